// Fast quantise path: fp16 input, rotation block of 32 or 64, 2-4 bits, no
// QJL, no norm correction (those layouts use the general kernel).
//
// A CTA quantises a contiguous range of tiles of 128 vectors x one rotation
// block.  The rotation of a tile is one small dense product on the tensor
// cores,
//   Y = X B,  B[k][n] = D_k H[n][k]  (entries +-1, exact in fp16),
// tcgen05.mma (M = 128 vectors, N = K = block) with the fp16 input tile and
// B in shared memory and the fp32 result in TMEM: the products are exact and
// the sums fp32, as in a scalar transform.  One consumer thread owns one
// vector (its TMEM lane), so the norm, the codes and the packed words of a
// vector never leave the thread.
//
// Roles: a producer thread loads input tiles with TMA (one 128-row box per
// tile, rows past the end zero-filled, 128- or 64-byte swizzled rows, the
// layout the MMA reads) ten stages deep, an MMA warp issues the products
// into eight TMEM accumulators, and four groups of four consumer warps take
// turns on the finished ones.  They meet only on mbarriers.  The producer
// issues the first loads before the CTA's set-up (B, the cell table, TMEM),
// and the kernel is launched as a programmatic dependent of the previous one
// in the stream, so both the set-up and the launch overlap other work.
//
// Codes come from the cell-table bucketize of tq_tc.cuh: one shared load and
// one compare per code.
//
// Every mbarrier wait is bounded.  A wait longer than the caller's limit
// records TQ_ERR_TIMEOUT in this file's device status word and goes on; one
// longer than the hard bound stops its role.  Before the CTA frees its TMEM
// and leaves, the producer waits for every load it issued and the MMA warp
// for every product (a final commit), so nothing in flight outlives it.
#include <mutex>

#include "tq_tc.cuh"

namespace tq {
namespace {

using namespace tcq;

// One CTA per SM.  Consumer warps: kGroups groups of four, group g takes the
// CTA's tiles i with i % kGroups == g; in a group, one vector per thread (one
// TMEM lane each)
constexpr int kGroups = 4;
constexpr int kConsumers = 4 * kGroups;
constexpr int kThreads = 32 * (kConsumers + 2);   // + a producer warp and an MMA warp
constexpr int kTileCols = 64;               // input columns per tile: one or two rotation blocks
constexpr int kStages = 10;                 // input stages (16 KB each)
constexpr int kAcc = 2 * kGroups;           // TMEM accumulators of 64 columns (two per group, all 512)

// first failure status of a quantise launch since the last read (0 = none)
__device__ int g_quant_status;

struct FastQuantArgs {
  const __half* x;
  int64_t n_vec;
  int64_t stride;   // elements between rows
  uint32_t* codes;  // [records][words per vector]
  uint16_t* scales;
  RowMap map;       // vector -> record
  int64_t n_tiles;  // ceil(n_vec / 128) * d / 64
  int64_t per_cta;  // tiles of each CTA (a contiguous range)
  uint64_t report_ns, hard_ns;   // wait limits (see WaitLimits)
  CellTable ct;     // bucketize cells
};

template <int BLK, int BITS>
__global__ void __launch_bounds__(kThreads, 1) quantize_tc_kernel(const CodecParams P, const FastQuantArgs a,
                                                                   const __grid_constant__ CUtensorMap xmap) {
  constexpr int CPR = BLK / 8;              // 16-byte chunks per row of B
  constexpr int BPT = kTileCols / BLK;      // rotation blocks per tile
  constexpr int STAGE = 128 * kTileCols * 2;   // bytes of one input tile
  constexpr uint32_t kCols = kAcc * kTileCols;  // TMEM columns: kAcc fp32 accumulators
  constexpr int WPB = BLK * BITS / 32;      // packed words per block
  // f32 accumulate, f16 A and B, both K-major, N = BLK, M = 128
  constexpr uint32_t kIdesc = (1u << 4) | ((uint32_t)(BLK >> 3) << 17) | ((uint32_t)(128 >> 4) << 24);
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // full: stage s loaded (TMA bytes); empty: its products read it;
  // tfull: accumulator b written; tempty: accumulator b read (4 warps)
  // drain: the MMA warp's last commit (every product it issued is done)
  __shared__ __align__(8) uint64_t s_full[kStages], s_empty[kStages], s_tfull[kAcc], s_tempty[kAcc], s_drain;
  __shared__ uint32_t s_tmem;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int nb = P.nb;
  const int tpg = nb / BPT;                 // tiles per 128-vector group
  // swizzled tiles want 1024-byte alignment (the launch adds the slack)
  uint8_t* smem = smem_raw + ((1024u - (su32(smem_raw) & 1023u)) & 1023u);
  uint8_t* s_x = smem;                                           // [kStages][128 rows x 64 columns] swizzled
  uint8_t* s_b = smem + kStages * STAGE;                         // [nb][BLK n x BLK k] core matrices
  uint32_t* s_cell = reinterpret_cast<uint32_t*>(s_b + (size_t)nb * BLK * BLK * 2);   // [C + 1][32]

  const int64_t t_begin = (int64_t)blockIdx.x * a.per_cta;
  const int64_t t_end = imin64(t_begin + a.per_cta, a.n_tiles);
  const int n = (int)(t_end > t_begin ? t_end - t_begin : 0);   // tiles of this CTA
  const uint32_t xs = su32(s_x), bs = su32(s_b);
  if (warp == kConsumers && lane == 0) {
    // barriers first, then (once the kernels this one depends on are done)
    // the first kStages tiles, so their loads overlap the set-up below
#pragma unroll
    for (int s = 0; s < kStages; ++s) {
      asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;\n" ::"r"(su32(&s_full[s])) : "memory");
      asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;\n" ::"r"(su32(&s_empty[s])) : "memory");
    }
#pragma unroll
    for (int b = 0; b < kAcc; ++b) {
      asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;\n" ::"r"(su32(&s_tfull[b])) : "memory");
      asm volatile("mbarrier.init.shared::cta.b64 [%0], 4;\n" ::"r"(su32(&s_tempty[b])) : "memory");
    }
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;\n" ::"r"(su32(&s_drain)) : "memory");
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
    asm volatile("prefetch.tensormap [%0];\n" ::"l"(reinterpret_cast<uint64_t>(&xmap)) : "memory");
    asm volatile("griddepcontrol.wait;\n" ::: "memory");
    int64_t vg = t_begin / tpg;
    int jt = (int)(t_begin - vg * tpg);
    for (int i = 0; i < n && i < kStages; ++i) {
      arrive_expect_tx(su32(&s_full[i]), STAGE);
      tma_load_2d(xs + i * STAGE, &xmap, jt * kTileCols, (int)(vg * 128), su32(&s_full[i]));
      if (++jt == tpg) { jt = 0; ++vg; }
    }
  }
  // B of every block j, stored as B^T (row n, column k): 8 k values per 16 bytes
  for (int idx = tid; idx < nb * BLK * CPR; idx += kThreads) {
    const int j = idx / (BLK * CPR);
    const int rem = idx - j * (BLK * CPR);
    const int nn = rem / CPR, ch = rem % CPR;
    uint32_t w[4];
#pragma unroll
    for (int e = 0; e < 8; e += 2) {
      uint32_t h2 = 0;
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        const int k = 8 * ch + e + q;
        const int c = j * BLK + k;
        const uint32_t neg = (__popc(nn & k) + (P.sign_bits[c >> 5] >> (c & 31))) & 1u;
        h2 |= (neg ? 0xBC00u : 0x3C00u) << (16 * q);
      }
      w[e >> 1] = h2;
    }
    *reinterpret_cast<uint4*>(s_b + (size_t)j * BLK * BLK * 2 + cm_off(nn, 8 * ch, BLK)) =
        make_uint4(w[0], w[1], w[2], w[3]);
  }
  for (int idx = tid; idx < (a.ct.n_cells + 1) * 32; idx += kThreads) s_cell[idx] = a.ct.cell[idx >> 5];
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;\n" ::"r"(su32(&s_tmem)),
                 "n"(kCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n" ::: "memory");
  }
  fence_async_smem();   // B, written by ordinary stores
  fence_before();
  __syncthreads();
  fence_after();
  const uint32_t tmem = s_tmem;

  // the next kernel in the stream may start its own set-up now
  asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
  int failed = 0;   // a wait of this thread gave up (hard bound); its role stops
  int late = 0;     // a wait of this thread passed the report limit
  auto wait = [&](uint32_t bar, uint32_t parity) { return bar_wait(bar, parity, a.report_ns, a.hard_ns, late); };

  if (warp == kConsumers) {
    // ================= producer (one thread): tile i >= kStages into stage
    // i % kStages once the products of tile i - kStages have read it
    if (lane == 0) {
      int64_t vg = (t_begin + kStages) / tpg;
      int jt = (int)(t_begin + kStages - vg * tpg);
      int i = kStages;
      for (; i < n; ++i) {
        const int s = i % kStages;
        if (!wait(su32(&s_empty[s]), (uint32_t)(i / kStages - 1) & 1)) {
          failed = 1;
          break;
        }
        arrive_expect_tx(su32(&s_full[s]), STAGE);
        tma_load_2d(xs + s * STAGE, &xmap, jt * kTileCols, (int)(vg * 128), su32(&s_full[s]));
        if (++jt == tpg) { jt = 0; ++vg; }
      }
      // drain: every load issued has landed before the CTA may leave (at
      // most one phase per stage is outstanding, so a parity wait is exact)
      const int issued = i < n ? i : n;
      for (int q = issued > kStages ? issued - kStages : 0; q < issued; ++q)
        bar_wait(su32(&s_full[q % kStages]), (uint32_t)(q / kStages) & 1, a.hard_ns, a.hard_ns, late);
    }
    __syncwarp();
  } else if (warp == kConsumers + 1) {
    // ================= MMA: for each block jj of tile i, columns
    // jj*BLK.. of accumulator b = X(stage, block jj) B_j, once the stage has
    // landed and accumulator b has been read
    int jt = (int)(t_begin % tpg);
    for (int i = 0; i < n; ++i) {
      const int s = i % kStages, b = i % kAcc;
      const bool ok = wait(su32(&s_full[s]), (uint32_t)(i / kStages) & 1) &&
                      (i < kAcc || wait(su32(&s_tempty[b]), (uint32_t)(i / kAcc - 1) & 1));
      if (!__all_sync(kFull, ok)) {
        failed = 1;
        break;
      }
      fence_after();
      __syncwarp();
      const uint64_t da = sdesc_swz(xs + s * STAGE, kTileCols * 2);
#pragma unroll
      for (int jj = 0; jj < BPT; ++jj) {
        const uint64_t db = sdesc(bs + (uint32_t)((jt * BPT + jj) * BLK * BLK * 2), 128, BLK * 16);
        // K step k: 32 bytes further along the swizzled A rows (block jj
        // starts jj*BLK*2 bytes in), two core matrices further along B
#pragma unroll
        for (int k = 0; k < BLK / 16; ++k)
          mma_ss_elect(tmem + b * kTileCols + jj * BLK, da + (jj * BLK * 2) / 16 + 2 * k, db + 16 * k, kIdesc, k > 0);
      }
      commit_elect(su32(&s_empty[s]));
      commit_elect(su32(&s_tfull[b]));
      if (++jt == tpg) jt = 0;
    }
    // drain: every product issued is done before TMEM is freed
    commit_elect(su32(&s_drain));
    __all_sync(kFull, bar_wait(su32(&s_drain), 0, a.hard_ns, a.hard_ns, late));
  } else {
    // ================= consumers: one vector per thread (TMEM lane
    // 32 (warp % 4) + lane, columns = coordinates of the tile)
    const int words_per_vec = P.code_bytes / 4;
    const float2 cells2 = make_float2((float)a.ct.n_cells, (float)a.ct.n_cells);
    const float2 magic2 = make_float2(kMagic, kMagic);
    // cell c of this lane's copy at s_cell + 4 (32 c + lane); the magic bits
    // of round(s C) + 1.5 * 2^23 are folded into the base (mod 2^32)
    const uint32_t cell_base = su32(s_cell) + 4u * lane - (__float_as_uint(kMagic) << 7);
    const int grp = warp >> 2, wq = warp & 3;   // group, quarter of the TMEM lanes
    int64_t vg = (t_begin + grp) / tpg;
    int jt = (int)(t_begin + grp - vg * tpg);
    for (int i = grp; i < n; i += kGroups) {
      const int b = i % kAcc;
      if (!__all_sync(kFull, wait(su32(&s_tfull[b]), (uint32_t)(i / kAcc) & 1))) {
        failed = 1;
        break;
      }
      fence_after();
      const uint32_t taddr = tmem + ((uint32_t)(32 * wq) << 16) + (uint32_t)(b * kTileCols);
      const int64_t v = vg * 128 + 32 * wq + lane;
      const int64_t r = v < a.n_vec ? map_row(a.map, v) : -1;
#pragma unroll
      for (int jj = 0; jj < BPT; ++jj) {
        const int j = jt * BPT + jj;
        const uint32_t tb = taddr + jj * BLK;
        // pass 1: ||y||^2 = BLK ||x||^2 over the block's columns
        float2 s2 = make_float2(0.f, 0.f);
#pragma unroll
        for (int c0 = 0; c0 < BLK; c0 += 32) {
          uint32_t vv[32];
          TQ_LD32(tb + c0, vv);
          asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory");
#pragma unroll
          for (int c = 0; c < 32; c += 2)
            s2 = __ffma2_rn(make_float2(__uint_as_float(vv[c]), __uint_as_float(vv[c + 1])),
                            make_float2(__uint_as_float(vv[c]), __uint_as_float(vv[c + 1])), s2);
        }
        const float ss = s2.x + s2.y;
        const float A1 = ss > 0.f ? a.ct.inv2r * rsqrtf(ss) : 0.f;
        // pass 2, 32 coordinates at a time: nibble word c holds the codes of
        // coordinates 8c .. 8c+7; a coordinate pair forms one byte, inserted
        // with a byte permute
        uint32_t N[BLK / 8];
#pragma unroll
        for (int c0 = 0; c0 < BLK; c0 += 32) {
          uint32_t vv[32];
          TQ_LD32(tb + c0, vv);
          asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory");
#pragma unroll
          for (int cc = 0; cc < 4; ++cc) {
            uint32_t w = 0;
#pragma unroll
            for (int m = 0; m < 4; ++m) {
              const float y0 = __uint_as_float(vv[8 * cc + 2 * m]), y1 = __uint_as_float(vv[8 * cc + 2 * m + 1]);
              const float2 s = make_float2(__saturatef(fmaf(y0, A1, 0.5f)), __saturatef(fmaf(y1, A1, 0.5f)));
              const float2 u = __ffma2_rn(s, cells2, magic2);
              const uint32_t e0 = lds32(cell_base + (__float_as_uint(u.x) << 7));
              const uint32_t e1 = lds32(cell_base + (__float_as_uint(u.y) << 7));
              // low byte: count of e0 | count of e1 << 4 (higher bytes are dropped)
              const uint32_t pair = (e0 & 0x0Fu) | ((e1 << 4) & ~0x0Fu);
              w = prmt(w, pair, m == 0 ? 0x3214u : m == 1 ? 0x3240u : m == 2 ? 0x3410u : 0x4210u);
              add_if_gt(w, s.x, e0, 1u << (8 * m));
              add_if_gt(w, s.y, e1, 1u << (8 * m + 4));
            }
            N[c0 / 8 + cc] = w;
          }
        }
        // packed words of the block (32-code groups of four nibble words)
        uint32_t W[WPB];
#pragma unroll
        for (int gi = 0; gi < BLK / 32; ++gi) {
          const uint32_t* G = N + 4 * gi;
          if (BITS == 4) {
#pragma unroll
            for (int w = 0; w < 4; ++w) W[4 * gi + w] = G[w];
          } else if (BITS == 3) {
#pragma unroll
            for (int w = 0; w < 3; ++w) W[3 * gi + w] = G[w] | (((G[3] >> w) & 0x11111111u) << 3);
          } else {
#pragma unroll
            for (int w = 0; w < 2; ++w) W[2 * gi + w] = G[w] | (G[w + 2] << 2);
          }
        }
        if (r >= 0) {
          uint32_t* dst = a.codes + r * words_per_vec + j * WPB;
          // widest store the record and block alignment allow
          if (WPB % 4 == 0 && words_per_vec % 4 == 0) {
#pragma unroll
            for (int w = 0; w < WPB; w += 4)
              *reinterpret_cast<uint4*>(dst + w) = make_uint4(W[w], W[w + 1], W[w + 2], W[w + 3]);
          } else if (WPB % 2 == 0 && words_per_vec % 2 == 0) {
#pragma unroll
            for (int w = 0; w < WPB; w += 2) *reinterpret_cast<uint2*>(dst + w) = make_uint2(W[w], W[w + 1]);
          } else {
#pragma unroll
            for (int w = 0; w < WPB; ++w) dst[w] = W[w];
          }
          a.scales[r * nb + j] = f2h(sqrtf(ss * (1.0f / BLK)));
        }
      }
      fence_before();
      __syncwarp();
      if (lane == 0) asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(su32(&s_tempty[b])) : "memory");
      jt += kGroups;   // the group's next tile
      while (jt >= tpg) { jt -= tpg; ++vg; }
    }
  }
  if (failed || late) atomicCAS(&g_quant_status, 0, (int)TQ_ERR_TIMEOUT);
  fence_before();
  __syncthreads();
  if (warp == 0) {
    fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;\n" ::"r"(tmem), "n"(kCols) : "memory");
  }
}

// Launch shape of one kernel instantiation on one device, worked out once.
struct LaunchShape {
  bool ready = false;
  int sms = 0, occ = 0;
  size_t smem = 0;
};

template <int BLK, int BITS>
int launch_fast(const CodecParams& P, FastQuantArgs& a, cudaStream_t st) {
  static std::mutex mu;
  static LaunchShape shapes[64][5];   // [device][nb - 1 for nb = 1, 2, 4, 8 -> index by log2]
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return TQ_ERR_CUDA;
  int lg = 0;
  while ((1 << lg) < P.nb && lg < 4) ++lg;
  auto kern = quantize_tc_kernel<BLK, BITS>;
  LaunchShape sh;
  {
    std::lock_guard<std::mutex> lock(mu);
    LaunchShape& c = shapes[dev][lg];
    if (!c.ready) {
      int sms = 0, smem_sm = 0, smem_blk_res = 0;
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
      cudaDeviceGetAttribute(&smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev);
      cudaDeviceGetAttribute(&smem_blk_res, cudaDevAttrReservedSharedMemoryPerBlock, dev);
      // stages (+ 1024 bytes of alignment slack), B of every block, cell table
      const size_t smem = 1024 + (size_t)kStages * 128 * kTileCols * 2 + (size_t)P.nb * BLK * BLK * 2 +
                          (size_t)(kMaxCells + 1) * 32 * 4;
      cudaFuncAttributes fa;
      if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess ||
          cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, 100) != cudaSuccess ||
          cudaFuncGetAttributes(&fa, kern) != cudaSuccess)
        return TQ_ERR_CUDA;
      // CTAs per SM: shared memory, registers, and TMEM (kAcc * 64 of 512 columns)
      int occ = (int)((size_t)smem_sm / (smem + fa.sharedSizeBytes + (size_t)smem_blk_res));
      const int by_regs = 65536 / (kThreads * (fa.numRegs > 0 ? fa.numRegs : 1));
      occ = occ < by_regs ? occ : by_regs;
      occ = occ < 512 / (kAcc * kTileCols) ? occ : 512 / (kAcc * kTileCols);
      c.sms = sms > 0 ? sms : 1;
      c.occ = occ > 0 ? occ : 1;
      c.smem = smem;
      c.ready = true;
    }
    sh = c;
  }
  CUtensorMap xmap;
  if (!make_rows_map(a.x, P.d, a.n_vec, a.stride, &xmap)) return TQ_ERR_UNSUPPORTED;
  const WaitLimits wl = wait_limits();
  a.report_ns = wl.report_ns;
  a.hard_ns = wl.hard_ns;
  a.n_tiles = (a.n_vec + 127) / 128 * (P.d / kTileCols);
  // every CTA takes the same number of tiles, so no CTA runs a tail alone
  const int64_t max_ctas = (int64_t)sh.sms * sh.occ;
  a.per_cta = (a.n_tiles + max_ctas - 1) / max_ctas;
  const int64_t blocks = (a.n_tiles + a.per_cta - 1) / a.per_cta;
  // programmatic dependent launch: this kernel's set-up may overlap the tail
  // of the previous kernel in the stream (its loads wait for that kernel)
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)blocks);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = sh.smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, kern, P, a, xmap) != cudaSuccess) return TQ_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? TQ_OK : TQ_ERR_CUDA;
}

}  // namespace

bool quantize_fast_eligible(const CodecParams& P, bool f32_input) {
  if (f32_input || P.m || P.nc || (P.blk != 32 && P.blk != 64) || P.bits < 2 || P.bits > 4 || P.d % kTileCols)
    return false;
  CellTable ct;
  return make_cells(P, &ct);
}

int launch_quantize_fast(const CodecParams& P, const void* x, int64_t n_vec, int64_t stride, uint8_t* codes,
                         uint16_t* scales, const RowMap& map, cudaStream_t st) {
  FastQuantArgs a;
  if (!make_cells(P, &a.ct)) return TQ_ERR_UNSUPPORTED;
  a.map = map;
  a.x = static_cast<const __half*>(x);
  a.n_vec = n_vec;
  a.stride = stride;
  a.codes = reinterpret_cast<uint32_t*>(codes);
  a.scales = scales;
  if (P.blk == 64) {
    if (P.bits == 4) return launch_fast<64, 4>(P, a, st);
    if (P.bits == 3) return launch_fast<64, 3>(P, a, st);
    return launch_fast<64, 2>(P, a, st);
  }
  if (P.bits == 4) return launch_fast<32, 4>(P, a, st);
  if (P.bits == 3) return launch_fast<32, 3>(P, a, st);
  return launch_fast<32, 2>(P, a, st);
}

// First failure status a fast quantise launch recorded since the last read
// with clear set (0 = none).
int quantize_fast_status(int clear, int* status) {
  int s = 0;
  if (cudaMemcpyFromSymbol(&s, g_quant_status, sizeof(int)) != cudaSuccess) return TQ_ERR_CUDA;
  if (clear && s != 0) {
    const int zero = 0;
    if (cudaMemcpyToSymbol(g_quant_status, &zero, sizeof(int)) != cudaSuccess) return TQ_ERR_CUDA;
  }
  *status = s;
  return TQ_OK;
}

}  // namespace tq
