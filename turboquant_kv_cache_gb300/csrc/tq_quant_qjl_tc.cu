// Quantise with the QJL residual stage on the tensor cores: head_dim 128 (one
// norm per vector, the QJL layouts' block), fp16 input, m <= 128 projection
// rows, no norm correction.  Other QJL layouts use tq_quant_qjl.cu.
//
// Per tile of 128 vectors (one per TMEM lane):
//   1. Y = X (D H^T): the unnormalised rotation, one tcgen05 product (M 128,
//      N 128, K 128) of the TMA-loaded tile and the +-1 matrix;
//   2. per vector, in its thread: the norm (||y||^2 = 128 ||x||^2), the codes
//      (cell-table bucketize of tq_tc.cuh), and the residual in the rotated
//      domain, e = y / ||y|| - c (a zero vector has e = 0);
//   3. the projection of the residual back in the input domain,
//      S r = S (D H e / sqrt(128)) = S' e with S' = S D H / sqrt(128), which
//      each CTA builds once (a Walsh-Hadamard transform of every row of S
//      times D, in registers, while its first tiles load).  S' e runs as three fp16 products, S'_hi e_hi + S'_lo e_hi +
//      S'_hi e_lo (e scaled by 2^12 so its low halves stay normal), with fp32
//      accumulation: about 22 significant bits, so a sign can differ from the
//      exact one only for |S r| far below 1e-5.  e goes to TMEM (fp16 pairs,
//      the A operand), S' stays in shared memory, and the result overwrites
//      Y's columns, which have been read by then;
//   4. sign bits [S r >= 0], rho = ||e|| (fp16), codes and the fp16 norm.
//
// Roles: a producer thread (TMA, three stages of 32 KB), a warp issuing the
// rotations, a warp issuing the projections, and two groups of four consumer
// warps; group g owns TMEM columns 256 g .. 256 g + 255 (Y or S'e, then e)
// and takes the CTA's tiles i with i % 2 == g.  They meet only on
// mbarriers, every wait bounded at two levels as in tq_quant_fast.cu, and
// the producer and both product warps drain what they issued before the CTA
// frees its TMEM.
#include <mutex>

#include "tq_tc.cuh"

namespace tq {
namespace {

using namespace tcq;

constexpr int kD = 128;                      // head_dim (= block)
constexpr int kCons = 8;                     // consumer warps (two groups)
constexpr int kWarpProd = kCons, kWarpRot = kCons + 1, kWarpProj = kCons + 2;
constexpr int kThreads = 32 * (kCons + 3);
constexpr int kStages = 3;
constexpr uint32_t kStage = 128 * kD * 2;    // one tile: two 64-column swizzled boxes
constexpr uint32_t kBox = 128 * 64 * 2;
constexpr float kEScale = 4096.f;            // e * 2^12 before the fp16 split

// first failure status of a QJL quantise launch since the last read (0 = none)
__device__ int g_qjl_status;

struct QjlTcArgs {
  const __half* x;
  int64_t n_vec;
  int64_t stride;   // elements between rows
  const float* S;   // [m][128] fp32
  uint32_t* codes;
  uint16_t* scales;
  uint32_t* qjl;    // [records][m / 32]
  uint16_t* rnorm;
  RowMap map;       // vector -> record
  int64_t n_tiles;  // ceil(n_vec / 128)
  int64_t per_cta;  // tiles of each CTA (a contiguous range)
  uint64_t report_ns, hard_ns;
  CellTable ct;
  float cent[16];
};

template <int BITS>
__global__ void __launch_bounds__(kThreads, 1) quantize_qjl_tc_kernel(const CodecParams P, const QjlTcArgs a,
                                                                        const __grid_constant__ CUtensorMap xmap) {
  constexpr int WPV = kD * BITS / 32;   // code words per vector
  constexpr uint32_t kIdescRot = (1u << 4) | ((uint32_t)(kD >> 3) << 17) | ((uint32_t)(128 >> 4) << 24);
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // full / empty: stage landed / read by the rotation; tfull: Y in TMEM;
  // eready: e in TMEM and Y read (4 warps); pfull: S'e in TMEM; rfree: S'e
  // read (4 warps); drain: the product warps' last commits
  __shared__ __align__(8) uint64_t s_full[kStages], s_empty[kStages], s_tfull[2], s_eready[2], s_pfull[2],
      s_rfree[2], s_drain[2];
  __shared__ uint32_t s_tmem;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int m = P.m;
  uint8_t* smem = smem_raw + ((1024u - (su32(smem_raw) & 1023u)) & 1023u);
  uint8_t* s_x = smem;                                   // [kStages][2][128 rows x 64] swizzled
  uint8_t* s_b = s_x + kStages * kStage;                 // D H^T as [n][k] core matrices (32 KB)
  uint8_t* s_shi = s_b + kD * kD * 2;                    // S'_hi as [j][k] core matrices (m x 256 B)
  uint8_t* s_slo = s_shi + (size_t)m * kD * 2;           // S'_lo
  uint32_t* s_cell = reinterpret_cast<uint32_t*>(s_slo + (size_t)m * kD * 2);   // [C + 1][32]
  float* s_cent = reinterpret_cast<float*>(s_cell + (a.ct.n_cells + 1) * 32);   // [16][32]

  const int64_t t_begin = (int64_t)blockIdx.x * a.per_cta;
  const int64_t t_end = imin64(t_begin + a.per_cta, a.n_tiles);
  const int n = (int)(t_end > t_begin ? t_end - t_begin : 0);
  const uint32_t xs = su32(s_x);

  // S and the input may come from the previous kernel in the stream
  asm volatile("griddepcontrol.wait;\n" ::: "memory");
  if (warp == kWarpProd && lane == 0) {
    // barriers first (the other roles use them only after the set-up
    // barrier), then the first tiles, which load while the CTA sets up
    asm volatile("prefetch.tensormap [%0];\n" ::"l"(reinterpret_cast<uint64_t>(&xmap)) : "memory");
#pragma unroll
    for (int s = 0; s < kStages; ++s) {
      asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;\n" ::"r"(su32(&s_full[s])) : "memory");
      asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;\n" ::"r"(su32(&s_empty[s])) : "memory");
    }
#pragma unroll
    for (int b = 0; b < 2; ++b) {
      asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;\n" ::"r"(su32(&s_tfull[b])) : "memory");
      asm volatile("mbarrier.init.shared::cta.b64 [%0], 4;\n" ::"r"(su32(&s_eready[b])) : "memory");
      asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;\n" ::"r"(su32(&s_pfull[b])) : "memory");
      asm volatile("mbarrier.init.shared::cta.b64 [%0], 4;\n" ::"r"(su32(&s_rfree[b])) : "memory");
      asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;\n" ::"r"(su32(&s_drain[b])) : "memory");
    }
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
    for (int i = 0; i < n && i < kStages; ++i) {
      const int y = (int)((t_begin + i) * 128);
      arrive_expect_tx(su32(&s_full[i]), kStage);
      tma_load_2d(xs + i * kStage, &xmap, 0, y, su32(&s_full[i]));
      tma_load_2d(xs + i * kStage + kBox, &xmap, 64, y, su32(&s_full[i]));
    }
  }
  // S' = S D H / sqrt(128), one row per warp at a time: lane l holds
  // columns 4l .. 4l+3; the Walsh-Hadamard strides 1 and 2 stay in the lane,
  // strides 4 .. 64 pair lane l with lane l ^ (stride / 4)
  {
    const float inv_sqrt_d = 0.08838834764831845f;   // 1 / sqrt(128)
    const uint32_t dsg = (P.sign_bits[(4 * lane) >> 5] >> ((4 * lane) & 31)) & 0xFu;
    for (int j = warp; j < m; j += kThreads / 32) {
      const float4 sv = *reinterpret_cast<const float4*>(a.S + (size_t)j * kD + 4 * lane);
      float v[4] = {(dsg & 1u) ? -sv.x : sv.x, (dsg & 2u) ? -sv.y : sv.y, (dsg & 4u) ? -sv.z : sv.z,
                    (dsg & 8u) ? -sv.w : sv.w};
      float t0 = v[0] + v[1], t1 = v[0] - v[1], t2 = v[2] + v[3], t3 = v[2] - v[3];
      v[0] = t0 + t2; v[2] = t0 - t2; v[1] = t1 + t3; v[3] = t1 - t3;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const bool upper = lane & o;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float w = __shfl_xor_sync(kFull, v[e], o);
          v[e] = upper ? w - v[e] : v[e] + w;
        }
      }
      // fp16 high / low halves, rows j = N, columns k = K (core matrices)
      const __half2 h01 = __floats2half2_rn(v[0] * inv_sqrt_d, v[1] * inv_sqrt_d);
      const __half2 h23 = __floats2half2_rn(v[2] * inv_sqrt_d, v[3] * inv_sqrt_d);
      const float2 f01 = __half22float2(h01), f23 = __half22float2(h23);
      const __half2 l01 = __floats2half2_rn(v[0] * inv_sqrt_d - f01.x, v[1] * inv_sqrt_d - f01.y);
      const __half2 l23 = __floats2half2_rn(v[2] * inv_sqrt_d - f23.x, v[3] * inv_sqrt_d - f23.y);
      const uint32_t off = cm_off(j, 4 * lane, kD);   // 8-byte aligned: 4 columns of one core-matrix row
      *reinterpret_cast<uint2*>(s_shi + off) =
          make_uint2(*reinterpret_cast<const uint32_t*>(&h01), *reinterpret_cast<const uint32_t*>(&h23));
      *reinterpret_cast<uint2*>(s_slo + off) =
          make_uint2(*reinterpret_cast<const uint32_t*>(&l01), *reinterpret_cast<const uint32_t*>(&l23));
    }
  }
  // D H^T as B^T[n][k] = H[n][k] D_k (entries +-1)
  for (int idx = tid; idx < kD * (kD / 8); idx += kThreads) {
    const int nn = idx / (kD / 8), ch = idx % (kD / 8);
    uint32_t w[4];
#pragma unroll
    for (int e = 0; e < 8; e += 2) {
      uint32_t h2 = 0;
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        const int k = 8 * ch + e + q;
        const uint32_t neg = (__popc(nn & k) + (P.sign_bits[k >> 5] >> (k & 31))) & 1u;
        h2 |= (neg ? 0xBC00u : 0x3C00u) << (16 * q);
      }
      w[e >> 1] = h2;
    }
    *reinterpret_cast<uint4*>(s_b + cm_off(nn, 8 * ch, kD)) = make_uint4(w[0], w[1], w[2], w[3]);
  }
  for (int idx = tid; idx < (a.ct.n_cells + 1) * 32; idx += kThreads) s_cell[idx] = a.ct.cell[idx >> 5];
  for (int idx = tid; idx < 16 * 32; idx += kThreads) s_cent[idx] = a.cent[idx >> 5];
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;\n" ::"r"(su32(&s_tmem)),
                 "n"(512)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n" ::: "memory");
  }
  // B and S' were written by ordinary stores and are read by the tensor cores
  fence_async_smem();
  fence_before();
  __syncthreads();
  fence_after();
  const uint32_t tmem = s_tmem;
  asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");

  int failed = 0, late = 0;
  auto wait = [&](uint32_t bar, uint32_t parity) { return bar_wait(bar, parity, a.report_ns, a.hard_ns, late); };

  if (warp == kWarpProd) {
    // ================= producer (one thread): tile i >= kStages into stage
    // i % kStages once the rotation of tile i - kStages has read it
    if (lane == 0) {
      int i = kStages;
      for (; i < n; ++i) {
        const int s = i % kStages;
        if (!wait(su32(&s_empty[s]), (uint32_t)(i / kStages - 1) & 1)) {
          failed = 1;
          break;
        }
        const int y = (int)((t_begin + i) * 128);
        arrive_expect_tx(su32(&s_full[s]), kStage);
        tma_load_2d(xs + s * kStage, &xmap, 0, y, su32(&s_full[s]));
        tma_load_2d(xs + s * kStage + kBox, &xmap, 64, y, su32(&s_full[s]));
      }
      // drain: every load issued has landed (at most one phase per stage)
      if (i > n) i = n;
      for (int q = i > kStages ? i - kStages : 0; q < i; ++q)
        bar_wait(su32(&s_full[q % kStages]), (uint32_t)(q / kStages) & 1, a.hard_ns, a.hard_ns, late);
    }
    __syncwarp();
  } else if (warp == kWarpRot) {
    // ================= rotations: Y(b) = X(stage) (D H^T) once the stage has
    // landed and group b has read the previous S'e of its columns
    const uint64_t db = sdesc(su32(s_b), 128, kD * 16);
    for (int i = 0; i < n; ++i) {
      const int s = i % kStages, b = i & 1;
      const bool ok = wait(su32(&s_full[s]), (uint32_t)(i / kStages) & 1) &&
                      (i < 2 || wait(su32(&s_rfree[b]), (uint32_t)(i / 2 - 1) & 1));
      if (!__all_sync(kFull, ok)) {
        failed = 1;
        break;
      }
      fence_after();
      __syncwarp();
      // K steps of 16 columns: steps 0-3 in the first 64-column box, 4-7 in
      // the second, 32 bytes apart along the swizzled rows
#pragma unroll
      for (int k = 0; k < kD / 16; ++k) {
        const uint64_t da = sdesc_swz(xs + s * kStage + (k >> 2) * kBox, 128) + 2 * (k & 3);
        mma_ss_elect(tmem + 256 * b, da, db + 16 * k, kIdescRot, k > 0);
      }
      commit_elect(su32(&s_empty[s]));
      commit_elect(su32(&s_tfull[b]));
    }
    commit_elect(su32(&s_drain[0]));
    __all_sync(kFull, bar_wait(su32(&s_drain[0]), 0, a.hard_ns, a.hard_ns, late));
  } else if (warp == kWarpProj) {
    // ================= projections: S'e into group b's first 128 columns
    // once e is in its last 128 (hi pairs, then lo pairs)
    const uint32_t idesc = (1u << 4) | ((uint32_t)(m >> 3) << 17) | ((uint32_t)(128 >> 4) << 24);
    const uint64_t dhi = sdesc(su32(s_shi), 128, kD * 16), dlo = sdesc(su32(s_slo), 128, kD * 16);
    for (int i = 0; i < n; ++i) {
      const int b = i & 1;
      if (!__all_sync(kFull, wait(su32(&s_eready[b]), (uint32_t)(i / 2) & 1))) {
        failed = 1;
        break;
      }
      fence_after();
      __syncwarp();
      const uint32_t d = tmem + 256 * b, ehi = d + 128, elo = d + 192;
#pragma unroll
      for (int k = 0; k < kD / 16; ++k) mma_ts_elect(d, ehi + 8 * k, dhi + 16 * k, idesc, k > 0);
#pragma unroll
      for (int k = 0; k < kD / 16; ++k) mma_ts_elect(d, ehi + 8 * k, dlo + 16 * k, idesc, 1);
#pragma unroll
      for (int k = 0; k < kD / 16; ++k) mma_ts_elect(d, elo + 8 * k, dhi + 16 * k, idesc, 1);
      commit_elect(su32(&s_pfull[b]));
    }
    commit_elect(su32(&s_drain[1]));
    __all_sync(kFull, bar_wait(su32(&s_drain[1]), 0, a.hard_ns, a.hard_ns, late));
  } else {
    // ================= consumers: group g = warp / 4, vector 32 (warp % 4) + lane
    const int g = warp >> 2, wq = warp & 3;
    const int words_per_vec = P.code_bytes / 4;
    const float2 cells2 = make_float2((float)a.ct.n_cells, (float)a.ct.n_cells);
    const float2 magic2 = make_float2(kMagic, kMagic);
    const uint32_t cell_base = su32(s_cell) + 4u * lane - (__float_as_uint(kMagic) << 7);
    const uint32_t cent_base = su32(s_cent) + 4u * lane;
    const uint32_t lanes = (uint32_t)(32 * wq) << 16;
    for (int i = g; i < n; i += 2) {
      const int b = g;
      if (!__all_sync(kFull, wait(su32(&s_tfull[b]), (uint32_t)(i / 2) & 1))) {
        failed = 1;
        break;
      }
      fence_after();
      const uint32_t ty = tmem + lanes + 256 * b, te = ty + 128;
      // pass 1: ||y||^2 = 128 ||x||^2
      float2 s2 = make_float2(0.f, 0.f);
#pragma unroll
      for (int c0 = 0; c0 < kD; c0 += 32) {
        uint32_t v[32];
        TQ_LD32(ty + c0, v);
        asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory");
#pragma unroll
        for (int c = 0; c < 32; c += 2)
          s2 = __ffma2_rn(make_float2(__uint_as_float(v[c]), __uint_as_float(v[c + 1])),
                          make_float2(__uint_as_float(v[c]), __uint_as_float(v[c + 1])), s2);
      }
      const float ss = s2.x + s2.y;
      const float inv = ss > 0.f ? rsqrtf(ss) : 0.f;        // y / ||y|| = y * inv
      const float A1 = a.ct.inv2r * inv;
      const float ez = ss > 0.f ? kEScale : 0.f;            // a zero vector has e = 0
      // pass 2: codes (nibble words), e = y / ||y|| - c as fp16 hi / lo pairs
      uint32_t N[kD / 8];
      float r2 = 0.f;
#pragma unroll
      for (int c0 = 0; c0 < kD; c0 += 32) {
        uint32_t v[32], hi[16], lo[16];
        TQ_LD32(ty + c0, v);
        asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory");
#pragma unroll
        for (int pr = 0; pr < 16; ++pr) {
          const float y0 = __uint_as_float(v[2 * pr]), y1 = __uint_as_float(v[2 * pr + 1]);
          const float2 s = make_float2(__saturatef(fmaf(y0, A1, 0.5f)), __saturatef(fmaf(y1, A1, 0.5f)));
          const float2 u = __ffma2_rn(s, cells2, magic2);
          const uint32_t e0 = lds32(cell_base + (__float_as_uint(u.x) << 7));
          const uint32_t e1 = lds32(cell_base + (__float_as_uint(u.y) << 7));
          const uint32_t k0 = (e0 & 15u) + (s.x > __uint_as_float(e0) ? 1u : 0u);
          const uint32_t k1 = (e1 & 15u) + (s.y > __uint_as_float(e1) ? 1u : 0u);
          const int nw = (c0 + 2 * pr) >> 3, nib = (2 * pr) & 7;
          const uint32_t part = (k0 << (4 * nib)) | (k1 << (4 * nib + 4));
          N[nw] = nib == 0 ? part : (N[nw] | part);
          const float c0v = __uint_as_float(lds32(cent_base + (k0 << 7)));
          const float c1v = __uint_as_float(lds32(cent_base + (k1 << 7)));
          const float2 e = make_float2((fmaf(y0, inv, -c0v)) * ez, (fmaf(y1, inv, -c1v)) * ez);
          r2 = fmaf(e.x, e.x, fmaf(e.y, e.y, r2));
          const __half2 h2 = __floats2half2_rn(e.x, e.y);
          const float2 hf = __half22float2(h2);
          const __half2 l2 = __floats2half2_rn(e.x - hf.x, e.y - hf.y);
          hi[pr] = *reinterpret_cast<const uint32_t*>(&h2);
          lo[pr] = *reinterpret_cast<const uint32_t*>(&l2);
        }
        // coordinates c0 .. c0+31 are columns c0/2 .. c0/2+15 of each half
        TQ_ST16(te + c0 / 2, hi);
        TQ_ST16(te + 64 + c0 / 2, lo);
      }
      asm volatile("tcgen05.wait::st.sync.aligned;\n" ::: "memory");
      fence_before();
      __syncwarp();
      if (lane == 0) asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(su32(&s_eready[b])) : "memory");

      // codes and norm while the projection runs
      const int64_t v = (t_begin + i) * 128 + 32 * wq + lane;
      const int64_t r = v < a.n_vec ? map_row(a.map, v) : -1;
      uint32_t W[WPV];
#pragma unroll
      for (int gi = 0; gi < kD / 32; ++gi) {
        const uint32_t* G = N + 4 * gi;
        if (BITS == 4) {
#pragma unroll
          for (int w = 0; w < 4; ++w) W[4 * gi + w] = G[w];
        } else if (BITS == 3) {
#pragma unroll
          for (int w = 0; w < 3; ++w) W[3 * gi + w] = G[w] | (((G[3] >> w) & 0x11111111u) << 3);
        } else if (BITS == 2) {
#pragma unroll
          for (int w = 0; w < 2; ++w) W[2 * gi + w] = G[w] | (G[w + 2] << 2);
        } else {
          W[gi] = G[0] | (G[1] << 1) | (G[2] << 2) | (G[3] << 3);
        }
      }
      if (r >= 0) {
        uint32_t* dst = a.codes + r * words_per_vec;
        if (WPV % 4 == 0) {
#pragma unroll
          for (int w = 0; w < WPV; w += 4) *reinterpret_cast<uint4*>(dst + w) = make_uint4(W[w], W[w + 1], W[w + 2], W[w + 3]);
        } else {
#pragma unroll
          for (int w = 0; w < WPV; ++w) dst[w] = W[w];
        }
        a.scales[r] = f2h(sqrtf(ss * (1.0f / kD)));
        a.rnorm[r] = f2h(sqrtf(r2) * (1.0f / kEScale));
      }

      // sign bits of S'e
      if (!__all_sync(kFull, wait(su32(&s_pfull[b]), (uint32_t)(i / 2) & 1))) {
        failed = 1;
        break;
      }
      fence_after();
      uint32_t bits[4] = {0u, 0u, 0u, 0u};
#pragma unroll
      for (int c0 = 0; c0 < 128; c0 += 32) {
        if (c0 < m) {
          uint32_t pv[32];
          TQ_LD32(ty + c0, pv);
          asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory");
          uint32_t w = 0;
#pragma unroll
          for (int c = 0; c < 32; ++c) w |= (__uint_as_float(pv[c]) >= 0.f ? 1u : 0u) << c;
          bits[c0 / 32] = w;
        }
      }
      fence_before();
      __syncwarp();
      if (lane == 0) asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(su32(&s_rfree[b])) : "memory");
      if (r >= 0) {
        uint32_t* q = a.qjl + r * (m / 32);
        if (m == 128) {
          *reinterpret_cast<uint4*>(q) = make_uint4(bits[0], bits[1], bits[2], bits[3]);
        } else {
          for (int w = 0; w < m / 32; ++w) q[w] = bits[w];
        }
      }
    }
  }
  if (failed || late) atomicCAS(&g_qjl_status, 0, (int)TQ_ERR_TIMEOUT);
  fence_before();
  __syncthreads();
  if (warp == 0) {
    fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;\n" ::"r"(tmem), "n"(512) : "memory");
  }
}

struct Shape {
  bool ready = false;
  int sms = 0;
};

template <int BITS>
int launch_qjl_tc(const CodecParams& P, QjlTcArgs& a, cudaStream_t st) {
  static std::mutex mu;
  static Shape shapes[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return TQ_ERR_CUDA;
  auto kern = quantize_qjl_tc_kernel<BITS>;
  // stages (+ 1024 bytes of alignment slack), D H^T, S'_hi and S'_lo at the
  // largest m, cells, centroids
  const size_t smem = 1024 + (size_t)kStages * kStage + (size_t)kD * kD * 2 + 2 * (size_t)128 * kD * 2 +
                      (size_t)(kMaxCells + 1) * 32 * 4 + 16 * 32 * 4;
  int sms;
  {
    std::lock_guard<std::mutex> lock(mu);
    Shape& c = shapes[dev];
    if (!c.ready) {
      if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
        return TQ_ERR_CUDA;
      int v = 0;
      cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev);
      c.sms = v > 0 ? v : 1;
      c.ready = true;
    }
    sms = c.sms;
  }
  CUtensorMap xmap;
  if (!make_rows_map(a.x, kD, a.n_vec, a.stride, &xmap)) return TQ_ERR_UNSUPPORTED;
  const WaitLimits wl = wait_limits();
  a.report_ns = wl.report_ns;
  a.hard_ns = wl.hard_ns;
  a.n_tiles = (a.n_vec + 127) / 128;
  a.per_cta = (a.n_tiles + sms - 1) / sms;   // one CTA per SM (all 512 TMEM columns)
  const int64_t blocks = (a.n_tiles + a.per_cta - 1) / a.per_cta;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)blocks);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
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

// fp16 QJL layouts at head_dim 128, m <= 128, no norm correction.
bool quantize_qjl_tc_eligible(const CodecParams& P, bool f32_input) {
  if (f32_input || !P.m || P.nc || P.d != kD || P.blk != kD || P.m > 128 || P.m % 32 || P.bits < 1 || P.bits > 4)
    return false;
  CellTable ct;
  return make_cells(P, &ct);
}

int launch_quantize_qjl_tc(const CodecParams& P, const void* x, int64_t n_vec, int64_t stride, const float* S,
                           uint8_t* codes, uint16_t* scales, uint8_t* qjl_bits, uint16_t* qjl_rnorm, const RowMap& map,
                           cudaStream_t st) {
  QjlTcArgs a;
  if (!make_cells(P, &a.ct)) return TQ_ERR_UNSUPPORTED;
  a.x = static_cast<const __half*>(x);
  a.n_vec = n_vec;
  a.stride = stride;
  a.S = S;
  a.codes = reinterpret_cast<uint32_t*>(codes);
  a.scales = scales;
  a.qjl = reinterpret_cast<uint32_t*>(qjl_bits);
  a.rnorm = qjl_rnorm;
  a.map = map;
  for (int k = 0; k < 16; ++k) a.cent[k] = P.centroids[k];
  switch (P.bits) {
    case 1: return launch_qjl_tc<1>(P, a, st);
    case 2: return launch_qjl_tc<2>(P, a, st);
    case 3: return launch_qjl_tc<3>(P, a, st);
    default: return launch_qjl_tc<4>(P, a, st);
  }
}

// First failure status a QJL tensor-core quantise launch recorded since the
// last read with clear set (0 = none).
int quantize_qjl_tc_status(int clear, int* status) {
  int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_qjl_status, sizeof(int)) != cudaSuccess) return TQ_ERR_CUDA;
  if (clear && v != 0) {
    const int zero = 0;
    if (cudaMemcpyToSymbol(g_qjl_status, &zero, sizeof(int)) != cudaSuccess) return TQ_ERR_CUDA;
  }
  *status = v;
  return TQ_OK;
}

}  // namespace tq
