// Prefill attention over the packed cache on the 5th-generation tensor cores
// (tcgen05, TMEM accumulators).
//
// Rows: every (batch, KV head) owns R = Tq*G query rows (query i, head h ->
// row i*G + h).  A CTA takes 128 rows (one per thread and per TMEM lane) and
// one slice of the context, walking it in 64-token tiles:
//   * the tile's K and V records are decoded by all 128 threads into shared
//     memory (rotated domain, centroid * block norm, fp16) in the canonical
//     no-swizzle core-matrix layout (8 rows x 16 bytes per core matrix), which
//     serves K as a K-major B operand of S = Q K^T and V as an MN-major B
//     operand of O = P V; both tiles are double-buffered so the decode of the
//     next tile overlaps the MMAs of the current one;
//   * one thread issues S = Q^ K^^T (M 128, N 64, K d) into TMEM;
//   * each thread reads its row of S, applies the causal / context mask and
//     an online softmax in base 2 (the reference max moves only when a score
//     exceeds it by more than 2^8), writes P as fp16 back into TMEM;
//   * one thread issues O += P V^ (A = P from TMEM, M 128, N d, K 64).
// Q^ = H D q per K block times softmax_scale * log2 e is prepared once per
// call by a small kernel.  Partial (m, l, O) per row and context slice go to
// the workspace in the decode-split format, and the decode combine kernel
// merges the slices and rotates each output row back (D H per V block).
// Every mbarrier wait is bounded: on expiry the CTA records an error word in
// the workspace, frees its TMEM and returns.
#include <cuda_runtime.h>
#include <math.h>

#include "tq_device.cuh"
#include "tq_lut.cuh"

namespace tq {

int decode_combine(const CodecParams& PV, const float* part, int n_split, uint16_t* out, int rows, cudaStream_t s);
int sm_count();

namespace {

constexpr int kRowsTc = 128;     // query rows per CTA (TMEM lanes)
constexpr int kThrTc = 256;      // 8 warps: all decode; warps 0-3 own the 128 TMEM rows
constexpr int kThrTcConst = kThrTc;
constexpr int kTok = 64;         // tokens per KV tile
constexpr int kProducerWarps = 8;   // decoding warps of the warp-specialised kernel
constexpr uint32_t kColS = 0, kColP = 64;
// TMEM columns: S (64 fp32) at 0, P (64 fp16 = 32 columns) at 64, Q^ (D fp16
// = D/2 columns) at 128, O (D fp32) after it; a power of two >= the total
template <int D> __host__ __device__ constexpr uint32_t col_o() { return 128u + D / 2; }
template <int D> __host__ __device__ constexpr uint32_t tmem_cols() { return col_o<D>() + D <= 256u ? 256u : 512u; }
constexpr float kLazyP = 8.0f;
constexpr int kWaitLimit = 1 << 24;

__device__ __forceinline__ uint32_t su32(const void* p) { return static_cast<uint32_t>(__cvta_generic_to_shared(p)); }

// byte offset of element (row, col) in a core-matrix tile of `cols` columns:
// core matrix (row/8, col/8) at ((row/8) * (cols/8) + col/8) * 128, row-major
// 8 x 16 bytes inside.
__device__ __forceinline__ uint32_t cm_off(int row, int col, int cols) {
  return (uint32_t)(((row >> 3) * (cols >> 3) + (col >> 3)) * 128 + (row & 7) * 16 + (col & 7) * 2);
}

__device__ __forceinline__ uint64_t sdesc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  return (uint64_t)((saddr >> 4) & 0x3FFF) | ((uint64_t)((lbo >> 4) & 0x3FFF) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFF) << 32) | ((uint64_t)1 << 46);
}

__device__ __forceinline__ void mma_ss(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, int acc) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d),
      "l"(a), "l"(b), "r"(idesc), "r"(acc)
      : "memory");
}

__device__ __forceinline__ void mma_ts(uint32_t d, uint32_t a, uint64_t b, uint32_t idesc, int acc) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(d),
      "r"(a), "l"(b), "r"(idesc), "r"(acc)
      : "memory");
}

__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool bar_wait(uint32_t bar, uint32_t phase) {
  uint32_t done = 0;
  for (int it = 0; it < kWaitLimit && !done; ++it)
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(done)
        : "r"(bar), "r"(phase)
        : "memory");
  return done != 0;
}

__device__ __forceinline__ void fence_before() { asm volatile("tcgen05.fence::before_thread_sync;\n" ::: "memory"); }
__device__ __forceinline__ void fence_after() { asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory"); }

#define TQ_LD32(taddr, v)                                                                                          \
  asm volatile(                                                                                                    \
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,"  \
      "%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n"                                             \
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),            \
        "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15]),      \
        "=r"(v[16]), "=r"(v[17]), "=r"(v[18]), "=r"(v[19]), "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]),    \
        "=r"(v[24]), "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31])     \
      : "r"(taddr))

#define TQ_ST32(taddr, v)                                                                                          \
  asm volatile(                                                                                                    \
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,"   \
      "%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};\n" ::"r"(taddr),                              \
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]),           \
      "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]), "r"(v[16]), "r"(v[17]),   \
      "r"(v[18]), "r"(v[19]), "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]), "r"(v[24]), "r"(v[25]), "r"(v[26]),  \
      "r"(v[27]), "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31])                                                   \
      : "memory")

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}

__device__ __forceinline__ float ex2f(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// fp16 centroid byte tables: lo/hi bytes of entries 0-3 / 4-7 (t[0..3]) and,
// for 4-bit codebooks, of entries 8-11 / 12-15 (t[4..7]).
// Packed bytes of tokens [t0, t0 + n) of one array (codes or scales; `sb`
// bytes per token) staged into smem: the copy starts at the 16-byte boundary
// at or below the first byte and never reads past the last byte needed.
// Returns the offset of the first byte inside the staging area.
__device__ __forceinline__ int stage_bytes(uint8_t* dst, const uint8_t* src_base, int64_t first_rec, int n, int sb,
                                           int tid, int nthr) {
  const int64_t s = first_rec * sb, e = s + (int64_t)n * sb;
  const int64_t s0 = s & ~(int64_t)15;
  const int chunks = (int)((e - s0 + 15) >> 4);
  for (int c = tid; c < chunks; c += nthr) {
    const int64_t at = s0 + 16 * (int64_t)c;
    const int64_t rem = e - at;
    const int bytes = rem >= 16 ? 16 : (int)rem;
    asm volatile("cp.async.ca.shared.global [%0], [%1], 16, %2;\n" ::"r"(su32(dst + 16 * c)), "l"(src_base + at),
                 "r"(bytes));
  }
  return (int)(s - s0);
}

struct PackedSlot {   // offsets of the four arrays inside one staging slot
  int kc, ks, vc, vs;
};

__device__ __forceinline__ uint32_t lds32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.b32 %0, [%1];\n" : "=r"(v) : "r"(addr));
  return v;
}
__device__ __forceinline__ uint16_t lds16(uint32_t addr) {
  uint16_t v;
  asm volatile("ld.shared.u16 %0, [%1];\n" : "=h"(v) : "r"(addr));
  return v;
}
__device__ __forceinline__ void sts128(uint32_t addr, uint4 v) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};\n" ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
               : "memory");
}

// Per-thread constants of the tile decoder: the thread's (token, 32-value
// group) work items and their byte offsets, the same for every tile.
template <int D, int NT = kThrTcConst>
struct ItemPlan {
  static constexpr int G8 = D / 32;
  static constexpr int N = (kTok * G8 + NT - 1) / NT;   // items per decoding thread
  int tok[N];
  uint32_t code_off[N], sc_off[N], dst_off[N];
};

template <int D, int NT = kThrTcConst>
__device__ __forceinline__ ItemPlan<D, NT> make_plan(const CodecParams& P, int tid) {
  ItemPlan<D, NT> pl;
  constexpr int G8 = D / 32;
#pragma unroll
  for (int k = 0; k < ItemPlan<D, NT>::N; ++k) {
    const int item = tid + k * NT;
    const int tok = 8 * (item / (8 * G8)) + (item & 7);
    const int grp = (item >> 3) % G8;
    pl.tok[k] = item < kTok * G8 ? tok : kTok;   // kTok: no item
    pl.code_off[k] = (uint32_t)(tok * P.code_bytes + grp * 4 * P.bits);
    pl.sc_off[k] = (uint32_t)(tok * P.nb * 2 + ((32 * grp) / P.blk) * 2);
    pl.dst_off[k] = cm_off(tok, 32 * grp, D);
  }
  return pl;
}

// Decode one kTok-token tile from its staged packed bytes (shared addresses
// codes / scales) into a core-matrix tile [kTok][D] at shared address tile:
// rotated, scaled fp16; tokens >= n_valid become zeros.  Work items are
// (token, 32-value group) pairs, so every thread runs the same instructions;
// 8 consecutive items are 8 tokens of one group, which spread one 16-byte
// store per lane over all banks.  Up to 3 bits the group's fp16 table is the
// centroids times its norm; 4-bit codes multiply after the lookup.
template <int D, int BITS, int NT>
__device__ __forceinline__ void decode_tile_items(const ItemPlan<D, NT>& pl, const uint32_t* c2, const Tab& fixed,
                                                  uint32_t codes, uint32_t scales, int n_valid, uint32_t tile) {
#pragma unroll
  for (int k = 0; k < ItemPlan<D, NT>::N; ++k) {
    if (pl.tok[k] >= kTok) continue;   // only when kTok * D/32 is not a multiple of the thread count
    const uint32_t dst = tile + pl.dst_off[k];
    if (n_valid == kTok || pl.tok[k] < n_valid) {
      uint32_t w[4], n[4];
#pragma unroll
      for (int b = 0; b < BITS; ++b) w[b] = lds32(codes + pl.code_off[k] + 4 * b);
      chunk_words<BITS>(w, n);
      const uint32_t sc = lds16(scales + pl.sc_off[k]);
      Tab T;
      uint32_t s2 = 0;
      if (BITS == 4) {
        T = fixed;
        s2 = sc | (sc << 16);
      } else {
        T = make_tab_p<BITS>(c2, sc);
      }
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t o[4];
        lut8<BITS>(n[c], T, o);
        if (BITS == 4) {
#pragma unroll
          for (int e = 0; e < 4; ++e) o[e] = lut_hmul2(o[e], s2);
        }
        sts128(dst + 128 * c, make_uint4(o[0], o[1], o[2], o[3]));
      }
    } else {
#pragma unroll
      for (int c = 0; c < 4; ++c) sts128(dst + 128 * c, make_uint4(0u, 0u, 0u, 0u));
    }
  }
}

// One codebook in the forms the tile decoder uses: fp16 centroid pairs
// (16 entries, unused ones zero) and, for 4-bit codes, the unscaled tables.
struct CodeTabs {
  uint32_t c2[8];
  Tab fixed;
};
__device__ __forceinline__ CodeTabs make_code_tabs(const CodecParams& P) {
  CodeTabs c;
#pragma unroll
  for (int k = 0; k < 8; ++k)
    c.c2[k] = (uint32_t)f2h(P.centroids[2 * k]) | ((uint32_t)f2h(P.centroids[2 * k + 1]) << 16);
  c.fixed = make_tab_p<4>(c.c2, 0x3C00u);
  return c;
}

template <int D, int NT>
__device__ __forceinline__ void decode_tile_smem(int bits, const ItemPlan<D, NT>& pl, const CodeTabs& ct,
                                                 uint32_t codes, uint32_t scales, int n_valid, uint32_t tile) {
  switch (bits) {
    case 4: decode_tile_items<D, 4, NT>(pl, ct.c2, ct.fixed, codes, scales, n_valid, tile); break;
    case 3: decode_tile_items<D, 3, NT>(pl, ct.c2, ct.fixed, codes, scales, n_valid, tile); break;
    case 2: decode_tile_items<D, 2, NT>(pl, ct.c2, ct.fixed, codes, scales, n_valid, tile); break;
    default: decode_tile_items<D, 1, NT>(pl, ct.c2, ct.fixed, codes, scales, n_valid, tile); break;
  }
}

struct PrefillTcArgs {
  const uint8_t* kc;
  const uint8_t* ks;
  const uint8_t* vc;
  const uint8_t* vs;
  const __half* qhat;   // [B*Hkv][R_pad][D]
  float* part;          // [(b*Hq + h)*Tq + i][n_split][D + 4]
  int* err;
  int64_t S_cap, ctx;
  int Hq, Hkv, Tq, R_pad, n_split, causal;
  int64_t per;          // tokens per split (multiple of kTok)
  int slot_bytes;       // one packed staging slot
  PackedSlot slot;
};


template <int D>
__global__ void __launch_bounds__(kThrTc, 1) prefill_tc_kernel(const CodecParams PK, const CodecParams PV,
                                                               const PrefillTcArgs a) {
  constexpr uint32_t kTmemCols = tmem_cols<D>();
  constexpr uint32_t kColQ = 128;                 // Q^ as the A operand of S, D/2 columns
  constexpr uint32_t kColO = col_o<D>();          // O accumulator, D columns
  constexpr uint32_t kTileBytes = kTok * D * 2;
  constexpr uint32_t kGroupBytes = (D / 8) * 128;   // one 8-row band of a [rows][D] core-matrix tile
  extern __shared__ __align__(1024) uint8_t smem[];
  // buffers b = 0, 1: decoded K and V tiles, staged packed bytes
  const uint32_t a_smem = su32(smem);
  auto aK = [&](int kb) { return a_smem + (uint32_t)kb * kTileBytes; };
  auto aV = [&](int kb) { return a_smem + (uint32_t)(2 + kb) * kTileBytes; };
  auto aPk = [&](int kb) { return a_smem + 4 * kTileBytes + (uint32_t)(kb * a.slot_bytes); };
  auto sPk = [&](int kb) { return smem + 4 * kTileBytes + kb * a.slot_bytes; };
  __shared__ __align__(8) uint64_t bar_s, bar_o;
  __shared__ uint32_t tmem_base;
  __shared__ int s_off[2][4];   // byte offsets of the staged arrays per slot

  const int tid = threadIdx.x, warp = tid >> 5;
  const bool row_warp = warp < 4;
  const int G = a.Hq / a.Hkv;
  const int rt = blockIdx.x;          // row tile
  const int split = blockIdx.y;
  const int bh = blockIdx.z;
  const int b = bh / a.Hkv, kvh = bh % a.Hkv;
  const int R = a.Tq * G;
  const int row = rt * kRowsTc + (tid & 127);   // row of this thread (row warps)
  const bool row_ok = row_warp && row < R;
  const int qi = row < R ? row / G : a.Tq - 1;
  const int64_t pos = a.ctx - a.Tq + qi;

  const int last_row = min(rt * kRowsTc + kRowsTc, R) - 1;
  const int64_t max_pos = a.causal ? a.ctx - a.Tq + last_row / G : a.ctx - 1;
  const int64_t t_lo = (int64_t)split * a.per;
  const int64_t t_hi = imin64(imin64(t_lo + a.per, a.ctx), max_pos + 1);
  const int n_tiles = t_hi > t_lo ? (int)((t_hi - t_lo + kTok - 1) / kTok) : 0;
  const int64_t rec0 = (int64_t)bh * a.S_cap;

  auto stage = [&](int tile, int slot) {   // packed bytes of `tile` into staging slot `slot`
    if (tile < n_tiles) {
      const int64_t t0 = t_lo + (int64_t)tile * kTok;
      const int n = (int)imin64(kTok, t_hi - t0);
      uint8_t* base = sPk(slot);
      const int o0 = stage_bytes(base + a.slot.kc, a.kc, rec0 + t0, n, PK.code_bytes, tid, kThrTc);
      const int o1 = stage_bytes(base + a.slot.ks, a.ks, rec0 + t0, n, 2 * PK.nb, tid, kThrTc);
      const int o2 = stage_bytes(base + a.slot.vc, a.vc, rec0 + t0, n, PV.code_bytes, tid, kThrTc);
      const int o3 = stage_bytes(base + a.slot.vs, a.vs, rec0 + t0, n, 2 * PV.nb, tid, kThrTc);
      if (tid == 0) {
        s_off[slot][0] = o0; s_off[slot][1] = o1; s_off[slot][2] = o2; s_off[slot][3] = o3;
      }
    }
    asm volatile("cp.async.commit_group;\n" ::);
  };
  auto n_valid_of = [&](int tile) { return (int)imin64(kTok, t_hi - (t_lo + (int64_t)tile * kTok)); };
  const CodeTabs lk = make_code_tabs(PK), lv = make_code_tabs(PV);
  const ItemPlan<D> plk = make_plan<D>(PK, tid), plv = make_plan<D>(PV, tid);
  const int kbits = PK.bits, vbits = PV.bits;

  stage(0, 0);
  stage(1, 1);
  if (tid == 0) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;\n" ::"r"(su32(&bar_s)) : "memory");
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;\n" ::"r"(su32(&bar_o)) : "memory");
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;\n" ::"r"(su32(&tmem_base)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n" ::: "memory");
  }
  fence_before();
  __syncthreads();
  fence_after();
  const uint32_t tmem = tmem_base;
  const uint32_t lane_base = tmem + ((uint32_t)(32 * (warp & 3)) << 16);
  // Q^ rows into TMEM (A operand of S: 2 fp16 per column)
  if (row_warp) {
    const __half* src = a.qhat + ((int64_t)bh * a.R_pad + (int64_t)rt * kRowsTc + tid) * D;
#pragma unroll 1
    for (int c0 = 0; c0 < D / 2; c0 += 32) {
      uint32_t w[32];
#pragma unroll
      for (int j = 0; j < 32; j += 4) {
        const uint4 v = *reinterpret_cast<const uint4*>(src + 2 * (c0 + j));
        w[j] = v.x; w[j + 1] = v.y; w[j + 2] = v.z; w[j + 3] = v.w;
      }
      TQ_ST32(lane_base + kColQ + c0, w);
    }
    asm volatile("tcgen05.wait::st.sync.aligned;\n" ::: "memory");
  }
  // tile 0 decoded before the first MMA
  asm volatile("cp.async.wait_group 1;\n" ::);
  __syncthreads();
  if (n_tiles > 0) {
    decode_tile_smem<D, kThrTcConst>(kbits, plk, lk, aPk(0) + a.slot.kc + s_off[0][0], aPk(0) + a.slot.ks + s_off[0][1], n_valid_of(0),
                        aK(0));
    decode_tile_smem<D, kThrTcConst>(vbits, plv, lv, aPk(0) + a.slot.vc + s_off[0][2], aPk(0) + a.slot.vs + s_off[0][3], n_valid_of(0),
                        aV(0));
  }
  asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
  fence_before();
  __syncthreads();
  fence_after();

  const uint32_t idesc_s = (1u << 4) | ((uint32_t)(kTok >> 3) << 17) | ((uint32_t)(kRowsTc >> 4) << 24);
  const uint32_t idesc_o = (1u << 4) | (1u << 16) | ((uint32_t)(D >> 3) << 17) | ((uint32_t)(kRowsTc >> 4) << 24);
  auto issue_s = [&](int kb) {   // S = Q^ (TMEM) K^(buffer kb)^T
#pragma unroll 4
    for (int s = 0; s < D / 16; ++s)
      mma_ts(tmem + kColS, tmem + kColQ + 8 * s, sdesc(aK(kb) + s * 256, 128, kGroupBytes), idesc_s, s > 0);
    mma_commit(su32(&bar_s));
  };
  auto issue_o = [&](int vb, bool first) {   // O += P (TMEM) V^(buffer vb)
#pragma unroll
    for (int s = 0; s < kTok / 16; ++s)
      mma_ts(tmem + kColO, tmem + kColP + 8 * s, sdesc(aV(vb) + s * 2 * kGroupBytes, kGroupBytes, 128), idesc_o,
             (first && s == 0) ? 0 : 1);
    mma_commit(su32(&bar_o));
  };

  bool ok = true;
  if (tid == 0 && n_tiles > 0) issue_s(0);
  float m_run = -INFINITY, l_run = 0.f;
  bool o_started = false;

  for (int t = 0; t < n_tiles && ok; ++t) {
    const int cur = t & 1, nxt = cur ^ 1;
    const int64_t t0 = t_lo + (int64_t)t * kTok;
    stage(t + 2, cur);                              // slot cur held tile t (already decoded)
    asm volatile("cp.async.wait_group 1;\n" ::);    // tile t+1 staged (own copies)
    __syncthreads();
    if (t + 1 < n_tiles)
      decode_tile_smem<D, kThrTcConst>(kbits, plk, lk, aPk(nxt) + a.slot.kc + s_off[nxt][0], aPk(nxt) + a.slot.ks + s_off[nxt][1],
                          n_valid_of(t + 1), aK(nxt));
    if (t >= 1) ok = ok && bar_wait(su32(&bar_o), (t - 1) & 1);          // O(t-1) done: P and V(nxt) free
    if (t + 1 < n_tiles)
      decode_tile_smem<D, kThrTcConst>(vbits, plv, lv, aPk(nxt) + a.slot.vc + s_off[nxt][2], aPk(nxt) + a.slot.vs + s_off[nxt][3],
                          n_valid_of(t + 1), aV(nxt));
    if (row_warp) {
      ok = ok && bar_wait(su32(&bar_s), t & 1);                          // S(t) ready
      fence_after();
      // ---- softmax on this thread's row of S
      uint32_t sv[32], sw[32];
      TQ_LD32(lane_base + kColS, sv);
      TQ_LD32(lane_base + kColS + 32, sw);
      asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory");
      // columns [0, nv_row) of this tile are valid for this row (context end,
      // causal limit); only tiles on a boundary need the mask
      const int64_t lim = a.causal ? imin64(t_hi, pos + 1) : t_hi;
      const int64_t room = lim - t0;
      const int nv_row = row_ok ? (room <= 0 ? 0 : (room >= kTok ? kTok : (int)room)) : 0;
      if (__any_sync(0xffffffffu, nv_row < kTok)) {
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          if (c >= nv_row) sv[c] = __float_as_uint(-INFINITY);
          if (c + 32 >= nv_row) sw[c] = __float_as_uint(-INFINITY);
        }
      }
      float mx = -INFINITY;
#pragma unroll
      for (int c = 0; c < 32; ++c) mx = fmaxf(mx, fmaxf(__uint_as_float(sv[c]), __uint_as_float(sw[c])));
      const bool need = mx > m_run + kLazyP;
      if (__any_sync(0xffffffffu, need)) {
        const float m_new = need ? mx : m_run;
        const float alpha = (need && m_run != -INFINITY) ? ex2f(m_run - m_new) : 1.f;
        m_run = m_new;
        l_run *= alpha;
        if (o_started) {   // rescale this row of O (alpha = 1 for rows that keep m)
#pragma unroll 1
          for (int c0 = 0; c0 < D; c0 += 32) {
            uint32_t ov[32];
            TQ_LD32(lane_base + kColO + c0, ov);
            asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory");
#pragma unroll
            for (int j = 0; j < 32; ++j) ov[j] = __float_as_uint(__uint_as_float(ov[j]) * alpha);
            TQ_ST32(lane_base + kColO + c0, ov);
          }
        }
      }
      const float mref = m_run == -INFINITY ? 0.f : m_run;
      uint32_t pw[32];
      float sum = 0.f;
#pragma unroll
      for (int c = 0; c < 32; ++c) {
        const float p0 = ex2f(__uint_as_float(c < 16 ? sv[2 * c] : sw[2 * c - 32]) - mref);
        const float p1 = ex2f(__uint_as_float(c < 16 ? sv[2 * c + 1] : sw[2 * c + 1 - 32]) - mref);
        sum += p0 + p1;
        const __half2 h = __floats2half2_rn(p0, p1);
        pw[c] = *reinterpret_cast<const uint32_t*>(&h);
      }
      l_run += sum;
      TQ_ST32(lane_base + kColP, pw);
      asm volatile("tcgen05.wait::st.sync.aligned;\n" ::: "memory");
    }
    asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");   // decoded tiles -> tensor core
    fence_before();
    ok = __syncthreads_and(ok) != 0;   // a timed-out wait stops the whole CTA together
    fence_after();
    if (ok && tid == 0) {
      issue_o(cur, !o_started);
      if (t + 1 < n_tiles) issue_s(nxt);
    }
    o_started = true;
  }
  if (n_tiles > 0 && ok) ok = bar_wait(su32(&bar_o), (n_tiles - 1) & 1);
  ok = __syncthreads_and(ok) != 0;
  // the combine kernel may be scheduled now; it waits for this grid to finish
  asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
  fence_after();
  asm volatile("cp.async.wait_group 0;\n" ::);
  // ---- partial (m, l, O) of this row for this context slice
  if (row_warp) {
    const int h = kvh * G + row % G;
    float* dst = a.part + ((((int64_t)b * a.Hq + h) * a.Tq + qi) * a.n_split + split) * (D + 4);
    if (ok && n_tiles > 0) {
      for (int c0 = 0; c0 < D; c0 += 32) {
        uint32_t ov[32];
        TQ_LD32(lane_base + kColO + c0, ov);
        asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory");
        if (row_ok) {
#pragma unroll
          for (int j = 0; j < 32; ++j) dst[2 + c0 + j] = __uint_as_float(ov[j]);
          if (c0 == 0) {
            dst[0] = m_run;
            dst[1] = l_run;
          }
        }
      }
    } else if (row_ok) {
      dst[0] = -INFINITY;
      dst[1] = 0.f;
      for (int j = 0; j < D; ++j) dst[2 + j] = 0.f;
    }
  }
  if (!ok && tid == 0) atomicExch(a.err, 1);
  fence_before();
  __syncthreads();
  if (warp == 0) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;\n" ::"r"(tmem), "r"(kTmemCols) : "memory");
  }
}

// Warp-specialised prefill: warps 0-3 (consumers) own the 128 TMEM rows, run
// the softmax and (one thread) issue the MMAs; the NP producer warps stage
// the packed bytes and decode K/V tiles into double buffers.  Handoffs go
// through mbarriers: kfull/vfull (a decoded tile is in buffer b; the
// producers arrive), kfree/vfree (the MMA that read buffer b is done; a
// tcgen05.commit arrives), s_done / o_done (S(t) written / O(t) done).  Every
// barrier is waited on at most one phase behind its last completion, so a
// parity wait is never confused by a later phase.  Waits are bounded: a wait
// that gives up raises a CTA-wide abort flag, after which the roles run out
// their loops (keeping the named-barrier counts) without further work.
template <int D, int NP>
__global__ void __launch_bounds__(128 + 32 * NP, 1) prefill_ws_kernel(const CodecParams PK, const CodecParams PV,
                                                                      const PrefillTcArgs a) {
  constexpr int kThr = 128 + 32 * NP;
  constexpr int kProd = 32 * NP;
  constexpr uint32_t kTmemCols = tmem_cols<D>();
  constexpr uint32_t kColQ = 128;
  constexpr uint32_t kColO = col_o<D>();
  constexpr uint32_t kTileBytes = kTok * D * 2;
  constexpr uint32_t kGroupBytes = (D / 8) * 128;
  extern __shared__ __align__(1024) uint8_t smem[];
  __shared__ __align__(8) uint64_t bars[10];   // kfull[2], vfull[2], kfree[2], vfree[2], s_done, o_done
  __shared__ uint32_t tmem_base;
  __shared__ int s_off[2][4];
  __shared__ volatile int s_abort;

  const int tid = threadIdx.x, warp = tid >> 5;
  const bool consumer = warp < 4;
  const int G = a.Hq / a.Hkv;
  const int rt = blockIdx.x, split = blockIdx.y, bh = blockIdx.z;
  const int b = bh / a.Hkv, kvh = bh % a.Hkv;
  const int R = a.Tq * G;
  const int row = rt * kRowsTc + (tid & 127);
  const bool row_ok = consumer && row < R;
  const int qi = row < R ? row / G : a.Tq - 1;
  const int64_t pos = a.ctx - a.Tq + qi;
  const int last_row = min(rt * kRowsTc + kRowsTc, R) - 1;
  const int64_t max_pos = a.causal ? a.ctx - a.Tq + last_row / G : a.ctx - 1;
  const int64_t t_lo = (int64_t)split * a.per;
  const int64_t t_hi = imin64(imin64(t_lo + a.per, a.ctx), max_pos + 1);
  const int n_tiles = t_hi > t_lo ? (int)((t_hi - t_lo + kTok - 1) / kTok) : 0;
  const int64_t rec0 = (int64_t)bh * a.S_cap;

  const uint32_t a_smem = su32(smem);
  auto aK = [&](int kb) { return a_smem + (uint32_t)kb * kTileBytes; };
  auto aV = [&](int kb) { return a_smem + (uint32_t)(2 + kb) * kTileBytes; };
  auto aPk = [&](int kb) { return a_smem + 4 * kTileBytes + (uint32_t)(kb * a.slot_bytes); };
  uint8_t* const pk_base = smem + 4 * kTileBytes;
  const uint32_t kfull = su32(&bars[0]), vfull = su32(&bars[2]), kfree = su32(&bars[4]), vfree = su32(&bars[6]);
  const uint32_t s_done = su32(&bars[8]), o_done = su32(&bars[9]);
  auto n_valid_of = [&](int tile) { return (int)imin64(kTok, t_hi - (t_lo + (int64_t)tile * kTok)); };
  auto wait = [&](uint32_t bar, uint32_t parity) {
    if (s_abort) return false;
    if (bar_wait(bar, parity)) return true;
    s_abort = 1;
    return false;
  };

  if (tid == 0) {
    s_abort = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(su32(&bars[i])), "r"(kProd) : "memory");
      asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;\n" ::"r"(su32(&bars[4 + i])) : "memory");
    }
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;\n" ::"r"(s_done) : "memory");
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;\n" ::"r"(o_done) : "memory");
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;\n" ::"r"(su32(&tmem_base)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n" ::: "memory");
  }
  fence_before();
  __syncthreads();
  fence_after();
  const uint32_t tmem = tmem_base;

  if (!consumer) {
    // ================= producers: stage and decode
    const int ptid = tid - 128;
    const CodeTabs lk = make_code_tabs(PK), lv = make_code_tabs(PV);
    const ItemPlan<D, kProd> plk = make_plan<D, kProd>(PK, ptid), plv = make_plan<D, kProd>(PV, ptid);
    auto stage = [&](int tile) {
      const int slot = tile & 1;
      if (tile < n_tiles) {
        const int64_t t0 = t_lo + (int64_t)tile * kTok;
        const int n = (int)imin64(kTok, t_hi - t0);
        uint8_t* base = pk_base + slot * a.slot_bytes;
        const int o0 = stage_bytes(base + a.slot.kc, a.kc, rec0 + t0, n, PK.code_bytes, ptid, kProd);
        const int o1 = stage_bytes(base + a.slot.ks, a.ks, rec0 + t0, n, 2 * PK.nb, ptid, kProd);
        const int o2 = stage_bytes(base + a.slot.vc, a.vc, rec0 + t0, n, PV.code_bytes, ptid, kProd);
        const int o3 = stage_bytes(base + a.slot.vs, a.vs, rec0 + t0, n, 2 * PV.nb, ptid, kProd);
        if (ptid == 0) {
          s_off[slot][0] = o0; s_off[slot][1] = o1; s_off[slot][2] = o2; s_off[slot][3] = o3;
        }
      }
      asm volatile("cp.async.commit_group;\n" ::);
    };
    stage(0);
    stage(1);
    for (int t = 0; t < n_tiles; ++t) {
      const int kb = t & 1;
      const uint32_t use = (uint32_t)(t >> 1);   // use number of buffer kb
      asm volatile("cp.async.wait_group 1;\n" ::);
      asm volatile("bar.sync 1, %0;\n" ::"n"(kProd) : "memory");   // tile t staged (all producers' copies)
      const int nv = n_valid_of(t);
      if (t >= 2) wait(kfree + 8 * kb, (use - 1) & 1);   // S(t-2) has read K buffer kb
      if (!s_abort)
        decode_tile_smem<D, kProd>(PK.bits, plk, lk, aPk(kb) + a.slot.kc + s_off[kb][0],
                                   aPk(kb) + a.slot.ks + s_off[kb][1], nv, aK(kb));
      asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
      asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(kfull + 8 * kb) : "memory");
      if (t >= 2) wait(vfree + 8 * kb, (use - 1) & 1);   // O(t-2) has read V buffer kb
      if (!s_abort)
        decode_tile_smem<D, kProd>(PV.bits, plv, lv, aPk(kb) + a.slot.vc + s_off[kb][2],
                                   aPk(kb) + a.slot.vs + s_off[kb][3], nv, aV(kb));
      asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
      asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(vfull + 8 * kb) : "memory");
      asm volatile("bar.sync 1, %0;\n" ::"n"(kProd) : "memory");   // every producer is done with slot kb
      stage(t + 2);
    }
    asm volatile("cp.async.wait_group 0;\n" ::);
  } else {
    // ================= consumers: softmax rows, one thread issues the MMAs
    const uint32_t lane_base = tmem + ((uint32_t)(32 * warp) << 16);
    {
      const __half* src = a.qhat + ((int64_t)bh * a.R_pad + (int64_t)rt * kRowsTc + tid) * D;
#pragma unroll 1
      for (int c0 = 0; c0 < D / 2; c0 += 32) {
        uint32_t w[32];
#pragma unroll
        for (int j = 0; j < 32; j += 4) {
          const uint4 v = *reinterpret_cast<const uint4*>(src + 2 * (c0 + j));
          w[j] = v.x; w[j + 1] = v.y; w[j + 2] = v.z; w[j + 3] = v.w;
        }
        TQ_ST32(lane_base + kColQ + c0, w);
      }
      asm volatile("tcgen05.wait::st.sync.aligned;\n" ::: "memory");
    }
    fence_before();
    asm volatile("bar.sync 2, 128;\n" ::: "memory");
    fence_after();
    const uint32_t idesc_s = (1u << 4) | ((uint32_t)(kTok >> 3) << 17) | ((uint32_t)(kRowsTc >> 4) << 24);
    const uint32_t idesc_o = (1u << 4) | (1u << 16) | ((uint32_t)(D >> 3) << 17) | ((uint32_t)(kRowsTc >> 4) << 24);
    auto issue_s = [&](int t) {   // S = Q^ (TMEM) K^(buffer)^T, once K(t) is decoded
      const int kb = t & 1;
      if (!wait(kfull + 8 * kb, (uint32_t)(t >> 1) & 1)) return;
      fence_after();
#pragma unroll 4
      for (int s = 0; s < D / 16; ++s)
        mma_ts(tmem + kColS, tmem + kColQ + 8 * s, sdesc(aK(kb) + s * 256, 128, kGroupBytes), idesc_s, s > 0);
      mma_commit(s_done);
      mma_commit(kfree + 8 * kb);
    };
    auto issue_o = [&](int t) {   // O += P (TMEM) V^(buffer), once V(t) is decoded
      const int kb = t & 1;
      if (!wait(vfull + 8 * kb, (uint32_t)(t >> 1) & 1)) return;
      fence_after();
#pragma unroll
      for (int s = 0; s < kTok / 16; ++s)
        mma_ts(tmem + kColO, tmem + kColP + 8 * s, sdesc(aV(kb) + s * 2 * kGroupBytes, kGroupBytes, 128), idesc_o,
               (t == 0 && s == 0) ? 0 : 1);
      mma_commit(o_done);
      mma_commit(vfree + 8 * kb);
    };
    if (tid == 0 && n_tiles > 0) issue_s(0);
    float m_run = -INFINITY, l_run = 0.f;
    for (int t = 0; t < n_tiles; ++t) {
      const int64_t t0 = t_lo + (int64_t)t * kTok;
      uint32_t sv[32], sw[32];
      const bool have_s = wait(s_done, (uint32_t)t & 1);   // S(t) written
      fence_after();
      if (have_s) {
        TQ_LD32(lane_base + kColS, sv);
        TQ_LD32(lane_base + kColS + 32, sw);
        asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory");
      } else {
#pragma unroll
        for (int c = 0; c < 32; ++c) sv[c] = sw[c] = __float_as_uint(-INFINITY);
      }
      const int64_t lim = a.causal ? imin64(t_hi, pos + 1) : t_hi;
      const int64_t room = lim - t0;
      const int nv_row = row_ok ? (room <= 0 ? 0 : (room >= kTok ? kTok : (int)room)) : 0;
      if (__any_sync(0xffffffffu, nv_row < kTok)) {
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          if (c >= nv_row) sv[c] = __float_as_uint(-INFINITY);
          if (c + 32 >= nv_row) sw[c] = __float_as_uint(-INFINITY);
        }
      }
      float mx = -INFINITY;
#pragma unroll
      for (int c = 0; c < 32; ++c) mx = fmaxf(mx, fmaxf(__uint_as_float(sv[c]), __uint_as_float(sw[c])));
      // O(t-1) must be done before P is rewritten or O rescaled
      if (t >= 1) wait(o_done, (uint32_t)(t - 1) & 1);
      fence_after();
      const bool need = mx > m_run + kLazyP;
      if (__any_sync(0xffffffffu, need)) {
        const float m_new = need ? mx : m_run;
        const float alpha = (need && m_run != -INFINITY) ? ex2f(m_run - m_new) : 1.f;
        m_run = m_new;
        l_run *= alpha;
        if (t >= 1) {
#pragma unroll 1
          for (int c0 = 0; c0 < D; c0 += 32) {
            uint32_t ov[32];
            TQ_LD32(lane_base + kColO + c0, ov);
            asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory");
#pragma unroll
            for (int j = 0; j < 32; ++j) ov[j] = __float_as_uint(__uint_as_float(ov[j]) * alpha);
            TQ_ST32(lane_base + kColO + c0, ov);
          }
        }
      }
      const float mref = m_run == -INFINITY ? 0.f : m_run;
      uint32_t pw[32];
      float sum = 0.f;
#pragma unroll
      for (int c = 0; c < 32; ++c) {
        const float p0 = ex2f(__uint_as_float(c < 16 ? sv[2 * c] : sw[2 * c - 32]) - mref);
        const float p1 = ex2f(__uint_as_float(c < 16 ? sv[2 * c + 1] : sw[2 * c + 1 - 32]) - mref);
        sum += p0 + p1;
        const __half2 h = __floats2half2_rn(p0, p1);
        pw[c] = *reinterpret_cast<const uint32_t*>(&h);
      }
      l_run += sum;
      TQ_ST32(lane_base + kColP, pw);
      asm volatile("tcgen05.wait::st.sync.aligned;\n" ::: "memory");
      fence_before();
      asm volatile("bar.sync 2, 128;\n" ::: "memory");   // P(t) complete, S(t) read by every row
      fence_after();
      if (tid == 0 && !s_abort) {
        issue_o(t);
        if (t + 1 < n_tiles) issue_s(t + 1);
      }
    }
    if (n_tiles > 0) wait(o_done, (uint32_t)(n_tiles - 1) & 1);
    fence_after();
    const bool ok = !s_abort;
    const int h = kvh * G + row % G;
    float* dst = a.part + ((((int64_t)b * a.Hq + h) * a.Tq + qi) * a.n_split + split) * (D + 4);
    if (ok && n_tiles > 0) {
      for (int c0 = 0; c0 < D; c0 += 32) {
        uint32_t ov[32];
        TQ_LD32(lane_base + kColO + c0, ov);
        asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory");
        if (row_ok) {
#pragma unroll
          for (int j = 0; j < 32; ++j) dst[2 + c0 + j] = __uint_as_float(ov[j]);
          if (c0 == 0) {
            dst[0] = m_run;
            dst[1] = l_run;
          }
        }
      }
    } else if (row_ok) {
      dst[0] = -INFINITY;
      dst[1] = 0.f;
      for (int j = 0; j < D; ++j) dst[2 + j] = 0.f;
    }
  }
  // the combine kernel may be scheduled now; it waits for this grid to finish
  asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
  fence_before();
  __syncthreads();
  if (tid == 0 && s_abort) atomicExch(a.err, 1);
  if (warp == 0) {
    fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;\n" ::"r"(tmem), "r"(kTmemCols) : "memory");
  }
}

// Q^ = (H D q per K block) * softmax_scale * log2 e, fp16, rows i*G + h of
// each (batch, KV head), zero padded to R_pad rows.
template <int D>
__global__ void __launch_bounds__(D) prefill_rotate_q_kernel(const CodecParams PK, const uint16_t* __restrict__ q,
                                                              __half* __restrict__ qhat, int Hq, int Hkv, int Tq,
                                                              int R_pad, float qscale) {
  __shared__ float s[D];
  const int r = blockIdx.x;        // padded row
  const int bh = blockIdx.y;
  const int b = bh / Hkv, kvh = bh % Hkv;
  const int G = Hq / Hkv;
  const int i = threadIdx.x;
  const bool ok = r < Tq * G;
  float v = 0.f;
  if (ok) {
    const int qi = r / G, h = kvh * G + r % G;
    v = h2f(q[(((int64_t)b * Hq + h) * Tq + qi) * D + i]);
    v = flip(v, (PK.sign_bits[i >> 5] >> (i & 31)) & 1u);
  }
  s[i] = v;
  for (int hs = 1; hs < PK.blk; hs <<= 1) {
    __syncthreads();
    const float x = s[i], y = s[i ^ hs];
    __syncthreads();
    s[i] = (i & hs) ? (y - x) : (x + y);
  }
  __syncthreads();
  qhat[((int64_t)bh * R_pad + r) * D + i] = __float2half_rn(s[i] * PK.inv_sqrt_blk * qscale);
}

template <int D>
size_t tc_smem(int slot_bytes) {  // double-buffered decoded K and V tiles + two packed staging slots
  return 4 * (size_t)kTok * D * 2 + 2 * (size_t)slot_bytes;
}

}  // namespace

int prefill_tc_splits(int B, int Hkv, int G, int Tq, int64_t ctx) {
  // One CTA per SM at a time: pick the context split that fills whole waves
  // best (at least 90% of the last wave busy), preferring fewer splits, each
  // split at least 4 tiles long.
  const int row_tiles = (Tq * G + kRowsTc - 1) / kRowsTc;
  const int64_t ctas = (int64_t)row_tiles * B * Hkv;
  const int sms = sm_count();
  const int64_t max_by_len = (ctx + 4 * kTok - 1) / (4 * kTok);
  int best = 1;
  double best_eff = 0.0;
  for (int ns = 1; ns <= 32 && ns <= max_by_len; ++ns) {
    const int64_t n = ctas * ns;
    const int64_t waves = (n + sms - 1) / sms;
    const double eff = (double)n / (double)(waves * sms);
    if (eff > best_eff + 1e-9 && (ns == 1 || eff >= 0.9 || eff > best_eff + 0.05)) {
      best = ns;
      best_eff = eff;
    }
    if (eff >= 0.97) break;
  }
  return best;
}

size_t prefill_tc_workspace(int B, int Hq, int Hkv, int d, int Tq, int64_t ctx) {
  const int G = Hq / Hkv;
  const int R_pad = (Tq * G + kRowsTc - 1) / kRowsTc * kRowsTc;
  const int ns = prefill_tc_splits(B, Hkv, G, Tq, ctx);
  const size_t qbytes = (size_t)B * Hkv * R_pad * d * 2;
  const size_t pbytes = (size_t)B * Hq * Tq * ns * (d + 4) * 4;
  return 256 + ((qbytes + 255) / 256) * 256 + pbytes;
}

int launch_prefill_tc(const CodecParams& PK, const CodecParams& PV, const uint8_t* kc, const uint16_t* ks,
                      const uint8_t* vc, const uint16_t* vs, const uint16_t* q, int B, int Hq, int Hkv, int Tq,
                      int64_t S_cap, int64_t ctx, int causal, float qscale, uint16_t* out, void* ws,
                      cudaStream_t st) {
  const int d = PK.d;
  const int G = Hq / Hkv;
  const int R_pad = (Tq * G + kRowsTc - 1) / kRowsTc * kRowsTc;
  const int ns = prefill_tc_splits(B, Hkv, G, Tq, ctx);
  uint8_t* base = static_cast<uint8_t*>(ws);
  int* err = reinterpret_cast<int*>(base);
  const size_t qbytes = (size_t)B * Hkv * R_pad * d * 2;
  __half* qhat = reinterpret_cast<__half*>(base + 256);
  float* part = reinterpret_cast<float*>(base + 256 + ((qbytes + 255) / 256) * 256);
  if (cudaMemsetAsync(err, 0, sizeof(int), st) != cudaSuccess) return TQ_ERR_CUDA;
  int64_t per = (ctx + ns - 1) / ns;
  per = (per + kTok - 1) / kTok * kTok;
  // staging slot: each array padded to 16 bytes plus 16 bytes of alignment slack
  auto pad = [](int bytes) { return (bytes + 16 + 15) / 16 * 16; };
  PackedSlot slot;
  slot.kc = 0;
  slot.ks = slot.kc + pad(kTok * PK.code_bytes);
  slot.vc = slot.ks + pad(kTok * 2 * PK.nb);
  slot.vs = slot.vc + pad(kTok * PV.code_bytes);
  const int slot_bytes = slot.vs + pad(kTok * 2 * PV.nb);
  PrefillTcArgs a{kc, reinterpret_cast<const uint8_t*>(ks), vc, reinterpret_cast<const uint8_t*>(vs), qhat, part,
                  err, S_cap, ctx, Hq, Hkv, Tq, R_pad, ns, causal, per, slot_bytes, slot};
  dim3 qgrid(R_pad, B * Hkv);
  dim3 grid(R_pad / kRowsTc, ns, B * Hkv);
  switch (d) {
    case 64: {
      prefill_rotate_q_kernel<64><<<qgrid, 64, 0, st>>>(PK, q, qhat, Hq, Hkv, Tq, R_pad, qscale);
      const size_t sm = tc_smem<64>(slot_bytes);
      if (cudaFuncSetAttribute(prefill_ws_kernel<64, kProducerWarps>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)sm))
        return TQ_ERR_CUDA;
      prefill_ws_kernel<64, kProducerWarps><<<grid, 128 + 32 * kProducerWarps, sm, st>>>(PK, PV, a);
      break;
    }
    case 128: {
      prefill_rotate_q_kernel<128><<<qgrid, 128, 0, st>>>(PK, q, qhat, Hq, Hkv, Tq, R_pad, qscale);
      const size_t sm = tc_smem<128>(slot_bytes);
      if (cudaFuncSetAttribute(prefill_ws_kernel<128, kProducerWarps>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)sm))
        return TQ_ERR_CUDA;
      prefill_ws_kernel<128, kProducerWarps><<<grid, 128 + 32 * kProducerWarps, sm, st>>>(PK, PV, a);
      break;
    }
    default: {
      prefill_rotate_q_kernel<256><<<qgrid, 256, 0, st>>>(PK, q, qhat, Hq, Hkv, Tq, R_pad, qscale);
      const size_t sm = tc_smem<256>(slot_bytes);
      if (cudaFuncSetAttribute(prefill_ws_kernel<256, kProducerWarps>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)sm))
        return TQ_ERR_CUDA;
      prefill_ws_kernel<256, kProducerWarps><<<grid, 128 + 32 * kProducerWarps, sm, st>>>(PK, PV, a);
      break;
    }
  }
  if (cudaGetLastError() != cudaSuccess) return TQ_ERR_CUDA;
  return decode_combine(PV, part, ns, out, B * Hq * Tq, st);
}

}  // namespace tq
