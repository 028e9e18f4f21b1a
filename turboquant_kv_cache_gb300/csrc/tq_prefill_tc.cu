// Prefill attention over the packed cache on the 5th-generation tensor cores
// (tcgen05, TMEM accumulators).
//
// Rows: every (batch, KV head) owns R = Tq*G query rows (query i, head h ->
// row i*G + h).  A CTA takes 128 rows (one per consumer thread and per TMEM
// lane) and one slice of the context, walking it in 64-token tiles, with two
// warp roles:
//   * producer warps stage the packed K/V bytes with cp.async and decode each
//     tile into shared memory (rotated domain, centroid * block norm, fp16)
//     in the canonical no-swizzle core-matrix layout (8 rows x 16 bytes per
//     core matrix), which serves K as a K-major B operand of S = Q K^T and V
//     as an MN-major B operand of O = P V; K and V tiles are double-buffered,
//     so decoding runs ahead of the MMAs;
//   * consumer warps: one thread issues S = Q^ K^^T (M 128, N 64, K d) into
//     TMEM and O += P V^ (A = P from TMEM, M 128, N d, K 64); each consumer
//     thread reads its row of S, applies the causal / context mask and an
//     online softmax in base 2 (the reference max moves only when a score
//     exceeds it by more than 2^8) and writes P as fp16 back into TMEM.
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
constexpr int kTok = 64;         // tokens per KV tile
constexpr int kProducerWarps = 8;   // decoding warps without register rebalancing
constexpr int kProducerWarpsRB = 16; // decoding warps with setmaxnreg rebalancing
constexpr int kConsRegs = 128, kDecRegs = 88;
constexpr uint32_t kColS = 0, kColP = 64;
// TMEM columns: S (64 fp32) at 0, two P buffers (64 fp16 = 32 columns each) at
// 64 and 96, Q^ (D fp16 = D/2 columns) at 128, O (D fp32) after it; a power
// of two >= the total (exactly 512 at head_dim 256)
template <int D> __host__ __device__ constexpr uint32_t col_o() { return 128u + D / 2; }
template <int D> __host__ __device__ constexpr uint32_t tmem_cols() { return col_o<D>() + D <= 256u ? 256u : 512u; }
constexpr float kLazyP = 8.0f;
constexpr uint32_t kSuspendNs = 1000000;        // try_wait sleep hint
constexpr uint64_t kWaitNs = 2000000000ull;     // give up a wait after 2 s

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

__device__ __forceinline__ void mma_ts(uint32_t d, uint32_t a, uint64_t b, uint32_t idesc, int acc) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(d),
      "r"(a), "l"(b), "r"(idesc), "r"(acc)
      : "memory");
}

__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n" ::"r"(bar) : "memory");
}

__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Wait for the phase of parity `phase` of an mbarrier.  The thread sleeps in
// try_wait (suspend-time hint 1 ms; it wakes as soon as the phase completes)
// instead of spinning; the whole wait is bounded by kWaitNs of wall time.
__device__ __forceinline__ bool bar_wait(uint32_t bar, uint32_t phase) {
  uint32_t done = 0;
  uint64_t t0 = 0;
  for (int it = 0; !done; ++it) {
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(done)
        : "r"(bar), "r"(phase), "r"(kSuspendNs)
        : "memory");
    if (done) break;
    if (it == 0) {
      t0 = global_ns();
    } else if (global_ns() - t0 > kWaitNs) {
      return false;
    }
  }
  return true;
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


__device__ __forceinline__ float ex2f(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// fp16 centroid byte tables: lo/hi bytes of entries 0-3 / 4-7 (t[0..3]) and,
// for 4-bit codebooks, of entries 8-11 / 12-15 (t[4..7]).
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
template <int D, int NT>
struct ItemPlan {
  static constexpr int G8 = D / 32;
  static constexpr int N = (kTok * G8 + NT - 1) / NT;   // items per decoding thread
  int tok[N];
  uint32_t code_off[N], sc_off[N], dst_off[N];
};

template <int D, int NT>
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

// Packed words and fp16 norm of a thread's items of one tile, loaded from
// global memory (read-only path) a tile ahead of their decode.
template <int D, int NT>
struct ItemRegs {
  uint32_t w[ItemPlan<D, NT>::N][4];
  uint32_t sc[ItemPlan<D, NT>::N];
};

__device__ __forceinline__ uint32_t ldg32(const uint8_t* p) {
  uint32_t v;
  asm volatile("ld.global.nc.b32 %0, [%1];" : "=r"(v) : "l"(p));
  return v;
}
__device__ __forceinline__ uint32_t ldg16(const uint8_t* p) {
  unsigned short v;
  asm volatile("ld.global.nc.u16 %0, [%1];" : "=h"(v) : "l"(p));
  return v;
}

template <int D, int NT, int BITS>
__device__ __forceinline__ void load_items_b(const ItemPlan<D, NT>& pl, const uint8_t* codes, const uint8_t* scales,
                                             int n_valid, ItemRegs<D, NT>& r) {
#pragma unroll
  for (int k = 0; k < ItemPlan<D, NT>::N; ++k) {
    if (pl.tok[k] < n_valid) {
      const uint8_t* c = codes + pl.code_off[k];
      if (BITS == 4) {
        uint4 v;
        asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
                     : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                     : "l"(c));
        r.w[k][0] = v.x; r.w[k][1] = v.y; r.w[k][2] = v.z; r.w[k][3] = v.w;
      } else if (BITS == 2) {
        uint2 v;
        asm volatile("ld.global.nc.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(c));
        r.w[k][0] = v.x; r.w[k][1] = v.y;
      } else {
#pragma unroll
        for (int b = 0; b < BITS; ++b) r.w[k][b] = ldg32(c + 4 * b);
      }
      r.sc[k] = ldg16(scales + pl.sc_off[k]);
    }
  }
}

template <int D, int NT>
__device__ __forceinline__ void load_items(int bits, const ItemPlan<D, NT>& pl, const uint8_t* codes,
                                           const uint8_t* scales, int n_valid, ItemRegs<D, NT>& r) {
  switch (bits) {
    case 4: load_items_b<D, NT, 4>(pl, codes, scales, n_valid, r); break;
    case 3: load_items_b<D, NT, 3>(pl, codes, scales, n_valid, r); break;
    case 2: load_items_b<D, NT, 2>(pl, codes, scales, n_valid, r); break;
    default: load_items_b<D, NT, 1>(pl, codes, scales, n_valid, r); break;
  }
}

// Decode a thread's items of one tile from registers into the core-matrix
// tile at shared address `tile` (same rules as decode_tile_items).
template <int D, int NT, int BITS>
__device__ __forceinline__ void decode_regs_b(const ItemPlan<D, NT>& pl, const ItemRegs<D, NT>& r, const uint32_t* c2,
                                              const Tab& fixed, int n_valid, uint32_t tile) {
#pragma unroll
  for (int k = 0; k < ItemPlan<D, NT>::N; ++k) {
    if (pl.tok[k] >= kTok) continue;
    const uint32_t dst = tile + pl.dst_off[k];
    if (n_valid == kTok || pl.tok[k] < n_valid) {
      uint32_t n[4];
      chunk_words<BITS>(r.w[k], n);
      const uint32_t sc = r.sc[k];
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
__device__ __forceinline__ void decode_regs(int bits, const ItemPlan<D, NT>& pl, const ItemRegs<D, NT>& r,
                                            const CodeTabs& ct, int n_valid, uint32_t tile) {
  switch (bits) {
    case 4: decode_regs_b<D, NT, 4>(pl, r, ct.c2, ct.fixed, n_valid, tile); break;
    case 3: decode_regs_b<D, NT, 3>(pl, r, ct.c2, ct.fixed, n_valid, tile); break;
    case 2: decode_regs_b<D, NT, 2>(pl, r, ct.c2, ct.fixed, n_valid, tile); break;
    default: decode_regs_b<D, NT, 1>(pl, r, ct.c2, ct.fixed, n_valid, tile); break;
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
};


// Warp-specialised prefill: warps 0-3 (consumers) own the 128 TMEM rows, run
// the softmax and (one thread) issue the MMAs; the NP producer warps stage
// the packed bytes and decode K/V tiles into double buffers.  Handoffs go
// through mbarriers: kfull/vfull (a decoded tile is in buffer b; the
// producers arrive), kfree/vfree (the MMA that read buffer b is done; a
// tcgen05.commit arrives), s_done (S(t) written) and pfree (the O product that
// read P buffer b is done; P is double-buffered in TMEM).  Every
// barrier is waited on at most one phase behind its last completion, so a
// parity wait is never confused by a later phase.  Waits are bounded: a wait
// that gives up raises a CTA-wide abort flag, after which the roles run out
// their loops (keeping the named-barrier counts) without further work.
template <int D, int NP, int NB, bool RB>
__global__ void __launch_bounds__(128 + 32 * NP, 1) prefill_ws_kernel(const CodecParams PK, const CodecParams PV,
                                                                      const PrefillTcArgs a) {
  constexpr int kProd = 32 * NP;
  constexpr int kHalf = kProd / 2;   // decoders per side (K or V)
  constexpr uint32_t kTmemCols = tmem_cols<D>();
  constexpr uint32_t kColQ = 128;
  constexpr uint32_t kColO = col_o<D>();
  constexpr uint32_t kTileBytes = kTok * D * 2;
  constexpr uint32_t kGroupBytes = (D / 8) * 128;
  extern __shared__ __align__(1024) uint8_t smem[];
  // kfull[NB], vfull[NB], kfree[NB], vfree[NB], s_done, pfree[2]
  __shared__ __align__(8) uint64_t bars[4 * NB + 3];
  __shared__ uint32_t tmem_base;
  __shared__ volatile int s_abort;
  __shared__ CodeTabs s_tabs[2];   // K and V codebooks (fp16 pairs, unscaled 4-bit tables)

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
  // NB decoded K buffers, then NB decoded V buffers
  auto aK = [&](int kb) { return a_smem + (uint32_t)kb * kTileBytes; };
  auto aV = [&](int kb) { return a_smem + (uint32_t)(NB + kb) * kTileBytes; };
  const uint32_t kfull = su32(&bars[0]), vfull = su32(&bars[NB]), kfree = su32(&bars[2 * NB]),
                 vfree = su32(&bars[3 * NB]);
  const uint32_t s_done = su32(&bars[4 * NB]), pfree = su32(&bars[4 * NB + 1]);  // pfree[b]: O that read P buffer b is done
  auto n_valid_of = [&](int tile) { return (int)imin64(kTok, t_hi - (t_lo + (int64_t)tile * kTok)); };
  auto wait = [&](uint32_t bar, uint32_t parity) {
    if (s_abort) return false;
    if (bar_wait(bar, parity)) return true;
    s_abort = 1;
    return false;
  };

  if (tid == 0) {
    s_tabs[0] = make_code_tabs(PK);
    s_tabs[1] = make_code_tabs(PV);
  }
  if (tid == 0) {
    s_abort = 0;
#pragma unroll
    for (int i = 0; i < 2 * NB; ++i)   // kfull, vfull: every decoder of that side arrives
      asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(su32(&bars[i])), "r"(kHalf) : "memory");
#pragma unroll
    for (int i = 2 * NB; i < 4 * NB + 3; ++i)   // one arrival: a tcgen05.commit
      asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;\n" ::"r"(su32(&bars[i])) : "memory");
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
    // ================= decoders: half the decoder warps fill the NB K buffers,
    // the other half the NB V buffers, each at its own pace (K waits only for
    // the S products, V only for the O products).  Each thread loads its
    // items' packed words for tile t+1 into registers before decoding tile t,
    // so the global latency hides behind the decode.
    if (RB) asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;\n" ::"n"(kDecRegs));
    const bool kside = warp < 4 + NP / 2;
    const int ptid = tid - (kside ? 128 : 128 + kHalf);
    const CodecParams& P = kside ? PK : PV;
    const CodeTabs& ct = s_tabs[kside ? 0 : 1];
    const uint8_t* codes = kside ? a.kc : a.vc;
    const uint8_t* scales = kside ? a.ks : a.vs;
    const uint32_t full = kside ? kfull : vfull, free_bar = kside ? kfree : vfree;
    const ItemPlan<D, kHalf> pl = make_plan<D, kHalf>(P, ptid);
    ItemRegs<D, kHalf> ra, rn;
    auto load = [&](int t, ItemRegs<D, kHalf>& r) {
      const int64_t rec = rec0 + t_lo + (int64_t)t * kTok;
      load_items<D, kHalf>(P.bits, pl, codes + rec * P.code_bytes, scales + rec * 2 * P.nb, n_valid_of(t), r);
    };
    auto step = [&](int t, const ItemRegs<D, kHalf>& r, ItemRegs<D, kHalf>& next) {
      if (t + 1 < n_tiles) load(t + 1, next);
      const int kb = t % NB;
      if (t >= NB) wait(free_bar + 8 * kb, (uint32_t)(t / NB - 1) & 1);   // the product NB tiles back is done
      if (!s_abort) decode_regs<D, kHalf>(P.bits, pl, r, ct, n_valid_of(t), kside ? aK(kb) : aV(kb));
      asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
      asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(full + 8 * kb) : "memory");
    };
    if (n_tiles > 0) load(0, ra);
    for (int t = 0; t < n_tiles; t += 2) {
      step(t, ra, rn);
      if (t + 1 < n_tiles) step(t + 1, rn, ra);
    }
  } else {
    // ================= consumers: softmax rows, one thread issues the MMAs
    if (RB) asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;\n" ::"n"(kConsRegs));
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
      const int kb = t % NB;
      if (!wait(kfull + 8 * kb, (uint32_t)(t / NB) & 1)) return;
      fence_after();
#pragma unroll 4
      for (int s = 0; s < D / 16; ++s)
        mma_ts(tmem + kColS, tmem + kColQ + 8 * s, sdesc(aK(kb) + s * 256, 128, kGroupBytes), idesc_s, s > 0);
      mma_commit(s_done);
      mma_commit(kfree + 8 * kb);
    };
    auto issue_o = [&](int t) {   // O += P (TMEM) V^(buffer), once V(t) is decoded
      const int kb = t % NB, pb = t & 1;
      if (!wait(vfull + 8 * kb, (uint32_t)(t / NB) & 1)) return;
      fence_after();
#pragma unroll
      for (int s = 0; s < kTok / 16; ++s)
        mma_ts(tmem + kColO, tmem + kColP + 32 * pb + 8 * s, sdesc(aV(kb) + s * 2 * kGroupBytes, kGroupBytes, 128),
               idesc_o, (t == 0 && s == 0) ? 0 : 1);
      mma_commit(pfree + 8 * pb);
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
      // every row has S(t) in registers: S(t+1) can overwrite it and run on
      // the tensor pipe while this softmax proceeds
      fence_before();
      asm volatile("bar.sync 2, 128;\n" ::: "memory");
      fence_after();
      if (tid == 0 && !s_abort && t + 1 < n_tiles) issue_s(t + 1);
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
        if (t >= 1) {
          // O(t-1), the last product issued on O, must be done before O is rescaled
          wait(pfree + 8 * ((t - 1) & 1), (uint32_t)((t - 1) >> 1) & 1);
          fence_after();
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
      // P buffer t&1 was last read by O(t-2)
      if (t >= 2) wait(pfree + 8 * (t & 1), (uint32_t)((t - 2) >> 1) & 1);
      fence_after();
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
      TQ_ST32(lane_base + kColP + 32 * (t & 1), pw);
      asm volatile("tcgen05.wait::st.sync.aligned;\n" ::: "memory");
      fence_before();
      asm volatile("bar.sync 2, 128;\n" ::: "memory");   // P(t) complete
      fence_after();
      if (tid == 0 && !s_abort) issue_o(t);
    }
    if (n_tiles > 0) wait(pfree + 8 * ((n_tiles - 1) & 1), (uint32_t)((n_tiles - 1) >> 1) & 1);
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
size_t tc_smem(int nb) {  // nb decoded K tiles and nb decoded V tiles
  return (size_t)2 * nb * kTok * D * 2;
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

// The warp-specialised kernel with 16 decoder warps and setmaxnreg moving
// registers to the consumers, when its launch register count makes that
// split exact (launch total >= consumer + decoder shares); otherwise 8
// decoder warps without rebalancing.
template <int D>
int launch_ws(const CodecParams& PK, const CodecParams& PV, const PrefillTcArgs& a, dim3 grid, cudaStream_t st) {
  const size_t sm = tc_smem<D>(3);
  static int use_rb = -1;   // decided once per process (the kernel image is fixed)
  if (use_rb < 0) {
    cudaFuncAttributes fa;
    use_rb = 0;
    if (cudaFuncGetAttributes(&fa, prefill_ws_kernel<D, kProducerWarpsRB, 3, true>) == cudaSuccess) {
      const long launch = (long)(128 + 32 * kProducerWarpsRB) * fa.numRegs;
      const long need = 128L * kConsRegs + 32L * kProducerWarpsRB * kDecRegs;
      use_rb = (fa.numRegs >= kDecRegs && fa.numRegs <= kConsRegs && launch >= need) ? 1 : 0;
    }
  }
  if (use_rb) {
    auto k = prefill_ws_kernel<D, kProducerWarpsRB, 3, true>;
    if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm)) return TQ_ERR_CUDA;
    k<<<grid, 128 + 32 * kProducerWarpsRB, sm, st>>>(PK, PV, a);
  } else {
    auto k = prefill_ws_kernel<D, kProducerWarps, 3, false>;
    if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm)) return TQ_ERR_CUDA;
    k<<<grid, 128 + 32 * kProducerWarps, sm, st>>>(PK, PV, a);
  }
  return cudaGetLastError() == cudaSuccess ? TQ_OK : TQ_ERR_CUDA;
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
  PrefillTcArgs a{kc, reinterpret_cast<const uint8_t*>(ks), vc, reinterpret_cast<const uint8_t*>(vs), qhat, part,
                  err, S_cap, ctx, Hq, Hkv, Tq, R_pad, ns, causal, per};
  dim3 qgrid(R_pad, B * Hkv);
  dim3 grid(R_pad / kRowsTc, ns, B * Hkv);
  int r;
  switch (d) {
    case 64:
      prefill_rotate_q_kernel<64><<<qgrid, 64, 0, st>>>(PK, q, qhat, Hq, Hkv, Tq, R_pad, qscale);
      r = launch_ws<64>(PK, PV, a, grid, st);
      break;
    case 128:
      prefill_rotate_q_kernel<128><<<qgrid, 128, 0, st>>>(PK, q, qhat, Hq, Hkv, Tq, R_pad, qscale);
      r = launch_ws<128>(PK, PV, a, grid, st);
      break;
    default:
      prefill_rotate_q_kernel<256><<<qgrid, 256, 0, st>>>(PK, q, qhat, Hq, Hkv, Tq, R_pad, qscale);
      r = launch_ws<256>(PK, PV, a, grid, st);
      break;
  }
  if (r != TQ_OK) return r;
  if (cudaGetLastError() != cudaSuccess) return TQ_ERR_CUDA;
  return decode_combine(PV, part, ns, out, B * Hq * Tq, st);
}

}  // namespace tq
