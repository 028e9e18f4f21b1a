// Prefill attention over the packed cache on the 5th-generation tensor cores
// (tcgen05, TMEM accumulators).
//
// Rows: every (batch, KV head) owns R = Tq*G query rows (query i, head h ->
// row i*G + h).  A CTA takes 128 rows (one per softmax thread and per TMEM
// lane) and one slice of the context, walking it in 64-token tiles, with
// three warp roles:
//   * decoder warps (one group for K, one for V) load the packed codes and
//     block norms of the next tile into registers and decode the current one
//     into shared memory (rotated domain, centroid * block norm, fp16) in the
//     canonical no-swizzle core-matrix layout (8 rows x 16 bytes per core
//     matrix), which serves K as a K-major B operand of S = Q K^T and V as an
//     MN-major B operand of O = P V; each side has a ring of three buffers;
//   * two MMA warps issue S = Q^ K^^T (A = Q^ from TMEM, M 128, N 64, K d)
//     and O += P V^ (A = P from TMEM, M 128, N d, K 64) as their inputs
//     become ready;
//   * the softmax warps read their row of S, apply the causal / context mask
//     and an online softmax in base 2 (the reference max moves only when a
//     score exceeds it by more than 2^8) and write P as fp16 back into TMEM
//     (two P buffers, so P(t+1) is written while O(t) runs).
// Q^ = H D q per K block times softmax_scale * log2 e is prepared once per
// call by a small kernel.  Partial (m, l, O) per row and context slice go to
// the workspace in the decode-split format, and the decode combine kernel
// merges the slices and rotates each output row back (D H per V block).
// Every mbarrier wait is bounded.  A wait longer than the caller's limit
// (tq_set_wait_limit_ns) records TQ_ERR_TIMEOUT in this file's device status
// word and goes on waiting, so the launch still completes; a wait longer than
// the hard bound raises the CTA's abort flag, the roles run out their loops
// without work, and the CTA frees its TMEM and returns.  That abort path does
// not wait for products or peer copies already in flight: it is the last
// resort for a device that has stopped making progress, not a way to cancel.
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
// decoding warps (K side, V side): 9 + 9 with setmaxnreg rebalancing (24 warps
// in all, so every decoder thread has at most one 32-code item of its half
// tile at head_dim 256), 4 + 2 without (12 warps)
constexpr int kDecK_RB = 9, kDecV_RB = 9, kDecK = 4, kDecV = 2;
constexpr int kConsRegs = 128, kDecRegs = 64;
constexpr uint32_t kColS = 0, kColP = 64;
// TMEM columns: S (64 fp32) at 0, two P buffers (64 fp16 = 32 columns each) at
// 64 and 96, Q^ (D fp16 = D/2 columns) at 128, O (D fp32) after it; a power
// of two >= the total (exactly 512 at head_dim 256)
template <int D> __host__ __device__ constexpr uint32_t col_o() { return 128u + D / 2; }
template <int D> __host__ __device__ constexpr uint32_t tmem_cols() { return col_o<D>() + D <= 256u ? 256u : 512u; }
constexpr float kLazyP = 8.0f;

// first failure status of a prefill launch since the last read (0 = none)
__device__ int g_prefill_status;
constexpr uint32_t kSuspendNs = 1000000;        // try_wait sleep hint

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

// Warp-wide forms: every lane of a converged warp executes them and the lane
// that elect.sync picks (the same one each time for a full, converged warp)
// issues the MMA or the commit, so an MMA and the commit that tracks it come
// from one thread.
__device__ __forceinline__ void mma_ts_elect(uint32_t d, uint32_t a, uint64_t b, uint32_t idesc, int acc) {
  asm volatile(
      "{\n .reg .pred p, e;\n elect.sync _|e, 0xffffffff;\n setp.ne.b32 p, %4, 0;\n"
      " @e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(d),
      "r"(a), "l"(b), "r"(idesc), "r"(acc)
      : "memory");
}
__device__ __forceinline__ void commit_elect(uint32_t bar) {
  asm volatile(
      "{\n .reg .pred e;\n elect.sync _|e, 0xffffffff;\n"
      " @e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n}\n" ::"r"(bar)
      : "memory");
}
// The same, arriving on the mbarrier at this offset in both CTAs of the pair.
__device__ __forceinline__ void commit_elect_pair(uint32_t bar) {
  const uint16_t mask = 0x3;
  asm volatile(
      "{\n .reg .pred e;\n elect.sync _|e, 0xffffffff;\n"
      " @e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;\n}\n" ::"r"(bar),
      "h"(mask)
      : "memory");
}


__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Wait for the phase of parity `phase` of an mbarrier.  The thread sleeps in
// try_wait (suspend-time hint 1 ms; it wakes as soon as the phase completes)
// instead of spinning.  Past report_ns of wall time the wait sets `late` and
// goes on; past hard_ns it gives up (returns false).
// CLUSTER: the arrivals come from the other CTA of the pair as well, so the
// wait acquires at cluster scope.
template <bool CLUSTER = false>
__device__ __forceinline__ bool bar_wait(uint32_t bar, uint32_t phase, uint64_t report_ns, uint64_t hard_ns,
                                         volatile int& late) {
  uint32_t done;
  if (CLUSTER)
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.test_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(done)
        : "r"(bar), "r"(phase)
        : "memory");
  else
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(done)
        : "r"(bar), "r"(phase)
        : "memory");
  if (done) return true;
  // try_wait sleeps until the phase completes (up to its hint), so the
  // elapsed time is checked after every return, the successful one too
  const uint64_t t0 = global_ns();
  for (;;) {
    if (CLUSTER)
      asm volatile(
          "{\n .reg .pred p;\n mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2, %3;\n"
          " selp.u32 %0, 1, 0, p;\n}\n"
          : "=r"(done)
          : "r"(bar), "r"(phase), "r"(kSuspendNs)
          : "memory");
    else
      asm volatile(
          "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n selp.u32 %0, 1, 0, p;\n}\n"
          : "=r"(done)
          : "r"(bar), "r"(phase), "r"(kSuspendNs)
          : "memory");
    const uint64_t el = global_ns() - t0;
    if (el > report_ns) late = 1;
    if (done) return true;
    if (el > hard_ns) return false;
  }
}

__device__ __forceinline__ void fence_before() { asm volatile("tcgen05.fence::before_thread_sync;\n" ::: "memory"); }
__device__ __forceinline__ void fence_after() { asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory"); }
// every thread of both CTAs of the cluster
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\nbarrier.cluster.wait.acquire.aligned;\n" ::: "memory");
}

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
__device__ __forceinline__ uint32_t mapa_peer(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;\n" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}

// Per-thread constants of the tile decoder: the thread's (token, 32-value
// group) work items and their byte offsets, the same for every tile.
// A thread decodes items of the TOK tokens of a tile that start at tok0
// (all of the tile, or the half a CTA of a pair decodes).
template <int D, int NT>
struct ItemPlan {
  static constexpr int G8 = D / 32;
  static constexpr int TOK = kTok / 2;
  static constexpr int N = (TOK * G8 + NT - 1) / NT;   // items per decoding thread
  int tok[N];
  uint32_t code_off[N], sc_off[N], dst_off[N];
};

template <int D, int NT>
__device__ __forceinline__ ItemPlan<D, NT> make_plan(const CodecParams& P, int tid, int tok0) {
  ItemPlan<D, NT> pl;
  constexpr int G8 = D / 32;
  constexpr int TOK = ItemPlan<D, NT>::TOK;
#pragma unroll
  for (int k = 0; k < ItemPlan<D, NT>::N; ++k) {
    const int item = tid + k * NT;
    const int tok = tok0 + 8 * (item / (8 * G8)) + (item & 7);
    const int grp = (item >> 3) % G8;
    pl.tok[k] = item < TOK * G8 ? tok : kTok;   // kTok: no item
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
// straight into a 32-bit register (zero-extended by the load itself, so no
// instruction has to wait for the value before it is used)
__device__ __forceinline__ uint32_t ldg16(const uint8_t* p) {
  uint32_t v;
  asm volatile("ld.global.nc.u16 %0, [%1];" : "=r"(v) : "l"(p));
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
      } else if (BITS == 3) {
        // 12 bytes at a 4-byte aligned offset: two 8-byte loads of the 16
        // bytes around them (the decode picks the three words, so nothing
        // waits on the loads here).  An 8-byte aligned group is never the
        // last of its row (the last group index, d/32 - 1, is odd), so the
        // second load stays inside the row.
        const uint8_t* c8 = c - (pl.code_off[k] & 4u);
        asm volatile("ld.global.nc.v2.u32 {%0,%1}, [%2];" : "=r"(r.w[k][0]), "=r"(r.w[k][1]) : "l"(c8));
        asm volatile("ld.global.nc.v2.u32 {%0,%1}, [%2];" : "=r"(r.w[k][2]), "=r"(r.w[k][3]) : "l"(c8 + 8));
      } else {
        r.w[k][0] = ldg32(c);
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
// EXACT (the keys): each (token, block) table holds the fp32 products of the
// centroids and the block norm rounded once to fp16 (make_tab_f32).
template <int D, int NT, int BITS, bool EXACT>
__device__ __forceinline__ void decode_regs_b(const ItemPlan<D, NT>& pl, const ItemRegs<D, NT>& r, const uint32_t* c2,
                                              const Tab& fixed, const float* cent, int n_valid, uint32_t tile) {
  auto sts2 = [&](uint32_t off, uint4 v) { sts128(tile + off, v); };
#pragma unroll
  for (int k = 0; k < ItemPlan<D, NT>::N; ++k) {
    if (pl.tok[k] >= kTok) continue;
    const uint32_t dst = pl.dst_off[k];
    if (n_valid == kTok || pl.tok[k] < n_valid) {
      uint32_t n[4];
      if (BITS == 3) {   // the group's three words out of the 16 loaded bytes
        const bool sh = (pl.code_off[k] & 4u) != 0;
        const uint32_t w3[3] = {sh ? r.w[k][1] : r.w[k][0], sh ? r.w[k][2] : r.w[k][1], sh ? r.w[k][3] : r.w[k][2]};
        chunk_words<3>(w3, n);
      } else {
        chunk_words<BITS>(r.w[k], n);
      }
      const uint32_t sc = r.sc[k];
      Tab T;
      uint32_t s2 = 0;
      if (EXACT) {
        T = make_tab_f32<BITS>(cent, h2f((uint16_t)sc));
      } else if (BITS == 4) {
        T = fixed;
        s2 = sc | (sc << 16);
      } else {
        T = make_tab_p<BITS>(c2, sc);
      }
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t o[4];
        lut8<BITS>(n[c], T, o);
        if (BITS == 4 && !EXACT) {
#pragma unroll
          for (int e = 0; e < 4; ++e) o[e] = lut_hmul2(o[e], s2);
        }
        sts2(dst + 128 * c, make_uint4(o[0], o[1], o[2], o[3]));
      }
    } else {
#pragma unroll
      for (int c = 0; c < 4; ++c) sts2(dst + 128 * c, make_uint4(0u, 0u, 0u, 0u));
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

template <int D, int NT, bool EXACT>
__device__ __forceinline__ void decode_regs(int bits, const ItemPlan<D, NT>& pl, const ItemRegs<D, NT>& r,
                                            const CodeTabs& ct, const float* cent, int n_valid, uint32_t tile) {
  switch (bits) {
    case 4: decode_regs_b<D, NT, 4, EXACT>(pl, r, ct.c2, ct.fixed, cent, n_valid, tile); break;
    case 3: decode_regs_b<D, NT, 3, EXACT>(pl, r, ct.c2, ct.fixed, cent, n_valid, tile); break;
    case 2: decode_regs_b<D, NT, 2, EXACT>(pl, r, ct.c2, ct.fixed, cent, n_valid, tile); break;
    default: decode_regs_b<D, NT, 1, EXACT>(pl, r, ct.c2, ct.fixed, cent, n_valid, tile); break;
  }
}


struct PrefillTcArgs {
  const uint8_t* kc;
  const uint8_t* ks;
  const uint8_t* vc;
  const uint8_t* vs;
  const __half* qhat;   // [B*Hkv][R_pad][D]
  float* part;          // [(b*Hq + h)*Tq + i][n_split][D + 4]
  uint64_t report_ns, hard_ns;   // wait limits (see WaitLimits)
  int64_t S_cap, ctx;
  int Hq, Hkv, Tq, R_pad, n_split, causal;
  int64_t per;          // tokens per split (multiple of kTok)
  PageMap pages;        // paging of both caches (table NULL: contiguous)
};


// Record of token 0 of a tile as the decoders address it: the item offsets
// carry the token within the tile.  Contiguous caches: one base per
// (batch, KV head).  Paged caches: the record of this CTA's half, less the
// half's offset (a half never crosses a page: both are 32-token aligned).
struct ContigRec {
  int64_t rec0;
  __device__ __forceinline__ int64_t tile(int64_t t0, int, int) const { return rec0 + t0; }
};
struct PagedRec {
  PageMap pm;
  int64_t S_cap;
  int H, b, h;
  __device__ __forceinline__ int64_t tile(int64_t t0, int half0, int nv) const {
    return nv > half0 ? cache_rec(pm, H, S_cap, b, h, t0 + half0) - half0 : 0;
  }
};

// A decoder role: NT threads of each CTA of a pair decode half of every tile
// of one side (K or V), tokens [32 rank, 32 rank + 32), into the NB-deep ring
// of shared buffers; in the core-matrix layout that half is one contiguous
// block (32 d fp16), which one thread then copies into the same place in the
// peer CTA with a bulk shared::cluster copy that completes on the peer's full
// barrier.  So each CTA holds whole tiles for its own MMAs at half the decode
// work.  Each thread loads its items' packed words two tiles ahead into
// registers, so the global latency hides behind two tile decodes.  Buffer t % NB is refilled once the products that read it NB tiles
// earlier have completed in both CTAs (its free barrier takes a commit from
// each; the peer's commit also implies that the copy out of this buffer has
// landed).  Before returning, the role waits for the products of its last
// tiles, so no arrival from the peer can still be on its way to this CTA.
// BAR_ID: the named barrier that gathers the side's NT threads.
template <int D, int NT, int NB, int BAR_ID, class RecOf, class NValid, class Wait>
__device__ __forceinline__ void decoder_role(const CodecParams& P, const CodeTabs& ct, const uint8_t* codes,
                                             const uint8_t* scales, int ptid, uint32_t full, uint32_t free_bar,
                                             uint32_t buf0, uint32_t tile_bytes, RecOf rec_of, int64_t t_lo,
                                             int n_tiles, uint32_t rank, NValid n_valid_of, Wait wait,
                                             volatile int& abort) {
  constexpr uint32_t kHalfBytes = 32u * D * 2;
  const ItemPlan<D, NT> pl = make_plan<D, NT>(P, ptid, (int)rank * ItemPlan<D, NT>::TOK);
  const uint32_t half_off = rank * kHalfBytes;
  const uint32_t peer_buf0 = mapa_peer(buf0, rank ^ 1u), peer_full = mapa_peer(full, rank ^ 1u);
  ItemRegs<D, NT> r0, r1, r2;
  auto load = [&](int t, ItemRegs<D, NT>& r) {
    const int nv = n_valid_of(t);
    const int64_t rec = rec_of.tile(t_lo + (int64_t)t * kTok, (int)rank * ItemPlan<D, NT>::TOK, nv);
    load_items<D, NT>(P.bits, pl, codes + rec * P.code_bytes, scales + rec * 2 * P.nb, nv, r);
  };
  // tile t decodes from registers loaded two steps earlier; the load of tile
  // t+2 is issued after tile t's arrivals, so no arrival waits on it
  auto step = [&](int t, const ItemRegs<D, NT>& r, ItemRegs<D, NT>& next2) {
    const int kb = t % NB;
    if (t >= NB) wait(free_bar + 8 * kb, (uint32_t)(t / NB - 1) & 1);   // the products NB tiles back are done
    const uint32_t tile = buf0 + (uint32_t)kb * tile_bytes;
    if (!abort) decode_regs<D, NT, BAR_ID == 1>(P.bits, pl, r, ct, P.centroids, n_valid_of(t), tile);
    // the stores before the tensor cores and the bulk copy (async proxy) read them
    asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
    asm volatile("bar.sync %0, %1;\n" ::"n"(BAR_ID), "n"(NT) : "memory");
    if (ptid == NT - 32) {   // the last warp's first thread: it has no item when the half tile has fewer items than threads
      asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(full + 8 * kb) : "memory");
      if (!abort) {
        // only a byte count: the data itself is ordered by the copy's complete_tx
        const uint32_t pbar = peer_full + 8 * kb;
        asm volatile("mbarrier.arrive.expect_tx.relaxed.cluster.shared::cluster.b64 _, [%0], %1;\n" ::"r"(pbar),
                     "n"(kHalfBytes)
                     : "memory");
        asm volatile(
            "cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n" ::"r"(
                peer_buf0 + (uint32_t)kb * tile_bytes + half_off),
            "r"(tile + half_off), "n"(kHalfBytes), "r"(pbar)
            : "memory");
      }
    }
    if (t + 2 < n_tiles) load(t + 2, next2);
  };
  if (n_tiles > 0) load(0, r0);
  if (n_tiles > 1) load(1, r1);
  for (int t = 0; t < n_tiles; t += 3) {
    step(t, r0, r2);
    if (t + 1 < n_tiles) step(t + 1, r1, r0);
    if (t + 2 < n_tiles) step(t + 2, r2, r1);
  }
  for (int t = n_tiles > NB ? n_tiles - NB : 0; t < n_tiles; ++t) wait(free_bar + 8 * (t % NB), (uint32_t)(t / NB) & 1);
}

// Warp-specialised prefill, launched as clusters of two CTAs that take
// consecutive 128-row tiles of the same (batch, KV head, context slice) and
// share the tile decode (see decoder_role).  Warps 0-3 (softmax) own the 128
// TMEM rows; warp 4 issues the S products and warp 5 the O products; NK warps
// decode K tiles and NV warps decode V tiles into NB-deep rings of shared
// buffers, each side at its own pace.
// Handoffs go through mbarriers:
//   kfull/vfull[b]  a decoded tile is in buffer b (one arrival for this CTA's
//                   half, one with the byte count of the peer's half, whose
//                   bulk copy completes the transaction)
//   kfree/vfree[b]  the products that read buffer b are done in both CTAs
//                   (a multicast tcgen05.commit from each)
//   q_full          Q^ is in TMEM (one arrival per softmax warp)
//   s_full          S(t) is in TMEM (commit)
//   s_free          every softmax warp holds S(t) in registers (one arrival per warp)
//   p_full[b]       P(t), t & 1 = b, is in TMEM (one arrival per softmax warp)
//   o_done[b]       O += P(t) V(t), t & 1 = b, is done (commit)
// S(t+1) is issued as soon as S(t) has been read, so it runs on the tensor
// pipe during the softmax of tile t, and O(t) as soon as P(t) is written.  Every barrier is waited on at most one phase behind its last
// completion, so a parity wait is never confused by a later phase.  Waits are
// bounded: a wait that gives up raises a CTA-wide abort flag, after which the
// roles run out their loops without further work or waits.
template <int D, int NK, int NV, int NB, bool RB>
__global__ void __launch_bounds__(192 + 32 * (NK + NV), 1) prefill_ws_kernel(const CodecParams PK, const CodecParams PV,
                                                                             const PrefillTcArgs a) {
  static_assert((192 + 32 * (NK + NV)) % 128 == 0, "whole warpgroups (setmaxnreg acts per warpgroup)");
  constexpr int kNK = 32 * NK, kNV = 32 * NV;
  constexpr uint32_t kTmemCols = tmem_cols<D>();
  constexpr uint32_t kColQ = 128;
  constexpr uint32_t kColO = col_o<D>();
  constexpr uint32_t kTileBytes = kTok * D * 2;
  constexpr uint32_t kGroupBytes = (D / 8) * 128;
  extern __shared__ __align__(1024) uint8_t smem[];
  // kfull[NB], vfull[NB], kfree[NB], vfree[NB], q_full, s_full, s_free, p_full[2], o_done[2]
  __shared__ __align__(8) uint64_t bars[4 * NB + 7];
  __shared__ uint32_t tmem_base;
  __shared__ volatile int s_abort;   // a wait passed the hard bound: the roles run out without work
  __shared__ volatile int s_late;    // a wait passed the caller's limit (reported, not stopped)
  __shared__ CodeTabs s_tabs[2];   // K and V codebooks (fp16 pairs, unscaled 4-bit tables)

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  uint32_t rank;   // 0 or 1 within the pair
  asm volatile("mov.u32 %0, %%cluster_ctarank;\n" : "=r"(rank));
  const int G = a.Hq / a.Hkv;
  const int rt = blockIdx.x, split = blockIdx.y, bh = blockIdx.z;
  const int b = bh / a.Hkv, kvh = bh % a.Hkv;
  const int R = a.Tq * G;
  // both CTAs of the pair walk the same tiles: the causal limit of the pair's last row
  const int last_row = min((rt & ~1) * kRowsTc + 2 * kRowsTc, R) - 1;
  const int64_t max_pos = a.causal ? a.ctx - a.Tq + last_row / G : a.ctx - 1;
  const int64_t t_lo = (int64_t)split * a.per;
  const int64_t t_hi = imin64(imin64(t_lo + a.per, a.ctx), max_pos + 1);
  const int n_tiles = t_hi > t_lo ? (int)((t_hi - t_lo + kTok - 1) / kTok) : 0;

  const uint32_t a_smem = su32(smem);
  // NB decoded K buffers, then NB decoded V buffers
  auto aK = [&](int kb) { return a_smem + (uint32_t)kb * kTileBytes; };
  auto aV = [&](int kb) { return a_smem + (uint32_t)(NB + kb) * kTileBytes; };
  const uint32_t kfull = su32(&bars[0]), vfull = su32(&bars[NB]), kfree = su32(&bars[2 * NB]),
                 vfree = su32(&bars[3 * NB]);
  const uint32_t q_full = su32(&bars[4 * NB]), s_full = su32(&bars[4 * NB + 1]), s_free = su32(&bars[4 * NB + 2]),
                 p_full = su32(&bars[4 * NB + 3]), o_done = su32(&bars[4 * NB + 5]);
  auto n_valid_of = [&](int tile) { return (int)imin64(kTok, t_hi - (t_lo + (int64_t)tile * kTok)); };
  auto wait = [&](uint32_t bar, uint32_t parity) {
    if (s_abort) return false;
    if (bar_wait(bar, parity, a.report_ns, a.hard_ns, s_late)) return true;
    s_abort = 1;
    return false;
  };
  auto wait_cl = [&](uint32_t bar, uint32_t parity) {   // barriers the peer CTA arrives on
    if (s_abort) return false;
    if (bar_wait<true>(bar, parity, a.report_ns, a.hard_ns, s_late)) return true;
    s_abort = 1;
    return false;
  };

  if (tid == 0) {
    s_tabs[0] = make_code_tabs(PK);
    s_tabs[1] = make_code_tabs(PV);
    s_abort = 0;
    s_late = 0;
#pragma unroll
    for (int i = 0; i < NB; ++i) {
      asm volatile("mbarrier.init.shared::cta.b64 [%0], 2;\n" ::"r"(kfull + 8 * i) : "memory");
      asm volatile("mbarrier.init.shared::cta.b64 [%0], 2;\n" ::"r"(vfull + 8 * i) : "memory");
      asm volatile("mbarrier.init.shared::cta.b64 [%0], 2;\n" ::"r"(kfree + 8 * i) : "memory");
      asm volatile("mbarrier.init.shared::cta.b64 [%0], 2;\n" ::"r"(vfree + 8 * i) : "memory");
    }
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 4;\n" ::"r"(q_full) : "memory");
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;\n" ::"r"(s_full) : "memory");
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 4;\n" ::"r"(s_free) : "memory");
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      asm volatile("mbarrier.init.shared::cta.b64 [%0], 4;\n" ::"r"(p_full + 8 * i) : "memory");
      asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;\n" ::"r"(o_done + 8 * i) : "memory");
    }
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;\n" ::"r"(su32(&tmem_base)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n" ::: "memory");
  }
  // both CTAs' barriers are initialised before either arrives on the other's
  fence_before();
  cluster_sync();
  fence_after();
  const uint32_t tmem = tmem_base;
  // a softmax warp's signal: its lanes' TMEM accesses are complete, then one arrival
  auto warp_arrive = [&](uint32_t bar) {
    fence_before();
    __syncwarp();
    if (lane == 0) asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(bar) : "memory");
  };

  if (warp >= 6) {
    // ================= decoders: NK warps fill the K ring, NV warps the V
    // ring.  Each thread loads its items' packed words for tile t+1 into
    // registers before decoding tile t, so the global latency hides behind
    // the decode.
    if (RB) asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;\n" ::"n"(kDecRegs));
    // the contiguous and the paged cache get their own copy of the role, so
    // the contiguous one keeps its single base address
    const ContigRec crec{(int64_t)bh * a.S_cap};
    const PagedRec prec{a.pages, a.S_cap, a.Hkv, b, kvh};
    if (warp < 6 + NK) {
      if (a.pages.table)
        decoder_role<D, kNK, NB, 1>(PK, s_tabs[0], a.kc, a.ks, tid - 192, kfull, kfree, aK(0), kTileBytes, prec, t_lo,
                                    n_tiles, rank, n_valid_of, wait_cl, s_abort);
      else
        decoder_role<D, kNK, NB, 1>(PK, s_tabs[0], a.kc, a.ks, tid - 192, kfull, kfree, aK(0), kTileBytes, crec, t_lo,
                                    n_tiles, rank, n_valid_of, wait_cl, s_abort);
    } else {
      if (a.pages.table)
        decoder_role<D, kNV, NB, 2>(PV, s_tabs[1], a.vc, a.vs, tid - 192 - kNK, vfull, vfree, aV(0), kTileBytes,
                                    prec, t_lo, n_tiles, rank, n_valid_of, wait_cl, s_abort);
      else
        decoder_role<D, kNV, NB, 2>(PV, s_tabs[1], a.vc, a.vs, tid - 192 - kNK, vfull, vfree, aV(0), kTileBytes,
                                    crec, t_lo, n_tiles, rank, n_valid_of, wait_cl, s_abort);
    }
  } else if (warp == 4) {
    // ================= S issue: S(t) = Q^ (TMEM) K^(t)^T once K(t) is decoded
    // and S(t-1) has been read.  The whole warp walks the schedule, one
    // elected lane issues each MMA and commit.  S and O have a warp each, so
    // neither stream of MMAs waits behind the other's handoffs.
    if (RB) asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;\n" ::"n"(kDecRegs));
    const uint32_t idesc_s = (1u << 4) | ((uint32_t)(kTok >> 3) << 17) | ((uint32_t)(kRowsTc >> 4) << 24);
    bool ok = n_tiles > 0 && wait(q_full, 0);
    for (int t = 0; t < n_tiles && ok; ++t) {
      const int kb = t % NB;
      ok = wait_cl(kfull + 8 * kb, (uint32_t)(t / NB) & 1) && (t == 0 || wait(s_free, (uint32_t)(t - 1) & 1));
      if (!ok) break;
      fence_after();
      __syncwarp();
      // fully unrolled: back-to-back MMAs in straight-line code keep the
      // tensor pipe fed; an issue loop with a branch per MMA does not
      const uint64_t dk = sdesc(aK(kb), 128, kGroupBytes);   // + 16 per 16 columns of d (256 bytes)
#pragma unroll
      for (int s = 0; s < D / 16; ++s)
        mma_ts_elect(tmem + kColS, tmem + kColQ + 8 * s, dk + (uint64_t)(16 * s), idesc_s, s > 0);
      commit_elect(s_full);
      commit_elect_pair(kfree + 8 * kb);
    }
  } else if (warp == 5) {
    // ================= O issue: O += P(t) (TMEM) V^(t) once P(t) is written
    // and V(t) decoded
    if (RB) asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;\n" ::"n"(kDecRegs));
    const uint32_t idesc_o = (1u << 4) | (1u << 16) | ((uint32_t)(D >> 3) << 17) | ((uint32_t)(kRowsTc >> 4) << 24);
    bool ok = true;
    for (int t = 0; t < n_tiles && ok; ++t) {
      const int vb = t % NB, pb = t & 1;
      ok = wait(p_full + 8 * pb, (uint32_t)(t >> 1) & 1) && wait_cl(vfull + 8 * vb, (uint32_t)(t / NB) & 1);
      if (!ok) break;
      fence_after();
      __syncwarp();
      const uint64_t dv = sdesc(aV(vb), kGroupBytes, 128);   // + per 16 tokens (2 groups)
#pragma unroll
      for (int s = 0; s < kTok / 16; ++s)
        mma_ts_elect(tmem + kColO, tmem + kColP + 32 * pb + 8 * s, dv + (uint64_t)(s * (2 * kGroupBytes >> 4)),
                     idesc_o, (t == 0 && s == 0) ? 0 : 1);
      commit_elect(o_done + 8 * pb);
      commit_elect_pair(vfree + 8 * vb);
    }
  } else {
    // ================= softmax: one row per thread
    if (RB) asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;\n" ::"n"(kConsRegs));
    const int row = rt * kRowsTc + tid;
    const bool row_ok = row < R;
    const int qi = row_ok ? row / G : a.Tq - 1;
    const int64_t pos = a.ctx - a.Tq + qi;
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
    warp_arrive(q_full);
    float m_run = -INFINITY, l_run = 0.f;
    for (int t = 0; t < n_tiles; ++t) {
      const int64_t t0 = t_lo + (int64_t)t * kTok;
      uint32_t sv[32], sw[32];
      const bool have_s = wait(s_full, (uint32_t)t & 1);   // S(t) written
      fence_after();
      if (have_s) {
        TQ_LD32(lane_base + kColS, sv);
        TQ_LD32(lane_base + kColS + 32, sw);
        asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory");
      } else {
#pragma unroll
        for (int c = 0; c < 32; ++c) sv[c] = sw[c] = __float_as_uint(-INFINITY);
      }
      warp_arrive(s_free);   // S(t+1) may overwrite S now
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
      float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
      for (int c = 0; c < 32; ++c)
        m4[c & 3] = fmaxf(m4[c & 3], fmaxf(__uint_as_float(sv[c]), __uint_as_float(sw[c])));
      const float mx = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
      const bool need = mx > m_run + kLazyP;
      if (__any_sync(0xffffffffu, need)) {
        const float m_new = need ? mx : m_run;
        const float alpha = (need && m_run != -INFINITY) ? ex2f(m_run - m_new) : 1.f;
        m_run = m_new;
        l_run *= alpha;
        if (t >= 1) {
          // O(t-1), the last product issued on O, must be done before O is rescaled
          wait(o_done + 8 * ((t - 1) & 1), (uint32_t)((t - 1) >> 1) & 1);
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
      if (t >= 2) wait(o_done + 8 * (t & 1), (uint32_t)((t - 2) >> 1) & 1);
      fence_after();
      const float mref = m_run == -INFINITY ? 0.f : m_run;
      uint32_t pw[32];
      float s4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int c = 0; c < 32; ++c) {
        const float p0 = ex2f(__uint_as_float(c < 16 ? sv[2 * c] : sw[2 * c - 32]) - mref);
        const float p1 = ex2f(__uint_as_float(c < 16 ? sv[2 * c + 1] : sw[2 * c + 1 - 32]) - mref);
        s4[c & 3] += p0 + p1;
        const __half2 h = __floats2half2_rn(p0, p1);
        pw[c] = *reinterpret_cast<const uint32_t*>(&h);
      }
      l_run += (s4[0] + s4[1]) + (s4[2] + s4[3]);
      TQ_ST32(lane_base + kColP + 32 * (t & 1), pw);
      asm volatile("tcgen05.wait::st.sync.aligned;\n" ::: "memory");
      warp_arrive(p_full + 8 * (t & 1));
    }
    if (n_tiles > 0) wait(o_done + 8 * ((n_tiles - 1) & 1), (uint32_t)((n_tiles - 1) >> 1) & 1);
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
  // neither CTA leaves while the other may still store into its shared memory
  fence_before();
  cluster_sync();
  if (tid == 0 && (s_abort || s_late)) atomicCAS(&g_prefill_status, 0, (int)TQ_ERR_TIMEOUT);
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
  const int row_tiles = (Tq * G + 2 * kRowsTc - 1) / (2 * kRowsTc) * 2;   // whole CTA pairs
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

// Q^ rows are padded to whole CTA pairs (256 rows).
size_t prefill_tc_workspace(int B, int Hq, int Hkv, int d, int Tq, int64_t ctx) {
  const int G = Hq / Hkv;
  const int R_pad = (Tq * G + 2 * kRowsTc - 1) / (2 * kRowsTc) * (2 * kRowsTc);
  const int ns = prefill_tc_splits(B, Hkv, G, Tq, ctx);
  const size_t qbytes = (size_t)B * Hkv * R_pad * d * 2;
  const size_t pbytes = (size_t)B * Hq * Tq * ns * (d + 4) * 4;
  return ((qbytes + 255) / 256) * 256 + pbytes;
}

// The warp-specialised kernel with 18 decoder warps and setmaxnreg moving
// registers to the softmax warps, when its launch register count makes that
// split exact (launch total >= softmax + other shares); otherwise 6 decoder
// warps without rebalancing.
template <int D>
int launch_ws(const CodecParams& PK, const CodecParams& PV, const PrefillTcArgs& a, dim3 grid, cudaStream_t st) {
  const size_t sm = tc_smem<D>(3);
  constexpr int kThreadsRB = 192 + 32 * (kDecK_RB + kDecV_RB), kThreads = 192 + 32 * (kDecK + kDecV);
  static int use_rb = -1;   // decided once per process (the kernel image is fixed)
  if (use_rb < 0) {
    cudaFuncAttributes fa;
    use_rb = 0;
    if (cudaFuncGetAttributes(&fa, prefill_ws_kernel<D, kDecK_RB, kDecV_RB, 3, true>) == cudaSuccess) {
      const long launch = (long)kThreadsRB * fa.numRegs;
      const long need = 128L * kConsRegs + (long)(kThreadsRB - 128) * kDecRegs;
      use_rb = (fa.numRegs >= kDecRegs && fa.numRegs <= kConsRegs && launch >= need) ? 1 : 0;
    }
  }
  // clusters of two CTAs along x (grid.x is even)
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.dynamicSmemBytes = sm;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e;
  if (use_rb) {
    auto k = prefill_ws_kernel<D, kDecK_RB, kDecV_RB, 3, true>;
    if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm)) return TQ_ERR_CUDA;
    cfg.blockDim = dim3(kThreadsRB);
    e = cudaLaunchKernelEx(&cfg, k, PK, PV, a);
  } else {
    auto k = prefill_ws_kernel<D, kDecK, kDecV, 3, false>;
    if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm)) return TQ_ERR_CUDA;
    cfg.blockDim = dim3(kThreads);
    e = cudaLaunchKernelEx(&cfg, k, PK, PV, a);
  }
  return e == cudaSuccess ? TQ_OK : TQ_ERR_CUDA;
}

int launch_prefill_tc(const CodecParams& PK, const CodecParams& PV, const uint8_t* kc, const uint16_t* ks,
                      const uint8_t* vc, const uint16_t* vs, const uint16_t* q, int B, int Hq, int Hkv, int Tq,
                      int64_t S_cap, int64_t ctx, int causal, float qscale, uint16_t* out, void* ws,
                      const PageMap& pages, cudaStream_t st) {
  const int d = PK.d;
  const int G = Hq / Hkv;
  const int R_pad = (Tq * G + 2 * kRowsTc - 1) / (2 * kRowsTc) * (2 * kRowsTc);
  const int ns = prefill_tc_splits(B, Hkv, G, Tq, ctx);
  uint8_t* base = static_cast<uint8_t*>(ws);
  const size_t qbytes = (size_t)B * Hkv * R_pad * d * 2;
  __half* qhat = reinterpret_cast<__half*>(base);
  float* part = reinterpret_cast<float*>(base + ((qbytes + 255) / 256) * 256);
  const WaitLimits wl = wait_limits();
  int64_t per = (ctx + ns - 1) / ns;
  per = (per + kTok - 1) / kTok * kTok;
  PrefillTcArgs a{kc, reinterpret_cast<const uint8_t*>(ks), vc, reinterpret_cast<const uint8_t*>(vs), qhat, part,
                  wl.report_ns, wl.hard_ns, S_cap, ctx, Hq, Hkv, Tq, R_pad, ns, causal, per, pages};
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

// First failure status a prefill launch recorded since the last read with
// clear set (0 = none).
int prefill_tc_status(int clear, int* status) {
  int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_prefill_status, sizeof(int)) != cudaSuccess) return TQ_ERR_CUDA;
  if (clear && v != 0) {
    const int zero = 0;
    if (cudaMemcpyToSymbol(g_prefill_status, &zero, sizeof(int)) != cudaSuccess) return TQ_ERR_CUDA;
  }
  *status = v;
  return TQ_OK;
}

}  // namespace tq
