// Building blocks of the tensor-core quantise kernels (tq_quant_fast.cu,
// tq_quant_qjl.cu): TMA loads, tcgen05 MMAs and their shared-memory
// descriptors, mbarrier waits bounded at two levels, and the cell-table
// bucketize (host table builder included).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstring>

#include "tq_device.cuh"

namespace tq {
namespace tcq {

constexpr float kMagic = 12582912.0f;       // 1.5 * 2^23
constexpr int kMaxCells = 64;
constexpr uint32_t kSuspendNs = 100000;     // try_wait sleep hint
constexpr unsigned kPollNs = 128;           // sleep between polls of an mbarrier

struct CellTable {
  int n_cells;      // C
  float inv2r;      // 1 / (2R), R beyond the outermost boundary
  uint32_t cell[kMaxCells + 1];
};

__device__ __forceinline__ uint32_t su32(const void* p) { return static_cast<uint32_t>(__cvta_generic_to_shared(p)); }

__device__ __forceinline__ uint32_t lds32(uint32_t a) {
  uint32_t v;
  asm volatile("ld.shared.b32 %0, [%1];" : "=r"(v) : "r"(a));
  return v;
}

// TMA: the 2-D box at (x, y) of a tensor map into shared memory, completing
// on an mbarrier
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];\n" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
      : "memory");
}
__device__ __forceinline__ void arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(bar), "r"(bytes) : "memory");
}

// byte offset of element (row, col) in a core-matrix tile of `cols` columns:
// core matrix (row/8, col/8) at ((row/8) * (cols/8) + col/8) * 128, row-major
// 8 x 16 bytes inside
__host__ __device__ __forceinline__ uint32_t cm_off(int row, int col, int cols) {
  return (uint32_t)(((row >> 3) * (cols >> 3) + (col >> 3)) * 128 + (row & 7) * 16 + (col & 7) * 2);
}

// shared-memory matrix descriptor, no swizzle: lbo = byte step between core
// matrices along K, sbo = along M / N
__device__ __forceinline__ uint64_t sdesc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  return (uint64_t)((saddr >> 4) & 0x3FFF) | ((uint64_t)((lbo >> 4) & 0x3FFF) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFF) << 32) | ((uint64_t)1 << 46);
}

// descriptor of a K-major operand whose rows are `row_bytes` (128 or 64)
// long, 16-byte chunks swizzled within each 8-row atom (128B / 64B modes);
// the atom stride is 8 rows
__device__ __forceinline__ uint64_t sdesc_swz(uint32_t saddr, int row_bytes) {
  const uint64_t mode = row_bytes == 128 ? 2 : 4;
  return (uint64_t)((saddr >> 4) & 0x3FFF) | ((uint64_t)1 << 16) | ((uint64_t)((8 * row_bytes) >> 4) << 32) |
         ((uint64_t)1 << 46) | (mode << 61);
}

// warp-wide: the lane elect.sync picks issues the MMA / the commit, so an MMA
// and the commit that tracks it come from one thread
__device__ __forceinline__ void mma_ss_elect(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, int acc) {
  asm volatile(
      "{\n .reg .pred p, e;\n elect.sync _|e, 0xffffffff;\n setp.ne.b32 p, %4, 0;\n"
      " @e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d),
      "l"(a), "l"(b), "r"(idesc), "r"(acc)
      : "memory");
}
// the same with the A operand in TMEM (fp16 pairs, one row per lane)
__device__ __forceinline__ void mma_ts_elect(uint32_t d, uint32_t a_tmem, uint64_t b, uint32_t idesc, int acc) {
  asm volatile(
      "{\n .reg .pred p, e;\n elect.sync _|e, 0xffffffff;\n setp.ne.b32 p, %4, 0;\n"
      " @e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(d),
      "r"(a_tmem), "l"(b), "r"(idesc), "r"(acc)
      : "memory");
}
__device__ __forceinline__ void commit_elect(uint32_t bar) {
  asm volatile(
      "{\n .reg .pred e;\n elect.sync _|e, 0xffffffff;\n"
      " @e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n}\n" ::"r"(bar)
      : "memory");
}
__device__ __forceinline__ void fence_before() { asm volatile("tcgen05.fence::before_thread_sync;\n" ::: "memory"); }
__device__ __forceinline__ void fence_after() { asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory"); }
// generic-proxy writes to shared memory (stores, cp.async) before the tensor
// cores read them
__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory"); }

__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Wait for phase `parity` of an mbarrier.  Past report_ns of wall time the
// wait sets `late` and goes on; past hard_ns it gives up (returns false).
// Callers combine the lanes' results with __all_sync, so a warp takes one
// decision even when its lanes time out at different moments.
__device__ __forceinline__ bool bar_wait(uint32_t bar, uint32_t parity, uint64_t report_ns, uint64_t hard_ns,
                                         int& late) {
  uint32_t done = 0;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(done)
      : "r"(bar), "r"(parity)
      : "memory");
  if (done) return true;
  // try_wait may itself sleep until the phase completes (up to its hint), so
  // the elapsed time is checked after every return, the successful one too
  const uint64_t t0 = global_ns();
  for (;;) {
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(done)
        : "r"(bar), "r"(parity), "r"(kSuspendNs)
        : "memory");
    const uint64_t el = global_ns() - t0;
    if (el > report_ns) late = 1;
    if (done) return true;
    if (el > hard_ns) return false;
    __nanosleep(kPollNs);   // leave the issue slots to the warps that have work
  }
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

// 16 consecutive 32-bit TMEM columns of this thread's lane from registers
#define TQ_ST16(taddr, v)                                                                                          \
  asm volatile(                                                                                                    \
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};\n" ::  \
          "r"(taddr),                                                                                              \
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]),           \
      "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])                            \
      : "memory")

// w += inc when s > the boundary held in entry e (as a float)
__device__ __forceinline__ void add_if_gt(uint32_t& w, float s, uint32_t e, uint32_t inc) {
  asm("{\n .reg .pred p;\n setp.gt.f32 p, %1, %2;\n @p add.u32 %0, %0, %3;\n}"
      : "+r"(w)
      : "f"(s), "f"(__uint_as_float(e)), "r"(inc));
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}

// The cell table of a codebook for the bucketize below; false when no
// C <= kMaxCells separates the boundaries.
//
// Bucketize, code = #{k : y > beta_k}: with s = sat(y / (2R ||y||) + 1/2)
// in [0, 1], round(s*C) picks one of C+1 cells that hold at most one
// boundary each (rounding is monotone, so every boundary in a lower cell is
// below s and every one in a higher cell above it).  A cell entry holds that
// boundary in s units with the count of boundaries below the cell in its low
// four mantissa bits (a shift of at most 15 ulp, far inside the 1e-5 tie
// band); code = count + (s > boundary).  Kernels replicate the table per
// lane so the lookup has no bank conflicts.
inline bool make_cells(const CodecParams& P, CellTable* a) {
  const int K = 1 << P.bits;
  float bmax = 0.f;
  for (int k = 0; k < K - 1; ++k) bmax = std::fmax(bmax, std::fabs(P.bounds[k]));
  if (!(bmax > 0.f) || !std::isfinite(bmax)) return false;
  a->inv2r = 0.5f / (bmax * 1.0625f);
  float sig[16];
  for (int k = 0; k < K - 1; ++k) sig[k] = std::fmaf(P.bounds[k], a->inv2r, 0.5f);
  for (int C = 16; C <= kMaxCells; C *= 2) {
    int cellk[16];
    bool ok = true;
    for (int k = 0; k < K - 1; ++k) {
      cellk[k] = (int)std::nearbyintf(sig[k] * (float)C);
      if (k > 0 && cellk[k] <= cellk[k - 1]) ok = false;
    }
    if (!ok) continue;
    a->n_cells = C;
    for (int c = 0; c <= C; ++c) {
      uint32_t below = 0;
      float bnd = 2.0f;
      for (int k = 0; k < K - 1; ++k) {
        if (cellk[k] < c) ++below;
        if (cellk[k] == c) bnd = sig[k];
      }
      uint32_t bits;
      std::memcpy(&bits, &bnd, 4);
      a->cell[c] = (bits & ~15u) | below;
    }
    return true;
  }
  return false;
}

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// cuTensorMapEncodeTiled from the driver (a host-only encoding call)
inline EncodeTiledFn encode_tiled() {
  static EncodeTiledFn fn = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      p = nullptr;
    return reinterpret_cast<EncodeTiledFn>(p);
  }();
  return fn;
}

// Tensor map of fp16 rows: [n_vec][d], rows `stride` elements apart, read in
// boxes of 128 rows x 64 columns (128-byte rows, 128-byte swizzle: the layout
// sdesc_swz(., 128) names); rows past n_vec read as zero.  False when the rows
// cannot be described (row coordinates are 32-bit).
inline bool make_rows_map(const __half* x, int d, int64_t n_vec, int64_t stride, CUtensorMap* map) {
  const EncodeTiledFn fn = encode_tiled();
  if (!fn || n_vec >= ((int64_t)1 << 31) - 128) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)d, (cuuint64_t)n_vec};
  const cuuint64_t strides[1] = {(cuuint64_t)stride * 2};
  const cuuint32_t box[2] = {64u, 128u};
  const cuuint32_t estr[2] = {1u, 1u};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<__half*>(x), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace tcq
}  // namespace tq
