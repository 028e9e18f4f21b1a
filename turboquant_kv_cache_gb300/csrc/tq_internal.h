// Internal definitions shared by the host layer and the CUDA kernels of
// libtq.  Nothing here is part of the public ABI (include/tq.h).
#pragma once

#include <stddef.h>
#include <stdint.h>

#include <type_traits>

#include "tq.h"

namespace tq {

constexpr int kMaxDim = 256;
constexpr int kMaxQjl = 256;
constexpr int kMaxQjlV = 128;   // QJL rows of V the decode takes

// Everything a kernel needs to know about one codec layout, passed by value
// as a kernel parameter (no device-side state in the library).
struct CodecParams {
  int d;         // head_dim
  int blk;       // rotation / norm block
  int bits;      // MSE bits
  int m;         // QJL rows (0 = none)
  int nc;        // norm correction
  int nb;        // d / blk
  int code_bytes;  // d * bits / 8
  int qjl_bytes;   // m / 8
  float inv_sqrt_blk;                 // 1 / sqrt(blk)
  uint32_t sign_bits[kMaxDim / 32];   // bit i set <=> D_i = -1
  float centroids[16];                // ascending, 2^bits used
  float bounds[16];                   // 2^bits - 1 used
};

// Fills `p` from a public layout; returns TQ_OK or a tq_status.  For 8-bit
// codes the centroid and boundary arrays stay empty: see Codebook8.
int make_params(const tq_layout* layout, CodecParams* p);

// The 256-level codebook of an 8-bit layout.  Too large for CodecParams
// (which every kernel takes), so only the kernels that read 8-bit codes
// take it, as a separate by-value parameter.
struct Codebook8 {
  float c[256];   // centroids, ascending
  float b[256];   // 255 midpoints, then +inf
};
struct NoCodebook8 {};
template <bool W8>
using Codebook8Param = typename std::conditional<W8, Codebook8, NoCodebook8>::type;

int make_codebook8(const tq_layout* layout, Codebook8* cb);

// Validates a public layout without building tables.
int check_layout(const tq_layout* layout);

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Paging of a cache (tq_kv_view): table == NULL for contiguous
// [B, H, S_cap] records.
struct PageMap {
  const int32_t* table;   // device [B][pages_per_seq], or NULL
  int32_t page_size, pages_per_seq;
};

// Where quantised vector i is stored.  pos == NULL: record i.  Otherwise the
// input holds n_new new tokens of every (batch, head) of a cache of H heads
// and S_cap slots, vector i = (b*H + h)*n_new + j, and it goes to the record
// of slot pos[b] + j (contiguous or paged, see PageMap); a slot outside
// [0, S_cap) is not written.
struct RowMap {
  const int32_t* pos;   // device [B], or NULL
  int32_t n_new, H;
  int64_t S_cap;
  PageMap pages;
};

// Checks a view's paging against the call's S_cap; TQ_OK or TQ_ERR_ARG.
inline int check_paging(const tq_kv_view* v, int64_t S_cap) {
  if (!v->page_table) return TQ_OK;
  if (v->page_size <= 0 || v->page_size % 32 || v->pages_per_seq <= 0) return TQ_ERR_ARG;
  return (int64_t)v->page_size * v->pages_per_seq >= S_cap ? TQ_OK : TQ_ERR_ARG;
}
inline bool same_paging(const tq_kv_view* a, const tq_kv_view* b) {
  return a->page_table == b->page_table && (!a->page_table || (a->page_size == b->page_size &&
                                                               a->pages_per_seq == b->pages_per_seq));
}

// Bounded device-side waits.  A wait longer than the caller's limit
// (tq_set_wait_limit_ns; default kDefaultWaitNs) records TQ_ERR_TIMEOUT in
// the device status word of its translation unit and goes on waiting; one
// longer than the hard bound stops its CTA.
constexpr uint64_t kDefaultWaitNs = 2000000000ull;
struct WaitLimits {
  uint64_t report_ns;   // record TQ_ERR_TIMEOUT past this
  uint64_t hard_ns;     // stop past this (>= report_ns, at least 2 s)
};
WaitLimits wait_limits();

// Device status words of the translation units whose kernels wait (read, and
// reset when clear != 0, on the current device; synchronous).
int quantize_fast_status(int clear, int* status);
int quantize_qjl_tc_status(int clear, int* status);
int prefill_tc_status(int clear, int* status);

}  // namespace tq
