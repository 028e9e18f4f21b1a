// Device helpers shared by the libtq kernels.
#pragma once

#include <cuda_fp16.h>
#include <stdint.h>

#include "tq_internal.h"

namespace tq {

constexpr unsigned kFull = 0xffffffffu;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kSqrtHalfPi = 1.2533141373155003f;  // sqrt(pi/2), QJL estimator constant

__host__ __device__ __forceinline__ int64_t imin64(int64_t a, int64_t b) { return a < b ? a : b; }

__device__ __forceinline__ float h2f(uint16_t h) { return __half2float(__ushort_as_half(h)); }
__device__ __forceinline__ uint16_t f2h(float f) { return __half_as_ushort(__float2half_rn(f)); }

// Sign bits of D for 8 consecutive coordinates starting at i0 (i0 % 8 == 0).
__device__ __forceinline__ uint32_t sign_byte(const CodecParams& P, int i0) {
  return (P.sign_bits[i0 >> 5] >> (i0 & 31)) & 0xffu;
}

// Record of token t of (batch b, head h) in a cache of H heads and S_cap
// slots, contiguous or paged.
__device__ __forceinline__ int64_t cache_rec(const PageMap& pm, int H, int64_t S_cap, int b, int h, int64_t t) {
  if (!pm.table) return ((int64_t)b * H + h) * S_cap + t;
  const int64_t page = pm.table[(int64_t)b * pm.pages_per_seq + t / pm.page_size];
  return (page * H + h) * pm.page_size + t % pm.page_size;
}

// Record of quantised vector i under a RowMap, or -1 when it is not stored.
__device__ __forceinline__ int64_t map_row(const RowMap& m, int64_t i) {
  if (!m.pos) return i;
  const int64_t bh = i / m.n_new;
  const int64_t slot = (int64_t)m.pos[bh / m.H] + (i - bh * m.n_new);
  if (slot < 0 || slot >= m.S_cap) return -1;
  return cache_rec(m.pages, m.H, m.S_cap, (int)(bh / m.H), (int)(bh % m.H), slot);
}

__device__ __forceinline__ float flip(float v, uint32_t bit) {
  return __uint_as_float(__float_as_uint(v) ^ (bit << 31));
}

// Unnormalised Walsh-Hadamard butterfly over 8 register values (strides
// 1, 2, 4 of the natural / Sylvester ordering).
__device__ __forceinline__ void wht8(float* v) {
#pragma unroll
  for (int h = 1; h < 8; h <<= 1) {
#pragma unroll
    for (int r = 0; r < 8; ++r) {
      if ((r & h) == 0) {
        const float a = v[r], b = v[r + h];
        v[r] = a + b;
        v[r + h] = a - b;
      }
    }
  }
}

// Cross-lane butterfly stages: lanes hold 8 consecutive coordinates each;
// the transform spans `lanes` lanes (a power of two, <= 32), lane bit o
// selects the upper half of the stride-8*o butterfly.
__device__ __forceinline__ void wht_cross(float* v, int sub, int lanes) {
  for (int o = 1; o < lanes; o <<= 1) {
#pragma unroll
    for (int r = 0; r < 8; ++r) {
      const float p = __shfl_xor_sync(kFull, v[r], o);
      v[r] = (sub & o) ? (p - v[r]) : (v[r] + p);
    }
  }
}

__device__ __forceinline__ float group_sum(float v, int lanes) {
  for (int o = 1; o < lanes; o <<= 1) v += __shfl_xor_sync(kFull, v, o);
  return v;
}

// Nibble word (8 codes, code k in bits 4k..4k+3) of the 8-code chunk w
// (0..3) of a 32-code group whose packed words start at `g`.
__device__ __forceinline__ uint32_t load_chunk(const uint32_t* g, int bits, int w) {
  switch (bits) {
    case 4: return g[w];
    case 3:
      if (w < 3) return g[w] & 0x77777777u;
      return ((g[0] >> 3) & 0x11111111u) | ((g[1] >> 2) & 0x22222222u) | ((g[2] >> 1) & 0x44444444u);
    case 2:
      return w < 2 ? (g[w] & 0x33333333u) : ((g[w - 2] >> 2) & 0x33333333u);
    default:
      return (g[0] >> w) & 0x11111111u;
  }
}

// load_chunk over a group whose k-th packed word is word(k) (for groups
// that are not 4-byte aligned, e.g. inside a block record).
template <class Word>
__device__ __forceinline__ uint32_t load_chunk_by(Word word, int bits, int w) {
  switch (bits) {
    case 4: return word(w);
    case 3:
      if (w < 3) return word(w) & 0x77777777u;
      return ((word(0) >> 3) & 0x11111111u) | ((word(1) >> 2) & 0x22222222u) | ((word(2) >> 1) & 0x44444444u);
    case 2:
      return w < 2 ? (word(w) & 0x33333333u) : ((word(w - 2) >> 2) & 0x33333333u);
    default:
      return (word(0) >> w) & 0x11111111u;
  }
}

// Code of coordinate i (0..d-1) of one packed vector record.
__device__ __forceinline__ int code_at(const uint32_t* rec, int bits, int i) {
  const uint32_t* g = rec + (i >> 5) * bits;
  const int s = i & 31;
  const uint32_t n = load_chunk(g, bits, s >> 3);
  return (n >> (4 * (s & 7))) & 0xf;
}

}  // namespace tq
