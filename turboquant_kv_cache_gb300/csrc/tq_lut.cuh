// Code -> fp16 lookup helpers shared by the tensor-core decode and prefill
// kernels: nibble words of a packed 32-code group, fp16 centroid tables
// (optionally scaled by a block norm) split into low / high bytes, and the
// byte-permute lookup that turns a nibble word into four fp16 pairs.
#pragma once

#include "tq_device.cuh"

namespace tq {

__device__ __forceinline__ uint32_t lut_lds32(uint32_t a) {
  uint32_t v;
  asm volatile("ld.shared.b32 %0, [%1];" : "=r"(v) : "r"(a));
  return v;
}
__device__ __forceinline__ uint2 lut_lds64(uint32_t a) {
  uint2 v;
  asm volatile("ld.shared.v2.b32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(a));
  return v;
}
__device__ __forceinline__ uint4 lut_lds128(uint32_t a) {
  uint4 v;
  asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a));
  return v;
}
__device__ __forceinline__ uint32_t lut_hmul2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
// Byte permute with the selector taken as is (the C intrinsic masks it).
__device__ __forceinline__ uint32_t lut_prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}

// Nibble words (code k of chunk c in bits 4k..4k+2) of one 32-code group,
// from its packed words w (see the layout in include/tq.h).
template <int BITS>
__device__ __forceinline__ void chunk_words(const uint32_t* w, uint32_t* n) {
  if (BITS == 4) {
    n[0] = w[0]; n[1] = w[1]; n[2] = w[2]; n[3] = w[3];
  } else if (BITS == 3) {
    n[0] = w[0] & 0x77777777u;
    n[1] = w[1] & 0x77777777u;
    n[2] = w[2] & 0x77777777u;
    // chunk 3 rides in bit 3 of every nibble; the shifts run as high-half
    // multiplies, off the integer logic pipe
    n[3] = __umulhi(w[0] & 0x88888888u, 1u << 29) + __umulhi(w[1] & 0x88888888u, 1u << 30) +
           __umulhi(w[2] & 0x88888888u, 1u << 31);
  } else if (BITS == 2) {
    n[0] = w[0] & 0x33333333u;
    n[1] = w[1] & 0x33333333u;
    n[2] = __umulhi(w[0], 1u << 30) & 0x33333333u;
    n[3] = __umulhi(w[1], 1u << 30) & 0x33333333u;
  } else {  // 1 bit: bit c of nibble k is code 8c + k
    n[0] = w[0] & 0x11111111u;
    n[1] = __umulhi(w[0], 1u << 31) & 0x11111111u;
    n[2] = __umulhi(w[0], 1u << 30) & 0x11111111u;
    n[3] = __umulhi(w[0], 1u << 29) & 0x11111111u;
  }
}

// Packed words of one 32-code group at shared address a (4-byte aligned;
// 8- or 16-byte aligned for 2 and 4 bits).
template <int BITS>
__device__ __forceinline__ void load_group(uint32_t a, uint32_t* w) {
  if (BITS == 4) {
    const uint4 v = lut_lds128(a);
    w[0] = v.x; w[1] = v.y; w[2] = v.z; w[3] = v.w;
  } else if (BITS == 3) {
    w[0] = lut_lds32(a); w[1] = lut_lds32(a + 4); w[2] = lut_lds32(a + 8);
  } else if (BITS == 2) {
    const uint2 v = lut_lds64(a);
    w[0] = v.x; w[1] = v.y;
  } else {
    w[0] = lut_lds32(a);
  }
}

// Lookup tables of one codebook (optionally scaled): low and high bytes of
// the fp16 values, entries 0-7 in t[0..3], entries 8-15 in t[4..7].
struct Tab {
  uint32_t t[8];
};

// fp16 centroid pairs (c0,c1), (c2,c3), ... of a codebook (up to 16 entries)
template <int BITS>
struct Cent {
  uint32_t c2[(1 << BITS) / 2];
};

template <int BITS>
__device__ __forceinline__ Cent<BITS> make_cent(const CodecParams& P) {
  Cent<BITS> c;
#pragma unroll
  for (int k = 0; k < (1 << BITS) / 2; ++k)
    c.c2[k] = (uint32_t)f2h(P.centroids[2 * k]) | ((uint32_t)f2h(P.centroids[2 * k + 1]) << 16);
  return c;
}

// Byte tables from fp16 entry pairs h[k] = (e_2k, e_2k+1).
template <int BITS>
__device__ __forceinline__ Tab tab_from_pairs(const uint32_t* h) {
  Tab T;
  if (BITS == 1) {
    T.t[0] = lut_prmt(h[0], h[0], 0x6420);
    T.t[2] = lut_prmt(h[0], h[0], 0x7531);
    T.t[1] = T.t[0];
    T.t[3] = T.t[2];
  } else if (BITS == 2) {
    T.t[0] = lut_prmt(h[0], h[1], 0x6420);
    T.t[2] = lut_prmt(h[0], h[1], 0x7531);
    T.t[1] = T.t[0];
    T.t[3] = T.t[2];
  } else {
    T.t[0] = lut_prmt(h[0], h[1], 0x6420);
    T.t[1] = lut_prmt(h[2], h[3], 0x6420);
    T.t[2] = lut_prmt(h[0], h[1], 0x7531);
    T.t[3] = lut_prmt(h[2], h[3], 0x7531);
    if (BITS == 4) {
      T.t[4] = lut_prmt(h[4], h[5], 0x6420);
      T.t[5] = lut_prmt(h[6], h[7], 0x6420);
      T.t[6] = lut_prmt(h[4], h[5], 0x7531);
      T.t[7] = lut_prmt(h[6], h[7], 0x7531);
    }
  }
  return T;
}

// tables of the centroids (fp16 pairs c2[k] = (c_2k, c_2k+1)) times the fp16
// norm s (s = 1.0 for unscaled): fp16 products of the fp16 centroids
template <int BITS>
__device__ __forceinline__ Tab make_tab_p(const uint32_t* c2, uint32_t s) {
  const uint32_t s2 = s | (s << 16);
  uint32_t h[8];
#pragma unroll
  for (int k = 0; k < (1 << BITS) / 2; ++k) h[k] = lut_hmul2(c2[k], s2);
  return tab_from_pairs<BITS>(h);
}

template <int BITS>
__device__ __forceinline__ Tab make_tab(const Cent<BITS>& c, uint32_t s) {
  return make_tab_p<BITS>(c.c2, s);
}

// Tables of the centroids c (fp32) times the norm s, each entry the fp32
// product rounded once to fp16.  The fp16-product tables above round the
// centroid first and the product again; for keys that double rounding is
// the largest error of the attention output, because the softmax turns a
// score error into a relative weight error (with heavy-tailed keys at long
// context it alone exceeds the 2e-3 attention tolerance).
template <int BITS>
__device__ __forceinline__ Tab make_tab_f32(const float* c, float s) {
  uint32_t h[8];
#pragma unroll
  for (int k = 0; k < (1 << BITS) / 2; ++k) {
    const __half2 v = __floats2half2_rn(c[2 * k] * s, c[2 * k + 1] * s);
    h[k] = *reinterpret_cast<const uint32_t*>(&v);
  }
  return tab_from_pairs<BITS>(h);
}

// Four fp16x2 registers (codes 0-1, 2-3, 4-5, 6-7) of a nibble word.
template <int BITS>
__device__ __forceinline__ void lut8(uint32_t n, const Tab& T, uint32_t* o) {
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    const uint32_t s = half ? __umulhi(n, 1u << 16) : n;
    uint32_t lo, hi;
    if (BITS == 4) {
      const uint32_t s7 = s & 0x7777u;
      const uint32_t lo0 = lut_prmt(T.t[0], T.t[1], s7), hi0 = lut_prmt(T.t[2], T.t[3], s7);
      const uint32_t lo1 = lut_prmt(T.t[4], T.t[5], s7), hi1 = lut_prmt(T.t[6], T.t[7], s7);
      // byte mask 0xff where bit 3 of the nibble is set: bit 3 moved to the
      // byte-select bit 2 picks 0x00 / 0xff from the constant pair
      const uint32_t m = lut_prmt(0u, 0xffffffffu, __umulhi(s, 1u << 31));
      lo = (lo0 & ~m) | (lo1 & m);
      hi = (hi0 & ~m) | (hi1 & m);
    } else {
      lo = lut_prmt(T.t[0], T.t[1], s);
      hi = lut_prmt(T.t[2], T.t[3], s);
    }
    o[2 * half] = lut_prmt(lo, hi, 0x5140);
    o[2 * half + 1] = lut_prmt(lo, hi, 0x7362);
  }
}

}  // namespace tq
