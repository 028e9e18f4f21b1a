// Recursive polar-angle quantizer ("TurboQuant: 3-Bit Compression with
// Zero Overhead", cneuralnets, Part 1): a vector of d = 2^k values becomes
// its L2 norm and d - 1 angles (pairs of coordinates, then pairs of radii,
// to atan2 and sqrt, level by level), each angle rounded on a uniform grid
// of 2^b points over [-pi, pi]; decoding rebuilds the tree from the root
// with r cos / r sin.
//
// One warp per vector: lane l holds the d/32 consecutive coordinates
// E*l .. E*l+E-1, so the first log2(E) levels of the tree stay in the lane
// and the last five pair lanes through shuffles.  Angle indices go to a
// per-warp byte array in shared memory in storage order (level 1 first, a
// 0 index after the root's), then lane p packs 8-code chunk p into the same
// nibble-word layout as the MSE codes.
#include <cuda_runtime.h>
#include <math.h>

#include "tq_device.cuh"

namespace tq {
namespace {

constexpr int kPolWarps = 4;
constexpr float kPi = 3.14159265358979323846f;

// first angle of level L (1-based) in storage order: d - d / 2^(L-1)
template <int D>
__device__ __forceinline__ int level_off(int L) {
  return D - (D >> (L - 1));
}

__device__ __forceinline__ int angle_code(float theta, float steps) {
  const float t = rintf((theta + kPi) * (steps / (2.f * kPi)));
  return (int)fminf(fmaxf(t, 0.f), steps);
}

template <int D>
__global__ void __launch_bounds__(kPolWarps * 32) polar_quantize_kernel(const void* __restrict__ x, int x_f32,
                                                                        int64_t n_vec, int64_t stride, int bits,
                                                                        uint32_t* __restrict__ codes,
                                                                        uint16_t* __restrict__ radius) {
  constexpr int E = D / 32;
  constexpr int LE = E == 8 ? 3 : (E == 4 ? 2 : 1);   // in-lane levels
  constexpr int LD = LE + 5;                            // all levels: log2(D)
  __shared__ uint8_t s_idx[kPolWarps][D];
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t v = (int64_t)blockIdx.x * kPolWarps + w;
  if (v >= n_vec) return;   // whole warps only
  const float steps = (float)((1 << bits) - 1);
  float r[E];
  if (x_f32) {
    const float* xr = static_cast<const float*>(x) + v * stride + E * lane;
#pragma unroll
    for (int e = 0; e < E; ++e) r[e] = xr[e];
  } else {
    const uint16_t* xr = static_cast<const uint16_t*>(x) + v * stride + E * lane;
#pragma unroll
    for (int e = 0; e < E; ++e) r[e] = h2f(xr[e]);
  }
  uint8_t* idx = s_idx[w];
  // levels inside the lane: pair j of level L holds values 2j, 2j+1
  int cnt = E;
#pragma unroll
  for (int L = 1; L <= LE; ++L) {
#pragma unroll
    for (int j = 0; j < E / 2; ++j) {
      if (j < cnt / 2) {
        const float a = r[2 * j], b = r[2 * j + 1];
        idx[level_off<D>(L) + lane * (cnt / 2) + j] = (uint8_t)angle_code(atan2f(b, a), steps);
        r[j] = sqrtf(fmaf(a, a, b * b));
      }
    }
    cnt /= 2;
  }
  // levels across lanes: lane pairs (l, l + s), s = 1, 2, 4, 8, 16
  float rr = r[0];
#pragma unroll
  for (int s = 1, L = LE + 1; s < 32; s <<= 1, ++L) {
    const float b = __shfl_down_sync(kFull, rr, s);
    if ((lane & (2 * s - 1)) == 0) {
      idx[level_off<D>(L) + lane / (2 * s)] = (uint8_t)angle_code(atan2f(b, rr), steps);
      rr = sqrtf(fmaf(rr, rr, b * b));
    }
  }
  static_assert(LD >= 6, "head_dim of 64 or more");
  if (lane == 0) {
    idx[D - 1] = 0;
    radius[v] = f2h(rr);
  }
  __syncwarp();
  // pack: lane p (p < D/8) forms the nibble word of 8-code chunk p, then the
  // lanes of a 32-code group combine them as the MSE codes are combined
  uint32_t nib = 0;
  if (lane < D / 8) {
#pragma unroll
    for (int k = 0; k < 8; ++k) nib |= (uint32_t)idx[8 * lane + k] << (4 * k);
  }
  const uint32_t n1 = __shfl_sync(kFull, nib, lane + 1 < 32 ? lane + 1 : lane);
  const uint32_t n2 = __shfl_sync(kFull, nib, lane + 2 < 32 ? lane + 2 : lane);
  const uint32_t n3 = __shfl_sync(kFull, nib, lane | 3);
  if (lane < D / 8) {
    const int gi = lane >> 2, wq = lane & 3;
    uint32_t* rec = codes + v * (D * bits / 32);
    switch (bits) {
      case 4: rec[gi * 4 + wq] = nib; break;
      case 3:
        if (wq < 3) rec[gi * 3 + wq] = nib | (((n3 >> wq) & 0x11111111u) << 3);
        break;
      case 2:
        if (wq < 2) rec[gi * 2 + wq] = nib | (n2 << 2);
        break;
      default:
        if (wq == 0) rec[gi] = nib | (n1 << 1) | (n2 << 2) | (n3 << 3);
        break;
    }
  }
}

template <int D>
__global__ void __launch_bounds__(kPolWarps * 32) polar_dequantize_kernel(const uint32_t* __restrict__ codes,
                                                                          const uint16_t* __restrict__ radius,
                                                                          int64_t n_vec, int bits, void* __restrict__ out,
                                                                          int out_f32) {
  constexpr int E = D / 32;
  constexpr int LE = E == 8 ? 3 : (E == 4 ? 2 : 1);
  __shared__ float s_th[kPolWarps][D];
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t v = (int64_t)blockIdx.x * kPolWarps + w;
  if (v >= n_vec) return;
  const float step = 2.f * kPi / (float)((1 << bits) - 1);
  float* th = s_th[w];
  if (lane < D / 8) {
    const uint32_t n = load_chunk(codes + v * (D * bits / 32) + (lane >> 2) * bits, bits, lane & 3);
#pragma unroll
    for (int k = 0; k < 8; ++k) th[8 * lane + k] = (float)((n >> (4 * k)) & 0xf) * step - kPi;
  }
  __syncwarp();
  // levels across lanes, root first: the lanes of a group of 2s take the
  // parent's r cos (lower half) or r sin (upper half)
  float rr = h2f(radius[v]);
#pragma unroll
  for (int s = 16, L = LE + 5; s >= 1; s >>= 1, --L) {
    const int p = lane & ~(2 * s - 1);
    const float rp = __shfl_sync(kFull, rr, p);
    float sn, cs;
    sincosf(th[level_off<D>(L) + p / (2 * s)], &sn, &cs);
    rr = (lane & s) ? rp * sn : rp * cs;
  }
  // levels inside the lane, from level LE down to 1
  float r[E];
  r[0] = rr;
  int cnt = 1;
#pragma unroll
  for (int L = LE; L >= 1; --L) {
#pragma unroll
    for (int j = E / 2 - 1; j >= 0; --j) {
      if (j < cnt) {
        float sn, cs;
        sincosf(th[level_off<D>(L) + lane * cnt + j], &sn, &cs);
        const float pr = r[j];
        r[2 * j] = pr * cs;
        r[2 * j + 1] = pr * sn;
      }
    }
    cnt *= 2;
  }
  if (out_f32) {
    float* o = static_cast<float*>(out) + v * D + E * lane;
#pragma unroll
    for (int e = 0; e < E; ++e) o[e] = r[e];
  } else {
    uint16_t* o = static_cast<uint16_t*>(out) + v * D + E * lane;
#pragma unroll
    for (int e = 0; e < E; ++e) o[e] = f2h(r[e]);
  }
}

bool polar_shape_ok(int d, int bits) { return (d == 64 || d == 128 || d == 256) && bits >= 1 && bits <= 4; }

}  // namespace
}  // namespace tq

extern "C" int tq_polar_code_bytes(int head_dim, int bits, int64_t* code_bytes) {
  if (!code_bytes) return TQ_ERR_ARG;
  if (!tq::polar_shape_ok(head_dim, bits)) return TQ_ERR_UNSUPPORTED;
  *code_bytes = (int64_t)head_dim * bits / 8;
  return TQ_OK;
}

extern "C" int tq_polar_quantize(const void* x, int x_dtype, int64_t n_vec, int head_dim, int64_t x_row_stride,
                                 int bits, uint8_t* codes, uint16_t* radius, void* stream) {
  if (!tq::polar_shape_ok(head_dim, bits)) return TQ_ERR_UNSUPPORTED;
  if (n_vec < 0 || (x_dtype != TQ_F16 && x_dtype != TQ_F32) || x_row_stride < head_dim) return TQ_ERR_ARG;
  if (n_vec == 0) return TQ_OK;
  if (!x || !codes || !radius) return TQ_ERR_ARG;
  if (!tq::aligned16(codes) || (reinterpret_cast<uintptr_t>(radius) & 1) ||
      (reinterpret_cast<uintptr_t>(x) & (x_dtype == TQ_F32 ? 3 : 1)))
    return TQ_ERR_ALIGN;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const unsigned grid = (unsigned)((n_vec + tq::kPolWarps - 1) / tq::kPolWarps);
  const int f32 = x_dtype == TQ_F32;
  uint32_t* c = reinterpret_cast<uint32_t*>(codes);
  switch (head_dim) {
    case 64: tq::polar_quantize_kernel<64><<<grid, tq::kPolWarps * 32, 0, s>>>(x, f32, n_vec, x_row_stride, bits, c, radius); break;
    case 128: tq::polar_quantize_kernel<128><<<grid, tq::kPolWarps * 32, 0, s>>>(x, f32, n_vec, x_row_stride, bits, c, radius); break;
    default: tq::polar_quantize_kernel<256><<<grid, tq::kPolWarps * 32, 0, s>>>(x, f32, n_vec, x_row_stride, bits, c, radius); break;
  }
  return cudaGetLastError() == cudaSuccess ? TQ_OK : TQ_ERR_CUDA;
}

extern "C" int tq_polar_dequantize(const uint8_t* codes, const uint16_t* radius, int64_t n_vec, int head_dim,
                                   int bits, void* out, int out_dtype, void* stream) {
  if (!tq::polar_shape_ok(head_dim, bits)) return TQ_ERR_UNSUPPORTED;
  if (n_vec < 0 || (out_dtype != TQ_F16 && out_dtype != TQ_F32)) return TQ_ERR_ARG;
  if (n_vec == 0) return TQ_OK;
  if (!codes || !radius || !out) return TQ_ERR_ARG;
  if (!tq::aligned16(codes) || !tq::aligned16(out) || (reinterpret_cast<uintptr_t>(radius) & 1)) return TQ_ERR_ALIGN;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const unsigned grid = (unsigned)((n_vec + tq::kPolWarps - 1) / tq::kPolWarps);
  const int f32 = out_dtype == TQ_F32;
  const uint32_t* c = reinterpret_cast<const uint32_t*>(codes);
  switch (head_dim) {
    case 64: tq::polar_dequantize_kernel<64><<<grid, tq::kPolWarps * 32, 0, s>>>(c, radius, n_vec, bits, out, f32); break;
    case 128: tq::polar_dequantize_kernel<128><<<grid, tq::kPolWarps * 32, 0, s>>>(c, radius, n_vec, bits, out, f32); break;
    default: tq::polar_dequantize_kernel<256><<<grid, tq::kPolWarps * 32, 0, s>>>(c, radius, n_vec, bits, out, f32); break;
  }
  return cudaGetLastError() == cudaSuccess ? TQ_OK : TQ_ERR_CUDA;
}
