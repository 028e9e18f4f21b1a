// Quantise and dequantise kernels of libtq.
//
// Thread mapping: every thread owns 8 consecutive coordinates of one vector
// (one 16-byte fp16 load), d/8 threads form a vector, 32/(d/8) vectors share
// a warp.  The Walsh-Hadamard transform runs in registers for strides 1..4
// and across lanes with shuffles for strides 8..block/2; norms and QJL
// reductions are shuffle reductions over the lanes of a block / vector.
#include <cuda_runtime.h>

#include "tq_device.cuh"

namespace tq {

bool quantize_fast_eligible(const CodecParams& P, bool f32_input);
int launch_quantize_fast(const CodecParams& P, const void* x, int64_t n_vec, int64_t stride, uint8_t* codes,
                         uint16_t* scales, const RowMap& map, cudaStream_t st);
bool quantize_qjl_eligible(const CodecParams& P);
bool quantize_qjl_tc_eligible(const CodecParams& P, bool f32_input);
int launch_quantize_qjl_tc(const CodecParams& P, const void* x, int64_t n_vec, int64_t stride, const float* S,
                           uint8_t* codes, uint16_t* scales, uint8_t* qjl_bits, uint16_t* qjl_rnorm, const RowMap& map,
                           cudaStream_t st);
int launch_quantize_qjl(const CodecParams& P, const void* x, bool f32, int64_t n_vec, int64_t stride, const float* S,
                        uint8_t* codes, uint16_t* scales, uint8_t* qjl_bits, uint16_t* qjl_rnorm, const RowMap& map,
                        cudaStream_t st);

namespace {

constexpr int kThreads = 256;

struct QuantArgs {
  const void* x;
  int64_t n_vec;
  int64_t stride;  // elements between rows
  const float* S;
  uint32_t* codes;
  uint16_t* scales;
  uint32_t* qjl;
  uint16_t* rnorm;
  RowMap map;   // vector -> record
};

// W8: one byte per code (256 levels, table in `cb`); otherwise 1..4 bits
// with the table in P.
template <int D, bool F32, bool W8>
__global__ void __launch_bounds__(kThreads) quantize_kernel(const CodecParams P, const QuantArgs a,
                                                            const Codebook8Param<W8> cb) {
  constexpr int TPV = D / 8;       // threads per vector
  constexpr int VPW = 32 / TPV;    // vectors per warp
  constexpr int NC = W8 ? 256 : 16;
  __shared__ float s_cent[NC];
  __shared__ float s_bnd[NC];
  __shared__ float s_r[kThreads / 32][VPW][D];        // QJL residual staging
  __shared__ uint32_t s_bits[kThreads / 32][VPW][kMaxQjl / 32];
  if constexpr (W8) {
    for (int k = threadIdx.x; k < NC; k += kThreads) {
      s_cent[k] = cb.c[k];
      s_bnd[k] = cb.b[k];
    }
  } else if (threadIdx.x < 16) {
    s_cent[threadIdx.x] = P.centroids[threadIdx.x];
    s_bnd[threadIdx.x] = P.bounds[threadIdx.x];
  }
  __syncthreads();

  const int lane = threadIdx.x & 31;
  const int wid = threadIdx.x >> 5;
  const int sub = lane % TPV;
  const int vs = lane / TPV;
  const int tpb = P.blk / 8;  // threads per rotation block
  const int K = 1 << P.bits;
  const int i0 = sub * 8;
  const uint32_t sb = sign_byte(P, i0);
  const int64_t nwarps = (int64_t)gridDim.x * (kThreads / 32);
  const int words_per_vec = P.code_bytes / 4;

  for (int64_t base = ((int64_t)blockIdx.x * (kThreads / 32) + wid) * VPW; base < a.n_vec;
       base += nwarps * VPW) {
    const int64_t v = base + vs;
    const bool valid = v < a.n_vec;
    const int64_t rv = valid ? map_row(a.map, v) : -1;   // output record
    float x[8];
    if (valid) {
      if (F32) {
        const float4* p = reinterpret_cast<const float4*>(static_cast<const float*>(a.x) + v * a.stride + i0);
        const float4 u0 = p[0], u1 = p[1];
        x[0] = u0.x; x[1] = u0.y; x[2] = u0.z; x[3] = u0.w;
        x[4] = u1.x; x[5] = u1.y; x[6] = u1.z; x[7] = u1.w;
      } else {
        const uint4 u = *reinterpret_cast<const uint4*>(static_cast<const __half*>(a.x) + v * a.stride + i0);
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int r = 0; r < 4; ++r) {
          const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w[r]));
          x[2 * r] = f.x;
          x[2 * r + 1] = f.y;
        }
      }
    } else {
#pragma unroll
      for (int r = 0; r < 8; ++r) x[r] = 0.f;
    }
    // S2: block norm.  S3: y = H (D u), computed unnormalised then scaled.
    float ss = 0.f;
#pragma unroll
    for (int r = 0; r < 8; ++r) ss = fmaf(x[r], x[r], ss);
    ss = group_sum(ss, tpb);
    const float n = sqrtf(ss);
#pragma unroll
    for (int r = 0; r < 8; ++r) x[r] = flip(x[r], (sb >> r) & 1u);
    wht8(x);
    wht_cross(x, sub, tpb);
    const float inv = n > 0.f ? 1.f / (n * sqrtf((float)P.blk)) : 0.f;
    // S4: code = #{k : y > beta_k}
    int code[8];
    float c[8];
    uint32_t nib = 0;          // 1..4 bits: code r in bits 4r..4r+3
    uint32_t byt[2] = {0, 0};  // 8 bits: code r in byte r
#pragma unroll
    for (int r = 0; r < 8; ++r) {
      const float y = x[r] * inv;
      x[r] = y;
      int k = 0;
      if constexpr (W8) {
        // the same count by bisection over the 255 ascending boundaries:
        // after the step of size s, k = #{j < k + s : y > beta_j} rounded
        // down to a multiple of s (indices stay <= 254)
#pragma unroll
        for (int step = 128; step >= 1; step >>= 1) k += (y > s_bnd[k + step - 1]) ? step : 0;
        byt[r >> 2] |= (uint32_t)k << (8 * (r & 3));
      } else {
        for (int j = 0; j < K - 1; ++j) k += (y > s_bnd[j]) ? 1 : 0;
        nib |= (uint32_t)k << (4 * r);
      }
      code[r] = k;
      c[r] = s_cent[k];
    }
    float scale = n;
    if (P.nc && !P.m) {  // S5: n / ||c|| (the rotation is orthonormal)
      float cn = 0.f;
#pragma unroll
      for (int r = 0; r < 8; ++r) cn = fmaf(c[r], c[r], cn);
      cn = group_sum(cn, tpb);
      scale = n > 0.f ? n / sqrtf(cn) : 0.f;
    }
    if (P.m) {  // S6: QJL residual, block == d
      float rr[8];
      float r2 = 0.f;
#pragma unroll
      for (int r = 0; r < 8; ++r) {
        rr[r] = n > 0.f ? x[r] - c[r] : 0.f;
        r2 = fmaf(rr[r], rr[r], r2);
      }
      r2 = group_sum(r2, TPV);
      const float rho = sqrtf(r2);
      // back to the input domain: r = D H (y - c)
      wht8(rr);
      wht_cross(rr, sub, TPV);
#pragma unroll
      for (int r = 0; r < 8; ++r) s_r[wid][vs][i0 + r] = flip(rr[r] * P.inv_sqrt_blk, (sb >> r) & 1u);
      __syncwarp();
      uint32_t word = 0;
      for (int j = 0; j < P.m / TPV; ++j) {
        const int row = TPV * j + sub;
        const float* srow = a.S + (int64_t)row * D;
        float dot = 0.f;
        for (int k = 0; k < D; ++k) dot = fmaf(__ldg(srow + k), s_r[wid][vs][k], dot);
        const uint32_t bal = __ballot_sync(kFull, dot >= 0.f);
        const uint32_t mine = TPV == 32 ? bal : (bal >> (vs * TPV)) & ((1u << (TPV & 31)) - 1u);
        word |= mine << ((TPV * j) & 31);
        if (((TPV * (j + 1)) & 31) == 0) {
          if (sub == 0) s_bits[wid][vs][(TPV * j) >> 5] = word;
          word = 0;
        }
      }
      __syncwarp();
      if (rv >= 0 && sub < P.m / 32) a.qjl[rv * (P.m / 32) + sub] = s_bits[wid][vs][sub];
      const float rho16 = __half2float(__float2half_rn(rho));
      if (rv >= 0 && sub == 0) a.rnorm[rv] = f2h(rho);
      if (P.nc) {  // renormalise the QJL-corrected direction
        float u[8];
#pragma unroll
        for (int r = 0; r < 8; ++r) u[r] = c[r];
        wht8(u);
        wht_cross(u, sub, TPV);
        const float coef = rho16 * kSqrtHalfPi / (float)P.m;
        float t2 = 0.f;
#pragma unroll
        for (int r = 0; r < 8; ++r) {
          float corr = 0.f;
          for (int i = 0; i < P.m; ++i) {
            const float sgn = ((s_bits[wid][vs][i >> 5] >> (i & 31)) & 1u) ? 1.f : -1.f;
            corr = fmaf(sgn, __ldg(a.S + (int64_t)i * D + i0 + r), corr);
          }
          const float e = flip(u[r] * P.inv_sqrt_blk, (sb >> r) & 1u) + coef * corr;
          t2 = fmaf(e, e, t2);
        }
        t2 = group_sum(t2, TPV);
        scale = n > 0.f ? n / sqrtf(t2) : 0.f;
      }
      __syncwarp();
    }
    // S7: pack and store
    if (rv >= 0 && (sub % tpb) == 0) a.scales[rv * P.nb + sub / tpb] = f2h(scale);
    uint32_t* rec = a.codes + rv * words_per_vec;
    if constexpr (W8) {   // bytes 8 sub .. 8 sub + 7 of the record
      if (rv >= 0) *reinterpret_cast<uint2*>(rec + 2 * sub) = make_uint2(byt[0], byt[1]);
      continue;
    }
    const int gi = sub >> 2, w = sub & 3;
    const uint32_t n1 = __shfl_sync(kFull, nib, lane + 1 < 32 ? lane + 1 : lane);
    const uint32_t n2 = __shfl_sync(kFull, nib, lane + 2 < 32 ? lane + 2 : lane);
    const uint32_t n3 = __shfl_sync(kFull, nib, lane | 3);
    if (rv >= 0) {
      switch (P.bits) {
        case 4: rec[gi * 4 + w] = nib; break;
        case 3:
          if (w < 3) rec[gi * 3 + w] = nib | (((n3 >> w) & 0x11111111u) << 3);
          break;
        case 2:
          if (w < 2) rec[gi * 2 + w] = nib | (n2 << 2);
          break;
        default:
          if (w == 0) rec[gi] = nib | (n1 << 1) | (n2 << 2) | (n3 << 3);
          break;
      }
    }
  }
}

struct DequantArgs {
  const uint32_t* codes;
  const uint16_t* scales;
  const uint32_t* qjl;
  const uint16_t* rnorm;
  const float* S;
  int64_t n_vec;
  void* out;
};

template <int D, bool F32, bool W8>
__global__ void __launch_bounds__(kThreads) dequantize_kernel(const CodecParams P, const DequantArgs a,
                                                              const Codebook8Param<W8> cb) {
  constexpr int TPV = D / 8;
  constexpr int VPW = 32 / TPV;
  __shared__ float s_cent[W8 ? 256 : 16];
  if constexpr (W8) {
    for (int k = threadIdx.x; k < 256; k += kThreads) s_cent[k] = cb.c[k];
  } else if (threadIdx.x < 16) {
    s_cent[threadIdx.x] = P.centroids[threadIdx.x];
  }
  __syncthreads();
  const int lane = threadIdx.x & 31;
  const int wid = threadIdx.x >> 5;
  const int sub = lane % TPV;
  const int vs = lane / TPV;
  const int tpb = P.blk / 8;
  const int i0 = sub * 8;
  const uint32_t sb = sign_byte(P, i0);
  const int64_t nwarps = (int64_t)gridDim.x * (kThreads / 32);
  const int words_per_vec = P.code_bytes / 4;
  const int64_t step = nwarps * VPW;
  // the packed words a thread's chunk needs: word wi of its group, and for the
  // fourth 3-bit chunk (bit 3 of every nibble) words 0..2
  const int w = sub & 3;
  const int wi = P.bits == 4 ? w : P.bits == 3 ? (w < 3 ? w : 0) : P.bits == 2 ? (w & 1) : 0;
  const bool three = P.bits == 3 && w == 3;
  // kBatch iterations at a time: every load of the batch is issued before the
  // first decode, so a warp keeps kBatch vector pairs of reads in flight
  constexpr int kBatch = D >= 256 ? 2 : 4;
  for (int64_t base = ((int64_t)blockIdx.x * (kThreads / 32) + wid) * VPW; base < a.n_vec;
       base += kBatch * step) {
    uint32_t r0[kBatch], r1[kBatch], r2[kBatch], sc16[kBatch];
#pragma unroll
    for (int k = 0; k < kBatch; ++k) {
      const int64_t v = base + k * step + vs;
      r0[k] = r1[k] = r2[k] = sc16[k] = 0;
      if (v < a.n_vec) {
        if constexpr (W8) {
          const uint32_t* g = a.codes + v * words_per_vec + 2 * sub;
          r0[k] = __ldg(g);
          r1[k] = __ldg(g + 1);
        } else {
          const uint32_t* g = a.codes + v * words_per_vec + (sub >> 2) * P.bits;
          r0[k] = __ldg(g + wi);
          if (three) {
            r1[k] = __ldg(g + 1);
            r2[k] = __ldg(g + 2);
          }
        }
        sc16[k] = __ldg(a.scales + v * P.nb + sub / tpb);
      }
    }
#pragma unroll
    for (int k = 0; k < kBatch; ++k) {
      const int64_t v = base + k * step + vs;
      if (base + k * step >= a.n_vec) break;   // the warp's vectors of this and later iterations are all past the end
      const bool valid = v < a.n_vec;
      float x[8];
      if constexpr (W8) {   // bytes 8 sub .. 8 sub + 7 of the record
#pragma unroll
        for (int r = 0; r < 8; ++r) x[r] = s_cent[((r < 4 ? r0[k] : r1[k]) >> (8 * (r & 3))) & 0xff];
      } else {
        uint32_t nib;
        if (three)
          nib = ((r0[k] >> 3) & 0x11111111u) | ((r1[k] >> 2) & 0x22222222u) | ((r2[k] >> 1) & 0x44444444u);
        else if (P.bits == 4)
          nib = r0[k];
        else if (P.bits == 3)
          nib = r0[k] & 0x77777777u;
        else if (P.bits == 2)
          nib = w < 2 ? (r0[k] & 0x33333333u) : ((r0[k] >> 2) & 0x33333333u);
        else
          nib = (r0[k] >> w) & 0x11111111u;
#pragma unroll
        for (int r = 0; r < 8; ++r) x[r] = s_cent[(nib >> (4 * r)) & 0xf];
      }
      wht8(x);
      wht_cross(x, sub, tpb);
#pragma unroll
      for (int r = 0; r < 8; ++r) x[r] = flip(x[r] * P.inv_sqrt_blk, (sb >> r) & 1u);
      if (P.m && valid) {
        const float coef = h2f(a.rnorm[v]) * kSqrtHalfPi / (float)P.m;
        const uint32_t* bits = a.qjl + v * (P.m / 32);
#pragma unroll
        for (int r = 0; r < 8; ++r) {
          float corr = 0.f;
          for (int i = 0; i < P.m; ++i) {
            const float sgn = ((__ldg(bits + (i >> 5)) >> (i & 31)) & 1u) ? 1.f : -1.f;
            corr = fmaf(sgn, __ldg(a.S + (int64_t)i * D + i0 + r), corr);
          }
          x[r] = fmaf(coef, corr, x[r]);
        }
      }
      if (valid) {
        const float sc = h2f((uint16_t)sc16[k]);
        if (F32) {
          float4* o = reinterpret_cast<float4*>(static_cast<float*>(a.out) + v * D + i0);
          o[0] = make_float4(x[0] * sc, x[1] * sc, x[2] * sc, x[3] * sc);
          o[1] = make_float4(x[4] * sc, x[5] * sc, x[6] * sc, x[7] * sc);
        } else {
          uint32_t wv[4];
#pragma unroll
          for (int r = 0; r < 4; ++r) {
            const __half2 h = __floats2half2_rn(x[2 * r] * sc, x[2 * r + 1] * sc);
            wv[r] = *reinterpret_cast<const uint32_t*>(&h);
          }
          *reinterpret_cast<uint4*>(static_cast<__half*>(a.out) + v * D + i0) = make_uint4(wv[0], wv[1], wv[2], wv[3]);
        }
      }
    }
  }
}

int grid_for(int64_t n_vec, int vpw) {
  int dev = 0, sms = 152;
  if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int64_t warps = (n_vec + vpw - 1) / vpw;
  const int64_t blocks = (warps + kThreads / 32 - 1) / (kThreads / 32);
  const int64_t cap = (int64_t)sms * 8;
  return (int)(blocks < cap ? (blocks > 0 ? blocks : 1) : cap);
}

// cb8: the 256-level table when P.bits == 8, else unused
template <int D>
int launch_quantize(const CodecParams& P, const QuantArgs& a, bool f32, const Codebook8& cb8, cudaStream_t st) {
  const int g = grid_for(a.n_vec, 32 / (D / 8));
  const NoCodebook8 none{};
  if (P.bits == 8) {
    if (f32) quantize_kernel<D, true, true><<<g, kThreads, 0, st>>>(P, a, cb8);
    else quantize_kernel<D, false, true><<<g, kThreads, 0, st>>>(P, a, cb8);
  } else {
    if (f32) quantize_kernel<D, true, false><<<g, kThreads, 0, st>>>(P, a, none);
    else quantize_kernel<D, false, false><<<g, kThreads, 0, st>>>(P, a, none);
  }
  return cudaGetLastError() == cudaSuccess ? TQ_OK : TQ_ERR_CUDA;
}

template <int D>
int launch_dequantize(const CodecParams& P, const DequantArgs& a, bool f32, const Codebook8& cb8, cudaStream_t st) {
  const int g = grid_for(a.n_vec, 32 / (D / 8));
  const NoCodebook8 none{};
  if (P.bits == 8) {
    if (f32) dequantize_kernel<D, true, true><<<g, kThreads, 0, st>>>(P, a, cb8);
    else dequantize_kernel<D, false, true><<<g, kThreads, 0, st>>>(P, a, cb8);
  } else {
    if (f32) dequantize_kernel<D, true, false><<<g, kThreads, 0, st>>>(P, a, none);
    else dequantize_kernel<D, false, false><<<g, kThreads, 0, st>>>(P, a, none);
  }
  return cudaGetLastError() == cudaSuccess ? TQ_OK : TQ_ERR_CUDA;
}

}  // namespace
}  // namespace tq

namespace tq {
namespace {

// tq_quantize_kv and tq_append_kv: checks, then the fastest eligible kernel.
int quantize_common(const tq_layout* layout, const void* x, tq_dtype x_dtype, int64_t n_vec, int64_t x_row_stride,
                    const float* S, uint8_t* codes, uint16_t* scales, uint8_t* qjl_bits, uint16_t* qjl_rnorm,
                    const RowMap& map, void* stream) {
  CodecParams P;
  int st = make_params(layout, &P);
  if (st != TQ_OK) return st;
  if (x_dtype != TQ_F16 && x_dtype != TQ_F32) return TQ_ERR_ARG;
  if (n_vec < 0 || x_row_stride < P.d) return TQ_ERR_ARG;
  if (n_vec == 0) return TQ_OK;
  if (!x || !codes || !scales) return TQ_ERR_ARG;
  if (P.m && (!S || !qjl_bits || !qjl_rnorm)) return TQ_ERR_ARG;
  const int esz = x_dtype == TQ_F32 ? 4 : 2;
  if (!aligned16(x) || (x_row_stride * esz) % 16 || !aligned16(codes) || !aligned16(scales)) return TQ_ERR_ALIGN;
  if (P.m && (!aligned16(S) || !aligned16(qjl_bits) || !aligned16(qjl_rnorm))) return TQ_ERR_ALIGN;
  QuantArgs a{x, n_vec, x_row_stride, S, reinterpret_cast<uint32_t*>(codes), scales,
              reinterpret_cast<uint32_t*>(qjl_bits), qjl_rnorm, map};
  Codebook8 cb8;
  if (P.bits == 8 && make_codebook8(layout, &cb8) != TQ_OK) return TQ_ERR_UNSUPPORTED;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const bool f32 = x_dtype == TQ_F32;
  if (quantize_fast_eligible(P, f32)) {
    // TQ_ERR_UNSUPPORTED: the input cannot be described to the tensor-memory
    // loads (e.g. 2^32 rows or more); the general kernel takes it
    const int fst = launch_quantize_fast(P, x, n_vec, x_row_stride, codes, scales, map, s);
    if (fst != TQ_ERR_UNSUPPORTED) return fst;
  }
  if (quantize_qjl_tc_eligible(P, f32)) {
    // TQ_ERR_UNSUPPORTED: more rows than the tensor-memory loads describe
    const int qst = launch_quantize_qjl_tc(P, x, n_vec, x_row_stride, S, codes, scales, qjl_bits, qjl_rnorm, map, s);
    if (qst != TQ_ERR_UNSUPPORTED) return qst;
  }
  if (quantize_qjl_eligible(P))
    return launch_quantize_qjl(P, x, f32, n_vec, x_row_stride, S, codes, scales, qjl_bits, qjl_rnorm, map, s);
  switch (P.d) {
    case 64: return launch_quantize<64>(P, a, f32, cb8, s);
    case 128: return launch_quantize<128>(P, a, f32, cb8, s);
    default: return launch_quantize<256>(P, a, f32, cb8, s);
  }
}

}  // namespace
}  // namespace tq

extern "C" int tq_quantize_kv(const tq_layout* layout, const void* x, tq_dtype x_dtype, int64_t n_vec,
                              int64_t x_row_stride, const float* S, uint8_t* codes, uint16_t* scales,
                              uint8_t* qjl_bits, uint16_t* qjl_rnorm, void* stream) {
  const tq::RowMap identity{nullptr, 1, 1, 0, {nullptr, 0, 0}};
  return tq::quantize_common(layout, x, x_dtype, n_vec, x_row_stride, S, codes, scales, qjl_bits, qjl_rnorm,
                             identity, stream);
}

extern "C" int tq_append_kv(const tq_layout* layout, const void* x, tq_dtype x_dtype, int B, int H, int n_new,
                            int64_t x_row_stride, const int32_t* pos, int64_t S_cap, const int32_t* page_table,
                            int page_size, int pages_per_seq, const float* S, uint8_t* codes, uint16_t* scales,
                            uint8_t* qjl_bits, uint16_t* qjl_rnorm, void* stream) {
  if (B < 0 || H < 0 || n_new < 0 || S_cap < 0) return TQ_ERR_ARG;
  if ((int64_t)B * H * n_new == 0) return TQ_OK;
  if (!pos || S_cap == 0) return TQ_ERR_ARG;
  if (page_table && (page_size <= 0 || page_size % 32 || pages_per_seq <= 0 ||
                     (int64_t)page_size * pages_per_seq < S_cap))
    return TQ_ERR_ARG;
  const tq::RowMap map{pos, n_new, H, S_cap, {page_table, page_table ? page_size : 0, page_table ? pages_per_seq : 0}};
  return tq::quantize_common(layout, x, x_dtype, (int64_t)B * H * n_new, x_row_stride, S, codes, scales, qjl_bits,
                             qjl_rnorm, map, stream);
}

extern "C" int tq_dequantize_kv(const tq_layout* layout, const uint8_t* codes, const uint16_t* scales,
                                const uint8_t* qjl_bits, const uint16_t* qjl_rnorm, const float* S,
                                int64_t n_vec, void* out, tq_dtype out_dtype, void* stream) {
  tq::CodecParams P;
  int st = tq::make_params(layout, &P);
  if (st != TQ_OK) return st;
  if (out_dtype != TQ_F16 && out_dtype != TQ_F32) return TQ_ERR_ARG;
  if (n_vec < 0) return TQ_ERR_ARG;
  if (n_vec == 0) return TQ_OK;
  if (!codes || !scales || !out) return TQ_ERR_ARG;
  if (P.m && (!S || !qjl_bits || !qjl_rnorm)) return TQ_ERR_ARG;
  if (!tq::aligned16(codes) || !tq::aligned16(scales) || !tq::aligned16(out)) return TQ_ERR_ALIGN;
  tq::DequantArgs a{reinterpret_cast<const uint32_t*>(codes), scales,
                    reinterpret_cast<const uint32_t*>(qjl_bits), qjl_rnorm, S, n_vec, out};
  tq::Codebook8 cb8;
  if (P.bits == 8 && tq::make_codebook8(layout, &cb8) != TQ_OK) return TQ_ERR_UNSUPPORTED;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const bool f32 = out_dtype == TQ_F32;
  switch (P.d) {
    case 64: return tq::launch_dequantize<64>(P, a, f32, cb8, s);
    case 128: return tq::launch_dequantize<128>(P, a, f32, cb8, s);
    default: return tq::launch_dequantize<256>(P, a, f32, cb8, s);
  }
}
