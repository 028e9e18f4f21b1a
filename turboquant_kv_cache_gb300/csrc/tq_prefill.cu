// Prefill attention over the packed cache: Tq queries per (batch, q-head),
// causal, on tensor cores over K/V tiles decoded into shared memory.
//
// Every (batch, KV head) owns Tq*G query rows (query i, head h -> row
// i*G + h).  A CTA takes 64 rows (16 per warp) and walks the context in
// 64-token tiles: the tile's K and V are decoded cooperatively into shared
// memory in the rotated domain (centroid * block scale, fp16), QK^T and PV
// run as m16n8k16 fp16 MMAs with fp32 accumulation and an fp32 online
// softmax, and the output is rotated back (D H per V block) once at the end.
// The query is rotated once by K's D and H ("llama.cpp-turboquant", "Fused
// tile path": <Hc, q> = <c, Hq>; V accumulated rotated, H applied once).
#include <cuda_runtime.h>
#include <math.h>

#include "tq_device.cuh"

namespace tq {
namespace {

constexpr int kPfWarps = 4;
constexpr int kPfThreads = kPfWarps * 32;
constexpr int kRows = 16 * kPfWarps;  // query rows per CTA
constexpr int kTile = 64;             // tokens per KV tile

struct PrefillArgs {
  const uint32_t* kc;
  const uint16_t* ks;
  const uint32_t* vc;
  const uint16_t* vs;
  const uint16_t* q;
  uint16_t* out;
  int64_t S_cap, ctx;
  int Hq, Hkv, Tq, causal;
  float qscale;
};

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void ldsm_x4(uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3, const void* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(smem_u32(p)));
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3, const void* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(smem_u32(p)));
}

__device__ __forceinline__ void mma16816(float* c, uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                                         uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t pack_h2(float lo, float hi) {
  const __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}

// Decode one tile of `kTile` tokens of a packed cache into smem rows
// [token][D + 8] fp16 (rotated domain, times the block scale).
template <int D>
__device__ void decode_tile(const CodecParams& P, const uint32_t* __restrict__ codes,
                            const uint16_t* __restrict__ scales, int64_t rec0, int64_t t0, int64_t t_lim,
                            const float* cent, __half* dst) {
  constexpr int CH = D / 8;  // 8-code chunks per token
  const int words = P.code_bytes / 4;
  for (int task = threadIdx.x; task < kTile * CH; task += kPfThreads) {
    const int tok = task / CH, ch = task % CH;
    const int64_t t = t0 + tok;
    uint4 packed = make_uint4(0, 0, 0, 0);
    if (t < t_lim) {
      const uint32_t* rec = codes + (rec0 + t) * words;
      const uint32_t nib = load_chunk(rec + (ch >> 2) * P.bits, P.bits, ch & 3);
      const float sc = h2f(scales[(rec0 + t) * P.nb + (ch * 8) / P.blk]);
      packed.x = pack_h2(cent[nib & 0xf] * sc, cent[(nib >> 4) & 0xf] * sc);
      packed.y = pack_h2(cent[(nib >> 8) & 0xf] * sc, cent[(nib >> 12) & 0xf] * sc);
      packed.z = pack_h2(cent[(nib >> 16) & 0xf] * sc, cent[(nib >> 20) & 0xf] * sc);
      packed.w = pack_h2(cent[(nib >> 24) & 0xf] * sc, cent[(nib >> 28) & 0xf] * sc);
    }
    *reinterpret_cast<uint4*>(dst + tok * (D + 8) + ch * 8) = packed;
  }
}

template <int D>
__global__ void __launch_bounds__(kPfThreads) prefill_kernel(const CodecParams PK, const CodecParams PV,
                                                             const PrefillArgs a) {
  extern __shared__ __align__(16) unsigned char smem[];
  __half* sQ = reinterpret_cast<__half*>(smem);                     // [kRows][D+8]
  __half* sK = sQ + kRows * (D + 8);                                // [kTile][D+8]
  __half* sV = sK + kTile * (D + 8);                                // [kTile][D+8]
  float* sF = reinterpret_cast<float*>(sV + kTile * (D + 8));       // [kRows][D] fp32 staging
  __shared__ float s_centK[16], s_centV[16];

  const int G = a.Hq / a.Hkv;
  const int bh = blockIdx.y;
  const int b = bh / a.Hkv, kvh = bh % a.Hkv;
  const int row0 = blockIdx.x * kRows;
  const int n_rows = a.Tq * G;
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const int g = lane >> 2, t = lane & 3;

  if (threadIdx.x < 16) {
    s_centK[threadIdx.x] = PK.centroids[threadIdx.x];
    s_centV[threadIdx.x] = PV.centroids[threadIdx.x];
  }
  // q rows -> rotate by K's D and H per block -> scale -> fp16
  for (int e = threadIdx.x; e < kRows * D; e += kPfThreads) {
    const int r = e / D, i = e % D;
    const int row = row0 + r;
    float v = 0.f;
    if (row < n_rows) {
      const int qi = row / G, h = kvh * G + row % G;
      v = h2f(a.q[(((int64_t)b * a.Hq + h) * a.Tq + qi) * D + i]);
      if ((PK.sign_bits[i >> 5] >> (i & 31)) & 1u) v = -v;
    }
    sF[e] = v;
  }
  for (int h = 1; h < PK.blk; h <<= 1) {
    __syncthreads();
    for (int e = threadIdx.x; e < kRows * D / 2; e += kPfThreads) {
      const int r = e / (D / 2), k = e % (D / 2);
      const int i = (k / h) * 2 * h + (k % h);
      float* rr = sF + r * D;
      const float x = rr[i], y = rr[i + h];
      rr[i] = x + y;
      rr[i + h] = x - y;
    }
  }
  __syncthreads();
  const float qn = PK.inv_sqrt_blk * a.qscale;
  for (int e = threadIdx.x; e < kRows * D; e += kPfThreads) {
    const int r = e / D, i = e % D;
    sQ[r * (D + 8) + i] = __float2half_rn(sF[e] * qn);
  }
  __syncthreads();

  // rows of this lane: warp rows wid*16 + g and + 8
  int pos[2];
#pragma unroll
  for (int hr = 0; hr < 2; ++hr) {
    const int row = row0 + wid * 16 + g + 8 * hr;
    const int qi = row < n_rows ? row / G : a.Tq - 1;
    pos[hr] = (int)(a.ctx - a.Tq + qi);
  }
  int max_pos = (int)(a.ctx - 1);
  if (a.causal) {
    const int last_row = min(row0 + kRows, n_rows) - 1;
    max_pos = (int)(a.ctx - a.Tq + last_row / G);
  }
  const int64_t t_lim = a.ctx;

  constexpr int NT = D / 8;   // n-tiles of the output
  float o[NT][4];
#pragma unroll
  for (int n = 0; n < NT; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
  float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.f, 0.f};
  const int64_t rec0 = (int64_t)bh * a.S_cap;

  for (int64_t t0 = 0; t0 <= max_pos; t0 += kTile) {
    __syncthreads();
    decode_tile<D>(PK, a.kc, a.ks, rec0, t0, t_lim, s_centK, sK);
    decode_tile<D>(PV, a.vc, a.vs, rec0, t0, t_lim, s_centV, sV);
    __syncthreads();
    // S = Q K^T for this warp's 16 rows x 64 tokens
    float s[kTile / 8][4];
#pragma unroll
    for (int n = 0; n < kTile / 8; ++n) s[n][0] = s[n][1] = s[n][2] = s[n][3] = 0.f;
    const __half* qbase = sQ + (wid * 16) * (D + 8);
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
      uint32_t a0, a1, a2, a3;
      ldsm_x4(a0, a1, a2, a3, qbase + (lane & 15) * (D + 8) + kk * 16 + (lane >> 4) * 8);
#pragma unroll
      for (int n = 0; n < kTile / 8; n += 2) {
        uint32_t b0, b1, b2, b3;
        // matrices: (tokens n*8..+7, k 0-7), (same, k 8-15), (tokens +8, k 0-7), (tokens +8, k 8-15)
        const int tok = n * 8 + (lane & 7) + ((lane >> 4) << 3);
        const int kof = kk * 16 + ((lane >> 3) & 1) * 8;
        ldsm_x4(b0, b1, b2, b3, sK + tok * (D + 8) + kof);
        mma16816(s[n], a0, a1, a2, a3, b0, b1);
        mma16816(s[n + 1], a0, a1, a2, a3, b2, b3);
      }
    }
    // mask + online softmax (base 2); rows g (regs 0,1) and g+8 (regs 2,3)
    float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
    for (int n = 0; n < kTile / 8; ++n)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int hr = e >> 1;
        const int64_t tok = t0 + n * 8 + 2 * t + (e & 1);
        const bool ok = tok < t_lim && (!a.causal || tok <= pos[hr]);
        s[n][e] = ok ? s[n][e] : -INFINITY;
        mx[hr] = fmaxf(mx[hr], s[n][e]);
      }
    float alpha[2], mnew[2];
#pragma unroll
    for (int hr = 0; hr < 2; ++hr) {
      mx[hr] = fmaxf(mx[hr], __shfl_xor_sync(kFull, mx[hr], 1));
      mx[hr] = fmaxf(mx[hr], __shfl_xor_sync(kFull, mx[hr], 2));
      mnew[hr] = fmaxf(m_run[hr], mx[hr]);
      alpha[hr] = (m_run[hr] == -INFINITY) ? 0.f : exp2f(m_run[hr] - mnew[hr]);
      m_run[hr] = mnew[hr];
    }
    float rs[2] = {0.f, 0.f};
    uint32_t pa[kTile / 16][4];
#pragma unroll
    for (int n = 0; n < kTile / 8; ++n) {
      float p[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int hr = e >> 1;
        p[e] = (mnew[hr] == -INFINITY) ? 0.f : exp2f(s[n][e] - mnew[hr]);
        rs[hr] += p[e];
      }
      // C layout of n-tile n -> A fragment of k-tile n/2
      const int kt = n >> 1;
      if ((n & 1) == 0) {
        pa[kt][0] = pack_h2(p[0], p[1]);
        pa[kt][1] = pack_h2(p[2], p[3]);
      } else {
        pa[kt][2] = pack_h2(p[0], p[1]);
        pa[kt][3] = pack_h2(p[2], p[3]);
      }
    }
#pragma unroll
    for (int hr = 0; hr < 2; ++hr) {
      rs[hr] += __shfl_xor_sync(kFull, rs[hr], 1);
      rs[hr] += __shfl_xor_sync(kFull, rs[hr], 2);
      l_run[hr] = l_run[hr] * alpha[hr] + rs[hr];
    }
#pragma unroll
    for (int n = 0; n < NT; ++n) {
      o[n][0] *= alpha[0];
      o[n][1] *= alpha[0];
      o[n][2] *= alpha[1];
      o[n][3] *= alpha[1];
    }
    // O += P V
#pragma unroll
    for (int kt = 0; kt < kTile / 16; ++kt) {
#pragma unroll
      for (int n = 0; n < NT; n += 2) {
        uint32_t b0, b1, b2, b3;
        // matrices: (tokens kt*16+0..7, coords n*8..), (tokens +8, same), (tokens 0..7, coords +8), (tokens +8, +8)
        const int tok = kt * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
        const int col = n * 8 + (lane >> 4) * 8;
        ldsm_x4_t(b0, b1, b2, b3, sV + tok * (D + 8) + col);
        mma16816(o[n], pa[kt][0], pa[kt][1], pa[kt][2], pa[kt][3], b0, b1);
        mma16816(o[n + 1], pa[kt][0], pa[kt][1], pa[kt][2], pa[kt][3], b2, b3);
      }
    }
  }
  // normalise, rotate back per V block, store
  __syncthreads();
#pragma unroll
  for (int hr = 0; hr < 2; ++hr) {
    const float inv = l_run[hr] > 0.f ? 1.f / l_run[hr] : 0.f;
    const int r = wid * 16 + g + 8 * hr;
#pragma unroll
    for (int n = 0; n < NT; ++n) {
      sF[r * D + n * 8 + 2 * t] = o[n][2 * hr] * inv;
      sF[r * D + n * 8 + 2 * t + 1] = o[n][2 * hr + 1] * inv;
    }
  }
  for (int h = 1; h < PV.blk; h <<= 1) {
    __syncthreads();
    for (int e = threadIdx.x; e < kRows * D / 2; e += kPfThreads) {
      const int r = e / (D / 2), k = e % (D / 2);
      const int i = (k / h) * 2 * h + (k % h);
      float* rr = sF + r * D;
      const float x = rr[i], y = rr[i + h];
      rr[i] = x + y;
      rr[i + h] = x - y;
    }
  }
  __syncthreads();
  for (int e = threadIdx.x; e < kRows * D; e += kPfThreads) {
    const int r = e / D, i = e % D;
    const int row = row0 + r;
    if (row >= n_rows) continue;
    const int qi = row / G, h = kvh * G + row % G;
    const float v = flip(sF[e] * PV.inv_sqrt_blk, (PV.sign_bits[i >> 5] >> (i & 31)) & 1u);
    a.out[(((int64_t)b * a.Hq + h) * a.Tq + qi) * D + i] = f2h(v);
  }
}

template <int D>
size_t prefill_smem() {
  return (size_t)(kRows + 2 * kTile) * (D + 8) * sizeof(__half) + (size_t)kRows * D * sizeof(float);
}

template <int D>
int launch_prefill(const CodecParams& PK, const CodecParams& PV, const PrefillArgs& a, int B, cudaStream_t st) {
  const size_t smem = prefill_smem<D>();
  if (cudaFuncSetAttribute(prefill_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
      cudaSuccess)
    return TQ_ERR_CUDA;
  const int rows = a.Tq * (a.Hq / a.Hkv);
  dim3 grid((rows + kRows - 1) / kRows, B * a.Hkv);
  prefill_kernel<D><<<grid, kPfThreads, smem, st>>>(PK, PV, a);
  return cudaGetLastError() == cudaSuccess ? TQ_OK : TQ_ERR_CUDA;
}

}  // namespace
}  // namespace tq

extern "C" int tq_prefill_workspace_bytes(int B, int Hq, int Hkv, int head_dim, int Tq, int64_t ctx,
                                          size_t* bytes) {
  if (B <= 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv || Tq < 0 || ctx < Tq || !bytes) return TQ_ERR_ARG;
  if (head_dim != 64 && head_dim != 128 && head_dim != 256) return TQ_ERR_UNSUPPORTED;
  *bytes = 0;
  return TQ_OK;
}

extern "C" int tq_prefill_attn(const tq_kv_view* K, const tq_kv_view* V, const uint16_t* q, int B, int Hq, int Hkv,
                               int Tq, int64_t S_cap, int64_t ctx, int causal, float softmax_scale, uint16_t* out,
                               void* workspace, size_t workspace_bytes, void* stream) {
  (void)workspace;
  (void)workspace_bytes;
  if (!K || !V || !q || !out) return TQ_ERR_ARG;
  tq::CodecParams PK, PV;
  int st = tq::make_params(&K->layout, &PK);
  if (st != TQ_OK) return st;
  st = tq::make_params(&V->layout, &PV);
  if (st != TQ_OK) return st;
  if (PK.d != PV.d || PK.m || PV.m) return TQ_ERR_UNSUPPORTED;
  if (B <= 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv || Tq < 0 || ctx < Tq || ctx > S_cap) return TQ_ERR_ARG;
  if (!K->codes || !K->scales || !V->codes || !V->scales) return TQ_ERR_ARG;
  if (!tq::aligned16(K->codes) || !tq::aligned16(V->codes) || !tq::aligned16(q) || !tq::aligned16(out))
    return TQ_ERR_ALIGN;
  if (Tq == 0) return TQ_OK;
  const float sm = softmax_scale > 0.f ? softmax_scale : 1.0f / sqrtf((float)PK.d);
  tq::PrefillArgs a{reinterpret_cast<const uint32_t*>(K->codes), K->scales,
                    reinterpret_cast<const uint32_t*>(V->codes), V->scales, q, out, S_cap, ctx, Hq, Hkv, Tq,
                    causal ? 1 : 0, sm * tq::kLog2e};
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  switch (PK.d) {
    case 64: return tq::launch_prefill<64>(PK, PV, a, B, s);
    case 128: return tq::launch_prefill<128>(PK, PV, a, B, s);
    default: return tq::launch_prefill<256>(PK, PV, a, B, s);
  }
}
