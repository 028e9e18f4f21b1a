// Quantise with the QJL residual stage (block = head_dim, no norm
// correction): the projection S r of every vector runs on tensor cores.
//
// A persistent CTA converts S once into fp16 high/low halves in shared
// memory, then loops over tiles of 64 vectors:
//   1. per vector (the same steps as the general quantise kernel): norm,
//      y = H D u, codes, fp16 norm; the residual back in the input domain,
//      r = D H (y - c) / sqrt(d), goes to shared memory as fp16 high/low
//      halves of r * 2^12 (the scale keeps the low halves normal);
//   2. S r for the tile as m16n8k16 MMAs, rows = vectors, k = coordinates,
//      columns = projection rows, from three products (hi*hi + hi*lo +
//      lo*hi) accumulated in fp32: about 22 significant bits, so a sign can
//      differ from the exact one only for |S r| far below 1e-5;
//   3. sign bits [S r >= 0] packed from warp ballots, rho = ||y - c|| as
//      fp16, stored per vector.
#include <cuda_runtime.h>

#include "tq_device.cuh"

namespace tq {
namespace {

constexpr int kQT = 256;     // threads
constexpr int kQV = 64;      // vectors per tile
constexpr float kRScale = 4096.f;

struct QjlArgs {
  const void* x;
  int64_t n_vec;
  int64_t stride;
  const float* S;
  uint32_t* codes;
  uint16_t* scales;
  uint8_t* qjl;
  uint16_t* rnorm;
  RowMap map;   // vector -> record
};

__device__ __forceinline__ uint32_t su32(const void* p) { return static_cast<uint32_t>(__cvta_generic_to_shared(p)); }

__device__ __forceinline__ void mma16816(float* c, const uint32_t* a, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// fp16 high half of v and fp16 of the remainder
__device__ __forceinline__ void split_h(float v, uint16_t& hi, uint16_t& lo) {
  hi = f2h(v);
  lo = f2h(v - h2f(hi));
}

// bit t of the low 4 bits moved to bit 2t
__device__ __forceinline__ uint32_t spread4(uint32_t x) {
  x = (x | (x << 2)) & 0x33u;
  return (x | (x << 1)) & 0x55u;
}

template <int D, bool F32>
__global__ void __launch_bounds__(kQT, 2) quantize_qjl_kernel(const CodecParams P, const QjlArgs a) {
  constexpr int LD = D + 8;        // padded row (fp16 elements): conflict-free fragment loads
  constexpr int TPV = D / 8;       // threads per vector
  constexpr int VPW = 32 / TPV;    // vectors per warp and pass
  const int m = P.m;
  extern __shared__ __align__(16) uint8_t smem[];
  uint16_t* sShi = reinterpret_cast<uint16_t*>(smem);          // [m][LD]
  uint16_t* sSlo = sShi + m * LD;                               // [m][LD]
  uint16_t* sRhi = sSlo + m * LD;                               // [kQV][LD]
  uint16_t* sRlo = sRhi + kQV * LD;                             // [kQV][LD]
  uint8_t* sBits = reinterpret_cast<uint8_t*>(sRlo + kQV * LD);  // [kQV][m/8]
  float* sRho = reinterpret_cast<float*>(sBits + kQV * 32);     // [kQV]
  __shared__ float s_cent[16], s_bnd[16];

  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  if (tid < 16) {
    s_cent[tid] = P.centroids[tid];
    s_bnd[tid] = P.bounds[tid];
  }
  for (int e = tid; e < m * D; e += kQT) {
    uint16_t hi, lo;
    split_h(a.S[e], hi, lo);
    sShi[(e / D) * LD + e % D] = hi;
    sSlo[(e / D) * LD + e % D] = lo;
  }
  __syncthreads();

  const int sub = lane % TPV, vs = lane / TPV;
  const int i0 = sub * 8;
  const uint32_t sb = sign_byte(P, i0);
  const int K = 1 << P.bits;
  const int words_per_vec = P.code_bytes / 4;
  const int64_t n_tiles = (a.n_vec + kQV - 1) / kQV;
  const int g = lane >> 2, t = lane & 3;

  for (int64_t tile = blockIdx.x; tile < n_tiles; tile += gridDim.x) {
    const int64_t v0 = tile * kQV;
    // ---- 1. codes, norm, residual per vector
    for (int lv = wid * VPW + vs; lv < kQV; lv += (kQT / 32) * VPW) {
      const int64_t v = v0 + lv;
      const bool valid = v < a.n_vec;
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
      float ss = 0.f;
#pragma unroll
      for (int r = 0; r < 8; ++r) ss = fmaf(x[r], x[r], ss);
      ss = group_sum(ss, TPV);
      const float n = sqrtf(ss);
#pragma unroll
      for (int r = 0; r < 8; ++r) x[r] = flip(x[r], (sb >> r) & 1u);
      wht8(x);
      wht_cross(x, sub, TPV);
      const float inv = n > 0.f ? 1.f / (n * sqrtf((float)D)) : 0.f;
      uint32_t nib = 0;
      float rr[8];
      float r2 = 0.f;
#pragma unroll
      for (int r = 0; r < 8; ++r) {
        const float y = x[r] * inv;
        int k = 0;
        for (int j = 0; j < K - 1; ++j) k += (y > s_bnd[j]) ? 1 : 0;
        nib |= (uint32_t)k << (4 * r);
        rr[r] = n > 0.f ? y - s_cent[k] : 0.f;
        r2 = fmaf(rr[r], rr[r], r2);
      }
      r2 = group_sum(r2, TPV);
      // back to the input domain: r = D H (y - c) / sqrt(d)
      wht8(rr);
      wht_cross(rr, sub, TPV);
      uint32_t hw[4], lw[4];
#pragma unroll
      for (int r = 0; r < 8; r += 2) {
        uint16_t h0, l0, h1, l1;
        split_h(flip(rr[r] * P.inv_sqrt_blk, (sb >> r) & 1u) * kRScale, h0, l0);
        split_h(flip(rr[r + 1] * P.inv_sqrt_blk, (sb >> (r + 1)) & 1u) * kRScale, h1, l1);
        hw[r / 2] = (uint32_t)h0 | ((uint32_t)h1 << 16);
        lw[r / 2] = (uint32_t)l0 | ((uint32_t)l1 << 16);
      }
      *reinterpret_cast<uint4*>(sRhi + lv * LD + i0) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
      *reinterpret_cast<uint4*>(sRlo + lv * LD + i0) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
      if (sub == 0) sRho[lv] = sqrtf(r2);
      // codes and the fp16 norm (one block per vector)
      const int64_t rv = valid ? map_row(a.map, v) : -1;
      if (rv >= 0 && sub == 0) a.scales[rv] = f2h(n);
      const int gi = sub >> 2, w = sub & 3;
      uint32_t* rec = a.codes + rv * words_per_vec;
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
    __syncthreads();

    // ---- 2. S r on tensor cores; warp w takes column tiles w, w+8, ...
    for (int nt = wid; nt < m / 8; nt += kQT / 32) {
      float acc[kQV / 16][4];
#pragma unroll
      for (int mt = 0; mt < kQV / 16; ++mt) acc[mt][0] = acc[mt][1] = acc[mt][2] = acc[mt][3] = 0.f;
      const uint16_t* bh = sShi + (nt * 8 + g) * LD + 2 * t;
      const uint16_t* bl = sSlo + (nt * 8 + g) * LD + 2 * t;
#pragma unroll 2
      for (int k0 = 0; k0 < D; k0 += 16) {
        const uint32_t bh0 = *reinterpret_cast<const uint32_t*>(bh + k0);
        const uint32_t bh1 = *reinterpret_cast<const uint32_t*>(bh + k0 + 8);
        const uint32_t bl0 = *reinterpret_cast<const uint32_t*>(bl + k0);
        const uint32_t bl1 = *reinterpret_cast<const uint32_t*>(bl + k0 + 8);
#pragma unroll
        for (int mt = 0; mt < kQV / 16; ++mt) {
          const uint16_t* ah = sRhi + (mt * 16 + g) * LD + k0 + 2 * t;
          const uint16_t* al = sRlo + (mt * 16 + g) * LD + k0 + 2 * t;
          const uint32_t A_h[4] = {*reinterpret_cast<const uint32_t*>(ah), *reinterpret_cast<const uint32_t*>(ah + 8 * LD),
                                   *reinterpret_cast<const uint32_t*>(ah + 8),
                                   *reinterpret_cast<const uint32_t*>(ah + 8 * LD + 8)};
          const uint32_t A_l[4] = {*reinterpret_cast<const uint32_t*>(al), *reinterpret_cast<const uint32_t*>(al + 8 * LD),
                                   *reinterpret_cast<const uint32_t*>(al + 8),
                                   *reinterpret_cast<const uint32_t*>(al + 8 * LD + 8)};
          mma16816(acc[mt], A_h, bh0, bh1);
          mma16816(acc[mt], A_h, bl0, bl1);
          mma16816(acc[mt], A_l, bh0, bh1);
        }
      }
      // signs: acc[mt][2*hr + e] is row (vector) mt*16 + 8*hr + g, column
      // (projection row) nt*8 + 2t + e; a ballot collects bit (4g + t)
#pragma unroll
      for (int mt = 0; mt < kQV / 16; ++mt)
#pragma unroll
        for (int hr = 0; hr < 2; ++hr) {
          const uint32_t b0 = __ballot_sync(kFull, acc[mt][2 * hr] >= 0.f);
          const uint32_t b1 = __ballot_sync(kFull, acc[mt][2 * hr + 1] >= 0.f);
          if (t == 0) {
            const uint32_t byte = spread4((b0 >> (4 * g)) & 0xfu) | (spread4((b1 >> (4 * g)) & 0xfu) << 1);
            sBits[(mt * 16 + 8 * hr + g) * (m / 8) + nt] = (uint8_t)byte;
          }
        }
    }
    __syncthreads();

    // ---- 3. sign bits and rho out
    const int bpv = m / 8;
    for (int e = tid; e < kQV * bpv / 4; e += kQT) {
      const int lv = (4 * e) / bpv;
      const int64_t v = v0 + lv;
      const int64_t rv = v < a.n_vec ? map_row(a.map, v) : -1;
      if (rv >= 0)
        *reinterpret_cast<uint32_t*>(a.qjl + rv * bpv + (4 * e) % bpv) = *reinterpret_cast<const uint32_t*>(sBits + 4 * e);
    }
    for (int lv = tid; lv < kQV; lv += kQT) {
      const int64_t v = v0 + lv;
      const int64_t rv = v < a.n_vec ? map_row(a.map, v) : -1;
      if (rv >= 0) a.rnorm[rv] = f2h(sRho[lv]);
    }
    __syncthreads();
  }
}

template <int D>
size_t qjl_smem(int m) {
  constexpr int LD = D + 8;
  return (size_t)2 * m * LD * 2 + (size_t)2 * kQV * LD * 2 + (size_t)kQV * 32 + (size_t)kQV * 4;
}

template <int D, bool F32>
int launch_qjl(const CodecParams& P, const QjlArgs& a, cudaStream_t st) {
  const size_t smem = qjl_smem<D>(P.m);
  auto kern = quantize_qjl_kernel<D, F32>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
    return TQ_ERR_CUDA;
  int dev = 0, sms = 152;
  if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int64_t tiles = (a.n_vec + kQV - 1) / kQV;
  const int per_sm = smem <= 110 * 1024 ? 2 : 1;
  const int grid = (int)(tiles < (int64_t)sms * per_sm ? tiles : (int64_t)sms * per_sm);
  kern<<<grid > 0 ? grid : 1, kQT, smem, st>>>(P, a);
  return cudaGetLastError() == cudaSuccess ? TQ_OK : TQ_ERR_CUDA;
}

}  // namespace

// QJL layouts without norm correction whose tables fit in shared memory.
bool quantize_qjl_eligible(const CodecParams& P) {
  if (!P.m || P.nc || P.blk != P.d) return false;
  switch (P.d) {
    case 64: return qjl_smem<64>(P.m) <= 220 * 1024;
    case 128: return qjl_smem<128>(P.m) <= 220 * 1024;
    case 256: return qjl_smem<256>(P.m) <= 220 * 1024;
    default: return false;
  }
}

int launch_quantize_qjl(const CodecParams& P, const void* x, bool f32, int64_t n_vec, int64_t stride, const float* S,
                        uint8_t* codes, uint16_t* scales, uint8_t* qjl_bits, uint16_t* qjl_rnorm, const RowMap& map,
                        cudaStream_t st) {
  QjlArgs a{x, n_vec, stride, S, reinterpret_cast<uint32_t*>(codes), scales, qjl_bits, qjl_rnorm, map};
  switch (P.d) {
    case 64: return f32 ? launch_qjl<64, true>(P, a, st) : launch_qjl<64, false>(P, a, st);
    case 128: return f32 ? launch_qjl<128, true>(P, a, st) : launch_qjl<128, false>(P, a, st);
    default: return f32 ? launch_qjl<256, true>(P, a, st) : launch_qjl<256, false>(P, a, st);
  }
}

}  // namespace tq
