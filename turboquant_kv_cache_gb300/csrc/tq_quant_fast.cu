// Fast quantise path: fp16 input, rotation block of 32 or 64, 2-4 bits, no
// QJL, no norm correction (those layouts use the general kernel).
//
// One thread owns one (vector, block): the whole block sits in registers, so
// the Walsh-Hadamard butterflies need no shuffles.  A warp takes 32 vectors
// at one block index j, so the sign pattern D_j is the same for every lane.
// Rows arrive through a per-warp double buffer filled by 16-byte cp.async
// (coalesced), stored with an XOR swizzle so the per-thread 16-byte reads
// are free of bank conflicts.
//
// Bucketize: code = #{k : y > beta_k}.  With a = |y| scaled by 2^20 / beta
// units, each positive boundary contributes sat(a*A - B_k) (an exact 0/1
// step except within 2^-20 of the boundary, far inside the 1e-5 tie band);
// the sign picks the half of the codebook.  The code is turned into an
// integer by adding 1.5*2^23 (round to nearest) and packed with integer
// multiply-adds.
#include <cuda_runtime.h>

#include "tq_device.cuh"

namespace tq {
namespace {

constexpr int kFW = 4;            // warps per CTA
constexpr float kStepScale = 1048576.0f;   // 2^20
constexpr float kMagic = 12582912.0f;      // 1.5 * 2^23

struct FastQuantArgs {
  const __half* x;
  int64_t n_vec;
  int64_t stride;   // elements between rows
  uint32_t* codes;  // [records][words per vector]
  uint16_t* scales;
  RowMap map;       // vector -> record
  float bstep[8];   // 2^20 * positive boundaries beta_{K/2} .. beta_{K-2}
  uint32_t sgn[128];  // fp16x2 +-1 multipliers of D, pairs (2i, 2i+1)
};

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void cp_async16(void* dst, const void* src, int bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(smem_u32(dst)), "l"(src), "r"(bytes));
}

template <int BLK>
__device__ __forceinline__ int swz(int item, int k) {
  return BLK == 64 ? (k ^ (item & 7)) : (k ^ ((item >> 1) & 3));
}

template <int BLK, int BITS>
__global__ void __launch_bounds__(kFW * 32) quantize_fast_kernel(const CodecParams P, const FastQuantArgs a) {
  constexpr int CPI = BLK / 8;               // 16-byte chunks per item
  constexpr int TILE_BYTES = 32 * BLK * 2;
  constexpr int HALF_K = (1 << BITS) / 2;    // codes per half of the codebook
  constexpr int WPB = BLK * BITS / 32;       // packed words per block
  __shared__ __align__(128) uint8_t s_buf[kFW][2][TILE_BYTES];

  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const int nb = P.nb;
  const int64_t vec_tiles = (a.n_vec + 31) / 32;
  const int64_t n_tiles = vec_tiles * nb;
  const int64_t gw = (int64_t)blockIdx.x * kFW + wid;
  const int64_t stride_w = (int64_t)gridDim.x * kFW;
  const int words_per_vec = P.code_bytes / 4;

  auto issue = [&](int64_t tile, int buf) {
    const int j = (int)(tile % nb);
    const int64_t v0 = (tile / nb) * 32;
    uint8_t* dst = s_buf[wid][buf];
#pragma unroll
    for (int r = 0; r < CPI; ++r) {
      const int c = lane + 32 * r;
      const int item = c / CPI, k = c % CPI;
      const int64_t v = v0 + item;
      const bool ok = v < a.n_vec;
      const __half* src = ok ? a.x + v * a.stride + (int64_t)j * BLK + k * 8 : a.x;
      cp_async16(dst + item * BLK * 2 + swz<BLK>(item, k) * 16, src, ok ? 16 : 0);
    }
    asm volatile("cp.async.commit_group;\n" ::);
  };

  int64_t tile = gw;
  int buf = 0;
  if (tile < n_tiles) issue(tile, 0);
  for (; tile < n_tiles; tile += stride_w, buf ^= 1) {
    const int64_t nx = tile + stride_w;
    if (nx < n_tiles) {
      issue(nx, buf ^ 1);
      asm volatile("cp.async.wait_group 1;\n" ::);
    } else {
      asm volatile("cp.async.wait_group 0;\n" ::);
    }
    __syncwarp();
    const int j = (int)(tile % nb);
    const int64_t v = (tile / nb) * 32 + lane;
    const uint8_t* src = s_buf[wid][buf] + lane * BLK * 2;

    // load, apply D, widen to fp32 pairs (2i, 2i+1)
    float2 x[BLK / 2];
    float2 ss2 = make_float2(0.f, 0.f);
#pragma unroll
    for (int k = 0; k < CPI; ++k) {
      const uint4 u = *reinterpret_cast<const uint4*>(src + swz<BLK>(lane, k) * 16);
      const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const uint32_t sg = a.sgn[(j * BLK) / 2 + 4 * k + e];
        const __half2 h = __hmul2(*reinterpret_cast<const __half2*>(&w[e]), *reinterpret_cast<const __half2*>(&sg));
        x[4 * k + e] = __half22float2(h);
        ss2 = __ffma2_rn(x[4 * k + e], x[4 * k + e], ss2);
      }
    }
    __syncwarp();   // the buffer is refilled two tiles later
    // unnormalised Walsh-Hadamard transform: stride 1 inside each pair, the
    // wider strides on whole pairs with packed fp32x2 adds
#pragma unroll
    for (int i = 0; i < BLK / 2; ++i) {
      const float p = x[i].x, q = x[i].y;
      x[i] = make_float2(p + q, p - q);
    }
    const float2 neg1 = make_float2(-1.f, -1.f);
#pragma unroll
    for (int h = 1; h < BLK / 2; h <<= 1) {
#pragma unroll
      for (int i = 0; i < BLK / 2; ++i) {
        if ((i & h) == 0) {
          const float2 p = x[i], q = x[i + h];
          x[i] = __fadd2_rn(p, q);
          x[i + h] = __ffma2_rn(q, neg1, p);
        }
      }
    }
    const float n = sqrtf(ss2.x + ss2.y);
    // a*A - B_k with A = 2^20 / (n sqrt(blk)): |y| > beta_k  <=>  step = 1
    const float A = n > 0.f ? kStepScale / (n * sqrtf((float)BLK)) : 0.f;
    const float2 base2 = make_float2((float)HALF_K - 0.5f, (float)HALF_K - 0.5f);
    const float2 magic2 = make_float2(kMagic, kMagic);
    // integer of the magic-shifted code is (bits - magic bits); the magic part
    // of all 8 nibbles is removed once per chunk
    const uint32_t magic_all = __float_as_uint(kMagic) * 0x11111111u;
    uint32_t words[WPB];
    uint32_t nib[BLK / 8];
#pragma unroll
    for (int c = 0; c < BLK / 8; ++c) {
      uint32_t acc = 0u - magic_all;
#pragma unroll
      for (int r2 = 0; r2 < 4; ++r2) {
        const float2 y = x[4 * c + r2];
        const float ay0 = fabsf(y.x), ay1 = fabsf(y.y);
        float2 cnt = make_float2(0.5f, 0.5f);
#pragma unroll
        for (int kk = 0; kk < HALF_K - 1; ++kk)
          cnt = __fadd2_rn(cnt, make_float2(__saturatef(fmaf(ay0, A, -a.bstep[kk])),
                                            __saturatef(fmaf(ay1, A, -a.bstep[kk]))));
        // code = HALF_K - 1 - cnt + 0.5 (y <= 0) or HALF_K - 0.5 + cnt (y > 0)
        const float2 sc = make_float2(copysignf(cnt.x, y.x), copysignf(cnt.y, y.y));
        // small exact sum first; adding 1.5*2^23 then rounds it to an integer
        const float2 codef = __fadd2_rn(__fadd2_rn(base2, sc), magic2);
        acc += __float_as_uint(codef.x) << (8 * r2);
        acc += __float_as_uint(codef.y) << (8 * r2 + 4);
      }
      nib[c] = n > 0.f ? acc : (uint32_t)(HALF_K - 1) * 0x11111111u;
    }
    // pack nibble chunks into the layout's words
#pragma unroll
    for (int gi = 0; gi < BLK / 32; ++gi) {
      const uint32_t* N = nib + 4 * gi;
      if (BITS == 4) {
#pragma unroll
        for (int w = 0; w < 4; ++w) words[4 * gi + w] = N[w];
      } else if (BITS == 3) {
#pragma unroll
        for (int w = 0; w < 3; ++w) words[3 * gi + w] = N[w] | (((N[3] >> w) & 0x11111111u) << 3);
      } else {
#pragma unroll
        for (int w = 0; w < 2; ++w) words[2 * gi + w] = N[w] | (N[w + 2] << 2);
      }
    }
    const int64_t r = v < a.n_vec ? map_row(a.map, v) : -1;
    if (r >= 0) {
      uint32_t* dst = a.codes + r * words_per_vec + j * WPB;
#pragma unroll
      for (int w = 0; w < WPB; ++w) dst[w] = words[w];
      a.scales[r * nb + j] = f2h(n);
    }
  }
}

template <int BLK, int BITS>
int launch_fast(const CodecParams& P, const FastQuantArgs& a, cudaStream_t st) {
  int dev = 0, sms = 152;
  if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int64_t tiles = (a.n_vec + 31) / 32 * P.nb;
  int64_t blocks = (tiles + kFW - 1) / kFW;
  const int64_t cap = (int64_t)sms * 8;
  if (blocks > cap) blocks = cap;
  quantize_fast_kernel<BLK, BITS><<<(int)(blocks > 0 ? blocks : 1), kFW * 32, 0, st>>>(P, a);
  return cudaGetLastError() == cudaSuccess ? TQ_OK : TQ_ERR_CUDA;
}

}  // namespace

bool quantize_fast_eligible(const CodecParams& P, bool f32_input) {
  return !f32_input && !P.m && !P.nc && (P.blk == 32 || P.blk == 64) && P.bits >= 2 && P.bits <= 4;
}

int launch_quantize_fast(const CodecParams& P, const void* x, int64_t n_vec, int64_t stride, uint8_t* codes,
                         uint16_t* scales, const RowMap& map, cudaStream_t st) {
  FastQuantArgs a;
  a.map = map;
  a.x = static_cast<const __half*>(x);
  a.n_vec = n_vec;
  a.stride = stride;
  a.codes = reinterpret_cast<uint32_t*>(codes);
  a.scales = scales;
  const int K = 1 << P.bits;
  for (int k = 0; k < 8; ++k) a.bstep[k] = 0.f;
  // positive boundaries beta_{K/2} .. beta_{K-2}, in units of the rotated
  // unit vector, times 2^20
  for (int k = K / 2; k < K - 1; ++k) a.bstep[k - K / 2] = P.bounds[k] * kStepScale;
  for (int i = 0; i < 128; ++i) {
    const int c0 = 2 * i, c1 = 2 * i + 1;
    const uint16_t h0 = (c0 < P.d && ((P.sign_bits[c0 >> 5] >> (c0 & 31)) & 1u)) ? 0xBC00 : 0x3C00;
    const uint16_t h1 = (c1 < P.d && ((P.sign_bits[c1 >> 5] >> (c1 & 31)) & 1u)) ? 0xBC00 : 0x3C00;
    a.sgn[i] = (uint32_t)h0 | ((uint32_t)h1 << 16);
  }
  if (P.blk == 64) {
    if (P.bits == 4) return launch_fast<64, 4>(P, a, st);
    if (P.bits == 3) return launch_fast<64, 3>(P, a, st);
    return launch_fast<64, 2>(P, a, st);
  }
  if (P.bits == 4) return launch_fast<32, 4>(P, a, st);
  if (P.bits == 3) return launch_fast<32, 3>(P, a, st);
  return launch_fast<32, 2>(P, a, st);
}

}  // namespace tq
