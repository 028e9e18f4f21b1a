// GGML-style blocks of the packed cache (llama.cpp-turboquant, "GGML
// Types" and "How it works"): every 32 values become one block of the fp16
// norm of their rotation block followed by their packed codes, 2 + 4*bits
// bytes (14 at 3 bits, 18 at 4 bits).  With a 128-value rotation block this
// is the page's layout: one norm per 128-chunk, stored in each of its four
// 32-value blocks.  Conversion both ways.  A CTA converts a tile of 1024
// consecutive blocks: it stages the side it reads in shared memory with
// coalesced loads, then writes the other side as whole 16-byte words
// gathered from there (a tile of 8k blocks starts on a 16-byte boundary of
// both sides).  Buffers off those boundaries take one thread per block.
#include <cuda_runtime.h>

#include "tq_device.cuh"

namespace tq {
namespace {

__global__ void to_blocks_kernel(const uint8_t* __restrict__ codes, const uint16_t* __restrict__ scales,
                                 int64_t n_blocks, int groups, int bits, int nb, int blk, uint8_t* __restrict__ out) {
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n_blocks) return;
  const int64_t v = i / groups;
  const int j = (int)(i - v * groups);
  const int gb = 4 * bits, bb = 2 + gb;
  uint16_t* dst = reinterpret_cast<uint16_t*>(out + i * bb);   // blocks are 2-byte aligned
  dst[0] = scales[v * nb + (32 * j) / blk];
  const uint16_t* src = reinterpret_cast<const uint16_t*>(codes + (v * groups + j) * gb);
  for (int k = 0; k < gb / 2; ++k) dst[1 + k] = src[k];
}

__global__ void from_blocks_kernel(const uint8_t* __restrict__ blocks, int64_t n_blocks, int groups, int bits,
                                   int nb, int blk, uint8_t* __restrict__ codes, uint16_t* __restrict__ scales) {
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n_blocks) return;
  const int64_t v = i / groups;
  const int j = (int)(i - v * groups);
  const int gb = 4 * bits, bb = 2 + gb;
  const uint16_t* src = reinterpret_cast<const uint16_t*>(blocks + i * bb);
  if ((32 * j) % blk == 0) scales[v * nb + (32 * j) / blk] = src[0];
  uint16_t* dst = reinterpret_cast<uint16_t*>(codes + (v * groups + j) * gb);
  for (int k = 0; k < gb / 2; ++k) dst[k] = src[1 + k];
}

constexpr int kTileBlocks = 1024;   // blocks per CTA tile (a multiple of 8)
constexpr int kTileThreads = 256;

// Codes of a tile, as 16-bit words, staged from 16-byte loads.
template <int GB>
__device__ __forceinline__ void stage16(uint16_t* dst, const uint8_t* src, int bytes) {
  const uint4* s4 = reinterpret_cast<const uint4*>(src);
  uint4* d4 = reinterpret_cast<uint4*>(dst);
  for (int k = threadIdx.x; k < bytes / 16; k += kTileThreads) d4[k] = __ldg(s4 + k);
  // a ragged tail (fewer than 16 bytes) in 16-bit words
  for (int k = (bytes / 16) * 8 + threadIdx.x; k < bytes / 2; k += kTileThreads)
    dst[k] = __ldg(reinterpret_cast<const uint16_t*>(src) + k);
}

// to blocks: one thread per 8 consecutive blocks (8 * (2 + 4 bits) bytes out,
// a whole number of 16-byte words): their codes in 16-byte loads, their 8
// norms, and each output word assembled from two halfwords at positions
// known at compile time.  The words go through shared memory so that the
// CTA's stores are contiguous; a CTA whose range runs past the end writes
// its last, ragged group block by block.
// threads of a to-blocks CTA (8 blocks a thread): its staged codes and
// output words within 40 KB, a power of two of at most 256
template <int BITS>
__host__ __device__ constexpr int g8_threads() {
  constexpr int per_thread = 8 * (4 * BITS + 2 + 4 * BITS);   // code bytes in + block bytes out
  return 40960 / per_thread >= 256 ? 256 : 40960 / per_thread >= 128 ? 128 : 64;
}

template <int BITS>
__global__ void __launch_bounds__(g8_threads<BITS>()) to_blocks_g8(const uint8_t* __restrict__ codes,
                                                            const uint16_t* __restrict__ scales, int64_t n_blocks,
                                                            int gshift, int jshift, int nb,
                                                            uint8_t* __restrict__ out) {
  constexpr int GB = 4 * BITS, BB = 2 + GB, HW = GB / 2;   // bytes of codes / of a block; code halfwords
  constexpr int kT = g8_threads<BITS>();
  __shared__ uint4 s_out[kT * BB / 2];           // the CTA's output words
  __shared__ uint4 s_in[kT * GB / 2];            // the CTA's codes
  const int64_t cta0 = (int64_t)blockIdx.x * kT * 8;   // the CTA's first block
  const int64_t i0 = cta0 + (int64_t)threadIdx.x * 8;
  const int mask = (1 << gshift) - 1;
  if (cta0 + (int64_t)kT * 8 > n_blocks) {
    // the last CTA: plain per-thread stores (no barrier, threads past the end leave)
    if (i0 >= n_blocks) return;
  }
  auto norm_of = [&](int64_t i) -> uint32_t {
    return __ldg(scales + (i >> gshift) * nb + ((int)(i & mask) >> jshift));
  };
  const bool last_cta = cta0 + (int64_t)kT * 8 > n_blocks;
  if (last_cta && i0 + 8 > n_blocks) {
    for (int64_t i = i0; i < n_blocks; ++i) {
      uint16_t* dst = reinterpret_cast<uint16_t*>(out + i * BB);
      dst[0] = (uint16_t)norm_of(i);
      const uint16_t* src = reinterpret_cast<const uint16_t*>(codes + i * GB);
      for (int k = 0; k < HW; ++k) dst[1 + k] = src[k];
    }
    return;
  }
  uint32_t cw[2 * GB];   // the 8 blocks' codes: 8 GB bytes
  const uint4* c4;
  if (last_cta) {
    c4 = reinterpret_cast<const uint4*>(codes + i0 * GB);
  } else {
    // the CTA's codes in one contiguous, coalesced pass
    const uint4* g4 = reinterpret_cast<const uint4*>(codes + cta0 * GB);
#pragma unroll
    for (int q = 0; q < GB / 2; ++q) s_in[q * kT + threadIdx.x] = __ldg(g4 + q * kT + threadIdx.x);
    __syncthreads();
    c4 = s_in + threadIdx.x * (GB / 2);
  }
#pragma unroll
  for (int k = 0; k < GB / 2; ++k) {
    const uint4 v = c4[k];
    cw[4 * k] = v.x; cw[4 * k + 1] = v.y; cw[4 * k + 2] = v.z; cw[4 * k + 3] = v.w;
  }
  uint32_t nr[8];
#pragma unroll
  for (int b = 0; b < 8; ++b) nr[b] = norm_of(i0 + b);
  // halfword o of the 8 blocks: a norm at the start of each block, codes after it
  auto hw = [&](int o) -> uint32_t {
    const int b = o / (BB / 2), k = o - b * (BB / 2);
    if (k == 0) return nr[b];
    const int c = b * HW + k - 1;
    return (cw[c >> 1] >> (16 * (c & 1))) & 0xFFFFu;
  };
  // a lane's words sit BB / 2 words apart: with BB / 2 odd for every width, eight
  // consecutive lanes hit eight different 16-byte bank groups
  uint4* o4 = last_cta ? reinterpret_cast<uint4*>(out + i0 * BB) : s_out + threadIdx.x * (BB / 2);
#pragma unroll
  for (int q = 0; q < BB / 2; ++q) {
    uint32_t w[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) w[e] = hw(8 * q + 2 * e) | (hw(8 * q + 2 * e + 1) << 16);
    o4[q] = make_uint4(w[0], w[1], w[2], w[3]);
  }
  if (last_cta) return;
  __syncthreads();
  uint4* dst = reinterpret_cast<uint4*>(out + cta0 * BB);
#pragma unroll
  for (int q = 0; q < BB / 2; ++q) dst[q * kT + threadIdx.x] = s_out[q * kT + threadIdx.x];
}

// from blocks: a tile of blocks into shared memory, then the codes as
// 16-byte words and each rotation block's norm (from its first 32-value block)
template <int BITS>
__global__ void __launch_bounds__(kTileThreads) from_blocks_tiled(const uint8_t* __restrict__ blocks,
                                                                 int64_t n_blocks, int gshift, int nb, int blk,
                                                                 uint8_t* __restrict__ codes,
                                                                 uint16_t* __restrict__ scales) {
  constexpr int GB = 4 * BITS, BB = 2 + GB;
  __shared__ __align__(16) uint16_t s_blk[kTileBlocks * BB / 2];
  const int64_t i0 = (int64_t)blockIdx.x * kTileBlocks;
  const int n = (int)(n_blocks - i0 < kTileBlocks ? n_blocks - i0 : kTileBlocks);
  stage16<BB>(s_blk, blocks + i0 * BB, n * BB);
  __syncthreads();
  uint8_t* dst = codes + i0 * GB;
  const int bytes = n * GB;
  auto code_half = [&](int k) -> uint32_t {   // code halfword k of the tile
    const int b = k / (GB / 2);
    return s_blk[b * (BB / 2) + 1 + (k - b * (GB / 2))];
  };
  for (int c = threadIdx.x; c < bytes / 16; c += kTileThreads) {
    uint32_t w[4];
#pragma unroll
    for (int h = 0; h < 4; ++h) w[h] = code_half(8 * c + 2 * h) | (code_half(8 * c + 2 * h + 1) << 16);
    *reinterpret_cast<uint4*>(dst + 16 * c) = make_uint4(w[0], w[1], w[2], w[3]);
  }
  for (int k = (bytes / 16) * 8 + threadIdx.x; k < bytes / 2; k += kTileThreads)
    reinterpret_cast<uint16_t*>(dst)[k] = (uint16_t)code_half(k);
  const int groups_mask = (1 << gshift) - 1;
  for (int b = threadIdx.x; b < n; b += kTileThreads) {
    const int64_t i = i0 + b;
    const int j = (int)(i & groups_mask);
    if ((32 * j) % blk == 0) scales[(i >> gshift) * nb + (32 * j) / blk] = s_blk[b * (BB / 2)];
  }
}

template <int BITS>
void launch_to_tiled(const uint8_t* codes, const uint16_t* scales, int64_t n, int gshift, int nb, int blk,
                     uint8_t* out, cudaStream_t st) {
  int jshift = 0;
  while ((32 << jshift) < blk) ++jshift;
  const int64_t groups8 = (n + 7) / 8;
  constexpr int kT = g8_threads<BITS>();
  to_blocks_g8<BITS><<<(unsigned)((groups8 + kT - 1) / kT), kT, 0, st>>>(
      codes, scales, n, gshift, jshift, nb, out);
}
template <int BITS>
void launch_from_tiled(const uint8_t* blocks, int64_t n, int gshift, int nb, int blk, uint8_t* codes,
                       uint16_t* scales, cudaStream_t st) {
  from_blocks_tiled<BITS><<<(unsigned)((n + kTileBlocks - 1) / kTileBlocks), kTileThreads, 0, st>>>(
      blocks, n, gshift, nb, blk, codes, scales);
}

// log2 of the blocks per vector when the tiled kernels apply (a power of two
// >= 2, at most 8 norms per vector, rotation blocks of a power of two times
// 32 values), else -1
int tiled_shift(int groups, int nb, int blk) {
  if (groups < 2 || (groups & (groups - 1)) || nb > 8 || blk < 32 || ((blk / 32) & (blk / 32 - 1)) || blk % 32)
    return -1;
  int s = 0;
  while ((1 << s) < groups) ++s;
  return s;
}

int block_args(const tq_layout* layout, CodecParams* P) {
  const int st = make_params(layout, P);
  if (st != TQ_OK) return st;
  return P->m ? TQ_ERR_UNSUPPORTED : TQ_OK;   // QJL vectors have no block form on the page
}

}  // namespace
}  // namespace tq

extern "C" int tq_to_blocks(const tq_layout* layout, const uint8_t* codes, const uint16_t* scales, int64_t n_vec,
                            uint8_t* blocks, void* stream) {
  tq::CodecParams P;
  int st = tq::block_args(layout, &P);
  if (st != TQ_OK) return st;
  if (n_vec < 0) return TQ_ERR_ARG;
  if (n_vec == 0) return TQ_OK;
  if (!codes || !scales || !blocks) return TQ_ERR_ARG;
  if ((reinterpret_cast<uintptr_t>(codes) & 3) || (reinterpret_cast<uintptr_t>(scales) & 1) ||
      (reinterpret_cast<uintptr_t>(blocks) & 1))
    return TQ_ERR_ALIGN;
  const int groups = P.d / 32;
  const int64_t n = n_vec * groups;
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  const int gshift = tq::tiled_shift(groups, P.nb, P.blk);
  if (gshift >= 0 && tq::aligned16(codes) && tq::aligned16(blocks)) {
    switch (P.bits) {
      case 1: tq::launch_to_tiled<1>(codes, scales, n, gshift, P.nb, P.blk, blocks, cs); break;
      case 2: tq::launch_to_tiled<2>(codes, scales, n, gshift, P.nb, P.blk, blocks, cs); break;
      case 3: tq::launch_to_tiled<3>(codes, scales, n, gshift, P.nb, P.blk, blocks, cs); break;
      case 4: tq::launch_to_tiled<4>(codes, scales, n, gshift, P.nb, P.blk, blocks, cs); break;
      default: tq::launch_to_tiled<8>(codes, scales, n, gshift, P.nb, P.blk, blocks, cs); break;
    }
  } else {
    tq::to_blocks_kernel<<<(unsigned)((n + 255) / 256), 256, 0, cs>>>(codes, scales, n, groups, P.bits, P.nb, P.blk,
                                                                      blocks);
  }
  return cudaGetLastError() == cudaSuccess ? TQ_OK : TQ_ERR_CUDA;
}

extern "C" int tq_from_blocks(const tq_layout* layout, const uint8_t* blocks, int64_t n_vec, uint8_t* codes,
                              uint16_t* scales, void* stream) {
  tq::CodecParams P;
  int st = tq::block_args(layout, &P);
  if (st != TQ_OK) return st;
  if (n_vec < 0) return TQ_ERR_ARG;
  if (n_vec == 0) return TQ_OK;
  if (!codes || !scales || !blocks) return TQ_ERR_ARG;
  if ((reinterpret_cast<uintptr_t>(codes) & 3) || (reinterpret_cast<uintptr_t>(scales) & 1) ||
      (reinterpret_cast<uintptr_t>(blocks) & 1))
    return TQ_ERR_ALIGN;
  const int groups = P.d / 32;
  const int64_t n = n_vec * groups;
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  const int gshift = tq::tiled_shift(groups, P.nb, P.blk);
  if (gshift >= 0 && tq::aligned16(codes) && tq::aligned16(blocks)) {
    switch (P.bits) {
      case 1: tq::launch_from_tiled<1>(blocks, n, gshift, P.nb, P.blk, codes, scales, cs); break;
      case 2: tq::launch_from_tiled<2>(blocks, n, gshift, P.nb, P.blk, codes, scales, cs); break;
      case 3: tq::launch_from_tiled<3>(blocks, n, gshift, P.nb, P.blk, codes, scales, cs); break;
      case 4: tq::launch_from_tiled<4>(blocks, n, gshift, P.nb, P.blk, codes, scales, cs); break;
      default: tq::launch_from_tiled<8>(blocks, n, gshift, P.nb, P.blk, codes, scales, cs); break;
    }
  } else {
    tq::from_blocks_kernel<<<(unsigned)((n + 255) / 256), 256, 0, cs>>>(blocks, n, groups, P.bits, P.nb, P.blk,
                                                                        codes, scales);
  }
  return cudaGetLastError() == cudaSuccess ? TQ_OK : TQ_ERR_CUDA;
}
