// GGML-style blocks of the packed cache (llama.cpp-turboquant, "GGML
// Types" and "How it works"): every 32 values become one block of the fp16
// norm of their rotation block followed by their packed codes, 2 + 4*bits
// bytes (14 at 3 bits, 18 at 4 bits).  With a 128-value rotation block this
// is the page's layout: one norm per 128-chunk, stored in each of its four
// 32-value blocks.  Conversion both ways; one thread per 32-value block.
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
  tq::to_blocks_kernel<<<(unsigned)((n + 255) / 256), 256, 0, static_cast<cudaStream_t>(stream)>>>(
      codes, scales, n, groups, P.bits, P.nb, P.blk, blocks);
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
  tq::from_blocks_kernel<<<(unsigned)((n + 255) / 256), 256, 0, static_cast<cudaStream_t>(stream)>>>(
      blocks, n, groups, P.bits, P.nb, P.blk, codes, scales);
  return cudaGetLastError() == cudaSuccess ? TQ_OK : TQ_ERR_CUDA;
}
