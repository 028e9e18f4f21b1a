// Prefill attention over the packed cache (tensor-core path; filled in below).
#include <cuda_runtime.h>

#include "tq_device.cuh"

extern "C" int tq_prefill_workspace_bytes(int B, int Hq, int Hkv, int head_dim, int Tq, int64_t ctx,
                                          size_t* bytes) {
  if (B <= 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv || Tq < 0 || ctx < Tq || !bytes) return TQ_ERR_ARG;
  if (head_dim != 64 && head_dim != 128 && head_dim != 256) return TQ_ERR_UNSUPPORTED;
  *bytes = 0;
  return TQ_OK;
}

extern "C" int tq_prefill_attn(const tq_kv_view*, const tq_kv_view*, const uint16_t*, int, int, int, int,
                               int64_t, int64_t, int, float, uint16_t*, void*, size_t, void*) {
  return TQ_ERR_UNSUPPORTED;
}
