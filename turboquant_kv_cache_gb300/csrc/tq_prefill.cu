// C entry points of prefill attention; the kernels are in tq_prefill_tc.cu.
#include <cuda_runtime.h>
#include <math.h>

#include "tq_device.cuh"

namespace tq {
size_t prefill_tc_workspace(int B, int Hq, int Hkv, int d, int Tq, int64_t ctx);
int launch_prefill_tc(const CodecParams& PK, const CodecParams& PV, const uint8_t* kc, const uint16_t* ks,
                      const uint8_t* vc, const uint16_t* vs, const uint16_t* q, int B, int Hq, int Hkv, int Tq,
                      int64_t S_cap, int64_t ctx, int causal, float qscale, uint16_t* out, void* ws,
                      const PageMap& pages, cudaStream_t st);
}  // namespace tq

extern "C" int tq_prefill_workspace_bytes(int B, int Hq, int Hkv, int head_dim, int Tq, int64_t ctx,
                                          size_t* bytes) {
  if (B <= 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv || Tq < 0 || ctx < Tq || !bytes) return TQ_ERR_ARG;
  if (head_dim != 64 && head_dim != 128 && head_dim != 256) return TQ_ERR_UNSUPPORTED;
  *bytes = Tq == 0 ? 0 : tq::prefill_tc_workspace(B, Hq, Hkv, head_dim, Tq, ctx);
  return TQ_OK;
}

extern "C" int tq_prefill_attn(const tq_kv_view* K, const tq_kv_view* V, const uint16_t* q, int B, int Hq, int Hkv,
                               int Tq, int64_t S_cap, int64_t ctx, int causal, float softmax_scale, uint16_t* out,
                               void* workspace, size_t workspace_bytes, void* stream) {
  if (!K || !V || !q || !out) return TQ_ERR_ARG;
  tq::CodecParams PK, PV;
  int st = tq::make_params(&K->layout, &PK);
  if (st != TQ_OK) return st;
  st = tq::make_params(&V->layout, &PV);
  if (st != TQ_OK) return st;
  if (PK.d != PV.d || PK.m || PV.m || PK.bits > 4 || PV.bits > 4) return TQ_ERR_UNSUPPORTED;
  if (B <= 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv || Tq < 0 || ctx < Tq || ctx > S_cap) return TQ_ERR_ARG;
  if (!K->codes || !K->scales || !V->codes || !V->scales) return TQ_ERR_ARG;
  if (tq::check_paging(K, S_cap) != TQ_OK || !tq::same_paging(K, V)) return TQ_ERR_ARG;
  if (!tq::aligned16(K->codes) || !tq::aligned16(V->codes) || !tq::aligned16(q) || !tq::aligned16(out))
    return TQ_ERR_ALIGN;
  if (Tq == 0) return TQ_OK;
  const size_t need = tq::prefill_tc_workspace(B, Hq, Hkv, PK.d, Tq, ctx);
  if (!workspace || workspace_bytes < need) return TQ_ERR_WORKSPACE;
  if (!tq::aligned16(workspace)) return TQ_ERR_ALIGN;
  const float sm = softmax_scale > 0.f ? softmax_scale : 1.0f / sqrtf((float)PK.d);
  return tq::launch_prefill_tc(PK, PV, K->codes, K->scales, V->codes, V->scales, q, B, Hq, Hkv, Tq, S_cap, ctx,
                               causal ? 1 : 0, sm * tq::kLog2e, out, workspace,
                               {K->page_table, K->page_table ? K->page_size : 0, K->page_table ? K->pages_per_seq : 0},
                               static_cast<cudaStream_t>(stream));
}
