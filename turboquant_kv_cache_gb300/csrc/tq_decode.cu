// Fused decode attention over the packed cache, computed in the Hadamard
// domain, plus the split-K combine that rotates the output back.
//
// Per CTA: one (batch, KV head) and one slice of the context.  The G query
// heads of the GQA group share every K/V record read.  The query is rotated
// once (q^ = H D q per K block, times softmax_scale * log2 e); a score is
// sum_j scaleK_j <q^_j, c(codes_j)> (+ the QJL term); V is accumulated
// rotated, sum_t p_t scaleV c(codes_t); the combine merges the splits by
// log-sum-exp and applies D H once per output ("llama.cpp-turboquant",
// "Fused tile path: K and V decoded inside attention").
#include <cuda_runtime.h>
#include <math.h>

#include <mutex>

#include "tq_device.cuh"

namespace tq {

int decode_auto_splits(int B, int Hkv, int64_t ctx, int per_sm = 4);
int decode_tc_ctas_per_sm(const CodecParams& PK, const CodecParams& PV);
int decode_tc_max_ctas_per_sm();
bool decode_tc_blocks_eligible(const CodecParams& PK, const CodecParams& PV, int G, int64_t S_cap,
                               const uint8_t* k_blocks, const uint8_t* v_blocks);
int launch_decode_tc_blocks(const CodecParams& PK, const CodecParams& PV, const uint8_t* k_blocks,
                            const uint8_t* v_blocks, const uint16_t* q, const int32_t* kv_len, float* part, int B,
                            int Hq, int Hkv, int64_t S_cap, int64_t ctx, int n_split, float qscale, cudaStream_t st);
bool decode_tc_eligible(const CodecParams& PK, const CodecParams& PV, int G, int64_t S_cap, const tq_kv_view* K,
                        const tq_kv_view* V);
size_t decode_tc_extra_bytes(int B, int Hq);
int launch_decode_tc(const CodecParams& PK, const CodecParams& PV, const tq_kv_view* K, const tq_kv_view* V,
                     const uint16_t* q, const int32_t* kv_len, float* part, size_t part_bytes, int B, int Hq, int Hkv,
                     int64_t S_cap, int64_t ctx, int n_split, int slots, bool pdl, float qscale, const Codebook8* cbk,
                     cudaStream_t st);
size_t decode_ws_bytes(int B, int Hq, int d, int n_split);

namespace {

constexpr int kWarps = 4;
constexpr int kDecThreads = kWarps * 32;

struct DecodeArgs {
  const uint32_t* kc;
  const uint16_t* ks;
  const uint32_t* kq;   // QJL bits
  const uint16_t* kr;   // QJL rho
  const float* S;
  const uint32_t* vc;
  const uint16_t* vs;
  const uint32_t* vq;   // QJL bits of V
  const uint16_t* vr;   // QJL rho of V
  const float* Sv;      // V's QJL projection [m][d]
  const uint16_t* q;
  const int32_t* kv_len;
  float* part;          // [B*Hq][slots][d + 4]
  PageMap pages;        // paging of both caches (table NULL: contiguous)
  int64_t S_cap;
  int64_t ctx;
  int Hq, Hkv, n_split;
  int slots;            // split slots per row (n_split, or more for extra partials)
  float qscale;         // softmax_scale * log2(e)
  int pdl;              // launched as a programmatic dependent of the kernel before it
  // block layout (AOS kernels only): per token d/32 blocks of [fp16 norm of
  // the rotation block, 4*bits code bytes], read as 16-bit units
  const uint16_t* kblk = nullptr;
  const uint16_t* vblk = nullptr;
};

// The packed words of one 32-code group stored inside a block record
// (2-byte aligned): g16 points at the block's first code byte.
__device__ __forceinline__ void block_group_words(const uint16_t* g16, int bits, uint32_t gw[4]) {
#pragma unroll
  for (int k = 0; k < 4; ++k)
    gw[k] = k < bits ? (uint32_t)g16[2 * k] | ((uint32_t)g16[2 * k + 1] << 16) : 0u;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v = fmaxf(v, __shfl_xor_sync(kFull, v, o));
  return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
  return v;
}

// In-place orthonormal Walsh-Hadamard on rows of a shared [rows][D] array,
// in blocks of `blk`, executed by the whole CTA.
template <int D>
__device__ void smem_wht(float* a, int rows, int blk, float norm) {
  for (int h = 1; h < blk; h <<= 1) {
    __syncthreads();
    for (int e = threadIdx.x; e < rows * D / 2; e += blockDim.x) {
      const int row = e / (D / 2), k = e % (D / 2);
      const int i = (k / h) * 2 * h + (k % h);
      float* r = a + row * D;
      const float x = r[i], y = r[i + h];
      r[i] = x + y;
      r[i + h] = x - y;
    }
  }
  __syncthreads();
  for (int e = threadIdx.x; e < rows * D; e += blockDim.x) a[e] *= norm;
  __syncthreads();
}

// QV: V carries a QJL residual (m <= kMaxQjlV rows).  The split then also
// accumulates sum_t p_t s_t rho_t (2 b_t - 1) (m values, lane holds rows
// lane + 32 k), and its epilogue adds sqrt(pi/2)/m S^T of that, rotated into
// V's coded domain, to the accumulator: the QJL term of every value, applied
// once per split instead of once per token.
// K8: keys of one byte per code, their 256-level table in `cbk`.
// AOS: K and V read from the block layout (a.kblk, a.vblk) instead of the
// separate code and norm arrays (no QJL, no 8-bit codes, contiguous cache).
template <int D, int G, bool QV, bool K8, bool AOS = false>
__global__ void __launch_bounds__(kDecThreads) decode_split_kernel(const CodecParams PK, const CodecParams PV,
                                                                   const DecodeArgs a,
                                                                   const Codebook8Param<K8> cbk) {
  constexpr int CPL = D / 32;  // V coordinates per lane
  constexpr int CQ = QV ? kMaxQjlV / 32 : 1;   // QJL rows of V per lane
  __shared__ float s_q[G][D];          // q, then q^ (rotated, scaled)
  __shared__ float s_qT[D][G];         // q^ transposed: coordinate-major
  __shared__ float s_sq[kMaxQjl][G];   // S q (QJL keys)
  __shared__ float s_centK[K8 ? 256 : 16], s_centV[16];
  __shared__ float s_p[kWarps][32][G];
  __shared__ float s_ml[kWarps][2][G];
  __shared__ float s_acc[kWarps][D];   // one head at a time in the final merge
  __shared__ float s_accq[QV ? kWarps : 1][QV ? kMaxQjlV : 1];
  __shared__ float s_aq[QV ? kMaxQjlV : 1];
  __shared__ float s_proj[QV ? D : 1];

  const int split = blockIdx.x;
  const int bh = blockIdx.y;           // b * Hkv + kv head
  const int b = bh / a.Hkv;
  const int kvh = bh % a.Hkv;
  const int h0 = kvh * G;
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;

  if constexpr (K8) {
    for (int k = threadIdx.x; k < 256; k += kDecThreads) s_centK[k] = cbk.c[k];
  } else if (threadIdx.x < 16) {
    s_centK[threadIdx.x] = PK.centroids[threadIdx.x];
  }
  if (threadIdx.x < 16) s_centV[threadIdx.x] = PV.centroids[threadIdx.x];
  for (int e = threadIdx.x; e < G * D; e += kDecThreads) {
    const int h = e / D, i = e % D;
    s_q[h][i] = h2f(a.q[((int64_t)b * a.Hq + h0 + h) * D + i]);
  }
  __syncthreads();
  if (PK.m) {  // S q in the input domain, scaled like the scores
    for (int e = threadIdx.x; e < PK.m * G; e += kDecThreads) {
      const int i = e / G, h = e % G;
      float acc = 0.f;
      for (int k = 0; k < D; ++k) acc = fmaf(__ldg(a.S + (int64_t)i * D + k), s_q[h][k], acc);
      s_sq[i][h] = acc * a.qscale;
    }
    __syncthreads();  // s_q is rotated in place below
  }
  for (int e = threadIdx.x; e < G * D; e += kDecThreads) {
    const int h = e / D, i = e % D;
    if ((PK.sign_bits[i >> 5] >> (i & 31)) & 1u) s_q[h][i] = -s_q[h][i];
  }
  smem_wht<D>(&s_q[0][0], G, PK.blk, PK.inv_sqrt_blk * a.qscale);
  for (int e = threadIdx.x; e < G * D; e += kDecThreads) {
    const int h = e / D, i = e % D;
    s_qT[i][h] = s_q[h][i];
  }
  __syncthreads();

  int64_t len = a.ctx;
  if (a.kv_len) len = imin64(len, (int64_t)a.kv_len[b]);
  const int64_t per = (a.ctx + a.n_split - 1) / a.n_split;
  const int64_t t_begin = (int64_t)split * per;
  const int64_t t_end = imin64(t_begin + per, len);

  float m_run[G], l_run[G], acc[G][CPL], accq[G][CQ];
#pragma unroll
  for (int h = 0; h < G; ++h) {
    m_run[h] = -INFINITY;
    l_run[h] = 0.f;
#pragma unroll
    for (int k = 0; k < CPL; ++k) acc[h][k] = 0.f;
#pragma unroll
    for (int k = 0; k < CQ; ++k) accq[h][k] = 0.f;
  }
  const int mq = QV ? PV.m / 32 : 0;   // QJL words of a V record
  const int kwords = PK.code_bytes / 4, vwords = PV.code_bytes / 4;
  auto rec_of = [&](int64_t t) { return cache_rec(a.pages, a.Hkv, a.S_cap, b, kvh, t); };

  for (int64_t c0 = t_begin + (int64_t)wid * 32; c0 < t_end; c0 += kWarps * 32) {
    const int64_t t = c0 + lane;
    const bool valid = t < t_end;
    float s[G];
#pragma unroll
    for (int h = 0; h < G; ++h) s[h] = 0.f;
    if (valid && AOS) {
      const int kb16 = 1 + 2 * PK.bits;   // 16-bit units per 32-value block
      const uint16_t* tr = a.kblk + rec_of(t) * (int64_t)(D / 32) * kb16;
      const int gpb = PK.blk / 32;
      for (int j = 0; j < PK.nb; ++j) {
        float part[G];
#pragma unroll
        for (int h = 0; h < G; ++h) part[h] = 0.f;
        for (int gg = 0; gg < gpb; ++gg) {
          const int gi = j * gpb + gg;
          uint32_t gw[4];
          block_group_words(tr + gi * kb16 + 1, PK.bits, gw);
#pragma unroll
          for (int w = 0; w < 4; ++w) {
            const uint32_t nib = load_chunk(gw, PK.bits, w);
#pragma unroll
            for (int r = 0; r < 8; ++r) {
              const float c = s_centK[(nib >> (4 * r)) & 0xf];
              const int i = gi * 32 + w * 8 + r;
#pragma unroll
              for (int h = 0; h < G; ++h) part[h] = fmaf(c, s_qT[i][h], part[h]);
            }
          }
        }
        const float scj = h2f(tr[j * gpb * kb16]);   // the norm heads each block of the rotation block
#pragma unroll
        for (int h = 0; h < G; ++h) s[h] = fmaf(scj, part[h], s[h]);
      }
    } else if (valid) {
      const int64_t rt = rec_of(t);
      const uint32_t* rec = a.kc + rt * kwords;
      const uint16_t* sc = a.ks + rt * PK.nb;
      const int gpb = PK.blk / 32;  // 32-code groups per block
      for (int j = 0; j < PK.nb; ++j) {
        float part[G];
#pragma unroll
        for (int h = 0; h < G; ++h) part[h] = 0.f;
        for (int gg = 0; gg < gpb; ++gg) {
          const int gi = j * gpb + gg;
          const uint32_t* gw = rec + gi * PK.bits;
          if constexpr (K8) {
            // 32 bytes, code i of the group in byte i: two 16-byte loads
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
              const uint4 u = reinterpret_cast<const uint4*>(gw)[hf];
              const uint32_t wv[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
              for (int w = 0; w < 4; ++w) {
#pragma unroll
                for (int r = 0; r < 4; ++r) {
                  const float c = s_centK[(wv[w] >> (8 * r)) & 0xff];
                  const int i = gi * 32 + hf * 16 + w * 4 + r;
#pragma unroll
                  for (int h = 0; h < G; ++h) part[h] = fmaf(c, s_qT[i][h], part[h]);
                }
              }
            }
          } else {
#pragma unroll
            for (int w = 0; w < 4; ++w) {
              const uint32_t nib = load_chunk(gw, PK.bits, w);
#pragma unroll
              for (int r = 0; r < 8; ++r) {
                const float c = s_centK[(nib >> (4 * r)) & 0xf];
                const int i = gi * 32 + w * 8 + r;
#pragma unroll
                for (int h = 0; h < G; ++h) part[h] = fmaf(c, s_qT[i][h], part[h]);
              }
            }
          }
        }
        const float scj = h2f(sc[j]);
#pragma unroll
        for (int h = 0; h < G; ++h) s[h] = fmaf(scj, part[h], s[h]);
      }
      if (PK.m) {
        const float coef = h2f(sc[0]) * h2f(a.kr[rt]) * kSqrtHalfPi / (float)PK.m;
        const uint32_t* qb = a.kq + rt * (PK.m / 32);
        float part[G];
#pragma unroll
        for (int h = 0; h < G; ++h) part[h] = 0.f;
        for (int i = 0; i < PK.m; ++i) {
          const float sgn = ((qb[i >> 5] >> (i & 31)) & 1u) ? 1.f : -1.f;
#pragma unroll
          for (int h = 0; h < G; ++h) part[h] = fmaf(sgn, s_sq[i][h], part[h]);
        }
#pragma unroll
        for (int h = 0; h < G; ++h) s[h] = fmaf(coef, part[h], s[h]);
      }
    } else {
#pragma unroll
      for (int h = 0; h < G; ++h) s[h] = -INFINITY;
    }
    // online softmax (base 2), one update per 32-token chunk
#pragma unroll
    for (int h = 0; h < G; ++h) {
      const float mx = warp_max(s[h]);
      const float m_new = fmaxf(m_run[h], mx);
      const float p = valid ? exp2f(s[h] - m_new) : 0.f;
      const float alpha = m_run[h] == -INFINITY ? 0.f : exp2f(m_run[h] - m_new);
      l_run[h] = l_run[h] * alpha + warp_sum(p);
      m_run[h] = m_new;
#pragma unroll
      for (int k = 0; k < CPL; ++k) acc[h][k] *= alpha;
      if (QV) {
#pragma unroll
        for (int k = 0; k < CQ; ++k) accq[h][k] *= alpha;
      }
      s_p[wid][lane][h] = p;
    }
    __syncwarp();
    const int n_tok = (int)imin64(32, t_end - c0);
    for (int tt = 0; tt < n_tok; ++tt) {
      if constexpr (AOS) {
        const int vb16 = 1 + 2 * PV.bits;
        const uint16_t* tr = a.vblk + rec_of(c0 + tt) * (int64_t)(D / 32) * vb16;
#pragma unroll
        for (int k = 0; k < CPL; ++k) {
          // coordinate lane + 32 k: group k, position lane
          const uint16_t* g16 = tr + k * vb16 + 1;
          const auto word = [g16](int j) { return (uint32_t)g16[2 * j] | ((uint32_t)g16[2 * j + 1] << 16); };
          const int code = (load_chunk_by(word, PV.bits, lane >> 3) >> (4 * (lane & 7))) & 0xf;
          const int i = lane + 32 * k;
          const float v = s_centV[code] * h2f(tr[(i / PV.blk) * (PV.blk / 32) * vb16]);
#pragma unroll
          for (int h = 0; h < G; ++h) acc[h][k] = fmaf(s_p[wid][tt][h], v, acc[h][k]);
        }
        continue;
      }
      const int64_t r = rec_of(c0 + tt);
      const uint32_t* rec = a.vc + r * vwords;
      const uint16_t* sc = a.vs + r * PV.nb;
#pragma unroll
      for (int k = 0; k < CPL; ++k) {
        const int i = lane + 32 * k;
        const float v = s_centV[code_at(rec, PV.bits, i)] * h2f(sc[i / PV.blk]);
#pragma unroll
        for (int h = 0; h < G; ++h) acc[h][k] = fmaf(s_p[wid][tt][h], v, acc[h][k]);
      }
      if (QV) {
        // the norm times rho weighs the +-1 signs of the token
        const float wr = h2f(sc[0]) * h2f(a.vr[r]);
        const uint32_t* qb = a.vq + r * mq;
#pragma unroll
        for (int k = 0; k < CQ; ++k) {
          if (k < mq) {
            const float sgn = ((qb[k] >> lane) & 1u) ? wr : -wr;
#pragma unroll
            for (int h = 0; h < G; ++h) accq[h][k] = fmaf(s_p[wid][tt][h], sgn, accq[h][k]);
          }
        }
      }
    }
    __syncwarp();
  }
  // merge the warps of the CTA
  if (lane == 0) {
#pragma unroll
    for (int h = 0; h < G; ++h) {
      s_ml[wid][0][h] = m_run[h];
      s_ml[wid][1][h] = l_run[h];
    }
  }
#pragma unroll
  for (int h = 0; h < G; ++h) {
    __syncthreads();
#pragma unroll
    for (int k = 0; k < CPL; ++k) s_acc[wid][lane + 32 * k] = acc[h][k];
    if (QV) {
#pragma unroll
      for (int k = 0; k < CQ; ++k) s_accq[wid][lane + 32 * k] = accq[h][k];
    }
    __syncthreads();
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) M = fmaxf(M, s_ml[w][0][h]);
    if (QV) {
      // the merged sign sums, then sqrt(pi/2)/m S^T of them (input domain),
      // then into V's coded domain: D signs, H per block over sqrt(blk)
      for (int k = threadIdx.x; k < PV.m; k += kDecThreads) {
        float v = 0.f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) {
          const float mw = s_ml[w][0][h];
          v += (mw == -INFINITY ? 0.f : exp2f(mw - M)) * s_accq[w][k];
        }
        s_aq[k] = v;
      }
      __syncthreads();
      for (int i = threadIdx.x; i < D; i += kDecThreads) {
        float v = 0.f;
        for (int k = 0; k < PV.m; ++k) v = fmaf(__ldg(a.Sv + (int64_t)k * D + i), s_aq[k], v);
        s_proj[i] = flip(v * (kSqrtHalfPi / (float)PV.m), (PV.sign_bits[i >> 5] >> (i & 31)) & 1u);
      }
      smem_wht<D>(s_proj, 1, PV.blk, PV.inv_sqrt_blk);
    }
    float* dst = a.part + (((int64_t)b * a.Hq + h0 + h) * a.slots + split) * (D + 4);
    for (int i = threadIdx.x; i < D + 2; i += kDecThreads) {
      float val = 0.f;
      if (i == 0) {
        val = M;
      } else {
#pragma unroll
        for (int w = 0; w < kWarps; ++w) {
          const float mw = s_ml[w][0][h];
          const float wt = mw == -INFINITY ? 0.f : exp2f(mw - M);
          val += wt * (i == 1 ? s_ml[w][1][h] : s_acc[w][i - 2]);
        }
        if (QV && i >= 2) val += s_proj[i - 2];
      }
      dst[i] = val;
    }
  }
  // finish only after the kernel this one may overlap (a no-op otherwise)
  asm volatile("griddepcontrol.wait;\n" ::: "memory");
}

// Final step of a merged row: divide by the total mass, rotate back (D H per
// V block) with in-lane and shuffle butterflies, store fp16.  Lane holds the
// D/32 consecutive coordinates E*lane .. E*lane+E-1.
template <int D>
__device__ __forceinline__ void finish_row(const CodecParams& PV, float* o, float L, uint16_t* dst_row, int lane) {
  constexpr int E = D / 32;
  const float inv = L > 0.f ? PV.inv_sqrt_blk / L : 0.f;
  // unnormalised Walsh-Hadamard per V block: strides below E inside the
  // lane, the rest across lanes
  for (int h = 1; h < E && h < PV.blk; h <<= 1) {
#pragma unroll
    for (int e = 0; e < E; ++e) {
      if ((e & h) == 0) {
        const float x = o[e], y = o[e + h];
        o[e] = x + y;
        o[e + h] = x - y;
      }
    }
  }
  for (int h = E; h < PV.blk; h <<= 1) {
    const int lo = h / E;
#pragma unroll
    for (int e = 0; e < E; ++e) {
      const float q = __shfl_xor_sync(kFull, o[e], lo);
      o[e] = (lane & lo) ? (q - o[e]) : (o[e] + q);
    }
  }
  uint32_t packed[E / 2];
#pragma unroll
  for (int e = 0; e < E; e += 2) {
    const int i = E * lane + e;
    const float v0 = flip(o[e] * inv, (PV.sign_bits[i >> 5] >> (i & 31)) & 1u);
    const float v1 = flip(o[e + 1] * inv, (PV.sign_bits[(i + 1) >> 5] >> ((i + 1) & 31)) & 1u);
    packed[e / 2] = (uint32_t)f2h(v0) | ((uint32_t)f2h(v1) << 16);
  }
  uint16_t* dst = dst_row + E * lane;
  if (E == 8) {
    *reinterpret_cast<uint4*>(dst) = make_uint4(packed[0], packed[1 % (E / 2)], packed[2 % (E / 2)], packed[3 % (E / 2)]);
  } else if (E == 4) {
    *reinterpret_cast<uint2*>(dst) = make_uint2(packed[0], packed[1 % (E / 2)]);
  } else {
    *reinterpret_cast<uint32_t*>(dst) = packed[0];
  }
}

constexpr int kCombWarps = 2;  // rows per CTA: many small CTAs spread the L2 reads over the SMs

// One warp per output row (b, head[, query]); lane holds the D/32 consecutive
// coordinates E*lane .. E*lane+E-1.  Merges the split partials (log-sum-exp
// weights), divides by the total mass and rotates back (D H per V block)
// with in-lane and shuffle butterflies.  Launched as a programmatic
// dependent of the split kernel: the wait below holds until that grid has
// finished and its partials are visible.
template <int D>
__global__ void __launch_bounds__(kCombWarps * 32) decode_combine_kernel(const CodecParams PV, const float* __restrict__ part,
                                                             int n_split, uint16_t* __restrict__ out, int rows) {
  asm volatile("griddepcontrol.wait;\n" ::: "memory");
  constexpr int E = D / 32;
  const int row = blockIdx.x * kCombWarps + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  if (row >= rows) return;
  const float* p = part + (int64_t)row * n_split * (D + 4);
  // Up to kPre splits (more go to the wide kernel): their values are loaded
  // before anything else, so that every load of the row is in flight at
  // once, one round trip to L2 instead of a chain of them.  Lane s holds
  // split s's (m, l).
  constexpr int kPre = 64 / E;   // 32, 16, 8 splits for d = 64, 128, 256
  float2 v[kPre][E / 2];
#pragma unroll
  for (int j = 0; j < kPre; ++j)
#pragma unroll
    for (int e = 0; e < E / 2; ++e)
      v[j][e] = j < n_split ? *reinterpret_cast<const float2*>(p + j * (D + 4) + 2 + E * lane + 2 * e)
                            : make_float2(0.f, 0.f);
  const float m_l = lane < n_split ? p[lane * (D + 4)] : -INFINITY;
  const float l_l = lane < n_split ? p[lane * (D + 4) + 1] : 0.f;
  float M = m_l;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(kFull, M, o));
  // weight of split s: exp2(m_s - M), zero for an empty split
  const float w_l = m_l == -INFINITY ? 0.f : exp2f(m_l - M);
  float L = w_l * l_l;
  float o[E];
#pragma unroll
  for (int e = 0; e < E; ++e) o[e] = 0.f;
#pragma unroll
  for (int j = 0; j < kPre; ++j) {
    const float w = __shfl_sync(kFull, w_l, j);   // zero for j >= n_split
#pragma unroll
    for (int e = 0; e < E / 2; ++e) {
      o[2 * e] = fmaf(w, v[j][e].x, o[2 * e]);
      o[2 * e + 1] = fmaf(w, v[j][e].y, o[2 * e + 1]);
    }
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) L += __shfl_xor_sync(kFull, L, off);
  finish_row<D>(PV, o, L, out + (int64_t)row * D, lane);
}

// Many splits (more than the narrow kernel preloads): one CTA per row, the
// warps take interleaved subsets of the splits, then one warp sums them.
constexpr int kWideWarps = 8;

template <int D>
__global__ void __launch_bounds__(kWideWarps * 32) decode_combine_wide_kernel(const CodecParams PV,
                                                                             const float* __restrict__ part,
                                                                             int n_split, uint16_t* __restrict__ out) {
  asm volatile("griddepcontrol.wait;\n" ::: "memory");
  constexpr int E = D / 32;
  __shared__ float s_o[kWideWarps][D];
  __shared__ float s_x[kWideWarps];
  const int row = blockIdx.x, w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const float* p = part + (int64_t)row * n_split * (D + 4);
  float M = -INFINITY;
  for (int s = threadIdx.x; s < n_split; s += kWideWarps * 32) M = fmaxf(M, p[s * (D + 4)]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(kFull, M, o));
  if (lane == 0) s_x[w] = M;
  __syncthreads();
  M = s_x[0];
#pragma unroll
  for (int i = 1; i < kWideWarps; ++i) M = fmaxf(M, s_x[i]);
  float o[E];
#pragma unroll
  for (int e = 0; e < E; ++e) o[e] = 0.f;
  float L = 0.f;
#pragma unroll 4
  for (int s = w; s < n_split; s += kWideWarps) {
    const float* ps = p + s * (D + 4);
    const float ms = ps[0];
    const float wt = ms == -INFINITY ? 0.f : exp2f(ms - M);
    L = fmaf(wt, ps[1], L);
#pragma unroll
    for (int e = 0; e < E; e += 2) {
      const float2 v = *reinterpret_cast<const float2*>(ps + 2 + E * lane + e);
      o[e] = fmaf(wt, v.x, o[e]);
      o[e + 1] = fmaf(wt, v.y, o[e + 1]);
    }
  }
  __syncthreads();  // every warp has read s_x
#pragma unroll
  for (int e = 0; e < E; ++e) s_o[w][E * lane + e] = o[e];
  if (lane == 0) s_x[w] = L;
  __syncthreads();
  if (w != 0) return;
  L = 0.f;
#pragma unroll
  for (int i = 0; i < kWideWarps; ++i) L += s_x[i];
#pragma unroll
  for (int e = 0; e < E; ++e) {
    float v = 0.f;
#pragma unroll
    for (int i = 0; i < kWideWarps; ++i) v += s_o[i][E * lane + e];
    o[e] = v;
  }
  finish_row<D>(PV, o, L, out + (int64_t)row * D, lane);
}

// Partials of the fp16 residual window, one CTA per (batch, KV head) and its
// G <= 8 q heads, as split slot `slot` of their rows.  The window is walked
// in chunks of 128 tokens with an online base-2 softmax: thread t scores
// token t of the chunk against every head (its key row loaded with 16-byte
// reads, all in flight at once; q in shared memory), one warp per head pair
// takes the chunk maximum and sum, then warp w accumulates tokens w, w+4, ...
// with lane holding D/32 consecutive coordinates (8- or 16-byte value
// reads).  The four warps' accumulators are summed in shared memory and
// rotated into V's coded domain (D signs, then H per V block over
// sqrt(blk)), so the combine merges and rotates them back with the
// quantised splits.  The kernel is small and latency-bound: every loop keeps
// its loads independent so that they overlap.
constexpr int kWinCh = 128;
constexpr int kWinMaxG = 8;

template <int D>
__global__ void __launch_bounds__(128) decode_window_kernel(const CodecParams PV, const uint16_t* __restrict__ q,
                                                            const uint16_t* __restrict__ kw,
                                                            const uint16_t* __restrict__ vw,
                                                            const int32_t* __restrict__ win_len, int win, int W_cap,
                                                            int Hq, int Hkv, float qscale, float* __restrict__ part,
                                                            int slots, int slot) {
  constexpr int E = D / 32;
  constexpr int KH = D / 8 > 16 ? 16 : D / 8;   // 16-byte key reads in flight per pass
  __shared__ float s_q[kWinMaxG][D];
  __shared__ float s_p[kWinMaxG][kWinCh];
  __shared__ float s_acc[4][kWinMaxG][D];
  __shared__ float s_m[kWinMaxG], s_al[kWinMaxG], s_l[kWinMaxG];
  // the decode kernel that follows reads nothing of this one's output: it
  // may start now (it waits for this grid before it finishes)
  asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
  const int bh = blockIdx.x, b = bh / Hkv, kvh = bh % Hkv, G = Hq / Hkv;
  const int tid = threadIdx.x, w = tid >> 5, lane = tid & 31;
  int wl = win_len ? win_len[b] : win;
  wl = wl < 0 ? 0 : (wl > W_cap ? W_cap : wl);
  for (int e = tid; e < G * D; e += 128) s_q[e / D][e % D] = h2f(q[((int64_t)b * Hq + kvh * G) * D + e]) * qscale;
  if (tid < kWinMaxG) {
    s_m[tid] = -INFINITY;
    s_l[tid] = 0.f;
  }
  float acc[kWinMaxG][E];
#pragma unroll
  for (int h = 0; h < kWinMaxG; ++h)
#pragma unroll
    for (int e = 0; e < E; ++e) acc[h][e] = 0.f;
  const uint16_t* kb = kw + ((int64_t)b * Hkv + kvh) * W_cap * D;
  const uint16_t* vb = vw + ((int64_t)b * Hkv + kvh) * W_cap * D + E * lane;
  __syncthreads();
  for (int c0 = 0; c0 < wl; c0 += kWinCh) {
    const int n = min(kWinCh, wl - c0);
    // scores: thread tid takes token c0 + tid
    float sc[kWinMaxG];
#pragma unroll
    for (int h = 0; h < kWinMaxG; ++h) sc[h] = tid < n ? 0.f : -INFINITY;
    if (tid < n) {
      const uint4* kr = reinterpret_cast<const uint4*>(kb + (int64_t)(c0 + tid) * D);
#pragma unroll
      for (int p0 = 0; p0 < D / 8; p0 += KH) {
        uint4 u[KH];
#pragma unroll
        for (int k = 0; k < KH; ++k) u[k] = kr[p0 + k];
#pragma unroll
        for (int k = 0; k < KH; ++k) {
          const uint32_t wv[4] = {u[k].x, u[k].y, u[k].z, u[k].w};
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const float2 kk = __half22float2(*reinterpret_cast<const __half2*>(&wv[j]));
            const int i = 8 * (p0 + k) + 2 * j;
#pragma unroll
            for (int h = 0; h < kWinMaxG; ++h)
              if (h < G) sc[h] = fmaf(s_q[h][i], kk.x, fmaf(s_q[h][i + 1], kk.y, sc[h]));
          }
        }
      }
    }
#pragma unroll
    for (int h = 0; h < kWinMaxG; ++h)
      if (h < G) s_p[h][tid] = sc[h];
    __syncthreads();
    // chunk maximum, new running maximum, probabilities and their sum: warp w
    // takes heads w and w + 4
    for (int h = w; h < G; h += 4) {
      float mx = -INFINITY;
#pragma unroll
      for (int k = 0; k < kWinCh / 32; ++k) mx = fmaxf(mx, s_p[h][lane + 32 * k]);
      mx = warp_max(mx);
      const float mo = s_m[h], mn = fmaxf(mo, mx);
      float sum = 0.f;
#pragma unroll
      for (int k = 0; k < kWinCh / 32; ++k) {
        const float pv = exp2f(s_p[h][lane + 32 * k] - mn);
        s_p[h][lane + 32 * k] = pv;
        sum += pv;
      }
      sum = warp_sum(sum);
      __syncwarp();
      if (lane == 0) {
        const float al = mo == -INFINITY ? 0.f : exp2f(mo - mn);
        s_al[h] = al;
        s_m[h] = mn;
        s_l[h] = s_l[h] * al + sum;
      }
    }
    __syncthreads();
    // values: warp w takes tokens w, w + 4, ...
#pragma unroll
    for (int h = 0; h < kWinMaxG; ++h) {
      const float al = h < G ? s_al[h] : 0.f;
#pragma unroll
      for (int e = 0; e < E; ++e) acc[h][e] *= al;
    }
#pragma unroll 8
    for (int t = w; t < n; t += 4) {
      float vv[E];
      const uint16_t* vr = vb + (int64_t)(c0 + t) * D;
      if (E == 8) {
        const uint4 u = *reinterpret_cast<const uint4*>(vr);
        const uint32_t wv[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&wv[j]));
          vv[2 * j] = f.x;
          vv[2 * j + 1] = f.y;
        }
      } else if (E == 4) {
        const uint2 u = *reinterpret_cast<const uint2*>(vr);
        const float2 f0 = __half22float2(*reinterpret_cast<const __half2*>(&u.x));
        const float2 f1 = __half22float2(*reinterpret_cast<const __half2*>(&u.y));
        vv[0] = f0.x; vv[1 % E] = f0.y; vv[2 % E] = f1.x; vv[3 % E] = f1.y;
      } else {
        const uint32_t u = *reinterpret_cast<const uint32_t*>(vr);
        const float2 f0 = __half22float2(*reinterpret_cast<const __half2*>(&u));
        vv[0] = f0.x; vv[1 % E] = f0.y;
      }
#pragma unroll
      for (int h = 0; h < kWinMaxG; ++h) {
        if (h < G) {
          const float pv = s_p[h][t];
#pragma unroll
          for (int e = 0; e < E; ++e) acc[h][e] = fmaf(pv, vv[e], acc[h][e]);
        }
      }
    }
    __syncthreads();   // s_p is rewritten by the next chunk
  }
#pragma unroll
  for (int h = 0; h < kWinMaxG; ++h)
#pragma unroll
    for (int e = 0; e < E; ++e)
      if (h < G) s_acc[w][h][E * lane + e] = acc[h][e];
  __syncthreads();
  // sum the warps, then into V's coded domain, one warp per head: D signs,
  // unnormalised Walsh-Hadamard per V block (in the lane below E, across
  // lanes above), then 1 / sqrt(blk)
  for (int h = w; h < G; h += 4) {
    float o[E];
#pragma unroll
    for (int e = 0; e < E; ++e) {
      const int i = E * lane + e;
      const float x = (s_acc[0][h][i] + s_acc[1][h][i]) + (s_acc[2][h][i] + s_acc[3][h][i]);
      o[e] = flip(x, (PV.sign_bits[i >> 5] >> (i & 31)) & 1u);
    }
    for (int hs = 1; hs < E && hs < PV.blk; hs <<= 1) {
#pragma unroll
      for (int e = 0; e < E; ++e) {
        if ((e & hs) == 0) {
          const float x = o[e], y = o[e + hs];
          o[e] = x + y;
          o[e + hs] = x - y;
        }
      }
    }
    for (int hs = E; hs < PV.blk; hs <<= 1) {
      const int lo = hs / E;
#pragma unroll
      for (int e = 0; e < E; ++e) {
        const float x = __shfl_xor_sync(kFull, o[e], lo);
        o[e] = (lane & lo) ? (x - o[e]) : (o[e] + x);
      }
    }
    float* dst = part + (((int64_t)b * Hq + kvh * G + h) * slots + slot) * (D + 4);
#pragma unroll
    for (int e = 0; e < E; ++e) dst[2 + E * lane + e] = o[e] * PV.inv_sqrt_blk;
    if (lane == 0) {
      dst[0] = s_m[h];
      dst[1] = s_l[h];
    }
  }
}

template <int D, int G, bool QV, bool K8>
int launch_decode(const CodecParams& PK, const CodecParams& PV, const DecodeArgs& a, int B,
                  const Codebook8Param<K8>& cbk, cudaStream_t st) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)a.n_split, (unsigned)(B * a.Hkv));
  cfg.blockDim = dim3(kDecThreads);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = a.pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, decode_split_kernel<D, G, QV, K8>, PK, PV, a, cbk) != cudaSuccess) return TQ_ERR_CUDA;
  if (cudaGetLastError() != cudaSuccess) return TQ_ERR_CUDA;
  return TQ_OK;
}

// cbk: the 256-level key table when PK.bits == 8 (values then without QJL)
template <int D>
int launch_decode_g(int G, const CodecParams& PK, const CodecParams& PV, const DecodeArgs& a, int B,
                    const Codebook8& cbk, cudaStream_t st) {
  const NoCodebook8 none{};
  if (PK.bits == 8) {
    if (PV.m) return TQ_ERR_UNSUPPORTED;
    switch (G) {
      case 1: return launch_decode<D, 1, false, true>(PK, PV, a, B, cbk, st);
      case 2: return launch_decode<D, 2, false, true>(PK, PV, a, B, cbk, st);
      case 4: return launch_decode<D, 4, false, true>(PK, PV, a, B, cbk, st);
      case 8: return launch_decode<D, 8, false, true>(PK, PV, a, B, cbk, st);
      default: return TQ_ERR_UNSUPPORTED;
    }
  }
  switch (G) {
    case 1: return PV.m ? launch_decode<D, 1, true, false>(PK, PV, a, B, none, st)
                        : launch_decode<D, 1, false, false>(PK, PV, a, B, none, st);
    case 2: return PV.m ? launch_decode<D, 2, true, false>(PK, PV, a, B, none, st)
                        : launch_decode<D, 2, false, false>(PK, PV, a, B, none, st);
    case 4: return PV.m ? launch_decode<D, 4, true, false>(PK, PV, a, B, none, st)
                        : launch_decode<D, 4, false, false>(PK, PV, a, B, none, st);
    case 8: return PV.m ? launch_decode<D, 8, true, false>(PK, PV, a, B, none, st)
                        : launch_decode<D, 8, false, false>(PK, PV, a, B, none, st);
    default: return TQ_ERR_UNSUPPORTED;
  }
}

// The split kernel over the block layout (no QJL, no 8-bit codes).
template <int D>
int launch_decode_blocks(int G, const CodecParams& PK, const CodecParams& PV, const DecodeArgs& a, int B,
                         cudaStream_t st) {
  const dim3 grid((unsigned)a.n_split, (unsigned)(B * a.Hkv));
  const NoCodebook8 none{};
  switch (G) {
    case 1: decode_split_kernel<D, 1, false, false, true><<<grid, kDecThreads, 0, st>>>(PK, PV, a, none); break;
    case 2: decode_split_kernel<D, 2, false, false, true><<<grid, kDecThreads, 0, st>>>(PK, PV, a, none); break;
    case 4: decode_split_kernel<D, 4, false, false, true><<<grid, kDecThreads, 0, st>>>(PK, PV, a, none); break;
    case 8: decode_split_kernel<D, 8, false, false, true><<<grid, kDecThreads, 0, st>>>(PK, PV, a, none); break;
    default: return TQ_ERR_UNSUPPORTED;
  }
  return cudaGetLastError() == cudaSuccess ? TQ_OK : TQ_ERR_CUDA;
}

}  // namespace

int decode_combine(const CodecParams& PV, const float* part, int n_split, uint16_t* out, int rows, cudaStream_t s) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)((rows + kCombWarps - 1) / kCombWarps));
  cfg.blockDim = dim3(kCombWarps * 32);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e;
  if (n_split > 64 / (PV.d / 32)) {   // beyond the narrow kernel's preload window
    cfg.gridDim = dim3((unsigned)rows);
    cfg.blockDim = dim3(kWideWarps * 32);
    switch (PV.d) {
      case 64: e = cudaLaunchKernelEx(&cfg, decode_combine_wide_kernel<64>, PV, part, n_split, out); break;
      case 128: e = cudaLaunchKernelEx(&cfg, decode_combine_wide_kernel<128>, PV, part, n_split, out); break;
      default: e = cudaLaunchKernelEx(&cfg, decode_combine_wide_kernel<256>, PV, part, n_split, out); break;
    }
    return e == cudaSuccess && cudaGetLastError() == cudaSuccess ? TQ_OK : TQ_ERR_CUDA;
  }
  switch (PV.d) {
    case 64: e = cudaLaunchKernelEx(&cfg, decode_combine_kernel<64>, PV, part, n_split, out, rows); break;
    case 128: e = cudaLaunchKernelEx(&cfg, decode_combine_kernel<128>, PV, part, n_split, out, rows); break;
    default: e = cudaLaunchKernelEx(&cfg, decode_combine_kernel<256>, PV, part, n_split, out, rows); break;
  }
  return e == cudaSuccess && cudaGetLastError() == cudaSuccess ? TQ_OK : TQ_ERR_CUDA;
}

int sm_count() {
  int dev = 0, sms = 152;
  if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  return sms;
}

int decode_auto_splits(int B, int Hkv, int64_t ctx, int per_sm) {
  // one wave at per_sm (default four) 4-warp CTAs per SM
  const int units = B * Hkv;
  int want = (per_sm * sm_count()) / units;
  const int64_t max_by_len = (ctx + 255) / 256;
  if (want > max_by_len) want = (int)max_by_len;
  if (want < 1) want = 1;
  if (want > 4096) want = 4096;
  return want;
}

// Split partials [B*Hq][n_split][d + 4] fp32, then (256-byte aligned) the
// tensor-core path's per-call extras (S q rows of QJL keys).
size_t decode_part_bytes(int B, int Hq, int d, int n_split) {
  return (size_t)B * Hq * n_split * (d + 4) * sizeof(float);
}

size_t decode_ws_bytes(int B, int Hq, int d, int n_split) {
  return (decode_part_bytes(B, Hq, d, n_split) + 255) / 256 * 256 + decode_tc_extra_bytes(B, Hq);
}

}  // namespace tq

extern "C" int tq_decode_workspace_bytes(int B, int Hq, int Hkv, int head_dim, int64_t ctx, int n_split,
                                         size_t* bytes, int* n_split_out) {
  if (B <= 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv || ctx < 0 || n_split < 0 || !bytes) return TQ_ERR_ARG;
  if (head_dim != 64 && head_dim != 128 && head_dim != 256) return TQ_ERR_UNSUPPORTED;
  // the layout decides the kernel and its residency; size for the most splits any choice takes
  const int per_sm = tq::decode_tc_max_ctas_per_sm() > 4 ? tq::decode_tc_max_ctas_per_sm() : 4;
  const int ns = n_split ? n_split : tq::decode_auto_splits(B, Hkv, ctx, per_sm);
  *bytes = tq::decode_ws_bytes(B, Hq, head_dim, ns);
  if (n_split_out) *n_split_out = ns;
  return TQ_OK;
}

namespace tq {
namespace {

// The fp16 residual window of a decode call (see tq_decode_attn_window).
struct Window {
  const uint16_t* k;
  const uint16_t* v;
  const int32_t* len;
  int win, W_cap;
};

int decode_impl(const tq_kv_view* K, const tq_kv_view* V, const uint16_t* q, int B, int Hq, int Hkv, int64_t S_cap,
                const int32_t* kv_len, int64_t ctx, float softmax_scale, uint16_t* out, void* workspace,
                size_t workspace_bytes, int n_split, void* stream, const Window* win) {
  if (!K || !V || !q || !out) return TQ_ERR_ARG;
  CodecParams PK, PV;
  int st = make_params(&K->layout, &PK);
  if (st != TQ_OK) return st;
  st = make_params(&V->layout, &PV);
  if (st != TQ_OK) return st;
  if (PK.d != PV.d || PV.m > kMaxQjlV) return TQ_ERR_UNSUPPORTED;
  // 8-bit codes: keys only (the value path reads 1..4-bit codes), no QJL
  // on the values beside them
  if (PV.bits > 4 || (PK.bits > 4 && PV.m)) return TQ_ERR_UNSUPPORTED;
  Codebook8 cbk;
  if (PK.bits == 8 && make_codebook8(&K->layout, &cbk) != TQ_OK) return TQ_ERR_UNSUPPORTED;
  if (B <= 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv || ctx < 0 || ctx > S_cap || n_split < 0) return TQ_ERR_ARG;
  if (!K->codes || !K->scales || !V->codes || !V->scales) return TQ_ERR_ARG;
  if (PK.m && (!K->qjl_bits || !K->qjl_rnorm || !K->S)) return TQ_ERR_ARG;
  if (PV.m && (!V->qjl_bits || !V->qjl_rnorm || !V->S)) return TQ_ERR_ARG;
  if (check_paging(K, S_cap) != TQ_OK || !same_paging(K, V)) return TQ_ERR_ARG;
  if (win && (!win->k || !win->v || win->W_cap < 0 || win->win < 0 || win->win > win->W_cap)) return TQ_ERR_ARG;
  if (win && Hq / Hkv > kWinMaxG) return TQ_ERR_UNSUPPORTED;
  if (!aligned16(K->codes) || !aligned16(V->codes) || !aligned16(q) || !aligned16(out)) return TQ_ERR_ALIGN;
  if (win && (reinterpret_cast<uintptr_t>(win->k) % 8 || reinterpret_cast<uintptr_t>(win->v) % 8))
    return TQ_ERR_ALIGN;
  const int G = Hq / Hkv;
  const bool tc = decode_tc_eligible(PK, PV, G, S_cap, K, V);
  const int ns = n_split ? n_split : decode_auto_splits(B, Hkv, ctx, tc ? decode_tc_ctas_per_sm(PK, PV) : 4);
  const int slots = ns + (win ? 1 : 0);
  const size_t need = decode_ws_bytes(B, Hq, PK.d, slots);
  if (!workspace || workspace_bytes < need) return TQ_ERR_WORKSPACE;
  if (!aligned16(workspace)) return TQ_ERR_ALIGN;
  const float sm = softmax_scale > 0.f ? softmax_scale : 1.0f / sqrtf((float)PK.d);
  DecodeArgs a{reinterpret_cast<const uint32_t*>(K->codes), K->scales,
               reinterpret_cast<const uint32_t*>(K->qjl_bits), K->qjl_rnorm, K->S,
               reinterpret_cast<const uint32_t*>(V->codes), V->scales,
               reinterpret_cast<const uint32_t*>(V->qjl_bits), V->qjl_rnorm, V->S, q, kv_len,
               static_cast<float*>(workspace),
               {K->page_table, K->page_table ? K->page_size : 0, K->page_table ? K->pages_per_seq : 0},
               S_cap, ctx, Hq, Hkv, ns, slots, sm * kLog2e, 0};
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (win) {
    // the window's partial first; the split kernel overlaps it
    const int units = B * Hkv;
    switch (PK.d) {
      case 64:
        decode_window_kernel<64><<<units, 128, 0, s>>>(PV, q, win->k, win->v, win->len, win->win, win->W_cap, Hq,
                                                       Hkv, a.qscale, a.part, slots, ns);
        break;
      case 128:
        decode_window_kernel<128><<<units, 128, 0, s>>>(PV, q, win->k, win->v, win->len, win->win, win->W_cap, Hq,
                                                        Hkv, a.qscale, a.part, slots, ns);
        break;
      default:
        decode_window_kernel<256><<<units, 128, 0, s>>>(PV, q, win->k, win->v, win->len, win->win, win->W_cap, Hq,
                                                        Hkv, a.qscale, a.part, slots, ns);
        break;
    }
    if (cudaGetLastError() != cudaSuccess) return TQ_ERR_CUDA;
    a.pdl = 1;
  }
  if (tc) {
    st = launch_decode_tc(PK, PV, K, V, q, kv_len, a.part, decode_part_bytes(B, Hq, PK.d, slots), B, Hq, Hkv, S_cap,
                          ctx, ns, slots, a.pdl != 0, a.qscale, &cbk, s);
  } else {
    switch (PK.d) {
      case 64: st = launch_decode_g<64>(G, PK, PV, a, B, cbk, s); break;
      case 128: st = launch_decode_g<128>(G, PK, PV, a, B, cbk, s); break;
      default: st = launch_decode_g<256>(G, PK, PV, a, B, cbk, s); break;
    }
  }
  if (st != TQ_OK) return st;
  return decode_combine(PV, a.part, slots, out, B * Hq, s);
}

}  // namespace
}  // namespace tq

namespace tq {
namespace {

int decode_blocks_impl(const tq_layout* Lk, const uint8_t* k_blocks, const tq_layout* Lv, const uint8_t* v_blocks,
                       const uint16_t* q, int B, int Hq, int Hkv, int64_t S_cap, const int32_t* kv_len, int64_t ctx,
                       float softmax_scale, uint16_t* out, void* workspace, size_t workspace_bytes, int n_split,
                       void* stream) {
  if (!Lk || !Lv || !q || !out) return TQ_ERR_ARG;
  CodecParams PK, PV;
  int st = make_params(Lk, &PK);
  if (st != TQ_OK) return st;
  st = make_params(Lv, &PV);
  if (st != TQ_OK) return st;
  // the block form has no QJL data; 8-bit codes are read by the packed path only
  if (PK.d != PV.d || PK.m || PV.m || PK.bits > 4 || PV.bits > 4) return TQ_ERR_UNSUPPORTED;
  if (B <= 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv || ctx < 0 || ctx > S_cap || n_split < 0) return TQ_ERR_ARG;
  if (Hq / Hkv != 1 && Hq / Hkv != 2 && Hq / Hkv != 4 && Hq / Hkv != 8) return TQ_ERR_UNSUPPORTED;
  if (!k_blocks || !v_blocks) return TQ_ERR_ARG;
  if ((reinterpret_cast<uintptr_t>(k_blocks) & 1) || (reinterpret_cast<uintptr_t>(v_blocks) & 1) ||
      !aligned16(q) || !aligned16(out))
    return TQ_ERR_ALIGN;
  const bool tc = decode_tc_blocks_eligible(PK, PV, Hq / Hkv, S_cap, k_blocks, v_blocks);
  const int ns = n_split ? n_split : decode_auto_splits(B, Hkv, ctx, tc ? decode_tc_ctas_per_sm(PK, PV) : 4);
  const size_t need = decode_ws_bytes(B, Hq, PK.d, ns);
  if (!workspace || workspace_bytes < need) return TQ_ERR_WORKSPACE;
  if (!aligned16(workspace)) return TQ_ERR_ALIGN;
  const float sm = softmax_scale > 0.f ? softmax_scale : 1.0f / sqrtf((float)PK.d);
  DecodeArgs a{};
  a.q = q;
  a.kv_len = kv_len;
  a.part = static_cast<float*>(workspace);
  a.pages = {nullptr, 0, 0};
  a.S_cap = S_cap;
  a.ctx = ctx;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.n_split = ns;
  a.slots = ns;
  a.qscale = sm * kLog2e;
  a.kblk = reinterpret_cast<const uint16_t*>(k_blocks);
  a.vblk = reinterpret_cast<const uint16_t*>(v_blocks);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int G = Hq / Hkv;
  if (tc) {
    st = launch_decode_tc_blocks(PK, PV, k_blocks, v_blocks, q, kv_len, a.part, B, Hq, Hkv, S_cap, ctx, ns, a.qscale,
                                 s);
  } else {
    switch (PK.d) {
      case 64: st = launch_decode_blocks<64>(G, PK, PV, a, B, s); break;
      case 128: st = launch_decode_blocks<128>(G, PK, PV, a, B, s); break;
      default: st = launch_decode_blocks<256>(G, PK, PV, a, B, s); break;
    }
  }
  if (st != TQ_OK) return st;
  return decode_combine(PV, a.part, ns, out, B * Hq, s);
}

}  // namespace
}  // namespace tq

extern "C" int tq_decode_attn_blocks(const tq_layout* k_layout, const uint8_t* k_blocks, const tq_layout* v_layout,
                                     const uint8_t* v_blocks, const uint16_t* q, int B, int Hq, int Hkv,
                                     int64_t S_cap, const int32_t* kv_len, int64_t ctx, float softmax_scale,
                                     uint16_t* out, void* workspace, size_t workspace_bytes, int n_split,
                                     void* stream) {
  return tq::decode_blocks_impl(k_layout, k_blocks, v_layout, v_blocks, q, B, Hq, Hkv, S_cap, kv_len, ctx,
                                softmax_scale, out, workspace, workspace_bytes, n_split, stream);
}

extern "C" int tq_decode_attn(const tq_kv_view* K, const tq_kv_view* V, const uint16_t* q, int B, int Hq,
                              int Hkv, int64_t S_cap, const int32_t* kv_len, int64_t ctx, float softmax_scale,
                              uint16_t* out, void* workspace, size_t workspace_bytes, int n_split,
                              void* stream) {
  return tq::decode_impl(K, V, q, B, Hq, Hkv, S_cap, kv_len, ctx, softmax_scale, out, workspace, workspace_bytes,
                         n_split, stream, nullptr);
}

extern "C" int tq_decode_window_workspace_bytes(int B, int Hq, int Hkv, int head_dim, int64_t ctx, int n_split,
                                                size_t* bytes) {
  int ns = 0;
  size_t b0 = 0;
  const int st = tq_decode_workspace_bytes(B, Hq, Hkv, head_dim, ctx, n_split, &b0, &ns);
  if (st != TQ_OK) return st;
  *bytes = tq::decode_ws_bytes(B, Hq, head_dim, ns + 1);
  return TQ_OK;
}

extern "C" int tq_decode_attn_window(const tq_kv_view* K, const tq_kv_view* V, const uint16_t* q, int B, int Hq,
                                     int Hkv, int64_t S_cap, const int32_t* kv_len, int64_t ctx,
                                     const uint16_t* k_win, const uint16_t* v_win, int W_cap,
                                     const int32_t* win_len, int win, float softmax_scale, uint16_t* out,
                                     void* workspace, size_t workspace_bytes, int n_split, void* stream) {
  const tq::Window w{k_win, v_win, win_len, win, W_cap};
  return tq::decode_impl(K, V, q, B, Hq, Hkv, S_cap, kv_len, ctx, softmax_scale, out, workspace, workspace_bytes,
                         n_split, stream, &w);
}

// ---------------------------------------------------------------------------
// Decode attention without any allocation by the caller or the library.
//
// Some callers cannot call cudaMalloc at the point where they decode: a
// serving runtime or plugin host that owns every device allocation through
// its own fixed pool and forbids new ones after start-up, or a hot path that
// cannot afford cudaMalloc's implicit device synchronisation.  For them the
// split-K partials live in one fixed array of device memory that belongs to
// this library.  Each GPU that loads the library keeps this array for the
// life of the process.
namespace tq {
namespace {

constexpr size_t kStaticDecodeScratch = size_t(TQ_DECODE_STATIC_SCRATCH_BYTES);
static __device__ __align__(256) unsigned char g_decode_scratch[kStaticDecodeScratch];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void* g_scratch_addr[kMaxDevices] = {};

}  // namespace
}  // namespace tq

extern "C" int tq_decode_attn_static(const tq_kv_view* K, const tq_kv_view* V, const uint16_t* q, int B, int Hq,
                                     int Hkv, int64_t S_cap, const int32_t* kv_len, int64_t ctx,
                                     float softmax_scale, uint16_t* out, int n_split, void* stream) {
  if (!K || !V) return TQ_ERR_ARG;
  size_t need = 0;
  int st = tq_decode_workspace_bytes(B, Hq, Hkv, K->layout.head_dim, ctx, n_split, &need, nullptr);
  if (st != TQ_OK) return st;
  if (need > tq::kStaticDecodeScratch) return TQ_ERR_WORKSPACE;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= tq::kMaxDevices) return TQ_ERR_CUDA;
  void* scratch = nullptr;
  {
    // Host code cannot use the array's name as a device address: ask the
    // runtime for this device's copy once, with this device current.
    std::lock_guard<std::mutex> lock(tq::g_scratch_mu);
    if (!tq::g_scratch_addr[dev]) {
      void* p = nullptr;
      if (cudaGetSymbolAddress(&p, tq::g_decode_scratch) != cudaSuccess || !p) {
        cudaGetLastError();  // leave no error behind for the caller's next launch check
        return TQ_ERR_CUDA;
      }
      tq::g_scratch_addr[dev] = p;
    }
    scratch = tq::g_scratch_addr[dev];
  }
  return tq_decode_attn(K, V, q, B, Hq, Hkv, S_cap, kv_len, ctx, softmax_scale, out, scratch,
                        tq::kStaticDecodeScratch, n_split, stream);
}
