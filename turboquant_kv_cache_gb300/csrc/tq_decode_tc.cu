// Tensor-core decode attention over the packed cache, GQA groups of 4.
//
// Same mathematics as the CUDA-core split kernel (scores <H D q, c> times the
// block norms, plus the QJL term for QJL keys; online softmax in base 2; V
// accumulated in the rotated domain; partials merged and rotated back by the
// combine kernel), mapped onto m16n8k16 fp16 MMAs with fp32 accumulation.
//
//  * Work split: a CTA owns (batch, KV head, context slice).  A pipeline of
//    one warp (head_dim 128) or two warps (head_dim 256, each taking 128
//    dimensions and exchanging partial scores through shared memory) walks
//    32-token steps of the slice; the CTA's pipelines interleave the steps.
//  * Staging: each pipeline streams its own steps (K codes, K norms, QJL
//    bits and rho, V codes, V norms) into a 3-slot ring with 16-byte
//    cp.async, two steps ahead of the one being computed.  Past the end of
//    the slice the copies zero-fill.
//  * Code -> fp16: an 8-code chunk of the packed layout is a nibble word;
//    byte permutes against the low-byte and high-byte tables of the fp16
//    centroids give four codes per two permutes (16-entry tables for 4-bit
//    codes pick between two 8-entry halves by bit 3).  With one norm per 32
//    values the tables of a (token, block) are the centroids times that
//    norm (built once per block); 4-bit codes multiply by the norm after the
//    lookup instead; per-vector norms multiply the score (K) or p (V).
//  * K side: lane t of a quad decodes 32-block t of tokens g and g+8 of a
//    16-token MMA tile; the B operand is q^ of head (g & 3), so every lane
//    ends with the scores of its own two heads.  QJL sign bits enter as a
//    second accumulator whose A operand is 2*s (0 or 2.0, built from the bit
//    word by a shift and a mask) against S q.
//  * V side: the same decode into row fragments, movmatrix transposes them
//    into A fragments with tokens along k, B holds p (fp16) of the head
//    columns; the accumulator columns of a lane are the heads of its scores.
//  * Softmax: the running max only moves when a score exceeds it by more
//    than 2^8 (lazy rescaling); partial (m, l, acc) per CTA go to the
//    workspace in the split-kernel format.
#include <cuda_runtime.h>
#include <math.h>

#include <type_traits>

#include "tq_device.cuh"
#include "tq_lut.cuh"

namespace tq {

int decode_combine(const CodecParams& PV, const float* part, int n_split, uint16_t* out, int rows, cudaStream_t s);

namespace {

constexpr int kG = 4;          // q heads per KV head
constexpr int kTok = 32;       // tokens per step
constexpr int kThreads = 128;  // 4 warps
constexpr int kSlots = 3;
constexpr int kQjlM = 128;     // QJL rows supported here
constexpr float kLazy = 8.0f;  // rescale threshold, log2 units

// AOS: the caches are arrays of 32-value blocks, [fp16 norm | packed codes of
// the group] (2 + 4*bits bytes), a token's blocks contiguous; a token's record
// holds its norms, so there is no separate norm stream.
// QV: values with a QJL residual (m = 128, one norm per vector, head_dim 128).
template <int D, int KB, int VB, bool KPV, bool VPV, bool QJL, bool AOS = false, bool QV = false>
struct Cfg {
  static constexpr int NH = D / 128;  // warps per pipeline
  static constexpr int P = 4 / NH;    // pipelines per CTA
  static constexpr int KBB = 2 + 4 * KB, VBB = 2 + 4 * VB;   // block bytes (AOS)
  static constexpr int KREC = AOS ? (D / 32) * KBB : D * KB / 8;
  static constexpr int KSB = AOS ? 0 : (KPV ? 2 : D / 16);
  static constexpr int QB = QJL ? kQjlM / 8 : 0;
  static constexpr int QR = QJL ? 2 : 0;
  static constexpr int VREC = AOS ? (D / 32) * VBB : D * VB / 8;
  static constexpr int VSB = AOS ? 0 : (VPV ? 2 : D / 16);
  static constexpr int OKC = 0;
  static constexpr int OKS = OKC + kTok * KREC;
  static constexpr int OQB = OKS + kTok * KSB;
  static constexpr int OQR = OQB + kTok * QB;
  static constexpr int OVC = OQR + kTok * QR;
  static constexpr int OVS = OVC + kTok * VREC;
  static constexpr int VQB = QV ? kQjlM / 8 : 0;   // V QJL sign bits per token
  static constexpr int VQR = QV ? 2 : 0;           // V rho per token
  static constexpr int OVQ = OVS + kTok * VSB;
  static constexpr int OVR = OVQ + kTok * VQB;
  static constexpr int STAGE = OVR + kTok * VQR;
  static constexpr int MINB = QV ? 3 : 4;          // CTAs per SM the register budget is cut for
  static constexpr size_t K8OFF = (size_t)P * kSlots * STAGE + (size_t)4 * kG * kTok * 2 +
                                  (NH > 1 ? (size_t)4 * 32 * 8 * 4 : 0);
  static constexpr size_t SMEM = K8OFF                             // rings, p per warp, score exchange
                                 + (KB == 8 ? (size_t)256 * 32 * 4 : 0);   // 8-bit key table, one copy per lane
  static_assert(STAGE % 16 == 0 && OVC % 16 == 0, "stage sub-arrays stay 16-byte aligned");
  static_assert((size_t)P * kSlots * STAGE >= (size_t)P * kG * D * 4 + (QV ? (size_t)(P + 2) * kG * kQjlM * 4 : 0),
                "ring too small for the merge");
};

// fp16 centroids of the 256-level key codebook (8-bit keys only)
struct K8Tab {
  uint16_t c[256];
};
struct NoK8Tab {};
template <int KB>
using K8Param = typename std::conditional<KB == 8, K8Tab, NoK8Tab>::type;

struct TcArgs {
  const uint8_t* kc;
  const uint8_t* ks;
  const uint8_t* kq;   // QJL bits
  const uint8_t* kr;   // QJL rho
  const uint8_t* vc;
  const uint8_t* vs;
  const uint8_t* vq;   // V QJL bits
  const uint8_t* vr;   // V QJL rho
  const float* Sv;     // V's QJL matrix [128][D]
  const uint16_t* q;
  const uint16_t* sq;  // S q * scale, fp16 [B*Hq][128] (QJL)
  const float* sqsum;  // per-head sum of sq (QJL)
  const int32_t* kv_len;
  float* part;
  PageMap pages;       // paging of both caches (table NULL: contiguous)
  int64_t S_cap;
  int64_t ctx;
  int64_t per;  // tokens per split (multiple of 128)
  int Hq, Hkv, n_split;
  int slots;    // split slots per row of the partials (n_split, or more for extra partials)
  int pdl;      // launched as a programmatic dependent of the kernel before it
  float qscale;
};

__device__ __forceinline__ uint32_t su32(const void* p) { return static_cast<uint32_t>(__cvta_generic_to_shared(p)); }
__device__ __forceinline__ void cp16(uint32_t dst, const void* src, int bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src), "r"(bytes));
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;\n" ::); }
template <int N>
__device__ __forceinline__ void cp_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N));
}
__device__ __forceinline__ void mma16816(float* c, uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                                         uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t movtrans(uint32_t x) {
  uint32_t y;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;\n" : "=r"(y) : "r"(x));
  return y;
}
__device__ __forceinline__ uint32_t hmul2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
// Byte permute with the selector taken as is (the C intrinsic masks it).
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ uint32_t lds32(uint32_t a) {
  uint32_t v;
  asm volatile("ld.shared.b32 %0, [%1];" : "=r"(v) : "r"(a));
  return v;
}
__device__ __forceinline__ uint32_t lds16(uint32_t a) {
  unsigned short v;
  asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(a));
  return v;
}
__device__ __forceinline__ uint2 lds64(uint32_t a) {
  uint2 v;
  asm volatile("ld.shared.v2.b32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(a));
  return v;
}
__device__ __forceinline__ uint4 lds128(uint32_t a) {
  uint4 v;
  asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a));
  return v;
}
__device__ __forceinline__ void sts16(uint32_t a, uint32_t v) {
  asm volatile("st.shared.u16 [%0], %1;" ::"r"(a), "h"((unsigned short)v));
}
__device__ __forceinline__ void sts128f(uint32_t a, float x, float y, float z, float w) {
  asm volatile("st.shared.v4.f32 [%0], {%1,%2,%3,%4};" ::"r"(a), "f"(x), "f"(y), "f"(z), "f"(w));
}
__device__ __forceinline__ float4 lds128f(uint32_t a) {
  float4 v;
  asm volatile("ld.shared.v4.f32 {%0,%1,%2,%3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(a));
  return v;
}
// Named barrier of the two warps of pipeline pi (ids 1 and 2; 0 is __syncthreads).
__device__ __forceinline__ void pair_sync(int pi) {
  if (pi == 0)
    asm volatile("bar.sync 1, 64;" ::: "memory");
  else
    asm volatile("bar.sync 2, 64;" ::: "memory");
}
__device__ __forceinline__ uint32_t pack_h2(float lo, float hi) {
  const __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}
__device__ __forceinline__ float2 unpack_h2(uint32_t v) {
  return __half22float2(*reinterpret_cast<const __half2*>(&v));
}

// One step (kTok tokens) of a per-token stream of BYTES bytes per token,
// as 16-byte copies spread over the pipeline's 32 * NH lanes.
template <int BYTES, int NH>
__device__ __forceinline__ void copy_full(uint32_t dst, const uint8_t* src, int plane) {
  if (BYTES == 0) return;
  constexpr int CH = kTok * BYTES / 16, STEP = 32 * NH;
#pragma unroll
  for (int k = 0; k < (CH + STEP - 1) / STEP; ++k) {
    const int c = plane + k * STEP;
    if (CH % STEP == 0 || c < CH) cp16(dst + 16 * c, src + 16 * c, 16);
  }
}

// The same for a step with only nv valid tokens: the rest is zero-filled.
template <int BYTES, int NH>
__device__ __forceinline__ void copy_part(uint32_t dst, const uint8_t* base, int64_t tok0, int nv, int plane) {
  if (BYTES == 0) return;
  constexpr int CH = kTok * BYTES / 16, STEP = 32 * NH;
  const uint8_t* src = base + tok0 * BYTES;
#pragma unroll
  for (int k = 0; k < (CH + STEP - 1) / STEP; ++k) {
    const int c = plane + k * STEP;
    if (CH % STEP == 0 || c < CH) {
      int bytes = nv * BYTES - 16 * c;
      bytes = bytes < 0 ? 0 : (bytes > 16 ? 16 : bytes);
      cp16(dst + 16 * c, bytes ? src + 16 * c : base, bytes);
    }
  }
}

// The packed words of a 32-code group at shared address `addr`; with AOS the
// group's codes follow its 2-byte norm, so they start 2 bytes past a word
// boundary for every other group (sh = 2): bits+1 aligned words and a byte
// permute per word.
template <int BITS, bool AOS>
__device__ __forceinline__ void group_words(uint32_t addr, uint32_t* w) {
  if (!AOS) {
    load_group<BITS>(addr, w);
  } else {
    const uint32_t base = addr & ~3u, sh = addr & 3u;
    uint32_t x[BITS + 1];
#pragma unroll
    for (int i = 0; i <= BITS; ++i) x[i] = lds32(base + 4 * i);
#pragma unroll
    for (int i = 0; i < BITS; ++i) w[i] = sh ? prmt(x[i], x[i + 1], 0x5432u) : x[i];
  }
}

template <int D, int KB, int VB, bool KPV, bool VPV, bool QJL, bool AOS = false, bool QV = false>
__global__ void __launch_bounds__(kThreads, Cfg<D, KB, VB, KPV, VPV, QJL, AOS, QV>::MINB)
    decode_tc_kernel(const CodecParams PK, const CodecParams PV, const TcArgs a, const K8Param<KB> k8) {
  using C = Cfg<D, KB, VB, KPV, VPV, QJL, AOS, QV>;
  constexpr int NH = C::NH, P = C::P;
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ float s_ml[4][2][kG];

  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, tid = threadIdx.x;
  const int g = lane >> 2, t = lane & 3;
  const int pi = wid / NH, hw = wid % NH;  // pipeline, dimension half
  const int split = blockIdx.x, bh = blockIdx.y;
  const int b = bh / a.Hkv, kvh = bh % a.Hkv, h0 = kvh * kG;

  int64_t len = a.ctx;
  if (a.kv_len) len = imin64(len, (int64_t)a.kv_len[b]);
  const int64_t t_begin = (int64_t)split * a.per;
  const int64_t t_end = imin64(t_begin + a.per, len);
  const int n_sub = t_end > t_begin ? (int)((t_end - t_begin + kTok - 1) / kTok) : 0;
  const int n_it = n_sub > pi ? (n_sub - pi + P - 1) / P : 0;
  const uint32_t ring = su32(smem) + pi * kSlots * C::STAGE;
  const int plane = hw * 32 + lane;  // lane within the pipeline

  // ---- staging: every 16-byte chunk of every stream of a step, spread over
  // the pipeline's lanes; zero-filled past the end of the slice
  int ld_it = 0;
  auto load_next = [&](int slot) {
    const int64_t t0 = t_begin + (int64_t)kTok * (pi + P * ld_it);
    // a step never crosses a page: steps and pages are both 32-token aligned
    const int64_t tok0 = cache_rec(a.pages, a.Hkv, a.S_cap, b, kvh, t0);
    const uint32_t dst = ring + slot * C::STAGE;
    const int64_t rem = t_end - t0;
    if (rem >= kTok) {
      copy_full<C::KREC, NH>(dst + C::OKC, a.kc + tok0 * C::KREC, plane);
      copy_full<C::KSB, NH>(dst + C::OKS, a.ks + tok0 * C::KSB, plane);
      if (QJL) {
        copy_full<C::QB, NH>(dst + C::OQB, a.kq + tok0 * C::QB, plane);
        copy_full<C::QR, NH>(dst + C::OQR, a.kr + tok0 * C::QR, plane);
      }
      copy_full<C::VREC, NH>(dst + C::OVC, a.vc + tok0 * C::VREC, plane);
      copy_full<C::VSB, NH>(dst + C::OVS, a.vs + tok0 * C::VSB, plane);
      if (QV) {
        copy_full<C::VQB, NH>(dst + C::OVQ, a.vq + tok0 * C::VQB, plane);
        copy_full<C::VQR, NH>(dst + C::OVR, a.vr + tok0 * C::VQR, plane);
      }
    } else {
      const int nv = (int)rem;
      copy_part<C::KREC, NH>(dst + C::OKC, a.kc, tok0, nv, plane);
      copy_part<C::KSB, NH>(dst + C::OKS, a.ks, tok0, nv, plane);
      if (QJL) {
        copy_part<C::QB, NH>(dst + C::OQB, a.kq, tok0, nv, plane);
        copy_part<C::QR, NH>(dst + C::OQR, a.kr, tok0, nv, plane);
      }
      copy_part<C::VREC, NH>(dst + C::OVC, a.vc, tok0, nv, plane);
      copy_part<C::VSB, NH>(dst + C::OVS, a.vs, tok0, nv, plane);
      if (QV) {
        copy_part<C::VQB, NH>(dst + C::OVQ, a.vq, tok0, nv, plane);
        copy_part<C::VQR, NH>(dst + C::OVR, a.vr, tok0, nv, plane);
      }
    }
    ++ld_it;
  };
#pragma unroll
  for (int s = 0; s < kSlots - 1; ++s) {
    if (s < n_it) load_next(s);
    cp_commit();
  }

  // ---- q^ = H (D q) of head (g & 3) over this lane's 32-block, times
  // softmax_scale * log2 e (K's layout), as B fragments
  uint32_t bq[4][2][2];
  {
    const float qn = PK.inv_sqrt_blk * a.qscale;
    const int blk = 4 * hw + t;  // the lane's 32-value group
    const uint4* qp = reinterpret_cast<const uint4*>(a.q + ((int64_t)b * a.Hq + h0 + (g & 3)) * D + 32 * blk);
    const uint32_t sb = PK.sign_bits[blk];
    float v[32];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const uint4 u = qp[k];
      const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 f = unpack_h2(w[e]);
        v[8 * k + 2 * e] = flip(f.x, (sb >> (8 * k + 2 * e)) & 1u);
        v[8 * k + 2 * e + 1] = flip(f.y, (sb >> (8 * k + 2 * e + 1)) & 1u);
      }
    }
    // Walsh-Hadamard over the block (when the K block is the whole vector,
    // the cross-block stages follow below through shuffles)
#pragma unroll
    for (int hs = 1; hs < 32; hs <<= 1)
#pragma unroll
      for (int i = 0; i < 32; ++i)
        if ((i & hs) == 0) {
          const float x = v[i], y = v[i + hs];
          v[i] = x + y;
          v[i + hs] = x - y;
        }
    if (KPV) {
      // blocks of 128 (head_dim 128): butterflies across the quad's lanes
#pragma unroll
      for (int o = 1; o < 4; o <<= 1)
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const float p = __shfl_xor_sync(kFull, v[i], o);
          v[i] = (t & o) ? (p - v[i]) : (v[i] + p);
        }
    }
#pragma unroll
    for (int s2 = 0; s2 < 4; ++s2)
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        const float* qh = v + 8 * s2 + 4 * half;
        bq[s2][half][0] = pack_h2(qh[0] * qn, qh[1] * qn);
        bq[s2][half][1] = pack_h2(qh[2] * qn, qh[3] * qn);
      }
  }
  // QJL: B fragments of S q for rows (32t + p, 32t + p + 16), and the sums
  uint32_t bj[QJL ? 8 : 1][2];
  float sqs[2] = {0.f, 0.f};
  if (QJL) {
    asm volatile("griddepcontrol.wait;\n" ::: "memory");
    const uint16_t* sq = a.sq + ((int64_t)b * a.Hq + h0 + (g & 3)) * kQjlM + 32 * t;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      bj[j][0] = (uint32_t)sq[2 * j] | ((uint32_t)sq[2 * j + 16] << 16);
      bj[j][1] = (uint32_t)sq[2 * j + 1] | ((uint32_t)sq[2 * j + 17] << 16);
    }
    sqs[0] = a.sqsum[(int64_t)b * a.Hq + h0 + ((2 * t) & 3)];
    sqs[1] = a.sqsum[(int64_t)b * a.Hq + h0 + ((2 * t + 1) & 3)];
  }

  // 8-bit keys: centroid c of lane l at k8base + 128 c + 4 l (fp16 in the low half)
  uint32_t k8base = 0;
  if constexpr (KB == 8) {
    k8base = su32(smem + C::K8OFF);
    uint32_t* t8 = reinterpret_cast<uint32_t*>(smem + C::K8OFF);
    for (int e = tid; e < 256 * 32; e += kThreads) t8[e] = k8.c[e >> 5];
    __syncthreads();
    k8base += 4u * lane;
  }
  const Cent<KB == 8 ? 4 : KB> kcent = make_cent<KB == 8 ? 4 : KB>(PK);
  const Cent<VB> vcent = make_cent<VB>(PV);
  const uint32_t one_h = 0x3C00u;
  // tables that do not depend on the token
  Tab kfix, vfix;
  if (KPV || KB == 4) kfix = make_tab<KB == 8 ? 4 : KB>(kcent, one_h);
  if (VPV) vfix = make_tab<VB>(vcent, one_h);

  float acc[4][2][4];
#pragma unroll
  for (int s = 0; s < 4; ++s)
#pragma unroll
    for (int pr = 0; pr < 2; ++pr) acc[s][pr][0] = acc[s][pr][1] = acc[s][pr][2] = acc[s][pr][3] = 0.f;
  // QV: Z[j][head] = sum_t rho_t (2 s_tj - 1) p_t norm_t, rows j in 8 tiles of 16
  // (same fragment layout as acc: row 16 mt + g (+8), heads of columns 2t, 2t+1)
  float zq[QV ? 8 : 1][4];
#pragma unroll
  for (int mt = 0; mt < (QV ? 8 : 1); ++mt) zq[mt][0] = zq[mt][1] = zq[mt][2] = zq[mt][3] = 0.f;
  // running max / partial sums of the lane's heads 2(t&1), 2(t&1)+1
  float m_run[2] = {-INFINITY, -INFINITY}, l_part[2] = {0.f, 0.f};
  const uint32_t pBase = su32(smem + (size_t)P * kSlots * C::STAGE) + wid * kG * kTok * 2;
  const uint32_t pW = pBase + 2 * ((2 * (t & 1)) * kTok + g);
  const uint32_t pR = pBase + 2 * ((g & 3) * kTok + 2 * t);
  const uint32_t xBase = su32(smem + (size_t)P * kSlots * C::STAGE + 4 * kG * kTok * 2);
  const int grp = 4 * hw + t;  // the lane's 32-value group of K and V

  for (int it = 0; it < n_it; ++it) {
    const int slot = it % kSlots;
    cp_wait<kSlots - 2>();
    if (NH > 1) pair_sync(pi); else __syncwarp();
    // both warps are past the previous step: its slot takes the next load
    if (it + kSlots - 1 < n_it) load_next((it + kSlots - 1) % kSlots);
    cp_commit();
    const uint32_t st = ring + slot * C::STAGE;
    const int64_t tbase = t_begin + (int64_t)kTok * (pi + P * it);

    // ---- scores: S[u][r][c] for token 16u + 8r + g, head 2(t&1) + c
    float S[2][2][2];
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      float Pm[4] = {0.f, 0.f, 0.f, 0.f};
      float Pq[4] = {0.f, 0.f, 0.f, 0.f};
      const int tok0 = 16 * u + g, tok1 = tok0 + 8;
      uint32_t w0[KB == 8 ? 8 : 4], w1[KB == 8 ? 8 : 4], n0[4], n1[4];
      if constexpr (KB == 8) {
        // one byte per code: the group's 32 codes are 32 bytes
        const uint32_t a0 = st + C::OKC + tok0 * C::KREC + grp * 32, a1 = st + C::OKC + tok1 * C::KREC + grp * 32;
        const uint4 u0 = lds128(a0), u1 = lds128(a0 + 16), v0 = lds128(a1), v1 = lds128(a1 + 16);
        w0[0] = u0.x; w0[1] = u0.y; w0[2] = u0.z; w0[3] = u0.w; w0[4] = u1.x; w0[5] = u1.y; w0[6] = u1.z; w0[7] = u1.w;
        w1[0] = v0.x; w1[1] = v0.y; w1[2] = v0.z; w1[3] = v0.w; w1[4] = v1.x; w1[5] = v1.y; w1[6] = v1.z; w1[7] = v1.w;
      } else {
        group_words<KB, AOS>(st + C::OKC + tok0 * C::KREC + (AOS ? grp * C::KBB + 2 : grp * 4 * KB), w0);
        group_words<KB, AOS>(st + C::OKC + tok1 * C::KREC + (AOS ? grp * C::KBB + 2 : grp * 4 * KB), w1);
        chunk_words<KB>(w0, n0);
        chunk_words<KB>(w1, n1);
      }
      // the group's norm: its block header (AOS) or the norm stream
      auto knorm = [&](int tok) {
        return lds16(AOS ? st + C::OKC + tok * C::KREC + grp * C::KBB : st + C::OKS + tok * C::KSB + 2 * grp);
      };
      Tab T0, T1;
      uint32_t s0h = 0, s1h = 0;
      if (KPV || KB == 4 || KB == 8) {
        T0 = kfix;
        T1 = kfix;
        if (!KPV) {
          s0h = knorm(tok0);
          s1h = knorm(tok1);
          s0h |= s0h << 16;
          s1h |= s1h << 16;
        }
      } else {
        T0 = make_tab<KB == 8 ? 4 : KB>(kcent, knorm(tok0));
        T1 = make_tab<KB == 8 ? 4 : KB>(kcent, knorm(tok1));
      }
#pragma unroll
      for (int s = 0; s < 4; ++s) {
        uint32_t x0[4], x1[4];
        if constexpr (KB == 8) {
          // codes 8s .. 8s+7 are bytes of words 2s, 2s+1; each pair of
          // table words gives an fp16 pair (low halves)
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const uint32_t wa = w0[2 * s + (e >> 1)], wb = w1[2 * s + (e >> 1)];
            const int sh = 16 * (e & 1);
            const uint32_t lo0 = lds32(k8base + (((wa >> sh) & 0xFFu) << 7));
            const uint32_t hi0 = lds32(k8base + (((wa >> (sh + 8)) & 0xFFu) << 7));
            const uint32_t lo1 = lds32(k8base + (((wb >> sh) & 0xFFu) << 7));
            const uint32_t hi1 = lds32(k8base + (((wb >> (sh + 8)) & 0xFFu) << 7));
            x0[e] = prmt(lo0, hi0, 0x5410u);
            x1[e] = prmt(lo1, hi1, 0x5410u);
          }
        } else {
          lut8<KB>(n0[s], T0, x0);
          lut8<KB>(n1[s], T1, x1);
        }
        if ((KB == 4 || KB == 8) && !KPV) {
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            x0[e] = hmul2(x0[e], s0h);
            x1[e] = hmul2(x1[e], s1h);
          }
        }
        mma16816(Pm, x0[0], x1[0], x0[1], x1[1], bq[s][0][0], bq[s][0][1]);
        mma16816(Pm, x0[2], x1[2], x0[3], x1[3], bq[s][1][0], bq[s][1][1]);
      }
      if (QJL) {
        const uint32_t q0 = lds32(st + C::OQB + tok0 * C::QB + 4 * t);
        const uint32_t q1 = lds32(st + C::OQB + tok1 * C::QB + 4 * t);
        // 2*s as fp16 (0 or 2.0): bits p and p+16 land on bits 14 and 30
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const int p0 = 2 * j, p1 = 2 * j + 1;
          const uint32_t a0 = (p0 <= 14 ? (q0 << (14 - p0)) : (q0 >> (p0 - 14))) & 0x40004000u;
          const uint32_t a2 = (p1 <= 14 ? (q0 << (14 - p1)) : (q0 >> (p1 - 14))) & 0x40004000u;
          const uint32_t a1 = (p0 <= 14 ? (q1 << (14 - p0)) : (q1 >> (p0 - 14))) & 0x40004000u;
          const uint32_t a3 = (p1 <= 14 ? (q1 << (14 - p1)) : (q1 >> (p1 - 14))) & 0x40004000u;
          mma16816(Pq, a0, a1, a2, a3, bj[j][0], bj[j][1]);
        }
      }
      if (KPV) {
        // one norm per vector (AOS: every block header holds it; block 0's)
        const float sc0 = h2f((uint16_t)lds16(AOS ? st + C::OKC + tok0 * C::KREC : st + C::OKS + tok0 * C::KSB));
        const float sc1 = h2f((uint16_t)lds16(AOS ? st + C::OKC + tok1 * C::KREC : st + C::OKS + tok1 * C::KSB));
        if (QJL) {
          const float r0 = sc0 * h2f((uint16_t)lds16(st + C::OQR + tok0 * 2));
          const float r1 = sc1 * h2f((uint16_t)lds16(st + C::OQR + tok1 * 2));
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            S[u][0][c] = fmaf(r0, Pq[c] - sqs[c], sc0 * Pm[c]);
            S[u][1][c] = fmaf(r1, Pq[2 + c] - sqs[c], sc1 * Pm[2 + c]);
          }
        } else {
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            S[u][0][c] = sc0 * Pm[c];
            S[u][1][c] = sc1 * Pm[2 + c];
          }
        }
      } else {
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          S[u][0][c] = Pm[c];
          S[u][1][c] = Pm[2 + c];
        }
      }
    }
    if (NH > 1) {
      // the other half of the dimensions: same lane of the partner warp
      const uint32_t mine = xBase + ((pi * 2 + hw) * 32 + lane) * 32;
      const uint32_t other = xBase + ((pi * 2 + (hw ^ 1)) * 32 + lane) * 32;
      sts128f(mine, S[0][0][0], S[0][0][1], S[0][1][0], S[0][1][1]);
      sts128f(mine + 16, S[1][0][0], S[1][0][1], S[1][1][0], S[1][1][1]);
      pair_sync(pi);
      const float4 o0 = lds128f(other), o1 = lds128f(other + 16);
      S[0][0][0] += o0.x; S[0][0][1] += o0.y; S[0][1][0] += o0.z; S[0][1][1] += o0.w;
      S[1][0][0] += o1.x; S[1][0][1] += o1.y; S[1][1][0] += o1.z; S[1][1][1] += o1.w;
    }
    if (tbase + kTok > t_end) {  // the slice's last step
#pragma unroll
      for (int u = 0; u < 2; ++u)
#pragma unroll
        for (int r = 0; r < 2; ++r)
          if (tbase + 16 * u + 8 * r + g >= t_end) S[u][r][0] = S[u][r][1] = -INFINITY;
    }

    // ---- online softmax with lazy rescaling
    bool need = false;
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      const float m = fmaxf(fmaxf(S[0][0][c], S[0][1][c]), fmaxf(S[1][0][c], S[1][1][c]));
      need |= m > m_run[c] + kLazy;
    }
    if (__any_sync(kFull, need)) {
      float al[2];
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        float m = fmaxf(fmaxf(S[0][0][c], S[0][1][c]), fmaxf(S[1][0][c], S[1][1][c]));
        m = fmaxf(m, __shfl_xor_sync(kFull, m, 4));
        m = fmaxf(m, __shfl_xor_sync(kFull, m, 8));
        m = fmaxf(m, __shfl_xor_sync(kFull, m, 16));
        const float mn = fmaxf(m_run[c], m);
        al[c] = (m_run[c] == -INFINITY) ? 0.f : ex2(m_run[c] - mn);
        m_run[c] = mn;
        l_part[c] *= al[c];
      }
#pragma unroll
      for (int s = 0; s < 4; ++s)
#pragma unroll
        for (int pr = 0; pr < 2; ++pr) {
          acc[s][pr][0] *= al[0];
          acc[s][pr][1] *= al[1];
          acc[s][pr][2] *= al[0];
          acc[s][pr][3] *= al[1];
        }
      if (QV) {
#pragma unroll
        for (int mt = 0; mt < 8; ++mt) {
          zq[mt][0] *= al[0];
          zq[mt][1] *= al[1];
          zq[mt][2] *= al[0];
          zq[mt][3] *= al[1];
        }
      }
    }
#pragma unroll
    for (int u = 0; u < 2; ++u)
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        float vs = 1.f;
        if (VPV)
          vs = h2f((uint16_t)lds16(AOS ? st + C::OVC + (16 * u + 8 * r + g) * C::VREC
                                       : st + C::OVS + (16 * u + 8 * r + g) * C::VSB));
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          // no valid token seen yet implies every score here is -inf
          const float mref = m_run[c] == -INFINITY ? 0.f : m_run[c];
          const float p = ex2(S[u][r][c] - mref);
          l_part[c] += p;
          if (t < 2) sts16(pW + 2 * (c * kTok + 16 * u + 8 * r), f2h(VPV ? p * vs : p));
        }
      }
    __syncwarp();

    // ---- V side: O^T[coord, head] += V^T P, 16 tokens per k step
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const uint32_t pb0 = lds32(pR + 2 * 16 * u);
      const uint32_t pb1 = lds32(pR + 2 * (16 * u + 8));
      const int tok0 = 16 * u + g, tok1 = tok0 + 8;
      uint32_t w0[4], w1[4], n0[4], n1[4];
      group_words<VB, AOS>(st + C::OVC + tok0 * C::VREC + (AOS ? grp * C::VBB + 2 : grp * 4 * VB), w0);
      group_words<VB, AOS>(st + C::OVC + tok1 * C::VREC + (AOS ? grp * C::VBB + 2 : grp * 4 * VB), w1);
      chunk_words<VB>(w0, n0);
      chunk_words<VB>(w1, n1);
      Tab T0, T1;
      if (VPV) {
        T0 = vfix;
        T1 = vfix;
      } else {
        T0 = make_tab<VB>(vcent, lds16(AOS ? st + C::OVC + tok0 * C::VREC + grp * C::VBB
                                           : st + C::OVS + tok0 * C::VSB + 2 * grp));
        T1 = make_tab<VB>(vcent, lds16(AOS ? st + C::OVC + tok1 * C::VREC + grp * C::VBB
                                           : st + C::OVS + tok1 * C::VSB + 2 * grp));
      }
#pragma unroll
      for (int s = 0; s < 4; ++s) {
        uint32_t x0[4], x1[4];
        lut8<VB>(n0[s], T0, x0);
        lut8<VB>(n1[s], T1, x1);
#pragma unroll
        for (int pr = 0; pr < 2; ++pr)
          mma16816(acc[s][pr], movtrans(x0[pr]), movtrans(x0[pr + 2]), movtrans(x1[pr]), movtrans(x1[pr + 2]), pb0,
                   pb1);
      }
      if constexpr (QV) {
        // A = rho_t (2 s_tj - 1) as fp16, rows j, columns the tokens of this
        // k step: the lane's columns are tokens ta, ta+1 and tb, tb+1.  Sign
        // word w of a token shifted so that bit 32 w + 8 k + g lands on bit
        // 8 k + 7; a byte permute brings the bits of two tokens to bits 15 and
        // 31, and one logic op keeps them inverted (set where s = 0) and signs
        // the rho pair with them.
        const int ta = 16 * u + 2 * t, tb = ta + 8;
        const uint32_t ra = lds32(st + C::OVR + 2 * ta), rb = lds32(st + C::OVR + 2 * tb);
        const uint4 qa0 = lds128(st + C::OVQ + 16 * ta), qa1 = lds128(st + C::OVQ + 16 * (ta + 1));
        const uint4 qb0 = lds128(st + C::OVQ + 16 * tb), qb1 = lds128(st + C::OVQ + 16 * (tb + 1));
        const uint32_t sh = 7 - g;
        const uint32_t wa0[4] = {qa0.x, qa0.y, qa0.z, qa0.w}, wa1[4] = {qa1.x, qa1.y, qa1.z, qa1.w};
        const uint32_t wb0[4] = {qb0.x, qb0.y, qb0.z, qb0.w}, wb1[4] = {qb1.x, qb1.y, qb1.z, qb1.w};
#pragma unroll
        for (int wi = 0; wi < 4; ++wi) {
          const uint32_t xa0 = wa0[wi] << sh, xa1 = wa1[wi] << sh;
          const uint32_t xb0 = wb0[wi] << sh, xb1 = wb1[wi] << sh;
#pragma unroll
          for (int hf = 0; hf < 2; ++hf) {   // row tiles mt = 2 wi + hf: rows 32 wi + 16 hf + g (+8)
            const int mt = 2 * wi + hf, k0 = 2 * hf, k1 = 2 * hf + 1;
            // result bytes 1 and 3 take byte k of the first and second token
            const uint32_t s0 = (uint32_t)((4 + k0) << 12 | k0 << 4), s1 = (uint32_t)((4 + k1) << 12 | k1 << 4);
            const uint32_t r0 = (~prmt(xa0, xa1, s0) & 0x80008000u) ^ ra;   // row 16 mt + g, tokens ta, ta+1
            const uint32_t r1 = (~prmt(xa0, xa1, s1) & 0x80008000u) ^ ra;   // row + 8
            const uint32_t r2 = (~prmt(xb0, xb1, s0) & 0x80008000u) ^ rb;   // row, tokens tb, tb+1
            const uint32_t r3 = (~prmt(xb0, xb1, s1) & 0x80008000u) ^ rb;
            mma16816(zq[mt], r0, r1, r2, r3, pb0, pb1);
          }
        }
      }
    }
    __syncwarp();
  }
  // the combine kernel may be scheduled now; it waits for this grid to finish
  asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");

  // ---- merge the pipelines through shared memory, then write the partial
  float l_run[2];
#pragma unroll
  for (int c = 0; c < 2; ++c) {
    float v = l_part[c];
    v += __shfl_xor_sync(kFull, v, 4);
    v += __shfl_xor_sync(kFull, v, 8);
    v += __shfl_xor_sync(kFull, v, 16);
    l_run[c] = v;
  }
  cp_wait<0>();
  __syncthreads();
  float* sO = reinterpret_cast<float*>(smem);  // [P][kG][D]
  {
    float* ow = sO + pi * kG * D;
    if (t < 2) {
      // accumulator row g of tile (s, pr): coordinate of the transposed
      // fragment, lane t's columns are heads 2t, 2t+1
      const int blk = 4 * hw + (g >> 1), e = g & 1;
#pragma unroll
      for (int s = 0; s < 4; ++s)
#pragma unroll
        for (int pr = 0; pr < 2; ++pr) {
          const int c0 = 32 * blk + 8 * s + 2 * pr + e;
          const int c1 = c0 + 4;
          ow[(2 * t) * D + c0] = acc[s][pr][0];
          ow[(2 * t + 1) * D + c0] = acc[s][pr][1];
          ow[(2 * t) * D + c1] = acc[s][pr][2];
          ow[(2 * t + 1) * D + c1] = acc[s][pr][3];
        }
    }
    if (hw == 0 && g == 0 && t < 2) {
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        s_ml[pi][0][2 * t + c] = m_run[c];
        s_ml[pi][1][2 * t + c] = l_run[c];
      }
    }
    if (QV && t < 2) {
      float* zw = sO + P * kG * D + pi * kG * kQjlM;   // [P][kG][128]
#pragma unroll
      for (int mt = 0; mt < (QV ? 8 : 0); ++mt) {
        const int j = 16 * mt + g;
        zw[(2 * t) * kQjlM + j] = zq[mt][0];
        zw[(2 * t + 1) * kQjlM + j] = zq[mt][1];
        zw[(2 * t) * kQjlM + j + 8] = zq[mt][2];
        zw[(2 * t + 1) * kQjlM + j + 8] = zq[mt][3];
      }
    }
  }
  __syncthreads();
  // QV: the pipelines' sign sums merged with the softmax weights, then
  // sqrt(pi/2)/m S^T of them (input domain), then into V's coded domain: D
  // signs and the block's Walsh-Hadamard transform over sqrt(blk)
  float* s_prj = sO + P * kG * D + P * kG * kQjlM + kG * kQjlM;   // [kG][D]
  if constexpr (QV) {
    float* s_az = sO + P * kG * D + P * kG * kQjlM;              // [kG][128]
    const float* zs = sO + P * kG * D;
    for (int e = tid; e < kG * kQjlM; e += kThreads) {
      const int h = e / kQjlM;
      float M = -INFINITY;
#pragma unroll
      for (int w = 0; w < P; ++w) M = fmaxf(M, s_ml[w][0][h]);
      float v = 0.f;
#pragma unroll
      for (int w = 0; w < P; ++w) {
        const float mw = s_ml[w][0][h];
        v += (mw == -INFINITY ? 0.f : exp2f(mw - M)) * zs[w * kG * kQjlM + e];
      }
      s_az[e] = v;
    }
    __syncthreads();
    // warp w: rows 32 w .. 32 w + 31 of S, lane l: columns 4 l .. 4 l + 3;
    // the four warps' partial products meet in the (now free) sign-sum area
    static_assert(kThreads == 128 && kG == 4 && D == 128 && kQjlM == 128, "QV layout: 4 warps x 32 rows x 128 columns");
    float* red = sO + P * kG * D;   // [4 warps][kG][D]
    {
      const int j0 = 32 * wid, c0 = 4 * lane;
      const float4* sp = reinterpret_cast<const float4*>(a.Sv + (int64_t)j0 * D + c0);
      float v[kG][4] = {};
#pragma unroll 8
      for (int jj = 0; jj < 32; ++jj) {
        const float4 s4 = __ldg(sp + jj * (D / 4));
#pragma unroll
        for (int h = 0; h < kG; ++h) {
          const float z = s_az[h * kQjlM + j0 + jj];
          v[h][0] = fmaf(s4.x, z, v[h][0]);
          v[h][1] = fmaf(s4.y, z, v[h][1]);
          v[h][2] = fmaf(s4.z, z, v[h][2]);
          v[h][3] = fmaf(s4.w, z, v[h][3]);
        }
      }
#pragma unroll
      for (int h = 0; h < kG; ++h) sts128f(su32(red + (wid * kG + h) * D + c0), v[h][0], v[h][1], v[h][2], v[h][3]);
    }
    __syncthreads();
    // warp h: head h.  Sum the partials, sqrt(pi/2)/m, V's signs D, then the
    // unnormalised 128-point Walsh-Hadamard (one V block per vector): strides
    // 1 and 2 inside the lane, 4 .. 64 across lanes
    {
      const int h = wid, c0 = 4 * lane;
      const float coef = kSqrtHalfPi / (float)kQjlM;
      const uint32_t sb = PV.sign_bits[c0 >> 5] >> (c0 & 31);
      float x[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        float v = 0.f;
#pragma unroll
        for (int w = 0; w < 4; ++w) v += red[(w * kG + h) * D + c0 + e];
        x[e] = flip(v * coef, (sb >> e) & 1u);
      }
      float y0 = x[0] + x[1], y1 = x[0] - x[1], y2 = x[2] + x[3], y3 = x[2] - x[3];
      x[0] = y0 + y2;
      x[2] = y0 - y2;
      x[1] = y1 + y3;
      x[3] = y1 - y3;
#pragma unroll
      for (int m = 1; m < 32; m <<= 1) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float o = __shfl_xor_sync(kFull, x[e], m);
          x[e] = (lane & m) ? o - x[e] : x[e] + o;
        }
      }
      sts128f(su32(s_prj + h * D + c0), x[0], x[1], x[2], x[3]);
    }
    __syncthreads();
  }
  for (int e = tid; e < kG * (D + 2); e += kThreads) {
    const int h = e / (D + 2), i = e % (D + 2);
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < P; ++w) M = fmaxf(M, s_ml[w][0][h]);
    float val = 0.f;
    if (i == 0) {
      val = M;
    } else {
#pragma unroll
      for (int w = 0; w < P; ++w) {
        const float mw = s_ml[w][0][h];
        const float wt = mw == -INFINITY ? 0.f : exp2f(mw - M);
        val += wt * (i == 1 ? s_ml[w][1][h] : sO[(w * kG + h) * D + i - 2]);
      }
      if (QV && i >= 2) val += s_prj[h * D + i - 2] * PV.inv_sqrt_blk;
    }
    a.part[(((int64_t)b * a.Hq + h0 + h) * a.slots + split) * (D + 4) + i] = val;
  }
  // finish only after the kernel this one may overlap (a no-op otherwise)
  asm volatile("griddepcontrol.wait;\n" ::: "memory");
}

// S q of every (batch, q head) for QJL keys, times softmax_scale * log2 e *
// sqrt(pi/2) / m, rounded to fp16, and the sum of each row of it.  One CTA
// per (batch, KV head) serves its 4 q heads; thread i owns row i of S.  The
// decode launched after it may start at once (its CTAs stage their first
// cache steps, then wait for this grid to finish before reading S q); the
// whole row of S is loaded before q, one round trip for both.
template <int D>
__global__ void __launch_bounds__(kQjlM) qjl_prep_kernel(const uint16_t* __restrict__ q, const float* __restrict__ S,
                                                         float coef, uint16_t* __restrict__ sq,
                                                         float* __restrict__ sqsum) {
  asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
  __shared__ __align__(16) float s_q[kG][D];
  __shared__ float s_red[kG][kQjlM / 32];
  const int grp = blockIdx.x, i = threadIdx.x;  // rows grp*4 .. grp*4+3 of q
  float4 sr[D / 4];
  const float4* Si = reinterpret_cast<const float4*>(S + (int64_t)i * D);
#pragma unroll
  for (int j4 = 0; j4 < D / 4; ++j4) sr[j4] = __ldg(Si + j4);
  for (int e = i; e < kG * D; e += kQjlM) s_q[e / D][e % D] = h2f(q[(int64_t)grp * kG * D + e]);
  __syncthreads();
  float v[kG] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int j4 = 0; j4 < D / 4; ++j4) {
    const float4 sv = sr[j4];
#pragma unroll
    for (int h = 0; h < kG; ++h) {
      const float4 qh = *reinterpret_cast<const float4*>(s_q[h] + 4 * j4);
      v[h] = fmaf(sv.x, qh.x, fmaf(sv.y, qh.y, fmaf(sv.z, qh.z, fmaf(sv.w, qh.w, v[h]))));
    }
  }
#pragma unroll
  for (int h = 0; h < kG; ++h) {
    const uint16_t hv = f2h(v[h] * coef);
    sq[((int64_t)grp * kG + h) * kQjlM + i] = hv;
    float r = h2f(hv);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) r += __shfl_xor_sync(kFull, r, o);
    if ((i & 31) == 0) s_red[h][i >> 5] = r;
  }
  __syncthreads();
  if (i < kG) {
    float tot = 0.f;
#pragma unroll
    for (int w = 0; w < kQjlM / 32; ++w) tot += s_red[i][w];
    sqsum[(int64_t)grp * kG + i] = tot;
  }
}

template <int D, int KB, int VB, bool KPV, bool VPV, bool QJL, bool AOS = false, bool QV = false>
int launch_cfg(const CodecParams& PK, const CodecParams& PV, const TcArgs& a, int B, cudaStream_t st,
               const K8Param<KB>& k8 = K8Param<KB>{}) {
  using C = Cfg<D, KB, VB, KPV, VPV, QJL, AOS, QV>;
  auto kern = decode_tc_kernel<D, KB, VB, KPV, VPV, QJL, AOS, QV>;
  static bool attr_set[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return TQ_ERR_CUDA;
  if (!attr_set[dev]) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::SMEM) != cudaSuccess)
      return TQ_ERR_CUDA;
    attr_set[dev] = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)a.n_split, (unsigned)(B * a.Hkv));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = C::SMEM;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = (QJL || a.pdl) ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, kern, PK, PV, a, k8) != cudaSuccess) return TQ_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? TQ_OK : TQ_ERR_CUDA;
}

}  // namespace

// Eligible layouts: head_dim 128 or 256 with 4 q heads per KV head; K codes
// of 2-4 bits, V codes of 3 bits, each with one norm per 32 values or per
// vector (the combinations instantiated below); 8-bit K with 4-bit V, one
// norm per 32 values, at head_dim 128; QJL keys with m = 128 on
// 2-bit per-vector K at head_dim 128; values with a QJL residual (m = 128)
// on 2- or 3-bit per-vector V at head_dim 128, beside 2-bit per-vector K with
// or without QJL keys; every array 16-byte aligned and every per-token
// stream's row pitch (S_cap times its bytes per token) a multiple of 16.
bool decode_tc_eligible(const CodecParams& PK, const CodecParams& PV, int G, int64_t S_cap, const tq_kv_view* K,
                        const tq_kv_view* V) {
  if (G != kG || PK.d != PV.d || (PK.d != 128 && PK.d != 256)) return false;
  const bool kpv = PK.blk == PK.d, vpv = PV.blk == PV.d;
  // 8-bit keys beside 4-bit values (k8v4), one norm per 32 values, head_dim 128
  const bool k8v4 = PK.bits == 8 && PV.bits == 4 && PK.d == 128 && PK.blk == 32 && PV.blk == 32 && !PK.m && !PV.m;
  // values with a QJL residual: m = 128, one norm per vector, 2- or 3-bit
  // codes, beside 2-bit per-vector keys (with or without QJL keys of m = 128)
  const bool qv = PV.m != 0;
  if (qv && !(PV.m == kQjlM && vpv && PK.d == 128 && (PV.bits == 2 || PV.bits == 3) && kpv && PK.bits == 2 &&
              (!PK.m || PK.m == kQjlM)))
    return false;
  if (PV.bits != 3 && !k8v4 && !qv) return false;
  // every per-token stream must keep 16-byte aligned rows for cp.async
  const int64_t streams[8] = {PK.code_bytes, 2 * PK.nb,       PK.qjl_bytes, PK.m ? 2 : 0,
                              PV.code_bytes, 2 * PV.nb,       PV.qjl_bytes, PV.m ? 2 : 0};
  // (a paged cache's rows are its pages)
  const int64_t row = K->page_table ? K->page_size : S_cap;
  for (int i = 0; i < 8; ++i)
    if ((row * streams[i]) % 16 != 0) return false;
  if ((!kpv && PK.blk != 32) || (!vpv && PV.blk != 32)) return false;
  bool ok;
  if (k8v4 || qv) {
    ok = true;
  } else if (PK.d == 256) {
    ok = !kpv && !vpv && !PK.m && PK.bits >= 2 && PK.bits <= 4;
  } else if (PK.m) {
    ok = PK.m == kQjlM && kpv && vpv && PK.bits == 2;
  } else if (kpv) {
    ok = PK.bits == 2;
  } else {
    ok = PK.bits == 3 || ((PK.bits == 2 || PK.bits == 4) && !vpv);
  }
  if (!ok) return false;
  if (!aligned16(K->codes) || !aligned16(K->scales) || !aligned16(V->codes) || !aligned16(V->scales)) return false;
  if (PK.m && (!aligned16(K->qjl_bits) || !aligned16(K->qjl_rnorm) || !K->S || !aligned16(K->S))) return false;
  if (PV.m && (!aligned16(V->qjl_bits) || !aligned16(V->qjl_rnorm) || !V->S || !aligned16(V->S))) return false;
  return true;
}

// CTAs of the kernel resident per SM (the register budget it is built for).
int decode_tc_ctas_per_sm(const CodecParams& PK, const CodecParams& PV) {
  if (PV.m) return Cfg<128, 2, 2, true, true, false, false, true>::MINB;
  if (PK.bits == 8) return Cfg<128, 8, 4, false, false, false>::MINB;
  return Cfg<128, 2, 3, true, true, false>::MINB;
}
// The most any layout uses: the split count a workspace is sized for.
int decode_tc_max_ctas_per_sm() {
  const int a = Cfg<128, 2, 2, true, true, false, false, true>::MINB, b = Cfg<128, 8, 4, false, false, false>::MINB,
            c = Cfg<128, 2, 3, true, true, false>::MINB;
  return a > b ? (a > c ? a : c) : (b > c ? b : c);
}

int64_t decode_tc_per_split(int64_t ctx, int n_split) {
  int64_t per = (ctx + n_split - 1) / n_split;
  per = (per + kThreads - 1) / kThreads * kThreads;
  return per > 0 ? per : kThreads;
}

// Extra workspace after the partials: S q rows and their sums (QJL keys).
size_t decode_tc_extra_bytes(int B, int Hq) {
  return (size_t)B * Hq * (kQjlM * 2 + 4) + 256;
}

// Writes the partials of splits 0 .. n_split-1 into rows of `slots` slots;
// the caller merges them (decode_combine).
int launch_decode_tc(const CodecParams& PK, const CodecParams& PV, const tq_kv_view* K, const tq_kv_view* V,
                     const uint16_t* q, const int32_t* kv_len, float* part, size_t part_bytes, int B, int Hq, int Hkv,
                     int64_t S_cap, int64_t ctx, int n_split, int slots, bool pdl, float qscale, const Codebook8* cbk,
                     cudaStream_t st) {
  TcArgs a{};
  a.kc = K->codes;
  a.ks = reinterpret_cast<const uint8_t*>(K->scales);
  a.kq = K->qjl_bits;
  a.kr = reinterpret_cast<const uint8_t*>(K->qjl_rnorm);
  a.vc = V->codes;
  a.vs = reinterpret_cast<const uint8_t*>(V->scales);
  a.vq = V->qjl_bits;
  a.vr = reinterpret_cast<const uint8_t*>(V->qjl_rnorm);
  a.Sv = V->S;
  a.q = q;
  a.kv_len = kv_len;
  a.part = part;
  a.pages = {K->page_table, K->page_table ? K->page_size : 0, K->page_table ? K->pages_per_seq : 0};
  a.S_cap = S_cap;
  a.ctx = ctx;
  a.per = decode_tc_per_split(ctx, n_split);
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.n_split = n_split;
  a.slots = slots;
  a.pdl = pdl ? 1 : 0;
  a.qscale = qscale;
  if (PK.m) {
    uint8_t* extra = reinterpret_cast<uint8_t*>(part) + ((part_bytes + 255) / 256) * 256;
    uint16_t* sq = reinterpret_cast<uint16_t*>(extra);
    float* sqsum = reinterpret_cast<float*>(extra + (((size_t)B * Hq * kQjlM * 2 + 15) / 16) * 16);
    a.sq = sq;
    a.sqsum = sqsum;
    if (PK.d != 128) return TQ_ERR_UNSUPPORTED;
    qjl_prep_kernel<128><<<B * Hkv, kQjlM, 0, st>>>(q, K->S, qscale * kSqrtHalfPi / (float)PK.m, sq, sqsum);
    if (cudaGetLastError() != cudaSuccess) return TQ_ERR_CUDA;
  }
  const bool kpv = PK.blk == PK.d, vpv = PV.blk == PV.d;
  int r;
  if (PK.bits == 8) {
    if (!cbk) return TQ_ERR_ARG;
    K8Tab tab;
    for (int k = 0; k < 256; ++k) {
      const __half h = __float2half_rn(cbk->c[k]);
      tab.c[k] = *reinterpret_cast<const uint16_t*>(&h);
    }
    r = launch_cfg<128, 8, 4, false, false, false>(PK, PV, a, B, st, tab);
  } else if (PK.d == 256) {
    r = PK.bits == 4 ? launch_cfg<256, 4, 3, false, false, false>(PK, PV, a, B, st)
        : PK.bits == 3 ? launch_cfg<256, 3, 3, false, false, false>(PK, PV, a, B, st)
                       : launch_cfg<256, 2, 3, false, false, false>(PK, PV, a, B, st);
  } else if (PV.m) {
    if (PK.m)
      r = PV.bits == 2 ? launch_cfg<128, 2, 2, true, true, true, false, true>(PK, PV, a, B, st)
                       : launch_cfg<128, 2, 3, true, true, true, false, true>(PK, PV, a, B, st);
    else
      r = PV.bits == 2 ? launch_cfg<128, 2, 2, true, true, false, false, true>(PK, PV, a, B, st)
                       : launch_cfg<128, 2, 3, true, true, false, false, true>(PK, PV, a, B, st);
  } else if (PK.m) {
    r = launch_cfg<128, 2, 3, true, true, true>(PK, PV, a, B, st);
  } else if (kpv) {
    r = vpv ? launch_cfg<128, 2, 3, true, true, false>(PK, PV, a, B, st)
            : launch_cfg<128, 2, 3, true, false, false>(PK, PV, a, B, st);
  } else {
    r = PK.bits == 4 ? launch_cfg<128, 4, 3, false, false, false>(PK, PV, a, B, st)
        : PK.bits == 3 ? (vpv ? launch_cfg<128, 3, 3, false, true, false>(PK, PV, a, B, st)
                              : launch_cfg<128, 3, 3, false, false, false>(PK, PV, a, B, st))
                       : launch_cfg<128, 2, 3, false, false, false>(PK, PV, a, B, st);
  }
  return r;
}

// The block form (arrays of [fp16 norm | packed codes] 32-value blocks) on
// the same kernel: head_dim 128 or 256, 4 q heads per KV head, K codes of 2-4
// bits and V codes of 3 bits with one norm per 32 values, contiguous caches
// whose arrays are 16-byte aligned with 16-byte multiples of row pitch.
bool decode_tc_blocks_eligible(const CodecParams& PK, const CodecParams& PV, int G, int64_t S_cap,
                               const uint8_t* k_blocks, const uint8_t* v_blocks) {
  if (G != kG || PK.d != PV.d || (PK.d != 128 && PK.d != 256) || PV.bits != 3 || PK.bits < 2 || PK.bits > 4)
    return false;
  if (PK.blk != 32 || PV.blk != 32 || PK.m || PV.m) return false;
  const int64_t krec = (int64_t)(PK.d / 32) * (2 + 4 * PK.bits), vrec = (int64_t)(PV.d / 32) * (2 + 4 * PV.bits);
  if ((S_cap * krec) % 16 || (S_cap * vrec) % 16) return false;
  return aligned16(k_blocks) && aligned16(v_blocks);
}

int launch_decode_tc_blocks(const CodecParams& PK, const CodecParams& PV, const uint8_t* k_blocks,
                            const uint8_t* v_blocks, const uint16_t* q, const int32_t* kv_len, float* part, int B,
                            int Hq, int Hkv, int64_t S_cap, int64_t ctx, int n_split, float qscale, cudaStream_t st) {
  TcArgs a{};
  a.kc = k_blocks;
  a.vc = v_blocks;
  a.q = q;
  a.kv_len = kv_len;
  a.part = part;
  a.pages = {nullptr, 0, 0};
  a.S_cap = S_cap;
  a.ctx = ctx;
  a.per = decode_tc_per_split(ctx, n_split);
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.n_split = n_split;
  a.slots = n_split;
  a.pdl = 0;
  a.qscale = qscale;
  if (PK.d == 256) {
    return PK.bits == 4 ? launch_cfg<256, 4, 3, false, false, false, true>(PK, PV, a, B, st)
           : PK.bits == 3 ? launch_cfg<256, 3, 3, false, false, false, true>(PK, PV, a, B, st)
                          : launch_cfg<256, 2, 3, false, false, false, true>(PK, PV, a, B, st);
  }
  return PK.bits == 4 ? launch_cfg<128, 4, 3, false, false, false, true>(PK, PV, a, B, st)
         : PK.bits == 3 ? launch_cfg<128, 3, 3, false, false, false, true>(PK, PV, a, B, st)
                        : launch_cfg<128, 2, 3, false, false, false, true>(PK, PV, a, B, st);
}

}  // namespace tq
