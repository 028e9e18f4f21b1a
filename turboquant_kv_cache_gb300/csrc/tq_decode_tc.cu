// Tensor-core decode attention for the turbo3 cache (3-bit codes, one fp16
// norm per 32 values) at head_dim 128 with GQA groups of 4.
//
// Same mathematics as the CUDA-core split kernel (scores <H D q, c> scaled
// by the block norms, online softmax in base 2, V accumulated in the rotated
// domain, partials merged and rotated back by the combine kernel), mapped
// onto m16n8k16 fp16 MMAs with fp32 accumulation:
//
//  * Staging: a CTA owns (batch, KV head, context slice).  64-token tiles of
//    K codes / K scales / V codes / V scales stream into a 4-stage shared
//    memory ring with 16-byte cp.async (zero-filled past the slice).  Each of
//    the 4 warps takes 16 tokens of a tile.
//  * Code -> fp16: an 8-code chunk of the packed layout is a nibble word;
//    byte permutes against two 8-byte tables (low and high bytes of the fp16
//    centroids) give the fp16 values, four codes per two permutes.
//  * K side: lane t of a quad decodes, at step s, chunk s of group (t+s)&3,
//    so every lane runs the same instructions (chunk 3 needs the bit-3
//    gather).  The MMA columns are (head, block) pairs and q^ is masked to
//    each block's coordinates, so one accumulator collects all K tiles; the
//    epilogue weights the 4 block columns by the tokens' block norms.
//  * V side: chunks decode the same way into row fragments, movmatrix
//    transposes them into B fragments (tokens along k), and the A operand
//    holds P' = p * scaleV with rows (head, block); the accumulator entry
//    whose row block matches its column's block is the output.
//  * Softmax: the running max only moves when a score exceeds it by more
//    than 2^8 (lazy rescaling); partial (m, l, acc) per CTA go to the
//    workspace in the split-kernel format.
#include <cuda_runtime.h>
#include <math.h>

#include "tq_device.cuh"

namespace tq {

int decode_combine(const CodecParams& PV, const float* part, int n_split, uint16_t* out, int rows, cudaStream_t s);

namespace {

constexpr int kW = 4;                 // warps per CTA
constexpr int kT = kW * 32;           // threads per CTA
constexpr int kWarpTok = 32;          // tokens per warp per step (two 16-token MMA tiles)
constexpr int kTileTok = kWarpTok * kW;   // tokens per stage
constexpr int kStages = 3;
constexpr int kD = 128;
constexpr int kG = 4;                 // q heads per KV head
constexpr int kRecC = 48;             // code bytes per token (128 coords x 3 bits)
constexpr int kRecS = 8;              // scale bytes per token (4 blocks x fp16)
constexpr int kOffKc = 0;
constexpr int kOffKs = kOffKc + kTileTok * kRecC;
constexpr int kOffVc = kOffKs + kTileTok * kRecS;
constexpr int kOffVs = kOffVc + kTileTok * kRecC;
constexpr int kStageBytes = kOffVs + kTileTok * kRecS;   // 14336
constexpr float kLazy = 8.0f;         // rescale threshold, log2 units

struct TcArgs {
  const uint8_t* kc;
  const uint8_t* ks;
  const uint8_t* vc;
  const uint8_t* vs;
  const uint16_t* q;
  const int32_t* kv_len;
  float* part;
  int64_t S_cap;
  int64_t ctx;
  int64_t per;          // tokens per split (multiple of kTileTok)
  int Hq, Hkv, n_split;
  float qscale;
};

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void cp_async16(void* dst, const void* src, int bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(smem_u32(dst)), "l"(src), "r"(bytes));
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
  const __half2 r = __hmul2(*reinterpret_cast<const __half2*>(&a), *reinterpret_cast<const __half2*>(&b));
  return *reinterpret_cast<const uint32_t*>(&r);
}

__device__ __forceinline__ uint32_t pack_h2(float lo, float hi) {
  const __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}

__device__ __forceinline__ float2 unpack_h2(uint32_t v) {
  return __half22float2(*reinterpret_cast<const __half2*>(&v));
}

// Nibble words of the four 8-code chunks of one 3-bit group (words w0..w2).
// Chunk 3's bits ride in bit 3 of every nibble; the shifts of the gather are
// done as high-half multiplies so they leave the integer logic pipe.
__device__ __forceinline__ void chunks3(uint32_t w0, uint32_t w1, uint32_t w2, uint32_t* n) {
  n[0] = w0 & 0x77777777u;
  n[1] = w1 & 0x77777777u;
  n[2] = w2 & 0x77777777u;
  n[3] = __umulhi(w0 & 0x88888888u, 1u << 29) + __umulhi(w1 & 0x88888888u, 1u << 30) +
         __umulhi(w2 & 0x88888888u, 1u << 31);
}

// Byte permute with the selector taken as is: every selector here has bit 3
// of each nibble clear, so no masking is needed (the C intrinsic masks).
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

// Four fp16x2 registers (codes 0-1, 2-3, 4-5, 6-7) of a nibble word: byte
// permutes against the low-byte and high-byte tables of the fp16 centroids.
__device__ __forceinline__ void lut8(uint32_t n, uint32_t tl0, uint32_t tl1, uint32_t th0, uint32_t th1,
                                     uint32_t* o) {
  uint32_t lo = prmt(tl0, tl1, n);
  uint32_t hi = prmt(th0, th1, n);
  o[0] = prmt(lo, hi, 0x5140);
  o[1] = prmt(lo, hi, 0x7362);
  const uint32_t n2 = __umulhi(n, 1u << 16);
  lo = prmt(tl0, tl1, n2);
  hi = prmt(th0, th1, n2);
  o[2] = prmt(lo, hi, 0x5140);
  o[3] = prmt(lo, hi, 0x7362);
}

__global__ void __launch_bounds__(kT, 4) decode_tc_kernel(const CodecParams PK, const CodecParams PV, const TcArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t* ring = smem;                                                 // [kStages][kStageBytes]
  uint16_t* sPh = reinterpret_cast<uint16_t*>(smem + kStages * kStageBytes);  // [kW][kG][kWarpTok] fp16 p
  uint16_t* sVT = sPh + kW * kG * kWarpTok;                             // [kW][4 blocks][kWarpTok] fp16
  __shared__ float s_ml[kW][2][kG];

  const int split = blockIdx.x;
  const int bh = blockIdx.y;
  const int b = bh / a.Hkv, kvh = bh % a.Hkv;
  const int h0 = kvh * kG;
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const int g = lane >> 2, t = lane & 3;

  int64_t len = a.ctx;
  if (a.kv_len) len = imin64(len, (int64_t)a.kv_len[b]);
  const int64_t t_begin = (int64_t)split * a.per;
  const int64_t t_end = imin64(t_begin + a.per, len);
  const int n_tiles = t_end > t_begin ? (int)((t_end - t_begin + kTileTok - 1) / kTileTok) : 0;
  const int64_t rec0 = (int64_t)bh * a.S_cap;

  auto load_stage = [&](int slot, int tile) {
    uint8_t* dst = ring + slot * kStageBytes;
    const int64_t t0 = t_begin + (int64_t)tile * kTileTok;
    const int nv = (int)imin64(kTileTok, t_end - t0);
    // codes: 3 chunks of 16 B per token
    for (int c = tid; c < kTileTok * 3; c += kT) {
      const bool ok = c / 3 < nv;
      const int64_t off = ok ? (rec0 + t0) * kRecC + (int64_t)c * 16 : 0;
      cp_async16(dst + kOffKc + c * 16, a.kc + off, ok ? 16 : 0);
      cp_async16(dst + kOffVc + c * 16, a.vc + off, ok ? 16 : 0);
    }
    // scales: one 16 B chunk per two tokens
    if (tid < kTileTok / 2) {
      const int c = tid;
      const int bytes = (int)imin64(16, (int64_t)(nv - 2 * c) * kRecS);
      const bool ok = bytes > 0;
      const int64_t off = ok ? (rec0 + t0) * kRecS + (int64_t)c * 16 : 0;
      cp_async16(dst + kOffKs + c * 16, a.ks + off, ok ? bytes : 0);
      cp_async16(dst + kOffVs + c * 16, a.vs + off, ok ? bytes : 0);
    }
  };

  // prologue: start the first stages while the query is rotated
#pragma unroll
  for (int st = 0; st < kStages - 1; ++st) {
    if (st < n_tiles) load_stage(st, st);
    cp_commit();
  }

  // B fragments of the K side.  Lane t of a quad owns 32-block t; K tile
  // (s, half) holds chunk s, codes 4*half..4*half+3 of every block; the
  // columns are (head, block) pairs, zero unless the block is the lane's.
  // Each lane rotates its own two (head, block t) slices of q in registers:
  // q^ = H (D q) per 32-block, times softmax_scale * log2 e (K's layout).
  const float qn = PK.inv_sqrt_blk * a.qscale;
  const bool on = (g & 3) == t;
  uint32_t bq[4][2][2][2];
#pragma unroll
  for (int nt = 0; nt < 2; ++nt) {
    const int h = 2 * nt + (g >> 2);
    const uint4* qp = reinterpret_cast<const uint4*>(a.q + ((int64_t)b * a.Hq + h0 + h) * kD + 32 * t);
    const uint32_t sb = PK.sign_bits[t];
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
#pragma unroll
    for (int hs = 1; hs < 32; hs <<= 1) {
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        if ((i & hs) == 0) {
          const float x = v[i], y = v[i + hs];
          v[i] = x + y;
          v[i + hs] = x - y;
        }
      }
    }
#pragma unroll
    for (int s2 = 0; s2 < 4; ++s2)
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        const float* qh = v + 8 * s2 + 4 * half;
        bq[s2][half][nt][0] = on ? pack_h2(qh[0] * qn, qh[1] * qn) : 0u;
        bq[s2][half][nt][1] = on ? pack_h2(qh[2] * qn, qh[3] * qn) : 0u;
      }
  }
  // fp16 centroid tables: low / high bytes of codes 0-3 and 4-7
  uint32_t ktl0, ktl1, kth0, kth1, vtl0, vtl1, vth0, vth1;
  {
    uint32_t lo[2] = {0, 0}, hi[2] = {0, 0}, vlo[2] = {0, 0}, vhi[2] = {0, 0};
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const uint32_t hk = f2h(PK.centroids[k]), hv = f2h(PV.centroids[k]);
      lo[k >> 2] |= (hk & 0xffu) << (8 * (k & 3));
      hi[k >> 2] |= (hk >> 8) << (8 * (k & 3));
      vlo[k >> 2] |= (hv & 0xffu) << (8 * (k & 3));
      vhi[k >> 2] |= (hv >> 8) << (8 * (k & 3));
    }
    ktl0 = lo[0]; ktl1 = lo[1]; kth0 = hi[0]; kth1 = hi[1];
    vtl0 = vlo[0]; vtl1 = vlo[1]; vth0 = vhi[0]; vth1 = vhi[1];
  }

  // V accumulator: M tile (s, pr) = coords of chunk s, codes {2pr, 2pr+1}
  // (rows 0-7) and {2pr+4, 2pr+5} (rows 8-15) of block g/2; columns = heads.
  float acc[4][2][4];
#pragma unroll
  for (int s = 0; s < 4; ++s)
#pragma unroll
    for (int pr = 0; pr < 2; ++pr) acc[s][pr][0] = acc[s][pr][1] = acc[s][pr][2] = acc[s][pr][3] = 0.f;
  // running max per lane head (2*nt + t/2), warp-uniform; per-lane partial sums
  float m_run[2] = {-INFINITY, -INFINITY}, l_part[2] = {0.f, 0.f};
  uint16_t* myP = sPh + wid * kG * kWarpTok;
  uint16_t* myVT = sVT + wid * 4 * kWarpTok;
  const int tok0 = kWarpTok * wid;
  // per-lane byte offsets inside a stage
  const int offK = kOffKc + (tok0 + g) * kRecC + 12 * t;
  const int offKs = kOffKs + (tok0 + g) * kRecS + 4 * (t & 1);
  const int offV = kOffVc + (tok0 + g) * kRecC + 12 * t;
  const int offVs = kOffVs + (tok0 + lane) * kRecS;
  uint16_t* pW = myP + (t >> 1) * kWarpTok + g;              // p writes: head 2*nt + t/2
  const uint16_t* pR = myP + (g & 3) * kWarpTok + 2 * t;     // p reads: head g (g < 4)
  const uint16_t* vR = myVT + (g >> 1) * kWarpTok + 2 * t;   // scale pairs: block g/2

  for (int tile = 0; tile < n_tiles; ++tile) {
    cp_wait<kStages - 2>();
    __syncthreads();
    {
      const int nx = tile + kStages - 1;
      if (nx < n_tiles) load_stage(nx % kStages, nx);
      cp_commit();
    }
    const uint8_t* st = ring + (tile % kStages) * kStageBytes;
    const int64_t tbase = t_begin + (int64_t)tile * kTileTok + tok0;
    const bool partial = tbase + kWarpTok > t_end;   // only the slice's last tile

    // V scales of the warp's 32 tokens, transposed to [block][token]
    {
      const uint2 sv = *reinterpret_cast<const uint2*>(st + offVs);
      myVT[0 * kWarpTok + lane] = (uint16_t)(sv.x & 0xffffu);
      myVT[1 * kWarpTok + lane] = (uint16_t)(sv.x >> 16);
      myVT[2 * kWarpTok + lane] = (uint16_t)(sv.y & 0xffffu);
      myVT[3 * kWarpTok + lane] = (uint16_t)(sv.y >> 16);
    }

    // ---- scores S[token, (h, j)] for two 16-token tiles
    float S[2][2][2];   // [tile u][row r][nt]
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      // two accumulator chains per n tile (even / odd chunk) for more ILP
      float P[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
      float Q[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
      const uint32_t* k0 = reinterpret_cast<const uint32_t*>(st + offK + 16 * u * kRecC);
      const uint32_t* k1 = reinterpret_cast<const uint32_t*>(st + offK + (16 * u + 8) * kRecC);
      uint32_t n0[4], n1[4];
      chunks3(k0[0], k0[1], k0[2], n0);
      chunks3(k1[0], k1[1], k1[2], n1);
#pragma unroll
      for (int s = 0; s < 4; ++s) {
        uint32_t x0[4], x1[4];
        lut8(n0[s], ktl0, ktl1, kth0, kth1, x0);
        lut8(n1[s], ktl0, ktl1, kth0, kth1, x1);
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
          float* c = (s & 1) ? Q[nt] : P[nt];
          mma16816(c, x0[0], x1[0], x0[1], x1[1], bq[s][0][nt][0], bq[s][0][nt][1]);
          mma16816(c, x0[2], x1[2], x0[3], x1[3], bq[s][1][nt][0], bq[s][1][nt][1]);
        }
      }
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) P[nt][e] += Q[nt][e];
      // weight the block columns by the block norms; column pair (j0, j0+1)
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        const float2 scf = unpack_h2(*reinterpret_cast<const uint32_t*>(st + offKs + (16 * u + 8 * r) * kRecS));
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
          float v = fmaf(scf.x, P[nt][2 * r], scf.y * P[nt][2 * r + 1]);
          S[u][r][nt] = v + __shfl_xor_sync(kFull, v, 1);
        }
      }
    }
    if (partial) {
#pragma unroll
      for (int u = 0; u < 2; ++u)
#pragma unroll
        for (int r = 0; r < 2; ++r)
          if (tbase + 16 * u + g + 8 * r >= t_end) S[u][r][0] = S[u][r][1] = -INFINITY;
    }
    // ---- online softmax with lazy rescaling: the reference max moves only
    // when some score exceeds it by more than 2^8
    bool need = false;
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      const float m = fmaxf(fmaxf(S[0][0][nt], S[0][1][nt]), fmaxf(S[1][0][nt], S[1][1][nt]));
      need |= m > m_run[nt] + kLazy;
    }
    if (__any_sync(kFull, need)) {
      float al[2];
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        float m = fmaxf(fmaxf(S[0][0][nt], S[0][1][nt]), fmaxf(S[1][0][nt], S[1][1][nt]));
        m = fmaxf(m, __shfl_xor_sync(kFull, m, 4));
        m = fmaxf(m, __shfl_xor_sync(kFull, m, 8));
        m = fmaxf(m, __shfl_xor_sync(kFull, m, 16));
        const float mn = fmaxf(m_run[nt], m);
        al[nt] = (m_run[nt] == -INFINITY) ? 0.f : ex2(m_run[nt] - mn);
        m_run[nt] = mn;
        l_part[nt] *= al[nt];
      }
      // V accumulator columns are heads 2t, 2t+1 (lanes t < 2)
      const float aA = al[t & 1];
      const float aB = __shfl_xor_sync(kFull, al[t & 1], 2);
#pragma unroll
      for (int s = 0; s < 4; ++s)
#pragma unroll
        for (int pr = 0; pr < 2; ++pr) {
          acc[s][pr][0] *= aA;
          acc[s][pr][1] *= aB;
          acc[s][pr][2] *= aA;
          acc[s][pr][3] *= aB;
        }
    }
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      // no valid token seen yet implies every score here is -inf
      const float mref = m_run[nt] == -INFINITY ? 0.f : m_run[nt];
#pragma unroll
      for (int u = 0; u < 2; ++u)
#pragma unroll
        for (int r = 0; r < 2; ++r) {
          const float p = ex2(S[u][r][nt] - mref);   // -inf scores give 0
          l_part[nt] += p;
          if ((t & 1) == 0) pW[2 * nt * kWarpTok + 16 * u + 8 * r] = f2h(p);
        }
    }
    __syncwarp();
    // ---- V side: O^T[coord, h] += (V^ * scaleV)^T P, 16 tokens per k step
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      uint32_t pb0 = *reinterpret_cast<const uint32_t*>(pR + 16 * u);
      uint32_t pb1 = *reinterpret_cast<const uint32_t*>(pR + 16 * u + 8);
      if (g >= kG) pb0 = pb1 = 0u;
      const uint32_t sv01 = *reinterpret_cast<const uint32_t*>(vR + 16 * u);
      const uint32_t sv89 = *reinterpret_cast<const uint32_t*>(vR + 16 * u + 8);
      const uint32_t* v0 = reinterpret_cast<const uint32_t*>(st + offV + 16 * u * kRecC);
      const uint32_t* v1 = reinterpret_cast<const uint32_t*>(st + offV + (16 * u + 8) * kRecC);
      uint32_t n0[4], n1[4];
      chunks3(v0[0], v0[1], v0[2], n0);
      chunks3(v1[0], v1[1], v1[2], n1);
#pragma unroll
      for (int s = 0; s < 4; ++s) {
        uint32_t x0[4], x1[4];
        lut8(n0[s], vtl0, vtl1, vth0, vth1, x0);
        lut8(n1[s], vtl0, vtl1, vth0, vth1, x1);
#pragma unroll
        for (int pr = 0; pr < 2; ++pr) {
          const uint32_t a0 = hmul2(movtrans(x0[pr]), sv01);
          const uint32_t a1 = hmul2(movtrans(x0[pr + 2]), sv01);
          const uint32_t a2 = hmul2(movtrans(x1[pr]), sv89);
          const uint32_t a3 = hmul2(movtrans(x1[pr + 2]), sv89);
          mma16816(acc[s][pr], a0, a1, a2, a3, pb0, pb1);
        }
      }
    }
    __syncwarp();
  }
  // the combine kernel may be scheduled now; it waits for this grid to finish
  asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
  // full sums per head: the 8 lanes g of a (t) column hold partial sums
  float l_run[2];
#pragma unroll
  for (int nt = 0; nt < 2; ++nt) {
    float v = l_part[nt];
    v += __shfl_xor_sync(kFull, v, 4);
    v += __shfl_xor_sync(kFull, v, 8);
    v += __shfl_xor_sync(kFull, v, 16);
    l_run[nt] = v;
  }
  cp_wait<0>();
  __syncthreads();

  // ---- per-warp results to shared memory (reusing the ring), then merge
  float* sO = reinterpret_cast<float*>(ring);   // [kW][kG][kD]
  {
    float* ow = sO + wid * kG * kD;
    if (t < 2) {
      const int blk = g >> 1, e = g & 1;
#pragma unroll
      for (int s = 0; s < 4; ++s)
#pragma unroll
        for (int pr = 0; pr < 2; ++pr) {
          const int c0 = 32 * blk + 8 * s + 2 * pr + e;     // row g
          const int c1 = c0 + 4;                            // row g + 8
          ow[(2 * t) * kD + c0] = acc[s][pr][0];
          ow[(2 * t + 1) * kD + c0] = acc[s][pr][1];
          ow[(2 * t) * kD + c1] = acc[s][pr][2];
          ow[(2 * t + 1) * kD + c1] = acc[s][pr][3];
        }
    }
    if (g == 0 && (t & 1) == 0) {
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        const int h = 2 * nt + (t >> 1);
        s_ml[wid][0][h] = m_run[nt];
        s_ml[wid][1][h] = l_run[nt];
      }
    }
  }
  __syncthreads();
  for (int e = tid; e < kG * (kD + 2); e += kT) {
    const int h = e / (kD + 2), i = e % (kD + 2);
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kW; ++w) M = fmaxf(M, s_ml[w][0][h]);
    float val = 0.f;
    if (i == 0) {
      val = M;
    } else {
#pragma unroll
      for (int w = 0; w < kW; ++w) {
        const float mw = s_ml[w][0][h];
        const float wt = mw == -INFINITY ? 0.f : exp2f(mw - M);
        val += wt * (i == 1 ? s_ml[w][1][h] : sO[(w * kG + h) * kD + i - 2]);
      }
    }
    a.part[(((int64_t)b * a.Hq + h0 + h) * a.n_split + split) * (kD + 4) + i] = val;
  }
}

constexpr size_t kSmem = (size_t)kStages * kStageBytes + (size_t)kW * kG * kWarpTok * 2 +
                         (size_t)kW * 4 * kWarpTok * 2;
static_assert((size_t)kStages * kStageBytes >= (size_t)kW * kG * kD * 4, "ring too small for the merge");

}  // namespace

// Eligible: d 128, K and V 3-bit with 32-value blocks, no QJL / norm
// correction dependence (the scale is whatever is stored), 4 q heads per KV
// head, even S_cap and 16-byte aligned scale arrays.
bool decode_tc_eligible(const CodecParams& PK, const CodecParams& PV, int G, int64_t S_cap, const void* ks,
                        const void* vs) {
  return PK.d == 128 && PV.d == 128 && PK.bits == 3 && PV.bits == 3 && PK.blk == 32 && PV.blk == 32 && !PK.m &&
         !PV.m && G == kG && (S_cap % 2) == 0 && aligned16(ks) && aligned16(vs);
}

int64_t decode_tc_per_split(int64_t ctx, int n_split) {
  int64_t per = (ctx + n_split - 1) / n_split;
  per = (per + kTileTok - 1) / kTileTok * kTileTok;
  return per > 0 ? per : kTileTok;
}

int launch_decode_tc(const CodecParams& PK, const CodecParams& PV, const uint8_t* kc, const uint16_t* ks,
                     const uint8_t* vc, const uint16_t* vs, const uint16_t* q, const int32_t* kv_len, float* part,
                     int B, int Hq, int Hkv, int64_t S_cap, int64_t ctx, int n_split, float qscale,
                     uint16_t* out, cudaStream_t st) {
  static bool attr_set[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return TQ_ERR_CUDA;
  if (!attr_set[dev]) {
    if (cudaFuncSetAttribute(decode_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmem) !=
        cudaSuccess)
      return TQ_ERR_CUDA;
    attr_set[dev] = true;
  }
  TcArgs a{kc, reinterpret_cast<const uint8_t*>(ks), vc, reinterpret_cast<const uint8_t*>(vs), q, kv_len, part,
           S_cap, ctx, decode_tc_per_split(ctx, n_split), Hq, Hkv, n_split, qscale};
  dim3 grid(n_split, B * Hkv);
  decode_tc_kernel<<<grid, kT, kSmem, st>>>(PK, PV, a);
  if (cudaGetLastError() != cudaSuccess) return TQ_ERR_CUDA;
  return decode_combine(PV, part, n_split, out, B * Hq, st);
}

}  // namespace tq
