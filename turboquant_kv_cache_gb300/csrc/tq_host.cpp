// Host layer of libtq: the Lloyd-Max codebook solver, the sign vector,
// layout checks and sizes, status strings.  Pure C++ (no device code).
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>
#include <cstring>
#include <mutex>
#include <utility>

#include "tq_internal.h"

namespace tq {
namespace {

constexpr int kMaxBits = 8;                 // host codebooks: 1..8 bits
constexpr int kMaxLevels = 1 << kMaxBits;
constexpr double kInvSqrt2 = 0.70710678118654752440;
constexpr double kInvSqrt2Pi = 0.39894228040143267794;

double density(double t) { return std::isinf(t) ? 0.0 : kInvSqrt2Pi * std::exp(-0.5 * t * t); }

// P(a < Z <= b) for a standard normal Z, written with erfc so that both
// tails keep their relative precision.
double cell_mass(double a, double b) {
  if (b <= 0.0) return cell_mass(-b, -a);
  if (a >= 0.0) return 0.5 * (std::erfc(a * kInvSqrt2) - std::erfc(b * kInvSqrt2));
  return 1.0 - 0.5 * std::erfc(-a * kInvSqrt2) - 0.5 * std::erfc(b * kInvSqrt2);
}

// Lloyd-Max quantiser of the standard normal with `levels` outputs: the
// fixed point of "boundaries = midpoints, centroids = conditional means"
// ("TurboQuant From Scratch", section 2, step 3).  The iteration starts from
// evenly spaced levels on [-2, 2]; for a log-concave density the fixed point
// is unique, so the start only affects the iteration count.  Up to 16 levels.
void solve_unit_codebook_lloyd(int levels, double* c) {
  for (int k = 0; k < levels; ++k) c[k] = levels == 1 ? 0.0 : -2.0 + 4.0 * k / (levels - 1);
  double edge[17];
  double last = INFINITY;
  for (int it = 0; it < 1000000; ++it) {
    edge[0] = -INFINITY;
    edge[levels] = INFINITY;
    for (int k = 1; k < levels; ++k) edge[k] = 0.5 * (c[k - 1] + c[k]);
    double moved = 0.0;
    for (int k = 0; k < levels; ++k) {
      const double next = (density(edge[k]) - density(edge[k + 1])) / cell_mass(edge[k], edge[k + 1]);
      moved = std::fmax(moved, std::fabs(next - c[k]));
      c[k] = next;
    }
    // Linear convergence: run to the fixed point, i.e. until nothing moves
    // or the step stalls at rounding level.
    if (moved == 0.0 || (moved < 1e-15 && moved >= last)) break;
    last = moved;
  }
}

// x with P(Z <= x) = p for a standard normal Z, by bisection on erfc (only
// used for a starting point, so speed does not matter).
double normal_quantile(double p) {
  double lo = -40.0, hi = 40.0;
  for (int it = 0; it < 200 && hi - lo > 1e-15; ++it) {
    const double mid = 0.5 * (lo + hi);
    if (0.5 * std::erfc(-mid * kInvSqrt2) < p) lo = mid; else hi = mid;
  }
  return 0.5 * (lo + hi);
}

// The same fixed point for many levels (256 at 8 bits), where the Lloyd
// iteration's linear rate is far too slow: Newton's method on
// F_k(c) = m_k(c) - c_k, m_k the mean of cell [l_k, u_k] whose edges are the
// midpoints to the neighbouring centroids.  With P the cell's mass,
// dm/du = phi(u) (u - m) / P and dm/dl = phi(l) (m - l) / P, and each edge
// moves by half of a neighbour's step, so the Jacobian is tridiagonal and
// each step is one forward/backward sweep.  Starting point: the centroid
// density of high-resolution quantisation theory (proportional to the cube
// root of the source density, i.e. N(0, 3) quantiles).
void solve_unit_codebook_newton(int levels, double* c) {
  double lo[kMaxLevels], di[kMaxLevels], up[kMaxLevels], rhs[kMaxLevels];
  for (int k = 0; k < levels; ++k) c[k] = std::sqrt(3.0) * normal_quantile((k + 0.5) / levels);
  double last = INFINITY;
  for (int it = 0; it < 500; ++it) {
    for (int k = 0; k < levels; ++k) {
      const double l = k == 0 ? -INFINITY : 0.5 * (c[k - 1] + c[k]);
      const double u = k + 1 == levels ? INFINITY : 0.5 * (c[k] + c[k + 1]);
      const double P = cell_mass(l, u);
      const double m = (density(l) - density(u)) / P;
      const double dmu = std::isinf(u) ? 0.0 : density(u) * (u - m) / P;
      const double dml = std::isinf(l) ? 0.0 : density(l) * (m - l) / P;
      lo[k] = 0.5 * dml;
      up[k] = 0.5 * dmu;
      di[k] = 0.5 * (dml + dmu) - 1.0;
      rhs[k] = c[k] - m;
    }
    for (int k = 1; k < levels; ++k) {
      const double w = lo[k] / di[k - 1];
      di[k] -= w * up[k - 1];
      rhs[k] -= w * rhs[k - 1];
    }
    double moved = 0.0, next = 0.0;
    for (int k = levels - 1; k >= 0; --k) {
      const double step = (rhs[k] - (k + 1 < levels ? up[k] * next : 0.0)) / di[k];
      next = step;
      c[k] += step;
      moved = std::fmax(moved, std::fabs(step));
    }
    // quadratic convergence until rounding level, then stop once the step
    // no longer shrinks
    if (moved == 0.0 || (moved < 1e-15 && moved >= last)) break;
    last = moved;
  }
}

void solve_unit_codebook(int levels, double* c) {
  if (levels <= 16) solve_unit_codebook_lloyd(levels, c);
  else solve_unit_codebook_newton(levels, c);
  // The density is symmetric, so is the exact codebook; symmetrise away the
  // rounding residue so that the middle boundary is exactly zero.
  double sym[kMaxLevels];
  for (int k = 0; k < levels; ++k) sym[k] = 0.5 * (c[k] - c[levels - 1 - k]);
  for (int k = 0; k < levels; ++k) c[k] = sym[k];
}

// Lloyd-Max quantiser of one coordinate of a uniformly random unit vector
// in R^blk: density f(x) = (1 - x^2)^a / B(1/2, a + 1) on [-1, 1] with
// a = (blk - 3)/2, i.e. (x + 1)/2 ~ Beta((blk - 1)/2, (blk - 1)/2)
// (llama.cpp-turboquant, "How it works": the exact Beta distribution of
// the rotated coordinates).  blk is even here, so a is a half-integer and
// J_p(x) = int_0^x (1 - t^2)^p dt follows from J_{1/2}(x) =
// (x sqrt(1 - x^2) + asin x)/2 by J_p = x (1 - x^2)^p / (2p + 1) +
// 2p/(2p + 1) J_{p-1}, every term positive for x >= 0.  The first moment of a
// cell is exact: int x (1 - x^2)^a dx = -(1 - x^2)^(a + 1) / (2 (a + 1)).
double beta_J(double x, double a) {
  const double ax = std::fabs(x);
  const double w = std::fmax(0.0, 1.0 - ax * ax);
  const double sw = std::sqrt(w);
  double J = 0.5 * (ax * sw + std::asin(std::fmin(ax, 1.0)));
  double wp = w * sw;   // w^p, p = 3/2, 5/2, ...
  for (double p = 1.5; p <= a + 1e-9; p += 1.0, wp *= w) J = ax * wp / (2.0 * p + 1.0) + (2.0 * p / (2.0 * p + 1.0)) * J;
  return x < 0.0 ? -J : J;
}

// One Lloyd step for the Beta density: boundaries at midpoints, centroids
// the conditional means of their cells.
void beta_lloyd_step(int levels, double a, double norm, const double* c, double* out) {
  double edge[17];
  edge[0] = -1.0;
  edge[levels] = 1.0;
  for (int k = 1; k < levels; ++k) edge[k] = 0.5 * (c[k - 1] + c[k]);
  double J[17];
  for (int k = 0; k <= levels; ++k) J[k] = beta_J(edge[k], a);
  for (int k = 0; k < levels; ++k) {
    const double e0 = edge[k], e1 = edge[k + 1];
    const double mass = (J[k + 1] - J[k]) / norm;
    const double mom = (std::pow(std::fmax(0.0, 1.0 - e0 * e0), a + 1.0) -
                        std::pow(std::fmax(0.0, 1.0 - e1 * e1), a + 1.0)) / (2.0 * (a + 1.0) * norm);
    out[k] = mom / mass;
  }
}

// The fixed point of the Lloyd step, found by Newton's method on
// F(c) = step(c) - c (finite-difference Jacobian, at most 16 x 16) from the
// scaled Gaussian codebook, then polished with plain steps until nothing
// moves.  Plain Lloyd converges linearly and slowly here; Newton needs a
// handful of iterations.
void solve_beta_codebook(int levels, int blk, double* c) {
  const double a = 0.5 * (blk - 3);
  const double norm = 2.0 * beta_J(1.0, a);   // B(1/2, a + 1)
  solve_unit_codebook(levels, c);
  for (int k = 0; k < levels; ++k) c[k] /= std::sqrt(static_cast<double>(blk));
  const double h = 1e-7 / std::sqrt(static_cast<double>(blk));
  double F[16], Jm[16][17], tp[16], tm[16], cp[16];
  for (int it = 0; it < 60; ++it) {
    beta_lloyd_step(levels, a, norm, c, F);
    double res = 0.0;
    for (int k = 0; k < levels; ++k) {
      F[k] -= c[k];
      res = std::fmax(res, std::fabs(F[k]));
    }
    if (res < 1e-15 / std::sqrt(static_cast<double>(blk))) break;
    for (int jcol = 0; jcol < levels; ++jcol) {
      for (int k = 0; k < levels; ++k) cp[k] = c[k];
      cp[jcol] = c[jcol] + h;
      beta_lloyd_step(levels, a, norm, cp, tp);
      cp[jcol] = c[jcol] - h;
      beta_lloyd_step(levels, a, norm, cp, tm);
      for (int k = 0; k < levels; ++k) Jm[k][jcol] = (tp[k] - tm[k]) / (2.0 * h) - (k == jcol ? 1.0 : 0.0);
    }
    for (int k = 0; k < levels; ++k) Jm[k][levels] = -F[k];
    // Gaussian elimination with partial pivoting
    for (int col = 0; col < levels; ++col) {
      int piv = col;
      for (int r = col + 1; r < levels; ++r)
        if (std::fabs(Jm[r][col]) > std::fabs(Jm[piv][col])) piv = r;
      if (piv != col)
        for (int q = 0; q <= levels; ++q) std::swap(Jm[col][q], Jm[piv][q]);
      if (Jm[col][col] == 0.0) break;
      for (int r = col + 1; r < levels; ++r) {
        const double f = Jm[r][col] / Jm[col][col];
        for (int q = col; q <= levels; ++q) Jm[r][q] -= f * Jm[col][q];
      }
    }
    for (int r = levels - 1; r >= 0; --r) {
      double v = Jm[r][levels];
      for (int q = r + 1; q < levels; ++q) v -= Jm[r][q] * cp[q];
      cp[r] = v / Jm[r][r];
    }
    for (int k = 0; k < levels; ++k) c[k] += cp[k];
  }
  double last = INFINITY;
  for (int it = 0; it < 100000; ++it) {
    beta_lloyd_step(levels, a, norm, c, tp);
    double moved = 0.0;
    for (int k = 0; k < levels; ++k) {
      moved = std::fmax(moved, std::fabs(tp[k] - c[k]));
      c[k] = tp[k];
    }
    if (moved == 0.0 || (moved < 1e-16 && moved >= last)) break;
    last = moved;
  }
  double sym[16];
  for (int k = 0; k < levels; ++k) sym[k] = 0.5 * (c[k] - c[levels - 1 - k]);
  for (int k = 0; k < levels; ++k) c[k] = sym[k];
}

struct CodebookCache {
  std::mutex mu;
  bool ready[kMaxBits + 1] = {};
  double unit[kMaxBits + 1][kMaxLevels];
  // Beta codebooks per (bits, log2 block) for blocks 32..256
  bool beta_ready[5][9] = {};
  double beta[5][9][16];
};

CodebookCache& cache() {
  static CodebookCache c;
  return c;
}

const double* beta_codebook(int bits, int blk) {
  int lb = 0;
  while ((1 << lb) < blk) ++lb;
  CodebookCache& cc = cache();
  std::lock_guard<std::mutex> lock(cc.mu);
  if (!cc.beta_ready[bits][lb]) {
    solve_beta_codebook(1 << bits, blk, cc.beta[bits][lb]);
    cc.beta_ready[bits][lb] = true;
  }
  return cc.beta[bits][lb];
}

const double* unit_codebook(int bits) {
  CodebookCache& cc = cache();
  std::lock_guard<std::mutex> lock(cc.mu);
  if (!cc.ready[bits]) {
    solve_unit_codebook(1 << bits, cc.unit[bits]);
    cc.ready[bits] = true;
  }
  return cc.unit[bits];
}

uint64_t splitmix64_next(uint64_t& state) {
  state += 0x9E3779B97F4A7C15ull;
  uint64_t z = state;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

bool pow2(int v) { return v > 0 && (v & (v - 1)) == 0; }

}  // namespace

int check_layout(const tq_layout* L) {
  if (!L) return TQ_ERR_ARG;
  if (L->codebook != TQ_CODEBOOK_GAUSSIAN && L->codebook != TQ_CODEBOOK_BETA) return TQ_ERR_ARG;
  if (L->head_dim != 64 && L->head_dim != 128 && L->head_dim != 256) return TQ_ERR_UNSUPPORTED;
  if (!pow2(L->block) || L->block < 32 || L->head_dim % L->block) return TQ_ERR_UNSUPPORTED;
  // 1..4 bits, or one byte per code (Gaussian codebook, no QJL)
  if (!((L->bits >= 1 && L->bits <= 4) || L->bits == 8)) return TQ_ERR_UNSUPPORTED;
  if (L->bits == 8 && (L->codebook != TQ_CODEBOOK_GAUSSIAN || L->qjl_m)) return TQ_ERR_UNSUPPORTED;
  if (L->norm_correct != 0 && L->norm_correct != 1) return TQ_ERR_ARG;
  if (L->qjl_m < 0) return TQ_ERR_ARG;
  if (L->qjl_m > 0 && (L->qjl_m % 32 || L->qjl_m > kMaxQjl || L->block != L->head_dim))
    return TQ_ERR_UNSUPPORTED;
  return TQ_OK;
}

int make_params(const tq_layout* L, CodecParams* p) {
  const int st = check_layout(L);
  if (st != TQ_OK) return st;
  std::memset(p, 0, sizeof(*p));
  p->d = L->head_dim;
  p->blk = L->block;
  p->bits = L->bits;
  p->m = L->qjl_m;
  p->nc = L->norm_correct;
  p->nb = L->head_dim / L->block;
  p->code_bytes = L->head_dim * L->bits / 8;
  p->qjl_bytes = L->qjl_m / 8;
  p->inv_sqrt_blk = static_cast<float>(1.0 / std::sqrt(static_cast<double>(L->block)));
  uint64_t state = L->sign_seed;
  for (int i = 0; i < L->head_dim; ++i)
    if (splitmix64_next(state) >> 63) p->sign_bits[i >> 5] |= 1u << (i & 31);
  if (L->bits > 4) return TQ_OK;   // 8-bit tables: make_codebook8
  double c[16], b[16];
  tq_codebook_kind(L->bits, L->block, L->codebook, c, b);
  const int K = 1 << L->bits;
  for (int k = 0; k < K; ++k) p->centroids[k] = static_cast<float>(c[k]);
  for (int k = 0; k + 1 < K; ++k) p->bounds[k] = static_cast<float>(b[k]);
  return TQ_OK;
}

namespace {
std::atomic<uint64_t> g_wait_limit_ns{0};   // 0: the default
}  // namespace

WaitLimits wait_limits() {
  const uint64_t v = g_wait_limit_ns.load(std::memory_order_relaxed);
  const uint64_t report = v ? v : kDefaultWaitNs;
  return WaitLimits{report, report > kDefaultWaitNs ? report : kDefaultWaitNs};
}

int make_codebook8(const tq_layout* L, Codebook8* cb) {
  const int st = check_layout(L);
  if (st != TQ_OK) return st;
  if (L->bits != 8) return TQ_ERR_ARG;
  double c[256], b[256];
  tq_codebook_kind(8, L->block, L->codebook, c, b);
  for (int k = 0; k < 256; ++k) cb->c[k] = static_cast<float>(c[k]);
  for (int k = 0; k < 255; ++k) cb->b[k] = static_cast<float>(b[k]);
  cb->b[255] = INFINITY;   // never compared: 255 boundaries
  return TQ_OK;
}

}  // namespace tq

extern "C" {

int tq_codebook_f64(int bits, int block, double* centroids, double* boundaries) {
  if (bits < 1 || bits > tq::kMaxBits || block < 1 || !centroids) return TQ_ERR_ARG;
  const double* u = tq::unit_codebook(bits);
  const int K = 1 << bits;
  const double sigma = 1.0 / std::sqrt(static_cast<double>(block));
  for (int k = 0; k < K; ++k) centroids[k] = u[k] * sigma;
  if (boundaries)
    for (int k = 0; k + 1 < K; ++k) boundaries[k] = 0.5 * (centroids[k] + centroids[k + 1]);
  return TQ_OK;
}

int tq_codebook_kind(int bits, int block, int kind, double* centroids, double* boundaries) {
  if (kind == TQ_CODEBOOK_GAUSSIAN) return tq_codebook_f64(bits, block, centroids, boundaries);
  if (kind != TQ_CODEBOOK_BETA || bits < 1 || bits > 4 || !centroids) return TQ_ERR_ARG;
  if (block < 32 || block > 256 || (block & (block - 1))) return TQ_ERR_UNSUPPORTED;
  const double* u = tq::beta_codebook(bits, block);
  const int K = 1 << bits;
  for (int k = 0; k < K; ++k) centroids[k] = u[k];
  if (boundaries)
    for (int k = 0; k + 1 < K; ++k) boundaries[k] = 0.5 * (centroids[k] + centroids[k + 1]);
  return TQ_OK;
}

int tq_codebook(int bits, int block, float* centroids, float* boundaries) {
  double c[tq::kMaxLevels], b[tq::kMaxLevels];
  const int st = tq_codebook_f64(bits, block, c, b);
  if (st != TQ_OK) return st;
  const int K = 1 << bits;
  for (int k = 0; k < K; ++k) centroids[k] = static_cast<float>(c[k]);
  if (boundaries)
    for (int k = 0; k + 1 < K; ++k) boundaries[k] = static_cast<float>(b[k]);
  return TQ_OK;
}

int tq_signs(uint64_t sign_seed, int d, int8_t* out) {
  if (d < 0 || (d > 0 && !out)) return TQ_ERR_ARG;
  uint64_t state = sign_seed;
  for (int i = 0; i < d; ++i) out[i] = (tq::splitmix64_next(state) >> 63) ? -1 : 1;
  return TQ_OK;
}

int tq_layout_sizes(const tq_layout* layout, int64_t* code_bytes_per_vec, int64_t* scales_per_vec,
                    int64_t* qjl_bytes_per_vec) {
  const int st = tq::check_layout(layout);
  if (st != TQ_OK) return st;
  if (code_bytes_per_vec) *code_bytes_per_vec = int64_t(layout->head_dim) * layout->bits / 8;
  if (scales_per_vec) *scales_per_vec = layout->head_dim / layout->block;
  if (qjl_bytes_per_vec) *qjl_bytes_per_vec = layout->qjl_m / 8;
  return TQ_OK;
}

const char* tq_strerror(int status) {
  switch (status) {
    case TQ_OK: return "ok";
    case TQ_ERR_ARG: return "invalid argument (null pointer, shape or stride)";
    case TQ_ERR_UNSUPPORTED: return "unsupported layout (head_dim, block, bits, qjl_m)";
    case TQ_ERR_ALIGN: return "pointer not aligned as required";
    case TQ_ERR_WORKSPACE: return "workspace missing or too small";
    case TQ_ERR_CUDA: return "CUDA launch failed";
    case TQ_ERR_TIMEOUT: return "device-side wait gave up";
    default: return "unknown tq status";
  }
}

int tq_version(void) { return 100; }

int tq_set_wait_limit_ns(uint64_t ns) {
  tq::g_wait_limit_ns.store(ns, std::memory_order_relaxed);
  return TQ_OK;
}

int tq_device_status(int device, int clear, int* status) {
  if (!status) return TQ_ERR_ARG;
  int prev = 0;
  if (cudaGetDevice(&prev) != cudaSuccess) return TQ_ERR_CUDA;
  if (device != prev && cudaSetDevice(device) != cudaSuccess) return TQ_ERR_ARG;
  int st = cudaDeviceSynchronize() == cudaSuccess ? TQ_OK : TQ_ERR_CUDA;
  int q = 0, j = 0, p = 0;
  if (st == TQ_OK) st = tq::quantize_fast_status(clear, &q);
  if (st == TQ_OK) st = tq::quantize_qjl_tc_status(clear, &j);
  if (st == TQ_OK) st = tq::prefill_tc_status(clear, &p);
  if (device != prev) cudaSetDevice(prev);
  if (st != TQ_OK) return st;
  *status = q != 0 ? q : (j != 0 ? j : p);
  return TQ_OK;
}

}  // extern "C"
