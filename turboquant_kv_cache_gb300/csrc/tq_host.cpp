// Host layer of libtq: the Lloyd-Max codebook solver, the sign vector,
// layout checks and sizes, status strings.  Pure C++ (no device code).
#include <cmath>
#include <cstring>
#include <mutex>

#include "tq_internal.h"

namespace tq {
namespace {

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
// is unique, so the start only affects the iteration count.
void solve_unit_codebook(int levels, double* c) {
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
  // The density is symmetric, so is the exact codebook; symmetrise away the
  // rounding residue so that the middle boundary is exactly zero.
  double sym[16];
  for (int k = 0; k < levels; ++k) sym[k] = 0.5 * (c[k] - c[levels - 1 - k]);
  for (int k = 0; k < levels; ++k) c[k] = sym[k];
}

struct CodebookCache {
  std::mutex mu;
  bool ready[5] = {false, false, false, false, false};
  double unit[5][16];
};

CodebookCache& cache() {
  static CodebookCache c;
  return c;
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
  if (L->reserved != 0) return TQ_ERR_ARG;
  if (L->head_dim != 64 && L->head_dim != 128 && L->head_dim != 256) return TQ_ERR_UNSUPPORTED;
  if (!pow2(L->block) || L->block < 32 || L->head_dim % L->block) return TQ_ERR_UNSUPPORTED;
  if (L->bits < 1 || L->bits > 4) return TQ_ERR_UNSUPPORTED;
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
  double c[16], b[16];
  tq_codebook_f64(L->bits, L->block, c, b);
  const int K = 1 << L->bits;
  for (int k = 0; k < K; ++k) p->centroids[k] = static_cast<float>(c[k]);
  for (int k = 0; k + 1 < K; ++k) p->bounds[k] = static_cast<float>(b[k]);
  return TQ_OK;
}

}  // namespace tq

extern "C" {

int tq_codebook_f64(int bits, int block, double* centroids, double* boundaries) {
  if (bits < 1 || bits > 4 || block < 1 || !centroids) return TQ_ERR_ARG;
  const double* u = tq::unit_codebook(bits);
  const int K = 1 << bits;
  const double sigma = 1.0 / std::sqrt(static_cast<double>(block));
  for (int k = 0; k < K; ++k) centroids[k] = u[k] * sigma;
  if (boundaries)
    for (int k = 0; k + 1 < K; ++k) boundaries[k] = 0.5 * (centroids[k] + centroids[k + 1]);
  return TQ_OK;
}

int tq_codebook(int bits, int block, float* centroids, float* boundaries) {
  double c[16], b[16];
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

}  // extern "C"
