// Host side of libtq: context creation (codebook fit, method randomness),
// cache sizing, argument validation and dispatch to the CUDA launchers.
//
// Codebook: Lloyd-Max quantiser of the unit-sphere coordinate marginal
// f(t) ~ (1 - t^2)^((d-3)/2) ("KVQuant++" forum post, "Codebook design";
// "Statistical Inference and Quality Measures of KV Cache Quantisations
// Inspired by TurboQuant", technical summary, "Theoretical framework" and
// "Quantisation schemes"). Cell masses and first moments are integrated with
// composite Gauss-Legendre quadrature in fp64; the Lloyd iteration alternates
// midpoint boundaries and conditional-mean centroids until no centroid moves
// by more than 1e-15 (or the step stalls at the fp64 noise floor).
//
// Method randomness: SplitMix64 (Steele, Lea & Flood, OOPSLA 2014) at counter
// stream*2^32 + i + 1; D from the top bit of stream 1, S by the cosine branch
// of Box-Muller on stream 2, evaluated in double with libm, rounded to float.

#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdlib>
#include <cstring>
#include <map>
#include <mutex>
#include <new>
#include <utility>
#include <vector>

#include "tq_internal.h"

namespace {

// ---------------------------------------------------------------- SplitMix64

constexpr uint64_t kGamma = 0x9E3779B97F4A7C15ull;

uint64_t mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

uint64_t draw(uint64_t seed, uint64_t stream, uint64_t i) {
  uint64_t counter = (stream << 32) + i + 1;
  return mix64(seed + counter * kGamma);
}

void make_diag(uint64_t seed, int d, int8_t *out) {
  for (int i = 0; i < d; ++i) out[i] = (draw(seed, 1, i) >> 63) ? -1 : 1;
}

void make_sketch(uint64_t seed, int d, float *out) {
  const double scale = std::ldexp(1.0, -53);
  const double two_pi = 2.0 * M_PI;
  for (int k = 0; k < d * d; ++k) {
    uint64_t w1 = draw(seed, 2, 2 * (uint64_t)k);
    uint64_t w2 = draw(seed, 2, 2 * (uint64_t)k + 1);
    double u1 = (double)((w1 >> 11) + 1) * scale;
    double u2 = (double)(w2 >> 11) * scale;
    out[k] = (float)(std::sqrt(-2.0 * std::log(u1)) * std::cos(two_pi * u2));
  }
}

// The dense rotation's Gaussian matrix: the same Box-Muller recipe on stream 3, kept in double.
void make_rotation_gaussian(uint64_t seed, int d, double *out) {
  const double scale = std::ldexp(1.0, -53);
  const double two_pi = 2.0 * M_PI;
  for (int k = 0; k < d * d; ++k) {
    uint64_t w1 = draw(seed, 3, 2 * (uint64_t)k);
    uint64_t w2 = draw(seed, 3, 2 * (uint64_t)k + 1);
    double u1 = (double)((w1 >> 11) + 1) * scale;
    double u2 = (double)(w2 >> 11) * scale;
    out[k] = std::sqrt(-2.0 * std::log(u1)) * std::cos(two_pi * u2);
  }
}

// Blocked record layout of a TQ-scheme context: planes in tq_plane order, each 16 tokens of
// its per-token bytes (the side plane only with side codes on).
void build_layout(tq_ctx *c) {
  const int d = c->d;
  const int tok[TQ_NUM_PLANES] = {(int)(c->k.bits * d / 8), 4, c->k.qjl ? d / 8 : 0, c->k.qjl ? 4 : 0,
                                  (int)(c->v.bits * d / 8), 4, c->v.qjl ? d / 8 : 0, c->v.qjl ? 4 : 0,
                                  2 * c->side_rank};
  int off = 0;
  for (int p = 0; p < TQ_NUM_PLANES; ++p) {
    c->lay.off[p] = off;
    c->lay.tok[p] = tok[p];
    off += tq::kBlockTokens * tok[p];
  }
  c->lay.bb = off;
}

// Eigen-decomposition of a symmetric d x d matrix A (row-major, destroyed) by cyclic Jacobi
// rotations: eigenvalues to w, eigenvectors to the columns of V (row-major).
void jacobi_eigen(std::vector<double> &A, int d, std::vector<double> &w, std::vector<double> &V) {
  V.assign((size_t)d * d, 0.0);
  for (int i = 0; i < d; ++i) V[(size_t)i * d + i] = 1.0;
  for (int sweep = 0; sweep < 100; ++sweep) {
    double off = 0.0, tot = 0.0;
    for (int i = 0; i < d; ++i)
      for (int j = 0; j < d; ++j) {
        const double a = A[(size_t)i * d + j] * A[(size_t)i * d + j];
        tot += a;
        if (i != j) off += a;
      }
    if (off <= 1e-30 * tot) break;
    for (int p = 0; p < d - 1; ++p)
      for (int q = p + 1; q < d; ++q) {
        const double apq = A[(size_t)p * d + q];
        if (apq == 0.0) continue;
        const double app = A[(size_t)p * d + p], aqq = A[(size_t)q * d + q];
        const double theta = (aqq - app) / (2.0 * apq);
        const double t = (theta >= 0.0 ? 1.0 : -1.0) / (std::fabs(theta) + std::sqrt(theta * theta + 1.0));
        const double c = 1.0 / std::sqrt(t * t + 1.0), s = t * c;
        for (int k = 0; k < d; ++k) {  // columns p, q
          const double akp = A[(size_t)k * d + p], akq = A[(size_t)k * d + q];
          A[(size_t)k * d + p] = c * akp - s * akq;
          A[(size_t)k * d + q] = s * akp + c * akq;
        }
        for (int k = 0; k < d; ++k) {  // rows p, q
          const double apk = A[(size_t)p * d + k], aqk = A[(size_t)q * d + k];
          A[(size_t)p * d + k] = c * apk - s * aqk;
          A[(size_t)q * d + k] = s * apk + c * aqk;
        }
        for (int k = 0; k < d; ++k) {
          const double vkp = V[(size_t)k * d + p], vkq = V[(size_t)k * d + q];
          V[(size_t)k * d + p] = c * vkp - s * vkq;
          V[(size_t)k * d + q] = s * vkp + c * vkq;
        }
      }
  }
  w.resize(d);
  for (int i = 0; i < d; ++i) w[i] = A[(size_t)i * d + i];
}

// Sign of det(A) (A d x d, row-major, copied) by Gaussian elimination with partial pivoting.
int det_sign(std::vector<double> A, int d) {
  int sign = 1;
  for (int c = 0; c < d; ++c) {
    int p = c;
    for (int r = c + 1; r < d; ++r)
      if (std::fabs(A[r * d + c]) > std::fabs(A[p * d + c])) p = r;
    if (A[p * d + c] == 0.0) return 0;
    if (p != c) {
      for (int k = 0; k < d; ++k) std::swap(A[p * d + k], A[c * d + k]);
      sign = -sign;
    }
    if (A[c * d + c] < 0.0) sign = -sign;
    for (int r = c + 1; r < d; ++r) {
      const double f = A[r * d + c] / A[c * d + c];
      for (int k = c; k < d; ++k) A[r * d + k] -= f * A[c * d + k];
    }
  }
  return sign;
}

// ---------------------------------------------------------------- codebook

struct GaussLegendre {
  std::vector<double> x, w;  // nodes/weights on [-1, 1]
  explicit GaussLegendre(int n) : x(n), w(n) {
    for (int i = 0; i < n; ++i) {
      double z = std::cos(M_PI * (i + 0.75) / (n + 0.5));
      for (int it = 0; it < 100; ++it) {
        double p0 = 1.0, p1 = z;
        for (int k = 2; k <= n; ++k) {
          double p2 = ((2.0 * k - 1.0) * z * p1 - (k - 1.0) * p0) / k;
          p0 = p1;
          p1 = p2;
        }
        double dp = n * (z * p1 - p0) / (z * z - 1.0);
        double dz = p1 / dp;
        z -= dz;
        if (std::fabs(dz) < 1e-16) {
          // recompute the derivative at the converged node for the weight
          double q0 = 1.0, q1 = z;
          for (int k = 2; k <= n; ++k) {
            double q2 = ((2.0 * k - 1.0) * z * q1 - (k - 1.0) * q0) / k;
            q0 = q1;
            q1 = q2;
          }
          dp = n * (z * q1 - q0) / (z * z - 1.0);
          x[i] = z;
          w[i] = 2.0 / ((1.0 - z * z) * dp * dp);
          break;
        }
      }
    }
  }
};

// (mass, first moment) of the unnormalised density g(t) = (1 - t^2)^e on [lo, hi]
std::pair<double, double> cell_integrals(double lo, double hi, double e, const GaussLegendre &gl) {
  if (hi <= lo) return {0.0, 0.0};
  const double panel = 1.0 / 32.0;
  int panels = std::max(1, (int)std::ceil((hi - lo) / panel));
  double h = (hi - lo) / panels;
  double mass = 0.0, mom = 0.0;
  for (int p = 0; p < panels; ++p) {
    double a = lo + p * h;
    double mid = a + 0.5 * h, half = 0.5 * h;
    for (size_t i = 0; i < gl.x.size(); ++i) {
      double t = mid + half * gl.x[i];
      double g = std::exp(e * std::log1p(-t * t));
      mass += gl.w[i] * half * g;
      mom += gl.w[i] * half * g * t;
    }
  }
  return {mass, mom};
}

struct Codebook64 {
  std::vector<double> c, b;
};

Codebook64 fit_lloyd_max(int d, int bits) {
  static const GaussLegendre gl(24);
  const int L = 1 << bits;
  const double e = 0.5 * (d - 3);
  const double sigma = 1.0 / std::sqrt((double)d);
  std::vector<double> c(L), cn(L), edges(L + 1);
  for (int i = 0; i < L; ++i) c[i] = sigma * 2.5 * ((2.0 * (i + 0.5) / L) - 1.0);
  double best = INFINITY;
  int since_best = 0;
  for (int it = 0; it < 400000; ++it) {
    edges[0] = -1.0;
    edges[L] = 1.0;
    for (int i = 1; i < L; ++i) edges[i] = 0.5 * (c[i - 1] + c[i]);
    double step = 0.0;
    for (int i = 0; i < L; ++i) {
      auto mm = cell_integrals(edges[i], edges[i + 1], e, gl);
      cn[i] = mm.second / mm.first;
      step = std::max(step, std::fabs(cn[i] - c[i]));
    }
    c.swap(cn);
    if (step < 1e-15) break;
    if (step < best) {
      best = step;
      since_best = 0;
    } else if (++since_best > 2000) {
      break;
    }
  }
  Codebook64 out;
  out.c.resize(L);
  for (int i = 0; i < L; ++i) out.c[i] = 0.5 * (c[i] - c[L - 1 - i]);
  out.b.resize(L - 1);
  for (int i = 0; i + 1 < L; ++i) out.b[i] = 0.5 * (out.c[i] + out.c[i + 1]);
  out.b[L / 2 - 1] = 0.0;
  return out;
}

const Codebook64 &cached_codebook(int d, int bits) {
  static std::mutex mu;
  static std::map<std::pair<int, int>, Codebook64> cache;
  std::lock_guard<std::mutex> lock(mu);
  auto key = std::make_pair(d, bits);
  auto it = cache.find(key);
  if (it == cache.end()) it = cache.emplace(key, fit_lloyd_max(d, bits)).first;
  return it->second;
}

// ---------------------------------------------------------------- helpers

bool aligned16(const void *p) { return p == nullptr || ((uintptr_t)p & 15u) == 0; }

tq_status cuda_status(cudaError_t e) { return e == cudaSuccess ? TQ_OK : TQ_ERR_CUDA; }

bool is_tq_scheme(int s) { return s == TQ_SCHEME_KV || s == TQ_SCHEME_KQV || s == TQ_SCHEME_QKQV; }

void roles_for(int scheme, int n, tq::Role *k, tq::Role *v) {
  switch (scheme) {
    case TQ_SCHEME_KV: *k = {n, false, false}; *v = {n, false, false}; break;
    case TQ_SCHEME_KQV: *k = {n, true, false}; *v = {n - 1, true, true}; break;
    case TQ_SCHEME_QKQV: *k = {n - 1, true, true}; *v = {n - 1, true, true}; break;
    default: *k = {2, false, false}; *v = {2, false, false}; break;  // KIVI
  }
}

size_t code_bytes(int bits, int d) { return (size_t)bits * d / 8; }

}  // namespace

namespace tq {

void choose_splits(int batch, int heads_kv, int max_len, int requested, int *splits, int *chunk) {
  int s = requested;
  if (s <= 0) {
    // Pick the split count that minimises (rounds of CTAs on 152 SMs x 2 CTAs)
    // x (chunk tokens + a fixed per-CTA setup cost of about 64 tokens), with
    // chunks of at least 256 tokens.
    const long long slots = 152LL * 2;
    const long long units = std::max(1, batch * heads_kv);
    const int s_max = std::max(1, std::min(1024, max_len / 256));
    double best = 1e300;
    s = 1;
    for (int c = 1; c <= s_max; ++c) {
      const long long ctas = units * c;
      const long long rounds = (ctas + slots - 1) / slots;
      const double cost = (double)rounds * ((double)((max_len + c - 1) / c) + 64.0);
      if (cost < best * 0.999) {
        best = cost;
        s = c;
      }
    }
  }
  s = std::max(1, std::min(s, std::max(1, max_len)));
  int c = (max_len + s - 1) / s;
  c = (c + 31) / 32 * 32;  // whole 32-token tiles
  *splits = s;
  *chunk = c;
}

bool draw_dense_rotation(uint64_t seed, int d, double *M) {
  // G = Q R with a positive diagonal: Q's columns are G's columns orthonormalised in order
  // (modified Gram-Schmidt, each column taken through the projections twice); a reflection
  // (det Q = sign det G = -1) becomes a rotation by negating the last column; M = Q^T
  std::vector<double> G((size_t)d * d), Q((size_t)d * d);
  make_rotation_gaussian(seed, d, G.data());
  for (int j = 0; j < d; ++j) {
    std::vector<double> v(d);
    for (int i = 0; i < d; ++i) v[i] = G[(size_t)i * d + j];
    for (int pass = 0; pass < 2; ++pass)
      for (int c = 0; c < j; ++c) {
        double dot = 0.0;
        for (int i = 0; i < d; ++i) dot += Q[(size_t)i * d + c] * v[i];
        for (int i = 0; i < d; ++i) v[i] -= dot * Q[(size_t)i * d + c];
      }
    double nn = 0.0;
    for (int i = 0; i < d; ++i) nn += v[i] * v[i];
    nn = std::sqrt(nn);
    if (!(nn > 0.0)) return false;
    for (int i = 0; i < d; ++i) Q[(size_t)i * d + j] = v[i] / nn;
  }
  const int s = det_sign(G, d);
  if (s == 0) return false;
  if (s < 0)
    for (int i = 0; i < d; ++i) Q[(size_t)i * d + d - 1] = -Q[(size_t)i * d + d - 1];
  for (int i = 0; i < d; ++i)
    for (int k = 0; k < d; ++k) M[(size_t)i * d + k] = Q[(size_t)k * d + i];
  return true;
}

bool build_cell_table(const float *bounds, const float *centroids, int bits, int stride, CellTable *out) {
  const int nb = (1 << bits) - 1;
  double bmax = 0.0;
  for (int j = 0; j < nb; ++j) bmax = std::max(bmax, std::fabs((double)bounds[j]));
  const double eps = 0.5 / stride;  // cell k: t * 63 in [k - eps, k + 1 - eps)
  const double u0 = std::max(bmax * 1.05, 0.05);
  for (int step = 0; step < 2000; ++step) {
    const double U = u0 * std::pow(1.0005, step);
    const float inv2u = (float)(1.0 / (2.0 * U));
    int cell[16];
    bool ok = true;
    for (int j = 0; j < nb && ok; ++j) {
      const double t = (double)bounds[j] * (double)inv2u + 0.5;
      const double s = t * (kCells - 1) + eps;
      const double fl = std::floor(s);
      cell[j] = (int)fl;
      ok = t > 0.0 && t < 1.0 && std::min(s - fl, fl + 1.0 - s) >= kCellMargin && (j == 0 || cell[j] > cell[j - 1]);
    }
    if (!ok) continue;
    out->inv2u = inv2u;
    out->stride = stride;
    for (int k = 0; k < kCells; ++k) {
      int below = 0, inside = -1;
      for (int j = 0; j < nb; ++j) {
        if (cell[j] < k) ++below;
        if (cell[j] == k) inside = j;
      }
      CellEntry &e = out->e[k];
      e.below = below;
      e.thr = inside >= 0 ? bounds[inside] : __builtin_huge_valf();
      e.c_lo = centroids[below] * 1024.f;
      e.c_hi = centroids[inside >= 0 ? below + 1 : below] * 1024.f;
    }
    return true;
  }
  return false;
}

}  // namespace tq

extern "C" {

int tq_abi_version(void) { return TQ_ABI_VERSION; }

const char *tq_status_str(int s) {
  switch (s) {
    case TQ_OK: return "ok";
    case TQ_ERR_ARG: return "invalid argument";
    case TQ_ERR_UNSUPPORTED: return "unsupported by this build";
    case TQ_ERR_CAPACITY: return "append past cache capacity";
    case TQ_ERR_CUDA: return "CUDA error";
    case TQ_ERR_TIMEOUT: return "bounded device wait timed out";
    case TQ_ERR_STATE: return "call does not fit the context's scheme";
    case TQ_ERR_ALIGN: return "pointer not 16-byte aligned";
    case TQ_ERR_WORKSPACE: return "workspace too small";
    default: return "unknown status";
  }
}

tq_status tq_codebook_f64(int d, int bits, double *h_c, double *h_b) {
  if (d < 4 || (d & (d - 1)) || d > 4096 || bits < 1 || bits > 4) return TQ_ERR_ARG;
  const Codebook64 &cb = cached_codebook(d, bits);
  if (h_c) std::memcpy(h_c, cb.c.data(), cb.c.size() * sizeof(double));
  if (h_b) std::memcpy(h_b, cb.b.data(), cb.b.size() * sizeof(double));
  return TQ_OK;
}

tq_status tq_draw_params(uint64_t seed, int d, int8_t *h_diag, float *h_sketch) {
  if (d < 4 || (d & (d - 1)) || d > 4096) return TQ_ERR_ARG;
  if (h_diag) make_diag(seed, d, h_diag);
  if (h_sketch) make_sketch(seed, d, h_sketch);
  return TQ_OK;
}

tq_status tq_init(int d, int bits, int scheme, uint64_t seed, tq_ctx **out) {
  if (!out) return TQ_ERR_ARG;
  *out = nullptr;
  if (scheme < TQ_SCHEME_KV || scheme > TQ_SCHEME_KIVI) return TQ_ERR_ARG;
  if (d < 4 || (d & (d - 1))) return TQ_ERR_ARG;
  if (bits < 2 || bits > 4) return TQ_ERR_ARG;
  if (d != tq::kD) return TQ_ERR_UNSUPPORTED;
  if (scheme == TQ_SCHEME_KIVI && bits != 2) return TQ_ERR_UNSUPPORTED;

  tq_ctx *c = new (std::nothrow) tq_ctx();
  if (!c) return TQ_ERR_ARG;
  c->d = d;
  c->bits = bits;
  c->scheme = scheme;
  c->seed = seed;
  roles_for(scheme, bits, &c->k, &c->v);
  if (is_tq_scheme(scheme)) {
    const Codebook64 &ck = cached_codebook(d, c->k.bits);
    const Codebook64 &cv = cached_codebook(d, c->v.bits);
    for (size_t i = 0; i < ck.c.size(); ++i) c->k_centroids[i] = (float)ck.c[i];
    for (size_t i = 0; i < ck.b.size(); ++i) c->k_bounds[i] = (float)ck.b[i];
    for (size_t i = 0; i < cv.c.size(); ++i) c->v_centroids[i] = (float)cv.c[i];
    for (size_t i = 0; i < cv.b.size(); ++i) c->v_bounds[i] = (float)cv.b[i];
  }
  if (is_tq_scheme(scheme)) {
    // the bulk append's code search: 16-byte entries for sketched roles (they also need the
    // code's centroid), 8-byte ones otherwise
    if (!tq::build_cell_table(c->k_bounds, c->k_centroids, c->k.bits, c->k.qjl ? 512 : 256, &c->cells[0]) ||
        !tq::build_cell_table(c->v_bounds, c->v_centroids, c->v.bits, c->v.qjl ? 512 : 256, &c->cells[1])) {
      delete c;
      return TQ_ERR_UNSUPPORTED;
    }
  }
  make_diag(seed, d, c->diag);
  c->sketch = (float *)std::malloc(sizeof(float) * d * d);
  if (!c->sketch) {
    delete c;
    return TQ_ERR_ARG;
  }
  make_sketch(seed, d, c->sketch);
  {  // an upper bound of the largest row norm of S (certifies the tensor-core signs)
    double m = 0.0;
    for (int j = 0; j < d; ++j) {
      double ss = 0.0;
      for (int k = 0; k < d; ++k) ss += (double)c->sketch[j * d + k] * c->sketch[j * d + k];
      m = std::max(m, std::sqrt(ss));
    }
    c->sketch_rowmax = (float)(m * (1.0 + 1e-6));
  }
  if (scheme != TQ_SCHEME_KIVI) build_layout(c);

  tq::DevParams *hp = (tq::DevParams *)std::calloc(1, sizeof(tq::DevParams));
  if (!hp) {
    std::free(c->sketch);
    delete c;
    return TQ_ERR_ARG;
  }
  std::memcpy(hp->k_centroids, c->k_centroids, sizeof(hp->k_centroids));
  std::memcpy(hp->k_bounds, c->k_bounds, sizeof(hp->k_bounds));
  std::memcpy(hp->v_centroids, c->v_centroids, sizeof(hp->v_centroids));
  std::memcpy(hp->v_bounds, c->v_bounds, sizeof(hp->v_bounds));
  for (int i = 0; i < d; ++i) hp->diag[i] = (float)c->diag[i];
  std::memcpy(hp->sketch, c->sketch, sizeof(float) * d * d);
  hp->error = 0;

  cudaError_t e = cudaGetDevice(&c->device);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&c->num_sms, cudaDevAttrMultiProcessorCount, c->device);
  if (e == cudaSuccess) e = cudaMalloc((void **)&c->dparams, sizeof(tq::DevParams));
  if (e == cudaSuccess) e = cudaMemcpy(c->dparams, hp, sizeof(tq::DevParams), cudaMemcpyHostToDevice);
  if (e == cudaSuccess && tq::launch_operand_prep(c->dparams, nullptr) != TQ_OK) e = cudaErrorUnknown;
  if (e == cudaSuccess && tq::launch_sketch_transpose(c->dparams, nullptr) != TQ_OK) e = cudaErrorUnknown;
  if (e == cudaSuccess) e = cudaStreamSynchronize(nullptr);
  if (e == cudaSuccess) e = cudaStreamCreateWithFlags((cudaStream_t *)&c->side_stream, cudaStreamNonBlocking);
  if (e == cudaSuccess) e = cudaEventCreateWithFlags((cudaEvent_t *)&c->ev_fork, cudaEventDisableTiming);
  if (e == cudaSuccess) e = cudaEventCreateWithFlags((cudaEvent_t *)&c->ev_join, cudaEventDisableTiming);
  std::free(hp);
  if (e != cudaSuccess) {
    if (c->ev_join) cudaEventDestroy((cudaEvent_t)c->ev_join);
    if (c->ev_fork) cudaEventDestroy((cudaEvent_t)c->ev_fork);
    if (c->side_stream) cudaStreamDestroy((cudaStream_t)c->side_stream);
    if (c->dparams) cudaFree(c->dparams);
    std::free(c->sketch);
    delete c;
    return TQ_ERR_CUDA;
  }
  *out = c;
  return TQ_OK;
}

void tq_destroy(tq_ctx *ctx) {
  if (!ctx) return;
  if (ctx->side_u) cudaFree(ctx->side_u);
  if (ctx->side_ur) cudaFree(ctx->side_ur);
  if (ctx->side_urs) cudaFree(ctx->side_urs);
  if (ctx->ev_join) cudaEventDestroy((cudaEvent_t)ctx->ev_join);
  if (ctx->ev_fork) cudaEventDestroy((cudaEvent_t)ctx->ev_fork);
  if (ctx->side_stream) cudaStreamDestroy((cudaStream_t)ctx->side_stream);
  if (ctx->dparams) cudaFree(ctx->dparams);
  std::free(ctx->sketch);
  delete ctx;
}

tq_status tq_draw_rotation(uint64_t seed, int d, float *h_rotation) {
  if (!h_rotation || d < 4 || d > 1024 || (d & (d - 1))) return TQ_ERR_ARG;
  std::vector<double> M((size_t)d * d);
  if (!tq::draw_dense_rotation(seed, d, M.data())) return TQ_ERR_ARG;
  for (size_t i = 0; i < M.size(); ++i) h_rotation[i] = (float)M[i];
  return TQ_OK;
}

tq_status tq_set_rotation(tq_ctx *ctx, int rotation) {
  if (!ctx) return TQ_ERR_ARG;
  if (ctx->scheme == TQ_SCHEME_KIVI) return TQ_ERR_STATE;
  if (rotation != TQ_ROTATION_WHT && rotation != TQ_ROTATION_DENSE) return TQ_ERR_ARG;
  if (ctx->side_rank) return TQ_ERR_STATE;  // side-code bases are set in the rotated coordinates
  if (rotation == TQ_ROTATION_DENSE && ctx->rotation != TQ_ROTATION_DENSE) {
    const int d = ctx->d;
    std::vector<float> M((size_t)d * d), MT((size_t)d * d);
    if (tq_draw_rotation(ctx->seed, d, M.data()) != TQ_OK) return TQ_ERR_ARG;
    for (int i = 0; i < d; ++i)
      for (int k = 0; k < d; ++k) MT[(size_t)k * d + i] = M[(size_t)i * d + k];
    cudaError_t e = cudaMemcpy(ctx->dparams->rot, M.data(), sizeof(float) * d * d, cudaMemcpyHostToDevice);
    if (e == cudaSuccess)
      e = cudaMemcpy(ctx->dparams->rot_t, MT.data(), sizeof(float) * d * d, cudaMemcpyHostToDevice);
    if (e == cudaSuccess && tq::launch_rotation_prep(ctx->dparams, nullptr) != TQ_OK) e = cudaErrorUnknown;
    if (e == cudaSuccess) e = cudaStreamSynchronize(nullptr);
    if (e != cudaSuccess) return TQ_ERR_CUDA;
  }
  ctx->rotation = rotation;
  return TQ_OK;
}

tq_status tq_principal_basis(const float *h_x, int n, int d, int rank, float *h_basis) {
  if (!h_x || !h_basis || n <= 0 || d <= 0 || d > 1024 || rank <= 0 || rank > d) return TQ_ERR_ARG;
  std::vector<double> C((size_t)d * d, 0.0), w, V;
  for (int j = 0; j < n; ++j) {
    const float *x = h_x + (size_t)j * d;
    for (int a = 0; a < d; ++a)
      for (int b = a; b < d; ++b) C[(size_t)a * d + b] += (double)x[a] * x[b];
  }
  for (int a = 0; a < d; ++a)
    for (int b = 0; b < a; ++b) C[(size_t)a * d + b] = C[(size_t)b * d + a];
  jacobi_eigen(C, d, w, V);
  std::vector<int> order(d);
  for (int i = 0; i < d; ++i) order[i] = i;
  std::stable_sort(order.begin(), order.end(), [&](int x, int y) { return w[x] > w[y]; });
  for (int r = 0; r < rank; ++r) {
    const int col = order[r];
    int imax = 0;
    for (int i = 1; i < d; ++i)
      if (std::fabs(V[(size_t)i * d + col]) > std::fabs(V[(size_t)imax * d + col])) imax = i;
    const double sgn = V[(size_t)imax * d + col] < 0.0 ? -1.0 : 1.0;
    for (int i = 0; i < d; ++i) h_basis[(size_t)i * rank + r] = (float)(sgn * V[(size_t)i * d + col]);
  }
  return TQ_OK;
}

tq_status tq_set_side_basis(tq_ctx *ctx, int rank, int heads_kv, const float *h_basis) {
  if (!ctx) return TQ_ERR_ARG;
  if (ctx->scheme == TQ_SCHEME_KIVI || ctx->k.qjl) return TQ_ERR_STATE;
  if (rank < 0 || rank > 8) return TQ_ERR_ARG;
  const int d = ctx->d;
  if (ctx->side_u) cudaFree(ctx->side_u);
  if (ctx->side_ur) cudaFree(ctx->side_ur);
  if (ctx->side_urs) cudaFree(ctx->side_urs);
  ctx->side_u = ctx->side_ur = ctx->side_urs = nullptr;
  ctx->side_rank = 0;
  ctx->side_heads = 0;
  if (rank == 0) {
    build_layout(ctx);
    return TQ_OK;
  }
  if (heads_kv <= 0 || !h_basis) return TQ_ERR_ARG;
  // orthonormal columns per head
  for (int h = 0; h < heads_kv; ++h) {
    const float *U = h_basis + (size_t)h * d * rank;
    for (int a = 0; a < rank; ++a)
      for (int b = 0; b < rank; ++b) {
        double s = 0.0;
        for (int i = 0; i < d; ++i) s += (double)U[(size_t)i * rank + a] * U[(size_t)i * rank + b];
        if (std::fabs(s - (a == b ? 1.0 : 0.0)) > 1e-3) return TQ_ERR_ARG;
      }
  }
  // the bases in the rotated coordinates the codes live in: U_rot = H D U (orthonormal H),
  // M U (dense rotation) or U (unrotated keys); and in code-storage order
  const size_t n = (size_t)heads_kv * d * rank;
  std::vector<float> ur(n), urs(n);
  std::vector<float> M;
  if (ctx->k.rotate && ctx->rotation == TQ_ROTATION_DENSE) {
    M.resize((size_t)d * d);
    if (tq_draw_rotation(ctx->seed, d, M.data()) != TQ_OK) return TQ_ERR_ARG;
  }
  const double inv_sqrt_d = 1.0 / std::sqrt((double)d);
  for (int h = 0; h < heads_kv; ++h) {
    const float *U = h_basis + (size_t)h * d * rank;
    float *R = ur.data() + (size_t)h * d * rank;
    for (int k = 0; k < rank; ++k)
      for (int i = 0; i < d; ++i) {
        double acc = 0.0;
        if (!ctx->k.rotate) {
          acc = U[(size_t)i * rank + k];
        } else if (!M.empty()) {
          for (int j = 0; j < d; ++j) acc += (double)M[(size_t)i * d + j] * U[(size_t)j * rank + k];
        } else {
          for (int j = 0; j < d; ++j)
            acc += ((__builtin_popcount(i & j) & 1) ? -1.0 : 1.0) * ctx->diag[j] * U[(size_t)j * rank + k];
          acc *= inv_sqrt_d;
        }
        R[(size_t)i * rank + k] = (float)acc;
      }
    // code-storage order: offset o = 32 t + 2 m + e holds coordinate 8 m + 2 t + e
    float *S = urs.data() + (size_t)h * d * rank;
    for (int o = 0; o < d; ++o) {
      const int t = o >> 5, m = (o >> 1) & 15, e = o & 1;
      const int i = 8 * m + 2 * t + e;
      for (int k = 0; k < rank; ++k) S[(size_t)o * rank + k] = R[(size_t)i * rank + k];
    }
  }
  cudaError_t e = cudaMalloc((void **)&ctx->side_u, n * sizeof(float));
  if (e == cudaSuccess) e = cudaMalloc((void **)&ctx->side_ur, n * sizeof(float));
  if (e == cudaSuccess) e = cudaMalloc((void **)&ctx->side_urs, n * sizeof(float));
  if (e == cudaSuccess) e = cudaMemcpy(ctx->side_u, h_basis, n * sizeof(float), cudaMemcpyHostToDevice);
  if (e == cudaSuccess) e = cudaMemcpy(ctx->side_ur, ur.data(), n * sizeof(float), cudaMemcpyHostToDevice);
  if (e == cudaSuccess) e = cudaMemcpy(ctx->side_urs, urs.data(), n * sizeof(float), cudaMemcpyHostToDevice);
  if (e != cudaSuccess) {
    if (ctx->side_u) cudaFree(ctx->side_u);
    if (ctx->side_ur) cudaFree(ctx->side_ur);
    if (ctx->side_urs) cudaFree(ctx->side_urs);
    ctx->side_u = ctx->side_ur = ctx->side_urs = nullptr;
    build_layout(ctx);
    return TQ_ERR_CUDA;
  }
  ctx->side_rank = rank;
  ctx->side_heads = heads_kv;
  build_layout(ctx);
  return TQ_OK;
}

tq_status tq_set_kivi(tq_ctx *ctx, int group, int window, int k_per_channel, int v_per_token) {
  if (!ctx) return TQ_ERR_ARG;
  if (ctx->scheme != TQ_SCHEME_KIVI) return TQ_ERR_STATE;
  if (group <= 0 || window < 0 || window % (group > 0 ? group : 1)) return TQ_ERR_ARG;
  if (group != 32 || window > 4096) return TQ_ERR_UNSUPPORTED;
  ctx->kivi_group = group;
  ctx->kivi_window = window;
  ctx->kivi_k_per_channel = k_per_channel ? 1 : 0;
  ctx->kivi_v_per_token = v_per_token ? 1 : 0;
  return TQ_OK;
}

tq_status tq_cache_sizes_get(const tq_ctx *ctx, int batch, int heads_kv, int capacity, tq_cache_sizes *out) {
  if (!ctx || !out || batch <= 0 || heads_kv <= 0 || capacity <= 0) return TQ_ERR_ARG;
  std::memset(out, 0, sizeof(*out));
  const size_t slots = (size_t)batch * heads_kv * capacity;
  const int d = ctx->d;
  if (ctx->scheme == TQ_SCHEME_KIVI) {
    const int G = ctx->kivi_group;
    if (capacity % G) return TQ_ERR_ARG;
    out->k_codes = slots * (d / 4);
    out->v_codes = slots * (d / 4);
    const size_t per_channel = (size_t)batch * heads_kv * (capacity / G) * d * 2 * sizeof(uint16_t);
    const size_t per_token = slots * (d / G) * 2 * sizeof(uint16_t);
    out->k_stats = ctx->kivi_k_per_channel ? per_channel : per_token;
    out->v_stats = ctx->kivi_v_per_token ? per_token : per_channel;
    const size_t win = (size_t)batch * heads_kv * (ctx->kivi_window + G) * d * sizeof(uint16_t);
    out->k_window = win;
    out->v_window = win;
    out->record_bytes = 2 * (d / 4 + (size_t)(d / G) * 4);
    return TQ_OK;
  }
  const size_t blocks = (size_t)batch * heads_kv * (tq::cap16_of(capacity) / tq::kBlockTokens);
  out->block_bytes = (size_t)ctx->lay.bb;
  out->records = blocks * ctx->lay.bb;
  size_t rec = 0;
  for (int p = 0; p < TQ_NUM_PLANES; ++p) {
    out->plane_offset[p] = (size_t)ctx->lay.off[p];
    out->plane_bytes[p] = (size_t)ctx->lay.tok[p];
    rec += (size_t)ctx->lay.tok[p];
  }
  out->record_bytes = rec;
  return TQ_OK;
}

static tq_status append_tq_both(const tq_ctx *ctx, const tq_cache *cache, const void *d_k, const void *d_v,
                                int dtype, int batch, int heads_kv, int n_new, const int32_t *d_seq_lens,
                                void *stream);

// Block-0 bases of the four planes of role `which` (0 keys, 1 values) in the blocked
// records (nullptr for a plane the role does not use).
static void set_role_planes(const tq_ctx *ctx, const tq_cache *c, int which, uint8_t *&codes, float *&norms,
                            uint8_t *&signs, float *&rnorms) {
  const int p0 = which ? TQ_PLANE_V_CODES : TQ_PLANE_K_CODES;
  auto at = [&](int p) -> uint8_t * { return ctx->lay.tok[p] ? c->records + ctx->lay.off[p] : nullptr; };
  codes = at(p0);
  norms = reinterpret_cast<float *>(at(p0 + 1));
  signs = at(p0 + 2);
  rnorms = reinterpret_cast<float *>(at(p0 + 3));
}

static tq_status check_cache(const tq_ctx *ctx, const tq_cache *c, int batch, int heads_kv) {
  if (!c) return TQ_ERR_ARG;
  if (c->batch != batch || c->heads_kv != heads_kv || c->capacity <= 0) return TQ_ERR_ARG;
  const void *planes[] = {c->records, c->k_codes, c->v_codes, c->k_stats, c->v_stats, c->k_window, c->v_window};
  for (const void *p : planes)
    if (!aligned16(p)) return TQ_ERR_ALIGN;
  if (ctx->scheme == TQ_SCHEME_KIVI) {
    if (!c->k_codes || !c->v_codes || !c->k_stats || !c->v_stats || !c->k_window || !c->v_window)
      return TQ_ERR_ARG;
    if (c->capacity % ctx->kivi_group) return TQ_ERR_ARG;
    if (c->block_table) return TQ_ERR_UNSUPPORTED;  // paging covers the blocked TQ records only
    return TQ_OK;
  }
  if (!c->records) return TQ_ERR_ARG;
  if (c->block_table && c->pool_blocks <= 0) return TQ_ERR_ARG;
  if (ctx->side_rank && heads_kv != ctx->side_heads) return TQ_ERR_ARG;  // one basis per KV head
  return TQ_OK;
}

tq_status tq_cache_bytes(const tq_ctx *ctx, int batch, int heads_kv, int capacity, tq_cache_sizes *out) {
  return tq_cache_sizes_get(ctx, batch, heads_kv, capacity, out);
}

tq_status tq_append_quantize(const tq_ctx *ctx, const tq_cache *cache, const void *d_k, const void *d_v,
                             int dtype, int batch, int heads_kv, int n_new, const int32_t *d_seq_lens,
                             void *stream) {
  if (!ctx || !d_k || !d_v || !d_seq_lens) return TQ_ERR_ARG;
  if (dtype != TQ_F32 && dtype != TQ_BF16) return TQ_ERR_ARG;
  if (batch <= 0 || heads_kv <= 0 || n_new < 0) return TQ_ERR_ARG;
  tq_status s = check_cache(ctx, cache, batch, heads_kv);
  if (s != TQ_OK) return s;
  if (!aligned16(d_k) || !aligned16(d_v)) return TQ_ERR_ALIGN;
  if (n_new == 0) return TQ_OK;
  if (ctx->scheme == TQ_SCHEME_KIVI) {
    tq::KiviAppendArgs a{ctx, cache, d_k, d_v, dtype, batch, heads_kv, n_new, d_seq_lens, &ctx->dparams->error};
    if (ctx->prof_append_start) cudaEventRecord((cudaEvent_t)ctx->prof_append_start, (cudaStream_t)stream);
    s = (tq_status)tq::launch_append_kivi(a, stream);
    if (ctx->prof_append_stop) cudaEventRecord((cudaEvent_t)ctx->prof_append_stop, (cudaStream_t)stream);
    return s;
  }
  if (ctx->prof_append_start) cudaEventRecord((cudaEvent_t)ctx->prof_append_start, (cudaStream_t)stream);
  s = append_tq_both(ctx, cache, d_k, d_v, dtype, batch, heads_kv, n_new, d_seq_lens, stream);
  if (ctx->prof_append_stop) cudaEventRecord((cudaEvent_t)ctx->prof_append_stop, (cudaStream_t)stream);
  return s;
}

static tq_status append_tq_both(const tq_ctx *ctx, const tq_cache *cache, const void *d_k, const void *d_v,
                                int dtype, int batch, int heads_kv, int n_new, const int32_t *d_seq_lens,
                                void *stream) {
  tq_status s;
  tq::AppendArgs a{};
  a.dtype = dtype;
  a.batch = batch;
  a.heads = heads_kv;
  a.n_new = n_new;
  a.capacity = cache->capacity;
  a.seq_lens = d_seq_lens;
  a.params = ctx->dparams;
  a.error = &ctx->dparams->error;
  a.ctx = ctx;
  // K
  a.x = d_k;
  a.bb = ctx->lay.bb;
  a.cap16 = tq::cap16_of(cache->capacity);
  a.btab = cache->block_table;
  a.pool_blocks = cache->pool_blocks;
  set_role_planes(ctx, cache, 0, a.codes, a.norms, a.signs, a.rnorms);
  a.vt = 0;
  a.side_rank = ctx->side_rank;
  a.side = ctx->side_rank ? reinterpret_cast<uint16_t *>(cache->records + ctx->lay.off[TQ_PLANE_K_SIDE]) : nullptr;
  a.side_ur = ctx->side_ur;
  a.side_urs = ctx->side_urs;
  a.role = ctx->k;
  a.centroids = ctx->dparams->k_centroids;
  a.bounds = ctx->dparams->k_bounds;
  if (tq::append_small_fits(ctx, (long long)batch * heads_kv * n_new)) {
    // few vectors (a decode step): keys and values in one warp-per-vector launch
    tq::AppendArgs v = a;
    v.side_rank = 0;
    v.side = nullptr;
    v.x = d_v;
    set_role_planes(ctx, cache, 1, v.codes, v.norms, v.signs, v.rnorms);
    v.vt = 1;
    v.role = ctx->v;
    v.centroids = ctx->dparams->v_centroids;
    v.bounds = ctx->dparams->v_bounds;
    return (tq_status)tq::launch_append_small(a, v, ctx, stream);
  }
  // K on the library's side stream, V on the caller's, joined before returning
  cudaStream_t st = (cudaStream_t)stream, side = (cudaStream_t)ctx->side_stream;
  const bool fork = side && cudaEventRecord((cudaEvent_t)ctx->ev_fork, st) == cudaSuccess &&
                    cudaStreamWaitEvent(side, (cudaEvent_t)ctx->ev_fork, 0) == cudaSuccess;
  s = (tq_status)tq::launch_append_tq(a, fork ? (void *)side : stream);
  const bool recorded = fork && cudaEventRecord((cudaEvent_t)ctx->ev_join, side) == cudaSuccess;
  if (fork && !recorded && s == TQ_OK) s = TQ_ERR_CUDA;
  if (s != TQ_OK) {
    if (recorded) cudaStreamWaitEvent(st, (cudaEvent_t)ctx->ev_join, 0);
    return s;
  }
  // V on the caller's stream, then the caller's stream waits for K
  a.side_rank = 0;
  a.side = nullptr;
  a.x = d_v;
  set_role_planes(ctx, cache, 1, a.codes, a.norms, a.signs, a.rnorms);
  a.vt = 1;
  a.role = ctx->v;
  a.centroids = ctx->dparams->v_centroids;
  a.bounds = ctx->dparams->v_bounds;
  s = (tq_status)tq::launch_append_tq(a, stream);
  if (recorded && cudaStreamWaitEvent(st, (cudaEvent_t)ctx->ev_join, 0) != cudaSuccess && s == TQ_OK)
    s = TQ_ERR_CUDA;
  return s;
}

tq_status tq_workspace_size(const tq_ctx *ctx, int batch, int heads_q, int heads_kv, int max_len, int splits,
                            size_t *out) {
  if (!ctx || !out || batch <= 0 || heads_q <= 0 || heads_kv <= 0 || max_len <= 0 || splits < 0)
    return TQ_ERR_ARG;
  int s, chunk;
  tq::choose_splits(batch, heads_kv, max_len, splits, &s, &chunk);
  // prepared queries | decode-tile prefix over batches | decode-step lengths | partial
  // records (split-K per (row, split), or the persistent kernel's kPersistGroups x G per
  // (CTA + KV head) slot)
  size_t qprep = (size_t)batch * heads_q * 2 * ctx->d * sizeof(float);
  size_t prefix = ((size_t)(batch + 1) * sizeof(int32_t) + 15) / 16 * 16;
  size_t lens = ((size_t)batch * sizeof(int32_t) + 15) / 16 * 16;
  size_t split_parts = (size_t)batch * heads_q * s * tq::kPartialFloats * sizeof(float);
  size_t persist_parts = (size_t)tq::kPersistGroups * (size_t)(heads_q / heads_kv) *
                         ((size_t)ctx->num_sms + (size_t)batch * heads_kv) * tq::kPartialFloats * sizeof(float);
  *out = qprep + prefix + lens + std::max(split_parts, persist_parts);
  return TQ_OK;
}

// Carve a workspace of tq_workspace_size bytes (layout above).
static void workspace_layout(const tq_ctx *ctx, void *ws, int batch, int heads_q, tq::DecodeArgs &a,
                             int32_t **step_lens) {
  a.qprep = (float *)ws;
  a.tile_prefix = (int32_t *)(a.qprep + (size_t)batch * heads_q * 2 * ctx->d);
  int32_t *lens = (int32_t *)((char *)a.tile_prefix + ((size_t)(batch + 1) * sizeof(int32_t) + 15) / 16 * 16);
  if (step_lens) *step_lens = lens;
  a.partials = (float *)((char *)lens + ((size_t)batch * sizeof(int32_t) + 15) / 16 * 16);
}

tq_status tq_workspace_bytes(const tq_ctx *ctx, int batch, int heads_q, int heads_kv, int max_len, int splits,
                             size_t *out) {
  return tq_workspace_size(ctx, batch, heads_q, heads_kv, max_len, splits, out);
}

tq_status tq_decode_attention(const tq_ctx *ctx, const tq_cache *cache, const void *d_q, int q_dtype, int batch,
                              int heads_q, int heads_kv, const int32_t *d_seq_lens, int max_len, int splits,
                              void *d_workspace, size_t ws_bytes, float *d_out, void *stream) {
  if (!ctx || !d_q || !d_seq_lens || !d_workspace || !d_out) return TQ_ERR_ARG;
  if (q_dtype != TQ_F32 && q_dtype != TQ_BF16) return TQ_ERR_ARG;
  if (batch <= 0 || heads_q <= 0 || heads_kv <= 0 || max_len <= 0 || splits < 0) return TQ_ERR_ARG;
  if (heads_q % heads_kv) return TQ_ERR_ARG;
  if (heads_q / heads_kv > tq::kMaxGroup) return TQ_ERR_UNSUPPORTED;
  tq_status s = check_cache(ctx, cache, batch, heads_kv);
  if (s != TQ_OK) return s;
  if (max_len > cache->capacity) return TQ_ERR_ARG;
  if (!aligned16(d_q) || !aligned16(d_workspace) || !aligned16(d_out)) return TQ_ERR_ALIGN;
  size_t need = 0;
  tq_workspace_size(ctx, batch, heads_q, heads_kv, max_len, splits, &need);
  if (ws_bytes < need) return TQ_ERR_WORKSPACE;
  tq::DecodeArgs a{};
  a.ctx = ctx;
  a.cache = cache;
  a.q = d_q;
  a.q_dtype = q_dtype;
  a.batch = batch;
  a.heads_q = heads_q;
  a.heads_kv = heads_kv;
  a.max_len = max_len;
  tq::choose_splits(batch, heads_kv, max_len, splits, &a.splits, &a.chunk);
  a.seq_lens = d_seq_lens;
  workspace_layout(ctx, d_workspace, batch, heads_q, a, nullptr);
  a.out = d_out;
  if (ctx->scheme == TQ_SCHEME_KIVI) return (tq_status)tq::launch_decode_kivi(a, stream);
  return (tq_status)tq::launch_decode_tq(a, stream);
}

tq_status tq_decode_step(const tq_ctx *ctx, const tq_cache *cache, const void *d_q, int q_dtype,
                         const void *d_k_new, const void *d_v_new, int kv_dtype, int batch, int heads_q,
                         int heads_kv, const int32_t *d_seq_lens, int max_len, void *d_workspace, size_t ws_bytes,
                         float *d_out, void *stream) {
  if (!ctx || !d_q || !d_k_new || !d_v_new || !d_seq_lens || !d_workspace || !d_out) return TQ_ERR_ARG;
  if (q_dtype != TQ_F32 && q_dtype != TQ_BF16) return TQ_ERR_ARG;
  if (kv_dtype != TQ_F32 && kv_dtype != TQ_BF16) return TQ_ERR_ARG;
  if (batch <= 0 || heads_q <= 0 || heads_kv <= 0 || max_len <= 0) return TQ_ERR_ARG;
  if (heads_q % heads_kv) return TQ_ERR_ARG;
  if (heads_q / heads_kv > tq::kMaxGroup) return TQ_ERR_UNSUPPORTED;
  tq_status s = check_cache(ctx, cache, batch, heads_kv);
  if (s != TQ_OK) return s;
  if (max_len > cache->capacity) return TQ_ERR_ARG;
  if (!aligned16(d_q) || !aligned16(d_k_new) || !aligned16(d_v_new) || !aligned16(d_workspace) ||
      !aligned16(d_out))
    return TQ_ERR_ALIGN;
  size_t need = 0;
  tq_workspace_size(ctx, batch, heads_q, heads_kv, max_len, 0, &need);
  if (ws_bytes < need) return TQ_ERR_WORKSPACE;
  if (ctx->scheme != TQ_SCHEME_KIVI) {
    // one decode kernel that also appends the new tokens and prepares the queries
    tq::DecodeArgs a{};
    a.ctx = ctx;
    a.cache = cache;
    a.q = d_q;
    a.q_dtype = q_dtype;
    a.batch = batch;
    a.heads_q = heads_q;
    a.heads_kv = heads_kv;
    a.max_len = max_len;
    tq::choose_splits(batch, heads_kv, max_len, 0, &a.splits, &a.chunk);
    a.seq_lens = d_seq_lens;
    workspace_layout(ctx, d_workspace, batch, heads_q, a, nullptr);
    a.out = d_out;
    const tq::StepArgs st{d_k_new, d_v_new, kv_dtype};
    const int r = tq::launch_decode_step_tq(a, st, stream);
    if (r != TQ_ERR_UNSUPPORTED) return (tq_status)r;
  }
  // otherwise: the append, then the decode over the lengths plus one
  tq::DecodeArgs lay{};
  int32_t *lens = nullptr;
  workspace_layout(ctx, d_workspace, batch, heads_q, lay, &lens);
  s = (tq_status)tq::launch_step_lengths(d_seq_lens, batch, cache->capacity, lens, stream);
  if (s != TQ_OK) return s;
  s = tq_append_quantize(ctx, cache, d_k_new, d_v_new, kv_dtype, batch, heads_kv, 1, d_seq_lens, stream);
  if (s != TQ_OK) return s;
  return tq_decode_attention(ctx, cache, d_q, q_dtype, batch, heads_q, heads_kv, lens, max_len, 0, d_workspace,
                             ws_bytes, d_out, stream);
}

tq_status tq_dequantize(const tq_ctx *ctx, const tq_cache *cache, int batch, int heads_kv, int t0, int t1,
                        const int32_t *d_seq_lens, float *d_k, float *d_v, void *stream) {
  if (!ctx || batch <= 0 || heads_kv <= 0 || t0 < 0 || t1 < t0) return TQ_ERR_ARG;
  tq_status s = check_cache(ctx, cache, batch, heads_kv);
  if (s != TQ_OK) return s;
  if (t1 > cache->capacity) return TQ_ERR_ARG;
  if (t1 == t0) return TQ_OK;
  if (ctx->scheme == TQ_SCHEME_KIVI) {
    if (!d_seq_lens) return TQ_ERR_ARG;
    tq::KiviDequantArgs a{ctx, cache, batch, heads_kv, t0, t1, d_seq_lens, d_k, d_v};
    return (tq_status)tq::launch_dequant_kivi(a, stream);
  }
  for (int which = 0; which < 2; ++which) {
    float *out = which ? d_v : d_k;
    if (!out) continue;
    tq::DequantArgs a{};
    a.batch = batch;
    a.heads = heads_kv;
    a.capacity = cache->capacity;
    a.t0 = t0;
    a.t1 = t1;
    a.params = ctx->dparams;
    a.out = out;
    a.rot = ctx->rotation == TQ_ROTATION_DENSE ? ctx->dparams->rot : nullptr;
    a.bb = ctx->lay.bb;
    a.cap16 = tq::cap16_of(cache->capacity);
    a.btab = cache->block_table;
    a.pool_blocks = cache->pool_blocks;
    a.error = &ctx->dparams->error;
    a.vt = which;
    uint8_t *codes, *signs;
    float *norms, *rnorms;
    set_role_planes(ctx, cache, which, codes, norms, signs, rnorms);
    a.codes = codes; a.norms = norms; a.signs = signs; a.rnorms = rnorms;
    if (which == 0) {
      a.role = ctx->k; a.centroids = ctx->dparams->k_centroids;
      if (ctx->side_rank) {
        a.side_rank = ctx->side_rank;
        a.side = reinterpret_cast<const uint16_t *>(cache->records + ctx->lay.off[TQ_PLANE_K_SIDE]);
        a.side_u = ctx->side_u;
      }
    } else {
      a.role = ctx->v; a.centroids = ctx->dparams->v_centroids;
    }
    s = (tq_status)tq::launch_dequant_tq(a, stream);
    if (s != TQ_OK) return s;
  }
  return TQ_OK;
}

tq_status tq_export_params(const tq_ctx *ctx, int *k_bits, float *k_c, float *k_b, int *v_bits, float *v_c,
                           float *v_b, int8_t *diag, float *sketch) {
  if (!ctx) return TQ_ERR_ARG;
  const int Lk = 1 << ctx->k.bits, Lv = 1 << ctx->v.bits;
  if (k_bits) *k_bits = ctx->k.bits;
  if (v_bits) *v_bits = ctx->v.bits;
  if (k_c) std::memcpy(k_c, ctx->k_centroids, sizeof(float) * Lk);
  if (k_b) std::memcpy(k_b, ctx->k_bounds, sizeof(float) * (Lk - 1));
  if (v_c) std::memcpy(v_c, ctx->v_centroids, sizeof(float) * Lv);
  if (v_b) std::memcpy(v_b, ctx->v_bounds, sizeof(float) * (Lv - 1));
  if (diag) std::memcpy(diag, ctx->diag, ctx->d);
  if (sketch) std::memcpy(sketch, ctx->sketch, sizeof(float) * ctx->d * ctx->d);
  return TQ_OK;
}

tq_status tq_set_profile_events(tq_ctx *ctx, void *start, void *stop, void *append_start, void *append_stop) {
  if (!ctx) return TQ_ERR_ARG;
  ctx->prof_decode_start = start;
  ctx->prof_decode_stop = stop;
  ctx->prof_append_start = append_start;
  ctx->prof_append_stop = append_stop;
  return TQ_OK;
}

tq_status tq_get_device_error(const tq_ctx *ctx, void *stream, int *code) {
  if (!ctx || !code) return TQ_ERR_ARG;
  cudaStream_t st = (cudaStream_t)stream;
  cudaError_t e = cudaStreamSynchronize(st);
  int v = 0;
  if (e == cudaSuccess) e = cudaMemcpy(&v, &ctx->dparams->error, sizeof(int), cudaMemcpyDeviceToHost);
  if (e == cudaSuccess) e = cudaMemset(&ctx->dparams->error, 0, sizeof(int));
  if (e == cudaSuccess) e = cudaDeviceSynchronize();
  *code = v;
  return cuda_status(e);
}

}  // extern "C"
