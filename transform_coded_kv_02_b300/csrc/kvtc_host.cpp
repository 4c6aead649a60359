// Host side of the transform-coded KV cache library: calibration (statistics, KLT, attention-aware
// importances, reverse water-filling), the parameter table and its device copy, persistence, and the
// argument checks in front of every kernel launch.
//
// Method sources: "KV Cache Compression Through the Lens of Transform Coding" (AATC) - Key points (additive
// white-noise key/value distortion; transform coding + reverse water-filling over a calibration set);
// "SPECTRA: Pushing the KV Cache Beyond the 2-Bit Cliff" - abstract (rotate into a basis from the cache's
// own statistics); "SPHERICAL KV ..." page, first abstract (RDKV: widths from full precision to zero by
// reverse water-filling, once) and third abstract (NOVA-KV: transforms from calibration statistics, fixed
// per-token bit count).
#include <math.h>
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <algorithm>
#include <atomic>
#include <cstdint>
#include <numeric>
#include <thread>
#include <vector>

#include "kvtc_internal.h"

using namespace kvtc;

// ------------------------------------------------------------------------------------------------------
// errors
// ------------------------------------------------------------------------------------------------------
static thread_local std::string g_err;

void kvtc::set_error(const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_err = buf;
}
void kvtc::clear_error() { g_err.clear(); }

extern "C" const char* kv_last_error(void) { return g_err.c_str(); }
extern "C" int kv_version(void) { return 1; }

#define KV_REQUIRE(cond, code, ...)   \
  do {                                \
    if (!(cond)) {                    \
      kvtc::set_error(__VA_ARGS__);   \
      return code;                    \
    }                                 \
  } while (0)

static kv_status cuda_fail(cudaError_t e, const char* what) {
  kvtc::set_error("%s: %s", what, cudaGetErrorString(e));
  return KV_ERR_CUDA;
}

// ------------------------------------------------------------------------------------------------------
// symmetric eigensolver: cyclic Jacobi (Golub & Van Loan, "Matrix Computations", symmetric Jacobi /
// cyclic-by-row), eigenvalues descending, eigenvector columns sign-normalised so that the entry of
// largest magnitude is positive (lowest index on ties).
// ------------------------------------------------------------------------------------------------------
static void jacobi_eigh(const double* sym, int d, double* evals, double* evecs /*[d][d] cols*/) {
  std::vector<double> A(sym, sym + (size_t)d * d), V((size_t)d * d, 0.0);
  for (int i = 0; i < d; ++i) V[(size_t)i * d + i] = 1.0;
  double fro = 0.0;
  for (size_t i = 0; i < A.size(); ++i) fro += A[i] * A[i];
  fro = sqrt(fro);
  for (int sweep = 0; sweep < 100; ++sweep) {
    double off = 0.0;
    for (int p = 0; p < d; ++p)
      for (int q = 0; q < d; ++q)
        if (p != q) off += A[(size_t)p * d + q] * A[(size_t)p * d + q];
    if (sqrt(off) <= 1e-15 * fro || off == 0.0) break;
    for (int p = 0; p < d - 1; ++p) {
      for (int q = p + 1; q < d; ++q) {
        const double apq = A[(size_t)p * d + q];
        if (apq == 0.0) continue;
        const double app = A[(size_t)p * d + p], aqq = A[(size_t)q * d + q];
        // skip rotations that cannot change the diagonal in double precision
        if (fabs(apq) < 1e-300 || (fabs(apq) * 1e18 < fabs(app) && fabs(apq) * 1e18 < fabs(aqq))) {
          A[(size_t)p * d + q] = A[(size_t)q * d + p] = 0.0;
          continue;
        }
        const double tau = (aqq - app) / (2.0 * apq);
        const double t = (tau >= 0 ? 1.0 : -1.0) / (fabs(tau) + sqrt(1.0 + tau * tau));
        const double c = 1.0 / sqrt(1.0 + t * t), s = t * c;
        for (int k = 0; k < d; ++k) {  // A <- A J (columns p, q)
          const double akp = A[(size_t)k * d + p], akq = A[(size_t)k * d + q];
          A[(size_t)k * d + p] = c * akp - s * akq;
          A[(size_t)k * d + q] = s * akp + c * akq;
        }
        for (int k = 0; k < d; ++k) {  // A <- J^T A (rows p, q)
          const double apk = A[(size_t)p * d + k], aqk = A[(size_t)q * d + k];
          A[(size_t)p * d + k] = c * apk - s * aqk;
          A[(size_t)q * d + k] = s * apk + c * aqk;
        }
        A[(size_t)p * d + q] = A[(size_t)q * d + p] = 0.0;
        for (int k = 0; k < d; ++k) {  // V <- V J
          const double vkp = V[(size_t)k * d + p], vkq = V[(size_t)k * d + q];
          V[(size_t)k * d + p] = c * vkp - s * vkq;
          V[(size_t)k * d + q] = s * vkp + c * vkq;
        }
      }
    }
  }
  std::vector<int> order(d);
  std::iota(order.begin(), order.end(), 0);
  std::stable_sort(order.begin(), order.end(),
                   [&](int a, int b) { return A[(size_t)a * d + a] > A[(size_t)b * d + b]; });
  for (int i = 0; i < d; ++i) {
    const int src = order[i];
    evals[i] = A[(size_t)src * d + src];
    int jmax = 0;
    double amax = -1.0;
    for (int k = 0; k < d; ++k) {
      const double a = fabs(V[(size_t)k * d + src]);
      if (a > amax) { amax = a; jmax = k; }
    }
    const double sgn = V[(size_t)jmax * d + src] < 0 ? -1.0 : 1.0;
    for (int k = 0; k < d; ++k) evecs[(size_t)k * d + i] = sgn * V[(size_t)k * d + src];
  }
}

// ------------------------------------------------------------------------------------------------------
// reverse water-filling: b_i(theta) = clip(1/2 log2(lam_i/theta), 0, Bmax), sum b_i = C by bisection on
// log2(theta) in [log2(min lam) - 40, log2(max lam)] (200 halvings); integer widths = floors, then one bit
// each to the largest fractional parts (compared at 1e-9), ties to larger lam then lower index.
// ------------------------------------------------------------------------------------------------------
static void water_fill(const double* lam, int d, int budget, int bmax, int32_t* out) {
  std::vector<double> b(d, 0.0), l2(d, -INFINITY);
  int npos = 0;
  double lo = INFINITY, hi = -INFINITY;
  for (int i = 0; i < d; ++i)
    if (lam[i] > 0) {
      l2[i] = log2(lam[i]);
      lo = std::min(lo, l2[i]);
      hi = std::max(hi, l2[i]);
      ++npos;
    }
  if (budget > 0 && npos > 0) {
    if ((long long)budget >= (long long)bmax * npos) {
      for (int i = 0; i < d; ++i) b[i] = lam[i] > 0 ? bmax : 0.0;
    } else {
      auto eval = [&](double t, std::vector<double>* dst) {
        double sum = 0.0;
        for (int i = 0; i < d; ++i) {
          double x = 0.5 * (l2[i] - t);
          x = x < 0 ? 0.0 : (x > bmax ? (double)bmax : x);
          if (dst) (*dst)[i] = x;
          sum += x;
        }
        return sum;
      };
      lo -= 40.0;
      for (int it = 0; it < 200; ++it) {
        const double mid = 0.5 * (lo + hi);
        if (eval(mid, nullptr) > budget) lo = mid; else hi = mid;
      }
      eval(0.5 * (lo + hi), &b);
    }
  }
  long long used = 0;
  std::vector<long long> fk(d);
  for (int i = 0; i < d; ++i) {
    out[i] = (int32_t)floor(b[i]);
    used += out[i];
    fk[i] = llrint((b[i] - out[i]) * 1e9);
  }
  long long rem = (long long)budget - used;
  std::vector<int> cand;
  for (int i = 0; i < d; ++i)
    if (out[i] < bmax && lam[i] > 0) cand.push_back(i);
  std::sort(cand.begin(), cand.end(), [&](int a, int c) {
    if (fk[a] != fk[c]) return fk[a] > fk[c];
    if (lam[a] != lam[c]) return lam[a] > lam[c];
    return a < c;
  });
  for (size_t k = 0; k < cand.size() && rem > 0; ++k, --rem) out[cand[k]] += 1;
}

static int record_words(float bits, int d) { return (int)floor((double)bits * d / 32.0 + 1e-9); }

// ------------------------------------------------------------------------------------------------------
// calibration of one set
// ------------------------------------------------------------------------------------------------------
struct SetResult {
  std::vector<float> T[2], mu[2], sigma[2], Tinv[2];
  std::vector<int32_t> widths[2];
  std::vector<double> eig[2], imp[2];
  bool ok = true;
  std::string err;
};

static bool finite_all(const float* x, size_t n) {
  for (size_t i = 0; i < n; ++i)
    if (!std::isfinite(x[i])) return false;
  return true;
}

static void moments(const float* x, int64_t n, int d, bool centre, std::vector<double>& mean,
                    std::vector<double>& cov) {
  mean.assign(d, 0.0);
  cov.assign((size_t)d * d, 0.0);
  if (centre) {
    for (int64_t t = 0; t < n; ++t)
      for (int i = 0; i < d; ++i) mean[i] += x[t * d + i];
    for (int i = 0; i < d; ++i) mean[i] /= (double)n;
  }
  std::vector<double> row(d);
  for (int64_t t = 0; t < n; ++t) {
    for (int i = 0; i < d; ++i) row[i] = (double)x[t * d + i] - mean[i];
    for (int i = 0; i < d; ++i) {
      const double ri = row[i];
      double* c = &cov[(size_t)i * d];
      for (int j = i; j < d; ++j) c[j] += ri * row[j];
    }
  }
  for (int i = 0; i < d; ++i)
    for (int j = i; j < d; ++j) {
      const double v = cov[(size_t)i * d + j] / (double)n;
      cov[(size_t)i * d + j] = v;
      cov[(size_t)j * d + i] = v;
    }
}

// ------------------------------------------------------------------------------------------------------
// fixed-width record layout [NOVA-KV: fixed per-token bit count, fixed-width layout]: storage channels
// (2k, 2k+1) share a slot of width max(b_2k, b_2k+1) at the same bit of the low and the high half of one
// code word; slots are placed first-fit in pair order.
// ------------------------------------------------------------------------------------------------------
bool kvtc::slot_layout(const int32_t* w, int d, int rw, int* word, int* pos) {
  int used[MAX_RW] = {0};
  const int nw = rw - 1;
  for (int k = 0; k < d / 2; ++k) {
    const int sw = std::max(w[2 * k], w[2 * k + 1]);
    word[k] = pos[k] = -1;
    if (sw == 0) continue;
    int u = 0;
    while (u < nw && used[u] + sw > 16) ++u;
    if (u >= nw) return false;
    word[k] = u;
    pos[k] = used[u];
    used[u] += sw;
  }
  return true;
}

// Value records hold two tokens: channel j has one slot of width b_j at the same bit of the low half (earlier
// token) and the high half (later token) of one of the 2 rw - 2 code words; slots are placed first-fit in
// storage order.
bool kvtc::token_slot_layout(const int32_t* w, int d, int rw, int* word, int* pos) {
  int used[2 * MAX_RW] = {0};
  const int nw = 2 * rw - 2;
  for (int j = 0; j < d; ++j) {
    word[j] = pos[j] = -1;
    if (w[j] == 0) continue;
    int u = 0;
    while (u < nw && used[u] + w[j] > 16) ++u;
    if (u >= nw) return false;
    word[j] = u;
    pos[j] = used[u];
    used[u] += w[j];
  }
  return true;
}

// Order of the cost 3 (lambda_2k + lambda_2k+1) 4^-w of taking one bit from a pair: log2 at 1e-9
// resolution (less the common log2 3), so that costs equal in exact arithmetic compare equal.
static long long fit_cost_key(double pair_importance, int width) {
  if (!(pair_importance > 0.0)) return -(1LL << 62);
  return (long long)std::nearbyint(std::log2(pair_importance) * 1e9) - 2000000000LL * width;
}

// Raise the narrower channel of each pair to the slot width, then take single bits from the cheapest pair
// (ties: the later pair) until the first-fit placement succeeds.
static void fit_layout(int32_t* w, const double* imp, int d, int rw) {
  const int np = d / 2;
  std::vector<int32_t> sw(np), wide(d);
  std::vector<double> plam(np);
  for (int k = 0; k < np; ++k) {
    sw[k] = std::max(w[2 * k], w[2 * k + 1]);
    plam[k] = imp[2 * k] + imp[2 * k + 1];
  }
  std::vector<int> word(np), pos(np);
  for (;;) {
    for (int k = 0; k < np; ++k) wide[2 * k] = wide[2 * k + 1] = sw[k];
    if (kvtc::slot_layout(wide.data(), d, rw, word.data(), pos.data())) break;
    int best = -1;
    long long best_key = 0;
    for (int k = 0; k < np; ++k) {
      if (sw[k] <= 0) continue;
      const long long key = fit_cost_key(plam[k], sw[k]);
      if (best < 0 || key <= best_key) {
        best = k;
        best_key = key;
      }
    }
    if (best < 0) break;  // nothing left to take (cannot happen for rw >= 1)
    --sw[best];
  }
  for (int j = 0; j < d; ++j) w[j] = wide[j];
}

// Take single bits from the cheapest channel (ties: the later channel) until the token-pair layout holds.
static void fit_token_layout(int32_t* w, const double* imp, int d, int rw) {
  std::vector<int> word(d), pos(d);
  while (!kvtc::token_slot_layout(w, d, rw, word.data(), pos.data())) {
    int best = -1;
    long long best_key = 0;
    for (int j = 0; j < d; ++j) {
      if (w[j] <= 0) continue;
      const long long key = fit_cost_key(imp[j], w[j]);
      if (best < 0 || key <= best_key) {
        best = j;
        best_key = key;
      }
    }
    if (best < 0) break;
    --w[best];
  }
}

// U: basis as columns (column e = row of T for basis index e). Uinv (null for an orthogonal U): the inverse of
// U^T, whose column e pairs with basis index e; kept in storage order beside T.
static void build_tensor(const std::vector<double>& mu_raw, const std::vector<double>& lam,
                         const std::vector<double>& U, const std::vector<double>& imp, int rw, int bmax,
                         int d, SetResult& r, int t, const std::vector<double>* Uinv = nullptr) {
  std::vector<int32_t> w(d);
  water_fill(imp.data(), d, 32 * rw - 32, bmax, w.data());
  std::vector<int> order(d);
  std::iota(order.begin(), order.end(), 0);
  std::sort(order.begin(), order.end(), [&](int a, int b) {
    if (w[a] != w[b]) return w[a] > w[b];
    if (imp[a] != imp[b]) return imp[a] > imp[b];
    return a < b;
  });
  std::vector<int32_t> ws(d);
  std::vector<double> imps(d);
  for (int j = 0; j < d; ++j) {
    ws[j] = w[order[j]];
    imps[j] = imp[order[j]];
  }
  if (t == 0)
    fit_layout(ws.data(), imps.data(), d, rw);  // keys: channel pairs share slots
  else
    fit_token_layout(ws.data(), imps.data(), d, rw);  // values: token pairs share slots
  r.T[t].resize((size_t)d * d);
  r.mu[t].resize(d);
  r.sigma[t].resize(d);
  r.widths[t].resize(d);
  r.eig[t].resize(d);
  r.imp[t].resize(d);
  for (int j = 0; j < d; ++j) {
    const int e = order[j];
    double m = 0.0;
    for (int k = 0; k < d; ++k) {
      const double u = U[(size_t)k * d + e];  // column e of U = row j of T
      r.T[t][(size_t)j * d + k] = (float)u;
      m += u * mu_raw[k];
    }
    r.mu[t][j] = (float)m;
    r.sigma[t][j] = (float)sqrt(std::max(lam[e], 0.0));
    r.widths[t][j] = r.sigma[t][j] > 0.f ? ws[j] : 0;
    r.eig[t][j] = lam[e];
    r.imp[t][j] = imps[j];
  }
  r.Tinv[t].clear();
  if (Uinv) {
    r.Tinv[t].resize((size_t)d * d);
    for (int k = 0; k < d; ++k)
      for (int j = 0; j < d; ++j) r.Tinv[t][(size_t)k * d + j] = (float)(*Uinv)[(size_t)k * d + order[j]];
  }
}

// Attention-aware orthogonal key basis, from the KLT U (columns; replaced in place). With white quantisation
// noise in basis U the key distortion is sum_i w_i D_i (w_i = u_i^T M_Q u_i); water-filling against the
// coefficient variances s_i = u_i^T Sigma_K u_i makes it proportional (high-rate model) to (prod_i s_i w_i)^(1/d),
// of which the KLT minimises only prod s_i. [NOVA-KV] derives the key transform from this distortion (its optimum
// is not orthogonal); here the transform stays orthogonal and sum_i log s_i + log w_i falls by cyclic Jacobi
// sweeps: each pair (i < j, row order) is rotated by the grid angle -pi/4 + k pi/(2 grid) that minimises its four
// log terms (the first such k), when that beats no rotation by more than 1e-10. Both matrices get 1e-12 tr/d
// added on the diagonal.
static void attention_aware_basis(const std::vector<double>& sk, const std::vector<double>& mq, int d,
                                  std::vector<double>& U) {
  constexpr int SWEEPS = 8, GRID = 48;
  std::vector<double> A(sk), B(mq);
  double ta = 0.0, tb = 0.0;
  for (int i = 0; i < d; ++i) {
    ta += A[(size_t)i * d + i];
    tb += B[(size_t)i * d + i];
  }
  for (int i = 0; i < d; ++i) {
    A[(size_t)i * d + i] += 1e-12 * ta / d;
    B[(size_t)i * d + i] += 1e-12 * tb / d;
  }
  // a = U^T A U, b = U^T B U
  auto congruence = [&](const std::vector<double>& M, std::vector<double>& out) {
    std::vector<double> MU((size_t)d * d, 0.0);
    for (int r = 0; r < d; ++r)
      for (int c = 0; c < d; ++c) {
        double acc = 0.0;
        for (int k = 0; k < d; ++k) acc += M[(size_t)r * d + k] * U[(size_t)k * d + c];
        MU[(size_t)r * d + c] = acc;
      }
    out.assign((size_t)d * d, 0.0);
    for (int r = 0; r < d; ++r)
      for (int c = 0; c < d; ++c) {
        double acc = 0.0;
        for (int k = 0; k < d; ++k) acc += U[(size_t)k * d + r] * MU[(size_t)k * d + c];
        out[(size_t)r * d + c] = acc;
      }
  };
  std::vector<double> a, b;
  congruence(A, a);
  congruence(B, b);
  double cs[GRID], sn[GRID], f[GRID];
  for (int k = 0; k < GRID; ++k) {
    const double phi = -M_PI / 4 + k * (M_PI / 2 / GRID);
    cs[k] = cos(phi);
    sn[k] = sin(phi);
  }
  const int k0 = GRID / 2;  // phi = 0
  auto rotate = [&](std::vector<double>& M, int i, int j, double c, double s) {
    for (int r = 0; r < d; ++r) {  // columns i, j
      const double mi = M[(size_t)r * d + i], mj = M[(size_t)r * d + j];
      M[(size_t)r * d + i] = mi * c + mj * s;
      M[(size_t)r * d + j] = mi * -s + mj * c;
    }
    for (int col = 0; col < d; ++col) {  // rows i, j
      const double mi = M[(size_t)i * d + col], mj = M[(size_t)j * d + col];
      M[(size_t)i * d + col] = c * mi + s * mj;
      M[(size_t)j * d + col] = -s * mi + c * mj;
    }
  };
  for (int sweep = 0; sweep < SWEEPS; ++sweep)
    for (int i = 0; i < d - 1; ++i)
      for (int j = i + 1; j < d; ++j) {
        const double aii = a[(size_t)i * d + i], ajj = a[(size_t)j * d + j], aij = a[(size_t)i * d + j];
        const double bii = b[(size_t)i * d + i], bjj = b[(size_t)j * d + j], bij = b[(size_t)i * d + j];
        int kb = 0;
        for (int k = 0; k < GRID; ++k) {
          const double c = cs[k], s = sn[k];
          f[k] = log(c * c * aii + 2 * c * s * aij + s * s * ajj) + log(s * s * aii - 2 * c * s * aij + c * c * ajj) +
                 log(c * c * bii + 2 * c * s * bij + s * s * bjj) + log(s * s * bii - 2 * c * s * bij + c * c * bjj);
          if (f[k] < f[kb]) kb = k;
        }
        if (!(f[kb] < f[k0] - 1e-10)) continue;
        const double c = cs[kb], s = sn[kb];
        for (int r = 0; r < d; ++r) {  // U columns i, j
          const double ui = U[(size_t)r * d + i], uj = U[(size_t)r * d + j];
          U[(size_t)r * d + i] = ui * c + uj * s;
          U[(size_t)r * d + j] = ui * -s + uj * c;
        }
        rotate(a, i, j, c, s);
        rotate(b, i, j, c, s);
      }
}

// Statistics, transforms and importances of one set (everything before the record budget is applied).
struct SetPrep {
  std::vector<double> mk, lk, uk, ik, mv, lv, uv, iv;
  std::vector<double> ukinv;  // key_basis 2: the inverse of uk^T (columns pair with uk's)
  double rho = 0.0;  // weight of key against value distortion (joint allocation)
};

static void prepare_one(const kv_calib_set& s, const kv_calib_opts& o, SetPrep& P, SetResult& r) {
  const int d = o.d;
  if (!finite_all(s.k, (size_t)s.n_tok * d) || !finite_all(s.v, (size_t)s.n_tok * d) ||
      !finite_all(s.q, (size_t)s.n_q * d)) {
    r.ok = false;
    r.err = "non-finite calibration data";
    return;
  }
  std::vector<double> ck, cv, mq, cq;
  std::vector<double>&mk = P.mk, &mv = P.mv, &lk = P.lk, &lv = P.lv, &uk = P.uk, &uv = P.uv, &ik = P.ik, &iv = P.iv;
  moments(s.k, s.n_tok, d, true, mk, ck);
  moments(s.v, s.n_tok, d, true, mv, cv);
  moments(s.q, s.n_q, d, false, mq, cq);
  lk.assign(d, 0.0);
  lv.assign(d, 0.0);
  uk.assign((size_t)d * d, 0.0);
  uv.assign((size_t)d * d, 0.0);
  jacobi_eigh(ck.data(), d, lk.data(), uk.data());
  jacobi_eigh(cv.data(), d, lv.data(), uv.data());
  if (o.key_basis == 2) {
    // [NOVA-KV]'s non-orthogonal key transform under the high-resolution model: T = c V^T M_Q^(1/2), V the KLT of
    // M_Q^(1/2) Sigma_K M_Q^(1/2). Then e^T M_Q e = |T e|^2 / c^2 (the attention-aware key distortion is
    // mean-squared in the transform domain) and the coefficients are uncorrelated with variances c^2 lambda, so
    // plain water-filling on those variances allocates the bits. c = the largest column norm of
    // (V^T M_Q^(1/2))^-1 = M_Q^(-1/2) V, so that every column of T^-1 has norm <= 1. M_Q gets 1e-12 tr/d on the
    // diagonal.
    std::vector<double> M(cq), lq(d), Q((size_t)d * d);
    double tq = 0.0;
    for (int i = 0; i < d; ++i) tq += M[(size_t)i * d + i];
    for (int i = 0; i < d; ++i) M[(size_t)i * d + i] += 1e-12 * tq / d;
    jacobi_eigh(M.data(), d, lq.data(), Q.data());
    std::vector<double> mh((size_t)d * d, 0.0), mih((size_t)d * d, 0.0);
    for (int a = 0; a < d; ++a)
      for (int b = 0; b < d; ++b) {
        double s1 = 0.0, s2 = 0.0;
        for (int i = 0; i < d; ++i) {
          const double l = std::max(lq[i], 1e-300), qa = Q[(size_t)a * d + i] * Q[(size_t)b * d + i];
          s1 += qa * std::sqrt(l);
          s2 += qa / std::sqrt(l);
        }
        mh[(size_t)a * d + b] = s1;
        mih[(size_t)a * d + b] = s2;
      }
    std::vector<double> tmpm((size_t)d * d, 0.0), A((size_t)d * d, 0.0), V((size_t)d * d);
    for (int a = 0; a < d; ++a)
      for (int b = 0; b < d; ++b) {
        double acc = 0.0;
        for (int i = 0; i < d; ++i) acc += ck[(size_t)a * d + i] * mh[(size_t)i * d + b];
        tmpm[(size_t)a * d + b] = acc;
      }
    for (int a = 0; a < d; ++a)
      for (int b = 0; b < d; ++b) {
        double acc = 0.0;
        for (int i = 0; i < d; ++i) acc += mh[(size_t)a * d + i] * tmpm[(size_t)i * d + b];
        A[(size_t)a * d + b] = acc;
      }
    std::vector<double> lam(d);
    jacobi_eigh(A.data(), d, lam.data(), V.data());
    // U = (V^T M_Q^(1/2))^T = M_Q^(1/2) V (columns), Uinv = M_Q^(-1/2) V (columns), then scaled by c and 1/c
    std::vector<double> U((size_t)d * d), Ui((size_t)d * d);
    for (int a = 0; a < d; ++a)
      for (int e = 0; e < d; ++e) {
        double s1 = 0.0, s2 = 0.0;
        for (int i = 0; i < d; ++i) {
          s1 += mh[(size_t)a * d + i] * V[(size_t)i * d + e];
          s2 += mih[(size_t)a * d + i] * V[(size_t)i * d + e];
        }
        U[(size_t)a * d + e] = s1;
        Ui[(size_t)a * d + e] = s2;
      }
    double c = 0.0;
    for (int e = 0; e < d; ++e) {
      double n2 = 0.0;
      for (int a = 0; a < d; ++a) n2 += Ui[(size_t)a * d + e] * Ui[(size_t)a * d + e];
      c = std::max(c, std::sqrt(n2));
    }
    for (size_t i = 0; i < U.size(); ++i) {
      U[i] *= c;
      Ui[i] /= c;
    }
    uk.swap(U);
    P.ukinv.swap(Ui);
    for (int i = 0; i < d; ++i) lk[i] = std::max(lam[i], 0.0) * c * c;
  }
  if (o.key_basis == 1) {  // attention-aware key basis; the variances are then the diagonal of U^T Sigma_K U
    attention_aware_basis(ck, cq, d, uk);
    for (int i = 0; i < d; ++i) {
      double acc = 0.0;
      for (int a = 0; a < d; ++a) {
        double row = 0.0;
        for (int b = 0; b < d; ++b) row += ck[(size_t)a * d + b] * uk[(size_t)b * d + i];
        acc += uk[(size_t)a * d + i] * row;
      }
      lk[i] = acc;
    }
  }
  // key importances: sigma_i^2 * u_i^T M_Q u_i (key_basis 2: the coefficient variances, the distortion being
  // mean-squared in that domain); value importances: sigma_i^2
  ik.assign(d, 0.0);
  iv.assign(d, 0.0);
  std::vector<double> tmp(d);
  for (int i = 0; i < d; ++i) {
    iv[i] = std::max(lv[i], 0.0);
    if (o.key_basis == 2) {
      ik[i] = std::max(lk[i], 0.0);
      continue;
    }
    for (int a = 0; a < d; ++a) {
      double acc = 0.0;
      for (int b = 0; b < d; ++b) acc += cq[(size_t)a * d + b] * uk[(size_t)b * d + i];
      tmp[a] = acc;
    }
    double w = 0.0;
    for (int a = 0; a < d; ++a) w += uk[(size_t)a * d + i] * tmp[a];
    ik[i] = std::max(lk[i], 0.0) * w;
  }
  for (int i = 0; i < d; ++i)
    if (!std::isfinite(ik[i]) || !std::isfinite(iv[i])) {
      r.ok = false;
      r.err = "non-finite statistics";
      return;
    }
  // Key against value distortion in the attention output: to first order a key error e_t moves the output by
  // p_t alpha (q.e_t)(v_t - o), so with white noise E|do|^2 = sum_t p_t^2 (alpha^2 |v_t - o|^2 sum_i w_i D^K_i
  // + sum_i D^V_i) (additive, factored over tokens and channels: [AATC] Key points, first bullet). With
  // |v_t - o|^2 at its mean tr(Sigma_V) and alpha = 1/sqrt(d): rho = tr(Sigma_V) / d.
  double tr = 0.0;
  for (int i = 0; i < d; ++i) tr += std::max(lv[i], 0.0);
  P.rho = tr / d;
}

// Integer water-filling of imp at 32 rw - 32 code bits; returns sum_i imp_i 4^-b_i (the white-noise distortion
// of a b-bit channel is proportional to sigma^2 4^-b).
static double budget_distortion(const std::vector<double>& imp, int rw, int bmax, int d) {
  std::vector<int32_t> w(d);
  water_fill(imp.data(), d, 32 * rw - 32, bmax, w.data());
  double acc = 0.0;
  for (int i = 0; i < d; ++i) acc += imp[i] * ldexp(1.0, -2 * w[i]);
  return acc;
}

static void build_one(const SetPrep& P, int rwk, int rwv, const kv_calib_opts& o, SetResult& r) {
  build_tensor(P.mk, P.lk, P.uk, P.ik, rwk, o.max_bits, o.d, r, 0, P.ukinv.empty() ? nullptr : &P.ukinv);
  build_tensor(P.mv, P.lv, P.uv, P.iv, rwv, o.max_bits, o.d, r, 1);
}

static kv_status check_budget(float bits, int d, int bmax, int* rw_out) {
  const int rw = record_words(bits, d);
  KV_REQUIRE(rw >= 1 && rw <= 1 + bmax * d / 32, KV_ERR_BUDGET,
             "budget %.4f bits/element gives %d record words (valid 1..%d)", bits, rw, 1 + bmax * d / 32);
  *rw_out = rw;
  return KV_OK;
}

extern "C" kv_status kv_calibrate(int n_sets, const kv_calib_set* sets, const kv_calib_opts* opts,
                                  kv_params** out) {
  clear_error();
  KV_REQUIRE(sets && opts && out && n_sets >= 1, KV_ERR_INVALID_ARG, "kv_calibrate: null argument or n_sets < 1");
  KV_REQUIRE(opts->d == D, KV_ERR_UNSUPPORTED, "kv_calibrate: d=%d unsupported (128 only)", opts->d);
  KV_REQUIRE(opts->max_bits >= 1 && opts->max_bits <= MAX_BITS, KV_ERR_INVALID_ARG, "max_bits must be 1..8");
  int rwk, rwv;
  kv_status st;
  if ((st = check_budget(opts->bits_k, opts->d, opts->max_bits, &rwk)) != KV_OK) return st;
  if ((st = check_budget(opts->bits_v, opts->d, opts->max_bits, &rwv)) != KV_OK) return st;
  for (int i = 0; i < n_sets; ++i) {
    KV_REQUIRE(sets[i].k && sets[i].v && sets[i].q, KV_ERR_INVALID_ARG, "set %d: null pointer", i);
    KV_REQUIRE(sets[i].n_tok >= 2 && sets[i].n_q >= 1, KV_ERR_INVALID_ARG, "set %d: need n_tok >= 2, n_q >= 1", i);
  }
  KV_REQUIRE(opts->joint == 0 || opts->joint == 1, KV_ERR_INVALID_ARG, "joint must be 0 or 1");
  KV_REQUIRE(opts->key_basis >= 0 && opts->key_basis <= 2, KV_ERR_INVALID_ARG, "key_basis must be 0, 1 or 2");
  std::vector<SetResult> res(n_sets);
  std::vector<SetPrep> prep(n_sets);
  int nth = opts->n_threads > 0 ? opts->n_threads : (int)std::max(1u, std::thread::hardware_concurrency());
  nth = std::min(nth, n_sets);
  auto parallel = [&](auto&& fn) {  // fn(i) for every set, on nth host threads
    std::atomic<int> next{0};
    auto worker = [&]() {
      for (int i; (i = next.fetch_add(1)) < n_sets;) fn(i);
    };
    std::vector<std::thread> pool;
    for (int t = 1; t < nth; ++t) pool.emplace_back(worker);
    worker();
    for (auto& th : pool) th.join();
  };
  parallel([&](int i) { prepare_one(sets[i], *opts, prep[i], res[i]); });
  for (int i = 0; i < n_sets; ++i)
    KV_REQUIRE(res[i].ok, KV_ERR_NUMERIC, "set %d: %s", i, res[i].err.c_str());
  if (opts->joint) {
    // one split of the record between keys and values for the whole table (the cache holds one record length
    // per tensor): the split that minimises the summed distortion; objectives within a relative 1e-9 of the
    // minimum tie, ties go to the split nearest the separate allocation's, then to fewer key words
    const int r_total = rwk + rwv, rmax = 1 + opts->max_bits * opts->d / 32;
    std::vector<int> cands;
    for (int r = 1; r < r_total; ++r)
      if (r <= rmax && r_total - r <= rmax) cands.push_back(r);
    std::vector<double> J(cands.size() * (size_t)n_sets);
    parallel([&](int i) {
      for (size_t c = 0; c < cands.size(); ++c)
        J[c * n_sets + i] = prep[i].rho * budget_distortion(prep[i].ik, cands[c], opts->max_bits, opts->d) +
                            budget_distortion(prep[i].iv, r_total - cands[c], opts->max_bits, opts->d);
    });
    std::vector<double> Jc(cands.size(), 0.0);
    double jmin = INFINITY;
    for (size_t c = 0; c < cands.size(); ++c) {
      for (int i = 0; i < n_sets; ++i) Jc[c] += J[c * n_sets + i];
      jmin = std::min(jmin, Jc[c]);
    }
    int best = -1;
    for (size_t c = 0; c < cands.size(); ++c) {
      if (!(Jc[c] <= jmin * (1.0 + 1e-9))) continue;
      if (best < 0 || std::abs(cands[c] - rwk) < std::abs(best - rwk) ||
          (std::abs(cands[c] - rwk) == std::abs(best - rwk) && cands[c] < best))
        best = cands[c];
    }
    KV_REQUIRE(best >= 1, KV_ERR_NUMERIC, "joint allocation: no finite split");
    rwv = r_total - best;
    rwk = best;
  }
  parallel([&](int i) { build_one(prep[i], rwk, rwv, *opts, res[i]); });
  kv_params* p = new kv_params();
  p->d = opts->d;
  p->n_sets = n_sets;
  p->max_bits = opts->max_bits;
  p->r_words[0] = rwk;
  p->r_words[1] = rwv;
  for (int t = 0; t < 2; ++t) {
    for (int i = 0; i < n_sets; ++i) {
      auto app = [](auto& dst, const auto& src) { dst.insert(dst.end(), src.begin(), src.end()); };
      app(p->T[t], res[i].T[t]);
      app(p->mu[t], res[i].mu[t]);
      app(p->sigma[t], res[i].sigma[t]);
      app(p->widths[t], res[i].widths[t]);
      app(p->eig[t], res[i].eig[t]);
      app(p->imp[t], res[i].imp[t]);
      app(p->Tinv[t], res[i].Tinv[t]);
    }
  }
  *out = p;
  return KV_OK;
}

extern "C" kv_status kv_params_get_inverse(const kv_params* p, int set, int tensor, float* Tinv) {
  clear_error();
  KV_REQUIRE(p && Tinv && (tensor == 0 || tensor == 1) && set >= 0 && set < p->n_sets, KV_ERR_INVALID_ARG,
             "kv_params_get_inverse: bad argument");
  KV_REQUIRE(!p->Tinv[tensor].empty(), KV_ERR_UNSUPPORTED, "tensor %d has an orthogonal transform (no inverse)",
             tensor);
  const size_t n = (size_t)p->d * p->d;
  memcpy(Tinv, &p->Tinv[tensor][(size_t)set * n], n * 4);
  return KV_OK;
}

extern "C" kv_status kv_params_set_inverse(kv_params* p, int tensor, const float* Tinv) {
  clear_error();
  KV_REQUIRE(p && (tensor == 0 || tensor == 1), KV_ERR_INVALID_ARG, "kv_params_set_inverse: bad argument");
  const size_t n = (size_t)p->n_sets * p->d * p->d;
  if (!Tinv) {
    p->Tinv[tensor].clear();
    return KV_OK;
  }
  KV_REQUIRE(finite_all(Tinv, n), KV_ERR_INVALID_ARG, "kv_params_set_inverse: non-finite entries");
  p->Tinv[tensor].assign(Tinv, Tinv + n);
  return KV_OK;
}

static constexpr double kPi = 3.14159265358979323846;

extern "C" kv_status kv_params_set_rope(kv_params* p, double base) {
  clear_error();
  KV_REQUIRE(p, KV_ERR_INVALID_ARG, "kv_params_set_rope: null table");
  KV_REQUIRE(std::isfinite(base) && base >= 0.0, KV_ERR_INVALID_ARG, "rotary base %g must be finite and >= 0", base);
  p->rope_base = base;
  return KV_OK;
}
extern "C" double kv_params_get_rope(const kv_params* p) { return p ? p->rope_base : 0.0; }

extern "C" kv_status kv_params_from_arrays(int d, int n_sets, const float* T_k, const float* mu_k,
                                           const float* sigma_k, const int32_t* widths_k, int r_words_k,
                                           const float* T_v, const float* mu_v, const float* sigma_v,
                                           const int32_t* widths_v, int r_words_v, kv_params** out) {
  clear_error();
  KV_REQUIRE(out && T_k && mu_k && sigma_k && widths_k && T_v && mu_v && sigma_v && widths_v && n_sets >= 1,
             KV_ERR_INVALID_ARG, "kv_params_from_arrays: null argument");
  KV_REQUIRE(d == D, KV_ERR_UNSUPPORTED, "d=%d unsupported (128 only)", d);
  const float* Ts[2] = {T_k, T_v};
  const float* mus[2] = {mu_k, mu_v};
  const float* sgs[2] = {sigma_k, sigma_v};
  const int32_t* ws[2] = {widths_k, widths_v};
  const int rws[2] = {r_words_k, r_words_v};
  kv_params* p = new kv_params();
  p->d = d;
  p->n_sets = n_sets;
  p->max_bits = MAX_BITS;
  for (int t = 0; t < 2; ++t) {
    if (rws[t] < 1 || rws[t] > MAX_RW) {
      delete p;
      KV_REQUIRE(false, KV_ERR_BUDGET, "r_words %d out of range 1..%d", rws[t], MAX_RW);
    }
    p->r_words[t] = rws[t];
    const size_t n = (size_t)n_sets * d;
    p->T[t].assign(Ts[t], Ts[t] + n * d);
    p->mu[t].assign(mus[t], mus[t] + n);
    p->sigma[t].assign(sgs[t], sgs[t] + n);
    p->widths[t].assign(ws[t], ws[t] + n);
    p->eig[t].resize(n);
    p->imp[t].assign(n, 0.0);
    for (int s = 0; s < n_sets; ++s) {
      for (int j = 0; j < d; ++j) {
        const size_t i = (size_t)s * d + j;
        if (!(p->sigma[t][i] > 0.f)) p->widths[t][i] = 0;
        if (p->widths[t][i] < 0 || p->widths[t][i] > MAX_BITS) {
          delete p;
          KV_REQUIRE(false, KV_ERR_INVALID_ARG, "set %d channel %d: width out of range 0..8", s, j);
        }
        p->eig[t][i] = (double)p->sigma[t][i] * p->sigma[t][i];
      }
      int word[D], pos[D];
      const int32_t* wt = &p->widths[t][(size_t)s * d];
      if (!(t == 0 ? kvtc::slot_layout(wt, d, rws[t], word, pos) : kvtc::token_slot_layout(wt, d, rws[t], word, pos))) {
        delete p;
        KV_REQUIRE(false, KV_ERR_BUDGET, "set %d tensor %d: widths do not fit the %d-word record layout", s, t,
                   rws[t]);
      }
    }
  }
  *out = p;
  return KV_OK;
}

// ------------------------------------------------------------------------------------------------------
// device copy of the table, with the derived arrays the kernels use
// ------------------------------------------------------------------------------------------------------
static uint16_t f32_to_bf16_rn(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  const uint32_t r = u + 0x7FFFu + ((u >> 16) & 1u);
  return (uint16_t)(r >> 16);
}
static float bf16_to_f32(uint16_t h) {
  const uint32_t u = (uint32_t)h << 16;
  float f;
  memcpy(&f, &u, 4);
  return f;
}

// Slot descriptor: code word u (0-based within the record's code words), bit r, width of the low-half and of
// the high-half code: u | r << 8 | b_lo << 16 | b_hi << 24 (all zero for an empty slot). Key slots hold the
// channel pair (2k, 2k+1) of one token; value slots hold channel j of the record's two tokens.
static uint32_t slot_descriptor(int u, int r, int b0, int b1) {
  if (u < 0 || (b0 == 0 && b1 == 0)) return 0u;
  return (uint32_t)u | ((uint32_t)r << 8) | ((uint32_t)b0 << 16) | ((uint32_t)b1 << 24);
}

static size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// The decode's order of the MMA channel dimension. The logit MMA's k index and the P.V MMA's row index may take the
// channels in any order (the q' operands and the value sums follow it), so a lane's two key pair slots of a
// 16-channel block - and a lane's two value channels - are coupled from one code word wherever the word holds two:
// the decode then loads that word once for both. items: n_blocks * lanes * 2 (pairs, or channels), word[item] (-1:
// no slot). A couple's slot 0 is real whenever it has a real slot; a real left alone in its word takes an item
// without a slot as partner (its couple still needs one load), or, where the blocks the decode reads (capacity
// couples) could not hold every real item that way, another lone real. Order: couples of one word, lone reals with
// a slotless partner, couples across words, slotless couples. Blocks whose couples all need one load get their bit
// in single_mask.
static void couple_positions(const int* word, int n_blocks, int lanes, int capacity, std::vector<int>& order,
                             uint32_t& single_mask) {
  const int n = n_blocks * lanes * 2;
  std::vector<std::pair<int, int>> same, lone, cross, empty;
  std::vector<int> dummies, left;
  int max_word = -1;
  for (int i = 0; i < n; ++i) max_word = std::max(max_word, word[i]);
  for (int u = 0; u <= max_word; ++u) {
    int held = -1;
    for (int i = 0; i < n; ++i)
      if (word[i] == u) {
        if (held < 0) {
          held = i;
        } else {
          same.emplace_back(held, i);
          held = -1;
        }
      }
    if (held >= 0) left.push_back(held);
  }
  for (int i = 0; i < n; ++i)
    if (word[i] < 0) dummies.push_back(i);
  const int L = (int)left.size();
  int x = std::max(0, (int)same.size() + L - capacity);  // couples across words needed to fit the capacity
  x = std::min(x, L / 2);
  x = std::max(x, (L - (int)dummies.size() + 1) / 2);   // and where slotless partners run out
  x = std::min(x, L / 2);
  int li = 0;
  for (int c = 0; c < x; ++c, li += 2) cross.emplace_back(left[li], left[li + 1]);
  size_t di = 0;
  std::vector<int> rest;
  for (; li < L; ++li) {
    if (di < dummies.size())
      lone.emplace_back(left[li], dummies[di++]);
    else
      rest.push_back(left[li]);
  }
  for (; di < dummies.size(); ++di) rest.push_back(dummies[di]);  // (reals first: left over only when unpaired)
  std::vector<int> rr, dd;
  for (int r : rest) (word[r] >= 0 ? rr : dd).push_back(r);
  for (size_t i = 0; i + 1 < rr.size(); i += 2) cross.emplace_back(rr[i], rr[i + 1]);
  if (rr.size() % 2) dd.insert(dd.begin(), rr.back());
  for (size_t i = 0; i + 1 < dd.size(); i += 2) empty.emplace_back(dd[i], dd[i + 1]);
  std::vector<std::pair<int, int>> all(same);
  const size_t n_one = same.size() + lone.size();  // couples needing one load: same, lone, and the slotless ones
  all.insert(all.end(), lone.begin(), lone.end());
  all.insert(all.end(), cross.begin(), cross.end());
  all.insert(all.end(), empty.begin(), empty.end());
  order.assign(n, 0);
  single_mask = 0u;
  for (int b = 0; b < n_blocks; ++b) {
    bool single = true;
    for (int l = 0; l < lanes; ++l) {
      const size_t c = (size_t)b * lanes + l;
      order[(b * lanes + l) * 2 + 0] = all[c].first;
      order[(b * lanes + l) * 2 + 1] = all[c].second;
      const bool one = c < n_one || c >= n_one + cross.size();
      single = single && one;
    }
    if (single) single_mask |= 1u << b;
  }
}

extern "C" kv_status kv_params_upload(kv_params* p, kv_stream_t stream) {
  clear_error();
  KV_REQUIRE(p, KV_ERR_INVALID_ARG, "kv_params_upload: null");
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (p->dev_blob) {
    cudaFree(p->dev_blob);
    p->dev_blob = nullptr;
  }
  const int S = p->n_sets, d = p->d;
  // host staging of every device array, laid out in one blob
  struct Piece { size_t off, bytes; };
  std::vector<uint8_t> blob;
  auto reserve = [&](size_t bytes) {
    const size_t off = align_up(blob.size(), 256);
    blob.resize(off + bytes);
    return Piece{off, bytes};
  };
  Piece pT[2], pTT[2], pTq[2], pTs[2], pmu[2], psg[2], pinv[2], pbase[2], pw[2], pnz[2], psl[2], psc[2], pws[2],
      pws2[2], psmx[2], pslp[2], pidx[2], pmask;
  for (int t = 0; t < 2; ++t) {
    pT[t] = reserve((size_t)S * d * d * 4);
    pTT[t] = reserve((size_t)S * d * d * 4);
    pTq[t] = p->Tinv[t].empty() ? pTT[t] : reserve((size_t)S * d * d * 4);
    pTs[t] = reserve((size_t)S * 3 * d * d * 2);
    pmu[t] = reserve((size_t)S * d * 4);
    psg[t] = reserve((size_t)S * d * 4);
    pinv[t] = reserve((size_t)S * d * 4);
    pbase[t] = reserve((size_t)S * d * 4);
    psc[t] = reserve((size_t)S * d * d * 4);
    pws[t] = reserve((size_t)S * d * 4);
    pws2[t] = reserve((size_t)S * d * 4);
    psmx[t] = reserve((size_t)S * 4);
    pw[t] = reserve((size_t)S * d);
    pnz[t] = reserve((size_t)S * 4);
    psl[t] = reserve((size_t)S * d * 4);
    pslp[t] = reserve((size_t)S * (t == 0 ? 64 : 128) * 4);
    pidx[t] = reserve((size_t)S * (t == 0 ? 64 : 128));
  }
  pmask = reserve((size_t)S * 4);
  // the rotary embedding's frequencies as fractions of a turn, 64-bit fixed point
  const bool has_rope = p->rope_base > 0.0;
  const Piece prope = has_rope ? reserve((size_t)(D / 2) * 8) : Piece{0, 0};
  if (has_rope) {
    unsigned long long* rt = (unsigned long long*)&blob[prope.off];
    for (int i = 0; i < D / 2; ++i) {
      const double f = std::pow(p->rope_base, -2.0 * i / D) / (2.0 * kPi);  // turns per position, < 1/(2 pi)
      rt[i] = (unsigned long long)std::llround(std::ldexp(f, 64));
    }
  }
  int single_word = 3;
  for (int t = 0; t < 2; ++t) {
    float* T = (float*)&blob[pT[t].off];
    float* TT = (float*)&blob[pTT[t].off];
    uint16_t* Ts = (uint16_t*)&blob[pTs[t].off];
    float* mu = (float*)&blob[pmu[t].off];
    float* sg = (float*)&blob[psg[t].off];
    float* inv = (float*)&blob[pinv[t].off];
    float* base = (float*)&blob[pbase[t].off];
    float* tsc = (float*)&blob[psc[t].off];
    float* wsum = (float*)&blob[pws[t].off];
    float* wsum2 = (float*)&blob[pws2[t].off];
    float* smx = (float*)&blob[psmx[t].off];
    uint8_t* w8 = (uint8_t*)&blob[pw[t].off];
    int32_t* nz = (int32_t*)&blob[pnz[t].off];
    uint32_t* sl = (uint32_t*)&blob[psl[t].off];
    const bool has_inv = !p->Tinv[t].empty();
    float* Tq = (float*)&blob[pTq[t].off];
    for (int s = 0; s < S; ++s) {
      const float* Tsrc = &p->T[t][(size_t)s * d * d];
      // inverse of T: Inv(k, j) = (T^-1)[k][j], T[j][k] for an orthogonal T
      const float* Isrc = has_inv ? &p->Tinv[t][(size_t)s * d * d] : nullptr;
      auto Inv = [&](int k, int j) -> double {
        return has_inv ? (double)Isrc[(size_t)k * d + j] : (double)Tsrc[(size_t)j * d + k];
      };
      if (has_inv)
        for (size_t i = 0; i < (size_t)d * d; ++i) Tq[(size_t)s * d * d + i] = Isrc[i];
      for (int j = 0; j < d; ++j)
        for (int k = 0; k < d; ++k) {
          const float v = Tsrc[(size_t)j * d + k];
          T[(size_t)s * d * d + (size_t)j * d + k] = v;
          TT[(size_t)s * d * d + (size_t)k * d + j] = v;
          const uint16_t hi = f32_to_bf16_rn(v);
          const float r1 = v - bf16_to_f32(hi);
          const uint16_t mid = f32_to_bf16_rn(r1);
          const float r2 = r1 - bf16_to_f32(mid);
          const uint16_t lo = f32_to_bf16_rn(r2);
          Ts[((size_t)s * 3 + 0) * d * d + (size_t)j * d + k] = hi;
          Ts[((size_t)s * 3 + 1) * d * d + (size_t)j * d + k] = mid;
          Ts[((size_t)s * 3 + 2) * d * d + (size_t)j * d + k] = lo;
        }
      int n_nz = 0;
      std::vector<int32_t> wv(d);
      for (int j = 0; j < d; ++j) {
        const size_t i = (size_t)s * d + j;
        mu[i] = p->mu[t][i];
        sg[i] = p->sigma[t][i];
        const int w = p->sigma[t][i] > 0.f ? p->widths[t][i] : 0;
        inv[i] = w > 0 ? (float)(1.0 / (double)p->sigma[t][i]) : 0.f;
        w8[i] = (uint8_t)w;
        wv[j] = w;
        if (w > 0) n_nz = j + 1;
      }
      nz[s] = n_nz;
      for (int k = 0; k < d; ++k) {
        double acc = 0.0;
        for (int j = 0; j < d; ++j) acc += Inv(k, j) * (double)p->mu[t][(size_t)s * d + j];
        base[(size_t)s * d + k] = (float)acc;
      }
      // The decode's folded constants. Slot width w_j: the wider code width of a key channel pair (both channels
      // share one slot), b_j itself for values. Scaled rows T'[j][k] = T[j][k] sigma_j (0 for zero-width rows);
      // w_k = sum_{b_j > 0} T[j][k] sigma_j; w2_k = sum_{b_j > 0} T[j][k] sigma_j (2^(w_j - b_j) - 2^(-b_j - 1));
      // smax = max_{b_j > 0} sigma_j 2^(w_j - b_j). Keys: q.w, q.w2 and smax give the logit constants and the
      // scale of the q coefficients; values: the rows and vectors map rotated-basis sums to the original basis.
      std::vector<int> slotw(d);
      for (int j = 0; j < d; ++j) slotw[j] = t == 0 ? std::max(wv[j], wv[j ^ 1]) : wv[j];
      // (with an inverse, |(T^-T q)_j| <= |q| |column j of T^-1|: the column norm enters the bound)
      double smax = 0.0;
      for (int j = 0; j < d; ++j)
        if (wv[j] > 0) {
          double cn = 1.0;
          if (has_inv) {
            double n2 = 0.0;
            for (int k = 0; k < d; ++k) n2 += Inv(k, j) * Inv(k, j);
            cn = std::sqrt(n2);
          }
          smax = std::max(smax, cn * (double)p->sigma[t][(size_t)s * d + j] * std::ldexp(1.0, slotw[j] - wv[j]));
        }
      smx[s] = (float)smax;
      for (int k = 0; k < d; ++k) {
        double wacc = 0.0, wacc2 = 0.0;
        for (int j = 0; j < d; ++j) {
          const double tj = Inv(k, j);
          const double sj = (double)p->sigma[t][(size_t)s * d + j];
          const int bj = wv[j];
          tsc[(size_t)s * d * d + (size_t)j * d + k] = bj > 0 ? (float)(tj * sj) : 0.f;
          if (bj > 0) {
            wacc += tj * sj;
            wacc2 += tj * sj * (std::ldexp(1.0, slotw[j] - bj) - std::ldexp(1.0, -bj - 1));
          }
        }
        wsum[(size_t)s * d + k] = (float)wacc;
        wsum2[(size_t)s * d + k] = (float)wacc2;
      }
      int word[D], pos[D];
      uint32_t* sls = sl + (size_t)s * d;
      if (t == 0) {  // key slots: one per channel pair (entries d/2 .. d-1 unused)
        kvtc::slot_layout(wv.data(), d, p->r_words[t], word, pos);
        for (int k = 0; k < d / 2; ++k) sls[k] = slot_descriptor(word[k], pos[k], wv[2 * k], wv[2 * k + 1]);
        for (int k = d / 2; k < d; ++k) sls[k] = 0u;
      } else {       // value slots: one per channel, the same width for both tokens of a record
        kvtc::token_slot_layout(wv.data(), d, p->r_words[t], word, pos);
        for (int j = 0; j < d; ++j) sls[j] = slot_descriptor(word[j], pos[j], wv[j], wv[j]);
      }
      // the decode's lane order (keys: 8 blocks x 4 lanes x 2 pair slots; values: 8 blocks x 8 lanes x 2
      // channels), the slot descriptors in that order, and the blocks whose couples share a word
      {
        const int lanes = t == 0 ? 4 : 8, n_items = 8 * lanes * 2;
        std::vector<int> ord;
        uint32_t single = 0u;
        // the decode reads the channel blocks below the last nonzero width: their items (zero-width ones too) are
        // ordered among themselves; the blocks past them keep the storage order
        const int blocks_read = (n_nz + 15) / 16;
        if (blocks_read > 0) couple_positions(word, blocks_read, lanes, blocks_read * lanes, ord, single);
        for (int i = (int)ord.size(); i < n_items; ++i) ord.push_back(i);
        uint32_t* slp = (uint32_t*)&blob[pslp[t].off] + (size_t)s * n_items;
        uint8_t* idx = (uint8_t*)&blob[pidx[t].off] + (size_t)s * n_items;
        for (int i = 0; i < n_items; ++i) {
          slp[i] = sls[ord[i]];
          idx[i] = (uint8_t)ord[i];
        }
        uint32_t* msk = (uint32_t*)&blob[pmask.off] + s;
        *msk = t == 0 ? single : (*msk | (single << 8));
        const uint32_t need = (1u << blocks_read) - 1u;  // the blocks the decode reads
        if ((single & need) != need) single_word &= ~(1 << t);
      }
    }
  }
  void* dblob = nullptr;
  e = cudaMalloc(&dblob, blob.size());
  if (e != cudaSuccess) return cuda_fail(e, "cudaMalloc(params)");
  e = cudaMemcpyAsync(dblob, blob.data(), blob.size(), cudaMemcpyHostToDevice, (cudaStream_t)stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize((cudaStream_t)stream);
  if (e != cudaSuccess) {
    cudaFree(dblob);
    return cuda_fail(e, "upload params");
  }
  p->dev_blob = dblob;
  p->dev_bytes = blob.size();
  p->device = dev;
  uint8_t* b = (uint8_t*)dblob;
  for (int t = 0; t < 2; ++t) {
    TensorDev& td = p->dev.t[t];
    td.T = (const float*)(b + pT[t].off);
    td.TT = (const float*)(b + pTT[t].off);
    td.Tq = (const float*)(b + pTq[t].off);
    td.Tsplit = (const __nv_bfloat16*)(b + pTs[t].off);
    td.mu = (const float*)(b + pmu[t].off);
    td.sigma = (const float*)(b + psg[t].off);
    td.inv_sigma = (const float*)(b + pinv[t].off);
    td.base = (const float*)(b + pbase[t].off);
    td.Tsc = (const float*)(b + psc[t].off);
    td.wsum = (const float*)(b + pws[t].off);
    td.wsum2 = (const float*)(b + pws2[t].off);
    td.smax = (const float*)(b + psmx[t].off);
    td.widths = (const uint8_t*)(b + pw[t].off);
    td.nz = (const int32_t*)(b + pnz[t].off);
    td.slots = (const uint32_t*)(b + psl[t].off);
    td.slp = (const uint32_t*)(b + pslp[t].off);
    td.idx = (const uint8_t*)(b + pidx[t].off);
    td.single = (const uint32_t*)(b + pmask.off);
    td.r_words = p->r_words[t];
    const int32_t* nzh = (const int32_t*)&blob[pnz[t].off];
    td.min_nz = S > 0 ? *std::min_element(nzh, nzh + S) : 0;
    td.max_nz = S > 0 ? *std::max_element(nzh, nzh + S) : 0;
  }
  p->dev.n_sets = S;
  p->dev.single_word = single_word;
  p->dev.rope_turns = has_rope ? (const unsigned long long*)(b + prope.off) : nullptr;
  return KV_OK;
}

extern "C" int kv_params_num_sets(const kv_params* p) { return p ? p->n_sets : 0; }
extern "C" int kv_params_record_words(const kv_params* p, int tensor) {
  return (p && (tensor == 0 || tensor == 1)) ? p->r_words[tensor] : 0;
}

extern "C" kv_status kv_params_info(const kv_params* p, int set, int tensor, int32_t* widths, double* eigvals,
                                    double* importance, float* T, float* mu, float* sigma) {
  clear_error();
  KV_REQUIRE(p && set >= 0 && set < p->n_sets && (tensor == 0 || tensor == 1), KV_ERR_INVALID_ARG,
             "kv_params_info: bad argument");
  const int d = p->d;
  const size_t o = (size_t)set * d;
  for (int j = 0; j < d; ++j) {
    if (widths) widths[j] = p->widths[tensor][o + j];
    if (eigvals) eigvals[j] = p->eig[tensor][o + j];
    if (importance) importance[j] = p->imp[tensor][o + j];
    if (mu) mu[j] = p->mu[tensor][o + j];
    if (sigma) sigma[j] = p->sigma[tensor][o + j];
  }
  if (T) memcpy(T, &p->T[tensor][o * d], (size_t)d * d * 4);
  return KV_OK;
}

extern "C" void kv_params_free(kv_params* p) {
  if (!p) return;
  if (p->dev_blob) cudaFree(p->dev_blob);
  delete p;
}

// ------------------------------------------------------------------------------------------------------
// persistence: "KVTC" magic, version, dims, arrays, CRC-32 (IEEE 802.3 polynomial, reflected) of the payload
// ------------------------------------------------------------------------------------------------------
static uint32_t crc32(const uint8_t* data, size_t n) {
  uint32_t c = 0xFFFFFFFFu;
  for (size_t i = 0; i < n; ++i) {
    c ^= data[i];
    for (int k = 0; k < 8; ++k) c = (c >> 1) ^ (0xEDB88320u & (0u - (c & 1u)));
  }
  return ~c;
}

static const uint32_t FILE_MAGIC = 0x4354564Bu;  // "KVTC"
// 2: a per-tensor inverse (non-orthogonal transform) after version 1's data; 3: then the rotary embedding's base
static const uint32_t FILE_VERSION = 3;

extern "C" kv_status kv_params_save(const kv_params* p, const char* path) {
  clear_error();
  KV_REQUIRE(p && path, KV_ERR_INVALID_ARG, "kv_params_save: null");
  std::vector<uint8_t> pay;
  auto put = [&](const void* src, size_t n) {
    const uint8_t* s = (const uint8_t*)src;
    pay.insert(pay.end(), s, s + n);
  };
  int32_t hdr[5] = {p->d, p->n_sets, p->max_bits, p->r_words[0], p->r_words[1]};
  put(hdr, sizeof(hdr));
  for (int t = 0; t < 2; ++t) {
    put(p->T[t].data(), p->T[t].size() * 4);
    put(p->mu[t].data(), p->mu[t].size() * 4);
    put(p->sigma[t].data(), p->sigma[t].size() * 4);
    put(p->widths[t].data(), p->widths[t].size() * 4);
    put(p->eig[t].data(), p->eig[t].size() * 8);
    put(p->imp[t].data(), p->imp[t].size() * 8);
  }
  for (int t = 0; t < 2; ++t) {
    const int32_t has = p->Tinv[t].empty() ? 0 : 1;
    put(&has, 4);
    if (has) put(p->Tinv[t].data(), p->Tinv[t].size() * 4);
  }
  put(&p->rope_base, 8);
  FILE* f = fopen(path, "wb");
  KV_REQUIRE(f, KV_ERR_IO, "cannot open %s for writing", path);
  const uint32_t head[4] = {FILE_MAGIC, FILE_VERSION, (uint32_t)pay.size(), crc32(pay.data(), pay.size())};
  bool ok = fwrite(head, sizeof(head), 1, f) == 1 && fwrite(pay.data(), 1, pay.size(), f) == pay.size();
  ok = (fclose(f) == 0) && ok;
  KV_REQUIRE(ok, KV_ERR_IO, "write to %s failed", path);
  return KV_OK;
}

extern "C" kv_status kv_params_load(const char* path, kv_params** out) {
  clear_error();
  KV_REQUIRE(path && out, KV_ERR_INVALID_ARG, "kv_params_load: null");
  FILE* f = fopen(path, "rb");
  KV_REQUIRE(f, KV_ERR_IO, "cannot open %s", path);
  uint32_t head[4];
  if (fread(head, sizeof(head), 1, f) != 1 || head[0] != FILE_MAGIC || head[1] < 1 || head[1] > FILE_VERSION) {
    fclose(f);
    KV_REQUIRE(false, KV_ERR_IO, "%s: not a parameter file of version 1..%u", path, FILE_VERSION);
  }
  std::vector<uint8_t> pay(head[2]);
  const size_t got = fread(pay.data(), 1, pay.size(), f);
  fclose(f);
  KV_REQUIRE(got == pay.size(), KV_ERR_IO, "%s: truncated", path);
  KV_REQUIRE(crc32(pay.data(), pay.size()) == head[3], KV_ERR_IO, "%s: checksum mismatch", path);
  size_t pos = 0;
  auto get = [&](void* dst, size_t n) {
    if (pos + n > pay.size()) return false;
    memcpy(dst, &pay[pos], n);
    pos += n;
    return true;
  };
  int32_t hdr[5];
  KV_REQUIRE(get(hdr, sizeof(hdr)), KV_ERR_IO, "%s: truncated header", path);
  KV_REQUIRE(hdr[0] == D && hdr[1] >= 1 && hdr[3] >= 1 && hdr[4] >= 1 && hdr[3] <= MAX_RW && hdr[4] <= MAX_RW,
             KV_ERR_IO, "%s: bad dimensions", path);
  kv_params* p = new kv_params();
  p->d = hdr[0];
  p->n_sets = hdr[1];
  p->max_bits = hdr[2];
  p->r_words[0] = hdr[3];
  p->r_words[1] = hdr[4];
  const size_t n = (size_t)p->n_sets * p->d;
  bool ok = true;
  for (int t = 0; t < 2 && ok; ++t) {
    p->T[t].resize(n * p->d);
    p->mu[t].resize(n);
    p->sigma[t].resize(n);
    p->widths[t].resize(n);
    p->eig[t].resize(n);
    p->imp[t].resize(n);
    ok = get(p->T[t].data(), n * p->d * 4) && get(p->mu[t].data(), n * 4) && get(p->sigma[t].data(), n * 4) &&
         get(p->widths[t].data(), n * 4) && get(p->eig[t].data(), n * 8) && get(p->imp[t].data(), n * 8);
  }
  for (int t = 0; t < 2 && ok && head[1] >= 2; ++t) {
    int32_t has = 0;
    ok = get(&has, 4) && (has == 0 || has == 1);
    if (ok && has) {
      p->Tinv[t].resize(n * p->d);
      ok = get(p->Tinv[t].data(), n * p->d * 4);
    }
  }
  if (ok && head[1] >= 3) ok = get(&p->rope_base, 8) && std::isfinite(p->rope_base) && p->rope_base >= 0.0;
  if (!ok || pos != pay.size()) {
    delete p;
    KV_REQUIRE(false, KV_ERR_IO, "%s: payload size mismatch", path);
  }
  *out = p;
  return KV_OK;
}

// ------------------------------------------------------------------------------------------------------
// sizing
// ------------------------------------------------------------------------------------------------------
extern "C" size_t kv_cache_bytes(const kv_params* p, int tensor, int B, int Hkv, int64_t T_cap) {
  if (!p || (tensor != 0 && tensor != 1) || B < 1 || Hkv < 1 || T_cap < 1) return 0;
  return (size_t)B * Hkv * (size_t)T_cap * p->r_words[tensor] * 4;
}

static int current_device() {
  int dev = 0;
  cudaGetDevice(&dev);
  return dev;
}

extern "C" size_t kv_decode_workspace_bytes(const kv_params* p, int B, int Hkv, int Hq, int64_t T_cap) {
  if (!p || B < 1 || Hkv < 1 || Hq < Hkv || T_cap < 1) return 0;
  return kvtc::decode_layout(B, Hkv, Hq, T_cap, current_device()).total;
}

extern "C" size_t kv_decode_bf16_workspace_bytes(int B, int Hkv, int Hq, int64_t T_cap) {
  if (B < 1 || Hkv < 1 || Hq < Hkv || T_cap < 1) return 0;
  return kvtc::decode_bf16_layout(B, Hkv, T_cap, current_device()).total;
}

// ------------------------------------------------------------------------------------------------------
// validated entry points
// ------------------------------------------------------------------------------------------------------
static bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

static kv_status check_params_on_device(const kv_params* p, int* dev_out = nullptr) {
  KV_REQUIRE(p, KV_ERR_INVALID_ARG, "null parameter table");
  KV_REQUIRE(p->dev_blob, KV_ERR_INVALID_ARG, "parameter table not uploaded (kv_params_upload)");
  const int dev = current_device();
  KV_REQUIRE(p->device == dev, KV_ERR_INVALID_ARG, "parameter table uploaded to device %d, current device is %d",
             p->device, dev);
  if (dev_out) *dev_out = dev;
  return KV_OK;
}

static kv_status check_cache(const kv_params* p, const kv_cache* c, int B) {
  KV_REQUIRE(c && c->k_rec && c->v_rec, KV_ERR_INVALID_ARG, "null cache");
  KV_REQUIRE(aligned16(c->k_rec) && aligned16(c->v_rec), KV_ERR_INVALID_ARG, "cache buffers must be 16-byte aligned");
  KV_REQUIRE(c->B >= 1 && c->Hkv >= 1 && c->T_cap >= 16 && c->T_cap % 16 == 0, KV_ERR_INVALID_ARG,
             "cache dims B=%d Hkv=%d T_cap=%lld (T_cap must be a positive multiple of 16)", c->B, c->Hkv,
             (long long)c->T_cap);
  KV_REQUIRE(B >= 1 && B <= c->B, KV_ERR_INVALID_ARG, "batch %d outside cache batch %d", B, c->B);
  const long long need = c->per_seq_params ? (long long)c->B * c->Hkv : c->Hkv;
  KV_REQUIRE(need <= p->n_sets, KV_ERR_INVALID_ARG, "cache needs %lld parameter sets, table has %d", need, p->n_sets);
  return KV_OK;
}

static int g_encode_path = 0;

extern "C" kv_status kv_debug_set_encode_path(int path) {
  KV_REQUIRE(path >= 0 && path <= 2, KV_ERR_INVALID_ARG, "encode path 0..2");
  g_encode_path = path;
  return KV_OK;
}

extern "C" kv_status kv_encode(const kv_params* p, const kv_cache* c, const void* k, const void* v, int dtype,
                               int B, int64_t t_new, const int64_t* dst_pos_dev, kv_stream_t stream) {
  clear_error();
  kv_status st;
  if ((st = check_params_on_device(p)) != KV_OK) return st;
  if ((st = check_cache(p, c, B)) != KV_OK) return st;
  KV_REQUIRE(dtype == KV_DTYPE_BF16 || dtype == KV_DTYPE_F32, KV_ERR_UNSUPPORTED, "dtype %d unsupported", dtype);
  KV_REQUIRE(t_new >= 0 && t_new <= c->T_cap, KV_ERR_INVALID_ARG, "t_new=%lld outside 0..T_cap", (long long)t_new);
  if (t_new == 0) return KV_OK;
  KV_REQUIRE(k && v && dst_pos_dev, KV_ERR_INVALID_ARG, "null k, v or dst_pos");
  KV_REQUIRE(aligned16(k) && aligned16(v), KV_ERR_INVALID_ARG, "k and v must be 16-byte aligned");
  return kvtc::launch_encode(p->dev, kvtc::dense_view(*c), k, v, dtype, B, t_new, dst_pos_dev, g_encode_path,
                             (cudaStream_t)stream);
}

namespace kvtc {
// Argument checks shared by the decode entry points (everything except the workspace).
kv_status check_decode_args(const kv_params* p, const kv_cache* c, const void* q, int B, int Hq,
                            const int32_t* seq_lens_dev, float softmax_scale, const float* out, int* dev) {
  kv_status st;
  if ((st = check_params_on_device(p, dev)) != KV_OK) return st;
  if ((st = check_cache(p, c, B)) != KV_OK) return st;
  KV_REQUIRE(q && seq_lens_dev && out, KV_ERR_INVALID_ARG, "null q, seq_lens or out");
  KV_REQUIRE(Hq >= c->Hkv && Hq % c->Hkv == 0, KV_ERR_INVALID_ARG, "Hq=%d not a multiple of Hkv=%d", Hq, c->Hkv);
  KV_REQUIRE(Hq / c->Hkv <= MAX_G, KV_ERR_UNSUPPORTED, "g = Hq/Hkv = %d > 8", Hq / c->Hkv);
  KV_REQUIRE(aligned16(q) && aligned16(out), KV_ERR_INVALID_ARG, "q and out must be 16-byte aligned");
  KV_REQUIRE(std::isfinite(softmax_scale), KV_ERR_INVALID_ARG, "non-finite softmax scale");
  return KV_OK;
}
}  // namespace kvtc

extern "C" kv_status kv_attend_decode(const kv_params* p, const kv_cache* c, const void* q, int B, int Hq,
                                      const int32_t* seq_lens_dev, float softmax_scale, float* out,
                                      void* workspace, size_t ws_bytes, kv_stream_t stream) {
  clear_error();
  kv_status st;
  int dev = 0;
  if ((st = kvtc::check_decode_args(p, c, q, B, Hq, seq_lens_dev, softmax_scale, out, &dev)) != KV_OK) return st;
  KV_REQUIRE(workspace && aligned16(workspace), KV_ERR_INVALID_ARG, "workspace null or not 16-byte aligned");
  const DecodeLayout L = kvtc::decode_layout(B, c->Hkv, Hq, c->T_cap, dev);
  KV_REQUIRE(ws_bytes >= L.total, KV_ERR_INVALID_ARG, "workspace %zu bytes < %zu needed", ws_bytes, L.total);
  return kvtc::launch_decode(p->dev, kvtc::dense_view(*c), q, B, Hq, seq_lens_dev, nullptr, softmax_scale, out,
                             workspace, L, (cudaStream_t)stream);
}

// ------------------------------------------------------------------------------------------------------
// paged, multi-layer cache
// ------------------------------------------------------------------------------------------------------
namespace kvtc {
CacheView dense_view(const kv_cache& c) {
  CacheView v{};
  v.rec[0] = c.k_rec;
  v.rec[1] = c.v_rec;
  v.bt = nullptr;
  v.T_cap = c.T_cap;
  v.B = c.B;
  v.Hkv = c.Hkv;
  v.per_seq = c.per_seq_params;
  v.set_base = 0;
  v.sets_per_layer = c.per_seq_params ? c.B * c.Hkv : c.Hkv;
  return v;
}

static CacheView paged_view(const kv_paged_cache& c) {
  CacheView v{};
  v.rec[0] = c.k_pages;
  v.rec[1] = c.v_pages;
  v.bt = c.block_table;
  v.T_cap = (long long)c.max_pages * c.page_tokens;
  v.n_pages = c.n_pages;
  v.P = c.page_tokens;
  v.P_shift = 0;
  while ((1 << v.P_shift) < c.page_tokens) ++v.P_shift;
  v.max_pages = c.max_pages;
  v.B = c.B;
  v.Hkv = c.Hkv;
  v.per_seq = c.per_seq_params;
  v.sets_per_layer = c.per_seq_params ? c.B * c.Hkv : c.Hkv;
  v.set_base = c.first_layer * v.sets_per_layer;
  return v;
}
}  // namespace kvtc

static kv_status check_paged_cache(const kv_params* p, const kv_paged_cache* c) {
  KV_REQUIRE(c && c->k_pages && c->v_pages && c->block_table, KV_ERR_INVALID_ARG, "null paged cache or block table");
  KV_REQUIRE(aligned16(c->k_pages) && aligned16(c->v_pages), KV_ERR_INVALID_ARG,
             "page pools must be 16-byte aligned");
  KV_REQUIRE(c->page_tokens >= 32 && c->page_tokens <= (1 << 20) && (c->page_tokens & (c->page_tokens - 1)) == 0,
             KV_ERR_INVALID_ARG, "page_tokens=%d must be a power of two from 32 to 2^20", c->page_tokens);
  KV_REQUIRE(c->n_pages >= 1 && c->max_pages >= 1 && c->B >= 1 && c->Hkv >= 1 && c->n_layers >= 1 &&
                 c->first_layer >= 0,
             KV_ERR_INVALID_ARG, "paged cache dims n_pages=%lld max_pages=%d B=%d Hkv=%d n_layers=%d first_layer=%d",
             (long long)c->n_pages, c->max_pages, c->B, c->Hkv, c->n_layers, c->first_layer);
  KV_REQUIRE((long long)c->n_layers * c->B <= 65535 && c->Hkv <= 65535, KV_ERR_UNSUPPORTED,
             "n_layers * B = %lld and Hkv = %d must stay within 65535", (long long)c->n_layers * c->B, c->Hkv);
  KV_REQUIRE((long long)c->max_pages * c->page_tokens < (1LL << 31), KV_ERR_INVALID_ARG,
             "max_pages * page_tokens = %lld must stay below 2^31", (long long)c->max_pages * c->page_tokens);
  const long long S = c->per_seq_params ? (long long)c->B * c->Hkv : c->Hkv;
  KV_REQUIRE((c->first_layer + (long long)c->n_layers) * S <= p->n_sets, KV_ERR_INVALID_ARG,
             "layers %d..%d need %lld parameter sets, table has %d", c->first_layer, c->first_layer + c->n_layers - 1,
             (c->first_layer + (long long)c->n_layers) * S, p->n_sets);
  return KV_OK;
}

extern "C" size_t kv_paged_cache_bytes(const kv_params* p, int tensor, int64_t n_pages, int page_tokens, int Hkv) {
  if (!p || (tensor != 0 && tensor != 1) || n_pages < 1 || page_tokens < 1 || Hkv < 1) return 0;
  return (size_t)n_pages * Hkv * (size_t)page_tokens * p->r_words[tensor] * 4;
}

extern "C" kv_status kv_encode_paged(const kv_params* p, const kv_paged_cache* c, const void* k, const void* v,
                                     int dtype, int64_t t_new, const int64_t* dst_pos_dev, kv_stream_t stream) {
  clear_error();
  kv_status st;
  if ((st = check_params_on_device(p)) != KV_OK) return st;
  if ((st = check_paged_cache(p, c)) != KV_OK) return st;
  KV_REQUIRE(dtype == KV_DTYPE_BF16 || dtype == KV_DTYPE_F32, KV_ERR_UNSUPPORTED, "dtype %d unsupported", dtype);
  const long long cap = (long long)c->max_pages * c->page_tokens;
  KV_REQUIRE(t_new >= 0 && t_new <= cap, KV_ERR_INVALID_ARG, "t_new=%lld outside 0..%lld", (long long)t_new, cap);
  if (t_new == 0) return KV_OK;
  KV_REQUIRE(k && v && dst_pos_dev, KV_ERR_INVALID_ARG, "null k, v or dst_pos");
  KV_REQUIRE(aligned16(k) && aligned16(v), KV_ERR_INVALID_ARG, "k and v must be 16-byte aligned");
  return kvtc::launch_encode(p->dev, kvtc::paged_view(*c), k, v, dtype, c->n_layers * c->B, t_new, dst_pos_dev,
                             g_encode_path, (cudaStream_t)stream);
}

extern "C" size_t kv_decode_paged_workspace_bytes(const kv_params* p, const kv_paged_cache* c, int Hq) {
  if (!p || !c || c->B < 1 || c->n_layers < 1 || c->Hkv < 1 || Hq < c->Hkv || c->max_pages < 1 || c->page_tokens < 1)
    return 0;
  return kvtc::decode_layout(c->n_layers * c->B, c->Hkv, Hq, (int64_t)c->max_pages * c->page_tokens,
                             current_device()).total;
}

extern "C" kv_status kv_attend_decode_paged(const kv_params* p, const kv_paged_cache* c, const void* q, int Hq,
                                            const int32_t* seq_lens_dev, const int32_t* q_pos_dev,
                                            float softmax_scale, float* out, void* workspace, size_t ws_bytes,
                                            kv_stream_t stream) {
  clear_error();
  kv_status st;
  int dev = 0;
  if ((st = check_params_on_device(p, &dev)) != KV_OK) return st;
  if ((st = check_paged_cache(p, c)) != KV_OK) return st;
  KV_REQUIRE(q && seq_lens_dev && out, KV_ERR_INVALID_ARG, "null q, seq_lens or out");
  KV_REQUIRE(Hq >= c->Hkv && Hq % c->Hkv == 0, KV_ERR_INVALID_ARG, "Hq=%d not a multiple of Hkv=%d", Hq, c->Hkv);
  KV_REQUIRE(Hq / c->Hkv <= MAX_G, KV_ERR_UNSUPPORTED, "g = Hq/Hkv = %d > 8", Hq / c->Hkv);
  KV_REQUIRE(aligned16(q) && aligned16(out), KV_ERR_INVALID_ARG, "q and out must be 16-byte aligned");
  KV_REQUIRE(std::isfinite(softmax_scale), KV_ERR_INVALID_ARG, "non-finite softmax scale");
  KV_REQUIRE(!q_pos_dev || p->dev.rope_turns, KV_ERR_INVALID_ARG,
             "query positions given but the parameter table has no rotary embedding (kv_params_set_rope, then upload)");
  KV_REQUIRE(workspace && aligned16(workspace), KV_ERR_INVALID_ARG, "workspace null or not 16-byte aligned");
  const int Z = c->n_layers * c->B;
  const DecodeLayout L = kvtc::decode_layout(Z, c->Hkv, Hq, (int64_t)c->max_pages * c->page_tokens, dev);
  KV_REQUIRE(ws_bytes >= L.total, KV_ERR_INVALID_ARG, "workspace %zu bytes < %zu needed", ws_bytes, L.total);
  return kvtc::launch_decode(p->dev, kvtc::paged_view(*c), q, Z, Hq, seq_lens_dev, q_pos_dev, softmax_scale, out,
                             workspace, L, (cudaStream_t)stream);
}

// ------------------------------------------------------------------------------------------------------
// token-axis allocation
// ------------------------------------------------------------------------------------------------------
extern "C" size_t kv_token_weights_workspace_bytes(int B, int Hkv, int64_t T) {
  if (B < 1 || Hkv < 1 || T < 1) return 0;
  return kvtc::token_layout(B, Hkv, T).total;
}

extern "C" kv_status kv_token_weights(const void* q_obs, int W, const void* k, int B, int Hkv, int Hq, int64_t T,
                                      float softmax_scale, float* weights, void* workspace, size_t ws_bytes,
                                      kv_stream_t stream) {
  clear_error();
  KV_REQUIRE(q_obs && k && weights && workspace, KV_ERR_INVALID_ARG, "null q_obs, k, weights or workspace");
  KV_REQUIRE(aligned16(q_obs) && aligned16(k) && aligned16(workspace), KV_ERR_INVALID_ARG,
             "q_obs, k and workspace must be 16-byte aligned");
  KV_REQUIRE(B >= 1 && Hkv >= 1 && Hq >= Hkv && Hq % Hkv == 0 && W >= 1 && T >= 1, KV_ERR_INVALID_ARG,
             "bad shape B=%d Hkv=%d Hq=%d W=%d T=%lld", B, Hkv, Hq, W, (long long)T);
  KV_REQUIRE((Hq / Hkv) * W <= 128, KV_ERR_UNSUPPORTED, "(Hq / Hkv) * W = %d observation rows > 128", (Hq / Hkv) * W);
  KV_REQUIRE((long long)B * Hkv * T < (1LL << 31) - 128 && (long long)B * Hq * W < (1LL << 31) - 128, KV_ERR_UNSUPPORTED,
             "B * Hkv * T rows exceed the tensor maps' 32-bit coordinates");
  KV_REQUIRE(std::isfinite(softmax_scale), KV_ERR_INVALID_ARG, "non-finite softmax scale");
  const kvtc::TokenLayout L = kvtc::token_layout(B, Hkv, T);
  KV_REQUIRE(ws_bytes >= L.total, KV_ERR_INVALID_ARG, "workspace %zu bytes < %zu needed", ws_bytes, L.total);
  return kvtc::launch_token_weights(q_obs, W, k, B, Hkv, Hq, T, softmax_scale, weights, workspace,
                                    (cudaStream_t)stream);
}

extern "C" kv_status kv_token_select(const float* weights, int B, int Hkv, int64_t T, int64_t keep,
                                     int32_t* keep_idx, kv_stream_t stream) {
  clear_error();
  KV_REQUIRE(weights && keep_idx, KV_ERR_INVALID_ARG, "null weights or keep_idx");
  KV_REQUIRE(B >= 1 && Hkv >= 1 && T >= 1 && T < (1LL << 31) && keep >= 0 && keep <= T, KV_ERR_INVALID_ARG,
             "bad shape B=%d Hkv=%d T=%lld keep=%lld", B, Hkv, (long long)T, (long long)keep);
  if (keep == 0) return KV_OK;
  return kvtc::launch_token_select(weights, B, Hkv, T, keep, keep_idx, (cudaStream_t)stream);
}

extern "C" kv_status kv_cache_compact(const kv_params* p, const kv_cache* src, const kv_cache* dst, int B,
                                      const int32_t* keep_idx, int64_t keep, kv_stream_t stream) {
  clear_error();
  kv_status st;
  if ((st = check_params_on_device(p)) != KV_OK) return st;
  if ((st = check_cache(p, src, B)) != KV_OK) return st;
  if ((st = check_cache(p, dst, B)) != KV_OK) return st;
  KV_REQUIRE(keep_idx, KV_ERR_INVALID_ARG, "null keep_idx");
  KV_REQUIRE(src->Hkv == dst->Hkv, KV_ERR_INVALID_ARG, "source and destination KV heads differ");
  KV_REQUIRE(src->k_rec != dst->k_rec && src->v_rec != dst->v_rec, KV_ERR_INVALID_ARG,
             "compaction needs a destination distinct from its source");
  KV_REQUIRE(keep >= 0 && keep <= dst->T_cap && keep <= src->T_cap, KV_ERR_INVALID_ARG,
             "keep=%lld outside 0..T_cap", (long long)keep);
  if (keep == 0) return KV_OK;
  return kvtc::launch_compact(p->dev, *src, *dst, B, keep_idx, keep, (cudaStream_t)stream);
}

extern "C" kv_status kv_attend_decode_bf16(const void* k, const void* v, int B, int Hkv, int Hq, int64_t T_cap,
                                           const void* q, const int32_t* seq_lens_dev, float softmax_scale,
                                           float* out, void* workspace, size_t ws_bytes, kv_stream_t stream) {
  clear_error();
  KV_REQUIRE(k && v && q && seq_lens_dev && out && workspace, KV_ERR_INVALID_ARG, "null argument");
  KV_REQUIRE(B >= 1 && Hkv >= 1 && T_cap >= 16 && T_cap % 16 == 0, KV_ERR_INVALID_ARG,
             "bad dims B=%d Hkv=%d T_cap=%lld", B, Hkv, (long long)T_cap);
  KV_REQUIRE(Hq >= Hkv && Hq % Hkv == 0, KV_ERR_INVALID_ARG, "Hq=%d not a multiple of Hkv=%d", Hq, Hkv);
  KV_REQUIRE(Hq / Hkv <= MAX_G, KV_ERR_UNSUPPORTED, "g = %d > 8", Hq / Hkv);
  KV_REQUIRE(aligned16(k) && aligned16(v) && aligned16(q) && aligned16(out) && aligned16(workspace),
             KV_ERR_INVALID_ARG, "buffers must be 16-byte aligned");
  const DecodeLayout L = kvtc::decode_bf16_layout(B, Hkv, T_cap, current_device());
  KV_REQUIRE(ws_bytes >= L.total, KV_ERR_INVALID_ARG, "workspace %zu bytes < %zu needed", ws_bytes, L.total);
  return kvtc::launch_decode_bf16(k, v, B, Hkv, Hq, T_cap, q, seq_lens_dev, softmax_scale, out, workspace, L,
                                  (cudaStream_t)stream);
}

extern "C" kv_status kv_check_status(kv_stream_t stream) {
  clear_error();
  cudaError_t e = cudaStreamSynchronize((cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "stream");
  unsigned st = 0;
  kv_status r = kvtc::read_and_clear_device_status(&st);
  if (r != KV_OK) return r;
  if (st & ST_TIMEOUT) {
    kvtc::set_error("a device-side bounded wait ran out");
    return KV_ERR_TIMEOUT;
  }
  if (st & ST_BAD_INDEX) {
    kvtc::set_error("a kernel skipped an out-of-range record write");
    return KV_ERR_DEVICE;
  }
  return KV_OK;
}

extern "C" kv_status kv_debug_quantize_pack(const kv_params* p, int set, int tensor, const float* y_dev, int64_t n,
                                            uint32_t* rec_dev, int variant, kv_stream_t stream) {
  clear_error();
  kv_status st;
  if ((st = check_params_on_device(p)) != KV_OK) return st;
  KV_REQUIRE(set >= 0 && set < p->n_sets && (tensor == 0 || tensor == 1) && n >= 0 && variant >= 0 && variant <= 2,
             KV_ERR_INVALID_ARG, "kv_debug_quantize_pack: bad argument");
  if (n == 0) return KV_OK;
  KV_REQUIRE(y_dev && rec_dev, KV_ERR_INVALID_ARG, "null buffer");
  return kvtc::launch_debug_quantize_pack(p->dev, set, tensor, y_dev, n, rec_dev, variant, (cudaStream_t)stream);
}

extern "C" kv_status kv_debug_unpack(const kv_params* p, int set, int tensor, const uint32_t* rec_dev, int64_t n,
                                     uint16_t* codes_dev, kv_stream_t stream) {
  clear_error();
  kv_status st;
  if ((st = check_params_on_device(p)) != KV_OK) return st;
  KV_REQUIRE(set >= 0 && set < p->n_sets && (tensor == 0 || tensor == 1) && n >= 0, KV_ERR_INVALID_ARG,
             "kv_debug_unpack: bad argument");
  if (n == 0) return KV_OK;
  KV_REQUIRE(rec_dev && codes_dev, KV_ERR_INVALID_ARG, "null buffer");
  return kvtc::launch_debug_unpack(p->dev, set, tensor, rec_dev, n, codes_dev, (cudaStream_t)stream);
}

extern "C" kv_status kv_debug_water_fill(const double* lam, int d, int budget_bits, int max_bits, int32_t* widths) {
  clear_error();
  KV_REQUIRE(lam && widths && d >= 1 && budget_bits >= 0 && max_bits >= 1 && max_bits <= 16, KV_ERR_INVALID_ARG,
             "kv_debug_water_fill: bad argument");
  water_fill(lam, d, budget_bits, max_bits, widths);
  return KV_OK;
}

extern "C" kv_status kv_debug_eigh(const double* sym, int d, double* evals, double* evecs) {
  clear_error();
  KV_REQUIRE(sym && evals && evecs && d >= 1 && d <= 1024, KV_ERR_INVALID_ARG, "kv_debug_eigh: bad argument");
  jacobi_eigh(sym, d, evals, evecs);
  return KV_OK;
}

extern "C" kv_status kv_debug_set_wait_limit_ns(long long ns) {
  KV_REQUIRE(ns > 0, KV_ERR_INVALID_ARG, "wait limit must be positive");
  kvtc::set_wait_limit_ns(ns);
  return KV_OK;
}

extern "C" kv_status kv_debug_decode_plan(const kv_params* p, int B, int Hkv, int Hq, int64_t T_cap,
                                          int32_t* info) {
  clear_error();
  kv_status st;
  int dev = 0;
  if ((st = check_params_on_device(p, &dev)) != KV_OK) return st;
  KV_REQUIRE(info && B >= 1 && Hkv >= 1 && Hq >= Hkv && Hq % Hkv == 0 && Hq / Hkv <= MAX_G && T_cap >= 16 &&
                 T_cap % 16 == 0,
             KV_ERR_INVALID_ARG, "kv_debug_decode_plan: bad argument");
  kv_cache c{};
  c.B = B;
  c.Hkv = Hkv;
  c.T_cap = T_cap;
  const DecodeLayout L = kvtc::decode_layout(B, Hkv, Hq, T_cap, dev);
  return kvtc::launch_decode(p->dev, kvtc::dense_view(c), nullptr, B, Hq, nullptr, nullptr, 1.f, nullptr, nullptr, L,
                             nullptr, info);
}

extern "C" kv_status kv_debug_wait_timeout_selftest(kv_stream_t stream) {
  clear_error();
  return kvtc::launch_wait_selftest((cudaStream_t)stream);
}
