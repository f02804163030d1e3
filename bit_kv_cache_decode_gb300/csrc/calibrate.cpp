// Offline calibration of OSCAR's rotations and clip thresholds on the host
// (MarkTechPost article "Together AI 开源 OSCAR…", section "OSCAR 有何不同做法":
// C_Q = (1/N) sum q^T q, C_S = (1/N) V^T S^T S V, U_Q / U_S their eigenvectors,
// R = U H_Had P_br; section "服务系统：混合精度缓存布局" and visual-guide step 4:
// percentile clip thresholds c_K = 0.96, c_V = 0.92).
//
// Eigenvectors come from the cyclic Jacobi method in double precision: plane
// rotations chosen to zero one off-diagonal entry at a time, swept over all
// pairs until the off-diagonal mass is negligible.
#include <algorithm>
#include <cmath>
#include <cstdint>
#include <vector>

#include "../../include/oscar.h"

namespace {

constexpr int D = 128;

// Symmetric eigen-decomposition: a (n x n, row-major, destroyed) -> eigenvalues w
// (descending) and eigenvector columns u (row-major n x n), each column's
// largest-magnitude entry positive.
void jacobi_eigen(std::vector<double>& a, int n, std::vector<double>& w, std::vector<double>& u) {
  std::vector<double> v((size_t)n * n, 0.0);
  for (int i = 0; i < n; ++i) v[(size_t)i * n + i] = 1.0;
  double total = 0.0;
  for (double x : a) total += x * x;
  for (int sweep = 0; sweep < 100; ++sweep) {
    double off = 0.0;
    for (int p = 0; p < n; ++p)
      for (int q = p + 1; q < n; ++q) off += a[(size_t)p * n + q] * a[(size_t)p * n + q];
    if (off <= 1e-30 * total) break;
    for (int p = 0; p < n - 1; ++p) {
      for (int q = p + 1; q < n; ++q) {
        const double apq = a[(size_t)p * n + q];
        if (std::fabs(apq) <= 1e-300) continue;
        const double theta = (a[(size_t)q * n + q] - a[(size_t)p * n + p]) / (2.0 * apq);
        const double t = (theta >= 0 ? 1.0 : -1.0) / (std::fabs(theta) + std::sqrt(theta * theta + 1.0));
        const double c = 1.0 / std::sqrt(t * t + 1.0), s = t * c;
        for (int k = 0; k < n; ++k) {             // columns p, q: A <- A J
          const double akp = a[(size_t)k * n + p], akq = a[(size_t)k * n + q];
          a[(size_t)k * n + p] = c * akp - s * akq;
          a[(size_t)k * n + q] = s * akp + c * akq;
        }
        for (int k = 0; k < n; ++k) {             // rows p, q: A <- J^T A
          const double apk = a[(size_t)p * n + k], aqk = a[(size_t)q * n + k];
          a[(size_t)p * n + k] = c * apk - s * aqk;
          a[(size_t)q * n + k] = s * apk + c * aqk;
        }
        for (int k = 0; k < n; ++k) {             // V <- V J
          const double vkp = v[(size_t)k * n + p], vkq = v[(size_t)k * n + q];
          v[(size_t)k * n + p] = c * vkp - s * vkq;
          v[(size_t)k * n + q] = s * vkp + c * vkq;
        }
      }
    }
  }
  std::vector<int> order(n);
  for (int i = 0; i < n; ++i) order[i] = i;
  std::stable_sort(order.begin(), order.end(),
                   [&](int x, int y) { return a[(size_t)x * n + x] > a[(size_t)y * n + y]; });
  w.assign(n, 0.0);
  u.assign((size_t)n * n, 0.0);
  for (int j = 0; j < n; ++j) {
    const int src = order[j];
    w[j] = a[(size_t)src * n + src];
    int imax = 0;
    for (int i = 1; i < n; ++i)
      if (std::fabs(v[(size_t)i * n + src]) > std::fabs(v[(size_t)imax * n + src])) imax = i;
    const double sgn = v[(size_t)imax * n + src] < 0 ? -1.0 : 1.0;
    for (int i = 0; i < n; ++i) u[(size_t)i * n + j] = sgn * v[(size_t)i * n + src];
  }
}

// x R for R = U H P_br (row vector x, U row-major with eigenvector columns).
void rotate_row(const double* x, const std::vector<double>& u, double* out) {
  double z[D];
  for (int j = 0; j < D; ++j) {
    double s = 0.0;
    for (int i = 0; i < D; ++i) s += x[i] * u[(size_t)i * D + j];
    z[j] = s;
  }
  for (int len = 1; len < D; len <<= 1)           // Walsh-Hadamard butterflies
    for (int i = 0; i < D; ++i)
      if ((i & len) == 0) {
        const double a = z[i], b = z[i + len];
        z[i] = a + b;
        z[i + len] = a - b;
      }
  const double inv = 1.0 / std::sqrt((double)D);
  for (int j = 0; j < D; ++j) {
    int r = 0;                                    // 7-bit reversal of j
    for (int bit = 0; bit < 7; ++bit)
      if (j & (1 << bit)) r |= 1 << (6 - bit);
    out[j] = z[r] * inv;                          // (w P_br)[j] = w[bitrev(j)]
  }
}

// Per-channel c-quantile of |X R| with linear interpolation between order statistics.
void thresholds(const float* x, int n, const std::vector<double>& u, double c, float* tau) {
  std::vector<double> col((size_t)D * n);
  std::vector<double> row(D), rot(D);
  for (int t = 0; t < n; ++t) {
    for (int i = 0; i < D; ++i) row[i] = x[(size_t)t * D + i];
    rotate_row(row.data(), u, rot.data());
    for (int j = 0; j < D; ++j) col[(size_t)j * n + t] = std::fabs(rot[j]);
  }
  for (int j = 0; j < D; ++j) {
    double* a = col.data() + (size_t)j * n;
    std::sort(a, a + n);
    const double pos = (n - 1) * c;
    const int lo = (int)std::floor(pos);
    const int hi = std::min(lo + 1, n - 1);
    tau[j] = (float)(a[lo] + (pos - lo) * (a[hi] - a[lo]));
  }
}

}  // namespace

extern "C" int oscar_calibrate(const float* Q, const float* K, const float* V, int N, float sm_scale, float c_K,
                               float c_V, float* U_K, float* U_V, float* tau_K, float* tau_V, double* eig_K,
                               double* eig_V) {
  if (!Q || !K || !V || N < 2 || !U_K || !U_V || !tau_K || !tau_V) return OSCAR_ERR_INVALID_ARG;
  if (!(c_K >= 0.f && c_K <= 1.f && c_V >= 0.f && c_V <= 1.f) || !(sm_scale > 0.f)) return OSCAR_ERR_INVALID_ARG;
  // C_Q = (1/N) Q^T Q
  std::vector<double> cq((size_t)D * D, 0.0);
  for (int t = 0; t < N; ++t) {
    const float* q = Q + (size_t)t * D;
    for (int i = 0; i < D; ++i) {
      const double qi = q[i];
      double* r = cq.data() + (size_t)i * D;
      for (int j = 0; j < D; ++j) r[j] += qi * q[j];
    }
  }
  for (double& x : cq) x /= N;
  // C_S = (1/N) (S V)^T (S V), S = row softmax of sm_scale Q K^T
  std::vector<double> cs((size_t)D * D, 0.0), logits(N), sv(D);
  for (int t = 0; t < N; ++t) {
    const float* q = Q + (size_t)t * D;
    double m = -INFINITY;
    for (int s = 0; s < N; ++s) {
      const float* k = K + (size_t)s * D;
      double dot = 0.0;
      for (int i = 0; i < D; ++i) dot += (double)q[i] * k[i];
      logits[s] = sm_scale * dot;
      m = std::max(m, logits[s]);
    }
    double z = 0.0;
    for (int s = 0; s < N; ++s) { logits[s] = std::exp(logits[s] - m); z += logits[s]; }
    std::fill(sv.begin(), sv.end(), 0.0);
    for (int s = 0; s < N; ++s) {
      const double p = logits[s] / z;
      const float* vr = V + (size_t)s * D;
      for (int i = 0; i < D; ++i) sv[i] += p * vr[i];
    }
    for (int i = 0; i < D; ++i) {
      double* r = cs.data() + (size_t)i * D;
      for (int j = 0; j < D; ++j) r[j] += sv[i] * sv[j];
    }
  }
  for (double& x : cs) x /= N;
  std::vector<double> wk, uk, wv, uv;
  jacobi_eigen(cq, D, wk, uk);
  jacobi_eigen(cs, D, wv, uv);
  for (size_t i = 0; i < (size_t)D * D; ++i) {
    U_K[i] = (float)uk[i];
    U_V[i] = (float)uv[i];
  }
  if (eig_K) std::copy(wk.begin(), wk.end(), eig_K);
  if (eig_V) std::copy(wv.begin(), wv.end(), eig_V);
  thresholds(K, N, uk, c_K, tau_K);
  thresholds(V, N, uv, c_V, tau_V);
  return OSCAR_OK;
}

// Lloyd-Max codebook of one (layer, kv head, kind) (news article "超越 TurboQuant…", section "总结与展望":
// a Lloyd-Max codebook inside the attention-aware rotation). Lloyd's iteration on the pooled normalised
// group values u = (y - min) / (max - min) of the clipped calibration rows; cell i holds the u in
// (t_{i-1}, t_i], t the midpoints between neighbouring levels, and each level moves to its cell's mean.
extern "C" int oscar_calibrate_codebook(const float* x_rot, int N, const float* tau, uint8_t* cb) {
  if (!x_rot || !tau || !cb || N < 1) return OSCAR_ERR_INVALID_ARG;
  constexpr int G = 64;
  std::vector<double> u;
  u.reserve((size_t)N * D);
  float y[G];
  for (int n = 0; n < N; ++n)
    for (int g = 0; g < D / G; ++g) {
      float mn = INFINITY, mx = -INFINITY;
      for (int j = 0; j < G; ++j) {
        const float t = tau[g * G + j];
        y[j] = std::min(std::max(x_rot[(size_t)n * D + g * G + j], -t), t);
        mn = std::min(mn, y[j]);
        mx = std::max(mx, y[j]);
      }
      if (!(mx > mn)) continue;
      const double range = (double)mx - (double)mn;
      for (int j = 0; j < G; ++j) u.push_back(((double)y[j] - (double)mn) / range);
    }
  std::sort(u.begin(), u.end());
  std::vector<double> csum(u.size() + 1, 0.0);
  for (size_t i = 0; i < u.size(); ++i) csum[i + 1] = csum[i] + u[i];
  double c[4] = {0.0, 1.0 / 3.0, 2.0 / 3.0, 1.0};
  for (int it = 0; it < 1000; ++it) {
    size_t edge[5];
    edge[0] = 0;
    edge[4] = u.size();
    for (int i = 0; i < 3; ++i)
      edge[i + 1] = (size_t)(std::upper_bound(u.begin(), u.end(), 0.5 * (c[i] + c[i + 1])) - u.begin());
    double nc[4], moved = 0.0;
    for (int i = 0; i < 4; ++i) {
      nc[i] = edge[i + 1] > edge[i] ? (csum[edge[i + 1]] - csum[edge[i]]) / (double)(edge[i + 1] - edge[i]) : c[i];
      moved = std::max(moved, std::fabs(nc[i] - c[i]));
    }
    std::copy(nc, nc + 4, c);
    if (moved <= 1e-12) break;
  }
  int k[4];
  for (int i = 0; i < 4; ++i) k[i] = (int)std::min(std::max(std::rint(255.0 * c[i]), 0.0), 255.0);
  std::sort(k, k + 4);
  for (int i = 0; i < 4; ++i) cb[i] = (uint8_t)k[i];
  return OSCAR_OK;
}
