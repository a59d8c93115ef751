// Host-side construction of the handle's tables, in fp64.
//
// * R: a Haar-random orthogonal matrix (intelliparadigm.com, "TurboQuant技术",
//   §2.1.1 step 1; 甲子光年 article §2 第一階段 "隨機旋轉"), taken as the Q
//   factor of a seeded d x d standard Gaussian matrix G = Q T with the signs
//   fixed so that diag(T) > 0 (Mezzadri 2007).  Householder QR written here.
// * S: m x d standard Gaussian (QJL projection, intelliparadigm.com §2.1.2).
//   S' = S R^T lets the kernels project the residual in the rotated space.
// * Codebooks: the Lloyd-Max quantizer for one coordinate of a random unit
//   vector, whose law is Beta (甲子光年 §2 第一階段 "Beta分布"): density
//   f_d(x) = C_d (1 - x^2)^((d-3)/2) on [-1, 1].  Cell masses by composite
//   Gauss-Legendre quadrature over the cell; cell first moments by the closed
//   form  int x (1-x^2)^a dx = -(1-x^2)^(a+1) / (2(a+1)).
// * Random numbers: SplitMix64 (Steele, Lea & Flood 2014, finaliser constants
//   of Vigna's splitmix64.c); uniforms ((z >> 11) + 1) * 2^-53; normals by
//   Box-Muller in pairs (cos, then sin); one stream: G row-major, then S.
#include <algorithm>
#include <cmath>
#include <vector>

#include "tq_internal.h"

namespace tq {
namespace {

class SplitMix64 {
 public:
  explicit SplitMix64(uint64_t seed) : state_(seed) {}
  uint64_t next() {
    state_ += 0x9E3779B97F4A7C15ull;
    uint64_t z = state_;
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
  }
  double uniform() { return static_cast<double>((next() >> 11) + 1) * 0x1.0p-53; }

 private:
  uint64_t state_;
};

std::vector<double> normal_stream(uint64_t seed, size_t count) {
  SplitMix64 gen(seed);
  std::vector<double> out;
  out.reserve(count + 1);
  while (out.size() < count) {
    double u1 = gen.uniform();
    double u2 = gen.uniform();
    double radius = std::sqrt(-2.0 * std::log(u1));
    double angle = 2.0 * M_PI * u2;
    out.push_back(radius * std::cos(angle));
    out.push_back(radius * std::sin(angle));
  }
  out.resize(count);
  return out;
}

// Q of A = Q T (A: n x n row-major) with diag(T) made positive.
std::vector<double> haar_q(std::vector<double> a, int n) {
  std::vector<std::vector<double>> reflectors;
  std::vector<double> diag(n);
  for (int k = 0; k < n; ++k) {
    double norm2 = 0.0;
    for (int i = k; i < n; ++i) norm2 += a[i * n + k] * a[i * n + k];
    double norm = std::sqrt(norm2);
    double alpha = a[k * n + k] > 0.0 ? -norm : norm;
    std::vector<double> v(n - k);
    for (int i = k; i < n; ++i) v[i - k] = a[i * n + k];
    v[0] -= alpha;
    double vv = 0.0;
    for (double x : v) vv += x * x;
    if (vv > 0.0) {
      for (int j = k; j < n; ++j) {
        double s = 0.0;
        for (int i = k; i < n; ++i) s += v[i - k] * a[i * n + j];
        s *= 2.0 / vv;
        for (int i = k; i < n; ++i) a[i * n + j] -= s * v[i - k];
      }
      double inv = 1.0 / std::sqrt(vv);
      for (double& x : v) x *= inv;
    } else {
      std::fill(v.begin(), v.end(), 0.0);
    }
    diag[k] = a[k * n + k];
    reflectors.push_back(std::move(v));
  }
  // Q = H_0 H_1 ... H_{n-1}: apply the reflectors to the identity from the right end.
  std::vector<double> q(static_cast<size_t>(n) * n, 0.0);
  for (int i = 0; i < n; ++i) q[i * n + i] = 1.0;
  for (int k = n - 1; k >= 0; --k) {
    const std::vector<double>& v = reflectors[k];
    for (int j = 0; j < n; ++j) {
      double s = 0.0;
      for (int i = k; i < n; ++i) s += v[i - k] * q[i * n + j];
      s *= 2.0;
      for (int i = k; i < n; ++i) q[i * n + j] -= s * v[i - k];
    }
  }
  for (int j = 0; j < n; ++j) {
    if (diag[j] < 0.0) {
      for (int i = 0; i < n; ++i) q[i * n + j] = -q[i * n + j];
    }
  }
  return q;
}

// Gauss-Legendre nodes/weights on [-1, 1] by Newton's method on P_n.
void gauss_legendre(int n, std::vector<double>* x, std::vector<double>* w) {
  x->assign(n, 0.0);
  w->assign(n, 0.0);
  for (int i = 0; i < n; ++i) {
    double z = std::cos(M_PI * (i + 0.75) / (n + 0.5));
    double dp = 1.0;
    for (int it = 0; it < 100; ++it) {
      double p0 = 1.0, p1 = z;
      for (int k = 2; k <= n; ++k) {
        double p2 = ((2.0 * k - 1.0) * z * p1 - (k - 1.0) * p0) / k;
        p0 = p1;
        p1 = p2;
      }
      dp = n * (z * p1 - p0) / (z * z - 1.0);
      double dz = p1 / dp;
      z -= dz;
      if (std::fabs(dz) < 1e-17) break;
    }
    (*x)[i] = z;
    (*w)[i] = 2.0 / ((1.0 - z * z) * dp * dp);
  }
}

class BetaCoordinateLaw {
 public:
  explicit BetaCoordinateLaw(int d) : d_(d), a_((d - 3) / 2.0) {
    c_ = std::exp(std::lgamma(d / 2.0) - std::lgamma((d - 1) / 2.0)) / std::sqrt(M_PI);
    gauss_legendre(12, &gx_, &gw_);
    panel_ = std::min(0.01, 0.1 / std::sqrt(static_cast<double>(d)));
  }
  double pdf(double x) const {
    double t = 1.0 - x * x;
    return t > 0.0 ? c_ * std::pow(t, a_) : 0.0;
  }
  // P(lo < X <= hi) by composite Gauss-Legendre over the cell itself.
  double mass(double lo, double hi) const {
    int panels = std::max(1, static_cast<int>(std::ceil((hi - lo) / panel_)));
    double h = (hi - lo) / panels;
    double total = 0.0;
    for (int p = 0; p < panels; ++p) {
      double mid = lo + (p + 0.5) * h;
      double acc = 0.0;
      for (size_t i = 0; i < gx_.size(); ++i) acc += gw_[i] * pdf(mid + 0.5 * h * gx_[i]);
      total += 0.5 * h * acc;
    }
    return total;
  }
  // int_{-1}^{x} u f(u) du.
  double first_moment_to(double x) const {
    double a1 = a_ + 1.0;
    double t = std::max(0.0, 1.0 - x * x);
    return -c_ * std::pow(t, a1) / (2.0 * a1);
  }

 private:
  int d_;
  double a_;
  double c_;
  double panel_;
  std::vector<double> gx_, gw_;
};

double standard_normal_quantile(double p) {
  double lo = -40.0, hi = 40.0;
  for (int it = 0; it < 200; ++it) {
    double mid = 0.5 * (lo + hi);
    if (0.5 * std::erfc(-mid / std::sqrt(2.0)) < p) lo = mid; else hi = mid;
  }
  return 0.5 * (lo + hi);
}

// Lloyd-Max: boundaries at level midpoints, levels at cell centroids; start
// from normal quantile midpoints scaled by 1/sqrt(d); stop when no level moves
// by more than 1e-13 in the sqrt(d)-scaled coordinate.
void lloyd_max(int d, int bits, std::vector<double>* levels, std::vector<double>* bounds) {
  const int count = 1 << bits;
  const double scale = std::sqrt(static_cast<double>(d));
  BetaCoordinateLaw law(d);
  std::vector<double> c(count), t(count - 1), edges(count + 1);
  for (int i = 0; i < count; ++i) c[i] = standard_normal_quantile((i + 0.5) / count) / scale;
  for (int it = 0; it < 100000; ++it) {
    for (int i = 0; i + 1 < count; ++i) t[i] = 0.5 * (c[i] + c[i + 1]);
    edges[0] = -1.0;
    edges[count] = 1.0;
    for (int i = 0; i + 1 < count; ++i) edges[i + 1] = t[i];
    double moved = 0.0;
    for (int i = 0; i < count; ++i) {
      double num = law.first_moment_to(edges[i + 1]) - law.first_moment_to(edges[i]);
      double next = num / law.mass(edges[i], edges[i + 1]);
      moved = std::max(moved, std::fabs(next - c[i]) * scale);
      c[i] = next;
    }
    if (moved < 1e-13) break;
  }
  // The coordinate law is even, so the exact codebook is odd-symmetric with a
  // middle boundary of exactly 0 (a coordinate at 0 then takes the lower level
  // by the tie rule); the iteration's rounding leaves a ~1e-16 residue there.
  std::vector<double> sym(count);
  for (int i = 0; i < count; ++i) sym[i] = 0.5 * (c[i] - c[count - 1 - i]);
  c = sym;
  for (int i = 0; i + 1 < count; ++i) t[i] = 0.5 * (c[i] + c[i + 1]);
  *levels = c;
  *bounds = t;
}

}  // namespace

void build_host_tables(int d, int qjl_m, uint64_t seed, int k_mse_bits, int v_bits, HostTables* out) {
  std::vector<double> normals = normal_stream(seed, static_cast<size_t>(d) * d + static_cast<size_t>(qjl_m) * d);
  std::vector<double> g(normals.begin(), normals.begin() + static_cast<size_t>(d) * d);
  out->R = haar_q(g, d);
  out->S.assign(normals.begin() + static_cast<size_t>(d) * d, normals.end());
  out->Sp.assign(static_cast<size_t>(qjl_m) * d, 0.0);
  for (int k = 0; k < qjl_m; ++k) {
    for (int j = 0; j < d; ++j) {
      double s = 0.0;
      for (int i = 0; i < d; ++i) s += out->S[k * d + i] * out->R[j * d + i];
      out->Sp[k * d + j] = s;
    }
  }
  lloyd_max(d, k_mse_bits, &out->k_levels, &out->k_bounds);
  lloyd_max(d, v_bits, &out->v_levels, &out->v_bounds);
}

}  // namespace tq
