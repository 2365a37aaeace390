// Latency gate: per-request choice between dense decode, the projection
// branch, KV selection and their composition.
//
// "Where Activation Sparsity and KV-Cache Sparsity Cross in LLM Decoding":
// §3.1 (a step reads every projection weight once plus a KV term that grows
// with the context), §3.2 (projection keep saves context-independent bytes,
// KV keep saves context-dependent ones; a step may switch branch), §3.3 (the
// gate adds kernel costs to the byte account; a fixed token budget puts
// r_KV = b/n; a batch reads the union of its sequences' channels), §5.4 and
// App. I (dispatch per request, charging the scoring pass to requests that
// select), App. D (byte-scaled dense time, interpolated log-log across the
// sweep contexts, plus each branch's kernel cost, interpolated linearly;
// equal-latency crossing).
// "Deja Vu: Contextual Sparsity for Efficient LLMs at Inference Time" §2.3
// Eq. 1-2 (the weight rows and cache rows a sparse layer reads), §4.1 (the
// predictor's two low-rank layers), App. C.1 (union over the batch).
//
// Host code only: no CUDA call, callable without a device.
#include <cmath>

#include "../../include/dv.h"

namespace {

constexpr double kElt = 2.0;  // fp16
constexpr int kScan = 8192;   // log-spaced bracketing points of the crossing search

bool is_sparse(int m) { return m == DV_MODE_ACT || m == DV_MODE_COMPOSED; }
bool is_retained(int m) { return m == DV_MODE_KV || m == DV_MODE_COMPOSED; }

int keep_k(float keep, int N) {
  if (keep >= 1.f) return N;
  const double k = std::floor((double)keep * (double)N + 1e-9);
  return k < 1.0 ? 1 : (k > N ? N : (int)k);
}

int check_plan_args(const dv_dims* D, const dv_keep* K, const dv_request* R) {
  if (!D || !K || !R) return DV_ERR_NULL;
  if (D->d < 1 || D->h < 1 || D->h_kv < 1 || D->h % D->h_kv != 0 || D->d_h < 1 || D->F < 1 ||
      D->r < 0)
    return DV_ERR_DIMS;
  for (float k : {K->neuron, K->head, K->kv})
    if (!(k > 0.f && k <= 1.f)) return DV_ERR_KEEP;
  if (R->B < 1 || R->steps < 1 || R->kv_budget < 0) return DV_ERR_DIMS;
  if (R->union_N < 0 || R->union_N > D->F || R->union_H < 0 || R->union_H > D->h_kv)
    return DV_ERR_DIMS;
  return DV_OK;
}

int check_model(const dv_cost_model* C) {
  if (!C) return DV_ERR_NULL;
  if (C->n_ctx < 2 || C->n_ctx > DV_PLAN_MAX_CTX) return DV_ERR_DIMS;
  for (int i = 0; i < C->n_ctx; ++i) {
    if (!std::isfinite(C->ctx[i]) || C->ctx[i] <= 0.0) return DV_ERR_DIMS;
    if (i && !(C->ctx[i] > C->ctx[i - 1])) return DV_ERR_DIMS;
    if (!std::isfinite(C->dense_us[i]) || C->dense_us[i] <= 0.0) return DV_ERR_DIMS;
    if (!std::isfinite(C->select_us[i]) || C->select_us[i] < 0.0) return DV_ERR_DIMS;
    for (int m = 0; m < 4; ++m)
      if (!std::isfinite(C->cost_us[m][i])) return DV_ERR_DIMS;
  }
  return DV_OK;
}

// Units of one kind read by a sparse step: the selected count, or for a batch
// the union (given, else its expectation under independent uniform draws).
double sparse_count(int k, int N, int B, int given) {
  if (B == 1) return k;
  if (given > 0) return given;
  double miss = 1.0;  // P(a unit is outside one sequence's set) ^ B
  for (int b = 0; b < B; ++b) miss *= 1.0 - (double)k / N;
  return N * (1.0 - miss);
}

double bytes_of(int m, const dv_dims* D, const dv_keep* K, const dv_request* R, double n) {
  const double d = D->d, dh = D->d_h, G = D->h / D->h_kv;
  double UN = D->F, UH = D->h_kv, pred = 0.0;
  if (is_sparse(m)) {
    UN = sparse_count(keep_k(K->neuron, D->F), D->F, R->B, R->union_N);
    UH = sparse_count(keep_k(K->head, D->h_kv), D->h_kv, R->B, R->union_H);
    const double scored = (K->neuron < 1.f ? D->F : 0) + (K->head < 1.f ? D->h_kv : 0);
    if (scored > 0) pred = kElt * D->r * (d + scored);  // P1 [r][d] + the scored P2 rows
  }
  double t = n;  // cached keys read per unit per sequence, before the new token
  if (is_retained(m)) t = R->kv_budget > 0 ? std::fmin(n, (double)R->kv_budget) : K->kv * n;
  const double w_attn = UH * (2.0 * G * dh + 2.0 * dh) * d * kElt;  // q, o slices + k, v rows
  const double w_mlp = UN * 2.0 * d * kElt;                         // fc1 row + fc2^T row
  const double kv = R->B * UH * 2.0 * dh * (t + 1.0) * kElt;
  return w_attn + w_mlp + kv + pred;
}

// Piecewise-linear in (log x, log y); the first / last segment continues
// beyond the first / last knot.
double interp_loglog(double x, const double* xs, const double* ys, int n) {
  int i = 0;
  while (i < n - 2 && x > xs[i + 1]) ++i;
  const double lx0 = std::log(xs[i]), lx1 = std::log(xs[i + 1]);
  const double ly0 = std::log(ys[i]), ly1 = std::log(ys[i + 1]);
  const double f = (std::log(x) - lx0) / (lx1 - lx0);
  return std::exp(ly0 + f * (ly1 - ly0));
}

// Piecewise-linear in x; constant beyond the end knots.
double interp_lin(double x, const double* xs, const double* ys, int n) {
  if (x <= xs[0]) return ys[0];
  if (x >= xs[n - 1]) return ys[n - 1];
  int i = 0;
  while (x > xs[i + 1]) ++i;
  const double f = (x - xs[i]) / (xs[i + 1] - xs[i]);
  return ys[i] + f * (ys[i + 1] - ys[i]);
}

double time_of(int m, const dv_dims* D, const dv_keep* K, const dv_request* R,
               const dv_cost_model* C, double n) {
  const int nc = C->n_ctx;
  double t = interp_loglog(n, C->ctx, C->dense_us, nc) * bytes_of(m, D, K, R, n) /
             bytes_of(DV_MODE_DENSE, D, K, R, n);
  t += interp_lin(n, C->ctx, C->cost_us[m], nc);
  if (is_retained(m)) t += interp_lin(n, C->ctx, C->select_us, nc) / R->steps;
  return t;
}

}  // namespace

extern "C" {

int dv_plan_bytes(const dv_dims* dims, const dv_keep* keep, const dv_request* req, double n,
                  double bytes[4]) {
  int rc = check_plan_args(dims, keep, req);
  if (rc != DV_OK) return rc;
  if (!bytes) return DV_ERR_NULL;
  if (!std::isfinite(n) || n < 0.0) return DV_ERR_DIMS;
  for (int m = 0; m < 4; ++m) bytes[m] = bytes_of(m, dims, keep, req, n);
  return DV_OK;
}

int dv_cost_calibrate(const dv_dims* dims, const dv_keep* keep, const dv_request* req, int n_ctx,
                      const double* ctx, const double* measured_us, const double* select_us,
                      dv_cost_model* out) {
  int rc = check_plan_args(dims, keep, req);
  if (rc != DV_OK) return rc;
  if (!ctx || !measured_us || !out) return DV_ERR_NULL;
  if (n_ctx < 2 || n_ctx > DV_PLAN_MAX_CTX) return DV_ERR_DIMS;
  dv_cost_model C = {};
  C.n_ctx = n_ctx;
  for (int i = 0; i < n_ctx; ++i) {
    C.ctx[i] = ctx[i];
    C.dense_us[i] = measured_us[i];
    C.select_us[i] = select_us ? select_us[i] : 0.0;
    const double dense_bytes = bytes_of(DV_MODE_DENSE, dims, keep, req, ctx[i]);
    for (int m = 0; m < 4; ++m) {
      const double t = measured_us[(size_t)m * n_ctx + i];
      if (!std::isfinite(t)) return DV_ERR_DIMS;
      C.cost_us[m][i] =
          m == DV_MODE_DENSE ? 0.0
                             : t - C.dense_us[i] * bytes_of(m, dims, keep, req, ctx[i]) / dense_bytes;
    }
  }
  if ((rc = check_model(&C)) != DV_OK) return rc;
  *out = C;
  return DV_OK;
}

int dv_plan_decode(const dv_dims* dims, const dv_keep* keep, const dv_request* req,
                   const dv_cost_model* cm, double n, dv_plan* out) {
  int rc = check_plan_args(dims, keep, req);
  if (rc != DV_OK) return rc;
  if ((rc = check_model(cm)) != DV_OK) return rc;
  if (!out) return DV_ERR_NULL;
  if (!std::isfinite(n) || n <= 0.0) return DV_ERR_DIMS;
  unsigned admit = req->modes ? req->modes : 0xFu;
  if (req->B > 1) admit &= (1u << DV_MODE_DENSE) | (1u << DV_MODE_ACT);
  dv_plan P = {};
  P.choice = -1;
  for (int m = 0; m < 4; ++m) {
    P.bytes[m] = bytes_of(m, dims, keep, req, n);
    P.us[m] = time_of(m, dims, keep, req, cm, n);
    if ((admit >> m & 1u) && (P.choice < 0 || P.us[m] < P.us[P.choice])) P.choice = m;
  }
  *out = P;
  return P.choice < 0 ? DV_ERR_UNSUPPORTED : DV_OK;
}

int dv_plan_crossing(const dv_dims* dims, const dv_keep* keep, const dv_request* req,
                     const dv_cost_model* cm, int mode_a, int mode_b, double n_lo, double n_hi,
                     double* n_star) {
  int rc = check_plan_args(dims, keep, req);
  if (rc != DV_OK) return rc;
  if ((rc = check_model(cm)) != DV_OK) return rc;
  if (!n_star) return DV_ERR_NULL;
  if (mode_a < 0 || mode_a > 3 || mode_b < 0 || mode_b > 3 || mode_a == mode_b) return DV_ERR_DIMS;
  if (!std::isfinite(n_lo) || !std::isfinite(n_hi) || !(n_lo > 0.0) || !(n_hi > n_lo))
    return DV_ERR_DIMS;
  auto diff = [&](double x) {
    return time_of(mode_a, dims, keep, req, cm, x) - time_of(mode_b, dims, keep, req, cm, x);
  };
  *n_star = -1.0;
  const double l0 = std::log(n_lo), step = (std::log(n_hi) - l0) / (kScan - 1);
  double xa = n_lo, fa = diff(xa);
  if (fa == 0.0) {
    *n_star = xa;
    return DV_OK;
  }
  for (int i = 1; i < kScan; ++i) {
    const double xb = i == kScan - 1 ? n_hi : std::exp(l0 + step * i);
    const double fb = diff(xb);
    if (fb == 0.0) {
      *n_star = xb;
      return DV_OK;
    }
    if ((fa < 0.0) != (fb < 0.0)) {
      double lo = xa, hi = xb, flo = fa;
      for (int it = 0; it < 200 && hi - lo > 1e-12 * hi; ++it) {
        const double mid = 0.5 * (lo + hi), fm = diff(mid);
        if (fm == 0.0) {
          lo = hi = mid;
          break;
        }
        if ((fm < 0.0) == (flo < 0.0)) {
          lo = mid;
          flo = fm;
        } else {
          hi = mid;
        }
      }
      *n_star = 0.5 * (lo + hi);
      return DV_OK;
    }
    xa = xb;
    fa = fb;
  }
  return DV_OK;
}

}  // extern "C"
