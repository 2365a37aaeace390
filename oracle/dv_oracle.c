/*
 * dv_oracle.c -- plain, slow, single-threaded fp64 CPU oracle for the Deja Vu
 * contextual-sparsity decode step and its composition with attention-scored
 * KV-token selection.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing on the product path may call, link or load
 * this file: only the tests, the smoke check and the benchmark's CPU-baseline
 * leg use it. It shares no code, header, table or constant with the CUDA
 * library; its inputs come from the seeded generators and the pages.
 *
 * Sources (page title, then section / equation):
 *   [DV]  "Deja Vu: Contextual Sparsity for Efficient LLMs at Inference Time"
 *         (arXiv 2310.17157, paper text): §2.3 Eq. 1 (sparsified MLP),
 *         §2.3 Eq. 2 (sparsified MHA), §2.3 budget, §4.1 "Design" (two-layer
 *         predictor), §4.2 "Approach" (head predictor, missing KV), §4.3
 *         (look-ahead), §5.2 / App. C.1 (union sparsity), App. C.3 (residual
 *         form of a layer), App. D (W2 and W^O stored transposed).
 *   [BX]  "Where Activation Sparsity and KV-Cache Sparsity Cross in LLM
 *         Decoding" (arXiv 2609.33889, summary page): §4.1 Setup and App. A
 *         (attention-scored KV selection: 4 sinks, 64-query observation window,
 *         pooled across query heads, width-7 average, top positions per KV
 *         head within the budget, gathered in a contiguous buffer).
 *
 * Conventions: every fp16 input is an IEEE binary16 bit pattern (uint16_t),
 * decoded exactly to double; all arithmetic is double; fp16 outputs are
 * rounded once, to nearest-even. Matrices are row-major. Weight layouts:
 * fc1 [F][d] (row j = neuron j's input weights, (W1)^T), fc2T [F][d]
 * (row j = neuron j's output weights, (W2)^T, App. D), Wq [h*dh][d],
 * Wk/Wv [hkv*dh][d], WoT [h*dh][d] (row j*dh+c = output weights of dim c of
 * head j, (W^O)^T, App. D). KV cache [hkv][n_max][dh].
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------ */
/* IEEE 754 binary16 <-> double                                             */
/* ------------------------------------------------------------------------ */

/* Exact decode: value = (-1)^s * (1024 + m) * 2^(e-25) for 1 <= e <= 30,
 * (-1)^s * m * 2^-24 for e = 0, inf / nan for e = 31. */
double or_h2d(uint16_t h) {
  int s = (h >> 15) & 1, e = (h >> 10) & 0x1f, m = h & 0x3ff;
  double v;
  if (e == 0)
    v = ldexp((double)m, -24);
  else if (e == 31)
    v = m ? NAN : INFINITY;
  else
    v = ldexp((double)(m | 0x400), e - 25);
  return s ? -v : v;
}

/* Round a double to the nearest binary16, ties to even. In the binade
 * [2^E, 2^(E+1)) (E >= -14) representable halves are spaced 2^(E-10); below
 * 2^-14 (subnormals) the spacing is 2^-24. Magnitudes that round to 2^16 or
 * beyond become infinity. */
uint16_t or_d2h(double x) {
  uint16_t sign = signbit(x) ? 0x8000 : 0;
  if (isnan(x)) return (uint16_t)(sign | 0x7e00);
  double a = fabs(x);
  if (isinf(a)) return (uint16_t)(sign | 0x7c00);
  if (a == 0.0) return sign;
  int e2;
  frexp(a, &e2);          /* a in [2^(e2-1), 2^e2) */
  int E = e2 - 1;
  if (E < -14) E = -14;
  double q = ldexp(1.0, E - 10);
  double r = nearbyint(a / q); /* a/q is exact; default mode rounds half to even */
  double v = r * q;
  if (v >= 65536.0) return (uint16_t)(sign | 0x7c00);
  if (v < ldexp(1.0, -14)) return (uint16_t)(sign | (uint16_t)(v / ldexp(1.0, -24)));
  frexp(v, &e2);
  int Ev = e2 - 1;
  int m = (int)(v / ldexp(1.0, Ev - 10)) - 1024;
  return (uint16_t)(sign | ((Ev + 15) << 10) | m);
}

static double H2D_TABLE[65536];
static int h2d_ready = 0;
static void h2d_init(void) {
  if (h2d_ready) return;
  for (int i = 0; i < 65536; ++i) H2D_TABLE[i] = or_h2d((uint16_t)i);
  h2d_ready = 1;
}
#define H(p, i) (H2D_TABLE[(p)[(i)]])
#define HOPT(p, i, dflt) ((p) ? H2D_TABLE[(p)[(i)]] : (dflt))

void or_h2d_array(const uint16_t* in, double* out, int64_t n) {
  h2d_init();
  for (int64_t i = 0; i < n; ++i) out[i] = H(in, i);
}

void or_d2h_array(const double* in, uint16_t* out, int64_t n) {
  for (int64_t i = 0; i < n; ++i) out[i] = or_d2h(in[i]);
}

/* ------------------------------------------------------------------------ */
/* LayerNorm (OPT pre-LN: the block input y is normalised before the       */
/* projections; [DV] App. C.3 writes a layer as y + MHA(y), then + MLP).    */
/* z = (x - mean) / sqrt(var + eps) * g + b, var the biased variance.      */
/* g == NULL means 1, b == NULL means 0.                                    */
/* ------------------------------------------------------------------------ */
void or_layernorm(const uint16_t* x, int d, const uint16_t* g, const uint16_t* b,
                  double eps, double* z) {
  h2d_init();
  double mean = 0.0;
  for (int i = 0; i < d; ++i) mean += H(x, i);
  mean /= d;
  double var = 0.0;
  for (int i = 0; i < d; ++i) {
    double t = H(x, i) - mean;
    var += t * t;
  }
  var /= d;
  double inv = 1.0 / sqrt(var + eps);
  for (int i = 0; i < d; ++i) z[i] = (H(x, i) - mean) * inv * HOPT(g, i, 1.0) + HOPT(b, i, 0.0);
}

/* ------------------------------------------------------------------------ */
/* Sparsity predictor ([DV] §4.1 "Design": a small two-layer fully         */
/* connected network per block; §4.2: the head predictor has the same      */
/* architecture, one class per head). Low-rank form: u = act(P1 y) with    */
/* P1 [r][d], then s = P2 u with P2 [N][r]. act = identity, or ReLU when   */
/* relu != 0. y is the layer input y_l ([DV] §4.3, SP(y_l)).               */
/* ------------------------------------------------------------------------ */
void or_predict(const uint16_t* y, int d, const uint16_t* P1, int r, const uint16_t* P2,
                int N, int relu, double* s) {
  h2d_init();
  double* u = (double*)malloc(sizeof(double) * (size_t)r);
  for (int j = 0; j < r; ++j) {
    double acc = 0.0;
    const uint16_t* row = P1 + (size_t)j * d;
    for (int i = 0; i < d; ++i) acc += H(row, i) * H(y, i);
    u[j] = (relu && acc < 0.0) ? 0.0 : acc;
  }
  for (int n = 0; n < N; ++n) {
    double acc = 0.0;
    const uint16_t* row = P2 + (size_t)n * r;
    for (int j = 0; j < r; ++j) acc += H(row, j) * u[j];
    s[n] = acc;
  }
  free(u);
}

/* ------------------------------------------------------------------------ */
/* Top-k set formation ([DV] §2.3 budget |S| <= (1 - sparsity) * N; §4.1   */
/* the predictor picks the set at a test-time sparsity level). The k       */
/* largest scores; equal scores go to the lower index; -0 equals +0. The   */
/* set is returned in ascending index order. Returns 0, or -1 on bad       */
/* arguments or a NaN score.                                                */
/* ------------------------------------------------------------------------ */
typedef struct {
  double v;
  int32_t i;
} scored_t;

static int cmp_scored_desc(const void* a, const void* b) {
  const scored_t* x = (const scored_t*)a;
  const scored_t* y = (const scored_t*)b;
  if (x->v > y->v) return -1;
  if (x->v < y->v) return 1;
  return (x->i < y->i) ? -1 : (x->i > y->i);
}

static int cmp_i32(const void* a, const void* b) {
  int32_t x = *(const int32_t*)a, y = *(const int32_t*)b;
  return (x > y) - (x < y);
}

int or_topk(const double* s, int N, int k, int32_t* idx) {
  if (N < 1 || k < 1 || k > N) return -1;
  scored_t* t = (scored_t*)malloc(sizeof(scored_t) * (size_t)N);
  for (int i = 0; i < N; ++i) {
    if (isnan(s[i])) {
      free(t);
      return -1;
    }
    t[i].v = (s[i] == 0.0) ? 0.0 : s[i];
    t[i].i = i;
  }
  qsort(t, (size_t)N, sizeof(scored_t), cmp_scored_desc);
  for (int i = 0; i < k; ++i) idx[i] = t[i].i;
  qsort(idx, (size_t)k, sizeof(int32_t), cmp_i32);
  free(t);
  return 0;
}

/* Union of B index sets of width k over [0, N) ([DV] App. C.1: the union of
 * the neurons / heads activated by any input of the batch). Writes the union
 * ascending into out, returns its size. */
int or_union(const int32_t* idx, int B, int k, int N, int32_t* out) {
  uint8_t* mark = (uint8_t*)calloc((size_t)N, 1);
  for (int b = 0; b < B; ++b)
    for (int t = 0; t < k; ++t) mark[idx[(size_t)b * k + t]] = 1;
  int c = 0;
  for (int i = 0; i < N; ++i)
    if (mark[i]) out[c++] = i;
  free(mark);
  return c;
}

/* ------------------------------------------------------------------------ */
/* MLP block ([DV] §2.3 Eq. 1): MLP_S(y) = sigma(y W1_S) (W2_S)^T with the */
/* bias terms of OPT, sigma = ReLU, on z = LN2(x).                         */
/* Two independent forms:                                                   */
/*   gather form: loops only over the neurons j in idx;                    */
/*   masked-dense form: computes every neuron, multiplies its activation   */
/*   by mask[j] (mask == NULL: dense).                                      */
/* delta[d] receives the block output (b2 included, residual excluded).    */
/* act, if not NULL, receives the activation of each visited neuron.       */
/* ------------------------------------------------------------------------ */
void or_mlp_gather(const uint16_t* x, int d, const uint16_t* ln_g, const uint16_t* ln_b,
                   double eps, const uint16_t* fc1, const uint16_t* b1, const uint16_t* fc2T,
                   const uint16_t* b2, const int32_t* idx, int k, double* delta, double* act) {
  h2d_init();
  double* z = (double*)malloc(sizeof(double) * (size_t)d);
  or_layernorm(x, d, ln_g, ln_b, eps, z);
  for (int i = 0; i < d; ++i) delta[i] = HOPT(b2, i, 0.0);
  for (int t = 0; t < k; ++t) {
    int j = idx[t];
    const uint16_t* w1 = fc1 + (size_t)j * d;
    double a = HOPT(b1, j, 0.0);
    for (int i = 0; i < d; ++i) a += z[i] * H(w1, i);
    if (a < 0.0) a = 0.0;
    if (act) act[t] = a;
    const uint16_t* w2 = fc2T + (size_t)j * d;
    for (int i = 0; i < d; ++i) delta[i] += a * H(w2, i);
  }
  free(z);
}

void or_mlp_masked(const uint16_t* x, int d, int F, const uint16_t* ln_g,
                   const uint16_t* ln_b, double eps, const uint16_t* fc1, const uint16_t* b1,
                   const uint16_t* fc2T, const uint16_t* b2, const uint8_t* mask,
                   double* delta, double* act) {
  h2d_init();
  double* z = (double*)malloc(sizeof(double) * (size_t)d);
  or_layernorm(x, d, ln_g, ln_b, eps, z);
  double* a = (double*)malloc(sizeof(double) * (size_t)F);
  for (int j = 0; j < F; ++j) {
    double s = HOPT(b1, j, 0.0);
    for (int i = 0; i < d; ++i) s += z[i] * H(fc1, (size_t)j * d + i);
    a[j] = (s > 0.0 ? s : 0.0) * (mask ? (double)mask[j] : 1.0);
    if (act) act[j] = a[j];
  }
  for (int i = 0; i < d; ++i) {
    double s = HOPT(b2, i, 0.0);
    for (int j = 0; j < F; ++j) s += a[j] * H(fc2T, (size_t)j * d + i);
    delta[i] = s;
  }
  free(a);
  free(z);
}

/* ------------------------------------------------------------------------ */
/* Attention of one query over a list of cached positions plus the new     */
/* token ([DV] §2.3 Eq. 2: H = D^-1 exp(q K^T) V, D = exp(q K^T) 1), with  */
/* the scale applied to the scores. The softmax subtracts the maximum      */
/* score first (same value, no overflow).                                   */
/*   q[dh]; Kbase/Vbase: rows of one KV head [n_max][dh];                   */
/*   pos[0..cnt-1]: cached positions to attend to (NULL: 0..cnt-1);        */
/*   knew/vnew[dh]: the new token's key and value (already fp16-rounded).  */
/* ------------------------------------------------------------------------ */
void or_attend(const double* q, int dh, const uint16_t* Kbase, const uint16_t* Vbase,
               const int32_t* pos, int cnt, const double* knew, const double* vnew,
               double scale, double* Hout) {
  h2d_init();
  int m = cnt + 1;
  double* sc = (double*)malloc(sizeof(double) * (size_t)m);
  for (int t = 0; t < cnt; ++t) {
    int p = pos ? pos[t] : t;
    const uint16_t* kr = Kbase + (size_t)p * dh;
    double s = 0.0;
    for (int c = 0; c < dh; ++c) s += q[c] * H(kr, c);
    sc[t] = s * scale;
  }
  {
    double s = 0.0;
    for (int c = 0; c < dh; ++c) s += q[c] * knew[c];
    sc[cnt] = s * scale;
  }
  double mx = sc[0];
  for (int t = 1; t < m; ++t)
    if (sc[t] > mx) mx = sc[t];
  double D = 0.0;
  for (int t = 0; t < m; ++t) {
    sc[t] = exp(sc[t] - mx);
    D += sc[t];
  }
  for (int c = 0; c < dh; ++c) Hout[c] = 0.0;
  for (int t = 0; t < cnt; ++t) {
    int p = pos ? pos[t] : t;
    const uint16_t* vr = Vbase + (size_t)p * dh;
    for (int c = 0; c < dh; ++c) Hout[c] += sc[t] * H(vr, c);
  }
  for (int c = 0; c < dh; ++c) Hout[c] += sc[cnt] * vnew[c];
  for (int c = 0; c < dh; ++c) Hout[c] /= D;
  free(sc);
}

/* Projection of z onto rows [row0, row0 + dh) of a [*][d] matrix plus bias. */
static void project(const double* z, int d, const uint16_t* W, const uint16_t* bias, int row0,
                    int dh, double* out) {
  for (int c = 0; c < dh; ++c) {
    const uint16_t* w = W + (size_t)(row0 + c) * d;
    double s = HOPT(bias, row0 + c, 0.0);
    for (int i = 0; i < d; ++i) s += z[i] * H(w, i);
    out[c] = s;
  }
}

/* ------------------------------------------------------------------------ */
/* MHA block for one decode token ([DV] §2.3 Eq. 2, MHA_S(y) = sum over    */
/* i in S_A of H_i(y) W^O_i), with OPT biases, z = LN1(x), GQA mapping     */
/* q head j -> KV head j / (h / hkv). The selection unit is a KV head and  */
/* the h/hkv query heads that read it (for MHA, hkv == h: one head).       */
/* The attended keys are positions 0..n-1 of the cache plus the new token, */
/* whose k and v are rounded to fp16 first (the cache holds fp16).         */
/*                                                                          */
/* Gather form: loops over the units in sel[0..ksel-1]. For each selected  */
/* unit it returns the new k, v (fp16 bits) in knew/vnew [hkv][dh]          */
/* (untouched for other units) and the per-query-head outputs in           */
/* Hout [h][dh] (zero for unselected heads).                                */
/* Masked form: computes every head, then multiplies head outputs by       */
/* mask[unit] (mask == NULL: dense) and returns knew/vnew for all units.   */
/* delta[d] = sum of H_j W^O_j + bo (residual excluded).                    */
/* ------------------------------------------------------------------------ */
typedef struct {
  int d, h, hkv, dh, n, n_max;
  double eps, scale;
} or_attn_dims;

static void attn_unit(const or_attn_dims* D, const double* z, const uint16_t* Wq,
                      const uint16_t* bq, const uint16_t* Wk, const uint16_t* bk,
                      const uint16_t* Wv, const uint16_t* bv, const uint16_t* Kc,
                      const uint16_t* Vc, const int32_t* pos, int cnt, int u,
                      uint16_t* knew16, uint16_t* vnew16, double* Hout) {
  int dh = D->dh, G = D->h / D->hkv;
  double* kv = (double*)malloc(sizeof(double) * (size_t)dh * 3);
  double *kd = kv, *vd = kv + dh, *q = kv + 2 * dh;
  project(z, D->d, Wk, bk, u * dh, dh, kd);
  project(z, D->d, Wv, bv, u * dh, dh, vd);
  for (int c = 0; c < dh; ++c) {
    knew16[(size_t)u * dh + c] = or_d2h(kd[c]);
    vnew16[(size_t)u * dh + c] = or_d2h(vd[c]);
    kd[c] = or_h2d(knew16[(size_t)u * dh + c]);
    vd[c] = or_h2d(vnew16[(size_t)u * dh + c]);
  }
  const uint16_t* Kb = Kc + (size_t)u * D->n_max * dh;
  const uint16_t* Vb = Vc + (size_t)u * D->n_max * dh;
  for (int g = 0; g < G; ++g) {
    int j = u * G + g;
    project(z, D->d, Wq, bq, j * dh, dh, q);
    or_attend(q, dh, Kb, Vb, pos, cnt, kd, vd, D->scale, Hout + (size_t)j * dh);
  }
  free(kv);
}

static void attn_out(const or_attn_dims* D, const double* Hout, const uint16_t* WoT,
                     const uint16_t* bo, double* delta) {
  for (int i = 0; i < D->d; ++i) delta[i] = HOPT(bo, i, 0.0);
  for (int j = 0; j < D->h; ++j)
    for (int c = 0; c < D->dh; ++c) {
      double hv = Hout[(size_t)j * D->dh + c];
      if (hv == 0.0) continue;
      const uint16_t* w = WoT + ((size_t)j * D->dh + c) * D->d;
      for (int i = 0; i < D->d; ++i) delta[i] += hv * H(w, i);
    }
}

void or_attn_gather(const or_attn_dims* D, const uint16_t* x, const uint16_t* ln_g,
                    const uint16_t* ln_b, const uint16_t* Wq, const uint16_t* bq,
                    const uint16_t* Wk, const uint16_t* bk, const uint16_t* Wv,
                    const uint16_t* bv, const uint16_t* WoT, const uint16_t* bo,
                    const uint16_t* Kc, const uint16_t* Vc, const int32_t* sel, int ksel,
                    uint16_t* knew16, uint16_t* vnew16, double* Hout, double* delta) {
  h2d_init();
  double* z = (double*)malloc(sizeof(double) * (size_t)D->d);
  or_layernorm(x, D->d, ln_g, ln_b, D->eps, z);
  memset(Hout, 0, sizeof(double) * (size_t)D->h * D->dh);
  for (int t = 0; t < ksel; ++t)
    attn_unit(D, z, Wq, bq, Wk, bk, Wv, bv, Kc, Vc, NULL, D->n, sel[t], knew16, vnew16, Hout);
  attn_out(D, Hout, WoT, bo, delta);
  free(z);
}

void or_attn_masked(const or_attn_dims* D, const uint16_t* x, const uint16_t* ln_g,
                    const uint16_t* ln_b, const uint16_t* Wq, const uint16_t* bq,
                    const uint16_t* Wk, const uint16_t* bk, const uint16_t* Wv,
                    const uint16_t* bv, const uint16_t* WoT, const uint16_t* bo,
                    const uint16_t* Kc, const uint16_t* Vc, const uint8_t* mask,
                    uint16_t* knew16, uint16_t* vnew16, double* Hout, double* delta) {
  h2d_init();
  double* z = (double*)malloc(sizeof(double) * (size_t)D->d);
  or_layernorm(x, D->d, ln_g, ln_b, D->eps, z);
  int G = D->h / D->hkv;
  for (int u = 0; u < D->hkv; ++u)
    attn_unit(D, z, Wq, bq, Wk, bk, Wv, bv, Kc, Vc, NULL, D->n, u, knew16, vnew16, Hout);
  if (mask)
    for (int j = 0; j < D->h; ++j)
      for (int c = 0; c < D->dh; ++c) Hout[(size_t)j * D->dh + c] *= (double)mask[j / G];
  attn_out(D, Hout, WoT, bo, delta);
  free(z);
}

/* Attention over a retained subset of positions: for every KV head u the
 * keys are kept[u][0..cnt[u]-1] (positions into the full cache) plus the new
 * token. Used for the composition with KV selection ([BX] §4.1, App. A: the
 * retained entries are read instead of the whole cache). All heads are
 * computed. Hout [h][dh]; knew16/vnew16 as above; delta = attention output. */
void or_attn_kvsel(const or_attn_dims* D, const uint16_t* x, const uint16_t* ln_g,
                   const uint16_t* ln_b, const uint16_t* Wq, const uint16_t* bq,
                   const uint16_t* Wk, const uint16_t* bk, const uint16_t* Wv,
                   const uint16_t* bv, const uint16_t* WoT, const uint16_t* bo,
                   const uint16_t* Kc, const uint16_t* Vc, const int32_t* kept, int kept_ld,
                   const int32_t* cnt, uint16_t* knew16, uint16_t* vnew16, double* Hout,
                   double* delta) {
  h2d_init();
  double* z = (double*)malloc(sizeof(double) * (size_t)D->d);
  or_layernorm(x, D->d, ln_g, ln_b, D->eps, z);
  for (int u = 0; u < D->hkv; ++u)
    attn_unit(D, z, Wq, bq, Wk, bk, Wv, bv, Kc, Vc, kept + (size_t)u * kept_ld, cnt[u], u,
              knew16, vnew16, Hout);
  attn_out(D, Hout, WoT, bo, delta);
  free(z);
}

/* ------------------------------------------------------------------------ */
/* Attention-scored KV selection ([BX] §4.1 and App. A), step by step.     */
/*                                                                          */
/* 1. or_kv_pool: the last W cached positions are the observation window;  */
/*    obs query t (0 <= t < W) sits at position p_t = n - W + t and        */
/*    attends causally to positions 0..p_t. For every query head j and    */
/*    obs query t the softmax of scale * q_obs[j][t] . K[u][p] over        */
/*    p <= p_t is added to pooled[u][p], u the KV head of j: the pool is    */
/*    the sum over the obs queries and over the query heads of the group.  */
/* 2. or_kv_smooth: centred moving average of width w (odd), zero padding  */
/*    beyond [0, n), divided by w.                                          */
/* 3. or_kv_choose: the sinks {0..n_sinks-1} and the window {n-W..n-1} are */
/*    forced; the remaining budget b - |forced| (b the per-head budget) is */
/*    filled with the highest smoothed scores, equal scores to the lower   */
/*    position. Returns the kept positions ascending.                       */
/* ------------------------------------------------------------------------ */
void or_kv_pool(const uint16_t* q_obs /* [h][W][dh] */, const uint16_t* K /* [hkv][n_max][dh] */,
                int h, int hkv, int dh, int n, int n_max, int W, double scale,
                double* pooled /* [hkv][n] */) {
  h2d_init();
  int G = h / hkv;
  memset(pooled, 0, sizeof(double) * (size_t)hkv * n);
  double* sc = (double*)malloc(sizeof(double) * (size_t)n);
  for (int j = 0; j < h; ++j) {
    int u = j / G;
    const uint16_t* Kb = K + (size_t)u * n_max * dh;
    for (int t = 0; t < W; ++t) {
      int pt = n - W + t;
      const uint16_t* q = q_obs + ((size_t)j * W + t) * dh;
      double mx = -INFINITY;
      for (int p = 0; p <= pt; ++p) {
        double s = 0.0;
        for (int c = 0; c < dh; ++c) s += H(q, c) * H(Kb, (size_t)p * dh + c);
        sc[p] = s * scale;
        if (sc[p] > mx) mx = sc[p];
      }
      double Z = 0.0;
      for (int p = 0; p <= pt; ++p) {
        sc[p] = exp(sc[p] - mx);
        Z += sc[p];
      }
      for (int p = 0; p <= pt; ++p) pooled[(size_t)u * n + p] += sc[p] / Z;
    }
  }
  free(sc);
}

void or_kv_smooth(const double* in, int n, int w, double* out) {
  int half = w / 2;
  for (int p = 0; p < n; ++p) {
    double s = 0.0;
    for (int o = -half; o <= half; ++o) {
      int q = p + o;
      if (q >= 0 && q < n) s += in[q];
    }
    out[p] = s / w;
  }
}

int or_kv_choose(const double* sm, int n, int n_sinks, int W, int b, int32_t* kept) {
  uint8_t* take = (uint8_t*)calloc((size_t)n, 1);
  int forced = 0;
  for (int p = 0; p < n; ++p)
    if (p < n_sinks || p >= n - W) {
      take[p] = 1;
      ++forced;
    }
  int extra = b - forced;
  if (extra > 0) {
    scored_t* t = (scored_t*)malloc(sizeof(scored_t) * (size_t)n);
    int m = 0;
    for (int p = 0; p < n; ++p)
      if (!take[p]) {
        t[m].v = (sm[p] == 0.0) ? 0.0 : sm[p];
        t[m].i = p;
        ++m;
      }
    qsort(t, (size_t)m, sizeof(scored_t), cmp_scored_desc);
    if (extra > m) extra = m;
    for (int i = 0; i < extra; ++i) take[t[i].i] = 1;
    free(t);
  }
  int c = 0;
  for (int p = 0; p < n; ++p)
    if (take[p]) kept[c++] = p;
  free(take);
  return c;
}
