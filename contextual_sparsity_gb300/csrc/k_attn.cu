// k_attn.cu -- attention over the KV cache (sm_103a).
//
// Split-K flash-decoding ("Where Activation Sparsity and KV-Cache Sparsity
// Cross in LLM Decoding", §4.1: dense and sparse modes read the cache through
// the same split-K kernel): the keys of each selected unit are cut into
// splits, every CTA keeps an online softmax (running max m, sum l and
// unnormalised output o, base-2 exponent) over its split, and a separate
// combine merges the splits: H = sum_s 2^(m_s-M) o_s / sum_s 2^(m_s-M) l_s
// ("Deja Vu", §2.3 Eq. 2: H = D^-1 exp(q K^T) V). A unit is one KV head and
// its G = h/h_kv query heads, so a K/V row is read once for all of them.
//
// Attention-scored KV selection ("Where ...", §4.1, App. A): causal softmax of
// the observation-window queries over the cache, pooled over the window and
// the query heads of each KV head, smoothed by a centred mean, sinks and the
// window forced, top positions per KV head, gathered into a contiguous buffer.
#include <cooperative_groups.h>

#include "dv_internal.h"

namespace dv {

namespace cg = cooperative_groups;

constexpr float kLog2e = 1.4426950408889634f;

// ---------------------------------------------------------------------------
// Split-K flash-decode
// ---------------------------------------------------------------------------
struct SplitParams {
  const float* q;  // [B][k][G][DH], already scaled by softmax_scale
  const uint16_t *K, *V;
  const uint16_t *Kr, *Vr;
  const int32_t* kept_count;
  const int32_t* idx;
  const int32_t* dev_count;
  int k, h_kv, n, n_max, b_max, retained, C, S;
  float* part;  // [B][k][G][S][DH + 2]
  float* H;     // [B][k][G][DH] combined head outputs
  int* cnt;     // [B][k] splits finished per unit (zero between launches)
  int* st;
};

// Online-softmax merge of (m2, l2, o2) into (m, l, o) (base 2).
template <int N>
DV_DEV void merge(float& m, float& l, float* o, float m2, float l2, const float* o2) {
  const float M = fmaxf(m, m2);
  if (M == -INFINITY) return;
  const float w1 = (m == -INFINITY) ? 0.f : exp2f(m - M);
  const float w2 = (m2 == -INFINITY) ? 0.f : exp2f(m2 - M);
  l = l * w1 + l2 * w2;
#pragma unroll
  for (int i = 0; i < N; ++i) o[i] = o[i] * w1 + o2[i] * w2;
  m = M;
}

// Each CTA owns a contiguous range of keys of one unit and walks it in chunks
// of kChunk keys: a chunk's K and V rows (contiguous in the cache or in the
// retained buffer) arrive by two 1-D bulk copies into one of NST shared-memory
// stages, so up to NST chunks are in flight at once. Two stages (64 KB at
// d_h 128) leave room on the SM for the side-stream kernels; three serve long
// ranges, where the bytes in flight set the pace.
//
// The splits of a unit are combined either through global memory (their
// partials written, an atomic count, the last split to finish combines:
// any number of splits) or, when they are at most kClusterSplits, as one
// thread-block cluster: each split leaves its partial in shared memory and
// rank 0 reads the others through distributed shared memory (no global
// partials, no fence, no atomic).
constexpr int kChunk = 64;
constexpr int kClusterSplits = 8;
constexpr int kLongRangeChunks = 4;  // more chunks per CTA than this: three stages

template <int DH, int G, bool CL, int NST>
__global__ void __launch_bounds__(128) k_splitk(const SplitParams p) {
  constexpr int LPK = DH / 8;            // lanes per key (8 dims each)
  constexpr int KPW = 32 / LPK;          // keys per warp step
  constexpr int U = kChunk / (4 * KPW);  // warp steps per chunk
  __shared__ float red[4][G][DH + 2];
  __shared__ float cpart[G][DH + 2];     // cluster combine: this split's (m, l, o)
  __shared__ __align__(8) uint64_t kv_bar[NST];
  __shared__ float cw[G][kSplitsMax];    // global combine: weight of each split
  __shared__ float cinv[G];              // global combine: 1 / sum of weighted l
  __shared__ int last;
  extern __shared__ __align__(128) uint16_t kv_smem[];  // [NST][K, V][kChunk][DH]

  const int s = blockIdx.x, e = blockIdx.y, b = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int sub = lane % LPK, grp = lane / LPK;
  pdl_wait();  // q and the new key/value come from the previous kernel
  if (threadIdx.x == 0) pdl_launch_dependents();

  int kk = p.k;
  if (p.dev_count) kk = min(kk, *p.dev_count);
  if (e >= kk) return;  // uniform over a unit's splits (one cluster)
  int u = p.idx ? p.idx[e] : e;
  if (u < 0 || u >= p.h_kv) {
    if (threadIdx.x == 0) flag(p.st, DV_DEV_BAD_INDEX);
    u = 0;
  }

  const uint16_t *Kb, *Vb;
  int count;
  if (p.retained) {
    Kb = p.Kr + (size_t)u * p.b_max * DH;
    Vb = p.Vr + (size_t)u * p.b_max * DH;
    count = min(p.kept_count[u] + 1, p.b_max);
  } else {
    Kb = p.K + (((size_t)b * p.h_kv + u) * p.n_max) * DH;
    Vb = p.V + (((size_t)b * p.h_kv + u) * p.n_max) * DH;
    count = p.n + 1;
  }
  const int t0 = min(count, s * p.C);
  const int t1 = min(count, t0 + p.C);
  const int nch = (t1 - t0 + kChunk - 1) / kChunk;

  if (threadIdx.x == 0) {
#pragma unroll
    for (int i = 0; i < NST; ++i) mbar_init(&kv_bar[i], 1);
    fence_mbar_init();
  }
  __syncthreads();
  // Thread 0 only: chunk c into stage c % NST.
  auto issue = [&](int c) {
    const int a0 = t0 + c * kChunk, a1 = min(t1, a0 + kChunk);
    const uint32_t bytes = (uint32_t)(a1 - a0) * DH * 2;
    uint16_t* stg = kv_smem + (size_t)(c % NST) * 2 * kChunk * DH;
    const uint64_t pol = policy_evict_first();
    mbar_arrive_expect_tx(&kv_bar[c % NST], 2 * bytes);
    bulk_g2s(stg, Kb + (size_t)a0 * DH, bytes, &kv_bar[c % NST], pol);
    bulk_g2s(stg + kChunk * DH, Vb + (size_t)a0 * DH, bytes, &kv_bar[c % NST], pol);
  };
  if (threadIdx.x == 0 && nch > 0) {
    // K/V rows were written by generic stores (the new token, by the QKV
    // kernel); order them before the async-proxy reads.
    asm volatile("fence.proxy.async.global;" ::: "memory");
    for (int c = 0; c < min(nch, NST); ++c) issue(c);
  }
  // The queries load while the first copies are in flight.
  float q[G][8];
#pragma unroll
  for (int g = 0; g < G; ++g) {
    const float* qs = p.q + (((size_t)b * p.k + e) * G + g) * DH + sub * 8;
#pragma unroll
    for (int i = 0; i < 8; ++i) q[g][i] = qs[i] * kLog2e;
  }
  float m[G], l[G], o[G][8];
#pragma unroll
  for (int g = 0; g < G; ++g) {
    m[g] = -INFINITY;
    l[g] = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) o[g][i] = 0.f;
  }

  int failed = -1;  // first chunk whose copies did not arrive in time
  for (int c = 0; c < nch; ++c) {
    bool staged = mbar_wait(&kv_bar[c % NST], (c / NST) & 1);
    if (!staged && lane == 0) flag(p.st, DV_DEV_TIMEOUT);
    if (!__syncthreads_and(staged)) {
      failed = c;
      break;
    }
    const uint16_t* sK = kv_smem + (size_t)(c % NST) * 2 * kChunk * DH;
    const uint16_t* sV = sK + kChunk * DH;
    const int na = min(kChunk, t1 - (t0 + c * kChunk));
    // Every lane runs every step (the shuffles below need all of them); a
    // lane whose key lies past the chunk carries a zero weight.
    uint4 kv[U], vv[U];
    bool valid[U];
#pragma unroll
    for (int j = 0; j < U; ++j) {
      const int t = warp * KPW + grp + j * 4 * KPW;  // key within the chunk
      valid[j] = t < na;
      if (valid[j]) {
        kv[j] = *reinterpret_cast<const uint4*>(sK + (size_t)t * DH + sub * 8);
        vv[j] = *reinterpret_cast<const uint4*>(sV + (size_t)t * DH + sub * 8);
      } else {
        kv[j] = make_uint4(0, 0, 0, 0);
        vv[j] = kv[j];
      }
    }
    __syncthreads();  // the stage is in registers everywhere: refill it
    if (threadIdx.x == 0 && c + NST < nch) issue(c + NST);
    float sc[U][G];
#pragma unroll
    for (int j = 0; j < U; ++j) {
      float kf[8];
      h8_to_f8(kv[j], kf);
#pragma unroll
      for (int g = 0; g < G; ++g) {
        float t = 0.f;
#pragma unroll
        for (int i = 0; i < 8; ++i) t = fmaf(q[g][i], kf[i], t);
#pragma unroll
        for (int off = LPK / 2; off > 0; off >>= 1) t += __shfl_xor_sync(0xffffffffu, t, off);
        sc[j][g] = valid[j] ? t : -INFINITY;
      }
    }
#pragma unroll
    for (int g = 0; g < G; ++g) {
      float mx = m[g];
#pragma unroll
      for (int j = 0; j < U; ++j) mx = fmaxf(mx, sc[j][g]);
      if (mx == -INFINITY) continue;
      const float corr = (m[g] == -INFINITY) ? 0.f : exp2f(m[g] - mx);
      l[g] *= corr;
#pragma unroll
      for (int i = 0; i < 8; ++i) o[g][i] *= corr;
#pragma unroll
      for (int j = 0; j < U; ++j) {
        const float pj = valid[j] ? exp2f(sc[j][g] - mx) : 0.f;
        l[g] += pj;
        float vf[8];
        h8_to_f8(vv[j], vf);
#pragma unroll
        for (int i = 0; i < 8; ++i) o[g][i] = fmaf(pj, vf[i], o[g][i]);
      }
      m[g] = mx;
    }
  }
  if (failed >= 0 && threadIdx.x == 0) {
    // Give the copies still in flight one more bounded wait before the CTA's
    // shared memory goes away.
    for (int c = failed; c < min(nch, failed + NST); ++c)
      mbar_wait(&kv_bar[c % NST], (c / NST) & 1);
  }
  // Merge the KPW key groups of the warp (lanes with equal sub).
#pragma unroll
  for (int off = 16; off >= LPK; off >>= 1) {
#pragma unroll
    for (int g = 0; g < G; ++g) {
      const float m2 = __shfl_xor_sync(0xffffffffu, m[g], off);
      const float l2 = __shfl_xor_sync(0xffffffffu, l[g], off);
      float o2[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) o2[i] = __shfl_xor_sync(0xffffffffu, o[g][i], off);
      merge<8>(m[g], l[g], o[g], m2, l2, o2);
    }
  }
  if (grp == 0) {
#pragma unroll
    for (int g = 0; g < G; ++g) {
      if (sub == 0) {
        red[warp][g][0] = m[g];
        red[warp][g][1] = l[g];
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) red[warp][g][2 + sub * 8 + i] = o[g][i];
    }
  }
  __syncthreads();
  // Merge the 4 warps: this split's partial (m, l, o).
  for (int i = threadIdx.x; i < G * (DH + 2); i += blockDim.x) {
    const int g = i / (DH + 2), c = i % (DH + 2);
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < 4; ++w) M = fmaxf(M, red[w][g][0]);
    float val;
    if (c == 0) {
      val = M;
    } else {
      val = 0.f;
      if (M != -INFINITY) {
#pragma unroll
        for (int w = 0; w < 4; ++w) {
          const float mw = red[w][g][0];
          if (mw != -INFINITY) val += exp2f(mw - M) * red[w][g][c];
        }
      }
    }
    if (CL) cpart[g][c] = val;
    else p.part[((((size_t)b * p.k + e) * G + g) * p.S + s) * (DH + 2) + c] = val;
  }

  if (CL) {
    // H = sum_s 2^(m_s - M) o_s / sum_s 2^(m_s - M) l_s over the cluster's
    // splits, read by rank 0 in rank order.
    cg::cluster_group cluster = cg::this_cluster();
    cluster.sync();
    if (cluster.block_rank() == 0) {
      const int ns = (int)cluster.num_blocks();
      for (int i = threadIdx.x; i < G * DH; i += blockDim.x) {
        const int g = i / DH, c = i % DH;
        float M = -INFINITY;
        for (int r = 0; r < ns; ++r) M = fmaxf(M, cluster.map_shared_rank(&cpart[g][0], r)[0]);
        float L = 0.f, O = 0.f;
        for (int r = 0; r < ns; ++r) {
          const float* pr = cluster.map_shared_rank(&cpart[g][0], r);
          const float lr = pr[1];
          const float w = (lr > 0.f) ? exp2f(pr[0] - M) : 0.f;
          L += w * lr;
          O += w * pr[2 + c];
        }
        p.H[(((size_t)b * p.k + e) * G + g) * DH + c] = L > 0.f ? O / L : 0.f;
      }
    }
    cluster.sync();  // the peers' shared memory stays until rank 0 has read it
    return;
  }

  // The last split of this unit to finish combines all splits (no waiting:
  // the others have already published their partials):
  // H = sum_s 2^(m_s - M) o_s / sum_s 2^(m_s - M) l_s.
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) last = (atomicAdd(&p.cnt[(size_t)b * p.k + e], 1) == p.S - 1);
  __syncthreads();
  if (!last) return;
  __threadfence();
  const float* ubase = p.part + (((size_t)b * p.k + e) * G) * p.S * (DH + 2);
  for (int g = warp; g < G; g += 4) {  // one warp per query head: split weights
    const float* base = ubase + (size_t)g * p.S * (DH + 2);
    float ms[kSplitsMax / 32], ls[kSplitsMax / 32];
    float M = -INFINITY;
#pragma unroll
    for (int j = 0; j < kSplitsMax / 32; ++j) {
      const int t = lane + 32 * j;
      ms[j] = t < p.S ? __ldcg(base + (size_t)t * (DH + 2)) : -INFINITY;
      ls[j] = t < p.S ? __ldcg(base + (size_t)t * (DH + 2) + 1) : 0.f;
      M = fmaxf(M, ms[j]);
    }
    M = warp_max(M);
    float L = 0.f;
#pragma unroll
    for (int j = 0; j < kSplitsMax / 32; ++j) {
      const float w = (ls[j] > 0.f) ? exp2f(ms[j] - M) : 0.f;
      if (lane + 32 * j < kSplitsMax) cw[g][lane + 32 * j] = w;
      L += w * ls[j];
    }
    L = warp_sum(L);
    if (lane == 0) cinv[g] = L > 0.f ? 1.f / L : 0.f;
  }
  __syncthreads();
  // O[g][c] = sum_s w[g][s] o_s[g][c]: 128 / DH threads per column, each
  // over every (128 / DH)-th group of 8 splits, with all G x 8 loads issued
  // before they are summed.
  constexpr int TPC = 128 / DH;
  const int c = threadIdx.x % DH, tp = threadIdx.x / DH;
  float O[G];
#pragma unroll
  for (int g = 0; g < G; ++g) O[g] = 0.f;
  for (int t0s = tp * 8; t0s < p.S; t0s += 8 * TPC) {
    float v[G][8];
#pragma unroll
    for (int j = 0; j < 8; ++j)
#pragma unroll
      for (int g = 0; g < G; ++g)
        v[g][j] = (t0s + j < p.S) ? __ldcg(ubase + ((size_t)g * p.S + t0s + j) * (DH + 2) + 2 + c)
                                  : 0.f;
#pragma unroll
    for (int j = 0; j < 8; ++j)
#pragma unroll
      for (int g = 0; g < G; ++g)
        if (t0s + j < p.S) O[g] = fmaf(cw[g][t0s + j], v[g][j], O[g]);
  }
  if (TPC > 1) {
    __syncthreads();  // red is free: the split partial was written above
    if (tp == 1)
#pragma unroll
      for (int g = 0; g < G; ++g) red[0][g][c] = O[g];
    __syncthreads();
  }
  if (tp == 0) {
#pragma unroll
    for (int g = 0; g < G; ++g) {
      const float o = TPC > 1 ? O[g] + red[0][g][c] : O[g];
      p.H[(((size_t)b * p.k + e) * G + g) * DH + c] = o * cinv[g];
    }
  }
  if (threadIdx.x == 0) p.cnt[(size_t)b * p.k + e] = 0;
}

SplitPlan split_plan(int max_keys, int units, int B, int target_ctas) {
  // About target_ctas CTAs in all; each split a whole number of chunks; at
  // most kSplitsMax splits per unit.
  SplitPlan pl;
  const long long ub = std::max(1LL, (long long)units * B);
  long long S = (std::max(1, target_ctas) + ub - 1) / ub;
  S = std::max(1LL, std::min<long long>(S, std::min<long long>(kSplitsMax, (max_keys + kChunk - 1) / kChunk)));
  long long per = (max_keys + S - 1) / S;
  per = std::max<long long>(kChunk, (per + kChunk - 1) / kChunk * kChunk);
  pl.C = (int)per;
  pl.S = (int)std::max(1LL, (max_keys + per - 1) / per);
  return pl;
}

template <int DH, bool CL, int NST>
static void* splitk_fn(int G) {
  switch (G) {
    case 1: return (void*)k_splitk<DH, 1, CL, NST>;
    case 2: return (void*)k_splitk<DH, 2, CL, NST>;
    case 4: return (void*)k_splitk<DH, 4, CL, NST>;
    case 8: return (void*)k_splitk<DH, 8, CL, NST>;
    default: return nullptr;
  }
}

template <int DH>
static void* splitk_pick(int G, bool cl, int nst) {
  if (cl) return splitk_fn<DH, true, 2>(G);
  return nst == 3 ? splitk_fn<DH, false, 3>(G) : splitk_fn<DH, false, 2>(G);
}

int launch_splitk(const float* q, int B, int dh, int G, int h_kv, const int32_t* idx, int k,
                  const int32_t* dev_count, const uint16_t* K, const uint16_t* V, int n, int n_max,
                  const uint16_t* Kr, const uint16_t* Vr, const int32_t* kept_count, int b_max,
                  int retained, SplitPlan plan, float* part, float* H, int* cnt, int* st,
                  cudaStream_t stream, bool pdl) {
  const bool cl = plan.S <= kClusterSplits;
  const int nst = (!cl && (plan.C + kChunk - 1) / kChunk > kLongRangeChunks) ? 3 : 2;
  void* fn = nullptr;
  if (dh == 128) fn = splitk_pick<128>(G, cl, nst);
  if (dh == 64) fn = splitk_pick<64>(G, cl, nst);
  if (!fn) return DV_ERR_UNSUPPORTED;
  SplitParams p{q, K, V, Kr, Vr, kept_count, idx, dev_count, k, h_kv, n, n_max, b_max,
                retained, plan.C, plan.S, part, H, cnt, st};
  void* args[] = {&p};
  const size_t smem = (size_t)nst * 2 * kChunk * dh * 2;  // nst stages of K and V
  if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
    return DV_ERR_LAUNCH;
  note_launch(DV_TAG_SPLITK, 0, stream);
  const cudaError_t e = launch_k(fn, dim3(plan.S, k, B), dim3(128), smem, stream, args, pdl,
                                 cl ? plan.S : 0);
  note_launch(DV_TAG_SPLITK, 1, stream);
  return e == cudaSuccess ? DV_OK : DV_ERR_LAUNCH;
}

// ---------------------------------------------------------------------------
// Attention-scored KV selection
// ---------------------------------------------------------------------------
// Tile: 128 positions x (G*W) queries of one KV head. Scores in base 2.
constexpr int KP = 64;  // positions per CTA

struct KvSelParams {
  const uint16_t* q_obs;  // [h][W][dh]
  const uint16_t* K;      // [h_kv][n_max][dh]
  int h, h_kv, dh, W, n, n_max, nchunks;
  float scale2;           // softmax_scale * log2(e)
  float* stats;           // [h*W][nchunks][2] (m, Z) partials
  float* mz;              // [h*W][2] combined
  float* pooled;          // [h_kv][n]
};

// Scores of the G*W window queries of KV head u against KP positions:
// thread (qi, pj) owns queries qi*4..qi*4+3 and positions pj*4..pj*4+3.
// PASS 0: per-query partial (max, sum 2^(s-max)) over the chunk.
// PASS 1: pooled[u][p] += sum over queries of 2^(s - M_q) / Z_q.
template <int PASS>
__global__ void __launch_bounds__(256) k_kv_score(const KvSelParams p) {
  extern __shared__ __align__(16) float sm[];
  const int chunk = blockIdx.x, u = blockIdx.y;
  const int G = p.h / p.h_kv, NQ = G * p.W;  // NQ <= 512
  const int dh = p.dh;
  float* qT = sm;                 // [dh][NQ]
  float* kT = qT + dh * NQ;       // [dh][KP]
  float* acc = kT + dh * KP;      // PASS 1: [NQ/4][KP]
  const int p0 = chunk * KP;
  for (int i = threadIdx.x; i < NQ * dh; i += blockDim.x) {
    const int qi = i / dh, c = i % dh;
    const int g = qi / p.W, t = qi % p.W;
    const int j = u * G + g;
    qT[c * NQ + qi] = h2f(p.q_obs[((size_t)j * p.W + t) * dh + c]) * p.scale2;
  }
  for (int i = threadIdx.x; i < KP * dh; i += blockDim.x) {
    const int pp = i / dh, c = i % dh;
    const int pos = p0 + pp;
    kT[c * KP + pp] = pos < p.n ? h2f(p.K[((size_t)u * p.n_max + pos) * dh + c]) : 0.f;
  }
  __syncthreads();
  const int nqg = NQ / 4, npg = KP / 4;  // query groups, position groups
  for (int task = threadIdx.x; task < nqg * npg; task += blockDim.x) {
    const int qg = task / npg, pg = task % npg;
    float s[4][4];
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
      for (int c = 0; c < 4; ++c) s[a][c] = 0.f;
    for (int c = 0; c < dh; ++c) {
      const float4 qa = *reinterpret_cast<const float4*>(qT + c * NQ + qg * 4);
      const float4 kb = *reinterpret_cast<const float4*>(kT + c * KP + pg * 4);
      const float qv[4] = {qa.x, qa.y, qa.z, qa.w}, kv[4] = {kb.x, kb.y, kb.z, kb.w};
#pragma unroll
      for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) s[a][cc] = fmaf(qv[a], kv[cc], s[a][cc]);
    }
    // Causal limit: query t sits at position n - W + t.
#pragma unroll
    for (int a = 0; a < 4; ++a) {
      const int qi = qg * 4 + a;
      const int t = qi % p.W;
      const int lim = p.n - p.W + t;
#pragma unroll
      for (int cc = 0; cc < 4; ++cc) {
        const int pos = p0 + pg * 4 + cc;
        if (pos > lim || pos >= p.n) s[a][cc] = -INFINITY;
      }
    }
    if (PASS == 0) {
      // write per-(query, position-group) partial max/sum into acc-like scratch
#pragma unroll
      for (int a = 0; a < 4; ++a) {
        float mx = fmaxf(fmaxf(s[a][0], s[a][1]), fmaxf(s[a][2], s[a][3]));
        float z = 0.f;
        if (mx != -INFINITY)
#pragma unroll
          for (int cc = 0; cc < 4; ++cc) z += exp2f(s[a][cc] - mx);
        const int qi = qg * 4 + a;
        acc[(qi * npg + pg) * 2] = mx;
        acc[(qi * npg + pg) * 2 + 1] = z;
      }
    } else {
      float colsum[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int a = 0; a < 4; ++a) {
        const int qi = qg * 4 + a;
        const int j = u * G + qi / p.W, t = qi % p.W;
        const float M = p.mz[((size_t)j * p.W + t) * 2];
        const float Zi = 1.0f / p.mz[((size_t)j * p.W + t) * 2 + 1];
#pragma unroll
        for (int cc = 0; cc < 4; ++cc)
          if (s[a][cc] != -INFINITY) colsum[cc] += exp2f(s[a][cc] - M) * Zi;
      }
#pragma unroll
      for (int cc = 0; cc < 4; ++cc) acc[qg * KP + pg * 4 + cc] = colsum[cc];
    }
  }
  __syncthreads();
  if (PASS == 0) {
    // Combine the position groups per query -> stats[query][chunk].
    for (int qi = threadIdx.x; qi < NQ; qi += blockDim.x) {
      float M = -INFINITY;
      for (int pg = 0; pg < npg; ++pg) M = fmaxf(M, acc[(qi * npg + pg) * 2]);
      float Z = 0.f;
      if (M != -INFINITY)
        for (int pg = 0; pg < npg; ++pg) {
          const float mp = acc[(qi * npg + pg) * 2];
          if (mp != -INFINITY) Z += exp2f(mp - M) * acc[(qi * npg + pg) * 2 + 1];
        }
      const int j = u * G + qi / p.W, t = qi % p.W;
      float* dst = p.stats + (((size_t)j * p.W + t) * p.nchunks + chunk) * 2;
      dst[0] = M;
      dst[1] = Z;
    }
  } else {
    for (int pp = threadIdx.x; pp < KP; pp += blockDim.x) {
      const int pos = p0 + pp;
      if (pos >= p.n) continue;
      float tot = 0.f;
      for (int qg = 0; qg < nqg; ++qg) tot += acc[qg * KP + pp];
      p.pooled[(size_t)u * p.n + pos] = tot;
    }
  }
}

// (M, Z) per window query from the chunk partials.
__global__ void k_kv_mz(const float* __restrict__ stats, int nq, int nchunks,
                        float* __restrict__ mz) {
  const int qi = blockIdx.x * blockDim.x + threadIdx.x;
  if (qi >= nq) return;
  const float* s = stats + (size_t)qi * nchunks * 2;
  float M = -INFINITY;
  for (int c = 0; c < nchunks; ++c) M = fmaxf(M, s[c * 2]);
  float Z = 0.f;
  for (int c = 0; c < nchunks; ++c)
    if (s[c * 2] != -INFINITY) Z += exp2f(s[c * 2] - M) * s[c * 2 + 1];
  mz[qi * 2] = M;
  mz[qi * 2 + 1] = Z;
}

// Centred width-w mean (zero padded, / w); forced positions get +inf keys.
__global__ void k_kv_smooth(const float* __restrict__ pooled, int n, int w, int n_sinks, int W,
                            float* __restrict__ keys, float* __restrict__ user) {
  const int u = blockIdx.y;
  const int pos = blockIdx.x * blockDim.x + threadIdx.x;
  if (pos >= n) return;
  const float* row = pooled + (size_t)u * n;
  const int half = w / 2;
  float s = 0.f;
  for (int o = -half; o <= half; ++o) {
    const int q = pos + o;
    if (q >= 0 && q < n) s += row[q];
  }
  s = s / (float)w;
  if (user) user[(size_t)u * n + pos] = s;
  const bool forced = pos < n_sinks || pos >= n - W;
  keys[(size_t)u * n + pos] = forced ? INFINITY : s;
}

// Gather the kept rows into the retained buffer; record positions and count.
__global__ void k_kv_gather(const uint16_t* __restrict__ K, const uint16_t* __restrict__ V,
                            int n_max, int dh, const int32_t* __restrict__ kept, int ld_kept,
                            int cnt, uint16_t* __restrict__ Kr, uint16_t* __restrict__ Vr,
                            int32_t* __restrict__ kept_pos, int32_t* __restrict__ kept_count,
                            int b_max) {
  const int u = blockIdx.y;
  const int vec = dh / 8;
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < cnt * vec; i += gridDim.x * blockDim.x) {
    const int r = i / vec, c = i % vec;
    const int pos = kept[(size_t)u * ld_kept + r];
    const size_t src = ((size_t)u * n_max + pos) * dh + c * 8;
    const size_t dst = ((size_t)u * b_max + r) * dh + c * 8;
    *reinterpret_cast<uint4*>(Kr + dst) = *reinterpret_cast<const uint4*>(K + src);
    *reinterpret_cast<uint4*>(Vr + dst) = *reinterpret_cast<const uint4*>(V + src);
    if (c == 0) kept_pos[(size_t)u * b_max + r] = pos;
  }
  if (blockIdx.x == 0 && threadIdx.x == 0) kept_count[u] = cnt;
}

size_t kv_select_ws_floats(int h, int h_kv, int W, int n) {
  const size_t nchunks = (n + KP - 1) / KP;
  return (size_t)h * W * nchunks * 2 + (size_t)h * W * 2 + 2 * (size_t)h_kv * n +
         (size_t)h_kv * n;  // stats, mz, pooled + keys, kept indices (int32)
}

int launch_kv_select(const uint16_t* q_obs, int h, int h_kv, int dh, int W, const uint16_t* K,
                     const uint16_t* V, int n, int n_max, float scale, int n_sinks, int smooth,
                     int b, uint16_t* Kr, uint16_t* Vr, int32_t* kept_pos, int32_t* kept_count,
                     int b_max, float* sel_scores, float* ws_f, size_t ws_floats, int* st,
                     cudaStream_t stream) {
  const int G = h / h_kv;
  if (G * W > 512 || (G * W) % 4 != 0 || W > n) return DV_ERR_UNSUPPORTED;
  const int nchunks = (n + KP - 1) / KP;
  if (kv_select_ws_floats(h, h_kv, W, n) > ws_floats) return DV_ERR_WORKSPACE;
  float* stats = ws_f;
  float* mz = stats + (size_t)h * W * nchunks * 2;
  float* pooled = mz + (size_t)h * W * 2;
  float* keys = pooled + (size_t)h_kv * n;
  int32_t* kept = reinterpret_cast<int32_t*>(keys + (size_t)h_kv * n);
  // The scoring contraction on the tensor cores where its shape allows
  // (d_h 64 or 128, G W a multiple of 64 up to 256); CUDA cores otherwise.
  int rc_tc = launch_kv_scores_tc(q_obs, K, h, h_kv, dh, W, n, n_max, scale * kLog2e, stats,
                                  (size_t)h * W * nchunks * 2, pooled, st, stream);
  if (rc_tc != DV_OK && rc_tc != DV_ERR_UNSUPPORTED) return rc_tc;
  KvSelParams p{q_obs, K, h, h_kv, dh, W, n, n_max, nchunks, scale * kLog2e, stats, mz, pooled};
  const int NQ = G * W;
  const size_t smem0 = (size_t)(dh * NQ + dh * KP) * 4 + (size_t)NQ * (KP / 4) * 2 * 4;
  const size_t smem1 = (size_t)(dh * NQ + dh * KP) * 4 + (size_t)(NQ / 4) * KP * 4;
  if (smem0 > 227 * 1024 || smem1 > 227 * 1024) return DV_ERR_UNSUPPORTED;
  if (rc_tc == DV_ERR_UNSUPPORTED) {
    cudaFuncSetAttribute(k_kv_score<0>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem0);
    cudaFuncSetAttribute(k_kv_score<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem1);
    note_launch(DV_TAG_KVSEL, 0, stream);
    k_kv_score<0><<<dim3(nchunks, h_kv), 256, smem0, stream>>>(p);
    note_launch(DV_TAG_KVSEL, 1, stream);
    note_launch(DV_TAG_KVSEL, 0, stream);
    k_kv_mz<<<(h * W + 127) / 128, 128, 0, stream>>>(stats, h * W, nchunks, mz);
    note_launch(DV_TAG_KVSEL, 1, stream);
    note_launch(DV_TAG_KVSEL, 0, stream);
    k_kv_score<1><<<dim3(nchunks, h_kv), 256, smem1, stream>>>(p);
    note_launch(DV_TAG_KVSEL, 1, stream);
  }
  note_launch(DV_TAG_KVSEL, 0, stream);
  k_kv_smooth<<<dim3((n + 255) / 256, h_kv), 256, 0, stream>>>(pooled, n, smooth, n_sinks, W, keys,
                                                               sel_scores);
  note_launch(DV_TAG_KVSEL, 1, stream);
  int forced = std::min(n, n_sinks) + W;
  if (n_sinks > n - W) forced = n;  // sinks overlap the window
  const int kk = std::min(n, std::max(b, forced));
  if (kk > b_max - 1) return DV_ERR_DIMS;
  int rc = launch_topk(keys, h_kv, n, n, nullptr, kk, kept, n, st, stream);
  if (rc != DV_OK) return rc;
  note_launch(DV_TAG_KVSEL, 0, stream);
  k_kv_gather<<<dim3(std::max(1, std::min(64, (kk * (dh / 8) + 255) / 256)), h_kv), 256, 0,
                stream>>>(K, V, n_max, dh, kept, n, kk, Kr, Vr, kept_pos, kept_count, b_max);
  note_launch(DV_TAG_KVSEL, 1, stream);
  return cudaGetLastError() == cudaSuccess ? DV_OK : DV_ERR_LAUNCH;
}

// Append the new token K/V[u][n] at Kr/Vr[u][kept_count[u]].
__global__ void k_kv_append(const uint16_t* __restrict__ K, const uint16_t* __restrict__ V, int dh,
                            int n, int n_max, uint16_t* __restrict__ Kr, uint16_t* __restrict__ Vr,
                            const int32_t* __restrict__ kept_count, int b_max) {
  const int u = blockIdx.x;
  const int slot = kept_count[u];
  if (slot < 0 || slot >= b_max) return;
  for (int c = threadIdx.x; c < dh; c += blockDim.x) {
    Kr[((size_t)u * b_max + slot) * dh + c] = K[((size_t)u * n_max + n) * dh + c];
    Vr[((size_t)u * b_max + slot) * dh + c] = V[((size_t)u * n_max + n) * dh + c];
  }
}

int launch_kv_append(const uint16_t* K, const uint16_t* V, int h_kv, int dh, int n, int n_max,
                     uint16_t* Kr, uint16_t* Vr, const int32_t* kept_count, int b_max,
                     cudaStream_t stream) {
  note_launch(DV_TAG_KVAPPEND, 0, stream);
  k_kv_append<<<h_kv, 128, 0, stream>>>(K, V, dh, n, n_max, Kr, Vr, kept_count, b_max);
  note_launch(DV_TAG_KVAPPEND, 1, stream);
  return cudaGetLastError() == cudaSuccess ? DV_OK : DV_ERR_LAUNCH;
}

__global__ void k_kv_advance(int32_t* kept_count, int h_kv, int b_max) {
  const int u = threadIdx.x;
  if (u < h_kv && kept_count[u] + 1 < b_max) kept_count[u] += 1;
}

int launch_kv_advance(int32_t* kept_count, int h_kv, int b_max, cudaStream_t stream) {
  note_launch(DV_TAG_KVADVANCE, 0, stream);
  k_kv_advance<<<1, 32 * ((h_kv + 31) / 32), 0, stream>>>(kept_count, h_kv, b_max);
  note_launch(DV_TAG_KVADVANCE, 1, stream);
  return cudaGetLastError() == cudaSuccess ? DV_OK : DV_ERR_LAUNCH;
}

}  // namespace dv
