// k_select.cu -- set formation on the device (sm_103a).
//
// Top-k ("Deja Vu", §2.3: |S| <= (1 - sparsity) N; §4.1: the predictor's set at
// a test-time sparsity level): one CTA per row runs an MSB-first radix select
// over order-preserving 32-bit keys (4 passes of 8 bits, shared-memory
// histogram), finds the k-th largest key T and how many keys equal to T are
// needed, then compacts in index order with two block scans, so the set comes
// out ascending and equal scores go to the lower index -- bit-exact and
// deterministic. The union of a batch's sets ("Deja Vu", App. C.1) is a
// shared-memory bitmap compacted the same way.
#include <cooperative_groups.h>

#include "dv_internal.h"

namespace cg = cooperative_groups;

namespace dv {

constexpr int kTopkThreads = 256;  // small: fits next to a weight-streaming CTA

// Order-preserving key: larger float -> larger key; -0 and +0 map together.
DV_DEV uint32_t fkey(float f) {
  if (f == 0.f) return 0x80000000u;
  const uint32_t b = __float_as_uint(f);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

// Block-wide exclusive scan of one int per thread; returns the prefix and
// writes the total to *total. Uses `tmp` (32 ints) in shared memory.
DV_DEV int block_exscan(int v, int* tmp, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) tmp[warp] = x;
  __syncthreads();
  if (warp == 0) {
    const int nw = blockDim.x >> 5;
    int w = lane < nw ? tmp[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    tmp[lane] = w;  // inclusive prefix of warp totals
  }
  __syncthreads();
  const int before = (warp > 0 ? tmp[warp - 1] : 0) + x - v;
  *total = tmp[(blockDim.x >> 5) - 1];
  __syncthreads();
  return before;
}

__global__ void __launch_bounds__(kTopkThreads) k_topk(const float* __restrict__ scores, int ld,
                                                       int N, const int* __restrict__ k_per_row,
                                                       int k_default, int32_t* __restrict__ idx,
                                                       int ld_idx, int* st) {
  __shared__ uint32_t hist[256];
  __shared__ uint32_t whist[256 * (kTopkThreads / 32)];
  __shared__ int tmp[32];
  __shared__ uint32_t sh_prefix, sh_krem;
  const int row = blockIdx.x;
  const float* s = scores + (size_t)row * ld;
  int32_t* out = idx + (size_t)row * ld_idx;
  int k = k_per_row ? k_per_row[row] : k_default;
  k = max(0, min(k, N));
  const int tid = threadIdx.x;
  if (k == 0) return;

  // NaN check (sets the status bit; NaN keys sort below everything finite).
  bool nan_seen = false;
  for (int i = tid; i < N; i += blockDim.x) nan_seen |= isnan(s[i]);
  if (__syncthreads_or(nan_seen) && tid == 0) flag(st, DV_DEV_NONFINITE);

  uint32_t prefix = 0, mask = 0, krem = (uint32_t)k;
  const int warp = tid >> 5, nwarp = blockDim.x >> 5;
  for (int pass = 0; pass < 4; ++pass) {
    const int shift = 24 - 8 * pass;
    for (int i = tid; i < 256 * nwarp; i += blockDim.x) whist[i] = 0;
    __syncthreads();
    uint32_t* my = whist + warp * 256;  // per-warp histogram: no cross-warp contention
    for (int i = tid; i < N; i += blockDim.x) {
      const float f = s[i];
      const uint32_t key = isnan(f) ? 0u : fkey(f);
      if ((key & mask) == prefix) atomicAdd(&my[(key >> shift) & 255u], 1u);
    }
    __syncthreads();
    for (int i = tid; i < 256; i += blockDim.x) {
      uint32_t t = 0;
      for (int w = 0; w < nwarp; ++w) t += whist[w * 256 + i];
      hist[i] = t;
    }
    __syncthreads();
    if (tid < 32) {
      // lane L owns digits [255 - 8L - 7, 255 - 8L], scanned from the top.
      uint32_t c[8], loc = 0;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        c[j] = hist[255 - 8 * tid - j];
        loc += c[j];
      }
      uint32_t incl = loc;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
        if (tid >= o) incl += y;
      }
      const uint32_t excl = incl - loc;  // keys with a higher digit than my range
      if (excl < krem && krem <= incl) {
        uint32_t above = excl;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          if (above + c[j] >= krem) {
            const uint32_t digit = 255 - 8 * tid - j;
            sh_prefix = prefix | (digit << shift);
            sh_krem = krem - above;
            break;
          }
          above += c[j];
        }
      }
    }
    __syncthreads();
    prefix = sh_prefix;
    krem = sh_krem;
    mask |= 255u << shift;
    __syncthreads();
  }
  const uint32_t T = prefix;  // the k-th largest key; krem of the keys == T are taken

  // Ordered compaction: thread t owns [c0, c1).
  const int per = (N + blockDim.x - 1) / blockDim.x;
  const int c0 = min(N, tid * per), c1 = min(N, c0 + per);
  int gt = 0, eq = 0;
  for (int i = c0; i < c1; ++i) {
    const float f = s[i];
    const uint32_t key = isnan(f) ? 0u : fkey(f);
    gt += key > T;
    eq += key == T;
  }
  int tot;
  const int eq_before = block_exscan(eq, tmp, &tot);
  int take_eq = min(eq, max(0, (int)krem - eq_before));
  const int pos0 = block_exscan(gt + take_eq, tmp, &tot);
  int pos = pos0;
  for (int i = c0; i < c1; ++i) {
    const float f = s[i];
    const uint32_t key = isnan(f) ? 0u : fkey(f);
    if (key > T) {
      out[pos++] = i;
    } else if (key == T && take_eq > 0) {
      out[pos++] = i;
      --take_eq;
    }
  }
}

DV_DEV uint32_t key_of(float f) { return isnan(f) ? 0u : fkey(f); }

// Scanning hist[0, nb) from the top bin down, find the bin where the running
// count reaches krem: sh[0] = that bin, sh[1] = krem minus the keys above it.
DV_DEV void select_bin(const uint32_t* hist, int nb, uint32_t krem, uint32_t* sh, int* tmp) {
  const int per = nb / (int)blockDim.x;
  const int top = nb - 1 - per * (int)threadIdx.x;
  uint32_t loc = 0;
  for (int j = 0; j < per; ++j) loc += hist[top - j];
  int total;
  const uint32_t excl = (uint32_t)block_exscan((int)loc, tmp, &total);
  if (excl < krem && krem <= excl + loc) {
    uint32_t above = excl;
    for (int j = 0; j < per; ++j) {
      const uint32_t c = hist[top - j];
      if (above + c >= krem) {
        sh[0] = (uint32_t)(top - j);
        sh[1] = krem - above;
        break;
      }
      above += c;
    }
  }
  __syncthreads();
}

// ---------------------------------------------------------------------------
// Cluster top-k: one cluster of 8 CTAs per row. CTA r of the cluster owns
// positions [r C, (r+1) C) (C = ceil(N / 8)) and keeps their keys in shared
// memory (one coalesced read of the row; every later pass is a short rolled
// loop, so the code stays small -- the kernel runs once per prediction, with
// a cold instruction cache). Cluster exchanges go through distributed shared
// memory, each CTA reading its peers in rank order, so all CTAs take the same
// decisions:
//   1. the row's smallest and largest score (and key);
//   2. a histogram over kRangeBins equal value ranges of [min, max] (any
//      monotone map of the scores is exact here: bins only narrow the search;
//      equal ranges spread the keys out, so few atomics collide and few keys
//      share the bin holding the k-th largest score, b1);
//   3. b1's keys of all CTAs gathered; their exact ranks (greater keys, then
//      equal keys at lower positions) give the k-th largest key T and how
//      many keys equal to T are taken -- or, when more than kCandMax keys
//      share b1, an MSB-first radix select (8 bits a pass) over b1's keys;
//   4. ordered compaction: per-warp segments counted with ballots, the CTAs'
//      counts exchanged, then the indices written in ascending order, keys
//      equal to T to the lowest positions first.
// No global atomics, no spin.
// ---------------------------------------------------------------------------
constexpr int kClusterTopk = 8;
constexpr int kRangeBins = 2048;
constexpr int kCandCta = 256;   // b1 keys one CTA can hold for the exchange
constexpr int kCandMax = 512;   // b1 keys of the whole row ranked in shared memory

// Inverse of fkey (NaN's key 0 comes back as a NaN).
DV_DEV float key_float(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

struct RangeBins {
  bool byval;
  float fmn, vscale;
  uint32_t kmn;
  float kscale;
  DV_DEV int operator()(uint32_t key) const {
    float t;
    if (byval) {
      const float f = key_float(key);
      t = isnan(f) ? 0.f : (f - fmn) * vscale;
    } else {
      t = __uint2float_rn(key - kmn) * kscale;
    }
    return min(kRangeBins - 1, max(0, (int)t));
  }
};

__global__ void __cluster_dims__(kClusterTopk, 1, 1) __launch_bounds__(kTopkThreads, 4)
    k_topk_cluster(const float* __restrict__ scores, int ld, int N, int k,
                   int32_t* __restrict__ idx, int ld_idx, int* st) {
  constexpr int NT = kTopkThreads, NW = NT / 32;
  cg::cluster_group cluster = cg::this_cluster();
  extern __shared__ uint32_t keys[];                    // [C] this CTA's keys
  __shared__ __align__(16) uint32_t hist[kRangeBins];   // this CTA's (peers read it)
  __shared__ __align__(16) uint32_t ghist[kRangeBins];  // the cluster's; per-warp in the radix path
  __shared__ uint32_t lkey[kCandCta];                   // this CTA's b1 keys (peers read them)
  __shared__ int lpos[kCandCta];
  __shared__ uint32_t ckey[kCandMax];                   // the row's b1 keys
  __shared__ int cpos[kCandMax];
  __shared__ float mmf[2];                              // this CTA's min, max score (peers read)
  __shared__ uint32_t mmk[2];                           // this CTA's min, max key (peers read)
  __shared__ int lcount;                                // (peers read)
  __shared__ int tot[2];                                // keys > T, == T here (peers read)
  __shared__ int wgt[NW], weq[NW];
  __shared__ int tmp[32];
  __shared__ float tmpf[2][NW];
  __shared__ uint32_t tmpk[2][NW];
  __shared__ uint32_t sh[2];
  const int rank = (int)cluster.block_rank();
  const int row = blockIdx.x / kClusterTopk;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const float* s = scores + (size_t)row * ld;
  int32_t* out = idx + (size_t)row * ld_idx;
  const int C = (N + kClusterTopk - 1) / kClusterTopk;
  const int c0 = min(N, rank * C), c1 = min(N, c0 + C), cn = c1 - c0;
  k = max(1, min(k, N));

  bool nan_seen = false;
  float fmn = INFINITY, fmx = -INFINITY;
  uint32_t kmn = 0xFFFFFFFFu, kmx = 0u;
  // eight loads in flight per thread (one round trip per 8 NT scores, not per NT)
  for (int i0 = 0; i0 < cn; i0 += 8 * NT) {
    float fv[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int i = i0 + j * NT + tid;
      fv[j] = i < cn ? s[c0 + i] : 0.f;
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int i = i0 + j * NT + tid;
      if (i >= cn) continue;
      const float f = fv[j];
      nan_seen |= isnan(f);
      if (!isnan(f)) {
        fmn = fminf(fmn, f);
        fmx = fmaxf(fmx, f);
      }
      const uint32_t key = key_of(f);
      kmn = min(kmn, key);
      kmx = max(kmx, key);
      keys[i] = key;
    }
  }
  for (int i = tid; i < kRangeBins; i += NT) hist[i] = 0;
  if (tid == 0) lcount = 0;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    fmn = fminf(fmn, __shfl_xor_sync(0xffffffffu, fmn, o));
    fmx = fmaxf(fmx, __shfl_xor_sync(0xffffffffu, fmx, o));
    kmn = min(kmn, __shfl_xor_sync(0xffffffffu, kmn, o));
    kmx = max(kmx, __shfl_xor_sync(0xffffffffu, kmx, o));
  }
  if (lane == 0) {
    tmpf[0][warp] = fmn;
    tmpf[1][warp] = fmx;
    tmpk[0][warp] = kmn;
    tmpk[1][warp] = kmx;
  }
  if (__syncthreads_or(nan_seen) && tid == 0) flag(st, DV_DEV_NONFINITE);
  if (tid == 0) {
    for (int w = 1; w < NW; ++w) {
      tmpf[0][0] = fminf(tmpf[0][0], tmpf[0][w]);
      tmpf[1][0] = fmaxf(tmpf[1][0], tmpf[1][w]);
      tmpk[0][0] = min(tmpk[0][0], tmpk[0][w]);
      tmpk[1][0] = max(tmpk[1][0], tmpk[1][w]);
    }
    mmf[0] = tmpf[0][0];
    mmf[1] = tmpf[1][0];
    mmk[0] = tmpk[0][0];
    mmk[1] = tmpk[1][0];
  }
  cluster.sync();  // (1)
  fmn = INFINITY;
  fmx = -INFINITY;
  kmn = 0xFFFFFFFFu;
  kmx = 0u;
  {
    // the peers' values: all remote reads issued before any is used
    float pf0[kClusterTopk], pf1[kClusterTopk];
    uint32_t pk0[kClusterTopk], pk1[kClusterTopk];
#pragma unroll
    for (int r = 0; r < kClusterTopk; ++r) {
      const float* pf = cluster.map_shared_rank(mmf, r);
      const uint32_t* pk = cluster.map_shared_rank(mmk, r);
      pf0[r] = pf[0];
      pf1[r] = pf[1];
      pk0[r] = pk[0];
      pk1[r] = pk[1];
    }
#pragma unroll
    for (int r = 0; r < kClusterTopk; ++r) {
      fmn = fminf(fmn, pf0[r]);
      fmx = fmaxf(fmx, pf1[r]);
      kmn = min(kmn, pk0[r]);
      kmx = max(kmx, pk1[r]);
    }
  }
  // Bins by value when the scores' range is finite, else by key.
  RangeBins bin_of;
  bin_of.byval = isfinite(fmn) && isfinite(fmx);
  bin_of.fmn = fmn;
  bin_of.vscale = bin_of.byval ? (float)kRangeBins / fmaxf(fmx - fmn, 1e-30f) : 0.f;
  bin_of.kmn = kmn;
  bin_of.kscale = (float)kRangeBins / ((float)(kmx - kmn) + 1.f);

  for (int i = tid; i < cn; i += NT) atomicAdd(&hist[bin_of(keys[i])], 1u);
  cluster.sync();  // (2)
  for (int b0 = tid * 4; b0 < kRangeBins; b0 += 4 * NT) {
    uint4 h[kClusterTopk];
#pragma unroll
    for (int r = 0; r < kClusterTopk; ++r)
      h[r] = *reinterpret_cast<const uint4*>(cluster.map_shared_rank(hist, r) + b0);
    uint4 t = make_uint4(0, 0, 0, 0);
#pragma unroll
    for (int r = 0; r < kClusterTopk; ++r) {
      t.x += h[r].x; t.y += h[r].y; t.z += h[r].z; t.w += h[r].w;
    }
    *reinterpret_cast<uint4*>(ghist + b0) = t;
  }
  __syncthreads();
  select_bin(ghist, kRangeBins, (uint32_t)k, sh, tmp);
  const int b1 = (int)sh[0];
  uint32_t krem = sh[1];

  for (int i = tid; i < cn; i += NT)
    if (bin_of(keys[i]) == b1) {
      const int c = atomicAdd(&lcount, 1);
      if (c < kCandCta) {
        lkey[c] = keys[i];
        lpos[c] = c0 + i;
      }
    }
  cluster.sync();  // (3)
  int nc = 0;
  bool fits = true;
  int crs[kClusterTopk];  // the ranks' b1 counts
#pragma unroll
  for (int r = 0; r < kClusterTopk; ++r) crs[r] = *cluster.map_shared_rank(&lcount, r);
#pragma unroll
  for (int r = 0; r < kClusterTopk; ++r) {
    fits &= crs[r] <= kCandCta;
    nc += crs[r];
  }
  fits &= nc <= kCandMax;

  uint32_t T;  // the k-th largest key; krem of the keys equal to T are taken
  if (fits) {
    // one key per thread and rank at most (kCandCta == NT): the ranks' reads
    // are issued together
    uint32_t kv[kClusterTopk];
    int pv[kClusterTopk];
#pragma unroll
    for (int r = 0; r < kClusterTopk; ++r) {
      if (tid < crs[r]) {
        kv[r] = cluster.map_shared_rank(lkey, r)[tid];
        pv[r] = cluster.map_shared_rank(lpos, r)[tid];
      }
    }
    int off = 0;
#pragma unroll
    for (int r = 0; r < kClusterTopk; ++r) {
      if (tid < crs[r]) {
        ckey[off + tid] = kv[r];
        cpos[off + tid] = pv[r];
      }
      off += crs[r];
    }
    __syncthreads();
    for (int c = tid; c < nc; c += NT) {
      const uint32_t kc = ckey[c];
      const int pc = cpos[c];
      int r = 0;
      for (int c2 = 0; c2 < nc; ++c2) {
        const uint32_t k2 = ckey[c2];
        r += (k2 > kc) || (k2 == kc && cpos[c2] < pc);
      }
      if (r == (int)krem - 1) sh[0] = kc;
    }
    __syncthreads();
    T = sh[0];
    int g = 0;
    for (int c = tid; c < nc; c += NT) g += ckey[c] > T;
    int gtot;
    block_exscan(g, tmp, &gtot);
    krem -= (uint32_t)gtot;
  } else {
    // Radix select over b1's keys; per-warp histograms in ghist, the CTA's in
    // hist (read by the peers between the two cluster barriers of a pass).
    uint32_t prefix = 0, mask = 0;
    uint32_t* whist = ghist;
    for (int pass = 0; pass < 4; ++pass) {
      const int shift = 24 - 8 * pass;
      for (int i = tid; i < NW * 256; i += NT) whist[i] = 0;
      __syncthreads();
      for (int i = tid; i < cn; i += NT) {
        const uint32_t key = keys[i];
        if (bin_of(key) == b1 && (key & mask) == prefix)
          atomicAdd(&whist[warp * 256 + ((key >> shift) & 255u)], 1u);
      }
      __syncthreads();
      {
        uint32_t t = 0;
        for (int w = 0; w < NW; ++w) t += whist[w * 256 + tid];
        hist[tid] = t;
      }
      cluster.sync();
      {
        uint32_t hr[kClusterTopk];
#pragma unroll
        for (int r = 0; r < kClusterTopk; ++r) hr[r] = cluster.map_shared_rank(hist, r)[tid];
        uint32_t t = 0;
#pragma unroll
        for (int r = 0; r < kClusterTopk; ++r) t += hr[r];
        whist[tid] = t;
      }
      __syncthreads();
      select_bin(whist, 256, krem, sh, tmp);
      prefix |= sh[0] << shift;
      krem = sh[1];
      mask |= 255u << shift;
      cluster.sync();  // the peers are done reading hist
    }
    T = prefix;
  }

  // Ordered compaction over warp segments (multiples of 32 positions).
  const int seg = (cn + NT - 1) / NT * 32;
  const int w0 = min(cn, warp * seg), w1 = min(cn, w0 + seg);
  int gt = 0, eq = 0;
  for (int base = w0; base < w1; base += 32) {
    const int i = base + lane;
    const bool v = i < w1;
    const uint32_t key = v ? keys[i] : 0u;
    gt += __popc(__ballot_sync(0xffffffffu, v && key > T));
    eq += __popc(__ballot_sync(0xffffffffu, v && key == T));
  }
  if (lane == 0) {
    wgt[warp] = gt;
    weq[warp] = eq;
  }
  __syncthreads();
  if (tid == 0) {
    int a = 0, b = 0;
    for (int w = 0; w < NW; ++w) {
      a += wgt[w];
      b += weq[w];
    }
    tot[0] = a;
    tot[1] = b;
  }
  cluster.sync();  // (4)
  int pos = 0, eqb = 0;
  {
    int t0[kClusterTopk], t1[kClusterTopk];
#pragma unroll
    for (int r = 0; r < kClusterTopk; ++r) {
      if (r < rank) {
        const int* o = cluster.map_shared_rank(tot, r);
        t0[r] = o[0];
        t1[r] = o[1];
      }
    }
#pragma unroll
    for (int r = 0; r < kClusterTopk; ++r) {
      if (r < rank) {
        pos += t0[r] + min(t1[r], max(0, (int)krem - eqb));
        eqb += t1[r];
      }
    }
  }
  for (int w = 0; w < warp; ++w) {
    pos += wgt[w] + min(weq[w], max(0, (int)krem - eqb));
    eqb += weq[w];
  }
  const unsigned lt = (1u << lane) - 1u;
  for (int base = w0; base < w1; base += 32) {
    const int i = base + lane;
    const bool v = i < w1;
    const uint32_t key = v ? keys[i] : 0u;
    const unsigned me = __ballot_sync(0xffffffffu, v && key == T);
    const bool take = v && (key > T || (key == T && eqb + __popc(me & lt) < (int)krem));
    const unsigned mt = __ballot_sync(0xffffffffu, take);
    if (take) out[pos + __popc(mt & lt)] = c0 + i;
    pos += __popc(mt);
    eqb += __popc(me);
  }
  cluster.sync();  // (5) keep this CTA's shared memory alive until all peers read it
}

// ---------------------------------------------------------------------------
// Short rows (N <= kSmallN, e.g. the head scores): one CTA of 256 threads per
// row (small enough to share an SM with a weight-streaming CTA) loads the
// row's keys into shared memory once, runs the 4-pass radix select there and
// compacts in index order with warp ballots over per-warp segments.
// ---------------------------------------------------------------------------
constexpr int kSmallN = 4096;


__global__ void __launch_bounds__(kTopkThreads, 4) k_topk_small(const float* __restrict__ scores,
                                                                 int ld, int N, int k,
                                                                 int32_t* __restrict__ idx,
                                                                 int ld_idx, int* st) {
  constexpr int NW = kTopkThreads / 32;
  __shared__ uint32_t keys[kSmallN];
  __shared__ uint32_t hist[256];
  __shared__ int tmp[32];
  __shared__ uint32_t sh[2];
  __shared__ int wgt[NW], weq[NW];
  const float* s = scores + (size_t)blockIdx.x * ld;
  int32_t* out = idx + (size_t)blockIdx.x * ld_idx;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  k = max(1, min(k, N));

  bool nan_seen = false;
  for (int i = tid; i < N; i += kTopkThreads) {
    const float f = s[i];
    nan_seen |= isnan(f);
    keys[i] = key_of(f);
  }
  if (__syncthreads_or(nan_seen) && tid == 0) flag(st, DV_DEV_NONFINITE);

  if (N <= 2 * kTopkThreads) {
    // Short rows: the rank of each key (greater keys, then equal keys at lower
    // positions) by one pass over the row; it is taken when its rank is below
    // k. The taken positions come out ascending through two block scans
    // (positions tid, then kTopkThreads + tid).
    bool take[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int i = h * kTopkThreads + tid;
      take[h] = false;
      if (i < N) {
        const uint32_t ki = keys[i];
        int r = 0;
        for (int j = 0; j < N; ++j) {
          const uint32_t kj = keys[j];
          r += (kj > ki) || (kj == ki && j < i);
        }
        take[h] = r < k;
      }
    }
    int base = 0;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      int tot;
      const int before = block_exscan(take[h] ? 1 : 0, tmp, &tot);
      if (take[h]) out[base + before] = h * kTopkThreads + tid;
      base += tot;
    }
    return;
  }

  uint32_t prefix = 0, mask = 0, krem = (uint32_t)k;
  for (int pass = 0; pass < 4; ++pass) {
    const int shift = 24 - 8 * pass;
    for (int i = tid; i < 256; i += kTopkThreads) hist[i] = 0;
    __syncthreads();
    for (int i = tid; i < N; i += kTopkThreads)
      if ((keys[i] & mask) == prefix) atomicAdd(&hist[(keys[i] >> shift) & 255u], 1u);
    __syncthreads();
    select_bin(hist, 256, krem, sh, tmp);
    prefix |= sh[0] << shift;
    krem = sh[1];
    mask |= 255u << shift;
  }
  const uint32_t T = prefix;  // the k-th largest key; krem of the keys equal to T are taken

  // Ordered compaction over warp segments (multiples of 32 positions).
  const int seg = (N + kTopkThreads - 1) / kTopkThreads * 32;
  const int w0 = min(N, warp * seg), w1 = min(N, w0 + seg);
  int gt = 0, eq = 0;
  for (int base = w0; base < w1; base += 32) {
    const int i = base + lane;
    const bool v = i < w1;
    const uint32_t key = v ? keys[i] : 0u;
    gt += __popc(__ballot_sync(0xffffffffu, v && key > T));
    eq += __popc(__ballot_sync(0xffffffffu, v && key == T));
  }
  if (lane == 0) {
    wgt[warp] = gt;
    weq[warp] = eq;
  }
  __syncthreads();
  int pos = 0, eqb = 0;
  for (int w = 0; w < warp; ++w) {
    pos += wgt[w] + min(weq[w], max(0, (int)krem - eqb));
    eqb += weq[w];
  }
  const unsigned lt = (1u << lane) - 1u;
  for (int base = w0; base < w1; base += 32) {
    const int i = base + lane;
    const bool v = i < w1;
    const uint32_t key = v ? keys[i] : 0u;
    const unsigned me = __ballot_sync(0xffffffffu, v && key == T);
    const bool take = v && (key > T || (key == T && eqb + __popc(me & lt) < (int)krem));
    const unsigned mt = __ballot_sync(0xffffffffu, take);
    if (take) out[pos + __popc(mt & lt)] = i;
    pos += __popc(mt);
    eqb += __popc(me);
  }
}

constexpr int kClusterMaxN = 131072;  // 64 KB of keys per CTA (opt-in shared memory)

static int launch_topk_cluster(const float* scores, int B, int ld, int N, int k, int32_t* idx,
                               int ld_idx, int* st, cudaStream_t stream) {
  // The keys go in dynamic shared memory; together with the static arrays
  // they can pass the 48 KB that needs no opt-in, so the limit is always set.
  const size_t smem = (size_t)((N + kClusterTopk - 1) / kClusterTopk) * 4;
  if (cudaFuncSetAttribute((const void*)k_topk_cluster, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)smem) != cudaSuccess)
    return DV_ERR_LAUNCH;
  k_topk_cluster<<<B * kClusterTopk, kTopkThreads, smem, stream>>>(scores, ld, N, k, idx, ld_idx, st);
  return cudaGetLastError() == cudaSuccess ? DV_OK : DV_ERR_LAUNCH;
}

int launch_topk(const float* scores, int B, int ld, int N, const int* k_per_row, int k,
                int32_t* idx, int ld_idx, int* st, cudaStream_t stream) {
  int rc = DV_ERR_UNSUPPORTED;
  note_launch(DV_TAG_TOPK, 0, stream);
  if (!k_per_row && N <= kSmallN) {
    k_topk_small<<<B, kTopkThreads, 0, stream>>>(scores, ld, N, k, idx, ld_idx, st);
    rc = cudaGetLastError() == cudaSuccess ? DV_OK : DV_ERR_LAUNCH;
  } else if (!k_per_row && N <= kClusterMaxN) {
    rc = launch_topk_cluster(scores, B, ld, N, k, idx, ld_idx, st, stream);
  } else {
    k_topk<<<B, kTopkThreads, 0, stream>>>(scores, ld, N, k_per_row, k, idx, ld_idx, st);
    rc = cudaGetLastError() == cudaSuccess ? DV_OK : DV_ERR_LAUNCH;
  }
  note_launch(DV_TAG_TOPK, 1, stream);
  return rc;
}

// Union of B ascending sets of width k over [0, N): bitmap, then ordered
// compaction over 32-bit words.
__global__ void __launch_bounds__(256) k_union(const int32_t* __restrict__ idx, int B, int k,
                                                int N, int32_t* __restrict__ out,
                                                int32_t* __restrict__ count) {
  extern __shared__ uint32_t bits[];
  __shared__ int tmp[32];
  const int words = (N + 31) / 32;
  for (int w = threadIdx.x; w < words; w += blockDim.x) bits[w] = 0;
  __syncthreads();
  // Eight indices in flight per thread (one dependent load per iteration
  // would make this loop latency-bound).
  const int nidx = B * k;
  for (int i0 = threadIdx.x; i0 < nidx; i0 += 8 * blockDim.x) {
    int j[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int i = i0 + u * blockDim.x;
      j[u] = i < nidx ? __ldg(idx + i) : -1;
    }
#pragma unroll
    for (int u = 0; u < 8; ++u)
      if (j[u] >= 0 && j[u] < N) atomicOr(&bits[j[u] >> 5], 1u << (j[u] & 31));
  }
  __syncthreads();
  const int per = (words + blockDim.x - 1) / blockDim.x;
  const int w0 = min(words, (int)threadIdx.x * per), w1 = min(words, w0 + per);
  int c = 0;
  for (int w = w0; w < w1; ++w) c += __popc(bits[w]);
  int tot;
  int pos = block_exscan(c, tmp, &tot);
  for (int w = w0; w < w1; ++w) {
    uint32_t m = bits[w];
    while (m) {
      const int b = __ffs(m) - 1;
      out[pos++] = w * 32 + b;
      m &= m - 1;
    }
  }
  if (threadIdx.x == 0) *count = tot;
}

int launch_union(const int32_t* idx, int B, int k, int N, int32_t* out, int32_t* count,
                 cudaStream_t stream) {
  const size_t smem = (size_t)((N + 31) / 32) * 4;
  if (smem > 200 * 1024) return DV_ERR_UNSUPPORTED;
  if (smem + 1024 > 48 * 1024 &&  // with the static scan buffer
      cudaFuncSetAttribute(k_union, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
          cudaSuccess)
    return DV_ERR_LAUNCH;
  note_launch(DV_TAG_UNION, 0, stream);
  k_union<<<1, 256, smem, stream>>>(idx, B, k, N, out, count);
  note_launch(DV_TAG_UNION, 1, stream);
  return cudaGetLastError() == cudaSuccess ? DV_OK : DV_ERR_LAUNCH;
}

}  // namespace dv
