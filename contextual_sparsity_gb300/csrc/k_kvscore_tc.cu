// k_kvscore_tc.cu -- the scoring pass of attention-scored KV selection on the
// fifth-generation tensor cores ("Where Activation Sparsity and KV-Cache
// Sparsity Cross in LLM Decoding", §4.1 and App. A: the last 64 prompt
// positions' queries attend causally over the cache; their softmax
// probabilities, pooled over the window and the query heads of a KV head,
// score the positions).
//
// Per KV head u the NQ = G * W window queries (G query heads x W positions,
// contiguous rows of q_obs) meet the n cached keys: a dense contraction of
// NQ x d_h by d_h x n. Two launches over the same grid (KV head, key range):
//   pass 0  S = Q K^T per 256-key tile (M = 128 queries per instruction,
//           N = 256 keys, K = d_h; one 256-column accumulator per query
//           tile), each query's running max and sum of 2^(s - max) over the
//           CTA's key range, written per split;
//   pass 1  the splits combined per query (M_q, L_q), then S^T = K Q^T per
//           128-key tile (M = 128 keys, N = NQ queries) so that each TMEM
//           lane is one key: pooled[u][key] = sum_q 2^(s - M_q) / L_q over the
//           queries whose position admits the key, a per-thread sum.
// Key tiles and the queries are brought by tiled TMA loads (128-byte
// swizzle, no multicast) into shared memory; one thread issues tcgen05.mma
// into TMEM accumulators (two buffers); sixteen warps read them back with
// tcgen05.ld. Scores are in base 2 (scaled by softmax_scale * log2 e).
#include "dv_internal.h"
#include "dv_tc.cuh"

namespace dv {

namespace {

constexpr int kTcKeys = 128;      // keys per pass-1 tile (M = 128 keys)
constexpr int kTcStages = 4;      // pass-1 K tiles in flight
// Pass 0 takes 256 keys per tile (N = 256, the instruction width that keeps
// the tensor pipe at full rate) in two stages of the same total size.
template <int PASS> constexpr int tc_keys() { return PASS == 0 ? 256 : kTcKeys; }
template <int PASS> constexpr int tc_stages() { return PASS == 0 ? 2 : kTcStages; }
constexpr int kBoxBytes = 128 * 128;  // one TMA box: 128 rows x 64 fp16
constexpr int kEpiWarps = 16;  // 4 per TMEM lane quadrant
constexpr int kThreads = (kEpiWarps + 2) * 32;  // + producer warp + MMA warp
constexpr uint32_t kTmemCols = 512;

struct KvTcParams {
  int h_kv, W, n, n_max, NQ, MT, KB, nsplit, tiles, tiles0;  // tiles0: pass-0 (256-key) tiles
  float scale2;
  float* stats;   // [h_kv][NQ][nsplit][2]
  float* pooled;  // [h_kv][n]
  int* st;
};

struct KvTcSmem {
  uint32_t q, k, bars, misc, total;  // byte offsets from the 1024-aligned base
};

__host__ __device__ inline KvTcSmem kvtc_layout(int KB, int MTQ) {
  KvTcSmem L{};
  L.q = 0;
  L.k = L.q + KB * MTQ * kBoxBytes;
  L.bars = L.k + kTcStages * KB * kBoxBytes;
  L.misc = L.bars + 256;
  // misc: tmem slot, abort flag, then cst[256], lim[256] (pass 0: the second
  // key half's max and sum per query), red[2][4][128] (pass 1)
  L.total = L.misc + 16 + 256 * 4 * 2 + 2 * 4 * 128 * 4;
  return L;
}

template <int PASS>
__global__ void __launch_bounds__(kThreads, 1)
    k_kvscore_tc(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmQ,
                 const KvTcParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~uintptr_t(1023));
  const int MTQ = (p.NQ + 127) / 128;
  const KvTcSmem L = kvtc_layout(p.KB, MTQ);
  uint8_t* sQ = sm + L.q;
  uint8_t* sK = sm + L.k;
  uint64_t* full = reinterpret_cast<uint64_t*>(sm + L.bars);
  uint64_t* empty = full + kTcStages;
  uint64_t* qbar = empty + kTcStages;
  uint64_t* accf = qbar + 1;
  uint64_t* acce = accf + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + L.misc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + L.misc + 4);
  float* cst = reinterpret_cast<float*>(sm + L.misc + 16);
  int* lims = reinterpret_cast<int*>(cst + 256);
  float* red = reinterpret_cast<float*>(lims + 256);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int u = blockIdx.y, split = blockIdx.x;
  constexpr int KT = tc_keys<PASS>(), NS = tc_stages<PASS>();
  const int tiles = PASS == 0 ? p.tiles0 : p.tiles;
  const int t0 = (int)((long long)tiles * split / p.nsplit);
  const int t1 = (int)((long long)tiles * (split + 1) / p.nsplit);
  const int ntiles = t1 - t0;
  // pass 0: a warp per (TMEM lane quadrant, query tile, key half of a tile);
  // pass 1: a warp per (lane quadrant, 64 query columns)
  const int epi_warps = PASS == 0 ? 8 * p.MT : 4 * (p.NQ / 64);

  if (tid == 0) {
    for (int s = 0; s < kTcStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(qbar, 1);
    for (int a = 0; a < 2; ++a) {
      mbar_init(&accf[a], 1);
      // pass 0: each accumulator is read by the 8 warps of one query tile
      mbar_init(&acce[a], PASS == 0 ? 8 : epi_warps);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kEpiWarps + 1) {
    tmem_alloc(tmem_slot, kTmemCols);
    tc_fence_before();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  auto give_up = [&]() {
    *abort_flag = 1;
    flag(p.st, DV_DEV_TIMEOUT);
  };

  if (warp == kEpiWarps) {
    // ---------------- producer: the queries once, then the key tiles ----------
    if (lane == 0) {
      tma_prefetch_map(&tmK);
      tma_prefetch_map(&tmQ);
      mbar_arrive_expect_tx(qbar, p.KB * MTQ * kBoxBytes);
      for (int kb = 0; kb < p.KB; ++kb)
        for (int mt = 0; mt < MTQ; ++mt)
          tma_load_2d(sQ + (kb * MTQ + mt) * kBoxBytes, &tmQ, kb * 64, u * p.NQ + mt * 128, qbar);
      int i = 0;
      constexpr int KBLK = KT / 128;  // 128-row boxes per 64-column slice of a tile
      for (; i < ntiles && !*abort_flag; ++i) {
        const int s = i % NS;
        if (i >= NS && !mbar_wait(&empty[s], ((i / NS) & 1) ^ 1)) {
          give_up();
          break;
        }
        mbar_arrive_expect_tx(&full[s], p.KB * KBLK * kBoxBytes);
        const int row = u * p.n_max + (t0 + i) * KT;
        // slice kb of the tile: its KBLK boxes of 128 keys back to back, so
        // the KT rows form one 128-byte-swizzled operand
        for (int kb = 0; kb < p.KB; ++kb)
          for (int kbk = 0; kbk < KBLK; ++kbk)
            tma_load_2d(sK + ((s * p.KB + kb) * KBLK + kbk) * kBoxBytes, &tmK, kb * 64,
                        row + kbk * 128, &full[s]);
      }
      // every issued copy lands before the CTA exits
      if (!mbar_wait(qbar, 0)) flag(p.st, DV_DEV_TIMEOUT);
      for (int j = (i > NS ? i - NS : 0); j < i; ++j)
        if (!mbar_wait(&full[j % NS], (j / NS) & 1)) flag(p.st, DV_DEV_TIMEOUT);
    }
    __syncwarp();
  } else if (warp == kEpiWarps + 1) {
    // ---------------- MMA issuer (one thread) ----------------------------------
    if (lane == 0) {
      const uint32_t sq = smem_addr(sQ), sk = smem_addr(sK);
      bool ok = mbar_wait(qbar, 0);
      if (!ok) give_up();
      for (int i = 0; i < ntiles && ok && !*abort_flag; ++i) {
        const int s = i % NS, a = i & 1;
        if (!mbar_wait(&full[s], (i / NS) & 1)) {
          give_up();
          break;
        }
        if (PASS == 0) {
          // 256 columns of TMEM per query tile: with two query tiles each has
          // its own accumulator (buffer mt, used once per key tile), with one
          // the two buffers alternate between key tiles
          const uint32_t kst = sk + s * p.KB * 2 * kBoxBytes;
          const uint32_t idesc = idesc_f16_f32(128, KT);
          for (int mt = 0; mt < p.MT && ok; ++mt) {
            const int b = p.MT == 2 ? mt : a;
            const int use = p.MT == 2 ? i : (i >> 1);  // earlier uses of buffer b
            if (use >= 1 && !mbar_wait(&acce[b], (use - 1) & 1)) {
              give_up();
              ok = false;
              break;
            }
            tc_fence_after();
            for (int kk = 0; kk < p.KB * 4; ++kk) {
              const int kb = kk >> 2, ko = kk & 3;
              tc_mma_f16(tmem + b * KT, sdesc_k128(sq + (kb * MTQ + mt) * kBoxBytes + ko * 32),
                         sdesc_k128(kst + kb * 2 * kBoxBytes + ko * 32), idesc, kk > 0);
            }
            tc_commit(&accf[b]);  // this query tile's scores are ready
          }
          if (!ok) break;
          tc_commit(&empty[s]);  // the stage is free once these products are done
          continue;
        }
        if (i >= 2 && !mbar_wait(&acce[a], ((i >> 1) & 1) ^ 1)) {
          give_up();
          break;
        }
        tc_fence_after();
        const uint32_t kst = sk + s * p.KB * kBoxBytes;
        {
          const uint32_t idesc = idesc_f16_f32(128, p.NQ);
          for (int kk = 0; kk < p.KB * 4; ++kk) {
            const int kb = kk >> 2, ko = kk & 3;
            tc_mma_f16(tmem + a * p.NQ, sdesc_k128(kst + kb * kBoxBytes + ko * 32),
                       sdesc_k128(sq + kb * MTQ * kBoxBytes + ko * 32), idesc, kk > 0);
          }
        }
        tc_commit(&empty[s]);  // the stage is free once these products are done
        tc_commit(&accf[a]);   // and the accumulator is ready
      }
    }
    __syncwarp();
  } else if (PASS == 0) {
    // ---------------- pass 0 epilogue: running max / sum per query --------------
    if (warp < epi_warps) {
      const int hq = warp / (4 * p.MT), rest = warp % (4 * p.MT);
      const int q = rest & 3, mt = rest >> 2;  // q = warp % 4: this warp's lane quadrant
      const int qi = mt * 128 + q * 32 + lane;
      const int lim = qi < p.NQ ? p.n - p.W + qi % p.W : -1;  // last admitted key
      const float s2 = p.scale2;
      float m = -INFINITY, l = 0.f;
      for (int i = 0; i < ntiles; ++i) {
        const int b = p.MT == 2 ? mt : (i & 1);     // this query tile's accumulator
        const int use = p.MT == 2 ? i : (i >> 1);  // earlier uses of buffer b
        if (*abort_flag) break;
        if (!mbar_wait(&accf[b], use & 1)) {
          give_up();
          break;
        }
        tc_fence_after();
        const uint32_t ta = tmem + ((uint32_t)(q * 32) << 16) + b * KT + hq * (KT / 2);
        // this query's 128 scores of the tile's key half, 64 at a time
#pragma unroll 1
        for (int c = 0; c < 2; ++c) {
          uint32_t r[64];
          tmem_ld32_nw(ta + c * 64, r);
          tmem_ld32_nw(ta + c * 64 + 32, r + 32);
          tmem_wait_ld();
          if (c == 1) {  // the accumulator is read: the next key tile may overwrite it
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&acce[b]);
          }
          const int key0 = (t0 + i) * KT + hq * (KT / 2) + c * 64;
          float v[64];
#pragma unroll
          for (int j = 0; j < 64; ++j) v[j] = __uint_as_float(r[j]);
          if (key0 + 63 > p.n - p.W) {  // the causal limit cuts these keys for some query
#pragma unroll
            for (int j = 0; j < 64; ++j)
              if (key0 + j > lim) v[j] = -INFINITY;
          }
          float mx = v[0];
#pragma unroll
          for (int j = 1; j < 64; ++j) mx = fmaxf(mx, v[j]);
          mx *= s2;  // scale > 0: the max of the scaled scores
          if (mx > m) {
            l *= ex2_approx(m - mx);
            m = mx;
          }
          if (m != -INFINITY) {
            float acc0 = 0.f, acc1 = 0.f;
#pragma unroll
            for (int j = 0; j < 64; j += 2) {
              acc0 += ex2_approx(fmaf(v[j], s2, -m));
              acc1 += ex2_approx(fmaf(v[j + 1], s2, -m));
            }
            l += acc0 + acc1;
          }
        }
      }
      // the two key halves of each query meet in shared memory
      if (hq == 1) {
        cst[qi] = m;
        reinterpret_cast<float*>(lims)[qi] = l;
      }
      consumer_sync(epi_warps * 32);
      if (hq == 0 && qi < p.NQ) {
        const float m1 = cst[qi], l1 = reinterpret_cast<const float*>(lims)[qi];
        const float M = fmaxf(m, m1);
        float L = 0.f;
        if (m != -INFINITY) L += l * ex2_approx(m - M);
        if (m1 != -INFINITY) L += l1 * ex2_approx(m1 - M);
        float* dst = p.stats + (((size_t)u * p.NQ + qi) * p.nsplit + split) * 2;
        dst[0] = M;
        dst[1] = L;
      }
    }
  } else {
    // ---------------- pass 1 epilogue: pooled probabilities per key ------------
    // The splits' (max, sum) of every query of this KV head, combined.
    for (int qi = tid; qi < p.NQ; qi += kEpiWarps * 32) {
      const float* s = p.stats + ((size_t)u * p.NQ + qi) * p.nsplit * 2;
      float M = -INFINITY;
      for (int j = 0; j < p.nsplit; ++j) M = fmaxf(M, s[2 * j]);
      float Ls = 0.f;
      for (int j = 0; j < p.nsplit; ++j)
        if (s[2 * j] != -INFINITY) Ls += exp2f(s[2 * j] - M) * s[2 * j + 1];
      cst[qi] = (Ls > 0.f) ? -(M + log2f(Ls)) : -INFINITY;
      lims[qi] = p.n - p.W + qi % p.W;
    }
    consumer_sync(kEpiWarps * 32);
    const int q = warp & 3, half = warp >> 2;  // half: which 64 query columns
    const int cols = 64;
    bool dead = false;
    for (int i = 0; i < ntiles && warp < epi_warps; ++i) {
      const int a = i & 1;
      const int key0 = (t0 + i) * kTcKeys;
      const int key = key0 + q * 32 + lane;
      float sum = 0.f;
      if (!dead && (*abort_flag || !mbar_wait(&accf[a], (i >> 1) & 1))) {
        give_up();
        dead = true;
      }
      if (!dead) {
        tc_fence_after();
        const bool nomask = key0 + kTcKeys - 1 <= p.n - p.W;  // every query admits every key
        const uint32_t ta = tmem + ((uint32_t)(q * 32) << 16) + a * p.NQ + half * cols;
        const float s2 = p.scale2;
        float acc0 = 0.f, acc1 = 0.f;
#pragma unroll 1
        for (int c = 0; c < cols / 32; c += 2) {  // two 32-column loads in flight (one at an odd end)
          uint32_t r[64];
          const int nc = (c + 1 < cols / 32) ? 2 : 1;
          tmem_ld32_nw(ta + c * 32, r);
          if (nc == 2) tmem_ld32_nw(ta + c * 32 + 32, r + 32);
          tmem_wait_ld();
          for (int h = 0; h < nc; ++h) {
            const int qb = half * cols + (c + h) * 32;
            const float4* cs = reinterpret_cast<const float4*>(cst + qb);
            if (nomask) {
#pragma unroll
              for (int j4 = 0; j4 < 8; ++j4) {
                const float4 cc = cs[j4];
                acc0 += ex2_approx(fmaf(__uint_as_float(r[h * 32 + 4 * j4]), s2, cc.x));
                acc1 += ex2_approx(fmaf(__uint_as_float(r[h * 32 + 4 * j4 + 1]), s2, cc.y));
                acc0 += ex2_approx(fmaf(__uint_as_float(r[h * 32 + 4 * j4 + 2]), s2, cc.z));
                acc1 += ex2_approx(fmaf(__uint_as_float(r[h * 32 + 4 * j4 + 3]), s2, cc.w));
              }
            } else {
#pragma unroll
              for (int j = 0; j < 32; ++j)
                if (key <= lims[qb + j])
                  acc0 += ex2_approx(fmaf(__uint_as_float(r[h * 32 + j]), s2, cst[qb + j]));
            }
          }
        }
        sum = acc0 + acc1;
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&acce[a]);
      }
      // the column parts of a key meet in shared memory (double buffered by
      // tile parity, so one barrier per tile suffices), summed in part order
      float* rb = red + (i & 1) * (4 * 128);
      if (half > 0) rb[half * 128 + q * 32 + lane] = sum;
      consumer_sync(epi_warps * 32);
      if (half == 0 && !dead && key < p.n) {
        float tot = sum;
        for (int h2 = 1; h2 < epi_warps / 4; ++h2) tot += rb[h2 * 128 + q * 32 + lane];
        p.pooled[(size_t)u * p.n + key] = tot;
      }
    }
  }
  __syncthreads();
  if (warp == kEpiWarps + 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace

// Both passes of the scoring on the tensor cores, writing pooled [h_kv][n]
// (the caller smooths, selects and gathers). DV_ERR_UNSUPPORTED for shapes
// this form does not take (the caller then uses the CUDA-core kernels).
int launch_kv_scores_tc(const uint16_t* q_obs, const uint16_t* K, int h, int h_kv, int dh, int W,
                        int n, int n_max, float scale2, float* stats, size_t stats_floats,
                        float* pooled, int* st, cudaStream_t stream) {
  const int G = h / h_kv, NQ = G * W;
  if (!(dh == 64 || dh == 128) || NQ % 64 != 0 || NQ > 256 || n < 1 || W > n)
    return DV_ERR_UNSUPPORTED;
  KvTcParams p{};
  p.h_kv = h_kv;
  p.W = W;
  p.n = n;
  p.n_max = n_max;
  p.NQ = NQ;
  p.MT = (NQ + 127) / 128;
  p.KB = dh / 64;
  p.tiles = (n + kTcKeys - 1) / kTcKeys;
  p.tiles0 = (n + tc_keys<0>() - 1) / tc_keys<0>();
  const int per_head = std::max(1, sm_count() / h_kv);
  p.nsplit = std::max(1, std::min(p.tiles, per_head));
  p.scale2 = scale2;
  p.stats = stats;
  p.pooled = pooled;
  p.st = st;
  if ((size_t)h_kv * NQ * p.nsplit * 2 > stats_floats) return DV_ERR_WORKSPACE;
  CUtensorMap tmK, tmQ;
  if (!make_tmap_f16_sw128(&tmK, K, dh, (uint64_t)h_kv * n_max, dh, 128) ||
      !make_tmap_f16_sw128(&tmQ, q_obs, dh, (uint64_t)h * W, dh, 128))
    return DV_ERR_UNSUPPORTED;
  const KvTcSmem L = kvtc_layout(p.KB, p.MT);
  const size_t smem = L.total + 1024;  // + alignment of the dynamic base to 1024
  if (smem > 227 * 1024) return DV_ERR_UNSUPPORTED;
  if (cudaFuncSetAttribute(k_kvscore_tc<0>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)smem) != cudaSuccess ||
      cudaFuncSetAttribute(k_kvscore_tc<1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)smem) != cudaSuccess)
    return DV_ERR_LAUNCH;
  const dim3 grid(p.nsplit, h_kv);
  note_launch(DV_TAG_KVSEL, 0, stream);
  k_kvscore_tc<0><<<grid, kThreads, smem, stream>>>(tmK, tmQ, p);
  note_launch(DV_TAG_KVSEL, 1, stream);
  note_launch(DV_TAG_KVSEL, 0, stream);
  k_kvscore_tc<1><<<grid, kThreads, smem, stream>>>(tmK, tmQ, p);
  note_launch(DV_TAG_KVSEL, 1, stream);
  return cudaGetLastError() == cudaSuccess ? DV_OK : DV_ERR_LAUNCH;
}

}  // namespace dv
