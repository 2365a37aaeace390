// k_union_tc.cu -- the sparse MLP of a batch of 8..64 sequences over the union
// of their neuron sets, on the fifth-generation tensor cores (sm_103a).
//
// "Deja Vu: Contextual Sparsity for Efficient LLMs at Inference Time", §5.2
// and App. C.1: a batch computes every row over the union U of its sequences'
// sets, which turns the per-sequence gathers into one dense contraction:
//   H = relu(Z W1_U^T + b1_U)   (B x |U|),  Z = LN2(x) in fp16
//   out = x + H W2_U + b2       (B x d)
// fp16 operands (the 16-bit activations), fp32 accumulation in TMEM.
//
// Launches: LN2 of the B inputs (fp16 Z); the fc1 contraction; the fc2^T
// contraction; a fixed-order reduce of the fc2 partial sums (+ b2, + x).
//   fc1: D[128 union rows][Bp] += fc1[U rows][64-column slice] * Z[Bp][slice]^T.
//        The union rows are gathered by TMA (tile::gather4, four rows per
//        instruction, 128-byte swizzle), Z slices by tiled TMA loads. Work
//        units are (row tile, K range); the CTA that completes a row tile's
//        last K range sums the ranges' fp32 partials in range order, adds b1,
//        applies ReLU and writes H (fp16) -- deterministic.
//   fc2: D[128 output columns][Bp] += fc2T[U rows][128 columns]^T * H[Bp][rows]^T.
//        A is MN-major here (an fc2T row is contiguous along the output
//        columns): each gathered union row lands as 128-byte rows of
//        64-column blocks. Work units are (256-column tile, union-row range),
//        two M = 128 tiles that read 512 contiguous bytes of every row; each
//        writes an fp32 partial [range][B][d], summed in range order.
// Bp = max(B, 16) (the instruction shape with M = 128 takes N in steps of
// 16; rows B..Bp-1 of Z and H feed only columns of D that are never read).
// Eight producer warps issue the copies (one gather4 per lane), one thread
// issues tcgen05.mma, four warps read the accumulators back (tcgen05.ld).
#include <algorithm>

#include "dv_internal.h"
#include "dv_tc.cuh"
#include "k_union_tc.h"

namespace dv {

namespace {

// Ring stages: fc1 stages are 128 rows x 64 columns (16 KB); fc2 stages are
// 64 union rows x 256 output columns (32 KB), so that one unit reads 512
// contiguous bytes of each fc2^T row.
template <int PHASE> constexpr int u_stages() { return PHASE == 1 ? 8 : 4; }
template <int PHASE> constexpr int u_abytes() { return PHASE == 1 ? 128 * 128 : 64 * 512; }
constexpr int kUCols2 = 256;         // output columns of one fc2 unit (two M = 128 tiles)
// Warps: 0-3 epilogue, 4..4+kUProd-1 producers (each issues a quarter of a
// stage's copies: one warp issuing all of them sets the pace), then the MMA
// issuer and the index warp.
constexpr int kUProd = 8;
constexpr int kUMmaWarp = 4 + kUProd;
constexpr int kUIdxWarp = kUMmaWarp + 1;
constexpr int kUThreads = (kUIdxWarp + 1) * 32;
// gather4 copies per producer warp and stage: fc1 32 per stage, fc2 64
template <int PHASE> constexpr int u_ops_per_prod() { return (PHASE == 1 ? 32 : 64) / kUProd; }
constexpr int kUIdxMax = 4096;       // union indices one fc2 unit stages in shared memory
// Each K step of a stage accumulates into its own TMEM accumulator (kUChains
// independent chains, summed by the epilogue): with N = Bp as small as 16 one
// instruction's latency, not its work, would otherwise set the pace.
constexpr int kUChains = 2;
constexpr uint32_t kUTmemCols = 512; // 2 buffers x kUChains x (1 or 2 tiles) x Bp (<= 64) columns
constexpr int kUMaxStages = 8;

struct UnionTcParams {
  int B, Bp, d, F, k, kpad, ksplit1, ksplit2;
  const uint16_t* W;  // the phase's weight rows (fc1 or fc2T), [F][d]
  const int32_t* U;
  const int32_t* dev_count;
  const uint16_t* b1;
  uint16_t* H;    // [Bp][kpad]
  float* part1;   // [ceil(k/128)][ksplit1][Bp][128]
  int* cnt1;      // [ceil(k/128)]
  float* part2;   // [ksplit2][B][d]
  int* st;
};

struct USmem {
  uint32_t a, b, idx, bars, misc, total;
};

template <int PHASE>
__host__ __device__ inline USmem u_layout(int Bp) {
  USmem L{};
  L.a = 0;
  L.b = L.a + u_stages<PHASE>() * u_abytes<PHASE>();
  L.idx = L.b + u_stages<PHASE>() * Bp * 128;
  L.bars = L.idx + 2 * kUIdxMax * 4;  // two index buffers: the next unit's fill ahead
  L.misc = L.bars + 256;
  L.total = L.misc + 64;
  return L;
}

DV_DEV int union_count(const UnionTcParams& p) {
  int kk = p.k;
  if (p.dev_count) {
    const int c = *p.dev_count;
    kk = c < kk ? (c < 0 ? 0 : c) : kk;
  }
  return kk;
}

// A union index as a row coordinate. Positions past the union's end and
// entries that are not rows of the matrix (reported) read row 0 instead: the
// fc1 epilogue writes H = 0 for them, so they add nothing in either phase,
// and no copy addresses a row outside the matrix.
DV_DEV int row_of(const UnionTcParams& p, int j, int kk, bool& bad) {
  if (j >= kk) return 0;
  const int r = p.U[j];
  if (r < 0 || r >= p.F) {
    bad = true;
    return 0;
  }
  return r;
}

// TMEM -> registers: Bp (16, 32 or 64) columns of this thread's lane.
DV_DEV void tmem_ld_row(uint32_t taddr, int Bp, float* v) {
  if (Bp == 16) {
    tmem_ld16(taddr, v);
  } else {
    tmem_ld32(taddr, v);
    if (Bp == 64) tmem_ld32(taddr + 32, v + 32);
  }
}

template <int PHASE, int BP>
__global__ void __launch_bounds__(kUThreads, 1)
    k_union_mlp_tc(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
                   const UnionTcParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~uintptr_t(1023));
  constexpr int kUStages = u_stages<PHASE>();
  constexpr int kABytes = u_abytes<PHASE>();
  constexpr int kUOpsPerProd = u_ops_per_prod<PHASE>();
  constexpr int NT = PHASE == 1 ? 1 : 2;  // M = 128 tiles of one unit
  const USmem L = u_layout<PHASE>(BP);
  uint8_t* sA = sm + L.a;
  uint8_t* sB = sm + L.b;
  int* sidx = reinterpret_cast<int*>(sm + L.idx);
  uint64_t* full = reinterpret_cast<uint64_t*>(sm + L.bars);
  uint64_t* empty = full + kUStages;
  uint64_t* accf = empty + kUStages;
  uint64_t* acce = accf + 2;
  uint64_t* ifull = acce + 2;   // index buffer b holds the next unit's rows
  uint64_t* iempty = ifull + 2; // the producer is done with index buffer b
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + L.misc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + L.misc + 4);
  volatile int* last_flag = reinterpret_cast<volatile int*>(sm + L.misc + 8);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  constexpr uint32_t bBytes = BP * 128;

  if (tid == 0) {
    for (int s = 0; s < kUStages; ++s) {
      mbar_init(&full[s], kUProd);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&accf[a], 1);
      mbar_init(&acce[a], 4);
      mbar_init(&ifull[a], 1);
      mbar_init(&iempty[a], kUProd);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kUMmaWarp) {
    tmem_alloc(tmem_slot, kUTmemCols);
    tc_fence_before();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // The index list and Z / H come from the kernels before this one.
  pdl_wait();
  if (tid == 0) pdl_launch_dependents();

  const int kk = union_count(p);
  // units: fc1 (row tile, K range); fc2 (256-column tile, union-row range)
  const int KB = (p.d + 63) / 64;  // 64-column slices of d
  const int ntile = PHASE == 1 ? (kk + 127) / 128 : (p.d + kUCols2 - 1) / kUCols2;
  const int ksplit = PHASE == 1 ? p.ksplit1 : p.ksplit2;
  const int JS = (kk + 63) / 64;   // 64-row stages of the union (fc2)
  const int nunits = ntile * ksplit;
  // fc1 numbers a row tile's K ranges consecutively (the CTAs of one tile run
  // together and the last of them sums the ranges); fc2 numbers the column
  // tiles of one union-row range consecutively, so that CTAs running at the
  // same time read neighbouring 512-byte pieces of the same weight rows.
  auto unit_tile = [&](int u) { return PHASE == 1 ? u / ksplit : u % ntile; };
  auto unit_part = [&](int u) { return PHASE == 1 ? u % ksplit : u / ntile; };
  auto stage_range = [&](int part, int& s0, int& s1) {
    const int tot = PHASE == 1 ? KB : JS;
    s0 = (int)((long long)tot * part / ksplit);
    s1 = (int)((long long)tot * (part + 1) / ksplit);
  };
  auto give_up = [&]() {
    *abort_flag = 1;
    flag(p.st, DV_DEV_TIMEOUT);
  };

  if (warp == kUIdxWarp) {
    // ---------------- index warp: each unit's union rows, one unit ahead -------
    bool bad = false;
    int n = 0;
    for (int u = blockIdx.x; u < nunits && !*abort_flag; u += gridDim.x, ++n) {
      const int buf = n & 1;
      int go = 1;
      if (lane == 0 && n >= 2 && !mbar_wait(&iempty[buf], ((n >> 1) & 1) ^ 1)) {
        give_up();
        go = 0;
      }
      if (!__shfl_sync(0xffffffffu, go, 0)) break;
      __syncwarp();  // lane 0's wait orders the producer's reads before these writes
      int s0, s1;
      stage_range(unit_part(u), s0, s1);
      const int j0 = PHASE == 1 ? unit_tile(u) * 128 : s0 * 64;
      const int nj = PHASE == 1 ? 128 : (s1 - s0) * 64;
      int* dst = sidx + buf * kUIdxMax;
      for (int i0 = 0; i0 < nj; i0 += 32 * 16) {
        int v[16];
#pragma unroll
        for (int r = 0; r < 16; ++r) {
          const int i = i0 + r * 32 + lane;
          v[r] = i < nj ? row_of(p, j0 + i, kk, bad) : 0;
        }
#pragma unroll
        for (int r = 0; r < 16; ++r) {
          const int i = i0 + r * 32 + lane;
          if (i < nj) dst[i] = v[r];
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&ifull[buf]);
    }
    if (__any_sync(0xffffffffu, bad) && lane == 0) flag(p.st, DV_DEV_BAD_INDEX);
    __syncwarp();
  } else if (warp >= 4 && warp < 4 + kUProd) {
    // ---------------- producers: copies o = pw*8 .. pw*8+7 of every stage ------
    const int pw = warp - 4;
    const int o = pw * kUOpsPerProd + lane;  // this lane's gather4 (lanes < 8)
    const uint32_t my_tx = kUOpsPerProd * 512 + (pw == 0 ? bBytes : 0);
    int it = 0, n = 0;
    if (lane == 0 && pw == 0) {
      tma_prefetch_map(&tmW);
      tma_prefetch_map(&tmX);
    }
    for (int u = blockIdx.x; u < nunits && !*abort_flag; u += gridDim.x, ++n) {
      const int tile = unit_tile(u), part = unit_part(u);
      int s0, s1;
      stage_range(part, s0, s1);
      const int buf = n & 1;
      int ready = 1;
      if (lane == 0 && !mbar_wait(&ifull[buf], (n >> 1) & 1)) {
        give_up();
        ready = 0;
      }
      if (!__shfl_sync(0xffffffffu, ready, 0)) break;
      __syncwarp();  // lane 0's wait orders the index warp's writes before these reads
      const int* sidx_u = sidx + buf * kUIdxMax;
      for (int sI = s0; sI < s1; ++sI, ++it) {
        const int s = it % kUStages;
        int go = 1;
        if (lane == 0) {
          if (*abort_flag) {
            go = 0;
          } else if (it >= kUStages && !mbar_wait(&empty[s], ((it / kUStages) & 1) ^ 1)) {
            give_up();
            go = 0;
          }
          if (go) mbar_arrive_expect_tx(&full[s], my_tx);
        }
        if (!__shfl_sync(0xffffffffu, go, 0)) break;
        uint8_t* a = sA + s * kABytes;
        if (lane < kUOpsPerProd) {
          if (PHASE == 1) {
            // rows 4 o .. 4 o + 3 of the tile, columns sI*64 .. +63
            const int* r = sidx_u + 4 * o;
            tma_gather4(a + o * 512, &tmW, sI * 64, r[0], r[1], r[2], r[3], &full[s]);
          } else {
            // union rows (sI - s0)*64 + 4 (o % 16) .. +3, output-column block
            // o / 16 (64 columns; four blocks per unit)
            const int mb = o >> 4, r4 = (o & 15) * 4;
            const int* r = sidx_u + (sI - s0) * 64 + r4;
            tma_gather4(a + mb * 8192 + r4 * 128, &tmW, tile * kUCols2 + mb * 64, r[0], r[1],
                        r[2], r[3], &full[s]);
          }
        }
        if (lane == 0 && pw == 0) tma_load_2d(sB + s * bBytes, &tmX, sI * 64, 0, &full[s]);
        __syncwarp();
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&iempty[buf]);  // this warp's copies of the unit are issued
    }
    if (lane == 0)  // every issued copy lands before the CTA exits
      for (int j = (it > kUStages ? it - kUStages : 0); j < it; ++j)
        if (!mbar_wait(&full[j % kUStages], (j / kUStages) & 1)) flag(p.st, DV_DEV_TIMEOUT);
    __syncwarp();
  } else if (warp == kUMmaWarp) {
    // ---------------- MMA issuer (one thread) ---------------------------------
    if (lane == 0) {
      const uint32_t a0 = smem_addr(sA), b0 = smem_addr(sB);
      const uint32_t idesc = idesc_f16_f32(128, BP, PHASE == 2);
      int it = 0, nu = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < nunits && ok && !*abort_flag; u += gridDim.x) {
        int s0, s1;
        stage_range(unit_part(u), s0, s1);
        if (s1 == s0) continue;
        const int a = nu & 1;
        if (nu >= 2 && !mbar_wait(&acce[a], ((nu >> 1) & 1) ^ 1)) {
          give_up();
          break;
        }
        for (int sI = s0; sI < s1; ++sI, ++it) {
          const int s = it % kUStages;
          if (*abort_flag || !mbar_wait(&full[s], (it / kUStages) & 1)) {
            give_up();
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll
          for (int t = 0; t < NT; ++t)
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) {
              // fc1: A K-major (16 columns = 32 bytes per step); fc2: A MN-major
              // (16 union rows = 2048 bytes per step, column blocks 8 KB apart,
              // tile t at blocks 2t and 2t + 1)
              const uint64_t ad =
                  PHASE == 1 ? sdesc_k128(a0 + s * kABytes + ks * 32)
                             : sdesc_sw128(a0 + s * kABytes + t * 16384 + ks * 2048, 8192, 1024);
              tc_mma_f16(tmem + ((a * NT + t) * kUChains + ks % kUChains) * BP, ad,
                         sdesc_k128(b0 + s * bBytes + ks * 32), idesc, sI > s0 || ks >= kUChains);
            }
          tc_commit(&empty[s]);
        }
        if (!ok) break;
        tc_commit(&accf[a]);
        ++nu;
      }
    }
    __syncwarp();
  } else {
    // ---------------- epilogue: 4 warps, thread = TMEM lane = row / column ----
    const int row = warp * 32 + lane;
    const uint32_t tl = tmem + ((uint32_t)(warp * 32) << 16);
    int nu = 0;
    bool dead = false;
    for (int u = blockIdx.x; u < nunits; u += gridDim.x) {
      const int tile = unit_tile(u), part = unit_part(u);
      int s0, s1;
      stage_range(part, s0, s1);
      if constexpr (PHASE == 2) {
        // partial sums of this union-row range for the unit's 256 output
        // columns (zeros for an empty range: the reduce adds every range)
        const bool have = s1 > s0;
        const int a = nu & 1;
        if (have && !dead && (*abort_flag || !mbar_wait(&accf[a], (nu >> 1) & 1))) {
          give_up();
          dead = true;
        }
        if (have && !dead) tc_fence_after();
        // sequences in pieces of at most 32 columns (BP = 64 would otherwise
        // hold 2 x 64 accumulators per thread at once)
        constexpr int PC = BP < 32 ? BP : 32;
#pragma unroll 1
        for (int t = 0; t < NT; ++t) {
          const int c = tile * kUCols2 + t * 128 + row;
#pragma unroll 1
          for (int b0 = 0; b0 < BP; b0 += PC) {
            float v[PC];
#pragma unroll
            for (int b = 0; b < PC; ++b) v[b] = 0.f;
            if (have && !dead) {
              const uint32_t base = tl + (a * NT + t) * kUChains * BP + b0;
              tmem_ld_row(base, PC, v);
#pragma unroll
              for (int ch = 1; ch < kUChains; ++ch) {
                float w[PC];
                tmem_ld_row(base + ch * BP, PC, w);
#pragma unroll
                for (int b = 0; b < PC; ++b) v[b] += w[b];
              }
            }
            if (c < p.d && !dead)
#pragma unroll
              for (int b = 0; b < PC; ++b)
                if (b0 + b < p.B) p.part2[((size_t)part * p.B + b0 + b) * p.d + c] = v[b];
          }
        }
        if (have && !dead) {
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&acce[a]);
        }
        if (have) ++nu;
        continue;
      }
      float v[BP];
#pragma unroll
      for (int b = 0; b < BP; ++b) v[b] = 0.f;
      if (s1 > s0) {
        const int a = nu & 1;
        if (!dead && (*abort_flag || !mbar_wait(&accf[a], (nu >> 1) & 1))) {
          give_up();
          dead = true;
        }
        if (!dead) {
          tc_fence_after();
          tmem_ld_row(tl + a * kUChains * BP, BP, v);
#pragma unroll
          for (int c = 1; c < kUChains; ++c) {
            float w[BP];
            tmem_ld_row(tl + (a * kUChains + c) * BP, BP, w);
#pragma unroll
            for (int b = 0; b < BP; ++b) v[b] += w[b];
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&acce[a]);
        }
        ++nu;
      }
      // fc1: partial sums of this K range, or the whole dot product
      const int j = tile * 128 + row;
      bool last = true;
      if (ksplit > 1) {
        float* my = p.part1 + ((size_t)(tile * ksplit + part) * BP) * 128 + row;
        if (!dead)
#pragma unroll
          for (int b = 0; b < BP; ++b) my[b * 128] = v[b];
        __threadfence();
        consumer_sync(128);
        if (row == 0) *last_flag = (atomicAdd(&p.cnt1[tile], 1) == ksplit - 1);
        consumer_sync(128);
        last = *last_flag;
        if (last) {
          __threadfence();
#pragma unroll
          for (int b = 0; b < BP; ++b) v[b] = 0.f;
          for (int q = 0; q < ksplit; ++q) {
            const float* src = p.part1 + ((size_t)(tile * ksplit + q) * BP) * 128 + row;
#pragma unroll
            for (int b = 0; b < BP; ++b) v[b] += __ldcg(src + b * 128);
          }
          if (row == 0) p.cnt1[tile] = 0;  // ready for the next call
        }
      }
      if (last && !dead) {
        float bias = 0.f;
        const bool on = j < kk && p.U[j] >= 0 && p.U[j] < p.F;
        if (on && p.b1) bias = h2f(p.b1[p.U[j]]);
#pragma unroll
        for (int b = 0; b < BP; ++b)
          p.H[(size_t)b * p.kpad + j] = on ? f2h(fmaxf(v[b] + bias, 0.f)) : (uint16_t)0;
      }
    }
  }
  __syncthreads();
  if (warp == kUMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, kUTmemCols);
  }
}

// Z[b] = fp16(LN2(x[b])): one CTA per sequence, two passes in fp32 over
// 8-column vectors (d is a multiple of 64). CTA 0 also clears the fc1
// tile counters (the fc1 launch that follows counts on them).
constexpr int kULnThreads = 512;

__global__ void __launch_bounds__(kULnThreads) k_union_ln(const uint16_t* __restrict__ x, int d,
                                                         const uint16_t* __restrict__ g,
                                                         const uint16_t* __restrict__ bb,
                                                         float eps, uint16_t* __restrict__ Z,
                                                         int* __restrict__ cnt1, int ncnt) {
  __shared__ float red[kULnThreads / 32];
  __shared__ float stat[2];
  pdl_wait();
  if (threadIdx.x == 0) pdl_launch_dependents();
  const int b = blockIdx.x, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  constexpr int nw = kULnThreads / 32;
  if (b == 0)
    for (int i = threadIdx.x; i < ncnt; i += kULnThreads) cnt1[i] = 0;
  const uint16_t* xr = x + (size_t)b * d;
  const int nv = d / 8;
  float s = 0.f;
  for (int v = threadIdx.x; v < nv; v += kULnThreads) {
    float f[8];
    h8_to_f8(*reinterpret_cast<const uint4*>(xr + v * 8), f);
#pragma unroll
    for (int e = 0; e < 8; ++e) s += f[e];
  }
  s = warp_sum(s);
  if (lane == 0) red[warp] = s;
  __syncthreads();
  if (threadIdx.x == 0) {
    float t = 0.f;
    for (int w = 0; w < nw; ++w) t += red[w];
    stat[0] = t / d;
  }
  __syncthreads();
  const float mu = stat[0];
  float q = 0.f;
  for (int v = threadIdx.x; v < nv; v += kULnThreads) {
    float f[8];
    h8_to_f8(*reinterpret_cast<const uint4*>(xr + v * 8), f);
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const float c = f[e] - mu;
      q = fmaf(c, c, q);
    }
  }
  q = warp_sum(q);
  __syncthreads();
  if (lane == 0) red[warp] = q;
  __syncthreads();
  if (threadIdx.x == 0) {
    float t = 0.f;
    for (int w = 0; w < nw; ++w) t += red[w];
    stat[1] = 1.0f / sqrtf(t / d + eps);
  }
  __syncthreads();
  const float inv = stat[1];
  for (int v = threadIdx.x; v < nv; v += kULnThreads) {
    float f[8], gg[8], be[8];
    h8_to_f8(*reinterpret_cast<const uint4*>(xr + v * 8), f);
    if (g) {
      h8_to_f8(*reinterpret_cast<const uint4*>(g + v * 8), gg);
    } else {
#pragma unroll
      for (int e = 0; e < 8; ++e) gg[e] = 1.f;
    }
    if (bb) {
      h8_to_f8(*reinterpret_cast<const uint4*>(bb + v * 8), be);
    } else {
#pragma unroll
      for (int e = 0; e < 8; ++e) be[e] = 0.f;
    }
    uint16_t o[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) o[e] = f2h((f[e] - mu) * inv * gg[e] + be[e]);
    uint4 pk;
    pk.x = (uint32_t)o[0] | ((uint32_t)o[1] << 16);
    pk.y = (uint32_t)o[2] | ((uint32_t)o[3] << 16);
    pk.z = (uint32_t)o[4] | ((uint32_t)o[5] << 16);
    pk.w = (uint32_t)o[6] | ((uint32_t)o[7] << 16);
    *reinterpret_cast<uint4*>(Z + (size_t)b * d + v * 8) = pk;
  }
}

// out[b] = fp16(x[b] + (sum_g part2[g][b] + b2)), the fc2 union-row ranges
// summed in range order: one thread per (sequence, 4 columns), eight
// partials' loads in flight.
__global__ void __launch_bounds__(256) k_union_reduce(const float* __restrict__ part, int G, int B,
                                                     int d, const uint16_t* __restrict__ x,
                                                     const uint16_t* __restrict__ bias,
                                                     uint16_t* __restrict__ out) {
  pdl_wait();
  if (threadIdx.x == 0) pdl_launch_dependents();
  const int n4 = d / 4;
  const long long i = (long long)blockIdx.x * 256 + threadIdx.x;
  if (i >= (long long)B * n4) return;
  const int b = (int)(i / n4), c4 = (int)(i % n4);
  const size_t stride = (size_t)B * d;
  const float* src = part + (size_t)b * d + c4 * 4;
  float4 s = make_float4(0.f, 0.f, 0.f, 0.f);
  int g0 = 0;
  for (; g0 + 8 <= G; g0 += 8) {
    float4 t[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) t[j] = __ldcg(reinterpret_cast<const float4*>(src + (g0 + j) * stride));
#pragma unroll
    for (int j = 0; j < 8; ++j) { s.x += t[j].x; s.y += t[j].y; s.z += t[j].z; s.w += t[j].w; }
  }
  for (; g0 < G; ++g0) {
    const float4 t = __ldcg(reinterpret_cast<const float4*>(src + g0 * stride));
    s.x += t.x; s.y += t.y; s.z += t.z; s.w += t.w;
  }
  const float r[4] = {s.x, s.y, s.z, s.w};
  const uint16_t* xr = x ? x + (size_t)b * d + c4 * 4 : nullptr;
  uint16_t o[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const float bv = bias ? h2f(bias[c4 * 4 + e]) : 0.f;
    o[e] = f2h((xr ? h2f(xr[e]) : 0.f) + (r[e] + bv));
  }
  uint2 pk;
  pk.x = (uint32_t)o[0] | ((uint32_t)o[1] << 16);
  pk.y = (uint32_t)o[2] | ((uint32_t)o[3] << 16);
  *reinterpret_cast<uint2*>(out + (size_t)b * d + c4 * 4) = pk;
}

// Host-side plan of one call (shared by the workspace size and the launch).
struct UnionPlan {
  int Bp, kpad, ntile1, ksplit1, ksplit2;
  size_t off_z, off_h, off_p1, off_cnt, off_p2, total;
};

size_t al256(size_t x) { return (x + 255) / 256 * 256; }

UnionPlan union_plan(int B, int d, int k) {
  UnionPlan P{};
  const int sms = sm_count();
  P.Bp = B < 16 ? 16 : B;
  P.ntile1 = (k + 127) / 128;
  P.kpad = P.ntile1 * 128;
  const int KB = (d + 63) / 64;
  // about eight units per SM in each phase (balance: the units of a phase
  // are equal, so a CTA's share differs by at most one), at least four
  // K slices per fc1 unit, and a union-row range per fc2 unit that fits its
  // index stage
  P.ksplit1 = std::max(1, std::min((8 * sms + P.ntile1 - 1) / P.ntile1, std::max(1, KB / 4)));
  const int nct = (d + kUCols2 - 1) / kUCols2, JS = (k + 63) / 64;
  const int need = (JS * 64 + kUIdxMax - 1) / kUIdxMax;
  P.ksplit2 = std::max(need, std::min((8 * sms + nct - 1) / nct, JS));
  P.ksplit2 = std::max(1, P.ksplit2);
  size_t off = 0;
  P.off_z = off;
  off += al256((size_t)P.Bp * d * 2);
  P.off_h = off;
  off += al256((size_t)P.Bp * P.kpad * 2);
  P.off_p1 = off;
  off += al256((size_t)P.ntile1 * P.ksplit1 * P.Bp * 128 * 4);
  P.off_cnt = off;
  off += al256((size_t)P.ntile1 * 4);
  P.off_p2 = off;
  off += al256((size_t)P.ksplit2 * B * d * 4);
  P.total = off;
  return P;
}

}  // namespace

size_t union_tc_ws_bytes(int B, int d, int k) { return union_plan(B, d, k).total; }

int launch_union_mlp_tc(const uint16_t* x, int B, int d, int F, const uint16_t* ln_g,
                        const uint16_t* ln_b, float eps, const uint16_t* fc1, const uint16_t* b1,
                        const uint16_t* fc2T, const uint16_t* b2, const int32_t* U, int k,
                        const int32_t* dev_count, bool resid, uint16_t* out, int* st, void* ws,
                        cudaStream_t s) {
  const UnionPlan P = union_plan(B, d, k);
  uint8_t* w = static_cast<uint8_t*>(ws);
  uint16_t* Z = reinterpret_cast<uint16_t*>(w + P.off_z);
  UnionTcParams p{};
  p.B = B;
  p.Bp = P.Bp;
  p.d = d;
  p.F = F;
  p.k = k;
  p.kpad = P.kpad;
  p.ksplit1 = P.ksplit1;
  p.ksplit2 = P.ksplit2;
  p.U = U;
  p.dev_count = dev_count;
  p.b1 = b1;
  p.H = reinterpret_cast<uint16_t*>(w + P.off_h);
  p.part1 = reinterpret_cast<float*>(w + P.off_p1);
  p.cnt1 = reinterpret_cast<int*>(w + P.off_cnt);
  p.part2 = reinterpret_cast<float*>(w + P.off_p2);
  p.st = st;
  CUtensorMap tW1, tZ, tW2, tH;
  if (!make_tmap_f16_sw128(&tW1, fc1, d, F, d, 1) || !make_tmap_f16_sw128(&tZ, Z, d, P.Bp, d, P.Bp) ||
      !make_tmap_f16_sw128(&tW2, fc2T, d, F, d, 1) ||
      !make_tmap_f16_sw128(&tH, p.H, P.kpad, P.Bp, P.kpad, P.Bp))
    return DV_ERR_UNSUPPORTED;
  const size_t smem = std::max(u_layout<1>(P.Bp).total, u_layout<2>(P.Bp).total) + 1024;
  const void* k1 = P.Bp == 16 ? (const void*)k_union_mlp_tc<1, 16>
                 : P.Bp == 32 ? (const void*)k_union_mlp_tc<1, 32> : (const void*)k_union_mlp_tc<1, 64>;
  const void* k2 = P.Bp == 16 ? (const void*)k_union_mlp_tc<2, 16>
                 : P.Bp == 32 ? (const void*)k_union_mlp_tc<2, 32> : (const void*)k_union_mlp_tc<2, 64>;
  if (cudaFuncSetAttribute(k1, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
          cudaSuccess ||
      cudaFuncSetAttribute(k2, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
          cudaSuccess)
    return DV_ERR_LAUNCH;
  note_launch(DV_TAG_MLP, 0, s);
  k_union_ln<<<B, kULnThreads, 0, s>>>(x, d, ln_g, ln_b, eps, Z, p.cnt1, P.ntile1);
  note_launch(DV_TAG_MLP, 1, s);
  if (cudaGetLastError() != cudaSuccess) return DV_ERR_LAUNCH;
  const int grid = sm_count();
  {
    p.W = fc1;
    void* args[] = {&tW1, &tZ, &p};
    note_launch(DV_TAG_MLP, 0, s);
    const cudaError_t e = launch_k(k1, dim3(grid), dim3(kUThreads), smem, s, args, true);
    note_launch(DV_TAG_MLP, 1, s);
    if (e != cudaSuccess) return DV_ERR_LAUNCH;
  }
  {
    p.W = fc2T;
    void* args[] = {&tW2, &tH, &p};
    note_launch(DV_TAG_MLP, 0, s);
    const cudaError_t e = launch_k(k2, dim3(grid), dim3(kUThreads), smem, s, args, true);
    note_launch(DV_TAG_MLP, 1, s);
    if (e != cudaSuccess) return DV_ERR_LAUNCH;
  }
  {
    const float* part = p.part2;
    int G = P.ksplit2, Bv = B, dv_ = d;
    const uint16_t* xres = resid ? x : nullptr;
    void* args[] = {&part, &G, &Bv, &dv_, &xres, &b2, &out};
    const long long n = (long long)B * (d / 4);
    note_launch(DV_TAG_REDUCE, 0, s);
    const cudaError_t e = launch_k((const void*)k_union_reduce, dim3((unsigned)((n + 255) / 256)),
                                   dim3(256), 0, s, args, true);
    note_launch(DV_TAG_REDUCE, 1, s);
    if (e != cudaSuccess) return DV_ERR_LAUNCH;
  }
  return DV_OK;
}

}  // namespace dv
