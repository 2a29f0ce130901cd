// ts_lm_head_argmax / ts_tree_accept_hidden: the target LM head's per-row argmax computed in
// the epilogue of the LM-head GEMM, so the [rows, V] logits never reach HBM.
//
// Source: "jialefu.github.io — EAGLE-4 efficient LM head", section "A variant based on local
// Top-k" (fuse the selection with the vocabulary-tile matrix multiplication and keep the
// scores on chip; each tile keeps only its local winners and the tiles' winners are merged).
// For top-1 the merge is exact: the row maximum is the maximum of the tiles' maxima, and the
// lowest index among equal values survives when each tile reports its first maximum and the
// merge breaks ties by index.  The greedy check that consumes it: "lesty.tech — EAGLE-2 vs.
// Medusa", section 4.
//
// logits[r, n] = sum_k hidden[r, k] * weight[n, k] (bf16 inputs, fp32 accumulation on the
// tensor cores).  CTA (mt, g) owns rows [128 mt, 128 mt + 128) and the vocabulary tiles
// [g * tpg, (g + 1) * tpg) of 256 columns; it leaves one (max, first index) per row.
//
// Warp roles (192 threads):
//   warp 0      TMA producer: per (tile, 64-wide K chunk) one 128x64 box of hidden and one
//               256x64 box of weight (128-byte swizzle) into a 4-stage ring; rows past M or N
//               and columns past K read zeros.
//   warp 1      TMEM allocator + the MMA-issuing thread: tcgen05.mma kind::f16, M=128, N=256,
//               four K=16 steps per chunk, into one of two 256-column accumulators, so the
//               next tile's MMAs run while the previous tile's epilogue reads its accumulator.
//   warps 2..5  epilogue, one thread per row (warp w reads TMEM lanes 32 (w % 4) ..): running
//               maximum over the tile's columns in increasing order (strict > keeps the first
//               index), columns past N skipped.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <climits>
#include <cmath>
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace ts {
namespace lm {

constexpr int BM = 128, BN = 256, BK = 64;
constexpr int STAGES = 4;
constexpr uint32_t A_BYTES = BM * BK * 2;   // 16 KB
constexpr uint32_t B_BYTES = BN * BK * 2;   // 32 KB
constexpr uint32_t STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int THREADS = 192;
constexpr uint32_t TMEM_COLS = 2 * BN;      // two accumulators
constexpr uint32_t OFF_BAR = STAGES * STAGE_BYTES;
// full[ST] empty[ST] acc_full[2] acc_empty[2] drain
constexpr int NBAR = 2 * STAGES + 5;
constexpr uint32_t OFF_MISC = OFF_BAR + NBAR * 8;
constexpr uint32_t SMEM_BYTES = OFF_MISC + 16 + 1024;  // + alignment slack

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const void* tmap, uint32_t bar, int c0, int c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(c0), "r"(c1), "r"(bar)
      : "memory");
}

// Wait bounded by time only (the abort path: let in-flight copies and MMAs land).
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try(bar, parity)) {
    if (global_timer_ns() - t0 > kWaitLimitNs) return;
  }
}

// Sorted (value descending) list of KL entries in registers: insert (cv, ci) without branches.
// The new list is computed from the old one: entry e becomes cv where cv is better than the old
// entry e but not than entry e-1, the old entry e-1 where cv is better than both, else stays.
// `full` compares (value, then lower index); without it a strict value compare is enough,
// because a list fed columns in increasing order keeps the earlier of equal values.
template <int KL, bool full>
__device__ __forceinline__ void list_insert(float (&v)[KL], int (&id)[KL], float cv, int ci) {
#pragma unroll
  for (int e = KL - 1; e >= 0; --e) {
    const bool gt = full ? (cv > v[e] || (cv == v[e] && ci < id[e])) : cv > v[e];
    bool gtp = false;
    if (e > 0) gtp = full ? (cv > v[e - 1] || (cv == v[e - 1] && ci < id[e - 1])) : cv > v[e - 1];
    const float nv = gtp ? v[e > 0 ? e - 1 : 0] : cv;
    const int ni = gtp ? id[e > 0 ? e - 1 : 0] : ci;
    v[e] = gt ? nv : v[e];
    id[e] = gt ? ni : id[e];
  }
}

// KT == 0: running (max, first index) over the CTA's columns -> part_v / part_i [M, S].
// KT >= 1: a vocabulary tile is vt consecutive 256-column tiles, split into vs parts of pt = vt/vs
// tiles; for every part, the KT best columns (value descending, ties -> lower index) with their
// values -> plv / pli [M, NV, vs, KT] (index INT_MAX where a part has fewer columns).  The CTA's
// tile range starts on a part boundary; gather_logits_kernel merges the parts of a tile.
template <int KT>
__global__ void __launch_bounds__(THREADS, 1)
    lm_head_kernel(const __grid_constant__ CUtensorMap tma_h, const __grid_constant__ CUtensorMap tma_w,
                   int M, int N, int K, int tpg, float* __restrict__ part_v, int* __restrict__ part_i,
                   int S, int vt, int pt, int vs, float* __restrict__ plv, int* __restrict__ pli, int32_t* status) {
  extern __shared__ unsigned char smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  unsigned char* sptr = smem_raw + (sbase - raw);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int mt = blockIdx.x, g = blockIdx.y;
  const int NT = (N + BN - 1) / BN;
  const int tile0 = g * tpg;
  const int ntile = max(0, min(NT, tile0 + tpg) - tile0);
  const int KC = (K + BK - 1) / BK;

  auto bar = [&](int i) -> uint32_t { return sbase + OFF_BAR + 8u * i; };
  auto full = [&](int s) { return bar(s); };
  auto empty = [&](int s) { return bar(STAGES + s); };
  auto acc_full = [&](int b) { return bar(2 * STAGES + b); };
  auto acc_empty = [&](int b) { return bar(2 * STAGES + 2 + b); };
  const uint32_t drain = bar(2 * STAGES + 4);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sptr + OFF_MISC);
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(sptr + OFF_MISC + 4);

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full(s), 1);
      mbar_init(empty(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(acc_full(b), 1);
      mbar_init(acc_empty(b), 4);  // one arrival per epilogue warp
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  pdl_wait();
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_holder), TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;

  if (warp == 0) {
    // ------------------------------ TMA producer ------------------------------
    if (lane == 0) {
      int issued = 0;
      for (int i = 0; i < ntile; ++i) {
        const int n0 = (tile0 + i) * BN;
        for (int kc = 0; kc < KC; ++kc) {
          const int it = i * KC + kc, s = it % STAGES;
          if (it >= STAGES && !mbar_wait(empty(s), ((it / STAGES) & 1) ^ 1, abort_flag, status)) break;
          mbar_expect_tx(full(s), STAGE_BYTES);
          const uint32_t dst = sbase + s * STAGE_BYTES;
          tma_load_2d(dst, &tma_h, full(s), kc * BK, mt * BM);
          tma_load_2d(dst + A_BYTES, &tma_w, full(s), kc * BK, n0);
          issued = it + 1;
        }
        if (*abort_flag) break;
      }
      if (*abort_flag) {
        for (int it = max(0, issued - STAGES); it < issued; ++it) drain_wait(full(it % STAGES), (it / STAGES) & 1);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------ MMA issuer ------------------------------
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(BM, BN, 0, 0);
      bool ok = true;
      for (int i = 0; i < ntile && ok; ++i) {
        const int ab = i & 1;
        if (i >= 2 && !mbar_wait(acc_empty(ab), ((i >> 1) - 1) & 1, abort_flag, status)) break;
        tc_fence_after();
        const uint32_t d = tmem + ab * BN;
        for (int kc = 0; kc < KC; ++kc) {
          const int it = i * KC + kc, s = it % STAGES;
          if (!mbar_wait(full(s), (it / STAGES) & 1, abort_flag, status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_s = sbase + s * STAGE_BYTES, b_s = a_s + A_BYTES;
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk) {
            const uint64_t ad = sdesc_sw128(a_s + kk * 32, 16, 1024);
            const uint64_t bd = sdesc_sw128(b_s + kk * 32, 16, 1024);
            mma_ss(d, ad, bd, idesc, (kc | kk) != 0 ? 1u : 0u);
          }
          tc_commit(empty(s));
        }
        if (!ok) break;
        tc_commit(acc_full(ab));
      }
      if (*abort_flag) {
        // one more commit covers every MMA issued so far: TMEM is released only after them
        tc_commit(drain);
        drain_wait(drain, 0);
      }
    }
    __syncwarp();
  } else {
    // ------------------------------ epilogue ------------------------------
    const int q = warp & 3;                 // TMEM lane quarter of this warp
    const int r = q * 32 + lane;            // row within the tile
    const uint32_t lane_off = static_cast<uint32_t>(q * 32) << 16;
    constexpr int KL = KT > 0 ? KT : 1;
    float lv[KL];
    int li[KL];
#pragma unroll
    for (int e = 0; e < KL; ++e) {
      lv[e] = -INFINITY;
      li[e] = INT_MAX;
    }
    // KT >= 1: a second list takes the odd columns (two independent dependency chains, no
    // branches); the two are merged when a part ends
    float ov[KL];
    int oi[KL];
#pragma unroll
    for (int e = 0; e < KL; ++e) {
      ov[e] = -INFINITY;
      oi[e] = INT_MAX;
    }
    const int row = mt * BM + r;
    for (int i = 0; i < ntile; ++i) {
      const int ab = i & 1;
      if (!mbar_wait_warp(acc_full(ab), (i >> 1) & 1, abort_flag, status)) break;
      tc_fence_after();
      const int n0 = (tile0 + i) * BN;
#pragma unroll 1
      for (int c = 0; c < BN / 32; ++c) {
        uint32_t u[32];
        tmem_ld32(tmem + lane_off + ab * BN + 32u * c, u);
        const int nb = n0 + 32 * c;
        if constexpr (KT > 0) {
#pragma unroll
          for (int j = 0; j < 32; j += 2) {
            list_insert<KL, false>(lv, li, nb + j < N ? __uint_as_float(u[j]) : -INFINITY, nb + j);
            list_insert<KL, false>(ov, oi, nb + j + 1 < N ? __uint_as_float(u[j + 1]) : -INFINITY, nb + j + 1);
          }
        } else {
#pragma unroll
          for (int j = 0; j < 32; ++j) {  // the running maximum, first index on ties
            const float cv = __uint_as_float(u[j]);
            if (nb + j < N && cv > lv[0]) {
              lv[0] = cv;
              li[0] = nb + j;
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(acc_empty(ab));
      if (KT > 0) {
        const int t = tile0 + i;
        if ((t + 1) % pt == 0 || t == NT - 1) {  // a part of a vocabulary tile ends here
#pragma unroll
          for (int e = 0; e < KL; ++e) {  // merge the odd-column list in
            list_insert<KL, true>(lv, li, ov[e], oi[e]);
            ov[e] = -INFINITY;
            oi[e] = INT_MAX;
          }
          if (row < M && !*abort_flag) {
            const int NV = (NT + vt - 1) / vt;
            const long long o = ((static_cast<long long>(row) * NV + t / vt) * vs + (t % vt) / pt) * KL;
#pragma unroll
            for (int e = 0; e < KL; ++e) {
              plv[o + e] = lv[e];
              pli[o + e] = li[e];
            }
          }
#pragma unroll
          for (int e = 0; e < KL; ++e) {
            lv[e] = -INFINITY;
            li[e] = INT_MAX;
          }
        }
      }
    }
    if (KT == 0 && row < M && !*abort_flag) {
      part_v[static_cast<long long>(row) * S + g] = lv[0];
      part_i[static_cast<long long>(row) * S + g] = li[0];
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

// Merge the S partials of each row: first index among equal maxima.
__global__ void __launch_bounds__(256) lm_head_merge_kernel(const float* __restrict__ part_v,
                                                            const int* __restrict__ part_i, int S, int M,
                                                            int32_t* __restrict__ argmax, float* __restrict__ max_logit) {
  pdl_wait();
  const int row = blockIdx.x * blockDim.x + threadIdx.x;
  if (row >= M) return;
  float bv = -INFINITY;
  int bi = INT_MAX;
  for (int s = 0; s < S; ++s) {
    const float v = part_v[static_cast<long long>(row) * S + s];
    const int i = part_i[static_cast<long long>(row) * S + s];
    if (better(v, i, bv, bi)) {
      bv = v;
      bi = i;
    }
  }
  argmax[row] = bi;
  if (max_logit != nullptr) max_logit[row] = bv;
}

// ---------------------------------------------------------------------------------------------
// The draft's two-stage efficient LM head ("jialefu.github.io — EAGLE-4 efficient LM head",
// sections "EAGLE Efficient LM Head" and "A variant based on local Top-k"):
//   u = bf16(B h) (lowrank_proj_kernel), scores = A u with the k_tile best ids of every
//   vocabulary tile kept in the GEMM epilogue (lm_head_kernel<KT>), exact logits W[c] h of the
//   candidates (gather_logits_kernel), and the k best candidates with log-probabilities over
//   the candidate set (head_topk_kernel).
// ---------------------------------------------------------------------------------------------

// One warp per output u[row][j] = sum_k B[j][k] h[row][k] (fp32, lanes over 8-element chunks,
// then a shuffle sum), rounded to bf16.  d % 8 == 0.
__global__ void __launch_bounds__(256) lowrank_proj_kernel(const __nv_bfloat16* __restrict__ hidden,
                                                          const __nv_bfloat16* __restrict__ lr_b, int d, int rank,
                                                          __nv_bfloat16* __restrict__ u) {
  pdl_wait();
  const int row = blockIdx.x, j = blockIdx.y * 8 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  if (j >= rank) return;
  const uint4* h4 = reinterpret_cast<const uint4*>(hidden + static_cast<long long>(row) * d);
  const uint4* b4 = reinterpret_cast<const uint4*>(lr_b + static_cast<long long>(j) * d);
  auto dot8 = [](const uint4& x, const uint4& y, float acc) {
    acc = fmaf(bf16_lo(x.x), bf16_lo(y.x), acc);
    acc = fmaf(bf16_hi(x.x), bf16_hi(y.x), acc);
    acc = fmaf(bf16_lo(x.y), bf16_lo(y.y), acc);
    acc = fmaf(bf16_hi(x.y), bf16_hi(y.y), acc);
    acc = fmaf(bf16_lo(x.z), bf16_lo(y.z), acc);
    acc = fmaf(bf16_hi(x.z), bf16_hi(y.z), acc);
    acc = fmaf(bf16_lo(x.w), bf16_lo(y.w), acc);
    return fmaf(bf16_hi(x.w), bf16_hi(y.w), acc);
  };
  // eight 16-byte pairs in flight per lane before any is used (a row of 4096 is two batches)
  const int n8 = d / 8;
  float acc0 = 0.f, acc1 = 0.f;
  int c = lane;
  for (; c + 7 * 32 < n8; c += 8 * 32) {
    uint4 x[8], y[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      x[e] = __ldg(h4 + c + 32 * e);
      y[e] = __ldg(b4 + c + 32 * e);
    }
#pragma unroll
    for (int e = 0; e < 8; e += 2) {
      acc0 = dot8(x[e], y[e], acc0);
      acc1 = dot8(x[e + 1], y[e + 1], acc1);
    }
  }
  for (; c < n8; c += 32) acc0 = dot8(__ldg(h4 + c), __ldg(b4 + c), acc0);
  float acc = acc0 + acc1;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
  if (lane == 0) u[static_cast<long long>(row) * rank + j] = __float2bfloat16_rn(acc);
}

// One warp per candidate slot c = (vocabulary tile, rank e < kt).  The warp first merges the
// tile's part lists (value descending, ties -> lower id; lane j holds entry j, at most 32) and
// takes the e-th best as the candidate (-1 when the tile has fewer columns), writes it to cand,
// then computes logits[row][c] = W[cand] . h[row] (fp32), -inf for an empty slot.
__global__ void __launch_bounds__(256) gather_logits_kernel(const __nv_bfloat16* __restrict__ hidden,
                                                           const __nv_bfloat16* __restrict__ weight, int V, int d,
                                                           const float* __restrict__ plv, const int* __restrict__ pli,
                                                           int kt, int vt, int pt, int vs, int NT,
                                                           int32_t* __restrict__ cand, int C,
                                                           float* __restrict__ logits, int32_t* status) {
  pdl_wait();
  const int row = blockIdx.x, c = blockIdx.y * 8 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  if (c >= C) return;
  const int vtile = c / kt, e = c % kt;
  const int NV = (NT + vt - 1) / vt;
  const int parts = (min(vt, NT - vtile * vt) + pt - 1) / pt;  // parts that hold columns
  const int n = parts * kt;
  float v = -INFINITY;
  int vid = INT_MAX;
  if (lane < n) {
    const long long o = (static_cast<long long>(row) * NV + vtile) * vs * kt + lane;
    v = plv[o];
    vid = pli[o];
  }
  int rank = 0;
  for (int j = 0; j < n; ++j) {
    const float vj = __shfl_sync(0xffffffffu, v, j);
    const int ij = __shfl_sync(0xffffffffu, vid, j);
    rank += ij != INT_MAX && (vj > v || (vj == v && ij < vid));
  }
  const unsigned hit = __ballot_sync(0xffffffffu, lane < n && vid != INT_MAX && rank == e);
  const int id = hit ? __shfl_sync(0xffffffffu, vid, __ffs(hit) - 1) : -1;
  if (lane == 0) cand[static_cast<long long>(row) * C + c] = id;
  float acc = -INFINITY;
  if (id >= 0 && id < V) {
    const uint4* h4 = reinterpret_cast<const uint4*>(hidden + static_cast<long long>(row) * d);
    const uint4* w4 = reinterpret_cast<const uint4*>(weight + static_cast<long long>(id) * d);
    acc = 0.f;
    for (int k = lane; k < d / 8; k += 32) {
      const uint4 x = __ldg(h4 + k), y = __ldg(w4 + k);
      acc = fmaf(bf16_lo(x.x), bf16_lo(y.x), acc);
      acc = fmaf(bf16_hi(x.x), bf16_hi(y.x), acc);
      acc = fmaf(bf16_lo(x.y), bf16_lo(y.y), acc);
      acc = fmaf(bf16_hi(x.y), bf16_hi(y.y), acc);
      acc = fmaf(bf16_lo(x.z), bf16_lo(y.z), acc);
      acc = fmaf(bf16_hi(x.z), bf16_hi(y.z), acc);
      acc = fmaf(bf16_lo(x.w), bf16_lo(y.w), acc);
      acc = fmaf(bf16_hi(x.w), bf16_hi(y.w), acc);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
  } else if (id >= V && lane == 0) {
    report(status, TS_ERR_DEVICE_CHECK);
  }
  if (lane == 0) logits[static_cast<long long>(row) * C + c] = acc;
}

// One warp per row, for candidate sets of at most kHeadWarpMaxC: the same k best candidates
// and log-probabilities as head_topk_kernel below.  Every lane keeps the best of its own share
// (a stride-32 slice in shared memory); a pick is a 5-step shuffle reduction of the 32 lane
// bests, after which only the lane that held the pick rescans its share.  No block barrier.
constexpr int kHeadRows = 4;
constexpr int kHeadWarpMaxC = 1024;
__global__ void __launch_bounds__(kHeadRows * 32) head_topk_warp_kernel(const float* __restrict__ logits,
                                                                       const int32_t* __restrict__ cand, int M,
                                                                       int C, int k, int32_t* __restrict__ top_tok,
                                                                       float* __restrict__ top_logp) {
  extern __shared__ unsigned char smem_raw[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  float* sl = reinterpret_cast<float*>(smem_raw) + static_cast<size_t>(warp) * 2 * C;
  int* si = reinterpret_cast<int*>(sl + C);
  pdl_wait();
  const int row = blockIdx.x * kHeadRows + warp;
  if (row >= M) return;
  const float* lr = logits + static_cast<long long>(row) * C;
  const int32_t* cr = cand + static_cast<long long>(row) * C;
  float mx = -INFINITY, bv = -INFINITY;
  int bi = INT_MAX, bc = -1;
  for (int c = lane; c < C; c += 32) {
    const int id = cr[c];
    const float l = id >= 0 ? lr[c] : -INFINITY;
    const int ii = id >= 0 ? id : INT_MAX;
    sl[c] = l;
    si[c] = ii;
    mx = fmaxf(mx, l);
    if (better(l, ii, bv, bi)) bv = l, bi = ii, bc = c;
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
  float sum = 0.f;
  for (int c = lane; c < C; c += 32)
    if (sl[c] != -INFINITY) sum += expf(sl[c] - mx);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
  const float lse = mx + logf(sum);
  for (int j = 0; j < k; ++j) {
    float v = bv;
    int i = bi;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, v, off);
      const int oi = __shfl_xor_sync(0xffffffffu, i, off);
      if (better(ov, oi, v, i)) v = ov, i = oi;
    }
    if (lane == 0) {
      top_tok[static_cast<long long>(row) * k + j] = i == INT_MAX ? -1 : i;
      top_logp[static_cast<long long>(row) * k + j] = i == INT_MAX ? -INFINITY : v - lse;
    }
    if (i != INT_MAX && bi == i) {  // this lane held the pick: take it out, find its next best
      sl[bc] = -INFINITY;
      si[bc] = INT_MAX;
      bv = -INFINITY, bi = INT_MAX, bc = -1;
      for (int c = lane; c < C; c += 32)
        if (better(sl[c], si[c], bv, bi)) bv = sl[c], bi = si[c], bc = c;
    }
  }
}

// One CTA per row (larger candidate sets): the k best candidates (logit descending, ties ->
// lower id) and their log-probabilities over the candidate set (logit - logsumexp of the
// candidates' logits).
constexpr int kHeadThreads = 256;
__device__ __forceinline__ void block_best_pair(float& v, int& i, float* s_v, int* s_i) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    const float ov = __shfl_xor_sync(0xffffffffu, v, off);
    const int oi = __shfl_xor_sync(0xffffffffu, i, off);
    if (better(ov, oi, v, i)) {
      v = ov;
      i = oi;
    }
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __syncthreads();
  if (lane == 0) {
    s_v[warp] = v;
    s_i[warp] = i;
  }
  __syncthreads();
  v = s_v[0];
  i = s_i[0];
  for (int w = 1; w < kHeadThreads / 32; ++w)
    if (better(s_v[w], s_i[w], v, i)) {
      v = s_v[w];
      i = s_i[w];
    }
}

__global__ void __launch_bounds__(kHeadThreads) head_topk_kernel(const float* __restrict__ logits,
                                                                const int32_t* __restrict__ cand, int C, int k,
                                                                int32_t* __restrict__ top_tok,
                                                                float* __restrict__ top_logp) {
  extern __shared__ unsigned char smem_raw[];
  float* sl = reinterpret_cast<float*>(smem_raw);
  int* si = reinterpret_cast<int*>(sl + C);
  __shared__ float s_v[kHeadThreads / 32];
  __shared__ int s_i[kHeadThreads / 32];
  pdl_wait();
  const int row = blockIdx.x;
  float mx = -INFINITY;
  for (int c = threadIdx.x; c < C; c += kHeadThreads) {
    const int id = cand[static_cast<long long>(row) * C + c];
    const float l = logits[static_cast<long long>(row) * C + c];
    sl[c] = id >= 0 ? l : -INFINITY;
    si[c] = id >= 0 ? id : INT_MAX;
    mx = fmaxf(mx, sl[c]);
  }
  int dummy = 0;
  block_best_pair(mx, dummy, s_v, s_i);
  float sum = 0.f;
  for (int c = threadIdx.x; c < C; c += kHeadThreads)
    if (sl[c] != -INFINITY) sum += expf(sl[c] - mx);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
  __syncthreads();
  if ((threadIdx.x & 31) == 0) s_v[threadIdx.x >> 5] = sum;
  __syncthreads();
  float tot = 0.f;
  for (int w = 0; w < kHeadThreads / 32; ++w) tot += s_v[w];
  const float lse = mx + logf(tot);
  for (int j = 0; j < k; ++j) {
    float bv = -INFINITY;
    int bi = INT_MAX, bc = -1;
    for (int c = threadIdx.x; c < C; c += kHeadThreads)
      if (better(sl[c], si[c], bv, bi)) {
        bv = sl[c];
        bi = si[c];
        bc = c;
      }
    int who = bi;
    block_best_pair(bv, who, s_v, s_i);
    if (bi == who && bc >= 0 && who != INT_MAX) sl[bc] = -INFINITY, si[bc] = INT_MAX;  // take it out
    if (threadIdx.x == 0) {
      top_tok[static_cast<long long>(row) * k + j] = who == INT_MAX ? -1 : who;
      top_logp[static_cast<long long>(row) * k + j] = who == INT_MAX ? -INFINITY : bv - lse;
    }
    __syncthreads();
  }
}

using EncodeFn = PFN_cuTensorMapEncodeTiled_v12000;

static EncodeFn get_encode() {
  static EncodeFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeFn>(f);
  });
  return fn;
}

// [rows, K] bf16 row-major, boxes of box_rows x 64 with 128-byte swizzle.
static bool encode_rows(CUtensorMap* map, const void* base, int rows, int K, int box_rows) {
  EncodeFn enc = get_encode();
  if (enc == nullptr) return false;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(K) * 2};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(BK), static_cast<cuuint32_t>(box_rows)};
  const cuuint32_t estr[2] = {1u, 1u};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Vocabulary tiles per CTA: with MT row tiles, about one wave of CTAs (the MT CTAs of one
// vocabulary range are adjacent in launch order, so they share the weight tiles in L2).
// With vocabulary tiles of vt GEMM tiles (the efficient head's local top-k), a tile is split into
// vs parts (a power of two dividing vt, with vs * kt <= 32 part-list entries per tile) when that
// brings the grid closer to one wave; a CTA takes whole parts.
static void plan(int M, int N, int num_sms, int* groups, int* tpg, int vt = 1, int kt = 1, int* pt_out = nullptr,
                 int* vs_out = nullptr) {
  const int MT = (M + BM - 1) / BM;
  const int NT = (N + BN - 1) / BN;
  const int NV = (NT + vt - 1) / vt;  // vocabulary tiles
  int cap = num_sms / MT;
  if (cap < 1) cap = 1;
  int vs = 1;
  while (2 * vs <= vt && vt % (2 * vs) == 0 && 2 * vs * kt <= 32 &&
         static_cast<long long>(NV) * 2 * vs <= cap)
    vs *= 2;
  const int pt = vt / vs;
  const int NP = (NT + pt - 1) / pt;  // parts; a CTA takes whole ones
  int G = cap;
  if (G > NP) G = NP;
  const int t = (NP + G - 1) / G * pt;
  *tpg = t;
  *groups = (NT + t - 1) / t;
  if (pt_out) *pt_out = pt;
  if (vs_out) *vs_out = vs;
}

}  // namespace lm

size_t lm_head_partials(int M, int N, int num_sms) {
  int G, t;
  lm::plan(M, N, num_sms, &G, &t);
  return static_cast<size_t>(G);
}

size_t lm_head_workspace_bytes(int M, int N, int num_sms) {
  return static_cast<size_t>(M) * lm_head_partials(M, N, num_sms) * 8 + 256;
}

int lm_head_partials_launch(const void* hidden, const void* weight, int M, int N, int K, float* part_v,
                            int* part_i, int* S_out, int32_t* dev_status, cudaStream_t stream, int num_sms) {
  int G, tpg;
  lm::plan(M, N, num_sms, &G, &tpg);
  CUtensorMap mh, mw;
  if (!lm::encode_rows(&mh, hidden, M, K, lm::BM) || !lm::encode_rows(&mw, weight, N, K, lm::BN))
    return TS_ERR_CUDA;
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(once, [] {
    attr_err = cudaFuncSetAttribute(lm::lm_head_kernel<0>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    lm::SMEM_BYTES);
  });
  if (attr_err != cudaSuccess) return TS_ERR_CUDA;
  const int MT = (M + lm::BM - 1) / lm::BM;
  if (launch_pdl(lm::lm_head_kernel<0>, dim3(MT, G), dim3(lm::THREADS), lm::SMEM_BYTES, stream, mh, mw, M, N, K,
                 tpg, part_v, part_i, G, 1, 1, 1, static_cast<float*>(nullptr), static_cast<int*>(nullptr),
                 dev_status) != cudaSuccess)
    return TS_ERR_CUDA;
  count_launches(1);
  *S_out = G;
  return TS_OK;
}

int lm_head_argmax_launch(const void* hidden, const void* weight, int M, int N, int K, int32_t* argmax,
                          float* max_logit, void* workspace, int32_t* dev_status, cudaStream_t stream,
                          int num_sms) {
  const int G = static_cast<int>(lm_head_partials(M, N, num_sms));
  float* part_v = static_cast<float*>(workspace);
  int* part_i = reinterpret_cast<int*>(part_v + static_cast<size_t>(M) * G);
  int S = 0;
  const int rc = lm_head_partials_launch(hidden, weight, M, N, K, part_v, part_i, &S, dev_status, stream, num_sms);
  if (rc != TS_OK) return rc;
  if (launch_pdl(lm::lm_head_merge_kernel, dim3((M + 255) / 256), dim3(256), 0, stream, part_v, part_i, S, M, argmax,
                 max_logit) != cudaSuccess)
    return TS_ERR_CUDA;
  count_launches(1);
  return TS_OK;
}


int efficient_head_candidates(int V, int tile_tokens, int k_tile) {
  return (V + tile_tokens - 1) / tile_tokens * k_tile;
}

size_t efficient_head_workspace_bytes(int M, int V, int rank, int tile_tokens, int k_tile) {
  const size_t C = static_cast<size_t>(efficient_head_candidates(V, tile_tokens, k_tile));
  const size_t u = (static_cast<size_t>(M) * rank * 2 + 255) / 256 * 256;
  // part lists: at most tile_tokens / 256 parts per vocabulary tile, k_tile (value, id) each
  const size_t vt = static_cast<size_t>(tile_tokens / lm::BN);
  const size_t parts = (static_cast<size_t>(M) * (C / k_tile) * vt * k_tile * 8 + 255) / 256 * 256;
  return u + static_cast<size_t>(M) * C * 8 + parts + 256;
}

template <int KT>
static cudaError_t launch_scores(const CUtensorMap& mh, const CUtensorMap& mw, int M, int V, int rank, int tpg,
                                 int G, int vt, int pt, int vs, float* plv, int* pli, int32_t* status,
                                 cudaStream_t stream) {
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(once, [] {
    attr_err = cudaFuncSetAttribute(lm::lm_head_kernel<KT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    lm::SMEM_BYTES);
  });
  if (attr_err != cudaSuccess) return attr_err;
  const int MT = (M + lm::BM - 1) / lm::BM;
  return launch_pdl(lm::lm_head_kernel<KT>, dim3(MT, G), dim3(lm::THREADS), lm::SMEM_BYTES, stream, mh, mw, M, V,
                    rank, tpg, static_cast<float*>(nullptr), static_cast<int*>(nullptr), 0, vt, pt, vs, plv, pli,
                    status);
}

int efficient_head_launch(const void* hidden, const void* lr_b, const void* lr_a, const void* weight, int M, int V,
                          int d, int rank, int tile_tokens, int k_tile, int k, int32_t* top_tok, float* top_logp,
                          int32_t* cand_out, void* workspace, int32_t* dev_status, cudaStream_t stream,
                          int num_sms) {
  const int C = efficient_head_candidates(V, tile_tokens, k_tile);
  unsigned char* ws = static_cast<unsigned char*>(workspace);
  __nv_bfloat16* u = reinterpret_cast<__nv_bfloat16*>(ws);
  const size_t u_bytes = (static_cast<size_t>(M) * rank * 2 + 255) / 256 * 256;
  int32_t* cand = cand_out != nullptr ? cand_out : reinterpret_cast<int32_t*>(ws + u_bytes);
  float* logits = reinterpret_cast<float*>(ws + u_bytes + static_cast<size_t>(M) * C * 4);
  const int vt = tile_tokens / lm::BN;
  const size_t nv = static_cast<size_t>(C / k_tile);
  float* plv = reinterpret_cast<float*>(ws + u_bytes + static_cast<size_t>(M) * C * 8);
  int* pli = reinterpret_cast<int*>(plv + static_cast<size_t>(M) * nv * vt * k_tile);
  // 1. u = bf16(B h)
  if (launch_pdl(lm::lowrank_proj_kernel, dim3(M, (rank + 7) / 8), dim3(256), 0, stream,
                 static_cast<const __nv_bfloat16*>(hidden), static_cast<const __nv_bfloat16*>(lr_b), d, rank, u) !=
      cudaSuccess)
    return TS_ERR_CUDA;
  // 2. scores = A u with the local top-k_tile of every part of every vocabulary tile
  int G, tpg, pt, vs;
  lm::plan(M, V, num_sms, &G, &tpg, vt, k_tile, &pt, &vs);
  CUtensorMap mu, ma;
  if (!lm::encode_rows(&mu, u, M, rank, lm::BM) || !lm::encode_rows(&ma, lr_a, V, rank, lm::BN)) return TS_ERR_CUDA;
  cudaError_t e;
  switch (k_tile) {
    case 1: e = launch_scores<1>(mu, ma, M, V, rank, tpg, G, vt, pt, vs, plv, pli, dev_status, stream); break;
    case 2: e = launch_scores<2>(mu, ma, M, V, rank, tpg, G, vt, pt, vs, plv, pli, dev_status, stream); break;
    case 3: e = launch_scores<3>(mu, ma, M, V, rank, tpg, G, vt, pt, vs, plv, pli, dev_status, stream); break;
    case 4: e = launch_scores<4>(mu, ma, M, V, rank, tpg, G, vt, pt, vs, plv, pli, dev_status, stream); break;
    case 5: e = launch_scores<5>(mu, ma, M, V, rank, tpg, G, vt, pt, vs, plv, pli, dev_status, stream); break;
    case 6: e = launch_scores<6>(mu, ma, M, V, rank, tpg, G, vt, pt, vs, plv, pli, dev_status, stream); break;
    case 7: e = launch_scores<7>(mu, ma, M, V, rank, tpg, G, vt, pt, vs, plv, pli, dev_status, stream); break;
    default: e = launch_scores<8>(mu, ma, M, V, rank, tpg, G, vt, pt, vs, plv, pli, dev_status, stream); break;
  }
  if (e != cudaSuccess) return TS_ERR_CUDA;
  // 3. the candidates (merged part lists) and their exact logits
  const int NT = (V + lm::BN - 1) / lm::BN;
  if (launch_pdl(lm::gather_logits_kernel, dim3(M, (C + 7) / 8), dim3(256), 0, stream,
                 static_cast<const __nv_bfloat16*>(hidden), static_cast<const __nv_bfloat16*>(weight), V, d,
                 static_cast<const float*>(plv), static_cast<const int*>(pli), k_tile, vt, pt, vs, NT, cand, C,
                 logits, dev_status) != cudaSuccess)
    return TS_ERR_CUDA;
  // 4. the k best candidates and their log-probabilities over the candidate set
  if (C <= lm::kHeadWarpMaxC) {
    if (launch_pdl(lm::head_topk_warp_kernel, dim3((M + lm::kHeadRows - 1) / lm::kHeadRows), dim3(lm::kHeadRows * 32),
                   static_cast<size_t>(lm::kHeadRows) * C * 8, stream, logits, cand, M, C, k, top_tok,
                   top_logp) != cudaSuccess)
      return TS_ERR_CUDA;
    count_launches(4);
    return TS_OK;
  }
  const size_t smem = static_cast<size_t>(C) * 8;
  if (smem > 48 * 1024 &&
      cudaFuncSetAttribute(lm::head_topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem)) !=
          cudaSuccess)
    return TS_ERR_CUDA;
  if (launch_pdl(lm::head_topk_kernel, dim3(M), dim3(lm::kHeadThreads), smem, stream, logits, cand, C, k, top_tok,
                 top_logp) != cudaSuccess)
    return TS_ERR_CUDA;
  count_launches(4);
  return TS_OK;
}

}  // namespace ts
