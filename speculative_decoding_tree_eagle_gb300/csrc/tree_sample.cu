// ts_tree_accept_sample kernel: stochastic (temperature T > 0) verification of the draft tree
// by multi-round rejection sampling.
//
// Source: "lesty.tech — EAGLE-2 vs. Medusa", section 4 (Mathematical Verification: Lossless
// Rejection Sampling): a candidate x proposed by q is kept with probability min(1, p(x)/q(x));
// after a rejection one token is drawn from the normalised max(0, p - q).  On the tree the
// children of the current node are tried in flat order, each rejection replacing p by that
// residual (and removing x from q); the first kept child becomes the current node.  Point
// proposals (q = a unit mass on each candidate) make a rejection simply remove the token's
// mass from p.
//
// Two kernels; the launcher picks by vocabulary size.
//
// sample_cluster_kernel (V <= 131072): one thread-block cluster of up to 8 CTAs per sequence,
// each CTA holding its slice of the vocabulary in registers (see the cluster section below):
// a visited node's rows are read from HBM once, draft-mode residual updates run on the
// registers, and cluster-wide sums go through exchange records read over DSMEM.
//
// sample_kernel (larger vocabularies): one CTA of 512 threads per sequence streams the rows.
// At each visited node u:
//   pass A  one read of the target row: a per-thread running (max, sum of 2^(s - max)) with
//           s = logit * log2(e) / T, merged across the block; in draft mode also the draft
//           row of u (q = its exp, renormalised).  Warp 0 first lists u's children in flat
//           order (ballot over the parent array) and gathers their tokens, uniforms and
//           logits.
//   trials  point mode decides all children on one thread: keep x iff r * Z_left < e(x),
//           Z_left losing e(x) of every rejected token.  Draft mode decides one child at a
//           time; each rejection runs one residual pass (w = max(0, p - q) into one of two
//           workspace rows per sequence, plus the proposal's remaining mass).
//   bonus   when no child is kept: the inverse CDF over token ids.  Every warp sums its
//           contiguous segment of the residual (pieces of 32 x VEC ids, lane-ordered
//           inclusive scans), one thread finds the segment holding r * total, and that warp
//           rescans it with the same arithmetic to the token.
//   Rejected tokens of the current node are kept in a shared-memory bitmap over the vocabulary.
#include <cmath>
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace ts {
namespace {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / kWarp;
constexpr float kLog2e = 1.4426950408889634f;
constexpr unsigned kFull = 0xffffffffu;
constexpr int kSampleMaxBitmapBytes = TS_SAMPLE_MAX_VOCAB / 8;

struct SampleArgs {
  const void* logits;
  const int32_t* tokens;
  const int32_t* parents;
  const float* uniforms;
  const float* draft_logp;
  const int32_t* node_row;
  int R, m, V;
  float c;  // log2(e) / T
  int q_draft;
  int32_t* accept_len;
  int32_t* accept_path;
  int32_t* bonus;
  float* resid;  // [B, 2, Vp] in draft mode
  long long Vp;
  int32_t* dev_status;
};

// VEC consecutive values of a row as fp32.  VEC is 1, 4 or 8; for VEC > 1 the index is a
// multiple of VEC and the row start is 16-byte aligned.
template <int VEC>
__device__ __forceinline__ void load_vec(const float* p, long long i, float (&v)[VEC]) {
  if constexpr (VEC == 1) {
    v[0] = __ldg(p + i);
  } else {
#pragma unroll
    for (int h = 0; h < VEC / 4; ++h) {
      const float4 f = __ldg(reinterpret_cast<const float4*>(p + i) + h);
      v[4 * h + 0] = f.x;
      v[4 * h + 1] = f.y;
      v[4 * h + 2] = f.z;
      v[4 * h + 3] = f.w;
    }
  }
}

template <int VEC>
__device__ __forceinline__ void load_vec(const __nv_bfloat16* p, long long i, float (&v)[VEC]) {
  if constexpr (VEC == 1) {
    v[0] = __bfloat162float(p[i]);
  } else {
    static_assert(VEC == 8, "bf16 rows are read 8 values at a time");
    const uint4 w = __ldg(reinterpret_cast<const uint4*>(p + i));
    v[0] = bf16_lo(w.x), v[1] = bf16_hi(w.x), v[2] = bf16_lo(w.y), v[3] = bf16_hi(w.y);
    v[4] = bf16_lo(w.z), v[5] = bf16_hi(w.z), v[6] = bf16_lo(w.w), v[7] = bf16_hi(w.w);
  }
}

// Residual rows are written by this kernel, so they are read through L2 (ld.global.cg),
// never through the read-only path.
template <int VEC>
__device__ __forceinline__ void load_vec_cg(const float* p, long long i, float (&v)[VEC]) {
  if constexpr (VEC == 1) {
    v[0] = __ldcg(p + i);
  } else {
#pragma unroll
    for (int h = 0; h < VEC / 4; ++h) {
      const float4 f = __ldcg(reinterpret_cast<const float4*>(p + i) + h);
      v[4 * h + 0] = f.x;
      v[4 * h + 1] = f.y;
      v[4 * h + 2] = f.z;
      v[4 * h + 3] = f.w;
    }
  }
}

template <int VEC>
__device__ __forceinline__ void store_vec(float* p, long long i, const float (&v)[VEC]) {
  if constexpr (VEC == 1) {
    p[i] = v[0];
  } else {
#pragma unroll
    for (int h = 0; h < VEC / 4; ++h)
      reinterpret_cast<float4*>(p + i)[h] = make_float4(v[4 * h], v[4 * h + 1], v[4 * h + 2], v[4 * h + 3]);
  }
}

// 2^(s - M) of a scaled logit; 0 for s = -inf.  The rounding of every step is fixed (no
// contraction) so that every pass recomputes the same value.
__device__ __forceinline__ float mass(float s, float M) { return ex2_approx(__fsub_rn(s, M)); }

// Merge running (max, sum of 2^(s - max)) pairs.
__device__ __forceinline__ void ms_merge(float& M, float& S, float M2, float S2) {
  const float Mn = fmaxf(M, M2);
  if (Mn == -INFINITY) return;
  S = S * ex2_approx(M - Mn) + S2 * ex2_approx(M2 - Mn);
  M = Mn;
}

// This thread's (max, sum) over row * scale.
template <typename T, int VEC>
__device__ __forceinline__ void row_max_sum(const T* row, int V, float scale, float& M, float& S) {
  M = -INFINITY;
  S = 0.f;
#pragma unroll 4
  for (long long i = static_cast<long long>(threadIdx.x) * VEC; i < V; i += kThreads * VEC) {
    float v[VEC];
    load_vec<VEC>(row, i, v);
    float vm = -INFINITY;
#pragma unroll
    for (int j = 0; j < VEC; ++j) {
      v[j] = __fmul_rn(v[j], scale);
      vm = fmaxf(vm, v[j]);
    }
    if (vm == -INFINITY) continue;
    if (vm > M) {
      S *= ex2_approx(M - vm);
      M = vm;
    }
#pragma unroll
    for (int j = 0; j < VEC; ++j) S += mass(v[j], M);
  }
}

// Block-wide merge of (M, S); every thread gets the result.  Uses red[0..2*kWarps).
__device__ __forceinline__ void block_max_sum(float& M, float& S, float* red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int off = 16; off; off >>= 1) {
    const float M2 = __shfl_xor_sync(kFull, M, off), S2 = __shfl_xor_sync(kFull, S, off);
    ms_merge(M, S, M2, S2);
  }
  if (lane == 0) red[warp] = M, red[kWarps + warp] = S;
  __syncthreads();
  M = lane < kWarps ? red[lane] : -INFINITY;
  S = lane < kWarps ? red[kWarps + lane] : 0.f;
#pragma unroll
  for (int off = 16; off; off >>= 1) {
    const float M2 = __shfl_xor_sync(kFull, M, off), S2 = __shfl_xor_sync(kFull, S, off);
    ms_merge(M, S, M2, S2);
  }
  __syncthreads();  // red may be reused right after
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int off = 16; off; off >>= 1) x += __shfl_xor_sync(kFull, x, off);
  return x;
}

__device__ __forceinline__ float warp_incl_scan(float x) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const float y = __shfl_up_sync(kFull, x, off);
    if (lane >= off) x = __fadd_rn(x, y);
  }
  return x;
}

__device__ __forceinline__ bool excluded(const uint32_t* bits, int x) { return (bits[x >> 5] >> (x & 31)) & 1u; }

struct Level {           // state of the current node, written by thread 0
  float M, invZ;         // target row: max of the scaled logits, 1 / sum of masses
  float Mq, Zq;          // draft row (draft mode): max of log2 q, remaining mass
  float Zleft;           // point mode: mass not yet rejected
  float invZw;           // 1 / sum of the residual row in use
  int src;               // 0: p from the logits, 1 + h: p from residual row h
  int nk, acc, nrej;     // children, kept child slot (-1 none), rejected tokens
};

// Residual value of id i..i+VEC-1 for the bonus draw.
template <typename T, int VEC>
__device__ __forceinline__ void bonus_values(const T* row, const float* wrow, const Level& L, const uint32_t* bits,
                                             bool use_excl, float c, long long i, int V, float (&v)[VEC]) {
  if (i >= V) {
#pragma unroll
    for (int j = 0; j < VEC; ++j) v[j] = 0.f;
    return;
  }
  if (L.src == 0) {
    load_vec<VEC>(row, i, v);
    const uint32_t w = use_excl ? (bits[i >> 5] >> (i & 31)) : 0u;
#pragma unroll
    for (int j = 0; j < VEC; ++j) v[j] = ((w >> j) & 1u) ? 0.f : mass(__fmul_rn(v[j], c), L.M);
  } else {
    load_vec_cg<VEC>(wrow, i, v);
  }
}

template <typename T, int VEC>
__global__ void __launch_bounds__(kThreads, 1) sample_kernel(const SampleArgs a) {
  extern __shared__ uint32_t s_bits[];  // ceil(V / 32) words: tokens rejected at this node
  __shared__ int s_par[TS_MAX_NODES], s_tok[TS_MAX_NODES], s_nrow[TS_MAX_NODES], s_path[TS_MAX_NODES];
  __shared__ int s_kid[TS_MAX_NODES], s_kx[TS_MAX_NODES], s_rej[TS_MAX_NODES];
  __shared__ float s_kr[TS_MAX_NODES], s_ks[TS_MAX_NODES], s_kd[TS_MAX_NODES];
  __shared__ unsigned char s_has[TS_MAX_NODES];
  __shared__ float s_red[4 * kWarps];
  __shared__ double s_seg[kWarps];
  __shared__ Level L;
  __shared__ int s_u, s_plen, s_sel, s_y, s_retry;
  __shared__ double s_tl;

  const int b = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int m = a.m, V = a.V;
  const long long bm = static_cast<long long>(b) * m;
  pdl_wait();

  // ---- load and check the tree -------------------------------------------------------
  const int words = (V + 31) >> 5;
  for (int i = tid; i < words; i += kThreads) s_bits[i] = 0u;
  for (int i = tid; i < m; i += kThreads) s_has[i] = 0;
  __syncthreads();
  int bad = 0;
  for (int i = tid; i < m; i += kThreads) {
    const int p = a.parents[bm + i], t = a.tokens[bm + i];
    s_par[i] = p;
    s_tok[i] = t;
    if (i == 0 ? p != -1 : (p < 0 || p >= i || t < 0 || t >= V)) bad = 1;
    else if (i > 0) s_has[p] = 1;
  }
  __syncthreads();
  if (a.q_draft) {
    for (int i = tid; i < m; i += kThreads) {
      const int r = a.node_row[bm + i];
      s_nrow[i] = r;
      if (s_has[i] && (r < 0 || r >= a.R)) bad = 1;
    }
  }
  if (__syncthreads_or(bad)) {
    if (tid == 0) {
      report(a.dev_status, TS_ERR_DEVICE_CHECK);
      a.accept_len[b] = 0;
      a.bonus[b] = -1;
    }
    for (int i = tid; i < m; i += kThreads) a.accept_path[bm + i] = -1;
    return;
  }

  const T* logits = static_cast<const T*>(a.logits);
  float* const resid0 = a.resid ? a.resid + static_cast<long long>(b) * 2 * a.Vp : nullptr;
  if (tid == 0) s_u = 0, s_plen = 1, s_path[0] = 0, L.nrej = 0;
  __syncthreads();

  for (;;) {
    const int u = s_u;
    const T* row = logits + (bm + u) * static_cast<long long>(V);
    const float* drow = nullptr;
    if (a.q_draft && s_has[u])
      drow = a.draft_logp + (static_cast<long long>(b) * a.R + s_nrow[u]) * static_cast<long long>(V);

    // children of u in flat order; the first 32 children's tokens, uniforms and logits are
    // fetched before pass A and stored after it, so their latency hides under the stream
    int nk = 0, px = 0;
    float pr = 0.f, pl = 0.f, pd = 0.f;
    if (warp == 0) {
      for (int base = 0; base < m; base += 32) {
        const int c = base + lane;
        const bool is = c < m && s_par[c] == u;
        const unsigned bal = __ballot_sync(kFull, is);
        if (is) s_kid[nk + __popc(bal & ((1u << lane) - 1u))] = c;
        nk += __popc(bal);
      }
      __syncwarp();
      if (lane < nk) {
        const int c = s_kid[lane];
        px = s_tok[c];
        pr = a.uniforms[bm + c];
        float lx[1];
        load_vec<1>(row, px, lx);
        pl = lx[0];
        if (drow) pd = __ldg(drow + px);
      }
    }

    // pass A: the target row's (max, sum); the draft row's in draft mode
    float M, S;
    row_max_sum<T, VEC>(row, V, a.c, M, S);
    if (warp == 0) {
      if (lane < nk) {
        s_kx[lane] = px;
        s_kr[lane] = pr;
        s_ks[lane] = __fmul_rn(pl, a.c);
        s_kd[lane] = __fmul_rn(pd, kLog2e);
      }
      for (int j = 32 + lane; j < nk; j += 32) {
        const int c = s_kid[j], x = s_tok[c];
        s_kx[j] = x;
        s_kr[j] = a.uniforms[bm + c];
        float lx[1];
        load_vec<1>(row, x, lx);
        s_ks[j] = __fmul_rn(lx[0], a.c);
        s_kd[j] = drow ? __fmul_rn(__ldg(drow + x), kLog2e) : 0.f;
      }
      if (lane == 0) L.nk = nk;
    }
    block_max_sum(M, S, s_red);
    float Mq = -INFINITY, Sq = 0.f;
    if (drow) {
      row_max_sum<float, VEC>(drow, V, kLog2e, Mq, Sq);
      block_max_sum(Mq, Sq, s_red);
    }
    if (tid == 0) {
      L.M = M;
      L.invZ = 1.f / S;
      L.Mq = Mq;
      L.Zq = Sq;
      L.Zleft = S;
      L.src = 0;
      L.invZw = 0.f;
      L.acc = -1;
      if (!a.q_draft) {  // point proposals: every trial on this thread
        float Zl = S;
        for (int j = 0; j < L.nk; ++j) {
          const int x = s_kx[j];
          const bool in = excluded(s_bits, x);
          const float e = in ? 0.f : mass(s_ks[j], M);
          if (s_kr[j] * Zl < e) {
            L.acc = j;
            break;
          }
          if (!in) {
            Zl -= e;
            s_bits[x >> 5] |= 1u << (x & 31);
            s_rej[L.nrej++] = x;
          }
        }
        L.Zleft = Zl;
      }
    }
    __syncthreads();

    if (a.q_draft) {  // draft proposals: one trial at a time, one residual pass per rejection
      for (int j = 0; j < L.nk; ++j) {
        const int x = s_kx[j];
        if (tid == 0) {
          const float p = L.src == 0 ? mass(s_ks[j], L.M) * L.invZ
                                     : __ldcg(resid0 + (L.src - 1) * a.Vp + x) * L.invZw;
          const float q = (excluded(s_bits, x) || !(L.Zq > 0.f)) ? 0.f : mass(s_kd[j], L.Mq) / L.Zq;
          if (s_kr[j] * q < p) L.acc = j;
        }
        __syncthreads();
        if (L.acc >= 0) break;
        // rejected: w = max(0, p - q) over the vocabulary; the proposal loses x
        const int src = L.src;
        const float M0 = L.M, invZ = L.invZ, invZw = L.invZw, Mq0 = L.Mq;
        const float invZq = L.Zq > 0.f ? 1.f / L.Zq : 0.f;
        const float* wsrc = src ? resid0 + (src - 1) * a.Vp : nullptr;
        float* wdst = resid0 + (src == 1 ? 1 : 0) * a.Vp;
        float sw = 0.f, sq = 0.f;
        for (long long i = static_cast<long long>(tid) * VEC; i < V; i += kThreads * VEC) {
          float p[VEC], q[VEC], w[VEC];
          if (src == 0) {
            load_vec<VEC>(row, i, p);
#pragma unroll
            for (int t = 0; t < VEC; ++t) p[t] = mass(__fmul_rn(p[t], a.c), M0) * invZ;
          } else {
            load_vec_cg<VEC>(wsrc, i, p);
#pragma unroll
            for (int t = 0; t < VEC; ++t) p[t] *= invZw;
          }
          load_vec<VEC>(drow, i, q);
          const uint32_t bw = s_bits[i >> 5] >> (i & 31);
#pragma unroll
          for (int t = 0; t < VEC; ++t) {
            const float qm = ((bw >> t) & 1u) ? 0.f : mass(__fmul_rn(q[t], kLog2e), Mq0);
            if (i + t != x) sq += qm;
            w[t] = fmaxf(0.f, p[t] - qm * invZq);
            sw += w[t];
          }
          store_vec<VEC>(wdst, i, w);
        }
        sw = warp_sum(sw);
        sq = warp_sum(sq);
        if (lane == 0) s_red[warp] = sw, s_red[kWarps + warp] = sq;
        __syncthreads();
        if (tid == 0) {
          float tw = 0.f, tq = 0.f;
          for (int w = 0; w < kWarps; ++w) tw += s_red[w], tq += s_red[kWarps + w];
          if (tw > 0.f) {  // a residual of zero mass leaves p as it was
            L.src = src == 1 ? 2 : 1;
            L.invZw = 1.f / tw;
          }
          L.Zq = tq;
          if (!excluded(s_bits, x)) {
            s_bits[x >> 5] |= 1u << (x & 31);
            s_rej[L.nrej++] = x;
          }
        }
        __syncthreads();
      }
    }

    if (L.acc >= 0) {  // walk down to the kept child
      __syncthreads();
      if (tid == 0) {
        const int c = s_kid[L.acc];
        s_path[s_plen++] = c;
        s_u = c;
        for (int j = 0; j < L.nrej; ++j) s_bits[s_rej[j] >> 5] &= ~(1u << (s_rej[j] & 31));
        L.nrej = 0;
      }
      __syncthreads();
      continue;
    }
    break;
  }

  // ---- bonus: inverse CDF over the residual of the last node ----------------------------
  // Lane and piece sums are fp32 (at most 32 x VEC small terms); the running sum over pieces
  // and segments is fp64, so the cumulative bounds stay far inside one token's mass.
  const int u = s_u;
  const T* row = logits + (bm + u) * static_cast<long long>(V);
  const float* wrow = L.src ? resid0 + (L.src - 1) * a.Vp : nullptr;
  const Level Lc = L;
  const long long piece = 32LL * VEC;
  const long long npieces = (V + piece - 1) / piece;
  const long long per_warp = (npieces + kWarps - 1) / kWarps;
  const long long pc0 = warp * per_warp, pc1 = min(npieces, (warp + 1) * per_warp);
  bool use_excl = !a.q_draft;
  for (;;) {
    double run = 0.0;
    for (long long pc = pc0; pc < pc1; ++pc) {
      float v[VEC];
      bonus_values<T, VEC>(row, wrow, Lc, s_bits, use_excl, a.c, pc * piece + lane * VEC, V, v);
      float ls = 0.f;
#pragma unroll
      for (int j = 0; j < VEC; ++j) ls = __fadd_rn(ls, v[j]);
      const float incl = warp_incl_scan(ls);
      run += static_cast<double>(__shfl_sync(kFull, incl, 31));
    }
    if (lane == 0) s_seg[warp] = run;
    __syncthreads();
    if (tid == 0) {
      double total = 0.0;
      for (int w = 0; w < kWarps; ++w) total += s_seg[w];
      s_retry = 0;
      s_sel = -1;
      if (!(total > 0.0)) {
        s_retry = use_excl;  // every remaining token has zero mass: draw from p itself
      } else {
        double t = static_cast<double>(a.uniforms[bm]) * total;
        if (!(t < total)) t = __longlong_as_double(__double_as_longlong(total) - 1);
        // the first segment whose upper bound passes t, else the last one with mass
        double pre = 0.0, pre_sel = 0.0;
        for (int w = 0; w < kWarps; ++w) {
          const double nxt = pre + s_seg[w];
          if (s_seg[w] > 0.0) {
            s_sel = w;
            pre_sel = pre;
            if (nxt > t) break;
          }
          pre = nxt;
        }
        s_tl = t - pre_sel;
      }
    }
    __syncthreads();
    if (!s_retry) break;
    use_excl = false;
    __syncthreads();
  }

  if (warp == s_sel) {
    const double tl = s_tl;
    double run = 0.0;
    int y = -1, lastnz = -1;
    for (long long pc = pc0; pc < pc1; ++pc) {
      const long long i0 = pc * piece + lane * VEC;
      float v[VEC];
      bonus_values<T, VEC>(row, wrow, Lc, s_bits, use_excl, a.c, i0, V, v);
      float ls = 0.f;
      int mynz = -1;
#pragma unroll
      for (int j = 0; j < VEC; ++j) {
        ls = __fadd_rn(ls, v[j]);
        if (v[j] > 0.f) mynz = static_cast<int>(i0) + j;
      }
      const float incl = warp_incl_scan(ls);
      float excl = __shfl_up_sync(kFull, incl, 1);
      if (lane == 0) excl = 0.f;
      const unsigned nzb = __ballot_sync(kFull, mynz >= 0);
      if (nzb) lastnz = __shfl_sync(kFull, mynz, 31 - __clz(nzb));
      const unsigned hit = __ballot_sync(kFull, run + static_cast<double>(incl) > tl);
      if (hit) {
        const int Ls = __ffs(hit) - 1;
        int yy = -1;
        if (lane == Ls) {
          double acc = run + static_cast<double>(excl);
#pragma unroll
          for (int j = 0; j < VEC; ++j) {
            acc += static_cast<double>(v[j]);
            if (yy < 0 && acc > tl) yy = static_cast<int>(i0) + j;
          }
          if (yy < 0) yy = mynz;
        }
        y = __shfl_sync(kFull, yy, Ls);
        break;
      }
      run += static_cast<double>(__shfl_sync(kFull, incl, 31));
    }
    if (y < 0) y = lastnz;
    if (lane == 0) s_y = y;
  }
  if (s_sel < 0 && tid == 0) s_y = -1;
  __syncthreads();
  if (tid == 0) {
    a.accept_len[b] = s_plen;
    a.bonus[b] = s_y;
    if (s_y < 0) report(a.dev_status, TS_ERR_DEVICE_CHECK);  // the target row had no mass
  }
  for (int i = tid; i < m; i += kThreads) a.accept_path[bm + i] = i < s_plen ? s_path[i] : -1;
}

// =====================================================================================
// Cluster path (V <= kClusterMaxVocab): one thread-block cluster of C <= 8 CTAs per
// sequence.  CTA r owns the vocabulary slice [r*NT*EPT, (r+1)*NT*EPT); every thread keeps EPT
// of its ids in registers (chunk j covers NT*VEC consecutive ids, thread t its VEC ids at
// offset t*VEC), so a node's target row (and draft row) is read from HBM once and every
// residual update, sum and the inverse CDF run on registers.  Cluster-wide values go through
// a small exchange record per CTA read over distributed shared memory.  Every CTA takes every
// decision itself from the same data in the same order, so the CTAs stay in lockstep
// without broadcasts and execute the same cluster barriers.
// =====================================================================================
namespace cl {

constexpr int NT = 512;
constexpr int NW = NT / kWarp;
constexpr int CMAX = 8;
constexpr int EPT_MAX = 32;

// One CTA's share of a cluster exchange (two buffers, alternated: one cluster barrier per
// exchange suffices, since a CTA rewrites a buffer only after every CTA has passed the
// barrier that follows its last read of it).
struct __align__(16) Xch {
  float M, S;      // node start: target slice (max of scaled logits, sum of 2^(s - max))
  float Mq, Sq;    // node start, draft mode: the same for the draft slice (log2 units)
  float w, q;      // residual step: sum of the new residual, remaining proposal mass
  float pnext, wnext;  // residual step: current / new residual at the next child (owner only)
  double tot;      // final draw: mass of the slice
  double pad;
};

__device__ __forceinline__ double ld_peer_f64(uint32_t local, uint32_t rank) {
  double v;
  asm volatile("ld.shared::cluster.f64 %0, [%1];" : "=d"(v) : "r"(dsmem_addr(local, rank)) : "memory");
  return v;
}

// Warp 0: lane r < C fetches 16 bytes of rank r's exchange record (one load per lane, all in
// flight together).  The merges below reduce over the lanes in a fixed butterfly order, the
// same in every CTA of the cluster.
__device__ __forceinline__ float4 fetch4(uint32_t local, int C, float4 dflt) {
  const int lane = threadIdx.x & 31;
  return lane < C ? ld_dsmem_f4(dsmem_addr(local, lane)) : dflt;
}
__device__ __forceinline__ float warp_max_f(float x) {
#pragma unroll
  for (int off = 16; off; off >>= 1) x = fmaxf(x, __shfl_xor_sync(kFull, x, off));
  return x;
}
__device__ __forceinline__ float warp_sum_f(float x) {
#pragma unroll
  for (int off = 16; off; off >>= 1) x += __shfl_xor_sync(kFull, x, off);
  return x;
}

// Whether id x lies in this thread's registers, and in which.
template <int VEC, int EPT>
__device__ __forceinline__ bool owns(long long x, long long slice0, int tid, int& reg) {
  const long long off = x - slice0;
  if (off < 0 || off >= static_cast<long long>(NT) * EPT) return false;
  const int o = static_cast<int>(off);
  const int rem = o % (NT * VEC);
  if (rem / VEC != tid) return false;
  reg = (o / (NT * VEC)) * VEC + rem % VEC;
  return true;
}

// Block max and sum of 2^(s - max) over this thread's values; valid in thread 0 only.
template <int EPT>
__device__ __forceinline__ float2 block_max_sum_t0(const float (&s)[EPT], float* red) {
  __syncthreads();  // thread 0 may still be reading red[] from the previous reduction
  float M = -INFINITY;
#pragma unroll
  for (int i = 0; i < EPT; ++i) M = fmaxf(M, s[i]);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int off = 16; off; off >>= 1) M = fmaxf(M, __shfl_xor_sync(kFull, M, off));
  if (lane == 0) red[warp] = M;
  __syncthreads();
  float Mc = red[0];
  for (int w = 1; w < NW; ++w) Mc = fmaxf(Mc, red[w]);
  float S = 0.f;
  if (Mc != -INFINITY) {
#pragma unroll
    for (int i = 0; i < EPT; ++i) S += mass(s[i], Mc);
  }
#pragma unroll
  for (int off = 16; off; off >>= 1) S += __shfl_xor_sync(kFull, S, off);
  __syncthreads();  // every thread has read red[] before it is overwritten
  if (lane == 0) red[warp] = S;
  __syncthreads();
  float St = 0.f;
  if (threadIdx.x == 0)
    for (int w = 0; w < NW; ++w) St += red[w];
  return make_float2(Mc, St);
}

// Block sums of four floats in a fixed order; the result is valid in thread 0 only.
__device__ __forceinline__ float4 block_sum4_t0(float a, float b, float c, float d, float* red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  __syncthreads();  // thread 0 may still be reading red[] from the previous reduction
#pragma unroll
  for (int off = 16; off; off >>= 1) {
    a += __shfl_xor_sync(kFull, a, off);
    b += __shfl_xor_sync(kFull, b, off);
    c += __shfl_xor_sync(kFull, c, off);
    d += __shfl_xor_sync(kFull, d, off);
  }
  if (lane == 0) red[warp] = a, red[NW + warp] = b, red[2 * NW + warp] = c, red[3 * NW + warp] = d;
  __syncthreads();
  float4 r = make_float4(0.f, 0.f, 0.f, 0.f);
  if (threadIdx.x == 0)
    for (int w = 0; w < NW; ++w) r.x += red[w], r.y += red[NW + w], r.z += red[2 * NW + w], r.w += red[3 * NW + w];
  return r;
}

__device__ __forceinline__ double warp_incl_scan_f64(double x) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const double y = __shfl_up_sync(kFull, x, off);
    if (lane >= off) x += y;
  }
  return x;
}

// Float-float sums for the inverse CDF: (hi, lo) with hi + lo the running sum.  Each addition
// is an exact two-sum (the rounding error of hi + b is recovered in full), so the pair keeps
// about 44 bits; the fp32 pipe is used because this GPU's fp64 rate is a small fraction of
// its fp32 rate.  The two-sum is symmetric in its operands, so the butterfly reductions give
// every lane the same pair.
struct DF {
  float hi, lo;
};
__device__ __forceinline__ DF df_two_sum(float a, float b) {
  const float s = __fadd_rn(a, b);
  const float bb = __fsub_rn(s, a);
  return {s, __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb))};
}
__device__ __forceinline__ DF df_add(DF a, DF b) {
  const DF s = df_two_sum(a.hi, b.hi);
  const float lo = __fadd_rn(s.lo, __fadd_rn(a.lo, b.lo));
  const float hi = __fadd_rn(s.hi, lo);
  return {hi, __fsub_rn(lo, __fsub_rn(hi, s.hi))};
}
__device__ __forceinline__ DF df_add1(DF a, float b) { return df_add(a, DF{b, 0.f}); }
__device__ __forceinline__ double df_to_d(DF a) { return static_cast<double>(a.hi) + static_cast<double>(a.lo); }
__device__ __forceinline__ DF df_shfl(DF a, int src) {
  return {__shfl_sync(kFull, a.hi, src), __shfl_sync(kFull, a.lo, src)};
}
__device__ __forceinline__ DF df_warp_sum(DF a) {
#pragma unroll
  for (int off = 16; off; off >>= 1) a = df_add(a, DF{__shfl_xor_sync(kFull, a.hi, off), __shfl_xor_sync(kFull, a.lo, off)});
  return a;
}
__device__ __forceinline__ DF df_warp_incl_scan(DF a) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const DF y{__shfl_up_sync(kFull, a.hi, off), __shfl_up_sync(kFull, a.lo, off)};
    if (lane >= off) a = df_add(a, y);
  }
  return a;
}
__device__ __forceinline__ DF df_warp_excl(DF inc) {
  DF e{__shfl_up_sync(kFull, inc.hi, 1), __shfl_up_sync(kFull, inc.lo, 1)};
  if ((threadIdx.x & 31) == 0) e = DF{0.f, 0.f};
  return e;
}

struct State {        // the walk's state, written by thread 0 of every CTA (identical values)
  float M, invZ;      // target row: max of the scaled logits, 1 / total mass
  float Mq, invZq;    // draft row: max (log2 units), 1 / remaining proposal mass (0 if none)
  float pinv;         // p = pv * pinv (pv: registers; the target masses, later the residual)
  float pnext;        // draft mode: p at the next child after a residual step
  int u, plen, nk, acc, nrej, apply, sel, chunk, retry;
  double tl, tc;      // final draw: target within the selected slice / chunk
};

}  // namespace cl

template <typename T, int VEC, int EPT>
__global__ void __launch_bounds__(cl::NT, 1) sample_cluster_kernel(const SampleArgs a, int C) {
  using namespace cl;
  constexpr int NCH = EPT / VEC;  // chunks per thread
  __shared__ int s_par[TS_MAX_NODES], s_tok[TS_MAX_NODES], s_nrow[TS_MAX_NODES], s_path[TS_MAX_NODES];
  __shared__ int s_kid[TS_MAX_NODES], s_kx[TS_MAX_NODES], s_rej[TS_MAX_NODES];
  __shared__ float s_kr[TS_MAX_NODES], s_ks[TS_MAX_NODES], s_kd[TS_MAX_NODES];
  __shared__ unsigned char s_has[TS_MAX_NODES];
  __shared__ float s_red[4 * NW];
  __shared__ DF s_dred[NW * NCH];
  __shared__ double s_ct[NCH], s_cpre[NCH];
  __shared__ Xch s_x[2];
  __shared__ State st;
  __shared__ int s_y, s_last;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint32_t rank = cluster_ctarank();
  const int b = blockIdx.x / C;
  const int m = a.m, V = a.V;
  const long long bm = static_cast<long long>(b) * m;
  const long long slice0 = static_cast<long long>(rank) * NT * EPT;
  pdl_wait();

  // ---- load and check the tree: every CTA of the cluster reads the same data and takes
  //      the same exit, before any cluster barrier ------------------------------------------
  for (int i = tid; i < m; i += NT) s_has[i] = 0;
  __syncthreads();
  int bad = 0;
  for (int i = tid; i < m; i += NT) {
    const int p = a.parents[bm + i], t = a.tokens[bm + i];
    s_par[i] = p;
    s_tok[i] = t;
    if (i == 0 ? p != -1 : (p < 0 || p >= i || t < 0 || t >= V)) bad = 1;
    else if (i > 0) s_has[p] = 1;
  }
  __syncthreads();
  if (a.q_draft) {
    for (int i = tid; i < m; i += NT) {
      const int r = a.node_row[bm + i];
      s_nrow[i] = r;
      if (s_has[i] && (r < 0 || r >= a.R)) bad = 1;
    }
  }
  if (__syncthreads_or(bad)) {
    if (rank == 0) {
      if (tid == 0) {
        report(a.dev_status, TS_ERR_DEVICE_CHECK);
        a.accept_len[b] = 0;
        a.bonus[b] = -1;
      }
      for (int i = tid; i < m; i += NT) a.accept_path[bm + i] = -1;
    }
    return;
  }

  const T* logits = static_cast<const T*>(a.logits);
  if (tid == 0) st.u = 0, st.plen = 1, s_path[0] = 0;
  __syncthreads();
  int xb = 0;          // exchange buffer
  float pv[EPT], qv[EPT];

  for (;;) {
    const int u = st.u;
    const T* row = logits + (bm + u) * static_cast<long long>(V);
    const bool draft = a.q_draft && s_has[u];
    const float* drow =
        draft ? a.draft_logp + (static_cast<long long>(b) * a.R + s_nrow[u]) * static_cast<long long>(V) : nullptr;

    // children of u in flat order; the first 32 children's tokens, uniforms and logits are
    // fetched before the slice loads and stored after them
    int nk = 0, px = 0;
    float pr = 0.f, pl = 0.f, pd = 0.f;
    if (warp == 0) {
      for (int base = 0; base < m; base += 32) {
        const int c = base + lane;
        const bool is = c < m && s_par[c] == u;
        const unsigned bal = __ballot_sync(kFull, is);
        if (is) s_kid[nk + __popc(bal & ((1u << lane) - 1u))] = c;
        nk += __popc(bal);
      }
      __syncwarp();
      if (lane < nk) {
        const int c = s_kid[lane];
        px = s_tok[c];
        pr = a.uniforms[bm + c];
        float lx[1];
        load_vec<1>(row, px, lx);
        pl = lx[0];
        if (drow) pd = __ldg(drow + px);
      }
    }

    // this CTA's slice of the target row (scaled logits) and of the draft row (log2 units)
#pragma unroll
    for (int jc = 0; jc < NCH; ++jc) {
      const long long i0 = slice0 + (static_cast<long long>(jc) * NT + tid) * VEC;
      float v[VEC];
      if (i0 < V) {
        load_vec<VEC>(row, i0, v);
      } else {
#pragma unroll
        for (int t = 0; t < VEC; ++t) v[t] = -INFINITY;
      }
#pragma unroll
      for (int t = 0; t < VEC; ++t) pv[jc * VEC + t] = __fmul_rn(v[t], a.c);
    }
    if (drow) {
#pragma unroll
      for (int jc = 0; jc < NCH; ++jc) {
        const long long i0 = slice0 + (static_cast<long long>(jc) * NT + tid) * VEC;
        float v[VEC];
        if (i0 < V) {
          load_vec<VEC>(drow, i0, v);
        } else {
#pragma unroll
          for (int t = 0; t < VEC; ++t) v[t] = -INFINITY;
        }
#pragma unroll
        for (int t = 0; t < VEC; ++t) qv[jc * VEC + t] = __fmul_rn(v[t], kLog2e);
      }
    }
    if (warp == 0) {
      if (lane < nk) {
        s_kx[lane] = px;
        s_kr[lane] = pr;
        s_ks[lane] = __fmul_rn(pl, a.c);
        s_kd[lane] = __fmul_rn(pd, kLog2e);
      }
      for (int j = 32 + lane; j < nk; j += 32) {
        const int c = s_kid[j], x = s_tok[c];
        s_kx[j] = x;
        s_kr[j] = a.uniforms[bm + c];
        float lx[1];
        load_vec<1>(row, x, lx);
        s_ks[j] = __fmul_rn(lx[0], a.c);
        s_kd[j] = drow ? __fmul_rn(__ldg(drow + x), kLog2e) : 0.f;
      }
      if (lane == 0) st.nk = nk;
    }

    // node start: (max, sum) of the slices, merged over the cluster in rank order
    const float2 t2 = block_max_sum_t0<EPT>(pv, s_red);
    float2 q2 = make_float2(-INFINITY, 0.f);
    if (drow) q2 = block_max_sum_t0<EPT>(qv, s_red);
    if (tid == 0) s_x[xb].M = t2.x, s_x[xb].S = t2.y, s_x[xb].Mq = q2.x, s_x[xb].Sq = q2.y;
    cluster_sync_all();
    float M = 0.f, Z = 0.f, Mq = 0.f, Zq = 0.f;
    if (warp == 0) {
      const float4 f = fetch4(smem_u32(&s_x[xb]) + offsetof(Xch, M), C, make_float4(-INFINITY, 0.f, -INFINITY, 0.f));
      M = warp_max_f(f.x);
      Mq = warp_max_f(f.z);
      Z = warp_sum_f(f.x != -INFINITY ? f.y * ex2_approx(f.x - M) : 0.f);
      Zq = warp_sum_f(f.z != -INFINITY ? f.w * ex2_approx(f.z - Mq) : 0.f);
    }
    if (tid == 0) {
      st.M = M;
      st.invZ = 1.f / Z;
      st.Mq = Mq;
      st.invZq = Zq > 0.f ? 1.f / Zq : 0.f;
      st.pinv = st.invZ;
      st.acc = -1;
      st.nrej = 0;
    }
    if (warp == 0 && !a.q_draft) {
      // Point proposals: child j is kept iff r_j * Z_left(j) < e(x_j), Z_left(j) = Z minus the
      // mass of the distinct tokens rejected before it.  Lane j takes child j (32 at a time):
      // a prefix sum gives Z_left, a ballot the first kept child; a token repeated among the
      // siblings has no mass left after its first trial.
      const int nk_ = st.nk;
      float base = 0.f;
      int acc = -1, nrej = 0;
      for (int g0 = 0; g0 < nk_ && acc < 0; g0 += 32) {
        const int j = g0 + lane;
        const bool valid = j < nk_;
        const int x = valid ? s_kx[j] : -1 - lane;
        bool dup = (__match_any_sync(kFull, x) & ((1u << lane) - 1u)) != 0;
        if (valid && !dup)
          for (int r = 0; r < nrej; ++r) dup |= s_rej[r] == x;
        const float e = (valid && !dup) ? mass(s_ks[j], M) : 0.f;
        const float inc = warp_incl_scan(e);
        float exc = __shfl_up_sync(kFull, inc, 1);
        if (lane == 0) exc = 0.f;
        const float Zl = __fsub_rn(Z, __fadd_rn(base, exc));
        const unsigned kb = __ballot_sync(kFull, valid && s_kr[j] * Zl < e);
        const int first = kb ? __ffs(kb) - 1 : 32;
        const bool rej = valid && !dup && lane < first;
        const unsigned rb = __ballot_sync(kFull, rej);
        __syncwarp();
        if (rej) s_rej[nrej + __popc(rb & ((1u << lane) - 1u))] = x;
        __syncwarp();
        nrej += __popc(rb);
        base = __fadd_rn(base, __shfl_sync(kFull, inc, 31));
        if (kb) acc = g0 + first;
      }
      if (lane == 0) st.acc = acc, st.nrej = nrej;
    }
    xb ^= 1;
    __syncthreads();
    // masses in registers: pv = 2^(s - M) (p = pv / Z), qv = 2^(d - Mq)
    {
      const float M = st.M;
#pragma unroll
      for (int i = 0; i < EPT; ++i) pv[i] = mass(pv[i], M);
      if (drow) {
        const float Mq = st.Mq;
#pragma unroll
        for (int i = 0; i < EPT; ++i) qv[i] = mass(qv[i], Mq);
      }
    }

    if (draft) {  // draft proposals: one trial at a time, one residual step per rejection
      for (int j = 0; j < st.nk; ++j) {
        if (tid == 0) {
          const int x = s_kx[j];
          bool in = false;
          for (int r = 0; r < st.nrej; ++r) in |= s_rej[r] == x;
          const float p = j == 0 ? mass(s_ks[0], st.M) * st.invZ : st.pnext;
          const float q = in ? 0.f : mass(s_kd[j], st.Mq) * st.invZq;
          st.acc = s_kr[j] * q < p ? j : -1;
        }
        __syncthreads();
        if (st.acc >= 0) break;
        // rejected x: w = max(0, p - q) on the registers; x leaves the proposal
        const int x = s_kx[j];
        const bool has_next = j + 1 < st.nk;
        int rx = -1, rn = -1;
        const bool own_x = owns<VEC, EPT>(x, slice0, tid, rx);
        const bool own_n = has_next && owns<VEC, EPT>(s_kx[j + 1], slice0, tid, rn);
        const float pinv = st.pinv, invZq = st.invZq;
        float sw = 0.f, sq = 0.f, pn = 0.f, wn = 0.f;
#pragma unroll
        for (int i = 0; i < EPT; ++i) {
          const float p = pv[i] * pinv;
          const float w = fmaxf(0.f, p - qv[i] * invZq);
          sw += w;
          if (!(own_x && i == rx)) sq += qv[i];
          if (own_n && i == rn) pn = p, wn = w;
        }
        const float4 r4 = block_sum4_t0(sw, sq, pn, wn, s_red);
        if (tid == 0) s_x[xb].w = r4.x, s_x[xb].q = r4.y, s_x[xb].pnext = r4.z, s_x[xb].wnext = r4.w;
        cluster_sync_all();
        float tw = 0.f, tq = 0.f, tp = 0.f, tn = 0.f;
        if (warp == 0) {
          const float4 f = fetch4(smem_u32(&s_x[xb]) + offsetof(Xch, w), C, make_float4(0.f, 0.f, 0.f, 0.f));
          tw = warp_sum_f(f.x);
          tq = warp_sum_f(f.y);
          tp = warp_sum_f(f.z);
          tn = warp_sum_f(f.w);
        }
        if (tid == 0) {
          st.apply = tw > 0.f;  // a residual of zero mass leaves p as it was
          if (tw > 0.f) {
            st.pinv = 1.f / tw;
            st.pnext = tn / tw;
          } else {
            st.pnext = tp;
          }
          st.invZq = tq > 0.f ? 1.f / tq : 0.f;
          bool in = false;
          for (int r = 0; r < st.nrej; ++r) in |= s_rej[r] == x;
          if (!in) s_rej[st.nrej++] = x;
        }
        xb ^= 1;
        __syncthreads();
        if (st.apply) {
#pragma unroll
          for (int i = 0; i < EPT; ++i) pv[i] = fmaxf(0.f, pv[i] * pinv - qv[i] * invZq);
        }
        if (own_x) {
#pragma unroll
          for (int i = 0; i < EPT; ++i)
            if (i == rx) qv[i] = 0.f;
        }
      }
    }

    if (st.acc >= 0) {  // walk down to the kept child
      __syncthreads();
      if (tid == 0) {
        const int c = s_kid[st.acc];
        s_path[st.plen++] = c;
        st.u = c;
      }
      __syncthreads();
      continue;
    }
    break;
  }

  // ---- final draw: inverse CDF over the residual of the last node ----------------------------
  // Chunk, slice and prefix sums are float-float pairs; slices are merged in rank order.
  uint32_t ex = 0;  // point mode: this thread's registers holding tokens rejected at this node
  if (!a.q_draft) {
    for (int r = 0; r < st.nrej; ++r) {
      int reg;
      if (owns<VEC, EPT>(s_rej[r], slice0, tid, reg)) ex |= 1u << reg;
    }
  }
  bool use_excl = true;
  for (;;) {
#pragma unroll
    for (int jc = 0; jc < NCH; ++jc) {
      DF cs{0.f, 0.f};
#pragma unroll
      for (int t = 0; t < VEC; ++t) {
        const int i = jc * VEC + t;
        cs = df_add1(cs, (use_excl && ((ex >> i) & 1u)) ? 0.f : pv[i]);
      }
      cs = df_warp_sum(cs);
      if (lane == 0) s_dred[warp * NCH + jc] = cs;
    }
    __syncthreads();
    if (warp == 0) {
      DF ct{0.f, 0.f};
      if (lane < NCH)
        for (int w = 0; w < NW; ++w) ct = df_add(ct, s_dred[w * NCH + lane]);
      const DF inc = df_warp_incl_scan(ct);
      const DF exc = df_warp_excl(inc);
      if (lane < NCH) s_ct[lane] = df_to_d(ct), s_cpre[lane] = df_to_d(exc);
      const DF tot = df_shfl(inc, NCH - 1);
      if (lane == 0) s_x[xb].tot = df_to_d(tot);
    }
    cluster_sync_all();
    if (warp == 0) {  // slice totals over the cluster: fp64 scan over the ranks, then a ballot
      double f = 0.0;
      if (lane < C) f = ld_peer_f64(smem_u32(&s_x[xb]) + offsetof(Xch, tot), lane);
      const double inc = warp_incl_scan_f64(f);
      double exc = __shfl_up_sync(kFull, inc, 1);
      if (lane == 0) exc = 0.0;
      const double total = __shfl_sync(kFull, inc, 31);
      if (lane == 0) st.retry = 0, st.sel = -1;
      if (!(total > 0.0)) {
        if (lane == 0) st.retry = use_excl && !a.q_draft;  // no mass left: draw from p itself
      } else {
        double t = static_cast<double>(a.uniforms[bm]) * total;
        if (!(t < total)) t = __longlong_as_double(__double_as_longlong(total) - 1);
        // the first slice whose upper bound passes t, else the last one with mass
        const bool has = lane < C && f > 0.0;
        const unsigned hp = __ballot_sync(kFull, has && inc > t), hh = __ballot_sync(kFull, has);
        const int sel = hp ? __ffs(hp) - 1 : 31 - __clz(hh);
        const double pre_sel = __shfl_sync(kFull, exc, sel);
        if (lane == 0) st.sel = sel, st.tl = t - pre_sel;
      }
    }
    xb ^= 1;
    __syncthreads();
    if (!st.retry) break;
    use_excl = false;
  }

  if (static_cast<int>(rank) == st.sel) {  // this CTA's slice holds the draw
    if (tid == 0) s_y = 0x7fffffff, s_last = -1;
    if (warp == 0) {
      const double tl = st.tl;
      const bool has = lane < NCH && s_ct[lane] > 0.0;
      const bool pass = has && s_cpre[lane] + s_ct[lane] > tl;
      const unsigned hp = __ballot_sync(kFull, pass), hh = __ballot_sync(kFull, has);
      const int ch = hp ? __ffs(hp) - 1 : (hh ? 31 - __clz(hh) : 0);
      if (lane == 0) st.chunk = ch, st.tc = tl - s_cpre[ch];
    }
    __syncthreads();
    const int ch = st.chunk;
    const double tc = st.tc;
    const long long id0 = slice0 + (static_cast<long long>(ch) * NT + tid) * VEC;
    float v[VEC];
#pragma unroll
    for (int t = 0; t < VEC; ++t) v[t] = 0.f;
#pragma unroll
    for (int jc = 0; jc < NCH; ++jc) {
      if (jc == ch) {
#pragma unroll
        for (int t = 0; t < VEC; ++t) {
          const int i = jc * VEC + t;
          v[t] = (use_excl && ((ex >> i) & 1u)) ? 0.f : pv[i];
        }
      }
    }
    DF mine{0.f, 0.f};
    int lastnz = -1;
#pragma unroll
    for (int t = 0; t < VEC; ++t) {
      mine = df_add1(mine, v[t]);
      if (v[t] > 0.f) lastnz = static_cast<int>(id0 + t);
    }
    const DF inc = df_warp_incl_scan(mine);
    const DF exc = df_warp_excl(inc);
    if (lane == 31) s_dred[warp] = inc;
    __syncthreads();
    DF pre{0.f, 0.f};
    for (int w = 0; w < warp; ++w) pre = df_add(pre, s_dred[w]);
    pre = df_add(pre, exc);
    if (lastnz >= 0) atomicMax(&s_last, lastnz);
    if (lastnz >= 0 && df_to_d(pre) <= tc && df_to_d(df_add(pre, mine)) > tc) {
      DF acc = pre;
      int y = -1;
#pragma unroll
      for (int t = 0; t < VEC; ++t) {
        acc = df_add1(acc, v[t]);
        if (y < 0 && df_to_d(acc) > tc) y = static_cast<int>(id0 + t);
      }
      atomicMin(&s_y, y >= 0 ? y : lastnz);
    }
    __syncthreads();
    if (tid == 0) {
      const int y = s_y != 0x7fffffff ? s_y : s_last;
      a.bonus[b] = y;
      if (y < 0) report(a.dev_status, TS_ERR_DEVICE_CHECK);
    }
  }
  if (rank == 0) {
    if (tid == 0) {
      a.accept_len[b] = st.plen;
      if (st.sel < 0) {  // the target row had no mass
        a.bonus[b] = -1;
        report(a.dev_status, TS_ERR_DEVICE_CHECK);
      }
    }
    for (int i = tid; i < m; i += NT) a.accept_path[bm + i] = i < st.plen ? s_path[i] : -1;
  }
  cluster_sync_all();  // no CTA leaves while a peer may still read its exchange record
}

template <typename T, int VEC, int EPT>
int launch_cluster(const SampleArgs& a, int B, int C, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(B) * C);
  cfg.blockDim = dim3(cl::NT);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = C;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  if (cudaLaunchKernelEx(&cfg, sample_cluster_kernel<T, VEC, EPT>, a, C) != cudaSuccess) return TS_ERR_CUDA;
  count_launches(1);
  return TS_OK;
}

// Registers per thread and cluster size for a vocabulary: the smallest EPT whose cluster of
// at most CMAX CTAs covers V.
template <typename T, int VEC>
int dispatch_cluster(const SampleArgs& a, int B, cudaStream_t stream) {
  const int V = a.V;
  if (V <= cl::CMAX * cl::NT * 8) return launch_cluster<T, VEC, 8>(a, B, (V + cl::NT * 8 - 1) / (cl::NT * 8), stream);
  if (V <= cl::CMAX * cl::NT * 16)
    return launch_cluster<T, VEC, 16>(a, B, (V + cl::NT * 16 - 1) / (cl::NT * 16), stream);
  return launch_cluster<T, VEC, 32>(a, B, (V + cl::NT * 32 - 1) / (cl::NT * 32), stream);
}


template <typename T, int VEC>
int launch_one(const SampleArgs& a, int B, cudaStream_t stream) {
  const size_t smem = static_cast<size_t>((a.V + 31) / 32) * 4;
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(once, [] {
    attr_err = cudaFuncSetAttribute(sample_kernel<T, VEC>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    kSampleMaxBitmapBytes);
  });
  if (attr_err != cudaSuccess) return TS_ERR_CUDA;
  if (launch_pdl(sample_kernel<T, VEC>, dim3(B), dim3(kThreads), smem, stream, a) != cudaSuccess)
    return TS_ERR_CUDA;
  count_launches(1);
  return TS_OK;
}

}  // namespace

size_t tree_accept_sample_workspace_bytes(int B, int V, int q_mode) {
  if (q_mode != TS_Q_DRAFT) return 0;
  const long long Vp = (V + 7LL) / 8 * 8;
  return static_cast<size_t>(B) * 2 * Vp * sizeof(float) + 256;
}

int tree_accept_sample_launch(const void* logits, ts_dtype dt, const int32_t* tokens, const int32_t* parents,
                              const float* uniforms, const float* draft_logp, const int32_t* node_row, int R,
                              int B, int m, int V, float temperature, int q_mode, int32_t* accept_len,
                              int32_t* accept_path, int32_t* bonus, void* workspace, int32_t* dev_status,
                              cudaStream_t stream) {
  SampleArgs a;
  a.logits = logits;
  a.tokens = tokens;
  a.parents = parents;
  a.uniforms = uniforms;
  a.draft_logp = draft_logp;
  a.node_row = node_row;
  a.R = R;
  a.m = m;
  a.V = V;
  a.c = static_cast<float>(1.4426950408889634 / static_cast<double>(temperature));
  a.q_draft = q_mode == TS_Q_DRAFT;
  a.accept_len = accept_len;
  a.accept_path = accept_path;
  a.bonus = bonus;
  a.Vp = (V + 7LL) / 8 * 8;
  a.resid = nullptr;
  if (a.q_draft) {
    const uintptr_t p = (reinterpret_cast<uintptr_t>(workspace) + 255) & ~static_cast<uintptr_t>(255);
    a.resid = reinterpret_cast<float*>(p);
  }
  a.dev_status = dev_status;
  const bool al = (reinterpret_cast<uintptr_t>(logits) & 15) == 0 &&
                  (!a.q_draft || (reinterpret_cast<uintptr_t>(draft_logp) & 15) == 0);
  if (V <= cl::CMAX * cl::NT * cl::EPT_MAX) {  // the row fits the registers of one cluster
    if (dt == TS_BF16) {
      if (al && V % 8 == 0) return dispatch_cluster<__nv_bfloat16, 8>(a, B, stream);
      return dispatch_cluster<__nv_bfloat16, 1>(a, B, stream);
    }
    if (al && V % 4 == 0) return dispatch_cluster<float, 4>(a, B, stream);
    return dispatch_cluster<float, 1>(a, B, stream);
  }
  if (dt == TS_BF16) {
    if (al && V % 8 == 0) return launch_one<__nv_bfloat16, 8>(a, B, stream);
    return launch_one<__nv_bfloat16, 1>(a, B, stream);
  }
  if (al && V % 4 == 0) return launch_one<float, 4>(a, B, stream);
  return launch_one<float, 1>(a, B, stream);
}

}  // namespace ts
