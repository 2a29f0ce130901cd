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
// One CTA of 512 threads per sequence walks its tree.  At each visited node u:
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
// Rejected tokens of the current node are kept in a shared-memory bitmap over the vocabulary.
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
  if (dt == TS_BF16) {
    if (al && V % 8 == 0) return launch_one<__nv_bfloat16, 8>(a, B, stream);
    return launch_one<__nv_bfloat16, 1>(a, B, stream);
  }
  if (al && V % 4 == 0) return launch_one<float, 4>(a, B, stream);
  return launch_one<float, 1>(a, B, stream);
}

}  // namespace ts
