// ts_tree_build kernels: EAGLE-2 dynamic draft-tree construction.
//
// Source: "rainlin.net/posts/eagle" (EAGLE series), section 7.1 Expansion and section 7.2
// Reranking; section 四 for the flattened order and the mask; "lesty.tech — EAGLE-2 vs.
// Medusa", section 5 for the parent-walk mask.
//
// Two launches:
//   1. row_topk_kernel — the HBM stream.  One CTA per draft row [V] fp32, one warp per
//      segment; the warps share lower bounds of the row's k-th best so that almost every
//      element costs one comparison, and the row's top-k goes to the workspace.
//   2. tree_kernel — one CTA per sequence, all on chip: read each row's top-k,
//      expand layer by layer (value = parent value + log-prob, fp64, root -> leaf order),
//      pick each layer's frontier by rank, rerank every candidate with per-layer binary
//      searches, flatten by (depth, parent position, child rank), and build each node's
//      ancestor mask by walking its parent pointers.
#include <climits>
#include <cmath>

#include "common.cuh"
#include "internal.h"

namespace ts {
namespace {

constexpr int kTreeThreads = 512;

// Warp-wide sorted top-k list: lane r < k holds the r-th best (value, index); lanes >= k
// hold the sentinel (-inf, INT_MAX).  `thr_*` mirror lane k-1 (the current k-th best).
struct WarpTopk {
  float v;
  int i;
  float thr_v;
  int thr_i;
};

__device__ __forceinline__ void wtopk_init(WarpTopk& t) {
  t.v = -INFINITY;
  t.i = INT_MAX;
  t.thr_v = -INFINITY;
  t.thr_i = INT_MAX;
}

// Insert (cv, ci) (same value in every lane) into the warp list of length k.
__device__ __forceinline__ void wtopk_insert(WarpTopk& t, float cv, int ci, int k) {
  const int lane = threadIdx.x & 31;
  const unsigned gt = __ballot_sync(0xffffffffu, lane < k && better(cv, ci, t.v, t.i));
  if (gt == 0u) return;
  const int pos = __ffs(gt) - 1;  // the list is sorted, so "better than lane r" holds from pos on
  const float up_v = __shfl_up_sync(0xffffffffu, t.v, 1);
  const int up_i = __shfl_up_sync(0xffffffffu, t.i, 1);
  if (lane == pos) {
    t.v = cv;
    t.i = ci;
  } else if (lane > pos && lane < k) {
    t.v = up_v;
    t.i = up_i;
  }
  t.thr_v = __shfl_sync(0xffffffffu, t.v, k - 1);
  t.thr_i = __shfl_sync(0xffffffffu, t.i, k - 1);
}

// Offer one element per lane; the lanes whose element beats the current k-th best are
// inserted one at a time (after an insertion the threshold rises, so later lanes re-check).
__device__ __forceinline__ void wtopk_offer(WarpTopk& t, float x, int ix, int k) {
  unsigned cand = __ballot_sync(0xffffffffu, better(x, ix, t.thr_v, t.thr_i));
  while (cand) {
    const int src = __ffs(cand) - 1;
    const float cv = __shfl_sync(0xffffffffu, x, src);
    const int ci = __shfl_sync(0xffffffffu, ix, src);
    wtopk_insert(t, cv, ci, k);
    cand &= ~(1u << src);
    cand &= __ballot_sync(0xffffffffu, better(x, ix, t.thr_v, t.thr_i));
  }
}

// Monotone map of a float to an unsigned key (larger value -> larger key, -0 == +0), and back
// (the inverse returns +0 for both zeros).
__device__ __forceinline__ unsigned float_order_key(float v) {
  if (v == 0.0f) v = 0.0f;
  const unsigned b = __float_as_uint(v);
  return (b >> 31) ? ~b : (b | 0x80000000u);
}
__device__ __forceinline__ float key_to_float(unsigned key) {
  return __uint_as_float((key & 0x80000000u) ? (key & 0x7fffffffu) : ~key);
}

// 64-bit candidate key: value key in the high word, 0xffffffff - index in the low word, so that
// "larger key" is exactly better() (larger value, then smaller index).  0 = no candidate.
__device__ __forceinline__ unsigned long long cand_key(float v, int i) {
  return (static_cast<unsigned long long>(float_order_key(v)) << 32) |
         (0xffffffffu - static_cast<unsigned>(i));
}

// Merge the n (<= 32) keys buf[0..n) into the warp's sorted key list lk (lane r < k holds the
// r-th best, 0 beyond): every key's rank in the union is counted, the k best are scattered
// through `scratch` (k slots) and read back.
__device__ __forceinline__ unsigned long long merge_keys(unsigned long long lk,
                                                         const unsigned long long* buf, int n, int k,
                                                         unsigned long long* scratch, int lane) {
  const unsigned long long ck = lane < n ? buf[lane] : 0ull;
  int rc = 0, rl = lane;
#pragma unroll 8
  for (int j = 0; j < 32; ++j) {
    const unsigned long long o = __shfl_sync(0xffffffffu, ck, j);
    rc += o > ck;
    rl += o > lk;
  }
  for (int j = 0; j < k; ++j) rc += __shfl_sync(0xffffffffu, lk, j) > ck;
  if (lane < k) scratch[lane] = 0ull;
  __syncwarp();
  if (ck != 0ull && rc < k) scratch[rc] = ck;
  if (lane < k && lk != 0ull && rl < k) scratch[rl] = lk;
  __syncwarp();
  const unsigned long long r = lane < k ? scratch[lane] : 0ull;
  __syncwarp();
  return r;
}

// The J largest of the 32 lanes' keys (0 = none), in order; lane 0 stores them to dst.
__device__ __forceinline__ unsigned warp_kth_key(unsigned key, int J, unsigned* dst, int lane) {
  unsigned top = 0u;
  for (int j = 0; j < J; ++j) {
    top = __reduce_max_sync(0xffffffffu, key);
    const unsigned holders = __ballot_sync(0xffffffffu, key == top);
    if (lane == __ffs(holders) - 1) key = 0u;
    if (dst != nullptr && lane == 0) dst[j] = top;
  }
  return top;
}

// Four consecutive elements 4q..4q+3 of a row; positions at or past `end` read -inf.
template <bool VEC>
__device__ __forceinline__ float4 load_quad(const float* __restrict__ x, int q, int end) {
  const float4 neg = make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
  if (VEC) return 4 * q < end ? __ldcs(reinterpret_cast<const float4*>(x) + q) : neg;
  const int e = 4 * q;
  return make_float4(e < end ? __ldcs(x + e) : -INFINITY, e + 1 < end ? __ldcs(x + e + 1) : -INFINITY,
                     e + 2 < end ? __ldcs(x + e + 2) : -INFINITY, e + 3 < end ? __ldcs(x + e + 3) : -INFINITY);
}

// One CTA per draft row, one warp per segment of seg_len elements (a multiple of 4).  Each warp
// streams its segment four elements per lane at a time, U quads per lane per batch with the
// next batch's loads in flight while the current one is examined, and keeps a sorted warp
// top-k list.  An element is examined only if it can still reach the row's top-k: three lower
// bounds of the row's k-th best value are shared through shared memory,
//   (a) the k-th largest of all warps' top-J lane maxima over their first batch (J = ceil(k/S):
//       S*J >= k distinct elements are at least that large),
//   (b) the smallest of the warps' current J-th best values (again S*J >= k elements above it),
//   (c) the warp's own k-th best,
// and a batch is skipped with one vote when no lane's maximum reaches their maximum.  At the
// end every warp keeps only its list entries at or above the final bounds, and one warp merges
// them (rank counting on 64-bit keys) into the row's top-k.
template <bool VEC>
__global__ void __launch_bounds__(1024) row_topk_kernel(const float* __restrict__ logp, int V,
                                                        int seg_len, int k,
                                                        float* __restrict__ row_v,
                                                        int* __restrict__ row_i) {
  constexpr int U = 4;
  __shared__ unsigned s_pro[32];
  __shared__ float s_jth[32];
  __shared__ float s_kth[32];
  __shared__ unsigned long long s_surv[32 * TS_MAX_TOPK];
  __shared__ unsigned long long s_scratch[TS_MAX_TOPK];
  __shared__ int s_n;
  pdl_wait();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int S = blockDim.x >> 5;
  const int J = (k + S - 1) / S;
  const long long row = blockIdx.x;
  const float* x = logp + row * static_cast<long long>(V);
  const int begin = warp * seg_len;
  const int end = min(V, begin + seg_len);
  const int q0 = begin >> 2, q1 = (end + 3) >> 2;
  if (lane == 0) s_jth[warp] = -INFINITY;
  if (threadIdx.x == 0) s_n = 0;
  WarpTopk t;
  wtopk_init(t);
  float4 nx[U];
#pragma unroll
  for (int u = 0; u < U; ++u) nx[u] = load_quad<VEC>(x, q0 + u * 32 + lane, end);

  // (a): every warp contributes its J largest lane maxima of the first batch
  float t_pro;
  {
    float lm = -INFINITY;
#pragma unroll
    for (int u = 0; u < U; ++u) lm = fmaxf(lm, fmaxf(fmaxf(nx[u].x, nx[u].y), fmaxf(nx[u].z, nx[u].w)));
    warp_kth_key(lm == lm ? float_order_key(lm) : 0u, J, s_pro + warp * J, lane);
    __syncthreads();
    const unsigned kth = warp_kth_key(lane < S * J ? s_pro[lane] : 0u, k, nullptr, lane);
    t_pro = kth == 0u ? -INFINITY : key_to_float(kth);
  }

  float pub = -INFINITY;  // this warp's J-th best as last published
  for (int qb = q0; qb < q1; qb += U * 32) {
    float4 a[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      a[u] = nx[u];
      nx[u] = load_quad<VEC>(x, qb + (U + u) * 32 + lane, end);
    }
    // (b): the smallest J-th best over the warps
    float jm = lane < S ? *reinterpret_cast<volatile float*>(&s_jth[lane]) : INFINITY;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) jm = fminf(jm, __shfl_xor_sync(0xffffffffu, jm, off));
    const float lo = fmaxf(fmaxf(t_pro, jm), t.thr_v);
    float bm = -INFINITY;
#pragma unroll
    for (int u = 0; u < U; ++u) bm = fmaxf(bm, fmaxf(fmaxf(a[u].x, a[u].y), fmaxf(a[u].z, a[u].w)));
    if (__ballot_sync(0xffffffffu, bm >= lo) == 0u) continue;
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int q = qb + u * 32 + lane;
      const float mx = fmaxf(fmaxf(a[u].x, a[u].y), fmaxf(a[u].z, a[u].w));
      const bool hot = 4 * q < end && mx >= lo;  // (the -inf padding past the end must not enter)
      if (__ballot_sync(0xffffffffu, hot) == 0u) continue;
      unsigned cm = 0u;
      if (hot) {
        const int left = end - 4 * q;  // elements of this quad inside the segment (>= 1)
        cm = (a[u].x >= lo ? 1u : 0u) | (a[u].y >= lo && left > 1 ? 2u : 0u) |
             (a[u].z >= lo && left > 2 ? 4u : 0u) | (a[u].w >= lo && left > 3 ? 8u : 0u);
      }
      // one offer per candidate element (lanes without one offer the sentinel)
      while (__ballot_sync(0xffffffffu, cm != 0u)) {
        const int c = __ffs(cm) - 1;
        const float xv = c == 0 ? a[u].x : c == 1 ? a[u].y : c == 2 ? a[u].z : a[u].w;
        wtopk_offer(t, cm ? xv : -INFINITY, cm ? 4 * q + c : INT_MAX, k);
        cm &= cm - 1u;
      }
    }
    const float jv = __shfl_sync(0xffffffffu, t.v, J - 1);
    if (jv > pub) {
      pub = jv;
      if (lane == 0) s_jth[warp] = jv;
    }
  }

  // final bounds; the surviving list entries of all warps go to one array
  if (lane == 0) s_kth[warp] = t.thr_v;
  __syncthreads();
  {
    float jm = lane < S ? s_jth[lane] : INFINITY;
    float km = lane < S ? s_kth[lane] : -INFINITY;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      jm = fminf(jm, __shfl_xor_sync(0xffffffffu, jm, off));
      km = fmaxf(km, __shfl_xor_sync(0xffffffffu, km, off));
    }
    const float lof = fmaxf(t_pro, fmaxf(jm, km));
    const bool keep = lane < k && t.i != INT_MAX && t.v >= lof;
    const unsigned msk = __ballot_sync(0xffffffffu, keep);
    int base = 0;
    if (lane == 0 && msk != 0u) base = atomicAdd(&s_n, __popc(msk));
    base = __shfl_sync(0xffffffffu, base, 0);
    if (keep) s_surv[base + __popc(msk & ((1u << lane) - 1u))] = cand_key(t.v, t.i);
  }
  __syncthreads();
  if (warp == 0) {
    const int n = s_n;
    unsigned long long lk = 0ull;
    for (int c0 = 0; c0 < n; c0 += 32) lk = merge_keys(lk, s_surv + c0, min(32, n - c0), k, s_scratch, lane);
    if (lane < k) {
      float v = -INFINITY;
      int idx = INT_MAX;
      if (lk != 0ull) {
        idx = static_cast<int>(0xffffffffu - static_cast<unsigned>(lk));
        v = key_to_float(static_cast<unsigned>(lk >> 32));
        if (v == 0.0f) v = x[idx];  // keep the sign of a zero
      }
      row_v[row * k + lane] = v;
      row_i[row * k + lane] = idx;
    }
  }
}

// Shared-memory layout of tree_kernel (sizes depend on k, depth, R, m).
struct TreeSmem {
  int N;  // candidates
  int off_val, off_key, off_code, off_skey, off_rtok, off_rlp, off_tok, off_lrank, off_sorted;
  int off_cpar, off_flat, off_sel, off_cnt, off_par, off_err, off_slist, total;
};

__host__ __device__ inline int align8(int x) { return (x + 7) & ~7; }

__host__ __device__ inline TreeSmem tree_smem_layout(int k, int depth, int R, int m) {
  TreeSmem L;
  L.N = k + (depth - 1) * k * k;
  int o = 0;
  L.off_val = o;    o = align8(o + 8 * L.N);              // fp64 value (sum of log-probs)
  L.off_key = o;    o = align8(o + 8 * L.N);              // order-preserving integer key
  L.off_code = o;   o = align8(o + 8 * L.N);              // path code: child ranks in base k
  L.off_skey = o;   o = align8(o + 8 * L.N);              // per layer: keys in rank order
  L.off_rtok = o;   o = align8(o + 4 * R * k);            // row top-k tokens
  L.off_rlp = o;    o = align8(o + 4 * R * k);            // row top-k log-probs
  L.off_tok = o;    o = align8(o + 4 * L.N);              // candidate token
  L.off_lrank = o;  o = align8(o + 2 * L.N);              // rank within its layer
  L.off_sorted = o; o = align8(o + 2 * L.N);              // per layer: ids by rank
  L.off_cpar = o;   o = align8(o + 2 * L.N);              // parent candidate (-1 for layer 1)
  L.off_flat = o;   o = align8(o + 2 * L.N);              // flat index or -1
  L.off_sel = o;    o = align8(o + L.N);                  // selected flag
  L.off_cnt = o;    o = align8(o + 4 * (depth + 2));      // selected per layer
  L.off_par = o;    o = align8(o + 4 * m);                // flat parent
  L.off_err = o;    o = align8(o + 4);
  L.off_slist = o;  o = align8(o + 2 * (depth + 1) * m);  // per depth: its selected candidates
  L.total = o;
  return L;
}

__device__ __forceinline__ int layer_base(int l, int k) {  // first candidate id of layer l >= 1
  return l == 1 ? 0 : k + (l - 2) * k * k;
}
__device__ __forceinline__ int layer_size(int l, int k) { return l == 1 ? k : k * k; }
__device__ __forceinline__ int layer_of(int x, int k, int depth) {
  if (x < k) return 1;
  const int l = 2 + (x - k) / (k * k);
  return l > depth ? depth : l;
}

// Monotone map of a double to an unsigned key (larger value -> larger key).  -0 and +0 get
// the same key, so integer comparisons order values exactly as fp64 comparisons do.
__device__ __forceinline__ unsigned long long order_key(double v) {
  unsigned long long b = static_cast<unsigned long long>(__double_as_longlong(v));
  if ((b << 1) == 0ull) b = 0ull;  // -0 -> +0 (integer test: no fp64 compare)
  return (b >> 63) ? ~b : (b | 0x8000000000000000ull);
}

__global__ void __launch_bounds__(kTreeThreads) tree_kernel(
    const float* __restrict__ part_v, const int* __restrict__ part_i,
    const int32_t* __restrict__ root_tokens, int R, int k, int depth, int m, int W,
    int32_t* __restrict__ tokens, int32_t* __restrict__ parents, int32_t* __restrict__ depth_out,
    uint64_t* __restrict__ mask, double* __restrict__ values, int32_t* __restrict__ node_row, int32_t* status) {
  extern __shared__ __align__(16) unsigned char smem[];
  pdl_wait();
  const TreeSmem L = tree_smem_layout(k, depth, R, m);
  double* cV = reinterpret_cast<double*>(smem + L.off_val);
  unsigned long long* ckey = reinterpret_cast<unsigned long long*>(smem + L.off_key);
  unsigned long long* ccode = reinterpret_cast<unsigned long long*>(smem + L.off_code);
  unsigned long long* skey = reinterpret_cast<unsigned long long*>(smem + L.off_skey);
  int* rtok = reinterpret_cast<int*>(smem + L.off_rtok);
  float* rlp = reinterpret_cast<float*>(smem + L.off_rlp);
  int* ctok = reinterpret_cast<int*>(smem + L.off_tok);
  short* lrank = reinterpret_cast<short*>(smem + L.off_lrank);
  short* sorted = reinterpret_cast<short*>(smem + L.off_sorted);
  short* cpar = reinterpret_cast<short*>(smem + L.off_cpar);
  short* cflat = reinterpret_cast<short*>(smem + L.off_flat);
  unsigned char* sel = smem + L.off_sel;
  int* cnt = reinterpret_cast<int*>(smem + L.off_cnt);
  int* fpar = reinterpret_cast<int*>(smem + L.off_par);
  int* err = reinterpret_cast<int*>(smem + L.off_err);
  short* slist = reinterpret_cast<short*>(smem + L.off_slist);

  const int b = blockIdx.x;
  const int tid = threadIdx.x;
  const long long out0 = static_cast<long long>(b) * m;

  if (tid == 0) *err = 0;
  if (m > 1) {
    // 1. The rows' top-k lists (row_topk_kernel's output).
    for (int e = tid; e < R * k; e += kTreeThreads) {
      rlp[e] = part_v[static_cast<long long>(b) * R * k + e];
      rtok[e] = part_i[static_cast<long long>(b) * R * k + e];
    }
    for (int x = tid; x < depth + 2; x += kTreeThreads) cnt[x] = 0;
    __syncthreads();
    // every row list must be in order (value descending, ties -> lower token), as the row
    // streams and the efficient head emit them
    for (int e = tid; e < R * k; e += kTreeThreads) {
      if (e % k == 0) continue;
      if (rlp[e - 1] < rlp[e] || (rlp[e - 1] == rlp[e] && rtok[e - 1] > rtok[e])) *err = 1;
    }
    __syncthreads();
    if (*err) {
      if (tid == 0) report(status, TS_ERR_DEVICE_CHECK);
      return;
    }

    // 2. Expansion, layer by layer: value = parent value + log-prob (fp64, root -> leaf);
    //    frontier slot j of layer l-1 is the candidate of rank j in that layer.  A candidate's
    //    path code is its parent's code times k plus its child rank.
    for (int l = 1; l <= depth; ++l) {
      const int base = layer_base(l, k), n = layer_size(l, k);
      for (int t = tid; t < n; t += kTreeThreads) {
        double v;
        int tok, par;
        unsigned long long code;
        if (l == 1) {
          tok = rtok[t];
          v = 0.0 + static_cast<double>(rlp[t]);
          par = -1;
          code = static_cast<unsigned long long>(t);
        } else {
          const int j = t / k, c = t - j * k;
          par = sorted[layer_base(l - 1, k) + j];
          const int row = 1 + (l - 2) * k + j;
          tok = rtok[row * k + c];
          v = cV[par] + static_cast<double>(rlp[row * k + c]);
          code = ccode[par] * static_cast<unsigned long long>(k) + static_cast<unsigned long long>(c);
        }
        const unsigned long long key = order_key(v);
        ctok[base + t] = tok;
        cV[base + t] = v;
        ckey[base + t] = key;
        ccode[base + t] = code;
        cpar[base + t] = static_cast<short>(par);
      }
      __syncthreads();
      // rank inside the layer: value descending, ties -> lower layer-local index.  Layer 1 is
      // the root row's top-k, already in that order.  Otherwise P threads per candidate count
      // the candidates that come first, each over every P-th candidate (eight independent
      // shared loads in flight), and add up by shuffles.  (Counting with broadcast loads beat
      // per-slot searches over the sorted runs here: the layer is small and the searches'
      // dependent steps cost more than the extra comparisons.)
      if (l == 1) {
        for (int t = tid; t < n; t += kTreeThreads) {
          lrank[t] = static_cast<short>(t);
          sorted[t] = static_cast<short>(t);
          skey[t] = ckey[t];
        }
      } else {
        int P = 1;
        while (P < 32 && 2 * P * n <= kTreeThreads) P *= 2;
        for (int q0 = 0; q0 < n * P; q0 += kTreeThreads) {
          const int q = q0 + tid;
          const int t = q / P, part = q & (P - 1);
          const bool live = t < n;
          const unsigned long long kv = live ? ckey[base + t] : 0ull;
          int before = 0;
          if (live) {
            int u = part;
            for (; u + 7 * P < n; u += 8 * P) {
              unsigned long long kw[8];
#pragma unroll
              for (int e = 0; e < 8; ++e) kw[e] = ckey[base + u + e * P];
#pragma unroll
              for (int e = 0; e < 8; ++e) before += (kw[e] > kv) | ((kw[e] == kv) & (u + e * P < t));
            }
            for (; u < n; u += P) {
              const unsigned long long kw = ckey[base + u];
              before += (kw > kv) | ((kw == kv) & (u < t));
            }
          }
          for (int off = P >> 1; off > 0; off >>= 1) before += __shfl_xor_sync(0xffffffffu, before, off);
          if (live && part == 0) {
            lrank[base + t] = static_cast<short>(before);
            sorted[base + before] = static_cast<short>(base + t);
            skey[base + before] = kv;
          }
        }
      }
      __syncthreads();
    }

    // 3. Rerank: global rank = rank in own layer + for every other layer the number of
    //    its candidates that come first (higher value, or equal value and shallower), found
    //    by binary search in that layer's sorted keys; a candidate stops counting once its
    //    rank rules it out.
    for (int x = tid; x < L.N; x += kTreeThreads) {
      const int l = layer_of(x, k, depth);
      const unsigned long long kv = ckey[x];
      int g = lrank[x];
      for (int l2 = 1; l2 <= depth && g < m - 1; ++l2) {
        if (l2 == l) continue;
        const unsigned long long* keys2 = skey + layer_base(l2, k);
        const bool shallower = l2 < l;
        int lo = 0, hi = layer_size(l2, k);
        while (lo < hi) {
          const int mid = (lo + hi) >> 1;
          const unsigned long long kw = keys2[mid];
          if (shallower ? (kw >= kv) : (kw > kv)) lo = mid + 1; else hi = mid;
        }
        g += lo;
      }
      const bool s = g < m - 1;
      sel[x] = s ? 1 : 0;
      cflat[x] = -1;
      if (s) slist[l * m + atomicAdd(&cnt[l], 1)] = static_cast<short>(x);
    }
    __syncthreads();
    // connectivity: every selected node's parent must be selected
    for (int x = tid; x < L.N; x += kTreeThreads) {
      if (sel[x] && x >= k && !sel[cpar[x]]) *err = 1;
    }
    __syncthreads();
    if (*err) {
      if (tid == 0) report(status, TS_ERR_DEVICE_CHECK);
      return;
    }

    // 4. Flatten: root, then by depth, and inside a depth by (parent's flat index, child
    //    rank), which is the order of the path codes.  A node's flat index = 1 + the selected
    //    nodes of shallower depths + the selected nodes of its depth with a smaller code.
    for (int e = tid; e < depth * m; e += kTreeThreads) {
      const int l = 1 + e / m, pos = e - (l - 1) * m;
      const int nl = cnt[l];
      if (pos >= nl) continue;
      const int x = slist[l * m + pos];
      int f = 1;
      for (int l2 = 1; l2 < l; ++l2) f += cnt[l2];
      const unsigned long long code = ccode[x];
      const short* sl = slist + l * m;
      int q = 0;
      for (; q + 8 <= nl; q += 8) {
        short ids[8];
#pragma unroll
        for (int e2 = 0; e2 < 8; ++e2) ids[e2] = sl[q + e2];
#pragma unroll
        for (int e2 = 0; e2 < 8; ++e2) f += ccode[ids[e2]] < code ? 1 : 0;
      }
      for (; q < nl; ++q) f += ccode[sl[q]] < code ? 1 : 0;
      cflat[x] = static_cast<short>(f);
    }
    __syncthreads();
    for (int x = tid; x < L.N; x += kTreeThreads) {
      if (!sel[x]) continue;
      const int f = cflat[x];
      const int pf = x < k ? 0 : cflat[cpar[x]];
      fpar[f] = pf;
      tokens[out0 + f] = ctok[x];
      parents[out0 + f] = pf;
      const int lx = layer_of(x, k, depth);
      depth_out[out0 + f] = lx;
      if (values) values[out0 + f] = cV[x];
      // the draft row a node was expanded with: frontier slot lrank of layer lx (< depth)
      if (node_row) node_row[out0 + f] = (lx < depth && lrank[x] < k) ? 1 + (lx - 1) * k + lrank[x] : -1;
    }
  }
  if (tid == 0) {
    fpar[0] = -1;
    tokens[out0] = root_tokens[b];
    parents[out0] = -1;
    depth_out[out0] = 0;
    if (values) values[out0] = 0.0;
    if (node_row) node_row[out0] = m > 1 ? 0 : -1;
  }
  __syncthreads();
  // the next kernel's CTAs may be placed now: only the short mask pass is left
  pdl_launch_dependents();
  // 5. Mask rows: walk the parent pointers from each node to the root.
  for (int i = tid; i < m; i += kTreeThreads) {
    uint64_t w0 = 0, w1 = 0, w2 = 0, w3 = 0;
    int n = i;
    for (int steps = 0; n >= 0 && steps <= m; ++steps) {
      const uint64_t bit = 1ull << (n & 63);
      const int q = n >> 6;
      w0 |= q == 0 ? bit : 0ull;
      w1 |= q == 1 ? bit : 0ull;
      w2 |= q == 2 ? bit : 0ull;
      w3 |= q == 3 ? bit : 0ull;
      n = fpar[n];
    }
    uint64_t* dst = mask + (out0 + i) * W;
    dst[0] = w0;
    if (W > 1) dst[1] = w1;
    if (W > 2) dst[2] = w2;
    if (W > 3) dst[3] = w3;
  }
}

}  // namespace

// Warps per draft row (one CTA of S warps per row): as many as keep every row's CTA resident at
// once (at most 1024 threads per SM at 64 registers a thread), at most 32, and segments of
// about 1024 elements or more; the segment length is a multiple of 4 (16-byte loads).
static void build_plan(int B, int V, int k, int depth, int num_sms, int* S_out, int* seg_out) {
  if (num_sms < 1) num_sms = 1;
  const int R = 1 + (depth - 1) * k;
  const long long rows = static_cast<long long>(B) * R;
  const long long per_sm = (rows + num_sms - 1) / num_sms;
  int S = per_sm >= 32 ? 1 : static_cast<int>(32 / per_sm);
  const int max_by_len = (V + 1023) / 1024;
  if (S > max_by_len) S = max_by_len;
  if (S < 1) S = 1;
  int seg = (V + S - 1) / S;
  seg = (seg + 3) & ~3;
  S = (V + seg - 1) / seg;
  *S_out = S;
  *seg_out = seg;
}

size_t tree_build_workspace_bytes(int B, int V, int k, int depth, int num_sms) {
  int S, seg;
  build_plan(B, V, k, depth, num_sms, &S, &seg);
  const long long R = 1 + static_cast<long long>(depth - 1) * k;
  return static_cast<size_t>(B) * R * k * 8 + 256;  // each row's merged top-k
}

int tree_build_launch(const float* draft_logp, const int32_t* root_tokens, int B, int V, int k,
                      int depth, int m, int32_t* tokens, int32_t* parents, int32_t* depth_out,
                      uint64_t* mask, double* values, int32_t* node_row, void* workspace, int32_t* dev_status,
                      cudaStream_t stream, int num_sms) {
  const int R = 1 + (depth - 1) * k;
  int S, seg;
  build_plan(B, V, k, depth, num_sms, &S, &seg);
  const long long rows = static_cast<long long>(B) * R;
  float* part_v = static_cast<float*>(workspace);
  int* part_i = reinterpret_cast<int*>(part_v + rows * k);
  const int W = (m + 63) / 64;
  int launches = 0;
  if (m > 1) {
    const bool vec = (V % 4 == 0) && (reinterpret_cast<uintptr_t>(draft_logp) % 16 == 0);
    if (rows > 0x7fffffffLL) return TS_ERR_UNSUPPORTED;
    const dim3 grid(static_cast<unsigned>(rows)), block(32 * S);
    const cudaError_t e = vec ? launch_pdl(row_topk_kernel<true>, grid, block, 0, stream, draft_logp, V, seg, k,
                                           part_v, part_i)
                              : launch_pdl(row_topk_kernel<false>, grid, block, 0, stream, draft_logp, V, seg,
                                           k, part_v, part_i);
    if (e != cudaSuccess) return TS_ERR_CUDA;
    ++launches;
  }
  const TreeSmem L = tree_smem_layout(k, depth, R, m);
  const int smem = L.total;
  if (smem > 48 * 1024) {
    if (cudaFuncSetAttribute(tree_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) !=
        cudaSuccess)
      return TS_ERR_CUDA;
  }
  if (launch_pdl(tree_kernel, dim3(B), dim3(kTreeThreads), smem, stream, part_v, part_i, root_tokens, R, k,
                 depth, m, W, tokens, parents, depth_out, mask, values, node_row, dev_status) != cudaSuccess)
    return TS_ERR_CUDA;
  ++launches;
  count_launches(launches);
  return cudaGetLastError() == cudaSuccess ? TS_OK : TS_ERR_CUDA;
}


int tree_build_from_topk_launch(const int32_t* row_tok, const float* row_logp, const int32_t* root_tokens, int B,
                                int k, int depth, int m, int32_t* tokens, int32_t* parents, int32_t* depth_out,
                                uint64_t* mask, double* values, int32_t* node_row, int32_t* dev_status,
                                cudaStream_t stream) {
  const int R = 1 + (depth - 1) * k;
  const int W = (m + 63) / 64;
  const TreeSmem L = tree_smem_layout(k, depth, R, m);
  if (L.total > 48 * 1024 &&
      cudaFuncSetAttribute(tree_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, L.total) != cudaSuccess)
    return TS_ERR_CUDA;
  if (launch_pdl(tree_kernel, dim3(B), dim3(kTreeThreads), L.total, stream, row_logp, row_tok, root_tokens, R, k,
                 depth, m, W, tokens, parents, depth_out, mask, values, node_row, dev_status) != cudaSuccess)
    return TS_ERR_CUDA;
  count_launches(1);
  return TS_OK;
}
}  // namespace ts
