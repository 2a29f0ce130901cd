// ts_tree_build kernels: EAGLE-2 dynamic draft-tree construction.
//
// Source: "rainlin.net/posts/eagle" (EAGLE series), section 7.1 Expansion and section 7.2
// Reranking; section 四 for the flattened order and the mask; "lesty.tech — EAGLE-2 vs.
// Medusa", section 5 for the parent-walk mask.
//
// Two launches:
//   1. row_topk_kernel — the HBM stream.  Every draft row [V] fp32 is split into S
//      segments; one CTA per (row, segment) keeps a per-thread sorted top-k in registers
//      while streaming the segment with 16-byte loads, then merges its 256 lists to one
//      top-k with warp shuffles.  Partials go to the workspace.
//   2. tree_kernel — one CTA per sequence, all on chip: merge each row's S partial lists,
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

constexpr int kTopkThreads = 128;
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

// Monotone map of a float to an unsigned key (larger value -> larger key, -0 == +0).
__device__ __forceinline__ unsigned float_order_key(float v) {
  if (v == 0.0f) v = 0.0f;
  const unsigned b = __float_as_uint(v);
  return (b >> 31) ? ~b : (b | 0x80000000u);
}

// One warp per (draft row, segment); a CTA holds kTopkThreads / 32 such warps.  Each warp
// streams its segment with 16-byte loads (8 in flight per lane) through its warp top-k
// list.  A lane first tests the maximum of its 4 loaded values against the warp's current
// k-th best; only then are the 4 values offered one by one, so once the list holds good
// values an element costs about one comparison.
__global__ void __launch_bounds__(kTopkThreads) row_topk_kernel(
    const float* __restrict__ logp, int V, int seg_len, int S, int k, int vec, long long items,
    float* __restrict__ part_v, int* __restrict__ part_i) {
  const int lane = threadIdx.x & 31;
  const long long item = static_cast<long long>(blockIdx.x) * (kTopkThreads / 32) + (threadIdx.x >> 5);
  if (item >= items) return;
  const long long row = item / S;
  const int seg = static_cast<int>(item % S);
  const float* x = logp + row * static_cast<long long>(V);
  const int begin = seg * seg_len;
  const int end = min(V, begin + seg_len);
  WarpTopk t;
  wtopk_init(t);
  if (vec) {
    constexpr int U = 8;
    const float4* x4 = reinterpret_cast<const float4*>(x);
    const int b4 = begin >> 2, e4 = end >> 2;
    for (int i0 = b4; i0 < e4; i0 += U * 32) {
      float4 a[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int i = i0 + u * 32 + lane;
        a[u] = i < e4 ? __ldcs(x4 + i) : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int i = i0 + u * 32 + lane;
        const float mx = fmaxf(fmaxf(a[u].x, a[u].y), fmaxf(a[u].z, a[u].w));
        const bool hot = i < e4 && mx >= t.thr_v;
        if (__ballot_sync(0xffffffffu, hot) == 0u) continue;
        // lanes without a candidate offer the sentinel (-inf, INT_MAX), which never enters
        wtopk_offer(t, hot ? a[u].x : -INFINITY, hot ? (i << 2) : INT_MAX, k);
        wtopk_offer(t, hot ? a[u].y : -INFINITY, hot ? (i << 2) + 1 : INT_MAX, k);
        wtopk_offer(t, hot ? a[u].z : -INFINITY, hot ? (i << 2) + 2 : INT_MAX, k);
        wtopk_offer(t, hot ? a[u].w : -INFINITY, hot ? (i << 2) + 3 : INT_MAX, k);
      }
    }
  } else {
    for (int i0 = begin; i0 < end; i0 += 32) {
      const int i = i0 + lane;
      wtopk_offer(t, i < end ? __ldcs(x + i) : -INFINITY, i < end ? i : INT_MAX, k);
    }
  }
  if (lane < k) {
    const long long o = item * k + lane;
    part_v[o] = t.v;
    part_i[o] = t.i;
  }
}

// Shared-memory layout of tree_kernel (sizes depend on k, depth, R, m).
struct TreeSmem {
  int N;  // candidates
  int off_val, off_key, off_rtok, off_rlp, off_tok, off_lrank, off_sorted, off_flat, off_sel;
  int off_cntc, off_cnt, off_par, off_err, off_stage, off_racc, total;
};

__host__ __device__ inline int align8(int x) { return (x + 7) & ~7; }

__host__ __device__ inline TreeSmem tree_smem_layout(int k, int depth, int R, int m, int S) {
  TreeSmem L;
  L.N = k + (depth - 1) * k * k;
  int o = 0;
  L.off_val = o;    o = align8(o + 8 * L.N);              // fp64 value (sum of log-probs)
  L.off_key = o;    o = align8(o + 8 * L.N);              // order-preserving integer key
  L.off_rtok = o;   o = align8(o + 4 * R * k);            // row top-k tokens
  L.off_rlp = o;    o = align8(o + 4 * R * k);            // row top-k log-probs
  L.off_tok = o;    o = align8(o + 4 * L.N);              // candidate token
  L.off_lrank = o;  o = align8(o + 2 * L.N);              // rank within its layer
  L.off_sorted = o; o = align8(o + 2 * L.N);              // per layer: ids by rank
  L.off_flat = o;   o = align8(o + 2 * L.N);              // flat index or -1
  L.off_sel = o;    o = align8(o + L.N);                  // selected flag
  L.off_cntc = o;   o = align8(o + 4 * (depth + 1) * k);  // selected children per frontier slot
  L.off_cnt = o;    o = align8(o + 4 * (depth + 2));      // selected per layer
  L.off_par = o;    o = align8(o + 4 * m);                // flat parent
  L.off_err = o;    o = align8(o + 4);
  L.off_racc = o;   o = align8(o + 4 * k * k);            // rank accumulators of one layer
  L.off_stage = o;  o = align8(o + 8 * (kTreeThreads / 32) * S * k);  // per-warp partial lists
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
  if (v == 0.0) v = 0.0;
  const unsigned long long b = static_cast<unsigned long long>(__double_as_longlong(v));
  return (b >> 63) ? ~b : (b | 0x8000000000000000ull);
}

__global__ void __launch_bounds__(kTreeThreads) tree_kernel(
    const float* __restrict__ part_v, const int* __restrict__ part_i,
    const int32_t* __restrict__ root_tokens, int R, int S, int k, int depth, int m, int W,
    int32_t* __restrict__ tokens, int32_t* __restrict__ parents, int32_t* __restrict__ depth_out,
    uint64_t* __restrict__ mask, double* __restrict__ values, int32_t* status) {
  extern __shared__ __align__(16) unsigned char smem[];
  const TreeSmem L = tree_smem_layout(k, depth, R, m, S);
  double* cV = reinterpret_cast<double*>(smem + L.off_val);
  unsigned long long* ckey = reinterpret_cast<unsigned long long*>(smem + L.off_key);
  int* rtok = reinterpret_cast<int*>(smem + L.off_rtok);
  float* rlp = reinterpret_cast<float*>(smem + L.off_rlp);
  int* ctok = reinterpret_cast<int*>(smem + L.off_tok);
  short* lrank = reinterpret_cast<short*>(smem + L.off_lrank);
  short* sorted = reinterpret_cast<short*>(smem + L.off_sorted);
  short* cflat = reinterpret_cast<short*>(smem + L.off_flat);
  unsigned char* sel = smem + L.off_sel;
  int* cntc = reinterpret_cast<int*>(smem + L.off_cntc);
  int* cnt = reinterpret_cast<int*>(smem + L.off_cnt);
  int* fpar = reinterpret_cast<int*>(smem + L.off_par);
  int* err = reinterpret_cast<int*>(smem + L.off_err);

  const int b = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  constexpr int nwarps = kTreeThreads / 32;
  const long long out0 = static_cast<long long>(b) * m;

  if (tid == 0) *err = 0;
  if (m > 1) {
    // 1. Merge each row's S sorted segment lists (k each) into the row's top-k.  The
    //    warp first copies the row's S*k partials to shared memory (independent loads).
    float* wv = reinterpret_cast<float*>(smem + L.off_stage) + warp * S * k;
    int* wi = reinterpret_cast<int*>(smem + L.off_stage + 4 * nwarps * S * k) + warp * S * k;
    for (int r = warp; r < R; r += nwarps) {
      const long long base = (static_cast<long long>(b) * R + r) * S * k;
      for (int e0 = lane; e0 < S * k; e0 += 8 * 32) {  // 8 independent loads in flight
        float v8[8];
        int i8[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const int e = e0 + 32 * u;
          if (e < S * k) {
            v8[u] = part_v[base + e];
            i8[u] = part_i[base + e];
          }
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const int e = e0 + 32 * u;
          if (e < S * k) {
            wv[e] = v8[u];
            wi[e] = i8[u];
          }
        }
      }
      __syncwarp();
      // k rounds: the best head among the S lists (largest value, then lowest id) is taken
      // with two warp reductions on an order-preserving 32-bit key and the id.
      int ptr = 0;
      for (int j = 0; j < k; ++j) {
        float v = -INFINITY;
        int i = INT_MAX;
        if (lane < S && ptr < k) {
          v = wv[lane * k + ptr];
          i = wi[lane * k + ptr];
        }
        const unsigned key = float_order_key(v);
        const unsigned kmax = __reduce_max_sync(0xffffffffu, key);
        const int imin = __reduce_min_sync(0xffffffffu, key == kmax ? i : INT_MAX);
        const bool win = key == kmax && i == imin;
        const int wl = __ffs(__ballot_sync(0xffffffffu, win)) - 1;
        const float best_v = __shfl_sync(0xffffffffu, v, wl < 0 ? 0 : wl);
        if (lane < S && ptr < k && win) ++ptr;
        if (lane == 0) {
          rtok[r * k + j] = imin;
          rlp[r * k + j] = best_v;
        }
      }
      __syncwarp();
    }
    for (int x = tid; x < (depth + 1) * k; x += kTreeThreads) cntc[x] = 0;
    for (int x = tid; x < depth + 2; x += kTreeThreads) cnt[x] = 0;
    __syncthreads();

    // 2. Expansion, layer by layer: value = parent value + log-prob (fp64, root -> leaf);
    //    frontier slot j of layer l-1 is the candidate of rank j in that layer.
    for (int l = 1; l <= depth; ++l) {
      const int base = layer_base(l, k), n = layer_size(l, k);
      for (int t = tid; t < n; t += kTreeThreads) {
        double v;
        int tok;
        if (l == 1) {
          tok = rtok[t];
          v = 0.0 + static_cast<double>(rlp[t]);
        } else {
          const int j = t / k, c = t % k;
          const int par = sorted[layer_base(l - 1, k) + j];
          const int row = 1 + (l - 2) * k + j;
          tok = rtok[row * k + c];
          v = cV[par] + static_cast<double>(rlp[row * k + c]);
        }
        ctok[base + t] = tok;
        cV[base + t] = v;
        ckey[base + t] = order_key(v);
        if (l > 1) reinterpret_cast<int*>(smem + L.off_racc)[t] = t % k;
      }
      __syncthreads();
      // rank inside the layer (value descending, ties -> lower layer-local index).  Layer 1
      // is the root row's top-k, already in order.  A later layer is k sorted lists (the k
      // children of each frontier slot, in child-rank order): the rank of child c of slot j
      // is c plus, for every other slot, the number of its children that come first, found
      // by a binary search; one thread per (candidate, other slot) pair.
      if (l == 1) {
        for (int t = tid; t < n; t += kTreeThreads) {
          lrank[t] = static_cast<short>(t);
          sorted[t] = static_cast<short>(t);
        }
      } else {
        int* racc = reinterpret_cast<int*>(smem + L.off_racc);
        for (int q = tid; q < n * k; q += kTreeThreads) {
          const int t = q / k, j2 = q % k, j = t / k;
          if (j2 == j) continue;
          const unsigned long long kv = ckey[base + t];
          int lo = 0, hi = k;  // children of slot j2 that come before candidate t
          while (lo < hi) {
            const int mid = (lo + hi) >> 1;
            const unsigned long long kw = ckey[base + j2 * k + mid];
            if (j2 < j ? (kw >= kv) : (kw > kv)) lo = mid + 1; else hi = mid;
          }
          if (lo) atomicAdd(&racc[t], lo);
        }
        __syncthreads();
        for (int t = tid; t < n; t += kTreeThreads) {
          const int rank = racc[t];
          lrank[base + t] = static_cast<short>(rank);
          sorted[base + rank] = static_cast<short>(base + t);
        }
      }
      __syncthreads();
    }

    // 3. Rerank: global rank = rank in own layer + for every other layer the number of
    //    its candidates that come first (higher value, or equal value and shallower),
    //    found by binary search in that layer's sorted order.
    for (int x = tid; x < L.N; x += kTreeThreads) {
      const int l = layer_of(x, k, depth);
      const unsigned long long kv = ckey[x];
      int g = lrank[x];
      for (int l2 = 1; l2 <= depth; ++l2) {
        if (l2 == l) continue;
        const int base2 = layer_base(l2, k), n2 = layer_size(l2, k);
        const bool shallower = l2 < l;
        int lo = 0, hi = n2;
        while (lo < hi) {
          const int mid = (lo + hi) >> 1;
          const unsigned long long kw = ckey[sorted[base2 + mid]];
          if (shallower ? (kw >= kv) : (kw > kv)) lo = mid + 1; else hi = mid;
        }
        g += lo;
      }
      const bool s = g < m - 1;
      sel[x] = s ? 1 : 0;
      cflat[x] = -1;
      if (s) {
        atomicAdd(&cnt[l], 1);
        const int slot = (l == 1) ? 0 : (x - layer_base(l, k)) / k;
        atomicAdd(&cntc[l * k + slot], 1);
      }
    }
    __syncthreads();
    // connectivity: every selected node's parent must be selected
    for (int x = tid; x < L.N; x += kTreeThreads) {
      if (!sel[x] || x < k) continue;
      const int l = layer_of(x, k, depth);
      const int j = (x - layer_base(l, k)) / k;
      if (!sel[sorted[layer_base(l - 1, k) + j]]) *err = 1;
    }
    __syncthreads();
    if (*err) {
      if (tid == 0) report(status, TS_ERR_DEVICE_CHECK);
      return;
    }

    // 4. Flatten: root, then by (depth, parent's flat index, child rank).  A node's
    //    position in its depth = selected children of parents placed before its parent
    //    + selected siblings of lower rank.
    int off = 1;
    for (int l = 1; l <= depth; ++l) {
      const int base = layer_base(l, k), n = layer_size(l, k);
      for (int t = tid; t < n; t += kTreeThreads) {
        const int x = base + t;
        if (!sel[x]) continue;
        const int j = (l == 1) ? 0 : t / k, c = t % k;
        int pos = 0, pf = 0;
        if (l > 1) {
          const int pbase = layer_base(l - 1, k);
          pf = cflat[sorted[pbase + j]];
          for (int j2 = 0; j2 < k; ++j2) {
            if (j2 == j || cntc[l * k + j2] == 0) continue;
            if (cflat[sorted[pbase + j2]] < pf) pos += cntc[l * k + j2];
          }
        }
        for (int c2 = 0; c2 < c; ++c2) pos += sel[base + j * k + c2];
        const int f = off + pos;
        cflat[x] = static_cast<short>(f);
        fpar[f] = pf;
        tokens[out0 + f] = ctok[x];
        parents[out0 + f] = pf;
        depth_out[out0 + f] = l;
        if (values) values[out0 + f] = cV[x];
      }
      off += cnt[l];
      __syncthreads();
    }
  }
  if (tid == 0) {
    fpar[0] = -1;
    tokens[out0] = root_tokens[b];
    parents[out0] = -1;
    depth_out[out0] = 0;
    if (values) values[out0] = 0.0;
  }
  __syncthreads();
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

// Segments per draft row (one warp each): at least 8 warps per SM when the rows allow it,
// at most 32 (one per lane of the merging warp), segment length a multiple of 4 (16-byte
// loads) and at least 1024 floats.
static void build_plan(int B, int V, int k, int depth, int num_sms, int* S_out, int* seg_out) {
  if (num_sms < 1) num_sms = 1;
  const int R = 1 + (depth - 1) * k;
  const long long rows = static_cast<long long>(B) * R;
  int S = (V + 16383) / 16384;
  const long long want = (8LL * num_sms + rows - 1) / rows;
  if (want > S) S = static_cast<int>(want);
  const int max_by_len = (V + 1023) / 1024;
  if (S > max_by_len) S = max_by_len;
  if (S > 32) S = 32;
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
  return static_cast<size_t>(B) * R * S * k * 8 + 256;
}

int tree_build_launch(const float* draft_logp, const int32_t* root_tokens, int B, int V, int k,
                      int depth, int m, int32_t* tokens, int32_t* parents, int32_t* depth_out,
                      uint64_t* mask, double* values, void* workspace, int32_t* dev_status,
                      cudaStream_t stream, int num_sms) {
  const int R = 1 + (depth - 1) * k;
  int S, seg;
  build_plan(B, V, k, depth, num_sms, &S, &seg);
  const long long rows = static_cast<long long>(B) * R;
  float* part_v = static_cast<float*>(workspace);
  int* part_i = reinterpret_cast<int*>(part_v + rows * S * k);
  const int W = (m + 63) / 64;
  int launches = 0;
  if (m > 1) {
    const int vec = (V % 4 == 0) && (reinterpret_cast<uintptr_t>(draft_logp) % 16 == 0);
    const long long grid = (rows * S + kTopkThreads / 32 - 1) / (kTopkThreads / 32);
    if (grid > 0x7fffffffLL) return TS_ERR_UNSUPPORTED;
    row_topk_kernel<<<static_cast<unsigned>(grid), kTopkThreads, 0, stream>>>(draft_logp, V, seg, S, k,
                                                                              vec, rows * S, part_v, part_i);
    ++launches;
  }
  const TreeSmem L = tree_smem_layout(k, depth, R, m, S);
  const int smem = L.total;
  if (smem > 48 * 1024) {
    if (cudaFuncSetAttribute(tree_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) !=
        cudaSuccess)
      return TS_ERR_CUDA;
  }
  tree_kernel<<<B, kTreeThreads, smem, stream>>>(part_v, part_i, root_tokens, R, S, k, depth, m,
                                                  W, tokens, parents, depth_out, mask, values,
                                                  dev_status);
  ++launches;
  count_launches(launches);
  return cudaGetLastError() == cudaSuccess ? TS_OK : TS_ERR_CUDA;
}

}  // namespace ts
