// ts_tree_prune kernels: cost-aware pruning of the draft tree before verification.
//
// Sources: "jialefu.github.io — EAGLE-4 efficient LM head", section EAGLE-Harness (prune the
// tree from draft and target costs and the draft confidence); "rainlin.net/posts/eagle",
// sections 7.1 (value = product of the confidences on the root path) and 六 (the confidence
// tracks the acceptance rate).  Expected tokens of a tree: 1 + sum exp(value); candidate trees
// are the prefixes of the rerank order; one node count n for the batch maximises expected
// tokens per unit of round time.
//
// Three launches, chained with programmatic dependent launch:
//   prune_rank_kernel     one CTA per sequence: every non-root node's position in the rerank
//                         order (value descending, shallower, lower index; values compared as
//                         integer order keys, since this GPU's fp64 pipe is narrow), then the
//                         prefix sums of exp(value) in that order -> workspace.
//   prune_choose_kernel   one CTA: rate(n) for n = 1..m from the prefix sums; first maximum.
//   prune_compact_kernel  one CTA per sequence: the kept nodes (the root and rerank positions
//                         below n - 1) in flat order, parents re-indexed, the ancestor mask
//                         rebuilt, every row written with stride n.
#include "common.cuh"
#include "internal.h"

namespace ts {
namespace {

constexpr int kPT = 256;  // threads per CTA; m <= TS_MAX_NODES = 256
constexpr int kPW = kPT / 32;
constexpr float kLog2eP = 1.4426950408889634f;

// Unsigned order key of a double: integer order equals numeric order.
__device__ __forceinline__ uint64_t dkey(double v) {
  const uint64_t b = static_cast<uint64_t>(__double_as_longlong(v));
  return (b >> 63) ? ~b : (b | 0x8000000000000000ull);
}

// Exclusive block scan of one float per thread (fixed order); also returns the total.
__device__ __forceinline__ float block_excl_scan(float x, float* s_w, float& total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  float inc = x;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const float y = __shfl_up_sync(0xffffffffu, inc, off);
    if (lane >= off) inc = __fadd_rn(inc, y);
  }
  float exc = __shfl_up_sync(0xffffffffu, inc, 1);
  if (lane == 0) exc = 0.f;
  if (lane == 31) s_w[warp] = inc;
  __syncthreads();
  float pre = 0.f;
  total = 0.f;
  for (int w = 0; w < kPW; ++w) {
    if (w < warp) pre = __fadd_rn(pre, s_w[w]);
    total = __fadd_rn(total, s_w[w]);
  }
  __syncthreads();
  return __fadd_rn(pre, exc);
}

__global__ void __launch_bounds__(kPT) prune_rank_kernel(const int32_t* __restrict__ parents,
                                                        const int32_t* __restrict__ depth,
                                                        const double* __restrict__ values, int m,
                                                        int32_t* __restrict__ rank_ws, float* __restrict__ cum_ws,
                                                        int32_t* __restrict__ bad_ws, int32_t* status) {
  __shared__ uint64_t s_key[TS_MAX_NODES];
  __shared__ int s_dep[TS_MAX_NODES];
  __shared__ float s_e[TS_MAX_NODES];
  __shared__ float s_w[kPW];
  const int b = blockIdx.x, i = threadIdx.x;
  const long long bm = static_cast<long long>(b) * m;
  pdl_wait();
  int bad = 0;
  float e = 0.f;
  if (i < m) {
    const double v = values[bm + i];
    s_key[i] = dkey(v);
    s_dep[i] = depth[bm + i];
    const int p = parents[bm + i];
    if (i == 0 ? p != -1 : (p < 0 || p >= i)) bad = 1;
    e = ex2_approx(__fmul_rn(static_cast<float>(v), kLog2eP));
    s_e[i] = 0.f;
  }
  bad = __syncthreads_or(bad);
  // position of node i among the non-root nodes: the count of nodes before it
  int r = -1;
  if (i > 0 && i < m) {
    const uint64_t ki = s_key[i];
    const int di = s_dep[i];
    r = 0;
    for (int j = 1; j < m; ++j) {
      const uint64_t kj = s_key[j];
      r += (kj > ki) || (kj == ki && (s_dep[j] < di || (s_dep[j] == di && j < i)));
    }
    s_e[r] = e;
  }
  __syncthreads();
  // cum[k] = sum of exp(value) over the first k nodes of the order (k = 0..m-1)
  float total;
  const float x = (i < m - 1) ? s_e[i] : 0.f;
  const float pre = block_excl_scan(x, s_w, total);
  if (i < m) {
    rank_ws[bm + i] = r;
    cum_ws[bm + i] = bad ? 0.f : pre;
  }
  if (i == 0) {
    bad_ws[b] = bad;
    if (bad) report(status, TS_ERR_DEVICE_CHECK);
  }
}

// rate(n) = sum_b (1 + cum[b][n-1]) / (t_draft + t_fixed + t_node * B * n) for n = 1..m; the
// first maximum is written to n_out (sequences with a bad tree count 0 tokens).
__global__ void __launch_bounds__(kPT) prune_choose_kernel(const float* __restrict__ cum_ws,
                                                          const int32_t* __restrict__ bad_ws, int B, int m,
                                                          float t_base, float t_node_b, int32_t* __restrict__ n_out) {
  __shared__ float s_r[kPW];
  __shared__ int s_n[kPW];
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  pdl_wait();
  float rate = -1.f;
  int n = 0x7fffffff;
  if (t < m) {
    float tok = 0.f;
    for (int b = 0; b < B; ++b)
      if (!bad_ws[b]) tok = __fadd_rn(tok, __fadd_rn(1.f, cum_ws[static_cast<long long>(b) * m + t]));
    n = t + 1;
    rate = tok / (t_base + t_node_b * static_cast<float>(n));
  }
#pragma unroll
  for (int off = 16; off; off >>= 1) {
    const float r2 = __shfl_xor_sync(0xffffffffu, rate, off);
    const int n2 = __shfl_xor_sync(0xffffffffu, n, off);
    if (r2 > rate || (r2 == rate && n2 < n)) rate = r2, n = n2;
  }
  if (lane == 0) s_r[warp] = rate, s_n[warp] = n;
  __syncthreads();
  if (t == 0) {
    for (int w = 1; w < kPW; ++w)
      if (s_r[w] > rate || (s_r[w] == rate && s_n[w] < n)) rate = s_r[w], n = s_n[w];
    n_out[0] = n;
  }
}

__global__ void __launch_bounds__(kPT) prune_compact_kernel(
    const int32_t* __restrict__ tokens, const int32_t* __restrict__ parents, const int32_t* __restrict__ depth,
    const double* __restrict__ values, const int32_t* __restrict__ node_row, int m,
    const int32_t* __restrict__ rank_ws, const float* __restrict__ cum_ws, const int32_t* __restrict__ bad_ws,
    const int32_t* __restrict__ n_in, int32_t* __restrict__ tokens_out, int32_t* __restrict__ parents_out,
    int32_t* __restrict__ depth_out, uint64_t* __restrict__ mask_out, double* __restrict__ values_out,
    int32_t* __restrict__ node_row_out, int32_t* __restrict__ kept_out, float* __restrict__ expected_out,
    int32_t* status) {
  __shared__ int s_new[TS_MAX_NODES];     // old flat index -> new index (-1: pruned)
  __shared__ int s_npar[TS_MAX_NODES];    // new index -> new parent
  __shared__ int s_w[kPW];
  const int b = blockIdx.x, i = threadIdx.x, lane = i & 31, warp = i >> 5;
  const long long bm = static_cast<long long>(b) * m;
  pdl_wait();
  const int n = n_in[0];
  const int W = (n + 63) / 64;
  const long long bn = static_cast<long long>(b) * n;
  if (bad_ws[b] != 0) {  // the tree failed its checks (already reported): rows of -1
    for (int j = i; j < n; j += kPT) {
      tokens_out[bn + j] = -1, parents_out[bn + j] = -1, depth_out[bn + j] = -1, kept_out[bn + j] = -1;
      values_out[bn + j] = 0.0;
      if (node_row_out) node_row_out[bn + j] = -1;
      for (int w = 0; w < W; ++w) mask_out[(bn + j) * W + w] = 0ull;
    }
    if (i == 0) expected_out[b] = 0.f;
    return;
  }
  const int r = i < m ? rank_ws[bm + i] : 0;
  const bool kept = i < m && (i == 0 || (r >= 0 && r < n - 1));
  // new index: the kept nodes before i in flat order
  const unsigned bal = __ballot_sync(0xffffffffu, kept);
  if (lane == 0) s_w[warp] = __popc(bal);
  __syncthreads();
  int idx = __popc(bal & ((1u << lane) - 1u));
  for (int w = 0; w < warp; ++w) idx += s_w[w];
  if (i < m) s_new[i] = kept ? idx : -1;
  __syncthreads();
  int np = -1, broken = 0;
  if (kept && i > 0) {
    np = s_new[parents[bm + i]];  // parents were checked: 0 <= parent < i
    broken = np < 0;              // a kept node whose parent was pruned: a value above its parent's
  }
  if (kept) s_npar[idx] = np;
  if (__syncthreads_or(broken)) {
    if (i == 0) report(status, TS_ERR_DEVICE_CHECK);
    for (int j = i; j < n; j += kPT) {
      tokens_out[bn + j] = -1, parents_out[bn + j] = -1, depth_out[bn + j] = -1, kept_out[bn + j] = -1;
      values_out[bn + j] = 0.0;
      if (node_row_out) node_row_out[bn + j] = -1;
      for (int w = 0; w < W; ++w) mask_out[(bn + j) * W + w] = 0ull;
    }
    if (i == 0) expected_out[b] = 0.f;
    return;
  }
  if (kept) {
    tokens_out[bn + idx] = tokens[bm + i];
    parents_out[bn + idx] = np;
    depth_out[bn + idx] = depth[bm + i];
    values_out[bn + idx] = values[bm + i];
    kept_out[bn + idx] = i;
    if (node_row_out) node_row_out[bn + idx] = node_row[bm + i];
    uint64_t mw[(TS_MAX_NODES + 63) / 64] = {0ull, 0ull, 0ull, 0ull};
    for (int c = idx, hops = 0; c >= 0 && hops <= n; c = s_npar[c], ++hops) mw[c >> 6] |= 1ull << (c & 63);
    for (int w = 0; w < W; ++w) mask_out[(bn + idx) * W + w] = mw[w];
  }
  if (i == 0) expected_out[b] = __fadd_rn(1.f, cum_ws[bm + n - 1]);
}

}  // namespace

size_t tree_prune_workspace_bytes(int B, int m) {
  // rank [B, m] int32, cum [B, m] float, bad [B] int32
  return static_cast<size_t>(B) * m * 8 + static_cast<size_t>(B) * 4 + 256;
}

int tree_prune_launch(const int32_t* tokens, const int32_t* parents, const int32_t* depth, const double* values,
                      const int32_t* node_row, int B, int m, double t_draft, double t_fixed, double t_node,
                      int32_t* n_out, int32_t* tokens_out, int32_t* parents_out, int32_t* depth_out, uint64_t* mask_out,
                      double* values_out, int32_t* node_row_out, int32_t* kept_out, float* expected_out,
                      void* workspace, int32_t* dev_status, cudaStream_t stream) {
  int32_t* rank_ws = static_cast<int32_t*>(workspace);
  float* cum_ws = reinterpret_cast<float*>(rank_ws + static_cast<size_t>(B) * m);
  int32_t* bad_ws = reinterpret_cast<int32_t*>(cum_ws + static_cast<size_t>(B) * m);
  const float t_base = static_cast<float>(t_draft + t_fixed);
  const float t_node_b = static_cast<float>(t_node * B);
  if (launch_pdl(prune_rank_kernel, dim3(B), dim3(kPT), 0, stream, parents, depth, values, m, rank_ws, cum_ws, bad_ws,
                 dev_status) != cudaSuccess)
    return TS_ERR_CUDA;
  if (launch_pdl(prune_choose_kernel, dim3(1), dim3(kPT), 0, stream, static_cast<const float*>(cum_ws),
                 static_cast<const int32_t*>(bad_ws), B, m, t_base, t_node_b, n_out) != cudaSuccess)
    return TS_ERR_CUDA;
  if (launch_pdl(prune_compact_kernel, dim3(B), dim3(kPT), 0, stream, tokens, parents, depth, values, node_row, m,
                 static_cast<const int32_t*>(rank_ws), static_cast<const float*>(cum_ws),
                 static_cast<const int32_t*>(bad_ws), static_cast<const int32_t*>(n_out), tokens_out, parents_out,
                 depth_out, mask_out, values_out, node_row_out, kept_out, expected_out, dev_status) != cudaSuccess)
    return TS_ERR_CUDA;
  count_launches(3);
  return TS_OK;
}

}  // namespace ts
