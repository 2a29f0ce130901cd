// ts_tree_accept kernels: greedy verification of the draft tree.
//
// Source: "lesty.tech — EAGLE-2 vs. Medusa", section 4 (greedy acceptance: a draft token is
// kept iff it is the base model's argmax in its context); "rainlin.net/posts/eagle",
// section 3.2 (the longest valid branch is accepted).
//
// Two launches:
//   1. argmax_kernel — the HBM stream over the [B*m, V] target logits.  Each CTA reduces
//      one segment of one row with 16-byte loads (4 in flight per thread), a per-thread
//      running (max, first index), a warp-shuffle and a shared-memory reduction.  Partial
//      (value, index) pairs go to the workspace.
//   2. accept_kernel — one CTA per sequence: merge the partials of each node's row, check
//      the parent array, mark each node valid if every node on its root path carries the
//      argmax of its parent, pick the deepest valid node (ties -> lowest index) with a
//      block max over a packed key, and write the path, its length and the bonus token.
#include <cuda.h>

#include <climits>
#include <cmath>
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace ts {
namespace {

constexpr int kArgThreads = 256;
constexpr int kAcceptThreads = 256;

__device__ __forceinline__ void upd(float& bv, int& bi, float v, int i) {
  if (better(v, i, bv, bi)) {
    bv = v;
    bi = i;
  }
}

__device__ __forceinline__ void block_best(float& v, int& i) {
  __shared__ float s_v[32];
  __shared__ int s_i[32];
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    const float ov = __shfl_xor_sync(0xffffffffu, v, off);
    const int oi = __shfl_xor_sync(0xffffffffu, i, off);
    upd(v, i, ov, oi);
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) {
    s_v[warp] = v;
    s_i[warp] = i;
  }
  __syncthreads();
  if (warp == 0) {
    const int nw = blockDim.x >> 5;
    v = lane < nw ? s_v[lane] : -INFINITY;
    i = lane < nw ? s_i[lane] : INT_MAX;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, v, off);
      const int oi = __shfl_xor_sync(0xffffffffu, i, off);
      upd(v, i, ov, oi);
    }
  }
}

// Running first maximum of one thread over increasing indices: a value replaces the best
// only when it is strictly larger, so among equal values the first (lowest) index stays and
// NaN, which compares larger than nothing, is never taken.
__device__ __forceinline__ void run_max(float& bv, int& bi, float v, int i) {
  const bool gt = v > bv;
  bi = gt ? i : bi;
  bv = gt ? v : bv;
}

// The 16-byte loads a thread examines: kArgU per batch, kArgThreads apart; the next batch is
// loaded while the current one is examined (2 x kArgU x 16 B in flight per thread).  Past the
// segment end the slots hold -inf, which never replaces a best value.  The loads are issued
// as written (volatile), so the next batch's loads are not moved below the current batch's
// comparisons.
constexpr int kArgU = 4;

__device__ __forceinline__ uint4 ld_stream(const void* p) {
  uint4 v;
  asm volatile("ld.global.cs.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// After a thread's scan: if no value above -inf was seen, its answer is its first element
// that is not NaN (the maximum is -inf there, or nothing but NaN was seen and it stays unset).
template <typename LoadF>
__device__ __forceinline__ void first_not_nan(float& bv, int& bi, int begin, int end, int stride, LoadF ld) {
  if (bi != INT_MAX) return;
  for (int i = begin; i < end; i += stride) {
    const float v = ld(i);
    if (v == v) {
      bv = v;
      bi = i;
      return;
    }
  }
}

// bf16 rows: 8 values per 16-byte load, two independent running maxima (the low and the
// high four values of every load), merged at the end.
__global__ void __launch_bounds__(kArgThreads) argmax_bf16_kernel(
    const __nv_bfloat16* __restrict__ logits, int V, int seg_len, int S, int vec,
    float* __restrict__ part_v, int* __restrict__ part_i) {
  pdl_launch_dependents();
  pdl_wait();
  const long long row = blockIdx.x / S;
  const int seg = blockIdx.x % S;
  const __nv_bfloat16* x = logits + row * static_cast<long long>(V);
  const unsigned short* xs = reinterpret_cast<const unsigned short*>(x);
  const int begin = seg * seg_len, end = min(V, begin + seg_len);
  float bv = -INFINITY;
  int bi = INT_MAX;
  if (vec) {
    const uint4* x8 = reinterpret_cast<const uint4*>(x);
    const int b8 = begin >> 3, e8 = end >> 3;
    constexpr int step = kArgU * kArgThreads;
    const uint4 ninf = make_uint4(0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u);
    float bv1 = -INFINITY;
    int bi1 = INT_MAX;
    uint4 cur[kArgU], nxt[kArgU];
    int i0 = b8 + threadIdx.x;
#pragma unroll
    for (int u = 0; u < kArgU; ++u) cur[u] = i0 + u * kArgThreads < e8 ? ld_stream(x8 + i0 + u * kArgThreads) : ninf;
    for (; i0 < e8; i0 += step) {
#pragma unroll
      for (int u = 0; u < kArgU; ++u) {
        const int j = i0 + step + u * kArgThreads;
        nxt[u] = j < e8 ? ld_stream(x8 + j) : ninf;
      }
#pragma unroll
      for (int u = 0; u < kArgU; ++u) {
        const int base = (i0 + u * kArgThreads) << 3;
        run_max(bv, bi, bf16_lo(cur[u].x), base + 0);
        run_max(bv1, bi1, bf16_lo(cur[u].z), base + 4);
        run_max(bv, bi, bf16_hi(cur[u].x), base + 1);
        run_max(bv1, bi1, bf16_hi(cur[u].z), base + 5);
        run_max(bv, bi, bf16_lo(cur[u].y), base + 2);
        run_max(bv1, bi1, bf16_lo(cur[u].w), base + 6);
        run_max(bv, bi, bf16_hi(cur[u].y), base + 3);
        run_max(bv1, bi1, bf16_hi(cur[u].w), base + 7);
      }
#pragma unroll
      for (int u = 0; u < kArgU; ++u) cur[u] = nxt[u];
    }
    upd(bv, bi, bv1, bi1);
    // a thread's elements in increasing order: its loads, each load's 8 values
    if (bi == INT_MAX) {
      for (int i = b8 + threadIdx.x; i < e8 && bi == INT_MAX; i += kArgThreads)
        first_not_nan(bv, bi, i << 3, (i << 3) + 8, 1,
                      [&](int k) { return __uint_as_float(static_cast<uint32_t>(xs[k]) << 16); });
    }
  } else {
    for (int i = begin + threadIdx.x; i < end; i += kArgThreads)
      upd(bv, bi, __uint_as_float(static_cast<uint32_t>(xs[i]) << 16), i);
  }
  block_best(bv, bi);
  if (threadIdx.x == 0) {
    part_v[row * S + seg] = bv;
    part_i[row * S + seg] = bi;
  }
}

// fp32 rows: 4 values per 16-byte load, two running maxima (the first and the second pair).
__global__ void __launch_bounds__(kArgThreads) argmax_f32_kernel(
    const float* __restrict__ logits, int V, int seg_len, int S, int vec,
    float* __restrict__ part_v, int* __restrict__ part_i) {
  pdl_launch_dependents();
  pdl_wait();
  const long long row = blockIdx.x / S;
  const int seg = blockIdx.x % S;
  const float* x = logits + row * static_cast<long long>(V);
  const int begin = seg * seg_len, end = min(V, begin + seg_len);
  float bv = -INFINITY;
  int bi = INT_MAX;
  if (vec) {
    const float4* x4 = reinterpret_cast<const float4*>(x);
    const int b4 = begin >> 2, e4 = end >> 2;
    constexpr int step = kArgU * kArgThreads;
    const float4 ninf = make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
    float bv1 = -INFINITY;
    int bi1 = INT_MAX;
    float4 cur[kArgU], nxt[kArgU];
    int i0 = b4 + threadIdx.x;
    auto ldf4 = [](const float4* q) {
      const uint4 w = ld_stream(q);
      return make_float4(__uint_as_float(w.x), __uint_as_float(w.y), __uint_as_float(w.z), __uint_as_float(w.w));
    };
#pragma unroll
    for (int u = 0; u < kArgU; ++u) cur[u] = i0 + u * kArgThreads < e4 ? ldf4(x4 + i0 + u * kArgThreads) : ninf;
    for (; i0 < e4; i0 += step) {
#pragma unroll
      for (int u = 0; u < kArgU; ++u) {
        const int j = i0 + step + u * kArgThreads;
        nxt[u] = j < e4 ? ldf4(x4 + j) : ninf;
      }
#pragma unroll
      for (int u = 0; u < kArgU; ++u) {
        const int base = (i0 + u * kArgThreads) << 2;
        run_max(bv, bi, cur[u].x, base + 0);
        run_max(bv1, bi1, cur[u].z, base + 2);
        run_max(bv, bi, cur[u].y, base + 1);
        run_max(bv1, bi1, cur[u].w, base + 3);
      }
#pragma unroll
      for (int u = 0; u < kArgU; ++u) cur[u] = nxt[u];
    }
    upd(bv, bi, bv1, bi1);
    if (bi == INT_MAX) {
      for (int i = b4 + threadIdx.x; i < e4 && bi == INT_MAX; i += kArgThreads)
        first_not_nan(bv, bi, i << 2, (i << 2) + 4, 1, [&](int k) { return x[k]; });
    }
  } else {
    for (int i = begin + threadIdx.x; i < end; i += kArgThreads) upd(bv, bi, __ldcs(x + i), i);
  }
  block_best(bv, bi);
  if (threadIdx.x == 0) {
    part_v[row * S + seg] = bv;
    part_i[row * S + seg] = bi;
  }
}

__global__ void __launch_bounds__(kAcceptThreads) accept_kernel(
    const float* __restrict__ part_v, const int* __restrict__ part_i, int S,
    const int32_t* __restrict__ tokens, const int32_t* __restrict__ parents, int m,
    int32_t* __restrict__ argmax, int32_t* __restrict__ accept_len,
    int32_t* __restrict__ accept_path, int32_t* __restrict__ bonus, int32_t* status) {
  __shared__ int s_amax[TS_MAX_NODES];
  __shared__ int s_par[TS_MAX_NODES];
  __shared__ int s_tok[TS_MAX_NODES];
  __shared__ unsigned s_key[32];
  pdl_wait();
  const int b = blockIdx.x, i = threadIdx.x;
  const long long r0 = static_cast<long long>(b) * m;
  bool bad = false;
  if (i < m) {
    float bv = -INFINITY;
    int bi = INT_MAX;
#pragma unroll 4
    for (int s = 0; s < S; ++s) upd(bv, bi, part_v[(r0 + i) * S + s], part_i[(r0 + i) * S + s]);
    if (bi == INT_MAX) bi = -1;  // nothing but NaN in the row
    s_amax[i] = bi;
    argmax[r0 + i] = bi;
    const int p = parents[r0 + i];
    s_par[i] = p;
    s_tok[i] = tokens[r0 + i];
    bad = (i == 0) ? (p != -1) : (p < 0 || p >= i);
  }
  const bool any_bad = __syncthreads_or(bad);
  pdl_launch_dependents();  // only on-chip work is left
  if (any_bad) {
    if (i == 0) {
      report(status, TS_ERR_DEVICE_CHECK);
      accept_len[b] = 0;
      bonus[b] = -1;
    }
    for (int j = i; j < m; j += blockDim.x) accept_path[r0 + j] = -1;
    return;
  }
  // valid node: every node on the root path carries its parent's argmax token
  unsigned key = 0u;
  if (i < m) {
    int n = i, d = 0;
    bool ok = true;
    while (n != 0) {
      const int p = s_par[n];
      if (s_tok[n] != s_amax[p]) {
        ok = false;
        break;
      }
      n = p;
      ++d;
    }
    // deepest first, then lowest index; 0 means "not valid" (the root's key is 0xFFFF)
    if (ok) key = (static_cast<unsigned>(d) << 16) | (0xFFFFu - static_cast<unsigned>(i));
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) key = max(key, __shfl_xor_sync(0xffffffffu, key, off));
  if ((i & 31) == 0) s_key[i >> 5] = key;
  __syncthreads();
  if (i < 32) {
    key = (i < static_cast<int>(blockDim.x >> 5)) ? s_key[i] : 0u;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) key = max(key, __shfl_xor_sync(0xffffffffu, key, off));
    if (i == 0) s_key[0] = key;
  }
  __syncthreads();
  key = s_key[0];
  const int best = static_cast<int>(0xFFFFu - (key & 0xFFFFu));
  const int dbest = static_cast<int>(key >> 16);
  for (int j = dbest + 1 + i; j < m; j += blockDim.x) accept_path[r0 + j] = -1;
  if (i == 0) {
    int n = best;
    for (int j = dbest; j >= 0; --j) {
      accept_path[r0 + j] = n;
      n = s_par[n];
    }
    accept_len[b] = dbest + 1;
    bonus[b] = s_amax[best];
  }
}

}  // namespace

static void accept_plan(ts_dtype dt, int B, int m, int V, int num_sms, int* S_out, int* seg_out) {
  if (num_sms < 1) num_sms = 1;
  const long long rows = static_cast<long long>(B) * m;
  const int gran = dt == TS_BF16 ? 8 : 4;
  int S = (V + 65535) / 65536;
  const long long want = (4LL * num_sms + rows - 1) / rows;
  if (want > S) S = static_cast<int>(want);
  const int max_by_len = (V + 2047) / 2048;
  if (S > max_by_len) S = max_by_len;
  if (S < 1) S = 1;
  int seg = (V + S - 1) / S;
  seg = (seg + gran - 1) / gran * gran;
  S = (V + seg - 1) / seg;
  *S_out = S;
  *seg_out = seg;
}

int accept_from_partials_launch(const float* part_v, const int* part_i, int S, const int32_t* tokens,
                                const int32_t* parents, int B, int m, int32_t* argmax, int32_t* accept_len,
                                int32_t* accept_path, int32_t* bonus, int32_t* dev_status, cudaStream_t stream) {
  if (launch_pdl(accept_kernel, dim3(B), dim3(kAcceptThreads), 0, stream, part_v, part_i, S, tokens, parents, m,
                 argmax, accept_len, accept_path, bonus, dev_status) != cudaSuccess)
    return TS_ERR_CUDA;
  count_launches(1);
  return TS_OK;
}

size_t tree_accept_workspace_bytes(ts_dtype dt, int B, int m, int V, int num_sms) {
  int S, seg;
  accept_plan(dt, B, m, V, num_sms, &S, &seg);
  return static_cast<size_t>(B) * m * S * 8 + 256;
}

int tree_accept_launch(const void* logits, ts_dtype dt, const int32_t* tokens,
                       const int32_t* parents, int B, int m, int V, int32_t* argmax,
                       int32_t* accept_len, int32_t* accept_path, int32_t* bonus, void* workspace,
                       int32_t* dev_status, cudaStream_t stream, int num_sms) {
  int S, seg;
  accept_plan(dt, B, m, V, num_sms, &S, &seg);
  const long long rows = static_cast<long long>(B) * m;
  float* part_v = static_cast<float*>(workspace);
  int* part_i = reinterpret_cast<int*>(part_v + rows * S);
  const long long grid = rows * S;
  if (grid > 0x7fffffffLL) return TS_ERR_UNSUPPORTED;
  if (dt == TS_BF16) {
    const int vec = (V % 8 == 0) && (reinterpret_cast<uintptr_t>(logits) % 16 == 0);
    launch_pdl(argmax_bf16_kernel, dim3(static_cast<unsigned>(grid)), dim3(kArgThreads), 0, stream,
               static_cast<const __nv_bfloat16*>(logits), V, seg, S, vec, part_v, part_i);
  } else {
    const int vec = (V % 4 == 0) && (reinterpret_cast<uintptr_t>(logits) % 16 == 0);
    launch_pdl(argmax_f32_kernel, dim3(static_cast<unsigned>(grid)), dim3(kArgThreads), 0, stream,
               static_cast<const float*>(logits), V, seg, S, vec, part_v, part_i);
  }
  launch_pdl(accept_kernel, dim3(B), dim3(kAcceptThreads), 0, stream, part_v, part_i, S, tokens, parents, m,
             argmax, accept_len, accept_path, bonus, dev_status);
  count_launches(2);
  return cudaGetLastError() == cudaSuccess ? TS_OK : TS_ERR_CUDA;
}

// ---------------------------------------------------------------------------------------
// ts_tree_accept_noalloc: tree_accept with its scratch in a fixed device array.
//
// Some callers cannot allocate device memory at the moment they verify a tree: a serving
// engine that hands all free HBM to its KV-cache pool at start-up and forbids later
// cudaMalloc calls, or a plugin hosted by a framework that owns every device allocation.
// This variant needs no workspace from them: its scratch (the per-segment partial argmax
// pairs) lives in the file-scope array below, which every GPU that loads this library keeps
// until the process exits.  The device address of the array is looked up with the device
// current on the first call made in a CUDA context (a device's first call, and the first
// call after a cudaDeviceReset, which creates a new context), and cached with the context.
// ---------------------------------------------------------------------------------------
namespace {

constexpr size_t kNoAllocScratchBytes = 1u << 20;  // 1 MiB
__device__ __align__(256) unsigned char g_accept_scratch[kNoAllocScratchBytes];

constexpr int kNoAllocMaxDevices = 64;
std::mutex g_noalloc_mu;
void* g_noalloc_ptr[kNoAllocMaxDevices] = {};
unsigned long long g_noalloc_ctx_id[kNoAllocMaxDevices] = {};  // 0: no address cached

using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);

// The two driver calls that name the current context, fetched once through the runtime (the
// library links the runtime only).  A context's ID is unique for the life of the process, so
// a context made after a reset never matches an ID cached for the one it replaced, even where
// the driver hands back the same context handle.
struct CtxCalls {
  CtxGetCurrentFn get_current = nullptr;
  CtxGetIdFn get_id = nullptr;
};

const CtxCalls& ctx_calls() {
  static CtxCalls calls;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      calls.get_current = reinterpret_cast<CtxGetCurrentFn>(f);
    f = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      calls.get_id = reinterpret_cast<CtxGetIdFn>(f);
  });
  return calls;
}

// ID of the current context, 0 if the runtime has not set this thread's context up yet.
int current_ctx_id(unsigned long long* id) {
  const CtxCalls& c = ctx_calls();
  if (c.get_current == nullptr || c.get_id == nullptr) return TS_ERR_CUDA;
  CUcontext ctx = nullptr;
  if (c.get_current(&ctx) != CUDA_SUCCESS) return TS_ERR_CUDA;
  *id = 0;
  if (ctx != nullptr && c.get_id(ctx, id) != CUDA_SUCCESS) return TS_ERR_CUDA;
  return TS_OK;
}

int noalloc_scratch(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kNoAllocMaxDevices) return TS_ERR_CUDA;
  unsigned long long id = 0;
  if (current_ctx_id(&id) != TS_OK) return TS_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (id == 0 || g_noalloc_ptr[dev] == nullptr || g_noalloc_ctx_id[dev] != id) {
    // In host code the array's name is only a host-side stand-in: the kernels must get the
    // device address, which the runtime reports for the current device and context (setting
    // the context up first if needed).
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_accept_scratch) != cudaSuccess || p == nullptr) return TS_ERR_CUDA;
    if (current_ctx_id(&id) != TS_OK || id == 0) return TS_ERR_CUDA;
    g_noalloc_ptr[dev] = p;
    g_noalloc_ctx_id[dev] = id;
  }
  *out = g_noalloc_ptr[dev];
  return TS_OK;
}

}  // namespace
}  // namespace ts

extern "C" int ts_tree_accept_noalloc(const void* logits, ts_dtype dt, const int32_t* tokens,
                                      const int32_t* parents, int B, int m, int V,
                                      int32_t* argmax, int32_t* accept_len,
                                      int32_t* accept_path, int32_t* bonus,
                                      int32_t* dev_status, void* stream) {
  if (B <= 0 || m <= 0 || V <= 0 || (dt != TS_F32 && dt != TS_BF16)) return TS_ERR_INVALID;
  if (m > TS_MAX_NODES) return TS_ERR_UNSUPPORTED;
  if (!logits || !tokens || !parents || !argmax || !accept_len || !accept_path || !bonus)
    return TS_ERR_INVALID;
  const int sms = ts::device_sm_count();
  if (sms <= 0) return TS_ERR_CUDA;
  if (ts::tree_accept_workspace_bytes(dt, B, m, V, sms) > ts::kNoAllocScratchBytes)
    return TS_ERR_UNSUPPORTED;  // the request needs more scratch than the fixed array holds
  void* scratch = nullptr;
  const int rc = ts::noalloc_scratch(&scratch);
  if (rc != TS_OK) return rc;
  return ts::tree_accept_launch(logits, dt, tokens, parents, B, m, V, argmax, accept_len,
                                accept_path, bonus, scratch, dev_status,
                                static_cast<cudaStream_t>(stream), sms);
}
