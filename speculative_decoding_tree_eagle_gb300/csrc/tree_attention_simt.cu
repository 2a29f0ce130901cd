// ts_tree_attention, CUDA-core path: fp32 inputs (any head dim <= 256) and bf16 shapes the
// tensor-core path does not take.  fp32 arithmetic and accumulation, accurate expf.
//
// Source: "rainlin.net/posts/eagle", section 四 Tree Attention (each node attends to its
// root-to-node ancestors); "lesty.tech — EAGLE-2 vs. Medusa", section 8 (the tree's K/V
// follow the committed prefix in the same paged sequence).
//
// One CTA per (query head, sequence); each warp owns one node at a time and streams the
// node's visible keys (prefix, then the mask's tree positions) with an online softmax.
// Lanes split the head dimension; the dot product is a warp-shuffle sum.
#include <cmath>

#include "common.cuh"
#include "internal.h"

namespace ts {
namespace {

constexpr int kSimtWarps = 4;

template <typename T>
__device__ __forceinline__ float ld_f(const T* p);
template <>
__device__ __forceinline__ float ld_f<float>(const float* p) { return __ldg(p); }
template <>
__device__ __forceinline__ float ld_f<__nv_bfloat16>(const __nv_bfloat16* p) {
  return __bfloat162float(*p);
}
template <typename T>
__device__ __forceinline__ void st_f(T* p, float v);
template <>
__device__ __forceinline__ void st_f<float>(float* p, float v) { *p = v; }
template <>
__device__ __forceinline__ void st_f<__nv_bfloat16>(__nv_bfloat16* p, float v) {
  *p = __float2bfloat16_rn(v);
}

template <typename T>
__global__ void __launch_bounds__(kSimtWarps * 32) tree_attn_simt_kernel(
    const T* __restrict__ q, const T* __restrict__ kc, const T* __restrict__ vc,
    const int32_t* __restrict__ block_table, int max_blocks, const int32_t* __restrict__ prefix_len,
    int max_prefix, const uint64_t* __restrict__ mask, int m, int Hq, int Hkv, int d, int bs,
    int num_blocks, float scale, T* __restrict__ out, float* __restrict__ lse, int32_t* status) {
  constexpr int DPL = 8;  // up to 256 / 32 head-dim elements per lane
  pdl_wait();
  const int h = blockIdx.x, b = blockIdx.y;
  const int g = Hq / Hkv, kh = h / g;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int L = prefix_len[b];
  if (L < 0 || L > max_prefix) {
    if (threadIdx.x == 0) report(status, TS_ERR_DEVICE_CHECK);
    return;
  }
  const int W = (m + 63) >> 6;
  for (int i = warp; i < m; i += kSimtWarps) {
    const long long qo = ((static_cast<long long>(b) * m + i) * Hq + h) * d;
    float qv[DPL], acc[DPL];
#pragma unroll
    for (int j = 0; j < DPL; ++j) {
      const int c = lane + 32 * j;
      qv[j] = c < d ? ld_f(q + qo + c) : 0.f;
      acc[j] = 0.f;
    }
    float mloc = -INFINITY, l = 0.f;
    const uint64_t* mrow = mask + (static_cast<long long>(b) * m + i) * W;
    for (int pos = 0; pos < L + m; ++pos) {
      if (pos >= L) {
        const int t = pos - L;
        if (!((mrow[t >> 6] >> (t & 63)) & 1ull)) continue;
      }
      const int e = block_table[static_cast<long long>(b) * max_blocks + pos / bs];
      if (e < 0 || e >= num_blocks) {
        if (lane == 0) report(status, TS_ERR_DEVICE_CHECK);
        continue;
      }
      const long long ko = ((static_cast<long long>(e) * Hkv + kh) * bs + pos % bs) * d;
      float s = 0.f;
#pragma unroll
      for (int j = 0; j < DPL; ++j) {
        const int c = lane + 32 * j;
        if (c < d) s = fmaf(qv[j], ld_f(kc + ko + c), s);
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
      s *= scale;
      const float mnew = fmaxf(mloc, s);
      const float corr = expf(mloc - mnew);
      const float pe = expf(s - mnew);
      l = l * corr + pe;
#pragma unroll
      for (int j = 0; j < DPL; ++j) {
        const int c = lane + 32 * j;
        if (c < d) acc[j] = acc[j] * corr + pe * ld_f(vc + ko + c);
      }
      mloc = mnew;
    }
    const float inv = 1.f / l;
#pragma unroll
    for (int j = 0; j < DPL; ++j) {
      const int c = lane + 32 * j;
      if (c < d) st_f(out + qo + c, acc[j] * inv);
    }
    if (lse != nullptr && lane == 0) lse[(static_cast<long long>(b) * m + i) * Hq + h] = mloc + logf(l);
  }
}

}  // namespace

int attention_simt_launch(const AttnArgs& a) {
  dim3 grid(a.Hq, a.B);
  if (a.dt == TS_F32) {
    launch_pdl(tree_attn_simt_kernel<float>, grid, dim3(kSimtWarps * 32), 0, a.stream,
        static_cast<const float*>(a.q), static_cast<const float*>(a.k_cache),
        static_cast<const float*>(a.v_cache), a.block_table, a.max_blocks, a.prefix_len,
        a.max_prefix, a.mask, a.m, a.Hq, a.Hkv, a.d, a.block_size, a.num_blocks, a.scale,
        static_cast<float*>(a.out), a.lse, a.dev_status);
  } else {
    launch_pdl(tree_attn_simt_kernel<__nv_bfloat16>, grid, dim3(kSimtWarps * 32), 0, a.stream,
        static_cast<const __nv_bfloat16*>(a.q), static_cast<const __nv_bfloat16*>(a.k_cache),
        static_cast<const __nv_bfloat16*>(a.v_cache), a.block_table, a.max_blocks, a.prefix_len,
        a.max_prefix, a.mask, a.m, a.Hq, a.Hkv, a.d, a.block_size, a.num_blocks, a.scale,
        static_cast<__nv_bfloat16*>(a.out), a.lse, a.dev_status);
  }
  count_launches(1);
  return cudaGetLastError() == cudaSuccess ? TS_OK : TS_ERR_CUDA;
}

}  // namespace ts
