// ts_kv_commit: keep the accepted path's K/V rows after a verify step and release the
// scratch pages that held only rejected tree nodes.
//
// Source: "lesty.tech — EAGLE-2 vs. Medusa", section 8 (speculative rollback: the tree's K/V
// sit in reserved scratch pages; only the accepted path survives, the block table commits
// it and the rejected pages return to the free pool).  With multi-token pages the accepted
// rows are compacted first: node accept_path[j] (logical position L + accept_path[j]) moves
// to L + j, then the pages past the committed length are released.
//
// One CTA per sequence.  A thread owns one (KV head, 16-byte column) of the rows and moves
// the accepted rows in increasing j, eight at a time (loads of a batch before its stores).
// That order never overwrites a row before it is read: a destination j is below every later
// source accept_path[j'] >= j' > j, and inside a batch every load precedes every store.
// Validation (thread-parallel) happens before anything is written; a sequence that breaks
// the contract is reported and left untouched.  The block-table and prefix-length updates
// follow a barrier, after every move has read the old table.
#include "common.cuh"
#include "internal.h"

namespace ts {
namespace {

constexpr int kCommitThreads = 512;
constexpr int kBatch = 8;
constexpr int kMaxPages = TS_MAX_NODES + 2;  // pages a tree of <= 256 nodes can touch (any page size)

template <typename Chunk>
__global__ void __launch_bounds__(kCommitThreads) kv_commit_kernel(
    unsigned char* __restrict__ kc, unsigned char* __restrict__ vc, int num_blocks, int bs, int Hkv,
    int row_bytes, int32_t* __restrict__ table, int max_blocks, int32_t* __restrict__ prefix_len,
    const int32_t* __restrict__ accept_path, const int32_t* __restrict__ accept_len, int m,
    int32_t* __restrict__ freed, int32_t* __restrict__ freed_count, int32_t* status) {
  __shared__ int s_path[TS_MAX_NODES];
  __shared__ int s_page[kMaxPages];
  pdl_wait();
  const int b = blockIdx.x, tid = threadIdx.x;
  const int L = prefix_len[b];
  const int a = accept_len[b];
  // page counts in 64 bits: a prefix length near INT_MAX must fail the max_blocks check
  const long long used64 = L >= 0 ? (static_cast<long long>(L) + m + bs - 1) / bs : 0;
  bool bad = L < 0 || a < 1 || a > m || used64 > max_blocks;
  const int n_used = bad ? 0 : static_cast<int>(used64);
  const int n_keep = bad ? 0 : static_cast<int>((static_cast<long long>(L) + a + bs - 1) / bs);
  const int p0 = bad ? 0 : L / bs;                 // first page a tree position touches
  bad = bad || n_used - p0 > kMaxPages;
  if (!bad) {
    for (int j = tid; j < a; j += blockDim.x) {
      const int pj = accept_path[static_cast<long long>(b) * m + j];
      s_path[j] = pj;
      if (j == 0 ? pj != 0 : (pj >= m || pj <= accept_path[static_cast<long long>(b) * m + j - 1])) bad = true;
    }
    for (int i = p0 + tid; i < n_used; i += blockDim.x) {
      const int pg = table[static_cast<long long>(b) * max_blocks + i];
      s_page[i - p0] = pg;
      if (pg < 0 || pg >= num_blocks) bad = true;
    }
  }
  if (__syncthreads_or(bad)) {
    // inputs untouched; the outputs still say "nothing released"
    for (int i = tid; i < max_blocks; i += blockDim.x) freed[static_cast<long long>(b) * max_blocks + i] = -1;
    if (tid == 0) {
      freed_count[b] = 0;
      report(status, TS_ERR_DEVICE_CHECK);
    }
    return;
  }
  // row moves: column c of every row = (head h, chunk q)
  const int cpr = row_bytes / static_cast<int>(sizeof(Chunk));  // chunks per head row
  const int ncol = Hkv * cpr;
  auto addr = [&](int pos, int h, int q) -> long long {
    const int page = s_page[pos / bs - p0];
    return ((static_cast<long long>(page) * Hkv + h) * bs + pos % bs) * row_bytes +
           static_cast<long long>(q) * sizeof(Chunk);
  };
  for (int c = tid; c < ncol; c += blockDim.x) {
    const int h = c / cpr, q = c - h * cpr;
    for (int j0 = 1; j0 < a; j0 += kBatch) {
      Chunk rk[kBatch], rv[kBatch];
#pragma unroll
      for (int u = 0; u < kBatch; ++u) {
        const int j = j0 + u;
        if (j < a && s_path[j] != j) {
          const long long src = addr(L + s_path[j], h, q);
          rk[u] = *reinterpret_cast<const Chunk*>(kc + src);
          rv[u] = *reinterpret_cast<const Chunk*>(vc + src);
        }
      }
#pragma unroll
      for (int u = 0; u < kBatch; ++u) {
        const int j = j0 + u;
        if (j < a && s_path[j] != j) {
          const long long dst = addr(L + j, h, q);
          *reinterpret_cast<Chunk*>(kc + dst) = rk[u];
          *reinterpret_cast<Chunk*>(vc + dst) = rv[u];
        }
      }
    }
  }
  __syncthreads();  // every move has read the old table before any entry changes
  for (int i = tid; i < max_blocks; i += blockDim.x) {
    const long long o = static_cast<long long>(b) * max_blocks;
    const int k = i + n_keep;  // logical page whose id goes to freed[i]
    if (k < n_used) {
      freed[o + i] = s_page[k - p0];
      table[o + k] = -1;
    } else {
      freed[o + i] = -1;
    }
  }
  if (tid == 0) {
    freed_count[b] = n_used > n_keep ? n_used - n_keep : 0;
    prefix_len[b] = L + a;
  }
}

}  // namespace

int kv_commit_launch(void* k_cache, void* v_cache, ts_dtype dt, int num_blocks, int block_size,
                     int Hkv, int d, int32_t* block_table, int max_blocks, int32_t* prefix_len,
                     const int32_t* accept_path, const int32_t* accept_len, int B, int m,
                     int32_t* freed_blocks, int32_t* freed_count, int32_t* dev_status,
                     cudaStream_t stream) {
  const int row_bytes = d * (dt == TS_BF16 ? 2 : 4);
  const bool wide = row_bytes % 16 == 0 && (reinterpret_cast<uintptr_t>(k_cache) % 16 == 0) &&
                    (reinterpret_cast<uintptr_t>(v_cache) % 16 == 0);
  cudaError_t e;
  if (wide)
    e = launch_pdl(kv_commit_kernel<uint4>, dim3(B), dim3(kCommitThreads), 0, stream,
                   static_cast<unsigned char*>(k_cache), static_cast<unsigned char*>(v_cache), num_blocks,
                   block_size, Hkv, row_bytes, block_table, max_blocks, prefix_len, accept_path, accept_len,
                   m, freed_blocks, freed_count, dev_status);
  else
    e = launch_pdl(kv_commit_kernel<uint32_t>, dim3(B), dim3(kCommitThreads), 0, stream,
                   static_cast<unsigned char*>(k_cache), static_cast<unsigned char*>(v_cache), num_blocks,
                   block_size, Hkv, row_bytes, block_table, max_blocks, prefix_len, accept_path, accept_len,
                   m, freed_blocks, freed_count, dev_status);
  count_launches(1);
  return e == cudaSuccess ? TS_OK : TS_ERR_CUDA;
}

}  // namespace ts
