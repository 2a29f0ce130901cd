// Internal launch entry points behind the C ABI (host side).  Arguments are already
// validated by the C-ABI layer when these are called.
#pragma once

#include <cuda_runtime.h>
#include <cstddef>
#include <cstdint>

#include "treespec.h"

namespace ts {

int device_sm_count();

size_t tree_build_workspace_bytes(int B, int V, int k, int depth, int num_sms);
int tree_build_launch(const float* draft_logp, const int32_t* root_tokens, int B, int V, int k,
                      int depth, int m, int32_t* tokens, int32_t* parents, int32_t* depth_out,
                      uint64_t* mask, double* values, int32_t* node_row, void* workspace, int32_t* dev_status,
                      cudaStream_t stream, int num_sms);

size_t tree_accept_workspace_bytes(ts_dtype dt, int B, int m, int V, int num_sms);
int tree_accept_launch(const void* logits, ts_dtype dt, const int32_t* tokens,
                       const int32_t* parents, int B, int m, int V, int32_t* argmax,
                       int32_t* accept_len, int32_t* accept_path, int32_t* bonus, void* workspace,
                       int32_t* dev_status, cudaStream_t stream, int num_sms);

struct AttnArgs {
  const void* q;
  const void* k_cache;
  const void* v_cache;
  ts_dtype dt;
  int num_blocks, block_size;
  const int32_t* block_table;
  int max_blocks;
  const int32_t* prefix_len;
  int max_prefix;
  const uint64_t* mask;
  int B, m, Hq, Hkv, d;
  float scale;
  void* out;
  float* lse;
  void* workspace;
  int32_t* dev_status;
  cudaStream_t stream;
};

// Whether the tensor-core path handles this shape (bf16, d == 128, block size 16..128).
bool attention_uses_tc(ts_dtype dt, int d, int block_size);
size_t attention_tc_workspace_bytes(int B, int m, int Hq, int Hkv, int max_prefix, int num_sms);
int attention_tc_launch(const AttnArgs& a, int num_sms);
// {row groups of 128 rows, chunks, tiles per chunk, split mode, multicast width} of the
// tensor-core launch.
void attention_tc_plan(int B, int m, int Hq, int Hkv, int max_prefix, int num_sms, int* out5);
int attention_simt_launch(const AttnArgs& a);

// accept_kernel on precomputed per-row partials (value, index) [B*m, S].
int accept_from_partials_launch(const float* part_v, const int* part_i, int S, const int32_t* tokens,
                                const int32_t* parents, int B, int m, int32_t* argmax, int32_t* accept_len,
                                int32_t* accept_path, int32_t* bonus, int32_t* dev_status, cudaStream_t stream);

// LM-head GEMM with the per-row argmax in its epilogue (lm_head.cu).
size_t lm_head_partials(int M, int N, int num_sms);
size_t lm_head_workspace_bytes(int M, int N, int num_sms);
int lm_head_partials_launch(const void* hidden, const void* weight, int M, int N, int K, float* part_v,
                            int* part_i, int* S_out, int32_t* dev_status, cudaStream_t stream, int num_sms);
int lm_head_argmax_launch(const void* hidden, const void* weight, int M, int N, int K, int32_t* argmax,
                          float* max_logit, void* workspace, int32_t* dev_status, cudaStream_t stream,
                          int num_sms);

int tree_build_from_topk_launch(const int32_t* row_tok, const float* row_logp, const int32_t* root_tokens, int B,
                                int k, int depth, int m, int32_t* tokens, int32_t* parents, int32_t* depth_out,
                                uint64_t* mask, double* values, int32_t* node_row, int32_t* dev_status,
                                cudaStream_t stream);

// Stochastic verification by multi-round rejection sampling (tree_sample.cu).
size_t tree_accept_sample_workspace_bytes(int B, int V, int q_mode);
int tree_accept_sample_launch(const void* logits, ts_dtype dt, const int32_t* tokens, const int32_t* parents,
                              const float* uniforms, const float* draft_logp, const int32_t* node_row, int R,
                              int B, int m, int V, float temperature, int q_mode, int32_t* accept_len,
                              int32_t* accept_path, int32_t* bonus, void* workspace, int32_t* dev_status,
                              cudaStream_t stream);

// Cost-aware pruning before verification (tree_prune.cu).
size_t tree_prune_workspace_bytes(int B, int m);
int tree_prune_launch(const int32_t* tokens, const int32_t* parents, const int32_t* depth, const double* values,
                      const int32_t* node_row, int B, int m, double t_draft, double t_fixed, double t_node,
                      int32_t* n_out, int32_t* tokens_out, int32_t* parents_out, int32_t* depth_out, uint64_t* mask_out,
                      double* values_out, int32_t* node_row_out, int32_t* kept_out, float* expected_out,
                      void* workspace, int32_t* dev_status, cudaStream_t stream);

// Bounded-wait self-test (selftest.cu).
int selftest_bounded_wait_launch(int mode, int32_t* result, int32_t* dev_status, cudaStream_t stream);

int efficient_head_candidates(int V, int tile_tokens, int k_tile);
size_t efficient_head_workspace_bytes(int M, int V, int rank, int tile_tokens, int k_tile);
int efficient_head_launch(const void* hidden, const void* lr_b, const void* lr_a, const void* weight, int M, int V,
                          int d, int rank, int tile_tokens, int k_tile, int k, int32_t* top_tok, float* top_logp,
                          int32_t* cand_out, void* workspace, int32_t* dev_status, cudaStream_t stream,
                          int num_sms);

int kv_commit_launch(void* k_cache, void* v_cache, ts_dtype dt, int num_blocks, int block_size,
                     int Hkv, int d, int32_t* block_table, int max_blocks, int32_t* prefix_len,
                     const int32_t* accept_path, const int32_t* accept_len, int B, int m,
                     int32_t* freed_blocks, int32_t* freed_count, int32_t* dev_status,
                     cudaStream_t stream);

}  // namespace ts
