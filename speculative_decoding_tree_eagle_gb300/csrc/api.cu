// C ABI of libtreespec.so (declared in include/treespec.h): host-side argument validation,
// workspace sizing and dispatch to the kernels.  Nothing here allocates device memory.
#include <atomic>
#include <cmath>
#include <cstdint>

#include "common.cuh"
#include "internal.h"

namespace ts {

static std::atomic<uint64_t> g_launches{0};

void count_launches(int n) { g_launches.fetch_add(static_cast<uint64_t>(n), std::memory_order_relaxed); }

int device_sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return n;
}

static bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

static int check_build(int B, int V, int k, int depth, int m) {
  if (B <= 0 || V <= 0 || k <= 0 || depth <= 0 || m <= 0) return TS_ERR_INVALID;
  if (k > TS_MAX_TOPK || depth > TS_MAX_DEPTH || m > TS_MAX_NODES) return TS_ERR_UNSUPPORTED;
  if (k > V) return TS_ERR_INVALID;
  const long long ncand = k + static_cast<long long>(depth - 1) * k * k;
  if (m - 1 > ncand) return TS_ERR_INVALID;
  const long long R = 1 + static_cast<long long>(depth - 1) * k;
  if (static_cast<long long>(B) * R * V > (1LL << 40)) return TS_ERR_UNSUPPORTED;
  return TS_OK;
}

static int check_attention(ts_dtype dt, int B, int m, int Hq, int Hkv, int d, int max_prefix) {
  if (B <= 0 || m <= 0 || Hq <= 0 || Hkv <= 0 || d <= 0 || max_prefix < 0) return TS_ERR_INVALID;
  if (dt != TS_F32 && dt != TS_BF16) return TS_ERR_INVALID;
  if (Hq % Hkv != 0) return TS_ERR_INVALID;
  if (m > TS_MAX_NODES || d > 256 || static_cast<long long>(B) * Hkv > 65535)
    return TS_ERR_UNSUPPORTED;
  return TS_OK;
}

static int check_accept(ts_dtype dt, int B, int m, int V) {
  if (B <= 0 || m <= 0 || V <= 0) return TS_ERR_INVALID;
  if (dt != TS_F32 && dt != TS_BF16) return TS_ERR_INVALID;
  if (m > TS_MAX_NODES) return TS_ERR_UNSUPPORTED;
  return TS_OK;
}

}  // namespace ts

static bool aligned16_ptr(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

extern "C" {

const char* ts_status_string(int status) {
  switch (status) {
    case TS_OK: return "TS_OK";
    case TS_ERR_INVALID: return "TS_ERR_INVALID: invalid argument";
    case TS_ERR_UNSUPPORTED: return "TS_ERR_UNSUPPORTED: size outside the supported range";
    case TS_ERR_WORKSPACE: return "TS_ERR_WORKSPACE: workspace too small";
    case TS_ERR_CUDA: return "TS_ERR_CUDA: CUDA launch or driver call failed";
    case TS_ERR_TIMEOUT: return "TS_ERR_TIMEOUT: a bounded device wait timed out";
    case TS_ERR_DEVICE_CHECK: return "TS_ERR_DEVICE_CHECK: bad input data found on the device";
    default: return "unknown ts_status";
  }
}

int ts_version(void) { return 1; }

uint64_t ts_launch_count(void) { return ts::g_launches.load(std::memory_order_relaxed); }

size_t ts_tree_build_workspace(int B, int V, int k, int depth, int m) {
  if (ts::check_build(B, V, k, depth, m) != TS_OK) return 0;
  return ts::tree_build_workspace_bytes(B, V, k, depth, ts::device_sm_count());
}

int ts_tree_build(const float* draft_logp, const int32_t* root_tokens, int B, int V, int k,
                  int depth, int m, int32_t* tokens, int32_t* parents, int32_t* depth_out,
                  uint64_t* mask, double* values, int32_t* node_row, void* workspace, size_t ws_bytes,
                  int32_t* dev_status, void* stream) {
  const int rc = ts::check_build(B, V, k, depth, m);
  if (rc != TS_OK) return rc;
  if (!draft_logp || !root_tokens || !tokens || !parents || !depth_out || !mask || !workspace)
    return TS_ERR_INVALID;
  const int sms = ts::device_sm_count();
  if (sms <= 0) return TS_ERR_CUDA;
  if (ws_bytes < ts::tree_build_workspace_bytes(B, V, k, depth, sms)) return TS_ERR_WORKSPACE;
  return ts::tree_build_launch(draft_logp, root_tokens, B, V, k, depth, m, tokens, parents,
                               depth_out, mask, values, node_row, workspace, dev_status,
                               static_cast<cudaStream_t>(stream), sms);
}

size_t ts_tree_attention_workspace(ts_dtype dt, int B, int m, int Hq, int Hkv, int d,
                                   int max_prefix) {
  if (ts::check_attention(dt, B, m, Hq, Hkv, d, max_prefix) != TS_OK) return 0;
  if (ts::attention_uses_tc(dt, d, 16))
    return ts::attention_tc_workspace_bytes(B, m, Hq, Hkv, max_prefix, ts::device_sm_count());
  return 256;
}

// num_sms <= 0: the current device's SM count, looked up only for the tensor-core path
static int attention_plan(ts_dtype dt, int B, int m, int Hq, int Hkv, int d, int max_prefix,
                          int block_size, int num_sms, int* plan_out) {
  const int rc = ts::check_attention(dt, B, m, Hq, Hkv, d, max_prefix);
  if (rc != TS_OK) return rc;
  if (!plan_out || block_size <= 0) return TS_ERR_INVALID;
  if (!ts::attention_uses_tc(dt, d, block_size)) {
    plan_out[0] = 0;
    plan_out[1] = 0;
    plan_out[2] = 1;
    plan_out[3] = 0;
    plan_out[4] = 0;
    plan_out[5] = 1;
    return TS_OK;
  }
  plan_out[0] = 1;
  ts::attention_tc_plan(B, m, Hq, Hkv, max_prefix, num_sms > 0 ? num_sms : ts::device_sm_count(), plan_out + 1);
  return TS_OK;
}

int ts_tree_attention_plan(ts_dtype dt, int B, int m, int Hq, int Hkv, int d, int max_prefix,
                           int block_size, int* plan_out) {
  return attention_plan(dt, B, m, Hq, Hkv, d, max_prefix, block_size, 0, plan_out);
}

int ts_tree_attention_plan_for_sms(ts_dtype dt, int B, int m, int Hq, int Hkv, int d, int max_prefix,
                                   int block_size, int num_sms, int* plan_out) {
  if (num_sms < 1) return TS_ERR_INVALID;
  return attention_plan(dt, B, m, Hq, Hkv, d, max_prefix, block_size, num_sms, plan_out);
}

int ts_tree_attention(const void* q, const void* k_cache, const void* v_cache, ts_dtype dt,
                      int num_blocks, int block_size, const int32_t* block_table,
                      int max_blocks, const int32_t* prefix_len, int max_prefix,
                      const uint64_t* mask, int B, int m, int Hq, int Hkv, int d,
                      float scale, void* out, float* lse, void* workspace, size_t ws_bytes,
                      int32_t* dev_status, void* stream) {
  int rc = ts::check_attention(dt, B, m, Hq, Hkv, d, max_prefix);
  if (rc != TS_OK) return rc;
  if (!q || !k_cache || !v_cache || !block_table || !prefix_len || !mask || !out)
    return TS_ERR_INVALID;
  if (num_blocks <= 0 || block_size <= 0 || max_blocks <= 0 || !std::isfinite(scale))
    return TS_ERR_INVALID;
  if (static_cast<long long>(max_blocks) * block_size < static_cast<long long>(max_prefix) + m)
    return TS_ERR_INVALID;
  ts::AttnArgs a{q, k_cache, v_cache, dt, num_blocks, block_size, block_table, max_blocks,
                 prefix_len, max_prefix, mask, B, m, Hq, Hkv, d, scale, out, lse, workspace,
                 dev_status, static_cast<cudaStream_t>(stream)};
  if (ts::attention_uses_tc(dt, d, block_size)) {
    if (!ts::aligned16(q) || !ts::aligned16(k_cache) || !ts::aligned16(v_cache) || !ts::aligned16(out))
      return TS_ERR_INVALID;
    const int sms = ts::device_sm_count();
    if (sms <= 0) return TS_ERR_CUDA;
    const size_t need = ts::attention_tc_workspace_bytes(B, m, Hq, Hkv, max_prefix, sms);
    if (need > 256 && (!workspace || ws_bytes < need)) return TS_ERR_WORKSPACE;
    if (!ts::aligned16(workspace) && need > 256) return TS_ERR_INVALID;
    return ts::attention_tc_launch(a, sms);
  }
  return ts::attention_simt_launch(a);
}

size_t ts_tree_accept_workspace(ts_dtype dt, int B, int m, int V) {
  if (ts::check_accept(dt, B, m, V) != TS_OK) return 0;
  return ts::tree_accept_workspace_bytes(dt, B, m, V, ts::device_sm_count());
}

int ts_tree_accept(const void* logits, ts_dtype dt, const int32_t* tokens,
                   const int32_t* parents, int B, int m, int V, int32_t* argmax,
                   int32_t* accept_len, int32_t* accept_path, int32_t* bonus, void* workspace,
                   size_t ws_bytes, int32_t* dev_status, void* stream) {
  const int rc = ts::check_accept(dt, B, m, V);
  if (rc != TS_OK) return rc;
  if (!logits || !tokens || !parents || !argmax || !accept_len || !accept_path || !bonus ||
      !workspace)
    return TS_ERR_INVALID;
  const int sms = ts::device_sm_count();
  if (sms <= 0) return TS_ERR_CUDA;
  if (ws_bytes < ts::tree_accept_workspace_bytes(dt, B, m, V, sms)) return TS_ERR_WORKSPACE;
  return ts::tree_accept_launch(logits, dt, tokens, parents, B, m, V, argmax, accept_len,
                                accept_path, bonus, workspace, dev_status,
                                static_cast<cudaStream_t>(stream), sms);
}

static int check_lm_head(const void* hidden, const void* weight, long long M, int N, int K) {
  if (M <= 0 || N <= 0 || K <= 0 || K % 8 != 0) return TS_ERR_INVALID;
  if (!hidden || !weight || !aligned16_ptr(hidden) || !aligned16_ptr(weight)) return TS_ERR_INVALID;
  if (M > (1LL << 24)) return TS_ERR_UNSUPPORTED;
  return TS_OK;
}

size_t ts_lm_head_argmax_workspace(int M, int N, int K) {
  if (M <= 0 || N <= 0 || K <= 0 || K % 8 != 0) return 0;
  return ts::lm_head_workspace_bytes(M, N, ts::device_sm_count());
}

int ts_lm_head_argmax(const void* hidden, const void* weight, int M, int N, int K, int32_t* argmax,
                      float* max_logit, void* workspace, size_t ws_bytes, int32_t* dev_status,
                      void* stream) {
  const int rc = check_lm_head(hidden, weight, M, N, K);
  if (rc != TS_OK) return rc;
  if (!argmax || !workspace) return TS_ERR_INVALID;
  const int sms = ts::device_sm_count();
  if (sms <= 0) return TS_ERR_CUDA;
  if (ws_bytes < ts::lm_head_workspace_bytes(M, N, sms)) return TS_ERR_WORKSPACE;
  return ts::lm_head_argmax_launch(hidden, weight, M, N, K, argmax, max_logit, workspace, dev_status,
                                   static_cast<cudaStream_t>(stream), sms);
}

size_t ts_tree_accept_hidden_workspace(int B, int m, int V, int K) {
  if (B <= 0 || m <= 0 || m > TS_MAX_NODES) return 0;
  return ts_lm_head_argmax_workspace(B * m, V, K);
}

int ts_tree_accept_hidden(const void* hidden, const void* weight, const int32_t* tokens,
                          const int32_t* parents, int B, int m, int V, int K, int32_t* argmax,
                          int32_t* accept_len, int32_t* accept_path, int32_t* bonus, void* workspace,
                          size_t ws_bytes, int32_t* dev_status, void* stream) {
  if (B <= 0 || m <= 0) return TS_ERR_INVALID;
  if (m > TS_MAX_NODES) return TS_ERR_UNSUPPORTED;
  const long long M = static_cast<long long>(B) * m;
  const int rc = check_lm_head(hidden, weight, M, V, K);
  if (rc != TS_OK) return rc;
  if (!tokens || !parents || !argmax || !accept_len || !accept_path || !bonus || !workspace)
    return TS_ERR_INVALID;
  const int sms = ts::device_sm_count();
  if (sms <= 0) return TS_ERR_CUDA;
  const int Mi = static_cast<int>(M);
  if (ws_bytes < ts::lm_head_workspace_bytes(Mi, V, sms)) return TS_ERR_WORKSPACE;
  const int G = static_cast<int>(ts::lm_head_partials(Mi, V, sms));
  float* part_v = static_cast<float*>(workspace);
  int* part_i = reinterpret_cast<int*>(part_v + M * G);
  int S = 0;
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int r1 = ts::lm_head_partials_launch(hidden, weight, Mi, V, K, part_v, part_i, &S, dev_status, st, sms);
  if (r1 != TS_OK) return r1;
  return ts::accept_from_partials_launch(part_v, part_i, S, tokens, parents, B, m, argmax, accept_len,
                                         accept_path, bonus, dev_status, st);
}

int ts_efficient_head_candidates(int V, int tile_tokens, int k_tile) {
  if (V <= 0 || tile_tokens <= 0 || tile_tokens % 256 != 0 || k_tile < 1 || k_tile > 8) return 0;
  return ts::efficient_head_candidates(V, tile_tokens, k_tile);
}

static int check_efficient_head(const void* hidden, const void* lr_b, const void* lr_a, const void* weight, int M,
                                int V, int d, int rank, int tile_tokens, int k_tile, int k) {
  if (M <= 0 || V <= 0 || d <= 0 || rank <= 0 || d % 8 != 0 || rank % 8 != 0) return TS_ERR_INVALID;
  if (tile_tokens <= 0 || tile_tokens % 256 != 0 || k_tile < 1 || k_tile > tile_tokens) return TS_ERR_INVALID;
  if (k_tile > 8 || k < 1 || k > TS_MAX_TOPK) return TS_ERR_UNSUPPORTED;
  const long long C = static_cast<long long>((V + tile_tokens - 1) / tile_tokens) * k_tile;
  if (k > C) return TS_ERR_INVALID;
  if (C * 8 > 200 * 1024 || M > 65535) return TS_ERR_UNSUPPORTED;
  if (!hidden || !lr_b || !lr_a || !weight) return TS_ERR_INVALID;
  if (!aligned16_ptr(hidden) || !aligned16_ptr(lr_b) || !aligned16_ptr(lr_a) || !aligned16_ptr(weight))
    return TS_ERR_INVALID;
  return TS_OK;
}

size_t ts_efficient_head_workspace(int M, int V, int d, int rank, int tile_tokens, int k_tile) {
  const void* p = reinterpret_cast<const void*>(static_cast<uintptr_t>(256));
  if (check_efficient_head(p, p, p, p, M, V, d, rank, tile_tokens, k_tile, 1) != TS_OK) return 0;
  return ts::efficient_head_workspace_bytes(M, V, rank, tile_tokens, k_tile);
}

int ts_efficient_head(const void* hidden, const void* lr_b, const void* lr_a, const void* weight, int M,
                      int V, int d, int rank, int tile_tokens, int k_tile, int k, int32_t* top_tok,
                      float* top_logp, int32_t* candidates, void* workspace, size_t ws_bytes,
                      int32_t* dev_status, void* stream) {
  const int rc = check_efficient_head(hidden, lr_b, lr_a, weight, M, V, d, rank, tile_tokens, k_tile, k);
  if (rc != TS_OK) return rc;
  if (!top_tok || !top_logp || !workspace) return TS_ERR_INVALID;
  if (ws_bytes < ts::efficient_head_workspace_bytes(M, V, rank, tile_tokens, k_tile)) return TS_ERR_WORKSPACE;
  const int sms = ts::device_sm_count();
  if (sms <= 0) return TS_ERR_CUDA;
  return ts::efficient_head_launch(hidden, lr_b, lr_a, weight, M, V, d, rank, tile_tokens, k_tile, k, top_tok,
                                   top_logp, candidates, workspace, dev_status, static_cast<cudaStream_t>(stream),
                                   sms);
}

int ts_tree_build_from_topk(const int32_t* row_tok, const float* row_logp, const int32_t* root_tokens,
                            int B, int k, int depth, int m, int32_t* tokens, int32_t* parents,
                            int32_t* depth_out, uint64_t* mask, double* values, int32_t* node_row,
                            int32_t* dev_status, void* stream) {
  if (B <= 0 || k <= 0 || depth <= 0 || m <= 0) return TS_ERR_INVALID;
  if (k > TS_MAX_TOPK || depth > TS_MAX_DEPTH || m > TS_MAX_NODES) return TS_ERR_UNSUPPORTED;
  const long long ncand = k + static_cast<long long>(depth - 1) * k * k;
  if (m - 1 > ncand) return TS_ERR_INVALID;
  if (!row_tok || !row_logp || !root_tokens || !tokens || !parents || !depth_out || !mask) return TS_ERR_INVALID;
  return ts::tree_build_from_topk_launch(row_tok, row_logp, root_tokens, B, k, depth, m, tokens, parents, depth_out,
                                         mask, values, node_row, dev_status, static_cast<cudaStream_t>(stream));
}

int ts_kv_commit(void* k_cache, void* v_cache, ts_dtype dt, int num_blocks, int block_size,
                 int Hkv, int d, int32_t* block_table, int max_blocks, int32_t* prefix_len,
                 const int32_t* accept_path, const int32_t* accept_len, int B, int m,
                 int32_t* freed_blocks, int32_t* freed_count, int32_t* dev_status, void* stream) {
  if (B <= 0 || m <= 0 || num_blocks <= 0 || block_size <= 0 || Hkv <= 0 || d <= 0 || max_blocks <= 0)
    return TS_ERR_INVALID;
  if (dt != TS_F32 && dt != TS_BF16) return TS_ERR_INVALID;
  if ((d * (dt == TS_BF16 ? 2 : 4)) % 4 != 0) return TS_ERR_INVALID;
  if (m > TS_MAX_NODES || B > 65535) return TS_ERR_UNSUPPORTED;
  if (!k_cache || !v_cache || !block_table || !prefix_len || !accept_path || !accept_len ||
      !freed_blocks || !freed_count)
    return TS_ERR_INVALID;
  return ts::kv_commit_launch(k_cache, v_cache, dt, num_blocks, block_size, Hkv, d, block_table,
                              max_blocks, prefix_len, accept_path, accept_len, B, m, freed_blocks,
                              freed_count, dev_status, static_cast<cudaStream_t>(stream));
}

size_t ts_tree_accept_sample_workspace(int B, int V, int q_mode) {
  if (B <= 0 || V <= 0 || (q_mode != TS_Q_POINT && q_mode != TS_Q_DRAFT)) return 0;
  return ts::tree_accept_sample_workspace_bytes(B, V, q_mode);
}

int ts_tree_accept_sample(const void* logits, ts_dtype dt, const int32_t* tokens, const int32_t* parents,
                          const float* uniforms, const float* draft_logp, const int32_t* node_row, int R,
                          int B, int m, int V, float temperature, int q_mode, int32_t* accept_len,
                          int32_t* accept_path, int32_t* bonus, void* workspace, size_t ws_bytes,
                          int32_t* dev_status, void* stream) {
  if (B <= 0 || m <= 0 || V <= 0) return TS_ERR_INVALID;
  if (dt != TS_F32 && dt != TS_BF16) return TS_ERR_INVALID;
  if (q_mode != TS_Q_POINT && q_mode != TS_Q_DRAFT) return TS_ERR_INVALID;
  if (!(temperature > 0.f) || !std::isfinite(temperature)) return TS_ERR_INVALID;
  if (m > TS_MAX_NODES || V > TS_SAMPLE_MAX_VOCAB || B > 65535) return TS_ERR_UNSUPPORTED;
  if (!logits || !tokens || !parents || !uniforms || !accept_len || !accept_path || !bonus) return TS_ERR_INVALID;
  if (q_mode == TS_Q_DRAFT && (!draft_logp || !node_row || R <= 0)) return TS_ERR_INVALID;
  const size_t need = ts::tree_accept_sample_workspace_bytes(B, V, q_mode);
  if (need > 0 && (!workspace || ws_bytes < need)) return workspace ? TS_ERR_WORKSPACE : TS_ERR_INVALID;
  return ts::tree_accept_sample_launch(logits, dt, tokens, parents, uniforms, draft_logp, node_row, R, B, m, V,
                                       temperature, q_mode, accept_len, accept_path, bonus, workspace, dev_status,
                                       static_cast<cudaStream_t>(stream));
}

size_t ts_tree_prune_workspace(int B, int m) {
  if (B <= 0 || m <= 0 || m > TS_MAX_NODES) return 0;
  return ts::tree_prune_workspace_bytes(B, m);
}

int ts_tree_prune(const int32_t* tokens, const int32_t* parents, const int32_t* depth, const double* values,
                  const int32_t* node_row, int B, int m, double t_draft, double t_fixed, double t_node,
                  int32_t* n_out, int32_t* tokens_out, int32_t* parents_out, int32_t* depth_out,
                  uint64_t* mask_out, double* values_out, int32_t* node_row_out, int32_t* kept_out,
                  float* expected_out, void* workspace, size_t ws_bytes, int32_t* dev_status, void* stream) {
  if (B <= 0 || m <= 0) return TS_ERR_INVALID;
  if (m > TS_MAX_NODES || B > 65535) return TS_ERR_UNSUPPORTED;
  if (!(t_draft >= 0.0) || !(t_fixed >= 0.0) || !(t_node >= 0.0) || !std::isfinite(t_draft) ||
      !std::isfinite(t_fixed) || !std::isfinite(t_node) || !(t_draft + t_fixed + t_node > 0.0))
    return TS_ERR_INVALID;
  if (!tokens || !parents || !depth || !values || !n_out || !tokens_out || !parents_out || !depth_out || !mask_out ||
      !values_out || !kept_out || !expected_out || !workspace)
    return TS_ERR_INVALID;
  if (node_row_out && !node_row) return TS_ERR_INVALID;
  if (ws_bytes < ts::tree_prune_workspace_bytes(B, m)) return TS_ERR_WORKSPACE;
  return ts::tree_prune_launch(tokens, parents, depth, values, node_row, B, m, t_draft, t_fixed, t_node, n_out,
                               tokens_out, parents_out, depth_out, mask_out, values_out, node_row_out, kept_out,
                               expected_out, workspace, dev_status, static_cast<cudaStream_t>(stream));
}

int ts_selftest_bounded_wait(int mode, int32_t* result, int32_t* dev_status, void* stream) {
  if ((mode != 0 && mode != 1) || !result) return TS_ERR_INVALID;
  return ts::selftest_bounded_wait_launch(mode, result, dev_status, static_cast<cudaStream_t>(stream));
}

}  // extern "C"
