/*
 * treespec.h — C ABI of libtreespec.so: the tree-verify hot path of EAGLE-2-style
 * speculative decoding on one GB300 (sm_103a).
 *
 * Three operations, each a set of hand-written CUDA kernels:
 *   ts_tree_build      dynamic draft-tree construction (expand, rerank, flatten, mask)
 *   ts_tree_attention  every tree node attends to the paged KV prefix + its own ancestors
 *   ts_tree_accept     per-node argmax of the target logits + longest matching root path
 *   ts_tree_accept_sample  the same verification at temperature T > 0 (rejection sampling)
 *   ts_tree_prune      cost-aware pruning of the tree before verification
 *
 * Conventions shared by every entry point
 *   - Every tensor argument is a DEVICE pointer owned by the caller.  The library never
 *     allocates device memory; scratch space is the caller's `workspace`, sized by the
 *     matching *_workspace() query (any contents on entry; not zeroed by the caller).
 *   - Every call is asynchronous on `stream` (a cudaStream_t; NULL = legacy default
 *     stream) and returns after the launches are queued.
 *   - Arguments are validated on the host before anything is launched: bad sizes or null
 *     pointers return TS_ERR_INVALID, sizes outside the supported range return
 *     TS_ERR_UNSUPPORTED, a too-small workspace returns TS_ERR_WORKSPACE.  Nothing is
 *     launched in those cases.  A failed launch returns TS_ERR_CUDA.
 *   - Problems the host cannot see (a block id out of range, a parent index that does
 *     not precede its child, a prefix length above `max_prefix`, a bounded wait that
 *     timed out) are reported on the device: the first such error code is stored into
 *     `*dev_status` (an int32 device word, may be NULL to ignore) and the affected work is
 *     skipped.  Kernels never trap.  The caller zeroes *dev_status and reads it after the
 *     stream has synchronised.
 *   - The library keeps no state that affects results and is safe to call from several
 *     host threads.  It caches launch set-up per process, under locks: kernel attributes,
 *     cluster occupancy and encoded K/V tensor maps (filled by the first calls, which
 *     should come before any stream capture) and the no-allocation scratch address.  The
 *     attribute and occupancy caches assume one GPU model per process; the tested use is
 *     one process per GPU.  Calls that share a workspace must be ordered on one stream.
 *
 * Notation: B sequences, m tree nodes per sequence INCLUDING the root (node 0), k draft
 * top-k, depth draft layers below the root, V vocabulary, Hq query heads, Hkv KV heads
 * (Hq % Hkv == 0, g = Hq / Hkv), d head dim, W = ceil(m / 64) mask words per node.
 */
#ifndef TREESPEC_H
#define TREESPEC_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  TS_OK = 0,
  TS_ERR_INVALID = -1,       /* null pointer, non-positive size, inconsistent sizes */
  TS_ERR_UNSUPPORTED = -2,   /* valid but outside the supported range (limits below) */
  TS_ERR_WORKSPACE = -3,     /* workspace smaller than the *_workspace() query */
  TS_ERR_CUDA = -4,          /* a CUDA launch or driver call failed */
  TS_ERR_TIMEOUT = -5,       /* device: a bounded wait gave up (written to *dev_status) */
  TS_ERR_DEVICE_CHECK = -6   /* device: bad data found in an input (written to *dev_status) */
} ts_status;

typedef enum { TS_F32 = 0, TS_BF16 = 1 } ts_dtype;

/* Limits (host-checked).  m <= TS_MAX_NODES, k <= TS_MAX_TOPK, depth <= TS_MAX_DEPTH. */
#define TS_MAX_NODES 256
#define TS_MAX_TOPK 16
#define TS_MAX_DEPTH 16
/* ts_tree_accept_sample: V <= TS_SAMPLE_MAX_VOCAB. */
#define TS_SAMPLE_MAX_VOCAB (1 << 20)

/* Proposal q of ts_tree_accept_sample (see there). */
typedef enum { TS_Q_POINT = 0, TS_Q_DRAFT = 1 } ts_q_mode;

/* Human-readable name of a ts_status value (static string, never NULL). */
const char* ts_status_string(int status);

/* Library ABI version (this header describes version 1). */
int ts_version(void);

/* Total number of CUDA kernels this process has launched through the library so far
 * (monotonic, thread-safe; a diagnostic for counting launches around a timed region). */
uint64_t ts_launch_count(void);

/* ------------------------------------------------------------------------------------
 * ts_tree_build — EAGLE-2 dynamic draft tree.
 * Source: "rainlin.net/posts/eagle" (EAGLE series), section 7.1 Expansion (expand the top-k
 * nodes of the deepest layer by global acceptance value = product of the draft confidences
 * on the root path, kept here as a sum of log-probabilities), section 7.2 Reranking (top-m
 * of all nodes, shallower first, still a connected tree; flatten; build the mask), section 四
 * (each node sees exactly its root-to-node path); "lesty.tech — EAGLE-2 vs. Medusa",
 * section 5 (the mask from the parent array).
 *
 * draft_logp  [B, R, V] fp32, R = 1 + (depth-1)*k, row-major.  Draft log-probabilities
 *             (<= 0).  Row 0 is the root's next-token distribution; row 1 + (l-2)*k + j is
 *             the distribution after the j-th selected frontier node of layer l-1 (frontier
 *             slots in order of value, highest first).  Read only.
 * root_tokens [B] int32: token of node 0 (the last committed token).
 * k, depth, m 1 <= k <= 16, 1 <= depth <= 16, 1 <= m <= 256, m - 1 <= k + (depth-1)*k*k.
 * Outputs ([B, m] row-major unless stated):
 *   tokens    int32 token of each flattened node (node 0 = root).
 *   parents   int32 flat index of the parent, -1 for the root; parents precede children.
 *   depth_out int32 depth below the root (root 0).
 *   mask      uint64 [B, m, W]: bit (j % 64) of word j / 64 of row i is set iff node j is
 *             node i or one of its ancestors.
 *   values    fp64 (optional, NULL to skip): global value = summed log-probs, root 0.
 *   node_row  int32 [B, m] (optional, NULL to skip): the draft row each node was expanded with
 *             (0 for the root, 1 + (l-1)k + slot for frontier slot `slot` of layer l), -1 for
 *             a node that was not expanded (it has no children).
 * Order of the flattened nodes: root, then by (depth, parent's flat index, rank of the
 * child within its parent's top-k).  Top-k ties -> lower token id; frontier ties -> lower
 * layer-local index; rerank ties -> shallower, then lower layer-local index.
 * Device errors: a selection that is not a connected tree (possible only if some
 * log-prob > 0) -> TS_ERR_DEVICE_CHECK for that sequence.
 * --------------------------------------------------------------------------------- */
size_t ts_tree_build_workspace(int B, int V, int k, int depth, int m);
int ts_tree_build(const float* draft_logp, const int32_t* root_tokens,
                  int B, int V, int k, int depth, int m,
                  int32_t* tokens, int32_t* parents, int32_t* depth_out, uint64_t* mask,
                  double* values, int32_t* node_row,
                  void* workspace, size_t ws_bytes, int32_t* dev_status, void* stream);

/* ------------------------------------------------------------------------------------
 * ts_tree_attention — tree attention over a paged KV cache, batched, GQA.
 * Source: "rainlin.net/posts/eagle", section 四 Tree Attention (the flattened tree is fed in
 * one pass; node i attends only to its root-to-node ancestors, which equals verifying
 * every path separately); "lesty.tech — EAGLE-2 vs. Medusa", section 5 (mask held on chip,
 * no re-reads) and section 8 (the tree's K/V sit in blocks of the same paged sequence,
 * after the committed prefix).
 *
 * For sequence b, query head h (KV head h / g) and node i:
 *   keys = prefix positions 0..L_b-1  U  { L_b + t : mask bit t of row i is set }
 *   out  = softmax(scale * q . k^T) . v over those keys,  lse = log of the softmax sum
 * q          [B, m, Hq, d]  (dt: fp32 or bf16), 16-byte aligned.
 * k_cache,
 * v_cache    [num_blocks, Hkv, block_size, d] (dt), 16-byte aligned.  Logical position p
 *            of sequence b lives in block block_table[b*max_blocks + p/block_size], row
 *            p % block_size.  Positions L_b .. L_b+m-1 hold the tree nodes' K/V (already
 *            written by the caller, with whatever positional encoding it applies).
 * block_table [B, max_blocks] int32; entries for positions >= L_b + m are not read.
 * prefix_len [B] int32, 0 <= L_b <= max_prefix, and L_b + m <= max_blocks*block_size.
 * max_prefix host-side upper bound of prefix_len (sizes the launch and the workspace).
 * mask       [B, m, W] uint64 as produced by ts_tree_build.
 * scale      softmax scale (normally 1/sqrt(d)).
 * out        [B, m, Hq, d] (dt).  lse: [B, m, Hq] fp32 natural-log sum-exp (NULL ok).
 * Supported: fp32 any d <= 256 (CUDA-core path, fp32 accumulation); bf16 with d == 128
 * and block_size in {16, 32, 64, 128} (tcgen05 tensor-core path, TMA-staged K/V, fp32
 * accumulation, P rounded to bf16 for the PV product).  m <= 256.
 * Device errors: block id outside [0, num_blocks) or prefix_len outside [0, max_prefix]
 * -> TS_ERR_DEVICE_CHECK; a pipeline wait that exceeded its time bound -> TS_ERR_TIMEOUT.
 * --------------------------------------------------------------------------------- */
size_t ts_tree_attention_workspace(ts_dtype dt, int B, int m, int Hq, int Hkv, int d,
                                   int max_prefix);
int ts_tree_attention(const void* q, const void* k_cache, const void* v_cache, ts_dtype dt,
                      int num_blocks, int block_size, const int32_t* block_table,
                      int max_blocks, const int32_t* prefix_len, int max_prefix,
                      const uint64_t* mask, int B, int m, int Hq, int Hkv, int d,
                      float scale, void* out, float* lse,
                      void* workspace, size_t ws_bytes, int32_t* dev_status, void* stream);

/* Launch plan ts_tree_attention would use for these sizes on the current device (a
 * diagnostic; the pages have no counterpart).  Writes 6 ints to plan_out: [0] path (0 =
 * CUDA-core, 1 = tensor-core), [1] row groups of 128 rows (one CTA each), [2] chunks per
 * (sequence, KV head, row group), [3] 128-key tiles per chunk, [4] split mode (0 = one chunk,
 * 1 = chunks merged inside a thread-block cluster, 2 = chunks merged through the workspace),
 * [5] row groups that share each K/V tile through TMA multicast (1 = none).  Returns TS_OK or
 * the validation error ts_tree_attention would return. */
int ts_tree_attention_plan(ts_dtype dt, int B, int m, int Hq, int Hkv, int d, int max_prefix,
                           int block_size, int* plan_out);

/* The same plan for a GPU with num_sms streaming multiprocessors in place of the current
 * device's count (sizing ahead of time, or for a share of the SMs; 152 on a GB300).  The row
 * groups, chunks and tiles per chunk follow from the sizes and num_sms alone; multicast and
 * the in-cluster merge are chosen only where the current device reports that it can
 * co-schedule such clusters, so with no device present the plan uses neither.
 * num_sms < 1 -> TS_ERR_INVALID; otherwise as ts_tree_attention_plan. */
int ts_tree_attention_plan_for_sms(ts_dtype dt, int B, int m, int Hq, int Hkv, int d, int max_prefix,
                                   int block_size, int num_sms, int* plan_out);

/* ------------------------------------------------------------------------------------
 * ts_tree_accept — greedy verification of the tree.
 * Source: "lesty.tech — EAGLE-2 vs. Medusa", section 4 (greedy: a draft token is accepted iff
 * it is the base model's argmax given its context, here its parent's position);
 * "rainlin.net/posts/eagle", section 3.2 (accept the longest valid branch).
 *
 * logits     [B, m, V] (dt), row (b, i) = target distribution after node i's root path.
 * tokens, parents [B, m] int32 (as from ts_tree_build; parents precede children).
 * Outputs:
 *   argmax      [B, m] int32, first index of the row maximum (ties -> lowest id; -0 == +0).
 *               NaN entries are never the argmax (-inf is an ordinary value); a row of
 *               nothing but NaN gives -1, which matches no token.
 *   accept_len  [B] int32 >= 1: nodes on the accepted path, root included.
 *   accept_path [B, m] int32: flat indices root..accepted node, then -1.
 *   bonus       [B] int32: argmax at the accepted node (the token the step emits after
 *               the accepted drafts).
 * A node is valid when every non-root node on its root path has token == argmax of its
 * parent.  The accepted node is the deepest valid node, ties -> lowest flat index.
 * Device errors: parents[0] != -1 or parents[i] not in [0, i) -> TS_ERR_DEVICE_CHECK, and
 * that sequence's outputs are accept_len 0, path all -1, bonus -1.
 * --------------------------------------------------------------------------------- */
size_t ts_tree_accept_workspace(ts_dtype dt, int B, int m, int V);
int ts_tree_accept(const void* logits, ts_dtype dt, const int32_t* tokens,
                   const int32_t* parents, int B, int m, int V,
                   int32_t* argmax, int32_t* accept_len, int32_t* accept_path, int32_t* bonus,
                   void* workspace, size_t ws_bytes, int32_t* dev_status, void* stream);

/* ------------------------------------------------------------------------------------
 * ts_tree_accept_noalloc — ts_tree_accept for callers that cannot allocate device memory.
 * The pages have no counterpart to this entry point; it exists for deployment.
 *
 * Who needs it: a serving engine that hands all free HBM to its KV-cache pool at start-up
 * and allows no later cudaMalloc, or a plugin whose host framework owns every device
 * allocation.  Such callers pass only inputs and outputs; the scratch comes from a 1 MiB array compiled into
 * the library (a file-scope __device__ array that every GPU which loads the library keeps
 * until the process exits).  No cudaMalloc, cudaFree or allocating library routine is
 * called.
 *
 * Arguments, outputs, ordering rules and device errors are those of ts_tree_accept.
 * Limit: B * m * S partial (value, index) pairs of 8 bytes must fit in 1 MiB, S being the
 * number of vocabulary segments per logits row the launch uses (at most ceil(V / 2048);
 * for example B * m = 512 rows of V = 128256 use S = 2).  Larger requests return
 * TS_ERR_UNSUPPORTED without launching anything.
 * The first call on a device looks up the array's device address with that device current
 * and caches it under the current CUDA context's ID (a cudaDeviceReset leads to a new
 * context, so the next call looks it up again); make that first call before any stream
 * capture.  All calls share the one
 * array (its previous contents are irrelevant: every slot is written before it is read), so
 * calls that may overlap on the GPU (different streams, or different host threads without
 * ordering) race and must be serialised by the caller.
 * --------------------------------------------------------------------------------- */
int ts_tree_accept_noalloc(const void* logits, ts_dtype dt, const int32_t* tokens,
                           const int32_t* parents, int B, int m, int V,
                           int32_t* argmax, int32_t* accept_len, int32_t* accept_path,
                           int32_t* bonus, int32_t* dev_status, void* stream);


/*
 * ts_lm_head_argmax — per-row argmax of the target LM head, computed in the epilogue of the
 * LM-head GEMM so that the [M, N] logits are never written to HBM.
 *
 * Source: "jialefu.github.io — EAGLE-4 efficient LM head", section "A variant based on local
 * Top-k" (selection fused with the vocabulary-tile matrix multiplication, scores kept on chip,
 * the tiles' winners merged); for top-1 the merge is exact.  Consumed by the greedy check of
 * "lesty.tech — EAGLE-2 vs. Medusa", section 4.
 *
 * logits[r][n] = sum_k hidden[r][k] * weight[n][k], bf16 inputs, fp32 accumulation (tensor
 * cores; the summation order is the hardware's).  argmax[r] = the first n with the largest
 * logit (ties -> lowest n); max_logit[r] (optional, NULL ok) = that logit.
 * hidden  [M, K] bf16, device, 16-byte aligned.   weight [N, K] bf16 (one row per vocabulary
 * entry, the usual LM-head layout), device, 16-byte aligned.   K % 8 == 0.
 * argmax [M] int32, max_logit [M] fp32: device outputs.  workspace: caller-owned device
 * memory of ts_lm_head_argmax_workspace(M, N, K) bytes.  Two launches on `stream`.
 * Errors: TS_ERR_INVALID (sizes, alignment, null pointers), TS_ERR_WORKSPACE (too small)
 * before any launch; TS_ERR_CUDA if a launch or the tensor-map encoding fails; a pipeline
 * wait that times out sets *dev_status to TS_ERR_TIMEOUT.
 */
size_t ts_lm_head_argmax_workspace(int M, int N, int K);
int ts_lm_head_argmax(const void* hidden, const void* weight, int M, int N, int K, int32_t* argmax,
                      float* max_logit, void* workspace, size_t ws_bytes, int32_t* dev_status,
                      void* stream);

/*
 * ts_tree_accept_hidden — ts_tree_accept starting from the target's final hidden states
 * instead of its logits: the per-node argmax comes from the fused LM-head GEMM above (no
 * logits in HBM), then the same acceptance walk.  hidden [B, m, K] bf16, weight [V, K] bf16;
 * other arguments and outputs as ts_tree_accept.  Workspace: ts_tree_accept_hidden_workspace.
 */
size_t ts_tree_accept_hidden_workspace(int B, int m, int V, int K);
int ts_tree_accept_hidden(const void* hidden, const void* weight, const int32_t* tokens,
                          const int32_t* parents, int B, int m, int V, int K, int32_t* argmax,
                          int32_t* accept_len, int32_t* accept_path, int32_t* bonus, void* workspace,
                          size_t ws_bytes, int32_t* dev_status, void* stream);


/*
 * ts_efficient_head — the draft model's two-stage efficient LM head.
 *
 * Source: "jialefu.github.io — EAGLE-4 efficient LM head", sections "EAGLE Efficient LM Head"
 * (a low-rank head scores the whole vocabulary cheaply and candidates are chosen by top-k;
 * the full LM-head rows of the candidates are gathered and their logits recomputed from the
 * hidden states) and "A variant based on local Top-k" (the selection is fused into the
 * vocabulary-tile matrix multiplication, each tile keeping its own k_tile best).
 *
 * Per row r of hidden [M, d]:  u = bf16(lr_b @ h)  (lr_b [rank, d]);  scores = lr_a @ u
 * (lr_a [V, rank], fp32 accumulation, never written to HBM);  the vocabulary is cut into tiles
 * of tile_tokens ids and each keeps its k_tile best (score descending, ties -> lower id) ->
 * candidates [M, C], C = ts_efficient_head_candidates(V, tile_tokens, k_tile) (-1 in empty
 * slots);  logits[c] = weight[c] @ h (weight [V, d], fp32);  top_tok [M, k] = the k best
 * candidates (logit descending, ties -> lower id), top_logp [M, k] = logit - logsumexp over
 * the candidates' logits; where short tiles leave a row fewer than k candidates, its last
 * entries are top_tok -1, top_logp -inf.  Rows of top_tok / top_logp are what
 * ts_tree_build_from_topk reads.
 * All bf16 tensors row-major, device, 16-byte aligned; d % 8 == 0, rank % 8 == 0,
 * tile_tokens % 256 == 0, 1 <= k_tile <= 8, 1 <= k <= min(16, C).  candidates may be NULL.
 * Four launches on `stream`; workspace of ts_efficient_head_workspace(...) bytes.
 * Errors: TS_ERR_INVALID / TS_ERR_UNSUPPORTED / TS_ERR_WORKSPACE before any launch;
 * TS_ERR_CUDA on a launch or tensor-map failure; a timed-out pipeline wait sets *dev_status.
 */
int ts_efficient_head_candidates(int V, int tile_tokens, int k_tile);
size_t ts_efficient_head_workspace(int M, int V, int d, int rank, int tile_tokens, int k_tile);
int ts_efficient_head(const void* hidden, const void* lr_b, const void* lr_a, const void* weight, int M,
                      int V, int d, int rank, int tile_tokens, int k_tile, int k, int32_t* top_tok,
                      float* top_logp, int32_t* candidates, void* workspace, size_t ws_bytes,
                      int32_t* dev_status, void* stream);

/*
 * ts_tree_build_from_topk — ts_tree_build starting from each draft row's top-k list instead of
 * the full rows (for a drafter whose head already returns the top-k, such as
 * ts_efficient_head): row_tok / row_logp [B, 1 + (depth-1) k, k], each row in order (value
 * descending, ties -> lower token; a row out of order sets *dev_status to
 * TS_ERR_DEVICE_CHECK and the sequence's outputs are not written).  Expansion, rerank,
 * flatten and mask as ts_tree_build.  One launch; no workspace.
 * Sources: "jialefu.github.io — EAGLE-4 efficient LM head", section "EAGLE Efficient LM Head"
 * (the draft head hands on only its top candidates per position); "rainlin.net/posts/eagle",
 * sections 7.1-7.2 (expansion and rerank over those candidates).
 */
int ts_tree_build_from_topk(const int32_t* row_tok, const float* row_logp, const int32_t* root_tokens,
                            int B, int k, int depth, int m, int32_t* tokens, int32_t* parents,
                            int32_t* depth_out, uint64_t* mask, double* values, int32_t* node_row,
                            int32_t* dev_status, void* stream);

/*
 * ts_kv_commit — after ts_tree_accept, keep the accepted path's K/V rows in the paged cache
 * and release the scratch pages that held only rejected tree nodes.
 *
 * Source: "lesty.tech — EAGLE-2 vs. Medusa", section 8 (speculative rollback: the tree's K/V
 * are written into reserved scratch pages during the verify pass; only the accepted path
 * survives, the block table commits it and the rejected pages return to the free pool).
 * With multi-token pages the page's "update the pointers only" holds for whole pages; the
 * accepted rows inside the tree's pages are compacted first.
 *
 * Tree node i of sequence b sits at logical position prefix_len[b] + i (the layout
 * ts_tree_attention reads).  For every sequence, with L = prefix_len[b], a = accept_len[b]:
 *   - the K and V rows of node accept_path[b][j] move to logical position L + j, for every
 *     KV head and j = 0..a-1 (every row is read before it can be overwritten);
 *   - prefix_len[b] becomes L + a;
 *   - the block-table entries of logical pages ceil((L+a)/bs) .. ceil((L+m)/bs)-1 are listed,
 *     in that order, in freed_blocks[b][0..] (the rest of the row is -1; freed_count[b] of
 *     them) and set to -1 in the block table.
 *
 * k_cache, v_cache   [num_blocks, Hkv, block_size, d] of dt (TS_F32 or TS_BF16), device, in/out.
 * block_table        [B, max_blocks] int32, device, in/out.
 * prefix_len         [B] int32, device, in/out.
 * accept_path        [B, m] int32, device (ts_tree_accept's output; -1 padded).
 * accept_len         [B] int32, device (1..m).
 * freed_blocks       [B, max_blocks] int32, device, out.   freed_count [B] int32, device, out.
 * All pointers are caller-owned device memory; nothing is allocated; one launch on `stream`.
 * Errors: TS_ERR_INVALID (null pointer, non-positive size, d * element size not a multiple
 * of 4) and TS_ERR_UNSUPPORTED (m > TS_MAX_NODES) before any launch.  A sequence whose
 * prefix length is negative, whose accept length is outside 1..m, whose path does not start
 * at the root or does not increase, whose pages do not fit max_blocks or whose touched page
 * ids are out of range is left untouched and *dev_status is set to TS_ERR_DEVICE_CHECK.
 */
int ts_kv_commit(void* k_cache, void* v_cache, ts_dtype dt, int num_blocks, int block_size,
                 int Hkv, int d, int32_t* block_table, int max_blocks, int32_t* prefix_len,
                 const int32_t* accept_path, const int32_t* accept_len, int B, int m,
                 int32_t* freed_blocks, int32_t* freed_count, int32_t* dev_status, void* stream);

/* ------------------------------------------------------------------------------------
 * ts_tree_accept_sample — verification of the tree when the target samples at temperature
 * T > 0: multi-round rejection sampling.
 * Source: "lesty.tech — EAGLE-2 vs. Medusa", section 4 (Mathematical Verification: Lossless
 * Rejection Sampling): a candidate x proposed by q is kept with probability min(1, p(x)/q(x));
 * after a rejection one token is drawn from max(0, p - q) / (1 - sum min(p, q)).
 *
 * Per sequence, starting at the root: p = softmax(logits[node] / T).  The node's children
 * are tried in increasing flat index; child c with token x is kept iff
 * uniforms[b][c] * q(x) < p(x).  The first kept child becomes the current node.  After a
 * rejection p becomes max(0, p - q) renormalised (unchanged if that has zero mass) and x
 * leaves q (q(x) = 0, q renormalised).  When no child is kept (or there are none), one token
 * is drawn from the current p by inverse CDF over increasing token ids with
 * uniforms[b][0]: the smallest y whose cumulative mass exceeds uniforms[b][0] * total.
 *   q_mode TS_Q_POINT: q is a unit mass on each candidate (the trial reads r < p(x), a
 *     rejection removes x's mass from p).  Lossless for children chosen deterministically,
 *     such as the draft's top-k of ts_tree_build.
 *   q_mode TS_Q_DRAFT: q = exp(draft_logp[b][node_row[b][node]]) renormalised (the draft
 *     row that proposed the node's children, as ts_tree_build's node_row output names it).
 *     Lossless for children drawn from q without replacement.
 *
 * logits      [B, m, V] (dt), row (b, i) = target logits after node i's root path.
 * tokens, parents [B, m] int32 (parents[0] == -1, parents[i] in [0, i); tokens in [0, V)).
 * uniforms    [B, m] float, each in [0, 1): entry c decides the trial of child c (a node is
 *             tried at most once), entry 0 draws the final token.
 * draft_logp  [B, R, V] float log-probabilities, node_row [B, m] int32 — TS_Q_DRAFT only
 *             (may be NULL for TS_Q_POINT); a node with children needs node_row in [0, R).
 * temperature finite, > 0.
 * Outputs: accept_len [B] (kept nodes, root included), accept_path [B, m] (flat indices from
 * the root, then -1), bonus [B] (the drawn token).
 * Workspace: ts_tree_accept_sample_workspace(B, V, q_mode) bytes (0 for TS_Q_POINT; the
 * pointer may then be NULL).  Limits: m <= TS_MAX_NODES, V <= TS_SAMPLE_MAX_VOCAB.
 * Device errors: a bad parent, token or node_row, or a target row without mass (every logit
 * -inf or NaN) -> TS_ERR_DEVICE_CHECK; for a bad tree that sequence's outputs are
 * accept_len 0, path all -1, bonus -1.  One launch, one CTA per sequence.
 * --------------------------------------------------------------------------------- */
size_t ts_tree_accept_sample_workspace(int B, int V, int q_mode);
int ts_tree_accept_sample(const void* logits, ts_dtype dt, const int32_t* tokens, const int32_t* parents,
                          const float* uniforms, const float* draft_logp, const int32_t* node_row, int R,
                          int B, int m, int V, float temperature, int q_mode, int32_t* accept_len,
                          int32_t* accept_path, int32_t* bonus, void* workspace, size_t ws_bytes,
                          int32_t* dev_status, void* stream);

/* ------------------------------------------------------------------------------------
 * ts_tree_prune — cost-aware pruning of the draft tree before verification.
 * Sources: "jialefu.github.io — EAGLE-4 efficient LM head", section EAGLE-Harness (prune the
 * tree from draft and target costs and the draft confidence; the page gives no formula);
 * "rainlin.net/posts/eagle", sections 7.1 (value = product of the confidences on the root
 * path) and 六 (the confidence tracks the acceptance rate).
 *
 * Expected tokens of verifying a tree: 1 + sum over its non-root nodes of exp(values).  The
 * candidate trees are the prefixes of the rerank order (value descending, then shallower,
 * then lower flat index), each a connected tree because values never increase along a path.
 * One node count n (root included) is chosen for the whole batch, the first maximum over
 * n = 1..m of
 *     sum_b (1 + sum of exp(values) over the first n-1 nodes of b) / (t_draft + t_fixed + t_node*B*n)
 * (t_draft: the round's drafting time; t_fixed, t_node: the verification pass's fixed and
 * per-node time; any unit, all >= 0 with a positive sum).  exp and the sums run in fp32.
 *
 * tokens, parents, depth [B, m] int32 and values [B, m] double: a tree as ts_tree_build
 *   writes it; node_row [B, m] int32 optional (NULL: node_row_out is not written).
 * Outputs (device, capacity for n = m; written COMPACTLY with row stride n, so after
 * reading *n_out the first B*n entries form [B, n]):
 *   n_out [1] int32; tokens_out, parents_out, depth_out, node_row_out, kept_out (the old
 *   flat index of each kept node) [B, n] int32; values_out [B, n] double; mask_out
 *   [B, n, ceil(n/64)] uint64 (the ancestor mask of the pruned tree); expected_out [B] float
 *   (1 + the kept nodes' sum of exp(values)).  Kept nodes keep their flat order.
 * Workspace: ts_tree_prune_workspace(B, m) bytes.  Limits: m <= TS_MAX_NODES.
 * Device errors: a parent not preceding its child, or a kept node whose parent is not kept
 * (a value above its parent's) -> TS_ERR_DEVICE_CHECK.  Three launches, no host sync.
 * --------------------------------------------------------------------------------- */
size_t ts_tree_prune_workspace(int B, int m);
int ts_tree_prune(const int32_t* tokens, const int32_t* parents, const int32_t* depth, const double* values,
                  const int32_t* node_row, int B, int m, double t_draft, double t_fixed, double t_node,
                  int32_t* n_out, int32_t* tokens_out, int32_t* parents_out, int32_t* depth_out,
                  uint64_t* mask_out, double* values_out, int32_t* node_row_out, int32_t* kept_out,
                  float* expected_out, void* workspace, size_t ws_bytes, int32_t* dev_status, void* stream);

/* ------------------------------------------------------------------------------------
 * ts_selftest_bounded_wait — failure-detection check of the bounded pipeline waits.
 * The pages have no counterpart; it exists so that the timeout path can be tested without
 * faulting or hanging a GPU.  One CTA, two warps, each waiting on its own mbarrier through
 * the same bounded wait every kernel of the library uses:
 *   mode 0: nothing arrives.  After the wait limit (2 s) the first wait to give up raises
 *           the CTA's abort flag and stores TS_ERR_TIMEOUT in *dev_status, the other leaves
 *           on the flag, and the kernel returns; the context stays usable.
 *   mode 1: both barriers are completed first; both waits succeed at once.
 * result [2] int32 device: 1 if warp w's wait succeeded, else 0.  One launch.
 * --------------------------------------------------------------------------------- */
int ts_selftest_bounded_wait(int mode, int32_t* result, int32_t* dev_status, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* TREESPEC_H */
