// ts_tree_attention, tensor-core path (bf16, head dim 128) for sm_103a.
//
// Source: "rainlin.net/posts/eagle", section 四 Tree Attention (node i attends to the
// prefix and to its own root-to-node ancestors only; one pass verifies every path);
// "lesty.tech — EAGLE-2 vs. Medusa", section 5 (the tree mask stays on chip, no global
// re-reads) and section 8 (tree K/V sit in the same paged sequence after the prefix).
//
// Work unit: (sequence b, KV head, row group, chunk of 128-key tiles).  The g query heads
// that share a KV head and the m tree nodes are packed into GEMM rows, row = node*g +
// head-in-group, so every K/V byte fetched serves up to 128 query rows on the tensor cores;
// row groups past the first (m*g > 128) read the same K/V tiles, adjacent in launch order so
// the second read comes from L2.  One CTA per SM.
//
// Warp roles (12 warps + extra producers):
//   warps 0,3 (+ extra)  K producers; warp 0 first stages the chunk's physical block ids in
//                        shared memory.  One thread per producer warp issues TMA loads: per
//                        128-key tile one box of min(block_size,64) rows x 64 bf16 (128-byte
//                        swizzle) per page and head-dim half, an even share of the tile's boxes
//                        per producer; positions past the sequence load an out-of-range block
//                        (zero fill).  K ring of SK stages, V ring of SV stages.
//   warp 2 (+ extra)     V producers (same scheme on the V ring).
//   warp 1               TMEM allocator + the single thread that issues tcgen05.mma:
//                          S_t  = Q K_t^T    (M=128, N=128, K=128; A, B from shared memory)
//                          O   += P_t V_t    (M=128, N=128, K=128; A = P from TMEM, B = V MN-major)
//                        S and P are double-buffered: Q K^T of tile t+2 is issued right after
//                        P V of tile t, so the tensor cores work while the softmax of tile t+1
//                        runs.
//   warps 4..11          softmax, two threads per row (TMEM lane): warps 4..7 take keys 0..63
//                        of every tile, warps 8..11 keys 64..127.  First each stages its row's
//                        head-dim half of Q in shared memory (the MMA thread waits for all of
//                        them on an mbarrier).  Per tile each loads its 64 scores,
//                        applies the tree mask on the tiles that reach the tree, exchanges its
//                        row maximum with its partner through shared memory, and runs the
//                        online softmax in the log2 domain with lazy rescaling of its half of O
//                        (only when the running max grows by more than 2^8), writing P as bf16
//                        into TMEM; then the epilogue.  Only the warps that hold rows of this
//                        group take part.
// TMEM columns: O [0,128), S_0 [128,256), S_1 [256,384), P_0 [384,448), P_1 [448,512).
// Split over chunks of one (sequence, KV head, row group):
//   direct   one chunk: the epilogue writes O / l.
//   cluster  the chunks are the CTAs of one thread-block cluster (<= 8): after a cluster
//            barrier each CTA stores its fp32 O rows and (max, sum) straight into the shared
//            memory of the CTA that owns those rows (distributed shared memory), and after a
//            second barrier every owner merges its rows locally and writes the output: no
//            partials in HBM and no second launch.
//   global   more chunks than a cluster holds: fp32 partials go to the workspace and
//            combine_kernel merges them.
// Chunks are balanced: chunk c of a sequence of T tiles covers [ceil(c*T/nc), ceil((c+1)*T/nc)).
#include <cuda.h>
#include <cudaTypedefs.h>

#include <cmath>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace ts {
namespace tc {

constexpr int BN = 128;   // keys per tile
constexpr int BM = 128;   // rows per CTA
constexpr int HD = 128;   // head dim
constexpr uint32_t QHALF = BM * 128;   // 128 rows x 64 bf16 = 16 KB
constexpr uint32_t QTILE = 2 * QHALF;  // both head-dim halves
constexpr uint32_t KHALF = BN * 128;   // 128 keys x 64 bf16 = 16 KB
constexpr uint32_t KTILE = 2 * KHALF;  // 32 KB
constexpr float kRescaleThreshold = 8.0f;  // log2 units
constexpr int kMaxChunkBoxes = 2048;       // physical-block ids a CTA stages in shared memory
constexpr int kMaxCluster = 8;
constexpr int kMaxSortedSeqs = 64;  // batches up to this size are dispatched longest first
constexpr float kLn2 = 0.69314718055994530942f;

enum Mode { kDirect = 0, kCluster = 1, kGlobal = 2 };

struct Cfg {
  static constexpr int SK = 3;  // K ring stages (K is consumed two tiles ahead of V)
  static constexpr int SV = 2;  // V ring stages
  // A TMA instruction keeps its issuing thread busy for on the order of 100 cycles, and a
  // 128-key tile of 16-token pages is 16 K boxes (2 KB) and 8 V boxes (4 KB), so K has three
  // issuing warps: warps 0 and 3, and warp 12 after the softmax warps; warp 2 issues V (the
  // warps after the softmax warps would take further V parts, then further K parts).  Measured
  // on the long-context and Llama-2-70B shapes, 3 + 1 issuers beat 4 + 2 by 1-2%.
  static constexpr int K_PRODUCERS = 3;
  static constexpr int V_PRODUCERS = 1;
  // softmax: two threads per row (warps 4..7 the first 64 keys of a tile, warps 8..11 the
  // other 64; warp w reaches TMEM lanes 32*(w%4) .. +31), which exchange their row maxima
  // through shared memory once per tile
  static constexpr int EXTRA_WARP = 12;
  // the P V issuer has a warp of its own after the extra producers (warp 1 issues Q K^T)
  static constexpr int PV_WARP = EXTRA_WARP + (K_PRODUCERS - 2) + (V_PRODUCERS - 1);
  static constexpr int THREADS = 32 * (PV_WARP + 1);
  static constexpr uint32_t TMEM_COLS = 512;
  static constexpr uint32_t COL_S = 128;
  static constexpr uint32_t COL_P = 384;
  static constexpr uint32_t OFF_Q = 0;
  static constexpr uint32_t OFF_K = QTILE;
  static constexpr uint32_t OFF_V = OFF_K + SK * KTILE;
  static constexpr uint32_t OFF_BAR = OFF_V + SV * KTILE;
  // full_k[SK] empty_k[SK] full_v[SV] empty_v[SV] s_full[2] p_full[2] o_ready o_final
  // xchg[4 quadrants][2 parities] (p_full is per S buffer: a fast softmax warp may reach tile
  // t+1 while slower warps still work on tile t, and their arrivals must not mix)
  // + q_ready, p_free[2] (P V has read that P buffer), qk_done
  static constexpr int NBAR = 2 * SK + 2 * SV + 6 + 8 + 1 + 3;
  static constexpr uint32_t OFF_XCH = OFF_BAR + NBAR * 8;         // [2 parities][2 halves][128 rows] fp32
  static constexpr uint32_t OFF_MISC = OFF_XCH + 2 * 2 * BM * 4;
  static constexpr uint32_t OFF_ML = OFF_MISC + 16;            // (max, sum) per row, cluster merge
  static constexpr uint32_t OFF_BLK = OFF_ML + BM * 8;
  static constexpr uint32_t SMEM_BYTES = OFF_BLK + 4 * kMaxChunkBoxes + 1024;  // + alignment slack
  static_assert(COL_P + 64 * 2 <= TMEM_COLS, "TMEM budget");
  static_assert(SK * KTILE >= BM * 512, "O rows must fit in the K ring for the merge");
  static_assert(SMEM_BYTES <= 232448, "shared memory budget");
};

struct Params {
  const __nv_bfloat16* q;
  const int32_t* block_table;
  const int32_t* prefix_len;
  const uint64_t* mask;
  __nv_bfloat16* out;
  float* lse;
  float* part_o;
  float2* part_ml;
  int32_t* status;
  int B, m, Hq, Hkv, g, rows, W, max_blocks, num_blocks, block_size, max_prefix, tpc, nchunk, mode;
  int mc;  // row groups sharing each K/V tile through TMA multicast (a cluster along x), 1 = none
  int split_issue;  // 1: Q K^T and P V issued by two threads (warp 1, PV_WARP); 0: warp 1 issues both
  float scale_log2;
};

// Wait bounded by time only (used on the abort path, to let in-flight copies and MMAs land
// before shared memory and TMEM are released).
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try(bar, parity)) {
    if (global_timer_ns() - t0 > kWaitLimitNs) return;
  }
}

// Byte offset of 16-byte chunk c of parked O row R (rows of 512 B; the chunk index is
// XOR-swizzled with the row so a warp writing 32 rows spreads over all banks).
__device__ __forceinline__ uint32_t orow_off(int R, int c) {
  return static_cast<uint32_t>(R) * 512u + (static_cast<uint32_t>(c ^ (R & 31)) << 4);
}

// Visibility of keys kb .. kb+63 for one row: the prefix keys (< L), then the row's ancestor
// bits of the tree positions (key - L) the 64 keys cover; positions at or past m are never
// visible.  `mw` are the row's mask words (m <= 256, so at most four).
__device__ __forceinline__ uint64_t visible64(int kb, int L, int m, uint64_t mw0, uint64_t mw1, uint64_t mw2,
                                              uint64_t mw3) {
  const int pre = L - kb;  // prefix keys among these 64
  if (pre >= 64) return ~0ull;
  const int tt0 = pre > 0 ? 0 : -pre;  // first tree position
  const int ntree = m - tt0;           // tree positions left from tt0
  uint64_t tb = 0ull;
  if (ntree > 0) {
    const int q = tt0 >> 6, sh = tt0 & 63;
    const uint64_t lo = q == 0 ? mw0 : q == 1 ? mw1 : q == 2 ? mw2 : q == 3 ? mw3 : 0ull;
    const uint64_t hi = q == 0 ? mw1 : q == 1 ? mw2 : q == 2 ? mw3 : 0ull;
    tb = sh == 0 ? lo : (lo >> sh) | (hi << (64 - sh));
    if (ntree < 64) tb &= (1ull << ntree) - 1ull;
  }
  return pre > 0 ? (((1ull << pre) - 1ull) | (tb << pre)) : tb;
}

__global__ void __launch_bounds__(Cfg::THREADS, 1)
    tree_attn_tc_kernel(const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
                        const Params p) {
  using C = Cfg;
  constexpr int SK = C::SK;
  constexpr int SV = C::SV;
  extern __shared__ unsigned char smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  unsigned char* sptr = smem_raw + (sbase - raw);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rg = blockIdx.x, chunk = blockIdx.y;
  const int slot = blockIdx.z / p.Hkv, kvh = blockIdx.z % p.Hkv;
  pdl_wait();
  // Launch order by decreasing prefix length (ties -> lower index): the CTAs of the longest
  // sequences are dispatched first and the short ones fill in behind them.
  int b = slot;
  if (p.B > 1 && p.B <= kMaxSortedSeqs) {
    int* s_len = reinterpret_cast<int*>(sptr + C::OFF_BLK);  // (the block-id area, not used yet)
    int* s_pick = s_len + kMaxSortedSeqs;
    if (threadIdx.x < p.B) s_len[threadIdx.x] = p.prefix_len[threadIdx.x];
    __syncthreads();
    if (threadIdx.x < p.B) {
      const int Lb = s_len[threadIdx.x];
      int rank = 0;
      for (int j = 0; j < p.B; ++j) {
        const int Lj = s_len[j];
        rank += (Lj > Lb) | ((Lj == Lb) & (j < static_cast<int>(threadIdx.x)));
      }
      if (rank == slot) *s_pick = threadIdx.x;
    }
    __syncthreads();
    b = *s_pick;
    __syncthreads();
  }
  const int bk = b * p.Hkv + kvh;
  const int L = p.prefix_len[b];
  // (the whole cluster shares b, so every CTA of a cluster returns here together)
  if (L < 0 || L > p.max_prefix) {
    if (threadIdx.x == 0 && rg == 0 && chunk == 0) report(p.status, TS_ERR_DEVICE_CHECK);
    return;
  }
  const int nkeys = L + p.m;
  const int T = (nkeys + BN - 1) / BN;
  // chunk c covers tiles [c*tpc, (c+1)*tpc) of this sequence (tpc from the longest allowed
  // prefix), so a shorter sequence uses fewer chunks and its CTAs past the end leave at once;
  // the last chunk, which holds the masked tree tile, is never the longest
  const int t0 = chunk * p.tpc;
  const int nt = max(0, min(T, t0 + p.tpc) - t0);
  if (nt == 0 && p.mode != kCluster) return;  // (an idle CTA of a cluster still merges)
  // a sequence whose tiles all fall into one chunk is written directly also in the global mode
  const bool direct = p.mode == kDirect || (p.mode == kGlobal && T <= p.tpc);
  const int R0 = rg * BM;
  const int rows_here = min(p.rows - R0, BM);
  const int nact = (rows_here + 31) / 32;  // softmax warps that hold rows of this group
  // Multicast: the mc row groups of one (sequence, KV head, chunk) form a cluster; each CTA
  // issues 1/mc of every tile's boxes to all of them, so a K/V tile leaves L2 once per
  // cluster.  A stage may be refilled only when every CTA of the cluster has released it, so
  // the empty barriers count one release per CTA (the MMA thread's commits are multicast).
  // The cluster is mc x nc CTAs in the chunk-merge mode (rank = x + mc*y), mc x 1 otherwise;
  // the row groups of one chunk (same y) share the multicasts.
  const int mc = p.mc;
  const int crank = rg % mc;
  const uint16_t mc_mask =
      static_cast<uint16_t>(((1u << mc) - 1u) << (p.mode == kCluster ? mc * chunk : 0));

  auto bar = [&](int idx) -> uint32_t { return sbase + C::OFF_BAR + 8u * idx; };
  auto full_k = [&](int s) { return bar(s); };
  auto empty_k = [&](int s) { return bar(SK + s); };
  auto full_v = [&](int s) { return bar(2 * SK + s); };
  auto empty_v = [&](int s) { return bar(2 * SK + SV + s); };
  auto s_full = [&](int sb) { return bar(2 * SK + 2 * SV + sb); };
  auto p_full = [&](int sb) { return bar(2 * SK + 2 * SV + 2 + sb); };
  const uint32_t o_ready = bar(2 * SK + 2 * SV + 4);
  const uint32_t o_final = bar(2 * SK + 2 * SV + 5);
  auto xchg_bar = [&](int q, int par) { return bar(2 * SK + 2 * SV + 6 + 2 * q + par); };
  const uint32_t q_ready = bar(2 * SK + 2 * SV + 14);  // Q staged by the softmax threads
  auto p_free = [&](int sb) { return bar(2 * SK + 2 * SV + 15 + sb); };
  const uint32_t qk_done = bar(2 * SK + 2 * SV + 17);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sptr + C::OFF_MISC);
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(sptr + C::OFF_MISC + 4);

  if (threadIdx.x == 0) {
    for (int s = 0; s < SK; ++s) {
      mbar_init(full_k(s), C::K_PRODUCERS);  // each producer warp registers its share of the bytes
      mbar_init(empty_k(s), mc);
    }
    for (int s = 0; s < SV; ++s) {
      mbar_init(full_v(s), C::V_PRODUCERS);
      mbar_init(empty_v(s), mc);
    }
    for (int sb = 0; sb < 2; ++sb) {
      mbar_init(s_full(sb), 1);
      mbar_init(p_full(sb), 64 * nact);
    }
    for (int q = 0; q < 4; ++q) {
      mbar_init(xchg_bar(q, 0), 64);
      mbar_init(xchg_bar(q, 1), 64);
    }
    mbar_init(o_ready, 1);
    mbar_init(o_final, 1);
    mbar_init(q_ready, 64 * nact);
    mbar_init(p_free(0), 1);
    mbar_init(p_free(1), 1);
    mbar_init(qk_done, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_holder), C::TMEM_COLS);
    tmem_relinquish();
  }
  // Physical block of every TMA box row group of this chunk -> shared memory (warp 0,
  // coalesced, 4 independent loads in flight per lane); out-of-range ids are reported and
  // replaced by the out-of-bounds block, positions past the sequence get it too.
  const int rpb = min(p.block_size, 64);  // rows per box
  const int bpt = BN / rpb;               // box rows per tile
  int* s_blk = reinterpret_cast<int*>(sptr + C::OFF_BLK);
  if (warp == 0) {
    const int nbox = nt * bpt;
    for (int e0 = lane; e0 < nbox; e0 += 4 * 32) {
      int ids[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int e = e0 + 32 * u;
        const int key = t0 * BN + e * rpb;
        ids[u] = -1;
        if (e < nbox && key < nkeys)
          ids[u] = __ldg(p.block_table + static_cast<long long>(b) * p.max_blocks + key / p.block_size);
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int e = e0 + 32 * u;
        if (e >= nbox) break;
        const int key = t0 * BN + e * rpb;
        int phys = p.num_blocks;
        if (key < nkeys) {
          if (ids[u] >= 0 && ids[u] < p.num_blocks) phys = ids[u];
          else report(p.status, TS_ERR_DEVICE_CHECK);
        }
        s_blk[e] = phys;
      }
    }
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;

  // per-row softmax state, kept for the epilogue
  float m_ref = -INFINITY, l_sum = 0.f;
  bool ok = true;

  if (warp == 0 || warp == 2 || warp == 3 || (warp >= C::EXTRA_WARP && warp < C::PV_WARP)) {
    // ------------------------------ TMA producers ------------------------------
    // Part `part` of `nparts` issues boxes [part*nbox/nparts, (part+1)*nbox/nparts) of every
    // tile (a part may hold none: it still registers its zero bytes once per tile).
    if (lane == 0) {
      const int e = warp - C::EXTRA_WARP;  // index among the warps after the softmax warps
      const int kv = (warp == 0 || warp == 3 || (e >= 0 && e >= C::V_PRODUCERS - 1)) ? 0 : 1;
      const int part = warp == 0 ? 0 : warp == 3 ? 1 : warp == 2 ? 0 : kv == 1 ? e + 1 : 2 + e - (C::V_PRODUCERS - 1);
      const int nparts = kv == 0 ? C::K_PRODUCERS : C::V_PRODUCERS;
      const int ST = kv == 0 ? SK : SV;
      const void* map = kv == 0 ? static_cast<const void*>(&tmk) : static_cast<const void*>(&tmv);
      // K: per box row j of the tile and head-dim half h one box of rpb rows x 128 B, placed
      // at h*KHALF + j*rpb*128 (each half of the tile is one K-major operand of 128 keys).
      // V: per box row j one box of both halves (rpb rows x 2 x 128 B, two-half tensor map),
      // placed at j*rpb*256 as [half][rows]: a P V step of 16 keys reads one page.
      const int nbox = kv == 0 ? 2 * bpt : bpt;
      // boxes this thread issues (its share among the cluster's mc*nparts issuers) and the
      // bytes it registers on this CTA's barrier (its share of the whole tile, which lands here
      // whichever CTA issued it)
      const int gi = crank * nparts + part, ng = mc * nparts;
      const int b_begin = gi * nbox / ng, b_end = (gi + 1) * nbox / ng;
      const int x_count = (part + 1) * nbox / nparts - part * nbox / nparts;
      const uint32_t box_bytes = kv == 0 ? rpb * 128 : rpb * 256;
      int issued = 0;
      for (int t = 0; t < nt; ++t) {
        const int s = t % ST;
        const uint32_t ph = (t / ST) & 1;
        const uint32_t fb = kv == 0 ? full_k(s) : full_v(s);
        const uint32_t eb = kv == 0 ? empty_k(s) : empty_v(s);
        if (!mbar_wait(eb, ph ^ 1u, abort_flag, p.status)) break;
        mbar_expect_tx(fb, static_cast<uint32_t>(x_count) * box_bytes);
        if (kv == 0) {
          const uint32_t dst0 = sbase + C::OFF_K + s * KTILE;
          for (int e2 = b_begin; e2 < b_end; ++e2) {
            const int j = e2 >> 1, h = e2 & 1;
            const int blk = s_blk[t * bpt + j];  // num_blocks (out of range) -> zero fill
            const int rin = blk < p.num_blocks ? (j * rpb) & (p.block_size - 1) : 0;
            if (mc > 1)
              tma_load_4d_mc(dst0 + h * KHALF + j * rpb * 128, map, fb, h * 64, rin, kvh, blk, mc_mask);
            else
              tma_load_4d(dst0 + h * KHALF + j * rpb * 128, map, fb, h * 64, rin, kvh, blk);
          }
        } else {
          const uint32_t dst0 = sbase + C::OFF_V + s * KTILE;
          for (int j = b_begin; j < b_end; ++j) {
            const int blk = s_blk[t * bpt + j];
            const int rin = blk < p.num_blocks ? (j * rpb) & (p.block_size - 1) : 0;
            if (mc > 1)
              tma_load_5d_mc(dst0 + j * rpb * 256, map, fb, 0, rin, 0, kvh, blk, mc_mask);
            else
              tma_load_5d(dst0 + j * rpb * 256, map, fb, 0, rin, 0, kvh, blk);
          }
        }
        issued = t + 1;
      }
      if (mc > 1 && part == 0 && !*abort_flag) {
        // every CTA of the cluster has released every stage of this ring: no release of a
        // peer is still on its way to this CTA's barriers when it exits
        for (int s = 0; s < ST && s < nt; ++s) {
          const int uses = (nt - s + ST - 1) / ST;
          if (!mbar_wait(kv == 0 ? empty_k(s) : empty_v(s), (uses - 1) & 1, abort_flag, p.status)) break;
        }
      }
      if (*abort_flag) {
        for (int t = max(0, issued - ST); t < issued; ++t)
          drain_wait(kv == 0 ? full_k(t % ST) : full_v(t % ST), (t / ST) & 1);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------ MMA issue ------------------------------
    // With several row groups (split_issue) warp 1 issues only Q K^T and the P V issuer warp
    // P V, so neither waits behind the other's barrier; with one row group warp 1 issues both.
    // Split: S_t = Q K_t^T (M=128, N=128, K=128; A, B from shared memory) into S buffer t%2, once K_t
    // is in and the softmax is done with the buffer's previous tile (its p_full: it has read S
    // and written P)
    if (lane == 0 && nt > 0 && !p.split_issue) {
      // one thread issues both: S_t = Q K_t^T and O += P_t V_t; S and P are double-buffered, Q K^T
      // of tile t+2 is issued right after P V of tile t (in issue order, so P V has read P before
      // the softmax of tile t+2 rewrites it), and the tensor cores work while the softmax of
      // tile t+1 runs
      constexpr uint32_t idq = idesc_bf16_f32(128, BN, 0, 0);
      constexpr uint32_t idp = idesc_bf16_f32(128, HD, 0, 1);
      auto qk = [&](int sk, int sb) {
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint32_t h = kk >> 2, ko = (kk & 3) * 32;
          const uint64_t a = sdesc_sw128(sbase + C::OFF_Q + h * QHALF + ko, 16, 1024);
          const uint64_t bd = sdesc_sw128(sbase + C::OFF_K + sk * KTILE + h * KHALF + ko, 16, 1024);
          mma_ss(tmem + C::COL_S + 128u * sb, a, bd, idq, kk > 0 ? 1u : 0u);
        }
        tc_commit(s_full(sb));
      };
      uint64_t vdesc[BN / 16];
#pragma unroll
      for (int kk = 0; kk < BN / 16; ++kk) {
        const int key = 16 * kk;
        const uint32_t off = (key / rpb) * rpb * 256 + (key % rpb) * 128;
        vdesc[kk] = sdesc_sw128(sbase + C::OFF_V + off, rpb * 128, 1024);
      }
      auto pv = [&](int sv, int sb, bool first) {
#pragma unroll
        for (int kk = 0; kk < BN / 16; ++kk)
          mma_ts(tmem, tmem + C::COL_P + 64u * sb + 8u * kk, vdesc[kk] + static_cast<uint64_t>(sv * (KTILE >> 4)), idp,
                 (first && kk == 0) ? 0u : 1u);
      };
      bool mok = mbar_wait(q_ready, 0, abort_flag, p.status);
      for (int t = 0; mok && t < 2 && t < nt; ++t) {
        mok = mbar_wait(full_k(t % SK), (t / SK) & 1, abort_flag, p.status);
        if (!mok) break;
        tc_fence_after();
        qk(t % SK, t & 1);
        if (mc > 1) tc_commit_mc(empty_k(t % SK), mc_mask);
        else tc_commit(empty_k(t % SK));
      }
      for (int t = 0; mok && t < nt; ++t) {
        const int sv = t % SV;
        mok = mbar_wait(full_v(sv), (t / SV) & 1, abort_flag, p.status);
        if (!mok) break;
        mok = mbar_wait(p_full(t & 1), (t >> 1) & 1, abort_flag, p.status);
        if (!mok) break;
        tc_fence_after();
        pv(sv, t & 1, t == 0);
        tc_commit(o_ready);
        if (mc > 1) tc_commit_mc(empty_v(sv), mc_mask);
        else tc_commit(empty_v(sv));
        const int tn = t + 2;
        if (tn < nt) {
          mok = mbar_wait(full_k(tn % SK), (tn / SK) & 1, abort_flag, p.status);
          if (!mok) break;
          tc_fence_after();
          qk(tn % SK, tn & 1);
          if (mc > 1) tc_commit_mc(empty_k(tn % SK), mc_mask);
          else tc_commit(empty_k(tn % SK));
        }
      }
      tc_commit(o_final);
      if (!mok) drain_wait(o_final, 0);
    }
    if (lane == 0 && nt > 0 && p.split_issue) {
      constexpr uint32_t idq = idesc_bf16_f32(128, BN, 0, 0);
      bool mok = mbar_wait(q_ready, 0, abort_flag, p.status);
      for (int t = 0; mok && t < nt; ++t) {
        const int sb = t & 1, sk = t % SK;
        if (t >= 2) {
          mok = mbar_wait(p_full(sb), ((t - 2) >> 1) & 1, abort_flag, p.status);
          if (!mok) break;
        }
        mok = mbar_wait(full_k(sk), (t / SK) & 1, abort_flag, p.status);
        if (!mok) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint32_t h = kk >> 2, ko = (kk & 3) * 32;
          const uint64_t a = sdesc_sw128(sbase + C::OFF_Q + h * QHALF + ko, 16, 1024);
          const uint64_t bd = sdesc_sw128(sbase + C::OFF_K + sk * KTILE + h * KHALF + ko, 16, 1024);
          mma_ss(tmem + C::COL_S + 128u * sb, a, bd, idq, kk > 0 ? 1u : 0u);
        }
        tc_commit(s_full(sb));
        if (mc > 1) tc_commit_mc(empty_k(sk), mc_mask);
        else tc_commit(empty_k(sk));
      }
      tc_commit(qk_done);
      if (!mok) drain_wait(qk_done, 0);
    }
    __syncwarp();
  } else if (warp == C::PV_WARP && p.split_issue) {
    // ------------------------------ P V issuer ------------------------------
    // O += P_t V_t (M=128, N=128, K=128; A = P from TMEM, B = V MN-major) once V_t and P_t are
    // in; its commits tell the softmax that O holds this tile (o_ready) and that the P buffer
    // may be rewritten (p_free)
    if (lane == 0 && nt > 0) {
      constexpr uint32_t idp = idesc_bf16_f32(128, HD, 0, 1);
      // B = V keys 16kk .. 16kk+15, MN-major: 64 head-dim columns per 128-byte row, 8-key
      // groups 1 KB apart (stride offset), the second head-dim half rpb*128 further (leading
      // offset); the keys sit in box row (16kk)/rpb at row (16kk)%rpb.  Descriptors of stage 0;
      // a stage adds KTILE (in 16-byte units) to the start address field.
      uint64_t vdesc[BN / 16];
#pragma unroll
      for (int kk = 0; kk < BN / 16; ++kk) {
        const int key = 16 * kk;
        const uint32_t off = (key / rpb) * rpb * 256 + (key % rpb) * 128;
        vdesc[kk] = sdesc_sw128(sbase + C::OFF_V + off, rpb * 128, 1024);
      }
      bool mok = true;
      for (int t = 0; mok && t < nt; ++t) {
        const int sv = t % SV, sb = t & 1;
        mok = mbar_wait(full_v(sv), (t / SV) & 1, abort_flag, p.status);
        if (!mok) break;
        mok = mbar_wait(p_full(sb), (t >> 1) & 1, abort_flag, p.status);
        if (!mok) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < BN / 16; ++kk)
          mma_ts(tmem, tmem + C::COL_P + 64u * sb + 8u * kk, vdesc[kk] + static_cast<uint64_t>(sv * (KTILE >> 4)),
                 idp, (t == 0 && kk == 0) ? 0u : 1u);
        tc_commit(o_ready);
        tc_commit(p_free(sb));
        if (mc > 1) tc_commit_mc(empty_v(sv), mc_mask);
        else tc_commit(empty_v(sv));
      }
      tc_commit(o_final);
      if (!mok) drain_wait(o_final, 0);
    }
    __syncwarp();
  } else if (warp >= 4 && warp < C::EXTRA_WARP) {
    // ------------------------------ softmax ------------------------------
    const int q4 = warp & 3;        // TMEM lane quadrant: rows 32*q4 .. +31
    const int hh = (warp - 4) >> 2; // keys 64*hh .. +63 of every tile, O columns 64*hh .. +63
    if (q4 < nact && nt > 0) {
      const int r = q4 * 32 + lane;
      const int grow = R0 + r;
      const bool valid = r < rows_here;
      const int node = valid ? grow / p.g : 0;
      uint64_t mw0 = 0, mw1 = 0, mw2 = 0, mw3 = 0;
      if (valid) {
        const uint64_t* mrow = p.mask + (static_cast<long long>(b) * p.m + node) * p.W;
        mw0 = mrow[0];
        if (p.W > 1) mw1 = mrow[1];
        if (p.W > 2) mw2 = mrow[2];
        if (p.W > 3) mw3 = mrow[3];
      }
      const uint32_t lane_off = static_cast<uint32_t>(q4 * 32) << 16;
      const uint32_t tO = tmem + lane_off + 64u * hh;
      {  // this row's head-dim half hh of Q -> shared memory in the 128-byte-swizzled K-major
         // layout (16-byte chunk j of row r at chunk j ^ (r % 8)); zeros for padding rows.  The
         // softmax threads stage Q after the CTA's set-up, while the producers start loading.
        const long long qoff =
            ((static_cast<long long>(b) * p.m + node) * p.Hq + kvh * p.g + (valid ? grow % p.g : 0)) * HD + 64 * hh;
        uint4 qv[8];
#pragma unroll
        for (int j = 0; j < 8; ++j)
          qv[j] = valid ? __ldg(reinterpret_cast<const uint4*>(p.q + qoff) + j) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
        for (int j = 0; j < 8; ++j)
          *reinterpret_cast<uint4*>(sptr + C::OFF_Q + hh * QHALF + r * 128 + ((j ^ (r & 7)) << 4)) = qv[j];
        fence_proxy_async_smem();
        mbar_arrive(q_ready);
      }
      const float sl2 = p.scale_log2;
      float* xch = reinterpret_cast<float*>(sptr + C::OFF_XCH);
      // the partner thread's value for exchange round `round` (both threads of a row take part
      // in every round; rounds alternate between two buffers, each with its own barrier)
      auto exchange = [&](int round, float v, float* other) -> bool {
        const int par = round & 1;
        xch[(par * 2 + hh) * BM + r] = v;
        mbar_arrive(xchg_bar(q4, par));
        if (!mbar_wait_warp(xchg_bar(q4, par), (round >> 1) & 1, abort_flag, p.status)) return false;
        *other = xch[(par * 2 + (hh ^ 1)) * BM + r];
        return true;
      };
      for (int t = 0; t < nt; ++t) {
        const int sb = t & 1;
        const uint32_t tS = tmem + lane_off + C::COL_S + 128u * sb + 64u * hh;
        const uint32_t tP = tmem + lane_off + C::COL_P + 64u * sb + 32u * hh;
        ok = mbar_wait_warp(s_full(sb), (t >> 1) & 1, abort_flag, p.status);
        if (!ok) break;
        tc_fence_after();
        const int key0 = (t0 + t) * BN;
        float s[64];
        {
          uint32_t u[64];
          tmem_ld64(tS, u);
#pragma unroll
          for (int c = 0; c < 64; ++c) s[c] = __uint_as_float(u[c]);
        }
        if (key0 + BN > L) {
          // one visibility bit per column (prefix columns, then this row's ancestors)
          const uint64_t vis = visible64(key0 + 64 * hh, L, p.m, mw0, mw1, mw2, mw3);
#pragma unroll
          for (int c = 0; c < 64; ++c) s[c] = ((vis >> c) & 1ull) ? s[c] : -INFINITY;
        }
        float mx;
        {  // eight independent running maxima, then a tree; then the partner's half
          float m8[8];
#pragma unroll
          for (int c = 0; c < 8; ++c) m8[c] = s[c];
#pragma unroll
          for (int c = 8; c < 64; ++c) m8[c & 7] = fmaxf(m8[c & 7], s[c]);
          mx = fmaxf(fmaxf(fmaxf(m8[0], m8[1]), fmaxf(m8[2], m8[3])), fmaxf(fmaxf(m8[4], m8[5]), fmaxf(m8[6], m8[7])));
          float mo;
          ok = exchange(t, mx, &mo);
          if (!ok) break;
          mx = fmaxf(mx, mo);
        }
        if (!valid) mx = -INFINITY;
        const float mt = mx * sl2;
        float alpha = 1.f;
        int resc = 0;
        if (mt > m_ref + kRescaleThreshold) {
          if (m_ref != -INFINITY) {
            alpha = ex2_approx(m_ref - mt);
            resc = 1;
          }
          l_sum *= alpha;
          m_ref = mt;
        }
        // padding rows take an infinite reference, so every exponential of theirs is 0
        const float mu = !valid ? INFINITY : (m_ref == -INFINITY) ? 0.f : m_ref;
        {
          float rs4[4] = {0.f, 0.f, 0.f, 0.f};
          uint32_t pk[32];
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            const float x0 = fmaf(s[2 * c], sl2, -mu), x1 = fmaf(s[2 * c + 1], sl2, -mu);
            const float p0 = ex2_approx(x0);
            const float p1 = ex2_approx(x1);
            rs4[c & 3] += p0 + p1;
            pk[c] = pack_bf16x2(p0, p1);
          }
          if (p.split_issue && t >= 2) {  // P V of tile t-2 has read this P buffer
            ok = mbar_wait_warp(p_free(sb), ((t >> 1) - 1) & 1, abort_flag, p.status);
            if (!ok) break;
            tc_fence_after();
          }
          tmem_st32(tP, pk);
          l_sum += (rs4[0] + rs4[1]) + (rs4[2] + rs4[3]);
        }
        if (__any_sync(0xffffffffu, resc)) {
          // O must hold P V of tile t-1 before it is rescaled (the partner warp rescales the
          // other 64 columns of the same rows with the same factor)
          ok = mbar_wait_warp(o_ready, (t - 1) & 1, abort_flag, p.status);
          if (!ok) break;
          tc_fence_after();
#pragma unroll 1
          for (int cc = 0; cc < 2; ++cc) {
            uint32_t o[32];
            tmem_ld32(tO + 32u * cc, o);
#pragma unroll
            for (int j = 0; j < 32; ++j) o[j] = __float_as_uint(__uint_as_float(o[j]) * alpha);
            tmem_st32(tO + 32u * cc, o);
          }
        }
        tmem_st_wait();
        if (key0 + BN > nkeys) {
          // zero V rows past the end of the sequence (their P is 0, but the cache slots may
          // hold non-finite garbage and 0 * inf would poison O)
          const int sv = t % SV;
          ok = mbar_wait_warp(full_v(sv), (t / SV) & 1, abort_flag, p.status);
          if (!ok) break;
          const int jv = nkeys - key0;
          const int nz = (BN - jv) * 16;
          for (int c = (hh * nact + q4) * 32 + lane; c < nz; c += 64 * nact) {
            const int key = jv + (c >> 4), h = (c >> 3) & 1, j = c & 7;
            const int off = (key / rpb) * rpb * 256 + h * rpb * 128 + (key % rpb) * 128 + j * 16;
            *reinterpret_cast<uint4*>(sptr + C::OFF_V + sv * KTILE + off) = make_uint4(0u, 0u, 0u, 0u);
          }
          fence_proxy_async_smem();
        }
        tc_fence_before();
        mbar_arrive(p_full(sb));
      }
      if (ok) {  // the row's sum over both halves
        float lo;
        ok = exchange(nt, l_sum, &lo);
        if (ok) l_sum += lo;
      }
      if (ok) ok = mbar_wait_warp(o_final, 0, abort_flag, p.status);
      if (ok) {
        tc_fence_after();
        const int head = kvh * p.g + (valid ? grow % p.g : 0);
        if (direct) {
          const float inv = (valid && l_sum > 0.f) ? 1.f / l_sum : 0.f;
          __nv_bfloat16* dst = p.out + ((static_cast<long long>(b) * p.m + node) * p.Hq + head) * HD + 64 * hh;
#pragma unroll 1
          for (int cc = 0; cc < 2; ++cc) {
            uint32_t o[32];
            tmem_ld32(tO + 32u * cc, o);
            if (valid) {
#pragma unroll
              for (int v4 = 0; v4 < 4; ++v4) {
                uint4 w;
                w.x = pack_bf16x2(__uint_as_float(o[8 * v4 + 0]) * inv, __uint_as_float(o[8 * v4 + 1]) * inv);
                w.y = pack_bf16x2(__uint_as_float(o[8 * v4 + 2]) * inv, __uint_as_float(o[8 * v4 + 3]) * inv);
                w.z = pack_bf16x2(__uint_as_float(o[8 * v4 + 4]) * inv, __uint_as_float(o[8 * v4 + 5]) * inv);
                w.w = pack_bf16x2(__uint_as_float(o[8 * v4 + 6]) * inv, __uint_as_float(o[8 * v4 + 7]) * inv);
                *reinterpret_cast<uint4*>(dst + cc * 32 + v4 * 8) = w;
              }
            }
          }
          if (valid && hh == 0 && p.lse != nullptr)
            p.lse[(static_cast<long long>(b) * p.m + node) * p.Hq + head] = (m_ref + log2f(l_sum)) * kLn2;
        } else if (p.mode == kGlobal) {
          const long long prow = (static_cast<long long>(bk) * p.rows + grow) * p.nchunk + chunk;
          float* dst = p.part_o + prow * HD + 64 * hh;
#pragma unroll 1
          for (int cc = 0; cc < 2; ++cc) {
            uint32_t o[32];
            tmem_ld32(tO + 32u * cc, o);
            if (valid) {
#pragma unroll
              for (int v4 = 0; v4 < 8; ++v4)
                *reinterpret_cast<float4*>(dst + cc * 32 + v4 * 4) =
                    make_float4(__uint_as_float(o[4 * v4]), __uint_as_float(o[4 * v4 + 1]),
                                __uint_as_float(o[4 * v4 + 2]), __uint_as_float(o[4 * v4 + 3]));
            }
          }
          if (valid && hh == 0) p.part_ml[prow] = make_float2(m_ref, l_sum);
        }
        // cluster mode: O stays in TMEM until every CTA of the cluster has left its loop
      }
    }
  }

  if (p.mode == kCluster) {
    // Merge through distributed shared memory.  Rows of the row group are split evenly over
    // the cs CTAs ("owners"); slot (c, row) of an owner's receive area holds CTA c's partial.
    // 1) barrier: every CTA has left its loop, so all K rings are idle and reusable;
    // 2) every CTA pushes its (max, sum) and fp32 O rows into the owners' rings with remote
    //    stores (no round trips); 3) barrier: all pushes are visible; 4) each owner merges
    //    its rows from local shared memory and writes the output.
    const int cs = p.nchunk;
    const int q = chunk;  // this CTA's place among the chunks of its row group
    auto rank_of = [&](int c) { return static_cast<uint32_t>(crank + mc * c); };
    const int per = BM / cs;  // cs divides 128
    tc_fence_before();
    cluster_sync_all();
    if (warp >= 4 && warp < C::EXTRA_WARP) {
      const int hh = (warp - 4) >> 2;
      const int Rl = (warp & 3) * 32 + lane;
      const bool have = ok && nt > 0 && Rl < rows_here;
      const int owner = Rl / per;
      const int slot = q * per + (Rl - owner * per);
      if (hh == 0) {
        const float2 ml = have ? make_float2(m_ref, l_sum) : make_float2(-INFINITY, 0.f);
        st_dsmem_f2(dsmem_addr(sbase + C::OFF_ML + 8u * slot, rank_of(owner)), ml);
      }
      if (__any_sync(0xffffffffu, have)) {  // tcgen05.ld is warp-wide
        tc_fence_after();
        const uint32_t tO = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16) + 64u * hh;
#pragma unroll 1
        for (int cc = 0; cc < 2; ++cc) {
          uint32_t o[32];
          tmem_ld32(tO + 32u * cc, o);
          if (have) {
#pragma unroll
            for (int v4 = 0; v4 < 8; ++v4)
              st_dsmem_u4(dsmem_addr(sbase + C::OFF_K + orow_off(slot, 16 * hh + cc * 8 + v4), rank_of(owner)),
                          make_uint4(o[4 * v4], o[4 * v4 + 1], o[4 * v4 + 2], o[4 * v4 + 3]));
          }
        }
      }
    }
    cluster_sync_all();
    // owner merge: one warp per row, lane c handles 16-byte chunk c of the row
    const float2* ml_local = reinterpret_cast<const float2*>(sptr + C::OFF_ML);
    for (int rr = warp; rr < per; rr += C::THREADS / 32) {
      const int Rl = q * per + rr;
      if (Rl >= rows_here) break;
      const int grow = R0 + Rl;
      float M = -INFINITY;
      float2 mls[kMaxCluster];
#pragma unroll
      for (int c = 0; c < kMaxCluster; ++c) {
        mls[c] = c < cs ? ml_local[c * per + rr] : make_float2(-INFINITY, 0.f);
        if (mls[c].y > 0.f) M = fmaxf(M, mls[c].x);
      }
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
      float Ls = 0.f;
#pragma unroll
      for (int c = 0; c < kMaxCluster; ++c) {
        if (!(mls[c].y > 0.f)) continue;
        const float w = ex2_approx(mls[c].x - M);
        Ls += w * mls[c].y;
        const float4 o = *reinterpret_cast<const float4*>(sptr + C::OFF_K + orow_off(c * per + rr, lane));
        acc.x += w * o.x;
        acc.y += w * o.y;
        acc.z += w * o.z;
        acc.w += w * o.w;
      }
      const float inv = Ls > 0.f ? 1.f / Ls : 0.f;
      const int node = grow / p.g, head = kvh * p.g + grow % p.g;
      const long long oo = ((static_cast<long long>(b) * p.m + node) * p.Hq + head) * HD + lane * 4;
      uint2 w2;
      w2.x = pack_bf16x2(acc.x * inv, acc.y * inv);
      w2.y = pack_bf16x2(acc.z * inv, acc.w * inv);
      *reinterpret_cast<uint2*>(p.out + oo) = w2;
      if (lane == 0 && p.lse != nullptr)
        p.lse[(static_cast<long long>(b) * p.m + node) * p.Hq + head] = (M + log2f(Ls)) * kLn2;
    }
  }
  tc_fence_before();
  if (mc > 1) cluster_sync_all();  // no CTA leaves while a peer may still address its shared memory
  else __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

// Split-K merge for the global mode: one warp per (sequence, KV head, row); rows of
// sequences that fit in one chunk were written directly by the attention kernel.
__global__ void __launch_bounds__(256) combine_kernel(const float* __restrict__ part_o,
                                                      const float2* __restrict__ part_ml,
                                                      const int32_t* __restrict__ prefix_len,
                                                      Params p, int total_rows) {
  pdl_wait();
  const int wid = blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (wid >= total_rows) return;
  const int bk = wid / p.rows, grow = wid % p.rows;
  const int b = bk / p.Hkv, kvh = bk % p.Hkv;
  const int L = prefix_len[b];
  if (L < 0 || L > p.max_prefix) return;
  const int T = (L + p.m + BN - 1) / BN;
  const int nc = p.nchunk;
  if (T <= p.tpc) return;  // one chunk: written directly by the attention kernel
  const long long prow = static_cast<long long>(wid) * nc;
  // chunk c holds tiles [c*tpc, (c+1)*tpc); chunks past the end wrote nothing.  The used
  // chunks are merged four at a time, all their loads issued before any is used, into a
  // running (max, sum, O) in the log2 domain.
  const int used = min(nc, (T + p.tpc - 1) / p.tpc);
  float M = -INFINITY, Ls = 0.f;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int c0 = 0; c0 < used; c0 += 4) {
    float2 ml[4];
    float4 o[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const bool have = c0 + u < used;
      ml[u] = have ? part_ml[prow + c0 + u] : make_float2(-INFINITY, 0.f);
      o[u] = have ? reinterpret_cast<const float4*>(part_o + (prow + c0 + u) * HD)[lane] : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      if (!(ml[u].y > 0.f)) continue;
      if (ml[u].x > M) {
        const float r = exp2f(M - ml[u].x);  // 0 while M is -inf
        Ls *= r;
        acc.x *= r;
        acc.y *= r;
        acc.z *= r;
        acc.w *= r;
        M = ml[u].x;
      }
      const float w = exp2f(ml[u].x - M);
      Ls += w * ml[u].y;
      acc.x += w * o[u].x;
      acc.y += w * o[u].y;
      acc.z += w * o[u].z;
      acc.w += w * o[u].w;
    }
  }
  const float inv = Ls > 0.f ? 1.f / Ls : 0.f;
  const int node = grow / p.g, head = kvh * p.g + grow % p.g;
  const long long oo = ((static_cast<long long>(b) * p.m + node) * p.Hq + head) * HD + lane * 4;
  uint2 w;
  w.x = pack_bf16x2(acc.x * inv, acc.y * inv);
  w.y = pack_bf16x2(acc.z * inv, acc.w * inv);
  *reinterpret_cast<uint2*>(p.out + oo) = w;
  if (lane == 0 && p.lse != nullptr)
    p.lse[(static_cast<long long>(b) * p.m + node) * p.Hq + head] = (M + log2f(Ls)) * kLn2;
}

static cudaError_t set_smem_attr() {
  static std::once_flag once;
  static cudaError_t err = cudaSuccess;
  std::call_once(once, [] {
    err = cudaFuncSetAttribute(tree_attn_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM_BYTES);
  });
  return err;
}

// How many clusters of cx x cy CTAs (one per SM) the device runs at once; 0 if unknown.
static int active_clusters(int cx, int cy) {
  static std::mutex mu;
  static int cache[kMaxCluster + 1][kMaxCluster + 1] = {};
  static bool done[kMaxCluster + 1][kMaxCluster + 1] = {};
  if (cx < 1 || cy < 1 || cx * cy > kMaxCluster) return 0;
  std::lock_guard<std::mutex> lock(mu);
  if (done[cx][cy]) return cache[cx][cy];
  done[cx][cy] = true;
  if (set_smem_attr() != cudaSuccess) return 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(cx, cy, 1);
  cfg.blockDim = dim3(Cfg::THREADS, 1, 1);
  cfg.dynamicSmemBytes = Cfg::SMEM_BYTES;
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeClusterDimension;
  attr.val.clusterDim.x = cx;
  attr.val.clusterDim.y = cy;
  attr.val.clusterDim.z = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, tree_attn_tc_kernel, &cfg) != cudaSuccess) {
    cudaGetLastError();
    n = 0;
  }
  cache[cx][cy] = n;
  return n;
}

struct Plan {
  int rowgroups, mc, nc, tpc, mode;
};

// Row groups that share each K/V tile through TMA multicast: all of them up to four, else the
// largest of 4, 3, 2 that divides their number; 1 when the device cannot co-schedule such
// clusters or TREESPEC_ATTN_MC=1 is set (tests and tuning).
static int multicast_width(int rowgroups) {
  if (const char* ov = std::getenv("TREESPEC_ATTN_MC"))
    if (std::strcmp(ov, "1") == 0) return 1;
  int mc = 1;
  if (rowgroups <= 4) mc = rowgroups;
  else if (rowgroups % 4 == 0) mc = 4;
  else if (rowgroups % 3 == 0) mc = 3;
  else if (rowgroups % 2 == 0) mc = 2;
  if (mc > 1 && active_clusters(mc, 1) <= 0) mc = 1;
  return mc;
}

// Makespan model (microseconds).  A CTA streams tpc tiles of 128 keys at the larger of its
// own pipeline rate (tau_c per tile) and its share of the HBM bandwidth when `active` CTAs
// stream at once (each K/V tile is 64 KB, shared by the row groups of a unit), plus a fixed
// cost per CTA (set-up, pipeline fill and drain, epilogue) and the merge of the split.
struct CostModel {
  double tau_c, c0, hbm_bytes_per_us, cluster_merge, global_merge;
};

static double makespan(const CostModel& cm, int unit_groups, int tpc, long long waves, long long active,
                       double merge) {
  const double tau_h = 65536.0 * static_cast<double>(active) / static_cast<double>(unit_groups) / cm.hbm_bytes_per_us;
  const double tau = cm.tau_c > tau_h ? cm.tau_c : tau_h;
  return static_cast<double>(waves) * (tpc * tau + cm.c0) + merge;
}

static Plan make_plan(int B, int m, int Hq, int Hkv, int max_prefix, int num_sms) {
  Plan pl;
  if (num_sms < 1) num_sms = 1;
  const int rows = m * (Hq / Hkv);
  pl.rowgroups = (rows + BM - 1) / BM;
  const int T = (max_prefix + m + BN - 1) / BN;
  const long long units = static_cast<long long>(B) * Hkv * pl.rowgroups;
  pl.mc = multicast_width(pl.rowgroups);
  // CTAs resident at once: clusters of mc row groups are placed whole
  long long slots = num_sms;
  if (pl.mc > 1) slots = static_cast<long long>(active_clusters(pl.mc, 1)) * pl.mc;
  // calibrated on the GB300 (128-row CTAs: ~1.25 us per 128-key tile; ~20 us per CTA of set-up,
  // pipeline fill, drain and epilogue, which makes fewer and longer CTAs the better split)
  const CostModel cm{1.25, 20.0, 6.5e6, 1.5, 3.0};
  double best = -1.0;
  pl.nc = 1;
  pl.tpc = T;
  pl.mode = kDirect;
  const int max_nc = T < 1024 ? T : 1024;
  for (int nc = 1; nc <= max_nc; ++nc) {
    const int tpc = (T + nc - 1) / nc;
    if ((T + tpc - 1) / tpc != nc) continue;
    if (tpc * (BN / 16) > kMaxChunkBoxes) continue;  // box ids staged for the smallest pages
    const long long ctas = units * nc;
    const long long waves = (ctas + slots - 1) / slots;
    const long long active = ctas < slots ? ctas : slots;
    const double cost = makespan(cm, pl.rowgroups, tpc, waves, active, nc > 1 ? cm.global_merge : 0.0);
    if (best < 0 || cost < best) {
      best = cost;
      pl.nc = nc;
      pl.tpc = tpc;
      pl.mode = nc > 1 ? kGlobal : kDirect;
    }
  }
  // The model assumes every sequence is max_prefix long.  When it keeps one chunk and a wave
  // of such CTAs leaves SMs idle, a batch of several sequences is split in two chunks of
  // ceil(T/2) tiles: with prefixes of mixed lengths only the sequences longer than that use the
  // second chunk (the others' CTAs leave at once), and the longest sequences, dispatched
  // first, no longer set the whole call's length.
  if (pl.nc == 1 && B > 1 && units < num_sms && T >= 4) {
    const int tpc = (T + 1) / 2;
    if (tpc * (BN / 16) <= kMaxChunkBoxes) {
      pl.nc = 2;
      pl.tpc = tpc;
      pl.mode = kGlobal;
    }
  }
  // Optional override for tests and tuning: TREESPEC_ATTN_SPLIT=direct | cluster:N | global:N
  // (ignored when the requested split is not feasible for these sizes; the chunk cluster is
  // only used without multicast).
  if (const char* ov = std::getenv("TREESPEC_ATTN_SPLIT")) {
    int n = 0;
    if (std::strcmp(ov, "direct") == 0) {
      if (T * (BN / 16) <= kMaxChunkBoxes) {
        pl.nc = 1;
        pl.tpc = T;
        pl.mode = kDirect;
        return pl;
      }
    } else if (std::sscanf(ov, "cluster:%d", &n) == 1 && (n == 2 || n == 4 || n == 8) && T >= n &&
               pl.mc * n <= kMaxCluster) {
      const int tpc = (T + n - 1) / n;
      if ((T + tpc - 1) / tpc == n && tpc * (BN / 16) <= kMaxChunkBoxes && active_clusters(pl.mc, n) > 0) {
        pl.nc = n;
        pl.tpc = tpc;
        pl.mode = kCluster;
        return pl;
      }
    } else if (std::sscanf(ov, "global:%d", &n) == 1 && n >= 2 && n <= T) {
      const int tpc = (T + n - 1) / n;
      if (tpc * (BN / 16) <= kMaxChunkBoxes) {
        pl.nc = (T + tpc - 1) / tpc;
        pl.tpc = tpc;
        pl.mode = pl.nc > 1 ? kGlobal : kDirect;
        return pl;
      }
    }
  }
  for (int cs = 2; pl.mc * cs <= kMaxCluster; cs *= 2) {
    if (T < cs) break;
    const int tpc = (T + cs - 1) / cs;
    if ((T + tpc - 1) / tpc != cs) continue;
    if (tpc * (BN / 16) > kMaxChunkBoxes) continue;
    const int act = active_clusters(pl.mc, cs);  // clusters of mc row groups x cs chunks
    if (act <= 0) continue;
    const long long clusters = units / pl.mc;
    const long long waves = (clusters + act - 1) / act;
    const long long ctas = units * cs;
    const long long active = ctas < static_cast<long long>(act) * pl.mc * cs ? ctas
                                                                            : static_cast<long long>(act) * pl.mc * cs;
    const double cost = makespan(cm, pl.rowgroups, tpc, waves, active, cm.cluster_merge);
    if (cost < best) {
      best = cost;
      pl.nc = cs;
      pl.tpc = tpc;
      pl.mode = kCluster;
    }
  }
  return pl;
}

using EncodeFn = PFN_cuTensorMapEncodeTiled_v12000;

static EncodeFn get_encode() {
  static EncodeFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeFn>(f);
  });
  return fn;
}

// Tensor maps of a paged cache [num_blocks, Hkv, bs, 128] bf16, 128-byte swizzle.
//   kHalfBox: dims {128, bs, Hkv, blocks}, box {64, rows, 1, 1}: one head-dim half of `rows`
//             rows (rows = min(bs, 64)).
//   kPageBox: dims {64, bs, 2, Hkv, blocks} (the head dim split into its two halves, the half
//             index strided by 128 B), box {64, rows, 2, 1, 1}: both halves of `rows` rows in
//             one copy, landing as [half][rows][64].
enum MapKind { kHalfBox = 0, kPageBox = 1 };

static bool encode_kv_map(CUtensorMap* map, const void* base, int num_blocks, int Hkv, int bs, int kind) {
  EncodeFn enc = get_encode();
  if (enc == nullptr) return false;
  const cuuint32_t rows = static_cast<cuuint32_t>(bs < 64 ? bs : 64);
  const cuuint64_t row_b = static_cast<cuuint64_t>(HD) * 2;
  const cuuint64_t head_b = static_cast<cuuint64_t>(bs) * row_b;
  const cuuint64_t block_b = static_cast<cuuint64_t>(Hkv) * head_b;
  const cuuint32_t estr[5] = {1u, 1u, 1u, 1u, 1u};
  if (kind == kHalfBox) {
    const cuuint64_t dims[4] = {static_cast<cuuint64_t>(HD), static_cast<cuuint64_t>(bs),
                                static_cast<cuuint64_t>(Hkv), static_cast<cuuint64_t>(num_blocks)};
    const cuuint64_t strides[3] = {row_b, head_b, block_b};
    const cuuint32_t box[4] = {64u, rows, 1u, 1u};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
  }
  const cuuint64_t dims[5] = {64u, static_cast<cuuint64_t>(bs), 2u, static_cast<cuuint64_t>(Hkv),
                              static_cast<cuuint64_t>(num_blocks)};
  const cuuint64_t strides[4] = {row_b, 128u, head_b, block_b};
  const cuuint32_t box[5] = {64u, rows, 2u, 1u, 1u};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Small cache of encoded K/V tensor maps keyed by (base pointer, shape, kind): encoding is a
// host-side driver call, and serving loops reuse the same cache tensors every step.
struct MapEntry {
  const void* base;
  int num_blocks, Hkv, bs, kind;
  CUtensorMap map;
  uint64_t stamp;
};

static bool cached_kv_map(CUtensorMap* out, const void* base, int num_blocks, int Hkv, int bs, int kind) {
  constexpr int kSlots = 16;
  static MapEntry cache[kSlots] = {};
  static uint64_t clock = 0;
  static std::mutex mu;
  std::lock_guard<std::mutex> lock(mu);
  ++clock;
  int victim = 0;
  for (int i = 0; i < kSlots; ++i) {
    MapEntry& e = cache[i];
    if (e.stamp != 0 && e.base == base && e.num_blocks == num_blocks && e.Hkv == Hkv && e.bs == bs &&
        e.kind == kind) {
      e.stamp = clock;
      *out = e.map;
      return true;
    }
    if (e.stamp < cache[victim].stamp) victim = i;
  }
  MapEntry e{base, num_blocks, Hkv, bs, kind, {}, clock};
  if (!encode_kv_map(&e.map, base, num_blocks, Hkv, bs, kind)) return false;
  cache[victim] = e;
  *out = e.map;
  return true;
}

// A failed CUDA call maps to TS_ERR_CUDA; with TREESPEC_DEBUG set in the environment the
// call site and the CUDA error string also go to stderr.
static int cuda_fail(cudaError_t e, const char* where) {
  if (std::getenv("TREESPEC_DEBUG") != nullptr)
    std::fprintf(stderr, "treespec: tree_attention %s: %s\n", where, cudaGetErrorString(e));
  return TS_ERR_CUDA;
}

static int launch_kernel(const CUtensorMap& mk, const CUtensorMap& mv, const Params& prm, const Plan& pl, int B,
                         int Hkv, cudaStream_t stream) {
  const cudaError_t ea = set_smem_attr();
  if (ea != cudaSuccess) return cuda_fail(ea, "shared-memory attribute");
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(pl.rowgroups, pl.nc, B * Hkv);
  cfg.blockDim = dim3(Cfg::THREADS, 1, 1);
  cfg.dynamicSmemBytes = Cfg::SMEM_BYTES;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (pl.mode == kCluster || pl.mc > 1) {
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = pl.mc;
    attr[1].val.clusterDim.y = pl.mode == kCluster ? pl.nc : 1;
    attr[1].val.clusterDim.z = 1;
    cfg.numAttrs = 2;
  }
  const cudaError_t el = cudaLaunchKernelEx(&cfg, tree_attn_tc_kernel, mk, mv, prm);
  return el == cudaSuccess ? TS_OK : cuda_fail(el, "launch");
}

}  // namespace tc

bool attention_uses_tc(ts_dtype dt, int d, int block_size) {
  return dt == TS_BF16 && d == tc::HD &&
         (block_size == 16 || block_size == 32 || block_size == 64 || block_size == 128);
}

size_t attention_tc_workspace_bytes(int B, int m, int Hq, int Hkv, int max_prefix, int num_sms) {
  const tc::Plan pl = tc::make_plan(B, m, Hq, Hkv, max_prefix, num_sms);
  if (pl.mode != tc::kGlobal) return 256;
  const size_t prow = static_cast<size_t>(B) * Hkv * m * (Hq / Hkv) * pl.nc;
  return prow * tc::HD * 4 + prow * 8 + 512;
}

void attention_tc_plan(int B, int m, int Hq, int Hkv, int max_prefix, int num_sms, int* out5) {
  const tc::Plan pl = tc::make_plan(B, m, Hq, Hkv, max_prefix, num_sms);
  out5[0] = pl.rowgroups;
  out5[1] = pl.nc;
  out5[2] = pl.tpc;
  out5[3] = pl.mode;
  out5[4] = pl.mc;
}

int attention_tc_launch(const AttnArgs& a, int num_sms) {
  const tc::Plan pl = tc::make_plan(a.B, a.m, a.Hq, a.Hkv, a.max_prefix, num_sms);
  CUtensorMap mk, mv;
  if (!tc::cached_kv_map(&mk, a.k_cache, a.num_blocks, a.Hkv, a.block_size, tc::kHalfBox) ||
      !tc::cached_kv_map(&mv, a.v_cache, a.num_blocks, a.Hkv, a.block_size, tc::kPageBox))
    return tc::cuda_fail(cudaErrorInvalidValue, "tensor map encode");
  tc::Params prm;
  prm.q = static_cast<const __nv_bfloat16*>(a.q);
  prm.block_table = a.block_table;
  prm.prefix_len = a.prefix_len;
  prm.mask = a.mask;
  prm.out = static_cast<__nv_bfloat16*>(a.out);
  prm.lse = a.lse;
  prm.status = a.dev_status;
  prm.B = a.B;
  prm.m = a.m;
  prm.Hq = a.Hq;
  prm.Hkv = a.Hkv;
  prm.g = a.Hq / a.Hkv;
  prm.rows = a.m * prm.g;
  prm.W = (a.m + 63) / 64;
  prm.max_blocks = a.max_blocks;
  prm.num_blocks = a.num_blocks;
  prm.block_size = a.block_size;
  prm.max_prefix = a.max_prefix;
  prm.tpc = pl.tpc;
  prm.nchunk = pl.nc;
  prm.mode = pl.mode;
  prm.mc = pl.mc;
  // two MMA-issuing threads pay off where the tensor cores set the pace (several row groups);
  // with one row group the single issuer is 2% faster
  prm.split_issue = pl.rowgroups >= 2 ? 1 : 0;
  if (const char* ov = std::getenv("TREESPEC_ATTN_ISSUE")) {
    if (std::strcmp(ov, "1") == 0) prm.split_issue = 0;
    else if (std::strcmp(ov, "2") == 0) prm.split_issue = 1;
  }
  prm.scale_log2 = a.scale * 1.4426950408889634f;
  const size_t prow = static_cast<size_t>(a.B) * a.Hkv * prm.rows * pl.nc;
  prm.part_o = pl.mode == tc::kGlobal ? static_cast<float*>(a.workspace) : nullptr;
  prm.part_ml = pl.mode == tc::kGlobal
                    ? reinterpret_cast<float2*>(static_cast<char*>(a.workspace) + prow * tc::HD * 4)
                    : nullptr;
  const int rc = tc::launch_kernel(mk, mv, prm, pl, a.B, a.Hkv, a.stream);
  if (rc != TS_OK) return rc;
  int launches = 1;
  if (pl.mode == tc::kGlobal) {
    const int total_rows = a.B * a.Hkv * prm.rows;
    const cudaError_t ec = launch_pdl(tc::combine_kernel, dim3((total_rows + 7) / 8), dim3(256), 0, a.stream,
                                      prm.part_o, prm.part_ml, a.prefix_len, prm, total_rows);
    if (ec != cudaSuccess) return tc::cuda_fail(ec, "combine launch");
    ++launches;
  }
  count_launches(launches);
  const cudaError_t eg = cudaGetLastError();
  return eg == cudaSuccess ? TS_OK : tc::cuda_fail(eg, "after launch");
}

}  // namespace ts
