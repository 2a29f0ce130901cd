// ts_tree_attention, tensor-core path (bf16, head dim 128) for sm_103a.
//
// Source: "rainlin.net/posts/eagle", section 四 Tree Attention (node i attends to the
// prefix and to its own root-to-node ancestors only; one pass verifies every path);
// "lesty.tech — EAGLE-2 vs. Medusa", section 5 (the tree mask stays on chip, no global
// re-reads) and section 8 (tree K/V sit in the same paged sequence after the prefix).
//
// Work unit: (sequence b, KV head, row group, chunk of 64-key tiles).  The g query heads
// that share a KV head and the m tree nodes are packed into GEMM rows, row = node*g +
// head-in-group, so every K/V byte fetched from HBM serves m*g query rows on the tensor
// cores.  A row group is one (NM = 1) or two (NM = 2) 128-row M tiles.  One CTA per SM.
//
// Warp roles (4 + 4*NM warps, then the extra producer warps; 288 threads for NM = 1, 384 for 2):
//   warps 0,2,3 and the warps after the softmax warps
//               warp 0 stages the chunk's physical block ids in shared memory; then one
//               thread per producer warp issues TMA loads (K: warps 0 and 3; V: warp 2 and,
//               for one-tile groups, the last warp; each an even share of every tile's
//               boxes): per 64-key tile one box of min(block_size,64) rows x 64 bf16
//               (128-byte swizzle) per page and head-dim half; positions past the sequence
//               load an out-of-range block (zero fill).  STAGES-deep ring; each full barrier
//               expects every producer of its operand.
//   warp 1      TMEM allocator + the single thread that issues tcgen05.mma:
//                 S_i = Q_i K^T     (M=128, N=64, K=128; A, B from shared memory)
//                 O_i += P_i V      (M=128, N=128, K=64; A = P from TMEM, B = V MN-major)
//   warps 4..   softmax, one thread per row (TMEM lane): load S, apply the tree mask on the
//               tiles that reach the tree, online softmax in the log2 domain with lazy
//               rescaling of O (only when the running max grows by more than 2^8), write P
//               as bf16 into TMEM; then the epilogue.
// Overlap: with one M tile, S and P are double-buffered in TMEM (S = Q K^T of tile t+2 runs
// while tile t's softmax runs); with two M tiles the MMAs of one tile run during the
// other tile's softmax.  P never aliases S.
// TMEM columns: O_i at 128*i; S_{i,s} at 128*NM + 64*(i*SB + s); P_{i,s} after the S
// buffers, 32 columns each.
// Split over chunks of one (sequence, KV head, row group):
//   direct   one chunk: the epilogue writes O / l.
//   cluster  the chunks are the CTAs of one thread-block cluster (<= 8): after a cluster
//            barrier each CTA stores its fp32 O rows and (max, sum) straight into the shared
//            memory of the CTA that owns those rows (distributed shared memory), and after a
//            second barrier every owner merges its rows locally and writes the output: no
//            partials in HBM and no second launch.
// Chunks are balanced: chunk c of a sequence of T tiles covers [c*T/nc, (c+1)*T/nc).
//   global   more chunks than a cluster holds: fp32 partials go to the workspace and
//            combine_kernel merges them.
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

constexpr int BN = 64;    // keys per tile
constexpr int BM = 128;   // rows per M tile
constexpr int HD = 128;   // head dim
constexpr uint32_t QHALF = BM * 128;   // 128 rows x 64 bf16 = 16 KB
constexpr uint32_t QTILE = 2 * QHALF;  // both head-dim halves
constexpr uint32_t KHALF = BN * 128;   // 64 keys x 64 bf16 = 8 KB
constexpr uint32_t KTILE = 2 * KHALF;  // 16 KB
constexpr float kRescaleThreshold = 8.0f;  // log2 units
constexpr int kMaxChunkBoxes = 2048;       // physical-block ids a CTA stages in shared memory
constexpr int kMaxCluster = 8;
constexpr float kLn2 = 0.69314718055994530942f;

enum Mode { kDirect = 0, kCluster = 1, kGlobal = 2 };

template <int NM>
struct Cfg {
  static constexpr int SB = NM == 1 ? 2 : 1;  // S / P buffers per M tile
  static constexpr int STAGES = NM == 1 ? 5 : 4;
  // A TMA instruction holds its issuing thread for a while (~0.19 us for a page-sized box),
  // so the boxes of a tile are spread over K_PRODUCERS + V_PRODUCERS warps.  Two-tile groups
  // are bound by their MMAs (a tile takes ~1.7 us, ~142 cycles per tcgen05.mma, against
  // ~0.8 us of box issue per producer warp) and keep a single V warp; more producer warps
  // (up to four of each) measured no faster in either group.  Warps 0 and 3 issue K, warp 2
  // V, and the warps after the softmax warps (from EXTRA_WARP on) the remaining V parts,
  // then K parts.
  static constexpr int K_PRODUCERS = 2;
  static constexpr int V_PRODUCERS = NM == 1 ? 2 : 1;
  static constexpr int EXTRA_WARP = 4 + 4 * NM;
  static constexpr int THREADS = 32 * (EXTRA_WARP + (K_PRODUCERS - 2) + (V_PRODUCERS - 1));
  static constexpr uint32_t TMEM_COLS = 512;
  static constexpr uint32_t COL_S = 128 * NM;
  static constexpr uint32_t COL_P = COL_S + 64 * NM * SB;
  static constexpr uint32_t OFF_Q = 0;
  static constexpr uint32_t OFF_K = NM * QTILE;
  static constexpr uint32_t OFF_V = OFF_K + STAGES * KTILE;
  static constexpr uint32_t OFF_BAR = OFF_V + STAGES * KTILE;
  // full_k[ST] full_v[ST] empty_k[ST] empty_v[ST] s_full[NM*SB] p_full[NM*SB] o_ready[NM] o_final[NM]
  // (p_full is per S buffer: with two buffers a fast softmax warp may reach tile t+1 while
  // slower warps of its M tile still work on tile t, and their arrivals must not mix)
  static constexpr int NBAR = 4 * STAGES + 2 * NM * SB + 2 * NM;
  static constexpr uint32_t OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr uint32_t OFF_ML = OFF_MISC + 16;            // (max, sum) per row, cluster merge
  static constexpr uint32_t OFF_BLK = OFF_ML + NM * BM * 8;
  static constexpr uint32_t SMEM_BYTES = OFF_BLK + 4 * kMaxChunkBoxes + 1024;  // + alignment slack
  static_assert(COL_P + 32 * NM * SB <= TMEM_COLS, "TMEM budget");
  static_assert(2 * STAGES * KTILE >= NM * BM * 512, "O rows must fit in the K/V ring for the merge");
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
  int m, Hq, Hkv, g, rows, W, max_blocks, num_blocks, block_size, max_prefix, tpc, nchunk, mode;
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

template <int NM>
__global__ void __launch_bounds__(Cfg<NM>::THREADS, 1)
    tree_attn_tc_kernel(const __grid_constant__ CUtensorMap tmk,
                        const __grid_constant__ CUtensorMap tmv, const Params p) {
  using C = Cfg<NM>;
  constexpr int ST = C::STAGES;
  constexpr int SB = C::SB;
  extern __shared__ unsigned char smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  unsigned char* sptr = smem_raw + (sbase - raw);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rg = blockIdx.x, chunk = blockIdx.y, bk = blockIdx.z;
  const int b = bk / p.Hkv, kvh = bk % p.Hkv;
  pdl_wait();
  const int L = p.prefix_len[b];
  // (the whole cluster shares b, so every CTA of a cluster returns here together)
  if (L < 0 || L > p.max_prefix) {
    if (threadIdx.x == 0 && rg == 0 && chunk == 0) report(p.status, TS_ERR_DEVICE_CHECK);
    return;
  }
  const int nkeys = L + p.m;
  const int T = (nkeys + BN - 1) / BN;
  // balanced chunks: chunk c covers tiles [ceil(c*T/nc), ceil((c+1)*T/nc)) of this sequence,
  // so the chunks that get one tile more are the first ones and the last chunk, which holds
  // the masked tree tile, is never the longest
  const int t0 = static_cast<int>((static_cast<long long>(chunk) * T + p.nchunk - 1) / p.nchunk);
  const int nt = static_cast<int>((static_cast<long long>(chunk + 1) * T + p.nchunk - 1) / p.nchunk) - t0;
  if (nt == 0 && p.mode != kCluster) return;  // (an idle CTA of a cluster still merges)
  // a sequence whose tiles all fall into one chunk is written directly also in the global mode
  const bool direct = p.mode == kDirect || (p.mode == kGlobal && min(T, p.nchunk) == 1);
  const int R0 = rg * NM * BM;
  const int rows_here = min(p.rows - R0, NM * BM);
  const int nma = (rows_here + BM - 1) / BM;

  auto bar = [&](int idx) -> uint32_t { return sbase + C::OFF_BAR + 8u * idx; };
  auto full_k = [&](int s) { return bar(s); };
  auto full_v = [&](int s) { return bar(ST + s); };
  auto empty_k = [&](int s) { return bar(2 * ST + s); };
  auto empty_v = [&](int s) { return bar(3 * ST + s); };
  auto s_full = [&](int i, int sb) { return bar(4 * ST + i * SB + sb); };
  auto p_full = [&](int i, int sb) { return bar(4 * ST + NM * SB + i * SB + sb); };
  auto o_ready = [&](int i) { return bar(4 * ST + 2 * NM * SB + i); };
  auto o_final = [&](int i) { return bar(4 * ST + 2 * NM * SB + NM + i); };
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sptr + C::OFF_MISC);
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(sptr + C::OFF_MISC + 4);
  float2* s_ml = reinterpret_cast<float2*>(sptr + C::OFF_ML);

  if (threadIdx.x == 0) {
    for (int s = 0; s < ST; ++s) {
      mbar_init(full_k(s), C::K_PRODUCERS);  // each producer warp registers its own bytes
      mbar_init(full_v(s), C::V_PRODUCERS);
      mbar_init(empty_k(s), 1);
      mbar_init(empty_v(s), 1);
    }
    for (int i = 0; i < NM; ++i) {
      for (int sb = 0; sb < SB; ++sb) {
        mbar_init(s_full(i, sb), 1);
        mbar_init(p_full(i, sb), 128);
      }
      mbar_init(o_ready(i), 1);
      mbar_init(o_final(i), 1);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_holder), C::TMEM_COLS);
    tmem_relinquish();
  }
  // Q rows of this row group -> shared memory in the 128-byte-swizzled K-major layout
  // (16-byte chunk j of row r stored at chunk j ^ (r % 8)); padding rows are zero.  Loads
  // are issued in batches of 4 per thread so their latencies overlap.
  for (int c0 = threadIdx.x; c0 < NM * BM * 16; c0 += 4 * C::THREADS) {
    uint4 v[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int c = c0 + u * C::THREADS;
      const int row = c >> 4, h = (c >> 3) & 1, j = c & 7;
      const int grow = R0 + row;
      v[u] = make_uint4(0u, 0u, 0u, 0u);
      if (nt > 0 && c < NM * BM * 16 && grow < p.rows) {
        const int node = grow / p.g, head = kvh * p.g + grow % p.g;
        const long long off = ((static_cast<long long>(b) * p.m + node) * p.Hq + head) * HD + h * 64 + j * 8;
        v[u] = __ldg(reinterpret_cast<const uint4*>(p.q + off));
      }
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int c = c0 + u * C::THREADS;
      if (c >= NM * BM * 16) break;
      const int row = c >> 4, h = (c >> 3) & 1, j = c & 7;
      const int i = row >> 7, r = row & 127;
      *reinterpret_cast<uint4*>(sptr + C::OFF_Q + i * QTILE + h * QHALF + r * 128 + ((j ^ (r & 7)) << 4)) = v[u];
    }
  }
  // Physical block of every TMA box of this chunk -> shared memory (warp 0, coalesced,
  // 4 independent loads in flight per lane); out-of-range ids are reported and replaced by
  // the out-of-bounds block, positions past the sequence get the out-of-bounds block too.
  const int rpb = min(p.block_size, BN);
  const int bpt = BN / rpb;
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

  if (warp == 0 || warp == 2 || warp == 3 || warp >= C::EXTRA_WARP) {
    // ------------------------------ TMA producers ------------------------------
    // Part `part` of `nparts` issues boxes [part*nbox/nparts, (part+1)*nbox/nparts) of every
    // tile (a part may hold none: it still registers its zero bytes once per tile).
    if (lane == 0) {
      const int e = warp - C::EXTRA_WARP;  // index among the warps after the softmax warps
      const int kv = (warp == 0 || warp == 3 || (e >= 0 && e >= C::V_PRODUCERS - 1)) ? 0 : 1;
      const int part = warp == 0 ? 0 : warp == 3 ? 1 : warp == 2 ? 0 : kv == 1 ? e + 1 : 2 + e - (C::V_PRODUCERS - 1);
      const int nparts = kv == 0 ? C::K_PRODUCERS : C::V_PRODUCERS;
      const void* map = kv == 0 ? static_cast<const void*>(&tmk) : static_cast<const void*>(&tmv);
      const int nbox = 2 * bpt;                    // boxes per tile: pages x head-dim halves
      const int b_begin = part * nbox / nparts, b_end = (part + 1) * nbox / nparts;
      int issued = 0;
      for (int t = 0; t < nt; ++t) {
        const int s = t % ST;
        const uint32_t ph = (t / ST) & 1;
        const int key0 = (t0 + t) * BN;
        const uint32_t fb = kv == 0 ? full_k(s) : full_v(s);
        const uint32_t eb = kv == 0 ? empty_k(s) : empty_v(s);
        if (!mbar_wait(eb, ph ^ 1u, abort_flag, p.status)) break;
        mbar_expect_tx(fb, static_cast<uint32_t>(b_end - b_begin) * rpb * 128);
        const uint32_t dst0 = sbase + (kv == 0 ? C::OFF_K : C::OFF_V) + s * KTILE;
        for (int e = b_begin; e < b_end; ++e) {
          const int j = e >> 1, h = e & 1;      // page j of the tile, head-dim half h
          const int blk = s_blk[t * bpt + j];  // num_blocks (out of range) -> zero fill
          const int rin = blk < p.num_blocks ? (key0 + j * rpb) % p.block_size : 0;
          tma_load_4d(dst0 + h * KHALF + j * rpb * 128, map, fb, h * 64, rin, kvh, blk);
        }
        issued = t + 1;
      }
      if (*abort_flag) {
        for (int t = max(0, issued - ST); t < issued; ++t)
          drain_wait(kv == 0 ? full_k(t % ST) : full_v(t % ST), (t / ST) & 1);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------ MMA issuer ------------------------------
    if (lane == 0 && nt > 0) {
      constexpr uint32_t idq = idesc_bf16_f32(128, BN, 0, 0);
      constexpr uint32_t idp = idesc_bf16_f32(128, HD, 0, 1);
      auto tO = [&](int i) { return tmem + 128u * i; };
      auto tS = [&](int i, int sb) { return tmem + C::COL_S + 64u * (i * SB + sb); };
      auto tP = [&](int i, int sb) { return tmem + C::COL_P + 32u * (i * SB + sb); };
      auto qk = [&](int i, int s, int sb) {
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint32_t h = kk >> 2, ko = (kk & 3) * 32;
          const uint64_t a = sdesc_sw128(sbase + C::OFF_Q + i * QTILE + h * QHALF + ko, 16, 1024);
          const uint64_t bd = sdesc_sw128(sbase + C::OFF_K + s * KTILE + h * KHALF + ko, 16, 1024);
          mma_ss(tS(i, sb), a, bd, idq, kk > 0 ? 1u : 0u);
        }
        tc_commit(s_full(i, sb));
      };
      auto pv = [&](int i, int s, int sb, bool first) {
#pragma unroll
        for (int kk = 0; kk < BN / 16; ++kk) {
          // B = V tile, MN-major: 64 head-dim columns per 128-byte row, 8-key groups 1 KB
          // apart (stride offset), the second head-dim half KHALF further (leading offset).
          const uint64_t bd = sdesc_sw128(sbase + C::OFF_V + s * KTILE + kk * 2048, KHALF, 1024);
          mma_ts(tO(i), tP(i, sb) + 8u * kk, bd, idp, (first && kk == 0) ? 0u : 1u);
        }
      };
      bool mok = true;
      for (int t = 0; mok && t < SB && t < nt; ++t) {
        mok = mbar_wait(full_k(t % ST), (t / ST) & 1, abort_flag, p.status);
        if (!mok) break;
        tc_fence_after();
        for (int i = 0; i < nma; ++i) qk(i, t % ST, t % SB);
        tc_commit(empty_k(t % ST));
      }
      for (int t = 0; mok && t < nt; ++t) {
        const int s = t % ST;
        mok = mbar_wait(full_v(s), (t / ST) & 1, abort_flag, p.status);
        if (!mok) break;
        tc_fence_after();
        const int tn = t + SB;
        for (int i = 0; i < nma; ++i) {
          mok = mbar_wait(p_full(i, t % SB), (t / SB) & 1, abort_flag, p.status);
          if (!mok) break;
          tc_fence_after();
          pv(i, s, t % SB, t == 0);
          tc_commit(o_ready(i));
          if (tn < nt) {
            if (i == 0) {
              mok = mbar_wait(full_k(tn % ST), (tn / ST) & 1, abort_flag, p.status);
              if (!mok) break;
              tc_fence_after();
            }
            qk(i, tn % ST, tn % SB);
            if (i == nma - 1) tc_commit(empty_k(tn % ST));
          }
        }
        if (!mok) break;
        tc_commit(empty_v(s));
      }
      for (int i = 0; i < nma; ++i) tc_commit(o_final(i));
      if (!mok) {
        for (int i = 0; i < nma; ++i) drain_wait(o_final(i), 0);
      }
    }
    __syncwarp();
  } else if (warp >= 4 && warp < C::EXTRA_WARP) {
    // ------------------------------ softmax ------------------------------
    const int i = (warp - 4) >> 2;
    const int q4 = warp & 3;
    if (i < nma && nt > 0) {
      const int r = q4 * 32 + lane;
      const int grow = R0 + i * BM + r;
      const bool valid = grow < p.rows;
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
      const uint32_t tO = tmem + lane_off + 128u * i;
      const float sl2 = p.scale_log2;
      for (int t = 0; t < nt; ++t) {
        const int sb = t % SB;
        const uint32_t tS = tmem + lane_off + C::COL_S + 64u * (i * SB + sb);
        const uint32_t tP = tmem + lane_off + C::COL_P + 32u * (i * SB + sb);
        ok = mbar_wait_warp(s_full(i, sb), (t / SB) & 1, abort_flag, p.status);
        if (!ok) break;
        tc_fence_after();
        float s[BN];
        {
          uint32_t u[BN];
          tmem_ld64(tS, u);
#pragma unroll
          for (int c = 0; c < BN; ++c) s[c] = __uint_as_float(u[c]);
        }
        const int key0 = (t0 + t) * BN;
        float mx = -INFINITY;
        if (key0 + BN > L) {
          // one visibility bit per column: the prefix columns, then this row's ancestor bits of
          // the tree positions the tile covers (positions at or past m are never visible)
          const int pre = L - key0;             // prefix columns in this tile (< 64)
          const int tt0 = pre > 0 ? 0 : -pre;   // first tree position in this tile
          const int q = tt0 >> 6, sh = tt0 & 63;
          const uint64_t lo = q == 0 ? mw0 : q == 1 ? mw1 : q == 2 ? mw2 : q == 3 ? mw3 : 0ull;
          const uint64_t hi = q == 0 ? mw1 : q == 1 ? mw2 : q == 2 ? mw3 : 0ull;
          uint64_t tb = sh == 0 ? lo : (lo >> sh) | (hi << (64 - sh));
          const int ntree = p.m - tt0;          // tree positions left from tt0
          if (ntree < 64) tb &= ntree > 0 ? (1ull << ntree) - 1ull : 0ull;
          const uint64_t vis = pre > 0 ? (((1ull << pre) - 1ull) | (tb << pre)) : tb;
#pragma unroll
          for (int c = 0; c < BN; ++c) s[c] = ((vis >> c) & 1ull) ? s[c] : -INFINITY;
        }
        {  // eight independent running maxima, then a tree
          float m8[8];
#pragma unroll
          for (int c = 0; c < 8; ++c) m8[c] = s[c];
#pragma unroll
          for (int c = 8; c < BN; ++c) m8[c & 7] = fmaxf(m8[c & 7], s[c]);
          mx = fmaxf(fmaxf(fmaxf(m8[0], m8[1]), fmaxf(m8[2], m8[3])), fmaxf(fmaxf(m8[4], m8[5]), fmaxf(m8[6], m8[7])));
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
        const float mu = (m_ref == -INFINITY) ? 0.f : m_ref;
        uint32_t pk[32];
        float rs4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          const float p0 = valid ? ex2_approx(fmaf(s[2 * c], sl2, -mu)) : 0.f;
          const float p1 = valid ? ex2_approx(fmaf(s[2 * c + 1], sl2, -mu)) : 0.f;
          rs4[c & 3] += p0 + p1;
          pk[c] = pack_bf16x2(p0, p1);
        }
        l_sum += (rs4[0] + rs4[1]) + (rs4[2] + rs4[3]);
        tmem_st32(tP, pk);
        if (__any_sync(0xffffffffu, resc)) {
          // O must hold P V of tile t-1 before it is rescaled
          ok = mbar_wait_warp(o_ready(i), (t - 1) & 1, abort_flag, p.status);
          if (!ok) break;
          tc_fence_after();
#pragma unroll 1
          for (int cc = 0; cc < 4; ++cc) {
            uint32_t o[32];
            tmem_ld32(tO + 32u * cc, o);
#pragma unroll
            for (int j = 0; j < 32; ++j) o[j] = __float_as_uint(__uint_as_float(o[j]) * alpha);
            tmem_st32(tO + 32u * cc, o);
          }
        }
        tmem_st_wait();
        if (i == 0 && key0 + BN > nkeys) {
          // zero V rows past the end of the sequence (their P is 0, but the cache slots may
          // hold non-finite garbage and 0 * inf would poison O)
          const int s_ = t % ST;
          ok = mbar_wait_warp(full_v(s_), (t / ST) & 1, abort_flag, p.status);
          if (!ok) break;
          const int jv = nkeys - key0;
          const int nz = (BN - jv) * 16;
          for (int c = q4 * 32 + lane; c < nz; c += 128) {
            const int row = jv + (c >> 4), h = (c >> 3) & 1, j = c & 7;
            *reinterpret_cast<uint4*>(sptr + C::OFF_V + s_ * KTILE + h * KHALF + row * 128 + j * 16) =
                make_uint4(0u, 0u, 0u, 0u);
          }
          fence_proxy_async_smem();
        }
        tc_fence_before();
        mbar_arrive(p_full(i, sb));
      }
      if (ok) ok = mbar_wait_warp(o_final(i), 0, abort_flag, p.status);
      if (ok) {
        tc_fence_after();
        const int head = kvh * p.g + (valid ? grow % p.g : 0);
        if (direct) {
          const float inv = (valid && l_sum > 0.f) ? 1.f / l_sum : 0.f;
          __nv_bfloat16* dst = p.out + ((static_cast<long long>(b) * p.m + node) * p.Hq + head) * HD;
#pragma unroll 1
          for (int cc = 0; cc < 4; ++cc) {
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
          if (valid && p.lse != nullptr)
            p.lse[(static_cast<long long>(b) * p.m + node) * p.Hq + head] = (m_ref + log2f(l_sum)) * kLn2;
        } else if (p.mode == kGlobal) {
          const long long prow = (static_cast<long long>(bk) * p.rows + grow) * p.nchunk + chunk;
          float* dst = p.part_o + prow * HD;
#pragma unroll 1
          for (int cc = 0; cc < 4; ++cc) {
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
          if (valid) p.part_ml[prow] = make_float2(m_ref, l_sum);
        }
        // cluster mode: O stays in TMEM until every CTA of the cluster has left its loop
      }
    }
  }

  if (p.mode == kCluster) {
    // Merge through distributed shared memory.  Rows of the row group are split evenly over
    // the cs CTAs ("owners"); slot (c, row) of an owner's receive area holds CTA c's partial.
    // 1) barrier: every CTA has left its loop, so all K/V rings are idle and reusable;
    // 2) every CTA pushes its (max, sum) and fp32 O rows into the owners' rings with remote
    //    stores (no round trips); 3) barrier: all pushes are visible; 4) each owner merges
    //    its rows from local shared memory and writes the output.
    const int cs = p.nchunk;
    const int q = static_cast<int>(cluster_ctarank());
    const int per = NM * BM / cs;  // cs divides 128
    tc_fence_before();
    cluster_sync_all();
    if (warp >= 4 && warp < C::EXTRA_WARP) {
      const int i = (warp - 4) >> 2;
      const int Rl = i * BM + (warp & 3) * 32 + lane;
      const bool have = ok && i < nma && nt > 0 && R0 + Rl < p.rows;
      const int owner = Rl / per;
      const int slot = q * per + (Rl - owner * per);
      const float2 ml = have ? make_float2(m_ref, l_sum) : make_float2(-INFINITY, 0.f);
      st_dsmem_f2(dsmem_addr(sbase + C::OFF_ML + 8u * slot, owner), ml);
      if (__any_sync(0xffffffffu, have)) {  // tcgen05.ld is warp-wide
        tc_fence_after();
        const uint32_t tO = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16) + 128u * i;
#pragma unroll 1
        for (int cc = 0; cc < 4; ++cc) {
          uint32_t o[32];
          tmem_ld32(tO + 32u * cc, o);
          if (have) {
#pragma unroll
            for (int v4 = 0; v4 < 8; ++v4)
              st_dsmem_u4(dsmem_addr(sbase + C::OFF_K + orow_off(slot, cc * 8 + v4), owner),
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
      const int grow = R0 + Rl;
      if (grow >= p.rows) break;
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
  __syncthreads();
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
  if (min(T, nc) <= 1) return;  // written directly by the attention kernel
  const long long prow = static_cast<long long>(wid) * nc;
  // chunk c holds tiles [ceil(c*T/nc), ceil((c+1)*T/nc)); empty chunks wrote nothing
  auto empty = [&](int c) {
    return (static_cast<long long>(c + 1) * T + nc - 1) / nc == (static_cast<long long>(c) * T + nc - 1) / nc;
  };
  float M = -INFINITY;
#pragma unroll 4
  for (int c = 0; c < nc; ++c) {
    if (empty(c)) continue;
    const float2 ml = part_ml[prow + c];
    if (ml.y > 0.f) M = fmaxf(M, ml.x);
  }
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  float Ls = 0.f;
#pragma unroll 4
  for (int c = 0; c < nc; ++c) {
    if (empty(c)) continue;
    const float2 ml = part_ml[prow + c];
    if (!(ml.y > 0.f)) continue;
    const float w = exp2f(ml.x - M);
    Ls += w * ml.y;
    const float4 o = reinterpret_cast<const float4*>(part_o + (prow + c) * HD)[lane];
    acc.x += w * o.x;
    acc.y += w * o.y;
    acc.z += w * o.z;
    acc.w += w * o.w;
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

template <int NM>
static cudaError_t set_smem_attr() {
  static std::once_flag once;
  static cudaError_t err = cudaSuccess;
  std::call_once(once, [] {
    err = cudaFuncSetAttribute(tree_attn_tc_kernel<NM>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               Cfg<NM>::SMEM_BYTES);
  });
  return err;
}

// How many clusters of `cs` CTAs (one per SM) the device runs at once; 0 if unknown.
template <int NM>
static int active_clusters(int cs) {
  static std::mutex mu;
  static int cache[kMaxCluster + 1] = {};
  static bool done[kMaxCluster + 1] = {};
  std::lock_guard<std::mutex> lock(mu);
  if (done[cs]) return cache[cs];
  done[cs] = true;
  if (set_smem_attr<NM>() != cudaSuccess) return 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(1, cs, 1);
  cfg.blockDim = dim3(Cfg<NM>::THREADS, 1, 1);
  cfg.dynamicSmemBytes = Cfg<NM>::SMEM_BYTES;
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeClusterDimension;
  attr.val.clusterDim.x = 1;
  attr.val.clusterDim.y = cs;
  attr.val.clusterDim.z = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, tree_attn_tc_kernel<NM>, &cfg) != cudaSuccess) {
    cudaGetLastError();
    n = 0;
  }
  cache[cs] = n;
  return n;
}

struct Plan {
  int NM, rowgroups, nc, tpc, mode;
};

// Makespan model in 64-key-tile units: waves x (tiles per CTA + fixed cost per CTA) plus,
// for the global mode, the partial write/read and the combine launch.
static Plan make_plan(int B, int m, int Hq, int Hkv, int max_prefix, int num_sms) {
  Plan pl;
  if (num_sms < 1) num_sms = 1;
  const int rows = m * (Hq / Hkv);
  pl.NM = rows > BM ? 2 : 1;
  pl.rowgroups = (rows + pl.NM * BM - 1) / (pl.NM * BM);
  const int T = (max_prefix + m + BN - 1) / BN;
  const long long units = static_cast<long long>(B) * Hkv * pl.rowgroups;
  const int c0 = 3;
  const int rows_cta = rows < pl.NM * BM ? rows : pl.NM * BM;
  const int cglob = 4 + (rows_cta * 2 + BN - 1) / BN;
  long long best = -1;
  pl.nc = 1;
  pl.tpc = T;
  pl.mode = kDirect;
  const int max_nc = T < 4096 ? T : 4096;
  for (int nc = 1; nc <= max_nc; ++nc) {
    const int tpc = (T + nc - 1) / nc;
    if ((T + tpc - 1) / tpc != nc) continue;
    if (tpc * (BN / 16) > kMaxChunkBoxes) continue;  // box ids staged for the smallest pages
    const long long waves = (units * nc + num_sms - 1) / num_sms;
    const long long cost = waves * (tpc + c0) + (nc > 1 ? waves * cglob : 0);
    if (best < 0 || cost < best) {
      best = cost;
      pl.nc = nc;
      pl.tpc = tpc;
      pl.mode = nc > 1 ? kGlobal : kDirect;
    }
  }
  // Optional override for tests and tuning: TREESPEC_ATTN_SPLIT=direct | cluster:N | global:N
  // (ignored when the requested split is not feasible for these sizes).
  if (const char* ov = std::getenv("TREESPEC_ATTN_SPLIT")) {
    int n = 0;
    if (std::strcmp(ov, "direct") == 0) {
      if (T * (BN / 16) <= kMaxChunkBoxes) {
        pl.nc = 1;
        pl.tpc = T;
        pl.mode = kDirect;
        return pl;
      }
    } else if (std::sscanf(ov, "cluster:%d", &n) == 1 && (n == 2 || n == 4 || n == 8) && T >= n) {
      const int tpc = (T + n - 1) / n;
      const int act = pl.NM == 1 ? active_clusters<1>(n) : active_clusters<2>(n);
      if ((T + tpc - 1) / tpc == n && tpc * (BN / 16) <= kMaxChunkBoxes && act > 0) {
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
  for (int cs = 2; cs <= kMaxCluster; cs *= 2) {
    if (T < cs) break;
    const int tpc = (T + cs - 1) / cs;
    if ((T + tpc - 1) / tpc != cs) continue;
    if (tpc * (BN / 16) > kMaxChunkBoxes) continue;
    const int act = pl.NM == 1 ? active_clusters<1>(cs) : active_clusters<2>(cs);
    if (act <= 0) continue;
    const long long waves = (units + act - 1) / act;
    const long long cost = waves * (tpc + c0 + 1);
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

static bool encode_kv_map(CUtensorMap* map, const void* base, int num_blocks, int Hkv, int bs) {
  EncodeFn enc = get_encode();
  if (enc == nullptr) return false;
  const cuuint64_t dims[4] = {static_cast<cuuint64_t>(HD), static_cast<cuuint64_t>(bs),
                              static_cast<cuuint64_t>(Hkv), static_cast<cuuint64_t>(num_blocks)};
  const cuuint64_t strides[3] = {static_cast<cuuint64_t>(HD) * 2, static_cast<cuuint64_t>(bs) * HD * 2,
                                 static_cast<cuuint64_t>(Hkv) * bs * HD * 2};
  const cuuint32_t box[4] = {64u, static_cast<cuuint32_t>(bs < BN ? bs : BN), 1u, 1u};
  const cuuint32_t estr[4] = {1u, 1u, 1u, 1u};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Small cache of encoded K/V tensor maps keyed by (base pointer, shape): encoding is a
// host-side driver call, and serving loops reuse the same cache tensors every step.
struct MapEntry {
  const void* base;
  int num_blocks, Hkv, bs;
  CUtensorMap map;
  uint64_t stamp;
};

static bool cached_kv_map(CUtensorMap* out, const void* base, int num_blocks, int Hkv, int bs) {
  constexpr int kSlots = 16;
  static MapEntry cache[kSlots] = {};
  static uint64_t clock = 0;
  static std::mutex mu;
  std::lock_guard<std::mutex> lock(mu);
  ++clock;
  int victim = 0;
  for (int i = 0; i < kSlots; ++i) {
    MapEntry& e = cache[i];
    if (e.stamp != 0 && e.base == base && e.num_blocks == num_blocks && e.Hkv == Hkv && e.bs == bs) {
      e.stamp = clock;
      *out = e.map;
      return true;
    }
    if (e.stamp < cache[victim].stamp) victim = i;
  }
  MapEntry e{base, num_blocks, Hkv, bs, {}, clock};
  if (!encode_kv_map(&e.map, base, num_blocks, Hkv, bs)) return false;
  cache[victim] = e;
  *out = e.map;
  return true;
}

template <int NM>
static int launch_nm(const CUtensorMap& mk, const CUtensorMap& mv, const Params& prm, const Plan& pl,
                     int B, int Hkv, cudaStream_t stream) {
  if (set_smem_attr<NM>() != cudaSuccess) return TS_ERR_CUDA;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(pl.rowgroups, pl.nc, B * Hkv);
  cfg.blockDim = dim3(Cfg<NM>::THREADS, 1, 1);
  cfg.dynamicSmemBytes = Cfg<NM>::SMEM_BYTES;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (pl.mode == kCluster) {
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = 1;
    attr[1].val.clusterDim.y = pl.nc;
    attr[1].val.clusterDim.z = 1;
    cfg.numAttrs = 2;
  }
  return cudaLaunchKernelEx(&cfg, tree_attn_tc_kernel<NM>, mk, mv, prm) == cudaSuccess ? TS_OK : TS_ERR_CUDA;
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

void attention_tc_plan(int B, int m, int Hq, int Hkv, int max_prefix, int num_sms, int* out4) {
  const tc::Plan pl = tc::make_plan(B, m, Hq, Hkv, max_prefix, num_sms);
  out4[0] = pl.NM;
  out4[1] = pl.nc;
  out4[2] = pl.tpc;
  out4[3] = pl.mode;
}

int attention_tc_launch(const AttnArgs& a, int num_sms) {
  const tc::Plan pl = tc::make_plan(a.B, a.m, a.Hq, a.Hkv, a.max_prefix, num_sms);
  CUtensorMap mk, mv;
  if (!tc::cached_kv_map(&mk, a.k_cache, a.num_blocks, a.Hkv, a.block_size) ||
      !tc::cached_kv_map(&mv, a.v_cache, a.num_blocks, a.Hkv, a.block_size))
    return TS_ERR_CUDA;
  tc::Params prm;
  prm.q = static_cast<const __nv_bfloat16*>(a.q);
  prm.block_table = a.block_table;
  prm.prefix_len = a.prefix_len;
  prm.mask = a.mask;
  prm.out = static_cast<__nv_bfloat16*>(a.out);
  prm.lse = a.lse;
  prm.status = a.dev_status;
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
  prm.scale_log2 = a.scale * 1.4426950408889634f;
  const size_t prow = static_cast<size_t>(a.B) * a.Hkv * prm.rows * pl.nc;
  prm.part_o = pl.mode == tc::kGlobal ? static_cast<float*>(a.workspace) : nullptr;
  prm.part_ml = pl.mode == tc::kGlobal
                    ? reinterpret_cast<float2*>(static_cast<char*>(a.workspace) + prow * tc::HD * 4)
                    : nullptr;
  const int rc = pl.NM == 1 ? tc::launch_nm<1>(mk, mv, prm, pl, a.B, a.Hkv, a.stream)
                            : tc::launch_nm<2>(mk, mv, prm, pl, a.B, a.Hkv, a.stream);
  if (rc != TS_OK) return rc;
  int launches = 1;
  if (pl.mode == tc::kGlobal) {
    const int total_rows = a.B * a.Hkv * prm.rows;
    if (launch_pdl(tc::combine_kernel, dim3((total_rows + 7) / 8), dim3(256), 0, a.stream, prm.part_o,
                   prm.part_ml, a.prefix_len, prm, total_rows) != cudaSuccess)
      return TS_ERR_CUDA;
    ++launches;
  }
  count_launches(launches);
  return cudaGetLastError() == cudaSuccess ? TS_OK : TS_ERR_CUDA;
}

}  // namespace ts
