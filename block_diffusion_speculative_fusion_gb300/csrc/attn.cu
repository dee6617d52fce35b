// Draft block attention: softmax(scale * Q K^T) V, GQA, where the keys/values
// of sequence b are its ctx_len[b] context rows in the paged pools followed by
// the block's own rows; no mask, or the in-block causal mask.
//   DFlash page, section 块扩散 (bidirectional attention inside the block),
//   KV 注入 step 3 (Attention(Q_draft, [K_draft; K_ctx], [V_draft; V_ctx])) and
//   块扩散的双向注意力问题 (the causal variant: block position i sees 0 .. i).
//
// bf16 / D = 128 path (the serving shapes): a persistent, warp-specialised
// tcgen05 kernel (below). The n_q * (Hq/Hkv) query rows that share a kv head
// are packed into the MMA's M dimension (GQA packing), so each K/V byte is read
// from HBM once per kv head. Context pages arrive by TMA into a ring of 64-row
// stages; Q, S, P and O live in TMEM; the online softmax runs in fp32. A
// context split over several CTAs leaves fp32 partials that a small second
// kernel merges; it is launched as a programmatic dependent of the first, so
// its launch overlaps the first kernel's tail.
//
// Generic path (fp32, or shapes outside the bf16 kernel): one CTA per query
// row with fp32 CUDA-core arithmetic; used for the tiny fp32 configuration.
#include <algorithm>

#include "common.cuh"
#include "internal.h"
#include "tc.cuh"
#include "tma.cuh"

namespace dflash {

namespace attn {
constexpr int kD = 128;
constexpr int kTileK = 64;                   // keys per tile
constexpr int kMinSplitTiles = 8;            // smallest range of the partition, in tiles
constexpr int kMaxWarps = 8;                 // M <= 128 packed query rows
}  // namespace attn

struct AttnParams {
  const bf16* q;
  const bf16* k_blk;
  const bf16* v_blk;
  const int32_t* page_table;
  const int32_t* ctx_len;
  const uint8_t* active;   // [B] or null: sequences with 0 take no tiles
  bf16* out;
  float* part_o;     // [n_slots][Mi][128]: fp32 partial O of the split pieces
  float2* part_ml;   // [n_slots][Mi]: their row max (log2 units) and sum
  int32_t* plan_ws;  // [B + 2]: the partition's range size, then cum[0..B] (read by the merge kernel)
  int* err;
  int B, n_q, n_kv, Hq, Hkv, G, M, page_size, max_pages, num_pages, n_slots, max_ctx;
  int causal;        // 1: query i sees block rows j <= i + n_kv - n_q
  // work items: hpi kv heads (1 or 2) per item, Gi = hpi * G query heads and
  // Mi = n_q * Gi packed rows per item, n_groups = Hkv / hpi items per split of
  // a sequence, TK = 64 / hpi keys per tile, br = K/V rows per TMA box
  int hpi, Gi, Mi, n_groups, TK, br;
  float scale_log2;  // softmax scale * log2(e)
  unsigned long long wait_ns;   // limit of every bounded wait on a work barrier
};

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// Byte offset of 16-byte chunk `c` (0..7) of row `r` in a [rows][64] bf16 half
// tile with the 128-byte TMA swizzle (chunk index XOR row mod 8).
__device__ __forceinline__ uint32_t swz(int r, int c) { return (uint32_t)(r * 128 + ((c ^ (r & 7)) << 4)); }

// ===========================================================================
// tcgen05 path: persistent, warp-specialised, TMEM accumulators.
//   softmax     warps q and q + 4 for q < W = ceil(M / 32): TMEM lane quarter q
//               (packed query row 32 q + lane), key columns 0-31 / 32-63
//   producer    warp 2 (W <= 2) or 12: walks the CTA's pieces of the static
//               partition, fetches their page rows, streams context K/V pages
//               by TMA into a ring of 64-row stages
//   MMA         the warp after the producer: TMEM allocator, one issuing thread
//   epilogue    warps 8 + q: write the next item's Q rows into TMEM, read O out
//               of TMEM, normalise, store
// A work item (piece) is a run of tiles of one (sequence, kv-head group),
// from a static partition that gives every CTA the same number of tiles
// (see AttnItem). Per 64-row tile t: S_t = Q K_t^T (M = 128,
// N = 64, Q from TMEM) into TMEM buffer t % 2; the softmax threads read their
// S row and write P_t (bf16 pairs) back into TMEM, and the MMA thread
// accumulates O += P_t V_t (M = 128, N = 128, P from TMEM, V read MN-major)
// into the item's TMEM O buffer. The running max is only raised (O rescaled
// in TMEM) when a tile's max exceeds it
// by more than 2^8, so rescaling is rare. The K/V ring runs across item
// boundaries. The MMA thread issues P_{t-1} V_{t-1} as soon as P_{t-1} is
// ready, also while it still waits for tile t to land, so that a stage goes
// back to the producer without waiting for the next tile; a new item's S MMAs
// start while the epilogue still reads the previous item's O, and only its
// first P V waits for the O buffer.
// ===========================================================================
namespace attn_tc {
constexpr int kTileK = 64;
constexpr int kMaxStages = 6;
constexpr int kTileBytes = 2 * 64 * 128;   // K (or V) of one tile: two d-halves x 64 keys x 128 B
constexpr int kTmemCols = 512;   // S0 [0,64), S1 [64,128), O0 [128,256), O1 [256,384), P0/P1 [384,448), Q [448,512)
constexpr uint32_t kPCol = 384;      // P_t (bf16 pairs) at kPCol + 32 (t % 2)
constexpr uint32_t kQCol = 448;      // Q of the current item (bf16 pairs, A operand of S = Q K^T)
constexpr float kRescaleLog2 = 8.f;
constexpr int kGrid = 152;                  // persistent CTAs: one per SM
constexpr int kMaxSeqs = 1024;              // sequences per call on this path
constexpr int kPtMax = 512;                 // page-table entries of one item
constexpr int kClaimAhead = 3;              // tiles before a piece's end at which the next one's pages are fetched
constexpr int kBarBytes = (2 * kMaxStages + 33) * 8 + 2 * 32 + (kMaxSeqs + 1) * 4 + 2 * kPtMax * 4 +
                          (2 * 2 * 128 + 2 * 4 * 128) * 4 + 64;
}  // namespace attn_tc

// Work is a static, balanced partition of the launch's tiles. Every (sequence
// b, kv-head group g) owns nt_b consecutive tiles -- its context tiles, then
// the block's own rows as one more tile -- in the order b-major, g-minor; the
// resulting sequence of N tiles is cut into ranges of `share` tiles (the mean
// work of one CTA, at least 8 tiles, at most what one page-table window
// holds), and CTA c takes ranges c, c + grid, ... A piece is the part of one
// range that falls in one (b, g); a (b, g) cut by range borders is computed
// in pieces whose fp32 partial results a second kernel (attn_merge_kernel)
// merges once the grid has finished. Partials sit in two slots per range: 2 v
// for the piece that starts range v, 2 v + 1 for a piece that starts inside it
// (only a (b, g)'s first piece can).

struct AttnItem {
  int b, g, split, nsplit, t0, C, n_tiles_ctx, n_tiles;   // b < 0: no more pieces
};

__device__ __forceinline__ int ctx_tiles(const AttnParams& p, int b) {
  const int C = max(0, min(p.ctx_len[b], p.max_ctx));
  return (C + p.TK - 1) / p.TK;
}

__device__ __forceinline__ int group_tiles(const AttnParams& p, int b) {
  if (p.active && !p.active[b]) return 0;   // an inactive sequence takes no tiles
  return ctx_tiles(p, b) + (p.n_kv > 0 ? 1 : 0);
}

struct AttnPlan {
  int N, share, R;   // tiles of the launch, tiles per range, ranges
};

// cum[b] (b = 0..B) = tiles per group of the sequences before b; whole warp.
__device__ __forceinline__ void plan_cum_warp(const AttnParams& p, int* cum, int lane) {
  const int per = (p.B + 31) / 32;
  const int r0 = lane * per, r1 = min(p.B, r0 + per);
  int tot = 0;
  for (int b = r0; b < r1; ++b) tot += group_tiles(p, b);
  int incl = tot;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  int run = incl - tot;
  for (int b = r0; b < r1; ++b) {
    cum[b] = run;
    run += group_tiles(p, b);
  }
  if (lane == 31) cum[p.B] = incl;
#ifdef DFLASH_DEBUG
  // context lengths outside [0, max_ctx] are clamped; debug builds record them
  if (blockIdx.x == 0)
    for (int b = r0; b < r1; ++b)
      if (p.ctx_len[b] < 0 || p.ctx_len[b] > p.max_ctx) record_dev_error(p.err, kDevErrBadCtxLen);
#endif
}

__device__ __forceinline__ AttnPlan make_plan(const AttnParams& p, const int* cum) {
  AttnPlan q;
  q.N = p.n_groups * cum[p.B];
  // one page more than a piece spans, for pieces that start inside a page
  const int window = (attn_tc::kPtMax - 1) * p.page_size / p.TK;
  q.share = min(window, max(attn::kMinSplitTiles, (q.N + attn_tc::kGrid - 1) / attn_tc::kGrid));
  q.R = (q.N + q.share - 1) / q.share;
  return q;
}

// The next piece of this CTA: `v` is the current range, `pos` the next tile of
// the launch sequence to hand out. Returns false when the CTA has no more work.
__device__ __forceinline__ bool next_piece(const AttnParams& p, const int* cum, const AttnPlan& q, int& v, int& pos,
                                           AttnItem& it) {
  while (v < q.R) {
    const int e = min(q.N, (v + 1) * q.share);
    if (pos < e) {
      int lo = 0, hi = p.B - 1;
      while (lo < hi) {      // last sequence whose tiles start at or before pos
        const int mid = (lo + hi + 1) >> 1;
        if (p.n_groups * cum[mid] <= pos) lo = mid; else hi = mid - 1;
      }
      const int b = lo, nt = cum[b + 1] - cum[b];
      const int gb = p.n_groups * cum[b];
      const int g = (pos - gb) / nt;
      const int base = gb + g * nt;
      const int t0 = pos - base, t1 = min(nt, e - base);
      it.b = b;
      it.g = g;
      it.C = max(0, min(p.ctx_len[b], p.max_ctx));
      it.t0 = t0;
      it.n_tiles = t1 - t0;
      it.n_tiles_ctx = max(0, min(t1, ctx_tiles(p, b)) - t0);
      it.split = v - base / q.share;
      it.nsplit = (base + nt - 1) / q.share - base / q.share + 1;
      pos = base + t1;
      return true;
    }
    v += attn_tc::kGrid;
    pos = v * q.share;
  }
  return false;
}

// 2^x on the special-function unit (flush-to-zero; P is rounded to bf16 anyway).
__device__ __forceinline__ float ex2_ftz(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

template <int kThreadsT, int HPI>
__global__ void __launch_bounds__(kThreadsT, 1)
attn_tc_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
               const __grid_constant__ CUtensorMap kbmap, const __grid_constant__ CUtensorMap vbmap,
               const AttnParams p, int S) {
  using namespace attn_tc;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // Roles, with W = ceil(Mi / 32) TMEM lane quarters holding real rows:
  //   softmax   warps q and q + 4 for q < W (half h = 0, 1 of the pair)
  //   epilogue  warps 8 + q for q < W (O read-out of finished items)
  //   producer  warp 2 (W <= 2) or 12; MMA issuer the warp after it
  // One head per item: half h takes keys 32h .. 32h + 31 of every tile (SPL = 2
  // column halves; the row max is exchanged). Two heads per item: half h takes
  // every other tile of an item whole (ALT = 2 tile groups) and accumulates
  // into its own TMEM O; the epilogue merges the two.
  constexpr int TK = kTileK / HPI;          // keys per tile (of each of the HPI heads)
  constexpr int SPL = HPI == 1 ? 2 : 1;     // softmax warps sharing one tile's row
  constexpr int ALT = HPI == 1 ? 1 : 2;     // softmax warp groups taking alternate tiles
  constexpr int NK = TK / SPL;              // keys of a tile per softmax thread
  constexpr int NCOL = NK * HPI;            // S columns per softmax thread (both heads)
  const int W = (p.Mi + 31) / 32;
  const int n_sm = 2 * W;                   // softmax warps
  const int n_tile_sm = n_sm / ALT;         // softmax warps that consume one tile
  const int prod_warp = W <= 2 ? 2 : 12, mma_warp = prod_warp + 1;
  const int quarter = warp & 3, chalf = (warp >> 2) & 1;
  const bool is_softmax = warp < 8 && quarter < W && warp != prod_warp && warp != mma_warp;
  const bool is_epi = warp >= 8 && warp < 12 && quarter < W;

  // shared memory: [S stages: K | V][barriers, tables]. Q lives in TMEM (columns
  // kQCol..kQCol+63, the S MMA's A operand): the epilogue warps write the next
  // item's Q rows there once the current item's last S has read them.
  // A 128-row MMA reads all 128 lanes; lanes past the item's rows only produce
  // padding rows of S, P and O, which are never used.
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* kv_s = smem;                      // stage s: K at s*2*T, V at s*2*T + T
  uint64_t* bars = reinterpret_cast<uint64_t*>(kv_s + S * 2 * kTileBytes);
  constexpr int KS = kMaxStages;
  uint64_t* kv_full = bars;               // [KS]
  uint64_t* kv_empty = bars + KS;         // [KS]
  uint64_t* s_full = bars + 2 * KS;       // [2]
  uint64_t* s_empty = s_full + 2;         // [2]
  uint64_t* p_full = s_full + 4;          // [2]
  uint64_t* pv_done = s_full + 6;         // [2]
  uint64_t* q_full = s_full + 8;          // [2]  epilogue warps -> MMA: Q of the item in TMEM
  uint64_t* q_empty = s_full + 10;        // [2]  MMA -> epilogue warps: the item's last S has read Q
  uint64_t* it_full = s_full + 12;        // [2]
  uint64_t* it_empty = s_full + 14;       // [2]
  uint64_t* o_full = s_full + 16;         // [2]  MMA -> epilogue: last P V of the item done
  uint64_t* o_empty = s_full + 18;        // [2]  epilogue -> MMA: O buffer read out
  uint64_t* mma_done = s_full + 20;
  uint64_t* xbar = s_full + 21;           // [4 quarters][2]: the two softmax warps of a quarter
  uint64_t* l_full = s_full + 29;         // [2]  softmax -> epilogue: row max and sums of the item
  // (s_full + 31, + 32: spare)
  AttnItem* ring = reinterpret_cast<AttnItem*>(s_full + 33);  // [2] pieces in flight (b < 0: none left)
  int* cum = reinterpret_cast<int*>(ring + 2);                // [B + 1] tiles per group before sequence b
  int* pt_s = cum + (kMaxSeqs + 1);                           // [2][kPtMax] page rows of two pieces
  float* xch = reinterpret_cast<float*>(pt_s + 2 * kPtMax);    // [2 tiles][2 halves][128] tile maxima
  float* ml_s = xch + 2 * 2 * 128;     // [2 slots][4][128]: (m, l) of softmax half 0, then of half 1
  uint32_t* tmem_base_sm = reinterpret_cast<uint32_t*>(ml_s + 2 * 4 * 128);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_base_sm + 1);
  int* consumed_sm = reinterpret_cast<int*>(tmem_base_sm + 2);

  if (tid == 0) {
    for (int i = 0; i < kMaxStages; ++i) {
      mbar_init(&kv_full[i], 1);
      mbar_init(&kv_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s_full[i], 1);
      mbar_init(&s_empty[i], n_tile_sm);
      mbar_init(&p_full[i], n_tile_sm);
      mbar_init(&pv_done[i], 1);
      mbar_init(&q_full[i], W);
      mbar_init(&q_empty[i], 1);
      mbar_init(&it_full[i], 1);
      mbar_init(&it_empty[i], 1 + n_sm + W);
      mbar_init(&o_full[i], 1);
      mbar_init(&o_empty[i], W);
      mbar_init(&l_full[i], n_sm);
    }
    mbar_init(mma_done, 1);
    for (int i = 0; i < 8; ++i) mbar_init(&xbar[i], 2);
    *abort_flag = 0;
    *consumed_sm = 0;
    fence_barrier_init();
  }
  if (warp == mma_warp) tmem_alloc(tmem_base_sm, kTmemCols);
  // the merge kernel that follows may be scheduled once every CTA has got here;
  // it waits for this grid to complete before it reads anything
  dependents_may_launch();
  // ---- work list: the tiles per group of every sequence, prefix-summed ----
  if (warp == 0) plan_cum_warp(p, cum, lane);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_base_sm;
  const AttnPlan plan = make_plan(p, cum);
  if (blockIdx.x == 0 && warp == 0) {
    for (int b = lane; b <= p.B; b += 32) p.plan_ws[1 + b] = cum[b];
    if (lane == 0) p.plan_ws[0] = plan.share;
  }
  int producer_issued = 0;

  if (warp == prod_warp) {
    // ------------------------------ producer ------------------------------
    // The next item's page rows are fetched while the current item's last tiles
    // stream, so that item boundaries leave no gap in the K/V stream.
    const int ps = p.page_size;
    const uint64_t pol_kv = l2_policy_evict_first();   // every page row is read once
    int item_seq = 0, tile_seq = 0;
    bool ok = true;
    // page rows of item `item` into table `tb` (whole warp). Every lane issues
    // its loads together before storing any, so the fetch costs one memory
    // latency instead of one per round.
    auto load_pages = [&](const AttnItem& it, int tb) {
      const int lp0 = it.t0 * TK / ps;
      const int n_lp = ((it.t0 + it.n_tiles_ctx) * TK + ps - 1) / ps - lp0;
      const int32_t* ptb = p.page_table + (size_t)it.b * p.max_pages;
      constexpr int kPer = kPtMax / 32;
      int phys[kPer];
#pragma unroll
      for (int u = 0; u < kPer; ++u) {
        const int lp = lp0 + u * 32 + lane;
        // pages past the context (or bad entries) read page 0; masked later
        const bool use = u * 32 + lane < n_lp && lp * ps < it.C && lp < p.max_pages;
        phys[u] = use ? __ldg(ptb + lp) : 0;
      }
      bool bad = false;
#pragma unroll
      for (int u = 0; u < kPer; ++u) {
        // an entry outside [0, num_pages) for a position inside the context is
        // an input error: record it and read page 0 instead (never out of bounds)
        const bool in_range = phys[u] >= 0 && phys[u] < p.num_pages;
        const int ph = in_range ? phys[u] : 0;
        bad |= !in_range;
        if (u * 32 + lane < n_lp) pt_s[tb * kPtMax + u * 32 + lane] = ph * ps;
      }
      if (__any_sync(0xffffffffu, bad) && lane == 0) atomicCAS(p.err, 0, kDevErrBadPage);
      __syncwarp();
    };
    // this CTA's ranges: blockIdx.x, blockIdx.x + grid, ...
    int rv = (int)blockIdx.x, rpos = (int)blockIdx.x * plan.share;
    AttnItem cur;
    bool have = next_piece(p, cum, plan, rv, rpos, cur);
    if (have) load_pages(cur, 0);
    while (ok) {
      const int slot = item_seq & 1;
      bool w = true;
      if (lane == 0) w = wait_or_abort(&it_empty[slot], (uint32_t)(((item_seq >> 1) & 1) ^ 1), abort_flag, p.err, 21, p.wait_ns);
      if (!__shfl_sync(0xffffffffu, w ? 1 : 0, 0)) break;
      if (lane == 0) {
        AttnItem pub = cur;
        if (!have) pub.b = -1;
        ring[slot] = pub;
        mbar_arrive(&it_full[slot]);    // release semantics publish the ring entry
      }
      if (!have) break;
      const AttnItem it = cur;
      const int* pt = pt_s + slot * kPtMax;
      // the next piece's page rows are fetched a few tiles before this one ends
      AttnItem nxt;
      bool have_n = false;
      const int j_claim = max(0, it.n_tiles - kClaimAhead);
      for (int j = 0; j < it.n_tiles && ok; ++j, ++tile_seq) {
        if (lane == 0) {
          const int st = tile_seq % S;
          uint8_t* ks = kv_s + st * 2 * kTileBytes;
          uint8_t* vs = ks + kTileBytes;
          if (!wait_or_abort(&kv_empty[st], (uint32_t)(((tile_seq / S) & 1) ^ 1), abort_flag, p.err, 23, p.wait_ns)) {
            ok = false;
          } else if (j < it.n_tiles_ctx) {
            mbar_arrive_expect_tx(&kv_full[st], 2 * kTileBytes);
            // box jb: br keys of each of the HPI heads, landing [key][head][64 d] per
            // d-half, so that tile row n holds key n / HPI of head n % HPI
            const int br = p.br;
            const int lp0 = it.t0 * TK / ps;
            for (int jb = 0; jb < TK / br; ++jb) {
              const int key0 = (it.t0 + j) * TK + jb * br;
              const int row = pt[key0 / ps - lp0] + key0 % ps;
              const int off = jb * HPI * br * 128;
              for (int h = 0; h < 2; ++h) {
                tma_load_3d_hint(ks + h * (kTileBytes / 2) + off, &kmap, &kv_full[st], h * 64, it.g * HPI, row, pol_kv);
                tma_load_3d_hint(vs + h * (kTileBytes / 2) + off, &vmap, &kv_full[st], h * 64, it.g * HPI, row, pol_kv);
              }
            }
            ++producer_issued;
          } else {
            // the block's own n_kv K/V rows of the HPI heads; rows past n_kv are
            // masked (K) and zeroed (V) by the softmax warps
            mbar_arrive_expect_tx(&kv_full[st], (uint32_t)(4 * HPI * p.n_kv * 128));
            for (int h = 0; h < 2; ++h) {
              tma_load_3d(ks + h * (kTileBytes / 2), &kbmap, &kv_full[st], h * 64, it.g * HPI, it.b * p.n_kv);
              tma_load_3d(vs + h * (kTileBytes / 2), &vbmap, &kv_full[st], h * 64, it.g * HPI, it.b * p.n_kv);
            }
            ++producer_issued;
          }
        }
        ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
        if (ok && j == j_claim) {
          have_n = next_piece(p, cum, plan, rv, rpos, nxt);
          if (have_n) load_pages(nxt, slot ^ 1);
        }
      }
      cur = nxt;
      have = have_n;
      ++item_seq;
    }
    __syncwarp();
  } else if (warp == mma_warp) {
    // ------------------------------ MMA issuer ------------------------------
    if (lane == 0) {
      const uint32_t id_s = idesc_bf16_ab(128, kTileK, 0);
      const uint32_t id_pv = idesc_bf16_ab(128, attn::kD, 1);
      int consumed = 0, item_seq = 0, tile_seq = 0;
      bool ok = true;
      while (ok) {
        const int slot = item_seq & 1;
        const uint32_t par = (uint32_t)((item_seq >> 1) & 1);
        if (!wait_or_abort(&it_full[slot], par, abort_flag, p.err, 24, p.wait_ns)) break;
        const AttnItem it = ring[slot];
        mbar_arrive(&it_empty[slot]);
        if (it.b < 0) break;
        // O: one buffer per item slot (ALT = 1), or both buffers for every item (ALT = 2)
        const int oi = ALT == 2 ? 0 : slot;
        const uint32_t opar = ALT == 2 ? (uint32_t)(item_seq & 1) : par;
        if (!wait_or_abort(&q_full[0], (uint32_t)(item_seq & 1), abort_flag, p.err, 25, p.wait_ns)) break;
        tc_fence_after();
        // The item's S MMAs go ahead while the epilogue still reads the previous
        // item's O; only its first P V waits for the O buffer (o_ready).
        bool o_ready = false;
        // O += P_t V_t once P_t is in TMEM; then stage t % S is free again
        auto pv_issue = [&](int t, int j) {
          tc_fence_after();
          // P_t from TMEM (8 packed columns per 16-row K step), V_t MN-major from smem
          const uint32_t pa = tmem_base + kPCol + (uint32_t)((t & 1) * 32);
          const uint32_t va = smem_u32(kv_s + (t % S) * 2 * kTileBytes + kTileBytes);
          const uint32_t o_tmem = tmem_base + 128 + (uint32_t)((ALT == 2 ? (t & 1) : slot) * attn::kD);
#pragma unroll
          for (int i = 0; i < kTileK / 16; ++i)
            tc_mma_bf16_ta(o_tmem, pa + (uint32_t)(i * 8), sdesc_sw128_mn(va + i * 2048, kTileBytes / 2), id_pv,
                           (j >= ALT || i > 0) ? 1u : 0u);
          tc_commit(&pv_done[t & 1]);
          tc_commit(&kv_empty[t % S]);
          ++consumed;
        };
        auto issue_pv = [&](int t, int j) -> bool {
          if (!o_ready) {
            if (!wait_or_abort(&o_empty[oi], opar ^ 1u, abort_flag, p.err, 26, p.wait_ns)) return false;
            o_ready = true;
          }
          if (!wait_or_abort(&p_full[t & 1], (uint32_t)((t >> 1) & 1), abort_flag, p.err, 27, p.wait_ns)) return false;
          pv_issue(t, j);
          return true;
        };
        // Wait for K/V tile t; while it is in flight, issue the P V of tile t - 1
        // as soon as its P is ready, so that stage (t - 1) % S goes back to the
        // producer without waiting for tile t to land.
        auto wait_tile = [&](int t, int j, bool& pv_pending) -> bool {
          uint64_t* full = &kv_full[t % S];
          const uint32_t par = (uint32_t)((t / S) & 1);
          if (mbar_try_wait(full, par)) return true;
          const uint64_t t_start = global_timer_ns();
          while (true) {
            for (int i = 0; i < 32; ++i) {
              if (mbar_try_wait(full, par)) return true;
              if (pv_pending) {
                if (!o_ready) o_ready = mbar_try_wait(&o_empty[oi], opar ^ 1u);
                if (o_ready && mbar_try_wait(&p_full[(t - 1) & 1], (uint32_t)(((t - 1) >> 1) & 1))) {
                  pv_issue(t - 1, j - 1);
                  pv_pending = false;
                }
              }
            }
            if (*abort_flag) return false;
            if (global_timer_ns() - t_start > p.wait_ns) {
              *abort_flag = 1;
              atomicCAS(p.err, 0, 28);
              return false;
            }
          }
        };
        for (int j = 0; j < it.n_tiles && ok; ++j) {
          const int t = tile_seq + j;
          const int st = t % S;
          bool pv_pending = j >= 1;   // the P V of tile t - 1 is still to issue
          if (!wait_tile(t, j, pv_pending)) { ok = false; break; }
          if (!wait_or_abort(&s_empty[t & 1], (uint32_t)(((t >> 1) & 1) ^ 1), abort_flag, p.err, 29, p.wait_ns)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t ka = smem_u32(kv_s + st * 2 * kTileBytes);
#pragma unroll
          for (int i = 0; i < attn::kD / 16; ++i) {
            const uint32_t off = (uint32_t)((i >> 2) * (kTileBytes / 2) + (i & 3) * 32);
            // Q from TMEM: 8 packed columns per 16-wide K step
            tc_mma_bf16_ta(tmem_base + (uint32_t)((t & 1) * kTileK), tmem_base + kQCol + (uint32_t)(i * 8),
                           sdesc_sw128(ka + off),
                        id_s, i > 0 ? 1u : 0u);
          }
          tc_commit(&s_full[t & 1]);
          if (j == it.n_tiles - 1) tc_commit(&q_empty[0]);   // Q is no longer read
          if (pv_pending) ok = issue_pv(t - 1, j - 1);
        }
        if (!ok) break;
        if (!issue_pv(tile_seq + it.n_tiles - 1, it.n_tiles - 1)) break;
        tc_commit(&o_full[oi]);
        tile_seq += it.n_tiles;
        ++item_seq;
      }
      *consumed_sm = consumed;
      tc_commit(mma_done);
      mbar_wait_bounded(mma_done, 0, p.err, 30);
    }
    __syncwarp();
  } else if (is_softmax) {
    // ------------------------------ softmax ------------------------------
    const int r = quarter * 32 + lane;              // packed query row = TMEM lane
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    // this warp's NK keys of a tile: keys kk0 .. kk0 + NK - 1 of the row's own
    // kv head hr; key kk of head h sits in S column (and V row) kk * HPI + h, so
    // the warp's columns are c0 .. c0 + 31 for both heads together
    const int hr = HPI == 1 ? 0 : (r % p.Gi) / p.G;
    const int kk0 = ALT == 2 ? 0 : chalf * NK;
    const int c0 = ALT == 2 ? 0 : chalf * NCOL;
    constexpr int OCOLS = attn::kD / SPL;           // O columns this thread rescales
    const uint32_t oc0 = (uint32_t)(ALT == 2 ? 0 : chalf * OCOLS);
    int item_seq = 0, tile_seq = 0;
    bool ok = true;
    int xs = 0;   // exchanges with the partner warp so far (both warps make the same sequence)
    // publish this warp's shared-memory values to its partner and wait for the partner's
    auto pair_exchange = [&]() -> bool {
      uint64_t* bar = &xbar[quarter * 2 + (xs & 1)];
      const uint32_t par = (uint32_t)((xs >> 1) & 1);
      ++xs;
      __syncwarp();
      if (lane == 0) mbar_arrive(bar);
      return __all_sync(0xffffffffu, wait_or_abort(bar, par, abort_flag, p.err, 37, p.wait_ns));
    };
    while (ok) {
      const int slot = item_seq & 1;
      const uint32_t par = (uint32_t)((item_seq >> 1) & 1);
      if (!__all_sync(0xffffffffu, wait_or_abort(&it_full[slot], par, abort_flag, p.err, 31, p.wait_ns))) break;
      const AttnItem it = ring[slot];
      __syncwarp();
      if (lane == 0) mbar_arrive(&it_empty[slot]);
      if (it.b < 0) break;
      const int t0 = it.t0;
      const uint32_t o_col = 128 + (uint32_t)((ALT == 2 ? chalf : slot) * attn::kD) + oc0;
      float m_run = -CUDART_INF_F, l_part = 0.f;
      // ALT = 2: this half takes the item's tiles t with t % 2 == half
      for (int j = ALT == 2 ? ((chalf - tile_seq) & 1) : 0; j < it.n_tiles; j += ALT) {
        const int t = tile_seq + j;
        const int sb = t & 1;
        if (!__all_sync(0xffffffffu, wait_or_abort(&s_full[sb], (uint32_t)((t >> 1) & 1), abort_flag, p.err, 32, p.wait_ns))) {
          ok = false;
          break;
        }
        tc_fence_after();
        float sv[NK];
        {
          // a TMEM load takes one column address for the whole warp, whose lanes
          // may hold rows of both heads: load both heads' columns and select
          uint32_t raw[NCOL];
#pragma unroll
          for (int c = 0; c < NCOL; c += 32) tmem_ld32(tmem_base + lane_off + (uint32_t)(sb * kTileK + c0 + c), raw + c);
          tmem_ld_wait();
#pragma unroll
          for (int c = 0; c < NK; ++c)
            sv[c] = __uint_as_float(HPI == 1 ? raw[c] : (hr ? raw[HPI * c + 1] : raw[HPI * c]));
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&s_empty[sb]);
        // keys 0 .. valid - 1 of the tile are real (per head); scores stay
        // unscaled here (the scale is > 0, so the max commutes with it)
        const int valid = (j < it.n_tiles_ctx) ? min(TK, it.C - (t0 + j) * TK) : p.n_kv;
        // keys this row sees: causal rows (packed row r is query r / Gi) stop
        // at their own block position
        const int seen = (p.causal && j >= it.n_tiles_ctx) ? min(valid, r / p.Gi + 1 + p.n_kv - p.n_q) : valid;
        float mx[4] = {-CUDART_INF_F, -CUDART_INF_F, -CUDART_INF_F, -CUDART_INF_F};
        if (seen < TK) {
#pragma unroll
          for (int c = 0; c < NK; ++c)
            if (kk0 + c >= seen) sv[c] = -CUDART_INF_F;
        }
#pragma unroll
        for (int c = 0; c < NK; ++c) mx[c & 3] = fmaxf(mx[c & 3], sv[c]);
        float mt = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])) * p.scale_log2;
        if constexpr (SPL == 2) {
          // tile max of the row over both column halves
          float* xb = xch + (t & 1) * 256;
          xb[chalf * 128 + r] = mt;
          if (!pair_exchange()) {
            ok = false;
            break;
          }
          mt = fmaxf(xb[r], xb[128 + r]);
        }
        const bool raise = mt > m_run + kRescaleLog2 || (m_run == -CUDART_INF_F && mt != -CUDART_INF_F);
        const float m_new = raise ? mt : m_run;
        const float alpha = raise ? (m_run == -CUDART_INF_F ? 0.f : exp2f(m_run - m_new)) : 1.f;
        if (j >= ALT && __any_sync(0xffffffffu, raise)) {
          // O must hold every earlier tile of the item before it is rescaled
          // (the last one into this O is tile t - ALT)
          if (!__all_sync(0xffffffffu, wait_or_abort(&pv_done[(t - ALT) & 1], (uint32_t)(((t - ALT) >> 1) & 1),
                                                     abort_flag, p.err, 33, p.wait_ns))) {
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll
          for (int c = 0; c < OCOLS / 32; ++c) {
            uint32_t o[32];
            tmem_ld32(tmem_base + lane_off + o_col + c * 32, o);
            tmem_ld_wait();
#pragma unroll
            for (int q = 0; q < 32; ++q) o[q] = __float_as_uint(__uint_as_float(o[q]) * alpha);
            tmem_st32(tmem_base + lane_off + o_col + c * 32, o);
          }
          tmem_st_wait();
        }
        m_run = m_new;
        const float base = (m_run == -CUDART_INF_F) ? 0.f : m_run;
        float rs[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int c = 0; c < NK; ++c) {
          sv[c] = ex2_ftz(fmaf(sv[c], p.scale_log2, -base));
          rs[c & 3] += sv[c];
        }
        l_part = l_part * alpha + ((rs[0] + rs[1]) + (rs[2] + rs[3]));
        // P buffer t & 1 was last read by the P V of tile t - 2
        if (t >= 2 && !__all_sync(0xffffffffu, wait_or_abort(&pv_done[sb], (uint32_t)(((t - 2) >> 1) & 1),
                                                           abort_flag, p.err, 34, p.wait_ns))) {
          ok = false;
          break;
        }
        // P_t (bf16) into its TMEM buffer: K entry n of the row (the S column /
        // V row n) in packed column n / 2; this thread's NCOL entries start at
        // c0, with 0 in the entries of the other head
        {
          const uint32_t pcol = tmem_base + lane_off + kPCol + (uint32_t)(sb * 32 + c0 / 2);
          if constexpr (HPI == 1) {
            uint32_t pk[NCOL / 2];
#pragma unroll
            for (int i = 0; i < NCOL / 2; ++i) pk[i] = pack_bf16(sv[2 * i], sv[2 * i + 1]);
            tmem_st16(pcol, pk);
          } else {
            uint32_t pk[NCOL / 2];
#pragma unroll
            for (int i = 0; i < NCOL / 2; ++i) pk[i] = hr ? pack_bf16(0.f, sv[i]) : pack_bf16(sv[i], 0.f);
            tmem_st32(pcol, pk);
          }
          tmem_st_wait();
        }
        if (valid < TK) {
          // V rows of keys past the valid ones may hold anything (P is 0 there,
          // but 0 * NaN is NaN): zero them. V row n holds key n / HPI.
          uint8_t* vs = kv_s + (t % S) * 2 * kTileBytes + kTileBytes;
          // the warps that take this tile: its group (ALT = 2), or both halves
          const int me = ALT == 2 ? quarter * 32 + lane : (chalf * W + quarter) * 32 + lane;
          for (int n = me; n < kTileK; n += n_tile_sm * 32) {
            if (n / HPI < valid) continue;
            for (int ch = 0; ch < 16; ++ch)
              *reinterpret_cast<uint4*>((ch < 8 ? vs : vs + kTileBytes / 2) + swz(n, ch & 7)) =
                  make_uint4(0, 0, 0, 0);
          }
          fence_proxy_async_smem();
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&p_full[sb]);
      }
      if (!ok) break;
      // hand the row max and this half's row sums to the epilogue warps; the
      // slot is free again once the epilogue has finished item_seq - 2 (it then
      // wrote this item's Q, which the item's first S MMA waited for)
      float* mls = ml_s + slot * 512;
      mls[256 * chalf + r] = m_run;
      mls[256 * chalf + 128 + r] = l_part;
      __syncwarp();
      if (lane == 0) mbar_arrive(&l_full[slot]);
      tile_seq += it.n_tiles;
      ++item_seq;
    }
  } else if (is_epi) {
    // ------------------------------ epilogue ------------------------------
    // Per item: put the next item's Q rows into TMEM (once this item's last S
    // has read the buffer), then read this item's O out.
    const int r = quarter * 32 + lane;
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    // the ring entry of item number `seq` into `out`: 0 (a piece), -1 (no more)
    // or -2 (gave up)
    auto read_item = [&](int seq, AttnItem& out) -> int {
      const int sl = seq & 1;
      if (!__all_sync(0xffffffffu, wait_or_abort(&it_full[sl], (uint32_t)((seq >> 1) & 1), abort_flag, p.err, 38, p.wait_ns)))
        return -2;
      out = ring[sl];
      __syncwarp();
      if (lane == 0) mbar_arrive(&it_empty[sl]);
      return out.b < 0 ? -1 : 0;
    };
    // this lane's packed query row r of item `item` (r = i * Gi + head) into
    // TMEM columns kQCol..kQCol+63; rows past Mi stay unwritten (padding lanes)
    auto put_q = [&](const AttnItem& qi, int seq) -> bool {
      uint32_t qv[64];
      if (r < p.Mi) {
        const int i = r / p.Gi, hh = r - i * p.Gi;
        const uint4* src = reinterpret_cast<const uint4*>(
            p.q + ((size_t)(qi.b * p.n_q + i) * p.Hq + qi.g * p.Gi + hh) * attn::kD);
#pragma unroll
        for (int k = 0; k < 16; ++k) {
          const uint4 v = __ldg(src + k);
          qv[4 * k] = v.x; qv[4 * k + 1] = v.y; qv[4 * k + 2] = v.z; qv[4 * k + 3] = v.w;
        }
      } else {
#pragma unroll
        for (int k = 0; k < 64; ++k) qv[k] = 0u;
      }
      // the previous item's last S must have read the buffer
      if (seq > 0 &&
          !__all_sync(0xffffffffu, wait_or_abort(&q_empty[0], (uint32_t)((seq - 1) & 1), abort_flag, p.err, 40, p.wait_ns)))
        return false;
      tc_fence_after();
      tmem_st32(tmem_base + lane_off + kQCol, qv);
      tmem_st32(tmem_base + lane_off + kQCol + 32, qv + 32);
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&q_full[0]);
      return true;
    };
    int item_seq = 0;
    AttnItem it_cur, it_nxt;
    int st_cur = read_item(0, it_cur);
    bool qok = st_cur == 0 ? put_q(it_cur, 0) : false;
    while (st_cur == 0 && qok) {
      const int st_nxt = read_item(item_seq + 1, it_nxt);
      if (st_nxt == -2) break;
      if (st_nxt == 0 && !put_q(it_nxt, item_seq + 1)) break;
      const int slot = item_seq & 1;
      const uint32_t par = (uint32_t)((item_seq >> 1) & 1);
      const AttnItem it = it_cur;
      const int oi = ALT == 2 ? 0 : slot;
      const uint32_t opar = ALT == 2 ? (uint32_t)(item_seq & 1) : par;
      if (!__all_sync(0xffffffffu, wait_or_abort(&l_full[slot], par, abort_flag, p.err, 39, p.wait_ns))) break;
      if (!__all_sync(0xffffffffu, wait_or_abort(&o_full[oi], opar, abort_flag, p.err, 35, p.wait_ns))) break;
      tc_fence_after();
      const float* mls = ml_s + slot * 512;
      const float ma = mls[r], la = mls[128 + r], mb = mls[256 + r], lb = mls[384 + r];
      // one O (ALT = 1: the halves' sums share one max) or two O merged (ALT = 2)
      float m_run, l_run, wa = 1.f, wb = 0.f;
      if (ALT == 1) {
        m_run = ma;
        l_run = la + lb;
      } else {
        // which half is "a" depends on where the item fell in the CTA's tile
        // count: the merge is written without contraction into FMAs, so that it
        // is symmetric in a and b and its rounding does not depend on that
        m_run = fmaxf(ma, mb);
        wa = la > 0.f ? exp2f(ma - m_run) : 0.f;
        wb = lb > 0.f ? exp2f(mb - m_run) : 0.f;
        l_run = __fadd_rn(__fmul_rn(la, wa), __fmul_rn(lb, wb));
      }
      const bool single = (it.nsplit == 1);
      const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
      // partial slot of a split piece: two per range, one for the piece that
      // starts the range and one for the piece that starts inside it
      const int nt_b = cum[it.b + 1] - cum[it.b];
      const int start = p.n_groups * cum[it.b] + it.g * nt_b + it.t0;
      const size_t cta = 2 * (size_t)(start / plan.share) + (start % plan.share != 0 ? 1 : 0);
      const uint32_t o_col = 128 + (uint32_t)((ALT == 2 ? 0 : slot) * attn::kD);
      for (int c = 0; c < attn::kD / 32; ++c) {
        uint32_t o[32];
        tmem_ld32(tmem_base + lane_off + o_col + c * 32, o);
        if (ALT == 2) {
          uint32_t ob[32];
          tmem_ld32(tmem_base + lane_off + o_col + attn::kD + c * 32, ob);
          tmem_ld_wait();
#pragma unroll
          for (int q = 0; q < 32; ++q) {
            // a half that took no tile has l = 0 and an O that was never written
            const float xa = wa != 0.f ? __fmul_rn(__uint_as_float(o[q]), wa) : 0.f;
            const float xb = wb != 0.f ? __fmul_rn(__uint_as_float(ob[q]), wb) : 0.f;
            o[q] = __float_as_uint(__fadd_rn(xa, xb));
          }
        } else {
          tmem_ld_wait();
        }
        if (r < p.Mi) {
          if (single) {
            const int i = r / p.Gi, hh = r - i * p.Gi;
            bf16* dst = p.out + ((size_t)(it.b * p.n_q + i) * p.Hq + it.g * p.Gi + hh) * attn::kD + c * 32;
#pragma unroll
            for (int q = 0; q < 32; q += 8) {
              uint4 v;
              v.x = pack_bf16(__uint_as_float(o[q + 0]) * inv, __uint_as_float(o[q + 1]) * inv);
              v.y = pack_bf16(__uint_as_float(o[q + 2]) * inv, __uint_as_float(o[q + 3]) * inv);
              v.z = pack_bf16(__uint_as_float(o[q + 4]) * inv, __uint_as_float(o[q + 5]) * inv);
              v.w = pack_bf16(__uint_as_float(o[q + 6]) * inv, __uint_as_float(o[q + 7]) * inv);
              *reinterpret_cast<uint4*>(dst + q) = v;
            }
          } else {
            float* dst = p.part_o + (cta * p.Mi + r) * attn::kD + c * 32;
#pragma unroll
            for (int q = 0; q < 32; q += 4)
              *reinterpret_cast<float4*>(dst + q) = make_float4(__uint_as_float(o[q]), __uint_as_float(o[q + 1]),
                                                                __uint_as_float(o[q + 2]), __uint_as_float(o[q + 3]));
          }
        }
      }
      if (!single && r < p.Mi) p.part_ml[cta * p.Mi + r] = make_float2(m_run, l_run);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&o_empty[oi]);
      it_cur = it_nxt;
      st_cur = st_nxt;
      ++item_seq;
    }
  }

  // ------------------------------ teardown ------------------------------
  tc_fence_before();
  __syncthreads();
  if (warp == prod_warp && lane == 0 && *abort_flag)
    for (int i = *consumed_sm; i < producer_issued; ++i)
      mbar_wait_bounded(&kv_full[i % S], (uint32_t)((i / S) & 1), p.err, 36);
  __syncthreads();
  if (warp == mma_warp) {
    tc_fence_after();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

// ===========================================================================
// Split merge: for every (sequence, kv-head group) whose tiles the partition cut
// into pieces, out = sum over the pieces s (in split order) of
// 2^(m_s - m) O_s / sum_s 2^(m_s - m) l_s. Thread: one packed row, 8 or 16 columns.
// ===========================================================================
constexpr int kMergeThreads = 512;

// COLS columns of one packed row per thread; the partial sums of PRE = 64 /
// COLS pieces are loaded at a time (with the first group, the statistics too).
template <int COLS>
__global__ void __launch_bounds__(kMergeThreads)
attn_merge_kernel(const AttnParams p) {
  constexpr int PRE = 64 / COLS, V4 = COLS / 4, UPR = attn::kD / COLS;
  // launched while the attention grid runs: wait for it to complete
  wait_for_prior_grid();
  const int grp = blockIdx.x;
  const int b = grp / p.n_groups, g = grp - b * p.n_groups;
  const int* cum = p.plan_ws + 1;
  const int share = p.plan_ws[0];
  const int nt = cum[b + 1] - cum[b];
  if (nt == 0) return;                       // inactive sequence
  const int base = p.n_groups * cum[b] + g * nt;
  const int nsplit = (base + nt - 1) / share - base / share + 1;
  if (nsplit < 2) return;                    // written whole by its one piece
  const int u = blockIdx.y * kMergeThreads + threadIdx.x;
  if (u >= p.Mi * UPR) return;
  const int r = u / UPR, c0 = (u - r * UPR) * COLS;
  // piece sp of the group sits in range base / share + sp; only the first piece
  // can start inside its range (slot 2 v + 1), the others start theirs (2 v)
  const int v0 = base / share, in0 = base % share != 0 ? 1 : 0;
  auto slot_of = [&](int sp) -> size_t { return 2 * (size_t)(v0 + sp) + (sp == 0 ? in0 : 0); };
  const float2* ml = p.part_ml + r;
  const float4* src0 = reinterpret_cast<const float4*>(p.part_o + (size_t)r * attn::kD + c0);
  const size_t sstride = (size_t)p.Mi * attn::kD / 4;   // float4 per slot
  const size_t mstride = (size_t)p.Mi;                  // float2 per slot
  float2 mv[PRE];
  float4 x[PRE][V4];
#pragma unroll
  for (int j = 0; j < PRE; ++j) {
    if (j < nsplit) {
      mv[j] = __ldg(ml + slot_of(j) * mstride);
#pragma unroll
      for (int q = 0; q < V4; ++q) x[j][q] = __ldg(src0 + slot_of(j) * sstride + q);
    }
  }
  float mx = -CUDART_INF_F;
#pragma unroll
  for (int j = 0; j < PRE; ++j)
    if (j < nsplit) mx = fmaxf(mx, mv[j].x);
  for (int s0 = PRE; s0 < nsplit; s0 += PRE) {
    float2 w4[PRE];
#pragma unroll
    for (int j = 0; j < PRE; ++j)
      if (s0 + j < nsplit) w4[j] = __ldg(ml + slot_of(s0 + j) * mstride);
#pragma unroll
    for (int j = 0; j < PRE; ++j)
      if (s0 + j < nsplit) mx = fmaxf(mx, w4[j].x);
  }
  float L = 0.f;
#pragma unroll
  for (int j = 0; j < PRE; ++j)
    if (j < nsplit) L += mv[j].x == -CUDART_INF_F ? 0.f : mv[j].y * exp2f(mv[j].x - mx);
  for (int sp = PRE; sp < nsplit; ++sp) {
    const float2 v = __ldg(ml + slot_of(sp) * mstride);
    L += v.x == -CUDART_INF_F ? 0.f : v.y * exp2f(v.x - mx);
  }
  const float inv_l = L > 0.f ? 1.f / L : 0.f;
  float acc[COLS];
#pragma unroll
  for (int q = 0; q < COLS; ++q) acc[q] = 0.f;
  for (int s0 = 0; s0 < nsplit; s0 += PRE) {
    if (s0 > 0) {
#pragma unroll
      for (int j = 0; j < PRE; ++j) {
        if (s0 + j < nsplit) {
          mv[j] = __ldg(ml + slot_of(s0 + j) * mstride);
#pragma unroll
          for (int q = 0; q < V4; ++q) x[j][q] = __ldg(src0 + slot_of(s0 + j) * sstride + q);
        }
      }
    }
#pragma unroll
    for (int j = 0; j < PRE; ++j) {
      if (s0 + j < nsplit) {
        const float w = mv[j].x == -CUDART_INF_F ? 0.f : exp2f(mv[j].x - mx) * inv_l;
#pragma unroll
        for (int q = 0; q < V4; ++q) {
          acc[4 * q + 0] += w * x[j][q].x;
          acc[4 * q + 1] += w * x[j][q].y;
          acc[4 * q + 2] += w * x[j][q].z;
          acc[4 * q + 3] += w * x[j][q].w;
        }
      }
    }
  }
  const int i = r / p.Gi, hh = r - i * p.Gi;
  bf16* dst = p.out + ((size_t)(b * p.n_q + i) * p.Hq + g * p.Gi + hh) * attn::kD + c0;
#pragma unroll
  for (int q = 0; q < COLS; q += 8) {
    uint4 v;
    v.x = pack_bf16(acc[q + 0], acc[q + 1]);
    v.y = pack_bf16(acc[q + 2], acc[q + 3]);
    v.z = pack_bf16(acc[q + 4], acc[q + 5]);
    v.w = pack_bf16(acc[q + 6], acc[q + 7]);
    *reinterpret_cast<uint4*>(dst + q) = v;
  }
}

// ===========================================================================
// Generic path: one CTA per (query position, q head, sequence), fp32 math.
// ===========================================================================
template <typename T>
__global__ void __launch_bounds__(128)
attn_generic_kernel(const T* __restrict__ q, const T* __restrict__ k_blk, const T* __restrict__ v_blk,
                    const T* __restrict__ k_pool, const T* __restrict__ v_pool,
                    const int32_t* __restrict__ page_table, const int32_t* __restrict__ ctx_len,
                    const uint8_t* __restrict__ active, T* __restrict__ out, int n_q, int n_kv, int Hq,
                    int Hkv, int D, int page_size, int max_pages, int num_pages, float scale, int causal,
                    int* __restrict__ err) {
  constexpr int KC = 128;   // keys per chunk (one per thread)
  __shared__ float qs[256];
  __shared__ float ps[KC];
  __shared__ int rowidx[KC];
  __shared__ float red[4];
  const int i = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  if (active && !active[b]) return;   // an inactive sequence: nothing read or written
  const int g = h / (Hq / Hkv);
  const int tid = threadIdx.x;
  const int C = max(0, ctx_len[b]);
  const int T_total = C + n_kv;
  for (int d = tid; d < D; d += blockDim.x) qs[d] = to_f32(q[((size_t)(b * n_q + i) * Hq + h) * D + d]);
  float o0 = 0.f, o1 = 0.f;    // d = tid and d = tid + 128
  float m_run = -CUDART_INF_F, l_run = 0.f;
  __syncthreads();
  for (int c0 = 0; c0 < T_total; c0 += KC) {
    const int key = c0 + tid;
    float sc = -CUDART_INF_F;
    const T* krow = nullptr;
    int vrow_kind = -1;
    if (key < T_total) {
      if (key < C) {
        const int lp = key / page_size;
        int phys = (lp < max_pages) ? page_table[(size_t)b * max_pages + lp] : -1;
        if (phys < 0 || phys >= num_pages) {
          // input error (recorded); page 0 is read instead, never out of bounds
          if (err) atomicCAS(err, 0, kDevErrBadPage);
          phys = 0;
        }
        const size_t row = (size_t)phys * page_size + key % page_size;
        krow = k_pool + (row * Hkv + g) * D;
        vrow_kind = (int)row;
      } else {
        krow = k_blk + ((size_t)(b * n_kv + (key - C)) * Hkv + g) * D;
        vrow_kind = -2 - (key - C);
      }
      float acc = 0.f;
      for (int d = 0; d < D; ++d) acc += qs[d] * to_f32(krow[d]);
      sc = acc * scale;
      if (causal && key >= C && key - C > i + n_kv - n_q) sc = -CUDART_INF_F;
    }
    rowidx[tid] = vrow_kind;
    // chunk max
    float mx = sc;
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    if ((tid & 31) == 0) red[tid >> 5] = mx;
    __syncthreads();
    mx = fmaxf(fmaxf(red[0], red[1]), fmaxf(red[2], red[3]));
    const float mnew = fmaxf(m_run, mx);
    const float alpha = (m_run == -CUDART_INF_F) ? 0.f : expf(m_run - mnew);
    const float pw = (sc == -CUDART_INF_F) ? 0.f : expf(sc - mnew);
    ps[tid] = pw;
    __syncthreads();
    float psum = 0.f;
    for (int j = 0; j < KC; ++j) psum += ps[j];
    l_run = l_run * alpha + psum;
    m_run = mnew;
    o0 *= alpha;
    o1 *= alpha;
    const int nk = min(KC, T_total - c0);
    for (int j = 0; j < nk; ++j) {
      const int rk = rowidx[j];
      const T* vrow = rk >= 0 ? v_pool + ((size_t)rk * Hkv + g) * D
                              : v_blk + ((size_t)(b * n_kv + (-2 - rk)) * Hkv + g) * D;
      if (tid < D) o0 += ps[j] * to_f32(vrow[tid]);
      if (tid + 128 < D) o1 += ps[j] * to_f32(vrow[tid + 128]);
    }
    __syncthreads();
  }
  const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
  T* dst = out + ((size_t)(b * n_q + i) * Hq + h) * D;
  if (tid < D) dst[tid] = from_f32<T>(o0 * inv);
  if (tid + 128 < D) dst[tid + 128] = from_f32<T>(o1 * inv);
}

// ===========================================================================
// Host side
// ===========================================================================
static bool bf16_fast_ok(const AttnArgs& a) {
  const int M = a.n_q * (a.Hq / a.Hkv);
  // (the kernel takes row maxima of unscaled scores: the scale must be > 0)
  return a.dtype == 1 && a.D == 128 && M <= 16 * attn::kMaxWarps && a.n_kv >= 1 && a.n_kv <= attn::kTileK &&
         a.scale > 0.f && a.scale < 3.0e38f &&
         a.B <= attn_tc::kMaxSeqs &&
         (a.page_size == 8 || a.page_size == 16 || a.page_size == 32 || a.page_size == 64) &&
         a.num_pages * (long)a.page_size < (1L << 31) &&
         (reinterpret_cast<uintptr_t>(a.k_pool) & 15) == 0 && (reinterpret_cast<uintptr_t>(a.v_pool) & 15) == 0 &&
         (reinterpret_cast<uintptr_t>(a.q) & 15) == 0 && (reinterpret_cast<uintptr_t>(a.k_blk) & 15) == 0 &&
         (reinterpret_cast<uintptr_t>(a.v_blk) & 15) == 0 && (reinterpret_cast<uintptr_t>(a.out) & 15) == 0;
}

// Kv heads per work item: two heads share one item (and one TMA box per page
// and d-half, twice the size of a one-head box) when their packed query rows
// fit the 128 MMA rows and the pages and the block fit the paired box layout.
static int attn_hpi(int n_q, int n_kv, int Hq, int Hkv, int page_size) {
  const int G = Hq / Hkv;
  const bool pair = Hkv % 2 == 0 && 2 * n_q * G <= 128 && page_size >= 16 && n_kv <= attn::kTileK / 2;
  return pair ? 2 : 1;
}

// Partial slots: two per range of the partition (its first piece and a piece
// starting inside it). The ranges number at most max(grid, N / window): a
// range holds at least N / grid tiles unless the page-table window caps it.
static int attn_slots(int B, int n_groups, int max_ctx, int TK, int page_size) {
  const long n_max = (long)B * n_groups * ((max_ctx + TK - 1) / TK + 1);
  const long window = (long)(attn_tc::kPtMax - 1) * page_size / TK;
  return (int)(2 * std::max<long>(attn_tc::kGrid, (n_max + window - 1) / window));
}

size_t attn_ws_bytes(int B, int n_q, int n_kv, int Hq, int Hkv, int D, int max_ctx, int page_size, int dtype) {
  if (dtype != 1 || D != 128) return 0;
  const int hpi = attn_hpi(n_q, n_kv, Hq, Hkv, page_size);
  const int Mi = hpi * n_q * (Hq / Hkv);
  const size_t ctas = (size_t)attn_slots(B, Hkv / hpi, max_ctx, attn::kTileK / hpi, page_size);
  return align_up(ctas * Mi * 128 * sizeof(float)) + align_up(ctas * Mi * sizeof(float2)) +
         align_up((size_t)(B + 2) * sizeof(int32_t));
}

template <int kThreadsT, int HPI>
static cudaError_t launch_attn_tc(const CUtensorMap& kmap, const CUtensorMap& vmap, const CUtensorMap& kbmap,
                                  const CUtensorMap& vbmap, const AttnParams& p,
                                  int S, size_t smem, cudaStream_t st, int* launches) {
  static SmemOptIn opt_in;
  cudaError_t e = opt_in.ensure(attn_tc_kernel<kThreadsT, HPI>, smem);
  if (e != cudaSuccess) return e;
  // a plain launch: as a dependent of the kernel before it, the CTAs reach the
  // SMs in a different order and the kernel measured 2 % slower
  attn_tc_kernel<kThreadsT, HPI><<<attn_tc::kGrid, kThreadsT, smem, st>>>(kmap, vmap, kbmap, vbmap, p, S);
  cudaError_t le = cudaGetLastError();
  if (le != cudaSuccess) return le;
  // the split merge, a programmatic dependent of the attention grid
  // few (sequence, group)s (small batches, many pieces each): 8 columns per
  // thread, every piece's loads at once; many: 16 columns, four pieces at once.
  // A masked call counts as few: it serves the later looped-draft stages, where
  // a minority of the batch is still drafting (DLoop shape, 4 or 10 of 32
  // active: 8 % faster; 20 of 32: 1.5 % slower).
  const bool narrow = p.active != nullptr || p.B * p.n_groups < attn_tc::kGrid / 2;
  const int cols = narrow ? 8 : 16;
  const dim3 mg(p.B * p.n_groups, (p.Mi * (attn::kD / cols) + kMergeThreads - 1) / kMergeThreads);
  if (narrow)
    le = launch_dependent(attn_merge_kernel<8>, mg, dim3(kMergeThreads), 0, st, p);
  else
    le = launch_dependent(attn_merge_kernel<16>, mg, dim3(kMergeThreads), 0, st, p);
  if (le != cudaSuccess) return le;
  *launches = 2;
  return cudaGetLastError();
}

cudaError_t launch_block_attn(const AttnArgs& a, int* launches) {
  *launches = 1;
  if (!bf16_fast_ok(a)) {
    dim3 grid(a.n_q, a.Hq, a.B);
    if (a.dtype == 0)
      attn_generic_kernel<float><<<grid, 128, 0, a.stream>>>(
          (const float*)a.q, (const float*)a.k_blk, (const float*)a.v_blk, (const float*)a.k_pool,
          (const float*)a.v_pool, a.page_table, a.ctx_len, a.active, (float*)a.out, a.n_q, a.n_kv, a.Hq, a.Hkv,
          a.D, a.page_size, a.max_pages, a.num_pages, a.scale, a.causal, a.err);
    else
      attn_generic_kernel<bf16><<<grid, 128, 0, a.stream>>>(
          (const bf16*)a.q, (const bf16*)a.k_blk, (const bf16*)a.v_blk, (const bf16*)a.k_pool,
          (const bf16*)a.v_pool, a.page_table, a.ctx_len, a.active, (bf16*)a.out, a.n_q, a.n_kv, a.Hq, a.Hkv,
          a.D, a.page_size, a.max_pages, a.num_pages, a.scale, a.causal, a.err);
    return cudaGetLastError();
  }
  using namespace attn;
  AttnParams p;
  p.q = (const bf16*)a.q;
  p.k_blk = (const bf16*)a.k_blk;
  p.v_blk = (const bf16*)a.v_blk;
  p.page_table = a.page_table;
  p.ctx_len = a.ctx_len;
  p.active = a.active;
  p.out = (bf16*)a.out;
  p.B = a.B; p.n_q = a.n_q; p.n_kv = a.n_kv; p.Hq = a.Hq; p.Hkv = a.Hkv; p.G = a.Hq / a.Hkv;
  p.causal = a.causal;
  p.M = a.n_q * p.G;
  p.page_size = a.page_size; p.max_pages = a.max_pages; p.num_pages = a.num_pages;
  p.hpi = attn_hpi(a.n_q, a.n_kv, a.Hq, a.Hkv, a.page_size);
  p.Gi = p.hpi * p.G;
  p.Mi = p.hpi * p.M;
  p.n_groups = a.Hkv / p.hpi;
  p.TK = kTileK / p.hpi;
  p.br = p.hpi == 1 ? a.page_size : std::min(a.page_size, 32);
  p.n_slots = attn_slots(a.B, p.n_groups, a.max_ctx, p.TK, a.page_size);
  p.max_ctx = a.max_ctx;
  p.scale_log2 = a.scale * kLog2e;
  p.wait_ns = wait_limit_ns();
  const int M = p.Mi;
  const size_t ctas = (size_t)p.n_slots;
  char* ws = (char*)a.scratch;
  p.part_o = (float*)ws;
  p.part_ml = (float2*)(ws + align_up(ctas * M * 128 * sizeof(float)));
  p.plan_ws = (int32_t*)(ws + align_up(ctas * M * 128 * sizeof(float)) + align_up(ctas * M * sizeof(float2)));
  p.err = a.err;
  // K/V pools and the block rows as [row][head][d]: a box of {64 d, hpi heads,
  // br rows} lands as [row][head][64 d]
  CUtensorMap kmap, vmap, kbmap, vbmap;
  {
    const uint64_t dims[3] = {(uint64_t)kD, (uint64_t)a.Hkv, (uint64_t)a.num_pages * a.page_size};
    const uint64_t strides[2] = {(uint64_t)kD * 2, (uint64_t)a.Hkv * kD * 2};
    const uint32_t box[3] = {64, (uint32_t)p.hpi, (uint32_t)p.br};
    const uint64_t bd[3] = {(uint64_t)kD, (uint64_t)a.Hkv, (uint64_t)a.B * a.n_kv};
    const uint64_t bs[2] = {(uint64_t)kD * 2, (uint64_t)a.Hkv * kD * 2};
    const uint32_t bb[3] = {64, (uint32_t)p.hpi, (uint32_t)a.n_kv};
    if (!encode_tensor_map(&kmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(a.k_pool), dims,
                           strides, box, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_tensor_map(&vmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(a.v_pool), dims,
                           strides, box, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_tensor_map(&kbmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(a.k_blk), bd, bs, bb,
                           CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_tensor_map(&vbmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(a.v_blk), bd, bs, bb,
                           CU_TENSOR_MAP_SWIZZLE_128B))
      return cudaErrorNotSupported;   // tensor-map encoding refused a layout
  }
  // K/V stages that fit beside the Q buffer (at most the barrier count)
  const size_t fixed = 1024 + attn_tc::kBarBytes;   // Q lives in TMEM
  const int S = (int)std::min<size_t>(attn_tc::kMaxStages, (232448 - fixed) / (2 * attn_tc::kTileBytes));
  const size_t smem = fixed + (size_t)S * 2 * attn_tc::kTileBytes;
  // warps 0-9 (two softmax quarters, producer, MMA, epilogue 8-9) or 0-13
  const bool wide = (M + 31) / 32 > 2;
  cudaError_t e;
  if (wide)
    e = p.hpi == 2 ? launch_attn_tc<448, 2>(kmap, vmap, kbmap, vbmap, p, S, smem, a.stream, launches)
                   : launch_attn_tc<448, 1>(kmap, vmap, kbmap, vbmap, p, S, smem, a.stream, launches);
  else
    e = p.hpi == 2 ? launch_attn_tc<320, 2>(kmap, vmap, kbmap, vbmap, p, S, smem, a.stream, launches)
                   : launch_attn_tc<320, 1>(kmap, vmap, kbmap, vbmap, p, S, smem, a.stream, launches);
  return e;
}

}  // namespace dflash
