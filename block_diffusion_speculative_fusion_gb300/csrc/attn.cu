// Draft block attention: softmax(scale * Q K^T) V with no mask, GQA, where the
// keys/values of sequence b are its ctx_len[b] context rows in the paged pools
// followed by the block's own rows.
//   DFlash page, section 块扩散 (bidirectional attention inside the block) and
//   KV 注入 step 3 (Attention(Q_draft, [K_draft; K_ctx], [V_draft; V_ctx])).
//
// bf16 / D = 128 path (the serving shapes): one CTA per (key split, kv head,
// sequence). The n_q * (Hq/Hkv) query rows that share a kv head are packed into
// the M dimension (GQA packing), so each K/V byte is read from HBM once per
// kv head. Context pages arrive by TMA (one 128B-swizzled box per page half)
// into a 3-stage ring; scores and P V run on mma.sync bf16 tensor cores with an
// online softmax in fp32. Splits of one (sequence, kv head) are merged by the
// last CTA to finish (completion ticket, no waiting).
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
constexpr int kStages = 3;
constexpr int kHalfBytes = kTileK * 128;     // [64 keys][64 d] bf16 = 8 KB
constexpr int kTileBytes = 2 * kHalfBytes;   // K (or V) of one tile = 16 KB
constexpr int kTilesPerSplit = 16;           // 1024 keys per CTA
constexpr int kMaxWarps = 8;                 // M <= 128 packed query rows
}  // namespace attn

struct AttnParams {
  const bf16* q;
  const bf16* k_blk;
  const bf16* v_blk;
  const int32_t* page_table;
  const int32_t* ctx_len;
  bf16* out;
  float* part_o;     // [B * Hkv * max_splits][M][128]
  float2* part_ml;   // [B * Hkv * max_splits][M]  (max in log2 units, sum)
  int32_t* counters; // [B * Hkv]
  int* err;
  int B, n_q, n_kv, Hq, Hkv, G, M, page_size, max_pages, num_pages, max_splits, max_ctx;
  float scale_log2;  // softmax scale * log2(e)
};

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr));
}
__device__ __forceinline__ void mma_bf16_16816(float* c, const uint32_t* a, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// Byte offset of 16-byte chunk `c` (0..7) of row `r` in a [rows][64] bf16 half
// tile with the 128-byte TMA swizzle (chunk index XOR row mod 8).
__device__ __forceinline__ uint32_t swz(int r, int c) { return (uint32_t)(r * 128 + ((c ^ (r & 7)) << 4)); }

// Copy one 128-element bf16 row into two swizzled half tiles (or zero it).
__device__ __forceinline__ void put_row(uint8_t* half0, uint8_t* half1, int r, const bf16* src, int chunk) {
  uint4 v = src ? *reinterpret_cast<const uint4*>(src + chunk * 8) : make_uint4(0, 0, 0, 0);
  uint8_t* h = chunk < 8 ? half0 : half1;
  *reinterpret_cast<uint4*>(h + swz(r, chunk & 7)) = v;
}

__global__ void __launch_bounds__(256, 1)
attn_bf16_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                 const AttnParams p) {
  using namespace attn;
  const int split = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
  // a length outside [0, max_ctx] would overrun the split workspace: clamp it
  const int C = max(0, min(p.ctx_len[b], p.max_ctx));
  const int n_ctx_tiles = (C + kTileK - 1) / kTileK;
  const int nsplit = max(1, (n_ctx_tiles + kTilesPerSplit - 1) / kTilesPerSplit);
  if (split >= nsplit) return;
  const int t0 = split * kTilesPerSplit;
  const int n_tiles_ctx = max(0, min(n_ctx_tiles, t0 + kTilesPerSplit) - t0);
  const bool has_blk = (split == nsplit - 1) && p.n_kv > 0;
  const int n_tiles = n_tiles_ctx + (has_blk ? 1 : 0);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int nwarps = blockDim.x >> 5;
  const int Mpad = nwarps * 16;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* kv = smem;                                        // stage s: K at s*2*T, V at s*2*T + T
  // Q halves [Mpad][64] x 2 live in the last stage until they are in registers
  uint8_t* qs = smem + (kStages - 1) * 2 * kTileBytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kStages * 2 * kTileBytes);

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) mbar_init(&bars[s], 1);
    fence_barrier_init();
  }
  // Q rows of this kv head: packed row r = i * G + hh  (position i, head g*G + hh)
  for (int idx = tid; idx < Mpad * 16; idx += blockDim.x) {
    const int r = idx >> 4, ch = idx & 15;
    const bf16* src = nullptr;
    if (r < p.M) {
      const int i = r / p.G, hh = r - i * p.G;
      src = p.q + ((size_t)(b * p.n_q + i) * p.Hq + g * p.G + hh) * kD;
    }
    put_row(qs, qs + Mpad * 128, r, src, ch);
  }
  __syncthreads();

  const int ps = p.page_size;
  auto issue = [&](int tile, int stage) {
    uint64_t* bar = &bars[stage];
    mbar_arrive_expect_tx(bar, 2 * kTileBytes);
    const int key0 = (t0 + tile) * kTileK;
    uint8_t* kdst = kv + stage * 2 * kTileBytes;
    uint8_t* vdst = kdst + kTileBytes;
    for (int pg = 0; pg < kTileK / ps; ++pg) {
      const int lp = key0 / ps + pg;
      int row = 0;   // pages past the context (or bad table entries) read page 0; masked below
      if (lp * ps < C && lp < p.max_pages) {
        const int phys = p.page_table[(size_t)b * p.max_pages + lp];
        if (phys >= 0 && phys < p.num_pages) row = phys * ps;
      }
      for (int h = 0; h < 2; ++h) {
        tma_load_3d(kdst + h * kHalfBytes + pg * ps * 128, &kmap, bar, h * 64, g, row);
        tma_load_3d(vdst + h * kHalfBytes + pg * ps * 128, &vmap, bar, h * 64, g, row);
      }
    }
  };
  if (tid == 0)
    for (int s = 0; s < kStages - 1 && s < n_tiles_ctx; ++s) issue(s, s);

  // Q fragments of this warp's 16 rows, all 8 k-slices of D = 128
  uint32_t qa[8][4];
  {
    const int r = warp * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
      const int ch = (kk & 3) * 2 + (lane >> 4);
      const uint32_t addr = smem_u32(qs + (kk >> 2) * Mpad * 128) + swz(r, ch);
      ldsm_x4(addr, qa[kk][0], qa[kk][1], qa[kk][2], qa[kk][3]);
    }
  }
  __syncthreads();   // the last stage is free for TMA once every warp holds its Q fragments

  float o[16][4];
#pragma unroll
  for (int n = 0; n < 16; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
  float m_run[2] = {-CUDART_INF_F, -CUDART_INF_F};
  float l_run[2] = {0.f, 0.f};
  const int qd = lane & 3;    // thread's column pair within an n-tile
  bool failed = false;
  int fail_t = 0;

  for (int t = 0; t < n_tiles; ++t) {
    const int stage = t % kStages;
    const bool is_blk = (t == n_tiles_ctx);
    if (tid == 0 && t + kStages - 1 < n_tiles_ctx) issue(t + kStages - 1, (t + kStages - 1) % kStages);
    uint8_t* ks = kv + stage * 2 * kTileBytes;
    uint8_t* vs = ks + kTileBytes;
    int valid;
    if (!is_blk) {
      const bool ok = mbar_wait_bounded(&bars[stage], (uint32_t)((t / kStages) & 1), p.err, 1);
      if (__syncthreads_or(!ok)) { failed = true; fail_t = t; break; }
      valid = min(kTileK, C - (t0 + t) * kTileK);
    } else {
      for (int idx = tid; idx < kTileK * 16; idx += blockDim.x) {
        const int r = idx >> 4, ch = idx & 15;
        const size_t off = ((size_t)(b * p.n_kv + r) * p.Hkv + g) * kD;
        put_row(ks, ks + kHalfBytes, r, r < p.n_kv ? p.k_blk + off : nullptr, ch);
        put_row(vs, vs + kHalfBytes, r, r < p.n_kv ? p.v_blk + off : nullptr, ch);
      }
      __syncthreads();
      valid = p.n_kv;
    }

    // ---- S = Q K^T for this warp's 16 rows x 64 keys ----
    float s[8][4];
#pragma unroll
    for (int n = 0; n < 8; ++n) s[n][0] = s[n][1] = s[n][2] = s[n][3] = 0.f;
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
      const uint32_t kbase = smem_u32(ks + (kk >> 2) * kHalfBytes);
#pragma unroll
      for (int np = 0; np < 4; ++np) {
        const int r = np * 16 + (lane & 7) + (lane >> 4) * 8;
        const int ch = (kk & 3) * 2 + ((lane >> 3) & 1);
        uint32_t b0, b1, b2, b3;
        ldsm_x4(kbase + swz(r, ch), b0, b1, b2, b3);
        mma_bf16_16816(s[2 * np], qa[kk], b0, b1);
        mma_bf16_16816(s[2 * np + 1], qa[kk], b2, b3);
      }
    }
    // ---- online softmax (base 2) ----
    float mx[2] = {m_run[0], m_run[1]};
#pragma unroll
    for (int n = 0; n < 8; ++n)
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int key = n * 8 + qd * 2 + (j & 1);
        const float v = key < valid ? s[n][j] * p.scale_log2 : -CUDART_INF_F;
        s[n][j] = v;
        mx[j >> 1] = fmaxf(mx[j >> 1], v);
      }
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 1));
      mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 2));
    }
    float alpha[2], base[2];
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      base[r] = (mx[r] == -CUDART_INF_F) ? 0.f : mx[r];
      alpha[r] = (m_run[r] == -CUDART_INF_F) ? 0.f : exp2f(m_run[r] - base[r]);
      m_run[r] = mx[r];
    }
    float rs[2] = {0.f, 0.f};
#pragma unroll
    for (int n = 0; n < 8; ++n)
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float e = exp2f(s[n][j] - base[j >> 1]);
        s[n][j] = e;
        rs[j >> 1] += e;
      }
#pragma unroll
    for (int r = 0; r < 2; ++r) l_run[r] = l_run[r] * alpha[r] + rs[r];
#pragma unroll
    for (int n = 0; n < 16; ++n) {
      o[n][0] *= alpha[0]; o[n][1] *= alpha[0];
      o[n][2] *= alpha[1]; o[n][3] *= alpha[1];
    }
    // ---- O += P V ----
#pragma unroll
    for (int kv4 = 0; kv4 < 4; ++kv4) {
      uint32_t a[4];
      a[0] = pack_bf16(s[2 * kv4][0], s[2 * kv4][1]);
      a[1] = pack_bf16(s[2 * kv4][2], s[2 * kv4][3]);
      a[2] = pack_bf16(s[2 * kv4 + 1][0], s[2 * kv4 + 1][1]);
      a[3] = pack_bf16(s[2 * kv4 + 1][2], s[2 * kv4 + 1][3]);
      const int r = kv4 * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
      // keys of this thread's B fragments: kv4*16 + qd*2 + {0,1} (+8 for b1/b3)
      const int kb = kv4 * 16 + qd * 2;
      const bool partial = valid < kTileK;
#pragma unroll
      for (int dp = 0; dp < 8; ++dp) {
        const int ch = (dp & 3) * 2 + (lane >> 4);
        uint32_t b0, b1, b2, b3;
        ldsm_x4_t(smem_u32(vs + (dp >> 2) * kHalfBytes) + swz(r, ch), b0, b1, b2, b3);
        if (partial) {   // rows past the valid keys may hold anything: zero them
          const uint32_t m0 = (kb < valid ? 0xffffu : 0u) | (kb + 1 < valid ? 0xffff0000u : 0u);
          const uint32_t m1 = (kb + 8 < valid ? 0xffffu : 0u) | (kb + 9 < valid ? 0xffff0000u : 0u);
          b0 &= m0; b2 &= m0; b1 &= m1; b3 &= m1;
        }
        mma_bf16_16816(o[2 * dp], a, b0, b1);
        mma_bf16_16816(o[2 * dp + 1], a, b2, b3);
      }
    }
    __syncthreads();   // every warp is done with this stage before it is refilled
  }

  if (failed) {
    // A TMA did not land in time (error recorded): wait, again bounded, for the
    // copies this CTA still has in flight, so none lands after the CTA exits.
    if (tid == 0)
      for (int tt = fail_t; tt < min(n_tiles_ctx, fail_t + kStages); ++tt)
        mbar_wait_bounded(&bars[tt % kStages], (uint32_t)((tt / kStages) & 1), p.err, 1);
    __syncthreads();
    return;
  }

#pragma unroll
  for (int r = 0; r < 2; ++r) {
    l_run[r] += __shfl_xor_sync(0xffffffffu, l_run[r], 1);
    l_run[r] += __shfl_xor_sync(0xffffffffu, l_run[r], 2);
  }
  const int g8 = lane >> 2;
  const int rows[2] = {warp * 16 + g8, warp * 16 + g8 + 8};

  if (nsplit == 1) {
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      const int row = rows[r];
      if (row >= p.M) continue;
      const float inv = l_run[r] > 0.f ? 1.f / l_run[r] : 0.f;
      const int i = row / p.G, hh = row - i * p.G;
      bf16* dst = p.out + ((size_t)(b * p.n_q + i) * p.Hq + g * p.G + hh) * kD;
#pragma unroll
      for (int n = 0; n < 16; ++n) {
        const int d = n * 8 + qd * 2;
        *reinterpret_cast<__nv_bfloat162*>(dst + d) =
            __floats2bfloat162_rn(o[n][2 * r] * inv, o[n][2 * r + 1] * inv);
      }
    }
    return;
  }

  // ---- split partials, then the last split of this (sequence, kv head) merges ----
  const size_t group = (size_t)b * p.Hkv + g;
  const size_t cta = group * p.max_splits + split;
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    const int row = rows[r];
    if (row >= p.M) continue;
    float* dst = p.part_o + (cta * p.M + row) * kD;
#pragma unroll
    for (int n = 0; n < 16; ++n)
      *reinterpret_cast<float2*>(dst + n * 8 + qd * 2) = make_float2(o[n][2 * r], o[n][2 * r + 1]);
    if (qd == 0) p.part_ml[cta * p.M + row] = make_float2(m_run[r], l_run[r]);
  }
  if (!take_ticket_is_last(&p.counters[group], nsplit)) return;

  for (int idx = tid; idx < p.M * (kD / 4); idx += blockDim.x) {
    const int row = idx / (kD / 4), d4 = idx - row * (kD / 4);
    float M = -CUDART_INF_F;
    for (int sp = 0; sp < nsplit; ++sp) M = fmaxf(M, __ldcg(&p.part_ml[(group * p.max_splits + sp) * p.M + row]).x);
    float L = 0.f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    if (M != -CUDART_INF_F) {
      for (int sp = 0; sp < nsplit; ++sp) {
        const size_t c2 = group * p.max_splits + sp;
        const float2 ml = __ldcg(&p.part_ml[c2 * p.M + row]);
        const float w = (ml.x == -CUDART_INF_F) ? 0.f : exp2f(ml.x - M);
        L += ml.y * w;
        const float4 v = __ldcg(reinterpret_cast<const float4*>(p.part_o + (c2 * p.M + row) * kD) + d4);
        acc.x += v.x * w; acc.y += v.y * w; acc.z += v.z * w; acc.w += v.w * w;
      }
    }
    const float inv = L > 0.f ? 1.f / L : 0.f;
    const int i = row / p.G, hh = row - i * p.G;
    bf16* dst = p.out + ((size_t)(b * p.n_q + i) * p.Hq + g * p.G + hh) * kD + d4 * 4;
    reinterpret_cast<__nv_bfloat162*>(dst)[0] = __floats2bfloat162_rn(acc.x * inv, acc.y * inv);
    reinterpret_cast<__nv_bfloat162*>(dst)[1] = __floats2bfloat162_rn(acc.z * inv, acc.w * inv);
  }
  reset_ticket(&p.counters[group]);
}

// ===========================================================================
// tcgen05 path: persistent, warp-specialised, TMEM accumulators.
//   softmax     warps 0..W-1 (W = ceil(M / 32)): thread r owns packed query
//               row r (TMEM lane r)
//   producer    warp 2 (W <= 2) or 4: claims work items, loads Q, streams
//               context K/V pages by TMA into a ring of 64-key stages
//   MMA         the next warp: TMEM allocator and single-thread MMA issuer
// A work item is (key split, kv head, sequence). Per 64-key tile t:
// S_t = Q K_t^T (M = 128, N = 64) into TMEM buffer t % 2; the softmax threads
// read their S row, write P_t (bf16) to shared memory, and the MMA thread
// accumulates O += P_t V_t (M = 128, N = 128, V read MN-major) into the item's
// TMEM O buffer. The running max is only raised (O rescaled in TMEM) when a
// tile's max exceeds it by more than 2^8, so rescaling is rare. Q and O are
// double-buffered per item so that one item's output overlaps the next
// item's MMAs; the K/V ring runs across item boundaries.
// ===========================================================================
namespace attn_tc {
constexpr int kTileK = 64;
constexpr int kMaxStages = 5;
constexpr int kTileBytes = 2 * 64 * 128;   // K (or V) of one tile: two d-halves x 64 keys x 128 B
constexpr int kMaxThreads = 448;
constexpr int kTmemCols = 512;              // S0 [0,64), S1 [64,128), O0 [128,256), O1 [256,384)
constexpr float kRescaleLog2 = 8.f;
constexpr int kGrid = 152;                  // persistent CTAs: one per SM
constexpr int kMaxSeqs = 1024;              // sequences per call on this path
constexpr int kPtMax = 128;                 // page-table entries of one item (page size >= 8)
constexpr int kBarBytes = 41 * 8 + 2 * 4 + (kMaxSeqs + 1) * 4 + 2 * kPtMax * 4 + (2 * 2 * 128 + 2 * 3 * 128) * 4 + 64;
}  // namespace attn_tc

struct AttnItem {
  int b, g, split, nsplit, C, n_tiles_ctx, n_tiles;
};

__device__ __forceinline__ int item_splits(const AttnParams& p, int b) {
  const int C = max(0, min(p.ctx_len[b], p.max_ctx));
  const int n_ctx_tiles = (C + attn_tc::kTileK - 1) / attn_tc::kTileK;
  return max(1, (n_ctx_tiles + attn::kTilesPerSplit - 1) / attn::kTilesPerSplit);
}

// Work item k (0 <= k < cum[B]) in sequence-major, then kv-head, then split
// order; cum[b] = number of items of sequences before b.
__device__ __forceinline__ void decode_item(const AttnParams& p, const int* cum, int k, AttnItem& it) {
  int lo = 0, hi = p.B - 1;
  while (lo < hi) {          // last b with cum[b] <= k
    const int mid = (lo + hi + 1) >> 1;
    if (cum[mid] <= k) lo = mid; else hi = mid - 1;
  }
  it.b = lo;
  it.C = max(0, min(p.ctx_len[it.b], p.max_ctx));
  const int n_ctx_tiles = (it.C + attn_tc::kTileK - 1) / attn_tc::kTileK;
  it.nsplit = max(1, (n_ctx_tiles + attn::kTilesPerSplit - 1) / attn::kTilesPerSplit);
  const int rem = k - cum[it.b];
  it.g = rem / it.nsplit;
  it.split = rem - it.g * it.nsplit;
  const int t0 = it.split * attn::kTilesPerSplit;
  it.n_tiles_ctx = max(0, min(n_ctx_tiles, t0 + attn::kTilesPerSplit) - t0);
  it.n_tiles = it.n_tiles_ctx + ((it.split == it.nsplit - 1 && p.n_kv > 0) ? 1 : 0);
}

// 2^x on the special-function unit (flush-to-zero; P is rounded to bf16 anyway).
__device__ __forceinline__ float ex2_ftz(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

template <int kThreadsT>
__global__ void __launch_bounds__(kThreadsT, 1)
attn_tc_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
               const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap kbmap,
               const __grid_constant__ CUtensorMap vbmap, const AttnParams p, int Ms, int S, int32_t* sched) {
  using namespace attn_tc;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // Roles, with W = ceil(M / 32) TMEM lane quarters holding real rows:
  //   softmax   warps q and q + 4 for q < W (key columns 0-31 / 32-63 of a tile)
  //   epilogue  warps 8 + q for q < W (O read-out of finished items)
  //   producer  warp 2 (W <= 2) or 12; MMA issuer the warp after it
  const int W = (p.M + 31) / 32;
  const int n_sm = 2 * W;                    // softmax warps
  const int prod_warp = W <= 2 ? 2 : 12, mma_warp = prod_warp + 1;
  const int quarter = warp & 3, chalf = (warp >> 2) & 1;
  const bool is_softmax = warp < 8 && quarter < W && warp != prod_warp && warp != mma_warp;
  const bool is_epi = warp >= 8 && warp < 12 && quarter < W;

  // shared memory: [Q0][Q1: 2 atoms x Ms rows each][P0][P1: Ms rows each][S stages: K | V][barriers, tables]
  // A 128-row MMA reads past the Ms stored rows into the next buffer; those
  // padding rows only produce padding rows of S, P and O, which are never used.
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int atom = Ms * 128;                 // one 64-wide column block of Ms rows
  uint8_t* q_s = smem;                       // Q buffer i at + 2 i atom: d 0-63, then d 64-127
  uint8_t* p_s = smem + 4 * atom;            // P buffer i at + i atom
  uint8_t* kv_s = smem + 6 * atom;           // stage s: K at s*2*T, V at s*2*T + T
  uint64_t* bars = reinterpret_cast<uint64_t*>(kv_s + S * 2 * kTileBytes);
  uint64_t* kv_full = bars;          // [5]
  uint64_t* kv_empty = bars + 5;     // [5]
  uint64_t* s_full = bars + 10;      // [2]
  uint64_t* s_empty = bars + 12;     // [2]
  uint64_t* p_full = bars + 14;      // [2]
  uint64_t* pv_done = bars + 16;     // [2]
  uint64_t* q_full = bars + 18;      // [2]
  uint64_t* q_empty = bars + 20;     // [2]
  uint64_t* it_full = bars + 22;     // [2]
  uint64_t* it_empty = bars + 24;    // [2]
  uint64_t* o_full = bars + 26;      // [2]  MMA -> epilogue: last P V of the item done
  uint64_t* o_empty = bars + 28;     // [2]  epilogue -> MMA: O buffer read out
  uint64_t* mma_done = bars + 30;
  uint64_t* xbar = bars + 31;        // [4 quarters][2]: the two softmax warps of a quarter
  uint64_t* l_full = bars + 39;      // [2]  softmax -> epilogue: row max and sums of the item
  int* ring = reinterpret_cast<int*>(bars + 41);               // [2] item ids
  int* cum = ring + 2;                                         // [B + 1] item prefix per sequence
  int* pt_s = cum + (kMaxSeqs + 1);                            // [2][kPtMax] page rows of two items
  float* xch = reinterpret_cast<float*>(pt_s + 2 * kPtMax);    // [2 tiles][2 halves][128] tile maxima
  float* ml_s = xch + 2 * 2 * 128;                             // [2 slots][3][128]: m, l half 0, l half 1
  uint32_t* tmem_base_sm = reinterpret_cast<uint32_t*>(ml_s + 2 * 3 * 128);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_base_sm + 1);
  int* consumed_sm = reinterpret_cast<int*>(tmem_base_sm + 2);

  if (tid == 0) {
    for (int i = 0; i < kMaxStages; ++i) {
      mbar_init(&kv_full[i], 1);
      mbar_init(&kv_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s_full[i], 1);
      mbar_init(&s_empty[i], n_sm);
      mbar_init(&p_full[i], n_sm);
      mbar_init(&pv_done[i], 1);
      mbar_init(&q_full[i], 1);
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
  if (warp == 0) {
    // cum[b] = sum over b' < b of Hkv * splits(b'): lane-contiguous runs, then a warp scan
    const int per = (p.B + 31) / 32;
    const int b0 = lane * per, b1 = min(p.B, b0 + per);
    int tot = 0;
    for (int bb = b0; bb < b1; ++bb) tot += p.Hkv * item_splits(p, bb);
    int incl = tot;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    int run = incl - tot;
    for (int bb = b0; bb < b1; ++bb) {
      cum[bb] = run;
      run += p.Hkv * item_splits(p, bb);
    }
    if (lane == 31) cum[p.B] = incl;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_base_sm;
  const int n_items = cum[p.B];
  int producer_issued = 0;

  if (warp == prod_warp) {
    // ------------------------------ producer ------------------------------
    // Items are claimed two ahead, and the page rows and Q of the next item are
    // fetched while the current item's tiles stream, so that item boundaries
    // leave no gap in the K/V stream.
    const int ps = p.page_size;
    int item_seq = 0, tile_seq = 0;
    bool ok = true;
    // page rows of item `item` into table `tb` (whole warp)
    auto load_pages = [&](int item, int tb) {
      AttnItem it;
      decode_item(p, cum, item, it);
      const int lp0 = it.split * attn::kTilesPerSplit * kTileK / ps;
      const int n_lp = it.n_tiles_ctx * kTileK / ps;
      for (int i = lane; i < n_lp; i += 32) {
        const int lp = lp0 + i;
        int row = 0;   // pages past the context (or bad entries) read page 0; masked later
        if (lp * ps < it.C && lp < p.max_pages) {
          const int phys = p.page_table[(size_t)it.b * p.max_pages + lp];
          if (phys >= 0 && phys < p.num_pages) row = phys * ps;
        }
        pt_s[tb * kPtMax + i] = row;
      }
      __syncwarp();
    };
    // Q of item `item` into Q buffer `slot` (lane 0); false on abort
    auto load_q = [&](int item, int seq) -> bool {
      const int slot = seq & 1;
      bool w = true;
      if (lane == 0) {
        w = wait_or_abort(&q_empty[slot], (uint32_t)(((seq >> 1) & 1) ^ 1), abort_flag, p.err, 22);
        if (w) {
          AttnItem it;
          decode_item(p, cum, item, it);
          uint8_t* qb = q_s + slot * 2 * atom;
          // one TMA box [n_q][G][64] per d-half lands in the packed row order r = i * G + hh
          mbar_arrive_expect_tx(&q_full[slot], (uint32_t)(2 * p.M * 128));
          tma_load_3d(qb, &qmap, &q_full[slot], 0, it.g * p.G, it.b * p.n_q);
          tma_load_3d(qb + atom, &qmap, &q_full[slot], 64, it.g * p.G, it.b * p.n_q);
        }
      }
      return __shfl_sync(0xffffffffu, w ? 1 : 0, 0) != 0;
    };
    int cur = 0, nxt = 0;
    if (lane == 0) {
      cur = atomicAdd(&sched[0], 1);
      nxt = atomicAdd(&sched[0], 1);
    }
    cur = __shfl_sync(0xffffffffu, cur, 0);
    nxt = __shfl_sync(0xffffffffu, nxt, 0);
    if (cur < n_items) {
      load_pages(cur, 0);
      ok = load_q(cur, 0);
    }
    while (ok) {
      const bool last = cur >= n_items;
      const int slot = item_seq & 1;
      bool w = true;
      if (lane == 0) w = wait_or_abort(&it_empty[slot], (uint32_t)(((item_seq >> 1) & 1) ^ 1), abort_flag, p.err, 21);
      if (!__shfl_sync(0xffffffffu, w ? 1 : 0, 0)) break;
      if (lane == 0) {
        ring[slot] = last ? -1 : cur;
        mbar_arrive(&it_full[slot]);    // release semantics publish the ring entry
      }
      if (last) break;
      int claimed = 0;                  // item after next; needed one item from now
      if (lane == 0 && nxt < n_items) claimed = atomicAdd(&sched[0], 1);
      AttnItem it;
      decode_item(p, cum, cur, it);
      const int* pt = pt_s + slot * kPtMax;
      for (int j = 0; j < it.n_tiles && ok; ++j, ++tile_seq) {
        if (lane == 0) {
          const int st = tile_seq % S;
          uint8_t* ks = kv_s + st * 2 * kTileBytes;
          uint8_t* vs = ks + kTileBytes;
          if (!wait_or_abort(&kv_empty[st], (uint32_t)(((tile_seq / S) & 1) ^ 1), abort_flag, p.err, 23)) {
            ok = false;
          } else if (j < it.n_tiles_ctx) {
            mbar_arrive_expect_tx(&kv_full[st], 2 * kTileBytes);
            for (int pg = 0; pg < kTileK / ps; ++pg) {
              const int row = pt[j * (kTileK / ps) + pg];
              for (int h = 0; h < 2; ++h) {
                tma_load_3d(ks + h * (kTileBytes / 2) + pg * ps * 128, &kmap, &kv_full[st], h * 64, it.g, row);
                tma_load_3d(vs + h * (kTileBytes / 2) + pg * ps * 128, &vmap, &kv_full[st], h * 64, it.g, row);
              }
            }
            ++producer_issued;
          } else {
            // the block's own n_kv K/V rows; rows past n_kv are masked (K) and
            // zeroed (V) by the softmax warps
            mbar_arrive_expect_tx(&kv_full[st], (uint32_t)(4 * p.n_kv * 128));
            for (int h = 0; h < 2; ++h) {
              tma_load_3d(ks + h * (kTileBytes / 2), &kbmap, &kv_full[st], h * 64, it.g, it.b * p.n_kv);
              tma_load_3d(vs + h * (kTileBytes / 2), &vbmap, &kv_full[st], h * 64, it.g, it.b * p.n_kv);
            }
            ++producer_issued;
          }
        }
        ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
        // a few tiles into this item, fetch the next item's page rows and Q
        if (ok && j == min(2, it.n_tiles - 1) && nxt < n_items) {
          load_pages(nxt, slot ^ 1);
          ok = load_q(nxt, item_seq + 1);
        }
      }
      cur = nxt;
      nxt = __shfl_sync(0xffffffffu, nxt < n_items ? claimed : nxt, 0);
      ++item_seq;
    }
    // the last CTA to finish resets the work counter for the next launch
    if (lane == 0) {
      __threadfence();
      if (atomicAdd(&sched[1], 1) == (int)gridDim.x - 1) {
        sched[0] = 0;
        sched[1] = 0;
        __threadfence();
      }
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
        if (!wait_or_abort(&it_full[slot], par, abort_flag, p.err, 24)) break;
        const int item = *reinterpret_cast<volatile int*>(&ring[slot]);
        mbar_arrive(&it_empty[slot]);
        if (item < 0) break;
        AttnItem it;
        decode_item(p, cum, item, it);
        if (!wait_or_abort(&q_full[slot], par, abort_flag, p.err, 25)) break;
        if (!wait_or_abort(&o_empty[slot], par ^ 1u, abort_flag, p.err, 26)) break;
        tc_fence_after();
        const uint32_t qa = smem_u32(q_s + slot * 2 * atom);
        const uint32_t o_tmem = tmem_base + 128 + (uint32_t)(slot * attn::kD);
        auto issue_pv = [&](int t, int j) -> bool {
          if (!wait_or_abort(&p_full[t & 1], (uint32_t)((t >> 1) & 1), abort_flag, p.err, 27)) return false;
          tc_fence_after();
          const uint32_t pa = smem_u32(p_s + (t & 1) * atom);
          const uint32_t va = smem_u32(kv_s + (t % S) * 2 * kTileBytes + kTileBytes);
#pragma unroll
          for (int i = 0; i < kTileK / 16; ++i)
            tc_mma_bf16(o_tmem, sdesc_sw128(pa + i * 32), sdesc_sw128_mn(va + i * 2048, kTileBytes / 2), id_pv,
                        (j > 0 || i > 0) ? 1u : 0u);
          tc_commit(&pv_done[t & 1]);
          tc_commit(&kv_empty[t % S]);
          ++consumed;
          return true;
        };
        for (int j = 0; j < it.n_tiles && ok; ++j) {
          const int t = tile_seq + j;
          const int st = t % S;
          if (!wait_or_abort(&kv_full[st], (uint32_t)((t / S) & 1), abort_flag, p.err, 28)) { ok = false; break; }
          if (!wait_or_abort(&s_empty[t & 1], (uint32_t)(((t >> 1) & 1) ^ 1), abort_flag, p.err, 29)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t ka = smem_u32(kv_s + st * 2 * kTileBytes);
#pragma unroll
          for (int i = 0; i < attn::kD / 16; ++i) {
            const uint32_t off = (uint32_t)((i >> 2) * (kTileBytes / 2) + (i & 3) * 32);
            const uint32_t qoff = (uint32_t)((i >> 2) * atom + (i & 3) * 32);
            tc_mma_bf16(tmem_base + (uint32_t)((t & 1) * kTileK), sdesc_sw128(qa + qoff), sdesc_sw128(ka + off),
                        id_s, i > 0 ? 1u : 0u);
          }
          tc_commit(&s_full[t & 1]);
          if (j == it.n_tiles - 1) tc_commit(&q_empty[slot]);   // Q is no longer read
          if (j >= 1) ok = issue_pv(t - 1, j - 1);
        }
        if (!ok) break;
        if (!issue_pv(tile_seq + it.n_tiles - 1, it.n_tiles - 1)) break;
        tc_commit(&o_full[slot]);
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
    const int c0 = chalf * 32;                      // this warp's 32 key columns of a tile
    const uint32_t oc0 = (uint32_t)(chalf * 64);    // and 64 of the 128 O columns for rescaling
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
      return __all_sync(0xffffffffu, wait_or_abort(bar, par, abort_flag, p.err, 37));
    };
    while (ok) {
      const int slot = item_seq & 1;
      const uint32_t par = (uint32_t)((item_seq >> 1) & 1);
      if (!__all_sync(0xffffffffu, wait_or_abort(&it_full[slot], par, abort_flag, p.err, 31))) break;
      const int item = *reinterpret_cast<volatile int*>(&ring[slot]);
      __syncwarp();
      if (lane == 0) mbar_arrive(&it_empty[slot]);
      if (item < 0) break;
      AttnItem it;
      decode_item(p, cum, item, it);
      const int t0 = it.split * attn::kTilesPerSplit;
      const uint32_t o_col = 128 + (uint32_t)(slot * attn::kD) + oc0;
      float m_run = -CUDART_INF_F, l_part = 0.f;
      for (int j = 0; j < it.n_tiles; ++j) {
        const int t = tile_seq + j;
        const int sb = t & 1;
        if (!__all_sync(0xffffffffu, wait_or_abort(&s_full[sb], (uint32_t)((t >> 1) & 1), abort_flag, p.err, 32))) {
          ok = false;
          break;
        }
        tc_fence_after();
        float sv[32];
        {
          uint32_t raw[32];
          tmem_ld32(tmem_base + lane_off + (uint32_t)(sb * kTileK + c0), raw);
          tmem_ld_wait();
#pragma unroll
          for (int c = 0; c < 32; ++c) sv[c] = __uint_as_float(raw[c]);
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&s_empty[sb]);
        const int valid = (j < it.n_tiles_ctx) ? min(kTileK, it.C - (t0 + j) * kTileK) : p.n_kv;
        float mx[4] = {-CUDART_INF_F, -CUDART_INF_F, -CUDART_INF_F, -CUDART_INF_F};
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          sv[c] = (c0 + c) < valid ? sv[c] * p.scale_log2 : -CUDART_INF_F;
          mx[c & 3] = fmaxf(mx[c & 3], sv[c]);
        }
        // tile max of the row over both column halves
        float* xb = xch + (t & 1) * 256;
        xb[chalf * 128 + r] = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3]));
        if (!pair_exchange()) {
          ok = false;
          break;
        }
        const float mt = fmaxf(xb[r], xb[128 + r]);
        const bool raise = mt > m_run + kRescaleLog2 || (m_run == -CUDART_INF_F && mt != -CUDART_INF_F);
        const float m_new = raise ? mt : m_run;
        const float alpha = raise ? (m_run == -CUDART_INF_F ? 0.f : exp2f(m_run - m_new)) : 1.f;
        if (j >= 1 && __any_sync(0xffffffffu, raise)) {
          // O must hold every earlier tile of the item before it is rescaled
          if (!__all_sync(0xffffffffu, wait_or_abort(&pv_done[(t - 1) & 1], (uint32_t)(((t - 1) >> 1) & 1),
                                                     abort_flag, p.err, 33))) {
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll
          for (int c = 0; c < 2; ++c) {
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
        for (int c = 0; c < 32; ++c) {
          sv[c] = ex2_ftz(sv[c] - base);
          rs[c & 3] += sv[c];
        }
        l_part = l_part * alpha + ((rs[0] + rs[1]) + (rs[2] + rs[3]));
        // P buffer t & 1 was last read by the P V of tile t - 2
        if (t >= 2 && !__all_sync(0xffffffffu, wait_or_abort(&pv_done[sb], (uint32_t)(((t - 2) >> 1) & 1),
                                                           abort_flag, p.err, 34))) {
          ok = false;
          break;
        }
        uint8_t* prow = p_s + sb * atom;
#pragma unroll
        for (int ch = 0; ch < 4; ++ch) {
          uint4 v;
          v.x = pack_bf16(sv[ch * 8 + 0], sv[ch * 8 + 1]);
          v.y = pack_bf16(sv[ch * 8 + 2], sv[ch * 8 + 3]);
          v.z = pack_bf16(sv[ch * 8 + 4], sv[ch * 8 + 5]);
          v.w = pack_bf16(sv[ch * 8 + 6], sv[ch * 8 + 7]);
          *reinterpret_cast<uint4*>(prow + swz(r, chalf * 4 + ch)) = v;
        }
        if (valid < kTileK) {
          // V rows past the valid keys may hold anything (P is 0 there, but 0 * NaN is NaN)
          uint8_t* vs = kv_s + (t % S) * 2 * kTileBytes + kTileBytes;
          const int me = (chalf * W + quarter) * 32 + lane;
          for (int vr = valid + me; vr < kTileK; vr += n_sm * 32)
            for (int ch = 0; ch < 16; ++ch)
              *reinterpret_cast<uint4*>((ch < 8 ? vs : vs + kTileBytes / 2) + swz(vr, ch & 7)) =
                  make_uint4(0, 0, 0, 0);
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&p_full[sb]);
      }
      if (!ok) break;
      // hand the row max and this half's row sums to the epilogue warps; the
      // slot is free again once the epilogue of item_seq - 2 released O (the
      // MMA only started this item after that)
      float* mls = ml_s + slot * 384;
      if (chalf == 0) mls[r] = m_run;
      mls[128 * (1 + chalf) + r] = l_part;
      __syncwarp();
      if (lane == 0) mbar_arrive(&l_full[slot]);
      tile_seq += it.n_tiles;
      ++item_seq;
    }
  } else if (is_epi) {
    // ------------------------------ epilogue ------------------------------
    const int r = quarter * 32 + lane;
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    int item_seq = 0;
    while (true) {
      const int slot = item_seq & 1;
      const uint32_t par = (uint32_t)((item_seq >> 1) & 1);
      if (!__all_sync(0xffffffffu, wait_or_abort(&it_full[slot], par, abort_flag, p.err, 38))) break;
      const int item = *reinterpret_cast<volatile int*>(&ring[slot]);
      __syncwarp();
      if (lane == 0) mbar_arrive(&it_empty[slot]);
      if (item < 0) break;
      AttnItem it;
      decode_item(p, cum, item, it);
      if (!__all_sync(0xffffffffu, wait_or_abort(&l_full[slot], par, abort_flag, p.err, 39))) break;
      if (!__all_sync(0xffffffffu, wait_or_abort(&o_full[slot], par, abort_flag, p.err, 35))) break;
      tc_fence_after();
      const float* mls = ml_s + slot * 384;
      const float m_run = mls[r];
      const float l_run = mls[128 + r] + mls[256 + r];
      const bool single = (it.nsplit == 1);
      const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
      const size_t cta = ((size_t)it.b * p.Hkv + it.g) * p.max_splits + it.split;
      const uint32_t o_col = 128 + (uint32_t)(slot * attn::kD);
      for (int c = 0; c < attn::kD / 32; ++c) {
        uint32_t o[32];
        tmem_ld32(tmem_base + lane_off + o_col + c * 32, o);
        tmem_ld_wait();
        if (r < p.M) {
          if (single) {
            const int i = r / p.G, hh = r - i * p.G;
            bf16* dst = p.out + ((size_t)(it.b * p.n_q + i) * p.Hq + it.g * p.G + hh) * attn::kD + c * 32;
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
            float* dst = p.part_o + (cta * p.M + r) * attn::kD + c * 32;
#pragma unroll
            for (int q = 0; q < 32; q += 4)
              *reinterpret_cast<float4*>(dst + q) = make_float4(__uint_as_float(o[q]), __uint_as_float(o[q + 1]),
                                                                __uint_as_float(o[q + 2]), __uint_as_float(o[q + 3]));
          }
        }
      }
      if (!single && r < p.M) p.part_ml[cta * p.M + r] = make_float2(m_run, l_run);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&o_empty[slot]);
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

// Merge the split partials of every (sequence, kv head) that was split.
__global__ void __launch_bounds__(256)
attn_merge_kernel(const AttnParams p) {
  const int g = blockIdx.x, b = blockIdx.y;
  const int C = max(0, min(p.ctx_len[b], p.max_ctx));
  const int n_ctx_tiles = (C + attn_tc::kTileK - 1) / attn_tc::kTileK;
  const int nsplit = max(1, (n_ctx_tiles + attn::kTilesPerSplit - 1) / attn::kTilesPerSplit);
  if (nsplit == 1) return;
  const size_t group = (size_t)b * p.Hkv + g;
  for (int idx = threadIdx.x; idx < p.M * (attn::kD / 4); idx += blockDim.x) {
    const int row = idx / (attn::kD / 4), d4 = idx - row * (attn::kD / 4);
    float M = -CUDART_INF_F;
    for (int sp = 0; sp < nsplit; ++sp) M = fmaxf(M, p.part_ml[(group * p.max_splits + sp) * p.M + row].x);
    float L = 0.f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    if (M != -CUDART_INF_F) {
      for (int sp = 0; sp < nsplit; ++sp) {
        const size_t c2 = group * p.max_splits + sp;
        const float2 ml = p.part_ml[c2 * p.M + row];
        const float w = (ml.x == -CUDART_INF_F) ? 0.f : exp2f(ml.x - M);
        L += ml.y * w;
        const float4 v = reinterpret_cast<const float4*>(p.part_o + (c2 * p.M + row) * attn::kD)[d4];
        acc.x += v.x * w; acc.y += v.y * w; acc.z += v.z * w; acc.w += v.w * w;
      }
    }
    const float inv = L > 0.f ? 1.f / L : 0.f;
    const int i = row / p.G, hh = row - i * p.G;
    bf16* dst = p.out + ((size_t)(b * p.n_q + i) * p.Hq + g * p.G + hh) * attn::kD + d4 * 4;
    reinterpret_cast<__nv_bfloat162*>(dst)[0] = __floats2bfloat162_rn(acc.x * inv, acc.y * inv);
    reinterpret_cast<__nv_bfloat162*>(dst)[1] = __floats2bfloat162_rn(acc.z * inv, acc.w * inv);
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
                    T* __restrict__ out, int n_q, int n_kv, int Hq, int Hkv, int D, int page_size,
                    int max_pages, int num_pages, float scale) {
  constexpr int KC = 128;   // keys per chunk (one per thread)
  __shared__ float qs[256];
  __shared__ float ps[KC];
  __shared__ int rowidx[KC];
  __shared__ float red[4];
  const int i = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
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
        int phys = (lp < max_pages) ? page_table[(size_t)b * max_pages + lp] : 0;
        if (phys < 0 || phys >= num_pages) phys = 0;
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
  return a.dtype == 1 && a.D == 128 && M <= 16 * attn::kMaxWarps && a.n_kv >= 1 && a.n_kv <= attn::kTileK &&
         a.B <= attn_tc::kMaxSeqs &&
         (a.page_size == 8 || a.page_size == 16 || a.page_size == 32 || a.page_size == 64) &&
         a.num_pages * (long)a.page_size < (1L << 31) &&
         (reinterpret_cast<uintptr_t>(a.k_pool) & 15) == 0 && (reinterpret_cast<uintptr_t>(a.v_pool) & 15) == 0 &&
         (reinterpret_cast<uintptr_t>(a.q) & 15) == 0 && (reinterpret_cast<uintptr_t>(a.k_blk) & 15) == 0 &&
         (reinterpret_cast<uintptr_t>(a.v_blk) & 15) == 0 && (reinterpret_cast<uintptr_t>(a.out) & 15) == 0;
}

static int attn_max_splits(int max_ctx) {
  const int tiles = (max_ctx + attn::kTileK - 1) / attn::kTileK;
  return std::max(1, (tiles + attn::kTilesPerSplit - 1) / attn::kTilesPerSplit);
}

size_t attn_ws_bytes(int B, int n_q, int n_kv, int Hq, int Hkv, int D, int max_ctx, int dtype) {
  if (dtype != 1 || D != 128) return 0;
  const int M = n_q * (Hq / Hkv);
  const size_t ctas = (size_t)B * Hkv * attn_max_splits(max_ctx);
  return align_up(ctas * M * 128 * sizeof(float)) + align_up(ctas * M * sizeof(float2));
}

cudaError_t launch_block_attn(const AttnArgs& a, int* launches) {
  *launches = 1;
  if (!bf16_fast_ok(a)) {
    dim3 grid(a.n_q, a.Hq, a.B);
    if (a.dtype == 0)
      attn_generic_kernel<float><<<grid, 128, 0, a.stream>>>(
          (const float*)a.q, (const float*)a.k_blk, (const float*)a.v_blk, (const float*)a.k_pool,
          (const float*)a.v_pool, a.page_table, a.ctx_len, (float*)a.out, a.n_q, a.n_kv, a.Hq, a.Hkv,
          a.D, a.page_size, a.max_pages, a.num_pages, a.scale);
    else
      attn_generic_kernel<bf16><<<grid, 128, 0, a.stream>>>(
          (const bf16*)a.q, (const bf16*)a.k_blk, (const bf16*)a.v_blk, (const bf16*)a.k_pool,
          (const bf16*)a.v_pool, a.page_table, a.ctx_len, (bf16*)a.out, a.n_q, a.n_kv, a.Hq, a.Hkv,
          a.D, a.page_size, a.max_pages, a.num_pages, a.scale);
    return cudaGetLastError();
  }
  using namespace attn;
  CUtensorMap kmap, vmap;
  const uint64_t dims[3] = {(uint64_t)kD, (uint64_t)a.Hkv, (uint64_t)a.num_pages * a.page_size};
  const uint64_t strides[2] = {(uint64_t)kD * 2, (uint64_t)a.Hkv * kD * 2};
  const uint32_t box[3] = {64, 1, (uint32_t)a.page_size};
  if (!encode_tensor_map(&kmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(a.k_pool), dims,
                         strides, box, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_tensor_map(&vmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(a.v_pool), dims,
                         strides, box, CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorNotSupported;   // tensor-map encoding refused the pool layout
  AttnParams p;
  p.q = (const bf16*)a.q;
  p.k_blk = (const bf16*)a.k_blk;
  p.v_blk = (const bf16*)a.v_blk;
  p.page_table = a.page_table;
  p.ctx_len = a.ctx_len;
  p.out = (bf16*)a.out;
  p.B = a.B; p.n_q = a.n_q; p.n_kv = a.n_kv; p.Hq = a.Hq; p.Hkv = a.Hkv; p.G = a.Hq / a.Hkv;
  p.M = a.n_q * p.G;
  p.page_size = a.page_size; p.max_pages = a.max_pages; p.num_pages = a.num_pages;
  p.max_splits = attn_max_splits(a.max_ctx);
  p.max_ctx = a.max_ctx;
  p.scale_log2 = a.scale * kLog2e;
  const int M = p.M;
  const size_t ctas = (size_t)a.B * a.Hkv * p.max_splits;
  char* ws = (char*)a.scratch;
  p.part_o = (float*)ws;
  p.part_ml = (float2*)(ws + align_up(ctas * M * 128 * sizeof(float)));
  p.counters = a.counters;
  p.err = a.err;
  CUtensorMap qmap, kbmap, vbmap;
  {
    const uint64_t qd[3] = {(uint64_t)kD, (uint64_t)a.Hq, (uint64_t)a.B * a.n_q};
    const uint64_t qs[2] = {(uint64_t)kD * 2, (uint64_t)a.Hq * kD * 2};
    const uint32_t qb[3] = {64, (uint32_t)(a.Hq / a.Hkv), (uint32_t)a.n_q};
    const uint64_t bd[3] = {(uint64_t)kD, (uint64_t)a.Hkv, (uint64_t)a.B * a.n_kv};
    const uint64_t bs[2] = {(uint64_t)kD * 2, (uint64_t)a.Hkv * kD * 2};
    const uint32_t bb[3] = {64, 1, (uint32_t)a.n_kv};
    if (!encode_tensor_map(&qmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(a.q), qd, qs, qb,
                           CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_tensor_map(&kbmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(a.k_blk), bd, bs, bb,
                           CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_tensor_map(&vbmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(a.v_blk), bd, bs, bb,
                           CU_TENSOR_MAP_SWIZZLE_128B))
      return cudaErrorNotSupported;
  }
  const int Ms = M <= 64 ? 64 : 128;     // stored query rows per operand atom
  const int S = Ms == 64 ? 5 : 3;        // K/V stages that fit beside Q and P
  const size_t smem = 1024 + 6 * (size_t)Ms * 128 + (size_t)S * 2 * attn_tc::kTileBytes + attn_tc::kBarBytes;
  // warps 0-9 (two softmax quarters, producer, MMA, epilogue 8-9) or 0-13
  const bool wide = (M + 31) / 32 > 2;
  static size_t smem_set[2] = {0, 0};   // largest dynamic shared memory opted into so far
  if (smem > smem_set[wide]) {
    cudaError_t e = wide ? cudaFuncSetAttribute(attn_tc_kernel<448>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                (int)smem)
                         : cudaFuncSetAttribute(attn_tc_kernel<320>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                (int)smem);
    if (e != cudaSuccess) return e;
    smem_set[wide] = smem;
  }
  if (wide)
    attn_tc_kernel<448><<<attn_tc::kGrid, 448, smem, a.stream>>>(kmap, vmap, qmap, kbmap, vbmap, p, Ms, S, a.sched);
  else
    attn_tc_kernel<320><<<attn_tc::kGrid, 320, smem, a.stream>>>(kmap, vmap, qmap, kbmap, vbmap, p, Ms, S, a.sched);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if (p.max_splits > 1) {
    attn_merge_kernel<<<dim3(a.Hkv, a.B), 256, 0, a.stream>>>(p);
    *launches = 2;
  }
  return cudaGetLastError();
}

}  // namespace dflash
