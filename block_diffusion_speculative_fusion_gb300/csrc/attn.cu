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
  return a.dtype == 1 && a.D == 128 && M <= 16 * attn::kMaxWarps && a.n_kv <= attn::kTileK &&
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

cudaError_t launch_block_attn(const AttnArgs& a) {
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
  const int nwarps = (M + 15) / 16;
  const size_t smem = 1024 + kStages * 2 * kTileBytes + kStages * 8;
  static size_t smem_set = 0;   // largest dynamic shared memory opted into so far
  if (smem > smem_set) {
    cudaError_t e = cudaFuncSetAttribute(attn_bf16_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    smem_set = smem;
  }
  dim3 grid(p.max_splits, a.Hkv, a.B);
  attn_bf16_kernel<<<grid, nwarps * 32, smem, a.stream>>>(kmap, vmap, p);
  return cudaGetLastError();
}

}  // namespace dflash
