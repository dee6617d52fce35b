// Target-context KV materialisation.
//   DFlash page, KV 注入 step 2: h_ctx = W_f [h_l1; ...; h_lm] + b_f
//   DFlash page, KV 注入 step 3: K^(l) = h_ctx W_K^(l), V^(l) = h_ctx W_V^(l)
//   SGLang page, 4.1: kv_proj, k_norm, k_rope(positions), then a prefix-valid
//     write of the first commit_len rows of each sequence; 5.1: position ->
//     KV slot through the request's page table.
//
// Pipeline (one stream, no host synchronisation; the number of committed rows
// is known only on the device):
//   plan      1 CTA: prefix sum of commit_len -> compact row list, new_len
//   gather    committed hidden rows -> a dense [T, m*d] operand
//   GEMM 1    partial sums of H W_f^T (split over K)
//   bias      h_ctx = sum of partials + b_f, rounded to the I/O type
//   GEMM 2    partial sums of h_ctx W_kv^T for all L layers at once
//   epilogue  per token: sum partials, k_norm, RoPE, cast, paged write
// GEMMs run on tcgen05 tensor cores for bf16 (gemm_tc.cu) and on CUDA cores
// for fp32 or shapes the tensor-core kernel does not take.
#include <algorithm>
#include <cmath>

#include "common.cuh"
#include "internal.h"

namespace dflash {

// RoPE frequencies theta^(-2i/D) for i < D/2, computed on the host in double
// and passed by value (D <= 256)
struct RopeFreq {
  double f[128];
};

// ---------------------------------------------------------------------------
// gather: committed rows hidden[b, j, :] -> a dense X[t, :], t in prefix order
// of the sequences. Every CTA forms the prefix of commit_len itself (threads
// own contiguous runs of sequences, then one block scan), so no separate plan
// launch is needed; CTA 0 also writes the plan the later kernels read (T, the
// GEMMs' k-block ranges) and new_len. Rows go one per CTA pass, 256 threads x
// 16-byte vectors, ten loads in flight per thread. The same pass records each
// row's sequence, index, pool slot and RoPE (cos, sin) coefficients.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256)
mat_gather_kernel(const int32_t* __restrict__ commit_len, const int32_t* __restrict__ start_pos, int B,
                  int rows_max, const uint8_t* __restrict__ hidden, uint8_t* __restrict__ X, size_t row_bytes,
                  int32_t* __restrict__ meta, int32_t* __restrict__ row_b, int32_t* __restrict__ row_j,
                  int32_t* __restrict__ new_len, int tc, int N1, int K1, int N2, int K2,
                  const __grid_constant__ RopeFreq inv_freq, float2* __restrict__ rope, int half,
                  const int32_t* __restrict__ page_table, int page_size, int max_pages, int num_pages,
                  long long* __restrict__ slots, int* __restrict__ err) {
  dependents_may_launch();   // the GEMM that follows may be scheduled (it waits for this grid)
  __shared__ int scan[256];
  __shared__ int run_start[257];
  const int tid = threadIdx.x;
  const int per = (B + 255) / 256;
  const int b0 = tid * per, b1 = min(B, b0 + per);
  int local = 0;
  for (int b = b0; b < b1; ++b) local += max(0, min(commit_len[b], rows_max));
#ifdef DFLASH_DEBUG
  // commit lengths outside [0, rows_max] are clamped; debug builds record them
  if (blockIdx.x == 0)
    for (int b = b0; b < b1; ++b)
      if (commit_len[b] < 0 || commit_len[b] > rows_max) record_dev_error(err, kDevErrBadCommitLen);
#else
  (void)err;
#endif
  scan[tid] = local;
  __syncthreads();
  for (int off = 1; off < 256; off <<= 1) {
    const int v = tid >= off ? scan[tid - off] : 0;
    __syncthreads();
    scan[tid] += v;
    __syncthreads();
  }
  run_start[tid] = scan[tid] - local;
  if (tid == 255) run_start[256] = scan[255];
  __syncthreads();
  const int T = run_start[256];
  if (blockIdx.x == 0) {
    if (tid == 0) {
      meta[0] = T;
      // tensor-core GEMMs: k-block range per persistent CTA for T rows (0: fixed splits)
      meta[1] = tc ? gemm_tc_per(T, N1, K1) : 0;
      meta[2] = tc ? gemm_tc_per(T, N2, K2) : 0;
    }
    if (new_len)
      for (int b = b0; b < b1; ++b) new_len[b] = start_pos[b] + max(0, min(commit_len[b], rows_max));
  }
  const bool vec = (row_bytes % 16) == 0 && (reinterpret_cast<uintptr_t>(hidden) & 15) == 0 &&
                   (reinterpret_cast<uintptr_t>(X) & 15) == 0;
  const long nvec = (long)(row_bytes / 16);
  for (int r = blockIdx.x; r < T; r += gridDim.x) {
    // the sequence of row r: the last run starting at or before r, then its sequences
    int lo = 0, hi = 255;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (run_start[mid] <= r) lo = mid; else hi = mid - 1;
    }
    int b = lo * per, j = r - run_start[lo];
    for (const int be = min(B, b + per) - 1; b < be; ++b) {
      const int n = max(0, min(commit_len[b], rows_max));
      if (j < n) break;
      j -= n;
    }
    const uint8_t* src = hidden + ((size_t)b * rows_max + j) * row_bytes;
    uint8_t* dst = X + (size_t)r * row_bytes;
    if (vec) {
      constexpr int U = 10;
      for (long v0 = 0; v0 < nvec; v0 += U * 256) {
        uint4 val[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const long v = v0 + u * 256 + tid;
          if (v < nvec) val[u] = __ldg(reinterpret_cast<const uint4*>(src) + v);
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const long v = v0 + u * 256 + tid;
          if (v < nvec) reinterpret_cast<uint4*>(dst)[v] = val[u];
        }
      }
    } else {
      for (size_t e = tid; e < row_bytes; e += 256) dst[e] = src[e];
    }
    const int pos = start_pos[b] + j;
    if (tid == 0) {
      row_b[r] = b;
      row_j[r] = j;
      // the pool slot of the row (-1: position outside the page table)
      const int lp = pos / page_size;
      long long sl = -1;
      if (pos >= 0 && lp < max_pages) {
        const int phys = page_table[(size_t)b * max_pages + lp];
        if (phys >= 0 && phys < num_pages) sl = (long long)phys * page_size + pos % page_size;
      }
      slots[r] = sl;
#ifdef DFLASH_DEBUG
      // a committed row without a pool slot is not written; debug builds record it
      if (sl < 0) record_dev_error(err, kDevErrBadPosition);
#endif
    }
    // RoPE (cos, sin) of the row's position, pair i: the angle pos * theta^(-2i/D)
    // in double (it reaches ~1e4 radians), reduced to [-pi, pi] by Cody-Waite
    // subtraction of k * 2 pi with 2 pi split into a double and its remainder,
    // then sin/cos in fp32 on the reduced angle
    if (rope)
      for (int i = tid; i < half; i += 256) {
        const double a = (double)pos * inv_freq.f[i];
        const double k = rint(a * 0.15915494309189535);
        double rr = fma(-k, 6.283185307179586, a);
        rr = fma(-k, 2.4492935982947064e-16, rr);
        float sf, cf;
        sincosf((float)rr, &sf, &cf);
        rope[(size_t)r * half + i] = make_float2(cf, sf);
      }
  }
}

// ---------------------------------------------------------------------------
// CUDA-core GEMM: part[s][t][n] = sum_{k in split s} X[t][k] W[n][k]
// 64 x 64 output tile per CTA, 4 x 4 per thread, K steps of 16.
// ---------------------------------------------------------------------------
template <typename T>
__global__ void __launch_bounds__(256)
gemm_simt_kernel(const T* __restrict__ X, const T* __restrict__ W, float* __restrict__ part,
                 const int32_t* __restrict__ meta, int T_max, int N, int K, int k_per_split) {
  wait_for_prior_grid();   // a dependent launch: the rows come from the kernel before
  dependents_may_launch();
  __shared__ float As[16][68];
  __shared__ float Bs[16][68];
  const int n0 = blockIdx.x * 64, t0 = blockIdx.y * 64, s = blockIdx.z;
  const int Tv = min(meta[0], T_max);
  if (t0 >= Tv) return;
  const int k_begin = s * k_per_split, k_end = min(K, k_begin + k_per_split);
  const int tid = threadIdx.x, ty = tid >> 4, tx = tid & 15;
  float acc[4][4] = {};
  const int lr = tid >> 2, lk = (tid & 3) * 4;
  for (int k0 = k_begin; k0 < k_end; k0 += 16) {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int k = k0 + lk + q;
      const int tr = t0 + lr, nr = n0 + lr;
      As[lk + q][lr] = (tr < Tv && k < k_end) ? to_f32(X[(size_t)tr * K + k]) : 0.f;
      Bs[lk + q][lr] = (nr < N && k < k_end) ? to_f32(W[(size_t)nr * K + k]) : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int k = 0; k < 16; ++k) {
      float a[4], bb[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) { a[i] = As[k][ty * 4 + i]; bb[i] = Bs[k][tx * 4 + i]; }
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], bb[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int t = t0 + ty * 4 + i;
    if (t >= Tv) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int n = n0 + tx * 4 + j;
      if (n < N) part[((size_t)s * T_max + t) * N + n] = acc[i][j];
    }
  }
}

// ---------------------------------------------------------------------------
// h_ctx = sum of split partials + b_f, rounded to the I/O type
// ---------------------------------------------------------------------------
template <typename T>
__global__ void __launch_bounds__(256)
mat_bias_kernel(const float* __restrict__ part, int splits, const T* __restrict__ b_f, T* __restrict__ h,
                const int32_t* __restrict__ meta, int T_max, int d, int K1) {
  wait_for_prior_grid();   // a dependent launch: the partial sums come from the GEMM before
  dependents_may_launch();
  // grid-stride over the committed rows only; 4 consecutive features per
  // thread (d % 4 == 0: they share one output tile, hence one segment count)
  const int d4 = d / 4;
  const long Tn = (long)min(meta[0], T_max) * d4;
  const SegRule rule = seg_rule(d, K1, meta[1], splits, min(meta[0], T_max));
  const long stride = (long)gridDim.x * blockDim.x;
  // two items of 4 features per thread, two segments a pass: four loads in flight
  constexpr int U = 2;
  for (long idx = blockIdx.x * (long)blockDim.x + threadIdx.x; idx < Tn; idx += U * stride) {
    float4 v[U];
    int segs[U];
    int smax = 0;
#pragma unroll
    for (int k = 0; k < U; ++k) {
      const long i = idx + k * stride;
      v[k] = make_float4(0.f, 0.f, 0.f, 0.f);
      segs[k] = 0;
      if (i < Tn) {
        const int t = (int)(i / d4), f = 4 * (int)(i - (long)t * d4);
        if (b_f) v[k] = make_float4(to_f32(b_f[f]), to_f32(b_f[f + 1]), to_f32(b_f[f + 2]), to_f32(b_f[f + 3]));
        segs[k] = seg_count(rule, t, f);
        smax = max(smax, segs[k]);
      }
    }
    for (int s = 0; s < smax; s += 2) {
      float4 x[2][U];
#pragma unroll
      for (int k = 0; k < U; ++k) {
        const long i = idx + k * stride;
        const int t = (int)(i / d4), f = 4 * (int)(i - (long)t * d4);
#pragma unroll
        for (int q = 0; q < 2; ++q)
          if (s + q < segs[k]) x[q][k] = *reinterpret_cast<const float4*>(part + ((size_t)(s + q) * T_max + t) * d + f);
      }
#pragma unroll
      for (int q = 0; q < 2; ++q)
#pragma unroll
        for (int k = 0; k < U; ++k)
          if (s + q < segs[k]) {
            v[k].x += x[q][k].x; v[k].y += x[q][k].y; v[k].z += x[q][k].z; v[k].w += x[q][k].w;
          }
    }
#pragma unroll
    for (int k = 0; k < U; ++k) {
      const long i = idx + k * stride;
      if (i < Tn) {
        const int t = (int)(i / d4), f = 4 * (int)(i - (long)t * d4);
        T* o = h + (size_t)t * d + f;
        o[0] = from_f32<T>(v[k].x); o[1] = from_f32<T>(v[k].y); o[2] = from_f32<T>(v[k].z); o[3] = from_f32<T>(v[k].w);
      }
    }
  }
}

// ---------------------------------------------------------------------------
// epilogue: one warp per (committed token, layer, K|V, kv head) vector of D
// values, grid-stride. K: RMSNorm over D, then rotate-half RoPE at the token's
// absolute position (cos/sin table from the gather kernel); then the cast and
// the paged write.
// ---------------------------------------------------------------------------
// D = 128 fast path: lane l owns elements 4l .. 4l + 3 of the vector (one float4
// of each partial sum), the RoPE partner d + 64 of lane l < 16 sits in lane l + 16
// and is fetched by a shuffle; stores are 8 bytes per lane.
template <typename T>
__device__ __forceinline__ void store4(T* dst, float4 v);
template <>
__device__ __forceinline__ void store4<float>(float* dst, float4 v) {
  *reinterpret_cast<float4*>(dst) = v;
}
template <>
__device__ __forceinline__ void store4<bf16>(bf16* dst, float4 v) {
  uint2 u;
  __nv_bfloat162 a = __floats2bfloat162_rn(v.x, v.y), b = __floats2bfloat162_rn(v.z, v.w);
  u.x = *reinterpret_cast<uint32_t*>(&a);
  u.y = *reinterpret_cast<uint32_t*>(&b);
  *reinterpret_cast<uint2*>(dst) = u;
}

// One unit = (committed token t, layer l, K or V, up to kEpiHeads kv heads): the
// heads' partial-sum vectors are all loaded before any is finished, and the
// token's RoPE coefficients and the layer's norm weights are loaded once for them.
constexpr int kEpiHeads = 8;

constexpr int kEpiCtasPerSm = 2;   // 104 registers a thread

template <typename T>
__global__ void __launch_bounds__(256, kEpiCtasPerSm)
mat_epilogue_d128_kernel(const float* __restrict__ part, int splits, const int32_t* __restrict__ meta,
                         const long long* __restrict__ slots, const T* __restrict__ k_norm_w, float rms_eps,
                         const float2* __restrict__ rope, MatPools pools, int T_max, int L, int Hkv, int K2) {
  wait_for_prior_grid();   // a dependent launch: the partial sums come from the GEMM before
  dependents_may_launch();
  constexpr int D = 128, half = 64, NH = kEpiHeads;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nwarps = blockDim.x >> 5;
  const int d0 = 4 * lane;
  const int N = L * 2 * Hkv * D;
  const int Tr = min(meta[0], T_max);
  const SegRule rule = seg_rule(N, K2, meta[2], splits, Tr);
  // heads per unit: up to kEpiHeads, fewer when that leaves warps without a unit
  const long warps = (long)gridDim.x * nwarps;
  int hs = NH;
  while (hs > 1 && (long)Tr * L * 2 * ((Hkv + hs - 1) / hs) < warps) hs >>= 1;
  const int hchunks = (Hkv + hs - 1) / hs;
  const long units = (long)Tr * L * 2 * hchunks;
  for (long u = (long)blockIdx.x * nwarps + warp; u < units; u += warps) {
    long r = u;
    const int hc = (int)(r % hchunks);
    r /= hchunks;
    const int kv = (int)(r & 1);
    r >>= 1;
    const int l = (int)(r % L);
    const int t = (int)(r / L);
    const int h0 = hc * hs, nh = min(hs, Hkv - h0);
    const int v0 = (l * 2 + kv) * Hkv + h0;    // vector index of head h0: (l, K|V, h) -> features v * D
    const long long slot = slots[t];
    // a 128-wide vector lies in one 128-feature GEMM tile: one segment count each
    int segs[NH];
    int smax = 0;
#pragma unroll
    for (int i = 0; i < NH; ++i) {
      segs[i] = i < nh ? seg_count(rule, t, (v0 + i) * D) : 0;
      smax = max(smax, segs[i]);
    }
    // the first segment straight into the sums, the others (split tiles) added
    const float* src0 = part + (size_t)t * N + (size_t)v0 * D + d0;
    float4 x[NH];
#pragma unroll
    for (int i = 0; i < NH; ++i)
      x[i] = segs[i] > 0 ? *reinterpret_cast<const float4*>(src0 + i * D) : make_float4(0.f, 0.f, 0.f, 0.f);
    for (int sg = 1; sg < smax; ++sg) {
      const float* src = part + ((size_t)sg * T_max + t) * N + (size_t)v0 * D + d0;
      float4 y[NH];
#pragma unroll
      for (int i = 0; i < NH; ++i)
        if (sg < segs[i]) y[i] = *reinterpret_cast<const float4*>(src + i * D);
#pragma unroll
      for (int i = 0; i < NH; ++i)
        if (sg < segs[i]) {
          x[i].x += y[i].x; x[i].y += y[i].y; x[i].z += y[i].z; x[i].w += y[i].w;
        }
    }
    T* dst = (kv == 0 ? (T*)pools.k[l] : (T*)pools.v[l]) + ((size_t)slot * Hkv + h0) * D + d0;
    if (kv == 0) {
      float4 w = make_float4(1.f, 1.f, 1.f, 1.f);
      if (k_norm_w) {
        const T* wv = k_norm_w + (size_t)l * D + d0;
        w = make_float4(to_f32(wv[0]), to_f32(wv[1]), to_f32(wv[2]), to_f32(wv[3]));
      }
      float2 c0 = make_float2(1.f, 0.f), c1 = c0, c2 = c0, c3 = c0;
      if (rope) {
        const float2* c = rope + (size_t)t * half + (d0 & (half - 1));
        c0 = c[0]; c1 = c[1]; c2 = c[2]; c3 = c[3];
      }
      // RMSNorm over D then rotate-half RoPE: the partner of element d < 64 is
      // d + 64, held by lane + 16
      const float sgn = d0 < half ? -1.f : 1.f;
#pragma unroll
      for (int i = 0; i < NH; ++i) {
        float4 a = x[i];
        if (k_norm_w) {
          float ss = a.x * a.x + a.y * a.y + a.z * a.z + a.w * a.w;
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
          const float sc = 1.f / sqrtf(ss / D + rms_eps);
          a = make_float4(a.x * (sc * w.x), a.y * (sc * w.y), a.z * (sc * w.z), a.w * (sc * w.w));
        }
        if (rope) {
          float4 y;
          y.x = __shfl_xor_sync(0xffffffffu, a.x, 16);
          y.y = __shfl_xor_sync(0xffffffffu, a.y, 16);
          y.z = __shfl_xor_sync(0xffffffffu, a.z, 16);
          y.w = __shfl_xor_sync(0xffffffffu, a.w, 16);
          a = make_float4(a.x * c0.x + sgn * y.x * c0.y, a.y * c1.x + sgn * y.y * c1.y,
                          a.z * c2.x + sgn * y.z * c2.y, a.w * c3.x + sgn * y.w * c3.y);
        }
        if (i < nh && slot >= 0) store4<T>(dst + i * D, a);
      }
    } else if (slot >= 0) {
#pragma unroll
      for (int i = 0; i < NH; ++i)
        if (i < nh) store4<T>(dst + i * D, x[i]);
    }
  }
}

template <typename T>
__global__ void __launch_bounds__(256)
mat_epilogue_kernel(const float* __restrict__ part, int splits, const int32_t* __restrict__ meta,
                    const int32_t* __restrict__ row_b, const int32_t* __restrict__ row_j,
                    const int32_t* __restrict__ start_pos, const int32_t* __restrict__ page_table,
                    const T* __restrict__ k_norm_w, float rms_eps, const float2* __restrict__ rope, MatPools pools,
                    int T_max, int L, int Hkv, int D, int page_size, int max_pages, int num_pages, int K2) {
  wait_for_prior_grid();   // a dependent launch: the partial sums come from the GEMM before
  dependents_may_launch();
  extern __shared__ float esm[];             // [warps][D] staging
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nwarps = blockDim.x >> 5;
  float* xs = esm + warp * D;
  const int NV = L * 2 * Hkv;
  const int N = NV * D;
  const int half = D / 2;
  const SegRule rule = seg_rule(N, K2, meta[2], splits, min(meta[0], T_max));
  const long tasks = (long)min(meta[0], T_max) * NV;
  for (long task = (long)blockIdx.x * nwarps + warp; task < tasks; task += (long)gridDim.x * nwarps) {
    const int t = (int)(task / NV), v = (int)(task - (long)t * NV);
    const int b = row_b[t];
    const int pos = start_pos[b] + row_j[t];
    const int lp = pos / page_size;
    if (pos < 0 || lp >= max_pages) continue;
    const int phys = page_table[(size_t)b * max_pages + lp];
    if (phys < 0 || phys >= num_pages) continue;
    const size_t slot = (size_t)phys * page_size + pos % page_size;
    const int h = v % Hkv, kv = (v / Hkv) & 1, l = v / (2 * Hkv);
    const int n0 = v * D;                    // column of (l, kv, h) in [L, 2, Hkv*D]
    float ss = 0.f;
    for (int d = lane; d < D; d += 32) {
      float x = 0.f;
      const int segs = seg_count(rule, t, n0 + d);
      for (int s = 0; s < segs; ++s) x += part[((size_t)s * T_max + t) * N + n0 + d];
      xs[d] = x;
      ss += x * x;
    }
    __syncwarp();
    T* dst = (kv == 0 ? (T*)pools.k[l] : (T*)pools.v[l]) + (slot * Hkv + h) * D;
    if (kv == 1) {
      for (int d = lane; d < D; d += 32) dst[d] = from_f32<T>(xs[d]);
      __syncwarp();
      continue;
    }
    float scale = 1.f;
    if (k_norm_w) {
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
      scale = 1.f / sqrtf(ss / D + rms_eps);
    }
    for (int d = lane; d < D; d += 32) {
      float x = xs[d] * scale;
      if (k_norm_w) x *= to_f32(k_norm_w[(size_t)l * D + d]);
      if (rope) {
        const int i = d < half ? d : d - half;
        const int dp = d < half ? d + half : d - half;
        float y = xs[dp] * scale;
        if (k_norm_w) y *= to_f32(k_norm_w[(size_t)l * D + dp]);
        const float2 c = rope[(size_t)t * half + i];
        x = d < half ? x * c.x - y * c.y : x * c.x + y * c.y;
      }
      dst[d] = from_f32<T>(x);
    }
    __syncwarp();
  }
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
MatPlan mat_plan(int B, int rows_max, int m, int d, int L, int Hkv, int D, int dtype) {
  MatPlan p;
  p.B = B;
  p.T_max = B * rows_max;
  p.K1 = m * d;
  p.N1 = d;
  p.K2 = d;
  p.N2 = L * 2 * Hkv * D;
  p.tc = dtype == 1 && gemm_tc_supported(p.K1, p.N1) && gemm_tc_supported(p.K2, p.N2);
  if (p.tc) {
    p.S1 = gemm_tc_splits(p.T_max, p.N1, p.K1);
    p.S2 = gemm_tc_splits(p.T_max, p.N2, p.K2);
  } else {
    p.S1 = std::max(1, std::min(8, (p.K1 + 4095) / 4096));
    p.S2 = std::max(1, std::min(8, (p.K2 + 4095) / 4096));
  }
  return p;
}

size_t mat_ws_bytes(const MatPlan& p, int dtype) {
  const size_t el = dtype == 1 ? 2 : 4;
  const size_t Nmax = std::max(p.N1, p.N2);
  size_t s = align_up(sizeof(int32_t) * (64 + 2 * (size_t)p.T_max + p.B + 1));
  s += align_up(sizeof(float2) * (size_t)p.T_max * 128);   // RoPE (cos, sin) per committed row
  s += align_up(sizeof(long long) * (size_t)p.T_max);       // pool slot per committed row
  s += align_up((size_t)p.T_max * p.K1 * el);     // gathered operand X
  s += align_up((size_t)p.T_max * p.N1 * el);     // h_ctx
  s += align_up((size_t)std::max(p.S1, p.S2) * p.T_max * Nmax * sizeof(float));
  return s;
}

template <typename T>
static cudaError_t run_gemm(const MatPlan& p, bool tc, const void* X, const void* W, float* part,
                            const int32_t* meta, int N, int K, int S, int per_idx, int* err, cudaStream_t st) {
  if (tc) return launch_gemm_tc(X, W, part, meta, p.T_max, N, K, per_idx, err, st);
  const int kps = ((K + S - 1) / S + 15) / 16 * 16;
  dim3 grid((N + 63) / 64, (p.T_max + 63) / 64, S);
  cudaError_t e = launch_dependent(gemm_simt_kernel<T>, grid, dim3(256), 0, st, (const T*)X, (const T*)W, part, meta,
                                   p.T_max, N, K, kps);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

template <typename T>
static cudaError_t launch_mat_t(const MatArgs& a, int* launches) {
  const MatPlan p = mat_plan(a.B, a.rows_max, a.m, a.d, a.L, a.Hkv, a.D, a.dtype);
  const size_t el = sizeof(T);
  char* ws = (char*)a.scratch;
  int32_t* meta = (int32_t*)ws;
  int32_t* row_b = meta + 64;
  int32_t* row_j = row_b + p.T_max;
  ws += align_up(sizeof(int32_t) * (64 + 2 * (size_t)p.T_max + p.B + 1));
  RopeFreq inv_freq;
  for (int i = 0; i < 128; ++i)
    inv_freq.f[i] = i < a.D / 2 && a.rope_theta > 0.f ? std::exp(-(2.0 * i / a.D) * std::log((double)a.rope_theta)) : 0.0;
  float2* rope = a.rope_theta > 0.f ? (float2*)ws : nullptr;
  ws += align_up(sizeof(float2) * (size_t)p.T_max * 128);
  long long* slots = (long long*)ws;
  ws += align_up(sizeof(long long) * (size_t)p.T_max);
  T* X = (T*)ws;
  ws += align_up((size_t)p.T_max * p.K1 * el);
  T* h = (T*)ws;
  ws += align_up((size_t)p.T_max * p.N1 * el);
  float* part = (float*)ws;
  cudaStream_t st = a.stream;
  int n = 0;
  const size_t row_bytes = (size_t)p.K1 * el;
  // grid-stride kernels over the committed rows: a few waves of the 152 SMs
  const int gs = 4 * 152;
  mat_gather_kernel<<<gs, 256, 0, st>>>(a.commit_len, a.start_pos, a.B, a.rows_max, (const uint8_t*)a.hidden,
                                        (uint8_t*)X, row_bytes, meta, row_b, row_j, a.new_len, p.tc ? 1 : 0, p.N1,
                                        p.K1, p.N2, p.K2, inv_freq, rope, a.D / 2, a.page_table, a.page_size,
                                        a.max_pages, a.num_pages, slots, a.err);
  ++n;
  cudaError_t e = run_gemm<T>(p, p.tc, X, a.W_f, part, meta, p.N1, p.K1, p.S1, 1, a.err, st);
  if (e != cudaSuccess) return e;
  ++n;
  e = launch_dependent(mat_bias_kernel<T>, dim3(gs), dim3(256), 0, st, part, p.S1, (const T*)a.b_f, h, meta, p.T_max,
                       p.N1, p.K1);
  if (e != cudaSuccess) return e;
  ++n;
  e = run_gemm<T>(p, p.tc, h, a.W_kv, part, meta, p.N2, p.K2, p.S2, 2, a.err, st);
  if (e != cudaSuccess) return e;
  ++n;
  if (a.D == 128) {
    e = launch_dependent(mat_epilogue_d128_kernel<T>, dim3(kEpiCtasPerSm * 152), dim3(256), 0, st, part, p.S2, meta,
                         slots, (const T*)a.k_norm_w, a.rms_eps, rope, a.pools, p.T_max, a.L, a.Hkv, p.K2);
  } else {
    const size_t esmem = sizeof(float) * 8 * (size_t)a.D;
    e = launch_dependent(mat_epilogue_kernel<T>, dim3(gs), dim3(256), esmem, st, part, p.S2, meta, row_b, row_j,
                         a.start_pos, a.page_table, (const T*)a.k_norm_w, a.rms_eps, rope, a.pools, p.T_max, a.L,
                         a.Hkv, a.D, a.page_size, a.max_pages, a.num_pages, p.K2);
  }
  if (e != cudaSuccess) return e;
  ++n;
  *launches = n;
  return cudaGetLastError();
}

cudaError_t launch_materialize(const MatArgs& a, int* launches) {
  return a.dtype == 0 ? launch_mat_t<float>(a, launches) : launch_mat_t<bf16>(a, launches);
}

}  // namespace dflash
