// Vocabulary-wide verify and gate kernels: greedy rule, sampled rule with
// residual resample, and the DLoop block gate.
//
// Every kernel streams each logit exactly once with 16-byte loads (HBM bound),
// splitting rows into chunks so that small batches still cover every SM. The
// per-sequence decision is fused into the same launch: the last CTA of a
// sequence (completion ticket, no spinning) combines the chunk partials.
//
//   greedy rule  -- SGLang DFlash engineering page, section 3 (accept rule code)
//   sampled rule -- speculative-decoding page, sections 3 (min(1, p/q) and the
//                   residual max(0, p - q) / (1 - beta)) and 4 (cascade discard)
//   gate         -- DLoop page, mechanism 1 (c_s = sum log p_draft(x_i) >= g)
#include "common.cuh"
#include "internal.h"

namespace dflash {

constexpr int kThreads = 256;
constexpr int kMaxRows = 256;    // n_max + 1 limit (drafts per verify <= 255)

// Visit elements [e0, e1) of row z: 16-byte vectors in the aligned middle,
// scalars at both ends. fv(f, first_index) gets N unpacked values, fs(v, i) one.
template <typename T, int UNROLL, typename FV, typename FS>
__device__ __forceinline__ void for_range(const T* z, int e0, int e1, FV&& fv, FS&& fs) {
  constexpr int N = VecTraits<T>::N;
  const uintptr_t addr = reinterpret_cast<uintptr_t>(z + e0);
  int head = (int)(((16u - (unsigned)(addr & 15u)) & 15u) / sizeof(T));
  head = min(head, e1 - e0);
  const int a = e0 + head;
  const int nvec = (e1 - a) / N;
  const int b = a + nvec * N;
  for (int e = e0 + (int)threadIdx.x; e < a; e += blockDim.x) fs(ld_scalar(z + e), e);
  for (int e = b + (int)threadIdx.x; e < e1; e += blockDim.x) fs(ld_scalar(z + e), e);
  const uint4* vp = reinterpret_cast<const uint4*>(z + a);
  int v = threadIdx.x;
  for (; v + (UNROLL - 1) * (int)blockDim.x < nvec; v += UNROLL * blockDim.x) {
    uint4 r[UNROLL];
#pragma unroll
    for (int u = 0; u < UNROLL; ++u) r[u] = ld_stream16(vp + v + u * blockDim.x);
#pragma unroll
    for (int u = 0; u < UNROLL; ++u) {
      float f[N];
      unpack16<T>(r[u], f);
      fv(f, a + (v + u * (int)blockDim.x) * N);
    }
  }
  for (; v < nvec; v += blockDim.x) {
    float f[N];
    unpack16<T>(ld_stream16(vp + v), f);
    fv(f, a + v * N);
  }
}

// ---------------------------------------------------------------------------
// Block reductions (deterministic tree order)
// ---------------------------------------------------------------------------
__device__ __forceinline__ VI block_vi(VI x) {
  __shared__ VI sh[kThreads / 32];
  x = warp_vi(x);
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  __syncthreads();
  if (l == 0) sh[w] = x;
  __syncthreads();
  if (w == 0) {
    x = (l < (int)(blockDim.x >> 5)) ? sh[l] : VI{-CUDART_INF_F, INT32_MAX};
    x = warp_vi(x);
  }
  return x;  // valid in thread 0
}

__device__ __forceinline__ MS block_ms(MS x, float k2) {
  __shared__ MS sh[kThreads / 32];
  x = warp_ms(x, k2);
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  __syncthreads();
  if (l == 0) sh[w] = x;
  __syncthreads();
  if (w == 0) {
    x = (l < (int)(blockDim.x >> 5)) ? sh[l] : MS{-CUDART_INF_F, 0.f};
    x = warp_ms(x, k2);
  }
  return x;  // valid in thread 0
}

// 2^x on the special-function unit, flushing denormal results to zero (terms
// below 2^-126 of a row maximum do not change a sum that contains 1).
__device__ __forceinline__ float ex2_ftz(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Streaming (max, sum exp2((z - max) * k2)) of elements [e0, e1) of one row.
// The same code serves target and draft rows, so identical rows give
// bit-identical statistics.
template <typename T>
__device__ __forceinline__ MS row_chunk_ms(const T* z, int e0, int e1, float k2) {
  constexpr int N = VecTraits<T>::N;
  MS acc{-CUDART_INF_F, 0.f};
  auto add_vec = [&](const float* f, int) {
    float vm = f[0];
#pragma unroll
    for (int j = 1; j < N; ++j) vm = fmaxf(vm, f[j]);
    if (vm > acc.m) {
      acc.s = (acc.m == -CUDART_INF_F) ? 0.f : acc.s * exp2f((acc.m - vm) * k2);
      acc.m = vm;
    }
    if (acc.m == -CUDART_INF_F) return;
    float s = 0.f;
#pragma unroll
    for (int j = 0; j < N; ++j) s += ex2_ftz((f[j] - acc.m) * k2);
    acc.s += s;
  };
  auto add_one = [&](float v, int) {
    if (v > acc.m) {
      acc.s = (acc.m == -CUDART_INF_F) ? 0.f : acc.s * exp2f((acc.m - v) * k2);
      acc.m = v;
    }
    if (acc.m != -CUDART_INF_F) acc.s += ex2_ftz((v - acc.m) * k2);
  };
  for_range<T, 4>(z, e0, e1, add_vec, add_one);
  return block_ms(acc, k2);
}

// ===========================================================================
// Greedy rule
// ===========================================================================
template <typename T>
__global__ void __launch_bounds__(kThreads)
greedy_kernel(const T* __restrict__ logits, const int64_t* __restrict__ cand,
              const int32_t* __restrict__ n_draft, int R, int V, int nch, int chunk,
              VI* __restrict__ parts, int32_t* __restrict__ counters,
              int32_t* __restrict__ accept_len, int64_t* __restrict__ bonus,
              int32_t* __restrict__ commit_len, int64_t* __restrict__ out_tokens,
              int64_t* __restrict__ target_pred) {
  const int c = blockIdx.x;
  const int row = blockIdx.y;
  const int b = row / R, i = row - b * R;
  const int nb = n_draft ? n_draft[b] : R - 1;
  VI best{-CUDART_INF_F, INT32_MAX};
  if (i <= nb) {
    const T* z = logits + (size_t)row * V;
    const int e0 = c * chunk, e1 = min(V, e0 + chunk);
    constexpr int N = VecTraits<T>::N;
    auto on_vec = [&](const float* f, int i0) {
#pragma unroll
      for (int j = 0; j < N; ++j)
        if (vi_better(f[j], i0 + j, best)) best = VI{f[j], i0 + j};
    };
    auto on_one = [&](float v, int e) {
      if (vi_better(v, e, best)) best = VI{v, e};
    };
    for_range<T, 4>(z, e0, e1, on_vec, on_one);
    best = block_vi(best);
  }
  if (threadIdx.x == 0) parts[(size_t)row * nch + c] = best;
  if (!take_ticket_is_last_t0(&counters[b], R * nch)) return;

  // ---- last CTA of sequence b: argmax per row, then the accept rule ----
  __shared__ int32_t tp[kMaxRows];
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  for (int r = w; r <= nb; r += blockDim.x >> 5) {
    VI x{-CUDART_INF_F, INT32_MAX};
    const VI* pr = parts + ((size_t)b * R + r) * nch;
    for (int cc = l; cc < nch; cc += 32) {
      const int2 raw = __ldcg(reinterpret_cast<const int2*>(pr + cc));
      const VI y{__int_as_float(raw.x), raw.y};
      if (vi_better(y.v, y.i, x)) x = y;
    }
    x = warp_vi(x);
    if (l == 0) tp[r] = (x.i == INT32_MAX) ? 0 : x.i;
  }
  __syncthreads();
  __shared__ int s_acc;
  if (threadIdx.x == 0) {
    const int64_t* cb = cand + (size_t)b * R;
    int a = 0;
    while (a < nb && cb[a + 1] == (int64_t)tp[a]) ++a;   // cumulative product of matches
    s_acc = a;
    accept_len[b] = a;
    commit_len[b] = a + 1;
    bonus[b] = tp[a];
  }
  __syncthreads();
  const int a = s_acc;
  for (int r = threadIdx.x; r < R; r += blockDim.x) {
    if (out_tokens)
      out_tokens[(size_t)b * R + r] = r < a ? cand[(size_t)b * R + r + 1] : (r == a ? (int64_t)tp[a] : -1);
    if (target_pred) target_pred[(size_t)b * R + r] = r <= nb ? (int64_t)tp[r] : -1;
  }
  reset_ticket(&counters[b]);
}

// ===========================================================================
// Sampled rule, pass 1: row statistics, then the sequential accept test
// ===========================================================================
struct SampleJob {
  int32_t row;     // target row the bonus is drawn from (= accept_len)
  int32_t mode;    // 0: residual max(0, p - q) at that row, 1: p at that row
  float mt, st;    // target row (max, scaled sum)
  float md, sd;    // draft row (max, scaled sum); unused in mode 1
  int32_t acc;
  int32_t flags;
};

template <typename T>
__global__ void __launch_bounds__(kThreads)
sample_stats_kernel(const T* __restrict__ zt, const T* __restrict__ zd,
                    const int64_t* __restrict__ cand, const int32_t* __restrict__ n_draft,
                    const float* __restrict__ u_acc, int n_max, int V, int nch, int chunk,
                    float k2, MS* __restrict__ parts, float* __restrict__ zx,
                    int32_t* __restrict__ counters, SampleJob* __restrict__ jobs,
                    int32_t* __restrict__ accept_len, int32_t* __restrict__ commit_len,
                    int64_t* __restrict__ out_tokens, float* __restrict__ probs) {
  const int R = n_max + 1;
  const int RR = R + n_max;              // target rows then draft rows of a sequence
  const int c = blockIdx.x;
  const int b = blockIdx.y / RR, r = blockIdx.y - b * RR;
  const int nb = n_draft ? n_draft[b] : n_max;
  const bool is_t = r < R;
  const int ri = is_t ? r : r - R;       // row index within its tensor
  const bool valid = is_t ? (ri <= nb) : (ri < nb);
  MS ms{-CUDART_INF_F, 0.f};
  if (valid) {
    const T* z = is_t ? zt + ((size_t)b * R + ri) * V : zd + ((size_t)b * n_max + ri) * V;
    const int e0 = c * chunk, e1 = min(V, e0 + chunk);
    ms = row_chunk_ms<T>(z, e0, e1, k2);
    if (threadIdx.x == 0 && ri < nb) {
      const int64_t x = cand[(size_t)b * R + ri + 1];
      if (x >= e0 && x < e1) zx[((size_t)b * RR + r)] = ld_scalar(z + x);
    }
  }
  if (threadIdx.x == 0) parts[((size_t)b * RR + r) * nch + c] = ms;
  if (!take_ticket_is_last_t0(&counters[b], RR * nch)) return;

  // ---- last CTA of sequence b ----
  __shared__ MS rs[2 * kMaxRows];
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  for (int rr = w; rr < RR; rr += blockDim.x >> 5) {
    const bool t = rr < R;
    const int rix = t ? rr : rr - R;
    if (t ? rix > nb : rix >= nb) continue;
    MS x{-CUDART_INF_F, 0.f};
    const MS* pr = parts + ((size_t)b * RR + rr) * nch;
    for (int cc = l; cc < nch; cc += 32) {
      const float2 raw = __ldcg(reinterpret_cast<const float2*>(pr + cc));
      x = ms_merge(x, MS{raw.x, raw.y}, k2);
    }
    // fixed-order combine across lanes
    x = warp_ms(x, k2);
    if (l == 0) rs[rr] = x;
  }
  __syncthreads();
  __shared__ int s_a;
  if (threadIdx.x == 0) {
    int a = 0, flags = 0;
    bool rejected = false;
    for (int i = 1; i <= nb; ++i) {
      const MS pt = rs[i - 1], pd = rs[R + i - 1];
      const float zxt = __ldcg(zx + (size_t)b * RR + (i - 1));
      const float zxd = __ldcg(zx + (size_t)b * RR + R + (i - 1));
      const float et = exp2f((zxt - pt.m) * k2), ed = exp2f((zxd - pd.m) * k2);
      const float px = et / pt.s, qx = ed / pd.s;
      if (probs) {
        probs[(size_t)b * (2 * n_max + 1) + (i - 1)] = px;
        probs[(size_t)b * (2 * n_max + 1) + n_max + (i - 1)] = qx;
      }
      float ratio;
      if (ed == 0.f) {
        flags |= 8;                      // DFLASH_FLAG_INVALID
        ratio = CUDART_INF_F;
      } else {
        // p/q = exp2((zt_x - mt) - (zd_x - md)) * sd / st, differences taken first
        ratio = exp2f(((zxt - pt.m) - (zxd - pd.m)) * k2) * (pd.s / pt.s);
      }
      const float u = u_acc[(size_t)b * n_max + (i - 1)];
      if (ratio < 1.f && fabsf(u - ratio) < 1e-6f) flags |= 1;   // ACCEPT_BOUNDARY
      if (u < ratio) {
        ++a;
      } else {
        rejected = true;
        break;
      }
    }
    if (probs)
      for (int i = a + (rejected ? 1 : 0) + 1; i <= n_max; ++i) {
        probs[(size_t)b * (2 * n_max + 1) + (i - 1)] = 0.f;
        probs[(size_t)b * (2 * n_max + 1) + n_max + (i - 1)] = 0.f;
      }
    SampleJob j;
    j.row = a;
    j.mode = rejected ? 0 : 1;
    j.mt = rs[a].m;
    j.st = rs[a].s;
    j.md = rejected ? rs[R + a].m : 0.f;
    j.sd = rejected ? rs[R + a].s : 1.f;
    j.acc = a;
    j.flags = flags;
    jobs[b] = j;
    accept_len[b] = a;
    commit_len[b] = a + 1;
    s_a = a;
  }
  __syncthreads();
  if (out_tokens) {
    // accepted drafts now; the bonus slot and padding are written by pass 2
    const int a = s_a;
    for (int rr = threadIdx.x; rr < a; rr += blockDim.x)
      out_tokens[(size_t)b * R + rr] = cand[(size_t)b * R + rr + 1];
  }
  reset_ticket(&counters[b]);
}

// ===========================================================================
// Sampled rule, pass 2: inverse-CDF draw of the bonus from the residual
// max(0, p - q) (or from p after a full accept), in ascending token order.
// Each thread owns one 16-byte vector of the chunk, so the CDF order is the
// token order and every thread's partial sum is recomputed identically.
// ===========================================================================
template <typename T>
__device__ __forceinline__ void resample_weights(const T* zt_row, const T* zd_row, int e0, int V,
                                                 const SampleJob& j, float k2, bool use_p,
                                                 float* wgt) {
  constexpr int N = VecTraits<T>::N;
  const float inv_st = 1.f / j.st;
  const float inv_sd = 1.f / j.sd;
#pragma unroll
  for (int q = 0; q < N; ++q) wgt[q] = 0.f;
  const int base = e0 + (int)threadIdx.x * N;
  if (base >= V) return;
  float ft[N], fd[N];
  if (base + N <= V && ((reinterpret_cast<uintptr_t>(zt_row + base) & 15u) == 0) &&
      (use_p || (reinterpret_cast<uintptr_t>(zd_row + base) & 15u) == 0)) {
    unpack16<T>(*reinterpret_cast<const uint4*>(zt_row + base), ft);
    if (!use_p) unpack16<T>(*reinterpret_cast<const uint4*>(zd_row + base), fd);
  } else {
#pragma unroll
    for (int q = 0; q < N; ++q) {
      ft[q] = base + q < V ? ld_scalar(zt_row + base + q) : -CUDART_INF_F;
      fd[q] = (!use_p && base + q < V) ? ld_scalar(zd_row + base + q) : -CUDART_INF_F;
    }
  }
#pragma unroll
  for (int q = 0; q < N; ++q) {
    const float p = exp2f((ft[q] - j.mt) * k2) * inv_st;
    if (use_p) {
      wgt[q] = p;
    } else {
      const float qq = exp2f((fd[q] - j.md) * k2) * inv_sd;
      wgt[q] = fmaxf(0.f, p - qq);
    }
  }
}

template <typename T>
__global__ void __launch_bounds__(kThreads)
sample_resample_kernel(const T* __restrict__ zt, const T* __restrict__ zd,
                       const int64_t* __restrict__ cand, const float* __restrict__ u_final,
                       int n_max, int V, int nch, float k2, const SampleJob* __restrict__ jobs,
                       float2* __restrict__ parts, int32_t* __restrict__ counters,
                       int64_t* __restrict__ bonus, int64_t* __restrict__ out_tokens,
                       uint8_t* __restrict__ flags_out, float* __restrict__ probs) {
  constexpr int N = VecTraits<T>::N;
  const int chunk = kThreads * N;
  const int c = blockIdx.x, b = blockIdx.y;
  const int R = n_max + 1;
  const SampleJob j = jobs[b];
  const T* zt_row = zt + ((size_t)b * R + j.row) * V;
  const T* zd_row = zd + ((size_t)b * n_max + min(j.row, max(n_max - 1, 0))) * V;
  const int e0 = c * chunk;
  float wr[N], wp[N];
  resample_weights<T>(zt_row, zd_row, e0, V, j, k2, j.mode == 1, wr);
  float sr = 0.f;
#pragma unroll
  for (int q = 0; q < N; ++q) sr += wr[q];
  float sp = sr;
  if (j.mode == 0) {
    resample_weights<T>(zt_row, zd_row, e0, V, j, k2, true, wp);
    sp = 0.f;
#pragma unroll
    for (int q = 0; q < N; ++q) sp += wp[q];
  }
  // block sums of the residual and of p (p is the fallback when Z == 0)
  __shared__ float shr[kThreads / 32], shp[kThreads / 32];
  float xr = sr, xp = sp;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    xr += __shfl_xor_sync(0xffffffffu, xr, o);
    xp += __shfl_xor_sync(0xffffffffu, xp, o);
  }
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  if (l == 0) { shr[w] = xr; shp[w] = xp; }
  __syncthreads();
  if (threadIdx.x == 0) {
    float tr = 0.f, tp = 0.f;
    for (int q = 0; q < (int)(blockDim.x >> 5); ++q) { tr += shr[q]; tp += shp[q]; }
    parts[(size_t)b * nch + c] = make_float2(tr, tp);
  }
  if (!take_ticket_is_last_t0(&counters[b], nch)) return;

  // ---- last CTA of sequence b: locate the chunk, then the token ----
  // Column x of the partials holds the drawn weights (residual, or p after a
  // full accept); column y holds p, used when the residual mass is zero.
  __shared__ double s_target, s_before, s_Z;
  __shared__ int s_chunk, s_degenerate;
  if (threadIdx.x == 0) {
    double Zr = 0.0, Zp = 0.0;
    for (int cc = 0; cc < nch; ++cc) {
      const float2 v = __ldcg(parts + (size_t)b * nch + cc);
      Zr += v.x;
      Zp += v.y;
    }
    const int degenerate = (j.mode == 0 && Zr == 0.0) ? 1 : 0;
    const double Z = degenerate ? Zp : Zr;
    const double target = (double)u_final[b] * Z;
    double cum = 0.0, before = 0.0;
    int cstar = -1, last_nz = 0;
    for (int cc = 0; cc < nch; ++cc) {
      const float2 v = __ldcg(parts + (size_t)b * nch + cc);
      const double sc = degenerate ? v.y : v.x;
      if (sc > 0.0) last_nz = cc;
      if (cstar < 0 && cum + sc > target) { cstar = cc; before = cum; }
      cum += sc;
    }
    if (cstar < 0) {   // rounding put the target past the last step
      cstar = last_nz;
      before = 0.0;
      for (int cc = 0; cc < last_nz; ++cc) {
        const float2 v = __ldcg(parts + (size_t)b * nch + cc);
        before += degenerate ? v.y : v.x;
      }
    }
    s_target = target;
    s_before = before;
    s_Z = Z;
    s_chunk = cstar;
    s_degenerate = degenerate;
  }
  __syncthreads();
  const bool usep = (j.mode == 1) || s_degenerate;
  const int e0s = s_chunk * chunk;
  float wv[N];
  resample_weights<T>(zt_row, zd_row, e0s, V, j, k2, usep, wv);
  double ts = 0.0;
  {
    float f = 0.f;
#pragma unroll
    for (int q = 0; q < N; ++q) f += wv[q];
    ts = f;
  }
  // exclusive scan of per-thread sums over the block, in fp64
  __shared__ double scan_sh[kThreads];
  scan_sh[threadIdx.x] = ts;
  __syncthreads();
  for (int off = 1; off < (int)blockDim.x; off <<= 1) {
    const double v = (threadIdx.x >= (unsigned)off) ? scan_sh[threadIdx.x - off] : 0.0;
    __syncthreads();
    scan_sh[threadIdx.x] += v;
    __syncthreads();
  }
  const double incl = scan_sh[threadIdx.x];
  const double excl = incl - ts;
  __shared__ int s_y, s_lastpos;
  __shared__ double s_clo, s_chi;
  if (threadIdx.x == 0) { s_y = INT32_MAX; s_lastpos = -1; }
  __syncthreads();
  const double target = s_target;
  double cum = s_before + excl;
  const int base = e0s + (int)threadIdx.x * N;
  for (int q = 0; q < N; ++q) {
    if (wv[q] > 0.f) atomicMax(&s_lastpos, base + q);
  }
  if (ts > 0.0 && cum <= target && cum + ts > target) {
    for (int q = 0; q < N; ++q) {
      const double nxt = cum + (double)wv[q];
      if (nxt > target) {
        s_y = base + q;        // unique: the thread ranges are disjoint
        s_clo = cum;
        s_chi = nxt;
        break;
      }
      cum = nxt;
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int y = s_y;
    double clo, chi;
    int flags = j.flags;
    if (y == INT32_MAX) {       // rounding: fall back to the last positive weight
      y = s_lastpos >= 0 ? s_lastpos : 0;
      clo = s_target;
      chi = s_target;
    } else {
      clo = s_clo;
      chi = s_chi;
    }
    const double Z = s_Z;
    const double u = u_final[b];
    if (Z > 0.0 && (fabs(clo / Z - u) < 1e-6 || fabs(chi / Z - u) < 1e-6)) flags |= 2;  // CDF_BOUNDARY
    if (s_degenerate) flags |= 4;                                                         // DEGENERATE
    bonus[b] = y;
    if (flags_out) flags_out[b] = (uint8_t)flags;
    if (probs) probs[(size_t)b * (2 * n_max + 1) + 2 * n_max] = (float)Z;
  }
  __shared__ int64_t s_yb;
  if (threadIdx.x == 0) s_yb = bonus[b];
  if (out_tokens) {
    __syncthreads();
    const int64_t yb = s_yb;
    for (int rr = j.acc + (int)threadIdx.x; rr < R; rr += blockDim.x)
      out_tokens[(size_t)b * R + rr] = (rr == j.acc) ? yb : -1;
  }
  reset_ticket(&counters[b]);
}

// ===========================================================================
// DLoop gate
// ===========================================================================
template <typename T>
__global__ void __launch_bounds__(kThreads)
gate_kernel(const T* __restrict__ z, const int64_t* __restrict__ tokens,
            const uint8_t* __restrict__ active, int k, int V, int nch, int chunk, float k2,
            float inv_t, float g, MS* __restrict__ parts, float* __restrict__ zx,
            int32_t* __restrict__ counters, float* __restrict__ c_s, uint8_t* __restrict__ cont,
            float* __restrict__ row_lse, uint8_t* __restrict__ flags) {
  const int c = blockIdx.x;
  const int row = blockIdx.y;
  const int b = row / k, i = row - b * k;
  const bool on = active ? active[b] != 0 : true;
  MS ms{-CUDART_INF_F, 0.f};
  const bool need = on || row_lse != nullptr;
  if (need) {
    const T* zr = z + (size_t)row * V;
    const int e0 = c * chunk, e1 = min(V, e0 + chunk);
    ms = row_chunk_ms<T>(zr, e0, e1, k2);
    if (threadIdx.x == 0) {
      const int64_t x = tokens[row];
      if (x >= e0 && x < e1) zx[row] = ld_scalar(zr + x);
    }
  }
  if (threadIdx.x == 0) parts[(size_t)row * nch + c] = ms;
  if (!take_ticket_is_last_t0(&counters[b], k * nch)) return;

  __shared__ MS rs[kMaxRows];
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  if (need) {
    for (int ii = w; ii < k; ii += blockDim.x >> 5) {
      MS x{-CUDART_INF_F, 0.f};
      const MS* pr = parts + ((size_t)b * k + ii) * nch;
      for (int cc = l; cc < nch; cc += 32) {
        const float2 raw = __ldcg(reinterpret_cast<const float2*>(pr + cc));
        x = ms_merge(x, MS{raw.x, raw.y}, k2);
      }
      x = warp_ms(x, k2);
      if (l == 0) rs[ii] = x;
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    double csum = 0.0;
    for (int ii = 0; ii < k; ++ii) {
      const MS r = rs[ii];
      if (need && row_lse) row_lse[(size_t)b * k + ii] = r.m * inv_t + logf(r.s);
      if (on) {
        const float zxv = __ldcg(zx + (size_t)b * k + ii);
        // log q(x) = (z_x - max) / T - ln(sum exp((z - max) / T))
        csum += (double)((zxv - r.m) * inv_t) - (double)logf(r.s);
      }
    }
    const float cval = on ? (float)csum : 0.f;
    c_s[b] = cval;
    cont[b] = (on && csum >= (double)g) ? 1 : 0;
    if (flags) flags[b] = (on && fabs(csum - (double)g) < 1e-4) ? 1 : 0;
  }
  reset_ticket(&counters[b]);
}

// ===========================================================================
// Host launchers
// ===========================================================================
static int vec_elems(int dtype) { return dtype == 0 ? 4 : 8; }

// Chunks per row: the grid (rows x chunks) is sized to one wave of resident
// CTAs (8 per SM) so that no partial wave trails the kernel; each thread
// handles at least one 16-byte vector per chunk.
ChunkPlan plan_chunks(int rows, int V, int dtype, int num_sms) {
  const int per_thread_vec = kThreads * vec_elems(dtype);
  const int units = (V + per_thread_vec - 1) / per_thread_vec;   // vector rounds for a whole row
  const long wave = 8L * num_sms;
  long nch = wave / (rows > 0 ? rows : 1);
  if (nch < 1) nch = 1;
  if (nch > units) nch = units;
  ChunkPlan p;
  p.chunk = (int)((units + nch - 1) / nch) * per_thread_vec;
  p.nch = (V + p.chunk - 1) / p.chunk;
  return p;
}

int resample_chunks(int V, int dtype) {
  const int chunk = kThreads * vec_elems(dtype);
  return (V + chunk - 1) / chunk;
}

size_t verify_greedy_ws_bytes(int B, int n_max, int V, int dtype, int num_sms) {
  const int R = n_max + 1;
  ChunkPlan p = plan_chunks(B * R, V, dtype, num_sms);
  return (size_t)B * R * p.nch * sizeof(VI);
}

size_t verify_sample_ws_bytes(int B, int n_max, int V, int dtype, int num_sms) {
  const int RR = 2 * n_max + 1;
  ChunkPlan p = plan_chunks(B * RR, V, dtype, num_sms);
  size_t s = 0;
  s += align_up((size_t)B * RR * p.nch * sizeof(MS));             // stats partials
  s += align_up((size_t)B * RR * sizeof(float));                  // z at candidates
  s += align_up((size_t)B * sizeof(SampleJob));                   // per-sequence job
  s += align_up((size_t)B * resample_chunks(V, dtype) * sizeof(float2));
  return s;
}

size_t gate_ws_bytes(int B, int k, int V, int dtype, int num_sms) {
  ChunkPlan p = plan_chunks(B * k, V, dtype, num_sms);
  return align_up((size_t)B * k * p.nch * sizeof(MS)) + align_up((size_t)B * k * sizeof(float));
}

template <typename T>
static cudaError_t launch_greedy_t(const VerifyArgs& a, int num_sms) {
  const int R = a.n_max + 1;
  ChunkPlan p = plan_chunks(a.B * R, a.V, a.dtype, num_sms);
  dim3 grid(p.nch, a.B * R);
  greedy_kernel<T><<<grid, kThreads, 0, a.stream>>>(
      (const T*)a.target_logits, a.cand, a.n_draft, R, a.V, p.nch, p.chunk,
      (VI*)a.scratch, a.counters, a.accept_len, a.bonus, a.commit_len, a.out_tokens,
      a.target_pred);
  return cudaGetLastError();
}

cudaError_t launch_verify_greedy(const VerifyArgs& a, int num_sms) {
  return a.dtype == 0 ? launch_greedy_t<float>(a, num_sms) : launch_greedy_t<bf16>(a, num_sms);
}

template <typename T>
static cudaError_t launch_sample_t(const VerifyArgs& a, int num_sms) {
  const int R = a.n_max + 1, RR = 2 * a.n_max + 1;
  ChunkPlan p = plan_chunks(a.B * RR, a.V, a.dtype, num_sms);
  char* ws = (char*)a.scratch;
  MS* parts = (MS*)ws;
  ws += align_up((size_t)a.B * RR * p.nch * sizeof(MS));
  float* zx = (float*)ws;
  ws += align_up((size_t)a.B * RR * sizeof(float));
  SampleJob* jobs = (SampleJob*)ws;
  ws += align_up((size_t)a.B * sizeof(SampleJob));
  float2* rparts = (float2*)ws;
  const float k2 = kLog2e / a.temperature;
  dim3 g1(p.nch, a.B * RR);
  sample_stats_kernel<T><<<g1, kThreads, 0, a.stream>>>(
      (const T*)a.target_logits, (const T*)a.draft_logits, a.cand, a.n_draft, a.u_accept,
      a.n_max, a.V, p.nch, p.chunk, k2, parts, zx, a.counters, jobs, a.accept_len,
      a.commit_len, a.out_tokens, a.probs);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int nch2 = resample_chunks(a.V, a.dtype);
  dim3 g2(nch2, a.B);
  sample_resample_kernel<T><<<g2, kThreads, 0, a.stream>>>(
      (const T*)a.target_logits, (const T*)a.draft_logits, a.cand, a.u_final, a.n_max, a.V,
      nch2, k2, jobs, rparts, a.counters + a.B, a.bonus, a.out_tokens, a.flags, a.probs);
  (void)R;
  return cudaGetLastError();
}

cudaError_t launch_verify_sample(const VerifyArgs& a, int num_sms) {
  return a.dtype == 0 ? launch_sample_t<float>(a, num_sms) : launch_sample_t<bf16>(a, num_sms);
}

template <typename T>
static cudaError_t launch_gate_t(const GateArgs& a, int num_sms) {
  ChunkPlan p = plan_chunks(a.B * a.k, a.V, a.dtype, num_sms);
  char* ws = (char*)a.scratch;
  MS* parts = (MS*)ws;
  ws += align_up((size_t)a.B * a.k * p.nch * sizeof(MS));
  float* zx = (float*)ws;
  dim3 grid(p.nch, a.B * a.k);
  gate_kernel<T><<<grid, kThreads, 0, a.stream>>>(
      (const T*)a.draft_logits, a.tokens, a.active, a.k, a.V, p.nch, p.chunk,
      kLog2e / a.temperature, 1.f / a.temperature, a.g, parts, zx, a.counters, a.c_s, a.cont,
      a.row_lse, a.flags);
  return cudaGetLastError();
}

cudaError_t launch_gate(const GateArgs& a, int num_sms) {
  return a.dtype == 0 ? launch_gate_t<float>(a, num_sms) : launch_gate_t<bf16>(a, num_sms);
}

}  // namespace dflash
