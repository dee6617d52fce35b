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
#include "stream.cuh"

namespace dflash {

constexpr int kCtasPerSm = 4;    // resident CTAs per SM the streaming kernels are planned for
constexpr int kMaxRows = 256;    // n_max + 1 limit (drafts per verify <= 255)
constexpr int kMaxDrawChunks = 1024;   // vocabulary <= 1024 x 16384

// ===========================================================================
// Greedy rule
// ===========================================================================
template <typename T>
__global__ void __launch_bounds__(kThreads, kCtasPerSm)
greedy_kernel(const T* __restrict__ logits, const int64_t* __restrict__ cand,
              const int32_t* __restrict__ n_draft, int R, int V, int nch, int chunk,
              VI* __restrict__ parts, int32_t* __restrict__ counters,
              int32_t* __restrict__ accept_len, int64_t* __restrict__ bonus,
              int32_t* __restrict__ commit_len, int64_t* __restrict__ out_tokens,
              int64_t* __restrict__ target_pred, int* __restrict__ err) {
  const int c = blockIdx.x;
  const int row = blockIdx.y;
  const int b = row / R, i = row - b * R;
  // drafts of sequence b, clamped to [0, R - 1] (an out-of-range count is recorded)
  int nb = n_draft ? n_draft[b] : R - 1;
  if (nb < 0 || nb > R - 1) {
    if (c == 0 && i == 0 && threadIdx.x == 0) record_dev_error(err, kDevErrBadNDraft);
    nb = min(max(nb, 0), R - 1);
  }
  VI best{-CUDART_INF_F, INT32_MAX};
  if (i <= nb) {
    const T* z = logits + (size_t)row * V;
    const int e0 = c * chunk, e1 = min(V, e0 + chunk);
    constexpr int N = VecTraits<T>::N;
    auto on_vec = [&](const uint4& u, int i0) {
      const float vm = vec_max<T>(u);          // packed max; the index search is rare
      if (vm > best.v || (vm == best.v && i0 < best.i)) {
        float f[N];
        unpack16<T>(u, f);
#pragma unroll
        for (int j = N - 1; j >= 0; --j)
          if (f[j] == vm) best = VI{vm, i0 + j};   // ends on the lowest index
      }
    };
    auto on_one = [&](float v, int e) {
      if (vi_better(v, e, best)) best = VI{v, e};
    };
    for_range<T, 8>(z, e0, e1, on_vec, on_one);
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

struct SampleJob {
  int32_t row;     // target row the bonus is drawn from (= accept_len)
  int32_t mode;    // 0: residual max(0, p - q) at that row, 1: p at that row
  float mt, st;    // target row (max, scaled sum)
  float md, sd;    // draft row (max, scaled sum); unused in mode 1
  int32_t acc;
  int32_t flags;
};

// ===========================================================================
// Sampled rule, pass 2: inverse-CDF draw of the bonus from the residual
// max(0, p - q) (or from p after a full accept) in ascending token order:
// chunk sums, then segment sums of the chosen chunk (fp64 prefix), then a warp
// scan over the chosen 64-token segment.
// ===========================================================================
// Weights of the 16-byte vectors (t, d) at token e: residual, or p (use_p),
// and the p values themselves. Tokens past V weigh 0.
template <typename T>
__device__ __forceinline__ void pair_weights(const uint4& vt, const uint4& vd, const SampleJob& j, float k2,
                                             bool use_p, float* w, float* pv) {
  constexpr int N = VecTraits<T>::N;
  float ft[N], fd[N];
  unpack16<T>(vt, ft);
  if (!use_p) unpack16<T>(vd, fd);
  const float inv_st = 1.f / j.st, inv_sd = 1.f / j.sd;
#pragma unroll
  for (int q = 0; q < N; ++q) {
    pv[q] = ex2_ftz(fmaf(ft[q], k2, -j.mt)) * inv_st;
    w[q] = use_p ? pv[q] : fmaxf(0.f, pv[q] - ex2_ftz(fmaf(fd[q], k2, -j.md)) * inv_sd);
  }
}


// Pass 2 grid: CTA (c, b) owns tokens [c * kDrawChunk, (c + 1) * kDrawChunk) of
// sequence b's drawn row; thread t owns the contiguous segment of kDrawSeg
// tokens at c * kDrawChunk + t * kDrawSeg. The CDF order is chunk, thread, token.
constexpr int kDrawSeg = 64;                      // tokens per thread
constexpr int kDrawChunk = kThreads * kDrawSeg;   // tokens per CTA

template <typename T>
__global__ void __launch_bounds__(kThreads)
sample_draw_kernel(const T* __restrict__ zt, const T* __restrict__ zd, const float* __restrict__ u_final,
                   int n_max, int V, int nch, float k2, const SampleJob* __restrict__ jobs,
                   float2* __restrict__ parts, float2* __restrict__ segs, int32_t* __restrict__ counters,
                   int64_t* __restrict__ bonus, int64_t* __restrict__ out_tokens, uint8_t* __restrict__ flags_out,
                   float* __restrict__ probs) {
  wait_for_prior_grid();   // a dependent launch: the jobs come from the statistics kernel
  constexpr int N = VecTraits<T>::N;
  constexpr int NV = kDrawSeg / N;
  const int c = blockIdx.x, b = blockIdx.y;
  const int R = n_max + 1;
  const SampleJob j = jobs[b];
  const bool usep_r = (j.mode == 1);
  const T* zt_row = zt + ((size_t)b * R + j.row) * V;
  const T* zd_row = zd + ((size_t)b * n_max + min(j.row, max(n_max - 1, 0))) * V;
  // ---- pass 1: segment sums of the drawn weights (residual, or p) and of p ----
  // The chunk of both rows is staged in shared memory with coalesced copies
  // (vector v of the chunk at stage[v]); each thread then reads its own
  // contiguous segment, its vectors in a rotated order so that a quarter warp
  // hits distinct banks.
  extern __shared__ __align__(16) uint4 draw_stage[];   // [2][kThreads * NV]
  {
    uint4* st_t = draw_stage;
    uint4* st_d = draw_stage + kThreads * NV;
    const bool al_t = (reinterpret_cast<uintptr_t>(zt_row) & 15u) == 0;
    const bool al_d = (reinterpret_cast<uintptr_t>(zd_row) & 15u) == 0;
#pragma unroll
    for (int k = 0; k < NV; ++k) {
      const int v = k * kThreads + (int)threadIdx.x;
      const int e = c * kDrawChunk + v * N;
      if (al_t && e + N <= V) cp_async16(&st_t[v], zt_row + e);
      else st_t[v] = load_vec_or_pad<T>(zt_row, e, V);
      if (!usep_r) {
        if (al_d && e + N <= V) cp_async16(&st_d[v], zd_row + e);
        else st_d[v] = load_vec_or_pad<T>(zd_row, e, V);
      }
    }
    cp_async_wait_all();
    __syncthreads();
  }
  float sr = 0.f, sp = 0.f;
  {
    uint4 vt[NV], vd[NV];
#pragma unroll
    for (int i = 0; i < NV; ++i) {
      const int v = (int)threadIdx.x * NV + ((i + (int)threadIdx.x) & (NV - 1));
      vt[i] = draw_stage[v];
      if (!usep_r) vd[i] = draw_stage[kThreads * NV + v];
    }
#pragma unroll
    for (int i = 0; i < NV; ++i) {
      float w[N], pv[N];
      pair_weights<T>(vt[i], vd[i], j, k2, usep_r, w, pv);
#pragma unroll
      for (int q = 0; q < N; ++q) {
        sr += w[q];
        sp += pv[q];
      }
    }
  }
  segs[((size_t)b * nch + c) * kThreads + threadIdx.x] = make_float2(sr, sp);
  __shared__ float shr[kThreads / 32], shp[kThreads / 32];
  float xr = sr, xp = sp;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    xr += __shfl_xor_sync(0xffffffffu, xr, o);
    xp += __shfl_xor_sync(0xffffffffu, xp, o);
  }
  const int wid = threadIdx.x >> 5, l = threadIdx.x & 31;
  if (l == 0) { shr[wid] = xr; shp[wid] = xp; }
  __syncthreads();
  if (threadIdx.x == 0) {
    float tr = 0.f, tp = 0.f;
    for (int q = 0; q < (int)(blockDim.x >> 5); ++q) { tr += shr[q]; tp += shp[q]; }
    parts[(size_t)b * nch + c] = make_float2(tr, tp);
  }
  if (!take_ticket_is_last(&counters[b], nch)) return;

  // ---- last CTA of sequence b: chunk, then segment, then token ----
  __shared__ float2 csum[kMaxDrawChunks];
  __shared__ double s_target, s_Z, s_before;
  __shared__ int s_chunk, s_degenerate, s_seg, s_y;
  __shared__ double s_clo, s_chi;
  for (int cc = threadIdx.x; cc < nch; cc += blockDim.x) csum[cc] = __ldcg(parts + (size_t)b * nch + cc);
  __syncthreads();
  if (threadIdx.x == 0) {
    double Zr = 0.0, Zp = 0.0;
    for (int cc = 0; cc < nch; ++cc) {
      Zr += csum[cc].x;
      Zp += csum[cc].y;
    }
    const int degenerate = (j.mode == 0 && Zr == 0.0) ? 1 : 0;
    const double Z = degenerate ? Zp : Zr;
    const double target = (double)u_final[b] * Z;
    double cum = 0.0, before = 0.0;
    int cstar = -1, last_nz = 0;
    for (int cc = 0; cc < nch; ++cc) {
      const double sc = degenerate ? csum[cc].y : csum[cc].x;
      if (sc > 0.0) last_nz = cc;
      if (cstar < 0 && cum + sc > target) { cstar = cc; before = cum; }
      cum += sc;
    }
    if (cstar < 0) {   // rounding put the target past the last step
      cstar = last_nz;
      before = 0.0;
      for (int cc = 0; cc < last_nz; ++cc) before += degenerate ? csum[cc].y : csum[cc].x;
    }
    s_target = target;
    s_Z = Z;
    s_before = before;
    s_chunk = cstar;
    s_degenerate = degenerate;
    s_seg = -1;
    s_y = INT32_MAX;
  }
  __syncthreads();
  const bool degenerate = s_degenerate != 0;
  // segment sums of the chosen chunk (written by its CTA) and their fp64 prefix
  const float2 sv = __ldcg(segs + ((size_t)b * nch + s_chunk) * kThreads + threadIdx.x);
  const float ts = degenerate ? sv.y : sv.x;
  double incl = ts;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const double x = __shfl_up_sync(0xffffffffu, incl, o);
    if (l >= o) incl += x;
  }
  __shared__ double wsum[kThreads / 32];
  if (l == 31) wsum[wid] = incl;
  __syncthreads();
  double base = s_before;
  for (int q = 0; q < wid; ++q) base += wsum[q];
  const double excl = base + incl - (double)ts;
  if (ts > 0.f && excl <= s_target && excl + (double)ts > s_target) {
    s_seg = threadIdx.x;        // unique: the segment ranges are disjoint
    s_clo = excl;
  }
  __syncthreads();
  // warp 0 walks the chosen segment: lane k holds tokens [2k, 2k + 2) of it
  if (wid == 0) {
    int seg = s_seg;
    double sbase = s_clo;
    if (seg < 0) {              // rounding: take the last segment with weight
      seg = kThreads - 1;
      sbase = s_target;
    }
    const int es = s_chunk * kDrawChunk + seg * kDrawSeg;
    float w2[2];
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      const int e = es + 2 * l + q;
      float wt = 0.f;
      if (e < V) {
        // the same arithmetic as the segment sums of pass 1
        const float pt = ex2_ftz(fmaf(to_f32(zt_row[e]), k2, -j.mt)) * (1.f / j.st);
        if (usep_r || degenerate) {
          wt = pt;
        } else {
          const float qd = ex2_ftz(fmaf(to_f32(zd_row[e]), k2, -j.md)) * (1.f / j.sd);
          wt = fmaxf(0.f, pt - qd);
        }
      }
      w2[q] = wt;
    }
    const float pair = w2[0] + w2[1];
    float inc = pair;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float x = __shfl_up_sync(0xffffffffu, inc, o);
      if (l >= o) inc += x;
    }
    const float rel = (float)(s_target - sbase);
    const float ex = inc - pair;
    int yl = INT32_MAX;
    double clo = 0.0, chi = 0.0;
    if (s_seg >= 0 && ex <= rel && inc > rel) {
      const bool first = ex + w2[0] > rel;
      yl = es + 2 * l + (first ? 0 : 1);
      clo = sbase + (double)(first ? ex : ex + w2[0]);
      chi = sbase + (double)(first ? ex + w2[0] : inc);
    }
    // lowest lane that holds the crossing (ties from rounding resolve low)
    const unsigned hit = __ballot_sync(0xffffffffu, yl != INT32_MAX);
    int lastw = -1;
#pragma unroll
    for (int q = 0; q < 2; ++q)
      if (w2[q] > 0.f) lastw = es + 2 * l + q;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) lastw = max(lastw, __shfl_xor_sync(0xffffffffu, lastw, o));
    if (hit) {
      const int src = __ffs(hit) - 1;
      if (l == src) {
        s_y = yl;
        s_clo = clo;
        s_chi = chi;
      }
    } else if (l == 0) {
      s_y = lastw >= 0 ? lastw : es;
      s_clo = s_target;
      s_chi = s_target;
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    const int y = s_y;
    const double Z = s_Z, u = u_final[b];
    int flags = j.flags;
    if (Z > 0.0 && (fabs(s_clo / Z - u) < 1e-6 || fabs(s_chi / Z - u) < 1e-6)) flags |= 2;  // CDF_BOUNDARY
    if (degenerate) flags |= 4;                                                           // DEGENERATE
    bonus[b] = y;
    if (flags_out) flags_out[b] = (uint8_t)flags;
    if (probs) probs[(size_t)b * (2 * n_max + 1) + 2 * n_max] = (float)Z;
    if (out_tokens) {
      out_tokens[(size_t)b * R + j.acc] = y;
      for (int rr = j.acc + 1; rr < R; ++rr) out_tokens[(size_t)b * R + rr] = -1;
    }
  }
  reset_ticket(&counters[b]);
}

// ===========================================================================
// Sampled rule, pass 1: row statistics, then the sequential accept test
// ===========================================================================

template <typename T>
__global__ void __launch_bounds__(kThreads, kCtasPerSm)
sample_stats_kernel(const T* __restrict__ zt, const T* __restrict__ zd, const float* __restrict__ draft_lse,
                    const int64_t* __restrict__ cand, const int32_t* __restrict__ n_draft,
                    const float* __restrict__ u_acc, int n_max, int V, int nch, int chunk,
                    float k2, MS* __restrict__ parts, float* __restrict__ zx,
                    int32_t* __restrict__ counters, SampleJob* __restrict__ jobs,
                    int32_t* __restrict__ accept_len, int32_t* __restrict__ commit_len,
                    int64_t* __restrict__ out_tokens, float* __restrict__ probs, int* __restrict__ err) {
  dependents_may_launch();   // the draw may be scheduled (it waits for this grid)
  const int R = n_max + 1;
  const int RR = R + n_max;              // target rows then draft rows of a sequence
  // with the draft rows' log-sum-exps supplied, only the target rows stream
  const int RS = draft_lse ? R : RR;
  const int c = blockIdx.x;
  const int b = blockIdx.y / RS, r = blockIdx.y - b * RS;
  // drafts of sequence b, clamped to [0, n_max] (an out-of-range count is recorded)
  int nb = n_draft ? n_draft[b] : n_max;
  if (nb < 0 || nb > n_max) {
    if (c == 0 && r == 0 && threadIdx.x == 0) record_dev_error(err, kDevErrBadNDraft);
    nb = min(max(nb, 0), n_max);
  }
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
  if (!take_ticket_is_last_t0(&counters[b], RS * nch)) return;

  // ---- last CTA of sequence b ----
  __shared__ MS rs[2 * kMaxRows];
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  if (draft_lse) {
    // draft row i: log2 of sum 2^(z k2) is LSE(z / T) * log2(e); as a (max, sum)
    // pair that is (lse2, 1), and q(x) = 2^(z_x k2 - lse2)
    for (int i = threadIdx.x; i < nb; i += blockDim.x) {
      rs[R + i] = MS{draft_lse[(size_t)b * n_max + i] * kLog2e, 1.f};
      const int64_t x = cand[(size_t)b * R + i + 1];
      zx[(size_t)b * RR + R + i] = (x >= 0 && x < V) ? ld_scalar(zd + ((size_t)b * n_max + i) * V + x)
                                                      : -CUDART_INF_F;
    }
  }
  for (int rr = w; rr < RS; rr += blockDim.x >> 5) {
    const bool t = rr < R;
    const int rix = t ? rr : rr - R;
    if (t ? rix > nb : rix >= nb) continue;
    MS2 x{-CUDART_INF_F, 0.f, 0.f};
    const MS* pr = parts + ((size_t)b * RR + rr) * nch;
    for (int cc = l; cc < nch; cc += 32) {
      const float2 raw = __ldcg(reinterpret_cast<const float2*>(pr + cc));
      x = ms2_merge(x, MS2{raw.x, raw.y, 0.f});
    }
    // fixed-order combine across lanes (compensated sums, rounded once)
    x = warp_ms2(x);
    if (l == 0) rs[rr] = MS{x.m, x.hi + x.lo};
  }
  __syncthreads();
  // Every candidate's p(x), q(x) and p/q at once, one thread each. The
  // numerator of p(x) is the very term the row sum holds for x (same exponent
  // fma, same ex2), so where x carries most of its row the approximation
  // errors of numerator and sum cancel; the fp32 exponent's rounding
  // residual r (z * k2 is exact in fp64 for bf16 or fp32 z) is put back as a
  // factor 1 + r ln 2. The quotients are formed in fp64.
  __shared__ double s_ratio[kMaxRows];
  __shared__ float s_px[kMaxRows], s_qx[kMaxRows];
  __shared__ uint8_t s_inv[kMaxRows];
  for (int i = (int)threadIdx.x + 1; i <= nb; i += blockDim.x) {
    const MS pt = rs[i - 1], pd = rs[R + i - 1];
    const float zxt = __ldcg(zx + (size_t)b * RR + (i - 1));
    const float zxd = zx[(size_t)b * RR + R + (i - 1)];
    const double k2d = (double)k2;
    const float at = fmaf(zxt, k2, -pt.m), ad = fmaf(zxd, k2, -pd.m);   // as in the row sums
    const double rt = ((double)zxt * k2d - (double)pt.m) - (double)at;
    const double rd = ((double)zxd * k2d - (double)pd.m) - (double)ad;
    const double px = (double)ex2_ftz(at) * (1.0 + rt * 0.6931471805599453) / (double)pt.s;
    const double qx = (double)ex2_ftz(ad) * (1.0 + rd * 0.6931471805599453) / (double)pd.s;
    s_px[i - 1] = (float)px;
    s_qx[i - 1] = (float)qx;
    // q(x) = 0: the candidate was not drawn from q (infinite ratio, flagged)
    s_inv[i - 1] = qx > 0.0 ? 0 : 1;
    s_ratio[i - 1] = qx > 0.0 ? px / qx : (double)CUDART_INF_F;
  }
  __syncthreads();
  __shared__ int s_a, s_eval;
  if (threadIdx.x == 0) {
    int a = 0, flags = 0;
    bool rejected = false;
    for (int i = 1; i <= nb; ++i) {
      const double ratio = s_ratio[i - 1];
      if (s_inv[i - 1]) flags |= 8;      // DFLASH_FLAG_INVALID
      const double u = (double)u_acc[(size_t)b * n_max + (i - 1)];
      if (ratio < 1.0 && fabs(u - ratio) < 1e-6) flags |= 1;   // ACCEPT_BOUNDARY
      if (u < ratio) {
        ++a;
      } else {
        rejected = true;
        break;
      }
    }
    s_eval = a + (rejected ? 1 : 0);
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
  if (probs)
    for (int i = threadIdx.x; i < n_max; i += blockDim.x) {
      const bool ev = i < s_eval;      // candidates the rule evaluated; 0 past them
      probs[(size_t)b * (2 * n_max + 1) + i] = ev ? s_px[i] : 0.f;
      probs[(size_t)b * (2 * n_max + 1) + n_max + i] = ev ? s_qx[i] : 0.f;
    }
  if (out_tokens) {
    // accepted drafts now; the bonus slot and padding are written by the draw
    const int a = s_a;
    for (int rr = threadIdx.x; rr < a; rr += blockDim.x)
      out_tokens[(size_t)b * R + rr] = cand[(size_t)b * R + rr + 1];
  }
  reset_ticket(&counters[b]);
}

// ===========================================================================
// DLoop gate
// ===========================================================================
template <typename T>
__global__ void __launch_bounds__(kThreads, kCtasPerSm)
gate_kernel(const T* __restrict__ z, const int64_t* __restrict__ tokens,
            const uint8_t* __restrict__ active, int k, int V, int nch, int chunk, float k2,
            float inv_t, float g, GateLayout lay, MS* __restrict__ parts, float* __restrict__ zx,
            int32_t* __restrict__ counters, float* __restrict__ c_s, uint8_t* __restrict__ cont,
            float* __restrict__ row_lse, uint8_t* __restrict__ flags, int32_t* __restrict__ n_verify) {
  const int c = blockIdx.x;
  const int row = blockIdx.y;             // b * k + i: the i-th row of this stage of sequence b
  const int b = row / k, i = row - b * k;
  const bool on = active ? active[b] != 0 : true;
  MS ms{-CUDART_INF_F, 0.f};
  const bool need = on || (row_lse != nullptr && lay.lse_inactive);
  if (need) {
    const T* zr = z + ((size_t)b * lay.z_rows + lay.z_row0 + i) * V;
    const int e0 = c * chunk, e1 = min(V, e0 + chunk);
    ms = row_chunk_ms<T>(zr, e0, e1, k2);
    if (threadIdx.x == 0) {
      const int64_t x = tokens[(size_t)b * lay.tok_stride + lay.tok0 + i];
      if (x >= e0 && x < e1) zx[row] = ld_scalar(zr + x);
    }
  }
  if (threadIdx.x == 0) parts[(size_t)row * nch + c] = ms;
  if (!take_ticket_is_last_t0(&counters[b], k * nch)) return;

  __shared__ MS rs[kMaxRows];
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  if (need) {
    for (int ii = w; ii < k; ii += blockDim.x >> 5) {
      MS2 x{-CUDART_INF_F, 0.f, 0.f};
      const MS* pr = parts + ((size_t)b * k + ii) * nch;
      for (int cc = l; cc < nch; cc += 32) {
        const float2 raw = __ldcg(reinterpret_cast<const float2*>(pr + cc));
        x = ms2_merge(x, MS2{raw.x, raw.y, 0.f});
      }
      x = warp_ms2(x);
      if (l == 0) rs[ii] = MS{x.m, x.hi + x.lo};
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    double csum = 0.0;
    for (int ii = 0; ii < k; ++ii) {
      const MS r = rs[ii];
      // natural-log values from log2-unit statistics: ln v = ln 2 * log2 v
      if (need && row_lse) row_lse[(size_t)b * lay.lse_stride + lay.lse0 + ii] = (r.m + log2f(r.s)) * 0.6931471805599453f;
      if (on) {
        const float zxv = __ldcg(zx + (size_t)b * k + ii);
        // log2 q(x) = (z_x k2 - m) - log2(sum)
        csum += ((double)fmaf(zxv, k2, -r.m) - (double)log2f(r.s)) * 0.6931471805599453;
      }
    }
    const float cval = on ? (float)csum : 0.f;
    c_s[b] = cval;
    cont[b] = (on && csum >= (double)g) ? 1 : 0;
    if (flags) flags[b] = (on && fabs(csum - (double)g) < 1e-4) ? 1 : 0;
    // looped draft: the stage's k tokens join the verify whatever its gate says
    if (n_verify && on) n_verify[b] += k;
  }
  reset_ticket(&counters[b]);
}

// ===========================================================================
// Draft-side token choice over the MASK rows (DFlash page, inference steps:
// each MASK position's logits give a draft token, argmax or one sample per
// position). One CTA per row (persistent over rows): the row goes in chunks of
// 256 segments of kSelVecs 16-byte vectors, each thread loading its own
// contiguous segment straight from global memory (a warp's lines are used
// whole over its 8 loads; no staging, no block barrier while streaming); each
// thread keeps its segment's record (max * k2, sum of 2^(z k2 - max k2)) and
// the running (max, lowest index). A sampled row then takes one block scan
// over the records in token order and one warp walk over the chosen segment
// (inverse CDF, ascending token order).
// ===========================================================================
constexpr int kSelVecs = 8;                      // 16-byte vectors per thread and chunk
constexpr int kSelCtasPerSm = 4;                 // resident CTAs per SM


template <typename T>
__global__ void __launch_bounds__(kThreads, kSelCtasPerSm)
draft_select_kernel(const T* __restrict__ z, const int64_t* __restrict__ anchor, const int32_t* __restrict__ n_draft,
                    const float* __restrict__ u_draft, int B, int n_max, int V, int nch, float k2, int sampled,
                    float2* __restrict__ rec, int64_t* __restrict__ cand, float* __restrict__ q_x,
                    float* __restrict__ row_lse, uint8_t* __restrict__ flags, int* __restrict__ err) {
  constexpr int N = VecTraits<T>::N;
  constexpr int NV = kSelVecs;
  constexpr int SEG = NV * N;                      // contiguous tokens per thread and chunk
  constexpr int CHUNK = kThreads * SEG;            // tokens per chunk
  constexpr int TPL = SEG / 32;                    // tokens per lane in the segment walk
  const bool need_sum = sampled || row_lse != nullptr;   // argmax alone needs no exponentials
  const int tid = threadIdx.x, wid = tid >> 5, l = tid & 31;
  __shared__ double s_wsum[kThreads / 32];
  __shared__ double s_Z, s_cbefore;
  __shared__ int s_j, s_y;
  __shared__ float s_qx;
  __shared__ uint8_t s_flag;

  for (int row = blockIdx.x; row < B * n_max; row += gridDim.x) {
    const int b = row / n_max, i = row - b * n_max;
    // drafts of sequence b, clamped to [0, n_max] (an out-of-range count is recorded)
    const int nd = n_draft ? n_draft[b] : n_max;
    if ((nd < 0 || nd > n_max) && i == 0 && tid == 0) record_dev_error(err, kDevErrBadNDraft);
    const int nb = min(max(nd, 0), n_max);
    const size_t crow = (size_t)b * (n_max + 1);
    if (i == 0 && tid == 0) cand[crow] = anchor[b];
    if (i >= nb) {   // position not drafted: padding
      if (tid == 0) {
        cand[crow + i + 1] = -1;
        if (q_x) q_x[row] = 0.f;
        if (row_lse) row_lse[row] = 0.f;
        if (flags) flags[row] = 0;
      }
      continue;
    }
    const T* zr = z + (size_t)row * V;
    float2* rr = rec + (size_t)row * nch * kThreads;
    const bool aligned = (reinterpret_cast<uintptr_t>(zr) & 15u) == 0;
    // each thread loads its own contiguous segment of every chunk straight
    // from global memory (its 8 vectors in a rotated order; the lines a warp
    // touches are used whole over those loads), no staging and no block barrier
    const uint4* zv = reinterpret_cast<const uint4*>(zr);
    VI best{-CUDART_INF_F, INT32_MAX};
    for (int c = 0; c < nch; ++c) {
      const int e0 = c * CHUNK + tid * SEG;
      uint4 vv[NV];
      float vmax[NV];
      float tmax = -CUDART_INF_F;
#pragma unroll
      for (int k = 0; k < NV; ++k) {
        const int e = e0 + ((k + tid) & (NV - 1)) * N;
        vv[k] = (aligned && e + N <= V) ? __ldg(zv + e / N) : load_vec_or_pad<T>(zr, e, V);
      }
#pragma unroll
      for (int k = 0; k < NV; ++k) {
        vmax[k] = vec_max<T>(vv[k]);
        tmax = fmaxf(tmax, vmax[k]);
      }
      // lowest index of the segment's max, searched only when it can win
      if (tmax != -CUDART_INF_F && tmax >= best.v) {
        int ebest = INT32_MAX;
#pragma unroll
        for (int k = 0; k < NV; ++k) {
          const int ek = e0 + ((k + tid) & (NV - 1)) * N;
          if (vmax[k] == tmax && ek < ebest) {
            float f[N];
            unpack16<T>(vv[k], f);
            int q = N - 1;
#pragma unroll
            for (int qq = N - 1; qq >= 0; --qq)
              if (f[qq] == tmax) q = qq;
            ebest = ek + q;
          }
        }
        if (vi_better(tmax, ebest, best)) best = VI{tmax, ebest};
      }
      if (need_sum) {
        const float mt = tmax == -CUDART_INF_F ? -CUDART_INF_F : ms_offset(tmax, k2);
        float st = 0.f;
        if (tmax != -CUDART_INF_F) {
#pragma unroll
          for (int k = 0; k < NV; ++k) {
            float f[N];
            unpack16<T>(vv[k], f);
#pragma unroll
            for (int q = 0; q < N; ++q) st += ex2_ftz(fmaf(f[q], k2, -mt));
          }
        }
        rr[c * kThreads + tid] = make_float2(mt, st);
      }
    }
    // ---- the row's max and its lowest index ----
    const VI rb = block_vi(best);
    __shared__ VI s_best;
    if (tid == 0) s_best = rb;
    __syncthreads();
    const VI arg = s_best;
    const float m2M = ms_offset(arg.v, k2);   // integer-valued: record rescales are exact
    if (!need_sum) {
      if (tid == 0) {
        cand[crow + i + 1] = arg.i;
        if (q_x) q_x[row] = 1.f;
        if (flags) flags[row] = 0;
      }
      continue;
    }
    // ---- records in token order: thread t holds records t*nch .. t*nch + nch - 1
    // (record j = chunk j / 256, segment j % 256), weights in row units ----
    double loc = 0.0;
    for (int r = 0; r < nch; ++r) {
      const int j = tid * nch + r;
      const float2 w2 = rr[(j / kThreads) * kThreads + (j % kThreads)];
      if (w2.x != -CUDART_INF_F) loc += (double)w2.y * (double)pow2i(w2.x - m2M);
    }
    double inc = loc;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const double x = __shfl_up_sync(0xffffffffu, inc, o);
      if (l >= o) inc += x;
    }
    if (l == 31) s_wsum[wid] = inc;
    if (tid == 0) { s_j = -1; s_y = -1; }
    __syncthreads();
    double base = 0.0, Z = 0.0;
    for (int q = 0; q < kThreads / 32; ++q) {
      if (q < wid) base += s_wsum[q];
      Z += s_wsum[q];
    }
    if (tid == 0) {
      s_Z = Z;
      if (row_lse) row_lse[row] = (float)(((double)m2M + log2(Z)) * 0.6931471805599453);
    }
    if (!sampled) {
      if (tid == 0) {
        cand[crow + i + 1] = arg.i;
        if (q_x) q_x[row] = 1.f;
        if (flags) flags[row] = 0;
      }
      __syncthreads();
      continue;
    }
    const double u = (double)u_draft[row];
    const double target = u * Z;
    const double excl = base + inc - loc;
    if (loc > 0.0 && excl <= target && excl + loc > target) {
      // the crossing record is one of this thread's: walk them in order
      double cum = excl;
      int jsel = tid * nch + nch - 1;
      for (int r = 0; r < nch; ++r) {
        const int j = tid * nch + r;
        const float2 w2 = rr[(j / kThreads) * kThreads + (j % kThreads)];
        const double w = w2.x == -CUDART_INF_F ? 0.0 : (double)w2.y * (double)pow2i(w2.x - m2M);
        if (w > 0.0 && cum + w > target) { jsel = j; break; }
        cum += w;
      }
      s_j = jsel;
      s_cbefore = cum;
    }
    __syncthreads();
    if (wid == 0) {
      int j = s_j;
      const bool found = j >= 0;
      double cbefore = s_cbefore;
      if (!found) j = nch * kThreads - 1;     // rounding: resolved below to the last token with weight
      const int cj = j / kThreads, tj = j % kThreads;
      const float2 w2 = rr[cj * kThreads + tj];
      const float mt = w2.x;
      const double f = mt == -CUDART_INF_F ? 0.0 : (double)pow2i(mt - m2M);   // segment units -> row units
      const int es = cj * CHUNK + tj * SEG;
      float w[TPL];
      float lsum = 0.f;
#pragma unroll
      for (int q = 0; q < TPL; ++q) {
        const int e = es + TPL * l + q;
        w[q] = (e < V && mt != -CUDART_INF_F) ? ex2_ftz(fmaf(to_f32(zr[e]), k2, -mt)) : 0.f;
        lsum += w[q];
      }
      float incw = lsum;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const float x = __shfl_up_sync(0xffffffffu, incw, o);
        if (l >= o) incw += x;
      }
      const float rel = found ? (float)((target - cbefore) / f) : 0.f;
      const float ex = incw - lsum;
      int yl = INT32_MAX;
      float run_sel = 0.f, wy = 0.f;
      if (found && ex <= rel && incw > rel) {
        float run = ex;
        bool done = false;
#pragma unroll
        for (int q = 0; q < TPL; ++q) {
          if (!done && (q == TPL - 1 || run + w[q] > rel)) {
            yl = es + TPL * l + q;
            run_sel = run;
            wy = w[q];
            done = true;
          }
          run += w[q];
        }
      }
      const unsigned hit = __ballot_sync(0xffffffffu, yl != INT32_MAX);
      if (hit) {
        if (l == __ffs(hit) - 1) {
          const double c_lo = (cbefore + f * (double)run_sel) / Z, c_hi = (cbefore + f * (double)(run_sel + wy)) / Z;
          s_y = yl;
          s_qx = (float)((double)wy * f / Z);
          s_flag = (fabs(c_lo - u) < 1e-6 || fabs(c_hi - u) < 1e-6) ? 2 : 0;   // CDF_BOUNDARY
        }
      } else if (l == 0) {
        s_y = -1;   // the target lies past every step (rounding)
      }
    }
    __syncthreads();
    if (s_y < 0) {
      // rounding put the target past the last step: the last token with weight,
      // found by a block-wide search from the end of the row
      __shared__ int s_last;
      if (tid == 0) s_last = -1;
      __syncthreads();
      for (int top = V - 1; top >= 0; top -= kThreads) {
        const int e = top - tid;
        const bool wt = e >= 0 && ex2_ftz(fmaf(to_f32(zr[e]), k2, -m2M)) > 0.f;
        if (wt) atomicMax(&s_last, e);
        if (__syncthreads_or(wt)) break;
      }
      if (tid == 0) {
        const int y = s_last >= 0 ? s_last : arg.i;
        s_y = y;
        s_qx = (float)((double)ex2_ftz(fmaf(to_f32(zr[y]), k2, -m2M)) / s_Z);
        s_flag = 2;
      }
      __syncthreads();
    }
    if (tid == 0) {
      cand[crow + i + 1] = s_y;
      if (q_x) q_x[row] = s_qx;
      if (flags) flags[row] = s_flag;
    }
    __syncthreads();
  }
}

// ===========================================================================
// Host launchers
// ===========================================================================
static int vec_elems(int dtype) { return dtype == 0 ? 4 : 8; }

// Chunks per row: the grid (rows x chunks) is sized to one wave of resident
// CTAs (kCtasPerSm per SM) so that no partial wave trails the kernel; each thread
// handles at least one 16-byte vector per chunk.
ChunkPlan plan_chunks(int rows, int V, int dtype, int num_sms) {
  const int per_thread_vec = kThreads * vec_elems(dtype);
  const int units = (V + per_thread_vec - 1) / per_thread_vec;   // vector rounds for a whole row
  const long wave = (long)kCtasPerSm * num_sms;
  long nch = wave / (rows > 0 ? rows : 1);
  if (nch < 1) nch = 1;
  if (nch > units) nch = units;
  ChunkPlan p;
  p.chunk = (int)((units + nch - 1) / nch) * per_thread_vec;
  p.nch = (V + p.chunk - 1) / p.chunk;
  return p;
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
  const int nch2 = (V + kDrawChunk - 1) / kDrawChunk;
  s += align_up((size_t)B * nch2 * sizeof(float2));                // chunk sums
  s += align_up((size_t)B * nch2 * kThreads * sizeof(float2));     // segment sums
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
      a.target_pred, a.err);
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
  const int nch2 = (a.V + kDrawChunk - 1) / kDrawChunk;
  float2* dparts = (float2*)ws;
  ws += align_up((size_t)a.B * nch2 * sizeof(float2));
  float2* dsegs = (float2*)ws;
  const float k2 = kLog2e / a.temperature;
  dim3 g1(p.nch, a.B * (a.draft_lse ? R : RR));
  sample_stats_kernel<T><<<g1, kThreads, 0, a.stream>>>(
      (const T*)a.target_logits, (const T*)a.draft_logits, a.draft_lse, a.cand, a.n_draft, a.u_accept,
      a.n_max, a.V, p.nch, p.chunk, k2, parts, zx, a.counters, jobs, a.accept_len, a.commit_len,
      a.out_tokens, a.probs, a.err);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  constexpr int kDrawSmem = 2 * kDrawChunk * (int)sizeof(T);   // the chunk of both rows
  static SmemOptIn opt_in;
  e = opt_in.ensure(sample_draw_kernel<T>, kDrawSmem);
  if (e != cudaSuccess) return e;
  e = launch_dependent(sample_draw_kernel<T>, dim3(nch2, a.B), dim3(kThreads), kDrawSmem, a.stream,
                       (const T*)a.target_logits, (const T*)a.draft_logits, a.u_final, a.n_max, a.V, nch2, k2, jobs,
                       dparts, dsegs, a.counters, a.bonus, a.out_tokens, a.flags, a.probs);
  if (e != cudaSuccess) return e;
  (void)R;
  return cudaGetLastError();
}

cudaError_t launch_verify_sample(const VerifyArgs& a, int num_sms) {
  return a.dtype == 0 ? launch_sample_t<float>(a, num_sms) : launch_sample_t<bf16>(a, num_sms);
}

static int sel_chunk(int dtype) { return kThreads * kSelVecs * vec_elems(dtype); }

size_t draft_select_ws_bytes(int B, int n_max, int V, int dtype) {
  const size_t rows = (size_t)B * n_max;
  const int nch = (V + sel_chunk(dtype) - 1) / sel_chunk(dtype);
  return align_up(rows * nch * kThreads * sizeof(float2));
}

template <typename T>
static cudaError_t launch_draft_select_t(const DraftSelectArgs& a) {
  const int nch = (a.V + sel_chunk(a.dtype) - 1) / sel_chunk(a.dtype);
  const long rows = (long)a.B * a.n_max;
  const bool sampled = a.temperature > 0.f;
  const float k2 = kLog2e / (sampled ? a.temperature : 1.f);
  const int grid = (int)std::min<long>(rows, (long)kSelCtasPerSm * a.num_sms);
  draft_select_kernel<T><<<grid, kThreads, 0, a.stream>>>(
      (const T*)a.draft_logits, a.anchor, a.n_draft, a.u_draft, a.B, a.n_max, a.V, nch, k2, sampled ? 1 : 0,
      (float2*)a.scratch, a.cand, a.q_x, a.row_lse, a.flags, a.err);
  return cudaGetLastError();
}

cudaError_t launch_draft_select(const DraftSelectArgs& a) {
  return a.dtype == 0 ? launch_draft_select_t<float>(a) : launch_draft_select_t<bf16>(a);
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
      kLog2e / a.temperature, 1.f / a.temperature, a.g, a.layout, parts, zx, a.counters, a.c_s, a.cont,
      a.row_lse, a.flags, a.n_verify);
  return cudaGetLastError();
}

cudaError_t launch_gate(const GateArgs& a, int num_sms) {
  return a.dtype == 0 ? launch_gate_t<float>(a, num_sms) : launch_gate_t<bf16>(a, num_sms);
}

}  // namespace dflash
