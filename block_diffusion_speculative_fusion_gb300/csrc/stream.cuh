// Vocabulary-row streaming helpers shared by the verify, gate, draft-select
// and DDTree kernels: coalesced 16-byte row visits, deterministic block
// reductions of (value, index) and (max, scaled sum) pairs, and 16-byte
// global -> shared copies.
#pragma once

#include "common.cuh"

namespace dflash {

constexpr int kThreads = 256;   // threads of every streaming CTA

// Visit elements [e0, e1) of row z: 16-byte vectors in the aligned middle,
// scalars at both ends. fv(u, first_index) gets one raw 16-byte vector, fs(v, i)
// one value. A thread visits its vectors in ascending index order.
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
    for (int u = 0; u < UNROLL; ++u) fv(r[u], a + (v + u * (int)blockDim.x) * N);
  }
  for (; v < nvec; v += blockDim.x) fv(ld_stream16(vp + v), a + v * N);
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

__device__ __forceinline__ MS block_ms(MS x) {
  __shared__ MS sh[kThreads / 32];
  x = warp_ms(x);
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  __syncthreads();
  if (l == 0) sh[w] = x;
  __syncthreads();
  if (w == 0) {
    x = (l < (int)(blockDim.x >> 5)) ? sh[l] : MS{-CUDART_INF_F, 0.f};
    x = warp_ms(x);
  }
  return x;  // valid in thread 0
}

// Block tree of (max, sum) pairs with compensated fp32 sums; the result
// (valid in thread 0) is rounded to one fp32 sum.
__device__ __forceinline__ MS block_ms2(MS2 x) {
  __shared__ MS2 sh2[kThreads / 32];
  x = warp_ms2(x);
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  __syncthreads();
  if (l == 0) sh2[w] = x;
  __syncthreads();
  if (w == 0) {
    x = (l < (int)(blockDim.x >> 5)) ? sh2[l] : MS2{-CUDART_INF_F, 0.f, 0.f};
    x = warp_ms2(x);
  }
  return MS{x.m, x.hi + x.lo};
}

// 2^x on the special-function unit, flushing denormal results to zero (terms
// below 2^-126 of a row maximum do not change a sum that contains 1).
__device__ __forceinline__ float ex2_ftz(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Streaming statistics of elements [e0, e1) of one row in log2 units:
// m = rint(max(z) * k2), s = sum 2^(fma(z, k2, -m)). The same code serves target and
// draft rows, so identical rows give bit-identical statistics.
// The thread's running sum is compensated (Kahan): a thread adds some 60
// vector sums of a 128k-token row, whose plain fp32 sum errs by ~sqrt(60) ulps
// (~5e-7 relative), as much as the 1e-6 decision band of the sampled rule; the
// block combines the threads' sums as compensated fp32 pairs.
template <typename T>
__device__ __forceinline__ MS row_chunk_ms(const T* z, int e0, int e1, float k2) {
  constexpr int N = VecTraits<T>::N;
  float zmax = -CUDART_INF_F;   // running max in logit units (exact comparisons)
  MS acc{-CUDART_INF_F, 0.f};
  float comp = 0.f;             // Kahan compensation of acc.s
  auto kadd = [&](float x) {
    const float y = x - comp;
    const float t = acc.s + y;
    comp = (t - acc.s) - y;
    acc.s = t;
  };
  auto raise_to = [&](float v) {
    const float m2 = ms_offset(v, k2);
    const float f = (acc.m == -CUDART_INF_F) ? 0.f : pow2i(acc.m - m2);   // exact power of two
    acc.s *= f;
    comp *= f;
    acc.m = m2;
    zmax = v;
  };
  auto add_vec = [&](const uint4& u, int) {
    const float vm = vec_max<T>(u);
    if (vm > zmax) raise_to(vm);
    if (zmax == -CUDART_INF_F) return;
    float f[N];
    unpack16<T>(u, f);
    float s = 0.f;
#pragma unroll
    for (int j = 0; j < N; ++j) s += ex2_ftz(fmaf(f[j], k2, -acc.m));
    kadd(s);
  };
  auto add_one = [&](float v, int) {
    if (v > zmax) raise_to(v);
    if (zmax != -CUDART_INF_F) kadd(ex2_ftz(fmaf(v, k2, -acc.m)));
  };
  for_range<T, 8>(z, e0, e1, add_vec, add_one);
  return block_ms2(MS2{acc.m, acc.s, -comp});
}


template <typename T>
__device__ __forceinline__ uint4 load_vec_or_pad(const T* row, int e, int V) {
  constexpr int N = VecTraits<T>::N;
  if (e + N <= V && (reinterpret_cast<uintptr_t>(row + e) & 15u) == 0)
    return __ldg(reinterpret_cast<const uint4*>(row + e));
  T tmp[N];
#pragma unroll
  for (int q = 0; q < N; ++q) tmp[q] = (e + q < V) ? row[e + q] : from_f32<T>(-CUDART_INF_F);
  return *reinterpret_cast<const uint4*>(tmp);
}

// 16-byte global -> shared copy that bypasses registers (L2 only)
__device__ __forceinline__ void cp_async16(void* smem_dst, const void* gmem_src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"((uint32_t)__cvta_generic_to_shared(smem_dst)),
               "l"(gmem_src)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_one() { asm volatile("cp.async.wait_group 1;" ::: "memory"); }

}  // namespace dflash
