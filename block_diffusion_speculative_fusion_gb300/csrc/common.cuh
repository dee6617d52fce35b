// Shared device helpers of the DFlash kernels (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math_constants.h>
#include <stdint.h>

namespace dflash {

typedef __nv_bfloat16 bf16;

constexpr float kLog2e = 1.4426950408889634f;

// ---------------------------------------------------------------------------
// Programmatic dependent launch. A kernel started with launch_dependent() may
// be scheduled while the kernel before it in the stream is still running (once
// every CTA of that kernel has executed dependents_may_launch() or ended); it
// executes wait_for_prior_grid() before it touches memory that earlier work
// writes or reads. Both instructions do nothing in a kernel launched plainly.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void wait_for_prior_grid() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void dependents_may_launch() { asm volatile("griddepcontrol.launch_dependents;"); }

template <typename... KArgs, typename... Args>
inline cudaError_t launch_dependent(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                                    Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args&&>(args)...);
}

// ---------------------------------------------------------------------------
// 16-byte vectors of logits, unpacked to fp32
// ---------------------------------------------------------------------------
template <typename T> struct VecTraits;
template <> struct VecTraits<float> { static constexpr int N = 4; };
template <> struct VecTraits<bf16> { static constexpr int N = 8; };

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// Streaming 16-byte load that does not allocate in L1 (every logit is read once).
__device__ __forceinline__ uint4 ld_stream16(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p));
  return r;
}

template <typename T>
__device__ __forceinline__ void unpack16(const uint4& u, float* f);
template <>
__device__ __forceinline__ void unpack16<float>(const uint4& u, float* f) {
  f[0] = __uint_as_float(u.x); f[1] = __uint_as_float(u.y);
  f[2] = __uint_as_float(u.z); f[3] = __uint_as_float(u.w);
}
template <>
__device__ __forceinline__ void unpack16<bf16>(const uint4& u, float* f) {
  f[0] = bf16_lo(u.x); f[1] = bf16_hi(u.x); f[2] = bf16_lo(u.y); f[3] = bf16_hi(u.y);
  f[4] = bf16_lo(u.z); f[5] = bf16_hi(u.z); f[6] = bf16_lo(u.w); f[7] = bf16_hi(u.w);
}

__device__ __forceinline__ float ld_scalar(const float* p) { return __ldg(p); }
__device__ __forceinline__ float ld_scalar(const bf16* p) { return __bfloat162float(*p); }

__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(bf16 x) { return __bfloat162float(x); }
template <typename T> __device__ __forceinline__ T from_f32(float x);
template <> __device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ bf16 from_f32<bf16>(float x) { return __float2bfloat16_rn(x); }

// ---------------------------------------------------------------------------
// Completion tickets: the last CTA of a group does the group's epilogue.
// Every thread has already written its part of the CTA's partial results; each
// publishes its writes with a device-scope fence, then thread 0 takes a ticket.
// Readers in the last CTA must load partials through L2 (__ldcg). No CTA waits.
// ---------------------------------------------------------------------------
__device__ __forceinline__ bool take_ticket_is_last(int32_t* counter, int group_size) {
  __shared__ int s_last;
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) {
    int t = atomicAdd(counter, 1);
    s_last = (t == group_size - 1);
  }
  __syncthreads();
  const bool last = s_last != 0;
  if (last) __threadfence();
  return last;
}

__device__ __forceinline__ void reset_ticket(int32_t* counter) {
  if (threadIdx.x == 0) atomicExch(counter, 0);
}

// Variant for results written by thread 0 alone: only thread 0 fences.
__device__ __forceinline__ bool take_ticket_is_last_t0(int32_t* counter, int group_size) {
  __shared__ int s_last0;
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    const int t = atomicAdd(counter, 1);
    s_last0 = (t == group_size - 1);
    if (s_last0) __threadfence();
  }
  __syncthreads();
  return s_last0 != 0;
}

// ---------------------------------------------------------------------------
// Online max / scaled-sum pairs in log2 units: a row's statistics are an
// integer-valued offset m = rint(max(z) * k2) and s = sum 2^(fma(z, k2, -m)),
// every exponent formed by one fused multiply-add, so that the same expression
// evaluated later for one element of the row is consistent with the sum.
// Because the offsets are integers, rescaling a partial sum to another offset
// multiplies it by an exact power of two: merging partials adds no rounding
// beyond the one addition (a non-integer offset would put an exp2 rounding
// into every merge of the reduction tree).
// ---------------------------------------------------------------------------
struct MS { float m; float s; };

// 2^k for an integer-valued k <= 0, exact (0 below the normal range).
__device__ __forceinline__ float pow2i(float k) {
  const int ki = (int)k;
  return ki < -126 ? 0.f : __int_as_float((ki + 127) << 23);
}

// The integer-valued log2 offset of a row whose largest logit is v.
__device__ __forceinline__ float ms_offset(float v, float k2) { return rintf(v * k2); }

__device__ __forceinline__ MS ms_merge(MS a, MS b) {
  const float M = fmaxf(a.m, b.m);
  if (M == -CUDART_INF_F) return MS{M, 0.f};
  const float sa = (a.m == -CUDART_INF_F) ? 0.f : a.s * pow2i(a.m - M);
  const float sb = (b.m == -CUDART_INF_F) ? 0.f : b.s * pow2i(b.m - M);
  return MS{M, sa + sb};
}

// The same pair with the sum carried as an unevaluated fp32 pair hi + lo, for
// reduction trees whose partial sums must not lose digits (a 256-thread tree
// in plain fp32 errs by up to 8 ulps). Merges use an exact power-of-two
// rescale and an error-free two-sum, fp32 arithmetic only (fp64 is slow here).
struct MS2 { float m; float hi; float lo; };

__device__ __forceinline__ MS2 ms2_merge(MS2 a, MS2 b) {
  const float M = fmaxf(a.m, b.m);
  if (M == -CUDART_INF_F) return MS2{M, 0.f, 0.f};
  const float fa = (a.m == -CUDART_INF_F) ? 0.f : pow2i(a.m - M);
  const float fb = (b.m == -CUDART_INF_F) ? 0.f : pow2i(b.m - M);
  const float ah = a.hi * fa, al = a.lo * fa, bh = b.hi * fb, bl = b.lo * fb;   // exact
  const float s = ah + bh;
  const float bp = s - ah;
  const float e = (ah - (s - bp)) + (bh - bp);     // s + e == ah + bh exactly
  const float lo = (al + bl) + e;
  const float hi = s + lo;
  return MS2{M, hi, lo - (hi - s)};
}

__device__ __forceinline__ MS2 warp_ms2(MS2 v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    MS2 w{__shfl_xor_sync(0xffffffffu, v.m, o), __shfl_xor_sync(0xffffffffu, v.hi, o),
          __shfl_xor_sync(0xffffffffu, v.lo, o)};
    v = ms2_merge(v, w);
  }
  return v;
}

__device__ __forceinline__ MS warp_ms(MS v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    MS w{__shfl_xor_sync(0xffffffffu, v.m, o), __shfl_xor_sync(0xffffffffu, v.s, o)};
    v = ms_merge(v, w);
  }
  return v;
}

// Largest of the 8 (bf16) or 4 (fp32) values of a 16-byte vector.
template <typename T> __device__ __forceinline__ float vec_max(const uint4& u);
template <> __device__ __forceinline__ float vec_max<bf16>(const uint4& u) {
  const __nv_bfloat162 a = __hmax2(*reinterpret_cast<const __nv_bfloat162*>(&u.x),
                                   *reinterpret_cast<const __nv_bfloat162*>(&u.y));
  const __nv_bfloat162 b = __hmax2(*reinterpret_cast<const __nv_bfloat162*>(&u.z),
                                   *reinterpret_cast<const __nv_bfloat162*>(&u.w));
  const __nv_bfloat162 c = __hmax2(a, b);
  return fmaxf(__low2float(c), __high2float(c));
}
template <> __device__ __forceinline__ float vec_max<float>(const uint4& u) {
  return fmaxf(fmaxf(__uint_as_float(u.x), __uint_as_float(u.y)), fmaxf(__uint_as_float(u.z), __uint_as_float(u.w)));
}

// (value, index) maximum with the lowest index among equal values.
struct VI { float v; int32_t i; };

__device__ __forceinline__ bool vi_better(float v, int32_t i, const VI& b) {
  return v > b.v || (v == b.v && i < b.i);
}

__device__ __forceinline__ VI warp_vi(VI a) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    VI w{__shfl_xor_sync(0xffffffffu, a.v, o), __shfl_xor_sync(0xffffffffu, a.i, o)};
    if (vi_better(w.v, w.i, a)) a = w;
  }
  return a;
}

}  // namespace dflash
