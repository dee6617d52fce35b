// tcgen05 tensor-core GEMM for the context-KV projections (sm_103a):
//   part[seg][t][n] = sum over one K segment of W[n][k] * X[t][k]
// with W [N, K] (weights, K contiguous) and X [T, K] (committed rows, K
// contiguous), bf16 in, fp32 out.
//
// Weights are the A operand (M = 128 output features per tile) and the rows
// are the B operand. When all T rows fit 512, a tile covers them as two MMA
// groups of up to 256 rows that share each k-block's weight tile, so a
// decode-sized T reads each weight byte from HBM once; larger T uses tiles of
// 256 rows, whose smaller stages make a deeper ring. The rows
// of a pass are loaded with 256-, 64- and 16-row boxes, so a short second
// group costs only the rows it has; the ring of stages is laid out at run time
// for the number of rows present.
//
// Weight tiles are loaded with an L2 evict-first policy: each weight byte is
// read once, and without the hint the weight stream pushes the split-K
// partial sums out of L2 before the kernels that sum them run.
//
// Persistent CTAs (one per SM): when there are at least GRID tiles, whole
// waves of GRID tiles go one per CTA (concurrent tiles then share their rows
// and weights in L2); the remaining tiles' (tile, 64-wide k-block) space is
// split into equal contiguous ranges (stream-K style). A range that covers
// part of a tile writes that tile's partial sum to its own segment slot, and
// the consumers sum a tile's segments in a fixed order, so results are
// deterministic.
//
// Per CTA: warp 0 = TMA producer, warp 1 = TMEM allocator and single-thread
// MMA issuer, warps 2-5 = epilogue (TMEM -> registers -> global). With one
// group per pass, two 256-column TMEM accumulators let the epilogue of one
// range piece overlap the MMAs of the next; with two groups they are the two
// groups' accumulators. Every mbarrier wait is bounded: a wait that gives up
// records an error code, the CTA drains its own copies and MMAs (again
// bounded), frees TMEM and returns.
#include <algorithm>

#include "common.cuh"
#include "internal.h"
#include "tc.cuh"
#include "tma.cuh"

namespace dflash {

namespace tc {
using namespace tcplan;
constexpr int A_BYTES = BM * BK * 2;    // 16 KB: one k-block of 128 weight rows
constexpr int MAX_STAGES = 12;   // barrier area: 8 * (2 * 12 + 5) + 12 bytes <= 256
constexpr int THREADS = 192;
constexpr int TMEM_COLS = 512;          // two 256-column fp32 accumulators
constexpr int SMEM_BYTES = 232448;      // all of it: the ring is sized at run time
constexpr int RING_BYTES = SMEM_BYTES - 1024 - 256;
}  // namespace tc

struct TcWork {
  int T, per, PR, P, total, MT, KB;
  int full, waves;    // tiles handed out whole (waves of GRID), and how many waves
  int lo, hi;         // this CTA's k-block range over the split tiles
  int rows_max;       // rows of the largest pass, rounded up to 16
  int stage_bytes, stages, nbuf;
};

__device__ __forceinline__ TcWork tc_work(const int32_t* meta, int per_idx, int MT, int KB, int T_max) {
  TcWork w;
  w.T = min(meta[0], T_max);
  w.per = meta[per_idx];
  w.MT = MT;
  w.KB = KB;
  w.PR = gemm_tc_pass_rows(w.T);
  w.P = (w.T + w.PR - 1) / w.PR;
  w.total = MT * w.P * KB;
  w.full = gemm_tc_full_tiles(w.T, MT * tc::BM);
  w.waves = w.full / tc::GRID;
  w.lo = w.full * KB + (int)blockIdx.x * w.per;
  w.hi = min(w.total, w.lo + w.per);
  w.rows_max = min(w.PR, (w.T + 15) / 16 * 16);
  w.stage_bytes = (tc::A_BYTES + w.rows_max * tc::BK * 2 + 1023) / 1024 * 1024;
  w.stages = min(tc::MAX_STAGES, tc::RING_BYTES / w.stage_bytes);
  w.nbuf = w.rows_max <= tc::BN ? 2 : 1;
  return w;
}

struct TcPiece {
  int tile, kb0, kb1, m_tile, r0, rows, ng, seg;
};
// The pieces of this CTA in order: its whole tiles (one per wave), then its
// k-block range over the split tiles. `wave` and `pos` carry the position.
__device__ __forceinline__ bool tc_next(const TcWork& w, int& wave, int& pos, TcPiece& c) {
  if (wave < w.waves) {
    c.tile = wave * tc::GRID + (int)blockIdx.x;
    c.kb0 = 0;
    c.kb1 = w.KB;
    c.seg = 0;
    ++wave;
  } else if (pos < w.hi) {
    c.tile = pos / w.KB;
    c.kb0 = pos - c.tile * w.KB;
    c.kb1 = min(w.KB, c.kb0 + (w.hi - pos));
    c.seg = (int)blockIdx.x - ((c.tile - w.full) * w.KB) / w.per;
    pos += c.kb1 - c.kb0;
  } else {
    return false;
  }
  c.m_tile = c.tile % w.MT;
  c.r0 = (c.tile / w.MT) * w.PR;
  c.rows = min(w.PR, w.T - c.r0);
  c.ng = (c.rows + tc::BN - 1) / tc::BN;
  return true;
}

__global__ void __launch_bounds__(tc::THREADS, 1)
gemm_tc_kernel(const __grid_constant__ CUtensorMap wmap, const __grid_constant__ CUtensorMap xmap_l,
               const __grid_constant__ CUtensorMap xmap_m, const __grid_constant__ CUtensorMap xmap_s,
               float* __restrict__ part, const int32_t* __restrict__ meta, int per_idx, int T_max, int N, int MT,
               int KB, int box_l, int box_m, int* err, unsigned long long wait_ns) {
  using namespace tc;
  // a dependent launch: the rows and the plan come from the kernel before
  wait_for_prior_grid();
  dependents_may_launch();
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + RING_BYTES);
  uint64_t* empty = full + MAX_STAGES;
  uint64_t* tfull = empty + MAX_STAGES;   // [2]
  uint64_t* tempty = tfull + 2;           // [2]
  uint64_t* mma_done = tempty + 2;
  uint32_t* tmem_base_sm = reinterpret_cast<uint32_t*>(mma_done + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_base_sm + 1);
  int* consumed_sm = reinterpret_cast<int*>(tmem_base_sm + 2);

  const TcWork w = tc_work(meta, per_idx, MT, KB, T_max);
  if (w.per <= 0 || (w.waves == 0 && w.lo >= w.hi)) return;
  const int S = w.stages;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int producer_issued = 0;
  if (threadIdx.x == 0) {
    for (int s = 0; s < MAX_STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], 4);
    }
    mbar_init(mma_done, 1);
    *abort_flag = 0;
    *consumed_sm = 0;
    fence_barrier_init();
  }
  if (warp == 1) tmem_alloc(tmem_base_sm, TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_base_sm;

  if (warp == 0) {
    // ------------------------------ TMA producer ------------------------------
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int issued = 0;
      bool ok = true;
      const uint64_t pol_w = l2_policy_evict_first();
      int wave = 0, pos = w.lo;
      TcPiece c;
      while (ok && tc_next(w, wave, pos, c)) {
        const int rows16 = (c.rows + 15) / 16 * 16;
        for (int kb = c.kb0; kb < c.kb1; ++kb) {
          if (!wait_or_abort(&empty[stage], phase ^ 1u, abort_flag, err, 2, wait_ns)) { ok = false; break; }
          uint8_t* sa = smem + stage * w.stage_bytes;
          mbar_arrive_expect_tx(&full[stage], (uint32_t)(A_BYTES + rows16 * BK * 2));
          tma_load_2d_hint(sa, &wmap, &full[stage], kb * BK, c.m_tile * BM, pol_w);
          // the pass's rows in the largest boxes that fit (all multiples of 16)
          for (int r = 0; r < rows16;) {
            const int left = rows16 - r;
            const CUtensorMap* map = left >= box_l ? &xmap_l : (left >= box_m ? &xmap_m : &xmap_s);
            const int n = left >= box_l ? box_l : (left >= box_m ? box_m : 16);
            tma_load_2d(sa + A_BYTES + r * BK * 2, map, &full[stage], kb * BK, c.r0 + r);
            r += n;
          }
          ++issued;
          if (++stage == S) { stage = 0; phase ^= 1u; }
        }
      }
      producer_issued = issued;
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------ MMA issuer ------------------------------
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int buf = 0;
      uint32_t buf_phase = 0;
      int consumed = 0;
      bool ok = true;
      int wave = 0, pos = w.lo;
      TcPiece c;
      while (ok && tc_next(w, wave, pos, c)) {
        if (!wait_or_abort(&tempty[buf], buf_phase ^ 1u, abort_flag, err, 4, wait_ns)) break;
        tc_fence_after();
        for (int kb = c.kb0; kb < c.kb1; ++kb) {
          if (!wait_or_abort(&full[stage], phase, abort_flag, err, 5, wait_ns)) { ok = false; break; }
          tc_fence_after();
          const uint32_t sa = smem_u32(smem + stage * w.stage_bytes);
          const uint64_t adesc = sdesc_sw128(sa);
          for (int g = 0; g < c.ng; ++g) {
            const int rows_g = min(BN, c.rows - g * BN);
            const uint32_t idesc = idesc_bf16(BM, (rows_g + 15) / 16 * 16);
            const uint64_t bdesc = sdesc_sw128(sa + A_BYTES + g * BN * BK * 2);
            const uint32_t d_tmem = tmem_base + (uint32_t)((buf + g) * BN);
#pragma unroll
            for (int j = 0; j < BK / 16; ++j)   // 16 bf16 = 32 bytes of K per instruction
              tc_mma_bf16(d_tmem, adesc + (uint64_t)(j * 2), bdesc + (uint64_t)(j * 2), idesc,
                          (kb > c.kb0 || j > 0) ? 1u : 0u);
          }
          tc_commit(&empty[stage]);       // stage is free once these MMAs have read it
          ++consumed;
          if (++stage == S) { stage = 0; phase ^= 1u; }
        }
        if (!ok) break;
        tc_commit(&tfull[buf]);           // accumulators ready for the epilogue
        if (w.nbuf == 2) {
          if (++buf == 2) { buf = 0; buf_phase ^= 1u; }
        } else {
          buf_phase ^= 1u;
        }
      }
      *consumed_sm = consumed;
      // every MMA issued by this thread has completed before TMEM is released
      tc_commit(mma_done);
      mbar_wait_bounded(mma_done, 0, err, 6);
    }
    __syncwarp();
  } else {
    // ------------------------------ epilogue (warps 2..5) ------------------------------
    const int quarter = warp & 3;         // TMEM lanes [32 q, 32 q + 32) belong to warp q mod 4
    int buf = 0;
    uint32_t buf_phase = 0;
    int wave = 0, pos = w.lo;
    TcPiece c;
    while (tc_next(w, wave, pos, c)) {
      const int seg = c.seg;
      // a warp-wide decision: the TMEM loads below are warp-collective
      if (!__all_sync(0xffffffffu, wait_or_abort(&tfull[buf], buf_phase, abort_flag, err, 7, wait_ns))) break;
      tc_fence_after();
      const int f = c.m_tile * BM + quarter * 32 + lane;
      for (int g = 0; g < c.ng; ++g) {
        const int rows_g = min(BN, c.rows - g * BN);
        float* dst = part + ((size_t)seg * T_max + (size_t)(c.r0 + g * BN)) * N + f;
        const uint32_t tbase = tmem_base + ((uint32_t)(quarter * 32) << 16) + (uint32_t)((buf + g) * BN);
        for (int c0 = 0; c0 < rows_g; c0 += 16) {
          uint32_t r[16];
          tmem_ld16(tbase + (uint32_t)c0, r);
          tmem_ld_wait();
#pragma unroll
          for (int q = 0; q < 16; ++q)
            if (c0 + q < rows_g) dst[(size_t)(c0 + q) * N] = __uint_as_float(r[q]);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tempty[buf]);
      if (w.nbuf == 2) {
        if (++buf == 2) { buf = 0; buf_phase ^= 1u; }
      } else {
        buf_phase ^= 1u;
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  // After an abort, copies issued but never consumed may still be in flight:
  // wait for them (bounded) so that none lands after this CTA has exited.
  if (warp == 0 && lane == 0 && *abort_flag)
    for (int i = *consumed_sm; i < producer_issued; ++i)
      mbar_wait_bounded(&full[i % S], (uint32_t)((i / S) & 1), err, 3);
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
bool gemm_tc_supported(int K, int N) { return K % tc::BK == 0 && N % tc::BM == 0 && K >= tc::BK; }

// Upper bound of the segment count of any tile: a CTA range covers at least
// ceil(MT * KB / GRID) k-blocks, so a tile of KB k-blocks meets at most
// ceil(GRID / MT) + 1 ranges.
int gemm_tc_splits(int /*T_max*/, int N, int /*K*/) { return gemm_tc_slots(N); }

cudaError_t launch_gemm_tc(const void* X, const void* W, float* part, const int32_t* meta, int T_max, int N, int K,
                           int per_idx, int* err, cudaStream_t st) {
  using namespace tc;
  CUtensorMap wmap, xmap_l, xmap_m, xmap_s;
  {
    const uint64_t dims[2] = {(uint64_t)K, (uint64_t)N};
    const uint64_t strides[1] = {(uint64_t)K * 2};
    const uint32_t box[2] = {BK, BM};
    if (!encode_tensor_map(&wmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(W), dims, strides, box,
                           CU_TENSOR_MAP_SWIZZLE_128B))
      return cudaErrorNotSupported;
  }
  // row boxes of 256 (or all of a small T_max), 64 and 16 rows
  const int t16 = (T_max + 15) / 16 * 16;
  const int box_l = std::min(BN, t16), box_m = std::min(64, t16);
  {
    const uint64_t dims[2] = {(uint64_t)K, (uint64_t)T_max};
    const uint64_t strides[1] = {(uint64_t)K * 2};
    const uint32_t bl[2] = {BK, (uint32_t)box_l}, bm[2] = {BK, (uint32_t)box_m}, bs[2] = {BK, 16};
    if (!encode_tensor_map(&xmap_l, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(X), dims, strides, bl,
                           CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_tensor_map(&xmap_m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(X), dims, strides, bm,
                           CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_tensor_map(&xmap_s, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(X), dims, strides, bs,
                           CU_TENSOR_MAP_SWIZZLE_128B))
      return cudaErrorNotSupported;
  }
  static SmemOptIn opt_in;
  cudaError_t e = opt_in.ensure(gemm_tc_kernel, SMEM_BYTES);
  if (e != cudaSuccess) return e;
  e = launch_dependent(gemm_tc_kernel, dim3(GRID), dim3(THREADS), SMEM_BYTES, st, wmap, xmap_l, xmap_m, xmap_s, part,
                       meta, per_idx, T_max, N, N / BM, K / BK, box_l, box_m, err, wait_limit_ns());
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace dflash
