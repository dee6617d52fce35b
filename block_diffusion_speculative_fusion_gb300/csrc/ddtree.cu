// DDTree kernels (speculative-decoding page, section 6): the per-position
// top-K of the draft's marginals (6.1), the best-first tree within a node
// budget (6.3), and the greedy walk of the verified tree (6.5).
//
//   ddtree_topk_kernel    one CTA per draft row: one coalesced pass for the
//                         row's log-sum-exp and the threads' maxima (the K-th
//                         largest of which bounds the row's K-th value from
//                         below), a second pass collecting the values above
//                         that bound, K block rounds over the collected ones
//   ddtree_build_kernel   one warp per sequence: the candidate frontier as
//                         64-bit order keys in shared memory, each pop a
//                         warp-wide minimum (each lane loads 8 of its slots at
//                         once, then two hardware warp reductions, high word
//                         then low word); siblings enter lazily (a node's
//                         next sibling is pushed when it pops), which pops the
//                         same nodes in the same order as pushing all K
//   ddtree_verify_kernel  argmax of every node's target row (chunks, one wave)
//                         and, in the last CTA of a sequence (completion
//                         ticket), the walk from the root
#include <algorithm>

#include "common.cuh"
#include "internal.h"
#include "stream.cuh"

namespace dflash {

// (value, index) order of the top-K: larger value first, then lower index
__device__ __forceinline__ bool tk_better(float v, int i, float w, int j) { return v > w || (v == w && i < j); }

// Candidates of one row's top-K: a lower bound t0 on the row's K-th largest
// value is the K-th largest of the threads' maxima (K threads hold a value at
// least that large); the values >= t0 are collected in shared memory and the K
// best are taken from them. Rows whose values >= t0 overflow the buffer (mass
// ties) take K block-wide passes instead.
constexpr int kTopkCap = 2048;

template <typename T>
__global__ void __launch_bounds__(kThreads)
ddtree_topk_kernel(const T* __restrict__ z, int rows, int V, int K, float k2, int64_t* __restrict__ tok,
                   float* __restrict__ logp) {
  constexpr int N = VecTraits<T>::N;
  __shared__ float c_v[kTopkCap];
  __shared__ int c_i[kTopkCap];
  __shared__ float s_max[kThreads];
  __shared__ int s_cnt;
  __shared__ float s_t0, s_lse2;
  for (int row = blockIdx.x; row < rows; row += gridDim.x) {
    const T* zr = z + (size_t)row * V;
    // ---- pass 1: the row's log-sum-exp and every thread's max ----
    float zmax = -CUDART_INF_F;
    MS acc{-CUDART_INF_F, 0.f};
    auto raise_to = [&](float v) {
      const float m2 = ms_offset(v, k2);
      acc.s = (acc.m == -CUDART_INF_F) ? 0.f : acc.s * pow2i(acc.m - m2);
      acc.m = m2;
      zmax = v;
    };
    auto on_vec = [&](const uint4& u, int) {
      const float vm = vec_max<T>(u);
      if (vm > zmax) raise_to(vm);
      float f[N];
      unpack16<T>(u, f);
      float sum = 0.f;
#pragma unroll
      for (int q = 0; q < N; ++q) sum += ex2_ftz(fmaf(f[q], k2, -acc.m));
      acc.s += sum;
    };
    auto on_one = [&](float v, int) {
      if (v > zmax) raise_to(v);
      if (zmax != -CUDART_INF_F) acc.s += ex2_ftz(fmaf(v, k2, -acc.m));
    };
    for_range<T, 8>(zr, 0, V, on_vec, on_one);
    s_max[threadIdx.x] = zmax;
    const MS tot = block_ms(acc);
    if (threadIdx.x == 0) {
      s_lse2 = tot.m + log2f(tot.s);
      s_cnt = 0;
    }
    __syncthreads();
    // t0: the K-th largest thread max in (value desc, thread asc) order. Warp 0
    // holds the 256 maxima (lane l: threads l, l + 32, ...) and takes the best
    // one K times; a taken entry becomes (-inf, INT_MAX), behind every other.
    if (threadIdx.x < 32) {
      const int l = threadIdx.x;
      float mv[kThreads / 32];
      int mj[kThreads / 32];
#pragma unroll
      for (int u = 0; u < kThreads / 32; ++u) {
        mv[u] = s_max[l + 32 * u];
        mj[u] = l + 32 * u;
      }
      float t = -CUDART_INF_F;
      for (int r = 0; r < K; ++r) {
        float bv = -CUDART_INF_F;
        int bj = INT32_MAX;
#pragma unroll
        for (int u = 0; u < kThreads / 32; ++u)
          if (mv[u] > bv || (mv[u] == bv && mj[u] < bj)) { bv = mv[u]; bj = mj[u]; }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
          const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
          const int oj = __shfl_xor_sync(0xffffffffu, bj, o);
          if (ov > bv || (ov == bv && oj < bj)) { bv = ov; bj = oj; }
        }
        t = bv;
        if (bj != INT32_MAX && (bj & 31) == l) {
#pragma unroll
          for (int u = 0; u < kThreads / 32; ++u)
            if (mj[u] == bj) { mv[u] = -CUDART_INF_F; mj[u] = INT32_MAX; }
        }
      }
      if (l == 0) s_t0 = t;
    }
    __syncthreads();
    const float t0 = s_t0;
    // ---- pass 2: collect the values >= t0 (the row is read again, mostly from L2) ----
    auto push = [&](float v, int e) {
      const int slot = atomicAdd(&s_cnt, 1);
      if (slot < kTopkCap) { c_v[slot] = v; c_i[slot] = e; }
    };
    auto col_vec = [&](const uint4& u, int i0) {
      if (vec_max<T>(u) < t0) return;
      float f[N];
      unpack16<T>(u, f);
#pragma unroll
      for (int q = 0; q < N; ++q)
        if (f[q] >= t0) push(f[q], i0 + q);
    };
    auto col_one = [&](float v, int e) {
      if (v >= t0) push(v, e);
    };
    for_range<T, 8>(zr, 0, V, col_vec, col_one);
    __syncthreads();
    const int cnt = s_cnt;
    if (cnt <= kThreads) {
      // ---- the K best at once: each candidate's rank in (value desc, index asc)
      // order (indices are distinct), rank r < K written to slot r ----
      if ((int)threadIdx.x < cnt) {
        const float v = c_v[threadIdx.x];
        const int e = c_i[threadIdx.x];
        int rank = 0;
        for (int j = 0; j < cnt; ++j) rank += tk_better(c_v[j], c_i[j], v, e) ? 1 : 0;
        if (rank < K) {
          tok[(size_t)row * K + rank] = e;
          logp[(size_t)row * K + rank] = (v * k2 - s_lse2) * 0.6931471805599453f;
        }
      }
      for (int r = cnt + (int)threadIdx.x; r < K; r += kThreads) {   // fewer candidates than K
        tok[(size_t)row * K + r] = -1;
        logp[(size_t)row * K + r] = -CUDART_INF_F;
      }
      __syncthreads();
      continue;
    }
    // ---- the K best: K rounds of a block-wide (value desc, index asc) maximum ----
    for (int r = 0; r < K; ++r) {
      VI best{-CUDART_INF_F, INT32_MAX};
      if (cnt <= kTopkCap) {
        for (int j = threadIdx.x; j < cnt; j += kThreads)
          if (vi_better(c_v[j], c_i[j], best)) best = VI{c_v[j], c_i[j]};
      } else {
        // overflow (mass ties): a pass over the row that skips the ones taken
        const int64_t* done = tok + (size_t)row * K;
        for (int e = threadIdx.x; e < V; e += kThreads) {
          const float v = ld_scalar(zr + e);
          bool taken = false;
          for (int q = 0; q < r; ++q) taken |= (done[q] == e);
          if (!taken && vi_better(v, e, best)) best = VI{v, e};
        }
      }
      best = block_vi(best);
      __shared__ VI s_w;
      if (threadIdx.x == 0) {
        s_w = best;
        tok[(size_t)row * K + r] = best.i == INT32_MAX ? -1 : best.i;
        logp[(size_t)row * K + r] = best.i == INT32_MAX ? -CUDART_INF_F : (best.v * k2 - s_lse2) * 0.6931471805599453f;
      }
      __syncthreads();
      if (cnt <= kTopkCap)
        for (int j = threadIdx.x; j < cnt; j += kThreads)
          if (c_i[j] == s_w.i) c_v[j] = -CUDART_INF_F, c_i[j] = INT32_MAX;
      __syncthreads();
    }
  }
}

// Frontier candidates as 64-bit keys whose unsigned order is the pop order:
// high word = the path log-probability mapped to a descending unsigned order,
// low word = depth (bits 17-24), parent pop index + 1 (bits 4-16, 0 = root),
// rank (bits 0-3). Smaller key pops first: larger log-probability, then smaller
// depth, earlier parent, lower rank.
__device__ __forceinline__ uint64_t cand_key(float lp, int depth, int parent, int rank) {
  uint32_t u = __float_as_uint(lp);
  u = (u & 0x80000000u) ? ~u : (u | 0x80000000u);   // ascending with lp
  return ((uint64_t)(~u) << 32) | ((uint32_t)depth << 17) | ((uint32_t)(parent + 1) << 4) | (uint32_t)rank;
}
__device__ __forceinline__ float key_lp(uint64_t k) {
  uint32_t u = ~(uint32_t)(k >> 32);
  u = (u & 0x80000000u) ? (u & 0x7fffffffu) : ~u;
  return __uint_as_float(u);
}
__device__ __forceinline__ int key_depth(uint64_t k) { return (int)((k >> 17) & 0xff); }
__device__ __forceinline__ int key_parent(uint64_t k) { return (int)((k >> 4) & 0x1fff) - 1; }
__device__ __forceinline__ int key_rank(uint64_t k) { return (int)(k & 0xf); }

// One warp per sequence, everything warp-synchronous; the frontier (at most
// one candidate more than the nodes taken), the taken nodes' log-probs and the
// sequence's top-K table live in shared memory.
__global__ void __launch_bounds__(32)
ddtree_build_kernel(const int64_t* __restrict__ tok, const float* __restrict__ logp, int n, int K, int budget,
                    int64_t* __restrict__ node_token, int32_t* __restrict__ node_parent,
                    int32_t* __restrict__ node_depth, float* __restrict__ node_logp, int32_t* __restrict__ n_nodes,
                    uint8_t* __restrict__ flags) {
  extern __shared__ __align__(16) unsigned char tree_smem[];
  uint64_t* fr = reinterpret_cast<uint64_t*>(tree_smem);          // frontier keys, capacity budget + 1
  int64_t* tk = reinterpret_cast<int64_t*>(fr + budget + 1);     // top-K tokens [n][K]
  float* nlp = reinterpret_cast<float*>(tk + (size_t)n * K);     // taken nodes' log-probs [budget]
  float* lb = nlp + budget;                                      // top-K log-probs [n][K]
  const int b = blockIdx.x, l = threadIdx.x;
  for (int j = l; j < n * K; j += 32) {
    lb[j] = logp[(size_t)b * n * K + j];
    tk[j] = tok[(size_t)b * n * K + j];
  }
  __syncwarp();
  int f = 0;
  if (n > 0 && K > 0) {
    if (l == 0) fr[0] = cand_key(lb[0], 1, -1, 0);
    f = 1;
  }
  __syncwarp();
  int cnt = 0;
  bool tie = false;
  // Near ties: a distinct candidate within 1e-5 of a pop either pops later,
  // with all pops in between inside that gap (consecutive pops closer than
  // 1e-5 but not equal), or is still waiting when the budget runs out (checked
  // after the loop); exact ties follow the key order and are not flagged.
  float prev = CUDART_INF_F;
  while (f > 0 && cnt < budget) {
    // the first key in pop order, and its slot (keys are distinct); each lane
    // loads 8 of its slots before comparing, so the loads overlap
    uint64_t bk = ~0ull;
    int bi = -1;
    for (int j0 = l; j0 < f; j0 += 32 * 8) {
      uint64_t kk[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) kk[u] = j0 + 32 * u < f ? fr[j0 + 32 * u] : ~0ull;
#pragma unroll
      for (int u = 0; u < 8; ++u)
        if (kk[u] < bk) { bk = kk[u]; bi = j0 + 32 * u; }
    }
    {
      // warp minimum of the 64-bit keys: the high words, then the low words of
      // the lanes holding the smallest high word; the key is distinct, so one
      // lane holds it and passes on its slot
      const uint32_t hi = (uint32_t)(bk >> 32), lo = (uint32_t)bk;
      const uint32_t mhi = __reduce_min_sync(0xffffffffu, hi);
      const uint32_t mlo = __reduce_min_sync(0xffffffffu, hi == mhi ? lo : 0xffffffffu);
      const uint64_t mk = ((uint64_t)mhi << 32) | mlo;
      const unsigned who = __ballot_sync(0xffffffffu, bk == mk);
      bi = __shfl_sync(0xffffffffu, bi, who ? __ffs(who) - 1 : 0);
      bk = mk;
    }
    const float lp = key_lp(bk);
    const int depth = key_depth(bk), parent = key_parent(bk), rank = key_rank(bk);
    if (prev != lp && prev - lp < 1e-5f) tie = true;
    prev = lp;
    const bool sib = rank + 1 < K, child = depth < n;
    __syncwarp();
    if (l == 0) {
      // every shared-memory read first (the tables share one buffer with the
      // frontier, so reads after a store would wait for it)
      const uint64_t last = fr[f - 1];
      const int64_t token = tk[(depth - 1) * K + rank];
      const float plp = (sib && parent >= 0) ? nlp[parent] : 0.f;
      const float lsib = sib ? lb[(depth - 1) * K + rank + 1] : 0.f;
      const float lch = child ? lb[depth * K] : 0.f;
      const size_t o = (size_t)b * budget + cnt;
      node_token[o] = token;
      node_parent[o] = parent;
      node_depth[o] = depth;
      node_logp[o] = lp;
      nlp[cnt] = lp;
      // the taken slot takes the last candidate; then the next sibling and the first child enter
      fr[bi] = last;
      int nf = f - 1;
      if (sib) fr[nf++] = cand_key(plp + lsib, depth, parent, rank + 1);
      if (child) fr[nf++] = cand_key(lp + lch, depth + 1, cnt, 0);
    }
    f = f - 1 + (sib ? 1 : 0) + (child ? 1 : 0);
    ++cnt;
    __syncwarp();
  }
  if (f > 0 && cnt > 0) {
    // the budget ran out: the nearest distinct candidate left behind
    float v = -CUDART_INF_F;
    for (int j0 = l; j0 < f; j0 += 32 * 8) {
      uint64_t kk[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) kk[u] = j0 + 32 * u < f ? fr[j0 + 32 * u] : 0ull;
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const float x = key_lp(kk[u]);
        if (j0 + 32 * u < f && x != prev) v = fmaxf(v, x);
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    if (v != -CUDART_INF_F && prev - v < 1e-5f) tie = true;
  }
  for (int j = cnt + l; j < budget; j += 32) {
    const size_t o = (size_t)b * budget + j;
    node_token[o] = -1;
    node_parent[o] = -1;
    node_depth[o] = -1;
    node_logp[o] = 0.f;
  }
  if (l == 0) {
    n_nodes[b] = cnt;
    if (flags) flags[b] = tie ? 1 : 0;
  }
}

// Greedy walk of the verified tree: rows b * (budget + 1) + r, r = 0 the root
template <typename T>
__global__ void __launch_bounds__(kThreads, 4)
ddtree_verify_kernel(const T* __restrict__ zt, const int64_t* __restrict__ node_token,
                     const int32_t* __restrict__ node_parent, const int32_t* __restrict__ n_nodes, int budget, int V,
                     int nch, int chunk, VI* __restrict__ parts, int32_t* __restrict__ counters,
                     int32_t* __restrict__ accept_len, int64_t* __restrict__ bonus, int32_t* __restrict__ commit_len,
                     int32_t* __restrict__ path, int64_t* __restrict__ out_tokens) {
  constexpr int N = VecTraits<T>::N;
  const int R = budget + 1;
  const int c = blockIdx.x, row = blockIdx.y;
  const int b = row / R, r = row - b * R;
  const int nn = min(max(n_nodes[b], 0), budget);
  VI best{-CUDART_INF_F, INT32_MAX};
  if (r <= nn) {
    const T* z = zt + (size_t)row * V;
    const int e0 = c * chunk, e1 = min(V, e0 + chunk);
    auto on_vec = [&](const uint4& u, int i0) {
      const float vm = vec_max<T>(u);
      if (vm > best.v || (vm == best.v && i0 < best.i)) {
        float f[N];
        unpack16<T>(u, f);
#pragma unroll
        for (int j = N - 1; j >= 0; --j)
          if (f[j] == vm) best = VI{vm, i0 + j};
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

  // ---- last CTA of sequence b: the target's prediction at every node, then the walk ----
  extern __shared__ int32_t tp[];   // [R]
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  for (int rr = w; rr <= nn; rr += blockDim.x >> 5) {
    VI x{-CUDART_INF_F, INT32_MAX};
    const VI* pr = parts + ((size_t)b * R + rr) * nch;
    for (int cc = l; cc < nch; cc += 32) {
      const int2 raw = __ldcg(reinterpret_cast<const int2*>(pr + cc));
      const VI y{__int_as_float(raw.x), raw.y};
      if (vi_better(y.v, y.i, x)) x = y;
    }
    x = warp_vi(x);
    if (l == 0) tp[rr] = (x.i == INT32_MAX) ? 0 : x.i;
  }
  __shared__ int s_next;
  __syncthreads();
  int cur = -1, a = 0;
  const int64_t* ntb = node_token + (size_t)b * budget;
  const int32_t* npb = node_parent + (size_t)b * budget;
  while (true) {
    const int t = tp[cur + 1];
    if (threadIdx.x == 0) s_next = INT32_MAX;
    __syncthreads();
    // the child of cur holding the target's token (siblings hold distinct tokens)
    for (int j = threadIdx.x; j < nn; j += blockDim.x)
      if (npb[j] == cur && ntb[j] == (int64_t)t) atomicMin(&s_next, j);
    __syncthreads();
    const int nxt = s_next;
    __syncthreads();
    if (nxt == INT32_MAX) break;
    if (threadIdx.x == 0) {
      if (path) path[(size_t)b * budget + a] = nxt;
      if (out_tokens) out_tokens[(size_t)b * R + a] = t;
    }
    ++a;
    cur = nxt;
  }
  const int bt = tp[cur + 1];
  if (threadIdx.x == 0) {
    accept_len[b] = a;
    commit_len[b] = a + 1;
    bonus[b] = bt;
  }
  for (int j = a + threadIdx.x; j < R; j += blockDim.x) {
    if (out_tokens) out_tokens[(size_t)b * R + j] = j == a ? (int64_t)bt : -1;
    if (path && j < budget) path[(size_t)b * budget + j] = -1;
  }
  reset_ticket(&counters[b]);
}

// ---------------------------------------------------------------------------
// Host launchers
// ---------------------------------------------------------------------------
template <typename T>
static cudaError_t launch_topk_t(const TreeArgs& a) {
  const int rows = a.B * a.n;
  const int grid = std::min(rows, 4 * a.num_sms);
  const float k2 = kLog2e / a.temperature;
  ddtree_topk_kernel<T><<<grid, kThreads, 0, a.stream>>>((const T*)a.logits, rows, a.V, a.K, k2, a.topk_tok,
                                                        a.topk_logp);
  return cudaGetLastError();
}

cudaError_t launch_ddtree_topk(const TreeArgs& a) {
  return a.dtype == 0 ? launch_topk_t<float>(a) : launch_topk_t<bf16>(a);
}

size_t ddtree_build_smem(int budget, int n, int K) {
  return (size_t)(budget + 1) * 8 + (size_t)n * K * 8 + (size_t)budget * 4 + (size_t)n * K * 4;
}

cudaError_t launch_ddtree_build(const TreeArgs& a) {
  const size_t smem = ddtree_build_smem(a.budget, a.n, a.K);
  static SmemOptIn opt_in;
  if (smem > 48 * 1024) {
    cudaError_t e = opt_in.ensure(ddtree_build_kernel, smem);
    if (e != cudaSuccess) return e;
  }
  ddtree_build_kernel<<<a.B, 32, smem, a.stream>>>(a.topk_tok, a.topk_logp, a.n, a.K, a.budget, a.node_token,
                                                   a.node_parent, a.node_depth, a.node_logp, a.n_nodes, a.flags);
  return cudaGetLastError();
}

size_t ddtree_verify_ws_bytes(int B, int budget, int V, int dtype, int num_sms) {
  ChunkPlan p = plan_chunks(B * (budget + 1), V, dtype, num_sms);
  return (size_t)B * (budget + 1) * p.nch * sizeof(VI);
}

template <typename T>
static cudaError_t launch_tree_verify_t(const TreeArgs& a) {
  const int R = a.budget + 1;
  ChunkPlan p = plan_chunks(a.B * R, a.V, a.dtype, a.num_sms);
  dim3 grid(p.nch, a.B * R);
  ddtree_verify_kernel<T><<<grid, kThreads, (size_t)R * sizeof(int32_t), a.stream>>>(
      (const T*)a.logits, a.node_token, a.node_parent, a.n_nodes, a.budget, a.V, p.nch, p.chunk, (VI*)a.scratch,
      a.counters, a.accept_len, a.bonus, a.commit_len, a.path, a.out_tokens);
  return cudaGetLastError();
}

cudaError_t launch_ddtree_verify(const TreeArgs& a) {
  return a.dtype == 0 ? launch_tree_verify_t<float>(a) : launch_tree_verify_t<bf16>(a);
}

}  // namespace dflash
