/*
 * Host-side cost of one call through the C ABI of libdflash, measured from C:
 * the wall-clock time a call takes to validate its arguments and enqueue its
 * kernels (no synchronisation inside the timed loop), per entry point, on
 * small problems whose device time is negligible next to the host time.
 * Prints one JSON object. Measurement harness only (it allocates its own
 * device buffers with cudaMalloc); the library itself allocates nothing.
 */
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdio.h>
#include <string.h>
#include <time.h>

#include "../../include/dflash.h"

static double now_us(void) {
  struct timespec ts;
  clock_gettime(CLOCK_MONOTONIC, &ts);
  return ts.tv_sec * 1e6 + ts.tv_nsec * 1e-3;
}

static void* dzero(size_t bytes) {
  void* p = NULL;
  if (cudaMalloc(&p, bytes ? bytes : 16) != cudaSuccess) return NULL;
  cudaMemset(p, 0, bytes ? bytes : 16);
  return p;
}

#define BATCH 64
#define ROUNDS 20

int main(void) {
  cudaStream_t s;
  if (cudaStreamCreate(&s) != cudaSuccess) { printf("{\"error\": \"no CUDA device\"}\n"); return 1; }
  int rc = 0;
  double t_greedy = 0, t_attn = 0, t_mat = 0;

  /* greedy verify: B = 1, 3 drafts, V = 1000, fp32 */
  {
    dflash_verify_dims d = {1, 3, 1000, DFLASH_F32};
    const size_t ws_bytes = dflash_verify_greedy_workspace_size(&d);
    void* logits = dzero(4 * 1000 * 4);
    int64_t* cand = (int64_t*)dzero(4 * 8);
    int32_t *acc = (int32_t*)dzero(4), *commit = (int32_t*)dzero(4);
    int64_t* bonus = (int64_t*)dzero(8);
    void* ws = dzero(ws_bytes);
    for (int r = 0; r < ROUNDS; ++r) {
      cudaStreamSynchronize(s);
      const double t0 = now_us();
      for (int i = 0; i < BATCH; ++i)
        rc |= dflash_verify_greedy(&d, logits, cand, NULL, acc, bonus, commit, NULL, NULL, ws, ws_bytes, s);
      t_greedy += now_us() - t0;
    }
  }
  /* block attention: B = 1, 16 queries x 32 heads, 8 kv heads, D = 128, 16-token
   * pages, 64 context rows, bf16 (the tensor-core path: four tensor maps per call) */
  {
    dflash_attn_dims d = {1, 16, 16, 32, 8, 128, 16, 8, 8, 128, DFLASH_BF16, 0};
    const size_t ws_bytes = dflash_block_attn_workspace_size(&d);
    void* q = dzero(16 * 32 * 128 * 2);
    void* kb = dzero(16 * 8 * 128 * 2);
    void* vb = dzero(16 * 8 * 128 * 2);
    void* kp = dzero(8 * 16 * 8 * 128 * 2);
    void* vp = dzero(8 * 16 * 8 * 128 * 2);
    int32_t pt_h[8] = {0, 1, 2, 3, 4, 5, 6, 7}, cl_h[1] = {64};
    int32_t* pt = (int32_t*)dzero(sizeof(pt_h));
    int32_t* cl = (int32_t*)dzero(sizeof(cl_h));
    cudaMemcpy(pt, pt_h, sizeof(pt_h), cudaMemcpyHostToDevice);
    cudaMemcpy(cl, cl_h, sizeof(cl_h), cudaMemcpyHostToDevice);
    void* out = dzero(16 * 32 * 128 * 2);
    void* ws = dzero(ws_bytes);
    for (int r = 0; r < ROUNDS; ++r) {
      cudaStreamSynchronize(s);
      const double t0 = now_us();
      for (int i = 0; i < BATCH; ++i)
        rc |= dflash_block_attn(&d, q, kb, vb, kp, vp, pt, cl, 0.08838834764831845f, out, ws, ws_bytes, s);
      t_attn += now_us() - t0;
    }
  }
  /* materialisation: B = 1, 4 rows, m = 5, d = 256, 1 draft layer of 1 kv head,
   * D = 128, bf16 (two tensor-core GEMMs: six tensor maps per call) */
  {
    dflash_ctx_kv_dims d = {1, 4, 5, 256, 1, 1, 128, 16, 1, 1, DFLASH_BF16};
    const size_t ws_bytes = dflash_materialize_workspace_size(&d);
    void* hidden = dzero(4 * 5 * 256 * 2);
    int32_t c_h[1] = {4};
    int32_t* commit = (int32_t*)dzero(4);
    int32_t* start = (int32_t*)dzero(4);
    cudaMemcpy(commit, c_h, 4, cudaMemcpyHostToDevice);
    void* wf = dzero(256 * 1280 * 2);
    void* wkv = dzero(2 * 128 * 256 * 2);
    void* kpool = dzero(16 * 128 * 2);
    void* vpool = dzero(16 * 128 * 2);
    void* kps[1] = {kpool};
    void* vps[1] = {vpool};
    int32_t* pt = (int32_t*)dzero(4);
    void* ws = dzero(ws_bytes);
    for (int r = 0; r < ROUNDS; ++r) {
      cudaStreamSynchronize(s);
      const double t0 = now_us();
      for (int i = 0; i < BATCH; ++i)
        rc |= dflash_materialize_ctx_kv(&d, hidden, commit, start, wf, NULL, wkv, NULL, 1e-6f, 0.f, kps, vps, pt,
                                        NULL, ws, ws_bytes, s);
      t_mat += now_us() - t0;
    }
  }
  cudaStreamSynchronize(s);
  const double n = (double)BATCH * ROUNDS;
  printf("{\"verify_greedy_us\": %.3f, \"block_attn_us\": %.3f, \"materialize_ctx_kv_us\": %.3f, "
         "\"calls_each\": %d, \"status\": %d, \"error\": \"%s\"}\n",
         t_greedy / n, t_attn / n, t_mat / n, BATCH * ROUNDS, rc, rc ? dflash_last_error() : "");
  return rc ? 1 : 0;
}
