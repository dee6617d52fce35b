// Internal interface between the C ABI layer (api.cu) and the kernel files.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <mutex>

namespace dflash {

inline size_t align_up(size_t x, size_t a = 256) { return (x + a - 1) / a * a; }

// Limit in nanoseconds of the bounded waits on work barriers in the
// tensor-core kernels (attention, context GEMMs); read at each launch.
// Default 2 s; dflash_set_wait_limit_ns changes it for the whole process.
unsigned long long wait_limit_ns();

// Device error word code: a page-table entry outside [0, num_pages) inside a
// context (attention reads page 0 for it).
constexpr int kDevErrBadPage = 100;
constexpr int kDevErrBadNDraft = 101;
constexpr int kDevErrBadCtxLen = 102;      // recorded in DFLASH_DEBUG builds only
constexpr int kDevErrBadCommitLen = 103;   // recorded in DFLASH_DEBUG builds only
constexpr int kDevErrBadPosition = 104;    // recorded in DFLASH_DEBUG builds only

// Record an input error in the workspace error word (the first code stays).
__device__ __forceinline__ void record_dev_error(int* err, int code) {
  if (err) atomicCAS(err, 0, code);
}

// Opt a kernel into `bytes` of dynamic shared memory on the calling thread's
// current device. The attribute belongs to each device's context, so it is set
// once per device (and again only to raise it), under a lock so that concurrent
// callers cannot lower it for each other. One object per kernel.
class SmemOptIn {
 public:
  template <class Kernel>
  cudaError_t ensure(Kernel* kernel, size_t bytes) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const bool tracked = dev >= 0 && dev < kDevices;
    std::lock_guard<std::mutex> lock(mu_);
    if (tracked && bytes <= set_[dev]) return cudaSuccess;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
    if (e == cudaSuccess && tracked) set_[dev] = bytes;
    return e;
  }

 private:
  static constexpr int kDevices = 64;
  std::mutex mu_;
  size_t set_[kDevices] = {};
};

struct ChunkPlan {
  int chunk;   // elements per chunk (multiple of one 16-byte vector per thread)
  int nch;     // chunks per row
};

ChunkPlan plan_chunks(int rows, int V, int dtype, int num_sms);

// ---------------------------------------------------------------- verify ---
struct VerifyArgs {
  int B, n_max, V, dtype;
  float temperature;
  const void* target_logits;
  const void* draft_logits;
  const int64_t* cand;
  const int32_t* n_draft;
  const float* u_accept;
  const float* u_final;
  const float* draft_lse;   // [B, n_max] LSE(draft row / T), or null (streamed)
  int32_t* accept_len;
  int64_t* bonus;
  int32_t* commit_len;
  int64_t* out_tokens;
  int64_t* target_pred;
  uint8_t* flags;
  float* probs;
  int32_t* counters;   // zeroed region at the workspace start
  int* err;            // the workspace's error word
  void* scratch;       // workspace after the counter region
  cudaStream_t stream;
};

size_t verify_greedy_ws_bytes(int B, int n_max, int V, int dtype, int num_sms);
size_t verify_sample_ws_bytes(int B, int n_max, int V, int dtype, int num_sms);
cudaError_t launch_verify_greedy(const VerifyArgs& a, int num_sms);
cudaError_t launch_verify_sample(const VerifyArgs& a, int num_sms);

// ------------------------------------------------------------------ gate ---
// Where a gate call finds its rows: sequence b's i-th row of the stage is row
// z_row0 + i of z_rows rows of that sequence; its token is tokens[b *
// tok_stride + tok0 + i]; its LSE goes to row_lse[b * lse_stride + lse0 + i].
// The plain gate is z_rows = tok_stride = lse_stride = k and zero offsets.
struct GateLayout {
  int z_rows, z_row0, tok_stride, tok0, lse_stride, lse0;
  int lse_inactive;   // 1: row LSEs of inactive sequences are computed too
};

struct GateArgs {
  int B, k, V, dtype;
  GateLayout layout;
  int32_t* n_verify;  // [B] or nullptr: += k for every active sequence
  float temperature, g;
  const void* draft_logits;
  const int64_t* tokens;
  const uint8_t* active;
  float* c_s;
  uint8_t* cont;
  float* row_lse;
  uint8_t* flags;
  int32_t* counters;
  void* scratch;
  cudaStream_t stream;
};

size_t gate_ws_bytes(int B, int k, int V, int dtype, int num_sms);
cudaError_t launch_gate(const GateArgs& a, int num_sms);

// Draft-side token choice over the MASK rows (argmax or one inverse-CDF sample
// per row, with q(x) and the row's log-sum-exp).
struct DraftSelectArgs {
  int B, n_max, V, dtype;
  float temperature;          // 0: argmax
  const void* draft_logits;   // [B, n_max, V]
  const int64_t* anchor;      // [B]
  const int32_t* n_draft;     // [B] or null
  const float* u_draft;       // [B, n_max] (sampled)
  int64_t* cand;              // [B, n_max + 1]
  float* q_x;                 // [B, n_max] or null
  float* row_lse;             // [B, n_max] or null
  uint8_t* flags;             // [B, n_max] or null
  int32_t* counters;          // zeroed region at the workspace start, one per row
  int* err;                   // the workspace's error word
  void* scratch;
  cudaStream_t stream;
  int num_sms;                // persistent grid: resident CTAs x SMs
};
constexpr int kSelMaxVocab = 1024 * 256 * 32;   // chunks x tokens per chunk (fp32)
size_t draft_select_ws_bytes(int B, int n_max, int V, int dtype);
cudaError_t launch_draft_select(const DraftSelectArgs& a);

// DDTree: per-position top-K, best-first tree within a node budget, greedy walk.
constexpr int kTreeMaxK = 16;
constexpr int kTreeMaxBudget = 4096;
struct TreeArgs {
  int B, n, V, dtype, K, budget;
  float temperature;
  const void* logits;         // topk: draft logits [B, n, V]; verify: target logits [B, budget + 1, V]
  int64_t* topk_tok;          // [B, n, K]
  float* topk_logp;           // [B, n, K]
  int64_t* node_token;        // [B, budget]
  int32_t* node_parent;       // [B, budget]
  int32_t* node_depth;        // [B, budget]
  float* node_logp;           // [B, budget]
  int32_t* n_nodes;           // [B]
  uint8_t* flags;             // [B] or null
  int32_t* accept_len;        // [B]
  int64_t* bonus;             // [B]
  int32_t* commit_len;        // [B]
  int32_t* path;              // [B, budget] or null
  int64_t* out_tokens;        // [B, budget + 1] or null
  int32_t* counters;          // zeroed region at the workspace start
  void* scratch;
  cudaStream_t stream;
  int num_sms;
};
cudaError_t launch_ddtree_topk(const TreeArgs& a);
size_t ddtree_build_smem(int budget, int n, int K);
cudaError_t launch_ddtree_build(const TreeArgs& a);
size_t ddtree_verify_ws_bytes(int B, int budget, int V, int dtype, int num_sms);
cudaError_t launch_ddtree_verify(const TreeArgs& a);

// ------------------------------------------------------------- attention ---
struct AttnArgs {
  int B, n_q, n_kv, Hq, Hkv, D, page_size, max_pages, num_pages, max_ctx, dtype;
  int causal;   // 1: query i sees block rows j <= i + n_kv - n_q
  const void* q;
  const void* k_blk;
  const void* v_blk;
  const void* k_pool;
  const void* v_pool;
  const int32_t* page_table;
  const int32_t* ctx_len;
  const uint8_t* active;   // [B] or null: sequences with 0 are skipped
  float scale;
  void* out;
  int* err;
  void* scratch;
  cudaStream_t stream;
};

size_t attn_ws_bytes(int B, int n_q, int n_kv, int Hq, int Hkv, int D, int max_ctx, int page_size, int dtype);
cudaError_t launch_block_attn(const AttnArgs& a, int* launches);

// ----------------------------------------------------------- materialise ---
constexpr int kMaxLayers = 16;
struct MatPools {
  void* k[kMaxLayers];
  void* v[kMaxLayers];
};

struct MatArgs {
  int B, rows_max, m, d, L, Hkv, D, page_size, max_pages, num_pages, dtype;
  const void* hidden;
  const int32_t* commit_len;
  const int32_t* start_pos;
  const void* W_f;
  const void* b_f;
  const void* W_kv;
  const void* k_norm_w;
  float rms_eps, rope_theta;
  MatPools pools;
  const int32_t* page_table;
  int32_t* new_len;
  int32_t* counters;
  int* err;
  void* scratch;
  cudaStream_t stream;
};

struct MatPlan {
  int B, T_max, K1, N1, K2, N2, S1, S2;
  bool tc;   // GEMMs on tcgen05 tensor cores
};

MatPlan mat_plan(int B, int rows_max, int m, int d, int L, int Hkv, int D, int dtype);
size_t mat_ws_bytes(const MatPlan& p, int dtype);
cudaError_t launch_materialize(const MatArgs& a, int* launches);

// tcgen05 GEMM: part[seg][t][n] = sum over one K segment of X[t][k] W[n][k], bf16 in, fp32 out.
namespace tcplan {
constexpr int BM = 128;      // output features per tile (MMA M)
constexpr int BN = 256;      // rows per MMA group (MMA N upper bound)
constexpr int BP = 512;      // rows per tile at most: two MMA groups share each weight k-block
constexpr int BK = 64;       // K per k-block: one 128-byte swizzle atom of bf16
constexpr int GRID = 152;    // persistent CTAs: one per SM of a GB300
constexpr int MIN_PER = 8;   // smallest k-block range per CTA
}  // namespace tcplan

// Rows per tile for T rows: all of them as two MMA groups sharing each weight
// k-block when they fit one tile (decode-sized commits read every weight byte
// once), else 256 (one group per tile, which leaves room for a deeper ring).
inline __host__ __device__ int gemm_tc_pass_rows(int T) { return T <= tcplan::BP ? tcplan::BP : tcplan::BN; }
// Tiles of a GEMM over T rows: N/BM x ceil(T/rows per tile). When the rows
// take more than one pass and there are at least GRID tiles, whole waves of
// GRID tiles are handed out one per CTA (the CTAs of a wave then work on a few
// passes at once and share their rows and weights in L2); the rest are split
// over the CTAs in contiguous k-block ranges (stream-K).
inline __host__ __device__ int gemm_tc_tiles(int T, int N) {
  const int PR = gemm_tc_pass_rows(T);
  return (N / tcplan::BM) * ((T + PR - 1) / PR);
}
inline __host__ __device__ int gemm_tc_full_tiles(int T, int N) {
  if (T <= gemm_tc_pass_rows(T)) return 0;
  return (gemm_tc_tiles(T, N) / tcplan::GRID) * tcplan::GRID;
}
// Partial-sum slots per output element: ceil(GRID / MT) + 1.
inline __host__ __device__ int gemm_tc_slots(int N) {
  const int MT = N / tcplan::BM;
  return (tcplan::GRID + MT - 1) / MT + 1;
}
// k-block range per CTA over the split tiles; at least KB / (slots - 1), so
// that no tile spans more segments than there are slots.
inline __host__ __device__ int gemm_tc_per(int T, int N, int K) {
  const int KB = K / tcplan::BK, S = gemm_tc_slots(N);
  const long rem = (long)(gemm_tc_tiles(T, N) - gemm_tc_full_tiles(T, N)) * KB;
  long per = (rem + tcplan::GRID - 1) / tcplan::GRID;
  const long floor_per = (KB + S - 2) / (S - 1);
  if (per < floor_per) per = floor_per;
  if (per < tcplan::MIN_PER) per = tcplan::MIN_PER;
  return (int)per;
}
// Number of K segments (CTA ranges) that split tile `tile` (counted from the
// first split tile) spans.
inline __host__ __device__ int gemm_tc_tile_segs(int tile, int KB, int per) {
  return ((tile + 1) * KB - 1) / per - (tile * KB) / per + 1;
}
// Which partial-sum slots hold an output element's sums: the per-call
// constants of a GEMM over T rows with segment rule `per` (0: fixed S splits),
// taken once per thread, and the count for element (t, n).
struct SegRule {
  int per, S, PR, MT, KB, full;
};
inline __host__ __device__ SegRule seg_rule(int N, int K, int per, int S, int T) {
  SegRule r;
  r.per = per;
  r.S = S;
  r.PR = gemm_tc_pass_rows(T);
  r.MT = N / tcplan::BM;
  r.KB = K / tcplan::BK;
  r.full = per > 0 ? gemm_tc_full_tiles(T, N) : 0;
  return r;
}
inline __host__ __device__ int seg_count(const SegRule& r, int t, int n) {
  if (r.per <= 0) return r.S;
  const int tile = (t / r.PR) * r.MT + n / tcplan::BM;
  if (tile < r.full) return 1;
  return gemm_tc_tile_segs(tile - r.full, r.KB, r.per);
}

bool gemm_tc_supported(int K, int N);
int gemm_tc_splits(int T_max, int N, int K);
cudaError_t launch_gemm_tc(const void* X, const void* W, float* part, const int32_t* meta, int T_max, int N,
                           int K, int per_idx, int* err, cudaStream_t st);

}  // namespace dflash
