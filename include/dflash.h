/*
 * dflash.h -- C ABI of the GB300 (sm_103a) DFlash hot path.
 *
 * Five operations of one block-diffusion speculative-decoding step, each a
 * hand-written CUDA kernel sequence:
 *   dflash_materialize_ctx_kv  target-context K/V materialisation into the paged
 *                              draft KV cache of every draft layer
 *   dflash_block_attn          the draft block's bidirectional (unmasked) GQA
 *                              attention over [context K/V ; block K/V]
 *   dflash_verify_greedy       the greedy accept rule over the vocabulary
 *   dflash_verify_sample       the min(1, p/q) accept rule with residual resample
 *   dflash_gate                the DLoop block gate c_s >= g
 *
 * Conventions shared by every call:
 *   - Tensor arguments are DEVICE pointers owned by the caller; the library
 *     never allocates, frees or keeps them. Shapes are row-major with the last
 *     dimension contiguous, as stated per argument.
 *   - Scratch memory is a caller-owned device workspace of at least
 *     dflash_*_workspace_size(dims) bytes, 256-byte aligned. Its first
 *     DFLASH_WS_COUNTER_BYTES bytes hold completion counters: they must be zero
 *     before a workspace is first used (e.g. allocate it zeroed) and every call
 *     that completes leaves them zero again. One workspace may serve any number
 *     of calls issued in order on one stream; calls that overlap on the GPU
 *     must use different workspaces.
 *   - Every call is asynchronous on the given stream and performs no host
 *     synchronisation. Outputs are valid once the stream reaches that point.
 *     A call's first kernel is an ordinary launch, so it starts after all
 *     earlier work in the stream; a call's later kernels (the attention split
 *     merge, the materialisation's GEMMs, bias and epilogue, the sampled
 *     draw) are programmatic dependent launches that may become resident
 *     while the kernel before them runs but read nothing until it completes.
 *   - Return value: DFLASH_OK, or an error code with a message available from
 *     dflash_last_error() (thread-local). Argument errors are detected on the
 *     host before anything is launched; DFLASH_ERR_CUDA reports a launch error.
 *   - dtype selects the element type of every floating-point tensor of the
 *     call: DFLASH_F32 (float) or DFLASH_BF16 (bfloat16). Accumulation is fp32.
 *
 * Citations name the source page and its section:
 *   [DFlash]  "DFlash 块扩散解码：以并行扩散替代自回归草稿" -- sections 块扩散,
 *             KV 注入, 验证流程.
 *   [SGLang]  "详解SGlang 最新DFlash投机解码算法的工程实现" -- section 3 (decode,
 *             greedy rule), 4.1 (KV materialisation), 5.1 (KV headroom).
 *   [SpecDec] "让大模型快 8 倍：从投机解码到 DDTree" -- sections 3 and 4.
 *   [DLoop]   "DLoop 完全拆解" -- 机制一 (confidence gate) and the looped verify.
 */
#ifndef DFLASH_H
#define DFLASH_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t; NULL is the legacy default stream. */
typedef struct CUstream_st* dflash_stream_t;

enum {
  DFLASH_OK = 0,
  DFLASH_ERR_INVALID_ARG = 1,   /* null pointer, bad size, inconsistent shape */
  DFLASH_ERR_UNSUPPORTED = 2,   /* valid but outside the compiled kernels */
  DFLASH_ERR_WORKSPACE = 3,     /* workspace too small or misaligned */
  DFLASH_ERR_CUDA = 4           /* a CUDA launch or API call failed */
};

enum { DFLASH_F32 = 0, DFLASH_BF16 = 1 };

/* Bits of the per-sequence flags of dflash_verify_sample. A flagged sequence's
 * integer outputs are valid draws but may differ from an exact-arithmetic
 * evaluation, because a uniform sat within 1e-6 of a decision boundary. */
enum {
  DFLASH_FLAG_ACCEPT_BOUNDARY = 1,  /* |u - p(x)/q(x)| < 1e-6 at an evaluated test */
  DFLASH_FLAG_CDF_BOUNDARY = 2,     /* u_final within 1e-6 of a CDF step */
  DFLASH_FLAG_DEGENERATE = 4,       /* zero residual mass; bonus drawn from p */
  DFLASH_FLAG_INVALID = 8           /* q(x) == 0: candidate was not drawn from q */
};

/* Bit of the per-sequence flags of dflash_gate: |c_s - g| < 1e-4. */
enum { DFLASH_FLAG_GATE_BOUNDARY = 1 };

#define DFLASH_WS_COUNTER_BYTES 16384

/*
 * Device-side error word. The last 4 bytes of a workspace's counter region
 * (byte offset DFLASH_WS_ERROR_WORD_OFFSET) hold an int32 that a kernel sets
 * when something goes wrong on the device; the first code written stays and
 * nothing clears it. It cannot be returned by the (asynchronous) call itself:
 * a caller that wants to know reads it once the stream has passed the call
 * (for example a 4-byte cudaMemcpy). Values:
 *   0                        no error
 *   1 .. 99                  a tensor-core kernel gave up a bounded wait (the
 *                            value names the wait; see dflash_set_wait_limit_ns).
 *                            The kernel returned early: that call's outputs are
 *                            invalid and completion counters of the workspace
 *                            may be left part-counted, so zero the whole counter
 *                            region (DFLASH_WS_COUNTER_BYTES) before the next call.
 *   DFLASH_DEVERR_BAD_PAGE   dflash_block_attn met a page-table entry outside
 *                            [0, num_pages) for a position inside a context; it
 *                            read page 0 for that position (never out of bounds),
 *                            so that call's output is invalid. Counters stay
 *                            consistent; clear the word to reuse the workspace.
 *   DFLASH_DEVERR_BAD_N_DRAFT  a verify or draft-select call met an n_draft[b]
 *                            outside [0, n_max]; it used the value clamped to
 *                            that range (never out of bounds), so sequence b's
 *                            outputs are those of the clamped count.
 * Only in a library built with DFLASH_DEBUG defined (the Python build's
 * debug library); release builds clamp these inputs without a record:
 *   DFLASH_DEVERR_BAD_CTX_LEN    dflash_block_attn met a ctx_len[b] outside
 *                            [0, max_ctx] (clamped to that range).
 *   DFLASH_DEVERR_BAD_COMMIT_LEN dflash_materialize_ctx_kv met a commit_len[b]
 *                            outside [0, rows_max] (clamped to that range).
 *   DFLASH_DEVERR_BAD_POSITION   dflash_materialize_ctx_kv met a committed row
 *                            whose position has no valid pool slot (a negative
 *                            position, a page past max_pages, or a page-table
 *                            entry outside [0, num_pages)); the row is not
 *                            written.
 * Calls that can set it: dflash_block_attn, dflash_materialize_ctx_kv, the
 * verify calls (greedy, sampled, sampled with LSEs) and
 * dflash_draft_select. The gate and DDTree kernels never set it.
 */
#define DFLASH_WS_ERROR_WORD_OFFSET (DFLASH_WS_COUNTER_BYTES - 4)
enum {
  DFLASH_DEVERR_BAD_PAGE = 100,
  DFLASH_DEVERR_BAD_N_DRAFT = 101,
  DFLASH_DEVERR_BAD_CTX_LEN = 102,
  DFLASH_DEVERR_BAD_COMMIT_LEN = 103,
  DFLASH_DEVERR_BAD_POSITION = 104
};

/* ------------------------------------------------------------------------- */
/* (a) Target-context KV materialisation                                      */
/* ------------------------------------------------------------------------- */
typedef struct {
  int32_t B;          /* sequences */
  int32_t rows_max;   /* rows per sequence in `hidden` (>= every commit_len) */
  int32_t m;          /* captured target layers */
  int32_t d;          /* d_model */
  int32_t L;          /* draft layers (1..16) */
  int32_t Hkv;        /* kv heads of a draft layer */
  int32_t D;          /* head dim (even) */
  int32_t page_size;  /* rows per KV page */
  int32_t max_pages;  /* row stride of page_table */
  int32_t num_pages;  /* pages in every pool; table entries must be < num_pages */
  int32_t dtype;      /* DFLASH_F32 | DFLASH_BF16 */
} dflash_ctx_kv_dims;

/*
 * Writes, for every sequence b and every row j < commit_len[b], the context K/V
 * of all L draft layers into the paged pools; no other pool row is touched.
 *
 *   h_ctx = W_f [h_l1; ...; h_lm] + b_f              [DFlash] KV 注入, step 2
 *   K^(l) = W_K^(l) h_ctx,  V^(l) = W_V^(l) h_ctx    [DFlash] KV 注入, step 3
 *   K^(l) <- k_norm, then RoPE at position start_pos[b] + j, then a
 *   prefix-valid write of the first commit_len[b] rows  [SGLang] 4.1
 *   slot of position p: page_table[b][p / page_size] * page_size + p % page_size
 *                                                     [SGLang] 5.1
 *
 * hidden     [B, rows_max, m*d]  captured target hidden of each candidate row
 * commit_len [B] int32  rows to write, 0 <= commit_len[b] <= rows_max
 * start_pos  [B] int32  absolute position of row 0 (the committed prefix length)
 * W_f [d, m*d], b_f [d] (nullable: no bias); stored [out, in]
 * W_kv       [L, 2, Hkv*D, d]  K then V projection of each draft layer, [out, in]
 * k_norm_w   [L, D] or NULL. Non-null: K <- K / sqrt(mean(K^2) + rms_eps) * w over D
 * rope_theta  > 0: rotate-half RoPE, pair (i, i + D/2) turned by
 *             pos * rope_theta^(-2i/D); 0 disables RoPE
 * k_pools, v_pools  HOST arrays of L device pointers, each [num_pages, page_size, Hkv, D]
 * page_table [B, max_pages] int32
 * new_len    [B] int32 or NULL: start_pos[b] + commit_len[b]; must not alias start_pos
 *
 * bf16 calls round h_ctx to bf16 before the K/V projection. Positions whose
 * page index is >= max_pages or whose page is outside [0, num_pages) are
 * skipped, not written.
 */
size_t dflash_materialize_workspace_size(const dflash_ctx_kv_dims* dims);
int dflash_materialize_ctx_kv(const dflash_ctx_kv_dims* dims,
                              const void* hidden, const int32_t* commit_len,
                              const int32_t* start_pos,
                              const void* W_f, const void* b_f, const void* W_kv,
                              const void* k_norm_w, float rms_eps, float rope_theta,
                              void* const* k_pools, void* const* v_pools,
                              const int32_t* page_table, int32_t* new_len,
                              void* workspace, size_t ws_bytes, dflash_stream_t stream);

/* ------------------------------------------------------------------------- */
/* (b) Draft block attention                                                  */
/* ------------------------------------------------------------------------- */
typedef struct {
  int32_t B;          /* sequences */
  int32_t n_q;        /* query rows of the block (k) */
  int32_t n_kv_blk;   /* the block's own K/V rows (k, plus rows a looped stage appends) */
  int32_t Hq, Hkv, D; /* Hq % Hkv == 0 */
  int32_t page_size;
  int32_t max_pages;  /* row stride of page_table */
  int32_t num_pages;
  int32_t max_ctx;    /* upper bound on every ctx_len[b] (sizes the launch) */
  int32_t dtype;
  int32_t causal;     /* 0: no mask; 1: in-block causal (needs n_kv_blk >= n_q), see below */
} dflash_attn_dims;

/*
 * out = softmax(scale * Q K^T) V, where for sequence b the keys and values are
 * the ctx_len[b] context rows of the paged pools followed by the n_kv_blk rows
 * of the block; q-head h reads kv-head h / (Hq / Hkv).
 *   [DFlash] 块扩散: the draft attends bidirectionally inside the block;
 *   [DFlash] KV 注入, step 3: Attention(Q_draft, [K_draft; K_ctx], [V_draft; V_ctx]).
 * causal = 0: no mask (every query row sees every key).
 * causal = 1: query row i sees every context row and the block rows
 *   j <= i + n_kv_blk - n_q (query i sits at block row i + n_kv_blk - n_q), the
 *   in-block causal variant of [DFlash] 块扩散的双向注意力问题 (JetSpec: block
 *   position i sees positions 0 .. i). n_kv_blk < n_q is rejected (INVALID_ARG).
 *
 * q [B, n_q, Hq, D]; k_blk, v_blk [B, n_kv_blk, Hkv, D]
 * k_pool, v_pool  one draft layer's pools [num_pages, page_size, Hkv, D]
 * page_table [B, max_pages] int32; ctx_len [B] int32, 0 <= ctx_len[b] <= max_ctx.
 *   Entries for positions inside a context must lie in [0, num_pages); an entry
 *   outside is read as page 0 and sets DFLASH_DEVERR_BAD_PAGE in the workspace's
 *   error word. Entries past a context are not read.
 * scale: softmax scale (1/sqrt(D) for the standard form)
 * out [B, n_q, Hq, D]
 * Repeated calls on the same inputs return identical bits: the bf16 kernel
 * divides the work by a static partition that depends on the dims and ctx_len
 * only, and merges split contexts in a fixed order.
 */
size_t dflash_block_attn_workspace_size(const dflash_attn_dims* dims);
int dflash_block_attn(const dflash_attn_dims* dims,
                      const void* q, const void* k_blk, const void* v_blk,
                      const void* k_pool, const void* v_pool,
                      const int32_t* page_table, const int32_t* ctx_len, float scale,
                      void* out, void* workspace, size_t ws_bytes, dflash_stream_t stream);

/*
 * dflash_block_attn for the sequences whose active[b] != 0 only. The looped
 * draft of [DLoop] 机制一 stops drafting a sequence once its stage gate fails
 * (c_s < g): later stages attend only for the sequences still going, and the
 * gate's cont output (dflash_gate, dflash_gate_stage) is this mask.
 * active [B] uint8 (device), or NULL: every sequence, exactly as
 * dflash_block_attn. The rows out[b] of an inactive sequence are not written;
 * its ctx_len[b] and page-table row are not read. The work of the call shrinks
 * with the active sequences (they alone are divided among the SMs); the bf16
 * kernel's partition of the work, and so the rounding of its split merges,
 * then depends on the mask as well: active rows may differ in the last bits
 * from dflash_block_attn's, and repeat bit for bit for the same mask.
 * Workspace: dflash_block_attn_workspace_size(dims).
 */
int dflash_block_attn_active(const dflash_attn_dims* dims,
                             const void* q, const void* k_blk, const void* v_blk,
                             const void* k_pool, const void* v_pool,
                             const int32_t* page_table, const int32_t* ctx_len, const uint8_t* active,
                             float scale, void* out, void* workspace, size_t ws_bytes,
                             dflash_stream_t stream);

/* ------------------------------------------------------------------------- */
/* (c) Verify                                                                 */
/* ------------------------------------------------------------------------- */
typedef struct {
  int32_t B;      /* sequences */
  int32_t n_max;  /* maximum drafts per sequence (row stride of cand is n_max+1) */
  int32_t V;      /* vocabulary */
  int32_t dtype;  /* type of the logits */
} dflash_verify_dims;

/*
 * Greedy rule, [SGLang] 3 and [DFlash] 验证流程:
 *   target_pred[i] = argmax_v target_logits[b, i, v]   (lowest index among ties)
 *   accept_len = number of leading i < n_b with cand[b, i+1] == target_pred[i]
 *   bonus = target_pred[accept_len];  commit_len = accept_len + 1
 *   out_tokens = cand[b, 1..accept_len] followed by bonus, then -1 padding.
 *
 * target_logits [B, n_max+1, V]; cand [B, n_max+1] int64, cand[:, 0] the anchor
 * n_draft [B] int32 in [0, n_max], or NULL for n_max everywhere
 * accept_len, commit_len [B] int32; bonus [B] int64
 * out_tokens [B, n_max+1] int64 or NULL; target_pred [B, n_max+1] int64 or NULL
 *   (argmax of rows 0..n_b, -1 beyond)
 */
size_t dflash_verify_greedy_workspace_size(const dflash_verify_dims* dims);
int dflash_verify_greedy(const dflash_verify_dims* dims,
                         const void* target_logits, const int64_t* cand,
                         const int32_t* n_draft,
                         int32_t* accept_len, int64_t* bonus, int32_t* commit_len,
                         int64_t* out_tokens, int64_t* target_pred,
                         void* workspace, size_t ws_bytes, dflash_stream_t stream);

/*
 * dflash_verify_greedy without a caller workspace. The pages have no
 * counterpart: this is a deployment variant of dflash_verify_greedy (same
 * arguments minus the workspace, same kernels, same results).
 *
 * It serves callers that cannot allocate device memory at the call site: a
 * plain C host that holds no device allocator, or a serving loop that reserves
 * all device memory up front (weights, paged KV pools) and permits no
 * allocation per decode round. Scratch is a fixed array of
 * DFLASH_NOALLOC_SCRATCH_BYTES in device memory of the library's module, one
 * per device; the call allocates nothing.
 *   - Limit: dims whose dflash_verify_greedy_workspace_size exceeds
 *     DFLASH_NOALLOC_SCRATCH_BYTES are rejected with DFLASH_ERR_UNSUPPORTED
 *     before anything is launched (B*(n_max+1) up to about 30000 rows fit).
 *   - Set-up: the first call on a device (the device current on the calling
 *     thread) resolves the array's address with cudaGetSymbolAddress, which may
 *     load the module on that device. Later calls only read the cached address.
 *   - Zero state: the array's counter region must be zero when a call starts.
 *     Module load zeroes it and every completed call leaves it zero; nothing
 *     else writes it.
 *   - Races: all calls on one device share the array. Calls must be ordered on
 *     the GPU (one stream, or streams ordered by events); calls that overlap
 *     in time, from any thread or stream, corrupt each other's results.
 */
#define DFLASH_NOALLOC_SCRATCH_BYTES (256 * 1024)
int dflash_verify_greedy_noalloc(const dflash_verify_dims* dims,
                                 const void* target_logits, const int64_t* cand,
                                 const int32_t* n_draft,
                                 int32_t* accept_len, int64_t* bonus, int32_t* commit_len,
                                 int64_t* out_tokens, int64_t* target_pred,
                                 dflash_stream_t stream);

/*
 * Sampled rule, [SpecDec] 3 and 4, [DLoop] looped verify:
 *   p_r = softmax(target_logits[b, r] / T), q_r = softmax(draft_logits[b, r] / T)
 *   for i = 1..n_b: x = cand[b, i]; accept iff u_accept[b, i-1] < p_{i-1}(x) / q_{i-1}(x);
 *   stop at the first rejection (later drafts are discarded).
 *   On a rejection at draft i: bonus ~ max(0, p_{i-1} - q_{i-1}) / Z with
 *   Z = sum_y max(0, p_{i-1}(y) - q_{i-1}(y)) (= 1 - beta); if all n_b are
 *   accepted: bonus ~ p_{n_b}. The draw is the inverse CDF in ascending token
 *   order: the smallest y with C(y) > u_final[b] * Z. If Z == 0 the draw uses p.
 *
 * target_logits [B, n_max+1, V]; draft_logits [B, n_max, V] (row i-1 is the law
 *   cand[b, i] was drawn from); cand [B, n_max+1] int64; n_draft [B] or NULL
 * u_accept [B, n_max] float, u_final [B] float: uniforms on [0, 1)
 * temperature > 0
 * accept_len, commit_len [B] int32; bonus [B] int64; out_tokens [B, n_max+1] int64
 *   or NULL; flags [B] uint8 or NULL (DFLASH_FLAG_* bits)
 * probs [B, 2*n_max + 1] float or NULL: p(x_i) for i = 1..n_max, then q(x_i),
 *   then the mass Z of the distribution the bonus was drawn from (1 for p).
 *   Entries of draft positions that were not evaluated are 0.
 */
size_t dflash_verify_sample_workspace_size(const dflash_verify_dims* dims);
int dflash_verify_sample(const dflash_verify_dims* dims, float temperature,
                         const void* target_logits, const void* draft_logits,
                         const int64_t* cand, const int32_t* n_draft,
                         const float* u_accept, const float* u_final,
                         int32_t* accept_len, int64_t* bonus, int32_t* commit_len,
                         int64_t* out_tokens, uint8_t* flags, float* probs,
                         void* workspace, size_t ws_bytes, dflash_stream_t stream);

/*
 * dflash_verify_sample with the draft rows' log-sum-exps supplied instead of
 * streamed. In [DLoop] 机制一 the gate score comes from the draft logits each
 * stage already produced, and the stage's dflash_gate call (row_lse) leaves
 * LSE(draft_logits[b, i] / T) for every row of the stage; the looped verify
 * over the stages' concatenated rows then reads only the target rows, one
 * draft logit per candidate and, for the bonus draw, the draft row at the
 * rejected position.
 * draft_row_lse [B, n_max] float: LSE(draft_logits[b, i] / T) in natural-log
 *   units (entries i >= n_b are not read). Every other argument and output as
 *   dflash_verify_sample; the workspace size is dflash_verify_sample's.
 * Same rule and same results as dflash_verify_sample whenever draft_row_lse
 * holds the rows' log-sum-exps (up to their float rounding, which the
 * boundary flags cover).
 */
int dflash_verify_sample_lse(const dflash_verify_dims* dims, float temperature,
                             const void* target_logits, const void* draft_logits,
                             const float* draft_row_lse, const int64_t* cand,
                             const int32_t* n_draft, const float* u_accept, const float* u_final,
                             int32_t* accept_len, int64_t* bonus, int32_t* commit_len,
                             int64_t* out_tokens, uint8_t* flags, float* probs,
                             void* workspace, size_t ws_bytes, dflash_stream_t stream);

/* ------------------------------------------------------------------------- */
/* DLoop block gate                                                           */
/* ------------------------------------------------------------------------- */
typedef struct {
  int32_t B;      /* sequences */
  int32_t k;      /* drafted tokens of the stage's block */
  int32_t V;
  int32_t dtype;  /* type of the logits */
} dflash_gate_dims;

/*
 * [DLoop] 机制一: c_s = sum_{i<k} log softmax(draft_logits[b, i] / T)[tokens[b, i]];
 * cont = (c_s >= g). Inactive sequences (active[b] == 0) get c = 0, cont = 0.
 *
 * draft_logits [B, k, V]; tokens [B, k] int64; active [B] uint8 or NULL (all active)
 * c_s [B] float; cont [B] uint8; row_lse [B, k] float or NULL (LSE of row / T);
 * flags [B] uint8 or NULL (DFLASH_FLAG_GATE_BOUNDARY)
 */
size_t dflash_gate_workspace_size(const dflash_gate_dims* dims);
int dflash_gate(const dflash_gate_dims* dims, float temperature, float g,
                const void* draft_logits, const int64_t* tokens, const uint8_t* active,
                float* c_s, uint8_t* cont, float* row_lse, uint8_t* flags,
                void* workspace, size_t ws_bytes, dflash_stream_t stream);

/*
 * One stage of the DLoop looped draft, read from the looped layout that the
 * verify of all stages takes, so that the stages chain on the device with no
 * host synchronisation. [DLoop] 机制一: a stage's block is drafted only while
 * every earlier gate said continue; the stage whose gate says stop is still
 * verified. [DLoop] looped verify: the S_b drafted blocks are concatenated
 * into one candidate list of S_b * k tokens checked by the sampled rule.
 *
 * dims: B, k (tokens of one stage), V, dtype. 0 <= stage, (stage + 1) * k <= n_max.
 * draft_logits [B, n_max, V]: stage s's rows are rows s*k .. s*k + k - 1
 * cand [B, n_max + 1] int64: cand[:, 0] the anchor, stage s's tokens at 1 + s*k ..
 * active [B] uint8 or NULL (all): sequences still drafting at this stage, i.e.
 *   the previous stage's cont (stage 0: NULL or all ones)
 * c_s, cont [B]; flags [B] or NULL: as dflash_gate (0 for inactive sequences)
 * row_lse [B, n_max] float or NULL: LSE(row / T) of this stage's rows of the
 *   active sequences, written at columns s*k .. s*k + k - 1 (other entries are
 *   left as they are): after the last stage it is the draft_row_lse of
 *   dflash_verify_sample_lse
 * n_verify [B] int32 or NULL: every active sequence adds k (its block joins the
 *   verify whether or not its gate continues); zero it before stage 0, and after
 *   the last stage it is the n_draft of the looped verify (S_b * k)
 * The workspace is dflash_gate_workspace_size(dims).
 */
int dflash_gate_stage(const dflash_gate_dims* dims, int32_t stage, int32_t n_max, float temperature,
                      float g, const void* draft_logits, const int64_t* cand, const uint8_t* active,
                      float* c_s, uint8_t* cont, float* row_lse, uint8_t* flags, int32_t* n_verify,
                      void* workspace, size_t ws_bytes, dflash_stream_t stream);

/* ------------------------------------------------------------------------- */
/* Draft-side token choice                                                    */
/* ------------------------------------------------------------------------- */
/*
 * The candidates of one round from the draft's MASK-position logits:
 *   [DFlash] 推理流程 step 4 and its decode listing: draft token i is the argmax
 *   of MASK position i's logits; [SpecDec] DFlash section: one token sampled
 *   from each position's distribution; candidates = [anchor] + draft tokens.
 * dims: B, n_max (MASK positions per sequence), V, dtype (dflash_verify_dims).
 * draft_logits [B, n_max, V] (row i <-> draft position i + 1); anchor [B] int64;
 * n_draft [B] int32 in [0, n_max] or NULL (n_max everywhere).
 * temperature == 0: argmax (lowest index among ties); q_x = 1; row_lse = LSE(z).
 * temperature > 0: x ~ softmax(z / T) by inverse CDF with u_draft[b, i] in
 *   ascending token order (smallest y with C(y) > u * Z); q_x = softmax(z / T)[x];
 *   row_lse = LSE(z / T); flags[b, i] = DFLASH_FLAG_CDF_BOUNDARY when u lies
 *   within 1e-6 of C(y-1)/Z or C(y)/Z as the kernel evaluates them.
 * u_draft [B, n_max] float (required when temperature > 0, else ignored).
 * Outputs: cand [B, n_max+1] int64 (cand[:, 0] = anchor, -1 past n_b);
 *   q_x, row_lse [B, n_max] float or NULL (0 past n_b); flags [B, n_max] uint8
 *   or NULL. Rows: B * n_max <= 4095; V <= 8388608.
 */
size_t dflash_draft_select_workspace_size(const dflash_verify_dims* dims);
int dflash_draft_select(const dflash_verify_dims* dims, float temperature,
                        const void* draft_logits, const int64_t* anchor, const int32_t* n_draft,
                        const float* u_draft, int64_t* cand, float* q_x, float* row_lse,
                        uint8_t* flags, void* workspace, size_t ws_bytes, dflash_stream_t stream);

/* ------------------------------------------------------------------------- */
/* DDTree: draft tree from the per-position marginals                         */
/* ------------------------------------------------------------------------- */
typedef struct {
  int32_t B;       /* sequences */
  int32_t n;       /* drafted positions (tree depth), <= 255 */
  int32_t V;       /* vocabulary */
  int32_t dtype;   /* type of the logits */
  int32_t K;       /* candidates per position, 1..16 */
  int32_t budget;  /* tree nodes (the root, the verified anchor, takes none), 1..4096 */
} dflash_tree_dims;

/*
 * [SpecDec] 6.1: the K most probable tokens of every drafted position.
 * draft_logits [B, n, V] (row i <-> position i + 1); temperature > 0.
 * topk_tok [B, n, K] int64 sorted by probability (ties: lower token index
 * first); topk_logp [B, n, K] float = log softmax(z / T) at those tokens.
 * No workspace.
 */
int dflash_ddtree_topk(const dflash_tree_dims* dims, float temperature, const void* draft_logits,
                       int64_t* topk_tok, float* topk_logp, dflash_stream_t stream);

/*
 * [SpecDec] 6.2 and 6.3: the best-first tree within `budget` nodes. The root's
 * candidate children are the position-1 top-K; each step takes the candidate
 * of highest path log-probability (the sum of its positions' topk_logp) into
 * the tree and makes its children (the next position's top-K) candidates;
 * it stops at `budget` nodes or when no candidate is left. Equal
 * probabilities: smaller depth, then earlier parent, then lower rank first.
 * Outputs per sequence, in the order the nodes were taken (a parent precedes
 * its children): node_token [B, budget] int64, node_parent [B, budget] int32
 * (index of the parent node, -1 = root), node_depth [B, budget] int32
 * (position 1..n), node_logp [B, budget] float (-1 / -1 / -1 / 0 past
 * n_nodes), n_nodes [B] int32, flags [B] uint8 or NULL (1: at some step a
 * candidate of different log-probability trailed the taken one by less than
 * 1e-5; exact ties follow the order above). No workspace.
 */
int dflash_ddtree_build(const dflash_tree_dims* dims, const int64_t* topk_tok, const float* topk_logp,
                        int64_t* node_token, int32_t* node_parent, int32_t* node_depth, float* node_logp,
                        int32_t* n_nodes, uint8_t* flags, dflash_stream_t stream);

/*
 * [SpecDec] 6.5 greedy tree walk with the greedy accept rule ([SGLang] 3):
 * from the root, the target's prediction (argmax, lowest index on ties) at the
 * current node selects the child holding that token, which is accepted and
 * becomes current; the walk stops at the first node with no such child, whose
 * prediction is the bonus.
 * target_logits [B, budget + 1, V]: row 0 after the anchor (the root), row
 * 1 + j after the path to node j (rows past n_nodes are not read).
 * accept_len, commit_len (= accept_len + 1) [B] int32; bonus [B] int64;
 * path [B, budget] int32 or NULL (accepted node indices, -1 padded);
 * out_tokens [B, budget + 1] int64 or NULL (accepted tokens then the bonus).
 */
size_t dflash_ddtree_verify_workspace_size(const dflash_tree_dims* dims);
int dflash_ddtree_verify_greedy(const dflash_tree_dims* dims, const void* target_logits,
                                const int64_t* node_token, const int32_t* node_parent,
                                const int32_t* n_nodes, int32_t* accept_len, int64_t* bonus,
                                int32_t* commit_len, int32_t* path, int64_t* out_tokens,
                                void* workspace, size_t ws_bytes, dflash_stream_t stream);

/* ------------------------------------------------------------------------- */
/* Diagnostics                                                                */
/* ------------------------------------------------------------------------- */
/*
 * Limit, in nanoseconds, of every bounded wait of the tensor-core kernels
 * (dflash_block_attn for bf16, dflash_materialize_ctx_kv for bf16) on the
 * barriers between their roles (copy landed, MMA done, buffer free). A wait
 * that runs out sets the error word (see DFLASH_WS_ERROR_WORD_OFFSET) and the
 * kernel returns early after draining its own copies and MMAs under a fixed
 * 2 s limit. The value is process-wide and read when a call launches (a kernel
 * captured in a CUDA graph keeps the value it was captured with). ns = 0
 * restores the default of 2 000 000 000 (2 s), far above any wait of a working
 * launch. Always returns DFLASH_OK.
 */
int dflash_set_wait_limit_ns(uint64_t ns);
uint64_t dflash_wait_limit_ns(void);
/* Message of the last error on this thread ("" if none). */
const char* dflash_last_error(void);
/* Number of kernel launches (memsets included) the last successful call on this
 * thread enqueued. */
int dflash_last_launch_count(void);

#ifdef __cplusplus
}
#endif
#endif /* DFLASH_H */
