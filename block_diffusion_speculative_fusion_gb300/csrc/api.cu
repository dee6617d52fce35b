// C ABI of libdflash: host-side validation, workspace layout and dispatch.
// Nothing here allocates device memory; every call is asynchronous on the
// caller's stream.
#include <atomic>
#include <cstdarg>
#include <cstdio>
#include <mutex>
#include <string>

#include <nvtx3/nvToolsExt.h>

#include "../../include/dflash.h"
#include "internal.h"

namespace {

// One NVTX range per call that launches work, named after the entry point, so
// that a profiler recording NVTX shows each call's kernels under its name
// (header-only NVTX: without a tool attached a range costs a few nanoseconds).
struct CallRange {
  explicit CallRange(const char* name) { nvtxRangePushA(name); }
  ~CallRange() { nvtxRangePop(); }
  CallRange(const CallRange&) = delete;
  CallRange& operator=(const CallRange&) = delete;
};

thread_local std::string g_err;
thread_local int g_launches = 0;

constexpr unsigned long long kDefaultWaitNs = 2000000000ull;
std::atomic<unsigned long long> g_wait_ns{kDefaultWaitNs};

// Kernel plans are sized for the 152-SM GB300 so that workspace sizes depend on
// the dims alone (no device query, callable without a GPU).
constexpr int kPlanSms = 152;
// The last int of the counter region is a sticky device-side error word.
constexpr int kMaxCounters = DFLASH_WS_COUNTER_BYTES / 4 - 1;

int fail(int code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_err = buf;
  return code;
}

int ok(int launches) {
  g_err.clear();
  g_launches = launches;
  return DFLASH_OK;
}

int cuda_fail(cudaError_t e, const char* what) {
  return fail(DFLASH_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

bool bad_dtype(int dt) { return dt != DFLASH_F32 && dt != DFLASH_BF16; }

int check_ws(void* ws, size_t have, size_t need) {
  if (need > 0 && ws == nullptr) return fail(DFLASH_ERR_WORKSPACE, "workspace is NULL (need %zu bytes)", need);
  if (have < need) return fail(DFLASH_ERR_WORKSPACE, "workspace of %zu bytes < required %zu", have, need);
  if ((reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return fail(DFLASH_ERR_WORKSPACE, "workspace not 256-byte aligned");
  return DFLASH_OK;
}

int check_verify_dims(const dflash_verify_dims* d, bool sampled) {
  if (!d) return fail(DFLASH_ERR_INVALID_ARG, "dims is NULL");
  if (d->B < 1 || d->n_max < 0 || d->V < 1) return fail(DFLASH_ERR_INVALID_ARG, "bad dims B=%d n_max=%d V=%d", d->B, d->n_max, d->V);
  if (bad_dtype(d->dtype)) return fail(DFLASH_ERR_INVALID_ARG, "bad dtype %d", d->dtype);
  if (d->n_max + 1 > 256) return fail(DFLASH_ERR_UNSUPPORTED, "n_max=%d > 255", d->n_max);
  if (sampled && (long)d->V > 1024L * 16384L) return fail(DFLASH_ERR_UNSUPPORTED, "V=%d too large", d->V);
  if (d->B > kMaxCounters) return fail(DFLASH_ERR_UNSUPPORTED, "B=%d too large", d->B);
  (void)sampled;
  if ((long)d->B * (2L * d->n_max + 1) > 65535L) return fail(DFLASH_ERR_UNSUPPORTED, "B*(2*n_max+1) > 65535");
  return DFLASH_OK;
}

}  // namespace

namespace dflash {
unsigned long long wait_limit_ns() { return g_wait_ns.load(std::memory_order_relaxed); }
}  // namespace dflash

extern "C" {

const char* dflash_last_error(void) { return g_err.c_str(); }
int dflash_last_launch_count(void) { return g_launches; }

int dflash_set_wait_limit_ns(uint64_t ns) {
  g_wait_ns.store(ns == 0 ? kDefaultWaitNs : (unsigned long long)ns, std::memory_order_relaxed);
  g_err.clear();
  return DFLASH_OK;
}
uint64_t dflash_wait_limit_ns(void) { return g_wait_ns.load(std::memory_order_relaxed); }

// ------------------------------------------------------------------ verify ---
size_t dflash_verify_greedy_workspace_size(const dflash_verify_dims* d) {
  if (check_verify_dims(d, false) != DFLASH_OK) return 0;
  return DFLASH_WS_COUNTER_BYTES + dflash::verify_greedy_ws_bytes(d->B, d->n_max, d->V, d->dtype, kPlanSms);
}

int dflash_verify_greedy(const dflash_verify_dims* d, const void* target_logits, const int64_t* cand,
                         const int32_t* n_draft, int32_t* accept_len, int64_t* bonus,
                         int32_t* commit_len, int64_t* out_tokens, int64_t* target_pred,
                         void* workspace, size_t ws_bytes, dflash_stream_t stream) {
  CallRange range_("dflash_verify_greedy");
  int rc = check_verify_dims(d, false);
  if (rc) return rc;
  if (!target_logits || !cand || !accept_len || !bonus || !commit_len)
    return fail(DFLASH_ERR_INVALID_ARG, "verify_greedy: a required pointer is NULL");
  rc = check_ws(workspace, ws_bytes, dflash_verify_greedy_workspace_size(d));
  if (rc) return rc;
  dflash::VerifyArgs a{};
  a.B = d->B; a.n_max = d->n_max; a.V = d->V; a.dtype = d->dtype; a.temperature = 1.f;
  a.target_logits = target_logits; a.cand = cand; a.n_draft = n_draft;
  a.accept_len = accept_len; a.bonus = bonus; a.commit_len = commit_len;
  a.out_tokens = out_tokens; a.target_pred = target_pred;
  a.counters = (int32_t*)workspace;
  a.err = (int*)workspace + kMaxCounters;
  a.scratch = (char*)workspace + DFLASH_WS_COUNTER_BYTES;
  a.stream = (cudaStream_t)stream;
  cudaError_t e = dflash::launch_verify_greedy(a, kPlanSms);
  if (e != cudaSuccess) return cuda_fail(e, "verify_greedy launch");
  return ok(1);
}

}  // extern "C"

// ------------------------------------------- verify, greedy, no allocation ---
// Scratch for dflash_verify_greedy_noalloc: a fixed device array in this
// module, one instance per device. It is laid out like a caller workspace
// (counters first, then the chunk partials). Static device storage is zero
// when the module loads, which is the state the completion counters need; a
// call that completes leaves them zero again.
namespace {

__device__ __align__(256) unsigned char g_noalloc_scratch[DFLASH_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mu;
void* g_noalloc_ptr[kMaxDevices] = {};

// Device address of the current device's scratch array. The first call on a
// device resolves it (cudaGetSymbolAddress, which may load the module on that
// device); later calls read the cached pointer.
int noalloc_scratch(void** out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "verify_greedy_noalloc: cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return fail(DFLASH_ERR_UNSUPPORTED, "device %d >= %d", dev, kMaxDevices);
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (!g_noalloc_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return cuda_fail(e, "verify_greedy_noalloc: cudaGetSymbolAddress");
    if (!p || (reinterpret_cast<uintptr_t>(p) & 255u) != 0)
      return fail(DFLASH_ERR_CUDA, "verify_greedy_noalloc: scratch address %p not 256-byte aligned", p);
    g_noalloc_ptr[dev] = p;
  }
  *out = g_noalloc_ptr[dev];
  return DFLASH_OK;
}

}  // namespace

extern "C" {

int dflash_verify_greedy_noalloc(const dflash_verify_dims* d, const void* target_logits, const int64_t* cand,
                                 const int32_t* n_draft, int32_t* accept_len, int64_t* bonus,
                                 int32_t* commit_len, int64_t* out_tokens, int64_t* target_pred,
                                 dflash_stream_t stream) {
  CallRange range_("dflash_verify_greedy_noalloc");
  int rc = check_verify_dims(d, false);
  if (rc) return rc;
  if (!target_logits || !cand || !accept_len || !bonus || !commit_len)
    return fail(DFLASH_ERR_INVALID_ARG, "verify_greedy_noalloc: a required pointer is NULL");
  const size_t need = dflash_verify_greedy_workspace_size(d);
  if (need > DFLASH_NOALLOC_SCRATCH_BYTES)
    return fail(DFLASH_ERR_UNSUPPORTED,
                "verify_greedy_noalloc: B=%d n_max=%d V=%d needs %zu bytes of scratch > the fixed %d; "
                "use dflash_verify_greedy with a caller workspace",
                d->B, d->n_max, d->V, need, (int)DFLASH_NOALLOC_SCRATCH_BYTES);
  void* scratch = nullptr;
  rc = noalloc_scratch(&scratch);
  if (rc) return rc;
  return dflash_verify_greedy(d, target_logits, cand, n_draft, accept_len, bonus, commit_len, out_tokens,
                              target_pred, scratch, DFLASH_NOALLOC_SCRATCH_BYTES, stream);
}

size_t dflash_verify_sample_workspace_size(const dflash_verify_dims* d) {
  if (check_verify_dims(d, true) != DFLASH_OK) return 0;
  return DFLASH_WS_COUNTER_BYTES + dflash::verify_sample_ws_bytes(d->B, d->n_max, d->V, d->dtype, kPlanSms);
}

int dflash_verify_sample(const dflash_verify_dims* d, float temperature, const void* target_logits,
                         const void* draft_logits, const int64_t* cand, const int32_t* n_draft,
                         const float* u_accept, const float* u_final, int32_t* accept_len,
                         int64_t* bonus, int32_t* commit_len, int64_t* out_tokens, uint8_t* flags,
                         float* probs, void* workspace, size_t ws_bytes, dflash_stream_t stream) {
  CallRange range_("dflash_verify_sample");
  int rc = check_verify_dims(d, true);
  if (rc) return rc;
  if (!(temperature > 0.f)) return fail(DFLASH_ERR_INVALID_ARG, "temperature must be > 0");
  if (!target_logits || !cand || !u_final || !accept_len || !bonus || !commit_len ||
      (d->n_max > 0 && (!draft_logits || !u_accept)))
    return fail(DFLASH_ERR_INVALID_ARG, "verify_sample: a required pointer is NULL");
  rc = check_ws(workspace, ws_bytes, dflash_verify_sample_workspace_size(d));
  if (rc) return rc;
  dflash::VerifyArgs a{};
  a.B = d->B; a.n_max = d->n_max; a.V = d->V; a.dtype = d->dtype; a.temperature = temperature;
  a.target_logits = target_logits; a.draft_logits = draft_logits; a.cand = cand;
  a.n_draft = n_draft; a.u_accept = u_accept; a.u_final = u_final;
  a.accept_len = accept_len; a.bonus = bonus; a.commit_len = commit_len;
  a.out_tokens = out_tokens; a.flags = flags; a.probs = probs;
  a.counters = (int32_t*)workspace;
  a.err = (int*)workspace + kMaxCounters;
  a.scratch = (char*)workspace + DFLASH_WS_COUNTER_BYTES;
  a.stream = (cudaStream_t)stream;
  cudaError_t e = dflash::launch_verify_sample(a, kPlanSms);
  if (e != cudaSuccess) return cuda_fail(e, "verify_sample launch");
  return ok(2);
}

int dflash_verify_sample_lse(const dflash_verify_dims* d, float temperature, const void* target_logits,
                             const void* draft_logits, const float* draft_row_lse, const int64_t* cand,
                             const int32_t* n_draft, const float* u_accept, const float* u_final,
                             int32_t* accept_len, int64_t* bonus, int32_t* commit_len, int64_t* out_tokens,
                             uint8_t* flags, float* probs, void* workspace, size_t ws_bytes,
                             dflash_stream_t stream) {
  CallRange range_("dflash_verify_sample_lse");
  int rc = check_verify_dims(d, true);
  if (rc) return rc;
  if (!(temperature > 0.f)) return fail(DFLASH_ERR_INVALID_ARG, "temperature must be > 0");
  if (!target_logits || !cand || !u_final || !accept_len || !bonus || !commit_len ||
      (d->n_max > 0 && (!draft_logits || !u_accept || !draft_row_lse)))
    return fail(DFLASH_ERR_INVALID_ARG, "verify_sample_lse: a required pointer is NULL");
  rc = check_ws(workspace, ws_bytes, dflash_verify_sample_workspace_size(d));
  if (rc) return rc;
  dflash::VerifyArgs a{};
  a.B = d->B; a.n_max = d->n_max; a.V = d->V; a.dtype = d->dtype; a.temperature = temperature;
  a.target_logits = target_logits; a.draft_logits = draft_logits; a.cand = cand;
  a.n_draft = n_draft; a.u_accept = u_accept; a.u_final = u_final;
  a.draft_lse = d->n_max > 0 ? draft_row_lse : nullptr;
  a.accept_len = accept_len; a.bonus = bonus; a.commit_len = commit_len;
  a.out_tokens = out_tokens; a.flags = flags; a.probs = probs;
  a.counters = (int32_t*)workspace;
  a.err = (int*)workspace + kMaxCounters;
  a.scratch = (char*)workspace + DFLASH_WS_COUNTER_BYTES;
  a.stream = (cudaStream_t)stream;
  cudaError_t e = dflash::launch_verify_sample(a, kPlanSms);
  if (e != cudaSuccess) return cuda_fail(e, "verify_sample_lse launch");
  return ok(2);
}

// -------------------------------------------------------------------- gate ---
static int check_gate_dims(const dflash_gate_dims* d) {
  if (!d) return fail(DFLASH_ERR_INVALID_ARG, "dims is NULL");
  if (d->B < 1 || d->k < 1 || d->V < 1) return fail(DFLASH_ERR_INVALID_ARG, "bad dims B=%d k=%d V=%d", d->B, d->k, d->V);
  if (bad_dtype(d->dtype)) return fail(DFLASH_ERR_INVALID_ARG, "bad dtype %d", d->dtype);
  if (d->k > 256) return fail(DFLASH_ERR_UNSUPPORTED, "k=%d > 256", d->k);
  if (d->B > kMaxCounters) return fail(DFLASH_ERR_UNSUPPORTED, "B=%d too large", d->B);
  if ((long)d->B * d->k > 65535L) return fail(DFLASH_ERR_UNSUPPORTED, "B*k > 65535");
  return DFLASH_OK;
}

size_t dflash_gate_workspace_size(const dflash_gate_dims* d) {
  if (check_gate_dims(d) != DFLASH_OK) return 0;
  return DFLASH_WS_COUNTER_BYTES + dflash::gate_ws_bytes(d->B, d->k, d->V, d->dtype, kPlanSms);
}

int dflash_gate(const dflash_gate_dims* d, float temperature, float g, const void* draft_logits,
                const int64_t* tokens, const uint8_t* active, float* c_s, uint8_t* cont,
                float* row_lse, uint8_t* flags, void* workspace, size_t ws_bytes,
                dflash_stream_t stream) {
  CallRange range_("dflash_gate");
  int rc = check_gate_dims(d);
  if (rc) return rc;
  if (!(temperature > 0.f)) return fail(DFLASH_ERR_INVALID_ARG, "temperature must be > 0");
  if (!draft_logits || !tokens || !c_s || !cont) return fail(DFLASH_ERR_INVALID_ARG, "gate: a required pointer is NULL");
  rc = check_ws(workspace, ws_bytes, dflash_gate_workspace_size(d));
  if (rc) return rc;
  dflash::GateArgs a{};
  a.B = d->B; a.k = d->k; a.V = d->V; a.dtype = d->dtype; a.temperature = temperature; a.g = g;
  a.layout = dflash::GateLayout{d->k, 0, d->k, 0, d->k, 0, 1};
  a.n_verify = nullptr;
  a.draft_logits = draft_logits; a.tokens = tokens; a.active = active;
  a.c_s = c_s; a.cont = cont; a.row_lse = row_lse; a.flags = flags;
  a.counters = (int32_t*)workspace;
  a.scratch = (char*)workspace + DFLASH_WS_COUNTER_BYTES;
  a.stream = (cudaStream_t)stream;
  cudaError_t e = dflash::launch_gate(a, kPlanSms);
  if (e != cudaSuccess) return cuda_fail(e, "gate launch");
  return ok(1);
}

int dflash_gate_stage(const dflash_gate_dims* d, int32_t stage, int32_t n_max, float temperature, float g,
                      const void* draft_logits, const int64_t* cand, const uint8_t* active, float* c_s,
                      uint8_t* cont, float* row_lse, uint8_t* flags, int32_t* n_verify, void* workspace,
                      size_t ws_bytes, dflash_stream_t stream) {
  CallRange range_("dflash_gate_stage");
  int rc = check_gate_dims(d);
  if (rc) return rc;
  if (!(temperature > 0.f)) return fail(DFLASH_ERR_INVALID_ARG, "temperature must be > 0");
  if (stage < 0 || n_max < 1 || (long)(stage + 1) * d->k > (long)n_max)
    return fail(DFLASH_ERR_INVALID_ARG, "stage %d of %d tokens does not fit n_max=%d", stage, d->k, n_max);
  if (n_max + 1 > 256) return fail(DFLASH_ERR_UNSUPPORTED, "n_max=%d > 255", n_max);
  if (!draft_logits || !cand || !c_s || !cont)
    return fail(DFLASH_ERR_INVALID_ARG, "gate_stage: a required pointer is NULL");
  rc = check_ws(workspace, ws_bytes, dflash_gate_workspace_size(d));
  if (rc) return rc;
  dflash::GateArgs a{};
  a.B = d->B; a.k = d->k; a.V = d->V; a.dtype = d->dtype; a.temperature = temperature; a.g = g;
  // stage rows s*k .. of [B, n_max, V]; tokens after the anchor in [B, n_max + 1]
  a.layout = dflash::GateLayout{n_max, stage * d->k, n_max + 1, 1 + stage * d->k, n_max, stage * d->k, 0};
  a.n_verify = n_verify;
  a.draft_logits = draft_logits; a.tokens = cand; a.active = active;
  a.c_s = c_s; a.cont = cont; a.row_lse = row_lse; a.flags = flags;
  a.counters = (int32_t*)workspace;
  a.scratch = (char*)workspace + DFLASH_WS_COUNTER_BYTES;
  a.stream = (cudaStream_t)stream;
  cudaError_t e = dflash::launch_gate(a, kPlanSms);
  if (e != cudaSuccess) return cuda_fail(e, "gate_stage launch");
  return ok(1);
}

// ------------------------------------------------------------ draft select ---
static int check_select_dims(const dflash_verify_dims* d) {
  if (!d) return fail(DFLASH_ERR_INVALID_ARG, "dims is NULL");
  if (d->B < 1 || d->n_max < 1 || d->V < 1)
    return fail(DFLASH_ERR_INVALID_ARG, "bad dims B=%d n_max=%d V=%d", d->B, d->n_max, d->V);
  if (bad_dtype(d->dtype)) return fail(DFLASH_ERR_INVALID_ARG, "bad dtype %d", d->dtype);
  if ((long)d->B * d->n_max > kMaxCounters)
    return fail(DFLASH_ERR_UNSUPPORTED, "B*n_max=%ld > %d rows", (long)d->B * d->n_max, kMaxCounters);
  if (d->V > dflash::kSelMaxVocab) return fail(DFLASH_ERR_UNSUPPORTED, "V=%d too large", d->V);
  return DFLASH_OK;
}

size_t dflash_draft_select_workspace_size(const dflash_verify_dims* d) {
  if (check_select_dims(d) != DFLASH_OK) return 0;
  return DFLASH_WS_COUNTER_BYTES + dflash::draft_select_ws_bytes(d->B, d->n_max, d->V, d->dtype);
}

int dflash_draft_select(const dflash_verify_dims* d, float temperature, const void* draft_logits,
                        const int64_t* anchor, const int32_t* n_draft, const float* u_draft, int64_t* cand,
                        float* q_x, float* row_lse, uint8_t* flags, void* workspace, size_t ws_bytes,
                        dflash_stream_t stream) {
  CallRange range_("dflash_draft_select");
  int rc = check_select_dims(d);
  if (rc) return rc;
  if (!(temperature >= 0.f) || !(temperature < 3.0e38f))
    return fail(DFLASH_ERR_INVALID_ARG, "temperature must be >= 0 and finite");
  if (!draft_logits || !anchor || !cand) return fail(DFLASH_ERR_INVALID_ARG, "draft_select: a required pointer is NULL");
  if (temperature > 0.f && !u_draft) return fail(DFLASH_ERR_INVALID_ARG, "draft_select: sampling needs u_draft");
  rc = check_ws(workspace, ws_bytes, dflash_draft_select_workspace_size(d));
  if (rc) return rc;
  dflash::DraftSelectArgs a{};
  a.B = d->B; a.n_max = d->n_max; a.V = d->V; a.dtype = d->dtype; a.temperature = temperature;
  a.draft_logits = draft_logits; a.anchor = anchor; a.n_draft = n_draft; a.u_draft = u_draft;
  a.cand = cand; a.q_x = q_x; a.row_lse = row_lse; a.flags = flags;
  a.num_sms = kPlanSms;
  a.counters = (int32_t*)workspace;
  a.err = (int*)workspace + kMaxCounters;
  a.scratch = (char*)workspace + DFLASH_WS_COUNTER_BYTES;
  a.stream = (cudaStream_t)stream;
  cudaError_t e = dflash::launch_draft_select(a);
  if (e != cudaSuccess) return cuda_fail(e, "draft_select launch");
  return ok(1);
}

// ------------------------------------------------------------------ DDTree ---
static int check_tree_dims(const dflash_tree_dims* d) {
  if (!d) return fail(DFLASH_ERR_INVALID_ARG, "dims is NULL");
  if (d->B < 1 || d->n < 1 || d->V < 1 || d->K < 1 || d->budget < 1)
    return fail(DFLASH_ERR_INVALID_ARG, "bad tree dims B=%d n=%d V=%d K=%d budget=%d", d->B, d->n, d->V, d->K,
                d->budget);
  if (bad_dtype(d->dtype)) return fail(DFLASH_ERR_INVALID_ARG, "bad dtype %d", d->dtype);
  if (d->K > dflash::kTreeMaxK || d->K > d->V)
    return fail(DFLASH_ERR_UNSUPPORTED, "K=%d outside [1, min(V, %d)]", d->K, dflash::kTreeMaxK);
  if (d->budget > dflash::kTreeMaxBudget) return fail(DFLASH_ERR_UNSUPPORTED, "budget=%d > %d", d->budget,
                                                      dflash::kTreeMaxBudget);
  if (d->n > 255) return fail(DFLASH_ERR_UNSUPPORTED, "n=%d > 255", d->n);
  if (d->B > kMaxCounters) return fail(DFLASH_ERR_UNSUPPORTED, "B=%d too large", d->B);
  if ((long)d->B * (d->budget + 1) > 65535L) return fail(DFLASH_ERR_UNSUPPORTED, "B*(budget+1) > 65535");
  return DFLASH_OK;
}

int dflash_ddtree_topk(const dflash_tree_dims* d, float temperature, const void* draft_logits, int64_t* topk_tok,
                       float* topk_logp, dflash_stream_t stream) {
  CallRange range_("dflash_ddtree_topk");
  int rc = check_tree_dims(d);
  if (rc) return rc;
  if (!(temperature > 0.f) || !(temperature < 3.0e38f)) return fail(DFLASH_ERR_INVALID_ARG, "temperature must be > 0");
  if (!draft_logits || !topk_tok || !topk_logp) return fail(DFLASH_ERR_INVALID_ARG, "ddtree_topk: a pointer is NULL");
  dflash::TreeArgs a{};
  a.B = d->B; a.n = d->n; a.V = d->V; a.dtype = d->dtype; a.K = d->K; a.budget = d->budget;
  a.temperature = temperature; a.logits = draft_logits; a.topk_tok = topk_tok; a.topk_logp = topk_logp;
  a.stream = (cudaStream_t)stream; a.num_sms = kPlanSms;
  cudaError_t e = dflash::launch_ddtree_topk(a);
  if (e != cudaSuccess) return cuda_fail(e, "ddtree_topk launch");
  return ok(1);
}

int dflash_ddtree_build(const dflash_tree_dims* d, const int64_t* topk_tok, const float* topk_logp,
                        int64_t* node_token, int32_t* node_parent, int32_t* node_depth, float* node_logp,
                        int32_t* n_nodes, uint8_t* flags, dflash_stream_t stream) {
  CallRange range_("dflash_ddtree_build");
  int rc = check_tree_dims(d);
  if (rc) return rc;
  if (!topk_tok || !topk_logp || !node_token || !node_parent || !node_depth || !node_logp || !n_nodes)
    return fail(DFLASH_ERR_INVALID_ARG, "ddtree_build: a required pointer is NULL");
  dflash::TreeArgs a{};
  a.B = d->B; a.n = d->n; a.V = d->V; a.dtype = d->dtype; a.K = d->K; a.budget = d->budget;
  a.topk_tok = const_cast<int64_t*>(topk_tok); a.topk_logp = const_cast<float*>(topk_logp);
  a.node_token = node_token; a.node_parent = node_parent; a.node_depth = node_depth; a.node_logp = node_logp;
  a.n_nodes = n_nodes; a.flags = flags; a.stream = (cudaStream_t)stream; a.num_sms = kPlanSms;
  cudaError_t e = dflash::launch_ddtree_build(a);
  if (e != cudaSuccess) return cuda_fail(e, "ddtree_build launch");
  return ok(1);
}

size_t dflash_ddtree_verify_workspace_size(const dflash_tree_dims* d) {
  if (check_tree_dims(d) != DFLASH_OK) return 0;
  return DFLASH_WS_COUNTER_BYTES + dflash::ddtree_verify_ws_bytes(d->B, d->budget, d->V, d->dtype, kPlanSms);
}

int dflash_ddtree_verify_greedy(const dflash_tree_dims* d, const void* target_logits, const int64_t* node_token,
                                const int32_t* node_parent, const int32_t* n_nodes, int32_t* accept_len,
                                int64_t* bonus, int32_t* commit_len, int32_t* path, int64_t* out_tokens,
                                void* workspace, size_t ws_bytes, dflash_stream_t stream) {
  CallRange range_("dflash_ddtree_verify_greedy");
  int rc = check_tree_dims(d);
  if (rc) return rc;
  if (!target_logits || !node_token || !node_parent || !n_nodes || !accept_len || !bonus || !commit_len)
    return fail(DFLASH_ERR_INVALID_ARG, "ddtree_verify_greedy: a required pointer is NULL");
  rc = check_ws(workspace, ws_bytes, dflash_ddtree_verify_workspace_size(d));
  if (rc) return rc;
  dflash::TreeArgs a{};
  a.B = d->B; a.n = d->n; a.V = d->V; a.dtype = d->dtype; a.K = d->K; a.budget = d->budget;
  a.logits = target_logits; a.node_token = const_cast<int64_t*>(node_token);
  a.node_parent = const_cast<int32_t*>(node_parent); a.n_nodes = const_cast<int32_t*>(n_nodes);
  a.accept_len = accept_len; a.bonus = bonus; a.commit_len = commit_len; a.path = path; a.out_tokens = out_tokens;
  a.counters = (int32_t*)workspace;
  a.scratch = (char*)workspace + DFLASH_WS_COUNTER_BYTES;
  a.stream = (cudaStream_t)stream; a.num_sms = kPlanSms;
  cudaError_t e = dflash::launch_ddtree_verify(a);
  if (e != cudaSuccess) return cuda_fail(e, "ddtree_verify launch");
  return ok(1);
}

// --------------------------------------------------------------- attention ---
static int check_attn_dims(const dflash_attn_dims* d) {
  if (!d) return fail(DFLASH_ERR_INVALID_ARG, "dims is NULL");
  if (d->B < 1 || d->n_q < 1 || d->n_kv_blk < 0 || d->Hq < 1 || d->Hkv < 1 || d->D < 2 ||
      d->page_size < 1 || d->max_pages < 1 || d->num_pages < 1 || d->max_ctx < 0)
    return fail(DFLASH_ERR_INVALID_ARG, "bad attention dims");
  if (d->Hq % d->Hkv) return fail(DFLASH_ERR_INVALID_ARG, "Hq=%d not a multiple of Hkv=%d", d->Hq, d->Hkv);
  if (bad_dtype(d->dtype)) return fail(DFLASH_ERR_INVALID_ARG, "bad dtype %d", d->dtype);
  if ((long)d->max_ctx > (long)d->max_pages * d->page_size)
    return fail(DFLASH_ERR_INVALID_ARG, "max_ctx=%d exceeds max_pages*page_size", d->max_ctx);
  if (d->D > 256) return fail(DFLASH_ERR_UNSUPPORTED, "D=%d > 256", d->D);
  if (d->n_q > 65535 || d->Hq > 65535 || d->B > 65535) return fail(DFLASH_ERR_UNSUPPORTED, "grid too large");
  if (d->causal != 0 && d->causal != 1) return fail(DFLASH_ERR_INVALID_ARG, "causal=%d is not 0 or 1", d->causal);
  if (d->causal && d->n_kv_blk < d->n_q)
    return fail(DFLASH_ERR_INVALID_ARG, "causal needs n_kv_blk=%d >= n_q=%d", d->n_kv_blk, d->n_q);
  return DFLASH_OK;
}

size_t dflash_block_attn_workspace_size(const dflash_attn_dims* d) {
  if (check_attn_dims(d) != DFLASH_OK) return 0;
  return DFLASH_WS_COUNTER_BYTES +
         dflash::attn_ws_bytes(d->B, d->n_q, d->n_kv_blk, d->Hq, d->Hkv, d->D, d->max_ctx, d->page_size, d->dtype);
}

}  // extern "C"

namespace {

int block_attn_call(const dflash_attn_dims* d, const void* q, const void* k_blk, const void* v_blk,
                    const void* k_pool, const void* v_pool, const int32_t* page_table, const int32_t* ctx_len,
                    const uint8_t* active, float scale, void* out, void* workspace, size_t ws_bytes,
                    dflash_stream_t stream) {
  int rc = check_attn_dims(d);
  if (rc) return rc;
  if (!q || !k_pool || !v_pool || !page_table || !ctx_len || !out || (d->n_kv_blk > 0 && (!k_blk || !v_blk)))
    return fail(DFLASH_ERR_INVALID_ARG, "block_attn: a required pointer is NULL");
  rc = check_ws(workspace, ws_bytes, dflash_block_attn_workspace_size(d));
  if (rc) return rc;
  dflash::AttnArgs a{};
  a.B = d->B; a.n_q = d->n_q; a.n_kv = d->n_kv_blk; a.Hq = d->Hq; a.Hkv = d->Hkv; a.D = d->D;
  a.page_size = d->page_size; a.max_pages = d->max_pages; a.num_pages = d->num_pages;
  a.max_ctx = d->max_ctx; a.dtype = d->dtype; a.causal = d->causal;
  a.q = q; a.k_blk = k_blk; a.v_blk = v_blk; a.k_pool = k_pool; a.v_pool = v_pool;
  a.page_table = page_table; a.ctx_len = ctx_len; a.active = active; a.scale = scale; a.out = out;
  a.err = (int*)workspace + kMaxCounters;
  a.scratch = (char*)workspace + DFLASH_WS_COUNTER_BYTES;
  a.stream = (cudaStream_t)stream;
  int launches = 0;
  cudaError_t e = dflash::launch_block_attn(a, &launches);
  if (e != cudaSuccess) return cuda_fail(e, "block_attn launch");
  return ok(launches);
}

}  // namespace

extern "C" {

int dflash_block_attn(const dflash_attn_dims* d, const void* q, const void* k_blk, const void* v_blk,
                      const void* k_pool, const void* v_pool, const int32_t* page_table,
                      const int32_t* ctx_len, float scale, void* out, void* workspace, size_t ws_bytes,
                      dflash_stream_t stream) {
  CallRange range_("dflash_block_attn");
  return block_attn_call(d, q, k_blk, v_blk, k_pool, v_pool, page_table, ctx_len, nullptr, scale, out, workspace,
                         ws_bytes, stream);
}

int dflash_block_attn_active(const dflash_attn_dims* d, const void* q, const void* k_blk, const void* v_blk,
                             const void* k_pool, const void* v_pool, const int32_t* page_table,
                             const int32_t* ctx_len, const uint8_t* active, float scale, void* out,
                             void* workspace, size_t ws_bytes, dflash_stream_t stream) {
  CallRange range_("dflash_block_attn_active");
  return block_attn_call(d, q, k_blk, v_blk, k_pool, v_pool, page_table, ctx_len, active, scale, out, workspace,
                         ws_bytes, stream);
}

// ------------------------------------------------------------- materialise ---
static int check_mat_dims(const dflash_ctx_kv_dims* d) {
  if (!d) return fail(DFLASH_ERR_INVALID_ARG, "dims is NULL");
  if (d->B < 1 || d->rows_max < 1 || d->m < 1 || d->d < 1 || d->L < 1 || d->Hkv < 1 || d->D < 2 ||
      d->page_size < 1 || d->max_pages < 1 || d->num_pages < 1)
    return fail(DFLASH_ERR_INVALID_ARG, "bad materialise dims");
  if (d->D % 2) return fail(DFLASH_ERR_INVALID_ARG, "D=%d must be even (RoPE pairs)", d->D);
  if (bad_dtype(d->dtype)) return fail(DFLASH_ERR_INVALID_ARG, "bad dtype %d", d->dtype);
  if (d->L > dflash::kMaxLayers) return fail(DFLASH_ERR_UNSUPPORTED, "L=%d > %d", d->L, dflash::kMaxLayers);
  if (d->D > 256) return fail(DFLASH_ERR_UNSUPPORTED, "D=%d > 256", d->D);
  if ((long)d->B * d->rows_max > 65535L) return fail(DFLASH_ERR_UNSUPPORTED, "B*rows_max > 65535");
  const long el = d->dtype == DFLASH_BF16 ? 2 : 4;
  if (((long)d->m * d->d * el) % 16 || ((long)d->d * el) % 16)
    return fail(DFLASH_ERR_UNSUPPORTED, "rows of hidden and W_kv must be multiples of 16 bytes");
  return DFLASH_OK;
}

size_t dflash_materialize_workspace_size(const dflash_ctx_kv_dims* d) {
  if (check_mat_dims(d) != DFLASH_OK) return 0;
  const dflash::MatPlan p = dflash::mat_plan(d->B, d->rows_max, d->m, d->d, d->L, d->Hkv, d->D, d->dtype);
  return DFLASH_WS_COUNTER_BYTES + dflash::mat_ws_bytes(p, d->dtype);
}

int dflash_materialize_ctx_kv(const dflash_ctx_kv_dims* d, const void* hidden, const int32_t* commit_len,
                              const int32_t* start_pos, const void* W_f, const void* b_f, const void* W_kv,
                              const void* k_norm_w, float rms_eps, float rope_theta, void* const* k_pools,
                              void* const* v_pools, const int32_t* page_table, int32_t* new_len,
                              void* workspace, size_t ws_bytes, dflash_stream_t stream) {
  CallRange range_("dflash_materialize_ctx_kv");
  int rc = check_mat_dims(d);
  if (rc) return rc;
  if (!hidden || !commit_len || !start_pos || !W_f || !W_kv || !k_pools || !v_pools || !page_table)
    return fail(DFLASH_ERR_INVALID_ARG, "materialize: a required pointer is NULL");
  if (new_len && new_len == start_pos) return fail(DFLASH_ERR_INVALID_ARG, "new_len must not alias start_pos");
  if (rope_theta < 0.f || !(rms_eps >= 0.f)) return fail(DFLASH_ERR_INVALID_ARG, "bad rope_theta or rms_eps");
  rc = check_ws(workspace, ws_bytes, dflash_materialize_workspace_size(d));
  if (rc) return rc;
  dflash::MatArgs a{};
  a.B = d->B; a.rows_max = d->rows_max; a.m = d->m; a.d = d->d; a.L = d->L; a.Hkv = d->Hkv; a.D = d->D;
  a.page_size = d->page_size; a.max_pages = d->max_pages; a.num_pages = d->num_pages; a.dtype = d->dtype;
  a.hidden = hidden; a.commit_len = commit_len; a.start_pos = start_pos; a.W_f = W_f; a.b_f = b_f;
  a.W_kv = W_kv; a.k_norm_w = k_norm_w; a.rms_eps = rms_eps; a.rope_theta = rope_theta;
  for (int l = 0; l < d->L; ++l) {
    if (!k_pools[l] || !v_pools[l]) return fail(DFLASH_ERR_INVALID_ARG, "pool pointer of layer %d is NULL", l);
    a.pools.k[l] = k_pools[l];
    a.pools.v[l] = v_pools[l];
  }
  a.page_table = page_table; a.new_len = new_len;
  a.counters = (int32_t*)workspace;
  a.err = (int*)workspace + kMaxCounters;
  a.scratch = (char*)workspace + DFLASH_WS_COUNTER_BYTES;
  a.stream = (cudaStream_t)stream;
  int launches = 0;
  cudaError_t e = dflash::launch_materialize(a, &launches);
  if (e != cudaSuccess) return cuda_fail(e, "materialize launch");
  return ok(launches);
}

}  // extern "C"
