// C-ABI entry points: host-side argument checks, then the launchers.
#include <atomic>
#include <cstdarg>
#include <cstdio>
#include <cstring>

#include "importance.cuh"
#include "refresh.cuh"
#include "ts_common.cuh"

namespace ts {

static thread_local char g_last_error[512] = {0};

std::atomic<long long> g_wait_limit{kDefaultWaitCycles};
long long wait_limit_cycles() { return g_wait_limit.load(); }

int fail(int code, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_last_error, sizeof(g_last_error), fmt, ap);
  va_end(ap);
  return code;
}

void clear_error() { g_last_error[0] = 0; }

int launch_status(const char* what) {
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return fail(TS_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
  return TS_OK;
}

static int check_ws(const void* ws, size_t have, size_t need, const char* what) {
  if (need == 0) return TS_OK;
  if (!ws) return fail(TS_ERR_WORKSPACE, "%s: workspace is NULL (%zu bytes needed)", what, need);
  if (reinterpret_cast<uintptr_t>(ws) % 256)
    return fail(TS_ERR_WORKSPACE, "%s: workspace must be 256-byte aligned", what);
  if (have < need)
    return fail(TS_ERR_WORKSPACE, "%s: workspace has %zu bytes, %zu needed", what, have, need);
  return TS_OK;
}

static int check_attn_shape(int T, int Hq, int Hkv, int d, const char* what) {
  if (T < 1 || Hq < 1 || Hkv < 1)
    return fail(TS_ERR_INVALID_ARG, "%s: T, Hq, Hkv must be >= 1 (T=%d Hq=%d Hkv=%d)", what, T, Hq, Hkv);
  if (T > 64) return fail(TS_ERR_UNSUPPORTED, "%s: T=%d > 64 tree nodes", what, T);
  if (Hq % Hkv) return fail(TS_ERR_INVALID_ARG, "%s: Hq=%d not a multiple of Hkv=%d", what, Hq, Hkv);
  if (d != 64 && d != 128) return fail(TS_ERR_UNSUPPORTED, "%s: head dim %d not in {64,128}", what, d);
  if (T * (Hq / Hkv) > 512)
    return fail(TS_ERR_UNSUPPORTED, "%s: T*Hq/Hkv = %d > 512 query rows per KV head", what, T * (Hq / Hkv));
  return TS_OK;
}

int launch_kv_commit_batched(int n_layers, void* const* k, void* const* v, int64_t L,
                             int64_t L_cap, int Hkv, int d, int T, const int32_t* path,
                             const int32_t* n_path, int32_t* status, cudaStream_t st);

size_t reject_ws_bytes(int V);
int launch_reject_accept(const float* logits, const float* q, const int32_t* tree_tokens,
                         const int32_t* parents, int T, const int32_t* prior, int n_prior, int W,
                         int V, float penalty, float temperature, float top_p, float min_p,
                         int literal, const float* u_accept, const float* u_draw, int32_t* path,
                         int32_t* n_path, int32_t* bonus, void* ws, int32_t* status,
                         cudaStream_t st);
int launch_kv_append_batched(int n_layers, void* const* k, void* const* v, const void* krows,
                             const void* vrows, int64_t L, int64_t L_cap, int Hkv, int d, int T,
                             bool v_fp16, int32_t* status, cudaStream_t st);

}  // namespace ts

using namespace ts;

extern "C" {

const char* ts_status_string(int s) {
  switch (s) {
    case TS_OK: return "ok";
    case TS_ERR_INVALID_ARG: return "invalid argument";
    case TS_ERR_UNSUPPORTED: return "unsupported configuration";
    case TS_ERR_CUDA: return "CUDA error";
    case TS_ERR_TIMEOUT: return "device-side wait timed out";
    case TS_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
    default: return "unknown status";
  }
}

const char* ts_last_error(void) { return g_last_error; }

int ts_version(void) { return 100; }

int ts_set_wait_limit(int64_t cycles) {
  clear_error();
  ts::g_wait_limit.store(cycles > 0 ? (long long)cycles : ts::kDefaultWaitCycles);
  return TS_OK;
}

size_t ts_verify_workspace_bytes(int T, int Hq, int Hkv, int d, int64_t L) {
  if (check_attn_shape(T, Hq, Hkv, d, "ts_verify_workspace_bytes") != TS_OK || L < 0) return 0;
  return verify_plan(T, Hq, Hkv, d, L).ws_bytes;
}

int ts_verify_attention_flags(const void* q, const void* k, const void* v, int64_t L,
                              int64_t L_cap, const int32_t* parents, int T, int Hq, int Hkv, int d,
                              int n_imp, float* o, float* lse, float* imp, void* workspace,
                              size_t workspace_bytes, int flags, int32_t* status, void* stream) {
  clear_error();
  const char* W = "ts_verify_attention";
  if (flags & ~TS_VERIFY_V_FP16) return fail(TS_ERR_INVALID_ARG, "%s: unknown flags 0x%x", W, flags);
  int rc = check_attn_shape(T, Hq, Hkv, d, W);
  if (rc) return rc;
  if (!q || !k || !v || !parents || !o) return fail(TS_ERR_INVALID_ARG, "%s: NULL tensor", W);
  if (L < 0 || L + T > L_cap)
    return fail(TS_ERR_INVALID_ARG, "%s: need 0 <= L and L+T <= L_cap (L=%lld T=%d L_cap=%lld)", W,
                (long long)L, T, (long long)L_cap);
  if (L_cap > (int64_t(1) << 31) - 1) return fail(TS_ERR_UNSUPPORTED, "%s: L_cap >= 2^31", W);
  if (n_imp > T) return fail(TS_ERR_INVALID_ARG, "%s: n_imp=%d > T=%d", W, n_imp, T);
  if (n_imp <= 0) n_imp = T;
  VerifyPlan p = verify_plan(T, Hq, Hkv, d, L);
  rc = check_ws(workspace, workspace_bytes, p.ws_bytes, W);
  if (rc) return rc;
  return launch_verify(q, k, v, L, L_cap, parents, T, Hq, Hkv, d, n_imp,
                       (flags & TS_VERIFY_V_FP16) != 0, o, lse, imp, workspace, status,
                       static_cast<cudaStream_t>(stream));
}

int ts_verify_attention(const void* q, const void* k, const void* v, int64_t L, int64_t L_cap,
                        const int32_t* parents, int T, int Hq, int Hkv, int d, int n_imp,
                        float* o, float* lse, float* imp, void* workspace,
                        size_t workspace_bytes, int32_t* status, void* stream) {
  return ts_verify_attention_flags(q, k, v, L, L_cap, parents, T, Hq, Hkv, d, n_imp, o, lse, imp,
                                   workspace, workspace_bytes, 0, status, stream);
}

int ts_importance_softmax(const void* q, const void* k, const float* lse, int64_t L,
                          int64_t L_cap, int T, int Hq, int Hkv, int d, int n_imp, float* imp,
                          int32_t* status, void* stream) {
  clear_error();
  const char* W = "ts_importance_softmax";
  int rc = check_attn_shape(T, Hq, Hkv, d, W);
  if (rc) return rc;
  if (L < 0 || L > L_cap)
    return fail(TS_ERR_INVALID_ARG, "%s: need 0 <= L <= L_cap (L=%lld L_cap=%lld)", W,
                (long long)L, (long long)L_cap);
  if (L == 0) return TS_OK;   // nothing to write (imp may then be empty)
  if (!q || !k || !lse || !imp) return fail(TS_ERR_INVALID_ARG, "%s: NULL tensor", W);
  if (L_cap > (int64_t(1) << 31) - 1) return fail(TS_ERR_UNSUPPORTED, "%s: L_cap >= 2^31", W);
  if (n_imp > T) return fail(TS_ERR_INVALID_ARG, "%s: n_imp=%d > T=%d", W, n_imp, T);
  if (n_imp <= 0) n_imp = T;
  if (importance_softmax_plan(T, Hq, Hkv, d, n_imp, L > 0 ? L : 1).smem > 227 * 1024)
    return fail(TS_ERR_UNSUPPORTED, "%s: %d importance query rows exceed one SM's shared memory",
                W, n_imp * (Hq / Hkv));
  return launch_importance_softmax(q, k, lse, L, L_cap, T, Hq, Hkv, d, n_imp, imp, status,
                                   static_cast<cudaStream_t>(stream));
}

size_t ts_select_workspace_bytes(int Hkv, int64_t L) {
  if (Hkv < 1 || L < 0) return 0;
  return select_plan(Hkv, L, 1).ws_bytes;
}

size_t ts_select_batched_workspace_bytes(int n_layers, int Hkv, int64_t L) {
  if (n_layers < 1 || Hkv < 1 || L < 0) return 0;
  return select_plan(Hkv, L, n_layers).ws_bytes;
}

int ts_partial_kv_select_gather(const float* imp, const void* k, const void* v, int64_t L,
                                int64_t L_cap, int Hkv, int d, int B, int S, int R,
                                int32_t* idx, void* kd, void* vd, int64_t* n_out,
                                void* workspace, size_t workspace_bytes, int32_t* status,
                                void* stream) {
  clear_error();
  const char* W = "ts_partial_kv_select_gather";
  if (Hkv < 1) return fail(TS_ERR_INVALID_ARG, "%s: Hkv=%d", W, Hkv);
  if (d != 64 && d != 128) return fail(TS_ERR_UNSUPPORTED, "%s: head dim %d not in {64,128}", W, d);
  if (B < 0 || S < 0 || R < 0) return fail(TS_ERR_INVALID_ARG, "%s: B, S, R must be >= 0", W);
  if (L < 0 || L > L_cap) return fail(TS_ERR_INVALID_ARG, "%s: need 0 <= L <= L_cap", W);
  if (L_cap > (int64_t(1) << 31) - 1) return fail(TS_ERR_UNSUPPORTED, "%s: L_cap >= 2^31", W);
  int64_t N = L < (int64_t)S + B + R ? L : (int64_t)S + B + R;
  if (n_out) *n_out = N;
  if (L == 0) return TS_OK;
  if (!imp || !k || !v || !idx || !kd || !vd) return fail(TS_ERR_INVALID_ARG, "%s: NULL tensor", W);
  SelectPlan p = select_plan(Hkv, L, 1);
  int rc = check_ws(workspace, workspace_bytes, p.ws_bytes, W);
  if (rc) return rc;
  return launch_select_gather(imp, k, v, L, L_cap, Hkv, d, B, S, R, idx, kd, vd, N, workspace,
                              status, static_cast<cudaStream_t>(stream));
}

int ts_partial_kv_select_gather_noalloc(const float* imp, const void* k, const void* v,
                                        int64_t L, int64_t L_cap, int Hkv, int d, int B, int S,
                                        int R, int32_t* idx, void* kd, void* vd, int64_t* n_out,
                                        int32_t* status, void* stream) {
  clear_error();
  const char* W = "ts_partial_kv_select_gather_noalloc";
  if (Hkv < 1) return fail(TS_ERR_INVALID_ARG, "%s: Hkv=%d", W, Hkv);
  if (d != 64 && d != 128) return fail(TS_ERR_UNSUPPORTED, "%s: head dim %d not in {64,128}", W, d);
  if (B < 0 || S < 0 || R < 0) return fail(TS_ERR_INVALID_ARG, "%s: B, S, R must be >= 0", W);
  if (L < 0 || L > L_cap) return fail(TS_ERR_INVALID_ARG, "%s: need 0 <= L <= L_cap", W);
  if (L_cap > (int64_t(1) << 31) - 1) return fail(TS_ERR_UNSUPPORTED, "%s: L_cap >= 2^31", W);
  const size_t need = select_plan(Hkv, L, 1).ws_bytes;
  if (need > kNoAllocScratchBytes)
    return fail(TS_ERR_UNSUPPORTED,
                "%s: Hkv=%d, L=%lld needs %zu bytes of scratch; the fixed array holds %zu "
                "(about Hkv*L <= 1.2M positions); use ts_partial_kv_select_gather with a workspace",
                W, Hkv, (long long)L, need, kNoAllocScratchBytes);
  int64_t N = L < (int64_t)S + B + R ? L : (int64_t)S + B + R;
  if (n_out) *n_out = N;
  if (L == 0) return TS_OK;
  if (!imp || !k || !v || !idx || !kd || !vd) return fail(TS_ERR_INVALID_ARG, "%s: NULL tensor", W);
  void* scratch = nullptr;
  int rc = select_scratch(&scratch);
  if (rc) return rc;
  return launch_select_gather(imp, k, v, L, L_cap, Hkv, d, B, S, R, idx, kd, vd, N, scratch,
                              status, static_cast<cudaStream_t>(stream));
}

size_t ts_refresh_workspace_bytes(int n_layers, int Hkv, int64_t L, int64_t N_cap) {
  if (n_layers < 1 || Hkv < 1 || L < 0 || N_cap < 0) return 0;
  return refresh_ws_bytes(n_layers * Hkv, L, N_cap);
}

static int refresh_common(const char* W, int n_layers, int64_t L, int64_t L_cap, int Hkv, int d,
                          int B, int S, int R, int64_t N_cap, int64_t N_prev, int64_t* n_out,
                          int64_t* N_new, void* workspace, size_t workspace_bytes) {
  if (n_layers < 1 || n_layers > 65535)
    return fail(TS_ERR_INVALID_ARG, "%s: n_layers=%d", W, n_layers);
  if (Hkv < 1) return fail(TS_ERR_INVALID_ARG, "%s: Hkv=%d", W, Hkv);
  if (d != 64 && d != 128) return fail(TS_ERR_UNSUPPORTED, "%s: head dim %d not in {64,128}", W, d);
  if (B < 0 || S < 0 || R < 0) return fail(TS_ERR_INVALID_ARG, "%s: B, S, R must be >= 0", W);
  if (L < 0 || L > L_cap) return fail(TS_ERR_INVALID_ARG, "%s: need 0 <= L <= L_cap", W);
  if (L_cap > (int64_t(1) << 31) - 1) return fail(TS_ERR_UNSUPPORTED, "%s: L_cap >= 2^31", W);
  const int64_t N = L < (int64_t)S + B + R ? L : (int64_t)S + B + R;
  if (N_cap < N)
    return fail(TS_ERR_INVALID_ARG, "%s: N_cap=%lld < min(L, S+B+R)=%lld", W, (long long)N_cap,
                (long long)N);
  if (N_prev < 0 || N_prev > N)
    return fail(TS_ERR_INVALID_ARG, "%s: need 0 <= N_prev <= min(L, S+B+R) (N_prev=%lld, N=%lld)",
                W, (long long)N_prev, (long long)N);
  if (n_out) *n_out = N;
  *N_new = N;
  if (L == 0) return TS_OK;
  return check_ws(workspace, workspace_bytes, refresh_ws_bytes(n_layers * Hkv, L, N_cap), W);
}

int ts_partial_kv_refresh_incremental(const float* imp, const void* k, const void* v, int64_t L,
                                      int64_t L_cap, int Hkv, int d, int B, int S, int R,
                                      int32_t* idx, void* kd, void* vd, int64_t N_cap,
                                      int64_t N_prev, int64_t* n_out, int32_t* n_written,
                                      void* workspace, size_t workspace_bytes, int32_t* status,
                                      void* stream) {
  clear_error();
  const char* W = "ts_partial_kv_refresh_incremental";
  int64_t N_new = 0;
  int rc = refresh_common(W, 1, L, L_cap, Hkv, d, B, S, R, N_cap, N_prev, n_out, &N_new, workspace,
                          workspace_bytes);
  if (rc || L == 0) return rc;
  if (!imp || !k || !v || !idx || !kd || !vd) return fail(TS_ERR_INVALID_ARG, "%s: NULL tensor", W);
  return launch_refresh_incremental(1, imp, nullptr, k, nullptr, v, nullptr, L, L_cap, Hkv, d, B,
                                    S, R, N_prev, N_new, N_cap, idx, nullptr, kd, nullptr, vd,
                                    nullptr, n_written, workspace, status,
                                    static_cast<cudaStream_t>(stream));
}

int ts_partial_kv_refresh_incremental_batched(int n_layers, const float* const* imp,
                                              const void* const* k, const void* const* v,
                                              int64_t L, int64_t L_cap, int Hkv, int d, int B,
                                              int S, int R, int32_t* const* idx, void* const* kd,
                                              void* const* vd, int64_t N_cap, int64_t N_prev,
                                              int64_t* n_out, int32_t* n_written, void* workspace,
                                              size_t workspace_bytes, int32_t* status,
                                              void* stream) {
  clear_error();
  const char* W = "ts_partial_kv_refresh_incremental_batched";
  int64_t N_new = 0;
  int rc = refresh_common(W, n_layers, L, L_cap, Hkv, d, B, S, R, N_cap, N_prev, n_out, &N_new,
                          workspace, workspace_bytes);
  if (rc || L == 0) return rc;
  if (!imp || !k || !v || !idx || !kd || !vd) return fail(TS_ERR_INVALID_ARG, "%s: NULL array", W);
  return launch_refresh_incremental(n_layers, nullptr, imp, nullptr, k, nullptr, v, L, L_cap, Hkv,
                                    d, B, S, R, N_prev, N_new, N_cap, nullptr, idx, nullptr, kd,
                                    nullptr, vd, n_written, workspace, status,
                                    static_cast<cudaStream_t>(stream));
}

int ts_partial_kv_select_gather_batched(int n_layers, const float* const* imp,
                                        const void* const* k, const void* const* v, int64_t L,
                                        int64_t L_cap, int Hkv, int d, int B, int S, int R,
                                        int32_t* const* idx, void* const* kd, void* const* vd,
                                        int64_t* n_out, void* workspace, size_t workspace_bytes,
                                        int32_t* status, void* stream) {
  clear_error();
  const char* W = "ts_partial_kv_select_gather_batched";
  if (n_layers < 1 || n_layers > 65535)
    return fail(TS_ERR_INVALID_ARG, "%s: n_layers=%d", W, n_layers);
  if (Hkv < 1) return fail(TS_ERR_INVALID_ARG, "%s: Hkv=%d", W, Hkv);
  if (d != 64 && d != 128) return fail(TS_ERR_UNSUPPORTED, "%s: head dim %d not in {64,128}", W, d);
  if (B < 0 || S < 0 || R < 0) return fail(TS_ERR_INVALID_ARG, "%s: B, S, R must be >= 0", W);
  if (L < 0 || L > L_cap) return fail(TS_ERR_INVALID_ARG, "%s: need 0 <= L <= L_cap", W);
  if (L_cap > (int64_t(1) << 31) - 1) return fail(TS_ERR_UNSUPPORTED, "%s: L_cap >= 2^31", W);
  int64_t N = L < (int64_t)S + B + R ? L : (int64_t)S + B + R;
  if (n_out) *n_out = N;
  if (L == 0) return TS_OK;
  if (!imp || !k || !v || !idx || !kd || !vd) return fail(TS_ERR_INVALID_ARG, "%s: NULL array", W);
  SelectPlan p = select_plan(Hkv, L, n_layers);
  int rc = check_ws(workspace, workspace_bytes, p.ws_bytes, W);
  if (rc) return rc;
  return launch_select_gather_batched(n_layers, imp, k, v, L, L_cap, Hkv, d, B, S, R, idx, kd, vd,
                                      N, workspace, status, static_cast<cudaStream_t>(stream));
}

size_t ts_sample_workspace_bytes(int T, int V) {
  if (T < 1 || T > 64 || V < 1 || V > 262144) return 0;
  return sample_ws_bytes(T, V);
}

int ts_penalized_sample_accept_flags(const float* logits, const int32_t* tree_tokens,
                                     const int32_t* parents, int T, const int32_t* prior,
                                     int n_prior, int W, int V, float penalty, float temperature,
                                     float top_p, float min_p, const float* uniforms,
                                     int32_t* sampled, int32_t* path, int32_t* n_path,
                                     int32_t* bonus, void* workspace, size_t workspace_bytes,
                                     int flags, int32_t* status, void* stream) {
  clear_error();
  const char* F = "ts_penalized_sample_accept";
  if (flags & ~TS_PENALTY_CTRL_LITERAL) return fail(TS_ERR_INVALID_ARG, "%s: unknown flags 0x%x", F, flags);
  if (T < 1) return fail(TS_ERR_INVALID_ARG, "%s: T=%d", F, T);
  if (T > 64) return fail(TS_ERR_UNSUPPORTED, "%s: T=%d > 64", F, T);
  if (V < 1) return fail(TS_ERR_INVALID_ARG, "%s: V=%d", F, V);
  if (V > 262144) return fail(TS_ERR_UNSUPPORTED, "%s: V=%d > 262144", F, V);
  if (n_prior < 0 || W < 0) return fail(TS_ERR_INVALID_ARG, "%s: n_prior, W must be >= 0", F);
  if (!(penalty > 0.f) || !(temperature > 0.f))
    return fail(TS_ERR_INVALID_ARG, "%s: penalty and temperature must be > 0", F);
  if (!(top_p > 0.f) || !(min_p >= 0.f))
    return fail(TS_ERR_INVALID_ARG, "%s: need top_p > 0 and min_p >= 0", F);
  if (!logits || !tree_tokens || !parents || !uniforms || !sampled || !path || !n_path || !bonus ||
      (n_prior > 0 && !prior))
    return fail(TS_ERR_INVALID_ARG, "%s: NULL tensor", F);
  int rc = check_ws(workspace, workspace_bytes, sample_ws_bytes(T, V), F);
  if (rc) return rc;
  // kernel mode word: bit 0 eta pool, bit 1 literal penalty, bit 2 rejection
  const int mode = (flags & TS_PENALTY_CTRL_LITERAL) ? 2 : 0;
  return launch_sample_accept(logits, tree_tokens, parents, T, prior, n_prior, W, V, penalty,
                              temperature, top_p, min_p, mode, 0.f, 0.f, uniforms, sampled, path,
                              n_path, bonus, workspace, nullptr, nullptr, status,
                              static_cast<cudaStream_t>(stream));
}

int ts_penalized_sample_accept(const float* logits, const int32_t* tree_tokens,
                               const int32_t* parents, int T, const int32_t* prior, int n_prior,
                               int W, int V, float penalty, float temperature, float top_p,
                               float min_p, const float* uniforms, int32_t* sampled,
                               int32_t* path, int32_t* n_path, int32_t* bonus, void* workspace,
                               size_t workspace_bytes, int32_t* status, void* stream) {
  return ts_penalized_sample_accept_flags(logits, tree_tokens, parents, T, prior, n_prior, W, V,
                                          penalty, temperature, top_p, min_p, uniforms, sampled,
                                          path, n_path, bonus, workspace, workspace_bytes, 0,
                                          status, stream);
}

int ts_penalized_sample_accept_eta(const float* logits, const int32_t* tree_tokens,
                                   const int32_t* parents, int T, const int32_t* prior,
                                   int n_prior, int W, int V, float penalty, float temperature,
                                   float eta_epsilon, float eta_alpha, const float* uniforms,
                                   int32_t* sampled, int32_t* path, int32_t* n_path,
                                   int32_t* bonus, void* workspace, size_t workspace_bytes,
                                   int32_t* status, void* stream) {
  clear_error();
  const char* F = "ts_penalized_sample_accept_eta";
  if (T < 1) return fail(TS_ERR_INVALID_ARG, "%s: T=%d", F, T);
  if (T > 64) return fail(TS_ERR_UNSUPPORTED, "%s: T=%d > 64", F, T);
  if (V < 1) return fail(TS_ERR_INVALID_ARG, "%s: V=%d", F, V);
  if (V > 262144) return fail(TS_ERR_UNSUPPORTED, "%s: V=%d > 262144", F, V);
  if (n_prior < 0 || W < 0) return fail(TS_ERR_INVALID_ARG, "%s: n_prior, W must be >= 0", F);
  if (!(penalty > 0.f) || !(temperature > 0.f))
    return fail(TS_ERR_INVALID_ARG, "%s: penalty and temperature must be > 0", F);
  if (!(eta_epsilon >= 0.f) || !(eta_alpha >= 0.f) || !(eta_alpha <= 1.f))
    return fail(TS_ERR_INVALID_ARG, "%s: need eta_epsilon >= 0 and 0 <= eta_alpha <= 1", F);
  if (!logits || !tree_tokens || !parents || !uniforms || !sampled || !path || !n_path || !bonus ||
      (n_prior > 0 && !prior))
    return fail(TS_ERR_INVALID_ARG, "%s: NULL tensor", F);
  int rc = check_ws(workspace, workspace_bytes, sample_ws_bytes(T, V), F);
  if (rc) return rc;
  return launch_sample_accept(logits, tree_tokens, parents, T, prior, n_prior, W, V, penalty,
                              temperature, 1.f, 0.f, 1, eta_epsilon, eta_alpha, uniforms, sampled,
                              path, n_path, bonus, workspace, nullptr, nullptr, status,
                              static_cast<cudaStream_t>(stream));
}

int ts_kv_commit(void* k, void* v, int64_t L, int64_t L_cap, int Hkv, int d, int T,
                 const int32_t* path, const int32_t* n_path, int32_t* status, void* stream) {
  clear_error();
  const char* F = "ts_kv_commit";
  if (Hkv < 1 || T < 1) return fail(TS_ERR_INVALID_ARG, "%s: Hkv, T must be >= 1", F);
  if (T > 64) return fail(TS_ERR_UNSUPPORTED, "%s: T=%d > 64", F, T);
  if (d != 64 && d != 128) return fail(TS_ERR_UNSUPPORTED, "%s: head dim %d", F, d);
  if (L < 0 || L + T > L_cap) return fail(TS_ERR_INVALID_ARG, "%s: need L+T <= L_cap", F);
  if (!k || !v || !path || !n_path) return fail(TS_ERR_INVALID_ARG, "%s: NULL tensor", F);
  return launch_kv_commit(k, v, L, L_cap, Hkv, d, T, path, n_path, status,
                          static_cast<cudaStream_t>(stream));
}

int ts_kv_commit_batched(int n_layers, void* const* k, void* const* v, int64_t L, int64_t L_cap,
                         int Hkv, int d, int T, const int32_t* path, const int32_t* n_path,
                         int32_t* status, void* stream) {
  clear_error();
  const char* F = "ts_kv_commit_batched";
  if (n_layers < 1 || n_layers > 65535) return fail(TS_ERR_INVALID_ARG, "%s: n_layers=%d", F, n_layers);
  if (Hkv < 1 || T < 1) return fail(TS_ERR_INVALID_ARG, "%s: Hkv, T must be >= 1", F);
  if (T > 64) return fail(TS_ERR_UNSUPPORTED, "%s: T=%d > 64", F, T);
  if (d != 64 && d != 128) return fail(TS_ERR_UNSUPPORTED, "%s: head dim %d", F, d);
  if (L < 0 || L + T > L_cap) return fail(TS_ERR_INVALID_ARG, "%s: need L+T <= L_cap", F);
  if (!k || !v || !path || !n_path) return fail(TS_ERR_INVALID_ARG, "%s: NULL array", F);
  return launch_kv_commit_batched(n_layers, k, v, L, L_cap, Hkv, d, T, path, n_path, status,
                                  static_cast<cudaStream_t>(stream));
}

int ts_kv_append_batched_flags(int n_layers, void* const* k, void* const* v, const void* k_rows,
                               const void* v_rows, int64_t L, int64_t L_cap, int Hkv, int d,
                               int T, int flags, int32_t* status, void* stream) {
  clear_error();
  const char* F = "ts_kv_append_batched";
  if (flags & ~TS_KV_V_FP16) return fail(TS_ERR_INVALID_ARG, "%s: unknown flags 0x%x", F, flags);
  if (n_layers < 1 || n_layers > 65535) return fail(TS_ERR_INVALID_ARG, "%s: n_layers=%d", F, n_layers);
  if (Hkv < 1 || T < 1) return fail(TS_ERR_INVALID_ARG, "%s: Hkv, T must be >= 1", F);
  if (T > 64) return fail(TS_ERR_UNSUPPORTED, "%s: T=%d > 64", F, T);
  if (d != 64 && d != 128) return fail(TS_ERR_UNSUPPORTED, "%s: head dim %d", F, d);
  if (L < 0 || L + T > L_cap) return fail(TS_ERR_INVALID_ARG, "%s: need L+T <= L_cap", F);
  if (!k || !v || !k_rows || !v_rows) return fail(TS_ERR_INVALID_ARG, "%s: NULL array", F);
  if ((reinterpret_cast<uintptr_t>(k_rows) | reinterpret_cast<uintptr_t>(v_rows)) & 15)
    return fail(TS_ERR_INVALID_ARG, "%s: k_rows and v_rows must be 16-byte aligned", F);
  return launch_kv_append_batched(n_layers, k, v, k_rows, v_rows, L, L_cap, Hkv, d, T,
                                  (flags & TS_KV_V_FP16) != 0, status,
                                  static_cast<cudaStream_t>(stream));
}

int ts_kv_append_batched(int n_layers, void* const* k, void* const* v, const void* k_rows,
                         const void* v_rows, int64_t L, int64_t L_cap, int Hkv, int d, int T,
                         void* stream) {
  return ts_kv_append_batched_flags(n_layers, k, v, k_rows, v_rows, L, L_cap, Hkv, d, T, 0,
                                    nullptr, stream);
}

size_t ts_reject_workspace_bytes(int V) {
  if (V < 1 || V > 262144) return 0;
  return reject_ws_bytes(V);
}

int ts_rejection_sample_accept(const float* logits, const float* q, const int32_t* tree_tokens,
                               const int32_t* parents, int T, const int32_t* prior, int n_prior,
                               int W, int V, float penalty, float temperature, float top_p,
                               float min_p, const float* u_accept, const float* u_draw,
                               int32_t* path, int32_t* n_path, int32_t* bonus, void* workspace,
                               size_t workspace_bytes, int flags, int32_t* status, void* stream) {
  clear_error();
  const char* F = "ts_rejection_sample_accept";
  if (flags & ~TS_PENALTY_CTRL_LITERAL) return fail(TS_ERR_INVALID_ARG, "%s: unknown flags 0x%x", F, flags);
  if (T < 1) return fail(TS_ERR_INVALID_ARG, "%s: T=%d", F, T);
  if (T > 64) return fail(TS_ERR_UNSUPPORTED, "%s: T=%d > 64", F, T);
  if (V < 1) return fail(TS_ERR_INVALID_ARG, "%s: V=%d", F, V);
  if (V > 262144) return fail(TS_ERR_UNSUPPORTED, "%s: V=%d > 262144", F, V);
  if (n_prior < 0 || W < 0) return fail(TS_ERR_INVALID_ARG, "%s: n_prior, W must be >= 0", F);
  if (!(penalty > 0.f) || !(temperature > 0.f))
    return fail(TS_ERR_INVALID_ARG, "%s: penalty and temperature must be > 0", F);
  if (!(top_p > 0.f) || !(min_p >= 0.f))
    return fail(TS_ERR_INVALID_ARG, "%s: need top_p > 0 and min_p >= 0", F);
  if (!logits || !q || !tree_tokens || !parents || !u_accept || !u_draw || !path || !n_path ||
      !bonus || (n_prior > 0 && !prior))
    return fail(TS_ERR_INVALID_ARG, "%s: NULL tensor", F);
  int rc = check_ws(workspace, workspace_bytes, reject_ws_bytes(V), F);
  if (rc) return rc;
  return launch_reject_accept(logits, q, tree_tokens, parents, T, prior, n_prior, W, V, penalty,
                              temperature, top_p, min_p, (flags & TS_PENALTY_CTRL_LITERAL) ? 1 : 0,
                              u_accept, u_draw, path, n_path, bonus, workspace, status,
                              static_cast<cudaStream_t>(stream));
}

size_t ts_ngram_table_bytes(int V, int cap) {
  if (V < 1 || cap < 1 || cap > 64) return 0;
  return ngram_table_bytes(V, cap);
}

int ts_ngram_insert(int32_t* table, int V, int cap, const int32_t* tokens, int n_tokens,
                    int start, int32_t* status, void* stream) {
  clear_error();
  const char* F = "ts_ngram_insert";
  if (V < 1) return fail(TS_ERR_INVALID_ARG, "%s: V must be >= 1", F);
  if (cap < 1 || cap > 64) return fail(TS_ERR_UNSUPPORTED, "%s: cap=%d outside [1, 64]", F, cap);
  if (n_tokens < 0 || start < 0) return fail(TS_ERR_INVALID_ARG, "%s: negative length", F);
  if (!table || (n_tokens > 0 && !tokens)) return fail(TS_ERR_INVALID_ARG, "%s: NULL tensor", F);
  return launch_ngram_insert(table, V, cap, tokens, n_tokens, start, status,
                             static_cast<cudaStream_t>(stream));
}

int ts_ngram_build_tree(const int32_t* table, int V, int cap, const int32_t* root_token,
                        const int32_t* head_topk, int n_heads, int head_k, int k,
                        const uint32_t* rand_keys, int T_max, int32_t* parents,
                        int32_t* tokens, int32_t* n_nodes, int32_t* status, void* stream) {
  clear_error();
  const char* F = "ts_ngram_build_tree";
  if (V < 1) return fail(TS_ERR_INVALID_ARG, "%s: V must be >= 1", F);
  if (cap < 1 || cap > 64) return fail(TS_ERR_UNSUPPORTED, "%s: cap=%d outside [1, 64]", F, cap);
  if (T_max < 1 || T_max > 64) return fail(TS_ERR_UNSUPPORTED, "%s: T_max=%d outside [1, 64]", F, T_max);
  if (n_heads < 0 || head_k < 0 || k < 0 || k > cap)
    return fail(TS_ERR_INVALID_ARG, "%s: need n_heads, head_k >= 0 and 0 <= k <= cap", F);
  if (!table || !root_token || !parents || !tokens || !n_nodes || (k > 0 && !rand_keys) ||
      (n_heads * head_k > 0 && !head_topk))
    return fail(TS_ERR_INVALID_ARG, "%s: NULL tensor", F);
  return launch_ngram_tree(table, V, cap, root_token, head_topk, n_heads, head_k, k, rand_keys,
                           T_max, parents, tokens, n_nodes, status,
                           static_cast<cudaStream_t>(stream));
}

}  // extern "C"
