/*
 * tokenswift_gb300.h — C ABI of the GB300 (sm_103a) per-step decode hot path of
 * TokenSwift-style lossless ultra-long generation.
 *
 * Source method: "TokenSwift: Lossless Acceleration of Ultra Long Sequence
 * Generation" (Wu, Shen, Jia, Wang, Zheng; ICML 2025).  One decoding step
 * drafts with a partial KV cache, verifies the draft tree with the full KV
 * cache, samples with a contextual penalty and accepts the longest exactly
 * matching draft, then updates the KV cache (§3.1 Overview, Figure 2).
 *
 * Conventions shared by every call:
 *   - Every tensor pointer is a DEVICE pointer owned by the caller, unless a
 *     parameter says "host".  Tensors are dense row-major in the layout given.
 *     bf16 tensors are passed as `const void*` holding IEEE bfloat16 values.
 *   - A V cache may hold IEEE binary16 (fp16) values instead: the calls that
 *     only move cache rows (gather, refresh, commit) copy bytes and take
 *     either; (1) reads an fp16 V cache with TS_VERIFY_V_FP16 and
 *     ts_kv_append_batched_flags writes one with TS_KV_V_FP16.
 *   - The library allocates no device memory.  Scratch space is a caller
 *     buffer (`workspace`, 256-byte aligned) of at least the size reported by
 *     the matching *_workspace_bytes() query.
 *   - Every call only enqueues work on `stream` (a cudaStream_t; NULL = the
 *     legacy default stream) and returns without synchronising.
 *   - Return value: TS_OK, or a ts_status code for arguments rejected on the
 *     host before anything was enqueued (a message is then available from
 *     ts_last_error(), per calling thread), or TS_ERR_CUDA if a launch failed.
 *   - `status` is an optional (may be NULL) device int32 the caller zeroes;
 *     kernels write a nonzero ts_status into it when they meet bad device-side
 *     data (a parent index or token id out of range) or a bounded wait that
 *     ran out.  They never trap.  Read it after synchronising the stream.
 *   - Limits: 1 <= T <= 64 tree nodes (parents[0] = -1, parents[i] < i);
 *     Hq % Hkv == 0; d in {64, 128}; T*Hq/Hkv <= 512; vocabulary V <= 262144.
 *   - Concurrent calls that share a workspace buffer race; give each stream
 *     its own workspace.
 */
#ifndef TOKENSWIFT_GB300_H
#define TOKENSWIFT_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum ts_status {
  TS_OK = 0,
  TS_ERR_INVALID_ARG = 1,  /* argument out of its documented domain        */
  TS_ERR_UNSUPPORTED = 2,  /* valid but outside the library's limits       */
  TS_ERR_CUDA = 3,         /* a CUDA launch or runtime call failed          */
  TS_ERR_TIMEOUT = 4,      /* a bounded device-side wait ran out            */
  TS_ERR_WORKSPACE = 5     /* workspace missing, too small or misaligned    */
} ts_status;

/* Static description of a status code. */
const char* ts_status_string(int status);
/* Message of the last failed call on this thread ("" if none). */
const char* ts_last_error(void);
/* Library ABI version (major*100 + minor). */
int ts_version(void);

/* Limit of one bounded device-side wait, in SM clock cycles, for kernels
 * launched after this call (from any thread): the verification kernel of (1)
 * gives up a wait on another warp's or the copy engine's progress after
 * `cycles` clocks, writes TS_ERR_TIMEOUT into `status`, waits for its own
 * copies and tensor-core work in flight (with the default limit), releases
 * its tensor memory and returns; that call's outputs are then undefined.
 * `cycles` <= 0 restores the default, 2^31 cycles (about one second).  A
 * small limit exists to exercise the expiry path; the paper has no
 * counterpart.  Returns TS_OK. */
int ts_set_wait_limit(int64_t cycles);

/* ------------------------------------------------------------------------
 * (1) Tree verification attention + attention importance.
 *
 * §3.1 Overview: the target model verifies the draft with the FULL KV cache;
 * §E Tree-Based Attention: each tree token attends only to its predecessors;
 * §3.3 Dynamic KV Cache Management: importance of a cached pair is the
 * query-key dot product, with GQA query heads partitioned per KV head and
 * their scores aggregated.
 *
 * For tree node i, query head h, KV head kv = h / (Hq/Hkv):
 *   s_j = q[i,h,:] . k[kv,j,:] / sqrt(d) over j in [0, L) and j = L + a for
 *   every node a on the root path of i (i itself included);
 *   o[i,h,:] = softmax_j(s) . v[kv,j,:]  (fp32),
 *   lse[i,h] = ln sum_j exp(s_j)          (fp32),
 *   imp[kv,j] = sum over the last n_imp nodes i and the heads h of group kv
 *               of s_{i,h,j}, for j in [0, L)   (fp32).
 *
 * q       [T, Hq, d] bf16 (post-RoPE tree queries)
 * k, v    [Hkv, L_cap, d] bf16; rows [0,L) = committed cache, rows
 *         [L, L+T) = the tree tokens' own keys/values.  L + T <= L_cap.
 * parents [T] int32, device; parents[0] = -1, 0 <= parents[i] < i.
 * n_imp   number of trailing tree queries used for importance (<= 0: all T).
 * o       [T, Hq, d] fp32 out.   lse [T, Hq] fp32 out, or NULL.
 * imp     [Hkv, L] fp32 out, or NULL to skip importance.
 * workspace >= ts_verify_workspace_bytes(T, Hq, Hkv, d, L).
 *
 * Precision: Q.K^T in bf16 with fp32 accumulation; the probabilities are
 * rounded to fp16 for the P.V product (fp32 accumulation), so V values must
 * lie in the fp16 range |v| < 65504.  Larger values saturate to +-65504 and
 * the kernel writes TS_ERR_UNSUPPORTED into `status`.
 * ------------------------------------------------------------------------ */
size_t ts_verify_workspace_bytes(int T, int Hq, int Hkv, int d, int64_t L);
int ts_verify_attention(const void* q, const void* k, const void* v,
                        int64_t L, int64_t L_cap, const int32_t* parents,
                        int T, int Hq, int Hkv, int d, int n_imp,
                        float* o, float* lse, float* imp,
                        void* workspace, size_t workspace_bytes,
                        int32_t* status, void* stream);
/* The same call with flags.  TS_VERIFY_V_FP16: v [Hkv, L_cap, d] holds fp16
 * values (a V cache kept in the precision of the P.V product, as
 * ts_kv_append_batched_flags with TS_KV_V_FP16 writes it).  The kernel then
 * skips its per-tile bf16 -> fp16 conversion; for V values that fp16
 * represents exactly (normal bf16 values below 65504 in magnitude, the
 * conversion rounding the rest exactly as the bf16 path does) the outputs are
 * bit-identical to the bf16 call on the same values.  Unknown flag bits:
 * TS_ERR_INVALID_ARG. */
#define TS_VERIFY_V_FP16 1
int ts_verify_attention_flags(const void* q, const void* k, const void* v,
                              int64_t L, int64_t L_cap, const int32_t* parents,
                              int T, int Hq, int Hkv, int d, int n_imp,
                              float* o, float* lse, float* imp,
                              void* workspace, size_t workspace_bytes, int flags,
                              int32_t* status, void* stream);

/* ------------------------------------------------------------------------
 * (1b) Softmax-weighted importance (a variant of the importance of (1)).
 *
 * §3.3 Dynamic KV Cache Management ranks cached pairs by query-key scores,
 * GQA query heads partitioned per KV head and their scores aggregated.  This
 * call aggregates the normalised attention weights instead: the probability
 * mass each committed position receives from the importance queries.
 *
 *   imp[kv,j] = sum over the last n_imp nodes i and the heads h of group kv
 *               of exp(q[i,h,:] . k[kv,j,:] / sqrt(d) - lse[i,h]),
 *               for j in [0, L)   (fp32)
 *
 * q       [T, Hq, d] bf16, the same tree queries given to (1).
 * k       [Hkv, L_cap, d] bf16; only rows [0, L) are read.  0 <= L <= L_cap.
 * lse     [T, Hq] fp32, device: each row's natural-log log-sum-exp over
 *         everything it attends to, as (1) returns it.
 * n_imp   number of trailing tree queries (<= 0: all T), n_imp <= T.
 * imp     [Hkv, L] fp32 out (row stride L); call (1) with imp = NULL and pass
 *         this array to (2).
 * L = 0 writes nothing and accepts NULL buffers.
 * No workspace: every position is written by one thread.  The K cache is
 * read once more (V is not read); the scores use bf16 operands with fp32
 * accumulation, the exponentials fp32.  Unsupported: n_imp*Hq/Hkv query
 * rows whose staging exceeds the shared memory of one SM (more than 448 rows
 * at d = 128).  The caller owns every buffer; nothing is allocated.
 * ------------------------------------------------------------------------ */
int ts_importance_softmax(const void* q, const void* k, const float* lse,
                          int64_t L, int64_t L_cap, int T, int Hq, int Hkv,
                          int d, int n_imp, float* imp,
                          int32_t* status, void* stream);

/* ------------------------------------------------------------------------
 * (2) Dynamic partial KV cache: top-B selection and gather.
 *
 * §3.3 Dynamic KV Cache Management: a fixed budget; the initial |S| pairs are
 * preserved and less important pairs are replaced; §3.1: the partial cache is
 * what drafting attends to.
 *
 * Per KV head: if L <= S+B+R every position is kept; otherwise the kept set
 * is [0,S) (sinks) + [L-R, L) (recent) + the B best positions of [S, L-R)
 * ranked by (imp desc, position asc).  The N = min(L, S+B+R) kept positions
 * are written in ascending order to idx[kv, 0:N] and their K/V rows are
 * copied bit for bit into kd/vd[kv, 0:N, :].
 *
 * imp     [Hkv, L] fp32 (typically from ts_verify_attention)
 * k, v    [Hkv, L_cap, d] bf16 full cache
 * idx     [Hkv, N] int32 out;  kd, vd [Hkv, N, d] bf16 out
 * n_out   HOST int64 out (may be NULL): N
 * workspace >= ts_select_workspace_bytes(Hkv, L).
 * ------------------------------------------------------------------------ */
size_t ts_select_workspace_bytes(int Hkv, int64_t L);
int ts_partial_kv_select_gather(const float* imp, const void* k, const void* v,
                                int64_t L, int64_t L_cap, int Hkv, int d,
                                int B, int S, int R,
                                int32_t* idx, void* kd, void* vd, int64_t* n_out,
                                void* workspace, size_t workspace_bytes,
                                int32_t* status, void* stream);

/* Allocation-free form of (2).  The pages have no counterpart: this entry
 * point exists for callers that may not allocate device memory -- a plugin
 * running inside a host runtime that owns every device allocation, or a
 * serving loop that forbids allocation (and the synchronisation it can bring)
 * once running.  It takes no workspace: its scratch is one fixed 10 MiB array
 * of device memory inside the library, which every GPU that loads the library
 * holds until the process exits.  That covers Hkv*L up to about 1.2 million
 * cached positions (e.g. 8 KV heads at 102,400 tokens); larger shapes return
 * TS_ERR_UNSUPPORTED with the size they would need.  Inputs and outputs are
 * the caller's, exactly as in ts_partial_kv_select_gather, and the results are
 * identical.  The first call on a device looks up the array's device address
 * (with that device current) and caches it; make that first call before any
 * stream capture.  All calls on a device share the array and each call
 * overwrites what the previous one left there (the parts that must start at
 * zero are cleared on the stream by every call), so calls that overlap on the
 * GPU -- on different streams, or from different host threads -- race and
 * must be serialised by the caller.  The cached address belongs to the
 * device's current context: after cudaDeviceReset (or any teardown of the
 * primary context) the array lives at a new address and the cache is stale,
 * so reload the library (a new process) before calling this again on that
 * device. */
int ts_partial_kv_select_gather_noalloc(const float* imp, const void* k, const void* v,
                                        int64_t L, int64_t L_cap, int Hkv, int d,
                                        int B, int S, int R,
                                        int32_t* idx, void* kd, void* vd, int64_t* n_out,
                                        int32_t* status, void* stream);

/* Batched form of (2): the same selection and gather for n_layers layers in
 * one pipeline of launches.  The refreshed partial cache of a layer is only
 * read by the next step's drafting, so a step may verify every layer first
 * and refresh all partial caches together.  imp, k, v, idx, kd, vd are DEVICE
 * arrays of n_layers pointers (each pointing at that layer's tensor with the
 * single-layer layout above); L, L_cap, Hkv, d, B, S, R are shared.
 * workspace >= ts_select_batched_workspace_bytes(n_layers, Hkv, L). */
size_t ts_select_batched_workspace_bytes(int n_layers, int Hkv, int64_t L);
int ts_partial_kv_select_gather_batched(int n_layers, const float* const* imp,
                                        const void* const* k, const void* const* v,
                                        int64_t L, int64_t L_cap, int Hkv, int d,
                                        int B, int S, int R,
                                        int32_t* const* idx, void* const* kd, void* const* vd,
                                        int64_t* n_out, void* workspace, size_t workspace_bytes,
                                        int32_t* status, void* stream);

/* ------------------------------------------------------------------------
 * (2b) Incremental partial-cache refresh.
 *
 * §3.3 Dynamic KV Cache Management: the budgeted cache keeps the initial |S|
 * pairs and replaces the less important pairs as generation proceeds.  The
 * kept set is the one (2) computes (same ranking, same tie rule); instead of
 * rewriting the compact cache in position order it is updated in place:
 *   - slot s < N_prev keeps its row while idx[kv,s] stays selected;
 *   - the newly selected positions, ascending, take the freed slots in
 *     ascending slot order, then slots N_prev .. N_new-1, where
 *     N_new = min(L, S+B+R) (the cache grows until it reaches the budget);
 *   - only those rows are copied (K and V, bit for bit).
 * Afterwards idx[kv, 0:N_new] holds exactly the kept set, in slot order, and
 * kd/vd[kv, s, :] = k/v[kv, idx[kv, s], :].  Attention over the compact
 * cache does not depend on the slot order.
 *
 * imp     [Hkv, L] fp32.   k, v [Hkv, L_cap, d] bf16.
 * idx     [Hkv, N_cap] int32, in/out; kd, vd [Hkv, N_cap, d] bf16, in/out;
 *         N_cap >= min(L, S+B+R) is the fixed row stride.
 * N_prev  slots valid before the call, 0 <= N_prev <= N_new (0 on the first
 *         call: the result then equals (2)'s ascending output).
 * n_out   N_new (may be NULL).
 * n_written [n_layers * Hkv] int32 device out, or NULL: rows written per
 *         (layer, KV head).
 * workspace >= ts_refresh_workspace_bytes(n_layers, Hkv, L, N_cap).
 * Previous slots holding a position outside [0, L), or the same position
 * twice, are reported as TS_ERR_INVALID_ARG in `status`; the contents are
 * then unspecified, but no access leaves the buffers.  The batched form
 * takes device arrays of per-layer pointers, as in (2).
 * ------------------------------------------------------------------------ */
size_t ts_refresh_workspace_bytes(int n_layers, int Hkv, int64_t L, int64_t N_cap);
int ts_partial_kv_refresh_incremental(const float* imp, const void* k, const void* v,
                                      int64_t L, int64_t L_cap, int Hkv, int d,
                                      int B, int S, int R, int32_t* idx, void* kd,
                                      void* vd, int64_t N_cap, int64_t N_prev,
                                      int64_t* n_out, int32_t* n_written,
                                      void* workspace, size_t workspace_bytes,
                                      int32_t* status, void* stream);
int ts_partial_kv_refresh_incremental_batched(int n_layers, const float* const* imp,
                                              const void* const* k, const void* const* v,
                                              int64_t L, int64_t L_cap, int Hkv, int d,
                                              int B, int S, int R, int32_t* const* idx,
                                              void* const* kd, void* const* vd,
                                              int64_t N_cap, int64_t N_prev,
                                              int64_t* n_out, int32_t* n_written,
                                              void* workspace, size_t workspace_bytes,
                                              int32_t* status, void* stream);

/* ------------------------------------------------------------------------
 * (3) Contextual-penalty sampling and exact-match tree acceptance.
 *
 * §3.4 Contextual Penalty: penalise the most recent W tokens; §D.1: top-p
 * keeps the smallest set of tokens whose cumulative probability exceeds
 * top_p (every token when top_p >= 1), min-p keeps tokens with
 * p >= min_p * p_max; Table 11 sets penalty 1.2, window 1024, temperature
 * 1.0, top-p 0.9, min-p 0.05; §3.1: the longest draft that matches the
 * target's own tokens is accepted.
 *
 * For every node i (in parallel): the window is the last W tokens of
 * (prior[0:n_prior] followed by the drafted tokens on the root path of i,
 * root excluded); each distinct windowed token t gets x_t/penalty if x_t > 0,
 * else x_t*penalty; all logits are divided by temperature; p = softmax;
 * tokens ranked by (p desc, id asc); rank r is kept iff the mass of the ranks
 * before it is <= top_p (or top_p >= 1) AND p >= min_p * p_max (rank 0
 * always kept); the draw is the first kept rank whose cumulative kept mass
 * exceeds uniforms[i] times the kept mass.  sampled[i] receives it.
 * Acceptance: root accepted; node c accepted iff its parent is accepted and
 * tree_tokens[c] == sampled[parents[c]]; the deepest accepted node (ties to
 * the lower index) gives path[0:n_path] (root first) and bonus = its sample.
 *
 * logits [T, V] fp32; tree_tokens [T] int32 (tree_tokens[0] = root token,
 * which is also prior[n_prior-1]); parents [T]; prior [n_prior] int32;
 * uniforms [T] fp32 in [0,1); sampled [T] int32 out; path [T] int32 out;
 * n_path [1] int32 out; bonus [1] int32 out.  All device pointers.
 * temperature > 0, penalty > 0, 0 < top_p, 0 <= min_p.
 * workspace >= ts_sample_workspace_bytes(T, V).
 * ------------------------------------------------------------------------ */
size_t ts_sample_workspace_bytes(int T, int V);
int ts_penalized_sample_accept(const float* logits, const int32_t* tree_tokens,
                               const int32_t* parents, int T,
                               const int32_t* prior, int n_prior, int W, int V,
                               float penalty, float temperature, float top_p, float min_p,
                               const float* uniforms,
                               int32_t* sampled, int32_t* path, int32_t* n_path,
                               int32_t* bonus,
                               void* workspace, size_t workspace_bytes,
                               int32_t* status, void* stream);

/* The same call with flags.  TS_PENALTY_CTRL_LITERAL: the literal CTRL
 * penalty, every windowed logit divided by `penalty` whatever its sign
 * (without the flag, non-positive windowed logits are multiplied by it).
 * Unknown flag bits are rejected (TS_ERR_INVALID_ARG). */
#define TS_PENALTY_CTRL_LITERAL 1
int ts_penalized_sample_accept_flags(const float* logits, const int32_t* tree_tokens,
                                     const int32_t* parents, int T,
                                     const int32_t* prior, int n_prior, int W, int V,
                                     float penalty, float temperature,
                                     float top_p, float min_p,
                                     const float* uniforms,
                                     int32_t* sampled, int32_t* path, int32_t* n_path,
                                     int32_t* bonus,
                                     void* workspace, size_t workspace_bytes, int flags,
                                     int32_t* status, void* stream);

/* eta-sampling variant (§D.1, Table 12): the same window, penalty,
 * temperature, draw and acceptance, with the kept set {p >= eta},
 * eta = min(eta_epsilon, eta_alpha * exp(-H)) and H the entropy (nats) of
 * the penalised, tempered distribution, in place of top-p and min-p.
 * eta_epsilon >= 0, 0 <= eta_alpha <= 1 (then eta <= p_max and the kept set
 * is never empty).  Same workspace as ts_penalized_sample_accept. */
int ts_penalized_sample_accept_eta(const float* logits, const int32_t* tree_tokens,
                                   const int32_t* parents, int T,
                                   const int32_t* prior, int n_prior, int W, int V,
                                   float penalty, float temperature,
                                   float eta_epsilon, float eta_alpha,
                                   const float* uniforms,
                                   int32_t* sampled, int32_t* path, int32_t* n_path,
                                   int32_t* bonus,
                                   void* workspace, size_t workspace_bytes,
                                   int32_t* status, void* stream);

/* ------------------------------------------------------------------------
 * (3b) Rejection-sampling acceptance (speculative sampling over the tree).
 *
 * A. Lossless Nature of Speculative Decoding: acceptance and rejection
 * cases together reproduce the target distribution.  From the root, at each
 * accepted node n the children are tried in index order as draws from
 * q[n, :] (the draft distribution that proposed n's children).  Child c with
 * token x is accepted iff u_accept[c] * q[n, x] < p_n(x); p_n is node n's
 * target distribution, formed exactly as in (3): penalty window along n's
 * root path, temperature, top-p and min-p, renormalised over the kept set.
 * On a rejection p_n becomes max(p_n - q[n, :], 0), renormalised, and the
 * next child is tried.  When no child is accepted, the bonus token is drawn
 * from the current p_n with u_draw[n], by inverse CDF over token ids.
 *
 * logits [T, V] fp32; q [T, V] fp32 (rows sum to 1); tree_tokens, parents
 * [T] int32; prior [n_prior] int32 ending with the root token; u_accept,
 * u_draw [T] fp32 in [0, 1).  Outputs as in (3): path [T] int32 (node
 * indices, root first), n_path [1], bonus [1].  flags:
 * TS_PENALTY_CTRL_LITERAL as in (3).  workspace >=
 * ts_reject_workspace_bytes(V).
 * Every node's outcome (its accepted child, or its bonus token) depends only
 * on that node's row, window and children, so all nodes are resolved in
 * parallel (the slices and merge of (3), then the chain over the node's
 * kept set) and the path follows the outcomes from the root.
 * ------------------------------------------------------------------------ */
size_t ts_reject_workspace_bytes(int V);
int ts_rejection_sample_accept(const float* logits, const float* q,
                               const int32_t* tree_tokens, const int32_t* parents, int T,
                               const int32_t* prior, int n_prior, int W, int V,
                               float penalty, float temperature, float top_p, float min_p,
                               const float* u_accept, const float* u_draw,
                               int32_t* path, int32_t* n_path, int32_t* bonus,
                               void* workspace, size_t workspace_bytes, int flags,
                               int32_t* status, void* stream);

/* ------------------------------------------------------------------------
 * (4) KV commit of the accepted path.
 *
 * §3.1: after verification the KV cache is updated with the accepted draft.
 * For t = 1 .. n_path-1: row L + path[t] of every KV head is copied to row
 * L + t (the root's row is already at L), in k and v, in place.  path and
 * n_path are device arrays as written by ts_penalized_sample_accept, so no
 * host synchronisation is needed between the two calls.  1 <= n_path <= T.
 * ------------------------------------------------------------------------ */
int ts_kv_commit(void* k, void* v, int64_t L, int64_t L_cap, int Hkv, int d, int T,
                 const int32_t* path, const int32_t* n_path,
                 int32_t* status, void* stream);
/* Every layer in one launch: k and v are device arrays of n_layers pointers,
 * each layer's cache [Hkv, L_cap, d] bf16 as above; the same path moves the
 * same rows in every layer. */
int ts_kv_commit_batched(int n_layers, void* const* k, void* const* v, int64_t L,
                         int64_t L_cap, int Hkv, int d, int T, const int32_t* path,
                         const int32_t* n_path, int32_t* status, void* stream);

/* The draft tree's own K/V rows written into every layer's cache (what the
 * verification forward produces for the tree tokens, §3.1): rows [L, L+T)
 * of KV head kv of layer l are set from k_rows / v_rows
 * [n_layers][Hkv][T][d] bf16 (device, 16-byte aligned, packed).  k and v
 * are device arrays of n_layers cache pointers as in ts_kv_commit_batched.
 * L + T <= L_cap.  One launch; the copies are bit for bit. */
int ts_kv_append_batched(int n_layers, void* const* k, void* const* v,
                         const void* k_rows, const void* v_rows, int64_t L,
                         int64_t L_cap, int Hkv, int d, int T, void* stream);
/* The same with flags.  TS_KV_V_FP16: the V caches hold fp16; each bf16
 * value of v_rows is rounded to the nearest fp16 on the way in (exact for
 * normal values below 65504 in magnitude); larger magnitudes saturate to
 * +-65504, NaN stays NaN, and either writes TS_ERR_UNSUPPORTED to `status`
 * (may be NULL).  K rows are copied bit for bit.  Unknown flag bits:
 * TS_ERR_INVALID_ARG. */
#define TS_KV_V_FP16 1
int ts_kv_append_batched_flags(int n_layers, void* const* k, void* const* v,
                               const void* k_rows, const void* v_rows, int64_t L,
                               int64_t L_cap, int Hkv, int d, int T, int flags,
                               int32_t* status, void* stream);

/* ------------------------------------------------------------------------
 * (5) Token reutilization: the 4-gram table and the draft-tree builder.
 *
 * §3.1: after verification the n-gram table is updated; §3.2 / §3.4:
 * frequent n-grams supply extra draft candidates, with random selection
 * among several valid ones; §B.2 / Table 10: 4-grams, at most k retrieved
 * (k = 20, Table 11); §4.4.1 / §B.2: the extra heads' candidates form the
 * ternary full tree [1,3,3,3].
 *
 * Table: one int32 device buffer of ts_ngram_table_bytes(V, cap) bytes,
 * zeroed by the caller before first use, owned by the caller.  The 4-gram
 * (a, b, c, d) is stored under key a as the continuation (b, c, d); each key
 * keeps at most cap distinct continuations (cap <= 64), the oldest
 * overwritten first; a repeated continuation is neither duplicated nor moved.
 * ------------------------------------------------------------------------ */
size_t ts_ngram_table_bytes(int V, int cap);

/* Insert the 4-grams ending at positions start .. n_tokens-1 of tokens
 * [n_tokens] (device int32; positions below 3 have no 4-gram), in position
 * order.  A token outside [0, V) skips its 4-grams and sets
 * TS_ERR_INVALID_ARG in *status (device word, may be NULL). */
int ts_ngram_insert(int32_t* table, int V, int cap, const int32_t* tokens, int n_tokens,
                    int start, int32_t* status, void* stream);

/* Draft tree for the next step.  root_token [1] (device; e.g. the bonus
 * token written by ts_penalized_sample_accept), head_topk [n_heads][head_k]
 * (device int32: candidate c of extra head d+1), rand_keys [cap] (device
 * uint32, the random keys of the root's stored continuations, oldest slot
 * first).  The root's continuations are selected: all of them (oldest
 * first) when at most k are stored, else the k with the smallest
 * (rand_keys[slot], slot) in that order.  The tree is the root, then the
 * heads' tree in breadth-first order (depth-d nodes carry head d's
 * candidates), then each selected continuation merged as a path from the
 * root (an existing child with the same token is followed, else a node is
 * appended while fewer than T_max exist).  Outputs (device int32): parents
 * [T_max] (parents[0] = -1, parents[i] < i), tokens [T_max], n_nodes [1];
 * entries past n_nodes are left untouched.  1 <= T_max <= 64,
 * 0 <= n_heads * head_k, k <= cap. */
int ts_ngram_build_tree(const int32_t* table, int V, int cap, const int32_t* root_token,
                        const int32_t* head_topk, int n_heads, int head_k, int k,
                        const uint32_t* rand_keys, int T_max, int32_t* parents,
                        int32_t* tokens, int32_t* n_nodes, int32_t* status, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* TOKENSWIFT_GB300_H */
