// Shared internals of the tokenswift_gb300 library (host + device helpers).
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>
#include <stddef.h>

#include "tokenswift_gb300.h"

namespace ts {

// ---------------------------------------------------------------- host side
int fail(int code, const char* fmt, ...);     // record message, return code
void clear_error();
int launch_status(const char* what);          // TS_ERR_CUDA if the last launch failed

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }
__host__ __device__ __forceinline__ int64_t imax64(int64_t a, int64_t b) { return a > b ? a : b; }
__host__ __device__ __forceinline__ int64_t imin64(int64_t a, int64_t b) { return a < b ? a : b; }

// ---------------------------------------------------------------- device side
__device__ __forceinline__ float bf2f(__nv_bfloat16 x) { return __bfloat162float(x); }

__device__ __forceinline__ void unpack_bf16x8(const uint4& u, float* f) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ int warp_sum_int(int v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Order-preserving map float -> uint32 (larger float -> larger key); -0.0 and
// +0.0 compare equal as floats, so both map to the key of +0.0.
__device__ __forceinline__ uint32_t float_key(float f) {
  uint32_t u = __float_as_uint(f);
  if ((u << 1) == 0u) u = 0u;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ void set_status(int32_t* status, int code) {
  if (status) atomicCAS(status, 0, code);
}

// Ancestor-or-self bit masks of the draft tree (T <= 64), computed by one
// thread; invalid parent indices are reported and treated as the root.
__device__ __forceinline__ void tree_masks(const int32_t* parents, int T,
                                           unsigned long long* anc, int32_t* status) {
  for (int i = 0; i < T; ++i) {
    int p = parents[i];
    unsigned long long m = 1ull << i;
    if (i == 0) {
      if (p != -1) set_status(status, TS_ERR_INVALID_ARG);
    } else if (p < 0 || p >= i) {
      set_status(status, TS_ERR_INVALID_ARG);
    } else {
      m |= anc[p];
    }
    anc[i] = m;
  }
}

// Programmatic dependent launch: a kernel launched with pdl_config may
// become resident while the previous kernel of its stream is finishing; it
// must call griddep_wait() before reading anything that kernel wrote.  A
// kernel calls griddep_launch_dependents() once the next kernel may be
// scheduled (that kernel still waits for this one's completion and memory).
__device__ __forceinline__ void griddep_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void griddep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
inline void pdl_config(cudaLaunchConfig_t* cfg, cudaLaunchAttribute* attr, dim3 grid, dim3 block,
                       size_t smem, cudaStream_t st) {
  cfg->gridDim = grid;
  cfg->blockDim = block;
  cfg->dynamicSmemBytes = smem;
  cfg->stream = st;
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg->attrs = attr;
  cfg->numAttrs = 1;
}

// ---------------------------------------------------------------- launchers
constexpr int kGb300Sms = 152;   // streaming multiprocessors of one GB300

// Split partials of the verification attention.  part_o holds each partial
// row normalised (O / l) in fp16, column-octet major: the 16 bytes holding
// columns [8*c8, 8*c8+8) of packed row R of split s of KV head kv sit at
// uint4 index ((kv * n_split + s) * (D/8) + c8) * M + R, so consecutive rows
// are consecutive uint4s (a warp holding 32 rows stores 512 contiguous
// bytes).  part_ml holds the fp32 (m, l) pairs at (kv * n_split + s) * M + R.
__host__ __device__ __forceinline__ size_t part_o8_index(int kv, int s, int n_split, int c8,
                                                         int D, int M, int R) {
  return (((size_t)kv * n_split + s) * (D / 8) + c8) * M + R;
}

// The cache [0, L) (plus the T tree rows, in the last split) is cut into
// n_split key splits, the same cut for every row group of a KV head, so that
// every key tile is read by all row groups at about the same time and leaves
// HBM once.
struct VerifyPlan {
  int M;               // packed query rows per KV head (T * G)
  int n_pt;            // row groups of up to 256 rows (pair-tile CTAs, one per split)
  int n_two;           // a last group of <= 128 rows (two-stream CTAs, one per two splits)
  int n_split;         // KV splits per head
  int64_t keys_per_split;   // a multiple of 128
  size_t part_o_bytes, part_ml_bytes, ws_bytes;
};
VerifyPlan verify_plan(int T, int Hq, int Hkv, int d, int64_t L);
int tc_splits(int Hkv, int n_rg, int64_t L, int nsm);
int verify_splits(int Hkv, int n_pt, int n_two, int64_t L, int nsm);
int launch_verify_tc(const void* q, const void* k, const void* v, int64_t L, int64_t L_cap,
                     const int32_t* parents, int T, int Hq, int Hkv, int d, int n_imp,
                     int64_t keys_per_split, int n_split, int n_pt, int n_two, bool v_fp16,
                     uint4* part_o, float* part_ml, float* imp, int32_t* status,
                     cudaStream_t st);

// Limit (SM clock cycles) of one bounded device wait in the kernels with
// cross-warp waits; ts_set_wait_limit sets it for later launches.
constexpr long long kDefaultWaitCycles = 1ll << 31;
long long wait_limit_cycles();
int launch_verify(const void* q, const void* k, const void* v, int64_t L, int64_t L_cap,
                  const int32_t* parents, int T, int Hq, int Hkv, int d, int n_imp,
                  bool v_fp16, float* o, float* lse, float* imp, void* ws, int32_t* status,
                  cudaStream_t st);

struct SelectPlan {
  int64_t chunk;       // positions per gather CTA
  int64_t n_chunks;
  size_t ws_bytes;
};
SelectPlan select_plan(int Hkv, int64_t L, int n_layers);
int launch_select_gather(const float* imp, const void* k, const void* v, int64_t L,
                         int64_t L_cap, int Hkv, int d, int B, int S, int R, int32_t* idx,
                         void* kd, void* vd, int64_t N, void* ws, int32_t* status,
                         cudaStream_t st);

int launch_select_gather_batched(int n_layers, const float* const* imp, const void* const* k,
                                 const void* const* v, int64_t L, int64_t L_cap, int Hkv, int d,
                                 int B, int S, int R, int32_t* const* idx, void* const* kd,
                                 void* const* vd, int64_t N, void* ws, int32_t* status,
                                 cudaStream_t st);

// Fixed scratch of the allocation-free selection entry point.
constexpr size_t kNoAllocScratchBytes = size_t(10) << 20;
int select_scratch(void** out);   // device address of that scratch (current device)

size_t sample_ws_bytes(int T, int V);
int launch_sample_accept(const float* logits, const int32_t* tree_tokens, const int32_t* parents,
                         int T, const int32_t* prior, int n_prior, int W, int V, float penalty,
                         float temperature, float top_p, float min_p, int eta_mode, float eta_eps,
                         float eta_alpha, const float* uniforms, int32_t* sampled, int32_t* path,
                         int32_t* n_path, int32_t* bonus, void* ws, const float* q_draft,
                         const float* u_draw, int32_t* status, cudaStream_t st);
size_t ngram_table_bytes(int V, int cap);
int launch_ngram_insert(int32_t* table, int V, int cap, const int32_t* tokens, int n_tokens,
                        int start, int32_t* status, cudaStream_t st);
int launch_ngram_tree(const int32_t* table, int V, int cap, const int32_t* root_token,
                      const int32_t* head_topk, int n_heads, int head_k, int k,
                      const uint32_t* rand_keys, int T_max, int32_t* parents, int32_t* tokens,
                      int32_t* n_nodes, int32_t* status, cudaStream_t st);
int launch_kv_commit(void* k, void* v, int64_t L, int64_t L_cap, int Hkv, int d, int T,
                     const int32_t* path, const int32_t* n_path, int32_t* status,
                     cudaStream_t st);

}  // namespace ts
