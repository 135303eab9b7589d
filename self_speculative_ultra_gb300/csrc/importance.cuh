// Softmax-weighted importance pass (importance_softmax.cu): plan and launcher.
#pragma once

#include "ts_common.cuh"

namespace ts {

struct ImpSoftmaxPlan {
  int Rs;                  // staged importance query rows (a multiple of 32)
  int chunk_rows;          // rows per MMA chunk (<= 256); Rs = chunks * chunk_rows
  int n_split;             // key splits per KV head
  int64_t keys_per_split;  // a multiple of 128
  size_t smem;             // dynamic shared memory of one CTA
};

ImpSoftmaxPlan importance_softmax_plan(int T, int Hq, int Hkv, int d, int n_imp, int64_t L);
int launch_importance_softmax(const void* q, const void* k, const float* lse, int64_t L,
                              int64_t L_cap, int T, int Hq, int Hkv, int d, int n_imp, float* imp,
                              int32_t* status, cudaStream_t st);

}  // namespace ts
