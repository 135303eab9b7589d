// Incremental partial-cache refresh (select_gather.cu): workspace size and
// launchers.  The compact cache keeps a fixed row stride N_cap; slots
// [0, N_prev) hold the previous step's rows, [0, N_new) the new ones.
#pragma once

#include "ts_common.cuh"

namespace ts {

size_t refresh_ws_bytes(int n_heads_total, int64_t L, int64_t N_cap);
int launch_refresh_incremental(int n_layers, const float* imp1, const float* const* imp,
                               const void* k1, const void* const* k, const void* v1,
                               const void* const* v, int64_t L, int64_t L_cap, int Hkv, int d,
                               int B, int S, int R, int64_t N_prev, int64_t N_new, int64_t N_cap,
                               int32_t* idx1, int32_t* const* idx, void* kd1, void* const* kd,
                               void* vd1, void* const* vd, int32_t* n_written, void* ws,
                               int32_t* status, cudaStream_t st);

}  // namespace ts
