// Cross-split merge of the tree verification attention and the host-side
// plan of the tcgen05 split kernel (verify_tc.cu).
//
// "TokenSwift: Lossless Acceleration of Ultra Long Sequence Generation":
// §3.1 Overview (verification with the full KV cache), §E Tree-Based
// Attention (a tree token attends only to its predecessors).
//
// Work decomposition: for KV head kv the M = T*G query rows of its group are
// packed (row r = node r / G, head kv*G + r % G) and the committed cache
// [0, L) is cut into n_split key ranges; the last range also takes the T
// tree rows under the ancestor mask.  Every (row, split) gets one
// unnormalised partial (O, m, l) in the log2 domain; the merge kernel below
// combines the splits of every row.
#include "ts_common.cuh"

namespace ts {

namespace {

// One CTA per (KV head, block of 8 packed rows); thread (c4, r) owns
// columns [4*c4, 4*c4+4) of row r.  The row's (m, l) pairs give the maximum
// over the splits first, so every split's weight 2^(m_s - max) is known
// before its partial is read and the partial loads of all splits are
// independent (unrolled, several in flight).  Launched as a programmatic
// dependent of the verification kernel: it waits for that grid's partials
// before its first load, then lets the next kernel of the stream start its
// set-up as this grid's CTAs retire.
constexpr int kMaxSplits = 1024;
constexpr int kMergeRows = 8;
__global__ void __launch_bounds__(256)
verify_merge(const float* __restrict__ part_o, const float* __restrict__ part_ml, int T, int Hq,
             int Hkv, int D, int n_split, float* __restrict__ o, float* __restrict__ lse) {
  griddep_wait();
  griddep_launch_dependents();
  const int kv = blockIdx.y;
  const int G = Hq / Hkv, M = T * G;
  const int tid = threadIdx.x, r = tid % kMergeRows, c4 = tid / kMergeRows;
  const int R = blockIdx.x * kMergeRows + r;
  if (R >= M) return;
  const float4* src =
      reinterpret_cast<const float4*>(part_o) + part_o4_index(kv, 0, n_split, c4, D, M, R);
  const size_t step = (size_t)(D / 4) * M;              // float4s between splits
  const float2* ml = reinterpret_cast<const float2*>(part_ml) + (size_t)kv * n_split * M + R;
  float mmax = -INFINITY;
#pragma unroll 8
  for (int s = 0; s < n_split; ++s) mmax = fmaxf(mmax, __ldg(&ml[(size_t)s * M]).x);
  // every row sees at least its own tree node, so mmax is finite; an empty
  // split has m = -inf and weight 0
  float lrun = 0.f;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 8
  for (int s = 0; s < n_split; ++s) {
    const float2 mv = __ldg(&ml[(size_t)s * M]);
    const float4 ov = __ldg(&src[(size_t)s * step]);
    const float w = exp2f(mv.x - mmax);
    lrun += w * mv.y;
    acc.x += w * ov.x;
    acc.y += w * ov.y;
    acc.z += w * ov.z;
    acc.w += w * ov.w;
  }
  const float inv = 1.f / lrun;
  const int i = R / G, h = kv * G + R % G;
  reinterpret_cast<float4*>(o + ((size_t)i * Hq + h) * D)[c4] =
      make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
  if (lse && c4 == 0) lse[(size_t)i * Hq + h] = (mmax + log2f(lrun)) * 0.6931471805599453f;
}

}  // namespace

VerifyPlan verify_plan(int T, int Hq, int Hkv, int d, int64_t L) {
  VerifyPlan p{};
  p.M = T * (Hq / Hkv);
  // rows are taken 256 at a time while more than 128 remain; a remainder of
  // at most 128 rows is served by two-stream CTAs
  int rows = p.M;
  p.n_pt = 0;
  while (rows > 128) {
    ++p.n_pt;
    rows -= 256;
  }
  p.n_two = rows > 0 ? 1 : 0;
  int n = verify_splits(Hkv, p.n_pt, p.n_two, L, kGb300Sms);
  int64_t kps = (L + n - 1) / n;
  kps = (kps + 127) / 128 * 128;
  if (kps < 128) kps = 128;
  p.keys_per_split = kps;
  p.n_split = (int)((L + kps - 1) / kps);
  if (p.n_split < 1) p.n_split = 1;
  if (p.n_split > kMaxSplits) {   // bounds the split partials of very long caches
    p.keys_per_split = ((L + kMaxSplits - 1) / kMaxSplits + 127) / 128 * 128;
    p.n_split = (int)((L + p.keys_per_split - 1) / p.keys_per_split);
  }
  p.part_o_bytes = align_up((size_t)Hkv * p.n_split * p.M * d * sizeof(float), 256);
  p.part_ml_bytes = align_up((size_t)Hkv * p.n_split * p.M * 2 * sizeof(float), 256);
  p.ws_bytes = p.part_o_bytes + p.part_ml_bytes;
  return p;
}

int launch_verify(const void* q, const void* k, const void* v, int64_t L, int64_t L_cap,
                  const int32_t* parents, int T, int Hq, int Hkv, int d, int n_imp, float* o,
                  float* lse, float* imp, void* ws, int32_t* status, cudaStream_t st) {
  VerifyPlan p = verify_plan(T, Hq, Hkv, d, L);
  float* part_o = static_cast<float*>(ws);
  float* part_ml = reinterpret_cast<float*>(static_cast<char*>(ws) + p.part_o_bytes);
  int rc = launch_verify_tc(q, k, v, L, L_cap, parents, T, Hq, Hkv, d, n_imp, p.keys_per_split,
                            p.n_split, p.n_pt, p.n_two, part_o, part_ml, imp, status, st);
  if (rc) return rc;
  dim3 mgrid((p.M + kMergeRows - 1) / kMergeRows, Hkv);
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  pdl_config(&cfg, attr, mgrid, dim3(kMergeRows * (d / 4)), 0, st);
  cudaLaunchKernelEx(&cfg, verify_merge, static_cast<const float*>(part_o),
                     static_cast<const float*>(part_ml), T, Hq, Hkv, d, p.n_split, o, lse);
  return launch_status("verify_merge");
}

}  // namespace ts
