// Cross-split merge of the tree verification attention and the host-side
// plan of the tcgen05 split kernel (verify_tc.cu).
//
// "TokenSwift: Lossless Acceleration of Ultra Long Sequence Generation":
// §3.1 Overview (verification with the full KV cache), §E Tree-Based
// Attention (a tree token attends only to its predecessors).
//
// Work decomposition: for KV head kv the M = T*G query rows of its group are
// packed (row r = node r / G, head kv*G + r % G) and the committed cache
// [0, L) is cut into n_split key ranges, the same cut for every row group;
// the last range also takes the T tree rows under the ancestor mask.  Every
// (row, split) gets one partial (O / l in fp16, m and l in the log2 domain);
// the merge kernel below combines the splits of every row.
#include "ts_common.cuh"

namespace ts {

namespace {

// Thread (row R, 8-column octet c8, split group j) folds splits j, j + NG,
// j + 2*NG, ... of its row with the online-softmax recurrence, kPer partial
// loads in flight at once (one round trip for up to NG * kPer splits); the
// NG states of a (row, octet) sit in lanes 32/NG apart of one warp and are
// combined by shuffles.  A warp covers 32/NG consecutive rows x NG split
// groups of one octet, so each group's loads are contiguous.  A partial is
// stored normalised (O_s / l_s, fp16), so split s enters with weight
// 2^(m_s - m) * l_s.  NG (1, 2 or 4) is the largest that keeps the grid
// within one wave of the SMs: a second wave of merge CTAs holds SMs the
// next verification grid waits for.  Launched as a programmatic dependent
// of the verification kernel: it waits for that grid's partials before its
// first load, then lets the next kernel of the stream start its set-up as
// this grid's CTAs retire.
constexpr int kMaxSplits = 1024;
constexpr int kPer = 5;              // loads in flight per thread
constexpr int kMergeThreads = 256;   // 8 warps: 8 column octets per CTA
constexpr int kMergeCtasPerSm = 4;   // at <= 64 registers
template <int NG>
__global__ void __launch_bounds__(kMergeThreads, kMergeCtasPerSm)
verify_merge(const uint4* __restrict__ part_o, const float* __restrict__ part_ml, int T, int Hq,
             int Hkv, int D, int n_split, float* __restrict__ o, float* __restrict__ lse) {
  constexpr int kRows = 32 / NG;      // rows per warp
  griddep_wait();
  griddep_launch_dependents();
  const int kv = blockIdx.z;
  const int G = Hq / Hkv, M = T * G;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int r = lane % kRows, j = lane / kRows;                  // row in block, split group
  const int c8 = blockIdx.y * (kMergeThreads / 32) + warp;       // column octet
  const int R = blockIdx.x * kRows + r;
  const bool live = R < M && c8 < D / 8;
  const int Rc = live ? R : 0, cc = live ? c8 : 0;
  // a thread with no row folds no split
  const int n_fold = live ? n_split : 0;
  const uint4* src = part_o + part_o8_index(kv, 0, n_split, cc, D, M, Rc);
  const size_t step = (size_t)(D / 8) * M;              // uint4s between splits
  const float2* ml = reinterpret_cast<const float2*>(part_ml) + (size_t)kv * n_split * M + Rc;
  float mrun = -INFINITY, lrun = 0.f;
  float acc[8];
#pragma unroll
  for (int x = 0; x < 8; ++x) acc[x] = 0.f;
  auto unpack = [](uint32_t w, float& a, float& b) {
    const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w));
    a = f.x;
    b = f.y;
  };
  for (int s0 = j; s0 < n_fold; s0 += NG * kPer) {
    uint4 ov[kPer];
    float2 mv[kPer];
#pragma unroll
    for (int k = 0; k < kPer; ++k) {
      const int s = s0 + k * NG;
      if (s < n_fold) {
        ov[k] = __ldg(&src[(size_t)s * step]);
        mv[k] = __ldg(&ml[(size_t)s * M]);
      } else {
        ov[k] = make_uint4(0u, 0u, 0u, 0u);
        mv[k] = make_float2(-INFINITY, 0.f);
      }
    }
    float mb = mrun;
#pragma unroll
    for (int k = 0; k < kPer; ++k) mb = fmaxf(mb, mv[k].x);
    if (mb == -INFINITY) continue;                      // no key seen yet
    const float fr = exp2f(mrun - mb);                  // 0 while mrun = -inf
    lrun *= fr;
#pragma unroll
    for (int x = 0; x < 8; ++x) acc[x] *= fr;
#pragma unroll
    for (int k = 0; k < kPer; ++k) {
      const float w = exp2f(mv[k].x - mb) * mv[k].y;    // 0 for an empty split
      lrun += w;
      const uint32_t wd[4] = {ov[k].x, ov[k].y, ov[k].z, ov[k].w};
#pragma unroll
      for (int x = 0; x < 4; ++x) {
        float a, b;
        unpack(wd[x], a, b);
        acc[2 * x] += w * a;
        acc[2 * x + 1] += w * b;
      }
    }
    mrun = mb;
  }
  // combine the split groups (lanes r, r + kRows, ...)
#pragma unroll
  for (int off = kRows; off < 32; off <<= 1) {
    const float m2 = __shfl_xor_sync(0xffffffffu, mrun, off);
    const float l2 = __shfl_xor_sync(0xffffffffu, lrun, off);
    const float mn = fmaxf(mrun, m2);
    const float f1 = mrun == -INFINITY ? 0.f : exp2f(mrun - mn);
    const float f2 = m2 == -INFINITY ? 0.f : exp2f(m2 - mn);
#pragma unroll
    for (int x = 0; x < 8; ++x) {
      const float a2 = __shfl_xor_sync(0xffffffffu, acc[x], off);
      acc[x] = acc[x] * f1 + a2 * f2;
    }
    lrun = lrun * f1 + l2 * f2;
    mrun = mn;
  }
  if (!live || j != 0) return;
  const float inv = 1.f / lrun;
  const int i = R / G, h = kv * G + R % G;
  float4* orow = reinterpret_cast<float4*>(o + ((size_t)i * Hq + h) * D) + 2 * c8;
  orow[0] = make_float4(acc[0] * inv, acc[1] * inv, acc[2] * inv, acc[3] * inv);
  orow[1] = make_float4(acc[4] * inv, acc[5] * inv, acc[6] * inv, acc[7] * inv);
  if (lse && c8 == 0) lse[(size_t)i * Hq + h] = (mrun + log2f(lrun)) * 0.6931471805599453f;
}

}  // namespace

// Keys per split for n splits of [0, L): whole 128-key tiles, at most
// kMaxSplits splits (bounds the partials of very long caches).
static void cut(int64_t L, int n, int& n_out, int64_t& kps) {
  kps = (L + n - 1) / n;
  kps = (kps + 127) / 128 * 128;
  if (kps < 128) kps = 128;
  n_out = (int)((L + kps - 1) / kps);
  if (n_out < 1) n_out = 1;
  if (n_out > kMaxSplits) {
    kps = ((L + kMaxSplits - 1) / kMaxSplits + 127) / 128 * 128;
    n_out = (int)((L + kps - 1) / kps);
  }
}

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
  cut(L, verify_splits(Hkv, p.n_pt, p.n_two, L, kGb300Sms), p.n_split, p.keys_per_split);
  p.part_o_bytes = align_up((size_t)Hkv * p.n_split * p.M * d * sizeof(__half), 256);
  p.part_ml_bytes = align_up((size_t)Hkv * p.n_split * p.M * 2 * sizeof(float), 256);
  p.ws_bytes = p.part_o_bytes + p.part_ml_bytes;
  return p;
}

int launch_verify(const void* q, const void* k, const void* v, int64_t L, int64_t L_cap,
                  const int32_t* parents, int T, int Hq, int Hkv, int d, int n_imp, bool v_fp16,
                  float* o, float* lse, float* imp, void* ws, int32_t* status, cudaStream_t st) {
  VerifyPlan p = verify_plan(T, Hq, Hkv, d, L);
  uint4* part_o = static_cast<uint4*>(ws);
  float* part_ml = reinterpret_cast<float*>(static_cast<char*>(ws) + p.part_o_bytes);
  int rc = launch_verify_tc(q, k, v, L, L_cap, parents, T, Hq, Hkv, d, n_imp, p.keys_per_split,
                            p.n_split, p.n_pt, p.n_two, v_fp16, part_o, part_ml, imp, status, st);
  if (rc) return rc;
  const int ny = (d / 8 + 7) / 8;
  auto ctas = [&](int ng) { return (p.M + 32 / ng - 1) / (32 / ng) * ny * Hkv; };
  const int wave = kMergeCtasPerSm * kGb300Sms;
  const int ng = ctas(4) <= wave ? 4 : (ctas(2) <= wave ? 2 : 1);
  dim3 mgrid((p.M + 32 / ng - 1) / (32 / ng), ny, Hkv);
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  pdl_config(&cfg, attr, mgrid, dim3(kMergeThreads), 0, st);
  auto po = static_cast<const uint4*>(part_o);
  auto pm = static_cast<const float*>(part_ml);
  if (ng == 4)
    cudaLaunchKernelEx(&cfg, verify_merge<4>, po, pm, T, Hq, Hkv, d, p.n_split, o, lse);
  else if (ng == 2)
    cudaLaunchKernelEx(&cfg, verify_merge<2>, po, pm, T, Hq, Hkv, d, p.n_split, o, lse);
  else
    cudaLaunchKernelEx(&cfg, verify_merge<1>, po, pm, T, Hq, Hkv, d, p.n_split, o, lse);
  return launch_status("verify_merge");
}

}  // namespace ts
