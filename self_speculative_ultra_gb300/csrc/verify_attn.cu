// Tree verification attention with fused attention-importance (split-KV
// flash-decode on CUDA cores) and the cross-split merge.
//
// "TokenSwift: Lossless Acceleration of Ultra Long Sequence Generation":
// §3.1 Overview (verification with the full KV cache), §E Tree-Based
// Attention (a tree token attends only to its predecessors), §3.3 Dynamic KV
// Cache Management (importance = query-key dot products aggregated over the
// GQA group).
//
// Work decomposition: for KV head kv the M = T*G query rows of its group are
// packed (row r = node i*G + group member g), the committed cache [0, L) is
// cut into n_split key ranges, and the last range also takes the T tree rows
// under the ancestor mask.  Each CTA owns (row block, split, kv) and writes
// an unnormalised partial (acc, m, l) in the log2 domain; the merge kernel
// combines the splits.  Importance is linear in the queries, so
//   imp[kv,j] = (sum of the group's last n_imp queries) . k_j / sqrt(d)
// is computed once per key by the row-block-0 CTAs from the K tile they
// already hold.
#include <cstdlib>
#include <cstring>

#include "ts_common.cuh"

namespace ts {

namespace {

constexpr int kThreads = 256;
constexpr int kRows = 32;   // query rows per CTA: 8 warps x 4 rows
constexpr int kKeys = 64;   // keys per shared-memory tile
constexpr float kLog2e = 1.4426950408889634f;

template <int D>
struct SimpleSmem {
  float q[kRows][D];
  float k[kKeys][D + 1];
  float v[kKeys][D];
  float qsum[D];
  unsigned long long anc[64];
};

template <int D>
__global__ void __launch_bounds__(kThreads)
verify_split_simple(const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ k,
                    const __nv_bfloat16* __restrict__ v, int64_t L, int64_t L_cap,
                    const int32_t* __restrict__ parents, int T, int Hq, int Hkv, int n_imp,
                    int64_t keys_per_split, int n_split, float* __restrict__ part_o,
                    float* __restrict__ part_ml, float* __restrict__ imp, int32_t* status) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  SimpleSmem<D>& sm = *reinterpret_cast<SimpleSmem<D>*>(smem_raw);
  const int rb = blockIdx.x, split = blockIdx.y, kv = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = Hq / Hkv, M = T * G;
  constexpr int DL = D / 32;   // output dims per lane

  if (tid == 0) tree_masks(parents, T, sm.anc, (rb == 0 && split == 0 && kv == 0) ? status : nullptr);
  for (int e = tid; e < kRows * D; e += kThreads) {
    int r = e / D, c = e % D, row = rb * kRows + r;
    float val = 0.f;
    if (row < M) {
      int i = row / G, h = kv * G + row % G;
      val = bf2f(q[((size_t)i * Hq + h) * D + c]);
    }
    sm.q[r][c] = val;
  }
  const bool do_imp = (rb == 0) && imp != nullptr;
  if (do_imp) {
    for (int c = tid; c < D; c += kThreads) {
      float s = 0.f;
      for (int i = T - n_imp; i < T; ++i)
        for (int g = 0; g < G; ++g) s += bf2f(q[((size_t)i * Hq + kv * G + g) * D + c]);
      sm.qsum[c] = s;
    }
  }
  __syncthreads();

  const float scale = 1.0f / sqrtf((float)D);
  const float sl2 = scale * kLog2e;
  const int64_t j0 = (int64_t)split * keys_per_split;
  const int64_t j1 = min(L, j0 + keys_per_split);
  const int64_t jend = (split == n_split - 1) ? L + T : j1;

  float m[4], l[4], acc[4][DL];
#pragma unroll
  for (int rr = 0; rr < 4; ++rr) {
    m[rr] = -INFINITY;
    l[rr] = 0.f;
#pragma unroll
    for (int c = 0; c < DL; ++c) acc[rr][c] = 0.f;
  }

  const __nv_bfloat16* kh = k + (size_t)kv * L_cap * D;
  const __nv_bfloat16* vh = v + (size_t)kv * L_cap * D;
  for (int64_t t0 = j0; t0 < jend; t0 += kKeys) {
    __syncthreads();
    for (int e = tid; e < kKeys * (D / 8); e += kThreads) {
      int key = e / (D / 8), c8 = (e % (D / 8)) * 8;
      int64_t j = t0 + key;
      float fk[8], fv[8];
      if (j < jend) {
        uint4 uk = *reinterpret_cast<const uint4*>(kh + (size_t)j * D + c8);
        uint4 uv = *reinterpret_cast<const uint4*>(vh + (size_t)j * D + c8);
        unpack_bf16x8(uk, fk);
        unpack_bf16x8(uv, fv);
      } else {
#pragma unroll
        for (int x = 0; x < 8; ++x) fk[x] = fv[x] = 0.f;
      }
#pragma unroll
      for (int x = 0; x < 8; ++x) {
        sm.k[key][c8 + x] = fk[x];
        sm.v[key][c8 + x] = fv[x];
      }
    }
    __syncthreads();

    if (do_imp) {
      for (int key = warp; key < kKeys; key += kThreads / 32) {
        int64_t j = t0 + key;
        float s = 0.f;
#pragma unroll
        for (int c = lane; c < D; c += 32) s += sm.qsum[c] * sm.k[key][c];
        s = warp_sum(s);
        if (lane == 0 && j < j1) imp[(size_t)kv * L + j] = s * scale;
      }
    }

#pragma unroll
    for (int rr = 0; rr < 4; ++rr) {
      const int r = warp * 4 + rr, row = rb * kRows + r;
      if (row >= M) continue;
      const int i = row / G;
      float s[2];
#pragma unroll
      for (int h2 = 0; h2 < 2; ++h2) {
        int key = lane + 32 * h2;
        int64_t j = t0 + key;
        bool ok = j < jend && (j < L || ((sm.anc[i] >> (j - L)) & 1ull));
        float dot = 0.f;
        if (ok) {
#pragma unroll 8
          for (int c = 0; c < D; ++c) dot += sm.q[r][c] * sm.k[key][c];
        }
        s[h2] = ok ? dot * sl2 : -INFINITY;
      }
      float tmax = warp_max(fmaxf(s[0], s[1]));
      float mnew = fmaxf(m[rr], tmax);
      if (mnew == -INFINITY) continue;
      float alpha = exp2f(m[rr] - mnew);
      float p0 = exp2f(s[0] - mnew), p1 = exp2f(s[1] - mnew);
      l[rr] = l[rr] * alpha + warp_sum(p0 + p1);
#pragma unroll
      for (int c = 0; c < DL; ++c) acc[rr][c] *= alpha;
      for (int key = 0; key < kKeys; ++key) {
        float pk = __shfl_sync(0xffffffffu, key < 32 ? p0 : p1, key & 31);
#pragma unroll
        for (int c = 0; c < DL; ++c) acc[rr][c] += pk * sm.v[key][lane + 32 * c];
      }
      m[rr] = mnew;
    }
  }

#pragma unroll
  for (int rr = 0; rr < 4; ++rr) {
    const int row = rb * kRows + warp * 4 + rr;
    if (row >= M) continue;
    size_t base = ((size_t)kv * n_split + split) * M + row;
#pragma unroll
    for (int c = 0; c < DL; ++c) {
      const int col = lane + 32 * c;
      part_o[part_o4_index(kv, split, n_split, col >> 2, D, M, row) * 4 + (col & 3)] = acc[rr][c];
    }
    if (lane == 0) {
      part_ml[base * 2] = m[rr];
      part_ml[base * 2 + 1] = l[rr];
    }
  }
}

// One CTA per (KV head, block of 8 packed rows); thread (c4, r) owns
// columns [4*c4, 4*c4+4) of row r and folds the splits in with the
// online-softmax recurrence (running maximum, rescaled sum and accumulator),
// the loads of kMergeBatch splits in flight at once.  Launched as a
// programmatic dependent of the verification kernel: it waits for that grid's
// partials before its first load.
constexpr int kMaxSplits = 1024;
constexpr int kMergeRows = 8;
constexpr int kMergeBatch = 8;
__global__ void __launch_bounds__(256, 2)
verify_merge(const float* __restrict__ part_o, const float* __restrict__ part_ml, int T, int Hq,
             int Hkv, int D, int n_split, float* __restrict__ o, float* __restrict__ lse) {
  griddep_wait();
  const int kv = blockIdx.y;
  const int G = Hq / Hkv, M = T * G;
  const int tid = threadIdx.x, r = tid % kMergeRows, c4 = tid / kMergeRows;
  const int R = blockIdx.x * kMergeRows + r;
  if (R >= M) return;
  const float4* src =
      reinterpret_cast<const float4*>(part_o) + part_o4_index(kv, 0, n_split, c4, D, M, R);
  const size_t step = (size_t)(D / 4) * M;              // float4s between splits
  const float2* ml = reinterpret_cast<const float2*>(part_ml) + (size_t)kv * n_split * M + R;
  float mrun = -INFINITY, lrun = 0.f;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int s0 = 0; s0 < n_split; s0 += kMergeBatch) {
    float4 ov[kMergeBatch];
    float2 mv[kMergeBatch];
#pragma unroll
    for (int k = 0; k < kMergeBatch; ++k) {
      const int s = s0 + k;
      if (s < n_split) {
        ov[k] = src[(size_t)s * step];
        mv[k] = ml[(size_t)s * M];
      } else {
        ov[k] = make_float4(0.f, 0.f, 0.f, 0.f);
        mv[k] = make_float2(-INFINITY, 0.f);
      }
    }
    float mb = mrun;
#pragma unroll
    for (int k = 0; k < kMergeBatch; ++k) mb = fmaxf(mb, mv[k].x);
    if (mb == -INFINITY) continue;                      // no key seen yet
    const float fr = exp2f(mrun - mb);                  // 0 while mrun = -inf
    lrun *= fr;
    acc = make_float4(acc.x * fr, acc.y * fr, acc.z * fr, acc.w * fr);
#pragma unroll
    for (int k = 0; k < kMergeBatch; ++k) {
      const float w = exp2f(mv[k].x - mb);              // 0 for an empty split
      lrun += w * mv[k].y;
      acc.x += w * ov[k].x;
      acc.y += w * ov[k].y;
      acc.z += w * ov[k].z;
      acc.w += w * ov[k].w;
    }
    mrun = mb;
  }
  const float inv = 1.f / lrun;
  const int i = R / G, h = kv * G + R % G;
  reinterpret_cast<float4*>(o + ((size_t)i * Hq + h) * D)[c4] =
      make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
  if (lse && c4 == 0) lse[(size_t)i * Hq + h] = (mrun + log2f(lrun)) * 0.6931471805599453f;
}

}  // namespace

static bool use_simple_path() {
  static int v = -1;
  if (v < 0) {
    const char* e = getenv("TS_VERIFY_IMPL");
    v = (e && strcmp(e, "simple") == 0) ? 1 : 0;
  }
  return v == 1;
}

VerifyPlan verify_plan(int T, int Hq, int Hkv, int d, int64_t L) {
  VerifyPlan p{};
  p.M = T * (Hq / Hkv);
  if (!use_simple_path()) {
    // tcgen05 path: row groups of up to 256 packed query rows
    p.tc = true;
    p.pair = verify_pair_eligible(T, Hq, Hkv, d);
    p.n_rowblk = (p.M + 255) / 256;
    p.rows_per_cta = 256;
    // a CTA pair per (split, head) when the pair kernel applies
    int n = tc_splits(Hkv, p.pair ? 2 : p.n_rowblk, L, kGb300Sms);
    int64_t kps = (L + n - 1) / n;
    kps = (kps + 127) / 128 * 128;
    if (kps < 128) kps = 128;
    p.keys_per_split = kps;
    p.n_split = (int)((L + kps - 1) / kps);
  } else {
    p.tc = false;
    p.rows_per_cta = kRows;
    p.n_rowblk = (p.M + kRows - 1) / kRows;
    // aim for ~4 waves of the SMs, keys_per_split a multiple of the key tile
    int64_t target_ctas = 4 * kGb300Sms;
    int64_t per_head = (target_ctas + (int64_t)Hkv * p.n_rowblk - 1) / ((int64_t)Hkv * p.n_rowblk);
    if (per_head < 1) per_head = 1;
    int64_t kps = (L + per_head - 1) / per_head;
    kps = (kps + kKeys - 1) / kKeys * kKeys;
    if (kps < kKeys) kps = kKeys;
    p.keys_per_split = kps;
    p.n_split = (int)((L + kps - 1) / kps);
  }
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
  int rc;
  if (p.pair) {
    rc = launch_verify_pair(q, k, v, L, L_cap, parents, T, Hq, Hkv, n_imp, p.keys_per_split,
                            p.n_split, part_o, part_ml, imp, status, st);
  } else if (p.tc) {
    rc = launch_verify_tc(q, k, v, L, L_cap, parents, T, Hq, Hkv, d, n_imp, p.keys_per_split,
                          p.n_split, p.n_rowblk, part_o, part_ml, imp, status, st);
  } else {
    dim3 grid(p.n_rowblk, p.n_split, Hkv);
    auto qb = static_cast<const __nv_bfloat16*>(q);
    auto kb = static_cast<const __nv_bfloat16*>(k);
    auto vb = static_cast<const __nv_bfloat16*>(v);
    if (d == 128) {
      size_t sm = sizeof(SimpleSmem<128>);
      cudaFuncSetAttribute(verify_split_simple<128>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
      verify_split_simple<128><<<grid, kThreads, sm, st>>>(qb, kb, vb, L, L_cap, parents, T, Hq, Hkv,
                                                           n_imp, p.keys_per_split, p.n_split, part_o,
                                                           part_ml, imp, status);
    } else {
      size_t sm = sizeof(SimpleSmem<64>);
      cudaFuncSetAttribute(verify_split_simple<64>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
      verify_split_simple<64><<<grid, kThreads, sm, st>>>(qb, kb, vb, L, L_cap, parents, T, Hq, Hkv,
                                                          n_imp, p.keys_per_split, p.n_split, part_o,
                                                          part_ml, imp, status);
    }
    rc = launch_status("verify_split_simple");
  }
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
