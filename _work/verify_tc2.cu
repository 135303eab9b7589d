// Tree verification attention on a CTA pair (tcgen05 .cta_group::2), for a
// KV head whose packed query rows fill exactly two 128-row tiles (M = T*G =
// 256, d = 128: the LLaMA3.1-8B and Qwen2.5-7B decode shapes).
//
// "TokenSwift: Lossless Acceleration of Ultra Long Sequence Generation":
// §3.1 Overview (verification with the full KV cache), §E Tree-Based
// Attention (a tree token attends only to its predecessors), §3.3 Dynamic KV
// Cache Management (importance = query-key dot products, GQA scores
// aggregated per group).
//
// One cluster of two CTAs = (key split, KV head).  CTA r holds query rows
// [128r, 128r+128) and, of every 128-key tile, the K rows of keys
// [64r, 64r+64) and the V columns [64r, 64r+64): the M=256 MMAs issued by the
// even CTA read A by rows and B by columns from the two CTAs' shared memory,
// so each CTA stages half of every K/V tile (one HBM read per tile for the
// pair) and its TMEM holds its own rows of S and O.  With one row tile per
// SM, TMEM has room for two S buffers: Q.K^T of tile j+2 overlaps the
// softmax of tile j+1 and P.V of tile j, which breaks the per-tile chain
// softmax -> P.V -> next Q.K^T of the single-SM kernel.
//
// Warp roles per CTA (16 warps):
//   0        TMA producer: this CTA's K half (4-stage ring) and V half
//            (4-stage ring)
//   1        MMA issuer (even CTA only; both CTAs allocate TMEM here)
//   2,3      importance of this CTA's 64 keys per tile, from shared memory,
//            with the query sum over both CTAs' rows
//   4..7,    softmax, one thread per query row; warpgroup w takes the tiles
//   12..15   j = w (mod 2) into its own O_w (two online-softmax streams per
//            row, merged at the end): max pass and exponent pass over the
//            TMEM row, lazy running max (O_w and l rescaled only when the max
//            grows past 2^8), P = 2^(s*log2e/sqrt(d) - m) written over S in
//            fp16
//   8..11    V conversion bf16 -> fp16 in place (exact for |v| < 65504;
//            larger values saturate and are reported in the status word)
// Hand-offs between the CTAs are remote mbarrier arrivals on the even CTA's
// barriers (K landed, V converted, P written) and multicast MMA commits to
// both CTAs' barriers (S ready, stages free, P.V done, O final).  Every wait
// is bounded; on expiry a CTA records TS_ERR_TIMEOUT and runs to the end,
// where both CTAs meet before TMEM is freed.
#include <cstdlib>

#include "tc_ptx.cuh"
#include "ts_common.cuh"

namespace ts {

namespace {

constexpr int kNk = 128;                 // keys per tile
constexpr int kHalf = 64;                // keys (K) or dims (V) per CTA per tile
constexpr int kD = 128;
constexpr int kSK = 4;                   // K ring depth
constexpr int kSV = 4;                   // V ring depth
constexpr int kThreads = 512;            // 16 warps
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLazy = 8.0f;
constexpr long long kWaitCycles = 1ll << 31;
constexpr uint32_t kNegInf = 0xFF800000u;

struct Aux {
  uint64_t k_full[kSK], k_peer[kSK], k_empty[kSK];
  uint64_t v_full[kSV], v_conv[kSV], v_empty[kSV];
  uint64_t s_full[2], p_ready[2], o_final, drain;
  float ml_odd[128][2];                  // (m, l) of the odd-tile softmax stream, per row
  unsigned long long anc[64];
  int32_t par[64];
  float qpeer[kD];                       // the other CTA's partial query sum
  uint32_t tmem_base;
  volatile int32_t abort_flag;
};

struct Ly {
  static constexpr int kQPanel = 128 * 128;            // 128 rows x 64 bf16
  static constexpr int kQ = 0;                         // 2 panels
  static constexpr int kKPanel = kHalf * 128;          // 64 keys x 64 bf16
  static constexpr int kKStage = 2 * kKPanel;          // 16 KB
  static constexpr int kK = kQ + 2 * kQPanel;
  static constexpr int kVStage = kNk * 128;            // 128 keys x 64 bf16: 16 KB
  static constexpr int kV = kK + kSK * kKStage;
  static constexpr int kQsum = kV + kSV * kVStage;
  static constexpr int kAux = kQsum + kD * 4;
  static constexpr int kBytes = kAux + (int)sizeof(Aux);
  static constexpr int kAlloc = kBytes + 1024;
  static constexpr uint32_t kTmemCols = 512;
  // TMEM columns: O_b (tiles j with j % 2 == b) at 128b, S_b at 256 + 128b
  __host__ __device__ static constexpr uint32_t obase(int b) { return (uint32_t)(128 * b); }
  __host__ __device__ static constexpr uint32_t sbase(int b) { return (uint32_t)(256 + 128 * b); }
};

__device__ __forceinline__ void timeout(Aux* aux, int32_t* status) {
  aux->abort_flag = 1;
  set_status(status, TS_ERR_TIMEOUT);
}

__device__ __forceinline__ float fmax32(const uint32_t (&r)[32]) {
  float a = ptx::max3(__uint_as_float(r[0]), __uint_as_float(r[1]), __uint_as_float(r[2]));
  float b = ptx::max3(__uint_as_float(r[3]), __uint_as_float(r[4]), __uint_as_float(r[5]));
#pragma unroll
  for (int x = 6; x < 30; x += 4) {
    a = ptx::max3(a, __uint_as_float(r[x]), __uint_as_float(r[x + 1]));
    b = ptx::max3(b, __uint_as_float(r[x + 2]), __uint_as_float(r[x + 3]));
  }
  return ptx::max3(a, b, fmaxf(__uint_as_float(r[30]), __uint_as_float(r[31])));
}

__global__ void __launch_bounds__(kThreads, 1)
verify_pair_kernel(const __grid_constant__ CUtensorMap tmap_k, const __grid_constant__ CUtensorMap tmap_v,
                   const __nv_bfloat16* __restrict__ q, const int32_t* __restrict__ parents, int T,
                   int Hq, int Hkv, int n_imp, int64_t L, int64_t L_cap, int64_t keys_per_split,
                   int n_split, float* __restrict__ part_o, float* __restrict__ part_ml,
                   float* __restrict__ imp, int32_t* status) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~uintptr_t(1023));
  uint8_t* sq = sm + Ly::kQ;
  uint8_t* sk = sm + Ly::kK;
  uint8_t* sv = sm + Ly::kV;
  float* qsum = reinterpret_cast<float*>(sm + Ly::kQsum);
  Aux* aux = reinterpret_cast<Aux*>(sm + Ly::kAux);

  const uint32_t rank = ptx::cluster_ctarank();        // 0: issues the MMAs
  const int split = blockIdx.x >> 1, kv = blockIdx.y;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = Hq / Hkv, M = T * G;                   // M == 256
  const int64_t j0 = (int64_t)split * keys_per_split;
  const int64_t j1 = imin64(L, j0 + keys_per_split);
  const bool last = (split == n_split - 1);
  const int64_t jend = last ? L + T : j1;
  const int64_t jlim = last ? L : j1;
  const int n_tiles = (int)((jend - j0 + kNk - 1) / kNk);
  const bool do_imp = imp != nullptr;
  const float scale = 1.0f / sqrtf((float)kD);
  const float sl2 = scale * kLog2e;
  constexpr int C16 = kD / 8;

  griddep_wait();
  // ---------------------------------------------------------------- set-up
  if (tid == 0) {
    for (int s = 0; s < kSK; ++s) {
      ptx::mbar_init(&aux->k_full[s], 1);
      ptx::mbar_init(&aux->k_peer[s], 1);        // the odd CTA's half landed
      ptx::mbar_init(&aux->k_empty[s], 1 + 2);   // MMA commit + two importance warps
    }
    for (int s = 0; s < kSV; ++s) {
      ptx::mbar_init(&aux->v_full[s], 1);
      ptx::mbar_init(&aux->v_conv[s], 2 * 4);    // four conversion warps in each CTA
      ptx::mbar_init(&aux->v_empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      ptx::mbar_init(&aux->s_full[b], 1);
      ptx::mbar_init(&aux->p_ready[b], 2 * 4);   // four softmax warps in each CTA
    }
    ptx::mbar_init(&aux->o_final, 1);
    ptx::mbar_init(&aux->drain, 1);
    aux->abort_flag = 0;
    ptx::fence_mbar_init();
    // first K and V halves go out now; they complete on this CTA's barriers
    const uint64_t pol = ptx::l2_evict_first_policy();
    const int row0 = (int)(kv * L_cap + j0);
    for (int jj = 0; jj < min(n_tiles, kSK); ++jj) {
      ptx::mbar_arrive_expect_tx(&aux->k_full[jj], Ly::kKStage);
      for (int p = 0; p < 2; ++p)
        ptx::tma_load_2d(sk + jj * Ly::kKStage + p * Ly::kKPanel, &tmap_k, &aux->k_full[jj], p * 64,
                         row0 + jj * kNk + kHalf * (int)rank, pol);
    }
    for (int jj = 0; jj < min(n_tiles, kSV - 1); ++jj) {
      ptx::mbar_arrive_expect_tx(&aux->v_full[jj], Ly::kVStage);
      ptx::tma_load_2d(sv + jj * Ly::kVStage, &tmap_v, &aux->v_full[jj], kHalf * (int)rank,
                       row0 + jj * kNk, pol);
    }
  }
  if (tid < T) aux->par[tid] = parents[tid];
  if (warp == 1) {
    ptx::tmem_alloc2(&aux->tmem_base, Ly::kTmemCols);
    ptx::tmem_relinquish2();
  }
  // this CTA's 128 query rows -> two 128-byte-swizzled K-major panels
  constexpr int kQAll = 128 * C16, kQPer = (kQAll + kThreads - 1) / kThreads;
  {
    uint4 val[kQPer];
#pragma unroll
    for (int k = 0; k < kQPer; ++k) {
      const int e = tid + k * kThreads;
      const int t = e / C16, c = e % C16;
      const int R = 128 * (int)rank + t;
      val[k] = make_uint4(0, 0, 0, 0);
      if (e < kQAll && R < M) {
        const int i = R / G, h = kv * G + R % G;
        val[k] = __ldg(reinterpret_cast<const uint4*>(q + ((size_t)i * Hq + h) * kD + c * 8));
      }
    }
#pragma unroll
    for (int k = 0; k < kQPer; ++k) {
      const int e = tid + k * kThreads;
      if (e < kQAll) {
        const int t = e / C16, c = e % C16;
        const int p = c >> 3, cc = c & 7;
        *reinterpret_cast<uint4*>(sq + p * Ly::kQPanel + t * 128 + ((cc ^ (t & 7)) << 4)) = val[k];
      }
    }
  }
  __syncthreads();
  // partial query sum over this CTA's importance rows (rows >= (T-n_imp)*G),
  // folded by shuffles and across warps through the last V stage (filled
  // only from tile kSV-1 on), then sent to the other CTA
  float* qpart = reinterpret_cast<float*>(sv + (kSV - 1) * Ly::kVStage);
  if (do_imp) {
    const int cg = tid % C16, slice = tid / C16, nsl = kThreads / C16;
    const int p = cg >> 3, cc = cg & 7;
    uint64_t acc[4] = {0, 0, 0, 0};
    const int rlo = max(0, (T - n_imp) * G - 128 * (int)rank);
    for (int t = rlo + slice; t < 128; t += nsl) {
      const uint4 u =
          *reinterpret_cast<const uint4*>(sq + p * Ly::kQPanel + t * 128 + ((cc ^ (t & 7)) << 4));
      const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
      for (int x = 0; x < 4; ++x)
        acc[x] = ptx::add2(acc[x], ptx::f2(__uint_as_float(w[x] << 16),
                                           __uint_as_float(w[x] & 0xFFFF0000u)));
    }
    float f[8];
#pragma unroll
    for (int x = 0; x < 4; ++x) ptx::f2_split(acc[x], f[2 * x], f[2 * x + 1]);
#pragma unroll
    for (int off = C16; off < 32; off <<= 1)
#pragma unroll
      for (int x = 0; x < 8; ++x) f[x] += __shfl_xor_sync(0xffffffffu, f[x], off);
    if (lane < C16) {
      float4* dst = reinterpret_cast<float4*>(qpart + warp * kD + lane * 8);
      dst[0] = make_float4(f[0], f[1], f[2], f[3]);
      dst[1] = make_float4(f[4], f[5], f[6], f[7]);
    }
  }
  // ancestor-or-self masks: node t walks its parent chain (depth < 64)
  if (tid < T) {
    unsigned long long m = 0ull;
    bool bad = (tid == 0) ? (aux->par[0] != -1) : false;
    int a = tid;
    for (int step = 0; step < 64; ++step) {
      m |= 1ull << a;
      if (a == 0) break;
      const int pa = aux->par[a];
      if (pa < 0 || pa >= a) {
        bad = true;
        break;
      }
      a = pa;
    }
    aux->anc[tid] = m;
    if (bad && split == 0 && kv == 0 && rank == 0) set_status(status, TS_ERR_INVALID_ARG);
  }
  __syncthreads();
  if (do_imp && tid < kD) {
    float sum = 0.f;
#pragma unroll
    for (int w = 0; w < kThreads / 32; ++w) sum += qpart[w * kD + tid];
    qsum[tid] = sum;
    ptx::st_cluster_f32(ptx::mapa(ptx::smem_u32(&aux->qpeer[tid]), rank ^ 1u), sum);
  }
  ptx::fence_proxy_async_smem();
  ptx::tc_fence_before();
  // both CTAs' barriers are initialised and the query-sum halves exchanged
  ptx::cluster_sync();
  ptx::tc_fence_after();
  if (do_imp && tid < kD) qsum[tid] += aux->qpeer[tid];
  __syncthreads();
  const uint32_t tmem = aux->tmem_base;
  griddep_launch_dependents();
  // even CTA's barriers, as shared::cluster addresses
  auto lead = [&](uint64_t* bar) { return ptx::mapa(ptx::smem_u32(bar), 0u); };

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    // K(jj) then V(jj) per tile; the first kSK K halves and kSV-1 V halves
    // went out during the set-up
    if (lane == 0) {
      const uint64_t pol = ptx::l2_evict_first_policy();
      const int row0 = (int)(kv * L_cap + j0);
      for (int jj = 0; jj < n_tiles && !aux->abort_flag; ++jj) {
        if (jj >= kSK) {
          const int s = jj % kSK;
          if (!ptx::mbar_wait_cluster(&aux->k_empty[s], (uint32_t)(jj / kSK - 1) & 1u, kWaitCycles)) {
            timeout(aux, status);
            break;
          }
          ptx::mbar_arrive_expect_tx(&aux->k_full[s], Ly::kKStage);
          for (int p = 0; p < 2; ++p)
            ptx::tma_load_2d(sk + s * Ly::kKStage + p * Ly::kKPanel, &tmap_k, &aux->k_full[s],
                             p * 64, row0 + jj * kNk + kHalf * (int)rank, pol);
        }
        if (jj >= kSV - 1) {
          const int s = jj % kSV;
          if (jj >= kSV &&
              !ptx::mbar_wait_cluster(&aux->v_empty[s], (uint32_t)(jj / kSV - 1) & 1u, kWaitCycles)) {
            timeout(aux, status);
            break;
          }
          ptx::mbar_arrive_expect_tx(&aux->v_full[s], Ly::kVStage);
          ptx::tma_load_2d(sv + s * Ly::kVStage, &tmap_v, &aux->v_full[s], kHalf * (int)rank,
                           row0 + jj * kNk, pol);
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (rank == 0 && lane == 0) {
      constexpr uint32_t idesc_qk = ptx::idesc_bf16_f32(256, kNk, false);
      constexpr uint32_t idesc_pv = ptx::idesc_f16_f32(256, kD, true);
      const uint64_t qd0 = ptx::sdesc_sw128(ptx::smem_u32(sq), 16, 1024);
      const uint64_t kd0 = ptx::sdesc_sw128(ptx::smem_u32(sk), 16, 1024);
      const uint64_t vd0 = ptx::sdesc_sw128(ptx::smem_u32(sv), Ly::kVStage, 1024);
      auto qk = [&](int b, int j) {
        const uint64_t b0 = kd0 + (uint64_t)((j % kSK) * (Ly::kKStage >> 4));
#pragma unroll
        for (int ks = 0; ks < kD / 16; ++ks) {
          const uint32_t oa = (ks >> 2) * (Ly::kQPanel >> 4) + (ks & 3) * 2;
          const uint32_t ob = (ks >> 2) * (Ly::kKPanel >> 4) + (ks & 3) * 2;
          ptx::mma2_ss(tmem + Ly::sbase(b), qd0 + oa, b0 + ob, idesc_qk, ks > 0 ? 1u : 0u);
        }
        ptx::mma_commit2(&aux->s_full[b], 3);
        ptx::mma_commit2(&aux->k_empty[j % kSK], 3);
      };
      // O += P V in fp16: keys [32c, 32c+32) keep their P pairs in S columns
      // [32c, 32c+16); K-step ks reads the 8 columns at 32*(ks/2) + 8*(ks%2)
      auto pv = [&](int b, int j) {
        const uint64_t b0 = vd0 + (uint64_t)((j % kSV) * (Ly::kVStage >> 4));
#pragma unroll
        for (int ks = 0; ks < kNk / 16; ++ks) {
          const uint32_t acol = 32 * (ks >> 1) + 8 * (ks & 1);
          ptx::mma2_ts(tmem + Ly::obase(b), tmem + Ly::sbase(b) + acol, b0 + (uint64_t)(ks * 128),
                       idesc_pv, (j >= 2 || ks > 0) ? 1u : 0u);
        }
        ptx::mma_commit2(&aux->v_empty[j % kSV], 3);
      };
      // K tile j is complete when this CTA's half has landed and the odd CTA
      // has forwarded the landing of its half
      auto k_in = [&](int j) {
        const uint32_t par = (uint32_t)(j / kSK) & 1u;
        return ptx::mbar_wait_cluster(&aux->k_full[j % kSK], par, kWaitCycles) &&
               ptx::mbar_wait_cluster(&aux->k_peer[j % kSK], par, kWaitCycles);
      };
      bool ok = true;
      for (int j = 0; ok && j < min(2, n_tiles); ++j) {
        ok = k_in(j);
        if (ok) {
          ptx::tc_fence_after();
          qk(j, j);
        }
      }
      for (int j = 0; ok && j < n_tiles; ++j) {
        const int b = j & 1;
        ok = ptx::mbar_wait_cluster(&aux->v_conv[j % kSV], (uint32_t)(j / kSV) & 1u, kWaitCycles) &&
             ptx::mbar_wait_cluster(&aux->p_ready[b], (uint32_t)(j >> 1) & 1u, kWaitCycles);
        if (!ok) break;
        ptx::tc_fence_after();
        pv(b, j);
        if (j + 2 < n_tiles) {
          ok = k_in(j + 2);
          if (!ok) break;
          ptx::tc_fence_after();
          qk(b, j + 2);
        }
      }
      if (!ok) timeout(aux, status);
      ptx::mma_commit2(&aux->o_final, 3);
      ptx::mma_commit2(&aux->drain, 1);
      ptx::mbar_wait_cluster(&aux->drain, 0, kWaitCycles);
    } else if (rank == 1 && lane == 0) {
      // forward the landing of this CTA's K halves to the MMA issuer
      const uint32_t peer_bar = lead(&aux->k_peer[0]);
      for (int j = 0; j < n_tiles; ++j) {
        if (aux->abort_flag ||
            !ptx::mbar_wait_cluster(&aux->k_full[j % kSK], (uint32_t)(j / kSK) & 1u, kWaitCycles)) {
          timeout(aux, status);
          break;
        }
        // async-proxy (TMA) data, complete once k_full's phase completed
        ptx::mbar_arrive_cluster_relaxed(peer_bar + (uint32_t)((j % kSK) * sizeof(uint64_t)));
      }
    }
  } else if (warp < 4) {
    // ------------------------------------------------------------ importance
    const int t = tid - 64;   // key row t of this CTA's half of each tile
    for (int j = 0; j < n_tiles; ++j) {
      const int s = j % kSK;
      if (aux->abort_flag ||
          !ptx::mbar_wait_cluster(&aux->k_full[s], (uint32_t)(j / kSK) & 1u, kWaitCycles)) {
        timeout(aux, status);
        break;
      }
      const int64_t ja = j0 + (int64_t)j * kNk + kHalf * (int)rank + t;
      if (do_imp && ja < j1) {
        const uint8_t* ra = sk + s * Ly::kKStage + t * 128;
        uint64_t a0 = 0, a1 = 0;
#pragma unroll
        for (int c = 0; c < C16; ++c) {
          const int p = c >> 3, cc = c & 7;
          const uint4 u = *reinterpret_cast<const uint4*>(ra + p * Ly::kKPanel + ((cc ^ (t & 7)) << 4));
          const float4 q0 = *reinterpret_cast<const float4*>(qsum + 8 * c);
          const float4 q1 = *reinterpret_cast<const float4*>(qsum + 8 * c + 4);
          auto lohi = [](uint32_t w) {
            return ptx::f2(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
          };
          a0 = ptx::fma2(lohi(u.x), ptx::f2(q0.x, q0.y), a0);
          a1 = ptx::fma2(lohi(u.y), ptx::f2(q0.z, q0.w), a1);
          a0 = ptx::fma2(lohi(u.z), ptx::f2(q1.x, q1.y), a0);
          a1 = ptx::fma2(lohi(u.w), ptx::f2(q1.z, q1.w), a1);
        }
        float x0, x1;
        ptx::f2_split(ptx::add2(a0, a1), x0, x1);
        imp[(size_t)kv * L + ja] = (x0 + x1) * scale;
      }
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&aux->k_empty[s]);
    }
  } else if (warp >= 8 && warp < 12) {
    // ------------------------------------------------------------ V conversion
    const int t = tid - 8 * 32;
    constexpr int kChunks = Ly::kVStage / 16;
    float vmax = 0.f;
    for (int j = 0; j < n_tiles; ++j) {
      const int s = j % kSV;
      const bool got = !aux->abort_flag &&
                       ptx::mbar_wait_cluster(&aux->v_full[s], (uint32_t)(j / kSV) & 1u, kWaitCycles);
      if (!__all_sync(0xffffffffu, got)) {
        timeout(aux, status);
        break;
      }
      uint4* vt = reinterpret_cast<uint4*>(sv + s * Ly::kVStage);
#pragma unroll 8
      for (int e = t; e < kChunks; e += 128) {
        uint4 u = vt[e];
        uint32_t wd[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int x = 0; x < 4; ++x) {
          const float lo = __uint_as_float(wd[x] << 16), hi = __uint_as_float(wd[x] & 0xFFFF0000u);
          vmax = ptx::max3(vmax, fabsf(lo), fabsf(hi));
          wd[x] = ptx::pack_f16x2_sat(lo, hi);
        }
        vt[e] = make_uint4(wd[0], wd[1], wd[2], wd[3]);
      }
      ptx::fence_proxy_async_smem();   // generic writes -> the MMA's async-proxy reads
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive_cluster_relaxed(lead(&aux->v_conv[s]));
    }
    if (!(vmax <= 65504.f)) set_status(status, TS_ERR_UNSUPPORTED);
  } else {
    // ------------------------------------------------------------ softmax
    // warpgroup w (warps 4..7: w = 0, 12..15: w = 1) runs the online softmax
    // of the tiles j = w (mod 2) into O_w; the two streams merge at the end
    const int w = warp >= 12 ? 1 : 0;
    const int quarter = warp & 3;
    const int t = quarter * 32 + lane;
    const int R = 128 * (int)rank + t;
    const bool valid = R < M;
    const unsigned long long anc = valid ? aux->anc[R / G] : 0ull;
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    const uint32_t o_addr = tmem + lane_off + Ly::obase(w);
    float m_used = -INFINITY, l = 0.f;
    bool ok = true;
    const uint32_t p_ready_lead = lead(&aux->p_ready[w]);
    const int b = w;
    const uint32_t s_addr = tmem + lane_off + Ly::sbase(b);
    for (int j = w; j < n_tiles; j += 2) {
      bool got = !aux->abort_flag &&
                 ptx::mbar_wait_cluster(&aux->s_full[b], (uint32_t)(j >> 1) & 1u, kWaitCycles);
      if (!__all_sync(0xffffffffu, got)) {
        ok = false;
        break;
      }
      ptx::tc_fence_after();
      const int64_t key0 = j0 + (int64_t)j * kNk;
      const bool edge = key0 + kNk > jlim;
      auto clampk = [](int64_t v) { return (int)(v < 0 ? 0 : (v > kNk ? kNk : v)); };
      const int lim = clampk(jlim - key0);
      const int t_lo = clampk(L - key0);
      const int t_hi = clampk(jend - key0);
      const int sh = (int)(key0 - L);
      auto mask = [&](uint32_t (&r)[32], int c) {
#pragma unroll
        for (int x = 0; x < 32; ++x) {
          const int xx = 32 * c + x;
          const bool vis = xx < lim ||
                           (xx >= t_lo && xx < t_hi && ((anc >> ((xx + sh) & 63)) & 1ull));
          if (!vis) r[x] = kNegInf;
        }
      };
      // pass 1: tile maximum (chunks 0 and 1 stay in registers for pass 2)
      uint32_t ca[32], cb[32];
      ptx::tmem_ld32(s_addr + 64, ca);
      ptx::tmem_ld32(s_addr + 96, cb);
      ptx::tmem_ld_wait();
      if (edge) {
        mask(ca, 2);
        mask(cb, 3);
      }
      float mx = fmaxf(fmax32(ca), fmax32(cb));
      ptx::tmem_ld32(s_addr, ca);
      ptx::tmem_ld32(s_addr + 32, cb);
      ptx::tmem_ld_wait();
      if (edge) {
        mask(ca, 0);
        mask(cb, 1);
      }
      mx = fmaxf(mx, fmaxf(fmax32(ca), fmax32(cb)));
      // lazy running max.  S_b of tile j completing implies P V of tile j-2
      // (this stream's previous tile) did: Q K^T of tile j was issued after it
      const float ms = mx * sl2;
      const bool raise = ms > m_used + kLazy;
      const float f = raise ? ptx::ex2(m_used - ms) : 1.f;   // 0 when m_used = -inf
      if (raise) {
        l *= f;
        m_used = ms;
      }
      if (j >= 2 && __any_sync(0xffffffffu, raise)) {
#pragma unroll 1
        for (int c = 0; c < kD / 16; ++c) {
          uint32_t o[16];
          ptx::tmem_ld16(o_addr + c * 16, o);
          ptx::tmem_ld_wait();
#pragma unroll
          for (int x = 0; x < 16; ++x) o[x] = __float_as_uint(__uint_as_float(o[x]) * f);
          ptx::tmem_st16(o_addr + c * 16, o);
        }
        ptx::tmem_st_wait();
      }
      // pass 2: P = 2^(s*sl2 - m) -> fp16 pairs over the chunk's own columns;
      // m_used is still -inf only when every score so far is -inf: reference
      // 0 then gives 2^-inf = 0
      const float mref = (m_used == -INFINITY) ? 0.f : m_used;
      const uint64_t sl2x2 = ptx::f2(sl2, sl2);
      const uint64_t negm = ptx::f2(-mref, -mref);
      uint64_t lsum = 0;
      auto process = [&](uint32_t (&r)[32], int c) {
        if (edge && c >= 2) mask(r, c);
        uint32_t pw[16];
#pragma unroll
        for (int x = 0; x < 16; ++x) {
          float t0, t1;
          ptx::f2_split(ptx::fma2(ptx::f2(__uint_as_float(r[2 * x]), __uint_as_float(r[2 * x + 1])),
                                  sl2x2, negm),
                        t0, t1);
          const float p0 = ptx::ex2(t0), p1 = ptx::ex2(t1);
          lsum = ptx::add2(lsum, ptx::f2(p0, p1));
          pw[x] = ptx::pack_f16x2(p0, p1);
        }
        ptx::tmem_st16(s_addr + 32 * c, pw);
      };
      process(ca, 0);
      ptx::tmem_ld32(s_addr + 64, ca);
      process(cb, 1);
      ptx::tmem_ld_wait();
      ptx::tmem_ld32(s_addr + 96, cb);
      process(ca, 2);
      ptx::tmem_ld_wait();
      process(cb, 3);
      {
        float a, c;
        ptx::f2_split(lsum, a, c);
        l += a + c;
      }
      ptx::tmem_st_wait();
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive_cluster_relaxed(p_ready_lead);   // P is in TMEM
    }
    // epilogue: the odd stream hands (m, l) over, the even stream merges
    // O = O_0 2^(m_0 - m) + O_1 2^(m_1 - m) into the unnormalised partial
    bool fin = ok && !aux->abort_flag && ptx::mbar_wait_cluster(&aux->o_final, 0, kWaitCycles);
    const bool all_fin = __all_sync(0xffffffffu, fin);
    if (w == 1) {
      aux->ml_odd[t][0] = m_used;
      aux->ml_odd[t][1] = l;
    }
    ptx::named_bar_sync(1, 256);   // the two softmax warpgroups
    if (w == 0 && all_fin) {
      ptx::tc_fence_after();
      const float m1 = n_tiles >= 2 ? aux->ml_odd[t][0] : -INFINITY;
      const float l1 = n_tiles >= 2 ? aux->ml_odd[t][1] : 0.f;
      const float mm = fmaxf(m_used, m1);
      const float f0 = (m_used == -INFINITY) ? 0.f : ptx::ex2(m_used - mm);
      const float f1 = (m1 == -INFINITY) ? 0.f : ptx::ex2(m1 - mm);
      const uint32_t o1_addr = tmem + lane_off + Ly::obase(1);
      float4* dst = reinterpret_cast<float4*>(part_o) +
                    part_o4_index(kv, split, n_split, 0, kD, M, valid ? R : 0);
#pragma unroll 1
      for (int c = 0; c < kD / 16; ++c) {
        uint32_t o0[16], o1[16];
        ptx::tmem_ld16(o_addr + c * 16, o0);
        ptx::tmem_ld16(o1_addr + c * 16, o1);
        ptx::tmem_ld_wait();
        float v[16];
#pragma unroll
        for (int x = 0; x < 16; ++x) {
          const float a0 = f0 == 0.f ? 0.f : __uint_as_float(o0[x]) * f0;
          const float a1 = f1 == 0.f ? 0.f : __uint_as_float(o1[x]) * f1;
          v[x] = a0 + a1;
        }
        if (valid) {
#pragma unroll
          for (int x = 0; x < 4; ++x)
            dst[(size_t)(c * 4 + x) * M] = make_float4(v[4 * x], v[4 * x + 1], v[4 * x + 2], v[4 * x + 3]);
        }
      }
      const size_t base = ((size_t)kv * n_split + split) * M + R;
      if (valid) {
        part_ml[base * 2] = mm;
        part_ml[base * 2 + 1] = l * f0 + l1 * f1;
      }
    } else if (!all_fin) {
      timeout(aux, status);
    }
    if (!ok) timeout(aux, status);
  }

  ptx::tc_fence_before();
  __syncthreads();
  // both CTAs are done with each other's barriers, shared memory and TMEM
  ptx::cluster_sync();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc2(tmem, Ly::kTmemCols);
  }
}

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn2() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

// [Hkv*L_cap, 128] bf16 viewed in boxes of 64 columns x `rows` rows, 128-byte swizzle
int make_map(CUtensorMap* map, const void* base, int Hkv, int64_t L_cap, int rows) {
  EncodeTiledFn fn = encode_fn2();
  if (!fn) return fail(TS_ERR_CUDA, "cuTensorMapEncodeTiled is unavailable");
  cuuint64_t dims[2] = {(cuuint64_t)kD, (cuuint64_t)Hkv * (cuuint64_t)L_cap};
  cuuint64_t strides[1] = {(cuuint64_t)kD * 2};
  cuuint32_t box[2] = {64, (cuuint32_t)rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(TS_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
  return TS_OK;
}

}  // namespace

// Opt-in (TS_VERIFY_PAIR=1): on the LLaMA3.1-8B shape this kernel measures
// 0.112 ms per call against 0.100 ms for the single-SM kernel.  Each of its
// two softmax streams still waits on its own P.V -> Q.K^T round trip (about
// 4.0 K cycles per two tiles), which matches the single-SM kernel's per-tile
// chain.  The single-SM kernel stays the default.
bool verify_pair_eligible(int T, int Hq, int Hkv, int d) {
  const char* e = getenv("TS_VERIFY_PAIR");
  return e && e[0] == '1' && d == kD && T * (Hq / Hkv) == 256;
}

int launch_verify_pair(const void* q, const void* k, const void* v, int64_t L, int64_t L_cap,
                       const int32_t* parents, int T, int Hq, int Hkv, int n_imp,
                       int64_t keys_per_split, int n_split, float* part_o, float* part_ml,
                       float* imp, int32_t* status, cudaStream_t st) {
  CUtensorMap mk, mv;
  int rc = make_map(&mk, k, Hkv, L_cap, kHalf);
  if (rc) return rc;
  rc = make_map(&mv, v, Hkv, L_cap, kNk);
  if (rc) return rc;
  cudaFuncSetAttribute(verify_pair_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, Ly::kAlloc);
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[2];
  pdl_config(&cfg, attr, dim3(2 * n_split, Hkv), dim3(kThreads), Ly::kAlloc, st);
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = 2;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.numAttrs = 2;
  cudaLaunchKernelEx(&cfg, verify_pair_kernel, mk, mv, static_cast<const __nv_bfloat16*>(q), parents,
                     T, Hq, Hkv, n_imp, L, L_cap, keys_per_split, n_split, part_o, part_ml, imp,
                     status);
  return launch_status("verify_pair_kernel");
}

}  // namespace ts
