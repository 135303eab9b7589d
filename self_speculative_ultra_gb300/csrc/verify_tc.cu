// Tree verification attention on the 5th-generation tensor cores (tcgen05):
// split-KV flash-decode with the GQA group and the draft tree packed into the
// query tile, importance fused into the same K pass.
//
// "TokenSwift: Lossless Acceleration of Ultra Long Sequence Generation":
// §3.1 Overview (verification with the full KV cache), §E Tree-Based
// Attention (a tree token attends only to its predecessors), §3.3 Dynamic KV
// Cache Management (importance = query-key dot products, GQA scores
// aggregated per group).
//
// One CTA = (key split, KV head, row group).  The M = T*G query rows of the
// KV head's group are packed (row r = node r / G, head kv*G + r % G) into up
// to two 128-row tiles held in shared memory for the whole CTA, so every K/V
// tile is read from HBM once per step.  Per 128-key tile j:
//   TMA (warp 0)        K (2-stage) and V (3-stage) shared-memory rings
//                       (128-byte swizzle, L2 evict-first)
//   MMA (warp 1)        S_g = Q_g K^T (bf16, M=128, N=128, fp32 in TMEM); once
//                       the softmax has written P_g over S_g, O_g += P_g V in
//                       fp16 with P read from TMEM, then at once S_g of tile
//                       j+1.  The two row tiles ping-pong: the tensor core
//                       works on one while the other's softmax runs.
//   importance (2,3)    imp_j = (sum of the group's last n_imp queries) . k_j
//                       / sqrt(d) on CUDA cores from the same shared K tile
//                       (the importance is linear in the queries)
//   softmax (4..11)     one thread per query row, its scores read from TMEM
//                       twice (max pass, then exponent pass): tile max, lazy
//                       running max (O and l are rescaled only when the max
//                       grows past 2^8), P = 2^(s*log2e/sqrt(d) - m) written
//                       back over S in fp16 (relative rounding 2^-11, four
//                       times finer than bf16), row sums.  Tree mask and
//                       split limits only touch the tiles that need them.
//   V conversion (12..15) each V tile is converted in place from bf16 to fp16
//                       as soon as it lands (exact for |v| < 65504; larger
//                       values saturate and are reported in the status word).
// Each CTA writes an unnormalised partial (O, m, l) in the log2 domain; the
// merge kernel of verify_attn.cu combines the splits.
//
// Every mbarrier wait is bounded (~1 s of SM clocks); on expiry the CTA
// records TS_ERR_TIMEOUT in the status word, drains its own in-flight copies
// and MMAs (again bounded), frees its TMEM and returns.
#include <cstdlib>
#include <cstring>

#include "tc_ptx.cuh"
#include "ts_common.cuh"

namespace ts {

namespace {

constexpr int kNk = 128;                 // keys per tile
constexpr int kSK = 2;                   // K ring depth
constexpr int kSV = 3;                   // V ring depth
constexpr int kThreadsTc = 512;          // 16 warps
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLazy = 8.0f;            // running max refreshed only past +2^8
constexpr long long kWaitCycles = 1ll << 31;
constexpr uint32_t kNegInf = 0xFF800000u;

struct TcAux {
  uint64_t k_full[kSK], k_empty[kSK], v_full[kSV], v_conv[kSV], v_empty[kSV];
  uint64_t s_full[2], p_ready[2], o_final, drain;
  unsigned long long anc[64];
  int32_t par[64];
  uint32_t tmem_base;
  volatile int32_t abort_flag;
};

template <int D>
struct TcLayout {
  static constexpr int kPanel = 128 * 128;         // 128 rows x 64 bf16 (128-byte rows)
  static constexpr int kTile = 128 * D * 2;        // 128 rows x D bf16
  static constexpr int kQ = 0;
  static constexpr int kK = kQ + 2 * kTile;
  static constexpr int kV = kK + kSK * kTile;
  static constexpr int kQsum = kV + kSV * kTile;
  static constexpr int kAux = kQsum + D * 4;
  static constexpr int kBytes = kAux + (int)sizeof(TcAux);
  static constexpr int kAlloc = kBytes + 1024;     // slack to align the base to 1024 B
  static constexpr uint32_t kTmemCols = 512;
  // TMEM columns: O_g at g*D, S_g (128 fp32; later P) after both O tiles
  __host__ __device__ static constexpr uint32_t obase(int g) { return (uint32_t)(g * D); }
  __host__ __device__ static constexpr uint32_t sbase(int g) { return (uint32_t)(2 * D + g * kNk); }
};

__device__ __forceinline__ void timeout(TcAux* aux, int32_t* status) {
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

template <int D>
__global__ void __launch_bounds__(kThreadsTc, 1)
verify_tc_kernel(const __grid_constant__ CUtensorMap tmap_k, const __grid_constant__ CUtensorMap tmap_v,
                 const __nv_bfloat16* __restrict__ q, const int32_t* __restrict__ parents, int T,
                 int Hq, int Hkv, int n_imp, int64_t L, int64_t L_cap, int64_t keys_per_split,
                 int n_split, float* __restrict__ part_o, float* __restrict__ part_ml,
                 float* __restrict__ imp, int32_t* status) {
  using Ly = TcLayout<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~uintptr_t(1023));
  uint8_t* sq = sm + Ly::kQ;
  uint8_t* sk = sm + Ly::kK;
  uint8_t* sv = sm + Ly::kV;
  float* qsum = reinterpret_cast<float*>(sm + Ly::kQsum);
  TcAux* aux = reinterpret_cast<TcAux*>(sm + Ly::kAux);

  const int split = blockIdx.x, kv = blockIdx.y, rg = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = Hq / Hkv, M = T * G;
  const int r0 = rg * 256;
  const int nt = min(2, (M - r0 + 127) / 128);
  const int64_t j0 = (int64_t)split * keys_per_split;
  const int64_t j1 = min(L, j0 + keys_per_split);
  const bool last = (split == n_split - 1);
  const int64_t jend = last ? L + T : j1;
  const int64_t jlim = last ? L : j1;           // keys below need no mask
  const int n_tiles = (int)((jend - j0 + kNk - 1) / kNk);
  const bool do_imp = (imp != nullptr) && rg == 0;
  const float scale = 1.0f / sqrtf((float)D);
  const float sl2 = scale * kLog2e;
  const int n_pre = min(n_tiles, kSK);          // tiles loaded during the set-up
  static_assert(kSK < kSV, "early loads fill K and V stages alike; the last V stage is set-up scratch");

  // ---------------------------------------------------------------- set-up
  // launched as a programmatic dependent: nothing the previous kernel of the
  // stream wrote is read before this
  griddep_wait();
  if (tid == 0) {
    for (int s = 0; s < kSK; ++s) {
      ptx::mbar_init(&aux->k_full[s], 1);
      ptx::mbar_init(&aux->k_empty[s], 1 + 2);   // MMA commit + two importance warps
    }
    for (int s = 0; s < kSV; ++s) {
      ptx::mbar_init(&aux->v_full[s], 1);
      ptx::mbar_init(&aux->v_conv[s], 4);        // one arrival per conversion warp
      ptx::mbar_init(&aux->v_empty[s], 1);
    }
    for (int g = 0; g < 2; ++g) {
      ptx::mbar_init(&aux->s_full[g], 1);
      ptx::mbar_init(&aux->p_ready[g], 128);
    }
    ptx::mbar_init(&aux->o_final, 1);
    ptx::mbar_init(&aux->drain, 1);
    aux->abort_flag = 0;
    ptx::fence_mbar_init();
    // the first K and V tiles go out before the rest of the set-up, which
    // then runs under their HBM latency; every stage is free at this point
    const uint64_t pol = ptx::l2_evict_first_policy();
    const int row0 = (int)(kv * L_cap + j0);
    for (int jj = 0; jj < n_pre; ++jj) {
      ptx::mbar_arrive_expect_tx(&aux->k_full[jj], Ly::kTile);
      for (int p = 0; p < D / 64; ++p)
        ptx::tma_load_2d(sk + jj * Ly::kTile + p * Ly::kPanel, &tmap_k, &aux->k_full[jj], p * 64,
                         row0 + jj * kNk, pol);
      ptx::mbar_arrive_expect_tx(&aux->v_full[jj], Ly::kTile);
      for (int p = 0; p < D / 64; ++p)
        ptx::tma_load_2d(sv + jj * Ly::kTile + p * Ly::kPanel, &tmap_v, &aux->v_full[jj], p * 64,
                         row0 + jj * kNk, pol);
    }
  }
  if (tid < T) aux->par[tid] = parents[tid];
  if (warp == 1) {
    ptx::tmem_alloc(&aux->tmem_base, Ly::kTmemCols);
    ptx::tmem_relinquish();
  }
  // Q tiles -> shared memory in the 128-byte-swizzled K-major layout
  constexpr int C16 = D / 8;                     // 16-byte chunks per row
  constexpr int kQAll = 2 * 128 * C16, kQPer = (kQAll + kThreadsTc - 1) / kThreadsTc;
  {
    // all loads of a thread are in flight together, then all stores
    uint4 val[kQPer];
#pragma unroll
    for (int k = 0; k < kQPer; ++k) {
      const int e = tid + k * kThreadsTc;
      const int g = e / (128 * C16), rem = e % (128 * C16);
      const int t = rem / C16, c = rem % C16;
      const int R = r0 + g * 128 + t;
      val[k] = make_uint4(0, 0, 0, 0);
      if (e < kQAll && g < nt && R < M) {
        const int i = R / G, h = kv * G + R % G;
        val[k] = __ldg(reinterpret_cast<const uint4*>(q + ((size_t)i * Hq + h) * D + c * 8));
      }
    }
#pragma unroll
    for (int k = 0; k < kQPer; ++k) {
      const int e = tid + k * kThreadsTc;
      if (e < kQAll) {
        const int g = e / (128 * C16), rem = e % (128 * C16);
        const int t = rem / C16, c = rem % C16;
        const int p = c >> 3, cc = c & 7;
        *reinterpret_cast<uint4*>(sq + g * Ly::kTile + p * Ly::kPanel + t * 128 +
                                  ((cc ^ (t & 7)) << 4)) = val[k];
      }
    }
  }
  __syncthreads();
  // summed importance queries over the packed rows (T - n_imp) * G .. M - 1:
  // thread (16-byte column chunk, row slice) partial sums, rows of this
  // CTA's Q tiles (r0 = 0 here) read back from shared memory; the slices are
  // folded by shuffles, then across warps through the last V stage, which
  // the producer fills only after the set-up
  float* qpart = reinterpret_cast<float*>(sv + (kSV - 1) * Ly::kTile);
  if (do_imp) {
    const int cg = tid % C16, slice = tid / C16, nsl = kThreadsTc / C16;
    const int p = cg >> 3, cc = cg & 7;
    const int in_smem = min(M, nt * 128);
    uint64_t acc[4] = {0, 0, 0, 0};
    auto add8 = [&](const uint4& u) {
      const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
      for (int x = 0; x < 4; ++x)
        acc[x] = ptx::add2(acc[x], ptx::f2(__uint_as_float(w[x] << 16),
                                           __uint_as_float(w[x] & 0xFFFF0000u)));
    };
    int R = (T - n_imp) * G + slice;
#pragma unroll 4
    for (; R < in_smem; R += nsl) {
      const int tr = R & 127;
      add8(*reinterpret_cast<const uint4*>(sq + (R >> 7) * Ly::kTile + p * Ly::kPanel + tr * 128 +
                                           ((cc ^ (tr & 7)) << 4)));
    }
#pragma unroll 4
    for (; R < M; R += nsl) {
      const int i = R / G, h = kv * G + R % G;
      add8(__ldg(reinterpret_cast<const uint4*>(q + ((size_t)i * Hq + h) * D + cg * 8)));
    }
    float f[8];
#pragma unroll
    for (int x = 0; x < 4; ++x) ptx::f2_split(acc[x], f[2 * x], f[2 * x + 1]);
#pragma unroll
    for (int off = C16; off < 32; off <<= 1)
#pragma unroll
      for (int x = 0; x < 8; ++x) f[x] += __shfl_xor_sync(0xffffffffu, f[x], off);
    if (lane < C16) {
      float4* dst = reinterpret_cast<float4*>(qpart + warp * D + lane * 8);
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
    if (bad && split == 0 && kv == 0 && rg == 0) set_status(status, TS_ERR_INVALID_ARG);
  }
  if (do_imp) {
    __syncthreads();
    if (tid < D) {
      float sum = 0.f;
#pragma unroll
      for (int w = 0; w < kThreadsTc / 32; ++w) sum += qpart[w * D + tid];
      qsum[tid] = sum;
    }
  }
  ptx::fence_proxy_async_smem();
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = aux->tmem_base;
  griddep_launch_dependents();   // the merge kernel may take SMs as CTAs retire
  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const uint64_t pol = ptx::l2_evict_first_policy();
      const int row0 = (int)(kv * L_cap + j0);
      int jk = n_pre, jv = n_pre;   // tiles whose K / V load has been issued
      for (; jk < n_tiles; ++jk) {
        const int s = jk % kSK;
        if (jk >= kSK &&
            !ptx::mbar_wait(&aux->k_empty[s], (uint32_t)(jk / kSK - 1) & 1u, kWaitCycles)) {
          timeout(aux, status);
          break;
        }
        ptx::mbar_arrive_expect_tx(&aux->k_full[s], Ly::kTile);
        for (int p = 0; p < D / 64; ++p)
          ptx::tma_load_2d(sk + s * Ly::kTile + p * Ly::kPanel, &tmap_k, &aux->k_full[s], p * 64,
                           row0 + jk * kNk, pol);
        const int sv_ = jv % kSV;
        if (jv >= kSV &&
            !ptx::mbar_wait(&aux->v_empty[sv_], (uint32_t)(jv / kSV - 1) & 1u, kWaitCycles)) {
          timeout(aux, status);
          ++jk;
          break;
        }
        ptx::mbar_arrive_expect_tx(&aux->v_full[sv_], Ly::kTile);
        for (int p = 0; p < D / 64; ++p)
          ptx::tma_load_2d(sv + sv_ * Ly::kTile + p * Ly::kPanel, &tmap_v, &aux->v_full[sv_],
                           p * 64, row0 + jv * kNk, pol);
        ++jv;
        if (aux->abort_flag) {
          ++jk;
          break;
        }
      }
      if (aux->abort_flag) {
        // drain: wait (bounded) for the loads issued into each stage
        for (int t = max(0, jk - kSK); t < jk; ++t)
          ptx::mbar_wait(&aux->k_full[t % kSK], (uint32_t)(t / kSK) & 1u, kWaitCycles);
        for (int t = max(0, jv - kSV); t < jv; ++t)
          ptx::mbar_wait(&aux->v_full[t % kSV], (uint32_t)(t / kSV) & 1u, kWaitCycles);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_qk = ptx::idesc_bf16_f32(128, kNk, false);
      constexpr uint32_t idesc_pv = ptx::idesc_f16_f32(128, D, true);
      // operand descriptors: built once; a descriptor's start address is its
      // low field in 16-byte units, so tile, stage and K-step offsets are adds
      const uint64_t qd0 = ptx::sdesc_sw128(ptx::smem_u32(sq), 16, 1024);
      const uint64_t kd0 = ptx::sdesc_sw128(ptx::smem_u32(sk), 16, 1024);
      const uint64_t vd0 = ptx::sdesc_sw128(ptx::smem_u32(sv), Ly::kPanel, 1024);
      constexpr uint32_t kTile16 = Ly::kTile >> 4, kPanel16 = Ly::kPanel >> 4;
      auto qk = [&](int g, int j) {
        const uint64_t a0 = qd0 + (uint64_t)(g * kTile16);
        const uint64_t b0 = kd0 + (uint64_t)((j % kSK) * kTile16);
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          const uint32_t off = (ks >> 2) * kPanel16 + (ks & 3) * 2;   // 64-element panels, 32-byte K-steps
          ptx::mma_ss(tmem + Ly::sbase(g), a0 + off, b0 + off, idesc_qk, ks > 0 ? 1u : 0u);
        }
        ptx::mma_commit(&aux->s_full[g]);
      };
      // O += P V in fp16.  Keys [32c, 32c+32) of the tile keep their fp16 P
      // pairs in S_g columns [32c, 32c+16): K-step ks (16 keys) reads the 8
      // columns at 32*(ks/2) + 8*(ks%2); V advances 16 rows (2048 bytes).
      auto pv = [&](int g, int j) {
        const uint64_t b0 = vd0 + (uint64_t)((j % kSV) * kTile16);
        const uint32_t acc = j > 0 ? 1u : 0u;
#pragma unroll
        for (int ks = 0; ks < kNk / 16; ++ks) {
          const uint32_t acol = 32 * (ks >> 1) + 8 * (ks & 1);
          ptx::mma_ts(tmem + Ly::obase(g), tmem + Ly::sbase(g) + acol, b0 + (uint64_t)(ks * 128),
                      idesc_pv, ks > 0 ? 1u : acc);
        }
      };
      bool ok = ptx::mbar_wait(&aux->k_full[0], 0, kWaitCycles);
      if (ok) {
        ptx::tc_fence_after();
        for (int g = 0; g < nt; ++g) qk(g, 0);
        ptx::mma_commit(&aux->k_empty[0]);
      }
      for (int j = 0; ok && j < n_tiles; ++j) {
        if (!ptx::mbar_wait(&aux->v_conv[j % kSV], (uint32_t)(j / kSV) & 1u, kWaitCycles)) {
          ok = false;
          break;
        }
        const bool more = j + 1 < n_tiles;
        for (int g = 0; g < nt && ok; ++g) {
          if (!ptx::mbar_wait(&aux->p_ready[g], (uint32_t)j & 1u, kWaitCycles)) {
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          pv(g, j);
          if (more) {
            if (g == 0) {
              if (!ptx::mbar_wait(&aux->k_full[(j + 1) % kSK], (uint32_t)((j + 1) / kSK) & 1u,
                                  kWaitCycles)) {
                ok = false;
                break;
              }
              ptx::tc_fence_after();
            }
            qk(g, j + 1);
          }
        }
        if (!ok) break;
        ptx::mma_commit(&aux->v_empty[j % kSV]);
        if (more) ptx::mma_commit(&aux->k_empty[(j + 1) % kSK]);
      }
      if (!ok) timeout(aux, status);
      ptx::mma_commit(&aux->o_final);
      // drain this thread's MMAs before TMEM is freed
      ptx::mma_commit(&aux->drain);
      ptx::mbar_wait(&aux->drain, 0, kWaitCycles);
    }
  } else if (warp < 4) {
    // ------------------------------------------------------------ importance
    const int t = tid - 64;   // key rows t and t + 64 of each tile
    for (int j = 0; j < n_tiles; ++j) {
      const int s = j % kSK;
      if (aux->abort_flag || !ptx::mbar_wait(&aux->k_full[s], (uint32_t)(j / kSK) & 1u,
                                             kWaitCycles)) {
        timeout(aux, status);
        break;
      }
      const int64_t ja = j0 + (int64_t)j * kNk + t, jb = ja + 64;
      if (do_imp && ja < j1) {
        const uint8_t* ra = sk + s * Ly::kTile + t * 128;
        const uint8_t* rb = ra + 64 * 128;
        uint64_t a0 = 0, a1 = 0, b0 = 0, b1 = 0;
#pragma unroll
        for (int c = 0; c < C16; ++c) {
          const int p = c >> 3, cc = c & 7;
          const int off = p * Ly::kPanel + ((cc ^ (t & 7)) << 4);   // rows t, t+64: same swizzle
          const uint4 u = *reinterpret_cast<const uint4*>(ra + off);
          const uint4 v = *reinterpret_cast<const uint4*>(rb + off);
          const float4 q0 = *reinterpret_cast<const float4*>(qsum + 8 * c);
          const float4 q1 = *reinterpret_cast<const float4*>(qsum + 8 * c + 4);
          const uint64_t qa = ptx::f2(q0.x, q0.y), qb = ptx::f2(q0.z, q0.w);
          const uint64_t qc = ptx::f2(q1.x, q1.y), qd = ptx::f2(q1.z, q1.w);
          auto lohi = [](uint32_t w) {
            return ptx::f2(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
          };
          a0 = ptx::fma2(lohi(u.x), qa, a0);
          a1 = ptx::fma2(lohi(u.y), qb, a1);
          a0 = ptx::fma2(lohi(u.z), qc, a0);
          a1 = ptx::fma2(lohi(u.w), qd, a1);
          b0 = ptx::fma2(lohi(v.x), qa, b0);
          b1 = ptx::fma2(lohi(v.y), qb, b1);
          b0 = ptx::fma2(lohi(v.z), qc, b0);
          b1 = ptx::fma2(lohi(v.w), qd, b1);
        }
        float x0, x1, y0, y1;
        ptx::f2_split(ptx::add2(a0, a1), x0, x1);
        ptx::f2_split(ptx::add2(b0, b1), y0, y1);
        imp[(size_t)kv * L + ja] = (x0 + x1) * scale;
        if (jb < j1) imp[(size_t)kv * L + jb] = (y0 + y1) * scale;
      }
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&aux->k_empty[s]);
    }
  } else if (warp >= 12) {
    // ------------------------------------------------------------ V conversion
    // V tiles are converted in place from bf16 to fp16 as soon as they land,
    // ahead of the MMA's P V (the V ring is three tiles deep)
    const int t = tid - 12 * 32;
    constexpr int kChunks = Ly::kTile / 16;          // 16-byte chunks per V tile
    constexpr int kConvThreads = kThreadsTc - 12 * 32;
    float vmax = 0.f;                                // largest |v| (fp16 range check)
    for (int j = 0; j < n_tiles; ++j) {
      const int sv_ = j % kSV;
      const bool got = !aux->abort_flag &&
                       ptx::mbar_wait(&aux->v_full[sv_], (uint32_t)(j / kSV) & 1u, kWaitCycles);
      if (!__all_sync(0xffffffffu, got)) {
        timeout(aux, status);
        break;
      }
      uint4* vt = reinterpret_cast<uint4*>(sv + sv_ * Ly::kTile);
#pragma unroll 8
      for (int e = t; e < kChunks; e += kConvThreads) {
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
      if (lane == 0) ptx::mbar_arrive(&aux->v_conv[sv_]);
    }
    if (!(vmax <= 65504.f)) set_status(status, TS_ERR_UNSUPPORTED);
  } else {
    // ------------------------------------------------------------ softmax
    const int g = (warp - 4) >> 2;
    const int quarter = warp & 3;
    const int t = quarter * 32 + lane;            // row within the tile
    const int R = r0 + g * 128 + t;
    const bool valid = (g < nt) && (R < M);
    const unsigned long long anc = valid ? aux->anc[R / G] : 0ull;
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    const uint32_t s_addr = tmem + lane_off + Ly::sbase(g);
    const uint32_t o_addr = tmem + lane_off + Ly::obase(g);
    float m_used = -INFINITY, l = 0.f;
    bool ok = true;
    if (g < nt && ok) {
      // tcgen05.ld/st are warp-collective: every branch around them is warp-uniform
      for (int j = 0; j < n_tiles; ++j) {
        bool got = !aux->abort_flag &&
                   ptx::mbar_wait(&aux->s_full[g], (uint32_t)j & 1u, kWaitCycles);
        if (!__all_sync(0xffffffffu, got)) {
          ok = false;
          break;
        }
        ptx::tc_fence_after();
        const int64_t key0 = j0 + (int64_t)j * kNk;
        const bool edge = key0 + kNk > jlim;       // uniform: depends on the tile only
        // key0 + x is visible iff x < lim or (t_lo <= x < t_hi and its tree
        // node x + sh is on this row's root path)
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
        // pass 1: tile maximum; chunks 0 and 1 are loaded last and stay in
        // registers for pass 2
        float mx;
        uint32_t ca[32], cb[32];
        ptx::tmem_ld32(s_addr + 64, ca);
        ptx::tmem_ld32(s_addr + 96, cb);
        ptx::tmem_ld_wait();
        if (edge) {
          mask(ca, 2);
          mask(cb, 3);
        }
        mx = fmaxf(fmax32(ca), fmax32(cb));
        ptx::tmem_ld32(s_addr, ca);
        ptx::tmem_ld32(s_addr + 32, cb);
        ptx::tmem_ld_wait();
        if (edge) {
          mask(ca, 0);
          mask(cb, 1);
        }
        mx = fmaxf(mx, fmaxf(fmax32(ca), fmax32(cb)));
        // lazy running max: raise it only when the tile max exceeds it by 2^8.
        // S_g of this tile completing implies P_g V of the previous tile did
        // (MMAs of one thread complete in order), so O_g may be rescaled.
        const float ms = mx * sl2;
        const bool raise = ms > m_used + kLazy;
        const float f = raise ? ptx::ex2(m_used - ms) : 1.f;   // 0 when m_used = -inf
        if (raise) {
          l *= f;
          m_used = ms;
        }
        if (j > 0 && __any_sync(0xffffffffu, raise)) {
#pragma unroll 1
          for (int c = 0; c < D / 16; ++c) {
            uint32_t o[16];
            ptx::tmem_ld16(o_addr + c * 16, o);
            ptx::tmem_ld_wait();
#pragma unroll
            for (int x = 0; x < 16; ++x) o[x] = __float_as_uint(__uint_as_float(o[x]) * f);
            ptx::tmem_st16(o_addr + c * 16, o);
          }
          ptx::tmem_st_wait();
        }
        // pass 2: P = 2^(s*sl2 - m) -> fp16 pairs, written over the chunk's
        // own columns once it has been loaded; two chunks in flight
        // when the running max is still -inf every score of the row seen so
        // far, this tile included, is -inf: reference 0 then gives 2^-inf = 0
        const float mref = (m_used == -INFINITY) ? 0.f : m_used;
        const uint64_t sl2x2 = ptx::f2(sl2, sl2);
        const uint64_t negm = ptx::f2(-mref, -mref);
        uint64_t lsum = 0;
        // chunks 0 and 1 arrive masked from pass 1; chunks 2 and 3 are reloaded
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
        ptx::mbar_arrive(&aux->p_ready[g]);
      }
      // epilogue: final O row -> unnormalised partial
      bool fin = ok && !aux->abort_flag && ptx::mbar_wait(&aux->o_final, 0, kWaitCycles);
      if (__all_sync(0xffffffffu, fin)) {
        ptx::tc_fence_after();
        // column-quad-major partial: for each float4 column the warp's 32
        // rows are 512 contiguous bytes
        float4* dst = reinterpret_cast<float4*>(part_o) +
                      part_o4_index(kv, split, n_split, 0, D, M, valid ? R : 0);
        const size_t c4_stride = (size_t)M;
#pragma unroll 1
        for (int c = 0; c < D / 32; ++c) {
          uint32_t o[32];
          ptx::tmem_ld32(o_addr + c * 32, o);
          ptx::tmem_ld_wait();
          if (valid) {
#pragma unroll
            for (int x = 0; x < 8; ++x)
              dst[(size_t)(c * 8 + x) * c4_stride] =
                  make_float4(__uint_as_float(o[4 * x]), __uint_as_float(o[4 * x + 1]),
                              __uint_as_float(o[4 * x + 2]), __uint_as_float(o[4 * x + 3]));
          }
        }
        const size_t base = ((size_t)kv * n_split + split) * M + R;
        if (valid) {
          part_ml[base * 2] = m_used;
          part_ml[base * 2 + 1] = l;
        }
      } else {
        timeout(aux, status);
      }
    }
    if (!ok) timeout(aux, status);
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, Ly::kTmemCols);
  }
}

// ------------------------------------------------------------------ host side
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static bool tried = false;
  if (!tried) {
    tried = true;
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

int make_kv_map(CUtensorMap* map, const void* base, int Hkv, int64_t L_cap, int d) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return fail(TS_ERR_CUDA, "cuTensorMapEncodeTiled is unavailable");
  cuuint64_t dims[2] = {(cuuint64_t)d, (cuuint64_t)Hkv * (cuuint64_t)L_cap};
  cuuint64_t strides[1] = {(cuuint64_t)d * 2};
  cuuint32_t box[2] = {64, (cuuint32_t)kNk};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(TS_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
  return TS_OK;
}

}  // namespace

// Key splits per (KV head, row group): the count minimising waves x tiles per
// CTA (+ a fixed per-CTA cost), so the grid fills whole waves of the SMs.
int tc_splits(int Hkv, int n_rg, int64_t L, int nsm) {
  int64_t max_split = (L + kNk - 1) / kNk;
  if (max_split < 1) max_split = 1;
  if (max_split > 1024) max_split = 1024;
  int best = 1;
  int64_t best_cost = INT64_MAX;
  for (int n = 1; n <= max_split; ++n) {
    int64_t kps = ((L + n - 1) / n + kNk - 1) / kNk;    // tiles per split
    int64_t ctas = (int64_t)Hkv * n_rg * n;
    int64_t waves = (ctas + nsm - 1) / nsm;
    int64_t cost = waves * (kps + 3);
    if (cost < best_cost) {
      best_cost = cost;
      best = n;
    }
  }
  return best;
}

int launch_verify_tc(const void* q, const void* k, const void* v, int64_t L, int64_t L_cap,
                     const int32_t* parents, int T, int Hq, int Hkv, int d, int n_imp,
                     int64_t keys_per_split, int n_split, int n_rg, float* part_o,
                     float* part_ml, float* imp, int32_t* status, cudaStream_t st) {
  CUtensorMap mk, mv;
  int rc = make_kv_map(&mk, k, Hkv, L_cap, d);
  if (rc) return rc;
  rc = make_kv_map(&mv, v, Hkv, L_cap, d);
  if (rc) return rc;
  dim3 grid(n_split, Hkv, n_rg);
  auto qb = static_cast<const __nv_bfloat16*>(q);
  auto go = [&](auto kern, int smem) {
    cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    pdl_config(&cfg, attr, grid, dim3(kThreadsTc), smem, st);
    cudaLaunchKernelEx(&cfg, kern, mk, mv, qb, parents, T, Hq, Hkv, n_imp, L, L_cap,
                       keys_per_split, n_split, part_o, part_ml, imp, status);
  };
  if (d == 128)
    go(verify_tc_kernel<128>, TcLayout<128>::kAlloc);
  else
    go(verify_tc_kernel<64>, TcLayout<64>::kAlloc);
  return launch_status("verify_tc_kernel");
}

}  // namespace ts
