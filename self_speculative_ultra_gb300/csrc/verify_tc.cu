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
// The M = T*G query rows of a KV head's group are packed (row r = node r / G,
// head kv*G + r % G).  Rows are cut into groups of 256 (two 128-row query
// tiles) while more than 128 remain; a remainder of at most 128 rows forms a
// last group.  Two kinds of CTA:
//   pair-tile CTA (a group of up to 256 rows, one key split): two query
//     tiles in shared memory for the whole CTA, each K/V tile read once and
//     used by both; the tensor core ping-pongs between the two tiles.
//   two-stream CTA (a group of at most 128 rows, two consecutive key
//     splits): one query tile; the two splits are two independent key
//     streams (even / odd tiles of the sequence), each with its own S and O
//     in TMEM, so two softmax chains overlap as in the pair-tile CTA.  Its
//     streams cover the same key ranges as the pair-tile CTAs of the other
//     rows, which read the same tiles at the same pace (the second read is
//     an L2 hit).
// Per 128-key tile:
//   TMA (warp 0)         K (2 stages; 3 in a two-stream CTA, in the unused
//                        second query slot) and V (3 stages) shared-memory
//                        rings, 128-byte swizzle
//   MMA (warp 1)         S_g = Q K^T (bf16, M=128, N=128, fp32 in TMEM); once
//                        the softmax has written P_g over S_g, O_g += P_g V in
//                        fp16 with P read from TMEM, then S_g of group g's
//                        next tile
//   importance (2, 3)    imp_j = (sum of the group's last n_imp queries) . k_j
//                        / sqrt(d) on CUDA cores from the same shared K tile
//                        (the importance is linear in the queries)
//   V conversion (4..7)  with a bf16 V cache, each V tile converted in place
//                        to fp16 as it lands (exact for |v| < 65504; larger
//                        values saturate and are reported in the status
//                        word); with an fp16 V cache the MMA takes the tile as
//                        the copy engine wrote it and these warps are idle
//   softmax (8..15)      one thread per query row, all 128 scores of a tile
//                        read from TMEM into registers at once (the softmax
//                        warpgroups hold 192 registers a thread, the others
//                        64).  The tile is exponentiated against the running
//                        max m: P = 2^(s*log2e/sqrt(d) - m) in fp16 (relative
//                        rounding 2^-11), packed in registers; while the
//                        tile's row sum of P stays <= 2^15 it is written back
//                        over S as is, with no pass for the tile max.  Else
//                        (or while m is -inf) m is raised to the tile max, O
//                        and l are rescaled (after the tile's P stores) and
//                        P is recomputed.  Tree mask and split limits (as bit
//                        masks over 64 keys) only touch the tiles that need
//                        them.
// Each stream writes its partial per row: O / l in fp16 and (m, l) in the
// log2 domain; the merge kernel of verify_attn.cu combines the splits.
//
// Every mbarrier wait is bounded (a caller-settable limit, ~1 s of SM clocks
// by default); on expiry the CTA records TS_ERR_TIMEOUT in the status word,
// waits (with the default limit) for its own in-flight copies and MMAs,
// frees its TMEM and returns.  The producer always waits for every copy it
// issued before the CTA exits.
#include <cstdlib>
#include <cstring>

#include "tc_ptx.cuh"
#include "ts_common.cuh"

namespace ts {

namespace {

constexpr int kNk = 128;                 // keys per tile
constexpr int kSV = 3;                   // V ring depth
constexpr int kThreadsTc = 512;          // 16 warps
constexpr int kSoftmaxWarp0 = 8;         // warps 8..15
// registers a thread after the role split: the launch holds 512 x 128; the
// two softmax warpgroups take 192 (all 128 scores of a row in registers),
// the other two keep 64, so 2 x 128 x 64 + 2 x 128 x 192 = 65,536
constexpr int kRegsLow = 64;
constexpr int kRegsSoftmax = 192;
static_assert(2 * 128 * kRegsLow + 2 * 128 * kRegsSoftmax == kThreadsTc * 128,
              "the register split must use exactly the launch's registers");
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kFastSum = 32768.0f;     // a tile's P is kept while its row sum <= 2^15
constexpr long long kDrainCycles = 1ll << 31;
constexpr uint32_t kNegInf = 0xFF800000u;

struct TcAux {
  uint64_t k_full[3], k_empty[3], v_full[kSV], v_conv[kSV], v_empty[kSV];
  uint64_t s_full[2], p_ready[2], o_final, drain;
  uint32_t tmem_base;
  volatile int32_t abort_flag;
};

// The draft tree during the set-up: parents and ancestor-or-self masks.
struct SetupScratch {
  unsigned long long anc[64];
  int32_t par[64];
};

template <int D>
struct TcLayout {
  static constexpr int kPanel = 128 * 128;         // 128 rows x 64 bf16 (128-byte rows)
  static constexpr int kTile = 128 * D * 2;        // 128 rows x D bf16
  static constexpr int kQ = 0;                     // Q tile 0 | Q tile 1 (or K stage 2)
  static constexpr int kK = kQ + 2 * kTile;        // K stages 0, 1
  static constexpr int kV = kK + 2 * kTile;
  static constexpr int kQsum = kV + kSV * kTile;
  static constexpr int kTree = kQsum + D * 4;
  static constexpr int kAux = kTree + (int)sizeof(SetupScratch);
  static constexpr int kBytes = kAux + (int)sizeof(TcAux);
  static constexpr uint32_t kTmemCols = 512;
  // TMEM columns: O_g at g*D, S_g (128 fp32; later P) after both O tiles
  __host__ __device__ static constexpr uint32_t obase(int g) { return (uint32_t)(g * D); }
  __host__ __device__ static constexpr uint32_t sbase(int g) { return (uint32_t)(2 * D + g * kNk); }
};

__device__ __forceinline__ void timeout(TcAux* aux, int32_t* status) {
  aux->abort_flag = 1;
  set_status(status, TS_ERR_TIMEOUT);
}

// One key stream: the split it covers and its tiles.
// Key positions fit 31 bits (the cache capacity is checked on the host).
struct Stream {
  int j0, j1, jend, jlim;   // keys [j0, jend); below jlim no mask is needed
  int n;                    // tiles
};
__device__ __forceinline__ Stream make_stream(int split, int n_split, int64_t kps, int64_t L,
                                              int T) {
  Stream s;
  if (split >= n_split) {
    s.j0 = s.j1 = s.jend = s.jlim = 0;
    s.n = 0;
    return s;
  }
  const bool last = split == n_split - 1;
  s.j0 = (int)((int64_t)split * kps);
  s.j1 = (int)min(L, (int64_t)s.j0 + kps);
  s.jend = last ? (int)L + T : s.j1;
  s.jlim = last ? (int)L : s.j1;
  s.n = (s.jend - s.j0 + kNk - 1) / kNk;
  return s;
}

// Tile sequence of a CTA (the order of the K/V rings).  Pair-tile CTA: one
// stream, tile s is (both groups, k = s).  Two-stream CTA: the streams'
// tiles alternate (g0 k0, g1 k0, g0 k1, ...) while both have tiles, then the
// longer stream's remainder follows.
struct Seq {
  bool two;
  int n0, n1, nmin;
  __device__ __forceinline__ int total() const { return two ? n0 + n1 : n0; }
  __device__ __forceinline__ void decode(int s, int& g, int& k) const {
    if (!two) {
      g = 0;
      k = s;
    } else if (s < 2 * nmin) {
      g = s & 1;
      k = s >> 1;
    } else {
      g = n0 > n1 ? 0 : 1;
      k = nmin + (s - 2 * nmin);
    }
  }
  __device__ __forceinline__ int index(int g, int k) const {
    if (!two) return k;
    return k < nmin ? 2 * k + g : 2 * nmin + (k - nmin);
  }
};

__device__ __forceinline__ float fmax32(const uint32_t* r) {
  float a = ptx::max3(__uint_as_float(r[0]), __uint_as_float(r[1]), __uint_as_float(r[2]));
  float b = ptx::max3(__uint_as_float(r[3]), __uint_as_float(r[4]), __uint_as_float(r[5]));
#pragma unroll
  for (int x = 6; x < 30; x += 4) {
    a = ptx::max3(a, __uint_as_float(r[x]), __uint_as_float(r[x + 1]));
    b = ptx::max3(b, __uint_as_float(r[x + 2]), __uint_as_float(r[x + 3]));
  }
  return ptx::max3(a, b, fmaxf(__uint_as_float(r[30]), __uint_as_float(r[31])));
}

template <int D, bool kVF16>
__global__ void __launch_bounds__(kThreadsTc, 1)
verify_tc_kernel(const __grid_constant__ CUtensorMap tmap_k, const __grid_constant__ CUtensorMap tmap_v,
                 const __nv_bfloat16* __restrict__ q, const int32_t* __restrict__ parents, int T,
                 int Hq, int Hkv, int n_imp, int64_t L, int64_t L_cap, int64_t keys_per_split,
                 int n_split, int n_pairtile_groups, long long wait_limit,
                 uint4* __restrict__ part_o, float* __restrict__ part_ml, float* __restrict__ imp,
                 int32_t* status) {
  using Ly = TcLayout<D>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* sm = smem_raw;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // the 128-byte swizzle needs 1024-byte aligned tiles
  if ((ptx::smem_u32(sm) & 1023u) != 0) {
    if (tid == 0) set_status(status, TS_ERR_CUDA);
    return;
  }
  uint8_t* sq = sm + Ly::kQ;
  uint8_t* sk = sm + Ly::kK;
  uint8_t* sv = sm + Ly::kV;
  float* qsum = reinterpret_cast<float*>(sm + Ly::kQsum);
  SetupScratch* scr = reinterpret_cast<SetupScratch*>(sm + Ly::kTree);
  TcAux* aux = reinterpret_cast<TcAux*>(sm + Ly::kAux);

  // ---------------------------------------------------------------- which work
  const int kv = blockIdx.y, x = blockIdx.x;
  const int G = Hq / Hkv, M = T * G;
  const int n_pt = n_pairtile_groups * n_split;     // pair-tile CTAs per head
  Seq seq;
  seq.two = x >= n_pt;
  int r0;
  Stream st0, st1;
  if (!seq.two) {
    const int rg = x / n_split, split = x % n_split;
    r0 = rg * 256;
    st0 = make_stream(split, n_split, keys_per_split, L, T);
    st1 = st0;
  } else {
    const int pair = x - n_pt;
    r0 = n_pairtile_groups * 256;
    st0 = make_stream(2 * pair, n_split, keys_per_split, L, T);
    st1 = make_stream(2 * pair + 1, n_split, keys_per_split, L, T);
  }
  seq.n0 = st0.n;
  seq.n1 = seq.two ? st1.n : 0;
  seq.nmin = min(seq.n0, seq.n1);
  const int n_seq = seq.total();
  const int nt = seq.two ? 1 : min(2, (M - r0 + 127) / 128);   // query tiles held
  const int nK = seq.two ? 3 : 2;                              // K ring depth
  const bool do_imp = (imp != nullptr) && r0 == 0;
  const float scale = 1.0f / sqrtf((float)D);
  const float sl2 = scale * kLog2e;
  const int n_pre = min(n_seq, 2);             // tiles loaded during the set-up
  auto kaddr = [&](int st) -> uint8_t* { return st < 2 ? sk + st * Ly::kTile : sq + Ly::kTile; };
  auto key0_of = [&](int g, int k) -> int { return (g ? st1.j0 : st0.j0) + k * kNk; };

  // ---------------------------------------------------------------- set-up
  // barriers and TMEM first: neither reads what the previous kernel of the
  // stream wrote, so they overlap its tail (programmatic dependent launch)
  if (tid == 0) {
    for (int s = 0; s < 3; ++s) {
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
      ptx::mbar_init(&aux->p_ready[g], 4);       // one arrival per softmax warp
    }
    ptx::mbar_init(&aux->o_final, 1);
    ptx::mbar_init(&aux->drain, 1);
    aux->abort_flag = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 1) {
    ptx::tmem_alloc(&aux->tmem_base, Ly::kTmemCols);
    ptx::tmem_relinquish();
  }
  griddep_wait();
  __syncthreads();
  if (tid < T) scr->par[tid] = parents[tid];
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
    if (tid == 0) {
      // the first K/V tiles go out right behind the query loads; the rest
      // of the set-up runs under their HBM latency.  Every stage is free.
      const uint64_t pol = ptx::l2_evict_first_policy();
      for (int s = 0; s < n_pre; ++s) {
        int g, k;
        seq.decode(s, g, k);
        const int row = (int)(kv * L_cap + key0_of(g, k));
        ptx::mbar_arrive_expect_tx(&aux->k_full[s], Ly::kTile);
        for (int p = 0; p < D / 64; ++p)
          ptx::tma_load_2d(kaddr(s) + p * Ly::kPanel, &tmap_k, &aux->k_full[s], p * 64, row, pol);
        ptx::mbar_arrive_expect_tx(&aux->v_full[s], Ly::kTile);
        for (int p = 0; p < D / 64; ++p)
          ptx::tma_load_2d(sv + s * Ly::kTile + p * Ly::kPanel, &tmap_v, &aux->v_full[s], p * 64,
                           row, pol);
      }
    }
#pragma unroll
    for (int k = 0; k < kQPer; ++k) {
      const int e = tid + k * kThreadsTc;
      const int g = e / (128 * C16);
      if (e < kQAll && g < nt) {
        const int rem = e % (128 * C16);
        const int t = rem / C16, c = rem % C16;
        const int p = c >> 3, cc = c & 7;
        *reinterpret_cast<uint4*>(sq + g * Ly::kTile + p * Ly::kPanel + t * 128 +
                                  ((cc ^ (t & 7)) << 4)) = val[k];
      }
    }
  }
  __syncthreads();
  // summed importance queries over the packed rows (T - n_imp) * G .. M - 1
  // (r0 = 0 here): thread (16-byte column chunk, row slice) partial sums, the
  // rows of the CTA's query tiles read back from shared memory, the rest from
  // global memory; the slices are folded by shuffles, then across warps
  // through the last V stage, which the producer fills only after the set-up
  float* qpart = reinterpret_cast<float*>(sv + (kSV - 1) * Ly::kTile);
  constexpr int kQpartWarps = kThreadsTc / 32;
  static_assert(kQpartWarps * 128 * 4 <= 128 * 64 * 2, "qsum partials must fit one V stage");
  if (do_imp) {
    const int cg = tid % C16, slice = tid / C16, nsl = kThreadsTc / C16;
    const int p = cg >> 3, cc = cg & 7;
    const int in_smem = min(M, nt * 128);
    uint64_t acc[4] = {0, 0, 0, 0};
    auto add8 = [&](const uint4& u) {
      const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
      for (int x2 = 0; x2 < 4; ++x2)
        acc[x2] = ptx::add2(acc[x2], ptx::f2(__uint_as_float(w[x2] << 16),
                                             __uint_as_float(w[x2] & 0xFFFF0000u)));
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
    for (int x2 = 0; x2 < 4; ++x2) ptx::f2_split(acc[x2], f[2 * x2], f[2 * x2 + 1]);
#pragma unroll
    for (int off = C16; off < 32; off <<= 1)
#pragma unroll
      for (int x2 = 0; x2 < 8; ++x2) f[x2] += __shfl_xor_sync(0xffffffffu, f[x2], off);
    if (lane < C16) {
      float4* dst = reinterpret_cast<float4*>(qpart + warp * D + lane * 8);
      dst[0] = make_float4(f[0], f[1], f[2], f[3]);
      dst[1] = make_float4(f[4], f[5], f[6], f[7]);
    }
  }
  // ancestor-or-self masks: node t walks its parent chain (depth < 64)
  if (tid < T) {
    unsigned long long m = 0ull;
    bool bad = (tid == 0) ? (scr->par[0] != -1) : false;
    int a = tid;
    for (int step = 0; step < 64; ++step) {
      m |= 1ull << a;
      if (a == 0) break;
      const int pa = scr->par[a];
      if (pa < 0 || pa >= a) {
        bad = true;
        break;
      }
      a = pa;
    }
    scr->anc[tid] = m;
    if (bad && x == 0 && kv == 0) set_status(status, TS_ERR_INVALID_ARG);
  }
  __syncthreads();
  if (do_imp && tid < D) {
    float sum = 0.f;
#pragma unroll
    for (int w = 0; w < kQpartWarps; ++w) sum += qpart[w * D + tid];
    qsum[tid] = sum;
  }
  // each softmax thread: its query tile g and row t
  unsigned long long anc_row = 0ull;
  int sm_g = 0, sm_t = 0, sm_R = 0;
  bool sm_valid = false;
  if (warp >= kSoftmaxWarp0) {
    sm_g = (warp - kSoftmaxWarp0) >> 2;
    sm_t = (warp & 3) * 32 + lane;
    sm_R = seq.two ? r0 + sm_t : r0 + sm_g * 128 + sm_t;
    const bool active = seq.two ? (sm_g == 0 ? seq.n0 > 0 : seq.n1 > 0) : sm_g < nt;
    sm_valid = active && sm_R < M;
    anc_row = sm_valid ? scr->anc[sm_R / G] : 0ull;
  }
  ptx::fence_proxy_async_smem();
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = aux->tmem_base;
  griddep_launch_dependents();   // the merge kernel may take SMs as CTAs retire
  if (warp < kSoftmaxWarp0) {
    // producer, MMA, importance and V conversion run in kRegsLow registers
    // a thread; the softmax warpgroups take the registers they free
    ptx::regs_dec<kRegsLow>();
    if (warp == 0) {
      // ------------------------------------------------------------ producer
      if (lane == 0) {
        const uint64_t pol = ptx::l2_evict_first_policy();
        int s = n_pre, sv_next = n_pre;   // next tile to load (K), V loads issued
        for (; s < n_seq; ++s) {
          int g, k;
          seq.decode(s, g, k);
          const int row = (int)(kv * L_cap + key0_of(g, k));
          const int stK = s % nK;
          if (s >= nK &&
              !ptx::mbar_wait(&aux->k_empty[stK], (uint32_t)(s / nK - 1) & 1u, wait_limit)) {
            timeout(aux, status);
            break;
          }
          ptx::mbar_arrive_expect_tx(&aux->k_full[stK], Ly::kTile);
          for (int p = 0; p < D / 64; ++p)
            ptx::tma_load_2d(kaddr(stK) + p * Ly::kPanel, &tmap_k, &aux->k_full[stK], p * 64, row,
                             pol);
          const int stV = s % kSV;
          if (s >= kSV &&
              !ptx::mbar_wait(&aux->v_empty[stV], (uint32_t)(s / kSV - 1) & 1u, wait_limit)) {
            timeout(aux, status);
            ++s;          // this tile's K load is in flight
            break;
          }
          ptx::mbar_arrive_expect_tx(&aux->v_full[stV], Ly::kTile);
          for (int p = 0; p < D / 64; ++p)
            ptx::tma_load_2d(sv + stV * Ly::kTile + p * Ly::kPanel, &tmap_v, &aux->v_full[stV],
                             p * 64, row, pol);
          sv_next = s + 1;
          if (aux->abort_flag) {
            ++s;
            break;
          }
        }
        // drain: the copy engine writes this CTA's shared memory, so every
        // issued load must land before the CTA exits, whether or not a
        // consumer gave up waiting for it (in a normal run the consumers
        // already saw each of them and these waits return at once).  Earlier
        // loads into a stage completed before the stage was refilled.
        for (int t = max(0, s - nK); t < s; ++t)
          ptx::mbar_wait(&aux->k_full[t % nK], (uint32_t)(t / nK) & 1u, kDrainCycles);
        for (int t = max(0, sv_next - kSV); t < sv_next; ++t)
          ptx::mbar_wait(&aux->v_full[t % kSV], (uint32_t)(t / kSV) & 1u, kDrainCycles);
      }
    } else if (warp == 1) {
      // ------------------------------------------------------------ MMA issuer
      if (lane == 0) {
        constexpr uint32_t idesc_qk = ptx::idesc_bf16_f32(128, kNk, false);
        constexpr uint32_t idesc_pv = ptx::idesc_f16_f32(128, D, true);
        // operand descriptors: a descriptor's start address is its low field
        // in 16-byte units, so tile, stage and K-step offsets are adds
        const uint64_t qd0 = ptx::sdesc_sw128(ptx::smem_u32(sq), 16, 1024);
        const uint64_t vd0 = ptx::sdesc_sw128(ptx::smem_u32(sv), Ly::kPanel, 1024);
        constexpr uint32_t kTile16 = Ly::kTile >> 4;
        auto qk = [&](int g, int stK) {
          const uint64_t a0 = qd0 + (uint64_t)((seq.two ? 0 : g) * kTile16);
          const uint64_t b0 = ptx::sdesc_sw128(ptx::smem_u32(kaddr(stK)), 16, 1024);
  #pragma unroll
          for (int ks = 0; ks < D / 16; ++ks) {
            // 64-element panels, 32-byte K-steps
            const uint32_t off = (ks >> 2) * (Ly::kPanel >> 4) + (ks & 3) * 2;
            ptx::mma_ss(tmem + Ly::sbase(g), a0 + off, b0 + off, idesc_qk, ks > 0 ? 1u : 0u);
          }
          ptx::mma_commit(&aux->s_full[g]);
        };
        // O += P V in fp16 once the softmax has stored P (phase ph of the P
        // barrier).  The fp16 pair of keys 2x, 2x+1 sits in S_g column x:
        // K-step ks (16 keys) reads the 8 columns at 8*ks; V advances 16 rows
        // (2048 bytes).
        auto pv = [&](int g, int stV, bool acc, uint32_t ph) {
          if (!ptx::mbar_wait(&aux->p_ready[g], ph, wait_limit)) return false;
          ptx::tc_fence_after();
          const uint64_t b0 = vd0 + (uint64_t)(stV * kTile16);
  #pragma unroll
          for (int ks = 0; ks < kNk / 16; ++ks) {
            const uint32_t acol = 8 * ks;
            ptx::mma_ts(tmem + Ly::obase(g), tmem + Ly::sbase(g) + acol, b0 + (uint64_t)(ks * 128),
                        idesc_pv, (ks > 0 || acc) ? 1u : 0u);
          }
          return true;
        };
        auto wait_k = [&](int s) {
          if (!ptx::mbar_wait(&aux->k_full[s % nK], (uint32_t)(s / nK) & 1u, wait_limit)) return false;
          ptx::tc_fence_after();
          return true;
        };
        // V stages the P V product may read: converted (bf16 cache) or as
        // landed (fp16 cache)
        uint64_t* v_ready = kVF16 ? aux->v_full : aux->v_conv;
        bool ok = true;
        if (!seq.two) {
          if (n_seq > 0) {
            ok = wait_k(0);
            if (ok) {
              for (int g = 0; g < nt; ++g) qk(g, 0);
              ptx::mma_commit(&aux->k_empty[0]);
            }
          }
          for (int s = 0; ok && s < n_seq; ++s) {
            if (!ptx::mbar_wait(&v_ready[s % kSV], (uint32_t)(s / kSV) & 1u, wait_limit)) {
              ok = false;
              break;
            }
            const bool more = s + 1 < n_seq;
            for (int g = 0; g < nt && ok; ++g) {
              if (!pv(g, s % kSV, s > 0, (uint32_t)s & 1u)) {
                ok = false;
                break;
              }
              if (more) {
                if (g == 0 && !wait_k(s + 1)) {
                  ok = false;
                  break;
                }
                qk(g, (s + 1) % nK);
              }
            }
            if (!ok) break;
            ptx::mma_commit(&aux->v_empty[s % kSV]);
            if (more) ptx::mma_commit(&aux->k_empty[(s + 1) % nK]);
          }
        } else {
          // first tile of each stream
          for (int g = 0; g < 2 && ok; ++g) {
            if ((g ? seq.n1 : seq.n0) == 0) continue;
            const int s = seq.index(g, 0);
            ok = wait_k(s);
            if (ok) {
              qk(g, s % nK);
              ptx::mma_commit(&aux->k_empty[s % nK]);
            }
          }
          for (int s = 0; ok && s < n_seq; ++s) {
            int g, k;
            seq.decode(s, g, k);
            if (!ptx::mbar_wait(&v_ready[s % kSV], (uint32_t)(s / kSV) & 1u, wait_limit) ||
                !pv(g, s % kSV, k > 0, (uint32_t)k & 1u)) {
              ok = false;
              break;
            }
            ptx::mma_commit(&aux->v_empty[s % kSV]);
            if (k + 1 < (g ? seq.n1 : seq.n0)) {
              const int s2 = seq.index(g, k + 1);
              if (!wait_k(s2)) {
                ok = false;
                break;
              }
              qk(g, s2 % nK);
              ptx::mma_commit(&aux->k_empty[s2 % nK]);
            }
          }
        }
        if (!ok) timeout(aux, status);
        ptx::mma_commit(&aux->o_final);
        // drain this thread's MMAs before TMEM is freed
        ptx::mma_commit(&aux->drain);
        ptx::mbar_wait(&aux->drain, 0, kDrainCycles);
      }
    } else if (warp < 4) {
      // ------------------------------------------------------------ importance
      const int t = tid - 64;   // key rows t and t + 64 of each tile
      for (int s = 0; s < n_seq; ++s) {
        const int stK = s % nK;
        if (aux->abort_flag ||
            !ptx::mbar_wait(&aux->k_full[stK], (uint32_t)(s / nK) & 1u, wait_limit)) {
          timeout(aux, status);
          break;
        }
        int g, k;
        seq.decode(s, g, k);
        const int ja = key0_of(g, k) + t, jb = ja + 64;
        const int j1 = g ? st1.j1 : st0.j1;
        if (do_imp && ja < j1) {
          const uint8_t* ra = kaddr(stK) + t * 128;
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
        if (lane == 0) ptx::mbar_arrive(&aux->k_empty[stK]);
      }
    } else if (!kVF16) {
      // ------------------------------------------------------------ V conversion
      // V tiles are converted in place from bf16 to fp16 as soon as they land,
      // ahead of the MMA's P V (the V ring is three tiles deep)
      const int t = tid - 4 * 32;
      constexpr int kChunks = Ly::kTile / 16;          // 16-byte chunks per V tile
      constexpr int kConvThreads = 4 * 32;
      float vmax = 0.f;                                // largest |v| (fp16 range check)
      for (int s = 0; s < n_seq; ++s) {
        const int stV = s % kSV;
        const bool got = !aux->abort_flag &&
                         ptx::mbar_wait(&aux->v_full[stV], (uint32_t)(s / kSV) & 1u, wait_limit);
        if (!__all_sync(0xffffffffu, got)) {
          timeout(aux, status);
          break;
        }
        uint4* vt = reinterpret_cast<uint4*>(sv + stV * Ly::kTile);
  #pragma unroll 4
        for (int e = t; e < kChunks; e += kConvThreads) {
          uint4 u = vt[e];
          uint32_t wd[4] = {u.x, u.y, u.z, u.w};
  #pragma unroll
          for (int x2 = 0; x2 < 4; ++x2) {
            const float lo = __uint_as_float(wd[x2] << 16), hi = __uint_as_float(wd[x2] & 0xFFFF0000u);
            vmax = ptx::max3(vmax, fabsf(lo), fabsf(hi));
            wd[x2] = ptx::pack_f16x2_sat(lo, hi);
          }
          vt[e] = make_uint4(wd[0], wd[1], wd[2], wd[3]);
        }
        ptx::fence_proxy_async_smem();   // generic writes -> the MMA's async-proxy reads
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(&aux->v_conv[stV]);
      }
      if (!(vmax <= 65504.f)) set_status(status, TS_ERR_UNSUPPORTED);
    }
  } else {
    ptx::regs_inc<kRegsSoftmax>();
    // ------------------------------------------------------------ softmax
    // one thread per query row t of tile g: all 128 keys of each key tile
    const int g = sm_g;
    const bool active = seq.two ? (g == 0 ? seq.n0 > 0 : seq.n1 > 0) : g < nt;
    const int n_mine = seq.two ? (g == 0 ? seq.n0 : seq.n1) : n_seq;
    const Stream& my = (seq.two && g == 1) ? st1 : st0;
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t s_addr = tmem + lane_off + Ly::sbase(g);
    const uint32_t o_addr = tmem + lane_off + Ly::obase(g);
    float m_used = -INFINITY, l = 0.f;
    bool ok = true;
    // a warp whose 32 rows all lie past the last query row (the padding of
    // a short row group) only releases each tile's P: the MMA then reads
    // stale words in those rows, which feed O rows that are never written
    const bool warp_rows = __any_sync(0xffffffffu, sm_valid);
    if (active) {
      // tcgen05.ld/st are warp-collective: every branch around them is
      // warp-uniform
      for (int k = 0; k < n_mine; ++k) {
        bool got = !aux->abort_flag &&
                   ptx::mbar_wait(&aux->s_full[g], (uint32_t)k & 1u, wait_limit);
        got = __all_sync(0xffffffffu, got);
        const int key0 = my.j0 + k * kNk;
        const bool edge = key0 + kNk > my.jlim;     // uniform: depends on the tile only
        // visibility of the 64 keys [64*blk, 64*blk + 64) of the tile as a
        // bit mask: key0 + xx is visible iff xx < lim or (t_lo <= xx < t_hi
        // and its tree node xx + key0 - L is on this row's root path)
        auto block_mask = [&](int blk) -> uint64_t {
          auto clampk = [](int v) { return v < 0 ? 0 : (v > kNk ? kNk : v); };
          auto lowbits = [](int n) {
            return n >= 64 ? ~0ull : (n <= 0 ? 0ull : ((1ull << n) - 1ull));
          };
          const int h0 = 64 * blk;
          const int lim = clampk(my.jlim - key0);
          const int t_lo = clampk((int)L - key0);
          const int t_hi = clampk(my.jend - key0);
          uint64_t vis = lowbits(lim - h0);
          const int a = max(t_lo - h0, 0), b = min(t_hi - h0, 64);
          if (a < b) {
            const int base = h0 + key0 - (int)L;   // tree node of bit 0
            const uint64_t tb = base >= 0 ? (base < 64 ? (anc_row >> base) : 0ull)
                                          : (base > -64 ? (anc_row << -base) : 0ull);
            vis |= tb & (lowbits(b) & ~lowbits(a));
          }
          return vis;
        };
        auto apply = [](uint32_t* r, uint64_t vis) {
          const uint32_t v0 = (uint32_t)vis, v1 = (uint32_t)(vis >> 32);
#pragma unroll
          for (int x2 = 0; x2 < 32; ++x2) {
            if (!((v0 >> x2) & 1u)) r[x2] = kNegInf;
            if (!((v1 >> x2) & 1u)) r[32 + x2] = kNegInf;
          }
        };
        // all 128 scores of the row in registers: one TMEM round trip
        uint32_t r[kNk];
        auto load_s = [&]() {
          ptx::tc_fence_after();
#pragma unroll
          for (int c = 0; c < kNk / 32; ++c)
            ptx::tmem_ld32(s_addr + 32 * c, *reinterpret_cast<uint32_t(*)[32]>(r + 32 * c));
          ptx::tmem_ld_wait();
          if (edge) {
            apply(r, block_mask(0));
            apply(r + 64, block_mask(1));
          }
        };
        if (!got) {
          ok = false;
          break;
        }
        if (!warp_rows) {
          __syncwarp();
          if (lane == 0) ptx::mbar_arrive(&aux->p_ready[g]);
          continue;
        }
        load_s();
        // P = 2^(s*sl2 - m) -> fp16 pairs, in place: the pair of keys
        // 32c + 2i, 32c + 2i + 1 in r[32c + i] (i < 16), stored to S column
        // 16c + i.  Returns the tile's row sum of P.
        const uint64_t sl2x2 = ptx::f2(sl2, sl2);
        auto exp_pack = [&](float mref) -> float {
          const uint64_t negm = ptx::f2(-mref, -mref);
          // exponentials of 32-key chunk c (16 independent exponent pairs,
          // then 32 independent exponentials)
          auto chunk_exp = [&](int c, float (&pe)[32]) {
            const uint32_t* w = r + 32 * c;
#pragma unroll
            for (int x2 = 0; x2 < 16; ++x2)
              ptx::f2_split(ptx::fma2(ptx::f2(__uint_as_float(w[2 * x2]),
                                              __uint_as_float(w[2 * x2 + 1])),
                                      sl2x2, negm),
                            pe[2 * x2], pe[2 * x2 + 1]);
#pragma unroll
            for (int x = 0; x < 32; ++x) pe[x] = ptx::ex2(pe[x]);
          };
          // software-pipelined: chunk c + 1's exponentials are issued before
          // chunk c's sums and packs, which wait on the exponential unit's
          // results; two row-sum accumulators per chunk
          uint64_t acc[2 * (kNk / 32)];
          float pa[32], pb[32];
          chunk_exp(0, pa);
#pragma unroll
          for (int c = 0; c < kNk / 32; ++c) {
            float (&cur)[32] = (c & 1) ? pb : pa;
            float (&nxt)[32] = (c & 1) ? pa : pb;
            if (c + 1 < kNk / 32) chunk_exp(c + 1, nxt);
            uint32_t* w = r + 32 * c;
            uint64_t s0 = ptx::f2(cur[0], cur[1]), s1 = ptx::f2(cur[2], cur[3]);
#pragma unroll
            for (int x2 = 2; x2 < 16; x2 += 2) {
              s0 = ptx::add2(s0, ptx::f2(cur[2 * x2], cur[2 * x2 + 1]));
              s1 = ptx::add2(s1, ptx::f2(cur[2 * x2 + 2], cur[2 * x2 + 3]));
            }
            // packed pairs overwrite the chunk's first 16 score words, whose
            // scores were read by chunk_exp(c)
#pragma unroll
            for (int x2 = 0; x2 < 16; ++x2) w[x2] = ptx::pack_f16x2(cur[2 * x2], cur[2 * x2 + 1]);
            acc[2 * c] = s0;
            acc[2 * c + 1] = s1;
          }
          const uint64_t t = ptx::add2(ptx::add2(ptx::add2(acc[0], acc[1]), ptx::add2(acc[2], acc[3])),
                                       ptx::add2(ptx::add2(acc[4], acc[5]), ptx::add2(acc[6], acc[7])));
          float a, c;
          ptx::f2_split(t, a, c);
          return a + c;
        };
        // Lazy running max, decided after the exponentials: the tile is first
        // exponentiated against the running max m_used; if the row sum of
        // that P is at most 2^15, every P fits fp16 (largest finite 65504)
        // and is kept, with no pass for the tile max.  Otherwise (or while
        // m_used is still -inf) the scores are reloaded from TMEM (P is not
        // stored yet) and the max is raised to the tile max: a row sum above
        // 2^15 means some P exceeded 2^8, so the tile max lies more than 8
        // above m_used.  S_g of this tile completing implies P_g V of group
        // g's previous tile did (MMAs of one thread complete in order), so
        // O_g may be rescaled (below, before this tile's P is released).
        bool fast = m_used != -INFINITY;
        float lt = 0.f;
        if (__all_sync(0xffffffffu, fast)) {
          lt = exp_pack(m_used);
          fast = lt <= kFastSum;
        } else {
          fast = false;
        }
        bool raise = false;
        float f = 1.f;
        if (!__all_sync(0xffffffffu, fast)) {
          load_s();
          const float mx = fmaxf(fmaxf(fmax32(&r[0]), fmax32(&r[32])),
                                 fmaxf(fmax32(&r[64]), fmax32(&r[96])));
          const float ms = mx * sl2;
          raise = !fast && ms > m_used;
          f = raise ? ptx::ex2(m_used - ms) : 1.f;   // 0 when m_used = -inf
          if (raise) {
            l *= f;
            m_used = ms;
          }
          // while the running max is still -inf every score seen so far is
          // -inf: reference 0 then gives 2^-inf = 0
          lt = exp_pack(m_used == -INFINITY ? 0.f : m_used);
        }
        l += lt;
        {
          uint32_t lo[32], hi[32];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            lo[i] = r[i];
            lo[16 + i] = r[32 + i];
            hi[i] = r[64 + i];
            hi[16 + i] = r[96 + i];
          }
          ptx::tmem_st32(s_addr, lo);
          ptx::tmem_st32(s_addr + 32, hi);
        }
        ptx::tmem_st_wait();
        // O_g rescale for a raised max, once the scores and P words are no
        // longer held in registers: P_g V of this tile is issued only after
        // every thread has arrived below
        if (k > 0 && __any_sync(0xffffffffu, raise)) {
#pragma unroll 1
          for (int c = 0; c < D / 16; ++c) {
            uint32_t o[16];
            ptx::tmem_ld16(o_addr + c * 16, o);
            ptx::tmem_ld_wait();
#pragma unroll
            for (int x2 = 0; x2 < 16; ++x2) o[x2] = __float_as_uint(__uint_as_float(o[x2]) * f);
            ptx::tmem_st16(o_addr + c * 16, o);
          }
          ptx::tmem_st_wait();
        }
        // every lane has waited for its own TMEM stores; the warp's lanes
        // meet, then one lane arrives for the warp
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(&aux->p_ready[g]);
      }
      // epilogue: final O row -> the split's partial (O / l in fp16, m, l)
      bool fin = ok && !aux->abort_flag && ptx::mbar_wait(&aux->o_final, 0, wait_limit);
      if (!__all_sync(0xffffffffu, fin)) {
        timeout(aux, status);
      } else if (warp_rows) {
        ptx::tc_fence_after();
        const int split = (int)(my.j0 / keys_per_split);
        // the partial row normalised (O / l: a convex combination of V rows,
        // so |O / l| <= max |v| < 65504) in fp16, column-octet major: for
        // each 8-column octet the warp's 32 rows are 512 contiguous bytes
        uint4* dst = part_o + part_o8_index(kv, split, n_split, 0, D, M, sm_valid ? sm_R : 0);
        const size_t c8_stride = (size_t)M;
        const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll 1
        for (int c = 0; c < D / 32; ++c) {
          uint32_t o[32];
          ptx::tmem_ld32(o_addr + c * 32, o);
          ptx::tmem_ld_wait();
          if (sm_valid) {
            auto h2 = [&](int x) {
              return ptx::pack_f16x2(__uint_as_float(o[x]) * inv, __uint_as_float(o[x + 1]) * inv);
            };
#pragma unroll
            for (int x8 = 0; x8 < 4; ++x8)
              dst[(size_t)(c * 4 + x8) * c8_stride] =
                  make_uint4(h2(8 * x8), h2(8 * x8 + 2), h2(8 * x8 + 4), h2(8 * x8 + 6));
          }
        }
        if (sm_valid) {
          const size_t base = ((size_t)kv * n_split + split) * M + sm_R;
          part_ml[base * 2] = m_used;
          part_ml[base * 2 + 1] = l;
        }
      }
    }
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

int make_kv_map(CUtensorMap* map, const void* base, int Hkv, int64_t L_cap, int d,
                bool fp16 = false) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return fail(TS_ERR_CUDA, "cuTensorMapEncodeTiled is unavailable");
  cuuint64_t dims[2] = {(cuuint64_t)d, (cuuint64_t)Hkv * (cuuint64_t)L_cap};
  cuuint64_t strides[1] = {(cuuint64_t)d * 2};
  cuuint32_t box[2] = {64, (cuuint32_t)kNk};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(map, fp16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                  const_cast<void*>(base), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(TS_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
  return TS_OK;
}

}  // namespace

// Key splits per (KV head, row group): the count minimising waves x tiles per
// CTA (+ a fixed per-CTA cost), so the grid fills whole waves of the SMs.
int tc_splits(int Hkv, int n_rg, int64_t L, int nsm) {
  return verify_splits(Hkv, n_rg, 0, L, nsm);
}

// The same for the verification grid.  n_pt pair-tile row groups take one
// CTA per split; the two-stream row group takes one CTA per two consecutive
// splits of the same cut, so its CTAs read every key tile at about the time
// a pair-tile CTA reads it and the second read is an L2 hit: K and V leave
// HBM once.  (Separate cuts balanced for time were measured at 1.8 x the K/V
// bytes from HBM on the 14B shape.)  Time of a CTA in
// pair-tile tile steps: a pair-tile CTA ~ its tiles + kFixedTiles; a
// two-stream CTA ~ 2 * kTwoStep * its tiles per split + kFixedTiles, a
// two-stream step (one query tile, one key tile) costing kTwoStep of a
// pair-tile step (two query tiles).  The fixed cost of a CTA (set-up while
// its first tiles arrive, the last tile's drain and the epilogue, ~7 us)
// is about four pair-tile steps.
int64_t split_tiles(int64_t L, int n) { return ((L + n - 1) / n + kNk - 1) / kNk; }

int verify_splits(int Hkv, int n_pt, int n_two, int64_t L, int nsm) {
  constexpr double kTwoStep = 0.55;
  constexpr double kFixedTiles = 4.0;
  int64_t max_split = (L + kNk - 1) / kNk;
  if (max_split < 1) max_split = 1;
  if (max_split > 1024) max_split = 1024;
  double best_cost = 1e300;
  int best = 1;
  for (int n = 1; n <= max_split; ++n) {
    const int64_t ctas = (int64_t)Hkv * ((int64_t)n_pt * n + (int64_t)n_two * ((n + 1) / 2));
    const int64_t waves = (ctas + nsm - 1) / nsm;
    double t = 0.0;
    if (n_pt > 0) t = (double)split_tiles(L, n) + kFixedTiles;
    if (n_two > 0) t = fmax(t, 2.0 * kTwoStep * (double)split_tiles(L, n) + kFixedTiles);
    const double cost = (double)waves * t;
    if (cost < best_cost - 1e-9) {
      best_cost = cost;
      best = n;
    }
  }
  return best;
}

size_t verify_tc_smem_bytes(int d) {
  return d == 128 ? (size_t)TcLayout<128>::kBytes : (size_t)TcLayout<64>::kBytes;
}

int launch_verify_tc(const void* q, const void* k, const void* v, int64_t L, int64_t L_cap,
                     const int32_t* parents, int T, int Hq, int Hkv, int d, int n_imp,
                     int64_t keys_per_split, int n_split, int n_pt, int n_two, bool v_fp16,
                     uint4* part_o, float* part_ml, float* imp, int32_t* status,
                     cudaStream_t st) {
  CUtensorMap mk, mv;
  int rc = make_kv_map(&mk, k, Hkv, L_cap, d);
  if (rc) return rc;
  rc = make_kv_map(&mv, v, Hkv, L_cap, d, v_fp16);
  if (rc) return rc;
  const int per_head = n_pt * n_split + n_two * ((n_split + 1) / 2);
  dim3 grid(per_head, Hkv);
  auto qb = static_cast<const __nv_bfloat16*>(q);
  const long long limit = wait_limit_cycles();
  auto go = [&](auto kern, int smem) {
    // the warpgroups' register split (setmaxnreg) adds up to 128 registers
    // a thread at launch; any other count would leave the softmax
    // warpgroups waiting for registers that never come free
    cudaFuncAttributes fa{};
    if (cudaFuncGetAttributes(&fa, kern) != cudaSuccess || fa.numRegs != 128) {
      rc = fail(TS_ERR_CUDA, "verify kernel compiled to %d registers a thread; its register "
                "split needs 128", fa.numRegs);
      return;
    }
    cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    pdl_config(&cfg, attr, grid, dim3(kThreadsTc), smem, st);
    cudaLaunchKernelEx(&cfg, kern, mk, mv, qb, parents, T, Hq, Hkv, n_imp, L, L_cap,
                       keys_per_split, n_split, n_pt, limit, part_o, part_ml, imp, status);
  };
  if (d == 128)
    v_fp16 ? go(verify_tc_kernel<128, true>, TcLayout<128>::kBytes)
           : go(verify_tc_kernel<128, false>, TcLayout<128>::kBytes);
  else
    v_fp16 ? go(verify_tc_kernel<64, true>, TcLayout<64>::kBytes)
           : go(verify_tc_kernel<64, false>, TcLayout<64>::kBytes);
  if (rc) return rc;
  return launch_status("verify_tc_kernel");
}

}  // namespace ts
