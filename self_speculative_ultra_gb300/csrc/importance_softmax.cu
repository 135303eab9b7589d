// Softmax-weighted importance of the committed KV cache on the tcgen05
// tensor cores: the attention probability each cache position receives from
// the importance queries of its KV head's group.
//
// "TokenSwift: Lossless Acceleration of Ultra Long Sequence Generation",
// §3.3 Dynamic KV Cache Management: cache pairs are ranked by query-key
// scores, a GQA group's queries partitioned and their scores aggregated.
// This variant aggregates the normalised attention weights of those queries
// rather than their raw scores:
//
//   imp[kv, j] = sum_{i in last n_imp nodes, h in group kv}
//                2^(q[i,h].k[kv,j] * log2(e)/sqrt(d) - lse[i,h] * log2(e))
//
// with lse[i,h] the row's natural-log log-sum-exp from the verification
// pass (its softmax normaliser).  The normaliser is only known once the
// whole cache has been read, so this is a second pass over K (V is not read).
//
// One CTA = (key split, KV head).  The R = n_imp * G importance query rows
// are packed (row r = node T - n_imp + r / G, head kv * G + r % G) into
// shared memory once, padded to Rs rows (a multiple of 32, zero queries whose
// lse is +inf, so they add exactly 0), split into chunks of at most 256 rows.
// Per 128-key tile:
//   TMA (warp 0)      K tile into a 3-stage ring (128-byte swizzle, L2
//                     evict-first)
//   MMA (warp 1)      D[key, row] = K Q_c^T for each row chunk c (bf16,
//                     M = 128 keys, N = chunk rows, fp32 in TMEM); work items
//                     (tile, chunk) alternate between two 256-column TMEM
//                     halves, so the MMA of item n+1 runs under the epilogue
//                     of item n
//   epilogue          two sets of four warps (2..5 and 6..9), set b reading
//                     TMEM half b: one thread per key (TMEM lane) sums
//                     ex2(s * log2e/sqrt(d) - lse2[row]) over its columns,
//                     the row-wise lse2 values being shared-memory
//                     broadcasts.  With one row chunk the sets take alternate
//                     tiles; with two, set 0 takes chunk 0 and set 1 chunk 1
//                     of every tile, set 0's partial sums passing to set 1
//                     through a double-buffered shared array
// Each key of [0, L) is written by exactly one thread, so no workspace and no
// merge are needed.  Every mbarrier wait is bounded (~1 s of SM clocks); on
// expiry the CTA records TS_ERR_TIMEOUT, drains its own copies and MMAs
// (bounded), frees its TMEM and returns.
#include "importance.cuh"
#include "tc_ptx.cuh"

namespace ts {

namespace {

constexpr int kKeys = 128;               // keys per tile (MMA M)
constexpr int kStages = 3;               // K ring depth
constexpr int kThreads = 320;            // warp 0 TMA, warp 1 MMA, warps 2..9 epilogue
constexpr int kHalf = 256;               // TMEM columns per accumulator half
constexpr int kMaxChunk = 256;           // MMA N limit at M = 128
constexpr long long kWaitCycles = 1ll << 31;
constexpr float kLog2e = 1.4426950408889634f;

struct ImpAux {
  uint64_t k_full[kStages], k_empty[kStages];
  uint64_t t_full[2], t_empty[2];
  uint64_t red_full[2], red_empty[2];   // set 0 -> set 1 partial sums (two row chunks)
  uint64_t drain;
  float red[2][kKeys];
  uint32_t tmem_base;
  volatile int32_t abort_flag;
};

__host__ __device__ constexpr int imp_tile_bytes(int D) { return kKeys * D * 2; }

// dynamic shared memory: K ring | Q (Rs rows) | lse2 (Rs floats) | aux
__host__ __device__ inline size_t imp_smem_bytes(int D, int Rs) {
  return 1024 + (size_t)kStages * imp_tile_bytes(D) + (size_t)Rs * D * 2 + (size_t)Rs * 4 +
         sizeof(ImpAux);
}

// tcgen05.wait::ld with the loaded registers as operands, so that no use of
// them can be scheduled before the wait
__device__ __forceinline__ void ld_wait_keep(uint32_t (&r)[32]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]),
                 "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]),
                 "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15]), "+r"(r[16]), "+r"(r[17]),
                 "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]), "+r"(r[22]), "+r"(r[23]),
                 "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]),
                 "+r"(r[30]), "+r"(r[31])
               :
               : "memory");
}

__device__ __forceinline__ void sum_ex2_32(const uint32_t (&r)[32], const float* l2, float sl2,
                                           float& a0, float& a1, float& a2, float& a3) {
#pragma unroll
  for (int x = 0; x < 32; x += 4) {
    const float4 l = *reinterpret_cast<const float4*>(l2 + x);
    a0 += ptx::ex2(fmaf(__uint_as_float(r[x]), sl2, -l.x));
    a1 += ptx::ex2(fmaf(__uint_as_float(r[x + 1]), sl2, -l.y));
    a2 += ptx::ex2(fmaf(__uint_as_float(r[x + 2]), sl2, -l.z));
    a3 += ptx::ex2(fmaf(__uint_as_float(r[x + 3]), sl2, -l.w));
  }
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
importance_softmax_kernel(const __grid_constant__ CUtensorMap tmap_k,
                          const __nv_bfloat16* __restrict__ q, const float* __restrict__ lse, int T,
                          int Hq, int Hkv, int n_imp, int Rs, int chunk_rows, int64_t L,
                          int64_t L_cap, int64_t keys_per_split, float* __restrict__ imp,
                          int32_t* status) {
  constexpr int kTile = imp_tile_bytes(D);
  constexpr int kPanel = kKeys * 128;            // 128 keys x 64 bf16 (128-byte rows)
  constexpr int C16 = D / 8;                     // 16-byte chunks per row
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~uintptr_t(1023));
  uint8_t* sk = sm;
  uint8_t* sq = sm + kStages * kTile;
  const int panel_q = Rs * 128;                  // bytes of one 64-column panel of Q
  float* lse2 = reinterpret_cast<float*>(sq + (size_t)Rs * D * 2);
  ImpAux* aux = reinterpret_cast<ImpAux*>(lse2 + Rs);

  const int split = blockIdx.x, kv = blockIdx.y;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = Hq / Hkv, R = n_imp * G;
  const int n_chunks = Rs / chunk_rows;
  const int64_t j0 = (int64_t)split * keys_per_split;
  const int64_t j1 = min(L, j0 + keys_per_split);
  const int n_tiles = (int)((j1 - j0 + kKeys - 1) / kKeys);
  const int n_items = n_tiles * n_chunks;
  const float sl2 = kLog2e / sqrtf((float)D);
  const int n_pre = min(n_tiles, kStages);

  // ---------------------------------------------------------------- set-up
  griddep_wait();   // lse comes from the kernels before this one
  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      ptx::mbar_init(&aux->k_full[s], 1);
      ptx::mbar_init(&aux->k_empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      ptx::mbar_init(&aux->t_full[b], 1);
      ptx::mbar_init(&aux->t_empty[b], 4);     // one arrival per warp of the set reading half b
      ptx::mbar_init(&aux->red_full[b], 4);
      ptx::mbar_init(&aux->red_empty[b], 4);
    }
    ptx::mbar_init(&aux->drain, 1);
    aux->abort_flag = 0;
    ptx::fence_mbar_init();
    const uint64_t pol = ptx::l2_evict_first_policy();
    const int row0 = (int)(kv * L_cap + j0);
    for (int jt = 0; jt < n_pre; ++jt) {
      ptx::mbar_arrive_expect_tx(&aux->k_full[jt], kTile);
      for (int p = 0; p < D / 64; ++p)
        ptx::tma_load_2d(sk + jt * kTile + p * kPanel, &tmap_k, &aux->k_full[jt], p * 64,
                         row0 + jt * kKeys, pol);
    }
  }
  if (warp == 1) {
    ptx::tmem_alloc(&aux->tmem_base, 512);
    ptx::tmem_relinquish();
  }
  // importance query rows -> shared memory, 128-byte-swizzled K-major panels
  for (int e = tid; e < Rs * C16; e += kThreads) {
    const int r = e / C16, c = e % C16;
    uint4 val = make_uint4(0, 0, 0, 0);
    if (r < R) {
      const int i = T - n_imp + r / G, h = kv * G + r % G;
      val = __ldg(reinterpret_cast<const uint4*>(q + ((size_t)i * Hq + h) * D + c * 8));
    }
    const int p = c >> 3, cc = c & 7;
    *reinterpret_cast<uint4*>(sq + p * panel_q + r * 128 + ((cc ^ (r & 7)) << 4)) = val;
  }
  for (int r = tid; r < Rs; r += kThreads) {
    float v = INFINITY;
    if (r < R) {
      const int i = T - n_imp + r / G, h = kv * G + r % G;
      v = lse[(size_t)i * Hq + h] * kLog2e;
    }
    lse2[r] = v;
  }
  ptx::fence_proxy_async_smem();
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = aux->tmem_base;
  griddep_launch_dependents();

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const uint64_t pol = ptx::l2_evict_first_policy();
      const int row0 = (int)(kv * L_cap + j0);
      int jt = n_pre;
      for (; jt < n_tiles; ++jt) {
        const int s = jt % kStages;
        if (!ptx::mbar_wait(&aux->k_empty[s], (uint32_t)(jt / kStages - 1) & 1u, kWaitCycles)) {
          aux->abort_flag = 1;
          set_status(status, TS_ERR_TIMEOUT);
          break;
        }
        ptx::mbar_arrive_expect_tx(&aux->k_full[s], kTile);
        for (int p = 0; p < D / 64; ++p)
          ptx::tma_load_2d(sk + s * kTile + p * kPanel, &tmap_k, &aux->k_full[s], p * 64,
                           row0 + jt * kKeys, pol);
        if (aux->abort_flag) {
          ++jt;
          break;
        }
      }
      // every issued load must land before the CTA exits, whether or not a
      // consumer gave up waiting for it (normally these waits return at once)
      for (int t = max(0, jt - kStages); t < jt; ++t)
        ptx::mbar_wait(&aux->k_full[t % kStages], (uint32_t)(t / kStages) & 1u, kWaitCycles);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t idesc = ptx::idesc_bf16_f32(kKeys, chunk_rows, false);
      const uint64_t kd0 = ptx::sdesc_sw128(ptx::smem_u32(sk), 16, 1024);
      const uint64_t qd0 = ptx::sdesc_sw128(ptx::smem_u32(sq), 16, 1024);
      constexpr uint32_t kTile16 = kTile >> 4, kPanel16 = kPanel >> 4;
      const uint32_t qpanel16 = (uint32_t)panel_q >> 4, chunk16 = (uint32_t)(chunk_rows * 128) >> 4;
      bool ok = true;
      for (int it = 0; it < n_items && ok; ++it) {
        const int j = it / n_chunks, c = it % n_chunks, b = it & 1;
        if (c == 0 &&
            !ptx::mbar_wait(&aux->k_full[j % kStages], (uint32_t)(j / kStages) & 1u, kWaitCycles))
          ok = false;
        if (ok && it >= 2 &&
            !ptx::mbar_wait(&aux->t_empty[b], (uint32_t)(it / 2 - 1) & 1u, kWaitCycles))
          ok = false;
        if (!ok || aux->abort_flag) {
          ok = false;
          break;
        }
        ptx::tc_fence_after();
        const uint64_t a0 = kd0 + (uint64_t)((j % kStages) * kTile16);
        const uint64_t b0 = qd0 + (uint64_t)(c * chunk16);
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          // 64-element panels, 32-byte K-steps inside a panel
          const uint32_t offa = (ks >> 2) * kPanel16 + (ks & 3) * 2;
          const uint32_t offb = (ks >> 2) * qpanel16 + (ks & 3) * 2;
          ptx::mma_ss(tmem + (uint32_t)(b * kHalf), a0 + offa, b0 + offb, idesc, ks > 0 ? 1u : 0u);
        }
        ptx::mma_commit(&aux->t_full[b]);
        if (c == n_chunks - 1) ptx::mma_commit(&aux->k_empty[j % kStages]);
      }
      if (!ok) {
        aux->abort_flag = 1;
        set_status(status, TS_ERR_TIMEOUT);
      }
      ptx::mma_commit(&aux->drain);
      ptx::mbar_wait(&aux->drain, 0, kWaitCycles);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int set = (warp - 2) >> 2;             // reads TMEM half `set`: items set, set+2, ...
    const int qtr = warp & 3;                    // TMEM lane quarter of this warp
    const uint32_t lane_base = tmem + ((uint32_t)(32 * qtr) << 16) + (uint32_t)(set * kHalf);
    const int key_in_tile = 32 * qtr + lane;
    const int ng = chunk_rows / 32;
    for (int it = set; it < n_items; it += 2) {
      const int j = it / n_chunks, c = it % n_chunks;
      if (aux->abort_flag ||
          !ptx::mbar_wait(&aux->t_full[set], (uint32_t)(it / 2) & 1u, kWaitCycles)) {
        aux->abort_flag = 1;
        set_status(status, TS_ERR_TIMEOUT);
        break;
      }
      ptx::tc_fence_after();
      const float* l2 = lse2 + c * chunk_rows;
      float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
      uint32_t ra[32], rb[32];
      ptx::tmem_ld32(lane_base, ra);
      ld_wait_keep(ra);
      for (int g = 0; g < ng; g += 2) {
        if (g + 1 < ng) ptx::tmem_ld32(lane_base + (uint32_t)((g + 1) * 32), rb);
        sum_ex2_32(ra, l2 + g * 32, sl2, a0, a1, a2, a3);
        if (g + 1 < ng) {
          ld_wait_keep(rb);
          if (g + 2 < ng) ptx::tmem_ld32(lane_base + (uint32_t)((g + 2) * 32), ra);
          sum_ex2_32(rb, l2 + (g + 1) * 32, sl2, a0, a1, a2, a3);
          if (g + 2 < ng) ld_wait_keep(ra);
        }
      }
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&aux->t_empty[set]);
      float acc = (a0 + a1) + (a2 + a3);
      const int64_t key = j0 + (int64_t)j * kKeys + key_in_tile;
      if (n_chunks == 2) {
        // chunk 0 (set 0) hands its partial sums to chunk 1 (set 1)
        const int rb_ = j & 1;
        const uint32_t use = (uint32_t)(j >> 1);
        if (set == 0) {
          if (j >= 2 && !ptx::mbar_wait(&aux->red_empty[rb_], (use - 1) & 1u, kWaitCycles)) {
            aux->abort_flag = 1;
            set_status(status, TS_ERR_TIMEOUT);
            break;
          }
          aux->red[rb_][key_in_tile] = acc;
          __syncwarp();
          if (lane == 0) ptx::mbar_arrive(&aux->red_full[rb_]);
          continue;
        }
        if (!ptx::mbar_wait(&aux->red_full[rb_], use & 1u, kWaitCycles)) {
          aux->abort_flag = 1;
          set_status(status, TS_ERR_TIMEOUT);
          break;
        }
        acc += aux->red[rb_][key_in_tile];
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(&aux->red_empty[rb_]);
      }
      if (key < j1) imp[(size_t)kv * L + key] = acc;
    }
  }

  // ---------------------------------------------------------------- teardown
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, 512);
  }
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

int make_k_map(CUtensorMap* map, const void* base, int Hkv, int64_t L_cap, int d) {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult qr{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &qr) == cudaSuccess &&
        qr == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  if (!fn) return fail(TS_ERR_CUDA, "cuTensorMapEncodeTiled is unavailable");
  cuuint64_t dims[2] = {(cuuint64_t)d, (cuuint64_t)Hkv * (cuuint64_t)L_cap};
  cuuint64_t strides[1] = {(cuuint64_t)d * 2};
  cuuint32_t box[2] = {64, (cuuint32_t)kKeys};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(TS_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
  return TS_OK;
}

}  // namespace

ImpSoftmaxPlan importance_softmax_plan(int T, int Hq, int Hkv, int d, int n_imp, int64_t L) {
  ImpSoftmaxPlan p{};
  const int R = n_imp * (Hq / Hkv);
  const int n_chunks = (R + kMaxChunk - 1) / kMaxChunk;
  const int per = (R + n_chunks - 1) / n_chunks;
  p.chunk_rows = (per + 31) / 32 * 32;
  p.Rs = n_chunks * p.chunk_rows;
  // at least 120 KB, so that one CTA holds an SM (each allocates all 512
  // TMEM columns)
  p.smem = imp_smem_bytes(d, p.Rs);
  if (p.smem < 120 * 1024) p.smem = 120 * 1024;
  const int n = tc_splits(Hkv, 1, L, kGb300Sms);
  p.keys_per_split = ((L + n - 1) / n + kKeys - 1) / kKeys * kKeys;
  if (p.keys_per_split < kKeys) p.keys_per_split = kKeys;
  p.n_split = (int)((L + p.keys_per_split - 1) / p.keys_per_split);
  return p;
}

int launch_importance_softmax(const void* q, const void* k, const float* lse, int64_t L,
                              int64_t L_cap, int T, int Hq, int Hkv, int d, int n_imp, float* imp,
                              int32_t* status, cudaStream_t st) {
  if (L <= 0) return TS_OK;
  const ImpSoftmaxPlan p = importance_softmax_plan(T, Hq, Hkv, d, n_imp, L);
  CUtensorMap mk;
  int rc = make_k_map(&mk, k, Hkv, L_cap, d);
  if (rc) return rc;
  dim3 grid(p.n_split, Hkv);
  auto qb = static_cast<const __nv_bfloat16*>(q);
  auto go = [&](auto kern) {
    cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)p.smem);
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    pdl_config(&cfg, attr, grid, dim3(kThreads), p.smem, st);
    cudaLaunchKernelEx(&cfg, kern, mk, qb, lse, T, Hq, Hkv, n_imp, p.Rs, p.chunk_rows, L, L_cap,
                       p.keys_per_split, imp, status);
  };
  if (d == 128)
    go(importance_softmax_kernel<128>);
  else
    go(importance_softmax_kernel<64>);
  return launch_status("importance_softmax_kernel");
}

}  // namespace ts
