// Dynamic partial KV cache: exact top-B selection + ordered gather.
//
// "TokenSwift: Lossless Acceleration of Ultra Long Sequence Generation",
// §3.3 Dynamic KV Cache Management: a fixed budget that always keeps the
// initial |S| pairs and replaces the less important ones; §3.1: the partial
// cache is what drafting attends to.
//
// The ranking (imp desc, position asc) is a total order, so the kept
// candidates are exactly those ranked at or above the B-th one, (tau, j_tie):
//   keep(j) = key(j) > tau  or  (key(j) == tau and j <= j_tie),
// with key() the order-preserving uint32 image of the fp32 score.  Stage 1
// (one CTA per KV head) finds tau by a 4-pass 8-bit radix select over the
// candidates, j_tie by an ordered count of the positions whose key equals
// tau, and the number of kept positions in every chunk of the cache.  Stage 2
// (one CTA per chunk and KV head) re-evaluates keep(), compacts the kept
// positions in ascending order, and copies their K/V rows with 16-byte loads.
#include "ts_common.cuh"

namespace ts {

namespace {

constexpr int kSelThreads = 1024;
constexpr int kChunk = 1024;        // positions per stage-2 CTA
constexpr int kGatherThreads = 256;

struct SelectState {
  uint32_t tau;        // key of the B-th ranked candidate
  int32_t j_tie;       // largest kept position among those with key == tau
  int32_t select_all;  // L <= S+B+R: keep everything
  int32_t pad;
};

__device__ __forceinline__ bool keep_pos(const float* __restrict__ imp_h, int64_t j, int64_t L,
                                         int S, int R, const SelectState& st) {
  if (st.select_all || j < S || j >= L - R) return true;
  uint32_t key = float_key(imp_h[j]);
  return key > st.tau || (key == st.tau && j <= st.j_tie);
}

__device__ int block_excl_scan(int x, int* warp_buf, int* total) {
  // exclusive prefix over the block (blockDim.x multiple of 32, <= 1024)
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  int incl = x;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) warp_buf[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int w = lane < nw ? warp_buf[lane] : 0;
    int wi = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int y = __shfl_up_sync(0xffffffffu, wi, o);
      if (lane >= o) wi += y;
    }
    if (lane < nw) warp_buf[lane] = wi - w;
    if (lane == 31) *total = wi;
  }
  __syncthreads();
  int r = warp_buf[warp] + incl - x;
  __syncthreads();
  return r;
}

__global__ void __launch_bounds__(kSelThreads)
select_threshold(const float* __restrict__ imp, int64_t L, int B, int S, int R, int64_t n_chunks,
                 SelectState* __restrict__ state, int32_t* __restrict__ chunk_off) {
  const int kv = blockIdx.x, tid = threadIdx.x;
  const float* imp_h = imp + (size_t)kv * L;
  __shared__ int hist[256];
  __shared__ uint32_t s_prefix, s_mask;
  __shared__ int s_krem;
  __shared__ int warp_buf[32];
  __shared__ int s_total;
  __shared__ SelectState st;

  if (tid == 0) {
    st.select_all = (L <= (int64_t)S + B + R) ? 1 : 0;
    st.tau = 0;
    st.j_tie = -1;
    s_prefix = 0;
    s_mask = 0;
    s_krem = B;
  }
  __syncthreads();
  const int64_t lo = S, hi = L - R;
  if (!st.select_all && B > 0) {
    for (int pass = 0; pass < 4; ++pass) {
      const int shift = 24 - 8 * pass;
      for (int b = tid; b < 256; b += kSelThreads) hist[b] = 0;
      __syncthreads();
      const uint32_t pre = s_prefix, msk = s_mask;
      for (int64_t j = lo + tid; j < hi; j += kSelThreads) {
        uint32_t key = float_key(imp_h[j]);
        if ((key & msk) == pre) atomicAdd(&hist[(key >> shift) & 255], 1);
      }
      __syncthreads();
      if (tid == 0) {
        int krem = s_krem, cum = 0, b = 255;
        for (; b > 0; --b) {
          if (cum + hist[b] >= krem) break;
          cum += hist[b];
        }
        s_krem = krem - cum;
        s_prefix = pre | ((uint32_t)b << shift);
        s_mask = msk | (255u << shift);
      }
      __syncthreads();
    }
    // j_tie: the s_krem-th candidate (in position order) whose key == tau
    const uint32_t tau = s_prefix;
    const int need = s_krem;
    const int64_t n = hi - lo;
    const int64_t per = (n + kSelThreads - 1) / kSelThreads;
    const int64_t a = lo + tid * per, e = min(hi, a + per);
    int cnt = 0;
    for (int64_t j = a; j < e; ++j) cnt += float_key(imp_h[j]) == tau;
    int before = block_excl_scan(cnt, warp_buf, &s_total);
    if (before < need && before + cnt >= need) {
      int c = before;
      for (int64_t j = a; j < e; ++j) {
        if (float_key(imp_h[j]) == tau && ++c == need) {
          st.j_tie = (int32_t)j;
          break;
        }
      }
    }
    if (tid == 0) st.tau = tau;
    __syncthreads();
  } else if (!st.select_all) {
    // B == 0: keep only sinks and recent
    if (tid == 0) {
      st.tau = 0xFFFFFFFFu;
      st.j_tie = -1;
    }
    __syncthreads();
  }
  // kept positions per chunk, then exclusive offsets
  SelectState s = st;
  int32_t* off = chunk_off + (size_t)kv * (n_chunks + 1);
  const int warp = tid >> 5, lane = tid & 31;
  for (int64_t c = warp; c < n_chunks; c += kSelThreads / 32) {
    int cnt = 0;
    const int64_t a = c * kChunk, e = min(L, a + kChunk);
    for (int64_t j = a + lane; j < e; j += 32) cnt += keep_pos(imp_h, j, L, S, R, s);
    cnt = warp_sum_int(cnt);
    if (lane == 0) off[c] = cnt;
  }
  __syncthreads();
  if (tid == 0) {
    int run = 0;
    for (int64_t c = 0; c < n_chunks; ++c) {
      int x = off[c];
      off[c] = run;
      run += x;
    }
    off[n_chunks] = run;
    state[kv] = s;
  }
}

template <int D>
__global__ void __launch_bounds__(kGatherThreads)
select_gather(const float* __restrict__ imp, const __nv_bfloat16* __restrict__ k,
              const __nv_bfloat16* __restrict__ v, int64_t L, int64_t L_cap, int S, int R,
              int64_t N, int64_t n_chunks, const SelectState* __restrict__ state,
              const int32_t* __restrict__ chunk_off, int32_t* __restrict__ idx,
              __nv_bfloat16* __restrict__ kd, __nv_bfloat16* __restrict__ vd, int32_t* status) {
  const int64_t c = blockIdx.x;
  const int kv = blockIdx.y, tid = threadIdx.x;
  const float* imp_h = imp + (size_t)kv * L;
  const SelectState s = state[kv];
  const int32_t* off = chunk_off + (size_t)kv * (n_chunks + 1);
  __shared__ int warp_buf[32];
  __shared__ int s_total;
  __shared__ int32_t sel[kChunk];
  constexpr int PER = kChunk / kGatherThreads;   // positions per thread
  const int64_t a = c * kChunk + tid * PER;
  int flags = 0, cnt = 0;
#pragma unroll
  for (int x = 0; x < PER; ++x) {
    int64_t j = a + x;
    if (j < L && keep_pos(imp_h, j, L, S, R, s)) {
      flags |= 1 << x;
      ++cnt;
    }
  }
  int pos = block_excl_scan(cnt, warp_buf, &s_total);
  const int base = off[c];
  if (tid == 0 && base + s_total > N) set_status(status, TS_ERR_INVALID_ARG);
#pragma unroll
  for (int x = 0; x < PER; ++x) {
    if (flags & (1 << x)) {
      int64_t out = base + pos;
      if (out < N) idx[(size_t)kv * N + out] = (int32_t)(a + x);
      sel[pos] = (int32_t)(a + x);
      ++pos;
    }
  }
  __syncthreads();
  const int total = s_total;
  constexpr int V16 = D / 8;   // 16-byte vectors per row
  const uint4* ksrc = reinterpret_cast<const uint4*>(k + (size_t)kv * L_cap * D);
  const uint4* vsrc = reinterpret_cast<const uint4*>(v + (size_t)kv * L_cap * D);
  uint4* kdst = reinterpret_cast<uint4*>(kd + (size_t)kv * N * D);
  uint4* vdst = reinterpret_cast<uint4*>(vd + (size_t)kv * N * D);
  for (int e = tid; e < total * V16; e += kGatherThreads) {
    int r = e / V16, x = e % V16;
    int64_t out = base + r;
    if (out >= N) continue;
    int64_t j = sel[r];
    kdst[out * V16 + x] = ksrc[j * V16 + x];
    vdst[out * V16 + x] = vsrc[j * V16 + x];
  }
}

}  // namespace

SelectPlan select_plan(int Hkv, int64_t L) {
  SelectPlan p{};
  p.chunk = kChunk;
  p.n_chunks = (L + kChunk - 1) / kChunk;
  size_t st = align_up((size_t)Hkv * sizeof(SelectState), 256);
  size_t off = align_up((size_t)Hkv * (p.n_chunks + 1) * sizeof(int32_t), 256);
  p.ws_bytes = st + off;
  return p;
}

int launch_select_gather(const float* imp, const void* k, const void* v, int64_t L,
                         int64_t L_cap, int Hkv, int d, int B, int S, int R, int32_t* idx,
                         void* kd, void* vd, int64_t N, void* ws, int32_t* status,
                         cudaStream_t st) {
  SelectPlan p = select_plan(Hkv, L);
  SelectState* state = static_cast<SelectState*>(ws);
  int32_t* off = reinterpret_cast<int32_t*>(static_cast<char*>(ws) +
                                            align_up((size_t)Hkv * sizeof(SelectState), 256));
  select_threshold<<<Hkv, kSelThreads, 0, st>>>(imp, L, B, S, R, p.n_chunks, state, off);
  int rc = launch_status("select_threshold");
  if (rc) return rc;
  dim3 grid((unsigned)p.n_chunks, Hkv);
  auto kb = static_cast<const __nv_bfloat16*>(k);
  auto vb = static_cast<const __nv_bfloat16*>(v);
  if (d == 128)
    select_gather<128><<<grid, kGatherThreads, 0, st>>>(imp, kb, vb, L, L_cap, S, R, N, p.n_chunks,
                                                        state, off, idx,
                                                        static_cast<__nv_bfloat16*>(kd),
                                                        static_cast<__nv_bfloat16*>(vd), status);
  else
    select_gather<64><<<grid, kGatherThreads, 0, st>>>(imp, kb, vb, L, L_cap, S, R, N, p.n_chunks,
                                                       state, off, idx,
                                                       static_cast<__nv_bfloat16*>(kd),
                                                       static_cast<__nv_bfloat16*>(vd), status);
  return launch_status("select_gather");
}

}  // namespace ts
