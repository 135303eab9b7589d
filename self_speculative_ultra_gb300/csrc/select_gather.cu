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
// with key() the order-preserving uint32 image of the fp32 score.  Three
// kernels, each over (chunk of positions, KV head, layer), the last CTA of a
// (layer, head) finishing its stage (atomic ticket, no waiting):
//   select_hist     12-bit histogram of the candidate keys [S, L-R);
//                   last CTA: the bucket b holding the B-th best key
//   select_collect  count keys above bucket b per chunk, append the keys of
//                   bucket b to a list; last CTA: radix-select (tau, j_tie)
//                   inside the list, then kept positions per chunk and their
//                   exclusive offsets
//   select_gather   re-evaluate keep(), compact the kept positions in
//                   ascending order, copy their K/V rows with 16-byte loads
#include <mutex>

#include "refresh.cuh"
#include "ts_common.cuh"

namespace ts {

namespace {

constexpr int kChunk = 2048;        // positions per gather CTA (and per offset)
constexpr int kScan = 8192;         // positions per histogram / collect CTA
constexpr int kPerScan = kScan / kChunk;
constexpr int kThreads = 256;
constexpr int kHistBits = 12;
constexpr int kBins = 1 << kHistBits;

struct SelectState {
  uint32_t tau;        // key of the B-th ranked candidate
  int32_t j_tie;       // largest kept position among those with key == tau
  int32_t select_all;  // L <= S+B+R: keep everything
  int32_t bucket;      // top-12-bit bucket of tau
  int32_t above;       // candidates in buckets above `bucket`
  int32_t need;        // candidates to take from `bucket`
  int32_t pad[2];
};

struct Counters {
  uint32_t hist_ticket, collect_ticket, n_list, pad;
};

struct Ws {
  SelectState* state;   // [Hkv]
  Counters* cnt;        // [Hkv]
  uint32_t* hist;       // [Hkv][kBins]
  int32_t* gt;          // [Hkv][n_chunks]
  int32_t* off;         // [Hkv][n_chunks + 1]
  uint2* list;          // [Hkv][L]  (key, position)
  size_t zero_bytes;    // prefix (counters + histograms) zeroed per call
};

__host__ __device__ inline size_t a256(size_t x) { return (x + 255) / 256 * 256; }

__host__ __device__ inline Ws carve(void* base, int Hkv, int64_t L, int64_t n_chunks) {
  Ws w;
  char* p = static_cast<char*>(base);
  size_t o = 0;
  w.cnt = reinterpret_cast<Counters*>(p + o);
  o += a256((size_t)Hkv * sizeof(Counters));
  w.hist = reinterpret_cast<uint32_t*>(p + o);
  o += a256((size_t)Hkv * kBins * sizeof(uint32_t));
  w.zero_bytes = o;
  w.state = reinterpret_cast<SelectState*>(p + o);
  o += a256((size_t)Hkv * sizeof(SelectState));
  w.gt = reinterpret_cast<int32_t*>(p + o);
  o += a256((size_t)Hkv * n_chunks * sizeof(int32_t));
  w.off = reinterpret_cast<int32_t*>(p + o);
  o += a256((size_t)Hkv * (n_chunks + 1) * sizeof(int32_t));
  w.list = reinterpret_cast<uint2*>(p + o);
  return w;
}

__host__ inline size_t ws_total(int Hkv, int64_t L, int64_t n_chunks) {
  size_t o = a256((size_t)Hkv * sizeof(Counters)) + a256((size_t)Hkv * kBins * sizeof(uint32_t)) +
             a256((size_t)Hkv * sizeof(SelectState)) +
             a256((size_t)Hkv * n_chunks * sizeof(int32_t)) +
             a256((size_t)Hkv * (n_chunks + 1) * sizeof(int32_t)) +
             a256((size_t)Hkv * (L > 0 ? L : 1) * sizeof(uint2));
  return o;
}

// Incremental refresh workspace (used by select_collect when it also counts
// the newly selected positions, and by the refresh kernels below).
struct RefreshWs {
  uint32_t* bits;      // [heads][W32]
  uint32_t* ticket;    // [heads]
  int32_t* n_freed;    // [heads]
  int32_t* cnt;        // [heads][n_chunks]
  int32_t* off;        // [heads][n_chunks + 1]
  int32_t* freed;      // [heads][N_cap]
  int64_t w32;         // bitmap words per head
  size_t zero_bytes;   // bits + tickets, zeroed per call
};

__host__ __device__ inline RefreshWs carve_refresh(void* base, int HH, int64_t L, int64_t n_chunks,
                                                   int64_t N_cap) {
  RefreshWs r;
  char* p = static_cast<char*>(base);
  size_t o = 0;
  r.w32 = (L + 31) / 32 > 0 ? (L + 31) / 32 : 1;
  r.bits = reinterpret_cast<uint32_t*>(p + o);
  o += a256((size_t)HH * r.w32 * sizeof(uint32_t));
  r.ticket = reinterpret_cast<uint32_t*>(p + o);
  o += a256((size_t)HH * sizeof(uint32_t));
  r.zero_bytes = o;
  r.n_freed = reinterpret_cast<int32_t*>(p + o);
  o += a256((size_t)HH * sizeof(int32_t));
  r.cnt = reinterpret_cast<int32_t*>(p + o);
  o += a256((size_t)HH * n_chunks * sizeof(int32_t));
  r.off = reinterpret_cast<int32_t*>(p + o);
  o += a256((size_t)HH * (n_chunks + 1) * sizeof(int32_t));
  r.freed = reinterpret_cast<int32_t*>(p + o);
  return r;
}

__host__ inline size_t refresh_area_bytes(int HH, int64_t L, int64_t n_chunks, int64_t N_cap) {
  const int64_t w32 = (L + 31) / 32 > 0 ? (L + 31) / 32 : 1;
  return a256((size_t)HH * w32 * sizeof(uint32_t)) + a256((size_t)HH * sizeof(uint32_t)) +
         a256((size_t)HH * sizeof(int32_t)) + a256((size_t)HH * n_chunks * sizeof(int32_t)) +
         a256((size_t)HH * (n_chunks + 1) * sizeof(int32_t)) +
         a256((size_t)HH * (N_cap > 0 ? N_cap : 1) * sizeof(int32_t));
}

__device__ __forceinline__ bool bit_of(const uint32_t* bits, int64_t j) {
  return (bits[j >> 5] >> (j & 31)) & 1u;
}

// Per-layer tensors: device arrays of per-layer pointers (batched call) or,
// when those are null, the single layer's pointers.
struct Layers {
  const float* const* imp;
  const __nv_bfloat16* const* k;
  const __nv_bfloat16* const* v;
  int32_t* const* idx;
  __nv_bfloat16* const* kd;
  __nv_bfloat16* const* vd;
  const float* imp1;
  const __nv_bfloat16* k1;
  const __nv_bfloat16* v1;
  int32_t* idx1;
  __nv_bfloat16* kd1;
  __nv_bfloat16* vd1;
};
__device__ __forceinline__ const float* imp_of(const Layers& P, int l) { return P.imp ? P.imp[l] : P.imp1; }

__device__ __forceinline__ bool keep_pos(const float* __restrict__ imp_h, int64_t j, int64_t L,
                                         int S, int R, const SelectState& st) {
  if (st.select_all || j < S || j >= L - R) return true;
  uint32_t key = float_key(imp_h[j]);
  return key > st.tau || (key == st.tau && j <= st.j_tie);
}

// Visit positions [lo, hi) of one importance row: f(j, imp[j], valid) is
// called the same number of times by every lane (valid = false past the
// end), so f may use warp votes.  The aligned interior is read as float4s,
// four per thread in flight.
template <typename F>
__device__ __forceinline__ void for_each_pos(const float* __restrict__ imp_h, int64_t lo,
                                             int64_t hi, F f) {
  const int tid = threadIdx.x, nthr = blockDim.x;
  int64_t vlo = hi, vhi = hi;
  if ((reinterpret_cast<uintptr_t>(imp_h) & 15) == 0 && lo < hi) {
    vlo = imin64(hi, (lo + 3) & ~int64_t(3));
    vhi = imax64(vlo, hi & ~int64_t(3));
  }
  auto scalar = [&](int64_t a, int64_t b) {
    for (int64_t j0 = a; j0 < b; j0 += nthr) {
      const int64_t j = j0 + tid;
      const bool ok = j < b;
      f(j, ok ? imp_h[j] : 0.f, ok);
    }
  };
  scalar(lo, vlo);
  const float4* p4 = reinterpret_cast<const float4*>(imp_h) + vlo / 4;
  const int64_t nq = (vhi - vlo) / 4;
  for (int64_t q0 = 0; q0 < nq; q0 += 4 * nthr) {
    float4 v[4];
    bool ok[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int64_t q = q0 + k * nthr + tid;
      ok[k] = q < nq;
      v[k] = ok[k] ? __ldg(p4 + q) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int64_t j = vlo + 4 * (q0 + k * nthr + tid);
      f(j, v[k].x, ok[k]);
      f(j + 1, v[k].y, ok[k]);
      f(j + 2, v[k].z, ok[k]);
      f(j + 3, v[k].w, ok[k]);
    }
  }
  scalar(vhi, hi);
}

// exclusive prefix over the block (blockDim.x a multiple of 32)
__device__ int block_excl_scan(int x, int* warp_buf, int* total) {
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

// Block-parallel bucket search over nb buckets (nb a multiple of blockDim):
// thread t takes a run of nb/blockDim consecutive buckets in scan order
// (descending bucket index if `desc`), finds the bucket where the running
// count first reaches `need`, and publishes it with the count before it.
__device__ void find_bucket(const uint32_t* cnt, int nb, int need, bool desc, int* warp_buf,
                           int* s_total, int* s_b, int* s_before) {
  const int per = nb / blockDim.x, t = threadIdx.x;
  int mine = 0;
  for (int x = 0; x < per; ++x) {
    const int r = t * per + x;
    mine += (int)cnt[desc ? nb - 1 - r : r];
  }
  const int before = block_excl_scan(mine, warp_buf, s_total);
  if (mine > 0 && before < need && before + mine >= need) {
    int cum = before;
    for (int x = 0; x < per; ++x) {
      const int r = t * per + x, b = desc ? nb - 1 - r : r;
      const int c = (int)cnt[b];
      if (cum + c >= need) {
        *s_b = b;
        *s_before = cum;
        break;
      }
      cum += c;
    }
  }
  __syncthreads();
}

// Ticket taken by every CTA of a head once its writes are done; true in the
// last CTA to arrive (which then sees all of them).
__device__ bool last_of_head(uint32_t* ticket, uint32_t n, int* s_flag) {
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    *s_flag = (atomicAdd(ticket, 1u) == n - 1) ? 1 : 0;
  }
  __syncthreads();
  if (*s_flag) __threadfence();
  return *s_flag != 0;
}

__global__ void __launch_bounds__(kThreads)
select_hist(Layers P, int64_t L, int B, int S, int R, int64_t n_chunks, Ws w) {
  const int kv = blockIdx.y, tid = threadIdx.x, layer = blockIdx.z;
  const int hh = layer * gridDim.y + kv;   // (layer, KV head) slot in the workspace
  const int64_t c = blockIdx.x;
  const float* imp_h = imp_of(P, layer) + (size_t)kv * L;
  __shared__ uint32_t h[kBins];
  __shared__ int warp_buf[32], s_total, s_last;
  __shared__ int s_b, s_above;
  const bool all = L <= (int64_t)S + B + R;
  if (!all && B > 0) {
    for (int b = tid; b < kBins; b += kThreads) h[b] = 0;
    __syncthreads();
    const int64_t lo = imax64(S, c * kScan), hi = imin64(L - R, (c + 1) * kScan);
    for_each_pos(imp_h, lo, hi, [&](int64_t, float x, bool ok) {
      if (ok) atomicAdd(&h[float_key(x) >> (32 - kHistBits)], 1u);
    });
    __syncthreads();
    uint32_t* gh = w.hist + (size_t)hh * kBins;
    for (int b = tid; b < kBins; b += kThreads)
      if (h[b]) atomicAdd(&gh[b], h[b]);
  }
  if (!last_of_head(&w.cnt[hh].hist_ticket, (uint32_t)gridDim.x, &s_last)) return;
  // last CTA of this head: find the bucket of the B-th best key
  SelectState st{};
  st.select_all = all ? 1 : 0;
  st.tau = 0xFFFFFFFFu;   // B == 0: nothing beyond sinks and recent
  st.j_tie = -1;
  st.bucket = -1;
  if (!all && B > 0) {
    volatile uint32_t* gh = w.hist + (size_t)hh * kBins;
    // thread t owns buckets [kBins-16(t+1), kBins-16t), highest first
    constexpr int per = kBins / kThreads;
    const int top = kBins - 1 - tid * per;
    int mine = 0;
    for (int x = 0; x < per; ++x) mine += (int)gh[top - x];
    const int before = block_excl_scan(mine, warp_buf, &s_total);
    if (before < B && before + mine >= B) {
      int cum = before;
      for (int x = 0; x < per; ++x) {
        const int cnt = (int)gh[top - x];
        if (cum + cnt >= B) {
          s_b = top - x;
          s_above = cum;
          break;
        }
        cum += cnt;
      }
    }
    __syncthreads();
    st.bucket = s_b;
    st.above = s_above;
    st.need = B - s_above;
  }
  if (tid == 0) w.state[hh] = st;
}

// With r.bits set (the incremental refresh), the same pass also counts, per
// gather chunk, the selected positions missing from the previous slots'
// bitmap, and the last CTA of a head lists the freed slots and turns the
// counts into the refresh offsets (the importance rows are not read again).
__global__ void __launch_bounds__(kThreads, 4)
select_collect(Layers P, int64_t L, int S, int R, int64_t n_chunks, Ws w, RefreshWs r,
               int64_t N_prev, int64_t N_new, int64_t N_cap, int32_t* status) {
  const int kv = blockIdx.y, tid = threadIdx.x, lane = tid & 31, nthr = blockDim.x;
  const int layer = blockIdx.z, hh = layer * gridDim.y + kv;
  const int64_t c = blockIdx.x;
  const float* imp_h = imp_of(P, layer) + (size_t)kv * L;
  __shared__ int warp_buf[32], s_total, s_last;
  __shared__ uint32_t s_cnt[1024];
  __shared__ int s_gt[kPerScan];
  // bucket members gathered per warp in its own region of s_list (a
  // warp-uniform count, no atomic per vote), then appended to the head's
  // list with one global reservation per CTA
  constexpr int kListBuf = 2048;
  constexpr int kWarps = kThreads / 32, kWarpCap = kListBuf / kWarps;
  static_assert(kPerScan == 4, "the above-bucket counters are four registers");
  __shared__ uint2 s_list[kListBuf];
  __shared__ int s_wn[kWarps], s_gbase, s_gn[kPerScan];
  const SelectState st0 = w.state[hh];
  const bool work = !st0.select_all && st0.bucket >= 0;
  uint2* list = w.list + (size_t)hh * L;
  const uint32_t* rbits = r.bits ? r.bits + (size_t)hh * r.w32 : nullptr;
  if (work) {
    const uint32_t b = (uint32_t)st0.bucket;
    const int warp = tid >> 5;
    if (tid < kPerScan) {
      s_gt[tid] = 0;
      s_gn[tid] = 0;
    }
    __syncthreads();
    const int64_t lo = imax64(S, c * kScan), hi = imin64(L - R, (c + 1) * kScan);
    // keys above bucket b, counted per gather chunk in registers (and, for
    // the refresh, those missing from the previous slots)
    int g0 = 0, g1 = 0, g2 = 0, g3 = 0, n0 = 0, n1 = 0, n2 = 0, n3 = 0;
    uint2* wl = s_list + warp * kWarpCap;
    int wn = 0;   // bucket members this warp found (the same in every lane)
    for_each_pos(imp_h, lo, hi, [&](int64_t j, float x, bool ok) {
      const uint32_t key = ok ? float_key(x) : 0u, bk = key >> (32 - kHistBits);
      if (ok && bk > b) {
        const int ci = (int)(j / kChunk - c * kPerScan);
        g0 += ci == 0;
        g1 += ci == 1;
        g2 += ci == 2;
        g3 += ci == 3;
        if (rbits && !bit_of(rbits, j)) {
          n0 += ci == 0;
          n1 += ci == 1;
          n2 += ci == 2;
          n3 += ci == 3;
        }
      }
      const bool eq = ok && bk == b;
      const unsigned m = __ballot_sync(0xffffffffu, eq);
      if (m) {
        const int slot = wn + __popc(m & ((1u << lane) - 1));
        if (eq) {
          if (slot < kWarpCap)
            wl[slot] = make_uint2(key, (uint32_t)j);
          else   // the warp's region is full: straight to the head's list
            list[atomicAdd(&w.cnt[hh].n_list, 1u)] = make_uint2(key, (uint32_t)j);
        }
        wn += __popc(m);
      }
    });
    auto warp_sum = [](int v) {
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
      return v;
    };
    g0 = warp_sum(g0);
    g1 = warp_sum(g1);
    g2 = warp_sum(g2);
    g3 = warp_sum(g3);
    if (rbits) {
      n0 = warp_sum(n0);
      n1 = warp_sum(n1);
      n2 = warp_sum(n2);
      n3 = warp_sum(n3);
    }
    if (lane == 0) {
      if (g0) atomicAdd(&s_gt[0], g0);
      if (g1) atomicAdd(&s_gt[1], g1);
      if (g2) atomicAdd(&s_gt[2], g2);
      if (g3) atomicAdd(&s_gt[3], g3);
      if (n0) atomicAdd(&s_gn[0], n0);
      if (n1) atomicAdd(&s_gn[1], n1);
      if (n2) atomicAdd(&s_gn[2], n2);
      if (n3) atomicAdd(&s_gn[3], n3);
      s_wn[warp] = min(wn, kWarpCap);
    }
    __syncthreads();
    if (tid == 0) {
      int tot = 0;
      for (int x = 0; x < kWarps; ++x) tot += s_wn[x];
      s_gbase = tot ? (int)atomicAdd(&w.cnt[hh].n_list, (uint32_t)tot) : 0;
    }
    __syncthreads();
    {
      // warp x's entries go after those of warps 0..x-1
      int off = s_gbase;
      for (int x = 0; x < warp; ++x) off += s_wn[x];
      for (int e = lane; e < s_wn[warp]; e += 32) list[off + e] = wl[e];
    }
    __syncthreads();
    if (tid < kPerScan && c * kPerScan + tid < n_chunks) {
      w.gt[(size_t)hh * n_chunks + c * kPerScan + tid] = s_gt[tid];
      if (rbits) r.cnt[(size_t)hh * n_chunks + c * kPerScan + tid] = s_gn[tid];
    }
  }
  if (!last_of_head(&w.cnt[hh].collect_ticket, (uint32_t)gridDim.x, &s_last)) return;

  // ---- last CTA of this head: (tau, j_tie) inside bucket b, then offsets
  SelectState st = st0;
  __shared__ uint32_t s_new[1024];   // refresh: new kept positions per gather chunk
  for (int x = tid; x < 1024; x += nthr) {
    s_cnt[x] = 0;
    s_new[x] = 0;
  }
  __syncthreads();
  __shared__ int s_b, s_before;
  if (work) {
    const uint32_t n = *(volatile uint32_t*)&w.cnt[hh].n_list;
    // the head's bucket members, staged in shared memory when they fit
    const bool staged = n <= (uint32_t)kListBuf;
    if (staged)
      for (uint32_t e = tid; e < n; e += nthr) s_list[e] = __ldcg(&list[e]);
    auto member = [&](uint32_t e) { return staged ? s_list[e] : __ldcg(&list[e]); };
    uint32_t pre = (uint32_t)st.bucket << (32 - kHistBits);
    uint32_t msk = 0xFFFFFFFFu << (32 - kHistBits);
    int need = st.need;
    int n_eq = -1;
    // the remaining 20 key bits, two 10-bit levels, largest keys first
    for (int lvl = 0; lvl < 2; ++lvl) {
      const int shift = 10 - 10 * lvl;
      __syncthreads();
      for (uint32_t e = tid; e < n; e += nthr) {
        const uint32_t key = member(e).x;
        if ((key & msk) == pre) atomicAdd(&s_cnt[(key >> shift) & 1023u], 1u);
      }
      __syncthreads();
      find_bucket(s_cnt, 1024, need, true, warp_buf, &s_total, &s_b, &s_before);
      need -= s_before;
      pre |= (uint32_t)s_b << shift;
      msk |= 1023u << shift;
      // after the last level the bucket holds exactly the members whose key
      // equals tau
      if (lvl == 1) n_eq = (int)s_cnt[s_b];
      __syncthreads();
      for (int x = tid; x < 1024; x += nthr) s_cnt[x] = 0;
    }
    const uint32_t tau = pre;
    // the need-th smallest position among keys == tau: four 8-bit levels,
    // unless every member with key tau is kept (no tie at the cut)
    uint32_t ppre = n_eq == need ? 0x7FFFFFFFu : 0u, pmsk = 0;
    for (int lvl = 0; lvl < 4 && n_eq != need; ++lvl) {
      const int shift = 24 - 8 * lvl;
      __syncthreads();
      for (uint32_t e = tid; e < n; e += nthr) {
        const uint2 v = member(e);
        if (v.x == tau && (v.y & pmsk) == ppre) atomicAdd(&s_cnt[(v.y >> shift) & 255u], 1u);
      }
      __syncthreads();
      find_bucket(s_cnt, 256, need, false, warp_buf, &s_total, &s_b, &s_before);
      need -= s_before;
      ppre |= (uint32_t)s_b << shift;
      pmsk |= 255u << shift;
      for (int x = tid; x < 1024; x += nthr) s_cnt[x] = 0;
    }
    st.tau = tau;
    st.j_tie = (int32_t)ppre;
    __syncthreads();
    // kept positions of bucket b per chunk (n_chunks <= 1024)
    for (uint32_t e = tid; e < n; e += nthr) {
      const uint2 v = member(e);
      if (v.x > tau || (v.x == tau && (int32_t)v.y <= st.j_tie)) {
        atomicAdd(&s_cnt[v.y / kChunk], 1u);
        if (rbits && !bit_of(rbits, v.y)) atomicAdd(&s_new[v.y / kChunk], 1u);
      }
    }
  }
  __syncthreads();
  // offsets: forced (sinks, recent) + above-bucket + bucket picks; thread t
  // takes gather chunks [4t, 4t+4)
  int cnts[4], mine = 0;
#pragma unroll
  for (int x = 0; x < 4; ++x) {
    const int64_t ch = (int64_t)tid * 4 + x;
    int cnt = 0;
    if (ch < n_chunks) {
      const int64_t a = ch * kChunk, e = imin64(L, a + kChunk);
      if (st.select_all) {
        cnt = (int)(e - a);
      } else {
        const int64_t f1 = imax64(0, imin64(e, S) - a);
        const int64_t f2 = imax64(0, e - imax64(a, L - R));
        cnt = (int)(f1 + f2);
        if (work) cnt += __ldcg(&w.gt[(size_t)hh * n_chunks + ch]) + (int)s_cnt[ch];
      }
    }
    cnts[x] = cnt;
    mine += cnt;
  }
  int before = block_excl_scan(mine, warp_buf, &s_total);
  int32_t* off = w.off + (size_t)hh * (n_chunks + 1);
#pragma unroll
  for (int x = 0; x < 4; ++x) {
    const int64_t ch = (int64_t)tid * 4 + x;
    if (ch < n_chunks) off[ch] = before;
    before += cnts[x];
  }
  if (tid == 0) {
    off[n_chunks] = s_total;
    w.state[hh] = st;
  }
  if (!rbits) return;

  // ---- refresh: new kept positions per chunk (the scan's above-bucket
  // part, the bucket picks above, the sinks and the recent window, or with
  // everything kept the positions missing from the bitmap), their offsets,
  // and the previous slots whose position is no longer kept
  if (st.select_all) {
    for (int64_t wi = tid; wi < (L + 31) / 32; wi += nthr) {
      const int64_t rem = L - wi * 32;
      const uint32_t valid = rem >= 32 ? 0xFFFFFFFFu : ((1u << rem) - 1u);
      const int cnew = __popc(~rbits[wi] & valid);
      if (cnew) atomicAdd(&s_new[(wi * 32) / kChunk], (uint32_t)cnew);
    }
  } else {
    // sinks [0, S) and the recent window [L-R, L) (disjoint here, as L > S+B+R)
    for (int64_t x = tid; x < (int64_t)S + R; x += nthr) {
      const int64_t j = x < S ? x : L - R + (x - S);
      if (j >= 0 && j < L && !bit_of(rbits, j)) atomicAdd(&s_new[j / kChunk], 1u);
    }
  }
  __syncthreads();
  int ncnt[4], nmine = 0;
#pragma unroll
  for (int x = 0; x < 4; ++x) {
    const int64_t ch = (int64_t)tid * 4 + x;
    int cnt = 0;
    if (ch < n_chunks) {
      cnt = (int)s_new[ch];
      if (work) cnt += __ldcg(&r.cnt[(size_t)hh * n_chunks + ch]);
    }
    ncnt[x] = cnt;
    nmine += cnt;
  }
  int nbefore = block_excl_scan(nmine, warp_buf, &s_total);
  int32_t* roff = r.off + (size_t)hh * (n_chunks + 1);
#pragma unroll
  for (int x = 0; x < 4; ++x) {
    const int64_t ch = (int64_t)tid * 4 + x;
    if (ch < n_chunks) roff[ch] = nbefore;
    nbefore += ncnt[x];
  }
  const int n_new_total = s_total;
  // freed slots: their position is no longer selected (or was invalid)
  const int32_t* idx = (P.idx ? P.idx[layer] : P.idx1) + (size_t)kv * N_cap;
  int fbase = 0;
  for (int64_t s0 = 0; s0 < N_prev; s0 += nthr) {
    const int64_t sl = s0 + tid;
    int f = 0;
    if (sl < N_prev) {
      const int32_t p = idx[sl];
      f = !(p >= 0 && p < L && keep_pos(imp_h, p, L, S, R, st));
    }
    const int pos = block_excl_scan(f, warp_buf, &s_total);
    if (f) r.freed[(size_t)hh * N_cap + fbase + pos] = (int32_t)sl;
    fbase += s_total;
  }
  if (tid == 0) {
    roff[n_chunks] = n_new_total;
    r.n_freed[hh] = fbase;
    if ((int64_t)n_new_total != (int64_t)fbase + (N_new - N_prev))
      set_status(status, TS_ERR_INVALID_ARG);   // duplicate or invalid previous slots
  }
}

template <int D>
__global__ void __launch_bounds__(kThreads)
select_gather(Layers P, int64_t L, int64_t L_cap, int S, int R, int64_t N, int64_t n_chunks,
              Ws w, int32_t* status) {
  const int64_t c = blockIdx.x;
  const int kv = blockIdx.y, tid = threadIdx.x, layer = blockIdx.z;
  const int hh = layer * gridDim.y + kv;
  const float* imp_h = imp_of(P, layer) + (size_t)kv * L;
  const __nv_bfloat16* k = P.k ? P.k[layer] : P.k1;
  const __nv_bfloat16* v = P.v ? P.v[layer] : P.v1;
  int32_t* idx = P.idx ? P.idx[layer] : P.idx1;
  __nv_bfloat16* kd = P.kd ? P.kd[layer] : P.kd1;
  __nv_bfloat16* vd = P.vd ? P.vd[layer] : P.vd1;
  const SelectState s = w.state[hh];
  const int32_t* off = w.off + (size_t)hh * (n_chunks + 1);
  __shared__ int warp_buf[32];
  __shared__ int s_total;
  __shared__ int32_t sel[kChunk];
  constexpr int PER = kChunk / kThreads;   // positions per thread
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
  if (tid == 0 && (base + s_total > N || (c == n_chunks - 1 && off[n_chunks] != N)))
    set_status(status, TS_ERR_INVALID_ARG);
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
  for (int e = tid; e < total * V16; e += kThreads) {
    int r = e / V16, x = e % V16;
    int64_t out = base + r;
    if (out >= N) continue;
    int64_t j = sel[r];
    kdst[out * V16 + x] = ksrc[j * V16 + x];
    vdst[out * V16 + x] = vsrc[j * V16 + x];
  }
}

// ---------------------------------------------------------------------------
// Incremental refresh (§3.3: the budgeted cache replaces its less important
// pairs as generation proceeds).  A slot keeps its row while its position
// stays selected; newly selected positions, in ascending order, take the
// freed slots in ascending slot order, then the slots [N_prev, N_new) while
// the cache still grows.  Only those rows are copied.  Stages after the
// selection's histogram and collect kernels:
//   refresh_bits    bitmap of the previous slots' positions (before the
//                   selection's histogram)
//   select_collect  (with the bitmap) also counts per chunk the selected
//                   positions not in the bitmap; the last CTA of a head lists
//                   the freed slots in slot order and turns the counts into
//                   offsets
//   refresh_patch   per chunk: rank the new positions, write idx and copy
//                   their K/V rows into their slots
__global__ void __launch_bounds__(kThreads)
refresh_bits(Layers P, int64_t L, int64_t N_prev, int64_t N_cap, RefreshWs r, int32_t* status) {
  const int kv = blockIdx.y, layer = blockIdx.z, hh = layer * gridDim.y + kv;
  const int32_t* idx = (P.idx ? P.idx[layer] : P.idx1) + (size_t)kv * N_cap;
  uint32_t* bits = r.bits + (size_t)hh * r.w32;
  const int64_t s = (int64_t)blockIdx.x * kThreads + threadIdx.x;
  if (s < N_prev) {
    const int32_t p = idx[s];
    if (p >= 0 && p < L)
      atomicOr(bits + (p >> 5), 1u << (p & 31));
    else
      set_status(status, TS_ERR_INVALID_ARG);
  }
}

template <int D>
__global__ void __launch_bounds__(kThreads)
refresh_patch(Layers P, int64_t L, int64_t L_cap, int S, int R, int64_t N_prev, int64_t N_new,
              int64_t N_cap, int64_t n_chunks, Ws w, RefreshWs r, int32_t* n_written,
              int32_t* status) {
  const int64_t c = blockIdx.x;
  const int kv = blockIdx.y, tid = threadIdx.x, layer = blockIdx.z;
  const int hh = layer * gridDim.y + kv;
  const float* imp_h = imp_of(P, layer) + (size_t)kv * L;
  const __nv_bfloat16* k = P.k ? P.k[layer] : P.k1;
  const __nv_bfloat16* v = P.v ? P.v[layer] : P.v1;
  int32_t* idx = (P.idx ? P.idx[layer] : P.idx1) + (size_t)kv * N_cap;
  __nv_bfloat16* kd = P.kd ? P.kd[layer] : P.kd1;
  __nv_bfloat16* vd = P.vd ? P.vd[layer] : P.vd1;
  const uint32_t* bits = r.bits + (size_t)hh * r.w32;
  const SelectState st = w.state[hh];
  __shared__ int warp_buf[32];
  __shared__ int s_total;
  __shared__ int32_t s_pos[kChunk], s_slot[kChunk];
  constexpr int PER = kChunk / kThreads;
  const int64_t a = c * kChunk + tid * PER;
  int flags = 0, cnt = 0;
#pragma unroll
  for (int x = 0; x < PER; ++x) {
    const int64_t j = a + x;
    if (j < L && keep_pos(imp_h, j, L, S, R, st) && !bit_of(bits, j)) {
      flags |= 1 << x;
      ++cnt;
    }
  }
  int pos = block_excl_scan(cnt, warp_buf, &s_total);
  const int base = __ldcg(r.off + (size_t)hh * (n_chunks + 1) + c);
  const int nf = __ldcg(r.n_freed + hh);
  if (c == 0 && tid == 0 && n_written)
    n_written[hh] = __ldcg(r.off + (size_t)hh * (n_chunks + 1) + n_chunks);
#pragma unroll
  for (int x = 0; x < PER; ++x) {
    if (flags & (1 << x)) {
      const int g = base + pos;
      const int64_t slot = g < nf ? (int64_t)__ldcg(r.freed + (size_t)hh * N_cap + g)
                                  : N_prev + (g - nf);
      const bool ok = slot >= 0 && slot < N_new;
      if (ok) idx[slot] = (int32_t)(a + x);
      else set_status(status, TS_ERR_INVALID_ARG);
      s_pos[pos] = (int32_t)(a + x);
      s_slot[pos] = ok ? (int32_t)slot : -1;
      ++pos;
    }
  }
  __syncthreads();
  const int total = s_total;
  constexpr int V16 = D / 8;
  const uint4* ksrc = reinterpret_cast<const uint4*>(k + (size_t)kv * L_cap * D);
  const uint4* vsrc = reinterpret_cast<const uint4*>(v + (size_t)kv * L_cap * D);
  uint4* kdst = reinterpret_cast<uint4*>(kd + (size_t)kv * N_cap * D);
  uint4* vdst = reinterpret_cast<uint4*>(vd + (size_t)kv * N_cap * D);
  for (int e = tid; e < total * V16; e += kThreads) {
    const int rr = e / V16, x = e % V16;
    const int64_t slot = s_slot[rr];
    if (slot < 0) continue;
    const int64_t j = s_pos[rr];
    kdst[slot * V16 + x] = ksrc[j * V16 + x];
    vdst[slot * V16 + x] = vsrc[j * V16 + x];
  }
}

}  // namespace

SelectPlan select_plan(int Hkv, int64_t L, int n_layers) {
  SelectPlan p{};
  p.chunk = kChunk;
  p.n_chunks = (L + kChunk - 1) / kChunk;
  if (p.n_chunks < 1) p.n_chunks = 1;
  p.ws_bytes = ws_total(Hkv * n_layers, L, p.n_chunks);
  return p;
}

static int run_select(const Layers& P, int n_layers, int64_t L, int64_t L_cap, int Hkv, int d,
                      int B, int S, int R, int64_t N, void* ws, int32_t* status, cudaStream_t st) {
  SelectPlan p = select_plan(Hkv, L, n_layers);
  if (p.n_chunks > 1024)
    return fail(TS_ERR_UNSUPPORTED, "ts_partial_kv_select_gather: L > %d", 1024 * kChunk);
  Ws w = carve(ws, Hkv * n_layers, L, p.n_chunks);
  if (cudaMemsetAsync(ws, 0, w.zero_bytes, st) != cudaSuccess)
    return launch_status("select workspace reset");
  dim3 grid((unsigned)p.n_chunks, Hkv, n_layers);
  dim3 sgrid((unsigned)((L + kScan - 1) / kScan), Hkv, n_layers);
  select_hist<<<sgrid, kThreads, 0, st>>>(P, L, B, S, R, p.n_chunks, w);
  int rc = launch_status("select_hist");
  if (rc) return rc;
  RefreshWs no_refresh{};   // bits = null: selection only
  select_collect<<<sgrid, kThreads, 0, st>>>(P, L, S, R, p.n_chunks, w, no_refresh, 0, 0, 0,
                                            nullptr);
  rc = launch_status("select_collect");
  if (rc) return rc;
  if (d == 128)
    select_gather<128><<<grid, kThreads, 0, st>>>(P, L, L_cap, S, R, N, p.n_chunks, w, status);
  else
    select_gather<64><<<grid, kThreads, 0, st>>>(P, L, L_cap, S, R, N, p.n_chunks, w, status);
  return launch_status("select_gather");
}

int launch_select_gather(const float* imp, const void* k, const void* v, int64_t L,
                         int64_t L_cap, int Hkv, int d, int B, int S, int R, int32_t* idx,
                         void* kd, void* vd, int64_t N, void* ws, int32_t* status,
                         cudaStream_t st) {
  Layers P{};
  P.imp1 = imp;
  P.k1 = static_cast<const __nv_bfloat16*>(k);
  P.v1 = static_cast<const __nv_bfloat16*>(v);
  P.idx1 = idx;
  P.kd1 = static_cast<__nv_bfloat16*>(kd);
  P.vd1 = static_cast<__nv_bfloat16*>(vd);
  return run_select(P, 1, L, L_cap, Hkv, d, B, S, R, N, ws, status, st);
}

// ---------------------------------------------------------------------------
// Allocation-free variant: the scratch lives in one fixed device array of the
// library instead of a caller workspace.  Its device address is looked up once
// per device (with that device current) and cached; every call on a device
// shares the array, so calls that overlap on the GPU race on it.
namespace {
static __device__ __align__(256) unsigned char g_select_scratch[kNoAllocScratchBytes];
}

int select_scratch(void** out) {
  static std::mutex mu;
  static void* cached[64] = {nullptr};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(TS_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
  if (dev < 0 || dev >= 64) return fail(TS_ERR_UNSUPPORTED, "device ordinal %d >= 64", dev);
  std::lock_guard<std::mutex> lock(mu);
  if (!cached[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_select_scratch);
    if (e != cudaSuccess || !p)
      return fail(TS_ERR_CUDA, "cudaGetSymbolAddress(select scratch): %s", cudaGetErrorString(e));
    cached[dev] = p;
  }
  *out = cached[dev];
  return TS_OK;
}

int launch_select_gather_batched(int n_layers, const float* const* imp, const void* const* k,
                                 const void* const* v, int64_t L, int64_t L_cap, int Hkv, int d,
                                 int B, int S, int R, int32_t* const* idx, void* const* kd,
                                 void* const* vd, int64_t N, void* ws, int32_t* status,
                                 cudaStream_t st) {
  Layers P{};
  P.imp = imp;
  P.k = reinterpret_cast<const __nv_bfloat16* const*>(k);
  P.v = reinterpret_cast<const __nv_bfloat16* const*>(v);
  P.idx = idx;
  P.kd = reinterpret_cast<__nv_bfloat16* const*>(kd);
  P.vd = reinterpret_cast<__nv_bfloat16* const*>(vd);
  return run_select(P, n_layers, L, L_cap, Hkv, d, B, S, R, N, ws, status, st);
}

size_t refresh_ws_bytes(int HH, int64_t L, int64_t N_cap) {
  const SelectPlan p = select_plan(HH, L, 1);
  return ws_total(HH, L, p.n_chunks) + refresh_area_bytes(HH, L, p.n_chunks, N_cap);
}

int launch_refresh_incremental(int n_layers, const float* imp1, const float* const* imp,
                               const void* k1, const void* const* k, const void* v1,
                               const void* const* v, int64_t L, int64_t L_cap, int Hkv, int d,
                               int B, int S, int R, int64_t N_prev, int64_t N_new, int64_t N_cap,
                               int32_t* idx1, int32_t* const* idx, void* kd1, void* const* kd,
                               void* vd1, void* const* vd, int32_t* n_written, void* ws,
                               int32_t* status, cudaStream_t st) {
  Layers P{};
  P.imp = imp;
  P.k = reinterpret_cast<const __nv_bfloat16* const*>(k);
  P.v = reinterpret_cast<const __nv_bfloat16* const*>(v);
  P.idx = idx;
  P.kd = reinterpret_cast<__nv_bfloat16* const*>(kd);
  P.vd = reinterpret_cast<__nv_bfloat16* const*>(vd);
  P.imp1 = imp1;
  P.k1 = static_cast<const __nv_bfloat16*>(k1);
  P.v1 = static_cast<const __nv_bfloat16*>(v1);
  P.idx1 = idx1;
  P.kd1 = static_cast<__nv_bfloat16*>(kd1);
  P.vd1 = static_cast<__nv_bfloat16*>(vd1);
  const int HH = Hkv * n_layers;
  const SelectPlan p = select_plan(Hkv, L, n_layers);
  if (p.n_chunks > 1024)
    return fail(TS_ERR_UNSUPPORTED, "ts_partial_kv_refresh_incremental: L > %d", 1024 * kChunk);
  Ws w = carve(ws, HH, L, p.n_chunks);
  RefreshWs r = carve_refresh(static_cast<char*>(ws) + ws_total(HH, L, p.n_chunks), HH, L,
                              p.n_chunks, N_cap);
  if (cudaMemsetAsync(ws, 0, w.zero_bytes, st) != cudaSuccess ||
      cudaMemsetAsync(r.bits, 0, r.zero_bytes, st) != cudaSuccess)
    return launch_status("refresh workspace reset");
  dim3 grid((unsigned)p.n_chunks, Hkv, n_layers);
  dim3 sgrid((unsigned)((L + kScan - 1) / kScan), Hkv, n_layers);
  if (N_prev > 0) {
    dim3 bgrid((unsigned)((N_prev + kThreads - 1) / kThreads), Hkv, n_layers);
    refresh_bits<<<bgrid, kThreads, 0, st>>>(P, L, N_prev, N_cap, r, status);
    int rc = launch_status("refresh_bits");
    if (rc) return rc;
  }
  select_hist<<<sgrid, kThreads, 0, st>>>(P, L, B, S, R, p.n_chunks, w);
  int rc = launch_status("select_hist");
  if (rc) return rc;
  select_collect<<<sgrid, kThreads, 0, st>>>(P, L, S, R, p.n_chunks, w, r, N_prev, N_new, N_cap,
                                            status);
  rc = launch_status("select_collect");
  if (rc) return rc;
  if (d == 128)
    refresh_patch<128><<<grid, kThreads, 0, st>>>(P, L, L_cap, S, R, N_prev, N_new, N_cap,
                                                  p.n_chunks, w, r, n_written, status);
  else
    refresh_patch<64><<<grid, kThreads, 0, st>>>(P, L, L_cap, S, R, N_prev, N_new, N_cap,
                                                 p.n_chunks, w, r, n_written, status);
  return launch_status("refresh_patch");
}

}  // namespace ts
