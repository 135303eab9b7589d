// Rejection-sampling acceptance over the draft tree (speculative sampling).
//
// "TokenSwift: Lossless Acceleration of Ultra Long Sequence Generation",
// A. Lossless Nature of Speculative Decoding: acceptance and rejection cases
// together reproduce the target model's distribution.  §3.4 / Table 11 give
// the target's processing (contextual penalty over the last W tokens,
// temperature, top-p and min-p), the same as the exact-match path.
//
// Tree form (multi-candidate recursive rejection): from the root, at each
// accepted node n the children are tried in index order as draws from q[n],
// the draft distribution that proposed them.  Child c with token x is
// accepted iff u_accept[c] * q[n][x] < p(x), p being n's target
// distribution; on rejection p becomes max(p - q[n], 0) renormalised.  When
// no child is accepted, the bonus token is drawn from the current p with
// u_draw[n] by inverse CDF in token-id order.
//
// One CTA of 1024 threads walks the path (at most T nodes, each with its
// children); every step over the vocabulary is block-wide:
//   x' pass        window bitmap, penalty, temperature -> ws[V]; block max M
//   truncation     none when top_p >= 1 and min_p <= 0; otherwise the tokens
//                  with exp(x' - M) >= min_p are collected (at most kCand),
//                  bitonic-sorted by (x' desc, id asc), and the top-p cut is
//                  read off their prefix masses (Z over the whole vocabulary):
//                  rank r is kept while the mass before it is <= top_p * Z,
//                  the smallest set whose mass exceeds top_p (§D.1)
//   p pass         ws[t] = kept(t) ? exp(x'_t - M) / Z_kept : 0
//   per rejection  S = sum max(ws[t] - q[t], 0); when S > 0,
//                  ws[t] = max(ws[t] - q[t], 0) / S (S = 0 only when nothing
//                  of p is left above q, and p then stays as it is)
//   bonus          block exclusive scan of per-thread id-ordered segments;
//                  the last thread whose segment starts at or below the
//                  target owns the draw
// No waits on other CTAs or on barriers with timeouts: loops and block
// barriers only.  Token ids and parents are range-checked; a violation is
// reported in the status word.
#include "ts_common.cuh"

namespace ts {

namespace {

constexpr int kRThreads = 1024;
constexpr int kCand = 2048;   // min-p candidates sorted for the top-p cut

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// block-wide max / sum over kRThreads threads (every thread gets the result)
__device__ float block_max(float v, float* red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  v = warp_max(v);
  __syncthreads();
  if (lane == 0) red[warp] = v;
  __syncthreads();
  float r = red[lane];
  r = warp_max(r);
  return r;
}
__device__ float block_sum(float v, float* red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  v = warp_sum(v);
  __syncthreads();
  if (lane == 0) red[warp] = v;
  __syncthreads();
  float r = red[lane];
  r = warp_sum(r);
  return r;
}

// exclusive prefix of one float per thread, in thread order
__device__ float block_excl_scan_f(float v, float* red, float* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  float incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  __syncthreads();
  if (lane == 31) red[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const float w = red[lane];
    float wi = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float y = __shfl_up_sync(0xffffffffu, wi, o);
      if (lane >= o) wi += y;
    }
    red[lane] = wi - w;
    if (lane == 31) *total = wi;
  }
  __syncthreads();
  const float r = red[warp] + incl - v;
  __syncthreads();
  return r;
}

__global__ void __launch_bounds__(kRThreads, 1)
reject_accept_kernel(const float* __restrict__ logits, const float* __restrict__ q,
                     const int32_t* __restrict__ tree_tokens, const int32_t* __restrict__ parents,
                     int T, const int32_t* __restrict__ prior, int n_prior, int W, int V,
                     float penalty, float temperature, float top_p, float min_p, int literal,
                     const float* __restrict__ u_accept, const float* __restrict__ u_draw,
                     int32_t* __restrict__ path, int32_t* __restrict__ n_path,
                     int32_t* __restrict__ bonus, float* __restrict__ ws, int32_t* status) {
  extern __shared__ uint32_t bitmap[];   // (V + 31) / 32 words: the window, then the kept set
  __shared__ float red[32];
  __shared__ float s_ckey[kCand];
  __shared__ int32_t s_cid[kCand];
  __shared__ int s_ncand, s_nkeep, s_bonus, s_bad, s_owner, s_accept;
  __shared__ int s_path[64], s_drafted[64];
  __shared__ float s_tot, s_zk;
  const int tid = threadIdx.x;
  const int nwords = (V + 31) / 32;
  const bool no_trunc = top_p >= 1.0f && min_p <= 0.0f;
  const bool unit_temp = temperature == 1.0f;
  if (tid == 0) {
    s_bad = 0;
    s_path[0] = 0;
    for (int c = 0; c < T; ++c) {
      const int p = parents[c];
      if ((c == 0 && p != -1) || (c > 0 && (p < 0 || p >= c))) s_bad = 1;
    }
  }
  __syncthreads();
  int node = 0, np = 1, nd = 0;
  bool unsupported = false;
  for (int hop = 0; hop < T; ++hop) {
    // ---- window of this node: the last W tokens of (prior ++ drafted path)
    for (int x = tid; x < nwords; x += kRThreads) bitmap[x] = 0u;
    __syncthreads();
    const int total_win = n_prior + nd, wlen = min(W, total_win);
    for (int e = tid; e < wlen; e += kRThreads) {
      const int k = total_win - wlen + e;
      const int t = k < n_prior ? prior[k] : s_drafted[k - n_prior];
      if (t >= 0 && t < V)
        atomicOr(&bitmap[t >> 5], 1u << (t & 31));
      else
        s_bad = 1;
    }
    __syncthreads();
    // ---- x' (penalty, temperature) and its maximum
    const float* xin = logits + (size_t)node * V;
    float lmax = -INFINITY;
    for (int t = tid; t < V; t += kRThreads) {
      float x = xin[t];
      if ((bitmap[t >> 5] >> (t & 31)) & 1u)
        x = (literal || x > 0.f) ? __fdiv_rn(x, penalty) : __fmul_rn(x, penalty);
      if (!unit_temp) x = __fdiv_rn(x, temperature);
      ws[t] = x;
      lmax = fmaxf(lmax, x);
    }
    const float M = block_max(lmax, red);
    float zp = 0.f;
    for (int t = tid; t < V; t += kRThreads) zp += expf(ws[t] - M);
    const float Zall = block_sum(zp, red);
    // ---- truncation: min-p candidates, sorted, top-p prefix
    if (!no_trunc) {
      if (tid == 0) s_ncand = 0;
      __syncthreads();
      for (int t = tid; t < V; t += kRThreads) {
        if (expf(ws[t] - M) >= min_p) {
          const int k = atomicAdd(&s_ncand, 1);
          if (k < kCand) {
            s_ckey[k] = ws[t];
            s_cid[k] = t;
          }
        }
      }
      __syncthreads();
      const int nc = s_ncand;
      if (nc > kCand) {
        unsupported = true;   // every thread sees the same count
        break;
      }
      int P = 1;
      while (P < nc) P <<= 1;
      for (int k = nc + tid; k < P; k += kRThreads) {
        s_ckey[k] = -INFINITY;
        s_cid[k] = 0x7FFFFFFF;
      }
      __syncthreads();
      // bitonic sort, order (x' desc, id asc)
      for (int size = 2; size <= P; size <<= 1) {
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
          for (int i = tid; i < P; i += kRThreads) {
            const int j = i ^ stride;
            if (j > i) {
              const float ki = s_ckey[i], kj = s_ckey[j];
              const int ii = s_cid[i], ij = s_cid[j];
              const bool i_first = ki > kj || (ki == kj && ii < ij);
              if (((i & size) == 0) != i_first) {
                s_ckey[i] = kj;
                s_ckey[j] = ki;
                s_cid[i] = ij;
                s_cid[j] = ii;
              }
            }
          }
          __syncthreads();
        }
      }
      if (tid == 0) {
        const float cut = top_p >= 1.0f ? INFINITY : top_p * Zall;
        float before = 0.f, zk = 0.f;
        int nk = 0;
        for (int r = 0; r < nc; ++r) {
          if (r > 0 && before > cut) break;
          const float e = expf(s_ckey[r] - M);
          before += e;
          zk += e;
          nk = r + 1;
        }
        s_nkeep = nk;
        s_zk = zk;
      }
      __syncthreads();
      for (int x = tid; x < nwords; x += kRThreads) bitmap[x] = 0u;
      __syncthreads();
      for (int r = tid; r < s_nkeep; r += kRThreads)
        atomicOr(&bitmap[s_cid[r] >> 5], 1u << (s_cid[r] & 31));
      __syncthreads();
    }
    const float Zk = no_trunc ? Zall : s_zk;
    // ---- the target distribution p of this node
    for (int t = tid; t < V; t += kRThreads) {
      const bool kept = no_trunc || ((bitmap[t >> 5] >> (t & 31)) & 1u);
      ws[t] = kept ? __fdiv_rn(expf(ws[t] - M), Zk) : 0.f;
    }
    __syncthreads();
    // ---- the children, in index order
    const float* qn = q + (size_t)node * V;
    int next = -1;
    for (int c = node + 1; c < T; ++c) {
      if (parents[c] != node) continue;
      const int x = tree_tokens[c];
      if (x < 0 || x >= V) {
        if (tid == 0) s_bad = 1;
        continue;
      }
      // one thread decides, every thread branches on its decision
      if (tid == 0) s_accept = (u_accept[c] * qn[x] < ws[x]) ? 1 : 0;
      __syncthreads();
      if (s_accept) {
        next = c;
        break;
      }
      float part = 0.f;
      for (int t = tid; t < V; t += kRThreads) part += fmaxf(ws[t] - qn[t], 0.f);
      const float S = block_sum(part, red);
      if (S > 0.f)
        for (int t = tid; t < V; t += kRThreads) ws[t] = __fdiv_rn(fmaxf(ws[t] - qn[t], 0.f), S);
      __syncthreads();
    }
    if (next >= 0) {
      node = next;
      if (tid == 0) {
        s_path[np] = next;
        s_drafted[nd] = tree_tokens[next];
      }
      ++np;
      ++nd;
      __syncthreads();
      continue;
    }
    // ---- bonus: inverse CDF over token ids
    const int per = (V + kRThreads - 1) / kRThreads;
    const int t0 = min(V, tid * per), t1 = min(V, t0 + per);
    float seg = 0.f;
    for (int t = t0; t < t1; ++t) seg += ws[t];
    if (tid == 0) {
      s_bonus = 0x7FFFFFFF;
      s_owner = -1;
    }
    const float before = block_excl_scan_f(seg, red, &s_tot);
    const float target = u_draw[node] * s_tot;
    // the owner is the last thread with mass whose segment starts at or
    // below the target: the scan's rounding can leave a target between one
    // segment's end and the next one's start, and the owner then takes its
    // own last token with mass
    if (seg > 0.f && before <= target) atomicMax(&s_owner, tid);
    __syncthreads();
    if (tid == s_owner) {
      float cum = before;
      int pick = -1, last = -1;
      for (int t = t0; t < t1; ++t) {
        if (ws[t] > 0.f) last = t;
        cum += ws[t];
        if (cum > target) {
          pick = t;
          break;
        }
      }
      s_bonus = pick >= 0 ? pick : last;
    }
    __syncthreads();
    if (s_owner < 0 && tid == 0) s_bad = 2;   // no mass left anywhere: not a distribution
    __syncthreads();
    break;
  }
  if (tid == 0) {
    if (unsupported) {
      set_status(status, TS_ERR_UNSUPPORTED);
      path[0] = 0;
      *n_path = 1;
      *bonus = -1;
    } else {
      for (int k = 0; k < np; ++k) path[k] = s_path[k];
      *n_path = np;
      *bonus = s_bonus;
    }
    if (s_bad == 2) {
      // only reachable when every target and draft mass is zero or negative
      // (invalid q rows): no token carries mass, so no bonus is emitted
      *bonus = -1;
    }
    if (s_bad) set_status(status, TS_ERR_INVALID_ARG);
  }
}

}  // namespace

size_t reject_ws_bytes(int V) { return ((size_t)V * sizeof(float) + 255) / 256 * 256; }

int launch_reject_accept(const float* logits, const float* q, const int32_t* tree_tokens,
                         const int32_t* parents, int T, const int32_t* prior, int n_prior, int W,
                         int V, float penalty, float temperature, float top_p, float min_p,
                         int literal, const float* u_accept, const float* u_draw, int32_t* path,
                         int32_t* n_path, int32_t* bonus, void* ws, int32_t* status,
                         cudaStream_t st) {
  const size_t smem = (size_t)((V + 31) / 32) * sizeof(uint32_t);
  cudaFuncSetAttribute(reject_accept_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  reject_accept_kernel<<<1, kRThreads, smem, st>>>(
      logits, q, tree_tokens, parents, T, prior, n_prior, W, V, penalty, temperature, top_p, min_p,
      literal, u_accept, u_draw, path, n_path, bonus, static_cast<float*>(ws), status);
  return launch_status("reject_accept_kernel");
}

}  // namespace ts
