// Contextual-penalty sampling of every draft-tree node, exact-match tree
// acceptance, and the KV commit of the accepted path.
//
// "TokenSwift: Lossless Acceleration of Ultra Long Sequence Generation":
// §3.4 Contextual Penalty (penalty on the most recent W tokens), §D.1
// (top-p: smallest set whose cumulative probability exceeds p, every token
// when p >= 1; min-p: tokens with p >= p_base * p_max), Table 11 (penalty 1.2 over 1024 tokens, temperature
// 1.0, top-p 0.9, min-p 0.05), §3.1 Overview (exact-match verification, the
// longest valid draft is kept, then the KV cache is updated).
//
// Each tree node's vocabulary is split over kParts CTAs.  Every CTA marks
// the node's window in a shared-memory bitmap, writes the penalised/tempered
// logits x' of its slice once to the workspace, and publishes its slice
// maximum m_c, Z_c = sum exp(x' - m_c) and the tokens with
// exp(x' - m_c) >= min_p (a superset of the node's min-p set, as m_c <= the
// node maximum).  The last CTA of the node (atomic ticket, no waiting) takes
// the maximum over the slices, rescales and adds the Z_c, and keeps the
// candidates with e_t = exp(x'_t - max x') >= min_p.  In rank order (x' desc, id asc) both truncations keep a
// prefix: top-p keeps ranks up to the first whose inclusive mass exceeds
// top_p * Z, min-p keeps the ranks with e >= min_p.  So the kept set always
// lies inside the min-p set; when that set is small (the usual case:
// min-p 0.05 keeps the tokens within ln 20 of the top logit) its members are
// collected in the same pass that sums Z, sorted in shared memory, and the
// top-p cut and the draw are read off their prefix sums.  Otherwise "first
// rank whose inclusive mass crosses a target" is found without sorting by a
// radix descent over the 50-bit key (x' key, reversed id) carrying a
// (count, mass) histogram per digit: 3 levels on the fp32 key, 2 on the id.
// The last CTA to finish walks the tree and writes the accepted path.
//
// Rejection mode (A. Lossless Nature of Speculative Decoding): the same
// slice and merge phases give every node its truncated target p (the kept
// set above, renormalised); then, instead of a draw, the node's CTA runs the
// speculative-sampling chain over its children in index order: child c with
// token x is accepted iff u_accept[c] * q[i][x] < p(x); on rejection p
// becomes max(p - q[i], 0) renormalised (left as it is when nothing is
// left); with no child accepted, the bonus token is drawn from the current p
// by inverse CDF in token-id order with u_draw[i].  A node's outcome does not
// depend on which nodes the walk visits, so every node is resolved in
// parallel and the last CTA follows the outcomes from the root.  p and its
// residuals live on the kept set (usually tens of tokens: one warp runs the
// chain there); when the kept set overflows shared memory, or with no
// truncation at all, the chain runs over the node's vocabulary row.
#include "tc_ptx.cuh"
#include "ts_common.cuh"

namespace ts {

namespace {

constexpr int kThreads = 512;
constexpr int kParts = 4;                // CTAs per tree node
constexpr int kCapPart = 4096;           // candidates one slice may publish
constexpr int kBatch = 8;                // float4 loads of a thread in flight together
constexpr int kScan = 8;                 // loads of a thread in flight in the per-node scans
constexpr int kPool = kParts * kCapPart; // pool entries a node's scan compacts (its slices'
                                         // candidate area, unused once it scans the row)
constexpr int kMaxBuckets = 2048;
constexpr uint32_t kIdMask = 0x3FFFFu;   // V <= 2^18

enum FindMode { kMassGT = 1, kRank = 2 };

struct Found {
  int id;
  int rank;        // number of tokens ranked before it
  float cum_incl;  // sum of e over ranks <= its rank
};

constexpr int kCap = 4096;               // min-p candidates sorted in shared memory

struct SampleSmem {
  int cnt[kMaxBuckets];
  float mass[kMaxBuckets];
  uint32_t ckey[kCap];                    // float_key(x') of the min-p candidates
  int32_t cid[kCap];                      // their token ids
  int ncand;
  float red_f[32];
  int red_i[32];
  uint32_t kpre, kmask, ipre, imask;
  float mb;     // mass ranked before the current bucket range
  int cb;       // count ranked before the current bucket range
  int32_t ptok[64];
  int32_t par[64], tok[64], smp[64];     // the tree, staged once (T <= 64)
  int best;    // acceptance: depth * 256 + (255 - node) of the best node
  int plen;
  int last;
  int nkeep;   // rejection mode: the kept set's size, its mass, the outcome
  float zk;
  int outcome;
  uint32_t cut_key, cut_rid;
};

struct PartStat {
  float m;     // slice maximum of x'
  float z;     // sum over the slice of exp(x' - m)
  int n;       // tokens with exp(x' - m) >= min_p (may exceed kCapPart)
  float s;     // eta mode: sum over the slice of exp(x' - m) (x' - m)
};

// workspace: [counters | PartStat [T][kParts] | candidates [T][kParts][kCapPart] | x' [T][V]]
constexpr size_t kCounterBytes = 1024;   // node tickets [64] + step counter
struct SampleWs {
  int32_t* node_ticket;
  int32_t* counter;
  PartStat* stat;
  uint2* cand;     // (float_key(x'), token id)
  float* xs;
};
__host__ __device__ inline size_t a256s(size_t x) { return (x + 255) / 256 * 256; }
__host__ __device__ inline SampleWs carve_sample(void* base, int T) {
  char* p = static_cast<char*>(base);
  SampleWs w;
  w.node_ticket = reinterpret_cast<int32_t*>(p);
  w.counter = w.node_ticket + 64;
  size_t o = kCounterBytes;
  w.stat = reinterpret_cast<PartStat*>(p + o);
  o += a256s((size_t)T * kParts * sizeof(PartStat));
  w.cand = reinterpret_cast<uint2*>(p + o);
  o += a256s((size_t)T * kParts * kCapPart * sizeof(uint2));
  w.xs = reinterpret_cast<float*>(p + o);
  return w;
}

// inverse of float_key
__device__ __forceinline__ float key_float(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

__device__ float block_max(float v, SampleSmem& sm) {
  v = warp_max(v);
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  if (lane == 0) sm.red_f[w] = v;
  __syncthreads();
  float r = lane < (int)(blockDim.x >> 5) ? sm.red_f[lane] : -INFINITY;
  r = warp_max(r);
  __syncthreads();
  return r;
}
__device__ float block_sum(float v, SampleSmem& sm) {
  v = warp_sum(v);
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  if (lane == 0) sm.red_f[w] = v;
  __syncthreads();
  float r = lane < (int)(blockDim.x >> 5) ? sm.red_f[lane] : 0.f;
  r = warp_sum(r);
  __syncthreads();
  return r;
}
__device__ int block_sum_int(int v, SampleSmem& sm) {
  v = warp_sum_int(v);
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  if (lane == 0) sm.red_i[w] = v;
  __syncthreads();
  int r = lane < (int)(blockDim.x >> 5) ? sm.red_i[lane] : 0;
  r = warp_sum_int(r);
  __syncthreads();
  return r;
}

// One radix level: histogram the tokens matching the digits fixed so far,
// then (warp 0) pick the bucket holding the target and fold the buckets
// ranked above it into (mb, cb).  Returns nothing; updates the prefixes.
// Tokens with e = exp(x - xmax) < skip_e are left out: a caller whose target
// lies inside the rank prefix {e >= skip_e} (the kept pool ranks first) gets
// the same token without them, and the first levels, which put most tokens
// into a few buckets, take far fewer contended atomics.
// With kList, the level reads a `list` of n (float_key(x'), id) pairs (a
// node's kept pool, compacted by its scan) instead of the row xs.
template <bool kList>
__device__ __noinline__ void radix_level(const float* __restrict__ xs, int V, const uint2* list, int n,
                            float xmax, int mode, float target_mass, int target_rank, bool on_id,
                            int shift, int bits, float skip_e, SampleSmem& sm) {
  const int nb = 1 << bits;
  for (int b = threadIdx.x; b < nb; b += blockDim.x) {
    sm.cnt[b] = 0;
    sm.mass[b] = 0.f;
  }
  __syncthreads();
  const uint32_t kpre = sm.kpre, kmask = sm.kmask, ipre = sm.ipre, imask = sm.imask;
  // kScan loads of a thread in flight together, then their histogram updates
  const int n_in = kList ? n : V;
  for (int c0 = 0; c0 < n_in; c0 += blockDim.x * kScan) {
    uint32_t kx[kScan], ki[kScan];
#pragma unroll
    for (int u = 0; u < kScan; ++u) {
      const int j = c0 + u * blockDim.x + threadIdx.x;
      kx[u] = 0u;
      ki[u] = (uint32_t)j;
      if (j < n_in) {
        if (kList) {
          const uint2 v = list[j];
          kx[u] = v.x;
          ki[u] = v.y;
        } else {
          kx[u] = __float_as_uint(xs[j]);
        }
      }
    }
#pragma unroll
    for (int u = 0; u < kScan; ++u) {
      const int j = c0 + u * blockDim.x + threadIdx.x;
      if (j >= n_in) continue;
      const float x = kList ? key_float(kx[u]) : __uint_as_float(kx[u]);
      const int t = (int)ki[u];
      const uint32_t key = float_key(x), rid = kIdMask - (uint32_t)t;
      if ((key & kmask) != kpre || (rid & imask) != ipre) continue;
      const float e = expf(x - xmax);
      if (e < skip_e) continue;
      const uint32_t dig = ((on_id ? rid : key) >> shift) & (uint32_t)(nb - 1);
      atomicAdd(&sm.cnt[dig], 1);
      if (mode != kRank) atomicAdd(&sm.mass[dig], e);
    }
  }
  __syncthreads();
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x, per = nb / 32;
    // lane 0 owns the highest buckets (ranked first)
    const int top = nb - 1 - lane * per;
    float lm = 0.f;
    int lc = 0;
    for (int x = 0; x < per; ++x) {
      lm += sm.mass[top - x];
      lc += sm.cnt[top - x];
    }
    float im = lm;
    int ic = lc;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      float ym = __shfl_up_sync(0xffffffffu, im, o);
      int yc = __shfl_up_sync(0xffffffffu, ic, o);
      if (lane >= o) {
        im += ym;
        ic += yc;
      }
    }
    const float mb = sm.mb;
    const int cb = sm.cb;
    bool cross;
    if (mode == kMassGT) cross = lc > 0 && mb + im > target_mass;
    else cross = lc > 0 && cb + ic > target_rank;
    unsigned bal = __ballot_sync(0xffffffffu, cross);
    int src;
    if (bal) {
      src = __ffs(bal) - 1;
    } else {
      // rounding left the target beyond the last token: take the last one
      unsigned ne = __ballot_sync(0xffffffffu, lc > 0);
      src = 31 - __clz(ne);
    }
    if (lane == src) {
      float m = mb + im - lm;   // mass ranked before this lane's buckets
      int c = cb + ic - lc;
      int chosen = -1, last_ne = -1;
      float m_at = m;
      int c_at = c;
      for (int x = 0; x < per; ++x) {
        const int b = top - x;
        if (sm.cnt[b] == 0) continue;
        last_ne = b;
        m_at = m;
        c_at = c;
        const float mn = m + sm.mass[b];
        const int cn = c + sm.cnt[b];
        bool hit = (mode == kMassGT) ? (mn > target_mass) : (cn > target_rank);
        if (hit) {
          chosen = b;
          break;
        }
        m = mn;
        c = cn;
      }
      if (chosen < 0) chosen = last_ne;   // rounding fallback: last non-empty bucket
      sm.mb = m_at;
      sm.cb = c_at;
      const uint32_t dmask = (uint32_t)(nb - 1) << shift;
      if (on_id) {
        sm.ipre = ipre | ((uint32_t)chosen << shift);
        sm.imask = imask | dmask;
      } else {
        sm.kpre = kpre | ((uint32_t)chosen << shift);
        sm.kmask = kmask | dmask;
      }
    }
  }
  __syncthreads();
}

template <bool kList>
__device__ __noinline__ Found radix_find(const float* __restrict__ xs, int V, const uint2* list, int n,
                            float xmax, int mode, float target_mass, int target_rank, float skip_e,
                            SampleSmem& sm) {
  if (threadIdx.x == 0) {
    sm.kpre = sm.kmask = sm.ipre = sm.imask = 0;
    sm.mb = 0.f;
    sm.cb = 0;
  }
  int key_bits = 32;   // key bits the levels resolve, from the top
  if (kList) {
    // a compacted pool spans a narrow range of keys: its common leading
    // bits are fixed in the prefix, so the first level spreads the pool over
    // its buckets instead of piling it into a few contended ones
    uint32_t lo = 0xFFFFFFFFu, hi = 0u;
    for (int j = threadIdx.x; j < n; j += blockDim.x) {
      const uint32_t k = list[j].x;
      lo = min(lo, k);
      hi = max(hi, k);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      lo = min(lo, __shfl_xor_sync(0xffffffffu, lo, o));
      hi = max(hi, __shfl_xor_sync(0xffffffffu, hi, o));
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      sm.red_i[0] = (int)0xFFFFFFFFu;
      sm.red_i[1] = 0;
    }
    __syncthreads();
    if ((threadIdx.x & 31) == 0) {
      atomicMin(reinterpret_cast<unsigned*>(&sm.red_i[0]), lo);
      atomicMax(reinterpret_cast<unsigned*>(&sm.red_i[1]), hi);
    }
    __syncthreads();
    lo = (uint32_t)sm.red_i[0];
    hi = (uint32_t)sm.red_i[1];
    const int common = lo <= hi ? __clz(lo ^ hi) : 0;   // 32 when every key is equal
    key_bits = 32 - common;
    if (threadIdx.x == 0 && common > 0) {
      const uint32_t pm = common == 32 ? 0xFFFFFFFFu : ~(0xFFFFFFFFu >> common);
      sm.kpre = lo & pm;
      sm.kmask = pm;
    }
  }
  __syncthreads();
  // key levels of at most 11 bits from the highest unresolved one down,
  // then the 18 id bits in two levels of 9
  while (key_bits > 0) {
    const int b = key_bits < 11 ? key_bits : 11;
    key_bits -= b;
    radix_level<kList>(xs, V, list, n, xmax, mode, target_mass, target_rank, false, key_bits, b,
                       skip_e, sm);
  }
  radix_level<kList>(xs, V, list, n, xmax, mode, target_mass, target_rank, true, 9, 9, skip_e, sm);
  radix_level<kList>(xs, V, list, n, xmax, mode, target_mass, target_rank, true, 0, 9, skip_e, sm);
  Found f;
  f.id = (int)(kIdMask - sm.ipre);
  f.rank = sm.cb;
  // the token is fully determined: its own e completes the inclusive mass
  float xv = xs[f.id];
  f.cum_incl = sm.mb + expf(xv - xmax);
  __syncthreads();
  return f;
}


// ---------------------------------------------------------------- rejection
// The children of node i in index order are the nodes c > i with parents[c]
// = i (sm.par, sm.tok staged).  Outcome codes: child c (>= 1) or -1 - token.

// Bonus draw from the row p = xs[0, V) (all threads): per-thread contiguous
// segments of token ids, a block exclusive scan of their sums; the owner is
// the last thread with mass whose segment starts at or below the target
// (rounding can leave the target between two segments) and it takes the
// first token whose cumulative mass exceeds the target, else its last token
// with mass.  Returns -1 - token.
__device__ int bonus_dense(int i, int V, const float* __restrict__ xs,
                           const float* __restrict__ u_draw, SampleSmem& sm) {
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const int per = (V + kThreads - 1) / kThreads;
  const int t0 = min(V, tid * per), t1 = min(V, t0 + per);
  float seg = 0.f;
  for (int t = t0; t < t1; ++t) seg += xs[t];
  float incl = seg;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) sm.red_f[w] = incl;
  if (tid == 0) sm.best = -1;
  __syncthreads();
  if (w == 0) {
    const float v = lane < (kThreads >> 5) ? sm.red_f[lane] : 0.f;
    float wi = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float y = __shfl_up_sync(0xffffffffu, wi, o);
      if (lane >= o) wi += y;
    }
    if (lane < (kThreads >> 5)) sm.mass[lane] = wi - v;   // warps before this one
    if (lane == 31) sm.zk = wi;                           // total
  }
  __syncthreads();
  const float before = sm.mass[w] + incl - seg;
  const float target = u_draw[i] * sm.zk;
  if (seg > 0.f && before <= target) atomicMax(&sm.best, tid);
  __syncthreads();
  if (tid == sm.best) {
    float cum = before;
    int pick = -1, last = -1;
    for (int t = t0; t < t1; ++t) {
      if (xs[t] > 0.f) last = t;
      cum += xs[t];
      if (cum > target) {
        pick = t;
        break;
      }
    }
    sm.outcome = -1 - (pick >= 0 ? pick : last);
  }
  __syncthreads();
  const int oc = sm.best >= 0 ? sm.outcome : -1;   // no mass anywhere: token 0
  __syncthreads();
  return oc;
}

// Kept set in shared memory (ranks 0 .. nkeep-1 of sm.ckey / sm.cid, sorted
// by (x' desc, id asc)); warp 0 runs the chain with p and q of the kept
// tokens in two shared arrays, then the bonus draw in token-id order.
__device__ int reject_sparse(int i, int T, int V, float xmax, const float* __restrict__ qrow,
                             const float* __restrict__ u_accept, const float* __restrict__ u_draw,
                             float* __restrict__ xs, SampleSmem& sm) {
  const int tid = threadIdx.x, lane = tid & 31;
  const int nk = sm.nkeep;
  constexpr int kSparseBonus = 256;    // larger kept sets draw over the row
  float* pk = reinterpret_cast<float*>(sm.cnt);        // kCap floats (cnt and mass)
  float* qk = reinterpret_cast<float*>(sm.ckey);       // reuses the keys once p is formed
  const float zk = sm.zk;
  for (int r = tid; r < nk; r += kThreads) {
    const float e = expf(key_float(sm.ckey[r]) - xmax);
    pk[r] = __fdiv_rn(e, zk);
  }
  __syncthreads();
  for (int r = tid; r < nk; r += kThreads) qk[r] = __ldg(qrow + sm.cid[r]);
  __syncthreads();
  if (tid < 32) {
    int outcome = 0;
    for (int c = i + 1; c < T && outcome == 0; ++c) {
      if (sm.par[c] != i) continue;
      const int x = sm.tok[c];
      if (x < 0 || x >= V) continue;               // reported by the window pass
      float px = 0.f;
      for (int r = lane; r < nk; r += 32)
        if (sm.cid[r] == x) px = pk[r];
      px = warp_sum(px);                           // at most one lane holds x
      if (u_accept[c] * __ldg(qrow + x) < px) {
        outcome = c;
        break;
      }
      float part = 0.f;
      for (int r = lane; r < nk; r += 32) part += fmaxf(pk[r] - qk[r], 0.f);
      const float S = warp_sum(part);
      if (S > 0.f)
        for (int r = lane; r < nk; r += 32) pk[r] = __fdiv_rn(fmaxf(pk[r] - qk[r], 0.f), S);
      __syncwarp();
    }
    if (outcome == 0 && nk <= kSparseBonus) {
      // bonus: the smallest token id whose cumulative mass in id order
      // exceeds u * total; cum(r) sums the kept tokens with id <= cid[r]
      float tot = 0.f;
      for (int r = lane; r < nk; r += 32) tot += pk[r];
      tot = warp_sum(tot);
      const float target = u_draw[i] * tot;
      int pick = 0x7FFFFFFF, last = -1;
      for (int r = lane; r < nk; r += 32) {
        const int id = sm.cid[r];
        if (pk[r] > 0.f) last = max(last, id);
        float cum = 0.f;
        for (int r2 = 0; r2 < nk; ++r2)
          if (sm.cid[r2] <= id) cum += pk[r2];
        if (pk[r] > 0.f && cum > target) pick = min(pick, id);
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        pick = min(pick, __shfl_xor_sync(0xffffffffu, pick, o));
        last = max(last, __shfl_xor_sync(0xffffffffu, last, o));
      }
      // rounding can leave the target past the last cumulative sum
      outcome = -1 - (pick != 0x7FFFFFFF ? pick : last);
    }
    if (lane == 0) sm.outcome = outcome;
  }
  __syncthreads();
  if (sm.outcome != 0) return sm.outcome;
  // no child accepted and a large kept set: the row p over the vocabulary
  for (int t = tid; t < V; t += kThreads) xs[t] = 0.f;
  __syncthreads();
  for (int r = tid; r < nk; r += kThreads) xs[sm.cid[r]] = pk[r];
  __syncthreads();
  return bonus_dense(i, V, xs, u_draw, sm);
}

// The whole vocabulary row: p is materialised over x' in place (xs), each
// rejection is a block-wide pass, the bonus a block-wide scan in id order.
__device__ int reject_dense(int i, int T, int V, float xmax, float min_p, bool by_cut,
                            uint32_t cut_key, uint32_t cut_rid, float ZK, float* __restrict__ xs,
                            const float* __restrict__ qrow, const float* __restrict__ u_accept,
                            const float* __restrict__ u_draw, SampleSmem& sm) {
  const int tid = threadIdx.x;
  // p(t) = kept(t) ? e_t / ZK : 0, kept = rank at or above the cut token
  // (or, without a top-p cut, e_t >= min_p)
  for (int t = tid; t < V; t += kThreads) {
    const float x = xs[t];
    const float e = expf(x - xmax);
    bool kept;
    if (by_cut) {
      const uint32_t k = float_key(x), rid = kIdMask - (uint32_t)t;
      kept = k > cut_key || (k == cut_key && rid >= cut_rid);
    } else {
      kept = e >= min_p;
    }
    xs[t] = kept ? __fdiv_rn(e, ZK) : 0.f;
  }
  __syncthreads();
  int outcome = 0;
  for (int c = i + 1; c < T; ++c) {
    if (sm.par[c] != i) continue;
    const int x = sm.tok[c];
    if (x < 0 || x >= V) continue;
    // every thread reads the same two values after the barrier above
    if (u_accept[c] * __ldg(qrow + x) < xs[x]) {
      outcome = c;
      break;
    }
    float part = 0.f;
    for (int t = tid; t < V; t += kThreads) part += fmaxf(xs[t] - __ldg(qrow + t), 0.f);
    const float S = block_sum(part, sm);
    if (S > 0.f)
      for (int t = tid; t < V; t += kThreads)
        xs[t] = __fdiv_rn(fmaxf(xs[t] - __ldg(qrow + t), 0.f), S);
    __syncthreads();
  }
  if (outcome != 0) return outcome;
  return bonus_dense(i, V, xs, u_draw, sm);
}

__global__ void __launch_bounds__(kThreads, 2)
sample_accept_kernel(const float* __restrict__ logits, const int32_t* __restrict__ tree_tokens,
                     const int32_t* __restrict__ parents, int T, const int32_t* __restrict__ prior,
                     int n_prior, int W, int V, float penalty, float temperature, float top_p,
                     float min_p, int mode, float eta_eps, float eta_alpha,
                     const float* __restrict__ uniforms, int32_t* sampled,
                     int32_t* __restrict__ path, int32_t* __restrict__ n_path,
                     int32_t* __restrict__ bonus, SampleWs ws,
                     const float* __restrict__ q_draft, const float* __restrict__ u_draw,
                     int32_t* status) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  // mode bit 0: eta-sampling pool instead of top-p / min-p; bit 1: literal
  // CTRL penalty (every windowed logit divided by the penalty); bit 2:
  // rejection-sampling acceptance against the draft rows q_draft
  // (`uniforms` are then the per-child acceptance uniforms)
  const bool eta_mode = (mode & 1) != 0;
  const bool literal = (mode & 2) != 0;
  const bool reject = (mode & 4) != 0;
  SampleSmem& sm = *reinterpret_cast<SampleSmem*>(smem_raw);
  uint32_t* bitmap = reinterpret_cast<uint32_t*>(smem_raw + sizeof(SampleSmem));
  const int part = blockIdx.x, i = blockIdx.y, tid = threadIdx.x;
  const int lane = tid & 31;
  const int nwords = (V + 31) / 32;
  for (int w = tid; w < nwords; w += kThreads) bitmap[w] = 0u;
  // the window's committed tokens lie in prior[n_prior - W, n_prior)
  // whatever the root path's length: loaded with the tree, ahead of the
  // path walk (two tokens a thread cover W <= 1024)
  constexpr int kPre = 2;
  const int plo = n_prior > W ? n_prior - W : 0;
  int pre[kPre];
#pragma unroll
  for (int k = 0; k < kPre; ++k) {
    const int c = plo + tid + k * kThreads;
    pre[k] = c < n_prior ? prior[c] : 0;
  }
  if (tid < T) {
    sm.par[tid] = parents[tid];
    sm.tok[tid] = tree_tokens[tid];
  }
  __syncthreads();
  if (tid == 0) {
    // drafted tokens on the root path of node i, root excluded, root first
    int tmp[64], n = 0, a = i;
    bool ok = true;
    while (a > 0 && n < 64) {
      tmp[n++] = a;
      int p = sm.par[a];
      if (p < 0 || p >= a) {
        ok = false;
        break;
      }
      a = p;
    }
    if (!ok || a != 0) {
      set_status(status, TS_ERR_INVALID_ARG);
      n = 0;
    }
    for (int x = 0; x < n; ++x) sm.ptok[x] = sm.tok[tmp[n - 1 - x]];
    sm.plen = n;
    sm.ncand = 0;
  }
  __syncthreads();
  // window = last W tokens of prior ++ path tokens: c in [start, total)
  const int total = n_prior + sm.plen;
  const int start = total > W ? total - W : 0;
  auto mark = [&](int t) {
    if (t < 0 || t >= V)
      set_status(status, TS_ERR_INVALID_ARG);
    else
      atomicOr(&bitmap[t >> 5], 1u << (t & 31));
  };
#pragma unroll
  for (int k = 0; k < kPre; ++k) {
    const int c = plo + tid + k * kThreads;
    if (c >= start && c < n_prior) mark(pre[k]);
  }
  for (int c = plo + kPre * kThreads + tid; c < n_prior; c += kThreads)
    if (c >= start) mark(prior[c]);
  for (int c = max(start, n_prior) + tid; c < total; c += kThreads) mark(sm.ptok[c - n_prior]);
  __syncthreads();

  // this CTA's slice of the vocabulary: x' = penalised / tempered logits
  // slices are whole float4s when rows are 16-byte aligned (V % 4 == 0)
  const bool vec = (V & 3) == 0;
  int per = (V + kParts - 1) / kParts;
  if (vec) per = (per + 3) & ~3;
  const int t0 = min(V, part * per), t1 = min(V, t0 + per);
  const float* x_in = logits + (size_t)i * V;
  float* xs = ws.xs + (size_t)i * V;
  const bool unit_temp = temperature == 1.0f;     // x / 1 is x exactly
  auto xprime_pen = [&](float x, uint32_t pen) {
    if (pen) x = (literal || x > 0.f) ? __fdiv_rn(x, penalty) : __fmul_rn(x, penalty);
    if (!unit_temp) x = __fdiv_rn(x, temperature);
    return x;
  };
  auto xprime = [&](float x, int t) { return xprime_pen(x, (bitmap[t >> 5] >> (t & 31)) & 1u); };
  float lmax = -INFINITY;
  if (vec) {
    // kBatch float4 loads of a thread in flight together, then their x'
    const float4* in4 = reinterpret_cast<const float4*>(x_in);
    float4* xs4 = reinterpret_cast<float4*>(xs);
    for (int q0 = t0 / 4 + tid; q0 < t1 / 4; q0 += kThreads * kBatch) {
      float4 a[kBatch];
#pragma unroll
      for (int b = 0; b < kBatch; ++b) {
        const int q = q0 + b * kThreads;
        if (q < t1 / 4) a[b] = __ldcs(in4 + q);
      }
#pragma unroll
      for (int b = 0; b < kBatch; ++b) {
        const int q = q0 + b * kThreads;
        if (q < t1 / 4) {
          const int t = 4 * q;
          // the window bits of tokens t .. t+3 (t is a multiple of 4: one word)
          const uint32_t pb = bitmap[t >> 5] >> (t & 31);
          a[b].x = xprime_pen(a[b].x, pb & 1u);
          a[b].y = xprime_pen(a[b].y, (pb >> 1) & 1u);
          a[b].z = xprime_pen(a[b].z, (pb >> 2) & 1u);
          a[b].w = xprime_pen(a[b].w, (pb >> 3) & 1u);
          xs4[q] = a[b];
          lmax = fmaxf(lmax, fmaxf(fmaxf(a[b].x, a[b].y), fmaxf(a[b].z, a[b].w)));
        }
      }
    }
  } else {
    for (int t = t0 + tid; t < t1; t += kThreads) {
      const float x = xprime(x_in[t], t);
      xs[t] = x;
      lmax = fmaxf(lmax, x);
    }
  }
  const float mc = block_max(lmax, sm);
  // Z_c and the slice's tokens with exp(x' - m_c) >= min_p (each thread
  // rereads the values it wrote)
  uint2* cand = ws.cand + ((size_t)i * kParts + part) * kCapPart;
  float z = 0.f, se = 0.f;
  // Z_c (and the entropy term) with the fast exponential: its error, below
  // 1e-6 relative where a token carries mass, is under the fp32 rounding of
  // the sum itself.  The candidate test is only a superset filter, loosened
  // by 2^-16 for that error: the merge re-tests every candidate with expf.
  const float min_p_lo = min_p * (1.0f - 1.0f / 65536.0f);
  auto accumulate = [&](float x) -> float {
    const float e = __expf(x - mc);
    z += e;
    if (eta_mode) se += e * (x - mc);   // entropy term
    return e;
  };
  // eta's threshold is only known after the merge: the last CTA scans
  auto is_cand = [&](bool valid, float e) { return valid && !eta_mode && e >= min_p_lo; };
  auto append = [&](bool in, float x, int t) {
    const unsigned m = __ballot_sync(0xffffffffu, in);
    if (m) {
      int base = 0;
      if (lane == __ffs(m) - 1) base = atomicAdd(&sm.ncand, __popc(m));
      base = __shfl_sync(0xffffffffu, base, __ffs(m) - 1);
      const int slot = base + __popc(m & ((1u << lane) - 1));
      if (in && slot < kCapPart) cand[slot] = make_uint2(float_key(x), (uint32_t)t);
    }
  };
  if (vec) {
    // this thread's own x' values (it wrote them), kBatch loads in flight
    const float4* xs4 = reinterpret_cast<const float4*>(xs);
    for (int b0 = t0 / 4; b0 < t1 / 4; b0 += kThreads * kBatch) {
      float4 a[kBatch];
#pragma unroll
      for (int b = 0; b < kBatch; ++b) {
        const int q = b0 + b * kThreads + tid;
        a[b] = q < t1 / 4 ? xs4[q] : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int b = 0; b < kBatch; ++b) {
        const int q = b0 + b * kThreads + tid;
        const bool valid = q < t1 / 4;
        float e0 = 0.f, e1 = 0.f, e2 = 0.f, e3 = 0.f;
        if (valid) {
          e0 = accumulate(a[b].x);
          e1 = accumulate(a[b].y);
          e2 = accumulate(a[b].z);
          e3 = accumulate(a[b].w);
        }
        const bool c0 = is_cand(valid, e0), c1 = is_cand(valid, e1);
        const bool c2 = is_cand(valid, e2), c3 = is_cand(valid, e3);
        // candidates are rare: one vote for the warp's four tokens a lane,
        // then the per-token appends only where some lane has one
        if (__any_sync(0xffffffffu, c0 || c1 || c2 || c3)) {
          append(c0, a[b].x, 4 * q);
          append(c1, a[b].y, 4 * q + 1);
          append(c2, a[b].z, 4 * q + 2);
          append(c3, a[b].w, 4 * q + 3);
        }
      }
    }
  } else {
    for (int b0 = t0; b0 < t1; b0 += kThreads) {
      const int t = b0 + tid;
      const bool valid = t < t1;
      const float x = valid ? xs[t] : 0.f;
      const float e = valid ? accumulate(x) : 0.f;
      append(is_cand(valid, e), x, t);
    }
  }
  const float zc = block_sum(z, sm);
  const float sc = eta_mode ? block_sum(se, sm) : 0.f;
  if (tid == 0) {
    ws.stat[i * kParts + part] = PartStat{mc, zc, sm.ncand, sc};
    __threadfence();
    sm.last = atomicAdd(&ws.node_ticket[i], 1) == kParts - 1;
  }
  __syncthreads();
  if (!sm.last) return;

  // ---- last CTA of node i: merge the slices
  // the node's uniform (an input) is loaded now, off the draw's critical path
  const float u_node = reject ? 0.f : uniforms[i];
  __threadfence();
  const volatile PartStat* vst = ws.stat + i * kParts;
  float xmax = -INFINITY;
  bool overflow = false;
  // the slices' candidate counts, and where each list starts in their
  // concatenation
  int cat_off[kParts + 1];
  cat_off[0] = 0;
#pragma unroll
  for (int p = 0; p < kParts; ++p) {
    const int np_ = vst[p].n;
    xmax = fmaxf(xmax, vst[p].m);
    overflow |= np_ > kCapPart;
    cat_off[p + 1] = cat_off[p] + np_;
  }
  float Z = 0.f, Sx = 0.f;
  for (int p = 0; p < kParts; ++p) {
    const float m = vst[p].m;
    if (m != -INFINITY) {
      const float f = expf(m - xmax);
      Z += vst[p].z * f;
      Sx += (vst[p].s + vst[p].z * (m - xmax)) * f;
    }
  }
  // min-p keeps e >= min_p (relative to the maximum).  eta keeps
  // p >= eta = min(eps, alpha exp(-H)), i.e. e >= eta Z, with the entropy
  // H = ln Z - sum e (x' - max) / Z; it needs the full scan below.
  float thr = min_p;
  if (eta_mode) {
    const float H = logf(Z) - Sx / Z;
    thr = fminf(eta_eps, eta_alpha * expf(-H)) * Z;
    overflow = true;
  }
  if (tid == 0) {
    sm.ncand = 0;
    ws.node_ticket[i] = 0;
  }
  __syncthreads();
  // the node's min-p set {e >= min_p}, e = exp(x' - max x'), from the slices' supersets
  float zmin = 0.f;
  int nmin = 0;
  // the node's pool, compacted by the row scan below (the slices' candidate
  // lists there are not read on that path)
  uint2* pool = ws.cand + (size_t)i * kPool;
  if (!overflow) {
    // one pass over the concatenation of the slices' lists (their loads in
    // flight together, not slice after slice); the members' order in the
    // shared list does not matter, it is sorted below
    const int ntot = cat_off[kParts];
    for (int b0 = 0; b0 < ntot; b0 += kThreads) {
      const int r = b0 + tid;
      const bool have = r < ntot;
      uint2 c = make_uint2(0u, 0u);
      float e = 0.f;
      if (have) {
        int p = 0, off = 0;
#pragma unroll
        for (int x = 1; x < kParts; ++x)
          if (r >= cat_off[x]) {
            p = x;
            off = cat_off[x];
          }
        c = __ldcg(ws.cand + ((size_t)i * kParts + p) * kCapPart + (r - off));
        e = expf(key_float(c.x) - xmax);
      }
      const bool in = have && e >= min_p;
      if (in) {
        zmin += e;
        ++nmin;
      }
      const unsigned m = __ballot_sync(0xffffffffu, in);
      if (m) {
        int base = 0;
        if (lane == __ffs(m) - 1) base = atomicAdd(&sm.ncand, __popc(m));
        base = __shfl_sync(0xffffffffu, base, __ffs(m) - 1);
        const int slot = base + __popc(m & ((1u << lane) - 1));
        if (in && slot < kCap) {
          sm.ckey[slot] = c.x;
          sm.cid[slot] = (int32_t)c.y;
        }
      }
    }
  } else {
    // full scan of the node's x' (a slice overflowed, or eta); members
    // are collected while they fit.  kScan loads of a thread are in flight
    // together: the ballots between tokens would otherwise hold every load
    // behind the previous one.
    for (int c0 = 0; c0 < V; c0 += kThreads * kScan) {
      float xv[kScan];
#pragma unroll
      for (int u = 0; u < kScan; ++u) {
        const int t = c0 + u * kThreads + tid;
        xv[u] = t < V ? __ldcg(xs + t) : 0.f;
      }
#pragma unroll
      for (int u = 0; u < kScan; ++u) {
        const int t = c0 + u * kThreads + tid;
        const float x = xv[u];
        const float e = t < V ? expf(x - xmax) : 0.f;
        const bool in = t < V && e >= thr;
        if (in) {
          zmin += e;
          ++nmin;
        }
        const unsigned m = __ballot_sync(0xffffffffu, in);
        if (m) {
          int base = 0;
          if (lane == __ffs(m) - 1) base = atomicAdd(&sm.ncand, __popc(m));
          base = __shfl_sync(0xffffffffu, base, __ffs(m) - 1);
          const int slot = base + __popc(m & ((1u << lane) - 1));
          if (in && slot < kCap) {
            sm.ckey[slot] = float_key(x);
            sm.cid[slot] = t;
          }
          if (in && slot < kPool) pool[slot] = make_uint2(float_key(x), (uint32_t)t);
        }
      }
    }
  }
  float Zmin = block_sum(zmin, sm);
  int n_minp = block_sum_int(nmin, sm);
  const int n_minp_seen = n_minp;   // members the scan counted (before the min_p > 1 rule)
  int token;
  if (n_minp >= 1 && n_minp <= kCap) {
    // ---- fast path: the kept set is a rank prefix inside the min-p set.
    // Sort the candidates by (x' desc, id asc), prefix-sum their e in rank
    // order, cut at top-p (first inclusive mass > top_p*Z), draw (first
    // inclusive mass > u * kept mass).
    const float tp = (eta_mode || top_p >= 1.0f) ? INFINITY : top_p * Z;   // eta: no top-p cut
    if (n_minp <= kThreads) {
      // one candidate a thread.  (key, id) is a total order, so a
      // candidate's count of the candidates ranked before it is its sorted
      // position: the permutation a sorting network gives, with no network
      uint32_t ck = 0u;
      int32_t cv = 0;
      int rank = 0;
      const bool mine = tid < n_minp;
      if (mine) {
        ck = sm.ckey[tid];
        cv = sm.cid[tid];
        for (int j = 0; j < n_minp; ++j) {
          const uint32_t kj = sm.ckey[j];
          const int32_t ij = sm.cid[j];
          rank += (kj > ck || (kj == ck && ij < cv)) ? 1 : 0;
        }
      }
      if (tid == 0) {
        sm.cnt[0] = n_minp;       // first rank past the top-p mass (none yet)
        sm.cnt[1] = 0x7FFFFFFF;   // first kept rank past the draw's target
      }
      __syncthreads();
      if (mine) {
        sm.ckey[rank] = ck;
        sm.cid[rank] = cv;
      }
      __syncthreads();
      // inclusive masses in rank order, each an fp32 sum formed exactly as
      // one warp walking 32 ranks at a time forms it: every 32-rank chunk
      // scanned by shuffles, plus the total of the chunks before it, carried
      // chunk after chunk (the total of a chunk is its last lane's scan)
      const int w = tid >> 5, nchunk = (n_minp + 31) >> 5;
      float* chunk_tot = sm.mass + kThreads;        // [kThreads / 32]
      float* chunk_run = chunk_tot + 32;            // [kThreads / 32], then the whole total
      float incl = 0.f;
      if (w < nchunk) {
        incl = mine ? expf(key_float(sm.ckey[tid]) - xmax) : 0.f;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const float y = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += y;
        }
        if (lane == 31) chunk_tot[w] = incl;
      }
      __syncthreads();
      if (tid == 0) {
        float run = 0.f;
        for (int c = 0; c < nchunk; ++c) {
          chunk_run[c] = run;
          run = chunk_tot[c] + run;
        }
        chunk_run[32] = run;
      }
      __syncthreads();
      if (w < nchunk) incl += chunk_run[w];
      if (mine) {
        sm.mass[tid] = incl;
        if (incl > tp) atomicMin(&sm.cnt[0], tid);
      }
      __syncthreads();
      const int hit = sm.cnt[0];
      const int k_keep = hit < n_minp ? hit + 1 : n_minp;
      // top-p keeps the whole min-p set: the kept mass is the last chunk's
      // carried total
      const float zk = hit < n_minp ? sm.mass[hit] : chunk_run[32];
      const float target = reject ? -1.f : u_node * zk;
      if (tid < k_keep && incl > target) atomicMin(&sm.cnt[1], tid);
      __syncthreads();
      if (tid == 0) {
        const int d = sm.cnt[1];
        const int pick = d < k_keep ? d : k_keep - 1;
        sm.nkeep = k_keep;
        sm.zk = zk;
        sm.kpre = (uint32_t)sm.cid[pick];
      }
    } else {
      int np = 32;
      while (np < n_minp) np <<= 1;
      for (int q = n_minp + tid; q < np; q += kThreads) {
        sm.ckey[q] = 0u;            // below every real key
        sm.cid[q] = 0x7FFFFFFF;
      }
      __syncthreads();
      for (int size = 2; size <= np; size <<= 1) {
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
          for (int q = tid; q < np; q += kThreads) {
            const int qx = q ^ stride;
            if (qx > q) {
              const uint32_t ka = sm.ckey[q], kb = sm.ckey[qx];
              const int32_t ia = sm.cid[q], ib = sm.cid[qx];
              // a ranks before b: larger key, then smaller id
              const bool a_first = ka > kb || (ka == kb && ia < ib);
              const bool desc = (q & size) == 0;
              if (desc != a_first) {
                sm.ckey[q] = kb;
                sm.ckey[qx] = ka;
                sm.cid[q] = ib;
                sm.cid[qx] = ia;
              }
            }
          }
          __syncthreads();
        }
      }
      // the rank walks as a block pass, as for the smaller sets, with warp
      // w taking chunks w, w + 16, ... (the same fp32 sums: chunk scans by
      // shuffles, their totals carried chunk after chunk)
      constexpr int kWarps = kThreads / 32, kRounds = kCap / kThreads;
      const int w = tid >> 5, nchunk = (n_minp + 31) >> 5;
      float* chunk_tot = sm.mass;                 // [kCap / 32]
      float* chunk_run = sm.mass + kCap / 32;     // [kCap / 32], then the whole total
      float* zk_at_hit = chunk_run + kCap / 32 + 1;
      if (tid == 0) {
        sm.cnt[0] = n_minp;
        sm.cnt[1] = 0x7FFFFFFF;
      }
      float incl[kRounds];
#pragma unroll
      for (int k = 0; k < kRounds; ++k) {
        const int c = w + k * kWarps;
        incl[k] = 0.f;
        if (c < nchunk) {   // warp-uniform
          const int r = 32 * c + lane;
          float v = r < n_minp ? expf(key_float(sm.ckey[r]) - xmax) : 0.f;
#pragma unroll
          for (int o = 1; o < 32; o <<= 1) {
            const float y = __shfl_up_sync(0xffffffffu, v, o);
            if (lane >= o) v += y;
          }
          if (lane == 31) chunk_tot[c] = v;
          incl[k] = v;
        }
      }
      __syncthreads();
      if (tid == 0) {
        float run = 0.f;
        for (int c = 0; c < nchunk; ++c) {
          chunk_run[c] = run;
          run = chunk_tot[c] + run;
        }
        chunk_run[kCap / 32] = run;
      }
      __syncthreads();
#pragma unroll
      for (int k = 0; k < kRounds; ++k) {
        const int c = w + k * kWarps, r = 32 * c + lane;
        if (c < nchunk) {
          incl[k] += chunk_run[c];
          if (r < n_minp && incl[k] > tp) atomicMin(&sm.cnt[0], r);
        }
      }
      __syncthreads();
      const int hit = sm.cnt[0];
      const int k_keep = hit < n_minp ? hit + 1 : n_minp;
#pragma unroll
      for (int k = 0; k < kRounds; ++k)
        if (hit < n_minp && 32 * (w + k * kWarps) + lane == hit) *zk_at_hit = incl[k];
      __syncthreads();
      // top-p keeps the whole min-p set: the kept mass is the carried total
      const float zk = hit < n_minp ? *zk_at_hit : chunk_run[kCap / 32];
      const float target = reject ? -1.f : u_node * zk;
#pragma unroll
      for (int k = 0; k < kRounds; ++k) {
        const int r = 32 * (w + k * kWarps) + lane;
        if (r < k_keep && incl[k] > target) atomicMin(&sm.cnt[1], r);
      }
      __syncthreads();
      if (tid == 0) {
        const int d = sm.cnt[1];
        const int pick = d < k_keep ? d : k_keep - 1;
        sm.nkeep = k_keep;
        sm.zk = zk;
        sm.kpre = (uint32_t)sm.cid[pick];
      }
    }
    __syncthreads();
    token = reject ? reject_sparse(i, T, V, xmax, q_draft + (size_t)i * V, uniforms, u_draw, xs, sm)
                   : (int)sm.kpre;
    __syncthreads();
  } else {
    // ---- general path: radix descent with (count, mass) histograms
    if (n_minp == 0) {   // min_p > 1: only rank 0 (e = 1) survives
      n_minp = 1;
      Zmin = 1.f;
    }
    int k_keep = n_minp;
    float ZK = Zmin;
    // kept tokens: the rank prefix up to the top-p cut token, else the
    // min-p set (e >= min_p); 50-bit rank key (x' key, reversed id)
    uint32_t cut_key = 0u, cut_rid = 0u;
    bool by_cut = false;
    if (!eta_mode && top_p < 1.0f) {
      const Found f1 = radix_find<false>(xs, V, nullptr, 0, xmax, kMassGT, top_p * Z, 0, 0.f, sm);
      k_keep = min(n_minp, f1.rank + 1);
      ZK = (k_keep == f1.rank + 1) ? f1.cum_incl : Zmin;
      if (k_keep == f1.rank + 1) {
        by_cut = true;
        cut_key = float_key(xs[f1.id]);
        cut_rid = kIdMask - (uint32_t)f1.id;
      }
    }
    if (reject) {
      token = reject_dense(i, T, V, xmax, min_p, by_cut, cut_key, cut_rid, ZK, xs,
                           q_draft + (size_t)i * V, uniforms, u_draw, sm);
    } else {
      const float u = uniforms[i];
      // the draw lies inside the kept pool, a rank prefix of {e >= thr}
      // (with thr above 1 the pool is rank 0 alone, e = 1): the descent
      // reads the pool compacted by the scan when it holds all of it, else
      // the row, leaving out the tokens below the pool
      const float skip = fminf(thr, 1.f);
      const bool listed = overflow && n_minp_seen >= 1 && n_minp_seen <= kPool;
      const uint2* lst = listed ? pool : nullptr;
      const int nl = listed ? n_minp_seen : 0;
      auto find = [&](int mode, float mass, int rank) {
        return listed ? radix_find<true>(xs, V, lst, nl, xmax, mode, mass, rank, 0.f, sm)
                      : radix_find<false>(xs, V, nullptr, 0, xmax, mode, mass, rank, skip, sm);
      };
      Found f2 = find(kMassGT, u * ZK, 0);
      if (f2.rank >= k_keep) f2 = find(kRank, 0.f, k_keep - 1);
      token = f2.id;
    }
  }

  // publish this node's draw; the last CTA walks the tree
  if (tid == 0) {
    sampled[i] = token;
    __threadfence();
    int prev = atomicAdd(ws.counter, 1);
    sm.last = (prev == T - 1);
  }
  __syncthreads();
  if (!sm.last) return;
  // the last node: every draw is published; stage them, then walk the tree
  // in shared memory
  __threadfence();
  if (tid < T) sm.smp[tid] = __ldcg(sampled + tid);
  if (tid == 0) sm.best = 0;
  __syncthreads();
  if (reject) {
    // outcome of node n: an accepted child c >= 1, or -1 - (bonus token)
    if (tid == 0) {
      int node = 0, n = 1;
      path[0] = 0;
      while (sm.smp[node] >= 1 && n < T) {
        node = sm.smp[node];
        path[n++] = node;
      }
      *n_path = n;
      *bonus = sm.smp[node] >= 1 ? -1 : -1 - sm.smp[node];
      *ws.counter = 0;
    }
    return;
  }
  // node c is accepted iff every node a on its root path (root excluded)
  // carries the token its parent drew; the deepest accepted node wins, ties
  // to the smaller index: the largest key depth * 256 + (255 - c)
  if (tid < T) {
    int a = tid, depth = 0;
    bool acc = true;
    while (a > 0 && depth < 64) {
      const int p = sm.par[a];
      if (p < 0 || p >= a) {
        acc = false;
        break;
      }
      acc = acc && sm.tok[a] == sm.smp[p];
      a = p;
      ++depth;
    }
    if (acc) atomicMax(&sm.best, depth * 256 + (255 - tid));
  }
  __syncthreads();
  if (tid == 0) {
    const int best = 255 - (sm.best & 255), n = (sm.best >> 8) + 1;
    int a = best;
    for (int d = n - 1; d >= 0; --d) {
      path[d] = a;
      a = sm.par[a];
    }
    *n_path = n;
    *bonus = sm.smp[best];
    *ws.counter = 0;
  }
}

// Rows L+path[t] -> L+t of one KV head (t = 1..n-1).  The sources are staged
// in shared memory first, so overlapping moves are safe.
template <int D>
__device__ __forceinline__ void commit_head(__nv_bfloat16* __restrict__ k,
                                            __nv_bfloat16* __restrict__ v, int kv, int64_t L,
                                            int64_t L_cap, int T, const int32_t* __restrict__ path,
                                            const int32_t* __restrict__ n_path, int32_t* status) {
  constexpr int V16 = D / 8;
  __shared__ uint4 kb[63][V16], vb[63][V16];
  const int n = *n_path;
  if (n < 1 || n > T) {
    if (threadIdx.x == 0) set_status(status, TS_ERR_INVALID_ARG);
    return;
  }
  uint4* kh = reinterpret_cast<uint4*>(k + (size_t)kv * L_cap * D);
  uint4* vh = reinterpret_cast<uint4*>(v + (size_t)kv * L_cap * D);
  bool bad = false;
  for (int e = threadIdx.x; e < (n - 1) * V16; e += blockDim.x) {
    int t = e / V16 + 1, x = e % V16;
    int src = path[t];
    if (src < t || src >= T) {
      bad = true;
      continue;
    }
    kb[t - 1][x] = kh[(L + src) * V16 + x];
    vb[t - 1][x] = vh[(L + src) * V16 + x];
  }
  bad = __syncthreads_or(bad);
  if (bad) {
    if (threadIdx.x == 0) set_status(status, TS_ERR_INVALID_ARG);
    return;
  }
  for (int e = threadIdx.x; e < (n - 1) * V16; e += blockDim.x) {
    int t = e / V16 + 1, x = e % V16;
    kh[(L + t) * V16 + x] = kb[t - 1][x];
    vh[(L + t) * V16 + x] = vb[t - 1][x];
  }
}

template <int D>
__global__ void kv_commit_kernel(__nv_bfloat16* __restrict__ k, __nv_bfloat16* __restrict__ v,
                                 int64_t L, int64_t L_cap, int T, const int32_t* __restrict__ path,
                                 const int32_t* __restrict__ n_path, int32_t* status) {
  commit_head<D>(k, v, blockIdx.x, L, L_cap, T, path, n_path, status);
}

// every layer in one launch: CTA (KV head, layer), per-layer caches from
// device arrays of pointers
template <int D>
__global__ void kv_commit_batched_kernel(__nv_bfloat16* const* __restrict__ ks,
                                         __nv_bfloat16* const* __restrict__ vs, int64_t L,
                                         int64_t L_cap, int T, const int32_t* __restrict__ path,
                                         const int32_t* __restrict__ n_path, int32_t* status) {
  commit_head<D>(ks[blockIdx.y], vs[blockIdx.y], blockIdx.x, L, L_cap, T, path, n_path, status);
}

// The draft tree's own K/V rows into every layer's cache: rows [L, L+T) of
// KV head kv of layer l come from the packed arrays [n_layers][Hkv][T][D].
// CTA (KV head, layer); 16-byte copies (rows are 128 or 256 bytes).  With an
// fp16 V cache (kVF16) each bf16 value of v is rounded to the nearest fp16
// (exact for normal values below 65504 in magnitude); larger magnitudes
// saturate to +-65504 and TS_ERR_UNSUPPORTED goes to the status word.
template <int D, bool kVF16>
__global__ void kv_append_batched_kernel(__nv_bfloat16* const* __restrict__ ks,
                                         __nv_bfloat16* const* __restrict__ vs,
                                         const __nv_bfloat16* __restrict__ krows,
                                         const __nv_bfloat16* __restrict__ vrows, int64_t L,
                                         int64_t L_cap, int T, int32_t* status) {
  constexpr int V16 = D / 8;
  const int kv = blockIdx.x, layer = blockIdx.y, Hkv = gridDim.x;
  const size_t src = ((size_t)layer * Hkv + kv) * T * V16;
  const uint4* ksrc = reinterpret_cast<const uint4*>(krows) + src;
  const uint4* vsrc = reinterpret_cast<const uint4*>(vrows) + src;
  uint4* kdst = reinterpret_cast<uint4*>(ks[layer] + ((size_t)kv * L_cap + L) * D);
  uint4* vdst = reinterpret_cast<uint4*>(vs[layer] + ((size_t)kv * L_cap + L) * D);
  bool over = false;
  for (int e = threadIdx.x; e < T * V16; e += blockDim.x) {
    kdst[e] = ksrc[e];
    uint4 u = vsrc[e];
    if (kVF16) {
      uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
      for (int x = 0; x < 4; ++x) {
        const float lo = __uint_as_float(w[x] << 16), hi = __uint_as_float(w[x] & 0xFFFF0000u);
        over |= !(fabsf(lo) <= 65504.f) || !(fabsf(hi) <= 65504.f);
        w[x] = ptx::pack_f16x2_sat(lo, hi);   // the rounding of the in-kernel conversion
      }
      u = make_uint4(w[0], w[1], w[2], w[3]);
    }
    vdst[e] = u;
  }
  if (kVF16 && over && status) set_status(status, TS_ERR_UNSUPPORTED);
}

}  // namespace

size_t sample_ws_bytes(int T, int V) {
  return kCounterBytes + a256s((size_t)T * kParts * sizeof(PartStat)) +
         a256s((size_t)T * kParts * kCapPart * sizeof(uint2)) + a256s((size_t)T * V * sizeof(float));
}

// Rejection mode: the sampling workspace of up to 64 nodes, then the nodes'
// outcomes (64 int32).
size_t reject_ws_bytes(int V) { return sample_ws_bytes(64, V) + 256; }

int launch_reject_accept(const float* logits, const float* q, const int32_t* tree_tokens,
                         const int32_t* parents, int T, const int32_t* prior, int n_prior, int W,
                         int V, float penalty, float temperature, float top_p, float min_p,
                         int literal, const float* u_accept, const float* u_draw, int32_t* path,
                         int32_t* n_path, int32_t* bonus, void* ws, int32_t* status,
                         cudaStream_t st) {
  int32_t* outcome = reinterpret_cast<int32_t*>(static_cast<char*>(ws) + sample_ws_bytes(64, V));
  return launch_sample_accept(logits, tree_tokens, parents, T, prior, n_prior, W, V, penalty,
                              temperature, top_p, min_p, 4 | (literal ? 2 : 0), 0.f, 0.f,
                              u_accept, outcome, path, n_path, bonus, ws, q, u_draw, status, st);
}

int launch_sample_accept(const float* logits, const int32_t* tree_tokens, const int32_t* parents,
                         int T, const int32_t* prior, int n_prior, int W, int V, float penalty,
                         float temperature, float top_p, float min_p, int mode, float eta_eps,
                         float eta_alpha, const float* uniforms, int32_t* sampled, int32_t* path,
                         int32_t* n_path, int32_t* bonus, void* ws, const float* q_draft,
                         const float* u_draw, int32_t* status, cudaStream_t st) {
  const SampleWs w = carve_sample(ws, T);
  if (cudaMemsetAsync(ws, 0, kCounterBytes, st) != cudaSuccess)
    return launch_status("sample counter reset");
  size_t smem = sizeof(SampleSmem) + (size_t)((V + 31) / 32) * sizeof(uint32_t);
  cudaFuncSetAttribute(sample_accept_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  sample_accept_kernel<<<dim3(kParts, T), kThreads, smem, st>>>(
      logits, tree_tokens, parents, T, prior, n_prior, W, V, penalty, temperature, top_p, min_p,
      mode, eta_eps, eta_alpha, uniforms, sampled, path, n_path, bonus, w, q_draft, u_draw,
      status);
  return launch_status("sample_accept_kernel");
}

int launch_kv_commit(void* k, void* v, int64_t L, int64_t L_cap, int Hkv, int d, int T,
                     const int32_t* path, const int32_t* n_path, int32_t* status,
                     cudaStream_t st) {
  auto kb = static_cast<__nv_bfloat16*>(k);
  auto vb = static_cast<__nv_bfloat16*>(v);
  if (d == 128)
    kv_commit_kernel<128><<<Hkv, 256, 0, st>>>(kb, vb, L, L_cap, T, path, n_path, status);
  else
    kv_commit_kernel<64><<<Hkv, 256, 0, st>>>(kb, vb, L, L_cap, T, path, n_path, status);
  return launch_status("kv_commit_kernel");
}

int launch_kv_commit_batched(int n_layers, void* const* k, void* const* v, int64_t L,
                             int64_t L_cap, int Hkv, int d, int T, const int32_t* path,
                             const int32_t* n_path, int32_t* status, cudaStream_t st) {
  auto kb = reinterpret_cast<__nv_bfloat16* const*>(k);
  auto vb = reinterpret_cast<__nv_bfloat16* const*>(v);
  dim3 grid(Hkv, n_layers);
  if (d == 128)
    kv_commit_batched_kernel<128><<<grid, 256, 0, st>>>(kb, vb, L, L_cap, T, path, n_path, status);
  else
    kv_commit_batched_kernel<64><<<grid, 256, 0, st>>>(kb, vb, L, L_cap, T, path, n_path, status);
  return launch_status("kv_commit_batched_kernel");
}

int launch_kv_append_batched(int n_layers, void* const* k, void* const* v, const void* krows,
                             const void* vrows, int64_t L, int64_t L_cap, int Hkv, int d, int T,
                             bool v_fp16, int32_t* status, cudaStream_t st) {
  auto kb = reinterpret_cast<__nv_bfloat16* const*>(k);
  auto vb = reinterpret_cast<__nv_bfloat16* const*>(v);
  auto kr = static_cast<const __nv_bfloat16*>(krows);
  auto vr = static_cast<const __nv_bfloat16*>(vrows);
  dim3 grid(Hkv, n_layers);
  auto go = [&](auto kern) { kern<<<grid, 256, 0, st>>>(kb, vb, kr, vr, L, L_cap, T, status); };
  if (d == 128)
    v_fp16 ? go(kv_append_batched_kernel<128, true>) : go(kv_append_batched_kernel<128, false>);
  else
    v_fp16 ? go(kv_append_batched_kernel<64, true>) : go(kv_append_batched_kernel<64, false>);
  return launch_status("kv_append_batched_kernel");
}

}  // namespace ts
