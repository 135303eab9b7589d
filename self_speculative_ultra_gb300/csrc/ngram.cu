// Token reutilization: the on-device 4-gram table and the draft-tree builder.
//
// "TokenSwift: Lossless Acceleration of Ultra Long Sequence Generation":
// §3.1 Overview (after verification the n-gram table is updated), §3.2
// Multi-token Generation and Token Reutilization (frequent n-grams supply
// extra draft candidates), §3.4 (random selection among several valid
// n-grams), §B.2 Inference Details and Table 10 (4-grams, at most k
// retrieved n-grams; k = 20 in Table 11), §4.4.1 / §B.2 (the extra heads'
// candidates form the ternary full tree [1,3,3,3]).
//
// Table (one int32 buffer, zeroed by the caller once): meta [V][2] = (count,
// oldest slot) then continuations [V][cap][3].  The 4-gram (a, b, c, d) is
// stored under a as (b, c, d); each key keeps at most `cap` distinct
// continuations in a ring, the oldest overwritten first, a repeated one
// neither duplicated nor moved.
//
// ngram_insert_kernel: one warp walks the positions in order (the per-key
//   order is what the table's contents depend on); the 32 lanes compare the
//   key's stored continuations in parallel.  A decode step inserts at most a
//   few 4-grams (the accepted path); a long prefix is a one-time cost.
// ngram_tree_kernel: one CTA: the root's continuations are selected (all of
//   them when at most k, else the k with the smallest caller-supplied random
//   keys, ties to the lower slot, by a bitonic sort of at most 64 entries),
//   then one thread builds the tree: root, the heads' tree in breadth-first
//   order, and each selected continuation merged as a path from the root.
#include "ts_common.cuh"

namespace ts {

namespace {

constexpr int kMaxCap = 64;
constexpr int kMaxNodes = 64;

__global__ void __launch_bounds__(32)
ngram_insert_kernel(int32_t* __restrict__ table, int V, int cap, const int32_t* __restrict__ tokens,
                    int n_tokens, int start, int32_t* status) {
  const int lane = threadIdx.x;
  int32_t* meta = table;
  int32_t* cont = table + (size_t)V * 2;
  for (int p = max(start, 3); p < n_tokens; ++p) {
    const int a = tokens[p - 3], b = tokens[p - 2], c = tokens[p - 1], d = tokens[p];
    if (a < 0 || a >= V || b < 0 || b >= V || c < 0 || c >= V || d < 0 || d >= V) {
      if (lane == 0) set_status(status, TS_ERR_INVALID_ARG);
      continue;
    }
    const int count = meta[2 * a], head = meta[2 * a + 1];
    bool found = false;
    for (int i = lane; i < count; i += 32) {
      const int32_t* e = cont + ((size_t)a * cap + (head + i) % cap) * 3;
      found |= e[0] == b && e[1] == c && e[2] == d;
    }
    if (__any_sync(0xffffffffu, found)) continue;
    if (lane == 0) {
      int slot;
      if (count < cap) {
        slot = (head + count) % cap;
        meta[2 * a] = count + 1;
      } else {
        slot = head;                       // the oldest continuation gives way
        meta[2 * a + 1] = (head + 1) % cap;
      }
      int32_t* e = cont + ((size_t)a * cap + slot) * 3;
      e[0] = b;
      e[1] = c;
      e[2] = d;
    }
    __syncwarp();   // the next position's reads see this insertion
  }
}

__global__ void __launch_bounds__(kMaxCap)
ngram_tree_kernel(const int32_t* __restrict__ table, int V, int cap,
                  const int32_t* __restrict__ root_token, const int32_t* __restrict__ head_topk,
                  int n_heads, int head_k, int k, const uint32_t* __restrict__ rand_keys, int T_max,
                  int32_t* __restrict__ parents, int32_t* __restrict__ tokens,
                  int32_t* __restrict__ n_nodes, int32_t* status) {
  __shared__ uint32_t s_key[kMaxCap];
  __shared__ int32_t s_slot[kMaxCap];
  __shared__ int32_t s_chain[kMaxCap][3];
  __shared__ int32_t s_par[kMaxNodes], s_tok[kMaxNodes], s_first[kMaxNodes], s_next[kMaxNodes];
  const int tid = threadIdx.x;
  const int root = *root_token;
  const bool root_ok = root >= 0 && root < V;
  const int32_t* meta = table;
  const int32_t* cont = table + (size_t)V * 2;
  const int count = root_ok ? meta[2 * root] : 0, head = root_ok ? meta[2 * root + 1] : 0;
  const int n_sel = min(count, k);
  // selection: slots ordered by (random key, slot) when more than k are stored
  s_key[tid] = (tid < count && count > k) ? rand_keys[tid] : 0xFFFFFFFFu;
  s_slot[tid] = tid < count ? tid : 0x7FFFFFFF;
  __syncthreads();
  if (count > k) {
    for (int size = 2; size <= kMaxCap; size <<= 1) {
      for (int stride = size >> 1; stride > 0; stride >>= 1) {
        const int x = tid ^ stride;
        if (x > tid) {
          const uint32_t ka = s_key[tid], kb = s_key[x];
          const int32_t sa = s_slot[tid], sb = s_slot[x];
          const bool a_first = ka < kb || (ka == kb && sa < sb);
          const bool asc = (tid & size) == 0;
          if (asc != a_first) {
            s_key[tid] = kb;
            s_key[x] = ka;
            s_slot[tid] = sb;
            s_slot[x] = sa;
          }
        }
        __syncthreads();
      }
    }
  }
  if (tid < n_sel) {
    const int32_t* e = cont + ((size_t)root * cap + (head + s_slot[tid]) % cap) * 3;
    s_chain[tid][0] = e[0];
    s_chain[tid][1] = e[1];
    s_chain[tid][2] = e[2];
  }
  __syncthreads();
  if (tid != 0) return;
  if (!root_ok) set_status(status, TS_ERR_INVALID_ARG);
  int n = 0;
  auto add = [&](int p, int tok) {
    s_par[n] = p;
    s_tok[n] = tok;
    s_first[n] = -1;
    s_next[n] = -1;
    if (p >= 0) {
      // append to the end of p's child list, keeping insertion order
      if (s_first[p] < 0) {
        s_first[p] = n;
      } else {
        int c = s_first[p];
        while (s_next[c] >= 0) c = s_next[c];
        s_next[c] = n;
      }
    }
    return n++;
  };
  add(-1, root);
  // the heads' tree, breadth-first: depth-d nodes carry head d's candidates
  int lvl_lo = 0, lvl_hi = 1;
  for (int d = 0; d < n_heads; ++d) {
    const int next_lo = n;
    for (int p = lvl_lo; p < lvl_hi; ++p)
      for (int c = 0; c < head_k && n < T_max; ++c) add(p, head_topk[d * head_k + c]);
    lvl_lo = next_lo;
    lvl_hi = n;
  }
  // the selected continuations, each merged as a path from the root
  for (int i = 0; i < n_sel; ++i) {
    int cur = 0;
    for (int x = 0; x < 3; ++x) {
      const int tok = s_chain[i][x];
      int hit = -1;
      for (int c = s_first[cur]; c >= 0; c = s_next[c])
        if (s_tok[c] == tok) {
          hit = c;
          break;
        }
      if (hit < 0) {
        if (n >= T_max) break;
        hit = add(cur, tok);
      }
      cur = hit;
    }
  }
  for (int i = 0; i < n; ++i) {
    parents[i] = s_par[i];
    tokens[i] = s_tok[i];
  }
  *n_nodes = n;
}

}  // namespace

size_t ngram_table_bytes(int V, int cap) {
  return ((size_t)V * 2 + (size_t)V * cap * 3) * sizeof(int32_t);
}

int launch_ngram_insert(int32_t* table, int V, int cap, const int32_t* tokens, int n_tokens,
                        int start, int32_t* status, cudaStream_t st) {
  if (n_tokens <= max(start, 3)) return TS_OK;
  ngram_insert_kernel<<<1, 32, 0, st>>>(table, V, cap, tokens, n_tokens, start, status);
  return launch_status("ngram_insert_kernel");
}

int launch_ngram_tree(const int32_t* table, int V, int cap, const int32_t* root_token,
                      const int32_t* head_topk, int n_heads, int head_k, int k,
                      const uint32_t* rand_keys, int T_max, int32_t* parents, int32_t* tokens,
                      int32_t* n_nodes, int32_t* status, cudaStream_t st) {
  ngram_tree_kernel<<<1, kMaxCap, 0, st>>>(table, V, cap, root_token, head_topk, n_heads, head_k, k,
                                           rand_keys, T_max, parents, tokens, n_nodes, status);
  return launch_status("ngram_tree_kernel");
}

}  // namespace ts
