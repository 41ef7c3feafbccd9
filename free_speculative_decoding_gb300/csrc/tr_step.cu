// Draft retrieval, greedy acceptance, matrix update, KV commit and the fused
// post-forward step of Token Recycling.
//
// These parts move a few hundred bytes to a few hundred KB per sequence and
// are latency-bound: one CTA (or a handful) per sequence, the tree plan in
// kernel parameters, the per-node state in shared memory.
#include "tr_internal.cuh"

namespace {

constexpr int kThreads = 256;  // >= TR_MAX_NODES: one thread per tree node

__device__ __forceinline__ unsigned ld_acquire_u32(const unsigned *p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// ---------------------------------------------------------------------------
// retrieval: one warp expands the tree level by level
// ---------------------------------------------------------------------------

// Blog "token-recycling", 完整工作流程 steps 1-2: tok[0] = root, then for each
// level l = 1..D and each node n of it, tok[n] = M[tok[parent n]][rank n].
// Reads go through L2 (ld.global.cg) because in the fused step the rows may
// have been rewritten by another CTA of the same launch.
template <typename T>
__device__ void warp_retrieve(const T *Mb, long long V, int K, const TreeDev &tree, int root, int *tok_s,
                              int32_t *out, unsigned *status) {
  const int lane = threadIdx.x & 31;
  if (lane == 0) {
    if (root < 0 || (long long)root >= V) {
      tr_flag(status, TR_DEV_BAD_TOKEN);
      root = 0;
    }
    tok_s[0] = root;
  }
  __syncwarp();
  for (int l = 1; l <= tree.D; ++l) {
    const int lo = tree.level_off[l], hi = tree.level_off[l + 1];
    for (int n = lo + lane; n < hi; n += 32) {
      const int p = tree.parent[n], r = tree.rank[n];
      long long t = (long long)__ldcg(Mb + (long long)tok_s[p] * K + r);
      if (t < 0 || t >= V) {
        tr_flag(status, TR_DEV_BAD_TOKEN);
        t = 0;
      }
      tok_s[n] = (int)t;
    }
    __syncwarp();
  }
  for (int n = lane; n < tree.N; n += 32) out[n] = tok_s[n];
}

template <typename T>
__global__ void __launch_bounds__(32) retrieve_kernel(const T *M, long long V, int K,
                                                      const __grid_constant__ TreeDev tree, const int32_t *root,
                                                      int32_t *tree_tok, unsigned *status) {
  __shared__ int tok_s[TR_MAX_NODES];
  const int b = blockIdx.x;
  warp_retrieve<T>(M + (long long)b * V * K, V, K, tree, root[b], tok_s, tree_tok + (long long)b * tree.N, status);
}

// ---------------------------------------------------------------------------
// acceptance (one block per sequence)
// ---------------------------------------------------------------------------

struct AcceptSmem {
  int tok[TR_MAX_NODES];
  int top1[TR_MAX_NODES];
  int path[TR_MAX_NODES];
  unsigned long long nomatch[2];
  int warp_best[kThreads / 32];
  int best;      // chosen node n*
  int acc_len;
  int bonus;
  int L;
  int last;
};

// Blog step 4 / hyper.ai "Method": node n (n >= 1) matches when its token is
// its parent's greedy choice; a node is acceptable when every node on its root
// path matches; the deepest acceptable node wins, then the smallest index.
__device__ void block_accept(const TreeDev &tree, AcceptSmem &s) {
  const int n = threadIdx.x;
  const int warp = n >> 5, lane = n & 31;
  bool miss = false;
  if (n < tree.N && n > 0) miss = s.tok[n] != s.top1[tree.parent[n]];
  const unsigned bal = __ballot_sync(0xffffffffu, miss);
  if (warp < 4 && lane == 0) {
    // words: warps 0,1 -> nomatch[0]; warps 2,3 -> nomatch[1]
    unsigned long long w = (unsigned long long)bal << ((warp & 1) * 32);
    atomicOr(&s.nomatch[warp >> 1], w);
  }
  __syncthreads();
  int score = -1;
  if (n < tree.N) {
    const bool ok = ((tree.anc[n][0] & s.nomatch[0]) | (tree.anc[n][1] & s.nomatch[1])) == 0ull;
    if (ok) score = ((int)tree.depth[n] << 8) | (255 - n);
  }
  score = __reduce_max_sync(0xffffffffu, score);
  if (lane == 0) s.warp_best[warp] = score;
  __syncthreads();
  if (n == 0) {
    int best = s.warp_best[0];
    for (int w = 1; w < kThreads / 32; ++w) best = max(best, s.warp_best[w]);
    const int nstar = 255 - (best & 255);
    s.best = nstar;
    s.acc_len = tree.depth[nstar];
    s.bonus = s.top1[nstar];
  }
  __syncthreads();
  if (n < tree.N) {
    const int nstar = s.best;
    if ((tree.anc[nstar][n >> 6] >> (n & 63)) & 1ull) s.path[tree.depth[n]] = n;
  }
  __syncthreads();
}

// With ids_s, every node's whole top-K row is loaded into it in the same round
// trip as the top-1 IDs.
__device__ void load_tree_state(const TreeDev &tree, const int32_t *tok, const int32_t *ids, int K, AcceptSmem &s,
                                int32_t *ids_s = nullptr) {
  const int n = threadIdx.x;
  if (n < 2) s.nomatch[n] = 0ull;
  if (n < tree.N) {
    s.tok[n] = tok[n];
    if (ids_s) {
      int32_t v[TR_MAX_K];
#pragma unroll
      for (int k = 0; k < TR_MAX_K; ++k)
        if (k < K) v[k] = ids[(long long)n * K + k];
#pragma unroll
      for (int k = 0; k < TR_MAX_K; ++k)
        if (k < K) ids_s[n * K + k] = v[k];
      s.top1[n] = v[0];
    } else {
      s.top1[n] = ids[(long long)n * K];
    }
  }
  __syncthreads();
}

__device__ void write_accept_outputs(const TreeDev &tree, const AcceptSmem &s, int b, int32_t *acc_len,
                                     int32_t *path, int32_t *committed, int32_t *bonus) {
  const int i = threadIdx.x;
  const int W = tree.D + 1;
  if (i <= tree.D) {
    if (path) path[(long long)b * W + i] = i <= s.acc_len ? s.path[i] : -1;
    if (committed) {
      int c = -1;
      if (i < s.acc_len) c = s.tok[s.path[i + 1]];
      else if (i == s.acc_len) c = s.bonus;
      committed[(long long)b * W + i] = c;
    }
  }
  if (i == 0) {
    if (acc_len) acc_len[b] = s.acc_len;
    if (bonus) bonus[b] = s.bonus;
  }
}

// ---------------------------------------------------------------------------
// update: M[tok[n]] <- ids[n] for the writing nodes, last in BFS order wins
// ---------------------------------------------------------------------------

// `writer` marks the nodes that write (all of them, or the accepted path).
// A node stores its row only if no later writing node holds the same token,
// which is what a sequential BFS-order loop of overwrites leaves behind.
template <typename T>
__device__ void block_update(T *Mb, long long V, int K, const TreeDev &tree, const int *tok_s, const bool *writer,
                             const int32_t *ids, unsigned *status) {
  const int n = threadIdx.x;
  bool w = false;
  int t = 0;
  if (n < tree.N && writer[n]) {
    t = tok_s[n];
    w = true;
    for (int m = n + 1; m < tree.N; ++m)
      if (writer[m] && tok_s[m] == t) {
        w = false;
        break;
      }
    if (w && (t < 0 || (long long)t >= V)) {
      tr_flag(status, TR_DEV_BAD_TOKEN);
      w = false;
    }
  }
  if (w) {
    T *row = Mb + (long long)t * K;
    const int32_t *src = ids + (long long)n * K;
    for (int k = 0; k < K; ++k) row[k] = (T)src[k];
  }
}

// ---------------------------------------------------------------------------
// KV commit: append the path's K/V rows at positions L..L+acc_len
// ---------------------------------------------------------------------------

__device__ void block_commit(const uint4 *Kt, const uint4 *Vt, uint4 *Kc, uint4 *Vc, int N, int Hkv, int cap,
                             int d16, int b, int L, int acc, const int *path, int h_lo, int h_hi) {
  const int nh = h_hi - h_lo;
  const long long total = (long long)(acc + 1) * nh * d16;
  for (long long e = threadIdx.x; e < total; e += blockDim.x) {
    const int c = (int)(e % d16);
    const long long r = e / d16;
    const int h = h_lo + (int)(r % nh);
    const int i = (int)(r / nh);
    const int node = path[i];
    const long long src = (((long long)b * N + node) * Hkv + h) * d16 + c;
    const long long dst = (((long long)b * Hkv + h) * cap + (L + i)) * d16 + c;
    Kc[dst] = Kt[src];
    Vc[dst] = Vt[src];
  }
}

// ---------------------------------------------------------------------------
// kernels
// ---------------------------------------------------------------------------

__global__ void __launch_bounds__(kThreads) accept_kernel(const __grid_constant__ TreeDev tree, const int32_t *tree_tok,
                                                          const int32_t *ids, int K, int32_t *acc_len,
                                                          int32_t *path, int32_t *committed, int32_t *bonus) {
  __shared__ AcceptSmem s;
  const int b = blockIdx.x;
  load_tree_state(tree, tree_tok + (long long)b * tree.N, ids + (long long)b * tree.N * K, K, s);
  block_accept(tree, s);
  write_accept_outputs(tree, s, b, acc_len, path, committed, bonus);
}

template <typename T>
__global__ void __launch_bounds__(kThreads) update_kernel(T *M, long long V, int K, const __grid_constant__ TreeDev tree,
                                                          const int32_t *tree_tok, const int32_t *ids, int mode,
                                                          const int32_t *path, const int32_t *acc_len,
                                                          unsigned *status) {
  __shared__ int tok_s[TR_MAX_NODES];
  __shared__ bool writer[TR_MAX_NODES];
  const int b = blockIdx.x, n = threadIdx.x;
  if (n < tree.N) {
    tok_s[n] = tree_tok[(long long)b * tree.N + n];
    writer[n] = mode == TR_UPD_ALL;
  }
  __syncthreads();
  if (mode == TR_UPD_ACCEPTED && n == 0) {
    const int W = tree.D + 1;
    const int a = acc_len[b];
    for (int i = 0; i <= a && i < W; ++i) {
      const int m = path[(long long)b * W + i];
      if (m >= 0 && m < tree.N) writer[m] = true;
    }
  }
  __syncthreads();
  block_update<T>(M + (long long)b * V * K, V, K, tree, tok_s, writer, ids + (long long)b * tree.N * K, status);
}

__global__ void __launch_bounds__(kThreads) commit_kernel(const uint4 *Kt, const uint4 *Vt, uint4 *Kc, uint4 *Vc,
                                                          int32_t *L, int cap, int N, int Hkv, int d16,
                                                          int heads_per_cta, int D, const int32_t *path,
                                                          const int32_t *acc_len, unsigned *counters,
                                                          unsigned *status) {
  __shared__ int path_s[TR_MAX_NODES];
  __shared__ int last;
  const int b = blockIdx.x, part = blockIdx.y, G = gridDim.y;
  __shared__ int bad_path;
  const int acc = acc_len[b];
  const int Lb = L[b];
  if (threadIdx.x == 0) bad_path = 0;
  __syncthreads();
  if (threadIdx.x <= D) {
    const int node = path[(long long)b * (D + 1) + threadIdx.x];
    path_s[threadIdx.x] = node;
    if ((int)threadIdx.x <= acc && (node < 0 || node >= N)) bad_path = 1;
  }
  __syncthreads();
  const bool bad_len = Lb < 0 || Lb > cap || acc < 0 || acc > D || bad_path;
  const bool full = !bad_len && Lb + acc + 1 > cap;
  if (!bad_len && !full) {
    const int h_lo = part * heads_per_cta, h_hi = min(Hkv, h_lo + heads_per_cta);
    if (h_lo < h_hi) block_commit(Kt, Vt, Kc, Vc, N, Hkv, cap, d16, b, Lb, acc, path_s, h_lo, h_hi);
  }
  // the last CTA of sequence b to finish advances L[b]
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) {
    unsigned prev = G > 1 ? atomicAdd(&counters[b], 1u) : 0u;
    last = prev == (unsigned)(G - 1);
  }
  __syncthreads();
  if (last && threadIdx.x == 0) {
    if (bad_len) tr_flag(status, TR_DEV_BAD_LENGTH);
    else if (full) tr_flag(status, TR_DEV_CACHE_FULL);
    else L[b] = Lb + acc + 1;
    if (G > 1) counters[b] = 0u;
  }
}

// The fused end of a step for sequence b.  CTA 0 of the sequence evaluates
// the acceptance, updates M and retrieves the next tree at once: a small
// shared-memory table maps every token written this step to its last writer
// (BFS order), which both resolves duplicate writes and lets the retrieval
// take a rewritten row from the new top-K rows it already holds, so it never
// waits for its own global writes.  CTAs 1..G copy the accepted K/V rows
// (each evaluates the cheap acceptance itself from tree_tok); the last of them
// to finish advances L (CTA 0 does when there is no KV cache).
//
// tree_tok is both this step's tree (read by every CTA of the sequence) and
// the next step's tree (the output), so it is overwritten only once every CTA
// of the sequence has read it: each commit CTA counts itself in `loaded[b]`
// after loading, and CTA 0 counts itself after leaving the next tree in
// `stash[b]`.  Whoever arrives last writes tree_tok (CTA 0 straight from
// shared memory, a commit CTA by copying the stash) and resets the counter.
// No CTA waits for another, so any grid size and any scheduling order works.
struct FinishArgs {
  void *M;
  long long V;
  int K;
  const int32_t *ids;
  int32_t *tree_tok;
  int32_t *acc_len, *path, *committed, *root, *L;
  const uint4 *Kt, *Vt;
  uint4 *Kc, *Vc;
  int cap, Hkv, d16, heads_per_cta;
  int mode;
  unsigned *counters;  // [B] commit CTAs finished (the last advances L)
  unsigned *loaded;    // [B] CTAs that have read this step's tree_tok
  int32_t *stash;      // [B, N] the next tree, when a commit CTA arrives last
  unsigned *status;
};

constexpr int kHash = 2 * TR_MAX_NODES;  // open addressing, load factor <= 1/2

__device__ __forceinline__ int hash_slot(int t) { return (int)(((unsigned)t * 2654435761u) >> 24) & (kHash - 1); }

struct WriterTable {
  int key[kHash];   // token, -1 when empty
  int node[kHash];  // last writing node (largest BFS index) of that token
  __device__ __forceinline__ void insert(int t, int n) {
    for (int h = hash_slot(t);; h = (h + 1) & (kHash - 1)) {
      const int prev = atomicCAS(&key[h], -1, t);
      if (prev == -1 || prev == t) {
        atomicMax(&node[h], n);
        return;
      }
    }
  }
  __device__ __forceinline__ int find(int t) const {
    for (int h = hash_slot(t);; h = (h + 1) & (kHash - 1)) {
      const int k = key[h];
      if (k == t) return node[h];
      if (k == -1) return -1;
    }
  }
};

template <typename T>
__global__ void __launch_bounds__(kThreads) finish_kernel(FinishArgs a, const __grid_constant__ TreeDev tree) {
  __shared__ AcceptSmem s;
  __shared__ WriterTable wt;
  __shared__ int32_t ids_s[TR_MAX_NODES * TR_MAX_K];
  __shared__ int next_tok[TR_MAX_NODES];
  const int b = blockIdx.x, part = blockIdx.y, G = gridDim.y - 1;  // G commit CTAs
  const int N = tree.N, K = a.K, n = threadIdx.x;
  const int32_t *ids_b = a.ids + (long long)b * N * K;
  if (part == 0) {
    for (int h = n; h < kHash; h += blockDim.x) {
      wt.key[h] = -1;
      wt.node[h] = -1;
    }
  }
  load_tree_state(tree, a.tree_tok + (long long)b * N, ids_b, K, s, part == 0 ? ids_s : nullptr);
  if (part > 0) {
    // this CTA has read tree_tok; the last of the sequence's CTAs writes the next tree
    if (n == 0) {
      __threadfence();
      s.last = atomicAdd(&a.loaded[b], 1u) == (unsigned)G;
    }
    __syncthreads();
    if (s.last) {
      __threadfence();
      if (n < N) a.tree_tok[(long long)b * N + n] = __ldcg(a.stash + (long long)b * N + n);
      if (n == 0) a.loaded[b] = 0u;
    }
  }
  block_accept(tree, s);
  const int acc = s.acc_len;
  if (part == 0) {
    write_accept_outputs(tree, s, b, a.acc_len, a.path, a.committed, nullptr);
    T *Mb = (T *)a.M + (long long)b * a.V * K;
    // writers: every node, or the accepted path (all top-K rows are in ids_s)
    bool w = false;
    int t = 0;
    if (n < N) {
      w = a.mode == TR_UPD_ALL || ((tree.anc[s.best][n >> 6] >> (n & 63)) & 1ull);
      t = s.tok[n];
      if (w && (t < 0 || (long long)t >= a.V)) {
        tr_flag(a.status, TR_DEV_BAD_TOKEN);
        w = false;
      }
      if (w) wt.insert(t, n);
    }
    __syncthreads();
    // last writer in BFS order stores its row
    if (w && wt.find(t) == n) {
      T *row = Mb + (long long)t * K;
      for (int k = 0; k < K; ++k) row[k] = (T)ids_s[n * K + k];
    }
    // the next tree from the updated matrix: rows written this step come from ids_s
    if (n < 32) {
      const int lane = n;
      if (lane == 0) {
        int root = s.bonus;
        if (root < 0 || (long long)root >= a.V) {
          tr_flag(a.status, TR_DEV_BAD_TOKEN);
          root = 0;
        }
        next_tok[0] = root;
      }
      __syncwarp();
      for (int l = 1; l <= tree.D; ++l) {
        const int lo = tree.level_off[l], hi = tree.level_off[l + 1];
        for (int m = lo + lane; m < hi; m += 32) {
          const int tp = next_tok[tree.parent[m]], r = tree.rank[m];
          const int wr = wt.find(tp);
          long long v = wr >= 0 ? (long long)ids_s[wr * K + r] : (long long)Mb[(long long)tp * K + r];
          if (v < 0 || v >= a.V) {
            tr_flag(a.status, TR_DEV_BAD_TOKEN);
            v = 0;
          }
          next_tok[m] = (int)v;
        }
        __syncwarp();
      }
      // publish the next tree once every commit CTA has read this step's
      bool direct = G == 0;
      if (!direct) {
        unsigned seen = 0;
        if (lane == 0) seen = ld_acquire_u32(&a.loaded[b]);
        seen = __shfl_sync(0xffffffffu, seen, 0);
        if (seen == (unsigned)G) {
          direct = true;  // all of them already have: no arrival is left to come
        } else {
          int32_t *st = a.stash + (long long)b * N;
          for (int m = lane; m < N; m += 32) st[m] = next_tok[m];
          __threadfence();
          __syncwarp();
          unsigned prev = 0;
          if (lane == 0) prev = atomicAdd(&a.loaded[b], 1u);
          prev = __shfl_sync(0xffffffffu, prev, 0);
          direct = prev == (unsigned)G;  // the others arrived meanwhile
        }
        if (direct && lane == 0) a.loaded[b] = 0u;
      }
      if (direct) {
        int32_t *out = a.tree_tok + (long long)b * N;
        for (int m = lane; m < N; m += 32) out[m] = next_tok[m];
      }
      if (lane == 0) {
        a.root[b] = s.bonus;
        if (G == 0) {
          const int Lb = a.L[b];
          if (Lb < 0 || Lb > a.cap) tr_flag(a.status, TR_DEV_BAD_LENGTH);
          else if (a.Kc && Lb + acc + 1 > a.cap) tr_flag(a.status, TR_DEV_CACHE_FULL);
          else a.L[b] = Lb + acc + 1;
        }
      }
    }
    return;
  }
  // ---- KV commit of heads [h_lo, h_hi)
  if (threadIdx.x == 0) s.L = a.L[b];
  __syncthreads();
  const int Lb = s.L;
  const bool bad_len = Lb < 0 || Lb > a.cap;
  const bool full = !bad_len && Lb + acc + 1 > a.cap;
  if (!bad_len && !full) {
    const int h_lo = (part - 1) * a.heads_per_cta, h_hi = min(a.Hkv, h_lo + a.heads_per_cta);
    if (h_lo < h_hi) block_commit(a.Kt, a.Vt, a.Kc, a.Vc, N, a.Hkv, a.cap, a.d16, b, Lb, acc, s.path, h_lo, h_hi);
  }
  // the last commit CTA of the sequence advances L (every one has read it by then)
  __syncthreads();
  if (threadIdx.x == 0) {
    const unsigned prev = G > 1 ? atomicAdd(&a.counters[b], 1u) : 0u;
    if (prev == (unsigned)(G - 1)) {
      if (bad_len) tr_flag(a.status, TR_DEV_BAD_LENGTH);
      else if (full) tr_flag(a.status, TR_DEV_CACHE_FULL);
      else a.L[b] = Lb + acc + 1;
      if (G > 1) a.counters[b] = 0u;
    }
  }
}

int commit_heads_per_cta(int Hkv) {
  // about 8 CTAs per sequence share the copy
  return Hkv <= 8 ? 1 : (Hkv + 7) / 8;
}

}  // namespace

// ---------------------------------------------------------------------------
// ABI
// ---------------------------------------------------------------------------

extern "C" int tr_retrieve(const void *M, tr_itype mtype, int B, int64_t V, int K, const struct tr_tree *tree,
                           const int32_t *root, int32_t *tree_tok, tr_stream_t stream) {
  if (!M || !tree || !root || !tree_tok || B < 1 || V < 1 || K != tree->dev.K) return TR_E_INVAL;
  if (mtype != TR_I32 && mtype != TR_I64) return TR_E_INVAL;
  int rc = tr_check_device();
  if (rc != TR_OK) return rc;
  cudaStream_t s = (cudaStream_t)stream;
  if (mtype == TR_I64)
    retrieve_kernel<long long><<<B, 32, 0, s>>>((const long long *)M, V, K, tree->dev, root, tree_tok, tr_status_dev());
  else
    retrieve_kernel<int32_t><<<B, 32, 0, s>>>((const int32_t *)M, V, K, tree->dev, root, tree_tok, tr_status_dev());
  TR_LAUNCH_CHECK();
  return TR_OK;
}

extern "C" int tr_accept(const struct tr_tree *tree, int B, const int32_t *tree_tok, const int32_t *ids, int K,
                         int32_t *acc_len, int32_t *path, int32_t *committed, int32_t *bonus, tr_stream_t stream) {
  if (!tree || !tree_tok || !ids || B < 1 || K < 1 || K > TR_MAX_K) return TR_E_INVAL;
  int rc = tr_check_device();
  if (rc != TR_OK) return rc;
  accept_kernel<<<B, kThreads, 0, (cudaStream_t)stream>>>(tree->dev, tree_tok, ids, K, acc_len, path, committed, bonus);
  TR_LAUNCH_CHECK();
  return TR_OK;
}

extern "C" int tr_update(void *M, tr_itype mtype, int B, int64_t V, int K, const struct tr_tree *tree,
                         const int32_t *tree_tok, const int32_t *ids, tr_upd_mode mode, const int32_t *path,
                         const int32_t *acc_len, tr_stream_t stream) {
  if (!M || !tree || !tree_tok || !ids || B < 1 || V < 1 || K < 1 || K > TR_MAX_K) return TR_E_INVAL;
  if (mtype != TR_I32 && mtype != TR_I64) return TR_E_INVAL;
  if (mode != TR_UPD_ALL && mode != TR_UPD_ACCEPTED) return TR_E_INVAL;
  if (mode == TR_UPD_ACCEPTED && (!path || !acc_len)) return TR_E_INVAL;
  int rc = tr_check_device();
  if (rc != TR_OK) return rc;
  cudaStream_t s = (cudaStream_t)stream;
  if (mtype == TR_I64)
    update_kernel<long long><<<B, kThreads, 0, s>>>((long long *)M, V, K, tree->dev, tree_tok, ids, mode, path,
                                                    acc_len, tr_status_dev());
  else
    update_kernel<int32_t><<<B, kThreads, 0, s>>>((int32_t *)M, V, K, tree->dev, tree_tok, ids, mode, path, acc_len,
                                                   tr_status_dev());
  TR_LAUNCH_CHECK();
  return TR_OK;
}

extern "C" size_t tr_kv_commit_workspace_bytes(int B) { return B > 0 ? tr_align_up((size_t)B * 4, 256) : 0; }

extern "C" int tr_kv_commit(const void *Kt, const void *Vt, void *Kc, void *Vc, int32_t *L, int cap, int B, int Hkv,
                            int d, const struct tr_tree *tree, const int32_t *path, const int32_t *acc_len, void *ws,
                            size_t ws_bytes, tr_stream_t stream) {
  if (!Kt || !Vt || !Kc || !Vc || !L || !tree || !path || !acc_len || B < 1 || Hkv < 1 || cap < 1) return TR_E_INVAL;
  if (d < 8 || d % 8) return TR_E_INVAL;
  if (((uintptr_t)Kt | (uintptr_t)Vt | (uintptr_t)Kc | (uintptr_t)Vc) & 15) return TR_E_INVAL;
  const int hpc = commit_heads_per_cta(Hkv);
  const int G = (Hkv + hpc - 1) / hpc;
  if (G > 1 && (!ws || ws_bytes < tr_kv_commit_workspace_bytes(B))) return TR_E_INVAL;
  int rc = tr_check_device();
  if (rc != TR_OK) return rc;
  commit_kernel<<<dim3(B, G), kThreads, 0, (cudaStream_t)stream>>>(
      (const uint4 *)Kt, (const uint4 *)Vt, (uint4 *)Kc, (uint4 *)Vc, L, cap, tree->dev.N, Hkv, d / 8, hpc,
      tree->dev.D, path, acc_len, (unsigned *)ws, tr_status_dev());
  TR_LAUNCH_CHECK();
  return TR_OK;
}

// workspace of tr_step: [top-K workspace | commit counters [B] | tree-read
// counters [B] | next-tree stash [B, N]], each part 256-byte aligned
static size_t step_topk_ws(const tr_step_args *a) {
  const int64_t rows = (int64_t)a->B * a->tree->dev.N;
  if (a->logits) return tr_align_up(tr_topk_workspace_bytes(rows, a->V, a->K), 256);
  return tr_align_up(tr_lmhead_topk_workspace_bytes(rows, a->D, a->V, a->K), 256);
}

static size_t step_counters_bytes(int B) { return tr_align_up((size_t)B * 4, 256); }

extern "C" size_t tr_step_workspace_bytes(const tr_step_args *a) {
  if (!a || !a->tree || a->B < 1) return 0;
  return step_topk_ws(a) + 2 * step_counters_bytes(a->B) +
         tr_align_up((size_t)a->B * a->tree->dev.N * 4, 256);
}

extern "C" int tr_step(const tr_step_args *a, tr_stream_t stream) {
  if (!a || !a->tree || !a->M || !a->tree_tok || !a->ids || !a->root || !a->L) return TR_E_INVAL;
  if (a->B < 1 || a->V < 1 || a->K != a->tree->dev.K) return TR_E_INVAL;
  if (a->mtype != TR_I32 && a->mtype != TR_I64) return TR_E_INVAL;
  if (a->mode != TR_UPD_ALL && a->mode != TR_UPD_ACCEPTED) return TR_E_INVAL;
  if (!a->logits && (!a->H || !a->Wt)) return TR_E_INVAL;
  const bool commit = a->Kt != nullptr;
  if (commit) {
    if (!a->Vt || !a->Kc || !a->Vc || a->Hkv < 1 || a->cap < 1 || a->d < 8 || a->d % 8) return TR_E_INVAL;
    if (((uintptr_t)a->Kt | (uintptr_t)a->Vt | (uintptr_t)a->Kc | (uintptr_t)a->Vc) & 15) return TR_E_INVAL;
  }
  if (!a->ws || a->ws_bytes < tr_step_workspace_bytes(a)) return TR_E_INVAL;
  int rc = tr_check_device();
  if (rc != TR_OK) return rc;
  cudaStream_t s = (cudaStream_t)stream;
  const TreeDev &tree = a->tree->dev;
  const int64_t rows = (int64_t)a->B * tree.N;
  const size_t tk_ws = step_topk_ws(a);
  if (a->logits)
    rc = tr_topk(a->logits, a->ltype, rows, a->V, a->ld, a->K, a->ids, a->vals, a->ws, tk_ws, stream);
  else
    rc = tr_lmhead_topk(a->H, a->Wt, rows, a->D, a->V, a->K, a->ids, a->vals, a->ws, tk_ws, stream);
  if (rc != TR_OK) return rc;
  FinishArgs f;
  f.M = a->M;
  f.V = a->V;
  f.K = a->K;
  f.ids = a->ids;
  f.tree_tok = a->tree_tok;
  f.acc_len = a->acc_len;
  f.path = a->path;
  f.committed = a->committed;
  f.root = a->root;
  f.L = a->L;
  f.Kt = (const uint4 *)a->Kt;
  f.Vt = (const uint4 *)a->Vt;
  f.Kc = commit ? (uint4 *)a->Kc : nullptr;
  f.Vc = (uint4 *)a->Vc;
  f.cap = commit ? a->cap : INT32_MAX;
  f.Hkv = commit ? a->Hkv : 0;
  f.d16 = commit ? a->d / 8 : 0;
  f.heads_per_cta = commit ? commit_heads_per_cta(a->Hkv) : 1;
  f.mode = a->mode;
  f.counters = (unsigned *)((char *)a->ws + tk_ws);
  f.loaded = (unsigned *)((char *)a->ws + tk_ws + step_counters_bytes(a->B));
  f.stash = (int32_t *)((char *)a->ws + tk_ws + 2 * step_counters_bytes(a->B));
  f.status = tr_status_dev();
  const int G = commit ? (a->Hkv + f.heads_per_cta - 1) / f.heads_per_cta : 0;  // commit CTAs per sequence
  if (a->mtype == TR_I64)
    finish_kernel<long long><<<dim3(a->B, 1 + G), kThreads, 0, s>>>(f, tree);
  else
    finish_kernel<int32_t><<<dim3(a->B, 1 + G), kThreads, 0, s>>>(f, tree);
  TR_LAUNCH_CHECK();
  return TR_OK;
}
