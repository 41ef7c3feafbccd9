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
  float cw[TR_MAX_NODES];  // sampling: node n's weight 2^((x - max) c) in its parent's row
  float cz[TR_MAX_NODES];  // sampling: node n's normaliser Z (the same units)
  float cu[TR_MAX_NODES];  // sampling: the uniform of node n's test, U[parent n, rank n]
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
// acceptance under sampling
// ---------------------------------------------------------------------------

// Logits of one row, fp32 or bf16 (widened exactly).
template <typename LT>
struct Logit;
template <>
struct Logit<float> {
  static constexpr int kVec = 4;
  __device__ __forceinline__ static float at(const float *p) { return __ldg(p); }
  __device__ __forceinline__ static void vec(const float *p, float (&e)[4]) {
    const float4 q = __ldg(reinterpret_cast<const float4 *>(p));
    e[0] = q.x;
    e[1] = q.y;
    e[2] = q.z;
    e[3] = q.w;
  }
};
template <>
struct Logit<__nv_bfloat16> {
  static constexpr int kVec = 8;
  __device__ __forceinline__ static float at(const __nv_bfloat16 *p) {
    return __uint_as_float((uint32_t)__ldg(reinterpret_cast<const unsigned short *>(p)) << 16);
  }
  __device__ __forceinline__ static void vec(const __nv_bfloat16 *p, float (&e)[8]) {
    const uint4 q = __ldg(reinterpret_cast<const uint4 *>(p));
    const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      e[2 * i] = __uint_as_float(w[i] << 16);
      e[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
  }
};

__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

struct SampleArgs {
  const void *logits;  // [B*N, ld] of the logit type
  long long ld;
  const float2 *stats; // [B*N] (row maximum, sum of 2^((x - max) c))
  const float2 *sstats;// [B*N, nsteps] (step maximum, sum of 2^((x - step max) c)) per 8 KB step of a row
  int nsteps;          // steps per row
  const float *U;      // [B, N, K1] uniforms in [0, 1)
  int K1;              // K + 1
  float c;             // log2(e) / temperature
};

// Speculative-decoding lesson, the acceptance rule, applied to Token
// Recycling's deterministic children in rank order (q one-hot on the child's
// token): child x of the current node is accepted when U < r(x), r being the
// node's distribution with the already rejected siblings' tokens removed and
// renormalised; the walk continues from an accepted child and stops at a node
// whose children are all rejected.  In units of the row maximum, r(x) is
// w(x) / (Z - sum of the rejected distinct tokens' w).  Every CTA of the
// sequence computes the same walk (thread 0; the weights come in one parallel
// gather).  Sets s.best, s.acc_len and s.path.
template <typename LT>
__device__ void block_accept_sampled(const TreeDev &tree, AcceptSmem &s, const SampleArgs &sa, int b, long long V,
                                     unsigned *status) {
  const int n = threadIdx.x, N = tree.N;
  if (n < N) {
    const long long rown = (long long)b * N + n;
    s.cz[n] = sa.stats[rown].y;
    if (n > 0) {
      const long long rowp = (long long)b * N + tree.parent[n];
      s.cu[n] = __ldg(sa.U + rowp * sa.K1 + tree.rank[n]);
      const int x = s.tok[n];
      float w = 0.f;
      if (x >= 0 && (long long)x < V) {
        const float l = Logit<LT>::at((const LT *)sa.logits + rowp * sa.ld + x);
        w = ex2_approx(fmaf(l, sa.c, -sa.stats[rowp].x * sa.c));
      } else {
        tr_flag(status, TR_DEV_BAD_TOKEN);
      }
      s.cw[n] = w;
    }
  }
  __syncthreads();
  if (n == 0) {
    int cur = 0;
    while (true) {
      const int f = tree.child_first[cur], cnt = tree.child_count[cur];
      float rem = s.cz[cur];
      int next = -1;
      for (int i = 0; i < cnt; ++i) {
        const int ch = f + i, x = s.tok[ch];
        bool dup = false;  // an earlier (rejected) sibling holds the same token: r(x) is 0 now
        for (int j = 0; j < i; ++j) dup |= s.tok[f + j] == x;
        const float w = s.cw[ch];
        const float r = dup ? 0.f : w / fmaxf(rem, w);
        if (s.cu[ch] < r) {
          next = ch;
          break;
        }
        if (!dup) rem -= w;
      }
      if (next < 0) break;
      cur = next;
    }
    s.best = cur;
    s.acc_len = tree.depth[cur];
  }
  __syncthreads();
  if (n < N && ((tree.anc[s.best][n >> 6] >> (n & 63)) & 1ull)) s.path[tree.depth[n]] = n;
  __syncthreads();
}

// The draw at the final node n*: the smallest token y with
// r(0) + ... + r(y) > U[n*, K], r being n*'s distribution without its
// (rejected) children's tokens.  The top-K pass left a (maximum, sum) pair for
// every 8 KB step of the row, so warp 0 scans those step sums (less the
// rejected children's weights) in fp64 to find the step where the running sum
// crosses U times the total; the block then loads that one step, coalesced,
// each thread sums its slice of it, a block scan finds the slice, and its
// thread walks the slice.  Returns y on every thread.
template <typename LT>
__device__ int block_draw_residual(const TreeDev &tree, AcceptSmem &s, const SampleArgs &sa, int b, long long V) {
  constexpr int E = 8192 / (int)sizeof(LT);  // elements per step
  constexpr int PER = E / kThreads;          // elements per thread of one step
  constexpr int VW = Logit<LT>::kVec;
  static_assert(PER % VW == 0, "whole vectors per thread");
  __shared__ float rej_w[TR_MAX_K];   // weight of each rejected child's token (0 for a repeated token)
  __shared__ int step_hit;            // the step the target falls in
  __shared__ double step_base, target_s;
  __shared__ float wpart[kThreads / 32];
  __shared__ int winner, last_pos;
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5, N = tree.N;
  const int nstar = s.best;
  const long long row = (long long)b * N + nstar;
  const LT *x = (const LT *)sa.logits + row * sa.ld;
  const float M = sa.stats[row].x, mc = M * sa.c;
  const int f = tree.child_first[nstar], cnt = tree.child_count[nstar];
  if (t < cnt) {
    const int xr = s.tok[f + t];
    bool dup = xr < 0 || (long long)xr >= V;
    for (int j = 0; j < t; ++j) dup |= s.tok[f + j] == xr;
    rej_w[t] = dup ? 0.f : ex2_approx(fmaf(Logit<LT>::at(x + xr), sa.c, -mc));
  }
  if (t == 0) {
    winner = -1;
    last_pos = -1;
  }
  __syncthreads();
  if (warp == 0) {
    // the steps' weights in units of the row maximum, rejected tokens removed
    const float2 *ss = sa.sstats + row * sa.nsteps;
    auto step_w = [&](int st) -> double {
      if (st >= sa.nsteps) return 0.0;
      const float2 p = ss[st];
      double w = p.y == 0.f ? 0.0 : (double)p.y * (double)ex2_approx((p.x - M) * sa.c);
      for (int i = 0; i < cnt; ++i)
        if (s.tok[f + i] / E == st) w -= (double)rej_w[i];
      return w > 0.0 ? w : 0.0;
    };
    double total = 0.0;
    for (int g = 0; g < sa.nsteps; g += 32) {
      double w = step_w(g + lane);
#pragma unroll
      for (int off = 16; off; off >>= 1) w += __shfl_xor_sync(0xffffffffu, w, off);
      total += w;
    }
    const double target = (double)__ldg(sa.U + row * sa.K1 + (sa.K1 - 1)) * total;
    double base = 0.0;
    int hit = -1, last = -1;
    for (int g = 0; g < sa.nsteps && hit < 0; g += 32) {
      const double w = step_w(g + lane);
      double incl = w;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const double o = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += o;
      }
      const unsigned cross = __ballot_sync(0xffffffffu, w > 0.0 && base + incl > target);
      const unsigned pos = __ballot_sync(0xffffffffu, w > 0.0);
      if (pos) last = g + 31 - __clz(pos);
      if (cross) {
        const int l = __ffs(cross) - 1;
        hit = g + l;
        base += __shfl_sync(0xffffffffu, incl - w, l);
      } else {
        base += __shfl_sync(0xffffffffu, incl, 31);
      }
    }
    if (lane == 0) {
      if (hit < 0) {  // rounding left the total at or below the target: the last token with weight
        hit = last;
        base = -INFINITY;  // no slice claims the target, so the last slice with weight walks
      }
      step_hit = hit;
      step_base = base;
      target_s = target;
    }
  }
  __syncthreads();
  const int hit = step_hit;
  if (hit < 0) {  // no weight left at all (the children held it all)
    if (t == 0) s.bonus = s.top1[nstar];
    __syncthreads();
    return s.bonus;
  }
  // the step's elements, PER consecutive ones per thread
  const long long e0 = (long long)hit * E + (long long)t * PER;
  float w[PER];
#pragma unroll
  for (int v = 0; v < PER; v += VW) {
    float e[VW];
    if (e0 + v + VW <= V) {
      Logit<LT>::vec(x + e0 + v, e);
    } else {
#pragma unroll
      for (int q = 0; q < VW; ++q) e[q] = e0 + v + q < V ? Logit<LT>::at(x + e0 + v + q) : -INFINITY;
    }
#pragma unroll
    for (int q = 0; q < VW; ++q) w[v + q] = ex2_approx(fmaf(e[q], sa.c, -mc));
  }
  for (int i = 0; i < cnt; ++i) {  // rejected children's tokens carry no weight
    const long long o = (long long)s.tok[f + i] - e0;
    if (o >= 0 && o < PER)
#pragma unroll
      for (int q = 0; q < PER; ++q)
        if (q == o) w[q] = 0.f;
  }
  float z = 0.f;
#pragma unroll
  for (int q = 0; q < PER; ++q) z += w[q];
  // block scan of the slices' sums: incl of thread t is bitwise the excl of t + 1
  float incl = z;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const float o = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += o;
  }
  const float excl_w = __shfl_up_sync(0xffffffffu, incl, 1);
  if (lane == 31) wpart[warp] = incl;
  __syncthreads();
  if (t == 0) {
    float acc = 0.f;
    for (int k = 0; k < kThreads / 32; ++k) {
      const float tw = wpart[k];
      wpart[k] = acc;
      acc += tw;
    }
  }
  __syncthreads();
  const float woff = wpart[warp];
  incl += woff;
  const float excl = lane == 0 ? woff : excl_w + woff;
  const float rel = (float)(target_s - step_base);  // the target inside the step
  if (z > 0.f && excl <= rel && rel < incl) winner = t;
  if (z > 0.f) atomicMax(&last_pos, t);
  __syncthreads();
  const int wt = winner >= 0 ? winner : last_pos;
  if (t == wt) {
    float acc = excl;
    int y = -1, lastp = -1;
#pragma unroll
    for (int q = 0; q < PER; ++q) {
      if (w[q] > 0.f) lastp = q;
      acc += w[q];
      if (y < 0 && w[q] > 0.f && acc > rel) y = q;
    }
    s.bonus = (int)(e0 + (y >= 0 ? y : lastp));
  }
  __syncthreads();
  return s.bonus;
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

template <typename LT>
__global__ void __launch_bounds__(kThreads) accept_sampled_kernel(const __grid_constant__ TreeDev tree,
                                                                  const int32_t *tree_tok, const int32_t *ids, int K,
                                                                  long long V, SampleArgs sa, int32_t *acc_len,
                                                                  int32_t *path, int32_t *committed, int32_t *bonus,
                                                                  unsigned *status) {
  __shared__ AcceptSmem s;
  const int b = blockIdx.x;
  load_tree_state(tree, tree_tok + (long long)b * tree.N, ids + (long long)b * tree.N * K, K, s);
  block_accept_sampled<LT>(tree, s, sa, b, V, status);
  block_draw_residual<LT>(tree, s, sa, b, V);
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
  SampleArgs sa;       // acceptance under sampling (SAMPLE kernels only)
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

// SAMPLE: the acceptance samples at a temperature (block_accept_sampled and,
// in CTA 0, block_draw_residual for the committed token after the path); LT
// is then the logits' element type.  The matrix update, the KV commit and the
// next retrieval are the same either way.
template <typename T, typename LT, bool SAMPLE>
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
  if (SAMPLE)
    block_accept_sampled<LT>(tree, s, a.sa, b, a.V, a.status);
  else
    block_accept(tree, s);
  const int acc = s.acc_len;
  if (part == 0) {
    if (SAMPLE) block_draw_residual<LT>(tree, s, a.sa, b, a.V);
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

static size_t step_stash_bytes(const tr_step_args *a) { return tr_align_up((size_t)a->B * a->tree->dev.N * 4, 256); }

static size_t step_stats_bytes(const tr_step_args *a) { return tr_align_up((size_t)a->B * a->tree->dev.N * 8, 256); }

// per 8 KB step of every row (fp32 rows have the most steps)
static size_t step_sstats_bytes(const tr_step_args *a) {
  return tr_align_up((size_t)a->B * a->tree->dev.N * tr_softmax_steps(a->V, TR_F32) * 8, 256);
}

extern "C" size_t tr_step_workspace_bytes(const tr_step_args *a) {
  if (!a || !a->tree || a->B < 1) return 0;
  // + the rows' and their steps' softmax statistics of tr_step_sampled
  return step_topk_ws(a) + 2 * step_counters_bytes(a->B) + step_stash_bytes(a) + step_stats_bytes(a) +
         step_sstats_bytes(a);
}

template <typename T>
static void launch_finish(const FinishArgs &f, const TreeDev &tree, dim3 grid, cudaStream_t s, bool sample,
                          tr_ftype ltype) {
  if (!sample)
    finish_kernel<T, float, false><<<grid, kThreads, 0, s>>>(f, tree);
  else if (ltype == TR_F32)
    finish_kernel<T, float, true><<<grid, kThreads, 0, s>>>(f, tree);
  else
    finish_kernel<T, __nv_bfloat16, true><<<grid, kThreads, 0, s>>>(f, tree);
}

static int step_impl(const tr_step_args *a, float temperature, const float *U, tr_stream_t stream);

extern "C" int tr_step(const tr_step_args *a, tr_stream_t stream) { return step_impl(a, 0.f, nullptr, stream); }

extern "C" int tr_step_sampled(const tr_step_args *a, float temperature, const float *U, tr_stream_t stream) {
  if (!U || !(temperature > 0.f) || !(temperature < INFINITY)) return TR_E_INVAL;
  if (a && !a->logits) return TR_E_UNSUPPORTED;  // the draw reads the logits: not with the fused LM head
  return step_impl(a, temperature, U, stream);
}

static int step_impl(const tr_step_args *a, float temperature, const float *U, tr_stream_t stream) {
  const bool sample = U != nullptr;
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
  const size_t cnt_bytes = step_counters_bytes(a->B);
  float2 *stats = (float2 *)((char *)a->ws + tk_ws + 2 * cnt_bytes + step_stash_bytes(a));
  float2 *sstats = (float2 *)((char *)stats + step_stats_bytes(a));
  if (sample)
    rc = tr_topk_softmax(a->logits, a->ltype, rows, a->V, a->ld, a->K, temperature, a->ids, a->vals, (float *)stats,
                         (float *)sstats, a->ws, tk_ws, stream);
  else if (a->logits)
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
  f.loaded = (unsigned *)((char *)a->ws + tk_ws + cnt_bytes);
  f.stash = (int32_t *)((char *)a->ws + tk_ws + 2 * cnt_bytes);
  f.status = tr_status_dev();
  f.sa.logits = a->logits;
  f.sa.ld = a->ld;
  f.sa.stats = stats;
  f.sa.sstats = sstats;
  f.sa.nsteps = tr_softmax_steps(a->V, a->ltype);
  f.sa.U = U;
  f.sa.K1 = a->K + 1;
  f.sa.c = sample ? 1.4426950408889634f / temperature : 0.f;
  const int G = commit ? (a->Hkv + f.heads_per_cta - 1) / f.heads_per_cta : 0;  // commit CTAs per sequence
  const dim3 grid(a->B, 1 + G);
  if (a->mtype == TR_I64)
    launch_finish<long long>(f, tree, grid, s, sample, a->ltype);
  else
    launch_finish<int32_t>(f, tree, grid, s, sample, a->ltype);
  TR_LAUNCH_CHECK();
  return TR_OK;
}

extern "C" int tr_accept_sampled(const struct tr_tree *tree, int B, const int32_t *tree_tok, const int32_t *ids,
                                 int K, const void *logits, tr_ftype ltype, int64_t V, int64_t ld, const float *stats,
                                 const float *step_stats, float temperature, const float *U, int32_t *acc_len,
                                 int32_t *path, int32_t *committed, int32_t *bonus, tr_stream_t stream) {
  if (!tree || !tree_tok || !ids || !logits || !stats || !step_stats || !U || B < 1 || K < 1 || K > TR_MAX_K)
    return TR_E_INVAL;
  if (K != tree->dev.K || V < 1 || ld < V || (ltype != TR_F32 && ltype != TR_BF16)) return TR_E_INVAL;
  if (!(temperature > 0.f) || !(temperature < INFINITY)) return TR_E_INVAL;
  if (V > INT32_MAX) return TR_E_UNSUPPORTED;
  const size_t esz = ltype == TR_F32 ? 4 : 2;
  if ((uintptr_t)logits % 16 || (ld * (int64_t)esz) % 16) return TR_E_UNSUPPORTED;
  int rc = tr_check_device();
  if (rc != TR_OK) return rc;
  SampleArgs sa;
  sa.logits = logits;
  sa.ld = ld;
  sa.stats = (const float2 *)stats;
  sa.sstats = (const float2 *)step_stats;
  sa.nsteps = tr_softmax_steps(V, ltype);
  sa.U = U;
  sa.K1 = K + 1;
  sa.c = 1.4426950408889634f / temperature;
  cudaStream_t s = (cudaStream_t)stream;
  if (ltype == TR_F32)
    accept_sampled_kernel<float><<<B, kThreads, 0, s>>>(tree->dev, tree_tok, ids, K, V, sa, acc_len, path, committed,
                                                        bonus, tr_status_dev());
  else
    accept_sampled_kernel<__nv_bfloat16><<<B, kThreads, 0, s>>>(tree->dev, tree_tok, ids, K, V, sa, acc_len, path,
                                                                committed, bonus, tr_status_dev());
  TR_LAUNCH_CHECK();
  return TR_OK;
}
