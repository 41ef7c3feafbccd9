/*
 * tr.h -- C ABI of libtr, the GB300 (sm_103a) hot path of Token Recycling
 * speculative decoding.
 *
 * Token Recycling ("Turning Trash into Treasure: Accelerating Inference of
 * Large Language Models with Token Recycling", ACL 2025) keeps an adjacency
 * matrix M in V^{|V| x K}: row i holds K candidate successor tokens of token
 * i.  Every decoding step (hyper.ai summary, section "Method"; blog
 * "token-recycling", section 完整工作流程):
 *   1. retrieves a static, unbalanced draft tree rooted at the last committed
 *      token by expanding rows of M level by level       -> tr_retrieve
 *   2. verifies the flattened tree in one forward pass with tree attention
 *      (each node sees the prefix and its own ancestors)  -> tr_verify_attn
 *   3. takes each node's top-K next tokens                -> tr_topk, or
 *      the fused LM head + top-K                          -> tr_lmhead_topk
 *   4. accepts the longest path matching the target's greedy choice, plus
 *      the target's token after it (the bonus)            -> tr_accept
 *   5. overwrites M[token] with the top-K of every verified node
 *      (Chinese summary, section 方法, M[x~_i] = argtopk(p~_{i+1}))
 *                                                          -> tr_update
 * and commits the accepted nodes' K/V to the cache (tr_kv_commit).
 * tr_step fuses 3-5, the commit and the next step's retrieval.
 *
 * Conventions
 *  - Every tensor argument is a caller-owned DEVICE pointer on the current
 *    device, dense row-major with the layout stated at each call.  libtr never
 *    allocates device memory on these calls; scratch comes from the caller's
 *    workspace (see the *_workspace_bytes calls).
 *  - Every call is asynchronous on `stream` (NULL = the legacy default stream),
 *    makes no host synchronisation and can be captured in a CUDA graph.
 *  - Argument errors are found on the host and returned before any launch
 *    (TR_E_INVAL, TR_E_UNSUPPORTED).  A failed launch returns TR_E_CUDA.
 *  - Errors found on the device (a token ID outside [0, V), a full cache, a
 *    wait that ran out) set bits of a per-device status word and the kernel
 *    skips the faulty unit; kernels never trap.  tr_get_status reads and
 *    clears the word.
 *  - No exception crosses the ABI.  Calls keep no hidden state besides the
 *    status word and may run concurrently on different streams as long as
 *    they do not share output buffers or workspace.
 *  - Limits: tree nodes N <= 128, K <= 32, head dim d == 128.
 */
#ifndef TR_H
#define TR_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *tr_stream_t; /* a cudaStream_t */

typedef enum {
  TR_OK = 0,
  TR_E_INVAL = 1,       /* bad argument (null pointer, shape, alignment) */
  TR_E_UNSUPPORTED = 2, /* valid but not supported here (dtype, size, GPU) */
  TR_E_CUDA = 3,        /* a CUDA runtime call or launch failed */
  TR_E_DEVICE = 4,      /* returned by tr_get_status when device bits are set */
  TR_E_TIMEOUT = 5
} tr_status;

/* bits of the device status word */
#define TR_DEV_BAD_TOKEN 0x1u  /* a token ID outside [0, V) was read from M or root */
#define TR_DEV_CACHE_FULL 0x2u /* a KV commit would pass the cache capacity */
#define TR_DEV_BAD_LENGTH 0x4u /* a cache length L[b] outside [0, cap] */
#define TR_DEV_TIMEOUT 0x8u    /* a bounded device wait gave up */

typedef enum { TR_I32 = 0, TR_I64 = 1 } tr_itype;  /* element type of M */
typedef enum { TR_F32 = 0, TR_BF16 = 1 } tr_ftype; /* element type of logits */

/* hyper.ai summary, "Method" (hot start inherits the matrix of earlier
 * inference) and "Experiment" (all-zero and random-vocabulary ablations). */
typedef enum { TR_INIT_ZERO = 0, TR_INIT_RANDOM = 1, TR_INIT_INHERIT = 2 } tr_init_mode;

/* hyper.ai summary, "Experiment": updating from all draft tokens versus from
 * the accepted tokens only. */
typedef enum { TR_UPD_ALL = 0, TR_UPD_ACCEPTED = 1 } tr_upd_mode;

/* ------------------------------------------------------------------------ */
/* Static draft tree                                                         */
/* ------------------------------------------------------------------------ */

/* Opaque, immutable plan of a static draft tree (host memory only).
 *
 * hyper.ai summary, "Method": the tree is static (each node keeps its child
 * count on every step, so it can be preprocessed) and unbalanced (earlier,
 * more probable nodes in a layer get more children).  Blog "token-recycling",
 * 完整工作流程 step 2: child r of a node holding token x is M[x][r].
 *
 * child_counts: host array of n_nodes child counts, one per node in BFS
 *   (level-by-level) order, node 0 being the root.  Each count is in [0, K];
 *   the counts must describe exactly n_nodes nodes.  1 <= n_nodes <= 128.
 * K: number of candidates per matrix row, 1 <= K <= 32.
 * out: receives the plan; free it with tr_tree_destroy.  The plan is copied
 *   into each launch's parameters, so no device memory is involved.
 * Returns TR_E_INVAL for a malformed spec. */
int tr_tree_create(const int32_t *child_counts, int n_nodes, int K, struct tr_tree **out);
int tr_tree_destroy(struct tr_tree *tree);

/* Host copies of the plan (each array n_nodes long; parent[0] = -1); any
 * pointer may be NULL.  Returns the node count in *n_nodes and the depth of
 * the deepest node in *max_depth. */
int tr_tree_info(const struct tr_tree *tree, int *n_nodes, int *max_depth, int32_t *parent,
                 int32_t *rank, int32_t *depth);

/* ------------------------------------------------------------------------ */
/* Matrix initialisation                                                     */
/* ------------------------------------------------------------------------ */

/* Fills B adjacency matrices M [B, V, K] (element type mtype).
 *  TR_INIT_ZERO     every entry 0.
 *  TR_INIT_RANDOM   entry (b, i, j) = output number (b*V + i)*K + j of the
 *                   splitmix64 stream started at `seed`, modulo V.
 *  TR_INIT_INHERIT  every sequence copies src [V, K] (same element type), a
 *                   matrix left by earlier requests (hot start).
 * src is ignored unless mode == TR_INIT_INHERIT. */
int tr_init_matrix(void *M, tr_itype mtype, int B, int64_t V, int K, tr_init_mode mode,
                   const void *src, uint64_t seed, tr_stream_t stream);

/* ------------------------------------------------------------------------ */
/* 1. Draft retrieval                                                        */
/* ------------------------------------------------------------------------ */

/* Blog "token-recycling", 完整工作流程 steps 1-2; hyper.ai summary, "Method"
 * (BFS-like expansion of the fixed tree, root = last token of the context).
 *   M        [B, V, K] mtype, read only (the matrix before this step's update)
 *   root     [B] int32, the root token of each sequence
 *   tree_tok [B, N] int32 output, the tree's tokens in BFS order,
 *            tree_tok[b, 0] = root[b], tree_tok[b, n] = M[b, tok(parent n), rank n].
 * A token outside [0, V) (in root or read from M) sets TR_DEV_BAD_TOKEN and
 * is replaced by 0 so the expansion stays in bounds. */
int tr_retrieve(const void *M, tr_itype mtype, int B, int64_t V, int K, const struct tr_tree *tree,
                const int32_t *root, int32_t *tree_tok, tr_stream_t stream);

/* ------------------------------------------------------------------------ */
/* 2. Tree-attention verification                                            */
/* ------------------------------------------------------------------------ */

/* Blog "token-recycling", 完整工作流程 step 3 (flattened merged sequence; each
 * node sees only its own root-to-node path, siblings are invisible); the
 * speculative-decoding lesson's tree attention (each node attends only to its
 * ancestors).  For node i and query head h, with g = h / (Hq / Hkv):
 *   O[b,i,h] = softmax_j(scale * Q[b,i,h] . key_j) . value_j
 * over the keys  {Kc[b,g,p] : 0 <= p < L[b]}  and  {Kt[b,j,g] : j on the path
 * from the root to i, i included}.
 *   Q      [B, N, Hq, d]  bf16       Kt, Vt [B, N, Hkv, d] bf16 (this step's tree)
 *   Kc, Vc [B, Hkv, cap, d] bf16, the first L[b] positions valid
 *   L      [B] int32 (device), 0 <= L[b] <= cap
 *   O      [B, N, Hq, d]  fp32 output
 * d must be 128; Hq must be a multiple of Hkv; scale positive and finite.
 * All pointers 16-byte aligned.  Keys are read in tiles of 64 positions:
 * the cache rows from L[b] up to the next multiple of 64 (inside the buffer)
 * are read and given weight zero, so they must hold finite values (a
 * zero-initialised cache does).
 * ws: at least tr_verify_attn_workspace_bytes(...) bytes, zeroed once before
 * first use; every call leaves its counters at zero again.  TR_E_INVAL for a
 * bad argument, TR_E_UNSUPPORTED for d != 128, B > 1024 or sizes past the
 * kernel's 31-bit tile indexing. */
int tr_verify_attn(const void *Q, const void *Kt, const void *Vt, const void *Kc, const void *Vc,
                   const int32_t *L, int cap, int B, int Hq, int Hkv, int d, float scale,
                   const struct tr_tree *tree, float *O, void *ws, size_t ws_bytes, tr_stream_t stream);
size_t tr_verify_attn_workspace_bytes(int B, int Hq, int Hkv, int d, int cap, const struct tr_tree *tree);

/* ------------------------------------------------------------------------ */
/* 3. Top-K                                                                   */
/* ------------------------------------------------------------------------ */

/* Chinese hyper.ai summary, section 方法, argtopk of the update equation; blog
 * "token-recycling", 为什么叫 Token Recycling (keep the K most probable tokens
 * of every node's distribution).  For each row r < rows of logits [rows, ld]
 * (columns [0, V) used): ids[r, :] = the K largest entries, sorted by value
 * descending, ties to the lower token ID, -0.0 equal to +0.0; vals[r, :] their
 * values as fp32 (vals may be NULL).  Logits must be finite.
 *   ftype TR_F32 or TR_BF16; ids [rows, K] int32; vals [rows, K] fp32.
 * ws: tr_topk_workspace_bytes(rows, V, K) bytes, zeroed once before first use. */
int tr_topk(const void *logits, tr_ftype ftype, int64_t rows, int64_t V, int64_t ld, int K,
            int32_t *ids, float *vals, void *ws, size_t ws_bytes, tr_stream_t stream);
size_t tr_topk_workspace_bytes(int64_t rows, int64_t V, int K);

/* tr_topk plus each row's softmax statistics at temperature T, for acceptance
 * under sampling (speculative-decoding lesson, the acceptance rule, which
 * needs the target's probabilities p = softmax(x / T)): in the same single
 * read of the logits, stats[r, 0] = max_v x[r, v] and
 * stats[r, 1] = sum_v exp((x[r, v] - stats[r, 0]) / T), and the same pair
 * for every 8 KB step of the row (2048 fp32 or 4096 bf16 entries; step s
 * covers entries [s*E, (s+1)*E)): step_stats[r, s, 0] = the step's maximum,
 * step_stats[r, s, 1] = sum over the step of exp((x - that maximum) / T).
 * fp32 throughout (exp2 of the fp32-scaled difference): relative error
 * ~1e-6.
 *   stats [rows, 2], step_stats [rows, tr_softmax_steps(V, ftype), 2] fp32;
 *   temperature positive and finite.
 * logits and ld * element size must be 16-byte aligned (TR_E_UNSUPPORTED
 * otherwise).  ws: tr_topk_workspace_bytes(rows, V, K) bytes, zeroed once. */
int tr_topk_softmax(const void *logits, tr_ftype ftype, int64_t rows, int64_t V, int64_t ld, int K,
                    float temperature, int32_t *ids, float *vals, float *stats, float *step_stats, void *ws,
                    size_t ws_bytes, tr_stream_t stream);
/* Steps per row of tr_topk_softmax's step_stats: ceil(V * element size / 8192). */
int tr_softmax_steps(int64_t V, tr_ftype ftype);

/* Allocation-free variant of tr_topk (the paper has no counterpart; this is a
 * library convenience).  For callers that hold logits, ids and vals on the
 * device but cannot get more device memory: a plugin whose host framework owns
 * every device buffer and gives plugins no workspace, a serving loop that must
 * not call cudaMalloc (it can synchronise the device and stall every stream),
 * or a foreign-function caller without an allocator.
 * Same arguments and results as tr_topk, minus the workspace: the scratch
 * lives in a static device array of TR_TOPK_NOALLOC_SCRATCH_BYTES inside the
 * library, held by every GPU that loads it until the process exits.  Sizes
 * whose scratch (tr_topk_workspace_bytes(rows, V, K)) exceeds that maximum are
 * refused with TR_E_UNSUPPORTED before any launch.  The call allocates
 * nothing: it clears the array's arrival counters with cudaMemsetAsync and
 * launches the tr_topk kernel on the array.
 * The first call on each device looks up the array's device address (with
 * that device current); make that first call before any stream capture.
 * Every call on a device shares the one array and it keeps the previous
 * call's contents, so calls that overlap on the GPU (other streams, other
 * host threads) race: serialise them on one stream. */
#define TR_TOPK_NOALLOC_SCRATCH_BYTES (4u << 20)
int tr_topk_noalloc(const void *logits, tr_ftype ftype, int64_t rows, int64_t V, int64_t ld, int K,
                    int32_t *ids, float *vals, tr_stream_t stream);

/* Fused LM head + top-K: logits = H . Wt^T (bf16 operands, fp32 accumulation)
 * and the top-K of each row as in tr_topk, without writing the logits.  The
 * distributions of the verified nodes come from the target's final
 * projection (blog, 为什么叫 Token Recycling).
 *   H  [rows, D] bf16 hidden states     Wt [V, D] bf16 (vocabulary-major)
 *   ids [rows, K] int32, vals [rows, K] fp32 (may be NULL)
 * D must be a multiple of 64; rows, V any positive size.
 * ws: tr_lmhead_topk_workspace_bytes(rows, D, V, K) bytes, zeroed once. */
int tr_lmhead_topk(const void *H, const void *Wt, int64_t rows, int D, int64_t V, int K,
                   int32_t *ids, float *vals, void *ws, size_t ws_bytes, tr_stream_t stream);
size_t tr_lmhead_topk_workspace_bytes(int64_t rows, int D, int64_t V, int K);

/* ------------------------------------------------------------------------ */
/* 4. Acceptance                                                              */
/* ------------------------------------------------------------------------ */

/* Blog "token-recycling", 完整工作流程 step 4; hyper.ai summary, "Method": the
 * longest tree path whose every token equals its parent's greedy choice
 * (ids[., ., 0]) is accepted; the target's choice after its last node (the
 * speculative-decoding lesson's bonus token) is appended.  Ties between
 * equally long paths go to the smallest BFS index.
 *   tree_tok [B, N] int32; ids [B, N, K] int32 (only column 0 is read)
 *   acc_len  [B] int32 out, accepted draft tokens (0 .. max depth)
 *   path     [B, D+1] int32 out, node indices root..last accepted, -1 padded
 *   committed[B, D+1] int32 out, accepted tokens then the bonus, -1 padded
 *   bonus    [B] int32 out, the next root (may alias the root buffer given to
 *            tr_retrieve).  D = the tree's max depth. */
int tr_accept(const struct tr_tree *tree, int B, const int32_t *tree_tok, const int32_t *ids, int K,
              int32_t *acc_len, int32_t *path, int32_t *committed, int32_t *bonus, tr_stream_t stream);

/* Acceptance under sampling at temperature T.  The speculative-decoding
 * lesson's rule (accept a drafted x with probability min(1, p(x) / q(x));
 * on a rejection resample from norm(max(0, p - q))) applied to Token
 * Recycling's tree, whose children are deterministic (q one-hot on the child's
 * token; the hyper.ai summary, "Experiment", reports the method stays
 * effective under sampling but gives no rule for the tree): starting at the
 * root, the children of the current node are tried in rank order, child x
 * being accepted when U[b, n, i] < r(x), where r is the node's p =
 * softmax(logits / T) with the tokens of the siblings already rejected
 * removed and renormalised; the walk moves to an accepted child and stops at
 * a node n* whose children are all rejected (or a leaf).  The token committed
 * after the path is the inverse CDF of n*'s residual r at U[b, n*, K] over
 * token IDs in ascending order (the smallest y with r(0) + ... + r(y) > U).
 * As T -> 0 this is the greedy rule of tr_accept.
 *   tree_tok [B, N] int32; ids [B, N, K] int32 (the top-K; only a fallback
 *   when n*'s residual has no weight left); logits [B*N, ld] of ltype with
 *   16-byte aligned rows; stats and step_stats from tr_topk_softmax at the
 *   same T (the draw finds its step from the step sums, then reads that step
 *   of n*'s row only); U [B, N, K+1] fp32 uniforms in [0, 1) (the random
 *   numbers are inputs); outputs as in tr_accept (bonus = the drawn token).
 * fp32 arithmetic: a decision whose uniform lies within ~1e-6 of its
 * threshold may differ from exact arithmetic. */
int tr_accept_sampled(const struct tr_tree *tree, int B, const int32_t *tree_tok, const int32_t *ids, int K,
                      const void *logits, tr_ftype ltype, int64_t V, int64_t ld, const float *stats,
                      const float *step_stats, float temperature, const float *U, int32_t *acc_len,
                      int32_t *path, int32_t *committed, int32_t *bonus, tr_stream_t stream);

/* ------------------------------------------------------------------------ */
/* 5. Matrix update                                                           */
/* ------------------------------------------------------------------------ */

/* Chinese hyper.ai summary, 方法: M[x~_i] = argtopk(p~_{i+1}) for every node of
 * the verified tree, no conflict logic for duplicated tokens; blog, 为什么叫
 * Token Recycling: rejected-branch nodes write too.  For n = 0..N-1 in BFS
 * order M[b, tree_tok[b,n], :] = ids[b, n, :]; when a token occurs at several
 * writing nodes, the one latest in BFS order is the row that stays.
 * TR_UPD_ACCEPTED (the ablation) writes only the nodes of path[b, 0..acc_len[b]];
 * path and acc_len are ignored (may be NULL) for TR_UPD_ALL.
 * Tokens outside [0, V) are skipped and set TR_DEV_BAD_TOKEN. */
int tr_update(void *M, tr_itype mtype, int B, int64_t V, int K, const struct tr_tree *tree,
              const int32_t *tree_tok, const int32_t *ids, tr_upd_mode mode, const int32_t *path,
              const int32_t *acc_len, tr_stream_t stream);

/* ------------------------------------------------------------------------ */
/* KV commit and loop state                                                   */
/* ------------------------------------------------------------------------ */

/* The pages are silent on the cache; standard tree decoding is used: the
 * root (the previous bonus, which has no cached K/V yet) and the accepted
 * nodes are appended in path order,
 *   Kc[b, g, L[b] + i, :] = Kt[b, path[b, i], g, :]   (same for V), i <= acc_len[b],
 * then L[b] += acc_len[b] + 1.  A commit that would pass cap sets
 * TR_DEV_CACHE_FULL and leaves that sequence untouched.
 * ws: 4*B bytes of zeroed workspace (arrival counters); tr_kv_commit_workspace_bytes. */
int tr_kv_commit(const void *Kt, const void *Vt, void *Kc, void *Vc, int32_t *L, int cap, int B,
                 int Hkv, int d, const struct tr_tree *tree, const int32_t *path,
                 const int32_t *acc_len, void *ws, size_t ws_bytes, tr_stream_t stream);
size_t tr_kv_commit_workspace_bytes(int B);

/* ------------------------------------------------------------------------ */
/* Fused step                                                                 */
/* ------------------------------------------------------------------------ */

/* Everything after the target's forward pass of one step, in the order the
 * blog fixes (the whole tree is built from the old matrix, the update then
 * serves the next step): top-K of every node (from logits, or from H and Wt
 * through the fused LM head), acceptance, matrix update, KV commit, loop
 * state (L += acc_len + 1, root = bonus) and the next step's retrieval into
 * tree_tok. */
typedef struct tr_step_args {
  int B;
  int64_t V;
  int K;
  const struct tr_tree *tree;
  void *M;          /* [B, V, K] */
  tr_itype mtype;
  const void *logits; /* [B*N, ld] of ltype, or NULL to use H and Wt */
  tr_ftype ltype;
  int64_t ld;
  const void *H;    /* [B*N, D] bf16 (fused LM head) */
  const void *Wt;   /* [V, D] bf16 */
  int D;
  int32_t *tree_tok; /* [B, N] in: this step's tree; out: the next step's tree */
  int32_t *ids;      /* [B*N, K] out */
  float *vals;       /* [B*N, K] out, may be NULL */
  int32_t *acc_len;  /* [B] out */
  int32_t *path;     /* [B, D+1] out */
  int32_t *committed;/* [B, D+1] out */
  int32_t *root;     /* [B] in/out */
  int32_t *L;        /* [B] in/out */
  const void *Kt;    /* [B, N, Hkv, d] bf16, or NULL: no KV commit (L still advances) */
  const void *Vt;
  void *Kc;          /* [B, Hkv, cap, d] bf16 */
  void *Vc;
  int cap;
  int Hkv;
  int d;
  tr_upd_mode mode;
  void *ws;          /* tr_step_workspace_bytes(args) bytes, zeroed once */
  size_t ws_bytes;
} tr_step_args;

int tr_step(const tr_step_args *args, tr_stream_t stream);
size_t tr_step_workspace_bytes(const tr_step_args *args);

/* tr_step with the acceptance of tr_accept_sampled at temperature T: the
 * top-K also yields each row's softmax statistics (tr_topk_softmax), the walk
 * and the draw run in the fused step end, and the drawn token becomes the
 * next root.  The matrix update (the top-K of every verified node) and the
 * KV commit are those of tr_step.  U [B, N, K+1] fp32 uniforms on the device.
 * Logits only (TR_E_UNSUPPORTED with the fused LM head, whose logits are never
 * stored), 16-byte aligned rows; the same workspace as tr_step. */
int tr_step_sampled(const tr_step_args *args, float temperature, const float *U, tr_stream_t stream);

/* ------------------------------------------------------------------------ */
/* Status and workspace                                                       */
/* ------------------------------------------------------------------------ */

/* Waits for `stream`, copies the current device's status word to *host_out
 * and clears it.  Returns TR_OK when the word was 0, TR_E_DEVICE otherwise. */
int tr_get_status(int32_t *host_out, tr_stream_t stream);

/* Time limit of every bounded device wait (the tensor-core kernels' mbarrier
 * waits for copies and products, the top-K's waits for its bulk copies), in
 * nanoseconds, for the launches made after this call in this process; the
 * default is 2 s.  A wait that runs out sets TR_DEV_TIMEOUT, the kernel lets
 * the copies and products it has issued complete and returns, so the context
 * stays usable; the results of that launch are undefined and its workspace
 * must be cleared (tr_workspace_clear) before the next call that uses it.  A
 * limit far below a kernel's normal waits makes every launch give up: that is
 * how the timeout path is tested (limits under 100 us are enforced by polling,
 * since a hardware-suspended wait could outlast them).  ns in [1, 6e10];
 * *previous (may be NULL)
 * receives the limit that was in force.  TR_E_INVAL outside the range. */
int tr_set_wait_limit_ns(uint64_t ns, uint64_t *previous);

/* Zeroes a workspace (cudaMemsetAsync on stream). */
int tr_workspace_clear(void *ws, size_t ws_bytes, tr_stream_t stream);

/* Human-readable name of a tr_status value (static storage). */
const char *tr_status_string(int status);

#ifdef __cplusplus
}
#endif

#endif /* TR_H */
