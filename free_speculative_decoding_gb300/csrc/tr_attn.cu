// Tree-attention verification on the 5th-generation tensor cores.
//
// For node i and query head h (KV head g = h / (Hq/Hkv)) the output is the
// softmax-weighted sum over the cached keys [0, L[b]) and the tree nodes on the
// root-to-i path (blog "token-recycling", 完整工作流程 step 3; the
// speculative-decoding lesson's tree attention).
//
// Work decomposition (stream-K): a "pair" is (sequence, KV head, query
// head); its keys are ceil(L/64) cache tiles of 64 keys followed by
// ceil(N/64) tree tiles.  The tiles of all (sequence, KV head) are laid end to
// end and cut into equal contiguous ranges, one per CTA group (one CTA per
// SM, fewer for a small batch), so every SM streams the same number of K/V
// bytes whatever the mix of prefix lengths.  A group is GS CTAs, one per
// query head of a KV head (GS = Hq / Hkv when that fits the grid, else 1 and
// those heads are laid end to end as well): the CTAs of a group walk the
// same key tiles at the same pace, each for its own query head, so
// a K/V tile that one of them brings into L2 is read from there by the
// others.  A pair that lies inside one range is finished in place;
// a pair cut by range boundaries leaves an (m, l, O) partial per part (two
// slots per CTA), and the part that finishes last merges them.  In stream-K
// order that is usually a CTA's last segment, whose partner part finished long
// before: when every other part has already left its partial, the last part
// merges straight from its TMEM accumulators (one acquire load of the pair's
// counter decides) instead of writing, handing over and re-reading its own.
//
// Per CTA (12 warps, so each SM sub-partition hosts one helper warp and two
// softmax warps):
//   warp 0      TMA producer of the K ring: tiles of 64 keys from the cache
//               (2-D map over [B*Hkv*cap, d]) or the tree (3-D map over
//               [B*N, Hkv, d]);
//   warp 2      TMA producer of the V ring, same maps for V; the two rings
//               run independently, so a V stage still held by a PV product
//               never stops the K stream;
//   warp 1      loads Q (3-D map over [B*N, Hq, d]; one buffer, the next
//               segment's Q is prefetched into L2) and issues S = Q.K^T
//               (tcgen05.mma M128 x N64 x K128, fp32 in TMEM);
//   warp 3      issues O += P.V (M128 x N128 x K64) with P read from TMEM and V
//               from shared memory as an MN-major operand.  One thread
//               issues an MMA every ~68 cycles at best (measured), so the two
//               products come from two warps, which together keep the tensor
//               pipe busy; both run warp-uniformly and issue from one elected
//               lane;
//   warps 4..11 softmax, one query row per thread (one TMEM lane): the mask
//               (key < L for the cache, ancestor bit for the tree), exp2 with a
//               running maximum that only rescales O when it grows by more
//               than 2^8, and P written back over the S columns it came from.
//               P goes in two bf16 parts, hi = p truncated to bf16 and
//               lo = bf16(p - hi), both multiplied with V, so the weights reach
//               the accumulator with at most 2^-15 relative error instead of
//               bf16's 2^-9 (the truncation packs hi with one byte permute
//               instead of a conversion).  At the end
//               of a segment the same threads normalise O or write the
//               partial.
// TMEM holds two O accumulators (128 columns each) and four S/P buffers of
// 64 columns; a buffer is reused by the QK product four tiles later, once the
// PV product that read its P has completed.  The two softmax warpgroups take
// alternate tiles into their own accumulators (combined at the end of a
// segment).  Grouped-query heads also get one pair per query head: two heads
// per K/V tile (one warpgroup and one accumulator per head, 256 query rows
// per tile, half the K/V reads) measured slower on grouped-query shapes,
// which are bound by the tensor pipe and the exponentials.
//
// Every wait is bounded in time; a wait that gives up sets TR_DEV_TIMEOUT and
// raises a block-wide abort flag; the roles drain their in-flight copies and
// MMAs, TMEM is freed and the kernel returns.
#include <algorithm>

#include "tr_sm100.cuh"

namespace {

constexpr int kD = 128;             // head dimension
constexpr int BN = 64;              // keys per tile
constexpr float kRescaleLog2 = 8.f; // O is rescaled only when the row maximum grows by more than this
constexpr int kMaxB = 1024;
constexpr int kEarlyParts = 4;      // other parts a split pair may have for the direct merge

struct Cfg {
  // One Q buffer (the next segment's Q is prefetched into L2) leaves room for
  // five K and five V stages: a tile's copy lands ~1.25 us after it is issued,
  // and a stage is refilled only once the product that read it has completed,
  // so each ring must hold more than that latency's worth of tiles.  Measured
  // on one box against two Q buffers with 3 K + 5 V stages: 0.1294 -> 0.1229 ms
  // (batched workload), 0.1134 -> 0.1098 ms (grouped-query workload).
  static constexpr int KS = 5;                    // K ring stages
  static constexpr int VS = 5;                    // V ring stages
  static constexpr int GROUPS = 2;                // softmax warpgroups taking alternate tiles
  static constexpr int NSB = 4;                   // S/P buffers in TMEM
  static constexpr int Q_HALF = 128 * 128;        // 128 rows x 64 bf16 (one d-half), bytes
  static constexpr int KV_HALF = 64 * 128;        // 64 keys x 64 bf16
  static constexpr int KV_TILE = 2 * KV_HALF;
  static constexpr int OFF_Q = 0;
  static constexpr int Q_BUF = 2 * Q_HALF;
  static constexpr int OFF_K = OFF_Q + Q_BUF;
  static constexpr int OFF_V = OFF_K + KS * KV_TILE;
  static constexpr int OFF_BAR = OFF_V + VS * KV_TILE;
  static constexpr int SOFT = 256;                // softmax threads: two warpgroups
  static constexpr int THREADS = 128 + SOFT;
  static constexpr uint32_t TMEM_COLS = 512;
  __host__ __device__ static constexpr uint32_t o_col(int o) { return (uint32_t)(o * kD); }
  __host__ __device__ static constexpr uint32_t s_col(int buf) { return (uint32_t)(2 * kD + buf * BN); }
};
static_assert(Cfg::s_col(Cfg::NSB - 1) + BN <= Cfg::TMEM_COLS, "TMEM budget");

struct Bars {
  static constexpr int KS = Cfg::KS, VS = Cfg::VS, NSB = Cfg::NSB;
  uint64_t q_full, q_empty;
  uint64_t k_full[KS], k_empty[KS], v_full[VS], v_empty[VS];
  uint64_t s_full[NSB], p_full[NSB], pv_done[NSB];
  uint64_t o_full, o_empty, drain, ml_ready;
  uint64_t mrg_in, mrg_go;  // hand-off of a pair shared by several CTAs
  uint32_t tmem;
  int abort, mrg_last;
  int mrg_early;  // every other part of this split pair has already left its partial
  float2 ml_x[2][2][128];  // each warpgroup's (m, l) per row, by segment parity
  int Ls[kMaxB];
  int pref[kMaxB + 1];  // first tile of sequence b in the global tile order
};

struct AttnArgs {
  const int32_t *L;
  float *O;
  float *part_o;      // [grid, 2, N, d]
  float2 *part_ml;    // [grid, 2, N]
  int *cnt;           // [pairs] parts finished, back to zero after the merge
  unsigned *status;
  int B, N, Hq, Hkv, G, cap;  // G = Hq / Hkv query heads per KV head
  int GS;   // CTAs per group: one per query head of a KV head (G), or 1
  int HPS;  // query heads laid end to end per KV head in the tile order: G / GS
  int q_rows, c_rows, t_rows;  // TMA box heights (at most the tensor's extent)
  float scale_log2;
  unsigned long long wait_ns;  // limit of every bounded wait
};

__device__ __forceinline__ int tiles_per_pair(int Lb, int N) { return (Lb + BN - 1) / BN + (N + BN - 1) / BN; }

// Range of global tiles owned by CTA group c of `groups`.
__device__ __forceinline__ long long range_start(long long total, int c, int groups) { return total * c / groups; }

// Group whose range holds global tile t (the inverse of range_start).
__device__ __forceinline__ int range_owner(long long t, long long total, int groups) {
  return (int)(((t + 1) * groups + total - 1) / total - 1);
}

// A run of consecutive tiles of one pair inside one CTA's range.
struct Seg {
  int b, g, hg, pair, Lb;
  int j0, n;    // first tile within the pair, number of tiles
  int n_ct;     // cache tiles of the pair
  bool complete, first_of_cta;
};

__device__ __forceinline__ Seg decode(long long t, long long t_lo, long long t_hi, const int *pref, const int *Ls,
                                      const AttnArgs &a) {
  int lo = 0, hi = a.B - 1;  // largest b with pref[b] <= t
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (pref[mid] <= t) lo = mid;
    else hi = mid - 1;
  }
  Seg s;
  s.b = lo;
  s.Lb = Ls[lo];
  const int tpp = tiles_per_pair(s.Lb, a.N);
  const long long r = t - pref[lo];
  const int pib = (int)(r / tpp);
  s.j0 = (int)(r % tpp);
  s.g = pib / a.HPS;
  s.hg = (pib % a.HPS) * a.GS + (int)(blockIdx.x % a.GS);  // query head within the KV head
  s.pair = (s.b * a.Hkv + s.g) * a.G + s.hg;
  s.n = (int)min((long long)(tpp - s.j0), t_hi - t);
  s.n_ct = (s.Lb + BN - 1) / BN;
  s.complete = s.j0 == 0 && s.n == tpp;
  s.first_of_cta = t == t_lo;
  return s;
}

// Walks a CTA's tiles segment by segment: u is the tile's index inside the
// current segment, sc the segment's index inside the CTA.
struct Cursor {
  long long t;  // first tile of the current segment
  Seg sg;
  int u, sc;
  __device__ __forceinline__ void init(long long t_lo, long long t_hi, const int *pref, const int *Ls,
                                       const AttnArgs &a) {
    t = t_lo;
    u = 0;
    sc = 0;
    if (t < t_hi) sg = decode(t, t_lo, t_hi, pref, Ls, a);
  }
  __device__ __forceinline__ bool last() const { return u == sg.n - 1; }
  __device__ __forceinline__ void advance(long long t_lo, long long t_hi, const int *pref, const int *Ls,
                                          const AttnArgs &a) {
    if (++u < sg.n) return;
    t += sg.n;
    u = 0;
    ++sc;
    if (t < t_hi) sg = decode(t, t_lo, t_hi, pref, Ls, a);
  }
};

__global__ void __launch_bounds__(Cfg::THREADS, 1)
    attn_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmKc,
                   const __grid_constant__ CUtensorMap tmVc, const __grid_constant__ CUtensorMap tmKt,
                   const __grid_constant__ CUtensorMap tmVt, const AttnArgs a, const __grid_constant__ TreeDev tree) {
  using namespace sm100;
  using C = Cfg;
  constexpr int KS = C::KS, VS = C::VS, NSB = C::NSB, GROUPS = C::GROUPS;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  Bars *bars = (Bars *)(smem + C::OFF_BAR);
  volatile int *abort = &bars->abort;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int N = a.N;

  if (threadIdx.x == 0) {
    mbar_init(&bars->q_full, 1);
    mbar_init(&bars->q_empty, 1);
    for (int s = 0; s < KS; ++s) {
      mbar_init(&bars->k_full[s], 1);
      mbar_init(&bars->k_empty[s], 1);
    }
    for (int s = 0; s < VS; ++s) {
      mbar_init(&bars->v_full[s], 1);
      mbar_init(&bars->v_empty[s], 1);
    }
    for (int b = 0; b < NSB; ++b) {
      mbar_init(&bars->s_full[b], 1);
      mbar_init(&bars->p_full[b], 128);
      mbar_init(&bars->pv_done[b], 1);
    }
    mbar_init(&bars->o_full, 1);
    mbar_init(&bars->o_empty, C::SOFT);
    mbar_init(&bars->drain, 2);  // one commit from each MMA issuer
    mbar_init(&bars->ml_ready, 256);
    mbar_init(&bars->mrg_in, C::SOFT);
    mbar_init(&bars->mrg_go, 1);
    bars->abort = 0;
    fence_mbar_init();
  }
  // A TMA box shorter than a 64-key tile (a tree or cache tensor of fewer
  // than 64 rows: tiny batches) leaves the tile's last rows unwritten.  Their
  // keys get weight zero, but zero times a NaN left in shared memory would
  // still reach O, so the V ring starts zeroed then.
  if (a.t_rows < BN || a.c_rows < BN) {
    uint4 *vr = reinterpret_cast<uint4 *>(smem + C::OFF_V);
    for (int i = threadIdx.x; i < VS * C::KV_TILE / 16; i += blockDim.x) vr[i] = make_uint4(0u, 0u, 0u, 0u);
    fence_proxy_async_smem();  // the zeros come before the ring's first copies and products
  }
  for (int b = threadIdx.x; b < a.B; b += blockDim.x) {
    int Lb = a.L[b];
    if (Lb < 0 || Lb > a.cap) {
      if (blockIdx.x == 0) tr_flag(a.status, TR_DEV_BAD_LENGTH);
      Lb = Lb < 0 ? 0 : a.cap;
    }
    bars->Ls[b] = Lb;
  }
  if (warp == 1) tmem_alloc(&bars->tmem, C::TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (threadIdx.x == 0) {
    int acc = 0;
    for (int b = 0; b < a.B; ++b) {
      bars->pref[b] = acc;
      acc += tiles_per_pair(bars->Ls[b], N) * a.Hkv * a.HPS;
    }
    bars->pref[a.B] = acc;
  }
  __syncthreads();
  const uint32_t tmem = bars->tmem;
  const long long total = bars->pref[a.B];
  const int groups = (int)gridDim.x / a.GS, grp_id = (int)blockIdx.x / a.GS;
  const long long t_lo = range_start(total, grp_id, groups);
  const long long t_hi = range_start(total, grp_id + 1, groups);

  auto give_up = [&]() {
    if (!*abort) {
      *abort = 1;
      tr_flag(a.status, TR_DEV_TIMEOUT);
    }
  };

  // every wait of the warp-wide roles is warp-uniform: a lane that gives up
  // takes its whole warp with it, so warp-collective instructions stay converged
  auto wwait = [&](uint64_t *bar, uint32_t parity) -> bool {
    const bool mine = mbar_wait(bar, parity, abort, a.wait_ns);
    const bool all = __all_sync(0xffffffffu, mine);
    if (!all) give_up();
    return all;
  };

  if (warp == 0 || warp == 2) {
    // ------------------------------------------------------------ producers
    if (lane == 0) {
      const bool is_k = warp == 0;
      constexpr int SMAX = KS > VS ? KS : VS;
      const int NS = is_k ? KS : VS;
      uint64_t *full = is_k ? bars->k_full : bars->v_full;
      uint64_t *empty = is_k ? bars->k_empty : bars->v_empty;
      const CUtensorMap *mc = is_k ? &tmKc : &tmVc;
      const CUtensorMap *mt = is_k ? &tmKt : &tmVt;
      uint8_t *ring = smem + (is_k ? C::OFF_K : C::OFF_V);
      if (is_k) {
        tma_prefetch_desc(&tmKc);
        tma_prefetch_desc(&tmKt);
      } else {
        tma_prefetch_desc(&tmVc);
        tma_prefetch_desc(&tmVt);
      }
      const uint64_t kv_policy = l2_evict_first();  // the cache streams through once
      int cnt = 0, last[SMAX];
      for (int s = 0; s < SMAX; ++s) last[s] = -1;
      bool ok = true;
      for (long long t = t_lo; t < t_hi && ok && !*abort;) {
        const Seg sg = decode(t, t_lo, t_hi, bars->pref, bars->Ls, a);
        t += sg.n;
        for (int u = 0; u < sg.n; ++u) {
          const int j = sg.j0 + u;
          const bool cache = j < sg.n_ct;
          const int s = cnt % NS;
          const uint32_t ph = (cnt / NS) & 1;
          if (!mbar_wait(&empty[s], ph ^ 1, abort, a.wait_ns)) {
            give_up();
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&full[s], (uint32_t)(2 * (cache ? a.c_rows : a.t_rows) * 128));
          uint8_t *dst = ring + s * C::KV_TILE;
          for (int half = 0; half < 2; ++half) {
            if (cache)
              tma_load_2d_hint(dst + half * C::KV_HALF, mc, &full[s], half * 64, (sg.b * a.Hkv + sg.g) * a.cap + j * BN,
                               kv_policy);
            else
              tma_load_3d(dst + half * C::KV_HALF, mt, &full[s], half * 64, sg.g, sg.b * N + (j - sg.n_ct) * BN);
          }
          last[s] = (int)ph;
          ++cnt;
        }
      }
      if (*abort) {
        // let the copies already issued land before the CTA can exit
        for (int s = 0; s < NS; ++s)
          if (last[s] >= 0) mbar_drain(&full[s], (uint32_t)last[s]);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------- QK issuer
    // S = Q.K^T of tile i once its Q and K have landed and the S/P buffer's
    // previous PV product has completed.  The whole warp runs the loop, so its
    // control flow and operands stay warp-uniform; one elected lane issues.
    // This warp also loads Q into the one buffer, once the previous segment's
    // last product is done; the next segment's Q is prefetched into L2 meanwhile.
    constexpr uint32_t kIdesc = idesc_bf16_f32(128, BN);
    const uint64_t dq0 = desc_kmajor_sw128(smem_u32(smem + C::OFF_Q));
    const uint64_t dk0 = desc_kmajor_sw128(smem_u32(smem + C::OFF_K));
    int q_armed = -1;  // parity of the last Q load, -1 for none
    auto load_q = [&](const Seg &sg, int sc_of) {
      if (elect_one()) {
        mbar_arrive_expect_tx(&bars->q_full, (uint32_t)(2 * a.q_rows * 128));
        const int h = sg.g * a.G + sg.hg;
        for (int half = 0; half < 2; ++half)
          tma_load_3d(smem + C::OFF_Q + half * C::Q_HALF, &tmQ, &bars->q_full, half * 64, h, sg.b * N);
      }
      __syncwarp();
      q_armed = sc_of & 1;
    };
    Cursor cq;
    cq.init(t_lo, t_hi, bars->pref, bars->Ls, a);
    const int n_all = (int)(t_hi - t_lo);
    if (lane == 0) tma_prefetch_desc(&tmQ);
    if (n_all > 0) load_q(cq.sg, 0);
    for (int i = 0; i < n_all; ++i) {
      const int sb = i % NSB, ks = i % KS;
      if (cq.u == 0) {
        const long long t_next = cq.t + cq.sg.n;  // first tile of the next segment
        if (cq.sc > 0) {
          // the buffer held the previous segment's Q: refill it once its last product is done
          if (!wwait(&bars->q_empty, (cq.sc - 1) & 1)) break;
          load_q(cq.sg, cq.sc);
        }
        if (t_next < t_hi && lane == 0) {
          const Seg nx = decode(t_next, t_lo, t_hi, bars->pref, bars->Ls, a);
          for (int half = 0; half < 2; ++half)
            tma_prefetch_l2_3d(&tmQ, half * 64, nx.g * a.G + nx.hg, nx.b * N);
        }
        if (!wwait(&bars->q_full, cq.sc & 1)) break;
      }
      if (!wwait(&bars->k_full[ks], (i / KS) & 1)) break;
      if (i >= NSB && !wwait(&bars->pv_done[sb], ((i / NSB) - 1) & 1)) break;
      tc_fence_after();
      if (elect_one()) {
        // descriptor start addresses count 16-byte units
        const uint64_t dk = dk0 + (uint64_t)(ks * (C::KV_TILE >> 4));
#pragma unroll
        for (int k = 0; k < kD / 16; ++k)
          mma_bf16(tmem + C::s_col(sb), dq0 + (uint64_t)(((k >> 2) * C::Q_HALF + (k & 3) * 32) >> 4),
                   dk + (uint64_t)(((k >> 2) * C::KV_HALF + (k & 3) * 32) >> 4), kIdesc, k > 0 ? 1u : 0u);
        mma_commit(&bars->k_empty[ks]);
        mma_commit(&bars->s_full[sb]);
        if (cq.last()) mma_commit(&bars->q_empty);
      }
      __syncwarp();
      cq.advance(t_lo, t_hi, bars->pref, bars->Ls, a);
    }
    if (*abort) {
      // let the Q copy already issued land before the CTA can exit
      if (q_armed >= 0) mbar_drain(&bars->q_full, (uint32_t)q_armed);
    }
    if (elect_one()) mma_commit(&bars->drain);
    __syncwarp();
    mbar_drain(&bars->drain, 0);
  } else if (warp == 3) {
    // ------------------------------------------------------------- PV issuer
    // O += P.V of tile i once its P is in TMEM and its V has landed; the first
    // tile of a segment also waits for the previous segment's epilogue to have
    // read the accumulators.
    constexpr uint32_t kIdesc = idesc_bf16_f32(128, kD, true);
    const uint64_t dv0 = desc_mnmajor_sw128(smem_u32(smem + C::OFF_V), C::KV_HALF);
    Cursor cp;
    cp.init(t_lo, t_hi, bars->pref, bars->Ls, a);
    const int n_all = (int)(t_hi - t_lo);
    for (int i = 0; i < n_all; ++i) {
      const int sb = i % NSB, vs = i % VS;
      if (cp.u == 0 && !wwait(&bars->o_empty, (cp.sc & 1) ^ 1)) break;
      if (!wwait(&bars->p_full[sb], (i / NSB) & 1)) break;
      if (!wwait(&bars->v_full[vs], (i / VS) & 1)) break;
      tc_fence_after();
      if (elect_one()) {
        const uint64_t dv = dv0 + (uint64_t)(vs * (C::KV_TILE >> 4));
        const uint32_t first = cp.u >= GROUPS ? 1u : 0u;
        const uint32_t d_o = tmem + C::o_col(i & 1);  // tile i's warpgroup owns accumulator i & 1
        const uint32_t a_p = tmem + C::s_col(sb);
#pragma unroll
        for (int part = 0; part < 2; ++part)
#pragma unroll
          for (int k = 0; k < BN / 16; ++k)
            mma_bf16_ts(d_o, a_p + part * 32 + k * 8, dv + (uint64_t)(k * (2048 >> 4)), kIdesc,
                        (part > 0 || k > 0) ? 1u : first);
        mma_commit(&bars->v_empty[vs]);
        mma_commit(&bars->pv_done[sb]);
        if (cp.last()) mma_commit(&bars->o_full);
      }
      __syncwarp();
      cp.advance(t_lo, t_hi, bars->pref, bars->Ls, a);
    }
    if (elect_one()) mma_commit(&bars->drain);
    __syncwarp();
    mbar_drain(&bars->drain, 0);
  } else {
    // -------------------------------------------------------------- softmax
    const int grp = (warp - 4) >> 2;           // softmax warpgroup: takes tiles grp, grp + 2, ...
    const int oacc = grp;                      // this warpgroup's O accumulator
    const int quad = warp & 3;                 // TMEM lanes quad*32 .. +31
    const int r = quad * 32 + lane;
    const bool warp_active = quad * 32 < N;
    const bool row_valid = r < N;
    const int rn = row_valid ? r : 0;
    const unsigned long long anc0 = tree.anc[rn][0], anc1 = tree.anc[rn][1];
    const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
    int gt = 0, sc = 0, n_split = 0;
    bool ok = true;
    const int cg = (int)blockIdx.x % a.GS;  // this CTA's place in its group
    for (long long t = t_lo; t < t_hi && ok; ++sc) {
      const Seg sg = decode(t, t_lo, t_hi, bars->pref, bars->Ls, a);
      const long long p_first = t - sg.j0;  // the pair's first tile in the global order
      t += sg.n;
      const int T = sg.n;
      const int h = sg.g * a.G + sg.hg;
      float m_run = -INFINITY, l_run = 0.f;  // running maximum (log2 units) and sum
      int done_here = 0;  // tiles of this segment this warpgroup has folded into its accumulator
      for (int u = 0; u < T && ok; ++u) {
        const int gtt = gt + u, sb = gtt % NSB;
        if ((gtt & 1) != grp) continue;  // the other warpgroup's tile
        // also for inactive warps: their p_full arrival must not run ahead
        // into the buffer's next use
        if (!wwait(&bars->s_full[sb], (gtt / NSB) & 1)) {
          ok = false;
          break;
        }
        tc_fence_after();
        if (warp_active) {
          const uint32_t scol = tmem + lane_off + C::s_col(sb);
          float sv[BN];
          tmem_ld64(scol, sv);
          const int j = sg.j0 + u;
          const bool cache = j < sg.n_ct;
          const int key0 = j * BN;
          if (!(cache && key0 + BN <= sg.Lb)) {
            // a tile with invisible keys (the cache's last tile, the tree
            // tiles): -inf where the validity mask has a zero.  A full cache
            // tile needs none (its rows past N are never stored).
            unsigned long long vm;
            if (cache) {
              vm = (1ull << (sg.Lb - key0)) - 1;  // 1 <= Lb - key0 < 64 here
            } else {
              const int node0 = (j - sg.n_ct) * BN, nv = N - node0;
              vm = (node0 == 0 ? anc0 : anc1) & (nv >= 64 ? ~0ull : (1ull << nv) - 1);
            }
            if (!row_valid) vm = 0;
            const uint32_t vlo = (uint32_t)vm, vhi = (uint32_t)(vm >> 32);
#pragma unroll
            for (int c = 0; c < BN; ++c)
              if (!(((c < 32 ? vlo : vhi) >> (c & 31)) & 1u)) sv[c] = -INFINITY;
          }
          float mx4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};  // four independent chains
#pragma unroll
          for (int c = 0; c < BN; c += 2) mx4[(c >> 1) & 3] = fmax3(mx4[(c >> 1) & 3], sv[c], sv[c + 1]);
          // the scale is positive, so the maximum of the raw scores scales to the scaled maximum
          const float mx = fmaxf(fmaxf(mx4[0], mx4[1]), fmaxf(mx4[2], mx4[3])) * a.scale_log2;
          const float m_new = fmaxf(m_run, mx);
          const bool need = m_new > m_run + kRescaleLog2;  // also true for the row's first finite maximum
          if (__any_sync(0xffffffffu, need && done_here > 0)) {
            // O already holds this warpgroup's earlier tiles: wait for the last PV into it, then scale it
            const int gp = gtt - GROUPS;
            if (!wwait(&bars->pv_done[gp % NSB], (gp / NSB) & 1)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const float f = (need && m_run != -INFINITY) ? ex2(m_run - m_new) : 1.f;
#pragma unroll 1
            for (int c0 = 0; c0 < kD; c0 += 32) {
              float ov[32];
              tmem_ld32(tmem + lane_off + C::o_col(oacc) + c0, ov);
#pragma unroll
              for (int c = 0; c < 32; ++c) ov[c] *= f;
              tmem_st32(tmem + lane_off + C::o_col(oacc) + c0, ov);
            }
          }
          if (need) {
            l_run = m_run == -INFINITY ? 0.f : l_run * ex2(m_run - m_new);
            m_run = m_new;
          }
          // ex2(-inf) = 0 for masked keys; a row that has seen no visible key yet
          // (m_run = -inf, all its keys masked) subtracts 0 instead of -inf
          const float m_sub = m_run == -INFINITY ? 0.f : m_run;
          float l4[4] = {0.f, 0.f, 0.f, 0.f};  // four independent chains
          // P over the S columns just read: hi parts in the first 32, lo in the next 32
#pragma unroll
          for (int half = 0; half < 2; ++half) {
            uint32_t whi[16], wlo[16];
#pragma unroll
            for (int q = 0; q < 16; ++q) {
              const int c = half * 32 + 2 * q;
              const float p0 = ex2(fmaf(sv[c], a.scale_log2, -m_sub));
              const float p1 = ex2(fmaf(sv[c + 1], a.scale_log2, -m_sub));
              l4[q & 3] += p0 + p1;
              // hi: p truncated to bf16 (its upper 16 bits, packed by one byte
              // permute); lo: the exact remainder rounded to bf16
              const uint32_t u0 = __float_as_uint(p0), u1 = __float_as_uint(p1);
              const __nv_bfloat162 lo = __floats2bfloat162_rn(p0 - __uint_as_float(u0 & 0xffff0000u),
                                                              p1 - __uint_as_float(u1 & 0xffff0000u));
              whi[q] = __byte_perm(u0, u1, 0x7632);
              wlo[q] = *reinterpret_cast<const uint32_t *>(&lo);
            }
            tmem_st16_nowait(scol + half * 16, whi);
            tmem_st16_nowait(scol + 32 + half * 16, wlo);
          }
          tmem_wait_st();
          l_run += (l4[0] + l4[1]) + (l4[2] + l4[3]);
        }
        ++done_here;
        tc_fence_before();
        mbar_arrive(&bars->p_full[sb]);
      }
      if (!ok) break;
      // ---- end of the segment: normalised output or a partial
      if (!done_here) {
        m_run = -INFINITY;
        l_run = 0.f;
      }
      // the CTA groups that own parts of a split pair: group q owns
      // [total*q/groups, total*(q+1)/groups); its CTA for this query head is q*GS + cg
      const long long p_total = bars->pref[a.B];
      const long long p_last = p_first + tiles_per_pair(sg.Lb, N) - 1;
      const int pc0 = range_owner(p_first, p_total, groups), pc1 = range_owner(p_last, p_total, groups);
      // with fewer tiles than groups some ranges are empty, and such a group
      // between the owners holds no part of the pair
      auto owns = [&](int q) { return range_start(p_total, q, groups) < range_start(p_total, q + 1, groups); };
      int others = 0;  // parts of this pair in other CTAs
      if (!sg.complete)
        for (int q = pc0; q <= pc1; ++q) others += q != grp_id && owns(q) ? 1 : 0;
      // A split pair whose other parts have all left their partials (at most
      // kEarlyParts of them): this part merges straight from its accumulators
      // instead of writing a partial, handing over and reading it back.
      if (threadIdx.x == 128 && !sg.complete) {
        int seen;
        asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(seen) : "l"(a.cnt + sg.pair) : "memory");
        bars->mrg_early = others <= kEarlyParts && seen == others;
      }
      // both warpgroups publish their (m, l); each then finishes half of the d columns
      bars->ml_x[sc & 1][grp][r] = make_float2(m_run, l_run);
      mbar_arrive(&bars->ml_ready);
      if (!wwait(&bars->o_full, sc & 1)) break;
      tc_fence_after();
      if (!wwait(&bars->ml_ready, sc & 1)) break;
      const float2 other = bars->ml_x[sc & 1][grp ^ 1][r];
      const float M = fmaxf(m_run, other.x);
      const float wa = m_run == -INFINITY ? 0.f : ex2(m_run - M);   // this warpgroup's accumulator
      const float wb = other.x == -INFINITY ? 0.f : ex2(other.x - M);  // the other warpgroup's
      const float l = l_run * wa + other.y * wb;
      constexpr int COLS = kD / 2;  // columns this warpgroup finishes
      const int col0 = grp * COLS;
      const bool early = !sg.complete && bars->mrg_early;
      const int slot_pc0 = (pc0 * a.GS + cg) * 2 + (range_start(p_total, pc0, groups) < p_first ? 1 : 0);
      auto part_row = [&](int q) {
        const int slot = q == pc0 ? slot_pc0 : (q * a.GS + cg) * 2;
        return (long long)slot * N + r;
      };
      if (early) {
        if (warp_active) {
          // No fence is needed before reading the other parts: each part
          // fenced its writes before counting itself, the counter was read
          // with acquire semantics, and that thread's mbarrier arrival
          // (release) and this thread's wait (acquire) order these loads after it.
          // The first other part's row (this warpgroup's columns) and every
          // other part's (m, l) are requested before any is used: the loads
          // queue behind the other CTAs' K/V streams, so each round trip
          // costs microseconds.
          int rk[kEarlyParts];  // partial rows: below 2 * grid * N
          int nk = 0;
#pragma unroll 1
          for (int q = pc0; q <= pc1 && nk < kEarlyParts; ++q)
            if (q != grp_id && owns(q)) rk[nk++] = (int)part_row(q);
          float4 o1[COLS / 4];
          const float4 *src1 = reinterpret_cast<const float4 *>(a.part_o + (long long)rk[0] * kD + col0);
#pragma unroll
          for (int i = 0; i < COLS / 4; ++i) o1[i] = nk > 0 && row_valid ? __ldcg(src1 + i) : make_float4(0.f, 0.f, 0.f, 0.f);
          float2 mlk[kEarlyParts];
#pragma unroll
          for (int k = 0; k < kEarlyParts; ++k)
            mlk[k] = k < nk && row_valid ? __ldcg(&a.part_ml[rk[k]]) : make_float2(-INFINITY, 0.f);
          float Mx = M;  // this part's maximum from above
#pragma unroll
          for (int k = 0; k < kEarlyParts; ++k) Mx = fmaxf(Mx, mlk[k].x);
          const float wown = M == -INFINITY ? 0.f : ex2(M - Mx);
          float den = l * wown;
          float wk[kEarlyParts];
#pragma unroll
          for (int k = 0; k < kEarlyParts; ++k) {
            wk[k] = mlk[k].x == -INFINITY ? 0.f : ex2(mlk[k].x - Mx);
            den += mlk[k].y * wk[k];
          }
          const float inv = den > 0.f ? 1.f / den : 0.f;  // > 0 for a valid row: every node sees itself
          const float w0 = (grp == 0 ? wa : wb) * wown, w1 = (grp == 0 ? wb : wa) * wown;
          float *dst = a.O + (((long long)sg.b * N + r) * a.Hq + h) * kD;
#pragma unroll
          for (int ch = 0; ch < COLS / 32; ++ch) {
            const int c0 = col0 + ch * 32;
            float oa[32], ob[32];
            tmem_ld32(tmem + lane_off + C::o_col(0) + c0, oa);
            tmem_ld32(tmem + lane_off + C::o_col(1) + c0, ob);
            if (ch == COLS / 32 - 1) {
              // the last read of the accumulators: the next segment's PV may overwrite them
              tc_fence_before();
              mbar_arrive(&bars->o_empty);
            }
            if (row_valid) {
#pragma unroll
              for (int c = 0; c < 32; ++c) oa[c] = (w0 != 0.f ? oa[c] * w0 : 0.f) + (w1 != 0.f ? ob[c] * w1 : 0.f);
#pragma unroll
              for (int i = 0; i < 8; ++i) {
                const float4 v = o1[ch * 8 + i];
                oa[4 * i] += v.x * wk[0];
                oa[4 * i + 1] += v.y * wk[0];
                oa[4 * i + 2] += v.z * wk[0];
                oa[4 * i + 3] += v.w * wk[0];
              }
#pragma unroll 1
              for (int k = 1; k < nk; ++k) {
                const float4 *src = reinterpret_cast<const float4 *>(a.part_o + (long long)rk[k] * kD + c0);
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                  const float4 v = __ldcg(src + i);
                  oa[4 * i] += v.x * wk[k];
                  oa[4 * i + 1] += v.y * wk[k];
                  oa[4 * i + 2] += v.z * wk[k];
                  oa[4 * i + 3] += v.w * wk[k];
                }
              }
#pragma unroll
              for (int c = 0; c < 32; c += 4)
                *reinterpret_cast<float4 *>(dst + c + c0) =
                    make_float4(oa[c] * inv, oa[c + 1] * inv, oa[c + 2] * inv, oa[c + 3] * inv);
            }
          }
          if (threadIdx.x == 128) a.cnt[sg.pair] = 0;  // the workspace is left zeroed
        } else {
          tc_fence_before();
          mbar_arrive(&bars->o_empty);
        }
      } else if (warp_active) {
        const int slot = blockIdx.x * 2 + (sg.first_of_cta ? 0 : 1);
        const long long prow_idx = (long long)slot * N + r;
        const float scale_out = sg.complete ? (row_valid && l > 0.f ? 1.f / l : 0.f) : 1.f;
        // fold accumulator 0 with weight w0 and accumulator 1 with w1
        const float w0 = grp == 0 ? wa : wb;
        const float w1 = grp == 0 ? wb : wa;
        float *dst = sg.complete ? a.O + (((long long)sg.b * N + r) * a.Hq + h) * kD : a.part_o + prow_idx * kD;
#pragma unroll 1
        for (int c0 = col0; c0 < col0 + COLS; c0 += 32) {
          float oa[32], ob[32];
          tmem_ld32(tmem + lane_off + C::o_col(0) + c0, oa);
          tmem_ld32(tmem + lane_off + C::o_col(1) + c0, ob);
          if (c0 + 32 == col0 + COLS) {
            // the last read of the accumulators: the next segment's PV may overwrite them
            tc_fence_before();
            mbar_arrive(&bars->o_empty);
          }
          if (row_valid) {
#pragma unroll
            for (int c = 0; c < 32; ++c) {
              float v = w0 != 0.f ? oa[c] * w0 : 0.f;
              if (w1 != 0.f) v += ob[c] * w1;
              oa[c] = v * scale_out;
            }
#pragma unroll
            for (int c = 0; c < 32; c += 4)
              *reinterpret_cast<float4 *>(dst + c + c0) = make_float4(oa[c], oa[c + 1], oa[c + 2], oa[c + 3]);
          }
        }
        if (!sg.complete && row_valid && grp == 0) a.part_ml[prow_idx] = make_float2(M, l);
      } else {
        tc_fence_before();
        mbar_arrive(&bars->o_empty);
      }
      if (!sg.complete && !early) {
        // A pair shared by several CTAs (cut by range boundaries): each part
        // leaves its partial in a slot and counts itself; the last part to
        // finish merges them all and resets the counter.
        __threadfence();
        mbar_arrive(&bars->mrg_in);
        if (threadIdx.x == 128) {
          int is_last = 0;
          if (mbar_wait(&bars->mrg_in, n_split & 1, abort, a.wait_ns)) {
            __threadfence();
            is_last = atomicAdd(&a.cnt[sg.pair], 1) == others;
            __threadfence();
          } else {
            give_up();
          }
          bars->mrg_last = is_last;
          mbar_arrive(&bars->mrg_go);
        }
        if (!wwait(&bars->mrg_go, n_split & 1)) break;
        ++n_split;
        if (bars->mrg_last) {
          __threadfence();
          if (warp_active && row_valid) {
#pragma unroll 1
            for (int ch = col0; ch < col0 + COLS; ch += 64) {
              float Mx = -INFINITY;
#pragma unroll 1
              for (int q = pc0; q <= pc1; ++q)
                if (owns(q)) Mx = fmaxf(Mx, a.part_ml[part_row(q)].x);
              float acc[64];
#pragma unroll
              for (int i = 0; i < 64; ++i) acc[i] = 0.f;
              float den = 0.f;
#pragma unroll 1
              for (int q = pc0; q <= pc1; ++q) {
                if (!owns(q)) continue;
                const long long row = part_row(q);
                const float2 ml = a.part_ml[row];
                const float w = ml.x == -INFINITY ? 0.f : ex2(ml.x - Mx);
                den += ml.y * w;
                const float4 *src = reinterpret_cast<const float4 *>(a.part_o + row * kD + ch);
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                  const float4 v = src[i];
                  acc[4 * i] += v.x * w;
                  acc[4 * i + 1] += v.y * w;
                  acc[4 * i + 2] += v.z * w;
                  acc[4 * i + 3] += v.w * w;
                }
              }
              const float inv = 1.f / den;  // > 0: every node sees itself
              float4 *dst = reinterpret_cast<float4 *>(a.O + (((long long)sg.b * N + r) * a.Hq + h) * kD + ch);
#pragma unroll
              for (int i = 0; i < 16; ++i)
                dst[i] = make_float4(acc[4 * i] * inv, acc[4 * i + 1] * inv, acc[4 * i + 2] * inv, acc[4 * i + 3] * inv);
            }
          }
          if (threadIdx.x == 128) a.cnt[sg.pair] = 0;
        }
      }
      gt += T;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

size_t smem_bytes() { return (size_t)Cfg::OFF_BAR + sizeof(Bars) + 1024; }

struct Plan {
  int G, GS, HPS, pairs, grid;  // grid: CTAs the workspace is laid out for (one per SM)
  size_t o_off, ml_off, cnt_off, total;
};

// CTAs to launch: one per SM, but never so many that a CTA gets fewer than
// kMinTiles tiles of the largest possible work (cap keys per sequence): a
// small batch would otherwise cut every pair into many parts, each paying the
// start-up and the partial merge.  Always whole groups.
constexpr long long kMinTiles = 16;
int launch_grid(const Plan &p, int B, int Hkv, int cap, int N) {
  const long long most = (long long)B * Hkv * p.G * ((cap + BN - 1) / BN + (N + BN - 1) / BN);
  const long long want = (most + kMinTiles - 1) / kMinTiles;
  const long long g = std::max<long long>(1, std::min<long long>(p.grid, want) / p.GS);
  return (int)(g * p.GS);
}

Plan make_plan(int B, int Hq, int Hkv, int N) {
  Plan p;
  p.G = Hq / Hkv;
  // one query head per pair, also for grouped-query heads: two heads per
  // K/V tile halve the K/V reads but measured slower on the grouped-query
  // shapes tried (32 query / 8 KV heads, prefixes 4096 and 32768), which are
  // bound by the tensor pipe and the exponentials, not HBM
  p.pairs = B * Hkv * p.G;
  p.grid = tr_sm_count();
  // one CTA per query head of a KV head in each CTA group, when that fits
  // the grid; else those heads are laid end to end in the tile order
  p.GS = p.G <= p.grid ? p.G : 1;
  p.HPS = p.G / p.GS;
  const size_t rows = (size_t)p.grid * 2 * N;
  p.o_off = 0;
  p.ml_off = tr_align_up(rows * kD * sizeof(float), 256);
  p.cnt_off = p.ml_off + tr_align_up(rows * sizeof(float2), 256);
  p.total = p.cnt_off + tr_align_up((size_t)p.pairs * sizeof(int), 256);
  return p;
}

}  // namespace

extern "C" size_t tr_verify_attn_workspace_bytes(int B, int Hq, int Hkv, int d, int cap, const struct tr_tree *tree) {
  if (!tree || B < 1 || Hq < 1 || Hkv < 1 || Hq % Hkv || d != kD || cap < 0) return 0;
  return make_plan(B, Hq, Hkv, tree->dev.N).total;
}

extern "C" int tr_verify_attn(const void *Q, const void *Kt, const void *Vt, const void *Kc, const void *Vc,
                              const int32_t *L, int cap, int B, int Hq, int Hkv, int d, float scale,
                              const struct tr_tree *tree, float *O, void *ws, size_t ws_bytes, tr_stream_t stream) {
  if (!Q || !Kt || !Vt || !Kc || !Vc || !L || !tree || !O || B < 1 || Hq < 1 || Hkv < 1 || cap < 0) return TR_E_INVAL;
  if (Hq % Hkv || !(scale > 0.f) || !(scale < INFINITY)) return TR_E_INVAL;
  if (d != kD) return TR_E_UNSUPPORTED;
  const int N = tree->dev.N;
  // the global tile count must fit in 31 bits
  const long long max_tiles = (long long)B * Hkv * Hq * ((cap + BN - 1) / BN + (N + BN - 1) / BN);
  if (B > kMaxB || max_tiles >= (1LL << 31) || (long long)B * Hkv * cap >= (1LL << 31)) return TR_E_UNSUPPORTED;
  const Plan p = make_plan(B, Hq, Hkv, N);
  if (!ws || ws_bytes < p.total) return TR_E_INVAL;
  if (((uintptr_t)Q | (uintptr_t)Kt | (uintptr_t)Vt | (uintptr_t)Kc | (uintptr_t)Vc | (uintptr_t)O) & 15)
    return TR_E_INVAL;
  int rc = tr_check_device();
  if (rc != TR_OK) return rc;

  const uint32_t q_rows = (uint32_t)std::min<long long>(128, (long long)B * N);
  const uint32_t c_rows = (uint32_t)std::min<long long>(BN, (long long)B * Hkv * (cap > 0 ? cap : 1));
  const uint32_t t_rows = (uint32_t)std::min<long long>(BN, (long long)B * N);
  CUtensorMap tq, tkc, tvc, tkt, tvt;
  {
    const uint64_t dq[3] = {(uint64_t)kD, (uint64_t)Hq, (uint64_t)B * N};
    const uint64_t sq[2] = {(uint64_t)kD * 2, (uint64_t)Hq * kD * 2};
    const uint32_t bq[3] = {64, 1, q_rows};
    if ((rc = tr_make_tmap_bf16(&tq, Q, 3, dq, sq, bq)) != TR_OK) return rc;
    const uint64_t dc[2] = {(uint64_t)kD, (uint64_t)B * Hkv * (cap > 0 ? cap : 1)};
    const uint64_t sc[1] = {(uint64_t)kD * 2};
    const uint32_t bc[2] = {64, c_rows};
    if ((rc = tr_make_tmap_bf16(&tkc, Kc, 2, dc, sc, bc)) != TR_OK) return rc;
    if ((rc = tr_make_tmap_bf16(&tvc, Vc, 2, dc, sc, bc)) != TR_OK) return rc;
    const uint64_t dt[3] = {(uint64_t)kD, (uint64_t)Hkv, (uint64_t)B * N};
    const uint64_t st[2] = {(uint64_t)kD * 2, (uint64_t)Hkv * kD * 2};
    const uint32_t bt[3] = {64, 1, t_rows};
    if ((rc = tr_make_tmap_bf16(&tkt, Kt, 3, dt, st, bt)) != TR_OK) return rc;
    if ((rc = tr_make_tmap_bf16(&tvt, Vt, 3, dt, st, bt)) != TR_OK) return rc;
  }
  AttnArgs a;
  a.L = L;
  a.O = O;
  a.part_o = (float *)((char *)ws + p.o_off);
  a.part_ml = (float2 *)((char *)ws + p.ml_off);
  a.cnt = (int *)((char *)ws + p.cnt_off);
  a.status = tr_status_dev();
  a.B = B;
  a.N = N;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.G = p.G;
  a.GS = p.GS;
  a.HPS = p.HPS;
  a.cap = cap;
  a.q_rows = (int)q_rows;
  a.c_rows = (int)c_rows;
  a.t_rows = (int)t_rows;
  a.scale_log2 = scale * 1.4426950408889634f;
  a.wait_ns = tr_wait_limit_ns();
  cudaStream_t s = (cudaStream_t)stream;
  const int grid = launch_grid(p, B, Hkv, cap, N);
  static bool attr_set[64];
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && !attr_set[dev]) {
    TR_TRY_CUDA(cudaFuncSetAttribute(attn_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_bytes()));
    attr_set[dev] = true;
  }
  attn_tc_kernel<<<grid, Cfg::THREADS, smem_bytes(), s>>>(tq, tkc, tvc, tkt, tvt, a, tree->dev);
  TR_LAUNCH_CHECK();
  return TR_OK;
}
