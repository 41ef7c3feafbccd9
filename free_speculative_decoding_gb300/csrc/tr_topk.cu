// Per-row top-K over vocabulary logits (fp32 or bf16), ties to the lower ID.
//
// Keys are 64-bit: an order-preserving value code in the high word and the
// complemented ID in the low word, so a larger key is better and equal values
// prefer the lower ID.
//
// Rows whose start and stride are 16-byte aligned take the warp-streaming
// kernel.  Every row is cut into 8 KB steps; all rows' steps, in order, are
// cut into equal contiguous ranges, one per warp of a persistent grid (one
// CTA of 8 warps per SM).  Each warp pulls its steps through a private ring
// of three bulk copies (cp.async.bulk into shared memory, completing on an
// mbarrier) and examines each step where it landed: vector maxima are read
// from the stage, an element handed over is cleared there, and the stage is
// refilled once the step is done.  The warp keeps the current row's running
// top-K across its lanes (lane j holds the j-th best key).
// Only elements above a floor can enter: the K-th best value held, or on a
// segment's first step the K-th largest lane maximum.  A step with no lane
// maximum above the floor costs a vector maximum and one vote; otherwise each
// lane hands over its largest remaining element per pass and the warp inserts
// those keys by ballot and shuffle.  A row split between warps leaves one
// list per warp segment in the workspace; the warp that completes the row's
// step count merges them.
//
// Other rows take a plain scan: a row is cut into chunks of one 256-thread
// CTA each, every thread keeps a register list, and the chunks of a row merge
// inside a thread-block cluster (or, beyond 8 chunks, in the last CTA to
// finish).
#include "tr_internal.cuh"
#include "tr_lists.cuh"
#include "tr_sm100.cuh"

namespace {

constexpr unsigned kFull = 0xffffffffu;

template <typename T>
struct Elem;
template <>
struct Elem<float> {
  static constexpr int kVec = 4;
  __device__ __forceinline__ static float load1(const float *p) { return __ldcs(p); }
  __device__ __forceinline__ static uint4 nan_vec() { return make_uint4(0x7FC00000u, 0x7FC00000u, 0x7FC00000u, 0x7FC00000u); }
  __device__ __forceinline__ static void unpack(const uint4 &q, float (&e)[4]) {
    e[0] = __uint_as_float(q.x);
    e[1] = __uint_as_float(q.y);
    e[2] = __uint_as_float(q.z);
    e[3] = __uint_as_float(q.w);
  }
  // the vector with component k set to NaN
  __device__ __forceinline__ static uint4 clear(uint4 q, int k) {
    q.x = k == 0 ? 0x7FC00000u : q.x;
    q.y = k == 1 ? 0x7FC00000u : q.y;
    q.z = k == 2 ? 0x7FC00000u : q.z;
    q.w = k == 3 ? 0x7FC00000u : q.w;
    return q;
  }
  // maximum of the vector, NaN only if all four are NaN
  __device__ __forceinline__ static float vmax(const uint4 &q) {
    return fmaxf(fmaxf(__uint_as_float(q.x), __uint_as_float(q.y)), fmaxf(__uint_as_float(q.z), __uint_as_float(q.w)));
  }
};
template <>
struct Elem<__nv_bfloat16> {
  static constexpr int kVec = 8;
  __device__ __forceinline__ static uint4 nan_vec() { return make_uint4(0x7FC07FC0u, 0x7FC07FC0u, 0x7FC07FC0u, 0x7FC07FC0u); }
  __device__ __forceinline__ static void unpack(const uint4 &q, float (&e)[8]) {
    e[0] = __uint_as_float(q.x << 16);
    e[1] = __uint_as_float(q.x & 0xFFFF0000u);
    e[2] = __uint_as_float(q.y << 16);
    e[3] = __uint_as_float(q.y & 0xFFFF0000u);
    e[4] = __uint_as_float(q.z << 16);
    e[5] = __uint_as_float(q.z & 0xFFFF0000u);
    e[6] = __uint_as_float(q.w << 16);
    e[7] = __uint_as_float(q.w & 0xFFFF0000u);
  }
  // the vector with element k set to NaN (even k: low half of word k/2)
  __device__ __forceinline__ static uint4 clear(uint4 q, int k) {
    const uint32_t nan = (k & 1) ? 0x7FC00000u : 0x00007FC0u, keep = (k & 1) ? 0x0000FFFFu : 0xFFFF0000u;
    const int w = k >> 1;
    q.x = w == 0 ? (q.x & keep) | nan : q.x;
    q.y = w == 1 ? (q.y & keep) | nan : q.y;
    q.z = w == 2 ? (q.z & keep) | nan : q.z;
    q.w = w == 3 ? (q.w & keep) | nan : q.w;
    return q;
  }
  __device__ __forceinline__ static float vmax(const uint4 &q) {
    // packed maxima first (exact: a maximum needs no rounding; NaN is dropped
    // unless both inputs are NaN)
    const __nv_bfloat162 a = __hmax2(*reinterpret_cast<const __nv_bfloat162 *>(&q.x),
                                     *reinterpret_cast<const __nv_bfloat162 *>(&q.y));
    const __nv_bfloat162 b = __hmax2(*reinterpret_cast<const __nv_bfloat162 *>(&q.z),
                                     *reinterpret_cast<const __nv_bfloat162 *>(&q.w));
    const __nv_bfloat162 c = __hmax2(a, b);
    const uint32_t u = *reinterpret_cast<const uint32_t *>(&c);
    return fmaxf(__uint_as_float(u << 16), __uint_as_float(u & 0xFFFF0000u));
  }
  __device__ __forceinline__ static float load1(const __nv_bfloat16 *p) {
    const unsigned short u = __ldcs((const unsigned short *)p);
    return __uint_as_float((uint32_t)u << 16);
  }
};

// ---------------------------------------------------------------------------
// warp-streaming kernel (aligned rows)
// ---------------------------------------------------------------------------

constexpr int kVecs = 16;                // 16-byte vectors a lane loads per step
constexpr int kStep = 32 * kVecs * 16;   // bytes of a row one warp step covers (8 KB)
constexpr int kWarps = 8;                // warps per CTA (one CTA per SM)
constexpr int kStages = 3;               // steps a warp has in flight or in hand

struct alignas(128) WarpRing {
  unsigned char stage[kStages][kStep];
  uint64_t full[kStages];
};
constexpr size_t kRingSmem = sizeof(WarpRing) * kWarps + 128;  // +128: alignment of the base

// steps per row for elements of esz bytes
inline long long steps_per_row(long long V, size_t esz) { return (V * (long long)esz + kStep - 1) / kStep; }

// The contiguous step range [u0, u1) of warp w out of W over U steps, and the
// warp whose range holds step u.
__device__ __forceinline__ long long range_start(long long w, long long U, long long W) { return w * U / W; }
__device__ __forceinline__ long long warp_of(long long u, long long U, long long W) { return ((u + 1) * W - 1) / U; }

// K-th largest of the lanes' values (counting repeats), the same on every
// lane: a bitonic sort of the 32 values into descending lane order.
__device__ __forceinline__ float warp_kth(float v, int K, int lane) {
#pragma unroll
  for (int k = 2; k <= 32; k <<= 1) {
#pragma unroll
    for (int j = k >> 1; j > 0; j >>= 1) {
      const float o = __shfl_xor_sync(kFull, v, j);
      // blocks of k lanes alternate direction; the lower lane of a pair keeps
      // the larger value in a descending block
      const bool keep_max = ((lane & j) == 0) != ((lane & k) != 0);
      v = keep_max ? fmaxf(v, o) : fminf(v, o);
    }
  }
  return __shfl_sync(kFull, v, K - 1);
}

__device__ __forceinline__ void write_final(int32_t *ids, float *vals, long long row, int K, int lane,
                                            unsigned long long key) {
  if (lane < K) {
    ids[row * K + lane] = key ? (int32_t)tr_key_id(key) : -1;
    if (vals) vals[row * K + lane] = key ? tr_key_val(key) : -INFINITY;
  }
}

// (max, Z) of a row from the lanes' running pairs: Z = sum of 2^((x - max) c).
__device__ __forceinline__ float2 warp_stats(float m, float z, float c) {
  float M = m;
#pragma unroll
  for (int off = 16; off; off >>= 1) M = fmaxf(M, __shfl_xor_sync(kFull, M, off));
  float S = m == -INFINITY ? 0.f : z * sm100::ex2((m - M) * c);
#pragma unroll
  for (int off = 16; off; off >>= 1) S += __shfl_xor_sync(kFull, S, off);
  return make_float2(M, S);
}

// STATS: also the row's softmax statistics at temperature T, c = log2(e) / T:
// stats[row] = (max, sum of exp((x - max) / T)), and the same pair for every
// 8 KB step of the row, sstats[row * nch + step] = (step max, sum of
// exp((x - step max) / T) over the step), from which a sampled token can be
// located one step at a time.  Per step the warp takes the step's maximum,
// each lane sums its elements' exp2 against it, and a warp sum gives the
// step's pair; the lanes' running sums share one warp-wide running maximum
// (rescaled when it grows), are summed at the end of a row segment and, for
// a row split between warps, combined over the segments by the merging warp
// (pstats holds one pair per list slot).
template <typename T, int KMAX, bool STATS>
__global__ void __launch_bounds__(kWarps * 32, 1)
    topk_warp_kernel(const T *__restrict__ x, long long V, long long ld, int K, int nch, long long U, int32_t *ids,
                     float *vals, unsigned long long *part, unsigned *counters, unsigned *status,
                     unsigned long long wait_ns, float c, float2 *stats, float2 *pstats, float2 *sstats) {
  using namespace sm100;
  extern __shared__ unsigned char smem_raw[];
  const int lane = threadIdx.x & 31;
  WarpRing &ring = reinterpret_cast<WarpRing *>((reinterpret_cast<uintptr_t>(smem_raw) + 127) &
                                                ~uintptr_t(127))[threadIdx.x >> 5];
  const long long W = (long long)gridDim.x * kWarps;
  const long long gw = (long long)blockIdx.x * kWarps + (threadIdx.x >> 5);
  const long long u0 = range_start(gw, U, W), u1 = range_start(gw + 1, U, W);
  if (u0 >= u1) return;  // warps work alone: no block-wide barrier follows

  constexpr int kV = Elem<T>::kVec;
  const long long row_bytes = V * (long long)sizeof(T);
  const int n_steps = (int)(u1 - u0);

  // lane j < K: the j-th best key of the row segment so far
  unsigned long long lk = 0ull;
  bool have_k = false;  // K keys held: thr is the value of the K-th
  float thr = 0.f;
  long long cur = -1;   // row of the segment
  int seg_first = 0, seg_units = 0;
  float st_m = -INFINITY, st_z = 0.f;  // STATS: this lane's running maximum and sum

  // end of a row segment: the final list, or this segment's list for a merge
  auto flush = [&](long long row) {
    float2 rs = make_float2(0.f, 0.f);
    if (STATS) rs = warp_stats(st_m, st_z, c);
    if (seg_first == 0 && seg_units == nch) {
      write_final(ids, vals, row, K, lane, lk);
      if (STATS && lane == 0) stats[row] = rs;
      return;
    }
    if (lane < K) part[((unsigned long long)row * nch + seg_first) * KMAX + lane] = lk;
    if (STATS && lane == 0) pstats[(unsigned long long)row * nch + seg_first] = rs;
    __threadfence();
    __syncwarp();
    unsigned last = 0;
    if (lane == 0) last = atomicAdd(&counters[row], (unsigned)seg_units) + (unsigned)seg_units == (unsigned)nch;
    if (!__shfl_sync(kFull, last, 0)) return;
    __threadfence();
    // every warp segment of the row left its list at the slot of its first step
    TopList<KMAX> L;
    L.init();
    const long long r0 = row * nch;
    const long long wlo = warp_of(r0, U, W), whi = warp_of(r0 + nch - 1, U, W);
    float pm = -INFINITY, pz = 0.f;  // STATS: the segments' pairs this lane folds
    for (long long p = wlo + lane; p <= whi; p += 32) {
      const long long sp = range_start(p, U, W);
      if (sp >= range_start(p + 1, U, W)) continue;  // a warp without steps
      const long long first = (sp > r0 ? sp : r0) - r0;
      const unsigned long long *src = part + ((unsigned long long)row * nch + first) * KMAX;
      for (int j = 0; j < K; ++j) list_insert(L.k, __ldcg(src + j));
      if (STATS) {
        const float2 q = __ldcg(pstats + (unsigned long long)row * nch + first);
        const float nm = fmaxf(pm, q.x);
        pz = (pm == -INFINITY ? 0.f : pz * sm100::ex2((pm - nm) * c)) +
             (q.x == -INFINITY ? 0.f : q.y * sm100::ex2((q.x - nm) * c));
        pm = nm;
      }
    }
    const unsigned long long m = warp_merge<KMAX>(L, lane);
    write_final(ids, vals, row, K, lane, m);
    if (STATS) {
      const float2 q = warp_stats(pm, pz, c);
      if (lane == 0) stats[row] = q;
    }
    if (lane == 0) counters[row] = 0u;  // the workspace is left zeroed
  };

  // A ring of kStages bulk copies (cp.async.bulk into this warp's shared
  // memory) runs ahead of the step being examined.  Lane 0 issues the copy of
  // the next step (row ir, step ic of the row): its whole 16-byte vectors;
  // the row's ragged last bytes are read directly.
  const char *base = reinterpret_cast<const char *>(x);
  const long long stride = ld * (long long)sizeof(T);
  long long ir = u0 / nch;
  int ic = (int)(u0 - ir * nch), n_issued = 0;
  if (lane == 0) {
    for (int q = 0; q < kStages; ++q) mbar_init(&ring.full[q], 1);
    fence_mbar_init();
  }
  // the logits are read once: their lines go first, so the matrices the step
  // end gathers from stay in L2
  const uint64_t stream_policy = l2_evict_first();
  __syncwarp();
  auto issue = [&](int q) {
    const long long off = (long long)ic * kStep;
    const uint32_t bytes = (uint32_t)(min(row_bytes - off, (long long)kStep) & ~15ll);
    mbar_arrive_expect_tx(&ring.full[q], bytes);
    if (bytes) bulk_load_hint(ring.stage[q], base + ir * stride + off, bytes, &ring.full[q], stream_policy);
    if (++ic == nch) {
      ic = 0;
      ++ir;
    }
    ++n_issued;
  };
  if (lane == 0)
    for (int q = 0; q < kStages && q < n_steps; ++q) issue(q);

  // after the step is examined (its stage read and partly cleared): the
  // stage takes the next step to fetch
  auto refill = [&](int q) {
    __syncwarp();
    if (lane == 0) {
      fence_proxy_async_smem();  // the stage's generic reads and writes come before the next copy into it
      if (n_issued < n_steps) issue(q);
    }
  };

  auto process = [&](int q, long long r, int cc) {
    if (r != cur) {
      if (cur >= 0) flush(cur);
      cur = r;
      lk = 0ull;
      have_k = false;
      seg_first = cc;
      seg_units = 0;
      st_m = -INFINITY;
      st_z = 0.f;
    }
    ++seg_units;
    const long long off = (long long)cc * kStep;
    const long long nb = min(row_bytes - off, (long long)kStep);
    const long long id0 = off / (long long)sizeof(T);                      // first element of the step
    const long long et = id0 + (nb >> 4) * kV;                              // first element past the vectors
    const int ntail = (int)((nb & 15) / (long long)sizeof(T));
    float tv = lane < ntail ? Elem<T>::load1(x + r * ld + et + lane) : NAN;  // the row's ragged end

    // The step stays in the warp's stage until the refill: vector maxima come
    // straight from it, and an element handed over is cleared there (NaN).
    uint4 *sv = reinterpret_cast<uint4 *>(ring.stage[q]);
    const int nvec = (int)(nb >> 4);
    float vmx[kVecs];  // each vector's maximum (NaN when none of it can enter)
    if (nvec == 32 * kVecs) {
#pragma unroll
      for (int j = 0; j < kVecs; ++j) vmx[j] = Elem<T>::vmax(sv[j * 32 + lane]);
    } else {
#pragma unroll
      for (int j = 0; j < kVecs; ++j) vmx[j] = j * 32 + lane < nvec ? Elem<T>::vmax(sv[j * 32 + lane]) : NAN;
    }
    // NaN when the lane holds no element of the step (a short last step of a
    // row, or everything handed over), so that such a lane never takes part
    auto lane_max = [&]() {
      float m = tv;
#pragma unroll
      for (int j = 0; j < kVecs; ++j) m = fmaxf(m, vmx[j]);
      return m;
    };
    float lm = lane_max();
    if (STATS) {
      // every element of the step enters the sums, before the top-K passes
      // below clear any of them from the stage
      float sm = isnan(lm) ? -INFINITY : lm;  // the step's maximum (some lane holds an element)
#pragma unroll
      for (int off = 16; off; off >>= 1) sm = fmaxf(sm, __shfl_xor_sync(kFull, sm, off));
      const float smc = sm * c;
      float z4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int j = 0; j < kVecs; ++j) {
        if (j * 32 + lane < nvec) {
          float e[kV];
          Elem<T>::unpack(sv[j * 32 + lane], e);
#pragma unroll
          for (int qq = 0; qq < kV; ++qq) z4[qq & 3] += sm100::ex2(fmaf(e[qq], c, -smc));
        }
      }
      if (!isnan(tv)) z4[1] += sm100::ex2(fmaf(tv, c, -smc));
      const float zl = (z4[0] + z4[1]) + (z4[2] + z4[3]);
      float zs = zl;
#pragma unroll
      for (int off = 16; off; off >>= 1) zs += __shfl_xor_sync(kFull, zs, off);
      if (lane == 0) sstats[r * nch + cc] = make_float2(sm, zs);
      const float nm = fmaxf(st_m, sm);  // warp-wide, so every rescale factor is at most 1
      st_z = (st_m == -INFINITY ? 0.f : st_z * sm100::ex2((st_m - nm) * c)) + zl * sm100::ex2((sm - nm) * c);
      st_m = nm;
    }
    // An element enters only above the floor f: the K-th best value held,
    // when there is one (the held keys all come from earlier steps, with
    // lower IDs, so only a strictly larger value can enter); else the K-th
    // largest lane maximum, which K elements of this step reach (-inf when
    // fewer than K lanes hold an element).
    float f = have_k ? thr : warp_kth(isnan(lm) ? -INFINITY : lm, K, lane);
    bool strict = have_k;
    // Each pass takes every lane's largest remaining element above the floor
    // (the lowest ID among equal values), inserts those keys into the held
    // list, and clears them from the registers.
    while (__any_sync(kFull, strict ? lm > f : lm >= f)) {
      unsigned long long key = 0ull;
      if (strict ? lm > f : lm >= f) {
        // the lowest vector holding the lane maximum (the tail comes last)
        int jv = kVecs;
#pragma unroll
        for (int j = kVecs - 1; j >= 0; --j) jv = vmx[j] == lm ? j : jv;
        if (jv < kVecs) {
          uint4 w = sv[jv * 32 + lane];
          float e[kV];
          Elem<T>::unpack(w, e);
          int q0 = kV;
#pragma unroll
          for (int qq = kV - 1; qq >= 0; --qq) q0 = e[qq] == lm ? qq : q0;
          key = tr_key(tr_ord(lm), (uint32_t)(id0 + ((long long)jv * 32 + lane) * kV + q0));
          w = Elem<T>::clear(w, q0);
          sv[jv * 32 + lane] = w;
          const float wm = Elem<T>::vmax(w);
#pragma unroll
          for (int j = 0; j < kVecs; ++j) vmx[j] = j == jv ? wm : vmx[j];
        } else {
          key = tr_key(tr_ord(tv), (uint32_t)(et + lane));
          tv = NAN;
        }
      }
      // keys that cannot beat the K-th held key stay out
      const unsigned long long kth0 = __shfl_sync(kFull, lk, K - 1);
      if (key <= kth0) key = 0ull;
      unsigned mask = __ballot_sync(kFull, key != 0ull);
      while (mask) {
        const int src = __ffs(mask) - 1;
        mask &= mask - 1;
        const unsigned long long k = __shfl_sync(kFull, key, src);
        // its place is the number of larger held keys; the keys below it move
        // up one lane and the K-th falls off
        const int pos = __popc(__ballot_sync(kFull, lk > k));
        if (pos < K) {
          const unsigned long long up = __shfl_up_sync(kFull, lk, 1);
          if (lane == pos) lk = k;
          else if (lane > pos && lane < K) lk = up;
        }
      }
      const unsigned long long kth = __shfl_sync(kFull, lk, K - 1);
      if (kth) {
        have_k = true;
        thr = tr_key_val(kth);
        // keys of this step may tie the new K-th value with a lower ID
        f = thr;
        strict = false;
      }
      lm = lane_max();
    }
  };

  long long r = u0 / nch;
  int cs = (int)(u0 - r * nch);
  int q = 0;
  uint32_t ph = 0;
  int i = 0;
  for (; i < n_steps; ++i) {
    if (!__all_sync(kFull, mbar_wait_for(&ring.full[q], ph, wait_ns))) break;
    process(q, r, cs);
    refill(q);
    if (++cs == nch) {
      cs = 0;
      ++r;
    }
    if (++q == kStages) {
      q = 0;
      ph ^= 1u;
    }
  }
  if (i < n_steps) {
    // a copy that never landed: flag it and wait (bounded) for this warp's
    // other copies before the CTA's shared memory goes away
    if (lane == 0) tr_flag(status, TR_DEV_TIMEOUT);
    for (int j = i; j < i + kStages && j < n_steps; ++j)
      mbar_drain(&ring.full[j % kStages], (uint32_t)((j / kStages) & 1));
    return;
  }
  flush(cur);
}

// ---------------------------------------------------------------------------
// plain scan (rows that are not 16-byte aligned)
// ---------------------------------------------------------------------------

constexpr int kThreads = 256;
constexpr long long kScanChunk = 16384;  // elements of a row per CTA
constexpr int kMaxCluster = 8;           // portable thread-block cluster size
constexpr int kMaxSplits = 32;

// The K largest of n distinct keys in shared memory, sorted, into out[0..K)
// (0 where fewer than K): each key's rank is the number of larger keys.
__device__ __forceinline__ void rank_select(const unsigned long long *keys, int n, int K, unsigned long long *out) {
  for (int k = threadIdx.x; k < K; k += blockDim.x) out[k] = 0ull;
  __syncthreads();
  for (int k = threadIdx.x; k < n; k += blockDim.x) {
    const unsigned long long key = keys[k];
    int rank = 0;
#pragma unroll 8
    for (int j = 0; j < n; ++j) rank += keys[j] > key;
    if (rank < K && key) out[rank] = key;
  }
  __syncthreads();
}

__device__ __forceinline__ void st_cluster_u64(void *local_addr, unsigned rank, unsigned long long v) {
  const unsigned a = (unsigned)__cvta_generic_to_shared(local_addr);
  unsigned remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(a), "r"(rank));
  asm volatile("st.shared::cluster.u64 [%0], %1;" ::"r"(remote), "l"(v) : "memory");
}

// CLUSTER: the row's chunks form one thread-block cluster and merge through
// the first CTA's shared memory; otherwise through the workspace, the row's
// last CTA to finish merging (an arrival counter, no spin-wait).
template <typename T, int KMAX, bool CLUSTER>
__global__ void __launch_bounds__(kThreads) topk_scan_kernel(const T *logits, long long V, long long ld, int K,
                                                             long long chunk, int32_t *ids, float *vals,
                                                             unsigned long long *part, unsigned *counters) {
  __shared__ unsigned long long keys[kMaxSplits * TR_MAX_K];
  __shared__ unsigned long long top[TR_MAX_K];
  __shared__ unsigned long long warp_keys[kThreads / 32][KMAX];
  __shared__ int is_last;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int split = blockIdx.x, splits = gridDim.x;
  const long long row = blockIdx.y;
  const T *x = logits + row * ld;
  const long long lo = split * chunk;
  const long long hi = min(V, lo + chunk);

  TopList<KMAX> L;
  L.init();
  for (long long i = lo + tid; i < hi; i += kThreads) L.push(Elem<T>::load1(x + i), (uint32_t)i);
  unsigned long long mine = warp_merge<KMAX>(L, lane);
  if (lane < KMAX) warp_keys[warp][lane] = mine;
  __syncthreads();
  if (warp == 0) {
    L.init();
    if (lane < kThreads / 32)
#pragma unroll
      for (int j = 0; j < KMAX; ++j) L.k[j] = warp_keys[lane][j];
    mine = warp_merge<KMAX>(L, lane);
    if (lane < K) top[lane] = mine;
  }
  __syncthreads();

  if (CLUSTER) {
    // every chunk's list into the first CTA's shared memory, then one ranking there
    const unsigned cr = sm100::cluster_ctarank();
    if (tid < K) st_cluster_u64(&keys[cr * K + tid], 0, top[tid]);
    sm100::cluster_sync_all();
    if (cr != 0) return;
    rank_select(keys, splits * K, K, top);
  } else if (splits > 1) {
    // publish this chunk's top K; the row's last CTA to arrive ranks all chunks' keys
    if (tid < K) part[(row * splits + split) * KMAX + tid] = top[tid];
    __threadfence();
    __syncthreads();
    if (tid == 0) is_last = atomicAdd(&counters[row], 1u) == (unsigned)(splits - 1);
    __syncthreads();
    if (!is_last) return;
    __threadfence();
    const int n = splits * K;
    for (int k = tid; k < n; k += kThreads) keys[k] = __ldcg(part + (row * splits + k / K) * KMAX + k % K);
    rank_select(keys, n, K, top);
    if (tid == 0) counters[row] = 0u;
  }
  if (tid < K) {
    const unsigned long long key = top[tid];
    ids[row * K + tid] = key ? (int32_t)tr_key_id(key) : -1;
    if (vals) vals[row * K + tid] = key ? tr_key_val(key) : -INFINITY;
  }
}

// ---------------------------------------------------------------------------
// launch
// ---------------------------------------------------------------------------

// Workspace: per-(row, step) list slots of KMAX keys (fp32 step count: the
// most steps, so bf16 rows fit as well), then one arrival counter per row.
size_t part_bytes_for(long long rows, long long V, int K) {
  return tr_align_up((size_t)rows * (size_t)steps_per_row(V, 4) * tr_kmax(K) * 8, 256);
}

template <typename T, int KMAX, bool STATS>
cudaError_t launch_warp(const void *logits, long long rows, long long V, long long ld, int K, int32_t *ids,
                        float *vals, unsigned long long *part, unsigned *counters, float c, float2 *stats,
                        float2 *pstats, float2 *sstats, cudaStream_t s) {
  const int nch = (int)steps_per_row(V, sizeof(T));
  const long long U = rows * nch;
  const long long want = (U + kWarps - 1) / kWarps;
  const long long most = tr_sm_count();  // one CTA per SM, persistent
  const int grid = (int)(want < most ? want : most);
  static bool attr_set[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!attr_set[dev]) {
    const cudaError_t e = cudaFuncSetAttribute(topk_warp_kernel<T, KMAX, STATS>,
                                               cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kRingSmem);
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  topk_warp_kernel<T, KMAX, STATS><<<grid, kWarps * 32, kRingSmem, s>>>(
      (const T *)logits, V, ld, K, nch, U, ids, vals, part, counters, tr_status_dev(), tr_wait_limit_ns(), c, stats,
      pstats, sstats);
  return cudaGetLastError();
}

template <typename T, int KMAX>
cudaError_t launch_scan(const void *logits, long long rows, long long V, long long ld, int K, int32_t *ids,
                        float *vals, unsigned long long *part, unsigned *counters, cudaStream_t s) {
  long long splits = (V + kScanChunk - 1) / kScanChunk;
  if (splits > kMaxSplits) splits = kMaxSplits;
  const long long chunk = (V + splits - 1) / splits;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)splits, (unsigned)rows);
  cfg.blockDim = dim3(kThreads);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  const bool cluster = splits > 1 && splits <= kMaxCluster;
  if (cluster) {
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)splits;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, topk_scan_kernel<T, KMAX, true>, (const T *)logits, V, ld, K, chunk, ids, vals,
                              part, counters);
  }
  return cudaLaunchKernelEx(&cfg, topk_scan_kernel<T, KMAX, false>, (const T *)logits, V, ld, K, chunk, ids, vals,
                            part, counters);
}

// Workspace layout: [list slots | row counters | STATS: one (max, sum) pair per list slot].
size_t counters_bytes_for(long long rows) { return tr_align_up((size_t)rows * 4, 256); }
size_t pstats_bytes_for(long long rows, long long V) { return tr_align_up((size_t)rows * steps_per_row(V, 4) * 8, 256); }

template <typename T, int KMAX>
cudaError_t launch(const void *logits, long long rows, long long V, long long ld, int K, int32_t *ids, float *vals,
                   void *ws, float c, float2 *stats, float2 *sstats, cudaStream_t s) {
  unsigned long long *part = (unsigned long long *)ws;
  unsigned *counters = (unsigned *)((char *)ws + (ws ? part_bytes_for(rows, V, K) : 0));
  float2 *pstats = (float2 *)((char *)ws + (ws ? part_bytes_for(rows, V, K) + counters_bytes_for(rows) : 0));
  const bool aligned = ((uintptr_t)logits % 16 == 0) && ((ld * (long long)sizeof(T)) % 16 == 0);
  if (stats)
    return launch_warp<T, KMAX, true>(logits, rows, V, ld, K, ids, vals, part, counters, c, stats, pstats, sstats, s);
  if (aligned)
    return launch_warp<T, KMAX, false>(logits, rows, V, ld, K, ids, vals, part, counters, 0.f, nullptr, nullptr,
                                       nullptr, s);
  return launch_scan<T, KMAX>(logits, rows, V, ld, K, ids, vals, part, counters, s);
}

}  // namespace

extern "C" size_t tr_topk_workspace_bytes(int64_t rows, int64_t V, int K) {
  if (rows <= 0 || V <= 0 || K < 1 || K > TR_MAX_K) return 0;
  if (steps_per_row(V, 4) == 1) return 0;  // no row is ever split
  return part_bytes_for(rows, V, K) + counters_bytes_for(rows) + pstats_bytes_for(rows, V);
}

size_t tr_topk_counters_offset(int64_t rows, int64_t V, int K) { return part_bytes_for(rows, V, K); }

int tr_topk_launch(const void *logits, tr_ftype ftype, int64_t rows, int64_t V, int64_t ld, int K, int32_t *ids,
                   float *vals, void *ws, size_t ws_bytes, cudaStream_t s, float temperature, float *stats,
                   float *step_stats) {
  (void)ws_bytes;
  const int km = tr_kmax(K);
  const float c = stats ? 1.4426950408889634f / temperature : 0.f;
#define TR_TOPK_CASE(T, KM) \
  launch<T, KM>(logits, rows, V, ld, K, ids, vals, ws, c, (float2 *)stats, (float2 *)step_stats, s)
  cudaError_t e;
  if (ftype == TR_F32)
    e = km == 8 ? TR_TOPK_CASE(float, 8) : km == 16 ? TR_TOPK_CASE(float, 16) : TR_TOPK_CASE(float, 32);
  else
    e = km == 8 ? TR_TOPK_CASE(__nv_bfloat16, 8) : km == 16 ? TR_TOPK_CASE(__nv_bfloat16, 16)
                : TR_TOPK_CASE(__nv_bfloat16, 32);
#undef TR_TOPK_CASE
  if (e != cudaSuccess) return TR_E_CUDA;
  TR_LAUNCH_CHECK();
  return TR_OK;
}

extern "C" int tr_topk(const void *logits, tr_ftype ftype, int64_t rows, int64_t V, int64_t ld, int K, int32_t *ids,
                       float *vals, void *ws, size_t ws_bytes, tr_stream_t stream) {
  if (rows < 0 || V < 1 || K < 1 || K > TR_MAX_K || K > V || ld < V) return TR_E_INVAL;
  if (ftype != TR_F32 && ftype != TR_BF16) return TR_E_INVAL;
  if (V > INT32_MAX) return TR_E_UNSUPPORTED;
  if (rows == 0) return TR_OK;
  if (!logits || !ids) return TR_E_INVAL;
  const size_t need = tr_topk_workspace_bytes(rows, V, K);
  if (need && (!ws || ws_bytes < need)) return TR_E_INVAL;
  if (rows > 65535) return TR_E_UNSUPPORTED;  // grid.y limit of the plain scan
  int rc = tr_check_device();
  if (rc != TR_OK) return rc;
  return tr_topk_launch(logits, ftype, rows, V, ld, K, ids, vals, ws, ws_bytes, (cudaStream_t)stream);
}

extern "C" int tr_softmax_steps(int64_t V, tr_ftype ftype) {
  if (V < 1 || (ftype != TR_F32 && ftype != TR_BF16)) return 0;
  return (int)steps_per_row(V, ftype == TR_F32 ? 4 : 2);
}

extern "C" int tr_topk_softmax(const void *logits, tr_ftype ftype, int64_t rows, int64_t V, int64_t ld, int K,
                               float temperature, int32_t *ids, float *vals, float *stats, float *step_stats,
                               void *ws, size_t ws_bytes, tr_stream_t stream) {
  if (rows < 0 || V < 1 || K < 1 || K > TR_MAX_K || K > V || ld < V) return TR_E_INVAL;
  if (ftype != TR_F32 && ftype != TR_BF16) return TR_E_INVAL;
  if (!(temperature > 0.f) || !(temperature < INFINITY)) return TR_E_INVAL;
  if (V > INT32_MAX) return TR_E_UNSUPPORTED;
  if (rows == 0) return TR_OK;
  if (!logits || !ids || !stats || !step_stats) return TR_E_INVAL;
  const size_t esz = ftype == TR_F32 ? 4 : 2;
  if ((uintptr_t)logits % 16 || (ld * (int64_t)esz) % 16) return TR_E_UNSUPPORTED;  // streamed rows only
  const size_t need = tr_topk_workspace_bytes(rows, V, K);
  if (need && (!ws || ws_bytes < need)) return TR_E_INVAL;
  int rc = tr_check_device();
  if (rc != TR_OK) return rc;
  return tr_topk_launch(logits, ftype, rows, V, ld, K, ids, vals, ws, ws_bytes, (cudaStream_t)stream, temperature,
                        stats, step_stats);
}
