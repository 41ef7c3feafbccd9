// Per-row top-K over vocabulary logits (fp32 or bf16), ties to the lower ID.
//
// The kernel streams each row once from HBM with 16-byte loads.  A row is cut
// into `splits` chunks of about 8K elements so that the grid holds several
// waves of short CTAs on 152 SMs whatever the row count.  Each thread keeps a
// sorted register list of 64-bit keys (order-preserving value code in the
// high word, complemented ID in the low word, so larger key = better and equal
// values prefer the lower ID); a warp-wide floor computed from the lanes'
// maxima rejects all but about 1% of the elements with one compare.  Lists merge by warp shuffles, then across warps, then across
// the row's chunks in the last CTA to finish (an arrival counter in the
// workspace, no spin-wait).
#include "tr_internal.cuh"
#include "tr_lists.cuh"

namespace {

constexpr int kThreads = 256;
constexpr int kWindow = 16384;            // elements a CTA holds in registers (its whole chunk)
constexpr long long kChunk = kWindow;     // target elements per CTA
constexpr int kRankKeys = 1024;           // keys ranked directly (also all chunks' lists of a row)
constexpr int kMaxSplits = 32;

// K-th largest of the lanes' values (counting repeats), the same on every lane.
__device__ __forceinline__ float warp_kth(float v, int K, int lane) {
  float res = -INFINITY;
  for (int r = 0; r < K; ++r) {
    float m = v;
#pragma unroll
    for (int off = 16; off; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
    res = m;
    const unsigned who = __ballot_sync(0xffffffffu, v == m);
    if (lane == __ffs(who) - 1) v = -INFINITY;
  }
  return res;
}

template <typename T>
struct Elem;
template <>
struct Elem<float> {
  static constexpr int kVec = 4;
  template <int KMAX>
  __device__ __forceinline__ static void push_vec(TopList<KMAX> &L, const uint4 &q, uint32_t id) {
    L.push(__uint_as_float(q.x), id);
    L.push(__uint_as_float(q.y), id + 1);
    L.push(__uint_as_float(q.z), id + 2);
    L.push(__uint_as_float(q.w), id + 3);
  }
  __device__ __forceinline__ static float load1(const float *p) { return __ldcs(p); }
  __device__ __forceinline__ static float load_again(const float *p) { return __ldcg(p); }
  __device__ __forceinline__ static uint4 nan_vec() { return make_uint4(0x7FC00000u, 0x7FC00000u, 0x7FC00000u, 0x7FC00000u); }
  __device__ __forceinline__ static void unpack(const uint4 &q, float (&e)[4]) {
    e[0] = __uint_as_float(q.x);
    e[1] = __uint_as_float(q.y);
    e[2] = __uint_as_float(q.z);
    e[3] = __uint_as_float(q.w);
  }
  __device__ __forceinline__ static float vmax(const uint4 &q) {
    return fmaxf(fmaxf(__uint_as_float(q.x), __uint_as_float(q.y)), fmaxf(__uint_as_float(q.z), __uint_as_float(q.w)));
  }
};
template <>
struct Elem<__nv_bfloat16> {
  static constexpr int kVec = 8;
  template <int KMAX>
  __device__ __forceinline__ static void push_vec(TopList<KMAX> &L, const uint4 &q, uint32_t id) {
    L.push(__uint_as_float(q.x << 16), id);
    L.push(__uint_as_float(q.x & 0xFFFF0000u), id + 1);
    L.push(__uint_as_float(q.y << 16), id + 2);
    L.push(__uint_as_float(q.y & 0xFFFF0000u), id + 3);
    L.push(__uint_as_float(q.z << 16), id + 4);
    L.push(__uint_as_float(q.z & 0xFFFF0000u), id + 5);
    L.push(__uint_as_float(q.w << 16), id + 6);
    L.push(__uint_as_float(q.w & 0xFFFF0000u), id + 7);
  }
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
  __device__ __forceinline__ static float vmax(const uint4 &q) {
    const float a = fmaxf(fmaxf(__uint_as_float(q.x << 16), __uint_as_float(q.x & 0xFFFF0000u)),
                          fmaxf(__uint_as_float(q.y << 16), __uint_as_float(q.y & 0xFFFF0000u)));
    const float b = fmaxf(fmaxf(__uint_as_float(q.z << 16), __uint_as_float(q.z & 0xFFFF0000u)),
                          fmaxf(__uint_as_float(q.w << 16), __uint_as_float(q.w & 0xFFFF0000u)));
    return fmaxf(a, b);
  }
  __device__ __forceinline__ static float load_again(const __nv_bfloat16 *p) {
    return __uint_as_float((uint32_t)__ldcg((const unsigned short *)p) << 16);
  }
  __device__ __forceinline__ static float load1(const __nv_bfloat16 *p) {
    const unsigned short u = __ldcs((const unsigned short *)p);
    return __uint_as_float((uint32_t)u << 16);
  }
};

// The K largest of n distinct keys in shared memory, sorted, into out[0..K)
// (0 where fewer than K): each key's rank is the number of larger keys.
__device__ __forceinline__ void rank_select(const unsigned long long *keys, int n, int K, unsigned long long *out) {
  for (int k = threadIdx.x; k < K; k += blockDim.x) out[k] = 0ull;
  __syncthreads();
  for (int k = threadIdx.x; k < n; k += blockDim.x) {
    const unsigned long long key = keys[k];
    int rank = 0;
    for (int j = 0; j < n; ++j) rank += keys[j] > key;
    if (rank < K && key) out[rank] = key;
  }
  __syncthreads();
}

template <typename T, int KMAX, bool VEC>
__global__ void __launch_bounds__(kThreads) topk_kernel(const T *logits, long long V, long long ld, int K,
                                                        long long chunk, int32_t *ids, float *vals,
                                                        unsigned long long *part, unsigned *counters) {
  __shared__ unsigned short cand_o[kWindow];          // candidate offsets within the chunk
  __shared__ unsigned long long keys[kRankKeys];       // keys being ranked
  __shared__ unsigned long long top[TR_MAX_K];
  __shared__ unsigned long long warp_keys[kThreads / 32][KMAX];
  __shared__ float wfloor[kThreads / 32];
  __shared__ int count, is_last;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int split = blockIdx.x, splits = gridDim.x;
  const long long row = blockIdx.y;
  const T *x = logits + row * ld;
  const long long lo = split * chunk;
  const long long hi = min(V, lo + chunk);
  if (tid == 0) count = 0;

  bool ranked = false;
  if (VEC) {
    // The chunk sits in registers.  The K-th largest lane maximum of a warp is
    // reached by at least K elements of that warp, so no element strictly
    // below the largest such warp floor can be in the row's top K.  Elements
    // at or above it (about 1% of random logits) are compacted into shared
    // memory with one ballot per element position and ranked directly.
    constexpr int kV = Elem<T>::kVec;
    constexpr int NV = kWindow / (kThreads * kV);
    const uint4 *xv = reinterpret_cast<const uint4 *>(x + lo);
    const int nvec = (int)((hi - lo) / kV);
    uint4 buf[NV];
#pragma unroll
    for (int u = 0; u < NV; ++u) {
      const int i = u * kThreads + tid;
      buf[u] = i < nvec ? __ldcs(xv + i) : Elem<T>::nan_vec();  // NaN never passes a compare
    }
    float lm = -INFINITY;
#pragma unroll
    for (int u = 0; u < NV; ++u) lm = fmaxf(lm, Elem<T>::vmax(buf[u]));
    const float wk = warp_kth(lm, K, lane);
    if (lane == 0) wfloor[warp] = wk;
    __syncthreads();
    float floor_v = wfloor[0];
#pragma unroll
    for (int w = 1; w < kThreads / 32; ++w) floor_v = fmaxf(floor_v, wfloor[w]);
    const unsigned lt_mask = (1u << lane) - 1u;
#pragma unroll
    for (int u = 0; u < NV; ++u) {
      float e[kV];
      Elem<T>::unpack(buf[u], e);
#pragma unroll
      for (int q = 0; q < kV; ++q) {
        const bool c = e[q] >= floor_v;
        const unsigned bal = __ballot_sync(0xffffffffu, c);
        if (bal) {
          int base = 0;
          if (lane == 0) base = atomicAdd(&count, __popc(bal));
          base = __shfl_sync(0xffffffffu, base, 0);
          if (c) cand_o[base + __popc(bal & lt_mask)] = (unsigned short)((u * kThreads + tid) * kV + q);
        }
      }
    }
    // the ragged end of the chunk (fewer than one vector)
    const long long tail0 = lo + (long long)nvec * kV;
    if (tail0 + tid < hi) {
      const float v = Elem<T>::load1(x + tail0 + tid);
      if (v >= floor_v) cand_o[atomicAdd(&count, 1)] = (unsigned short)(tail0 + tid - lo);
    }
    __syncthreads();
    const int n = count;
    if (n <= kRankKeys) {
      for (int k = tid; k < n; k += kThreads) {
        const long long id = lo + cand_o[k];
        keys[k] = tr_key(tr_ord(Elem<T>::load_again(x + id)), (uint32_t)id);
      }
      rank_select(keys, n, K, top);
      ranked = true;
    } else {
      // many ties at the floor: fold the candidates through register lists
      TopList<KMAX> L;
      L.init();
      for (int k = tid; k < n; k += kThreads) {
        const long long id = lo + cand_o[k];
        L.push(Elem<T>::load_again(x + id), (uint32_t)id);
      }
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
      ranked = true;
    }
  }
  if (!ranked) {
    // rows that are not 16-byte aligned: a plain scan through register lists
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
  }

  if (splits > 1) {
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

template <typename T, int KMAX>
void launch(const void *logits, long long rows, long long V, long long ld, int K, int splits, long long chunk,
            bool vec, int32_t *ids, float *vals, void *ws, size_t part_bytes, cudaStream_t s) {
  unsigned long long *part = (unsigned long long *)ws;
  unsigned *counters = (unsigned *)((char *)ws + part_bytes);
  dim3 grid(splits, (unsigned)rows);
  if (vec)
    topk_kernel<T, KMAX, true><<<grid, kThreads, 0, s>>>((const T *)logits, V, ld, K, chunk, ids, vals, part, counters);
  else
    topk_kernel<T, KMAX, false><<<grid, kThreads, 0, s>>>((const T *)logits, V, ld, K, chunk, ids, vals, part,
                                                          counters);
}

long long plan_chunk(long long V, int splits) {
  // chunks are multiples of 8 elements so every chunk of an aligned row is 16-byte aligned
  long long c = (V + splits - 1) / splits;
  return (c + 7) / 8 * 8;
}

size_t part_bytes_for(long long rows, int splits, int K) {
  return splits > 1 ? tr_align_up((size_t)rows * splits * tr_kmax(K) * 8, 256) : 0;
}

}  // namespace

int tr_topk_plan_splits(int64_t rows, int64_t V) {
  (void)rows;
  long long s = (V + kChunk - 1) / kChunk;
  if (s < 1) s = 1;
  if (s > kMaxSplits) s = kMaxSplits;
  return (int)s;
}

extern "C" size_t tr_topk_workspace_bytes(int64_t rows, int64_t V, int K) {
  if (rows <= 0 || V <= 0 || K < 1 || K > TR_MAX_K) return 0;
  const int splits = tr_topk_plan_splits(rows, V);
  if (splits == 1) return 0;
  return part_bytes_for(rows, splits, K) + tr_align_up((size_t)rows * 4, 256);
}

int tr_topk_launch(const void *logits, tr_ftype ftype, int64_t rows, int64_t V, int64_t ld, int K, int32_t *ids,
                   float *vals, void *ws, size_t ws_bytes, cudaStream_t s) {
  const int splits = tr_topk_plan_splits(rows, V);
  const long long chunk = splits > 1 ? plan_chunk(V, splits) : V;
  const size_t esz = ftype == TR_F32 ? 4 : 2;
  const bool vec = ((uintptr_t)logits % 16 == 0) && ((ld * (int64_t)esz) % 16 == 0) && chunk <= kWindow;
  const size_t pb = part_bytes_for(rows, splits, K);
  const int km = tr_kmax(K);
#define TR_TOPK_CASE(T, KM) launch<T, KM>(logits, rows, V, ld, K, splits, chunk, vec, ids, vals, ws, pb, s)
  if (ftype == TR_F32) {
    if (km == 8) TR_TOPK_CASE(float, 8);
    else if (km == 16) TR_TOPK_CASE(float, 16);
    else TR_TOPK_CASE(float, 32);
  } else {
    if (km == 8) TR_TOPK_CASE(__nv_bfloat16, 8);
    else if (km == 16) TR_TOPK_CASE(__nv_bfloat16, 16);
    else TR_TOPK_CASE(__nv_bfloat16, 32);
  }
#undef TR_TOPK_CASE
  TR_LAUNCH_CHECK();
  (void)ws_bytes;
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
  if (rows > 65535) return TR_E_UNSUPPORTED;  // grid.y limit
  int rc = tr_check_device();
  if (rc != TR_OK) return rc;
  return tr_topk_launch(logits, ftype, rows, V, ld, K, ids, vals, ws, ws_bytes, (cudaStream_t)stream);
}
