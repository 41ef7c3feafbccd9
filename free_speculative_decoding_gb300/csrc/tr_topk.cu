// Per-row top-K over vocabulary logits (fp32 or bf16), ties to the lower ID.
//
// The kernel streams each row once from HBM with 16-byte loads.  A row is cut
// into `splits` chunks of at most 64 KB (16K fp32 or 32K bf16 elements), one
// CTA each, and a chunk sits in registers (64 KB over 256 threads).  Keys are
// 64-bit: an order-preserving value code in the high word and the
// complemented ID in the low word, so a larger key is better and equal values
// prefer the lower ID.  A floor taken from the lanes' maxima rejects all but
// a fraction of a percent of the elements; the rest are counted, given slots
// by a block-wide scan and ranked directly in shared memory.  The chunks of a
// row form one thread-block cluster (up to 8: V up to 131072 fp32 or 262144
// bf16) and merge through the first CTA's shared memory; longer rows merge in
// the last CTA to finish (an arrival counter in the workspace, no spin-wait).
#include "tr_internal.cuh"
#include "tr_lists.cuh"

namespace {

constexpr int kThreads = 256;
constexpr int kWindowBytes = 65536;      // bytes of a chunk a CTA holds in registers (64 a thread)
constexpr long long kChunkF32 = kWindowBytes / 4;  // elements per chunk of fp32 rows (the most splits)
constexpr int kRankKeys = 1024;           // keys ranked directly (also all chunks' lists of a row)
constexpr int kMaxSplits = 32;
constexpr int kMaxCluster = 8;  // portable thread-block cluster size

// K-th largest of the lanes' values (counting repeats), the same on every
// lane: a bitonic sort of the 32 values into descending lane order.
__device__ __forceinline__ float warp_kth(float v, int K, int lane) {
#pragma unroll
  for (int k = 2; k <= 32; k <<= 1) {
#pragma unroll
    for (int j = k >> 1; j > 0; j >>= 1) {
      const float o = __shfl_xor_sync(0xffffffffu, v, j);
      // blocks of k lanes alternate direction; the lower lane of a pair keeps
      // the larger value in a descending block
      const bool keep_max = ((lane & j) == 0) != ((lane & k) != 0);
      v = keep_max ? fmaxf(v, o) : fminf(v, o);
    }
  }
  return __shfl_sync(0xffffffffu, v, K - 1);
}

template <typename T>
struct Elem;
template <>
struct Elem<float> {
  static constexpr int kVec = 4;
  static constexpr bool kPrefilter = false;  // four compares cost less than a vector maximum
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
  static constexpr bool kPrefilter = true;   // packed maxima skip most unpacking
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
    // packed maxima first (exact: a maximum needs no rounding)
    const __nv_bfloat162 a = __hmax2(*reinterpret_cast<const __nv_bfloat162 *>(&q.x),
                                     *reinterpret_cast<const __nv_bfloat162 *>(&q.y));
    const __nv_bfloat162 b = __hmax2(*reinterpret_cast<const __nv_bfloat162 *>(&q.z),
                                     *reinterpret_cast<const __nv_bfloat162 *>(&q.w));
    const __nv_bfloat162 c = __hmax2(a, b);
    const uint32_t u = *reinterpret_cast<const uint32_t *>(&c);
    return fmaxf(__uint_as_float(u << 16), __uint_as_float(u & 0xFFFF0000u));
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
#pragma unroll 8
    for (int j = 0; j < n; ++j) rank += keys[j] > key;
    if (rank < K && key) out[rank] = key;
  }
  __syncthreads();
}

// Thread-block cluster helpers: the rank of this CTA in its cluster, a store
// into another CTA's shared memory, and the cluster-wide barrier.
__device__ __forceinline__ unsigned cluster_rank() {
  unsigned r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

__device__ __forceinline__ void st_cluster_u64(void *local_addr, unsigned rank, unsigned long long v) {
  const unsigned a = (unsigned)__cvta_generic_to_shared(local_addr);
  unsigned remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(a), "r"(rank));
  asm volatile("st.shared::cluster.u64 [%0], %1;" ::"r"(remote), "l"(v) : "memory");
}

__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// CLUSTER: the row's chunks form one thread-block cluster and merge through
// the first CTA's shared memory; otherwise through the workspace, the row's
// last CTA to finish merging (an arrival counter, no spin-wait).
template <typename T, int KMAX, bool VEC, bool CLUSTER>
__global__ void __launch_bounds__(kThreads, KMAX <= 8 ? 3 : 1) topk_kernel(const T *logits, long long V, long long ld, int K,
                                                        long long chunk, int32_t *ids, float *vals,
                                                        unsigned long long *part, unsigned *counters) {
  __shared__ unsigned long long keys[kRankKeys];       // candidate keys being ranked
  __shared__ unsigned long long top[TR_MAX_K];
  __shared__ unsigned long long gathered[kMaxCluster * TR_MAX_K];  // the cluster's lists (first CTA)
  __shared__ unsigned long long warp_keys[kThreads / 32][KMAX];
  __shared__ float wfloor[kThreads / 32];
  __shared__ int wcount[kThreads / 32];
  __shared__ int is_last;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int split = blockIdx.x, splits = gridDim.x;
  const long long row = blockIdx.y;
  const T *x = logits + row * ld;
  const long long lo = split * chunk;
  const long long hi = min(V, lo + chunk);

  bool ranked = false;
  if (VEC) {
    // The chunk sits in registers (64 bytes a thread).  The K-th largest
    // lane maximum of a warp is reached by at least K elements of that warp,
    // so no element strictly below the largest such warp floor can be in the
    // row's top K.  The elements at or above it (well under 1% of random
    // logits) are counted, given slots by a block-wide scan, and ranked.
    constexpr int kV = Elem<T>::kVec;
    constexpr int NV = kWindowBytes / (kThreads * 16);
    const uint4 *xv = reinterpret_cast<const uint4 *>(x + lo);
    const int nvec = (int)((hi - lo) / kV);
    uint4 buf[NV];
#pragma unroll
    for (int u = 0; u < NV; ++u) {
      const int i = u * kThreads + tid;
      buf[u] = i < nvec ? __ldcs(xv + i) : Elem<T>::nan_vec();  // NaN never passes a compare
    }
    // the ragged end of the chunk (fewer than one vector): one element for some threads
    const long long tail0 = lo + (long long)nvec * kV;
    const bool has_tail = tail0 + tid < hi;
    const float tail_v = has_tail ? Elem<T>::load1(x + tail0 + tid) : NAN;
    float lm = has_tail ? tail_v : -INFINITY;
#pragma unroll
    for (int u = 0; u < NV; ++u) lm = fmaxf(lm, Elem<T>::vmax(buf[u]));
    const float wk = warp_kth(lm, K, lane);
    if (lane == 0) wfloor[warp] = wk;
    __syncthreads();
    float floor_v = wfloor[0];
#pragma unroll
    for (int w = 1; w < kThreads / 32; ++w) floor_v = fmaxf(floor_v, wfloor[w]);
    // count, then a block-wide exclusive scan of the counts
    // (bf16: a vector whose maximum is below the floor is skipped whole)
    int cnt = has_tail && tail_v >= floor_v;
#pragma unroll
    for (int u = 0; u < NV; ++u) {
      if (!Elem<T>::kPrefilter || Elem<T>::vmax(buf[u]) >= floor_v) {
        float e[kV];
        Elem<T>::unpack(buf[u], e);
#pragma unroll
        for (int q = 0; q < kV; ++q) cnt += e[q] >= floor_v;
      }
    }
    int incl = cnt;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int o = __shfl_up_sync(0xffffffffu, incl, off);
      if (lane >= off) incl += o;
    }
    if (lane == 31) wcount[warp] = incl;
    __syncthreads();
    int base = incl - cnt, n = 0;
#pragma unroll
    for (int w = 0; w < kThreads / 32; ++w) {
      const int c = wcount[w];
      base += w < warp ? c : 0;
      n += c;
    }
    if (n <= kRankKeys) {
      // keys straight from the registers
      if (cnt) {
#pragma unroll
        for (int u = 0; u < NV; ++u) {
          if (!Elem<T>::kPrefilter || Elem<T>::vmax(buf[u]) >= floor_v) {
            float e[kV];
            Elem<T>::unpack(buf[u], e);
#pragma unroll
            for (int q = 0; q < kV; ++q)
              if (e[q] >= floor_v) keys[base++] = tr_key(tr_ord(e[q]), (uint32_t)(lo + (u * kThreads + tid) * kV + q));
          }
        }
        if (has_tail && tail_v >= floor_v) keys[base] = tr_key(tr_ord(tail_v), (uint32_t)(tail0 + tid));
      }
      __syncthreads();
      rank_select(keys, n, K, top);
      ranked = true;
    }
    // else: many elements tie at the floor; the plain scan below takes the chunk again
  }
  if (!ranked) {
    // rows that are not 16-byte aligned (or chunks with more than kRankKeys
    // elements at the floor): a plain scan through register lists
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

  if (CLUSTER) {
    // every chunk's list into the first CTA's shared memory, then one ranking there
    const unsigned cr = cluster_rank();
    if (tid < K) st_cluster_u64(&gathered[cr * K + tid], 0, top[tid]);
    cluster_sync();
    if (cr != 0) return;
    rank_select(gathered, splits * K, K, top);
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

template <typename T, int KMAX, bool VEC, bool CLUSTER>
cudaError_t launch_one(const void *logits, long long rows, long long V, long long ld, int K, int splits, long long chunk,
                int32_t *ids, float *vals, unsigned long long *part, unsigned *counters, cudaStream_t s) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(splits, (unsigned)rows);
  cfg.blockDim = dim3(kThreads);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  if (CLUSTER) {
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)splits;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
  }
  return cudaLaunchKernelEx(&cfg, topk_kernel<T, KMAX, VEC, CLUSTER>, (const T *)logits, V, ld, K, chunk, ids, vals,
                            part, counters);
}

template <typename T, int KMAX>
cudaError_t launch(const void *logits, long long rows, long long V, long long ld, int K, int splits, long long chunk,
            bool vec, int32_t *ids, float *vals, void *ws, size_t part_bytes, cudaStream_t s) {
  unsigned long long *part = (unsigned long long *)ws;
  unsigned *counters = (unsigned *)((char *)ws + part_bytes);
  const bool cluster = splits > 1 && splits <= kMaxCluster;
  if (vec)
    return cluster ? launch_one<T, KMAX, true, true>(logits, rows, V, ld, K, splits, chunk, ids, vals, part, counters, s)
                   : launch_one<T, KMAX, true, false>(logits, rows, V, ld, K, splits, chunk, ids, vals, part, counters, s);
  return cluster ? launch_one<T, KMAX, false, true>(logits, rows, V, ld, K, splits, chunk, ids, vals, part, counters, s)
                 : launch_one<T, KMAX, false, false>(logits, rows, V, ld, K, splits, chunk, ids, vals, part, counters, s);
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

// Chunks per row for elements of esz bytes; the workspace is laid out for
// fp32 (the most chunks), so it also fits bf16 rows.
static int plan_splits(int64_t V, size_t esz) {
  const long long per = kWindowBytes / (long long)esz;
  long long s = (V + per - 1) / per;
  if (s < 1) s = 1;
  if (s > kMaxSplits) s = kMaxSplits;
  return (int)s;
}

int tr_topk_plan_splits(int64_t rows, int64_t V) {
  (void)rows;
  return plan_splits(V, 4);
}

extern "C" size_t tr_topk_workspace_bytes(int64_t rows, int64_t V, int K) {
  if (rows <= 0 || V <= 0 || K < 1 || K > TR_MAX_K) return 0;
  const int splits = tr_topk_plan_splits(rows, V);
  if (splits == 1) return 0;
  return part_bytes_for(rows, splits, K) + tr_align_up((size_t)rows * 4, 256);
}

int tr_topk_launch(const void *logits, tr_ftype ftype, int64_t rows, int64_t V, int64_t ld, int K, int32_t *ids,
                   float *vals, void *ws, size_t ws_bytes, cudaStream_t s) {
  const size_t esz = ftype == TR_F32 ? 4 : 2;
  const int splits = plan_splits(V, esz);
  const long long chunk = splits > 1 ? plan_chunk(V, splits) : V;
  const bool vec = ((uintptr_t)logits % 16 == 0) && ((ld * (int64_t)esz) % 16 == 0) &&
                   chunk <= kWindowBytes / (long long)esz;
  // the partial lists are laid out for the fp32 chunk count (never fewer chunks)
  const size_t pb = part_bytes_for(rows, tr_topk_plan_splits(rows, V), K);
  const int km = tr_kmax(K);
#define TR_TOPK_CASE(T, KM) launch<T, KM>(logits, rows, V, ld, K, splits, chunk, vec, ids, vals, ws, pb, s)
  cudaError_t e;
  if (ftype == TR_F32)
    e = km == 8 ? TR_TOPK_CASE(float, 8) : km == 16 ? TR_TOPK_CASE(float, 16) : TR_TOPK_CASE(float, 32);
  else
    e = km == 8 ? TR_TOPK_CASE(__nv_bfloat16, 8) : km == 16 ? TR_TOPK_CASE(__nv_bfloat16, 16)
                : TR_TOPK_CASE(__nv_bfloat16, 32);
#undef TR_TOPK_CASE
  if (e != cudaSuccess) return TR_E_CUDA;
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
