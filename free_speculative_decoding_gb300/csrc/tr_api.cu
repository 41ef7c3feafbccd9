// Host side of libtr: tree plans, status word, device checks, matrix init.
#include <stdlib.h>
#include <string.h>

#include <atomic>

#include "tr_internal.cuh"

static __device__ unsigned int tr_dev_status_word = 0;

#define TR_MAX_DEVICES 64
// per-device caches, filled on a device's first call; atomic so that first
// calls from several host threads at once are well defined
static std::atomic<unsigned int *> g_status_ptr[TR_MAX_DEVICES];
static std::atomic<int> g_arch_ok[TR_MAX_DEVICES];  // 0 unknown, 1 ok, -1 unsupported
static std::atomic<int> g_sm_count[TR_MAX_DEVICES];

static int current_device() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= TR_MAX_DEVICES) return -1;
  return dev;
}

unsigned int *tr_status_dev() {
  int dev = current_device();
  if (dev < 0) return nullptr;
  unsigned int *s = g_status_ptr[dev].load(std::memory_order_acquire);
  if (!s) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, tr_dev_status_word) != cudaSuccess) return nullptr;
    s = (unsigned int *)p;
    g_status_ptr[dev].store(s, std::memory_order_release);
  }
  return s;
}

int tr_check_device() {
  int dev = current_device();
  if (dev < 0) {
    cudaGetLastError();
    return TR_E_CUDA;
  }
  if (g_arch_ok[dev].load() == 0) {
    int major = 0, minor = 0, sms = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return TR_E_CUDA;
    g_sm_count[dev].store(sms);
    g_arch_ok[dev].store((major == 10 && minor == 3) ? 1 : -1);
  }
  if (g_arch_ok[dev].load() < 0) return TR_E_UNSUPPORTED;
  if (!tr_status_dev()) return TR_E_CUDA;
  return TR_OK;
}

int tr_sm_count() {
  int dev = current_device();
  if (dev < 0) return 148;
  if (g_sm_count[dev].load() == 0) tr_check_device();
  const int n = g_sm_count[dev].load();
  return n > 0 ? n : 148;
}

// ---------------------------------------------------------------------------
// tree plans
// ---------------------------------------------------------------------------

extern "C" int tr_tree_create(const int32_t *child_counts, int n_nodes, int K, struct tr_tree **out) {
  if (!child_counts || !out || n_nodes < 1 || n_nodes > TR_MAX_NODES || K < 1 || K > TR_MAX_K)
    return TR_E_INVAL;
  *out = nullptr;
  tr_tree *t = (tr_tree *)calloc(1, sizeof(tr_tree));
  if (!t) return TR_E_INVAL;
  TreeDev &d = t->dev;
  int named = 1;  // nodes given an index so far (the root)
  d.parent[0] = 0;
  d.rank[0] = 0;
  d.depth[0] = 0;
  for (int n = 0; n < n_nodes; ++n) {
    int c = child_counts[n];
    if (c < 0 || c > K || n >= named || named + c > n_nodes) {
      free(t);
      return TR_E_INVAL;
    }
    t->child_counts[n] = c;
    d.child_first[n] = (uint8_t)(c ? named : 0);
    d.child_count[n] = (uint8_t)c;
    for (int r = 0; r < c; ++r) {
      d.parent[named] = (uint8_t)n;
      d.rank[named] = (uint8_t)r;
      d.depth[named] = (uint8_t)(d.depth[n] + 1);
      ++named;
    }
  }
  if (named != n_nodes) {
    free(t);
    return TR_E_INVAL;
  }
  d.N = n_nodes;
  d.K = K;
  int D = 0;
  for (int n = 0; n < n_nodes; ++n) D = d.depth[n] > D ? d.depth[n] : D;
  d.D = D;
  // nodes are in BFS order, so each level is a contiguous range
  int n = 0;
  for (int l = 0; l <= D + 1; ++l) {
    while (n < n_nodes && d.depth[n] < l) ++n;
    d.level_off[l] = (uint8_t)n;
  }
  for (int i = 0; i < n_nodes; ++i) {
    int m = i;
    while (true) {
      d.anc[i][m >> 6] |= 1ull << (m & 63);
      if (m == 0) break;
      m = d.parent[m];
    }
  }
  *out = t;
  return TR_OK;
}

extern "C" int tr_tree_destroy(struct tr_tree *tree) {
  free(tree);
  return TR_OK;
}

extern "C" int tr_tree_info(const struct tr_tree *tree, int *n_nodes, int *max_depth, int32_t *parent,
                            int32_t *rank, int32_t *depth) {
  if (!tree) return TR_E_INVAL;
  const TreeDev &d = tree->dev;
  if (n_nodes) *n_nodes = d.N;
  if (max_depth) *max_depth = d.D;
  for (int n = 0; n < d.N; ++n) {
    if (parent) parent[n] = n == 0 ? -1 : d.parent[n];
    if (rank) rank[n] = d.rank[n];
    if (depth) depth[n] = d.depth[n];
  }
  return TR_OK;
}

// ---------------------------------------------------------------------------
// status word, workspace
// ---------------------------------------------------------------------------

extern "C" int tr_get_status(int32_t *host_out, tr_stream_t stream) {
  if (!host_out) return TR_E_INVAL;
  int rc = tr_check_device();
  if (rc != TR_OK) return rc;
  unsigned int v = 0, zero = 0;
  TR_TRY_CUDA(cudaStreamSynchronize((cudaStream_t)stream));
  TR_TRY_CUDA(cudaMemcpy(&v, tr_status_dev(), sizeof(v), cudaMemcpyDeviceToHost));
  TR_TRY_CUDA(cudaMemcpy(tr_status_dev(), &zero, sizeof(zero), cudaMemcpyHostToDevice));
  *host_out = (int32_t)v;
  return v ? TR_E_DEVICE : TR_OK;
}

static std::atomic<unsigned long long> g_wait_limit_ns{2000000000ull};

unsigned long long tr_wait_limit_ns() { return g_wait_limit_ns.load(std::memory_order_relaxed); }

extern "C" int tr_set_wait_limit_ns(uint64_t ns, uint64_t *previous) {
  if (ns < 1 || ns > 60000000000ull) return TR_E_INVAL;
  const unsigned long long old = g_wait_limit_ns.exchange(ns);
  if (previous) *previous = old;
  return TR_OK;
}

extern "C" int tr_workspace_clear(void *ws, size_t ws_bytes, tr_stream_t stream) {
  if (!ws && ws_bytes) return TR_E_INVAL;
  if (!ws_bytes) return TR_OK;
  TR_TRY_CUDA(cudaMemsetAsync(ws, 0, ws_bytes, (cudaStream_t)stream));
  return TR_OK;
}

extern "C" const char *tr_status_string(int status) {
  switch (status) {
    case TR_OK: return "TR_OK";
    case TR_E_INVAL: return "TR_E_INVAL: invalid argument";
    case TR_E_UNSUPPORTED: return "TR_E_UNSUPPORTED: not supported on this device or configuration";
    case TR_E_CUDA: return "TR_E_CUDA: a CUDA call or launch failed";
    case TR_E_DEVICE: return "TR_E_DEVICE: the device status word has error bits set";
    case TR_E_TIMEOUT: return "TR_E_TIMEOUT: a bounded wait gave up";
    default: return "unknown tr_status";
  }
}

// ---------------------------------------------------------------------------
// matrix initialisation
// ---------------------------------------------------------------------------

__device__ __forceinline__ unsigned long long tr_splitmix64(unsigned long long state, unsigned long long index) {
  // splitmix64 (Steele, Lea, Flood 2014): output `index` of the stream at `state`
  unsigned long long z = state + (index + 1ull) * 0x9E3779B97F4A7C15ull;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

template <typename T>
__global__ void init_matrix_kernel(T *M, long long total, long long VK, long long V, int mode, const T *src,
                                   unsigned long long seed) {
  for (long long e = blockIdx.x * (long long)blockDim.x + threadIdx.x; e < total;
       e += (long long)gridDim.x * blockDim.x) {
    if (mode == TR_INIT_RANDOM)
      M[e] = (T)(tr_splitmix64(seed, (unsigned long long)e) % (unsigned long long)V);
    else
      M[e] = src[e % VK];
  }
}

extern "C" int tr_init_matrix(void *M, tr_itype mtype, int B, int64_t V, int K, tr_init_mode mode,
                              const void *src, uint64_t seed, tr_stream_t stream) {
  if (!M || B < 1 || V < 1 || K < 1 || K > TR_MAX_K) return TR_E_INVAL;
  if (mtype != TR_I32 && mtype != TR_I64) return TR_E_INVAL;
  if (mode != TR_INIT_ZERO && mode != TR_INIT_RANDOM && mode != TR_INIT_INHERIT) return TR_E_INVAL;
  if (mode == TR_INIT_INHERIT && !src) return TR_E_INVAL;
  if (mtype == TR_I32 && V > INT32_MAX) return TR_E_UNSUPPORTED;
  int rc = tr_check_device();
  if (rc != TR_OK) return rc;
  size_t esz = mtype == TR_I64 ? 8 : 4;
  long long VK = (long long)V * K, total = VK * B;
  cudaStream_t s = (cudaStream_t)stream;
  if (mode == TR_INIT_ZERO) {
    TR_TRY_CUDA(cudaMemsetAsync(M, 0, (size_t)total * esz, s));
    return TR_OK;
  }
  int grid = tr_sm_count() * 8;
  if (mtype == TR_I64)
    init_matrix_kernel<long long><<<grid, 256, 0, s>>>((long long *)M, total, VK, V, mode,
                                                      (const long long *)src, seed);
  else
    init_matrix_kernel<int32_t><<<grid, 256, 0, s>>>((int32_t *)M, total, VK, V, mode, (const int32_t *)src, seed);
  TR_LAUNCH_CHECK();
  return TR_OK;
}
