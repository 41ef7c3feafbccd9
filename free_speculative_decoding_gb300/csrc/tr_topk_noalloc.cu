// tr_topk_noalloc: the per-row top-K with its scratch in a fixed device array
// of this library instead of a caller-provided workspace.
//
// Who needs it: callers that hold their logits, IDs and values on the device
// but cannot obtain any more device memory -- a plugin inside a host framework
// whose memory planner owns every buffer and offers plugins no workspace, a
// latency-critical serving loop that must never call cudaMalloc (it can
// synchronise the whole device and stall every stream), or a thin
// foreign-function caller with tensors in hand but no allocator of its own.
//
// The scratch (per-chunk partial lists and per-row arrival counters, exactly
// what tr_topk keeps in its workspace) is a file-scope static __device__ array
// of TR_TOPK_NOALLOC_SCRATCH_BYTES.  Every GPU that loads the library holds it
// until the process exits.  In host code the array's name is only a host-side
// stand-in, never a device address, so its device address is looked up with
// cudaGetSymbolAddress once per device (on that device's first call, with the
// device current) and passed to the kernel.
#include <atomic>

#include "tr_internal.cuh"

static __device__ __align__(256) unsigned char g_topk_scratch[TR_TOPK_NOALLOC_SCRATCH_BYTES];

#define TR_NOALLOC_MAX_DEVICES 64
// per-device address cache; atomic so that first calls from several host
// threads at once are well defined (they all store the same address)
static std::atomic<void *> g_scratch_addr[TR_NOALLOC_MAX_DEVICES];

// Device address of this device's scratch array (looked up once per device).
static int scratch_address(void **out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= TR_NOALLOC_MAX_DEVICES) return TR_E_CUDA;
  void *p = g_scratch_addr[dev].load(std::memory_order_acquire);
  if (!p) {
    if (cudaGetSymbolAddress(&p, g_topk_scratch) != cudaSuccess || !p) return TR_E_CUDA;
    g_scratch_addr[dev].store(p, std::memory_order_release);
  }
  *out = p;
  return TR_OK;
}

extern "C" int tr_topk_noalloc(const void *logits, tr_ftype ftype, int64_t rows, int64_t V, int64_t ld, int K,
                               int32_t *ids, float *vals, tr_stream_t stream) {
  if (rows < 0 || V < 1 || K < 1 || K > TR_MAX_K || K > V || ld < V) return TR_E_INVAL;
  if (ftype != TR_F32 && ftype != TR_BF16) return TR_E_INVAL;
  if (V > INT32_MAX) return TR_E_UNSUPPORTED;
  if (rows == 0) return TR_OK;
  if (!logits || !ids) return TR_E_INVAL;
  if (rows > 65535) return TR_E_UNSUPPORTED;
  // the same scratch tr_topk would take from a workspace; refuse what the array cannot hold
  const size_t need = tr_topk_workspace_bytes(rows, V, K);
  if (need > (size_t)TR_TOPK_NOALLOC_SCRATCH_BYTES) return TR_E_UNSUPPORTED;
  int rc = tr_check_device();
  if (rc != TR_OK) return rc;
  void *scratch = nullptr;
  rc = scratch_address(&scratch);
  if (rc != TR_OK) return rc;
  cudaStream_t s = (cudaStream_t)stream;
  if (need) {
    // the arrival counters sit after the partial lists and must start at zero;
    // the array keeps whatever the previous call left there
    const size_t part = tr_topk_counters_offset(rows, V, K);
    if (cudaMemsetAsync((char *)scratch + part, 0, need - part, s) != cudaSuccess) return TR_E_CUDA;
  }
  return tr_topk_launch(logits, ftype, rows, V, ld, K, ids, vals, scratch, (size_t)TR_TOPK_NOALLOC_SCRATCH_BYTES, s);
}
