// Internal definitions shared by the libtr translation units.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "tr.h"

#define TR_MAX_NODES 128
#define TR_MAX_K 32

// Plan of a static draft tree, passed by value as a __grid_constant__ kernel
// parameter (about 2.7 KB), so launches need no device allocation and a CUDA
// graph captures the plan with the launch.
struct TreeDev {
  int N;          // nodes
  int D;          // depth of the deepest node
  int K;          // candidates per matrix row
  uint8_t level_off[TR_MAX_NODES + 2];  // level l holds nodes [level_off[l], level_off[l+1])
  uint8_t parent[TR_MAX_NODES];         // parent of node n (root: 0)
  uint8_t rank[TR_MAX_NODES];           // child index of n under its parent
  uint8_t depth[TR_MAX_NODES];
  uint8_t child_first[TR_MAX_NODES];    // children of n are nodes child_first[n] .. + child_count[n] - 1
  uint8_t child_count[TR_MAX_NODES];    // (BFS order keeps a node's children together, in rank order)
  unsigned long long anc[TR_MAX_NODES][2];  // bit j set iff node j is on the root->n path (n included)
};

struct tr_tree {
  TreeDev dev;
  int32_t child_counts[TR_MAX_NODES];
};

// Device address of the per-device status word (a static __device__ variable
// of tr_api.cu, looked up once per device); kernels receive it as an argument.
unsigned int *tr_status_dev();

__device__ __forceinline__ void tr_flag(unsigned int *status, unsigned int bits) { atomicOr(status, bits); }

// ---------------------------------------------------------------------------
// ordered keys for top-K: larger key = better; ties in value go to the lower id
// ---------------------------------------------------------------------------

// Monotone map of a finite float to uint32 (+0.0 and -0.0 map to the same code).
__device__ __forceinline__ uint32_t tr_ord(float v) {
  uint32_t u = __float_as_uint(v + 0.0f);  // -0.0 + 0.0 = +0.0 under round-to-nearest
  return u ^ ((uint32_t)((int32_t)u >> 31) | 0x80000000u);
}

__device__ __forceinline__ float tr_unord(uint32_t o) {
  uint32_t u = (o & 0x80000000u) ? (o ^ 0x80000000u) : ~o;
  return __uint_as_float(u);
}

__device__ __forceinline__ unsigned long long tr_key(uint32_t ord, uint32_t id) {
  return ((unsigned long long)ord << 32) | (unsigned long long)(0xFFFFFFFFu - id);
}

__device__ __forceinline__ uint32_t tr_key_id(unsigned long long k) {
  return 0xFFFFFFFFu - (uint32_t)(k & 0xFFFFFFFFull);
}

__device__ __forceinline__ float tr_key_val(unsigned long long k) { return tr_unord((uint32_t)(k >> 32)); }

// ---------------------------------------------------------------------------
// host helpers
// ---------------------------------------------------------------------------

int tr_check_device();  // TR_OK on an sm_103 device, else TR_E_UNSUPPORTED / TR_E_CUDA
unsigned long long tr_wait_limit_ns();  // limit of the bounded device waits (tr_set_wait_limit_ns)
int tr_sm_count();

#define TR_TRY_CUDA(expr)                         \
  do {                                            \
    cudaError_t _e = (expr);                      \
    if (_e != cudaSuccess) return TR_E_CUDA;      \
  } while (0)

#define TR_LAUNCH_CHECK()                         \
  do {                                            \
    if (cudaGetLastError() != cudaSuccess) return TR_E_CUDA; \
  } while (0)

static inline size_t tr_align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// smallest supported register-list width for K
static inline int tr_kmax(int K) { return K <= 8 ? 8 : (K <= 16 ? 16 : 32); }

// top-K internals shared with the step and the LM head
size_t tr_topk_counters_offset(int64_t rows, int64_t V, int K);  // byte offset of the arrival counters in the workspace
// stats != NULL: also each row's (max, sum of exp((x - max) / temperature)) into stats [rows, 2]
// and every 8 KB step's pair into step_stats [rows, tr_softmax_steps(V, ftype), 2]
// (16-byte aligned rows only: the caller checks)
int tr_topk_launch(const void *logits, tr_ftype ftype, int64_t rows, int64_t V, int64_t ld, int K,
                   int32_t *ids, float *vals, void *ws, size_t ws_bytes, cudaStream_t stream,
                   float temperature = 1.f, float *stats = nullptr, float *step_stats = nullptr);
