// Register top-K lists of 64-bit ordered keys and their warp-level merge,
// shared by the top-K kernel and the LM-head epilogue.
#pragma once

#include "tr_internal.cuh"

template <int KMAX>
struct TopList {
  unsigned long long k[KMAX];
  float thr;    // values below thr cannot enter: max(own KMAX-th value, floor)
  float floor;  // a value known to be beaten KMAX times elsewhere in the same merge group

  __device__ __forceinline__ void init() {
#pragma unroll
    for (int j = 0; j < KMAX; ++j) k[j] = 0ull;
    thr = -INFINITY;
    floor = -INFINITY;
  }

  // Raise the rejection threshold to f, the KMAX-th best value of another list
  // whose keys are merged with this one: a value strictly below f is beaten by
  // KMAX keys of that list, so it cannot be among the merged top KMAX.
  __device__ __forceinline__ void raise_floor(float f) {
    floor = fmaxf(floor, f);
    thr = fmaxf(thr, floor);
  }

  __device__ __forceinline__ void push(float v, uint32_t id) {
    if (v >= thr) {
      unsigned long long key = tr_key(tr_ord(v), id);
      if (key > k[KMAX - 1]) {
#pragma unroll
        for (int j = 0; j < KMAX; ++j) {
          const unsigned long long hi = k[j] > key ? k[j] : key;
          key = k[j] > key ? key : k[j];
          k[j] = hi;
        }
        thr = fmaxf(k[KMAX - 1] ? tr_key_val(k[KMAX - 1]) : -INFINITY, floor);
      }
    }
  }
};

// K rounds of a warp-wide maximum over the lanes' list heads; lane r returns
// the r-th largest key (0 when the warp holds fewer than r+1 keys).
template <int KMAX>
__device__ __forceinline__ unsigned long long warp_merge(TopList<KMAX> &L, int lane) {
  unsigned long long mine = 0ull;
#pragma unroll
  for (int r = 0; r < KMAX; ++r) {
    const unsigned long long head = L.k[0];
    unsigned long long m = head;
#pragma unroll
    for (int off = 16; off; off >>= 1) {
      const unsigned long long o = __shfl_xor_sync(0xffffffffu, m, off);
      m = o > m ? o : m;
    }
    if (m != 0ull && head == m) {
#pragma unroll
      for (int j = 0; j < KMAX - 1; ++j) L.k[j] = L.k[j + 1];
      L.k[KMAX - 1] = 0ull;
    }
    if (lane == r) mine = m;
  }
  return mine;
}

// Insert a key into a sorted (descending) register list, dropping the smallest.
template <int KMAX>
__device__ __forceinline__ void list_insert(unsigned long long (&k)[KMAX], unsigned long long key) {
  if (key > k[KMAX - 1]) {
#pragma unroll
    for (int t = 0; t < KMAX; ++t) {
      const unsigned long long h = k[t] > key ? k[t] : key;
      key = k[t] > key ? key : k[t];
      k[t] = h;
    }
  }
}
