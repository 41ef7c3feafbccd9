// Device-side generators of the synthetic workload (the target-model stand-in).
// Not part of Token Recycling; see tr_synth.h for the definitions.
#include "tr_internal.cuh"
#include "tr_synth.h"

namespace {

constexpr unsigned long long kGamma = 0x9E3779B97F4A7C15ull;
enum {
  TAG_NEXT = 1, TAG_ALT = 2, TAG_NOISE = 3, TAG_WARM = 5, TAG_H = 12, TAG_W = 13, TAG_CLASS = 14, TAG_E = 15,
  TAG_G = 16, TAG_U = 17
};
constexpr int kAlt = 7;
constexpr int kClasses = 16;

__device__ __forceinline__ unsigned long long mix64(unsigned long long z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

__device__ __forceinline__ unsigned long long chain(unsigned long long h, unsigned long long f) {
  return mix64(h + kGamma + f);
}

__device__ __forceinline__ unsigned long long hkey2(unsigned long long a, unsigned long long b) {
  return chain(chain(0ull, a), b);
}
__device__ __forceinline__ unsigned long long hkey3(unsigned long long a, unsigned long long b, unsigned long long c) {
  return chain(hkey2(a, b), c);
}
__device__ __forceinline__ unsigned long long hkey4(unsigned long long a, unsigned long long b, unsigned long long c,
                                                    unsigned long long d) {
  return chain(hkey3(a, b, c), d);
}
__device__ __forceinline__ unsigned long long hkey5(unsigned long long a, unsigned long long b, unsigned long long c,
                                                    unsigned long long d, unsigned long long e) {
  return chain(hkey4(a, b, c, d), e);
}

__device__ __forceinline__ float ih12(unsigned long long key, unsigned long long i) {
  int total = 0;
#pragma unroll
  for (int j = 0; j < 3; ++j) {
    const unsigned long long w = mix64(key + kGamma * (3ull * i + (unsigned long long)j + 1ull));
    total += (int)(w & 0xFFFFull) + (int)((w >> 16) & 0xFFFFull) + (int)((w >> 32) & 0xFFFFull) + (int)(w >> 48);
  }
  return (float)(total - 393210) * (1.0f / 65536.0f);
}

__device__ __forceinline__ unsigned short bf16_rne(float x) {
  return __bfloat16_as_ushort(__float2bfloat16_rn(x));
}

// row = b*N + n; 4 consecutive vocabulary entries per thread
__global__ void logits_kernel(unsigned long long seed, long long V, const __grid_constant__ TreeDev tree,
                              const int32_t *tree_tok, const int32_t *L, int bf16, void *out, long long ld) {
  const long long row = blockIdx.y;
  const int N = tree.N;
  const int b = (int)(row / N), n = (int)(row % N);
  const unsigned long long tok = (unsigned long long)(long long)tree_tok[row];
  const unsigned long long pos = (unsigned long long)(long long)(L[b] + tree.depth[n]);
  const unsigned long long rk = hkey5(seed, TAG_NOISE, (unsigned long long)b, pos, tok);
  const long long nxt = (long long)(hkey4(seed, TAG_NEXT, (unsigned long long)b, tok) % (unsigned long long)V);
  long long alt[kAlt];
#pragma unroll
  for (int j = 0; j < kAlt; ++j)
    alt[j] = (long long)(hkey5(seed, TAG_ALT, (unsigned long long)b, tok, (unsigned long long)j) % (unsigned long long)V);
  for (long long v = ((long long)blockIdx.x * blockDim.x + threadIdx.x); v < V; v += (long long)gridDim.x * blockDim.x) {
    float x = ih12(rk, (unsigned long long)v);
    float boost = 0.f;
    if (v == nxt) boost = 6.0f;
    else {
#pragma unroll
      for (int j = 0; j < kAlt; ++j)
        if (v == alt[j]) boost = 3.0f;
    }
    x = x + boost;
    if (bf16) ((unsigned short *)out)[row * ld + v] = bf16_rne(x);
    else ((float *)out)[row * ld + v] = x;
  }
}

__global__ void rows_kernel(unsigned long long seed, int tag, long long step, int n1, int n2, int d, long long nrows,
                            unsigned short *out) {
  for (long long e = (long long)blockIdx.x * blockDim.x + threadIdx.x; e < nrows * d;
       e += (long long)gridDim.x * blockDim.x) {
    const long long r = e / d;
    const int i = (int)(e % d);
    const long long i2 = r % n2, i1 = (r / n2) % n1, i0 = r / ((long long)n1 * n2);
    const unsigned long long key = chain(hkey5(seed, (unsigned long long)tag, (unsigned long long)step,
                                               (unsigned long long)i0, (unsigned long long)i1),
                                         (unsigned long long)i2);
    out[e] = bf16_rne(ih12(key, (unsigned long long)i));
  }
}

__global__ void cache_kernel(unsigned long long seed, int tag, int H, int cap, int d, const int32_t *L,
                             unsigned short *out) {
  const int b = blockIdx.z, h = blockIdx.y;
  const int Lb = min(max(L[b], 0), cap);
  for (long long e = (long long)blockIdx.x * blockDim.x + threadIdx.x; e < (long long)Lb * d;
       e += (long long)gridDim.x * blockDim.x) {
    const long long p = e / d;
    const int i = (int)(e % d);
    const unsigned long long key =
        hkey5(seed, (unsigned long long)tag, (unsigned long long)b, (unsigned long long)h, (unsigned long long)p);
    out[(((long long)b * H + h) * cap + p) * d + i] = bf16_rne(ih12(key, (unsigned long long)i));
  }
}

__device__ __forceinline__ float class_sign(unsigned long long seed, int c, int i) {
  return (hkey4(seed, TAG_E, (unsigned long long)c, (unsigned long long)i) & 1ull) == 0ull ? 1.0f : -1.0f;
}

__global__ void lm_hidden_kernel(unsigned long long seed, int D, const __grid_constant__ TreeDev tree,
                                 const int32_t *tree_tok, const int32_t *L, unsigned short *out) {
  const long long row = blockIdx.x;
  const int N = tree.N;
  const int b = (int)(row / N), n = (int)(row % N);
  const unsigned long long tok = (unsigned long long)(long long)tree_tok[row];
  const unsigned long long pos = (unsigned long long)(long long)(L[b] + tree.depth[n]);
  const unsigned long long key = hkey5(seed, TAG_H, (unsigned long long)b, pos, tok);
  const int c = (int)(hkey3(seed, TAG_CLASS, tok) % kClasses);
  for (int i = threadIdx.x; i < D; i += blockDim.x) {
    float x = ih12(key, (unsigned long long)i);
    x = rintf(x * 32.0f) / 32.0f;
    x = x + 0.25f * class_sign(seed, c, i);
    out[row * D + i] = bf16_rne(x);
  }
}

__global__ void lm_weight_kernel(unsigned long long seed, long long V, int D, unsigned short *out) {
  const long long v = blockIdx.x;
  __shared__ int hits[kClasses];
  __shared__ int n_hits;
  if (threadIdx.x == 0) {
    int m = 0;
    for (int c = 0; c < kClasses; ++c)
      if ((long long)(hkey3(seed, TAG_G, (unsigned long long)c) % (unsigned long long)V) == v) hits[m++] = c;
    n_hits = m;
  }
  __syncthreads();
  const unsigned long long key = hkey3(seed, TAG_W, (unsigned long long)v);
  for (int i = threadIdx.x; i < D; i += blockDim.x) {
    float x = ih12(key, (unsigned long long)i) * 0.02f;
    x = rintf(x * 1024.0f) / 1024.0f;
    for (int q = 0; q < n_hits; ++q) x = x + 0.0078125f * class_sign(seed, hits[q], i);
    out[v * D + i] = bf16_rne(x);
  }
}

template <typename T>
__global__ void warm_kernel(unsigned long long seed, int B, long long V, int K, T *M) {
  for (long long e = (long long)blockIdx.x * blockDim.x + threadIdx.x; e < (long long)B * V;
       e += (long long)gridDim.x * blockDim.x) {
    const unsigned long long b = (unsigned long long)(e / V), t = (unsigned long long)(e % V);
    const bool good = (hkey4(seed, TAG_WARM, b, t) & 1ull) == 0ull;
    T *row = M + e * K;
    for (int j = 0; j < K; ++j) {
      unsigned long long val;
      if (good && j == 0) val = hkey4(seed, TAG_NEXT, b, t);
      else if (good && j <= kAlt) val = hkey5(seed, TAG_ALT, b, t, (unsigned long long)(j - 1));
      else val = hkey5(seed, TAG_WARM, b, t, (unsigned long long)(j + 1));
      row[j] = (T)(long long)(val % (unsigned long long)V);
    }
  }
}

// out[(b*N + n)*K1 + j] = top 24 bits of output j of the stream at key (seed, 17, step, b, n), times 2^-24
__global__ void uniforms_kernel(unsigned long long seed, long long step, int N, int K1, long long total, float *out) {
  for (long long e = (long long)blockIdx.x * blockDim.x + threadIdx.x; e < total;
       e += (long long)gridDim.x * blockDim.x) {
    const unsigned long long j = (unsigned long long)(e % K1), bn = (unsigned long long)(e / K1);
    const unsigned long long key = hkey5(seed, TAG_U, (unsigned long long)step, bn / N, bn % N);
    out[e] = (float)(mix64(key + kGamma * (j + 1ull)) >> 40) * (1.0f / 16777216.0f);
  }
}

}  // namespace

extern "C" int trsyn_uniforms(uint64_t seed, int64_t step, int B, int N, int K1, float *out, tr_stream_t stream) {
  if (!out || B < 1 || N < 1 || K1 < 1) return TR_E_INVAL;
  int rc = tr_check_device();
  if (rc != TR_OK) return rc;
  uniforms_kernel<<<tr_sm_count() * 2, 256, 0, (cudaStream_t)stream>>>(seed, step, N, K1, (long long)B * N * K1, out);
  TR_LAUNCH_CHECK();
  return TR_OK;
}

extern "C" int trsyn_logits(uint64_t seed, int B, int64_t V, const struct tr_tree *tree, const int32_t *tree_tok,
                            const int32_t *L, tr_ftype ftype, void *out, int64_t ld, tr_stream_t stream) {
  if (!tree || !tree_tok || !L || !out || B < 1 || V < 1 || ld < V) return TR_E_INVAL;
  const long long rows = (long long)B * tree->dev.N;
  if (rows > 65535) return TR_E_UNSUPPORTED;
  int rc = tr_check_device();
  if (rc != TR_OK) return rc;
  const int threads = 256;
  const int gx = (int)((V + threads * 4 - 1) / (threads * 4));
  logits_kernel<<<dim3(gx, (unsigned)rows), threads, 0, (cudaStream_t)stream>>>(seed, V, tree->dev, tree_tok, L,
                                                                                ftype == TR_BF16, out, ld);
  TR_LAUNCH_CHECK();
  return TR_OK;
}

extern "C" int trsyn_rows_bf16(uint64_t seed, int tag, int64_t step, int n0, int n1, int n2, int d, void *out,
                               tr_stream_t stream) {
  if (!out || n0 < 1 || n1 < 1 || n2 < 1 || d < 1) return TR_E_INVAL;
  int rc = tr_check_device();
  if (rc != TR_OK) return rc;
  const long long nrows = (long long)n0 * n1 * n2;
  rows_kernel<<<tr_sm_count() * 8, 256, 0, (cudaStream_t)stream>>>(seed, tag, step, n1, n2, d, nrows,
                                                                   (unsigned short *)out);
  TR_LAUNCH_CHECK();
  return TR_OK;
}

extern "C" int trsyn_cache_bf16(uint64_t seed, int tag, int B, int H, int cap, int d, const int32_t *L, void *out,
                                tr_stream_t stream) {
  if (!out || !L || B < 1 || H < 1 || cap < 1 || d < 1 || B > 65535 || H > 65535) return TR_E_INVAL;
  int rc = tr_check_device();
  if (rc != TR_OK) return rc;
  cache_kernel<<<dim3(64, H, B), 256, 0, (cudaStream_t)stream>>>(seed, tag, H, cap, d, L, (unsigned short *)out);
  TR_LAUNCH_CHECK();
  return TR_OK;
}

extern "C" int trsyn_lm_hidden(uint64_t seed, int B, int D, const struct tr_tree *tree, const int32_t *tree_tok,
                               const int32_t *L, void *out, tr_stream_t stream) {
  if (!tree || !tree_tok || !L || !out || B < 1 || D < 1) return TR_E_INVAL;
  int rc = tr_check_device();
  if (rc != TR_OK) return rc;
  lm_hidden_kernel<<<B * tree->dev.N, 256, 0, (cudaStream_t)stream>>>(seed, D, tree->dev, tree_tok, L,
                                                                     (unsigned short *)out);
  TR_LAUNCH_CHECK();
  return TR_OK;
}

extern "C" int trsyn_lm_weight(uint64_t seed, int64_t V, int D, void *out, tr_stream_t stream) {
  if (!out || V < 1 || D < 1 || V > INT32_MAX) return TR_E_INVAL;
  int rc = tr_check_device();
  if (rc != TR_OK) return rc;
  lm_weight_kernel<<<(unsigned)V, 256, 0, (cudaStream_t)stream>>>(seed, V, D, (unsigned short *)out);
  TR_LAUNCH_CHECK();
  return TR_OK;
}

extern "C" int trsyn_warm_matrix(uint64_t seed, int B, int64_t V, int K, tr_itype mtype, void *M, tr_stream_t stream) {
  if (!M || B < 1 || V < 1 || K < 1 || K > TR_MAX_K) return TR_E_INVAL;
  int rc = tr_check_device();
  if (rc != TR_OK) return rc;
  const int grid = tr_sm_count() * 8;
  if (mtype == TR_I64)
    warm_kernel<long long><<<grid, 256, 0, (cudaStream_t)stream>>>(seed, B, V, K, (long long *)M);
  else
    warm_kernel<int32_t><<<grid, 256, 0, (cudaStream_t)stream>>>(seed, B, V, K, (int32_t *)M);
  TR_LAUNCH_CHECK();
  return TR_OK;
}
