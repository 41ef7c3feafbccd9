// Tree-attention verification: split-KV decode over the prefix cache plus the
// flattened draft tree, with the ancestor-only mask read from the tree plan.
//
// The key space of sequence b is [0, L[b] + N): positions below L[b] come
// from the cache, the rest are the tree nodes in BFS order.  It is cut into
// chunks of kChunk keys; one CTA handles one (sequence, query head, chunk),
// keeps an online softmax per tree node, and, when the sequence needs several
// chunks, publishes (m, l, unnormalised O) partials that the last CTA of the
// (sequence, head) to arrive merges (an arrival counter, no spin-wait).
#include "tr_internal.cuh"

namespace {

constexpr int kThreads = 256;
constexpr int kD = 128;       // head dimension
constexpr int kTile = 64;     // keys per tile
constexpr int kChunk = 1024;  // keys per CTA
constexpr int kKStride = kD + 1;

struct AttnArgs {
  const __nv_bfloat16 *Q, *Kt, *Vt, *Kc, *Vc;
  const int32_t *L;
  float *O;
  float *part_o;     // [B*Hq, CH, N, D]
  float2 *part_ml;   // [B*Hq, CH, N]
  unsigned *counters;  // [B*Hq]
  int cap, B, Hq, Hkv, CH;
  float scale;
  unsigned *status;
};

__device__ __forceinline__ float bf(const __nv_bfloat16 x) { return __bfloat162float(x); }

__global__ void __launch_bounds__(kThreads) attn_kernel(AttnArgs a, const __grid_constant__ TreeDev tree) {
  extern __shared__ float smem[];
  const int N = tree.N;
  float *Qs = smem;                          // [N][kD]
  float *Ks = Qs + TR_MAX_NODES * kD;        // [kTile][kKStride]
  float *Vs = Ks + kTile * kKStride;         // [kTile][kD]
  float *Ss = Vs + kTile * kD;               // [N][kTile]
  float *ms = Ss + TR_MAX_NODES * kTile;     // [N]
  float *ls = ms + TR_MAX_NODES;             // [N]
  float *cs = ls + TR_MAX_NODES;             // [N]
  __shared__ int is_last;

  const int c = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x;
  const int g = h / (a.Hq / a.Hkv);
  int Lb = a.L[b];
  if (Lb < 0 || Lb > a.cap) {
    if (tid == 0 && c == 0) tr_flag(a.status, TR_DEV_BAD_LENGTH);
    Lb = Lb < 0 ? 0 : a.cap;
  }
  const int total = Lb + N;
  const int nch = (total + kChunk - 1) / kChunk;
  if (c >= nch) return;
  const int k_lo = c * kChunk, k_hi = min(total, k_lo + kChunk);

  // queries of this head for every node
  for (int e = tid; e < N * kD; e += kThreads) {
    const int n = e / kD, i = e % kD;
    Qs[n * kD + i] = bf(a.Q[(((long long)b * N + n) * a.Hq + h) * kD + i]);
  }
  for (int n = tid; n < N; n += kThreads) {
    ms[n] = -INFINITY;
    ls[n] = 0.f;
  }
  // O accumulators: thread owns column i = tid % 128 of rows tid/128 + 2r
  const int oi = tid & (kD - 1), orow0 = tid >> 7;
  float acc[TR_MAX_NODES / 2];
#pragma unroll
  for (int r = 0; r < TR_MAX_NODES / 2; ++r) acc[r] = 0.f;
  __syncthreads();

  const long long cache_base = ((long long)b * a.Hkv + g) * a.cap;
  for (int t0 = k_lo; t0 < k_hi; t0 += kTile) {
    // stage K and V of keys [t0, t0 + kTile)
    for (int e = tid; e < kTile * kD; e += kThreads) {
      const int j = e / kD, i = e % kD;
      const int key = t0 + j;
      float kv = 0.f, vv = 0.f;
      if (key < k_hi) {
        if (key < Lb) {
          kv = bf(a.Kc[(cache_base + key) * kD + i]);
          vv = bf(a.Vc[(cache_base + key) * kD + i]);
        } else {
          const int node = key - Lb;
          kv = bf(a.Kt[(((long long)b * N + node) * a.Hkv + g) * kD + i]);
          vv = bf(a.Vt[(((long long)b * N + node) * a.Hkv + g) * kD + i]);
        }
      }
      Ks[j * kKStride + i] = kv;
      Vs[j * kD + i] = vv;
    }
    __syncthreads();
    // scores: thread owns key j = tid % 64 for rows tid/64 + 4r
    {
      const int j = tid & (kTile - 1), r0 = tid >> 6;
      const int key = t0 + j;
      float s[TR_MAX_NODES / 4];
#pragma unroll
      for (int r = 0; r < TR_MAX_NODES / 4; ++r) s[r] = 0.f;
      for (int i = 0; i < kD; ++i) {
        const float kk = Ks[j * kKStride + i];
#pragma unroll
        for (int r = 0; r < TR_MAX_NODES / 4; ++r) {
          const int n = r0 + 4 * r;
          if (n < N) s[r] = fmaf(Qs[n * kD + i], kk, s[r]);
        }
      }
#pragma unroll
      for (int r = 0; r < TR_MAX_NODES / 4; ++r) {
        const int n = r0 + 4 * r;
        if (n < N) {
          bool vis = key < k_hi;
          if (vis && key >= Lb) {
            const int node = key - Lb;
            vis = (tree.anc[n][node >> 6] >> (node & 63)) & 1ull;
          }
          Ss[n * kTile + j] = vis ? s[r] * a.scale : -INFINITY;
        }
      }
    }
    __syncthreads();
    // online softmax per row
    for (int n = tid; n < N; n += kThreads) {
      float mx = -INFINITY;
      for (int j = 0; j < kTile; ++j) mx = fmaxf(mx, Ss[n * kTile + j]);
      const float m_old = ms[n];
      const float m_new = fmaxf(m_old, mx);
      float corr = 1.f, sum = 0.f;
      if (m_new != -INFINITY) {
        corr = m_old == -INFINITY ? 0.f : expf(m_old - m_new);
        for (int j = 0; j < kTile; ++j) {
          const float sv = Ss[n * kTile + j];
          const float p = sv == -INFINITY ? 0.f : expf(sv - m_new);
          Ss[n * kTile + j] = p;
          sum += p;
        }
      } else {
        for (int j = 0; j < kTile; ++j) Ss[n * kTile + j] = 0.f;
      }
      ms[n] = m_new;
      ls[n] = ls[n] * corr + sum;
      cs[n] = corr;
    }
    __syncthreads();
#pragma unroll
    for (int r = 0; r < TR_MAX_NODES / 2; ++r) {
      const int n = orow0 + 2 * r;
      if (n < N) {
        float o = acc[r] * cs[n];
        for (int j = 0; j < kTile; ++j) o = fmaf(Ss[n * kTile + j], Vs[j * kD + oi], o);
        acc[r] = o;
      }
    }
    __syncthreads();
  }

  const long long bh = (long long)b * a.Hq + h;
  if (nch == 1) {
#pragma unroll
    for (int r = 0; r < TR_MAX_NODES / 2; ++r) {
      const int n = orow0 + 2 * r;
      if (n < N) a.O[(((long long)b * N + n) * a.Hq + h) * kD + oi] = acc[r] / ls[n];
    }
    return;
  }
  // publish the partial of this chunk
  float *po = a.part_o + (bh * a.CH + c) * (long long)N * kD;
#pragma unroll
  for (int r = 0; r < TR_MAX_NODES / 2; ++r) {
    const int n = orow0 + 2 * r;
    if (n < N) po[n * kD + oi] = acc[r];
  }
  for (int n = tid; n < N; n += kThreads) a.part_ml[(bh * a.CH + c) * N + n] = make_float2(ms[n], ls[n]);
  __threadfence();
  __syncthreads();
  if (tid == 0) is_last = atomicAdd(&a.counters[bh], 1u) == (unsigned)(nch - 1);
  __syncthreads();
  if (!is_last) return;
  __threadfence();
  // merge the chunks of this (sequence, head)
  for (int e = tid; e < N * kD; e += kThreads) {
    const int n = e / kD, i = e % kD;
    float M = -INFINITY;
    for (int q = 0; q < nch; ++q) M = fmaxf(M, __ldcg(&a.part_ml[(bh * a.CH + q) * N + n].x));
    float num = 0.f, den = 0.f;
    for (int q = 0; q < nch; ++q) {
      const float2 ml = __ldcg(&a.part_ml[(bh * a.CH + q) * N + n]);
      const float w = ml.x == -INFINITY ? 0.f : expf(ml.x - M);
      den += ml.y * w;
      num += __ldcg(&a.part_o[((bh * a.CH + q) * N + n) * (long long)kD + i]) * w;
    }
    a.O[(((long long)b * N + n) * a.Hq + h) * kD + i] = num / den;
  }
  if (tid == 0) a.counters[bh] = 0u;
}

constexpr size_t kSmemBytes =
    sizeof(float) * (TR_MAX_NODES * kD + kTile * kKStride + kTile * kD + TR_MAX_NODES * kTile + 3 * TR_MAX_NODES);

int max_chunks(int cap, int N) { return (cap + N + kChunk - 1) / kChunk; }

struct WsLayout {
  size_t o_off, ml_off, cnt_off, total;
};

WsLayout ws_layout(int B, int Hq, int cap, int N) {
  WsLayout w;
  const size_t CH = (size_t)max_chunks(cap, N);
  const size_t bh = (size_t)B * Hq;
  w.o_off = 0;
  w.ml_off = tr_align_up(bh * CH * N * kD * sizeof(float), 256);
  w.cnt_off = w.ml_off + tr_align_up(bh * CH * N * sizeof(float2), 256);
  w.total = w.cnt_off + tr_align_up(bh * sizeof(unsigned), 256);
  return w;
}

}  // namespace

extern "C" size_t tr_verify_attn_workspace_bytes(int B, int Hq, int Hkv, int d, int cap, const struct tr_tree *tree) {
  if (!tree || B < 1 || Hq < 1 || Hkv < 1 || d != kD || cap < 0) return 0;
  return ws_layout(B, Hq, cap, tree->dev.N).total;
}

extern "C" int tr_verify_attn(const void *Q, const void *Kt, const void *Vt, const void *Kc, const void *Vc,
                              const int32_t *L, int cap, int B, int Hq, int Hkv, int d, float scale,
                              const struct tr_tree *tree, float *O, void *ws, size_t ws_bytes, tr_stream_t stream) {
  if (!Q || !Kt || !Vt || !Kc || !Vc || !L || !tree || !O || B < 1 || Hq < 1 || Hkv < 1 || cap < 0) return TR_E_INVAL;
  if (Hq % Hkv) return TR_E_INVAL;
  if (d != kD) return TR_E_UNSUPPORTED;
  if (B > 65535 || Hq > 65535) return TR_E_UNSUPPORTED;
  const int N = tree->dev.N;
  const WsLayout w = ws_layout(B, Hq, cap, N);
  if (!ws || ws_bytes < w.total) return TR_E_INVAL;
  if (((uintptr_t)Q | (uintptr_t)Kt | (uintptr_t)Vt | (uintptr_t)Kc | (uintptr_t)Vc | (uintptr_t)O) & 15)
    return TR_E_INVAL;
  int rc = tr_check_device();
  if (rc != TR_OK) return rc;
  static bool attr_set[64];
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && !attr_set[dev]) {
    TR_TRY_CUDA(cudaFuncSetAttribute(attn_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes));
    attr_set[dev] = true;
  }
  AttnArgs a;
  a.Q = (const __nv_bfloat16 *)Q;
  a.Kt = (const __nv_bfloat16 *)Kt;
  a.Vt = (const __nv_bfloat16 *)Vt;
  a.Kc = (const __nv_bfloat16 *)Kc;
  a.Vc = (const __nv_bfloat16 *)Vc;
  a.L = L;
  a.O = O;
  a.part_o = (float *)((char *)ws + w.o_off);
  a.part_ml = (float2 *)((char *)ws + w.ml_off);
  a.counters = (unsigned *)((char *)ws + w.cnt_off);
  a.cap = cap;
  a.B = B;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.CH = max_chunks(cap, N);
  a.scale = scale;
  a.status = tr_status_dev();
  dim3 grid(a.CH, Hq, B);
  attn_kernel<<<grid, kThreads, kSmemBytes, (cudaStream_t)stream>>>(a, tree->dev);
  TR_LAUNCH_CHECK();
  return TR_OK;
}
