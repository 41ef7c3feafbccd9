// Fused LM head + top-K: logits = H . Wt^T never reach HBM; each
// (row block, vocabulary tile) keeps only its rows' top-K keys, and a merge
// kernel reduces the tiles' lists to the final top-K per row.
#include "tr_internal.cuh"
#include "tr_lists.cuh"

namespace {

constexpr int kThreads = 256;
constexpr int kBM = 64;    // rows per tile
constexpr int kBN = 128;   // vocabulary columns per tile
constexpr int kBK = 32;    // reduction step

// One 64 x 128 output tile on CUDA cores, fp32 accumulation of bf16 products,
// followed by a per-row top-K of the tile written as KMAX keys per row.
template <int KMAX>
__global__ void __launch_bounds__(kThreads) lmhead_tile_kernel(const __nv_bfloat16 *H, const __nv_bfloat16 *Wt,
                                                               long long rows, int D, long long V,
                                                               unsigned long long *part, int n_vt) {
  // operand tiles during the reduction, the output tile afterwards
  constexpr int kOperands = kBK * (kBM + 1) + kBK * (kBN + 1);
  constexpr int kOut = kBM * (kBN + 1);
  __shared__ float buf[kOperands > kOut ? kOperands : kOut];
  float (*Hs)[kBM + 1] = reinterpret_cast<float (*)[kBM + 1]>(buf);
  float (*Ws)[kBN + 1] = reinterpret_cast<float (*)[kBN + 1]>(buf + kBK * (kBM + 1));
  float (*Cs)[kBN + 1] = reinterpret_cast<float (*)[kBN + 1]>(buf);
  const int tid = threadIdx.x;
  const long long r0 = (long long)blockIdx.y * kBM;
  const long long v0 = (long long)blockIdx.x * kBN;
  // thread computes rows tr*4..+3 and columns tc + 16*j, j < 8
  const int tr = tid >> 4, tc = tid & 15;
  float acc[4][8];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[i][j] = 0.f;
  for (int k0 = 0; k0 < D; k0 += kBK) {
    for (int e = tid; e < kBM * kBK; e += kThreads) {
      const int r = e / kBK, k = e % kBK;
      const long long gr = r0 + r;
      Hs[k][r] = gr < rows ? __bfloat162float(H[gr * D + k0 + k]) : 0.f;
    }
    for (int e = tid; e < kBN * kBK; e += kThreads) {
      const int v = e / kBK, k = e % kBK;
      const long long gv = v0 + v;
      Ws[k][v] = gv < V ? __bfloat162float(Wt[gv * D + k0 + k]) : 0.f;
    }
    __syncthreads();
#pragma unroll 8
    for (int k = 0; k < kBK; ++k) {
      float hv[4], wv[8];
#pragma unroll
      for (int i = 0; i < 4; ++i) hv[i] = Hs[k][tr * 4 + i];
#pragma unroll
      for (int j = 0; j < 8; ++j) wv[j] = Ws[k][tc + 16 * j];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[i][j] = fmaf(hv[i], wv[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 8; ++j) Cs[tr * 4 + i][tc + 16 * j] = acc[i][j];
  __syncthreads();
  // per-row top-K of the tile: warp w takes rows w, w+8, ...
  const int warp = tid >> 5, lane = tid & 31;
  for (int r = warp; r < kBM; r += kThreads / 32) {
    const long long gr = r0 + r;
    if (gr >= rows) break;
    TopList<KMAX> L;
    L.init();
    for (int c = lane; c < kBN; c += 32) {
      const long long gv = v0 + c;
      if (gv < V) L.push(Cs[r][c], (uint32_t)gv);
    }
    const unsigned long long mine = warp_merge<KMAX>(L, lane);
    if (lane < KMAX) part[(gr * n_vt + blockIdx.x) * KMAX + lane] = mine;
  }
}

// Final merge: one warp per row reduces n_vt lists of KMAX keys.
template <int KMAX>
__global__ void __launch_bounds__(128) merge_lists_kernel(const unsigned long long *part, long long rows, int n_lists,
                                                          int K, int32_t *ids, float *vals) {
  const long long row = (long long)blockIdx.x * 4 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;
  TopList<KMAX> L;
  L.init();
  for (int t = lane; t < n_lists; t += 32) {
    const unsigned long long *src = part + (row * n_lists + t) * KMAX;
    for (int j = 0; j < KMAX; ++j) {
      const unsigned long long key = src[j];
      if (key == 0ull) break;
      list_insert<KMAX>(L.k, key);
    }
  }
  const unsigned long long mine = warp_merge<KMAX>(L, lane);
  if (lane < K) {
    ids[row * K + lane] = mine ? (int32_t)tr_key_id(mine) : -1;
    if (vals) vals[row * K + lane] = mine ? tr_key_val(mine) : -INFINITY;
  }
}

int n_vtiles(long long V) { return (int)((V + kBN - 1) / kBN); }

template <int KMAX>
void launch(const __nv_bfloat16 *H, const __nv_bfloat16 *Wt, long long rows, int D, long long V, int K, int32_t *ids,
            float *vals, unsigned long long *part, cudaStream_t s) {
  const int nvt = n_vtiles(V);
  dim3 grid(nvt, (unsigned)((rows + kBM - 1) / kBM));
  lmhead_tile_kernel<KMAX><<<grid, kThreads, 0, s>>>(H, Wt, rows, D, V, part, nvt);
  merge_lists_kernel<KMAX><<<(unsigned)((rows + 3) / 4), 128, 0, s>>>(part, rows, nvt, K, ids, vals);
}

}  // namespace

extern "C" size_t tr_lmhead_topk_workspace_bytes(int64_t rows, int D, int64_t V, int K) {
  if (rows <= 0 || D <= 0 || V <= 0 || K < 1 || K > TR_MAX_K) return 0;
  return tr_align_up((size_t)rows * n_vtiles(V) * tr_kmax(K) * 8, 256);
}

extern "C" int tr_lmhead_topk(const void *H, const void *Wt, int64_t rows, int D, int64_t V, int K, int32_t *ids,
                              float *vals, void *ws, size_t ws_bytes, tr_stream_t stream) {
  if (rows < 0 || D < 1 || V < 1 || K < 1 || K > TR_MAX_K || K > V) return TR_E_INVAL;
  if (D % 64) return TR_E_UNSUPPORTED;
  if (V > INT32_MAX || rows > 65535LL * kBM) return TR_E_UNSUPPORTED;
  if (rows == 0) return TR_OK;
  if (!H || !Wt || !ids) return TR_E_INVAL;
  if (!ws || ws_bytes < tr_lmhead_topk_workspace_bytes(rows, D, V, K)) return TR_E_INVAL;
  int rc = tr_check_device();
  if (rc != TR_OK) return rc;
  cudaStream_t s = (cudaStream_t)stream;
  const int km = tr_kmax(K);
  auto h = (const __nv_bfloat16 *)H;
  auto w = (const __nv_bfloat16 *)Wt;
  auto part = (unsigned long long *)ws;
  if (km == 8) launch<8>(h, w, rows, D, V, K, ids, vals, part, s);
  else if (km == 16) launch<16>(h, w, rows, D, V, K, ids, vals, part, s);
  else launch<32>(h, w, rows, D, V, K, ids, vals, part, s);
  TR_LAUNCH_CHECK();
  return TR_OK;
}
