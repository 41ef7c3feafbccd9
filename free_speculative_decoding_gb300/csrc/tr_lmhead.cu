// Fused LM head + top-K on the 5th-generation tensor cores.
//
// logits = H . Wt^T (bf16 operands, fp32 accumulation) never reach HBM.  A
// persistent kernel (one CTA per SM) walks 128 x 256 output tiles; per CTA:
//   warp 0      TMA producer: 128x64 H and 256x64 Wt tiles, 128-byte swizzle,
//               a 4-stage shared-memory ring guarded by mbarriers;
//   warp 1      allocates 512 TMEM columns (two 128x256 fp32 accumulators) and
//               issues tcgen05.mma (M=128, N=256, K=16) per 16-wide K slice,
//               committing each stage back to the producer and each finished
//               tile to the epilogue; the warp runs its loop warp-uniformly
//               and one elected lane issues;
//   warps 2..5  epilogue: each thread owns one TMEM lane (one hidden row) and
//               streams the tile's 256 fp32 logits from TMEM into a register
//               top-K list, then writes that list (one per row and tile).  Per
//               32-column chunk each lane marks the columns that can enter its
//               list; a chunk with any such column is staged in shared memory
//               and every lane walks only its own marks, so a warp pays for
//               its busiest row's insertions instead of one insertion per
//               column for all 32 rows.  A first read of the tile sets each
//               list's floor to the smallest of KMAX column-group maxima.
// A second kernel merges each row's per-tile lists into the final top-K.  The
// two accumulators let the epilogue of tile i overlap the MMAs of tile i+1.
//
// Every mbarrier wait is bounded in time; a wait that gives up sets
// TR_DEV_TIMEOUT, raises a block-wide abort flag, drains the copies and MMAs
// already issued, frees TMEM and returns.
#include "tr_lists.cuh"
#include "tr_sm100.cuh"

namespace {

constexpr int BM = 128, BN = 256, BK = 64, STAGES = 4;
constexpr int A_BYTES = BM * BK * 2, B_BYTES = BN * BK * 2, STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int TMEM_COLS = 2 * BN;
constexpr int kThreads = 192;
constexpr int kStageFloats = 128 * 33;  // epilogue: 32 logits per row, padded
constexpr size_t kSmemBytes = (size_t)STAGES * STAGE_BYTES + 1024 + 256 + kStageFloats * 4;
constexpr uint32_t kIdesc = sm100::idesc_bf16_f32(BM, BN);

struct Bars {
  uint64_t full[STAGES], empty[STAGES], tfull[2], tempty[2], drain;
  uint32_t tmem;
  int abort;
};

template <int KMAX>
__global__ void __launch_bounds__(kThreads, 1)
    lmhead_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB, int rows,
                     long long V, int D, int n_mt, int n_nt, unsigned long long *part, unsigned *status,
                     unsigned long long wait_ns) {
  using namespace sm100;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  Bars *bars = (Bars *)(smem + STAGES * STAGE_BYTES);
  float *stage = (float *)(smem + STAGES * STAGE_BYTES + 256);
  volatile int *abort = &bars->abort;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_tiles = n_mt * n_nt;
  const int nkb = D / BK;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&bars->full[s], 1);
      mbar_init(&bars->empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&bars->tfull[a], 1);
      mbar_init(&bars->tempty[a], 128);
    }
    mbar_init(&bars->drain, 1);
    bars->abort = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
  }
  if (warp == 1) tmem_alloc(&bars->tmem, TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem;

  auto give_up = [&]() {
    if (!*abort) {
      *abort = 1;
      tr_flag(status, TR_DEV_TIMEOUT);
    }
  };

  if (warp == 0) {
    if (lane == 0) {
      int it = 0;
      uint32_t armed_phase[STAGES];
      bool armed[STAGES];
      for (int s = 0; s < STAGES; ++s) armed[s] = false;
      for (int t = blockIdx.x; t < n_tiles && !*abort; t += gridDim.x) {
        const int mt = t % n_mt, nt = t / n_mt;
        for (int kb = 0; kb < nkb; ++kb, ++it) {
          const int s = it % STAGES;
          const uint32_t ph = (it / STAGES) & 1;
          if (!mbar_wait(&bars->empty[s], ph ^ 1, abort, wait_ns)) {
            give_up();
            break;
          }
          mbar_arrive_expect_tx(&bars->full[s], STAGE_BYTES);
          tma_load_2d(smem + s * STAGE_BYTES, &tmA, &bars->full[s], kb * BK, mt * BM);
          tma_load_2d(smem + s * STAGE_BYTES + A_BYTES, &tmB, &bars->full[s], kb * BK, nt * BN);
          armed[s] = true;
          armed_phase[s] = ph;
        }
      }
      if (*abort) {
        // let the copies already issued land before the CTA can exit
        for (int s = 0; s < STAGES; ++s)
          if (armed[s]) mbar_drain(&bars->full[s], armed_phase[s]);
      }
    }
  } else if (warp == 1) {
    // The whole warp runs the loop, so control flow and operands stay
    // warp-uniform; one elected lane issues the MMAs and commits.
    auto wwait = [&](uint64_t *bar, uint32_t parity) -> bool {
      const bool all = __all_sync(0xffffffffu, mbar_wait(bar, parity, abort, wait_ns));
      if (!all && lane == 0) give_up();
      return all;
    };
    const uint64_t da0 = desc_kmajor_sw128(smem_u32(smem));
    int it = 0, tc = 0;
    for (int t = blockIdx.x; t < n_tiles; t += gridDim.x, ++tc) {
      const int acc = tc & 1;
      const uint32_t aph = (tc >> 1) & 1;
      if (!wwait(&bars->tempty[acc], aph ^ 1)) break;
      tc_fence_after();
      const uint32_t d = tmem + (uint32_t)(acc * BN);
      bool ok = true;
      for (int kb = 0; kb < nkb; ++kb, ++it) {
        const int s = it % STAGES;
        const uint32_t ph = (it / STAGES) & 1;
        if (!wwait(&bars->full[s], ph)) {
          ok = false;
          break;
        }
        tc_fence_after();
        if (elect_one()) {
          // descriptor start addresses count 16-byte units
          const uint64_t da = da0 + (uint64_t)(s * (STAGE_BYTES >> 4));
          const uint64_t db = da + (uint64_t)(A_BYTES >> 4);
#pragma unroll
          for (int k = 0; k < BK / 16; ++k)
            mma_bf16(d, da + (uint64_t)(k * 2), db + (uint64_t)(k * 2), kIdesc, (kb | k) != 0 ? 1u : 0u);
          mma_commit(&bars->empty[s]);
          if (kb == nkb - 1) mma_commit(&bars->tfull[acc]);
        }
        __syncwarp();
      }
      if (!ok) break;
    }
    // every MMA issued so far completes before TMEM can be released
    if (elect_one()) mma_commit(&bars->drain);
    __syncwarp();
    mbar_drain(&bars->drain, 0);
  } else {
    const int lane_base = (warp & 3) * 32;  // TMEM lanes this warp may read
    int tc = 0;
    for (int t = blockIdx.x; t < n_tiles; t += gridDim.x, ++tc) {
      const int mt = t % n_mt, nt = t / n_mt;
      const int acc = tc & 1;
      const uint32_t aph = (tc >> 1) & 1;
      if (!mbar_wait(&bars->tfull[acc], aph, abort, wait_ns)) {
        give_up();
        break;
      }
      tc_fence_after();
      TopList<KMAX> L;
      L.init();
      const uint32_t taddr = tmem + ((uint32_t)lane_base << 16) + (uint32_t)(acc * BN);
      const long long col0 = (long long)nt * BN;
      float *mine = stage + (threadIdx.x - 64) * 33;  // this row's 32 staged logits (stride 33: no bank conflicts)
      {
        // a first read of the tile: the smallest of KMAX group maxima is
        // reached by KMAX elements of this row, so nothing below it can enter
        constexpr int GW = BN / KMAX;  // columns per group
        float fl = INFINITY;
#pragma unroll 1
        for (int c0 = 0; c0 < BN; c0 += 32) {
          float v[32];
          tmem_ld32(taddr + c0, v);
          const int n_in = (int)min((long long)32, V - (col0 + c0));
#pragma unroll
          for (int g = 0; g < 32 / GW; ++g) {
            float gm = -INFINITY;
#pragma unroll
            for (int j = g * GW; j < (g + 1) * GW; ++j) gm = j < n_in ? fmaxf(gm, v[j]) : gm;
            fl = fminf(fl, gm);
          }
        }
        L.raise_floor(fl);
      }
#pragma unroll 1
      for (int c0 = 0; c0 < BN; c0 += 32) {
        float v[32];
        tmem_ld32(taddr + c0, v);
        // columns that can enter this row's list (none past the vocabulary)
        const int n_in = (int)min((long long)32, V - (col0 + c0));
        uint32_t m = 0;
#pragma unroll
        for (int j = 0; j < 32; ++j) m |= (uint32_t)(j < n_in && v[j] >= L.thr) << j;
        if (__any_sync(0xffffffffu, m != 0u)) {
          // each lane walks only its own candidates, so the warp's cost is the
          // busiest row's candidate count rather than every column
#pragma unroll
          for (int j = 0; j < 32; ++j) mine[j] = v[j];  // lane-private: no barrier needed
          while (m) {
            const int j = __ffs(m) - 1;
            m &= m - 1;
            L.push(mine[j], (uint32_t)(col0 + c0 + j));
          }
        }
      }
      tc_fence_before();
      mbar_arrive(&bars->tempty[acc]);
      const int row = mt * BM + lane_base + lane;
      if (row < rows) {
        unsigned long long *dst = part + ((long long)row * n_nt + nt) * KMAX;
#pragma unroll
        for (int j = 0; j < KMAX; ++j) dst[j] = L.k[j];
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

// Final merge: one warp per row reduces n_lists lists of KMAX keys.  A lane
// takes every 32nd list; each list arrives with 16-byte loads issued before
// any key is used, and since a list is sorted, its first key that cannot
// enter ends it.
template <int KMAX>
__global__ void __launch_bounds__(128) merge_lists_kernel(const unsigned long long *part, long long rows, int n_lists,
                                                          int K, int32_t *ids, float *vals) {
  const long long row = (long long)blockIdx.x * 4 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;
  TopList<KMAX> L;
  L.init();
  constexpr int kLists = KMAX <= 8 ? 4 : (KMAX <= 16 ? 2 : 1);  // lists a lane holds in registers at once
  for (int t0 = lane; t0 < n_lists; t0 += 32 * kLists) {
    ulonglong2 buf[kLists][KMAX / 2];
#pragma unroll
    for (int q = 0; q < kLists; ++q) {
      const int t = t0 + 32 * q;
      const ulonglong2 *src = reinterpret_cast<const ulonglong2 *>(part + (row * n_lists + t) * KMAX);
#pragma unroll
      for (int j = 0; j < KMAX / 2; ++j) buf[q][j] = t < n_lists ? __ldcs(src + j) : make_ulonglong2(0ull, 0ull);
    }
#pragma unroll
    for (int q = 0; q < kLists; ++q)
#pragma unroll
      for (int j = 0; j < KMAX / 2; ++j) {
        if (buf[q][j].x <= L.k[KMAX - 1]) break;  // sorted: nothing further in this list enters
        list_insert<KMAX>(L.k, buf[q][j].x);
        if (buf[q][j].y <= L.k[KMAX - 1]) break;
        list_insert<KMAX>(L.k, buf[q][j].y);
      }
  }
  const unsigned long long mine = warp_merge<KMAX>(L, lane);
  if (lane < K) {
    ids[row * K + lane] = mine ? (int32_t)tr_key_id(mine) : -1;
    if (vals) vals[row * K + lane] = mine ? tr_key_val(mine) : -INFINITY;
  }
}

int n_ntiles(long long V) { return (int)((V + BN - 1) / BN); }

template <int KMAX>
int launch(const CUtensorMap &ta, const CUtensorMap &tb, long long rows, int D, long long V, int K, int32_t *ids,
           float *vals, unsigned long long *part, cudaStream_t s) {
  static bool attr_set[64];
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && !attr_set[dev]) {
    if (cudaFuncSetAttribute(lmhead_tc_kernel<KMAX>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes) !=
        cudaSuccess)
      return TR_E_CUDA;
    attr_set[dev] = true;
  }
  const int n_mt = (int)((rows + BM - 1) / BM), n_nt = n_ntiles(V);
  const int tiles = n_mt * n_nt;
  const int grid = tiles < tr_sm_count() ? tiles : tr_sm_count();
  lmhead_tc_kernel<KMAX><<<grid, kThreads, kSmemBytes, s>>>(ta, tb, (int)rows, V, D, n_mt, n_nt, part,
                                                            tr_status_dev(), tr_wait_limit_ns());
  merge_lists_kernel<KMAX><<<(unsigned)((rows + 3) / 4), 128, 0, s>>>(part, rows, n_nt, K, ids, vals);
  return TR_OK;
}

}  // namespace

extern "C" size_t tr_lmhead_topk_workspace_bytes(int64_t rows, int D, int64_t V, int K) {
  if (rows <= 0 || D <= 0 || V <= 0 || K < 1 || K > TR_MAX_K) return 0;
  return tr_align_up((size_t)rows * n_ntiles(V) * tr_kmax(K) * 8, 256);
}

extern "C" int tr_lmhead_topk(const void *H, const void *Wt, int64_t rows, int D, int64_t V, int K, int32_t *ids,
                              float *vals, void *ws, size_t ws_bytes, tr_stream_t stream) {
  if (rows < 0 || D < 1 || V < 1 || K < 1 || K > TR_MAX_K || K > V) return TR_E_INVAL;
  if (D % BK) return TR_E_UNSUPPORTED;
  if (V > INT32_MAX || rows > INT32_MAX / 2) return TR_E_UNSUPPORTED;
  if (rows == 0) return TR_OK;
  if (!H || !Wt || !ids) return TR_E_INVAL;
  if (((uintptr_t)H | (uintptr_t)Wt) & 15) return TR_E_INVAL;
  if (!ws || ws_bytes < tr_lmhead_topk_workspace_bytes(rows, D, V, K)) return TR_E_INVAL;
  int rc = tr_check_device();
  if (rc != TR_OK) return rc;
  CUtensorMap ta, tb;
  rc = tr_make_tmap_2d_bf16(&ta, H, (uint64_t)D, (uint64_t)rows, (uint64_t)D * 2, BK, BM);
  if (rc != TR_OK) return rc;
  rc = tr_make_tmap_2d_bf16(&tb, Wt, (uint64_t)D, (uint64_t)V, (uint64_t)D * 2, BK, BN);
  if (rc != TR_OK) return rc;
  cudaStream_t s = (cudaStream_t)stream;
  const int km = tr_kmax(K);
  auto part = (unsigned long long *)ws;
  if (km == 8) rc = launch<8>(ta, tb, rows, D, V, K, ids, vals, part, s);
  else if (km == 16) rc = launch<16>(ta, tb, rows, D, V, K, ids, vals, part, s);
  else rc = launch<32>(ta, tb, rows, D, V, K, ids, vals, part, s);
  if (rc != TR_OK) return rc;
  TR_LAUNCH_CHECK();
  return TR_OK;
}
