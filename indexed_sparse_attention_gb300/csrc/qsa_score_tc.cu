// Step 2 for many query rows (chunked prefill): block scoring as one dense
// contraction on the 5th-generation tensor cores (hipfire, "QSA sparse
// attention and the VMM KV backend", section 03: the wide scoring variant for
// prefill; section 02 for the score itself).
//
// For one sequence with R rows, the logits of index head h of row r against
// block b form the product of A = the index queries as an (4R x 128) bf16
// matrix (m = 4r + h) and the pooled keys.  The pooled keys are fp32; they are
// split once per call into three bf16 planes hi + mid + lo that sum to them
// exactly (each residual is the exact rounding error of the previous plane),
// laid out as one (blocks x 384) bf16 matrix B = [hi | mid | lo].  Against
// A' = [Q | Q | Q] (the same query tile reused for each plane) one product
// with K = 384 gives sum_c q_c (hi_c + mid_c + lo_c) = q . k exactly up to fp32
// accumulation: bf16 x bf16 products are exact in fp32.
//
// score_tc_kernel: persistent, one CTA per SM; CTA c takes a contiguous run of
// output tiles (128 row-heads = 32 rows x 128 blocks), block tile major, so
// one tile of key planes (128 blocks x 384 = 96 KB) stays in shared memory
// while the query tiles (32 KB) stream past it.
//   warp 0, lane 0  loads the key-plane tile (six 64-wide K slices) when the
//                   block tile changes, and each output tile's query tile as
//                   two 64-channel boxes through a 4-box ring, with 2-D
//                   tensor copies (128-byte swizzle);
//   warp 1          allocates 256 TMEM columns (two fp32 accumulators of
//                   128 columns); lane 0 issues tcgen05.mma (kind::f16,
//                   M = 128, N = 128, K = 16) into the accumulator the
//                   epilogue has released -- K slice kc pairs query half
//                   kc % 2 with key plane kc / 2 -- and commits the query
//                   boxes and, at a block-tile change, the key tile back to
//                   the producer, and each finished accumulator to the
//                   epilogue;
//   warps 2..9      read an accumulator with tcgen05.ld (warp w reads TMEM
//                   lanes 32 (w % 4) .., columns 64 ((w - 2) / 4) ..), release
//                   it, apply ReLU per head,
//                   add the four heads of a row across lanes, scale, mask
//                   blocks the row cannot see, and write the scores and group
//                   maxima -- while the MMAs of the next tile run.
// Tiles whose blocks no row of the tile can see are skipped by every role.
// Every wait on an mbarrier gives up after about two seconds instead of
// hanging (counted in a device counter).
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "qsa_tc.cuh"

namespace qsa {

namespace {

constexpr float kScale = 0.08838834764831845f;   // 1/sqrt(128)
constexpr int kTcM = 128;                        // row-heads per tile (32 rows)
constexpr int kTcN = 128;                        // blocks per tile
constexpr int kTcK = 64;                         // bf16 per 128-byte swizzled row
constexpr int kPlanesK = 3 * QSA_INDEX_DIM;      // 384
constexpr int kKSlices = kPlanesK / kTcK;        // 6
constexpr int kABoxes = 4;                       // query-box ring (two per output tile)
constexpr int kSliceBytes = kTcN * kTcK * 2;     // 16 KB of B per slice
constexpr int kBBytes = kKSlices * kSliceBytes;  // 96 KB key-plane tile
constexpr int kABoxBytes = kTcM * kTcK * 2;      // 16 KB: 128 row-heads x 64 channels
constexpr size_t kTcSmem = (size_t)kBBytes + (size_t)kABoxes * kABoxBytes + 1024;
constexpr int kEpiWarps = 8;                     // two per TMEM lane quarter, each half the columns
constexpr int kTcThreads = 64 + 32 * kEpiWarps;
constexpr int kEpiThreads = 32 * kEpiWarps;

__device__ int g_tc_wait_timeouts;

using namespace tc;

__device__ __forceinline__ bool wait_bar(uint64_t* b, uint32_t parity) {
  return bar_wait(b, parity, &g_tc_wait_timeouts);
}

// Both operands K-major with the 128-byte swizzle: 8-row groups 1,024 bytes apart.
__device__ __forceinline__ uint64_t umma_desc(const void* p) { return desc_sw128(p, 16, 1024); }

constexpr uint32_t kIdesc = idesc_bf16(kTcM, kTcN, false, false);

// ------------------------------------------------------------------ key planes
// planes[b][p * 128 + c], p = 0, 1, 2: bf16 hi, mid, lo of pooled[b][c].
__global__ void split_planes_kernel(const float* __restrict__ pooled, int64_t pstride, int64_t n_blocks,
                                    __nv_bfloat16* __restrict__ planes) {
  grid_dependency_sync();
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;   // (block, 4-channel group)
  if (i >= n_blocks * (QSA_INDEX_DIM / 4)) return;
  const int64_t b = i / (QSA_INDEX_DIM / 4);
  const int c = (int)(i % (QSA_INDEX_DIM / 4)) * 4;
  const float4 x = *reinterpret_cast<const float4*>(pooled + b * pstride + c);
  const float v[4] = {x.x, x.y, x.z, x.w};
  __nv_bfloat16 h[4], m[4], l[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    h[j] = __float2bfloat16_rn(v[j]);
    const float r1 = v[j] - __bfloat162float(h[j]);
    m[j] = __float2bfloat16_rn(r1);
    l[j] = __float2bfloat16_rn(r1 - __bfloat162float(m[j]));
  }
  __nv_bfloat16* row = planes + b * kPlanesK + c;
  *reinterpret_cast<uint2*>(row) = *reinterpret_cast<const uint2*>(h);
  *reinterpret_cast<uint2*>(row + QSA_INDEX_DIM) = *reinterpret_cast<const uint2*>(m);
  *reinterpret_cast<uint2*>(row + 2 * QSA_INDEX_DIM) = *reinterpret_cast<const uint2*>(l);
}

// ------------------------------------------------------------------ scoring
struct ScoreTcParams {
  CUtensorMap tmap_q;       // index queries of the sequence: [4 R, 128] bf16
  CUtensorMap tmap_k;       // key planes: [blocks, 384] bf16
  float* scores;
  int64_t ld;
  float* gmax;
  int64_t gld;
  int64_t n_tokens;
  int64_t block_lo;         // absolute id of the first block scored (column 0 of scores)
  int64_t n_blocks;         // blocks scored: block_lo .. block_lo + n_blocks - 1
  int32_t n_rows;
  int32_t row_begin;
};

struct TcTile {
  int m0, n0;
  bool live;   // some row of the tile sees some of its blocks
};

__device__ __forceinline__ TcTile tc_tile(const ScoreTcParams& P, int n_tiles_m, int t) {
  TcTile x;
  x.n0 = (t / n_tiles_m) * kTcN;
  x.m0 = (t % n_tiles_m) * kTcM;
  const int r_last = min(P.n_rows - 1, x.m0 / 4 + kTcM / 4 - 1);
  x.live = P.block_lo + x.n0 < visible_blocks(row_position(P.n_tokens, P.n_rows, r_last));
  return x;
}

__global__ void __launch_bounds__(kTcThreads, 1) score_tc_kernel(const __grid_constant__ ScoreTcParams P) {
  extern __shared__ uint8_t tc_raw[];
  __shared__ uint64_t b_full, b_empty, a_full[kABoxes], a_empty[kABoxes], acc_full[2], acc_empty[2];
  __shared__ uint32_t tmem_slot;
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(tc_raw) + 1023) & ~(uintptr_t)1023);
  uint8_t* smB = base;              // six boxes [128 blocks][64 of K]
  uint8_t* smA = base + kBBytes;    // kABoxes boxes [128 row-heads][64 channels]
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int n_tiles_m = (int)(((int64_t)P.n_rows * 4 + kTcM - 1) / kTcM);
  const int n_tiles = n_tiles_m * (int)((P.n_blocks + kTcN - 1) / kTcN);
  const int t0 = (int)((int64_t)n_tiles * blockIdx.x / gridDim.x);
  const int t1 = (int)((int64_t)n_tiles * (blockIdx.x + 1) / gridDim.x);

  if (tid == 0) {
    bar_init(&b_full, 1);
    bar_init(&b_empty, 1);
    for (int i = 0; i < kABoxes; ++i) {
      bar_init(&a_full[i], 1);
      bar_init(&a_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      bar_init(&acc_full[i], 1);
      bar_init(&acc_empty[i], kEpiThreads);
    }
    bar_init_fence();
  }
  if (warp == 1) {
    tmem_alloc(&tmem_slot, 2 * kTcN);
  }
  fence_before();
  __syncthreads();
  fence_after();
  const uint32_t tmem = tmem_slot;
  grid_dependency_sync();

  if (warp == 0) {
    if (lane == 0) {
      int b_loads = 0, boxes = 0, n_prev = -1;
      bool ok = true;
      for (int t = t0; t < t1 && ok; ++t) {
        const TcTile x = tc_tile(P, n_tiles_m, t);
        if (!x.live) continue;
        if (x.n0 != n_prev) {   // a new key-plane tile, once the MMAs are done with the last
          if (b_loads >= 1 && !(ok = wait_bar(&b_empty, (uint32_t)((b_loads - 1) & 1)))) break;
          bar_expect_tx(&b_full, kBBytes);
          for (int kc = 0; kc < kKSlices; ++kc) tma_2d(smB + kc * kSliceBytes, &P.tmap_k, kc * kTcK, x.n0, &b_full);
          ++b_loads;
          n_prev = x.n0;
        }
        for (int h = 0; h < 2; ++h, ++boxes) {
          const int q = boxes % kABoxes;
          if (boxes >= kABoxes && !(ok = wait_bar(&a_empty[q], (uint32_t)((boxes / kABoxes - 1) & 1)))) break;
          bar_expect_tx(&a_full[q], kABoxBytes);
          tma_2d(smA + q * kABoxBytes, &P.tmap_q, h * kTcK, x.m0, &a_full[q]);
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      int b_loads = 0, boxes = 0, tiles = 0, n_prev = -1;
      bool ok = true;
      for (int t = t0; t < t1 && ok; ++t) {
        const TcTile x = tc_tile(P, n_tiles_m, t);
        if (!x.live) continue;
        if (x.n0 != n_prev) {
          if (b_loads > 0) commit(&b_empty);   // the previous key tile is done once these MMAs finish
          if (!(ok = wait_bar(&b_full, (uint32_t)(b_loads & 1)))) break;
          ++b_loads;
          n_prev = x.n0;
        }
        const int acc = tiles & 1;
        if (tiles >= 2 && !(ok = wait_bar(&acc_empty[acc], (uint32_t)((tiles / 2 - 1) & 1)))) break;
        const int q0 = boxes % kABoxes, q1 = (boxes + 1) % kABoxes;
        if (!(ok = wait_bar(&a_full[q0], (uint32_t)((boxes / kABoxes) & 1)))) break;
        if (!(ok = wait_bar(&a_full[q1], (uint32_t)(((boxes + 1) / kABoxes) & 1)))) break;
        fence_after();
        const uint32_t d = tmem + (uint32_t)(acc * kTcN);
        for (int kc = 0; kc < kKSlices; ++kc) {
          // Slice kc is plane kc / 2, channels 64 (kc % 2) ..: the query half kc % 2.
          const uint8_t* a = smA + ((kc % 2) ? q1 : q0) * kABoxBytes;
          const uint8_t* b = smB + kc * kSliceBytes;
#pragma unroll
          for (int j = 0; j < kTcK / 16; ++j)
            mma_bf16(d, umma_desc(a + 32 * j), umma_desc(b + 32 * j), kIdesc, (kc | j) != 0 ? 1u : 0u);
        }
        commit(&a_empty[q0]);
        commit(&a_empty[q1]);
        commit(&acc_full[acc]);
        boxes += 2;
        ++tiles;
      }
    }
  } else {
    // Epilogue: TMEM lanes 32 (warp % 4) .. +31 = row-heads m of the tile.
    const int quarter = warp & 3;
    constexpr int kColGroups = kEpiWarps / 4;
    constexpr int kGroupCols = kTcN / kColGroups;
    const int cgrp = (warp - 2) / 4;   // columns [kGroupCols cgrp, + kGroupCols)
    const int m = quarter * 32 + lane;
    int tiles = 0;
    for (int t = t0; t < t1; ++t) {
      const TcTile x = tc_tile(P, n_tiles_m, t);
      if (!x.live) continue;
      const int acc = tiles & 1;
      if (!wait_bar(&acc_full[acc], (uint32_t)((tiles / 2) & 1))) break;
      fence_after();
      const int r = x.m0 / 4 + m / 4;   // row within the sequence
      const bool row_ok = r < P.n_rows;
      // Blocks of this launch's range the row can see (column index limit).
      const int64_t nb =
          row_ok ? min(P.n_blocks, visible_blocks(row_position(P.n_tokens, P.n_rows, r)) - P.block_lo) : 0;
      constexpr int kChunks = kGroupCols / 32;
      float v[kChunks][32];
#pragma unroll
      for (int c = 0; c < kChunks; ++c)
        tmem_ld32(tmem + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(acc * kTcN + kGroupCols * cgrp + 32 * c), v[c]);
      // The accumulator is in registers: the MMAs of a later tile may reuse it.
      fence_before();
      bar_arrive(&acc_empty[acc]);
#pragma unroll
      for (int c = 0; c < kChunks; ++c) {
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          float y = fmaxf(v[c][i], 0.f);
          y += __shfl_xor_sync(0xffffffffu, y, 1);
          y += __shfl_xor_sync(0xffffffffu, y, 2);
          v[c][i] = y * kScale;
        }
        if ((lane & 3) == 0 && row_ok) {
          const int64_t b0 = x.n0 + kGroupCols * cgrp + 32 * c;
          float* dst = P.scores + (int64_t)(P.row_begin + r) * P.ld + b0;
          if (b0 + 32 <= nb) {
#pragma unroll
            for (int i = 0; i < 32; i += 4)
              *reinterpret_cast<float4*>(dst + i) = make_float4(v[c][i], v[c][i + 1], v[c][i + 2], v[c][i + 3]);
          } else {
#pragma unroll
            for (int i = 0; i < 32; ++i)
              if (b0 + i < nb) dst[i] = v[c][i];
          }
          if (P.gmax) {
#pragma unroll
            for (int g = 0; g < 2; ++g) {
              if (b0 + 16 * g >= nb) continue;
              float mx = -INFINITY;
#pragma unroll
              for (int i = 0; i < 16; ++i)
                if (b0 + 16 * g + i < nb) mx = fmaxf(mx, v[c][16 * g + i]);
              P.gmax[(int64_t)(P.row_begin + r) * P.gld + b0 / 16 + g] = mx;
            }
          }
        }
      }
      ++tiles;
    }
  }
  fence_before();
  __syncthreads();
  if (warp == 1) {
    fence_after();
    tmem_dealloc(tmem, 2 * kTcN);
  }
}

PFN_cuTensorMapEncodeTiled_v12000 encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  return fn;
}

bool encode_bf16_2d(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer, uint64_t row_bytes,
                    uint32_t box_inner, uint32_t box_outer) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = encoder();
  if (!enc) return false;
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {row_bytes};
  const cuuint32_t box[2] = {box_inner, box_outer};
  const cuuint32_t elem[2] = {1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, elem,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

size_t score_tc_workspace_bytes(int64_t n_blocks) {
  return n_blocks > 0 ? (size_t)n_blocks * kPlanesK * 2 : 0;
}

cudaError_t launch_score_tc(const void* q_idx, int32_t row_begin, int32_t n_rows, int64_t n_tokens,
                            const float* pooled, int64_t pooled_stride, int64_t block_lo, int64_t n_blocks,
                            float* scores, int64_t ld, float* gmax, int64_t gld, void* workspace, cudaStream_t st) {
  const int64_t nb = n_blocks;
  if (nb <= 0 || n_rows <= 0) return cudaSuccess;
  __nv_bfloat16* planes = static_cast<__nv_bfloat16*>(workspace);
  const int64_t threads = nb * (QSA_INDEX_DIM / 4);
  cudaError_t e = launch_kernel(split_planes_kernel, dim3((unsigned)((threads + 255) / 256)), dim3(256), 0, st, 0u,
                                pooled + block_lo * pooled_stride, pooled_stride, nb, planes);
  if (e != cudaSuccess) return e;
  ScoreTcParams P;
  memset(&P, 0, sizeof(P));
  const __nv_bfloat16* q = static_cast<const __nv_bfloat16*>(q_idx) + (int64_t)row_begin * QSA_INDEX_HEADS * QSA_INDEX_DIM;
  if (!encode_bf16_2d(&P.tmap_q, q, QSA_INDEX_DIM, (uint64_t)n_rows * QSA_INDEX_HEADS, QSA_INDEX_DIM * 2, kTcK, kTcM) ||
      !encode_bf16_2d(&P.tmap_k, planes, kPlanesK, (uint64_t)nb, kPlanesK * 2, kTcK, kTcN))
    return cudaErrorNotSupported;
  P.scores = scores;
  P.ld = ld;
  P.gmax = gmax;
  P.gld = gld;
  P.n_tokens = n_tokens;
  P.block_lo = block_lo;
  P.n_blocks = n_blocks;
  P.n_rows = n_rows;
  P.row_begin = row_begin;
  if ((e = allow_dynamic_smem((const void*)score_tc_kernel, kTcSmem)) != cudaSuccess) return e;
  const int64_t tiles = ((nb + kTcN - 1) / kTcN) * (((int64_t)n_rows * 4 + kTcM - 1) / kTcM);
  const int sms = device_sm_count();
  const unsigned grid = (unsigned)(tiles < sms ? tiles : sms);
  return launch_kernel(score_tc_kernel, dim3(grid), dim3(kTcThreads), kTcSmem, st, 0u, P);
}

int score_tc_wait_timeouts() {
  int v = 0;
  return cudaMemcpyFromSymbol(&v, g_tc_wait_timeouts, sizeof(int)) == cudaSuccess ? v : -1;
}

}  // namespace qsa
