// Steps 1 and 2 of the QSA layer step: pooling index keys into block keys and
// scoring the pooled blocks (hipfire, "QSA sparse attention and the VMM KV
// backend", section 02 "How QSA chooses what to read"; section 03 names a
// few-row scoring variant for decode/verify and a wide one for prefill).
//
// Scoring is a streaming pass over the pooled keys: every 512-byte pooled
// block is read once per row-group of <= 8 query rows.  For bf16 index
// queries the dot products run on the tensor pipe with fp32 accumulation,
// and the fp32 pooled key is split so that no product loses precision:
//  - decode and verify (<= 8 rows on the TMA-ring and direct-load kernels,
//    <= 4 rows on the warp-level kernel): tf32 MMAs (m16n8k8) on two
//    planes, hi = the key rounded to tf32 and lo = key - hi (exact; the MMA
//    keeps at least its top 11 bits, so hi + lo is the key to within one
//    fp32 ulp); 3 integer/fp32 ops per key element;
//  - wider groups (prefill): bf16 MMAs (m16n8k16) on three planes hi + mid +
//    lo that sum to the key exactly.
// bf16 queries are exact in both formats.  Every tile of 16 blocks is one
// group of the group maxima the selection starts from.  fp32 index queries
// take a CUDA-core kernel.
//
// Steps 1 and 2 in one call (qsa_pool_score_blocks): on the few-row path the
// scoring launch pools the blocks the step's rows complete -- the consumer
// warp whose tile holds such a block averages the block's four index keys
// (the pooling kernel's order of operations), overwrites that row of the
// landed tile and stores it to the pooled keys -- so the step has no pooling
// launch; the other kernels get a pooling launch before them.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "qsa_internal.cuh"
#include "qsa_tc.cuh"

namespace qsa {

namespace {

constexpr float kScoreScale = 0.08838834764831845f;  // 1/sqrt(128)

// bf16x2 of (lo_elem, hi_elem), round to nearest even; lo_elem in bits 0..15.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo_elem, float hi_elem) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi_elem), "f"(lo_elem));
  return r;
}

// Split the fp32 pair (x, y) into three bf16x2 words with x = hx + mx + lx
// exactly (each residual is the exact rounding error of the previous step).
__device__ __forceinline__ void split3(float x, float y, uint32_t& hi, uint32_t& mid, uint32_t& lo) {
  hi = pack_bf16x2(x, y);
  const float rx = x - bf16_lo(hi), ry = y - bf16_hi(hi);
  mid = pack_bf16x2(rx, ry);
  const float sx = rx - bf16_lo(mid), sy = ry - bf16_hi(mid);
  lo = pack_bf16x2(sx, sy);
}

__device__ __forceinline__ void mma_bf16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void mma_tf32(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// x = hi + lo: hi is x rounded to 11 significant bits (to nearest, ties away
// from zero, by integer add and mask on the bit pattern), lo = x - hi exactly
// (|lo| <= 2^-12 |x|, a multiple of x's fp32 ulp, so it has <= 12 bits).
__device__ __forceinline__ void split_tf32(float x, uint32_t& hi, uint32_t& lo) {
  const uint32_t h = (__float_as_uint(x) + 0x1000u) & 0xffffe000u;
  hi = h;
  lo = __float_as_uint(x - __uint_as_float(h));
}

// ------------------------------------------------------------------ pooling
__global__ void pool_kernel(const void* __restrict__ idx, int dtype, int64_t tok_stride, int64_t first_block,
                            int64_t n_blocks, float* __restrict__ pooled, int64_t pstride) {
  // The scoring launch after this one may start at once: it reads blocks this
  // launch writes only after its own dependency wait.
  grid_dependency_release();
  grid_dependency_wait();
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;  // (block, 4-channel group)
  if (i >= n_blocks * (QSA_INDEX_DIM / 4)) return;
  const int64_t b = first_block + i / (QSA_INDEX_DIM / 4);
  const int d = (int)(i % (QSA_INDEX_DIM / 4)) * 4;
  float4 k[4];
  if (dtype == QSA_F32) {
    const float* src = static_cast<const float*>(idx) + 4 * b * tok_stride + d;
#pragma unroll
    for (int j = 0; j < 4; ++j) k[j] = *reinterpret_cast<const float4*>(src + j * tok_stride);
  } else {
    const __nv_bfloat16* src = static_cast<const __nv_bfloat16*>(idx) + 4 * b * tok_stride + d;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint2 w = *reinterpret_cast<const uint2*>(src + j * tok_stride);
      k[j] = make_float4(bf16_lo(w.x), bf16_hi(w.x), bf16_lo(w.y), bf16_hi(w.y));
    }
  }
  float4 m;
  m.x = (((k[0].x + k[1].x) + k[2].x) + k[3].x) * 0.25f;
  m.y = (((k[0].y + k[1].y) + k[2].y) + k[3].y) * 0.25f;
  m.z = (((k[0].z + k[1].z) + k[2].z) + k[3].z) * 0.25f;
  m.w = (((k[0].w + k[1].w) + k[2].w) + k[3].w) * 0.25f;
  *reinterpret_cast<float4*>(pooled + b * pstride + d) = m;
}

template <int NSEQ>
__device__ __forceinline__ int find_seq_by_work(const ScoreParams<NSEQ>& p, int64_t item) {
  int s = 0;
#pragma unroll
  for (int i = 1; i < NSEQ; ++i)
    if (i < p.n_seqs && item >= p.seq[i].work_begin) s = i;
  return s;
}

// ------------------------------------------------------------------ scoring, tensor pipe
// Persistent warps: warp w of the grid takes work items w, w + W, w + 2W, ...
// (W = warps in the grid); an item is one (16-block tile, group of <= 8
// rows).  Each warp streams its tiles' pooled keys into shared memory with
// cp.async, two tiles in flight, and runs the MMAs on the tile that landed.
// MMA columns are (row, head) pairs n = 4*row + head; NT n-tiles of 8
// columns cover 2*NT rows.  The 128 channels are visited in 8 k-steps of 16;
// inside a k-step, thread quad t holds physical channels 4t..4t+3, i.e.
// logical fragment columns (2t, 2t+1) <- channels (4t, 4t+1) and
// (2t+8, 2t+9) <- channels (4t+2, 4t+3).  A and B use the same channel
// permutation, so the dot products are unchanged and each thread reads one
// float4 per row per k-step.
constexpr int kScoreStages = 2;
constexpr int kRowPitch = 144;   // floats per staged row: 576 bytes keep the float4 reads conflict-free
constexpr int kStageFloats = kScoreTile * kRowPitch;


struct ScoreItem {
  int64_t b0;        // first block of the tile
  int64_t nb_last;   // complete blocks the group's last row sees
  int si;            // sequence
  int row0, rows;    // rows of the group within the sequence
  bool valid;        // item exists
  bool active;       // item has visible blocks
};

template <int NSEQ>
__device__ __forceinline__ ScoreItem score_item(const ScoreParams<NSEQ>& p, int64_t item) {
  ScoreItem x;
  x.valid = item < p.n_work;
  x.active = false;
  x.si = 0;
  x.b0 = 0;
  x.nb_last = 0;
  x.row0 = 0;
  x.rows = 0;
  if (!x.valid) return x;
  x.si = find_seq_by_work(p, item);
  const ScoreSeq& sq = p.seq[x.si];
  // Items of one sequence number < 2^31 (<= 2^14 tiles x groups of 8 rows).
  const int w = (int)(item - sq.work_begin);
  const int tile = sq.n_groups == 1 ? w : w / sq.n_groups;
  const int grp = w - tile * sq.n_groups;
  x.row0 = grp * kRowGroup;
  x.rows = min(kRowGroup, sq.n_rows - x.row0);
  x.b0 = (int64_t)tile * kScoreTile;
  x.nb_last = visible_blocks(row_position(sq.n_tokens, sq.n_rows, x.row0 + x.rows - 1));
  x.active = x.b0 < x.nb_last;
  return x;
}

// tf32 planes (rows groups of <= 4 rows): in every 16-channel k-step above,
// thread t's float4 of channels 4t..4t+3 feeds two m16n8k8 steps -- channels
// 4t, 4t+1 are fragment k = t, t+4 of the first, channels 4t+2, 4t+3 those of
// the second -- and the queries take the same mapping.
template <int NT, int NSEQ, int WARPS>
__global__ void __launch_bounds__(WARPS * 32, 1) score_mma_kernel(const ScoreParams<NSEQ> p) {
  constexpr bool kTf32 = NT <= 2;
  constexpr int kBq = kTf32 ? 4 : 2;
  extern __shared__ float4 score_smem4[];
  grid_dependency_sync();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int g = lane >> 2, t = lane & 3;
  float* my = reinterpret_cast<float*>(score_smem4) + warp * kScoreStages * kStageFloats;
  const int64_t W = (int64_t)gridDim.x * WARPS;
  int64_t item = (int64_t)blockIdx.x * WARPS + warp;

  // 16 rows x 32 chunks of 16 bytes; lane takes chunks lane, lane + 32, ...
  auto issue = [&](const ScoreItem& x, int stage) {
    if (!x.active) return;
    const ScoreSeq& sq = p.seq[x.si];
    float* dst = my + stage * kStageFloats;
    const float* src = sq.pooled + x.b0 * sq.pooled_stride;
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      const int c = lane + 32 * j, row = c >> 5, col = c & 31;
      const bool ok = x.b0 + row < x.nb_last;
      cp_async16(dst + row * kRowPitch + col * 4, ok ? src + row * sq.pooled_stride + col * 4 : src, ok);
    }
  };

  ScoreItem cur = score_item(p, item);
  ScoreItem nxt = score_item(p, item + W);
  issue(cur, 0);
  cp_async_commit();
  issue(nxt, 1);
  cp_async_commit();

  // B operand, the group's index queries: per n-tile and 16-channel step,
  // tf32 words (channels 4t, 4t+1, 4t+2, 4t+3) or packed bf16 pairs.
  uint32_t bq[NT][8][kBq];
  int bq_si = -1, bq_row0 = -1;
  int stage = 0;
  while (cur.valid) {
    cp_async_wait<1>();
    __syncwarp();
    if (cur.active) {
      const ScoreSeq& sq = p.seq[cur.si];
      if (cur.si != bq_si || cur.row0 != bq_row0) {
        const __nv_bfloat16* qb = static_cast<const __nv_bfloat16*>(p.q_idx);
#pragma unroll
        for (int j = 0; j < NT; ++j) {
          const int n = 8 * j + g, r = n >> 2, h = n & 3;
          const __nv_bfloat16* src =
              qb + ((int64_t)(sq.row_begin + cur.row0 + r) * QSA_INDEX_HEADS + h) * QSA_INDEX_DIM + 4 * t;
#pragma unroll
          for (int s = 0; s < 8; ++s) {
            uint2 v = make_uint2(0u, 0u);
            if (r < cur.rows) v = *reinterpret_cast<const uint2*>(src + 16 * s);
            if constexpr (kTf32) {
              bq[j][s][0] = v.x << 16;
              bq[j][s][1] = v.x & 0xffff0000u;
              bq[j][s][kBq - 2] = v.y << 16;
              bq[j][s][kBq - 1] = v.y & 0xffff0000u;
            } else {
              bq[j][s][0] = v.x;
              bq[j][s][1] = v.y;
            }
          }
        }
        bq_si = cur.si;
        bq_row0 = cur.row0;
      }
      const float* a = my + stage * kStageFloats;
      float acc[NT][4];
      if constexpr (kTf32) {
        // Separate accumulators per plane and k-step parity keep the MMA
        // dependency chains short.
        float ah[2][NT][4], al[2][NT][4];
#pragma unroll
        for (int q = 0; q < 2; ++q)
#pragma unroll
          for (int j = 0; j < NT; ++j)
#pragma unroll
            for (int e = 0; e < 4; ++e) ah[q][j][e] = al[q][j][e] = 0.f;
#pragma unroll
        for (int s = 0; s < 8; ++s) {
          const float4 ra = *reinterpret_cast<const float4*>(a + g * kRowPitch + 16 * s + 4 * t);
          const float4 rb = *reinterpret_cast<const float4*>(a + (g + 8) * kRowPitch + 16 * s + 4 * t);
          uint32_t h0, l0, h1, l1, h2, l2, h3, l3;
          split_tf32(ra.x, h0, l0);  // row g,   k = t     (channel 4t)
          split_tf32(rb.x, h1, l1);  // row g+8, k = t
          split_tf32(ra.y, h2, l2);  // row g,   k = t + 4 (channel 4t+1)
          split_tf32(rb.y, h3, l3);  // row g+8, k = t + 4
#pragma unroll
          for (int j = 0; j < NT; ++j) {
            mma_tf32(al[0][j], l0, l1, l2, l3, bq[j][s][0], bq[j][s][1]);
            mma_tf32(ah[0][j], h0, h1, h2, h3, bq[j][s][0], bq[j][s][1]);
          }
          split_tf32(ra.z, h0, l0);  // channel 4t+2
          split_tf32(rb.z, h1, l1);
          split_tf32(ra.w, h2, l2);  // channel 4t+3
          split_tf32(rb.w, h3, l3);
#pragma unroll
          for (int j = 0; j < NT; ++j) {
            mma_tf32(al[1][j], l0, l1, l2, l3, bq[j][s][kBq - 2], bq[j][s][kBq - 1]);
            mma_tf32(ah[1][j], h0, h1, h2, h3, bq[j][s][kBq - 2], bq[j][s][kBq - 1]);
          }
        }
#pragma unroll
        for (int j = 0; j < NT; ++j)
#pragma unroll
          for (int e = 0; e < 4; ++e) acc[j][e] = (ah[0][j][e] + ah[1][j][e]) + (al[0][j][e] + al[1][j][e]);
      } else {
        // One accumulator per bf16 part keeps the MMA dependency chains short.
        float accm[NT][4], accl[NT][4];
#pragma unroll
        for (int j = 0; j < NT; ++j)
#pragma unroll
          for (int e = 0; e < 4; ++e) acc[j][e] = accm[j][e] = accl[j][e] = 0.f;
#pragma unroll
        for (int s = 0; s < 8; ++s) {
          const float4 ra = *reinterpret_cast<const float4*>(a + g * kRowPitch + 16 * s + 4 * t);
          const float4 rb = *reinterpret_cast<const float4*>(a + (g + 8) * kRowPitch + 16 * s + 4 * t);
          uint32_t h0, m0, l0, h1, m1, l1, h2, m2, l2, h3, m3, l3;
          split3(ra.x, ra.y, h0, m0, l0);  // row g,   columns 2t, 2t+1
          split3(rb.x, rb.y, h1, m1, l1);  // row g+8, columns 2t, 2t+1
          split3(ra.z, ra.w, h2, m2, l2);  // row g,   columns 2t+8, 2t+9
          split3(rb.z, rb.w, h3, m3, l3);  // row g+8, columns 2t+8, 2t+9
#pragma unroll
          for (int j = 0; j < NT; ++j) {
            mma_bf16(accl[j], l0, l1, l2, l3, bq[j][s][0], bq[j][s][1]);
            mma_bf16(accm[j], m0, m1, m2, m3, bq[j][s][0], bq[j][s][1]);
            mma_bf16(acc[j], h0, h1, h2, h3, bq[j][s][0], bq[j][s][1]);
          }
        }
#pragma unroll
        for (int j = 0; j < NT; ++j)
#pragma unroll
          for (int e = 0; e < 4; ++e) acc[j][e] += accm[j][e] + accl[j][e];
      }
      // Epilogue: thread (g, t) holds columns 8j+2t, 8j+2t+1 = heads 2(t&1),
      // 2(t&1)+1 of row 2j + (t>>1) for blocks b0+g and b0+g+8; its
      // neighbour t^1 holds the other two heads.  The tile's maximum per row
      // is its group maximum.
#pragma unroll
      for (int j = 0; j < NT; ++j) {
        float v0 = fmaxf(acc[j][0], 0.f) + fmaxf(acc[j][1], 0.f);
        float v1 = fmaxf(acc[j][2], 0.f) + fmaxf(acc[j][3], 0.f);
        v0 += __shfl_xor_sync(0xffffffffu, v0, 1);
        v1 += __shfl_xor_sync(0xffffffffu, v1, 1);
        v0 *= kScoreScale;
        v1 *= kScoreScale;
        const int r = 2 * j + (t >> 1);
        const int64_t nb = r < cur.rows ? visible_blocks(row_position(sq.n_tokens, sq.n_rows, cur.row0 + r)) : 0;
        const bool ok0 = cur.b0 + g < nb, ok1 = cur.b0 + g + 8 < nb;
        const int64_t grow = sq.row_begin + cur.row0 + r;
        if ((t & 1) == 0 && r < cur.rows) {
          float* dst = p.scores + grow * p.ld;
          if (ok0) dst[cur.b0 + g] = v0;
          if (ok1) dst[cur.b0 + g + 8] = v1;
        }
        if (p.gmax) {
          float m = fmaxf(ok0 ? v0 : -INFINITY, ok1 ? v1 : -INFINITY);
          m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 4));
          m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 8));
          m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 16));
          if (g == 0 && (t & 1) == 0 && cur.b0 < nb) p.gmax[grow * p.gld + cur.b0 / kScoreTile] = m;
        }
      }
    }
    __syncwarp();
    const ScoreItem n2 = score_item(p, item + 2 * W);
    issue(n2, stage);
    cp_async_commit();
    cur = nxt;
    nxt = n2;
    item += W;
    stage ^= 1;
  }
  cp_async_wait<0>();
}

// ------------------------------------------------------------------ scoring, tensor pipe, TMA-fed
// The few-row path (2 to 4 rows per sequence, bf16 queries): persistent CTAs,
// each owning a contiguous range of items; an item is 4 tiles (64 blocks) of
// one sequence.  Warp 0 is the producer: lane L < kTmaItems loads the items
// of ring slot L, each with four 2-D tensor copies of 64 blocks x 32 channels
// (8 KB, 128-byte swizzle) completing on the slot's barrier, so a CTA keeps
// kTmaItems x 32 KB of pooled keys in flight and refills each slot as soon
// as it is consumed (the tensor-copy engine spends a fixed time per copy and
// per barrier transaction, so copies are issued from several lanes and are
// as large as the ring allows: 8 KB boxes in 4 slots took the 261,120-token
// verify's launch from 9.8 to 9.2 us against 4 KB boxes in 8 slots, with the
// same 128 KB in flight; a steady ring keeps HBM busier than requesting a
// CTA's whole range at once, and 192 KB rings were slower).  Two CTAs share
// an SM, each with two slots and four consumers: the same 128 KB in flight
// per SM, but two producers and half as many consumers per barrier, which
// took the same launch from 9.2 to 8.6 us.
// kTmaConsumers consumer warps run the tf32 MMAs of the kernel above, one
// tile at a time: tile j of the item in slot q belongs to consumer
// (kItemTiles q + j) % kTmaConsumers, so each consumer waits on a slot's
// barrier phases in order.  With the swizzle, the 16-byte chunk c of box row
// r (4 of its 32 channels) sits at chunk c ^ (r & 7).  In 16-channel step s,
// thread t reads chunk 2t + (s & 1) of box s / 2 -- channels
// 32 (s / 2) + 8t + 4 (s & 1) .. +3, split over the two m16n8k8 steps as above
// -- so the 8 lanes of one shared-memory phase (rows g, g ^ 1, t = 0..3)
// cover all 8 chunks of a bank row.  The queries take the same channel
// mapping.
constexpr int kItemTiles = 4;
constexpr int kItemBlocks = kItemTiles * kScoreTile;          // 64
constexpr int kTmaItems = 2;                                  // ring slots: 64 KB in flight per CTA
constexpr int kTmaConsumers = 4;
constexpr int kTmaCtasPerSm = 2;
constexpr int kBoxRows = kItemBlocks;
constexpr int kBoxBytes = kBoxRows * 128;                     // 64 rows x 32 fp32 = 8 KB
constexpr int kItemBytes = 4 * kBoxBytes;                     // 32 KB
static_assert((kTmaItems * kItemTiles) % kTmaConsumers == 0, "tile slots split evenly over consumers");
static_assert(kTmaItems <= 32, "one producer lane per ring slot");
constexpr int kPoolScratch = 4 * QSA_INDEX_DIM * 4;               // one block's four f32 index keys
constexpr size_t kTmaSmem = (size_t)kTmaItems * kItemBytes + 1024;   // + alignment slack
constexpr size_t kTmaPoolSmem = kTmaSmem + (size_t)kTmaConsumers * kPoolScratch;   // + a scratch per consumer

__device__ int g_score_wait_timeouts;   // waits that gave up (never expected)

// The index keys of token t (es bytes per element): from the appended
// tokens' input when the launch also appends t, else from the cache.
__device__ __forceinline__ const char* idx_row(const ScoreSeq& sq, int64_t t, int es) {
  if (sq.idx_new && t >= sq.first_new)
    return static_cast<const char*>(sq.idx_new) + (t - sq.first_new) * QSA_INDEX_DIM * es;
  return static_cast<const char*>(sq.idx_keys) + t * sq.idx_stride * es;
}

// Lane l's channels 4l .. 4l + 3 of the four index keys of block b.
__device__ __forceinline__ void load_index_keys(const ScoreSeq& sq, int64_t b, int lane, float4 (&k)[4]) {
  if (sq.idx_dtype == QSA_F32) {
#pragma unroll
    for (int j = 0; j < 4; ++j)
      k[j] = *reinterpret_cast<const float4*>(reinterpret_cast<const float*>(idx_row(sq, 4 * b + j, 4)) + 4 * lane);
  } else {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint2 w =
          *reinterpret_cast<const uint2*>(reinterpret_cast<const __nv_bfloat16*>(idx_row(sq, 4 * b + j, 2)) + 4 * lane);
      k[j] = make_float4(bf16_lo(w.x), bf16_hi(w.x), bf16_lo(w.y), bf16_hi(w.y));
    }
  }
}

// The pooling kernel's arithmetic: ((k0 + k1) + k2) + k3, times 0.25.
__device__ __forceinline__ float4 pool4(const float4 (&k)[4]) {
  float4 m;
  m.x = (((k[0].x + k[1].x) + k[2].x) + k[3].x) * 0.25f;
  m.y = (((k[0].y + k[1].y) + k[2].y) + k[3].y) * 0.25f;
  m.z = (((k[0].z + k[1].z) + k[2].z) + k[3].z) * 0.25f;
  m.w = (((k[0].w + k[1].w) + k[2].w) + k[3].w) * 0.25f;
  return m;
}

template <int NSEQ>
struct ScoreTmaParams {
  CUtensorMap tmap[NSEQ];      // pooled keys of sequence i: [n_tokens / 4 rows, 128] fp32
  int64_t item_begin[NSEQ];    // first item of sequence i
  int64_t n_items;
  ScoreParams<NSEQ> p;
  AppendParams ap;             // an append done by the launch (no items: none)
};

template <int NSEQ>
__device__ __forceinline__ int find_seq_by_item(const ScoreTmaParams<NSEQ>& P, int64_t item) {
  int s = 0;
#pragma unroll
  for (int i = 1; i < NSEQ; ++i)
    if (i < P.p.n_seqs && item >= P.item_begin[i]) s = i;
  return s;
}

// POOL: the launch also pools the step's completed blocks (qsa_pool_score_blocks).
template <int NT, int NSEQ, bool POOL>
__global__ void __launch_bounds__(32 * (1 + kTmaConsumers), kTmaCtasPerSm)
    score_tma_kernel(const __grid_constant__ ScoreTmaParams<NSEQ> P) {
  static_assert(NT <= 2, "the TMA path serves groups of <= 4 rows");
  extern __shared__ unsigned char tma_smem_raw[];
  __shared__ uint64_t full_bar[kTmaItems], empty_bar[kTmaItems];
  const ScoreParams<NSEQ>& p = P.p;
  unsigned char* items = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(tma_smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) {
    for (int i = 0; i < kTmaItems; ++i) {
      tc::bar_init(&full_bar[i], 1);
      tc::bar_init(&empty_bar[i], kItemTiles);
    }
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
  }
  __syncthreads();
  const int64_t i0 = P.n_items * blockIdx.x / gridDim.x;
  const int64_t i1 = P.n_items * (blockIdx.x + 1) / gridDim.x;
  const int n_items = (int)(i1 - i0);

  if (warp == 0) {
    // Producer: lane q issues the items of slot q, in order.  Pooled blocks
    // before the ones this step's rows complete are state from earlier steps
    // that no launch of this step writes: a slot's first item is requested
    // before the dependency wait when it holds only such blocks.
    bool waited = false;
    if (lane < kTmaItems) {
      uint64_t* fb = &full_bar[lane];
      uint64_t* eb = &empty_bar[lane];
      unsigned char* dst = items + (size_t)lane * kItemBytes;
      for (int n = lane; n < n_items; n += kTmaItems) {
        const int si = find_seq_by_item(P, i0 + n);
        const int64_t y = (i0 + n - P.item_begin[si]) * kItemBlocks;
        const ScoreSeq& sq = p.seq[si];
        const bool old_blocks = y + kItemBlocks <= (sq.n_tokens - sq.n_rows) / 4;
        if (!waited && !(n < kTmaItems && old_blocks)) {
          grid_dependency_wait();
          waited = true;
        }
        if (n >= kTmaItems && !tc::bar_wait_spin(eb, (uint32_t)((n / kTmaItems - 1) & 1), &g_score_wait_timeouts))
          break;
        tc::bar_expect_tx(fb, kItemBytes);
#pragma unroll
        for (int c = 0; c < 4; ++c) tc::tma_2d(dst + c * kBoxBytes, &P.tmap[si], 32 * c, (int)y, fb);
      }
    }
    if (!waited) grid_dependency_wait();
    grid_dependency_release();
    // The append's copies, on the lanes that issue no tensor copies.
    if (lane >= kTmaItems) {
      constexpr int kCopyLanes = 32 - kTmaItems;
      const int64_t n_copy = P.ap.kv_items + P.ap.idx_items;
      for (int64_t i = (int64_t)blockIdx.x * kCopyLanes + (lane - kTmaItems); i < n_copy;
           i += (int64_t)gridDim.x * kCopyLanes)
        append_copy(P.ap, i);
    }
    return;
  }
  grid_dependency_wait();
  grid_dependency_release();

  // Consumers.
  const int cw = warp - 1;
  const int g = lane >> 2, t = lane & 3;
  // The first block this warp pools (a completed block of the step in one of
  // its tiles): its four index keys are copied now into the warp's scratch,
  // so the copy overlaps the stream; any further ones are read when reached.
  unsigned char* keys_s = items + (size_t)kTmaItems * kItemBytes + (size_t)cw * kPoolScratch;
  int64_t pf_b = -1;
  int pf_si = -1;
#pragma unroll
  for (int s = 0; s < NSEQ; ++s) {
    if (!POOL || s >= p.n_seqs) break;
    const ScoreSeq& sq = p.seq[s];
    for (int64_t b = sq.pool_b0; b < sq.pool_b1 && pf_b < 0; ++b) {
      const int64_t item = P.item_begin[s] + b / kItemBlocks;
      if (item < i0 || item >= i1) continue;
      const int q = (int)((item - i0) % kTmaItems);
      const int j = (int)((b % kItemBlocks) / kScoreTile);
      if ((kItemTiles * q + j) % kTmaConsumers != cw) continue;
      const int es = sq.idx_dtype == QSA_F32 ? 4 : 2;
      const int chunks = QSA_INDEX_DIM * es / 16;   // per key row
      for (int c = lane; c < 4 * chunks; c += 32) {
        const char* src = idx_row(sq, 4 * b + c / chunks, es) + (c % chunks) * 16;
        const uint32_t dst = (uint32_t)__cvta_generic_to_shared(keys_s + c * 16);
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(dst), "l"(src) : "memory");
      }
      asm volatile("cp.async.commit_group;\n" ::: "memory");
      pf_b = b;
      pf_si = s;
    }
  }
  uint32_t bq[NT][8][2];   // packed bf16 pairs (channels +0, +1) and (+2, +3)
  int bq_si = -1;
  for (int n = 0; n < n_items; ++n) {
    const int q = n % kTmaItems;
    const int j = ((cw - kItemTiles * q) % kTmaConsumers + kTmaConsumers) % kTmaConsumers;
    if (j >= kItemTiles) continue;   // no tile of this item is ours
    const int64_t item = i0 + n;
    const int si = find_seq_by_item(P, item);
    const ScoreSeq& sq = p.seq[si];
    const int64_t tile = (item - P.item_begin[si]) * kItemTiles + j;
    const bool valid = tile < sq.n_tiles;
    const int64_t b0 = tile * kScoreTile;
    const int rows = sq.n_rows;   // one row group on this path
    if (valid && si != bq_si) {
      const __nv_bfloat16* qb = static_cast<const __nv_bfloat16*>(p.q_idx);
#pragma unroll
      for (int jj = 0; jj < NT; ++jj) {
        const int nn = 8 * jj + g, r = nn >> 2, h = nn & 3;
        const __nv_bfloat16* src = qb + ((int64_t)(sq.row_begin + r) * QSA_INDEX_HEADS + h) * QSA_INDEX_DIM + 8 * t;
#pragma unroll
        for (int s = 0; s < 8; ++s) {
          uint2 v = make_uint2(0u, 0u);
          if (r < rows) v = *reinterpret_cast<const uint2*>(src + 32 * (s >> 1) + 4 * (s & 1));
          bq[jj][s][0] = v.x;
          bq[jj][s][1] = v.y;
        }
      }
      bq_si = si;
    }
    if (!tc::bar_wait_spin(&full_bar[q], (uint32_t)((n / kTmaItems) & 1), &g_score_wait_timeouts)) break;
    float acc[NT][4];
    if (valid) {
      const unsigned char* tl = items + (size_t)q * kItemBytes + j * (kScoreTile * 128);
      // Step 1 for the tile's completed blocks: replace the rows the tensor
      // copy brought with the mean of their index keys, and store it.
      const int64_t plo = POOL ? max(sq.pool_b0, b0) : 0, phi = POOL ? min(sq.pool_b1, b0 + kScoreTile) : 0;
      for (int64_t b = plo; b < phi; ++b) {
        float4 k4[4];
        if (b == pf_b && si == pf_si) {
          asm volatile("cp.async.wait_all;\n" ::: "memory");
          __syncwarp();
          if (sq.idx_dtype == QSA_F32) {
#pragma unroll
            for (int e = 0; e < 4; ++e) k4[e] = *reinterpret_cast<const float4*>(keys_s + e * 512 + 16 * lane);
          } else {
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const uint2 w = *reinterpret_cast<const uint2*>(keys_s + e * 256 + 8 * lane);
              k4[e] = make_float4(bf16_lo(w.x), bf16_hi(w.x), bf16_lo(w.y), bf16_hi(w.y));
            }
          }
        } else {
          load_index_keys(sq, b, lane, k4);
        }
        const float4 m = pool4(k4);
        const int rr = (int)(b - b0);   // row of the tile
        *reinterpret_cast<float4*>(items + (size_t)q * kItemBytes + j * (kScoreTile * 128) + (lane >> 3) * kBoxBytes +
                                   rr * 128 + (((lane & 7) ^ (rr & 7)) << 4)) = m;
        *reinterpret_cast<float4*>(const_cast<float*>(sq.pooled) + b * sq.pooled_stride + 4 * lane) = m;
      }
      if (phi > plo) __syncwarp();
      float ah[2][NT][4], al[2][NT][4];
#pragma unroll
      for (int u = 0; u < 2; ++u)
#pragma unroll
        for (int jj = 0; jj < NT; ++jj)
#pragma unroll
          for (int e = 0; e < 4; ++e) ah[u][jj][e] = al[u][jj][e] = 0.f;
      // The tile's fragments into registers first: the slot is released
      // before the MMAs run, so its refill is requested one tile earlier.
      float4 fa[8], fb[8];
#pragma unroll
      for (int s = 0; s < 8; ++s) {
        // Rows g and g + 8 of the tile (same swizzle: g & 7), chunk 2t + (s & 1) of box s / 2.
        const unsigned char* box = tl + (s >> 1) * kBoxBytes;
        const int chunk = (2 * t + (s & 1)) ^ g;
        fa[s] = *reinterpret_cast<const float4*>(box + g * 128 + 16 * chunk);
        fb[s] = *reinterpret_cast<const float4*>(box + (g + 8) * 128 + 16 * chunk);
      }
      __syncwarp();
      if (lane == 0) tc::bar_arrive(&empty_bar[q]);
#pragma unroll
      for (int s = 0; s < 8; ++s) {
        const float4 ra = fa[s];
        const float4 rb = fb[s];
        uint32_t h0, l0, h1, l1, h2, l2, h3, l3;
        split_tf32(ra.x, h0, l0);  // row g,   k = t     (first channel of the chunk)
        split_tf32(rb.x, h1, l1);  // row g+8, k = t
        split_tf32(ra.y, h2, l2);  // row g,   k = t + 4 (second channel)
        split_tf32(rb.y, h3, l3);  // row g+8, k = t + 4
#pragma unroll
        for (int jj = 0; jj < NT; ++jj) {
          const uint32_t b0 = bq[jj][s][0] << 16, b1 = bq[jj][s][0] & 0xffff0000u;
          mma_tf32(al[0][jj], l0, l1, l2, l3, b0, b1);
          mma_tf32(ah[0][jj], h0, h1, h2, h3, b0, b1);
        }
        split_tf32(ra.z, h0, l0);  // third and fourth channels: the second k-step
        split_tf32(rb.z, h1, l1);
        split_tf32(ra.w, h2, l2);
        split_tf32(rb.w, h3, l3);
#pragma unroll
        for (int jj = 0; jj < NT; ++jj) {
          const uint32_t b0 = bq[jj][s][1] << 16, b1 = bq[jj][s][1] & 0xffff0000u;
          mma_tf32(al[1][jj], l0, l1, l2, l3, b0, b1);
          mma_tf32(ah[1][jj], h0, h1, h2, h3, b0, b1);
        }
      }
#pragma unroll
      for (int jj = 0; jj < NT; ++jj)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[jj][e] = (ah[0][jj][e] + ah[1][jj][e]) + (al[0][jj][e] + al[1][jj][e]);
    }
    if (!valid) {   // (a valid tile released its slot above)
      __syncwarp();
      if (lane == 0) tc::bar_arrive(&empty_bar[q]);
      continue;
    }
    // Epilogue as in score_mma_kernel: scores and the tile's group maximum.
#pragma unroll
    for (int jj = 0; jj < NT; ++jj) {
      float v0 = fmaxf(acc[jj][0], 0.f) + fmaxf(acc[jj][1], 0.f);
      float v1 = fmaxf(acc[jj][2], 0.f) + fmaxf(acc[jj][3], 0.f);
      v0 += __shfl_xor_sync(0xffffffffu, v0, 1);
      v1 += __shfl_xor_sync(0xffffffffu, v1, 1);
      v0 *= kScoreScale;
      v1 *= kScoreScale;
      const int r = 2 * jj + (t >> 1);
      const int64_t nb = r < rows ? visible_blocks(row_position(sq.n_tokens, sq.n_rows, r)) : 0;
      const bool ok0 = b0 + g < nb, ok1 = b0 + g + 8 < nb;
      const int64_t grow = sq.row_begin + r;
      if ((t & 1) == 0 && r < rows) {
        float* dst = p.scores + grow * p.ld;
        if (ok0) dst[b0 + g] = v0;
        if (ok1) dst[b0 + g + 8] = v1;
      }
      if (p.gmax) {
        float m = fmaxf(ok0 ? v0 : -INFINITY, ok1 ? v1 : -INFINITY);
        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 4));
        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 8));
        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 16));
        if (g == 0 && (t & 1) == 0 && b0 < nb) p.gmax[grow * p.gld + b0 / kScoreTile] = m;
      }
    }
  }
  // A key copy whose tile was never reached (a wait that gave up) lands before exit.
  if constexpr (POOL) asm volatile("cp.async.wait_all;\n" ::: "memory");
}

// ------------------------------------------------------------------ few-row scoring, direct loads
// Decode and verify (<= 8 rows per sequence, bf16 index queries): every
// pooled block is read once with plain 128-bit loads straight into registers,
// and the dot products run as tf32 MMAs (m16n8k8) on the two-plane split of
// the key (split_tf32), so no product loses precision beyond one fp32 ulp of
// the key.  MMA rows are (row, head) pairs rh = 4 row + head (NMT tiles of
// 16: <= 4 rows per tile), MMA columns are 8 blocks, and the 128 channels
// are 16 k-steps of 8.  The k-slots of a step are mapped to channels so
// that the four lanes of a quad read 64 contiguous bytes per load: lane
// (g, t) (g = lane / 4, t = lane % 4) holds block g's channels 16q + 4t ..
// 16q + 4t + 3 (q < 8) and supplies channel 16q + 4t + 2p (slot t) and
// 16q + 4t + 2p + 1 (slot t + 4) at k-step j = 2q + p; the queries use the
// same mapping, which leaves every dot product unchanged.
//
// Persistent warps: warp w of the grid takes tiles (16 blocks = 8 KB) w,
// w + W, w + 2W, ... of the call, so consecutive warps read consecutive
// memory.  A tile is two 8-block halves; the next tile's halves are loaded
// while the current one is multiplied, so every warp keeps 8 KB in flight.
// The epilogue adds the four heads' ReLUs across lanes, writes each row's
// visible scores and the tile's maximum per row (the group maximum).
// Step 1 rides along (qsa_pool_score_blocks): a half holding a block the
// step's rows complete replaces that block's loaded values with the mean of
// its four index keys (the pooling kernel's order of operations) and stores
// it to the pooled keys.
// Warps per CTA and CTAs per SM by row-head tiles (registers: ~220 per
// thread for one tile, the most for two).
template <int NMT>
struct DirShape {
  static constexpr int warps = 4;
  static constexpr int ctas_per_sm = NMT == 1 ? 3 : 2;
  // Per warp: query fragments, then a pooling scratch of two blocks.
  static constexpr size_t q_bytes = (size_t)NMT * 16 * 32 * sizeof(uint2);
  static constexpr size_t warp_bytes = q_bytes + 2 * 4 * QSA_INDEX_DIM * 4;
  static constexpr size_t smem = (size_t)warps * warp_bytes;
};

// split_tf32 issued where it is used (volatile), so the compiler does not
// hoist the splits of a whole half ahead of its MMAs and hold them all live.
__device__ __forceinline__ void split_tf32_at_use(float x, uint32_t& hi, uint32_t& lo) {
  asm volatile(
      "{\n\t.reg .b32 r, f;\n\t"
      "add.u32 r, %2, 0x1000;\n\t"
      "and.b32 %0, r, 0xffffe000;\n\t"
      "sub.f32 f, %3, %0;\n\t"
      "mov.b32 %1, f;\n\t}"
      : "=r"(hi), "=r"(lo)
      : "r"(__float_as_uint(x)), "f"(x));
}

struct HalfTile {
  float4 v[8];   // channels 16q + 4t .. 16q + 4t + 3 of block g of the half, q < 8
};

__device__ __forceinline__ float4 ld_stream(const float4* p) {
  float4 r;
  asm volatile("ld.global.nc.L1::no_allocate.L2::256B.v4.f32 {%0,%1,%2,%3}, [%4];\n"
               : "=f"(r.x), "=f"(r.y), "=f"(r.z), "=f"(r.w)
               : "l"(p));
  return r;
}

// Block b's channels 16q + 4t .. 16q + 4t + 3, q < 8 (zeros past the sequence's blocks).
__device__ __forceinline__ void load_half(HalfTile& h, const ScoreSeq& sq, int64_t b, int64_t nb, int t) {
  if (b < nb) {
    const float4* src = reinterpret_cast<const float4*>(sq.pooled + b * sq.pooled_stride + 4 * t);
#pragma unroll
    for (int q = 0; q < 8; ++q) h.v[q] = ld_stream(src + 4 * q);
  } else {
#pragma unroll
    for (int q = 0; q < 8; ++q) h.v[q] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
}

__device__ __forceinline__ float elem(const HalfTile& h, int e) {
  const float4 v = h.v[e >> 2];
  return (e & 3) == 0 ? v.x : (e & 3) == 1 ? v.y : (e & 3) == 2 ? v.z : v.w;
}

// Step 1 inside the scoring launch.  The index keys of the blocks a tile
// completes (at most 2: <= 8 rows complete <= 2 blocks) are copied into the
// warp's scratch with cp.async when the tile's pooled keys are requested,
// so they arrive with them.  Scratch slot i holds block
// max(pool_b0, b0) + i: its 4 tokens' 128 index-key channels as stored.
constexpr int kPoolSlotBytes = 4 * QSA_INDEX_DIM * 4;   // 4 tokens of f32 keys (bf16 use half)

__device__ __forceinline__ void pool_prefetch(unsigned char* scratch, const ScoreSeq& sq, int64_t b0, int lane) {
  const int64_t lo = max(sq.pool_b0, b0), hi = min(sq.pool_b1, b0 + (int64_t)kScoreTile);
  const int es = sq.idx_dtype == QSA_F32 ? 4 : 2;
  const int chunks = QSA_INDEX_DIM * es / 16;   // 16-byte chunks per token row
  for (int64_t b = lo; b < hi && b < lo + 2; ++b) {
    for (int c = lane; c < 4 * chunks; c += 32) {
      const char* src = idx_row(sq, 4 * b + c / chunks, es) + (c % chunks) * 16;
      const uint32_t dst = (uint32_t)__cvta_generic_to_shared(scratch + (b - lo) * kPoolSlotBytes + c * 16);
      asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(dst), "l"(src) : "memory");
    }
  }
  asm volatile("cp.async.commit_group;\n" ::: "memory");
}

// Block b = b0 + 8h + g of a tile with completed blocks: the mean of its
// four index keys (((k0 + k1) + k2) + k3, times 0.25) over the lane's
// channels 16q + 4t .. 16q + 4t + 3 replaces the loaded values and is stored
// to the pooled keys.  The warp's scratch must have landed.
__device__ __forceinline__ void pool_from_scratch(HalfTile& h, const unsigned char* scratch, const ScoreSeq& sq,
                                                  int64_t b0, int64_t b, int t) {
  const unsigned char* slot = scratch + (b - max(sq.pool_b0, b0)) * kPoolSlotBytes;
  float4* dst = reinterpret_cast<float4*>(const_cast<float*>(sq.pooled) + b * sq.pooled_stride + 4 * t);
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    float4 k[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int c = 16 * q + 4 * t;
      if (sq.idx_dtype == QSA_F32) {
        k[j] = *reinterpret_cast<const float4*>(slot + (j * QSA_INDEX_DIM + c) * 4);
      } else {
        const uint2 w = *reinterpret_cast<const uint2*>(slot + (j * QSA_INDEX_DIM + c) * 2);
        k[j] = make_float4(bf16_lo(w.x), bf16_hi(w.x), bf16_lo(w.y), bf16_hi(w.y));
      }
    }
    h.v[q] = pool4(k);
    dst[4 * q] = h.v[q];
  }
}

__device__ __forceinline__ bool tile_pools(const ScoreSeq& sq, int64_t b0) {
  return sq.pool_b1 > sq.pool_b0 && b0 < sq.pool_b1 && b0 + kScoreTile > sq.pool_b0;
}

// The MMAs of one half: s[mt] = the 16 x 8 (row-head x block) products.
// qs: this warp's query fragments, [mt][j][lane] = (rows g, g + 8) x the two
// channels of k-step j, as bf16 pairs.
template <int NMT>
__device__ __forceinline__ void mma_half(const HalfTile& h, const uint2* qs, int lane, float (&s)[NMT][4]) {
  float ah[NMT][2][4], al[NMT][2][4];
#pragma unroll
  for (int mt = 0; mt < NMT; ++mt)
#pragma unroll
    for (int c = 0; c < 2; ++c)
#pragma unroll
      for (int e = 0; e < 4; ++e) ah[mt][c][e] = al[mt][c][e] = 0.f;
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    uint32_t h0, l0, h1, l1;
    split_tf32_at_use(elem(h, 2 * j), h0, l0);       // k-slot t:     channel 16(j / 2) + 4t + 2(j % 2)
    split_tf32_at_use(elem(h, 2 * j + 1), h1, l1);   // k-slot t + 4: the next channel
#pragma unroll
    for (int mt = 0; mt < NMT; ++mt) {
      const uint2 w = qs[(mt * 16 + j) * 32 + lane];   // rows g, g + 8: the step's two channels
      const uint32_t a0 = w.x << 16, a1 = w.y << 16, a2 = w.x & 0xffff0000u, a3 = w.y & 0xffff0000u;
      mma_tf32(al[mt][j & 1], a0, a1, a2, a3, l0, l1);
      mma_tf32(ah[mt][j & 1], a0, a1, a2, a3, h0, h1);
    }
  }
#pragma unroll
  for (int mt = 0; mt < NMT; ++mt)
#pragma unroll
    for (int e = 0; e < 4; ++e) s[mt][e] = (ah[mt][0][e] + ah[mt][1][e]) + (al[mt][0][e] + al[mt][1][e]);
}

// The append a direct-load launch also does (APPEND), else nothing.
template <bool APPEND>
struct DirAppend {
  AppendParams ap;
};
template <>
struct DirAppend<false> {};

template <int NMT, int NSEQ, bool APPEND>
__global__ void __launch_bounds__(32 * DirShape<NMT>::warps, DirShape<NMT>::ctas_per_sm)
    score_direct_kernel(const __grid_constant__ ScoreParams<NSEQ> p, const __grid_constant__ DirAppend<APPEND> da) {
  constexpr int kWarps = DirShape<NMT>::warps;
  const int lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  const int64_t W = (int64_t)gridDim.x * kWarps;
  int64_t u = (int64_t)blockIdx.x * kWarps + (threadIdx.x >> 5);
  extern __shared__ __align__(16) unsigned char dir_smem[];
  uint2* qs = reinterpret_cast<uint2*>(dir_smem + (size_t)(threadIdx.x >> 5) * DirShape<NMT>::warp_bytes);
  unsigned char* scratch = dir_smem + (size_t)(threadIdx.x >> 5) * DirShape<NMT>::warp_bytes + DirShape<NMT>::q_bytes;
  HalfTile ha, hb;
  // The first tile's pooled keys: blocks older than those the step's rows
  // complete are state that no launch of this step writes, so they may be
  // requested before the dependency wait.
  bool waited = false;
  if (u < p.n_work) {
    const ScoreSeq& sq = p.seq[find_seq_by_work(p, u)];
    const int64_t b0 = (u - sq.work_begin) * kScoreTile;
    const int64_t nbs = sq.n_tokens / 4;
    if (b0 + kScoreTile > (sq.n_tokens - sq.n_rows) / 4) {
      grid_dependency_wait();
      waited = true;
    }
    load_half(ha, sq, b0 + g, nbs, t);
    load_half(hb, sq, b0 + 8 + g, nbs, t);
    if (tile_pools(sq, b0)) pool_prefetch(scratch, sq, b0, lane);
  }
  if (!waited) grid_dependency_wait();
  grid_dependency_release();
  // The append's copies, spread over the launch's threads.
  if constexpr (APPEND) {
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < da.ap.kv_items + da.ap.idx_items;
         i += (int64_t)gridDim.x * blockDim.x)
      append_copy(da.ap, i);
  }
  int q_si = -1;
  for (; u < p.n_work; u += W) {
    const int si = find_seq_by_work(p, u);
    const ScoreSeq& sq = p.seq[si];
    const int64_t b0 = (u - sq.work_begin) * kScoreTile;
    const int rows = sq.n_rows;
    if (si != q_si) {
      // Index queries of rows rh / 4 (heads rh % 4), rh = 16 mt + g + 8 hs:
      // channels 16q + 4t .. 16q + 4t + 3 as two bf16 pairs per q, laid out
      // as the fragments of k-steps j = 2q and 2q + 1.
      const __nv_bfloat16* qb = static_cast<const __nv_bfloat16*>(p.q_idx);
      __syncwarp();
#pragma unroll
      for (int mt = 0; mt < NMT; ++mt) {
        uint2 w[2][8];
#pragma unroll
        for (int hs = 0; hs < 2; ++hs) {
          const int rh = 16 * mt + g + 8 * hs, r = rh >> 2;
          const uint2* src = reinterpret_cast<const uint2*>(
              qb + ((int64_t)(sq.row_begin + r) * QSA_INDEX_HEADS + (rh & 3)) * QSA_INDEX_DIM + 4 * t);
#pragma unroll
          for (int q = 0; q < 8; ++q) w[hs][q] = r < rows ? src[4 * q] : make_uint2(0u, 0u);
        }
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          qs[(mt * 16 + 2 * q) * 32 + lane] = make_uint2(w[0][q].x, w[1][q].x);
          qs[(mt * 16 + 2 * q + 1) * 32 + lane] = make_uint2(w[0][q].y, w[1][q].y);
        }
      }
      __syncwarp();
      q_si = si;
    }
    // Step 1 for the tile's completed blocks, from the scratch requested with the tile.
    if (tile_pools(sq, b0)) {
      asm volatile("cp.async.wait_all;\n" ::: "memory");
      __syncwarp();
      const int64_t ba = b0 + g, bb = b0 + 8 + g;
      if (ba >= sq.pool_b0 && ba < sq.pool_b1) pool_from_scratch(ha, scratch, sq, b0, ba, t);
      if (bb >= sq.pool_b0 && bb < sq.pool_b1) pool_from_scratch(hb, scratch, sq, b0, bb, t);
      __syncwarp();   // the scratch is free for the next tile's copies
    }
    float sa[NMT][4], sb[NMT][4];
    mma_half<NMT>(ha, qs, lane, sa);
    const int64_t un = u + W;
    int sin = si;
    int64_t bn = 0, nbn = 0;
    if (un < p.n_work) {
      sin = find_seq_by_work(p, un);
      bn = (un - p.seq[sin].work_begin) * kScoreTile;
      nbn = p.seq[sin].n_tokens / 4;
      load_half(ha, p.seq[sin], bn + g, nbn, t);
      if (tile_pools(p.seq[sin], bn)) pool_prefetch(scratch, p.seq[sin], bn, lane);
    }
    mma_half<NMT>(hb, qs, lane, sb);
    if (un < p.n_work) load_half(hb, p.seq[sin], bn + 8 + g, nbn, t);
    // Epilogue: ReLU per head, the four heads added across lanes g % 4.
#pragma unroll
    for (int mt = 0; mt < NMT; ++mt) {
      float v[2][4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        v[0][e] = fmaxf(sa[mt][e], 0.f);
        v[1][e] = fmaxf(sb[mt][e], 0.f);
      }
#pragma unroll
      for (int hf = 0; hf < 2; ++hf)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          v[hf][e] += __shfl_xor_sync(0xffffffffu, v[hf][e], 4);
          v[hf][e] += __shfl_xor_sync(0xffffffffu, v[hf][e], 8);
          v[hf][e] *= kScoreScale;
        }
      // Lanes g = 0 and g = 4 hold rows 4 mt + g / 4 (elements 0, 1) and
      // 4 mt + 2 + g / 4 (elements 2, 3), blocks b0 + 8 hf + 2t (+ 1).
#pragma unroll
      for (int rr = 0; rr < 2; ++rr) {
        const int r = 4 * mt + 2 * rr + (g >> 2);
        const int64_t nb = r < rows ? visible_blocks(row_position(sq.n_tokens, sq.n_rows, r)) : 0;
        float m = -INFINITY;
#pragma unroll
        for (int hf = 0; hf < 2; ++hf)
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            const int64_t b = b0 + 8 * hf + 2 * t + c;
            if (b < nb) m = fmaxf(m, v[hf][2 * rr + c]);
          }
        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
        if ((g & 3) == 0 && r < rows) {
          float* dst = p.scores + (int64_t)(sq.row_begin + r) * p.ld;
#pragma unroll
          for (int hf = 0; hf < 2; ++hf)
#pragma unroll
            for (int c = 0; c < 2; ++c) {
              const int64_t b = b0 + 8 * hf + 2 * t + c;
              if (b < nb) dst[b] = v[hf][2 * rr + c];
            }
          if (p.gmax && t == 0 && b0 < nb) p.gmax[(int64_t)(sq.row_begin + r) * p.gld + b0 / kScoreTile] = m;
        }
      }
    }
  }
}

// ------------------------------------------------------------------ scoring, CUDA cores (fp32 queries)
// One CTA per (32-block tile, group of <= 8 rows); lane = (row, head) pair,
// warp w = blocks 4w..4w+3 of the tile.
constexpr int kSimtTile = 32;

template <int NSEQ>
__global__ void __launch_bounds__(256) score_simt_kernel(const ScoreParams<NSEQ> p) {
  __shared__ float q_s[32][QSA_INDEX_DIM + 1];
  __shared__ float k_s[kSimtTile][QSA_INDEX_DIM + 1];
  __shared__ float m_s[kRowGroup][kSimtTile];
  grid_dependency_sync();
  const int64_t item = blockIdx.x;
  if (item >= p.n_work) return;
  const int si = find_seq_by_work(p, item);
  const ScoreSeq& sq = p.seq[si];
  const int64_t w = item - sq.work_begin;
  const int64_t tile = w / sq.n_groups;
  const int grp = (int)(w - tile * sq.n_groups);
  const int row0 = grp * kRowGroup;
  const int rows = min(kRowGroup, sq.n_rows - row0);
  const int64_t b0 = tile * kSimtTile;
  const int64_t nb_last = visible_blocks(row_position(sq.n_tokens, sq.n_rows, row0 + rows - 1));
  if (b0 >= nb_last) return;

  const float* qf = static_cast<const float*>(p.q_idx);
  for (int i = threadIdx.x; i < 32 * QSA_INDEX_DIM; i += blockDim.x) {
    const int pair = i / QSA_INDEX_DIM, d = i % QSA_INDEX_DIM, r = pair >> 2, h = pair & 3;
    q_s[pair][d] = r < rows
                       ? qf[((int64_t)(sq.row_begin + row0 + r) * QSA_INDEX_HEADS + h) * QSA_INDEX_DIM + d]
                       : 0.f;
    const int64_t b = b0 + pair;
    k_s[pair][d] = b < nb_last ? sq.pooled[b * sq.pooled_stride + d] : 0.f;
  }
  __syncthreads();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  float acc[4] = {0.f, 0.f, 0.f, 0.f};
  for (int d = 0; d < QSA_INDEX_DIM; ++d) {
    const float qv = q_s[lane][d];
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[j] = fmaf(qv, k_s[4 * warp + j][d], acc[j]);
  }
  const int r = lane >> 2;
  const int64_t nb = r < rows ? visible_blocks(row_position(sq.n_tokens, sq.n_rows, row0 + r)) : 0;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    float v = fmaxf(acc[j], 0.f);
    v += __shfl_xor_sync(0xffffffffu, v, 1);
    v += __shfl_xor_sync(0xffffffffu, v, 2);
    v *= kScoreScale;
    const int64_t b = b0 + 4 * warp + j;
    if ((lane & 3) == 0) {
      if (b < nb) p.scores[(int64_t)(sq.row_begin + row0 + r) * p.ld + b] = v;
      m_s[r][4 * warp + j] = b < nb ? v : -INFINITY;
    }
  }
  if (!p.gmax) return;
  // The tile's two groups of 16 blocks: their maxima per row.
  __syncthreads();
  if (threadIdx.x < 2 * kRowGroup) {
    const int rr = threadIdx.x >> 1, half = threadIdx.x & 1;
    const int64_t nbr = rr < rows ? visible_blocks(row_position(sq.n_tokens, sq.n_rows, row0 + rr)) : 0;
    const int64_t gb0 = b0 + 16 * half;
    if (gb0 < nbr) {
      float m = -INFINITY;
      for (int i = 0; i < 16; ++i) m = fmaxf(m, m_s[rr][16 * half + i]);
      p.gmax[(int64_t)(sq.row_begin + row0 + rr) * p.gld + gb0 / QSA_SCORE_GROUP] = m;
    }
  }
}

}  // namespace

cudaError_t launch_pool(const void* idx, qsa_dtype dt, int64_t tok_stride, int64_t first_block, int64_t n_blocks,
                        float* pooled, int64_t pstride, cudaStream_t st) {
  const int64_t threads = n_blocks * (QSA_INDEX_DIM / 4);
  const int bs = 256;
  const int64_t grid = (threads + bs - 1) / bs;
  return launch_kernel(pool_kernel, dim3((unsigned)grid), dim3(bs), 0, st, 0, idx, (int)dt, tok_stride, first_block,
                       n_blocks, pooled, pstride);
}

// The work decomposition (tile size) differs between the two kernels; the host
// fills n_tiles / work_begin for kScoreTile (bf16) or kSimtTile (fp32).
int score_tile_blocks(qsa_dtype q_dtype) { return q_dtype == QSA_BF16 ? kScoreTile : kSimtTile; }

namespace {

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
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

// cudaErrorNotSupported: the TMA path does not apply (no encoder, a tensor
// map the driver refuses); the caller then launches the cp.async kernel.
template <int NSEQ>
cudaError_t launch_score_tma(const ScoreParams<NSEQ>& p, int max_rows_per_group, int sms, cudaStream_t st,
                             const AppendParams* ap) {
  PFN_cuTensorMapEncodeTiled_v12000 encode = tensor_map_encoder();
  if (!encode) return cudaErrorNotSupported;
  ScoreTmaParams<NSEQ> P;
  memset(&P, 0, sizeof(P));
  P.p = p;
  if (ap) P.ap = *ap;
  int64_t n_items = 0;
  for (int i = 0; i < p.n_seqs; ++i) {
    const ScoreSeq& q = p.seq[i];
    if (q.n_groups > 1) return cudaErrorNotSupported;   // one row group per sequence on this path
    P.item_begin[i] = n_items;
    n_items += (q.n_tiles + kItemTiles - 1) / kItemTiles;
    const int64_t rows = q.n_tokens / 4;
    if (rows < 1 || !q.pooled) continue;   // no tile of this sequence is loaded
    const cuuint64_t dims[2] = {(cuuint64_t)QSA_INDEX_DIM, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)q.pooled_stride * sizeof(float)};
    const cuuint32_t box[2] = {32, (cuuint32_t)kBoxRows};
    const cuuint32_t elem[2] = {1, 1};
    if (encode(&P.tmap[i], CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float*>(q.pooled), dims, strides, box, elem,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorNotSupported;
  }
  bool pool = false;
  for (int i = 0; i < p.n_seqs; ++i) pool |= p.seq[i].pool_b1 > p.seq[i].pool_b0;
  const size_t smem = pool ? kTmaPoolSmem : kTmaSmem;
  const void* k = max_rows_per_group <= 2 ? (pool ? (const void*)score_tma_kernel<1, NSEQ, true>
                                                  : (const void*)score_tma_kernel<1, NSEQ, false>)
                                          : (pool ? (const void*)score_tma_kernel<2, NSEQ, true>
                                                  : (const void*)score_tma_kernel<2, NSEQ, false>);
  cudaError_t e = allow_dynamic_smem(k, smem);
  if (e != cudaSuccess) return e;
  P.n_items = n_items;
  if (n_items == 0) return cudaSuccess;
  // As many items per CTA as the resident CTAs need, and then as few CTAs
  // as carry that many, so every CTA streams the same number of items.
  // (1,020 items of the 261,120-token verify: 255 CTAs of 4 items rather
  // than 304 of 3 or 4 -- the layer step 28.5 against 29.0 us in a 12-layer
  // graph, though the scoring launch alone takes 8.7 against 8.6; 300 CTAs
  // of 3.4 items took 29.1.)
  const int64_t ctas = (int64_t)sms * kTmaCtasPerSm;
  const int64_t per_cta = (n_items + ctas - 1) / ctas;
  const unsigned grid = (unsigned)((n_items + per_cta - 1) / per_cta);
  const dim3 block(32 * (1 + kTmaConsumers));
  if (max_rows_per_group <= 2) {
    if (pool) return launch_kernel(score_tma_kernel<1, NSEQ, true>, dim3(grid), block, smem, st, 0u, P);
    return launch_kernel(score_tma_kernel<1, NSEQ, false>, dim3(grid), block, smem, st, 0u, P);
  }
  if (pool) return launch_kernel(score_tma_kernel<2, NSEQ, true>, dim3(grid), block, smem, st, 0u, P);
  return launch_kernel(score_tma_kernel<2, NSEQ, false>, dim3(grid), block, smem, st, 0u, P);
}

template <int NMT, int NSEQ>
cudaError_t launch_direct(const ScoreParams<NSEQ>& p, const AppendParams* ap, unsigned grid, cudaStream_t st) {
  constexpr size_t smem = DirShape<NMT>::smem;
  const dim3 block(32 * DirShape<NMT>::warps);
  if (ap) {
    cudaError_t e = allow_dynamic_smem((const void*)score_direct_kernel<NMT, NSEQ, true>, smem);
    if (e != cudaSuccess) return e;
    return launch_kernel(score_direct_kernel<NMT, NSEQ, true>, dim3(grid), block, smem, st, 0u, p, DirAppend<true>{*ap});
  }
  cudaError_t e = allow_dynamic_smem((const void*)score_direct_kernel<NMT, NSEQ, false>, smem);
  if (e != cudaSuccess) return e;
  return launch_kernel(score_direct_kernel<NMT, NSEQ, false>, dim3(grid), block, smem, st, 0u, p, DirAppend<false>{});
}

}  // namespace

template <int NSEQ>
cudaError_t launch_score(const ScoreParams<NSEQ>& p_in, qsa_dtype q_dtype, int max_rows_per_group, cudaStream_t st,
                         const AppendParams* ap) {
  if (p_in.n_work == 0) return ap ? launch_append(*ap, st) : cudaSuccess;
  const int sms = device_sm_count();
  // 2 to 4 rows: the TMA ring (score_tma_kernel); 1 row and 5 to 8 rows:
  // direct loads.  (One row, measured at 65,536 tokens: the decode layer
  // chain takes 18.4 us with the direct kernel against 19.0 with the ring,
  // though the launch alone takes 3.6 against 3.3 us.)
  if (q_dtype == QSA_BF16 && max_rows_per_group >= 2 && max_rows_per_group <= 4) {
    cudaError_t e = launch_score_tma(p_in, max_rows_per_group, sms, st, ap);
    if (e != cudaErrorNotSupported) return e;
  }
  if (q_dtype == QSA_BF16 && max_rows_per_group <= kRowGroup) {
    bool one_group = true;
    for (int i = 0; i < p_in.n_seqs; ++i) one_group &= p_in.seq[i].n_groups == 1;
    if (one_group) {
      // Persistent: as many CTAs as fit on the SMs, no more than the tiles need.
      // (The balanced grid of the TMA ring -- equal tiles per warp, fewer
      // CTAs -- made the 8-row launch slower: 16.6 against 15.6 us.)
      auto grid_of = [&](int warps, int per_sm) {
        const int64_t need = (p_in.n_work + warps - 1) / warps;
        const int64_t ctas = (int64_t)sms * per_sm;
        return (unsigned)(need < ctas ? need : ctas);
      };
      if (max_rows_per_group <= 4)   // one row, or the TMA ring declined the call
        return launch_direct<1, NSEQ>(p_in, ap, grid_of(DirShape<1>::warps, DirShape<1>::ctas_per_sm), st);
      return launch_direct<2, NSEQ>(p_in, ap, grid_of(DirShape<2>::warps, DirShape<2>::ctas_per_sm), st);
    }
  }
  // The other kernels neither append nor pool: those launches come first
  // (the pooling then reads the appended keys from the cache).
  if (ap) {
    cudaError_t e = launch_append(*ap, st);
    if (e != cudaSuccess) return e;
  }
  ScoreParams<NSEQ> p = p_in;
  for (int i = 0; i < p.n_seqs; ++i) {
    ScoreSeq& sq = p.seq[i];
    if (sq.pool_b1 > sq.pool_b0) {
      cudaError_t e = launch_pool(sq.idx_keys, (qsa_dtype)sq.idx_dtype, sq.idx_stride, sq.pool_b0,
                                  sq.pool_b1 - sq.pool_b0, const_cast<float*>(sq.pooled), sq.pooled_stride, st);
      if (e != cudaSuccess) return e;
    }
    sq.pool_b0 = sq.pool_b1 = 0;
  }
  if (q_dtype == QSA_F32) {
    return launch_kernel(score_simt_kernel<NSEQ>, dim3((unsigned)p.n_work), dim3(256), 0, st, 0u, p);
  }
  constexpr int Ws = 12;
  const size_t smem = sizeof(float) * Ws * kScoreStages * kStageFloats;
  const int64_t need = (p.n_work + Ws - 1) / Ws;
  const unsigned grid = (unsigned)(need < sms ? need : sms);
  const void* k = max_rows_per_group <= 2   ? (const void*)score_mma_kernel<1, NSEQ, Ws>
                  : max_rows_per_group <= 4 ? (const void*)score_mma_kernel<2, NSEQ, Ws>
                                            : (const void*)score_mma_kernel<4, NSEQ, Ws>;
  cudaError_t e = allow_dynamic_smem(k, smem);
  if (e != cudaSuccess) return e;
  const dim3 block(Ws * 32);
  if (max_rows_per_group <= 2) return launch_kernel(score_mma_kernel<1, NSEQ, Ws>, dim3(grid), block, smem, st, 0u, p);
  if (max_rows_per_group <= 4) return launch_kernel(score_mma_kernel<2, NSEQ, Ws>, dim3(grid), block, smem, st, 0u, p);
  return launch_kernel(score_mma_kernel<4, NSEQ, Ws>, dim3(grid), block, smem, st, 0u, p);
}

template cudaError_t launch_score<1>(const ScoreParams<1>&, qsa_dtype, int, cudaStream_t, const AppendParams*);
template cudaError_t launch_score<kLaunchSeqs>(const ScoreParams<kLaunchSeqs>&, qsa_dtype, int, cudaStream_t,
                                               const AppendParams*);

int score_wait_timeouts() {
  int v = 0;
  return cudaMemcpyFromSymbol(&v, g_score_wait_timeouts, sizeof(int)) == cudaSuccess ? v : -1;
}

}  // namespace qsa
