// Row bookkeeping and K/V gathers shared by the attention kernels: the
// selected list of a query row (hipfire, "QSA sparse attention and the VMM KV
// backend", section 02: the 4 tokens of every selected block, then the
// incomplete tail block) and the lookup of a list entry in the sequence's KV
// segment table (MTPLX pull request #610).
#pragma once

#include <cuda_fp16.h>

#include "qsa_internal.cuh"

namespace qsa {
namespace attn {

namespace {
// Selected block ids outside [0, nb) met by this translation unit's kernels
// (skipped; read and cleared by qsa_check_device_status).
__device__ int g_bad_ids;
}  // namespace

// Per-row context: position, visible blocks, selected list length.  The
// list's longest possible length (cnt = min(sel_ld, nb)) is known without
// reading cnt, so the splits' ranges and id loads need not wait for it.
struct RowCtx {
  int64_t nb;
  int64_t tail;       // tail tokens 4 nb .. p
  int64_t n_list;     // 4 cnt + tail (set by set_count)
  int64_t n_max;      // 4 min(sel_ld, nb) + tail
  const int32_t* sel_row;
  int32_t cnt;
  int32_t seg_begin;
  int32_t n_segs;
};

template <int NSEQ>
__device__ __forceinline__ RowCtx make_row_ctx(const AttnParams<NSEQ>& p, int r) {
  int si = 0;
#pragma unroll
  for (int i = 1; i < NSEQ; ++i)
    if (i < p.n_seqs && r >= p.seq[i].row_begin) si = i;
  const AttnSeq sq = p.seq[si];
  const int64_t pos = row_position(sq.n_tokens, sq.n_rows, r - sq.row_begin);
  RowCtx c;
  c.nb = visible_blocks(pos);
  c.tail = pos + 1 - 4 * c.nb;
  c.n_max = 4 * min((int64_t)p.sel_ld, c.nb) + c.tail;
  c.n_list = c.n_max;
  c.cnt = 0;
  c.sel_row = p.sel + (int64_t)r * p.sel_ld;
  c.seg_begin = sq.seg_begin;
  c.n_segs = sq.n_segs;
  return c;
}

// The row's count as loaded (clamped to 0 .. min(sel_ld, nb)).
__device__ __forceinline__ void set_count(RowCtx& c, int32_t cnt, int32_t sel_ld) {
  cnt = max(0, min(cnt, sel_ld));
  if ((int64_t)cnt > c.nb) cnt = (int32_t)c.nb;
  c.cnt = cnt;
  c.n_list = 4 * (int64_t)cnt + c.tail;
}

// Entries [i0, i1) of the longest possible list that split `split` of n
// takes: whole 32-token tiles of the selected blocks' entries, balanced over
// the row; the last split also takes the tail tokens (at most 3), so they
// cost no split of their own.
__device__ __forceinline__ void split_range(const RowCtx& c, int split, int n, int64_t& i0, int64_t& i1) {
  const int64_t T = max((c.n_max - c.tail + 31) / 32, (int64_t)1);
  i0 = 32 * (T * split / n);
  i1 = split == n - 1 ? c.n_max : min(c.n_max, 32 * (T * (split + 1) / n));
}

// The block ids a split needs, staged in shared memory once: entries
// [blk0, blk0 + n) of the row's selection (n <= kIdCache).
constexpr int kIdCache = 512;

struct IdCache {
  const int32_t* ids;   // shared memory
  int64_t blk0;
  int n;
};

// Entry i of the row's selected list -> element offset of (KV head g, token)
// in its segment, and the segment.  False when the entry names an invalid
// block id or a token no segment covers.
template <int NSEQ>
__device__ __forceinline__ bool locate(const AttnParams<NSEQ>& p, const RowCtx& c, const IdCache& ic, int64_t i,
                                       int g, int& seg, int64_t& off, int64_t* tok_in_seg = nullptr) {
  int64_t t;
  if (i >= c.n_list) return false;
  if (i < 4 * (int64_t)c.cnt) {
    const int64_t k = (i >> 2) - ic.blk0;
    const int32_t b = (k >= 0 && k < ic.n) ? ic.ids[k] : __ldg(c.sel_row + (i >> 2));
    if (b < 0 || (int64_t)b >= c.nb) {
      atomicAdd(&g_bad_ids, 1);
      return false;
    }
    t = 4 * (int64_t)b + (i & 3);
  } else {
    t = 4 * c.nb + (i - 4 * (int64_t)c.cnt);
  }
  for (int s = 0; s < c.n_segs; ++s) {
    const Segment& sg = p.seg[c.seg_begin + s];
    if (t >= sg.first && t < sg.first + sg.n) {
      seg = c.seg_begin + s;
      off = (int64_t)g * sg.head_stride + (t - sg.first) * sg.tok_stride;
      if (tok_in_seg) *tok_in_seg = t - sg.first;
      return true;
    }
  }
  return false;
}

// Stage the ids of list entries [i0, i1) into ids_s (all threads call).
__device__ __forceinline__ IdCache stage_ids(const RowCtx& c, int64_t i0, int64_t i1, int32_t* ids_s) {
  IdCache ic;
  ic.ids = ids_s;
  ic.blk0 = i0 >> 2;
  const int64_t last = min(i1, c.n_max - c.tail);   // entries past the selected part are tail tokens
  int64_t n = last > i0 ? ((last - 1) >> 2) - ic.blk0 + 1 : 0;
  if (n > kIdCache) n = kIdCache;
  ic.n = (int)n;
  for (int k = threadIdx.x; k < ic.n; k += blockDim.x) ids_s[k] = __ldg(c.sel_row + ic.blk0 + k);
  return ic;
}


// ---------------------------------------------------------------- quantized K/V codes
// Two E4M3 codes (low byte first) -> two bf16 (low half first), exactly:
// E4M3 -> f16 -> f32 -> bf16 loses nothing (4 significant bits, exponents
// 2^-9 .. 2^8).
__device__ __forceinline__ uint32_t e4m3x2_to_bf16x2(uint32_t two_codes) {
  uint32_t h2;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"((unsigned short)two_codes));
  const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&h2));
  const __nv_bfloat162 b = __floats2bfloat162_rn(f.x, f.y);
  return *reinterpret_cast<const uint32_t*>(&b);
}
// Four int8 codes (low byte first) times a block scale d -> four bf16 (two
// words, low half first), each rounded once.  Code c becomes the binary32
// 2^23 + 128 + c exactly -- its biased byte c ^ 0x80 placed in the mantissa
// of 2^23 -- less 2^23 + 128; the product with d is exact in binary32 (8 x 11
// significant bits).
__device__ __forceinline__ void i8x4_to_bf16x4(uint32_t four_codes, float d, uint32_t& lo, uint32_t& hi) {
  const uint32_t u = four_codes ^ 0x80808080u;
  const float c0 = __uint_as_float(__byte_perm(u, 0x4b000000u, 0x7440)) - 8388736.0f;
  const float c1 = __uint_as_float(__byte_perm(u, 0x4b000000u, 0x7441)) - 8388736.0f;
  const float c2 = __uint_as_float(__byte_perm(u, 0x4b000000u, 0x7442)) - 8388736.0f;
  const float c3 = __uint_as_float(__byte_perm(u, 0x4b000000u, 0x7443)) - 8388736.0f;
  const __nv_bfloat162 a = __floats2bfloat162_rn(c0 * d, c1 * d);
  const __nv_bfloat162 b = __floats2bfloat162_rn(c2 * d, c3 * d);
  lo = *reinterpret_cast<const uint32_t*>(&a);
  hi = *reinterpret_cast<const uint32_t*>(&b);
}

}  // namespace attn
}  // namespace qsa
