// Appending a sequence's newest tokens to its caches in place, with the
// pooling of the blocks they complete (step 1) in the same launch: the step
// either side of the pooling in a QSA layer (hipfire, "QSA sparse attention
// and the VMM KV backend", section 02: a QSA layer writes an index key for
// every token besides its K/V, and every 4 consecutive index keys are
// averaged into one pooled block key; MTPLX pull request #482, optimisation
// 1: the new rows' K/V are written into the existing cache, not into a copy).
//
// One launch, three kinds of 16-byte work item (thread = item):
//   K and V rows of the new tokens -> the KV segment that covers each token
//   (quantized state: one warp per row quantizes it -- hipfire, section 02,
//   table "State formats": fp8 = E4M3 codes with an f16 scale per head and
//   token, scale = f16(amax / 448), code = nearest E4M3 to x / scale, ties
//   to even, saturated at 448; q8 = Q8_0, int8 codes with an f16 scale per
//   block of 32, scale = f16(amax / 127), code = nearest integer to
//   x / scale, halves away from zero, within +-127; all in binary32);
//   index keys of the new tokens  -> the index-key cache;
//   pooled keys of every block a new token completes -> pooled, averaging
//   the block's four index keys in the order ((k0 + k1) + k2) + k3, x 0.25
//   (the pooling kernel's arithmetic), reading the keys of new tokens from
//   the input and those of earlier tokens from the cache, so no item reads
//   what another item of the launch writes.
#include <cuda_fp16.h>

#include "qsa_internal.cuh"

namespace qsa {

namespace {

__device__ __forceinline__ float4 load_key4(const void* base, int dtype, int64_t row, int64_t stride, int d) {
  if (dtype == QSA_F32) return *reinterpret_cast<const float4*>(static_cast<const float*>(base) + row * stride + d);
  const uint2 w = *reinterpret_cast<const uint2*>(static_cast<const __nv_bfloat16*>(base) + row * stride + d);
  return make_float4(bf16_lo(w.x), bf16_hi(w.x), bf16_lo(w.y), bf16_hi(w.y));
}

// Two binary32 values -> two E4M3 codes (x0 in the low byte), nearest with
// ties to even, saturated at +-448.
__device__ __forceinline__ uint32_t f32x2_to_e4m3x2(float x0, float x1) {
  unsigned short r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(x1), "f"(x0));
  return r;
}

__device__ __forceinline__ const AppendSeg* seg_of(const AppendParams& p, int64_t t) {
  for (int s = 0; s < p.n_segs; ++s)
    if (t >= p.seg[s].first && t < p.seg[s].first + p.seg[s].n) return &p.seg[s];
  return nullptr;
}

// One warp quantizes one bf16 row of D values (8 per lane at D = 256) into
// codes and its f16 scale.
__device__ __forceinline__ void quantize_row(const AppendParams& p, int64_t row, int lane) {
  const int which = (int)(row / ((int64_t)p.n_kv_heads * p.n_new));   // 0: K, 1: V
  const int64_t hr = row % ((int64_t)p.n_kv_heads * p.n_new);
  const int h = (int)(hr / p.n_new);
  const int64_t j = hr % p.n_new;
  const int64_t t = p.n_tokens - p.n_new + j;
  const int per = p.head_dim / 32;                                      // 8 or 4 values per lane
  const __nv_bfloat16* src = static_cast<const __nv_bfloat16*>(which ? p.v_new : p.k_new) +
                             ((int64_t)h * p.n_new + j) * p.head_dim + lane * per;
  float x[8];
  if (per == 8) {
    const uint4 w = *reinterpret_cast<const uint4*>(src);
    const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      x[2 * k] = bf16_lo(u[k]);
      x[2 * k + 1] = bf16_hi(u[k]);
    }
  } else {
    const uint2 w = *reinterpret_cast<const uint2*>(src);
    x[0] = bf16_lo(w.x);
    x[1] = bf16_hi(w.x);
    x[2] = bf16_lo(w.y);
    x[3] = bf16_hi(w.y);
#pragma unroll
    for (int k = 4; k < 8; ++k) x[k] = 0.f;
  }
  float amax = 0.f;
#pragma unroll
  for (int k = 0; k < 8; ++k) amax = fmaxf(amax, fabsf(x[k]));
  // fp8: the whole row (all 32 lanes); q8: the lane's block of 32 elements
  // (32 / per lanes, aligned).
  const int span = p.kvq == 1 ? 32 : 32 / per;
  for (int o = 1; o < span; o <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  const __half sh = __float2half_rn(__fdiv_rn(amax, p.kvq == 1 ? 448.0f : 127.0f));
  const float sc = __half2float(sh);
  uint32_t c[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    if (sc == 0.f) {
      c[k] = 0u;
    } else if (p.kvq == 1) {
      c[k] = f32x2_to_e4m3x2(__fdiv_rn(x[2 * k], sc), __fdiv_rn(x[2 * k + 1], sc));
    } else {
      const float a = fminf(127.f, fmaxf(-127.f, roundf(__fdiv_rn(x[2 * k], sc))));
      const float b = fminf(127.f, fmaxf(-127.f, roundf(__fdiv_rn(x[2 * k + 1], sc))));
      c[k] = ((uint32_t)(int)a & 0xffu) | (((uint32_t)(int)b & 0xffu) << 8);
    }
  }
  const AppendSeg* sg = seg_of(p, t);
  if (!sg) return;
  uint8_t* dst = static_cast<uint8_t*>(which ? sg->v : sg->k) + (int64_t)h * sg->head_stride +
                 (t - sg->first) * sg->tok_stride + lane * per;
  if (per == 8)
    *reinterpret_cast<uint2*>(dst) = make_uint2(c[0] | (c[1] << 16), c[2] | (c[3] << 16));
  else
    *reinterpret_cast<uint32_t*>(dst) = c[0] | (c[1] << 16);
  const int rec_bytes = p.kvq == 1 ? 4 : p.head_dim / 8;
  __half* rec = reinterpret_cast<__half*>(static_cast<uint8_t*>(sg->kv_scale) +
                                          ((int64_t)h * sg->s_head_stride + (t - sg->first) * sg->s_tok_stride) *
                                              rec_bytes);
  if (p.kvq == 1) {
    if (lane == 0) rec[which] = sh;
  } else if (lane % span == 0) {
    rec[which * (p.head_dim / 32) + lane / span] = sh;
  }
}

__global__ void __launch_bounds__(256) append_kernel(const AppendParams p) {
  // Writes what earlier launches of the stream may read: wait for them first.
  grid_dependency_wait();
  grid_dependency_release();
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int64_t first_new = p.n_tokens - p.n_new;
  if (p.kvq && i < p.kv_items) {   // a whole warp per row (kv_items is a multiple of 32)
    quantize_row(p, i / 32, (int)(i % 32));
    return;
  }
  if (i < p.kv_items + p.idx_items) {
    append_copy(p, i);
    return;
  }
  const int64_t i2 = i - p.kv_items;
  const int64_t i3 = i2 - p.idx_items;
  if (i3 < p.pool_items) {
    const int64_t b = p.first_block + i3 / (QSA_INDEX_DIM / 4);
    const int d = (int)(i3 % (QSA_INDEX_DIM / 4)) * 4;
    float4 k[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int64_t t = 4 * b + q;
      k[q] = t >= first_new ? load_key4(p.idx_new, p.idx_dtype, t - first_new, QSA_INDEX_DIM, d)
                            : load_key4(p.idx_keys, p.idx_dtype, t, p.idx_stride, d);
    }
    float4 m;
    m.x = (((k[0].x + k[1].x) + k[2].x) + k[3].x) * 0.25f;
    m.y = (((k[0].y + k[1].y) + k[2].y) + k[3].y) * 0.25f;
    m.z = (((k[0].z + k[1].z) + k[2].z) + k[3].z) * 0.25f;
    m.w = (((k[0].w + k[1].w) + k[2].w) + k[3].w) * 0.25f;
    *reinterpret_cast<float4*>(p.pooled + b * p.pooled_stride + d) = m;
  }
}

}  // namespace

cudaError_t launch_append(const AppendParams& p, cudaStream_t st) {
  const int64_t items = p.kv_items + p.idx_items + p.pool_items;
  if (items == 0) return cudaSuccess;
  const int64_t grid = (items + 255) / 256;
  return launch_kernel(append_kernel, dim3((unsigned)grid), dim3(256), 0, st, 0u, p);
}

}  // namespace qsa
