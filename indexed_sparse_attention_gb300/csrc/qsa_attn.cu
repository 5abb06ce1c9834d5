// Steps 4 and 5 of the QSA layer step: exact softmax attention over only the
// selected rows, grouped-query, split over each row's selected list and
// merged by log-sum-exp.
//   hipfire, "QSA sparse attention and the VMM KV backend", section 02 (full
//   attention over the selected rows plus the incomplete tail block, at most
//   2,048 + 3 per query) and section 03 (one workgroup per KV group of 12
//   query heads, so each selected K/V row is read once);
//   MTPLX pull request #610 (attention over up to 12 KV segments in one
//   launch, partials merged by their log-sum-exp; rows with no visible key
//   merge to zeros; fp32 partials rounded once).
//
// One CTA per (query row, KV group, split): a split walks its share of the
// row's selected list (the 4 tokens of each selected block, then the tail) in
// tiles of 32 tokens -- split s of n takes tiles [s T / n, (s + 1) T / n) of
// the T tiles of the row's longest possible list -- and each token is located in the sequence's segment table
// and its K and V rows are gathered into shared memory with cp.async.  bf16
// K/V run on the tensor pipe (mma.sync m16n8k16: the 12 heads of a group
// padded to 16 rows against 32 gathered tokens) with an fp32 online softmax;
// fp32 K/V take a CUDA-core kernel.  A split writes its normalised partial
// output and lse; a second launch merges the splits by log-sum-exp (step 5,
// the kernel behind qsa_lse_merge).  A row with a single split is written
// directly.
#include <math.h>

#include <algorithm>

#include <cuda_fp16.h>

#include "qsa_attn_common.cuh"

namespace qsa {

namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr int kMaxSplits = 256;  // splits of one (row, KV group)

using namespace attn;

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ void ldsm_x4(uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3, const void* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(smem_u32(p)));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3, const void* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(smem_u32(p)));
}

__device__ __forceinline__ void mma_bf16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// ------------------------------------------------------------------ a split's result
// Normalised output and natural-log lse of one (row, head): to the final
// output when the row has a single split, else to the split's partial slot
// ([split][row * Hq + head][D] and [split][row * Hq + head], the layout of
// qsa_lse_merge's inputs).
template <int NSEQ>
__device__ __forceinline__ void store_result(const AttnParams<NSEQ>& p, int split, int r, int head, int d, float x0,
                                             float x1) {
  const int64_t rh = (int64_t)r * p.n_q_heads + head;
  if (p.n_splits == 1) {
    if (p.out_dtype == QSA_F32) {
      *reinterpret_cast<float2*>(static_cast<float*>(p.out) + rh * p.head_dim + d) = make_float2(x0, x1);
    } else {
      *reinterpret_cast<__nv_bfloat162*>(static_cast<__nv_bfloat16*>(p.out) + rh * p.head_dim + d) =
          __floats2bfloat162_rn(x0, x1);
    }
  } else {
    const int64_t R = (int64_t)p.total_rows * p.n_q_heads;
    *reinterpret_cast<float2*>(p.part_o + ((int64_t)split * R + rh) * p.head_dim + d) = make_float2(x0, x1);
  }
}

template <int NSEQ>
__device__ __forceinline__ void store_lse(const AttnParams<NSEQ>& p, int split, int r, int head, float lse) {
  const int64_t rh = (int64_t)r * p.n_q_heads + head;
  if (p.n_splits == 1) {
    if (p.lse) p.lse[rh] = lse;
  } else {
    p.part_lse[(int64_t)split * p.total_rows * p.n_q_heads + rh] = lse;
  }
}

// ------------------------------------------------------------------ tensor-pipe kernel (bf16 K/V)
// 8 warps.  Per 32-token tile: warp w computes the logits of tokens
// 8(w%4)..8(w%4)+7 over half w/4 of the channels (the two halves are added
// in shared memory), then softmax rows w and w+8, then P.V for channels
// [w*D/8, (w+1)*D/8).
constexpr int kTT = 32;        // tokens per tile
constexpr int kPStride = 40;   // bf16 per P row: 80-byte rows keep ldmatrix conflict-free
constexpr int kSStride = kTT + 4;
constexpr int kAttnThreads = 256;

// KVQ (quantized state): 1 = fp8 (E4M3 codes, one (K, V) scale pair per
// token), 2 = q8 (int8 codes, an f16 scale per 32 elements of each row).
// Each stage holds the codes (1 byte per element) and the tokens' scale
// records; the stage being consumed is converted to bf16 into one tile of the
// bf16 layout before the MMAs.
template <int D, int STAGES, int KVQ = 0>
struct MmaSmem {
  static constexpr bool F8 = KVQ != 0;
  static constexpr int kRec = KVQ == 1 ? 4 : KVQ == 2 ? D / 8 : 0;   // scale record bytes per token
  static constexpr int CH = D / 8;                     // 16-byte chunks per bf16 K/V/Q row
  static constexpr size_t q = 16 * D * 2;
  static constexpr size_t kv_tile = kTT * D * (F8 ? 1 : 2);   // one K or V tile as gathered
  static constexpr size_t s = 2 * 16 * kSStride * 4;   // logits, one plane per channel half
  static constexpr size_t pm = 16 * kPStride * 2;
  static constexpr size_t off_kv = q;                  // [STAGES][K tile, V tile]
  static constexpr size_t off_bf = off_kv + STAGES * 2 * kv_tile;   // fp8: the converted K, V tile
  static constexpr size_t off_s = off_bf + (F8 ? 2 * kTT * D * 2 : 0);
  static constexpr size_t off_p = off_s + s;
  static constexpr size_t off_m = off_p + pm;          // m, l, alpha: 3 x 16 floats
  static constexpr size_t off_valid = off_m + 3 * 16 * 4;
  static constexpr size_t off_sc = off_valid + STAGES * kTT * 4;   // scale records per stage
  static constexpr size_t off_ids = off_sc + (size_t)STAGES * kTT * kRec;
  static constexpr size_t bytes = off_ids + kIdCache * 4;
  // Three stages keep two CTAs per SM (228 KB per SM, 1 KB reserved per CTA).
  static_assert(STAGES != 3 || 2 * (bytes + 1024) <= 228 * 1024, "two CTAs per SM");
};

template <int D, int STAGES, int NSEQ, int KVQ = 0>
__global__ void __launch_bounds__(kAttnThreads, STAGES <= 3 ? 2 : 1) attn_mma_kernel(const AttnParams<NSEQ> p) {
  using L = MmaSmem<D, STAGES, KVQ>;
  constexpr bool F8 = KVQ != 0;
  constexpr int CH = L::CH;
  constexpr int KH = D / 32;   // k-steps (16 channels each) per channel half
  constexpr int NTD = D / 64;  // 8-channel n-tiles per warp in P.V
  extern __shared__ __align__(128) uint8_t smem[];
  __nv_bfloat16* q_s = reinterpret_cast<__nv_bfloat16*>(smem);
  __nv_bfloat16* kv_s = reinterpret_cast<__nv_bfloat16*>(smem + L::off_kv);
  float* s_s = reinterpret_cast<float*>(smem + L::off_s);
  __nv_bfloat16* p_s = reinterpret_cast<__nv_bfloat16*>(smem + L::off_p);
  float* m_s = reinterpret_cast<float*>(smem + L::off_m);
  float* l_s = m_s + 16;
  float* a_s = m_s + 32;
  int* valid_s = reinterpret_cast<int*>(smem + L::off_valid);
  int32_t* ids_s = reinterpret_cast<int32_t*>(smem + L::off_ids);
  uint8_t* kv8_s = smem + L::off_kv;                                        // fp8 stages
  __nv_bfloat16* kvb_s = reinterpret_cast<__nv_bfloat16*>(smem + L::off_bf);   // fp8: converted tile
  uint8_t* sc_s = smem + L::off_sc;                                         // scale records

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int quarter = warp & 3, half = warp >> 2;
  const int split = blockIdx.x, g = blockIdx.y, r = p.row_base + blockIdx.z;
  const int G = p.group, head0 = g * G;
  RowCtx c = make_row_ctx(p, r);
  int64_t i0, i1;
  split_range(c, split, p.n_splits, i0, i1);
  const int n_tiles = i1 > i0 ? (int)((i1 - i0 + kTT - 1) / kTT) : 0;
  const __nv_bfloat16* qg = static_cast<const __nv_bfloat16*>(p.q) + ((int64_t)r * p.n_q_heads + head0) * D;

  // Q of the group's heads, read while the split's block ids are staged.
  uint4 qv[(16 * CH + kAttnThreads - 1) / kAttnThreads];
#pragma unroll
  for (int k = 0; k < (16 * CH + kAttnThreads - 1) / kAttnThreads; ++k) {
    const int idx = tid + k * kAttnThreads;
    const int row = idx / CH, ch = idx % CH;
    qv[k] = make_uint4(0u, 0u, 0u, 0u);
    if (idx < 16 * CH && row < G) qv[k] = *reinterpret_cast<const uint4*>(qg + (int64_t)row * D + ch * 8);
  }
  // Q is an input of the step that no earlier launch of the step writes: its
  // loads above are issued before the wait for the selection.
  grid_dependency_wait();
  grid_dependency_release();
  const int32_t cnt_loaded = __ldg(p.cnt + r);   // in flight with the ids
  const IdCache ic = stage_ids(c, i0, i1, ids_s);
  set_count(c, cnt_loaded, p.sel_ld);
  __syncthreads();

  // Gather of one tile into a stage: thread -> token slot tid/8, chunks (tid&7) + 8j,
  // swizzled: chunk c of token row t lands at c ^ (t & 7).
  auto load_tile = [&](int it, int stage) {
    const int tk = tid >> 3, q8 = tid & 7;
    const int64_t i = i0 + (int64_t)it * kTT + tk;
    int seg = 0;
    int64_t off = 0, tseg = 0;
    const bool ok = i < i1 && locate(p, c, ic, i, g, seg, off, &tseg);
    if constexpr (F8) {
      // Codes of the token's K and V rows (D bytes each) into the stage, row
      // after row; the (K, V) scale pair of (head g, token) beside them.
      const uint8_t* ks = ok ? static_cast<const uint8_t*>(p.seg[seg].k) + off : static_cast<const uint8_t*>(p.q);
      const uint8_t* vs = ok ? static_cast<const uint8_t*>(p.seg[seg].v) + off : static_cast<const uint8_t*>(p.q);
      uint8_t* kd = kv8_s + (size_t)stage * 2 * L::kv_tile + tk * D;
      uint8_t* vd = kd + L::kv_tile;
#pragma unroll
      for (int j = 0; j < D / 128; ++j) {
        const int ch = 8 * j + q8;
        cp_async16(kd + ch * 16, ks + (ok ? ch * 16 : 0), ok);
        cp_async16(vd + ch * 16, vs + (ok ? ch * 16 : 0), ok);
      }
      const uint8_t* sp = ok ? p.seg[seg].kv_scale +
                                   ((int64_t)g * p.seg[seg].s_head_stride + tseg * p.seg[seg].s_tok_stride) * L::kRec
                             : static_cast<const uint8_t*>(p.q);
      uint8_t* sd = sc_s + (size_t)(stage * kTT + tk) * L::kRec;
      if constexpr (KVQ == 1) {
        if (q8 == 0) cp_async4(sd, sp, ok);
      } else {
        if (q8 < L::kRec / 16) cp_async16(sd + q8 * 16, sp + (ok ? q8 * 16 : 0), ok);
      }
      if (q8 == 0) valid_s[stage * kTT + tk] = ok ? 1 : 0;
      return;
    }
    const __nv_bfloat16* ks = ok ? static_cast<const __nv_bfloat16*>(p.seg[seg].k) + off : qg;
    const __nv_bfloat16* vs = ok ? static_cast<const __nv_bfloat16*>(p.seg[seg].v) + off : qg;
    __nv_bfloat16* kd = kv_s + (size_t)stage * 2 * kTT * D + tk * D;
    __nv_bfloat16* vd = kd + kTT * D;
    // The four tokens of a warp write different 128-byte segments (bank-conflict free).
#pragma unroll
    for (int j = 0; j < CH / 8; ++j) {
      const int ch = 8 * ((j + tk) % (CH / 8)) + q8;
      const int pc = ch ^ (tk & 7);
      cp_async16(kd + pc * 8, ks + (ok ? ch * 8 : 0), ok);
      cp_async16(vd + pc * 8, vs + (ok ? ch * 8 : 0), ok);
    }
    if (q8 == 0) valid_s[stage * kTT + tk] = ok ? 1 : 0;
  };

  // Put every stage's gather in flight first (one commit group per stage).
#pragma unroll
  for (int st = 0; st < STAGES; ++st) {
    if (st < n_tiles) load_tile(st, st);
    cp_async_commit();
  }

  // Q of the group's heads (rows >= G zero), swizzled like the K/V tiles.
#pragma unroll
  for (int k = 0; k < (16 * CH + kAttnThreads - 1) / kAttnThreads; ++k) {
    const int idx = tid + k * kAttnThreads;
    const int row = idx / CH, ch = idx % CH;
    if (idx < 16 * CH) *reinterpret_cast<uint4*>(q_s + (row * CH + (ch ^ (row & 7))) * 8) = qv[k];
  }
  for (int idx = tid; idx < 16 * kPStride; idx += kAttnThreads) p_s[idx] = __float2bfloat16(0.f);
  if (tid < 16) {
    m_s[tid] = -INFINITY;
    l_s[tid] = 0.f;
    a_s[tid] = 1.f;
  }
  __syncthreads();
  uint32_t qf[KH][4];
#pragma unroll
  for (int i = 0; i < KH; ++i) {
    const int row = (lane & 7) + 8 * ((lane >> 3) & 1);
    const int ch = 2 * (half * KH + i) + (lane >> 4);
    ldsm_x4(qf[i][0], qf[i][1], qf[i][2], qf[i][3], q_s + (row * CH + (ch ^ (row & 7))) * 8);
  }

  float o[NTD][4];
#pragma unroll
  for (int j = 0; j < NTD; ++j) o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.f;
  const float zscale = p.scale * kLog2e;
  const int gq = lane >> 2, t4 = lane & 3;

  // Commit groups: tile t < STAGES is group t (prologue); iteration j >= 1
  // commits group STAGES + j - 1 holding tile STAGES + j - 1.  So tile t is
  // group t, and at the top of iteration it the groups after it that may
  // still be pending number STAGES - 1 (it = 0) or STAGES - 2 (it >= 1).
  for (int it = 0; it < n_tiles; ++it) {
    const int stage = it % STAGES;
    if (it == 0) cp_async_wait<STAGES - 1>();
    else cp_async_wait<STAGES - 2>();
    __syncthreads();
    // Every thread is past tile it-1: its stage takes tile it-1+STAGES.
    if (it >= 1) {
      if (it - 1 + STAGES < n_tiles) load_tile(it - 1 + STAGES, (it - 1) % STAGES);
      cp_async_commit();
    }
    const __nv_bfloat16* kt = kv_s + (size_t)stage * 2 * kTT * D;
    if constexpr (F8) {
      // Codes -> bf16 into the swizzled layout the MMAs read: output chunk ch
      // (8 elements) of row tk sits at chunk ch ^ (tk & 7).
      const uint8_t* src = kv8_s + (size_t)stage * 2 * L::kv_tile;
#pragma unroll
      for (int k = 0; k < 2 * kTT * CH / kAttnThreads; ++k) {
        const int job = tid + k * kAttnThreads;
        const int kv = job / (kTT * CH), rem = job % (kTT * CH);
        const int tk = rem / CH, ch = rem % CH;
        const uint2 w = *reinterpret_cast<const uint2*>(src + kv * L::kv_tile + tk * D + ch * 8);
        uint4 o;
        if constexpr (KVQ == 1) {
          o.x = e4m3x2_to_bf16x2(w.x & 0xffffu);
          o.y = e4m3x2_to_bf16x2(w.x >> 16);
          o.z = e4m3x2_to_bf16x2(w.y & 0xffffu);
          o.w = e4m3x2_to_bf16x2(w.y >> 16);
        } else {
          // q8: code x the scale of its 32-element block (chunk ch lies in block ch / 4),
          // rounded once to bf16.
          const __half* rec = reinterpret_cast<const __half*>(sc_s + (size_t)(stage * kTT + tk) * L::kRec);
          const float d = __half2float(rec[kv * (D / 32) + ch / 4]);
          i8x4_to_bf16x4(w.x, d, o.x, o.y);
          i8x4_to_bf16x4(w.y, d, o.z, o.w);
        }
        *reinterpret_cast<uint4*>(kvb_s + (size_t)kv * kTT * D + (tk * CH + (ch ^ (tk & 7))) * 8) = o;
      }
      __syncthreads();
      kt = kvb_s;
    }
    const __nv_bfloat16* vt = kt + kTT * D;
    // Partial logits of tokens 8*quarter.. over this warp's channel half, two chains.
    {
      float sa[4] = {0.f, 0.f, 0.f, 0.f}, sb[4] = {0.f, 0.f, 0.f, 0.f};
      const int tk = 8 * quarter + (lane & 7);
#pragma unroll
      for (int i = 0; i < KH; i += 2) {
        uint32_t b0, b1, b2, b3;
        const int ch = 2 * (half * KH + i) + (lane >> 3);
        ldsm_x4(b0, b1, b2, b3, kt + (tk * CH + (ch ^ (tk & 7))) * 8);
        mma_bf16(sa, qf[i], b0, b1);
        mma_bf16(sb, qf[i + 1], b2, b3);
      }
      float* sp = s_s + half * 16 * kSStride;
      const int col = 8 * quarter + 2 * t4;
      *reinterpret_cast<float2*>(sp + gq * kSStride + col) = make_float2(sa[0] + sb[0], sa[1] + sb[1]);
      *reinterpret_cast<float2*>(sp + (gq + 8) * kSStride + col) = make_float2(sa[2] + sb[2], sa[3] + sb[3]);
    }
    __syncthreads();
    // Online softmax of rows warp and warp+8 (base-2 logits), one lane per token.
    {
      const bool valid = valid_s[stage * kTT + lane] != 0;
      float kscale = 1.f, vscale = 1.f;
      if constexpr (KVQ == 1) {
        const uint32_t pr = *reinterpret_cast<const uint32_t*>(sc_s + (stage * kTT + lane) * 4);
        kscale = __half2float(__ushort_as_half((unsigned short)(pr & 0xffffu)));
        vscale = __half2float(__ushort_as_half((unsigned short)(pr >> 16)));
      }
      float z[2], mo[2], mx[2];
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const int rr = warp + 8 * j;
        z[j] = -INFINITY;
        mo[j] = -INFINITY;
        if (rr < G) {
          const float s0 = s_s[rr * kSStride + lane] + s_s[16 * kSStride + rr * kSStride + lane];
          z[j] = valid ? s0 * kscale * zscale : -INFINITY;
          mo[j] = m_s[rr];
        }
        mx[j] = z[j];
      }
#pragma unroll
      for (int off = 16; off; off >>= 1) {
        mx[0] = fmaxf(mx[0], __shfl_xor_sync(0xffffffffu, mx[0], off));
        mx[1] = fmaxf(mx[1], __shfl_xor_sync(0xffffffffu, mx[1], off));
      }
      float pz[2], sm[2];
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const float mn = fmaxf(mo[j], mx[j]);
        pz[j] = mn == -INFINITY ? 0.f : exp2f(z[j] - mn);
        sm[j] = pz[j];
        mx[j] = mn;
      }
#pragma unroll
      for (int off = 16; off; off >>= 1) {
        sm[0] += __shfl_xor_sync(0xffffffffu, sm[0], off);
        sm[1] += __shfl_xor_sync(0xffffffffu, sm[1], off);
      }
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const int rr = warp + 8 * j;
        if (rr < G) {
          p_s[rr * kPStride + lane] = __float2bfloat16(KVQ == 1 ? pz[j] * vscale : pz[j]);
          if (lane == 0) {
            const float alpha = mo[j] == -INFINITY ? 0.f : exp2f(mo[j] - mx[j]);
            a_s[rr] = alpha;
            m_s[rr] = mx[j];
            l_s[rr] = l_s[rr] * alpha + sm[j];
          }
        }
      }
    }
    __syncthreads();
    // O += P V over channels [warp*D/8, (warp+1)*D/8).
    {
      const float al0 = gq < G ? a_s[gq] : 1.f, al1 = gq + 8 < G ? a_s[gq + 8] : 1.f;
#pragma unroll
      for (int j = 0; j < NTD; ++j) {
        o[j][0] *= al0;
        o[j][1] *= al0;
        o[j][2] *= al1;
        o[j][3] *= al1;
      }
#pragma unroll
      for (int kk = 0; kk < kTT / 16; ++kk) {
        uint32_t pa[4];
        {
          const int row = (lane & 7) + 8 * ((lane >> 3) & 1);
          const int ch = 2 * kk + (lane >> 4);
          ldsm_x4(pa[0], pa[1], pa[2], pa[3], p_s + row * kPStride + ch * 8);
        }
        const int tk = kk * 16 + (lane & 7) + 8 * ((lane >> 3) & 1);
#pragma unroll
        for (int j = 0; j < NTD; j += 2) {
          const int ch = warp * NTD + j + (lane >> 4);
          uint32_t b0, b1, b2, b3;
          ldsm_x4_t(b0, b1, b2, b3, vt + (tk * CH + (ch ^ (tk & 7))) * 8);
          mma_bf16(o[j], pa, b0, b1);
          mma_bf16(o[j + 1], pa, b2, b3);
        }
      }
    }
  }
  cp_async_wait<0>();
  __syncthreads();

  // Normalised result of heads gq and gq + 8 over this warp's channels.
#pragma unroll
  for (int hf = 0; hf < 2; ++hf) {
    const int row = gq + 8 * hf;
    if (row >= G) continue;
    const float l = l_s[row];
    const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll
    for (int j = 0; j < NTD; ++j) {
      const int d = warp * (D / 8) + j * 8 + 2 * t4;
      store_result(p, split, r, head0 + row, d, o[j][2 * hf] * inv, o[j][2 * hf + 1] * inv);
    }
    if (warp == 0 && t4 == 0) store_lse(p, split, r, head0 + row, l > 0.f ? (m_s[row] + log2f(l)) * kLn2 : -INFINITY);
  }
}

// ------------------------------------------------------------------ CUDA-core kernel (fp32 K/V)
// Thread -> channel d = tid % D and heads hs, hs + HS, ... (HS = 256 / D).
constexpr int kSimtTT = 32;

template <int D>
struct SimtSmem {
  static constexpr size_t q = 16 * D;                 // floats
  static constexpr size_t k = kSimtTT * (D + 1);
  static constexpr size_t v = kSimtTT * D;
  static constexpr size_t z = 16 * 33;
  static constexpr size_t floats = q + k + v + z + 3 * 16;
  static constexpr size_t bytes = floats * 4 + kSimtTT * 4 + kIdCache * 4;
};

template <int D, int NSEQ>
__global__ void __launch_bounds__(256) attn_simt_kernel(const AttnParams<NSEQ> p) {
  using L = SimtSmem<D>;
  constexpr int HS = 256 / D;
  constexpr int MAXH = 16 / HS;
  extern __shared__ __align__(16) float fsm[];
  float* q_s = fsm;                          // [16][D]
  float* k_s = q_s + L::q;                   // [32][D+1]
  float* v_s = k_s + L::k;                   // [32][D]
  float* z_s = v_s + L::v;                   // [16][33]
  float* m_s = z_s + L::z;
  float* l_s = m_s + 16;
  float* a_s = l_s + 16;
  int* ok_s = reinterpret_cast<int*>(a_s + 16);
  int32_t* ids_s = ok_s + kSimtTT;
  grid_dependency_sync();

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int split = blockIdx.x, g = blockIdx.y, r = p.row_base + blockIdx.z;
  const int G = p.group, head0 = g * G;
  RowCtx c = make_row_ctx(p, r);
  const int32_t cnt_loaded = __ldg(p.cnt + r);
  int64_t i0, i1;
  split_range(c, split, p.n_splits, i0, i1);
  const float zscale = p.scale * kLog2e;
  const IdCache ic = stage_ids(c, i0, i1, ids_s);
  set_count(c, cnt_loaded, p.sel_ld);

  const float* qg = static_cast<const float*>(p.q) + ((int64_t)r * p.n_q_heads + head0) * D;
  for (int idx = tid; idx < G * D; idx += 256) q_s[idx] = qg[idx];
  if (tid < 16) {
    m_s[tid] = -INFINITY;
    l_s[tid] = 0.f;
  }
  const int d = tid % D, hs = tid / D;
  float acc[MAXH];
#pragma unroll
  for (int j = 0; j < MAXH; ++j) acc[j] = 0.f;
  __syncthreads();

  for (int64_t base = i0; base < i1; base += kSimtTT) {
    const int nt = (int)((i1 - base) < (int64_t)kSimtTT ? (i1 - base) : (int64_t)kSimtTT);
    for (int tk = warp; tk < kSimtTT; tk += 8) {
      int seg = 0;
      int64_t off = 0;
      const bool ok = tk < nt && locate(p, c, ic, base + tk, g, seg, off);
      const float* ks = ok ? static_cast<const float*>(p.seg[seg].k) + off : nullptr;
      const float* vs = ok ? static_cast<const float*>(p.seg[seg].v) + off : nullptr;
      for (int dd = lane; dd < D; dd += 32) {
        k_s[tk * (D + 1) + dd] = ok ? ks[dd] : 0.f;
        v_s[tk * D + dd] = ok ? vs[dd] : 0.f;
      }
      if (lane == 0) ok_s[tk] = ok ? 1 : 0;
    }
    __syncthreads();
    for (int pr = tid; pr < G * kSimtTT; pr += 256) {
      const int hh = pr / kSimtTT, tk = pr % kSimtTT;
      float dot = 0.f;
      for (int dd = 0; dd < D; ++dd) dot = fmaf(q_s[hh * D + dd], k_s[tk * (D + 1) + dd], dot);
      z_s[hh * 33 + tk] = ok_s[tk] ? dot * zscale : -INFINITY;
    }
    __syncthreads();
    for (int hh = warp; hh < G; hh += 8) {
      const float z = z_s[hh * 33 + lane];
      const float mo = m_s[hh];
      const float mn = fmaxf(mo, warp_max(z));
      const float pz = mn == -INFINITY ? 0.f : exp2f(z - mn);
      const float sum = warp_sum(pz);
      z_s[hh * 33 + lane] = pz;
      if (lane == 0) {
        const float alpha = mo == -INFINITY ? 0.f : exp2f(mo - mn);
        a_s[hh] = alpha;
        m_s[hh] = mn;
        l_s[hh] = l_s[hh] * alpha + sum;
      }
    }
    __syncthreads();
#pragma unroll
    for (int j = 0; j < MAXH; ++j) {
      const int hh = hs + j * HS;
      if (hh < G) {
        float a = acc[j] * a_s[hh];
        for (int tk = 0; tk < kSimtTT; ++tk) a = fmaf(z_s[hh * 33 + tk], v_s[tk * D + d], a);
        acc[j] = a;
      }
    }
    __syncthreads();
  }
#pragma unroll
  for (int j = 0; j < MAXH; ++j) {
    const int hh = hs + j * HS;
    if (hh >= G) continue;
    const float l = l_s[hh];
    const float x = l > 0.f ? acc[j] / l : 0.f;
    const int64_t rh = (int64_t)r * p.n_q_heads + head0 + hh;
    if (p.n_splits == 1) {
      if (p.out_dtype == QSA_F32) static_cast<float*>(p.out)[rh * D + d] = x;
      else static_cast<__nv_bfloat16*>(p.out)[rh * D + d] = __float2bfloat16(x);
    } else {
      p.part_o[((int64_t)split * p.total_rows * p.n_q_heads + rh) * D + d] = x;
    }
    if (d == 0) store_lse(p, split, r, head0 + hh, l > 0.f ? (m_s[hh] + log2f(l)) * kLn2 : -INFINITY);
  }
}

// ------------------------------------------------------------------ step 5: merge of split partials
// One CTA of 8 warps per (row, head) when head_dim is 128 or 256: warp w
// takes partials w, w + 8, ...; lane l accumulates channels [l*CPL, (l+1)*CPL)
// of each, weighted by 2^(lse_s - m_w) against its own running maximum; the
// warps then combine in shared memory by the same rule.  Every load of a warp
// is independent of its other loads.
constexpr int kMergeWarps = 8;
constexpr int kMergeBatch = 8;   // partials a warp loads per pass

template <int CPL>   // channels per lane (4 or 8)
__global__ void __launch_bounds__(kMergeWarps * 32) merge_cta_kernel(const float* __restrict__ o_parts,
                                                                     const float* __restrict__ lse_parts,
                                                                     int n_parts, int64_t n_rows, int head_dim,
                                                                     void* __restrict__ out, int out_dtype,
                                                                     float* __restrict__ lse_out) {
  __shared__ float acc_s[kMergeWarps][32 * CPL];
  __shared__ float m_s[kMergeWarps], w_s[kMergeWarps];
  grid_dependency_sync();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t row = blockIdx.x;
  const int d0 = lane * CPL;
  // This warp's partials w, w + 8, ..., eight per pass: their lse values and
  // channels are loaded together (one round trip for up to 64 partials), then
  // added with an online rescale to the warp's running maximum m.
  float m = -INFINITY, wsum = 0.f;
  float acc[CPL];
#pragma unroll
  for (int c = 0; c < CPL; ++c) acc[c] = 0.f;
  for (int s0 = warp; s0 < n_parts; s0 += kMergeWarps * kMergeBatch) {
    float ls[kMergeBatch];
    float4 v[kMergeBatch][CPL / 4];
#pragma unroll
    for (int k = 0; k < kMergeBatch; ++k) {
      const int s = s0 + k * kMergeWarps;
      ls[k] = s < n_parts ? __ldg(lse_parts + (int64_t)s * n_rows + row) : -INFINITY;
#pragma unroll
      for (int c = 0; c < CPL / 4; ++c)
        v[k][c] = s < n_parts
                      ? __ldg(reinterpret_cast<const float4*>(o_parts + ((int64_t)s * n_rows + row) * head_dim + d0) + c)
                      : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    float mn = m;
#pragma unroll
    for (int k = 0; k < kMergeBatch; ++k) mn = fmaxf(mn, ls[k]);
    if (mn == -INFINITY) continue;
    const float rescale = m == -INFINITY ? 0.f : exp2f((m - mn) * kLog2e);
    wsum *= rescale;
#pragma unroll
    for (int c = 0; c < CPL; ++c) acc[c] *= rescale;
#pragma unroll
    for (int k = 0; k < kMergeBatch; ++k) {
      if (ls[k] == -INFINITY) continue;   // drops the values of a partial without keys
      const float w = exp2f((ls[k] - mn) * kLog2e);
      wsum += w;
#pragma unroll
      for (int c = 0; c < CPL / 4; ++c) {
        acc[4 * c + 0] = fmaf(w, v[k][c].x, acc[4 * c + 0]);
        acc[4 * c + 1] = fmaf(w, v[k][c].y, acc[4 * c + 1]);
        acc[4 * c + 2] = fmaf(w, v[k][c].z, acc[4 * c + 2]);
        acc[4 * c + 3] = fmaf(w, v[k][c].w, acc[4 * c + 3]);
      }
    }
    m = mn;
  }
#pragma unroll
  for (int c = 0; c < CPL; ++c) acc_s[warp][d0 + c] = acc[c];
  if (lane == 0) {
    m_s[warp] = m;
    w_s[warp] = wsum;
  }
  __syncthreads();
  if (warp != 0) return;
  float M = -INFINITY;
#pragma unroll
  for (int k = 0; k < kMergeWarps; ++k) M = fmaxf(M, m_s[k]);
  float f[kMergeWarps], W = 0.f;
#pragma unroll
  for (int k = 0; k < kMergeWarps; ++k) {
    f[k] = m_s[k] == -INFINITY ? 0.f : expf(m_s[k] - M);
    W += f[k] * w_s[k];
  }
  const float inv = W > 0.f ? 1.f / W : 0.f;
  float r[CPL];
#pragma unroll
  for (int c = 0; c < CPL; ++c) {
    float x = 0.f;
#pragma unroll
    for (int k = 0; k < kMergeWarps; ++k) x = fmaf(f[k], acc_s[k][d0 + c], x);
    r[c] = x * inv;
  }
  if (out_dtype == QSA_F32) {
    float* o = static_cast<float*>(out) + row * head_dim + d0;
#pragma unroll
    for (int c = 0; c < CPL / 4; ++c)
      reinterpret_cast<float4*>(o)[c] = make_float4(r[4 * c], r[4 * c + 1], r[4 * c + 2], r[4 * c + 3]);
  } else {
    __nv_bfloat162* o = reinterpret_cast<__nv_bfloat162*>(static_cast<__nv_bfloat16*>(out) + row * head_dim + d0);
#pragma unroll
    for (int c = 0; c < CPL / 2; ++c) o[c] = __floats2bfloat162_rn(r[2 * c], r[2 * c + 1]);
  }
  if (lane == 0 && lse_out) lse_out[row] = W > 0.f ? M + logf(W) : -INFINITY;
}

// Thread -> (row, 4 channels), for any head_dim that is a multiple of 4.
__global__ void __launch_bounds__(256) merge_kernel(const float* __restrict__ o_parts,
                                                     const float* __restrict__ lse_parts, int n_parts,
                                                     int64_t n_rows, int head_dim, void* __restrict__ out,
                                                     int out_dtype, float* __restrict__ lse_out) {
  grid_dependency_sync();
  const int q = head_dim / 4;
  const int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= n_rows * q) return;
  const int64_t row = idx / q;
  const int d = (int)(idx % q) * 4;
  float m = -INFINITY;
  for (int s0 = 0; s0 < n_parts; s0 += 8) {
    float l[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) l[j] = s0 + j < n_parts ? __ldg(lse_parts + (int64_t)(s0 + j) * n_rows + row) : -INFINITY;
#pragma unroll
    for (int j = 0; j < 8; ++j) m = fmaxf(m, l[j]);
  }
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  float wsum = 0.f;
  if (m != -INFINITY) {
    for (int s0 = 0; s0 < n_parts; s0 += 4) {
      float w[4];
      float4 v[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const bool in = s0 + j < n_parts;
        const float ls = in ? __ldg(lse_parts + (int64_t)(s0 + j) * n_rows + row) : -INFINITY;
        w[j] = ls == -INFINITY ? 0.f : expf(ls - m);
        v[j] = in && ls != -INFINITY
                   ? __ldg(reinterpret_cast<const float4*>(o_parts + ((int64_t)(s0 + j) * n_rows + row) * head_dim + d))
                   : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        wsum += w[j];
        acc.x = fmaf(w[j], v[j].x, acc.x);
        acc.y = fmaf(w[j], v[j].y, acc.y);
        acc.z = fmaf(w[j], v[j].z, acc.z);
        acc.w = fmaf(w[j], v[j].w, acc.w);
      }
    }
  }
  const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
  const float4 res = make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
  if (out_dtype == QSA_F32) {
    *reinterpret_cast<float4*>(static_cast<float*>(out) + row * head_dim + d) = res;
  } else {
    __nv_bfloat162* o2 = reinterpret_cast<__nv_bfloat162*>(static_cast<__nv_bfloat16*>(out) + row * head_dim + d);
    o2[0] = __floats2bfloat162_rn(res.x, res.y);
    o2[1] = __floats2bfloat162_rn(res.z, res.w);
  }
  if (d == 0 && lse_out) lse_out[row] = wsum > 0.f ? m + logf(wsum) : -INFINITY;
}

}  // namespace

static int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Splits per (row, KV group): about two CTAs per SM over the whole call, each
// split a whole number of 32-token tiles; one split for calls with enough
// rows (prefill).
AttnPlan attn_plan(qsa_dtype kv_dtype, int head_dim, int64_t pairs, int64_t n_list, int user_splits) {
  (void)kv_dtype;
  (void)head_dim;
  const int64_t sms = device_sm_count();
  // n_list counts up to 3 tail entries, which ride with the last split.
  const int64_t blocks_part = std::max<int64_t>(n_list - 3, 1);
  const int64_t max_splits = std::min<int64_t>(ceil_div(blocks_part, kTT), kMaxSplits);
  int64_t n = user_splits > 0 ? user_splits : ceil_div(2 * sms, pairs);
  n = std::max<int64_t>(1, std::min(n, max_splits));
  int64_t per = ceil_div(blocks_part, n);
  if (n > 1) per = ceil_div(per, kTT) * kTT;
  n = ceil_div(blocks_part, per);
  const int stages = per + 3 <= 2 * kTT ? 2 : 3;
  return AttnPlan{(int32_t)n, (int32_t)per, stages};
}

size_t attn_workspace_bytes(const AttnPlan& pl, int64_t rows, int n_q_heads, int head_dim) {
  if (pl.n_splits <= 1) return 0;
  const int64_t R = rows * n_q_heads;
  return 256 * (size_t)ceil_div(pl.n_splits * R * head_dim * 4, 256) + (size_t)pl.n_splits * R * 4;
}

void attn_workspace_layout(const AttnPlan& pl, int64_t rows, int n_q_heads, int head_dim, void* ws, float** part_o,
                           float** part_lse) {
  const int64_t R = rows * n_q_heads;
  *part_o = static_cast<float*>(ws);
  *part_lse = reinterpret_cast<float*>(static_cast<char*>(ws) + 256 * ceil_div(pl.n_splits * R * head_dim * 4, 256));
}

namespace {

template <int NSEQ, typename Kern>
cudaError_t launch_attn_kernel(Kern kernel, const AttnParams<NSEQ>& p, int n_rows, int threads, size_t smem,
                               cudaStream_t st) {
  cudaError_t e = allow_dynamic_smem((const void*)kernel, smem);
  if (e != cudaSuccess) return e;
  return launch_kernel(kernel, dim3((unsigned)p.n_splits, (unsigned)(p.n_q_heads / p.group), (unsigned)n_rows),
                       dim3((unsigned)threads), smem, st, 0u, p);
}

}  // namespace

template <int KVQ, int NSEQ>
cudaError_t launch_quantized(const AttnParams<NSEQ>& p, int n_rows, int stages, cudaStream_t st) {
  if (p.head_dim == 256) {
    if (stages == 2)
      return launch_attn_kernel(attn_mma_kernel<256, 2, NSEQ, KVQ>, p, n_rows, kAttnThreads,
                                MmaSmem<256, 2, KVQ>::bytes, st);
    return launch_attn_kernel(attn_mma_kernel<256, 3, NSEQ, KVQ>, p, n_rows, kAttnThreads,
                              MmaSmem<256, 3, KVQ>::bytes, st);
  }
  if (stages == 2)
    return launch_attn_kernel(attn_mma_kernel<128, 2, NSEQ, KVQ>, p, n_rows, kAttnThreads,
                              MmaSmem<128, 2, KVQ>::bytes, st);
  return launch_attn_kernel(attn_mma_kernel<128, 3, NSEQ, KVQ>, p, n_rows, kAttnThreads,
                            MmaSmem<128, 3, KVQ>::bytes, st);
}

template <int NSEQ>
cudaError_t launch_attn(const AttnParams<NSEQ>& p, int n_rows, qsa_dtype kv_dtype, int stages, cudaStream_t st) {
  if (n_rows == 0) return cudaSuccess;
  if (kv_dtype == QSA_FP8_E4M3) return launch_quantized<1, NSEQ>(p, n_rows, stages, st);
  if (kv_dtype == QSA_Q8_0) return launch_quantized<2, NSEQ>(p, n_rows, stages, st);
  if (kv_dtype == QSA_BF16) {
    if (p.head_dim == 256) {
      if (stages == 2)
        return launch_attn_kernel(attn_mma_kernel<256, 2, NSEQ>, p, n_rows, kAttnThreads, MmaSmem<256, 2>::bytes, st);
      return launch_attn_kernel(attn_mma_kernel<256, 3, NSEQ>, p, n_rows, kAttnThreads, MmaSmem<256, 3>::bytes, st);
    }
    if (stages == 2)
      return launch_attn_kernel(attn_mma_kernel<128, 2, NSEQ>, p, n_rows, kAttnThreads, MmaSmem<128, 2>::bytes, st);
    return launch_attn_kernel(attn_mma_kernel<128, 3, NSEQ>, p, n_rows, kAttnThreads, MmaSmem<128, 3>::bytes, st);
  }
  if (p.head_dim == 256)
    return launch_attn_kernel(attn_simt_kernel<256, NSEQ>, p, n_rows, 256, SimtSmem<256>::bytes, st);
  return launch_attn_kernel(attn_simt_kernel<128, NSEQ>, p, n_rows, 256, SimtSmem<128>::bytes, st);
}

template cudaError_t launch_attn<1>(const AttnParams<1>&, int, qsa_dtype, int, cudaStream_t);
template cudaError_t launch_attn<kLaunchSeqs>(const AttnParams<kLaunchSeqs>&, int, qsa_dtype, int, cudaStream_t);

cudaError_t launch_merge(const float* o_parts, const float* lse_parts, int n_parts, int64_t n_rows, int head_dim,
                         void* out, int out_dtype, float* lse_out, cudaStream_t st) {
  if (n_rows == 0) return cudaSuccess;
  if (head_dim == 256 || head_dim == 128) {
    const dim3 grid((unsigned)n_rows), block(kMergeWarps * 32);
    if (head_dim == 256)
      return launch_kernel(merge_cta_kernel<8>, grid, block, 0, st, 0u, o_parts, lse_parts, n_parts, n_rows, head_dim,
                           out, out_dtype, lse_out);
    return launch_kernel(merge_cta_kernel<4>, grid, block, 0, st, 0u, o_parts, lse_parts, n_parts, n_rows, head_dim,
                         out, out_dtype, lse_out);
  }
  const int64_t threads = n_rows * (head_dim / 4);
  const unsigned grid = (unsigned)((threads + 255) / 256);
  return launch_kernel(merge_kernel, dim3(grid), dim3(256), 0, st, 0u, o_parts, lse_parts, n_parts, n_rows, head_dim,
                       out, out_dtype, lse_out);
}

int attn_bad_ids_take() { return take_counter(attn::g_bad_ids); }

}  // namespace qsa
