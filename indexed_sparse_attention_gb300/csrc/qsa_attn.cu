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
// One CTA per (query row, KV group, split).  A split walks its share of the
// row's selected list (the 4 tokens of each selected block, then the tail) in
// tiles of 32 tokens; each token is located in the sequence's segment table
// and its K and V rows are gathered into shared memory.  bf16 K/V run on the
// tensor pipe (mma.sync m16n8k16: the 12 heads of a group padded to 16 rows
// against 32 gathered tokens), with an fp32 online softmax; fp32 K/V take a
// CUDA-core kernel.  Partials (normalised output, lse) of several splits are
// merged by the step-5 kernel.
#include <math.h>

#include "qsa_internal.cuh"

namespace qsa {

namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// Per-row context: position, visible blocks, selected list length.
struct RowCtx {
  int64_t nb;
  int64_t n_list;
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
  int32_t cnt = p.cnt[r];
  cnt = max(0, min(cnt, p.sel_ld));
  if ((int64_t)cnt > c.nb) cnt = (int32_t)c.nb;
  c.cnt = cnt;
  c.n_list = 4 * (int64_t)cnt + (pos + 1 - 4 * c.nb);
  c.sel_row = p.sel + (int64_t)r * p.sel_ld;
  c.seg_begin = sq.seg_begin;
  c.n_segs = sq.n_segs;
  return c;
}

// Entry i of the row's selected list -> element offset of (KV head g, token)
// in its segment, and the segment.  False when the entry names an invalid
// block id or a token no segment covers.
template <int NSEQ>
__device__ __forceinline__ bool locate(const AttnParams<NSEQ>& p, const RowCtx& c, int64_t i, int g,
                                       int& seg, int64_t& off) {
  int64_t t;
  if (i < 4 * (int64_t)c.cnt) {
    const int32_t b = __ldg(c.sel_row + (i >> 2));
    if (b < 0 || (int64_t)b >= c.nb) return false;
    t = 4 * (int64_t)b + (i & 3);
  } else {
    t = 4 * c.nb + (i - 4 * (int64_t)c.cnt);
  }
  for (int s = 0; s < c.n_segs; ++s) {
    const Segment& sg = p.seg[c.seg_begin + s];
    if (t >= sg.first && t < sg.first + sg.n) {
      seg = c.seg_begin + s;
      off = (int64_t)g * sg.head_stride + (t - sg.first) * sg.tok_stride;
      return true;
    }
  }
  return false;
}

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

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void cp_async16(void* dst, const void* src, bool valid) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(smem_u32(dst)), "l"(src),
               "r"(valid ? 16 : 0));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::); }
__device__ __forceinline__ void cp_async_wait1() { asm volatile("cp.async.wait_group 1;\n" ::); }

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

// Write one (row, head) result: to the final output when there is a single
// split, else to the split's partial slot.
template <int NSEQ>
__device__ __forceinline__ float* partial_row(const AttnParams<NSEQ>& p, int split, int r, int head) {
  return p.part_o + (((int64_t)split * p.total_rows + r) * p.n_q_heads + head) * p.head_dim;
}

// ------------------------------------------------------------------ tensor-pipe kernel (bf16 K/V)
constexpr int kTT = 32;        // tokens per tile
constexpr int kPStride = 40;   // bf16 per P row: 80-byte rows keep ldmatrix conflict-free

template <int D>
struct MmaSmem {
  static constexpr int CH = D / 8;  // 16-byte chunks per K/V/Q row
  static constexpr size_t q = 16 * D * 2;
  static constexpr size_t kv_stage = kTT * D * 2;
  static constexpr size_t s = 16 * (kTT + 4) * 4;
  static constexpr size_t pm = 16 * kPStride * 2;
  static constexpr size_t off_k = q;
  static constexpr size_t off_v = off_k + 2 * kv_stage;
  static constexpr size_t off_s = off_v + 2 * kv_stage;
  static constexpr size_t off_p = off_s + s;
  static constexpr size_t off_m = off_p + pm;           // m, l, alpha: 3 x 16 floats
  static constexpr size_t off_valid = off_m + 3 * 16 * 4;
  static constexpr size_t bytes = off_valid + 2 * kTT * 4;
};

template <int D, int NSEQ>
__global__ void __launch_bounds__(128) attn_mma_kernel(const AttnParams<NSEQ> p) {
  using L = MmaSmem<D>;
  constexpr int CH = L::CH;
  constexpr int NTD = D / 32;  // 8-channel n-tiles per warp in P.V (D/4 channels per warp)
  extern __shared__ __align__(128) uint8_t smem[];
  __nv_bfloat16* q_s = reinterpret_cast<__nv_bfloat16*>(smem);
  __nv_bfloat16* k_s = reinterpret_cast<__nv_bfloat16*>(smem + L::off_k);
  __nv_bfloat16* v_s = reinterpret_cast<__nv_bfloat16*>(smem + L::off_v);
  float* s_s = reinterpret_cast<float*>(smem + L::off_s);
  __nv_bfloat16* p_s = reinterpret_cast<__nv_bfloat16*>(smem + L::off_p);
  float* m_s = reinterpret_cast<float*>(smem + L::off_m);
  float* l_s = m_s + 16;
  float* a_s = m_s + 32;
  int* valid_s = reinterpret_cast<int*>(smem + L::off_valid);

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int split = blockIdx.x, g = blockIdx.y, r = p.row_base + blockIdx.z;
  const int G = p.group, head0 = g * G;
  const RowCtx c = make_row_ctx(p, r);
  const int64_t i0 = (int64_t)split * p.split_tokens;
  const int64_t i1 = min(c.n_list, i0 + p.split_tokens);
  const int n_tiles = i1 > i0 ? (int)((i1 - i0 + kTT - 1) / kTT) : 0;

  // Q of the group's heads (rows >= G zero), swizzled: chunk c of row h at c ^ (h & 7).
  const __nv_bfloat16* qg = static_cast<const __nv_bfloat16*>(p.q) + ((int64_t)r * p.n_q_heads + head0) * D;
  for (int idx = tid; idx < 16 * CH; idx += 128) {
    const int row = idx / CH, ch = idx % CH;
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (row < G) v = *reinterpret_cast<const uint4*>(qg + (int64_t)row * D + ch * 8);
    *reinterpret_cast<uint4*>(q_s + (row * CH + (ch ^ (row & 7))) * 8) = v;
  }
  for (int idx = tid; idx < 16 * kPStride; idx += 128) p_s[idx] = __float2bfloat16(0.f);
  if (tid < 16) {
    m_s[tid] = -INFINITY;
    l_s[tid] = 0.f;
    a_s[tid] = 1.f;
  }

  // Gather of one tile: thread -> token slot tid/4, chunks (tid&3) + 4j.
  auto load_tile = [&](int it, int stage) {
    const int tk = tid >> 2, q4 = tid & 3;
    const int64_t i = i0 + (int64_t)it * kTT + tk;
    int seg = 0;
    int64_t off = 0;
    const bool ok = i < i1 && locate(p, c, i, g, seg, off);
    const __nv_bfloat16* ks = ok ? static_cast<const __nv_bfloat16*>(p.seg[seg].k) + off : qg;
    const __nv_bfloat16* vs = ok ? static_cast<const __nv_bfloat16*>(p.seg[seg].v) + off : qg;
    __nv_bfloat16* kd = k_s + (size_t)stage * kTT * D + tk * D;
    __nv_bfloat16* vd = v_s + (size_t)stage * kTT * D + tk * D;
#pragma unroll
    for (int j = 0; j < CH / 4; ++j) {
      const int ch = q4 + 4 * j;
      const int pc = ch ^ (tk & 7);
      cp_async16(kd + pc * 8, ks + (ok ? ch * 8 : 0), ok);
      cp_async16(vd + pc * 8, vs + (ok ? ch * 8 : 0), ok);
    }
    if (q4 == 0) valid_s[stage * kTT + tk] = ok ? 1 : 0;
  };

  if (n_tiles > 0) load_tile(0, 0);
  cp_async_commit();
  __syncthreads();

  uint32_t qf[D / 16][4];
#pragma unroll
  for (int ks = 0; ks < D / 16; ++ks) {
    const int row = (lane & 7) + 8 * ((lane >> 3) & 1);
    const int ch = 2 * ks + (lane >> 4);
    ldsm_x4(qf[ks][0], qf[ks][1], qf[ks][2], qf[ks][3], q_s + (row * CH + (ch ^ (row & 7))) * 8);
  }

  float o[NTD][4];
#pragma unroll
  for (int j = 0; j < NTD; ++j) o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.f;
  const float zscale = p.scale * kLog2e;
  const int gq = lane >> 2, t4 = lane & 3;

  for (int it = 0; it < n_tiles; ++it) {
    const int stage = it & 1;
    if (it + 1 < n_tiles) load_tile(it + 1, stage ^ 1);
    cp_async_commit();
    cp_async_wait1();
    __syncthreads();
    const __nv_bfloat16* kt = k_s + (size_t)stage * kTT * D;
    const __nv_bfloat16* vt = v_s + (size_t)stage * kTT * D;
    // S = Q K^T for tokens 8w..8w+7 of the tile.
    {
      float sacc[4] = {0.f, 0.f, 0.f, 0.f};
      const int tk = 8 * warp + (lane & 7);
#pragma unroll
      for (int ks = 0; ks < D / 16; ks += 2) {
        uint32_t b0, b1, b2, b3;
        const int ch = 2 * ks + (lane >> 3);
        ldsm_x4(b0, b1, b2, b3, kt + (tk * CH + (ch ^ (tk & 7))) * 8);
        mma_bf16(sacc, qf[ks], b0, b1);
        mma_bf16(sacc, qf[ks + 1], b2, b3);
      }
      const int col = 8 * warp + 2 * t4;
      const bool v0 = valid_s[stage * kTT + col] != 0, v1 = valid_s[stage * kTT + col + 1] != 0;
      s_s[gq * (kTT + 4) + col] = v0 ? sacc[0] * zscale : -INFINITY;
      s_s[gq * (kTT + 4) + col + 1] = v1 ? sacc[1] * zscale : -INFINITY;
      s_s[(gq + 8) * (kTT + 4) + col] = v0 ? sacc[2] * zscale : -INFINITY;
      s_s[(gq + 8) * (kTT + 4) + col + 1] = v1 ? sacc[3] * zscale : -INFINITY;
    }
    __syncthreads();
    // Online softmax, one warp per head row, one lane per token (base-2 logits).
    for (int rr = warp; rr < G; rr += 4) {
      const float z = s_s[rr * (kTT + 4) + lane];
      const float mo = m_s[rr];
      const float mn = fmaxf(mo, warp_max(z));
      const float pz = mn == -INFINITY ? 0.f : exp2f(z - mn);
      const float sum = warp_sum(pz);
      p_s[rr * kPStride + lane] = __float2bfloat16(pz);
      if (lane == 0) {
        const float alpha = mo == -INFINITY ? 0.f : exp2f(mo - mn);
        a_s[rr] = alpha;
        m_s[rr] = mn;
        l_s[rr] = l_s[rr] * alpha + sum;
      }
    }
    __syncthreads();
    // O += P V over channels [warp*D/4, (warp+1)*D/4).
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
          const int ch = warp * (D / 32) + j + (lane >> 4);
          uint32_t b0, b1, b2, b3;
          ldsm_x4_t(b0, b1, b2, b3, vt + (tk * CH + (ch ^ (tk & 7))) * 8);
          mma_bf16(o[j], pa, b0, b1);
          mma_bf16(o[j + 1], pa, b2, b3);
        }
      }
    }
    __syncthreads();
  }

  // Finalise: normalised output and lse (natural log) for heads gq, gq+8.
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    const int row = gq + 8 * half;
    if (row >= G) continue;
    const float l = n_tiles > 0 ? l_s[row] : 0.f;
    const float m = n_tiles > 0 ? m_s[row] : -INFINITY;
    const float inv = l > 0.f ? 1.f / l : 0.f;
    const float lse = l > 0.f ? (m + log2f(l)) * kLn2 : -INFINITY;
    const int head = head0 + row;
    if (p.n_splits == 1) {
      const int64_t base = ((int64_t)r * p.n_q_heads + head) * D;
#pragma unroll
      for (int j = 0; j < NTD; ++j) {
        const int d = warp * (D / 4) + j * 8 + 2 * t4;
        const float x0 = o[j][2 * half] * inv, x1 = o[j][2 * half + 1] * inv;
        if (p.out_dtype == QSA_F32) {
          *reinterpret_cast<float2*>(static_cast<float*>(p.out) + base + d) = make_float2(x0, x1);
        } else {
          *reinterpret_cast<__nv_bfloat162*>(static_cast<__nv_bfloat16*>(p.out) + base + d) =
              __floats2bfloat162_rn(x0, x1);
        }
      }
      if (warp == 0 && t4 == 0 && p.lse) p.lse[(int64_t)r * p.n_q_heads + head] = lse;
    } else {
      float* dst = partial_row(p, split, r, head);
#pragma unroll
      for (int j = 0; j < NTD; ++j) {
        const int d = warp * (D / 4) + j * 8 + 2 * t4;
        *reinterpret_cast<float2*>(dst + d) = make_float2(o[j][2 * half] * inv, o[j][2 * half + 1] * inv);
      }
      if (warp == 0 && t4 == 0)
        p.part_lse[((int64_t)split * p.total_rows + r) * p.n_q_heads + head] = lse;
    }
  }
}

// ------------------------------------------------------------------ CUDA-core kernel (fp32 K/V)
// Thread -> channel d = tid % D and heads hs, hs + HS, ... (HS = 256 / D).
constexpr int kSimtTT = 32;

template <int D, int NSEQ>
__global__ void __launch_bounds__(256) attn_simt_kernel(const AttnParams<NSEQ> p) {
  constexpr int HS = 256 / D;
  constexpr int MAXH = 16 / HS;
  extern __shared__ __align__(16) float fsm[];
  float* q_s = fsm;                          // [16][D]
  float* k_s = q_s + 16 * D;                 // [32][D+1]
  float* v_s = k_s + kSimtTT * (D + 1);      // [32][D]
  float* z_s = v_s + kSimtTT * D;            // [16][33]
  float* m_s = z_s + 16 * 33;
  float* l_s = m_s + 16;
  float* a_s = l_s + 16;
  int* ok_s = reinterpret_cast<int*>(a_s + 16);

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int split = blockIdx.x, g = blockIdx.y, r = p.row_base + blockIdx.z;
  const int G = p.group, head0 = g * G;
  const RowCtx c = make_row_ctx(p, r);
  const int64_t i0 = (int64_t)split * p.split_tokens;
  const int64_t i1 = min(c.n_list, i0 + p.split_tokens);

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
      const bool ok = tk < nt && locate(p, c, base + tk, g, seg, off);
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
      z_s[hh * 33 + tk] = ok_s[tk] ? dot * p.scale : -INFINITY;
    }
    __syncthreads();
    for (int hh = warp; hh < G; hh += 8) {
      const float z = z_s[hh * 33 + lane];
      const float mo = m_s[hh];
      const float mn = fmaxf(mo, warp_max(z));
      const float pz = mn == -INFINITY ? 0.f : expf(z - mn);
      const float sum = warp_sum(pz);
      z_s[hh * 33 + lane] = pz;
      if (lane == 0) {
        const float alpha = mo == -INFINITY ? 0.f : expf(mo - mn);
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
  const bool any = i1 > i0;
#pragma unroll
  for (int j = 0; j < MAXH; ++j) {
    const int hh = hs + j * HS;
    if (hh >= G) continue;
    const float l = any ? l_s[hh] : 0.f;
    const float m = any ? m_s[hh] : -INFINITY;
    const float x = l > 0.f ? acc[j] / l : 0.f;
    const float lse = l > 0.f ? m + logf(l) : -INFINITY;
    const int head = head0 + hh;
    if (p.n_splits == 1) {
      const int64_t o = ((int64_t)r * p.n_q_heads + head) * D + d;
      if (p.out_dtype == QSA_F32) static_cast<float*>(p.out)[o] = x;
      else static_cast<__nv_bfloat16*>(p.out)[o] = __float2bfloat16(x);
      if (d == 0 && p.lse) p.lse[(int64_t)r * p.n_q_heads + head] = lse;
    } else {
      partial_row(p, split, r, head)[d] = x;
      if (d == 0) p.part_lse[((int64_t)split * p.total_rows + r) * p.n_q_heads + head] = lse;
    }
  }
}

template <int D>
constexpr size_t simt_smem_bytes() {
  return sizeof(float) * (16 * D + kSimtTT * (D + 1) + kSimtTT * D + 16 * 33 + 3 * 16) + sizeof(int) * kSimtTT;
}

// ------------------------------------------------------------------ step 5: log-sum-exp merge
// Thread -> (row, 4 channels).
__global__ void __launch_bounds__(256) merge_kernel(const float* __restrict__ o_parts,
                                                     const float* __restrict__ lse_parts, int n_parts,
                                                     int64_t n_rows, int head_dim, void* __restrict__ out,
                                                     int out_dtype, float* __restrict__ lse_out) {
  const int q = head_dim / 4;
  const int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= n_rows * q) return;
  const int64_t row = idx / q;
  const int d = (int)(idx % q) * 4;
  float m = -INFINITY;
  for (int s = 0; s < n_parts; ++s) m = fmaxf(m, lse_parts[(int64_t)s * n_rows + row]);
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  float wsum = 0.f;
  if (m != -INFINITY) {
    for (int s = 0; s < n_parts; ++s) {
      const float ls = lse_parts[(int64_t)s * n_rows + row];
      if (ls == -INFINITY) continue;
      const float w = expf(ls - m);
      const float4 v = *reinterpret_cast<const float4*>(o_parts + ((int64_t)s * n_rows + row) * head_dim + d);
      wsum += w;
      acc.x = fmaf(w, v.x, acc.x);
      acc.y = fmaf(w, v.y, acc.y);
      acc.z = fmaf(w, v.z, acc.z);
      acc.w = fmaf(w, v.w, acc.w);
    }
  }
  const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
  const float4 r = make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
  if (out_dtype == QSA_F32) {
    *reinterpret_cast<float4*>(static_cast<float*>(out) + row * head_dim + d) = r;
  } else {
    __nv_bfloat162* o2 = reinterpret_cast<__nv_bfloat162*>(static_cast<__nv_bfloat16*>(out) + row * head_dim + d);
    o2[0] = __floats2bfloat162_rn(r.x, r.y);
    o2[1] = __floats2bfloat162_rn(r.z, r.w);
  }
  if (d == 0 && lse_out) lse_out[row] = wsum > 0.f ? m + logf(wsum) : -INFINITY;
}

}  // namespace

template <int NSEQ>
cudaError_t launch_attn(const AttnParams<NSEQ>& p, int n_rows, qsa_dtype kv_dtype, cudaStream_t st) {
  if (n_rows == 0) return cudaSuccess;
  const dim3 grid((unsigned)p.n_splits, (unsigned)(p.n_q_heads / p.group), (unsigned)n_rows);
  cudaError_t e;
  if (kv_dtype == QSA_BF16) {
    if (p.head_dim == 256) {
      const size_t sm = MmaSmem<256>::bytes;
      if ((e = allow_dynamic_smem((const void*)attn_mma_kernel<256, NSEQ>, sm)) != cudaSuccess) return e;
      attn_mma_kernel<256, NSEQ><<<grid, 128, sm, st>>>(p);
    } else {
      const size_t sm = MmaSmem<128>::bytes;
      if ((e = allow_dynamic_smem((const void*)attn_mma_kernel<128, NSEQ>, sm)) != cudaSuccess) return e;
      attn_mma_kernel<128, NSEQ><<<grid, 128, sm, st>>>(p);
    }
  } else {
    if (p.head_dim == 256) {
      const size_t sm = simt_smem_bytes<256>();
      if ((e = allow_dynamic_smem((const void*)attn_simt_kernel<256, NSEQ>, sm)) != cudaSuccess) return e;
      attn_simt_kernel<256, NSEQ><<<grid, 256, sm, st>>>(p);
    } else {
      const size_t sm = simt_smem_bytes<128>();
      if ((e = allow_dynamic_smem((const void*)attn_simt_kernel<128, NSEQ>, sm)) != cudaSuccess) return e;
      attn_simt_kernel<128, NSEQ><<<grid, 256, sm, st>>>(p);
    }
  }
  return cudaGetLastError();
}

template cudaError_t launch_attn<1>(const AttnParams<1>&, int, qsa_dtype, cudaStream_t);
template cudaError_t launch_attn<kLaunchSeqs>(const AttnParams<kLaunchSeqs>&, int, qsa_dtype, cudaStream_t);

cudaError_t launch_merge(const float* o_parts, const float* lse_parts, int n_parts, int64_t n_rows, int head_dim,
                         void* out, int out_dtype, float* lse_out, cudaStream_t st) {
  const int64_t threads = n_rows * (head_dim / 4);
  if (threads == 0) return cudaSuccess;
  const unsigned grid = (unsigned)((threads + 255) / 256);
  merge_kernel<<<grid, 256, 0, st>>>(o_parts, lse_parts, n_parts, n_rows, head_dim, out, out_dtype, lse_out);
  return cudaGetLastError();
}

}  // namespace qsa
