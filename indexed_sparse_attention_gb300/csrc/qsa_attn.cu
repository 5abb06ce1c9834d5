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
#include <cooperative_groups.h>
#include <math.h>

#include <algorithm>
#include <mutex>
#include <vector>

#include "qsa_internal.cuh"

namespace cg = cooperative_groups;

namespace qsa {

namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr int kMaxSplits = 16;   // splits of one (row, KV group) = CTAs of one cluster

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
                                       int g, int& seg, int64_t& off) {
  int64_t t;
  if (i < 4 * (int64_t)c.cnt) {
    const int64_t k = (i >> 2) - ic.blk0;
    const int32_t b = (k >= 0 && k < ic.n) ? ic.ids[k] : __ldg(c.sel_row + (i >> 2));
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

// Stage the ids of list entries [i0, i1) into ids_s (all threads call).
__device__ __forceinline__ IdCache stage_ids(const RowCtx& c, int64_t i0, int64_t i1, int32_t* ids_s) {
  IdCache ic;
  ic.ids = ids_s;
  ic.blk0 = i0 >> 2;
  const int64_t last = min(i1, 4 * (int64_t)c.cnt);   // entries past 4*cnt are tail tokens
  int64_t n = last > i0 ? ((last - 1) >> 2) - ic.blk0 + 1 : 0;
  if (n > kIdCache) n = kIdCache;
  ic.n = (int)n;
  for (int k = threadIdx.x; k < ic.n; k += blockDim.x) ids_s[k] = __ldg(c.sel_row + ic.blk0 + k);
  return ic;
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
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N));
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

// ------------------------------------------------------------------ split merge (step 5)
// The CTAs of one cluster hold the partials of consecutive splits of the same
// (row, KV group): unnormalised output o_s[16][D] (fp32), running max m_s[16]
// of the base-2 logits and running sum l_s[16].  After a cluster barrier,
// CTA c merges the 4-channel groups c, c+CS, ... of every head across the
// cluster through distributed shared memory:
//   M = max_q m_q,  w_q = 2^(m_q - M),  out = sum_q w_q o_q / sum_q w_q l_q,
//   lse = (M + log2 sum_q w_q l_q) * ln 2,
// and a head whose splits saw no key gets out = 0 and lse = -inf.
// With several clusters per (row, KV group), each cluster writes its merged,
// normalised partial and lse to the workspace; the cluster that takes the
// last ticket merges all of them by the same rule (natural-log lse) and
// returns the ticket counter to zero.
constexpr int kMaxClusters = 32;   // clusters per (row, KV group)

struct MergeSmem {
  float mq[16][kMaxSplits];
  float lq[16][kMaxSplits];
  float w[16][kMaxSplits];
  float inv[16];
  float lse[16];
  float cw[16][kMaxClusters];
  float cinv[16];
  float clse[16];
  int last;
};

template <int NSEQ>
__device__ void merge_store(const AttnParams<NSEQ>& p, int r, int g, int G, int D, float* o_s, float* m_s,
                            float* l_s, MergeSmem* ms) {
  cg::cluster_group cluster = cg::this_cluster();
  const int S = (int)cluster.num_blocks();
  const int c = (int)cluster.block_rank();
  const int tid = threadIdx.x, nt = blockDim.x;
  const int head0 = g * G;
  cluster.sync();
  // Every split's running max and sum, one (head, split) pair per thread.
  for (int t = tid; t < G * S; t += nt) {
    const int h = t / S, q = t % S;
    ms->mq[h][q] = *cluster.map_shared_rank(m_s + h, q);
    ms->lq[h][q] = *cluster.map_shared_rank(l_s + h, q);
  }
  __syncthreads();
  if (tid < G) {
    float M = -INFINITY;
    for (int q = 0; q < S; ++q) M = fmaxf(M, ms->mq[tid][q]);
    float Lsum = 0.f;
    for (int q = 0; q < S; ++q) {
      const float mq = ms->mq[tid][q];
      const float w = mq == -INFINITY ? 0.f : exp2f(mq - M);
      ms->w[tid][q] = w;
      Lsum += w * ms->lq[tid][q];
    }
    ms->inv[tid] = Lsum > 0.f ? 1.f / Lsum : 0.f;
    ms->lse[tid] = Lsum > 0.f ? (M + log2f(Lsum)) * kLn2 : -INFINITY;
  }
  __syncthreads();
  const int NC = p.n_clusters;
  const int64_t pair = (int64_t)r * (p.n_q_heads / G) + g;
  const int64_t cid = blockIdx.x / S;
  // 4-channel groups c, c + S, c + 2S, ... of every head belong to this CTA
  // (any S <= 16; D / 4 >= 32 groups, so every CTA has at least one).
  const int nq = (D / 4 - c + S - 1) / S;
  for (int idx = tid; idx < G * nq; idx += nt) {
    const int h = idx / nq;
    const int d = 4 * (c + (idx % nq) * S);
    float4 v[kMaxSplits];
#pragma unroll
    for (int q = 0; q < kMaxSplits; ++q)
      if (q < S) v[q] = *reinterpret_cast<const float4*>(cluster.map_shared_rank(o_s + h * D + d, q));
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int q = 0; q < kMaxSplits; ++q) {
      if (q < S) {
        const float w = ms->w[h][q];
        acc.x = fmaf(w, v[q].x, acc.x);
        acc.y = fmaf(w, v[q].y, acc.y);
        acc.z = fmaf(w, v[q].z, acc.z);
        acc.w = fmaf(w, v[q].w, acc.w);
      }
    }
    const float inv = ms->inv[h];
    const float4 res = make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
    if (NC > 1) {
      *reinterpret_cast<float4*>(p.part_o + ((pair * NC + cid) * G + h) * D + d) = res;
    } else {
      const int64_t o = ((int64_t)r * p.n_q_heads + head0 + h) * D + d;
      if (p.out_dtype == QSA_F32) {
        *reinterpret_cast<float4*>(static_cast<float*>(p.out) + o) = res;
      } else {
        __nv_bfloat162* o2 = reinterpret_cast<__nv_bfloat162*>(static_cast<__nv_bfloat16*>(p.out) + o);
        o2[0] = __floats2bfloat162_rn(res.x, res.y);
        o2[1] = __floats2bfloat162_rn(res.z, res.w);
      }
    }
  }
  if (NC == 1) {
    if (c == 0 && tid < G && p.lse) p.lse[(int64_t)r * p.n_q_heads + head0 + tid] = ms->lse[tid];
    cluster.sync();  // keep this CTA's partial alive until every peer has read it
    return;
  }
  if (c == 0 && tid < G) p.part_lse[(pair * NC + cid) * G + tid] = ms->lse[tid];
  __threadfence();
  cluster.sync();    // this cluster's partial is written; peers are done reading o_s
  if (c == 0 && tid == 0) {
    const unsigned t = atomicAdd(p.counters + pair, 1u);
    const int last = t == (unsigned)(NC - 1);
    if (last) p.counters[pair] = 0u;   // every ticket is taken: ready for the next call
    for (int q = 0; q < S; ++q) cluster.map_shared_rank(ms, q)->last = last;
  }
  cluster.sync();
  if (!ms->last) return;
  __threadfence();
  // The last cluster merges the clusters' partials (natural-log lse).
  for (int t = tid; t < G * NC; t += nt) {
    const int h = t / NC, q = t % NC;
    ms->cw[h][q] = __ldcg(p.part_lse + (pair * NC + q) * G + h);
  }
  __syncthreads();
  if (tid < G) {
    float M = -INFINITY;
    for (int q = 0; q < NC; ++q) M = fmaxf(M, ms->cw[tid][q]);
    float Wsum = 0.f;
    for (int q = 0; q < NC; ++q) {
      const float lq = ms->cw[tid][q];
      const float w = lq == -INFINITY ? 0.f : expf(lq - M);
      ms->cw[tid][q] = w;
      Wsum += w;
    }
    ms->cinv[tid] = Wsum > 0.f ? 1.f / Wsum : 0.f;
    ms->clse[tid] = Wsum > 0.f ? M + logf(Wsum) : -INFINITY;
  }
  __syncthreads();
  for (int idx = tid; idx < G * nq; idx += nt) {
    const int h = idx / nq;
    const int d = 4 * (c + (idx % nq) * S);
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int q0 = 0; q0 < NC; q0 += 8) {
      float4 v[8];
#pragma unroll
      for (int j = 0; j < 8; ++j)
        v[j] = q0 + j < NC ? __ldcg(reinterpret_cast<const float4*>(p.part_o + ((pair * NC + q0 + j) * G + h) * D + d))
                           : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const float w = q0 + j < NC ? ms->cw[h][q0 + j] : 0.f;
        acc.x = fmaf(w, v[j].x, acc.x);
        acc.y = fmaf(w, v[j].y, acc.y);
        acc.z = fmaf(w, v[j].z, acc.z);
        acc.w = fmaf(w, v[j].w, acc.w);
      }
    }
    const float inv = ms->cinv[h];
    const int64_t o = ((int64_t)r * p.n_q_heads + head0 + h) * D + d;
    if (p.out_dtype == QSA_F32) {
      *reinterpret_cast<float4*>(static_cast<float*>(p.out) + o) =
          make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
    } else {
      __nv_bfloat162* o2 = reinterpret_cast<__nv_bfloat162*>(static_cast<__nv_bfloat16*>(p.out) + o);
      o2[0] = __floats2bfloat162_rn(acc.x * inv, acc.y * inv);
      o2[1] = __floats2bfloat162_rn(acc.z * inv, acc.w * inv);
    }
  }
  if (c == 0 && tid < G && p.lse) p.lse[(int64_t)r * p.n_q_heads + head0 + tid] = ms->clse[tid];
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

template <int D, int STAGES>
struct MmaSmem {
  static constexpr int CH = D / 8;                     // 16-byte chunks per K/V/Q row
  static constexpr size_t q = 16 * D * 2;
  static constexpr size_t kv_tile = kTT * D * 2;       // one K or V tile
  static constexpr size_t s = 2 * 16 * kSStride * 4;   // logits, one plane per channel half
  static constexpr size_t pm = 16 * kPStride * 2;
  static constexpr size_t off_kv = q;                  // [STAGES][K tile, V tile]
  static constexpr size_t off_s = off_kv + STAGES * 2 * kv_tile;
  static constexpr size_t off_p = off_s + s;
  static constexpr size_t off_m = off_p + pm;          // m, l, alpha: 3 x 16 floats
  static constexpr size_t off_valid = off_m + 3 * 16 * 4;
  static constexpr size_t off_ids = off_valid + STAGES * kTT * 4;
  static constexpr size_t bytes = off_ids + kIdCache * 4;
  // After the token loop the K/V stages hold the partial [16][D] fp32 and the
  // merge scratch.
  static constexpr size_t off_merge = off_kv + 16 * D * 4;
  static_assert(16 * D * 4 + sizeof(MergeSmem) <= STAGES * 2 * kv_tile, "merge data must fit the K/V stages");
  // Three stages keep two CTAs per SM (228 KB per SM, 1 KB reserved per CTA).
  static_assert(STAGES != 3 || 2 * (bytes + 1024) <= 228 * 1024, "two CTAs per SM");
};

template <int D, int STAGES, int NSEQ>
__global__ void __launch_bounds__(kAttnThreads, STAGES <= 3 ? 2 : 1) attn_mma_kernel(const AttnParams<NSEQ> p) {
  using L = MmaSmem<D, STAGES>;
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
  MergeSmem* msm = reinterpret_cast<MergeSmem*>(smem + L::off_merge);
  grid_dependency_sync();

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int quarter = warp & 3, half = warp >> 2;
  const int split = blockIdx.x, g = blockIdx.y, r = p.row_base + blockIdx.z;
  const int G = p.group, head0 = g * G;
  const RowCtx c = make_row_ctx(p, r);
  const int64_t i0 = (int64_t)split * p.split_tokens;
  const int64_t i1 = min(c.n_list, i0 + p.split_tokens);
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
  const IdCache ic = stage_ids(c, i0, i1, ids_s);
  __syncthreads();

  // Gather of one tile into a stage: thread -> token slot tid/8, chunks (tid&7) + 8j,
  // swizzled: chunk c of token row t lands at c ^ (t & 7).
  auto load_tile = [&](int it, int stage) {
    const int tk = tid >> 3, q8 = tid & 7;
    const int64_t i = i0 + (int64_t)it * kTT + tk;
    int seg = 0;
    int64_t off = 0;
    const bool ok = i < i1 && locate(p, c, ic, i, g, seg, off);
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
      float z[2], mo[2], mx[2];
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const int rr = warp + 8 * j;
        z[j] = -INFINITY;
        mo[j] = -INFINITY;
        if (rr < G) {
          const float s0 = s_s[rr * kSStride + lane] + s_s[16 * kSStride + rr * kSStride + lane];
          z[j] = valid ? s0 * zscale : -INFINITY;
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
          p_s[rr * kPStride + lane] = __float2bfloat16(pz[j]);
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

  // Unnormalised partial into shared memory (over the K/V stages), then merge.
  float* o_s = reinterpret_cast<float*>(kv_s);
#pragma unroll
  for (int hf = 0; hf < 2; ++hf) {
    const int row = gq + 8 * hf;
#pragma unroll
    for (int j = 0; j < NTD; ++j) {
      const int d = warp * (D / 8) + j * 8 + 2 * t4;
      *reinterpret_cast<float2*>(o_s + row * D + d) = make_float2(o[j][2 * hf], o[j][2 * hf + 1]);
    }
  }
  merge_store(p, r, g, G, D, o_s, m_s, l_s, msm);
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
  static constexpr size_t bytes = floats * 4 + kSimtTT * 4 + kIdCache * 4 + sizeof(MergeSmem);
  static_assert(16 * D <= k + v, "merge partial must fit the K/V tiles");
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
  MergeSmem* msm = reinterpret_cast<MergeSmem*>(ids_s + kIdCache);
  grid_dependency_sync();

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int split = blockIdx.x, g = blockIdx.y, r = p.row_base + blockIdx.z;
  const int G = p.group, head0 = g * G;
  const RowCtx c = make_row_ctx(p, r);
  const int64_t i0 = (int64_t)split * p.split_tokens;
  const int64_t i1 = min(c.n_list, i0 + p.split_tokens);
  const float zscale = p.scale * kLog2e;
  const IdCache ic = stage_ids(c, i0, i1, ids_s);

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
  float* o_s = k_s;  // [16][D] over the K/V tiles
#pragma unroll
  for (int j = 0; j < MAXH; ++j) {
    const int hh = hs + j * HS;
    if (hh < 16) o_s[hh * D + d] = hh < G ? acc[j] : 0.f;
  }
  merge_store(p, r, g, G, D, o_s, m_s, l_s, msm);
}


// ------------------------------------------------------------------ step 5 entry point: merge of given partials
// Thread -> (row, 4 channels).  The partials' lse values are read first in
// batches, so each thread's loads are independent of one another.
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

template <int NSEQ, typename Kern>
cudaError_t launch_attn_kernel(Kern kernel, const AttnParams<NSEQ>& p, int n_rows, int threads, size_t smem,
                               cudaStream_t st) {
  cudaError_t e = allow_dynamic_smem((const void*)kernel, smem);
  if (e != cudaSuccess) return e;
  const int cs = p.cluster_size;
  if (cs > 8) {
    e = allow_cluster16((const void*)kernel, threads, smem);
    if (e != cudaSuccess) return e;
  }
  return launch_kernel(kernel, dim3((unsigned)(cs * p.n_clusters), (unsigned)(p.n_q_heads / p.group), (unsigned)n_rows),
                       dim3((unsigned)threads), smem, st, (unsigned)cs, p);
}

}  // namespace

// The kernel variant a plan runs, with its block size and shared memory.
struct AttnVariant {
  const void* fn;
  int threads;
  size_t smem;
};

static AttnVariant attn_variant(qsa_dtype kv_dtype, int head_dim, int stages) {
  if (kv_dtype == QSA_BF16) {
    if (head_dim == 256)
      return stages == 5 ? AttnVariant{(const void*)attn_mma_kernel<256, 5, 1>, kAttnThreads, MmaSmem<256, 5>::bytes}
                         : AttnVariant{(const void*)attn_mma_kernel<256, 3, 1>, kAttnThreads, MmaSmem<256, 3>::bytes};
    return stages == 5 ? AttnVariant{(const void*)attn_mma_kernel<128, 5, 1>, kAttnThreads, MmaSmem<128, 5>::bytes}
                       : AttnVariant{(const void*)attn_mma_kernel<128, 3, 1>, kAttnThreads, MmaSmem<128, 3>::bytes};
  }
  return head_dim == 256 ? AttnVariant{(const void*)attn_simt_kernel<256, 1>, 256, SimtSmem<256>::bytes}
                         : AttnVariant{(const void*)attn_simt_kernel<128, 1>, 256, SimtSmem<128>::bytes};
}

// Clusters of `cs` CTAs of this variant that can be resident at once.
static int max_active_clusters(const AttnVariant& v, int cs) {
  struct Entry {
    int dev;
    const void* fn;
    int cs;
    int n;
  };
  static std::vector<Entry> cache;
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  std::lock_guard<std::mutex> lk(mu);
  for (const Entry& e : cache)
    if (e.dev == dev && e.fn == v.fn && e.cs == cs) return e.n;
  int n = 0;
  if (allow_dynamic_smem(v.fn, v.smem) == cudaSuccess) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)cs, 1, 1);
    cfg.blockDim = dim3((unsigned)v.threads, 1, 1);
    cfg.dynamicSmemBytes = v.smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)cs;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaOccupancyMaxActiveClusters(&n, v.fn, &cfg) != cudaSuccess) n = 0;
  }
  cache.push_back(Entry{dev, v.fn, cs, n});
  return n;
}

static int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Splits of each (row, KV group): `total` CTAs in n_clusters clusters of
// cluster_size, each split at most 5 tiles of 32 selected rows when the GPU
// has room for one CTA per SM, all of them resident at once.
AttnPlan attn_plan(qsa_dtype kv_dtype, int head_dim, int64_t pairs, int64_t n_list, int user_splits) {
  const int64_t sms = device_sm_count();
  const int64_t max_total = std::min<int64_t>(ceil_div(n_list, kTT), (int64_t)kMaxSplits * kMaxClusters);
  int64_t total;
  if (user_splits > 0) {
    total = std::min<int64_t>(user_splits, max_total);
  } else {
    total = std::max<int64_t>(1, sms / pairs);
    if (ceil_div(ceil_div(n_list, std::min(total, max_total)), kTT) > 5) total = std::max<int64_t>(1, 2 * sms / pairs);
    total = std::min(total, max_total);
    // Fewer CTAs when that keeps the tiles per CTA.
    const int64_t tiles = ceil_div(ceil_div(n_list, total), kTT);
    while (total > 1 && ceil_div(ceil_div(n_list, total - 1), kTT) == tiles) --total;
  }
  total = std::max<int64_t>(1, total);
  const int64_t tiles = ceil_div(ceil_div(n_list, total), kTT);
  const int stages = (tiles <= 5 && pairs * total <= sms) ? 5 : 3;
  const AttnVariant v = attn_variant(kv_dtype, head_dim, stages);
  AttnPlan best{1, 1, (int32_t)n_list, stages};
  bool found = false;
  // Cluster sizes to try, largest first: min(total, 8), then 6, 4, 3, 2, 1.
  const int first = (int)std::min<int64_t>(total, 8);
  const int sizes[6] = {first, 6, 4, 3, 2, 1};
  for (int k = 0; k < 6; ++k) {
    const int cs = sizes[k];
    if (k > 0 && cs >= first) continue;
    const int64_t nc = ceil_div(total, cs);
    if (nc > kMaxClusters) continue;
    const int64_t cs_b = ceil_div(total, nc);           // balance the clusters
    const int active = max_active_clusters(v, (int)cs_b);
    if (user_splits <= 0 && active > 0 && pairs * nc > active) continue;   // keep every cluster resident
    best = AttnPlan{(int32_t)cs_b, (int32_t)nc, (int32_t)ceil_div(n_list, cs_b * nc), stages};
    found = true;
    break;
  }
  if (!found) {
    const int64_t cs = std::min<int64_t>(total, 8);
    const int64_t nc = std::min<int64_t>(ceil_div(total, cs), kMaxClusters);
    best = AttnPlan{(int32_t)cs, (int32_t)nc, (int32_t)ceil_div(n_list, cs * nc), stages};
  }
  return best;
}

size_t attn_workspace_bytes(const AttnPlan& pl, int64_t pairs, int group, int head_dim) {
  if (pl.n_clusters <= 1) return 0;
  const size_t parts = (size_t)pairs * pl.n_clusters * group;
  return 256 * ceil_div(pairs * 4, 256) + 256 * ceil_div((int64_t)parts * 4, 256) + parts * head_dim * 4;
}

void attn_workspace_layout(const AttnPlan& pl, int64_t pairs, int group, void* ws, uint32_t** counters,
                           float** part_lse, float** part_o) {
  char* b = static_cast<char*>(ws);
  const size_t parts = (size_t)pairs * pl.n_clusters * group;
  *counters = reinterpret_cast<uint32_t*>(b);
  b += 256 * ceil_div(pairs * 4, 256);
  *part_lse = reinterpret_cast<float*>(b);
  b += 256 * ceil_div((int64_t)parts * 4, 256);
  *part_o = reinterpret_cast<float*>(b);
}

template <int NSEQ>
cudaError_t launch_attn(const AttnParams<NSEQ>& p, int n_rows, qsa_dtype kv_dtype, int stages, cudaStream_t st) {
  if (n_rows == 0) return cudaSuccess;
  if (kv_dtype == QSA_BF16) {
    if (p.head_dim == 256) {
      if (stages == 5)
        return launch_attn_kernel(attn_mma_kernel<256, 5, NSEQ>, p, n_rows, kAttnThreads, MmaSmem<256, 5>::bytes, st);
      return launch_attn_kernel(attn_mma_kernel<256, 3, NSEQ>, p, n_rows, kAttnThreads, MmaSmem<256, 3>::bytes, st);
    }
    if (stages == 5)
      return launch_attn_kernel(attn_mma_kernel<128, 5, NSEQ>, p, n_rows, kAttnThreads, MmaSmem<128, 5>::bytes, st);
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
  const int64_t threads = n_rows * (head_dim / 4);
  if (threads == 0) return cudaSuccess;
  const unsigned grid = (unsigned)((threads + 255) / 256);
  return launch_kernel(merge_kernel, dim3(grid), dim3(256), 0, st, 0, o_parts, lse_parts, n_parts, n_rows, head_dim,
                       out, out_dtype, lse_out);
}

}  // namespace qsa
