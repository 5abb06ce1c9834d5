// Step 4 for many query rows (chunked prefill) on the 5th-generation tensor
// cores: exact softmax attention of each row's 12-head KV group over only the
// row's selected K/V rows (hipfire, "QSA sparse attention and the VMM KV
// backend", section 02: at most 2,048 selected rows plus the incomplete tail
// block per query; section 03: one unit of work per KV group so each gathered
// K/V row serves all its query heads), over the KV segment table of MTPLX
// pull request #610.
//
// A unit is one (query row r, KV group g): the group's G <= 16 query heads
// against the row's list of n = 4 cnt + tail entries, in T = ceil(n / 128)
// tiles of 128 gathered tokens.  Two passes over the list, so the softmax
// needs no running rescale:
//   logits   S_t^T = K_t Q^T   tcgen05.mma, M = 128 tokens, N = 16 heads,
//                              K = head_dim; every tile's 16 fp32 columns stay
//                              in TMEM (up to 30 tiles = 480 columns);
//   softmax  the exact maximum m_h of each head over all tiles, then
//            P_t = exp(S_t - m) rounded to bf16 into shared memory, and the
//            row sums l_h in fp32;
//   output   O^T += V_t^T P_t^T  M = 128 channels per MMA (two for
//                              head_dim 256), N = 16 heads, K = 128 tokens,
//                              in 32 further TMEM columns; normalised by l,
//                              with the natural-log lse m + log l.
// Roles in a persistent CTA (one per SM; unit u goes to CTA u mod grid, KV
// group major, so the CTAs in flight read one KV head's cache):
//   warps 0-3  softmax and epilogue (warp w reads TMEM lanes 32 w ..);
//   warps 4-7  gather each unit's K tiles, then its V tiles, 16 bytes per
//              lane with cp.async (zero fill for list entries that name no
//              valid token), into a ring of 3 (head_dim 256) or 6 (128)
//              tile slots stored with the 128-byte swizzle, plus the query
//              tile and one validity bit per list entry;
//   warp 8     allocates TMEM; lane 0 issues the MMAs and commits them.
// Each K and V row is read once per unit and each MMA operand is read from
// shared memory by the tensor cores.  Every mbarrier wait gives up after
// about two seconds (counted; the CTA then runs to its end without waiting).
#include <math.h>

#include "qsa_attn_common.cuh"
#include "qsa_tc.cuh"

namespace qsa {

namespace {

using namespace attn;
using namespace tc;

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr int kTok = 128;                   // gathered tokens per tile (M of the logits MMA)
constexpr int kHeads = 16;                  // query heads of a group, padded (N of both MMAs)
constexpr int kMaxTiles = 30;               // logits tiles held in TMEM (16 columns each)
constexpr int kMaxList = kMaxTiles * kTok;  // 3,840 list entries
constexpr int kIdCap = kMaxList / 4;        // selected block ids staged per unit
constexpr int kSoftWarps = 4;
constexpr int kProdWarps = 4;
constexpr int kMmaWarp = kSoftWarps + kProdWarps;
constexpr int kThreads = 32 * (kMmaWarp + 1);
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kOCol = kMaxTiles * kHeads;   // O^T accumulators after the logits
constexpr int kSubBytes = kTok * 128;            // one 64-channel column block of a tile

// M = 128 tokens x N = 16 heads, both operands K-major; and the output
// product with V^T as an MN-major operand (channels contiguous).
constexpr uint32_t kIdescS = idesc_bf16(128, kHeads, false, false);
constexpr uint32_t kIdescO = idesc_bf16(128, kHeads, true, false);

__device__ int g_attn_tc_timeouts;

template <int D>
struct TcLayout {
  static constexpr int kSubs = D / 64;                     // 64-channel column blocks
  static constexpr int kTileBytes = kSubs * kSubBytes;     // 128 tokens x D bf16
  static constexpr int kSlots = 3 * 65536 / kTileBytes;    // 3 (D = 256) or 6 (D = 128)
  static constexpr int kQBytes = kSubs * kHeads * 128;
  static constexpr int kPBytes = 2 * kHeads * 128;         // 16 heads x 128 tokens (two 64-token blocks)
  static constexpr size_t off_q = (size_t)kSlots * kTileBytes;
  static constexpr size_t off_p = off_q + kQBytes;         // two P buffers
  static constexpr size_t off_ids = off_p + 2 * kPBytes;
  static constexpr size_t off_valid = off_ids + kIdCap * 4;   // validity bits of two units
  static constexpr size_t bytes = off_valid + 2 * (kMaxList / 32) * 4;
  static constexpr size_t alloc = bytes + 1024;            // room for the 1,024-byte alignment
  static_assert(off_q % 1024 == 0 && off_p % 1024 == 0, "swizzled tiles on 1,024-byte boundaries");
  static_assert(kOCol + kHeads * (D / 128) <= kTmemCols, "TMEM columns");
};

// One unit's row bookkeeping (every role derives the same values).
struct Unit {
  RowCtx c;
  int r, g;
  int n;   // list entries
  int T;   // tiles
};

template <int NSEQ>
__device__ __forceinline__ Unit unit_at(const AttnParams<NSEQ>& p, int n_rows, int u) {
  Unit x;
  x.g = u / n_rows;
  x.r = p.row_base + u % n_rows;
  x.c = make_row_ctx(p, x.r);
  set_count(x.c, __ldg(p.cnt + x.r), p.sel_ld);
  x.n = (int)x.c.n_list;
  x.T = (x.n + kTok - 1) / kTok;
  return x;
}

__device__ __forceinline__ void named_sync(int id, int threads) {
  asm volatile("bar.sync %0, %1;\n" ::"r"(id), "r"(threads) : "memory");
}

// Reduce 16 values per lane over the warp's 32 lanes by halving: after the
// call lane l holds the result for value index vi(l) = 8 b4 + 4 b3 + 2 b2 + b1
// (b_k = bit k of l) in v[0].
template <bool MAX>
__device__ __forceinline__ void warp_reduce16(float (&v)[16], int lane) {
#pragma unroll
  for (int step = 0; step < 4; ++step) {
    const int half = 8 >> step;   // values kept after this step
    const int bit = 16 >> step;   // partner lane distance
    const bool upper = (lane & bit) != 0;
#pragma unroll
    for (int i = 0; i < half; ++i) {
      const float send = upper ? v[i] : v[i + half];
      const float keep = upper ? v[i + half] : v[i];
      const float got = __shfl_xor_sync(0xffffffffu, send, bit);
      v[i] = MAX ? fmaxf(keep, got) : keep + got;
    }
  }
  const float got = __shfl_xor_sync(0xffffffffu, v[0], 1);
  v[0] = MAX ? fmaxf(v[0], got) : v[0] + got;
}
__device__ __forceinline__ int reduced_index(int lane) {
  return 8 * ((lane >> 4) & 1) + 4 * ((lane >> 3) & 1) + 2 * ((lane >> 2) & 1) + ((lane >> 1) & 1);
}

// The KV segments of a unit's sequence, copied to shared memory once per unit.
struct SegS {
  const __nv_bfloat16* k;
  const __nv_bfloat16* v;
  int64_t first, n, head_stride, tok_stride;
};

// List entry i of a unit -> its K or V row (KV head g), as locate() does,
// reading the ids and the segment table from shared memory.
__device__ __forceinline__ bool locate_tok(const RowCtx& c, const int32_t* ids, const SegS* segs, int g, int64_t i,
                                           bool v, const __nv_bfloat16*& src) {
  if (i >= c.n_list) return false;
  int64_t t;
  if (i < 4 * (int64_t)c.cnt) {
    const int32_t b = ids[i >> 2];
    if (b < 0 || (int64_t)b >= c.nb) {
      atomicAdd(&g_bad_ids, 1);
      return false;
    }
    t = 4 * (int64_t)b + (i & 3);
  } else {
    t = 4 * c.nb + (i - 4 * (int64_t)c.cnt);
  }
  for (int s = 0; s < c.n_segs; ++s) {
    const SegS& sg = segs[s];
    if (t >= sg.first && t < sg.first + sg.n) {
      src = (v ? sg.v : sg.k) + (int64_t)g * sg.head_stride + (t - sg.first) * sg.tok_stride;
      return true;
    }
  }
  return false;
}

template <int NSEQ>
__device__ __forceinline__ void store_out(const AttnParams<NSEQ>& p, int64_t idx, float x) {
  if (p.out_dtype == QSA_F32)
    static_cast<float*>(p.out)[idx] = x;
  else
    static_cast<__nv_bfloat16*>(p.out)[idx] = __float2bfloat16(x);
}

template <int D, int NSEQ>
__global__ void __launch_bounds__(kThreads, 1) attn_tc_kernel(const __grid_constant__ AttnParams<NSEQ> p, int n_rows) {
  using L = TcLayout<D>;
  constexpr int S = L::kSlots;
  extern __shared__ uint8_t tc_raw[];
  __shared__ uint64_t full[S], empty[S], p_full[2], p_empty[2], s_full, s_free, o_full, o_free, q_free, mma_done;
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag;
  __shared__ float red_m[kSoftWarps][kHeads], red_l[kSoftWarps][kHeads];
  __shared__ SegS segs_s[QSA_MAX_SEGMENTS];

  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(tc_raw) + 1023) & ~(uintptr_t)1023);
  uint8_t* ring = base;
  uint8_t* q_s = base + L::off_q;
  uint8_t* p_s = base + L::off_p;
  int32_t* ids_s = reinterpret_cast<int32_t*>(base + L::off_ids);
  uint32_t* valid_s = reinterpret_cast<uint32_t*>(base + L::off_valid);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int n_units = n_rows * (p.n_q_heads / p.group);
  volatile int* abrt = &abort_flag;

  if (tid == 0) {
    for (int i = 0; i < S; ++i) {
      bar_init(&full[i], kProdWarps);
      bar_init(&empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      bar_init(&p_full[i], 32 * kSoftWarps);
      bar_init(&p_empty[i], 1);
    }
    bar_init(&s_full, 1);
    bar_init(&s_free, 32 * kSoftWarps);
    bar_init(&o_full, 1);
    bar_init(&o_free, 32 * kSoftWarps);
    bar_init(&q_free, 1);
    bar_init(&mma_done, 1);
    abort_flag = 0;
    bar_init_fence();
  }
  if (warp == kMmaWarp) tmem_alloc(&tmem_slot, kTmemCols);
  fence_before();
  __syncthreads();
  fence_after();
  const uint32_t tmem = tmem_slot;
  // The selection (sel, cnt) comes from the previous launch.
  grid_dependency_wait();
  grid_dependency_release();

  if (warp >= kSoftWarps && warp < kMmaWarp) {
    // ------------------------------------------------------------ producers
    const int pw = warp - kSoftWarps, ptid = tid - 32 * kSoftWarps;
    const int c8 = lane & 7;
    int kv = 0, arrived = 0, live = 0;
    for (int u = blockIdx.x; u < n_units; u += gridDim.x) {
      const Unit x = unit_at(p, n_rows, u);
      if (x.T == 0) continue;
      const int head0 = x.g * p.group;
      // Every producer warp is past the previous unit's gathers: restage the
      // ids and the sequence's segment table.
      named_sync(2, 32 * kProdWarps);
      for (int k = ptid; k < x.c.cnt; k += 32 * kProdWarps) ids_s[k] = __ldg(x.c.sel_row + k);
      if (ptid < x.c.n_segs) {
        const Segment& sg = p.seg[x.c.seg_begin + ptid];
        segs_s[ptid] = SegS{static_cast<const __nv_bfloat16*>(sg.k), static_cast<const __nv_bfloat16*>(sg.v), sg.first,
                            sg.n, sg.head_stride, sg.tok_stride};
      }
      named_sync(2, 32 * kProdWarps);
      // The query tile (rows >= G zero), once the previous unit's logits MMAs are done with it;
      // its copies complete with the first K tile's.
      if (live > 0) bar_wait(&q_free, (uint32_t)((live - 1) & 1), &g_attn_tc_timeouts, abrt);
      {
        const __nv_bfloat16* qg = static_cast<const __nv_bfloat16*>(p.q) + ((int64_t)x.r * p.n_q_heads + head0) * D;
#pragma unroll
        for (int k = 0; k < kHeads * (D / 8) / (32 * kProdWarps); ++k) {
          const int idx = ptid + k * 32 * kProdWarps;
          const int row = idx / (D / 8), ch = idx % (D / 8);
          const bool ok = row < p.group;
          cp_async16(q_s + (ch >> 3) * (kHeads * 128) + row * 128 + (((ch & 7) ^ (row & 7)) << 4),
                     qg + (ok ? (int64_t)row * D + ch * 8 : 0), ok);
        }
      }
      uint32_t* vbits = valid_s + (live & 1) * (kMaxList / 32);
      for (int ph = 0; ph < 2; ++ph) {
        for (int t = 0; t < x.T; ++t, ++kv) {
          const int slot = kv % S;
          if (kv >= S) bar_wait(&empty[slot], (uint32_t)((kv / S - 1) & 1), &g_attn_tc_timeouts, abrt);
          uint8_t* dst = ring + slot * L::kTileBytes;
          // Lane l locates token 32 pw + l of the tile; each token's row is
          // then copied by 8 lanes, 16 bytes of each 64-channel block apiece.
          const __nv_bfloat16* mine = static_cast<const __nv_bfloat16*>(p.q);
          const bool ok_mine = locate_tok(x.c, ids_s, segs_s, x.g, (int64_t)t * kTok + 32 * pw + lane, ph != 0, mine);
          const uint32_t bits = __ballot_sync(0xffffffffu, ok_mine);
          if (ph == 0 && lane == 0) vbits[t * 4 + pw] = bits;
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const int from = 4 * j + (lane >> 3);
            const int tk = 32 * pw + from;
            const bool ok = (bits >> from) & 1u;
            const __nv_bfloat16* src = reinterpret_cast<const __nv_bfloat16*>(
                __shfl_sync(0xffffffffu, reinterpret_cast<uintptr_t>(mine), from));
            uint8_t* d0 = dst + tk * 128 + ((c8 ^ (tk & 7)) << 4);
#pragma unroll
            for (int s = 0; s < L::kSubs; ++s)
              cp_async16(d0 + s * kSubBytes, ok ? src + s * 64 + c8 * 8 : src, ok);
          }
          cp_async_commit();
          // The tile issued S - 1 tiles ago has landed once at most S - 1 groups are pending.
          if (kv + 1 - arrived > S - 1) {
            cp_async_wait<S - 1>();
            fence_async_smem();
            __syncwarp();
            if (lane == 0) bar_arrive(&full[arrived % S]);
            ++arrived;
          }
        }
      }
      // Hand over the unit's last tiles before staging the next unit.
      cp_async_wait<0>();
      fence_async_smem();
      __syncwarp();
      for (; arrived < kv; ++arrived)
        if (lane == 0) bar_arrive(&full[arrived % S]);
      ++live;
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issue
    if (lane == 0) {
      int kv = 0, live = 0, pc = 0;
      for (int u = blockIdx.x; u < n_units; u += gridDim.x) {
        const Unit x = unit_at(p, n_rows, u);
        if (x.T == 0) continue;
        // Logits: the softmax has read the previous unit's.
        if (live > 0) bar_wait(&s_free, (uint32_t)((live - 1) & 1), &g_attn_tc_timeouts, abrt);
        for (int t = 0; t < x.T; ++t, ++kv) {
          const int slot = kv % S;
          bar_wait(&full[slot], (uint32_t)((kv / S) & 1), &g_attn_tc_timeouts, abrt);
          fence_after();
          const uint8_t* a = ring + slot * L::kTileBytes;
          const uint32_t d = tmem + (uint32_t)(t * kHeads);
#pragma unroll
          for (int s = 0; s < L::kSubs; ++s)
#pragma unroll
            for (int k = 0; k < 4; ++k)
              mma_bf16(d, desc_sw128(a + s * kSubBytes + 32 * k, 16, 1024),
                       desc_sw128(q_s + s * (kHeads * 128) + 32 * k, 16, 1024), kIdescS, (s | k) != 0 ? 1u : 0u);
          commit(&empty[slot]);
        }
        commit(&s_full);
        commit(&q_free);
        // Output: the epilogue has read the previous unit's.
        if (live > 0) bar_wait(&o_free, (uint32_t)((live - 1) & 1), &g_attn_tc_timeouts, abrt);
        for (int t = 0; t < x.T; ++t, ++kv, ++pc) {
          const int slot = kv % S;
          bar_wait(&full[slot], (uint32_t)((kv / S) & 1), &g_attn_tc_timeouts, abrt);
          bar_wait(&p_full[pc & 1], (uint32_t)((pc >> 1) & 1), &g_attn_tc_timeouts, abrt);
          fence_after();
          const uint8_t* a = ring + slot * L::kTileBytes;
          const uint8_t* b = p_s + (pc & 1) * L::kPBytes;
#pragma unroll
          for (int h = 0; h < D / 128; ++h)
#pragma unroll
            for (int k = 0; k < kTok / 16; ++k)
              mma_bf16(tmem + kOCol + (uint32_t)(h * kHeads),
                       desc_sw128(a + h * 2 * kSubBytes + k * 2048, kSubBytes, 1024),
                       desc_sw128(b + (k >> 2) * (kHeads * 128) + (k & 3) * 32, 16, 1024), kIdescO,
                       (t | k) != 0 ? 1u : 0u);
          commit(&empty[slot]);
          commit(&p_empty[pc & 1]);
        }
        commit(&o_full);
        ++live;
      }
      // Every MMA has completed before TMEM is released.
      commit(&mma_done);
      bar_wait(&mma_done, 0u, &g_attn_tc_timeouts);
    }
  } else {
    // ------------------------------------------------------------ softmax and epilogue
    const int q = warp;   // TMEM lanes 32 q ..: tokens 32 q .. of a tile, channels 32 q .. of O^T
    const float c = p.scale * kLog2e;
    const int tk = 32 * q + lane;
    int live = 0, pc = 0;
    for (int u = blockIdx.x; u < n_units; u += gridDim.x) {
      const Unit x = unit_at(p, n_rows, u);
      const int head0 = x.g * p.group;
      const int64_t rh0 = (int64_t)x.r * p.n_q_heads + head0;
      if (x.T == 0) {   // nothing visible: zeros and lse = -inf
        for (int h = 0; h < p.group; ++h)
          for (int d = tk; d < D; d += kTok) store_out(p, (rh0 + h) * D + d, 0.f);
        if (q == 0 && lane < p.group && p.lse) p.lse[rh0 + lane] = -INFINITY;
        continue;
      }
      bar_wait(&s_full, (uint32_t)(live & 1), &g_attn_tc_timeouts, abrt);
      fence_after();
      const uint32_t* vbits = valid_s + (live & 1) * (kMaxList / 32);
      // Pass 1: the maximum logit of each head over the whole list.
      float mx[kHeads];
#pragma unroll
      for (int h = 0; h < kHeads; ++h) mx[h] = -INFINITY;
      for (int t = 0; t < x.T; t += 2) {
        float v[32];
        tmem_ld32(tmem_at(tmem, 32 * q, t * kHeads), v);
        const bool ok0 = (vbits[t * 4 + q] >> lane) & 1u;
        const bool ok1 = t + 1 < x.T && ((vbits[(t + 1) * 4 + q] >> lane) & 1u);
#pragma unroll
        for (int h = 0; h < kHeads; ++h) {
          if (ok0) mx[h] = fmaxf(mx[h], v[h]);
          if (ok1) mx[h] = fmaxf(mx[h], v[kHeads + h]);
        }
      }
      warp_reduce16<true>(mx, lane);
      if ((lane & 1) == 0) red_m[q][reduced_index(lane)] = mx[0];
      named_sync(1, 32 * kSoftWarps);
      float m[kHeads];
#pragma unroll
      for (int h = 0; h < kHeads; ++h)
        m[h] = fmaxf(fmaxf(red_m[0][h], red_m[1][h]), fmaxf(red_m[2][h], red_m[3][h]));
      // Pass 2: P = exp(S - m) in bf16 for the output MMAs, and the row sums.
      float ls[kHeads];
#pragma unroll
      for (int h = 0; h < kHeads; ++h) ls[h] = 0.f;
      for (int t = 0; t < x.T; ++t, ++pc) {
        const int buf = pc & 1;
        if (pc >= 2) bar_wait(&p_empty[buf], (uint32_t)(((pc >> 1) - 1) & 1), &g_attn_tc_timeouts, abrt);
        float v[kHeads];
        tmem_ld16(tmem_at(tmem, 32 * q, t * kHeads), v);
        const bool ok = (vbits[t * 4 + q] >> lane) & 1u;
        uint8_t* pb = p_s + buf * L::kPBytes + (tk >> 6) * (kHeads * 128) + (tk & 7) * 2;
        const int chunk = (tk & 63) >> 3;
#pragma unroll
        for (int h = 0; h < kHeads; ++h) {
          const float e = (ok && h < p.group && m[h] != -INFINITY) ? exp2f((v[h] - m[h]) * c) : 0.f;
          ls[h] += e;
          *reinterpret_cast<__nv_bfloat16*>(pb + h * 128 + ((chunk ^ (h & 7)) << 4)) = __float2bfloat16(e);
        }
        fence_async_smem();
        bar_arrive(&p_full[buf]);
      }
      fence_before();
      bar_arrive(&s_free);
      warp_reduce16<false>(ls, lane);
      if ((lane & 1) == 0) red_l[q][reduced_index(lane)] = ls[0];
      named_sync(1, 32 * kSoftWarps);
      float l[kHeads];
#pragma unroll
      for (int h = 0; h < kHeads; ++h) l[h] = (red_l[0][h] + red_l[1][h]) + (red_l[2][h] + red_l[3][h]);
      // Epilogue: O^T lanes are channels; write O / l and the lse.
      bar_wait(&o_full, (uint32_t)(live & 1), &g_attn_tc_timeouts, abrt);
      fence_after();
      float o[D / 128][kHeads];
#pragma unroll
      for (int h = 0; h < D / 128; ++h) tmem_ld16(tmem_at(tmem, 32 * q, kOCol + h * kHeads), o[h]);
      fence_before();
      bar_arrive(&o_free);
#pragma unroll
      for (int h = 0; h < kHeads; ++h) {
        if (h >= p.group) break;
        const float inv = l[h] > 0.f ? 1.f / l[h] : 0.f;
#pragma unroll
        for (int hh = 0; hh < D / 128; ++hh) store_out(p, (rh0 + h) * D + 128 * hh + tk, o[hh][h] * inv);
      }
      if (q == 0 && lane < p.group && p.lse) {
        float ml = -INFINITY, ll = 0.f;
#pragma unroll
        for (int h = 0; h < kHeads; ++h)
          if (h == lane) {
            ml = m[h];
            ll = l[h];
          }
        p.lse[rh0 + lane] = ll > 0.f ? (ml * c + log2f(ll)) * kLn2 : -INFINITY;
      }
      ++live;
    }
  }

  fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

template <int D, int NSEQ>
cudaError_t launch_d(const AttnParams<NSEQ>& p, int n_rows, cudaStream_t st) {
  const size_t smem = TcLayout<D>::alloc;
  cudaError_t e = allow_dynamic_smem((const void*)attn_tc_kernel<D, NSEQ>, smem);
  if (e != cudaSuccess) return e;
  const int64_t units = (int64_t)n_rows * (p.n_q_heads / p.group);
  const int sms = device_sm_count();
  const unsigned grid = (unsigned)(units < sms ? units : sms);
  return launch_kernel(attn_tc_kernel<D, NSEQ>, dim3(grid), dim3(kThreads), smem, st, 0u, p, n_rows);
}

}  // namespace

bool attn_tc_eligible(qsa_dtype kv_dtype, int head_dim, int group, int64_t max_list, int64_t rows) {
  return kv_dtype == QSA_BF16 && (head_dim == 128 || head_dim == 256) && group <= kHeads && max_list <= kMaxList &&
         rows >= kAttnTcMinRows;
}

template <int NSEQ>
cudaError_t launch_attn_tc(const AttnParams<NSEQ>& p, int n_rows, cudaStream_t st) {
  if (n_rows == 0) return cudaSuccess;
  if (p.n_splits != 1) return cudaErrorInvalidValue;
  return p.head_dim == 256 ? launch_d<256, NSEQ>(p, n_rows, st) : launch_d<128, NSEQ>(p, n_rows, st);
}

template cudaError_t launch_attn_tc<1>(const AttnParams<1>&, int, cudaStream_t);
template cudaError_t launch_attn_tc<kLaunchSeqs>(const AttnParams<kLaunchSeqs>&, int, cudaStream_t);

int attn_tc_bad_ids_take() { return take_counter(g_bad_ids); }

int attn_tc_wait_timeouts() {
  int v = 0;
  return cudaMemcpyFromSymbol(&v, g_attn_tc_timeouts, sizeof(int)) == cudaSuccess ? v : -1;
}

}  // namespace qsa
