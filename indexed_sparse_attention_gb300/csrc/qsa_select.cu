// Step 3 of the QSA layer step: per query row, the top-k pooled blocks by
// score, the lower block id first among equal scores, listed in ascending id
// order (hipfire, "QSA sparse attention and the VMM KV backend", section 02:
// a budget of 512 blocks = 2,048 tokens; section 03: selection by a radix
// select over the scores).
//
// One CTA per row runs an exact radix select over order-preserving 32-bit
// keys of the fp32 scores (-0.0 folded onto +0.0), restricted to candidate
// groups.  A group is QSA_SCORE_GROUP = 16 consecutive blocks; its maximum
// comes from the scoring kernel or is computed here from the scores.
//  1. Histogram the G group maxima on their top 12 key bits and find the bin
//     B of the k-th largest.  The k largest group maxima are the scores of k
//     different blocks, so the k-th best block score is at least the k-th
//     largest group maximum, whose key lies in bin B or above: every block of
//     the top k has a key in a bin >= B and sits in a group whose maximum is
//     in a bin >= B.  With fewer than k groups nothing is pruned.
//  2. Read the blocks of the candidate groups (maximum in a bin >= B) and
//     keep those whose own key is in a bin >= B as a (key, id) list.
//  3. Radix select over the list (12 + 12 + 8 key bits, stopping early when
//     a bin is taken whole) gives the k-th key K and how many entries equal
//     to K to keep -- the lowest ids.
//  4. The kept ids are marked in a bitmap over the row's blocks, which one
//     prefix scan turns into the ascending id list.
// A row whose candidates exceed the shared-memory capacity (many equal or
// nearly equal scores) runs steps 3 and 4 over its whole score row in
// global memory instead.
#include "qsa_internal.cuh"

namespace qsa {

namespace {

constexpr int kThreads = 1024;
constexpr int kWarps = kThreads / 32;

// NaN scores met among the candidates (read and cleared by
// qsa_check_device_status): order keys above +inf's or below -inf's.
__device__ int g_nan_keys;
constexpr int kGroup = QSA_SCORE_GROUP;
constexpr int kBins = 4096;                        // radix levels 1 and 2: 12 key bits each
constexpr int kBins3 = 256;                        // radix level 3: the last 8 key bits
constexpr int kGroupCap = 1024;                    // candidate groups read back (16,384 blocks)
constexpr int kListCap = 8192;                     // candidate (key, id) pairs kept
constexpr int kLoadBatch = 4;                                  // group maxima a thread loads per pass
constexpr int kChunkBatch = 4;                                  // float4 chunks a thread loads per pass
// Every region of SelLayout starts on a multiple of 4 words (the clears and
// the list's chunk loads use 16-byte accesses).
static_assert(kBins % 4 == 0 && kBins3 % 4 == 0 && kGroupCap % 4 == 0 && kListCap % 4 == 0,
              "shared-memory regions on 16-byte boundaries");


// Shared-memory layout (32-bit words); R1 holds the group-maximum keys, then
// the list keys.
struct SelLayout {
  int h1, h2, h3, cg, r1, r2, selw, eqw, total;
  __host__ __device__ SelLayout(int64_t max_nb) {
    const int groups = (int)((max_nb + kGroup - 1) / kGroup);
    const int nw = (int)((max_nb + 31) / 32);
    h1 = 0;                                        // group-maximum histogram, then radix level 2
    h2 = h1 + kBins;                               // radix level 1
    h3 = h2 + kBins;                               // radix level 3
    cg = h3 + kBins3;                              // candidate group ids
    r1 = cg + kGroupCap;
    r2 = r1 + (groups > kListCap ? (groups + 3) / 4 * 4 : kListCap);   // list ids (16-byte aligned)
    selw = r2 + kListCap;                          // kept ids, one bit per block
    eqw = selw + (nw + 3) / 4 * 4;                 // entries equal to the k-th key
    total = eqw + (nw + 3) / 4 * 4;
  }
};

__device__ __forceinline__ uint32_t lanes_below() {
  uint32_t m;
  asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
  return m;
}

// Exclusive prefix sum of v over the warps of the CTA (v uniform within each
// warp, warp order); *total = the sum over warps.  wt (NT / 32 words) must not
// be touched again before the next __syncthreads() after this call.
template <int NT>
__device__ __forceinline__ uint32_t warp_prefix(uint32_t v, uint32_t* wt, uint32_t* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (lane == 0) wt[warp] = v;
  __syncthreads();
  const uint32_t w = lane < NT / 32 ? wt[lane] : 0u;
  *total = __reduce_add_sync(0xffffffffu, w);
  return __reduce_add_sync(0xffffffffu, lane < warp ? w : 0u);
}

// Exclusive prefix sum of v over the CTA in thread order (same contract on wt).
template <int NT>
__device__ __forceinline__ uint32_t block_scan(uint32_t v, uint32_t* wt, uint32_t* total) {
  const int lane = threadIdx.x & 31;
  uint32_t x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  return warp_prefix<NT>(__shfl_sync(0xffffffffu, x, 31), wt, total) + x - v;
}

// Bin (of nbins = kBins or kBins3) holding the need-th largest key counted in
// hist: s_res[0] = the bin, s_res[1] = keys in higher bins.  The histogram
// holds at least need >= 1 keys.  Ends with a barrier.
template <int NT>
__device__ __forceinline__ void find_bin(const uint32_t* hist, int nbins, uint32_t need, uint32_t* wt,
                                         uint32_t* s_res) {
  const int tid = threadIdx.x;
  constexpr int P = kBins / NT;
  static_assert(kBins % (4 * NT) == 0 && NT >= kBins3 && NT <= 1024, "thread count");
  uint32_t c[P];   // c[j] = count of bin top - 1 - j
  int per, top;
  if (nbins == kBins) {
    per = P;
    top = kBins - P * tid;
#pragma unroll
    for (int q = 0; q < P / 4; ++q) {
      const uint4 u = *reinterpret_cast<const uint4*>(hist + top - 4 * (q + 1));
      c[4 * q] = u.w;
      c[4 * q + 1] = u.z;
      c[4 * q + 2] = u.y;
      c[4 * q + 3] = u.x;
    }
  } else {
    per = tid < nbins ? 1 : 0;
    top = nbins - tid;
    c[0] = per ? hist[top - 1] : 0u;
#pragma unroll
    for (int j = 1; j < P; ++j) c[j] = 0u;
  }
  uint32_t local = 0u;
#pragma unroll
  for (int j = 0; j < P; ++j) local += c[j];
  uint32_t total;
  const uint32_t above = block_scan<NT>(local, wt, &total);
  if (above < need && above + local >= need) {
    uint32_t acc = above;
#pragma unroll
    for (int j = 0; j < P; ++j) {
      if (j < per) {
        if (acc + c[j] >= need) {
          s_res[0] = (uint32_t)(top - 1 - j);
          s_res[1] = acc;
          break;
        }
        acc += c[j];
      }
    }
  }
  __syncthreads();
}

// Warp-aggregated shared-memory histogram increment (one atomic per distinct
// bin among the active lanes); all 32 lanes of the warp must call it.  Used
// where many keys can share a bin.
__device__ __forceinline__ void hist_add(uint32_t* hist, bool act, uint32_t bin) {
  const uint32_t peers = __match_any_sync(0xffffffffu, act ? bin : 0xffffffffu);
  if (act && (__ffs(peers) - 1) == (int)(threadIdx.x & 31)) atomicAdd(&hist[bin], (uint32_t)__popc(peers));
}

// Maximum of the scores of blocks 16g .. min(16g + 16, nb) - 1 (the row's
// stride keeps every group start 16-byte aligned).
__device__ __forceinline__ float group_max_of(const float* srow, int64_t g, int64_t nb) {
  const int64_t b0 = g * kGroup;
  float m = -INFINITY;
  if (b0 + kGroup <= nb) {
    const float4* v = reinterpret_cast<const float4*>(srow + b0);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float4 x = __ldg(v + j);
      m = fmaxf(m, fmaxf(fmaxf(x.x, x.y), fmaxf(x.z, x.w)));
    }
  } else {
    for (int64_t b = b0; b < nb; ++b) m = fmaxf(m, __ldg(srow + b));
  }
  return m;
}

// The k-th key of a candidate set by radix levels of 12, 12 and 8 key bits
// (stopping early when a bin is taken whole): entries whose masked key
// (key & mask) exceeds K are kept; of those equal to K, all when all_eq,
// else the `need` lowest ids.  for_each(f) calls f(key, id) for every
// candidate (key != 0), each exactly once over the CTA's threads, and
// for_each_warp(f) does the same with all 32 lanes of every warp calling f
// the same number of times (f(key, id, active)).  level1_done: the caller
// already filled the level-1 histogram (h2).  Ends with a barrier.
struct Threshold {
  uint32_t K, mask, need;
  bool all_eq;
};

template <int NT, typename ForEach, typename ForEachWarp>
__device__ __forceinline__ Threshold radix_threshold(uint32_t k, ForEach for_each, ForEachWarp for_each_warp,
                                                     uint32_t* sm, const SelLayout& L, bool level1_done,
                                                     uint32_t (*wt)[NT / 32], uint32_t* s_res) {
  uint32_t* h1 = sm + L.h1;
  uint32_t* h2 = sm + L.h2;
  uint32_t* h3 = sm + L.h3;
  if (!level1_done) {
    for_each_warp([&](uint32_t key, int32_t, bool act) { hist_add(h2, act, key >> 20); });
    __syncthreads();
  }
  uint32_t need = k;
  find_bin<NT>(h2, kBins, need, wt[0], s_res);
  const uint32_t b1 = s_res[0];
  need -= s_res[1];
  uint32_t K = b1 << 20, mask = 0xfff00000u;
  uint32_t n_eq = h2[b1];   // entries whose masked key equals K
  if (n_eq != need) {
    // Level 2: key bits 19..8 of the keys in bin b1.
    for_each([&](uint32_t key, int32_t) {
      if ((key & 0xfff00000u) == K) atomicAdd(&h1[(key >> 8) & (kBins - 1)], 1u);
    });
    __syncthreads();
    find_bin<NT>(h1, kBins, need, wt[1], s_res);
    const uint32_t b2 = s_res[0];
    need -= s_res[1];
    K |= b2 << 8;
    mask = 0xffffff00u;
    n_eq = h1[b2];
    if (n_eq != need) {
      // Level 3: the last 8 key bits.
      for_each([&](uint32_t key, int32_t) {
        if ((key & 0xffffff00u) == K) atomicAdd(&h3[key & (kBins3 - 1)], 1u);
      });
      __syncthreads();
      find_bin<NT>(h3, kBins3, need, wt[0], s_res);
      K |= s_res[0];
      mask = 0xffffffffu;
      need -= s_res[1];
      n_eq = h3[s_res[0]];
    }
  }
  return Threshold{K, mask, need, n_eq == need};
}

// Steps 3 and 4 over the candidates (for_each, for_each_warp and
// level1_done as for radix_threshold): the kept ids are marked in a bitmap
// over the row's blocks and written ascending to out.
template <int NT, typename ForEach, typename ForEachWarp>
__device__ __forceinline__ void radix_and_write(uint32_t k, int nw, ForEach for_each, ForEachWarp for_each_warp,
                                                uint32_t* sm, const SelLayout& L, bool level1_done,
                                                uint32_t (*wt)[NT / 32], uint32_t* s_res, int32_t* out) {
  const int tid = threadIdx.x;
  uint32_t* selw = sm + L.selw;
  uint32_t* eqw = sm + L.eqw;
  const Threshold th = radix_threshold<NT>(k, for_each, for_each_warp, sm, L, level1_done, wt, s_res);
  const uint32_t K = th.K, mask = th.mask, need = th.need;
  // Step 4: mark the kept ids.  Entries above K are kept; so are those equal
  // to K when all of them fit, else the `need` lowest ids among them.
  const bool all_eq = th.all_eq;
  for_each([&](uint32_t key, int32_t id) {
    if (key > 0xff800000u || key < 0x007fffffu) atomicAdd(&g_nan_keys, 1);
    const uint32_t m = key & mask;
    if (m > K || (all_eq && m == K)) atomicOr(&selw[id >> 5], 1u << (id & 31));
    else if (m == K) atomicOr(&eqw[id >> 5], 1u << (id & 31));
  });
  __syncthreads();
  const int wpt = (nw + NT - 1) / NT;
  const int a0 = min(nw, tid * wpt), a1 = min(nw, a0 + wpt);
  uint32_t total;
  if (!all_eq) {
    uint32_t c = 0u;
    for (int i = a0; i < a1; ++i) c += __popc(eqw[i]);
    uint32_t before = block_scan<NT>(c, wt[1], &total);
    for (int i = a0; i < a1; ++i) {
      uint32_t e = eqw[i];
      const uint32_t pc = __popc(e);
      if (before >= need) {
        e = 0u;
      } else if (before + pc > need) {   // keep the lowest need - before bits
        uint32_t keep = 0u;
        for (uint32_t j = 0; j < need - before; ++j) {
          keep |= e & (0u - e);
          e &= e - 1u;
        }
        e = keep;
      }
      before += pc;
      selw[i] |= e;
    }
    __syncthreads();
  }
  uint32_t c = 0u;
  for (int i = a0; i < a1; ++i) c += __popc(selw[i]);
  uint32_t at = block_scan<NT>(c, wt[0], &total);
  for (int i = a0; i < a1; ++i) {
    uint32_t e = selw[i];
    while (e) {
      const int b = __ffs(e) - 1;
      e &= e - 1u;
      // (Positions stay below k for scores that obey the contract; the bound
      // also keeps NaN keys from writing outside the row.)
      if (at < k) out[at] = i * 32 + b;
      ++at;
    }
  }
}

// MINB: CTAs per SM the register budget allows (2 for calls of many rows,
// whose CTAs then share SMs; 1 keeps the fewest-row latency lowest).
template <int NSEQ, int MINB, int NT>
__global__ void __launch_bounds__(NT, MINB) select_kernel(const SelectParams<NSEQ> p, int64_t max_nb) {
  extern __shared__ __align__(16) uint32_t sm[];
  __shared__ uint32_t wt[2][(NT / 32)];
  __shared__ uint32_t s_res[2];
  __shared__ uint32_t s_cnt;
  const SelLayout L(max_nb);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  // The three histograms and the two bitmaps, 16 bytes per store (every
  // region starts and ends on a multiple of 4 words).
  uint4* sm4 = reinterpret_cast<uint4*>(sm);
  for (int i = tid; i < L.cg / 4; i += NT) sm4[i] = make_uint4(0u, 0u, 0u, 0u);
  for (int i = L.selw / 4 + tid; i < L.total / 4; i += NT) sm4[i] = make_uint4(0u, 0u, 0u, 0u);
  if (tid == 0) {
    s_res[0] = 0u;
    s_res[1] = 0u;
    s_cnt = 0u;
  }
  grid_dependency_sync();
  const int r = p.row_base + (int)blockIdx.x;
  int si = 0;
#pragma unroll
  for (int i = 1; i < NSEQ; ++i)
    if (i < p.n_seqs && r >= p.seq[i].row_begin) si = i;
  const RowSeq sq = p.seq[si];
  const int64_t nb = visible_blocks(row_position(sq.n_tokens, sq.n_rows, r - sq.row_begin));
  const int k = p.top_k;
  int32_t* out = p.sel + (int64_t)r * k;
  if (nb <= k) {
    for (int i = tid; i < k; i += NT) out[i] = i < nb ? i : -1;
    if (tid == 0) p.cnt[r] = (int32_t)nb;
    return;
  }
  const float* srow = p.scores + (int64_t)r * p.ld;
  const int G = (int)((nb + kGroup - 1) / kGroup);   // <= kMaxGroups
  const int nw = (int)((nb + 31) / 32);
  uint32_t* r1 = sm + L.r1;
  uint32_t* r2 = sm + L.r2;
  uint32_t* cg = sm + L.cg;
  uint32_t* h1 = sm + L.h1;
  uint32_t* h2 = sm + L.h2;
  __syncthreads();   // histograms and bitmaps cleared

  // 1. Keys of the group maxima (all loads in flight at once) and their
  // top-12-bit histogram.
  if (p.gmax) {
    const float* grow = p.gmax + (int64_t)r * p.gld;
    for (int g0 = 0; g0 < G; g0 += kLoadBatch * NT) {
      float v[kLoadBatch];
#pragma unroll
      for (int j = 0; j < kLoadBatch; ++j) {
        const int g = g0 + tid + j * NT;
        v[j] = g < G ? __ldg(grow + g) : 0.f;
      }
#pragma unroll
      for (int j = 0; j < kLoadBatch; ++j) {
        const int g = g0 + tid + j * NT;
        if (g < G) {
          const uint32_t key = order_key(v[j]);
          r1[g] = key;
          atomicAdd(&h1[key >> 20], 1u);
        }
      }
    }
  } else {
#pragma unroll 1
    for (int g = tid; g < G; g += NT) {
      const uint32_t key = order_key(group_max_of(srow, g, nb));
      r1[g] = key;
      atomicAdd(&h1[key >> 20], 1u);
    }
  }
  __syncthreads();
  const bool prune = G >= k;
  uint32_t B = 0u;
  if (prune) {
    find_bin<NT>(h1, kBins, (uint32_t)k, wt[0], s_res);
    B = s_res[0];
  }

  // 2a. Candidate groups: warp w owns a contiguous run of groups, 32 per round.
  const int gpw = (G + (NT / 32) * 32 - 1) / ((NT / 32) * 32) * 32;
  const int ga = min(G, warp * gpw), gb = min(G, ga + gpw);
  uint32_t c = 0u;
  for (int g0 = ga; g0 < gb; g0 += 32) {
    const int g = g0 + lane;
    c += __popc(__ballot_sync(0xffffffffu, g < gb && (r1[g] >> 20) >= B));
  }
  uint32_t n_cg;
  uint32_t q = warp_prefix<NT>(c, wt[1], &n_cg);
  bool overflow = n_cg > (uint32_t)kGroupCap;
  if (!overflow) {
    const uint32_t below = lanes_below();
    for (int g0 = ga; g0 < gb; g0 += 32) {
      const int g = g0 + lane;
      const bool in = g < gb && (r1[g] >> 20) >= B;
      const uint32_t bal = __ballot_sync(0xffffffffu, in);
      if (in) cg[q + __popc(bal & below)] = (uint32_t)g;
      q += __popc(bal);
    }
  }
  for (int i = tid; i < kBins / 4; i += NT) sm4[L.h1 / 4 + i] = make_uint4(0u, 0u, 0u, 0u);   // reused by radix level 2
  __syncthreads();

  uint32_t n_list = 0u;
  if (!overflow) {
    // 2b. The candidate groups' blocks, 4 per float4 chunk, all loads in
    // flight at once; keys in a bin >= B join the list and its level-1
    // histogram.
    const int n_ch = (int)n_cg * (kGroup / 4);
    for (int c0 = 0; c0 < n_ch; c0 += kChunkBatch * NT) {
    float4 v[kChunkBatch];
#pragma unroll
    for (int j = 0; j < kChunkBatch; ++j) {
      const int ch = c0 + tid + j * NT;
      v[j] = make_float4(0.f, 0.f, 0.f, 0.f);
      // A chunk that starts below nb ends within the row stride (both
      // multiples of 4); its blocks >= nb are dropped below.
      const int64_t b0 = ch < n_ch ? (int64_t)cg[ch >> 2] * kGroup + 4 * (ch & 3) : nb;
      if (b0 < nb) v[j] = __ldg(reinterpret_cast<const float4*>(srow + b0));
    }
#pragma unroll
    for (int j = 0; j < kChunkBatch; ++j) {
      const int ch = c0 + tid + j * NT;
      if (ch < n_ch) {
        const int64_t b0 = (int64_t)cg[ch >> 2] * kGroup + 4 * (ch & 3);
        const float x[4] = {v[j].x, v[j].y, v[j].z, v[j].w};
        uint32_t key[4];
        int n = 0;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          key[e] = order_key(x[e]);
          if (b0 + e >= nb || (key[e] >> 20) < B) key[e] = 0u;
          n += key[e] != 0u;
        }
        if (n) {
          uint32_t at = atomicAdd(&s_cnt, (uint32_t)n);
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            if (key[e] != 0u) {
              if (at < (uint32_t)kListCap) {
                r1[at] = key[e];
                r2[at] = (uint32_t)(b0 + e);
              }
              ++at;
              atomicAdd(&h2[key[e] >> 20], 1u);
            }
          }
        }
      }
    }
    }
    __syncthreads();
    n_list = s_cnt;
    overflow = n_list > (uint32_t)kListCap;
  }
  if (!overflow) {
    const int n = (int)n_list;
    radix_and_write<NT>(
        (uint32_t)k, nw,
        [&](auto f) {
          for (int i = tid; i < n; i += NT) f(r1[i], (int32_t)r2[i]);
        },
        [&](auto f) {
          const int n_pad = (n + 31) / 32 * 32;
          for (int i = tid; i < n_pad; i += NT) f(i < n ? r1[i] : 0u, i < n ? (int32_t)r2[i] : 0, i < n);
        },
        sm, L, true, wt, s_res, out);
  } else {
    // The whole row from global memory (the level-1 histogram is rebuilt).
    if (n_list) {
      for (int i = tid; i < kBins; i += NT) h2[i] = 0u;
      __syncthreads();
    }
    const int nbi = (int)nb;
    radix_and_write<NT>(
        (uint32_t)k, nw,
        [&](auto f) {
          for (int b0 = tid; b0 < nbi; b0 += 8 * NT) {   // 8 loads in flight
            uint32_t kk[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              const int b = b0 + j * NT;
              kk[j] = b < nbi ? order_key(__ldg(srow + b)) : 0u;
            }
#pragma unroll
            for (int j = 0; j < 8; ++j)
              if (b0 + j * NT < nbi) f(kk[j], (int32_t)(b0 + j * NT));
          }
        },
        [&](auto f) {
          const int n_pad = (nbi + 31) / 32 * 32;   // warp-uniform trip counts
          for (int b0 = tid; b0 < n_pad; b0 += 8 * NT) {
            uint32_t kk[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              const int b = b0 + j * NT;
              kk[j] = b < nbi ? order_key(__ldg(srow + b)) : 0u;
            }
#pragma unroll
            for (int j = 0; j < 8; ++j) f(kk[j], (int32_t)(b0 + j * NT), b0 + j * NT < nbi);
          }
        },
        sm, L, false, wt, s_res, out);
  }
  if (tid == 0) p.cnt[r] = k;
}

// ------------------------------------------------------------------ selection over key-axis chunks
// One CTA per row merges the row's running top-k (keys and ids, ascending
// ids) with the scores of one chunk of blocks [block_lo, block_lo + n_blocks):
// the top-k of the union equals the top-k over the whole row once every chunk
// has been merged (the SGLang launcher notes, section 2.3: top-k of a union
// equals the top-k of the per-part top-k lists).  The union is laid out in
// ascending id order -- the running entries, whose ids precede the chunk's,
// then the chunk's blocks the row can see -- so the radix select's rule
// "lowest index among keys equal to the k-th" is the method's lowest-id rule.
// Once the running list holds k entries, a chunk block enters the union only
// with a key above the list's smallest (it cannot displace an entry of equal
// key and lower id), which leaves few chunk entries after the first chunks.
__global__ void __launch_bounds__(kThreads) merge_select_kernel(const MergeSelectParams p, int64_t max_union) {
  extern __shared__ __align__(16) uint32_t sm[];
  __shared__ uint32_t wt[2][kWarps];
  __shared__ uint32_t s_res[2];
  __shared__ int32_t out_s[QSA_MAX_TOP_K];
  const SelLayout L(max_union);
  const int tid = threadIdx.x;
  // The three histograms and the two bitmaps, 16 bytes per store.
  uint4* sm4 = reinterpret_cast<uint4*>(sm);
  for (int i = tid; i < L.cg / 4; i += kThreads) sm4[i] = make_uint4(0u, 0u, 0u, 0u);
  for (int i = L.selw / 4 + tid; i < L.total / 4; i += kThreads) sm4[i] = make_uint4(0u, 0u, 0u, 0u);
  if (tid == 0) {
    s_res[0] = 0u;
    s_res[1] = 0u;
  }
  grid_dependency_sync();
  const int r = (int)blockIdx.x;
  const int k = p.top_k;
  const int64_t nb = visible_blocks(row_position(p.n_tokens, p.n_rows, r));
  const int n_run = p.first ? 0 : max(0, min(k, p.run_cnt_in[r]));
  const int vis = (int)max((int64_t)0, min((int64_t)p.n_blocks, nb - p.block_lo));
  uint32_t* keys = sm + L.r1;
  uint32_t* ids = sm + L.r2;
  // The running entries, and their smallest key when they are k: a chunk
  // block can only enter with a larger key (on an equal key the running
  // entry's lower id wins).
  uint32_t run_min = 0xffffffffu;
  for (int u = tid; u < n_run; u += kThreads) {
    const uint32_t key = p.run_key_in[(int64_t)r * k + u];
    keys[u] = key;
    ids[u] = (uint32_t)p.run_id_in[(int64_t)r * k + u];
    run_min = min(run_min, key);
  }
#pragma unroll
  for (int o = 16; o; o >>= 1) run_min = min(run_min, __shfl_xor_sync(0xffffffffu, run_min, o));
  if ((tid & 31) == 0) wt[0][tid >> 5] = run_min;
  __syncthreads();
  run_min = (tid & 31) < kWarps ? wt[0][tid & 31] : 0xffffffffu;
#pragma unroll
  for (int o = 16; o; o >>= 1) run_min = min(run_min, __shfl_xor_sync(0xffffffffu, run_min, o));
  const uint32_t floor_key = n_run == k ? run_min : 0u;   // chunk keys must exceed this
  // The chunk's blocks above the floor, appended in id order: thread t takes
  // a contiguous run, a block-wide scan places it.
  const float* crow = p.chunk + (int64_t)r * p.ld_chunk;
  const int per = (vis + kThreads - 1) / kThreads;
  const int j0 = min(vis, tid * per), j1 = min(vis, j0 + per);
  uint32_t c = 0u;
  for (int j = j0; j < j1; ++j) c += order_key(__ldg(crow + j)) > floor_key;
  uint32_t total;
  uint32_t at = (uint32_t)n_run + block_scan<kThreads>(c, wt[1], &total);
  for (int j = j0; j < j1; ++j) {
    const uint32_t key = order_key(__ldg(crow + j));
    if (key > floor_key) {
      keys[at] = key;
      ids[at] = (uint32_t)(p.block_lo + j);
      ++at;
    }
  }
  const int n_union = n_run + (int)total;
  __syncthreads();
  int n_sel;
  if (n_union <= k) {
    n_sel = n_union;
    for (int i = tid; i < n_union; i += kThreads) out_s[i] = i;
  } else {
    n_sel = k;
    radix_and_write<kThreads>(
        (uint32_t)k, (n_union + 31) / 32,
        [&](auto f) {
          for (int i = tid; i < n_union; i += kThreads) f(keys[i], (int32_t)i);
        },
        [&](auto f) {
          const int n_pad = (n_union + 31) / 32 * 32;
          for (int i = tid; i < n_pad; i += kThreads) f(i < n_union ? keys[i] : 0u, (int32_t)i, i < n_union);
        },
        sm, L, false, wt, s_res, out_s);
  }
  __syncthreads();
  // The kept entries in ascending union index = ascending id order.
  const int64_t grow = (int64_t)p.row_begin + r;
  for (int i = tid; i < n_sel; i += kThreads) {
    const int u = out_s[i];
    const int32_t id = (int32_t)ids[u];
    if (p.last) {
      p.sel[grow * k + i] = id;
    } else {
      p.run_key_out[(int64_t)r * k + i] = keys[u];
      p.run_id_out[(int64_t)r * k + i] = id;
    }
  }
  if (p.last) {
    for (int i = n_sel + tid; i < k; i += kThreads) p.sel[grow * k + i] = -1;
    if (tid == 0) p.cnt[grow] = n_sel;
  } else if (tid == 0) {
    p.run_cnt_out[r] = n_sel;
  }
}

}  // namespace

size_t select_smem_bytes(int64_t max_nb) { return sizeof(uint32_t) * (size_t)SelLayout(max_nb).total; }

int merge_select_max_union() { return kListCap; }

int select_nan_keys_take() { return take_counter(g_nan_keys); }

cudaError_t launch_merge_select(const MergeSelectParams& p, cudaStream_t st) {
  if (p.n_rows == 0) return cudaSuccess;
  const int64_t max_union = (int64_t)p.top_k + p.n_blocks;
  if (max_union > kListCap || p.top_k > QSA_MAX_TOP_K) return cudaErrorInvalidValue;
  const size_t smem = select_smem_bytes(max_union);
  cudaError_t e = allow_dynamic_smem((const void*)merge_select_kernel, smem);
  if (e != cudaSuccess) return e;
  return launch_kernel(merge_select_kernel, dim3((unsigned)p.n_rows), dim3(kThreads), smem, st, 0u, p, max_union);
}

template <int NSEQ>
cudaError_t launch_select(const SelectParams<NSEQ>& p, int n_rows, int64_t max_nb, cudaStream_t st) {
  if (n_rows == 0) return cudaSuccess;
  const size_t smem = select_smem_bytes(max_nb);
  // More rows than SMs: CTAs of 512 threads, two per SM where shared memory
  // allows it (more rows in flight); few rows: 1,024 threads, whose per-row
  // latency is lowest.
  const bool many = n_rows > device_sm_count() && 2 * (smem + 2048) <= 228 * 1024;
  auto* kernel = many ? select_kernel<NSEQ, 2, 512> : select_kernel<NSEQ, 1, 1024>;
  cudaError_t e = allow_dynamic_smem((const void*)kernel, smem);
  if (e != cudaSuccess) return e;
  return launch_kernel(kernel, dim3((unsigned)n_rows), dim3(many ? 512 : 1024), smem, st, 0u, p, max_nb);
}

template cudaError_t launch_select<1>(const SelectParams<1>&, int, int64_t, cudaStream_t);
template cudaError_t launch_select<kLaunchSeqs>(const SelectParams<kLaunchSeqs>&, int, int64_t, cudaStream_t);

}  // namespace qsa
