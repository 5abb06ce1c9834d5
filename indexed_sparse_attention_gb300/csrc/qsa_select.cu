// Step 3 of the QSA layer step: per query row, keep the top-k complete
// blocks by score, lower block id winning ties (hipfire, "QSA sparse
// attention and the VMM KV backend", section 02: the top-scoring blocks
// within a 2,048-token budget of 512 blocks; section 03: a radix select from
// the scores).
//
// Scores map to order-preserving uint32 keys (-0.0 folded onto +0.0).  One
// thread-block cluster of S CTAs handles one row; CTA c owns a chunk of the
// row's blocks and keeps its keys in shared memory.  In one launch:
//   1. each CTA histograms its keys over the top 12 key bits (4096 bins);
//   2. the histograms are summed across the cluster through distributed
//      shared memory (CTA c sums bin slice c of every peer and broadcasts it),
//      and every CTA finds the bin B holding the row's k-th best key;
//   3. each CTA writes one bitmap word per 32 of its ids -- ids whose bin is
//      above B -- into CTA 0, and appends the ids in bin B (the candidates)
//      to CTA 0's candidate list;
//   4. CTA 0 resolves the candidates with two more radix passes over the low
//      20 key bits, keeps the lowest ids among keys equal to the k-th key,
//      and writes the row's ids in ascending order by a prefix popcount over
//      the bitmap.
// If bin B holds more candidates than the list takes (massive ties), CTA 0
// runs the remaining radix passes over the row's scores instead.
#include <cooperative_groups.h>

#include "qsa_internal.cuh"

namespace cg = cooperative_groups;

namespace qsa {

namespace {

constexpr int kBins = kSelBins;      // top 12 key bits
constexpr int kCandCap = 2048;       // candidates kept by CTA 0
constexpr int kThreads = 512;
constexpr int kMaxCluster = 16;

// Exclusive prefix sum of v over the CTA; *total gets the sum of all v.
__device__ __forceinline__ uint32_t block_exclusive_scan(uint32_t v, uint32_t* warp_sums, uint32_t* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int n_warps = blockDim.x >> 5;
  uint32_t x = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, x, off);
    if (lane >= off) x += y;
  }
  if (lane == 31) warp_sums[warp] = x;
  __syncthreads();
  if (warp == 0) {
    uint32_t s = lane < n_warps ? warp_sums[lane] : 0u;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const uint32_t y = __shfl_up_sync(0xffffffffu, s, off);
      if (lane >= off) s += y;
    }
    warp_sums[lane] = s;
  }
  __syncthreads();
  const uint32_t before = warp == 0 ? 0u : warp_sums[warp - 1];
  *total = warp_sums[n_warps - 1];
  __syncthreads();
  return before + x - v;
}

// Keep the n lowest set bits of w.
__device__ __forceinline__ uint32_t lowest_bits(uint32_t w, uint32_t n) {
  uint32_t out = 0;
  for (uint32_t i = 0; i < n && w; ++i) {
    const uint32_t b = w & (0u - w);
    out |= b;
    w ^= b;
  }
  return out;
}

// Bin of a histogram (nbins bins, read through hist(b)) that holds the
// need-th largest element counting from the top bin.  s_out[0] = bin,
// s_out[1] = elements in higher bins.
template <typename H>
__device__ __forceinline__ void find_bin(H hist, int nbins, uint32_t need, uint32_t* warp_sums, uint32_t* s_out) {
  const int nt = blockDim.x;
  const int per = nbins >= nt ? nbins / nt : 1;
  const int hi = nbins - (int)threadIdx.x * per;
  uint32_t local = 0u;
  if (hi > 0)
    for (int b = hi - 1; b >= hi - per; --b) local += hist(b);
  uint32_t total;
  const uint32_t above = block_exclusive_scan(local, warp_sums, &total);
  if (hi > 0 && above < need && above + local >= need) {
    uint32_t c = above;
    for (int b = hi - 1; b >= hi - per; --b) {
      const uint32_t h = hist(b);
      if (c + h >= need) {
        s_out[0] = (uint32_t)b;
        s_out[1] = c;
        break;
      }
      c += h;
    }
  }
  __syncthreads();
}

// Warp-aggregated shared-memory histogram increment (one atomic per
// distinct bin in the warp); all 32 lanes must call it.
__device__ __forceinline__ void hist_add(uint32_t* hist, bool act, uint32_t bin, int lane) {
  const uint32_t peers = __match_any_sync(0xffffffffu, act ? bin : 0xffffffffu);
  if (act && (__ffs(peers) - 1) == lane) atomicAdd(&hist[bin], (uint32_t)__popc(peers));
}

constexpr int kSubCap = 256;        // candidates sharing the k-th key's top 24 bits, resolved by rank

struct SelSmem {
  // offsets in 32-bit words
  int own, merged, keys, selw, eqw, ck, ci, h2, subk, subi, total;
  __host__ __device__ SelSmem(int chunk, int nw) {
    own = 0;
    merged = own + kBins;
    keys = merged + kBins;
    selw = keys + chunk;
    eqw = selw + nw;
    ck = eqw + nw;
    ci = ck + kCandCap;
    h2 = ci + kCandCap;      // second-level histogram (key bits 19..8) of the candidates, in CTA 0
    subk = h2 + kBins;
    subi = subk + kSubCap;
    total = subi + kSubCap;
  }
};

template <int NSEQ>
__global__ void __launch_bounds__(kThreads) select_kernel(const SelectParams<NSEQ> p, int chunk, int nw_max,
                                                            int cache_keys) {
  extern __shared__ uint32_t sm[];
  __shared__ uint32_t warp_sums[32];
  __shared__ uint32_t s_res[2];
  __shared__ uint32_t s_cand, s_sub;
  cg::cluster_group cluster = cg::this_cluster();
  grid_dependency_sync();
  const int S = (int)cluster.num_blocks();
  const int c = (int)cluster.block_rank();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int r = p.row_base + blockIdx.y;
  int si = 0;
#pragma unroll
  for (int i = 1; i < NSEQ; ++i)
    if (i < p.n_seqs && r >= p.seq[i].row_begin) si = i;
  const RowSeq sq = p.seq[si];
  const int n = (int)visible_blocks(row_position(sq.n_tokens, sq.n_rows, r - sq.row_begin));
  const int k = p.top_k;
  int32_t* out = p.sel + (int64_t)r * k;
  // Uniform across the cluster: every CTA of the row takes the same branch.
  if (n <= k) {
    if (c == 0) {
      for (int i = tid; i < k; i += kThreads) out[i] = i < n ? i : -1;
      if (tid == 0) p.cnt[r] = n;
    }
    return;
  }
  const int nw = (n + 31) >> 5;
  const SelSmem L(cache_keys ? chunk : 0, nw_max);
  uint32_t* own = sm + L.own;
  uint32_t* merged = sm + L.merged;
  uint32_t* keys = sm + L.keys;
  const float* srow = p.scores + (int64_t)r * p.ld;
  const int i0 = c * chunk;
  const int i1 = min(n, i0 + chunk);

  if (c == 0) {
    for (int i = tid; i < nw; i += kThreads) sm[L.eqw + i] = 0u;
    for (int b = tid; b < kBins; b += kThreads) sm[L.h2 + b] = 0u;
    if (tid == 0) {
      s_cand = 0u;
      s_sub = 0u;
    }
  }
  if (tid == 0) {   // a histogram that cannot hold the k-th key leaves bin 0
    s_res[0] = 0u;
    s_res[1] = 0u;
  }
  const uint32_t* hrow = p.hist ? p.hist + (int64_t)r * kBins : nullptr;
  if (hrow) {
    // The scoring kernel left the row's histogram: every CTA reads it.
    cluster.sync();   // peers are running and CTA 0's candidate state is zeroed
    find_bin([&](int b) { return __ldcg(hrow + b); }, kBins, (uint32_t)k, warp_sums, s_res);
  } else {
    // 1. Histogram of this CTA's keys (kept in shared memory for step 3).
    for (int b = tid; b < kBins; b += kThreads) own[b] = 0u;
    __syncthreads();
    // Loads are issued 8 per thread at a time, then counted.
    for (int base = i0 + warp * 32; base < i0 + chunk; base += 8 * kThreads) {
      float v[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int i = base + j * kThreads + lane;
        v[j] = i < i1 ? __ldg(srow + i) : 0.f;
      }
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int i = base + j * kThreads + lane;
        if (i < i1) {
          const uint32_t key = order_key(v[j]);
          if (cache_keys) keys[i - i0] = key;
          atomicAdd(&own[key >> 20], 1u);
        }
      }
    }
    cluster.sync();

    // 2. Sum bin slice c over the cluster and broadcast it to every CTA.
    {
      const int per = kBins / S;
      for (int b = c * per + tid; b < (c + 1) * per; b += kThreads) {
        uint32_t h[kMaxCluster];
#pragma unroll
        for (int q = 0; q < kMaxCluster; ++q) h[q] = q < S ? *cluster.map_shared_rank(own + b, q) : 0u;
        uint32_t sum = 0u;
#pragma unroll
        for (int q = 0; q < kMaxCluster; ++q) sum += h[q];
#pragma unroll
        for (int q = 0; q < kMaxCluster; ++q)
          if (q < S) *cluster.map_shared_rank(merged + b, q) = sum;
      }
    }
    cluster.sync();
    find_bin([&](int b) { return merged[b]; }, kBins, (uint32_t)k, warp_sums, s_res);
  }
  const uint32_t B = s_res[0];
  uint32_t need = (uint32_t)k - s_res[1];
  const bool overflow = (hrow ? __ldcg(hrow + B) : merged[B]) > (uint32_t)kCandCap;
  const bool cached = cache_keys && !hrow;

  // 3. Bitmap words (bin above B) and candidates (bin B) into CTA 0.
  uint32_t* selw0 = cluster.map_shared_rank(sm + L.selw, 0);
  uint32_t* ck0 = cluster.map_shared_rank(sm + L.ck, 0);
  uint32_t* ci0 = cluster.map_shared_rank(sm + L.ci, 0);
  uint32_t* cand0 = cluster.map_shared_rank(&s_cand, 0);
  uint32_t* h20 = cluster.map_shared_rank(sm + L.h2, 0);
  if (i0 < i1) {
    const int w0 = i0 >> 5, w1 = (i1 + 31) >> 5;
    for (int word = w0 + warp; word < w1; word += kThreads / 32) {
      const int i = word * 32 + lane;
      const bool in = i < i1;
      const uint32_t key = in ? (cached ? keys[i - i0] : order_key(srow[i])) : 0u;
      const uint32_t bin = key >> 20;
      const uint32_t gt = __ballot_sync(0xffffffffu, in && bin > B);
      const uint32_t eq = __ballot_sync(0xffffffffu, in && bin == B);
      if (lane == 0) selw0[word] = gt;
      if (!overflow && eq) {
        uint32_t base = 0u;
        if (lane == 0) base = atomicAdd(cand0, (uint32_t)__popc(eq));
        base = __shfl_sync(0xffffffffu, base, 0);
        if (eq & (1u << lane)) {
          const uint32_t at = base + __popc(eq & ((1u << lane) - 1u));
          ck0[at] = key;
          ci0[at] = (uint32_t)i;
          atomicAdd(h20 + ((key >> 8) & (kBins - 1)), 1u);
        }
      }
    }
  }
  cluster.sync();
  if (c != 0) return;

  // 4. CTA 0 finishes the row.
  uint32_t* selw = sm + L.selw;
  uint32_t* eqw = sm + L.eqw;
  uint32_t* hist = own;                 // free again: reused as radix scratch
  uint32_t prefix = B << 20;
  uint32_t pmask = 0xfff00000u;
  bool ranked = false;   // candidates resolved by rank: no "equal key" bitmap to apply
  if (!overflow) {
    const int C = (int)s_cand;
    const uint32_t* ck = sm + L.ck;
    const uint32_t* ci = sm + L.ci;
    uint32_t* subk = sm + L.subk;
    uint32_t* subi = sm + L.subi;
    // Second level: the bin of key bits 19..8 holding the k-th key.
    find_bin([&](int b) { return sm[L.h2 + b]; }, kBins, need, warp_sums, s_res);
    const uint32_t need2 = need - s_res[1];
    const uint32_t p24 = (B << 12) | s_res[0];
    for (int i = tid; i < C; i += kThreads) {
      const uint32_t key = ck[i], id = ci[i], k24 = key >> 8;
      if (k24 > p24) {
        atomicOr(&selw[id >> 5], 1u << (id & 31));
      } else if (k24 == p24) {
        const uint32_t j = atomicAdd(&s_sub, 1u);
        if (j < (uint32_t)kSubCap) {
          subk[j] = key;
          subi[j] = id;
        }
      }
    }
    __syncthreads();
    const int n_sub = (int)s_sub;
    if (n_sub <= kSubCap) {
      // Keep the need2 best of the few candidates left, by (key desc, id asc).
      for (int j = tid; j < n_sub; j += kThreads) {
        const uint32_t kj = subk[j], ij = subi[j];
        uint32_t rank = 0u;
        for (int i = 0; i < n_sub; ++i) rank += (subk[i] > kj) || (subk[i] == kj && subi[i] < ij);
        if (rank < need2) atomicOr(&selw[ij >> 5], 1u << (ij & 31));
      }
      ranked = true;
    } else {
      // Too many near-ties: a last radix pass over key bits 7..0.
      need = need2;
      prefix = p24 << 8;
      pmask = 0xffffff00u;
      for (int b = tid; b < 256; b += kThreads) hist[b] = 0u;
      __syncthreads();
      for (int i = tid; i < C; i += kThreads)
        if ((ck[i] & pmask) == prefix) atomicAdd(&hist[ck[i] & 255u], 1u);
      __syncthreads();
      find_bin([&](int b) { return hist[b]; }, 256, need, warp_sums, s_res);
      need -= s_res[1];
      prefix |= s_res[0];
      __syncthreads();
      for (int i = tid; i < C; i += kThreads) {
        const uint32_t key = ck[i], id = ci[i];
        if ((key >> 8) == p24) {
          if (key > prefix) atomicOr(&selw[id >> 5], 1u << (id & 31));
          else if (key == prefix) atomicOr(&eqw[id >> 5], 1u << (id & 31));
        }
      }
    }
  } else {
#pragma unroll 1
    for (int pass = 0; pass < 2; ++pass) {
      const int shift = pass == 0 ? 8 : 0;
      const int nbins = pass == 0 ? 4096 : 256;
      for (int b = tid; b < nbins; b += kThreads) hist[b] = 0u;
      __syncthreads();
      for (int base = warp * 32; base < n; base += kThreads) {
        const int i = base + lane;
        bool act = false;
        uint32_t bin = 0u;
        if (i < n) {
          const uint32_t key = order_key(srow[i]);
          act = (key & pmask) == prefix;
          bin = (key >> shift) & (uint32_t)(nbins - 1);
        }
        hist_add(hist, act, bin, lane);
      }
      __syncthreads();
      find_bin([&](int b) { return hist[b]; }, nbins, need, warp_sums, s_res);
      need -= s_res[1];
      prefix |= s_res[0] << shift;
      pmask |= (uint32_t)(nbins - 1) << shift;
      __syncthreads();
    }
    for (int word = warp; word < nw; word += kThreads / 32) {
      const int i = word * 32 + lane;
      const uint32_t key = i < n ? order_key(srow[i]) : 0u;
      const uint32_t gt = __ballot_sync(0xffffffffu, i < n && key > prefix);
      const uint32_t eq = __ballot_sync(0xffffffffu, i < n && key == prefix);
      if (lane == 0) {
        selw[word] = gt;
        eqw[word] = eq;
      }
    }
  }
  __syncthreads();
  // Keep the `need` lowest ids among keys equal to the k-th key (unless the
  // candidates were ranked), then write every chosen id in ascending order.
  const int wp = (nw + kThreads - 1) / kThreads;
  const int a0 = tid * wp, a1 = min(nw, a0 + wp);
  uint32_t local = 0u, total;
  if (!ranked) {
    for (int i = a0; i < a1; ++i) local += __popc(eqw[i]);
    uint32_t cpos = block_exclusive_scan(local, warp_sums, &total);
    local = 0u;
    for (int i = a0; i < a1; ++i) {
      uint32_t e = eqw[i];
      const uint32_t pc = __popc(e);
      if (cpos >= need) e = 0u;
      else if (cpos + pc > need) e = lowest_bits(e, need - cpos);
      cpos += pc;
      e |= selw[i];
      selw[i] = e;
      local += __popc(e);
    }
  } else {
    for (int i = a0; i < a1; ++i) local += __popc(selw[i]);
  }
  uint32_t at = block_exclusive_scan(local, warp_sums, &total);
  for (int i = a0; i < a1; ++i) {
    uint32_t e = selw[i];
    while (e) {
      const int b = __ffs(e) - 1;
      e &= e - 1u;
      if (at < (uint32_t)k) out[at] = i * 32 + b;
      ++at;
    }
  }
  if (tid == 0) p.cnt[r] = k;
  // Every CTA of the row read the histogram before the last cluster barrier:
  // return it to zero for the next call.
  if (hrow)
    for (int b = tid; b < kBins; b += kThreads) p.hist[(int64_t)r * kBins + b] = 0u;
}

}  // namespace

// Cluster size and chunk for rows of up to max_nb blocks: chunks of at most
// 2,048 keys when the cluster allows it, fewer CTAs per row when there are
// many rows.
void select_plan(int64_t rows, int64_t max_nb, int* cluster, int* chunk) {
  int s = 1;
  while (s < kMaxCluster && (max_nb + s - 1) / s > 2048) s <<= 1;
  const int64_t cap = 8 * (int64_t)device_sm_count();
  while (s > 1 && rows * s > cap) s >>= 1;
  int64_t ch = (max_nb + s - 1) / s;
  ch = (ch + 31) / 32 * 32;
  if (ch < 32) ch = 32;
  *cluster = s;
  *chunk = (int)ch;
}

constexpr int kKeyCacheMax = 16384;   // keys a CTA keeps in shared memory

size_t select_smem_bytes(int chunk, int nw_max) {
  return sizeof(uint32_t) * (size_t)SelSmem(chunk <= kKeyCacheMax ? chunk : 0, nw_max).total;
}

template <int NSEQ>
cudaError_t launch_select(const SelectParams<NSEQ>& p, int n_rows, int64_t max_nb, cudaStream_t st) {
  if (n_rows == 0) return cudaSuccess;
  int S = 1, chunk = 32;
  select_plan(n_rows, max_nb, &S, &chunk);
  const int nw_max = (int)((max_nb + 31) / 32);
  size_t smem = select_smem_bytes(chunk, nw_max);
  cudaError_t e = allow_dynamic_smem((const void*)select_kernel<NSEQ>, smem);
  if (e != cudaSuccess) return e;
  if (S > 8) {
    e = allow_cluster16((const void*)select_kernel<NSEQ>, kThreads, smem);
    if (e == cudaErrorNotSupported) {   // no 16-CTA cluster fits: use 8
      S = 8;
      chunk = (int)(((max_nb + 7) / 8 + 31) / 32 * 32);
    } else if (e != cudaSuccess) {
      return e;
    }
  }
  smem = select_smem_bytes(chunk, nw_max);
  if ((e = allow_dynamic_smem((const void*)select_kernel<NSEQ>, smem)) != cudaSuccess) return e;
  const int cache_keys = chunk <= kKeyCacheMax ? 1 : 0;
  return launch_kernel(select_kernel<NSEQ>, dim3((unsigned)S, (unsigned)n_rows), dim3(kThreads), smem, st,
                       (unsigned)S, p, chunk, nw_max, cache_keys);
}

template cudaError_t launch_select<1>(const SelectParams<1>&, int, int64_t, cudaStream_t);
template cudaError_t launch_select<kLaunchSeqs>(const SelectParams<kLaunchSeqs>&, int, int64_t, cudaStream_t);

}  // namespace qsa
