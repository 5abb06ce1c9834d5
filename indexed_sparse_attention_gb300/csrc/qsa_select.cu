// Step 3 of the QSA layer step: per query row, keep the top-k complete
// blocks by score, lower block id winning ties (hipfire, "QSA sparse
// attention and the VMM KV backend", section 02: the top-scoring blocks
// within a 2,048-token budget of 512 blocks; section 03: a radix select from
// the scores).
//
// One CTA of 1024 threads per row.  Scores map to order-preserving uint32
// keys (-0.0 folded onto +0.0).  Three radix passes (12 + 12 + 8 bits) find
// the exact key T of the k-th best block and how many blocks equal to T are
// still needed; a ballot pass then builds "> T" and "== T" bitmaps of the
// row, the lowest-id "== T" bits are kept, and a prefix popcount over the
// combined bitmap writes the kept ids in ascending order.
#include "qsa_internal.cuh"

namespace qsa {

namespace {

constexpr int kSelThreads = 1024;
constexpr int kHistBins = 4096;

__device__ __forceinline__ uint32_t order_key(float f) {
  uint32_t u = __float_as_uint(f);
  if (u == 0x80000000u) u = 0u;  // -0.0 ties with +0.0
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

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

template <int NSEQ>
__global__ void __launch_bounds__(kSelThreads) select_kernel(const SelectParams<NSEQ> p) {
  extern __shared__ uint32_t sm[];
  __shared__ uint32_t warp_sums[32];
  __shared__ uint32_t s_bin, s_above;
  uint32_t* hist = sm;
  const int r = p.row_base + blockIdx.x;
  int si = 0;
#pragma unroll
  for (int i = 1; i < NSEQ; ++i)
    if (i < p.n_seqs && r >= p.seq[i].row_begin) si = i;
  const RowSeq sq = p.seq[si];
  const int64_t pos = row_position(sq.n_tokens, sq.n_rows, r - sq.row_begin);
  const int64_t nb = visible_blocks(pos);
  const int k = p.top_k;
  int32_t* out = p.sel + (int64_t)r * k;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (nb <= k) {
    for (int i = tid; i < k; i += kSelThreads) out[i] = i < nb ? i : -1;
    if (tid == 0) p.cnt[r] = (int32_t)nb;
    return;
  }
  const float* srow = p.scores + (int64_t)r * p.ld;
  const int n = (int)nb;
  const int nw = (n + 31) >> 5;
  uint32_t* gtw = hist + kHistBins;
  uint32_t* eqw = gtw + nw;

  uint32_t prefix = 0u, pmask = 0u, need = (uint32_t)k;
#pragma unroll 1
  for (int pass = 0; pass < 3; ++pass) {
    const int shift = pass == 0 ? 20 : (pass == 1 ? 8 : 0);
    const int bits = pass == 2 ? 8 : 12;
    const uint32_t nbins = 1u << bits, bmask = nbins - 1u;
    for (int i = tid; i < (int)nbins; i += kSelThreads) hist[i] = 0u;
    __syncthreads();
    for (int base = warp * 32; base < n; base += kSelThreads) {
      const int i = base + lane;
      bool act = false;
      uint32_t bin = 0u;
      if (i < n) {
        const uint32_t key = order_key(srow[i]);
        act = (key & pmask) == prefix;
        bin = (key >> shift) & bmask;
      }
      // Warp-aggregated increments: one shared atomic per distinct bin.
      const uint32_t peers = __match_any_sync(0xffffffffu, act ? bin : 0xffffffffu);
      if (act && (__ffs(peers) - 1) == lane) atomicAdd(&hist[bin], (uint32_t)__popc(peers));
    }
    __syncthreads();
    // Thread i owns a run of bins taken from the top: bins [hi - per, hi).
    const int per = (int)(nbins >= (uint32_t)kSelThreads ? nbins / kSelThreads : 1u);
    const int hi = (int)nbins - tid * per;
    uint32_t local = 0u;
    if (hi > 0)
      for (int b = hi - 1; b >= hi - per; --b) local += hist[b];
    uint32_t total;
    const uint32_t above = block_exclusive_scan(local, warp_sums, &total);
    if (hi > 0 && above < need && above + local >= need) {
      uint32_t c = above;
      for (int b = hi - 1; b >= hi - per; --b) {
        if (c + hist[b] >= need) {
          s_bin = (uint32_t)b;
          s_above = c;
          break;
        }
        c += hist[b];
      }
    }
    __syncthreads();
    need -= s_above;
    prefix |= s_bin << shift;
    pmask |= bmask << shift;
    __syncthreads();
  }
  const uint32_t T = prefix;  // key of the k-th best block; `need` blocks equal to T are kept

  for (int word = warp; word < nw; word += kSelThreads / 32) {
    const int i = word * 32 + lane;
    const uint32_t key = i < n ? order_key(srow[i]) : 0u;
    const uint32_t gt = __ballot_sync(0xffffffffu, i < n && key > T);
    const uint32_t eq = __ballot_sync(0xffffffffu, i < n && key == T);
    if (lane == 0) {
      gtw[word] = gt;
      eqw[word] = eq;
    }
  }
  __syncthreads();
  const int wp = (nw + kSelThreads - 1) / kSelThreads;
  const int w0 = tid * wp, w1 = min(nw, w0 + wp);
  uint32_t local = 0u, total;
  for (int w = w0; w < w1; ++w) local += __popc(eqw[w]);
  uint32_t c = block_exclusive_scan(local, warp_sums, &total);
  local = 0u;
  for (int w = w0; w < w1; ++w) {
    uint32_t e = eqw[w];
    const uint32_t pc = __popc(e);
    if (c >= need) e = 0u;
    else if (c + pc > need) e = lowest_bits(e, need - c);
    c += pc;
    e |= gtw[w];
    eqw[w] = e;
    local += __popc(e);
  }
  uint32_t at = block_exclusive_scan(local, warp_sums, &total);
  for (int w = w0; w < w1; ++w) {
    uint32_t e = eqw[w];
    while (e) {
      const int b = __ffs(e) - 1;
      e &= e - 1u;
      if (at < (uint32_t)k) out[at] = w * 32 + b;
      ++at;
    }
  }
  if (tid == 0) p.cnt[r] = k;
}

}  // namespace

size_t select_smem_bytes(int64_t max_nb) {
  const int64_t nw = (max_nb + 31) / 32;
  return sizeof(uint32_t) * (size_t)(kHistBins + 2 * nw);
}

template <int NSEQ>
cudaError_t launch_select(const SelectParams<NSEQ>& p, int n_rows, int64_t max_nb, cudaStream_t st) {
  if (n_rows == 0) return cudaSuccess;
  const size_t smem = select_smem_bytes(max_nb);
  cudaError_t e = allow_dynamic_smem((const void*)select_kernel<NSEQ>, smem);
  if (e != cudaSuccess) return e;
  select_kernel<NSEQ><<<n_rows, kSelThreads, smem, st>>>(p);
  return cudaGetLastError();
}

template cudaError_t launch_select<1>(const SelectParams<1>&, int, int64_t, cudaStream_t);
template cudaError_t launch_select<kLaunchSeqs>(const SelectParams<kLaunchSeqs>&, int, int64_t, cudaStream_t);

}  // namespace qsa
