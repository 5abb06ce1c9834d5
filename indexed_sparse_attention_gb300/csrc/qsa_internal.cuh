// Internal declarations shared by the CUDA translation units of libqsa.so.
// Kernel parameters are passed by value (so a call can be captured in a CUDA
// graph); sequence and segment tables are copied into them on the host.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "qsa.h"

namespace qsa {

// Sequences one launch carries; larger calls are issued in chunks.
constexpr int kLaunchSeqs = 8;
// Query rows of one scoring row-group (4 index heads each: 32 MMA columns).
constexpr int kRowGroup = 8;
// Blocks per scoring tile (the MMA M dimension).
constexpr int kScoreTile = 16;

// ---------------------------------------------------------------- scoring
struct ScoreSeq {
  const float* pooled;
  int64_t pooled_stride;
  int64_t n_tokens;
  int64_t work_begin;    // first flattened (tile, row-group) item of this sequence
  int32_t row_begin;     // global index of the sequence's first row
  int32_t n_rows;
  int32_t n_tiles;       // ceil(floor(L/4) / kScoreTile)
  int32_t n_groups;      // ceil(n_rows / kRowGroup)
  // Optional step 1 inside the scoring launch: blocks [pool_b0, pool_b1) are
  // pooled from their four index keys (idx_keys, idx_stride elements between
  // tokens, idx_dtype) and written to pooled before they are scored.
  const void* idx_keys;
  int64_t idx_stride;
  int32_t idx_dtype;
  int64_t pool_b0, pool_b1;
  // With an append in the same launch: the index keys of tokens >= first_new
  // are read from idx_new ([n_new, 128] of idx_dtype) -- the launch itself
  // writes them into idx_keys, and no thread reads what another writes.
  const void* idx_new;
  int64_t first_new;
};

template <int NSEQ>
struct ScoreParams {
  ScoreSeq seq[NSEQ];
  int32_t n_seqs;
  int64_t n_work;        // total (tile, row-group) items
  const void* q_idx;     // [rows, 4, 128]
  float* scores;
  int64_t ld;
  float* gmax;           // optional [rows, gld]: max score of each group of QSA_SCORE_GROUP blocks
  int64_t gld;
};

static_assert(kScoreTile == QSA_SCORE_GROUP, "a scoring tile is one group of the group maxima");

__device__ __forceinline__ uint32_t order_key(float f) {
  uint32_t u = __float_as_uint(f);
  if (u == 0x80000000u) u = 0u;  // -0.0 ties with +0.0
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// ---------------------------------------------------------------- KV segments
struct Segment {
  const void* k;
  const void* v;
  int64_t first;
  int64_t n;
  int64_t head_stride;
  int64_t tok_stride;
  const uint8_t* kv_scale;     // quantized state: scale records (4 bytes fp8, D/8 bytes q8)
  int64_t s_head_stride;       // records
  int64_t s_tok_stride;
};

// ---------------------------------------------------------------- selection
struct RowSeq {
  int64_t n_tokens;
  int32_t row_begin;
  int32_t n_rows;
};

template <int NSEQ>
struct SelectParams {
  RowSeq seq[NSEQ];
  int32_t n_seqs;
  int32_t row_base;      // global index of this launch's first row
  const float* scores;
  int64_t ld;
  const float* gmax;     // optional group maxima [rows, gld] (from the scoring kernel)
  int64_t gld;
  int32_t top_k;
  int32_t* sel;
  int32_t* cnt;
};

// ---------------------------------------------------------------- attention
struct AttnSeq {
  int64_t n_tokens;
  int32_t row_begin;
  int32_t n_rows;
  int32_t seg_begin;
  int32_t n_segs;
};

template <int NSEQ>
struct AttnParams {
  AttnSeq seq[NSEQ];
  Segment seg[NSEQ * QSA_MAX_SEGMENTS];
  int32_t n_seqs;
  int32_t row_base;        // global index of this launch's first row
  const void* q;           // [rows, Hq, D]
  const int32_t* sel;
  const int32_t* cnt;
  int32_t sel_ld;
  int32_t n_q_heads;
  int32_t group;           // query heads per KV head
  int32_t head_dim;
  float scale;             // logit scale
  int32_t n_splits;        // splits per (row, KV group): split s takes tiles [s T / n, (s + 1) T / n)
                           // of the T 32-token tiles of a row's longest possible list
  int32_t total_rows;      // rows of the whole call (partial buffer stride)
  void* out;               // [rows, Hq, D] (single split)
  float* lse;              // [rows, Hq] or null (single split)
  float* part_o;           // [n_splits, rows * Hq, D] normalised partials (several splits)
  float* part_lse;         // [n_splits, rows * Hq]
  int32_t out_dtype;
};

// ---------------------------------------------------------------- appending tokens
struct AppendSeg {
  void* k;
  void* v;
  int64_t first, n, head_stride, tok_stride;   // elements
  void* kv_scale;                              // quantized state: scale records
  int64_t s_head_stride, s_tok_stride;         // records
};

struct AppendParams {
  AppendSeg seg[QSA_MAX_SEGMENTS];
  int32_t n_segs;
  int32_t n_kv_heads;
  int32_t head_dim;
  int32_t kvq;               // 1: fp8 state, 2: q8 state (k_new / v_new are bf16 and get quantized)
  int64_t n_tokens;          // L after the append
  int64_t n_new;             // tokens L - n_new .. L - 1 are appended
  const void* k_new;         // [Hkv, n_new, D]
  const void* v_new;
  int64_t row_bytes;         // D x kv element size
  int64_t row_chunks;        // row_bytes / 16
  int32_t kv_es;
  const void* idx_new;       // [n_new, 128]
  void* idx_keys;            // [>= L, idx_stride]
  int64_t idx_stride;
  int32_t idx_dtype;
  int32_t idx_es;
  int64_t idx_chunks;        // 128 x idx_es / 16
  float* pooled;
  int64_t pooled_stride;
  int64_t first_block;       // blocks first_block .. first_block + pool_items / 32 - 1 are pooled
  int64_t kv_items, idx_items, pool_items;
};

cudaError_t launch_append(const AppendParams& p, cudaStream_t st);

// Copy item i of an append with K/V state that is not quantized: items
// [0, kv_items) are 16-byte pieces of the new tokens' K and V rows
// (K or V, KV head, new token, piece), written into the segment that covers
// the token; items [kv_items, kv_items + idx_items) are 16-byte pieces of
// their index keys, written into the index-key cache.  Sets the piece's
// source and destination (dst null: no segment covers the token, or no item).
__device__ __forceinline__ void append_item(const AppendParams& p, int64_t i, const uint4*& src, uint4*& dst) {
  const int64_t first_new = p.n_tokens - p.n_new;
  dst = nullptr;
  if (i < p.kv_items) {
    const int64_t row = i / p.row_chunks, c = i % p.row_chunks;
    const int which = (int)(row / ((int64_t)p.n_kv_heads * p.n_new));   // 0: K, 1: V
    const int64_t hr = row % ((int64_t)p.n_kv_heads * p.n_new);
    const int h = (int)(hr / p.n_new);
    const int64_t j = hr % p.n_new;
    const int64_t t = first_new + j;
    src = reinterpret_cast<const uint4*>(static_cast<const char*>(which ? p.v_new : p.k_new) +
                                         ((int64_t)h * p.n_new + j) * p.row_bytes + c * 16);
    for (int s = 0; s < p.n_segs; ++s) {
      const AppendSeg& sg = p.seg[s];
      if (t >= sg.first && t < sg.first + sg.n) {
        dst = reinterpret_cast<uint4*>(static_cast<char*>(which ? sg.v : sg.k) +
                                       ((int64_t)h * sg.head_stride + (t - sg.first) * sg.tok_stride) * p.kv_es +
                                       c * 16);
        break;
      }
    }
    return;
  }
  const int64_t i2 = i - p.kv_items;
  if (i2 < p.idx_items) {
    const int64_t j = i2 / p.idx_chunks, c = i2 % p.idx_chunks;
    src = reinterpret_cast<const uint4*>(static_cast<const char*>(p.idx_new) + j * QSA_INDEX_DIM * p.idx_es + c * 16);
    dst = reinterpret_cast<uint4*>(static_cast<char*>(p.idx_keys) + (first_new + j) * p.idx_stride * p.idx_es +
                                   c * 16);
  }
}
__device__ __forceinline__ void append_copy(const AppendParams& p, int64_t i) {
  const uint4* src;
  uint4* dst;
  append_item(p, i, src, dst);
  if (dst) *dst = *src;
}

// ---------------------------------------------------------------- demand-mapped arena (qsa_arena.cu)
qsa_status arena_create(int32_t device, uint64_t reserve_bytes, qsa_arena** out, const char** why);
qsa_status arena_ensure(qsa_arena* a, uint64_t bytes, const char** why);
qsa_status arena_destroy(qsa_arena* a, const char** why);
void* arena_base(const qsa_arena* a);
uint64_t arena_mapped(const qsa_arena* a);
uint64_t arena_reserved(const qsa_arena* a);
uint64_t arena_granularity(const qsa_arena* a);

// ---------------------------------------------------------------- launchers
cudaError_t launch_pool(const void* idx, qsa_dtype dt, int64_t tok_stride, int64_t first_block,
                        int64_t n_blocks, float* pooled, int64_t pstride, cudaStream_t st);

// ap (optional): an append (K/V state not quantized, pool_items 0) done by
// the scoring launch itself where the kernel takes it (the few-row kernels),
// else by an append launch first.
template <int NSEQ>
cudaError_t launch_score(const ScoreParams<NSEQ>& p, qsa_dtype q_dtype, int max_rows_per_group,
                         cudaStream_t st, const AppendParams* ap = nullptr);

// Wide scoring on the tensor cores (one sequence; see qsa_score_tc.cu).
size_t score_tc_workspace_bytes(int64_t n_blocks);
// Scores blocks [block_lo, block_lo + n_blocks) into columns 0 .. n_blocks - 1.
cudaError_t launch_score_tc(const void* q_idx, int32_t row_begin, int32_t n_rows, int64_t n_tokens,
                            const float* pooled, int64_t pooled_stride, int64_t block_lo, int64_t n_blocks,
                            float* scores, int64_t ld, float* gmax, int64_t gld, void* workspace, cudaStream_t st);

template <int NSEQ>
cudaError_t launch_select(const SelectParams<NSEQ>& p, int n_rows, int64_t max_nb, cudaStream_t st);
size_t select_smem_bytes(int64_t max_nb);

// Selection over key-axis chunks: merge one chunk's scores into each row's
// running top-k (see qsa_select.cu).
struct MergeSelectParams {
  int64_t n_tokens;             // the sequence
  int32_t n_rows;
  int32_t row_begin;            // global index of its first row (sel, cnt)
  const float* chunk;           // [n_rows, ld_chunk] scores of blocks block_lo .. block_lo + n_blocks - 1
  int64_t ld_chunk;
  int64_t block_lo;
  int32_t n_blocks;
  int32_t top_k;
  const uint32_t* run_key_in;   // [n_rows, top_k] order keys of the running top-k (ascending ids)
  const int32_t* run_id_in;     // [n_rows, top_k]
  const int32_t* run_cnt_in;    // [n_rows]
  uint32_t* run_key_out;
  int32_t* run_id_out;
  int32_t* run_cnt_out;
  int32_t first;                // no running list yet
  int32_t last;                 // write sel and cnt instead of the running list
  int32_t* sel;
  int32_t* cnt;
};
cudaError_t launch_merge_select(const MergeSelectParams& p, cudaStream_t st);
// Largest top_k + chunk width the merge holds in shared memory.
int merge_select_max_union();

struct AttnPlan {
  int32_t n_splits;
  int32_t split_tokens;
  int32_t stages;
};

// Split plan for pairs = rows * Hkv (row, KV group) pairs whose selected lists
// are at most n_list entries; user_splits > 0 fixes the splits per pair.
AttnPlan attn_plan(qsa_dtype kv_dtype, int head_dim, int64_t pairs, int64_t n_list, int user_splits);
size_t attn_workspace_bytes(const AttnPlan& pl, int64_t rows, int n_q_heads, int head_dim);
void attn_workspace_layout(const AttnPlan& pl, int64_t rows, int n_q_heads, int head_dim, void* ws, float** part_o,
                           float** part_lse);

template <int NSEQ>
cudaError_t launch_attn(const AttnParams<NSEQ>& p, int n_rows, qsa_dtype kv_dtype, int stages, cudaStream_t st);

cudaError_t launch_merge(const float* o_parts, const float* lse_parts, int n_parts, int64_t n_rows,
                         int head_dim, void* out, int out_dtype, float* lse_out, cudaStream_t st);

// Attention on the tensor cores (see qsa_attn_tc.cu): bf16 K/V, head_dim 128
// or 256, at most 16 query heads per KV head, lists of at most 3,840 entries,
// one split, calls with at least kAttnTcMinRows query rows.
constexpr int kAttnTcMinRows = 512;
bool attn_tc_eligible(qsa_dtype kv_dtype, int head_dim, int group, int64_t max_list, int64_t rows);
template <int NSEQ>
cudaError_t launch_attn_tc(const AttnParams<NSEQ>& p, int n_rows, cudaStream_t st);

// Device-side waits that gave up after their time limit, per translation unit.
int score_wait_timeouts();
int score_tc_wait_timeouts();
int attn_tc_wait_timeouts();

// Reads a device-side event counter of the calling translation unit and
// clears it (-1 if it cannot be read).
template <typename T>
inline int take_counter(T& symbol) {
  int v = 0;
  if (cudaMemcpyFromSymbol(&v, symbol, sizeof(int)) != cudaSuccess) return -1;
  const int zero = 0;
  if (v != 0 && cudaMemcpyToSymbol(symbol, &zero, sizeof(int)) != cudaSuccess) return -1;
  return v;
}
// Counters behind qsa_check_device_status, each read and cleared.
int attn_bad_ids_take();        // selected ids outside [0, nb) (qsa_attn.cu)
int attn_tc_bad_ids_take();     // the same in the tensor-core attention
int select_nan_keys_take();     // NaN scores among selection candidates
int selftest_timeouts_take();   // expired waits of qsa_selftest_wait_timeout
cudaError_t launch_selftest_wait(int32_t limit_us, cudaStream_t st);

int device_sm_count();

// Raise a kernel's dynamic shared-memory limit (once per device and size).
cudaError_t allow_dynamic_smem(const void* kernel, size_t bytes);

// Blocks per scoring work item for the kernel that serves q_dtype.
int score_tile_blocks(qsa_dtype q_dtype);

// ---------------------------------------------------------------- launches
// Every kernel is launched with programmatic stream serialization: it may
// start while its predecessor on the stream finishes, and waits
// (griddepcontrol.wait) before it touches any memory the predecessor writes.
template <typename... KArgs, typename... Args>
cudaError_t launch_kernel(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                          unsigned cluster_x, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  int n = 0;
  attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[n].val.programmaticStreamSerializationAllowed = 1;
  ++n;
  if (cluster_x > 0) {
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = cluster_x;
    attr[n].val.clusterDim.y = 1;
    attr[n].val.clusterDim.z = 1;
    ++n;
  }
  cfg.attrs = attr;
  cfg.numAttrs = n;
  cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, args...);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

// ---------------------------------------------------------------- device helpers
// Wait until the grids this one depends on have completed and their writes
// are visible; then let this grid's dependents be scheduled.
__device__ __forceinline__ void grid_dependency_sync() {
  asm volatile("griddepcontrol.wait;\n" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
}
// The two halves, for kernels that do work between them.
__device__ __forceinline__ void grid_dependency_wait() { asm volatile("griddepcontrol.wait;\n" ::: "memory"); }
__device__ __forceinline__ void grid_dependency_release() {
  asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
}

// Asynchronous global -> shared copies (cp.async): a copy whose valid is
// false writes zeros and reads nothing; wait_group N waits until at most N
// committed groups are pending.
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ void cp_async16(void* dst, const void* src, bool valid) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(smem_u32(dst)), "l"(src),
               "r"(valid ? 16 : 0));
}
// 4-byte copy; src and dst 4-byte aligned.
__device__ __forceinline__ void cp_async4(void* dst, const void* src, bool valid) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;\n" ::"r"(smem_u32(dst)), "l"(src), "r"(valid ? 4 : 0));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N));
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;\n" ::: "memory"); }

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// Row r of a sequence at n_tokens L with n_rows M sits at L - M + j.
__device__ __forceinline__ int64_t row_position(int64_t L, int32_t n_rows, int32_t j) {
  return L - n_rows + j;
}
__device__ __forceinline__ int64_t visible_blocks(int64_t p) { return (p + 1) >> 2; }

}  // namespace qsa
