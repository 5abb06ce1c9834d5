// Host side of the C ABI declared in include/qsa.h: argument checks, the
// decomposition of a call into launches, and status reporting.  No entry
// point allocates device memory; scratch comes from the caller's workspace.
#include <math.h>
#include <stdarg.h>
#include <stdio.h>

#include <algorithm>
#include <mutex>
#include <string>
#include <vector>

#include <nvtx3/nvToolsExt.h>

#include "qsa_internal.cuh"

namespace {

thread_local std::string g_last_error;

// An NVTX range around each call that enqueues work (named after the entry
// point): a profiler attributes the call's launches to the QSA step they
// serve.  Without a profiler attached the push and pop are no-ops.
struct NvtxRange {
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
  NvtxRange(const NvtxRange&) = delete;
  NvtxRange& operator=(const NvtxRange&) = delete;
};

qsa_status fail(qsa_status s, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return s;
}

qsa_status ok() {
  g_last_error.clear();
  return QSA_OK;
}

qsa_status cuda_fail(cudaError_t e, const char* where) {
  return fail(QSA_ERR_CUDA, "%s: %s", where, cudaGetErrorString(e));
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool quantized(int d) { return d == QSA_FP8_E4M3 || d == QSA_Q8_0; }
size_t dtype_size(qsa_dtype d) { return d == QSA_F32 ? 4 : quantized(d) ? 1 : 2; }

bool valid_dtype(int d) { return d == QSA_F32 || d == QSA_BF16; }
// K/V state types: the value types plus the fp8 state.
bool valid_kv_dtype(int d) { return valid_dtype(d) || quantized(d); }

// Complete blocks the last (furthest) row of a sequence sees: floor(L / 4).
int64_t max_visible_blocks(const qsa_seq& s) { return s.n_tokens / 4; }
int64_t n_groups(int64_t blocks) { return (blocks + QSA_SCORE_GROUP - 1) / QSA_SCORE_GROUP; }

qsa_status check_rows(const qsa_seq* seqs, int32_t n_seqs, const char* fn, int64_t* total_rows) {
  if (!seqs || n_seqs < 1) return fail(QSA_ERR_INVALID_ARG, "%s: need at least one sequence", fn);
  int64_t rows = 0;
  for (int i = 0; i < n_seqs; ++i) {
    const qsa_seq& s = seqs[i];
    if (s.n_tokens < 1 || s.n_rows < 1 || s.n_rows > s.n_tokens)
      return fail(QSA_ERR_INVALID_ARG, "%s: sequence %d has n_tokens=%lld, n_rows=%d (need 1 <= n_rows <= n_tokens)",
                  fn, i, (long long)s.n_tokens, s.n_rows);
    if (max_visible_blocks(s) > QSA_MAX_BLOCKS)
      return fail(QSA_ERR_UNSUPPORTED, "%s: sequence %d has %lld complete blocks (max %d)", fn, i,
                  (long long)max_visible_blocks(s), QSA_MAX_BLOCKS);
    rows += s.n_rows;
  }
  if (rows > (int64_t)INT32_MAX / 64) return fail(QSA_ERR_UNSUPPORTED, "%s: too many rows", fn);
  *total_rows = rows;
  return QSA_OK;
}

cudaStream_t as_stream(void* s) { return static_cast<cudaStream_t>(s); }

std::mutex g_dev_mu;
int g_sm_count[64];

}  // namespace

namespace qsa {
cudaError_t allow_dynamic_smem(const void* kernel, size_t bytes) {
  if (bytes <= 48 * 1024) return cudaSuccess;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  struct Entry {
    int dev;
    const void* kernel;
    size_t bytes;
  };
  static std::vector<Entry> done;
  std::lock_guard<std::mutex> lk(g_dev_mu);
  for (const Entry& x : done)
    if (x.dev == dev && x.kernel == kernel && x.bytes >= bytes) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
  if (e == cudaSuccess) done.push_back(Entry{dev, kernel, bytes});
  return e;
}

int device_sm_count() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
  std::lock_guard<std::mutex> lk(g_dev_mu);
  if (g_sm_count[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
    g_sm_count[dev] = n;
  }
  return g_sm_count[dev];
}
}  // namespace qsa

using namespace qsa;

#define QSA_API extern "C" __attribute__((visibility("default")))

QSA_API const char* qsa_status_string(qsa_status s) {
  switch (s) {
    case QSA_OK: return "QSA_OK";
    case QSA_ERR_INVALID_ARG: return "QSA_ERR_INVALID_ARG";
    case QSA_ERR_UNSUPPORTED: return "QSA_ERR_UNSUPPORTED";
    case QSA_ERR_MISALIGNED: return "QSA_ERR_MISALIGNED";
    case QSA_ERR_WORKSPACE: return "QSA_ERR_WORKSPACE";
    case QSA_ERR_CUDA: return "QSA_ERR_CUDA";
    case QSA_ERR_DEVICE_CHECK: return "QSA_ERR_DEVICE_CHECK";
    case QSA_ERR_TIMEOUT: return "QSA_ERR_TIMEOUT";
  }
  return "QSA_ERR_UNKNOWN";
}

QSA_API const char* qsa_last_error(void) { return g_last_error.c_str(); }

QSA_API int32_t qsa_version(void) { return QSA_VERSION; }

QSA_API int32_t qsa_wait_timeouts(void) {
  const int a = score_wait_timeouts(), b = score_tc_wait_timeouts(), c = attn_tc_wait_timeouts();
  if (a < 0 || b < 0 || c < 0) return -1;
  return a + b + c;
}

QSA_API qsa_status qsa_check_device_status(void* stream) {
  const char* fn = "qsa_check_device_status";
  cudaError_t e = cudaStreamSynchronize(as_stream(stream));
  if (e != cudaSuccess) return cuda_fail(e, fn);
  static std::mutex mu;
  static int seen_waits[64];   // per device: qsa_wait_timeouts() at the previous call
  int dev = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return cuda_fail(e, fn);
  if (dev < 0 || dev >= 64) return fail(QSA_ERR_UNSUPPORTED, "%s: device %d", fn, dev);
  std::lock_guard<std::mutex> lock(mu);
  const int w = qsa_wait_timeouts(), st = selftest_timeouts_take();
  const int bad_a = attn_bad_ids_take(), bad_t = attn_tc_bad_ids_take(), nan = select_nan_keys_take();
  if (w < 0 || st < 0 || bad_a < 0 || bad_t < 0 || nan < 0)
    return fail(QSA_ERR_CUDA, "%s: the device counters could not be read", fn);
  const int waits = (w - seen_waits[dev]) + st, bad = bad_a + bad_t;
  seen_waits[dev] = w;
  if (waits > 0)
    return fail(QSA_ERR_TIMEOUT, "%s: %d device wait(s) gave up; %d out-of-range selected ids, %d NaN scores", fn,
                waits, bad, nan);
  if (bad > 0 || nan > 0)
    return fail(QSA_ERR_DEVICE_CHECK, "%s: %d out-of-range selected ids (skipped), %d NaN scores among the selection's candidates",
                fn, bad, nan);
  return ok();
}

QSA_API qsa_status qsa_selftest_wait_timeout(int32_t limit_us, void* stream) {
  const char* fn = "qsa_selftest_wait_timeout";
  if (limit_us < 1 || limit_us > 2000000)
    return fail(QSA_ERR_INVALID_ARG, "%s: limit_us=%d outside 1..2,000,000", fn, limit_us);
  cudaError_t e = launch_selftest_wait(limit_us, as_stream(stream));
  if (e != cudaSuccess) return cuda_fail(e, fn);
  return ok();
}

// ------------------------------------------------------------------ step 1
QSA_API qsa_status qsa_pool_index_keys(const void* idx_keys, qsa_dtype idx_dtype, int64_t tok_stride, int64_t first_block,
                               int64_t n_blocks, float* pooled, int64_t pooled_stride, void* stream) {
  const NvtxRange nvtx_range("qsa_pool_index_keys");
  const char* fn = "qsa_pool_index_keys";
  if (!valid_dtype(idx_dtype)) return fail(QSA_ERR_UNSUPPORTED, "%s: idx_dtype %d", fn, (int)idx_dtype);
  if (first_block < 0 || n_blocks < 0) return fail(QSA_ERR_INVALID_ARG, "%s: negative block range", fn);
  if (tok_stride < QSA_INDEX_DIM || pooled_stride < QSA_INDEX_DIM)
    return fail(QSA_ERR_INVALID_ARG, "%s: strides must be >= %d", fn, QSA_INDEX_DIM);
  if (n_blocks == 0) return ok();
  if (!idx_keys || !pooled) return fail(QSA_ERR_INVALID_ARG, "%s: null pointer", fn);
  if (!aligned16(idx_keys) || !aligned16(pooled) || (tok_stride * (int64_t)dtype_size(idx_dtype)) % 16 != 0 ||
      pooled_stride % 4 != 0)
    return fail(QSA_ERR_MISALIGNED, "%s: pointers and strides must be 16-byte aligned", fn);
  cudaError_t e = launch_pool(idx_keys, idx_dtype, tok_stride, first_block, n_blocks, pooled, pooled_stride,
                              as_stream(stream));
  if (e != cudaSuccess) return cuda_fail(e, fn);
  return ok();
}

// ------------------------------------------------------------------ step 2
namespace {
// Index-key caches of the sequences of a pooling + scoring call.
struct IdxKeys {
  const void* const* keys;   // host array: one device pointer per sequence
  int64_t tok_stride;
  qsa_dtype dtype;
};
}  // namespace

template <int NSEQ>
static qsa_status score_chunk(const qsa_seq* seqs, int n, int32_t row_begin, const void* q_idx, qsa_dtype qd,
                              float* scores, int64_t ld, float* gmax, int64_t gld, const IdxKeys* ik,
                              cudaStream_t st, const AppendParams* ap = nullptr) {
  ScoreParams<NSEQ> p{};
  p.gmax = gmax;
  p.gld = gld;
  const int tile = score_tile_blocks(qd);
  int64_t work = 0;
  int max_rows = 1;
  for (int i = 0; i < n; ++i) {
    ScoreSeq& q = p.seq[i];
    q.pooled = seqs[i].pooled;
    q.pooled_stride = seqs[i].pooled_stride;
    q.n_tokens = seqs[i].n_tokens;
    q.row_begin = row_begin;
    q.n_rows = seqs[i].n_rows;
    q.n_tiles = (int32_t)((max_visible_blocks(seqs[i]) + tile - 1) / tile);
    q.n_groups = (q.n_rows + kRowGroup - 1) / kRowGroup;
    q.work_begin = work;
    if (ik) {   // step 1 for the blocks the rows complete, inside the launch where the kernel allows it
      q.idx_keys = ik->keys[i];
      q.idx_stride = ik->tok_stride;
      q.idx_dtype = ik->dtype;
      q.pool_b0 = (seqs[i].n_tokens - seqs[i].n_rows) / 4;
      q.pool_b1 = seqs[i].n_tokens / 4;
    }
    if (ap) {   // (one sequence) the launch appends its newest tokens too
      q.idx_new = ap->idx_new;
      q.first_new = ap->n_tokens - ap->n_new;
    }
    work += (int64_t)q.n_tiles * q.n_groups;
    max_rows = std::max(max_rows, std::min(kRowGroup, q.n_rows));
    row_begin += seqs[i].n_rows;
  }
  p.n_seqs = n;
  p.n_work = work;
  p.q_idx = q_idx;
  p.scores = scores;
  p.ld = ld;
  cudaError_t e = launch_score<NSEQ>(p, qd, max_rows, st, ap);
  if (e != cudaSuccess) return cuda_fail(e, "qsa_score_blocks");
  return QSA_OK;
}

namespace {
// Sequences that take the tensor-core path: bf16 index queries, more rows
// than the few-row path serves (kRowGroup).
bool wide_seq(const qsa_seq& q, qsa_dtype qd) { return qd == QSA_BF16 && q.n_rows > kRowGroup && q.n_tokens / 4 > 0; }
}  // namespace

QSA_API size_t qsa_score_workspace_size(const qsa_seq* seqs, int32_t n_seqs, qsa_dtype q_idx_dtype) {
  if (!seqs || n_seqs < 1) return 0;
  size_t need = 0;
  for (int i = 0; i < n_seqs; ++i)
    if (wide_seq(seqs[i], q_idx_dtype)) need = std::max(need, score_tc_workspace_bytes(max_visible_blocks(seqs[i])));
  return need;
}

// ap: (one few-row sequence) the append the scoring launch does too.
// check_only: validate the arguments and launch nothing.
static qsa_status score_blocks_impl(const char* fn, const qsa_seq* seqs, int32_t n_seqs, const IdxKeys* ik,
                                   const void* q_idx, qsa_dtype q_idx_dtype, float* scores, int64_t ld,
                                   float* group_max, int64_t group_ld, void* workspace, size_t workspace_bytes,
                                   void* stream, const AppendParams* ap = nullptr, bool check_only = false) {
  int64_t rows = 0;
  qsa_status s = check_rows(seqs, n_seqs, fn, &rows);
  if (s != QSA_OK) return s;
  if (ik) {
    if (!ik->keys) return fail(QSA_ERR_INVALID_ARG, "%s: null idx_keys array", fn);
    if (!valid_dtype(ik->dtype)) return fail(QSA_ERR_UNSUPPORTED, "%s: idx_dtype %d", fn, (int)ik->dtype);
    if (ik->tok_stride < QSA_INDEX_DIM) return fail(QSA_ERR_INVALID_ARG, "%s: idx_tok_stride < %d", fn, QSA_INDEX_DIM);
    if ((ik->tok_stride * (int64_t)dtype_size(ik->dtype)) % 16 != 0)
      return fail(QSA_ERR_MISALIGNED, "%s: idx_tok_stride not a multiple of 16 bytes", fn);
  }
  if (!valid_dtype(q_idx_dtype)) return fail(QSA_ERR_UNSUPPORTED, "%s: q_idx_dtype %d", fn, (int)q_idx_dtype);
  if (!q_idx || !scores) return fail(QSA_ERR_INVALID_ARG, "%s: null pointer", fn);
  if (!aligned16(q_idx) || !aligned16(scores)) return fail(QSA_ERR_MISALIGNED, "%s: q_idx/scores not aligned", fn);
  if (group_max && (!aligned16(group_max) || group_ld % 4 != 0))
    return fail(QSA_ERR_MISALIGNED, "%s: group_max or group_ld not 16-byte aligned", fn);
  for (int i = 0; i < n_seqs; ++i) {
    const qsa_seq& q = seqs[i];
    if (group_max && n_groups(max_visible_blocks(q)) > group_ld)
      return fail(QSA_ERR_INVALID_ARG, "%s: group_ld=%lld < %lld groups of sequence %d", fn, (long long)group_ld,
                  (long long)n_groups(max_visible_blocks(q)), i);
    if (max_visible_blocks(q) > ld)
      return fail(QSA_ERR_INVALID_ARG, "%s: ld=%lld < %lld visible blocks of sequence %d", fn, (long long)ld,
                  (long long)max_visible_blocks(q), i);
    if (max_visible_blocks(q) > 0) {
      if (!q.pooled) return fail(QSA_ERR_INVALID_ARG, "%s: sequence %d has no pooled keys", fn, i);
      if (q.pooled_stride < QSA_INDEX_DIM) return fail(QSA_ERR_INVALID_ARG, "%s: pooled_stride < 128", fn);
      if (!aligned16(q.pooled) || q.pooled_stride % 4 != 0)
        return fail(QSA_ERR_MISALIGNED, "%s: pooled keys of sequence %d not 16-byte aligned", fn, i);
    }
    if (ik && q.n_tokens / 4 > (q.n_tokens - q.n_rows) / 4) {
      if (!ik->keys[i]) return fail(QSA_ERR_INVALID_ARG, "%s: sequence %d has no index keys", fn, i);
      if (!aligned16(ik->keys[i]))
        return fail(QSA_ERR_MISALIGNED, "%s: index keys of sequence %d not 16-byte aligned", fn, i);
    }
  }
  if (check_only) return QSA_OK;
  cudaStream_t st = as_stream(stream);
  const size_t tc_need = qsa_score_workspace_size(seqs, n_seqs, q_idx_dtype);
  if (ap) return (s = score_chunk<1>(seqs, 1, 0, q_idx, q_idx_dtype, scores, ld, group_max, group_ld, ik, st, ap)) ==
                         QSA_OK ? ok() : s;
  if (tc_need > 0 && workspace && workspace_bytes >= tc_need) {
    if (!aligned16(workspace)) return fail(QSA_ERR_MISALIGNED, "%s: workspace not aligned", fn);
    // Wide sequences on the tensor cores, one after the other (they share the
    // workspace in stream order); the others on the few-row path.
    int32_t row_begin = 0;
    for (int i = 0; i < n_seqs && s == QSA_OK; ++i) {
      const qsa_seq& q = seqs[i];
      if (wide_seq(q, q_idx_dtype)) {
        const int64_t pb0 = (q.n_tokens - q.n_rows) / 4, pb1 = q.n_tokens / 4;
        if (ik && pb1 > pb0) {   // step 1 first: the tensor-core kernel reads pooled keys only
          cudaError_t e = launch_pool(ik->keys[i], ik->dtype, ik->tok_stride, pb0, pb1 - pb0,
                                      const_cast<float*>(q.pooled), q.pooled_stride, st);
          if (e != cudaSuccess) return cuda_fail(e, fn);
        }
        cudaError_t e = launch_score_tc(q_idx, row_begin, q.n_rows, q.n_tokens, q.pooled, q.pooled_stride, 0,
                                        q.n_tokens / 4, scores, ld, group_max, group_ld, workspace, st);
        if (e == cudaErrorNotSupported)
          s = score_chunk<1>(seqs + i, 1, row_begin, q_idx, q_idx_dtype, scores, ld, group_max, group_ld, nullptr, st);
        else if (e != cudaSuccess)
          s = cuda_fail(e, fn);
      } else {
        IdxKeys one{ik ? ik->keys + i : nullptr, ik ? ik->tok_stride : 0, ik ? ik->dtype : QSA_F32};
        s = score_chunk<1>(seqs + i, 1, row_begin, q_idx, q_idx_dtype, scores, ld, group_max, group_ld,
                           ik ? &one : nullptr, st);
      }
      row_begin += q.n_rows;
    }
  } else if (n_seqs == 1) {
    s = score_chunk<1>(seqs, 1, 0, q_idx, q_idx_dtype, scores, ld, group_max, group_ld, ik, st);
  } else {
    int32_t row_begin = 0;
    for (int c = 0; c < n_seqs && s == QSA_OK; c += kLaunchSeqs) {
      const int n = std::min(kLaunchSeqs, n_seqs - c);
      IdxKeys part{ik ? ik->keys + c : nullptr, ik ? ik->tok_stride : 0, ik ? ik->dtype : QSA_F32};
      s = score_chunk<kLaunchSeqs>(seqs + c, n, row_begin, q_idx, q_idx_dtype, scores, ld, group_max, group_ld,
                                   ik ? &part : nullptr, st);
      for (int i = 0; i < n; ++i) row_begin += seqs[c + i].n_rows;
    }
  }
  return s == QSA_OK ? ok() : s;
}

QSA_API qsa_status qsa_score_blocks(const qsa_seq* seqs, int32_t n_seqs, const void* q_idx, qsa_dtype q_idx_dtype,
                                    float* scores, int64_t ld, float* group_max, int64_t group_ld, void* workspace,
                                    size_t workspace_bytes, void* stream) {
  const NvtxRange nvtx_range("qsa_score_blocks");
  return score_blocks_impl("qsa_score_blocks", seqs, n_seqs, nullptr, q_idx, q_idx_dtype, scores, ld, group_max,
                           group_ld, workspace, workspace_bytes, stream);
}

QSA_API qsa_status qsa_pool_score_blocks(const qsa_seq* seqs, int32_t n_seqs, const void* const* idx_keys,
                                         int64_t idx_tok_stride, qsa_dtype idx_dtype, const void* q_idx,
                                         qsa_dtype q_idx_dtype, float* scores, int64_t ld, float* group_max,
                                         int64_t group_ld, void* workspace, size_t workspace_bytes, void* stream) {
  const NvtxRange nvtx_range("qsa_pool_score_blocks");
  const IdxKeys ik{idx_keys, idx_tok_stride, idx_dtype};
  return score_blocks_impl("qsa_pool_score_blocks", seqs, n_seqs, &ik, q_idx, q_idx_dtype, scores, ld, group_max,
                           group_ld, workspace, workspace_bytes, stream);
}

// ------------------------------------------------------------------ step 3
QSA_API size_t qsa_select_workspace_size(const qsa_seq* seqs, int32_t n_seqs, int32_t top_k) {
  (void)seqs;
  (void)n_seqs;
  (void)top_k;
  return 0;
}

template <int NSEQ>
static qsa_status select_chunk(const qsa_seq* seqs, int n, int32_t row_begin, const float* scores, int64_t ld,
                               const float* gmax, int64_t gld, int32_t top_k, int32_t* sel, int32_t* cnt,
                               cudaStream_t st) {
  SelectParams<NSEQ> p{};
  p.gmax = gmax;
  p.gld = gld;
  int rows = 0;
  int64_t max_nb = 0;
  p.row_base = row_begin;
  for (int i = 0; i < n; ++i) {
    p.seq[i].n_tokens = seqs[i].n_tokens;
    p.seq[i].row_begin = row_begin + rows;
    p.seq[i].n_rows = seqs[i].n_rows;
    rows += seqs[i].n_rows;
    max_nb = std::max(max_nb, max_visible_blocks(seqs[i]));
  }
  p.n_seqs = n;
  p.scores = scores;
  p.ld = ld;
  p.top_k = top_k;
  p.sel = sel;
  p.cnt = cnt;
  cudaError_t e = launch_select<NSEQ>(p, rows, max_nb, st);
  if (e != cudaSuccess) return cuda_fail(e, "qsa_select_topk");
  return QSA_OK;
}

QSA_API qsa_status qsa_select_topk(const qsa_seq* seqs, int32_t n_seqs, const float* scores, int64_t ld,
                                   const float* group_max, int64_t group_ld, int32_t top_k, int32_t* sel, int32_t* cnt,
                                   void* workspace, size_t workspace_bytes, void* stream) {
  const NvtxRange nvtx_range("qsa_select_topk");
  const char* fn = "qsa_select_topk";
  int64_t rows = 0;
  qsa_status s = check_rows(seqs, n_seqs, fn, &rows);
  if (s != QSA_OK) return s;
  if (top_k < 1 || top_k > QSA_MAX_TOP_K)
    return fail(QSA_ERR_UNSUPPORTED, "%s: top_k=%d outside 1..%d", fn, top_k, QSA_MAX_TOP_K);
  if (!scores || !sel || !cnt) return fail(QSA_ERR_INVALID_ARG, "%s: null pointer", fn);
  if (!aligned16(scores) || ld % 4 != 0) return fail(QSA_ERR_MISALIGNED, "%s: scores or ld not 16-byte aligned", fn);
  if (group_max && (!aligned16(group_max) || group_ld % 4 != 0))
    return fail(QSA_ERR_MISALIGNED, "%s: group_max or group_ld not 16-byte aligned", fn);
  for (int i = 0; i < n_seqs; ++i) {
    if (max_visible_blocks(seqs[i]) > ld)
      return fail(QSA_ERR_INVALID_ARG, "%s: ld smaller than the visible blocks of sequence %d", fn, i);
    if (group_max && n_groups(max_visible_blocks(seqs[i])) > group_ld)
      return fail(QSA_ERR_INVALID_ARG, "%s: group_ld smaller than the groups of sequence %d", fn, i);
  }
  (void)workspace;
  (void)workspace_bytes;
  cudaStream_t st = as_stream(stream);
  if (n_seqs == 1) {
    s = select_chunk<1>(seqs, 1, 0, scores, ld, group_max, group_ld, top_k, sel, cnt, st);
  } else {
    int32_t row_begin = 0;
    for (int c = 0; c < n_seqs && s == QSA_OK; c += kLaunchSeqs) {
      const int n = std::min(kLaunchSeqs, n_seqs - c);
      s = select_chunk<kLaunchSeqs>(seqs + c, n, row_begin, scores, ld, group_max, group_ld, top_k, sel, cnt, st);
      for (int i = 0; i < n; ++i) row_begin += seqs[c + i].n_rows;
    }
  }
  return s == QSA_OK ? ok() : s;
}

// ------------------------------------------------------------------ steps 2 + 3 fused
namespace {
// Row stride of the group maxima a fused call keeps in its workspace.
int64_t fused_group_ld(const qsa_seq* seqs, int32_t n_seqs) {
  int64_t g = 0;
  for (int i = 0; i < n_seqs; ++i) g = std::max(g, n_groups(max_visible_blocks(seqs[i])));
  return std::max<int64_t>(4, (g + 3) / 4 * 4);
}
}  // namespace

// Bytes of group maxima a fused call keeps at the start of its workspace
// (256-byte multiple); the key planes of the tensor-core path follow.
size_t fused_gmax_bytes(const qsa_seq* seqs, int32_t n_seqs) {
  int64_t rows = 0;
  for (int i = 0; i < n_seqs; ++i) rows += std::max(0, seqs[i].n_rows);
  return (sizeof(float) * (size_t)rows * (size_t)fused_group_ld(seqs, n_seqs) + 255) / 256 * 256;
}

QSA_API size_t qsa_score_select_workspace_size(const qsa_seq* seqs, int32_t n_seqs, int32_t top_k) {
  (void)top_k;
  if (!seqs || n_seqs < 1) return 0;
  // Group maxima, the selection's scratch, then the scoring's (bf16 queries
  // assumed: the tensor-core planes are counted whenever a sequence is wide).
  return fused_gmax_bytes(seqs, n_seqs) + qsa_score_workspace_size(seqs, n_seqs, QSA_BF16);
}

QSA_API qsa_status qsa_score_select_topk(const qsa_seq* seqs, int32_t n_seqs, const void* q_idx,
                                         qsa_dtype q_idx_dtype, float* scores, int64_t ld, int32_t top_k,
                                         int32_t* sel, int32_t* cnt, void* workspace, size_t workspace_bytes,
                                         void* stream) {
  const NvtxRange nvtx_range("qsa_score_select_topk");
  const char* fn = "qsa_score_select_topk";
  int64_t rows = 0;
  qsa_status s = check_rows(seqs, n_seqs, fn, &rows);
  if (s != QSA_OK) return s;
  const size_t need = qsa_score_select_workspace_size(seqs, n_seqs, top_k);
  if (!workspace || workspace_bytes < need)
    return fail(QSA_ERR_WORKSPACE, "%s: workspace of %zu bytes needed, %zu given", fn, need,
                workspace ? workspace_bytes : (size_t)0);
  if (!aligned16(workspace)) return fail(QSA_ERR_MISALIGNED, "%s: workspace not aligned", fn);
  // Check the selection's own arguments before the scoring launch.
  if (top_k < 1 || top_k > QSA_MAX_TOP_K)
    return fail(QSA_ERR_UNSUPPORTED, "%s: top_k=%d outside 1..%d", fn, top_k, QSA_MAX_TOP_K);
  if (!sel || !cnt) return fail(QSA_ERR_INVALID_ARG, "%s: null pointer", fn);
  float* gmax = static_cast<float*>(workspace);
  const int64_t gld = fused_group_ld(seqs, n_seqs);
  const size_t gb = fused_gmax_bytes(seqs, n_seqs);
  void* planes = static_cast<char*>(workspace) + gb;
  const size_t planes_bytes = workspace_bytes - gb;
  if ((s = qsa_score_blocks(seqs, n_seqs, q_idx, q_idx_dtype, scores, ld, gmax, gld, planes, planes_bytes, stream)) !=
      QSA_OK)
    return s;
  return qsa_select_topk(seqs, n_seqs, scores, ld, gmax, gld, top_k, sel, cnt, nullptr, 0, stream);
}

// ------------------------------------------------------------------ steps 2 + 3 over key-axis chunks
namespace {

struct BlockedLayout {
  size_t chunk, planes, keys, ids, cnts, total;   // byte offsets of the parts
  int64_t ld_chunk;
};

BlockedLayout blocked_layout(const qsa_seq* seqs, int32_t n_seqs, int32_t top_k, int32_t block_keys) {
  auto up = [](size_t b) { return (b + 255) / 256 * 256; };
  int64_t rows = 0;
  for (int i = 0; i < n_seqs; ++i) rows = std::max<int64_t>(rows, seqs[i].n_rows);
  BlockedLayout L;
  L.ld_chunk = block_keys;
  const size_t chunk_b = up(sizeof(float) * (size_t)rows * (size_t)block_keys);
  const size_t planes_b = up(score_tc_workspace_bytes(block_keys));
  const size_t list_b = up(sizeof(uint32_t) * (size_t)rows * (size_t)top_k);
  const size_t cnt_b = up(sizeof(int32_t) * (size_t)std::max<int64_t>(rows, 1));
  L.chunk = 0;
  L.planes = chunk_b;
  L.keys = L.planes + planes_b;      // two running lists: keys[2], ids[2], counts[2]
  L.ids = L.keys + 2 * list_b;
  L.cnts = L.ids + 2 * list_b;
  L.total = L.cnts + 2 * cnt_b;
  return L;
}

}  // namespace

QSA_API size_t qsa_score_select_blocked_workspace_size(const qsa_seq* seqs, int32_t n_seqs, int32_t top_k,
                                                       int32_t block_keys) {
  if (!seqs || n_seqs < 1 || top_k < 1 || block_keys < 1) return 0;
  return blocked_layout(seqs, n_seqs, top_k, block_keys).total;
}

QSA_API qsa_status qsa_score_select_topk_blocked(const qsa_seq* seqs, int32_t n_seqs, const void* q_idx,
                                                 qsa_dtype q_idx_dtype, int32_t top_k, int32_t block_keys,
                                                 int32_t* sel, int32_t* cnt, void* workspace,
                                                 size_t workspace_bytes, void* stream) {
  const NvtxRange nvtx_range("qsa_score_select_topk_blocked");
  const char* fn = "qsa_score_select_topk_blocked";
  int64_t rows = 0;
  qsa_status s = check_rows(seqs, n_seqs, fn, &rows);
  if (s != QSA_OK) return s;
  if (q_idx_dtype != QSA_BF16)
    return fail(QSA_ERR_UNSUPPORTED, "%s: q_idx_dtype must be bf16 (tensor-core scoring)", fn);
  if (top_k < 1 || top_k > QSA_MAX_TOP_K)
    return fail(QSA_ERR_UNSUPPORTED, "%s: top_k=%d outside 1..%d", fn, top_k, QSA_MAX_TOP_K);
  if (block_keys < 128 || block_keys % 128 != 0 || top_k + block_keys > merge_select_max_union())
    return fail(QSA_ERR_UNSUPPORTED, "%s: block_keys=%d (a multiple of 128, top_k + block_keys <= %d)", fn,
                block_keys, merge_select_max_union());
  if (!q_idx || !sel || !cnt) return fail(QSA_ERR_INVALID_ARG, "%s: null pointer", fn);
  if (!aligned16(q_idx)) return fail(QSA_ERR_MISALIGNED, "%s: q_idx not 16-byte aligned", fn);
  for (int i = 0; i < n_seqs; ++i) {
    const qsa_seq& q = seqs[i];
    if (max_visible_blocks(q) > QSA_MAX_BLOCKS)
      return fail(QSA_ERR_UNSUPPORTED, "%s: sequence %d has more than %d blocks", fn, i, QSA_MAX_BLOCKS);
    if (max_visible_blocks(q) > 0) {
      if (!q.pooled) return fail(QSA_ERR_INVALID_ARG, "%s: sequence %d has no pooled keys", fn, i);
      if (q.pooled_stride < QSA_INDEX_DIM) return fail(QSA_ERR_INVALID_ARG, "%s: pooled_stride < 128", fn);
      if (!aligned16(q.pooled) || q.pooled_stride % 4 != 0)
        return fail(QSA_ERR_MISALIGNED, "%s: pooled keys of sequence %d not 16-byte aligned", fn, i);
    }
  }
  const BlockedLayout L = blocked_layout(seqs, n_seqs, top_k, block_keys);
  if (!workspace || workspace_bytes < L.total)
    return fail(QSA_ERR_WORKSPACE, "%s: workspace of %zu bytes needed, %zu given", fn, L.total,
                workspace ? workspace_bytes : (size_t)0);
  if (!aligned16(workspace)) return fail(QSA_ERR_MISALIGNED, "%s: workspace not aligned", fn);
  char* ws = static_cast<char*>(workspace);
  const size_t list_b = (L.ids - L.keys) / 2, cnt_b = (L.total - L.cnts) / 2;
  float* chunk = reinterpret_cast<float*>(ws + L.chunk);
  void* planes = ws + L.planes;
  cudaStream_t st = as_stream(stream);
  int32_t row_begin = 0;
  for (int i = 0; i < n_seqs; ++i) {
    const qsa_seq& q = seqs[i];
    const int64_t nbmax = max_visible_blocks(q);   // n_tokens / 4 (the last row sees the most)
    const int64_t n_chunks = std::max<int64_t>(1, (nbmax + block_keys - 1) / block_keys);
    const void* qi = static_cast<const char*>(q_idx) + (size_t)row_begin * QSA_INDEX_HEADS * QSA_INDEX_DIM * 2;
    for (int64_t c = 0; c < n_chunks; ++c) {
      const int64_t lo = c * block_keys;
      const int64_t n = std::max<int64_t>(0, std::min<int64_t>(block_keys, nbmax - lo));
      cudaError_t e = launch_score_tc(qi, 0, q.n_rows, q.n_tokens, q.pooled, q.pooled_stride, lo, n, chunk,
                                      L.ld_chunk, nullptr, 0, planes, st);
      if (e != cudaSuccess) return cuda_fail(e, fn);
      const int in = (int)(c & 1), out = 1 - in;
      MergeSelectParams m{};
      m.n_tokens = q.n_tokens;
      m.n_rows = q.n_rows;
      m.row_begin = row_begin;
      m.chunk = chunk;
      m.ld_chunk = L.ld_chunk;
      m.block_lo = lo;
      m.n_blocks = (int32_t)n;
      m.top_k = top_k;
      m.run_key_in = reinterpret_cast<const uint32_t*>(ws + L.keys + in * list_b);
      m.run_id_in = reinterpret_cast<const int32_t*>(ws + L.ids + in * list_b);
      m.run_cnt_in = reinterpret_cast<const int32_t*>(ws + L.cnts + in * cnt_b);
      m.run_key_out = reinterpret_cast<uint32_t*>(ws + L.keys + out * list_b);
      m.run_id_out = reinterpret_cast<int32_t*>(ws + L.ids + out * list_b);
      m.run_cnt_out = reinterpret_cast<int32_t*>(ws + L.cnts + out * cnt_b);
      m.first = c == 0;
      m.last = c == n_chunks - 1;
      m.sel = sel;
      m.cnt = cnt;
      if ((e = launch_merge_select(m, st)) != cudaSuccess) return cuda_fail(e, fn);
    }
    row_begin += q.n_rows;
  }
  return ok();
}

// ------------------------------------------------------------------ step 4
namespace {

// Longest selected list any row of the call can have: 4 tokens per listed
// block (at most min(sel_ld, visible blocks)) plus up to 3 tail tokens.
int64_t max_list(const qsa_seq* seqs, int32_t n_seqs, int32_t sel_ld) {
  int64_t m = 0;
  for (int i = 0; i < n_seqs; ++i) m = std::max(m, 4 * std::min<int64_t>(sel_ld, max_visible_blocks(seqs[i])) + 3);
  return m;
}

AttnPlan plan_splits(const qsa_seq* seqs, int32_t n_seqs, const qsa_attn_config* cfg, int32_t sel_ld, int64_t rows) {
  return attn_plan(cfg->kv_dtype, cfg->head_dim, rows * cfg->n_kv_heads, max_list(seqs, n_seqs, sel_ld),
                   cfg->n_splits);
}

size_t attn_ws_bytes(const AttnPlan& sp, int64_t rows, const qsa_attn_config* cfg) {
  return attn_workspace_bytes(sp, rows, cfg->n_q_heads, cfg->head_dim);
}

qsa_status check_attn_config(const qsa_attn_config* cfg, const char* fn) {
  if (!cfg) return fail(QSA_ERR_INVALID_ARG, "%s: null config", fn);
  if (cfg->n_q_heads < 1 || cfg->n_kv_heads < 1 || cfg->n_q_heads % cfg->n_kv_heads != 0)
    return fail(QSA_ERR_INVALID_ARG, "%s: n_q_heads=%d must be a positive multiple of n_kv_heads=%d", fn,
                cfg->n_q_heads, cfg->n_kv_heads);
  if (cfg->n_q_heads / cfg->n_kv_heads > 16)
    return fail(QSA_ERR_UNSUPPORTED, "%s: more than 16 query heads per KV head", fn);
  if (cfg->head_dim != 128 && cfg->head_dim != 256)
    return fail(QSA_ERR_UNSUPPORTED, "%s: head_dim=%d (supported: 128, 256)", fn, cfg->head_dim);
  if (!valid_dtype(cfg->q_dtype) || !valid_kv_dtype(cfg->kv_dtype) || !valid_dtype(cfg->out_dtype))
    return fail(QSA_ERR_UNSUPPORTED, "%s: unknown dtype", fn);
  if (quantized(cfg->kv_dtype) ? cfg->q_dtype != QSA_BF16 : cfg->q_dtype != cfg->kv_dtype)
    return fail(QSA_ERR_UNSUPPORTED, "%s: q_dtype must equal kv_dtype (bf16 with quantized K/V)", fn);
  if (!(cfg->scale >= 0.f) || isinf(cfg->scale)) return fail(QSA_ERR_INVALID_ARG, "%s: bad scale", fn);
  return QSA_OK;
}

qsa_status check_segments(const qsa_seq* seqs, int32_t n_seqs, const qsa_attn_config* cfg, const char* fn) {
  const int64_t es = (int64_t)dtype_size(cfg->kv_dtype);
  for (int i = 0; i < n_seqs; ++i) {
    const qsa_seq& s = seqs[i];
    if (s.n_segments < 1 || s.n_segments > QSA_MAX_SEGMENTS)
      return fail(QSA_ERR_INVALID_ARG, "%s: sequence %d has %d segments (1..%d)", fn, i, s.n_segments,
                  QSA_MAX_SEGMENTS);
    std::vector<std::pair<int64_t, int64_t>> ranges;
    for (int j = 0; j < s.n_segments; ++j) {
      const qsa_kv_segment& g = s.segments[j];
      if (!g.k || !g.v) return fail(QSA_ERR_INVALID_ARG, "%s: sequence %d segment %d has a null K/V", fn, i, j);
      if (g.first_token < 0 || g.n_tokens < 0)
        return fail(QSA_ERR_INVALID_ARG, "%s: sequence %d segment %d has a negative range", fn, i, j);
      if (g.tok_stride < cfg->head_dim || g.head_stride < 0)
        return fail(QSA_ERR_INVALID_ARG, "%s: sequence %d segment %d has bad strides", fn, i, j);
      if (!aligned16(g.k) || !aligned16(g.v) || (g.tok_stride * es) % 16 != 0 || (g.head_stride * es) % 16 != 0)
        return fail(QSA_ERR_MISALIGNED, "%s: sequence %d segment %d K/V not 16-byte aligned", fn, i, j);
      if (quantized(cfg->kv_dtype)) {
        if (!g.kv_scale) return fail(QSA_ERR_INVALID_ARG, "%s: sequence %d segment %d has no scales", fn, i, j);
        const uintptr_t align = cfg->kv_dtype == QSA_FP8_E4M3 ? 3u : 15u;
        if ((reinterpret_cast<uintptr_t>(g.kv_scale) & align) != 0)
          return fail(QSA_ERR_MISALIGNED, "%s: sequence %d segment %d scale records misaligned", fn, i, j);
        if (g.scale_head_stride < 0 || g.scale_tok_stride < 1)
          return fail(QSA_ERR_INVALID_ARG, "%s: sequence %d segment %d has bad scale strides", fn, i, j);
      }
      ranges.emplace_back(g.first_token, g.first_token + g.n_tokens);
    }
    std::sort(ranges.begin(), ranges.end());
    for (size_t j = 1; j < ranges.size(); ++j)
      if (ranges[j].first < ranges[j - 1].second)
        return fail(QSA_ERR_INVALID_ARG, "%s: sequence %d has overlapping segments", fn, i);
  }
  return QSA_OK;
}

template <int NSEQ>
qsa_status attn_chunk(const qsa_seq* seqs, int n, int32_t row_begin, const qsa_attn_config* cfg, const void* q,
                      const int32_t* sel, const int32_t* cnt, int32_t sel_ld, const AttnPlan& sp, int64_t total_rows,
                      bool tensor_cores, void* out, float* lse, float* part_o, float* part_lse, cudaStream_t st) {
  AttnParams<NSEQ> p{};
  int rows = 0, nseg = 0;
  p.row_base = row_begin;
  for (int i = 0; i < n; ++i) {
    AttnSeq& a = p.seq[i];
    a.n_tokens = seqs[i].n_tokens;
    a.row_begin = row_begin + rows;
    a.n_rows = seqs[i].n_rows;
    a.seg_begin = nseg;
    a.n_segs = seqs[i].n_segments;
    for (int j = 0; j < seqs[i].n_segments; ++j) {
      const qsa_kv_segment& g = seqs[i].segments[j];
      Segment& d = p.seg[nseg++];
      d.k = g.k;
      d.v = g.v;
      d.first = g.first_token;
      d.n = g.n_tokens;
      d.head_stride = g.head_stride;
      d.tok_stride = g.tok_stride;
      d.kv_scale = static_cast<const uint8_t*>(g.kv_scale);
      d.s_head_stride = g.scale_head_stride;
      d.s_tok_stride = g.scale_tok_stride;
    }
    rows += seqs[i].n_rows;
  }
  p.n_seqs = n;
  p.q = q;
  p.sel = sel;
  p.cnt = cnt;
  p.sel_ld = sel_ld;
  p.n_q_heads = cfg->n_q_heads;
  p.group = cfg->n_q_heads / cfg->n_kv_heads;
  p.head_dim = cfg->head_dim;
  p.scale = cfg->scale > 0.f ? cfg->scale : 1.0f / sqrtf((float)cfg->head_dim);
  p.n_splits = sp.n_splits;
  p.total_rows = (int32_t)total_rows;
  p.part_o = part_o;
  p.part_lse = part_lse;
  p.out = out;
  p.lse = lse;
  p.out_dtype = cfg->out_dtype;
  cudaError_t e = tensor_cores ? launch_attn_tc<NSEQ>(p, rows, st) : launch_attn<NSEQ>(p, rows, cfg->kv_dtype, sp.stages, st);
  if (e != cudaSuccess) return cuda_fail(e, "qsa_sparse_attn");
  return QSA_OK;
}

}  // namespace

QSA_API size_t qsa_attn_workspace_size(const qsa_seq* seqs, int32_t n_seqs, const qsa_attn_config* cfg, int32_t sel_ld) {
  int64_t rows = 0;
  if (check_rows(seqs, n_seqs, "qsa_attn_workspace_size", &rows) != QSA_OK) return 0;
  if (check_attn_config(cfg, "qsa_attn_workspace_size") != QSA_OK || sel_ld < 1) return 0;
  return attn_ws_bytes(plan_splits(seqs, n_seqs, cfg, sel_ld, rows), rows, cfg);
}

QSA_API qsa_status qsa_sparse_attn(const qsa_seq* seqs, int32_t n_seqs, const qsa_attn_config* cfg, const void* q,
                           const int32_t* sel, const int32_t* cnt, int32_t sel_ld, void* out, float* lse,
                           void* workspace, size_t workspace_bytes, void* stream) {
  const NvtxRange nvtx_range("qsa_sparse_attn");
  const char* fn = "qsa_sparse_attn";
  int64_t rows = 0;
  qsa_status s = check_rows(seqs, n_seqs, fn, &rows);
  if (s != QSA_OK) return s;
  if ((s = check_attn_config(cfg, fn)) != QSA_OK) return s;
  if (sel_ld < 1) return fail(QSA_ERR_INVALID_ARG, "%s: sel_ld < 1", fn);
  if (!q || !sel || !cnt || !out) return fail(QSA_ERR_INVALID_ARG, "%s: null pointer", fn);
  if (!aligned16(q) || !aligned16(out)) return fail(QSA_ERR_MISALIGNED, "%s: q/out not 16-byte aligned", fn);
  if ((s = check_segments(seqs, n_seqs, cfg, fn)) != QSA_OK) return s;
  const AttnPlan sp = plan_splits(seqs, n_seqs, cfg, sel_ld, rows);
  const size_t need = attn_ws_bytes(sp, rows, cfg);
  if (need > 0 && (!workspace || workspace_bytes < need))
    return fail(QSA_ERR_WORKSPACE, "%s: workspace of %zu bytes needed, %zu given", fn, need,
                workspace ? workspace_bytes : (size_t)0);
  if (need > 0 && !aligned16(workspace)) return fail(QSA_ERR_MISALIGNED, "%s: workspace not aligned", fn);
  float* part_o = nullptr;
  float* part_lse = nullptr;
  if (need > 0) attn_workspace_layout(sp, rows, cfg->n_q_heads, cfg->head_dim, workspace, &part_o, &part_lse);
  cudaStream_t st = as_stream(stream);
  // Calls with many rows and a single split run on the tensor cores.
  const bool tensor_cores = sp.n_splits == 1 &&
                            attn_tc_eligible(cfg->kv_dtype, cfg->head_dim, cfg->n_q_heads / cfg->n_kv_heads,
                                             max_list(seqs, n_seqs, sel_ld), rows);
  if (n_seqs == 1) {
    s = attn_chunk<1>(seqs, 1, 0, cfg, q, sel, cnt, sel_ld, sp, rows, tensor_cores, out, lse, part_o, part_lse, st);
  } else {
    int32_t row_begin = 0;
    for (int c = 0; c < n_seqs && s == QSA_OK; c += kLaunchSeqs) {
      const int n = std::min(kLaunchSeqs, n_seqs - c);
      s = attn_chunk<kLaunchSeqs>(seqs + c, n, row_begin, cfg, q, sel, cnt, sel_ld, sp, rows, tensor_cores, out, lse,
                                  part_o, part_lse, st);
      for (int i = 0; i < n; ++i) row_begin += seqs[c + i].n_rows;
    }
  }
  if (s != QSA_OK) return s;
  if (sp.n_splits > 1) {
    // Step 5 on the splits' partials.
    cudaError_t e = launch_merge(part_o, part_lse, sp.n_splits, rows * cfg->n_q_heads, cfg->head_dim, out,
                                 cfg->out_dtype, lse, st);
    if (e != cudaSuccess) return cuda_fail(e, fn);
  }
  return ok();
}

// ------------------------------------------------------------------ appending tokens (step 1 in place)
// The checks of an append and its launch parameters (pooling included).
static qsa_status build_append(const char* fn, const qsa_seq* seq, const qsa_attn_config* cfg, const void* k_new,
                               const void* v_new, const void* idx_new, void* idx_keys, int64_t idx_tok_stride,
                               qsa_dtype idx_dtype, AppendParams* out) {
  int64_t rows = 0;
  qsa_status s = check_rows(seq, 1, fn, &rows);
  if (s != QSA_OK) return s;
  if ((s = check_attn_config(cfg, fn)) != QSA_OK) return s;
  if (!valid_dtype(idx_dtype)) return fail(QSA_ERR_UNSUPPORTED, "%s: idx_dtype %d", fn, (int)idx_dtype);
  if (!k_new || !v_new || !idx_new || !idx_keys) return fail(QSA_ERR_INVALID_ARG, "%s: null pointer", fn);
  const int64_t idx_es = (int64_t)dtype_size(idx_dtype), kv_es = (int64_t)dtype_size(cfg->kv_dtype);
  if (idx_tok_stride < QSA_INDEX_DIM) return fail(QSA_ERR_INVALID_ARG, "%s: idx_tok_stride < 128", fn);
  if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(idx_new) || !aligned16(idx_keys) ||
      (idx_tok_stride * idx_es) % 16 != 0)
    return fail(QSA_ERR_MISALIGNED, "%s: pointers and strides must be 16-byte aligned", fn);
  if ((s = check_segments(seq, 1, cfg, fn)) != QSA_OK) return s;
  const int64_t L = seq->n_tokens, n_new = seq->n_rows;
  // Every new token must land in a segment (segments do not overlap).
  {
    std::vector<std::pair<int64_t, int64_t>> r;
    for (int j = 0; j < seq->n_segments; ++j)
      r.emplace_back(seq->segments[j].first_token, seq->segments[j].first_token + seq->segments[j].n_tokens);
    std::sort(r.begin(), r.end());
    int64_t t = L - n_new;
    for (const auto& e : r)
      if (e.first <= t && e.second > t) t = e.second;
    if (t < L) return fail(QSA_ERR_INVALID_ARG, "%s: token %lld is in no KV segment", fn, (long long)t);
  }
  const int64_t b0 = (L - n_new) / 4, b1 = L / 4;   // blocks the new tokens complete
  if (b1 > b0) {
    if (!seq->pooled) return fail(QSA_ERR_INVALID_ARG, "%s: no pooled keys to write", fn);
    if (seq->pooled_stride < QSA_INDEX_DIM || seq->pooled_stride % 4 != 0 || !aligned16(seq->pooled))
      return fail(QSA_ERR_MISALIGNED, "%s: pooled keys must be 16-byte aligned, stride >= 128", fn);
  }
  AppendParams p{};
  for (int j = 0; j < seq->n_segments; ++j) {
    const qsa_kv_segment& g = seq->segments[j];
    p.seg[j] = AppendSeg{const_cast<void*>(g.k), const_cast<void*>(g.v), g.first_token, g.n_tokens, g.head_stride,
                         g.tok_stride, const_cast<void*>(g.kv_scale), g.scale_head_stride, g.scale_tok_stride};
  }
  p.n_segs = seq->n_segments;
  p.n_kv_heads = cfg->n_kv_heads;
  p.head_dim = cfg->head_dim;
  p.kvq = cfg->kv_dtype == QSA_FP8_E4M3 ? 1 : cfg->kv_dtype == QSA_Q8_0 ? 2 : 0;
  p.n_tokens = L;
  p.n_new = n_new;
  p.k_new = k_new;
  p.v_new = v_new;
  p.kv_es = (int32_t)kv_es;
  p.row_bytes = cfg->head_dim * kv_es;
  p.row_chunks = p.row_bytes / 16;
  p.idx_new = idx_new;
  p.idx_keys = idx_keys;
  p.idx_stride = idx_tok_stride;
  p.idx_dtype = idx_dtype;
  p.idx_es = (int32_t)idx_es;
  p.idx_chunks = QSA_INDEX_DIM * idx_es / 16;
  p.pooled = const_cast<float*>(seq->pooled);
  p.pooled_stride = seq->pooled_stride;
  p.first_block = b0;
  // fp8 state: one warp (32 items) per K or V row, which it quantizes.
  p.kv_items = p.kvq ? 2 * (int64_t)cfg->n_kv_heads * n_new * 32 : 2 * (int64_t)cfg->n_kv_heads * n_new * p.row_chunks;
  p.idx_items = n_new * p.idx_chunks;
  p.pool_items = std::max<int64_t>(0, b1 - b0) * (QSA_INDEX_DIM / 4);
  *out = p;
  return QSA_OK;
}

QSA_API qsa_status qsa_append_tokens(const qsa_seq* seq, const qsa_attn_config* cfg, const void* k_new,
                                     const void* v_new, const void* idx_new, void* idx_keys, int64_t idx_tok_stride,
                                     qsa_dtype idx_dtype, void* stream) {
  const NvtxRange nvtx_range("qsa_append_tokens");
  const char* fn = "qsa_append_tokens";
  AppendParams p{};
  const qsa_status s = build_append(fn, seq, cfg, k_new, v_new, idx_new, idx_keys, idx_tok_stride, idx_dtype, &p);
  if (s != QSA_OK) return s;
  cudaError_t e = launch_append(p, as_stream(stream));
  if (e != cudaSuccess) return cuda_fail(e, fn);
  return ok();
}

QSA_API qsa_status qsa_append_score_blocks(const qsa_seq* seq, const qsa_attn_config* cfg, const void* k_new,
                                           const void* v_new, const void* idx_new, void* idx_keys,
                                           int64_t idx_tok_stride, qsa_dtype idx_dtype, const void* q_idx,
                                           qsa_dtype q_idx_dtype, float* scores, int64_t ld, float* group_max,
                                           int64_t group_ld, void* workspace, size_t workspace_bytes, void* stream) {
  const NvtxRange nvtx_range("qsa_append_score_blocks");
  const char* fn = "qsa_append_score_blocks";
  AppendParams p{};
  qsa_status s = build_append(fn, seq, cfg, k_new, v_new, idx_new, idx_keys, idx_tok_stride, idx_dtype, &p);
  if (s != QSA_OK) return s;
  // With at most 4 rows (K/V state not quantized, bf16 index queries) the
  // scoring launch appends and pools itself; otherwise the append launch,
  // pooling included, comes first and plain scoring follows.  (At 5 to 8
  // rows the scoring is bound by its MMAs and the copies lengthen it: the
  // 261,120-token 8-row step measured 19.9k layer-steps/s end to end fused
  // against 20.5k with the append launch.)
  if (!p.kvq && q_idx_dtype == QSA_BF16 && seq->n_rows <= 4) {
    p.pool_items = 0;
    const void* const keys[1] = {idx_keys};
    const IdxKeys ik{keys, idx_tok_stride, idx_dtype};
    return score_blocks_impl(fn, seq, 1, &ik, q_idx, q_idx_dtype, scores, ld, group_max, group_ld, workspace,
                             workspace_bytes, stream, &p);
  }
  // (Arguments of the scoring are checked before anything is launched.)
  if ((s = score_blocks_impl(fn, seq, 1, nullptr, q_idx, q_idx_dtype, scores, ld, group_max, group_ld, workspace,
                             workspace_bytes, stream, nullptr, true)) != QSA_OK)
    return s;
  cudaError_t e = launch_append(p, as_stream(stream));
  if (e != cudaSuccess) return cuda_fail(e, fn);
  return score_blocks_impl(fn, seq, 1, nullptr, q_idx, q_idx_dtype, scores, ld, group_max, group_ld, workspace,
                           workspace_bytes, stream);
}

// ------------------------------------------------------------------ demand-mapped arena
QSA_API qsa_status qsa_arena_create(int32_t device, uint64_t reserve_bytes, qsa_arena** arena) {
  const char* fn = "qsa_arena_create";
  if (!arena) return fail(QSA_ERR_INVALID_ARG, "%s: null output pointer", fn);
  *arena = nullptr;
  if (device < 0 || reserve_bytes == 0) return fail(QSA_ERR_INVALID_ARG, "%s: device %d, %llu bytes", fn, device,
                                                    (unsigned long long)reserve_bytes);
  const char* why = "";
  const qsa_status s = arena_create(device, reserve_bytes, arena, &why);
  return s == QSA_OK ? ok() : fail(s, "%s: %s", fn, why);
}

QSA_API qsa_status qsa_arena_ensure(qsa_arena* arena, uint64_t bytes) {
  const char* fn = "qsa_arena_ensure";
  if (!arena) return fail(QSA_ERR_INVALID_ARG, "%s: null arena", fn);
  const char* why = "";
  const qsa_status s = arena_ensure(arena, bytes, &why);
  return s == QSA_OK ? ok() : fail(s, "%s: %s", fn, why);
}

QSA_API void* qsa_arena_base(const qsa_arena* arena) { return arena ? arena_base(arena) : nullptr; }
QSA_API uint64_t qsa_arena_mapped(const qsa_arena* arena) { return arena ? arena_mapped(arena) : 0; }
QSA_API uint64_t qsa_arena_reserved(const qsa_arena* arena) { return arena ? arena_reserved(arena) : 0; }
QSA_API uint64_t qsa_arena_granularity(const qsa_arena* arena) { return arena ? arena_granularity(arena) : 0; }

QSA_API qsa_status qsa_arena_destroy(qsa_arena* arena) {
  const char* fn = "qsa_arena_destroy";
  if (!arena) return ok();
  const char* why = "";
  const qsa_status s = arena_destroy(arena, &why);
  return s == QSA_OK ? ok() : fail(s, "%s: %s", fn, why);
}

// ------------------------------------------------------------------ step 5
QSA_API qsa_status qsa_lse_merge(const float* o_parts, const float* lse_parts, int32_t n_parts, int64_t n_rows,
                         int32_t head_dim, void* out, qsa_dtype out_dtype, float* lse_out, void* stream) {
  const NvtxRange nvtx_range("qsa_lse_merge");
  const char* fn = "qsa_lse_merge";
  if (n_parts < 1 || n_rows < 0) return fail(QSA_ERR_INVALID_ARG, "%s: n_parts >= 1 and n_rows >= 0 required", fn);
  if (head_dim < 4 || head_dim % 4 != 0) return fail(QSA_ERR_UNSUPPORTED, "%s: head_dim must be a multiple of 4", fn);
  if (!valid_dtype(out_dtype)) return fail(QSA_ERR_UNSUPPORTED, "%s: out_dtype %d", fn, (int)out_dtype);
  if (n_rows == 0) return ok();
  if (!o_parts || !lse_parts || !out) return fail(QSA_ERR_INVALID_ARG, "%s: null pointer", fn);
  if (!aligned16(o_parts) || !aligned16(out)) return fail(QSA_ERR_MISALIGNED, "%s: o_parts/out not aligned", fn);
  cudaError_t e = launch_merge(o_parts, lse_parts, n_parts, n_rows, head_dim, out, out_dtype, lse_out,
                               as_stream(stream));
  if (e != cudaSuccess) return cuda_fail(e, fn);
  return ok();
}


// ------------------------------------------------------------------ attention without a caller workspace
// Some callers cannot give the library device memory: a host framework that
// owns every byte of device memory through its own pool and offers plugins no
// allocation, or a serving loop that must never call cudaMalloc because the
// call can synchronize the device and stall every stream.  For them
// qsa_sparse_attn_noalloc keeps the scratch the split merge needs in a fixed
// array of static device memory, part of the loaded library itself.
namespace {

constexpr size_t kNoAllocScratchBytes = QSA_NOALLOC_SCRATCH_BYTES;   // held by every GPU that loads the library
__device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_noalloc_mu;
void* g_noalloc_ptr[64];

// Device address of the scratch array on the current device (host code must
// not pass the array's name to a kernel).  Looked up on every call made
// outside a stream capture, so a device reset (which reloads the module)
// never leaves a stale address behind; a call inside a capture reuses the
// address an earlier call on that device found.
qsa_status noalloc_scratch(const char* fn, cudaStream_t st, void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, fn);
  if (dev < 0 || dev >= 64) return fail(QSA_ERR_UNSUPPORTED, "%s: device %d", fn, dev);
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  e = cudaStreamIsCapturing(st, &cap);
  if (e != cudaSuccess) return cuda_fail(e, fn);
  std::lock_guard<std::mutex> lk(g_noalloc_mu);
  if (cap == cudaStreamCaptureStatusNone) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return cuda_fail(e, "qsa_sparse_attn_noalloc: cudaGetSymbolAddress");
    g_noalloc_ptr[dev] = p;
  } else if (!g_noalloc_ptr[dev]) {
    return fail(QSA_ERR_INVALID_ARG, "%s: the first call on a device must come before any stream capture", fn);
  }
  *out = g_noalloc_ptr[dev];
  return QSA_OK;
}

}  // namespace

QSA_API qsa_status qsa_sparse_attn_noalloc(const qsa_seq* seqs, int32_t n_seqs, const qsa_attn_config* cfg,
                                           const void* q, const int32_t* sel, const int32_t* cnt, int32_t sel_ld,
                                           void* out, float* lse, void* stream) {
  const NvtxRange nvtx_range("qsa_sparse_attn_noalloc");
  const char* fn = "qsa_sparse_attn_noalloc";
  int64_t rows = 0;
  qsa_status s = check_rows(seqs, n_seqs, fn, &rows);
  if (s != QSA_OK) return s;
  if ((s = check_attn_config(cfg, fn)) != QSA_OK) return s;
  if (sel_ld < 1) return fail(QSA_ERR_INVALID_ARG, "%s: sel_ld < 1", fn);
  if (!q || !sel || !cnt || !out) return fail(QSA_ERR_INVALID_ARG, "%s: null pointer", fn);
  if (!aligned16(q) || !aligned16(out)) return fail(QSA_ERR_MISALIGNED, "%s: q/out not 16-byte aligned", fn);
  if ((s = check_segments(seqs, n_seqs, cfg, fn)) != QSA_OK) return s;
  const size_t need = qsa_attn_workspace_size(seqs, n_seqs, cfg, sel_ld);
  if (need > kNoAllocScratchBytes)
    return fail(QSA_ERR_UNSUPPORTED, "%s: this call needs %zu bytes of scratch; the built-in array holds %zu", fn,
                need, kNoAllocScratchBytes);
  void* scratch = nullptr;
  if (need > 0 && (s = noalloc_scratch(fn, as_stream(stream), &scratch)) != QSA_OK) return s;
  return qsa_sparse_attn(seqs, n_seqs, cfg, q, sel, cnt, sel_ld, out, lse, scratch, need > 0 ? kNoAllocScratchBytes : 0,
                         stream);
}
