/*
 * qsa.h -- C ABI of the GB300 (sm_103a) Qwen Sparse Attention layer-step
 * library, libqsa.so.
 *
 * One QSA layer step over a long KV cache, for decode, verify and prefill:
 *   1. qsa_pool_index_keys  average every 4 consecutive 128-wide index keys
 *                           into one pooled block key;
 *   2. qsa_score_blocks     score every complete block a query row can see as
 *                           (1/sqrt(128)) * sum over 4 index heads of
 *                           ReLU(q_h . pooled_block);
 *   3. qsa_select_topk      keep the 512 best blocks (2,048 tokens), lower id
 *                           winning ties; the incomplete tail block is always
 *                           attended and is implied, not listed;
 *   4. qsa_sparse_attn      exact softmax attention over only the selected
 *                           rows, 24 query heads over 2 KV heads, each
 *                           selected K/V row read once per 12-head group,
 *                           split over the selected rows and over KV segments;
 *   5. qsa_lse_merge        merge partial results by their log-sum-exp.
 * Sources: hipfire, "QSA sparse attention and the VMM KV backend", section 02
 * "How QSA chooses what to read" and section 03 "How hipfire runs it on RDNA"
 * (steps 1-4); MTPLX pull request #610 (segmented KV cache), "How it works,
 * in plain terms" and "What changes" (step 5 and KV segments).
 *
 * Conventions (all entry points):
 *  - Every function returns a qsa_status; nothing throws across the ABI.
 *    On failure, qsa_last_error() gives a one-line reason (per host thread).
 *  - Tensors are caller-owned DEVICE memory unless marked "host".  The
 *    library never allocates, frees, copies or resizes caller buffers.
 *  - Work is enqueued asynchronously on `stream` (a cudaStream_t; NULL means
 *    the legacy default stream).  Argument checks run on the host before any
 *    launch; a launch failure returns QSA_ERR_CUDA.  Errors of kernels that
 *    already ran surface on the stream as CUDA errors.
 *  - Descriptor arrays (qsa_seq) are HOST memory and are consumed before the
 *    call returns; their contents are copied into kernel parameters, so a
 *    call can be captured into a CUDA graph.
 *  - Rows: a call covers the query rows of n_seqs sequences, concatenated in
 *    sequence order (row index r = rows of earlier sequences + j).  Row j of
 *    a sequence with n_tokens = L and n_rows = M sits at absolute position
 *    p = L - M + j and sees tokens 0..p (causal).  Nothing past L is read,
 *    so the cache may hold more tokens than L: a run of consecutive rows
 *    anywhere in a cache is one descriptor with L = its last position + 1,
 *    and rows at scattered positions (or one sequence's rows split over
 *    several calls) are several descriptors over the same pooled keys and
 *    K/V segments.
 *  - Blocks: block b holds tokens 4b..4b+3.  A row at p sees
 *    nb(p) = floor((p+1)/4) complete blocks and a tail of (p+1) mod 4 tokens
 *    4*nb(p)..p.
 *  - Alignment: every device pointer must be 16-byte aligned and every row
 *    stride a multiple of 16 bytes (QSA_ERR_MISALIGNED otherwise).
 */
#ifndef QSA_H_
#define QSA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define QSA_VERSION 111            /* 1.1.1 */
#define QSA_INDEX_DIM 128          /* width of an index key and an index-query head */
#define QSA_INDEX_HEADS 4          /* index-query heads per query row */
#define QSA_BLOCK_TOKENS 4         /* tokens pooled into one block key */
#define QSA_TOP_K 512              /* the method's block budget */
#define QSA_MAX_TOP_K 1024         /* largest top_k qsa_select_topk accepts */
#define QSA_MAX_SEGMENTS 12        /* KV segments per sequence */
#define QSA_MAX_FEW_ROWS 8         /* rows per sequence on the few-row scoring path */
#define QSA_MAX_BLOCKS (1 << 18)   /* complete blocks per sequence (1,048,576 tokens) */
#define QSA_SCORE_GROUP 16         /* blocks per group of the group maxima (qsa_score_blocks) */

typedef enum qsa_status {
  QSA_OK = 0,
  QSA_ERR_INVALID_ARG = 1,   /* null pointer, negative size, inconsistent shapes */
  QSA_ERR_UNSUPPORTED = 2,   /* dtype / head_dim / head count / size the library does not build */
  QSA_ERR_MISALIGNED = 3,    /* pointer or stride not 16-byte aligned */
  QSA_ERR_WORKSPACE = 4,     /* workspace null or smaller than the *_workspace_size result */
  QSA_ERR_CUDA = 5,          /* a CUDA runtime call or launch failed */
  QSA_ERR_DEVICE_CHECK = 6,  /* qsa_check_device_status: kernels met inputs outside the contract */
  QSA_ERR_TIMEOUT = 7        /* qsa_check_device_status: a device-side wait gave up */
} qsa_status;

typedef enum qsa_dtype {
  QSA_F32 = 0,               /* IEEE binary32 */
  QSA_BF16 = 1,              /* bfloat16 */
  QSA_FP8_E4M3 = 2,          /* K/V state only: E4M3 codes with per-(head, token) f16 scales */
  QSA_Q8_0 = 3               /* K/V state only: int8 codes with an f16 scale per 32 elements */
} qsa_dtype;

/* One contiguous piece of a sequence's K/V cache (MTPLX pull request #610:
 * a cache kept as immutable per-turn segments plus a growing tail).
 * Element (h, t, d) of K -- KV head h, the segment's t-th token, channel d --
 * is at k[h * head_stride + t * tok_stride + d]; V likewise.  The segment
 * holds absolute tokens first_token .. first_token + n_tokens - 1.  Segments
 * of one sequence must not overlap; tokens no segment covers are not
 * attended.
 * Quantized state (hipfire, section 02, table "State formats"): k and v hold
 * 1-byte codes with the element layout above, and the scales of (h, t) form
 * one record at kv_scale + R * (h * scale_head_stride + t * scale_tok_stride)
 * bytes:
 *   QSA_FP8_E4M3  E4M3 codes, value = code * scale of the row; the record is
 *                 the K row's f16 scale then the V row's (R = 4, 4-byte
 *                 aligned);
 *   QSA_Q8_0      int8 codes, value = code * scale of its block of 32
 *                 elements; the record is the K row's D/32 f16 block scales
 *                 then the V row's (R = D/8 bytes, 16-byte aligned).
 * Unused for f32 / bf16 state. */
typedef struct qsa_kv_segment {
  const void* k;             /* device, kv_dtype */
  const void* v;             /* device, kv_dtype */
  int64_t first_token;
  int64_t n_tokens;
  int64_t head_stride;       /* elements between KV heads */
  int64_t tok_stride;        /* elements between tokens, >= head_dim */
  const void* kv_scale;      /* quantized state: device scale records */
  int64_t scale_head_stride; /* quantized state: records between KV heads */
  int64_t scale_tok_stride;  /* quantized state: records between tokens */
} qsa_kv_segment;

/* One sequence of a call (host struct). */
typedef struct qsa_seq {
  int64_t n_tokens;          /* L: tokens in the cache, this call's rows included */
  int32_t n_rows;            /* query rows, 1..L; row j sits at L - n_rows + j */
  int32_t n_segments;        /* qsa_sparse_attn: KV segments used, 1..QSA_MAX_SEGMENTS */
  const float* pooled;       /* qsa_score_blocks: device [>= floor(L/4)] x pooled_stride f32 */
  int64_t pooled_stride;     /* floats between pooled blocks, >= 128 */
  qsa_kv_segment segments[QSA_MAX_SEGMENTS];
} qsa_seq;

/* Attention shape and options (host struct). */
typedef struct qsa_attn_config {
  int32_t n_q_heads;         /* Hq, e.g. 24 */
  int32_t n_kv_heads;        /* Hkv, e.g. 2; Hq / Hkv must be <= 16 */
  int32_t head_dim;          /* 128 or 256 */
  qsa_dtype q_dtype;         /* dtype of q; kv_dtype, or bf16 with quantized K/V */
  qsa_dtype kv_dtype;        /* dtype of every segment's K and V */
  qsa_dtype out_dtype;       /* dtype of out */
  float scale;               /* logit scale; 0 means 1/sqrt(head_dim) */
  int32_t n_splits;          /* splits of each row's selected rows, <= 256; 0 = library's choice */
} qsa_attn_config;

/*
 * Demand-mapped device arena (hipfire, "QSA sparse attention and the VMM KV
 * backend", section 04 "VMM: reserve big, commit what you touch").  Reserves
 * a virtual address range for the largest cache and maps physical device
 * memory into it only as the cache grows; the base pointer never changes, so
 * segment descriptors and CUDA graphs captured with addresses inside the
 * arena stay valid across growth.  Host calls; not for concurrent use on one
 * arena from several threads without the caller's own ordering (ensure() is
 * internally locked).
 *   qsa_arena_create   reserve >= reserve_bytes (rounded up to the device's
 *                      recommended allocation granularity) on `device`;
 *                      nothing mapped yet
 *   qsa_arena_ensure   map physical memory so that [base, base + bytes) is
 *                      backed (granularity multiples; never unmaps); bytes
 *                      beyond the reservation: QSA_ERR_INVALID_ARG; device
 *                      memory exhausted: QSA_ERR_CUDA.  Mapping does not
 *                      disturb work in flight on already-mapped bytes.
 *   qsa_arena_base / _mapped / _reserved / _granularity   (0 / NULL for NULL)
 *   qsa_arena_destroy  waits for the device, unmaps and frees the physical
 *                      memory and the address range; NULL is a no-op
 * Errors: QSA_ERR_INVALID_ARG, QSA_ERR_CUDA (no device, driver refusal).
 */
typedef struct qsa_arena qsa_arena;
qsa_status qsa_arena_create(int32_t device, uint64_t reserve_bytes, qsa_arena** arena);
qsa_status qsa_arena_ensure(qsa_arena* arena, uint64_t bytes);
void* qsa_arena_base(const qsa_arena* arena);
uint64_t qsa_arena_mapped(const qsa_arena* arena);
uint64_t qsa_arena_reserved(const qsa_arena* arena);
uint64_t qsa_arena_granularity(const qsa_arena* arena);
qsa_status qsa_arena_destroy(qsa_arena* arena);

/* Human-readable name of a status code (static storage). */
const char* qsa_status_string(qsa_status status);

/* Reason for the last failing call on this host thread ("" if none). */
const char* qsa_last_error(void);

/* QSA_VERSION of the loaded library. */
int32_t qsa_version(void);

/*
 * Device-side waits that gave up since the library was loaded, summed over
 * its kernels.  The pipelined kernels wait on shared-memory barriers for
 * their own copies and tensor-core operations; each wait gives up after about
 * two seconds instead of hanging the GPU, and the kernel then runs to its end
 * with an invalid result.  0 in normal operation; -1 if the counters could
 * not be read.  Reads device memory: waits for the device to be idle.
 */
int32_t qsa_wait_timeouts(void);

/*
 * The device-side checks since the previous call (or since the library was
 * loaded), after synchronizing `stream`:
 *   QSA_ERR_TIMEOUT       a wait of a pipelined kernel (or of
 *                         qsa_selftest_wait_timeout) gave up -- that
 *                         launch's result is invalid;
 *   QSA_ERR_DEVICE_CHECK  the attention met selected block ids outside
 *                         [0, nb) among a row's first cnt entries (skipped),
 *                         or the selection met NaN scores among its
 *                         candidates (NaN ranks above every number);
 *   QSA_OK                neither.
 * qsa_last_error() gives the counts.  The counters belong to the current
 * device (each GPU keeps its own) and cover all its streams and threads; a
 * call reads and clears those of the current device.  Launches still running
 * on other streams may be counted by the next call.
 * Errors: QSA_ERR_CUDA (the stream or the counters could not be read).
 */
qsa_status qsa_check_device_status(void* stream);

/*
 * Test hook for the timeout path: one thread waits on a shared-memory
 * barrier that nothing completes, gives up after limit_us microseconds
 * (1 .. 2,000,000) and records the expired wait, which the next
 * qsa_check_device_status reports as QSA_ERR_TIMEOUT (qsa_wait_timeouts does
 * not count it).  The kernel ends by itself; the context stays usable.
 * Errors: QSA_ERR_INVALID_ARG (limit), QSA_ERR_CUDA (launch).
 */
qsa_status qsa_selftest_wait_timeout(int32_t limit_us, void* stream);

/*
 * Step 1 -- pooling (hipfire, section 02: every 4 consecutive index keys are
 * averaged into one pooled block key).
 *   pooled[b * pooled_stride + d] = ((k[4b][d] + k[4b+1][d]) + k[4b+2][d] + k[4b+3][d]) / 4
 * in fp32, for b in [first_block, first_block + n_blocks), d < 128, where
 * k[t][d] = idx_keys[t * tok_stride + d].  Blocks must be complete (the caller
 * guarantees tokens up to 4*(first_block + n_blocks) - 1 exist).  A decode or
 * verify step pools only the blocks its new tokens completed.
 *   idx_keys       device [tokens, tok_stride], idx_dtype
 *   pooled         device f32, written only at the listed blocks
 * n_blocks == 0 is a no-op.
 */
qsa_status qsa_pool_index_keys(const void* idx_keys, qsa_dtype idx_dtype, int64_t tok_stride,
                               int64_t first_block, int64_t n_blocks, float* pooled,
                               int64_t pooled_stride, void* stream);

/*
 * Appending tokens with in-place pooling (step 1 and the cache writes either
 * side of it: hipfire, section 02 -- a QSA layer writes K/V and an index key
 * for every token, and every 4 index keys are averaged into a pooled block
 * key; MTPLX pull request #482, optimisation 1 -- the new rows' K/V are
 * written into the existing cache).  For the n = seq->n_rows newest tokens
 * t = L - n .. L - 1 (L = seq->n_tokens, the cache length after the append):
 *   K/V:  head h of token t -> the segment s covering t, at
 *         s.k[h * s.head_stride + (t - s.first_token) * s.tok_stride + d]
 *         (s.v likewise), from k_new[(h * n + (t - L + n)) * D + d];
 *   index keys: idx_keys[t * idx_tok_stride + c] = idx_new[(t - L + n) * 128 + c];
 *   pooled keys of every block the new tokens complete (floor((L - n) / 4)
 *   <= b < floor(L / 4)), exactly as qsa_pool_index_keys computes them,
 *   reading earlier tokens' index keys from idx_keys.
 * One launch.  The library writes into the caller's caches here (and only
 * here): the segments' K/V and seq->pooled are written through their
 * pointers, which the descriptor declares const for the read-only calls.
 *   seq            host descriptor: n_tokens, n_rows (= n), n_segments,
 *                  segments, pooled, pooled_stride
 *   cfg            n_kv_heads, head_dim, kv_dtype (other fields checked as
 *                  for qsa_sparse_attn)
 *   k_new, v_new   device [Hkv, n, D] kv_dtype, contiguous; bf16 when the
 *                  state is quantized, and each (K or V, head, token) row is
 *                  then written in it: QSA_FP8_E4M3 -- scale = f16(f32(amax /
 *                  448)), codes = the E4M3 values nearest to f32(x / scale),
 *                  ties to even, saturated at 448; QSA_Q8_0 -- per block of
 *                  32, scale = f16(f32(amax / 127)), codes = the integers
 *                  nearest to f32(x / scale), halves away from zero, within
 *                  +-127 (0 codes where a scale is 0)
 *   idx_new        device [n, 128] idx_dtype, contiguous
 *   idx_keys       device index-key cache, [>= L, idx_tok_stride] idx_dtype
 * Errors: QSA_ERR_INVALID_ARG (a new token in no segment, null pointers,
 * n > L), QSA_ERR_MISALIGNED, QSA_ERR_UNSUPPORTED (dtypes, head_dim).
 */
qsa_status qsa_append_tokens(const qsa_seq* seq, const qsa_attn_config* cfg, const void* k_new, const void* v_new,
                             const void* idx_new, void* idx_keys, int64_t idx_tok_stride, qsa_dtype idx_dtype,
                             void* stream);

/*
 * qsa_append_tokens, then qsa_pool_score_blocks's step 2 (every visible
 * block of seq scored as qsa_score_blocks does), in one call for one
 * sequence: the same caches, pooled keys, scores and group maxima as the
 * two calls.  With bf16 index queries, at most 4 rows and K/V state that is
 * not quantized (bf16 or f32), the scoring launch does the whole append
 * itself -- the new tokens' K/V rows and index keys are copied by threads
 * that issue no loads of pooled keys, and the blocks they complete are
 * pooled from idx_new (new tokens) and idx_keys (earlier ones) before they
 * are scored -- so the step keeps one launch; otherwise an append launch
 * precedes the scoring.
 *   seq, cfg, k_new, v_new, idx_new, idx_keys, idx_tok_stride, idx_dtype
 *                  as qsa_append_tokens
 *   q_idx ... workspace_bytes, stream   as qsa_score_blocks (one sequence)
 * Errors: those of the two calls; nothing is launched when either's
 * arguments fail their checks.
 */
qsa_status qsa_append_score_blocks(const qsa_seq* seq, const qsa_attn_config* cfg, const void* k_new,
                                   const void* v_new, const void* idx_new, void* idx_keys, int64_t idx_tok_stride,
                                   qsa_dtype idx_dtype, const void* q_idx, qsa_dtype q_idx_dtype, float* scores,
                                   int64_t ld, float* group_max, int64_t group_ld, void* workspace,
                                   size_t workspace_bytes, void* stream);

/*
 * Step 2 -- block scoring (hipfire, section 02: four index-query heads score
 * every pooled block; section 03: a few-row variant for decode and verify
 * and a wide variant for prefill).
 *   scores[r * ld + b] = (1/sqrt(128)) * sum_{h<4} max(0, q_idx[r][h] . pooled_s[b])
 * for every b < nb(p_r); entries b >= nb(p_r) are left unwritten.  With
 * group_max given, also the maximum score of every group of QSA_SCORE_GROUP
 * consecutive blocks:
 *   group_max[r * group_ld + g] = max { scores[r * ld + b] : 16g <= b < min(16g + 16, nb(p_r)) }
 * for g < ceil(nb(p_r) / 16); other entries are left unwritten.
 *   seqs, n_seqs   host descriptors; uses n_tokens, n_rows, pooled, pooled_stride
 *   q_idx          device [rows, 4, 128], q_idx_dtype
 *   scores         device [rows, ld] f32, ld >= max_r nb(p_r)
 *   group_max      device [rows, group_ld] f32, group_ld >= max_r ceil(nb(p_r) / 16)
 *                  and a multiple of 4; may be NULL (not written)
 *   workspace      device scratch of >= qsa_score_workspace_size bytes, or NULL
 *                  (then sequences of more than 8 rows use a slower
 *                  warp-level tensor-pipe kernel); its contents need no
 *                  initialisation; calls sharing it must not run concurrently
 * Arithmetic: fp32 accumulation of products that lose nothing of the fp32
 * pooled key beyond one fp32 ulp (bf16 index queries on the tensor pipe:
 * for <= 8 rows per sequence the key is split into two tf32 parts; for more
 * rows into three bf16 parts that sum to it exactly; fp32 index queries on
 * the CUDA cores).
 */
qsa_status qsa_score_blocks(const qsa_seq* seqs, int32_t n_seqs, const void* q_idx,
                            qsa_dtype q_idx_dtype, float* scores, int64_t ld, float* group_max,
                            int64_t group_ld, void* workspace, size_t workspace_bytes, void* stream);

/*
 * Steps 1 and 2 in one call (hipfire, section 02): pools the blocks that each
 * sequence's rows complete -- blocks floor((L - n_rows) / 4) .. floor(L / 4)
 * - 1, from idx_keys[i] as qsa_pool_index_keys does, written into the
 * sequence's pooled array -- and scores every visible block as
 * qsa_score_blocks does.  On the few-row path (bf16 index queries, at most 4
 * rows per sequence) the scoring kernel pools those blocks itself, so the two
 * steps are one launch; elsewhere a pooling launch precedes the scoring.
 *   idx_keys        HOST array of n_seqs device pointers: sequence i's index
 *                   keys [>= L tokens] x idx_tok_stride of idx_dtype (f32 or
 *                   bf16), 16-byte aligned; may be NULL for a sequence whose
 *                   rows complete no block
 *   idx_tok_stride  elements between tokens, >= 128, a multiple of 16 bytes
 *   the rest        as qsa_score_blocks; seqs[i].pooled is written for the
 *                   completed blocks
 * Errors: as qsa_score_blocks and qsa_pool_index_keys.
 */
qsa_status qsa_pool_score_blocks(const qsa_seq* seqs, int32_t n_seqs, const void* const* idx_keys,
                                 int64_t idx_tok_stride, qsa_dtype idx_dtype, const void* q_idx, qsa_dtype q_idx_dtype,
                                 float* scores, int64_t ld, float* group_max, int64_t group_ld, void* workspace,
                                 size_t workspace_bytes, void* stream);

/*
 * Scratch bytes qsa_score_blocks can use: with bf16 index queries, sequences
 * of more than 4 rows (prefill chunks) are scored as one tensor-core product
 * (tcgen05) against the pooled keys split into three bf16 planes, kept in the
 * workspace (768 bytes per complete block of the largest such sequence).
 * 0 when no sequence takes that path.
 */
size_t qsa_score_workspace_size(const qsa_seq* seqs, int32_t n_seqs, qsa_dtype q_idx_dtype);

/*
 * Scratch bytes qsa_select_topk needs for these sequences.  The kernel keeps
 * all selection state in shared memory and this returns 0; the workspace
 * arguments are kept so that variants needing scratch keep the ABI.
 */
size_t qsa_select_workspace_size(const qsa_seq* seqs, int32_t n_seqs, int32_t top_k);

/*
 * Step 3 -- top-k block selection (hipfire, section 02: the top-scoring
 * blocks within a 2,048-token budget, 512 blocks, plus the incomplete block
 * at the end; section 03: a radix select from the scores).
 * Per row r: k_r = min(top_k, nb(p_r)) blocks, ordered by score descending,
 * then block id ascending (ties go to the lower id; -0.0 equals +0.0).
 *   sel[r * top_k + i], i < cnt[r]   the kept block ids, ascending
 *   sel[r * top_k + i], i >= cnt[r]  -1
 *   cnt[r]                           k_r
 * The tail block (tokens 4*nb(p_r)..p_r) is not listed; qsa_sparse_attn adds
 * it.  Scores must not be NaN.  top_k in 1..QSA_MAX_TOP_K.
 *   scores         device [rows, ld] f32 (as written by qsa_score_blocks)
 *   group_max      device [rows, group_ld] f32, the group maxima of exactly
 *                  these scores as qsa_score_blocks writes them; may be NULL,
 *                  and then the kernel takes the maxima from the scores
 *   sel, cnt       device int32 [rows, top_k], [rows]
 *   workspace      device scratch of >= qsa_select_workspace_size bytes
 *                  (may be NULL when that size is 0)
 * One CTA per row: the group maxima bound the k-th score from below, so
 * only groups whose maximum can reach the top k are read again, and an
 * exact radix select runs over their blocks.
 */
qsa_status qsa_select_topk(const qsa_seq* seqs, int32_t n_seqs, const float* scores, int64_t ld,
                           const float* group_max, int64_t group_ld, int32_t top_k, int32_t* sel,
                           int32_t* cnt, void* workspace, size_t workspace_bytes, void* stream);

/*
 * Steps 2 and 3 in one call: qsa_score_blocks writes the group maxima into
 * the workspace (followed by its own scratch) and qsa_select_topk starts
 * from them.  Results are those of
 * the two separate calls.
 *   workspace      device scratch of >= qsa_score_select_workspace_size bytes;
 *                  its contents need no initialisation.  Two calls that share
 *                  a workspace must not run concurrently.
 * Other arguments as for qsa_score_blocks and qsa_select_topk.
 */
size_t qsa_score_select_workspace_size(const qsa_seq* seqs, int32_t n_seqs, int32_t top_k);

qsa_status qsa_score_select_topk(const qsa_seq* seqs, int32_t n_seqs, const void* q_idx,
                                 qsa_dtype q_idx_dtype, float* scores, int64_t ld, int32_t top_k,
                                 int32_t* sel, int32_t* cnt, void* workspace, size_t workspace_bytes,
                                 void* stream);

/*
 * Steps 2 and 3 over the key axis in chunks, with memory flat in the context
 * length (the SGLang launcher notes, section 2.3: score the rows against key
 * blocks of B_k, keep each part's top-k with ids, take the top-k of the
 * kept candidates; the top-k of a union equals the top-k of the per-part
 * top-k lists, so the result is exact).  Per sequence, blocks
 * [c * block_keys, (c + 1) * block_keys) are scored on the tensor cores into
 * a chunk buffer and merged into each row's running top-k (keys and ids in
 * ascending id order, so the lowest id still wins among equal scores).
 * Output: sel and cnt exactly as qsa_select_topk writes them for the
 * scores qsa_score_blocks would write; no [rows, blocks] score buffer.
 *   q_idx_dtype    QSA_BF16 (the tensor-core scoring); else QSA_ERR_UNSUPPORTED
 *   top_k          1..QSA_MAX_TOP_K
 *   block_keys     blocks per chunk: a multiple of 128, at least 128, and
 *                  top_k + block_keys <= 8192
 *   workspace      device scratch of >= qsa_score_select_blocked_workspace_size
 *                  bytes (chunk scores, key planes and two running lists,
 *                  sized by the largest sequence's rows and block_keys, not
 *                  by the context); contents need no initialisation; calls
 *                  that share it must not run concurrently
 * Other arguments as for qsa_score_blocks and qsa_select_topk.  One scoring
 * and one merge launch per chunk of each sequence.
 */
size_t qsa_score_select_blocked_workspace_size(const qsa_seq* seqs, int32_t n_seqs, int32_t top_k,
                                               int32_t block_keys);

qsa_status qsa_score_select_topk_blocked(const qsa_seq* seqs, int32_t n_seqs, const void* q_idx,
                                         qsa_dtype q_idx_dtype, int32_t top_k, int32_t block_keys, int32_t* sel,
                                         int32_t* cnt, void* workspace, size_t workspace_bytes, void* stream);

/*
 * Scratch bytes qsa_sparse_attn needs for this call: the normalised partial
 * outputs and lse values of every split when a (row, KV group) is cut into
 * several splits (0 when each has one).  sel_ld is the row stride of sel (the
 * top_k used for selection).
 */
size_t qsa_attn_workspace_size(const qsa_seq* seqs, int32_t n_seqs, const qsa_attn_config* cfg,
                               int32_t sel_ld);

/*
 * Step 4 -- sparse grouped-query attention over the selected rows (hipfire,
 * section 02: full attention over only the selected rows, <= 2,048 + 3 per
 * query; section 03: one workgroup per KV group of 12 query heads, so each
 * selected row is read once, not once per head), split over each row's
 * selected rows and over the KV segments and merged by log-sum-exp (MTPLX
 * pull request #610).
 * For row r and query head h (KV head g = h / (Hq/Hkv)), the attended rows
 * are R_r = {4b..4b+3 : b in sel[r][0..cnt[r])} U {4*nb(p_r)..p_r}, kept
 * where a segment of the row's sequence covers them; with z_t = scale*q.k_t,
 *   lse[r][h] = log(sum_{t in R_r} exp z_t),
 *   out[r][h] = sum_{t in R_r} exp(z_t - lse) v_t.
 * A row with no attended key gets out = 0 and lse = -inf.  fp32 accumulation;
 * out is rounded once to out_dtype.
 *   seqs           host; uses n_tokens, n_rows, n_segments, segments
 *   q              device [rows, Hq, head_dim], cfg->q_dtype
 *   sel, cnt       device, as written by qsa_select_topk (row stride sel_ld);
 *                  ids outside 0..nb(p_r)-1 are skipped, never dereferenced
 *   out            device [rows, Hq, head_dim], cfg->out_dtype
 *   lse            device [rows, Hq] f32 (natural log); may be NULL
 *   workspace      device scratch of >= qsa_attn_workspace_size bytes (may be
 *                  NULL when that size is 0); its contents need no
 *                  initialisation.  Two calls that share a workspace must
 *                  not run concurrently.
 * Each row's selected list is cut into cfg->n_splits splits per KV group
 * (at most 256; 0 = library's choice, about two CTAs per SM); every split
 * writes its normalised partial and lse, and a second launch merges them by
 * the log-sum-exp rule of qsa_lse_merge.
 * Supported: head_dim 128 or 256; q and K/V both bf16 or both f32;
 * Hq / Hkv <= 16.
 */
qsa_status qsa_sparse_attn(const qsa_seq* seqs, int32_t n_seqs, const qsa_attn_config* cfg,
                           const void* q, const int32_t* sel, const int32_t* cnt, int32_t sel_ld,
                           void* out, float* lse, void* workspace, size_t workspace_bytes,
                           void* stream);

/*
 * qsa_sparse_attn without a workspace argument.  The pages have no
 * counterpart to this entry point; it exists for callers that cannot give the
 * library device memory -- for example a host framework that owns all device
 * memory through its own pool and offers plugins no allocation, or a serving
 * loop that must never call cudaMalloc because that call can synchronize the
 * device.  It computes exactly what qsa_sparse_attn computes, with the
 * scratch the split merge needs taken from one array of static device memory
 * inside libqsa.so: QSA_NOALLOC_SCRATCH_BYTES (4 MiB), which every GPU that
 * loads the library holds until the process exits.
 *  - A call made outside a stream capture looks up the array's device
 *    address on the current device (a cheap driver query, repeated so that a
 *    device reset never leaves a stale address); a call inside a capture uses
 *    the address an earlier call on that device found, so make one call on
 *    the device before capturing (else QSA_ERR_INVALID_ARG).  A call whose
 *    plan needs no scratch (one split) looks up nothing.
 *  - It allocates and frees nothing.
 *  - Every call on a device shares the array: calls whose work overlaps on
 *    the GPU (other streams, other threads) race and must not be issued.
 *  - A call whose split plan needs more than QSA_NOALLOC_SCRATCH_BYTES of
 *    scratch (qsa_attn_workspace_size) fails with QSA_ERR_UNSUPPORTED.
 * Arguments, layouts and errors are otherwise those of qsa_sparse_attn.
 */
#define QSA_NOALLOC_SCRATCH_BYTES ((size_t)4 << 20)

qsa_status qsa_sparse_attn_noalloc(const qsa_seq* seqs, int32_t n_seqs, const qsa_attn_config* cfg,
                                   const void* q, const int32_t* sel, const int32_t* cnt, int32_t sel_ld,
                                   void* out, float* lse, void* stream);

/*
 * Step 5 -- log-sum-exp merge of partial attention results (MTPLX pull
 * request #610: per-segment partials merged by their log-sum-exp equal
 * single-buffer attention; rows without a visible key merge to zeros, not
 * NaN; partials stay fp32 and the merge rounds once).
 * For i < n_rows (a row is one (query row, head) pair):
 *   m = max_s lse_parts[s][i];  w_s = exp(lse_parts[s][i] - m)
 *   out[i][:] = sum_s w_s o_parts[s][i][:] / sum_s w_s;  lse_out[i] = m + log(sum_s w_s)
 * and out = 0, lse_out = -inf when every lse_parts[s][i] is -inf.
 *   o_parts        device f32 [n_parts, n_rows, head_dim] (normalised partials)
 *   lse_parts      device f32 [n_parts, n_rows]
 *   out            device [n_rows, head_dim], out_dtype
 *   lse_out        device f32 [n_rows]; may be NULL
 * head_dim must be a multiple of 4; n_parts >= 1.
 */
qsa_status qsa_lse_merge(const float* o_parts, const float* lse_parts, int32_t n_parts,
                         int64_t n_rows, int32_t head_dim, void* out, qsa_dtype out_dtype,
                         float* lse_out, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* QSA_H_ */
