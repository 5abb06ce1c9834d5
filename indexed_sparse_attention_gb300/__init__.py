"""Python binding of libqsa.so, the GB300 (sm_103a) QSA layer-step library.

Argument marshalling only: every step runs in the library's CUDA kernels.
PyTorch provides device memory and streams.  There is no CPU fallback; if
the library is missing the calls raise.

The five calls follow one Qwen Sparse Attention layer step (hipfire, "QSA
sparse attention and the VMM KV backend", sections 02 and 03; MTPLX pull
request #610 for KV segments and the log-sum-exp merge):

    pool_index_keys -> score_blocks -> select_topk -> sparse_attn (-> lse_merge)
"""
from __future__ import annotations

import ctypes
import dataclasses
import math
import os
from typing import Sequence

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libqsa.so")

F32, BF16, FP8, Q8 = 0, 1, 2, 3   # FP8 / Q8: quantized K/V state (E4M3 / int8 codes + f16 scales)
INDEX_DIM = 128
INDEX_HEADS = 4
TOP_K = 512
MAX_TOP_K = 1024
MAX_SEGMENTS = 12
SCORE_GROUP = 16

STATUS = {0: "QSA_OK", 1: "QSA_ERR_INVALID_ARG", 2: "QSA_ERR_UNSUPPORTED", 3: "QSA_ERR_MISALIGNED",
          4: "QSA_ERR_WORKSPACE", 5: "QSA_ERR_CUDA", 6: "QSA_ERR_DEVICE_CHECK", 7: "QSA_ERR_TIMEOUT"}
ERR_DEVICE_CHECK, ERR_TIMEOUT = 6, 7


class QSAError(RuntimeError):
    """A library call returned a status other than QSA_OK."""

    def __init__(self, fn: str, status: int, detail: str):
        super().__init__(f"{fn}: {STATUS.get(status, status)}: {detail}")
        self.status = status


class KVSegment(ctypes.Structure):
    _fields_ = [("k", ctypes.c_void_p), ("v", ctypes.c_void_p), ("first_token", ctypes.c_int64),
                ("n_tokens", ctypes.c_int64), ("head_stride", ctypes.c_int64), ("tok_stride", ctypes.c_int64),
                ("kv_scale", ctypes.c_void_p), ("scale_head_stride", ctypes.c_int64),
                ("scale_tok_stride", ctypes.c_int64)]


class SeqDesc(ctypes.Structure):
    _fields_ = [("n_tokens", ctypes.c_int64), ("n_rows", ctypes.c_int32), ("n_segments", ctypes.c_int32),
                ("pooled", ctypes.c_void_p), ("pooled_stride", ctypes.c_int64),
                ("segments", KVSegment * MAX_SEGMENTS)]


class AttnConfig(ctypes.Structure):
    _fields_ = [("n_q_heads", ctypes.c_int32), ("n_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("q_dtype", ctypes.c_int32), ("kv_dtype", ctypes.c_int32), ("out_dtype", ctypes.c_int32),
                ("scale", ctypes.c_float), ("n_splits", ctypes.c_int32)]


_lib = None
EXPORTS = ("qsa_status_string", "qsa_last_error", "qsa_version", "qsa_pool_index_keys", "qsa_score_blocks", "qsa_score_workspace_size",
           "qsa_select_workspace_size", "qsa_select_topk", "qsa_score_select_workspace_size",
           "qsa_score_select_topk", "qsa_attn_workspace_size", "qsa_sparse_attn", "qsa_sparse_attn_noalloc",
           "qsa_lse_merge", "qsa_wait_timeouts", "qsa_score_select_blocked_workspace_size",
           "qsa_score_select_topk_blocked", "qsa_append_tokens", "qsa_arena_create", "qsa_arena_ensure",
           "qsa_arena_base", "qsa_arena_mapped", "qsa_arena_reserved", "qsa_arena_granularity", "qsa_arena_destroy",
           "qsa_check_device_status", "qsa_selftest_wait_timeout", "qsa_pool_score_blocks",
           "qsa_append_score_blocks")
NOALLOC_SCRATCH_BYTES = 4 << 20


def lib() -> ctypes.CDLL:
    """Load libqsa.so (built by ``indexed_sparse_attention_gb300.build``)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                           "`python -m indexed_sparse_attention_gb300.build`")
    L = ctypes.CDLL(LIB_PATH)
    vp, i32, i64, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
    seqp = ctypes.POINTER(SeqDesc)
    L.qsa_status_string.argtypes = [i32]
    L.qsa_status_string.restype = ctypes.c_char_p
    L.qsa_last_error.restype = ctypes.c_char_p
    L.qsa_version.restype = i32
    L.qsa_wait_timeouts.restype = i32
    L.qsa_check_device_status.argtypes = [vp]
    L.qsa_selftest_wait_timeout.argtypes = [i32, vp]
    L.qsa_pool_index_keys.argtypes = [vp, i32, i64, i64, i64, vp, i64, vp]
    L.qsa_score_blocks.argtypes = [seqp, i32, vp, i32, vp, i64, vp, i64, vp, sz, vp]
    L.qsa_pool_score_blocks.argtypes = [seqp, i32, ctypes.POINTER(vp), i64, i32, vp, i32, vp, i64, vp, i64, vp, sz, vp]
    L.qsa_score_workspace_size.argtypes = [seqp, i32, i32]
    L.qsa_score_workspace_size.restype = sz
    L.qsa_select_workspace_size.argtypes = [seqp, i32, i32]
    L.qsa_select_workspace_size.restype = sz
    L.qsa_select_topk.argtypes = [seqp, i32, vp, i64, vp, i64, i32, vp, vp, vp, sz, vp]
    L.qsa_score_select_workspace_size.argtypes = [seqp, i32, i32]
    L.qsa_score_select_workspace_size.restype = sz
    L.qsa_score_select_topk.argtypes = [seqp, i32, vp, i32, vp, i64, i32, vp, vp, vp, sz, vp]
    L.qsa_attn_workspace_size.argtypes = [seqp, i32, ctypes.POINTER(AttnConfig), i32]
    L.qsa_attn_workspace_size.restype = sz
    L.qsa_sparse_attn.argtypes = [seqp, i32, ctypes.POINTER(AttnConfig), vp, vp, vp, i32, vp, vp, vp, sz, vp]
    L.qsa_sparse_attn_noalloc.argtypes = [seqp, i32, ctypes.POINTER(AttnConfig), vp, vp, vp, i32, vp, vp, vp]
    L.qsa_lse_merge.argtypes = [vp, vp, i32, i64, i32, vp, i32, vp, vp]
    L.qsa_append_tokens.argtypes = [seqp, ctypes.POINTER(AttnConfig), vp, vp, vp, vp, i64, i32, vp]
    L.qsa_append_score_blocks.argtypes = [seqp, ctypes.POINTER(AttnConfig), vp, vp, vp, vp, i64, i32, vp, i32, vp, i64,
                                          vp, i64, vp, sz, vp]
    u64 = ctypes.c_uint64
    L.qsa_arena_create.argtypes = [i32, u64, ctypes.POINTER(vp)]
    L.qsa_arena_ensure.argtypes = [vp, u64]
    L.qsa_arena_destroy.argtypes = [vp]
    L.qsa_arena_base.argtypes = [vp]
    L.qsa_arena_base.restype = vp
    for name in ("qsa_arena_mapped", "qsa_arena_reserved", "qsa_arena_granularity"):
        getattr(L, name).argtypes = [vp]
        getattr(L, name).restype = u64
    L.qsa_score_select_blocked_workspace_size.argtypes = [seqp, i32, i32, i32]
    L.qsa_score_select_blocked_workspace_size.restype = sz
    L.qsa_score_select_topk_blocked.argtypes = [seqp, i32, vp, i32, i32, i32, vp, vp, vp, sz, vp]
    for name in ("qsa_pool_index_keys", "qsa_score_blocks", "qsa_select_topk", "qsa_score_select_topk",
                 "qsa_sparse_attn", "qsa_sparse_attn_noalloc", "qsa_lse_merge", "qsa_score_select_topk_blocked",
                 "qsa_append_tokens", "qsa_arena_create", "qsa_arena_ensure", "qsa_arena_destroy"):
        getattr(L, name).restype = i32
    _lib = L
    return L


def wait_timeouts() -> int:
    """Device-side barrier waits that gave up (0 in normal operation)."""
    return int(lib().qsa_wait_timeouts())


def check_device_status(stream=None) -> tuple[int, str]:
    """qsa_check_device_status: (status, reason) for the device-side checks
    since the previous call -- 0, ERR_TIMEOUT or ERR_DEVICE_CHECK."""
    st = int(lib().qsa_check_device_status(_stream(stream)))
    return st, (lib().qsa_last_error().decode() if st else "")


def selftest_wait_timeout(limit_us: int, stream=None):
    """Launch one bounded wait that nothing completes (a test of the
    timeout reporting)."""
    _check("qsa_selftest_wait_timeout", lib().qsa_selftest_wait_timeout(int(limit_us), _stream(stream)))


def _check(fn: str, status: int):
    if status != 0:
        raise QSAError(fn, status, lib().qsa_last_error().decode())


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return F32
    if t.dtype == torch.bfloat16:
        return BF16
    if t.dtype in (torch.float8_e4m3fn, torch.uint8):   # E4M3 codes
        return FP8
    if t.dtype == torch.int8:                            # Q8_0 codes
        return Q8
    raise TypeError(f"unsupported dtype {t.dtype}")


def _stream(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _ptr(t):
    return None if t is None else t.data_ptr()


@dataclasses.dataclass
class Segment:
    """A contiguous run of one sequence's K/V cache: k, v are [Hkv, n, D]
    views (channel stride 1) holding absolute tokens first_token .. +n-1.
    Quantized state: for fp8, k and v hold E4M3 codes (float8_e4m3fn or
    uint8) and kv_scale is an [Hkv, n, 2] float16 view of the (K, V) scale
    pairs; for q8 (Q8_0), k and v hold int8 codes and kv_scale is an
    [Hkv, n, 2 * D / 32] float16 view of the K then V block scales."""
    k: torch.Tensor
    v: torch.Tensor
    first_token: int = 0
    kv_scale: torch.Tensor | None = None


@dataclasses.dataclass
class Seq:
    """One sequence of a call.  Its n_rows query rows are its last tokens:
    row j sits at absolute position n_tokens - n_rows + j.  Nothing past
    n_tokens is read, so rows elsewhere in a longer cache take n_tokens =
    their last position + 1, and scattered rows take one Seq per run of
    consecutive positions over the same tensors."""
    n_tokens: int
    n_rows: int
    pooled: torch.Tensor | None = None       # [>= n_tokens // 4, >= 128] f32
    segments: Sequence[Segment] = ()
    idx_keys: torch.Tensor | None = None     # [>= n_tokens, 128] index keys (for pooling)

    @property
    def row_pos(self) -> list[int]:
        return [self.n_tokens - self.n_rows + j for j in range(self.n_rows)]


def make_seq_array(seqs: Sequence[Seq]):
    """Marshal Seq objects into the C descriptor array (host memory)."""
    arr = (SeqDesc * len(seqs))()
    for i, s in enumerate(seqs):
        d = arr[i]
        d.n_tokens = int(s.n_tokens)
        d.n_rows = int(s.n_rows)
        d.n_segments = len(s.segments)
        if len(s.segments) > MAX_SEGMENTS:
            raise ValueError(f"at most {MAX_SEGMENTS} segments per sequence")
        if s.pooled is not None:
            if s.pooled.dtype != torch.float32 or s.pooled.stride(-1) != 1:
                raise TypeError("pooled keys must be f32 with unit channel stride")
            d.pooled = s.pooled.data_ptr()
            d.pooled_stride = s.pooled.stride(0)
        for j, g in enumerate(s.segments):
            if g.k.stride(-1) != 1 or g.v.stride(-1) != 1 or g.k.stride() != g.v.stride():
                raise TypeError("segment k/v need unit channel stride and equal strides")
            sg = d.segments[j]
            sg.k, sg.v = g.k.data_ptr(), g.v.data_ptr()
            sg.first_token = int(g.first_token)
            sg.n_tokens = int(g.k.shape[1])
            sg.head_stride, sg.tok_stride = int(g.k.stride(0)), int(g.k.stride(1))
            if g.kv_scale is not None:
                ks = g.kv_scale
                rec = 2 if g.k.dtype != torch.int8 else 2 * g.k.shape[-1] // 32   # f16 per scale record
                if (ks.dtype != torch.float16 or ks.shape[-1] != rec or ks.stride(-1) != 1
                        or ks.stride(0) % rec or ks.stride(1) % rec):
                    raise TypeError(f"kv_scale must be a float16 [Hkv, n, {rec}] view of whole scale records")
                sg.kv_scale = ks.data_ptr()
                sg.scale_head_stride, sg.scale_tok_stride = int(ks.stride(0)) // rec, int(ks.stride(1)) // rec
    return arr


# ---------------------------------------------------------------------- the five steps

def pool_index_keys(idx_keys: torch.Tensor, pooled: torch.Tensor, first_block: int, n_blocks: int, stream=None):
    """Step 1: pooled[b] = mean of index keys 4b..4b+3 for the listed blocks."""
    _check("qsa_pool_index_keys", lib().qsa_pool_index_keys(
        idx_keys.data_ptr(), _dtype_code(idx_keys), idx_keys.stride(0), int(first_block), int(n_blocks),
        pooled.data_ptr(), pooled.stride(0), _stream(stream)))


def n_groups(n_tokens: int) -> int:
    """Groups of SCORE_GROUP blocks covering the complete blocks of n_tokens."""
    return (n_tokens // 4 + SCORE_GROUP - 1) // SCORE_GROUP


def score_workspace_size(seqs, q_idx: torch.Tensor, seq_array=None) -> int:
    arr = seq_array if seq_array is not None else make_seq_array(seqs)
    return int(lib().qsa_score_workspace_size(arr, len(arr), _dtype_code(q_idx)))


def score_blocks(seqs, q_idx: torch.Tensor, scores: torch.Tensor, stream=None, seq_array=None,
                 group_max: torch.Tensor | None = None, workspace: torch.Tensor | None = None):
    """Step 2: scores[r, b] for every complete block row r sees; with
    group_max, also each row's maximum over every group of 16 blocks.  A
    workspace is allocated when the call has a tensor-core (prefill) part and
    none is given."""
    arr = seq_array if seq_array is not None else make_seq_array(seqs)
    if workspace is None:
        need = score_workspace_size(None, q_idx, seq_array=arr)
        if need:
            workspace = torch.empty(need, dtype=torch.uint8, device=scores.device)
    _check("qsa_score_blocks", lib().qsa_score_blocks(
        arr, len(arr), q_idx.data_ptr(), _dtype_code(q_idx), scores.data_ptr(), scores.stride(0),
        _ptr(group_max), 0 if group_max is None else group_max.stride(0), _ptr(workspace),
        0 if workspace is None else workspace.numel(), _stream(stream)))


def _idx_key_array(seqs):
    """(host pointer array, token stride, dtype code) of the sequences' index
    keys for qsa_pool_score_blocks, or None when they are missing or differ
    in dtype or stride."""
    keys = [sq.idx_keys for sq in seqs]
    if not keys or any(k is None for k in keys) or len({(k.dtype, k.stride(0)) for k in keys}) != 1:
        return None
    return (ctypes.c_void_p * len(keys))(*[k.data_ptr() for k in keys]), keys[0].stride(0), _dtype_code(keys[0])


def pool_score_blocks(seqs, q_idx: torch.Tensor, scores: torch.Tensor, stream=None, seq_array=None,
                      group_max: torch.Tensor | None = None, workspace: torch.Tensor | None = None, idx_array=None):
    """Steps 1 and 2 in one call: pools the blocks each sequence's rows
    complete (from its idx_keys into its pooled keys) and scores every visible
    block, in one launch on the few-row path."""
    arr = seq_array if seq_array is not None else make_seq_array(seqs)
    ia = idx_array if idx_array is not None else _idx_key_array(seqs)
    if ia is None:
        raise ValueError("pool_score_blocks: every sequence needs index keys of one dtype and stride")
    if workspace is None:
        need = score_workspace_size(None, q_idx, seq_array=arr)
        if need:
            workspace = torch.empty(need, dtype=torch.uint8, device=scores.device)
    _check("qsa_pool_score_blocks", lib().qsa_pool_score_blocks(
        arr, len(arr), ia[0], ia[1], ia[2], q_idx.data_ptr(), _dtype_code(q_idx), scores.data_ptr(),
        scores.stride(0), _ptr(group_max), 0 if group_max is None else group_max.stride(0), _ptr(workspace),
        0 if workspace is None else workspace.numel(), _stream(stream)))


def select_topk(seqs, scores: torch.Tensor, sel: torch.Tensor, cnt: torch.Tensor, top_k: int = TOP_K,
                workspace: torch.Tensor | None = None, stream=None, seq_array=None,
                group_max: torch.Tensor | None = None):
    """Step 3: the top_k best blocks per row, ascending ids, -1 padded.
    group_max: the group maxima score_blocks wrote for these scores, or None."""
    arr = seq_array if seq_array is not None else make_seq_array(seqs)
    need = lib().qsa_select_workspace_size(arr, len(arr), top_k)
    if need and workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=scores.device)
    _check("qsa_select_topk", lib().qsa_select_topk(
        arr, len(arr), scores.data_ptr(), scores.stride(0), _ptr(group_max),
        0 if group_max is None else group_max.stride(0), int(top_k), sel.data_ptr(), cnt.data_ptr(),
        _ptr(workspace), 0 if workspace is None else workspace.numel(), _stream(stream)))


def score_select_topk(seqs, q_idx: torch.Tensor, scores: torch.Tensor, sel: torch.Tensor, cnt: torch.Tensor,
                      top_k: int = TOP_K, workspace: torch.Tensor | None = None, stream=None, seq_array=None):
    """Steps 2 and 3 in one call; the workspace holds the group maxima."""
    arr = seq_array if seq_array is not None else make_seq_array(seqs)
    need = lib().qsa_score_select_workspace_size(arr, len(arr), top_k)
    if need and workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=scores.device)
    _check("qsa_score_select_topk", lib().qsa_score_select_topk(
        arr, len(arr), q_idx.data_ptr(), _dtype_code(q_idx), scores.data_ptr(), scores.stride(0), int(top_k),
        sel.data_ptr(), cnt.data_ptr(), _ptr(workspace), 0 if workspace is None else workspace.numel(),
        _stream(stream)))


def append_tokens(seq: Seq, k_new: torch.Tensor, v_new: torch.Tensor, idx_new: torch.Tensor, stream=None,
                  cfg=None):
    """Write the seq.n_rows newest tokens' K/V ([Hkv, n, D]) and index keys
    ([n, 128]) into seq's segments and seq.idx_keys, and pool the blocks they
    complete into seq.pooled, in one launch."""
    if not (k_new.is_contiguous() and v_new.is_contiguous() and idx_new.is_contiguous()):
        raise ValueError("append_tokens: k_new, v_new and idx_new must be contiguous")
    arr = make_seq_array([seq])
    if cfg is None:   # only the KV heads, head_dim and the caches' dtype matter here
        kvd = _kv_dtype([seq])
        kvd = _dtype_code(k_new) if kvd is None else kvd
        cfg = AttnConfig(k_new.shape[0], k_new.shape[0], k_new.shape[2], BF16 if kvd in (FP8, Q8) else kvd, kvd, F32,
                         0.0, 0)
    idxk = seq.idx_keys
    _check("qsa_append_tokens", lib().qsa_append_tokens(
        arr, ctypes.byref(cfg), k_new.data_ptr(), v_new.data_ptr(), idx_new.data_ptr(), idxk.data_ptr(),
        idxk.stride(0), _dtype_code(idxk), _stream(stream)))


def append_score_blocks(seq: Seq, k_new: torch.Tensor, v_new: torch.Tensor, idx_new: torch.Tensor,
                        q_idx: torch.Tensor, scores: torch.Tensor, stream=None, cfg=None,
                        group_max: torch.Tensor | None = None, workspace: torch.Tensor | None = None, seq_array=None):
    """append_tokens and the scoring of every visible block (score_blocks)
    in one call for one sequence: one launch on the few-row path."""
    if not (k_new.is_contiguous() and v_new.is_contiguous() and idx_new.is_contiguous()):
        raise ValueError("append_score_blocks: k_new, v_new and idx_new must be contiguous")
    arr = seq_array if seq_array is not None else make_seq_array([seq])
    if cfg is None:
        kvd = _kv_dtype([seq])
        kvd = _dtype_code(k_new) if kvd is None else kvd
        cfg = AttnConfig(k_new.shape[0], k_new.shape[0], k_new.shape[2], BF16 if kvd in (FP8, Q8) else kvd, kvd, F32,
                         0.0, 0)
    if workspace is None:
        need = score_workspace_size(None, q_idx, seq_array=arr)
        if need:
            workspace = torch.empty(need, dtype=torch.uint8, device=scores.device)
    idxk = seq.idx_keys
    _check("qsa_append_score_blocks", lib().qsa_append_score_blocks(
        arr, ctypes.byref(cfg), k_new.data_ptr(), v_new.data_ptr(), idx_new.data_ptr(), idxk.data_ptr(),
        idxk.stride(0), _dtype_code(idxk), q_idx.data_ptr(), _dtype_code(q_idx), scores.data_ptr(), scores.stride(0),
        _ptr(group_max), 0 if group_max is None else group_max.stride(0), _ptr(workspace),
        0 if workspace is None else workspace.numel(), _stream(stream)))


class _DevicePtr:
    """A device byte range exposed through __cuda_array_interface__ (no ownership)."""

    def __init__(self, ptr: int, n_bytes: int):
        self.__cuda_array_interface__ = {"shape": (n_bytes,), "typestr": "|u1", "data": (ptr, False), "version": 3}


class Arena:
    """Demand-mapped device memory with one stable base pointer: reserve once,
    map more physical memory with ensure() as the cache grows.  Views from
    tensor() do not own the memory; the arena must outlive them."""

    def __init__(self, reserve_bytes: int, device: int | None = None):
        self.device = torch.cuda.current_device() if device is None else int(device)
        h = ctypes.c_void_p()
        _check("qsa_arena_create", lib().qsa_arena_create(self.device, int(reserve_bytes), ctypes.byref(h)))
        self._h = h.value

    def ensure(self, n_bytes: int):
        _check("qsa_arena_ensure", lib().qsa_arena_ensure(self._h, int(n_bytes)))

    @property
    def base(self) -> int:
        return int(lib().qsa_arena_base(self._h) or 0)

    @property
    def mapped(self) -> int:
        return int(lib().qsa_arena_mapped(self._h))

    @property
    def reserved(self) -> int:
        return int(lib().qsa_arena_reserved(self._h))

    @property
    def granularity(self) -> int:
        return int(lib().qsa_arena_granularity(self._h))

    def tensor(self, offset: int, shape, dtype) -> torch.Tensor:
        """A view of [offset, offset + bytes) (mapped already) as a tensor."""
        es = torch.empty(0, dtype=dtype).element_size()
        n = es
        for d in shape:
            n *= int(d)
        if offset < 0 or offset % 16 or offset + n > self.mapped:
            raise ValueError("arena view outside the mapped, 16-byte-aligned range")
        raw = torch.as_tensor(_DevicePtr(self.base + offset, n), device=f"cuda:{self.device}")
        return raw.view(dtype).view(tuple(shape))

    def destroy(self):
        if getattr(self, "_h", None):
            _check("qsa_arena_destroy", lib().qsa_arena_destroy(self._h))
            self._h = None

    def __del__(self):
        try:
            self.destroy()
        except Exception:
            pass


def score_select_blocked_workspace_size(seqs, top_k: int = TOP_K, block_keys: int = 4096, seq_array=None) -> int:
    arr = seq_array if seq_array is not None else make_seq_array(seqs)
    return int(lib().qsa_score_select_blocked_workspace_size(arr, len(arr), int(top_k), int(block_keys)))


def score_select_topk_blocked(seqs, q_idx: torch.Tensor, sel: torch.Tensor, cnt: torch.Tensor, top_k: int = TOP_K,
                              block_keys: int = 4096, workspace: torch.Tensor | None = None, stream=None,
                              seq_array=None):
    """Steps 2 and 3 over key-axis chunks of block_keys blocks (no score buffer)."""
    arr = seq_array if seq_array is not None else make_seq_array(seqs)
    need = score_select_blocked_workspace_size(None, top_k, block_keys, seq_array=arr)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q_idx.device)
    _check("qsa_score_select_topk_blocked", lib().qsa_score_select_topk_blocked(
        arr, len(arr), q_idx.data_ptr(), _dtype_code(q_idx), int(top_k), int(block_keys), sel.data_ptr(),
        cnt.data_ptr(), workspace.data_ptr(), workspace.numel(), _stream(stream)))


def _kv_dtype(seqs):
    """The K/V dtype code of the first segment (None without segments)."""
    for sq in seqs or ():
        for g in sq.segments:
            return _dtype_code(g.k)
    return None


def attn_config(q: torch.Tensor, n_kv_heads: int, out_dtype=None, scale: float = 0.0, n_splits: int = 0,
                kv_dtype: int | None = None):
    cfg = AttnConfig()
    cfg.n_q_heads, cfg.head_dim = q.shape[1], q.shape[2]
    cfg.n_kv_heads = n_kv_heads
    cfg.q_dtype = _dtype_code(q)
    cfg.kv_dtype = cfg.q_dtype if kv_dtype is None else kv_dtype
    cfg.out_dtype = _dtype_code(torch.empty(0, dtype=out_dtype)) if out_dtype is not None else F32
    cfg.scale = float(scale)
    cfg.n_splits = int(n_splits)
    return cfg


def attn_workspace_size(seqs, cfg: AttnConfig, sel_ld: int, seq_array=None) -> int:
    arr = seq_array if seq_array is not None else make_seq_array(seqs)
    return int(lib().qsa_attn_workspace_size(arr, len(arr), ctypes.byref(cfg), int(sel_ld)))


def sparse_attn(seqs, q: torch.Tensor, sel: torch.Tensor, cnt: torch.Tensor, out: torch.Tensor,
                lse: torch.Tensor | None = None, *, n_kv_heads: int = 2, scale: float = 0.0, n_splits: int = 0,
                workspace: torch.Tensor | None = None, stream=None, seq_array=None, cfg: AttnConfig | None = None):
    """Step 4 (+ the internal step-5 merge of its splits)."""
    arr = seq_array if seq_array is not None else make_seq_array(seqs)
    if cfg is None:
        cfg = attn_config(q, n_kv_heads, out.dtype, scale, n_splits, kv_dtype=_kv_dtype(seqs))
    need = lib().qsa_attn_workspace_size(arr, len(arr), ctypes.byref(cfg), sel.stride(0))
    if need and workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    _check("qsa_sparse_attn", lib().qsa_sparse_attn(
        arr, len(arr), ctypes.byref(cfg), q.data_ptr(), sel.data_ptr(), cnt.data_ptr(), sel.stride(0),
        out.data_ptr(), _ptr(lse), _ptr(workspace), 0 if workspace is None else workspace.numel(),
        _stream(stream)))


def sparse_attn_noalloc(seqs, q: torch.Tensor, sel: torch.Tensor, cnt: torch.Tensor, out: torch.Tensor,
                        lse: torch.Tensor | None = None, *, n_kv_heads: int = 2, scale: float = 0.0,
                        n_splits: int = 0, stream=None, seq_array=None, cfg: AttnConfig | None = None):
    """Step 4 for callers that cannot provide device scratch: the library's
    own static scratch array is used (see qsa_sparse_attn_noalloc in qsa.h)."""
    arr = seq_array if seq_array is not None else make_seq_array(seqs)
    if cfg is None:
        cfg = attn_config(q, n_kv_heads, out.dtype, scale, n_splits, kv_dtype=_kv_dtype(seqs))
    _check("qsa_sparse_attn_noalloc", lib().qsa_sparse_attn_noalloc(
        arr, len(arr), ctypes.byref(cfg), q.data_ptr(), sel.data_ptr(), cnt.data_ptr(), sel.stride(0),
        out.data_ptr(), _ptr(lse), _stream(stream)))


def lse_merge(o_parts: torch.Tensor, lse_parts: torch.Tensor, out: torch.Tensor,
              lse_out: torch.Tensor | None = None, stream=None):
    """Step 5: merge [S, R, D] partials by their log-sum-exp into out [R, D]."""
    S, R, D = o_parts.shape
    _check("qsa_lse_merge", lib().qsa_lse_merge(
        o_parts.data_ptr(), lse_parts.data_ptr(), S, R, D, out.data_ptr(), _dtype_code(out), _ptr(lse_out),
        _stream(stream)))


def n_pooled_slots(n_tokens: int) -> int:
    """Pooled-key rows a cache of n_tokens needs (one per started block)."""
    return (int(n_tokens) + 3) // 4


def score_scale() -> float:
    return 1.0 / math.sqrt(INDEX_DIM)


class LayerStep:
    """Preallocated buffers and descriptors for one QSA layer step of a batch
    of sequences, so the same step can be replayed (or captured in a CUDA
    graph) without re-marshalling.  Plumbing only: every step is a library
    call.

    ``run`` pools the blocks that the rows' tokens completed (the blocks
    ending at positions L - n_rows .. L - 1), scores every visible block,
    selects the top_k per row and attends over the selection.
    """

    def __init__(self, seqs: Sequence[Seq], q_idx: torch.Tensor, q: torch.Tensor, *, n_kv_heads: int = 2,
                 top_k: int = TOP_K, out_dtype=torch.float32, n_splits: int = 0, scale: float = 0.0):
        self.seqs = list(seqs)
        self.q_idx, self.q = q_idx, q
        self.top_k = int(top_k)
        dev = q.device
        rows = sum(s.n_rows for s in self.seqs)
        self.ld = max(1, max(s.n_tokens // 4 for s in self.seqs))
        self.ld = (self.ld + 3) // 4 * 4
        self.arr = make_seq_array(self.seqs)
        self.cfg = attn_config(q, n_kv_heads, out_dtype, scale, n_splits, kv_dtype=_kv_dtype(self.seqs))
        self.scores = torch.empty((rows, self.ld), dtype=torch.float32, device=dev)
        gld = max(1, max(n_groups(s.n_tokens) for s in self.seqs))
        self.group_max = torch.empty((rows, (gld + 3) // 4 * 4), dtype=torch.float32, device=dev)
        self.sel = torch.empty((rows, self.top_k), dtype=torch.int32, device=dev)
        self.cnt = torch.empty((rows,), dtype=torch.int32, device=dev)
        self.out = torch.empty((rows, q.shape[1], q.shape[2]), dtype=out_dtype, device=dev)
        self.lse = torch.empty((rows, q.shape[1]), dtype=torch.float32, device=dev)
        score_ws = score_workspace_size(None, q_idx, seq_array=self.arr)
        self.score_ws = torch.empty(max(score_ws, 16), dtype=torch.uint8, device=dev) if score_ws else None
        sel_ws = int(lib().qsa_score_select_workspace_size(self.arr, len(self.arr), self.top_k))
        attn_ws = attn_workspace_size(None, self.cfg, self.top_k, seq_array=self.arr)
        # Selection scratch: zero-filled once; every call leaves it zeroed.
        self.sel_ws = torch.empty(max(sel_ws, 16), dtype=torch.uint8, device=dev)
        self.ws = torch.empty(max(attn_ws, 16), dtype=torch.uint8, device=dev)
        # Blocks completed by each sequence's new rows: [first, last] of nb(p) over its rows.
        self.pool_jobs = []
        for s in self.seqs:
            if s.idx_keys is None or s.pooled is None:
                continue
            b0 = (s.n_tokens - s.n_rows) // 4
            b1 = s.n_tokens // 4
            if b1 > b0:
                self.pool_jobs.append((s.idx_keys, s.pooled, b0, b1 - b0))
        # Steps 1 and 2 in one call when every sequence has index keys and pooled keys.
        self.idx_array = _idx_key_array(self.seqs) if all(s.pooled is not None for s in self.seqs) else None

    def pool(self, stream=None):
        for idxk, pooled, b0, n in self.pool_jobs:
            pool_index_keys(idxk, pooled, b0, n, stream)

    def score(self, stream=None):
        score_blocks(None, self.q_idx, self.scores, stream, seq_array=self.arr, group_max=self.group_max,
                     workspace=self.score_ws)

    def pool_score(self, stream=None):
        """pool() then score(), as one call (one launch on the few-row path)."""
        if self.idx_array is None:
            self.pool(stream)
            self.score(stream)
            return
        pool_score_blocks(None, self.q_idx, self.scores, stream, seq_array=self.arr, group_max=self.group_max,
                          workspace=self.score_ws, idx_array=self.idx_array)

    def select(self, stream=None):
        select_topk(None, self.scores, self.sel, self.cnt, self.top_k, None, stream, seq_array=self.arr,
                    group_max=self.group_max)

    def score_select(self, stream=None):
        score_select_topk(None, self.q_idx, self.scores, self.sel, self.cnt, self.top_k, self.sel_ws, stream,
                          seq_array=self.arr)

    def attend(self, stream=None):
        sparse_attn(None, self.q, self.sel, self.cnt, self.out, self.lse, workspace=self.ws, stream=stream,
                    seq_array=self.arr, cfg=self.cfg)

    def append(self, new_tokens, stream=None):
        """Append each sequence's n_rows newest tokens (a (k_new, v_new,
        idx_new) triple per sequence) and pool the blocks they complete:
        replaces pool() when the caller hands the new tokens to the library."""
        for sq, (k_new, v_new, idx_new) in zip(self.seqs, new_tokens):
            append_tokens(sq, k_new, v_new, idx_new, stream, cfg=self.cfg)

    def append_score(self, new_tokens, stream=None):
        """append() then score() as one call (one launch on the few-row
        path); one sequence."""
        if len(self.seqs) != 1:
            self.append(new_tokens, stream)
            self.score(stream)
            return
        k_new, v_new, idx_new = new_tokens[0]
        append_score_blocks(self.seqs[0], k_new, v_new, idx_new, self.q_idx, self.scores, stream, cfg=self.cfg,
                            group_max=self.group_max, workspace=self.score_ws, seq_array=self.arr)

    def run(self, stream=None, new_tokens=None):
        """One layer step: pool (or append new_tokens and pool), score,
        select, attend (an NVTX range "qsa.layer_step" around the calls)."""
        torch.cuda.nvtx.range_push("qsa.layer_step")
        try:
            if new_tokens is None:
                self.pool_score(stream)
            else:
                self.append_score(new_tokens, stream)
            self.select(stream)
            self.attend(stream)
        finally:
            torch.cuda.nvtx.range_pop()
        return self.out, self.lse
