"""fp64 CPU oracle for one QSA layer step -- test infrastructure only.

Only the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` import this package.  The CUDA library neither imports nor links
it and the two share no code.

The arithmetic lives in ``qsa_oracle.c`` (plain C, IEEE fp64, no fast-math);
this module compiles it with gcc and wraps it with ctypes.  Inputs may be
numpy arrays or CPU torch tensors in fp32, bf16 or fp64; they are handed to C
in their stored format and widened exactly there.

Sources: hipfire, "QSA sparse attention and the VMM KV backend", sections 02
and 03 (steps 1-4), and MTPLX pull request #610, "How it works, in plain
terms" and "What changes" (step 5).  Each wrapper names the step it follows.
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "qsa_oracle.c")
_LIB_PATH = os.path.join(_HERE, "libqsa_oracle.so")
_lock = threading.Lock()
_lib = None

F32, BF16, F64 = 0, 1, 2

INDEX_DIM = 128          # width of one index key
INDEX_HEADS = 4          # index-query heads per query row
BLOCK_TOKENS = 4         # tokens pooled into one block key
TOP_K = 512              # block budget (2,048 tokens)
SCORE_SCALE = 1.0 / math.sqrt(128.0)


def build(force: bool = False) -> str:
    """Compile the C oracle into ``libqsa_oracle.so`` beside its source."""
    with _lock:
        if (not force and os.path.exists(_LIB_PATH)
                and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
            return _LIB_PATH
        tmp = _LIB_PATH + f".{os.getpid()}.tmp"
        cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-fno-fast-math",
               "-ffp-contract=off", _SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
        return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB_PATH)
        i64, i32, dbl, vp = ctypes.c_int64, ctypes.c_int, ctypes.c_double, ctypes.c_void_p
        lib.qsa_oracle_set_threads.argtypes = [i32]
        lib.qsa_oracle_set_threads.restype = i32
        lib.qsa_oracle_get_threads.restype = i32
        lib.qsa_oracle_visible_blocks.argtypes = [i64]
        lib.qsa_oracle_visible_blocks.restype = i64
        lib.qsa_oracle_tail_tokens.argtypes = [i64]
        lib.qsa_oracle_tail_tokens.restype = i64
        lib.qsa_oracle_pool.argtypes = [vp, i32, i64, i64, i64, i64, i64, vp]
        lib.qsa_oracle_pool.restype = i32
        lib.qsa_oracle_score.argtypes = [vp, i32, i64, i64, i64, vp, i64, vp, dbl, vp, i64]
        lib.qsa_oracle_score.restype = i32
        lib.qsa_oracle_select.argtypes = [vp, i64, i64, vp, i64, vp, vp, vp]
        lib.qsa_oracle_select.restype = i32
        lib.qsa_oracle_row_tokens.argtypes = [i64, vp, i32, vp, vp]
        lib.qsa_oracle_row_tokens.restype = i64
        lib.qsa_oracle_attn.argtypes = [vp, i32, i64, i64, i64, i64, vp, vp, i32, i64, vp, vp, vp,
                                        vp, i64, dbl, vp, vp]
        lib.qsa_oracle_attn.restype = i32
        lib.qsa_oracle_lse_merge.argtypes = [vp, vp, i64, i64, i64, vp, vp]
        lib.qsa_oracle_lse_merge.restype = i32
        lib.qsa_oracle_e4m3_decode.argtypes = [ctypes.c_uint8]
        lib.qsa_oracle_e4m3_decode.restype = dbl
        lib.qsa_oracle_e4m3_encode.argtypes = [dbl]
        lib.qsa_oracle_e4m3_encode.restype = ctypes.c_uint8
        lib.qsa_oracle_f16_decode.argtypes = [ctypes.c_uint16]
        lib.qsa_oracle_f16_decode.restype = dbl
        lib.qsa_oracle_f16_encode.argtypes = [dbl]
        lib.qsa_oracle_f16_encode.restype = ctypes.c_uint16
        lib.qsa_oracle_fp8_quantize.argtypes = [vp, i32, i64, i64, vp, vp]
        lib.qsa_oracle_fp8_quantize.restype = i32
        lib.qsa_oracle_fp8_dequantize.argtypes = [vp, vp, i64, i64, vp]
        lib.qsa_oracle_fp8_dequantize.restype = i32
        lib.qsa_oracle_q8_quantize.argtypes = [vp, i32, i64, i64, vp, vp]
        lib.qsa_oracle_q8_quantize.restype = i32
        lib.qsa_oracle_q8_dequantize.argtypes = [vp, vp, i64, i64, vp]
        lib.qsa_oracle_q8_dequantize.restype = i32
        _lib = lib
    return _lib


def set_threads(n: int) -> int:
    """Host threads the oracle's row loops may use; returns the value set."""
    return _load().qsa_oracle_set_threads(int(n))


def _stored(x):
    """(contiguous numpy array in stored format, dtype code) of an input."""
    try:
        import torch
        if isinstance(x, torch.Tensor):
            x = x.detach().cpu().contiguous()
            if x.dtype == torch.bfloat16:
                return x.view(torch.int16).numpy().view(np.uint16), BF16
            x = x.numpy()
    except ImportError:  # pragma: no cover
        pass
    x = np.ascontiguousarray(x)
    if x.dtype == np.float32:
        return x, F32
    if x.dtype == np.float64:
        return x, F64
    if x.dtype == np.uint16:          # raw bf16 bit patterns
        return x, BF16
    raise TypeError(f"oracle input dtype {x.dtype} not supported")


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def visible_blocks(p: int) -> int:
    """nb(p): complete blocks visible to a row at position p."""
    return int(_load().qsa_oracle_visible_blocks(int(p)))


def tail_tokens(p: int) -> int:
    """Tokens of the incomplete tail block visible to a row at position p."""
    return int(_load().qsa_oracle_tail_tokens(int(p)))


def pool(idxk, first_block: int = 0, n_blocks: int | None = None) -> np.ndarray:
    """Step 1: pooled block keys (mean of 4 index keys), fp64 [n_blocks, dim]."""
    a, code = _stored(idxk)
    n_tokens, dim = a.shape
    if n_blocks is None:
        n_blocks = n_tokens // BLOCK_TOKENS - first_block
    out = np.zeros((n_blocks, dim), dtype=np.float64)
    rc = _load().qsa_oracle_pool(_ptr(a), code, n_tokens, dim, dim, first_block, n_blocks, _ptr(out))
    if rc != 0:
        raise ValueError("pool: requested blocks are not complete")
    return out


def score(q_idx, pooled: np.ndarray, row_pos, scale: float = SCORE_SCALE, ld: int | None = None):
    """Step 2: fp64 block scores [M, ld]; -inf where b >= nb(p_r)."""
    q, qcode = _stored(q_idx)
    M, H, dim = q.shape
    pooled = np.ascontiguousarray(pooled, dtype=np.float64)
    pos = np.ascontiguousarray(np.asarray(row_pos, dtype=np.int64))
    if ld is None:
        ld = pooled.shape[0]
    out = np.empty((M, ld), dtype=np.float64)
    rc = _load().qsa_oracle_score(_ptr(q), qcode, M, H, dim, _ptr(pooled), pooled.shape[0], _ptr(pos),
                                  float(scale), _ptr(out), ld)
    if rc != 0:
        raise ValueError("score: a row sees more blocks than are pooled")
    return out


def select(scores: np.ndarray, row_pos, top_k: int = TOP_K):
    """Step 3: (sel [M, top_k] int32 ascending, -1 padded; cnt [M]; tau [M])."""
    s = np.ascontiguousarray(scores, dtype=np.float64)
    pos = np.ascontiguousarray(np.asarray(row_pos, dtype=np.int64))
    M, ld = s.shape
    sel = np.empty((M, top_k), dtype=np.int32)
    cnt = np.empty((M,), dtype=np.int32)
    tau = np.empty((M,), dtype=np.float64)
    rc = _load().qsa_oracle_select(_ptr(s), M, ld, _ptr(pos), top_k, _ptr(sel), _ptr(cnt), _ptr(tau))
    if rc != 0:
        raise ValueError("select: bad arguments")
    return sel, cnt, tau


def row_tokens(p: int, sel_row, cnt: int, visible=None) -> np.ndarray:
    """Token ids a row attends to: selected blocks' tokens plus its tail."""
    sel_row = np.ascontiguousarray(np.asarray(sel_row, dtype=np.int32))
    buf = np.empty((4 * max(int(cnt), 0) + 4,), dtype=np.int64)
    vis = None if visible is None else np.ascontiguousarray(visible, dtype=np.uint8)
    n = _load().qsa_oracle_row_tokens(int(p), _ptr(sel_row), int(cnt),
                                      None if vis is None else _ptr(vis), _ptr(buf))
    return buf[:n].copy()


def attn(q, k, v, row_pos, sel, cnt, scale: float | None = None, visible=None):
    """Step 4: (out [M, Hq, D] fp64, lse [M, Hq] fp64) over the selected rows.

    k and v are single buffers [Hkv, L, D]; ``visible`` ([L] bool) keeps only
    tokens some KV segment covers.
    """
    qa, qcode = _stored(q)
    ka, kcode = _stored(k)
    va, vcode = _stored(v)
    if kcode != vcode:
        raise TypeError("k and v must share a stored dtype")
    M, Hq, D = qa.shape
    Hkv, L, D2 = ka.shape
    if D2 != D or va.shape != ka.shape:
        raise ValueError("shape mismatch")
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    pos = np.ascontiguousarray(np.asarray(row_pos, dtype=np.int64))
    sel = np.ascontiguousarray(np.asarray(sel, dtype=np.int32))
    cnt = np.ascontiguousarray(np.asarray(cnt, dtype=np.int32))
    vis = None if visible is None else np.ascontiguousarray(visible, dtype=np.uint8)
    out = np.empty((M, Hq, D), dtype=np.float64)
    lse = np.empty((M, Hq), dtype=np.float64)
    rc = _load().qsa_oracle_attn(_ptr(qa), qcode, M, Hq, Hkv, D, _ptr(ka), _ptr(va), kcode, L,
                                 None if vis is None else _ptr(vis), _ptr(pos), _ptr(sel), _ptr(cnt),
                                 sel.shape[1], float(scale), _ptr(out), _ptr(lse))
    if rc != 0:
        raise ValueError("attn: bad arguments (row position or selected id out of range)")
    return out, lse


def lse_merge(o_parts, lse_parts):
    """Step 5: merge partials [S, R, D] / [S, R] by log-sum-exp."""
    o = np.ascontiguousarray(o_parts, dtype=np.float64)
    l = np.ascontiguousarray(lse_parts, dtype=np.float64)
    S, R, D = o.shape
    out = np.empty((R, D), dtype=np.float64)
    lse = np.empty((R,), dtype=np.float64)
    rc = _load().qsa_oracle_lse_merge(_ptr(o), _ptr(l), S, R, D, _ptr(out), _ptr(lse))
    if rc != 0:
        raise ValueError("lse_merge: bad arguments")
    return out, lse


def layer_step(q_idx, idxk, q, k, v, row_pos, top_k: int = TOP_K, scale: float | None = None,
               visible=None, pooled: np.ndarray | None = None):
    """Steps 1-4 for one sequence: returns a dict of every intermediate.

    ``pooled`` may carry block keys pooled earlier (state kept between
    steps); otherwise every complete block of ``idxk`` is pooled here.
    """
    if pooled is None:
        pooled = pool(idxk)
    s = score(q_idx, pooled, row_pos)
    sel, cnt, tau = select(s, row_pos, top_k)
    out, lse = attn(q, k, v, row_pos, sel, cnt, scale=scale, visible=visible)
    return {"pooled": pooled, "scores": s, "sel": sel, "cnt": cnt, "tau": tau, "out": out, "lse": lse}


# ---------------------------------------------------------------------- fp8 K/V state
# hipfire, "QSA sparse attention and the VMM KV backend", section 02, table
# "State formats": E4M3 K/V with an f16 scale per head and token (reading R9
# in qsa_oracle.c: how a row is written).

def e4m3_decode(code: int) -> float:
    return float(_load().qsa_oracle_e4m3_decode(int(code) & 0xFF))


def e4m3_encode(x: float) -> int:
    return int(_load().qsa_oracle_e4m3_encode(float(x)))


def f16_decode(bits: int) -> float:
    return float(_load().qsa_oracle_f16_decode(int(bits) & 0xFFFF))


def f16_encode(x: float) -> int:
    return int(_load().qsa_oracle_f16_encode(float(x)))


def fp8_quantize(x):
    """Rows [..., D] (fp32 / bf16 / fp64) -> (codes uint8 [..., D], f16 scale bits uint16 [...])."""
    a, code = _stored(x)
    D = a.shape[-1]
    rows = a.size // D
    codes = np.empty(a.shape, dtype=np.uint8)
    scales = np.empty(a.shape[:-1], dtype=np.uint16)
    _load().qsa_oracle_fp8_quantize(_ptr(a), code, rows, D, _ptr(codes), _ptr(scales))
    return codes, scales


def fp8_dequantize(codes, scales) -> np.ndarray:
    """(codes uint8 [..., D], f16 scale bits uint16 [...]) -> values fp64 [..., D] (exact)."""
    c = np.ascontiguousarray(np.asarray(codes, dtype=np.uint8))
    s_ = np.ascontiguousarray(np.asarray(scales, dtype=np.uint16))
    D = c.shape[-1]
    out = np.empty(c.shape, dtype=np.float64)
    _load().qsa_oracle_fp8_dequantize(_ptr(c), _ptr(s_), c.size // D, D, _ptr(out))
    return out


# ---------------------------------------------------------------------- q8 K/V state
# The same table: Q8_0 K/V -- blocks of 32 elements, an f16 scale and 32 int8
# codes each (reading R10 in qsa_oracle.c: how a block is written).

def q8_quantize(x):
    """Rows [..., D] -> (codes int8 [..., D], f16 scale bits uint16 [..., D // 32])."""
    a, code = _stored(x)
    D = a.shape[-1]
    rows = a.size // D
    codes = np.empty(a.shape, dtype=np.int8)
    scales = np.empty(a.shape[:-1] + (D // 32,), dtype=np.uint16)
    if _load().qsa_oracle_q8_quantize(_ptr(a), code, rows, D, _ptr(codes), _ptr(scales)) != 0:
        raise ValueError("q8_quantize: D must be a multiple of 32")
    return codes, scales


def q8_dequantize(codes, scales) -> np.ndarray:
    """(codes int8 [..., D], f16 scale bits [..., D // 32]) -> values fp64 [..., D] (exact)."""
    c = np.ascontiguousarray(np.asarray(codes, dtype=np.int8))
    s_ = np.ascontiguousarray(np.asarray(scales, dtype=np.uint16))
    D = c.shape[-1]
    out = np.empty(c.shape, dtype=np.float64)
    _load().qsa_oracle_q8_dequantize(_ptr(c), _ptr(s_), c.size // D, D, _ptr(out))
    return out
