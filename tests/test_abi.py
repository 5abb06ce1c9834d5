"""The C ABI without a GPU: the library loads, exports every declared entry
point, and rejects bad arguments on the host before any launch.

Device pointers below are fake aligned addresses: host-side checks never
dereference them, and every call here fails validation before it would
reach CUDA (or is a documented no-op).
"""
import ctypes
import os
import re

import pytest
import torch

import indexed_sparse_attention_gb300 as qsa
from indexed_sparse_attention_gb300 import build as qsa_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "qsa.h")

FAKE = 0x10000        # aligned, never dereferenced on the host
FAKE_MIS = 0x10004    # 4-byte aligned only


@pytest.fixture(scope="module")
def L():
    qsa_build.build()
    return qsa.lib()


def _declared():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[a-z_0-9]+\*?\s+\*?(qsa_[a-z_0-9]+)\(", text, re.M)))


def test_header_declares_the_five_steps():
    names = _declared()
    for n in ("qsa_pool_index_keys", "qsa_score_blocks", "qsa_select_topk", "qsa_sparse_attn", "qsa_lse_merge"):
        assert n in names


def test_every_declared_symbol_is_exported(L):
    for name in _declared():
        assert hasattr(L, name), name
    assert set(qsa.EXPORTS) <= set(_declared())


def test_status_strings_and_version(L):
    assert L.qsa_version() == 111
    for code, name in qsa.STATUS.items():
        assert L.qsa_status_string(code).decode() == name
    assert L.qsa_status_string(99).decode() == "QSA_ERR_UNKNOWN"


def test_selftest_wait_limits_checked_before_launch(L):
    for bad in (0, -3, 2_000_001):
        assert L.qsa_selftest_wait_timeout(bad, None) == 1
        assert "limit_us" in L.qsa_last_error().decode()


def _seq(n_tokens=4099, n_rows=4, pooled=FAKE, n_segments=1, segs=None):
    arr = (qsa.SeqDesc * 1)()
    d = arr[0]
    d.n_tokens, d.n_rows, d.n_segments = n_tokens, n_rows, n_segments
    d.pooled, d.pooled_stride = pooled, 128
    for j, (first, n) in enumerate(segs or [(0, n_tokens)]):
        s = d.segments[j]
        s.k, s.v, s.first_token, s.n_tokens = FAKE, FAKE, first, n
        s.head_stride, s.tok_stride = n * 256, 256
    return arr


def _cfg(**kw):
    c = qsa.AttnConfig()
    c.n_q_heads, c.n_kv_heads, c.head_dim = 24, 2, 256
    c.q_dtype = c.kv_dtype = qsa.BF16
    c.out_dtype = qsa.F32
    c.scale, c.n_splits = 0.0, 0
    for k, v in kw.items():
        setattr(c, k, v)
    return c


def test_pool_validation(L):
    assert L.qsa_pool_index_keys(FAKE, 7, 128, 0, 4, FAKE, 128, None) == 2
    assert L.qsa_pool_index_keys(FAKE, qsa.F32, 128, -1, 4, FAKE, 128, None) == 1
    assert L.qsa_pool_index_keys(FAKE, qsa.F32, 64, 0, 4, FAKE, 128, None) == 1
    assert L.qsa_pool_index_keys(FAKE_MIS, qsa.F32, 128, 0, 4, FAKE, 128, None) == 3
    assert L.qsa_pool_index_keys(FAKE, qsa.BF16, 132, 0, 4, FAKE, 128, None) == 3   # 264-byte rows
    assert L.qsa_pool_index_keys(None, qsa.F32, 128, 0, 4, FAKE, 128, None) == 1
    assert "null" in L.qsa_last_error().decode()
    assert L.qsa_pool_index_keys(None, qsa.F32, 128, 0, 0, None, 128, None) == 0     # empty range: no-op
    assert L.qsa_last_error().decode() == ""


def test_pool_score_validation(L):
    # Checks that run before any launch (a null key array, dtypes, strides,
    # a sequence that completes a block without keys).
    seq = _seq()
    keys = (ctypes.c_void_p * 1)(FAKE)
    none = (ctypes.c_void_p * 1)(None)
    mis = (ctypes.c_void_p * 1)(FAKE_MIS)
    args = (FAKE, qsa.BF16, FAKE, 1024, None, 0, None, 0, None)
    assert L.qsa_pool_score_blocks(seq, 1, None, 128, qsa.BF16, *args) == 1
    assert L.qsa_pool_score_blocks(seq, 1, keys, 128, 9, *args) == 2
    assert L.qsa_pool_score_blocks(seq, 1, keys, 64, qsa.BF16, *args) == 1
    assert L.qsa_pool_score_blocks(seq, 1, keys, 132, qsa.BF16, *args) == 3       # 264 bytes per token
    assert L.qsa_pool_score_blocks(seq, 1, none, 128, qsa.BF16, *args) == 1       # rows complete block 1,024
    assert L.qsa_pool_score_blocks(seq, 1, mis, 128, qsa.BF16, *args) == 3
    assert "qsa_pool_score_blocks" in L.qsa_last_error().decode()


def test_score_validation(L):
    seq = _seq()
    assert L.qsa_score_blocks(seq, 0, FAKE, qsa.BF16, FAKE, 1024, None, 0, None, 0, None) == 1
    assert L.qsa_score_blocks(seq, 1, FAKE, 9, FAKE, 1024, None, 0, None, 0, None) == 2
    assert L.qsa_score_blocks(seq, 1, FAKE, qsa.BF16, FAKE, 1023, None, 0, None, 0, None) == 1       # ld < 1,024 blocks
    assert L.qsa_score_blocks(seq, 1, FAKE_MIS, qsa.BF16, FAKE, 1024, None, 0, None, 0, None) == 3
    assert L.qsa_score_blocks(_seq(pooled=None), 1, FAKE, qsa.BF16, FAKE, 1024, None, 0, None, 0, None) == 1
    assert L.qsa_score_blocks(_seq(n_rows=5000), 1, FAKE, qsa.BF16, FAKE, 1024, None, 0, None, 0, None) == 1
    assert L.qsa_score_blocks(_seq(n_tokens=4 * (1 << 18) + 4), 1, FAKE, qsa.BF16, FAKE, 1 << 20, None, 0, None, 0, None) == 2


def test_group_max_validation(L):
    seq = _seq()   # 4,099 tokens: 1,024 blocks = 64 groups
    assert L.qsa_score_blocks(seq, 1, FAKE, qsa.BF16, FAKE, 1024, FAKE, 60, None, 0, None) == 1
    assert "group_ld" in L.qsa_last_error().decode()
    assert L.qsa_score_blocks(seq, 1, FAKE, qsa.BF16, FAKE, 1024, FAKE, 66, None, 0, None) == 3
    assert L.qsa_score_blocks(seq, 1, FAKE, qsa.BF16, FAKE, 1024, FAKE_MIS, 64, None, 0, None) == 3
    assert L.qsa_select_topk(seq, 1, FAKE, 1024, FAKE, 60, 512, FAKE, FAKE, None, 0, None) == 1
    assert L.qsa_select_topk(seq, 1, FAKE, 1024, FAKE_MIS, 64, 512, FAKE, FAKE, None, 0, None) == 3
    assert L.qsa_select_topk(seq, 1, FAKE, 1022, None, 0, 512, FAKE, FAKE, None, 0, None) == 3   # ld % 4
    assert L.qsa_score_select_workspace_size(seq, 1, 512) == 4 * 4 * 64
    assert L.qsa_score_select_topk(seq, 1, FAKE, qsa.BF16, FAKE, 1024, 512, FAKE, FAKE, FAKE, 1023, None) == 4


def test_select_validation(L):
    seq = _seq()
    assert L.qsa_select_workspace_size(seq, 1, 512) == 0
    assert L.qsa_select_topk(seq, 1, FAKE, 1024, None, 0, 0, FAKE, FAKE, None, 0, None) == 2
    assert L.qsa_select_topk(seq, 1, FAKE, 1024, None, 0, 2048, FAKE, FAKE, None, 0, None) == 2
    assert L.qsa_select_topk(seq, 1, FAKE, 1000, None, 0, 512, FAKE, FAKE, None, 0, None) == 1
    assert L.qsa_select_topk(seq, 1, FAKE, 1024, None, 0, 512, None, FAKE, None, 0, None) == 1


def test_attn_validation(L):
    seq = _seq()
    c = _cfg()
    assert L.qsa_sparse_attn(seq, 1, ctypes.byref(_cfg(head_dim=64)), FAKE, FAKE, FAKE, 512, FAKE, None, None, 0,
                             None) == 2
    assert L.qsa_sparse_attn(seq, 1, ctypes.byref(_cfg(n_q_heads=25)), FAKE, FAKE, FAKE, 512, FAKE, None, None,
                             0, None) == 1
    assert L.qsa_sparse_attn(seq, 1, ctypes.byref(_cfg(n_q_heads=34, n_kv_heads=2)), FAKE, FAKE, FAKE, 512, FAKE,
                             None, None, 0, None) == 2                                # 17 heads per KV head
    assert L.qsa_sparse_attn(seq, 1, ctypes.byref(_cfg(q_dtype=qsa.F32)), FAKE, FAKE, FAKE, 512, FAKE, None,
                             None, 0, None) == 2
    assert L.qsa_sparse_attn(_seq(n_segments=0), 1, ctypes.byref(c), FAKE, FAKE, FAKE, 512, FAKE, None, None, 0,
                             None) == 1
    assert L.qsa_sparse_attn(_seq(n_segments=2, segs=[(0, 3000), (2999, 1100)]), 1, ctypes.byref(c), FAKE, FAKE,
                             FAKE, 512, FAKE, None, None, 0, None) == 1             # overlapping segments
    assert "overlapping" in L.qsa_last_error().decode()
    assert L.qsa_sparse_attn(seq, 1, ctypes.byref(c), FAKE_MIS, FAKE, FAKE, 512, FAKE, None, None, 0, None) == 3
    # One split per (row, KV group) needs no scratch; several splits keep
    # their normalised partials and lse values in the workspace.
    assert L.qsa_attn_workspace_size(seq, 1, ctypes.byref(_cfg(n_splits=1)), 512) == 0
    c16 = _cfg(n_splits=16)
    need = L.qsa_attn_workspace_size(seq, 1, ctypes.byref(c16), 512)
    # (16 splits of 2,051 rows round to whole 32-row tiles: 13 splits of 160)
    assert need >= 13 * 4 * 24 * (256 + 1) * 4
    assert L.qsa_sparse_attn(seq, 1, ctypes.byref(c16), FAKE, FAKE, FAKE, 512, FAKE, None, FAKE, need - 1,
                             None) == 4
    assert L.qsa_sparse_attn(seq, 1, ctypes.byref(c16), FAKE, FAKE, FAKE, 512, FAKE, None, None, 0, None) == 4


def test_arena_validation(L):
    h = ctypes.c_void_p()
    assert L.qsa_arena_create(0, 1 << 20, None) == 1
    assert L.qsa_arena_create(-1, 1 << 20, ctypes.byref(h)) == 1
    assert L.qsa_arena_create(0, 0, ctypes.byref(h)) == 1
    assert L.qsa_arena_ensure(None, 16) == 1
    assert L.qsa_arena_destroy(None) == 0
    assert L.qsa_arena_base(None) is None and L.qsa_arena_mapped(None) == 0
    if not torch.cuda.is_available():
        # No GPU here: creation fails with a status and a reason, not a crash.
        assert L.qsa_arena_create(0, 1 << 20, ctypes.byref(h)) == 5
        assert L.qsa_last_error().decode().startswith("qsa_arena_create:")


def test_append_validation(L):
    c = qsa.AttnConfig(2, 2, 256, qsa.BF16, qsa.BF16, qsa.F32, 0.0, 0)
    seq = _seq(n_tokens=4099, n_rows=4)
    ok = lambda s, idx=FAKE, stride=128: L.qsa_append_tokens(s, ctypes.byref(c), FAKE, FAKE, FAKE, idx, stride,
                                                             qsa.BF16, None)
    assert ok(seq, idx=None) == 1                                       # null pointer
    assert ok(seq, stride=64) == 1                                      # index-key stride < 128
    assert ok(seq, idx=FAKE_MIS) == 3
    assert ok(_seq(n_tokens=4099, n_rows=4, segs=[(0, 4097)])) == 1     # tokens 4097, 4098 in no segment
    assert "no KV segment" in L.qsa_last_error().decode()
    assert ok(_seq(n_tokens=4099, n_rows=5000)) == 1                    # more new tokens than the cache


def test_append_score_validation(L):
    # The append's checks and the scoring's both run before anything is launched.
    c = qsa.AttnConfig(2, 2, 256, qsa.BF16, qsa.BF16, qsa.F32, 0.0, 0)
    seq = _seq(n_tokens=4099, n_rows=4)

    def call(s=seq, idx=FAKE, q=FAKE, scores=FAKE, ld=1028):
        return L.qsa_append_score_blocks(s, ctypes.byref(c), FAKE, FAKE, FAKE, idx, 128, qsa.BF16, q, qsa.BF16,
                                         scores, ld, None, 0, None, 0, None)
    assert call(idx=None) == 1                                              # append: null index keys
    assert call(_seq(n_tokens=4099, n_rows=4, segs=[(0, 4097)])) == 1        # append: token in no segment
    assert "no KV segment" in L.qsa_last_error().decode()
    assert call(q=None) == 1                                                # scoring: null index queries
    assert call(scores=FAKE_MIS) == 3                                       # scoring: misaligned scores
    assert call(ld=100) == 1                                                # scoring: ld below the blocks
    assert "qsa_append_score_blocks" in L.qsa_last_error().decode()


def test_blocked_score_select_validation(L):
    seq = _seq(n_tokens=40_000, n_rows=600)
    need = L.qsa_score_select_blocked_workspace_size(seq, 1, 512, 1024)
    assert need > 0
    # Flat in the context: the same rows at 10x the context need the same workspace.
    assert L.qsa_score_select_blocked_workspace_size(_seq(n_tokens=400_000, n_rows=600), 1, 512, 1024) == need
    args = lambda dt, k, bk, ws=need: (seq, 1, FAKE, dt, k, bk, FAKE, FAKE, FAKE, ws, None)
    assert L.qsa_score_select_topk_blocked(*args(qsa.F32, 512, 1024)) == 2       # bf16 queries only
    assert L.qsa_score_select_topk_blocked(*args(qsa.BF16, 512, 1000)) == 2      # not a multiple of 128
    assert L.qsa_score_select_topk_blocked(*args(qsa.BF16, 1024, 7424)) == 2     # top_k + block_keys > 8192
    assert L.qsa_score_select_topk_blocked(*args(qsa.BF16, 0, 1024)) == 2
    assert L.qsa_score_select_topk_blocked(*args(qsa.BF16, 512, 1024, need - 1)) == 4
    assert L.qsa_score_select_topk_blocked(seq, 1, FAKE, qsa.BF16, 512, 1024, None, FAKE, FAKE, need, None) == 1


def test_merge_validation(L):
    assert L.qsa_lse_merge(FAKE, FAKE, 0, 10, 256, FAKE, qsa.F32, None, None) == 1
    assert L.qsa_lse_merge(FAKE, FAKE, 2, 10, 6, FAKE, qsa.F32, None, None) == 2
    assert L.qsa_lse_merge(FAKE, FAKE, 2, 10, 256, FAKE, 5, None, None) == 2
    assert L.qsa_lse_merge(FAKE_MIS, FAKE, 2, 10, 256, FAKE, qsa.F32, None, None) == 3
    assert L.qsa_lse_merge(None, None, 2, 0, 256, None, qsa.F32, None, None) == 0   # no rows: no-op


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    monkeypatch.setattr(qsa, "_lib", None)
    monkeypatch.setattr(qsa, "LIB_PATH", str(tmp_path / "libqsa.so"))
    with pytest.raises(RuntimeError, match="missing"):
        qsa.lib()
