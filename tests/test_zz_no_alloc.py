"""qsa_sparse_attn_noalloc: attention for callers that cannot give the library
device memory (for example a framework whose pool owns every byte of device
memory, or a serving loop that must not call cudaMalloc because it can
synchronize the device).  The entry point uses a fixed scratch array inside
libqsa.so instead of a workspace; these checks call it through the C ABI and
compare it with qsa_sparse_attn, which takes a caller workspace, on two calls
in a row.

This file is collected last so that a run stopping at its first failure has
already run every other test; it also passes alone in a fresh process (its
first call is the one that looks up the scratch array on the device).
"""
import ctypes

import numpy as np
import pytest
import torch

import indexed_sparse_attention_gb300 as qsa
import oracle
from qsa_cases import ATTN_BF16_ABS, ATTN_BF16_REL, dev, to_np
from workloads import make_layer

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from indexed_sparse_attention_gb300 import build
    build.build()
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need CUDA")


def _selection(x):
    pooled = oracle.pool(x.idxk)
    s = oracle.score(x.q_idx, pooled, x.row_pos)
    return oracle.select(s, x.row_pos)


def _close(got, want_out, want_lse):
    out, lse = got
    err = np.abs(out.astype(np.float64) - want_out.astype(np.float64)).max()
    assert err <= ATTN_BF16_ABS and err <= ATTN_BF16_REL * np.abs(want_out).max(), err
    fin = np.isfinite(want_lse)
    assert np.array_equal(np.isfinite(lse), fin)
    assert np.abs(lse[fin] - want_lse[fin]).max() <= ATTN_BF16_ABS


@pytest.mark.parametrize("L,M,n_splits", [(9001, 4, 40), (65_536, 1, 0), (20_011, 2, 0)])
def test_noalloc_matches_workspace_entry_point(L, M, n_splits):
    x = make_layer(L=L, M=M, dtype=torch.bfloat16, seed=31, n_planted=64)
    sel, cnt = _selection(x)[:2]
    q, k, v = x.q.to(dev()), x.k.to(dev()), x.v.to(dev())
    seqs = qsa.make_seq_array([qsa.Seq(x.L, x.M, segments=[qsa.Segment(k, v, 0)])])
    seld, cntd = torch.from_numpy(sel).to(dev()), torch.from_numpy(cnt).to(dev())
    cfg = qsa.attn_config(q, 2, torch.float32, 0.0, n_splits)
    L_ = qsa.lib()
    need = L_.qsa_attn_workspace_size(seqs, 1, ctypes.byref(cfg), sel.shape[1])
    if n_splits:
        assert need > 0          # this case exercises the scratch the split merge needs
    stream = torch.cuda.current_stream().cuda_stream

    # The existing entry point, with a caller workspace (zero-filled once).
    ws = torch.zeros(max(need, 16), dtype=torch.uint8, device=dev())
    ref_out = torch.empty((M, 24, 256), device=dev())
    ref_lse = torch.empty((M, 24), device=dev())
    st = L_.qsa_sparse_attn(seqs, 1, ctypes.byref(cfg), q.data_ptr(), seld.data_ptr(), cntd.data_ptr(),
                            sel.shape[1], ref_out.data_ptr(), ref_lse.data_ptr(), ws.data_ptr(), ws.numel(), stream)
    assert st == 0, L_.qsa_last_error()
    torch.cuda.synchronize()
    want = (to_np(ref_out), to_np(ref_lse))

    # The allocation-free entry point, twice in a row: the second call finds
    # the scratch array as the first left it.
    for _ in range(2):
        out = torch.full((M, 24, 256), float("nan"), device=dev())
        lse = torch.full((M, 24), float("nan"), device=dev())
        st = L_.qsa_sparse_attn_noalloc(seqs, 1, ctypes.byref(cfg), q.data_ptr(), seld.data_ptr(), cntd.data_ptr(),
                                        sel.shape[1], out.data_ptr(), lse.data_ptr(), stream)
        assert st == 0, L_.qsa_last_error()
        torch.cuda.synchronize()
        _close((to_np(out), to_np(lse)), *want)


def test_noalloc_shapes_in_turn_leave_nothing_behind():
    """The shared array keeps the previous call's partials; a call with another
    shape or split count must not read them.  A 40-split call, a one-row
    65,536-token call with the library's own plan, then the 40-split call
    again, each against the workspace entry point."""
    L_ = qsa.lib()
    stream = torch.cuda.current_stream().cuda_stream
    for (L, M, n_splits) in ((9001, 4, 40), (65_536, 1, 0), (9001, 4, 40)):
        x = make_layer(L=L, M=M, dtype=torch.bfloat16, seed=37 + M, n_planted=64)
        sel, cnt = _selection(x)[:2]
        q, k, v = x.q.to(dev()), x.k.to(dev()), x.v.to(dev())
        seqs = qsa.make_seq_array([qsa.Seq(x.L, x.M, segments=[qsa.Segment(k, v, 0)])])
        seld, cntd = torch.from_numpy(sel).to(dev()), torch.from_numpy(cnt).to(dev())
        cfg = qsa.attn_config(q, 2, torch.float32, 0.0, n_splits)
        need = L_.qsa_attn_workspace_size(seqs, 1, ctypes.byref(cfg), sel.shape[1])
        ws = torch.zeros(max(need, 16), dtype=torch.uint8, device=dev())
        ref = [torch.empty((M, 24, 256), device=dev()), torch.empty((M, 24), device=dev())]
        got = [torch.full((M, 24, 256), float("nan"), device=dev()), torch.full((M, 24), float("nan"), device=dev())]
        assert L_.qsa_sparse_attn(seqs, 1, ctypes.byref(cfg), q.data_ptr(), seld.data_ptr(), cntd.data_ptr(),
                                  sel.shape[1], ref[0].data_ptr(), ref[1].data_ptr(), ws.data_ptr(), ws.numel(),
                                  stream) == 0, L_.qsa_last_error()
        assert L_.qsa_sparse_attn_noalloc(seqs, 1, ctypes.byref(cfg), q.data_ptr(), seld.data_ptr(), cntd.data_ptr(),
                                          sel.shape[1], got[0].data_ptr(), got[1].data_ptr(), stream) == 0, \
            L_.qsa_last_error()
        torch.cuda.synchronize()
        _close((to_np(got[0]), to_np(got[1])), to_np(ref[0]), to_np(ref[1]))


def test_noalloc_rejects_plans_beyond_its_scratch():
    # 2,048 prefill rows forced to 40 splits need far more than the built-in
    # 4 MiB; the call is refused on the host before any launch.
    arr = (qsa.SeqDesc * 1)()
    d = arr[0]
    d.n_tokens, d.n_rows, d.n_segments = 102_400, 2048, 1
    s = d.segments[0]
    s.k = s.v = 0x10000
    s.first_token, s.n_tokens, s.head_stride, s.tok_stride = 0, 102_400, 102_400 * 256, 256
    cfg = qsa.AttnConfig()
    cfg.n_q_heads, cfg.n_kv_heads, cfg.head_dim = 24, 2, 256
    cfg.q_dtype = cfg.kv_dtype = qsa.BF16
    cfg.out_dtype = qsa.F32
    cfg.scale, cfg.n_splits = 0.0, 40
    L_ = qsa.lib()
    assert L_.qsa_attn_workspace_size(arr, 1, ctypes.byref(cfg), 512) > qsa.NOALLOC_SCRATCH_BYTES
    st = L_.qsa_sparse_attn_noalloc(arr, 1, ctypes.byref(cfg), 0x10000, 0x10000, 0x10000, 512, 0x10000, None, None)
    assert st == 2 and "scratch" in L_.qsa_last_error().decode()
