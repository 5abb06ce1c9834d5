"""GPU parity at the workloads' full sizes: the 65,536-token decode (M = 1),
the 261,120-token verify (M = 4) -- over bf16, fp8 and q8 K/V state -- the
2,048-row prefill at a 100,352-token prefix (sampled rows), and the ragged
16-sequence segmented batch.  One layer each (layers are independent).
Tolerances as in qsa_cases."""
import os

import numpy as np
import pytest
import torch

import indexed_sparse_attention_gb300 as qsa
import oracle
from qsa_cases import (assert_attn_close, assert_scores_close, assert_selection_close, dev, pooled_buffer,
                       score_bound, to_np)
from workloads import make_layer, ragged_batch_spec, segment_cuts

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from indexed_sparse_attention_gb300 import build
    build.build()
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need CUDA")
    oracle.set_threads(len(os.sched_getaffinity(0)))
    yield
    oracle.set_threads(1)


def _gpu_step(x, segments=None):
    """Pool what earlier steps pooled, then run the whole step on the GPU."""
    pooled = pooled_buffer(x.L, dev())
    first_new = (x.L - x.M) // 4
    if first_new:
        qsa.pool_index_keys(x.idxk, pooled, 0, first_new)
    segs = segments if segments is not None else [qsa.Segment(x.k, x.v, 0)]
    step = qsa.LayerStep([qsa.Seq(x.L, x.M, pooled, segs, idx_keys=x.idxk)], x.q_idx, x.q)
    step.run()
    torch.cuda.synchronize()
    return step, pooled


def _host(x):
    return {k: getattr(x, k).cpu() for k in ("idxk", "q_idx", "q", "k", "v")}


@pytest.mark.parametrize("L,M", [(65_536, 1), (261_120, 4), (261_120, 8)])
def test_decode_and_verify_full_size(L, M):
    x = make_layer(L=L, M=M, dtype=torch.bfloat16, seed=0, n_planted=256, device=dev())
    step, _ = _gpu_step(x)
    h = _host(x)
    pooled_ref = oracle.pool(h["idxk"])
    s_ref = oracle.score(h["q_idx"], pooled_ref, x.row_pos)
    sel_ref, cnt_ref, tau = oracle.select(s_ref, x.row_pos)
    nb = s_ref.shape[1]
    assert_scores_close(to_np(step.scores)[:, :nb], s_ref, 2 * score_bound(h["q_idx"], pooled_ref, x.row_pos),
                        x.row_pos)
    sel, cnt = to_np(step.sel), to_np(step.cnt)
    assert_selection_close(sel, cnt, sel_ref, cnt_ref, tau, s_ref, x.row_pos)
    # The step's own output against the oracle on the same selection ...
    out_ref, lse_ref = oracle.attn(h["q"], h["k"], h["v"], x.row_pos, sel, cnt)
    assert_attn_close(to_np(step.out), to_np(step.lse), out_ref, lse_ref, True)
    # ... and attention given the oracle's selection.
    out = torch.empty_like(step.out)
    lse = torch.empty_like(step.lse)
    qsa.sparse_attn([qsa.Seq(L, M, segments=[qsa.Segment(x.k, x.v, 0)])], x.q,
                    torch.from_numpy(sel_ref).to(dev()), torch.from_numpy(cnt_ref).to(dev()), out, lse)
    torch.cuda.synchronize()
    out_ref2, lse_ref2 = oracle.attn(h["q"], h["k"], h["v"], x.row_pos, sel_ref, cnt_ref)
    assert_attn_close(to_np(out), to_np(lse), out_ref2, lse_ref2, True)
    # Every row attends 2,048 selected rows plus its tail.
    assert (cnt == 512).all()


@pytest.mark.parametrize("state", ["fp8", "q8"])
@pytest.mark.parametrize("L,M", [(65_536, 1), (261_120, 4)])
def test_decode_and_verify_full_size_quantized(L, M, state):
    # The quantized-state steps as the bench runs them: caches written by the
    # library's append of every token of the bf16 draw -- which must equal
    # the oracle's quantizer on the same draw -- then the whole step, against
    # the oracle's attention on the oracle's dequantized K/V.
    x = make_layer(L=L, M=M, dtype=torch.bfloat16, seed=0, n_planted=256, device=dev())
    D = x.k.shape[2]
    rec = 2 if state == "fp8" else 2 * D // 32
    kc = torch.zeros(x.k.shape, dtype=torch.uint8 if state == "fp8" else torch.int8, device=dev())
    vc = torch.zeros_like(kc)
    sc = torch.zeros((x.k.shape[0], L, rec), dtype=torch.float16, device=dev())
    seg = qsa.Segment(kc, vc, 0, kv_scale=sc)
    pooled = pooled_buffer(L, dev())
    qsa.append_tokens(qsa.Seq(L, L, pooled, [seg], idx_keys=x.idxk), x.k.contiguous(), x.v.contiguous(),
                      x.idxk.clone())
    step = qsa.LayerStep([qsa.Seq(L, M, pooled, [seg], idx_keys=x.idxk)], x.q_idx, x.q)
    step.run()
    torch.cuda.synchronize()
    h = _host(x)
    quant, dequant = ((oracle.fp8_quantize, oracle.fp8_dequantize) if state == "fp8"
                      else (oracle.q8_quantize, oracle.q8_dequantize))
    kq, ks = quant(h["k"])
    vq, vs = quant(h["v"])
    np.testing.assert_array_equal(to_np(kc), kq)
    np.testing.assert_array_equal(to_np(vc), vq)
    sb = to_np(sc.view(torch.int16)).view(np.uint16)
    np.testing.assert_array_equal(sb[..., :rec // 2] if state == "q8" else sb[..., 0], ks)
    np.testing.assert_array_equal(sb[..., rec // 2:] if state == "q8" else sb[..., 1], vs)
    pooled_ref = oracle.pool(h["idxk"])
    s_ref = oracle.score(h["q_idx"], pooled_ref, x.row_pos)
    sel_ref, cnt_ref, tau = oracle.select(s_ref, x.row_pos)
    sel, cnt = to_np(step.sel), to_np(step.cnt)
    assert_selection_close(sel, cnt, sel_ref, cnt_ref, tau, s_ref, x.row_pos)
    kd, vd = dequant(kq, ks), dequant(vq, vs)
    out_ref, lse_ref = oracle.attn(h["q"], kd, vd, x.row_pos, sel, cnt)
    assert_attn_close(to_np(step.out), to_np(step.lse), out_ref, lse_ref, True)


def test_prefill_chunk_sampled_rows():
    # 2,048 rows appended at a 100,352-token prefix; rows are independent, so
    # checking a sample of rows is exact for those rows.
    T, prefix = 2048, 100_352
    x = make_layer(L=prefix + T, M=T, dtype=torch.bfloat16, seed=4, n_planted=256, device=dev())
    step, _ = _gpu_step(x)
    rows = [0, 1, 2, 3, 4, 511, 512, 1023, 1024, 1535, 1536, 2043, 2044, 2045, 2046, 2047]
    h = _host(x)
    pos = [x.row_pos[r] for r in rows]
    pooled_ref = oracle.pool(h["idxk"])
    s_ref = oracle.score(h["q_idx"][rows], pooled_ref, pos)
    sel_ref, cnt_ref, tau = oracle.select(s_ref, pos)
    nb = s_ref.shape[1]
    assert_scores_close(to_np(step.scores)[rows, :nb], s_ref,
                        2 * score_bound(h["q_idx"][rows], pooled_ref, pos), pos)
    sel_all, cnt_all = to_np(step.sel), to_np(step.cnt)
    assert_selection_close(sel_all[rows], cnt_all[rows], sel_ref, cnt_ref, tau, s_ref, pos)
    # Attention given the oracle's selection for the sampled rows.
    sel_all[rows] = sel_ref
    cnt_all[rows] = cnt_ref
    out = torch.empty_like(step.out)
    lse = torch.empty_like(step.lse)
    qsa.sparse_attn([qsa.Seq(x.L, T, segments=[qsa.Segment(x.k, x.v, 0)])], x.q,
                    torch.from_numpy(sel_all).to(dev()), torch.from_numpy(cnt_all).to(dev()), out, lse)
    torch.cuda.synchronize()
    out_ref, lse_ref = oracle.attn(h["q"][rows], h["k"], h["v"], pos, sel_ref, cnt_ref)
    assert_attn_close(to_np(out)[rows], to_np(lse)[rows], out_ref, lse_ref, True)


def test_prefill_chunk_blocked_selection_equals_one_pass():
    # The 2,048-row chunk at a 100,352-token prefix: key-axis chunks of 4,096
    # blocks give the same selection as the [2,048, 25,600] score buffer.
    T, prefix = 2048, 100_352
    x = make_layer(L=prefix + T, M=T, dtype=torch.bfloat16, seed=4, n_planted=256, device=dev())
    step, _ = _gpu_step(x)
    sel = torch.empty_like(step.sel)
    cnt = torch.empty_like(step.cnt)
    seqs = [qsa.Seq(x.L, T, step.seqs[0].pooled)]
    qsa.score_select_topk_blocked(seqs, x.q_idx, sel, cnt, 512, 4096)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(to_np(cnt), to_np(step.cnt))
    np.testing.assert_array_equal(to_np(sel), to_np(step.sel))
    # ... and the blocked selection against the oracle on a sample of rows
    # (rows are independent), chunk edges included.
    rows = [0, 1, 1023, 1024, 2047]
    h = _host(x)
    pos = [x.row_pos[r] for r in rows]
    pooled_ref = oracle.pool(h["idxk"])
    s_ref = oracle.score(h["q_idx"][rows], pooled_ref, pos)
    sel_ref, cnt_ref, tau = oracle.select(s_ref, pos)
    assert_selection_close(to_np(sel)[rows], to_np(cnt)[rows], sel_ref, cnt_ref, tau, s_ref, pos)


@pytest.mark.parametrize("D", [256, 128])
def test_ragged_segmented_batch_full_size(D):
    # 16 sequences, 8 decoding one row and 8 verifying four, contexts
    # log-uniform in 4,096..262,144, each cache split into 3..12 separately
    # allocated segments at token positions (not block-aligned).
    spec = ragged_batch_spec(16, seed=0)
    xs, seqs, single = [], [], []
    for i, (L, M, ns) in enumerate(zip(spec.lengths, spec.rows, spec.n_segments)):
        x = make_layer(L=L, M=M, dtype=torch.bfloat16, seed=100 + i, n_planted=256, head_dim=D, device=dev())
        pooled = pooled_buffer(L, dev())
        if (L - M) // 4:
            qsa.pool_index_keys(x.idxk, pooled, 0, (L - M) // 4)
        cuts = segment_cuts(L, ns, seed=i)
        segs = [qsa.Segment(x.k[:, f:f + n].clone(), x.v[:, f:f + n].clone(), f) for f, n in cuts]
        seqs.append(qsa.Seq(L, M, pooled, segs, idx_keys=x.idxk))
        single.append(qsa.Seq(L, M, pooled, [qsa.Segment(x.k, x.v, 0)]))
        xs.append(x)
    q_idx = torch.cat([x.q_idx for x in xs])
    q = torch.cat([x.q for x in xs])
    step = qsa.LayerStep(seqs, q_idx, q)
    step.run()
    # Single-buffer attention on the same selection.
    out1 = torch.empty_like(step.out)
    lse1 = torch.empty_like(step.lse)
    qsa.sparse_attn(single, q, step.sel, step.cnt, out1, lse1)
    torch.cuda.synchronize()
    np.testing.assert_allclose(to_np(step.out), to_np(out1), atol=2e-3)
    row = 0
    sel_all, cnt_all = to_np(step.sel), to_np(step.cnt)
    for x in xs:
        h = _host(x)
        pooled_ref = oracle.pool(h["idxk"])
        s_ref = oracle.score(h["q_idx"], pooled_ref, x.row_pos)
        sel_ref, cnt_ref, tau = oracle.select(s_ref, x.row_pos)
        rs = slice(row, row + x.M)
        assert_selection_close(sel_all[rs], cnt_all[rs], sel_ref, cnt_ref, tau, s_ref, x.row_pos)
        out_ref, lse_ref = oracle.attn(h["q"], h["k"], h["v"], x.row_pos, sel_all[rs], cnt_all[rs])
        assert_attn_close(to_np(step.out)[rs], to_np(step.lse)[rs], out_ref, lse_ref, True)
        row += x.M
