"""GPU parity: every step of the CUDA library against the fp64 oracle on the
same seeded inputs, at sizes the oracle finishes in seconds that still span
several tiles and a ragged tail.  Tolerances are stated in qsa_cases."""
import math

import numpy as np
import pytest
import torch

import indexed_sparse_attention_gb300 as qsa
import oracle
from qsa_cases import (assert_attn_close, assert_pooled_close, assert_scores_close, assert_selection_close, dev,
                       oracle_layer, pool_all, pooled_buffer, score_bound, to_np, DeviceLayer)
from workloads import make_layer, segment_cuts

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from indexed_sparse_attention_gb300 import build
    build.build()
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need CUDA")


# ------------------------------------------------------------------ step 1
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_pool_matches_oracle(dtype):
    x = make_layer(L=4099, M=4, dtype=dtype, seed=0)
    idxk = x.idxk.to(dev())
    pooled = pooled_buffer(x.L, dev())
    pool_all(idxk, pooled, x.L)
    got = to_np(pooled)[:1024].astype(np.float64)
    want = oracle.pool(x.idxk)
    # Three fp32 additions and an exact scaling: |err| <= 3 u * mean_j |k_j| + u |mean|.
    u = 2.0 ** -24
    mag = np.abs(x.idxk.double().numpy()[:4096]).reshape(1024, 4, 128).mean(axis=1)
    bound = 3 * u * mag + u * np.abs(want)
    assert (np.abs(got - want) <= bound).all()
    assert np.isnan(to_np(pooled)[1024]).all()              # the incomplete block is not pooled
    # A sub-range writes only its blocks.
    part = pooled_buffer(x.L, dev())
    qsa.pool_index_keys(idxk, part, 10, 7)
    p = to_np(part)
    assert (np.abs(p[10:17] - want[10:17]) <= bound[10:17]).all()
    assert np.isnan(p[:10]).all() and np.isnan(p[17:]).all()


# ------------------------------------------------------------------ step 2
@pytest.mark.parametrize("dtype,L,M", [(torch.float32, 4099, 4), (torch.bfloat16, 4099, 4),
                                       (torch.bfloat16, 5003, 8), (torch.bfloat16, 777, 1),
                                       (torch.bfloat16, 6001, 6), (torch.bfloat16, 70_001, 2),
                                       (torch.float32, 3001, 3), (torch.bfloat16, 2100, 37)])
def test_scores_match_oracle(dtype, L, M):
    x = make_layer(L=L, M=M, dtype=dtype, seed=1)
    pooled_ref = oracle.pool(x.idxk)
    # The GPU scores the oracle's pooled keys rounded to fp32 ...
    pooled = torch.from_numpy(pooled_ref.astype(np.float32)).to(dev())
    q_idx = x.q_idx.to(dev())
    ld = (L // 4 + 7) // 8 * 8
    scores = torch.full((M, ld), float("nan"), device=dev())
    gld = (qsa.n_groups(L) + 3) // 4 * 4
    gmax = torch.full((M, gld), float("nan"), device=dev())
    seq = qsa.Seq(L, M, pooled)
    qsa.score_blocks([seq], q_idx, scores, group_max=gmax)
    ref = oracle.score(x.q_idx, pooled_ref.astype(np.float32).astype(np.float64), x.row_pos, ld=ld)
    bound = score_bound(x.q_idx, pooled_ref, x.row_pos)
    got = to_np(scores)
    assert_scores_close(got, ref, bound, x.row_pos)
    for r, p in enumerate(x.row_pos):                       # blocks a row cannot see stay unwritten
        assert np.isnan(got[r, oracle.visible_blocks(p):]).all()
    # Group maxima: exactly the maximum of the written scores of each group.
    gm = to_np(gmax)
    for r, p in enumerate(x.row_pos):
        nb = oracle.visible_blocks(p)
        G = (nb + 15) // 16
        want = np.array([got[r, 16 * g:min(16 * g + 16, nb)].max() for g in range(G)], dtype=np.float32)
        np.testing.assert_array_equal(gm[r, :G], want)
        assert np.isnan(gm[r, G:]).all()
    # ... and the chained GPU pool gives scores within the same bound.
    gp = pooled_buffer(L, dev())
    pool_all(x.idxk.to(dev()), gp, L)
    qsa.score_blocks([qsa.Seq(L, M, gp)], q_idx, scores)
    ref2 = oracle.score(x.q_idx, pooled_ref, x.row_pos, ld=ld)
    assert_scores_close(to_np(scores), ref2, 2 * bound, x.row_pos)


def test_scores_zero_query_and_nonnegative():
    x = make_layer(L=1600, M=2, dtype=torch.bfloat16, seed=2)
    pooled = pooled_buffer(x.L, dev())
    pool_all(x.idxk.to(dev()), pooled, x.L)
    scores = torch.empty((2, 400), device=dev())
    qsa.score_blocks([qsa.Seq(x.L, 2, pooled)], torch.zeros_like(x.q_idx).to(dev()), scores)
    got = to_np(scores)
    assert (got[0, :399] == 0).all() and (got[1] == 0).all()      # rows at 1,598 and 1,599
    qsa.score_blocks([qsa.Seq(x.L, 2, pooled)], x.q_idx.to(dev()), scores)
    got = to_np(scores)
    assert (got[0, :399] >= 0).all() and (got[1] >= 0).all()


# ------------------------------------------------------------------ steps 1 + 2 in one call
# (idx dtype, q_idx dtype): bf16/bf16 takes the few-row kernel that pools in
# place; f32 index queries, 600-row sequences (tensor cores) and ragged
# batches check the paths that pool in a launch of their own.
@pytest.mark.parametrize("Ls,Ms,idx_dtype,q_dtype", [
    ([261_120], [4], torch.bfloat16, torch.bfloat16), ([65_536], [1], torch.bfloat16, torch.bfloat16),
    ([261_120], [8], torch.bfloat16, torch.bfloat16), ([9001], [5], torch.bfloat16, torch.bfloat16),
    ([9003], [7], torch.float32, torch.bfloat16),
    ([9001], [3], torch.float32, torch.bfloat16), ([9001], [4], torch.bfloat16, torch.float32),
    ([4099], [600], torch.bfloat16, torch.bfloat16), ([4097], [1], torch.bfloat16, torch.bfloat16),
    ([9002], [1], torch.float32, torch.bfloat16), ([9002], [2], torch.bfloat16, torch.bfloat16),
    ([4099, 700, 30_000, 9, 2052, 65_540], [4, 1, 2, 3, 1, 4], torch.bfloat16, torch.bfloat16)])
def test_pool_score_equals_pool_then_score(Ls, Ms, idx_dtype, q_dtype):
    _pool_score_vs_separate(Ls, Ms, idx_dtype, q_dtype)


# Batches of 8 sequences, long and short mixed.  On a 152-SM GB300 each of
# these puts the completed blocks of two sequences in one consumer warp of
# the few-row kernel (the last items of a long and of a short sequence, 4
# items apart in one CTA), so one warp pools a second block from keys read
# when its tile is reached rather than from its prefetched copy.
@pytest.mark.parametrize("Ls,Ms", [
    ([386, 122_275, 255, 38, 79, 161_101, 214, 232], [1, 1, 3, 2, 3, 4, 2, 2]),
    ([176_377, 124, 109, 237, 188, 392, 351, 390], [3, 2, 1, 3, 3, 4, 4, 4]),
    ([102_237, 120, 145_450, 195_651, 24, 263, 196_566, 465], [4, 1, 1, 1, 2, 2, 4, 4])])
def test_pool_score_many_sequences(Ls, Ms):
    _pool_score_vs_separate(Ls, Ms, torch.bfloat16, torch.bfloat16)


def _pool_score_vs_separate(Ls, Ms, idx_dtype, q_dtype):
    runs = []
    for fused in (True, False):
        seqs, rows = [], 0
        q_parts = []
        for i, (L, M) in enumerate(zip(Ls, Ms)):
            x = make_layer(L=L, M=M, dtype=torch.float32, seed=100 + i, device=dev())
            idxk = x.idxk.to(idx_dtype)
            pooled = pooled_buffer(L, dev())              # NaN: new blocks must be written
            b0 = (L - M) // 4
            if b0:
                qsa.pool_index_keys(idxk, pooled, 0, b0)
            seqs.append(qsa.Seq(L, M, pooled, idx_keys=idxk))
            q_parts.append(x.q_idx.to(q_dtype))
            rows += M
        q_idx = torch.cat(q_parts)
        ld = (max(L // 4 for L in Ls) + 3) // 4 * 4
        scores = torch.full((rows, ld), float("nan"), device=dev())
        gmax = torch.full((rows, (qsa.n_groups(max(Ls)) + 3) // 4 * 4), float("nan"), device=dev())
        if fused:
            qsa.pool_score_blocks(seqs, q_idx, scores, group_max=gmax)
        else:
            for sq in seqs:
                b0, b1 = (sq.n_tokens - sq.n_rows) // 4, sq.n_tokens // 4
                if b1 > b0:
                    qsa.pool_index_keys(sq.idx_keys, sq.pooled, b0, b1 - b0)
            qsa.score_blocks(seqs, q_idx, scores, group_max=gmax)
        torch.cuda.synchronize()
        runs.append((seqs, scores, gmax, q_idx))
    (sa, sc_a, gm_a, q_a), (sb, sc_b, gm_b, _) = runs
    # The fused call against the oracle: the blocks it pooled, and every
    # visible score of a sample of rows (scores of the stored pooled keys).
    r = 0
    for qa in sa:
        L, M = qa.n_tokens, qa.n_rows
        assert_pooled_close(to_np(qa.pooled), qa.idx_keys.float(), range((L - M) // 4, L // 4))
        pos = qa.row_pos
        pooled_ref = to_np(qa.pooled)[:L // 4].astype(np.float64)
        s_ref = oracle.score(q_a[r:r + M].float().cpu(), pooled_ref, pos)
        nb = s_ref.shape[1]
        assert_scores_close(to_np(sc_a)[r:r + M, :nb], s_ref, score_bound(q_a[r:r + M].float(), pooled_ref, pos), pos)
        r += M
    r = 0
    for qa, qb in zip(sa, sb):
        L, M = qa.n_tokens, qa.n_rows
        assert torch.equal(qa.pooled[:L // 4], qb.pooled[:L // 4])
        for j in range(M):
            nb = (L - M + j + 1) // 4
            assert torch.equal(sc_a[r, :nb], sc_b[r, :nb])
            ng = (nb + 15) // 16
            assert torch.equal(gm_a[r, :ng], gm_b[r, :ng])
            r += 1


# ------------------------------------------------------------------ step 3
def group_maxima(scores_f32: np.ndarray, row_pos) -> np.ndarray:
    """Per row, the maximum score of every group of 16 visible blocks (the
    layout qsa_score_blocks writes), NaN elsewhere."""
    G = max((oracle.visible_blocks(p) + 15) // 16 for p in row_pos)
    out = np.full((len(row_pos), (G + 3) // 4 * 4), np.nan, dtype=np.float32)
    for r, p in enumerate(row_pos):
        nb = oracle.visible_blocks(p)
        for g in range((nb + 15) // 16):
            out[r, g] = scores_f32[r, 16 * g:min(16 * g + 16, nb)].max()
    return out


def _select_gpu(scores_f32: np.ndarray, row_pos, L, top_k=512, with_group_max=False):
    M, ld = scores_f32.shape
    n_rows = len(row_pos)
    s = torch.from_numpy(np.ascontiguousarray(scores_f32)).to(dev())
    sel = torch.full((M, top_k), -7, dtype=torch.int32, device=dev())
    cnt = torch.full((M,), -7, dtype=torch.int32, device=dev())
    gm = torch.from_numpy(group_maxima(scores_f32, row_pos)).to(dev()) if with_group_max else None
    qsa.select_topk([qsa.Seq(L, n_rows)], s, sel, cnt, top_k, group_max=gm)
    return to_np(sel), to_np(cnt)


def _select_case(scores_f32, L, M, top_k=512):
    row_pos = [L - M + j for j in range(M)]
    rs, rc, _ = oracle.select(scores_f32.astype(np.float64), row_pos, top_k)
    # Without group maxima (the kernel derives them) and with them.
    for with_gm in (False, True):
        sel, cnt = _select_gpu(scores_f32, row_pos, L, top_k, with_gm)
        np.testing.assert_array_equal(cnt, rc)
        np.testing.assert_array_equal(sel, rs)


@pytest.mark.parametrize("L,M,kind", [(4099, 4, "normal"), (261_120, 4, "normal"), (65_536, 1, "normal"),
                                      (9001, 3, "coarse"), (9001, 3, "zeros"), (9001, 2, "signed_zeros"),
                                      (9001, 2, "increasing"), (2051, 4, "normal"), (2052, 1, "normal"),
                                      (2049, 2, "normal"), (13, 4, "normal"), (1 << 20, 1, "coarse"),
                                      (262_144, 2, "zeros"), (100_003, 3, "planted_ties"),
                                      (40_000, 2, "negative")])
def test_select_bit_exact_on_fp32_scores(L, M, kind):
    rng = np.random.default_rng(L + M)
    nb = L // 4
    ld = (nb + 3) // 4 * 4
    s = np.zeros((M, ld), dtype=np.float32)
    if kind == "normal":
        s[:, :nb] = np.abs(rng.standard_normal((M, nb))).astype(np.float32) * 3
    elif kind == "coarse":
        s[:, :nb] = rng.integers(0, 40, size=(M, nb)).astype(np.float32) * 0.125
    elif kind == "signed_zeros":
        s[:, :nb] = np.where(rng.random((M, nb)) < 0.5, np.float32(-0.0), np.float32(0.0))
        s[:, 7::97] = 1.5
    elif kind == "increasing":
        s[:, :nb] = np.arange(nb, dtype=np.float32)[None]
    elif kind == "planted_ties":
        # 600 blocks share the top score: the 512 lowest ids among them win.
        s[:, :nb] = np.abs(rng.standard_normal((M, nb))).astype(np.float32)
        for r in range(M):
            s[r, rng.choice(nb - M, 600, replace=False)] = 9.0
    elif kind == "negative":
        s[:, :nb] = rng.standard_normal((M, nb)).astype(np.float32) - 4
    _select_case(s, L, M)


@pytest.mark.parametrize("top_k", [1, 7, 64, 512, 1000, 1024])
def test_select_other_budgets(top_k):
    rng = np.random.default_rng(top_k)
    L, M = 20_011, 2
    s = np.zeros((M, (L // 4 + 3) // 4 * 4), dtype=np.float32)     # row stride: a multiple of 16 bytes
    s[:, :L // 4] = rng.integers(0, 300, size=(M, L // 4)) * 0.5
    _select_case(s, L, M, top_k)


def test_select_ragged_sequences():
    rng = np.random.default_rng(5)
    Ls, Ms = [4099, 700, 30_000, 9, 2052, 65_540, 5000, 8001, 12_345], [4, 1, 2, 3, 1, 4, 8, 1, 2]
    ld = (max(L // 4 for L in Ls) + 3) // 4 * 4
    rows = sum(Ms)
    s = np.abs(rng.standard_normal((rows, ld))).astype(np.float32)
    s[3] = np.round(s[3] * 4) / 4   # ties
    seqs = [qsa.Seq(L, M) for L, M in zip(Ls, Ms)]
    sd = torch.from_numpy(s).to(dev())
    sel = torch.empty((rows, 512), dtype=torch.int32, device=dev())
    cnt = torch.empty((rows,), dtype=torch.int32, device=dev())
    qsa.select_topk(seqs, sd, sel, cnt)
    pos = [p for sq in seqs for p in sq.row_pos]
    rs, rc, _ = oracle.select(s.astype(np.float64), pos)
    np.testing.assert_array_equal(to_np(cnt), rc)
    np.testing.assert_array_equal(to_np(sel), rs)
    # With the group maxima score_blocks would write.
    gm = torch.from_numpy(group_maxima(s, pos)).to(dev())
    sel.fill_(-7)
    cnt.fill_(-7)
    qsa.select_topk(seqs, sd, sel, cnt, group_max=gm)
    np.testing.assert_array_equal(to_np(cnt), rc)
    np.testing.assert_array_equal(to_np(sel), rs)


# ------------------------------------------------------------------ appending tokens with in-place pooling
@pytest.mark.parametrize("L,n,kv_dtype,idx_dtype,n_segs", [
    (4099, 4, torch.bfloat16, torch.bfloat16, 1), (65_536, 1, torch.bfloat16, torch.bfloat16, 1),
    (2148, 2048, torch.bfloat16, torch.bfloat16, 3), (7, 1, torch.float32, torch.float32, 1),
    (3, 3, torch.float32, torch.bfloat16, 1), (9001, 5, torch.float32, torch.float32, 4),
    (2052, 9, torch.bfloat16, torch.float32, 2)])
def test_append_writes_caches_and_pools(L, n, kv_dtype, idx_dtype, n_segs):
    x = make_layer(L=L, M=min(n, L), dtype=torch.float32, seed=L + n, device=dev())
    k_full, v_full = x.k.to(kv_dtype), x.v.to(kv_dtype)
    idx_full = x.idxk.to(idx_dtype)
    # Caches hold the first L - n tokens; the rest is garbage (NaN) until the append.
    k_c, v_c = torch.full_like(k_full, float("nan")), torch.full_like(v_full, float("nan"))
    idx_c = torch.full_like(idx_full, float("nan"))
    k_c[:, :L - n], v_c[:, :L - n], idx_c[:L - n] = k_full[:, :L - n], v_full[:, :L - n], idx_full[:L - n]
    pooled = pooled_buffer(L, dev())
    b0 = (L - n) // 4
    if b0:
        qsa.pool_index_keys(idx_c, pooled, 0, b0)
    # Segments: views of the caches, one cut inside the new tokens when several.
    cuts = [0] + sorted({max(1, L - n + (n * j) // n_segs) for j in range(1, n_segs)} - {0, L}) + [L]
    segs = [qsa.Segment(k_c[:, a:b], v_c[:, a:b], a) for a, b in zip(cuts[:-1], cuts[1:])]
    seq = qsa.Seq(L, n, pooled, segs, idx_keys=idx_c)
    qsa.append_tokens(seq, k_full[:, L - n:].contiguous(), v_full[:, L - n:].contiguous(),
                      idx_full[L - n:].contiguous())
    torch.cuda.synchronize()
    assert torch.equal(k_c, k_full) and torch.equal(v_c, v_full) and torch.equal(idx_c, idx_full)
    ref = pooled_buffer(L, dev())
    if L // 4:
        qsa.pool_index_keys(idx_full, ref, 0, L // 4)
    torch.cuda.synchronize()
    # The blocks the append pooled, against the oracle's mean of the stored
    # index keys, and the same numbers as the pooling kernel.
    assert_pooled_close(to_np(pooled), idx_full.float(), range(b0, L // 4))
    assert torch.equal(pooled[:L // 4], ref[:L // 4])


# The append and the scoring in one call (qsa_append_score_blocks): one
# launch on the few-row path (bf16 index queries, <= 4 rows, K/V state not
# quantized), else an append launch then the scoring.  The caches, pooled
# keys, scores and group maxima equal those of the two separate calls, and
# the pooled keys and scores match the oracle.
@pytest.mark.parametrize("L,n,kv_dtype,idx_dtype,n_segs,q_dtype", [
    (65_536, 1, torch.bfloat16, torch.bfloat16, 1, torch.bfloat16),
    (261_120, 4, torch.bfloat16, torch.bfloat16, 1, torch.bfloat16),
    (9001, 8, torch.bfloat16, torch.float32, 3, torch.bfloat16),
    (9002, 2, torch.float32, torch.bfloat16, 2, torch.bfloat16),
    (4099, 3, torch.bfloat16, torch.bfloat16, 1, torch.float32),
    (2148, 20, torch.bfloat16, torch.bfloat16, 1, torch.bfloat16),
    (9003, 1, torch.bfloat16, torch.float32, 2, torch.bfloat16),
    (5, 3, torch.bfloat16, torch.bfloat16, 1, torch.bfloat16),
    (5, 5, torch.bfloat16, torch.bfloat16, 1, torch.bfloat16)])
def test_append_score_equals_append_then_score(L, n, kv_dtype, idx_dtype, n_segs, q_dtype):
    x = make_layer(L=L, M=n, dtype=torch.float32, seed=L + 3 * n, device=dev())
    k_full, v_full, idx_full = x.k.to(kv_dtype), x.v.to(kv_dtype), x.idxk.to(idx_dtype)
    q_idx = x.q_idx.to(q_dtype)
    ld = (L // 4 + 3) // 4 * 4
    runs = []
    for fused in (True, False):
        k_c, v_c = torch.full_like(k_full, float("nan")), torch.full_like(v_full, float("nan"))
        idx_c = torch.full_like(idx_full, float("nan"))
        k_c[:, :L - n], v_c[:, :L - n], idx_c[:L - n] = k_full[:, :L - n], v_full[:, :L - n], idx_full[:L - n]
        pooled = pooled_buffer(L, dev())
        b0 = (L - n) // 4
        if b0:
            qsa.pool_index_keys(idx_c, pooled, 0, b0)
        cuts = [0] + sorted({max(1, L - n + (n * j) // n_segs) for j in range(1, n_segs)} - {0, L}) + [L]
        segs = [qsa.Segment(k_c[:, a:b], v_c[:, a:b], a) for a, b in zip(cuts[:-1], cuts[1:])]
        seq = qsa.Seq(L, n, pooled, segs, idx_keys=idx_c)
        scores = torch.full((n, ld), float("nan"), device=dev())
        gmax = torch.full((n, (qsa.n_groups(L) + 3) // 4 * 4), float("nan"), device=dev())
        new = (k_full[:, L - n:].contiguous(), v_full[:, L - n:].contiguous(), idx_full[L - n:].contiguous())
        if fused:
            qsa.append_score_blocks(seq, *new, q_idx, scores, group_max=gmax)
        else:
            qsa.append_tokens(seq, *new)
            qsa.score_blocks([seq], q_idx, scores, group_max=gmax)
        torch.cuda.synchronize()
        runs.append((k_c, v_c, idx_c, pooled, scores, gmax, seq))
    (ka, va, ia, pa, sa, ga, seq), (kb, vb, ib, pb, sb, gb, _) = runs
    assert torch.equal(ka, k_full) and torch.equal(va, v_full) and torch.equal(ia, idx_full)
    nb = L // 4
    assert torch.equal(pa[:nb], pb[:nb])
    pos = seq.row_pos
    for r, p_ in enumerate(pos):
        vis = (p_ + 1) // 4
        assert torch.equal(sa[r, :vis], sb[r, :vis])
        ng = (vis + 15) // 16
        assert torch.equal(ga[r, :ng], gb[r, :ng])
    # Against the oracle: the blocks the call pooled, and the scores of the
    # stored pooled keys.
    if nb:
        assert_pooled_close(to_np(pa), idx_full.float(), range((L - n) // 4, nb))
        pooled_ref = to_np(pa)[:nb].astype(np.float64)
        s_ref = oracle.score(q_idx.float().cpu(), pooled_ref, pos)
        assert_scores_close(to_np(sa)[:, :s_ref.shape[1]], s_ref, score_bound(q_idx.float(), pooled_ref, pos), pos)


@pytest.mark.parametrize("M", [4, 1])
def test_layer_step_with_append_replays_in_a_graph(M):
    # The step with new tokens (append, pooling and scoring in one launch)
    # captured in a CUDA graph and replayed gives what the eager step gives,
    # caches included.
    L = 9001
    x = make_layer(L=L, M=M, dtype=torch.bfloat16, seed=43 + M, device=dev())
    new = [(x.k[:, L - M:].contiguous(), x.v[:, L - M:].contiguous(), x.idxk[L - M:].contiguous())]
    runs = []
    for graphed in (False, True):
        k_c, v_c, idx_c = x.k.clone(), x.v.clone(), x.idxk.clone()
        k_c[:, L - M:] = 0
        v_c[:, L - M:] = 0
        idx_c[L - M:] = 0
        pooled = pooled_buffer(L, dev())
        qsa.pool_index_keys(idx_c, pooled, 0, (L - M) // 4)
        step = qsa.LayerStep([qsa.Seq(L, M, pooled, [qsa.Segment(k_c, v_c, 0)], idx_keys=idx_c)], x.q_idx, x.q)
        if graphed:
            s = torch.cuda.Stream()
            s.wait_stream(torch.cuda.current_stream())
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=s):
                step.run(new_tokens=new)
            g.replay()
        else:
            step.run(new_tokens=new)
        torch.cuda.synchronize()
        runs.append((step.out.clone(), step.lse.clone(), k_c, v_c, idx_c, pooled))
    (oa, la, ka, va, ia, pa), (ob, lb, kb, vb, ib, pb) = runs
    assert torch.equal(oa, ob) and torch.equal(la, lb)
    assert torch.equal(ka, x.k) and torch.equal(kb, x.k) and torch.equal(vb, x.v) and torch.equal(ib, x.idxk)
    assert torch.equal(pa[:L // 4], pb[:L // 4])


def test_layer_step_with_append_equals_prewritten_caches():
    L, M = 9001, 4
    x = make_layer(L=L, M=M, dtype=torch.bfloat16, seed=41, device=dev())
    pa = pooled_buffer(L, dev())
    qsa.pool_index_keys(x.idxk, pa, 0, (L - M) // 4)
    step_a = qsa.LayerStep([qsa.Seq(L, M, pa, [qsa.Segment(x.k, x.v, 0)], idx_keys=x.idxk)], x.q_idx, x.q)
    out_a, lse_a = step_a.run()
    k_c, v_c, idx_c = x.k.clone(), x.v.clone(), x.idxk.clone()
    k_c[:, L - M:] = 0
    v_c[:, L - M:] = 0
    idx_c[L - M:] = 0
    pb = pooled_buffer(L, dev())
    qsa.pool_index_keys(idx_c, pb, 0, (L - M) // 4)
    step_b = qsa.LayerStep([qsa.Seq(L, M, pb, [qsa.Segment(k_c, v_c, 0)], idx_keys=idx_c)], x.q_idx, x.q)
    out_b, lse_b = step_b.run(new_tokens=[(x.k[:, L - M:].contiguous(), x.v[:, L - M:].contiguous(),
                                           x.idxk[L - M:].contiguous())])
    torch.cuda.synchronize()
    assert torch.equal(out_a, out_b) and torch.equal(lse_a, lse_b)
    assert torch.equal(k_c, x.k) and torch.equal(idx_c, x.idxk)


# ------------------------------------------------------------------ fp8 K/V state (E4M3 codes + f16 scales)
def _fp8_state(shape, seed):
    """Seeded E4M3 codes with exponents 2^-4 .. 2^2 and random signs/mantissas,
    and f16 (K, V) scale pairs 2^-4 .. 2^-1 per head and token: values of
    magnitude ~0.5 and at most ~4, like N(0, 1) K/V written as fp8."""
    g = torch.Generator().manual_seed(seed)
    Hkv, L, D = shape
    e = torch.randint(3, 10, (2, Hkv, L, D), generator=g)
    m = torch.randint(0, 8, (2, Hkv, L, D), generator=g)
    sgn = torch.randint(0, 2, (2, Hkv, L, D), generator=g)
    codes = ((sgn << 7) | (e << 3) | m).to(torch.uint8)
    expo = torch.randint(-4, -1, (Hkv, L, 2), generator=g).double()
    frac = 1 + torch.randint(0, 1024, (Hkv, L, 2), generator=g).double() / 1024
    scales = (frac * torch.pow(2.0, expo)).to(torch.float16)
    return codes[0], codes[1], scales


def _fp8_ref(kc, vc, scales):
    sb = scales.view(torch.int16).numpy().view(np.uint16)
    return oracle.fp8_dequantize(kc.numpy(), sb[..., 0]), oracle.fp8_dequantize(vc.numpy(), sb[..., 1])


# Many-row calls (one split per row) at both head sizes; 9,001-token rows
# have full 2,051-entry lists with ragged tails.
@pytest.mark.parametrize("L,M,D,n_splits", [(4099, 4, 256, 0), (9001, 1, 256, 0), (9001, 3, 128, 5),
                                            (2051, 4, 256, 1), (1200, 600, 256, 0), (1200, 600, 128, 0),
                                            (9001, 512, 128, 0)])
def test_fp8_attention_matches_oracle(L, M, D, n_splits):
    x = make_layer(L=L, M=M, dtype=torch.bfloat16, seed=L + D, head_dim=D)
    kc, vc, scales = _fp8_state((2, L, D), seed=L + M)
    sel, cnt, _ = _oracle_selection(x)
    kd, vd = _fp8_ref(kc, vc, scales)
    ref_out, ref_lse = oracle.attn(x.q, kd, vd, x.row_pos, sel, cnt)
    seg = [qsa.Segment(kc.to(dev()), vc.to(dev()), 0, kv_scale=scales.to(dev()))]
    out, lse = _attn_gpu(x, sel, cnt, segments=lambda k, v: seg, n_splits=n_splits)
    assert_attn_close(out, lse, ref_out, ref_lse, True)


@pytest.mark.parametrize("L,M", [(9001, 4), (1500, 520)])
def test_fp8_segments_equal_single_buffer(L, M):
    D = 256
    x = make_layer(L=L, M=M, dtype=torch.bfloat16, seed=61, head_dim=D)
    kc, vc, scales = _fp8_state((2, L, D), seed=62)
    kc, vc, scales = kc.to(dev()), vc.to(dev()), scales.to(dev())
    sel, cnt, _ = _oracle_selection(x)
    single, single_lse = _attn_gpu(x, sel, cnt,
                                   segments=lambda k, v: [qsa.Segment(kc, vc, 0, kv_scale=scales)])
    cuts = segment_cuts(L, 6, seed=4)
    segs = [qsa.Segment(kc[:, f:f + n].clone(), vc[:, f:f + n].clone(), f, kv_scale=scales[:, f:f + n].clone())
            for f, n in cuts]
    out, lse = _attn_gpu(x, sel, cnt, segments=lambda k, v: segs)
    np.testing.assert_allclose(out, single, atol=2e-3)
    kd, vd = _fp8_ref(kc.cpu(), vc.cpu(), scales.cpu())
    ref_out, ref_lse = oracle.attn(x.q, kd, vd, x.row_pos, sel, cnt)
    assert_attn_close(out, lse, ref_out, ref_lse, True)


@pytest.mark.parametrize("D", [256, 128])
def test_fp8_append_quantizes_like_oracle(D):
    L, n = 5003, 40
    x = make_layer(L=L, M=n, dtype=torch.bfloat16, seed=63, head_dim=D, device=dev())
    x.k[0, L - 3] = 0.0                                  # a zero row: scale 0, codes 0
    x.v[1, L - 2, 5] = 1000.0                            # a large element
    kc = torch.zeros((2, L, D), dtype=torch.uint8, device=dev())
    vc = torch.zeros_like(kc)
    scales = torch.zeros((2, L, 2), dtype=torch.float16, device=dev())
    idx_c = x.idxk.clone()
    pooled = pooled_buffer(L, dev())
    qsa.pool_index_keys(idx_c, pooled, 0, (L - n) // 4)
    seq = qsa.Seq(L, n, pooled, [qsa.Segment(kc, vc, 0, kv_scale=scales)], idx_keys=idx_c)
    qsa.append_tokens(seq, x.k[:, L - n:].contiguous(), x.v[:, L - n:].contiguous(), x.idxk[L - n:].contiguous())
    torch.cuda.synchronize()
    for which, src, codes in ((0, x.k, kc), (1, x.v, vc)):
        ref_c, ref_s = oracle.fp8_quantize(src[:, L - n:].cpu())
        np.testing.assert_array_equal(to_np(codes[:, L - n:]), ref_c)
        np.testing.assert_array_equal(to_np(scales[:, L - n:, which].view(torch.int16)).view(np.uint16), ref_s)
        assert (to_np(codes[:, :L - n]) == 0).all()        # earlier tokens untouched
    assert (to_np(kc[0, L - 3]) == 0).all() and float(scales[0, L - 3, 0]) == 0.0


def test_fp8_layer_step_matches_oracle():
    # A verify step over fp8 K/V written by the append, against the oracle's
    # quantization of the same rows and attention over its dequantized state.
    L, M = 9001, 4
    x = make_layer(L=L, M=M, dtype=torch.bfloat16, seed=64, device=dev())
    rows_k, rows_s = oracle.fp8_quantize(x.k.cpu())
    rows_v, rows_sv = oracle.fp8_quantize(x.v.cpu())
    kc = torch.from_numpy(rows_k).to(dev())
    vc = torch.from_numpy(rows_v).to(dev())
    sc = torch.from_numpy(np.stack([rows_s, rows_sv], axis=-1).view(np.float16).copy()).to(dev())
    kc[:, L - M:] = 0
    vc[:, L - M:] = 0
    pooled = pooled_buffer(L, dev())
    qsa.pool_index_keys(x.idxk, pooled, 0, (L - M) // 4)
    step = qsa.LayerStep([qsa.Seq(L, M, pooled, [qsa.Segment(kc, vc, 0, kv_scale=sc)], idx_keys=x.idxk)],
                         x.q_idx, x.q)
    step.run(new_tokens=[(x.k[:, L - M:].contiguous(), x.v[:, L - M:].contiguous(),
                          x.idxk[L - M:].contiguous())])
    torch.cuda.synchronize()
    ref = oracle_layer(x)
    kd = oracle.fp8_dequantize(rows_k, rows_s)
    vd = oracle.fp8_dequantize(rows_v, rows_sv)
    sel, cnt = to_np(step.sel), to_np(step.cnt)
    assert_selection_close(sel, cnt, ref["sel"], ref["cnt"], ref["tau"], ref["scores"], x.row_pos)
    ref_out, ref_lse = oracle.attn(x.q.cpu(), kd, vd, x.row_pos, sel, cnt)
    assert_attn_close(to_np(step.out), to_np(step.lse), ref_out, ref_lse, True)


# ------------------------------------------------------------------ q8 K/V state (Q8_0: int8 + f16 per 32)
def _q8_state(shape, seed):
    """Seeded int8 codes in [-127, 127] and f16 block scales 2^-7 .. 2^-6
    (values within about +-2), the K scales then the V scales of each row."""
    g = torch.Generator().manual_seed(seed)
    Hkv, L, D = shape
    codes = torch.randint(-127, 128, (2, Hkv, L, D), generator=g).to(torch.int8)
    expo = torch.randint(-7, -5, (Hkv, L, 2 * D // 32), generator=g).double()
    frac = 1 + torch.randint(0, 1024, (Hkv, L, 2 * D // 32), generator=g).double() / 1024
    return codes[0], codes[1], (frac * torch.pow(2.0, expo)).to(torch.float16)


def _q8_ref(kc, vc, scales):
    D = kc.shape[-1]
    sb = scales.view(torch.int16).numpy().view(np.uint16)
    return (oracle.q8_dequantize(kc.numpy(), sb[..., :D // 32]),
            oracle.q8_dequantize(vc.numpy(), sb[..., D // 32:]))


@pytest.mark.parametrize("L,M,D,n_splits", [(4099, 4, 256, 0), (9001, 1, 128, 0), (9001, 3, 256, 7),
                                            (1200, 600, 256, 0), (1200, 600, 128, 0), (9001, 512, 128, 0)])
def test_q8_attention_matches_oracle(L, M, D, n_splits):
    x = make_layer(L=L, M=M, dtype=torch.bfloat16, seed=L + D + 1, head_dim=D)
    kc, vc, scales = _q8_state((2, L, D), seed=L + M + 1)
    sel, cnt, _ = _oracle_selection(x)
    kd, vd = _q8_ref(kc, vc, scales)
    ref_out, ref_lse = oracle.attn(x.q, kd, vd, x.row_pos, sel, cnt)
    seg = [qsa.Segment(kc.to(dev()), vc.to(dev()), 0, kv_scale=scales.to(dev()))]
    out, lse = _attn_gpu(x, sel, cnt, segments=lambda k, v: seg, n_splits=n_splits)
    assert_attn_close(out, lse, ref_out, ref_lse, True)


@pytest.mark.parametrize("D", [256, 128])
def test_q8_append_quantizes_like_oracle(D):
    L, n = 5003, 40
    x = make_layer(L=L, M=n, dtype=torch.bfloat16, seed=65, head_dim=D, device=dev())
    x.k[0, L - 3, :32] = 0.0                             # a zero block: scale 0, codes 0
    x.v[1, L - 2, 5] = 1000.0                            # a large element
    kc = torch.zeros((2, L, D), dtype=torch.int8, device=dev())
    vc = torch.zeros_like(kc)
    scales = torch.zeros((2, L, 2 * D // 32), dtype=torch.float16, device=dev())
    idx_c = x.idxk.clone()
    pooled = pooled_buffer(L, dev())
    qsa.pool_index_keys(idx_c, pooled, 0, (L - n) // 4)
    seq = qsa.Seq(L, n, pooled, [qsa.Segment(kc, vc, 0, kv_scale=scales)], idx_keys=idx_c)
    qsa.append_tokens(seq, x.k[:, L - n:].contiguous(), x.v[:, L - n:].contiguous(), x.idxk[L - n:].contiguous())
    torch.cuda.synchronize()
    nb = D // 32
    for which, src, codes in ((0, x.k, kc), (1, x.v, vc)):
        ref_c, ref_s = oracle.q8_quantize(src[:, L - n:].cpu())
        np.testing.assert_array_equal(to_np(codes[:, L - n:]), ref_c)
        got_s = to_np(scales[:, L - n:, which * nb:(which + 1) * nb].contiguous().view(torch.int16)).view(np.uint16)
        np.testing.assert_array_equal(got_s, ref_s)
        assert (to_np(codes[:, :L - n]) == 0).all()


# ------------------------------------------------------------------ demand-mapped arena
def test_arena_grows_in_place():
    a = qsa.Arena(1 << 30)
    try:
        base, g = a.base, a.granularity
        assert base and a.mapped == 0 and a.reserved >= 1 << 30 and g > 0
        a.ensure(5_000_000)
        assert a.mapped >= 5_000_000 and a.mapped % g == 0
        v = a.tensor(0, (5_000_000 // 4,), torch.float32)
        v.copy_(torch.arange(v.numel(), device=dev(), dtype=torch.float32))
        a.ensure(300 << 20)
        assert a.base == base and a.mapped >= 300 << 20
        assert torch.equal(a.tensor(0, (5_000_000 // 4,), torch.float32),
                           torch.arange(5_000_000 // 4, device=dev(), dtype=torch.float32))
        w = a.tensor(a.mapped - 4096, (1024,), torch.float32)
        w.fill_(3.0)
        assert float(w.sum()) == 3072.0
        with pytest.raises(qsa.QSAError):
            a.ensure(a.reserved + 1)
    finally:
        a.destroy()


def test_arena_kv_cache_and_graph_survive_growth():
    # K and V of each token interleaved in one arena ([token][K|V][head][D]),
    # so the cache grows by mapping more of the same range; a CUDA graph
    # captured over the arena replays unchanged after growth.
    Hkv, D, cap = 2, 256, 16_384
    tok_bytes = 2 * Hkv * D * 2
    a = qsa.Arena(cap * tok_bytes)
    try:
        L1, L2, M = 6000, 12_000, 4
        x = make_layer(L=L2, M=M, dtype=torch.bfloat16, seed=51, device=dev())
        a.ensure(L1 * tok_bytes)

        def kv_views(L):
            t = a.tensor(0, (L, 2, Hkv, D), torch.bfloat16)
            return t[:, 0].permute(1, 0, 2), t[:, 1].permute(1, 0, 2)   # [Hkv, L, D] views, tok stride 2*Hkv*D

        def fill(t0, t1):
            t = a.tensor(0, (t1, 2, Hkv, D), torch.bfloat16)
            t[t0:t1, 0] = x.k[:, t0:t1].permute(1, 0, 2)
            t[t0:t1, 1] = x.v[:, t0:t1].permute(1, 0, 2)

        fill(0, L1)
        x1 = make_layer(L=L1, M=M, dtype=torch.bfloat16, seed=51, device=dev())
        sel, cnt, _ = _oracle_selection(x1)
        seld, cntd = torch.from_numpy(sel).to(dev()), torch.from_numpy(cnt).to(dev())
        q1 = x.q[:M].clone()
        ka, va = kv_views(L1)
        seqs1 = [qsa.Seq(L1, M, segments=[qsa.Segment(ka, va, 0)])]
        out_a = torch.empty((M, 24, D), device=dev())
        lse_a = torch.empty((M, 24), device=dev())
        ref_o = torch.empty_like(out_a)
        ref_l = torch.empty_like(lse_a)
        qsa.sparse_attn([qsa.Seq(L1, M, segments=[qsa.Segment(x.k[:, :L1].contiguous(), x.v[:, :L1].contiguous(),
                                                                0)])], q1, seld, cntd, ref_o, ref_l)
        qsa.sparse_attn(seqs1, q1, seld, cntd, out_a, lse_a)   # eager once (kernel attributes)
        torch.cuda.synchronize()
        assert torch.equal(out_a, ref_o) and torch.equal(lse_a, ref_l)
        g = torch.cuda.CUDAGraph()
        s_ = torch.cuda.Stream()
        with torch.cuda.graph(g, stream=s_):
            qsa.sparse_attn(seqs1, q1, seld, cntd, out_a, lse_a)
        # Grow: map and write tokens L1 .. L2 - 1; the base stays, the graph replays.
        base = a.base
        a.ensure(L2 * tok_bytes)
        fill(L1, L2)
        assert a.base == base
        out_a.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(out_a, ref_o) and torch.equal(lse_a, ref_l)
        # The grown cache against the oracle.
        sel2, cnt2, _ = _oracle_selection(x)
        kb, vb = kv_views(L2)
        out2, lse2 = torch.empty((M, 24, D), device=dev()), torch.empty((M, 24), device=dev())
        qsa.sparse_attn([qsa.Seq(L2, M, segments=[qsa.Segment(kb, vb, 0)])], x.q,
                        torch.from_numpy(sel2).to(dev()), torch.from_numpy(cnt2).to(dev()), out2, lse2)
        torch.cuda.synchronize()
        ref_out, ref_lse = oracle.attn(x.q, x.k, x.v, x.row_pos, sel2, cnt2)
        assert_attn_close(to_np(out2), to_np(lse2), ref_out, ref_lse, True)
        del ka, va, kb, vb
    finally:
        torch.cuda.synchronize()
        a.destroy()


# ------------------------------------------------------------------ steps 2 + 3 over key-axis chunks
def _blocked_vs_one_pass(seqs, q_idx, block_keys, top_k=512):
    """Selections of the chunked path and of score_blocks + select_topk."""
    rows = sum(sq.n_rows for sq in seqs)
    ld = max(1, max(sq.n_tokens // 4 for sq in seqs))
    ld = (ld + 3) // 4 * 4
    scores = torch.empty((rows, ld), dtype=torch.float32, device=dev())
    gm = torch.empty((rows, (qsa.n_groups(max(sq.n_tokens for sq in seqs)) + 3) // 4 * 4), device=dev())
    sel1 = torch.empty((rows, top_k), dtype=torch.int32, device=dev())
    cnt1 = torch.empty((rows,), dtype=torch.int32, device=dev())
    qsa.score_blocks(seqs, q_idx, scores, group_max=gm)
    qsa.select_topk(seqs, scores, sel1, cnt1, top_k, group_max=gm)
    sel2 = torch.full((rows, top_k), 12345, dtype=torch.int32, device=dev())
    cnt2 = torch.full((rows,), -7, dtype=torch.int32, device=dev())
    ws = torch.full((qsa.score_select_blocked_workspace_size(seqs, top_k, block_keys),), 0x7F, dtype=torch.uint8,
                    device=dev())
    qsa.score_select_topk_blocked(seqs, q_idx, sel2, cnt2, top_k, block_keys, workspace=ws)
    torch.cuda.synchronize()
    return to_np(sel1), to_np(cnt1), to_np(sel2), to_np(cnt2), scores


@pytest.mark.parametrize("L,M,block_keys", [(12_000, 600, 1024), (2500, 600, 128), (20_000, 520, 4096),
                                            (4099, 512, 256)])
def test_blocked_selection_equals_one_pass(L, M, block_keys):
    # Many rows score on the tensor cores in both paths, so the scores are the
    # same numbers and the selections must be identical.  Rows at small
    # positions see fewer than 512 blocks; the last chunk is ragged.
    x = make_layer(L=L, M=M, dtype=torch.bfloat16, seed=L + block_keys, device=dev())
    pooled = pooled_buffer(L, dev())
    pool_all(x.idxk, pooled, L)
    seqs = [qsa.Seq(L, M, pooled)]
    sel1, cnt1, sel2, cnt2, _ = _blocked_vs_one_pass(seqs, x.q_idx, block_keys)
    np.testing.assert_array_equal(cnt2, cnt1)
    np.testing.assert_array_equal(sel2, sel1)
    assert qsa.wait_timeouts() == 0


def test_blocked_selection_matches_oracle_and_ties():
    # A ragged batch (a prefill chunk and an 8-row verify); rows 0-2 of the
    # chunk have all-zero index queries, so every block ties at 0 and the
    # lowest ids must win.  Sampled rows against the oracle.
    xa = make_layer(L=9000, M=600, dtype=torch.bfloat16, seed=31, device=dev())
    xb = make_layer(L=5003, M=8, dtype=torch.bfloat16, seed=32, device=dev())
    xa.q_idx[:3] = 0
    pa, pb = pooled_buffer(9000, dev()), pooled_buffer(5003, dev())
    pool_all(xa.idxk, pa, 9000)
    pool_all(xb.idxk, pb, 5003)
    seqs = [qsa.Seq(9000, 600, pa), qsa.Seq(5003, 8, pb)]
    q_idx = torch.cat([xa.q_idx, xb.q_idx])
    sel1, cnt1, sel2, cnt2, _ = _blocked_vs_one_pass(seqs, q_idx, 1024)
    np.testing.assert_array_equal(cnt2, cnt1)
    np.testing.assert_array_equal(sel2, sel1)
    np.testing.assert_array_equal(sel2[0], np.arange(512))
    rows = [0, 1, 5, 300, 599]
    for x, sel, cnt, rr in ((xa, sel2[:600], cnt2[:600], rows), (xb, sel2[600:], cnt2[600:], list(range(8)))):
        h_idxk, h_q = x.idxk.cpu(), x.q_idx.cpu()
        pos = [x.row_pos[r] for r in rr]
        pooled_ref = oracle.pool(h_idxk)
        s_ref = oracle.score(h_q[rr], pooled_ref, pos)
        sel_ref, cnt_ref, tau = oracle.select(s_ref, pos)
        assert_selection_close(sel[rr], cnt[rr], sel_ref, cnt_ref, tau, s_ref, pos)


def test_blocked_selection_few_rows_matches_oracle():
    # Four rows: the one-pass path scores them on the few-row kernel (tf32
    # planes), the chunked path on the tensor cores; both against the oracle.
    L, M = 30_001, 4
    x = make_layer(L=L, M=M, dtype=torch.bfloat16, seed=33, device=dev())
    pooled = pooled_buffer(L, dev())
    pool_all(x.idxk, pooled, L)
    seqs = [qsa.Seq(L, M, pooled)]
    _, _, sel2, cnt2, _ = _blocked_vs_one_pass(seqs, x.q_idx, 2048)
    pooled_ref = oracle.pool(x.idxk.cpu())
    s_ref = oracle.score(x.q_idx.cpu(), pooled_ref, x.row_pos)
    sel_ref, cnt_ref, tau = oracle.select(s_ref, x.row_pos)
    assert_selection_close(sel2, cnt2, sel_ref, cnt_ref, tau, s_ref, x.row_pos)


# ------------------------------------------------------------------ step 4 (given the oracle's selection)
def _oracle_selection(x):
    pooled = oracle.pool(x.idxk)
    s = oracle.score(x.q_idx, pooled, x.row_pos)
    return oracle.select(s, x.row_pos)


def _attn_gpu(x, sel, cnt, *, segments=None, out_dtype=torch.float32, n_splits=0, device=None):
    device = device or dev()
    q = x.q.to(device)
    k, v = x.k.to(device), x.v.to(device)
    segs = segments(k, v) if segments else [qsa.Segment(k, v, 0)]
    out = torch.full((x.M, x.q.shape[1], x.q.shape[2]), float("nan"), dtype=out_dtype, device=device)
    lse = torch.full((x.M, x.q.shape[1]), float("nan"), device=device)
    seld = torch.from_numpy(np.ascontiguousarray(sel)).to(device)
    cntd = torch.from_numpy(np.ascontiguousarray(cnt)).to(device)
    qsa.sparse_attn([qsa.Seq(x.L, x.M, segments=segs)], q, seld, cntd, out, lse, n_splits=n_splits,
                    n_kv_heads=x.k.shape[0])
    torch.cuda.synchronize()
    return to_np(out.float()), to_np(lse)


@pytest.mark.parametrize("dtype,D", [(torch.float32, 256), (torch.bfloat16, 256), (torch.float32, 128),
                                     (torch.bfloat16, 128)])
@pytest.mark.parametrize("n_splits", [0, 1, 3, 16, 40])
def test_attention_matches_oracle(dtype, D, n_splits):
    x = make_layer(L=4099, M=4, dtype=dtype, seed=3, head_dim=D)
    sel, cnt, _ = _oracle_selection(x)
    out, lse = _attn_gpu(x, sel, cnt, n_splits=n_splits)
    ref_out, ref_lse = oracle.attn(x.q, x.k, x.v, x.row_pos, sel, cnt)
    assert_attn_close(out, lse, ref_out, ref_lse, dtype == torch.bfloat16)


# Other grouped-query shapes (up to 16 query heads per KV head), on the
# few-row path and on the tensor-core path (>= 512 rows).
@pytest.mark.parametrize("Hq,Hkv,M,D", [(32, 2, 4, 256), (8, 1, 4, 128), (4, 4, 3, 128), (32, 2, 520, 128),
                                        (8, 1, 600, 256), (16, 4, 512, 128)])
def test_attention_other_head_groupings(Hq, Hkv, M, D):
    L = 9001 if M <= 8 else 1500
    x = make_layer(L=L, M=M, dtype=torch.bfloat16, seed=7 * Hq + Hkv + M, n_q_heads=Hq, n_kv_heads=Hkv, head_dim=D)
    sel, cnt, _ = _oracle_selection(x)
    out, lse = _attn_gpu(x, sel, cnt)
    ref_out, ref_lse = oracle.attn(x.q, x.k, x.v, x.row_pos, sel, cnt)
    assert_attn_close(out, lse, ref_out, ref_lse, True)


# Budgets other than 512 blocks: lists of 4 top_k + tail entries (900 blocks
# at 520 rows fill 29 of the tensor-core path's 30 logit tiles; 1,024 blocks
# exceed them and run split-free on the warp-level path).
@pytest.mark.parametrize("top_k,M", [(64, 4), (1024, 4), (900, 520), (1024, 520)])
def test_attention_other_budgets(top_k, M):
    L = 20_011 if M <= 8 else 5000
    x = make_layer(L=L, M=M, dtype=torch.bfloat16, seed=top_k + M, head_dim=128)
    s = oracle.score(x.q_idx, oracle.pool(x.idxk), x.row_pos)
    sel, cnt, _ = oracle.select(s, x.row_pos, top_k)
    out, lse = _attn_gpu(x, sel, cnt)
    ref_out, ref_lse = oracle.attn(x.q, x.k, x.v, x.row_pos, sel, cnt)
    assert_attn_close(out, lse, ref_out, ref_lse, True)


# The split count the plan picks follows the number of rows (about two CTAs
# per SM over the call): 64 splits for one row down to 2 for 100 rows.
@pytest.mark.parametrize("M,D,out_dtype", [(1, 256, torch.float32), (16, 256, torch.float32),
                                           (32, 128, torch.bfloat16), (100, 256, torch.float32),
                                           (4, 128, torch.bfloat16)])
def test_attention_auto_split_counts(M, D, out_dtype):
    x = make_layer(L=9001, M=M, dtype=torch.bfloat16, seed=M + D, head_dim=D)
    sel, cnt, _ = _oracle_selection(x)
    out, lse = _attn_gpu(x, sel, cnt, out_dtype=out_dtype)
    ref_out, ref_lse = oracle.attn(x.q, x.k, x.v, x.row_pos, sel, cnt)
    assert_attn_close(out, lse, ref_out, ref_lse, True)


def test_attention_many_splits_reuse_workspace():
    # 40 splits per (row, KV group) merge through the workspace; a second call
    # on the same (now dirty) workspace gives the same result.
    x = make_layer(L=9001, M=3, dtype=torch.bfloat16, seed=13)
    sel, cnt, _ = _oracle_selection(x)
    q, k, v = x.q.to(dev()), x.k.to(dev()), x.v.to(dev())
    seqs = [qsa.Seq(x.L, x.M, segments=[qsa.Segment(k, v, 0)])]
    seld, cntd = torch.from_numpy(sel).to(dev()), torch.from_numpy(cnt).to(dev())
    cfg = qsa.attn_config(q, 2, torch.float32, 0.0, 40)
    need = qsa.attn_workspace_size(seqs, cfg, sel.shape[1])
    assert need > 0
    ws = torch.full((need,), 0x7F, dtype=torch.uint8, device=dev())
    outs = []
    for _ in range(2):
        out = torch.full((x.M, 24, 256), float("nan"), device=dev())
        lse = torch.full((x.M, 24), float("nan"), device=dev())
        qsa.sparse_attn(seqs, q, seld, cntd, out, lse, workspace=ws, cfg=cfg)
        torch.cuda.synchronize()
        outs.append((to_np(out), to_np(lse)))
    ref_out, ref_lse = oracle.attn(x.q, x.k, x.v, x.row_pos, sel, cnt)
    for o, l in outs:
        assert_attn_close(o, l, ref_out, ref_lse, True)
    np.testing.assert_array_equal(outs[0][0], outs[1][0])


def test_attention_bf16_output():
    x = make_layer(L=6007, M=2, dtype=torch.bfloat16, seed=4)
    sel, cnt, _ = _oracle_selection(x)
    out, lse = _attn_gpu(x, sel, cnt, out_dtype=torch.bfloat16)
    ref_out, ref_lse = oracle.attn(x.q, x.k, x.v, x.row_pos, sel, cnt)
    assert_attn_close(out, lse, ref_out, ref_lse, True)


@pytest.mark.parametrize("L,M", [(1, 1), (2, 2), (3, 1), (4, 4), (5, 3), (7, 1), (9, 4), (2051, 4), (2052, 1),
                                 (2055, 4), (4096, 1), (333, 8)])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_attention_degenerate_sizes(L, M, dtype):
    x = make_layer(L=L, M=M, dtype=dtype, seed=L, head_dim=128)
    sel, cnt, _ = _oracle_selection(x)
    out, lse = _attn_gpu(x, sel, cnt)
    ref_out, ref_lse = oracle.attn(x.q, x.k, x.v, x.row_pos, sel, cnt)
    assert_attn_close(out, lse, ref_out, ref_lse, dtype == torch.bfloat16)


def test_attention_skips_invalid_ids():
    # Out-of-range ids in the selection are skipped (never dereferenced);
    # the result equals attention without them.
    x = make_layer(L=3001, M=2, dtype=torch.bfloat16, seed=6)
    sel, cnt, _ = _oracle_selection(x)
    bad = sel.copy()
    bad[0, 3] = 10_000_000
    bad[1, 5] = -5
    out, lse = _attn_gpu(x, bad, cnt)
    keep0 = np.delete(sel[0, :cnt[0]], 3)
    keep1 = np.delete(sel[1, :cnt[1]], 5)
    ref_sel = np.full_like(sel, -1)
    ref_sel[0, :len(keep0)] = keep0
    ref_sel[1, :len(keep1)] = keep1
    ref_out, ref_lse = oracle.attn(x.q, x.k, x.v, x.row_pos, ref_sel, [len(keep0), len(keep1)])
    assert_attn_close(out, lse, ref_out, ref_lse, True)


# ------------------------------------------------------------------ step 4 on the tensor cores
# Calls with at least 512 query rows and a single split (chunked prefill) run
# on tcgen05; two forced splits take the mma.sync kernel and the merge on the
# same inputs.  Rows at small positions give short, ragged lists (2 to 10
# tiles of 128 tokens); the 6,000-token case gives full 2,051-entry lists.
@pytest.mark.parametrize("L,M,D", [(1200, 1000, 256), (6000, 600, 256), (1200, 700, 128)])
def test_attention_tensor_cores_matches_oracle(L, M, D):
    x = make_layer(L=L, M=M, dtype=torch.bfloat16, seed=L + M, head_dim=D)
    sel, cnt, _ = _oracle_selection(x)
    ref_out, ref_lse = oracle.attn(x.q, x.k, x.v, x.row_pos, sel, cnt)
    out, lse = _attn_gpu(x, sel, cnt)
    assert_attn_close(out, lse, ref_out, ref_lse, True)
    out2, lse2 = _attn_gpu(x, sel, cnt, n_splits=2)
    assert_attn_close(out2, lse2, ref_out, ref_lse, True)
    assert qsa.wait_timeouts() == 0


def test_attention_tensor_cores_edge_cases():
    # Out-of-range ids (skipped), a row with an empty list (count 0, no tail:
    # zeros and lse = -inf), KV segments with a hole, bf16 output.
    x = make_layer(L=2600, M=560, dtype=torch.bfloat16, seed=21)
    sel, cnt, _ = _oracle_selection(x)
    bad, bad_cnt = sel.copy(), cnt.copy()
    bad[1, 3] = 10_000_000
    bad[2, 5] = -5
    assert (x.row_pos[3] + 1) % 4 == 0
    bad_cnt[3] = 0
    ref_sel, ref_cnt = sel.copy(), cnt.copy()
    for r, j in ((1, 3), (2, 5)):
        keep = np.delete(sel[r, :cnt[r]], j)
        ref_sel[r] = -1
        ref_sel[r, :len(keep)] = keep
        ref_cnt[r] = len(keep)
    ref_cnt[3] = 0
    cuts = segment_cuts(x.L, 5, seed=3)
    kept = cuts[:2] + cuts[3:]
    vis = np.zeros(x.L, dtype=bool)
    for f, n in kept:
        vis[f:f + n] = True
    ref_out, ref_lse = oracle.attn(x.q, x.k, x.v, x.row_pos, ref_sel, ref_cnt, visible=vis)
    out, lse = _attn_gpu(x, bad, bad_cnt, segments=_segment_views(kept), out_dtype=torch.bfloat16)
    assert_attn_close(out, lse, ref_out, ref_lse, True)
    assert (out[3] == 0).all() and np.isneginf(lse[3]).all()
    assert qsa.wait_timeouts() == 0


# ------------------------------------------------------------------ segments and step 5
def _segment_views(cuts):
    def make(k, v):
        # Each segment is a separate allocation holding its tokens.
        return [qsa.Segment(k[:, f:f + n].clone(), v[:, f:f + n].clone(), f) for f, n in cuts]
    return make


@pytest.mark.parametrize("D", [256, 128])
def test_segmented_equals_single_buffer_and_oracle(D):
    x = make_layer(L=9001, M=4, dtype=torch.bfloat16, seed=7, head_dim=D)
    sel, cnt, _ = _oracle_selection(x)
    ref_out, ref_lse = oracle.attn(x.q, x.k, x.v, x.row_pos, sel, cnt)
    cuts = segment_cuts(x.L, 12, seed=1)
    single, single_lse = _attn_gpu(x, sel, cnt)
    seg, seg_lse = _attn_gpu(x, sel, cnt, segments=_segment_views(cuts))
    assert_attn_close(seg, seg_lse, ref_out, ref_lse, True)
    np.testing.assert_allclose(seg, single, atol=2e-3)
    # Per-segment calls merged by the step-5 entry point.
    parts_o, parts_l = [], []
    for f, n in cuts:
        o, l = _attn_gpu(x, sel, cnt, segments=_segment_views([(f, n)]))
        parts_o.append(o.reshape(-1, D))
        parts_l.append(l.reshape(-1))
    po = torch.from_numpy(np.stack(parts_o)).to(dev())
    pl = torch.from_numpy(np.stack(parts_l)).to(dev())
    merged = torch.empty((po.shape[1], D), device=dev())
    mlse = torch.empty((po.shape[1],), device=dev())
    qsa.lse_merge(po, pl, merged, mlse)
    assert_attn_close(to_np(merged).reshape(ref_out.shape), to_np(mlse).reshape(ref_lse.shape), ref_out, ref_lse,
                      True)


def test_segment_hole_matches_visibility_mask():
    x = make_layer(L=7000, M=3, dtype=torch.bfloat16, seed=8)
    sel, cnt, _ = _oracle_selection(x)
    cuts = segment_cuts(x.L, 5, seed=2)
    kept = cuts[:2] + cuts[3:]
    vis = np.zeros(x.L, dtype=bool)
    for f, n in kept:
        vis[f:f + n] = True
    out, lse = _attn_gpu(x, sel, cnt, segments=_segment_views(kept))
    ref_out, ref_lse = oracle.attn(x.q, x.k, x.v, x.row_pos, sel, cnt, visible=vis)
    assert_attn_close(out, lse, ref_out, ref_lse, True)
    # Only a segment far from every selected row: no visible key -> zeros, -inf.
    far = lambda k, v: [qsa.Segment(k[:, 0:4].clone(), v[:, 0:4].clone(), 10 ** 9)]
    out0, lse0 = _attn_gpu(x, sel, cnt, segments=far)
    assert (out0 == 0).all() and np.isneginf(lse0).all()


@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
def test_lse_merge_matches_oracle(out_dtype):
    rng = np.random.default_rng(9)
    S, R, D = 5, 300, 256
    o = rng.standard_normal((S, R, D)).astype(np.float32)
    l = (rng.standard_normal((S, R)) * 4).astype(np.float32)
    l[:, 7] = -np.inf                    # a row no part saw a key for
    l[2, 11:40] = -np.inf                # parts without keys for some rows
    out = torch.empty((R, D), dtype=out_dtype, device=dev())
    lse = torch.empty((R,), device=dev())
    qsa.lse_merge(torch.from_numpy(o).to(dev()), torch.from_numpy(l).to(dev()), out, lse)
    ref_o, ref_l = oracle.lse_merge(o.astype(np.float64), l.astype(np.float64))
    got = to_np(out.float())
    assert not np.isnan(got).any()
    tol = 1e-5 if out_dtype == torch.float32 else 1e-2
    np.testing.assert_allclose(got, ref_o, atol=tol, rtol=tol)
    fin = np.isfinite(ref_l)
    np.testing.assert_allclose(to_np(lse)[fin], ref_l[fin], atol=1e-5)
    assert np.isneginf(to_np(lse)[~fin]).all() and (got[7] == 0).all()


# ------------------------------------------------------------------ whole layer step
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_layer_step_tiny_verify(dtype):
    # 4,099 tokens, four verify rows at 4,095..4,098, 64 planted blocks.
    x = make_layer(L=4099, M=4, dtype=dtype, seed=0, n_planted=64)
    g = DeviceLayer(x).run()
    ref = oracle_layer(x)
    pooled_ref = oracle.pool(x.idxk)
    bound = score_bound(x.q_idx, pooled_ref, x.row_pos)
    nb = ref["scores"].shape[1]
    assert_scores_close(to_np(g.scores)[:, :nb], ref["scores"], 2 * bound, x.row_pos)
    sel, cnt = to_np(g.sel), to_np(g.cnt)
    assert_selection_close(sel, cnt, ref["sel"], ref["cnt"], ref["tau"], ref["scores"], x.row_pos)
    # Attention over the GPU's own selection against the oracle on that selection.
    ref_out, ref_lse = oracle.attn(x.q, x.k, x.v, x.row_pos, sel, cnt)
    assert_attn_close(to_np(g.out), to_np(g.lse), ref_out, ref_lse, dtype == torch.bfloat16)
    # The tail is attended: the row at 4,098 has 2,048 + 3 rows (lse vs q=0 is checked by the oracle pins).
    assert list(cnt) == [512] * 4


def test_layer_step_ragged_batch_small():
    # Several sequences in one call (decode and verify rows), bf16, segmented K/V.
    Ls, Ms, nsegs = [4099, 9001, 2051, 17_000], [1, 4, 2, 4], [3, 12, 1, 5]
    xs = [make_layer(L=L, M=M, dtype=torch.bfloat16, seed=20 + i, head_dim=128) for i, (L, M) in
          enumerate(zip(Ls, Ms))]
    seqs, keep = [], []
    for i, x in enumerate(xs):
        k, v = x.k.to(dev()), x.v.to(dev())
        idxk = x.idxk.to(dev())
        pooled = pooled_buffer(x.L, dev())
        pool_all(idxk, pooled, x.L)
        segs = _segment_views(segment_cuts(x.L, nsegs[i], seed=i))(k, v)
        seqs.append(qsa.Seq(x.L, x.M, pooled, segs, idx_keys=idxk))
        keep += [k, v, idxk, pooled]
    q_idx = torch.cat([x.q_idx for x in xs]).to(dev())
    q = torch.cat([x.q for x in xs]).to(dev())
    step = qsa.LayerStep(seqs, q_idx, q)
    step.run()
    torch.cuda.synchronize()
    # The fused scoring + selection entry point gives the same selection.
    sel0, cnt0 = step.sel.clone(), step.cnt.clone()
    step.sel.fill_(-5)
    step.cnt.fill_(-5)
    step.score_select()
    torch.cuda.synchronize()
    assert torch.equal(step.sel, sel0) and torch.equal(step.cnt, cnt0)
    row = 0
    for x in xs:
        ref = oracle_layer(x)
        rows = slice(row, row + x.M)
        sel, cnt = to_np(step.sel)[rows], to_np(step.cnt)[rows]
        assert_selection_close(sel, cnt, ref["sel"], ref["cnt"], ref["tau"], ref["scores"], x.row_pos)
        ref_out, ref_lse = oracle.attn(x.q, x.k, x.v, x.row_pos, sel, cnt)
        assert_attn_close(to_np(step.out)[rows], to_np(step.lse)[rows], ref_out, ref_lse, True)
        row += x.M


def test_layer_step_rows_at_any_position():
    # A row at position p sees tokens 0..p only, so a descriptor whose
    # n_tokens is its last row's position + 1 places a run of consecutive
    # rows anywhere in a longer cache (the last run below ends two tokens
    # before the cache's end), and rows at scattered positions are several
    # descriptors over one cache: the same pooled keys and K/V segments.
    L = 9001
    runs = [(1203, 1), (5000, 2), (7003, 1), (8997, 2)]   # (first position, rows)
    row_pos = [p + j for p, n in runs for j in range(n)]
    x = make_layer(L=L, M=len(row_pos), dtype=torch.bfloat16, seed=41, head_dim=256)
    k, v, idxk = x.k.to(dev()), x.v.to(dev()), x.idxk.to(dev())
    pooled = pooled_buffer(L, dev())
    pool_all(idxk, pooled, L)
    segs = [qsa.Segment(k, v, 0)]
    seqs = [qsa.Seq(p + n, n, pooled, segs, idx_keys=idxk) for p, n in runs]
    step = qsa.LayerStep(seqs, x.q_idx.to(dev()), x.q.to(dev()))
    step.run()
    torch.cuda.synchronize()
    ref = oracle.layer_step(x.q_idx, x.idxk, x.q, x.k, x.v, row_pos)
    sel, cnt = to_np(step.sel), to_np(step.cnt)
    assert_selection_close(sel, cnt, ref["sel"], ref["cnt"], ref["tau"], ref["scores"], row_pos)
    ref_out, ref_lse = oracle.attn(x.q, x.k, x.v, row_pos, sel, cnt)
    assert_attn_close(to_np(step.out), to_np(step.lse), ref_out, ref_lse, True)
    # The pooled keys the step rewrote (each run's completed block) are the oracle's.
    assert_pooled_close(to_np(pooled), x.idxk, [(p + n) // 4 - 1 for p, n in runs])


# ------------------------------------------------------------------ device-side checks
def test_device_status_clean_after_normal_work():
    qsa.check_device_status()   # clears what earlier tests left
    L, M = 9001, 4
    x = make_layer(L=L, M=M, dtype=torch.bfloat16, seed=71, device=dev())
    pooled = pooled_buffer(L, dev())
    qsa.pool_index_keys(x.idxk, pooled, 0, L // 4)
    step = qsa.LayerStep([qsa.Seq(L, M, pooled, [qsa.Segment(x.k, x.v, 0)], idx_keys=x.idxk)], x.q_idx, x.q)
    step.run()
    assert qsa.check_device_status() == (0, "")


@pytest.mark.parametrize("L,M", [(3001, 2), (1200, 600)])
def test_device_status_reports_out_of_range_ids(L, M):
    # Few rows (warp-level path) and >= 512 rows (tensor cores): the bad ids
    # are skipped and counted.
    qsa.check_device_status()
    x = make_layer(L=L, M=M, dtype=torch.bfloat16, seed=L + M)
    sel, cnt, _ = _oracle_selection(x)
    bad = sel.copy()
    bad[0, 3] = 10_000_000
    bad[M - 1, 5] = -5
    _attn_gpu(x, bad, cnt)
    st, why = qsa.check_device_status()
    assert st == qsa.ERR_DEVICE_CHECK and "out-of-range" in why
    assert qsa.check_device_status() == (0, "")     # read and cleared


def test_device_status_reports_nan_scores():
    qsa.check_device_status()
    L, M = 20_011, 2
    rng = np.random.default_rng(3)
    s = np.abs(rng.standard_normal((M, (L // 4 + 3) // 4 * 4))).astype(np.float32)
    s[0, 64:80] = 100.0        # the group of block 77 is surely a candidate
    s[0, 77] = np.nan
    _select_gpu(s, [L - M + j for j in range(M)], L)
    st, why = qsa.check_device_status()
    assert st == qsa.ERR_DEVICE_CHECK and "NaN" in why


def test_device_status_reports_expired_wait():
    # One wait on a barrier nothing completes, limited to 2 ms: reported as a
    # timeout, and the context stays usable.
    qsa.check_device_status()
    before = qsa.wait_timeouts()
    qsa.selftest_wait_timeout(2000)
    st, why = qsa.check_device_status()
    assert st == qsa.ERR_TIMEOUT and "gave up" in why
    assert qsa.wait_timeouts() == before          # the library's own kernels are not blamed
    x = make_layer(L=2052, M=1, dtype=torch.bfloat16, seed=9)
    sel, cnt, _ = _oracle_selection(x)
    out, lse = _attn_gpu(x, sel, cnt)
    ref_out, ref_lse = oracle.attn(x.q, x.k, x.v, x.row_pos, sel, cnt)
    assert_attn_close(out, lse, ref_out, ref_lse, True)
    assert qsa.check_device_status() == (0, "")
