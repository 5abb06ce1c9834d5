"""Pins of the fp64 CPU oracle against facts that do not come from the oracle.

Each test ties one step of the oracle to a closed form, a special case that
reduces to a library routine, an invariant, or a number the pages print, so
that a plausible slip in the oracle (a dropped term, a wrong sign or index, a
transposed operand, an off-by-one in the block or tail bookkeeping) fails.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from workloads import make_layer, segment_cuts

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---------------------------------------------------------------- block bookkeeping

def test_block_counts_and_tails():
    # Block b holds tokens 4b..4b+3; a row at p sees floor((p+1)/4) complete
    # blocks and (p+1) mod 4 tail tokens.
    assert [oracle.visible_blocks(p) for p in (0, 1, 2, 3, 4, 7)] == [0, 0, 0, 1, 1, 2]
    assert [oracle.tail_tokens(p) for p in (0, 1, 2, 3, 4, 7)] == [1, 2, 3, 0, 1, 0]
    # 4,099-token context: 1,025 pooled slots, 1,024 complete; the four verify
    # rows at 4,095..4,098 have tails 0, 1, 2, 3.
    assert math.ceil(4099 / 4) == 1025
    assert [oracle.visible_blocks(p) for p in range(4095, 4099)] == [1024] * 4
    assert [oracle.tail_tokens(p) for p in range(4095, 4099)] == [0, 1, 2, 3]
    # 261,120 tokens: 65,280 complete blocks and no tail on the last row.
    assert oracle.visible_blocks(261_119) == 65_280 and oracle.tail_tokens(261_119) == 0


def test_page_state_sizes_match_shapes():
    g = json.load(open(os.path.join(GOLDEN, "state_sizes.json")))
    n_kv_heads, head_dim, f32 = 2, 256, 4
    kv = 2 * n_kv_heads * head_dim * f32                        # K and V
    index_key = oracle.INDEX_DIM * f32                          # one per token
    pooled = oracle.INDEX_DIM * f32 / oracle.BLOCK_TOKENS       # one per 4 tokens
    assert kv + index_key + pooled == g["f32_bytes_per_token_per_layer"]
    mib = g["f32_bytes_per_token_per_layer"] * g["max_context_tokens"] * g["qsa_layers"] / 2**20
    assert mib == g["f32_context_state_mib"]
    assert oracle.TOP_K == g["block_budget"] and oracle.TOP_K * oracle.BLOCK_TOKENS == g["token_budget"]
    assert g["token_budget"] + 3 == g["max_rows_per_query"]
    mb = 2 * g["bf16_key_buffer_capacity"] * head_dim * 2 / 1e6
    assert round(mb) == g["bf16_key_buffer_mb_about"]


# ---------------------------------------------------------------- step 1: pooling

def test_pool_closed_form_arithmetic_sequence():
    # idxk[t, d] = t + d/2 -> the mean over a block's tokens 4b..4b+3 is 4b + 1.5 + d/2.
    L, dim = 23, 128
    t = np.arange(L, dtype=np.float64)[:, None]
    d = np.arange(dim, dtype=np.float64)[None, :]
    idxk = (t + d / 2).astype(np.float32)
    pooled = oracle.pool(idxk)
    assert pooled.shape == (L // 4, dim)
    b = np.arange(L // 4, dtype=np.float64)[:, None]
    np.testing.assert_array_equal(pooled, 4 * b + 1.5 + d / 2)
    # An offset range pools the same blocks.
    np.testing.assert_array_equal(oracle.pool(idxk, first_block=2, n_blocks=3), pooled[2:5])
    with pytest.raises(ValueError):
        oracle.pool(idxk, first_block=5, n_blocks=1)   # tokens 20..23: block not complete


def test_pool_reads_bf16_exactly():
    x = torch.randn(16, 128).to(torch.bfloat16)
    want = x.double().view(4, 4, 128).mean(dim=1).numpy()
    np.testing.assert_allclose(oracle.pool(x), want, rtol=0, atol=1e-15)


# ---------------------------------------------------------------- step 2: scoring

def test_score_closed_form_unit_heads():
    # Head h of the index query is the unit vector e_h; the pooled key starts
    # [1, -2, 3, 4]: dots 1, -2, 3, 4 -> ReLU sum 8 -> 8 / sqrt(128) = 1/sqrt(2).
    q_idx = np.zeros((1, 4, 128))
    for h in range(4):
        q_idx[0, h, h] = 1.0
    pooled = np.zeros((1, 128))
    pooled[0, :4] = [1.0, -2.0, 3.0, 4.0]
    s = oracle.score(q_idx, pooled, row_pos=[3])
    assert s.shape == (1, 1)
    assert abs(s[0, 0] - 1 / math.sqrt(2)) < 1e-15
    # Flipping the sign of the key makes only head 1 positive: 2 / sqrt(128).
    s2 = oracle.score(q_idx, -pooled, row_pos=[3])
    assert abs(s2[0, 0] - 2 / math.sqrt(128)) < 1e-15


def test_score_nonnegative_inputs_reduce_to_one_matvec():
    # With every entry >= 0 the ReLU is the identity, so the four-head sum is
    # one matrix-vector product with the summed index query.
    rng = np.random.default_rng(1)
    q_idx = rng.random((3, 4, 128))
    pooled = rng.random((40, 128))
    pos = [159, 160, 161]
    s = oracle.score(q_idx, pooled, row_pos=pos)
    for r, p in enumerate(pos):
        nb = (p + 1) // 4
        want = (pooled[:nb] @ q_idx[r].sum(axis=0)) / math.sqrt(128)
        np.testing.assert_allclose(s[r, :nb], want, rtol=1e-13)
        assert np.all(np.isneginf(s[r, nb:]))


def test_score_invariants():
    rng = np.random.default_rng(2)
    q_idx = rng.standard_normal((2, 4, 128))
    pooled = rng.standard_normal((64, 128))
    pos = [255, 255]
    s = oracle.score(q_idx, pooled, row_pos=pos)
    assert np.all(s >= 0)
    # Permuting the index heads leaves the score unchanged.
    s_perm = oracle.score(q_idx[:, [2, 0, 3, 1]], pooled, row_pos=pos)
    np.testing.assert_allclose(s, s_perm, rtol=1e-13)
    # A zero index query scores every block 0.
    assert np.all(oracle.score(np.zeros_like(q_idx), pooled, row_pos=pos) == 0)
    # Causality: a row at p = 9 sees blocks 0 and 1 only.
    s3 = oracle.score(q_idx[:1], pooled, row_pos=[9])
    assert np.all(np.isfinite(s3[0, :2])) and np.all(np.isneginf(s3[0, 2:]))


# ---------------------------------------------------------------- step 3: selection

def _brute_topk(scores_row, nb, k):
    order = sorted(range(nb), key=lambda b: (-scores_row[b], b))
    return sorted(order[:k])


def test_select_matches_python_sort_on_tiny_inputs():
    rng = np.random.default_rng(3)
    for trial in range(50):
        nb = int(rng.integers(1, 40))
        k = int(rng.integers(1, 12))
        # coarse values so that ties are common
        row = rng.integers(0, 6, size=nb).astype(np.float64) * 0.25
        p = 4 * nb - 1 + int(rng.integers(0, 4))      # nb complete blocks, tail 0..3
        sel, cnt, tau = oracle.select(row[None, :], [p], top_k=k)
        want = _brute_topk(row, oracle.visible_blocks(p), k)
        assert cnt[0] == len(want)
        assert sel[0, :cnt[0]].tolist() == want
        assert np.all(sel[0, cnt[0]:] == -1)


def test_select_special_cases():
    nb = 2000
    p = 4 * nb - 1
    # All ties: the lower ids win -> blocks 0..511.
    sel, cnt, tau = oracle.select(np.zeros((1, nb)), [p])
    assert cnt[0] == 512 and sel[0].tolist() == list(range(512)) and tau[0] == 0.0
    # Strictly increasing scores -> the last 512 blocks.
    sel, cnt, tau = oracle.select(np.arange(nb, dtype=np.float64)[None], [p])
    assert sel[0].tolist() == list(range(nb - 512, nb)) and tau[0] == nb - 512
    # Ties straddling the threshold: ids 0..505 score 9 and ids 1000..1009
    # score 5, so the six lowest of the tied tens are kept.
    row = np.zeros(nb)
    row[:506] = 9.0
    row[100:110] = 9.0
    row[1000:1010] = 5.0
    sel, cnt, _ = oracle.select(row[None], [p])
    assert sel[0].tolist() == list(range(506)) + list(range(1000, 1006))
    # top_k = 1 is numpy's argmax (first index of the maximum).
    rowr = np.random.default_rng(4).integers(0, 50, size=nb).astype(np.float64)
    sel, cnt, _ = oracle.select(rowr[None], [p], top_k=1)
    assert sel[0, 0] == int(np.argmax(rowr))
    # Fewer complete blocks than the budget: all of them, no threshold.
    sel, cnt, tau = oracle.select(np.ones((1, 100)), [399])
    assert cnt[0] == 100 and sel[0, :100].tolist() == list(range(100)) and np.isneginf(tau[0])
    # -0.0 ties with +0.0 (IEEE equality), so the lower id wins.
    row0 = np.array([0.0, -0.0, 0.0, 1.0])
    sel, cnt, _ = oracle.select(row0[None], [15], top_k=2)
    assert sel[0].tolist() == [0, 3]


def test_row_tokens_bound_and_tail():
    # |R_r| = 4 * min(512, nb) + tail <= 2,048 + 3, and the tail is always in.
    for p in (4095, 4096, 4097, 4098, 261_119, 10, 0):
        nb = oracle.visible_blocks(p)
        k = min(512, nb)
        sel_row = np.arange(nb - k, nb, dtype=np.int32)
        toks = oracle.row_tokens(p, sel_row, k)
        assert len(toks) == 4 * k + oracle.tail_tokens(p) <= 2051
        tail = list(range(4 * nb, p + 1))
        assert toks[len(toks) - len(tail):].tolist() == tail
        assert toks.max() <= p


# ---------------------------------------------------------------- step 4: attention

def _all_selected(M_pos, top_k=512):
    sel = np.full((len(M_pos), top_k), -1, dtype=np.int32)
    cnt = np.zeros(len(M_pos), dtype=np.int32)
    for r, p in enumerate(M_pos):
        nb = oracle.visible_blocks(p)
        assert nb <= top_k
        sel[r, :nb] = np.arange(nb)
        cnt[r] = nb
    return sel, cnt


def test_attention_zero_query_is_mean_and_log_count():
    # q = 0: every selected row weighs the same, so out = mean of V over R_r
    # and lse = ln |R_r| -- pins the row set, its size and the tail.
    x = make_layer(L=4099, M=4, seed=5, n_planted=0, head_dim=64)
    q = torch.zeros_like(x.q)
    pooled = oracle.pool(x.idxk)
    s = oracle.score(x.q_idx, pooled, x.row_pos)
    sel, cnt, _ = oracle.select(s, x.row_pos)
    out, lse = oracle.attn(q, x.k, x.v, x.row_pos, sel, cnt)
    v = x.v.double().numpy()
    for r, p in enumerate(x.row_pos):
        nb = oracle.visible_blocks(p)
        rows = [4 * b + j for b in sel[r, :cnt[r]] for j in range(4)] + list(range(4 * nb, p + 1))
        assert len(rows) == 2048 + (p + 1) % 4
        np.testing.assert_allclose(lse[r], math.log(len(rows)), rtol=0, atol=1e-12)
        for h in range(24):
            np.testing.assert_allclose(out[r, h], v[h // 12, rows].mean(axis=0), atol=1e-12)


def test_attention_dense_case_equals_torch_sdpa():
    # Context <= 2,048 + 3 tokens: every complete block fits the budget, so QSA
    # is plain causal grouped-query attention (torch's SDPA, fp64).
    L, M, D = 1203, 5, 64
    x = make_layer(L=L, M=M, seed=6, head_dim=D)
    sel, cnt = _all_selected(x.row_pos)
    out, lse = oracle.attn(x.q, x.k, x.v, x.row_pos, sel, cnt)
    q = x.q.double().permute(1, 0, 2)                       # [Hq, M, D]
    k = x.k.double().repeat_interleave(12, dim=0)            # [Hq, L, D]
    v = x.v.double().repeat_interleave(12, dim=0)
    mask = torch.arange(L)[None, :] <= torch.tensor(x.row_pos)[:, None]
    ref = torch.nn.functional.scaled_dot_product_attention(q, k, v, attn_mask=mask)
    np.testing.assert_allclose(out, ref.permute(1, 0, 2).numpy(), atol=1e-12)
    logits = torch.einsum("hmd,hld->hml", q, k) / math.sqrt(D)
    ref_lse = torch.logsumexp(logits.masked_fill(~mask, float("-inf")), dim=-1)
    np.testing.assert_allclose(lse, ref_lse.T.numpy(), atol=1e-11)


def test_attention_gqa_head_mapping():
    # Heads 0..11 read KV head 0 and heads 12..23 read KV head 1: zeroing V of
    # KV head 1 zeroes exactly the outputs of heads 12..23.
    x = make_layer(L=300, M=2, seed=7, head_dim=32)
    sel, cnt = _all_selected(x.row_pos)
    v = x.v.clone()
    v[1] = 0
    out, _ = oracle.attn(x.q, x.k, v, x.row_pos, sel, cnt)
    assert np.all(out[:, 12:] == 0) and np.all(np.abs(out[:, :12]).sum(axis=-1) > 0)


def test_attention_single_key():
    # A row at position 0 sees one token (its own, the tail): out = v_0 and
    # lse = scale * q . k_0.
    x = make_layer(L=1, M=1, seed=8, head_dim=16)
    sel = np.full((1, 512), -1, dtype=np.int32)
    out, lse = oracle.attn(x.q, x.k, x.v, [0], sel, [0])
    for h in range(24):
        g = h // 12
        np.testing.assert_allclose(out[0, h], x.v[g, 0].double().numpy(), atol=1e-15)
        want = float(x.q[0, h].double() @ x.k[g, 0].double()) / 4.0
        assert abs(lse[0, h] - want) < 1e-12


def test_attention_visibility_mask_matches_sdpa_mask():
    L, M, D = 700, 3, 32
    x = make_layer(L=L, M=M, seed=9, head_dim=D)
    sel, cnt = _all_selected(x.row_pos)
    visible = np.ones(L, dtype=bool)
    visible[100:350] = False
    out, lse = oracle.attn(x.q, x.k, x.v, x.row_pos, sel, cnt, visible=visible)
    q = x.q.double().permute(1, 0, 2)
    k = x.k.double().repeat_interleave(12, dim=0)
    v = x.v.double().repeat_interleave(12, dim=0)
    mask = (torch.arange(L)[None, :] <= torch.tensor(x.row_pos)[:, None]) & torch.from_numpy(visible)[None]
    ref = torch.nn.functional.scaled_dot_product_attention(q, k, v, attn_mask=mask)
    np.testing.assert_allclose(out, ref.permute(1, 0, 2).numpy(), atol=1e-12)
    # No visible key at all: zeros and -inf, no NaN.
    out0, lse0 = oracle.attn(x.q, x.k, x.v, x.row_pos, sel, cnt, visible=np.zeros(L, dtype=bool))
    assert np.all(out0 == 0) and np.all(np.isneginf(lse0))


# ---------------------------------------------------------------- step 5: merge

def test_merge_identities():
    rng = np.random.default_rng(10)
    o = rng.standard_normal((1, 6, 8))
    l = rng.standard_normal((1, 6))
    out, lse = oracle.lse_merge(o, l)
    np.testing.assert_array_equal(out, o[0])
    np.testing.assert_array_equal(lse, l[0])
    # Two parts with equal lse: the average, and lse + ln 2.
    o2 = rng.standard_normal((2, 6, 8))
    out, lse = oracle.lse_merge(o2, np.stack([l[0], l[0]]))
    np.testing.assert_allclose(out, o2.mean(axis=0), atol=1e-15)
    np.testing.assert_allclose(lse, l[0] + math.log(2), atol=1e-15)
    # Weights follow exp(lse): lse 0 and ln 3 weigh 1 : 3.
    out, lse = oracle.lse_merge(o2, np.stack([np.zeros(6), np.full(6, math.log(3))]))
    np.testing.assert_allclose(out, 0.25 * o2[0] + 0.75 * o2[1], atol=1e-15)
    np.testing.assert_allclose(lse, math.log(4), atol=1e-15)
    # A -inf part contributes nothing; all -inf gives zeros and -inf.
    out, lse = oracle.lse_merge(o2, np.stack([l[0], np.full(6, -np.inf)]))
    np.testing.assert_allclose(out, o2[0], atol=1e-15)
    out, lse = oracle.lse_merge(o2, np.full((2, 6), -np.inf))
    assert np.all(out == 0) and np.all(np.isneginf(lse)) and not np.any(np.isnan(out))
    # Order of the parts does not matter.
    o5 = rng.standard_normal((5, 4, 3))
    l5 = rng.standard_normal((5, 4)) * 3
    a = oracle.lse_merge(o5, l5)
    b = oracle.lse_merge(o5[::-1].copy(), l5[::-1].copy())
    np.testing.assert_allclose(a[0], b[0], atol=1e-14)
    np.testing.assert_allclose(a[1], b[1], atol=1e-14)


def test_segmented_merge_equals_single_buffer():
    # Attention per KV segment, merged by log-sum-exp, equals attention over
    # the whole buffer (the segmented-cache identity), including a segment
    # that holds no selected row.
    x = make_layer(L=9000, M=4, seed=11, head_dim=64)
    pooled = oracle.pool(x.idxk)
    s = oracle.score(x.q_idx, pooled, x.row_pos)
    sel, cnt, _ = oracle.select(s, x.row_pos)
    full_out, full_lse = oracle.attn(x.q, x.k, x.v, x.row_pos, sel, cnt)
    cuts = segment_cuts(x.L, 7, seed=3) + []
    parts_o, parts_l = [], []
    for first, n in cuts:
        vis = np.zeros(x.L, dtype=bool)
        vis[first:first + n] = True
        o, l = oracle.attn(x.q, x.k, x.v, x.row_pos, sel, cnt, visible=vis)
        parts_o.append(o.reshape(-1, 64))
        parts_l.append(l.reshape(-1))
    out, lse = oracle.lse_merge(np.stack(parts_o), np.stack(parts_l))
    np.testing.assert_allclose(out, full_out.reshape(-1, 64), atol=1e-12)
    np.testing.assert_allclose(lse, full_lse.reshape(-1), atol=1e-12)


def test_threads_do_not_change_results():
    x = make_layer(L=3000, M=2, seed=12, head_dim=32)
    old = oracle.set_threads(1)
    a = oracle.layer_step(x.q_idx, x.idxk, x.q, x.k, x.v, x.row_pos)
    oracle.set_threads(4)
    b = oracle.layer_step(x.q_idx, x.idxk, x.q, x.k, x.v, x.row_pos)
    oracle.set_threads(old)
    for key in ("scores", "sel", "cnt", "out", "lse"):
        np.testing.assert_array_equal(a[key], b[key])


def test_layer_step_reads_nothing_past_a_row():
    # A row at position p sees tokens 0..p only (causal, hipfire section 02):
    # its scores, selection, output and lse must not change when the cache is
    # cut right after p.  This is the reading under which rows inside a
    # longer cache are a descriptor with L = p + 1; a visibility bound taken
    # from the cache length rather than the row's position fails it.  Every
    # row here chooses 512 of more than 512 blocks.
    x = make_layer(L=6001, M=3, seed=13, head_dim=32)
    row_pos = [2500, 4001, 5998]
    full = oracle.layer_step(x.q_idx, x.idxk, x.q, x.k, x.v, row_pos)
    for r, p in enumerate(row_pos):
        cut = oracle.layer_step(x.q_idx[r:r + 1], x.idxk[:p + 1], x.q[r:r + 1], x.k[:, :p + 1], x.v[:, :p + 1], [p])
        nb = oracle.visible_blocks(p)
        assert nb > 512 and int(cut["cnt"][0]) == int(full["cnt"][r]) == 512
        np.testing.assert_array_equal(cut["scores"][0, :nb], full["scores"][r, :nb])
        np.testing.assert_array_equal(cut["sel"][0], full["sel"][r])
        np.testing.assert_array_equal(cut["out"][0], full["out"][r])
        np.testing.assert_array_equal(cut["lse"][0], full["lse"][r])


# ------------------------------------------------------------------ fp8 K/V state (E4M3 + f16 scale)
_FINITE = [c for c in range(256) if c not in (0x7F, 0xFF)]


def test_e4m3_decode_known_codes():
    # Format facts: bias 7, 3 mantissa bits, subnormals m * 2^-9, 448 the
    # largest finite value, S.1111.111 the only NaN.
    assert oracle.e4m3_decode(0x00) == 0.0 and math.copysign(1, oracle.e4m3_decode(0x80)) < 0
    assert oracle.e4m3_decode(0x01) == 2.0 ** -9 and oracle.e4m3_decode(0x07) == 7 * 2.0 ** -9
    assert oracle.e4m3_decode(0x08) == 2.0 ** -6
    assert oracle.e4m3_decode(0x38) == 1.0 and oracle.e4m3_decode(0x3F) == 1.875
    assert oracle.e4m3_decode(0x7E) == 448.0 and oracle.e4m3_decode(0xFE) == -448.0
    assert math.isnan(oracle.e4m3_decode(0x7F)) and math.isnan(oracle.e4m3_decode(0xFF))
    vals = sorted(oracle.e4m3_decode(c) for c in _FINITE if c < 0x80)
    assert len(set(vals)) == 127 and vals[-1] == 448.0       # 127 distinct non-negative values


def test_e4m3_encode_is_nearest_ties_to_even():
    table = [(c, oracle.e4m3_decode(c)) for c in _FINITE]
    for c, v in table:                                        # every finite code round-trips
        if c != 0x80:
            assert oracle.e4m3_encode(v) == c
    rng = np.random.default_rng(7)
    xs = np.concatenate([rng.standard_normal(1500) * 40, rng.standard_normal(500) * 0.01,
                         rng.uniform(-470, 470, 500)])
    for x in xs:
        c = oracle.e4m3_encode(x)
        got = oracle.e4m3_decode(c)
        target = max(-448.0, min(448.0, x))                   # saturation
        best = min(abs(target - v) for _, v in table)
        assert abs(target - got) == best, (x, c)
        ties = [cc for cc, v in table if abs(target - v) == best and (v != 0 or cc == 0)]
        if len(ties) > 1:                                     # a tie: the even mantissa
            assert c & 1 == 0
    # Exact halfway points.
    assert oracle.e4m3_encode(1.0625) == 0x38 and oracle.e4m3_encode(1.1875) == 0x3A
    assert oracle.e4m3_encode(2.0 ** -10) == 0x00 and oracle.e4m3_encode(3 * 2.0 ** -10) == 0x02
    assert oracle.e4m3_encode(1e6) == 0x7E and oracle.e4m3_encode(-1e6) == 0xFE


def test_f16_codec_matches_numpy():
    rng = np.random.default_rng(8)
    xs = np.concatenate([rng.standard_normal(3000), rng.standard_normal(1000) * 1e-5,
                         rng.standard_normal(500) * 3e4, [0.0, -0.0, 65504.0, 6.0e-8, 2.0 ** -24]])
    for x in xs:
        ref = int(np.array([x], dtype=np.float16).view(np.uint16)[0])
        assert oracle.f16_encode(float(x)) == ref, x
        assert oracle.f16_decode(ref) == float(np.array([ref], dtype=np.uint16).view(np.float16)[0])


def test_fp8_quantize_rows():
    rng = np.random.default_rng(9)
    x = rng.standard_normal((6, 256)).astype(np.float32)
    x[1] *= 1e-3
    x[2] = 0.0                                                # a zero row: scale 0, zero codes
    x[3, :] = np.arange(256, dtype=np.float32) * 0.5          # exact multiples
    x[4, 17] = -1000.0                                        # amax from a negative element
    codes, scales = oracle.fp8_quantize(x)
    deq = oracle.fp8_dequantize(codes, scales)
    for r in range(6):
        amax = float(np.abs(x[r]).max())
        s32 = np.float32(amax) / np.float32(448.0)
        assert scales[r] == np.array([s32], dtype=np.float16).view(np.uint16)[0]
        sc = float(np.array([scales[r]], dtype=np.uint16).view(np.float16)[0])
        if sc == 0:
            assert (codes[r] == 0).all() and (deq[r] == 0).all()
            continue
        for d in range(256):
            qv = float(np.float32(x[r, d]) / np.float32(sc))
            assert codes[r, d] == oracle.e4m3_encode(qv)
        # Relative error of a stored element: at most half an E4M3 step (2^-4
        # of the value) plus the f16 rounding of the scale, or a subnormal step.
        err = np.abs(deq[r] - x[r])
        assert (err <= np.abs(x[r]) * (2.0 ** -4 + 2.0 ** -10) + 2.0 ** -9 * sc * 1.01).all()
    # The element of largest magnitude lands at or next to 448.
    assert abs(oracle.e4m3_decode(codes[4, 17])) >= 416.0


def test_fp8_attention_is_attention_on_the_stored_values():
    # The oracle attends over fp8 state by dequantizing exactly; a row whose
    # values are exactly representable gives the same result as bf16 state.
    x = make_layer(L=600, M=2, seed=14, head_dim=64)
    k = np.round(x.k.numpy() * 4) / 4                         # quarters in [-4, 4]: exact in E4M3 at scale 1/8
    k = np.clip(k, -4, 4).astype(np.float32)
    codes = np.vectorize(lambda v: oracle.e4m3_encode(v * 8))(k).astype(np.uint8)
    scales = np.full(k.shape[:-1], oracle.f16_encode(0.125), dtype=np.uint16)
    kd = oracle.fp8_dequantize(codes, scales)
    np.testing.assert_array_equal(kd, k.astype(np.float64))
    pooled = oracle.pool(x.idxk)
    s = oracle.score(x.q_idx, pooled, x.row_pos)
    sel, cnt, _ = oracle.select(s, x.row_pos)
    v64 = x.v.numpy().astype(np.float64)
    a = oracle.attn(x.q, kd, v64, x.row_pos, sel, cnt)
    b = oracle.attn(x.q, k.astype(np.float64), v64, x.row_pos, sel, cnt)
    np.testing.assert_array_equal(a[0], b[0])


# ------------------------------------------------------------------ q8 K/V state (Q8_0 blocks of 32)
def test_q8_quantize_blocks():
    rng = np.random.default_rng(15)
    x = rng.standard_normal((5, 256)).astype(np.float32)
    x[1, :32] = 0.0                                           # a zero block
    x[2, 40] = 254.0                                          # amax 254: scale exactly 2
    x[3, 64:96] = np.arange(-16, 16, dtype=np.float32) * 0.5  # halves: ties away from zero
    codes, scales = oracle.q8_quantize(x)
    deq = oracle.q8_dequantize(codes, scales)
    f16 = lambda b: float(np.array([b], dtype=np.uint16).view(np.float16)[0])
    for r in range(5):
        for b in range(8):
            blk = x[r, 32 * b:32 * b + 32]
            s32 = np.float32(np.abs(blk).max()) / np.float32(127.0)
            assert scales[r, b] == np.array([s32], dtype=np.float16).view(np.uint16)[0]
            sc = f16(scales[r, b])
            want = np.zeros(32, dtype=np.int8) if sc == 0 else np.clip(
                np.sign(blk / np.float32(sc)) * np.floor(np.abs(blk / np.float32(sc)) + 0.5), -127, 127)
            np.testing.assert_array_equal(codes[r, 32 * b:32 * b + 32], want.astype(np.int8))
            np.testing.assert_array_equal(deq[r, 32 * b:32 * b + 32], codes[r, 32 * b:32 * b + 32] * sc)
    assert (codes[1, :32] == 0).all() and scales[1, 0] == 0
    assert codes[2, 40] == 127 and f16(scales[2, 1]) == 2.0
    assert np.abs(codes).max() <= 127
    # Error of a stored element: at most half a code step plus the scale's f16 rounding.
    steps = np.repeat(np.vectorize(f16)(scales), 32, axis=1)
    assert (np.abs(deq - x) <= 0.5 * steps * 1.001 + np.abs(x) * 2.0 ** -10).all()
