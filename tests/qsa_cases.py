"""Shared helpers for the GPU parity tests: run the CUDA library on seeded
workloads and compare with the oracle under the tolerances the tests state.

Tolerances (fp32 accumulation, derived from the arithmetic):
  * pooled keys: a mean of 4 stored values in fp32 -> |err| <= 2 ulp.
  * block scores: each of the 4 dot products has 128 fp32 products with fp32
    accumulation, so |err_h| <= gamma * sum_d |q_hd| |k_d| with
    gamma = 130 * 2^-24 (recursive-summation bound for n = 128, plus the fp32
    rounding of the pooled key); ReLU and the 4-term head sum do not amplify
    it, so |err| <= scale * (gamma * sum_h sum_d |q_hd||k_d| + 4 ulp(score)).
  * selection: bit-exact, except blocks whose oracle score is within 1e-6
    relative of the row's k-th score tau.
  * attention given the oracle's selection: max abs error <= 1e-4 for fp32
    K/V; for bf16 K/V max abs error <= 2e-2 and max error <= 1e-2 of the
    largest |output| (normwise relative).
"""
from __future__ import annotations

import math

import numpy as np
import torch

import indexed_sparse_attention_gb300 as qsa
import oracle

SCORE_GAMMA = 130 * 2.0 ** -24
ATTN_F32_ABS = 1e-4
ATTN_BF16_ABS = 2e-2
ATTN_BF16_REL = 1e-2
SEL_REL = 1e-6


def dev():
    return torch.device("cuda", 0)


def pooled_buffer(L: int, device) -> torch.Tensor:
    return torch.full((qsa.n_pooled_slots(L), 128), float("nan"), dtype=torch.float32, device=device)


def pool_all(idxk_dev: torch.Tensor, pooled: torch.Tensor, L: int):
    qsa.pool_index_keys(idxk_dev, pooled, 0, L // 4)


def assert_pooled_close(got: np.ndarray, idxk, blocks):
    """Pooled keys of the listed blocks against the oracle's fp64 mean of the
    four stored index keys: three fp32 additions and an exact scaling, so
    |err| <= 3 u mean_j |k_j| + u |mean| (u = 2^-24)."""
    blocks = np.asarray(list(blocks), dtype=np.int64)
    if blocks.size == 0:
        return
    if isinstance(idxk, torch.Tensor):
        idxk = idxk.cpu()
    keys = idxk.double().numpy() if isinstance(idxk, torch.Tensor) else np.asarray(idxk, dtype=np.float64)
    want = oracle.pool(idxk)[blocks]
    rows = keys[: 4 * (int(blocks.max()) + 1)].reshape(-1, 4, keys.shape[1])[blocks]
    u = 2.0 ** -24
    bound = 3 * u * np.abs(rows).mean(axis=1) + u * np.abs(want)
    err = np.abs(got[blocks].astype(np.float64) - want)
    assert (err <= bound).all(), f"pooled keys off by up to {err.max():.3e}"


def score_bound(q_idx, pooled_f64: np.ndarray, row_pos) -> np.ndarray:
    """Per-entry absolute error bound of an fp32 score (see module docstring)."""
    q = q_idx.double().cpu().numpy() if isinstance(q_idx, torch.Tensor) else np.asarray(q_idx, dtype=np.float64)
    aq = np.abs(q)                                # [M, 4, 128]
    ak = np.abs(pooled_f64)                       # [NB, 128]
    mag = np.einsum("mhd,bd->mb", aq, ak)         # sum_h sum_d |q||k|
    return oracle.SCORE_SCALE * (SCORE_GAMMA * mag) + 1e-30


def assert_scores_close(gpu: np.ndarray, ref: np.ndarray, bound: np.ndarray, row_pos):
    for r, p in enumerate(row_pos):
        nb = oracle.visible_blocks(p)
        g, o, b = gpu[r, :nb].astype(np.float64), ref[r, :nb], bound[r, :nb]
        tol = b + 4 * np.spacing(np.abs(o).astype(np.float32)).astype(np.float64)
        bad = np.abs(g - o) > tol
        assert not bad.any(), (f"row {r}: {bad.sum()} scores off; worst |err| "
                               f"{np.max(np.abs(g - o)):.3e} vs bound {tol[np.argmax(np.abs(g - o))]:.3e}")


def assert_selection_close(sel_gpu, cnt_gpu, sel_ref, cnt_ref, tau, scores_ref, row_pos, rel=SEL_REL):
    """Sets equal except blocks with |s - tau| <= rel*|tau|; counts equal."""
    for r in range(len(row_pos)):
        assert int(cnt_gpu[r]) == int(cnt_ref[r]), f"row {r}: count {cnt_gpu[r]} != {cnt_ref[r]}"
        c = int(cnt_ref[r])
        a = sel_gpu[r, :c]
        assert np.all(np.diff(a) > 0), f"row {r}: ids not strictly ascending"
        assert np.all(sel_gpu[r, c:] == -1)
        diff = set(a.tolist()) ^ set(sel_ref[r, :c].tolist())
        t = tau[r]
        for b in diff:
            assert np.isfinite(t) and abs(scores_ref[r, b] - t) <= rel * abs(t), \
                f"row {r}: block {b} (score {scores_ref[r, b]!r}, tau {t!r}) differs"


def assert_attn_close(out_gpu: np.ndarray, lse_gpu: np.ndarray, out_ref: np.ndarray, lse_ref: np.ndarray,
                      kv_bf16: bool):
    og = out_gpu.astype(np.float64)
    err = np.abs(og - out_ref)
    assert not np.isnan(og).any()
    fin = np.isfinite(lse_ref)
    assert np.array_equal(np.isfinite(lse_gpu), fin), "rows with / without keys differ"
    lerr = np.abs(lse_gpu[fin].astype(np.float64) - lse_ref[fin]) if fin.any() else np.zeros(1)
    if kv_bf16:
        assert err.max() <= ATTN_BF16_ABS, f"max abs err {err.max():.3e}"
        scale = max(np.abs(out_ref).max(), 1e-30)
        assert err.max() <= ATTN_BF16_REL * scale, f"normwise rel err {err.max() / scale:.3e}"
        assert lerr.max() <= ATTN_BF16_ABS, f"lse err {lerr.max():.3e}"
    else:
        assert err.max() <= ATTN_F32_ABS, f"max abs err {err.max():.3e}"
        assert lerr.max() <= ATTN_F32_ABS, f"lse err {lerr.max():.3e}"


def to_np(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().numpy()


class DeviceLayer:
    """One sequence's workload on the GPU, single-buffer K/V, all earlier
    blocks already pooled (the step pools what its rows complete)."""

    def __init__(self, x, device=None, *, out_dtype=torch.float32, n_splits=0, segments=None, top_k=512):
        device = device or dev()
        self.x = x
        self.idxk = x.idxk.to(device)
        self.q_idx = x.q_idx.to(device)
        self.q = x.q.to(device)
        self.k = x.k.to(device)
        self.v = x.v.to(device)
        self.pooled = pooled_buffer(x.L, device)
        first_new = (x.L - x.M) // 4
        if first_new > 0:
            qsa.pool_index_keys(self.idxk, self.pooled, 0, first_new)
        segs = segments if segments is not None else [qsa.Segment(self.k, self.v, 0)]
        self.seq = qsa.Seq(x.L, x.M, self.pooled, segs, idx_keys=self.idxk)
        self.step = qsa.LayerStep([self.seq], self.q_idx, self.q, out_dtype=out_dtype, n_splits=n_splits,
                                  top_k=top_k)

    def run(self):
        self.step.run()
        torch.cuda.synchronize()
        return self.step


def oracle_layer(x, top_k=512, visible=None):
    return oracle.layer_step(x.q_idx, x.idxk, x.q, x.k, x.v, x.row_pos, top_k=top_k, visible=visible)
