"""Seeded synthetic inputs for QSA layer steps.

This module only draws random numbers and lays them out; it holds none of the
method's arithmetic (no pooling, scoring, selection or attention).  Both the
CUDA path and the CPU oracle take their inputs from here.

Recipe (the same for every workload):
  * q, k, v, index keys and index queries ~ N(0, 1), drawn in fp32 from a
    torch.Generator seeded with (seed, layer) on the requested device;
  * "planted" blocks: a seeded permutation of the complete blocks picks
    ``n_planted`` distinct block ids, and +0.5 is added to all four tokens'
    index keys of those blocks (before any rounding), so that the block
    selection is not a uniform lottery;
  * bf16 workloads round every tensor to bf16 once, after planting.

The shapes follow the pages' workloads: 24 query heads over 2 KV heads at
head_dim 256 (MTPLX pull request #482, "Terms used in this document"), 128-wide
index keys with 4 index heads and a 512-block budget (hipfire, "QSA sparse
attention and the VMM KV backend", section 02), a 261,120-token context with
a fixed four-row verify (pull request #482), and a 2,048-row prefill chunk at a
~100k prefix (the SGLang launcher notes, section 1).
"""
from __future__ import annotations

import dataclasses
import math

import torch

INDEX_DIM = 128
INDEX_HEADS = 4


@dataclasses.dataclass
class LayerInputs:
    """One sequence's inputs for one QSA layer.

    Rows j = 0..M-1 sit at absolute positions L - M + j (the last M tokens).
    k and v are single buffers laid out [n_kv_heads, L, head_dim].
    """
    L: int
    M: int
    idxk: torch.Tensor        # [L, 128]
    q_idx: torch.Tensor       # [M, 4, 128]
    q: torch.Tensor           # [M, Hq, D]
    k: torch.Tensor           # [Hkv, L, D]
    v: torch.Tensor           # [Hkv, L, D]
    planted: torch.Tensor     # int64 block ids that got the +0.5 offset

    @property
    def row_pos(self) -> list[int]:
        return [self.L - self.M + j for j in range(self.M)]


def _gen(seed: int, stream: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed((int(seed) * 1_000_003 + int(stream) * 7_919) & 0x7FFF_FFFF_FFFF_FFFF)
    return g


def make_layer(L: int, M: int, *, dtype=torch.float32, seed: int = 0, layer: int = 0,
               n_planted: int = 64, n_q_heads: int = 24, n_kv_heads: int = 2, head_dim: int = 256,
               device="cpu") -> LayerInputs:
    """Draw one layer's inputs; deterministic in (seed, layer, device)."""
    if not (1 <= M <= L):
        raise ValueError("need 1 <= M <= L")
    g = _gen(seed, layer, device)
    f32 = torch.float32
    idxk = torch.randn((L, INDEX_DIM), generator=g, device=device, dtype=f32)
    q_idx = torch.randn((M, INDEX_HEADS, INDEX_DIM), generator=g, device=device, dtype=f32)
    q = torch.randn((M, n_q_heads, head_dim), generator=g, device=device, dtype=f32)
    k = torch.randn((n_kv_heads, L, head_dim), generator=g, device=device, dtype=f32)
    v = torch.randn((n_kv_heads, L, head_dim), generator=g, device=device, dtype=f32)
    complete = L // 4
    gp = torch.Generator(device="cpu")
    gp.manual_seed(int(seed) * 65_537 + int(layer) + 1)
    n_planted = min(int(n_planted), complete)
    planted = torch.randperm(complete, generator=gp)[:n_planted].sort().values
    if n_planted:
        tok = (planted.to(device).view(-1, 1) * 4 + torch.arange(4, device=device).view(1, 4)).reshape(-1)
        idxk[tok] += 0.5
    if dtype != f32:
        idxk, q_idx, q, k, v = (t.to(dtype) for t in (idxk, q_idx, q, k, v))
    return LayerInputs(L=L, M=M, idxk=idxk, q_idx=q_idx, q=q, k=k, v=v, planted=planted)


def segment_cuts(L: int, n_segments: int, *, seed: int) -> list[tuple[int, int]]:
    """Split tokens [0, L) into n_segments non-empty (first, n) ranges.

    Cut points are uniform over token positions (not block-aligned), as in a
    cache kept as one segment per finished turn plus a growing tail (MTPLX
    pull request #610, "How it works, in plain terms").
    """
    if not (1 <= n_segments <= L):
        raise ValueError("need 1 <= n_segments <= L")
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed) * 104_729 + L)
    cuts = (torch.randperm(L - 1, generator=g)[: n_segments - 1] + 1).sort().values.tolist()
    edges = [0] + cuts + [L]
    return [(edges[i], edges[i + 1] - edges[i]) for i in range(n_segments)]


@dataclasses.dataclass
class RaggedBatchSpec:
    """A ragged decode/verify batch: per sequence (L, M, n_segments)."""
    lengths: list[int]
    rows: list[int]
    n_segments: list[int]


def ragged_batch_spec(n_seqs: int = 16, *, seed: int = 0, min_len: int = 4096,
                      max_len: int = 262_144) -> RaggedBatchSpec:
    """Half the sequences decode one row, half verify four; contexts are
    log-uniform in [min_len, max_len]; each has 3-12 KV segments."""
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed) * 31_337 + 11)
    u = torch.rand((n_seqs,), generator=g, dtype=torch.float64)
    lengths = [int(round(math.exp(math.log(min_len) + float(x) * (math.log(max_len) - math.log(min_len)))))
               for x in u]
    rows = [1 if i < n_seqs // 2 else 4 for i in range(n_seqs)]
    n_segs = torch.randint(3, 13, (n_seqs,), generator=g).tolist()
    return RaggedBatchSpec(lengths=lengths, rows=rows, n_segments=n_segs)


# The five workloads, by name.  "layers" independent layers are drawn per
# step; rows sit at the end of each context.
WORKLOADS = {
    "tiny_verify_f32": dict(L=4099, M=4, dtype=torch.float32, layers=1, n_planted=64, head_dim=256),
    "decode_m1_65k_bf16": dict(L=65_536, M=1, dtype=torch.bfloat16, layers=12, n_planted=256, head_dim=256),
    "verify_m4_261k_bf16": dict(L=261_120, M=4, dtype=torch.bfloat16, layers=12, n_planted=256, head_dim=256),
    # A wider verify window (MTPLX #482 verifies 3-8 rows): eight rows on the
    # same 261,120-token cache.
    "verify_m8_261k_bf16": dict(L=261_120, M=8, dtype=torch.bfloat16, layers=12, n_planted=256, head_dim=256),
    "prefill_t2048_100k_bf16": dict(L=100_352 + 2048, M=2048, dtype=torch.bfloat16, layers=1, n_planted=256,
                                    head_dim=256),
    "ragged_segmented_bf16": dict(n_seqs=16, dtype=torch.bfloat16, n_planted=256, head_dims=(256, 128)),
    # The same decode and verify steps over quantized K/V state (fp8: E4M3 codes
    # with an f16 scale pair per head and token; q8: Q8_0, int8 codes with an
    # f16 scale per 32 elements), the caches written from the bf16 draw by the
    # library's own append, as a model's cache would be.
    "decode_m1_65k_fp8": dict(L=65_536, M=1, dtype=torch.bfloat16, layers=12, n_planted=256, head_dim=256,
                              kv_state="fp8"),
    "verify_m4_261k_fp8": dict(L=261_120, M=4, dtype=torch.bfloat16, layers=12, n_planted=256, head_dim=256,
                               kv_state="fp8"),
    "decode_m1_65k_q8": dict(L=65_536, M=1, dtype=torch.bfloat16, layers=12, n_planted=256, head_dim=256,
                             kv_state="q8"),
    "verify_m4_261k_q8": dict(L=261_120, M=4, dtype=torch.bfloat16, layers=12, n_planted=256, head_dim=256,
                              kv_state="q8"),
}
