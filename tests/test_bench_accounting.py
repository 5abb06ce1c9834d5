"""The bench's algorithmic bytes per layer-step, on the CPU.

The roofline fraction divides these bytes by a measured time, so they are
pinned here to the count written out by hand for the 261,120-token verify
(4 rows at positions 261,116..261,119, bf16 state, head_dim 256, 24 query
heads over 2 KV heads): the pooled keys once, the index queries, the pooling
of the one block the rows complete, each row's selected K/V tokens of both
KV heads, the queries and the fp32 outputs with their lse -- and neither the
dense K/V left unread nor the scores intermediate.
"""
from types import SimpleNamespace

import torch

import bench


def _verify_layer(kv_state=None):
    L, M, D = 261_120, 4, 256
    bf = torch.bfloat16
    x = SimpleNamespace(
        L=L, M=M,
        k=torch.empty((2, 0, D), dtype=bf if kv_state is None else torch.uint8),
        q=torch.empty((M, 24, D), dtype=bf),
        idxk=torch.empty((0, 128), dtype=bf),
        q_idx=torch.empty((M, 4, 128), dtype=bf),
        row_pos=[L - M + j for j in range(M)],
    )
    # The step pools the one block its rows complete: block 65,279.
    step = SimpleNamespace(pool_jobs=[(None, None, 65_279, 1)])
    return SimpleNamespace(x=x, kv_state=kv_state, step=step)


def test_verify_bytes_written_out():
    ab = bench.algorithmic_bytes(_verify_layer())
    pooled = 65_280 * 128 * 4                      # every complete block's fp32 key, once
    q_idx = 4 * 4 * 128 * 2                        # bf16 index queries
    pool = 4 * 128 * 2 + 128 * 4                   # one block: four bf16 index keys in, one key out
    tokens = (2048 + 1) + (2048 + 2) + (2048 + 3) + (2048 + 0)   # 512 blocks + the tail per row
    kv = tokens * 2 * (2 * 256 * 2)                # both KV heads, K and V rows of 256 bf16
    q = 4 * 24 * 256 * 2
    out = 4 * 24 * (256 * 4 + 4)                   # fp32 outputs and lse
    assert tokens == 8198
    assert ab["score"] == pooled + q_idx
    assert ab["pool"] == pool
    assert ab["score"] + ab["pool"] == 33_428_992
    assert ab["attn"] == kv + q + out
    assert ab["total"] == 50_366_336


def test_quantized_state_counts_codes_and_scale_records():
    # fp8: one byte per element and a 4-byte (K, V) scale pair per head and
    # token; q8: one byte per element and an f16 scale per 32 elements of
    # each of the two rows.
    tokens = 8198
    base = bench.algorithmic_bytes(_verify_layer())
    for state, per_tok in (("fp8", 2 * 256 + 4), ("q8", 2 * 256 + 2 * (256 // 32) * 2)):
        ab = bench.algorithmic_bytes(_verify_layer(state))
        assert ab["score"] == base["score"] and ab["pool"] == base["pool"]
        assert ab["attn"] - base["attn"] == tokens * 2 * (per_tok - 2 * 256 * 2)
