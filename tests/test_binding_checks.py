"""The Python binding checks every tensor's shape and dtype against the plan before a
call reaches the C ABI (which takes raw pointers and cannot check sizes).  Meta tensors
stand in for device tensors: only shapes and dtypes are looked at, no GPU is used."""
import numpy as np
import pytest
import torch

import segmented_kv_attention_msa_b300 as msa
from segmented_kv_attention_msa_b300 import build as B
from segmented_kv_attention_msa_b300 import workload as W


@pytest.fixture(scope="module", autouse=True)
def built():
    B.build()


def meta(*shape, dtype=torch.bfloat16):
    return torch.empty(*shape, dtype=dtype, device="meta")


def prefill_tensors(lay):
    T, Hq, Hkv, d, nb = lay.total_q, lay.num_heads_q, lay.num_heads_kv, lay.head_dim, lay.num_pool_blocks
    return dict(q=meta(T, Hq, d), k_chunk=meta(T, Hkv, d), v_chunk=meta(T, Hkv, d),
                k_pool=meta(nb, Hkv, 16, d), v_pool=meta(nb, Hkv, 16, d),
                out=meta(T, Hq, d), lse=meta(T, Hq, dtype=torch.float32))


@pytest.mark.parametrize("idx", [1, 2, 3])
def test_prefill_shapes_accepted_and_refused(idx):
    lay = W.make_layout(idx, tiler=msa.chunk_sizes if idx == 3 else None)
    plan = msa.Plan.from_layout(lay)
    good = prefill_tensors(lay)
    msa.check_prefill_args(plan, **good)
    # a larger pool is fine (the plan addresses blocks below num_pool_blocks only)
    bigger = dict(good, k_pool=meta(lay.num_pool_blocks + 3, lay.num_heads_kv, 16, lay.head_dim),
                  v_pool=meta(lay.num_pool_blocks + 3, lay.num_heads_kv, 16, lay.head_dim))
    msa.check_prefill_args(plan, **bigger)
    T, Hq, Hkv, d, nb = lay.total_q, lay.num_heads_q, lay.num_heads_kv, lay.head_dim, lay.num_pool_blocks
    bad = [dict(q=meta(T - 1, Hq, d)), dict(k_chunk=meta(T, Hkv + 1, d)), dict(v_chunk=meta(T, Hkv, d // 2)),
           dict(k_pool=meta(nb - 1, Hkv, 16, d)), dict(v_pool=meta(nb, Hkv, 8, d)),
           dict(out=meta(T, Hq, d, dtype=torch.float32)), dict(lse=meta(T, Hq - 1, dtype=torch.float32)),
           dict(q=meta(T, Hq, d, dtype=torch.float16))]
    for b in bad:
        with pytest.raises(ValueError):
            msa.check_prefill_args(plan, **dict(good, **b))


def test_decode_shapes_accepted_and_refused():
    lay = W.make_layout(4)
    plan = msa.Plan.from_layout(lay)
    B_, Hq, Hkv, d, nb = lay.num_seqs, lay.num_heads_q, lay.num_heads_kv, lay.head_dim, lay.num_pool_blocks
    good = dict(q=meta(B_, Hq, d), k_pool=meta(nb, Hkv, 16, d), v_pool=meta(nb, Hkv, 16, d),
                out=meta(B_, Hq, d), lse=meta(B_, Hq, dtype=torch.float32))
    msa.check_decode_args(plan, **good)
    for b in (dict(q=meta(B_ + 1, Hq, d)), dict(k_pool=meta(nb - 1, Hkv, 16, d)),
              dict(out=meta(B_, Hq, d + 8)), dict(lse=meta(B_, Hq))):
        with pytest.raises(ValueError):
            msa.check_decode_args(plan, **dict(good, **b))


def test_mode_mismatch_refused():
    lay = W.make_layout(1)
    plan = msa.Plan.from_layout(lay)
    t = prefill_tensors(lay)
    with pytest.raises(ValueError):
        msa.check_decode_args(plan, t["q"], t["k_pool"], t["v_pool"])
