"""Pool slots that hold no token may contain anything, NaN and Inf included.

A block's slots past its fill, and blocks no segment references, are not part of any
context (the paged pool of section 4.1 holds whole blocks; a recycled or freshly
allocated pool holds arbitrary bit patterns there).  The oracle reads only slots below
the fill, so the kernels must give the oracle's result whatever those slots hold.  Both
tests poison every unused slot (K with NaN, V with +Inf, then the reverse) and compare
with the oracle, and with a run on the same pool whose unused slots hold zeros.
"""
import math

import numpy as np
import pytest
import torch

import segmented_kv_attention_msa_b300 as msa
from segmented_kv_attention_msa_b300 import build as B
from segmented_kv_attention_msa_b300 import workload as W
from oracle import msa_oracle as O
from tests.helpers import assert_close, np64, workload_arrays

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    B.build()
    msa.lib()


def unused_slots(lay):
    """bool [blocks, 16]: slots that hold no token of any segment."""
    used = np.zeros((lay.num_pool_blocks, 16), bool)
    for (s, f, nb) in np.asarray(lay.segments).reshape(-1, 3):
        for i in range(int(nb)):
            b = int(lay.block_table[s, f + i])
            used[b, :int(lay.block_fill[b])] = True
    return ~used


def poison(t, mask, value):
    """Write `value` into every (block, slot) of `mask`, all heads and columns."""
    m = torch.from_numpy(mask).to(t.device)
    view = t.permute(0, 2, 1, 3)            # [blocks, 16, Hkv, d]
    view[m] = value


def _prefill_specs():
    rng = np.random.default_rng(61)
    partial = W.SeqSpec([(0, 37), (48, 100), (160, 9), (256, 250)],
                        np.concatenate([np.arange(37, 48), np.arange(148, 160), np.arange(169, 256),
                                        np.arange(506, 900)]))
    sparse = W.SeqSpec([(0, 16), (64, 7), (128, 40), (320, 33)],
                       np.sort(rng.choice(np.concatenate([np.arange(16, 64), np.arange(71, 128),
                                                          np.arange(168, 320), np.arange(353, 800)]),
                                          400, replace=False)))
    return [partial, sparse, W.random_prefill_spec(rng, 60, 0.5, 100, 500)]


@pytest.mark.parametrize("heads", [(8, 2, 128), (4, 4, 64), (32, 8, 128)])
@pytest.mark.parametrize("kval,vval", [(math.nan, math.inf), (math.inf, math.nan)])
def test_prefill_ignores_unused_slots(heads, kval, vval):
    Hq, Hkv, d = heads
    lay = W.custom_prefill(Hq, Hkv, d, _prefill_specs(), seed=62, qk_std=2.0 / math.sqrt(d), shuffle_segments=True)
    mask = unused_slots(lay)
    assert mask[lay.block_fill > 0].any()             # some referenced blocks are partial
    wl = W.make_values(lay, device="cuda")
    plan = msa.Plan.from_layout(lay).upload("cuda")
    poison(wl.k_pool, mask, 0.0)
    poison(wl.v_pool, mask, 0.0)
    clean_o, clean_l = msa.prefill(plan, wl.q, wl.k_chunk, wl.v_chunk, wl.k_pool, wl.v_pool)
    torch.cuda.synchronize()
    a = workload_arrays(wl)
    poison(wl.k_pool, mask, kval)
    poison(wl.v_pool, mask, vval)
    out, lse = msa.prefill(plan, wl.q, wl.k_chunk, wl.v_chunk, wl.k_pool, wl.v_pool)
    torch.cuda.synchronize()
    assert msa.get_status(plan) == 0
    assert torch.isfinite(out.float()).all() and torch.isfinite(lse).all()
    assert torch.equal(out, clean_o) and torch.equal(lse, clean_l)
    _, ro, rl = O.prefill(lay, a["q"], a["k_chunk"], a["v_chunk"], a["k_pool"], a["v_pool"], 1.0 / math.sqrt(d))
    assert_close(np64(out), ro, "prefill out")
    assert_close(np64(lse), rl, "prefill lse")


@pytest.mark.parametrize("kval,vval", [(math.nan, math.inf), (math.inf, math.nan)])
@pytest.mark.parametrize("split", [0, 2])
def test_decode_ignores_unused_slots(kval, vval, split):
    rng = np.random.default_rng(63)
    specs = []
    for _ in range(6):
        L = int(rng.integers(20, 1500))
        cut = int(rng.integers(1, max(2, L // 16))) * 16 if L > 32 else L
        runs = [(0, min(cut, L))] + ([(cut, L - cut)] if L > cut else [])
        specs.append(W.SeqSpec(runs, np.zeros(0)))
    lay = W.custom_decode(16, 4, 128, specs, seed=64, qk_std=0.4, shuffle_segments=True)
    mask = unused_slots(lay)
    assert mask[lay.block_fill > 0].any()
    wl = W.make_values(lay, device="cuda")
    plan = msa.Plan.from_layout(lay, decode_split_blocks=split).upload("cuda")
    poison(wl.k_pool, mask, 0.0)
    poison(wl.v_pool, mask, 0.0)
    clean_o, clean_l = msa.decode(plan, wl.q, wl.k_pool, wl.v_pool)
    torch.cuda.synchronize()
    kp, vp = np64(wl.k_pool), np64(wl.v_pool)
    poison(wl.k_pool, mask, kval)
    poison(wl.v_pool, mask, vval)
    out, lse = msa.decode(plan, wl.q, wl.k_pool, wl.v_pool)
    torch.cuda.synchronize()
    assert msa.get_status(plan) == 0
    assert torch.equal(out, clean_o) and torch.equal(lse, clean_l)
    _, ro, rl = O.decode(lay, np64(wl.q), kp, vp, 1.0 / math.sqrt(128))
    assert_close(np64(out), ro, "decode out")
    assert_close(np64(lse), rl, "decode lse")
