"""The kernels' give-up path, made to run on purpose without any GPU fault.

Every device wait is bounded (msa_set_wait_limit).  The test hook msa_set_test_drop makes
one CTA leave out one of its copies, so the wait for that copy runs out: the kernel must
record MSA_ERR_TIMEOUT in the status word, let every copy and MMA it started land, free
its tensor memory and return.  Each test then checks that the status is exactly TIMEOUT
(so the give-up path did run), re-initialises the workspace, and checks that the next
launch on the same context matches the CPU oracle.
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

MSA_ERR_TIMEOUT = -7
LIMIT_NS = 20_000_000   # 20 ms: long enough for every real copy, short for the test


@pytest.fixture(scope="module", autouse=True)
def built():
    B.build()
    msa.lib()


def _dropped_run(kernel, cta, index, launch):
    try:
        msa.set_wait_limit(LIMIT_NS)
        msa.set_test_drop(kernel, cta, index)
        launch()
        torch.cuda.synchronize()
    finally:
        msa.set_test_drop()
        msa.set_wait_limit(0)


def _decode_layout():
    specs = [W.SeqSpec([(0, 4096), (4112, 500)], np.zeros(0)) for _ in range(8)]
    return W.custom_decode(8, 2, 128, specs, seed=3, qk_std=0.5)


@pytest.mark.parametrize("index", [0, 1, 5])
def test_decode_gives_up_on_a_missing_block(index):
    lay = _decode_layout()
    wl = W.make_values(lay, device="cuda")
    plan = msa.Plan.from_layout(lay, decode_split_blocks=64).upload("cuda")
    _dropped_run("decode", 0, index, lambda: msa.decode(plan, wl.q, wl.k_pool, wl.v_pool))
    assert msa.get_status(plan) == MSA_ERR_TIMEOUT
    # the next launch, on a re-initialised workspace, is correct
    plan.upload("cuda")
    out, lse = msa.decode(plan, wl.q, wl.k_pool, wl.v_pool)
    torch.cuda.synchronize()
    assert msa.get_status(plan) == 0
    _, ro, rl = O.decode(lay, np64(wl.q), np64(wl.k_pool), np64(wl.v_pool), 1.0 / math.sqrt(128))
    assert_close(np64(out), ro, "decode out after a give-up")
    assert_close(np64(lse), rl, "decode lse after a give-up")


def _prefill_layout():
    rng = np.random.default_rng(51)
    specs = [W.random_prefill_spec(rng, 120, 0.5, 200, 1200), W.random_prefill_spec(rng, 40, 0.4, 60, 300)]
    return W.custom_prefill(8, 2, 128, specs, seed=51, qk_std=0.5)


@pytest.mark.parametrize("ctas,cta,index", [(148, 0, 0), (64, 3, 2), (64, 10, 7), (8, 1, 20)])
def test_prefill_gives_up_on_a_missing_tile(ctas, cta, index):
    """Drops at the first tile of a CTA, in the middle of a CTA's work and in a CTA that
    holds pieces of split work items (merged on the device by the last piece)."""
    lay = _prefill_layout()
    plan = msa.Plan.from_layout(lay, prefill_ctas=ctas).upload("cuda")
    sched = plan.export_schedule()
    mine = sched[sched[:, 0] == cta]
    assert mine[:, 5].sum() > index          # the CTA loads that many K tiles
    if ctas == 64:
        assert (sched[:, 6] > 1).any()       # the plan has split items
    wl = W.make_values(lay, device="cuda")
    _dropped_run("prefill", cta, index,
                  lambda: msa.prefill(plan, wl.q, wl.k_chunk, wl.v_chunk, wl.k_pool, wl.v_pool))
    assert msa.get_status(plan) == MSA_ERR_TIMEOUT
    plan.upload("cuda")
    out, lse = msa.prefill(plan, wl.q, wl.k_chunk, wl.v_chunk, wl.k_pool, wl.v_pool)
    torch.cuda.synchronize()
    assert msa.get_status(plan) == 0
    a = workload_arrays(wl)
    _, ro, rl = O.prefill(lay, a["q"], a["k_chunk"], a["v_chunk"], a["k_pool"], a["v_pool"], 1.0 / math.sqrt(128))
    assert_close(np64(out), ro, "prefill out after a give-up")
    assert_close(np64(lse), rl, "prefill lse after a give-up")


def test_hook_off_by_default_and_after_reset():
    """With the hook off (the default, and after turning it off) launches report no error."""
    lay = _decode_layout()
    wl = W.make_values(lay, device="cuda")
    plan = msa.Plan.from_layout(lay, decode_split_blocks=64).upload("cuda")
    msa.decode(plan, wl.q, wl.k_pool, wl.v_pool)
    assert msa.get_status(plan) == 0
    msa.set_test_drop("prefill", 0, 0)     # a prefill drop does not touch the decode
    try:
        msa.decode(plan, wl.q, wl.k_pool, wl.v_pool)
        assert msa.get_status(plan) == 0
    finally:
        msa.set_test_drop()
