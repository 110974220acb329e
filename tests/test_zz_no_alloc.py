"""msa_decode_no_alloc: the decode for callers that cannot allocate device memory.

Such callers (an engine that reserves nearly all of HBM for its KV-cache pool at
start-up, or a loop that must not call cudaMalloc/cudaFree because they can
synchronise the device) get a decode whose split-KV scratch lives in a fixed array
owned by the library.  The test calls it through the C ABI twice in a row and checks
each result against the regular msa_decode (which uses a caller workspace) and against
the CPU oracle, within the parity tolerance; checks that a plan needing more scratch
than the array holds is rejected; and makes one of its bounded waits run out (test
hook), reads MSA_ERR_TIMEOUT back through msa_get_status_no_alloc, and checks that the
next call is correct again.  This file is collected last on purpose.
"""
import ctypes
import math

import numpy as np
import pytest
import torch

import segmented_kv_attention_msa_b300 as msa
from segmented_kv_attention_msa_b300 import build as B
from segmented_kv_attention_msa_b300 import workload as W
from oracle import msa_oracle as O
from tests.helpers import assert_close, np64

pytestmark = pytest.mark.gpu

MSA_ERR_WORKSPACE = -5
MSA_ERR_TIMEOUT = -7


def _call(plan, q, k_pool, v_pool, out, lse, scale):
    stream = torch.cuda.current_stream().cuda_stream
    return msa.lib().msa_decode_no_alloc(plan.handle, plan.dev.data_ptr(), q.data_ptr(), k_pool.data_ptr(),
                                         v_pool.data_ptr(), out.data_ptr(), lse.data_ptr(),
                                         ctypes.c_float(scale), ctypes.c_void_p(stream))


def _status():
    return msa.lib().msa_get_status_no_alloc(ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def _layout():
    specs = []
    rng = np.random.default_rng(41)
    for _ in range(12):
        L = int(rng.integers(300, 5000))
        nb = -(-L // 16)
        cuts = np.sort(rng.choice(np.arange(1, nb), size=int(rng.integers(1, 8)), replace=False))
        edges = np.concatenate([[0], cuts, [nb]])
        specs.append(W.SeqSpec([(int(a) * 16, min(int(b) * 16, L) - int(a) * 16)
                                for a, b in zip(edges[:-1], edges[1:])], np.zeros(0)))
    return W.custom_decode(32, 8, 128, specs, seed=41, qk_std=0.3, shuffle_segments=True)


def test_no_alloc_decode_matches_regular_decode_twice():
    B.build()
    lay = _layout()
    wl = W.make_values(lay, device="cuda")
    plan = msa.Plan.from_layout(lay, decode_split_blocks=24).upload("cuda")
    assert plan.workspace_bytes <= (8 << 20)
    scale = 1.0 / math.sqrt(128)
    ref_o, ref_l = msa.decode(plan, wl.q, wl.k_pool, wl.v_pool, scale=scale)
    torch.cuda.synchronize()
    _, oro, orl = O.decode(lay, np64(wl.q), np64(wl.k_pool), np64(wl.v_pool), scale)
    for _ in range(2):
        out = torch.full_like(wl.q, float("nan"))
        lse = torch.full((lay.num_seqs, 32), float("nan"), dtype=torch.float32, device="cuda")
        assert _call(plan, wl.q, wl.k_pool, wl.v_pool, out, lse, scale) == 0
        torch.cuda.synchronize()
        assert _status() == 0
        assert_close(np64(out), np64(ref_o), "no-alloc decode out vs msa_decode")
        assert_close(np64(lse), np64(ref_l), "no-alloc decode lse vs msa_decode")
        assert_close(np64(out), oro, "no-alloc decode out vs oracle")
        assert_close(np64(lse), orl, "no-alloc decode lse vs oracle")


def test_no_alloc_decode_reports_a_wait_that_ran_out():
    """The wait limit of msa_set_wait_limit applies; a wait that runs out (one block left
    out by the test hook) is reported by msa_get_status_no_alloc, and the next call, which
    re-arms the shared scratch, is correct."""
    B.build()
    lay = _layout()
    wl = W.make_values(lay, device="cuda")
    plan = msa.Plan.from_layout(lay, decode_split_blocks=24).upload("cuda")
    scale = 1.0 / math.sqrt(128)
    ref_o, ref_l = msa.decode(plan, wl.q, wl.k_pool, wl.v_pool, scale=scale)
    out = torch.empty_like(wl.q)
    lse = torch.empty(lay.num_seqs, 32, dtype=torch.float32, device="cuda")
    try:
        msa.set_wait_limit(20_000_000)
        msa.set_test_drop("decode", 0, 1)
        assert _call(plan, wl.q, wl.k_pool, wl.v_pool, out, lse, scale) == 0
        assert _status() == MSA_ERR_TIMEOUT
    finally:
        msa.set_test_drop()
        msa.set_wait_limit(0)
    assert _status() == 0                     # read and cleared
    assert _call(plan, wl.q, wl.k_pool, wl.v_pool, out, lse, scale) == 0
    torch.cuda.synchronize()
    assert _status() == 0
    assert_close(np64(out), np64(ref_o), "no-alloc decode out after a give-up")
    assert_close(np64(lse), np64(ref_l), "no-alloc decode lse after a give-up")


def test_no_alloc_decode_rejects_oversized_plan():
    B.build()
    specs = [W.SeqSpec([(0, 16 * 700)], np.zeros(0))]
    lay = W.custom_decode(32, 8, 128, specs, seed=2)
    plan = msa.Plan.from_layout(lay, decode_split_blocks=1).upload("cuda")
    assert plan.workspace_bytes > (8 << 20)
    wl = W.make_values(lay, device="cuda")
    out = torch.empty_like(wl.q)
    lse = torch.empty(1, 32, dtype=torch.float32, device="cuda")
    assert _call(plan, wl.q, wl.k_pool, wl.v_pool, out, lse, 0.1) == MSA_ERR_WORKSPACE
