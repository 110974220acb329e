"""The MSA_DEBUG build (libmsa_debug.so): device-side bounds checks that never trap.

Its kernels check every work record, list entry, block id and block fill they read
against the plan and the pool; a bad one sets MSA_ERR_BLOCK_OOB in the status word and is
replaced by a safe value (a pool row past the end, which the tensor copy fills with
zeros).  The package loads this build when MSA_LIBRARY=debug, so each check runs in a
child process:
* clean runs (the tiny and the Llama-3-8B-shaped prefill, a GQA decode) report no error,
  match the CPU oracle and equal the regular build's results bit for bit;
* a plan image whose KV-tile block ids (prefill) or block list (decode) were overwritten
  on the device with ids past the pool reports MSA_ERR_BLOCK_OOB instead of reading
  outside the pool.
"""
import json
import math
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

import segmented_kv_attention_msa_b300 as msa
from segmented_kv_attention_msa_b300 import build as B
from segmented_kv_attention_msa_b300 import workload as W
from oracle import msa_oracle as O
from tests.helpers import assert_close, np64, workload_arrays

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
MSA_ERR_BLOCK_OOB = -4


def _decode_layout():
    specs = [W.SeqSpec([(0, 700), (704, 333), (1040, 90)], np.zeros(0)) for _ in range(5)]
    return W.custom_decode(16, 4, 128, specs, seed=71, qk_std=0.4)


def _align(x):
    return (x + 255) // 256 * 256


def child(outdir):
    """Runs inside MSA_LIBRARY=debug: clean runs, then corrupted plan images."""
    assert msa.LIB_PATH.endswith("libmsa_debug.so")
    res = {}
    for idx in (1, 2):
        lay = W.make_layout(idx)
        wl = W.make_values(lay, device="cuda")
        plan = msa.Plan.from_layout(lay).upload("cuda")
        out, lse = msa.prefill(plan, wl.q, wl.k_chunk, wl.v_chunk, wl.k_pool, wl.v_pool)
        torch.cuda.synchronize()
        res[f"prefill{idx}_status"] = msa.get_status(plan)
        np.save(os.path.join(outdir, f"prefill{idx}_out.npy"), out.view(torch.int16).cpu().numpy())
        np.save(os.path.join(outdir, f"prefill{idx}_lse.npy"), lse.cpu().numpy())
    lay = _decode_layout()
    wl = W.make_values(lay, device="cuda")
    plan = msa.Plan.from_layout(lay, decode_split_blocks=8).upload("cuda")
    out, lse = msa.decode(plan, wl.q, wl.k_pool, wl.v_pool)
    torch.cuda.synchronize()
    res["decode_status"] = msa.get_status(plan)
    np.save(os.path.join(outdir, "decode_out.npy"), out.view(torch.int16).cpu().numpy())
    np.save(os.path.join(outdir, "decode_lse.npy"), lse.cpu().numpy())

    # prefill with its KV tiles' pool block ids overwritten (image sections are 256-byte
    # aligned: query positions, query tiles of 8 int32, KV tiles of 32 int32 whose words
    # 8..15 are the units' block ids, negative for chunk rows)
    lay = W.make_layout(1)
    wl = W.make_values(lay, device="cuda")
    plan = msa.Plan.from_layout(lay).upload("cuda")
    st = plan.stats()
    k0 = (_align(lay.total_q * 4) + _align(st["num_q_tiles"] * 32)) // 4
    img = plan.dev.view(torch.int32)
    recs = img[k0:k0 + 32 * st["num_kv_tiles"]].view(-1, 32)
    blk = recs[:, 8:16]
    nblk = recs[:, 3:4]
    unit = torch.arange(8, device=blk.device)[None, :] < nblk
    pool_unit = unit & (blk >= 0)
    assert int(pool_unit.sum()) > 0
    blk[pool_unit] = lay.num_pool_blocks + 3
    msa.prefill(plan, wl.q, wl.k_chunk, wl.v_chunk, wl.k_pool, wl.v_pool)
    torch.cuda.synchronize()
    res["prefill_corrupt_status"] = msa.get_status(plan)

    # decode with one entry of its block list overwritten: find sequence 0's blocks, in
    # position order, as a run of the image
    lay = _decode_layout()
    wl = W.make_values(lay, device="cuda")
    plan = msa.Plan.from_layout(lay, decode_split_blocks=8).upload("cuda")
    rows = [int(b) for b in lay.block_table[0] if b >= 0]
    rows.sort(key=lambda b: int(lay.block_pos[b]))
    img_h = plan.dev.view(torch.int32).cpu().numpy()
    run = np.array(rows[:4], np.int32)
    hits = [i for i in range(len(img_h) - 4) if np.array_equal(img_h[i:i + 4], run)]
    assert len(hits) == 1, hits
    plan.dev.view(torch.int32)[hits[0] + 1] = lay.num_pool_blocks + 5
    msa.decode(plan, wl.q, wl.k_pool, wl.v_pool)
    torch.cuda.synchronize()
    res["decode_corrupt_status"] = msa.get_status(plan)
    with open(os.path.join(outdir, "res.json"), "w") as f:
        json.dump(res, f)


def test_debug_build(tmp_path):
    B.build()
    B.build(debug=True)
    env = dict(os.environ, MSA_LIBRARY="debug")
    code = f"import sys; sys.path.insert(0, {ROOT!r}); import tests.test_gpu_debug_build as T; T.child({str(tmp_path)!r})"
    r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout + r.stderr
    res = json.load(open(tmp_path / "res.json"))
    assert res["prefill1_status"] == 0 and res["prefill2_status"] == 0 and res["decode_status"] == 0
    assert res["prefill_corrupt_status"] == MSA_ERR_BLOCK_OOB
    assert res["decode_corrupt_status"] == MSA_ERR_BLOCK_OOB

    # the regular build gives the same bits, and both match the oracle
    for idx in (1, 2):
        lay = W.make_layout(idx)
        wl = W.make_values(lay, device="cuda")
        plan = msa.Plan.from_layout(lay).upload("cuda")
        out, lse = msa.prefill(plan, wl.q, wl.k_chunk, wl.v_chunk, wl.k_pool, wl.v_pool)
        torch.cuda.synchronize()
        assert np.array_equal(out.view(torch.int16).cpu().numpy(), np.load(tmp_path / f"prefill{idx}_out.npy"))
        assert np.array_equal(lse.cpu().numpy(), np.load(tmp_path / f"prefill{idx}_lse.npy"))
        a = workload_arrays(wl)
        _, ro, rl = O.prefill(lay, a["q"], a["k_chunk"], a["v_chunk"], a["k_pool"], a["v_pool"],
                              1.0 / math.sqrt(lay.head_dim))
        assert_close(np64(out), ro, f"prefill {idx} out")
        assert_close(np64(lse), rl, f"prefill {idx} lse")
    lay = _decode_layout()
    wl = W.make_values(lay, device="cuda")
    plan = msa.Plan.from_layout(lay, decode_split_blocks=8).upload("cuda")
    out, lse = msa.decode(plan, wl.q, wl.k_pool, wl.v_pool)
    torch.cuda.synchronize()
    assert np.array_equal(out.view(torch.int16).cpu().numpy(), np.load(tmp_path / "decode_out.npy"))
    assert np.array_equal(lse.cpu().numpy(), np.load(tmp_path / "decode_lse.npy"))
    _, ro, rl = O.decode(lay, np64(wl.q), np64(wl.k_pool), np64(wl.v_pool), 1.0 / math.sqrt(128))
    assert_close(np64(out), ro, "decode out")
    assert_close(np64(lse), rl, "decode lse")
