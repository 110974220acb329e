"""GPU checks of the write-back step (chunk K/V into pool blocks at their original
positions), called through the C ABI: the copy is bit-exact against the oracle, and a
prefill -> write-back -> decode sequence over the pool alone sees exactly the KV context
the prefill saw (pool segments plus the chunk), by position."""
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


@pytest.fixture(scope="module", autouse=True)
def built():
    B.build()
    msa.lib()


@pytest.mark.parametrize("hkv,d", [(8, 128), (2, 64)])
def test_kv_append_bit_exact(hkv, d):
    g = torch.Generator(device="cuda").manual_seed(hkv + d)
    nblocks, n = 40, 300
    kp = torch.randn(nblocks, hkv, 16, d, generator=g, device="cuda").to(torch.bfloat16)
    vp = torch.randn(nblocks, hkv, 16, d, generator=g, device="cuda").to(torch.bfloat16)
    kc = torch.randn(n, hkv, d, generator=g, device="cuda").to(torch.bfloat16)
    vc = torch.randn(n, hkv, d, generator=g, device="cuda").to(torch.bfloat16)
    rng = np.random.default_rng(d)
    slots = rng.permutation(nblocks * 16)[:n].astype(np.int32)
    slots[rng.choice(n, 20, replace=False)] = -1                     # skipped rows
    ref_k, ref_v = O.append(np64(kc), np64(vc), np64(kp), np64(vp), slots)
    msa.kv_append(torch.from_numpy(slots).cuda(), kc, vc, kp, vp)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(np64(kp), ref_k)
    np.testing.assert_array_equal(np64(vp), ref_v)


def _decode_layout_after_append(lay, s, new_blocks, block_pos, block_fill, q_pos_last):
    """Decode layout of sequence ``s`` over the pool alone: its old segments plus one
    segment per freshly written block."""
    row = [int(b) for b in lay.block_table[s] if b >= 0]
    segs = [(0, int(f), int(nb)) for (q, f, nb) in lay.segments if q == s]
    for b in new_blocks:
        segs.append((0, len(row), 1))
        row.append(int(b))
    table = np.array([row], np.int32)
    return W.Layout(mode="decode", num_heads_q=lay.num_heads_q, num_heads_kv=lay.num_heads_kv,
                    head_dim=lay.head_dim, num_seqs=1, num_pool_blocks=lay.num_pool_blocks,
                    block_pos=block_pos, block_fill=block_fill, block_table=table,
                    segments=np.array(segs, np.int32), cu_q=np.array([0, 1], np.int32),
                    q_pos=np.array([q_pos_last], np.int32), qk_std=lay.qk_std, v_std=lay.v_std,
                    name="after_append", seed=lay.seed)


@pytest.mark.parametrize("seed", [1, 2])
def test_prefill_append_decode(seed):
    rng = np.random.default_rng(seed)
    # old context of 60 blocks ending 7 tokens into block 60 (a partial cached block that the
    # new suffix continues), half of the whole blocks evicted and recomputed in the chunk
    cached = rng.random(60) < 0.5
    runs = [(p0, n) for (p0, n) in W._cached_runs_tokens(cached)] + [(60 * 16, 7)]
    evicted = np.flatnonzero(~cached)
    chunk = np.concatenate([np.arange(b * 16, b * 16 + 16) for b in evicted] + [np.arange(60 * 16 + 7, 60 * 16 + 90)])
    spec = W.SeqSpec(runs, chunk)
    lay = W.custom_prefill(8, 2, 128, [spec], seed=seed, qk_std=0.4, pool_slack=3.0)
    wl = W.make_values(lay, device="cuda")
    plan = msa.Plan.from_layout(lay).upload("cuda")
    out, lse = msa.prefill(plan, wl.q, wl.k_chunk, wl.v_chunk, wl.k_pool, wl.v_pool)
    torch.cuda.synchronize()
    # what the prefill saw, by position: pool segments plus the chunk
    p_ref, k_ref, v_ref = O.gather_by_position(lay, 0, np64(wl.k_pool), np64(wl.v_pool), np64(wl.k_chunk),
                                               np64(wl.v_chunk))
    # write the chunk back
    used = set(int(b) for b in lay.block_table[0] if b >= 0)
    free = [b for b in range(lay.num_pool_blocks) if b not in used]
    bp, bf = lay.block_pos.copy(), lay.block_fill.copy()
    dst, new = msa.append_plan(lay.q_pos, free, bp, bf, seq_blocks=sorted(used))
    msa.kv_append(torch.from_numpy(dst).cuda(), wl.k_chunk, wl.v_chunk, wl.k_pool, wl.v_pool)
    torch.cuda.synchronize()
    dl = _decode_layout_after_append(lay, 0, new, bp, bf, int(p_ref[-1]))
    dplan = msa.Plan.from_layout(dl).upload("cuda")
    k, v, pos = msa.gather(dplan, None, None, wl.k_pool, wl.v_pool)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(pos.cpu().numpy(), p_ref)
    np.testing.assert_array_equal(np64(k), k_ref)
    np.testing.assert_array_equal(np64(v), v_ref)
    # decode of a new query over the pool alone against the oracle
    q = torch.randn(1, 8, 128, device="cuda").mul_(0.4).to(torch.bfloat16)
    dout, dlse = msa.decode(dplan, q, wl.k_pool, wl.v_pool)
    torch.cuda.synchronize()
    assert msa.get_status(dplan) == 0
    _, ro, rl = O.decode(dl, np64(q), np64(wl.k_pool), np64(wl.v_pool), 1.0 / math.sqrt(128))
    assert_close(np64(dout), ro, "decode after write-back")
    assert_close(np64(dlse), rl, "decode lse after write-back")
