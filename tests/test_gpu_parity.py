"""GPU parity of the MSA kernels against the CPU oracle, called through the C ABI.

Tolerance (bf16 inputs, fp32 accumulation): |gpu - oracle| <= 1e-2 + 2e-2 |oracle|
per element on O and LSE.  Indexing (gather) is compared bit for bit, and so are two
runs on the same data and two runs whose pool blocks sit at permuted physical ids.
"""
import math

import numpy as np
import pytest
import torch

import segmented_kv_attention_msa_b300 as msa
from segmented_kv_attention_msa_b300 import build as B
from segmented_kv_attention_msa_b300 import workload as W
from oracle import msa_oracle as O
from tests.helpers import (DevicePool, assert_close, empty_sequence_specs, export_tables, np64,
                           workload_arrays)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    B.build()
    msa.lib()


def run_prefill(lay, wl=None, plan_kw=None, **kw):
    wl = wl or W.make_values(lay, device="cuda")
    plan = msa.Plan.from_layout(lay, **(plan_kw or {})).upload("cuda")
    out, lse = msa.prefill(plan, wl.q, wl.k_chunk, wl.v_chunk, wl.k_pool, wl.v_pool, **kw)
    torch.cuda.synchronize()
    assert msa.get_status(plan) == 0
    return wl, out, lse


def check_prefill(lay, rows=None, scale=None, wl=None, plan_kw=None):
    wl, out, lse = run_prefill(lay, wl, plan_kw, scale=scale)
    a = workload_arrays(wl)
    sc = 1.0 / math.sqrt(lay.head_dim) if scale is None else scale
    rows_, ref_o, ref_l = O.prefill(lay, a["q"], a["k_chunk"], a["v_chunk"], a["k_pool"], a["v_pool"], sc,
                                    rows=rows)
    assert_close(np64(out)[rows_], ref_o, "out")
    assert_close(np64(lse)[rows_], ref_l, "lse")
    return wl, out, lse


# ----------------------------------------------------------------------------- merge / gather

def test_merge_lse_kernel():
    g = torch.Generator().manual_seed(3)
    rows, H, d = 37, 5, 128
    oa = torch.randn(rows, H, d, generator=g)
    ob = torch.randn(rows, H, d, generator=g)
    la = torch.randn(rows, H, generator=g) * 4
    lb = torch.randn(rows, H, generator=g) * 4
    la[0, 0] = -math.inf
    lb[1, 1] = -math.inf
    la[2, 2] = lb[2, 2] = -math.inf
    o, l = msa.merge_lse(oa.cuda(), la.cuda(), ob.cuda(), lb.cuda())
    ref_o, ref_l = O.merge_lse([oa.numpy(), ob.numpy()], [la.numpy(), lb.numpy()])
    assert_close(np64(o), ref_o, "merged out")
    assert_close(np64(l), ref_l, "merged lse")


def test_decode_merge_invariant_gpu():
    """Decode over segments A and over segments B, merged by msa_merge_lse, equals decode over A u B."""
    specs = [W.SeqSpec([(0, 512), (512, 300), (1024, 77), (816, 208)], np.zeros(0)) for _ in range(3)]
    lay = W.custom_decode(8, 2, 128, specs, seed=21, qk_std=0.6)
    wl = W.make_values(lay, device="cuda")
    plan = msa.Plan.from_layout(lay).upload("cuda")
    whole_o, whole_l = msa.decode(plan, wl.q, wl.k_pool, wl.v_pool)
    parts = []
    for sel in (slice(0, None, 2), slice(1, None, 2)):
        sub = W.Layout(**{**vars(lay), "segments": lay.segments[sel].copy()})
        p = msa.Plan.from_layout(sub).upload("cuda")
        o, l = msa.decode(p, wl.q, wl.k_pool, wl.v_pool)
        parts.append((o.float().contiguous(), l))
    mo, ml = msa.merge_lse(parts[0][0], parts[0][1], parts[1][0], parts[1][1])
    torch.cuda.synchronize()
    assert_close(np64(mo), np64(whole_o), "merged decode out")
    assert_close(np64(ml), np64(whole_l), "merged decode lse")


@pytest.mark.parametrize("idx", [1, 2])
def test_gather_bit_exact(idx):
    lay = W.make_layout(idx)
    wl = W.make_values(lay, device="cuda")
    plan = msa.Plan.from_layout(lay).upload("cuda")
    k, v, pos = msa.gather(plan, wl.k_chunk, wl.v_chunk, wl.k_pool, wl.v_pool)
    torch.cuda.synchronize()
    a = workload_arrays(wl)
    p_ref, k_ref, v_ref = O.gather_by_position(lay, 0, a["k_pool"], a["v_pool"], a["k_chunk"], a["v_chunk"])
    np.testing.assert_array_equal(pos.cpu().numpy(), p_ref)
    np.testing.assert_array_equal(np64(k), k_ref)
    np.testing.assert_array_equal(np64(v), v_ref)
    # into caller buffers longer than the context: the same rows, the tail untouched
    n = k.shape[0]
    ko = torch.full((n + 5, lay.num_heads_kv, lay.head_dim), 7.0, dtype=torch.bfloat16, device="cuda")
    vo = torch.full_like(ko, 9.0)
    po = torch.full((n + 5,), -3, dtype=torch.int32, device="cuda")
    k2, v2, p2 = msa.gather(plan, wl.k_chunk, wl.v_chunk, wl.k_pool, wl.v_pool, out=(ko, vo, po))
    torch.cuda.synchronize()
    assert k2.data_ptr() == ko.data_ptr() and k2.shape[0] == n
    assert torch.equal(k2, k) and torch.equal(v2, v) and torch.equal(p2, pos)
    assert torch.all(ko[n:] == 7.0) and torch.all(vo[n:] == 9.0) and torch.all(po[n:] == -3)


def test_gather_decode_bit_exact():
    lay = W.make_layout(4)
    lay = W.Layout(**{**vars(lay)})
    wl = W.make_values(lay, device="cuda")
    plan = msa.Plan.from_layout(lay).upload("cuda")
    k, v, pos = msa.gather(plan, None, None, wl.k_pool, wl.v_pool)
    torch.cuda.synchronize()
    a = workload_arrays(wl)
    empty = np.zeros((0, lay.num_heads_kv, lay.head_dim))
    off = 0
    for s in range(lay.num_seqs):
        p_ref, k_ref, v_ref = O.gather_by_position(lay, s, a["k_pool"], a["v_pool"], empty, empty)
        n = len(p_ref)
        if s in (0, 17, 63):
            np.testing.assert_array_equal(pos[off:off + n].cpu().numpy(), p_ref)
            np.testing.assert_array_equal(np64(k[off:off + n]), k_ref)
            np.testing.assert_array_equal(np64(v[off:off + n]), v_ref)
        off += n
    assert off == k.shape[0]


# ----------------------------------------------------------------------------- decode

def check_decode(lay, seqs=None, **plan_kw):
    wl = W.make_values(lay, device="cuda")
    plan = msa.Plan.from_layout(lay, **plan_kw).upload("cuda")
    out, lse = msa.decode(plan, wl.q, wl.k_pool, wl.v_pool)
    torch.cuda.synchronize()
    assert msa.get_status(plan) == 0
    q = np64(wl.q)
    kp, vp = np64(wl.k_pool), np64(wl.v_pool)
    seqs_, ref_o, ref_l = O.decode(lay, q, kp, vp, 1.0 / math.sqrt(lay.head_dim), seqs=seqs)
    assert_close(np64(out)[seqs_], ref_o, "decode out")
    assert_close(np64(lse)[seqs_], ref_l, "decode lse")
    return plan, out, lse


@pytest.mark.parametrize("Hq,Hkv,d", [(32, 8, 128), (8, 8, 128), (4, 2, 64), (16, 2, 128), (6, 3, 64),
                                        (32, 2, 128), (8, 1, 64)])
@pytest.mark.parametrize("split", [0, 1, 3])
def test_decode_small(Hq, Hkv, d, split):
    rng = np.random.default_rng(Hq * 7 + d + split)
    specs = []
    for _ in range(5):
        L = int(rng.integers(1, 900))
        nb = -(-L // 16)
        cuts = np.sort(rng.choice(np.arange(1, nb), size=min(nb - 1, int(rng.integers(0, 6))), replace=False)) \
            if nb > 1 else np.array([], int)
        edges = np.concatenate([[0], cuts, [nb]])
        specs.append(W.SeqSpec([(int(a) * 16, min(int(b) * 16, L) - int(a) * 16)
                                for a, b in zip(edges[:-1], edges[1:])], np.zeros(0)))
    lay = W.custom_decode(Hq, Hkv, d, specs, seed=split, qk_std=1.0 / math.sqrt(d) * 4, shuffle_segments=True)
    check_decode(lay, decode_split_blocks=split)


def test_decode_sharp_logits():
    specs = [W.SeqSpec([(0, 1000), (1008, 333)], np.zeros(0)) for _ in range(4)]
    lay = W.custom_decode(32, 8, 128, specs, seed=5, qk_std=1.0)   # no 1/sqrt(d) pre-scaling
    check_decode(lay, decode_split_blocks=8)


def test_decode_workload4_all_sequences():
    """All 64 sequences of the decode workload against the oracle (the oracle reads the
    pool rows it needs straight from the device tensor)."""
    lay = W.make_layout(4)
    wl = W.make_values(lay, device="cuda")
    plan = msa.Plan.from_layout(lay).upload("cuda")
    out, lse = msa.decode(plan, wl.q, wl.k_pool, wl.v_pool)
    torch.cuda.synchronize()
    assert msa.get_status(plan) == 0
    seqs_, ref_o, ref_l = O.decode(lay, np64(wl.q), DevicePool(wl.k_pool), DevicePool(wl.v_pool),
                                   1.0 / math.sqrt(lay.head_dim))
    assert len(seqs_) == 64
    assert_close(np64(out), ref_o, "decode out")
    assert_close(np64(lse), ref_l, "decode lse")


def test_decode_deterministic_and_permutation_invariant():
    specs = [W.SeqSpec([(0, 700), (704, 90)], np.zeros(0)) for _ in range(3)]
    lay_a = W.custom_decode(8, 2, 128, specs, seed=1)
    lay_b = W.custom_decode(8, 2, 128, specs, seed=2)     # other physical placement
    wa = W.make_values(lay_a, device="cuda", seed=77)
    # re-place the same logical values at lay_b's block ids
    kb = torch.zeros(lay_b.num_pool_blocks, *wa.k_pool.shape[1:], dtype=wa.k_pool.dtype, device="cuda")
    vb = torch.zeros_like(kb)
    for (s, f, nb) in lay_a.segments:
        for i in range(nb):
            ba = int(lay_a.block_table[s, f + i])
            pos = int(lay_a.block_pos[ba])
            row_b = [x for x in lay_b.block_table[s] if x >= 0 and lay_b.block_pos[x] == pos and
                     lay_b.block_fill[x] > 0]
            kb[row_b[0]] = wa.k_pool[ba]
            vb[row_b[0]] = wa.v_pool[ba]
    pa = msa.Plan.from_layout(lay_a).upload("cuda")
    pb = msa.Plan.from_layout(lay_b).upload("cuda")
    o1, l1 = msa.decode(pa, wa.q, wa.k_pool, wa.v_pool)
    o2, l2 = msa.decode(pa, wa.q, wa.k_pool, wa.v_pool)
    o3, l3 = msa.decode(pb, wa.q, kb, vb)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    assert torch.equal(o1, o3) and torch.equal(l1, l3)


# ----------------------------------------------------------------------------- prefill

def test_prefill_workload1_all_rows():
    check_prefill(W.make_layout(1))


def test_prefill_workload2_all_rows():
    check_prefill(W.make_layout(2))


def test_prefill_workload3_sampled():
    lay = W.make_layout(3, tiler=msa.chunk_sizes)
    rng = np.random.default_rng(0)
    rows = np.sort(rng.choice(lay.total_q, 400, replace=False))
    rows = np.unique(np.concatenate([rows, lay.cu_q[:-1], lay.cu_q[1:] - 1]))
    check_prefill(lay, rows=rows)


def test_prefill_workload5_sampled():
    """Random rows, plus rows of every query tile whose work item is cut into pieces that
    are merged on the device, and of query tiles with partial (masked) mixed tiles."""
    lay = W.make_layout(5)
    plan = msa.Plan.from_layout(lay)
    sched = plan.export_schedule()
    _, kt, qt, cls = export_tables(plan.export())
    split_qt = np.unique(sched[sched[:, 6] > 1, 1])
    assert len(split_qt) > 0
    nkt = len(kt)
    mixed_partial = [i for i in range(len(qt))
                     if np.any((cls[i * nkt:(i + 1) * nkt] == O.PARTIAL) & (kt[:, 1] == O.MIXED))]
    assert len(mixed_partial) > 0
    rng = np.random.default_rng(1)
    pick_qt = np.unique(np.concatenate([rng.choice(split_qt, min(12, len(split_qt)), replace=False),
                                        rng.choice(mixed_partial, min(8, len(mixed_partial)), replace=False)]))
    rows = [rng.choice(lay.total_q, 64, replace=False), [0, lay.total_q - 1]]
    for i in pick_qt:
        r0, n = int(qt[i, 1]), int(qt[i, 2])
        rows.append([r0, r0 + n // 2, r0 + n - 1])
    check_prefill(lay, rows=np.unique(np.concatenate(rows)))


def _spec(pool_runs, chunk):
    return W.SeqSpec(pool_runs, np.asarray(chunk))


@pytest.mark.parametrize("case", ["no_cache", "prefix_only", "one_token", "single_segment",
                                  "partial_blocks", "ragged_multi", "future_blocks", "tiny_tiles",
                                  "sparse_chunk", "fragmented"])
@pytest.mark.parametrize("heads", [(32, 8, 128), (4, 4, 64), (6, 2, 128), (3, 3, 64), (32, 2, 128), (8, 1, 64)])
def test_prefill_edge_cases(case, heads):
    Hq, Hkv, d = heads
    rng = np.random.default_rng(hash(case) % 1000)
    if case == "no_cache":
        specs = [_spec([], np.arange(300))]
    elif case == "prefix_only":
        specs = [_spec([(0, 1024)], np.arange(1024, 1400))]
    elif case == "one_token":
        specs = [_spec([(0, 512), (528, 48)], [512]), _spec([(0, 16)], [16])]
    elif case == "single_segment":
        specs = [_spec([(256, 512)], np.concatenate([np.arange(0, 256), np.arange(768, 800)]))]
    elif case == "partial_blocks":
        specs = [_spec([(0, 37), (48, 100), (160, 9)], np.concatenate([np.arange(37, 48), np.arange(148, 160),
                                                                       np.arange(169, 420)]))]
    elif case == "ragged_multi":
        specs = [W.random_prefill_spec(rng, int(rng.integers(2, 70)), 0.5, int(rng.integers(1, 200)),
                                       int(rng.integers(1, 400))) for _ in range(5)]
    elif case == "future_blocks":
        specs = [_spec([(0, 128), (640, 512)], np.arange(128, 640))]
    elif case == "sparse_chunk":
        # chunk positions with gaps (held by neither side), so consecutive chunk rows of one
        # 16-key unit are not consecutive positions; partial pool blocks between them
        pool = [(0, 16), (64, 16), (128, 40)]
        free = np.concatenate([np.arange(16, 64), np.arange(80, 128), np.arange(168, 700)])
        specs = [_spec(pool, np.sort(rng.choice(free, 330, replace=False)))]
    elif case == "fragmented":
        # half of 96 blocks cached at random, everything else recomputed in this launch:
        # most KV tiles mix pool blocks and chunk rows
        specs = [W.random_prefill_spec(rng, 96, 0.5, 40), W.random_prefill_spec(rng, 30, 0.3, 7)]
    else:  # tiny_tiles: alternating single cached blocks and single chunk tokens
        runs = [(32 * i, 16) for i in range(20)]
        chunk = np.concatenate([np.arange(32 * i + 16, 32 * i + 17) for i in range(20)])
        specs = [_spec(runs, chunk)]
    lay = W.custom_prefill(Hq, Hkv, d, specs, seed=4, qk_std=1.0 / math.sqrt(d) * 3, shuffle_segments=True)
    check_prefill(lay)


@pytest.mark.parametrize("heads", [(4, 2, 64), (32, 8, 128)])
def test_prefill_empty_sequences(heads):
    """Sequences with no chunk rows between sequences that have some: rows of the others
    are unaffected and nothing is written for the empty ones."""
    Hq, Hkv, d = heads
    lay = W.custom_prefill(Hq, Hkv, d, empty_sequence_specs(), seed=3, qk_std=1.0 / math.sqrt(d) * 3)
    check_prefill(lay)


def test_prefill_without_query_rows():
    lay = W.custom_prefill(4, 2, 64, [W.SeqSpec([(0, 48)], np.array([], np.int64))], seed=3)
    wl = W.make_values(lay, device="cuda")
    plan = msa.Plan.from_layout(lay).upload("cuda")
    out, lse = msa.prefill(plan, wl.q, wl.k_chunk, wl.v_chunk, wl.k_pool, wl.v_pool)
    torch.cuda.synchronize()
    assert out.shape[0] == 0 and lse.shape[0] == 0
    assert msa.get_status(plan) == 0


def test_zero_rows_merge_and_append():
    o = torch.empty(0, 4, 64, dtype=torch.float32, device="cuda")
    l = torch.empty(0, 4, dtype=torch.float32, device="cuda")
    out, lse = msa.merge_lse(o, l, o, l)
    assert out.shape == (0, 4, 64) and lse.shape == (0, 4)
    kp = torch.zeros(2, 2, 16, 64, dtype=torch.bfloat16, device="cuda")
    vp = torch.zeros_like(kp)
    none = torch.empty(0, 2, 64, dtype=torch.bfloat16, device="cuda")
    msa.kv_append(torch.empty(0, dtype=torch.int32, device="cuda"), none, none, kp, vp)
    torch.cuda.synchronize()
    assert int(kp.count_nonzero()) == 0 and int(vp.count_nonzero()) == 0


def test_prefill_sharp_logits():
    rng = np.random.default_rng(5)
    spec = W.random_prefill_spec(rng, 64, 0.5, 200, 700)
    lay = W.custom_prefill(16, 4, 128, [spec], seed=5, qk_std=1.0)
    check_prefill(lay)


def test_prefill_planted_maxima():
    """Planted large logits at random keys force the running max to move across tiles."""
    rng = np.random.default_rng(6)
    spec = W.random_prefill_spec(rng, 80, 0.5, 300, 900)
    lay = W.custom_prefill(8, 2, 128, [spec], seed=6, qk_std=0.2)
    wl = W.make_values(lay, device="cuda")
    nb = lay.num_pool_blocks
    for _ in range(40):
        b = int(rng.integers(0, nb))
        t = int(rng.integers(0, 16))
        wl.k_pool[b, :, t, :] = wl.q[int(rng.integers(0, lay.total_q)), :2, :].mean(0) * 6
    for _ in range(10):
        r = int(rng.integers(0, lay.total_q))
        wl.k_chunk[r] = wl.q[r, ::4, :] * 6
    check_prefill(lay, wl=wl)


def test_prefill_deterministic_and_permutation_invariant():
    rng = np.random.default_rng(8)
    spec = W.random_prefill_spec(rng, 60, 0.6, 150, 600)
    lay_a = W.custom_prefill(8, 2, 128, [spec], seed=11)
    lay_b = W.custom_prefill(8, 2, 128, [spec], seed=12)
    wa = W.make_values(lay_a, device="cuda", seed=5)
    kb = torch.zeros(lay_b.num_pool_blocks, *wa.k_pool.shape[1:], dtype=torch.bfloat16, device="cuda")
    vb = torch.zeros_like(kb)
    pos_to_b = {int(lay_b.block_pos[x]): int(x) for x in lay_b.block_table[0] if x >= 0}
    for x in lay_a.block_table[0]:
        if x >= 0:
            kb[pos_to_b[int(lay_a.block_pos[x])]] = wa.k_pool[x]
            vb[pos_to_b[int(lay_a.block_pos[x])]] = wa.v_pool[x]
    pa = msa.Plan.from_layout(lay_a).upload("cuda")
    pb = msa.Plan.from_layout(lay_b).upload("cuda")
    o1, l1 = msa.prefill(pa, wa.q, wa.k_chunk, wa.v_chunk, wa.k_pool, wa.v_pool)
    o2, l2 = msa.prefill(pa, wa.q, wa.k_chunk, wa.v_chunk, wa.k_pool, wa.v_pool)
    o3, l3 = msa.prefill(pb, wa.q, wa.k_chunk, wa.v_chunk, kb, vb)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    assert torch.equal(o1, o3) and torch.equal(l1, l3)


@pytest.mark.parametrize("ctas", [1, 2, 5, 8, 24, 37, 64, 148, 1000])
def test_prefill_schedules(ctas):
    """The same layout balanced over different CTA counts: whole items, items cut into
    2 or more pieces merged on the device (8, 24 and 64 CTAs and up cut some); every
    schedule matches the oracle and is bit-reproducible."""
    rng = np.random.default_rng(31)
    specs = [W.random_prefill_spec(rng, 90, 0.5, 120, 900), W.random_prefill_spec(rng, 30, 0.3, 40, 300)]
    lay = W.custom_prefill(8, 2, 128, specs, seed=31, qk_std=0.5)
    plan = msa.Plan.from_layout(lay, prefill_ctas=ctas)
    sc = plan.export_schedule()
    if ctas in (8, 24) or ctas >= 64:
        assert (sc[:, 6] > 1).any()          # some items are split and merged
    wl, o1, l1 = check_prefill(lay, plan_kw={"prefill_ctas": ctas})
    _, o2, l2 = run_prefill(lay, wl, {"prefill_ctas": ctas})
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_prefill_split_sharp_logits():
    """Items cut into pieces whose maxima differ by a lot (unscaled logits, planted keys):
    the log-sum-exp merge of the pieces must still match the oracle."""
    rng = np.random.default_rng(32)
    spec = W.random_prefill_spec(rng, 120, 0.6, 64, 1024)
    lay = W.custom_prefill(4, 1, 128, [spec], seed=32, qk_std=1.0)
    wl = W.make_values(lay, device="cuda")
    for _ in range(12):
        b = int(rng.integers(0, lay.num_pool_blocks))
        wl.k_pool[b, :, int(rng.integers(0, 16)), :] = wl.q[int(rng.integers(0, lay.total_q)), :1, :] * 4
    check_prefill(lay, wl=wl, plan_kw={"prefill_ctas": 64})


def _with_segments(lay, segs):
    return W.Layout(**{**vars(lay), "segments": np.asarray(segs, np.int32).reshape(-1, 3)})


@pytest.mark.parametrize("seed", [41, 42])
def test_prefill_queries_only_and_per_segment_merge(seed):
    """Queries-only plans (KV = pool segments alone) match the oracle, including rows that
    see no key of their segment (O = 0, LSE = -inf); one launch per segment plus one over
    the chunk's own keys, merged by log-sum-exp on the GPU, matches the single MSA launch."""
    rng = np.random.default_rng(seed)
    spec = W.random_prefill_spec(rng, 70, 0.5, 150, 700)
    lay = W.custom_prefill(8, 2, 128, [spec], seed=seed, qk_std=0.6)
    wl = W.make_values(lay, device="cuda")
    a = workload_arrays(wl)
    sc = 1.0 / math.sqrt(128)
    whole_o, whole_l = run_prefill(lay, wl)[1:]
    parts = []
    for seg in lay.segments:
        sub = _with_segments(lay, [seg])
        plan = msa.Plan.from_layout(sub, chunk_queries_only=True).upload("cuda")
        o, l = msa.prefill(plan, wl.q, wl.k_chunk, wl.v_chunk, wl.k_pool, wl.v_pool)
        torch.cuda.synchronize()
        assert msa.get_status(plan) == 0
        _, ro, rl = O.prefill(sub, a["q"], a["k_chunk"], a["v_chunk"], a["k_pool"], a["v_pool"], sc,
                              chunk_keys=False)
        assert_close(np64(o), ro, "queries-only out")
        assert_close(np64(l), rl, "queries-only lse")
        parts.append((o, l))
    nothing = _with_segments(lay, [])
    parts.append(run_prefill(nothing, wl)[1:])
    assert any(torch.isinf(l).any() for _, l in parts[:-1])
    acc_o, acc_l = parts[0][0].float().contiguous(), parts[0][1]
    for o, l in parts[1:]:
        mo, ml = msa.merge_lse(acc_o, acc_l, o.float().contiguous(), l)
        acc_o, acc_l = mo.float().contiguous(), ml
    torch.cuda.synchronize()
    assert_close(np64(acc_o), np64(whole_o), "per-segment merged out")
    assert_close(np64(acc_l), np64(whole_l), "per-segment merged lse")
