"""Pins of the CPU oracle against things other than itself.

Each test ties the oracle to mathematics or an independent textbook routine:
brute-force causal attention over the contiguous sequence (the paper's lossless
claim: recomputed blocks at their original positions give exactly ordinary
attention), the LSE-merge invariant over disjoint key sets, closed forms, special
cases (no cache, prefix cache, single key, decode), a hand-worked example, and the
written rules of the plan and the chunk tiler.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

from oracle import msa_oracle as O
from segmented_kv_attention_msa_b300 import workload as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ----------------------------------------------------------------------------- helpers

def scatter_from_contiguous(layout, Kc, Vc, Qc):
    """Fill pool / chunk tensors of ``layout`` from a contiguous sequence per seq.

    Kc[s], Vc[s]: [L_s, Hkv, d] indexed by original position; Qc[s]: [L_s, Hq, d].
    Written with direct indexing of the block table (independent of the oracle).
    """
    Hkv, d, Hq = layout.num_heads_kv, layout.head_dim, layout.num_heads_q
    kp = np.zeros((layout.num_pool_blocks, Hkv, 16, d))
    vp = np.zeros_like(kp)
    for (s, first, nb) in layout.segments:
        for lb in range(first, first + nb):
            b = layout.block_table[s, lb]
            for t in range(layout.block_fill[b]):
                p = layout.block_pos[b] + t
                kp[b, :, t] = Kc[s][p]
                vp[b, :, t] = Vc[s][p]
    tq = layout.total_q
    q = np.zeros((tq, Hq, d))
    kc = np.zeros((tq, Hkv, d))
    vc = np.zeros((tq, Hkv, d))
    for s in range(layout.num_seqs):
        for r in range(layout.cu_q[s], layout.cu_q[s + 1]):
            p = layout.q_pos[r]
            q[r] = Qc[s][p]
            kc[r] = Kc[s][p]
            vc[r] = Vc[s][p]
    return q, kc, vc, kp, vp


def sdpa_rows(Qc, Kc, Vc, rows_pos, scale):
    """Full causal attention over the contiguous sequence via torch (fp64), at rows."""
    L, Hq, d = Qc.shape
    Hkv = Kc.shape[1]
    G = Hq // Hkv
    q = torch.tensor(Qc, dtype=torch.float64).permute(1, 0, 2)[None]
    k = torch.tensor(Kc, dtype=torch.float64).permute(1, 0, 2)[None].repeat_interleave(G, 1)
    v = torch.tensor(Vc, dtype=torch.float64).permute(1, 0, 2)[None].repeat_interleave(G, 1)
    o = torch.nn.functional.scaled_dot_product_attention(q, k, v, is_causal=True, scale=scale)
    s = (q @ k.transpose(-1, -2)) * scale
    mask = torch.ones(L, L, dtype=torch.bool).tril()
    s = s.masked_fill(~mask, float("-inf"))
    lse = torch.logsumexp(s, dim=-1)
    o = o[0].permute(1, 0, 2).numpy()
    lse = lse[0].permute(1, 0).numpy()
    return o[rows_pos], lse[rows_pos]


def random_contiguous(rng, L, Hq, Hkv, d):
    return (rng.standard_normal((L, Hq, d)), rng.standard_normal((L, Hkv, d)),
            rng.standard_normal((L, Hkv, d)))


def seq_len(spec):
    m = max([p0 + n for (p0, n) in spec.pool_runs] + [int(p) + 1 for p in spec.chunk_pos])
    return m


# ----------------------------------------------------------------------------- attention pins

@pytest.mark.parametrize("seed,Hq,Hkv,d,frac", [(1, 4, 2, 16, 0.5), (2, 2, 2, 8, 0.2),
                                                (3, 8, 2, 16, 0.8), (4, 3, 1, 4, 0.6)])
def test_prefill_equals_contiguous_causal_attention(seed, Hq, Hkv, d, frac):
    """Lossless claim (abstract): MSA over scattered segments equals ordinary causal
    attention over the contiguous sequence, at the chunk tokens' positions."""
    rng = np.random.default_rng(seed)
    specs = [W.random_prefill_spec(rng, old_blocks=int(rng.integers(3, 9)), cached_frac=frac,
                                   suffix=int(rng.integers(1, 40)),
                                   chunk=int(rng.integers(20, 90))) for _ in range(3)]
    lay = W.custom_prefill(Hq, Hkv, d, specs, seed=seed, shuffle_segments=True)
    Ls = [seq_len(s) for s in specs]
    contig = [random_contiguous(rng, L, Hq, Hkv, d) for L in Ls]
    q, kc, vc, kp, vp = scatter_from_contiguous(lay, [c[1] for c in contig], [c[2] for c in contig],
                                                [c[0] for c in contig])
    scale = 1.0 / math.sqrt(d)
    rows, out, lse = O.prefill(lay, q, kc, vc, kp, vp, scale)
    for s in range(lay.num_seqs):
        r0, r1 = lay.cu_q[s], lay.cu_q[s + 1]
        ref_o, ref_l = sdpa_rows(contig[s][0], contig[s][1], contig[s][2], lay.q_pos[r0:r1], scale)
        np.testing.assert_allclose(out[r0:r1], ref_o, rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(lse[r0:r1], ref_l, rtol=1e-12, atol=1e-12)


def test_prefill_fp32_mode_close_to_fp64():
    rng = np.random.default_rng(7)
    spec = W.random_prefill_spec(rng, 6, 0.5, 20, 60)
    lay = W.custom_prefill(4, 2, 16, [spec], seed=7)
    L = seq_len(spec)
    Qc, Kc, Vc = random_contiguous(rng, L, 4, 2, 16)
    args = scatter_from_contiguous(lay, [Kc], [Vc], [Qc])
    _, o64, l64 = O.prefill(lay, *args, 0.25)
    _, o32, l32 = O.prefill(lay, *args, 0.25, dtype=np.float32)
    np.testing.assert_allclose(o32, o64, rtol=1e-4, atol=1e-5)
    np.testing.assert_allclose(l32, l64, rtol=1e-5, atol=1e-5)


def test_nothing_cached_is_plain_causal_prefill():
    rng = np.random.default_rng(11)
    L = 70
    spec = W.SeqSpec([], np.arange(L))
    lay = W.custom_prefill(2, 1, 8, [spec], seed=11)
    Qc, Kc, Vc = random_contiguous(rng, L, 2, 1, 8)
    args = scatter_from_contiguous(lay, [Kc], [Vc], [Qc])
    _, out, lse = O.prefill(lay, *args, 0.3)
    ref_o, ref_l = sdpa_rows(Qc, Kc, Vc, np.arange(L), 0.3)
    np.testing.assert_allclose(out, ref_o, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(lse, ref_l, rtol=1e-12, atol=1e-12)


def test_prefix_cache_is_chunked_prefill():
    """Prefix caching (section 4.1's baseline) is the special case cached set = prefix."""
    rng = np.random.default_rng(12)
    spec = W.SeqSpec([(0, 48)], np.arange(48, 90))
    lay = W.custom_prefill(4, 4, 8, [spec], seed=12)
    Qc, Kc, Vc = random_contiguous(rng, 90, 4, 4, 8)
    args = scatter_from_contiguous(lay, [Kc], [Vc], [Qc])
    _, out, lse = O.prefill(lay, *args, 0.5)
    ref_o, ref_l = sdpa_rows(Qc, Kc, Vc, np.arange(48, 90), 0.5)
    np.testing.assert_allclose(out, ref_o, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(lse, ref_l, rtol=1e-12, atol=1e-12)


def test_decode_is_last_row_of_full_attention():
    rng = np.random.default_rng(13)
    specs = [W.SeqSpec([(0, 32), (48, 20), (32, 16)], np.zeros(0)),
             W.SeqSpec([(0, 16), (16, 9)], np.zeros(0))]
    lay = W.custom_decode(4, 2, 8, specs, seed=13, shuffle_segments=True)
    Ls = [68, 25]
    contig = [random_contiguous(rng, L, 4, 2, 8) for L in Ls]
    _, _, _, kp, vp = scatter_from_contiguous(lay, [c[1] for c in contig], [c[2] for c in contig],
                                              [c[0] for c in contig])
    q = np.stack([contig[s][0][Ls[s] - 1] for s in range(2)])
    _, out, lse = O.decode(lay, q, kp, vp, 0.35)
    for s in range(2):
        ref_o, ref_l = sdpa_rows(contig[s][0], contig[s][1], contig[s][2], [Ls[s] - 1], 0.35)
        np.testing.assert_allclose(out[s], ref_o[0], rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(lse[s], ref_l[0], rtol=1e-12, atol=1e-12)


def test_single_visible_key():
    rng = np.random.default_rng(5)
    q = rng.standard_normal((1, 2, 8))
    k = rng.standard_normal((3, 1, 8))
    v = rng.standard_normal((3, 1, 8))
    out, lse = O.attention(q, np.array([10]), k, v, np.array([10, 11, 12]), 0.7)
    for h in range(2):
        np.testing.assert_array_equal(out[0, h], v[0, 0])
        assert lse[0, h] == pytest.approx(0.7 * float(q[0, h] @ k[0, 0]), rel=1e-14)


def test_zero_query_gives_mean_and_log_count():
    """Q = 0: every visible logit is 0, so O = mean of visible V and LSE = ln(count)."""
    rng = np.random.default_rng(6)
    n, m = 5, 32
    q = np.zeros((n, 2, 4))
    k = rng.standard_normal((m, 1, 4))
    v = rng.standard_normal((m, 1, 4))
    kpos = rng.permutation(m)
    qpos = np.array([0, 3, 7, 15, 31])
    out, lse = O.attention(q, qpos, k, v, kpos, 1.0)
    for i, p in enumerate(qpos):
        vis = kpos <= p
        np.testing.assert_allclose(out[i, 0], v[vis, 0].mean(axis=0), rtol=1e-13, atol=1e-13)
        assert lse[i, 1] == pytest.approx(math.log(vis.sum()), abs=1e-14)


def test_equal_keys_give_mean():
    rng = np.random.default_rng(8)
    q = rng.standard_normal((3, 1, 4))
    k = np.tile(rng.standard_normal((1, 1, 4)), (16, 1, 1))
    v = rng.standard_normal((16, 1, 4))
    kpos = np.arange(16)
    out, lse = O.attention(q, np.array([3, 7, 15]), k, v, kpos, 0.5)
    for i, p in enumerate([3, 7, 15]):
        np.testing.assert_allclose(out[i, 0], v[:p + 1, 0].mean(axis=0), rtol=1e-12)
        x = 0.5 * float(q[i, 0] @ k[0, 0])
        assert lse[i, 0] == pytest.approx(x + math.log(p + 1), rel=1e-13)


def test_no_visible_key_gives_zero_and_neg_inf():
    q = np.ones((1, 1, 4))
    k = np.ones((2, 1, 4))
    v = np.ones((2, 1, 4))
    out, lse = O.attention(q, np.array([0]), k, v, np.array([5, 6]), 1.0)
    assert np.all(out == 0) and np.isneginf(lse[0, 0])


def test_worked_example():
    ex = json.load(open(os.path.join(GOLDEN, "worked_example_attention.json")))
    keys = ex["keys"]
    k = np.array([kk["k"] for kk in keys], float)[:, None, :]
    v = np.array([kk["v"] for kk in keys], float)[:, None, :]
    kpos = np.array([kk["pos"] for kk in keys])
    q = np.array([qq["q"] for qq in ex["queries"]], float)[:, None, :]
    qpos = np.array([qq["pos"] for qq in ex["queries"]])
    out, lse = O.attention(q, qpos, k, v, kpos, ex["scale"])
    env = {"e": math.e, "ln": math.log, "__builtins__": {}}
    for i, qq in enumerate(ex["queries"]):
        exp_o = [eval(s, env) for s in qq["out"]]
        exp_l = eval(qq["lse"], env)
        np.testing.assert_allclose(out[i, 0], exp_o, rtol=1e-14)
        assert lse[i, 0] == pytest.approx(exp_l, rel=1e-14)


# ----------------------------------------------------------------------------- merge invariant

@pytest.mark.parametrize("seed", [0, 1, 2])
def test_merge_of_disjoint_key_sets_equals_whole(seed):
    rng = np.random.default_rng(seed)
    n, m, Hq, Hkv, d = 6, 40, 4, 2, 8
    q = rng.standard_normal((n, Hq, d)) * 2
    k = rng.standard_normal((m, Hkv, d))
    v = rng.standard_normal((m, Hkv, d))
    kpos = rng.permutation(m)
    qpos = np.sort(rng.choice(m, n, replace=False))
    whole_o, whole_l = O.attention(q, qpos, k, v, kpos, 0.9)
    parts = rng.integers(0, 5, size=m)          # 5 subsets, some possibly empty
    o_parts, l_parts = [], []
    for r in range(6):                           # subset 5 is always empty
        sel = parts == r
        o, l = O.attention(q, qpos, k[sel], v[sel], kpos[sel], 0.9)
        o_parts.append(o)
        l_parts.append(l)
    mo, ml = O.merge_lse(o_parts, l_parts)
    np.testing.assert_allclose(mo, whole_o, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(ml, whole_l, rtol=1e-12, atol=1e-13)


def _layout_with_segments(lay, segs):
    return W.Layout(**{**vars(lay), "segments": np.asarray(segs, np.int32).reshape(-1, 3)})


@pytest.mark.parametrize("seed", [3, 4])
def test_per_segment_parts_merge_to_msa(seed):
    """The queries-only variant (KV = pool segments alone), one launch per segment plus one
    over the chunk's own keys, merged by log-sum-exp, equals MSA over the whole context:
    the one-launch result the method replaces many launches with (ablation baseline)."""
    rng = np.random.default_rng(seed)
    spec = W.random_prefill_spec(rng, 24, 0.5, 40, 150)
    lay = W.custom_prefill(4, 2, 16, [spec], seed=seed, qk_std=0.7)
    wl = W.make_values(lay)
    a = {k: getattr(wl, k).float().numpy().astype(np.float64) for k in ("q", "k_chunk", "v_chunk", "k_pool", "v_pool")}
    sc = 1.0 / 4.0
    _, whole_o, whole_l = O.prefill(lay, a["q"], a["k_chunk"], a["v_chunk"], a["k_pool"], a["v_pool"], sc)
    o_parts, l_parts = [], []
    for seg in lay.segments:
        _, o, l = O.prefill(_layout_with_segments(lay, [seg]), a["q"], a["k_chunk"], a["v_chunk"], a["k_pool"],
                            a["v_pool"], sc, chunk_keys=False)
        o_parts.append(o)
        l_parts.append(l)
    _, o, l = O.prefill(_layout_with_segments(lay, []), a["q"], a["k_chunk"], a["v_chunk"], a["k_pool"], a["v_pool"], sc)
    o_parts.append(o)
    l_parts.append(l)
    assert any(np.isneginf(x).any() for x in l_parts[:-1])   # some query sees nothing of some segment
    mo, ml = O.merge_lse(o_parts, l_parts)
    np.testing.assert_allclose(mo, whole_o, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(ml, whole_l, rtol=1e-12, atol=1e-13)


def test_merge_edge_cases():
    o1 = np.ones((2, 4))
    o2 = 3 * np.ones((2, 4))
    l1 = np.array([-np.inf, 0.0])
    l2 = np.array([-np.inf, -np.inf])
    o, l = O.merge_lse([o1, o2], [l1, l2])
    assert np.all(o[0] == 0) and np.isneginf(l[0])
    np.testing.assert_array_equal(o[1], o1[1])
    assert l[1] == 0.0
    # equal lse: plain average, lse + ln 2
    o, l = O.merge_lse([o1, o2], [np.zeros(2), np.zeros(2)])
    np.testing.assert_allclose(o, 2 * np.ones((2, 4)))
    np.testing.assert_allclose(l, math.log(2) * np.ones(2))


# ----------------------------------------------------------------------------- tiler

@pytest.mark.parametrize("R,lo,hi,expect", [
    (4096, 512, 4096, [4096]), (4097, 512, 4096, [2176, 1921]), (300, 512, 4096, [300]),
    (8192, 512, 4096, [4096, 4096]), (5000, 512, 4096, [2560, 2440]), (512, 512, 4096, [512]),
    (129, 1, 128, [128, 1]), (1000, 100, 256, [256, 256, 256, 232]), (0, 512, 4096, [])])
def test_chunk_tiler_rule(R, lo, hi, expect):
    assert O.chunk_sizes(R, lo, hi) == expect


def test_chunk_tiler_properties():
    rng = np.random.default_rng(0)
    for _ in range(2000):
        hi = 128 * int(rng.integers(1, 40))
        lo = int(rng.integers(1, hi + 1))
        R = int(rng.integers(1, 20 * hi))
        c = O.chunk_sizes(R, lo, hi)
        assert sum(c) == R and all(x > 0 for x in c)
        if R >= lo:
            assert len(c) == -(-R // hi)              # fewest chunks the maximum allows
            assert all(x <= hi for x in c)
            assert all(x == c[0] for x in c[:-1]) and c[-1] <= c[0]
            if len(c) > 1:
                assert c[0] % 128 == 0


# ----------------------------------------------------------------------------- canonical plan

def hand_layout():
    """A layout small enough to plan by hand: 1 sequence, 12 pool blocks in 4 segments
    given out of order, 20 chunk tokens in two runs, one cached block beyond the chunk."""
    nbk = 18
    block_pos = np.zeros(nbk, np.int32)
    block_fill = np.zeros(nbk, np.int32)
    row = [13, 10, 17, 11, 16, 12, 15, 14, 3, 1, 7, 0]
    pos = [0, 16, 32, 48, 64, 80, 96, 112, 128, 144, 176, 192]
    fill = [16] * 10 + [5, 16]
    for b, p, f in zip(row, pos, fill):
        block_pos[b] = p
        block_fill[b] = f
    q_pos = np.array(list(range(160, 176)) + list(range(181, 185)), np.int32)
    return W.Layout(mode="prefill", num_heads_q=2, num_heads_kv=1, head_dim=64, num_seqs=1,
                    num_pool_blocks=nbk, block_pos=block_pos, block_fill=block_fill,
                    block_table=np.array([row], np.int32),
                    segments=np.array([(0, 10, 1), (0, 0, 8), (0, 11, 1), (0, 8, 2)], np.int32),
                    cu_q=np.array([0, 20], np.int32), q_pos=q_pos, qk_std=1.0, v_std=1.0)


def hand_expected():
    toks = []
    row = [13, 10, 17, 11, 16, 12, 15, 14, 3, 1]
    for i, b in enumerate(row):
        toks += [(0, b, t, 16 * i + t) for t in range(16)]
    toks += [(1, r, 0, 160 + r) for r in range(16)]
    toks += [(0, 7, t, 176 + t) for t in range(5)]
    toks += [(1, 16 + r, 0, 181 + r) for r in range(4)]
    toks += [(0, 0, t, 192 + t) for t in range(16)]
    # units: 8 pool blocks (0-127) | block 3, block 1, chunk rows 0-15, block 7 (5 tokens),
    # chunk rows 16-19, block 0: one tile of 8 pool units, then one mixed tile of 6 units
    kts = [(0, O.POOL, 0, 128, 0, 127), (0, O.MIXED, 128, 16 + 16 + 16 + 5 + 4 + 16, 128, 207)]
    qts = [(0, 0, 20, 160, 184)]
    cls = [O.FULL, O.PARTIAL]
    head = [0, 1, len(toks), len(kts), len(qts), len(cls)]
    return np.array(head + [x for t in toks for x in t] + [x for t in kts for x in t]
                    + [x for t in qts for x in t] + cls, np.int32)


def test_canonical_plan_hand_example():
    np.testing.assert_array_equal(O.canonical_plan(hand_layout()), hand_expected())


def parse_plan(arr):
    mode, ns, nt, nk, nq, nc = arr[:6]
    o = 6
    toks = arr[o:o + 4 * nt].reshape(-1, 4); o += 4 * nt
    kts = arr[o:o + 6 * nk].reshape(-1, 6); o += 6 * nk
    qts = arr[o:o + 5 * nq].reshape(-1, 5); o += 5 * nq
    cls = arr[o:o + nc]; o += nc
    assert o == len(arr)
    return toks, kts, qts, cls


@pytest.mark.parametrize("idx", [1, 2])
def test_canonical_plan_invariants(idx):
    """Every KV token appears once in ascending position; tiles partition the list;
    each class agrees with brute-force visibility of its (query, key) pairs."""
    lay = W.make_layout(idx)
    toks, kts, qts, cls = parse_plan(O.canonical_plan(lay))
    npool = int(sum(lay.block_fill[lay.block_table[s, f + i]]
                    for (s, f, nb) in lay.segments for i in range(nb)))
    assert len(toks) == npool + lay.total_q
    assert np.all(np.diff(toks[:, 3]) > 0)
    for (src, idn, off, pos) in toks:
        if src == O.POOL:
            assert lay.block_pos[idn] + off == pos and off < lay.block_fill[idn]
        else:
            assert lay.q_pos[idn] == pos and off == 0
    assert kts[0, 2] == 0 and np.all(kts[1:, 2] == kts[:-1, 2] + kts[:-1, 3])
    assert kts[-1, 2] + kts[-1, 3] == len(toks)
    ci = 0
    for (s, r0, nr, qmin, qmax) in qts:
        qp = lay.q_pos[r0:r0 + nr]
        for (ks, src, tb, nt, kmin, kmax) in kts:
            kp = toks[tb:tb + nt, 3]
            if src == O.MIXED:
                assert set(toks[tb:tb + nt, 0].tolist()) == {O.POOL, O.CHUNK}
            else:
                assert np.all(toks[tb:tb + nt, 0] == src)
            assert kmin == kp[0] and kmax == kp[-1]
            vis = kp[None, :] <= qp[:, None]
            c = cls[ci]; ci += 1
            if not vis.any():
                assert c == O.SKIP
            elif vis.all() and nt == 128:
                assert c == O.FULL
            else:
                assert c == O.PARTIAL
    assert ci == len(cls)


def test_useful_flops_brute_force():
    lay = hand_layout()
    kp = O.canonical_tokens(lay, 0)[:, 3]
    pairs = sum(int((kp <= p).sum()) for p in lay.q_pos)
    assert O.useful_flops(lay) == pairs * 2 * 4 * 64


# ----------------------------------------------------------------------------- mutation check

def test_pins_catch_a_planted_mistake(monkeypatch):
    """Plant a plausible mistake in the oracle (mask off by one) and check a pin fails."""
    real = O.attention

    def wrong(q, q_pos, k, v, k_pos, scale, dtype=np.float64, causal=True):
        return real(q, np.asarray(q_pos) - 1, k, v, k_pos, scale, dtype, causal)

    monkeypatch.setattr(O, "attention", wrong)
    with pytest.raises(AssertionError):
        test_prefill_equals_contiguous_causal_attention(1, 4, 2, 16, 0.5)


# ----------------------------------------------------------------------------- write-back (oracle)

def test_append_plan_hand_example():
    """Placement worked by hand from the written rule (row at position p -> block holding
    position block p // 16, offset p % 16; a block met at offset 0 takes the next free
    block, one met part-way continues the sequence's block that holds it)."""
    bp = np.zeros(8, np.int64)
    bf = np.zeros(8, np.int64)
    bp[1], bf[1] = 0, 3                     # the sequence's block 1 holds positions 0, 1, 2
    dst, new, bp2, bf2 = O.append_plan([3, 4, 16, 17, 32], [7, 2, 5], bp, bf, seq_blocks=[1])
    assert dst.tolist() == [1 * 16 + 3, 1 * 16 + 4, 7 * 16 + 0, 7 * 16 + 1, 2 * 16 + 0]
    assert new.tolist() == [7, 2]
    assert (bp2[1], bf2[1]) == (0, 5)
    assert (bp2[7], bf2[7]) == (16, 2)
    assert (bp2[2], bf2[2]) == (32, 1)
    assert bf2[5] == 0 and bf[1] == 3       # block 5 untouched; the inputs are not modified


@pytest.mark.parametrize("q_pos,free,seq_blocks,why", [
    ([0, 2], [0], [], "hole inside a block"),
    ([5], [0], [], "part-way with no block to continue"),
    ([0, 16, 32], [0, 1], [], "too few free blocks"),
    ([4, 3], [0], [], "unsorted"),
])
def test_append_plan_rejects(q_pos, free, seq_blocks, why):
    with pytest.raises(ValueError):
        O.append_plan(q_pos, free, np.zeros(4, np.int64), np.zeros(4, np.int64), seq_blocks=seq_blocks)


@pytest.mark.parametrize("seed", range(5))
def test_append_plan_places_every_row_at_its_position(seed):
    """On random chunks (a new turn that continues a partial block, then gaps): every row
    lands in a block whose positions cover it, inside the block's fill, and no two rows
    share a slot."""
    rng = np.random.default_rng(seed)
    nblk = 64
    start = int(rng.integers(0, 200))
    pos = np.sort(rng.choice(np.arange(start, start + 400), int(rng.integers(1, 300)), replace=False))
    # make each position block's rows contiguous from the block's first row (no holes)
    keep = []
    for pb in np.unique(pos // 16):
        rows = pos[pos // 16 == pb]
        first = rows[0] if pb == pos[0] // 16 else pb * 16
        keep.extend(range(int(first), int(first) + len(rows)))
    pos = np.array(keep)
    bp = np.zeros(nblk, np.int64)
    bf = np.zeros(nblk, np.int64)
    seq_blocks = []
    if pos[0] % 16:
        bp[9], bf[9] = pos[0] // 16 * 16, pos[0] % 16
        seq_blocks = [9]
    free = [b for b in rng.permutation(nblk).tolist() if b != 9]
    dst, new, bp2, bf2 = O.append_plan(pos, free, bp, bf, seq_blocks=seq_blocks)
    assert len(set(dst.tolist())) == len(dst)
    for p, slot in zip(pos, dst):
        b, t = divmod(int(slot), 16)
        assert bp2[b] + t == p and t < bf2[b]


def test_append_copies_rows_to_their_slots():
    k_chunk = np.arange(3 * 2 * 4, dtype=np.float64).reshape(3, 2, 4)
    v_chunk = -k_chunk
    k_pool = np.full((3, 2, 16, 4), 7.0)
    v_pool = np.full((3, 2, 16, 4), 7.0)
    kp, vp = O.append(k_chunk, v_chunk, k_pool, v_pool, [2 * 16 + 5, -1, 0 * 16 + 15])
    assert np.array_equal(kp[2, :, 5, :], k_chunk[0]) and np.array_equal(vp[2, :, 5, :], v_chunk[0])
    assert np.array_equal(kp[0, :, 15, :], k_chunk[2]) and np.array_equal(vp[0, :, 15, :], v_chunk[2])
    changed = np.zeros((3, 16), bool)
    changed[2, 5] = changed[0, 15] = True
    assert np.all(kp.transpose(0, 2, 1, 3)[~changed] == 7.0)      # row 1 (slot -1) and the rest untouched
    assert np.all(vp.transpose(0, 2, 1, 3)[~changed] == 7.0)
    assert np.all(k_pool == 7.0)                                   # the inputs are not modified
