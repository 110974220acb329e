"""Host-side checks of libmsa.so (no GPU needed): every symbol declared in
include/msa.h is exported, the planner's canonical plan equals the oracle's bit for
bit, the chunk tiler equals the oracle's rule, decode splits partition the context,
useful-FLOP counts agree, and malformed layouts return the documented error codes."""
import os
import re
import subprocess

import numpy as np
import pytest

import segmented_kv_attention_msa_b300 as msa
from segmented_kv_attention_msa_b300 import build as B
from segmented_kv_attention_msa_b300 import workload as W
from oracle import msa_oracle as O
from tests.helpers import empty_sequence_specs, export_tables

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def built():
    B.build()
    return msa.lib()


def header_symbols():
    src = open(os.path.join(ROOT, "include", "msa.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(msa_[a-z_0-9]+)\s*\(", src)))


def test_header_symbols_exported():
    syms = header_symbols()
    assert len(syms) >= 18
    out = subprocess.run(["nm", "-D", "--defined-only", B.LIB], capture_output=True, text=True).stdout
    exported = set(re.findall(r"\bT (msa_\w+)", out))
    missing = [s for s in syms if s not in exported]
    assert not missing, missing
    # and the binding declares them all
    assert set(syms) <= set(msa.EXPORTS)


def test_version():
    assert msa.lib().msa_version() == 1


@pytest.mark.parametrize("idx", [1, 2, 5])
def test_plan_export_bit_exact(idx):
    lay = W.make_layout(idx)
    plan = msa.Plan.from_layout(lay)
    np.testing.assert_array_equal(plan.export(), O.canonical_plan(lay))


def test_plan_export_multiturn():
    lay = W.make_layout(3, tiler=O.chunk_sizes)
    lay2 = W.make_layout(3, tiler=msa.chunk_sizes)
    np.testing.assert_array_equal(lay.q_pos, lay2.q_pos)
    np.testing.assert_array_equal(lay.block_table, lay2.block_table)
    plan = msa.Plan.from_layout(lay)
    np.testing.assert_array_equal(plan.export(), O.canonical_plan(lay))


def test_plan_hand_example():
    from tests.test_oracle_pins import hand_expected, hand_layout
    plan = msa.Plan.from_layout(hand_layout())
    np.testing.assert_array_equal(plan.export(), hand_expected())


@pytest.mark.parametrize("seed", range(6))
def test_plan_random_layouts(seed):
    rng = np.random.default_rng(100 + seed)
    specs = [W.random_prefill_spec(rng, int(rng.integers(1, 40)), float(rng.random()),
                                   int(rng.integers(1, 300)), int(rng.integers(1, 700)))
             for _ in range(int(rng.integers(1, 5)))]
    lay = W.custom_prefill(8, 2, 64, specs, seed=seed, shuffle_segments=True)
    plan = msa.Plan.from_layout(lay)
    np.testing.assert_array_equal(plan.export(), O.canonical_plan(lay))
    assert plan.stats()["useful_flops"] == O.useful_flops(lay)


def sparse_spec(rng, nblocks):
    """A sequence whose pool runs start on block boundaries and may end in a partial block,
    and whose chunk holds random positions that no run holds (gaps anywhere), so chunk
    units of consecutive rows have non-consecutive positions and tiles mix sources."""
    runs, b = [], 0
    taken = np.zeros(nblocks * 16, bool)
    while b < nblocks:
        if rng.random() < 0.5:
            nb = min(int(rng.integers(1, 6)), nblocks - b)
            ntok = nb * 16 - int(rng.integers(0, 16)) if rng.random() < 0.4 else nb * 16
            runs.append((b * 16, ntok))
            taken[b * 16:b * 16 + ntok] = True
            b += nb
        else:
            b += int(rng.integers(1, 4))
    free = np.nonzero(~taken)[0]
    k = int(rng.integers(1, max(2, len(free))))
    return W.SeqSpec(runs, np.sort(rng.choice(free, size=min(k, len(free)), replace=False)))


@pytest.mark.parametrize("seed", range(8))
def test_plan_random_sparse_layouts(seed):
    rng = np.random.default_rng(5000 + seed)
    specs = [sparse_spec(rng, int(rng.integers(1, 30))) for _ in range(int(rng.integers(1, 5)))]
    lay = W.custom_prefill(8, 2, 64, specs, seed=seed, shuffle_segments=True)
    plan = msa.Plan.from_layout(lay)
    np.testing.assert_array_equal(plan.export(), O.canonical_plan(lay))
    assert plan.stats()["useful_flops"] == O.useful_flops(lay)


def test_decode_plan_tokens_and_splits():
    lay = W.make_layout(4)
    plan = msa.Plan.from_layout(lay)
    np.testing.assert_array_equal(plan.export(), O.canonical_plan(lay))
    sp = plan.export_splits()
    # splits partition each sequence's canonical block list, in order, none empty
    for s in range(lay.num_seqs):
        mine = sp[sp[:, 0] == s]
        nblk = sum(int(nb) for (q, f, nb) in lay.segments if q == s)
        assert mine[0, 1] == 0 and np.all(mine[:, 2] > 0)
        assert np.all(mine[1:, 1] == mine[:-1, 1] + mine[:-1, 2])
        assert mine[-1, 1] + mine[-1, 2] == nblk
    st = plan.stats()
    assert st["useful_flops"] == O.useful_flops(lay)
    assert st["num_work_items"] >= 2 * 148


def test_chunk_tiler_matches_oracle():
    rng = np.random.default_rng(1)
    for _ in range(3000):
        hi = 128 * int(rng.integers(1, 40))
        lo = int(rng.integers(0, hi + 1))
        R = int(rng.integers(0, 20 * hi))
        assert msa.chunk_sizes(R, lo, hi) == O.chunk_sizes(R, lo, hi)


def test_chunk_tiler_rejects_bad_max():
    with pytest.raises(msa.MSAError):
        msa.chunk_sizes(1000, 10, 100)


# ----------------------------------------------------------------------------- validation

def base_layout():
    from tests.test_oracle_pins import hand_layout
    return hand_layout()


def make(lay, **kw):
    args = dict(mode=lay.mode, num_heads_q=lay.num_heads_q, num_heads_kv=lay.num_heads_kv,
                head_dim=lay.head_dim, segments=lay.segments, block_table=lay.block_table,
                block_pos=lay.block_pos, block_fill=lay.block_fill, cu_q=lay.cu_q, q_pos=lay.q_pos)
    args.update(kw)
    return msa.Plan(**args)


def expect(code, **kw):
    with pytest.raises(msa.MSAError) as e:
        make(base_layout(), **kw)
    assert e.value.code == code


def test_validation_ok():
    make(base_layout())


def test_unsupported_head_dim():
    expect(-2, head_dim=96)


def test_unsupported_gqa():
    expect(-2, num_heads_q=3, num_heads_kv=2)


def test_plan_with_empty_sequences_matches_oracle():
    lay = W.custom_prefill(4, 2, 64, empty_sequence_specs(), seed=3)
    pl = msa.Plan.from_layout(lay)
    assert np.array_equal(pl.export(), O.canonical_plan(lay))
    sch = pl.export_schedule().reshape(-1, 9)
    ex = pl.export()
    n_tok, n_kt, n_qt = ex[2], ex[3], ex[4]
    qts = ex[6 + 4 * n_tok + 6 * n_kt:][:5 * n_qt].reshape(-1, 5)
    assert set(qts[:, 0].tolist()) == {0, 2}            # query tiles only where rows exist
    assert set(sch[:, 1].tolist()) == set(range(n_qt))   # and every one is scheduled


def test_plan_without_query_rows():
    lay = W.custom_prefill(4, 2, 64, [W.SeqSpec([(0, 48)], np.array([], np.int64))], seed=3)
    pl = msa.Plan.from_layout(lay)
    st = pl.stats()
    assert st["useful_flops"] == 0 and st["num_work_items"] == 0 and st["num_prefill_ctas"] == 0
    assert np.array_equal(pl.export(), O.canonical_plan(lay))
    assert pl.export_schedule().size == 0


def test_pool_rows_beyond_int32():
    """The pool seen as [blocks * Hkv * 16] rows must fit 32-bit TMA coordinates: one block
    more than that limit is refused, the limit itself is accepted."""
    lay = base_layout()
    hkv = 8  # planning does not look at K/V values; more heads keep the arrays small
    limit = (2 ** 31 - 1) // (hkv * 16)
    nb = len(lay.block_pos)
    for n, ok in ((limit, True), (limit + 1, False)):
        bp = np.zeros(n, np.int32)
        bf = np.zeros(n, np.int32)
        bp[:nb], bf[:nb] = lay.block_pos, lay.block_fill
        kw = dict(block_pos=bp, block_fill=bf, num_heads_q=hkv, num_heads_kv=hkv)
        if ok:
            make(lay, **kw)
        else:
            with pytest.raises(msa.MSAError) as e:
                make(lay, **kw)
            assert e.value.code == -2


def test_block_out_of_range():
    lay = base_layout()
    bt = lay.block_table.copy()
    bt[0, 3] = 99
    expect(-4, block_table=bt)


def test_logical_block_out_of_row():
    lay = base_layout()
    seg = lay.segments.copy()
    seg[0, 2] = 5
    expect(-4, segments=seg)


def test_position_overlap_pool_vs_chunk():
    lay = base_layout()
    qp = lay.q_pos.copy()
    qp[0] = 150         # inside the cached block at 144..159
    qp = np.sort(qp)
    expect(-3, q_pos=qp)


def test_position_overlap_two_blocks():
    lay = base_layout()
    bp = lay.block_pos.copy()
    bp[0] = 176         # block 0 now starts where block 7 does
    expect(-3, block_pos=bp)


def test_unsorted_q_pos():
    lay = base_layout()
    qp = lay.q_pos.copy()
    qp[[2, 3]] = qp[[3, 2]]
    expect(-1, q_pos=qp)


def test_inconsistent_run():
    lay = base_layout()
    bp = lay.block_pos.copy()
    bp[10] = 320        # second block of the first segment no longer follows the first
    expect(-1, block_pos=bp)


def test_partial_block_inside_run():
    lay = base_layout()
    bf = lay.block_fill.copy()
    bf[13] = 8          # first block of an 8-block run may not be partial
    expect(-1, block_fill=bf)


def test_decode_needs_one_query_per_sequence():
    lay = W.custom_decode(4, 2, 64, [W.SeqSpec([(0, 40)], np.zeros(0))], seed=0)
    with pytest.raises(msa.MSAError) as e:
        msa.Plan("decode", 4, 2, 64, lay.segments, lay.block_table, lay.block_pos, lay.block_fill,
                 np.array([0, 2], np.int32))
    assert e.value.code == -1


def _list_counts(plan):
    """Non-skipped KV tiles of every query tile, from the canonical export."""
    c = plan.export()
    _, _, ntok, nkt, nqt, ncls = c[:6]
    off = 6 + 4 * ntok
    kts = c[off:off + 6 * nkt].reshape(-1, 6)
    off += 6 * nkt
    qts = c[off:off + 5 * nqt].reshape(-1, 5)
    off += 5 * nqt
    cls = c[off:off + ncls]
    out, ci = [], 0
    for q in qts:
        n = int((kts[:, 0] == q[0]).sum())
        out.append(int((cls[ci:ci + n] != 0).sum()))
        ci += n
    return out


@pytest.mark.parametrize("idx,ctas", [(1, 0), (2, 0), (2, 1), (2, 7), (2, 500), (3, 0), (5, 0)])
def test_prefill_schedule_covers_every_item_once(idx, ctas):
    lay = W.make_layout(idx, tiler=msa.chunk_sizes)
    plan = msa.Plan.from_layout(lay, prefill_ctas=ctas)
    sc = plan.export_schedule()
    st = plan.stats()
    counts = _list_counts(plan)
    G = lay.num_heads_q // lay.num_heads_kv
    hpc = 2 if G % 2 == 0 else 1
    n_ctas = st["num_prefill_ctas"]
    assert 1 <= n_ctas <= (ctas or 148)
    assert np.all(np.diff(sc[:, 0]) >= 0) and set(sc[:, 0]) == set(range(n_ctas))
    assert st["num_work_items"] == len(sc)
    pieces = {}
    for (c, qt, g, h0, j0, n, nparts, slot0, slot) in sc:
        assert n >= 1 and 0 <= g < lay.num_heads_kv and h0 % hpc == 0 and h0 // G == g
        pieces.setdefault((qt, g, h0), []).append((j0, n, nparts, slot0, slot))
    # every (query tile, KV head, head pair) exactly once, its list covered in slot order
    assert len(pieces) == len(counts) * lay.num_heads_kv * (G // hpc)
    slots = []
    for (qt, g, h0), ps in pieces.items():
        ps.sort()
        assert all(p[2] == len(ps) for p in ps)
        assert ps[0][0] == 0 and sum(p[1] for p in ps) == counts[qt]
        assert all(a[0] + a[1] == b[0] for a, b in zip(ps[:-1], ps[1:]))
        if len(ps) == 1:
            assert ps[0][3] == -1 and ps[0][4] == -1
        else:
            assert [p[4] for p in ps] == [ps[0][3] + k for k in range(len(ps))]
            slots += [p[4] for p in ps]
    assert len(set(slots)) == len(slots)
    assert st["num_split_items"] == sum(1 for ps in pieces.values() if len(ps) > 1)


def _modelled_cta_cost(lay, ctas=148):
    """Per-CTA cost under the planner's cost model (full tile 8, masked tile 11, piece 22,
    split piece 40 more), from the exported schedule and tile classes: a query tile's list
    holds its FULL tiles first."""
    plan = msa.Plan.from_layout(lay, prefill_ctas=ctas)
    sc = plan.export_schedule()
    _, kt, qt, cls = export_tables(plan.export())
    per_seq = np.bincount(kt[:, 0], minlength=lay.num_seqs)
    nfull, off = [], 0
    for q in qt:
        nk = int(per_seq[q[0]])
        nfull.append(int((cls[off:off + nk] == O.FULL).sum()))
        off += nk
    cost = np.zeros(ctas)
    for c, q, g, h0, j0, n, nparts, s0, slot in sc:
        full = max(0, min(nfull[q] - j0, n))
        cost[c] += 8 * full + 11 * (n - full) + 22 + (40 if nparts > 1 else 0)
    return cost


@pytest.mark.parametrize("idx", [2, 3, 5])
def test_prefill_schedule_balance(idx):
    """The prefill workloads balance to within a few percent of modelled cost over 148
    CTAs once items may be cut (the last CTA may hold less)."""
    cost = _modelled_cta_cost(W.make_layout(idx, tiler=msa.chunk_sizes))
    assert cost.max() <= 1.03 * np.median(cost)


# ----------------------------------------------------------------------------- write-back placement

def _random_append_case(rng, nb=64):
    """A sequence whose chunk holds recomputed blocks (whole) and a suffix that may start
    inside a partially written block; returns (q_pos, block_pos, block_fill, free, cont)."""
    pool = nb * 2
    block_pos = np.zeros(pool, np.int32)
    block_fill = np.zeros(pool, np.int32)
    evicted = np.sort(rng.choice(nb, size=int(rng.integers(1, nb // 2)), replace=False))
    pos = np.concatenate([np.arange(b * 16, b * 16 + 16) for b in evicted])
    # the old context ends part-way into a cached block that the suffix continues
    cont = -1
    start = nb * 16 + int(rng.integers(0, 16))
    if start % 16:
        cont = int(rng.integers(0, pool))
        block_pos[cont] = start // 16 * 16
        block_fill[cont] = start % 16
    suffix = np.arange(start, start + int(rng.integers(1, 80)))
    q_pos = np.concatenate([pos, suffix]).astype(np.int32)
    free = [b for b in rng.permutation(pool).tolist() if b != cont][:len(q_pos) // 16 + 3]
    others = [b for b in rng.permutation(pool).tolist() if b != cont and b not in free][:5]
    seq_blocks = others + ([cont] if cont >= 0 else [])
    return q_pos, block_pos, block_fill, free, seq_blocks


def test_append_plan_matches_oracle():
    rng = np.random.default_rng(11)
    for _ in range(200):
        q_pos, bp, bf, free, sb = _random_append_case(rng)
        bp_c, bf_c = bp.copy(), bf.copy()
        dst, new = msa.append_plan(q_pos, free, bp_c, bf_c, seq_blocks=sb)
        d2, n2, bp2, bf2 = O.append_plan(q_pos, free, bp, bf, seq_blocks=sb)
        np.testing.assert_array_equal(dst, d2)
        np.testing.assert_array_equal(new, n2)
        np.testing.assert_array_equal(bp_c, bp2)
        np.testing.assert_array_equal(bf_c, bf2)


def test_append_plan_preserves_positions():
    """Pinned independently of the placement rule: every row lands in a distinct slot whose
    block position plus offset is the row's own position, inside the block's fill."""
    rng = np.random.default_rng(12)
    for _ in range(100):
        q_pos, bp, bf, free, sb = _random_append_case(rng)
        dst, new = msa.append_plan(q_pos, free, bp, bf, seq_blocks=sb)
        assert len(set(dst.tolist())) == len(dst)
        blk, off = dst // 16, dst % 16
        np.testing.assert_array_equal(bp[blk] + off, q_pos)
        assert np.all(off < bf[blk])
        assert set(new.tolist()) <= set(free) and len(new) == len(set(blk.tolist()) - set(sb))


def test_append_plan_errors():
    bp = np.zeros(8, np.int32)
    bf = np.zeros(8, np.int32)
    with pytest.raises(msa.MSAError):                       # a hole inside a block
        msa.append_plan([0, 1, 3], [0, 1], bp.copy(), bf.copy())
    with pytest.raises(msa.MSAError):                       # unsorted positions
        msa.append_plan([5, 4], [0, 1], bp.copy(), bf.copy())
    with pytest.raises(msa.MSAError) as e:                  # not enough free blocks
        msa.append_plan(list(range(40)), [0, 1], bp.copy(), bf.copy())
    assert e.value.code == -5
    with pytest.raises(msa.MSAError):                       # mid-block start without its block
        msa.append_plan([20, 21], [0, 1], bp.copy(), bf.copy())
    b2 = bp.copy(); f2 = bf.copy(); b2[3] = 16; f2[3] = 3
    with pytest.raises(msa.MSAError):                       # continued block's fill disagrees
        msa.append_plan([20, 21], [0, 1], b2, f2, seq_blocks=[3])
    b4 = bp.copy(); f4 = bf.copy(); b4[3] = 16; f4[3] = 4
    dst, new = msa.append_plan([20, 21, 32], [6], b4, f4, seq_blocks=[1, 3])   # continues block 3
    assert dst.tolist() == [3 * 16 + 4, 3 * 16 + 5, 6 * 16] and new.tolist() == [6] and f4[3] == 6
    with pytest.raises(msa.MSAError) as e:                  # block id outside the pool
        msa.append_plan([0], [9], bp.copy(), bf.copy())
    assert e.value.code == -4
    # nothing was written by a failed call
    b3 = bp.copy(); f3 = bf.copy()
    with pytest.raises(msa.MSAError):
        msa.append_plan([0, 1, 16, 18], [2, 5], b3, f3)
    assert not b3.any() and not f3.any()


def test_prefill_schedule_kv_head_phases():
    """When the KV of all heads is larger than L2 holds (the 131k-token context: 541 MB),
    every CTA runs its pieces KV head by KV head, and each head's work is balanced over
    the CTAs on its own; when it fits (the 8192-token context: 37 MB) the schedule is one
    longest-first walk whose CTAs mix heads."""
    big = W.make_layout(5)
    sc = msa.Plan.from_layout(big).export_schedule()
    for c in np.unique(sc[:, 0]):
        g = sc[sc[:, 0] == c, 2]
        assert np.all(np.diff(g) >= 0)                       # head 0 first, then head 1, ...
    _, kt, qt, cls = export_tables(msa.Plan.from_layout(big).export())
    per_head = np.zeros((148, big.num_heads_kv))
    for c, q, g, h0, j0, n, nparts, s0, slot in sc:
        per_head[c, g] += n
    for g in range(big.num_heads_kv):
        col = per_head[:, g]
        assert col.max() <= 1.06 * np.median(col)            # each head balanced on its own
    small = W.make_layout(2)
    sc2 = msa.Plan.from_layout(small).export_schedule()
    assert any(np.any(np.diff(sc2[sc2[:, 0] == c, 2]) < 0) for c in np.unique(sc2[:, 0]))
