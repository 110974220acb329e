"""The KV-block eviction policy (host C++ in libmsa.so) against its oracle and its pins.

Pins of the oracle itself: Eq. 10 in closed form; the piecewise exponential reuse
estimate (flat to the turning point, exponential after it, continuous, turning point
moved by beta ln lambda); the order-preserving rule of the appendix (Lemma 1: with the
exponential, two blocks that are not accessed never swap places; a hyperbolic decay
does swap some); Eq. 5 summed over a request in closed form.  Then the library's
O(log n) policy, its O(n) scan mode, LRU and prefix-only are driven by random operation
sequences beside the oracle: same victims (exact ties go to the smaller id; scores that
differ by less than 1e-12 relative may resolve either way and are accepted when both are
minimal), same lambda, same scores.  No GPU is needed.
"""
import math

import numpy as np
import pytest

import bench
import segmented_kv_attention_msa_b300 as msa
from segmented_kv_attention_msa_b300 import build as B
from segmented_kv_attention_msa_b300 import workload as W
from oracle import evict_oracle as E


@pytest.fixture(scope="module", autouse=True)
def built():
    B.build()
    msa.lib()


# ----------------------------------------------------------------------------- oracle pins

def test_eq10_closed_form():
    # lambda = exp((tau - tau0)/beta - tau/alpha)
    assert E.lambda_update(16.0, 0.0, 16.0, 64.0) == pytest.approx(math.exp(1.0 - 0.25), rel=1e-15)
    assert E.lambda_update(10.0, 10.0, 4.0, 1e300) == pytest.approx(1.0, rel=1e-15)
    assert E.lambda_update(0.0, 8.0, 2.0, 5.0) == pytest.approx(math.exp(-4.0), rel=1e-15)


def test_reuse_estimate_is_piecewise_exponential():
    beta, lam = 8.0, 1.7
    for count in (1, 2, 5):
        tp = E.turning_point(count, lam, beta)
        assert tp == pytest.approx(beta * math.log(lam * count))
        # flat before the turning point, continuous at it, exponential with scale beta after
        assert E.reuse_estimate(count, max(0.0, tp - 3.0), lam, beta) == 1.0
        assert E.reuse_estimate(count, tp, lam, beta) == pytest.approx(1.0, rel=1e-12)
        for dt in (tp + 1.0, tp + 5.0, tp + 40.0):
            assert E.reuse_estimate(count, dt, lam, beta) == pytest.approx(math.exp(-(dt - tp) / beta), rel=1e-12)
    # rescaling the frequency term by lambda moves the turning point by beta ln lambda
    assert E.turning_point(3, 2.5, beta) - E.turning_point(3, 1.0, beta) == pytest.approx(beta * math.log(2.5))


def test_order_preserving_rule():
    """Lemma 1 (appendix A.1): under exponential decay, blocks that are not accessed keep
    their order for all later times; a hyperbolic decay, continuous and non-negative too,
    does not."""
    rng = np.random.default_rng(3)
    o = E.EvictOracle(beta=5.0, lambda0=0.05, period=0)      # small lambda: every block decays
    for b in range(40):
        o.insert(b, int(rng.integers(0, 500)), float(rng.integers(0, 30)))
    t_grid = [40.0, 60.0, 100.0, 200.0]
    orders = [sorted(o.blocks, key=lambda i: (o.log_score(i, t), i)) for t in t_grid]
    assert all(x == orders[0] for x in orders)

    def hyper(b, t):
        return E.recompute_cost(b["pos"], o.k5, o.k_const) / (1.0 + (t - b["t_last"]))
    h_orders = [sorted(o.blocks, key=lambda i: (hyper(o.blocks[i], t), i)) for t in t_grid]
    assert any(x != h_orders[0] for x in h_orders)


def test_modelled_request_cost_closed_forms():
    k5, kc = 3e-6, 4e-5
    n = 37
    # nothing cached: sum over q of k5 (2 q) + kc
    assert E.modelled_recompute_cost([False] * n, k5, kc) == pytest.approx(k5 * n * (n - 1) + kc * n, rel=1e-12)
    # everything cached costs nothing
    assert E.modelled_recompute_cost([True] * n, k5, kc) == 0.0
    # a cached prefix of l blocks, then r recomputed: sum of k5 (l + 2 q) + kc
    l, r = 10, 7
    want = sum(k5 * (l + 2 * q) + kc for q in range(r))
    assert E.modelled_recompute_cost([True] * l + [False] * r, k5, kc) == pytest.approx(want, rel=1e-12)
    # Eq. 5 itself
    assert E.marginal_cost(4, 3, k5, kc) == pytest.approx(k5 * 10 + kc)


def test_bench_model_matches_oracle():
    rng = np.random.default_rng(9)
    for _ in range(50):
        hit = (rng.random(int(rng.integers(0, 300))) < 0.5).tolist()
        assert bench.modelled_recompute_cost(hit, 3e-6, 4e-5) == pytest.approx(
            E.modelled_recompute_cost(hit, 3e-6, 4e-5), rel=1e-12, abs=0.0)


# ----------------------------------------------------------------------------- library vs oracle

KW = dict(k5=3e-6, k_const=4e-5, beta=6.0, alpha=20.0, tau0=2.0, lambda0=1.0, window=8, period=3)


def _drive(policy_name, seed, n_ops=1500, **kw):
    kw = {**KW, **kw}
    rng = np.random.default_rng(seed)
    lib = msa.EvictionPolicy(policy_name, **kw)
    orc = E.EvictOracle(policy_name, **kw)
    now = 0.0
    next_id = 0
    cached = []
    for _ in range(n_ops):
        now += float(rng.integers(0, 3))
        r = rng.random()
        if r < 0.35 or not cached:
            pos = int(rng.integers(0, 64))
            lib.insert(next_id, pos, now)
            orc.insert(next_id, pos, now)
            cached.append(next_id)
            next_id += 1
        elif r < 0.7:
            b = cached[int(rng.integers(0, len(cached)))]
            lib.access(b, now)
            orc.access(b, now)
        elif r < 0.75:
            b = cached.pop(int(rng.integers(0, len(cached))))
            lib.remove(b)
            orc.remove(b)
        else:
            if policy_name in ("cost", "cost_scan"):
                ls = {i: orc.log_score(i, now) for i in orc.blocks}
            v_lib = lib.victim(now)
            v_orc = orc.victim(now)
            if v_lib != v_orc:
                assert policy_name in ("cost", "cost_scan"), (policy_name, v_lib, v_orc)
                m = min(ls.values())
                assert abs(ls[v_lib] - m) <= 1e-12 * max(1.0, abs(m)), (v_lib, v_orc, ls[v_lib], m)
                return lib, orc       # a valid near-tie; the two states differ from here on
            cached.remove(v_lib)
        assert len(lib) == len(orc)
        assert lib.check(now)
        assert lib.lam == pytest.approx(orc.lam, rel=1e-13)
    for b in cached[:20]:
        assert lib.score(b, now) == pytest.approx(orc.score(b, now), rel=1e-12, abs=1e-300)
    return lib, orc


@pytest.mark.parametrize("policy", ["cost", "cost_scan", "lru", "prefix"])
@pytest.mark.parametrize("seed", range(4))
def test_policy_matches_oracle(policy, seed):
    _drive(policy, seed)


@pytest.mark.parametrize("lambda0,period,alpha", [(0.02, 0, 20.0), (40.0, 0, 20.0), (1.0, 1, 20.0), (1.0, 1, 3.0)])
def test_cost_policy_both_classes(lambda0, period, alpha):
    """Mostly decaying blocks (small lambda), mostly flat ones (large lambda) and a lambda
    that moves after every eviction, growing with the lifespan (alpha > beta) or shrinking
    (alpha < beta), so that blocks cross the flat / decaying boundary both ways."""
    lib, orc = _drive("cost", 11, lambda0=lambda0, period=period, window=4, alpha=alpha)
    assert len(lib) > 50


def test_lambda_follows_eq10():
    """Evictions at known times: after each `period` evictions lambda = Eq. 10 of the mean
    lifespan over the window."""
    kw = {**KW, "period": 2, "window": 3, "lambda0": 1.0}
    p = msa.EvictionPolicy("lru", **kw)
    spans = []
    for b in range(6):
        p.insert(b, 0, float(b))           # inserted at time b
    for k, t in enumerate((10.0, 14.0, 15.0, 30.0)):
        v = p.victim(t)                    # LRU: block k, lifespan t - k
        assert v == k
        spans.append(t - k)
        if (k + 1) % 2 == 0:
            tau = sum(spans[-3:]) / len(spans[-3:])
            assert p.lam == pytest.approx(math.exp((tau - kw["tau0"]) / kw["beta"] - tau / kw["alpha"]), rel=1e-14)


def test_invalid_use():
    with pytest.raises(msa.MSAError):
        msa.EvictionPolicy("cost", beta=0.0)
    with pytest.raises(msa.MSAError):
        msa.EvictionPolicy("cost", k_const=0.0)
    p = msa.EvictionPolicy("cost")
    with pytest.raises(msa.MSAError):
        p.victim(0.0)                      # empty
    p.insert(3, 0, 0.0)
    with pytest.raises(msa.MSAError):
        p.insert(3, 1, 1.0)                # duplicate
    with pytest.raises(msa.MSAError):
        p.access(4, 1.0)                   # unknown
    with pytest.raises(msa.MSAError):
        p.insert(5, -1, 1.0)               # negative position


def test_replay_same_with_library_and_oracle():
    """The bench's trace replay gives the same hits and modelled cost with the library's
    policy and with the oracle, for every policy, on a small multi-turn trace."""
    trace = W.multiturn_trace(seed=7, sessions=8, requests=150, first_blocks=(4, 40), turn_blocks=(1, 6))
    for name in ("cost", "lru", "prefix"):
        a = bench.replay_trace(msa.EvictionPolicy(name), trace, capacity=120)
        b = bench.replay_trace(E.EvictOracle(name), trace, capacity=120)
        assert a["hits"] == b["hits"] and a["blocks"] == b["blocks"]
        assert a["modelled_ms"] == pytest.approx(b["modelled_ms"], rel=1e-12)
