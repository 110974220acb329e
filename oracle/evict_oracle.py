"""CPU oracle of the KV-block eviction policy -- test infrastructure only.

Plain statement of the cost-aware eviction rule, evaluated from its definition for every
cached block at every eviction (O(n) per eviction), against which the library's O(log n)
policy is checked.  Only the test suite uses it; it shares no code with the library.

Source: "Multi-Segment Attention: Enabling Efficient KV-Cache Management for Faster Large
Language Model Serving" (Shi, Chen, Chen, Miao, Cui):
* abstract: the eviction policy jointly weighs hit rate and position-aware recompute cost;
* Fig. 6 caption, Eq. 5: recomputing one more block costs
  Delta T_B = k5 (l1 + 2 q1) + (k2 - k3 + k5); (l1 + 2 q1) is approximated online (the
  approximation itself is cut off in the text);
* Fig. 7 / Fig. 8 captions: the reuse-time distribution and a piecewise exponential
  function; the policy runs in O(log n) against O(1) LRU and O(n) variants;
* Fig. 10 caption, Eq. 10: lambda rescales the frequency term, which moves the turning
  point of the piecewise exponential; lambda <- exp((tau - tau0)/beta - tau/alpha) with
  tau the mean lifespan of cache blocks over a sliding window;
* appendix A.1, Lemma 1: only an exponential keeps the order of two blocks that are not
  accessed (the order-preserving rule).

Readings where the text is cut off or silent (each listed in the design notes):
* (l1 + 2 q1) ~ p_b, the number of blocks before b in its sequence;
* reuse estimate of block b, dt after its last access: min(1, lambda F_b exp(-dt / beta)),
  flat until the turning point dt* = beta ln(lambda F_b), exponential after it; F_b is the
  number of accesses while cached;
* score = Delta T_B x reuse estimate (the recompute time that keeping b is expected to
  save); the smallest is evicted, ties to the smaller block id;
* tau = mean of (eviction time - insertion time) over the last `window` evictions, lambda
  refreshed every `period` evictions;
* modelled recompute cost of a request: Eq. 5's marginal cost summed over its recomputed
  blocks in position order, each with the cached (l1) and recomputed (q1) blocks before it.
"""
from __future__ import annotations

import math
from collections import deque
from typing import Dict, List, Sequence


def recompute_cost(pos_block: int, k5: float, k_const: float) -> float:
    """Eq. 5 with (l1 + 2 q1) approximated by the block's position p_b (in blocks);
    k_const = k2 - k3 + k5."""
    return k5 * pos_block + k_const


def reuse_estimate(count: int, dt: float, lam: float, beta: float) -> float:
    """Piecewise exponential reuse estimate: 1 up to the turning point beta ln(lam count),
    then lam count exp(-dt / beta)."""
    return min(1.0, lam * count * math.exp(-dt / beta))


def turning_point(count: int, lam: float, beta: float) -> float:
    return beta * math.log(lam * count)


def lambda_update(tau: float, tau0: float, beta: float, alpha: float) -> float:
    """Eq. 10."""
    return math.exp((tau - tau0) / beta - tau / alpha)


def marginal_cost(l1: int, q1: int, k5: float, k_const: float) -> float:
    """Eq. 5: the cost of recomputing one more block after l1 cached and q1 recomputed ones."""
    return k5 * (l1 + 2 * q1) + k_const


def modelled_recompute_cost(hit: Sequence[bool], k5: float, k_const: float) -> float:
    """Eq. 5 summed over the recomputed blocks of one request, in position order."""
    cost, l1, q1 = 0.0, 0, 0
    for h in hit:
        if h:
            l1 += 1
        else:
            cost += marginal_cost(l1, q1, k5, k_const)
            q1 += 1
    return cost


class EvictOracle:
    """The eviction rules evaluated from their definitions (O(n) per eviction).

    policy: "cost" (the score above), "lru" (least recently accessed first) or "prefix"
    (prefix caching: the block with the largest position first, then the least recent)."""

    def __init__(self, policy="cost", k5=3.07463e-6, k_const=3.49e-5, beta=16.0, alpha=64.0,
                 tau0=0.0, lambda0=1.0, window=64, period=16):
        self.policy = "cost" if policy == "cost_scan" else policy
        self.k5, self.k_const, self.beta, self.alpha, self.tau0 = k5, k_const, beta, alpha, tau0
        self.lam = lambda0
        self.window, self.period = window, period
        self.blocks: Dict[int, dict] = {}
        self.spans: deque = deque(maxlen=max(1, window))
        self.since = 0

    def __len__(self):
        return len(self.blocks)

    def insert(self, block: int, pos_block: int, now: float):
        if block in self.blocks:
            raise ValueError("block already cached")
        self.blocks[block] = {"pos": pos_block, "count": 1, "t_last": now, "t_ins": now}

    def access(self, block: int, now: float):
        b = self.blocks[block]
        b["count"] += 1
        b["t_last"] = now

    def remove(self, block: int):
        del self.blocks[block]

    def score(self, block: int, now: float) -> float:
        b = self.blocks[block]
        return (recompute_cost(b["pos"], self.k5, self.k_const) *
                reuse_estimate(b["count"], now - b["t_last"], self.lam, self.beta))

    def log_score(self, block: int, now: float) -> float:
        """ln of score(): the same product taken in logs, so that scores too small for
        fp64 (a block untouched for thousands of beta) still order as they should."""
        b = self.blocks[block]
        e = math.log(self.lam * b["count"]) - (now - b["t_last"]) / self.beta
        return math.log(recompute_cost(b["pos"], self.k5, self.k_const)) + min(0.0, e)

    def scores(self, now: float) -> Dict[int, float]:
        return {i: self.score(i, now) for i in self.blocks}

    def victim(self, now: float) -> int:
        if self.policy == "cost":
            order = sorted((self.log_score(i, now), i) for i in self.blocks)
        elif self.policy == "lru":
            order = sorted((b["t_last"], i) for i, b in self.blocks.items())
        else:
            order = sorted((-b["pos"], b["t_last"], i) for i, b in self.blocks.items())
        v = order[0][-1]
        span = now - self.blocks[v]["t_ins"]
        del self.blocks[v]
        if self.window > 0:
            self.spans.append(span)
            if self.period > 0:
                self.since += 1
                if self.since >= self.period:
                    self.since = 0
                    tau = math.fsum(self.spans) / len(self.spans)
                    self.lam = lambda_update(tau, self.tau0, self.beta, self.alpha)
        return v
