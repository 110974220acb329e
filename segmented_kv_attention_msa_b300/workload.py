"""Seeded synthetic workloads for Multi-Segment Attention (MSA).

This module builds the inputs that both the CUDA path and the CPU oracle consume:
a paged KV pool whose blocks carry their original token positions, a block table,
segment descriptors (runs of logical blocks with consecutive positions), the
positions of the query chunk (recomputed evicted blocks plus new tokens), and the
random Q/K/V values.  It performs none of the attention arithmetic and none of the
planning: it only lays data out.

The five named workloads follow the shapes the paper's serving setting implies
("Multi-Segment Attention: Enabling Efficient KV-Cache Management for Faster Large
Language Model Serving", abstract and Fig. 4 / section 4.1: cached segments that are
disjoint KV regions, evicted blocks recomputed on demand at their original
positions).  The pages publish no dataset that could be used here, so these
synthetic layouts stand in for the paper's LooGLE / BFCL traces.

Values are drawn with ``torch.randn`` from a ``torch.Generator`` seeded per
workload, on the device the caller asks for, and rounded to bf16 (round to
nearest even).  Layout metadata comes from ``numpy.random.default_rng(seed)``.
"""
from __future__ import annotations

import dataclasses
from typing import Callable, List, Optional, Sequence, Tuple

import numpy as np
import torch

BLOCK_SIZE = 16

# name of each numbered workload (the numbers are the order they are listed in)
WORKLOAD_NAMES = {
    1: "tiny_prefill_4h_d64_ctx512",
    2: "llama3_8b_layer_prefill_ctx8192_chunk2048",
    3: "multiturn_batch16_prefill",
    4: "decode_batch64_ctx4k_64k",
    5: "llama3_70b_layer_prefill_ctx131k_chunk8192",
}


def default_seed(index: int) -> int:
    return 20260000 + int(index)


@dataclasses.dataclass
class SeqSpec:
    """One sequence: pool-resident runs and the query chunk.

    pool_runs: list of (first_pos, n_tokens); first_pos is a multiple of 16 and the
        run occupies ceil(n_tokens/16) blocks, only the last of which may be partial.
    chunk_pos: sorted positions of the query-chunk tokens (prefill) or empty
        (decode: one query token per sequence sees the whole pool context).
    """
    pool_runs: List[Tuple[int, int]]
    chunk_pos: np.ndarray


@dataclasses.dataclass
class Layout:
    mode: str                      # "prefill" or "decode"
    num_heads_q: int
    num_heads_kv: int
    head_dim: int
    num_seqs: int
    num_pool_blocks: int
    block_pos: np.ndarray          # int32 [num_pool_blocks] original position of token 0 of the block
    block_fill: np.ndarray         # int32 [num_pool_blocks] valid tokens in the block (0 = unused)
    block_table: np.ndarray        # int32 [num_seqs, max_blocks] physical block of each logical block (-1 unused)
    segments: np.ndarray           # int32 [num_segments, 3] (seq, first_logical_block, num_blocks)
    cu_q: np.ndarray               # int32 [num_seqs + 1] query-row offsets
    q_pos: np.ndarray              # int32 [total_q] original position of each query row
    qk_std: float                  # std of the Q and K draws
    v_std: float
    name: str = ""
    seed: int = 0

    @property
    def total_q(self) -> int:
        return int(self.cu_q[-1])

    @property
    def max_blocks(self) -> int:
        return int(self.block_table.shape[1])


@dataclasses.dataclass
class Workload:
    layout: Layout
    q: torch.Tensor        # bf16 [total_q, Hq, d]
    k_chunk: torch.Tensor  # bf16 [total_q, Hkv, d]   (prefill; empty for decode)
    v_chunk: torch.Tensor
    k_pool: torch.Tensor   # bf16 [num_pool_blocks, Hkv, 16, d]
    v_pool: torch.Tensor


# ----------------------------------------------------------------------------- layout assembly

def assemble_layout(mode: str, num_heads_q: int, num_heads_kv: int, head_dim: int,
                    seqs: Sequence[SeqSpec], rng: np.random.Generator,
                    pool_slack: float = 1.25, qk_std: float = 1.0, v_std: float = 1.0,
                    name: str = "", seed: int = 0, shuffle_segments: bool = False) -> Layout:
    """Place every pool run of every sequence in a scattered paged pool.

    Physical block ids come from one random permutation of the pool; each run takes
    consecutive entries of it, so runs land scattered in the pool while staying
    block-granular.  The pool holds ``pool_slack`` times the blocks in use; the
    spare blocks keep fill 0.
    """
    runs_blocks = []
    for s in seqs:
        for (p0, n) in s.pool_runs:
            if p0 % BLOCK_SIZE != 0 or n <= 0:
                raise ValueError("pool runs start on a block boundary and are non-empty")
            runs_blocks.append((n + BLOCK_SIZE - 1) // BLOCK_SIZE)
    needed = int(sum(runs_blocks))
    num_pool_blocks = max(1, int(np.ceil(needed * pool_slack)))
    perm = rng.permutation(num_pool_blocks).astype(np.int32)
    block_pos = np.zeros(num_pool_blocks, np.int32)
    block_fill = np.zeros(num_pool_blocks, np.int32)
    rows: List[List[int]] = []
    segs: List[Tuple[int, int, int]] = []
    cursor = 0
    for si, s in enumerate(seqs):
        row: List[int] = []
        for (p0, n) in sorted(s.pool_runs):
            nb = (n + BLOCK_SIZE - 1) // BLOCK_SIZE
            ids = perm[cursor:cursor + nb]
            cursor += nb
            segs.append((si, len(row), nb))
            for k in range(nb):
                b = int(ids[k])
                block_pos[b] = p0 + BLOCK_SIZE * k
                block_fill[b] = min(BLOCK_SIZE, n - BLOCK_SIZE * k)
                row.append(b)
        rows.append(row)
    max_blocks = max(1, max(len(r) for r in rows))
    block_table = np.full((len(seqs), max_blocks), -1, np.int32)
    for si, r in enumerate(rows):
        block_table[si, :len(r)] = r
    segments = np.array(segs, np.int32).reshape(-1, 3)
    if shuffle_segments and len(segments) > 1:
        segments = segments[rng.permutation(len(segments))]
    if mode == "decode":
        cu_q = np.arange(len(seqs) + 1, dtype=np.int32)
        q_pos = np.array([_decode_qpos(s) for s in seqs], np.int32)
    else:
        lens = [len(s.chunk_pos) for s in seqs]
        cu_q = np.zeros(len(seqs) + 1, np.int32)
        cu_q[1:] = np.cumsum(lens)
        q_pos = (np.concatenate([np.asarray(s.chunk_pos, np.int64) for s in seqs])
                 if sum(lens) else np.zeros(0)).astype(np.int32)
    return Layout(mode=mode, num_heads_q=num_heads_q, num_heads_kv=num_heads_kv,
                  head_dim=head_dim, num_seqs=len(seqs), num_pool_blocks=num_pool_blocks,
                  block_pos=block_pos, block_fill=block_fill, block_table=block_table,
                  segments=segments, cu_q=cu_q, q_pos=q_pos, qk_std=qk_std, v_std=v_std,
                  name=name, seed=seed)


def _decode_qpos(s: SeqSpec) -> int:
    # the decode query is the newest token; its own K/V already sits in the pool
    return max(p0 + n for (p0, n) in s.pool_runs) - 1


# ----------------------------------------------------------------------------- values

def make_values(layout: Layout, device="cpu", seed: Optional[int] = None) -> Workload:
    """Draw Q, chunk K/V and pool K/V for a layout (fixed draw order), bf16 on ``device``."""
    seed = layout.seed if seed is None else seed
    gen = torch.Generator(device=device)
    gen.manual_seed(int(seed))
    Hq, Hkv, d = layout.num_heads_q, layout.num_heads_kv, layout.head_dim
    tq = layout.total_q
    nchunk = tq if layout.mode == "prefill" else 0

    def draw(shape, std):
        out = torch.empty(shape, dtype=torch.bfloat16, device=device)
        flat = out.view(-1)
        step = 1 << 26
        for i in range(0, flat.numel(), step):
            n = min(step, flat.numel() - i)
            x = torch.randn(n, generator=gen, device=device, dtype=torch.float32)
            if std != 1.0:
                x.mul_(std)
            flat[i:i + n].copy_(x)  # fp32 -> bf16 rounds to nearest even
        return out

    q = draw((tq, Hq, d), layout.qk_std)
    k_chunk = draw((nchunk, Hkv, d), layout.qk_std)
    v_chunk = draw((nchunk, Hkv, d), layout.v_std)
    k_pool = draw((layout.num_pool_blocks, Hkv, BLOCK_SIZE, d), layout.qk_std)
    v_pool = draw((layout.num_pool_blocks, Hkv, BLOCK_SIZE, d), layout.v_std)
    return Workload(layout, q, k_chunk, v_chunk, k_pool, v_pool)


# ----------------------------------------------------------------------------- helpers

def _composition(rng, total: int, parts: int, minimum: int) -> List[int]:
    """Uniform random composition of ``total`` into ``parts`` parts, each >= minimum."""
    free = total - parts * minimum
    if free < 0:
        raise ValueError("composition impossible")
    # stars and bars: choose parts-1 bar slots among free+parts-1
    bars = np.sort(rng.choice(free + parts - 1, size=parts - 1, replace=False)) if parts > 1 else np.array([], int)
    edges = np.concatenate([[-1], bars, [free + parts - 1]])
    return [int(e - s - 1) + minimum for s, e in zip(edges[:-1], edges[1:])]


def _blocks_to_runs(cached: np.ndarray) -> List[Tuple[int, int]]:
    """Boolean per-block mask -> list of (first_block, n_blocks) runs of True."""
    runs = []
    i, n = 0, len(cached)
    while i < n:
        if cached[i]:
            j = i
            while j < n and cached[j]:
                j += 1
            runs.append((i, j - i))
            i = j
        else:
            i += 1
    return runs


def _split_recompute(evicted_blocks_mask: np.ndarray, old_len: int, suffix: int,
                     chunk_sizes: Sequence[int]):
    """Order the recompute set (evicted blocks, then the new suffix) front to back and
    split it into chunks of the given sizes.  Every chunk but the last becomes
    pool-resident (already recomputed); the last chunk is the query chunk.

    Returns (pool runs of the earlier chunks as (first_pos, n_tokens), last-chunk positions).
    """
    ev = np.nonzero(evicted_blocks_mask)[0]
    rec = np.concatenate([
        (ev[:, None] * BLOCK_SIZE + np.arange(BLOCK_SIZE)[None, :]).reshape(-1),
        np.arange(old_len, old_len + suffix)]).astype(np.int64)
    total = sum(chunk_sizes)
    assert total == len(rec), (total, len(rec))
    last = chunk_sizes[-1]
    earlier = rec[:len(rec) - last]
    chunk = rec[len(rec) - last:]
    return _positions_to_runs(earlier), chunk


def _positions_to_runs(pos: np.ndarray) -> List[Tuple[int, int]]:
    """Sorted, block-aligned positions -> runs of consecutive positions (first_pos, n)."""
    runs = []
    if len(pos) == 0:
        return runs
    start = int(pos[0])
    prev = start
    for p in pos[1:]:
        p = int(p)
        if p != prev + 1:
            runs.append((start, prev - start + 1))
            start = p
        prev = p
    runs.append((start, prev - start + 1))
    return runs


def _cached_runs_tokens(cached_mask: np.ndarray) -> List[Tuple[int, int]]:
    return [(b0 * BLOCK_SIZE, nb * BLOCK_SIZE) for (b0, nb) in _blocks_to_runs(cached_mask)]


# ----------------------------------------------------------------------------- named workloads

def _wl1(rng, seed):
    L0, nb = 512, 32
    cached = np.zeros(nb, bool)
    cached[rng.choice(nb, 12, replace=False)] = True
    suffix = 64
    runs_pool, chunk = _split_recompute(~cached, L0, suffix, [20 * 16 + suffix])
    spec = SeqSpec(_cached_runs_tokens(cached) + runs_pool, chunk)
    return assemble_layout("prefill", 4, 4, 64, [spec], rng, qk_std=1.0, v_std=1.0,
                           name=WORKLOAD_NAMES[1], seed=seed)


def _wl2(rng, seed):
    nb, n_cached = 512, 307
    R = int(rng.integers(3, 11))
    run_lens = _composition(rng, n_cached, R, 1)
    # gaps g0 >= 0, g1..g_{R-1} >= 1, g_R >= 0, summing to the evicted count
    n_ev = nb - n_cached
    g = _composition(rng, n_ev + 2, R + 1, 1)
    g[0] -= 1
    g[-1] -= 1
    cached = np.zeros(nb, bool)
    b = g[0]
    for i in range(R):
        cached[b:b + run_lens[i]] = True
        b += run_lens[i] + g[i + 1]
    assert cached.sum() == n_cached
    suffix = 816
    runs_pool, chunk = _split_recompute(~cached, nb * BLOCK_SIZE, suffix, [2048, 2048])
    spec = SeqSpec(_cached_runs_tokens(cached) + runs_pool, chunk)
    s = 1.0 / np.sqrt(128.0)
    return assemble_layout("prefill", 32, 8, 128, [spec], rng, qk_std=s, v_std=1.0,
                           name=WORKLOAD_NAMES[2], seed=seed)


def _place_middle_holes(rng, nb_avail_end: int, lens: List[int]) -> List[Tuple[int, int]]:
    """Non-overlapping, non-adjacent block ranges inside [1, nb_avail_end)."""
    holes: List[Tuple[int, int]] = []
    for ln in lens:
        for _ in range(200):
            if nb_avail_end - 1 - ln < 1:
                break
            st = int(rng.integers(1, nb_avail_end - ln))
            ok = all(st + ln < a or st > a + l for (a, l) in holes)
            if ok:
                holes.append((st, ln))
                break
    return holes


def _wl3(rng, seed, tiler):
    if tiler is None:
        raise ValueError("the multi-turn batch workload needs the adaptive chunk tiler")
    specs = []
    for _ in range(16):
        L0 = int(rng.integers(2048, 32769)) // BLOCK_SIZE * BLOCK_SIZE
        nb = L0 // BLOCK_SIZE
        k = int(rng.poisson(6))
        evicted = np.zeros(nb, bool)
        if k >= 1:
            tl = min(int(rng.geometric(1.0 / 8.0)), nb - 1)
            evicted[nb - tl:] = True
            lens = [min(int(rng.geometric(1.0 / 8.0)), max(1, nb // 8)) for _ in range(k - 1)]
            for (st, ln) in _place_middle_holes(rng, nb - tl - 1, lens):
                evicted[st:st + ln] = True
        suffix = int(rng.integers(16, 513))
        R = int(evicted.sum()) * BLOCK_SIZE + suffix
        if R < 512:
            suffix += 512 - R
            R = 512
        sizes = list(tiler(R, 512, 4096))
        runs_pool, chunk = _split_recompute(evicted, L0, suffix, sizes)
        specs.append(SeqSpec(_cached_runs_tokens(~evicted) + runs_pool, chunk))
    s = 1.0 / np.sqrt(128.0)
    return assemble_layout("prefill", 32, 8, 128, specs, rng, qk_std=s, v_std=1.0,
                           name=WORKLOAD_NAMES[3], seed=seed)


def _wl4(rng, seed, batch: int = 64, lo: int = 4096, hi: int = 65536):
    specs = []
    for _ in range(batch):
        L = int(rng.integers(lo, hi + 1))
        nb = (L + BLOCK_SIZE - 1) // BLOCK_SIZE
        nseg = int(rng.integers(2, 33))
        cuts = np.sort(rng.choice(np.arange(1, nb), size=nseg - 1, replace=False))
        edges = np.concatenate([[0], cuts, [nb]])
        runs = []
        for a, b in zip(edges[:-1], edges[1:]):
            p0 = int(a) * BLOCK_SIZE
            n = min(int(b) * BLOCK_SIZE, L) - p0
            runs.append((p0, n))
        specs.append(SeqSpec(runs, np.zeros(0, np.int64)))
    s = 1.0 / np.sqrt(128.0)
    return assemble_layout("decode", 32, 8, 128, specs, rng, qk_std=s, v_std=1.0,
                           name=WORKLOAD_NAMES[4], seed=seed)


def _wl5(rng, seed):
    nb_total = 8192
    for _attempt in range(1000):
        cached = np.zeros(nb_total, bool)
        b, n_runs = 0, 0
        while b < nb_total:
            c = int(rng.geometric(1.0 / 25.0))
            cached[b:min(nb_total, b + c)] = True
            n_runs += 1
            b += c
            if b >= nb_total:
                break
            b += int(rng.geometric(1.0 / 8.0))
        if n_runs >= 200:
            break
    suffix = 1024
    R = int((~cached).sum()) * BLOCK_SIZE + suffix
    sizes = [R - 8192, 8192] if R > 8192 else [R]
    runs_pool, chunk = _split_recompute(~cached, nb_total * BLOCK_SIZE, suffix, sizes)
    spec = SeqSpec(_cached_runs_tokens(cached) + runs_pool, chunk)
    s = 1.0 / np.sqrt(128.0)
    return assemble_layout("prefill", 64, 8, 128, [spec], rng, qk_std=s, v_std=1.0,
                           name=WORKLOAD_NAMES[5], seed=seed)


def make_layout(index: int, seed: Optional[int] = None,
                tiler: Optional[Callable[[int, int, int], Sequence[int]]] = None,
                decode_batch: int = 64) -> Layout:
    """Layout of numbered workload ``index`` (1..5).  ``decode_batch`` shrinks the decode
    workload (4) to fewer sequences of the same distribution (for small profiling cases)."""
    seed = default_seed(index) if seed is None else int(seed)
    rng = np.random.default_rng(seed)
    if index == 1:
        return _wl1(rng, seed)
    if index == 2:
        return _wl2(rng, seed)
    if index == 3:
        return _wl3(rng, seed, tiler)
    if index == 4:
        lay = _wl4(rng, seed, batch=decode_batch)
        if decode_batch != 64:
            lay.name = f"decode_batch{decode_batch}_ctx4k_64k"
        return lay
    if index == 5:
        return _wl5(rng, seed)
    raise ValueError(f"unknown workload {index}")


def make_workload(index: int, seed: Optional[int] = None, device="cpu",
                  tiler=None) -> Workload:
    lay = make_layout(index, seed, tiler)
    return make_values(lay, device=device)


def custom_prefill(num_heads_q, num_heads_kv, head_dim, seqs: Sequence[SeqSpec], seed: int,
                   qk_std=1.0, v_std=1.0, shuffle_segments=False, pool_slack=1.25) -> Layout:
    rng = np.random.default_rng(seed)
    return assemble_layout("prefill", num_heads_q, num_heads_kv, head_dim, seqs, rng,
                           qk_std=qk_std, v_std=v_std, name="custom_prefill", seed=seed,
                           shuffle_segments=shuffle_segments, pool_slack=pool_slack)


def custom_decode(num_heads_q, num_heads_kv, head_dim, seqs: Sequence[SeqSpec], seed: int,
                  qk_std=1.0, v_std=1.0, shuffle_segments=False, pool_slack=1.25) -> Layout:
    rng = np.random.default_rng(seed)
    return assemble_layout("decode", num_heads_q, num_heads_kv, head_dim, seqs, rng,
                           qk_std=qk_std, v_std=v_std, name="custom_decode", seed=seed,
                           shuffle_segments=shuffle_segments, pool_slack=pool_slack)


def random_prefill_spec(rng: np.random.Generator, old_blocks: int, cached_frac: float,
                        suffix: int, chunk: Optional[int] = None) -> SeqSpec:
    """A sequence whose old context has randomly cached blocks; the chunk is the last
    ``chunk`` tokens of the recompute set (all of it if None)."""
    cached = rng.random(old_blocks) < cached_frac
    R = int((~cached).sum()) * BLOCK_SIZE + suffix
    c = R if chunk is None else min(chunk, R)
    sizes = [R - c, c] if R > c else [R]
    runs_pool, cpos = _split_recompute(~cached, old_blocks * BLOCK_SIZE, suffix, sizes)
    return SeqSpec(_cached_runs_tokens(cached) + runs_pool, cpos)


# ----------------------------------------------------------------------------- request traces

def multiturn_trace(seed: int = 20260100, sessions: int = 64, requests: int = 4000,
                    first_blocks=(16, 256), turn_blocks=(1, 16), popularity_sigma: float = 1.0):
    """A synthetic multi-session, multi-turn request trace (the paper's LooGLE / BFCL
    traces are not available).  Each session starts with a context of U[first_blocks]
    blocks; each of its turns adds U[turn_blocks] blocks and reads the whole context.  At
    every time step one session makes a request, picked with a fixed lognormal popularity
    weight, so reuse times are spread (popular sessions return soon, others rarely).
    Returns a list of (time, session, context blocks)."""
    rng = np.random.default_rng(seed)
    weights = rng.lognormal(0.0, popularity_sigma, sessions)
    weights /= weights.sum()
    length = rng.integers(first_blocks[0], first_blocks[1] + 1, sessions)
    grow = rng.integers(turn_blocks[0], turn_blocks[1] + 1, sessions)
    started = np.zeros(sessions, bool)
    trace = []
    for t in range(requests):
        s = int(rng.choice(sessions, p=weights))
        if started[s]:
            length[s] += grow[s]
        started[s] = True
        trace.append((t, s, int(length[s])))
    return trace
