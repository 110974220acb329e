"""CPU oracle for Multi-Segment Attention (MSA) -- test infrastructure only.

This module is the plain, slow, obviously correct statement of what the MSA hot path
computes.  It exists to check the CUDA path and to be timed as a CPU baseline; only
the test suite, the package smoke check and the benchmark's CPU-baseline leg use it.
It shares no code with the CUDA path and imports nothing from the package.

Source: "Multi-Segment Attention: Enabling Efficient KV-Cache Management for Faster
Large Language Model Serving" (Shi, Chen, Chen, Miao, Cui).

* Eq. 1 (Fig. 1): A = Q K^T / sqrt(d_k), O = softmax(A) V.
* Section 4.1 (Fig. 4 text): the KV context is a union of disjoint regions
  (non-contiguous cache segments, e.g. a prefix and a suffix); Fig. 5 is MSA.
* Abstract: evicted blocks are recomputed on demand so outputs stay exact
  (lossless); the result is therefore exactly ordinary causal attention over the
  contiguous sequence, evaluated at the original positions of the chunk's tokens.

Readings where the pages are silent (each listed in the design notes):
* the mask is causal by original position, key position <= query position,
  inclusive of the query itself;
* grouped-query attention maps query head h to KV head h // (Hq / Hkv);
* LSE is the natural log of the softmax denominator of the scaled logits;
* decode: the query is the newest token of its sequence, whose K/V already sits in
  the pool, so it sees every KV token of that sequence;
* a query with no visible key gets O = 0 and LSE = -inf.

Arithmetic is fp64 on the bf16-rounded inputs (exact in fp64), which is strictly
closer to the exact result than the fp32 the attention definition would otherwise
be written in; ``dtype=np.float32`` gives an fp32 variant.

Every function is pinned by tests against closed forms, brute force and invariants
(see tests/test_oracle_pins.py); the canonical plan and chunk tiler are pinned only
to their written rules (parity unpinned against the pages, which give no rule).
"""
from __future__ import annotations

import math
from typing import Dict, List, Optional, Sequence, Tuple

import numpy as np

BLOCK = 16
POOL, CHUNK, MIXED = 0, 1, 2
SKIP, FULL, PARTIAL = 0, 1, 2
TILE_ROWS = 128          # tokens per KV tile and per query tile
TILE_BLOCKS = TILE_ROWS // BLOCK


# ----------------------------------------------------------------------------- gather

def seq_units(layout, s: int) -> List[Tuple[int, int, int, int]]:
    """KV units of sequence ``s``: pool blocks and chunk tokens.

    Each unit is (first_pos, src, id, n_tokens): a pool block (src POOL, id = physical
    block) holds block_fill[id] tokens at positions block_pos[id] + t; a chunk token
    (src CHUNK, id = global query row) holds one token at q_pos[id].  Segments are
    runs of logical blocks of the sequence's block-table row (section 4.1: the
    cache is a set of disjoint regions).
    """
    units = []
    for (seq, first, nb) in np.asarray(layout.segments).reshape(-1, 3):
        if int(seq) != s:
            continue
        for lb in range(int(first), int(first) + int(nb)):
            b = int(layout.block_table[s, lb])
            units.append((int(layout.block_pos[b]), POOL, b, int(layout.block_fill[b])))
    if layout.mode == "prefill":
        for r in range(int(layout.cu_q[s]), int(layout.cu_q[s + 1])):
            units.append((int(layout.q_pos[r]), CHUNK, r, 1))
    units.sort()
    return units


def canonical_tokens(layout, s: int) -> np.ndarray:
    """Canonical KV order of sequence ``s``: rows (src, id, offset, pos) sorted by pos."""
    rows = []
    for (p0, src, idx, n) in seq_units(layout, s):
        for t in range(n):
            rows.append((src, idx, t, p0 + t))
    arr = np.array(rows, np.int64).reshape(-1, 4)
    pos = arr[:, 3]
    if len(pos) and np.any(np.diff(pos) <= 0):
        raise ValueError("KV positions of a sequence must be unique")
    return arr


def gather_by_position(layout, s: int, k_pool, v_pool, k_chunk, v_chunk, dtype=np.float64,
                       chunk_keys: bool = True):
    """K and V of sequence ``s`` in ascending original position (bit-exact copies).
    With ``chunk_keys=False`` the chunk's own rows are left out (pool segments only).

    Returns (pos [L], K [L, Hkv, d], V [L, Hkv, d]).
    """
    tok = canonical_tokens(layout, s)
    if not chunk_keys:
        tok = tok[tok[:, 0] == POOL]
    L = len(tok)
    Hkv, d = layout.num_heads_kv, layout.head_dim
    K = np.empty((L, Hkv, d), dtype)
    V = np.empty((L, Hkv, d), dtype)
    pool = tok[:, 0] == POOL
    if pool.any():
        K[pool] = k_pool[tok[pool, 1], :, tok[pool, 2], :]
        V[pool] = v_pool[tok[pool, 1], :, tok[pool, 2], :]
    ch = ~pool
    if ch.any():
        K[ch] = k_chunk[tok[ch, 1]]
        V[ch] = v_chunk[tok[ch, 1]]
    return tok[:, 3].copy(), K, V


# ----------------------------------------------------------------------------- attention (Eq. 1)

def attention(q: np.ndarray, q_pos: np.ndarray, k: np.ndarray, v: np.ndarray,
              k_pos: np.ndarray, scale: float, dtype=np.float64, causal: bool = True):
    """Eq. 1 with a causal mask by original position, for one sequence.

    q [n, Hq, d]; k, v [m, Hkv, d]; q_pos [n]; k_pos [m].
    Query head h reads KV head h // (Hq // Hkv).  For each row i and head h:
      x_j = scale * <q_i, k_j>   for every key j with k_pos[j] <= q_pos[i]
      O = sum_j exp(x_j - max x) v_j / sum_j exp(x_j - max x)
      LSE = max x + ln sum_j exp(x_j - max x)
    Returns O [n, Hq, d] and LSE [n, Hq] in ``dtype``.
    """
    n, Hq, d = q.shape
    Hkv = k.shape[1]
    G = Hq // Hkv
    out = np.zeros((n, Hq, d), dtype)
    lse = np.full((n, Hq), -np.inf, dtype)
    if n == 0 or k.shape[0] == 0:
        return out, lse
    if causal:
        visible = k_pos[None, :].astype(np.int64) <= q_pos[:, None].astype(np.int64)
    else:
        visible = np.ones((n, k.shape[0]), bool)
    any_vis = visible.any(axis=1)
    for h in range(Hq):
        g = h // G
        x = (q[:, h, :].astype(dtype) @ k[:, g, :].astype(dtype).T) * dtype(scale)
        x = np.where(visible, x, -np.inf)
        m = np.max(x, axis=1, keepdims=True)
        m = np.where(np.isfinite(m), m, 0.0)
        p = np.exp(x - m)
        l = p.sum(axis=1)
        o = p @ v[:, g, :].astype(dtype)
        with np.errstate(divide="ignore", invalid="ignore"):
            out[:, h, :] = np.where(any_vis[:, None], o / l[:, None], 0.0)
            lse[:, h] = np.where(any_vis, m[:, 0] + np.log(l), -np.inf)
    return out, lse


def prefill(layout, q, k_chunk, v_chunk, k_pool, v_pool, scale: float,
            rows: Optional[np.ndarray] = None, dtype=np.float64, row_block: int = 1024,
            chunk_keys: bool = True):
    """MSA prefill: every chunk token attends over pool segments plus the chunk's own
    fresh K/V, causally by original position (section 4.1, abstract, Eq. 1).

    Inputs are numpy arrays of the bf16 values (any float dtype).  ``rows`` selects
    global query rows to evaluate (all if None).  ``chunk_keys=False`` computes the
    partial attention over the pool segments alone (the chunk rows are queries only),
    one of the parts a log-sum-exp merge combines.  Returns (rows, O, LSE).
    """
    total = layout.total_q
    rows = np.arange(total) if rows is None else np.asarray(rows, np.int64)
    out = np.zeros((len(rows), layout.num_heads_q, layout.head_dim), dtype)
    lse = np.full((len(rows), layout.num_heads_q), -np.inf, dtype)
    cu = np.asarray(layout.cu_q, np.int64)
    seq_of = np.searchsorted(cu, rows, side="right") - 1
    for s in np.unique(seq_of):
        sel = np.nonzero(seq_of == s)[0]
        kpos, K, V = gather_by_position(layout, int(s), k_pool, v_pool, k_chunk, v_chunk, dtype, chunk_keys)
        for i in range(0, len(sel), row_block):
            part = sel[i:i + row_block]
            r = rows[part]
            o, l = attention(q[r], layout.q_pos[r], K, V, kpos, scale, dtype)
            out[part] = o
            lse[part] = l
    return rows, out, lse


def decode(layout, q, k_pool, v_pool, scale: float, seqs: Optional[Sequence[int]] = None,
           dtype=np.float64):
    """MSA decode: the newest token of each sequence attends over all of its pool
    segments (every KV token is visible).  q [num_seqs, Hq, d].  Returns (seqs, O, LSE)."""
    seqs = list(range(layout.num_seqs)) if seqs is None else list(seqs)
    out = np.zeros((len(seqs), layout.num_heads_q, layout.head_dim), dtype)
    lse = np.full((len(seqs), layout.num_heads_q), -np.inf, dtype)
    empty = np.zeros((0, layout.num_heads_kv, layout.head_dim), np.float32)
    for i, s in enumerate(seqs):
        kpos, K, V = gather_by_position(layout, s, k_pool, v_pool, empty, empty, dtype)
        o, l = attention(q[s:s + 1], np.array([0]), K, V, kpos, scale, dtype, causal=False)
        out[i] = o[0]
        lse[i] = l[0]
    return np.array(seqs), out, lse


# ----------------------------------------------------------------------------- LSE merge

def merge_lse(o_parts: Sequence[np.ndarray], lse_parts: Sequence[np.ndarray], dtype=np.float64):
    """Combine attention results over disjoint key sets.

    With m = max_r lse_r and w_r = exp(lse_r - m):  O = sum_r w_r O_r / sum_r w_r,
    LSE = m + ln sum_r w_r.  A part with lse = -inf has weight 0; if every part is
    -inf the result is O = 0, LSE = -inf.
    """
    lse = np.stack([np.asarray(x, dtype) for x in lse_parts])           # [R, ...]
    o = np.stack([np.asarray(x, dtype) for x in o_parts])               # [R, ..., d]
    m = lse.max(axis=0)
    finite = np.isfinite(m)
    m_safe = np.where(finite, m, 0.0)
    w = np.where(np.isfinite(lse), np.exp(lse - m_safe[None]), 0.0)
    den = w.sum(axis=0)
    with np.errstate(divide="ignore", invalid="ignore"):
        out = np.where(finite[..., None], (w[..., None] * o).sum(axis=0) / den[..., None], 0.0)
        l = np.where(finite, m_safe + np.log(den), -np.inf)
    return out, l


# ----------------------------------------------------------------------------- adaptive chunk tiler

def chunk_sizes(R: int, min_chunk: int, max_chunk: int) -> List[int]:
    """Chunk sizes for R remaining recompute tokens (adaptive chunking, abstract).

    The pages give no rule, so this is the written reading: take the fewest chunks
    the maximum allows, n = ceil(R / max_chunk); make them near-equal and aligned to
    the 128-token tile, c = min(R, roundup(ceil(R / n), 128)); cut front to back into
    ceil(R / c) chunks of c tokens, the last taking the remainder.  A set smaller than
    min_chunk is one chunk.  max_chunk must be a positive multiple of 128.
    """
    if R <= 0:
        return []
    if R < min_chunk:
        return [R]
    n = -(-R // max_chunk)
    c = -(-R // n)
    c = min(R, -(-c // 128) * 128)
    k = -(-R // c)
    return [c] * (k - 1) + [R - c * (k - 1)]


# ----------------------------------------------------------------------------- canonical plan

def canonical_plan(layout) -> np.ndarray:
    """The plan of the MSA prefill in canonical form, as an int32 array.

    Layout (all int32):
      header  [mode(0 prefill / 1 decode), num_seqs, n_tok, n_kt, n_qt, n_cls]
      n_tok x (src, id, offset, pos)   canonical KV order of each sequence in turn
      n_kt  x (seq, src, tok_begin, n_tok, minpos, maxpos)
      n_qt  x (seq, row0, nrows, minpos, maxpos)
      n_cls x class                    for each query tile, one per KV tile of its sequence
    KV tiles: the sequence's KV in position order is cut into units of at most 16 tokens
    -- a pool block is one unit; a run of chunk tokens with no pool block between them is
    cut front to back into units of 16 (the last may be shorter) -- and every 8
    consecutive units make a tile, whatever their sources (src POOL or CHUNK when all
    units are of that kind, else MIXED).  A tile's smallest and largest positions are
    those of its first and last token.  Query tiles: the sequence's
    chunk rows cut every 128.  Class of (query tile, KV tile): SKIP when the query
    tile's largest position is below the KV tile's smallest; FULL when the query
    tile's smallest position is at least the KV tile's largest and the KV tile holds
    128 tokens; PARTIAL otherwise.  For decode the KV tiles, query tiles and classes
    are empty (the decode split is an implementation choice).
    """
    mode = 0 if layout.mode == "prefill" else 1
    toks, kts, qts, cls = [], [], [], []
    base = 0
    for s in range(layout.num_seqs):
        units = seq_units(layout, s)
        tok = canonical_tokens(layout, s)
        toks.append(tok)
        if mode == 1:
            base += len(tok)
            continue
        # tile units: pool blocks, and runs of chunk tokens cut into pieces of <= 16
        tunits = []   # [src, n_tok, minpos, maxpos]
        for (p0, src, idx, n) in units:
            if src == CHUNK and tunits and tunits[-1][0] == CHUNK and tunits[-1][1] < BLOCK:
                tunits[-1][1] += 1
                tunits[-1][3] = p0
            else:
                tunits.append([src, n, p0, p0 + n - 1])
        # kv tiles: 8 units each
        seq_kts = []
        t_index = base
        for a in range(0, len(tunits), TILE_BLOCKS):
            grp = tunits[a:a + TILE_BLOCKS]
            srcs = {u[0] for u in grp}
            src = srcs.pop() if len(srcs) == 1 else MIXED
            ntok = sum(u[1] for u in grp)
            seq_kts.append([src, t_index, ntok, grp[0][2], grp[-1][3]])
            t_index += ntok
        for c in seq_kts:
            kts.append((s, c[0], c[1], c[2], c[3], c[4]))
        # q tiles
        r0, r1 = int(layout.cu_q[s]), int(layout.cu_q[s + 1])
        for a in range(r0, r1, TILE_ROWS):
            b = min(r1, a + TILE_ROWS)
            qmin, qmax = int(layout.q_pos[a]), int(layout.q_pos[b - 1])
            qts.append((s, a, b - a, qmin, qmax))
            for c in seq_kts:
                kmin, kmax, nk = c[3], c[4], c[2]
                if qmax < kmin:
                    cls.append(SKIP)
                elif qmin >= kmax and nk == TILE_ROWS:
                    cls.append(FULL)
                else:
                    cls.append(PARTIAL)
        base += len(tok)
    tok_all = np.concatenate(toks) if toks else np.zeros((0, 4), np.int64)
    head = [mode, layout.num_seqs, len(tok_all), len(kts), len(qts), len(cls)]
    parts = [np.array(head, np.int64), tok_all.reshape(-1),
             np.array(kts, np.int64).reshape(-1), np.array(qts, np.int64).reshape(-1),
             np.array(cls, np.int64)]
    return np.concatenate(parts).astype(np.int32)


def useful_flops(layout) -> int:
    """Visible (query, key) pairs x Hq x 4 d: the multiply-adds of QK^T and PV that
    the causal-by-position definition needs, nothing for masked or padded pairs."""
    total = 0
    for s in range(layout.num_seqs):
        kpos = canonical_tokens(layout, s)[:, 3]
        kpos = np.sort(kpos)
        r0, r1 = int(layout.cu_q[s]), int(layout.cu_q[s + 1])
        if layout.mode == "prefill":
            vis = np.searchsorted(kpos, layout.q_pos[r0:r1], side="right")
            total += int(vis.sum())
        else:
            total += len(kpos)
    return total * layout.num_heads_q * 4 * layout.head_dim


# ----------------------------------------------------------------------------- write-back

def append_plan(q_pos, free_blocks, block_pos, block_fill, seq_blocks=()):
    """Placement of one sequence's chunk rows in paged pool blocks (write-back).

    The abstract: evicted blocks are recomputed on demand, at their original positions;
    once recomputed (and for the new tokens) their K/V belongs in the cache again.  The
    pages give no placement rule; this is the library's rule, stated plainly: the row at
    position p goes to the pool block that holds position block p // 16, at offset p % 16.
    A position block first met at offset 0 takes the next free block; one first met
    part-way continues the sequence's block (among ``seq_blocks``) that holds it.  Slots of
    a block fill from its current fill upward without holes.

    Returns (dst_slot, new_blocks, block_pos, block_fill) with copies of the two arrays
    updated; raises ValueError where the library returns an error.
    """
    q_pos = [int(x) for x in q_pos]
    block_pos = np.array(block_pos, np.int64)
    block_fill = np.array(block_fill, np.int64)
    if any(b <= a for a, b in zip(q_pos[:-1], q_pos[1:])) or any(p < 0 for p in q_pos):
        raise ValueError("positions must be non-negative and strictly ascending")
    owner = {}           # position block -> physical block
    next_free = 0
    dst = []
    for p in q_pos:
        pb = p // BLOCK
        if pb not in owner:
            if p % BLOCK != 0:
                held = [b for b in seq_blocks if block_fill[b] > 0 and block_pos[b] == pb * BLOCK]
                if not held:
                    raise ValueError("a row part-way into a block needs the block that holds it")
                owner[pb] = int(held[-1])
            else:
                if next_free >= len(free_blocks):
                    raise ValueError("not enough free blocks")
                owner[pb] = int(free_blocks[next_free])
                next_free += 1
                block_pos[owner[pb]] = pb * BLOCK
                block_fill[owner[pb]] = 0
        b = owner[pb]
        if p % BLOCK != block_fill[b]:
            raise ValueError("a hole inside a block")
        block_fill[b] += 1
        dst.append(b * BLOCK + p % BLOCK)
    return (np.array(dst, np.int64), np.array(free_blocks[:next_free], np.int64), block_pos, block_fill)


def append(k_chunk, v_chunk, k_pool, v_pool, dst_slot):
    """Copy every chunk row's K and V (all KV heads) into its pool slot; rows with a
    negative slot are skipped.  Returns the new pools (the inputs are not modified)."""
    k_pool = np.array(k_pool, copy=True)
    v_pool = np.array(v_pool, copy=True)
    for row, slot in enumerate(np.asarray(dst_slot)):
        if slot < 0:
            continue
        b, t = divmod(int(slot), BLOCK)
        k_pool[b, :, t, :] = k_chunk[row]
        v_pool[b, :, t, :] = v_chunk[row]
    return k_pool, v_pool
