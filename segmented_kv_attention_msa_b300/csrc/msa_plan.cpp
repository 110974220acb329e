// Host planner of Multi-Segment Attention (MSA): validates segment descriptors and
// the paged block table, puts every sequence's KV context (pool segments plus the
// chunk's own tokens) in original-position order, cuts it into KV tiles, cuts the
// chunk into query tiles, classifies each (query tile, KV tile) pair by position
// (skip / full / partial), orders the CTA work list longest first, and splits decode
// contexts into split-KV units.  No CUDA call is made here.
//
// Paper: "Multi-Segment Attention: Enabling Efficient KV-Cache Management for Faster
// Large Language Model Serving", section 4.1 (a KV context of disjoint regions) and the
// abstract (evicted blocks recomputed at their original positions; adaptive chunking).
#include <algorithm>
#include <climits>
#include <cstring>
#include <new>
#include <numeric>
#include <vector>

#include "msa_internal.h"

using namespace msa;

namespace {

struct Unit {  // pool block or chunk token, ordered by first position
  int32_t first_pos, src, id, n;
};

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

msa_status_t build_units(const msa_plan_opts_t* opts, msa_mode_t mode, int32_t num_seqs,
                         const msa_segment_t* segs, int32_t num_segs, const int32_t* block_table,
                         int32_t max_blocks, const int32_t* block_pos, const int32_t* block_fill,
                         int32_t num_pool_blocks, const int32_t* cu_q, const int32_t* q_pos,
                         std::vector<std::vector<Unit>>& units) {
  units.assign(num_seqs, {});
  for (int32_t i = 0; i < num_segs; ++i) {
    const msa_segment_t& s = segs[i];
    if (s.seq < 0 || s.seq >= num_seqs || s.num_blocks <= 0 || s.first_logical_block < 0)
      return MSA_ERR_INVALID_ARG;
    if ((int64_t)s.first_logical_block + s.num_blocks > max_blocks) return MSA_ERR_BLOCK_OOB;
    const int32_t* row = block_table + (size_t)s.seq * max_blocks;
    for (int32_t k = 0; k < s.num_blocks; ++k) {
      int32_t b = row[s.first_logical_block + k];
      if (b < 0 || b >= num_pool_blocks) return MSA_ERR_BLOCK_OOB;
      int32_t f = block_fill[b], p = block_pos[b];
      if (f < 1 || f > kBlock || p < 0 || p % kBlock != 0) return MSA_ERR_INVALID_ARG;
      if (k + 1 < s.num_blocks) {
        int32_t bn = row[s.first_logical_block + k + 1];
        if (bn < 0 || bn >= num_pool_blocks) return MSA_ERR_BLOCK_OOB;
        if (f != kBlock || block_pos[bn] != p + kBlock) return MSA_ERR_INVALID_ARG;
      }
      units[s.seq].push_back({p, SRC_POOL, b, f});
    }
  }
  if (cu_q[0] != 0) return MSA_ERR_INVALID_ARG;
  for (int32_t s = 0; s < num_seqs; ++s) {
    int32_t r0 = cu_q[s], r1 = cu_q[s + 1];
    if (r1 < r0) return MSA_ERR_INVALID_ARG;
    if (mode == MSA_DECODE) {
      if (r1 - r0 != 1) return MSA_ERR_INVALID_ARG;
      continue;
    }
    for (int32_t r = r0; r < r1; ++r) {
      if (q_pos[r] < 0) return MSA_ERR_INVALID_ARG;
      if (r > r0 && q_pos[r] <= q_pos[r - 1]) return MSA_ERR_INVALID_ARG;
      if (!opts->chunk_queries_only) units[s].push_back({q_pos[r], SRC_CHUNK, r, 1});
    }
  }
  for (int32_t s = 0; s < num_seqs; ++s) {
    auto& us = units[s];
    std::sort(us.begin(), us.end(), [](const Unit& a, const Unit& b) {
      if (a.first_pos != b.first_pos) return a.first_pos < b.first_pos;
      if (a.src != b.src) return a.src < b.src;
      return a.id < b.id;
    });
    for (size_t i = 1; i < us.size(); ++i)
      if (us[i].first_pos <= us[i - 1].first_pos + us[i - 1].n - 1) return MSA_ERR_POS_OVERLAP;
    if (mode == MSA_DECODE && us.empty()) return MSA_ERR_INVALID_ARG;
  }
  return MSA_OK;
}

// A KV tile's unit: a pool block, or up to 16 chunk tokens that are consecutive in the
// canonical order (and so consecutive chunk rows).  One 16-row TMA box each.
struct TileUnit {
  int32_t src, id, first_pos, n;  // id: physical block, or the first chunk row
};

struct KTileHost {
  int32_t seq, src, tok_begin, ntok, minpos, maxpos, nunits;
  int32_t first_unit;  // into the flat TileUnit list
};


// ---------------------------------------------------------------- prefill schedule
//
// The prefill kernel is persistent: one CTA per SM walks a fixed list of pieces.  A work
// item is (query tile, KV head, pair of query heads) over the query tile's list of
// non-skipped KV tiles.  Items differ a lot in length (a query tile late in position sees
// many more keys), and a few hundred of them over 148 SMs balance poorly when each item
// stays whole.  So the items, longest first, are laid end to end and cut into `ctas`
// consecutive stretches of near-equal cost; an item that straddles a cut becomes several
// pieces, each computing a partial (O, max, sum) over its part of the list, merged on the
// device by the piece that finishes last (log-sum-exp merge).  The cost model counts a
// full tile as kWFull, a partial (masked) tile as kWPartial, each piece's set-up and
// epilogue as kWPiece, and each piece of a split item kWSplit more (its partial store, the
// hand-shake, and the merge that one of them does).  The weights are B300 measurements:
// per-CTA times of whole launches fitted by least squares to the CTAs' tile and piece
// counts (a full tile ~1.9 us of a CTA's time, a masked tile 1.34 times that, a piece 2.8
// full tiles, a split piece 5 more).  No piece is shorter than kMinPiece tiles.  The
// smallest stretch cost for which the walk fits in `ctas` CTAs is found by bisection.
constexpr int32_t kDefaultCtas = 148;
constexpr int64_t kWFull = 8, kWPartial = 11, kWPiece = 22, kWSplit = 40;
constexpr int32_t kMinPiece = 4;

struct ItemRef {
  int32_t qt, g, h0;
};

struct Cut {
  int32_t item, j0, n, cta;
};

// Walk the items with stretch cost T; returns false if more than `ctas` CTAs are needed.
bool walk_items(const std::vector<std::vector<int64_t>>& pre, const std::vector<int32_t>& order,
                int64_t T, int32_t ctas, std::vector<Cut>* cuts) {
  int32_t c = 0;
  int64_t cap = T;
  if (cuts) cuts->clear();
  for (int32_t it : order) {
    const std::vector<int64_t>& w = pre[it];  // prefix sums of tile weights, w[0] = 0
    const int32_t n = (int32_t)w.size() - 1;
    if (n == 0) {  // a query tile that sees no key: one empty piece writes its rows
      if (cap < kWPiece) {
        if (++c >= ctas) return false;
        cap = T;
      }
      if (cuts) cuts->push_back({it, 0, 0, c});
      cap -= kWPiece;
      continue;
    }
    int32_t j = 0;
    while (j < n) {
      // the rest of the item as one piece: a split piece if an earlier piece took its start
      const int64_t rest = w[n] - w[j] + kWPiece + (j > 0 ? kWSplit : 0);
      if (rest <= cap) {
        if (cuts) cuts->push_back({it, j, n - j, c});
        cap -= rest;
        j = n;
        break;
      }
      // longest prefix of the rest that fits in what is left of this CTA (a split piece)
      int32_t j2 = j;
      while (j2 < n && w[j2 + 1] - w[j] + kWPiece + kWSplit <= cap) ++j2;
      if (n - j2 < kMinPiece) j2 = n - kMinPiece;
      if (j2 - j >= kMinPiece) {
        if (cuts) cuts->push_back({it, j, j2 - j, c});
        j = j2;
      }
      if (++c >= ctas) return false;
      cap = T;
    }
  }
  return true;
}

// Cut one list of items (in `order`) into stretches over `ctas` CTAs, the smallest
// stretch cost that fits found by bisection; CTA indices run backwards when `reverse`.
void balance(const std::vector<std::vector<int64_t>>& pre, const std::vector<int32_t>& order, int32_t ctas,
             bool reverse, std::vector<Cut>& cuts) {
  int64_t total = 0;
  for (int32_t it : order) total += pre[it].back() + kWPiece;
  // with T = total everything fits in one CTA, so the bisection always ends feasible
  int64_t lo = (total + ctas - 1) / ctas, hi = total;
  while (lo < hi) {
    const int64_t mid = lo + (hi - lo) / 2;
    if (walk_items(pre, order, mid, ctas, nullptr)) hi = mid;
    else lo = mid + 1;
  }
  walk_items(pre, order, lo, ctas, &cuts);
  if (reverse)
    for (Cut& c : cuts) c.cta = ctas - 1 - c.cta;
}

// KV-head phases.  Every work item streams the KV tiles of its KV head.  When the KV of all
// heads together is larger than the L2 cache can hold, CTAs that run items of different
// heads at the same time evict each other's tiles, and every item re-reads its tiles from
// DRAM.  So then the items are balanced head by head and every CTA runs its share of head
// 0, then of head 1, and so on: at any time the CTAs read one head's KV (the walk runs
// forwards for even heads and backwards for odd ones, so that the remainders of the
// per-head balancing land on different CTAs).
constexpr int64_t kPhaseKvBytes = 96ll << 20;

void schedule_prefill(const std::vector<QTileRec>& qts, const std::vector<int32_t>& list,
                      const std::vector<ItemRef>& items, int32_t ctas, int32_t Hkv, int64_t kv_bytes,
                      std::vector<WorkRec>& work, std::vector<int32_t>& cta_begin, std::vector<int32_t>& sched) {
  work.clear();
  cta_begin.assign(1, 0);
  sched.clear();
  if (items.empty()) return;
  std::vector<std::vector<int64_t>> pre(items.size());
  for (size_t i = 0; i < items.size(); ++i) {
    const QTileRec& q = qts[items[i].qt];
    std::vector<int64_t>& w = pre[i];
    w.assign(q.list_count + 1, 0);
    for (int32_t j = 0; j < q.list_count; ++j)
      w[j + 1] = w[j] + (list[q.list_begin + j] < 0 ? kWPartial : kWFull);
  }
  ctas = std::max<int32_t>(1, ctas);
  const bool phased = kv_bytes > kPhaseKvBytes && Hkv > 1;
  const int32_t nphase = phased ? Hkv : 1;
  // longest first within each phase; ties keep (query tile, KV head, head) order
  std::vector<std::vector<Cut>> cuts(nphase);
  for (int32_t ph = 0; ph < nphase; ++ph) {
    std::vector<int32_t> order;
    for (int32_t i = 0; i < (int32_t)items.size(); ++i)
      if (!phased || items[i].g == ph) order.push_back(i);
    std::stable_sort(order.begin(), order.end(),
                     [&](int32_t a, int32_t b) { return pre[a].back() > pre[b].back(); });
    balance(pre, order, ctas, phased && (ph & 1), cuts[ph]);
  }
  // pieces per item (numbered in list order, the walk's order), partial slots for items
  // in several pieces
  std::vector<int32_t> nparts(items.size(), 0), slot0(items.size(), -1);
  std::vector<std::vector<int32_t>> part(nphase);
  for (int32_t ph = 0; ph < nphase; ++ph)
    for (const Cut& c : cuts[ph]) part[ph].push_back(nparts[c.item]++);
  int32_t slots = 0;
  for (const std::vector<Cut>& cs : cuts)
    for (const Cut& c : cs)
      if (nparts[c.item] > 1 && slot0[c.item] < 0) {
        slot0[c.item] = slots;
        slots += nparts[c.item];
      }
  // each CTA runs its pieces phase by phase; within a phase, pieces of split items first
  // (their merges then happen early), then whole items, each group in walk order
  std::vector<std::vector<std::vector<int32_t>>> by_cta(ctas, std::vector<std::vector<int32_t>>(nphase));
  for (int32_t ph = 0; ph < nphase; ++ph)
    for (int32_t i = 0; i < (int32_t)cuts[ph].size(); ++i) by_cta[cuts[ph][i].cta][ph].push_back(i);
  int32_t used = 0;
  for (int32_t c = 0; c < ctas; ++c)
    for (int32_t ph = 0; ph < nphase; ++ph)
      if (!by_cta[c][ph].empty()) used = c + 1;
  for (int32_t c = 0; c < used; ++c) {
    for (int32_t ph = 0; ph < nphase; ++ph)
      for (int pass = 0; pass < 2; ++pass)
        for (int32_t i : by_cta[c][ph]) {
          const Cut& cu = cuts[ph][i];
          const bool split = nparts[cu.item] > 1;
          if ((pass == 0) != split) continue;
          const ItemRef& r = items[cu.item];
          const int32_t slot = split ? slot0[cu.item] + part[ph][i] : -1;
          work.push_back({r.qt, r.g, r.h0, cu.j0, cu.n, nparts[cu.item], slot0[cu.item], slot});
          const int32_t rec[9] = {c, r.qt, r.g, r.h0, cu.j0, cu.n, nparts[cu.item], slot0[cu.item], slot};
          sched.insert(sched.end(), rec, rec + 9);
        }
    cta_begin.push_back((int32_t)work.size());
  }
}

}  // namespace

extern "C" msa_status_t msa_chunk_sizes(int32_t R, int32_t min_chunk, int32_t max_chunk,
                                        int32_t* sizes, int32_t capacity, int32_t* n) {
  if (!n || R < 0 || min_chunk < 0 || max_chunk <= 0 || max_chunk % kTileRows != 0)
    return MSA_ERR_INVALID_ARG;
  std::vector<int32_t> out;
  if (R > 0) {
    if (R < min_chunk) {
      out.push_back(R);
    } else {
      int64_t k0 = ceil_div(R, max_chunk);
      int64_t c = ceil_div(R, k0);
      c = std::min<int64_t>(R, ceil_div(c, kTileRows) * kTileRows);
      int64_t k = ceil_div(R, c);
      for (int64_t i = 0; i + 1 < k; ++i) out.push_back((int32_t)c);
      out.push_back((int32_t)(R - c * (k - 1)));
    }
  }
  *n = (int32_t)out.size();
  if (sizes) {
    if (capacity < (int32_t)out.size()) return MSA_ERR_WORKSPACE;
    std::copy(out.begin(), out.end(), sizes);
  }
  return MSA_OK;
}

extern "C" msa_status_t msa_plan_create(const msa_plan_opts_t* opts, msa_mode_t mode,
                                        int32_t num_seqs, const msa_segment_t* segs,
                                        int32_t num_segs, const int32_t* block_table,
                                        int32_t max_blocks, const int32_t* block_pos,
                                        const int32_t* block_fill, int32_t num_pool_blocks,
                                        const int32_t* cu_q, const int32_t* q_pos,
                                        msa_plan_t** out) {
  if (!out) return MSA_ERR_INVALID_ARG;
  *out = nullptr;
  if (!opts || num_seqs <= 0 || num_segs < 0 || max_blocks < 0 || num_pool_blocks < 0 || !cu_q)
    return MSA_ERR_INVALID_ARG;
  if (mode != MSA_PREFILL && mode != MSA_DECODE) return MSA_ERR_INVALID_ARG;
  if (num_segs > 0 && (!segs || !block_table || !block_pos || !block_fill)) return MSA_ERR_INVALID_ARG;
  for (int i = 0; i < 2; ++i)
    if (opts->reserved[i] != 0) return MSA_ERR_INVALID_ARG;
  if (opts->chunk_queries_only != 0 && opts->chunk_queries_only != 1) return MSA_ERR_INVALID_ARG;
  if (opts->prefill_ctas < 0) return MSA_ERR_INVALID_ARG;
  const int32_t Hq = opts->num_heads_q, Hkv = opts->num_heads_kv, d = opts->head_dim;
  if (Hq <= 0 || Hkv <= 0) return MSA_ERR_INVALID_ARG;
  if (Hq % Hkv != 0 || (d != 64 && d != 128) || opts->block_size != kBlock) return MSA_ERR_UNSUPPORTED;
  if (opts->decode_split_blocks < 0 || opts->decode_min_ctas < 0) return MSA_ERR_INVALID_ARG;
  if (mode == MSA_PREFILL && cu_q[num_seqs] > 0 && !q_pos) return MSA_ERR_INVALID_ARG;
  // the kernels see the pool as [num_pool_blocks * Hkv * 16] rows and the chunk K/V as
  // [total_q * Hkv] rows of one head each, addressed by 32-bit TMA coordinates
  if ((int64_t)num_pool_blocks * Hkv * kBlock > INT32_MAX) return MSA_ERR_UNSUPPORTED;
  if (mode == MSA_PREFILL && (int64_t)cu_q[num_seqs] * Hkv > INT32_MAX) return MSA_ERR_UNSUPPORTED;

  std::vector<std::vector<Unit>> units;
  msa_status_t st = build_units(opts, mode, num_seqs, segs, num_segs, block_table, max_blocks,
                                block_pos, block_fill, num_pool_blocks, cu_q, q_pos, units);
  if (st != MSA_OK) return st;

  msa_plan_t* P = new (std::nothrow) msa_plan_t();
  if (!P) return MSA_ERR_INVALID_ARG;
  P->mode = mode;
  P->num_seqs = num_seqs;
  P->Hq = Hq;
  P->Hkv = Hkv;
  P->d = d;
  P->G = Hq / Hkv;
  P->hpc = (P->G % 2 == 0) ? 2 : 1;
  P->total_q = cu_q[num_seqs];
  P->num_pool_blocks = num_pool_blocks;
  std::memset(&P->stats, 0, sizeof(P->stats));

  // ---- canonical token list
  std::vector<int32_t> toks;
  std::vector<int32_t> seq_tok_begin(num_seqs + 1, 0);
  for (int32_t s = 0; s < num_seqs; ++s) {
    seq_tok_begin[s] = (int32_t)(toks.size() / 4);
    for (const Unit& u : units[s])
      for (int32_t t = 0; t < u.n; ++t) {
        toks.push_back(u.src);
        toks.push_back(u.id);
        toks.push_back(u.src == SRC_POOL ? t : 0);
        toks.push_back(u.first_pos + t);
      }
  }
  seq_tok_begin[num_seqs] = (int32_t)(toks.size() / 4);
  P->n_tok = seq_tok_begin[num_seqs];

  std::vector<KTileHost> kts;
  std::vector<QTileRec> qts;
  std::vector<int32_t> cls;
  std::vector<int32_t> seq_kt_begin(num_seqs + 1, 0);
  std::vector<TileUnit> tunits;
  if (mode == MSA_PREFILL) {
    // KV tiles: the sequence's units in position order, 8 per tile, pool blocks and runs of
    // chunk tokens alike (a run of consecutive chunk tokens is cut into units of <= 16), so
    // a fragmented cache still gives full tiles
    for (int32_t s = 0; s < num_seqs; ++s) {
      seq_kt_begin[s] = (int32_t)kts.size();
      const size_t tu0 = tunits.size();
      for (const Unit& u : units[s]) {
        if (u.src == SRC_CHUNK && !tunits.empty() && tunits.size() > tu0 && tunits.back().src == SRC_CHUNK &&
            tunits.back().n < kBlock && tunits.back().id + tunits.back().n == u.id) {
          tunits.back().n += 1;
        } else {
          tunits.push_back({u.src, u.id, u.first_pos, u.n});
        }
      }
      int32_t t_index = seq_tok_begin[s];
      for (size_t a = tu0; a < tunits.size(); a += kTileBlocks) {
        const size_t b = std::min(tunits.size(), a + kTileBlocks);
        KTileHost t{s, tunits[a].src, t_index, 0, tunits[a].first_pos, 0, (int32_t)(b - a), (int32_t)a};
        for (size_t i = a; i < b; ++i) {
          if (tunits[i].src != t.src) t.src = SRC_MIXED;
          t.ntok += tunits[i].n;
        }
        // the last unit's last token: a chunk unit's tokens need not be at consecutive positions
        const TileUnit& lu = tunits[b - 1];
        t.maxpos = lu.src == SRC_POOL ? lu.first_pos + lu.n - 1 : q_pos[lu.id + lu.n - 1];
        t_index += t.ntok;
        kts.push_back(t);
      }
    }
    seq_kt_begin[num_seqs] = (int32_t)kts.size();
    for (int32_t s = 0; s < num_seqs; ++s) {
      for (int32_t a = cu_q[s]; a < cu_q[s + 1]; a += kTileRows) {
        int32_t b = std::min(cu_q[s + 1], a + kTileRows);
        QTileRec q{s, a, b - a, q_pos[a], q_pos[b - 1], 0, 0, 0};
        for (int32_t k = seq_kt_begin[s]; k < seq_kt_begin[s + 1]; ++k) {
          const KTileHost& t = kts[k];
          int32_t c;
          if (q.maxpos < t.minpos) c = CLS_SKIP;
          else if (q.minpos >= t.maxpos && t.ntok == kTileRows) c = CLS_FULL;
          else c = CLS_PARTIAL;
          cls.push_back(c);
        }
        qts.push_back(q);
      }
    }
  }
  P->n_kt = (int32_t)kts.size();
  P->n_qt = (int32_t)qts.size();

  // ---- canonical export
  P->canon = {(int32_t)mode, num_seqs, P->n_tok, P->n_kt, P->n_qt, (int32_t)cls.size()};
  P->canon.insert(P->canon.end(), toks.begin(), toks.end());
  for (const KTileHost& t : kts) {
    int32_t r[6] = {t.seq, t.src, t.tok_begin, t.ntok, t.minpos, t.maxpos};
    P->canon.insert(P->canon.end(), r, r + 6);
  }
  for (const QTileRec& q : qts) {
    int32_t r[5] = {q.seq, q.row0, q.nrows, q.minpos, q.maxpos};
    P->canon.insert(P->canon.end(), r, r + 5);
  }
  P->canon.insert(P->canon.end(), cls.begin(), cls.end());

  // ---- statistics shared by both modes
  int64_t pairs = 0;
  for (int32_t s = 0; s < num_seqs; ++s) {
    int32_t nt = seq_tok_begin[s + 1] - seq_tok_begin[s];
    if (mode == MSA_DECODE) {
      pairs += nt;
      continue;
    }
    // visible keys of each query = keys with pos <= q_pos (tokens are sorted by pos)
    const int32_t* tp = toks.data() + (size_t)seq_tok_begin[s] * 4;
    int32_t j = 0;
    for (int32_t r = cu_q[s]; r < cu_q[s + 1]; ++r) {
      while (j < nt && tp[(size_t)j * 4 + 3] <= q_pos[r]) ++j;
      pairs += j;
    }
  }
  P->stats.useful_flops = pairs * (int64_t)Hq * 4 * d;
  P->stats.kv_tokens = P->n_tok;
  P->stats.num_kv_tiles = P->n_kt;
  P->stats.num_q_tiles = P->n_qt;

  // ---- device image
  std::vector<int32_t> list;
  std::vector<ItemRef> items;
  std::vector<WorkRec> work;
  std::vector<int32_t> cta_begin{0}, sched;
  std::vector<KTileRec> ktr(kts.size());
  std::vector<SplitRec> splits;
  std::vector<int32_t> blist, bfill;
  std::vector<GatherRec> gather;

  if (mode == MSA_PREFILL) {
    for (size_t k = 0; k < kts.size(); ++k) {
      const KTileHost& t = kts[k];
      KTileRec& r = ktr[k];
      std::memset(&r, 0, sizeof(r));
      r.src = t.src;
      r.ntok = t.ntok;
      r.minpos = t.minpos;
      r.maxpos = t.maxpos;
      r.full = t.ntok == kTileRows;
      r.nblk = t.nunits;
      for (int32_t i = 0; i < t.nunits; ++i) {
        const TileUnit& u = tunits[t.first_unit + i];
        r.blk[i] = u.src == SRC_POOL ? u.id : -(u.id + 1);
        r.bpos[i] = u.first_pos;
        r.bfill[i] = u.n;
      }
    }
    size_t ci = 0;
    int64_t tile_pairs = 0, partial_pairs = 0;
    for (size_t qi = 0; qi < qts.size(); ++qi) {
      QTileRec& q = qts[qi];
      q.list_begin = (int32_t)list.size();
      int32_t s = q.seq;
      // full tiles first, then partial ones, each group in position order
      for (int pass = 0; pass < 2; ++pass) {
        for (int32_t k = seq_kt_begin[s]; k < seq_kt_begin[s + 1]; ++k) {
          int32_t c = cls[ci + (k - seq_kt_begin[s])];
          if (pass == 0 && c == CLS_FULL) list.push_back(k);
          if (pass == 1 && c == CLS_PARTIAL) list.push_back(k | (int32_t)0x80000000u);
        }
      }
      for (int32_t k = seq_kt_begin[s]; k < seq_kt_begin[s + 1]; ++k) {
        if (cls[ci + (k - seq_kt_begin[s])] == CLS_PARTIAL) ++partial_pairs;
      }
      ci += seq_kt_begin[s + 1] - seq_kt_begin[s];
      q.list_count = (int32_t)list.size() - q.list_begin;
      tile_pairs += q.list_count;
      for (int32_t g = 0; g < Hkv; ++g)
        for (int32_t h = 0; h < P->G; h += P->hpc) items.push_back({(int32_t)qi, g, g * P->G + h});
    }
    const int32_t ctas = opts->prefill_ctas > 0 ? opts->prefill_ctas : kDefaultCtas;
    const int64_t kv_bytes = (int64_t)P->n_tok * Hkv * P->d * 2 * 2;  // K and V, bf16
    schedule_prefill(qts, list, items, ctas, Hkv, kv_bytes, work, cta_begin, sched);
    P->n_ctas = (int32_t)cta_begin.size() - 1;
    P->n_slots = 0;
    for (const WorkRec& w : work)
      if (w.nparts > 1) P->n_slots = std::max(P->n_slots, w.slot + 1);
    P->sched_export = sched;
    P->stats.num_work_items = (int32_t)work.size();
    P->stats.num_prefill_ctas = P->n_ctas;
    for (const WorkRec& w : work)
      if (w.nparts > 1 && w.slot == w.slot0) ++P->stats.num_split_items;
    P->stats.num_tile_pairs = (int32_t)(tile_pairs * (Hq / P->hpc));
    P->stats.num_partial_pairs = (int32_t)(partial_pairs * (Hq / P->hpc));
    int64_t bytes = 0;
    bytes += (int64_t)P->total_q * Hq * d * 2 * 2;           // q read + out write
    bytes += (int64_t)P->total_q * Hq * 4;                   // lse
    bytes += (int64_t)P->n_tok * Hkv * d * 2 * 2;            // every KV token once, K and V
    P->stats.algorithmic_bytes = bytes;
  } else {
    // decode: canonical block list and split-KV units
    std::vector<int32_t> seq_blk_begin(num_seqs + 1, 0);
    for (int32_t s = 0; s < num_seqs; ++s) {
      seq_blk_begin[s] = (int32_t)blist.size();
      for (const Unit& u : units[s]) {
        blist.push_back(u.id);
        bfill.push_back(u.n);
      }
    }
    seq_blk_begin[num_seqs] = (int32_t)blist.size();
    int64_t total_blocks = (int64_t)blist.size();
    int64_t S = opts->decode_split_blocks;
    if (S == 0) {
      int64_t target = opts->decode_min_ctas ? opts->decode_min_ctas : 16 * 148;
      S = std::max<int64_t>(8, ceil_div(total_blocks * Hkv, target));
    }
    for (int32_t s = 0; s < num_seqs; ++s) {
      int32_t nb = seq_blk_begin[s + 1] - seq_blk_begin[s];
      int32_t ns = (int32_t)ceil_div(nb, S);
      int32_t per = (int32_t)ceil_div(nb, ns);
      int32_t first = (int32_t)splits.size();
      for (int32_t i = 0; i < ns; ++i) {
        int32_t b0 = i * per, b1 = std::min(nb, b0 + per);
        if (b1 <= b0) {
          ns = i;
          break;
        }
        int32_t ntok = 0;
        for (int32_t b = b0; b < b1; ++b) ntok += bfill[seq_blk_begin[s] + b];
        splits.push_back({s, seq_blk_begin[s] + b0, b1 - b0, i, 0, first, ntok, 0});
      }
      for (size_t i = first; i < splits.size(); ++i) splits[i].nsplit = (int32_t)(splits.size() - first);
      for (size_t i = first; i < splits.size(); ++i) {
        P->split_export.push_back(s);
        P->split_export.push_back(splits[i].blk_begin - seq_blk_begin[s]);
        P->split_export.push_back(splits[i].blk_count);
      }
    }
    P->stats.num_splits = (int32_t)splits.size();
    P->stats.num_work_items = (int32_t)splits.size() * Hkv;
    int64_t bytes = 0;
    bytes += (int64_t)P->n_tok * Hkv * d * 2 * 2;                 // K and V once
    bytes += (int64_t)num_seqs * Hq * d * 2 * 2;                  // q read + out write
    bytes += (int64_t)num_seqs * Hq * 4;                          // lse
    bytes += total_blocks * 8;                                    // block id + fill
    P->stats.algorithmic_bytes = bytes;
  }
  // gather units (both modes): one per pool block, one per run of chunk rows
  {
    int32_t out_row = 0;
    for (int32_t s = 0; s < num_seqs; ++s) {
      const auto& us = units[s];
      for (size_t i = 0; i < us.size(); ++i) {
        const Unit& u = us[i];
        if (u.src == SRC_POOL) {
          gather.push_back({SRC_POOL, u.id, u.n, out_row, u.first_pos, 0, 0, 0});
          out_row += u.n;
        } else {
          size_t j = i;
          while (j + 1 < us.size() && us[j + 1].src == SRC_CHUNK && us[j + 1].id == us[j].id + 1 &&
                 (j + 1 - i) < (size_t)kTileRows)
            ++j;
          int32_t n = (int32_t)(j - i + 1);
          gather.push_back({SRC_CHUNK, u.id, n, out_row, u.first_pos, 0, 0, 0});
          out_row += n;
          i = j;
        }
      }
    }
  }

  P->n_list = (int32_t)list.size();
  P->n_work = (int32_t)work.size();
  P->n_split = (int32_t)splits.size();
  P->n_blist = (int32_t)blist.size();
  P->n_gather = (int32_t)gather.size();

  // ---- lay out the image (every section 256-byte aligned)
  DevLayout L{};
  size_t off = 0;
  auto take = [&](size_t bytes) {
    size_t o = off;
    off = align_up(off + bytes, 256);
    return o;
  };
  L.qpos = take((size_t)P->total_q * 4);
  L.qtile = take(qts.size() * sizeof(QTileRec));
  L.ktile = take(ktr.size() * sizeof(KTileRec));
  L.list = take(list.size() * 4);
  L.work = take(work.size() * sizeof(WorkRec));
  L.cta = take(cta_begin.size() * 4);
  L.split = take(splits.size() * sizeof(SplitRec));
  L.blist = take(blist.size() * 4);
  L.bfill = take(bfill.size() * 4);
  L.gather = take(gather.size() * sizeof(GatherRec));
  L.total = std::max<size_t>(off, 256);
  P->dev = L;
  P->image.assign(L.total / 4, 0);
  auto put = [&](size_t o, const void* src, size_t bytes) {
    if (bytes) std::memcpy(reinterpret_cast<char*>(P->image.data()) + o, src, bytes);
  };
  if (mode == MSA_PREFILL && P->total_q) put(L.qpos, q_pos, (size_t)P->total_q * 4);
  put(L.qtile, qts.data(), qts.size() * sizeof(QTileRec));
  put(L.ktile, ktr.data(), ktr.size() * sizeof(KTileRec));
  put(L.list, list.data(), list.size() * 4);
  put(L.work, work.data(), work.size() * sizeof(WorkRec));
  put(L.cta, cta_begin.data(), cta_begin.size() * 4);
  put(L.split, splits.data(), splits.size() * sizeof(SplitRec));
  put(L.blist, blist.data(), blist.size() * 4);
  put(L.bfill, bfill.data(), bfill.size() * 4);
  put(L.gather, gather.data(), gather.size() * sizeof(GatherRec));

  // ---- workspace layout
  WsLayout W{};
  size_t wo = 0;
  W.status = 0;
  wo = kStatusBytes;
  W.counters = wo;
  wo = align_up(wo + (size_t)num_seqs * Hq * 4, 256);
  W.part_o = wo;
  wo = align_up(wo + (size_t)P->n_split * Hq * d * 4, 256);
  W.part_lse = wo;
  wo = align_up(wo + (size_t)P->n_split * Hq * 4, 256);
  // prefill: one merge counter per (split item, head of the pair), then per partial slot
  // and head the unnormalised O (fp32, d/4 x 128 rows of float4) and (max, sum) per row
  W.pf_counters = wo;
  wo = align_up(wo + (size_t)P->n_slots * P->hpc * 4, 256);
  W.pf_part_o = wo;
  wo = align_up(wo + (size_t)P->n_slots * P->hpc * kTileRows * d * 4, 256);
  W.pf_part_ml = wo;
  wo = align_up(wo + (size_t)P->n_slots * P->hpc * kTileRows * 8, 256);
  W.total = wo;
  P->ws = W;

  *out = P;
  return MSA_OK;
}

extern "C" void msa_plan_destroy(msa_plan_t* plan) { delete plan; }

extern "C" size_t msa_plan_device_bytes(const msa_plan_t* plan) { return plan ? plan->dev.total : 0; }

extern "C" size_t msa_workspace_bytes(const msa_plan_t* plan) { return plan ? plan->ws.total : 0; }

extern "C" msa_status_t msa_plan_export(const msa_plan_t* plan, int32_t* out, size_t capacity,
                                        size_t* n) {
  if (!plan || !n) return MSA_ERR_INVALID_ARG;
  *n = plan->canon.size();
  if (!out) return MSA_OK;
  if (capacity < plan->canon.size()) return MSA_ERR_WORKSPACE;
  std::copy(plan->canon.begin(), plan->canon.end(), out);
  return MSA_OK;
}

extern "C" msa_status_t msa_plan_export_splits(const msa_plan_t* plan, int32_t* out,
                                               size_t capacity, size_t* n) {
  if (!plan || !n) return MSA_ERR_INVALID_ARG;
  *n = plan->split_export.size();
  if (!out) return MSA_OK;
  if (capacity < plan->split_export.size()) return MSA_ERR_WORKSPACE;
  std::copy(plan->split_export.begin(), plan->split_export.end(), out);
  return MSA_OK;
}

extern "C" msa_status_t msa_plan_export_schedule(const msa_plan_t* plan, int32_t* out,
                                                 size_t capacity, size_t* n) {
  if (!plan || !n) return MSA_ERR_INVALID_ARG;
  *n = plan->sched_export.size();
  if (!out) return MSA_OK;
  if (capacity < plan->sched_export.size()) return MSA_ERR_WORKSPACE;
  std::copy(plan->sched_export.begin(), plan->sched_export.end(), out);
  return MSA_OK;
}

extern "C" msa_status_t msa_plan_get_stats(const msa_plan_t* plan, msa_plan_stats_t* stats) {
  if (!plan || !stats) return MSA_ERR_INVALID_ARG;
  *stats = plan->stats;
  return MSA_OK;
}

extern "C" const char* msa_status_string(msa_status_t s) {
  switch (s) {
    case MSA_OK: return "ok";
    case MSA_ERR_INVALID_ARG: return "invalid argument";
    case MSA_ERR_UNSUPPORTED: return "unsupported configuration";
    case MSA_ERR_POS_OVERLAP: return "two KV tokens of one sequence share a position";
    case MSA_ERR_BLOCK_OOB: return "block index out of range";
    case MSA_ERR_WORKSPACE: return "buffer too small or misaligned";
    case MSA_ERR_CUDA: return "CUDA error";
    case MSA_ERR_TIMEOUT: return "device wait timed out";
    case MSA_ERR_MODE: return "plan built for the other mode";
  }
  return "unknown status";
}

extern "C" int32_t msa_version(void) { return 1; }

// ---------------------------------------------------------------- write-back placement
// Rows of one sequence's chunk are grouped by position block (pos / 16); each group goes
// to one pool block at offsets pos % 16, extending the block without a hole.  A group that
// starts part-way into its position block continues the sequence's block holding it.
extern "C" msa_status_t msa_append_plan(const int32_t* q_pos, int32_t n, const int32_t* free_blocks,
                                        int32_t n_free, const int32_t* seq_blocks, int32_t n_seq_blocks,
                                        int32_t* block_pos, int32_t* block_fill, int32_t num_pool_blocks,
                                        int32_t* dst_slot, int32_t* new_blocks, int32_t* n_new) {
  if (n < 0 || n_free < 0 || n_seq_blocks < 0 || num_pool_blocks < 0 || !n_new) return MSA_ERR_INVALID_ARG;
  if (n > 0 && (!q_pos || !dst_slot || !block_pos || !block_fill)) return MSA_ERR_INVALID_ARG;
  if (n_free > 0 && (!free_blocks || !new_blocks)) return MSA_ERR_INVALID_ARG;
  if (n_seq_blocks > 0 && !seq_blocks) return MSA_ERR_INVALID_ARG;
  *n_new = 0;
  for (int32_t i = 0; i < n; ++i)
    if (q_pos[i] < 0 || (i > 0 && q_pos[i] <= q_pos[i - 1])) return MSA_ERR_INVALID_ARG;
  // first pass: validate and place, writing nothing
  struct Group { int32_t blk, base, first_off, i0, i1; };
  std::vector<Group> groups;
  int32_t used = 0;
  for (int32_t i = 0; i < n;) {
    const int32_t base = q_pos[i] / kBlock * kBlock;
    int32_t j = i;
    while (j < n && q_pos[j] / kBlock * kBlock == base) ++j;
    int32_t blk = -1, start = 0;
    if (q_pos[i] % kBlock != 0) {
      for (int32_t k = 0; k < n_seq_blocks; ++k) {
        const int32_t b = seq_blocks[k];
        if (b < 0 || b >= num_pool_blocks) return MSA_ERR_BLOCK_OOB;
        if (block_fill[b] > 0 && block_pos[b] == base) blk = b;
      }
      if (blk < 0) return MSA_ERR_INVALID_ARG;
      start = block_fill[blk];
    } else {
      if (used >= n_free) return MSA_ERR_WORKSPACE;
      blk = free_blocks[used++];
      if (blk < 0 || blk >= num_pool_blocks) return MSA_ERR_BLOCK_OOB;
    }
    for (int32_t r = i; r < j; ++r)
      if (q_pos[r] - base != start + (r - i)) return MSA_ERR_INVALID_ARG;  // a hole
    groups.push_back({blk, base, start, i, j});
    i = j;
  }
  // second pass: write
  for (const Group& gp : groups) {
    for (int32_t r = gp.i0; r < gp.i1; ++r) dst_slot[r] = gp.blk * kBlock + (q_pos[r] - gp.base);
    block_pos[gp.blk] = gp.base;
    block_fill[gp.blk] = gp.first_off + (gp.i1 - gp.i0);
  }
  for (int32_t u = 0; u < used; ++u) new_blocks[u] = free_blocks[u];
  *n_new = used;
  return MSA_OK;
}
