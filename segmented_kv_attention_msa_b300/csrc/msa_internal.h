// Internal layout of the MSA plan: host object and the int32 records of its device
// image.  Shared by the host planner and the kernels.
#pragma once
#include <stddef.h>
#include <stdint.h>

#include "msa.h"

#ifdef __cplusplus
#include <vector>
#endif

namespace msa {

constexpr int kBlock = 16;          // tokens per pool block
constexpr int kTileRows = 128;      // tokens per KV tile / rows per query tile
constexpr int kTileBlocks = kTileRows / kBlock;
constexpr int kStatusBytes = 256;   // workspace head: status word + scheduling counters

enum { SRC_POOL = 0, SRC_CHUNK = 1, SRC_MIXED = 2 };
enum { CLS_SKIP = 0, CLS_FULL = 1, CLS_PARTIAL = 2 };

// Query tile: `nrows` consecutive chunk rows of one sequence starting at global row
// `row0`; its non-skipped KV tiles are list[list_begin, list_begin + list_count).
struct QTileRec {
  int32_t seq, row0, nrows, minpos, maxpos, list_begin, list_count, pad;
};

// KV tile: nblk units of up to 16 rows, unit i at tile rows 16*i .. 16*i + 15.  A pool
// unit is block blk[i] >= 0 whose tokens sit at positions bpos[i] + t, t < bfill[i]; a
// chunk unit (blk[i] = -(r + 1)) is chunk rows r .. r + bfill[i] - 1, the first at
// position bpos[i].  src is SRC_POOL or SRC_CHUNK when every unit is of that kind, else
// SRC_MIXED; row0 is unused.
struct KTileRec {
  int32_t src, ntok, row0, nblk, minpos, maxpos, full, pad;
  int32_t blk[kTileBlocks];
  int32_t bpos[kTileBlocks];
  int32_t bfill[kTileBlocks];
};

// One piece of prefill work: query tile `qt`, KV head `g`, query heads h0 .. h0+hpc-1,
// over entries [j0, j0 + n) of the query tile's KV-tile list.  A work item (qt, g, h0)
// whose list is cut into nparts > 1 pieces (to balance the CTAs) writes one partial
// result per piece into workspace slot `slot` (slot0 .. slot0 + nparts - 1); the piece
// that finishes last (counter `slot0`) merges them.  nparts == 1: written directly.
struct WorkRec {
  int32_t qt, g, h0, j0, n, nparts, slot0, slot;
};

// One decode split-KV unit: canonical blocks [blk_begin, blk_begin + blk_count) of the
// flat block list, part `split_idx` of `nsplit` of sequence `seq`, whose first unit
// has global index `first_split`.
struct SplitRec {
  int32_t seq, blk_begin, blk_count, split_idx, nsplit, first_split, ntok, pad;
};

// Gather unit: `n` tokens copied to output rows [out_row, out_row + n); pool block
// `id` (slots 0..n-1, positions pos0 + t) or chunk rows id .. id+n-1.
struct GatherRec {
  int32_t src, id, n, out_row, pos0, pad0, pad1, pad2;
};

// Byte offsets of each section within the device image.
struct DevLayout {
  size_t qpos, qtile, ktile, list, work, cta, split, blist, bfill, gather, total;
};

// Byte offsets within the workspace.
struct WsLayout {
  size_t status, counters, part_o, part_lse, pf_counters, pf_part_o, pf_part_ml, total;
};

}  // namespace msa

#ifdef __cplusplus
struct msa_plan {
  msa_mode_t mode;
  int32_t num_seqs, Hq, Hkv, d, G, hpc, num_pool_blocks;
  int32_t total_q, n_tok, n_qt, n_kt, n_list, n_work, n_split, n_blist, n_gather;
  int32_t n_ctas, n_slots;          // prefill: CTAs of the launch, partial-result slots
  std::vector<int32_t> canon;       // canonical export
  std::vector<int32_t> split_export;
  std::vector<int32_t> sched_export;
  std::vector<int32_t> image;       // device image (int32 words)
  msa::DevLayout dev;
  msa::WsLayout ws;
  msa_plan_stats_t stats;
};
#endif
