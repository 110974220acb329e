// MSA prefill (TTFT path) for sm_103a.
//
// What it computes (paper "Multi-Segment Attention: Enabling Efficient KV-Cache
// Management for Faster Large Language Model Serving": Eq. 1, section 4.1, Fig. 5,
// abstract): every chunk token -- a recomputed evicted-block token or a new token, at
// its original position -- attends with softmax(q k^T * scale) over the union of
// disjoint KV regions: cached pool segments plus the chunk's own fresh K/V, masked
// causally by original position.  One launch covers all sequences; outputs O (bf16)
// and the natural-log LSE (fp32).
//
// How (one persistent CTA per SM, warp-specialised, 12 warps in 3 warpgroups):
//  * warp 10 (K producer): TMA loads of the Q tiles (two query heads sharing one KV head,
//    128 chunk rows each; the next work item's Q is prefetched into L2 when an item
//    starts) and of each K tile into a 3-deep ring.  A KV tile is 8 units of
//    at most 16 keys, each a paged pool block or a run of chunk rows, loaded as one
//    16-row box per unit and 64-column slab; pool blocks and chunk rows may share a
//    tile.  Missing units of a short tile are loaded from an out-of-range row and arrive
//    as zeros.
//  * warp 11 (V producer): the V tiles into a 2-deep ring, and for each tile a mask
//    record (per unit: its source, the position or chunk row of its first key and its
//    number of valid keys) used by partial tiles.  A pool block holding fewer than 16
//    keys may carry anything (NaN included) in its unused slots: those V rows are zeroed
//    in shared memory before the slot is marked full.
//  * warps 8 and 9 (MMA issuers, one thread each, warp 8 for head 0, warp 9 for head 1):
//    tcgen05.mma kind::f16.  S_t = Q_t K^T (both operands in 128-byte-swizzled shared
//    memory, accumulator in TMEM), then O_t += P_t V with P_t read from TMEM (it
//    overwrites S_t as bf16) and V as an MN-major shared-memory operand.  The two heads
//    ping-pong: while one softmax group works on S_0, the tensor core runs the other
//    head's GEMMs.  The issuers pass a turn between them so that the heads' blocks
//    alternate; each waits for its own head's P while the other issues.
//  * warps 0-3 / 4-7 (softmax groups, one per head): each thread owns one query row in
//    TMEM (tcgen05.ld 32x32b), masks partial tiles by a per-unit prefix cut, takes the
//    exponentials against the running reference max (re-doing the pass against the
//    tile's exact max only if the tile's sum of exponentials passes 2^16), writes P as
//    bf16 back to TMEM, and at the end normalises O and stores bf16 rows and the LSE.
//  * KV tiles whose smallest position exceeds the query tile's largest are never
//    loaded (the planner leaves them out of the work item's list); tiles that every
//    query row sees fully skip the mask.
//  * Registers: the softmax warpgroups hold a full 128-column row of S and run with 216
//    registers a thread; the third warpgroup (MMA issuers, producers) gives its share
//    back (setmaxnreg).
// TMEM: 512 columns = S_0 | S_1 | O_0 | O_1 (128 columns each).
#include <cuda.h>
#include <cuda_runtime.h>

#include <type_traits>

#include "msa_device.cuh"
#include "msa_kernels.h"
#include "msa_tmap.h"

namespace msa {

// 12 warps = 3 full warpgroups (setmaxnreg acts on whole warpgroups).
// At launch every thread gets kPfLaunchRegs registers (65536 / 384, rounded down to 8);
// the split below must fit in that total, and the host refuses to launch a build whose
// kernel was given fewer registers.
constexpr int kPfThreads = 384;
constexpr int kPfLaunchRegs = 168;
constexpr int kPfRegsSoftmax = 216;    // after setmaxnreg, warpgroups 0-1
constexpr int kPfRegsOther = 64;       // after setmaxnreg, warpgroup 2
static_assert(2 * 128 * kPfRegsSoftmax + 128 * kPfRegsOther <= kPfThreads * kPfLaunchRegs, "register split");
constexpr int kKStages = 3;            // K tiles in flight (a slot frees once its QK^T is done)
constexpr int kVStages = 2;            // V tiles (a slot frees once its PV is done)
constexpr int kSlabBytes = 128 * 128;  // 128 rows x 128 bytes (64 bf16)
constexpr int kMaskInts = 24;          // mask record: base[8], nvalid[8], src[8]

// Shared memory: small items first (barriers, mask records), then the operand tiles on
// a 1024-byte boundary (the 128-byte swizzle pattern repeats every 1024 bytes).
template <int D>
struct PfLayout {
  static constexpr int kTileBytes = 128 * D * 2;
  static constexpr int kNumBars = 31;
  static constexpr int kBar = 0;
  static constexpr int kMisc = (kBar + kNumBars * 8 + 15) / 16 * 16;  // TMEM base address, flags
  static constexpr int kMask = kMisc + 16;                             // int32 [kVStages][kMaskInts]
  static constexpr int kSmall = kMask + kVStages * kMaskInts * 4;
  static constexpr int kQ = 0;                         // offsets from the aligned tile base
  static constexpr int kK = kQ + 2 * kTileBytes;
  static constexpr int kV = kK + kKStages * kTileBytes;
  static constexpr int kTiles = kV + kVStages * kTileBytes;
  static constexpr int kBytes = kSmall + 1023 + kTiles;
};
static_assert(PfLayout<128>::kBytes <= 232448, "prefill shared memory exceeds 227 KB");
static_assert(PfLayout<128>::kMask % 16 == 0 && PfLayout<128>::kMisc % 16 == 0, "16-byte alignment");

// Bounded wait that also gives up as soon as another role of this CTA gave up.
__device__ __forceinline__ bool pf_wait(uint64_t* bar, uint32_t parity, const PrefillParams& p,
                                        volatile int* abort_flag) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (;;) {
#pragma unroll 1
    for (int i = 0; i < 32; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    if (global_timer_ns() - t0 > p.wait_ns) {
      set_status(p.status, MSA_ERR_TIMEOUT);
      *abort_flag = 1;
      return false;
    }
  }
}

// The same, taken by a whole warp: every lane leaves together, so no warp-collective
// tcgen05 instruction ever runs on a partial warp.
__device__ __forceinline__ bool pf_wait_warp(uint64_t* bar, uint32_t parity, const PrefillParams& p,
                                             volatile int* abort_flag) {
  const bool ok = pf_wait(bar, parity, p, abort_flag);
  return __all_sync(0xffffffffu, ok);
}

// d = a * b + c on two fp32 lanes at once (one packed FMA).
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
  float2 d;
  asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\tmov.b64 ra, {%2,%3};\n\tmov.b64 rb, {%4,%5};\n\t"
      "mov.b64 rc, {%6,%7};\n\tfma.rn.f32x2 rd, ra, rb, rc;\n\tmov.b64 {%0,%1}, rd;\n\t}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
  return d;
}
__device__ __forceinline__ float2 fadd2(float2 a, float2 b) {
  float2 d;
  asm("{\n\t.reg .b64 ra, rb, rd;\n\tmov.b64 ra, {%2,%3};\n\tmov.b64 rb, {%4,%5};\n\t"
      "add.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0,%1}, rd;\n\t}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return d;
}

// One query row's D accumulator columns from TMEM: all loads issued, then one wait.
template <int D>
__device__ __forceinline__ void tmem_ld_row(uint32_t taddr, uint32_t (&v)[D]) {
#pragma unroll
  for (int c = 0; c < D; c += 32) tmem_ld_x32(taddr + c, *reinterpret_cast<uint32_t(*)[32]>(&v[c]));
  tmem_wait_ld();
}

// A KV tile record spread over a warp: lane i holds word i of the 32-word record.
// Fields are read with warp shuffles, so every lane must take part.
struct TileRec {
  int v;
  __device__ __forceinline__ int get(int i) const { return __shfl_sync(0xffffffffu, v, i); }
};
__device__ __forceinline__ TileRec load_tile_rec(const PrefillParams& p, const int* lst, int j, int lane) {
  const int e = __ldg(lst + j);
  int ki = e & 0x7fffffff;
  if (!MSA_DCHECK(ki < p.n_kt, p.status)) ki = 0;
  const int* rec = reinterpret_cast<const int*>(p.kt + ki);
  return TileRec{__ldg(rec + lane)};
}

// MSA_DEBUG build: a work record must point inside the plan (query tile, list range, heads)
// before any role reads through it; a bad one sets MSA_ERR_BLOCK_OOB and the CTA gives up.
__device__ __forceinline__ bool work_ok(const PrefillParams& p, const WorkRec& wk) {
#ifdef MSA_DEBUG
  bool ok = wk.qt >= 0 && wk.qt < p.n_qt && wk.g >= 0 && wk.g < p.Hkv && wk.h0 >= 0 && wk.h0 + p.hpc <= p.Hq &&
            wk.j0 >= 0 && wk.n >= 0 && p.hpc >= 1 && p.hpc <= 2;
  if (ok) {
    const QTileRec qt = p.qt[wk.qt];
    ok = qt.list_begin >= 0 && qt.list_begin + wk.j0 + wk.n <= p.n_list && qt.row0 >= 0 && qt.nrows >= 0 &&
         qt.row0 + qt.nrows <= p.total_q;
  }
  return MSA_DCHECK(ok, p.status);
#else
  (void)p;
  (void)wk;
  return true;
#endif
}

// Issue the TMA loads of one K or V tile (whole warp calls; lane 0 posts the byte
// count, lane i < 8 loads the tile's unit i as one 16-row box: a paged pool block
// (blk >= 0) or 16 chunk rows starting at row -blk-1 (blk < 0)).  A unit past the
// tile's last one reads rows out of the pool map's range and arrives as zeros.
template <int D>
__device__ __forceinline__ void issue_kv_tile(const TileRec& rec, uint8_t* dst, uint64_t* bar,
                                              const CUtensorMap* tm_chunk, const CUtensorMap* tm_pool,
                                              int g, const PrefillParams& p, int lane) {
  constexpr int kSlabs = D / 64;
  const int nblk = rec.get(3);
  const int blk = rec.get(8 + (lane & 7));
  if (lane == 0) mbar_arrive_expect_tx(bar, 128 * D * 2);
  __syncwarp();
  if (lane < kTileBlocks) {
    uint8_t* d = dst + lane * 2048;
    bool chunk = false;
    int y = p.pool_rows;  // past the pool: the box arrives as zeros
    if (lane < nblk && MSA_DCHECK(blk < 0 ? -blk - 1 < p.total_q : blk < p.num_pool_blocks, p.status)) {
      chunk = blk < 0;
      if (!chunk) y = (blk * p.Hkv + g) * kBlock;
    }
    if (chunk) {
      for (int s = 0; s < kSlabs; ++s) tma_load_2d(d + s * kSlabBytes, tm_chunk, bar, g * D + s * 64, -blk - 1);
    } else {
      for (int s = 0; s < kSlabs; ++s) tma_load_2d(d + s * kSlabBytes, tm_pool, bar, s * 64, y);
    }
  }
}

template <int D>
__global__ void __launch_bounds__(kPfThreads, 1)
    msa_prefill_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_kc,
                       const __grid_constant__ CUtensorMap tm_vc, const __grid_constant__ CUtensorMap tm_kp,
                       const __grid_constant__ CUtensorMap tm_vp, const PrefillParams p) {
  using L = PfLayout<D>;
  constexpr int kSlabs = D / 64;
  constexpr uint32_t kIdescQK = idesc_bf16_f32(128, 128, false, false);
  constexpr uint32_t kIdescPV = idesc_bf16_f32(128, D, false, true);
  constexpr float kLn2 = 0.69314718055994531f;

  extern __shared__ uint8_t smem_raw[];
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem_raw + L::kBar);
  uint64_t* q_full = bars + 0;
  uint64_t* q_empty = bars + 1;
  uint64_t* k_full = bars + 2;     // [3]
  uint64_t* k_empty = bars + 5;    // [3]
  uint64_t* v_full = bars + 8;     // [2]
  uint64_t* v_empty = bars + 10;   // [2]
  uint64_t* m_full = bars + 12;    // [2] mask record of the tile held in V slot s
  uint64_t* s_full = bars + 14;    // [2] per head
  uint64_t* p_full = bars + 16;    // [2]
  uint64_t* o_full = bars + 18;    // [2]
  uint64_t* o_free = bars + 20;    // [2]
  uint64_t* drain = bars + 22;    // [2] one per MMA-issuing thread
  uint64_t* ep_bar = bars + 24;    // [2] split pieces: the head's 128 threads stored their partial
  uint64_t* ep_flag = bars + 26;   // [2] split pieces: merge counter read, last_flag[t] valid
  uint64_t* v_land = bars + 28;    // V tiles with unused pool slots: the copy landed (then fixed up)
  uint64_t* turn = bars + 29;      // [2] head t's issuer may start its next block
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem_raw + L::kMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem_raw + L::kMisc + 4);
  volatile int* last_flag = reinterpret_cast<volatile int*>(smem_raw + L::kMisc + 8);  // [2]
  int32_t* sMask = reinterpret_cast<int32_t*>(smem_raw + L::kMask);
  uint8_t* tiles = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw + L::kSmall) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = tiles + L::kQ;
  uint8_t* sK = tiles + L::kK;
  uint8_t* sV = tiles + L::kV;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int cta_w0 = __ldg(p.cta_begin + blockIdx.x), cta_w1 = __ldg(p.cta_begin + blockIdx.x + 1);

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    // Q, K and V slots are handed back once per head: each head's GEMMs come from
    // their own issuing thread, and one head's completion says nothing of the other's
    mbar_init(q_empty, p.hpc);
    for (int s = 0; s < kKStages; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&k_empty[s], p.hpc);
    }
    for (int s = 0; s < kVStages; ++s) {
      mbar_init(&v_full[s], 1);
      mbar_init(&v_empty[s], p.hpc);
      mbar_init(&m_full[s], 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(&s_full[t], 1);
      mbar_init(&p_full[t], 128);
      mbar_init(&o_full[t], 1);
      mbar_init(&o_free[t], 128);
      mbar_init(&ep_bar[t], 128);
      mbar_init(&ep_flag[t], 1);
    }
    mbar_init(&drain[0], 1);
    mbar_init(&drain[1], 1);
    mbar_init(v_land, 1);
    mbar_init(&turn[0], 1);
    mbar_init(&turn[1], 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 8) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  // The two register regions never merge again: each ends with its own barrier and
  // return, so the compiler can give each the register budget of its warpgroups.
  if (warp >= 8) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kPfRegsOther));
  if (warp == 10) {
    // ------------------------------------------------------------ K producer (and Q)
    int kit = 0, wi = 0;  // K tiles and work items issued
    int last_k[kKStages] = {-1, -1, -1};
    int last_wi = -1;
    for (int w = cta_w0; w < cta_w1; ++w) {
      const WorkRec wk = p.work[w];
      if (!work_ok(p, wk)) {
        *abort_flag = 1;
        goto kprod_done;
      }
      const QTileRec qt = p.qt[wk.qt];
      const int n = wk.n;
      if (n == 0) continue;
      const int* lst = p.list + qt.list_begin + wk.j0;
      TileRec cur = load_tile_rec(p, lst, 0, lane);
      if (!pf_wait_warp(q_empty, (wi & 1) ^ 1, p, abort_flag)) goto kprod_done;
      if (lane == 0) {
        mbar_arrive_expect_tx(q_full, p.hpc * L::kTileBytes);
        for (int t = 0; t < p.hpc; ++t)
          for (int s = 0; s < kSlabs; ++s)
            tma_load_2d(sQ + t * L::kTileBytes + s * kSlabBytes, &tm_q, q_full, (wk.h0 + t) * D + s * 64, qt.row0);
        // The next item's Q can load only once this item's last QK^T is done, and then
        // waits behind the K/V tiles in flight: bring it into L2 now, while this item runs.
        if (w + 1 < cta_w1) {
          const WorkRec wn = p.work[w + 1];
          if (wn.n > 0 && work_ok(p, wn)) {
            const int row0n = p.qt[wn.qt].row0;
            for (int t = 0; t < p.hpc; ++t)
              for (int s = 0; s < kSlabs; ++s) tma_prefetch_2d(&tm_q, (wn.h0 + t) * D + s * 64, row0n);
          }
        }
      }
      last_wi = wi;
      for (int j = 0; j < n; ++j) {
        TileRec nxt = cur;
        if (j + 1 < n) nxt = load_tile_rec(p, lst, j + 1, lane);
        const int ks = kit % kKStages;
        if (!pf_wait_warp(&k_empty[ks], ((kit / kKStages) & 1) ^ 1, p, abort_flag)) goto kprod_done;
        // (test hook: one CTA may leave out one K tile, so that the wait for it runs out)
        if (!(kit == p.drop_k && (int)blockIdx.x == p.drop_cta)) {
          issue_kv_tile<D>(cur, sK + ks * L::kTileBytes, &k_full[ks], &tm_kc, &tm_kp, wk.g, p, lane);
          last_k[ks] = kit;
        }
        ++kit;
        cur = nxt;
      }
      ++wi;
    }
  kprod_done:
    // every copy this warp started must land before the CTA may exit
    for (int s = 0; s < kKStages; ++s)
      if (last_k[s] >= 0) mbar_wait(&k_full[s], (last_k[s] / kKStages) & 1, 1000000000ull);
    if (last_wi >= 0) mbar_wait(q_full, last_wi & 1, 1000000000ull);
  } else if (warp == 11) {
    // ------------------------------------------------------------ V producer (and mask records)
    int vit = 0;
    int last_v[kVStages] = {-1, -1};
    int nfix = 0;               // V tiles whose copy landed on v_land
    bool land_pending = false;  // a copy on v_land has not been seen to land
    for (int w = cta_w0; w < cta_w1; ++w) {
      const WorkRec wk = p.work[w];
      if (!work_ok(p, wk)) {
        *abort_flag = 1;
        goto vprod_done;
      }
      const QTileRec qt = p.qt[wk.qt];
      const int n = wk.n;
      if (n == 0) continue;
      const int* lst = p.list + qt.list_begin + wk.j0;
      TileRec cur = load_tile_rec(p, lst, 0, lane);
      for (int j = 0; j < n; ++j) {
        TileRec nxt = cur;
        if (j + 1 < n) nxt = load_tile_rec(p, lst, j + 1, lane);
        const int vs = vit % kVStages;
        if (!pf_wait_warp(&v_empty[vs], ((vit / kVStages) & 1) ^ 1, p, abort_flag)) goto vprod_done;
        {
          // Pool units with unused slots (fill < 16): those slots may hold anything, NaN
          // included, and P.V spans the unit's 16 rows.  A masked key has P = 0, but
          // 0 x NaN is NaN, so their V rows are zeroed in shared memory before the MMA
          // reads the tile: the copy lands on v_land, this warp clears the rows, and only
          // then marks the slot full.  (Their K rows need nothing: the mask replaces
          // those logits by -inf.)
          uint8_t* vdst = sV + vs * L::kTileBytes;
          const int ui = lane & 7;
          const int u_n = cur.get(3), u_blk = cur.get(8 + ui), u_fill = cur.get(24 + ui);  // all lanes
          const bool fix_u = lane < kTileBlocks && ui < u_n && u_blk >= 0 && u_fill < kBlock;
          const unsigned fixmask = __ballot_sync(0xffffffffu, fix_u);
          if (fixmask == 0) {
            issue_kv_tile<D>(cur, vdst, &v_full[vs], &tm_vc, &tm_vp, wk.g, p, lane);
          } else {
            issue_kv_tile<D>(cur, vdst, v_land, &tm_vc, &tm_vp, wk.g, p, lane);
            land_pending = true;
            if (!pf_wait_warp(v_land, nfix & 1, p, abort_flag)) goto vprod_done;
            land_pending = false;
            ++nfix;
            for (int i = 0; i < kTileBlocks; ++i) {
              const int f = cur.get(24 + i);  // every lane takes part in the shuffle
              if (!((fixmask >> i) & 1)) continue;
              for (int s = 0; s < kSlabs; ++s) {
                uint4* z = reinterpret_cast<uint4*>(vdst + s * kSlabBytes + i * (kBlock * 128) + f * 128);
                for (int c = lane; c < (kBlock - f) * 8; c += 32) z[c] = make_uint4(0u, 0u, 0u, 0u);
              }
            }
            fence_proxy_async_smem();  // the zeroed rows, before the tensor core reads the tile
            __syncwarp();
            if (lane == 0) mbar_arrive(&v_full[vs]);
          }
        }
        last_v[vs] = vit;
        // mask record: per 16-row unit i, the first key's position (pool unit) or chunk
        // row (chunk unit), its number of valid keys and its source; chunk units are
        // compared by row index (chunk rows of one sequence are in position order)
        {
          const int nblk = cur.get(3);
          const int i = lane & 7;
          const int blk = cur.get(8 + i), bp = cur.get(16 + i), bf = cur.get(24 + i);
          const bool chunk = i < nblk && blk < 0;
          int val = 0;
          if (lane < 8) {
            val = chunk ? -blk - 1 : bp;
          } else if (lane < 16) {
            val = i < nblk ? bf : 0;
          } else if (lane < 24) {
            val = chunk ? SRC_CHUNK : SRC_POOL;
          }
          if (lane < kMaskInts) sMask[vs * kMaskInts + lane] = val;
          __syncwarp();
          if (lane == 0) mbar_arrive(&m_full[vs]);
        }
        ++vit;
        cur = nxt;
      }
    }
  vprod_done:
    for (int s = 0; s < kVStages; ++s)
      if (last_v[s] >= 0) mbar_wait(&v_full[s], (last_v[s] / kVStages) & 1, 1000000000ull);
    if (land_pending) mbar_wait(v_land, nfix & 1, 1000000000ull);
  } else if (warp - 8 < p.hpc) {
    // ------------------------------------------------------------ MMA issuers
    // Warp 8 issues head 0's GEMMs, warp 9 head 1's.  One thread cannot issue a
    // 128x128x16 MMA as fast as the tensor pipe retires it once a softmax warp shares
    // its scheduler, and a head's next block waits on its own P only: with a thread per
    // head, neither head's block queues behind the other's.
    const int t = warp - 8;
    if (lane == 0) {
      // one descriptor per operand ring, built once.  Slot and k-step offsets add to the
      // start-address field in the low word (addresses stay below 2^18, so the field never
      // carries); the high word (stride, version, swizzle) is the same for Q, K and V.
      // Plain arithmetic, not arrays indexed by slot: those would live in local memory.
      constexpr uint32_t kTileDesc = (uint32_t)(L::kTileBytes >> 4);
      const uint64_t qd0 = smem_desc_sw128(smem_u32(sQ), 16, 1024);
      const uint32_t desc_hi = (uint32_t)(qd0 >> 32);
      const uint32_t q_lo = (uint32_t)qd0 + (uint32_t)t * kTileDesc;
      const uint32_t k_lo = (uint32_t)smem_desc_sw128(smem_u32(sK), 16, 1024);
      const uint32_t v_lo = (uint32_t)smem_desc_sw128(smem_u32(sV), kSlabBytes, 1024);
      const uint32_t tS = tmem + t * 128, tO = tmem + 256 + t * 128;
      auto desc = [&](uint32_t lo) { return ((uint64_t)desc_hi << 32) | lo; };
      int it = 0, wi = 0, ks = 0, vs = 0;
      uint32_t kph = 0, vph = 0;  // phase bits of the K and V rings at (ks, vs)
      // The two heads' blocks take turns (0, 1, 0, 1, ...): left free, both issuers start
      // together, their GEMMs share the pipe and their softmax groups the MUFU, and the
      // two heads stay in step.  Block nb of head 1 follows block nb of head 0; block nb
      // of head 0 follows block nb - 1 of head 1.
      int nb = 0;
      auto my_turn = [&]() {
        if (p.hpc == 1 || (t == 0 && nb == 0)) return true;
        return pf_wait(&turn[t], (uint32_t)((t == 0 ? nb - 1 : nb) & 1), p, abort_flag);
      };
      auto pass_turn = [&]() {
        if (p.hpc == 2) mbar_arrive(&turn[1 - t]);
        ++nb;
      };
      // (the empty asm keeps the compiler from hoisting all 16 descriptors of a block out
      // of the loops: this warpgroup runs with 64 registers)
      auto issue_qk = [&](int kslot) {
        uint32_t qd = q_lo, kd = k_lo + (uint32_t)kslot * kTileDesc;
        asm volatile("" : "+r"(qd), "+r"(kd));
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (uint32_t)((((kk >> 2) * kSlabBytes) + (kk & 3) * 32) >> 4);
          umma_ss(tS, desc(qd + off), desc(kd + off), kIdescQK, kk > 0);
        }
      };
      auto issue_pv = [&](int vslot, bool acc) {
        uint32_t vd = v_lo + (uint32_t)vslot * kTileDesc;
        asm volatile("" : "+r"(vd));
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          umma_ts(tO, tS + kk * 8, desc(vd + (uint32_t)((kk * 2048) >> 4)), kIdescPV, (acc || kk > 0) ? 1u : 0u);
      };
      [&] {
        for (int w = cta_w0; w < cta_w1; ++w) {
          if (!work_ok(p, p.work[w])) {
            *abort_flag = 1;
            return;
          }
          const int n = p.work[w].n;
          if (n == 0) continue;
          if (!pf_wait(q_full, wi & 1, p, abort_flag)) return;
          if (!pf_wait(&k_full[ks], kph, p, abort_flag)) return;
          if (!my_turn()) return;
          tc_fence_after();
          issue_qk(ks);
          umma_commit(&s_full[t]);
          pass_turn();
          if (n == 1) umma_commit(q_empty);
          if (++ks == kKStages) { ks = 0; kph ^= 1; }
          for (int j = 0; j < n; ++j) {
            const bool has_next = j + 1 < n;
            if (!pf_wait(&p_full[t], (it + j) & 1, p, abort_flag)) return;
            if (!pf_wait(&v_full[vs], vph, p, abort_flag)) return;
            if (has_next && !pf_wait(&k_full[ks], kph, p, abort_flag)) return;
            if (j == 0 && !pf_wait(&o_free[t], (wi & 1) ^ 1, p, abort_flag)) return;
            if (!my_turn()) return;
            tc_fence_after();
            issue_pv(vs, j > 0);
            if (has_next) {
              issue_qk(ks);
              umma_commit(&s_full[t]);
              if (++ks == kKStages) { ks = 0; kph ^= 1; }
            } else {
              umma_commit(&o_full[t]);
            }
            pass_turn();
            // this head's K and V slots are handed back by its softmax group once it sees
            // the S (or O) that these GEMMs produced: that commit covers every MMA above
            if (j + 2 == n) umma_commit(q_empty);
            if (++vs == kVStages) { vs = 0; vph ^= 1; }
          }
          it += n;
          ++wi;
        }
      }();
      // every exit (done or aborted) waits for its MMAs in flight before TMEM is freed
      umma_commit(&drain[t]);
      mbar_wait(&drain[t], 0, 1000000000ull);
    }
    __syncwarp();
  }
    tc_fence_before();
    __syncthreads();
    if (warp == 8) {
      tc_fence_after();
      tmem_dealloc(tmem, 512);
    }
    return;
  }
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kPfRegsSoftmax));
  {
    // ------------------------------------------------------------ softmax groups
    const int t = warp >> 2, wq = warp & 3;
    const int r = wq * 32 + lane;
    const uint32_t lane_base = (uint32_t)(wq * 32) << 16;
    const uint32_t tS = tmem + lane_base + t * 128;
    const uint32_t tO = tmem + lane_base + 256 + t * 128;
    const float2 scale2 = make_float2(p.scale_log2, p.scale_log2);
    int it = 0, wi = 0, se = 0;  // tiles, pieces and split pieces done
    for (int w = cta_w0; w < cta_w1; ++w) {
      const WorkRec wk = p.work[w];
      if (!work_ok(p, wk)) {
        *abort_flag = 1;
        goto softmax_done;
      }
      const QTileRec qt = p.qt[wk.qt];
      const int n = wk.n;
      if (n == 0) {
        // a query tile that sees no key (a plan whose chunk rows are queries only): O = 0,
        // LSE = -inf; no other role takes part
        if (t < p.hpc && r < qt.nrows) {
          uint4* dst = reinterpret_cast<uint4*>(p.out + ((size_t)(qt.row0 + r) * p.Hq + wk.h0 + t) * D);
#pragma unroll
          for (int c = 0; c < D / 8; ++c) dst[c] = make_uint4(0u, 0u, 0u, 0u);
          p.lse[(size_t)(qt.row0 + r) * p.Hq + wk.h0 + t] = -INFINITY;
        }
        continue;
      }
      if (t >= p.hpc) {
        it += n;
        ++wi;
        continue;
      }
      const int h = wk.h0 + t;
      const bool valid = r < qt.nrows;
      // rows past the tile's end see every key (their values are finite and never stored)
      const int qp = valid ? __ldg(p.qpos + qt.row0 + r) : 0x7fffffff;
      const int qrow = valid ? qt.row0 + r : 0x7fffffff;
      float m_used = -INFINITY, l = 0.f;
      const int* lst = p.list + qt.list_begin + wk.j0;
      int e_next = __ldg(lst);
      for (int j = 0; j < n; ++j, ++it) {
        const int vs = it % kVStages;
        const bool partial = e_next < 0;
        if (j + 1 < n) e_next = __ldg(lst + j + 1);
        if (!pf_wait_warp(&s_full[t], it & 1, p, abort_flag)) goto softmax_done;
        if (lane == 0 && wq == 0) {
          // S of this tile for this head is done, and so is every MMA its issuing thread
          // started before it: for this head, this tile's K slot and the previous tile's
          // V slot are free
          mbar_arrive(&k_empty[it % kKStages]);
          if (j > 0) mbar_arrive(&v_empty[(it - 1) % kVStages]);
        }
        tc_fence_after();
        uint32_t s[128];
        tmem_ld_x64(tS + 0, *reinterpret_cast<uint32_t(*)[64]>(&s[0]));
        tmem_ld_x64(tS + 64, *reinterpret_cast<uint32_t(*)[64]>(&s[64]));
        tmem_wait_ld();
        if (partial) {
          // key (block b, slot u) is visible iff u < cut_b, cut_b = clamp(ref - base_b + 1, 0, nvalid_b)
          if (!pf_wait_warp(&m_full[vs], (it / kVStages) & 1, p, abort_flag)) goto softmax_done;
          const int4* mr = reinterpret_cast<const int4*>(sMask + vs * kMaskInts);
          const int4 b0 = mr[0], b1 = mr[1], f0 = mr[2], f1 = mr[3], s0 = mr[4], s1 = mr[5];
          const int base[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
          const int nv[8] = {f0.x, f0.y, f0.z, f0.w, f1.x, f1.y, f1.z, f1.w};
          const int sr[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
#pragma unroll
          for (int b = 0; b < 8; ++b) {
            // ref - base + 1 cannot overflow: a row past the end uses INT_MAX only against
            // bases >= 0, and then the cut is the unit's valid count
            const int ref = sr[b] == SRC_CHUNK ? qrow : qp;
            const int d = ref - base[b];
            const int cut = d < 0 ? 0 : (d >= nv[b] ? nv[b] : d + 1);
#pragma unroll
            for (int u = 0; u < 16; ++u)
              if (u >= cut) s[16 * b + u] = __float_as_uint(-INFINITY);
          }
        }
        // Exponents are taken against the reference max m_used of the earlier tiles.  The
        // result is exact for any reference (O and l share it); the reference only has to
        // keep the exponentials far from overflow.  So no max is tracked per element: only
        // if the tile's sum of exponentials exceeds 2^16 (some exponential above 2^16, or
        // not finite) is the tile's exact max found and the pass redone against it, with
        // O and l rescaled.  The first tile of a piece (reference still -inf) finds its
        // max first.
        float factor = 1.f;
        bool resc = false;
        const bool spec = !__any_sync(0xffffffffu, m_used == -INFINITY);
        if (!spec) {
          float m4[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) m4[i] = fmax3(__uint_as_float(s[i]), __uint_as_float(s[4 + i]), -INFINITY);
#pragma unroll
          for (int c = 8; c < 128; c += 8)
#pragma unroll
            for (int i = 0; i < 4; ++i)
              m4[i] = fmax3(m4[i], __uint_as_float(s[c + i]), __uint_as_float(s[c + 4 + i]));
          const float m_cand = fmax3(m4[0], m4[1], fmaxf(m4[2], m4[3])) * p.scale_log2;
          if (m_cand > m_used + 8.f) {
            resc = m_used != -INFINITY;
            if (resc) factor = fast_exp2(m_used - m_cand);
            l *= factor;
            m_used = m_cand;
          }
        }
        float2 acc[4];
        float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll 1
        for (int pass = 0; pass < 2; ++pass) {
          const float ms = (m_used == -INFINITY) ? 0.f : m_used;
          const float2 nms2 = make_float2(-ms, -ms);
#pragma unroll
          for (int i = 0; i < 4; ++i) acc[i] = make_float2(0.f, 0.f);
          uint32_t pk[64];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
#pragma unroll
            for (int c = 0; c < 16; ++c) {
              const int e = q * 32 + 2 * c;
              const float2 x = ffma2(make_float2(__uint_as_float(s[e]), __uint_as_float(s[e + 1])), scale2, nms2);
              const float2 pe = make_float2(fast_exp2(x.x), fast_exp2(x.y));
              acc[c & 3] = fadd2(acc[c & 3], pe);
              pk[q * 16 + c] = pack_bf16x2(pe.x, pe.y);
            }
          }
          // P leaves in two x32 stores after the whole pass: measured faster than a store
          // per 32 exponentials, which interleaves store issue with the exponential chain
          tmem_st_x32(tS, *reinterpret_cast<uint32_t(*)[32]>(&pk[0]));
          tmem_st_x32(tS + 32, *reinterpret_cast<uint32_t(*)[32]>(&pk[32]));
          if (pass == 1 || !spec) break;
          // the tile's sum of exponentials bounds its largest one: above 2^16 (or not
          // finite) the tile is redone against its exact max
          const float2 at = fadd2(fadd2(acc[0], acc[1]), fadd2(acc[2], acc[3]));
          const bool redo = !(at.x + at.y <= 65536.f);
          if (!__any_sync(0xffffffffu, redo)) break;
          if (redo) {
#pragma unroll
            for (int i = 0; i < 4; ++i) m4[i] = fmax3(__uint_as_float(s[i]), __uint_as_float(s[4 + i]), -INFINITY);
#pragma unroll
            for (int c = 8; c < 128; c += 8)
#pragma unroll
              for (int i = 0; i < 4; ++i)
                m4[i] = fmax3(m4[i], __uint_as_float(s[c + i]), __uint_as_float(s[c + 4 + i]));
            const float m_cand = fmax3(m4[0], m4[1], fmaxf(m4[2], m4[3])) * p.scale_log2;
            factor = fast_exp2(m_used - m_cand);
            l *= factor;
            m_used = m_cand;
            resc = true;
          }
          tmem_wait_st();  // the second pass overwrites these P columns
        }
        if (__any_sync(0xffffffffu, resc)) {
#pragma unroll 1
          for (int c = 0; c < D; c += 32) {
            uint32_t ov[32];
            tmem_ld_x32(tO + c, ov);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 32; ++i) ov[i] = __float_as_uint(__uint_as_float(ov[i]) * factor);
            tmem_st_x32(tO + c, ov);
          }
        }
        const float2 a = fadd2(fadd2(acc[0], acc[1]), fadd2(acc[2], acc[3]));
        l += a.x + a.y;
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(&p_full[t]);
      }
      // epilogue: O / l -> bf16, LSE = ln 2 * (m + log2 l)
      if (!pf_wait_warp(&o_full[t], wi & 1, p, abort_flag)) goto softmax_done;
      if (lane == 0 && wq == 0) mbar_arrive(&v_empty[(it - 1) % kVStages]);  // last tile's V
      tc_fence_after();
      if (wk.nparts == 1) {
        // O leaves TMEM first, every column in flight at once, and the O columns are handed
        // back before the rows are normalised and stored: this head's issuer may start the
        // next piece's P.V meanwhile
        uint32_t ov[D];
        tmem_ld_row<D>(tO, ov);
        tc_fence_before();
        mbar_arrive(&o_free[t]);
        const float inv = l > 0.f ? 1.f / l : 0.f;
        if (valid) {
          // 32-byte stores (rows start on 256-byte boundaries)
          __nv_bfloat16* dst = p.out + ((size_t)(qt.row0 + r) * p.Hq + h) * D;
#pragma unroll
          for (int c = 0; c < D; c += 16) {
            uint32_t w[8];
#pragma unroll
            for (int i = 0; i < 8; ++i)
              w[i] = pack_bf16x2(__uint_as_float(ov[c + 2 * i]) * inv, __uint_as_float(ov[c + 2 * i + 1]) * inv);
            st_global_v8(dst + c, w[0], w[1], w[2], w[3], w[4], w[5], w[6], w[7]);
          }
          p.lse[(size_t)(qt.row0 + r) * p.Hq + h] = l > 0.f ? (m_used + __log2f(l)) * kLn2 : -INFINITY;
        }
      } else {
        // one piece of a split work item: store the unnormalised partial (O, max, sum);
        // the piece that finishes last merges all of them in slot order (log-sum-exp
        // merge), so the result does not depend on which piece that is.
        const size_t sb = (size_t)wk.slot * p.hpc + t;
        float4* po = p.part_o + sb * (D / 4) * 128;
        uint32_t ov[D];
        tmem_ld_row<D>(tO, ov);
        tc_fence_before();
        mbar_arrive(&o_free[t]);
#pragma unroll
        for (int i = 0; i < D / 4; ++i)
          po[(size_t)i * 128 + r] = make_float4(__uint_as_float(ov[4 * i]), __uint_as_float(ov[4 * i + 1]),
                                                __uint_as_float(ov[4 * i + 2]), __uint_as_float(ov[4 * i + 3]));
        p.part_ml[sb * 128 + r] = make_float2(m_used, l);
        // publish the partial device-wide, then one thread bumps the item's counter; the
        // handshake inside the CTA uses bounded mbarrier waits
        __threadfence();
        mbar_arrive(&ep_bar[t]);
        int32_t* counter = p.counters + (size_t)wk.slot0 * p.hpc + t;
        if (r == 0) {
          if (!pf_wait(&ep_bar[t], se & 1, p, abort_flag)) goto softmax_done;
          last_flag[t] = (atomicAdd(counter, 1) == wk.nparts - 1) ? 1 : 0;
          mbar_arrive(&ep_flag[t]);
        }
        if (!pf_wait_warp(&ep_flag[t], se & 1, p, abort_flag)) goto softmax_done;
        ++se;
        if (last_flag[t]) {
          // The merge reads the parts from L2: every load of one part's half row is issued
          // before any is used, so each part costs one round trip, not one per column.
          __threadfence();
          const size_t s0 = (size_t)wk.slot0 * p.hpc + t;
          float mx = -INFINITY;
#pragma unroll 4
          for (int k = 0; k < wk.nparts; ++k) mx = fmaxf(mx, __ldcg(p.part_ml + (s0 + (size_t)k * p.hpc) * 128 + r).x);
          float den = 0.f, inv = 0.f;
          const size_t orow = ((size_t)(qt.row0 + r) * p.Hq + h) * D;
#pragma unroll 1
          for (int half = 0; half < 2; ++half) {
            float4 acc[D / 8];
#pragma unroll
            for (int i = 0; i < D / 8; ++i) acc[i] = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 1
            for (int k = 0; k < wk.nparts; ++k) {
              const size_t sk = s0 + (size_t)k * p.hpc;
              const float2 ml = __ldcg(p.part_ml + sk * 128 + r);
              const float4* pk = p.part_o + (sk * (D / 4) + (size_t)half * (D / 8)) * 128 + r;
              float4 x[D / 8];
#pragma unroll
              for (int i = 0; i < D / 8; ++i) x[i] = __ldcg(pk + (size_t)i * 128);
              const float wgt = (ml.x == -INFINITY) ? 0.f : fast_exp2(ml.x - mx);
              if (half == 0) den += wgt * ml.y;
#pragma unroll
              for (int i = 0; i < D / 8; ++i) {
                acc[i].x = fmaf(wgt, x[i].x, acc[i].x);
                acc[i].y = fmaf(wgt, x[i].y, acc[i].y);
                acc[i].z = fmaf(wgt, x[i].z, acc[i].z);
                acc[i].w = fmaf(wgt, x[i].w, acc[i].w);
              }
            }
            if (half == 0) inv = den > 0.f ? 1.f / den : 0.f;
            if (valid) {
              __nv_bfloat16* dst = p.out + orow + half * (D / 2);
#pragma unroll
              for (int i = 0; i < D / 8; i += 4)
                st_global_v8(dst + i * 4, pack_bf16x2(acc[i].x * inv, acc[i].y * inv),
                             pack_bf16x2(acc[i].z * inv, acc[i].w * inv),
                             pack_bf16x2(acc[i + 1].x * inv, acc[i + 1].y * inv),
                             pack_bf16x2(acc[i + 1].z * inv, acc[i + 1].w * inv),
                             pack_bf16x2(acc[i + 2].x * inv, acc[i + 2].y * inv),
                             pack_bf16x2(acc[i + 2].z * inv, acc[i + 2].w * inv),
                             pack_bf16x2(acc[i + 3].x * inv, acc[i + 3].y * inv),
                             pack_bf16x2(acc[i + 3].z * inv, acc[i + 3].w * inv));
            }
          }
          if (valid) p.lse[(size_t)(qt.row0 + r) * p.Hq + h] = den > 0.f ? (mx + __log2f(den)) * kLn2 : -INFINITY;
          if (r == 0) *counter = 0;  // re-arm for the next launch
        }
      }
      ++wi;
    }
  softmax_done:;
  }
  tc_fence_before();
  __syncthreads();
}

// ------------------------------------------------------------------ host side
template <int D>
static cudaError_t launch_prefill_t(const PrefillParams& p, const PrefillTensors& T, cudaStream_t stream) {
  CUtensorMap mq, mkc, mvc, mkp, mvp;
  const uint64_t pool_rows = (uint64_t)T.num_pool_blocks * p.Hkv * kBlock;
  if (!make_map(&mq, T.q, (uint64_t)p.Hq * D, T.total_q, 128)) return cudaErrorInvalidValue;
  if (!make_map(&mkc, T.k_chunk, (uint64_t)p.Hkv * D, T.total_q, 16)) return cudaErrorInvalidValue;
  if (!make_map(&mvc, T.v_chunk, (uint64_t)p.Hkv * D, T.total_q, 16)) return cudaErrorInvalidValue;
  // an empty pool still needs a valid map: point it at the chunk tensor; only rows past
  // its end are ever read from it (the zero fill of a tile's missing units)
  PrefillParams pp = p;
  if (pool_rows) {
    if (!make_map(&mkp, T.k_pool, D, pool_rows, 16)) return cudaErrorInvalidValue;
    if (!make_map(&mvp, T.v_pool, D, pool_rows, 16)) return cudaErrorInvalidValue;
  } else {
    if (!make_map(&mkp, T.k_chunk, D, (uint64_t)T.total_q * p.Hkv, 16)) return cudaErrorInvalidValue;
    if (!make_map(&mvp, T.v_chunk, D, (uint64_t)T.total_q * p.Hkv, 16)) return cudaErrorInvalidValue;
    pp.pool_rows = (int32_t)(T.total_q * p.Hkv);
  }
  const int smem = PfLayout<D>::kBytes;
  cudaError_t e = cudaFuncSetAttribute(msa_prefill_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  // the warpgroups' register split (setmaxnreg) must fit in what the launch allocates
  cudaFuncAttributes fa;
  e = cudaFuncGetAttributes(&fa, msa_prefill_kernel<D>);
  if (e != cudaSuccess) return e;
  if (fa.numRegs != kPfLaunchRegs) return cudaErrorInvalidConfiguration;

  const int grid = p.n_ctas;  // the planner balanced the pieces over this many CTAs
  if (grid == 0) return cudaSuccess;
  msa_prefill_kernel<D><<<grid, kPfThreads, smem, stream>>>(mq, mkc, mvc, mkp, mvp, pp);
  return cudaGetLastError();
}

cudaError_t launch_prefill(const PrefillParams& p, const PrefillTensors& T, cudaStream_t stream) {
  if (T.d == 128) return launch_prefill_t<128>(p, T, stream);
  return launch_prefill_t<64>(p, T, stream);
}

}  // namespace msa
