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
// How (one persistent CTA per SM, warp-specialised, 320 threads):
//  * warp 9 (producer): TMA loads of the Q tiles (two query heads sharing one KV head,
//    128 chunk rows each), of each K tile into a 3-deep ring and of each V tile into a
//    2-deep ring (a K slot frees as soon as its QK^T is done, so K runs well ahead).  A pool KV tile is 8
//    paged blocks, one 16-row box per block and 64-column slab; a chunk KV tile is one
//    128-row box per slab.  Missing blocks of a short pool tile are loaded from an
//    out-of-range row and arrive as zeros.  The producer also writes each tile's 128
//    key positions to shared memory for the masking of partial tiles.
//  * warp 8 (MMA issuer, one thread): tcgen05.mma kind::f16.  S_t = Q_t K^T (both
//    operands in 128-byte-swizzled shared memory, accumulator in TMEM), then
//    O_t += P_t V with P_t read from TMEM (it overwrites S_t as bf16) and V as an
//    MN-major shared-memory operand.  The two heads ping-pong: while one softmax group
//    works on S_0, the tensor core runs the other head's GEMMs.
//  * warps 0-3 / 4-7 (softmax groups, one per head): each thread owns one query row in
//    TMEM (tcgen05.ld 32x32b), applies the position mask on partial tiles only, keeps the
//    running max in log2 units, rescales the O accumulator in TMEM only when the max
//    grows by more than 2^8 (the result is exact either way: the final O is divided by
//    the sum taken with the same reference max), writes P as bf16 back to TMEM, and
//    at the end normalises O and stores bf16 rows and the LSE.
//  * KV tiles whose smallest position exceeds the query tile's largest are never
//    loaded (the planner leaves them out of the work item's list); tiles that every
//    query row sees fully skip the mask.
// TMEM: 512 columns = S_0 | S_1 | O_0 | O_1 (128 columns each).
#include <cuda.h>
#include <cuda_runtime.h>

#include "msa_device.cuh"
#include "msa_kernels.h"

namespace msa {


constexpr int kPfThreads = 320;
constexpr int kKStages = 3;            // K tiles in flight (a slot frees once its QK^T is done)
constexpr int kVStages = 2;            // V tiles (a slot frees once its PV is done)
constexpr int kSlabBytes = 128 * 128;  // 128 rows x 128 bytes (64 bf16)

// Shared memory: small items first (barriers, key positions), then the operand tiles on
// a 1024-byte boundary (the 128-byte swizzle pattern repeats every 1024 bytes).
template <int D>
struct PfLayout {
  static constexpr int kTileBytes = 128 * D * 2;
  static constexpr int kNumBars = 27;
  static constexpr int kBar = 0;
  static constexpr int kMisc = (kBar + kNumBars * 8 + 15) / 16 * 16;  // TMEM base address, abort flag
  static constexpr int kPos = (kMisc + 16 + 127) / 128 * 128;          // int32 [kVStages][128], read as int4
  static constexpr int kSmall = kPos + kVStages * 128 * 4;
  static constexpr int kQ = 0;                         // offsets from the aligned tile base
  static constexpr int kK = kQ + 2 * kTileBytes;
  static constexpr int kV = kK + kKStages * kTileBytes;
  static constexpr int kTiles = kV + kVStages * kTileBytes;
  static constexpr int kBytes = kSmall + 1023 + kTiles;
};
static_assert(PfLayout<128>::kBytes <= 232448, "prefill shared memory exceeds 227 KB");
static_assert(PfLayout<128>::kPos % 16 == 0 && PfLayout<128>::kMisc % 16 == 0, "16-byte alignment");

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

// A KV tile record spread over a warp: lane i holds word i of the 32-word record.
// Fields are read with warp shuffles, so every lane must take part.
struct TileRec {
  int v;
  __device__ __forceinline__ int get(int i) const { return __shfl_sync(0xffffffffu, v, i); }
};
__device__ __forceinline__ TileRec load_tile_rec(const PrefillParams& p, const int* lst, int j, int lane) {
  const int e = __ldg(lst + j);
  const int* rec = reinterpret_cast<const int*>(p.kt + (e & 0x7fffffff));
  return TileRec{__ldg(rec + lane)};
}

// Issue the TMA loads of one K or V tile (whole warp calls; lane 0 posts the byte
// count, lanes 0-7 load one 16-row paged block each, or lane 0 the 128-row chunk box).
template <int D>
__device__ __forceinline__ void issue_kv_tile(const TileRec& rec, uint8_t* dst, uint64_t* bar,
                                              const CUtensorMap* tm_chunk, const CUtensorMap* tm_pool,
                                              int g, int Hkv, int pool_rows, int lane) {
  constexpr int kSlabs = D / 64;
  const int src = rec.get(0), row0 = rec.get(2), nblk = rec.get(3);
  const int blk = rec.get(8 + (lane & 7));
  if (lane == 0) mbar_arrive_expect_tx(bar, 128 * D * 2);
  __syncwarp();
  if (src == SRC_CHUNK) {
    if (lane == 0)
      for (int s = 0; s < kSlabs; ++s) tma_load_2d(dst + s * kSlabBytes, tm_chunk, bar, g * D + s * 64, row0);
  } else if (lane < kTileBlocks) {
    // a missing block reads an out-of-range row and arrives as zeros
    const int y = (lane < nblk) ? (blk * Hkv + g) * kBlock : pool_rows;
    for (int s = 0; s < kSlabs; ++s) tma_load_2d(dst + s * kSlabBytes + lane * 2048, tm_pool, bar, s * 64, y);
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
  uint64_t* pos_full = bars + 12;  // [2] key positions of the tile held in V slot s
  uint64_t* s_full = bars + 14;    // [2] per head
  uint64_t* p_full = bars + 16;    // [2]
  uint64_t* o_full = bars + 18;    // [2]
  uint64_t* o_free = bars + 20;    // [2]
  uint64_t* drain = bars + 22;
  uint64_t* ep_bar = bars + 23;    // [2] split pieces: the head's 128 threads stored their partial
  uint64_t* ep_flag = bars + 25;   // [2] split pieces: merge counter read, last_flag[t] valid
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem_raw + L::kMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem_raw + L::kMisc + 4);
  volatile int* last_flag = reinterpret_cast<volatile int*>(smem_raw + L::kMisc + 8);  // [2]
  int32_t* sPos = reinterpret_cast<int32_t*>(smem_raw + L::kPos);
  uint8_t* tiles = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw + L::kSmall) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = tiles + L::kQ;
  uint8_t* sK = tiles + L::kK;
  uint8_t* sV = tiles + L::kV;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    mbar_init(q_empty, 1);
    for (int s = 0; s < kKStages; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&k_empty[s], 1);
    }
    for (int s = 0; s < kVStages; ++s) {
      mbar_init(&v_full[s], 1);
      mbar_init(&v_empty[s], 1);
      mbar_init(&pos_full[s], 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(&s_full[t], 1);
      mbar_init(&p_full[t], 128);
      mbar_init(&o_full[t], 1);
      mbar_init(&o_free[t], 128);
    }
    mbar_init(drain, 1);
    for (int t = 0; t < 2; ++t) {
      mbar_init(&ep_bar[t], 128);
      mbar_init(&ep_flag[t], 1);
    }
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

  if (warp == 9) {
    // ------------------------------------------------------------ producer
    // Per work item: Q, K0, K1, V0, K2, V1, ..., K(n-1), V(n-2), V(n-1).  K(j) waits for
    // the QK^T of the tile three back in its slot; V(j) waits for the PV of the tile two
    // back, which also frees that slot's key positions (that tile's softmax is done).
    int kit = 0, vit = 0, wi = 0;  // K tiles, V tiles and work items issued
    int last_k[kKStages] = {-1, -1, -1};
    int last_v[kVStages] = {-1, -1};
    int last_wi = -1;
    for (int w = __ldg(p.cta_begin + blockIdx.x), w1 = __ldg(p.cta_begin + blockIdx.x + 1); w < w1; ++w) {
      const WorkRec wk = p.work[w];
      const QTileRec qt = p.qt[wk.qt];
      const int n = wk.n;
      if (n == 0) continue;
      const int* lst = p.list + qt.list_begin + wk.j0;
      TileRec cur = load_tile_rec(p, lst, 0, lane);
      if (!pf_wait_warp(q_empty, (wi & 1) ^ 1, p, abort_flag)) goto producer_done;
      if (lane == 0) {
        mbar_arrive_expect_tx(q_full, p.hpc * L::kTileBytes);
        for (int t = 0; t < p.hpc; ++t)
          for (int s = 0; s < kSlabs; ++s)
            tma_load_2d(sQ + t * L::kTileBytes + s * kSlabBytes, &tm_q, q_full, (wk.h0 + t) * D + s * 64, qt.row0);
      }
      last_wi = wi;
      TileRec prev = cur;
      for (int j = 0; j <= n; ++j) {
        TileRec nxt = cur;
        if (j + 1 < n) nxt = load_tile_rec(p, lst, j + 1, lane);
        if (j < n) {
          const int ks = kit % kKStages;
          if (!pf_wait_warp(&k_empty[ks], ((kit / kKStages) & 1) ^ 1, p, abort_flag)) goto producer_done;
          issue_kv_tile<D>(cur, sK + ks * L::kTileBytes, &k_full[ks], &tm_kc, &tm_kp, wk.g, p.Hkv, p.pool_rows,
                           lane);
          last_k[ks] = kit;
          ++kit;
        }
        if (j >= 1) {
          // V and key positions of the previous tile
          const int vs = vit % kVStages;
          if (!pf_wait_warp(&v_empty[vs], ((vit / kVStages) & 1) ^ 1, p, abort_flag)) goto producer_done;
          issue_kv_tile<D>(prev, sV + vs * L::kTileBytes, &v_full[vs], &tm_vc, &tm_vp, wk.g, p.Hkv, p.pool_rows,
                           lane);
          last_v[vs] = vit;
          const int src = prev.get(0), ntok = prev.get(1), row0 = prev.get(2), nblk = prev.get(3);
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4) {
            const int r = q4 * 32 + lane;
            const int i = r >> 4, tt = r & 15;
            const int bp = prev.get(16 + i);
            const int bf = prev.get(24 + i);
            int pos;
            if (src == SRC_CHUNK) pos = (r < ntok) ? __ldg(p.qpos + row0 + r) : 0x7fffffff;
            else pos = (i < nblk && tt < bf) ? bp + tt : 0x7fffffff;
            sPos[vs * 128 + r] = pos;
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(&pos_full[vs]);
          ++vit;
        }
        prev = cur;
        cur = nxt;
      }
      ++wi;
    }
  producer_done:
    // every copy this warp started must land before the CTA may exit
    for (int s = 0; s < kKStages; ++s)
      if (last_k[s] >= 0) mbar_wait(&k_full[s], (last_k[s] / kKStages) & 1, 1000000000ull);
    for (int s = 0; s < kVStages; ++s)
      if (last_v[s] >= 0) mbar_wait(&v_full[s], (last_v[s] / kVStages) & 1, 1000000000ull);
    if (last_wi >= 0) mbar_wait(q_full, last_wi & 1, 1000000000ull);
  } else if (warp == 8) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      int it = 0, wi = 0;
      auto issue_qk = [&](int t, int ks) {
        const uint32_t qa = smem_u32(sQ + t * L::kTileBytes);
        const uint32_t ka = smem_u32(sK + ks * L::kTileBytes);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * kSlabBytes + (kk & 3) * 32;
          umma_ss(tmem + t * 128, smem_desc_sw128(qa + off, 16, 1024), smem_desc_sw128(ka + off, 16, 1024),
                  kIdescQK, kk > 0);
        }
      };
      auto issue_pv = [&](int t, int vs, bool acc) {
        const uint32_t va = smem_u32(sV + vs * L::kTileBytes);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          umma_ts(tmem + 256 + t * 128, tmem + t * 128 + kk * 8,
                  smem_desc_sw128(va + kk * 2048, kSlabBytes, 1024), kIdescPV, (acc || kk > 0) ? 1u : 0u);
      };
      for (int w = __ldg(p.cta_begin + blockIdx.x), w1 = __ldg(p.cta_begin + blockIdx.x + 1); w < w1; ++w) {
        const int n = p.work[w].n;
        if (n == 0) continue;
        if (!pf_wait(q_full, wi & 1, p, abort_flag)) goto mma_done;
        {
          const int ks0 = it % kKStages;
          if (!pf_wait(&k_full[ks0], (it / kKStages) & 1, p, abort_flag)) goto mma_done;
          tc_fence_after();
          for (int t = 0; t < p.hpc; ++t) {
            issue_qk(t, ks0);
            umma_commit(&s_full[t]);
          }
          umma_commit(&k_empty[ks0]);
          if (n == 1) umma_commit(q_empty);
        }
        for (int j = 0; j < n; ++j) {
          const int cur = it + j, vs = cur % kVStages;
          const int nxt = cur + 1, ksn = nxt % kKStages;
          const bool has_next = j + 1 < n;
          bool have_v = false, have_kn = false;
          for (int t = 0; t < p.hpc; ++t) {
            if (!pf_wait(&p_full[t], cur & 1, p, abort_flag)) goto mma_done;
            if (j == 0 && !pf_wait(&o_free[t], (wi & 1) ^ 1, p, abort_flag)) goto mma_done;
            if (!have_v) {
              if (!pf_wait(&v_full[vs], (cur / kVStages) & 1, p, abort_flag)) goto mma_done;
              have_v = true;
            }
            tc_fence_after();
            issue_pv(t, vs, j > 0);
            if (has_next) {
              if (!have_kn) {
                if (!pf_wait(&k_full[ksn], (nxt / kKStages) & 1, p, abort_flag)) goto mma_done;
                have_kn = true;
                tc_fence_after();
              }
              issue_qk(t, ksn);
              umma_commit(&s_full[t]);
            } else {
              umma_commit(&o_full[t]);
            }
          }
          if (has_next) umma_commit(&k_empty[ksn]);
          if (j + 2 == n) umma_commit(q_empty);
          umma_commit(&v_empty[vs]);
        }
        it += n;
        ++wi;
      }
    mma_done:
      umma_commit(drain);
      mbar_wait(drain, 0, 1000000000ull);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax groups
    const int t = warp >> 2, wq = warp & 3;
    const int r = wq * 32 + lane;
    const uint32_t lane_base = (uint32_t)(wq * 32) << 16;
    const uint32_t tS = tmem + lane_base + t * 128;
    const uint32_t tO = tmem + lane_base + 256 + t * 128;
    const float2 scale2 = make_float2(p.scale_log2, p.scale_log2);
    int it = 0, wi = 0, se = 0;  // tiles, pieces and split pieces done
    for (int w = __ldg(p.cta_begin + blockIdx.x), w1 = __ldg(p.cta_begin + blockIdx.x + 1); w < w1; ++w) {
      const WorkRec wk = p.work[w];
      const QTileRec qt = p.qt[wk.qt];
      const int n = wk.n;
      if (n == 0) continue;
      if (t >= p.hpc) {
        it += n;
        ++wi;
        continue;
      }
      const int h = wk.h0 + t;
      const bool valid = r < qt.nrows;
      const int qp = valid ? __ldg(p.qpos + qt.row0 + r) : -1;
      float m_used = -INFINITY, l = 0.f;
      const int* lst = p.list + qt.list_begin + wk.j0;
      int e_next = __ldg(lst);
      for (int j = 0; j < n; ++j, ++it) {
        const int vs = it % kVStages;
        const bool partial = e_next < 0;
        if (j + 1 < n) e_next = __ldg(lst + j + 1);
        if (!pf_wait_warp(&s_full[t], it & 1, p, abort_flag)) goto softmax_done;
        tc_fence_after();
        uint32_t s[128];
        tmem_ld_x32(tS + 0, *reinterpret_cast<uint32_t(*)[32]>(&s[0]));
        tmem_ld_x32(tS + 32, *reinterpret_cast<uint32_t(*)[32]>(&s[32]));
        tmem_ld_x32(tS + 64, *reinterpret_cast<uint32_t(*)[32]>(&s[64]));
        tmem_ld_x32(tS + 96, *reinterpret_cast<uint32_t(*)[32]>(&s[96]));
        tmem_wait_ld();
        if (partial) {
          if (!pf_wait_warp(&pos_full[vs], (it / kVStages) & 1, p, abort_flag)) goto softmax_done;
          const int4* kp4 = reinterpret_cast<const int4*>(sPos + vs * 128);
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            const int4 kp = kp4[c];
            if (kp.x > qp) s[4 * c + 0] = __float_as_uint(-INFINITY);
            if (kp.y > qp) s[4 * c + 1] = __float_as_uint(-INFINITY);
            if (kp.z > qp) s[4 * c + 2] = __float_as_uint(-INFINITY);
            if (kp.w > qp) s[4 * c + 3] = __float_as_uint(-INFINITY);
          }
        }
        // row max: eight independent chains, then a tree
        float m8[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) m8[i] = __uint_as_float(s[i]);
#pragma unroll
        for (int c = 8; c < 128; ++c) m8[c & 7] = fmaxf(m8[c & 7], __uint_as_float(s[c]));
        const float mx = fmaxf(fmaxf(fmaxf(m8[0], m8[1]), fmaxf(m8[2], m8[3])),
                               fmaxf(fmaxf(m8[4], m8[5]), fmaxf(m8[6], m8[7])));
        const float m_cand = mx * p.scale_log2;
        const bool need = m_cand > m_used + 8.f;
        const bool resc = need && (m_used != -INFINITY);
        float factor = 1.f;
        if (need) {
          if (resc) factor = fast_exp2(m_used - m_cand);
          l *= factor;
          m_used = m_cand;
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
          tmem_wait_st();
        }
        const float ms = (m_used == -INFINITY) ? 0.f : m_used;
        const float2 nms2 = make_float2(-ms, -ms);
        float2 acc[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[i] = make_float2(0.f, 0.f);
#pragma unroll
        for (int c = 0; c < 64; ++c) {
          const float2 x =
              ffma2(make_float2(__uint_as_float(s[2 * c]), __uint_as_float(s[2 * c + 1])), scale2, nms2);
          const float2 pe = make_float2(fast_exp2(x.x), fast_exp2(x.y));
          acc[c & 3] = fadd2(acc[c & 3], pe);
          s[c] = pack_bf16x2(pe.x, pe.y);
        }
        const float2 a = fadd2(fadd2(acc[0], acc[1]), fadd2(acc[2], acc[3]));
        l += a.x + a.y;
        tmem_st_x32(tS + 0, *reinterpret_cast<uint32_t(*)[32]>(&s[0]));
        tmem_st_x32(tS + 32, *reinterpret_cast<uint32_t(*)[32]>(&s[32]));
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(&p_full[t]);
      }
      // epilogue: O / l -> bf16, LSE = ln 2 * (m + log2 l)
      if (!pf_wait_warp(&o_full[t], wi & 1, p, abort_flag)) goto softmax_done;
      tc_fence_after();
      if (wk.nparts == 1) {
        const float inv = l > 0.f ? 1.f / l : 0.f;
        const size_t orow = ((size_t)(qt.row0 + r) * p.Hq + h) * D;
#pragma unroll 1
        for (int c = 0; c < D; c += 32) {
          uint32_t ov[32];
          tmem_ld_x32(tO + c, ov);
          tmem_wait_ld();
          if (valid) {
            uint4* dst = reinterpret_cast<uint4*>(p.out + orow + c);
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) {
              uint4 v;
              v.x = pack_bf16x2(__uint_as_float(ov[8 * q4 + 0]) * inv, __uint_as_float(ov[8 * q4 + 1]) * inv);
              v.y = pack_bf16x2(__uint_as_float(ov[8 * q4 + 2]) * inv, __uint_as_float(ov[8 * q4 + 3]) * inv);
              v.z = pack_bf16x2(__uint_as_float(ov[8 * q4 + 4]) * inv, __uint_as_float(ov[8 * q4 + 5]) * inv);
              v.w = pack_bf16x2(__uint_as_float(ov[8 * q4 + 6]) * inv, __uint_as_float(ov[8 * q4 + 7]) * inv);
              dst[q4] = v;
            }
          }
        }
        if (valid) p.lse[(size_t)(qt.row0 + r) * p.Hq + h] = l > 0.f ? (m_used + __log2f(l)) * kLn2 : -INFINITY;
        tc_fence_before();
        mbar_arrive(&o_free[t]);
      } else {
        // one piece of a split work item: store the unnormalised partial (O, max, sum);
        // the piece that finishes last merges all of them in slot order (log-sum-exp
        // merge), so the result does not depend on which piece that is.
        const size_t sb = (size_t)wk.slot * p.hpc + t;
        float4* po = p.part_o + sb * (D / 4) * 128;
#pragma unroll 1
        for (int c = 0; c < D; c += 32) {
          uint32_t ov[32];
          tmem_ld_x32(tO + c, ov);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 8; ++i)
            po[(size_t)(c / 4 + i) * 128 + r] = make_float4(__uint_as_float(ov[4 * i]), __uint_as_float(ov[4 * i + 1]),
                                                            __uint_as_float(ov[4 * i + 2]), __uint_as_float(ov[4 * i + 3]));
        }
        p.part_ml[sb * 128 + r] = make_float2(m_used, l);
        tc_fence_before();
        mbar_arrive(&o_free[t]);
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
          __threadfence();
          const size_t s0 = (size_t)wk.slot0 * p.hpc + t;
          float mx = -INFINITY;
          for (int k = 0; k < wk.nparts; ++k) mx = fmaxf(mx, __ldcg(p.part_ml + (s0 + (size_t)k * p.hpc) * 128 + r).x);
          float den = 0.f;
          for (int k = 0; k < wk.nparts; ++k) {
            const float2 ml = __ldcg(p.part_ml + (s0 + (size_t)k * p.hpc) * 128 + r);
            den += (ml.x == -INFINITY) ? 0.f : fast_exp2(ml.x - mx) * ml.y;
          }
          const float inv = den > 0.f ? 1.f / den : 0.f;
          if (valid) {
            const size_t orow = ((size_t)(qt.row0 + r) * p.Hq + h) * D;
#pragma unroll 1
            for (int c4 = 0; c4 < D / 4; c4 += 2) {
              float4 a0 = make_float4(0.f, 0.f, 0.f, 0.f), a1 = a0;
              for (int k = 0; k < wk.nparts; ++k) {
                const size_t sk = s0 + (size_t)k * p.hpc;
                const float mk = __ldcg(p.part_ml + sk * 128 + r).x;
                const float wgt = (mk == -INFINITY) ? 0.f : fast_exp2(mk - mx);
                const float4* pk = p.part_o + sk * (D / 4) * 128;
                const float4 x0 = __ldcg(pk + (size_t)c4 * 128 + r), x1 = __ldcg(pk + (size_t)(c4 + 1) * 128 + r);
                a0.x = fmaf(wgt, x0.x, a0.x); a0.y = fmaf(wgt, x0.y, a0.y);
                a0.z = fmaf(wgt, x0.z, a0.z); a0.w = fmaf(wgt, x0.w, a0.w);
                a1.x = fmaf(wgt, x1.x, a1.x); a1.y = fmaf(wgt, x1.y, a1.y);
                a1.z = fmaf(wgt, x1.z, a1.z); a1.w = fmaf(wgt, x1.w, a1.w);
              }
              uint4 v;
              v.x = pack_bf16x2(a0.x * inv, a0.y * inv);
              v.y = pack_bf16x2(a0.z * inv, a0.w * inv);
              v.z = pack_bf16x2(a1.x * inv, a1.y * inv);
              v.w = pack_bf16x2(a1.z * inv, a1.w * inv);
              *reinterpret_cast<uint4*>(p.out + orow + c4 * 4) = v;
            }
            p.lse[(size_t)(qt.row0 + r) * p.Hq + h] = den > 0.f ? (mx + __log2f(den)) * kLn2 : -INFINITY;
          }
          if (r == 0) *counter = 0;  // re-arm for the next launch
        }
      }
      ++wi;
    }
  softmax_done:;
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 8) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ------------------------------------------------------------------ host side
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn get_encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  }
  return fn;
}

// 2-D bf16 tensor map over `rows` rows of `cols` elements, 128-byte swizzle,
// box of 64 columns x box_rows rows; out-of-range elements read as zero.
static bool make_map(CUtensorMap* m, const void* base, uint64_t cols, uint64_t rows, uint32_t box_rows) {
  EncodeTiledFn fn = get_encode_fn();
  if (!fn || rows == 0 || cols == 0) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {64, box_rows};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}


template <int D>
static cudaError_t launch_prefill_t(const PrefillParams& p, const PrefillTensors& T, cudaStream_t stream) {
  CUtensorMap mq, mkc, mvc, mkp, mvp;
  const uint64_t pool_rows = (uint64_t)T.num_pool_blocks * p.Hkv * kBlock;
  if (!make_map(&mq, T.q, (uint64_t)p.Hq * D, T.total_q, 128)) return cudaErrorInvalidValue;
  if (!make_map(&mkc, T.k_chunk, (uint64_t)p.Hkv * D, T.total_q, 128)) return cudaErrorInvalidValue;
  if (!make_map(&mvc, T.v_chunk, (uint64_t)p.Hkv * D, T.total_q, 128)) return cudaErrorInvalidValue;
  // an empty pool still needs a valid map: point it at the chunk tensor (never read)
  if (pool_rows) {
    if (!make_map(&mkp, T.k_pool, D, pool_rows, 16)) return cudaErrorInvalidValue;
    if (!make_map(&mvp, T.v_pool, D, pool_rows, 16)) return cudaErrorInvalidValue;
  } else {
    if (!make_map(&mkp, T.k_chunk, D, (uint64_t)T.total_q * p.Hkv, 16)) return cudaErrorInvalidValue;
    if (!make_map(&mvp, T.v_chunk, D, (uint64_t)T.total_q * p.Hkv, 16)) return cudaErrorInvalidValue;
  }
  const int smem = PfLayout<D>::kBytes;
  cudaError_t e = cudaFuncSetAttribute(msa_prefill_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;

  const int grid = p.n_ctas;  // the planner balanced the pieces over this many CTAs
  if (grid == 0) return cudaSuccess;
  msa_prefill_kernel<D><<<grid, kPfThreads, smem, stream>>>(mq, mkc, mvc, mkp, mvp, p);
  return cudaGetLastError();
}

cudaError_t launch_prefill(const PrefillParams& p, const PrefillTensors& T, cudaStream_t stream) {
  if (T.d == 128) return launch_prefill_t<128>(p, T, stream);
  return launch_prefill_t<64>(p, T, stream);
}

}  // namespace msa
