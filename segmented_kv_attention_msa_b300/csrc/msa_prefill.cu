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
//    128 chunk rows each) and of each KV tile into a 2-stage ring.  A pool KV tile is 8
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
constexpr int kPfStages = 2;
constexpr int kSlabBytes = 128 * 128;  // 128 rows x 128 bytes (64 bf16)

template <int D>
struct PfLayout {
  static constexpr int kTileBytes = 128 * D * 2;
  static constexpr int kQ = 0;
  static constexpr int kK = kQ + 2 * kTileBytes;
  static constexpr int kV = kK + kPfStages * kTileBytes;
  static constexpr int kPos = kV + kPfStages * kTileBytes;
  static constexpr int kBar = kPos + kPfStages * 128 * 4;
  static constexpr int kNumBars = 17;
  static constexpr int kEnd = kBar + kNumBars * 8 + 16;
  static constexpr int kBytes = kEnd + 1024;  // slack for 1024-byte alignment of the base
};

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
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = sm + L::kQ;
  uint8_t* sK = sm + L::kK;
  uint8_t* sV = sm + L::kV;
  int32_t* sPos = reinterpret_cast<int32_t*>(sm + L::kPos);
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + L::kBar);
  uint64_t* q_full = bars + 0;
  uint64_t* q_empty = bars + 1;
  uint64_t* k_full = bars + 2;     // [2]
  uint64_t* v_full = bars + 4;     // [2]
  uint64_t* kv_empty = bars + 6;   // [2]
  uint64_t* s_full = bars + 8;     // [2] per head
  uint64_t* p_full = bars + 10;    // [2]
  uint64_t* o_full = bars + 12;    // [2]
  uint64_t* o_free = bars + 14;    // [2]
  uint64_t* drain = bars + 16;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + L::kNumBars);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    mbar_init(q_empty, 1);
    for (int s = 0; s < kPfStages; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&v_full[s], 1);
      mbar_init(&kv_empty[s], 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(&s_full[t], 1);
      mbar_init(&p_full[t], 128);
      mbar_init(&o_full[t], 1);
      mbar_init(&o_free[t], 128);
    }
    mbar_init(drain, 1);
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
    int it = 0, wi = 0;
    int last_it[kPfStages] = {-1, -1};
    int last_wi = -1;
    for (int w = blockIdx.x; w < p.n_work; w += gridDim.x) {
      const WorkRec wk = p.work[w];
      const QTileRec qt = p.qt[wk.qt];
      const int n = qt.list_count;
      if (n == 0) continue;
      if (!pf_wait_warp(q_empty, (wi & 1) ^ 1, p, abort_flag)) goto producer_done;
      if (lane == 0) {
        mbar_arrive_expect_tx(q_full, p.hpc * L::kTileBytes);
        for (int t = 0; t < p.hpc; ++t)
          for (int s = 0; s < kSlabs; ++s)
            tma_load_2d(sQ + t * L::kTileBytes + s * kSlabBytes, &tm_q, q_full, (wk.h0 + t) * D + s * 64, qt.row0);
      }
      last_wi = wi;
      for (int j = 0; j < n; ++j, ++it) {
        const int st = it % kPfStages;
        if (!pf_wait_warp(&kv_empty[st], ((it / kPfStages) & 1) ^ 1, p, abort_flag)) goto producer_done;
        const int e = p.list[qt.list_begin + j];
        const KTileRec* kt = p.kt + (e & 0x7fffffff);
        const int src = kt->src, ntok = kt->ntok, row0 = kt->row0, nblk = kt->nblk;
        for (int r = lane; r < 128; r += 32) {
          int pos;
          if (src == SRC_CHUNK) {
            pos = (r < ntok) ? p.qpos[row0 + r] : 0x7fffffff;
          } else {
            const int i = r >> 4, tt = r & 15;
            pos = (i < nblk && tt < kt->bfill[i]) ? kt->bpos[i] + tt : 0x7fffffff;
          }
          sPos[st * 128 + r] = pos;
        }
        __threadfence_block();
        __syncwarp();
        if (lane == 0) {
          uint8_t* dK = sK + st * L::kTileBytes;
          uint8_t* dV = sV + st * L::kTileBytes;
          mbar_arrive_expect_tx(&k_full[st], L::kTileBytes);
          if (src == SRC_CHUNK) {
            for (int s = 0; s < kSlabs; ++s)
              tma_load_2d(dK + s * kSlabBytes, &tm_kc, &k_full[st], wk.g * D + s * 64, row0);
          } else {
            for (int i = 0; i < kTileBlocks; ++i) {
              const int y = (i < nblk) ? (kt->blk[i] * p.Hkv + wk.g) * kBlock : p.pool_rows;
              for (int s = 0; s < kSlabs; ++s)
                tma_load_2d(dK + s * kSlabBytes + i * 2048, &tm_kp, &k_full[st], s * 64, y);
            }
          }
          mbar_arrive_expect_tx(&v_full[st], L::kTileBytes);
          if (src == SRC_CHUNK) {
            for (int s = 0; s < kSlabs; ++s)
              tma_load_2d(dV + s * kSlabBytes, &tm_vc, &v_full[st], wk.g * D + s * 64, row0);
          } else {
            for (int i = 0; i < kTileBlocks; ++i) {
              const int y = (i < nblk) ? (kt->blk[i] * p.Hkv + wk.g) * kBlock : p.pool_rows;
              for (int s = 0; s < kSlabs; ++s)
                tma_load_2d(dV + s * kSlabBytes + i * 2048, &tm_vp, &v_full[st], s * 64, y);
            }
          }
        }
        last_it[st] = it;
        __syncwarp();
      }
      ++wi;
    }
  producer_done:
    // every copy this warp started must land before the CTA may exit
    for (int s = 0; s < kPfStages; ++s)
      if (last_it[s] >= 0) {
        mbar_wait(&k_full[s], (last_it[s] / kPfStages) & 1, 1000000000ull);
        mbar_wait(&v_full[s], (last_it[s] / kPfStages) & 1, 1000000000ull);
      }
    if (last_wi >= 0) mbar_wait(q_full, last_wi & 1, 1000000000ull);
  } else if (warp == 8) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      int it = 0, wi = 0;
      auto issue_qk = [&](int t, int st) {
        const uint32_t qa = smem_u32(sQ + t * L::kTileBytes);
        const uint32_t ka = smem_u32(sK + st * L::kTileBytes);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * kSlabBytes + (kk & 3) * 32;
          umma_ss(tmem + t * 128, smem_desc_sw128(qa + off, 16, 1024), smem_desc_sw128(ka + off, 16, 1024),
                  kIdescQK, kk > 0);
        }
      };
      auto issue_pv = [&](int t, int st, bool acc) {
        const uint32_t va = smem_u32(sV + st * L::kTileBytes);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          umma_ts(tmem + 256 + t * 128, tmem + t * 128 + kk * 8,
                  smem_desc_sw128(va + kk * 2048, kSlabBytes, 1024), kIdescPV, (acc || kk > 0) ? 1u : 0u);
      };
      for (int w = blockIdx.x; w < p.n_work; w += gridDim.x) {
        const WorkRec wk = p.work[w];
        const int n = p.qt[wk.qt].list_count;
        if (n == 0) continue;
        if (!pf_wait(q_full, wi & 1, p, abort_flag)) goto mma_done;
        {
          const int st0 = it % kPfStages;
          if (!pf_wait(&k_full[st0], (it / kPfStages) & 1, p, abort_flag)) goto mma_done;
          tc_fence_after();
          for (int t = 0; t < p.hpc; ++t) {
            issue_qk(t, st0);
            umma_commit(&s_full[t]);
          }
          if (n == 1) umma_commit(q_empty);
        }
        for (int j = 0; j < n; ++j) {
          const int cur = it + j, st = cur % kPfStages;
          const int nxt = cur + 1, stn = nxt % kPfStages;
          const bool has_next = j + 1 < n;
          bool have_v = false, have_kn = false;
          for (int t = 0; t < p.hpc; ++t) {
            if (!pf_wait(&p_full[t], cur & 1, p, abort_flag)) goto mma_done;
            if (j == 0 && !pf_wait(&o_free[t], (wi & 1) ^ 1, p, abort_flag)) goto mma_done;
            if (!have_v) {
              if (!pf_wait(&v_full[st], (cur / kPfStages) & 1, p, abort_flag)) goto mma_done;
              have_v = true;
            }
            tc_fence_after();
            issue_pv(t, st, j > 0);
            if (has_next) {
              if (!have_kn) {
                if (!pf_wait(&k_full[stn], (nxt / kPfStages) & 1, p, abort_flag)) goto mma_done;
                have_kn = true;
                tc_fence_after();
              }
              issue_qk(t, stn);
              umma_commit(&s_full[t]);
            } else {
              umma_commit(&o_full[t]);
            }
          }
          if (j + 2 == n) umma_commit(q_empty);
          umma_commit(&kv_empty[st]);
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
    int it = 0, wi = 0;
    for (int w = blockIdx.x; w < p.n_work; w += gridDim.x) {
      const WorkRec wk = p.work[w];
      const QTileRec qt = p.qt[wk.qt];
      const int n = qt.list_count;
      if (n == 0) continue;
      if (t >= p.hpc) {
        it += n;
        ++wi;
        continue;
      }
      const int h = wk.h0 + t;
      const bool valid = r < qt.nrows;
      const int qp = valid ? p.qpos[qt.row0 + r] : -1;
      float m_used = -INFINITY, l = 0.f;
      for (int j = 0; j < n; ++j, ++it) {
        const int st = it % kPfStages;
        const bool partial = p.list[qt.list_begin + j] < 0;
        if (!pf_wait_warp(&s_full[t], it & 1, p, abort_flag)) goto softmax_done;
        tc_fence_after();
        uint32_t s[128];
        tmem_ld_x32(tS + 0, *reinterpret_cast<uint32_t(*)[32]>(&s[0]));
        tmem_ld_x32(tS + 32, *reinterpret_cast<uint32_t(*)[32]>(&s[32]));
        tmem_ld_x32(tS + 64, *reinterpret_cast<uint32_t(*)[32]>(&s[64]));
        tmem_ld_x32(tS + 96, *reinterpret_cast<uint32_t(*)[32]>(&s[96]));
        tmem_wait_ld();
        if (partial) {
          if (!pf_wait_warp(&k_full[st], (it / kPfStages) & 1, p, abort_flag)) goto softmax_done;
          const int4* kp4 = reinterpret_cast<const int4*>(sPos + st * 128);
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            const int4 kp = kp4[c];
            if (kp.x > qp) s[4 * c + 0] = __float_as_uint(-INFINITY);
            if (kp.y > qp) s[4 * c + 1] = __float_as_uint(-INFINITY);
            if (kp.z > qp) s[4 * c + 2] = __float_as_uint(-INFINITY);
            if (kp.w > qp) s[4 * c + 3] = __float_as_uint(-INFINITY);
          }
        }
        float mx = -INFINITY;
#pragma unroll
        for (int c = 0; c < 128; ++c) mx = fmaxf(mx, __uint_as_float(s[c]));
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
        float rowsum = 0.f;
#pragma unroll
        for (int c = 0; c < 64; ++c) {
          const float p0 = fast_exp2(fmaf(__uint_as_float(s[2 * c]), p.scale_log2, -ms));
          const float p1 = fast_exp2(fmaf(__uint_as_float(s[2 * c + 1]), p.scale_log2, -ms));
          rowsum += p0 + p1;
          s[c] = pack_bf16x2(p0, p1);
        }
        l += rowsum;
        tmem_st_x32(tS + 0, *reinterpret_cast<uint32_t(*)[32]>(&s[0]));
        tmem_st_x32(tS + 32, *reinterpret_cast<uint32_t(*)[32]>(&s[32]));
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(&p_full[t]);
      }
      // epilogue: O / l -> bf16, LSE = ln 2 * (m + log2 l)
      if (!pf_wait_warp(&o_full[t], wi & 1, p, abort_flag)) goto softmax_done;
      tc_fence_after();
      {
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
      }
      tc_fence_before();
      mbar_arrive(&o_free[t]);
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


static int num_sms() {
  static int n = 0;
  if (!n) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (n <= 0) n = 148;
  }
  return n;
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
  const int grid = p.n_work < num_sms() ? p.n_work : num_sms();
  if (grid == 0) return cudaSuccess;
  msa_prefill_kernel<D><<<grid, kPfThreads, smem, stream>>>(mq, mkc, mvc, mkp, mvp, p);
  return cudaGetLastError();
}

cudaError_t launch_prefill(const PrefillParams& p, const PrefillTensors& T, cudaStream_t stream) {
  if (T.d == 128) return launch_prefill_t<128>(p, T, stream);
  return launch_prefill_t<64>(p, T, stream);
}

}  // namespace msa
