// MSA decode (TPOT path): the newest token of each sequence attends over every KV
// token of its non-contiguous pool segments (paper: "Multi-Segment Attention ...",
// abstract -- TPOT gains come from attention over the segmented cache; section 4.1 --
// the context is a set of disjoint KV regions).
//
// Split-KV design for a bandwidth-bound scan on B300:
//  * grid = (split units) x (KV heads x head groups).  A split unit is a run of
//    canonical blocks of one sequence; the planner sizes units so the grid covers the
//    148 SMs many times over.
//  * each CTA handles GH query heads that share one KV head, so every K/V byte is read
//    from HBM once per head group;
//  * each of the 4 warps owns a ring of 3 shared-memory stages; a stage is one paged
//    block's K and V for this KV head, brought in by TMA as 128-byte-swizzled 16 x 64
//    boxes (8 KB at d = 128), so 192 KB per SM are in flight;
//  * the two small products of a block run on the warp-level tensor-core MMA
//    (m16n8k16, bf16 in, fp32 accumulate): S = Q K^T with the GH heads as rows of a
//    16-row tile, and O += P V with P kept in registers (the accumulator fragment of
//    S is the operand fragment of P).  K and V reach the registers through ldmatrix
//    (V transposed), conflict-free on the swizzled layout.  This keeps the instruction
//    count per byte low enough for the scan to stay bandwidth-bound;
//  * online softmax once per 16-token block in log2 units, rescaling O only when the
//    running max grows by more than 2^8 (exact either way: O and the sum share the
//    reference max);
//  * the split partials (O normalised, natural-log LSE) go to the workspace; the last
//    CTA of each (sequence, head group) merges them (LSE merge) and writes the bf16
//    output and fp32 LSE, then re-arms its counter.
#include <cuda.h>
#include <cuda_runtime.h>

#include "msa_device.cuh"
#include "msa_kernels.h"
#include "msa_tmap.h"

namespace msa {

constexpr int kDecWarps = 4;
constexpr int kDecStages = 3;

template <int D>
struct DecSmem {
  static constexpr int kSlabs = D / 64;
  static constexpr int kSlabBytes = kBlock * 128;         // 16 rows x 128 bytes
  static constexpr int kKVBytes = kSlabs * kSlabBytes;    // one block of K (or V) of one head
  static constexpr int kStageBytes = 2 * kKVBytes;        // K, then V
  static constexpr int kWarpBytes = kDecStages * kStageBytes;
  static constexpr int kRingBytes = kDecWarps * kWarpBytes;
  static constexpr int kBytes = kRingBytes + 1024;        // + alignment of the swizzled slabs
};

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
// d += A(16x16, row) * B(16x8, col), bf16 inputs, fp32 accumulators
__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Byte offset of 16-byte chunk `chunk` of row `row` in a 128-byte-swizzled slab (the
// chunk index is XORed with the row index modulo 8, as the TMA wrote it).
__device__ __forceinline__ uint32_t swz(int row, int chunk) { return row * 128 + ((chunk ^ (row & 7)) << 4); }

template <int D, int GH>
__global__ void __launch_bounds__(kDecWarps * 32, 2)
    msa_decode_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                      const DecodeParams p) {
  using S = DecSmem<D>;
  constexpr int NT = D / 8;  // 8-column output tiles of O
  static_assert(GH >= 1 && GH <= 8, "the heads of a group are rows 0..7 of the 16-row tile");

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ __align__(8) uint64_t full_bar[kDecWarps][kDecStages];
  __shared__ float mw[kDecWarps][GH];
  __shared__ float lw[kDecWarps][GH];
  __shared__ int32_t last_flag;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const SplitRec sp = p.split[blockIdx.x];
#ifdef MSA_DEBUG
  // the split must point inside the plan's block list, sequences and splits
  if (!MSA_DCHECK(sp.blk_begin >= 0 && sp.blk_count >= 0 && sp.blk_begin + sp.blk_count <= p.n_blist &&
                      sp.seq >= 0 && sp.seq < p.num_seqs && sp.first_split >= 0 && sp.nsplit >= 1 &&
                      sp.first_split + sp.nsplit <= (int)gridDim.x,
                  p.status))
    return;
#endif
  const int groups = p.G / GH;
  const int g = blockIdx.y / groups;
  const int h0 = g * p.G + (blockIdx.y % groups) * GH;

  if (tid == 0) {
    for (int w = 0; w < kDecWarps; ++w)
      for (int s = 0; s < kDecStages; ++s) mbar_init(&full_bar[w][s], 1);
    fence_barrier_init();
  }
  __syncthreads();

  // Q as A fragments: row r = lane/4 is head h0 + r (rows GH..15 are zero), columns
  // k0 = (lane%4)*2 and k0 + 8 of each 16-column step
  const int qr = lane >> 2, kq = (lane & 3) * 2;
  uint32_t qa[D / 16][2];
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk) {
    if (qr < GH) {
      const uint32_t* src =
          reinterpret_cast<const uint32_t*>(p.q + ((size_t)sp.seq * p.Hq + h0 + qr) * D + kk * 16 + kq);
      qa[kk][0] = src[0];
      qa[kk][1] = src[4];
    } else {
      qa[kk][0] = qa[kk][1] = 0u;
    }
  }

  uint8_t* ring = smem + warp * S::kWarpBytes;
  const uint32_t ring_u32 = smem_u32(ring);
  const int nb_w = sp.blk_count > warp ? (sp.blk_count - warp + kDecWarps - 1) / kDecWarps : 0;

  // test hook: warp 0 of one CTA may leave out one block, so that the wait for it runs out
  const int drop_k = ((int)blockIdx.x == p.drop_split && blockIdx.y == 0 && warp == 0) ? p.drop_k : -1;
  auto issue = [&](int k) {  // lane 0 only
    if (k == drop_k) return;
    const int bi = sp.blk_begin + warp + kDecWarps * k;
    const int phys = p.blist[bi];
    const int st = k % kDecStages;
    uint8_t* dst = ring + st * S::kStageBytes;
    // (a block id outside the pool reads rows past it, which arrive as zeros)
    const int y = MSA_DCHECK(phys >= 0 && phys < p.num_pool_blocks, p.status) ? (phys * p.Hkv + g) * kBlock
                                                                                : (int)p.pool_rows;
    mbar_arrive_expect_tx(&full_bar[warp][st], S::kStageBytes);
#pragma unroll
    for (int s = 0; s < S::kSlabs; ++s) tma_load_2d(dst + s * S::kSlabBytes, &tm_k, &full_bar[warp][st], s * 64, y);
#pragma unroll
    for (int s = 0; s < S::kSlabs; ++s)
      tma_load_2d(dst + S::kKVBytes + s * S::kSlabBytes, &tm_v, &full_bar[warp][st], s * 64, y);
  };

  if (lane == 0) {
    for (int k = 0; k < kDecStages && k < nb_w; ++k) issue(k);
  }
  __syncwarp();

  float m_used = -INFINITY, l_part = 0.f;  // row qr's reference max (log2 units); this lane's sum share
  float o[NT][4];
#pragma unroll
  for (int n = 0; n < NT; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;

  // ldmatrix lane roles: K (plain): matrices (tokens 0-7 | 8-15) x (chunk c | c+1);
  // V (transposed): (tokens 0-7 | 8-15) x chunk c, then chunk c+1
  const int k_tok = ((lane >> 4) << 3) + (lane & 7), k_dc = (lane >> 3) & 1;
  const int v_tok = (((lane >> 3) & 1) << 3) + (lane & 7), v_dc = lane >> 4;

  int k = 0;
  bool aborted = false;
  for (; k < nb_w; ++k) {
    const int st = k % kDecStages;
    const int bi = sp.blk_begin + warp + kDecWarps * k;
    int fill = p.bfill[bi];
    if (!MSA_DCHECK(fill >= 1 && fill <= kBlock, p.status)) fill = fill < 1 ? 0 : kBlock;
    if (!mbar_wait(&full_bar[warp][st], (k / kDecStages) & 1, p.wait_ns)) {
      set_status(p.status, MSA_ERR_TIMEOUT);
      aborted = true;
      break;
    }
    const uint32_t ks = ring_u32 + st * S::kStageBytes;
    const uint32_t vsb = ks + S::kKVBytes;
    if (fill < kBlock) {
      // slots past the block's fill are not part of the context: their V rows are
      // zeroed so that a masked key (P = 0) adds nothing even if the slot holds NaN
      uint8_t* vrow = ring + st * S::kStageBytes + S::kKVBytes;
      for (int i = lane; i < S::kSlabs * kBlock * 8; i += 32) {
        const int s = i / (kBlock * 8), row = (i / 8) % kBlock, c = i % 8;
        if (row >= fill) *reinterpret_cast<uint4*>(vrow + s * S::kSlabBytes + row * 128 + c * 16) = make_uint4(0, 0, 0, 0);
      }
      __syncwarp();
    }

    // ---- S = Q K^T (16 rows x 16 tokens)
    float sacc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
      const int slab = kk >> 2, c0 = (kk & 3) * 2;
      uint32_t b0, b1, b2, b3;
      ldsm_x4(ks + slab * S::kSlabBytes + swz(k_tok, c0 + k_dc), b0, b1, b2, b3);
      mma16816(sacc[0], qa[kk][0], 0u, qa[kk][1], 0u, b0, b1);
      mma16816(sacc[1], qa[kk][0], 0u, qa[kk][1], 0u, b2, b3);
    }

    // ---- online softmax for row qr over tokens 8n + kq + e (log2 units)
    float x[4];
#pragma unroll
    for (int n = 0; n < 2; ++n)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int tok = n * 8 + kq + e;
        x[n * 2 + e] = tok < fill ? sacc[n][e] * p.scale_log2 : -INFINITY;
      }
    float mx = fmaxf(fmaxf(x[0], x[1]), fmaxf(x[2], x[3]));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
    float factor = 1.f;
    const bool resc = mx > m_used + 8.f;
    if (resc) {
      factor = (m_used == -INFINITY) ? 0.f : fast_exp2(m_used - mx);
      l_part *= factor;
      m_used = mx;
    }
    if (__any_sync(0xffffffffu, resc)) {
#pragma unroll
      for (int n = 0; n < NT; ++n) {
        o[n][0] *= factor;
        o[n][1] *= factor;
      }
    }
    const float ms = (m_used == -INFINITY) ? 0.f : m_used;
    float pv[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      pv[i] = fast_exp2(x[i] - ms);
      l_part += pv[i];
    }
    const uint32_t pa0 = pack_bf16x2(pv[0], pv[1]), pa2 = pack_bf16x2(pv[2], pv[3]);

    // ---- O += P V (16 rows x D)
#pragma unroll
    for (int nd = 0; nd < D / 16; ++nd) {
      const int slab = nd >> 2, c0 = (nd & 3) * 2;
      uint32_t b0, b1, b2, b3;
      ldsm_x4_t(vsb + slab * S::kSlabBytes + swz(v_tok, c0 + v_dc), b0, b1, b2, b3);
      mma16816(o[2 * nd], pa0, 0u, pa2, 0u, b0, b1);
      mma16816(o[2 * nd + 1], pa0, 0u, pa2, 0u, b2, b3);
    }
    __syncwarp();
    if (lane == 0 && k + kDecStages < nb_w) {
      fence_proxy_async_smem();  // generic writes (zeroed rows) before the next TMA into this stage
      issue(k + kDecStages);
    }
    __syncwarp();
  }
  if (aborted) {
    // let the copies this warp still has in flight land before the CTA exits
    const int issued = nb_w < k + kDecStages ? nb_w : k + kDecStages;
    for (int kk = k; kk < issued; ++kk)
      if (kk != drop_k) mbar_wait(&full_bar[warp][kk % kDecStages], (kk / kDecStages) & 1, 1000000000ull);
  }

  // ---- combine the four lanes of a row (sum) and the warps (max, sum, O) in shared memory
  l_part += __shfl_xor_sync(0xffffffffu, l_part, 1);
  l_part += __shfl_xor_sync(0xffffffffu, l_part, 2);
  __syncthreads();
  float* ow = reinterpret_cast<float*>(smem);  // [warps][GH][D]
  if (qr < GH) {
    if ((lane & 3) == 0) {
      mw[warp][qr] = m_used;
      lw[warp][qr] = l_part;
    }
#pragma unroll
    for (int n = 0; n < NT; ++n) {
      ow[(warp * GH + qr) * D + n * 8 + kq] = o[n][0];
      ow[(warp * GH + qr) * D + n * 8 + kq + 1] = o[n][1];
    }
  }
  __syncthreads();

  const size_t gsplit = blockIdx.x;
  const bool single = sp.nsplit == 1;
  for (int idx = tid; idx < GH * D; idx += kDecWarps * 32) {
    const int hh = idx / D, i = idx % D;
    float m = -INFINITY;
#pragma unroll
    for (int w = 0; w < kDecWarps; ++w) m = fmaxf(m, mw[w][hh]);
    float L = 0.f, acc = 0.f;
#pragma unroll
    for (int w = 0; w < kDecWarps; ++w) {
      const float mwv = mw[w][hh];
      const float wt = (mwv == -INFINITY) ? 0.f : fast_exp2(mwv - m);
      L += wt * lw[w][hh];
      acc += wt * ow[(w * GH + hh) * D + i];
    }
    const float on = L > 0.f ? acc / L : 0.f;
    const float ls = L > 0.f ? (m + __log2f(L)) * 0.69314718055994531f : -INFINITY;
    const int h = h0 + hh;
    if (single) {
      p.out[((size_t)sp.seq * p.Hq + h) * D + i] = __float2bfloat16_rn(on);
      if (i == 0) p.lse[(size_t)sp.seq * p.Hq + h] = ls;
    } else {
      p.part_o[(gsplit * p.Hq + h) * D + i] = on;
      if (i == 0) p.part_lse[gsplit * p.Hq + h] = ls;
    }
  }
  if (single) return;

  // ---- last CTA of this (sequence, head group) merges the split partials
  __threadfence();
  __syncthreads();
  int32_t* counter = p.counters + (size_t)sp.seq * p.Hq + h0;
  if (tid == 0) last_flag = (atomicAdd(counter, 1) == sp.nsplit - 1);
  __syncthreads();
  if (!last_flag) return;
  __threadfence();
  for (int idx = tid; idx < GH * D; idx += kDecWarps * 32) {
    const int hh = idx / D, i = idx % D;
    const int h = h0 + hh;
    float m = -INFINITY;
    for (int r = 0; r < sp.nsplit; ++r)
      m = fmaxf(m, __ldcg(p.part_lse + (size_t)(sp.first_split + r) * p.Hq + h));
    float den = 0.f, acc = 0.f;
    for (int r = 0; r < sp.nsplit; ++r) {
      const size_t sr = (size_t)(sp.first_split + r);
      const float lr = __ldcg(p.part_lse + sr * p.Hq + h);
      const float wt = (lr == -INFINITY) ? 0.f : fast_exp2((lr - m) * 1.4426950408889634f);
      den += wt;
      acc += wt * __ldcg(p.part_o + (sr * p.Hq + h) * D + i);
    }
    p.out[((size_t)sp.seq * p.Hq + h) * D + i] = __float2bfloat16_rn(den > 0.f ? acc / den : 0.f);
    if (i == 0) p.lse[(size_t)sp.seq * p.Hq + h] = den > 0.f ? m + __logf(den) : -INFINITY;
  }
  if (tid == 0) *counter = 0;
}

template <int D, int GH>
cudaError_t launch_decode_t(const DecodeParams& p, int n_split, int head_groups, cudaStream_t stream) {
  CUtensorMap mk, mv;
  if (p.pool_rows <= 0) return cudaErrorInvalidValue;
  if (!make_map(&mk, p.k_pool, D, (uint64_t)p.pool_rows, kBlock)) return cudaErrorInvalidValue;
  if (!make_map(&mv, p.v_pool, D, (uint64_t)p.pool_rows, kBlock)) return cudaErrorInvalidValue;
  const int smem = DecSmem<D>::kBytes;
  cudaError_t e = cudaFuncSetAttribute(msa_decode_kernel<D, GH>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  dim3 grid(n_split, head_groups);
  msa_decode_kernel<D, GH><<<grid, kDecWarps * 32, smem, stream>>>(mk, mv, p);
  return cudaGetLastError();
}

cudaError_t launch_decode(const DecodeParams& p, int d, int n_split, cudaStream_t stream) {
  const int G = p.G;
  const int GH = (G % 8 == 0) ? 8 : (G % 4 == 0) ? 4 : (G % 2 == 0 ? 2 : 1);
  const int groups = p.Hkv * (G / GH);
  if (d == 128) {
    if (GH == 8) return launch_decode_t<128, 8>(p, n_split, groups, stream);
    if (GH == 4) return launch_decode_t<128, 4>(p, n_split, groups, stream);
    if (GH == 2) return launch_decode_t<128, 2>(p, n_split, groups, stream);
    return launch_decode_t<128, 1>(p, n_split, groups, stream);
  }
  if (GH == 8) return launch_decode_t<64, 8>(p, n_split, groups, stream);
  if (GH == 4) return launch_decode_t<64, 4>(p, n_split, groups, stream);
  if (GH == 2) return launch_decode_t<64, 2>(p, n_split, groups, stream);
  return launch_decode_t<64, 1>(p, n_split, groups, stream);
}

}  // namespace msa
