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
//  * each of the 4 warps owns a ring of 3 shared-memory stages filled by 1-D bulk
//    copies (cp.async.bulk, 4 KB K + 4 KB V per block at d = 128), so 24 KB per warp
//    and 192 KB per SM are in flight without register staging;
//  * scores: 8 lanes per token (16-element slice each) and a 3-step shuffle reduction;
//    online softmax once per 16-token block in log2 units; P.V: every lane owns a
//    4-element slice of d for all GH heads;
//  * the split partials (O normalised, natural-log LSE) go to the workspace; the last
//    CTA of each (sequence, head group) merges them (LSE merge) and writes the bf16
//    output and fp32 LSE, then re-arms its counter.
#include <cuda_runtime.h>

#include "msa_device.cuh"
#include "msa_kernels.h"

namespace msa {


constexpr int kDecWarps = 4;
constexpr int kDecStages = 3;

template <int D>
struct DecSmem {
  static constexpr int kBlkBytes = kBlock * D * 2;
  static constexpr int kStageBytes = 2 * kBlkBytes;
  static constexpr int kWarpBytes = kDecStages * kStageBytes;
  static constexpr int kRingBytes = kDecWarps * kWarpBytes;
};

template <int D, int GH>
__global__ void __launch_bounds__(kDecWarps * 32) msa_decode_kernel(const DecodeParams p) {
  constexpr int SL = D / 8;        // QK: d-slice per lane (8 lanes per token)
  constexpr int DL = D / 32;       // PV: d-slice per lane
  constexpr int NS = kBlock * GH;  // scores per block
  constexpr int EPL = NS >= 32 ? NS / 32 : 1;
  using S = DecSmem<D>;

  extern __shared__ __align__(1024) uint8_t smem[];
  __shared__ __align__(8) uint64_t full_bar[kDecWarps][kDecStages];
  __shared__ float sc[kDecWarps][NS];
  __shared__ float ps[kDecWarps][NS];
  __shared__ float fs[kDecWarps][GH];
  __shared__ int32_t last_flag;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const SplitRec sp = p.split[blockIdx.x];
  const int groups = p.G / GH;
  const int g = blockIdx.y / groups;
  const int h0 = g * p.G + (blockIdx.y % groups) * GH;

  if (tid == 0) {
    for (int w = 0; w < kDecWarps; ++w)
      for (int s = 0; s < kDecStages; ++s) mbar_init(&full_bar[w][s], 1);
    fence_barrier_init();
  }
  __syncthreads();

  // query slice for the score layout, pre-scaled into log2 units
  const int tg = lane >> 3, sub = lane & 7;
  float qf[GH][SL];
#pragma unroll
  for (int hh = 0; hh < GH; ++hh) {
    const uint4* src = reinterpret_cast<const uint4*>(p.q + ((size_t)sp.seq * p.Hq + h0 + hh) * D + sub * SL);
#pragma unroll
    for (int c = 0; c < SL / 8; ++c) {
      uint4 w = src[c];
      uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        qf[hh][c * 8 + 2 * e] = bf16_lo(ws[e]) * p.scale_log2;
        qf[hh][c * 8 + 2 * e + 1] = bf16_hi(ws[e]) * p.scale_log2;
      }
    }
  }

  uint8_t* ring = smem + warp * S::kWarpBytes;
  const int nb_w = sp.blk_count > warp ? (sp.blk_count - warp + kDecWarps - 1) / kDecWarps : 0;
  const size_t head_stride = (size_t)kBlock * D;  // elements per (block, head)

  auto issue = [&](int k) {
    const int bi = sp.blk_begin + warp + kDecWarps * k;
    const int phys = p.blist[bi];
    const int st = k % kDecStages;
    uint8_t* dst = ring + st * S::kStageBytes;
    const size_t off = ((size_t)phys * p.Hkv + g) * head_stride;
    mbar_arrive_expect_tx(&full_bar[warp][st], 2 * S::kBlkBytes);
    bulk_load(dst, p.k_pool + off, S::kBlkBytes, &full_bar[warp][st]);
    bulk_load(dst + S::kBlkBytes, p.v_pool + off, S::kBlkBytes, &full_bar[warp][st]);
  };

  if (lane == 0) {
    for (int k = 0; k < kDecStages && k < nb_w; ++k) issue(k);
  }
  __syncwarp();

  float m_run = -INFINITY, l_run = 0.f;  // per lane: head (lane % GH)
  float o[GH][DL];
#pragma unroll
  for (int hh = 0; hh < GH; ++hh)
#pragma unroll
    for (int i = 0; i < DL; ++i) o[hh][i] = 0.f;

  int k = 0;
  bool aborted = false;
  for (; k < nb_w; ++k) {
    const int st = k % kDecStages;
    const int bi = sp.blk_begin + warp + kDecWarps * k;
    const int fill = p.bfill[bi];
    if (!mbar_wait(&full_bar[warp][st], (k / kDecStages) & 1, p.wait_ns)) {
      set_status(p.status, MSA_ERR_TIMEOUT);
      aborted = true;
      break;
    }
    const __nv_bfloat16* Ks = reinterpret_cast<const __nv_bfloat16*>(ring + st * S::kStageBytes);
    const __nv_bfloat16* Vs = Ks + kBlock * D;

    // ---- scores: token t = 4*it + tg, lanes sub 0..7 split d
#pragma unroll
    for (int it = 0; it < kBlock / 4; ++it) {
      const int t = it * 4 + tg;
      const uint4* kr = reinterpret_cast<const uint4*>(Ks + t * D + sub * SL);
      float acc[GH];
#pragma unroll
      for (int hh = 0; hh < GH; ++hh) acc[hh] = 0.f;
#pragma unroll
      for (int c = 0; c < SL / 8; ++c) {
        uint4 w = kr[c];
        uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float k0 = bf16_lo(ws[e]), k1 = bf16_hi(ws[e]);
#pragma unroll
          for (int hh = 0; hh < GH; ++hh) {
            acc[hh] = fmaf(qf[hh][c * 8 + 2 * e], k0, acc[hh]);
            acc[hh] = fmaf(qf[hh][c * 8 + 2 * e + 1], k1, acc[hh]);
          }
        }
      }
#pragma unroll
      for (int hh = 0; hh < GH; ++hh) {
        acc[hh] += __shfl_xor_sync(0xffffffffu, acc[hh], 1);
        acc[hh] += __shfl_xor_sync(0xffffffffu, acc[hh], 2);
        acc[hh] += __shfl_xor_sync(0xffffffffu, acc[hh], 4);
      }
      if (sub < GH) {
        float v = acc[0];
#pragma unroll
        for (int hh = 1; hh < GH; ++hh)
          if (sub == hh) v = acc[hh];
        sc[warp][t * GH + sub] = (t < fill) ? v : -INFINITY;
      }
    }
    __syncwarp();

    // ---- online softmax over this block (log2 units)
    float x[EPL];
    float mx = -INFINITY;
#pragma unroll
    for (int j = 0; j < EPL; ++j) {
      const int e = lane + 32 * j;
      x[j] = (e < NS) ? sc[warp][e] : -INFINITY;
      mx = fmaxf(mx, x[j]);
    }
#pragma unroll
    for (int msk = GH; msk < 32; msk <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, msk));
    const float m_new = fmaxf(m_run, mx);
    const float factor = (m_run == -INFINITY) ? 0.f : fast_exp2(m_run - m_new);
    float lsum = 0.f;
#pragma unroll
    for (int j = 0; j < EPL; ++j) {
      const int e = lane + 32 * j;
      const float pe = fast_exp2(x[j] - m_new);
      if (e < NS) ps[warp][e] = pe;
      lsum += (e < NS) ? pe : 0.f;
    }
    l_run = l_run * factor + lsum;
    m_run = m_new;
    if (lane < GH) fs[warp][lane] = factor;
    __syncwarp();

    // ---- P.V: lane owns d-slice [lane*DL, lane*DL + DL)
#pragma unroll
    for (int hh = 0; hh < GH; ++hh) {
      const float f = fs[warp][hh];
#pragma unroll
      for (int i = 0; i < DL; ++i) o[hh][i] *= f;
    }
#pragma unroll 4
    for (int t = 0; t < fill; ++t) {
      float vv[DL];
      if constexpr (DL == 4) {
        uint2 w = *reinterpret_cast<const uint2*>(Vs + t * D + lane * 4);
        vv[0] = bf16_lo(w.x);
        vv[1] = bf16_hi(w.x);
        vv[2] = bf16_lo(w.y);
        vv[3] = bf16_hi(w.y);
      } else {
        uint32_t w = *reinterpret_cast<const uint32_t*>(Vs + t * D + lane * 2);
        vv[0] = bf16_lo(w);
        vv[1] = bf16_hi(w);
      }
#pragma unroll
      for (int hh = 0; hh < GH; ++hh) {
        const float pp = ps[warp][t * GH + hh];
#pragma unroll
        for (int i = 0; i < DL; ++i) o[hh][i] = fmaf(pp, vv[i], o[hh][i]);
      }
    }
    __syncwarp();
    if (lane == 0 && k + kDecStages < nb_w) issue(k + kDecStages);
    __syncwarp();
  }
  if (aborted) {
    // let the copies this warp still has in flight land before the CTA exits
    const int issued = nb_w < k + kDecStages ? nb_w : k + kDecStages;
    for (int kk = k; kk < issued; ++kk)
      mbar_wait(&full_bar[warp][kk % kDecStages], (kk / kDecStages) & 1, 1000000000ull);
  }

  // ---- combine lanes (l) and warps (m, l, O) in shared memory (the rings are idle now)
#pragma unroll
  for (int msk = GH; msk < 32; msk <<= 1) l_run += __shfl_xor_sync(0xffffffffu, l_run, msk);
  __syncthreads();
  float* mw = reinterpret_cast<float*>(smem);             // [warps][GH]
  float* lw = mw + kDecWarps * GH;                         // [warps][GH]
  float* ow = lw + kDecWarps * GH;                         // [warps][GH][D]
  if (lane < GH) {
    mw[warp * GH + lane] = m_run;
    lw[warp * GH + lane] = l_run;
  }
#pragma unroll
  for (int hh = 0; hh < GH; ++hh)
#pragma unroll
    for (int i = 0; i < DL; ++i) ow[(warp * GH + hh) * D + lane * DL + i] = o[hh][i];
  __syncthreads();

  const size_t gsplit = blockIdx.x;
  const bool single = sp.nsplit == 1;
  for (int idx = tid; idx < GH * D; idx += kDecWarps * 32) {
    const int hh = idx / D, i = idx % D;
    float m = -INFINITY;
#pragma unroll
    for (int w = 0; w < kDecWarps; ++w) m = fmaxf(m, mw[w * GH + hh]);
    float L = 0.f, acc = 0.f;
#pragma unroll
    for (int w = 0; w < kDecWarps; ++w) {
      const float mwv = mw[w * GH + hh];
      const float wt = (mwv == -INFINITY) ? 0.f : fast_exp2(mwv - m);
      L += wt * lw[w * GH + hh];
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
  const int smem = DecSmem<D>::kRingBytes;
  cudaError_t e = cudaFuncSetAttribute(msa_decode_kernel<D, GH>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  dim3 grid(n_split, head_groups);
  msa_decode_kernel<D, GH><<<grid, kDecWarps * 32, smem, stream>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_decode(const DecodeParams& p, int d, int n_split, cudaStream_t stream) {
  const int G = p.G;
  const int GH = (G % 4 == 0) ? 4 : (G % 2 == 0 ? 2 : 1);
  const int groups = p.Hkv * (G / GH);
  if (d == 128) {
    if (GH == 4) return launch_decode_t<128, 4>(p, n_split, groups, stream);
    if (GH == 2) return launch_decode_t<128, 2>(p, n_split, groups, stream);
    return launch_decode_t<128, 1>(p, n_split, groups, stream);
  }
  if (GH == 4) return launch_decode_t<64, 4>(p, n_split, groups, stream);
  if (GH == 2) return launch_decode_t<64, 2>(p, n_split, groups, stream);
  return launch_decode_t<64, 1>(p, n_split, groups, stream);
}

}  // namespace msa
