// Stand-alone LSE merge of two partial attention results, and the bit-exact gather
// of each sequence's KV context into original-position order.
#include <cuda_runtime.h>

#include "msa_device.cuh"
#include "msa_kernels.h"

namespace msa {

// Two attention results over disjoint key sets combine exactly through their
// log-sum-exp: with m = max(lse_a, lse_b) and w = exp(lse - m),
// O = (w_a O_a + w_b O_b) / (w_a + w_b), LSE = m + ln(w_a + w_b).
// One thread per (row, head, 4 elements of d).
__global__ void msa_merge_lse_kernel(const float4* __restrict__ oa, const float* __restrict__ la,
                                     const float4* __restrict__ ob, const float* __restrict__ lb,
                                     __nv_bfloat16* __restrict__ o, float* __restrict__ lse,
                                     int64_t n_rh, int d4) {
  const int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= n_rh * d4) return;
  const int64_t rh = idx / d4;
  const int c = (int)(idx % d4);
  const float a = la[rh], b = lb[rh];
  const float m = fmaxf(a, b);
  float4 r = make_float4(0.f, 0.f, 0.f, 0.f);
  float l = -INFINITY;
  if (m != -INFINITY) {
    const float wa = (a == -INFINITY) ? 0.f : expf(a - m);
    const float wb = (b == -INFINITY) ? 0.f : expf(b - m);
    const float inv = 1.f / (wa + wb);
    const float4 va = oa[idx], vb = ob[idx];
    r.x = (wa * va.x + wb * vb.x) * inv;
    r.y = (wa * va.y + wb * vb.y) * inv;
    r.z = (wa * va.z + wb * vb.z) * inv;
    r.w = (wa * va.w + wb * vb.w) * inv;
    l = m + logf(wa + wb);
  }
  __nv_bfloat162 lo = __floats2bfloat162_rn(r.x, r.y), hi = __floats2bfloat162_rn(r.z, r.w);
  uint2 packed;
  packed.x = *reinterpret_cast<uint32_t*>(&lo);
  packed.y = *reinterpret_cast<uint32_t*>(&hi);
  reinterpret_cast<uint2*>(o)[idx] = packed;
  if (c == 0) lse[rh] = l;
}

cudaError_t launch_merge_lse(const float* oa, const float* la, const float* ob, const float* lb, void* o,
                             float* lse, int64_t n_rh, int d, cudaStream_t stream) {
  const int d4 = d / 4;
  const int64_t n = n_rh * d4;
  if (n == 0) return cudaSuccess;
  const int threads = 256;
  const int64_t blocks = (n + threads - 1) / threads;
  msa_merge_lse_kernel<<<(unsigned)blocks, threads, 0, stream>>>(
      reinterpret_cast<const float4*>(oa), la, reinterpret_cast<const float4*>(ob), lb,
      reinterpret_cast<__nv_bfloat16*>(o), lse, n_rh, d4);
  return cudaGetLastError();
}

// Write-back: every (row, KV head, 16-byte piece) of the chunk's K and V moves to its
// pool slot; reads coalesced along the chunk row, writes along the pool row.  A thread
// moves kAppendPer pieces kAppendThreads apart, all loads before any store, so that each
// thread keeps several DRAM reads in flight.  A negative slot skips the row; a slot past
// the pool is ignored.
constexpr int kAppendPer = 4, kAppendThreads = 256;
__global__ void __launch_bounds__(kAppendThreads)
    msa_kv_append_kernel(const int32_t* __restrict__ dst_slot, const uint4* __restrict__ kc,
                         const uint4* __restrict__ vc, uint4* __restrict__ kp, uint4* __restrict__ vp, int64_t n,
                         int Hkv, int d8, int64_t pool_slots) {
  const int64_t per_row = (int64_t)Hkv * d8;
  const int64_t total = n * per_row;
  const int64_t base = (int64_t)blockIdx.x * (kAppendThreads * kAppendPer) + threadIdx.x;
  uint4 kr[kAppendPer], vr[kAppendPer];
  int64_t dst[kAppendPer];
#pragma unroll
  for (int k = 0; k < kAppendPer; ++k) {
    const int64_t idx = base + (int64_t)k * kAppendThreads;
    dst[k] = -1;
    if (idx < total) {
      const int64_t row = idx / per_row;
      const int rem = (int)(idx % per_row);
      const int g = rem / d8, c = rem % d8;
      const int64_t slot = dst_slot[row];
      if (slot >= 0 && slot < pool_slots) {
        const int64_t blk = slot / kBlock, t = slot % kBlock;
        dst[k] = ((blk * Hkv + g) * kBlock + t) * d8 + c;
        kr[k] = kc[idx];
        vr[k] = vc[idx];
      }
    }
  }
#pragma unroll
  for (int k = 0; k < kAppendPer; ++k)
    if (dst[k] >= 0) {
      kp[dst[k]] = kr[k];
      vp[dst[k]] = vr[k];
    }
}

cudaError_t launch_kv_append(const int32_t* dst_slot, const void* kc, const void* vc, void* kp, void* vp, int64_t n,
                             int Hkv, int d, int64_t pool_blocks, cudaStream_t stream) {
  const int d8 = d / 8;
  const int64_t total = n * Hkv * d8;
  if (total == 0) return cudaSuccess;
  const int threads = kAppendThreads;
  const int64_t blocks = (total + threads * kAppendPer - 1) / (threads * kAppendPer);
  msa_kv_append_kernel<<<(unsigned)blocks, threads, 0, stream>>>(
      dst_slot, reinterpret_cast<const uint4*>(kc), reinterpret_cast<const uint4*>(vc), reinterpret_cast<uint4*>(kp),
      reinterpret_cast<uint4*>(vp), n, Hkv, d8, pool_blocks * kBlock);
  return cudaGetLastError();
}

// Gather: one CTA per gather unit (a pool block or a run of consecutive chunk rows);
// copies its tokens' K and V rows for every KV head with 16-byte moves, each thread
// loading kGatherPer pieces of K and of V before it stores any, so that several DRAM
// reads per thread are in flight.
constexpr int kGatherPer = 4, kGatherThreads = 128;
__global__ void __launch_bounds__(kGatherThreads) msa_gather_kernel(const GatherParams p) {
  const GatherRec u = p.units[blockIdx.x];
  const int row_vec = p.d / 8;  // uint4 per (token, head) row
  const int per_tok = p.Hkv * row_vec;
  const int total = u.n * per_tok;
  const bool pool = u.src == SRC_POOL;
  const uint4* __restrict__ ks = pool ? p.k_pool : p.k_chunk;
  const uint4* __restrict__ vs = pool ? p.v_pool : p.v_chunk;
  uint4* __restrict__ ko = p.k_out;
  uint4* __restrict__ vo = p.v_out;
  for (int i0 = threadIdx.x; i0 < total; i0 += kGatherThreads * kGatherPer) {
    uint4 kr[kGatherPer], vr[kGatherPer];
    size_t dst[kGatherPer];
#pragma unroll
    for (int k = 0; k < kGatherPer; ++k) {
      const int i = i0 + k * kGatherThreads;
      if (i < total) {
        const int t = i / per_tok;
        const int rem = i % per_tok;
        const int g = rem / row_vec, c = rem % row_vec;
        dst[k] = ((size_t)(u.out_row + t) * p.Hkv + g) * row_vec + c;
        const size_t src = pool ? (((size_t)u.id * p.Hkv + g) * kBlock + t) * row_vec + c
                                : ((size_t)(u.id + t) * p.Hkv + g) * row_vec + c;
        kr[k] = ks[src];
        vr[k] = vs[src];
      }
    }
#pragma unroll
    for (int k = 0; k < kGatherPer; ++k)
      if (i0 + k * kGatherThreads < total) {
        ko[dst[k]] = kr[k];
        vo[dst[k]] = vr[k];
      }
  }
  if (p.pos_out)
    for (int t = threadIdx.x; t < u.n; t += blockDim.x)
      p.pos_out[u.out_row + t] = (u.src == SRC_POOL) ? u.pos0 + t : p.qpos[u.id + t];
}

cudaError_t launch_gather(const GatherParams& p, int n_units, cudaStream_t stream) {
  if (n_units == 0) return cudaSuccess;
  msa_gather_kernel<<<n_units, kGatherThreads, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace msa
