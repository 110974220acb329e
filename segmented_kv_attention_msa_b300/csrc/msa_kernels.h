// Parameter blocks and launchers of the MSA kernels (internal to libmsa.so).
#pragma once
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "msa_internal.h"

namespace msa {

struct PrefillParams {
  const int32_t* qpos;
  const QTileRec* qt;
  const KTileRec* kt;
  const int32_t* list;
  const WorkRec* work;
  const int32_t* cta_begin;  // pieces of CTA c: work[cta_begin[c] .. cta_begin[c + 1])
  __nv_bfloat16* out;
  float* lse;
  float4* part_o;            // split items: unnormalised O per (slot, head), [d/4][128] float4
  float2* part_ml;           // split items: (max in log2 units, sum) per (slot, head, row)
  int32_t* counters;         // split items: pieces finished per (first slot, head)
  int32_t* status;
  int32_t n_ctas, Hq, Hkv, hpc;
  int32_t pool_rows;  // rows of the pool tensor maps; a box starting here reads zeros
  float scale_log2;
  uint64_t wait_ns;
  int32_t drop_cta, drop_k;  // test hook: CTA drop_cta leaves out its K tile number drop_k (-1: none)
  int32_t n_qt, n_kt, n_list, total_q, num_pool_blocks;  // bounds checked by the MSA_DEBUG build
};

struct PrefillTensors {
  const void *q, *k_chunk, *v_chunk, *k_pool, *v_pool;
  int64_t total_q, num_pool_blocks;
  int d;
};

struct DecodeParams {
  const SplitRec* split;
  const int32_t* blist;
  const int32_t* bfill;
  const __nv_bfloat16* q;
  const __nv_bfloat16* k_pool;
  const __nv_bfloat16* v_pool;
  __nv_bfloat16* out;
  float* lse;
  float* part_o;
  float* part_lse;
  int32_t* counters;
  int32_t* status;
  int32_t Hq, Hkv, G;
  int64_t pool_rows;  // rows of the pool tensors seen as [num_blocks * Hkv * 16][d]
  float scale_log2;
  uint64_t wait_ns;
  int32_t drop_split, drop_k;  // test hook: warp 0 of CTA (drop_split, 0) leaves out its block drop_k (-1: none)
  int32_t n_blist, num_pool_blocks, num_seqs;  // bounds checked by the MSA_DEBUG build
};

struct GatherParams {
  const GatherRec* units;
  const int32_t* qpos;
  const uint4* k_chunk;
  const uint4* v_chunk;
  const uint4* k_pool;
  const uint4* v_pool;
  uint4* k_out;
  uint4* v_out;
  int32_t* pos_out;
  int32_t Hkv;
  int32_t d;
};

// Settings shared by every launch (set through the C ABI): the bound of each device wait
// and the test hook that leaves out one copy (kernel 0 = prefill, 1 = decode).
uint64_t wait_limit_ns();
void test_drop(int kernel, int32_t* cta, int32_t* index);

cudaError_t launch_prefill(const PrefillParams& p, const PrefillTensors& T, cudaStream_t stream);
cudaError_t launch_decode(const DecodeParams& p, int d, int n_split, cudaStream_t stream);
cudaError_t launch_merge_lse(const float* oa, const float* la, const float* ob, const float* lb, void* o,
                             float* lse, int64_t n_rh, int d, cudaStream_t stream);
cudaError_t launch_gather(const GatherParams& p, int n_units, cudaStream_t stream);
cudaError_t launch_kv_append(const int32_t* dst_slot, const void* kc, const void* vc, void* kp, void* vp, int64_t n,
                             int Hkv, int d, int64_t pool_blocks, cudaStream_t stream);

}  // namespace msa
