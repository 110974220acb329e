// C ABI entry points of libmsa.so that touch the GPU: plan upload, workspace set-up,
// the prefill / decode / merge / gather launches and the device status word.
#include <cuda_runtime.h>

#include <atomic>

#include "msa_kernels.h"

using namespace msa;

namespace {
constexpr uint64_t kDefaultWaitNs = 2000000000ull;  // 2 s per wait
std::atomic<uint64_t> g_wait_ns{kDefaultWaitNs};
// test hook: which kernel leaves out a copy, in which CTA, and which copy (-1: none)
std::atomic<int32_t> g_drop_kernel{-1}, g_drop_cta{-1}, g_drop_index{-1};

inline bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

template <typename T>
inline const T* at(const void* base, size_t off) {
  return reinterpret_cast<const T*>(reinterpret_cast<const char*>(base) + off);
}
}  // namespace

extern "C" void msa_set_wait_limit(int64_t ns) { g_wait_ns = ns > 0 ? (uint64_t)ns : kDefaultWaitNs; }

extern "C" void msa_set_test_drop(int32_t kernel, int32_t cta, int32_t index) {
  const bool on = (kernel == 0 || kernel == 1) && cta >= 0 && index >= 0;
  g_drop_kernel = on ? kernel : -1;
  g_drop_cta = on ? cta : -1;
  g_drop_index = on ? index : -1;
}

namespace msa {
uint64_t wait_limit_ns() { return g_wait_ns.load(); }
void test_drop(int kernel, int32_t* cta, int32_t* index) {
  const bool on = g_drop_kernel.load() == kernel;
  *cta = on ? g_drop_cta.load() : -1;
  *index = on ? g_drop_index.load() : -1;
}
}  // namespace msa

extern "C" msa_status_t msa_plan_upload(const msa_plan_t* plan, void* plan_dev, size_t bytes,
                                        cudaStream_t stream) {
  if (!plan || !plan_dev || !aligned(plan_dev, 16)) return MSA_ERR_INVALID_ARG;
  if (bytes < plan->dev.total) return MSA_ERR_WORKSPACE;
  if (cudaMemcpyAsync(plan_dev, plan->image.data(), plan->dev.total, cudaMemcpyHostToDevice, stream) !=
      cudaSuccess)
    return MSA_ERR_CUDA;
  return MSA_OK;
}

extern "C" msa_status_t msa_workspace_init(void* workspace, size_t bytes, cudaStream_t stream) {
  if (!workspace || !aligned(workspace, 256)) return MSA_ERR_INVALID_ARG;
  if (cudaMemsetAsync(workspace, 0, bytes, stream) != cudaSuccess) return MSA_ERR_CUDA;
  return MSA_OK;
}

extern "C" msa_status_t msa_get_status(void* workspace, cudaStream_t stream) {
  if (!workspace) return MSA_ERR_INVALID_ARG;
  int32_t word = 0;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return MSA_ERR_CUDA;
  if (cudaMemcpy(&word, workspace, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess) return MSA_ERR_CUDA;
  if (word != 0) {
    const int32_t zero = 0;
    if (cudaMemcpy(workspace, &zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess) return MSA_ERR_CUDA;
  }
  return (msa_status_t)word;
}

extern "C" msa_status_t msa_prefill(const msa_plan_t* plan, const void* plan_dev, const void* q,
                                    const void* k_chunk, const void* v_chunk, const void* k_pool,
                                    const void* v_pool, void* out, float* lse, float scale, void* workspace,
                                    size_t ws_bytes, cudaStream_t stream) {
  if (!plan) return MSA_ERR_INVALID_ARG;
  if (plan->mode != MSA_PREFILL) return MSA_ERR_MODE;
  if (plan->total_q == 0 || plan->n_work == 0) return MSA_OK;
  if (!plan_dev || !q || !k_chunk || !v_chunk || !out || !lse || !workspace) return MSA_ERR_INVALID_ARG;
  const void* ptrs[] = {plan_dev, q, k_chunk, v_chunk, out, lse};
  for (const void* p : ptrs)
    if (!aligned(p, 16)) return MSA_ERR_INVALID_ARG;
  if ((k_pool && !aligned(k_pool, 16)) || (v_pool && !aligned(v_pool, 16))) return MSA_ERR_INVALID_ARG;
  if (ws_bytes < plan->ws.total || !aligned(workspace, 256)) return MSA_ERR_WORKSPACE;
  const int64_t pool_blocks = plan->num_pool_blocks;
  if (pool_blocks > 0 && (!k_pool || !v_pool)) return MSA_ERR_INVALID_ARG;
  PrefillParams p{};
  p.qpos = at<int32_t>(plan_dev, plan->dev.qpos);
  p.qt = at<QTileRec>(plan_dev, plan->dev.qtile);
  p.kt = at<KTileRec>(plan_dev, plan->dev.ktile);
  p.list = at<int32_t>(plan_dev, plan->dev.list);
  p.work = at<WorkRec>(plan_dev, plan->dev.work);
  p.cta_begin = at<int32_t>(plan_dev, plan->dev.cta);
  p.out = reinterpret_cast<__nv_bfloat16*>(out);
  p.lse = lse;
  char* ws = reinterpret_cast<char*>(workspace);
  p.part_o = reinterpret_cast<float4*>(ws + plan->ws.pf_part_o);
  p.part_ml = reinterpret_cast<float2*>(ws + plan->ws.pf_part_ml);
  p.counters = reinterpret_cast<int32_t*>(ws + plan->ws.pf_counters);
  p.status = reinterpret_cast<int32_t*>(ws + plan->ws.status);
  p.n_ctas = plan->n_ctas;
  p.Hq = plan->Hq;
  p.Hkv = plan->Hkv;
  p.hpc = plan->hpc;
  p.pool_rows = (int32_t)(pool_blocks * plan->Hkv * kBlock);
  p.scale_log2 = scale * 1.4426950408889634f;
  p.wait_ns = g_wait_ns.load();
  test_drop(0, &p.drop_cta, &p.drop_k);
  p.n_qt = plan->n_qt;
  p.n_kt = plan->n_kt;
  p.n_list = plan->n_list;
  p.total_q = plan->total_q;
  p.num_pool_blocks = plan->num_pool_blocks;
  PrefillTensors T{q, k_chunk, v_chunk, k_pool, v_pool, plan->total_q, pool_blocks, plan->d};
  return launch_prefill(p, T, stream) == cudaSuccess ? MSA_OK : MSA_ERR_CUDA;
}

extern "C" msa_status_t msa_decode(const msa_plan_t* plan, const void* plan_dev, const void* q,
                                   const void* k_pool, const void* v_pool, void* out, float* lse, float scale,
                                   void* workspace, size_t ws_bytes, cudaStream_t stream) {
  if (!plan) return MSA_ERR_INVALID_ARG;
  if (plan->mode != MSA_DECODE) return MSA_ERR_MODE;
  if (!plan_dev || !q || !k_pool || !v_pool || !out || !lse || !workspace) return MSA_ERR_INVALID_ARG;
  const void* ptrs[] = {plan_dev, q, k_pool, v_pool, out, lse};
  for (const void* p : ptrs)
    if (!aligned(p, 16)) return MSA_ERR_INVALID_ARG;
  if (ws_bytes < plan->ws.total || !aligned(workspace, 256)) return MSA_ERR_WORKSPACE;
  if (plan->n_split == 0) return MSA_OK;
  char* ws = reinterpret_cast<char*>(workspace);
  DecodeParams p{};
  p.split = at<SplitRec>(plan_dev, plan->dev.split);
  p.blist = at<int32_t>(plan_dev, plan->dev.blist);
  p.bfill = at<int32_t>(plan_dev, plan->dev.bfill);
  p.q = reinterpret_cast<const __nv_bfloat16*>(q);
  p.k_pool = reinterpret_cast<const __nv_bfloat16*>(k_pool);
  p.v_pool = reinterpret_cast<const __nv_bfloat16*>(v_pool);
  p.out = reinterpret_cast<__nv_bfloat16*>(out);
  p.lse = lse;
  p.part_o = reinterpret_cast<float*>(ws + plan->ws.part_o);
  p.part_lse = reinterpret_cast<float*>(ws + plan->ws.part_lse);
  p.counters = reinterpret_cast<int32_t*>(ws + plan->ws.counters);
  p.status = reinterpret_cast<int32_t*>(ws + plan->ws.status);
  p.Hq = plan->Hq;
  p.Hkv = plan->Hkv;
  p.G = plan->G;
  p.pool_rows = (int64_t)plan->num_pool_blocks * plan->Hkv * kBlock;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.wait_ns = g_wait_ns.load();
  test_drop(1, &p.drop_split, &p.drop_k);
  p.n_blist = plan->n_blist;
  p.num_pool_blocks = plan->num_pool_blocks;
  p.num_seqs = plan->num_seqs;
  return launch_decode(p, plan->d, plan->n_split, stream) == cudaSuccess ? MSA_OK : MSA_ERR_CUDA;
}

extern "C" msa_status_t msa_merge_lse(const float* o_a, const float* lse_a, const float* o_b,
                                      const float* lse_b, void* o, float* lse, int32_t rows, int32_t heads,
                                      int32_t head_dim, cudaStream_t stream) {
  if (rows < 0 || heads <= 0 || head_dim <= 0 || head_dim % 4 != 0) return MSA_ERR_INVALID_ARG;
  if (rows == 0) return MSA_OK;
  if (!o_a || !lse_a || !o_b || !lse_b || !o || !lse) return MSA_ERR_INVALID_ARG;
  if (!aligned(o_a, 16) || !aligned(o_b, 16) || !aligned(o, 8)) return MSA_ERR_INVALID_ARG;
  return launch_merge_lse(o_a, lse_a, o_b, lse_b, o, lse, (int64_t)rows * heads, head_dim, stream) == cudaSuccess
             ? MSA_OK
             : MSA_ERR_CUDA;
}

extern "C" msa_status_t msa_gather(const msa_plan_t* plan, const void* plan_dev, const void* k_chunk,
                                   const void* v_chunk, const void* k_pool, const void* v_pool, void* k_out,
                                   void* v_out, int32_t* pos_out, size_t out_tokens, cudaStream_t stream) {
  if (!plan || !plan_dev || !k_out || !v_out) return MSA_ERR_INVALID_ARG;
  if (out_tokens < (size_t)plan->n_tok) return MSA_ERR_WORKSPACE;
  if (plan->mode == MSA_PREFILL && plan->total_q > 0 && (!k_chunk || !v_chunk)) return MSA_ERR_INVALID_ARG;
  const void* ptrs[] = {plan_dev, k_out, v_out, k_chunk, v_chunk, k_pool, v_pool};
  for (const void* p : ptrs)
    if (p && !aligned(p, 16)) return MSA_ERR_INVALID_ARG;
  GatherParams p{};
  p.units = at<GatherRec>(plan_dev, plan->dev.gather);
  p.qpos = at<int32_t>(plan_dev, plan->dev.qpos);
  p.k_chunk = reinterpret_cast<const uint4*>(k_chunk);
  p.v_chunk = reinterpret_cast<const uint4*>(v_chunk);
  p.k_pool = reinterpret_cast<const uint4*>(k_pool);
  p.v_pool = reinterpret_cast<const uint4*>(v_pool);
  p.k_out = reinterpret_cast<uint4*>(k_out);
  p.v_out = reinterpret_cast<uint4*>(v_out);
  p.pos_out = pos_out;
  p.Hkv = plan->Hkv;
  p.d = plan->d;
  return launch_gather(p, plan->n_gather, stream) == cudaSuccess ? MSA_OK : MSA_ERR_CUDA;
}

extern "C" msa_status_t msa_kv_append(const int32_t* dst_slot, const void* k_chunk, const void* v_chunk,
                                      void* k_pool, void* v_pool, int32_t n, int32_t num_heads_kv,
                                      int32_t head_dim, int32_t num_pool_blocks, cudaStream_t stream) {
  if (n < 0 || num_heads_kv <= 0 || num_pool_blocks < 0) return MSA_ERR_INVALID_ARG;
  if (head_dim != 64 && head_dim != 128) return MSA_ERR_UNSUPPORTED;
  if (n == 0) return MSA_OK;
  if (!dst_slot || !k_chunk || !v_chunk || !k_pool || !v_pool) return MSA_ERR_INVALID_ARG;
  const void* ptrs[] = {dst_slot, k_chunk, v_chunk, k_pool, v_pool};
  for (const void* p : ptrs)
    if (!aligned(p, 16)) return MSA_ERR_INVALID_ARG;
  return launch_kv_append(dst_slot, k_chunk, v_chunk, k_pool, v_pool, n, num_heads_kv, head_dim, num_pool_blocks,
                          stream) == cudaSuccess
             ? MSA_OK
             : MSA_ERR_CUDA;
}
