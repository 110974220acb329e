// msa_decode_no_alloc: the MSA decode for callers that cannot allocate device memory.
//
// The regular msa_decode needs a caller-allocated workspace for its split-KV partial
// results and merge counters.  Some callers cannot provide one: a serving engine that
// reserves nearly all of HBM for its KV-cache pool at start-up and hands out no further
// device memory, or a latency-critical loop that must not call cudaMalloc/cudaFree
// because those calls can synchronise the whole device.  This entry point takes the
// same inputs and outputs as msa_decode but keeps its scratch in a fixed array that the
// library owns for the life of the process, so it never allocates.
//
// The scratch array is a file-scope __device__ array.  In host code its name is only a
// host-side stand-in, not a device address, so its device address is looked up with
// cudaGetSymbolAddress once per device (with that device current) and passed to the
// kernel.
#include <cuda_runtime.h>

#include <mutex>

#include "msa_kernels.h"

namespace {

// Largest scratch one call may use: status word, merge counters and split partials
// (the plan's msa_workspace_bytes must not exceed this).  Every GPU that loads the
// library holds this much device memory until the process exits.
constexpr size_t kNoAllocScratchBytes = 8u << 20;  // 8 MiB

static __device__ __align__(256) unsigned char g_no_alloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device (set up on first use).
cudaError_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_mutex);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_no_alloc_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return cudaSuccess;
}

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

using namespace msa;

extern "C" msa_status_t msa_decode_no_alloc(const msa_plan_t* plan, const void* plan_dev, const void* q,
                                            const void* k_pool, const void* v_pool, void* out, float* lse,
                                            float scale, cudaStream_t stream) {
  if (!plan) return MSA_ERR_INVALID_ARG;
  if (plan->mode != MSA_DECODE) return MSA_ERR_MODE;
  if (!plan_dev || !q || !k_pool || !v_pool || !out || !lse) return MSA_ERR_INVALID_ARG;
  const void* ptrs[] = {plan_dev, q, k_pool, v_pool, out, lse};
  for (const void* p : ptrs)
    if (!aligned16(p)) return MSA_ERR_INVALID_ARG;
  if (plan->ws.total > kNoAllocScratchBytes) return MSA_ERR_WORKSPACE;  // too many split partials
  if (plan->n_split == 0) return MSA_OK;

  void* scratch = nullptr;
  if (scratch_address(&scratch) != cudaSuccess) return MSA_ERR_CUDA;
  char* ws = reinterpret_cast<char*>(scratch);

  // The array keeps whatever the previous call left; the status word and the merge
  // counters must start at zero.  (A memset is not an allocation.)
  if (cudaMemsetAsync(ws, 0, plan->ws.part_o, stream) != cudaSuccess) return MSA_ERR_CUDA;

  DecodeParams p{};
  p.split = reinterpret_cast<const SplitRec*>(reinterpret_cast<const char*>(plan_dev) + plan->dev.split);
  p.blist = reinterpret_cast<const int32_t*>(reinterpret_cast<const char*>(plan_dev) + plan->dev.blist);
  p.bfill = reinterpret_cast<const int32_t*>(reinterpret_cast<const char*>(plan_dev) + plan->dev.bfill);
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
  p.wait_ns = wait_limit_ns();  // the same bound as every other launch (msa_set_wait_limit)
  test_drop(1, &p.drop_split, &p.drop_k);
  p.n_blist = plan->n_blist;
  p.num_pool_blocks = plan->num_pool_blocks;
  p.num_seqs = plan->num_seqs;
  return launch_decode(p, plan->d, plan->n_split, stream) == cudaSuccess ? MSA_OK : MSA_ERR_CUDA;
}

// The status word sits at the start of the library's scratch array (offset 0 of the
// workspace layout).  Reading it needs no allocation either: a copy into a host int.
extern "C" msa_status_t msa_get_status_no_alloc(cudaStream_t stream) {
  void* scratch = nullptr;
  if (scratch_address(&scratch) != cudaSuccess) return MSA_ERR_CUDA;
  int32_t word = 0;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return MSA_ERR_CUDA;
  if (cudaMemcpy(&word, scratch, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess) return MSA_ERR_CUDA;
  if (word != 0) {
    const int32_t zero = 0;
    if (cudaMemcpy(scratch, &zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess) return MSA_ERR_CUDA;
  }
  return (msa_status_t)word;
}
