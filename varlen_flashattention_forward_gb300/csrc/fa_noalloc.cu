// fa_noalloc.cu -- fa_sparse_mla_decode_noalloc (include/fa_gb300.h): the
// sparse-MLA decode with its partial-result workspace taken from a fixed
// scratch buffer in device memory instead of an allocation.
//
// The buffer is a file-scope __device__ array in its own translation unit.
// Under lazy module loading (CUDA_MODULE_LOADING=LAZY, the default since CUDA
// 12.2) its device memory is committed on a device only when the first call
// there loads the module; under eager loading, every process that loads the
// library commits it on every device it uses, whether or not it calls this
// entry point.
#include <cstdint>
#include <mutex>

#include <cuda_runtime.h>

#include "../../include/fa_gb300.h"
#include "decode_plan.h"

namespace {

constexpr size_t kScratchBytes = FA_NOALLOC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

std::mutex g_mu;
void* g_scratch[kMaxDevices] = {};

// Device address of the scratch on the current device, looked up once per
// device with that device current and kept for the life of the process (a
// cudaDeviceReset invalidates it; the header forbids calls after one).
fa_status scratch_address(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return FA_ERR_LAUNCH;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return FA_ERR_LAUNCH;
    g_scratch[dev] = p;
  }
  *out = g_scratch[dev];
  return FA_OK;
}

}  // namespace

extern "C" fa_status fa_sparse_mla_decode_noalloc(const void* q, const void* kv_cache,
                                                  const int* page_table, const int* topk_idx,
                                                  int num_tokens, int num_heads, int topk,
                                                  int num_pages, int max_pages_per_tok,
                                                  float softmax_scale, void* out, float* lse,
                                                  fa_stream_t stream) {
  alignas(128) unsigned char plan[fa::kDecodePlanBytes];
  size_t ws_bytes = 0;
  bool launch = false;
  fa_status st = fa::decode_plan(q, kv_cache, page_table, topk_idx, num_tokens, num_heads, topk,
                                 num_pages, max_pages_per_tok, softmax_scale, out, lse, plan,
                                 &ws_bytes, &launch);
  if (st != FA_OK || !launch) return st;
  void* ws = nullptr;
  if (ws_bytes > 0) {
    if (ws_bytes > kScratchBytes) return FA_ERR_SCRATCH;
    st = scratch_address(&ws);
    if (st != FA_OK) return st;
  }
  return fa::decode_launch(plan, ws, reinterpret_cast<cudaStream_t>(stream));
}
