// sparse_decode_kernel.cuh -- sparse-MLA decode (kernel not yet in place:
// the launcher reports cudaErrorNotSupported, which the API maps to
// FA_ERR_LAUNCH).
#pragma once
#include <cstdint>
#include <cuda_runtime.h>

namespace fa {
constexpr int kDecodePage = 64;
struct DecodeArgs {
  const uint16_t* q;
  const uint16_t* cache;
  const int* page_table;
  const int* topk_idx;
  int num_tokens, num_heads, topk, num_pages, max_pages;
  float scale_log2;
  uint16_t* out;
  float* lse;
  unsigned int* status;
};
inline cudaError_t launch_sparse_decode(const DecodeArgs&, int, cudaStream_t) {
  return cudaErrorNotSupported;
}
}  // namespace fa
