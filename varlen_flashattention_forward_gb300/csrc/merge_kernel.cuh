// merge_kernel.cuh -- LSE-weighted merge of two partial attention results.
//
//   L = ln(e^{L_a} + e^{L_b}),   O = e^{L_a - L} O_a + e^{L_b - L} O_b
//
// over the same query rows and disjoint key sets (a context chunk attended
// without a mask and the new tokens attended causally, as in chunked
// prefill).  Source: merge_attn_states on the vLLM page
// "vllm.v1.attention.backends.mla.prefill.flash_attn" (FlashAttnPrefillBackend).
//
// Memory-bound elementwise work: one thread per 8 output elements (16-byte
// loads of both partials and one 16-byte store), grid-stride over all rows.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "sm103_ptx.cuh"

namespace fa {

struct MergeArgs {
  const uint16_t* oa;  // bf16 [T, H, d]
  const float* la;     // [H, T]
  const uint16_t* ob;
  const float* lb;
  uint16_t* out;       // bf16 [T, H, d]
  float* lse;          // [H, T] or null
  int total_q, num_heads, head_dim;
};

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

__global__ void __launch_bounds__(256) merge_states_kernel(const MergeArgs a) {
  const int chunks = a.head_dim >> 3;
  const int64_t total = (int64_t)a.total_q * a.num_heads * chunks;
  const float neg_inf = -__int_as_float(0x7f800000);
  for (int64_t g = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; g < total;
       g += (int64_t)gridDim.x * blockDim.x) {
    const int64_t row = g / chunks;
    const int c = (int)(g - row * chunks);
    const int t = (int)(row / a.num_heads);
    const int h = (int)(row - (int64_t)t * a.num_heads);
    const size_t li = (size_t)h * a.total_q + t;
    const float la = a.la[li], lb = a.lb[li];
    const float m = fmaxf(la, lb);
    uint4 res = make_uint4(0u, 0u, 0u, 0u);
    float L = neg_inf;
    if (m != neg_inf) {
      const float ea = __expf(la - m), eb = __expf(lb - m);
      const float inv = 1.f / (ea + eb);
      const float wa = ea * inv, wb = eb * inv;
      L = m + __logf(ea + eb);
      const size_t off = (size_t)row * a.head_dim + c * 8;
      const uint4 va = *reinterpret_cast<const uint4*>(a.oa + off);
      const uint4 vb = *reinterpret_cast<const uint4*>(a.ob + off);
      const uint32_t xa[4] = {va.x, va.y, va.z, va.w};
      const uint32_t xb[4] = {vb.x, vb.y, vb.z, vb.w};
      uint32_t r[4];
#pragma unroll
      for (int i = 0; i < 4; ++i)
        r[i] = ptx::pack_bf16x2(wa * bf16_lo(xa[i]) + wb * bf16_lo(xb[i]),
                                wa * bf16_hi(xa[i]) + wb * bf16_hi(xb[i]));
      res = make_uint4(r[0], r[1], r[2], r[3]);
    }
    *reinterpret_cast<uint4*>(a.out + (size_t)row * a.head_dim + c * 8) = res;
    if (a.lse && c == 0) a.lse[li] = L;
  }
}

inline cudaError_t launch_merge(const MergeArgs& a, int sm_count, cudaStream_t stream) {
  const int64_t total = (int64_t)a.total_q * a.num_heads * (a.head_dim >> 3);
  int64_t blocks = (total + 255) / 256;
  const int64_t cap = (int64_t)sm_count * 8;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  merge_states_kernel<<<(int)blocks, 256, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace fa
