// Test probe: the sm_103 reducing TMEM load (tcgen05.ld.red ... .max.f32, as
// wrapped by fa::ptx::tmem_ld32_max and used by the varlen softmax for the
// row max of unmasked tiles) must return the 32 stored values unchanged and
// a maximum bitwise equal to the software maximum of the same values.  One
// CTA of 128 threads; each thread owns TMEM lane = thread and writes 128
// fp32 values into columns [0, 128) of a 512-column allocation, including
// all -inf chunks and single -inf values (no -0, whose sign a maximum may
// take from either operand).  Exit status 0 on success.
#include <cmath>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <vector>

#include <cuda_runtime.h>

#include "sm103_ptx.cuh"

using namespace fa::ptx;

#define CK(x)                                                                  \
  do {                                                                         \
    cudaError_t e_ = (x);                                                      \
    if (e_ != cudaSuccess) {                                                   \
      std::printf("CUDA error %s: %s\n", #x, cudaGetErrorString(e_));         \
      return 2;                                                                \
    }                                                                          \
  } while (0)

__global__ void probe(const float* in, float* vals, float* hw_max, float* sw_max) {
  __shared__ uint32_t tbase;
  const int tid = threadIdx.x, warp = tid / 32;
  if (warp == 0) {
    tmem_alloc(smem_u32(&tbase), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tm = tbase + ((uint32_t)(warp * 32) << 16);
  for (int q = 0; q < 4; ++q) {
    uint32_t v[32];
    for (int c = 0; c < 32; ++c) v[c] = __float_as_uint(in[tid * 128 + q * 32 + c]);
    tmem_st32(tm + q * 32, v);
  }
  tmem_wait_st();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  for (int q = 0; q < 4; ++q) {
    float r[32], mx;
    tmem_ld32_max(tm + q * 32, r, mx);
    tmem_wait_ld();
    float sw = -INFINITY;
    for (int c = 0; c < 32; ++c) {
      asm volatile("" : "+f"(r[c]));
      vals[tid * 128 + q * 32 + c] = r[c];
      sw = fmaxf(sw, r[c]);
    }
    asm volatile("" : "+f"(mx));
    hw_max[tid * 4 + q] = mx;
    sw_max[tid * 4 + q] = sw;
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tbase, 512);
  }
}

static bool same_bits(float a, float b) {
  uint32_t x, y;
  std::memcpy(&x, &a, 4);
  std::memcpy(&y, &b, 4);
  return x == y;
}

int main() {
  const int n = 128 * 128;
  std::vector<float> in(n);
  std::srand(5);
  for (int i = 0; i < n; ++i) in[i] = (float)((std::rand() % 20001) - 10000) / 37.f;
  for (int t = 0; t < 128; t += 5)
    for (int c = 0; c < 32; ++c) in[t * 128 + c] = -INFINITY;  // an all -inf chunk
  for (int t = 1; t < 128; t += 7) in[t * 128 + 40] = -INFINITY;  // one -inf value
  float *din, *dv, *dh, *ds;
  CK(cudaMalloc(&din, n * 4));
  CK(cudaMalloc(&dv, n * 4));
  CK(cudaMalloc(&dh, 512 * 4));
  CK(cudaMalloc(&ds, 512 * 4));
  CK(cudaMemcpy(din, in.data(), n * 4, cudaMemcpyHostToDevice));
  probe<<<1, 128>>>(din, dv, dh, ds);
  CK(cudaGetLastError());
  CK(cudaDeviceSynchronize());
  std::vector<float> v(n), h(512), s(512);
  CK(cudaMemcpy(v.data(), dv, n * 4, cudaMemcpyDeviceToHost));
  CK(cudaMemcpy(h.data(), dh, 512 * 4, cudaMemcpyDeviceToHost));
  CK(cudaMemcpy(s.data(), ds, 512 * 4, cudaMemcpyDeviceToHost));
  int bad_v = 0, bad_hw_sw = 0, bad_host = 0;
  for (int i = 0; i < n; ++i) bad_v += !same_bits(v[i], in[i]);
  for (int t = 0; t < 128; ++t)
    for (int q = 0; q < 4; ++q) {
      float e = -INFINITY;
      for (int c = 0; c < 32; ++c) e = std::fmax(e, in[t * 128 + q * 32 + c]);
      bad_hw_sw += !same_bits(h[t * 4 + q], s[t * 4 + q]);
      bad_host += !same_bits(h[t * 4 + q], e);
    }
  std::printf("values %d, hardware vs software max %d, vs host max %d mismatches: %s\n", bad_v,
              bad_hw_sw, bad_host, (bad_v || bad_hw_sw || bad_host) ? "FAIL" : "PASS");
  return (bad_v || bad_hw_sw || bad_host) ? 1 : 0;
}
