// Gather ceiling of the sparse-MLA decode structure, without the attention.
//
// Each CTA stands for one decode token: it copies the 2048 rows (576 bf16,
// 1152 bytes each) that the token's top-k selects out of a paged latent cache
// into the same two-stage ring the decode kernel uses -- 64-row tiles of nine
// 64-column chunks (128-byte swizzle), gather threads issuing 16-byte
// cp.async with an evict-first policy, one full barrier per chunk and one free
// barrier per release group of chunks -- while one consumer warp releases each
// group as soon as its chunks have landed (no MMA, no softmax).  The kernel
// gathers with 128 threads; 192 and 256 show what more threads would give.  The rows of a
// CTA are 2048 distinct positions of a 32768-position context laid out on
// 64-row pages drawn from a seeded permutation of 65536 pages (4.8 GB), as in
// the decode workload.  The time of a launch is therefore the most the decode
// kernel's gather can deliver at that CTA count.
//
// Output, one line per configuration:
//   gather ctas=<C> threads=<G>: <us> us <GB/s> GB/s
// Every wait is bounded; a wait that runs out sets a flag, the threads let
// their own copies land and return, and the program reports TIMEOUT and exits
// non-zero.  Test fixture of tests/test_gpu_gather_ceiling.py.
#include <algorithm>
#include <cstdint>
#include <cstdio>
#include <random>
#include <vector>

#include <cuda_runtime.h>

#include "sm103_ptx.cuh"

using namespace fa::ptx;

#define CK(x)                                                                        \
  do {                                                                               \
    cudaError_t e_ = (x);                                                            \
    if (e_ != cudaSuccess) {                                                         \
      printf("CUDA error %s: %s\n", #x, cudaGetErrorString(e_));                     \
      return 1;                                                                      \
    }                                                                                \
  } while (0)

constexpr int kRowsPerCta = 2048, kKeys = 64, kChunks = 9, kChunkBytes = 8192;
constexpr int kRowElems = 576;
constexpr int kGroups = 4;  // chunk c is released with group min(c / 2, 3)
constexpr long long kWaitLimitNs = 2000000000ll;

__device__ __forceinline__ int group_of(int c) { return c < 8 ? c >> 1 : kGroups - 1; }

// Bounded wait on an mbarrier phase; false once the limit or another
// thread's timeout has been seen.
__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity, volatile int* flag) {
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t spin = 0;; ++spin) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((spin & 255u) == 255u) {
      if (*flag) return false;
      if ((long long)(globaltimer_ns() - t0) > kWaitLimitNs) {
        *flag = 1;
        return false;
      }
    }
  }
}

// blockDim = G gather threads + one consumer warp.
template <int G>
__global__ void __launch_bounds__(G + 32, 1)
    gather_ring(const uint16_t* cache, const int* rows, int* flag) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* ring = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  __shared__ uint64_t full[2][kChunks], freeb[2][kGroups];
  __shared__ int srows[kRowsPerCta];
  const int tid = threadIdx.x;
  for (int i = tid; i < kRowsPerCta; i += blockDim.x)
    srows[i] = rows[(size_t)blockIdx.x * kRowsPerCta + i];
  if (tid == 0) {
    for (int s = 0; s < 2; ++s) {
      for (int c = 0; c < kChunks; ++c) mbar_init(smem_u32(&full[s][c]), G);
      for (int g = 0; g < kGroups; ++g) mbar_init(smem_u32(&freeb[s][g]), 1);
    }
    fence_mbar_init();
  }
  __syncthreads();
  volatile int* vflag = flag;
  constexpr int n_tiles = kRowsPerCta / kKeys;
  if (tid < G) {
    const uint64_t read_once = make_policy_evict_first();
    bool ok = true;
    for (int j = 0; j < n_tiles && ok; ++j) {
      const int st = j & 1;
      const uint32_t d0 = smem_u32(ring + st * kChunks * kChunkBytes);
      for (int c = 0; c < kChunks && ok; ++c) {
        // The group that last read this chunk's slot, two tiles ago.
        if (j >= 2 && (c == 0 || group_of(c) != group_of(c - 1)))
          ok = wait_bounded(smem_u32(&freeb[st][group_of(c)]), ((j >> 1) - 1) & 1, vflag);
        if (!ok) break;
        // 64 rows x 8 units of 16 bytes per chunk, spread over G threads.
        for (int e = tid; e < kKeys * 8; e += G) {
          const int r = e >> 3, u = e & 7;
          cp_async_16_hint(d0 + c * kChunkBytes + r * 128 + ((u ^ (r & 7)) << 4),
                           cache + (size_t)srows[j * kKeys + r] * kRowElems + c * 64 + u * 8,
                           read_once);
        }
        cp_async_mbar_arrive(smem_u32(&full[st][c]));
      }
    }
    asm volatile("cp.async.wait_all;" ::: "memory");  // nothing in flight at exit
  } else if (tid == G) {
    bool ok = true;
    for (int j = 0; j < n_tiles && ok; ++j) {
      const int st = j & 1;
      for (int c = 0; c < kChunks && ok; ++c) {
        ok = wait_bounded(smem_u32(&full[st][c]), (j >> 1) & 1, vflag);
        if (ok && (c == kChunks - 1 || group_of(c) != group_of(c + 1)))
          mbar_arrive(smem_u32(&freeb[st][group_of(c)]));
      }
    }
  }
}

int main() {
  const int kPages = 65536, kPageRows = 64, kContextPages = 512;
  const long long nrows = (long long)kPages * kPageRows;
  int nsm = 0;
  CK(cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, 0));
  const int max_ctas = std::max(nsm, 128);
  uint16_t* cache = nullptr;
  CK(cudaMalloc(&cache, (size_t)nrows * kRowElems * 2));
  CK(cudaMemset(cache, 0, (size_t)nrows * kRowElems * 2));
  // Rows: per CTA, 2048 distinct positions of its own 512-page context.
  std::mt19937 rng(1234);
  std::vector<int> perm(kPages);
  for (int p = 0; p < kPages; ++p) perm[p] = p;
  std::shuffle(perm.begin(), perm.end(), rng);
  std::vector<int> rows((size_t)max_ctas * kRowsPerCta);
  std::vector<int> pos(kContextPages * kPageRows);
  for (int b = 0; b < max_ctas; ++b) {
    for (int i = 0; i < (int)pos.size(); ++i) pos[i] = i;
    std::shuffle(pos.begin(), pos.end(), rng);
    for (int k = 0; k < kRowsPerCta; ++k) {
      const int page = perm[(b * kContextPages + pos[k] / kPageRows) % kPages];
      rows[(size_t)b * kRowsPerCta + k] = page * kPageRows + pos[k] % kPageRows;
    }
  }
  for (int r : rows)
    if (r < 0 || r >= nrows) {
      printf("row out of range\n");
      return 1;
    }
  int* drows = nullptr;
  CK(cudaMalloc(&drows, rows.size() * sizeof(int)));
  CK(cudaMemcpy(drows, rows.data(), rows.size() * sizeof(int), cudaMemcpyHostToDevice));
  int* flag = nullptr;
  CK(cudaMalloc(&flag, sizeof(int)));
  CK(cudaMemset(flag, 0, sizeof(int)));
  void* l2_flush = nullptr;
  const size_t flush_bytes = 512u << 20;
  CK(cudaMalloc(&l2_flush, flush_bytes));
  cudaEvent_t e0, e1;
  CK(cudaEventCreate(&e0));
  CK(cudaEventCreate(&e1));
  const size_t smem = 2 * kChunks * kChunkBytes + 1024;
  int failures = 0;
  auto run = [&](auto kern, int g, int ctas) -> int {
    CK(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem));
    kern<<<ctas, g + 32, smem>>>(cache, drows, flag);
    CK(cudaGetLastError());
    CK(cudaDeviceSynchronize());
    std::vector<float> ts;
    for (int it = 0; it < 7; ++it) {
      CK(cudaMemsetAsync(l2_flush, it, flush_bytes));  // L2 cold, outside the events
      CK(cudaEventRecord(e0));
      kern<<<ctas, g + 32, smem>>>(cache, drows, flag);
      CK(cudaEventRecord(e1));
      CK(cudaEventSynchronize(e1));
      float ms = 0.f;
      CK(cudaEventElapsedTime(&ms, e0, e1));
      ts.push_back(ms);
    }
    std::sort(ts.begin(), ts.end());
    const float ms = ts[ts.size() / 2];
    int f = 0;
    CK(cudaMemcpy(&f, flag, sizeof(int), cudaMemcpyDeviceToHost));
    const double bytes = (double)ctas * kRowsPerCta * kRowElems * 2;
    printf("gather ctas=%d threads=%d: %.1f us %.0f GB/s%s\n", ctas, g, ms * 1e3,
           bytes / (ms * 1e-3) / 1e9, f ? " TIMEOUT" : "");
    if (f) ++failures;
    return 0;
  };
  for (int ctas : {128, nsm}) {
    if (run(gather_ring<128>, 128, ctas)) return 1;
    if (run(gather_ring<192>, 192, ctas)) return 1;
    if (run(gather_ring<256>, 256, ctas)) return 1;
  }
  return failures ? 2 : 0;
}
