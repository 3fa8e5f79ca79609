// sparse_decode_kernel.cuh -- sparse-MLA decode for sm_103a.
//
// All heads of a token share the token's top-k gathered latent rows (576 =
// 512 latent + 64 rope columns; the value is the 512 latent columns).  The
// work is the list of (token, group of up to 64 heads, 64-key tile) units,
// numbered unit-major; CTA b takes the contiguous tile range
// [b*T/grid, (b+1)*T/grid), so every SM gets the same number of tiles
// whatever the token count.  A range is cut into segments, one per
// (token, head group) it touches; a segment that covers all of its unit's
// tiles writes the final O and LSE, one that covers only a part writes
// O/l and its LSE in fp32 to a partial slot, and decode_merge_kernel combines
// the parts of each split unit by their LSE (the split-KV merge).
//
// The kernel works in the transposed form so that the tensor-core M
// dimension runs over keys:
//
//   Sᵀ[key, head]  = R[key, 0:576] · Q[head, 0:576]ᵀ     M = 64 keys, N = heads
//   Oᵀ[dv, head]  += R[key, 0:512]ᵀ · Pᵀ[key, head]       M = 128 (x4 tiles of dv)
//
//   gather warps 4-7    copy each 64-key tile into a 2-stage ring with 16-byte
//                       cp.async, one 64-column chunk at a time (128-byte
//                       swizzle: the UMMA K-major layout for Sᵀ and the
//                       MN-major layout for Oᵀ), each chunk on its own barrier;
//   MMA warp 8          TMA-loads Q at the start of each segment and issues
//                       the Sᵀ MMAs of a chunk as soon as it has landed;
//   MMA warp 9          issues Oᵀ += Rᵀ·Pᵀ as soon as Pᵀ is ready, one
//                       128-column m-tile at a time, and releases each m-tile's
//                       chunks as it completes (two issuers, so waiting for the
//                       next gathered tile never delays the current PV);
//   softmax warps 0-3   two threads per key of the tile, each with half of the
//                       heads: per-head maximum over the tile's keys (shuffle
//                       transpose-reduce + shared memory), exp2 with a lazily
//                       rescaled running maximum, per-thread partial row sums,
//                       and Pᵀ (bf16) written into the tile's rope columns,
//                       which are dead once Sᵀ is done; at the end of a
//                       segment, the normalised output.
//
// TMEM: Sᵀ double buffer at columns [0, 2*NP) (64-row layout: key r lives in
// lane 32*(r/16) + r%16), Oᵀ at [128, 128 + 4*NP) (row = lane).
//
// Method source: vLLM API page "vllm.v1.attention.backends.mla.
// flashattn_mla_sparse" -- FlashAttnMLASparseFA4Backend (BF16 cache only; head
// size 576 split into 512 latent + 64 rope; cache block size a multiple of 64;
// index_topk % 128 == 0 so the gathered indices are whole tiles; 8..128
// heads) and _fa4_varlen_scalars (one query row per token).  The merge of
// partial results is the log-sum-exp weighting of merge_attn_states and
// FA4SplitKVCombineKernel on the vLLM page "vllm.v1.attention.backends.mla.
// prefill.flash_attn", applied to any number of parts.
#pragma once

#include <atomic>
#include <cstdint>
#include <cstring>
#include <cuda.h>
#include <cuda_runtime.h>

#include "sm103_ptx.cuh"
#include "varlen_fwd_kernel.cuh"  // kStatusTimeout, bounded waits

namespace fa {

constexpr int kDecodePage = 64;
constexpr int kDecodeThreads = 384;   // softmax 0-3, gather 4-7, S issuer 8, PV issuer 9, idle 10-11
// Register split (launch: 168 x 384 = 64512): softmax 128 x 232, gather
// 128 x 88, control 128 x 96 = 53248.
constexpr uint32_t kDecodeSoftmaxRegs = 232;
constexpr uint32_t kDecodeGatherRegs = 88;
constexpr uint32_t kDecodeControlRegs = 96;
constexpr int kDecodeKeys = 64;       // keys per tile
constexpr int kDecodeMaxTopk = 2048;  // key slots of one CTA's range (row table in shared memory)
constexpr int kDecodeMaxTilesPerCta = kDecodeMaxTopk / 64;
// Measured cost of a split schedule's partial writes, segment switches and
// merge kernel, in tile times (one tile: ~2.7 us on one SM).
constexpr int kDecodeMergeCostTiles = 6;
constexpr int kDqk = 576, kDv = 512;
constexpr int kChunks = 9;            // 64-column chunks of a row: 8 latent + 1 rope
constexpr int kPvGroups = 4;          // PV m-tiles of 128 value columns
constexpr int kChunkBytes = kDecodeKeys * 128;            // one 64-column chunk
constexpr int kStageBytes = kChunks * kChunkBytes;        // 73728
constexpr int kQBytes = 9 * 64 * 128;                     // Q for up to 64 heads

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
  // Work split (see the file comment).
  int groups;             // head groups of up to 64 per token
  int n_tiles;            // tiles per unit: topk / 64
  int total_tiles;        // num_tokens * groups * n_tiles (< 2^31)
  int grid;               // CTAs; at most kDecodeMaxTilesPerCta tiles each
  // Ranges are cut in granules of `gran` tiles (1, or n_tiles for ranges of
  // whole units): total_tiles = (range_q * grid + range_r) * gran.
  int gran, range_q, range_r;
  float* part_o;          // [2 * grid][64][512] O/l of partial segments (NULL: none)
  float* part_lse;        // [2 * grid][64] their natural-log LSE
  uint64_t wait_limit_ns; // pipeline wait limit (bounded waits)
};

// First tile of CTA b's range: the first range_r CTAs take range_q + 1
// granules, the others range_q.
__host__ __device__ inline int decode_cta_lo(const DecodeArgs& a, int b) {
  return (b * a.range_q + (b < a.range_r ? b : a.range_r)) * a.gran;
}

// Chunk c of a stage is released when the PV m-tile that last reads it is
// done: m-tile g reads value chunks 2g and 2g+1, and every m-tile reads Pᵀ
// in the rope chunk 8, so chunk 8 goes with the last m-tile.
__host__ __device__ constexpr int release_group(int c) { return c < 8 ? c >> 1 : kPvGroups - 1; }

struct alignas(16) DecodeCtl {
  uint64_t q_full;
  uint64_t r_full[2][kChunks];     // chunk landed (128 gather-thread arrivals)
  uint64_t r_free[2][kPvGroups];   // the chunks of PV m-tile g may be overwritten
  uint64_t s_full[2];
  uint64_t s_free[2];
  uint64_t p_full[2];   // Pᵀ(j) written, indexed by j % 2
  uint64_t pv_done[2];  // PV(j) complete, indexed by j % 2
  uint64_t q_free;      // every S MMA of the segment done: Q may be replaced
  uint64_t o_free;      // the segment's Oᵀ has been read out (128 arrivals)
  uint64_t drain;
  uint32_t tmem_base;
  volatile int abort_flag;
  alignas(16) float red[4][64];  // per-warp partial maxima / sums
  float m_used[64];   // running maximum per head (scaled log2 units)
  alignas(16) float alpha[64];   // rescale factors of the current tile; after the
                                 // last tile, the reciprocal row sums
};

constexpr size_t kDecodeSmem = 1024 + kQBytes + 2 * kStageBytes +
                               sizeof(int) * kDecodeMaxTopk + sizeof(DecodeCtl);
static_assert(kDecodeSmem <= 232448, "decode shared memory exceeds the per-CTA limit");
static_assert((kQBytes + 2 * kStageBytes + sizeof(int) * kDecodeMaxTopk) % 16 == 0,
              "control block must stay 16-byte aligned");

__device__ __forceinline__ void named_bar_sync(int id, int n) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}

// Barrier over n threads that also ANDs a predicate (all must pass).
__device__ __forceinline__ int named_bar_and(int id, int n, int pred) {
  int r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 q, %1, 0;\n\t"
      "bar.red.and.pred p, %2, %3, q;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(r)
      : "r"(pred), "r"(id), "r"(n)
      : "memory");
  return r;
}

// Barrier over n threads that also ORs a predicate.
__device__ __forceinline__ int named_bar_or(int id, int n, int pred) {
  int r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 q, %1, 0;\n\t"
      "bar.red.or.pred p, %2, %3, q;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(r)
      : "r"(pred), "r"(id), "r"(n)
      : "memory");
  return r;
}

__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Max (kMax) or sum of V values per lane over the 16 lanes of each half-warp
// (the halves reduce independently), by repeated halving.  Afterwards a lane
// holds max(V / 16, 1) results in v[0 ..); their value indices are given by
// half_reduce_index.
template <int V, bool kMax>
__device__ __forceinline__ void half_warp_transpose_reduce(float* v, int lane) {
#pragma unroll
  for (int s = 0; s < 4; ++s) {
    const int o = 8 >> s;
    const int n = V >> s;  // values held before this step
    if (n >= 2) {
      const int half = n / 2;
      const bool upper = (lane & o) != 0;
#pragma unroll
      for (int i = 0; i < half; ++i) {
        const float send = upper ? v[i] : v[i + half];
        const float keep = upper ? v[i + half] : v[i];
        const float recv = __shfl_xor_sync(0xffffffffu, send, o);
        v[i] = kMax ? fmaxf(keep, recv) : keep + recv;
      }
    } else {
      const float recv = __shfl_xor_sync(0xffffffffu, v[0], o);
      v[0] = kMax ? fmaxf(v[0], recv) : v[0] + recv;
    }
  }
}
template <int V>
__device__ __forceinline__ int half_reduce_index(int lane, int i) {
  return V >= 16 ? (lane & 15) * (V / 16) + i : ((lane & 15) >> 1);
}
// Lanes that publish the results (for V = 8, lane pairs hold the same one).
template <int V>
__device__ __forceinline__ bool half_reduce_writer(int lane) {
  return V >= 16 || (lane & 1) == 0;
}

template <int NP>
__global__ void __launch_bounds__(kDecodeThreads, 1)
    sparse_decode_kernel(const __grid_constant__ CUtensorMap q_map, const DecodeArgs a) {
  static_assert(NP == 16 || NP == 32 || NP == 64, "head group width");
  constexpr uint32_t kSwP = NP == 64 ? ptx::kLayoutSw128 : (NP == 32 ? ptx::kLayoutSw64
                                                                     : ptx::kLayoutSw32);
  constexpr int kPRowBytes = NP * 2;  // one Pᵀ row (one key) in bytes
  constexpr int HP = NP / 2;          // heads per softmax thread
  constexpr int kRed = HP >= 16 ? HP / 16 : 1;  // reduced values per lane

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* q_s = smem;
  uint8_t* stage[2] = {smem + kQBytes, smem + kQBytes + kStageBytes};
  int* rows = reinterpret_cast<int*>(smem + kQBytes + 2 * kStageBytes);
  DecodeCtl* cb = reinterpret_cast<DecodeCtl*>(rows + kDecodeMaxTopk);
  volatile int* abort_flag = &cb->abort_flag;

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int heads = a.num_heads < 64 ? a.num_heads : 64;  // real heads in a group
  const int n_tiles = a.n_tiles;
  // This CTA's tiles: global tile lo + i, i in [0, n).
  const int lo = decode_cta_lo(a, blockIdx.x);
  const int n = decode_cta_lo(a, blockIdx.x + 1) - lo;
  // Tile i of the range is tile (pos0 + i) % n_tiles of unit
  // unit0 + (pos0 + i) / n_tiles (32-bit: pos0 < n_tiles, i < kDecodeMaxTilesPerCta).
  const int pos0 = lo % n_tiles;
  const int unit0 = lo / n_tiles;
  auto seg_first = [&](int i) { return i == 0 || (pos0 + i) % n_tiles == 0; };
  auto seg_last = [&](int i) { return i == n - 1 || (pos0 + i + 1) % n_tiles == 0; };
  auto unit_of = [&](int i) { return unit0 + (pos0 + i) / n_tiles; };

  // The merge kernel may be scheduled as SMs free up; it waits for this
  // grid to complete before it reads anything.
  ptx::grid_launch_dependents();
  if (tid == 0) {
    ptx::mbar_init(ptx::smem_u32(&cb->q_full), 1);
    for (int s = 0; s < 2; ++s) {
      for (int c = 0; c < kChunks; ++c) ptx::mbar_init(ptx::smem_u32(&cb->r_full[s][c]), 128);
      for (int g = 0; g < kPvGroups; ++g) ptx::mbar_init(ptx::smem_u32(&cb->r_free[s][g]), 1);
      ptx::mbar_init(ptx::smem_u32(&cb->s_full[s]), 1);
      ptx::mbar_init(ptx::smem_u32(&cb->s_free[s]), 128);
      ptx::mbar_init(ptx::smem_u32(&cb->p_full[s]), 128);
      ptx::mbar_init(ptx::smem_u32(&cb->pv_done[s]), 1);
    }
    ptx::mbar_init(ptx::smem_u32(&cb->q_free), 1);
    ptx::mbar_init(ptx::smem_u32(&cb->o_free), 128);
    ptx::mbar_init(ptx::smem_u32(&cb->drain), 2);
    cb->abort_flag = 0;
    ptx::fence_mbar_init();
    // The first segment's Q goes out before anything else, ahead of the
    // gathers of every CTA, so that the first S MMAs do not wait behind them.
    ptx::prefetch_tmap(&q_map);
    const int token = unit0 / a.groups;
    ptx::mbar_arrive_expect_tx(ptx::smem_u32(&cb->q_full), 9 * NP * 128);
    for (int c = 0; c < 9; ++c)
      ptx::tma_load_3d(ptx::smem_u32(q_s + c * NP * 128), &q_map, ptx::smem_u32(&cb->q_full),
                       c * 64, (unit0 - token * a.groups) * 64, token);
  }
  if (warp == 8) {
    ptx::tmem_alloc(ptx::smem_u32(&cb->tmem_base), 512);
    ptx::tmem_relinquish();
  }
  // Row table: physical cache row of every key slot of the range, -1 if the
  // slot is outside its token's context or its page is out of range.  All
  // index loads are issued before any page-table load, so the table costs
  // two dependent memory round trips.
  {
    constexpr int kPer = (kDecodeMaxTopk + kDecodeThreads - 1) / kDecodeThreads;
    const int64_t context = (int64_t)a.max_pages * kDecodePage;
    int p[kPer], page[kPer], token[kPer];
#pragma unroll
    for (int k = 0; k < kPer; ++k) {
      const int s = tid + k * kDecodeThreads;
      p[k] = -1;
      token[k] = 0;
      if (s < n * kDecodeKeys) {
        const int i = s / kDecodeKeys;
        token[k] = unit_of(i) / a.groups;
        const int slot = (pos0 + i) % n_tiles * kDecodeKeys + s % kDecodeKeys;
        p[k] = __ldg(a.topk_idx + (size_t)token[k] * a.topk + slot);
      }
    }
#pragma unroll
    for (int k = 0; k < kPer; ++k)
      page[k] = (p[k] >= 0 && p[k] < context)
                    ? __ldg(a.page_table + (size_t)token[k] * a.max_pages + p[k] / kDecodePage)
                    : -1;
#pragma unroll
    for (int k = 0; k < kPer; ++k) {
      const int s = tid + k * kDecodeThreads;
      if (s < n * kDecodeKeys)
        rows[s] = (page[k] >= 0 && page[k] < a.num_pages) ? page[k] * kDecodePage + p[k] % kDecodePage
                                                          : -1;
    }
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = cb->tmem_base;

  if (warp >= 4 && warp < 8) {
    ptx::regs_dec<kDecodeGatherRegs>();
    // ------------------------------------------------------------ gather
    // Tile i goes to stage i % 2, one 64-column chunk at a time, so that the
    // S MMAs can start on the first chunks while the rest are in flight.
    // Each thread copies the same 16-byte unit (ptid % 8) of 4 rows
    // (ptid / 8 + 16 k) per chunk; its copies of chunk c arrive on
    // r_full[stage][c] by themselves when they land
    // (cp.async.mbarrier.arrive.noinc; 128 arrivals expected), so no gather
    // warp blocks on its own copies.  Chunk c of tile i >= 2 waits for the
    // PV m-tile of tile i - 2 that last reads it.
    const int ptid = tid - 128;
    const int u = ptid & 7;
    const uint64_t read_once = ptx::make_policy_evict_first();  // each row is read once
    test_load_delay(a.wait_limit_ns);
    bool ok = true;
    for (int i = 0; i < n && ok; ++i) {
      const int st = i & 1;
      const uint32_t dst0 = ptx::smem_u32(stage[st]);
      int row[4];
#pragma unroll
      for (int k = 0; k < 4; ++k)  // invalid slots read row 0 (masked later)
        row[k] = max(rows[i * kDecodeKeys + (ptid >> 3) + 16 * k], 0);
      for (int c = 0; c < kChunks; ++c) {
        if (i >= 2 && (c == 0 || (c < 8 && release_group(c) != release_group(c - 1)))) {
          ok = wait_warp(ptx::smem_u32(&cb->r_free[st][release_group(c)]), ((i >> 1) - 1) & 1,
                         abort_flag, a.status, a.wait_limit_ns);
          if (!ok) break;
        }
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int r = (ptid >> 3) + 16 * k;
          ptx::cp_async_16_hint(dst0 + c * kChunkBytes + r * 128 + ((u ^ (r & 7)) << 4),
                                a.cache + (size_t)row[k] * kDqk + c * 64 + u * 8, read_once);
        }
        ptx::cp_async_mbar_arrive(ptx::smem_u32(&cb->r_full[st][c]));
      }
    }
    cp_async_wait<0>();  // nothing of this thread is in flight at exit
  } else if (warp >= 8) {
    ptx::regs_dec<kDecodeControlRegs>();
    // ------------------------------------------------------------ MMA issuers
    constexpr uint32_t idesc_s = ptx::idesc_bf16_f32(64, NP, false, false);
    constexpr uint32_t idesc_o = ptx::idesc_bf16_f32(128, NP, true, true);
    // Each issuer warp runs converged (warp-uniform waits); its MMAs go out
    // four at a time from one elected lane, as do its commits.
    if (warp == 8) {
      // Sᵀ(i) = R(i) Qᵀ into Sᵀ buffer i % 2, chunk by chunk as they land.
      const uint64_t qd = ptx::smem_desc(ptx::smem_u32(q_s), 16, 1024, ptx::kLayoutSw128);
      bool ok = true;
      int seg = 0;
      bool q_inflight = true;  // Q load number seg issued, its wait not yet passed
      for (int i = 0; i < n && ok; ++i) {
        const int st = i & 1;
        if (seg_first(i)) {
          if (seg > 0) {
            // Every S MMA that reads the current Q must be done before the
            // next segment's Q replaces it.
            ptx::mma_commit_elect(ptx::smem_u32(&cb->q_free));
            ok = wait_warp(ptx::smem_u32(&cb->q_free), (seg - 1) & 1, abort_flag, a.status, a.wait_limit_ns);
            if (!ok) break;
            // (Segment 0's Q was issued at kernel start.)
            if (lane == 0) {
              const int unit = unit_of(i);
              const int token = unit / a.groups;
              const int head0 = (unit - token * a.groups) * 64;
              ptx::mbar_arrive_expect_tx(ptx::smem_u32(&cb->q_full), 9 * NP * 128);
              for (int c = 0; c < 9; ++c)
                ptx::tma_load_3d(ptx::smem_u32(q_s + c * NP * 128), &q_map,
                                 ptx::smem_u32(&cb->q_full), c * 64, head0, token);
            }
            __syncwarp();
            q_inflight = true;
          }
          ok = wait_warp(ptx::smem_u32(&cb->q_full), seg & 1, abort_flag, a.status, a.wait_limit_ns);
          if (!ok) break;
          q_inflight = false;
          ++seg;
        }
        if (i >= 2) {
          ok = wait_warp(ptx::smem_u32(&cb->s_free[st]), ((i >> 1) - 1) & 1, abort_flag,
                         a.status, a.wait_limit_ns);
          if (!ok) break;
        }
        const uint64_t rd = ptx::smem_desc(ptx::smem_u32(stage[st]), 16, 1024, ptx::kLayoutSw128);
        const uint32_t d = tmem + (uint32_t)(st * NP);
        for (int c = 0; c < kChunks && ok; ++c) {
          ok = wait_warp(ptx::smem_u32(&cb->r_full[st][c]), (i >> 1) & 1, abort_flag, a.status, a.wait_limit_ns);
          if (!ok) break;
          // The gathered rows were written by cp.async (generic proxy); order
          // them before the tensor core's (async proxy) reads.
          ptx::fence_proxy_async_smem();
          ptx::tc_fence_after();
          // Four K=16 steps over the chunk's 64 columns (32 bytes apart).
          ptx::mma_ss4_elect<2, 2>(d, ptx::desc_add(rd, c * kChunkBytes),
                                   ptx::desc_add(qd, c * NP * 128), idesc_s, c > 0 ? 1u : 0u);
        }
        if (!ok) break;
        ptx::mma_commit_elect(ptx::smem_u32(&cb->s_full[st]));
      }
      ptx::mma_commit_elect(ptx::smem_u32(&cb->drain));
      wait_drain_warp(ptx::smem_u32(&cb->drain), 0, a.status);
      // A Q reload still in flight (the wait for it gave up) lands before
      // the CTA exits.
      if (q_inflight) wait_drain_warp(ptx::smem_u32(&cb->q_full), seg & 1, a.status);
    } else if (warp == 9) {
      // Oᵀ += R(i)[:, 0:512]ᵀ Pᵀ(i), one 128-column m-tile at a time; each
      // m-tile's commit releases the chunks it was the last to read.  The
      // first PV of a segment overwrites Oᵀ, so it waits until the softmax
      // warps have read out the previous segment's.
      bool ok = true;
      int seg = 0;
      for (int i = 0; i < n && ok; ++i) {
        const int st = i & 1;
        ok = wait_warp(ptx::smem_u32(&cb->p_full[st]), (i >> 1) & 1, abort_flag, a.status, a.wait_limit_ns);
        if (!ok) break;
        const bool first = seg_first(i);
        if (first) {
          if (seg > 0) {
            ok = wait_warp(ptx::smem_u32(&cb->o_free), (seg - 1) & 1, abort_flag, a.status, a.wait_limit_ns);
            if (!ok) break;
          }
          ++seg;
        }
        ptx::fence_proxy_async_smem();
        ptx::tc_fence_after();
        const uint32_t ra = ptx::smem_u32(stage[st]);
        // A = R[keys, 128m .. 128m+128)ᵀ: MN-major, two 64-wide chunks.
        const uint64_t ad = ptx::smem_desc(ra, kChunkBytes, 1024, ptx::kLayoutSw128);
        // B = Pᵀ[keys, heads] in the rope chunk: MN-major, NP wide.
        const uint64_t bd =
            ptx::smem_desc(ra + 8 * kChunkBytes, 8 * kPRowBytes, 8 * kPRowBytes, kSwP);
#pragma unroll
        for (int m = 0; m < kPvGroups; ++m) {
          // Four K=16 steps over the tile's 64 keys: 16 rows of R (128 bytes
          // each) and 16 rows of Pᵀ per step.
          ptx::mma_ss4_elect<16 * 128 / 16, 16 * kPRowBytes / 16>(
              tmem + 128u + (uint32_t)(m * NP), ptx::desc_add(ad, 2 * m * kChunkBytes), bd,
              idesc_o, first ? 0u : 1u);
          ptx::mma_commit_elect(ptx::smem_u32(&cb->r_free[st][m]));
        }
        ptx::mma_commit_elect(ptx::smem_u32(&cb->pv_done[st]));
      }
      ptx::mma_commit_elect(ptx::smem_u32(&cb->drain));
      wait_drain_warp(ptx::smem_u32(&cb->drain), 0, a.status);
    }
  } else {
    ptx::regs_inc<kDecodeSoftmaxRegs>();
    // ------------------------------------------------------------ softmax
    // Sᵀ has 64 key rows in TMEM lanes 32w + (0..15) of warp w's quarter.
    // Lane l of warp w takes key 16w + l % 16 and heads [HP*(l/16), +HP).
    const int half = lane >> 4;
    const int key_in_tile = warp * 16 + (lane & 15);
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
    const float sl2 = a.scale_log2;
    const float neg_inf = -__int_as_float(0x7f800000);
    float* l_inv = cb->alpha;  // after a segment's last tile: reciprocal row sums
    float lpart[HP];
#pragma unroll
    for (int h = 0; h < HP; ++h) lpart[h] = 0.f;
    if (tid < 64) cb->m_used[tid] = neg_inf;
    named_bar_sync(1, 128);
    bool ok = true;
    for (int seg = 0, i = 0; i < n && ok; ++seg) {
      const int seg_start = i;
      int seg_end = i;  // last tile of the segment
      while (!seg_last(seg_end)) ++seg_end;
      for (; i <= seg_end; ++i) {
        const int st = i & 1;
        const bool first = i == seg_start;
        // Every wait is followed by a warpgroup-wide agreement, so that no warp
        // can be left alone at a later named barrier after another gave up.
        ok = wait_warp(ptx::smem_u32(&cb->s_full[st]), (i >> 1) & 1, abort_flag, a.status, a.wait_limit_ns);
        ok = named_bar_and(3, 128, ok);
        if (!ok) break;
        ptx::tc_fence_after();
        uint32_t sr[HP];
        ptx::tmem_ld_16x2<HP>(tmem + lane_base + st * NP, sr);
        ptx::tmem_wait_ld();
        if constexpr (HP == 8) {
          ptx::reg_fence8(sr);
        } else {
#pragma unroll
          for (int c = 0; c < HP; c += 16) ptx::reg_fence16(sr + c);
        }
        ptx::tc_fence_before();
        ptx::mbar_arrive(ptx::smem_u32(&cb->s_free[st]));  // Sᵀ buffer may be reused
        const bool valid = rows[i * kDecodeKeys + key_in_tile] >= 0;
        float s[HP], v[HP];
#pragma unroll
        for (int h = 0; h < HP; ++h) {
          s[h] = valid ? __uint_as_float(sr[h]) : neg_inf;
          v[h] = s[h];
        }
        // Per-head maximum over the tile: 16 lanes, then 4 warps.
        half_warp_transpose_reduce<HP, true>(v, lane);
        if (half_reduce_writer<HP>(lane)) {
#pragma unroll
          for (int k = 0; k < kRed; ++k) cb->red[warp][half * HP + half_reduce_index<HP>(lane, k)] = v[k];
        }
        named_bar_sync(1, 128);
        int need = 0;
        if (tid < NP) {
          const float mt = fmaxf(fmaxf(cb->red[0][tid], cb->red[1][tid]),
                                 fmaxf(cb->red[2][tid], cb->red[3][tid])) * sl2;
          const float mu = cb->m_used[tid];
          float al = 1.f;
          if (mt > mu + kRescaleLog2) {
            need = 1;
            al = (mu == neg_inf) ? 0.f : ptx::ex2(mu - mt);
            cb->m_used[tid] = mt;
          }
          cb->alpha[tid] = al;
        }
        const int any = named_bar_or(2, 128, need);
        if (any) {
#pragma unroll
          for (int h = 0; h < HP; ++h) lpart[h] *= cb->alpha[half * HP + h];
          if (!first) {
            // Oᵀ holds the segment's earlier tiles: wait for the last PV, then
            // scale every head column by its factor.
            ok = wait_warp(ptx::smem_u32(&cb->pv_done[(i - 1) & 1]), ((i - 1) >> 1) & 1,
                           abort_flag, a.status, a.wait_limit_ns);
            ok = named_bar_and(3, 128, ok);
            if (!ok) break;
            ptx::tc_fence_after();
#pragma unroll
            for (int m = 0; m < kPvGroups; ++m) {
#pragma unroll
              for (int c = 0; c < NP; c += 16) {
                uint32_t o[16];
                const uint32_t addr = tmem + lane_base + 128u + m * NP + c;
                ptx::tmem_ld16(addr, o);
                ptx::tmem_wait_ld();
                ptx::reg_fence16(o);
#pragma unroll
                for (int k = 0; k < 16; ++k)
                  o[k] = __float_as_uint(__uint_as_float(o[k]) * cb->alpha[c + k]);
                ptx::tmem_st16(addr, o);
              }
            }
            ptx::tmem_wait_st();
          }
        }
        // Probabilities: this thread's half of the Pᵀ row of its key.
        {
          uint8_t* prow = stage[st] + 8 * kChunkBytes + key_in_tile * kPRowBytes;
#pragma unroll
          for (int g = 0; g < HP / 8; ++g) {
            uint32_t pk[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const int h0 = g * 8 + 2 * k;  // local head index
              const float b0 = cb->m_used[half * HP + h0], b1 = cb->m_used[half * HP + h0 + 1];
              const float p0 = valid ? ptx::ex2(fmaf(s[h0], sl2, -b0)) : 0.f;
              const float p1 = valid ? ptx::ex2(fmaf(s[h0 + 1], sl2, -b1)) : 0.f;
              lpart[h0] += p0;
              lpart[h0 + 1] += p1;
              pk[k] = ptx::pack_bf16x2(p0, p1);
            }
            // Swizzled 16-byte unit of row key_in_tile (the NP*2-byte-wide
            // layout: unit index XOR row bits).
            const int gu = half * (HP / 8) + g;
            const int unit = NP == 64 ? (gu ^ (key_in_tile & 7))
                                      : (NP == 32 ? (gu ^ ((key_in_tile >> 1) & 3))
                                                  : (gu ^ ((key_in_tile >> 2) & 1)));
            *reinterpret_cast<uint4*>(prow + unit * 16) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
          }
        }
        ptx::fence_proxy_async_smem();
        ptx::tc_fence_before();
        ptx::mbar_arrive(ptx::smem_u32(&cb->p_full[st]));
      }
      if (!ok) break;

      // ---------------------------------------------------- segment output
      const int unit = unit_of(seg_end);
      const int token = unit / a.groups;
      const int head0 = (unit - token * a.groups) * 64;
      // The whole unit is in this segment: final output; else a partial slot
      // (2b for the CTA's first segment, 2b + 1 for its last).
      const bool whole = (pos0 + seg_start) % n_tiles == 0 && (pos0 + seg_end + 1) % n_tiles == 0;
      const int slot = 2 * (int)blockIdx.x + (seg == 0 ? 0 : 1);
      // Row sums: reduce the per-thread partials over keys (16 lanes, 4 warps).
      half_warp_transpose_reduce<HP, false>(lpart, lane);
      if (half_reduce_writer<HP>(lane)) {
#pragma unroll
        for (int k = 0; k < kRed; ++k)
          cb->red[warp][half * HP + half_reduce_index<HP>(lane, k)] = lpart[k];
      }
      named_bar_sync(1, 128);
      if (tid < NP) {
        const float l = (cb->red[0][tid] + cb->red[1][tid]) + (cb->red[2][tid] + cb->red[3][tid]);
        l_inv[tid] = l > 0.f ? 1.f / l : 0.f;
        const float lse_v = l > 0.f ? (cb->m_used[tid] + __log2f(l)) * 0.69314718055994531f
                                    : neg_inf;
        if (tid < heads) {
          if (!whole)
            a.part_lse[(size_t)slot * 64 + tid] = lse_v;
          else if (a.lse)
            a.lse[(size_t)(head0 + tid) * a.num_tokens + token] = lse_v;
        }
      }
      if (tid < 64) cb->m_used[tid] = neg_inf;  // fresh running maximum for the next segment
      named_bar_sync(1, 128);
      // A commit tracks every earlier MMA of its issuer, so PV(i) done means
      // all of the segment's Oᵀ is final.
      ok = wait_warp(ptx::smem_u32(&cb->pv_done[seg_end & 1]), (seg_end >> 1) & 1, abort_flag,
                     a.status, a.wait_limit_ns);
      ok = named_bar_and(3, 128, ok);
      if (!ok) break;
      ptx::tc_fence_after();
      // Oᵀ has one value column per TMEM lane, the output wants value columns
      // contiguous per head.  Each thread packs heads (2k, 2k+1) of its column
      // and swaps with the neighbouring lane, after which the even lane holds
      // columns (c, c+1) of head 2k and the odd lane those of head 2k+1: one
      // store each (a bf16x2 word, or an fp32 pair for a partial).
      float li[NP];
#pragma unroll
      for (int h = 0; h < NP; h += 4) {
        const float4 v4 = *reinterpret_cast<const float4*>(l_inv + h);
        li[h] = v4.x; li[h + 1] = v4.y; li[h + 2] = v4.z; li[h + 3] = v4.w;
      }
      const bool odd = lane & 1;
      uint16_t* out_g = a.out + ((size_t)token * a.num_heads + head0) * kDv;
      float* po = a.part_o + (size_t)slot * 64 * kDv;
#pragma unroll 1
      for (int m = 0; m < kPvGroups; ++m) {
        const int dv_even = m * 128 + warp * 32 + (lane & ~1);
        uint32_t o[NP];
#pragma unroll
        for (int c = 0; c < NP; c += 16) ptx::tmem_ld16(tmem + lane_base + 128u + m * NP + c, o + c);
        ptx::tmem_wait_ld();
#pragma unroll
        for (int c = 0; c < NP; c += 16) ptx::reg_fence16(o + c);
        if (whole) {
#pragma unroll
          for (int k = 0; k < NP / 2; ++k) {
            const uint32_t w = ptx::pack_bf16x2(__uint_as_float(o[2 * k]) * li[2 * k],
                                                __uint_as_float(o[2 * k + 1]) * li[2 * k + 1]);
            const uint32_t r = __shfl_xor_sync(0xffffffffu, w, 1);
            const uint32_t pair = odd ? __byte_perm(w, r, 0x3276) : __byte_perm(w, r, 0x5410);
            const int h = 2 * k + (odd ? 1 : 0);
            if (h < heads) *reinterpret_cast<uint32_t*>(out_g + (size_t)h * kDv + dv_even) = pair;
          }
        } else {
#pragma unroll
          for (int k = 0; k < NP / 2; ++k) {
            const float e0 = __uint_as_float(o[2 * k]) * li[2 * k];
            const float e1 = __uint_as_float(o[2 * k + 1]) * li[2 * k + 1];
            const float r = __shfl_xor_sync(0xffffffffu, odd ? e0 : e1, 1);
            const int h = 2 * k + (odd ? 1 : 0);
            if (h < heads)
              *reinterpret_cast<float2*>(po + (size_t)h * kDv + dv_even) =
                  odd ? make_float2(r, e1) : make_float2(e0, r);
          }
        }
      }
      // Oᵀ has been read: the next segment's first PV may overwrite it.
      ptx::tc_fence_before();
      ptx::mbar_arrive(ptx::smem_u32(&cb->o_free));
#pragma unroll
      for (int h = 0; h < HP; ++h) lpart[h] = 0.f;
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 8) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, 512);
  }
}

// Merge of split units.  Block (x, y): boundary b = x + 1 between CTAs b-1
// and b, heads [8y, 8y + 8) of the group.  Only a boundary that falls inside
// a unit and is the first one inside it does work: the unit's parts come
// from CTA b-1 (its last segment, or its only one if it starts exactly at
// the unit) and CTAs b, b+1, ... (their first segments) while they start
// inside the unit.  O = sum_p w_p O_p with w_p = exp(lse_p - LSE) and LSE =
// log sum_p exp(lse_p); a unit whose parts all have lse = -inf (no valid
// key) gets O = 0, LSE = -inf.  The parts are summed in CTA order, so the
// result does not depend on timing.  Each thread owns 16 consecutive
// outputs of one head; with up to kMergeFast parts it issues every LSE load
// and then every partial load at once (two memory round trips).
constexpr int kMergeHeads = 8;  // heads per block: 8 x 512 outputs, 16 per thread
constexpr int kMergeFast = 2;

__device__ __forceinline__ int merge_part_slot(int b, int p, bool first_is_whole_start) {
  // part 0: CTA b-1 (slot 2(b-1) if its range starts at the unit, else its
  // last segment's slot 2(b-1)+1); part p >= 1: CTA b-1+p, first segment.
  return p == 0 ? 2 * (b - 1) + (first_is_whole_start ? 0 : 1) : 2 * (b - 1 + p);
}

__global__ void __launch_bounds__(256) decode_merge_kernel(const DecodeArgs a) {
  const int b = blockIdx.x + 1;
  const int lob = decode_cta_lo(a, b);
  const int n_tiles = a.n_tiles;
  if (lob % n_tiles == 0) return;
  const int unit = lob / n_tiles, u0 = unit * n_tiles, u1 = u0 + n_tiles;
  const int lop = decode_cta_lo(a, b - 1);
  if (lop > u0) return;  // an earlier boundary lies inside this unit
  const int heads = a.num_heads < 64 ? a.num_heads : 64;
  const int tid = threadIdx.x;
  const int h = blockIdx.y * kMergeHeads + tid / 32;  // 32 threads x 16 outputs per head
  if (h >= heads) return;
  int np = 1;
  while (b - 1 + np < a.grid && decode_cta_lo(a, b - 1 + np) < u1) ++np;
  const bool start0 = lop == u0;
  const int token = unit / a.groups;
  const int head0 = (unit - token * a.groups) * 64;
  const int dv0 = (tid & 31) * 16;
  const float neg_inf = -__int_as_float(0x7f800000);
  ptx::grid_dependency_wait();  // the decode grid's partials and outputs are complete
  float acc[16];
#pragma unroll
  for (int k = 0; k < 16; ++k) acc[k] = 0.f;
  float lse = neg_inf;
  if (np <= kMergeFast) {
    float l[kMergeFast];
#pragma unroll
    for (int p = 0; p < kMergeFast; ++p)
      l[p] = p < np ? __ldg(a.part_lse + (size_t)merge_part_slot(b, p, start0) * 64 + h) : neg_inf;
    float4 v[kMergeFast][4];
#pragma unroll
    for (int p = 0; p < kMergeFast; ++p) {
      if (p < np) {
        const float4* src = reinterpret_cast<const float4*>(
            a.part_o + ((size_t)merge_part_slot(b, p, start0) * 64 + h) * kDv + dv0);
#pragma unroll
        for (int k = 0; k < 4; ++k) v[p][k] = __ldg(src + k);
      }
    }
    float mx = neg_inf;
#pragma unroll
    for (int p = 0; p < kMergeFast; ++p) mx = fmaxf(mx, l[p]);
    if (mx != neg_inf) {
      float sum = 0.f;
#pragma unroll
      for (int p = 0; p < kMergeFast; ++p) sum += p < np ? expf(l[p] - mx) : 0.f;
      lse = mx + logf(sum);
#pragma unroll
      for (int p = 0; p < kMergeFast; ++p) {
        if (p < np) {
          const float wp = expf(l[p] - lse);
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            acc[4 * k] += wp * v[p][k].x;
            acc[4 * k + 1] += wp * v[p][k].y;
            acc[4 * k + 2] += wp * v[p][k].z;
            acc[4 * k + 3] += wp * v[p][k].w;
          }
        }
      }
    }
  } else {
    float mx = neg_inf;
    for (int p = 0; p < np; ++p)
      mx = fmaxf(mx, __ldg(a.part_lse + (size_t)merge_part_slot(b, p, start0) * 64 + h));
    if (mx != neg_inf) {
      float sum = 0.f;
      for (int p = 0; p < np; ++p)
        sum += expf(__ldg(a.part_lse + (size_t)merge_part_slot(b, p, start0) * 64 + h) - mx);
      lse = mx + logf(sum);
      for (int p = 0; p < np; ++p) {
        const int slot = merge_part_slot(b, p, start0);
        const float wp = expf(__ldg(a.part_lse + (size_t)slot * 64 + h) - lse);
        const float4* src =
            reinterpret_cast<const float4*>(a.part_o + ((size_t)slot * 64 + h) * kDv + dv0);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const float4 v = __ldg(src + k);
          acc[4 * k] += wp * v.x;
          acc[4 * k + 1] += wp * v.y;
          acc[4 * k + 2] += wp * v.z;
          acc[4 * k + 3] += wp * v.w;
        }
      }
    }
  }
  // The partial lines (each shared by two neighbouring lanes) have been read
  // for the last time: drop them from L2 instead of writing them back.
  __syncwarp();
  if ((tid & 1) == 0) {
    for (int p = 0; p < np; ++p)
      ptx::discard_l2_line(a.part_o + ((size_t)merge_part_slot(b, p, start0) * 64 + h) * kDv + dv0);
  }
  if (dv0 == 0 && a.lse) a.lse[(size_t)(head0 + h) * a.num_tokens + token] = lse;
  uint4 pk[2];
  uint32_t* w = reinterpret_cast<uint32_t*>(pk);
#pragma unroll
  for (int k = 0; k < 8; ++k) w[k] = ptx::pack_bf16x2(acc[2 * k], acc[2 * k + 1]);
  uint4* dst = reinterpret_cast<uint4*>(a.out + ((size_t)token * a.num_heads + head0 + h) * kDv + dv0);
  dst[0] = pk[0];
  dst[1] = pk[1];
}

template <int NP>
inline cudaError_t launch_decode_np(const CUtensorMap& map, const DecodeArgs& a,
                                    cudaStream_t stream) {
  // Set once per device; concurrent first calls may both set it (the call
  // is idempotent), the flag itself is atomic.
  static std::atomic<bool> attr_done[64];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!attr_done[dev].load(std::memory_order_acquire)) {
    e = cudaFuncSetAttribute(sparse_decode_kernel<NP>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)kDecodeSmem);
    if (e != cudaSuccess) return e;
    attr_done[dev].store(true, std::memory_order_release);
  }
  sparse_decode_kernel<NP><<<a.grid, kDecodeThreads, kDecodeSmem, stream>>>(map, a);
  e = cudaGetLastError();
  if (e != cudaSuccess || a.part_o == nullptr || a.grid < 2) return e;
  const int heads = a.num_heads < 64 ? a.num_heads : 64;
  cudaLaunchConfig_t cfg;
  std::memset(&cfg, 0, sizeof cfg);
  cfg.gridDim = dim3(a.grid - 1, (heads + kMergeHeads - 1) / kMergeHeads);
  cfg.blockDim = dim3(256);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, decode_merge_kernel, a);
}

}  // namespace fa
