// sparse_decode_kernel.cuh -- sparse-MLA decode for sm_103a.
//
// One CTA per (token, group of up to 64 query heads).  All heads of a token
// share the token's top-k gathered latent rows (576 = 512 latent + 64 rope
// columns; the value is the 512 latent columns).  The kernel works in the
// transposed form so that the tensor-core M dimension runs over keys:
//
//   Sᵀ[key, head]  = R[key, 0:576] · Q[head, 0:576]ᵀ     M = 64 keys, N = heads
//   Oᵀ[dv, head]  += R[key, 0:512]ᵀ · Pᵀ[key, head]       M = 128 (x4 tiles of dv)
//
//   producer warps 4-7  gather 64 rows per tile with 16-byte cp.async into a
//                       2-stage ring (128-byte swizzle, the UMMA K-major layout
//                       for Sᵀ and the MN-major layout for Oᵀ);
//   MMA warp 8          TMA-loads Q once and issues Sᵀ as soon as a tile has
//                       landed and its Sᵀ buffer is free;
//   MMA warp 9          issues Oᵀ += Rᵀ·Pᵀ as soon as Pᵀ is ready and
//                       releases the stage (two issuers, so waiting for the
//                       next gathered tile never delays the current PV);
//   softmax warps 0-3   one thread per key of the tile: per-head maximum over
//                       the tile's keys (shuffle transpose-reduce + shared
//                       memory), exp2 with a lazily rescaled running maximum,
//                       per-thread partial row sums, and Pᵀ (bf16) written into
//                       the tile's rope columns, which are dead once Sᵀ is done.
//
// TMEM: Sᵀ double buffer at columns [0, 2*NP) (64-row layout: key r lives in
// lane 32*(r/16) + r%16), Oᵀ at [128, 128 + 4*NP) (row = lane).
//
// Method source: vLLM API page "vllm.v1.attention.backends.mla.
// flashattn_mla_sparse" -- FlashAttnMLASparseFA4Backend (BF16 cache only; head
// size 576 split into 512 latent + 64 rope; cache block size a multiple of 64;
// index_topk % 128 == 0 so the gathered indices are whole tiles; 8..128
// heads) and _fa4_varlen_scalars (one query row per token).
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "sm103_ptx.cuh"
#include "varlen_fwd_kernel.cuh"  // kStatusTimeout, bounded waits

namespace fa {

constexpr int kDecodePage = 64;
constexpr int kDecodeThreads = 384;   // softmax 0-3, gather 4-7, S issuer 8, PV issuer 9, idle 10-11
// Register split (launch: 168 x 384 = 64512): softmax 128 x 240, gather
// 128 x 88, control 128 x 56 = 49152.
constexpr uint32_t kDecodeSoftmaxRegs = 240;
constexpr uint32_t kDecodeGatherRegs = 88;
constexpr uint32_t kDecodeControlRegs = 56;
constexpr int kDecodeKeys = 64;       // keys per tile
constexpr int kDecodeMaxTopk = 2048;  // row table held in shared memory
constexpr int kDqk = 576, kDv = 512;
constexpr int kRowBytes = kDqk * 2;                       // 1152
constexpr int kChunkBytes = kDecodeKeys * 128;            // one 64-column chunk
constexpr int kStageBytes = 9 * kChunkBytes;              // 73728
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
};

struct alignas(8) DecodeCtl {
  uint64_t q_full;
  uint64_t r_full[2];
  uint64_t r_free[2];
  uint64_t s_full[2];
  uint64_t s_free[2];
  uint64_t p_full[2];   // Pᵀ(j) written, indexed by j % 2
  uint64_t pv_done[2];  // PV(j) complete, indexed by j % 2
  uint64_t drain;
  uint32_t tmem_base;
  volatile int abort_flag;
  float red[4][64];   // per-warp partial maxima / sums
  float m_used[64];   // running maximum per head (scaled log2 units)
  float alpha[64];    // rescale factor of the current tile
  float l_tot[64];    // final row sums
};

constexpr size_t kDecodeSmem = 1024 + kQBytes + 2 * kStageBytes +
                               sizeof(int) * kDecodeMaxTopk + sizeof(DecodeCtl);
static_assert(kDecodeSmem <= 232448, "decode shared memory exceeds the per-CTA limit");

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

// Max (kMax) or sum over the 16 lanes of each half-warp of NP values per
// lane, by repeated halving: after the call lane l holds, in v[0 .. NP/16),
// the reduction for heads [l*NP/16, (l+1)*NP/16).
template <int NP, bool kMax>
__device__ __forceinline__ void half_warp_transpose_reduce(float* v, int lane) {
#pragma unroll
  for (int o = 8, n = NP; o >= 1; o >>= 1, n >>= 1) {
    const int half = n / 2;
    const bool upper = (lane & o) != 0;
#pragma unroll
    for (int i = 0; i < half; ++i) {
      const float send = upper ? v[i] : v[i + half];
      const float keep = upper ? v[i + half] : v[i];
      const float recv = __shfl_xor_sync(0xffffffffu, send, o);
      v[i] = kMax ? fmaxf(keep, recv) : keep + recv;
    }
  }
}

template <int NP>
__global__ void __launch_bounds__(kDecodeThreads, 1)
    sparse_decode_kernel(const __grid_constant__ CUtensorMap q_map, const DecodeArgs a) {
  static_assert(NP == 16 || NP == 32 || NP == 64, "head group width");
  constexpr uint32_t kSwP = NP == 64 ? ptx::kLayoutSw128 : (NP == 32 ? ptx::kLayoutSw64
                                                                     : ptx::kLayoutSw32);
  constexpr int kPRowBytes = NP * 2;  // one Pᵀ row (one key) in bytes
  constexpr int kPerLane = NP / 16;   // heads per lane after the transpose-reduce

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
  const int groups = (a.num_heads + 63) / 64;
  const int token = blockIdx.x / groups;
  const int group = blockIdx.x - token * groups;
  const int heads = a.num_heads < 64 ? a.num_heads : 64;  // real heads in this group
  const int head0 = group * 64;
  const int n_tiles = a.topk / kDecodeKeys;

  if (tid == 0) {
    ptx::mbar_init(ptx::smem_u32(&cb->q_full), 1);
    for (int s = 0; s < 2; ++s) {
      ptx::mbar_init(ptx::smem_u32(&cb->r_full[s]), 128);
      ptx::mbar_init(ptx::smem_u32(&cb->r_free[s]), 1);
      ptx::mbar_init(ptx::smem_u32(&cb->s_full[s]), 1);
      ptx::mbar_init(ptx::smem_u32(&cb->s_free[s]), 128);
    }
    for (int s = 0; s < 2; ++s) {
      ptx::mbar_init(ptx::smem_u32(&cb->p_full[s]), 128);
      ptx::mbar_init(ptx::smem_u32(&cb->pv_done[s]), 1);
    }
    ptx::mbar_init(ptx::smem_u32(&cb->drain), 2);
    cb->abort_flag = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 8) {
    ptx::tmem_alloc(ptx::smem_u32(&cb->tmem_base), 512);
    ptx::tmem_relinquish();
  }
  // Row table: physical cache row of every top-k slot, -1 if the slot is
  // outside the token's context or its page is out of range.
  {
    const int64_t context = (int64_t)a.max_pages * kDecodePage;
    const int* idx = a.topk_idx + (size_t)token * a.topk;
    const int* pt = a.page_table + (size_t)token * a.max_pages;
    for (int s = tid; s < a.topk; s += kDecodeThreads) {
      const int p = idx[s];
      int row = -1;
      if (p >= 0 && p < context) {
        const int page = pt[p / kDecodePage];
        if (page >= 0 && page < a.num_pages) row = page * kDecodePage + p % kDecodePage;
      }
      rows[s] = row;
    }
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = cb->tmem_base;

  if (warp >= 4 && warp < 8) {
    ptx::regs_dec<kDecodeGatherRegs>();
    // ------------------------------------------------------------ gather
    const int ptid = tid - 128;
    // Tile j goes to stage j % 2.  Each gather thread's copies of tile j
    // arrive on r_full[j % 2] by themselves when they land
    // (cp.async.mbarrier.arrive.noinc; the barrier expects 128 arrivals), so
    // no gather warp ever blocks on its own copies.  Stage reuse for tile j
    // waits for PV(j - 2), which needs only tiles <= j - 1.
    bool ok = true;
    for (int j = 0; j < n_tiles && ok; ++j) {
      if (j >= 2) {
        ok = wait_warp(ptx::smem_u32(&cb->r_free[j & 1]), ((j >> 1) - 1) & 1, abort_flag,
                       a.status);
        if (!ok) break;
      }
      const uint32_t dst0 = ptx::smem_u32(stage[j & 1]);
      const int* trow = rows + j * kDecodeKeys;
#pragma unroll 4
      for (int e = ptid; e < kDecodeKeys * 72; e += 128) {
        const int r = e / 72;
        const int c16 = e - r * 72;       // 16-byte unit within the row
        const int row = max(trow[r], 0);  // invalid slots read row 0 (masked later)
        const uint16_t* src = a.cache + (size_t)row * kDqk + c16 * 8;
        const int chunk = c16 >> 3, u = c16 & 7;
        const uint32_t dst = dst0 + chunk * kChunkBytes + r * 128 + ((u ^ (r & 7)) << 4);
        ptx::cp_async_16(dst, src);
      }
      ptx::cp_async_mbar_arrive(ptx::smem_u32(&cb->r_full[j & 1]));
    }
    cp_async_wait<0>();  // nothing of this thread is in flight at exit
  } else if (warp >= 8) {
    ptx::regs_dec<kDecodeControlRegs>();
    // ------------------------------------------------------------ MMA issuers
    constexpr uint32_t idesc_s = ptx::idesc_bf16_f32(64, NP, false, false);
    constexpr uint32_t idesc_o = ptx::idesc_bf16_f32(128, NP, true, true);
    if (warp == 8 && lane == 0) {
      // Sᵀ(j) = R(j) Qᵀ into Sᵀ buffer j % 2.
      ptx::prefetch_tmap(&q_map);
      ptx::mbar_arrive_expect_tx(ptx::smem_u32(&cb->q_full), 9 * NP * 128);
      for (int c = 0; c < 9; ++c)
        ptx::tma_load_3d(ptx::smem_u32(q_s + c * NP * 128), &q_map, ptx::smem_u32(&cb->q_full),
                         c * 64, head0, token);
      bool ok = wait_single(ptx::smem_u32(&cb->q_full), 0, abort_flag, a.status);
      const uint64_t qd = ptx::smem_desc(ptx::smem_u32(q_s), 16, 1024, ptx::kLayoutSw128);
      for (int j = 0; j < n_tiles && ok; ++j) {
        ok = wait_single(ptx::smem_u32(&cb->r_full[j & 1]), (j >> 1) & 1, abort_flag, a.status);
        if (ok && j >= 2)
          ok = wait_single(ptx::smem_u32(&cb->s_free[j & 1]), ((j >> 1) - 1) & 1, abort_flag,
                           a.status);
        if (!ok) break;
        // The gathered rows were written by cp.async (generic proxy); order
        // them before the tensor core's (async proxy) reads.
        ptx::fence_proxy_async_smem();
        ptx::tc_fence_after();
        const uint64_t rd =
            ptx::smem_desc(ptx::smem_u32(stage[j & 1]), 16, 1024, ptx::kLayoutSw128);
        const uint32_t d = tmem + (uint32_t)((j & 1) * NP);
#pragma unroll
        for (int k = 0; k < kDqk / 16; ++k) {
          const uint32_t in = (k & 3) * 32;
          ptx::mma_ss(d, ptx::desc_add(rd, (k >> 2) * kChunkBytes + in),
                      ptx::desc_add(qd, (k >> 2) * NP * 128 + in), idesc_s, k > 0 ? 1u : 0u);
        }
        ptx::mma_commit(ptx::smem_u32(&cb->s_full[j & 1]));
      }
      ptx::mma_commit(ptx::smem_u32(&cb->drain));
      wait_single(ptx::smem_u32(&cb->drain), 0, abort_flag, a.status);
    } else if (warp == 9 && lane == 0) {
      // Oᵀ += R(j)[:, 0:512]ᵀ Pᵀ(j), then release stage j % 2.
      bool ok = true;
      for (int j = 0; j < n_tiles && ok; ++j) {
        ok = wait_single(ptx::smem_u32(&cb->p_full[j & 1]), (j >> 1) & 1, abort_flag, a.status);
        if (!ok) break;
        ptx::fence_proxy_async_smem();
        ptx::tc_fence_after();
        const uint32_t ra = ptx::smem_u32(stage[j & 1]);
        // A = R[keys, 128m .. 128m+128)ᵀ: MN-major, two 64-wide chunks.
        const uint64_t ad = ptx::smem_desc(ra, kChunkBytes, 1024, ptx::kLayoutSw128);
        // B = Pᵀ[keys, heads] in the rope chunk: MN-major, NP wide.
        const uint64_t bd =
            ptx::smem_desc(ra + 8 * kChunkBytes, 8 * kPRowBytes, 8 * kPRowBytes, kSwP);
#pragma unroll
        for (int m = 0; m < 4; ++m) {
#pragma unroll
          for (int k = 0; k < kDecodeKeys / 16; ++k)
            ptx::mma_ss(tmem + 128u + (uint32_t)(m * NP),
                        ptx::desc_add(ad, 2 * m * kChunkBytes + k * 16 * 128),
                        ptx::desc_add(bd, k * 16 * kPRowBytes), idesc_o,
                        (j > 0 || k > 0) ? 1u : 0u);
        }
        ptx::mma_commit(ptx::smem_u32(&cb->pv_done[j & 1]));
        ptx::mma_commit(ptx::smem_u32(&cb->r_free[j & 1]));
      }
      ptx::mma_commit(ptx::smem_u32(&cb->drain));
      wait_single(ptx::smem_u32(&cb->drain), 0, abort_flag, a.status);
    }
    __syncwarp();
  } else {
    ptx::regs_inc<kDecodeSoftmaxRegs>();
    // ------------------------------------------------------------ softmax
    const int key_in_tile = warp * 16 + (lane & 15);  // meaningful for lanes 0-15
    const bool holds_key = lane < 16;
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
    const float sl2 = a.scale_log2;
    const float neg_inf = -__int_as_float(0x7f800000);
    float lpart[NP];
#pragma unroll
    for (int h = 0; h < NP; ++h) lpart[h] = 0.f;
    if (tid < 64) cb->m_used[tid] = neg_inf;
    named_bar_sync(1, 128);
    bool ok = true;
    for (int j = 0; j < n_tiles; ++j) {
      // Every wait is followed by a warpgroup-wide agreement, so that no warp
      // can be left alone at a later named barrier after another gave up.
      ok = wait_warp(ptx::smem_u32(&cb->s_full[j & 1]), (j >> 1) & 1, abort_flag, a.status);
      ok = named_bar_and(3, 128, ok);
      if (!ok) break;
      ptx::tc_fence_after();
      uint32_t sr[NP];
#pragma unroll
      for (int c = 0; c < NP; c += 16) ptx::tmem_ld16(tmem + lane_base + (j & 1) * NP + c, sr + c);
      ptx::tmem_wait_ld();
#pragma unroll
      for (int c = 0; c < NP; c += 16) ptx::reg_fence16(sr + c);
      ptx::tc_fence_before();
      ptx::mbar_arrive(ptx::smem_u32(&cb->s_free[j & 1]));  // Sᵀ buffer may be reused
      const bool valid = holds_key && rows[j * kDecodeKeys + key_in_tile] >= 0;
      float s[NP], v[NP];
#pragma unroll
      for (int h = 0; h < NP; ++h) {
        s[h] = valid ? __uint_as_float(sr[h]) : neg_inf;
        v[h] = s[h];
      }
      // Per-head maximum over the tile: 16 lanes, then 4 warps.
      half_warp_transpose_reduce<NP, true>(v, lane);
      if (holds_key) {
#pragma unroll
        for (int i = 0; i < kPerLane; ++i) cb->red[warp][lane * kPerLane + i] = v[i];
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
        float al[NP];
#pragma unroll
        for (int h = 0; h < NP; ++h) {
          al[h] = cb->alpha[h];
          lpart[h] *= al[h];
        }
        if (j > 0) {
          // Oᵀ holds the earlier tiles: wait for the last PV, then scale
          // every head column by its factor.
          ok = wait_warp(ptx::smem_u32(&cb->pv_done[(j - 1) & 1]), ((j - 1) >> 1) & 1,
                         abort_flag, a.status);
          ok = named_bar_and(3, 128, ok);
          if (!ok) break;
          ptx::tc_fence_after();
#pragma unroll
          for (int m = 0; m < 4; ++m) {
#pragma unroll
            for (int c = 0; c < NP; c += 16) {
              uint32_t o[16];
              const uint32_t addr = tmem + lane_base + 128u + m * NP + c;
              ptx::tmem_ld16(addr, o);
              ptx::tmem_wait_ld();
              ptx::reg_fence16(o);
#pragma unroll
              for (int i = 0; i < 16; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * al[c + i]);
              ptx::tmem_st16(addr, o);
            }
          }
          ptx::tmem_wait_st();
        }
      }
      // Probabilities and Pᵀ row for this thread's key.
      if (holds_key) {
        uint8_t* prow = stage[j & 1] + 8 * kChunkBytes + key_in_tile * kPRowBytes;
#pragma unroll
        for (int g = 0; g < NP / 8; ++g) {
          uint32_t pk[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int h0 = g * 8 + 2 * i;
            const float b0 = cb->m_used[h0], b1 = cb->m_used[h0 + 1];
            const float p0 = valid ? ptx::ex2(fmaf(s[h0], sl2, -b0)) : 0.f;
            const float p1 = valid ? ptx::ex2(fmaf(s[h0 + 1], sl2, -b1)) : 0.f;
            lpart[h0] += p0;
            lpart[h0 + 1] += p1;
            pk[i] = ptx::pack_bf16x2(p0, p1);
          }
          // Swizzled 16-byte unit g of row key_in_tile (pattern of the
          // NP*2-byte-wide layout: unit index XOR row bits).
          const int unit = kPerLane == 4 ? (g ^ (key_in_tile & 7))
                                         : (kPerLane == 2 ? (g ^ ((key_in_tile >> 1) & 3))
                                                          : (g ^ ((key_in_tile >> 2) & 1)));
          *reinterpret_cast<uint4*>(prow + unit * 16) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
        }
      }
      ptx::fence_proxy_async_smem();
      ptx::tc_fence_before();
      ptx::mbar_arrive(ptx::smem_u32(&cb->p_full[j & 1]));
    }
    if (ok) {
      // Row sums: reduce the per-thread partials over keys (16 lanes, 4 warps).
      half_warp_transpose_reduce<NP, false>(lpart, lane);
      if (holds_key) {
#pragma unroll
        for (int i = 0; i < kPerLane; ++i) cb->red[warp][lane * kPerLane + i] = lpart[i];
      }
      named_bar_sync(1, 128);
      if (tid < NP) {
        const float l = (cb->red[0][tid] + cb->red[1][tid]) + (cb->red[2][tid] + cb->red[3][tid]);
        cb->l_tot[tid] = l;
        if (a.lse && tid < heads) {
          const float m = cb->m_used[tid];
          a.lse[(size_t)(head0 + tid) * a.num_tokens + token] =
              l > 0.f ? (m + __log2f(l)) * 0.69314718055994531f : neg_inf;
        }
      }
      named_bar_sync(1, 128);
      // A commit tracks every earlier MMA of its issuer, so PV(n-1) done
      // means all of Oᵀ is final.
      ok = wait_warp(ptx::smem_u32(&cb->pv_done[(n_tiles - 1) & 1]), ((n_tiles - 1) >> 1) & 1,
                     abort_flag, a.status);
    }
    if (ok) {
      ptx::tc_fence_after();
      // Epilogue: lane = dv row within each 128-row tile of Oᵀ.
#pragma unroll 1
      for (int m = 0; m < 4; ++m) {
        const int dv = m * 128 + warp * 32 + lane;
#pragma unroll
        for (int c = 0; c < NP; c += 16) {
          uint32_t o[16];
          ptx::tmem_ld16(tmem + lane_base + 128u + m * NP + c, o);
          ptx::tmem_wait_ld();
          ptx::reg_fence16(o);
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const int h = c + i;
            if (h < heads) {
              const float l = cb->l_tot[h];
              const float val = l > 0.f ? __uint_as_float(o[i]) / l : 0.f;
              const uint32_t b = ptx::pack_bf16x2(val, 0.f) & 0xffffu;
              a.out[((size_t)token * a.num_heads + head0 + h) * kDv + dv] = (uint16_t)b;
            }
          }
        }
      }
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 8) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, 512);
  }
}

template <int NP>
inline cudaError_t launch_decode_np(const CUtensorMap& map, const DecodeArgs& a,
                                    cudaStream_t stream) {
  static bool attr_done[64] = {false};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!attr_done[dev]) {
    e = cudaFuncSetAttribute(sparse_decode_kernel<NP>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)kDecodeSmem);
    if (e != cudaSuccess) return e;
    attr_done[dev] = true;
  }
  const int groups = (a.num_heads + 63) / 64;
  sparse_decode_kernel<NP><<<a.num_tokens * groups, kDecodeThreads, kDecodeSmem, stream>>>(map, a);
  return cudaGetLastError();
}

}  // namespace fa
