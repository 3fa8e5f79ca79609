// sparse_decode_kernel.cuh -- sparse-MLA decode for sm_103a.
//
// One CTA per (token, group of up to 64 query heads).  All heads of a token
// share the token's top-k gathered latent rows R (576 = 512 latent + 64 rope
// columns; the value is the 512 latent columns).  Per tile of 128 keys:
//
//   S  = Q · R[:, 0:576]ᵀ        M = 64 heads, N = 128 keys, K = 576 (36 MMAs)
//   Oᵀ += R[:, 0:512]ᵀ · Pᵀ      M = 128 rows of d_v (x4), N = 64 heads, K = 128
//
// A tensor-core instruction costs about the same for M = 64 as for M = 128
// and for any N up to 128, so heads go on M for S (one MMA covers 128 keys)
// while Oᵀ keeps d_v on M.  TMEM: S double buffer at columns [0,128) and
// [128,256) (64-row layout: head h in lane 32*(h/16) + h%16), Oᵀ at
// [256,512) (row = lane).  One softmax thread per head owns a whole S row:
// max, exp2 and sum stay in registers.
//
// Rows are streamed as 64-column chunks of 128 keys (16 KB): for tile t the 9
// chunks used by S go through the S ring (consumed only by the S issuer),
// and for P·V the 8 latent chunks are gathered again (L2 hits) into the V
// ring (consumed only by the PV issuer), so a tile never has to be resident
// whole.  Each ring has exactly one in-order consumer, which is what makes
// its mbarrier parity waits unambiguous.  The gather fills them in the order
// S(0); then per tile t: S(t+1), V(t).  The V ring has an even number of
// slots and V groups of 8, so the two chunks of each 128-row d_v tile sit in
// adjacent slots (one MN-major operand).
//
//   gather warps 4-7   16-byte cp.async, one mbarrier arrival per thread and
//                      chunk when its copies land (cp.async.mbarrier.arrive);
//   warp 8             TMEM owner; TMA-loads Q; issues S as chunks land;
//   warp 9             issues Oᵀ += Vᵀ Pᵀ once Pᵀ(t) is written;
//   softmax warps 0-3  lanes 0-15 = heads; lazy rescale of Oᵀ columns.
//
// Method source: vLLM API page "vllm.v1.attention.backends.mla.
// flashattn_mla_sparse" -- FlashAttnMLASparseFA4Backend (BF16 cache only; head
// size 576 split into 512 latent + 64 rope; cache block size a multiple of 64;
// index_topk % 128 == 0 so the gathered indices are whole 128-key tiles;
// 8..128 heads) and _fa4_varlen_scalars (one query row per token).
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "sm103_ptx.cuh"
#include "varlen_fwd_kernel.cuh"  // kStatusTimeout, bounded waits, kRescaleLog2

namespace fa {

constexpr int kDecodePage = 64;
constexpr int kDecodeThreads = 384;  // softmax 0-3, gather 4-7, S issuer 8, PV issuer 9
// Register split (launch: 168 x 384 = 64512): softmax 128 x 240, gather
// 128 x 88, control 128 x 56 = 49152.
constexpr uint32_t kDecodeSoftmaxRegs = 240;
constexpr uint32_t kDecodeGatherRegs = 88;
constexpr uint32_t kDecodeControlRegs = 56;
constexpr int kDecodeKeys = 128;      // keys per tile
constexpr int kDecodeMaxTopk = 2048;  // row table held in shared memory
constexpr int kDqk = 576, kDv = 512;
constexpr int kChunkBytes = kDecodeKeys * 128;  // 128 keys x 64 columns bf16
constexpr int kRingS = 3;                       // S-ring chunk slots
constexpr int kRingV = 4;                       // V-ring chunk slots (even)
constexpr int kRing = kRingS + kRingV;
constexpr int kSGroup = 9;                      // chunks per tile for S
constexpr int kVGroup = 8;                      // chunks per tile for P·V
constexpr int kQBytes = 9 * 64 * 128;           // 64 heads x 576
constexpr int kPBytes = 64 * kDecodeKeys * 2;   // Pᵀ of one tile, 64 heads x 128 keys

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
  uint64_t full_s[kRingS];
  uint64_t free_s[kRingS];
  uint64_t full_v[kRingV];
  uint64_t free_v[kRingV];
  uint64_t s_full[2];
  uint64_t s_free[2];
  uint64_t p_full[2];  // per Pᵀ buffer: the softmax may run one tile ahead of PV
  uint64_t p_free[2];  // PV(t) complete, per Pᵀ buffer t % 2
  uint64_t drain;
  uint32_t tmem_base;
  volatile int abort_flag;
  uint32_t valid[kDecodeMaxTopk / 32];  // bit per top-k slot
  float alpha[64];
  float l_tot[64];
};

constexpr size_t kDecodeSmem = 1024 + kQBytes + 2 * kPBytes + (size_t)kRing * kChunkBytes +
                               sizeof(int) * kDecodeMaxTopk + sizeof(DecodeCtl);

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

__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.wait_all;" ::: "memory");
}


__global__ void __launch_bounds__(kDecodeThreads, 1)
    sparse_decode_kernel(const __grid_constant__ CUtensorMap q_map, const DecodeArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* q_s = smem;
  uint8_t* p_s = smem + kQBytes;  // two Pᵀ buffers
  uint8_t* ring_s = p_s + 2 * kPBytes;              // kRingS slots
  uint8_t* ring_v = ring_s + kRingS * kChunkBytes;   // kRingV slots
  int* rows = reinterpret_cast<int*>(ring_v + kRingV * kChunkBytes);
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
    for (int s = 0; s < kRingS; ++s) {
      ptx::mbar_init(ptx::smem_u32(&cb->full_s[s]), 128);
      ptx::mbar_init(ptx::smem_u32(&cb->free_s[s]), 1);
    }
    for (int s = 0; s < kRingV; ++s) {
      ptx::mbar_init(ptx::smem_u32(&cb->full_v[s]), 128);
      ptx::mbar_init(ptx::smem_u32(&cb->free_v[s]), 1);
    }
    for (int b = 0; b < 2; ++b) {
      ptx::mbar_init(ptx::smem_u32(&cb->s_full[b]), 1);
      ptx::mbar_init(ptx::smem_u32(&cb->s_free[b]), 128);
      ptx::mbar_init(ptx::smem_u32(&cb->p_free[b]), 1);
      ptx::mbar_init(ptx::smem_u32(&cb->p_full[b]), 128);
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
  // outside the token's context or its page is out of range; then a validity
  // bit per slot.
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
  __syncthreads();
  for (int w32 = tid; w32 < a.topk / 32; w32 += kDecodeThreads) {
    uint32_t bits = 0;
    for (int b = 0; b < 32; ++b) bits |= (rows[w32 * 32 + b] >= 0 ? 1u : 0u) << b;
    cb->valid[w32] = bits;
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = cb->tmem_base;

  if (warp >= 4 && warp < 8) {
    ptx::regs_dec<kDecodeGatherRegs>();
    // ------------------------------------------------------------ gather
    const int ptid = tid - 128;
    bool ok = true;
    int ps = 0, pv = 0;  // positions in the S and V rings
    // One chunk: 128 rows x 8 units of 16 bytes; thread ptid copies units
    // e = ptid + 128 i (row e / 8, unit e % 8) -- 8 per thread, consecutive
    // threads on consecutive 16-byte units of a row.
    auto fill = [&](uint8_t* ring, uint64_t* full, uint64_t* free_, int nslot, int& pos,
                    int tile, int col_chunk) -> bool {
      const int s = pos % nslot;
      if (pos >= nslot) {
        if (!wait_warp(ptx::smem_u32(&free_[s]), ((pos / nslot) - 1) & 1, abort_flag, a.status))
          return false;
      }
      const uint32_t dst0 = ptx::smem_u32(ring + s * kChunkBytes);
      const int* trow = rows + tile * kDecodeKeys;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int e = ptid + 128 * i;
        const int r = e >> 3, u = e & 7;
        const int row = max(trow[r], 0);  // invalid slots read row 0 (masked later)
        const uint16_t* src = a.cache + (size_t)row * kDqk + col_chunk * 64 + u * 8;
        ptx::cp_async_16(dst0 + r * 128 + ((u ^ (r & 7)) << 4), src);
      }
      ptx::cp_async_mbar_arrive(ptx::smem_u32(&full[s]));
      ++pos;
      return true;
    };
    for (int c = 0; c < kSGroup && ok; ++c)
      ok = fill(ring_s, cb->full_s, cb->free_s, kRingS, ps, 0, c);
    for (int t = 0; t < n_tiles && ok; ++t) {
      if (t + 1 < n_tiles)
        for (int c = 0; c < kSGroup && ok; ++c)
          ok = fill(ring_s, cb->full_s, cb->free_s, kRingS, ps, t + 1, c);
      for (int c = 0; c < kVGroup && ok; ++c)
        ok = fill(ring_v, cb->full_v, cb->free_v, kRingV, pv, t, c);
    }
    cp_async_wait_all();  // nothing of this thread is in flight at exit
  } else if (warp >= 8) {
    ptx::regs_dec<kDecodeControlRegs>();
    if (warp == 8 && lane == 0) {
      // ---------------------------------------------------------- S issuer
      constexpr uint32_t idesc_s = ptx::idesc_bf16_f32(64, kDecodeKeys, false, false);
      ptx::prefetch_tmap(&q_map);
      ptx::mbar_arrive_expect_tx(ptx::smem_u32(&cb->q_full), kQBytes);
      for (int c = 0; c < 9; ++c)
        ptx::tma_load_3d(ptx::smem_u32(q_s + c * 64 * 128), &q_map, ptx::smem_u32(&cb->q_full),
                         c * 64, head0, token);
      bool ok = wait_single(ptx::smem_u32(&cb->q_full), 0, abort_flag, a.status);
      const uint64_t qd = ptx::smem_desc(ptx::smem_u32(q_s), 16, 1024, ptx::kLayoutSw128);
      for (int t = 0; t < n_tiles && ok; ++t) {
        const int b = t & 1;
        if (t >= 2) {
          ok = wait_single(ptx::smem_u32(&cb->s_free[b]), ((t >> 1) - 1) & 1, abort_flag,
                           a.status);
          if (!ok) break;
        }
        const uint32_t d = tmem + (uint32_t)(b * kDecodeKeys);
        for (int c = 0; c < kSGroup && ok; ++c) {
          const int pp = t * kSGroup + c, s = pp % kRingS;
          ok = wait_single(ptx::smem_u32(&cb->full_s[s]), (pp / kRingS) & 1, abort_flag, a.status);
          if (!ok) break;
          // Rows landed by cp.async (generic proxy): order them before the
          // tensor core's (async proxy) reads.
          ptx::fence_proxy_async_smem();
          ptx::tc_fence_after();
          const uint64_t rd = ptx::smem_desc(ptx::smem_u32(ring_s + s * kChunkBytes), 16, 1024,
                                             ptx::kLayoutSw128);
#pragma unroll
          for (int k = 0; k < 4; ++k)
            ptx::mma_ss(d, ptx::desc_add(qd, c * 64 * 128 + k * 32), ptx::desc_add(rd, k * 32),
                        idesc_s, (c > 0 || k > 0) ? 1u : 0u);
          ptx::mma_commit(ptx::smem_u32(&cb->free_s[s]));
        }
        if (ok) ptx::mma_commit(ptx::smem_u32(&cb->s_full[b]));
      }
      ptx::mma_commit(ptx::smem_u32(&cb->drain));
      wait_single(ptx::smem_u32(&cb->drain), 0, abort_flag, a.status);
    } else if (warp == 9 && lane == 0) {
      // ---------------------------------------------------------- PV issuer
      constexpr uint32_t idesc_o = ptx::idesc_bf16_f32(128, 64, true, false);
      bool ok = true;
      for (int t = 0; t < n_tiles && ok; ++t) {
        ok = wait_single(ptx::smem_u32(&cb->p_full[t & 1]), (t >> 1) & 1, abort_flag, a.status);
        if (!ok) break;
        // B = Pᵀ(t): K-major [64 heads x 128 keys] in two 64-key chunks.
        const uint64_t pd =
            ptx::smem_desc(ptx::smem_u32(p_s + (t & 1) * kPBytes), 16, 1024, ptx::kLayoutSw128);
        for (int m = 0; m < 4 && ok; ++m) {
          const int pa = t * kVGroup + 2 * m, sa = pa % kRingV;  // even: sa + 1 < kRingV
          ok = wait_single(ptx::smem_u32(&cb->full_v[sa]), (pa / kRingV) & 1, abort_flag,
                           a.status);
          if (ok)
            ok = wait_single(ptx::smem_u32(&cb->full_v[sa + 1]), ((pa + 1) / kRingV) & 1,
                             abort_flag, a.status);
          if (!ok) break;
          ptx::fence_proxy_async_smem();
          ptx::tc_fence_after();
          // A = R[keys, 128m .. 128m+128)ᵀ: MN-major over two adjacent slots.
          const uint64_t ad = ptx::smem_desc(ptx::smem_u32(ring_v + sa * kChunkBytes),
                                             kChunkBytes, 1024, ptx::kLayoutSw128);
          const uint32_t d = tmem + 256u + (uint32_t)(m * 64);
#pragma unroll
          for (int k = 0; k < kDecodeKeys / 16; ++k)
            ptx::mma_ss(d, ptx::desc_add(ad, k * 16 * 128),
                        ptx::desc_add(pd, (k >> 2) * 64 * 128 + (k & 3) * 32), idesc_o,
                        (t > 0 || k > 0) ? 1u : 0u);
          ptx::mma_commit(ptx::smem_u32(&cb->free_v[sa]));
          ptx::mma_commit(ptx::smem_u32(&cb->free_v[sa + 1]));
        }
        if (!ok) break;
        ptx::mma_commit(ptx::smem_u32(&cb->p_free[t & 1]));
      }
      ptx::mma_commit(ptx::smem_u32(&cb->drain));
      wait_single(ptx::smem_u32(&cb->drain), 0, abort_flag, a.status);
    }
    __syncwarp();
  } else {
    ptx::regs_inc<kDecodeSoftmaxRegs>();
    // ------------------------------------------------------------ softmax
    const int h = warp * 16 + (lane & 15);  // head row (meaningful for lanes 0-15)
    const bool holds_row = lane < 16;
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
    const float sl2 = a.scale_log2;
    const float neg_inf = -__int_as_float(0x7f800000);
    float m_used = neg_inf, l = 0.f;
    bool ok = true;
    for (int t = 0; t < n_tiles; ++t) {
      // Every wait is followed by a warpgroup-wide agreement, so that no warp
      // can be left alone at a later named barrier after another gave up.
      ok = wait_warp(ptx::smem_u32(&cb->s_full[t & 1]), (t >> 1) & 1, abort_flag, a.status);
      ok = named_bar_and(3, 128, ok);
      if (!ok) break;
      ptx::tc_fence_after();
      uint32_t sr[kDecodeKeys];
#pragma unroll
      for (int q = 0; q < kDecodeKeys / 32; ++q)
        ptx::tmem_ld32(tmem + lane_base + (t & 1) * kDecodeKeys + q * 32, sr + q * 32);
      ptx::tmem_wait_ld();
#pragma unroll
      for (int q = 0; q < kDecodeKeys / 16; ++q) ptx::reg_fence16(sr + q * 16);
      ptx::tc_fence_before();
      ptx::mbar_arrive(ptx::smem_u32(&cb->s_free[t & 1]));  // S buffer may be reused
      float s[kDecodeKeys];
      uint32_t vb[kDecodeKeys / 32];
#pragma unroll
      for (int w = 0; w < kDecodeKeys / 32; ++w) vb[w] = cb->valid[t * (kDecodeKeys / 32) + w];
#pragma unroll
      for (int c = 0; c < kDecodeKeys; ++c)
        s[c] = ((vb[c >> 5] >> (c & 31)) & 1u) ? __uint_as_float(sr[c]) : neg_inf;
      float mx[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) mx[k] = fmaxf(s[k], s[k + 4]);
#pragma unroll
      for (int c = 8; c < kDecodeKeys; c += 8) {
#pragma unroll
        for (int k = 0; k < 4; ++k) mx[k] = ptx::max3(mx[k], s[c + k], s[c + k + 4]);
      }
      const float m_tile = ptx::max3(mx[0], mx[1], fmaxf(mx[2], mx[3])) * sl2;
      const int need = (holds_row && m_tile > m_used + kRescaleLog2) ? 1 : 0;
      float alpha = 1.f;
      if (need) {
        alpha = (m_used == neg_inf) ? 0.f : ptx::ex2(m_used - m_tile);
        m_used = m_tile;
        l *= alpha;
      }
      if (holds_row) cb->alpha[h] = alpha;
      if (named_bar_or(2, 128, need) && t > 0) {
        // Oᵀ holds the earlier tiles: wait for PV(t - 1) (use (t-1)/2 of its
        // Pᵀ buffer's barrier; the previous use was observed, so the parity
        // wait is unambiguous), then scale every head column by its factor.
        ok = wait_warp(ptx::smem_u32(&cb->p_free[(t - 1) & 1]), ((t - 1) >> 1) & 1, abort_flag,
                       a.status);
        ok = named_bar_and(3, 128, ok);
        if (!ok) break;
        ptx::tc_fence_after();
#pragma unroll 1
        for (int m = 0; m < 4; ++m) {
#pragma unroll
          for (int c = 0; c < 64; c += 16) {
            uint32_t o[16];
            const uint32_t addr = tmem + lane_base + 256u + m * 64 + c;
            ptx::tmem_ld16(addr, o);
            ptx::tmem_wait_ld();
            ptx::reg_fence16(o);
#pragma unroll
            for (int i = 0; i < 16; ++i)
              o[i] = __float_as_uint(__uint_as_float(o[i]) * cb->alpha[c + i]);
            ptx::tmem_st16(addr, o);
          }
        }
        ptx::tmem_wait_st();
      }
      const float base = (m_used == neg_inf) ? 0.f : m_used;
      const uint64_t sl2x2 = ptx::f2_pack(sl2, sl2);
      const uint64_t nbx2 = ptx::f2_pack(-base, -base);
      uint64_t ls2[4] = {0ull, 0ull, 0ull, 0ull};
      uint32_t pr[kDecodeKeys / 2];
#pragma unroll
      for (int c = 0; c < kDecodeKeys; c += 2) {
        float x0, x1;
        ptx::f2_unpack(ptx::fma2(ptx::f2_pack(s[c], s[c + 1]), sl2x2, nbx2), x0, x1);
        const float p0 = ptx::ex2(x0);  // masked keys: ex2(-inf) = 0
        const float p1 = ptx::ex2(x1);
        ls2[(c >> 1) & 3] = ptx::add2(ls2[(c >> 1) & 3], ptx::f2_pack(p0, p1));
        pr[c >> 1] = ptx::pack_bf16x2(p0, p1);
      }
      {
        float a0, a1, b0, b1;
        ptx::f2_unpack(ptx::add2(ls2[0], ls2[1]), a0, a1);
        ptx::f2_unpack(ptx::add2(ls2[2], ls2[3]), b0, b1);
        l += (a0 + b0) + (a1 + b1);
      }
      // Pᵀ buffer t % 2 is free once PV(t - 2) has completed.
      if (t >= 2) {
        ok = wait_warp(ptx::smem_u32(&cb->p_free[t & 1]), ((t >> 1) - 1) & 1, abort_flag,
                       a.status);
        ok = named_bar_and(3, 128, ok);
        if (!ok) break;
      }
      if (holds_row) {
        // Row h of the K-major [64 heads x 128 keys] buffer: two 64-key
        // chunks of 128 bytes per row, 16-byte units swizzled by row.
        uint8_t* pb = p_s + (t & 1) * kPBytes;
#pragma unroll
        for (int g = 0; g < kDecodeKeys / 8; ++g) {
          const int chunk = g >> 3, u = g & 7;
          *reinterpret_cast<uint4*>(pb + chunk * 64 * 128 + h * 128 + ((u ^ (h & 7)) << 4)) =
              make_uint4(pr[4 * g], pr[4 * g + 1], pr[4 * g + 2], pr[4 * g + 3]);
        }
      }
      ptx::fence_proxy_async_smem();
      ptx::tc_fence_before();
      ptx::mbar_arrive(ptx::smem_u32(&cb->p_full[t & 1]));
    }
    if (ok) {
      if (holds_row) {
        cb->l_tot[h] = l;
        if (a.lse && h < heads)
          a.lse[(size_t)(head0 + h) * a.num_tokens + token] =
              l > 0.f ? (m_used + __log2f(l)) * 0.69314718055994531f : neg_inf;
      }
      named_bar_sync(1, 128);
      // PVs complete in issue order: PV(n - 1) done means Oᵀ is final.
      ok = wait_warp(ptx::smem_u32(&cb->p_free[(n_tiles - 1) & 1]), ((n_tiles - 1) >> 1) & 1,
                     abort_flag, a.status);
    }
    if (ok) {
      ptx::tc_fence_after();
      // Epilogue: lane = d_v row within each 128-row tile of Oᵀ, columns = heads.
#pragma unroll 1
      for (int m = 0; m < 4; ++m) {
        const int dv = m * 128 + warp * 32 + lane;
#pragma unroll
        for (int c = 0; c < 64; c += 16) {
          uint32_t o[16];
          ptx::tmem_ld16(tmem + lane_base + 256u + m * 64 + c, o);
          ptx::tmem_wait_ld();
          ptx::reg_fence16(o);
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const int hh = c + i;
            if (hh < heads) {
              const float lh = cb->l_tot[hh];
              const float val = lh > 0.f ? __uint_as_float(o[i]) / lh : 0.f;
              const uint32_t bits = ptx::pack_bf16x2(val, 0.f) & 0xffffu;
              a.out[((size_t)token * a.num_heads + head0 + hh) * kDv + dv] = (uint16_t)bits;
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

inline cudaError_t launch_sparse_decode(const CUtensorMap& map, const DecodeArgs& a,
                                        cudaStream_t stream) {
  static bool attr_done[64] = {false};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!attr_done[dev]) {
    e = cudaFuncSetAttribute(sparse_decode_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)kDecodeSmem);
    if (e != cudaSuccess) return e;
    attr_done[dev] = true;
  }
  const int groups = (a.num_heads + 63) / 64;
  sparse_decode_kernel<<<a.num_tokens * groups, kDecodeThreads, kDecodeSmem, stream>>>(map, a);
  return cudaGetLastError();
}

}  // namespace fa
