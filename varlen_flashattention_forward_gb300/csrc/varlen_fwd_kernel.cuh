// varlen_fwd_kernel.cuh -- variable-length attention forward for sm_103a.
//
// One persistent CTA per SM walks its share of a static, longest-first list
// of work items (dealt in snake order, snake_item).
// A work item is (sequence, head, pair of 128-row query tiles).  Per item:
//
//   producer warp   TMA: Q tiles once, then K_j and V_j tiles into two rings
//                   of shared-memory slots (K ring, V ring) guarded by
//                   mbarriers; L2 prefetches where a ring is shallow (one K
//                   slot, one Q pair, split-KV streams).
//   MMA warps 9/10  one warp per query tile t, running converged; an
//                   elect.sync-chosen lane issues its tcgen05.mma groups:
//                     S_t = Q_t K_jᵀ          (SS form, fp32 accumulator in TMEM)
//                     O_t += P_t V_j          (TS form, P read from TMEM)
//                   Two issuers keep the two tiles' chains independent: a
//                   warp blocked on a full tensor-core queue while issuing
//                   one tile's MMAs cannot delay the other tile.  For
//                   d_qk == d_v they take turns per issue group (tile 0 group
//                   g, tile 1 group g, tile 0 group g+1, ...) so the tensor
//                   core alternates between the tiles and each tile's softmax
//                   runs while the other tile's MMAs execute (ping-pong);
//                   for MLA shapes and d_v <= 64 they run free
//                   (VarlenCfg::turns).
//   softmax WG t    one thread per query row (TMEM lane): loads S_t with the
//                   sm_103 reducing TMEM load (values + per-32-column max),
//                   masks only boundary tiles (software 3-input max there),
//                   exp2, lazy O rescale (threshold kRescaleLog2), writes P_t
//                   as bf16 into the S_t columns, or at d_v <= 64 into
//                   columns of its own so that S_t(j + 1) can be issued once
//                   S_t(j) is loaded (VarlenCfg::p_cols), in two halves for
//                   small d_v (VarlenCfg::split_pv), and at the end normalises O_t
//                   and writes O (through the dead Q tile and bulk copies
//                   where VarlenCfg::stage_o) and the LSE.
//
// TMEM (512 columns x 128 lanes x 32 bit):
//   [  0,128) S_0 / P_0   [128,256) S_1 / P_1   [256,384) O_0   [384,512) O_1
//   (d_v <= 64: P_t at [320 + 128 t, +64), beside O_t)
//
// Shared memory: one or two pairs of Q tiles, the K ring, the V ring,
// mbarriers, and the work list.  Q and K tiles are column chunks of
// the head dimension, 64 bf16 wide with the 128-byte swizzle (or one narrower
// tail chunk with the 32/64-byte swizzle); V tiles are atoms of 16, 32 or 64
// columns (v_atom_width).  Each is both the TMA box layout and the UMMA
// canonical layout (K-major for Q and K, MN-major for V).
//
// Method sources: sglang PR #41344 (FA4 path on Blackwell), "Motivation" and
// "Modifications" (the row max taken by tcgen05.ld.red on sm_103 for tiles
// that need no masking, the software reduction on masked tiles, bit-identical
// results; exp2 after the max; rescale threshold; only tiles that need
// masking are masked, and the first processed tile is a masked one); vLLM API page
// "vllm.v1.attention.backends.mla.prefill.flash_attn", FA4MLAPrefillKernel
// CompileKey (128-row query tile, q_stage of two tiles per CTA, static
// persistent scheduler).
#pragma once

#include <atomic>
#include <cstdint>
#include <cstring>
#include <cuda.h>
#include <cuda_runtime.h>

#include "sm103_ptx.cuh"

namespace fa {

constexpr int kVarlenThreads = 384;   // 2 softmax warpgroups + {producer, 2 MMA, 1 idle} warps
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;           // issuer of tile 0 (and TMEM owner); warp 10 issues tile 1
// Register split (launch: 168 per thread x 384 threads = 64512):
// softmax warpgroups 2 x 128 x 208 + control warpgroup 128 x 64 = 61440.
constexpr uint32_t kSoftmaxRegs = 208;
constexpr uint32_t kControlRegs = 64;
constexpr int kBM = 128;              // query rows per tile
constexpr int kBN = 128;              // keys per KV tile
constexpr int kRowsPerItem = 2 * kBM; // two query tiles per work item
constexpr int kMaxBatch = 2048;       // sequences per launch (larger batches: several launches)
constexpr float kRescaleLog2 = 8.0f;  // lazy rescale threshold, log2 units
constexpr int kSmemBudget = 232448;   // 227 KB opt-in per CTA
constexpr int kBarrierBytes = 480;    // VarlenBarriers, reserved in the smem budget

constexpr unsigned int kStatusTimeout = 1u;

// Head-dim chunking: full 64-element chunks plus an optional 16- or 32-element
// tail (dims padded to a multiple of 16 with TMA zero fill).
template <int D>
struct HeadDim {
  static constexpr int padded = (D + 15) / 16 * 16;
  static constexpr int full = padded / 64;
  static constexpr int tail = padded % 64;  // 0, 16 or 32
  static constexpr int chunks = full + (tail ? 1 : 0);
  static_assert(tail == 0 || tail == 16 || tail == 32, "unsupported head dim");
  // Byte offset of chunk c inside a tile of `rows` rows.
  __host__ __device__ static constexpr int chunk_off(int c, int rows) { return c * rows * 128; }
  __host__ __device__ static constexpr int chunk_width(int c) { return c < full ? 64 : tail; }
  static constexpr int tile_bytes(int rows) { return rows * padded * 2; }
};

template <int V>
struct IntTag {
  static constexpr int value = V;
};

__host__ __device__ constexpr uint32_t layout_for_width(int w) {
  return w == 64 ? ptx::kLayoutSw128 : (w == 32 ? ptx::kLayoutSw64 : ptx::kLayoutSw32);
}

// Width (elements) of the swizzle atoms V is stored in: the widest of 64,
// 32 and 16 that divides d_v rounded up to 16, so that a V tile holds no
// padding beyond that rounding (d_v = 80: five 16-wide atoms, 20 KB per 128
// keys, instead of two zero-filled 64-wide atoms, 32 KB).  The host encodes
// the V tensor map with the same box width.
__host__ __device__ constexpr int v_atom_width(int d_v) {
  return ((d_v + 15) / 16 * 16) % 64 == 0 ? 64
         : (((d_v + 15) / 16 * 16) % 32 == 0 ? 32 : 16);
}

template <int D_QK, int D_V>
struct VarlenCfg {
  using QK = HeadDim<D_QK>;
  using VD = HeadDim<D_V>;
  static constexpr int q_tile_bytes = QK::tile_bytes(kBM);
  static constexpr int k_tile_bytes = QK::tile_bytes(kBN);
  // V is stored MN-major as v_atoms atoms of v_atom columns (TMA zero-fills
  // columns past d_v), so that P V is one MMA of N = pv_n per 16 keys.
  static constexpr int v_atom = v_atom_width(D_V);
  static constexpr int v_atoms = VD::padded / v_atom;
  static constexpr int v_atom_bytes = kBN * v_atom * 2;
  static constexpr int v_tile_bytes = v_atoms * v_atom_bytes;
  static constexpr int pv_n = VD::padded;
  // K and V tiles live in two rings with their own slot sizes.
  static constexpr int k_slot_bytes = (k_tile_bytes + 1023) / 1024 * 1024;
  static constexpr int v_slot_bytes = (v_tile_bytes + 1023) / 1024 * 1024;
  static constexpr int sched_bytes_max = 8 * (kMaxBatch + 1) + 4 * kVarlenThreads;
  // Shared memory left for the rings next to `pairs` pairs of Q tiles.
  static constexpr int ring_bytes(int pairs) {
    return kSmemBudget - (1024 /*align*/ + pairs * 2 * q_tile_bytes + kBarrierBytes) -
           sched_bytes_max;
  }
  static constexpr int min_(int a, int b) { return a < b ? a : b; }
  // Equal K and V slot counts, at most 8 each.
  static constexpr int pairs_fit(int pairs) {
    return min_(8, ring_bytes(pairs) / (k_slot_bytes + v_slot_bytes));
  }
  // Two pairs of Q buffers, used by alternate work items, so that the next
  // item's Q loads while the current item runs (a short sequence's item is
  // only a few KV steps long, and its Q would otherwise wait for the
  // current item's last S); only where three K and three V slots still fit.
  static constexpr int q_pairs = pairs_fit(2) >= 3 ? 2 : 1;
  static constexpr int nk = pairs_fit(q_pairs);
  // With two Q pairs, a tile's O rows are staged in its item's Q tile (dead
  // once the item's last S is done) and written by one bulk copy per row;
  // the softmax warpgroup, not the issuer, then releases the Q buffer once
  // the copies have read it.  Plain 16-byte stores from one thread per row
  // touch 32 rows per warp instruction and hold up every later load and store
  // of the SM: measured on 256-token ViT windows, 21 % of the kernel time.
  static constexpr bool stage_o =
      q_pairs == 2 && kBM * D_V * 2 <= q_tile_bytes && (D_V * 2) % 16 == 0;
  // One more V slot where the rest allows: a KV step needs V_j first, and
  // V_{j+1} can then load while P V_j still reads V_j.
  static constexpr int nv = min_(8, nk + ((ring_bytes(q_pairs) - nk * (k_slot_bytes + v_slot_bytes)) /
                                          v_slot_bytes > 0 ? 1 : 0));
  static_assert(nk >= 1 && nv >= 2, "shared memory too small for the K and V rings");
  // L2 prefetches by the producer.  With one K slot (MLA), K_{j+1} of an
  // item as K_j goes out (causal 4 x 4096: 1979 -> 1927 us); in a split-KV
  // launch, K_{j+1} and V_{j+1} as K_j goes out (each part streams keys no
  // other CTA reads, and the two-slot rings of d128 keep too few bytes in
  // flight: 256 rows x 65536 keys 154 -> 140 us; where tiles are shared
  // between items the same prefetch cost 2-4 %); with one Q
  // pair and a deeper K ring (d96, d128), an item's Q and first K/V tiles
  // when it is published (256-token windows at d128: 64-66 us against
  // 66-68; for MLA the same prefetch cost back the gain of the K one).
  static constexpr bool k_prefetch = nk == 1;
  static constexpr bool item_prefetch = q_pairs == 1 && nk > 1;
  static_assert(pv_n <= 128, "O accumulator wider than its TMEM region");
  // Issue order between the two query tiles' MMA groups.  Strict turns
  // (ping-pong) for d_qk == d_v, where a group is short and free-running
  // issuers fall into lockstep (measured: ViT d80 0.57 vs 0.67 ms); free
  // running for d_qk > d_v (MLA 192/128: long S groups, one K slot),
  // where turns cost more than they save (causal 4 x 4096: 794 vs 699
  // TFLOP/s).
  // P in TMEM columns of its own, next to O_t, where d_v leaves them free
  // (d_v <= 64: 2 x (128 S + 64 O + 64 P) = 512 columns): S_t(j + 1) is then
  // issued as soon as the softmax has loaded S_t(j), not after it has
  // written P_t(j), so that the tile's next S runs during its exp2 phase
  // and the softmax of step j + 1 finds S waiting (ViT d64: 406 -> 396 us;
  // the step is then bound by the softmax's own exp2 and TMEM latency).
  static constexpr bool p_cols = pv_n <= 64;
  // Not with p_cols, where the two tiles' S issues taking turns measured
  // 7 % slower on ViT d64 (424.6 against 395.9 us free running).
  static constexpr bool turns = D_QK == D_V && !p_cols;
  // P V is issued in two halves of 64 keys: the softmax hands over the
  // first half of P before it computes the second, so that half of P V runs
  // while the softmax is still busy (it shortens each tile's chain softmax ->
  // P V -> S -> softmax by the half's tensor time).  Measured: ViT d80 +1 %;
  // d_v = 128 (ViT d128, MLA) -3 %, where the extra handover costs more.
  static constexpr bool split_pv = D_V <= 80;
  // Per-query-tile key ranges inside a work item (tile_kv_range) for the
  // MLA shapes, whose prefill is causal or windowed: sliding window (1024,
  // 0) 1287 -> 1214 us, causal 4 x 4096 2028 -> 1993 us.  The other head
  // dims run the item's whole range for both tiles: their state cost the
  // non-causal ViT and long-sequence loops 1-4 %.
  static constexpr bool tile_ranges = D_QK != D_V;
  // TMEM columns of the S/P and O regions of query tile t.
  __host__ __device__ static constexpr uint32_t s_col(int t) { return 128u * (uint32_t)t; }
  __host__ __device__ static constexpr uint32_t o_col(int t) { return 256u + 128u * (uint32_t)t; }
  // P_t (bf16 pairs, 64 columns): its own columns with p_cols, else S_t's.
  __host__ __device__ static constexpr uint32_t p_col(int t) {
    return p_cols ? o_col(t) + 64u : s_col(t);
  }
};

struct VarlenArgs {
  const int* cu_q;
  const int* cu_k;
  int batch;
  int num_heads;
  int num_heads_k;
  int total_q;
  int total_k;
  float scale_log2;  // softmax_scale * log2(e)
  int wl;            // window left, -1 = unbounded
  int wr;            // window right with causal folded in, -1 = unbounded
  uint16_t* out;     // bf16 [total_q, H, d_v]
  float* lse;        // [H, total_q] or null
  unsigned int* status;
  // Split-KV: CTAs per work item (the cluster size; 1 = no split).  With
  // split > 1 the grid holds one cluster per work item; rank r of a cluster
  // runs part r of the item's KV tiles and the cluster combines the parts
  // (split_combine).
  int split;
  // GQA head-group packing: P = 1 << pack_shift query heads that share a
  // key/value head fill one query tile together, row r of a tile being
  // token r / P and head r % P of the tile's 128 / P tokens (the Q tensor
  // maps load boxes of {64, P, 128 / P}), so that a K/V tile serves all P
  // heads at once.  0 = one head per tile.
  int pack_shift;
  uint64_t wait_limit_ns;  // pipeline wait limit (bounded waits)
};

struct VarlenMaps {
  CUtensorMap q_full, q_tail, k_full, k_tail, v_full;
  // O [total_q, H, d_v] through boxes of {d_v, 1, 128}, no swizzle: the
  // staged rows of one query tile (row r = token r) written by one store.
  CUtensorMap o_rows;
};

// Shared-memory control block (after the tiles).
struct alignas(8) VarlenBarriers {
  uint64_t q_full[4];  // [pair * 2 + tile]
  uint64_t q_free[4];
  uint64_t s_full[2];
  uint64_t p_full[2];
  uint64_t p_half[2];  // P_t(j) keys 0..63 written (split_pv)
  uint64_t o_full[2];
  uint64_t o_free[2];
  uint64_t drain;
  uint64_t turn[2];  // issuer t may issue its next group
  uint64_t s_free[2];   // p_cols: the softmax has loaded S_t(j)
  uint64_t pv_done[2];  // p_cols: P V_t(j) completed (not the tile's last)
  uint64_t k_full[8];   // K ring slot landed
  uint64_t k_free[8];   // K ring slot released (one arrival per issuer)
  uint64_t v_full[8];
  uint64_t v_free[8];
  uint32_t tmem_base;
  volatile int abort_flag;
};
static_assert(sizeof(VarlenBarriers) <= kBarrierBytes, "barrier block larger than reserved");

// Slot of the n-th tile loaded into a ring of Size slots (its fill parity is
// (n / Size) & 1).  A one-slot ring's (d_qk = 192) constant slot is hidden
// from the optimiser, which otherwise makes ptxas spill registers.
template <int Size>
__device__ __forceinline__ uint32_t ring_slot(uint32_t n) {
  uint32_t s = n % (uint32_t)Size;
  if (Size == 1) asm volatile("" : "+r"(s));
  return s;
}

// ------------------------------------------------------------ MMA groups
// The MMA issuer warps run converged, and each group of MMAs is one asm
// block in which elect.sync picks a lane and every tcgen05.mma is predicated
// on it.  The same MMAs issued from a lane-0 branch share the SM
// sub-partition's issue slots badly with the softmax warps there: measured
// on one SM with two exp2/FMA warps beside the issuer, 85 clk per MMA from
// the branch against 52 (the tensor-core rate of this group shape) this way.
// Descriptor offsets are assembly-time constant expressions.

// Block prologue: pa = accumulate, pz = overwrite, e = the elected lane.
#define FA_GROUP_BEGIN                                                  \
  "{\n\t.reg .pred e, pa, pz;\n\t.reg .b64 da, db;\n\t.reg .b32 ta;\n\t" \
  "setp.ne.b32 pa, %7, 0;\n\tsetp.eq.b32 pz, %7, 0;\n\t"                \
  "elect.sync _|e, 0xffffffff;\n\t"
// S += Q K^T for one K=16 step: both descriptors advanced by OFF (16-byte
// units).  Operands: %0 S columns, %1/%2 Q/K descriptors of the 64-wide
// chunks, %3/%4 of the tail chunk, %5 instruction descriptor, %6 the
// descriptor distance between 64-wide chunks, %7 the constant 1.
#define FA_SS(QD, KD, OFF, ACC)                                            \
  "add.s64 da, " QD ", " OFF ";\n\tadd.s64 db, " KD ", " OFF ";\n\t"       \
  "@e tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %5, " ACC ";\n\t"
// The four K=16 steps of 64-wide chunk C (128-byte swizzle: 32 bytes apart).
#define FA_SS_CHUNK(C, ACC0)                                                  \
  FA_SS("%1", "%2", "%6*" #C "+0", ACC0) FA_SS("%1", "%2", "%6*" #C "+2", "pa") \
  FA_SS("%1", "%2", "%6*" #C "+4", "pa") FA_SS("%1", "%2", "%6*" #C "+6", "pa")
#define FA_SS_TAIL(OFF) FA_SS("%3", "%4", OFF, "pa")

// S_t = Q_t K_j^T over the padded head dimension: FULL 64-wide chunks and a
// TAIL-wide (0, 16 or 32) last chunk, kBM == kBN so one offset addresses the
// same chunk of Q and K.
template <int FULL, int TAIL>
__device__ __forceinline__ void issue_s_group(uint32_t d, uint64_t qd, uint64_t kd, uint64_t qdt,
                                              uint64_t kdt, uint32_t idesc) {
  constexpr uint32_t kChunk = (uint32_t)(kBN * 128) >> 4;  // chunk distance, 16-byte units
#define FA_S_OPERANDS                                                                   \
  ::"r"(d), "l"(qd), "l"(kd), "l"(qdt), "l"(kdt), "r"(idesc), "n"(kChunk), "r"(1u) \
      : "memory"
  if constexpr (FULL == 1 && TAIL == 0) {
    asm volatile(FA_GROUP_BEGIN FA_SS_CHUNK(0, "pz") "}\n" FA_S_OPERANDS);
  } else if constexpr (FULL == 1 && TAIL == 16) {
    asm volatile(FA_GROUP_BEGIN FA_SS_CHUNK(0, "pz") FA_SS_TAIL("0") "}\n" FA_S_OPERANDS);
  } else if constexpr (FULL == 1 && TAIL == 32) {
    asm volatile(FA_GROUP_BEGIN FA_SS_CHUNK(0, "pz") FA_SS_TAIL("0") FA_SS_TAIL("2") "}\n"
                 FA_S_OPERANDS);
  } else if constexpr (FULL == 2 && TAIL == 0) {
    asm volatile(FA_GROUP_BEGIN FA_SS_CHUNK(0, "pz") FA_SS_CHUNK(1, "pa") "}\n" FA_S_OPERANDS);
  } else if constexpr (FULL == 3 && TAIL == 0) {
    asm volatile(FA_GROUP_BEGIN FA_SS_CHUNK(0, "pz") FA_SS_CHUNK(1, "pa") FA_SS_CHUNK(2, "pa")
                 "}\n" FA_S_OPERANDS);
  } else {
    static_assert(FULL < 0, "head dimension without an S issue group");
  }
#undef FA_S_OPERANDS
}

// O_t (+)= P_t V_j: eight K=16 steps over the 128 keys, P read from TMEM
// (8 columns of packed bf16 pairs per step), V descriptor advanced by %6
// (16-byte units) per step.  %4 = 0 overwrites O on the first step.
#define FA_TS(S, ACC)                                                          \
  "add.u32 ta, %1, 8*" S ";\n\tadd.s64 db, %2, %6*" S ";\n\t"                  \
  "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [ta], db, %3, " ACC ";\n\t"
template <uint32_t kStepDesc>
__device__ __forceinline__ void issue_pv_group(uint32_t o, uint32_t p, uint64_t vd, uint32_t idesc,
                                               uint32_t acc_first) {
  static_assert(kBN == 128, "eight K=16 steps per KV tile");
  asm volatile(
      "{\n\t.reg .pred e, pa, p0;\n\t.reg .b64 db;\n\t.reg .b32 ta;\n\t"
      "setp.ne.b32 pa, %5, 0;\n\tsetp.ne.b32 p0, %4, 0;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      FA_TS("0", "p0") FA_TS("1", "pa") FA_TS("2", "pa") FA_TS("3", "pa")
      FA_TS("4", "pa") FA_TS("5", "pa") FA_TS("6", "pa") FA_TS("7", "pa") "}\n"
      ::"r"(o), "r"(p), "l"(vd), "r"(idesc), "r"(acc_first), "r"(1u), "n"(kStepDesc)
      : "memory");
}
// Half of it: the four K=16 steps over keys [64 h, 64 h + 64) (P columns
// 32 h .. 32 h + 32, V rows 64 h ..).
template <uint32_t kStepDesc>
__device__ __forceinline__ void issue_pv_half(uint32_t o, uint32_t p, uint64_t vd, uint32_t idesc,
                                              uint32_t acc_first, int h) {
  const uint32_t ph = p + (uint32_t)(h * 32);
  const uint64_t vh = vd + (uint64_t)(h * 4 * kStepDesc);
  asm volatile(
      "{\n\t.reg .pred e, pa, p0;\n\t.reg .b64 db;\n\t.reg .b32 ta;\n\t"
      "setp.ne.b32 pa, %5, 0;\n\tsetp.ne.b32 p0, %4, 0;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      FA_TS("0", "p0") FA_TS("1", "pa") FA_TS("2", "pa") FA_TS("3", "pa") "}\n"
      ::"r"(o), "r"(ph), "l"(vh), "r"(idesc), "r"(acc_first), "r"(1u), "n"(kStepDesc)
      : "memory");
}
#undef FA_TS
#undef FA_SS_TAIL
#undef FA_SS_CHUNK
#undef FA_SS
#undef FA_GROUP_BEGIN

// Work items are sorted longest first and dealt to the CTAs in rounds of
// gridDim.x, the direction reversed every other round, so that the CTAs that
// take the longest item of one round take the shortest of the next.  For the
// packed ViT mix (6 images, 256 to 9216 tokens, 16 heads) the busiest CTA then
// carries 1.04x the mean work instead of 1.07x with a plain round robin;
// causal 4 x 4096: 1.01x instead of 1.14x.
__device__ __forceinline__ int snake_item(int round, int split) {
  if (split > 1) return round == 0 ? (int)blockIdx.x / split : 0x7fffffff;  // one item per cluster
  const int g = (int)gridDim.x, b = (int)blockIdx.x;
  return round * g + ((round & 1) ? g - 1 - b : b);
}

struct WorkItem {
  int q_start, k_start, lq, lk, head, kv_head, row0, n_qt, tile_lo, n_kv;
  int b0, nb;  // first sequence of the unit and how many (nb > 1: a pack)
};
// Row r of a work item (0 .. 255) is token row0 + (r >> pack_shift) of the
// sequence and query head head + r % P.
static_assert(sizeof(WorkItem) == 48, "work item slot size");

// Decoded work items, published by the producer (which runs ahead of the
// other roles) into a ring in shared memory: decoding an item (a search of
// the work list, reads of cu_seqlens, integer divisions) costs about 1000
// cycles, which the MMA issuers and softmax warps would otherwise spend at
// every item boundary.  Lives in the work-list scan's scratch (s_part), dead
// once the list is built.
constexpr int kItemSlots = 4;
constexpr int kItemReaders = 2 + 8;  // the issuer warps and the softmax warps
struct ItemRing {
  WorkItem slot[kItemSlots];
  uint64_t full[kItemSlots];
  uint64_t free_[kItemSlots];
};
static_assert(sizeof(ItemRing) <= 4 * kVarlenThreads, "item ring fits the scan scratch");

// Short segments: consecutive sequences of 1..kPackMaxLen query rows with as
// many keys and the same token offsets in Q and K (self-attention over one
// packed tensor, as in windowed ViT attention), whose first tokens fall in
// the same kPackBlock-token block, form one work unit, a pack of at most
// kPackBlock + kPackMaxLen rows.  Its query tiles run against its own key
// tiles under a block-diagonal mask: each row sees only its own segment
// (and the window inside it).  A 64-token window alone fills a quarter of a
// 128 x 128 score tile; packed, up to four share two query tiles and two
// key tiles.
constexpr int kPackMaxLen = 64;
constexpr int kPackBlock = kRowsPerItem - kPackMaxLen;  // 192
// A unit in the sorted list: first sequence | number of sequences << 16.
constexpr int kUnitShift = 16;
static_assert(kMaxBatch < (1 << kUnitShift), "unit encoding");

// ------------------------------------------------------------ bounded waits
// Time limit of the pipeline barrier waits, passed per launch (default
// kWaitLimitNs; fa_set_wait_limit_ns changes it).  Normal waits are
// microseconds; hitting the limit means the pipeline is broken.  The kernel
// then records kStatusTimeout, raises the CTA abort flag and unwinds instead
// of hanging.  Waits read the clock every 256 probes, or on every probe
// under limits below kShortWaitNs (a test setting, see test_load_delay).
constexpr uint64_t kWaitLimitNs = 4000000000ull;
constexpr uint64_t kShortWaitNs = 1000000ull;
// Limit of the unwind's own waits (for the copies and MMAs a CTA started),
// which do not give up on the abort flag.
constexpr uint64_t kDrainLimitNs = 4000000000ull;

__device__ __forceinline__ bool wait_single(uint32_t bar, uint32_t parity,
                                            volatile int* abort_flag, unsigned int* status,
                                            uint64_t limit_ns) {
  if (ptx::mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = ptx::globaltimer_ns();
  for (uint32_t spin = 1;; ++spin) {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    if ((spin & 255u) == 0 || limit_ns < kShortWaitNs) {
      if (*abort_flag) return false;
      if (ptx::globaltimer_ns() - t0 > limit_ns) {
        atomicOr(status, kStatusTimeout);
        *abort_flag = 1;
        return false;
      }
    }
  }
}

// Warp-uniform variant: every lane of the warp gets the same answer, so the
// warp stays converged for the warp-collective tcgen05 loads and stores.
__device__ __forceinline__ bool wait_warp(uint32_t bar, uint32_t parity,
                                          volatile int* abort_flag, unsigned int* status,
                                          uint64_t limit_ns) {
  const unsigned full = 0xffffffffu;
  if (__all_sync(full, ptx::mbar_try_wait(bar, parity))) return true;
  const uint64_t t0 = ptx::globaltimer_ns();
  for (uint32_t spin = 1;; ++spin) {
    if (__all_sync(full, ptx::mbar_try_wait(bar, parity))) return true;
    if ((spin & 255u) == 0 || limit_ns < kShortWaitNs) {
      int give_up = 0;
      if ((threadIdx.x & 31) == 0) {
        if (*abort_flag) {
          give_up = 1;
        } else if (ptx::globaltimer_ns() - t0 > limit_ns) {
          atomicOr(status, kStatusTimeout);
          *abort_flag = 1;
          give_up = 1;
        }
      }
      if (__shfl_sync(full, give_up, 0)) return false;
    }
  }
}

// Under a test limit (below kShortWaitNs) the loaders pause this long before
// their first copy, so that the first waits for their data outlast any
// suspension inside try_wait and run out; bounded like every wait.
constexpr uint64_t kTestLoadDelayNs = 50000000ull;
__device__ __forceinline__ void test_load_delay(uint64_t limit_ns) {
  if (limit_ns >= kShortWaitNs) return;
  const uint64_t t0 = ptx::globaltimer_ns();
  while (ptx::globaltimer_ns() - t0 < kTestLoadDelayNs) __nanosleep(10000);
}

// The unwind's waits: for copies and MMAs this CTA started, which complete
// whatever the rest of the pipeline does, so they ignore the abort flag;
// bounded all the same.
__device__ __forceinline__ bool wait_drain_single(uint32_t bar, uint32_t parity,
                                                  unsigned int* status) {
  if (ptx::mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = ptx::globaltimer_ns();
  for (uint32_t spin = 1;; ++spin) {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    if ((spin & 255u) == 0 && ptx::globaltimer_ns() - t0 > kDrainLimitNs) {
      atomicOr(status, kStatusTimeout);
      return false;
    }
  }
}
__device__ __forceinline__ bool wait_drain_warp(uint32_t bar, uint32_t parity,
                                                unsigned int* status) {
  const unsigned full = 0xffffffffu;
  if (__all_sync(full, ptx::mbar_try_wait(bar, parity))) return true;
  const uint64_t t0 = ptx::globaltimer_ns();
  for (uint32_t spin = 1;; ++spin) {
    if (__all_sync(full, ptx::mbar_try_wait(bar, parity))) return true;
    if ((spin & 255u) == 0) {
      int give_up = 0;
      if ((threadIdx.x & 31) == 0 && ptx::globaltimer_ns() - t0 > kDrainLimitNs) {
        atomicOr(status, kStatusTimeout);
        give_up = 1;
      }
      if (__shfl_sync(full, give_up, 0)) return false;
    }
  }
}

// ------------------------------------------------------------ work list
// Builds, in shared memory, the work units (sequences, or packs of short
// segments) sorted by key length (longest first, ties by index) and the
// prefix sum of their work-item counts.
// s_tmp: 5 * kMaxBatch ints of scratch (the K ring, empty until the producer
// starts), so that nothing is held in registers across the barriers.  Kept
// out of line: it runs once per CTA, and inlined it changed the register
// allocation of the pipeline loops (ViT d80 1.5 % slower).
// (The kernel arguments it needs come by value: a reference would make the
// compiler copy the whole argument block to local memory for the call.)
// Sequence b's token range [lo, hi) in a tensor of `total` tokens: the
// cu_seqlens entries clamped to [0, total] and hi to at least lo, so that a
// malformed array (decreasing, or reaching past the tensor) gives empty or
// shortened sequences and no access outside the tensors.
__device__ __forceinline__ int seq_lo(const int* cu, int b, int total) {
  return min(max(__ldg(cu + b), 0), total);
}
__device__ __forceinline__ int seq_hi(const int* cu, int b, int total) {
  return min(max(__ldg(cu + b + 1), seq_lo(cu, b, total)), total);
}

static __device__ __noinline__ void build_work_list(const int* cu_q, const int* cu_k, int B,
                                                    int total_q, int total_k,
                                                    int num_heads, int pack_shift, int* s_prefix,
                                                    int* s_sorted, int* s_part, int* s_tmp) {
  const int tid = threadIdx.x;
  int* t_lq = s_tmp;                 // query rows of sequence b
  int* t_key = s_tmp + kMaxBatch;    // sort key of the unit starting at b, -1 for members
  int* t_unit = s_tmp + 2 * kMaxBatch;  // nb of the unit starting at b (0 for members)
  uint64_t* t_sort = reinterpret_cast<uint64_t*>(s_tmp + 3 * kMaxBatch);  // sort keys
  // 1. The only global reads: s_prefix[b] = the kPackBlock-token block of a
  //    packable sequence's first token (-1 for any other sequence),
  //    s_sorted[b] = its key count.
  for (int b = tid; b < B; b += kVarlenThreads) {
    const int q0 = seq_lo(cu_q, b, total_q), k0 = seq_lo(cu_k, b, total_k);
    const int lq = seq_hi(cu_q, b, total_q) - q0, lk = seq_hi(cu_k, b, total_k) - k0;
    const bool pack = pack_shift == 0 && lq >= 1 && lq <= kPackMaxLen && lk == lq && k0 == q0;
    s_prefix[b] = pack ? q0 / kPackBlock : -1;
    s_sorted[b] = lk;
    t_lq[b] = lq;
  }
  __syncthreads();
  // 2. Units: a sequence starts one unless it continues its predecessor's
  //    pack.  Sort key = key rows; the item count (head groups x pairs of
  //    query tiles) goes where the sequence's key count was.
  const int tokens_per_item = kRowsPerItem >> pack_shift;
  for (int b = tid; b < B; b += kVarlenThreads) {
    const int blk = s_prefix[b];
    int nb = 0, key = -1;
    if (!(blk >= 0 && b > 0 && s_prefix[b - 1] == blk)) {
      nb = 1;
      key = s_sorted[b];
      if (blk >= 0)  // a pack: its members have as many query rows as keys
        for (; b + nb < B && s_prefix[b + nb] == blk; ++nb) key += s_sorted[b + nb];
      const int rows_q = blk >= 0 ? key : t_lq[b];
      t_lq[b] = (num_heads >> pack_shift) *
                ((max(rows_q, 0) + tokens_per_item - 1) >> (8 - pack_shift));
    } else {
      t_lq[b] = 0;
    }
    t_key[b] = key;
    t_unit[b] = nb;
  }
  __syncthreads();
  // 3. Longest first: the entries sorted by key, descending (ties in
  //    sequence order, members last), with a bitonic network over N = B
  //    rounded up to a power of two (padding entries sort after everything);
  //    then s_sorted[rank] = b | nb << kUnitShift and s_prefix[rank] = its
  //    item count.  Every CTA sorts the same keys the same way, so all agree
  //    on the order.
  int n_sort = 1;
  while (n_sort < B) n_sort <<= 1;
  for (int b = tid; b < n_sort; b += kVarlenThreads)
    t_sort[b] = b < B ? ((uint64_t)(uint32_t)(t_key[b] + 1) << 32) | (uint32_t)(0xffffffffu - b)
                      : 0ull;
  __syncthreads();
  for (int k = 2; k <= n_sort; k <<= 1) {
    for (int j = k >> 1; j > 0; j >>= 1) {
      for (int i = tid; i < n_sort / 2; i += kVarlenThreads) {
        const int lo = 2 * i - (i & (j - 1));  // the i-th pair (lo, lo + j)
        const uint64_t x = t_sort[lo], y = t_sort[lo + j];
        // Blocks of k entries alternate direction; the last merge is
        // descending.
        if (((lo & k) == 0) == (x < y)) {
          t_sort[lo] = y;
          t_sort[lo + j] = x;
        }
      }
      __syncthreads();
    }
  }
  for (int r = tid; r < B; r += kVarlenThreads) {
    const int b = (int)(0xffffffffu - (uint32_t)t_sort[r]);
    s_sorted[r] = b | (t_unit[b] << kUnitShift);
    s_prefix[r] = t_lq[b];
  }
  __syncthreads();
  // Block-wide exclusive scan of per-unit item counts in sorted order.
  const int per = (B + kVarlenThreads - 1) / kVarlenThreads;
  const int beg = tid * per;
  const int end = min(B, beg + per);
  int local = 0;
  for (int p = beg; p < end; ++p) local += s_prefix[p];
  s_part[tid] = local;
  __syncthreads();
  if (tid < 32) {
    // Warp 0 scans the kVarlenThreads partial sums, kPer per lane.
    constexpr int kPer = (kVarlenThreads + 31) / 32;
    int vals[kPer];
    int run = 0;
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
      const int idx = tid * kPer + i;
      vals[i] = idx < kVarlenThreads ? s_part[idx] : 0;
      run += vals[i];
    }
    int incl = run;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int n = __shfl_up_sync(0xffffffffu, incl, o);
      if (tid >= o) incl += n;
    }
    int excl = incl - run;
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
      const int idx = tid * kPer + i;
      if (idx < kVarlenThreads) s_part[idx] = excl;
      excl += vals[i];
    }
  }
  __syncthreads();
  int run = s_part[tid];
  for (int p = beg; p < end; ++p) {
    const int n = s_prefix[p];  // item count in, exclusive prefix out
    s_prefix[p] = run;
    run += n;
  }
  if (end == B && beg < end) s_prefix[B] = run;  // the thread owning the last chunk
  // The scratch in s_tmp is overwritten next by TMA (async proxy).
  ptx::fence_proxy_async_smem();
  __syncthreads();
}

__device__ __forceinline__ WorkItem decode_item(int it, const VarlenArgs& a,
                                                const int* s_prefix, const int* s_sorted,
                                                int split, int pack_shift) {
  // Largest sorted position p with prefix[p] <= it (skips empty sequences).
  int lo = 0, hi = a.batch - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (s_prefix[mid] <= it) lo = mid; else hi = mid - 1;
  }
  const int unit = s_sorted[lo];
  const int r = it - s_prefix[lo];
  WorkItem w;
  w.b0 = unit & ((1 << kUnitShift) - 1);
  w.nb = unit >> kUnitShift;
  // Read through the read-only data cache: every role decodes every item,
  // and these few words stay cached there.
  // (A pack's members are consecutive and contiguous, so its range runs
  // from its first member's start to its last member's end.)
  w.q_start = seq_lo(a.cu_q, w.b0, a.total_q);
  w.k_start = seq_lo(a.cu_k, w.b0, a.total_k);
  w.lq = seq_hi(a.cu_q, w.b0 + w.nb - 1, a.total_q) - w.q_start;
  w.lk = seq_hi(a.cu_k, w.b0 + w.nb - 1, a.total_k) - w.k_start;
  // An item covers 256 / P tokens of the sequence (1 << tshift) and P heads.
  static_assert(kRowsPerItem == 256, "tokens per item are 256 >> pack_shift");
  const int tshift = 8 - pack_shift;
  const int pairs = (w.lq + (1 << tshift) - 1) >> tshift;
  const int group = r / pairs;
  w.head = group << pack_shift;  // first query head of the item
  const int pair = pairs - 1 - (r - group * pairs);  // later rows first
  w.kv_head = w.head / (a.num_heads / a.num_heads_k);
  w.row0 = pair << tshift;  // first token of the item in the sequence
  const int row_end = min(w.lq, w.row0 + (1 << tshift));
  w.n_qt = (((row_end - w.row0) << pack_shift) + kBM - 1) / kBM;
  const int off = w.lk - w.lq;
  const int key_lo = a.wl >= 0 ? max(0, w.row0 + off - a.wl) : 0;
  const int key_hi = a.wr >= 0 ? min(w.lk, row_end + off + a.wr) : w.lk;
  if (key_hi <= key_lo) {
    w.tile_lo = 0;
    w.n_kv = 0;
  } else {
    w.tile_lo = key_lo / kBN;
    w.n_kv = (key_hi + kBN - 1) / kBN - w.tile_lo;
  }
  if (split > 1) {
    // Split-KV: this CTA's part of the item's KV tiles (its rank in the
    // cluster; parts differ in size by at most one tile, and may be empty).
    const int part = (int)blockIdx.x % split;
    const int p0 = w.n_kv * part / split;
    const int p1 = w.n_kv * (part + 1) / split;
    w.tile_lo += p0;
    w.n_kv = p1 - p0;
  }
  return w;
}

// Key tiles [jlo, jhi) of a work item (relative to its tile_lo) that query
// tile t of the item can see: the causal and window bounds of the tile's
// first and last rows.  The two query tiles of an item share its KV tiles
// but not all of them (a causal tile 0 cannot see the diagonal tile of
// tile 1; under a sliding window tile 1 cannot see the first tile of tile
// 0); the issuer of tile t and its softmax warpgroup both walk exactly these
// tiles.  Packs of short segments keep the item's whole range.
__device__ __forceinline__ void tile_kv_range(const WorkItem& w, int t, int wl, int wr,
                                              int pack_shift, int& jlo, int& jhi) {
  jlo = 0;
  jhi = w.n_kv;
  if (w.nb > 1 || w.n_kv == 0) return;
  const int off = w.lk - w.lq;
  const int r0 = w.row0 + ((t * kBM) >> pack_shift);                        // first token
  const int r1 = min(w.lq, w.row0 + (((t + 1) * kBM) >> pack_shift)) - 1;   // last token
  if (wl >= 0) jlo = max(0, max(0, r0 + off - wl) / kBN - w.tile_lo);
  if (wr >= 0) {
    const int khi = min(w.lk, r1 + off + wr + 1);  // keys < khi
    jhi = khi <= 0 ? 0 : min(w.n_kv, (khi + kBN - 1) / kBN - w.tile_lo);
  }
  if (jhi < jlo) jhi = jlo;
}

// ------------------------------------------------------------ split-KV combine
// Split-KV partials in shared memory, in the Q tiles and K/V rings of the
// item's CTAs (dead once the item's last MMA is done): row r of the item's
// 256 rows holds its unnormalised O (d_v fp32; 16 bytes of padding put the
// rows of a warp in different banks), then every row's (m, l) with m the
// running maximum in scaled log2 units, then the combining CTA's per-row
// weights of the parts.
constexpr int kMaxSplit = 16;
template <int D_V>
struct SplitStash {
  static constexpr int kRowBytes = D_V * 4 + 16;
  static constexpr int kMlOff = kRowsPerItem * kRowBytes;
  static constexpr int kWOff = kMlOff + kRowsPerItem * 8;
  static constexpr int kBytes = kWOff + kRowsPerItem * kMaxSplit * 4;
};

// The combine of one work item's parts, run by every thread of each CTA of
// the item's cluster once all of them have left their pipelines.  Rank r of
// S combines rows [r n / S, (r + 1) n / S) of the item's n rows, reading every
// part's row through distributed shared memory, in rank order:
//   M = max_s m_s,  w_s = 2^(m_s - M),  L = sum_s w_s l_s,
//   O = sum_s (w_s / L) O_s,  LSE = ln 2 (M + log2 L)
// (the LSE-weighted merge of split-KV partials of the vLLM flash_attn page,
// FA4SplitKVCombineKernel).  A row with no key in any part gets O = 0 and
// LSE = -inf.
template <int D_V>
static __device__ __noinline__ void split_combine(const VarlenArgs args, uint8_t* smem,
                                                  const int* s_prefix, const int* s_sorted,
                                                  int total_items) {
  using St = SplitStash<D_V>;
  const int S = args.split;
  const int rank = (int)blockIdx.x % S;
  const int it = (int)blockIdx.x / S;
  ptx::cluster_arrive_release();
  ptx::cluster_wait_acquire();  // every part is in its CTA's shared memory
  if (it < total_items) {
    const WorkItem w = decode_item(it, args, s_prefix, s_sorted, S, args.pack_shift);
    const int rows = min(kRowsPerItem, (w.lq - w.row0) << args.pack_shift);
    const int pmask = (1 << args.pack_shift) - 1;
    const int r_lo = rows * rank / S, r_hi = rows * (rank + 1) / S;
    const uint32_t base = ptx::smem_u32(smem);
    float* wgt = reinterpret_cast<float*>(smem + St::kWOff);
    const float neg_inf = -__int_as_float(0x7f800000);
    for (int r = r_lo + (int)threadIdx.x; r < r_hi; r += (int)blockDim.x) {
      float* wr = wgt + (r - r_lo) * kMaxSplit;
      float M = neg_inf;
      for (int sp = 0; sp < S; ++sp) {
        const float2 ml = ptx::ld_shared_cluster_v2(ptx::mapa_shared(base + St::kMlOff + r * 8, sp));
        wr[sp] = ml.y > 0.f ? ml.x : neg_inf;  // parts with no key of this row: weight 0
        M = fmaxf(M, wr[sp]);
      }
      float L = 0.f;
      for (int sp = 0; sp < S; ++sp) {
        const float2 ml = ptx::ld_shared_cluster_v2(ptx::mapa_shared(base + St::kMlOff + r * 8, sp));
        const float e = wr[sp] == neg_inf ? 0.f : ptx::ex2(wr[sp] - M);
        wr[sp] = e;
        L += e * ml.y;
      }
      const float inv = L > 0.f ? 1.f / L : 0.f;
      for (int sp = 0; sp < S; ++sp) wr[sp] *= inv;
      if (args.lse) {
        const size_t tok = (size_t)(w.q_start + w.row0 + (r >> args.pack_shift));
        args.lse[(size_t)(w.head + (r & pmask)) * args.total_q + tok] =
            L > 0.f ? (M + __log2f(L)) * 0.69314718055994531f : neg_inf;
      }
    }
    __syncthreads();
    constexpr int kGroups = D_V / 8;  // 8 output columns (16 bytes of bf16) per unit
    const int units = (r_hi - r_lo) * kGroups;
    for (int u = (int)threadIdx.x; u < units; u += (int)blockDim.x) {
      const int rr = u / kGroups, g = u - rr * kGroups;
      const int r = r_lo + rr;
      const float* wr = wgt + rr * kMaxSplit;
      float acc[8];
#pragma unroll
      for (int c = 0; c < 8; ++c) acc[c] = 0.f;
      for (int sp = 0; sp < S; ++sp) {
        const float ws = wr[sp];
        if (ws == 0.f) continue;
        const uint32_t a = ptx::mapa_shared(base + r * St::kRowBytes + g * 32, sp);
        const float4 v0 = ptx::ld_shared_cluster_v4(a);
        const float4 v1 = ptx::ld_shared_cluster_v4(a + 16);
        acc[0] += ws * v0.x; acc[1] += ws * v0.y; acc[2] += ws * v0.z; acc[3] += ws * v0.w;
        acc[4] += ws * v1.x; acc[5] += ws * v1.y; acc[6] += ws * v1.z; acc[7] += ws * v1.w;
      }
      const size_t tok = (size_t)(w.q_start + w.row0 + (r >> args.pack_shift));
      const int head = w.head + (r & pmask);
      uint4 pk;
      pk.x = ptx::pack_bf16x2(acc[0], acc[1]);
      pk.y = ptx::pack_bf16x2(acc[2], acc[3]);
      pk.z = ptx::pack_bf16x2(acc[4], acc[5]);
      pk.w = ptx::pack_bf16x2(acc[6], acc[7]);
      *reinterpret_cast<uint4*>(args.out + (tok * args.num_heads + head) * (size_t)D_V + 8 * g) = pk;
    }
  }
  __syncwarp();
  ptx::cluster_arrive_release();
  ptx::cluster_wait_acquire();  // no CTA leaves while another still reads its shared memory
}

// ------------------------------------------------------------ the kernel
// kGeneral selects the instantiation that runs split-KV (args.split > 1,
// launched in clusters of args.split CTAs) and GQA head-group packing
// (args.pack_shift > 0); the other one compiles with neither (split 1,
// one head per tile as constants): their extra state would otherwise cost
// the pipeline loops registers.
template <int D_QK, int D_V, bool kGeneral>
__global__ void __launch_bounds__(kVarlenThreads, 1)
    varlen_fwd_kernel(const __grid_constant__ VarlenMaps maps, const VarlenArgs args) {
  using C = VarlenCfg<D_QK, D_V>;
  const int split = kGeneral ? args.split : 1;
  const int pshift = kGeneral ? args.pack_shift : 0;
  using QK = typename C::QK;
  using VD = typename C::VD;
  constexpr int NK = C::nk, NV = C::nv;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  // Q tile t of buffer pair p at smem + (2p + t) * q_tile_bytes.
  uint8_t* const q_base = smem;
  uint8_t* k_ring = smem + 2 * C::q_pairs * C::q_tile_bytes;
  uint8_t* v_ring = k_ring + NK * C::k_slot_bytes;
  VarlenBarriers* cb = reinterpret_cast<VarlenBarriers*>(v_ring + NV * C::v_slot_bytes);
  // The scan scratch first (a fixed offset from the shared-memory base: the
  // decoded-item ring lives there once the list is built), then the list.
  int* s_part = reinterpret_cast<int*>(cb + 1);
  int* s_prefix = s_part + kVarlenThreads;
  int* s_sorted = s_prefix + (args.batch + 1);
  volatile int* abort_flag = &cb->abort_flag;

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;

  if (tid == 0) {
    for (int q = 0; q < 4; ++q) {
      ptx::mbar_init(ptx::smem_u32(&cb->q_full[q]), 1);
      ptx::mbar_init(ptx::smem_u32(&cb->q_free[q]), C::stage_o ? kBM : 1);
    }
    for (int t = 0; t < 2; ++t) {
      ptx::mbar_init(ptx::smem_u32(&cb->s_full[t]), 1);
      ptx::mbar_init(ptx::smem_u32(&cb->p_full[t]), kBM);
      ptx::mbar_init(ptx::smem_u32(&cb->p_half[t]), kBM);
      ptx::mbar_init(ptx::smem_u32(&cb->o_full[t]), 1);
      ptx::mbar_init(ptx::smem_u32(&cb->o_free[t]), kBM);
      ptx::mbar_init(ptx::smem_u32(&cb->s_free[t]), kBM);
      ptx::mbar_init(ptx::smem_u32(&cb->pv_done[t]), 1);
    }
    ptx::mbar_init(ptx::smem_u32(&cb->drain), 2);
    ptx::mbar_init(ptx::smem_u32(&cb->turn[0]), 1);
    ptx::mbar_init(ptx::smem_u32(&cb->turn[1]), 1);
    for (int s = 0; s < NK; ++s) {
      ptx::mbar_init(ptx::smem_u32(&cb->k_full[s]), 1);
      ptx::mbar_init(ptx::smem_u32(&cb->k_free[s]), 2);  // one release per issuer
    }
    for (int s = 0; s < NV; ++s) {
      ptx::mbar_init(ptx::smem_u32(&cb->v_full[s]), 1);
      ptx::mbar_init(ptx::smem_u32(&cb->v_free[s]), 2);
    }
    cb->abort_flag = 0;
    ptx::fence_mbar_init();
  }
  if (warp == kProducerWarp && lane == 0) {
    ptx::prefetch_tmap(&maps.q_full);
    ptx::prefetch_tmap(&maps.k_full);
    ptx::prefetch_tmap(&maps.v_full);
    if (QK::tail) {
      ptx::prefetch_tmap(&maps.q_tail);
      ptx::prefetch_tmap(&maps.k_tail);
    }
  }
  if (warp == kMmaWarp) {
    ptx::tmem_alloc(ptx::smem_u32(&cb->tmem_base), 512);
    ptx::tmem_relinquish();
  }
  static_assert(NK * C::k_slot_bytes >= 5 * kMaxBatch * (int)sizeof(int),
                "the K ring holds the work-list scratch");
  static_assert(SplitStash<D_V>::kBytes <= 2 * C::q_pairs * C::q_tile_bytes +
                                               NK * C::k_slot_bytes + NV * C::v_slot_bytes,
                "the split-KV partials fit in the Q tiles and K/V rings");
  build_work_list(args.cu_q, args.cu_k, args.batch, args.total_q, args.total_k, args.num_heads,
                  pshift, s_prefix, s_sorted, s_part,
                  reinterpret_cast<int*>(k_ring));  // ends with __syncthreads
  if (tid == 0) {
    // The decoded-item ring, in the scan scratch the list builder is done with.
    ItemRing* rg = reinterpret_cast<ItemRing*>(s_part);
    for (int sl = 0; sl < kItemSlots; ++sl) {
      ptx::mbar_init(ptx::smem_u32(&rg->full[sl]), 1);
      ptx::mbar_init(ptx::smem_u32(&rg->free_[sl]), kItemReaders);
    }
    ptx::fence_mbar_init();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = cb->tmem_base;
  const int total_items = s_prefix[args.batch];
  ItemRing* const ring = reinterpret_cast<ItemRing*>(s_part);

  if (warp >= 8) {
    ptx::regs_dec<kControlRegs>();
    if (warp == kProducerWarp) {
      // ---------------------------------------------------------- producer
      if (lane == 0) {
        test_load_delay(args.wait_limit_ns);
        // Per Q buffer b = 2 * pair + tile, bit b: parity of the q_free
        // phases consumed, of the Q loads issued, and whether any was issued.
        uint32_t qf_par = 0, qi_par = 0, qi_any = 0;
        uint32_t item_n = 0;  // items with KV tiles so far (selects the pair)
        // Tiles loaded into each ring so far: tile n goes to slot n % size,
        // fill parity (n / size) & 1.
        uint32_t kn = 0, vn = 0;
        bool ok = true;
        for (int r = 0; r * (int)gridDim.x < total_items && ok; ++r) {
          const int it = snake_item(r, split);
          if (it >= total_items) continue;
          const WorkItem w = decode_item(it, args, s_prefix, s_sorted, split, pshift);
          {
            // Publish the item (every one, empty or not: all roles walk the
            // same sequence).
            // Item of round r (only the last round can be without one, so r
            // counts the items of every role).
            const uint32_t sl = (uint32_t)r % kItemSlots;
            ok = wait_single(ptx::smem_u32(&ring->free_[sl]), (((uint32_t)r / kItemSlots) & 1) ^ 1,
                             abort_flag, args.status, args.wait_limit_ns);
            if (!ok) break;
            ring->slot[sl] = w;
            ptx::mbar_arrive(ptx::smem_u32(&ring->full[sl]));
          }
          if (w.n_kv == 0) continue;
          if (C::item_prefetch) {
            // One Q buffer pair: this item's Q and first K/V tiles load only
            // once the previous item's last S is done.  Fetch them into L2
            // while that item finishes, so that those loads come from there.
            for (int t = 0; t < w.n_qt; ++t) {
              const int row = w.q_start + w.row0 + t * (kBM >> pshift);
#pragma unroll
              for (int c = 0; c < QK::chunks; ++c)
                ptx::tma_prefetch_l2_3d(c < QK::full ? &maps.q_full : &maps.q_tail, c * 64,
                                        w.head, row);
            }
            const int krow = w.k_start + w.tile_lo * kBN;
#pragma unroll
            for (int c = 0; c < QK::chunks; ++c)
              ptx::tma_prefetch_l2_3d(c < QK::full ? &maps.k_full : &maps.k_tail, c * 64,
                                      w.kv_head, krow);
#pragma unroll
            for (int c = 0; c < C::v_atoms; ++c)
              ptx::tma_prefetch_l2_3d(&maps.v_full, c * C::v_atom, w.kv_head, krow);
          }
          const int pair = C::q_pairs == 2 ? (int)(item_n & 1) : 0;
          ++item_n;
          for (int t = 0; t < w.n_qt && ok; ++t) {
            const int b = 2 * pair + t;
            ok = wait_single(ptx::smem_u32(&cb->q_free[b]), ((qf_par >> b) & 1) ^ 1, abort_flag,
                             args.status, args.wait_limit_ns);
            qf_par ^= 1u << b;
            if (!ok) break;
            const uint32_t bar = ptx::smem_u32(&cb->q_full[b]);
            ptx::mbar_arrive_expect_tx(bar, C::q_tile_bytes);
            qi_par ^= 1u << b;
            qi_any |= 1u << b;
            const int row = w.q_start + w.row0 + t * (kBM >> pshift);
            uint8_t* qdst = q_base + b * C::q_tile_bytes;
#pragma unroll
            for (int c = 0; c < QK::chunks; ++c)
              ptx::tma_load_3d(ptx::smem_u32(qdst + QK::chunk_off(c, kBM)),
                               c < QK::full ? &maps.q_full : &maps.q_tail, bar, c * 64, w.head,
                               row);
          }
          for (int j = 0; j < w.n_kv && ok; ++j) {
            const int krow = w.k_start + (w.tile_lo + j) * kBN;
            // K_j into the K ring.
            const uint32_t ks = ring_slot<NK>(kn);
            ok = wait_single(ptx::smem_u32(&cb->k_free[ks]), ((kn / NK) & 1) ^ 1, abort_flag,
                             args.status, args.wait_limit_ns);
            if (!ok) break;
            {
              const uint32_t bar = ptx::smem_u32(&cb->k_full[ks]);
              uint8_t* dst = k_ring + ks * C::k_slot_bytes;
              ptx::mbar_arrive_expect_tx(bar, C::k_tile_bytes);
#pragma unroll
              for (int c = 0; c < QK::chunks; ++c)
                ptx::tma_load_3d(ptx::smem_u32(dst + QK::chunk_off(c, kBN)),
                                 c < QK::full ? &maps.k_full : &maps.k_tail, bar, c * 64,
                                 w.kv_head, krow);
              // With one K slot, K_{j+1} can only start loading once both
              // tiles' S_j are done, and the MMAs wait for it: fetch it into
              // L2 now, so that its load then comes from there.
              if (C::k_prefetch && j + 1 < w.n_kv) {
#pragma unroll
                for (int c = 0; c < QK::chunks; ++c)
                  ptx::tma_prefetch_l2_3d(c < QK::full ? &maps.k_full : &maps.k_tail, c * 64,
                                          w.kv_head, krow + kBN);
              }
              ++kn;
            }
            if (kGeneral && split > 1 && j + 1 < w.n_kv) {
              const int prow = krow + kBN;
#pragma unroll
              for (int c = 0; c < QK::chunks; ++c)
                ptx::tma_prefetch_l2_3d(c < QK::full ? &maps.k_full : &maps.k_tail, c * 64,
                                        w.kv_head, prow);
#pragma unroll
              for (int c = 0; c < C::v_atoms; ++c)
                ptx::tma_prefetch_l2_3d(&maps.v_full, c * C::v_atom, w.kv_head, prow);
            }
            // V_j into the V ring.
            const uint32_t vs = ring_slot<NV>(vn);
            ok = wait_single(ptx::smem_u32(&cb->v_free[vs]), ((vn / NV) & 1) ^ 1, abort_flag,
                             args.status, args.wait_limit_ns);
            if (!ok) break;
            {
              const uint32_t bar = ptx::smem_u32(&cb->v_full[vs]);
              uint8_t* dst = v_ring + vs * C::v_slot_bytes;
              ptx::mbar_arrive_expect_tx(bar, C::v_tile_bytes);
#pragma unroll
              for (int c = 0; c < C::v_atoms; ++c)
                ptx::tma_load_3d(ptx::smem_u32(dst + c * C::v_atom_bytes), &maps.v_full, bar,
                                 c * C::v_atom, w.kv_head, krow);
              ++vn;
            }
          }
        }
        if (!ok) {
          // Let every copy this thread started land before the CTA exits.
          for (int b = 0; b < 4; ++b)
            if ((qi_any >> b) & 1)
              wait_drain_single(ptx::smem_u32(&cb->q_full[b]), ((qi_par >> b) & 1) ^ 1,
                                args.status);
          // Slot s was last filled by tile s + size * ((n - 1 - s) / size).
          for (uint32_t s = 0; s < (uint32_t)NK && s < kn; ++s)
            wait_drain_single(ptx::smem_u32(&cb->k_full[s]), ((kn - 1 - s) / NK) & 1,
                              args.status);
          for (uint32_t s = 0; s < (uint32_t)NV && s < vn; ++s)
            wait_drain_single(ptx::smem_u32(&cb->v_full[s]), ((vn - 1 - s) / NV) & 1,
                              args.status);
        }
      }
      __syncwarp();
    } else if (warp == kMmaWarp || warp == kMmaWarp + 1) {
      // ---------------------------------------------------------- MMA issuers
      // The whole warp runs this converged (waits are warp-uniform); the
      // MMAs, commits and arrives are done by one elected lane.
      {
        const int t = warp - kMmaWarp;  // query tile this warp issues for
        constexpr uint32_t idesc_s = ptx::idesc_bf16_f32(kBM, kBN, false, false);
        uint32_t q_par = 0;   // bit b: parity of the q_full[b] phases consumed
        uint32_t item_n = 0;  // items with KV tiles so far (selects the Q pair)
        uint32_t pn = 0, ofn = 0;
        uint32_t sfn = 0;     // s_free phases consumed (p_cols)
        uint32_t groups = 0;  // issue groups done by this issuer
        // Wait for this issuer's turn; issuer 0 starts.
        auto take_turn = [&]() -> bool {
          if (!C::turns || (t == 0 && groups == 0)) return true;
          const uint32_t par = (t == 0 ? groups - 1 : groups) & 1;
          return wait_warp(ptx::smem_u32(&cb->turn[t]), par, abort_flag, args.status, args.wait_limit_ns);
        };
        auto pass_turn = [&]() {
          if (C::turns) ptx::mbar_arrive_elect(ptx::smem_u32(&cb->turn[t ^ 1]));
          ++groups;
        };
        uint32_t kn = 0, vn = 0;  // tiles consumed from each ring
        bool ok = true;

        // Descriptors are built once per buffer; the MMAs of a group add
        // constant offsets to them.
        constexpr uint32_t kQkTailSbo = 8 * (QK::tail ? QK::tail : 16) * 2;
        constexpr uint32_t kQkTailLay = layout_for_width(QK::tail ? QK::tail : 16);
        // Descriptors of this issuer's Q tile in the current item's pair.
        uint64_t q_desc = 0, q_desc_tail = 0;
        auto set_q = [&](int b) {
          const uint32_t qa = ptx::smem_u32(q_base + b * C::q_tile_bytes);
          q_desc = ptx::smem_desc(qa, 16, 1024, ptx::kLayoutSw128);
          q_desc_tail =
              ptx::smem_desc(qa + QK::chunk_off(QK::full, kBM), 16, kQkTailSbo, kQkTailLay);
        };
        auto issue_s = [&](const uint8_t* kbuf) {
          const uint32_t ka = ptx::smem_u32(kbuf);
          const uint64_t kd = ptx::smem_desc(ka, 16, 1024, ptx::kLayoutSw128);
          const uint64_t kd_tail =
              ptx::smem_desc(ka + QK::chunk_off(QK::full, kBN), 16, kQkTailSbo, kQkTailLay);
          issue_s_group<QK::full, QK::tail>(tmem + C::s_col(t), q_desc, kd, q_desc_tail, kd_tail,
                                            idesc_s);
        };
        auto issue_pv = [&](const uint8_t* vbuf, bool first) {
          // One MMA per 16 keys over all of d_v: MN-major B spanning
          // C::v_atoms atoms (LBO = atom stride), 8-key groups SBO apart.
          constexpr uint32_t idesc_pv = ptx::idesc_bf16_f32(kBM, C::pv_n, false, true);
          constexpr uint32_t kRowBytes = C::v_atom * 2;
          const uint64_t vd = ptx::smem_desc(ptx::smem_u32(vbuf), C::v_atom_bytes, 8 * kRowBytes,
                                             layout_for_width(C::v_atom));
          // 16 keys = 16 rows of kRowBytes: kRowBytes 16-byte units per step.
          issue_pv_group<kRowBytes>(tmem + C::o_col(t), tmem + C::p_col(t), vd, idesc_pv,
                                    first ? 0u : 1u);
        };
        auto issue_pv_h = [&](const uint8_t* vbuf, bool first, int h) {
          constexpr uint32_t idesc_pv = ptx::idesc_bf16_f32(kBM, C::pv_n, false, true);
          constexpr uint32_t kRowBytes = C::v_atom * 2;
          const uint64_t vd = ptx::smem_desc(ptx::smem_u32(vbuf), C::v_atom_bytes, 8 * kRowBytes,
                                             layout_for_width(C::v_atom));
          issue_pv_half<kRowBytes>(tmem + C::o_col(t), tmem + C::p_col(t), vd, idesc_pv,
                                   first ? 0u : 1u, h);
        };
        // Both issuers walk every KV tile of every item (to stay in phase on
        // the ring); an issuer whose tile is absent from the item only waits
        // and releases.
        for (int r = 0; r * (int)gridDim.x < total_items && ok; ++r) {
          const int it = snake_item(r, split);
          if (it >= total_items) continue;
          WorkItem w;
          {
            const uint32_t sl = (uint32_t)r % kItemSlots;
            ok = wait_warp(ptx::smem_u32(&ring->full[sl]), ((uint32_t)r / kItemSlots) & 1,
                           abort_flag, args.status, args.wait_limit_ns);
            if (!ok) break;
            w = ring->slot[sl];
            ptx::mbar_arrive_elect(ptx::smem_u32(&ring->free_[sl]));
          }
          if (w.n_kv == 0) continue;
          const bool mine = t < w.n_qt;
          // This tile's key tiles: S_t(j) for j in [jlo, jhi), issued at the
          // step before (or in the prologue), P V_t(j) at step j.
          int jlo = 0, jhi = 0;
          if (mine) {
            if (C::tile_ranges)
              tile_kv_range(w, t, args.wl, args.wr, pshift, jlo, jhi);
            else
              jhi = w.n_kv;
          }
          const int qb = 2 * (C::q_pairs == 2 ? (int)(item_n & 1) : 0) + t;  // Q buffer
          ++item_n;
          if (mine) {
            ok = wait_warp(ptx::smem_u32(&cb->q_full[qb]), (q_par >> qb) & 1, abort_flag,
                           args.status, args.wait_limit_ns);
            q_par ^= 1u << qb;
            if (!ok) break;
            set_q(qb);
          }
          // Prologue: S_t(0).
          {
            const uint32_t ks = ring_slot<NK>(kn);
            ok = wait_warp(ptx::smem_u32(&cb->k_full[ks]), (kn / NK) & 1, abort_flag,
                           args.status, args.wait_limit_ns);
            if (ok) ok = take_turn();
            if (!ok) break;
            ptx::tc_fence_after();
            const bool s0 = jlo == 0 && jhi > 0;  // (jhi > jlo only for an owned tile)
            if (s0) issue_s(k_ring + ks * C::k_slot_bytes);
            pass_turn();
            if (s0) ptx::mma_commit_elect(ptx::smem_u32(&cb->s_full[t]));
            // Q is free once the tile's last S is done (or it has none).
            if (!C::stage_o && mine && (jhi <= jlo || (s0 && jhi == 1)))
              ptx::mma_commit_elect(ptx::smem_u32(&cb->q_free[qb]));
            ptx::mma_commit_elect(ptx::smem_u32(&cb->k_free[ks]));
            ++kn;
          }
          if constexpr (C::p_cols) {
            for (int j = 0; j < w.n_kv && ok; ++j) {
              const bool has_next = j + 1 < w.n_kv;
              const bool pv = j >= jlo && j < jhi;              // P V_t(j) at this step
              const bool s_next = j + 1 >= jlo && j + 1 < jhi;  // S_t(j + 1) at this step
              // S_t(j + 1) once K_{j+1} has landed and the softmax has
              // loaded S_t(j) out of the columns it overwrites.
              if (has_next) {
                const uint32_t ks = ring_slot<NK>(kn);
                ok = wait_warp(ptx::smem_u32(&cb->k_full[ks]), (kn / NK) & 1, abort_flag,
                               args.status, args.wait_limit_ns);
                ++kn;
                if (!ok) break;
                if (pv && s_next) {
                  ok = wait_warp(ptx::smem_u32(&cb->s_free[t]), sfn & 1, abort_flag, args.status,
                                 args.wait_limit_ns);
                  ++sfn;
                  if (!ok) break;
                }
                ptx::tc_fence_after();
                if (s_next) {
                  issue_s(k_ring + ks * C::k_slot_bytes);
                  ptx::mma_commit_elect(ptx::smem_u32(&cb->s_full[t]));
                  if (!C::stage_o && j + 2 == jhi)
                    ptx::mma_commit_elect(ptx::smem_u32(&cb->q_free[qb]));
                }
                ptx::mma_commit_elect(ptx::smem_u32(&cb->k_free[ks]));
              }
              // P V_t(j) once V_j has landed and the softmax has written
              // P_t(j) (keys 0..63 first with split_pv).
              const uint32_t vs = ring_slot<NV>(vn);
              ok = wait_warp(ptx::smem_u32(&cb->v_full[vs]), (vn / NV) & 1, abort_flag,
                             args.status, args.wait_limit_ns);
              ++vn;
              if (!ok) break;
              if (pv) {
                if (j == jlo) {
                  ok = wait_warp(ptx::smem_u32(&cb->o_free[t]), (ofn & 1) ^ 1, abort_flag,
                                 args.status, args.wait_limit_ns);
                  ++ofn;
                  if (!ok) break;
                }
                if (C::split_pv) {
                  ok = wait_warp(ptx::smem_u32(&cb->p_half[t]), pn & 1, abort_flag, args.status,
                                 args.wait_limit_ns);
                  if (!ok) break;
                  ptx::tc_fence_after();
                  issue_pv_h(v_ring + vs * C::v_slot_bytes, j == jlo, 0);
                }
                ok = wait_warp(ptx::smem_u32(&cb->p_full[t]), pn & 1, abort_flag, args.status,
                               args.wait_limit_ns);
                ++pn;
                if (!ok) break;
                ptx::tc_fence_after();
                if (C::split_pv)
                  issue_pv_h(v_ring + vs * C::v_slot_bytes, false, 1);
                else
                  issue_pv(v_ring + vs * C::v_slot_bytes, j == jlo);
                // The softmax of step j + 1 rescales O_t and overwrites P_t
                // only after this P V; the tile's last one ends in o_full.
                ptx::mma_commit_elect(
                    ptx::smem_u32(j + 1 == jhi ? &cb->o_full[t] : &cb->pv_done[t]));
              }
              ptx::mma_commit_elect(ptx::smem_u32(&cb->v_free[vs]));
            }
          } else {
            for (int j = 0; j < w.n_kv && ok; ++j) {
              const bool has_next = j + 1 < w.n_kv;
              const bool pv = j >= jlo && j < jhi;                  // P V_t(j) at this step
              const bool s_next = j + 1 >= jlo && j + 1 < jhi;      // S_t(j + 1) at this step
              // Operands and turn first: they are normally settled long before
              // P_t(j) is, so the wait for P is the last thing before the MMAs.
              // With a one-slot K ring, K_{j+1} only starts loading once both
              // tiles' S(j) are done, so it is waited for after P V_j instead.
              constexpr bool kEarlyK = NK > 1;
              const uint32_t vs = ring_slot<NV>(vn);
              ok = wait_warp(ptx::smem_u32(&cb->v_full[vs]), (vn / NV) & 1, abort_flag,
                             args.status, args.wait_limit_ns);
              if (!ok) break;
              ++vn;
              const uint32_t ks = ring_slot<NK>(kn);
              auto wait_k = [&]() -> bool {
                const bool r = wait_warp(ptx::smem_u32(&cb->k_full[ks]), (kn / NK) & 1, abort_flag,
                                         args.status, args.wait_limit_ns);
                ++kn;
                return r;
              };
              if (kEarlyK && has_next) {
                ok = wait_k();
                if (!ok) break;
              }
              ok = take_turn();
              if (!ok) break;
              if (pv) {
                if (j == jlo) {
                  ok = wait_warp(ptx::smem_u32(&cb->o_free[t]), (ofn & 1) ^ 1, abort_flag,
                                 args.status, args.wait_limit_ns);
                  ++ofn;
                  if (!ok) break;
                }
                if (C::split_pv) {
                  ok = wait_warp(ptx::smem_u32(&cb->p_half[t]), pn & 1, abort_flag, args.status, args.wait_limit_ns);
                  if (!ok) break;
                  ptx::tc_fence_after();
                  issue_pv_h(v_ring + vs * C::v_slot_bytes, j == jlo, 0);
                }
                ok = wait_warp(ptx::smem_u32(&cb->p_full[t]), pn & 1, abort_flag, args.status, args.wait_limit_ns);
                ++pn;
                if (!ok) break;
                ptx::tc_fence_after();
                if (C::split_pv)
                  issue_pv_h(v_ring + vs * C::v_slot_bytes, false, 1);
                else
                  issue_pv(v_ring + vs * C::v_slot_bytes, j == jlo);
              }
              if (!kEarlyK && has_next) {
                ok = wait_k();
                if (!ok) break;
                ptx::tc_fence_after();
              }
              if (s_next) issue_s(k_ring + ks * C::k_slot_bytes);
              // The other issuer goes next, then the commits (a commit tracks
              // this thread's MMAs alone; issuing one costs the warp time that
              // would otherwise delay the other query tile's MMAs).
              pass_turn();
              if (s_next) ptx::mma_commit_elect(ptx::smem_u32(&cb->s_full[t]));
              if (pv && j + 1 == jhi) ptx::mma_commit_elect(ptx::smem_u32(&cb->o_full[t]));
              if (!C::stage_o && s_next && j + 2 == jhi)
                ptx::mma_commit_elect(ptx::smem_u32(&cb->q_free[qb]));
              if (has_next) ptx::mma_commit_elect(ptx::smem_u32(&cb->k_free[ks]));
              ptx::mma_commit_elect(ptx::smem_u32(&cb->v_free[vs]));
            }
          }
        }
        // Drain: every MMA issued by either issuer completes before TMEM is
        // freed (the barrier expects one arrival from each issuer).
        ptx::mma_commit_elect(ptx::smem_u32(&cb->drain));
        wait_drain_warp(ptx::smem_u32(&cb->drain), 0, args.status);
      }
    }
  } else {
    ptx::regs_inc<kSoftmaxRegs>();
    // ------------------------------------------------------------ softmax WG t
    const int t = warp >> 2;                 // query tile of this warpgroup
    const int row_in_tile = tid & 127;       // == TMEM lane
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t s_addr = tmem + lane_base + C::s_col(t);
    const uint32_t o_addr = tmem + lane_base + C::o_col(t);
    const uint32_t p_addr = tmem + lane_base + C::p_col(t);
    const float sl2 = args.scale_log2;
    const float neg_inf = -__int_as_float(0x7f800000);
    uint32_t sn = 0, on = 0;
    uint32_t pdn = 0;     // pv_done phases consumed (p_cols)
    uint32_t item_n = 0;  // items with KV tiles so far (selects the Q pair)
    int staged_qb = -1;   // Q buffer holding O rows still being copied out
    // Releases the Q buffer of the last staged O once its copies have read it.
    auto release_staged = [&]() {
      if (C::stage_o && staged_qb >= 0) {
        ptx::bulk_wait_read_all();
        ptx::mbar_arrive(ptx::smem_u32(&cb->q_free[staged_qb]));
        staged_qb = -1;
      }
    };
    bool ok = true;

    for (int r = 0; r * (int)gridDim.x < total_items && ok; ++r) {
      const int it = snake_item(r, split);
      if (it >= total_items) continue;
      WorkItem w;
      {
        const uint32_t sl = (uint32_t)r % kItemSlots;
        ok = wait_warp(ptx::smem_u32(&ring->full[sl]), ((uint32_t)r / kItemSlots) & 1, abort_flag,
                       args.status, args.wait_limit_ns);
        if (!ok) break;
        w = ring->slot[sl];
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(ptx::smem_u32(&ring->free_[sl]));
      }
      const int qb = 2 * (C::q_pairs == 2 ? (int)(item_n & 1) : 0) + t;  // this item's Q buffer
      if (w.n_kv > 0) ++item_n;
      if (t >= w.n_qt) continue;
      release_staged();
      // Query token of this row within the sequence.
      const int i = w.row0 + ((t * kBM + row_in_tile) >> pshift);
      const bool row_valid = i < w.lq;
      int jlo = 0, jhi = w.n_kv;  // this tile's key tiles (its issuer walks the same)
      if (C::tile_ranges) tile_kv_range(w, t, args.wl, args.wr, pshift, jlo, jhi);
      // Every row of the tile a token of one sequence (one head per tile):
      // the staged O rows leave with one tensor store instead of one bulk
      // copy per row (128 copies per tile queue up in the copy engine, ahead
      // of the next item's loads; 256-token ViT windows at d80: 54.0 -> 49.8
      // us).  Packs of short segments keep the per-row copies (measured:
      // the tile store made 64-token windows 8 % slower).
      const bool whole_o = C::stage_o && jhi > jlo && pshift == 0 && w.nb == 1 &&
                           w.row0 + (t + 1) * kBM <= w.lq;
      const int off = w.lk - w.lq;
      int lo_i = 0, hi_i = 0;
      if (row_valid && w.nb > 1) {
        // A pack of short segments: the row's own segment [s0, s1) (keys and
        // rows share token offsets there), then the window inside it.
        const int g = w.q_start + i;
        int lo = w.b0, hi = w.b0 + w.nb - 1;
        while (lo < hi) {
          const int mid = (lo + hi + 1) >> 1;
          if (seq_lo(args.cu_q, mid, args.total_q) <= g) lo = mid; else hi = mid - 1;
        }
        const int s0 = seq_lo(args.cu_q, lo, args.total_q) - w.q_start;
        const int s1 = seq_hi(args.cu_q, lo, args.total_q) - w.q_start;
        lo_i = args.wl >= 0 ? max(s0, i - args.wl) : s0;
        hi_i = args.wr >= 0 ? min(s1, i + args.wr + 1) : s1;
        if (hi_i < lo_i) hi_i = lo_i;
      } else if (row_valid) {
        lo_i = args.wl >= 0 ? max(0, i + off - args.wl) : 0;
        hi_i = args.wr >= 0 ? min(w.lk, i + off + args.wr + 1) : w.lk;
        if (hi_i < lo_i) hi_i = lo_i;
      }
      float m_used = neg_inf;  // running max, scaled log2 units
      float l = 0.f;
      for (int j = jlo; j < jhi; ++j) {
        ok = wait_warp(ptx::smem_u32(&cb->s_full[t]), sn & 1, abort_flag, args.status, args.wait_limit_ns);
        ++sn;
        if (!ok) break;
        ptx::tc_fence_after();
        // S through the sm_103 reducing TMEM load: the values and, per 32
        // columns, their maximum.
        float s[kBN], qmax[kBN / 32];
#pragma unroll
        for (int q = 0; q < kBN / 32; ++q) ptx::tmem_ld32_max(s_addr + q * 32, s + q * 32, qmax[q]);
        ptx::tmem_wait_ld();
#pragma unroll
        for (int q = 0; q < kBN / 16; ++q) ptx::reg_fence16f(s + q * 16);
#pragma unroll
        for (int q = 0; q < kBN / 32; ++q) ptx::reg_fence1f(qmax[q]);
        if (C::p_cols && j + 1 < jhi) {
          // S_t(j) is in registers: its columns may take S_t(j + 1).
          ptx::tc_fence_before();
          ptx::mbar_arrive(ptx::smem_u32(&cb->s_free[t]));
        }

        const int k0 = (w.tile_lo + j) * kBN;
        float row_max;
        if (k0 >= lo_i && k0 + kBN <= hi_i) {
          // Every key of the tile is visible to this row: the hardware max.
          row_max = ptx::max3(qmax[0], qmax[1], fmaxf(qmax[2], qmax[3]));
        } else {
          // Boundary tile for this row: mask keys outside [lo_i, hi_i) and
          // reduce in software (the hardware max is over the unmasked S).
          const unsigned span = (unsigned)(hi_i - lo_i);
#pragma unroll
          for (int c = 0; c < kBN; ++c)
            s[c] = ((unsigned)(k0 + c - lo_i) < span) ? s[c] : neg_inf;
          float mx[4];
#pragma unroll
          for (int k = 0; k < 4; ++k) mx[k] = fmaxf(s[k], s[k + 4]);
#pragma unroll
          for (int c = 8; c < kBN; c += 8) {
#pragma unroll
            for (int k = 0; k < 4; ++k) mx[k] = ptx::max3(mx[k], s[c + k], s[c + k + 4]);
          }
          row_max = ptx::max3(mx[0], mx[1], fmaxf(mx[2], mx[3]));
        }
        const float m_tile = row_max * sl2;  // -inf stays -inf
        const bool need = m_tile > m_used + kRescaleLog2;
        // O_t *= alpha for a rescale (the running max moved by more than the
        // threshold).  O_t must hold the sum of the earlier tiles: their P V
        // has completed (the commit that released this S tile came after
        // it; with p_cols, the pv_done wait before the call).
        auto rescale_o = [&](float alpha) {
#pragma unroll
          for (int c0 = 0; c0 < C::pv_n; c0 += 16) {
            uint32_t o[16];
            ptx::tmem_ld16(o_addr + c0, o);
            ptx::tmem_wait_ld();
            ptx::reg_fence16(o);
#pragma unroll
            for (int c = 0; c < 16; ++c) o[c] = __float_as_uint(__uint_as_float(o[c]) * alpha);
            ptx::tmem_st16(o_addr + c0, o);
          }
        };
        // With p_cols, P V_t(j - 1) may still be running: the wait for it
        // (and the O rescale) comes after the first half of the exp2s.
        bool rescale_late = false;
        float alpha_late = 1.f;
        if (__any_sync(0xffffffffu, need)) {
          const float m_new = fmaxf(m_used, m_tile);
          const float alpha = (m_used == neg_inf) ? 0.f : ptx::ex2(m_used - m_new);
          if (C::p_cols) {
            rescale_late = j > jlo;
            alpha_late = alpha;
          } else if (j > jlo) {
            rescale_o(alpha);
          }
          if (m_new != neg_inf) {
            l *= alpha;
            m_used = m_new;
          }
        }
        const float base = (m_used == neg_inf) ? 0.f : m_used;
        // exp2(s * scale_log2 - base) with packed fp32x2 FMA / ADD (one
        // instruction per element pair), MUFU ex2 per element, and the fp32
        // row sum in four packed accumulators.
        const uint64_t sl2x2 = ptx::f2_pack(sl2, sl2);
        const uint64_t nbx2 = ptx::f2_pack(-base, -base);
        uint32_t pr[kBN / 2];
        {
          uint64_t ls2[4] = {0ull, 0ull, 0ull, 0ull};
          // Keys [c0, c0 + 64): exp2, row sum, P as bf16 pairs.
          auto exp_half = [&](auto half) {
            constexpr int c0 = decltype(half)::value * (kBN / 2);
#pragma unroll
            for (int c = c0; c < c0 + kBN / 2; c += 2) {
              float x0, x1;
              ptx::f2_unpack(ptx::fma2(ptx::f2_pack(s[c], s[c + 1]), sl2x2, nbx2), x0, x1);
              const float p0 = ptx::ex2(x0);
              const float p1 = ptx::ex2(x1);
              ls2[(c >> 1) & 3] = ptx::add2(ls2[(c >> 1) & 3], ptx::f2_pack(p0, p1));
              pr[c >> 1] = ptx::pack_bf16x2(p0, p1);
            }
          };
          exp_half(IntTag<0>{});
          if (C::p_cols && j > jlo) {
            // P V_t(j - 1) has read P_t and added into O_t.
            if (!wait_warp(ptx::smem_u32(&cb->pv_done[t]), pdn & 1, abort_flag, args.status,
                           args.wait_limit_ns))
              ok = false;
            ++pdn;
            ptx::tc_fence_after();
            if (ok && rescale_late) rescale_o(alpha_late);
          }
          if (C::split_pv) {
            // The first 64 keys' P goes out before the rest is computed.
            ptx::tmem_st32(p_addr, pr);
            ptx::tmem_wait_st();
            ptx::tc_fence_before();
            ptx::mbar_arrive(ptx::smem_u32(&cb->p_half[t]));
          }
          exp_half(IntTag<1>{});
          float a0, a1, b0, b1;
          ptx::f2_unpack(ptx::add2(ls2[0], ls2[1]), a0, a1);
          ptx::f2_unpack(ptx::add2(ls2[2], ls2[3]), b0, b1);
          l += (a0 + b0) + (a1 + b1);
        }
        if (!ok) break;
#pragma unroll
        for (int q = C::split_pv ? 32 : 0; q < kBN / 2; q += 32) ptx::tmem_st32(p_addr + q, pr + q);
        ptx::tmem_wait_st();
        ptx::tc_fence_before();
        ptx::mbar_arrive(ptx::smem_u32(&cb->p_full[t]));
      }
      if (!ok) break;

      if (kGeneral && split > 1) {
        // Split-KV: this CTA holds one part of the item.  Its O stays in
        // TMEM for the cluster combine, and (m, l) go into the row's first
        // two S/P columns, dead once the last P V (before o_full) is done.
        if (jhi > jlo) {
          ok = wait_warp(ptx::smem_u32(&cb->o_full[t]), on & 1, abort_flag, args.status, args.wait_limit_ns);
          ++on;
          if (!ok) break;
          ptx::tc_fence_after();
          const uint32_t ml[2] = {__float_as_uint(m_used), __float_as_uint(l)};
          ptx::tmem_st2(s_addr, ml);
          ptx::tmem_wait_st();
        }
        continue;
      }

      // ---- epilogue: O / l -> bf16 rows, LSE
      uint32_t o[C::pv_n];
      if (jhi > jlo) {
        ok = wait_warp(ptx::smem_u32(&cb->o_full[t]), on & 1, abort_flag, args.status, args.wait_limit_ns);
        ++on;
        if (!ok) break;
        ptx::tc_fence_after();
#pragma unroll
        for (int c0 = 0; c0 < C::pv_n; c0 += 16) ptx::tmem_ld16(o_addr + c0, o + c0);
        ptx::tmem_wait_ld();
#pragma unroll
        for (int c0 = 0; c0 < C::pv_n; c0 += 16) ptx::reg_fence16(o + c0);
        ptx::tc_fence_before();
        ptx::mbar_arrive(ptx::smem_u32(&cb->o_free[t]));
      } else {
#pragma unroll
        for (int c = 0; c < C::pv_n; ++c) o[c] = 0u;
      }
      const bool staged = C::stage_o && jhi > jlo;
      // Query head of this row (packed heads: row % P).
      const int head = w.head + (row_in_tile & ((1 << pshift) - 1));
      uint8_t* const srow = q_base + qb * C::q_tile_bytes + row_in_tile * (D_V * 2);
      if (row_valid) {
        const float inv_l = l > 0.f ? 1.f / l : 0.f;
        const size_t tok = (size_t)(w.q_start + i);
        uint4* dst = reinterpret_cast<uint4*>(args.out +
                                              (tok * args.num_heads + head) * (size_t)D_V);
        auto pk = [&](int c) {
          return ptx::pack_bf16x2(__uint_as_float(o[c]) * inv_l, __uint_as_float(o[c + 1]) * inv_l);
        };
        if (!staged && D_V % 16 == 0 && ((reinterpret_cast<uintptr_t>(args.out) & 31) == 0)) {
          // Unstaged rows (one per thread, so each warp instruction touches
          // 32 rows): 32-byte stores, half as many instructions as 16-byte.
#pragma unroll
          for (int g = 0; g < D_V / 16; ++g) {
            uint32_t wv[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) wv[k] = pk(16 * g + 2 * k);
            ptx::st_global_v8(dst + 2 * g, wv);
          }
        } else {
#pragma unroll
          for (int g = 0; g < D_V / 8; ++g) {
            uint4 v;
            v.x = pk(8 * g + 0);
            v.y = pk(8 * g + 2);
            v.z = pk(8 * g + 4);
            v.w = pk(8 * g + 6);
            if (staged)
              reinterpret_cast<uint4*>(srow)[g] = v;
            else
              dst[g] = v;
          }
        }
        if (staged && !whole_o) {
          ptx::fence_proxy_async_smem();  // the copy engine reads the row
          ptx::bulk_store(dst, ptx::smem_u32(srow), D_V * 2);
          ptx::bulk_commit();
        }
        if (args.lse) {
          // Natural-log LSE: (m + log2 l) * ln 2.
          const float lse = l > 0.f ? (m_used + __log2f(l)) * 0.69314718055994531f : neg_inf;
          args.lse[(size_t)head * args.total_q + tok] = lse;
        }
      }
      if (whole_o) {
        ptx::fence_proxy_async_smem();  // the copy engine reads the staged rows
        ptx::named_bar_sync_n(2 + t, kBM);
        if (row_in_tile == 0) {  // its row is the tile's first: token q_start + i
          ptx::tma_store_3d(&maps.o_rows, ptx::smem_u32(srow), 0, head, w.q_start + i);
          ptx::bulk_commit();
        }
      }
      // The Q buffer (loaded for every item with key tiles) is released once
      // any staged rows have been read out.
      if (C::stage_o && w.n_kv > 0) staged_qb = qb;
    }
    release_staged();
    ptx::bulk_wait_all();  // every O row written before the CTA exits
    if (kGeneral && split > 1) {
      // Both warpgroups are past their last O wait, so every MMA of the item
      // has completed (each issuer's last commit covers all of its MMAs) and
      // the Q tiles and K/V rings are dead: the partial goes there.
      ptx::named_bar_sync_n(1, 256);
      const int it = (int)blockIdx.x / split;
      const WorkItem w = it < total_items ? decode_item(it, args, s_prefix, s_sorted, split, pshift) : WorkItem{};
      if (it < total_items && t < w.n_qt) {
        ptx::tc_fence_after();
        const int r = t * kBM + row_in_tile;  // row within the item
        uint8_t* row = smem + r * SplitStash<D_V>::kRowBytes;
        int jlo = 0, jhi = w.n_kv;
        if (C::tile_ranges) tile_kv_range(w, t, args.wl, args.wr, pshift, jlo, jhi);
        const bool has_o = jhi > jlo;
        float sp_m = neg_inf, sp_l = 0.f;
        if (has_o) {
          uint32_t ml[2];
          ptx::tmem_ld2(s_addr, ml);
          ptx::tmem_wait_ld();
          sp_m = __uint_as_float(ml[0]);
          sp_l = __uint_as_float(ml[1]);
        }
        if (has_o) {
#pragma unroll
          for (int c0 = 0; c0 < D_V; c0 += 16) {
            uint32_t o[16];
            ptx::tmem_ld16(o_addr + c0, o);
            ptx::tmem_wait_ld();
            ptx::reg_fence16(o);
#pragma unroll
            for (int c = 0; c < 16; c += 4)
              if (c0 + c < D_V)
                *reinterpret_cast<uint4*>(row + (c0 + c) * 4) =
                    make_uint4(o[c], o[c + 1], o[c + 2], o[c + 3]);
          }
        } else {
#pragma unroll
          for (int c = 0; c < D_V; c += 4)
            *reinterpret_cast<uint4*>(row + c * 4) = make_uint4(0u, 0u, 0u, 0u);
        }
        *reinterpret_cast<float2*>(smem + SplitStash<D_V>::kMlOff + r * 8) =
            make_float2(sp_m, sp_l);
      }
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (kGeneral && split > 1) split_combine<D_V>(args, smem, s_prefix, s_sorted, total_items);
  if (warp == kMmaWarp) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, 512);
  }
}

// Dynamic shared memory a launch needs for a given batch.
template <int D_QK, int D_V>
inline size_t varlen_smem_bytes(int batch) {
  using C = VarlenCfg<D_QK, D_V>;
  return (size_t)1024 + 2 * C::q_pairs * C::q_tile_bytes + (size_t)C::nk * C::k_slot_bytes +
         (size_t)C::nv * C::v_slot_bytes +
         sizeof(VarlenBarriers) + 8 * (size_t)(batch + 1) + 4 * kVarlenThreads + 16;
}

// What the host knows about a call's work, for the launch shape.
struct VarlenLaunch {
  int sm_count;
  long long item_bound;  // upper bound on the work items (query heads x 256-row pairs)
  long long kv_tiles;    // estimate of one item's KV tiles (performance only)
};

// Largest number of clusters of `split` CTAs of this kernel that can be
// resident at once on the current device (0 if none), queried once per
// device and cluster size.
template <int D_QK, int D_V>
int varlen_max_clusters(int dev, int split) {
  static std::atomic<int> cache[64][kMaxSplit + 1];  // value + 1; 0 = not yet queried
  const int c = cache[dev][split].load(std::memory_order_acquire);
  if (c > 0) return c - 1;
  cudaLaunchConfig_t cfg;
  std::memset(&cfg, 0, sizeof cfg);
  cfg.gridDim = dim3(split);
  cfg.blockDim = dim3(kVarlenThreads);
  cfg.dynamicSmemBytes = varlen_smem_bytes<D_QK, D_V>(kMaxBatch);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = split;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, varlen_fwd_kernel<D_QK, D_V, true>, &cfg) != cudaSuccess) {
    cudaGetLastError();  // not a sticky error: clear it and report no cluster
    n = 0;
  }
  cache[dev][split].store(n + 1, std::memory_order_release);
  return n;
}

// Split-KV when the work items cannot fill half of the SMs: the largest
// cluster size (at most kMaxSplit, 8 where larger clusters are unavailable)
// whose clusters, one per item, are all resident at once and whose parts
// keep at least four KV tiles.  1 = no split.
template <int D_QK, int D_V>
int varlen_split_choice(int dev, const VarlenLaunch& L, bool large_clusters) {
  if (L.item_bound < 1 || L.item_bound * 2 > L.sm_count || L.kv_tiles < 8) return 1;
  for (int s = large_clusters ? kMaxSplit : 8; s >= 2; --s) {
    if (L.kv_tiles < 4LL * s || L.item_bound * s > L.sm_count) continue;
    if (L.item_bound <= varlen_max_clusters<D_QK, D_V>(dev, s)) return s;
  }
  return 1;
}

// Launch shape the launcher below picks: CTAs and CTAs per work item.
template <int D_QK, int D_V>
cudaError_t varlen_plan_impl(const VarlenLaunch& L, int* grid, int* split) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  // Without the non-portable cluster-size permission set (the launcher sets
  // it on first use) the query still reports what is possible.
  cudaFuncSetAttribute(varlen_fwd_kernel<D_QK, D_V, true>,
                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                       (int)varlen_smem_bytes<D_QK, D_V>(kMaxBatch));
  const bool large = cudaFuncSetAttribute(varlen_fwd_kernel<D_QK, D_V, true>,
                                          cudaFuncAttributeNonPortableClusterSizeAllowed,
                                          1) == cudaSuccess;
  cudaGetLastError();
  *split = varlen_split_choice<D_QK, D_V>(dev, L, large);
  long long g = *split > 1 ? L.item_bound * *split
                           : (L.item_bound < L.sm_count ? L.item_bound : L.sm_count);
  *grid = (int)(g < 1 ? 1 : g);
  return cudaSuccess;
}

// Launches one instantiation: a persistent grid of at most one CTA per SM,
// or, for split-KV, one cluster per work item.  The dynamic shared-memory
// limit (for the largest supported batch) and the cluster-size permission
// are set once per device; concurrent first calls may both set them (the
// calls are idempotent), the flags themselves are atomic.
template <int D_QK, int D_V>
cudaError_t launch_varlen_impl(const VarlenMaps& maps, const VarlenArgs& args_in,
                               const VarlenLaunch& L, cudaStream_t stream) {
  static std::atomic<int> attr_done[64];  // 0 = not set, 1 = set, 2 = set with large clusters
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  int attrs = attr_done[dev].load(std::memory_order_acquire);
  if (attrs == 0) {
    e = cudaFuncSetAttribute(varlen_fwd_kernel<D_QK, D_V, false>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)varlen_smem_bytes<D_QK, D_V>(kMaxBatch));
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(varlen_fwd_kernel<D_QK, D_V, true>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)varlen_smem_bytes<D_QK, D_V>(kMaxBatch));
    if (e != cudaSuccess) return e;
    const bool large = cudaFuncSetAttribute(varlen_fwd_kernel<D_QK, D_V, true>,
                                            cudaFuncAttributeNonPortableClusterSizeAllowed,
                                            1) == cudaSuccess;
    if (!large) cudaGetLastError();
    attrs = large ? 2 : 1;
    attr_done[dev].store(attrs, std::memory_order_release);
  }
  VarlenArgs args = args_in;
  args.split = varlen_split_choice<D_QK, D_V>(dev, L, attrs == 2);
  const size_t smem = varlen_smem_bytes<D_QK, D_V>(args.batch);
  if (args.split == 1) {
    long long grid = L.item_bound < L.sm_count ? L.item_bound : L.sm_count;
    if (grid < 1) grid = 1;
    if (args.pack_shift == 0)
      varlen_fwd_kernel<D_QK, D_V, false><<<(int)grid, kVarlenThreads, smem, stream>>>(maps, args);
    else
      varlen_fwd_kernel<D_QK, D_V, true><<<(int)grid, kVarlenThreads, smem, stream>>>(maps, args);
    return cudaGetLastError();
  }
  cudaLaunchConfig_t cfg;
  std::memset(&cfg, 0, sizeof cfg);
  cfg.gridDim = dim3((unsigned)(L.item_bound * args.split));
  cfg.blockDim = dim3(kVarlenThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = args.split;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, varlen_fwd_kernel<D_QK, D_V, true>, maps, args);
}

}  // namespace fa

#define FA_DEFINE_VARLEN_LAUNCHER(DQK, DV)                                              \
  namespace fa {                                                                         \
  cudaError_t launch_varlen_##DQK##_##DV(const VarlenMaps& maps, const VarlenArgs& args, \
                                         const VarlenLaunch& L, cudaStream_t stream) {  \
    return launch_varlen_impl<DQK, DV>(maps, args, L, stream);                           \
  }                                                                                      \
  cudaError_t plan_varlen_##DQK##_##DV(const VarlenLaunch& L, int* grid, int* split) {   \
    return varlen_plan_impl<DQK, DV>(L, grid, split);                                    \
  }                                                                                      \
  }
