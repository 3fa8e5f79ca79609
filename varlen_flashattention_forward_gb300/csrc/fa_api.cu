// fa_api.cu -- host side of the C ABI declared in include/fa_gb300.h:
// argument validation, TMA descriptor encoding, dispatch over the compiled
// head-dim instantiations, and the device status word.
//
// No function here copies data or synchronises, except fa_get_device_status
// (documented as synchronising).  The only device memory the library
// allocates is the partial-result workspace of fa_sparse_mla_decode: one
// buffer per (device, stream), allocated by the first call on that stream
// whose work split needs it and reused by every later call; a call that needs
// more than the stream's buffer holds allocates a larger one and keeps the
// old one allocated (a CUDA graph captured earlier may still point at it).
#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <new>
#include <vector>

#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/fa_gb300.h"
#include "decode_plan.h"
#include "merge_kernel.cuh"
#include "sparse_decode_kernel.cuh"
#include "varlen_fwd_kernel.cuh"

namespace fa {
cudaError_t launch_varlen_64_64(const VarlenMaps&, const VarlenArgs&, const VarlenLaunch&,
                                 cudaStream_t);
cudaError_t plan_varlen_64_64(const VarlenLaunch&, int*, int*);
cudaError_t launch_varlen_72_72(const VarlenMaps&, const VarlenArgs&, const VarlenLaunch&,
                                 cudaStream_t);
cudaError_t plan_varlen_72_72(const VarlenLaunch&, int*, int*);
cudaError_t launch_varlen_80_80(const VarlenMaps&, const VarlenArgs&, const VarlenLaunch&,
                                 cudaStream_t);
cudaError_t plan_varlen_80_80(const VarlenLaunch&, int*, int*);
cudaError_t launch_varlen_96_96(const VarlenMaps&, const VarlenArgs&, const VarlenLaunch&,
                                 cudaStream_t);
cudaError_t plan_varlen_96_96(const VarlenLaunch&, int*, int*);
cudaError_t launch_varlen_128_128(const VarlenMaps&, const VarlenArgs&, const VarlenLaunch&,
                                 cudaStream_t);
cudaError_t plan_varlen_128_128(const VarlenLaunch&, int*, int*);
cudaError_t launch_varlen_192_128(const VarlenMaps&, const VarlenArgs&, const VarlenLaunch&,
                                 cudaStream_t);
cudaError_t plan_varlen_192_128(const VarlenLaunch&, int*, int*);
}  // namespace fa

// Device status word: bit 0 = a pipeline wait ran out of time.
__device__ unsigned int g_fa_status = 0;

namespace {

constexpr int kMaxDevices = 64;

struct DeviceInfo {
  bool ready = false;
  bool arch_ok = false;
  int sm_count = 0;
  unsigned int* status = nullptr;  // device address of g_fa_status
};

std::mutex g_mu;
DeviceInfo g_dev[kMaxDevices];

// Time limit of the kernels' pipeline waits, passed to every launch.
std::atomic<unsigned long long> g_wait_limit_ns{fa::kWaitLimitNs};

// Per-device facts, queried once.  The first call on a device therefore
// performs runtime queries (no stream work); make it before any stream
// capture if the call is to be captured.
fa_status device_info(DeviceInfo** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return FA_ERR_LAUNCH;
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceInfo& d = g_dev[dev];
  if (!d.ready) {
    int major = 0, minor = 0, sms = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return FA_ERR_LAUNCH;
    d.arch_ok = (major == 10 && minor == 3);
    d.sm_count = sms;
    void* p = nullptr;
    if (d.arch_ok) {
      if (cudaGetSymbolAddress(&p, g_fa_status) != cudaSuccess) return FA_ERR_LAUNCH;
    }
    d.status = static_cast<unsigned int*>(p);
    d.ready = true;
  }
  *out = &d;
  return d.arch_ok ? FA_OK : FA_ERR_ARCH;
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// 3-D bf16 tensor [tokens, heads, dim] (dim innermost) viewed through a box of
// {box_w, box_heads, box_rows}: shared-memory row r of a box is token
// r / box_heads, head r % box_heads.  The swizzle matches the box width
// (64 -> 128 B, 32 -> 64 B, 16 -> 32 B).  Elements past `dim` or `tokens`
// read as zero.
bool encode_rows(CUtensorMap* m, const void* base, int dim, int heads, int tokens, int box_w,
                 int box_rows, long long head_stride, long long row_stride, int box_heads = 1) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {(cuuint64_t)dim, (cuuint64_t)heads,
                        (cuuint64_t)(tokens > 0 ? tokens : 1)};
  // Strides in bytes of the head and token dimensions (elements are bf16).
  cuuint64_t strides[2] = {(cuuint64_t)head_stride * 2, (cuuint64_t)row_stride * 2};
  cuuint32_t box[3] = {(cuuint32_t)box_w, (cuuint32_t)box_heads, (cuuint32_t)box_rows};
  cuuint32_t estr[3] = {1u, 1u, 1u};
  CUtensorMapSwizzle swz = box_w == 64   ? CU_TENSOR_MAP_SWIZZLE_128B
                           : box_w == 32 ? CU_TENSOR_MAP_SWIZZLE_64B
                                         : CU_TENSOR_MAP_SWIZZLE_32B;
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Decode workspace of one (device, stream).  Calls on one stream run in
// order, so they can share it; calls on different streams get their own.
struct StreamWorkspace {
  int dev;
  cudaStream_t stream;
  void* ptr;
  size_t bytes;
};
std::vector<StreamWorkspace> g_ws;    // guarded by g_mu
std::vector<void*> g_ws_outgrown;     // replaced buffers, kept allocated

// The workspace of `stream` on the current device, at least `need` bytes.
// Allocates (cudaMalloc) only when the stream has none yet or a smaller one.
fa_status stream_workspace(cudaStream_t stream, size_t need, void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return FA_ERR_LAUNCH;
  std::lock_guard<std::mutex> lock(g_mu);
  StreamWorkspace* w = nullptr;
  for (auto& e : g_ws)
    if (e.dev == dev && e.stream == stream) w = &e;
  if (w && w->bytes >= need) {
    *out = w->ptr;
    return FA_OK;
  }
  // Round up to 4 MiB so that slowly growing requests reallocate rarely.
  const size_t bytes = (need + (4u << 20) - 1) / (4u << 20) * (4u << 20);
  void* p = nullptr;
  if (cudaMalloc(&p, bytes) != cudaSuccess) {
    cudaGetLastError();  // clear the sticky-free allocation error
    return FA_ERR_LAUNCH;
  }
  if (w) {
    g_ws_outgrown.push_back(w->ptr);
    w->ptr = p;
    w->bytes = bytes;
  } else {
    g_ws.push_back(StreamWorkspace{dev, stream, p, bytes});
  }
  *out = p;
  return FA_OK;
}

// Launch shape of a varlen call.  A sequence of l query rows has
// ceil(l / t) work items per head group (t = 256 / P tokens per item, P
// heads per group), and the sum of the ceilings is at most
// floor((total_q + (t - 1) batch) / t), so no more work items than
// item_bound exist (packed short segments only make fewer).  The KV tiles of one item
// are estimated from the max_seqlen_k hint (else total_k) and the window;
// they only steer the split-KV choice, never correctness.
// GQA head-group packing factor (log2): the largest power of two P <= 16
// that divides the group size num_heads / num_heads_k and still leaves a
// work item (256 / P tokens) at least as many tokens as a sequence is
// expected to have (the max_seqlen_q hint, else the mean).  Short query
// sequences then share each K/V tile among P heads instead of loading it
// once per head; long ones gain nothing from it and stay unpacked.
int pack_shift_for(int batch, int total_q, int num_heads, int num_heads_k, int max_seqlen_q) {
  const int g = num_heads / num_heads_k;
  long long lq = max_seqlen_q > 0 ? max_seqlen_q : ((long long)total_q + batch - 1) / batch;
  if (lq < 1) lq = 1;
  int shift = 0;
  while (shift < 4 && g % (2 << shift) == 0 && (fa::kRowsPerItem >> (shift + 1)) >= lq) ++shift;
  return shift;
}

fa::VarlenLaunch launch_shape(int sm_count, int batch, int total_q, int total_k, int num_heads,
                              int max_seqlen_k, int causal, int window_left, int window_right,
                              int pack_shift) {
  fa::VarlenLaunch L;
  L.sm_count = sm_count;
  // With packing an item holds 256 / P tokens of P heads.
  const long long tpi = fa::kRowsPerItem >> pack_shift;
  L.item_bound = (long long)(num_heads >> pack_shift) *
                 (((long long)total_q + (tpi - 1) * batch) / tpi);
  long long kv = total_k;
  if (max_seqlen_k > 0 && max_seqlen_k < kv) kv = max_seqlen_k;
  if (window_left >= 0 && (causal || window_right >= 0)) {
    const long long span =
        (long long)window_left + (causal ? 0 : window_right) + fa::kRowsPerItem;
    if (span < kv) kv = span;
  }
  L.kv_tiles = (kv + fa::kBN - 1) / fa::kBN;
  return L;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

int tail_width(int d) { return ((d + 15) / 16 * 16) % 64; }

}  // namespace

namespace {

// A strided [tokens, heads, dim] view: innermost dimension contiguous, head
// and token strides multiples of 16 bytes, no element reachable two ways.
bool valid_view(long long row_stride, long long head_stride, int heads, int dim) {
  if (row_stride <= 0 || head_stride <= 0) return false;
  if (row_stride % 8 != 0 || head_stride % 8 != 0) return false;
  if (head_stride < dim) return false;
  if (row_stride < (long long)(heads - 1) * head_stride + dim) return false;
  return row_stride < (1ll << 37) && head_stride < (1ll << 37);  // TMA stride range
}

}  // namespace

extern "C" fa_status fa_varlen_fwd(const void* q, const void* k, const void* v,
                                   const int* cu_seqlens_q, const int* cu_seqlens_k, int batch,
                                   int total_q, int total_k, int num_heads, int num_heads_k,
                                   int d_qk, int d_v, int max_seqlen_q, int max_seqlen_k,
                                   float softmax_scale, int causal, int window_left,
                                   int window_right, void* out, float* lse,
                                   fa_stream_t stream) {
  return fa_varlen_fwd_strided(
      q, (long long)num_heads * d_qk, d_qk, k, (long long)num_heads_k * d_qk, d_qk, v,
      (long long)num_heads_k * d_v, d_v, cu_seqlens_q, cu_seqlens_k, batch, total_q, total_k,
      num_heads, num_heads_k, d_qk, d_v, max_seqlen_q, max_seqlen_k, softmax_scale, causal,
      window_left, window_right, out, lse, stream);
}

extern "C" fa_status fa_varlen_fwd_strided(
    const void* q, long long q_row_stride, long long q_head_stride, const void* k,
    long long k_row_stride, long long k_head_stride, const void* v, long long v_row_stride,
    long long v_head_stride, const int* cu_seqlens_q, const int* cu_seqlens_k, int batch,
    int total_q, int total_k, int num_heads, int num_heads_k, int d_qk, int d_v,
    int max_seqlen_q, int max_seqlen_k, float softmax_scale, int causal, int window_left,
    int window_right, void* out, float* lse, fa_stream_t stream) {
  // ---- host validation (before any CUDA call); q and out may be null only
  // when they have no rows
  if ((total_q > 0 && (!q || !out)) || !cu_seqlens_q || !cu_seqlens_k) return FA_ERR_INVALID_ARG;
  if (total_k > 0 && (!k || !v)) return FA_ERR_INVALID_ARG;
  if (batch < 1 || total_q < 0 || total_k < 0 || num_heads < 1 || num_heads_k < 1 ||
      num_heads % num_heads_k != 0)
    return FA_ERR_INVALID_ARG;
  if (window_left < -1 || window_right < -1) return FA_ERR_INVALID_ARG;
  if (!(softmax_scale > 0.f) || !std::isfinite(softmax_scale)) return FA_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(out, 16) || (k && !aligned(k, 16)) || (v && !aligned(v, 16)) ||
      !aligned(cu_seqlens_q, 4) || !aligned(cu_seqlens_k, 4) || (lse && !aligned(lse, 4)))
    return FA_ERR_INVALID_ARG;
  typedef cudaError_t (*Launcher)(const fa::VarlenMaps&, const fa::VarlenArgs&,
                                  const fa::VarlenLaunch&, cudaStream_t);
  Launcher launch = nullptr;
  if (d_qk == 64 && d_v == 64) launch = fa::launch_varlen_64_64;
  else if (d_qk == 72 && d_v == 72) launch = fa::launch_varlen_72_72;
  else if (d_qk == 80 && d_v == 80) launch = fa::launch_varlen_80_80;
  else if (d_qk == 96 && d_v == 96) launch = fa::launch_varlen_96_96;
  else if (d_qk == 128 && d_v == 128) launch = fa::launch_varlen_128_128;
  else if (d_qk == 192 && d_v == 128) launch = fa::launch_varlen_192_128;
  if (!launch) return FA_ERR_UNSUPPORTED;
  if (!valid_view(q_row_stride, q_head_stride, num_heads, d_qk) ||
      (total_k > 0 && (!valid_view(k_row_stride, k_head_stride, num_heads_k, d_qk) ||
                       !valid_view(v_row_stride, v_head_stride, num_heads_k, d_v))))
    return FA_ERR_INVALID_ARG;
  // Token indices are 32-bit in the kernel.
  if ((int64_t)total_q * num_heads > INT32_MAX || (int64_t)total_k * num_heads_k > INT32_MAX)
    return FA_ERR_UNSUPPORTED;

  DeviceInfo* dev = nullptr;
  fa_status st = device_info(&dev);
  if (st != FA_OK) return st;
  if (total_q == 0) return FA_OK;

  // ---- TMA descriptors (host-only encoding, no device interaction)
  fa::VarlenMaps maps;
  std::memset(&maps, 0, sizeof maps);
  const void* kb = total_k > 0 ? k : q;  // never dereferenced when total_k == 0
  const void* vb = total_k > 0 ? v : q;
  const int kh = total_k > 0 ? num_heads_k : num_heads;
  const int vd = total_k > 0 ? d_v : d_qk;
  const int tk = total_k > 0 ? total_k : total_q;
  const long long krs = total_k > 0 ? k_row_stride : q_row_stride;
  const long long khs = total_k > 0 ? k_head_stride : q_head_stride;
  const long long vrs = total_k > 0 ? v_row_stride : q_row_stride;
  const long long vhs = total_k > 0 ? v_head_stride : q_head_stride;
  const int qt = tail_width(d_qk);
  const int pack_shift = pack_shift_for(batch, total_q, num_heads, num_heads_k, max_seqlen_q);
  const int qh = 1 << pack_shift;  // heads per Q box, fa::kBM / qh tokens
  bool ok = encode_rows(&maps.q_full, q, d_qk, num_heads, total_q, 64, fa::kBM / qh,
                        q_head_stride, q_row_stride, qh) &&
            encode_rows(&maps.k_full, kb, d_qk, kh, tk, 64, fa::kBN, khs, krs) &&
            encode_rows(&maps.v_full, vb, vd, kh, tk, fa::v_atom_width(vd), fa::kBN, vhs, vrs);
  if (ok && qt)
    ok = encode_rows(&maps.q_tail, q, d_qk, num_heads, total_q, qt, fa::kBM / qh, q_head_stride,
                     q_row_stride, qh) &&
         encode_rows(&maps.k_tail, kb, d_qk, kh, tk, qt, fa::kBN, khs, krs);
  if (ok) {
    // O as [total_q, H, d_v] through boxes of {d_v, 1, 128}, no swizzle.
    EncodeTiledFn fn = encode_fn();
    cuuint64_t dims[3] = {(cuuint64_t)d_v, (cuuint64_t)num_heads, (cuuint64_t)total_q};
    cuuint64_t strides[2] = {(cuuint64_t)d_v * 2, (cuuint64_t)num_heads * d_v * 2};
    cuuint32_t box[3] = {(cuuint32_t)d_v, 1u, (cuuint32_t)fa::kBM};
    cuuint32_t estr[3] = {1u, 1u, 1u};
    ok = fn && fn(&maps.o_rows, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, out, dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                  CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
                     CUDA_SUCCESS;
  }
  if (!ok) return FA_ERR_LAUNCH;

  fa::VarlenArgs args;
  args.num_heads = num_heads;
  args.num_heads_k = num_heads_k;
  args.total_q = total_q;
  args.total_k = total_k;
  args.scale_log2 = softmax_scale * 1.4426950408889634f;
  args.wl = window_left;
  // Causal is the window's right edge on the bottom-right diagonal
  // (window_right >= -1, so min(window_right, 0) is 0 whenever causal).
  args.wr = causal ? 0 : window_right;
  args.out = static_cast<uint16_t*>(out);
  args.lse = lse;
  args.status = dev->status;
  args.split = 1;
  args.pack_shift = pack_shift;
  args.wait_limit_ns = g_wait_limit_ns.load(std::memory_order_relaxed);

  // One launch per chunk of at most kMaxBatch sequences (the kernel keeps a
  // chunk's work list in shared memory).  cu_seqlens hold absolute token
  // offsets, so a chunk is the same arrays from its first sequence on; the
  // chunks' outputs and LSE rows are disjoint.
  for (long long b0 = 0; b0 < batch; b0 += fa::kMaxBatch) {
    const int nb = (int)std::min<long long>(fa::kMaxBatch, batch - b0);
    args.cu_q = cu_seqlens_q + b0;
    args.cu_k = cu_seqlens_k + b0;
    args.batch = nb;
    const fa::VarlenLaunch L = launch_shape(dev->sm_count, nb, total_q, total_k, num_heads,
                                            max_seqlen_k, causal, window_left, window_right,
                                            pack_shift);
    const cudaError_t e = launch(maps, args, L, reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return FA_ERR_LAUNCH;
  }
  return FA_OK;
}

extern "C" fa_status fa_varlen_fwd_plan(int batch, int total_q, int total_k, int num_heads,
                                        int num_heads_k, int d_qk, int d_v, int max_seqlen_q,
                                        int max_seqlen_k, int causal, int window_left,
                                        int window_right, int* grid, int* split,
                                        int* heads_per_tile) {
  if (!grid || !split || !heads_per_tile) return FA_ERR_INVALID_ARG;
  if (batch < 1 || total_q < 0 || total_k < 0 || num_heads < 1 || num_heads_k < 1 ||
      num_heads % num_heads_k != 0 || window_left < -1 || window_right < -1)
    return FA_ERR_INVALID_ARG;
  typedef cudaError_t (*Planner)(const fa::VarlenLaunch&, int*, int*);
  Planner plan = nullptr;
  if (d_qk == 64 && d_v == 64) plan = fa::plan_varlen_64_64;
  else if (d_qk == 72 && d_v == 72) plan = fa::plan_varlen_72_72;
  else if (d_qk == 80 && d_v == 80) plan = fa::plan_varlen_80_80;
  else if (d_qk == 96 && d_v == 96) plan = fa::plan_varlen_96_96;
  else if (d_qk == 128 && d_v == 128) plan = fa::plan_varlen_128_128;
  else if (d_qk == 192 && d_v == 128) plan = fa::plan_varlen_192_128;
  if (!plan) return FA_ERR_UNSUPPORTED;
  DeviceInfo* dev = nullptr;
  const fa_status st = device_info(&dev);
  if (st != FA_OK) return st;
  *grid = 0;
  *split = 1;
  const int pack_shift = pack_shift_for(batch, total_q, num_heads, num_heads_k, max_seqlen_q);
  *heads_per_tile = 1 << pack_shift;
  if (total_q == 0) return FA_OK;
  const fa::VarlenLaunch L =
      launch_shape(dev->sm_count, std::min(batch, fa::kMaxBatch), total_q, total_k, num_heads,
                   max_seqlen_k, causal, window_left, window_right, pack_shift);
  return plan(L, grid, split) == cudaSuccess ? FA_OK : FA_ERR_LAUNCH;
}

namespace {

// Work split of a decode call.  Each CTA takes a contiguous range of the
// (token, head group) units' 64-key tiles, at most kDecodeMaxTilesPerCta of
// them.  Either the ranges hold whole units, or they hold equal tile counts
// over whole waves of SMs and the units cut by a range end are merged by a
// second kernel.  The host takes the cut with the fewer tiles on the busiest
// SM, counting the merge as kDecodeMergeCostTiles tiles; the equal-tile cut
// is considered only up to two waves, which bounds its workspace.
struct DecodeSplit {
  long long grid;
  int gran;     // tiles per granule: 1 (equal tiles) or n_tiles (whole units)
  bool split;   // partial results and the merge kernel are needed
};

DecodeSplit decode_split(long long units, int n_tiles, long long sms) {
  auto ceil_div = [](long long x, long long y) { return (x + y - 1) / y; };
  const long long total = units * n_tiles;
  if (n_tiles > fa::kDecodeMaxTilesPerCta) {
    // A unit longer than one CTA's range (top-k above 2048): always the
    // equal-tile cut, over as many waves as it takes.
    DecodeSplit d;
    d.grid = std::min(ceil_div(total, fa::kDecodeMaxTilesPerCta * sms) * sms, total / 2);
    d.gran = 1;
    d.split = true;
    return d;
  }
  // Whole units per CTA.
  const long long upc = fa::kDecodeMaxTilesPerCta / n_tiles;
  const long long grid_u = std::max(ceil_div(units, upc), std::min(units, sms));
  const long long cost_u = ceil_div(grid_u, sms) * ceil_div(units, grid_u) * n_tiles;
  // Equal tile counts, over whole waves of SMs, at least 2 tiles per CTA.
  long long grid_t = ceil_div(total, fa::kDecodeMaxTilesPerCta * sms) * sms;
  grid_t = std::min(grid_t, std::max(1LL, total / 2));
  const bool cuts = units % grid_t != 0;
  const long long cost_t = ceil_div(grid_t, sms) * ceil_div(total, grid_t) +
                           (cuts ? fa::kDecodeMergeCostTiles : 0);
  DecodeSplit d;
  d.split = cuts && cost_t < cost_u && grid_t <= 2 * sms;
  const bool equal = d.split || (!cuts && grid_t <= 2 * sms);
  d.grid = equal ? grid_t : grid_u;
  d.gran = equal ? 1 : n_tiles;
  return d;
}

size_t decode_workspace_bytes(const DecodeSplit& d) {
  return d.split ? (size_t)2 * d.grid * 64 * (fa::kDv + 1) * sizeof(float) : 0;
}

// Everything fa_sparse_mla_decode does before it needs workspace memory:
// argument checks, the Q tensor map, the kernel arguments and the work split
// (see the comment below).  `*launch` is false when there is nothing to run.
struct DecodePlan {
  fa::DecodeArgs a;
  CUtensorMap qmap;
  int np = 64;          // head group width the kernel is instantiated for
  bool launch = false;
  bool split = false;   // partial results and the merge kernel are needed
  size_t o_bytes = 0;   // workspace: partial O, then partial LSE
  size_t l_bytes = 0;
};

fa_status plan_decode(const void* q, const void* kv_cache, const int* page_table,
                      const int* topk_idx, int num_tokens, int num_heads, int topk,
                      int num_pages, int max_pages_per_tok, float softmax_scale, void* out,
                      float* lse, DecodePlan* plan) {
  // q, page_table, topk_idx and out may be null only when there are no tokens.
  if (!kv_cache || (num_tokens > 0 && (!q || !page_table || !topk_idx || !out)))
    return FA_ERR_INVALID_ARG;
  if (num_tokens < 0 || num_pages < 1 || max_pages_per_tok < 1 || topk < 1)
    return FA_ERR_INVALID_ARG;
  if (!(softmax_scale > 0.f) || !std::isfinite(softmax_scale)) return FA_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(kv_cache, 16) || !aligned(out, 16) || !aligned(page_table, 4) ||
      !aligned(topk_idx, 4) || (lse && !aligned(lse, 4)))
    return FA_ERR_INVALID_ARG;
  if (num_heads != 8 && num_heads != 16 && num_heads != 32 && num_heads != 64 &&
      num_heads != 128)
    return FA_ERR_UNSUPPORTED;
  if (topk % 128 != 0 || (int64_t)topk > (int64_t)max_pages_per_tok * fa::kDecodePage)
    return FA_ERR_UNSUPPORTED;
  if ((int64_t)num_pages * fa::kDecodePage > INT32_MAX) return FA_ERR_UNSUPPORTED;
  const int groups = (num_heads + 63) / 64;
  const int n_tiles = topk / fa::kDecodeKeys;
  const long long units = (long long)num_tokens * groups;
  const long long total = units * n_tiles;
  if (total > INT32_MAX) return FA_ERR_UNSUPPORTED;
  DeviceInfo* dev = nullptr;
  fa_status st = device_info(&dev);
  if (st != FA_OK) return st;
  plan->launch = num_tokens > 0;
  if (!plan->launch) return FA_OK;
  // Q viewed as [tokens, heads, 576]; a box covers one token, np heads
  // (heads past num_heads read as zero) and 64 columns.
  const int np = num_heads >= 64 ? 64 : (num_heads <= 16 ? 16 : num_heads);
  plan->np = np;
  {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return FA_ERR_LAUNCH;
    cuuint64_t dims[3] = {576, (cuuint64_t)num_heads, (cuuint64_t)num_tokens};
    cuuint64_t strides[2] = {576 * 2, (cuuint64_t)num_heads * 576 * 2};
    cuuint32_t box[3] = {64u, (cuuint32_t)np, 1u};
    cuuint32_t estr[3] = {1u, 1u, 1u};
    if (fn(&plan->qmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(q), dims, strides,
           box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return FA_ERR_LAUNCH;
  }
  fa::DecodeArgs& a = plan->a;
  a.q = static_cast<const uint16_t*>(q);
  a.cache = static_cast<const uint16_t*>(kv_cache);
  a.page_table = page_table;
  a.topk_idx = topk_idx;
  a.num_tokens = num_tokens;
  a.num_heads = num_heads;
  a.topk = topk;
  a.num_pages = num_pages;
  a.max_pages = max_pages_per_tok;
  a.scale_log2 = softmax_scale * 1.4426950408889634f;
  a.out = static_cast<uint16_t*>(out);
  a.lse = lse;
  a.status = dev->status;
  a.groups = groups;
  a.n_tiles = n_tiles;
  const DecodeSplit sp = decode_split(units, n_tiles, dev->sm_count);
  plan->split = sp.split;
  a.total_tiles = (int)total;
  a.grid = (int)sp.grid;
  a.gran = sp.gran;
  const long long granules = total / a.gran;
  a.range_q = (int)(granules / sp.grid);
  a.range_r = (int)(granules % sp.grid);
  a.part_o = nullptr;
  a.part_lse = nullptr;
  a.wait_limit_ns = g_wait_limit_ns.load(std::memory_order_relaxed);
  if (plan->split) {
    plan->o_bytes = (size_t)2 * sp.grid * 64 * fa::kDv * sizeof(float);
    plan->l_bytes = (size_t)2 * sp.grid * 64 * sizeof(float);
  }
  return FA_OK;
}

// Launches the planned kernels; `ws` holds plan.o_bytes + plan.l_bytes when
// plan.split.
fa_status launch_decode(DecodePlan& plan, void* ws, cudaStream_t stream) {
  if (plan.split) {
    plan.a.part_o = static_cast<float*>(ws);
    plan.a.part_lse = reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + plan.o_bytes);
  }
  const cudaError_t e = plan.np == 64 ? fa::launch_decode_np<64>(plan.qmap, plan.a, stream)
                      : plan.np == 32 ? fa::launch_decode_np<32>(plan.qmap, plan.a, stream)
                                      : fa::launch_decode_np<16>(plan.qmap, plan.a, stream);
  return e == cudaSuccess ? FA_OK : FA_ERR_LAUNCH;
}

}  // namespace

namespace fa {

static_assert(sizeof(DecodePlan) <= kDecodePlanBytes && alignof(DecodePlan) <= 128,
              "decode plan storage");

fa_status decode_plan(const void* q, const void* kv_cache, const int* page_table,
                      const int* topk_idx, int num_tokens, int num_heads, int topk,
                      int num_pages, int max_pages_per_tok, float softmax_scale, void* out,
                      float* lse, void* plan, size_t* workspace_bytes, bool* launch) {
  DecodePlan* p = new (plan) DecodePlan();
  const fa_status st = plan_decode(q, kv_cache, page_table, topk_idx, num_tokens, num_heads, topk,
                                   num_pages, max_pages_per_tok, softmax_scale, out, lse, p);
  *launch = st == FA_OK && p->launch;
  *workspace_bytes = p->split ? p->o_bytes + p->l_bytes : 0;
  return st;
}

fa_status decode_launch(void* plan, void* workspace, cudaStream_t stream) {
  return launch_decode(*static_cast<DecodePlan*>(plan), workspace, stream);
}

}  // namespace fa

extern "C" fa_status fa_sparse_mla_decode(const void* q, const void* kv_cache,
                                          const int* page_table, const int* topk_idx,
                                          int num_tokens, int num_heads, int topk,
                                          int num_pages, int max_pages_per_tok,
                                          float softmax_scale, void* out, float* lse,
                                          fa_stream_t stream) {
  DecodePlan plan;
  fa_status st = plan_decode(q, kv_cache, page_table, topk_idx, num_tokens, num_heads, topk,
                             num_pages, max_pages_per_tok, softmax_scale, out, lse, &plan);
  if (st != FA_OK || !plan.launch) return st;
  cudaStream_t st_ = reinterpret_cast<cudaStream_t>(stream);
  void* ws = nullptr;
  if (plan.split) {
    st = stream_workspace(st_, plan.o_bytes + plan.l_bytes, &ws);
    if (st != FA_OK) return st;
  }
  return launch_decode(plan, ws, st_);
}

extern "C" fa_status fa_sparse_mla_decode_plan(int num_tokens, int num_heads, int topk,
                                               int* launches, size_t* workspace_bytes) {
  if (!launches || !workspace_bytes || num_tokens < 0 || topk < 1) return FA_ERR_INVALID_ARG;
  if (num_heads != 8 && num_heads != 16 && num_heads != 32 && num_heads != 64 &&
      num_heads != 128)
    return FA_ERR_UNSUPPORTED;
  if (topk % 128 != 0) return FA_ERR_UNSUPPORTED;
  const int groups = (num_heads + 63) / 64;
  const int n_tiles = topk / fa::kDecodeKeys;
  const long long units = (long long)num_tokens * groups;
  if (units * n_tiles > INT32_MAX) return FA_ERR_UNSUPPORTED;
  DeviceInfo* dev = nullptr;
  const fa_status st = device_info(&dev);
  if (st != FA_OK) return st;
  *launches = 0;
  *workspace_bytes = 0;
  if (num_tokens == 0) return FA_OK;
  const DecodeSplit d = decode_split(units, n_tiles, dev->sm_count);
  *launches = d.split && d.grid >= 2 ? 2 : 1;
  *workspace_bytes = decode_workspace_bytes(d);
  return FA_OK;
}

extern "C" fa_status fa_merge_attn_states(void* out, float* out_lse, const void* prefix_out,
                                          const float* prefix_lse, const void* suffix_out,
                                          const float* suffix_lse, int total_q, int num_heads,
                                          int head_dim, fa_stream_t stream) {
  if (!out || !prefix_out || !prefix_lse || !suffix_out || !suffix_lse) return FA_ERR_INVALID_ARG;
  if (total_q < 0 || num_heads < 1 || head_dim < 8 || head_dim % 8 != 0) return FA_ERR_INVALID_ARG;
  if (!aligned(out, 16) || !aligned(prefix_out, 16) || !aligned(suffix_out, 16) ||
      !aligned(prefix_lse, 4) || !aligned(suffix_lse, 4) || (out_lse && !aligned(out_lse, 4)))
    return FA_ERR_INVALID_ARG;
  if ((int64_t)total_q * num_heads > INT32_MAX) return FA_ERR_UNSUPPORTED;
  DeviceInfo* dev = nullptr;
  fa_status st = device_info(&dev);
  if (st != FA_OK) return st;
  if (total_q == 0) return FA_OK;
  fa::MergeArgs a;
  a.oa = static_cast<const uint16_t*>(prefix_out);
  a.la = prefix_lse;
  a.ob = static_cast<const uint16_t*>(suffix_out);
  a.lb = suffix_lse;
  a.out = static_cast<uint16_t*>(out);
  a.lse = out_lse;
  a.total_q = total_q;
  a.num_heads = num_heads;
  a.head_dim = head_dim;
  cudaError_t e = fa::launch_merge(a, dev->sm_count, reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? FA_OK : FA_ERR_LAUNCH;
}

extern "C" fa_status fa_get_device_status(void) {
  DeviceInfo* dev = nullptr;
  fa_status st = device_info(&dev);
  if (st != FA_OK) return st;
  if (cudaDeviceSynchronize() != cudaSuccess) return FA_ERR_LAUNCH;
  unsigned int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_fa_status, sizeof v) != cudaSuccess) return FA_ERR_LAUNCH;
  const unsigned int zero = 0;
  if (cudaMemcpyToSymbol(g_fa_status, &zero, sizeof zero) != cudaSuccess) return FA_ERR_LAUNCH;
  return (v & fa::kStatusTimeout) ? FA_ERR_DEVICE_TIMEOUT : FA_OK;
}

extern "C" fa_status fa_set_wait_limit_ns(unsigned long long ns) {
  g_wait_limit_ns.store(ns == 0 ? fa::kWaitLimitNs : ns, std::memory_order_relaxed);
  return FA_OK;
}

extern "C" const char* fa_status_string(fa_status s) {
  switch (s) {
    case FA_OK: return "ok";
    case FA_ERR_INVALID_ARG: return "invalid argument";
    case FA_ERR_UNSUPPORTED: return "unsupported configuration";
    case FA_ERR_ARCH: return "device is not sm_103 (GB300)";
    case FA_ERR_LAUNCH: return "CUDA launch or driver call failed";
    case FA_ERR_DEVICE_TIMEOUT: return "a kernel pipeline wait timed out";
    case FA_ERR_SCRATCH:
      return "the call needs more partial-result scratch than fa_sparse_mla_decode_noalloc's "
             "fixed buffer holds";
  }
  return "unknown status";
}
