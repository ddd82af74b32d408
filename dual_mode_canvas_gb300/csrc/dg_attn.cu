// Host side of the dg_attn C ABI (see include/dg_attn.h): argument checks,
// TMA tensor maps, workspace layout, kernel launches and the device status word.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include <nvtx3/nvToolsExt.h>

#include "dg_attn.h"
#include "kernels.cuh"
#include "acceptance.cuh"
#include "selfcond.cuh"

namespace dg {

__device__ int g_status;  // first device-side error since the last dg_attn_status()

// Scratch of dg_attn_forward_noalloc.  Host code must not use this name as an
// address: it reaches the kernels only through the device address looked up
// once per device (DeviceInfo::noalloc_scratch).
static __device__ __align__(256) uint8_t g_noalloc_scratch[DG_ATTN_NOALLOC_SCRATCH_BYTES];

namespace {

constexpr int kMaxDevices = 64;
constexpr int kVersion = 100;  // 0.1.0

struct DeviceInfo {
  bool ready = false;
  int num_sms = 0;
  int cc_major = 0, cc_minor = 0;
  int* status = nullptr;   // device address of g_status
  void* noalloc_scratch = nullptr;  // device address of g_noalloc_scratch
};

std::mutex g_mutex;

// An NVTX range around each C-ABI call (header-only NVTX: free unless a
// profiler is attached).
struct NvtxRange {
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
  NvtxRange(const NvtxRange&) = delete;
  NvtxRange& operator=(const NvtxRange&) = delete;
};
DeviceInfo g_dev[kMaxDevices];
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

// Per-head_dim kernel shapes: KV tile rows BN, K-ring and V-ring stages
// (shared memory holds the rings, up to 224 KB, and with QS the query tile),
// S/P buffers NS in TMEM (O, NS buffers of BN columns and, without QS, Q).
// - head_dim 64 has TMEM room for three buffers (64 + 3 x 128 + 32 columns),
//   so QK^T runs two tiles ahead of P.V.
// - bf16 head_dim 128 / 256 keep two: 96-key tiles with three buffers were
//   slower at head_dim 128 (max mix 0.902 vs 0.840 ms per call), and so was the
//   query tile in shared memory with three 128-key buffers (0.827 vs 0.820 ms;
//   at head_dim 256 the 64 KB query tile leaves five ring stages: denoise loop
//   0.198 vs 0.172 ms).
// - e4m3 tiles are half the bytes, so the same rings hold more stages.
//   head_dim 128 moves its query tile to shared memory for three buffers (max
//   mix 0.691 vs 0.698 ms).  head_dim 256 moves it there for 128-key tiles with
//   two buffers (256 + 2 x 128 columns; 3 K + 3 V stages of 32 KB and the 32 KB
//   query tile): denoise loop 0.116 vs 0.134 ms with 64-key tiles and three
//   buffers (which had beaten two 64-key buffers, 0.137 vs 0.145 ms); rings of
//   4 + 2 or 2 + 4 stages time the same.
template <int D, bool F8 = false> struct Shape;
template <> struct Shape<64> { static constexpr int BN = 128, NK = 6, NV = 6, NS = 3; static constexpr bool QS = false; };
template <> struct Shape<128> { static constexpr int BN = 128, NK = 4, NV = 3, NS = 2; static constexpr bool QS = false; };
template <> struct Shape<256> { static constexpr int BN = 64, NK = 4, NV = 3, NS = 2; static constexpr bool QS = false; };
template <> struct Shape<128, true> { static constexpr int BN = 128, NK = 6, NV = 6, NS = 3; static constexpr bool QS = true; };
template <> struct Shape<256, true> { static constexpr int BN = 128, NK = 3, NV = 3, NS = 2; static constexpr bool QS = true; };

int kv_tile_rows(int D, bool f8 = false) {
  if (f8) return D == 128 ? Shape<128, true>::BN : Shape<256, true>::BN;
  return D == 64 ? Shape<64>::BN : D == 128 ? Shape<128>::BN : Shape<256>::BN;
}

template <int D, bool F8 = false>
cudaError_t set_kernel_attrs() {
  using S = Shape<D, F8>;
  using C = FwdCfg<D, S::BN, S::NK, S::NV, F8, S::NS, S::QS>;
  return cudaFuncSetAttribute(fwd_kernel<D, S::BN, S::NK, S::NV, F8, S::NS, S::QS>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
}

cudaError_t set_sc_attrs() {
  return cudaFuncSetAttribute(sc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, ScCfg::SMEM_BYTES);
}

// One-time per-device setup (SM count, architecture, kernel attributes,
// status word address).  Returns DG_OK or an error code.
dg_status_t device_info(DeviceInfo** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return DG_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return DG_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_mutex);
  DeviceInfo& di = g_dev[dev];
  if (!di.ready) {
    cudaDeviceProp prop;
    if (cudaGetDeviceProperties(&prop, dev) != cudaSuccess) return DG_ERR_CUDA;
    di.num_sms = prop.multiProcessorCount;
    di.cc_major = prop.major;
    di.cc_minor = prop.minor;
    if (!(di.cc_major == 10 && di.cc_minor == 3)) return DG_ERR_UNSUPPORTED;
    if (!g_encode) {
      void* fn = nullptr;
      cudaDriverEntryPointQueryResult q;
      if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                           &q) != cudaSuccess ||
          q != cudaDriverEntryPointSuccess || fn == nullptr)
        return DG_ERR_CUDA;
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
    if (set_kernel_attrs<64>() != cudaSuccess || set_kernel_attrs<128>() != cudaSuccess ||
        set_kernel_attrs<256>() != cudaSuccess || set_kernel_attrs<128, true>() != cudaSuccess ||
        set_kernel_attrs<256, true>() != cudaSuccess || set_sc_attrs() != cudaSuccess)
      return DG_ERR_CUDA;
    void* sym = nullptr;
    if (cudaGetSymbolAddress(&sym, g_status) != cudaSuccess) return DG_ERR_CUDA;
    di.status = static_cast<int*>(sym);
    void* scratch = nullptr;
    if (cudaGetSymbolAddress(&scratch, g_noalloc_scratch) != cudaSuccess || scratch == nullptr)
      return DG_ERR_CUDA;
    di.noalloc_scratch = scratch;
    if (cudaMemset(di.status, 0, sizeof(int)) != cudaSuccess) return DG_ERR_CUDA;
    di.ready = true;
  }
  *out = &di;
  return DG_OK;
}

// Each query tile's KV tiles are visited in the rotated order that lines up
// the CTAs streaming the same KV (DG_ATTN_KV_ORDER=linear: ascending order).
bool rotate_kv_order() {
  const char* e = std::getenv("DG_ATTN_KV_ORDER");
  return !(e && std::strcmp(e, "linear") == 0);
}

// Persistent grid: one CTA per SM (DG_ATTN_NUM_CTAS caps the number of CTAs,
// for tests of the split-KV path).
int num_ctas_for(const DeviceInfo& di) {
  int n = std::min(di.num_sms, kMaxCtas);
  if (const char* e = std::getenv("DG_ATTN_NUM_CTAS")) {
    const int v = std::max(1, std::atoi(e));
    if (v < n) n = v;
  }
  return n;
}

inline size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

struct Layout {
  size_t hdr, seq_tile, seq_kv, tiles, unit_begin, part_lse, part_o, total;
  int max_tiles;
  bool local;  // at most kLocalMaxTiles tiles: one copy of the tile tables per CTA
};

Layout make_layout(int B, int total_q, int Hq, int Hkv, int D, int num_sms) {
  const int G = Hq / Hkv;
  const int TT = kRows / G;
  Layout l;
  const int64_t mt = (static_cast<int64_t>(total_q) + TT - 1) / TT + B;
  l.max_tiles = static_cast<int>(static_cast<int64_t>(Hkv) * mt);
  // small batches: every CTA of the attention grid builds the work list into
  // its own copy of the tables
  l.local = l.max_tiles <= kLocalMaxTiles;
  const size_t copies = l.local ? static_cast<size_t>(num_sms) : 1;
  size_t off = 0;
  l.hdr = off;        off = align256(off + sizeof(WorkHeader));
  l.seq_tile = off;   off = align256(off + sizeof(int64_t) * (B + 1));
  l.seq_kv = off;     off = align256(off + sizeof(int64_t) * (B + 1));
  l.tiles = off;      off = align256(off + sizeof(TileDesc) * static_cast<size_t>(l.max_tiles) * copies);
  l.unit_begin = off; off = align256(off + sizeof(int64_t) * (static_cast<size_t>(l.max_tiles) + 1) * copies);
  l.part_lse = off;   off = align256(off + sizeof(float) * 2 * static_cast<size_t>(num_sms) * kRows);
  l.part_o = off;     off = align256(off + sizeof(float) * 2 * static_cast<size_t>(num_sms) * kRows * D);
  l.total = off;
  return l;
}

bool sizes_ok(int B, int total_q, int Hq, int Hkv, int D) {
  if (B < 0 || total_q < 0 || Hq <= 0 || Hkv <= 0) return false;
  if (Hq % Hkv != 0 || Hq / Hkv > kRows) return false;
  if (D != 64 && D != 128 && D != 256) return false;
  return true;
}

// [rows, heads, D] tensor map of bf16 (or, with e4m3, of bytes), box {one
// 128-byte block of D, box_heads, box_rows}, 128-byte swizzle.
dg_status_t encode_map(CUtensorMap* map, const void* base, int rows, int heads, int D,
                       int box_heads, int box_rows, bool e4m3 = false) {
  const cuuint64_t es = e4m3 ? 1 : 2;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(heads),
                              static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(D) * es,
                                 static_cast<cuuint64_t>(heads) * D * es};
  const cuuint32_t box[3] = {static_cast<cuuint32_t>(128 / es), static_cast<cuuint32_t>(box_heads),
                             static_cast<cuuint32_t>(box_rows)};
  const cuuint32_t estr[3] = {1u, 1u, 1u};
  const CUresult r = g_encode(map, e4m3 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                              3, const_cast<void*>(base), dims,
                              strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? DG_OK : DG_ERR_INVALID_ARG;
}

// The paged V pool as a 4-D map {128-byte block of D, heads, rows, column
// blocks of D} (the last stride, 128 bytes, is the smallest: it walks the
// column blocks of one row), box {one block, one head, box_rows, every column
// block}: one box is a whole page of one head, landing as [column block][row].
dg_status_t encode_page_map(CUtensorMap* map, const void* base, int rows, int heads, int D, int box_rows,
                            bool e4m3) {
  const cuuint64_t es = e4m3 ? 1 : 2;
  const cuuint64_t nkb = static_cast<cuuint64_t>(D) * es / 128;
  const cuuint64_t dims[4] = {128 / es, static_cast<cuuint64_t>(heads), static_cast<cuuint64_t>(rows), nkb};
  const cuuint64_t strides[3] = {static_cast<cuuint64_t>(D) * es, static_cast<cuuint64_t>(heads) * D * es, 128};
  const cuuint32_t box[4] = {static_cast<cuuint32_t>(128 / es), 1u, static_cast<cuuint32_t>(box_rows),
                             static_cast<cuuint32_t>(nkb)};
  const cuuint32_t estr[4] = {1u, 1u, 1u, 1u};
  const CUresult r = g_encode(map, e4m3 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                              4, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? DG_OK : DG_ERR_INVALID_ARG;
}

template <int D, bool F8 = false>
dg_status_t launch(const CUtensorMap& mk, const CUtensorMap& mv,
                   const FwdParams& p, int num_ctas, int max_tiles, cudaStream_t stream,
                   cudaEvent_t ev_begin, cudaEvent_t ev_end) {
  using S = Shape<D, F8>;
  using C = FwdCfg<D, S::BN, S::NK, S::NV, F8, S::NS, S::QS>;
  if (ev_begin && cudaEventRecord(ev_begin, stream) != cudaSuccess) return DG_ERR_CUDA;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(num_ctas);
  cfg.blockDim = dim3(p.k_split ? kThreads : kThreads - 32);  // warp 7 only with k_split
  cfg.dynamicSmemBytes = C::SMEM_BYTES;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  // programmatic dependent of the work-list grid (the kernel waits for it)
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, fwd_kernel<D, S::BN, S::NK, S::NV, F8, S::NS, S::QS>, mk, mv, p) != cudaSuccess)
    return DG_ERR_CUDA;
  if (ev_end && cudaEventRecord(ev_end, stream) != cudaSuccess) return DG_ERR_CUDA;
  // the merge is a programmatic dependent of the attention grid (it waits
  // for it before reading the partials)
  cudaLaunchConfig_t ccfg = {};
  ccfg.gridDim = dim3(max_tiles, (kRows + kCombineWarps - 1) / kCombineWarps);
  ccfg.blockDim = dim3(kCombineWarps * 32);
  ccfg.stream = stream;
  cudaLaunchAttribute cattr[1];
  cattr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  cattr[0].val.programmaticStreamSerializationAllowed = 1;
  ccfg.attrs = cattr;
  ccfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&ccfg, combine_kernel<D>, p) != cudaSuccess) return DG_ERR_CUDA;
  return DG_OK;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

}  // namespace
}  // namespace dg

using namespace dg;

namespace {
// The attention grid builds the work list itself (no work-list grid) for
// contiguous K/V batches whose tile bound fits the per-CTA tables, but not in
// the e4m3 head_dim-128 shape, whose kernel reads the work-list grid's tables
// directly; DG_ATTN_FUSED_WL=0 keeps the separate grid everywhere.
bool fused_work_list(bool paged, bool f8, int head_dim, const Layout& lay) {
  const char* e = std::getenv("DG_ATTN_FUSED_WL");
  return !paged && lay.local && !(f8 && head_dim == 128) && !(e && std::strcmp(e, "0") == 0);
}
}  // namespace

extern "C" int32_t dg_attn_launches_per_call(int32_t num_seqs, int32_t total_q, int32_t num_q_heads,
                                             int32_t num_kv_heads, int32_t head_dim, int32_t paged,
                                             int32_t e4m3) {
  if (!sizes_ok(num_seqs, total_q, num_q_heads, num_kv_heads, head_dim)) return 0;
  // (the layout's tile bound does not depend on the SM count)
  const Layout lay = make_layout(num_seqs, total_q, num_q_heads, num_kv_heads, head_dim, 1);
  return fused_work_list(paged != 0, e4m3 != 0, head_dim, lay) ? 2 : 3;
}

extern "C" size_t dg_attn_workspace_size(int32_t num_seqs, int32_t total_q, int32_t num_q_heads,
                                         int32_t num_kv_heads, int32_t head_dim) {
  if (!sizes_ok(num_seqs, total_q, num_q_heads, num_kv_heads, head_dim)) return 0;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return make_layout(num_seqs, total_q, num_q_heads, num_kv_heads, head_dim, sms).total;
}

namespace {
// The host-visible argument checks of a forward call (everything but the
// workspace).  *nothing_to_do is set when the call is valid and has no work
// (no sequences or no query tokens).
dg_status_t check_args(const void* q, const void* k, const void* v, const int32_t* cu_q,
                       const int32_t* ctx_len, const uint8_t* mode, int32_t num_seqs,
                       int32_t total_q, int32_t total_kv, int32_t num_q_heads, int32_t num_kv_heads,
                       int32_t head_dim, int32_t window, float scale, const void* out,
                       const float* lse, bool paged, bool f8, bool* nothing_to_do) {
  *nothing_to_do = false;
  if (f8 && (head_dim == 64 || paged)) return DG_ERR_UNSUPPORTED;
  if (!sizes_ok(num_seqs, total_q, num_q_heads, num_kv_heads, head_dim))
    return (num_q_heads > 0 && num_kv_heads > 0 && num_q_heads % num_kv_heads == 0 &&
            num_q_heads / num_kv_heads > kRows) || (head_dim > 0 && head_dim != 64 &&
            head_dim != 128 && head_dim != 256 && head_dim % 8 == 0)
               ? DG_ERR_UNSUPPORTED
               : DG_ERR_INVALID_ARG;
  if (window < -1 || total_kv < 0 || !(scale > 0.f) || !std::isfinite(scale)) return DG_ERR_INVALID_ARG;
  if (num_seqs == 0 || total_q == 0) {
    *nothing_to_do = true;
    return num_seqs == 0 && total_q != 0 ? DG_ERR_INVALID_ARG : DG_OK;
  }
  if (!paged && total_kv < total_q) return DG_ERR_INVALID_ARG;
  if (!paged && (!k || !v || !aligned(k, 16) || !aligned(v, 16))) return DG_ERR_INVALID_ARG;
  if (!q || !cu_q || !ctx_len || !mode || !out) return DG_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(out, 16) ||
      !aligned(cu_q, 4) || !aligned(ctx_len, 4) || (lse && !aligned(lse, 4)))
    return DG_ERR_INVALID_ARG;
  return DG_OK;
}

// `pg` null: contiguous K/V (k, v, total_kv); otherwise the paged cache it
// describes (k, v unused).
dg_status_t forward_impl(const void* q, const void* k, const void* v, const int32_t* cu_q,
                         const int32_t* ctx_len, const uint8_t* mode, int32_t num_seqs,
                         int32_t total_q, int32_t total_kv, int32_t num_q_heads,
                         int32_t num_kv_heads, int32_t head_dim, int32_t window, float scale,
                         void* out, float* lse, void* workspace, size_t workspace_bytes,
                         void* stream_ptr, void* ev_begin, void* ev_end,
                         const PagedArgs* pg = nullptr, const float* e4m3_scales = nullptr) {
  // e4m3_scales = {q, k, v} scales: Q, K, V are e4m3 bytes (contiguous layout only)
  const bool f8 = e4m3_scales != nullptr;
  bool nothing_to_do = false;
  const dg_status_t chk = check_args(q, k, v, cu_q, ctx_len, mode, num_seqs, total_q, total_kv,
                                     num_q_heads, num_kv_heads, head_dim, window, scale, out, lse,
                                     pg != nullptr, f8, &nothing_to_do);
  if (chk != DG_OK || nothing_to_do) return chk;

  DeviceInfo* di = nullptr;
  const dg_status_t st = device_info(&di);
  if (st != DG_OK) return st;
  const Layout lay = make_layout(num_seqs, total_q, num_q_heads, num_kv_heads, head_dim, di->num_sms);
  if (!workspace || !aligned(workspace, 256) || workspace_bytes < lay.total) return DG_ERR_WORKSPACE;

  const int G = num_q_heads / num_kv_heads;
  const int TT = kRows / G;
  const int BN = kv_tile_rows(head_dim, f8);
  CUtensorMap mk, mv;
  // K/V tiles of BN rows; from a paged cache in boxes of at most one page
  // that divide the tile (pages and tiles start on multiples of the box)
  int box = BN;
  if (pg) {
    box = 1;
    while (box * 2 <= (1 << pg->page_shift) && BN % (box * 2) == 0) box *= 2;
  }
  const void* kmap = pg ? pg->k_cache : k;
  const void* vmap = pg ? pg->v_cache : v;
  const int map_rows = pg ? (pg->num_pages << pg->page_shift) : total_kv;
  // V pages of one MMA K step or half of one, and head_dim over several
  // 128-byte blocks: one box per page (DG_ATTN_V_PAGE_BOX=0 keeps a box per
  // block)
  const int kstep = f8 ? 32 : 16;
  const int nkb = head_dim * (f8 ? 1 : 2) / 128;
  const char* vpb_env = std::getenv("DG_ATTN_V_PAGE_BOX");
  const bool v_page_box = pg && (box == kstep || 2 * box == kstep) && box < BN && nkb > 1 &&
                          !(vpb_env && std::strcmp(vpb_env, "0") == 0);
  // K pages of 8 rows: one box per page as well (DG_ATTN_K_PAGE_BOX=0 keeps a
  // box per block)
  const char* kpb_env = std::getenv("DG_ATTN_K_PAGE_BOX");
  const bool k_page_box = pg && !f8 && box == 8 && box < BN && nkb > 1 &&
                          !(kpb_env && std::strcmp(kpb_env, "0") == 0);
  if ((k_page_box ? encode_page_map(&mk, kmap, map_rows, num_kv_heads, head_dim, box, f8)
                  : encode_map(&mk, kmap, map_rows, num_kv_heads, head_dim, 1, box, f8)) != DG_OK ||
      (v_page_box ? encode_page_map(&mv, vmap, map_rows, num_kv_heads, head_dim, box, f8)
                  : encode_map(&mv, vmap, map_rows, num_kv_heads, head_dim, 1, box, f8)) != DG_OK)
    return DG_ERR_INVALID_ARG;

  uint8_t* w = static_cast<uint8_t*>(workspace);
  FwdParams p;
  p.ws.hdr = reinterpret_cast<WorkHeader*>(w + lay.hdr);
  p.ws.seq_tile_off = reinterpret_cast<int64_t*>(w + lay.seq_tile);
  p.ws.seq_kv_off = reinterpret_cast<int64_t*>(w + lay.seq_kv);
  p.ws.tiles = reinterpret_cast<TileDesc*>(w + lay.tiles);
  p.ws.unit_begin = reinterpret_cast<int64_t*>(w + lay.unit_begin);
  p.ws.part_lse = reinterpret_cast<float*>(w + lay.part_lse);
  p.ws.part_o = reinterpret_cast<float*>(w + lay.part_o);
  p.q = q;
  p.out = static_cast<__nv_bfloat16*>(out);
  p.lse = lse;
  p.status = di->status;
  p.Hq = num_q_heads;
  p.G = G;
  p.TT = TT;
  p.window = window;
  p.block_table = pg ? pg->block_table : nullptr;
  p.page_shift = pg ? pg->page_shift : 0;
  p.page_box = box;
  p.v_page_box = v_page_box ? 1 : 0;
  p.k_page_box = k_page_box ? 1 : 0;
  // a K tile of 8 or more boxes: two warps issue them (DG_ATTN_K_SPLIT=0: one)
  const char* ks_env = std::getenv("DG_ATTN_K_SPLIT");
  const int k_boxes = k_page_box ? BN / box : (BN / box) * nkb;
  p.k_split = (k_boxes >= 8 && !(ks_env && std::strcmp(ks_env, "0") == 0)) ? 1 : 0;
  // segment weight in KV-tile units: a segment (Q load, pipeline fill,
  // epilogue) costs about the same time at every head_dim, a 64-key tile of
  // head_dim 256 less than a 128-key one.  Measured optima: 18 for 64-key
  // tiles (bf16 denoise loop 0.1698 vs 0.1732 ms at 8), 8 for 128-key tiles
  // of head_dim 128 (mixed batch 43.3 us; 4 / 14: 46.3 / 45.1 us), 12 for the
  // e4m3 128-key tiles of head_dim 256 (denoise loop 0.1155 ms; 5 / 8 / 18:
  // 0.1183 / 0.1165 / 0.1160 ms).
  // DG_ATTN_SEG_WEIGHT overrides it.
  p.seg_weight = BN == 64 ? 18 : (head_dim == 256 ? 12 : 8);
  if (const char* e = std::getenv("DG_ATTN_SEG_WEIGHT")) p.seg_weight = std::max(0, std::atoi(e));
  p.debug_skip_k_load = -1;
  if (const char* e = std::getenv("DG_ATTN_DEBUG_SKIP_K_LOAD")) p.debug_skip_k_load = std::atoi(e);
  p.Hkv = num_kv_heads;
  p.kv_rows = map_rows;
  p.total_q = total_q;
  p.bt_entries = pg ? static_cast<int64_t>(num_seqs) * pg->bt_stride : 0;
  p.debug_bad_kv_row = -1;
#ifdef DG_ATTN_DEBUG
  if (const char* e = std::getenv("DG_ATTN_DEBUG_BAD_KV_ROW")) p.debug_bad_kv_row = std::atoi(e);
#endif
  // e4m3: the q and k scales multiply every score, the v scale the output
  const float s_eff = f8 ? scale * e4m3_scales[0] * e4m3_scales[1] : scale;
  p.scale = s_eff;
  p.scale_log2 = s_eff * 1.4426950408889634f;
  p.v_scale = f8 ? e4m3_scales[2] : 1.f;

  cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
  PagedArgs pa = {};
  int append_ctas = 0;
  if (pg) {
    pa = *pg;
    if (pa.k_new) {
      const int64_t units = 2ll * total_q * num_kv_heads * head_dim / 8;
      append_ctas = static_cast<int>(std::min<int64_t>((units + 1023) / 1024, 2ll * di->num_sms));
    }
  }
  const int num_ctas = num_ctas_for(*di);
  p.num_slots = 2 * num_ctas;
  // Small batches with contiguous K/V have no work-list grid: every CTA of
  // the attention grid builds the list for itself (measured: the work-list
  // grid's launch and run cost a denoise step ~5 us on the critical path).
  p.fused_wl = fused_work_list(pg != nullptr, f8, head_dim, lay) ? 1 : 0;
  p.cu_q = cu_q;
  p.ctx_len = ctx_len;
  p.mode = mode;
  p.B = num_seqs;
  p.max_tiles = lay.max_tiles;
  p.tiles_stride = p.fused_wl ? lay.max_tiles : 0;
  p.ub_stride = p.fused_wl ? lay.max_tiles + 1 : 0;
  p.rotate = rotate_kv_order() ? 1 : 0;
  p.kv_total = pg ? 0 : total_kv;
  // a programmatic dependent of the stream's previous kernel (it waits for
  // that grid before reading anything), so in a loop of calls its launch
  // overlaps the previous call's merge
  cudaLaunchConfig_t wcfg = {};
  wcfg.gridDim = dim3(1 + append_ctas);
  wcfg.blockDim = dim3(1024);
  wcfg.stream = stream;
  cudaLaunchAttribute wattr[1];
  wattr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  wattr[0].val.programmaticStreamSerializationAllowed = 1;
  wcfg.attrs = wattr;
  wcfg.numAttrs = 1;
  if (!p.fused_wl &&
      cudaLaunchKernelEx(&wcfg, build_worklist_kernel, cu_q, ctx_len, mode, num_seqs, total_q,
                         pg ? INT32_MAX : total_kv, num_kv_heads, TT, BN, window, lay.max_tiles, num_ctas,
                         p.rotate, p.seg_weight, p.ws, pa, p.status) != cudaSuccess)
    return DG_ERR_CUDA;
  cudaEvent_t e0 = static_cast<cudaEvent_t>(ev_begin), e1 = static_cast<cudaEvent_t>(ev_end);
  if (f8) {
    if (head_dim == 128) return launch<128, true>(mk, mv, p, num_ctas, lay.max_tiles, stream, e0, e1);
    return launch<256, true>(mk, mv, p, num_ctas, lay.max_tiles, stream, e0, e1);
  }
  switch (head_dim) {
    case 64: return launch<64>(mk, mv, p, num_ctas, lay.max_tiles, stream, e0, e1);
    case 128: return launch<128>(mk, mv, p, num_ctas, lay.max_tiles, stream, e0, e1);
    default: return launch<256>(mk, mv, p, num_ctas, lay.max_tiles, stream, e0, e1);
  }
}
}  // namespace

extern "C" dg_status_t dg_attn_forward(const void* q, const void* k, const void* v,
                                       const int32_t* cu_q, const int32_t* ctx_len,
                                       const uint8_t* mode, int32_t num_seqs, int32_t total_q,
                                       int32_t total_kv, int32_t num_q_heads, int32_t num_kv_heads,
                                       int32_t head_dim, int32_t window, float scale, void* out,
                                       float* lse, void* workspace, size_t workspace_bytes,
                                       void* stream) {
  NvtxRange nvtx("dg_attn_forward");
  return forward_impl(q, k, v, cu_q, ctx_len, mode, num_seqs, total_q, total_kv, num_q_heads,
                      num_kv_heads, head_dim, window, scale, out, lse, workspace, workspace_bytes,
                      stream, nullptr, nullptr);
}

extern "C" dg_status_t dg_attn_forward_profiled(
    const void* q, const void* k, const void* v, const int32_t* cu_q, const int32_t* ctx_len,
    const uint8_t* mode, int32_t num_seqs, int32_t total_q, int32_t total_kv, int32_t num_q_heads,
    int32_t num_kv_heads, int32_t head_dim, int32_t window, float scale, void* out, float* lse,
    void* workspace, size_t workspace_bytes, void* stream, void* attn_begin_event,
    void* attn_end_event) {
  NvtxRange nvtx("dg_attn_forward_profiled");
  return forward_impl(q, k, v, cu_q, ctx_len, mode, num_seqs, total_q, total_kv, num_q_heads,
                      num_kv_heads, head_dim, window, scale, out, lse, workspace, workspace_bytes,
                      stream, attn_begin_event, attn_end_event);
}

// For callers that cannot allocate device memory (see the header): the same
// forward pass, with the workspace taken from the library's static scratch.
extern "C" dg_status_t dg_attn_forward_noalloc(const void* q, const void* k, const void* v,
                                               const int32_t* cu_q, const int32_t* ctx_len,
                                               const uint8_t* mode, int32_t num_seqs,
                                               int32_t total_q, int32_t total_kv,
                                               int32_t num_q_heads, int32_t num_kv_heads,
                                               int32_t head_dim, int32_t window, float scale,
                                               void* out, float* lse, void* stream) {
  NvtxRange nvtx("dg_attn_forward_noalloc");
  // the same argument checks as dg_attn_forward first, so a bad argument
  // reports DG_ERR_INVALID_ARG / DG_ERR_UNSUPPORTED whatever the sizes
  bool nothing_to_do = false;
  const dg_status_t chk = check_args(q, k, v, cu_q, ctx_len, mode, num_seqs, total_q, total_kv,
                                     num_q_heads, num_kv_heads, head_dim, window, scale, out, lse,
                                     false, false, &nothing_to_do);
  if (chk != DG_OK || nothing_to_do) return chk;
  DeviceInfo* di = nullptr;
  const dg_status_t st = device_info(&di);
  if (st != DG_OK) return st;
  const Layout lay = make_layout(num_seqs, total_q, num_q_heads, num_kv_heads, head_dim, di->num_sms);
  if (lay.total > DG_ATTN_NOALLOC_SCRATCH_BYTES) return DG_ERR_WORKSPACE;
  return forward_impl(q, k, v, cu_q, ctx_len, mode, num_seqs, total_q, total_kv, num_q_heads,
                      num_kv_heads, head_dim, window, scale, out, lse, di->noalloc_scratch,
                      DG_ATTN_NOALLOC_SCRATCH_BYTES, stream, nullptr, nullptr);
}

namespace {
dg_status_t forward_fp8(const void* q, const void* k, const void* v, const int32_t* cu_q,
                        const int32_t* ctx_len, const uint8_t* mode, int32_t num_seqs,
                        int32_t total_q, int32_t total_kv, int32_t num_q_heads, int32_t num_kv_heads,
                        int32_t head_dim, int32_t window, float scale, float q_scale, float k_scale,
                        float v_scale, void* out, float* lse, void* workspace,
                        size_t workspace_bytes, void* stream, void* ev_begin, void* ev_end) {
  if (!(q_scale > 0.f) || !(k_scale > 0.f) || !(v_scale > 0.f) || !std::isfinite(q_scale) ||
      !std::isfinite(k_scale) || !std::isfinite(v_scale))
    return DG_ERR_INVALID_ARG;
  const float sc[3] = {q_scale, k_scale, v_scale};
  return forward_impl(q, k, v, cu_q, ctx_len, mode, num_seqs, total_q, total_kv, num_q_heads,
                      num_kv_heads, head_dim, window, scale, out, lse, workspace, workspace_bytes,
                      stream, ev_begin, ev_end, nullptr, sc);
}
}  // namespace

extern "C" dg_status_t dg_attn_forward_fp8(const void* q, const void* k, const void* v,
                                           const int32_t* cu_q, const int32_t* ctx_len,
                                           const uint8_t* mode, int32_t num_seqs, int32_t total_q,
                                           int32_t total_kv, int32_t num_q_heads,
                                           int32_t num_kv_heads, int32_t head_dim, int32_t window,
                                           float scale, float q_scale, float k_scale, float v_scale,
                                           void* out, float* lse, void* workspace,
                                           size_t workspace_bytes, void* stream) {
  NvtxRange nvtx("dg_attn_forward_fp8");
  return forward_fp8(q, k, v, cu_q, ctx_len, mode, num_seqs, total_q, total_kv, num_q_heads,
                     num_kv_heads, head_dim, window, scale, q_scale, k_scale, v_scale, out, lse,
                     workspace, workspace_bytes, stream, nullptr, nullptr);
}

extern "C" dg_status_t dg_attn_forward_fp8_profiled(
    const void* q, const void* k, const void* v, const int32_t* cu_q, const int32_t* ctx_len,
    const uint8_t* mode, int32_t num_seqs, int32_t total_q, int32_t total_kv, int32_t num_q_heads,
    int32_t num_kv_heads, int32_t head_dim, int32_t window, float scale, float q_scale,
    float k_scale, float v_scale, void* out, float* lse, void* workspace, size_t workspace_bytes,
    void* stream, void* attn_begin_event, void* attn_end_event) {
  NvtxRange nvtx("dg_attn_forward_fp8_profiled");
  return forward_fp8(q, k, v, cu_q, ctx_len, mode, num_seqs, total_q, total_kv, num_q_heads,
                     num_kv_heads, head_dim, window, scale, q_scale, k_scale, v_scale, out, lse,
                     workspace, workspace_bytes, stream, attn_begin_event, attn_end_event);
}

namespace {
dg_status_t forward_paged(const void* q, const void* k_new, const void* v_new, void* k_cache,
                          void* v_cache, int32_t num_pages, int32_t page_size,
                          const int32_t* block_table, int32_t max_pages_per_seq,
                          const int32_t* cu_q, const int32_t* ctx_len, const uint8_t* mode,
                          int32_t num_seqs, int32_t total_q, int32_t num_q_heads,
                          int32_t num_kv_heads, int32_t head_dim, int32_t window, float scale,
                          void* out, float* lse, void* workspace, size_t workspace_bytes,
                          void* stream, void* ev_begin, void* ev_end) {
  if (page_size < 8 || page_size > 65536 || (page_size & (page_size - 1)) != 0)
    return DG_ERR_INVALID_ARG;
  if (num_pages < 1 || static_cast<int64_t>(num_pages) * page_size > INT32_MAX)
    return DG_ERR_INVALID_ARG;
  if (max_pages_per_seq < 1 || num_seqs < 0 ||
      static_cast<int64_t>(num_seqs) * max_pages_per_seq > INT32_MAX)
    return DG_ERR_INVALID_ARG;
  if (!k_cache || !v_cache || !block_table || !aligned(k_cache, 16) || !aligned(v_cache, 16) ||
      !aligned(block_table, 4))
    return DG_ERR_INVALID_ARG;
  if ((k_new == nullptr) != (v_new == nullptr)) return DG_ERR_INVALID_ARG;
  if (k_new && (!aligned(k_new, 16) || !aligned(v_new, 16))) return DG_ERR_INVALID_ARG;
  PagedArgs pg;
  pg.block_table = block_table;
  pg.bt_stride = max_pages_per_seq;
  pg.page_shift = 0;
  while ((1 << pg.page_shift) < page_size) ++pg.page_shift;
  pg.num_pages = num_pages;
  pg.k_new = static_cast<const __nv_bfloat16*>(k_new);
  pg.v_new = static_cast<const __nv_bfloat16*>(v_new);
  pg.k_cache = static_cast<__nv_bfloat16*>(k_cache);
  pg.v_cache = static_cast<__nv_bfloat16*>(v_cache);
  pg.Hkv = num_kv_heads;
  pg.D = head_dim;
  return forward_impl(q, nullptr, nullptr, cu_q, ctx_len, mode, num_seqs, total_q, 0, num_q_heads,
                      num_kv_heads, head_dim, window, scale, out, lse, workspace, workspace_bytes,
                      stream, ev_begin, ev_end, &pg);
}
}  // namespace

extern "C" dg_status_t dg_attn_forward_paged(
    const void* q, const void* k_new, const void* v_new, void* k_cache, void* v_cache,
    int32_t num_pages, int32_t page_size, const int32_t* block_table, int32_t max_pages_per_seq,
    const int32_t* cu_q, const int32_t* ctx_len, const uint8_t* mode, int32_t num_seqs,
    int32_t total_q, int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim, int32_t window,
    float scale, void* out, float* lse, void* workspace, size_t workspace_bytes, void* stream) {
  NvtxRange nvtx("dg_attn_forward_paged");
  return forward_paged(q, k_new, v_new, k_cache, v_cache, num_pages, page_size, block_table,
                       max_pages_per_seq, cu_q, ctx_len, mode, num_seqs, total_q, num_q_heads,
                       num_kv_heads, head_dim, window, scale, out, lse, workspace, workspace_bytes,
                       stream, nullptr, nullptr);
}

extern "C" dg_status_t dg_attn_forward_paged_profiled(
    const void* q, const void* k_new, const void* v_new, void* k_cache, void* v_cache,
    int32_t num_pages, int32_t page_size, const int32_t* block_table, int32_t max_pages_per_seq,
    const int32_t* cu_q, const int32_t* ctx_len, const uint8_t* mode, int32_t num_seqs,
    int32_t total_q, int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim, int32_t window,
    float scale, void* out, float* lse, void* workspace, size_t workspace_bytes, void* stream,
    void* attn_begin_event, void* attn_end_event) {
  NvtxRange nvtx("dg_attn_forward_paged_profiled");
  return forward_paged(q, k_new, v_new, k_cache, v_cache, num_pages, page_size, block_table,
                       max_pages_per_seq, cu_q, ctx_len, mode, num_seqs, total_q, num_q_heads,
                       num_kv_heads, head_dim, window, scale, out, lse, workspace, workspace_bytes,
                       stream, attn_begin_event, attn_end_event);
}

namespace {
// row statistics chunks per row: rows of a vocabulary that is not a multiple of
// 8 start up to 7 logits past a 16-byte boundary, and the chunks start there
int stat_chunks(int32_t vocab) {
  const int64_t span = static_cast<int64_t>(vocab) + (vocab % 8 ? 7 : 0);
  return static_cast<int>((span + kStatChunk - 1) / kStatChunk);
}
}  // namespace

namespace {
int stat_chunks(int32_t vocab);

// Self-conditioning plan: tiles, vocabulary splits and the workspace layout.
// The split count depends only on the shapes and the SM count, so the size
// query and the call agree.
struct ScPlan {
  int m_tiles, n_tiles, splits, kblocks, chunks;
  size_t off_stats, off_rowc, off_part, total;
};

ScPlan sc_plan(int rows, int vocab, int d, int num_sms) {
  ScPlan pl;
  pl.m_tiles = (rows + kRows - 1) / kRows;
  pl.n_tiles = (d + kScN - 1) / kScN;
  pl.kblocks = (vocab + kScK - 1) / kScK;
  pl.chunks = stat_chunks(vocab);
  // split the vocabulary so the units spread evenly over the CTAs (one per
  // SM): minimise ceil(units / CTAs) / splits (the time of the busiest CTA),
  // keeping at least 8 blocks per split
  const int64_t per_split = static_cast<int64_t>(pl.m_tiles) * pl.n_tiles;
  const int ctas = std::max(1, num_sms);
  const int smax = std::max(1, std::min(64, pl.kblocks / 8));
  pl.splits = 1;
  double best = 1e30;
  for (int S = 1; S <= smax; ++S) {
    const double cost = static_cast<double>((per_split * S + ctas - 1) / ctas) / S;
    if (cost < best - 1e-12) {
      best = cost;
      pl.splits = S;
    }
  }
  size_t off = 0;
  pl.off_stats = off;
  off = align256(off + sizeof(RowPartial) * static_cast<size_t>(rows) * pl.chunks);
  pl.off_rowc = off;
  off = align256(off + sizeof(float) * static_cast<size_t>(rows));
  pl.off_part = off;
  if (pl.splits > 1)
    off = align256(off + sizeof(float) * static_cast<size_t>(pl.splits) * pl.m_tiles * kRows *
                             static_cast<size_t>(pl.n_tiles) * kScN);
  pl.total = off;
  return pl;
}

bool sc_shapes_ok(int32_t rows, int32_t vocab, int32_t d) {
  return rows >= 1 && vocab >= 8 && vocab % 8 == 0 && d >= 8 && d % 8 == 0;
}

// stats_ready: the row statistics of these logits are already at the
// workspace's start (written by the acceptance step of the same call)
dg_status_t selfcond_impl(const void* logits, int32_t rows, int32_t vocab, const void* embedding,
                          int32_t d_model, float* out, void* workspace, size_t workspace_bytes,
                          void* stream_ptr, void* ev_begin, void* ev_end, bool stats_ready = false) {
  if (!sc_shapes_ok(rows, vocab, d_model)) return DG_ERR_INVALID_ARG;
  if (!logits || !embedding || !out || !aligned(logits, 16) || !aligned(embedding, 16) ||
      !aligned(out, 16))
    return DG_ERR_INVALID_ARG;
  DeviceInfo* di = nullptr;
  const dg_status_t st = device_info(&di);
  if (st != DG_OK) return st;
  const ScPlan pl = sc_plan(rows, vocab, d_model, di->num_sms);
  if (!workspace || !aligned(workspace, 256) || workspace_bytes < pl.total) return DG_ERR_WORKSPACE;
  int ncta = di->num_sms;
  const int64_t units = static_cast<int64_t>(pl.splits) * pl.m_tiles * pl.n_tiles;
  if (units < ncta) ncta = static_cast<int>(units);

  CUtensorMap ml, me;
  // logits [rows, vocab]: boxes of 64 entries x 128 rows; E [vocab, d]: boxes
  // of 64 columns x 64 vocabulary rows
  if (encode_map(&ml, logits, rows, 1, vocab, 1, kRows) != DG_OK ||
      encode_map(&me, embedding, vocab, 1, d_model, 1, kScK) != DG_OK)
    return DG_ERR_INVALID_ARG;

  uint8_t* w = static_cast<uint8_t*>(workspace);
  RowPartial* stats = reinterpret_cast<RowPartial*>(w + pl.off_stats);
  ScParams p;
  p.rowc = reinterpret_cast<float*>(w + pl.off_rowc);
  p.out = out;
  p.part = pl.splits > 1 ? reinterpret_cast<float*>(w + pl.off_part) : nullptr;
  p.status = di->status;
  p.rows = rows;
  p.vocab = vocab;
  p.d = d_model;
  p.m_tiles = pl.m_tiles;
  p.n_tiles = pl.n_tiles;
  p.splits = pl.splits;
  p.debug_skip_e_load = -1;
  if (const char* e = std::getenv("DG_SELFCOND_DEBUG_SKIP_E_LOAD")) p.debug_skip_e_load = std::atoi(e);
  p.kblocks = pl.kblocks;

  cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
  if (!stats_ready)
    row_stats_kernel<<<static_cast<unsigned>(rows) * pl.chunks, kStatThreads, 0, stream>>>(
        static_cast<const __nv_bfloat16*>(logits), vocab, pl.chunks, stats);
  sc_rowconst_kernel<<<(rows + 7) / 8, 256, 0, stream>>>(stats, rows, pl.chunks,
                                                         const_cast<float*>(p.rowc));
  if (cudaGetLastError() != cudaSuccess) return DG_ERR_CUDA;
  cudaEvent_t e0 = static_cast<cudaEvent_t>(ev_begin), e1 = static_cast<cudaEvent_t>(ev_end);
  if (e0 && cudaEventRecord(e0, stream) != cudaSuccess) return DG_ERR_CUDA;
  sc_kernel<<<ncta, kScThreads, ScCfg::SMEM_BYTES, stream>>>(ml, me, p);
  if (cudaGetLastError() != cudaSuccess) return DG_ERR_CUDA;
  if (e1 && cudaEventRecord(e1, stream) != cudaSuccess) return DG_ERR_CUDA;
  if (pl.splits > 1) {
    const dim3 grid(pl.m_tiles, (d_model + 31) / 32);
    sc_combine_kernel<<<grid, dim3(32, 8), 0, stream>>>(p);
    if (cudaGetLastError() != cudaSuccess) return DG_ERR_CUDA;
  }
  return DG_OK;
}
}  // namespace

extern "C" size_t dg_selfcond_workspace_size(int32_t rows, int32_t vocab, int32_t d_model) {
  if (!sc_shapes_ok(rows, vocab, d_model)) return 0;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return sc_plan(rows, vocab, d_model, sms).total;
}

extern "C" dg_status_t dg_selfcond_forward(const void* logits, int32_t rows, int32_t vocab,
                                           const void* embedding, int32_t d_model, float* out,
                                           void* workspace, size_t workspace_bytes, void* stream) {
  NvtxRange nvtx("dg_selfcond_forward");
  return selfcond_impl(logits, rows, vocab, embedding, d_model, out, workspace, workspace_bytes,
                       stream, nullptr, nullptr);
}

extern "C" dg_status_t dg_selfcond_forward_profiled(const void* logits, int32_t rows,
                                                    int32_t vocab, const void* embedding,
                                                    int32_t d_model, float* out, void* workspace,
                                                    size_t workspace_bytes, void* stream,
                                                    void* gemm_begin_event, void* gemm_end_event) {
  NvtxRange nvtx("dg_selfcond_forward_profiled");
  return selfcond_impl(logits, rows, vocab, embedding, d_model, out, workspace, workspace_bytes,
                       stream, gemm_begin_event, gemm_end_event);
}

extern "C" size_t dg_accept_workspace_size(int32_t rows, int32_t vocab) {
  if (rows < 0 || vocab < 1) return 0;
  const size_t chunks = static_cast<size_t>(stat_chunks(vocab));
  return align256(sizeof(RowPartial) * chunks * static_cast<size_t>(rows) + 1);
}

extern "C" dg_status_t dg_accept_step(const void* logits, int32_t rows, int32_t vocab,
                                      const int32_t* cu_rows, int32_t num_canvases,
                                      const uint8_t* accepted_in, const int32_t* argmax_prev,
                                      const int32_t* stable_in, float entropy_budget,
                                      float entropy_threshold, int32_t patience, int32_t step,
                                      int32_t max_steps, float* entropy_out, float* confidence_out,
                                      int32_t* argmax_out, uint8_t* accepted_out,
                                      int32_t* stable_out, uint8_t* converged_out, void* workspace,
                                      size_t workspace_bytes, void* stream_ptr) {
  NvtxRange nvtx("dg_accept_step");
  if (rows < 0 || vocab < 1 || num_canvases < 0 || patience < 0 || max_steps < 1 || step < 0 ||
      !std::isfinite(entropy_budget) || entropy_budget < 0.f || !std::isfinite(entropy_threshold))
    return DG_ERR_INVALID_ARG;
  if (rows == 0 || num_canvases == 0) return DG_OK;
  if (!logits || !cu_rows || !accepted_in || !argmax_prev || !stable_in || !entropy_out ||
      !confidence_out || !argmax_out || !accepted_out || !stable_out || !converged_out)
    return DG_ERR_INVALID_ARG;
  if (!aligned(logits, 16)) return DG_ERR_INVALID_ARG;
  if (!workspace || !aligned(workspace, 256) ||
      workspace_bytes < dg_accept_workspace_size(rows, vocab))
    return DG_ERR_WORKSPACE;
  DeviceInfo* di = nullptr;
  const dg_status_t st = device_info(&di);
  if (st != DG_OK) return st;
  const int chunks = stat_chunks(vocab);
  cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
  RowPartial* part = static_cast<RowPartial*>(workspace);
  row_stats_kernel<<<static_cast<unsigned>(rows) * chunks, kStatThreads, 0, stream>>>(
      static_cast<const __nv_bfloat16*>(logits), vocab, chunks, part);
  if (cudaGetLastError() != cudaSuccess) return DG_ERR_CUDA;
  AcceptParams ap;
  ap.part = part;
  ap.chunks = chunks;
  ap.cu_rows = cu_rows;
  ap.accepted_in = accepted_in;
  ap.argmax_prev = argmax_prev;
  ap.stable_in = stable_in;
  ap.budget = entropy_budget;
  ap.tau = entropy_threshold;
  ap.patience = patience;
  ap.step = step;
  ap.max_steps = max_steps;
  ap.entropy = entropy_out;
  ap.confidence = confidence_out;
  ap.argmax = argmax_out;
  ap.accepted_out = accepted_out;
  ap.stable_out = stable_out;
  ap.converged = converged_out;
  ap.status = di->status;
  accept_kernel<<<num_canvases, kAcceptThreads, 0, stream>>>(ap);
  if (cudaGetLastError() != cudaSuccess) return DG_ERR_CUDA;
  return DG_OK;
}

extern "C" dg_status_t dg_attn_status(void* stream_ptr) {
  DeviceInfo* di = nullptr;
  const dg_status_t st = device_info(&di);
  if (st != DG_OK) return st;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
  int h = 0;
  if (cudaMemcpyAsync(&h, di->status, sizeof(int), cudaMemcpyDeviceToHost, stream) != cudaSuccess)
    return DG_ERR_CUDA;
  if (cudaMemsetAsync(di->status, 0, sizeof(int), stream) != cudaSuccess) return DG_ERR_CUDA;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return DG_ERR_CUDA;
  return static_cast<dg_status_t>(h);
}

extern "C" const char* dg_attn_error_string(int32_t status) {
  switch (status) {
    case DG_OK: return "ok";
    case DG_ERR_INVALID_ARG: return "invalid argument";
    case DG_ERR_UNSUPPORTED: return "unsupported configuration or device";
    case DG_ERR_CUDA: return "CUDA runtime error";
    case DG_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
    case DG_ERR_DEVICE_TIMEOUT: return "a device-side wait timed out";
    case DG_ERR_DEVICE_BOUNDS: return "a device-side bounds check failed";
    default: return "unknown status";
  }
}

extern "C" int32_t dg_attn_version(void) { return kVersion; }

// The sampler's work on one denoise step's logits in one call: the acceptance
// step and the self-conditioning average share one pass of row statistics.
extern "C" size_t dg_sampler_workspace_size(int32_t rows, int32_t vocab, int32_t d_model) {
  const size_t a = dg_accept_workspace_size(rows, vocab);
  const size_t b = dg_selfcond_workspace_size(rows, vocab, d_model);
  if (a == 0 || b == 0) return 0;
  return a > b ? a : b;
}

extern "C" dg_status_t dg_sampler_step(const void* logits, int32_t rows, int32_t vocab,
                                       const int32_t* cu_rows, int32_t num_canvases,
                                       const uint8_t* accepted_in, const int32_t* argmax_prev,
                                       const int32_t* stable_in, float entropy_budget,
                                       float entropy_threshold, int32_t patience, int32_t step,
                                       int32_t max_steps, const void* embedding, int32_t d_model,
                                       float* entropy_out, float* confidence_out,
                                       int32_t* argmax_out, uint8_t* accepted_out,
                                       int32_t* stable_out, uint8_t* converged_out,
                                       float* selfcond_out, void* workspace,
                                       size_t workspace_bytes, void* stream) {
  NvtxRange nvtx("dg_sampler_step");
  if (rows == 0) return num_canvases >= 0 ? DG_OK : DG_ERR_INVALID_ARG;
  if (num_canvases < 1 || !sc_shapes_ok(rows, vocab, d_model)) return DG_ERR_INVALID_ARG;
  if (!embedding || !selfcond_out || !aligned(embedding, 16) || !aligned(selfcond_out, 16))
    return DG_ERR_INVALID_ARG;
  if (workspace_bytes < dg_sampler_workspace_size(rows, vocab, d_model)) return DG_ERR_WORKSPACE;
  const dg_status_t st = dg_accept_step(logits, rows, vocab, cu_rows, num_canvases, accepted_in,
                                        argmax_prev, stable_in, entropy_budget, entropy_threshold,
                                        patience, step, max_steps, entropy_out, confidence_out,
                                        argmax_out, accepted_out, stable_out, converged_out,
                                        workspace, workspace_bytes, stream);
  if (st != DG_OK) return st;
  return selfcond_impl(logits, rows, vocab, embedding, d_model, selfcond_out, workspace,
                       workspace_bytes, stream, nullptr, nullptr, true);
}
