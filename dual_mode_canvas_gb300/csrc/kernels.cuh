// Device side of the dual-mode attention forward pass.
//
//   build_worklist_kernel  one CTA: validates cu_q / ctx_len / mode, cuts every
//                          (sequence, KV head) into 128-row query tiles and
//                          computes each tile's visible KV-tile range; the
//                          range is the union of the rows' windows (causal:
//                          keys <= i, bidirectional: the whole sequence, both
//                          narrowed to [i-W, i+W] on sliding-window layers).
//                          Batches of at most kLocalMaxTiles tiles with
//                          contiguous K/V skip this grid: every CTA of the
//                          attention grid builds the same list for itself.
//   fwd_kernel<D,BN,NK,NV,F8,NS,QS> persistent, one CTA per SM.  The (tile,
//                          KV-tile) work units are split over the CTAs by
//                          weight; each CTA keeps the tiles of its range in a
//                          shared-memory window (all shapes but e4m3 head_dim
//                          128) and TMA-loads the K/V tiles it consumes from
//                          this GPU's memory into its own shared memory.  A tile cut between CTAs leaves fp32
//                          partials + LSE.
//                          Warp roles: warps 4 and 6 issue TMA loads (K ring,
//                          V ring; warp 7 shares the K boxes of tiles of small
//                          pages), warp 5 issues tcgen05 MMAs, warps 0-3 (one
//                          TMEM lane = one query row each) stage Q and run the
//                          online softmax and the epilogue.
//   combine_kernel<D>      merges the partials of cut tiles by their LSE.
//
// Paged KV cache (block-table indirection): K and V live in pools of pages of
// P = 2^page_shift token rows, [num_pages * P, Hkv, D]; block_table[s, p] is
// the physical page of positions p*P .. p*P+P-1 of sequence s.  The work-list
// launch then also appends the query tokens' K/V rows into their pages (CTAs
// 1.. of the launch) and checks every page-table entry the attention will
// read; the loaders look up each tile's pages and load them in boxes of
// min(P, BN) rows, one box per lane of the loader warp (V pages of one MMA K
// step or half of one, and K pages of 8 rows, in one box per page).
//
// Rules (DiffusionGemma, agentlenshq page, "dual-mode operation", "dynamic
// per-sequence causal attention", "symmetric sliding-window attention"): a
// causal query at position i sees keys j <= i, a bidirectional one every key of
// its sequence; a window W keeps j >= i - W and, when bidirectional, j <= i + W.
// One formula covers all four cases, so no warp branches on the mode:
//   visible(i, j) = (j >= i - WL) && (j <= min(i + WR, L - 1))
//   WL = W < 0 ? inf : W,   WR = causal ? 0 : (W < 0 ? inf : W)
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cstdint>
#include <type_traits>

#include "ptx.cuh"

namespace dg {

constexpr int kRows = 128;          // query rows per tile (UMMA M, TMEM lanes)
constexpr int kThreads = 256;       // 4 softmax warps + K loader + MMA issuer + V loader (+ K loader 2)
constexpr int kTmaWarp = 4;         // loads the K ring
constexpr int kMmaWarp = 5;         // issues tcgen05 MMAs, owns TMEM
constexpr int kVLoadWarp = 6;       // loads the V ring
constexpr int kTmaWarp2 = 7;        // with k_split, issues half of every K tile's boxes
constexpr uint32_t kTmemCols = 512;
constexpr uint64_t kWaitTimeoutNs = 250ull * 1000ull * 1000ull;
// Work-split weight of starting a segment (Q load, pipeline fill, epilogue),
// in KV-tile units: every tile occupies seg_weight + (its KV tiles) units of
// the split, the first seg_weight of them carrying no KV tile.  The host
// picks it per kernel shape (a segment costs about the same time whatever the
// shape, a KV tile does not).

// error codes shared with the host (same values as dg_status_t)
constexpr int kErrInvalid = 1;
constexpr int kErrTimeout = 5;
constexpr int kErrBounds = 6;

struct TileDesc {
  int32_t q_row0;    // global query row of the tile's first token
  int32_t n_tok;     // query tokens in the tile (1 .. TT)
  int32_t kv_row0;   // global K/V row of the sequence's first key (paged: its page-table row offset)
  int32_t pos0;      // absolute position of the tile's first token
  int32_t L;         // keys of the sequence (context + queries)
  int32_t kt_first;  // first KV tile of the tile's range (units of BN keys, sequence-relative)
  int32_t kvh;       // KV head
  int32_t causal;    // 1 causal (encoder), 0 bidirectional (denoise)
  int32_t kt_count;  // KV tiles in the range
  int32_t kt_rot;    // the KV tiles are visited from kt_first + kt_rot on, cyclically
  // split-KV merge: the tile's KV tiles are spread over comb_n CTAs from
  // comb_cta on (comb_n <= 1: written directly); the first of them wrote its
  // partial to slot comb_slot0, CTA comb_cta + i (i >= 1) to slot 2 (comb_cta + i)
  int32_t comb_cta;
  int32_t comb_n;
  int32_t comb_slot0;
  int32_t pad_;
};

// KV tile (sequence-relative, units of BN keys) visited j-th for a query tile.
__device__ __forceinline__ int kv_tile(const TileDesc& td, int j) {
  int x = j + td.kt_rot;
  if (x >= td.kt_count) x -= td.kt_count;
  return td.kt_first + x;
}

// The work list as one CTA of the attention kernel reads it: the descriptors
// and unit starts of a window of up to kWinTiles tiles, from the tile holding
// the CTA's first unit, in shared memory; tiles past the window from the
// global tables.  (A CTA's unit range spans one to three tiles in the
// configured workloads.)
constexpr int kWinTiles = 16;
struct WorkView {
  const TileDesc* g_tiles;  // global tile table (this CTA's copy, or the work-list grid's)
  const int64_t* g_ub;      // global unit starts, [num_tiles + 1]
  int t0, n;                // the window holds tiles t0 .. t0 + n - 1
  int scratch[2];
  TileDesc s_tiles[kWinTiles];
  int64_t s_ub[kWinTiles + 1];  // unit starts of tiles t0 .. t0 + n
  __device__ __forceinline__ int64_t ub(int t) const {
    const unsigned i = static_cast<unsigned>(t - t0);
    return i <= static_cast<unsigned>(n) ? s_ub[i] : g_ub[t];
  }
  __device__ __forceinline__ TileDesc tile(int t) const {
    const unsigned i = static_cast<unsigned>(t - t0);
    return i < static_cast<unsigned>(n) ? s_tiles[i] : g_tiles[t];
  }
};

struct WorkHeader {
  int32_t num_tiles;  // query tiles
  int32_t error;
  int64_t total_units;
};

struct Workspace {
  WorkHeader* hdr;
  int64_t* seq_tile_off;   // [B + 1] tiles before each sequence
  int64_t* seq_kv_off;     // [B + 1]
  TileDesc* tiles;         // [max_tiles]
  int64_t* unit_begin;     // [max_tiles + 1]
  float* part_lse;         // [2 * num_ctas][128]
  float* part_o;           // [2 * num_ctas][128][D]
};

struct FwdParams {
  Workspace ws;
  const void* q;       // bf16 or e4m3 [total_q, Hq, D]
  __nv_bfloat16* out;
  float* lse;
  int* status;
  int Hq, G, TT, window;
  // paged KV cache: block_table [B, bt_stride] (nullptr: contiguous K/V),
  // pages of 2^page_shift rows, TMA boxes of page_box rows
  const int32_t* block_table;
  int page_shift, page_box;
  // 1: the V tensor map is 4-D ({128-byte block, head, row, column block})
  // and one box brings a whole page (page_box rows, every column block of
  // head_dim): a page of one MMA K step (16 bf16 / 32 e4m3 rows), or of half
  // of one (8 bf16 rows), lands as [column block][row][128 bytes], which P.V
  // reads with the column-block stride of one page (and, for 8-row pages, the
  // next 8 rows one page further on).  Cuts a small-page V tile from NKB
  // boxes per page to one.
  int v_page_box;
  // 1: the same whole-page boxes for K, with 8-row pages only: a page is then
  // one 8-row swizzle group of every column block, so QK^T's B operand finds
  // consecutive 8-row groups of a column block one page (NKB * 1024 bytes)
  // apart.  (Larger pages hold several groups of a column block together, at
  // another stride than the next page's.)
  int k_page_box;
  // 1: two warps issue a K tile's TMA boxes, half each (each registers its
  // half of the bytes on K_FULL, which then counts two arrivals).  A K tile of
  // small pages is 16 or more boxes, and one warp issuing them one after the
  // other is what paces the loads (~75 clocks a box).
  int k_split;
  int seg_weight;  // the work list's segment weight (KV-tile units)
  // >= 0: the K loader skips the TMA load of this (per-CTA) KV tile, so the
  // MMA warp's bounded wait for it expires (tests of the timeout path)
  int debug_skip_k_load;
  // sizes the bounds-checking build checks every index against: K/V rows of
  // the tensor maps, KV heads, query rows, partial slots, page-table entries
  int Hkv, kv_rows, total_q, num_slots;
  int64_t bt_entries;
  // bounds-checking build only, >= 0: the K loader moves the row coordinate
  // of this (per-CTA) KV tile past the tensor, so its bounds check fails
  // (tests of the check; the load it guards is skipped)
  int debug_bad_kv_row;
  // 1: no work-list grid; every CTA of the attention grid builds the work
  // list itself from the metadata below (contiguous K/V, at most
  // kLocalMaxTiles tiles).  CTA c keeps its copy of the tables at ws.tiles +
  // c * tiles_stride and ws.unit_begin + c * ub_stride; CTA 0's copy, at the
  // base, is the one the split-KV merge reads.
  int fused_wl;
  int tiles_stride, ub_stride;  // max_tiles and max_tiles + 1 with fused_wl, else 0
  const int32_t* cu_q;
  const int32_t* ctx_len;
  const uint8_t* mode;
  int B, max_tiles, rotate;
  int64_t kv_total;  // K/V rows of the contiguous layout
  float scale, scale_log2;  // softmax scale (times the q and k scales for e4m3 inputs)
  float v_scale;            // e4m3 inputs: the v scale, applied in the epilogue (1 for bf16)
};

// Maximum of N registers by a tree of 3-input maxima: ceil(log3 N) dependent
// levels instead of a chain of N / 2.
template <int N>
struct TreeMax {
  static __device__ __forceinline__ float of(const float* v) {
    constexpr int M = (N + 2) / 3;
    float t[M];
#pragma unroll
    for (int i = 0; i < M; ++i) {
      if (3 * i + 2 < N) t[i] = max3f(v[3 * i], v[3 * i + 1], v[3 * i + 2]);
      else if (3 * i + 1 < N) t[i] = fmaxf(v[3 * i], v[3 * i + 1]);
      else t[i] = v[3 * i];
    }
    return TreeMax<M>::of(t);
  }
};
template <>
struct TreeMax<1> {
  static __device__ __forceinline__ float of(const float* v) { return v[0]; }
};
template <>
struct TreeMax<2> {
  static __device__ __forceinline__ float of(const float* v) { return fmaxf(v[0], v[1]); }
};

// a row of packed P -> TMEM (16, 32 or 64 columns)
__device__ __forceinline__ void store_packed_p(uint32_t taddr, const uint32_t (&r)[16]) { tmem_st16(taddr, r); }
__device__ __forceinline__ void store_packed_p(uint32_t taddr, const uint32_t (&r)[32]) { tmem_st32(taddr, r); }
__device__ __forceinline__ void store_packed_p(uint32_t taddr, const uint32_t (&r)[64]) { tmem_st64(taddr, r); }

__device__ __forceinline__ void record_error(int* status, int code) {
  atomicCAS(status, 0, code);
}

// Bounds checks of the debug build (compiled with DG_ATTN_DEBUG): every TMA
// coordinate, shared-memory destination, TMEM column and global index is
// checked against its buffer before the access.  A failed check records
// DG_ERR_DEVICE_BOUNDS in the status word, raises the CTA's abort flag (every
// role then leaves its loop through the bounded-wait exits) and the access is
// skipped.  Release builds compile the checks out.
#ifdef DG_ATTN_DEBUG
constexpr bool kBoundsChecks = true;
#else
constexpr bool kBoundsChecks = false;
#endif
__device__ __forceinline__ bool in_bounds(bool ok, int* status, volatile int* abort_flag) {
  if constexpr (kBoundsChecks) {
    if (!ok) {
      record_error(status, kErrBounds);
      if (abort_flag != nullptr) *abort_flag = 1;
    }
    return ok;
  } else {
    return true;
  }
}

// ------------------------------------------------------------ block scan
// Exclusive scan of one value per thread over a 1024-thread block; *total
// receives the block's sum.  Every thread of the block must call it.
__device__ int64_t block_scan_1024(int64_t x, int64_t* total) {
  __shared__ int64_t warp_part[32];
  __shared__ int64_t block_total;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int64_t incl = x;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int64_t y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) warp_part[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const int64_t w = warp_part[lane];
    int64_t wi = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int64_t y = __shfl_up_sync(0xffffffffu, wi, o);
      if (lane >= o) wi += y;
    }
    warp_part[lane] = wi - w;  // exclusive prefix of the warp sums
    if (lane == 31) block_total = wi;
  }
  __syncthreads();
  const int64_t r = warp_part[warp] + incl - x;
  *total = block_total;
  __syncthreads();  // the shared words are reused by the next call
  return r;
}

// ------------------------------------------------ paged cache: the append
struct PagedArgs {
  const int32_t* block_table;    // [B, bt_stride]; nullptr: contiguous K/V
  int bt_stride;                 // page-table entries per sequence
  int page_shift;                // pages of 2^page_shift rows
  int num_pages;
  const __nv_bfloat16* k_new;    // [total_q, Hkv, D] or nullptr (no append)
  const __nv_bfloat16* v_new;
  __nv_bfloat16* k_cache;        // [num_pages << page_shift, Hkv, D]
  __nv_bfloat16* v_cache;
  int Hkv, D;
};

// Writes row r of k_new / v_new (query token t of sequence s) at position
// ctx_len[s] + t of sequence s, 16 bytes per thread, grid-stride over the
// CTAs 1 .. gridDim.x-1.  Every write is checked against the page table and
// the pool; a bad entry records DG_ERR_INVALID_ARG and the row is skipped.
__device__ void append_rows(const int32_t* __restrict__ cu_q, const int32_t* __restrict__ ctx_len,
                            int B, int total_q, const PagedArgs& pg, int* status) {
  const int upr = pg.Hkv * pg.D / 8;  // 16-byte units per token row
  const int64_t units = static_cast<int64_t>(total_q) * upr;
  const int64_t step = static_cast<int64_t>(gridDim.x - 1) * blockDim.x;
  const int P = 1 << pg.page_shift;
  for (int64_t u = static_cast<int64_t>(blockIdx.x - 1) * blockDim.x + threadIdx.x; u < 2 * units;
       u += step) {
    const bool is_v = u >= units;
    const int64_t uu = is_v ? u - units : u;
    const int r = static_cast<int>(uu / upr);
    const int c = static_cast<int>(uu - static_cast<int64_t>(r) * upr);
    int lo = 0, hi = B - 1;  // sequence of row r: largest s with cu_q[s] <= r
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (cu_q[mid] <= r) lo = mid; else hi = mid - 1;
    }
    const int t = r - cu_q[lo];
    const int pos = ctx_len[lo] + t;
    if (t < 0 || pos < 0 || (pos >> pg.page_shift) >= pg.bt_stride) {
      record_error(status, kErrInvalid);
      continue;
    }
    const int page = pg.block_table[static_cast<int64_t>(lo) * pg.bt_stride + (pos >> pg.page_shift)];
    if (page < 0 || page >= pg.num_pages) {
      record_error(status, kErrInvalid);
      continue;
    }
    const int64_t row = (static_cast<int64_t>(page) << pg.page_shift) + (pos & (P - 1));
    const uint4* src = reinterpret_cast<const uint4*>((is_v ? pg.v_new : pg.k_new) +
                                                      static_cast<int64_t>(r) * pg.Hkv * pg.D) + c;
    uint4* dst = reinterpret_cast<uint4*>((is_v ? pg.v_cache : pg.k_cache) + row * pg.Hkv * pg.D) + c;
    *dst = __ldg(src);
  }
}

// --------------------------------------------------------- work splitting
// The U work units are cut into P = min(grid, U) contiguous CTA ranges, so no
// CTA range is empty.
__device__ __forceinline__ int active_ctas(int grid, int64_t U) {
  return U < grid ? static_cast<int>(U) : grid;
}

__device__ __forceinline__ int64_t cta_unit_begin(int c, int64_t U, int P) {
  return static_cast<int64_t>(c) * U / P;
}

// ------------------------------------------------------ work-list builder
// Per-sequence values of the builder live in shared memory for batches of up
// to this many sequences (larger batches read them back from the workspace).
constexpr int kWlSmemSeqs = 1024;
// Batches of at most this many query tiles (with contiguous K/V) have no
// work-list grid: each CTA of the attention grid builds the list itself.
constexpr int kLocalMaxTiles = 256;
// CTAs of the attention grid at most (the host caps the grid).
constexpr int kMaxCtas = 1024;

// Per-sequence values a tile descriptor is made from: first query row
// (q0[B] = total_q), cached tokens, mode, tiles and K/V rows before the
// sequence (shared memory or workspace).
struct SeqTables {
  const int32_t* q0;
  const int32_t* ctx;
  const uint8_t* mode;
  const int64_t* toff;
  const int64_t* kvoff;
};

// Descriptor of query tile `tile` (KV range and geometry; no split fields).
// Tiles run sequence by sequence, KV head by KV head, TT tokens each.
__device__ TileDesc make_tile_desc(int tile, const SeqTables& st, int B, int TT, int BN, int window,
                                   bool paged, int bt_stride) {
  // sequence owning this tile: largest s with tiles-before(s) <= tile
  int lo = 0, hi = B - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (st.toff[mid] <= tile) lo = mid; else hi = mid - 1;
  }
  const int s = lo;
  const int q0 = st.q0[s];
  const int n = st.q0[s + 1] - q0;
  const int c = st.ctx[s];
  const int L = c + n;
  const bool causal = st.mode[s] == 0;
  const int m_tiles = (n + TT - 1) / TT;
  const int local = tile - static_cast<int>(st.toff[s]);
  const int kvh = local / m_tiles;
  const int mt = local - kvh * m_tiles;
  const int t0 = mt * TT;
  const int pos_first = c + t0;
  const int i_max = c + min(n, t0 + TT) - 1;
  const int kv_lo = window < 0 ? 0 : max(0, pos_first - window);
  const int kv_hi = causal ? i_max : (window < 0 ? L - 1 : min(L - 1, i_max + window));
  TileDesc td;
  td.q_row0 = q0 + t0;
  td.n_tok = min(TT, n - t0);
  td.kv_row0 = paged ? s * bt_stride : static_cast<int>(st.kvoff[s]);
  td.pos0 = pos_first;
  td.L = L;
  td.kt_first = kv_lo / BN;
  td.kvh = kvh;
  td.causal = causal ? 1 : 0;
  td.kt_count = kv_hi / BN - kv_lo / BN + 1;
  td.kt_rot = 0;
  td.comb_cta = 0;
  td.comb_n = 0;
  td.comb_slot0 = 0;
  td.pad_ = 0;
  return td;
}

// Largest CTA c < P whose unit range starts at or before unit u, from the
// table of range starts cbeg[0 .. P] (cbeg[c] = cta_unit_begin(c, U, P)).
__device__ __forceinline__ int cta_of_unit_tab(int64_t u, const int64_t* cbeg, int P) {
  int lo = 0, hi = P - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (cbeg[mid] <= u) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// Fills cbeg[0 .. P] (shared memory); every thread of the block calls it.
__device__ __forceinline__ void fill_cta_starts(int64_t* cbeg, int64_t U, int P) {
  for (int c = threadIdx.x; c <= P; c += blockDim.x) cbeg[c] = cta_unit_begin(c, U, P);
  __syncthreads();
}

// The split fields of a tile whose units start at ub (its KV tiles at
// ub + seg_weight), given the starts cbeg[0 .. P] of the P CTA ranges (P = 0:
// no units): the CTAs holding its KV tiles, the partial slot of the first,
// and the KV visiting offset.  (A table lookup instead of the 64-bit divisions
// of cta_of_unit: those put ~2 us on the critical path of every call.)
__device__ void split_tile_desc(TileDesc& td, int64_t ub, int seg_weight, const int64_t* cbeg, int P,
                                bool rotate) {
  const int64_t r0 = ub + seg_weight, n = td.kt_count;
  if (P <= 0) return;
  const int c_lo = cta_of_unit_tab(r0, cbeg, P), c_hi = cta_of_unit_tab(r0 + n - 1, cbeg, P);
  td.comb_cta = c_lo;
  td.comb_n = c_hi - c_lo + 1;
  td.comb_slot0 = cbeg[c_lo] >= ub ? 2 * c_lo : 2 * c_lo + 1;
  // KV visiting order.  The CTAs' unit ranges are contiguous and equally
  // long (U / P units), so the CTAs sharing one query tile start at KV-tile
  // offsets a multiple of U / P apart.  Rotating each tile's KV tiles so
  // that the CTA holding its first KV tile reaches that KV tile at "time"
  // (units since the launch) equal to the KV tile's index gives every CTA
  // of every query tile a phase that is a multiple of U / P: the query
  // tiles of one (sequence, KV head) with the same KV range then stream the
  // same KV tiles at about the same time, and the later readers find them
  // in L2.  The order of the KV tiles does not change the result beyond
  // fp32 rounding.
  if (rotate && n > 1 && P > 1) td.kt_rot = static_cast<int>((r0 - cbeg[c_lo]) % n);
}

// CTA 0 builds the work list; with a paged cache, CTAs 1.. append the new K/V.
// One read of the metadata, scans in registers and shared memory, one write
// of the tile table: the attention kernel waits for this grid, so its length
// is on every call's critical path.
__global__ void __launch_bounds__(1024, 1)
build_worklist_kernel(const int32_t* __restrict__ cu_q, const int32_t* __restrict__ ctx_len,
                      const uint8_t* __restrict__ mode, int B, int total_q, int total_kv, int Hkv,
                      int TT, int BN, int window, int max_tiles, int num_ctas, int rotate, int seg_weight,
                      Workspace ws, PagedArgs pg, int* status) {
  // the attention kernel is launched as a programmatic dependent: its CTAs
  // become resident while this grid runs and wait for it to finish
  griddep_launch_dependents();
  // this grid is itself a programmatic dependent of the stream's previous
  // kernel (the last call's split-KV merge, in a loop of calls): it becomes
  // resident while that grid drains, and reads or writes nothing before it
  // has finished
  griddep_wait();
  if (blockIdx.x > 0) {
    append_rows(cu_q, ctx_len, B, total_q, pg, status);
    return;
  }
  __shared__ int bad;
  __shared__ int32_t s_q0[kWlSmemSeqs + 1];   // cu_q
  __shared__ int32_t s_ctx[kWlSmemSeqs];
  __shared__ uint8_t s_mode[kWlSmemSeqs];
  __shared__ int64_t s_toff[kWlSmemSeqs + 1];  // tiles before each sequence
  __shared__ int64_t s_kvoff[kWlSmemSeqs];     // K/V rows before each sequence
  __shared__ int64_t s_cbeg[kMaxCtas + 1];     // start unit of each CTA range
  const int tid = threadIdx.x;
  const bool paged = pg.block_table != nullptr;
  const bool small = B <= kWlSmemSeqs;
  if (tid == 0) bad = 0;
  __syncthreads();
  if (tid == 0 && (cu_q[0] != 0 || cu_q[B] != total_q)) atomicOr(&bad, 1);
  // ---- sequences: tiles and K/V rows, scanned 1024 sequences at a time
  int64_t carry_t = 0, carry_kv = 0;
  for (int base = 0; base < B; base += 1024) {
    const int s = base + tid;
    int64_t nt = 0, nkv = 0;
    if (s < B) {
      const int q0 = cu_q[s], q1 = cu_q[s + 1], c = ctx_len[s], md = mode[s];
      const int n = q1 - q0;
      if (n < 0 || c < 0 || md > 1) atomicOr(&bad, 1);
      const int64_t nn = n < 0 ? 0 : n;
      nt = static_cast<int64_t>(Hkv) * ((nn + TT - 1) / TT);
      nkv = static_cast<int64_t>(c < 0 ? 0 : c) + nn;
      if (small) {
        s_q0[s] = q0;
        s_ctx[s] = c;
        s_mode[s] = static_cast<uint8_t>(md);
      }
    }
    int64_t sum_t, sum_kv;
    const int64_t et = block_scan_1024(nt, &sum_t);
    const int64_t ekv = block_scan_1024(nkv, &sum_kv);
    if (s < B) {
      if (small) {
        s_toff[s] = carry_t + et;
        s_kvoff[s] = carry_kv + ekv;
      } else {
        ws.seq_tile_off[s] = carry_t + et;
        ws.seq_kv_off[s] = carry_kv + ekv;
      }
    }
    carry_t += sum_t;
    carry_kv += sum_kv;
  }
  if (tid == 0) {
    if (small) {
      s_toff[B] = carry_t;
      s_q0[B] = total_q;
    } else {
      ws.seq_tile_off[B] = carry_t;
    }
    if (carry_t > max_tiles || (!paged && carry_kv > total_kv)) bad = 1;
  }
  __syncthreads();
  auto q0_of = [&](int s) { return small ? s_q0[s] : cu_q[s]; };
  auto ctx_of = [&](int s) { return small ? s_ctx[s] : ctx_len[s]; };
  if (paged && !bad) {
    // every page the attention reads: pages 0 .. ceil(L / P) - 1 of each sequence
    for (int s = 0; s < B; ++s) {
      const int64_t L = static_cast<int64_t>(ctx_of(s)) + q0_of(s + 1) - q0_of(s);
      const int64_t need = (L + (1 << pg.page_shift) - 1) >> pg.page_shift;
      if (need > pg.bt_stride) {
        if (tid == 0) bad = 1;
        continue;
      }
      for (int64_t i = tid; i < need; i += 1024) {
        const int page = pg.block_table[static_cast<int64_t>(s) * pg.bt_stride + i];
        if (page < 0 || page >= pg.num_pages) atomicOr(&bad, 1);
      }
    }
  }
  __syncthreads();
  if (bad) {
    if (tid == 0) {
      ws.hdr->num_tiles = 0;
      ws.hdr->total_units = 0;
      ws.hdr->error = kErrInvalid;
      record_error(status, kErrInvalid);
    }
    return;
  }
  // ---- tiles: thread tid owns the consecutive tiles [t_begin, t_end)
  const int num_tiles = static_cast<int>(carry_t);
  const int per = (num_tiles + 1023) / 1024;
  const int t_begin = min(num_tiles, tid * per), t_end = min(num_tiles, t_begin + per);
  const SeqTables st{small ? s_q0 : cu_q, small ? s_ctx : ctx_len, small ? s_mode : mode,
                     small ? s_toff : ws.seq_tile_off, small ? s_kvoff : ws.seq_kv_off};
  auto make_tile = [&](int tile) { return make_tile_desc(tile, st, B, TT, BN, window, paged, pg.bt_stride); };
  // pass 1: the units of this thread's tiles, scanned over the block
  int64_t mine = 0;
  for (int t = t_begin; t < t_end; ++t) mine += seg_weight + make_tile(t).kt_count;
  int64_t U;
  int64_t ub = block_scan_1024(mine, &U);
  const int P = active_ctas(num_ctas, U);
  fill_cta_starts(s_cbeg, U, P);
  // pass 2: the finished descriptors, written once
  for (int t = t_begin; t < t_end; ++t) {
    TileDesc td = make_tile(t);
    split_tile_desc(td, ub, seg_weight, s_cbeg, P, rotate != 0);
    ws.tiles[t] = td;
    ws.unit_begin[t] = ub;
    ub += seg_weight + td.kt_count;
  }
  if (tid == 0) {
    ws.unit_begin[num_tiles] = U;
    ws.hdr->num_tiles = num_tiles;
    ws.hdr->total_units = U;
    ws.hdr->error = 0;
  }
}

// Exclusive scan of one value per thread over the block (a multiple of 32
// threads, at most 1024); *total receives the block's sum.  wsum: 33 words of
// shared scratch.  Every thread of the block must call it.
__device__ int64_t block_scan_excl(int64_t x, int64_t* total, int64_t* wsum) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nw = static_cast<int>(blockDim.x >> 5);
  int64_t incl = x;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int64_t y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) wsum[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const int64_t w = lane < nw ? wsum[lane] : 0;
    int64_t wi = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int64_t y = __shfl_up_sync(0xffffffffu, wi, o);
      if (lane >= o) wi += y;
    }
    if (lane < nw) wsum[lane] = wi - w;
    if (lane == 31) wsum[32] = wi;
  }
  __syncthreads();
  const int64_t r = wsum[warp] + incl - x;
  *total = wsum[32];
  __syncthreads();  // the shared words are reused by the next call
  return r;
}

// Bytes of shared scratch build_worklist_cta uses.
constexpr int kLocalWlScratch = 40 * 8 + (kMaxCtas + 1) * 8 + 2 * (kLocalMaxTiles + 1) * 8 +
                                2 * (kLocalMaxTiles + 1) * 4 + (kLocalMaxTiles + 1);

// This CTA's unit range [u_beg, u_end) of U units over the active CTAs (a CTA
// past them, or a call without work, has an empty range).
__device__ __forceinline__ void cta_range(int num_tiles, int64_t U, int64_t& u_beg, int64_t& u_end) {
  const int cta = static_cast<int>(blockIdx.x);
  const int P = U > 0 ? active_ctas(static_cast<int>(gridDim.x), U) : 1;
  const bool active = num_tiles > 0 && U > 0 && cta < P;
  u_beg = active ? cta_unit_begin(cta, U, P) : 0;
  u_end = active ? cta_unit_begin(cta + 1, U, P) : 0;
}

// The work list of one call, built by a CTA of the attention grid for itself
// (every CTA builds the same list): the checks, tiles, unit starts, visiting
// offsets and merge contributors of build_worklist_kernel, from the same
// helpers, written to this CTA's copy of the tile table and unit starts (CTA
// 0 also writes the header) and, for the tiles from the one holding this
// CTA's first unit on, to its shared-memory window.  Contiguous K/V and at
// most kLocalMaxTiles tiles.  scratch: kLocalWlScratch bytes of shared
// memory.  Every thread of the block calls it; it returns the tile and unit
// counts (both 0 for invalid metadata, which it records as
// DG_ERR_INVALID_ARG).  Kept out of line: inlined, its registers spilled the
// attention kernel's e4m3 shapes.
struct WlCounts {
  int64_t units;
  int num_tiles;
};
// The call's metadata and sizes the in-grid builder reads.  (Passed by value:
// a reference to the kernel's parameter block made the e4m3 head_dim-128
// kernel read its parameters from a local copy.)
struct WlArgs {
  const int32_t* cu_q;
  const int32_t* ctx_len;
  const uint8_t* mode;
  WorkHeader* hdr;
  int* status;
  int64_t kv_total;
  int B, total_q, Hkv, TT, window, seg_weight, max_tiles, rotate;
};
__device__ __noinline__ WlCounts build_worklist_cta(const WlArgs p, int BN, TileDesc* tiles, int64_t* ub_out,
                                                    uint8_t* scratch, WorkView* wv) {
  constexpr int S = kLocalMaxTiles + 1;
  int64_t* wsum = reinterpret_cast<int64_t*>(scratch);  // 33 used
  int64_t* s_cbeg = wsum + 40;                          // start unit of each CTA range
  int64_t* s_toff = s_cbeg + kMaxCtas + 1;              // tiles before each sequence
  int64_t* s_kvoff = s_toff + S;                        // K/V rows before each sequence
  int32_t* s_q0 = reinterpret_cast<int32_t*>(s_kvoff + S);
  int32_t* s_ctx = s_q0 + S;
  uint8_t* s_mode = reinterpret_cast<uint8_t*>(s_ctx + S);
  const int tid = threadIdx.x, nthr = static_cast<int>(blockDim.x);
  const int B = p.B;
  // ---- sequences: tiles and K/V rows (B <= kLocalMaxTiles), every load of
  // the metadata in one round trip
  int bad = 0;
  int64_t carry_t = 0, carry_kv = 0;
  for (int base = 0; base < B; base += nthr) {
    const int s = base + tid;
    int64_t nt = 0, nkv = 0;
    if (s < B) {
      const int q0 = p.cu_q[s], q1 = p.cu_q[s + 1], c = p.ctx_len[s], md = p.mode[s];
      const int n = q1 - q0;
      if (n < 0 || c < 0 || md > 1 || (s == 0 && q0 != 0) || (s == B - 1 && q1 != p.total_q)) bad = 1;
      const int64_t nn = n < 0 ? 0 : n;
      nt = static_cast<int64_t>(p.Hkv) * ((nn + p.TT - 1) / p.TT);
      nkv = static_cast<int64_t>(c < 0 ? 0 : c) + nn;
      s_q0[s] = q0;
      s_ctx[s] = c;
      s_mode[s] = static_cast<uint8_t>(md);
    }
    int64_t sum_t, sum_kv;
    const int64_t et = block_scan_excl(nt, &sum_t, wsum);
    const int64_t ekv = block_scan_excl(nkv, &sum_kv, wsum);
    if (s < B) {
      s_toff[s] = carry_t + et;
      s_kvoff[s] = carry_kv + ekv;
    }
    carry_t += sum_t;
    carry_kv += sum_kv;
  }
  if (tid == 0) {
    s_toff[B] = carry_t;
    s_q0[B] = p.total_q;
  }
  if (carry_t > p.max_tiles || carry_kv > p.kv_total) bad = 1;
  if (__syncthreads_or(bad)) {
    if (blockIdx.x == 0 && tid == 0) {
      p.hdr->num_tiles = 0;
      p.hdr->total_units = 0;
      p.hdr->error = kErrInvalid;
      record_error(p.status, kErrInvalid);
    }
    if (tid == 0) {
      wv->g_tiles = tiles;
      wv->g_ub = ub_out;
      wv->t0 = 0;
      wv->n = 0;
    }
    __syncthreads();
    return WlCounts{0, 0};
  }
  // ---- tiles: thread tid owns the consecutive tiles [t_begin, t_end)
  const int num_tiles = static_cast<int>(carry_t);
  const int per = (num_tiles + nthr - 1) / nthr;
  const int t_begin = min(num_tiles, tid * per), t_end = min(num_tiles, t_begin + per);
  const SeqTables st{s_q0, s_ctx, s_mode, s_toff, s_kvoff};
  int64_t mine = 0;
  for (int t = t_begin; t < t_end; ++t)
    mine += p.seg_weight + make_tile_desc(t, st, B, p.TT, BN, p.window, false, 0).kt_count;
  int64_t U;
  const int64_t ub0 = block_scan_excl(mine, &U, wsum);
  const int P = active_ctas(static_cast<int>(gridDim.x), U);
  int64_t u_beg, u_end;
  cta_range(num_tiles, U, u_beg, u_end);
  // the tile holding this CTA's first unit starts the window (found by the
  // one thread whose tiles hold that unit)
  if (tid == 0) wv->scratch[0] = 0;
  fill_cta_starts(s_cbeg, U, P);
  if (u_beg < u_end && ub0 <= u_beg && u_beg < ub0 + mine) {
    int64_t ub = ub0;
    for (int t = t_begin; t < t_end; ++t) {
      const int64_t len = p.seg_weight + make_tile_desc(t, st, B, p.TT, BN, p.window, false, 0).kt_count;
      if (ub <= u_beg && u_beg < ub + len) wv->scratch[0] = t;
      ub += len;
    }
  }
  __syncthreads();
  const int t0 = wv->scratch[0];
  const int nwin = u_beg < u_end ? min(kWinTiles, num_tiles - t0) : 0;
  int64_t ub = ub0;
  for (int t = t_begin; t < t_end; ++t) {
    TileDesc td = make_tile_desc(t, st, B, p.TT, BN, p.window, false, 0);
    split_tile_desc(td, ub, p.seg_weight, s_cbeg, P, p.rotate != 0);
    tiles[t] = td;
    ub_out[t] = ub;
    const int i = t - t0;
    if (i >= 0 && i < nwin) wv->s_tiles[i] = td;
    if (i >= 0 && i <= nwin) wv->s_ub[i] = ub;
    ub += p.seg_weight + td.kt_count;
  }
  if (tid == 0) {
    ub_out[num_tiles] = U;
    if (t0 + nwin == num_tiles) wv->s_ub[nwin] = U;
    wv->g_tiles = tiles;
    wv->g_ub = ub_out;
    wv->t0 = t0;
    wv->n = nwin;
    if (blockIdx.x == 0) {
      p.hdr->num_tiles = num_tiles;
      p.hdr->total_units = U;
      p.hdr->error = 0;
    }
  }
  __syncthreads();  // the tables and the window are complete for every thread of the CTA
  return WlCounts{U, num_tiles};
}

// The window of a work list the work-list grid wrote: the tile holding this
// CTA's first unit is found by a parallel search of the unit starts (rounds
// of one load per thread, each narrowing the range by the block size), then
// the window's descriptors are copied.  Every thread of the block calls it.
__device__ __noinline__ void load_window(const TileDesc* tiles, const int64_t* ubg, int num_tiles, int64_t U,
                                         WorkView* wv) {
  const int tid = threadIdx.x, nthr = static_cast<int>(blockDim.x);
  int64_t u_beg, u_end;
  cta_range(num_tiles, U, u_beg, u_end);
  int lo = 0, hi = num_tiles;  // the tile holding u_beg is in [lo, hi)
  while (u_beg < u_end && hi - lo > 1) {
    const int stride = (hi - lo + nthr - 1) / nthr;
    if (tid == 0) wv->scratch[0] = lo;
    __syncthreads();
    const int a = lo + tid * stride;
    if (a < hi) {
      const int b = min(hi, a + stride);
      if (ubg[a] <= u_beg && u_beg < ubg[b]) wv->scratch[0] = a;
    }
    __syncthreads();
    lo = wv->scratch[0];
    hi = min(hi, lo + stride);
    __syncthreads();
  }
  const int t0 = lo;
  const int nwin = u_beg < u_end ? min(kWinTiles, num_tiles - t0) : 0;
  if (tid < nwin) wv->s_tiles[tid] = tiles[t0 + tid];
  if (tid <= nwin && u_beg < u_end) wv->s_ub[tid] = ubg[t0 + tid];
  if (tid == 0) {
    wv->g_tiles = tiles;
    wv->g_ub = ubg;
    wv->t0 = t0;
    wv->n = nwin;
  }
  __syncthreads();
}

struct Seg {
  int tile;
  int j0, j1;   // KV-tile range within the tile's range
  int whole;    // segment covers every KV tile of its query tile
  int slot;     // partial slot when not whole
};

// Walks the segments of one CTA's unit range; every role walks the same
// list.  A query tile spans units [ub[t], ub[t+1]); its KV tiles are the units
// from ub[t] + seg_w on, so a range that only touches a tile's first seg_w
// units yields no segment of it.  The walk goes tile by tile from the tile
// holding the range's first unit (every tile has at least one KV tile, so the
// unit starts strictly increase).
struct SegIter {
  const WorkView* wv;
  int t;  // the tile holding unit u
  int64_t u, u_end;
  int cta;
  bool first;
  int seg_w;
  __device__ bool next(Seg& sg) {
    while (u < u_end) {
      const int tt = t;
      const int64_t r0 = wv->ub(tt) + seg_w, t1 = wv->ub(tt + 1);
      const int64_t b = u > r0 ? u : r0;
      const int64_t e = u_end < t1 ? u_end : t1;
      u = e;
      if (e == t1) ++t;
      if (b >= e) continue;
      sg.tile = tt;
      sg.j0 = static_cast<int>(b - r0);
      sg.j1 = static_cast<int>(e - r0);
      sg.whole = (b == r0 && e == t1) ? 1 : 0;
      sg.slot = first ? 2 * cta : 2 * cta + 1;
      first = false;
      return true;
    }
    return false;
  }
};

// The same walk over the global unit starts (a binary search per segment),
// for the kernel shape that reads the work-list grid's tables directly.
__device__ __forceinline__ int tile_of_unit(const int64_t* ub, int num_tiles, int64_t u) {
  int lo = 0, hi = num_tiles - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (ub[mid] <= u) lo = mid; else hi = mid - 1;
  }
  return lo;
}
struct SegIterG {
  const int64_t* ub;
  int num_tiles;
  int64_t u, u_end;
  int cta;
  bool first;
  int seg_w;
  __device__ bool next(Seg& sg) {
    while (u < u_end) {
      const int t = tile_of_unit(ub, num_tiles, u);
      const int64_t r0 = ub[t] + seg_w, t1 = ub[t + 1];
      const int64_t b = u > r0 ? u : r0;
      const int64_t e = u_end < t1 ? u_end : t1;
      u = e;
      if (b >= e) continue;
      sg.tile = t;
      sg.j0 = static_cast<int>(b - r0);
      sg.j1 = static_cast<int>(e - r0);
      sg.whole = (b == r0 && e == t1) ? 1 : 0;
      sg.slot = first ? 2 * cta : 2 * cta + 1;
      first = false;
      return true;
    }
    return false;
  }
};

// Bounded wait on an mbarrier phase.  Returns false (after recording a
// timeout) when the wait expired or another role of the CTA gave up.
__device__ __forceinline__ bool wait_phase(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                           int* status) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    if ((it & 255u) == 0 && global_timer_ns() - t0 > kWaitTimeoutNs) {
      *abort_flag = 1;
      record_error(status, kErrTimeout);
      return false;
    }
  }
}

// Short bounded wait used only while draining after an abort.
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (global_timer_ns() - t0 > kWaitTimeoutNs) return;
  }
}

// Waits for the P and V of one PV together and, in the same rounds, tests the
// K stage of the next QK^T (each test is its own block: measured faster than
// issuing the three tests of a round in one block, 413 vs 769 clocks from the
// last P arrival to the MMA warp seeing it on the max mix).
__device__ __forceinline__ bool wait_pv_probe_k(uint32_t pbar, uint32_t pparity, uint32_t vbar,
                                                uint32_t vparity, uint32_t kbar, uint32_t kparity,
                                                bool& k_ready, volatile int* abort_flag, int* status) {
  bool p_ok = false, v_ok = false;
  uint64_t t0 = 0;
  for (uint32_t it = 0;; ++it) {
    const bool tp = mbar_test_wait(pbar, pparity);
    const bool tv = mbar_test_wait(vbar, vparity);
    const bool tk = mbar_test_wait(kbar, kparity);
    p_ok = p_ok || tp;
    v_ok = v_ok || tv;
    k_ready = k_ready || tk;
    if (p_ok && v_ok) return true;
    if (*abort_flag) return false;
    if (it == 0) {
      t0 = global_timer_ns();
    } else if ((it & 255u) == 0 && global_timer_ns() - t0 > kWaitTimeoutNs) {
      *abort_flag = 1;
      record_error(status, kErrTimeout);
      return false;
    }
  }
}

// -------------------------------------------------------------- main kernel
// Element type of Q, K, V and of P: bf16 (tcgen05 kind::f16) or e4m3
// (kind::f8f6f4).  Sizes in elements of the 128-byte swizzle block, of one
// MMA K step (32 bytes) and of one 32-bit TMEM column.
template <bool F8>
struct Elem {
  static constexpr int SIZE = F8 ? 1 : 2;
  static constexpr int BLK = 128 / SIZE;
  static constexpr int KSTEP = 32 / SIZE;
  static constexpr int PER_WORD = 4 / SIZE;
  // e4m3 P: probabilities are scaled by 2^P_SHIFT so the small ones stay in
  // the normal range, and the running maximum is refreshed once it grew by
  // more than 2^LAZY, so a scaled P never exceeds 2^(LAZY + P_SHIFT) = 256
  // (the largest e4m3 is 448)
  static constexpr int P_SHIFT = F8 ? 5 : 0;
  static constexpr float LAZY = F8 ? 3.f : 8.f;
};

// Shared memory holds the K and V rings and, with QS, the query tile; S, P
// and O (and Q without QS) live in TMEM.
template <int D, int BN, int NK, int NV, bool F8 = false, int NS = 2, bool QS = false>
struct FwdCfg {
  using E = Elem<F8>;
  static constexpr int NKB = D * E::SIZE / 128;      // 128-byte column blocks of head_dim
  static constexpr int KV_BYTES = BN * D * E::SIZE;  // one K (or V) tile
  static constexpr int OFF_K = 0;
  static constexpr int OFF_V = OFF_K + NK * KV_BYTES;
  // QS: the query tile in shared memory, K-major with the 128-byte swizzle
  // (NKB blocks of 128 rows x 128 bytes), read by QK^T in SS form.  That frees
  // Q's TMEM columns for a third S/P buffer.
  static constexpr int OFF_Q = OFF_V + NV * KV_BYTES;
  static constexpr int Q_BYTES = QS ? kRows * D * E::SIZE : 0;
  static constexpr int OFF_BAR = OFF_Q + Q_BYTES;
  // barriers
  // S_FULL[s]: QK^T of the tile in K stage s is done (which also frees that
  // K stage); O_DONE[s]: likewise P.V of the tile in V stage s (which frees
  // that V stage)
  // (with soft release, K_EMPTY / V_EMPTY free the stages instead)
  static constexpr int B_Q_FULL = 0, B_K_FULL = 1, B_V_FULL = 1 + NK,
                       B_S_FULL = 1 + NK + NV, B_P_FULL = B_S_FULL + NK,
                       B_O_DONE = B_P_FULL + NS, B_K_EMPTY = B_O_DONE + NV, B_V_EMPTY = B_K_EMPTY + NK,
                       B_O_FREE = B_V_EMPTY + NV,
                       B_DRAIN = B_O_FREE + 1, NUM_BARS = B_DRAIN + 1;
  static constexpr int OFF_MISC = OFF_BAR + NUM_BARS * 8;
  static constexpr int SMEM_USED = OFF_MISC + 16;
  static constexpr int SMEM_BYTES = SMEM_USED + 1024;  // slack for 1024-byte alignment
  // TMEM columns: O (fp32, D), NS S buffers (fp32, BN; P overwrites the first
  // BN / PER_WORD columns, packed), Q (packed, D / PER_WORD; not with QS).
  // Tile g uses S buffer g % NS; the MMA warp issues QK^T NS - 1 tiles ahead
  // of P.V.
  static constexpr uint32_t TM_O = 0, TM_Q = D + NS * BN;
  static __device__ __forceinline__ uint32_t tm_s(uint32_t g) { return D + (g % NS) * BN; }
  static_assert(D % 64 == 0 && D >= 64 && D <= 256, "head_dim");
  static_assert(BN % 64 == 0 && BN >= 64 && BN <= 256, "kv tile");
  static_assert(NS == 2 || NS == 3, "two or three S/P buffers");
  static_assert(NKB >= 1, "head_dim of at least one 128-byte block");
  // Barrier reuse: S_FULL[g % NK] and O_DONE[g % NV] serve every NK-th (NV-th)
  // tile; a parity wait is sound while the barrier is at most one phase away
  // from the awaited one.  QK^T(g + NK) waits for P(g + NK - NS), so the
  // softmax has seen S(g) before S_FULL moves on when NK >= NS; the rescale
  // wait for PV(g - 1) at tile g needs PV(g - 1 - NV) done, which S(g) seen
  // implies (PV(g - NS) was issued before QK^T(g)) when NV >= NS - 1.
  static_assert(NK >= NS, "S_FULL reuse");
  static_assert(NV >= NS - 1, "O_DONE reuse");
  static_assert(OFF_Q % 1024 == 0, "the swizzled query tile starts on a 1024-byte boundary");
  static_assert(D + NS * BN + (QS ? 0 : D / E::PER_WORD) <= static_cast<int>(kTmemCols), "TMEM budget");
  // (the kernel's WorkView is static shared memory, beside this dynamic part)
  static_assert(SMEM_BYTES + sizeof(WorkView) <= 232448, "shared memory budget");
};

template <int D, int BN, int NK, int NV, bool F8 = false, int NS = 2, bool QS = false>
__global__ void __launch_bounds__(kThreads, 1)
fwd_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
           const FwdParams p) {
  using Cf = FwdCfg<D, BN, NK, NV, F8, NS, QS>;
  using E = Elem<F8>;
  // launched as a programmatic dependent of the work-list grid: the prologue
  // (barriers, TMEM, descriptor prefetch) overlaps that grid, and nothing it
  // wrote is read before it has finished.  The split-KV merge is this grid's
  // own dependent, released once every CTA has passed that wait (so the work
  // list is complete when the merge starts); it becomes resident as CTAs of
  // this grid exit and waits for this grid before reading the partials.
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_base = smem_u32(smem_raw);
  const uint32_t sbase = (raw_base + 1023u) & ~1023u;
  uint8_t* sptr = smem_raw + (sbase - raw_base);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // Soft release (64-key tiles): a softmax thread frees the K and V stages
  // with an arrive once it has seen S(g), so the loaders wait on K_EMPTY /
  // V_EMPTY; measured 1.5% faster there than freeing them through the MMA
  // warp's S_FULL / O_DONE commits, which the larger tiles use.  (It relies
  // on P.V running one tile behind QK^T: two S/P buffers.)
  constexpr bool soft_release = (BN == 64) && (NS == 2);
  constexpr int LA = NS - 1;  // P.V of tile g is issued after QK^T of tile g + LA

  const uint32_t sK = sbase + Cf::OFF_K;
  const uint32_t sV = sbase + Cf::OFF_V;
  const uint32_t sQ = sbase + Cf::OFF_Q;
  const uint32_t bars = sbase + Cf::OFF_BAR;
  auto bar = [&](int i) -> uint32_t { return bars + 8u * static_cast<uint32_t>(i); };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sptr + Cf::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sptr + Cf::OFF_MISC + 4);

  if (threadIdx.x == 0) {
    mbar_init(bar(Cf::B_Q_FULL), kRows);
    // S_FULL / O_DONE count one commit from the MMA warp.  Tile g uses
    // S_FULL[g % NK] and O_DONE[g % NV]: a wait for tile x never aliases,
    // since the next tile on the same barrier, x + NK (x + NV), cannot be
    // issued before P(x) exists.
    for (int s = 0; s < NK; ++s) {
      mbar_init(bar(Cf::B_K_FULL + s), p.k_split ? 2 : 1);
      mbar_init(bar(Cf::B_S_FULL + s), 1);
      mbar_init(bar(Cf::B_K_EMPTY + s), 1);
    }
    for (int s = 0; s < NV; ++s) {
      mbar_init(bar(Cf::B_V_FULL + s), 1);
      mbar_init(bar(Cf::B_O_DONE + s), 1);
      mbar_init(bar(Cf::B_V_EMPTY + s), 1);
    }
    // one P_FULL per S/P buffer in TMEM: tile g uses index g % NS
    for (int s = 0; s < NS; ++s) mbar_init(bar(Cf::B_P_FULL + s), kRows);
    mbar_init(bar(Cf::B_O_FREE), kRows);
    mbar_init(bar(Cf::B_DRAIN), 1);
    *abort_flag = 0;
    fence_barrier_init();
    fence_proxy_async_smem();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  if (warp == kTmaWarp && lane == 0) {
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // all 512 columns of all 128 lanes: the column offsets below are compile-time
  // constants within that range (checked by FwdCfg's static_asserts)
  in_bounds(tmem == 0u, p.status, abort_flag);

  griddep_wait();
  griddep_launch_dependents();
  const int cta = static_cast<int>(blockIdx.x);
  // The work list: built here by every CTA for itself (no work-list grid), or
  // read from the tables the work-list grid wrote; either way the CTA's first
  // tiles land in its shared-memory window.
  // (static shared memory: its address is a constant, so the roles hold no
  // register for it; measured against the window in the dynamic part, the
  // denoise step 1.7 us shorter)
  __shared__ WorkView wv_s;
  WorkView* wv = &wv_s;
  // The e4m3 head_dim-128 shape keeps the walk over the work-list grid's
  // global tables (the host never builds its list in the grid): with the
  // window and the in-grid build its kernel ran 3.7% slower on the max mix
  // (0.722 vs 0.696 ms), a code-generation effect at its 255-register limit
  // that no single part of the change accounted for.
  constexpr bool kGlobalWalk = F8 && D == 128;
  using Iter = std::conditional_t<kGlobalWalk, SegIterG, SegIter>;
  int num_tiles;
  int64_t U;
  if constexpr (kGlobalWalk) {
    num_tiles = p.ws.hdr->num_tiles;
    U = p.ws.hdr->total_units;
  } else if (p.fused_wl) {
    static_assert(NK * Cf::KV_BYTES >= kLocalWlScratch, "work-list scratch in the K ring");
    const WlArgs wa{p.cu_q, p.ctx_len, p.mode, p.ws.hdr, p.status, p.kv_total, p.B, p.total_q, p.Hkv, p.TT,
                    p.window, p.seg_weight, p.max_tiles, p.rotate};
    const WlCounts wc = build_worklist_cta(wa, BN, p.ws.tiles + static_cast<size_t>(cta) * p.tiles_stride,
                                           p.ws.unit_begin + static_cast<size_t>(cta) * p.ub_stride,
                                           sptr + Cf::OFF_K, wv);
    num_tiles = wc.num_tiles;
    U = wc.units;
    // the scratch was the K ring, which the TMA unit (async proxy) writes next
    fence_proxy_async_smem();
    __syncthreads();
  } else {
    num_tiles = p.ws.hdr->num_tiles;
    U = p.ws.hdr->total_units;
    load_window(p.ws.tiles, p.ws.unit_begin, num_tiles, U, wv);
  }
  const int P = U > 0 ? active_ctas(static_cast<int>(gridDim.x), U) : 1;
  // a CTA without work (no tiles, or more CTAs than units) walks an empty
  // range: every role finds nothing to do and the CTA frees its TMEM
  const bool active = num_tiles > 0 && U > 0 && cta < P;
  const int64_t u_beg = active ? cta_unit_begin(cta, U, P) : 0;
  const int64_t u_end = active ? cta_unit_begin(cta + 1, U, P) : 0;

  Iter it = [&]() -> Iter {
    if constexpr (kGlobalWalk) return SegIterG{p.ws.unit_begin, num_tiles, u_beg, u_end, cta, true, p.seg_weight};
    else return SegIter{wv, wv->t0, u_beg, u_end, cta, true, p.seg_weight};
  }();
  auto tile_at = [&](int t) -> TileDesc {
    if constexpr (kGlobalWalk) return p.ws.tiles[t];
    else return wv->tile(t);
  };
  const int G = p.G, TT = p.TT;

  if (warp == kTmaWarp || warp == kVLoadWarp || (warp == kTmaWarp2 && p.k_split)) {
    // ----------------------------------------------------------- producers
    // Warp 4 (with k_split, warps 4 and 7) loads the K ring, warp 6 the V
    // ring, each from this GPU's memory into this CTA's shared memory.  The
    // whole warp runs the loop with warp-uniform control flow; the TMA boxes
    // of one KV tile are spread over the lanes, one box per lane, so that a
    // paged tile's page lookups and box issues run side by side instead of
    // one after the other.
    const bool is_k = (warp != kVLoadWarp);
    const int nkw = is_k && p.k_split ? 2 : 1;       // warps sharing this ring's boxes
    const int kw = (warp == kTmaWarp2) ? 1 : 0;       // this warp's share
    const bool paged = p.block_table != nullptr;
    const int NR = is_k ? NK : NV;  // stages of this ring
    const uint32_t full0 = bar(is_k ? Cf::B_K_FULL : Cf::B_V_FULL);
    // a stage is free once its tile's QK^T (K) or P.V (V) is done
    const uint32_t empty0 = soft_release ? bar(is_k ? Cf::B_K_EMPTY : Cf::B_V_EMPTY)
                                         : bar(is_k ? Cf::B_S_FULL : Cf::B_O_DONE);
    const uint32_t ring = is_k ? sK : sV;
    const void* map = is_k ? static_cast<const void*>(&tm_k) : static_cast<const void*>(&tm_v);
    // boxes of a tile: (BN / box_rows) row blocks x NKB 128-byte column blocks
    // (at most 32: a box holds at least 8 rows, BN * NKB <= 256)
    const int box_rows = paged ? p.page_box : BN;
    const int nbr = BN / box_rows;
    const bool page_box = is_k ? p.k_page_box : p.v_page_box;  // one box per page, every column block
    const int box_i = lane * nkw + kw;              // boxes interleaved over the warps
    const bool has_box = box_i < (page_box ? nbr : nbr * Cf::NKB);
    const int br = page_box ? box_i : box_i % nbr, bk = page_box ? 0 : box_i / nbr;
    const uint32_t box_off = page_box ? static_cast<uint32_t>(br * (Cf::NKB * box_rows * 128))
                                      : static_cast<uint32_t>(bk * (BN * 128) + br * box_rows * 128);
    const uint32_t box_bytes = static_cast<uint32_t>((page_box ? Cf::NKB : 1) * box_rows * 128);
    const int pmask = (1 << p.page_shift) - 1;
    uint32_t stage = 0, phase = 0;
    uint32_t issued_mask = 0, issued_phase = 0;  // per stage: a load was issued / its phase
    int loads = 0;
    bool ok = true;
    Seg sg;
    while (ok && it.next(sg)) {
      const TileDesc td = tile_at(sg.tile);
      if (is_k && kw == 0) {
        // the next segment's Q rows go to L2 while this segment streams, so
        // the softmax warps load them at L2 latency at the segment switch
        Iter look = it;
        Seg nx;
        if (look.next(nx)) {
          const TileDesc tn = tile_at(nx.tile);
          for (int t = lane; t < tn.n_tok; t += 32)
            prefetch_l2_bulk(static_cast<const uint8_t*>(p.q) +
                                 (static_cast<size_t>(tn.q_row0 + t) * p.Hq + tn.kvh * G) * D * E::SIZE,
                             static_cast<uint32_t>(G * D * E::SIZE));
        }
      }
      // positions past the sequence's last key read its last page (checked
      // by the work-list launch); the softmax masks them
      const int last_page = (td.L - 1) >> p.page_shift;
      // This lane's page-table entry for KV tile j; the one for tile j + 1 is
      // read one iteration ahead, so its latency overlaps this tile's wait
      // and box issue (with 16-row pages the issue of a K tile's 16 boxes is
      // what paces the loader).
      auto page_entry = [&](int j, bool& ok_ent) -> int {
        const int pos = kv_tile(td, j) * BN + br * box_rows;
        const int64_t ent = static_cast<int64_t>(td.kv_row0) + min(pos >> p.page_shift, last_page);
        ok_ent = in_bounds(ent >= 0 && ent < p.bt_entries, p.status, abort_flag);
        return ok_ent ? __ldg(p.block_table + ent) : 0;
      };
      bool ok_next = true;
      int page_next = (paged && has_box && sg.j0 < sg.j1) ? page_entry(sg.j0, ok_next) : 0;
      for (int j = sg.j0; j < sg.j1; ++j) {
        const int page_cur = page_next;
        const bool ok_cur = ok_next;
        if (paged && has_box && j + 1 < sg.j1) page_next = page_entry(j + 1, ok_next);
        if (!__all_sync(0xffffffffu, wait_phase(empty0 + 8u * stage, phase ^ 1, abort_flag, p.status))) {
          ok = false;
          break;
        }
        if (is_k && loads++ == p.debug_skip_k_load) {
          if (++stage == static_cast<uint32_t>(NR)) { stage = 0; phase ^= 1; }
          continue;
        }
        // the expected bytes are registered before any box of the stage is issued
        if (lane == 0) mbar_arrive_expect_tx(full0 + 8u * stage, static_cast<uint32_t>(Cf::KV_BYTES / nkw));
        __syncwarp();
        if (has_box) {
          const int pos = kv_tile(td, j) * BN + br * box_rows;
          int row;
          bool ok_box = true;
          if (!paged) {
            row = td.kv_row0 + pos;
          } else {
            ok_box = ok_cur;
            row = (page_cur << p.page_shift) + (pos & pmask);
          }
          if constexpr (kBoundsChecks) {
            if (is_k && loads - 1 == p.debug_bad_kv_row) row += p.kv_rows;
          }
          const uint32_t dst = ring + stage * Cf::KV_BYTES + box_off;
          // a box starts inside the tensor (its rows past the end are zero-filled
          // by the TMA unit and masked) and lands inside its ring stage
          ok_box = ok_box &&
                   in_bounds(row >= 0 && row < p.kv_rows && td.kvh >= 0 && td.kvh < p.Hkv &&
                                 (bk + 1) * E::BLK <= D && (dst & 1023u) == 0u &&
                                 dst + box_bytes <= ring + NR * Cf::KV_BYTES,
                             p.status, abort_flag);
          if (ok_box) {
            if (page_box) tma_load_4d(dst, map, full0 + 8u * stage, 0, td.kvh, row, 0);
            else tma_load_3d(dst, map, full0 + 8u * stage, bk * E::BLK, td.kvh, row);
          }
        }
        issued_mask |= 1u << stage;
        issued_phase = (issued_phase & ~(1u << stage)) | (phase << stage);
        if (++stage == static_cast<uint32_t>(NR)) { stage = 0; phase ^= 1; }
      }
    }
    if (!ok) {
      // let loads already in flight land before the CTA's shared memory goes away
      for (int st = 0; st < NR; ++st)
        if (issued_mask & (1u << st)) drain_wait(full0 + 8u * st, (issued_phase >> st) & 1);
    }
    __syncwarp();
  } else if (warp == kMmaWarp) {
    // ---------------------------------------------------------- MMA issuer
    // per KV tile g: S[g % NS] = Q K^T (A = Q from TMEM), then, LA = NS - 1
    // tiles later, O += P V with P read from TMEM where it overwrote
    // S[g % NS].  MMAs of one thread execute in issue order, so QK(g + NS)
    // may reuse the buffer as soon as PV(g) has been issued.  The whole warp runs this loop with identical
    // (warp-uniform) operands and one elected lane issues each tcgen05 op:
    // issuing from a single divergent lane cost ~100 clocks per MMA.
    //
    // This warp's loop sets the pace: every mbarrier test and every commit
    // costs it 100-300 clocks, against ~1000 clocks of MMAs per tile.  So it
    // tests P, V and the next K together, and commits once per MMA batch: the
    // commit that tells the softmax warps S is ready also frees the K stage,
    // the one that marks P.V done also frees the V stage (or, with soft
    // release, a softmax thread frees both).
    {
      constexpr uint32_t idesc_qk = F8 ? idesc_e4m3_f32(kRows, BN, 0, 0) : idesc_bf16_f32(kRows, BN, 0, 0);
      constexpr uint32_t idesc_pv = F8 ? idesc_e4m3_f32(kRows, D, 0, 1) : idesc_bf16_f32(kRows, D, 0, 1);
      uint32_t k_stage = 0, k_phase = 0, v_stage = 0, v_phase = 0;
      uint32_t gj = 0;
      int seg_i = 0;
      bool ok = true;
      bool k_ready = false;  // the next QK's K stage was seen full by the last probe
      // V tile layout: [column block][BN rows][128 B] (column blocks BN * 128
      // bytes apart, 8-row groups 1024 apart, a K step KSTEP rows further on),
      // or with whole-page boxes [page][column block][page rows][128 B]:
      // column blocks page_box * 128 bytes apart, 8-row groups 1024 apart in a
      // page of one K step and one page (NKB * 1024) apart with 8-row pages, a
      // K step NKB * KSTEP * 128 bytes further on either way
      const uint32_t pv_lbo = p.v_page_box ? p.page_box * 128 : BN * 128;
      const uint32_t pv_sbo = (!F8 && p.v_page_box && p.page_box == 8) ? Cf::NKB * 1024 : 1024;
      const uint32_t pv_step_bytes = p.v_page_box ? Cf::NKB * E::KSTEP * 128 : E::KSTEP * 128;
      Seg sg;
      while (ok && it.next(sg)) {
        if (!__all_sync(0xffffffffu, wait_phase(bar(Cf::B_Q_FULL), seg_i & 1, abort_flag, p.status))) { ok = false; break; }
        tc_fence_after();
        const int n = sg.j1 - sg.j0;
        // e4m3: the loop body twice per iteration (measured: denoise loop
        // 0.1347 vs 0.1358 ms, max mix 0.697 vs 0.709 ms; bf16 was slower so)
        constexpr int kMmaUnroll = F8 ? 2 : 1;
#pragma unroll kMmaUnroll
        for (int jj = 0; jj < n + LA && ok; ++jj) {
          if (jj < n) {
            const uint32_t g = gj + jj;
            if (!k_ready &&
                !__all_sync(0xffffffffu, wait_phase(bar(Cf::B_K_FULL + k_stage), k_phase, abort_flag, p.status))) { ok = false; break; }
            k_ready = false;
            tc_fence_after();
            const uint32_t d_s = tmem + Cf::tm_s(g);
            const uint32_t k_base = sK + k_stage * Cf::KV_BYTES;
            // one batch of four K steps per 128-byte column block of K: A
            // advances 8 TMEM columns, B 32 bytes within the swizzle atom
#pragma unroll
            for (int kb = 0; kb < Cf::NKB; ++kb) {
              // column block kb: BN rows of 128 bytes, or with 8-row page
              // boxes 8 rows per page, pages NKB * 1024 bytes apart
              const uint64_t b = (!F8 && p.k_page_box)
                                     ? smem_desc_sw128(k_base + kb * 1024, 16, Cf::NKB * 1024)
                                     : smem_desc_sw128(k_base + kb * (BN * 128), 16, 1024);
              if constexpr (QS) {
                // A from the query tile in shared memory: 32 bytes per K step
                const uint64_t a = smem_desc_sw128(sQ + kb * (kRows * 128), 16, 1024);
                umma_ss_batch4_warp<F8>(d_s, a, b, idesc_qk, kb > 0 ? 1u : 0u, 2ull, 2ull);
              } else {
                umma_ts_batch_warp<F8, 4>(d_s, tmem + Cf::TM_Q + kb * 32, b, idesc_qk, kb > 0 ? 1u : 0u, 8u,
                                          2ull);
              }
            }
            umma_commit_warp(bar(Cf::B_S_FULL + k_stage));
            if (++k_stage == NK) { k_stage = 0; k_phase ^= 1; }
          }
          if (jj >= LA) {
            const uint32_t g = gj + jj - LA;
            const bool first = (jj == LA);
            if (first && seg_i > 0 &&
                !__all_sync(0xffffffffu, wait_phase(bar(Cf::B_O_FREE), (seg_i - 1) & 1, abort_flag, p.status))) { ok = false; break; }
            // k_stage / k_phase already name the next QK's stage (this segment
            // or the next); at the end of the work that phase never completes
            // and the probe just reads false
            bool kr = k_ready;
            const bool w = wait_pv_probe_k(bar(Cf::B_P_FULL + g % NS), (g / NS) & 1, bar(Cf::B_V_FULL + v_stage),
                                           v_phase, bar(Cf::B_K_FULL + k_stage), k_phase, kr, abort_flag, p.status);
            k_ready = __all_sync(0xffffffffu, kr);
            if (!__all_sync(0xffffffffu, w)) { ok = false; break; }
            tc_fence_after();
            const uint32_t p_tm = tmem + Cf::tm_s(g);
            const uint32_t v_base = sV + v_stage * Cf::KV_BYTES;
            // batches of (up to) four K steps: A advances 8 TMEM columns, B one
            // K step of V rows (KSTEP rows of 128 bytes)
            constexpr int kPvSteps = BN / E::KSTEP;
            constexpr int kPvBatch = kPvSteps % 4 == 0 ? 4 : 2;
            static_assert(kPvSteps % kPvBatch == 0, "P.V steps in batches of 2 or 4");
#pragma unroll
            for (int kb = 0; kb < kPvSteps / kPvBatch; ++kb) {
              const uint64_t b = smem_desc_sw128(v_base + kb * kPvBatch * pv_step_bytes, pv_lbo, pv_sbo);
              umma_ts_batch_warp<F8, kPvBatch>(tmem + Cf::TM_O, p_tm + kb * kPvBatch * 8, b, idesc_pv,
                                               (first && kb == 0) ? 0u : 1u, 8u,
                                               static_cast<uint64_t>(pv_step_bytes / 16));
            }
            umma_commit_warp(bar(Cf::B_O_DONE + v_stage));
            if (++v_stage == NV) { v_stage = 0; v_phase ^= 1; }
          }
        }
        if (!ok) break;
        gj += n;
        ++seg_i;
      }
      // every MMA issued by this thread has finished before TMEM is released
      umma_commit_warp(bar(Cf::B_DRAIN));
      drain_wait(bar(Cf::B_DRAIN), 0);
    }
    __syncwarp();
  } else if (warp < 4) {
    // ---------------------------------- Q load, softmax, epilogue (one row each)
    const int r = threadIdx.x;  // query row of the tile == TMEM lane
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(warp * 32) << 16);
    const int W = p.window;
    const float sl2 = p.scale_log2;
    const int t_row = r / G;
    const int g_row = r - t_row * G;
    uint32_t gj = 0;
    int seg_i = 0;
    bool ok = true;
    // This thread's row of a tile's Q, staged in registers as packed bf16
    // pairs: the loads of the next segment's row are issued at the start of
    // this segment's epilogue and land while O is drained.
    constexpr int kQW = D / E::PER_WORD;  // packed 32-bit words of a Q row
    uint32_t qw[kQW];
    // (rows past the tile's tokens load the last token's row; they write nothing)
    auto q_issue = [&](const TileDesc& t) {
      const int hq = t.kvh * G + (r < G * TT ? g_row : 0);
      const int qr = t.q_row0 + min(t_row, t.n_tok - 1);
      const bool q_ok = in_bounds(qr >= 0 && qr < p.total_q && hq >= 0 && hq < p.Hq, p.status, abort_flag);
      const uint4* src = reinterpret_cast<const uint4*>(
          static_cast<const uint8_t*>(p.q) + (static_cast<size_t>(q_ok ? qr : 0) * p.Hq + (q_ok ? hq : 0)) *
                                                 D * E::SIZE);
#pragma unroll
      for (int e = 0; e < kQW / 4; ++e) {
        const uint4 x = __ldg(src + e);
        qw[4 * e + 0] = x.x; qw[4 * e + 1] = x.y; qw[4 * e + 2] = x.z; qw[4 * e + 3] = x.w;
      }
    };
    // registers -> Q (its TMEM columns, or with QS the shared-memory tile);
    // the MMA warp may start QK^T after this
    auto q_commit = [&]() {
      if constexpr (QS) {
        // row r of each 128-byte column block, its 16-byte chunks placed by the
        // 128-byte swizzle (chunk c of row r at position c ^ (r % 8)), then
        // made visible to the tensor core's (async) proxy
        uint8_t* qrow = sptr + Cf::OFF_Q + r * 128;
#pragma unroll
        for (int kb = 0; kb < Cf::NKB; ++kb)
#pragma unroll
          for (int c = 0; c < 8; ++c)
            *reinterpret_cast<uint4*>(qrow + kb * (kRows * 128) + ((c ^ (r & 7)) << 4)) =
                make_uint4(qw[kb * 32 + 4 * c], qw[kb * 32 + 4 * c + 1], qw[kb * 32 + 4 * c + 2],
                           qw[kb * 32 + 4 * c + 3]);
        fence_proxy_async_smem();
      } else {
#pragma unroll
        for (int c = 0; c < kQW / 32; ++c)
          tmem_st32(lane_base + Cf::TM_Q + c * 32, *reinterpret_cast<uint32_t(*)[32]>(&qw[c * 32]));
        tc_fence_before();
      }
      mbar_arrive(bar(Cf::B_Q_FULL));
    };
    Seg sg;
    bool have = it.next(sg);
    if (have) {
      q_issue(tile_at(sg.tile));
      q_commit();
    }
    // With head_dim 256 and Q in TMEM the register file has room to stage
    // the next row during the epilogue; smaller head dims, and the shared-
    // memory query tile of 128-key e4m3 tiles (whose staged row spilled), load
    // it at the segment start.
    constexpr bool kStageQ = (D == 256) && !QS;
    bool q_loaded = true;  // the first segment's Q is already committed
    while (ok && have) {
      const TileDesc td = tile_at(sg.tile);
      if (!q_loaded) {
        q_issue(td);
        q_commit();
      }
      const int nt = td.n_tok;
      const bool row_ok = (t_row < TT) && (t_row < td.n_tok);
      const int tq = min(t_row, nt - 1);
      const int i = td.pos0 + tq;
      const int lo_r = W < 0 ? INT32_MIN / 2 : i - W;
      const int hi_r = min(td.L - 1, td.causal ? i : (W < 0 ? td.L - 1 : i + W));
      const int i_lo = td.pos0, i_hi = td.pos0 + nt - 1;
      const int lo_all = W < 0 ? INT32_MIN / 2 : i_hi - W;  // largest row lower bound
      const int hi_all = min(td.L - 1, td.causal ? i_lo : (W < 0 ? td.L - 1 : i_lo + W));
      float m_run = -INFINITY, l_run = 0.f;
      const int n = sg.j1 - sg.j0;
      for (int jj = 0; jj < n; ++jj) {
        const uint32_t g = gj + jj;
        const int kv0 = kv_tile(td, sg.j0 + jj) * BN;
        if (!__all_sync(0xffffffffu, wait_phase(bar(Cf::B_S_FULL + g % NK), (g / NK) & 1, abort_flag, p.status))) { ok = false; break; }
        if (soft_release && r == 0) {
          // S(g) complete: QK(g) and every MMA issued before it, PV(g - 2)
          // included, are done, so their K and V stages are free
          mbar_arrive(bar(Cf::B_K_EMPTY + g % NK));
          if (g >= 2) mbar_arrive(bar(Cf::B_V_EMPTY + (g - 2) % NV));
        }
        tc_fence_after();
        uint32_t sr[BN];
        const uint32_t s_addr = lane_base + Cf::tm_s(g);
        if constexpr (BN == 64) tmem_ld64(s_addr, sr);
        else tmem_ld128(s_addr, sr);
        float s[BN];
#pragma unroll
        for (int c = 0; c < BN; ++c) s[c] = __uint_as_float(sr[c]);
        const bool full_tile = (kv0 >= lo_all) && (kv0 + BN - 1 <= hi_all);
        if (!full_tile) {
#pragma unroll
          for (int c = 0; c < BN; ++c) {
            const int key = kv0 + c;
            s[c] = (key >= lo_r && key <= hi_r) ? s[c] : -INFINITY;
          }
        }
        // p = 2^(s * scale * log2(e) - base), two lanes per fp32x2 instruction,
        // packed for P.V; the row sum runs in four independent fp32x2
        // accumulators
        uint32_t pk[BN / E::PER_WORD];
        float rs;
        auto exps = [&](float base) {
          const uint64_t sl2x2 = f32x2(sl2, sl2), nbase2 = f32x2(-base, -base);
          uint64_t acc[4] = {0ull, 0ull, 0ull, 0ull};
#pragma unroll
          for (int c = 0; c < BN; c += 2) {
            float t0, t1;
            f32x2_split(fma_f32x2(f32x2(s[c], s[c + 1]), sl2x2, nbase2), t0, t1);
            const float p0 = ex2_approx(t0), p1 = ex2_approx(t1);
            if constexpr (F8) {
              // e4m3 pairs, two per 32-bit word, lower key in the lower byte
              const uint32_t h = pack_e4m3x2(p0, p1);
              if (((c >> 1) & 1) == 0) pk[c / 4] = h;
              else pk[c / 4] |= h << 16;
            } else {
              pk[c / 2] = pack_bf16x2(p0, p1);
            }
            acc[(c >> 1) & 3] = add_f32x2(acc[(c >> 1) & 3], f32x2(p0, p1));
          }
          float a0, a1, a2, a3, a4, a5, a6, a7;
          f32x2_split(acc[0], a0, a1);
          f32x2_split(acc[1], a2, a3);
          f32x2_split(acc[2], a4, a5);
          f32x2_split(acc[3], a6, a7);
          rs = ((a0 + a1) + (a2 + a3)) + ((a4 + a5) + (a6 + a7));
        };
        // With 128-key tiles the exponentials start against the running
        // maximum, before this tile's maximum is known: while the maximum grows
        // by at most 2^LAZY (every tile but a segment's first few) these are
        // exactly the p the lazy rescale keeps, so they need not wait for the
        // maximum tree, which runs alongside.  A row whose maximum grew by more
        // (or that has none yet) recomputes them against the new maximum.
        // Measured: e4m3 max mix 0.738 -> 0.689 ms, bf16 max mix 1% faster;
        // with 64-key tiles (head_dim 256) the extra live registers spill and
        // the tree is short, so there the maximum comes first.
        constexpr bool kSpeculate = (BN >= 128);
        if constexpr (kSpeculate)
          exps(m_run == -INFINITY ? 0.f : m_run * sl2 - static_cast<float>(E::P_SHIFT));
        // a tree of 3-input maxima (4 levels for 64 keys) instead of one chain
        const float mx = TreeMax<BN>::of(s);
        const float m_new = fmaxf(m_run, mx);
        float m_use = m_run, alpha = 1.f;
        bool rescale = false;
        const bool exact = (m_run == -INFINITY) || ((m_new - m_run) * sl2 > E::LAZY);
        if (exact) {
          m_use = m_new;
          if (m_run != -INFINITY) {
            alpha = ex2_approx((m_run - m_new) * sl2);
            rescale = true;
          }
        }
        if constexpr (kSpeculate) {
          if (__any_sync(0xffffffffu, exact) && exact)
            exps((m_use == -INFINITY) ? 0.f : m_use * sl2 - static_cast<float>(E::P_SHIFT));
        } else {
          exps((m_use == -INFINITY) ? 0.f : m_use * sl2 - static_cast<float>(E::P_SHIFT));
        }
        l_run = l_run * alpha + rs;
        m_run = m_use;
        if (jj > 0 && __any_sync(0xffffffffu, rescale)) {
          // the row maximum grew by more than 2^8: rescale O once PV(g-1) is done
          const uint32_t x = g - 1;
          if (!__all_sync(0xffffffffu, wait_phase(bar(Cf::B_O_DONE + x % NV), (x / NV) & 1, abort_flag, p.status))) { ok = false; break; }
          tc_fence_after();
#pragma unroll 1
          for (int c = 0; c < D / 32; ++c) {
            uint32_t o[32];
            tmem_ld32(lane_base + Cf::TM_O + c * 32, o);
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
            tmem_st32(lane_base + Cf::TM_O + c * 32, o);
          }
        }
        // P row (bf16 pairs) over the first BN/2 columns of this S buffer
        store_packed_p(s_addr, pk);
        tc_fence_before();
        mbar_arrive(bar(Cf::B_P_FULL + g % NS));
      }
      if (!ok) break;
      // ------------------------------------------------------------ epilogue
      // PV(g_last) done implies every earlier MMA of this CTA is done.  A
      // parity wait on O_DONE[x % NV] is only sound once PV(x - NV), the
      // previous commit on that barrier, is done.  S(g_last) seen implies
      // PV(g_last - NS) done; with NV < NS, PV(g_last - 1) is waited for first,
      // which implies PV(g_last - NV) for any NV >= 1.
      {
        const uint32_t x = gj + n - 1;
        bool w = true;
        if constexpr (NV < NS) {
          if (x >= 1) w = wait_phase(bar(Cf::B_O_DONE + (x - 1) % NV), ((x - 1) / NV) & 1, abort_flag, p.status);
        }
        if (!__all_sync(0xffffffffu,
                        w && wait_phase(bar(Cf::B_O_DONE + x % NV), (x / NV) & 1, abort_flag, p.status))) {
          ok = false;
          break;
        }
      }
      tc_fence_after();
      Seg nx;
      Iter look = it;
      const bool more = kStageQ && look.next(nx);
      if (more) q_issue(tile_at(nx.tile));
      const float inv_l = l_run > 0.f ? p.v_scale / l_run : 0.f;
      // l_run sums the probabilities scaled by 2^P_SHIFT
      const float lse_v = l_run > 0.f ? m_run * p.scale + logf(l_run) - E::P_SHIFT * 0.6931471805599453f
                                      : -INFINITY;
      if (sg.whole) {
        const int orow = td.q_row0 + t_row;
        const bool w_ok = !row_ok || in_bounds(orow >= 0 && orow < p.total_q && td.kvh * G + g_row < p.Hq,
                                               p.status, abort_flag);
        __nv_bfloat16* dst = p.out + (static_cast<size_t>(orow) * p.Hq + td.kvh * G + g_row) * D;
#pragma unroll 1
        for (int c = 0; c < D / 32; ++c) {
          uint32_t o[32];
          tmem_ld32(lane_base + Cf::TM_O + c * 32, o);
          if (row_ok && w_ok) {
            uint32_t w[16];
#pragma unroll
            for (int e = 0; e < 16; ++e)
              w[e] = pack_bf16x2(__uint_as_float(o[2 * e]) * inv_l, __uint_as_float(o[2 * e + 1]) * inv_l);
            uint4* d4 = reinterpret_cast<uint4*>(dst + c * 32);
#pragma unroll
            for (int e = 0; e < 4; ++e) d4[e] = make_uint4(w[4 * e], w[4 * e + 1], w[4 * e + 2], w[4 * e + 3]);
          }
        }
        if (row_ok && w_ok && p.lse != nullptr)
          p.lse[static_cast<size_t>(orow) * p.Hq + td.kvh * G + g_row] = lse_v;
      } else {
        const bool s_ok = in_bounds(sg.slot >= 0 && sg.slot < p.num_slots, p.status, abort_flag);
        float* dst = p.ws.part_o + (static_cast<size_t>(sg.slot) * kRows + r) * D;
#pragma unroll 1
        for (int c = 0; c < D / 32; ++c) {
          uint32_t o[32];
          tmem_ld32(lane_base + Cf::TM_O + c * 32, o);
          float4* d4 = reinterpret_cast<float4*>(dst + c * 32);
          if (s_ok) {
#pragma unroll
            for (int e = 0; e < 8; ++e)
              d4[e] = make_float4(__uint_as_float(o[4 * e]) * inv_l, __uint_as_float(o[4 * e + 1]) * inv_l,
                                  __uint_as_float(o[4 * e + 2]) * inv_l, __uint_as_float(o[4 * e + 3]) * inv_l);
          }
        }
        if (s_ok) p.ws.part_lse[static_cast<size_t>(sg.slot) * kRows + r] = lse_v;
      }
      if (more) q_commit();
      tc_fence_before();
      mbar_arrive(bar(Cf::B_O_FREE));
      gj += n;
      ++seg_i;
      have = it.next(sg);
      q_loaded = more;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// ------------------------------------------------------------------ combine
// One warp per (tile, row): the partial LSEs of the CTAs that shared the tile
// are reduced across lanes, then every lane merges its columns.
constexpr int kCombineWarps = 8;

template <int D>
__global__ void __launch_bounds__(kCombineWarps * 32)
combine_kernel(const FwdParams p) {
  // the next call's first grid (work list, or attention) may become
  // resident now: it waits for this grid before it reads or writes memory
  griddep_launch_dependents();
  const int tile = blockIdx.x;
  const int G = p.G;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r = blockIdx.y * kCombineWarps + warp;
  if (r >= G * p.TT) return;
  const int t = r / G, gi = r - t * G;
  // A tile table written by the work-list grid was complete before the
  // attention grid released this grid, so it is read before the wait and
  // only the partials wait for the attention grid (both loads issued
  // together; the descriptor of a tile past num_tiles is stale but lies
  // inside the workspace and is not used).  A table the attention grid built
  // itself is complete only once that grid has finished: read after the wait.
  const bool early = !p.fused_wl;
  if (!early) griddep_wait();
  const int num_tiles = p.ws.hdr->num_tiles;
  const TileDesc td = p.ws.tiles[tile];
  if (tile >= num_tiles || td.comb_n <= 1) return;  // no tile, or written directly by one CTA
  if (t >= td.n_tok) return;
  if (early) griddep_wait();
  const int nc = td.comb_n;
  // partial slot of contributor i: the first CTA's is recorded, the others
  // hold the tile in their first segment
  auto slot_of = [&](int i) { return i == 0 ? td.comb_slot0 : 2 * (td.comb_cta + i); };
  constexpr int E = D / 32;  // columns per lane
  const int orow = td.q_row0 + t;
  const int h = td.kvh * G + gi;
  // every partial slot this row reads and the row it writes
  if (!in_bounds(orow >= 0 && orow < p.total_q && h < p.Hq && td.comb_slot0 >= 0 &&
                     td.comb_slot0 < p.num_slots && slot_of(nc - 1) < p.num_slots,
                 p.status, nullptr))
    return;
  __nv_bfloat16* dst = p.out + (static_cast<size_t>(orow) * p.Hq + h) * D;
  if (nc <= 4) {
    // the usual case: every load of the row (up to four contributors' LSE and
    // columns) is issued at once, one memory round trip in all
    float lw[4];
    float acc4[4][E];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int sl = slot_of(min(u, nc - 1));
      lw[u] = u < nc ? p.ws.part_lse[static_cast<size_t>(sl) * kRows + r] : -INFINITY;
      const float* src = p.ws.part_o + (static_cast<size_t>(sl) * kRows + r) * D;
      if constexpr (E % 4 == 0) {
#pragma unroll
        for (int k = 0; k < E / 4; ++k) {
          const float4 x = u < nc ? *reinterpret_cast<const float4*>(src + (k * 32 + lane) * 4)
                                  : make_float4(0.f, 0.f, 0.f, 0.f);
          acc4[u][4 * k + 0] = x.x;
          acc4[u][4 * k + 1] = x.y;
          acc4[u][4 * k + 2] = x.z;
          acc4[u][4 * k + 3] = x.w;
        }
      } else {
        const float2 x = u < nc ? *reinterpret_cast<const float2*>(src + lane * 2) : make_float2(0.f, 0.f);
        acc4[u][0] = x.x;
        acc4[u][1] = x.y;
      }
    }
    const float M4 = fmaxf(fmaxf(lw[0], lw[1]), fmaxf(lw[2], lw[3]));
    float wsum4 = 0.f, acc[E];
#pragma unroll
    for (int e = 0; e < E; ++e) acc[e] = 0.f;
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const float w = lw[u] == -INFINITY ? 0.f : __expf(lw[u] - M4);
      wsum4 += w;
#pragma unroll
      for (int e = 0; e < E; ++e) acc[e] += w * acc4[u][e];
    }
    const float inv4 = wsum4 > 0.f ? 1.f / wsum4 : 0.f;
    if constexpr (E % 4 == 0) {
#pragma unroll
      for (int k = 0; k < E / 4; ++k) {
        const uint32_t w0 = pack_bf16x2(acc[4 * k + 0] * inv4, acc[4 * k + 1] * inv4);
        const uint32_t w1 = pack_bf16x2(acc[4 * k + 2] * inv4, acc[4 * k + 3] * inv4);
        *reinterpret_cast<uint2*>(dst + (k * 32 + lane) * 4) = make_uint2(w0, w1);
      }
    } else {
      *reinterpret_cast<uint32_t*>(dst + lane * 2) = pack_bf16x2(acc[0] * inv4, acc[1] * inv4);
    }
    if (lane == 0 && p.lse != nullptr)
      p.lse[static_cast<size_t>(orow) * p.Hq + h] = wsum4 > 0.f ? M4 + logf(wsum4) : -INFINITY;
    return;
  }
  // every contributor's LSE at once (lane i holds contributors i, i + 32, ...)
  float M = -INFINITY;
  for (int i = lane; i < nc; i += 32)
    M = fmaxf(M, p.ws.part_lse[static_cast<size_t>(slot_of(i)) * kRows + r]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  float acc[E];
#pragma unroll
  for (int e = 0; e < E; ++e) acc[e] = 0.f;
  float wsum = 0.f;
  for (int i0 = 0; i0 < nc; i0 += 32) {
    // lane j: weight and slot of contributor i0 + j
    const int cj = i0 + lane;
    const int sj = cj < nc ? slot_of(cj) : 0;
    const float lj = cj < nc ? p.ws.part_lse[static_cast<size_t>(sj) * kRows + r] : -INFINITY;
    const float wj = lj == -INFINITY ? 0.f : __expf(lj - M);
    float ws = wj;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ws += __shfl_xor_sync(0xffffffffu, ws, o);
    wsum += ws;
    const int nb = min(32, nc - i0);
    // four contributors' rows in flight at a time
    for (int b = 0; b < nb; b += 4) {
      float w[4];
      const float* src[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int j = min(b + u, nb - 1);
        w[u] = b + u < nb ? __shfl_sync(0xffffffffu, wj, j) : 0.f;
        const int sl = __shfl_sync(0xffffffffu, sj, j);
        src[u] = p.ws.part_o + (static_cast<size_t>(sl) * kRows + r) * D;
      }
      if constexpr (E % 4 == 0) {
        float4 x[4][E / 4];
#pragma unroll
        for (int u = 0; u < 4; ++u)
#pragma unroll
          for (int k = 0; k < E / 4; ++k) x[u][k] = *reinterpret_cast<const float4*>(src[u] + (k * 32 + lane) * 4);
#pragma unroll
        for (int u = 0; u < 4; ++u)
#pragma unroll
          for (int k = 0; k < E / 4; ++k) {
            acc[4 * k + 0] += w[u] * x[u][k].x;
            acc[4 * k + 1] += w[u] * x[u][k].y;
            acc[4 * k + 2] += w[u] * x[u][k].z;
            acc[4 * k + 3] += w[u] * x[u][k].w;
          }
      } else {
        float2 x[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) x[u] = *reinterpret_cast<const float2*>(src[u] + lane * 2);
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          acc[0] += w[u] * x[u].x;
          acc[1] += w[u] * x[u].y;
        }
      }
    }
  }
  const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
  if constexpr (E % 4 == 0) {
#pragma unroll
    for (int k = 0; k < E / 4; ++k) {
      const uint32_t w0 = pack_bf16x2(acc[4 * k + 0] * inv, acc[4 * k + 1] * inv);
      const uint32_t w1 = pack_bf16x2(acc[4 * k + 2] * inv, acc[4 * k + 3] * inv);
      *reinterpret_cast<uint2*>(dst + (k * 32 + lane) * 4) = make_uint2(w0, w1);
    }
  } else {
    *reinterpret_cast<uint32_t*>(dst + lane * 2) = pack_bf16x2(acc[0] * inv, acc[1] * inv);
  }
  if (lane == 0 && p.lse != nullptr)
    p.lse[static_cast<size_t>(orow) * p.Hq + h] = wsum > 0.f ? M + logf(wsum) : -INFINITY;
}

}  // namespace dg
