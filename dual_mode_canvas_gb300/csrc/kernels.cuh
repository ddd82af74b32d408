// Device side of the dual-mode attention forward pass.
//
//   build_worklist_kernel  one CTA: validates cu_q / ctx_len / mode, cuts every
//                          (sequence, KV head) into 128-row query tiles and
//                          computes each tile's visible KV-tile range; the
//                          range is the union of the rows' windows (causal:
//                          keys <= i, bidirectional: the whole sequence, both
//                          narrowed to [i-W, i+W] on sliding-window layers).
//   fwd_kernel<D,BN,NK,NV> persistent, one CTA per SM.  The (tile, KV-tile)
//                          work units are split evenly over the CTAs; a tile
//                          cut between CTAs leaves fp32 partials + LSE.
//                          Warp roles: warps 4 and 6 issue TMA loads (Q + K
//                          ring, V ring), warp 5 issues tcgen05 MMAs, warps
//                          0-3 (one TMEM lane = one query row each) run the
//                          online softmax and the epilogue.
//   combine_kernel<D>      merges the partials of cut tiles by their LSE.
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

#include "ptx.cuh"

namespace dg {

constexpr int kRows = 128;          // query rows per tile (UMMA M, TMEM lanes)
constexpr int kThreads = 224;       // 4 softmax warps + Q/K loader + MMA issuer + V loader
constexpr int kTmaWarp = 4;         // loads Q and the K ring
constexpr int kMmaWarp = 5;         // issues tcgen05 MMAs, owns TMEM
constexpr int kVLoadWarp = 6;       // loads the V ring
constexpr uint32_t kTmemCols = 512;
constexpr uint64_t kWaitTimeoutNs = 250ull * 1000ull * 1000ull;

// error codes shared with the host (same values as dg_status_t)
constexpr int kErrInvalid = 1;
constexpr int kErrTimeout = 5;

struct TileDesc {
  int32_t q_row0;    // global query row of the tile's first token
  int32_t n_tok;     // query tokens in the tile (1 .. TT)
  int32_t kv_row0;   // global K/V row of the sequence's first key
  int32_t pos0;      // absolute position of the tile's first token
  int32_t L;         // keys of the sequence (context + queries)
  int32_t kt_first;  // first KV tile touched (units of BN keys, sequence-relative)
  int32_t kvh;       // KV head
  int32_t causal;    // 1 causal (encoder), 0 bidirectional (denoise)
};

struct WorkHeader {
  int32_t num_tiles;
  int32_t error;
  int64_t total_units;
};

struct Workspace {
  WorkHeader* hdr;
  int64_t* seq_tile_off;   // [B + 1]
  int64_t* seq_kv_off;     // [B + 1]
  TileDesc* tiles;         // [max_tiles]
  int64_t* unit_begin;     // [max_tiles + 1]
  float* part_lse;         // [2 * num_ctas][128]
  float* part_o;           // [2 * num_ctas][128][D]
};

struct FwdParams {
  Workspace ws;
  __nv_bfloat16* out;
  float* lse;
  int* status;
  int Hq, G, TT, window;
  float scale, scale_log2;
};

__device__ __forceinline__ void record_error(int* status, int code) {
  atomicCAS(status, 0, code);
}

// ------------------------------------------------------------ block scan
// In-place exclusive scan of data[0..n) (int64); data[n] receives the total.
// Must be called by every thread of a 1024-thread block.
__device__ void block_exclusive_scan(int64_t* data, int n) {
  __shared__ int64_t warp_sums[32];
  __shared__ int64_t carry;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) carry = 0;
  __syncthreads();
  for (int base = 0; base < n; base += 1024) {
    const int idx = base + tid;
    int64_t x = idx < n ? data[idx] : 0;
    int64_t incl = x;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int64_t y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    if (lane == 31) warp_sums[warp] = incl;
    __syncthreads();
    if (warp == 0) {
      int64_t w = warp_sums[lane];
      int64_t wi = w;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        int64_t y = __shfl_up_sync(0xffffffffu, wi, o);
        if (lane >= o) wi += y;
      }
      warp_sums[lane] = wi - w;  // exclusive prefix of warp totals
    }
    __syncthreads();
    const int64_t c0 = carry;
    if (idx < n) data[idx] = c0 + warp_sums[warp] + incl - x;
    __syncthreads();
    if (tid == 1023) carry = c0 + warp_sums[31] + incl;
    __syncthreads();
  }
  if (tid == 0) data[n] = carry;
  __syncthreads();
}

// ------------------------------------------------------ work-list builder
__global__ void __launch_bounds__(1024, 1)
build_worklist_kernel(const int32_t* __restrict__ cu_q, const int32_t* __restrict__ ctx_len,
                      const uint8_t* __restrict__ mode, int B, int total_q, int total_kv, int Hkv,
                      int TT, int BN, int window, int max_tiles, Workspace ws, int* status) {
  __shared__ int bad;
  const int tid = threadIdx.x;
  if (tid == 0) bad = (cu_q[0] != 0 || cu_q[B] != total_q) ? 1 : 0;
  __syncthreads();
  for (int s = tid; s < B; s += 1024) {
    const int n = cu_q[s + 1] - cu_q[s];
    const int c = ctx_len[s];
    const int md = mode[s];
    if (n < 0 || c < 0 || md > 1) atomicOr(&bad, 1);
    const int64_t nn = n < 0 ? 0 : n;
    ws.seq_tile_off[s] = static_cast<int64_t>(Hkv) * ((nn + TT - 1) / TT);
    ws.seq_kv_off[s] = static_cast<int64_t>(c < 0 ? 0 : c) + nn;
  }
  __syncthreads();
  block_exclusive_scan(ws.seq_tile_off, B);
  block_exclusive_scan(ws.seq_kv_off, B);
  if (tid == 0) {
    if (ws.seq_tile_off[B] > max_tiles || ws.seq_kv_off[B] > total_kv) bad = 1;
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
  const int num_tiles = static_cast<int>(ws.seq_tile_off[B]);
  for (int tile = tid; tile < num_tiles; tile += 1024) {
    // sequence owning this tile: largest s with seq_tile_off[s] <= tile
    int lo = 0, hi = B - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (ws.seq_tile_off[mid] <= tile) lo = mid; else hi = mid - 1;
    }
    const int s = lo;
    const int n = cu_q[s + 1] - cu_q[s];
    const int c = ctx_len[s];
    const int L = c + n;
    const bool causal = mode[s] == 0;
    const int m_tiles = (n + TT - 1) / TT;
    const int local = tile - static_cast<int>(ws.seq_tile_off[s]);
    const int kvh = local / m_tiles;
    const int mt = local - kvh * m_tiles;
    const int t0 = mt * TT;
    const int n_tok = min(TT, n - t0);
    const int pos0 = c + t0;
    const int i_max = pos0 + n_tok - 1;
    const int kv_lo = window < 0 ? 0 : max(0, pos0 - window);
    const int kv_hi = causal ? i_max : (window < 0 ? L - 1 : min(L - 1, i_max + window));
    TileDesc td;
    td.q_row0 = cu_q[s] + t0;
    td.n_tok = n_tok;
    td.kv_row0 = static_cast<int>(ws.seq_kv_off[s]);
    td.pos0 = pos0;
    td.L = L;
    td.kt_first = kv_lo / BN;
    td.kvh = kvh;
    td.causal = causal ? 1 : 0;
    ws.tiles[tile] = td;
    ws.unit_begin[tile] = kv_hi / BN - kv_lo / BN + 1;
  }
  __syncthreads();
  block_exclusive_scan(ws.unit_begin, num_tiles);
  if (tid == 0) {
    ws.hdr->num_tiles = num_tiles;
    ws.hdr->total_units = ws.unit_begin[num_tiles];
    ws.hdr->error = 0;
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

// CTA whose unit range contains unit u (ranges are [begin(c), begin(c+1))).
__device__ __forceinline__ int cta_of_unit(int64_t u, int64_t U, int P) {
  int c = static_cast<int>((u * P) / U);
  if (c > P - 1) c = P - 1;
  while (c + 1 < P && cta_unit_begin(c + 1, U, P) <= u) ++c;
  while (c > 0 && cta_unit_begin(c, U, P) > u) --c;
  return c;
}

// Tile containing unit u: largest t with unit_begin[t] <= u.
__device__ __forceinline__ int tile_of_unit(const int64_t* ub, int num_tiles, int64_t u) {
  int lo = 0, hi = num_tiles - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (ub[mid] <= u) lo = mid; else hi = mid - 1;
  }
  return lo;
}

struct Seg {
  int tile;
  int j0, j1;   // KV-tile range within the tile's range
  int whole;    // segment covers every KV tile of its tile
  int slot;     // partial slot when not whole
};

// Walks the segments of one CTA's unit range; every role walks the same list.
struct SegIter {
  const int64_t* ub;
  int num_tiles;
  int64_t u, u_end;
  int cta;
  bool first;
  __device__ bool next(Seg& sg) {
    if (u >= u_end) return false;
    const int t = tile_of_unit(ub, num_tiles, u);
    const int64_t t0 = ub[t], t1 = ub[t + 1];
    const int64_t e = u_end < t1 ? u_end : t1;
    sg.tile = t;
    sg.j0 = static_cast<int>(u - t0);
    sg.j1 = static_cast<int>(e - t0);
    sg.whole = (u == t0 && e == t1) ? 1 : 0;
    sg.slot = first ? 2 * cta : 2 * cta + 1;
    u = e;
    first = false;
    return true;
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

// -------------------------------------------------------------- main kernel
template <int D, int BN, int NK, int NV>
struct FwdCfg {
  static constexpr int NKB = D / 64;                 // 128-byte column blocks of head_dim
  static constexpr int Q_BYTES = kRows * D * 2;
  static constexpr int KV_BYTES = BN * D * 2;        // one K (or V) tile
  static constexpr int P_BYTES = kRows * BN * 2;
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_K = OFF_Q + Q_BYTES;
  static constexpr int OFF_V = OFF_K + NK * KV_BYTES;
  static constexpr int OFF_P = OFF_V + NV * KV_BYTES;
  static constexpr int OFF_BAR = OFF_P + P_BYTES;
  // barriers
  static constexpr int B_Q_FULL = 0, B_Q_EMPTY = 1, B_K_FULL = 2, B_K_EMPTY = 2 + NK,
                       B_V_FULL = 2 + 2 * NK, B_V_EMPTY = 2 + 2 * NK + NV,
                       B_S_FULL = 2 + 2 * NK + 2 * NV, B_S_FREE = B_S_FULL + 2,
                       B_P_FULL = B_S_FREE + 2, B_O_DONE = B_P_FULL + 1, B_O_FREE = B_O_DONE + 1,
                       B_DRAIN = B_O_FREE + 1, NUM_BARS = B_DRAIN + 1;
  static constexpr int OFF_MISC = OFF_BAR + NUM_BARS * 8;
  static constexpr int SMEM_USED = OFF_MISC + 16;
  static constexpr int SMEM_BYTES = SMEM_USED + 1024;  // slack for 1024-byte alignment
  // TMEM columns
  static constexpr uint32_t TM_O = 0, TM_S0 = D, TM_S1 = D + BN;
  static_assert(D % 64 == 0 && D >= 64 && D <= 256, "head_dim");
  static_assert(BN % 64 == 0 && BN >= 64 && BN <= 256, "kv tile");
  static_assert(D + 2 * BN <= static_cast<int>(kTmemCols), "TMEM budget");
  static_assert(SMEM_BYTES <= 232448, "shared memory budget");
};

template <int D, int BN, int NK, int NV>
__global__ void __launch_bounds__(kThreads, 1)
fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
           const __grid_constant__ CUtensorMap tm_v, const FwdParams p) {
  using C = FwdCfg<D, BN, NK, NV>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_base = smem_u32(smem_raw);
  const uint32_t sbase = (raw_base + 1023u) & ~1023u;
  uint8_t* sptr = smem_raw + (sbase - raw_base);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  const WorkHeader* hdr = p.ws.hdr;
  const int num_tiles = hdr->num_tiles;
  const int64_t U = hdr->total_units;
  const int cta = blockIdx.x;
  if (num_tiles <= 0 || U <= 0) return;  // uniform over the CTA
  const int P = active_ctas(gridDim.x, U);
  if (cta >= P) return;
  const int64_t u_beg = cta_unit_begin(cta, U, P);
  const int64_t u_end = cta_unit_begin(cta + 1, U, P);

  const uint32_t sQ = sbase + C::OFF_Q;
  const uint32_t sK = sbase + C::OFF_K;
  const uint32_t sV = sbase + C::OFF_V;
  const uint32_t sP = sbase + C::OFF_P;
  const uint32_t bars = sbase + C::OFF_BAR;
  auto bar = [&](int i) -> uint32_t { return bars + 8u * static_cast<uint32_t>(i); };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sptr + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sptr + C::OFF_MISC + 4);

  if (threadIdx.x == 0) {
    mbar_init(bar(C::B_Q_FULL), 1);
    mbar_init(bar(C::B_Q_EMPTY), 1);
    for (int s = 0; s < NK; ++s) {
      mbar_init(bar(C::B_K_FULL + s), 1);
      mbar_init(bar(C::B_K_EMPTY + s), 1);
    }
    for (int s = 0; s < NV; ++s) {
      mbar_init(bar(C::B_V_FULL + s), 1);
      mbar_init(bar(C::B_V_EMPTY + s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar(C::B_S_FULL + b), 1);
      mbar_init(bar(C::B_S_FREE + b), kRows);
    }
    mbar_init(bar(C::B_P_FULL), kRows);
    mbar_init(bar(C::B_O_DONE), 1);
    mbar_init(bar(C::B_O_FREE), kRows);
    mbar_init(bar(C::B_DRAIN), 1);
    *abort_flag = 0;
    fence_barrier_init();
    fence_proxy_async_smem();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  if (warp == kTmaWarp && lane == 0) {
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  SegIter it{p.ws.unit_begin, num_tiles, u_beg, u_end, cta, true};
  const int G = p.G, TT = p.TT;

  if (warp == kTmaWarp || warp == kVLoadWarp) {
    // ----------------------------------------------------------- producers
    // warp 4 loads each segment's Q tile and the K ring, warp 6 the V ring,
    // so a K tile is fetched as soon as its slot's QK^T has retired
    if (lane == 0) {
      const bool is_k = (warp == kTmaWarp);
      const uint32_t q_tx = static_cast<uint32_t>(C::NKB * 64 * G * TT * 2);
      const uint32_t t_tx = static_cast<uint32_t>(C::NKB * 64 * BN * 2);
      const int NS = is_k ? NK : NV;
      const uint32_t full0 = bar(is_k ? C::B_K_FULL : C::B_V_FULL);
      const uint32_t empty0 = bar(is_k ? C::B_K_EMPTY : C::B_V_EMPTY);
      const uint32_t ring = is_k ? sK : sV;
      const void* map = is_k ? static_cast<const void*>(&tm_k) : static_cast<const void*>(&tm_v);
      uint32_t stage = 0, phase = 0;
      int seg_i = 0;
      int q_issued_seg = -1;
      uint32_t issued_mask = 0, issued_phase = 0;  // per stage: a load was issued / its phase
      bool ok = true;
      Seg sg;
      while (ok && it.next(sg)) {
        const TileDesc td = p.ws.tiles[sg.tile];
        if (is_k) {
          if (!wait_phase(bar(C::B_Q_EMPTY), (seg_i & 1) ^ 1, abort_flag, p.status)) { ok = false; break; }
          mbar_arrive_expect_tx(bar(C::B_Q_FULL), q_tx);
#pragma unroll
          for (int kb = 0; kb < C::NKB; ++kb)
            tma_load_3d(sQ + kb * (kRows * 128), &tm_q, bar(C::B_Q_FULL), kb * 64, td.kvh * G,
                        td.q_row0);
          q_issued_seg = seg_i;
        }
        for (int j = sg.j0; j < sg.j1; ++j) {
          if (!wait_phase(empty0 + 8u * stage, phase ^ 1, abort_flag, p.status)) { ok = false; break; }
          mbar_arrive_expect_tx(full0 + 8u * stage, t_tx);
          const int row = td.kv_row0 + (td.kt_first + j) * BN;
#pragma unroll
          for (int kb = 0; kb < C::NKB; ++kb)
            tma_load_3d(ring + stage * C::KV_BYTES + kb * (BN * 128), map, full0 + 8u * stage, kb * 64,
                        td.kvh, row);
          issued_mask |= 1u << stage;
          issued_phase = (issued_phase & ~(1u << stage)) | (phase << stage);
          if (++stage == static_cast<uint32_t>(NS)) { stage = 0; phase ^= 1; }
        }
        ++seg_i;
      }
      if (!ok) {
        // let loads already in flight land before the CTA's shared memory goes away
        if (q_issued_seg >= 0) drain_wait(bar(C::B_Q_FULL), q_issued_seg & 1);
        for (int st = 0; st < NS; ++st)
          if (issued_mask & (1u << st)) drain_wait(full0 + 8u * st, (issued_phase >> st) & 1);
      }
    }
    __syncwarp();
  } else if (warp == kMmaWarp) {
    // ---------------------------------------------------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_qk = idesc_bf16_f32(kRows, BN, 0, 0);
      constexpr uint32_t idesc_pv = idesc_bf16_f32(kRows, D, 0, 1);
      uint32_t k_stage = 0, k_phase = 0, v_stage = 0, v_phase = 0;
      uint32_t gj = 0;
      int seg_i = 0;
      bool ok = true;
      Seg sg;
      while (ok && it.next(sg)) {
        if (!wait_phase(bar(C::B_Q_FULL), seg_i & 1, abort_flag, p.status)) { ok = false; break; }
        tc_fence_after();
        const int n = sg.j1 - sg.j0;
        for (int jj = 0; jj <= n && ok; ++jj) {
          if (jj < n) {
            // S[g & 1] = Q K^T
            const uint32_t g = gj + jj;
            if (!wait_phase(bar(C::B_K_FULL + k_stage), k_phase, abort_flag, p.status) ||
                !wait_phase(bar(C::B_S_FREE + (g & 1)), ((g >> 1) & 1) ^ 1, abort_flag, p.status)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t d_s = tmem + ((g & 1) ? C::TM_S1 : C::TM_S0);
            const uint32_t k_base = sK + k_stage * C::KV_BYTES;
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
              const uint64_t a = smem_desc_sw128(sQ + (kk >> 2) * (kRows * 128) + (kk & 3) * 32, 16, 1024);
              const uint64_t b = smem_desc_sw128(k_base + (kk >> 2) * (BN * 128) + (kk & 3) * 32, 16, 1024);
              umma_bf16_ss(d_s, a, b, idesc_qk, kk > 0 ? 1u : 0u);
            }
            umma_commit(bar(C::B_S_FULL + (g & 1)));
            umma_commit(bar(C::B_K_EMPTY + k_stage));
            if (++k_stage == NK) { k_stage = 0; k_phase ^= 1; }
          }
          if (jj >= 1) {
            // O (+)= P V
            const uint32_t g = gj + jj - 1;
            const bool first = (jj == 1);
            if (first && seg_i > 0 &&
                !wait_phase(bar(C::B_O_FREE), (seg_i - 1) & 1, abort_flag, p.status)) { ok = false; break; }
            if (!wait_phase(bar(C::B_P_FULL), g & 1, abort_flag, p.status) ||
                !wait_phase(bar(C::B_V_FULL + v_stage), v_phase, abort_flag, p.status)) { ok = false; break; }
            tc_fence_after();
            const uint32_t v_base = sV + v_stage * C::KV_BYTES;
#pragma unroll
            for (int kk = 0; kk < BN / 16; ++kk) {
              const uint64_t a = smem_desc_sw128(sP + (kk >> 2) * (kRows * 128) + (kk & 3) * 32, 16, 1024);
              const uint64_t b = smem_desc_sw128(v_base + kk * 2048, BN * 128, 1024);
              umma_bf16_ss(tmem + C::TM_O, a, b, idesc_pv, (first && kk == 0) ? 0u : 1u);
            }
            umma_commit(bar(C::B_O_DONE));
            umma_commit(bar(C::B_V_EMPTY + v_stage));
            if (++v_stage == NV) { v_stage = 0; v_phase ^= 1; }
          }
        }
        if (!ok) break;
        umma_commit(bar(C::B_Q_EMPTY));
        gj += n;
        ++seg_i;
      }
      // every MMA issued by this thread has finished before TMEM is released
      umma_commit(bar(C::B_DRAIN));
      drain_wait(bar(C::B_DRAIN), 0);
    }
    __syncwarp();
  } else if (warp < 4) {
    // -------------------------------------------- softmax + epilogue (rows)
    const int r = threadIdx.x;  // query row of the tile == TMEM lane
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(warp * 32) << 16);
    const int W = p.window;
    const float sl2 = p.scale_log2;
    const int t_row = r / G;
    const int g_row = r - t_row * G;
    uint32_t gj = 0;
    int seg_i = 0;
    bool ok = true;
    Seg sg;
    while (ok && it.next(sg)) {
      const TileDesc td = p.ws.tiles[sg.tile];
      const bool row_ok = (t_row < TT) && (t_row < td.n_tok);
      const int i = td.pos0 + min(t_row, td.n_tok - 1);
      const int lo_r = W < 0 ? INT32_MIN / 2 : i - W;
      const int hi_r = min(td.L - 1, td.causal ? i : (W < 0 ? td.L - 1 : i + W));
      const int i_lo = td.pos0, i_hi = td.pos0 + td.n_tok - 1;
      const int lo_all = W < 0 ? INT32_MIN / 2 : i_hi - W;  // largest row lower bound
      const int hi_all = min(td.L - 1, td.causal ? i_lo : (W < 0 ? td.L - 1 : i_lo + W));
      // l_run: sum of the bf16 weights the PV MMA used (normalises O);
      // l_lse: the same sum before rounding (gives the LSE)
      float m_run = -INFINITY, l_run = 0.f, l_lse = 0.f;
      const int n = sg.j1 - sg.j0;
      for (int jj = 0; jj < n; ++jj) {
        const uint32_t g = gj + jj;
        const int kv0 = (td.kt_first + sg.j0 + jj) * BN;
        if (!__all_sync(0xffffffffu, wait_phase(bar(C::B_S_FULL + (g & 1)), (g >> 1) & 1, abort_flag, p.status))) { ok = false; break; }
        tc_fence_after();
        uint32_t sr[BN];
        const uint32_t s_addr = lane_base + ((g & 1) ? C::TM_S1 : C::TM_S0);
#pragma unroll
        for (int c = 0; c < BN / 32; ++c)
          tmem_ld32(s_addr + c * 32, *reinterpret_cast<uint32_t(*)[32]>(&sr[c * 32]));
        tc_fence_before();
        mbar_arrive(bar(C::B_S_FREE + (g & 1)));
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
        float mx = s[0];
#pragma unroll
        for (int c = 1; c < BN; ++c) mx = fmaxf(mx, s[c]);
        const float m_new = fmaxf(m_run, mx);
        float m_use = m_run, alpha = 1.f;
        bool rescale = false;
        if (m_run == -INFINITY) {
          m_use = m_new;
        } else if ((m_new - m_run) * sl2 > 8.f) {
          m_use = m_new;
          alpha = ex2_approx((m_run - m_new) * sl2);
          rescale = true;
        }
        const float base = (m_use == -INFINITY) ? 0.f : m_use * sl2;
        float rs = 0.f, rs_exact = 0.f;
        uint32_t pk[BN / 2];
#pragma unroll
        for (int c = 0; c < BN; c += 2) {
          const float p0 = ex2_approx(fmaf(s[c], sl2, -base));
          const float p1 = ex2_approx(fmaf(s[c + 1], sl2, -base));
          const uint32_t w = pack_bf16x2(p0, p1);
          pk[c / 2] = w;
          // normalise O by the bf16 weights the PV MMA multiplies, so O / l
          // stays a convex combination of the value rows
          rs += __uint_as_float(w << 16) + __uint_as_float(w & 0xFFFF0000u);
          rs_exact += p0 + p1;
        }
        l_run = l_run * alpha + rs;
        l_lse = l_lse * alpha + rs_exact;
        m_run = m_use;
        if (jj > 0) {
          // PV of the previous tile has finished: P buffer free, O stable
          if (!__all_sync(0xffffffffu, wait_phase(bar(C::B_O_DONE), (g - 1) & 1, abort_flag, p.status))) { ok = false; break; }
          if (__any_sync(0xffffffffu, rescale)) {
            tc_fence_after();
#pragma unroll 1
            for (int c = 0; c < D / 32; ++c) {
              uint32_t o[32];
              tmem_ld32(lane_base + C::TM_O + c * 32, o);
#pragma unroll
              for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
              tmem_st32(lane_base + C::TM_O + c * 32, o);
            }
          }
        }
        // P row -> shared memory, K-major with the 128-byte swizzle
#pragma unroll
        for (int c8 = 0; c8 < BN / 8; ++c8) {
          const int region = c8 >> 3, chunk = c8 & 7;
          const uint32_t addr = sP + region * (kRows * 128) + r * 128 + ((chunk ^ (r & 7)) << 4);
          st_shared_v4(addr, pk[c8 * 4 + 0], pk[c8 * 4 + 1], pk[c8 * 4 + 2], pk[c8 * 4 + 3]);
        }
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(bar(C::B_P_FULL));
      }
      if (!ok) break;
      // ------------------------------------------------------------ epilogue
      if (!__all_sync(0xffffffffu, wait_phase(bar(C::B_O_DONE), (gj + n - 1) & 1, abort_flag, p.status))) { ok = false; break; }
      tc_fence_after();
      const float inv_l = l_run > 0.f ? 1.f / l_run : 0.f;
      const float lse_v = l_lse > 0.f ? m_run * p.scale + logf(l_lse) : -INFINITY;
      if (sg.whole) {
        const int orow = td.q_row0 + t_row;
        const int h = td.kvh * G + g_row;
        __nv_bfloat16* dst = p.out + (static_cast<size_t>(orow) * p.Hq + h) * D;
#pragma unroll 1
        for (int c = 0; c < D / 32; ++c) {
          uint32_t o[32];
          tmem_ld32(lane_base + C::TM_O + c * 32, o);
          if (row_ok) {
            uint32_t w[16];
#pragma unroll
            for (int e = 0; e < 16; ++e)
              w[e] = pack_bf16x2(__uint_as_float(o[2 * e]) * inv_l, __uint_as_float(o[2 * e + 1]) * inv_l);
            uint4* d4 = reinterpret_cast<uint4*>(dst + c * 32);
#pragma unroll
            for (int e = 0; e < 4; ++e) d4[e] = make_uint4(w[4 * e], w[4 * e + 1], w[4 * e + 2], w[4 * e + 3]);
          }
        }
        if (row_ok && p.lse != nullptr) p.lse[static_cast<size_t>(orow) * p.Hq + h] = lse_v;
      } else {
        float* dst = p.ws.part_o + (static_cast<size_t>(sg.slot) * kRows + r) * D;
#pragma unroll 1
        for (int c = 0; c < D / 32; ++c) {
          uint32_t o[32];
          tmem_ld32(lane_base + C::TM_O + c * 32, o);
          float4* d4 = reinterpret_cast<float4*>(dst + c * 32);
#pragma unroll
          for (int e = 0; e < 8; ++e)
            d4[e] = make_float4(__uint_as_float(o[4 * e]) * inv_l, __uint_as_float(o[4 * e + 1]) * inv_l,
                                __uint_as_float(o[4 * e + 2]) * inv_l, __uint_as_float(o[4 * e + 3]) * inv_l);
        }
        p.ws.part_lse[static_cast<size_t>(sg.slot) * kRows + r] = lse_v;
      }
      tc_fence_before();
      mbar_arrive(bar(C::B_O_FREE));
      gj += n;
      ++seg_i;
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
combine_kernel(const FwdParams p, int num_ctas) {
  const WorkHeader* hdr = p.ws.hdr;
  const int tile = blockIdx.x;
  if (tile >= hdr->num_tiles) return;
  const int64_t U = hdr->total_units;
  const int P = active_ctas(num_ctas, U);
  const int64_t T0 = p.ws.unit_begin[tile], T1 = p.ws.unit_begin[tile + 1];
  const int c_lo = cta_of_unit(T0, U, P);
  const int c_hi = cta_of_unit(T1 - 1, U, P);
  if (c_lo == c_hi) return;  // written directly by one CTA
  const TileDesc td = p.ws.tiles[tile];
  const int G = p.G;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r = blockIdx.y * kCombineWarps + warp;
  if (r >= G * p.TT) return;
  const int t = r / G, gi = r - t * G;
  if (t >= td.n_tok) return;
  const int nc = c_hi - c_lo + 1;
  auto slot_of = [&](int c) { return cta_unit_begin(c, U, P) >= T0 ? 2 * c : 2 * c + 1; };
  float M = -INFINITY;
  for (int i = lane; i < nc; i += 32)
    M = fmaxf(M, p.ws.part_lse[static_cast<size_t>(slot_of(c_lo + i)) * kRows + r]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  constexpr int E = D / 32;  // columns per lane
  float acc[E];
#pragma unroll
  for (int e = 0; e < E; ++e) acc[e] = 0.f;
  float wsum = 0.f;
  for (int i = 0; i < nc; ++i) {
    const int slot = slot_of(c_lo + i);
    const float lk = p.ws.part_lse[static_cast<size_t>(slot) * kRows + r];
    if (lk == -INFINITY) continue;
    const float w = __expf(lk - M);
    wsum += w;
    const float* src = p.ws.part_o + (static_cast<size_t>(slot) * kRows + r) * D;
    if constexpr (E % 4 == 0) {
#pragma unroll
      for (int k = 0; k < E / 4; ++k) {
        const float4 x = *reinterpret_cast<const float4*>(src + (k * 32 + lane) * 4);
        acc[4 * k + 0] += w * x.x;
        acc[4 * k + 1] += w * x.y;
        acc[4 * k + 2] += w * x.z;
        acc[4 * k + 3] += w * x.w;
      }
    } else {
      const float2 x = *reinterpret_cast<const float2*>(src + lane * 2);
      acc[0] += w * x.x;
      acc[1] += w * x.y;
    }
  }
  const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
  const int orow = td.q_row0 + t;
  const int h = td.kvh * G + gi;
  __nv_bfloat16* dst = p.out + (static_cast<size_t>(orow) * p.Hq + h) * D;
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
