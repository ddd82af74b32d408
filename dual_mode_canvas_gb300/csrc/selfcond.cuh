// Self-conditioning input of a denoise step (DiffusionGemma, agentlenshq page,
// "self-conditioning for stability"; 24-ai.news page, the self-conditioning
// signal between iterations): the probability-weighted average of the token
// embeddings under the previous step's softmax,
//
//   Y[r, :] = sum_v p[r, v] E[v, :],   p[r, :] = softmax(logits[r, :]).
//
//   row_stats_kernel (acceptance.cuh) then sc_rowconst_kernel: per row the
//       constant c_r = m_r log2(e) + log2(s_r) of its softmax, so that
//       p = 2^(x log2(e) - c_r) needs one FMA and one ex2 per logit.
//   sc_kernel: a persistent tcgen05 GEMM.  Work units are (vocabulary split,
//       128-row tile, 256-column tile of E); CTAs take units round-robin with
//       the split outermost, so the CTAs running at any moment read the same
//       vocabulary range of logits and E and share it in L2.  Per 64-entry
//       vocabulary block: TMA brings the 128 x 64 logits tile of this CTA's
//       rows and the 64 x 256 E tile into this CTA's shared memory; several
//       warps per TMEM lane quadrant (one row and a share of the block's
//       columns per thread) turn the logits into bf16 probabilities written
//       straight to TMEM; the MMA warp accumulates P (A from TMEM) x E (B,
//       N-major in shared memory) into TMEM.
//   sc_combine_kernel: sums the splits' fp32 partials when there are several.
#pragma once

#include <cuda_bf16.h>
#include <cstdint>

#include "acceptance.cuh"
#include "kernels.cuh"
#include "ptx.cuh"

namespace dg {

constexpr int kScN = 256;   // embedding columns per tile (UMMA N)
constexpr int kScK = 64;    // vocabulary entries per block (one 128-byte row of bf16)
constexpr int kScNL = 3;    // logits ring stages (read into registers at once)
constexpr int kScNE = 5;    // embedding ring stages (held until the MMA is done)
constexpr int kScNP = 4;    // probability buffers in TMEM
// kScXW warps per TMEM lane quadrant compute probabilities, each 1/kScXW of a
// block's columns: warps 0-3 and 7.. ; warps 4 / 6 load, warp 5 issues MMAs
constexpr int kScXW = 2;
constexpr int kScXform = 128 * kScXW;           // probability threads
constexpr int kScThreads = kScXform + 3 * 32;

struct ScCfg {
  static constexpr int L_BYTES = kRows * kScK * 2;   // one logits tile, 16 KB
  static constexpr int E_BYTES = kScK * kScN * 2;    // one embedding tile, 32 KB
  static constexpr int OFF_L = 0;
  static constexpr int OFF_E = OFF_L + kScNL * L_BYTES;
  static constexpr int OFF_BAR = OFF_E + kScNE * E_BYTES;
  static constexpr int B_L_FULL = 0, B_L_EMPTY = kScNL, B_E_FULL = 2 * kScNL,
                       B_E_EMPTY = 2 * kScNL + kScNE, B_P_FULL = 2 * kScNL + 2 * kScNE,
                       B_P_EMPTY = B_P_FULL + kScNP, B_ACC_FULL = B_P_EMPTY + kScNP,
                       B_ACC_EMPTY = B_ACC_FULL + 1, B_DRAIN = B_ACC_EMPTY + 1,
                       NUM_BARS = B_DRAIN + 1;
  static constexpr int OFF_MISC = OFF_BAR + NUM_BARS * 8;
  static constexpr int SMEM_BYTES = OFF_MISC + 16 + 1024;  // slack for 1024-byte alignment
  // TMEM: the fp32 accumulator (kScN columns), then kScNP probability buffers
  // of kScK / 2 columns (packed bf16 pairs)
  static constexpr uint32_t TM_ACC = 0, TM_P = kScN;
  static_assert(kScN + kScNP * (kScK / 2) <= static_cast<int>(kTmemCols), "TMEM budget");
  static_assert(SMEM_BYTES <= 232448, "shared memory budget");
};

struct ScParams {
  const float* rowc;  // [rows] c_r
  float* out;         // [rows, d] fp32, written directly when splits == 1
  float* part;        // splits > 1: fp32 [splits, m_tiles, n_tiles, kScN, 128], each
                      // tile column-major so the epilogue's stores coalesce
  int* status;
  // >= 0: the E loader skips its load of this (per-CTA) block, so the MMA
  // warp's bounded wait for it expires (tests of the timeout path)
  int debug_skip_e_load;
  int rows, vocab, d;
  int m_tiles, n_tiles, splits, kblocks;
};

// a thread's packed probabilities -> TMEM (8 or 16 columns, by share size)
__device__ __forceinline__ void st_probs(uint32_t taddr, const uint32_t (&r)[8]) { tmem_st8(taddr, r); }
__device__ __forceinline__ void st_probs(uint32_t taddr, const uint32_t (&r)[16]) { tmem_st16(taddr, r); }

struct ScUnit {
  int split, mt, nt, kb0, kb1;
};

// Unit u: split outermost, then the row tile, then the E tile.
__device__ __forceinline__ ScUnit sc_unit(const ScParams& p, int64_t u) {
  const int64_t per_split = static_cast<int64_t>(p.m_tiles) * p.n_tiles;
  ScUnit w;
  w.split = static_cast<int>(u / per_split);
  const int rem = static_cast<int>(u - w.split * per_split);
  w.mt = rem / p.n_tiles;
  w.nt = rem - w.mt * p.n_tiles;
  w.kb0 = static_cast<int>(static_cast<int64_t>(w.split) * p.kblocks / p.splits);
  w.kb1 = static_cast<int>(static_cast<int64_t>(w.split + 1) * p.kblocks / p.splits);
  return w;
}

// One warp per row: lane c merges chunks c, c + 32, ..., the lanes then
// merge by shuffles and lane 0 writes c_r = m log2(e) + log2(s).
__global__ void __launch_bounds__(256) sc_rowconst_kernel(const RowPartial* __restrict__ part, int rows,
                                                           int chunks, float* __restrict__ rowc) {
  const int r = blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (r >= rows) return;  // warp-uniform
  float m = -INFINITY, s = 0.f, t = 0.f;
  int a = INT32_MAX;
  for (int c = lane; c < chunks; c += 32) {
    const RowPartial q = part[static_cast<size_t>(r) * chunks + c];
    merge_stats(m, s, t, a, q.m, q.s, q.t, q.arg);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
    const float s2 = __shfl_xor_sync(0xffffffffu, s, o);
    const float t2 = __shfl_xor_sync(0xffffffffu, t, o);
    const int a2 = __shfl_xor_sync(0xffffffffu, a, o);
    merge_stats(m, s, t, a, m2, s2, t2, a2);
  }
  if (lane == 0) rowc[r] = m * kLog2e + log2f(s);
}

__global__ void __launch_bounds__(kScThreads, 1)
sc_kernel(const __grid_constant__ CUtensorMap tm_l, const __grid_constant__ CUtensorMap tm_e,
          const ScParams p) {
  using Cf = ScCfg;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_base = smem_u32(smem_raw);
  const uint32_t sbase = (raw_base + 1023u) & ~1023u;
  uint8_t* sptr = smem_raw + (sbase - raw_base);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int cl = static_cast<int>(blockIdx.x);
  const int ncl = static_cast<int>(gridDim.x);
  const int64_t U = static_cast<int64_t>(p.splits) * p.m_tiles * p.n_tiles;

  const uint32_t sL = sbase + Cf::OFF_L;
  const uint32_t sE = sbase + Cf::OFF_E;
  const uint32_t bars = sbase + Cf::OFF_BAR;
  auto bar = [&](int i) -> uint32_t { return bars + 8u * static_cast<uint32_t>(i); };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sptr + Cf::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sptr + Cf::OFF_MISC + 4);

  if (threadIdx.x == 0) {
    for (int s = 0; s < kScNL; ++s) {
      mbar_init(bar(Cf::B_L_FULL + s), 1);
      mbar_init(bar(Cf::B_L_EMPTY + s), kScXform);
    }
    for (int s = 0; s < kScNE; ++s) {
      mbar_init(bar(Cf::B_E_FULL + s), 1);
      mbar_init(bar(Cf::B_E_EMPTY + s), 1);
    }
    for (int s = 0; s < kScNP; ++s) {
      mbar_init(bar(Cf::B_P_FULL + s), kScXform);
      mbar_init(bar(Cf::B_P_EMPTY + s), 1);
    }
    mbar_init(bar(Cf::B_ACC_FULL), 1);
    mbar_init(bar(Cf::B_ACC_EMPTY), kScXform);
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
    tma_prefetch_desc(&tm_l);
    tma_prefetch_desc(&tm_e);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == kTmaWarp || warp == kVLoadWarp) {
    // ----------------------------------------------------------- producers
    // warp 4 loads this CTA's logits tiles, warp 6 its E tiles, both from
    // this GPU's memory into this CTA's shared memory
    if (lane == 0) {
      const bool is_l = (warp == kTmaWarp);
      const int NS = is_l ? kScNL : kScNE;
      const uint32_t full0 = bar(is_l ? Cf::B_L_FULL : Cf::B_E_FULL);
      const uint32_t empty0 = bar(is_l ? Cf::B_L_EMPTY : Cf::B_E_EMPTY);
      uint32_t stage = 0, phase = 0;
      uint32_t issued_mask = 0, issued_phase = 0;
      int loads = 0;
      bool ok = true;
      for (int64_t u = cl; ok && u < U; u += ncl) {
        const ScUnit w = sc_unit(p, u);
        for (int kb = w.kb0; kb < w.kb1; ++kb) {
          if (!wait_phase(empty0 + 8u * stage, phase ^ 1, abort_flag, p.status)) { ok = false; break; }
          if (!is_l && loads++ == p.debug_skip_e_load) {
            // test hook: this stage is never filled, so the MMA warp's
            // bounded wait for it expires
            if (++stage == static_cast<uint32_t>(NS)) { stage = 0; phase ^= 1; }
            continue;
          }
          // (bounds-checking build) every box starts inside its tensor
          if (is_l) {
            mbar_arrive_expect_tx(full0 + 8u * stage, Cf::L_BYTES);
            if (in_bounds(kb * kScK < p.vocab && w.mt * kRows < p.rows, p.status, abort_flag))
              tma_load_3d(sL + stage * Cf::L_BYTES, &tm_l, full0 + 8u * stage, kb * kScK, 0,
                          w.mt * kRows);
          } else {
            mbar_arrive_expect_tx(full0 + 8u * stage, Cf::E_BYTES);
            const uint32_t dst = sE + stage * Cf::E_BYTES;
#pragma unroll
            for (int nb = 0; nb < kScN / 64; ++nb)
              // (column boxes of the last E tile past d_model are zero-filled by design)
              if (in_bounds(kb * kScK < p.vocab && w.nt < p.n_tiles, p.status, abort_flag))
                tma_load_3d(dst + nb * (kScK * 128), &tm_e, full0 + 8u * stage, w.nt * kScN + nb * 64, 0,
                            kb * kScK);
          }
          issued_mask |= 1u << stage;
          issued_phase = (issued_phase & ~(1u << stage)) | (phase << stage);
          if (++stage == static_cast<uint32_t>(NS)) { stage = 0; phase ^= 1; }
        }
      }
      if (!ok) {
        // let loads already in flight land before the CTA's shared memory goes away
        for (int st = 0; st < NS; ++st)
          if (issued_mask & (1u << st)) drain_wait(full0 + 8u * st, (issued_phase >> st) & 1);
      }
    }
    __syncwarp();
  } else if (warp == kMmaWarp) {
    // ---------------------------------------------------------- MMA issuer
    // ACC += P (128 x 64, bf16 in TMEM) x E (64 x 256, N-major in shared
    // memory), four K=16 steps per vocabulary block; one elected lane issues
    constexpr uint32_t idesc = idesc_bf16_f32(kRows, kScN, 0, 1);
    uint32_t e_stage = 0, e_phase = 0, g = 0, ui = 0;
    bool ok = true;
    for (int64_t u = cl; ok && u < U; u += ncl, ++ui) {
      const ScUnit w = sc_unit(p, u);
      // the accumulator is free once the previous unit's epilogue has read it
      if (ui > 0 &&
          !__all_sync(0xffffffffu, wait_phase(bar(Cf::B_ACC_EMPTY), (ui - 1) & 1, abort_flag, p.status))) {
        ok = false;
        break;
      }
      tc_fence_after();
      for (int kb = w.kb0; kb < w.kb1; ++kb, ++g) {
        const uint32_t ps = g % kScNP, pph = (g / kScNP) & 1;
        if (!__all_sync(0xffffffffu, wait_phase(bar(Cf::B_P_FULL + ps), pph, abort_flag, p.status) &&
                                         wait_phase(bar(Cf::B_E_FULL + e_stage), e_phase, abort_flag, p.status))) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t e_base = sE + e_stage * Cf::E_BYTES;
#pragma unroll
        for (int kk = 0; kk < kScK / 16; ++kk) {
          const uint64_t b = smem_desc_sw128(e_base + kk * 2048, kScK * 128, 1024);
          umma_bf16_ts_warp(tmem + Cf::TM_ACC, tmem + Cf::TM_P + ps * (kScK / 2) + kk * 8, b, idesc,
                            (kb == w.kb0 && kk == 0) ? 0u : 1u);
        }
        umma_commit_warp(bar(Cf::B_P_EMPTY + ps));
        umma_commit_warp(bar(Cf::B_E_EMPTY + e_stage));
        if (++e_stage == kScNE) { e_stage = 0; e_phase ^= 1; }
      }
      if (!ok) break;
      umma_commit_warp(bar(Cf::B_ACC_FULL));
    }
    // every MMA issued by this thread has finished before TMEM is released
    umma_commit_warp(bar(Cf::B_DRAIN));
    drain_wait(bar(Cf::B_DRAIN), 0);
    __syncwarp();
  } else {
    // ---------------- probabilities and epilogue: warps 0-3 and 7.. ; warp w
    // owns TMEM lanes 32 (w % 4) .. +31 (one row each) and column share h
    const int q = warp & 3;
    const int h = (warp < 4 ? warp : warp - 3) >> 2;
    const int r = q * 32 + lane;  // row of the tile == TMEM lane
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(q * 32) << 16);
    const uint64_t l2e2 = f32x2(kLog2e, kLog2e);
    constexpr int kPart = kScK / kScXW;  // logits per thread per block
    uint32_t l_stage = 0, l_phase = 0, g = 0, ui = 0;
    bool ok = true;
    for (int64_t u = cl; ok && u < U; u += ncl, ++ui) {
      const ScUnit w = sc_unit(p, u);
      const int row = w.mt * kRows + r;
      const bool row_ok = row < p.rows;
      // rows past the end (zero-filled by TMA) get p = 2^-inf = 0
      const float c = row_ok ? p.rowc[row] : INFINITY;
      const uint64_t nc2 = f32x2(-c, -c);
      for (int kb = w.kb0; kb < w.kb1; ++kb, ++g) {
        if (!__all_sync(0xffffffffu, wait_phase(bar(Cf::B_L_FULL + l_stage), l_phase, abort_flag, p.status))) {
          ok = false;
          break;
        }
        // this row's share: 16-byte chunks (8/kScXW) h .. , chunk j stored at j ^ (row & 7)
        constexpr int kChunks = kPart / 8;
        uint32_t x[kPart / 2];
        const uint32_t rb = sL + l_stage * Cf::L_BYTES + r * 128;
#pragma unroll
        for (int j = 0; j < kChunks; ++j) {
          const uint32_t a = rb + ((static_cast<uint32_t>(kChunks * h + j) ^ (r & 7)) << 4);
          asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                       : "=r"(x[4 * j]), "=r"(x[4 * j + 1]), "=r"(x[4 * j + 2]), "=r"(x[4 * j + 3])
                       : "r"(a));
        }
        mbar_arrive(bar(Cf::B_L_EMPTY + l_stage));
        if (++l_stage == kScNL) { l_stage = 0; l_phase ^= 1; }
        // p = 2^(x log2(e) - c_r), two logits per fp32x2 FMA
        uint32_t pk[kPart / 2];
#pragma unroll
        for (int i = 0; i < kPart / 2; ++i) {
          float t0, t1;
          f32x2_split(fma_f32x2(f32x2(__uint_as_float(x[i] << 16), __uint_as_float(x[i] & 0xFFFF0000u)),
                                l2e2, nc2),
                      t0, t1);
          pk[i] = pack_bf16x2(ex2_approx(t0), ex2_approx(t1));
        }
        if ((kb + 1) * kScK > p.vocab) {
          // the block past the vocabulary: those entries (zero-filled by TMA) get p = 0
#pragma unroll
          for (int i = 0; i < kPart / 2; ++i) {
            const int v0 = kb * kScK + h * kPart + 2 * i;
            if (v0 >= p.vocab) pk[i] = 0u;
            else if (v0 + 1 >= p.vocab) pk[i] &= 0xFFFFu;
          }
        }
        const uint32_t ps = g % kScNP, pph = (g / kScNP) & 1;
        if (!__all_sync(0xffffffffu, wait_phase(bar(Cf::B_P_EMPTY + ps), pph ^ 1, abort_flag, p.status))) {
          ok = false;
          break;
        }
        tc_fence_after();
        st_probs(lane_base + Cf::TM_P + ps * (kScK / 2) + h * (kPart / 2), pk);
        tc_fence_before();
        mbar_arrive(bar(Cf::B_P_FULL + ps));
      }
      if (!ok) break;
      // ------------------------------------------------------------ epilogue
      // this warp's share of the accumulator columns
      if (!__all_sync(0xffffffffu, wait_phase(bar(Cf::B_ACC_FULL), ui & 1, abort_flag, p.status))) {
        ok = false;
        break;
      }
      tc_fence_after();
      const int hc = h * (kScN / kScXW);
      if (p.splits == 1) {
        // one split: this row straight into out (small problems only)
        const int col0 = w.nt * kScN + hc;
        float* dst = p.out + static_cast<size_t>(row) * p.d + col0;
#pragma unroll 1
        for (int cc = 0; cc < kScN / kScXW / 32; ++cc) {
          uint32_t o[32];
          tmem_ld32(lane_base + Cf::TM_ACC + hc + cc * 32, o);
          if (row_ok) {
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              const int col = cc * 32 + 4 * e;
              if (col0 + col < p.d)
                *reinterpret_cast<float4*>(dst + col) =
                    make_float4(__uint_as_float(o[4 * e]), __uint_as_float(o[4 * e + 1]),
                                __uint_as_float(o[4 * e + 2]), __uint_as_float(o[4 * e + 3]));
            }
          }
        }
      } else if (w.mt < p.m_tiles &&
                 in_bounds(w.split < p.splits && w.nt < p.n_tiles, p.status, abort_flag)) {
        // column-major partial tile: for each column the warp writes 32
        // consecutive rows (128 bytes)
        float* dst = p.part + ((static_cast<size_t>(w.split) * p.m_tiles + w.mt) * p.n_tiles + w.nt) *
                                  (static_cast<size_t>(kScN) * kRows) + static_cast<size_t>(hc) * kRows + r;
#pragma unroll 1
        for (int cc = 0; cc < kScN / kScXW / 32; ++cc) {
          uint32_t o[32];
          tmem_ld32(lane_base + Cf::TM_ACC + hc + cc * 32, o);
#pragma unroll
          for (int e = 0; e < 32; ++e) dst[static_cast<size_t>(cc * 32 + e) * kRows] = __uint_as_float(o[e]);
        }
      }
      tc_fence_before();
      mbar_arrive(bar(Cf::B_ACC_EMPTY));
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// out[r, c] = sum over splits of the partial tiles: one CTA per 128 rows x
// 32 columns of out.  Each thread reads four rows of a column at a time
// (the tiles are column-major, so a warp reads 512 contiguous bytes), sums
// the splits, and the block writes out row by row through shared memory.
__global__ void __launch_bounds__(256, 4) sc_combine_kernel(const ScParams p) {
  __shared__ float t[32][kRows + 4];
  const int mt = blockIdx.x, c0 = blockIdx.y * 32;
  const int tx = threadIdx.x, ty = threadIdx.y;  // 32 x 8 threads
  const size_t tile = static_cast<size_t>(kScN) * kRows;
  const size_t split_stride4 = static_cast<size_t>(p.m_tiles) * p.n_tiles * tile / 4;
  const float4* src[4];
  bool ok[4];
  float4 acc[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int c = c0 + ty + 8 * k;
    ok[k] = c < p.d;
    const int nt = ok[k] ? c / kScN : 0, cl = ok[k] ? c - nt * kScN : 0;
    src[k] = reinterpret_cast<const float4*>(p.part + (static_cast<size_t>(mt) * p.n_tiles + nt) * tile +
                                             static_cast<size_t>(cl) * kRows) + tx;
    acc[k] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
#pragma unroll 2
  for (int s = 0; s < p.splits; ++s) {
    float4 v[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) v[k] = ok[k] ? __ldg(src[k] + s * split_stride4) : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      acc[k].x += v[k].x;
      acc[k].y += v[k].y;
      acc[k].z += v[k].z;
      acc[k].w += v[k].w;
    }
  }
#pragma unroll
  for (int k = 0; k < 4; ++k) *reinterpret_cast<float4*>(&t[ty + 8 * k][4 * tx]) = acc[k];
  __syncthreads();
  const int c = c0 + tx;
  for (int rr = ty; rr < kRows; rr += 8) {
    const int row = mt * kRows + rr;
    if (row < p.rows && c < p.d) p.out[static_cast<size_t>(row) * p.d + c] = t[tx][rr];
  }
}

}  // namespace dg
