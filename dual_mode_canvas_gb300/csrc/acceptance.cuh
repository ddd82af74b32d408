// Entropy-bounded acceptance of one denoise step (DiffusionGemma, agentlenshq
// page, "sampling loop and entropy-bounded denoising"; 24-ai.news page, "the
// mechanism for deciding finished tokens"):
//
//   row_stats_kernel     one CTA per (row, 16384-logit chunk): online softmax
//                        statistics of the chunk in one pass over HBM
//                        (max m, s = sum e^(x-m), t = sum e^(x-m) (x-m), the
//                        first index of the max).
//   accept_kernel        one CTA per canvas: merges each row's chunks in
//                        order (entropy H = ln s - t/s, confidence c = 1/s,
//                        argmax), ranks the open rows by confidence (bitonic
//                        sort, ties to the lower row), accepts them in that
//                        order while the running fp32 entropy sum stays within
//                        the budget (at least one per step), and runs the
//                        convergence test (argmax unchanged for `patience`
//                        steps and mean entropy under the threshold, or the
//                        step limit).
#pragma once

#include <cuda_bf16.h>
#include <cstdint>

#include "ptx.cuh"

namespace dg {

constexpr int kStatThreads = 256;
constexpr int kStatChunk = 16384;          // logits per CTA (32 KB of bf16)
constexpr int kStatVec = 8;                // bf16 per 16-byte load
constexpr int kAcceptThreads = 1024;       // max rows per canvas
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

struct RowPartial {
  float m;     // max logit of the chunk
  float s;     // sum e^(x - m)
  float t;     // sum e^(x - m) (x - m)
  int32_t arg; // first index of the max
};

// Combine (m2, s2, t2, a2) into (m, s, t, a); the argmax keeps the lower index on ties.
__device__ __forceinline__ void merge_stats(float& m, float& s, float& t, int& a, float m2, float s2,
                                            float t2, int a2) {
  if (s2 == 0.f) return;
  if (s == 0.f) {
    m = m2; s = s2; t = t2; a = a2;
    return;
  }
  const float mn = fmaxf(m, m2);
  const float d1 = m - mn, d2 = m2 - mn;
  const float e1 = exp2f(d1 * kLog2e), e2 = exp2f(d2 * kLog2e);
  t = e1 * (t + d1 * s) + e2 * (t2 + d2 * s2);
  s = e1 * s + e2 * s2;
  if (m2 > m || (m2 == m && a2 < a)) a = a2;
  m = mn;
}

__global__ void __launch_bounds__(kStatThreads, 3)
row_stats_kernel(const __nv_bfloat16* __restrict__ logits, int vocab, int chunks,
                 RowPartial* __restrict__ part) {
  const int row = blockIdx.x / chunks, chunk = blockIdx.x - row * chunks;
  const int64_t base = static_cast<int64_t>(row) * vocab;
  const int lo = chunk * kStatChunk;
  const int hi = min(vocab, lo + kStatChunk);
  const int tid = threadIdx.x;
  constexpr int kIters = kStatChunk / (kStatThreads * kStatVec);  // 8 loads per thread
  // pass 1: the thread's values in registers, its max and first argmax
  uint4 v[kIters];
  float m = -INFINITY;
  int a = INT32_MAX;
#pragma unroll
  for (int k = 0; k < kIters; ++k) {
    const int e0 = lo + (k * kStatThreads + tid) * kStatVec;
    if (e0 + kStatVec <= hi && ((base + e0) & 7) == 0) {
      v[k] = __ldg(reinterpret_cast<const uint4*>(logits + base + e0));
    } else {
      // ragged tail or a row that does not start 16-byte aligned: element loads, pad with -inf
      uint32_t w[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int i0 = e0 + 2 * j, i1 = i0 + 1;
        const unsigned short b0 = i0 < hi ? __bfloat16_as_ushort(logits[base + i0]) : 0xFF80u;
        const unsigned short b1 = i1 < hi ? __bfloat16_as_ushort(logits[base + i1]) : 0xFF80u;
        w[j] = static_cast<uint32_t>(b0) | (static_cast<uint32_t>(b1) << 16);
      }
      v[k] = make_uint4(w[0], w[1], w[2], w[3]);
    }
    const uint32_t w[4] = {v[k].x, v[k].y, v[k].z, v[k].w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float x0 = __uint_as_float(w[j] << 16), x1 = __uint_as_float(w[j] & 0xFFFF0000u);
      const int i0 = e0 + 2 * j;
      if (x0 > m) { m = x0; a = i0; }
      if (x1 > m) { m = x1; a = i0 + 1; }
    }
  }
  // pass 2 (registers only): s and t relative to the thread's max
  float s = 0.f, t = 0.f;
  if (m > -INFINITY) {
    const float nm = -m * kLog2e;
#pragma unroll
    for (int k = 0; k < kIters; ++k) {
      const uint32_t w[4] = {v[k].x, v[k].y, v[k].z, v[k].w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float x0 = __uint_as_float(w[j] << 16), x1 = __uint_as_float(w[j] & 0xFFFF0000u);
        const float e0 = ex2_approx(fmaf(x0, kLog2e, nm)), e1 = ex2_approx(fmaf(x1, kLog2e, nm));
        s += e0 + e1;
        // x - m is clamped so that padding (-inf) gives 0 * -1000 = 0, not 0 * -inf
        t = fmaf(e0, fmaxf(x0 - m, -1000.f), t);
        t = fmaf(e1, fmaxf(x1 - m, -1000.f), t);
      }
    }
  }
  // block reduction: warps by shuffles, then warp 0 over the warp results
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float m2 = __shfl_xor_sync(0xffffffffu, m, o), s2 = __shfl_xor_sync(0xffffffffu, s, o);
    const float t2 = __shfl_xor_sync(0xffffffffu, t, o);
    const int a2 = __shfl_xor_sync(0xffffffffu, a, o);
    merge_stats(m, s, t, a, m2, s2, t2, a2);
  }
  __shared__ RowPartial red[kStatThreads / 32];
  const int warp = tid >> 5, lane = tid & 31;
  if (lane == 0) red[warp] = RowPartial{m, s, t, a};
  __syncthreads();
  if (warp == 0) {
    RowPartial r = lane < kStatThreads / 32 ? red[lane] : RowPartial{-INFINITY, 0.f, 0.f, INT32_MAX};
    m = r.m; s = r.s; t = r.t; a = r.arg;
#pragma unroll
    for (int o = 4; o > 0; o >>= 1) {
      const float m2 = __shfl_xor_sync(0xffffffffu, m, o), s2 = __shfl_xor_sync(0xffffffffu, s, o);
      const float t2 = __shfl_xor_sync(0xffffffffu, t, o);
      const int a2 = __shfl_xor_sync(0xffffffffu, a, o);
      merge_stats(m, s, t, a, m2, s2, t2, a2);
    }
    if (lane == 0) part[blockIdx.x] = RowPartial{m, s, t, a};
  }
}

struct AcceptParams {
  const RowPartial* part;
  int chunks;
  const int32_t* cu_rows;      // [num_canvases + 1]
  const uint8_t* accepted_in;  // [rows]
  const int32_t* argmax_prev;  // [rows]
  const int32_t* stable_in;    // [num_canvases]
  float budget, tau;
  int patience, step, max_steps;
  float* entropy;              // [rows]
  float* confidence;           // [rows]
  int32_t* argmax;             // [rows]
  uint8_t* accepted_out;       // [rows]
  int32_t* stable_out;         // [num_canvases]
  uint8_t* converged;          // [num_canvases]
  int* status;
};

__global__ void __launch_bounds__(kAcceptThreads)
accept_kernel(const AcceptParams p) {
  __shared__ unsigned long long key[kAcceptThreads];
  __shared__ float Hs[kAcceptThreads];
  const int b = blockIdx.x;
  const int r0 = p.cu_rows[b], r1 = p.cu_rows[b + 1];
  const int n = r1 - r0;
  const int tid = threadIdx.x;
  if (n < 0 || n > kAcceptThreads) {
    if (tid == 0) atomicCAS(p.status, 0, 1);  // invalid canvas size
    return;
  }
  bool same = true;
  if (tid < n) {
    const int row = r0 + tid;
    float m = -INFINITY, s = 0.f, t = 0.f;
    int a = INT32_MAX;
    for (int c = 0; c < p.chunks; ++c) {
      const RowPartial q = p.part[static_cast<size_t>(row) * p.chunks + c];
      merge_stats(m, s, t, a, q.m, q.s, q.t, q.arg);
    }
    const float H = logf(s) - t / s;  // ln s - t / s
    const float conf = 1.f / s;
    p.entropy[row] = H;
    p.confidence[row] = conf;
    p.argmax[row] = a;
    Hs[tid] = H;
    same = (a == p.argmax_prev[row]);
    const bool open = p.accepted_in[row] == 0;
    // ascending order of the key = confidence descending, then row ascending;
    // closed rows sort last
    const uint32_t hi = open ? 0x7F800000u - __float_as_uint(conf) : 0xFFFFFFFFu;
    key[tid] = (static_cast<unsigned long long>(hi) << 32) | static_cast<uint32_t>(tid);
    p.accepted_out[row] = open ? 0 : 1;
  }
  int np2 = 1;
  while (np2 < n) np2 <<= 1;
  if (tid >= n && tid < np2) key[tid] = ~0ull;
  const bool all_same = __syncthreads_and(same) != 0;
  // bitonic sort of key[0 .. np2)
  for (int k = 2; k <= np2; k <<= 1) {
    for (int j = k >> 1; j > 0; j >>= 1) {
      if (tid < np2) {
        const int ixj = tid ^ j;
        if (ixj > tid) {
          const unsigned long long x = key[tid], y = key[ixj];
          const bool up = (tid & k) == 0;
          if ((x > y) == up) { key[tid] = y; key[ixj] = x; }
        }
      }
      __syncthreads();
    }
  }
  if (tid == 0 && n > 0) {
    // sequential fp32 running sum in ranking order, so the decision is reproducible
    float run = 0.f;
    for (int k = 0; k < n; ++k) {
      const unsigned long long x = key[k];
      if ((x >> 32) == 0xFFFFFFFFull) break;  // closed rows follow the open ones
      const int i = static_cast<int>(x & 0xFFFFFFFFull);
      run = __fadd_rn(run, Hs[i]);
      if (k > 0 && run > p.budget) break;
      p.accepted_out[r0 + i] = 1;
    }
    float total = 0.f;
    for (int i = 0; i < n; ++i) total = __fadd_rn(total, Hs[i]);
    const float mean = __fdiv_rn(total, static_cast<float>(n));
    const int stable = all_same ? p.stable_in[b] + 1 : 0;
    p.stable_out[b] = stable;
    p.converged[b] = ((stable >= p.patience && mean < p.tau) || (p.step + 1 >= p.max_steps)) ? 1 : 0;
  }
}

}  // namespace dg
