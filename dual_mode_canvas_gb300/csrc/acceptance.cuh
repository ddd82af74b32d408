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
  // a side whose weight underflows to 0 drops out: its d * s may overflow to
  // -inf (a chunk of masked logits has m = the lowest finite value), and
  // 0 * -inf would be NaN
  float tn = 0.f;
  if (e1 > 0.f) tn += e1 * (t + d1 * s);
  if (e2 > 0.f) tn += e2 * (t2 + d2 * s2);
  t = tn;
  s = e1 * s + e2 * s2;
  if (m2 > m || (m2 == m && a2 < a)) a = a2;
  m = mn;
}

// Chunks are laid out from the 16-byte boundary at or before the row's first
// logit, so every full 8-logit group is one aligned vector load whatever the
// vocabulary size or the buffer's alignment: chunk c of a row covers row
// positions [c K - off, (c + 1) K - off), off = the row start's misalignment
// in logits (0..7).  `chunks` must cover vocab + off.
__global__ void __launch_bounds__(kStatThreads, 4)
row_stats_kernel(const __nv_bfloat16* __restrict__ logits, int vocab, int chunks,
                 RowPartial* __restrict__ part) {
  const int row = blockIdx.x / chunks, chunk = blockIdx.x - row * chunks;
  const int64_t base = static_cast<int64_t>(row) * vocab;
  const int off = static_cast<int>(((reinterpret_cast<uintptr_t>(logits) >> 1) + base) & 7);
  const int tid = threadIdx.x;
  constexpr int kIters = kStatChunk / (kStatThreads * kStatVec);  // 8 vectors per thread
  // row position of the first logit of vector k of this thread
  auto first = [&](int k) { return chunk * kStatChunk - off + (k * kStatThreads + tid) * kStatVec; };
  // The lowest finite bf16: -inf logits (and positions outside the row) are
  // raised to it, so x - M stays finite and e * (x - M) is exactly 0.
  constexpr uint32_t kFloor2 = 0xFF7FFF7Fu;
  // pass 1a: every load of the thread is issued before any value is used
  uint4 v[kIters];
  bool has_data = false;
#pragma unroll
  for (int k = 0; k < kIters; ++k) {
    const int r0 = first(k);
    has_data |= (r0 + kStatVec > 0 && r0 < vocab);
    if (r0 >= 0 && r0 + kStatVec <= vocab) {
      v[k] = __ldg(reinterpret_cast<const uint4*>(logits + base + r0));
    } else {
      // the row's first or last group: element loads of the positions inside the row
      uint32_t w[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int i0 = r0 + 2 * j, i1 = i0 + 1;
        const unsigned short b0 = (i0 >= 0 && i0 < vocab) ? __bfloat16_as_ushort(logits[base + i0]) : 0xFF80u;
        const unsigned short b1 = (i1 >= 0 && i1 < vocab) ? __bfloat16_as_ushort(logits[base + i1]) : 0xFF80u;
        w[j] = static_cast<uint32_t>(b0) | (static_cast<uint32_t>(b1) << 16);
      }
      v[k] = make_uint4(w[0], w[1], w[2], w[3]);
    }
  }
  // pass 1b: clamp and the thread's max (packed pairs)
  uint32_t mx2 = kFloor2;
#pragma unroll
  for (int k = 0; k < kIters; ++k) {
    v[k].x = max_bf16x2(v[k].x, kFloor2);
    v[k].y = max_bf16x2(v[k].y, kFloor2);
    v[k].z = max_bf16x2(v[k].z, kFloor2);
    v[k].w = max_bf16x2(v[k].w, kFloor2);
    mx2 = max_bf16x2(mx2, max_bf16x2(max_bf16x2(v[k].x, v[k].y), max_bf16x2(v[k].z, v[k].w)));
  }
  // a thread with no position inside the row drops out
  const float mloc = has_data ? fmaxf(__uint_as_float(mx2 << 16), __uint_as_float(mx2 & 0xFFFF0000u))
                              : -INFINITY;
  // block maximum M (plain max, no exponentials)
  __shared__ float red_m[kStatThreads / 32];
  __shared__ float red_s[kStatThreads / 32], red_t[kStatThreads / 32];
  __shared__ int red_a[kStatThreads / 32];
  const int warp = tid >> 5, lane = tid & 31;
  float M = mloc;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  if (lane == 0) red_m[warp] = M;
  __syncthreads();
  M = red_m[0];
#pragma unroll
  for (int w = 1; w < kStatThreads / 32; ++w) M = fmaxf(M, red_m[w]);
  // pass 2 (registers only) against M, two lanes per fp32x2 instruction:
  // s = sum e, t = sum e * (x - M), e = 2^((x - M) log2 e)
  const uint64_t m2x = f32x2(M, M), l2e = f32x2(kLog2e, kLog2e);
  uint64_t s2 = 0ull, t2 = 0ull;
#pragma unroll
  for (int k = 0; k < kIters; ++k) {
    const uint32_t w[4] = {v[k].x, v[k].y, v[k].z, v[k].w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint64_t d = sub_f32x2(f32x2(__uint_as_float(w[j] << 16), __uint_as_float(w[j] & 0xFFFF0000u)), m2x);
      float y0, y1;
      f32x2_split(mul_f32x2(d, l2e), y0, y1);
      const uint64_t e = f32x2(ex2_approx(y0), ex2_approx(y1));
      s2 = add_f32x2(s2, e);
      t2 = fma_f32x2(e, d, t2);
    }
  }
  float s0, s1, t0, t1;
  f32x2_split(s2, s0, s1);
  f32x2_split(t2, t0, t1);
  float s = has_data ? s0 + s1 : 0.f, t = has_data ? t0 + t1 : 0.f;
  // first index of M: only threads holding M scan their values, in index
  // order (fully unrolled so the values stay in registers)
  int a = INT32_MAX;
  if (mloc == M) {
    const uint32_t mb = __float_as_uint(M) >> 16;
    const uint32_t mm2 = mb | (mb << 16);
#pragma unroll
    for (int k = kIters - 1; k >= 0; --k) {
      const uint32_t w[4] = {v[k].x, v[k].y, v[k].z, v[k].w};
      const int e0 = first(k);
#pragma unroll
      for (int j = 3; j >= 0; --j) {
        const uint32_t hit = eq_bf16x2(w[j], mm2);
        if (hit) a = e0 + 2 * j + ((hit & 1u) ? 0 : 1);
      }
    }
  }
  // block sums and the lowest index of M
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    s += __shfl_xor_sync(0xffffffffu, s, o);
    t += __shfl_xor_sync(0xffffffffu, t, o);
    a = min(a, __shfl_xor_sync(0xffffffffu, a, o));
  }
  if (lane == 0) {
    red_s[warp] = s;
    red_t[warp] = t;
    red_a[warp] = a;
  }
  __syncthreads();
  if (tid == 0) {
    float S = 0.f, T = 0.f;
    int A = INT32_MAX;
#pragma unroll
    for (int w = 0; w < kStatThreads / 32; ++w) {
      S += red_s[w];
      T += red_t[w];
      A = min(A, red_a[w]);
    }
    part[blockIdx.x] = S > 0.f ? RowPartial{M, S, T, A} : RowPartial{-INFINITY, 0.f, 0.f, INT32_MAX};
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
