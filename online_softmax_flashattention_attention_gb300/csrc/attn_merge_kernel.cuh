// Merge of partial attention states, sm_103a.
//
// A state (m, l, o~) summarises the keys one split absorbed: m the largest scaled score,
// l = sum exp(s_j - m), o~ = sum exp(s_j - m) v_j ("FlashAttention math", section "The
// running state").  States of disjoint key sets combine with the rescaling identity of
// the same page (section "The rescaling identity, derived"): every state is moved to
// the common reference m = max_s m_s by the factor exp(m_s - m) <= 1, then the sums add.
// The single final division gives O = o~ / l and LSE = m + ln l; a row whose states all
// saw no visible key (every m_s = -inf) gets O = 0, LSE = -inf.
//
// The merge reads S * (4 d + 8) bytes and writes 2 d + 4 bytes per row: it is bound by
// HBM bandwidth.  One warp owns one row; lane t holds columns [t * d/32, (t+1) * d/32),
// so each state's o~ row is one coalesced 256- or 512-byte read.  Rows are spread over
// a grid sized to the SM count (grid-stride loop).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "ptx.cuh"

namespace attn {

constexpr int kMergeThreads = 256;

struct MergeParams {
  const float* st_o;  // [S, rows, D]
  const float* st_m;  // [S, rows]
  const float* st_l;  // [S, rows]
  int S;
  long long rows;
  __nv_bfloat16* O;   // [rows, D]
  float* lse;         // [rows]
};

template <int D>
__global__ void __launch_bounds__(kMergeThreads) attn_merge_kernel(const MergeParams p) {
  constexpr int kPer = D / 32;  // columns per lane: 4 (d = 128) or 2 (d = 64)
  constexpr float kLog2e = 1.4426950408889634f;
  const int lane = threadIdx.x & 31;
  const long long warps = static_cast<long long>(gridDim.x) * (kMergeThreads / 32);
  for (long long row = static_cast<long long>(blockIdx.x) * (kMergeThreads / 32) + (threadIdx.x >> 5);
       row < p.rows; row += warps) {
    // the common reference: the largest running max over the states
    float mx = -INFINITY;
    for (int s = lane; s < p.S; s += 32) mx = fmaxf(mx, __ldg(p.st_m + static_cast<long long>(s) * p.rows + row));
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
    const float ref = (mx == -INFINITY) ? 0.f : mx;
    // l = sum_s exp(m_s - m) l_s  (an empty state has m_s = -inf, factor 0)
    float lsum = 0.f;
    for (int s = lane; s < p.S; s += 32) {
      const long long i = static_cast<long long>(s) * p.rows + row;
      lsum += ex2_approx((__ldg(p.st_m + i) - ref) * kLog2e) * __ldg(p.st_l + i);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) lsum += __shfl_xor_sync(0xffffffffu, lsum, off);
    // o~ = sum_s exp(m_s - m) o~_s, this lane's columns
    float acc[kPer];
#pragma unroll
    for (int k = 0; k < kPer; ++k) acc[k] = 0.f;
#pragma unroll 4
    for (int s = 0; s < p.S; ++s) {
      const long long i = static_cast<long long>(s) * p.rows + row;
      const float w = ex2_approx((__ldg(p.st_m + i) - ref) * kLog2e);
      const float* src = p.st_o + i * D + lane * kPer;
      if constexpr (kPer == 4) {
        const float4 v = __ldg(reinterpret_cast<const float4*>(src));
        acc[0] = fmaf(w, v.x, acc[0]);
        acc[1] = fmaf(w, v.y, acc[1]);
        acc[2] = fmaf(w, v.z, acc[2]);
        acc[3] = fmaf(w, v.w, acc[3]);
      } else {
        const float2 v = __ldg(reinterpret_cast<const float2*>(src));
        acc[0] = fmaf(w, v.x, acc[0]);
        acc[1] = fmaf(w, v.y, acc[1]);
      }
    }
    // the single final division
    const float inv = lsum > 0.f ? 1.f / lsum : 0.f;
    __nv_bfloat16* dst = p.O + row * D + lane * kPer;
    if constexpr (kPer == 4) {
      uint2 packed;
      packed.x = pack_bf16x2(acc[0] * inv, acc[1] * inv);
      packed.y = pack_bf16x2(acc[2] * inv, acc[3] * inv);
      *reinterpret_cast<uint2*>(dst) = packed;
    } else {
      *reinterpret_cast<uint32_t*>(dst) = pack_bf16x2(acc[0] * inv, acc[1] * inv);
    }
    if (lane == 0) p.lse[row] = lsum > 0.f ? mx + logf(lsum) : -INFINITY;
  }
}

}  // namespace attn
