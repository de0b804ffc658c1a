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
// memory bandwidth once enough loads are in flight.  One warp owns one row; lane t holds
// columns [t * d/32, (t+1) * d/32), so each state's o~ row is one coalesced 256- or
// 512-byte read.  States are taken eight at a time: all their loads are issued before
// any arithmetic, and the chunks fold into a running (M, L, o~) with the same identity,
// so a row costs one round trip to memory per eight states.  Rows are spread over a grid
// sized to the SM count (grid-stride loop).
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
  constexpr int kPer = D / 32;    // columns per lane: 4 (d = 128) or 2 (d = 64)
  constexpr int kChunk = 8;       // states loaded together: one round of independent loads
  constexpr float kLog2e = 1.4426950408889634f;
  const int lane = threadIdx.x & 31;
  griddep_wait();  // the states kernel before it in the stream has finished
  griddep_launch_dependents();
  const long long warps = static_cast<long long>(gridDim.x) * (kMergeThreads / 32);
  for (long long row = static_cast<long long>(blockIdx.x) * (kMergeThreads / 32) + (threadIdx.x >> 5);
       row < p.rows; row += warps) {
    // running merge over chunks of states: (M, L, acc) is the state of the states seen
    float M = -INFINITY, L = 0.f;
    float acc[kPer];
#pragma unroll
    for (int k = 0; k < kPer; ++k) acc[k] = 0.f;
    for (int s0 = 0; s0 < p.S; s0 += kChunk) {
      float ms[kChunk], ls[kChunk], os[kChunk][kPer];
      // every load of the chunk first (m and l are the same address for all lanes)
#pragma unroll
      for (int c = 0; c < kChunk; ++c) {
        const int s = s0 + c;
        ms[c] = -INFINITY;
        ls[c] = 0.f;
#pragma unroll
        for (int k = 0; k < kPer; ++k) os[c][k] = 0.f;
        if (s < p.S) {
          const long long i = static_cast<long long>(s) * p.rows + row;
          ms[c] = __ldg(p.st_m + i);
          ls[c] = __ldg(p.st_l + i);
          const float* src = p.st_o + i * D + lane * kPer;
          if constexpr (kPer == 4) {
            const float4 v = __ldg(reinterpret_cast<const float4*>(src));
            os[c][0] = v.x;
            os[c][1] = v.y;
            os[c][2] = v.z;
            os[c][3] = v.w;
          } else {
            const float2 v = __ldg(reinterpret_cast<const float2*>(src));
            os[c][0] = v.x;
            os[c][1] = v.y;
          }
        }
      }
      // new common reference, then every state (and the running one) rescaled to it
      float mc = M;
#pragma unroll
      for (int c = 0; c < kChunk; ++c) mc = fmaxf(mc, ms[c]);
      const float ref = (mc == -INFINITY) ? 0.f : mc;
      const float a = ex2_approx((M - ref) * kLog2e);  // 0 while nothing was seen
      L *= a;
#pragma unroll
      for (int k = 0; k < kPer; ++k) acc[k] *= a;
#pragma unroll
      for (int c = 0; c < kChunk; ++c) {
        const float w = ex2_approx((ms[c] - ref) * kLog2e);  // 0 for an empty state
        L = fmaf(w, ls[c], L);
#pragma unroll
        for (int k = 0; k < kPer; ++k) acc[k] = fmaf(w, os[c][k], acc[k]);
      }
      M = mc;
    }
    // the single final division
    const float inv = L > 0.f ? 1.f / L : 0.f;
    __nv_bfloat16* dst = p.O + row * D + lane * kPer;
    if constexpr (kPer == 4) {
      uint2 packed;
      packed.x = pack_bf16x2(acc[0] * inv, acc[1] * inv);
      packed.y = pack_bf16x2(acc[2] * inv, acc[3] * inv);
      *reinterpret_cast<uint2*>(dst) = packed;
    } else {
      *reinterpret_cast<uint32_t*>(dst) = pack_bf16x2(acc[0] * inv, acc[1] * inv);
    }
    if (lane == 0) p.lse[row] = L > 0.f ? M + logf(L) : -INFINITY;
  }
}

}  // namespace attn
