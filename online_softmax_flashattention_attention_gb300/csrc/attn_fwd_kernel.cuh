// Fused attention forward with the online-softmax recurrence, sm_103a.
//
// One CTA computes two tiles of 128 query rows (256 consecutive rows) of one
// (batch, head).  Warp roles:
//   warps 0-3  softmax of tile 0, warps 4-7 softmax of tile 1: thread t of a group owns
//              query row t of its tile (tensor-memory lane t).  Per key block it reads
//              the score row S from tensor memory, masks, takes the block max, computes
//              alpha and p = exp2(c*s - m), updates l, writes P (bf16) back into tensor
//              memory over its own S, and rescales the output accumulator o~ by alpha
//              when any row of its warp saw the max rise.  At the end it divides o~ by
//              l once and writes O (TMA store) and LSE.
//   warp 8     MMA issuer: tcgen05.mma S_t = Q_t K^T (both operands in shared memory)
//              and o~_t += P_t V (P from tensor memory, V from shared memory), alternating
//              between the two tiles so the tensor core works on one tile while the
//              other tile's softmax runs.
//   warp 9     producer: TMA loads of the two Q tiles and of K/V blocks into a ring of
//              shared-memory stages guarded by full/empty mbarriers.  Both tiles share
//              each K/V block.
//
// The recurrence is the block-wise update of "FlashAttention math" (aicassindra.com),
// section "The block-wise update, and the full algorithm", and of "2.2b: FlashAttention
// -- Online Softmax", section "The Complete Online Softmax Algorithm", carried in the
// log2 domain: with c = scale * log2(e), m2 = c * max(q.k) and p = exp2(c * q.k - m2),
// which equals exp(s - max s) for the scaled scores s.  Masked scores are -inf before
// the block max ("Pitfalls in implementing the recurrence").  While a row has seen no
// visible key its reference point is 0, so alpha = p = 0 and a row with no visible key
// ends with l = 0, O = 0 and LSE = -inf.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "ptx.cuh"

namespace attn {

constexpr int kBM = 128;           // query rows per tile (= tensor-memory lanes)
constexpr int kTiles = 2;          // query tiles per CTA
constexpr int kRowsPerCta = kBM * kTiles;
constexpr int kBN = 128;           // keys per block
constexpr int kWarpMma = 8;
constexpr int kWarpTma = 9;
constexpr int kThreads = 384;      // 2 softmax warpgroups + a warpgroup holding the MMA and producer warps
constexpr uint32_t kTmemCols = 512;
// Register split.  The CTA is launched with kLaunchRegs per thread (384 x 168 = 64512, the
// most three warps per scheduler partition allow); the MMA/producer warpgroup then gives
// registers back and the two softmax warpgroups take them:
// 2 x 128 x 208 + 128 x 88 = 64512.  The host refuses to launch a build whose register
// count differs from kLaunchRegs, since setmaxnreg.inc would then wait for registers
// that never come free.
constexpr int kLaunchRegs = 168;
constexpr int kSoftmaxRegs = 208;
constexpr int kOtherRegs = 88;
static_assert(2 * 128 * kSoftmaxRegs + 128 * kOtherRegs <= kThreads * kLaunchRegs, "register split");

struct FwdParams {
  int BH, H, Nq, Nk;
  int units_per_bh;        // ceil(Nq / 256)
  int causal;
  float c;                 // scale * log2(e)
  const int32_t* lens;     // per-batch key lengths or null
  float* lse;              // [BH, Nq]
  uint32_t* status;        // device status word (bit 0: a wait ran out)
  unsigned long long timeout_ns;
};

template <int D>
struct FwdCfg {
  static constexpr int kSub = D / 64;                 // 64-column swizzle sub-tiles per row tile
  static constexpr int kSubBytes = 128 * 128;         // 128 rows x 64 bf16 = 16 KiB
  static constexpr int kTileBytes = kSub * kSubBytes; // 128 rows x D bf16
  static constexpr int kStages = (D == 128) ? 2 : 4;  // K/V ring depth
  static constexpr int kOffQ = 0;                     // Q tile t at kOffQ + t * kTileBytes
  static constexpr int kOffK = kTiles * kTileBytes;
  static constexpr int kOffV = kOffK + kStages * kTileBytes;
  static constexpr int kOffBar = kOffV + kStages * kTileBytes;
  // barriers: q_full[2], k_full[S], k_empty[S], v_full[S], v_empty[S], s_full[2], p_full[2],
  // pv_done[2], mma_done
  static constexpr int kNumBars = 2 + 4 * kStages + 2 + 2 + 2 + 1;
  static constexpr int kOffMisc = kOffBar + 8 * kNumBars;  // tmem base, abort flag
  static constexpr int kSmemBytes = kOffMisc + 16;
  static constexpr int kSmemAlloc = kSmemBytes + 1024;     // slack to align the base to 1024 B
  // tensor-memory columns: S_t (P_t aliases its first 64 columns), then o~_t
  __host__ __device__ static constexpr uint32_t col_s(int t) { return 128u * t; }
  __host__ __device__ static constexpr uint32_t col_o(int t) { return 256u + D * t; }
  static constexpr uint32_t kIdescS = idesc_bf16_f32(kBM, kBN, 0);
  static constexpr uint32_t kIdescO = idesc_bf16_f32(kBM, D, 1);
};

// Visible keys of a row are exactly j < limit(row): both the key padding and the
// bottom-right causal bound are upper bounds on the key index.
__device__ __forceinline__ int row_key_limit(int row, int kv_len, int Nq, int Nk, int causal) {
  if (!causal) return kv_len;
  const long long lim = static_cast<long long>(row) + Nk - Nq + 1;
  return lim < kv_len ? static_cast<int>(lim < 0 ? 0 : lim) : kv_len;
}

__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmO,
                    const FwdParams p) {
  using C = FwdCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t sK = sbase + C::kOffK;
  const uint32_t sV = sbase + C::kOffV;
  const uint32_t bar0 = sbase + C::kOffBar;
  auto sQ = [&](int t) { return sbase + C::kOffQ + t * C::kTileBytes; };
  auto bar_q_full = [&](int t) { return bar0 + 8u * t; };
  auto bar_k_full = [&](int s) { return bar0 + 8u * (2 + s); };
  auto bar_k_empty = [&](int s) { return bar0 + 8u * (2 + C::kStages + s); };
  auto bar_v_full = [&](int s) { return bar0 + 8u * (2 + 2 * C::kStages + s); };
  auto bar_v_empty = [&](int s) { return bar0 + 8u * (2 + 3 * C::kStages + s); };
  auto bar_s_full = [&](int t) { return bar0 + 8u * (2 + 4 * C::kStages + t); };
  auto bar_p_full = [&](int t) { return bar0 + 8u * (4 + 4 * C::kStages + t); };
  auto bar_pv_done = [&](int t) { return bar0 + 8u * (6 + 4 * C::kStages + t); };
  const uint32_t bar_mma_done = bar0 + 8u * (8 + 4 * C::kStages);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kOffMisc);
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(smem + C::kOffMisc + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // ---- work unit: heads in order (their K/V stay in L2 while their units run);
  //      within a head, causal units longest first
  const int ub = p.units_per_bh;
  const int bh = blockIdx.x / ub;
  int u = blockIdx.x % ub;
  if (p.causal) u = ub - 1 - u;
  const int b = bh / p.H;
  const int q0 = u * kRowsPerCta;
  int kv_len = p.Nk;
  if (p.lens) {
    const int L = __ldg(p.lens + b);
    kv_len = L < 0 ? 0 : (L > p.Nk ? p.Nk : L);
  }
  // per tile: number of key blocks with a visible key, and the key limit of its first row
  int nb[kTiles], min_limit[kTiles];
  bool has_rows[kTiles];
#pragma unroll
  for (int t = 0; t < kTiles; ++t) {
    const int qt0 = q0 + t * kBM;
    has_rows[t] = qt0 < p.Nq;
    const int qlast = min(qt0 + kBM - 1, p.Nq - 1);
    const int max_limit = has_rows[t] ? row_key_limit(qlast, kv_len, p.Nq, p.Nk, p.causal) : 0;
    min_limit[t] = row_key_limit(qt0, kv_len, p.Nq, p.Nk, p.causal);
    nb[t] = max_limit > 0 ? (max_limit + kBN - 1) / kBN : 0;
  }
  const int nblk = max(nb[0], nb[1]);

  WaitCtx wc{abort_flag, p.status, p.timeout_ns};

  if (threadIdx.x == 0) {
    for (int t = 0; t < kTiles; ++t) {
      mbar_init(bar_q_full(t), 1);
      mbar_init(bar_s_full(t), 1);
      mbar_init(bar_p_full(t), 4);
      mbar_init(bar_pv_done(t), 1);
    }
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(bar_k_full(s), 1);
      mbar_init(bar_k_empty(s), 1);
      mbar_init(bar_v_full(s), 1);
      mbar_init(bar_v_empty(s), 1);
    }
    mbar_init(bar_mma_done, 1);
    *abort_flag = 0u;
    fence_mbar_init();
  }
  if (warp == kWarpMma) tmem_alloc<kTmemCols>(smem_u32(tmem_slot));
  if (warp == kWarpTma && lane == 0) {
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
    tma_prefetch_desc(&tmO);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp >= 8) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kOtherRegs));
    if (warp == kWarpTma) {
      // ============================================================== producer
      if (lane == 0 && nblk > 0) {
        const uint64_t pol_kv = policy_evict_last();
        const uint64_t pol_q = policy_evict_first();
#pragma unroll
        for (int t = 0; t < kTiles; ++t) {
          if (nb[t] == 0) continue;
          mbar_arrive_expect_tx(bar_q_full(t), C::kTileBytes);
          for (int s = 0; s < C::kSub; ++s)
            tma_load_3d(sQ(t) + s * C::kSubBytes, &tmQ, bar_q_full(t), s * 64, q0 + t * kBM, bh, pol_q);
        }
        int k_issued = 0, v_issued = 0;
        for (int j = 0; j < nblk; ++j) {
          const int st = j % C::kStages;
          const uint32_t ph = (j / C::kStages) & 1;
          if (!mbar_wait(bar_k_empty(st), ph ^ 1, wc, 1)) break;
          mbar_arrive_expect_tx(bar_k_full(st), C::kTileBytes);
          for (int s = 0; s < C::kSub; ++s)
            tma_load_3d(sK + st * C::kTileBytes + s * C::kSubBytes, &tmK, bar_k_full(st), s * 64, j * kBN, bh,
                        pol_kv);
          k_issued = j + 1;
          if (!mbar_wait(bar_v_empty(st), ph ^ 1, wc, 2)) break;
          mbar_arrive_expect_tx(bar_v_full(st), C::kTileBytes);
          for (int s = 0; s < C::kSub; ++s)
            tma_load_3d(sV + st * C::kTileBytes + s * C::kSubBytes, &tmV, bar_v_full(st), s * 64, j * kBN, bh,
                        pol_kv);
          v_issued = j + 1;
        }
        if (*abort_flag) {
          // let the copies already issued land before the CTA exits
          for (int i = (k_issued > C::kStages ? k_issued - C::kStages : 0); i < k_issued; ++i)
            mbar_wait_drain(bar_k_full(i % C::kStages), (i / C::kStages) & 1, p.timeout_ns);
          for (int i = (v_issued > C::kStages ? v_issued - C::kStages : 0); i < v_issued; ++i)
            mbar_wait_drain(bar_v_full(i % C::kStages), (i / C::kStages) & 1, p.timeout_ns);
        }
      }
    } else if (warp == kWarpMma) {
      // ============================================================== MMA issuer
      if (lane == 0 && nblk > 0) {
        // Shared-memory descriptors: the high word (stride 1024 B, version 1, 128-byte
        // swizzle) is the same for every operand; the low word holds the start address
        // (>> 4) and the leading byte offset, so a k-step is one add to the low word.
        const uint32_t dhi = (1024u >> 4) | (1u << 14) | (2u << 29);
        const uint32_t qlo0 = (sQ(0) >> 4) | (1u << 16);
        const uint32_t qlo1 = (sQ(1) >> 4) | (1u << 16);
        const uint32_t klo = (sK >> 4) | (1u << 16);
        const uint32_t vlo = (sV >> 4) | (static_cast<uint32_t>(C::kSubBytes >> 4) << 16);
        const uint32_t ts0 = tmem + C::col_s(0), ts1 = tmem + C::col_s(1);
        const uint32_t to0 = tmem + C::col_o(0), to1 = tmem + C::col_o(1);
        const int nb0 = nb[0], nb1 = nb[1];
        // S_t = Q_t K_j^T: 8 (d = 128) or 4 (d = 64) k-steps of 16
        auto issue_s = [&](int t, int j) {
          const uint32_t alo = t ? qlo1 : qlo0;
          const uint32_t blo = klo + (j % C::kStages) * (C::kTileBytes >> 4);
          const uint32_t d = t ? ts1 : ts0;
#pragma unroll
          for (int ks = 0; ks < D / 16; ++ks) {
            const uint32_t off = (ks / 4) * (C::kSubBytes >> 4) + (ks % 4) * 2;
            mma_ss(d, (static_cast<uint64_t>(dhi) << 32) | (alo + off), (static_cast<uint64_t>(dhi) << 32) | (blo + off),
                   C::kIdescS, ks > 0 ? 1u : 0u);
          }
          mma_commit(bar_s_full(t));
        };
        // o~_t += P_t V_j: 8 k-steps of 16 keys; A = P_t from tensor memory, B = V_j MN-major
        auto issue_pv = [&](int t, int j) {
          const uint32_t blo = vlo + (j % C::kStages) * (C::kTileBytes >> 4);
          const uint32_t a = t ? ts1 : ts0;
          const uint32_t d = t ? to1 : to0;
#pragma unroll
          for (int ks = 0; ks < kBN / 16; ++ks)
            mma_ts(d, a + ks * 8, (static_cast<uint64_t>(dhi) << 32) | (blo + ks * (16 * 128 >> 4)), C::kIdescO,
                   (j > 0 || ks > 0) ? 1u : 0u);
          mma_commit(bar_pv_done(t));
        };
        bool ok = mbar_wait(bar_k_full(0), 0, wc, 3);
        if (ok && nb0 > 0) {
          ok = mbar_wait(bar_q_full(0), 0, wc, 4);
          tc_fence_after();
          if (ok) issue_s(0, 0);
        }
        if (ok && nb1 > 0) {
          ok = mbar_wait(bar_q_full(1), 0, wc, 4);
          tc_fence_after();
          if (ok) issue_s(1, 0);
        }
        if (ok) mma_commit(bar_k_empty(0));
        for (int j = 0; ok && j < nblk; ++j) {
          const int st = j % C::kStages;
          ok = mbar_wait(bar_v_full(st), (j / C::kStages) & 1, wc, 5);
          bool k_next = false;
#pragma unroll
          for (int t = 0; t < kTiles; ++t) {
            const int nbt = t ? nb1 : nb0;
            if (!ok || j >= nbt) continue;
            ok = mbar_wait(bar_p_full(t), j & 1, wc, 6);
            if (!ok) continue;
            tc_fence_after();
            issue_pv(t, j);
            if (j + 1 < nbt) {
              if (!k_next) {
                ok = mbar_wait(bar_k_full((j + 1) % C::kStages), ((j + 1) / C::kStages) & 1, wc, 7);
                k_next = true;
              }
              // S_t(j+1) overwrites P_t(j): wait until P_t(j) V has been consumed
              ok = ok && mbar_wait(bar_pv_done(t), j & 1, wc, 8);
              if (!ok) continue;
              tc_fence_after();
              issue_s(t, j + 1);
            }
          }
          if (!ok) break;
          mma_commit(bar_v_empty(st));
          if (k_next) mma_commit(bar_k_empty((j + 1) % C::kStages));
        }
        // every MMA this thread issued must finish before tensor memory is released
        mma_commit(bar_mma_done);
        mbar_wait_drain(bar_mma_done, 0, p.timeout_ns);
      }
    }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kSoftmaxRegs));
    // ================================================================ softmax / epilogue
    const int t = warp >> 2;               // tile of this warpgroup
    const int r = threadIdx.x & 127;       // row within the tile = tensor-memory lane
    const int row = q0 + t * kBM + r;
    const int limit = row_key_limit(row, kv_len, p.Nq, p.Nk, p.causal);
    const uint32_t tl = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);
    const uint32_t colS = C::col_s(t), colO = C::col_o(t);
    const float c = p.c;
    const int my_nb = t ? nb[1] : nb[0];
    const int my_min_limit = t ? min_limit[1] : min_limit[0];
    const bool my_has_rows = t ? has_rows[1] : has_rows[0];
    float m = -INFINITY;  // running max, log2 domain
    float l = 0.f;        // running denominator
    bool ok = true;
    for (int j = 0; j < my_nb; ++j) {
      // every lane of the warp takes the same branch: the tcgen05 loads below are warp-wide
      ok = __all_sync(0xffffffffu, mbar_wait(bar_s_full(t), j & 1, wc, 9));
      if (!ok) break;
      tc_fence_after();
      uint32_t sr[kBN];
#pragma unroll
      for (int q = 0; q < kBN / 32; ++q) tmem_ld32(tl + colS + q * 32, sr + q * 32);
      tmem_wait_ld();
      float s[kBN];
#pragma unroll
      for (int k = 0; k < kBN; ++k) s[k] = __uint_as_float(sr[k]);
      const int kb = j * kBN;
      if (kb + kBN > my_min_limit) {
#pragma unroll
        for (int k = 0; k < kBN; ++k)
          if (kb + k >= limit) s[k] = -INFINITY;
      }
      // block max: four independent chains of 3-input max over s[0..kBN)
      float a0 = fmaxf(s[0], s[1]), a1 = fmaxf(s[2], s[3]), a2 = fmaxf(s[4], s[5]), a3 = fmaxf(s[6], s[7]);
#pragma unroll
      for (int k = 8; k < kBN; k += 8) {
        a0 = fmax3(a0, s[k], s[k + 1]);
        a1 = fmax3(a1, s[k + 2], s[k + 3]);
        a2 = fmax3(a2, s[k + 4], s[k + 5]);
        a3 = fmax3(a3, s[k + 6], s[k + 7]);
      }
      const float mx = fmaxf(fmaxf(a0, a1), fmaxf(a2, a3));
      const float m_new = fmaxf(m, mx * c);
      const float m_ref = (m_new == -INFINITY) ? 0.f : m_new;
      const float alpha = ex2_approx(m - m_ref);
      // p = exp2(c*s - m_ref), summed in fp32, packed to bf16 and stored 32 keys at a time
      const float2 c2 = make_float2(c, c);
      const float2 nm2 = make_float2(-m_ref, -m_ref);
      float2 acc0 = make_float2(0.f, 0.f), acc1 = make_float2(0.f, 0.f);
#pragma unroll
      for (int q = 0; q < kBN / 32; ++q) {
        uint32_t pk[16];
#pragma unroll
        for (int k = 0; k < 16; ++k) {
          float2 x = __ffma2_rn(make_float2(s[q * 32 + 2 * k], s[q * 32 + 2 * k + 1]), c2, nm2);
          x.x = ex2_approx(x.x);
          x.y = ex2_approx(x.y);
          if (k & 1)
            acc1 = __fadd2_rn(acc1, x);
          else
            acc0 = __fadd2_rn(acc0, x);
          pk[k] = pack_bf16x2(x.x, x.y);
        }
        tmem_st16(tl + colS + q * 16, pk);
      }
      const float2 acc = __fadd2_rn(acc0, acc1);
      l = l * alpha + (acc.x + acc.y);
      m = m_new;
      if (j > 0 && !__all_sync(0xffffffffu, alpha == 1.f)) {
        // o~ may be touched only after the previous P V product has landed in it
        ok = __all_sync(0xffffffffu, mbar_wait(bar_pv_done(t), (j - 1) & 1, wc, 10));
        if (!ok) break;
        tc_fence_after();
        const float2 al2 = make_float2(alpha, alpha);
#pragma unroll
        for (int q = 0; q < D / 64; ++q) {
          uint32_t o[64];
          tmem_ld32(tl + colO + q * 64, o);
          tmem_ld32(tl + colO + q * 64 + 32, o + 32);
          tmem_wait_ld();
#pragma unroll
          for (int k = 0; k < 32; ++k) {
            float2 v = __fmul2_rn(make_float2(__uint_as_float(o[2 * k]), __uint_as_float(o[2 * k + 1])), al2);
            o[2 * k] = __float_as_uint(v.x);
            o[2 * k + 1] = __float_as_uint(v.y);
          }
          tmem_st32(tl + colO + q * 64, o);
          tmem_st32(tl + colO + q * 64 + 32, o + 32);
        }
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_p_full(t));
    }
    // ---- epilogue: one division by l, O through shared memory and a TMA store, LSE direct
    if (ok && my_nb > 0) {
      ok = __all_sync(0xffffffffu, mbar_wait(bar_pv_done(t), (my_nb - 1) & 1, wc, 11));
      tc_fence_after();
    }
    // one decision for the four warps of this tile (the named barriers below need all of them)
    const bool give_up = bar_sync_or(1 + t, 128, !ok || *abort_flag != 0u);
    if (!give_up && my_has_rows) {
      const float inv = l > 0.f ? 1.f / l : 0.f;
      uint8_t* orow = smem + C::kOffQ + t * C::kTileBytes + r * 128;
#pragma unroll
      for (int q = 0; q < D / 32; ++q) {
        uint32_t o[32];
        if (my_nb > 0) {
          tmem_ld32(tl + colO + q * 32, o);
          tmem_wait_ld();
        } else {
#pragma unroll
          for (int k = 0; k < 32; ++k) o[k] = 0u;
        }
        // 32 columns = four 16-byte chunks of sub-tile q/2, chunk (q%2)*4 + ch, 128-byte swizzle
#pragma unroll
        for (int ch = 0; ch < 4; ++ch) {
          uint4 v;
          v.x = pack_bf16x2(__uint_as_float(o[ch * 8 + 0]) * inv, __uint_as_float(o[ch * 8 + 1]) * inv);
          v.y = pack_bf16x2(__uint_as_float(o[ch * 8 + 2]) * inv, __uint_as_float(o[ch * 8 + 3]) * inv);
          v.z = pack_bf16x2(__uint_as_float(o[ch * 8 + 4]) * inv, __uint_as_float(o[ch * 8 + 5]) * inv);
          v.w = pack_bf16x2(__uint_as_float(o[ch * 8 + 6]) * inv, __uint_as_float(o[ch * 8 + 7]) * inv);
          const int chunk = (q % 2) * 4 + ch;
          *reinterpret_cast<uint4*>(orow + (q / 2) * C::kSubBytes + ((chunk ^ (r & 7)) * 16)) = v;
        }
      }
      if (row < p.Nq) {
        const float lse = l > 0.f ? (m + __log2f(l)) * 0.69314718055994531f : -INFINITY;
        p.lse[static_cast<size_t>(bh) * p.Nq + row] = lse;
      }
      fence_proxy_async_smem();
      bar_sync_named(1 + t, 128);
      if (r == 0) {
        for (int s = 0; s < C::kSub; ++s) tma_store_3d(&tmO, sQ(t) + s * C::kSubBytes, s * 64, q0 + t * kBM, bh);
        tma_store_commit();
        tma_store_wait_all();
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kWarpMma) {
    tc_fence_after();
    tmem_dealloc<kTmemCols>(tmem);
  }
}

}  // namespace attn
