// Fused attention forward with the online-softmax recurrence, sm_103a.
//
// One CTA computes one tile of 128 query rows of one (batch, head).  Warp roles:
//   warps 0-3  softmax: thread t owns query row t (tensor-memory lane t).  Per key
//              block it reads the score row S from tensor memory, masks, takes the
//              block max, computes alpha and p = exp2(c*s - m), updates l, writes P
//              (bf16) back into tensor memory over its own S, and rescales the
//              output accumulator o~ by alpha when any row of its warp saw the max rise.
//              At the end it divides o~ by l once and writes O (TMA store) and LSE.
//   warp 4     producer: TMA loads of the Q tile and of K/V blocks into a ring of
//              shared-memory stages guarded by full/empty mbarriers.
//   warp 5     MMA issuer: tcgen05.mma S = Q K^T (both operands in shared memory) into
//              one of two tensor-memory score buffers, then o~ += P V (P from tensor
//              memory, V from shared memory) into the tensor-memory accumulator.
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

constexpr int kBM = 128;        // query rows per tile (= tensor-memory lanes)
constexpr int kBN = 128;        // keys per block
constexpr int kThreads = 192;   // 4 softmax warps + producer + MMA
constexpr uint32_t kTmemCols = 512;

struct FwdParams {
  int BH, H, Nq, Nk;
  int num_qtiles;
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
  static constexpr int kOffQ = 0;
  static constexpr int kOffK = kTileBytes;
  static constexpr int kOffV = kOffK + kStages * kTileBytes;
  static constexpr int kOffBar = kOffV + kStages * kTileBytes;
  // barriers: q, k_full[S], k_empty[S], v_full[S], v_empty[S], s_full[2], p_full[2], pv_done[2], mma_done
  static constexpr int kNumBars = 1 + 4 * kStages + 2 + 2 + 2 + 1;
  static constexpr int kOffMisc = kOffBar + 8 * kNumBars;  // tmem base, abort flag
  static constexpr int kSmemBytes = kOffMisc + 16;
  static constexpr int kSmemAlloc = kSmemBytes + 1024;     // slack to align the base to 1024 B
  // tensor-memory columns
  static constexpr uint32_t kColS0 = 0, kColS1 = 128, kColO = 256;
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

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmO,
                    const FwdParams p) {
  using C = FwdCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t sQ = sbase + C::kOffQ;
  const uint32_t sK = sbase + C::kOffK;
  const uint32_t sV = sbase + C::kOffV;
  const uint32_t bar0 = sbase + C::kOffBar;
  const uint32_t bar_q = bar0;
  auto bar_k_full = [&](int s) { return bar0 + 8u * (1 + s); };
  auto bar_k_empty = [&](int s) { return bar0 + 8u * (1 + C::kStages + s); };
  auto bar_v_full = [&](int s) { return bar0 + 8u * (1 + 2 * C::kStages + s); };
  auto bar_v_empty = [&](int s) { return bar0 + 8u * (1 + 3 * C::kStages + s); };
  auto bar_s_full = [&](int b) { return bar0 + 8u * (1 + 4 * C::kStages + b); };
  auto bar_p_full = [&](int b) { return bar0 + 8u * (3 + 4 * C::kStages + b); };
  auto bar_pv_done = [&](int b) { return bar0 + 8u * (5 + 4 * C::kStages + b); };
  const uint32_t bar_mma_done = bar0 + 8u * (7 + 4 * C::kStages);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kOffMisc);
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(smem + C::kOffMisc + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // ---- work unit: longest causal tiles first
  const int BH = p.BH;
  const int idx = blockIdx.x;
  const int qtile = p.causal ? (p.num_qtiles - 1 - idx / BH) : (idx / BH);
  const int bh = idx % BH;
  const int b = bh / p.H;
  const int q0 = qtile * kBM;
  int kv_len = p.Nk;
  if (p.lens) {
    const int L = __ldg(p.lens + b);
    kv_len = L < 0 ? 0 : (L > p.Nk ? p.Nk : L);
  }
  const int qlast = min(q0 + kBM - 1, p.Nq - 1);
  const int max_limit = row_key_limit(qlast, kv_len, p.Nq, p.Nk, p.causal);
  const int min_limit = row_key_limit(q0, kv_len, p.Nq, p.Nk, p.causal);
  const int nblk = max_limit > 0 ? (max_limit + kBN - 1) / kBN : 0;

  WaitCtx wc{abort_flag, p.status, p.timeout_ns};

  if (threadIdx.x == 0) {
    mbar_init(bar_q, 1);
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(bar_k_full(s), 1);
      mbar_init(bar_k_empty(s), 1);
      mbar_init(bar_v_full(s), 1);
      mbar_init(bar_v_empty(s), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar_s_full(i), 1);
      mbar_init(bar_p_full(i), 4);
      mbar_init(bar_pv_done(i), 1);
    }
    mbar_init(bar_mma_done, 1);
    *abort_flag = 0u;
    fence_mbar_init();
  }
  if (warp == 5) tmem_alloc<kTmemCols>(smem_u32(tmem_slot));
  if (warp == 4 && lane == 0) {
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
    tma_prefetch_desc(&tmO);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 4) {
    // ================================================================ producer
    if (lane == 0 && nblk > 0) {
      const uint64_t pol_kv = policy_evict_last();
      const uint64_t pol_q = policy_evict_first();
      mbar_arrive_expect_tx(bar_q, C::kTileBytes);
      for (int s = 0; s < C::kSub; ++s) tma_load_3d(sQ + s * C::kSubBytes, &tmQ, bar_q, s * 64, q0, bh, pol_q);
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
  } else if (warp == 5) {
    // ================================================================ MMA issuer
    if (lane == 0 && nblk > 0) {
      bool ok = mbar_wait(bar_q, 0, wc, 3);
      tc_fence_after();
      auto issue_pv = [&](int i) -> bool {
        const int sb = i & 1;
        if (!mbar_wait(bar_p_full(sb), (i >> 1) & 1, wc, 4)) return false;
        const int st = i % C::kStages;
        if (!mbar_wait(bar_v_full(st), (i / C::kStages) & 1, wc, 5)) return false;
        tc_fence_after();
        const uint32_t vbase = sV + st * C::kTileBytes;
#pragma unroll
        for (int ks = 0; ks < kBN / 16; ++ks) {
          const uint64_t bdesc = smem_desc_sw128(vbase + ks * 16 * 128, C::kSubBytes, 1024);
          mma_ts(tmem + C::kColO, tmem + (sb ? C::kColS1 : C::kColS0) + ks * 8, bdesc, C::kIdescO,
                 (i > 0 || ks > 0) ? 1u : 0u);
        }
        mma_commit(bar_pv_done(sb));
        mma_commit(bar_v_empty(st));
        return true;
      };
      for (int j = 0; ok && j < nblk; ++j) {
        const int sb = j & 1;
        if (j >= 2) {
          if (!mbar_wait(bar_pv_done(sb), ((j - 2) >> 1) & 1, wc, 6)) break;
        }
        const int st = j % C::kStages;
        if (!mbar_wait(bar_k_full(st), (j / C::kStages) & 1, wc, 7)) break;
        tc_fence_after();
        const uint32_t kbase = sK + st * C::kTileBytes;
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          const uint32_t off = (ks / 4) * C::kSubBytes + (ks % 4) * 32;
          const uint64_t adesc = smem_desc_sw128(sQ + off, 16, 1024);
          const uint64_t bdesc = smem_desc_sw128(kbase + off, 16, 1024);
          mma_ss(tmem + (sb ? C::kColS1 : C::kColS0), adesc, bdesc, C::kIdescS, ks > 0 ? 1u : 0u);
        }
        mma_commit(bar_s_full(sb));
        mma_commit(bar_k_empty(st));
        if (j >= 1 && !issue_pv(j - 1)) {
          ok = false;
          break;
        }
      }
      if (ok && !*abort_flag) issue_pv(nblk - 1);
      // every MMA this thread issued must finish before tensor memory is released
      mma_commit(bar_mma_done);
      mbar_wait_drain(bar_mma_done, 0, p.timeout_ns);
    }
  } else {
    // ================================================================ softmax / epilogue
    const int t = threadIdx.x;  // 0..127: row within the tile and tensor-memory lane
    const int row = q0 + t;
    const int limit = row_key_limit(row, kv_len, p.Nq, p.Nk, p.causal);
    const uint32_t tl = tmem + (static_cast<uint32_t>(warp * 32) << 16);
    const float c = p.c;
    float m = -INFINITY;  // running max, log2 domain
    float l = 0.f;        // running denominator
    bool ok = true;
    for (int j = 0; j < nblk; ++j) {
      const int sb = j & 1;
      const uint32_t scol = sb ? C::kColS1 : C::kColS0;
      // every lane of the warp takes the same branch: the tcgen05 loads below are warp-wide
      ok = __all_sync(0xffffffffu, mbar_wait(bar_s_full(sb), (j >> 1) & 1, wc, 8));
      if (!ok) break;
      tc_fence_after();
      uint32_t sr[kBN];
#pragma unroll
      for (int q = 0; q < kBN / 32; ++q) tmem_ld32(tl + scol + q * 32, sr + q * 32);
      tmem_wait_ld();
      float s[kBN];
#pragma unroll
      for (int k = 0; k < kBN; ++k) s[k] = __uint_as_float(sr[k]);
      const int kb = j * kBN;
      if (kb + kBN > min_limit) {
#pragma unroll
        for (int k = 0; k < kBN; ++k)
          if (kb + k >= limit) s[k] = -INFINITY;
      }
      float mx = s[0];
#pragma unroll
      for (int k = 1; k < kBN; ++k) mx = fmaxf(mx, s[k]);
      const float m_new = fmaxf(m, mx * c);
      const float m_ref = (m_new == -INFINITY) ? 0.f : m_new;
      const float alpha = ex2_approx(m - m_ref);
      float rs = 0.f;
#pragma unroll
      for (int k = 0; k < kBN; ++k) {
        s[k] = ex2_approx(fmaf(s[k], c, -m_ref));
        rs += s[k];
      }
      l = l * alpha + rs;
      m = m_new;
      uint32_t pk[kBN / 2];
#pragma unroll
      for (int k = 0; k < kBN / 2; ++k) pk[k] = pack_bf16x2(s[2 * k], s[2 * k + 1]);
      if (j > 0) {
        // o~ may be touched only after the previous P V product has landed in it
        ok = __all_sync(0xffffffffu, mbar_wait(bar_pv_done((j - 1) & 1), ((j - 1) >> 1) & 1, wc, 9));
        if (!ok) break;
        tc_fence_after();
        if (!__all_sync(0xffffffffu, alpha == 1.f)) {
#pragma unroll
          for (int q = 0; q < D / 32; ++q) {
            uint32_t o[32];
            tmem_ld32(tl + C::kColO + q * 32, o);
            tmem_wait_ld();
#pragma unroll
            for (int k = 0; k < 32; ++k) o[k] = __float_as_uint(__uint_as_float(o[k]) * alpha);
            tmem_st32(tl + C::kColO + q * 32, o);
          }
        }
      }
      tmem_st32(tl + scol, pk);
      tmem_st32(tl + scol + 32, pk + 32);
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_p_full(sb));
    }
    // ---- epilogue: one division by l, O through shared memory and a TMA store, LSE direct
    if (ok && nblk > 0) {
      ok = __all_sync(0xffffffffu,
                      mbar_wait(bar_pv_done((nblk - 1) & 1), ((nblk - 1) >> 1) & 1, wc, 10));
      tc_fence_after();
    }
    // one decision for all four softmax warps (the named barriers below need all of them)
    const bool give_up = bar_sync_or(1, 128, !ok || *abort_flag != 0u);
    if (!give_up) {
      const float inv = l > 0.f ? 1.f / l : 0.f;
      uint8_t* orow = smem + C::kOffQ + t * 128;
#pragma unroll
      for (int q = 0; q < D / 32; ++q) {
        uint32_t o[32];
        if (nblk > 0) {
          tmem_ld32(tl + C::kColO + q * 32, o);
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
          *reinterpret_cast<uint4*>(orow + (q / 2) * C::kSubBytes + ((chunk ^ (t & 7)) * 16)) = v;
        }
      }
      if (row < p.Nq) {
        const float lse = l > 0.f ? (m + __log2f(l)) * 0.69314718055994531f : -INFINITY;
        p.lse[static_cast<size_t>(bh) * p.Nq + row] = lse;
      }
      fence_proxy_async_smem();
      bar_sync_named(1, 128);
      if (t == 0) {
        for (int s = 0; s < C::kSub; ++s) tma_store_3d(&tmO, sQ + s * C::kSubBytes, s * 64, q0, bh);
        tma_store_commit();
        tma_store_wait_all();
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 5) {
    tc_fence_after();
    tmem_dealloc<kTmemCols>(tmem);
  }
}

}  // namespace attn
