// Fused attention forward at d = 64 with two query tiles per CTA, sm_103a.
//
// The same computation as attn_fwd_kernel -- the block-wise update of "FlashAttention
// math" (aicassindra.com), section "The block-wise update, and the full algorithm", in the
// log2 domain, with the same masking and fully-masked-row conventions -- scheduled for
// d = 64.  There one tile's softmax warps cannot keep the tensor core busy: a key block's
// exponentials take them about twice as long as the block's two products.  So a CTA takes
// two adjacent 128-row query tiles of one (batch, head) at a time, both reading every K/V
// block it loads, and the softmax warps of the two tiles share the scheduler partitions.
// Warp roles:
//   warps 0-3  softmax of tile 0 (thread r: row r of the tile, tensor-memory lane r)
//   warps 4-7  softmax of tile 1 (the same lanes)
//   warp 8     producer: TMA loads of the two Q tiles and of K_j, V_j into one ring of
//              shared-memory slots (K_j and V_j take one slot each, in load order)
//   warp 9     S issuer, warp 10 P V issuer (each warp runs its loop as a whole; one
//              elected lane issues every MMA and commit)
// The products of a pair of tiles form one sequence: for each key block j the pair loads,
// tile 0's, then tile 1's, q = 2 j + t.  A tile that lacks block j (it sees fewer keys,
// or lies past the end of its sequence) still takes its place in the sequence with an
// empty product, which moves the barriers on without any MMA or arithmetic, so that each
// tile's products stay two apart and every wait stays within one phase of its barrier.
// Product q writes its scores into score buffer q % 3.  With three buffers for two tiles a
// score product waits only for the P V product three places before it, which is always
// the other tile's, never this tile's previous one: neither tile runs S -> softmax ->
// P V -> S in series, and while one tile's softmax warps work the tensor core runs the
// other tile's products.  Tensor memory: three score buffers of 128 columns (P over the first 64 of
// its own buffer) and o~ of each tile (64 columns each), 512 columns in all.
#pragma once

#include "attn_fwd_kernel.cuh"

namespace attn {

// 8 softmax warps + producer + two MMA issuers + one warp without a role, which completes
// the third warpgroup so that setmaxnreg can move registers from that group (producer and
// issuers) to the softmax warps: 224 each instead of the 168 a 12-warp launch gives every
// thread (three warps per scheduler partition of 16384 registers), with no spills.
constexpr int kPairThreads = 384;
constexpr uint32_t kPairRegsSoftmax = 224;
constexpr uint32_t kPairRegsOther = 56;
static_assert(256 * kPairRegsSoftmax + 128 * kPairRegsOther <= 168 * kPairThreads, "register split");
constexpr int kPairWarpTma = 8;
constexpr int kPairWarpS = 9;
constexpr int kPairWarpPv = 10;
constexpr int kPairSBufs = 3;

struct PairCfg {
  static constexpr int D = 64;
  static constexpr int kTileBytes = 128 * 128;  // 128 rows x 64 bf16: one 128-byte-swizzled tile
  static constexpr int kSlots = 10;             // ring slots
  static constexpr int kOffQ = 0;               // Q tile t at kOffQ + t * kTileBytes
  static constexpr int kOffRing = 2 * kTileBytes;
  static constexpr int kOffBar = kOffRing + kSlots * kTileBytes;
  // barriers: q_full, q_free, full[kSlots], free[kSlots], s_full[3], p_full[3], pv_done[3],
  // o_done[2], drain[2]
  static constexpr int kNumBars = 2 + 2 * kSlots + 3 * kPairSBufs + 4;
  static constexpr int kOffMisc = kOffBar + 8 * kNumBars;  // tensor-memory base, abort flag
  static constexpr int kOffPerm = kOffMisc + 16;           // uint16 order of packed sequences
  static constexpr int kSmemBytes = kOffPerm + 2 * kMaxSortedSeqs;
  static constexpr int kSmemAlloc = kSmemBytes + 1024;     // slack to align the base to 1024 B
  static constexpr int kSmemAllocNoPerm = kOffPerm + 1024; // launches without seq_sort
  static_assert(kSmemAlloc <= 232448, "shared memory per CTA");
  __host__ __device__ static constexpr uint32_t col_s(int b) { return 128u * b; }
  __host__ __device__ static constexpr uint32_t col_o(int t) { return 128u * kPairSBufs + 64u * t; }
  static constexpr uint32_t kIdescS = idesc_bf16_f32(kBM, kBN, 0);
  static constexpr uint32_t kIdescO = idesc_bf16_f32(kBM, D, 1);
  static_assert(128u * kPairSBufs + 2u * D <= kTmemCols, "tensor memory");
};

// One work item = query tiles 2i and 2i + 1 of one (batch, head).  Tile 1 may lie past the
// end of the sequence (an odd tile count, or a shorter packed sequence): it then has no
// blocks and no rows.
struct PairItem {
  int bh, b, hh;
  int q_base, k_base;      // first rows of the sequence in the Q / K maps
  int Nq, Nk, bcoord;      // the sequence's lengths and its batch coordinate in the maps
  int kv_len;              // visible keys after padding
  int q0[2];               // first query row of each tile within its sequence
  int min_limit[2];        // smallest key limit of each tile's rows
  int nblk[2];             // key blocks 0 .. nblk[t] - 1 of tile t (0: nothing to compute)
  int nmax;                // max(nblk[0], nblk[1]): blocks the CTA loads
  bool valid[2];           // the tile has rows in its sequence
};

template <bool kPacked>  // as in decode
__device__ __forceinline__ PairItem decode_pair(const FwdParams& p, int item, const uint16_t* seq_perm) {
  PairItem it;
  const int npairs = (p.num_qtiles + 1) >> 1;
  // as decode: head major (heads in order) or rank major (pair rank r of every head, then
  // r + 1), order_div = npairs or B H; within a head, causal pairs longest first
  const int ua = item / p.order_div;
  const int ub = item - ua * p.order_div;
  it.bh = p.rank_major ? ub : ua;
  int pair = p.rank_major ? ua : ub;
  if (p.causal) pair = npairs - 1 - pair;
  it.b = it.bh / p.H;
  it.hh = it.bh - it.b * p.H;
  it.q_base = 0;
  it.k_base = 0;
  it.Nq = p.Nq;
  it.Nk = p.Nk;
  it.bcoord = it.b;
  if (p.cu_q) {
    if constexpr (kPacked) {
      if (p.seq_sort) {  // as in decode: the sequence of this rank in decreasing work
        it.b = seq_perm[it.b];
        it.bh = it.b * p.H + it.hh;
      }
    }
    const int qs = min(max(__ldg(p.cu_q + it.b), 0), p.total_q);
    const int qe = min(max(__ldg(p.cu_q + it.b + 1), qs), p.total_q);
    const int ks = min(max(__ldg(p.cu_k + it.b), 0), p.total_k);
    const int ke = min(max(__ldg(p.cu_k + it.b + 1), ks), p.total_k);
    it.q_base = qs;
    it.k_base = ks;
    it.Nq = qe - qs;
    it.Nk = ke - ks;
    it.bcoord = 0;
  }
  it.kv_len = it.Nk;
  if (p.lens) {
    const int L = __ldg(p.lens + it.b);
    it.kv_len = L < 0 ? 0 : (L > it.Nk ? it.Nk : L);
  }
#pragma unroll
  for (int t = 0; t < 2; ++t) {
    it.q0[t] = (2 * pair + t) * kBM;
    it.valid[t] = it.q0[t] < it.Nq;
    const int qlast = min(it.q0[t] + kBM - 1, it.Nq - 1);
    const int max_limit = row_key_limit(qlast, it.kv_len, it.Nq, it.Nk, p.causal);
    it.min_limit[t] = row_key_limit(it.q0[t], it.kv_len, it.Nq, it.Nk, p.causal);
    const int nvis = max_limit > 0 ? (max_limit + kBN - 1) / kBN : 0;
    it.nblk[t] = it.valid[t] ? nvis : 0;
  }
  it.nmax = max(it.nblk[0], it.nblk[1]);
  return it;
}

// Persistent like attn_fwd_kernel: one CTA per SM walks its pairs in item_of() order; the
// ring, the score buffers and their barrier phases run on from one pair to the next.  Every
// role counts the products over all its pairs (qn; 2 nmax per pair): product q completes
// phase (q / 3) & 1 of s_full, p_full and pv_done[q % 3], empty products included.
// o_done[t] completes once per pair in which tile t has blocks, when its last P V product
// has landed.  Each wait stays within one phase of its barrier: the phase before it has
// completed (a tile's previous product is two places back, and tcgen05 commits of one
// thread complete in order), and the phase after it needs an arrival that comes after the
// wait.
template <int kSoftPairs, bool kPacked>
__global__ void __launch_bounds__(kPairThreads, 1)
    attn_fwd_pair_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                         const __grid_constant__ CUtensorMap tmV, const FwdParams p) {
  using C = PairCfg;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t sQ = sbase + C::kOffQ;
  const uint32_t sRing = sbase + C::kOffRing;
  const uint32_t bar0 = sbase + C::kOffBar;
  const uint32_t bar_q_full = bar0;
  const uint32_t bar_q_free = bar0 + 8u;  // the pair's last S product has read both Q tiles
  auto bar_full = [&](int s) { return bar0 + 8u * (2 + s); };
  auto bar_free = [&](int s) { return bar0 + 8u * (2 + C::kSlots + s); };
  auto bar_s_full = [&](int b) { return bar0 + 8u * (2 + 2 * C::kSlots + b); };
  auto bar_p_full = [&](int b) { return bar0 + 8u * (2 + 2 * C::kSlots + kPairSBufs + b); };
  auto bar_pv_done = [&](int b) { return bar0 + 8u * (2 + 2 * C::kSlots + 2 * kPairSBufs + b); };
  auto bar_o_done = [&](int t) { return bar0 + 8u * (2 + 2 * C::kSlots + 3 * kPairSBufs + t); };
  auto bar_drain = [&](int i) { return bar0 + 8u * (4 + 2 * C::kSlots + 3 * kPairSBufs + i); };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kOffMisc);
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(smem + C::kOffMisc + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int G = static_cast<int>(gridDim.x);
  const int cta = static_cast<int>(blockIdx.x);
  WaitCtx wc{abort_flag, p.status, p.timeout_ns};

  if (threadIdx.x == 0) {
    mbar_init(bar_q_full, 1);
    mbar_init(bar_q_free, 1);
    for (int s = 0; s < C::kSlots; ++s) {
      mbar_init(bar_full(s), 1);
      mbar_init(bar_free(s), 1);
    }
    for (int b = 0; b < kPairSBufs; ++b) {
      mbar_init(bar_s_full(b), 1);
      mbar_init(bar_p_full(b), 4);  // the four softmax warps of the product's tile
      mbar_init(bar_pv_done(b), 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(bar_o_done(t), 1);
      mbar_init(bar_drain(t), 1);
    }
    *abort_flag = 0u;
    fence_mbar_init();
  }
  if (warp == kPairWarpPv) tmem_alloc<kTmemCols>(smem_u32(tmem_slot));
  if (warp == kPairWarpTma && lane == 0) {
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  griddep_wait();  // as in attn_fwd_kernel: the previous kernel has finished from here on
  griddep_launch_dependents();
  uint16_t* seq_perm = reinterpret_cast<uint16_t*>(smem + C::kOffPerm);
  if constexpr (kPacked) {
    if (p.seq_sort) rank_sequences(p, p.BH / p.H, reinterpret_cast<float*>(smem + C::kOffQ), seq_perm);
  }

  if (warp == kPairWarpTma) {
    // ================================================================ producer
    // Warp-wide like the MMA issuers below: one elected lane issues each copy.
    setmaxnreg_dec<kPairRegsOther>();
    {
      const uint64_t pol_kv = policy_evict_last();
      const uint64_t pol_q = policy_evict_first();
      int e = 0;   // ring entries loaded so far over all pairs (K_j, then V_j): slot e % kSlots
      int kq = 0;  // pairs with work so far: uses of the Q tiles
      // Slot s has a copy in flight when bit s of live is set; bit s of par is the phase
      // parity that copy completes (bit masks: an array indexed by the slot would live in
      // local memory).
      uint32_t live = 0, par = 0;
      bool ok = true;
      for (int ri = 0; ok; ++ri) {
        const int item = item_of(ri, cta, G);
        if (item >= p.num_items) break;
        const PairItem it = decode_pair<kPacked>(p, item, seq_perm);
        if (it.nmax == 0) continue;
        // the previous pair's Q tiles must have been read by its last S product
        if (kq > 0 && !__all_sync(0xffffffffu, mbar_wait(bar_q_free, (kq - 1) & 1, wc, 13))) break;
        mbar_arrive_expect_tx_elect(bar_q_full, ((it.nblk[0] > 0) + (it.nblk[1] > 0)) * C::kTileBytes);
#pragma unroll
        for (int t = 0; t < 2; ++t)
          if (it.nblk[t] > 0)
            tma_load_4d_elect(sQ + t * C::kTileBytes, &tmQ, bar_q_full, 0, it.q_base + it.q0[t], it.hh, it.bcoord,
                              pol_q);
        ++kq;
        for (int j = 0; ok && j < it.nmax; ++j) {
          for (int kv = 0; kv < 2; ++kv, ++e) {
            const int slot = e % C::kSlots;
            if (!__all_sync(0xffffffffu, mbar_wait(bar_free(slot), ((e / C::kSlots) & 1) ^ 1, wc, 1 + kv))) {
              ok = false;
              break;
            }
            const uint32_t bit = 1u << slot;
            live &= ~bit;
            // the test hook withholds K of one block: its full barrier never completes
            if (kv == 1 || j != p.fault_block) {
              mbar_arrive_expect_tx_elect(bar_full(slot), C::kTileBytes);
              tma_load_4d_elect(sRing + slot * C::kTileBytes, kv ? &tmV : &tmK, bar_full(slot), 0,
                                it.k_base + j * kBN, it.hh, it.bcoord, pol_kv);
              live |= bit;
              par = (par & ~bit) | (static_cast<uint32_t>((e / C::kSlots) & 1) << slot);
            }
          }
        }
      }
      // Let the copies still in flight land before this warp leaves (in a normal run they
      // were consumed long ago; after a failed wait nobody else will wait for them).
#pragma unroll
      for (int s = 0; s < C::kSlots; ++s)
        if ((live >> s) & 1u) mbar_wait_drain(bar_full(s), (par >> s) & 1u, p.timeout_ns);
    }
  } else if (warp == kPairWarpS || warp == kPairWarpPv) {
    // ================================================================ MMA issuers
    // The whole warp runs the issuer loop (warp-uniform control flow; measured on GB300,
    // 7-9 % faster than one lane running it alone); one elected lane issues each MMA and
    // commit.
    setmaxnreg_dec<kPairRegsOther>();
    {
      // descriptor high word: stride 1024 B, version 1, 128-byte swizzle (as attn_fwd_kernel)
      const uint32_t dhi = (1024u >> 4) | (1u << 14) | (2u << 29);
      int e = (warp == kPairWarpS) ? 0 : 1;  // this issuer's ring entries: K_j even, V_j odd
      int qn = 0;                             // products of the pairs before this one
      int kq = 0;
      bool ok = true;
      for (int ri = 0; ok; ++ri) {
        const int item = item_of(ri, cta, G);
        if (item >= p.num_items) break;
        const PairItem it = decode_pair<kPacked>(p, item, seq_perm);
        if (it.nmax == 0) continue;
        if (warp == kPairWarpS) {
          ok = __all_sync(0xffffffffu, mbar_wait(bar_q_full, kq & 1, wc, 3));
          const uint32_t klo = (sRing >> 4) | (1u << 16);
          for (int j = 0; ok && j < it.nmax; ++j, e += 2) {
            const int slot = e % C::kSlots;
            if (!(ok = __all_sync(0xffffffffu, mbar_wait(bar_full(slot), (e / C::kSlots) & 1, wc, 5)))) break;
#pragma unroll
            for (int t = 0; t < 2; ++t) {
              const int q = qn + 2 * j + t;
              const int b = q % kPairSBufs;
              // buffer b last held the P of product q - 3: its P V product must have read it
              if (q >= kPairSBufs &&
                  !(ok = __all_sync(0xffffffffu,
                                    mbar_wait(bar_pv_done(b), ((q - kPairSBufs) / kPairSBufs) & 1, wc, 4))))
                break;
              if (j < it.nblk[t]) {
                tc_fence_after();
                // S = Q_t K_j^T: 4 k-steps of 16 along d
                const uint32_t qlo = ((sQ + t * C::kTileBytes) >> 4) | (1u << 16);
                const uint32_t blo = klo + slot * (C::kTileBytes >> 4);
#pragma unroll
                for (int ks = 0; ks < C::D / 16; ++ks)
                  mma_ss_elect(tmem + C::col_s(b), (static_cast<uint64_t>(dhi) << 32) | (qlo + ks * 2),
                         (static_cast<uint64_t>(dhi) << 32) | (blo + ks * 2), C::kIdescS, ks > 0 ? 1u : 0u);
              }
              mma_commit_elect(bar_s_full(b));  // an empty product commits no MMA of its own
            }
            if (!ok) break;
            mma_commit_elect(bar_free(slot));  // K_j has been read by both tiles' products
          }
          if (!ok) break;
          mma_commit_elect(bar_q_free);
          ++kq;
        } else {
          const uint32_t vlo = (sRing >> 4) | (static_cast<uint32_t>(C::kTileBytes >> 4) << 16);
          for (int j = 0; ok && j < it.nmax; ++j, e += 2) {
            const int slot = e % C::kSlots;
            if (!(ok = __all_sync(0xffffffffu, mbar_wait(bar_full(slot), (e / C::kSlots) & 1, wc, 7)))) break;
#pragma unroll
            for (int t = 0; t < 2; ++t) {
              const int q = qn + 2 * j + t;
              const int b = q % kPairSBufs;
              if (!(ok = __all_sync(0xffffffffu, mbar_wait_poll(bar_p_full(b), (q / kPairSBufs) & 1, wc, 6)))) break;
              if (j >= it.nblk[t]) {  // an empty product
                mma_commit_elect(bar_pv_done(b));
                continue;
              }
              tc_fence_after();
              // o~_t (+)= P V_j: A = P from tensor memory, B = V_j MN-major.  The first
              // product of a pair overwrites o~_t; the softmax warps read the previous
              // pair's o~_t out before they hand over this pair's first P of tile t.
              const uint32_t blo = vlo + slot * (C::kTileBytes >> 4);
#pragma unroll
              for (int ks = 0; ks < kBN / 16; ++ks)
                mma_ts_elect(tmem + C::col_o(t), tmem + C::col_s(b) + ks * 8,
                       (static_cast<uint64_t>(dhi) << 32) | (blo + ks * (16 * 128 >> 4)), C::kIdescO,
                       (j > 0 || ks > 0) ? 1u : 0u);
              mma_commit_elect(bar_pv_done(b));
              if (j + 1 == it.nblk[t]) mma_commit_elect(bar_o_done(t));  // o~_t is complete
            }
            if (!ok) break;
            mma_commit_elect(bar_free(slot));  // V_j has been read by both tiles' products
          }
        }
        qn += 2 * it.nmax;
      }
      // every MMA this thread issued must finish before tensor memory is released
      const int di = warp == kPairWarpS ? 0 : 1;
      mma_commit_elect(bar_drain(di));
      mbar_wait_drain(bar_drain(di), 0, p.timeout_ns);
    }
  } else if (warp > kPairWarpPv) {
    setmaxnreg_dec<kPairRegsOther>();  // the warp without a role completes its warpgroup
  } else {
    // ================================================================ softmax / epilogue
    setmaxnreg_inc<kPairRegsSoftmax>();
    const int t = warp >> 2;          // the tile these warps serve
    const int r = threadIdx.x & 127;  // row within the tile = tensor-memory lane
    const uint32_t tl = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);
    const uint32_t colO = C::col_o(t);
    const float c = p.c;
    int qn = 0;  // products of the pairs before this one
    int nd = 0;  // pairs so far in which this tile had blocks: phase of o_done[t]
    bool ok = true;
    for (int ri = 0; ok; ++ri) {
      const int item = item_of(ri, cta, G);
      if (item >= p.num_items) break;
      const PairItem it = decode_pair<kPacked>(p, item, seq_perm);
      const int qbase = qn;
      qn += 2 * it.nmax;
      // this tile's fields, chosen by value (an array indexed by t would go to local memory)
      const int t_q0 = t ? it.q0[1] : it.q0[0];
      const int t_min_limit = t ? it.min_limit[1] : it.min_limit[0];
      const int nblk = t ? it.nblk[1] : it.nblk[0];
      const bool t_valid = t ? it.valid[1] : it.valid[0];
      const int row = t_q0 + r;
      const int limit = row_key_limit(row, it.kv_len, it.Nq, it.Nk, p.causal);
      float m = -INFINITY;  // running max, log2 domain
      float l = 0.f;        // running denominator
      // Checking a barrier costs a long round trip even when its phase completed long ago,
      // so the checks are issued early as non-blocking tests (as in attn_fwd_kernel): s_full
      // of the tile's next product and pv_done of its previous product, before the last
      // chunk of this block's exponentials.  Only a "not yet" leads to the (bounded) wait.
      bool s_seen = false;
      for (int j = 0; j < it.nmax; ++j) {
        const int q = qbase + 2 * j + t;
        const int b = q % kPairSBufs;
        const uint32_t colS = C::col_s(b);
        // every lane of the warp takes the same branch: the tcgen05 loads below are warp-wide
        if (!__all_sync(0xffffffffu, s_seen))
          ok = __all_sync(0xffffffffu, mbar_wait(bar_s_full(b), (q / kPairSBufs) & 1, wc, 9));
        if (!ok) break;
        if (j >= nblk) {  // an empty product: the tile lacks this block; only the barriers move
          s_seen = false;
          __syncwarp();
          if (lane == 0) mbar_arrive(bar_p_full(b));
          continue;
        }
        tc_fence_after();
        uint32_t sr[kBN];
#pragma unroll
        for (int x = 0; x < kBN / 32; ++x) tmem_ld32(tl + colS + x * 32, sr + x * 32);
        tmem_wait_ld();
        float s[kBN];
#pragma unroll
        for (int x = 0; x < kBN; ++x) s[x] = __uint_as_float(sr[x]);
        const int kb = j * kBN;
        if (kb + kBN > t_min_limit) {
#pragma unroll
          for (int x = 0; x < kBN; ++x)
            if (kb + x >= limit) s[x] = -INFINITY;
        }
        // block max: eight independent chains of 3-input max
        float a[8];
#pragma unroll
        for (int c8 = 0; c8 < 8; ++c8) a[c8] = fmaxf(s[2 * c8], s[2 * c8 + 1]);
#pragma unroll
        for (int x = 16; x < kBN; x += 16) {
#pragma unroll
          for (int c8 = 0; c8 < 8; ++c8) a[c8] = fmax3(a[c8], s[x + 2 * c8], s[x + 2 * c8 + 1]);
        }
        const float mx = fmaxf(fmaxf(fmax3(a[0], a[1], a[2]), fmax3(a[3], a[4], a[5])), fmaxf(a[6], a[7]));
        // the reference moves when the block max passes it by more than tau (tau = 0:
        // whenever the max rises); a row that has seen no visible key stays at -inf
        const float mb = mx * c;
        const float m_new = (mb > m + p.tau) ? mb : m;
        const float m_ref = (m_new == -INFINITY) ? 0.f : m_new;
        const float alpha = ex2_approx(m - m_ref);
        // p = exp2(c*s - m_ref), summed in fp32, packed to bf16 and stored 32 keys at a time
        const float2 c2 = make_float2(c, c);
        const float2 nm2 = make_float2(-m_ref, -m_ref);
        float2 acc0 = make_float2(0.f, 0.f), acc1 = make_float2(0.f, 0.f);
        const int qp = q - 2;  // the tile's previous product (j > 0)
        const int qx = q + 2;  // and its next (j + 1 < nmax)
        bool pv_seen = false;
        auto exp_block = [&](auto soft_tag) {
          constexpr bool kSoft = decltype(soft_tag)::value;
#pragma unroll
          for (int x4 = 0; x4 < kBN / 32; ++x4) {
            if (x4 == kBN / 32 - 1)
              s_seen = j + 1 < it.nmax && mbar_test_wait(bar_s_full(qx % kPairSBufs), (qx / kPairSBufs) & 1);
            if (x4 == 3)
              pv_seen = j > 0 && mbar_test_wait(bar_pv_done(qp % kPairSBufs), (qp / kPairSBufs) & 1);
            uint32_t pk[16];
#pragma unroll
            for (int x = 0; x < 16; ++x) {
              float2 v = __ffma2_rn(make_float2(s[x4 * 32 + 2 * x], s[x4 * 32 + 2 * x + 1]), c2, nm2);
              if (kSoft && (x * kSoftPairs) % 16 < kSoftPairs) {
                v = exp2_poly2(v);
              } else {
                v.x = ex2_approx(v.x);
                v.y = ex2_approx(v.y);
              }
              if (x & 1)
                acc1 = __fadd2_rn(acc1, v);
              else
                acc0 = __fadd2_rn(acc0, v);
              pk[x] = pack_bf16x2(v.x, v.y);
            }
            tmem_st16(tl + colS + x4 * 16, pk);
          }
        };
        // blocks with a masked key (-inf scores) keep every exponential on ex2.approx
        if (kSoftPairs > 0 && kb + kBN <= t_min_limit)
          exp_block(std::true_type{});
        else
          exp_block(std::false_type{});
        const float2 acc = __fadd2_rn(acc0, acc1);
        l = l * alpha + (acc.x + acc.y);
        m = m_new;
        if (j > 0 && !__all_sync(0xffffffffu, alpha == 1.f)) {
          // o~_t may be touched only after the tile's previous P V product has landed in it
          if (!__all_sync(0xffffffffu, pv_seen))
            ok = __all_sync(0xffffffffu, mbar_wait(bar_pv_done(qp % kPairSBufs), (qp / kPairSBufs) & 1, wc, 10));
          if (!ok) break;
          tc_fence_after();
          const float2 al2 = make_float2(alpha, alpha);
          uint32_t o[64];
          tmem_ld32(tl + colO, o);
          tmem_ld32(tl + colO + 32, o + 32);
          tmem_wait_ld();
#pragma unroll
          for (int x = 0; x < 32; ++x) {
            float2 v = __fmul2_rn(make_float2(__uint_as_float(o[2 * x]), __uint_as_float(o[2 * x + 1])), al2);
            o[2 * x] = __float_as_uint(v.x);
            o[2 * x + 1] = __float_as_uint(v.y);
          }
          tmem_st32(tl + colO, o);
          tmem_st32(tl + colO + 32, o + 32);
        }
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_p_full(b));
      }
      if (!t_valid) continue;  // a tile past the end of its sequence: no rows
      // ---- epilogue: one division by l; O and LSE out, straight from registers
      if (ok && nblk > 0) {
        // the tile's last P V product has landed in o~_t
        ok = __all_sync(0xffffffffu, mbar_wait(bar_o_done(t), nd & 1, wc, 11));
        ++nd;
        tc_fence_after();
      }
      if (!ok) break;
      const bool store = row < it.Nq;
      const float inv = l > 0.f ? 1.f / l : 0.f;
      uint4* dst = reinterpret_cast<uint4*>(p.o + it.b * p.os_b + it.hh * p.os_h +
                                            (it.q_base + (store ? row : 0)) * p.os_r);
#pragma unroll
      for (int x4 = 0; x4 < C::D / 32; ++x4) {
        uint32_t o[32];
        if (nblk > 0) {  // warp-wide load: every lane takes part, tail rows then skip the store
          tmem_ld32(tl + colO + x4 * 32, o);
          tmem_wait_ld();
        } else {
#pragma unroll
          for (int x = 0; x < 32; ++x) o[x] = 0u;
        }
        if (store) {
#pragma unroll
          for (int ch = 0; ch < 4; ++ch) {
            uint4 v;
            v.x = pack_bf16x2(__uint_as_float(o[ch * 8 + 0]) * inv, __uint_as_float(o[ch * 8 + 1]) * inv);
            v.y = pack_bf16x2(__uint_as_float(o[ch * 8 + 2]) * inv, __uint_as_float(o[ch * 8 + 3]) * inv);
            v.z = pack_bf16x2(__uint_as_float(o[ch * 8 + 4]) * inv, __uint_as_float(o[ch * 8 + 5]) * inv);
            v.w = pack_bf16x2(__uint_as_float(o[ch * 8 + 6]) * inv, __uint_as_float(o[ch * 8 + 7]) * inv);
            dst[x4 * 4 + ch] = v;
          }
        }
      }
      if (store) {
        const float lse = l > 0.f ? (m + __log2f(l)) * 0.69314718055994531f : -INFINITY;
        // [B, H, Nq], or [H, total_q] for packed sequences
        const size_t li = p.cu_q ? static_cast<size_t>(it.hh) * p.total_q + it.q_base + row
                                 : static_cast<size_t>(it.bh) * p.Nq + row;
        p.lse[li] = lse;
      }
      // o~_t has been read out (tcgen05 loads waited above): the next pair's first P V
      // product of this tile, ordered after this warp's next arrival on p_full, may
      // overwrite it
      tc_fence_before();
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kPairWarpPv) {
    tc_fence_after();
    // the base re-read from shared memory: keeping `tmem` live through every role's code
    // to here cost a spill (and so local memory) in the register-limited roles
    tmem_dealloc<kTmemCols>(*reinterpret_cast<volatile uint32_t*>(tmem_slot));
  }
}

}  // namespace attn
