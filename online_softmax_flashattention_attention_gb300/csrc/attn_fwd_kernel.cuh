// Fused attention forward with the online-softmax recurrence, sm_103a.
//
// A CTA computes tiles of 128 query rows of one (batch, head) at a time (persistently:
// one CTA per SM walks its tiles, see attn_fwd_kernel below).  Warp roles:
//   warps 0-3  softmax: thread r owns query row r of the tile (tensor-memory lane r).
//              Per key block it reads the score row S from tensor memory, masks, takes
//              the block max, computes alpha and p = exp2(c*s - m), updates l, writes P
//              (bf16) back into tensor memory over its own S and rescales the output
//              accumulator o~ by alpha when some row of its warp saw the max rise.  At the
//              end it divides o~ by l once and writes O and LSE.
//   warp 4     producer: TMA loads of the Q tile and of K/V blocks into a ring of
//              shared-memory stages guarded by full/free mbarriers.
//   warp 5     P V issuer: tcgen05.mma o~ += P_j V_j (P from tensor memory, V from shared
//              memory) as soon as the softmax warps have written P_j.
//   warp 6     S issuer: tcgen05.mma S_j = Q K_j^T (both operands in shared memory) into
//              score buffer j % 3, as soon as the buffer is free (P_{j-3} V done) and K_j
//              has landed.
// Three score buffers let the tensor core compute the next scores while the softmax
// warps work on S_j.  The two kinds of product come from two issuing warps: issuing a
// tcgen05.mma blocks while the tensor core is busy, and each issuer spends most of its
// time waiting on a barrier; with one issuer every such wait left the tensor core idle.
// One tile per CTA keeps a single busy softmax warp per scheduler partition (measured
// on GB300, a lightly loaded warp next to two busy warps gets its instructions issued
// only every 8-14 cycles).
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
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <type_traits>

#include "exp2_poly.cuh"
#include "ptx.cuh"

namespace attn {

constexpr int kBM = 128;           // query rows per tile (= tensor-memory lanes)
constexpr int kBN = 128;           // keys per block (kBNWide, kBNNarrow: d = 128 options of attn_fwd_ex)
constexpr int kBNWide = 192;
constexpr int kBNNarrow = 64;
constexpr int kWarpTma = 4;
constexpr int kWarpPv = 5;
constexpr int kWarpS = 6;
constexpr int kThreads = 224;      // 4 softmax warps + producer + two MMA issuers
constexpr uint32_t kTmemCols = 512;

struct FwdParams {
  int BH, H, Nq, Nk;
  int num_qtiles;          // ceil(Nq / 128)
  int causal;
  int rank_major;          // item order: 1 = tile rank major, 0 = head major (see decode)
  int order_div;           // B H when rank major, else the tiles (two-tile kernel: pairs) per head
  float c;                 // scale * log2(e)
  const int32_t* lens;     // per-batch key lengths or null
  float* lse;              // [BH, Nq]
  uint32_t* status;        // device status word (bit 0: a wait ran out)
  unsigned long long timeout_ns;
  int fault_block;         // test hook: the K block the producer never loads (-1: none)
  float tau;               // rescale threshold, log2 units: 0 = rescale whenever the max rises
  // Layout.  Every tensor map is 4-D, (d, rows, heads, batches), over any strides.  Packed
  // sequences (cu_q != null): sequence b is rows cu_q[b] .. cu_q[b+1] of Q / O and
  // cu_k[b] .. cu_k[b+1] of K / V in maps with one batch; Nq and Nk are then per sequence.
  const int32_t* cu_q;     // [B + 1] or null
  const int32_t* cu_k;     // [B + 1] or null
  int total_q, total_k;    // packed rows (the clamp for cu_q / cu_k)
  // O is stored straight from registers: element (b, h, row, x) at
  // o + b * os_b + h * os_h + row * os_r + x (packed sequences: row counted from cu_q[0])
  __nv_bfloat16* o;
  long long os_b, os_h, os_r;
  int num_items;           // work items: query tiles x splits
  // partial-state mode only: CTA (unit, split) absorbs key blocks [split * split_blocks,
  // (split + 1) * split_blocks) and writes the state (m, l, o~) instead of O and LSE
  int num_splits;          // >= 1
  int split_blocks;        // key blocks per split, >= 1
  int seq_sort;            // packed sequences: take them in decreasing work (rank_sequences)
  int o_v8;                // every O row starts on a 32-byte boundary: 32-byte stores
  float* st_o;             // [num_splits, BH, Nq, D] fp32 o~ (unnormalised)
  float* st_m;             // [num_splits, BH, Nq] running max of the scaled scores (natural log units)
  float* st_l;             // [num_splits, BH, Nq] running denominator
  // The one-tile kernel's decode divides by num_splits, order_div and H as
  // n / d = (umulhi(m, n) + n) >> s for 0 <= n < 2^31 (multiplier and shift set on the host
  // by set_divisors): measured on GB300, 1.02-1.05x on the short-tile workloads against
  // integer division, the same on long tiles.  (The two-tile kernel keeps the division: the
  // same change measured 0.955x there.)
  uint32_t dm_split, ds_split, dm_order, ds_order, dm_h, ds_h;
};

__device__ __forceinline__ int fast_div(int n, uint32_t m, uint32_t s) {
  const uint32_t u = static_cast<uint32_t>(n);
  return static_cast<int>((__umulhi(m, u) + u) >> s);
}

// Packed sequences are ranked by work for the item order when there are at most this many
// (a uint16 each in shared memory); more are taken in the order of cu_seqlens.
constexpr int kMaxSortedSeqs = 512;

// BN: keys per block.  128 everywhere by default.  At d = 128 a forward with O out can take
// 192- or 64-key blocks instead (attn_fwd_ex, key_block).  With 192, tensor memory holds two
// score buffers of 192 columns and o~ (512 columns), shared memory Q and two K/V stages of
// 48 KB; with 64, three score buffers of 64 columns and o~ (320 columns), Q and four K/V
// stages of 16 KB.  Both are measured slower on GB300: 192 because two score buffers leave
// the softmax warps waiting for scores, 64 because every block's hand-offs and rescale now
// cover half the keys.  They stay as options because they are the same recurrence over other
// blocks, which the tests compare with the 128-key build.
template <int D, int BN = kBN>
struct FwdCfg {
  static constexpr int kBNc = BN;
  static constexpr int kSub = D / 64;                   // 64-column swizzle sub-tiles per row tile
  static constexpr int kSubBytesQ = kBM * 128;          // 128 rows x 64 bf16 = 16 KiB
  static constexpr int kSubBytesKV = BN * 128;          // BN rows x 64 bf16
  static constexpr int kQBytes = kSub * kSubBytesQ;     // 128 rows x D bf16
  static constexpr int kKVBytes = kSub * kSubBytesKV;   // BN rows x D bf16
  // K/V ring depth.  At d = 128 with 128-key blocks, three stages each are all that fit beside
  // Q; measured on GB300, two stages each are 11-18 % slower, and two K with four V stages
  // run the same as three and three.
  static constexpr int kStages = BN > kBN ? 2 : (BN < kBN || D == 64) ? 4 : 3;
  static constexpr int kSBufs = BN > kBN ? 2 : 3;       // tensor-memory score buffers
  // How a tile's O leaves (measured on GB300): at d = 64 it is staged in the V stage of the
  // tile's last block and stored by TMA (a 16 KB tile in a 4-deep ring); at d = 128 the
  // stage would take a third of the ring while the store reads it, so each thread stores
  // its row straight from registers.
  static constexpr bool kStageO = (D == 64);
  static_assert(!kStageO || BN == kBM, "O is staged in a V stage of the tile's own size");
  static constexpr int kOffQ = 0;
  static constexpr int kOffK = kQBytes;
  static constexpr int kOffV = kOffK + kStages * kKVBytes;
  static constexpr int kOffBar = kOffV + kStages * kKVBytes;
  // barriers: q_full, q_free, (one unused slot), k_full[S], v_full[S], k_free[S],
  // v_free[S], s_full[B], pv_done[B], p_full[B], drain[2]
  static constexpr int kNumBars = 3 + 4 * kStages + 3 * kSBufs + 2;
  static constexpr int kOffMisc = kOffBar + 8 * kNumBars;  // tmem base, abort flag
  static constexpr int kOffPerm = kOffMisc + 16;           // uint16 order of packed sequences
  static constexpr int kSmemBytes = kOffPerm + 2 * kMaxSortedSeqs;
  static constexpr int kSmemAlloc = kSmemBytes + 1024;     // slack to align the base to 1024 B
  static constexpr int kSmemAllocNoPerm = kOffPerm + 1024; // launches without seq_sort
  static_assert(kSmemAlloc <= 232448, "shared memory per CTA");
  static_assert(kQBytes >= 4 * kMaxSortedSeqs, "the Q tile holds rank_sequences' scratch");
  // tensor-memory columns: S buffers b (P aliases the first BN / 2 columns), then o~
  __host__ __device__ static constexpr uint32_t col_s(int b) { return static_cast<uint32_t>(BN) * b; }
  static constexpr uint32_t kColO = static_cast<uint32_t>(BN) * kSBufs;
  static constexpr uint32_t kIdescS = idesc_bf16_f32(kBM, BN, 0);
  static constexpr uint32_t kIdescO = idesc_bf16_f32(kBM, D, 1);
  static_assert(kColO + D <= kTmemCols, "tensor memory");
};

// Visible keys of a row are exactly j < limit(row): both the key padding and the
// bottom-right causal bound are upper bounds on the key index.
__device__ __forceinline__ int row_key_limit(int row, int kv_len, int Nq, int Nk, int causal) {
  if (!causal) return kv_len;
  const long long lim = static_cast<long long>(row) + Nk - Nq + 1;
  return lim < kv_len ? static_cast<int>(lim < 0 ? 0 : lim) : kv_len;
}

// 2^x for two values on the FMA and ALU pipes instead of the MUFU unit.  Range reduction
// after Cody and Waite: j = rint(x) by adding and subtracting 1.5 * 2^23, f = x - j in
// [-1/2, 1/2], 2^f by the degree-4 polynomial of exp2_poly.cuh (relative error
// kExp2PolyMaxRelError), then j added to the exponent field.  Arguments below -125 are
// clamped to -125, so j >= -125 and the exponent field stays >= 1 (2^f >= 2^-1/2 has a
// field of 126): no wrap into the sign bit.  A clamped value is at most 2^-124.5, which
// is negligible next to l >= 1.  -inf is clamped too, so masked scores must not come here.
__device__ __forceinline__ float2 exp2_poly2(float2 x) {
  x.x = fmaxf(x.x, -125.f);
  x.y = fmaxf(x.y, -125.f);
  const float2 shifter = make_float2(12582912.f, 12582912.f);
  const float2 t = __fadd2_rn(x, shifter);                            // 1.5 * 2^23 + rint(x)
  const float2 nj = __ffma2_rn(t, make_float2(-1.f, -1.f), shifter);  // -rint(x), exact
  const float2 f = __fadd2_rn(x, nj);
  float2 r = __ffma2_rn(make_float2(kExp2C4, kExp2C4), f, make_float2(kExp2C3, kExp2C3));
  r = __ffma2_rn(r, f, make_float2(kExp2C2, kExp2C2));
  r = __ffma2_rn(r, f, make_float2(kExp2C1, kExp2C1));
  r = __ffma2_rn(r, f, make_float2(kExp2C0, kExp2C0));
  // the low bits of t hold rint(x) in two's complement: shifted into the exponent field
  r.x = __uint_as_float(__float_as_uint(r.x) + (__float_as_uint(t.x) << 23));
  r.y = __uint_as_float(__float_as_uint(r.y) + (__float_as_uint(t.y) << 23));
  return r;
}

__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

// One work item = one 128-row query tile of one (batch, head), or, in partial-state
// mode, one key split of such a tile.  decode() turns an item index into everything the
// roles need about it; every role of the CTA decodes the same items in the same order.
struct Item {
  int bh, b, hh;           // (batch, head)
  int q0;                  // first query row of the tile within its sequence
  int q_base, k_base;      // first rows of the sequence in the Q / K maps
  int Nq, Nk, bcoord;      // the sequence's lengths and its batch coordinate in the maps
  int kv_len;              // visible keys after padding
  int min_limit;           // smallest key limit of the tile's rows
  int split, jb0, nblk;    // key blocks jb0 .. jb0 + nblk - 1 (nblk = 0: nothing to compute)
  bool valid;              // false: a tile past the end of a shorter packed sequence
};

// Packed sequences: perm[r] = the sequence of rank r in decreasing work Lq * Lk (ties by
// index), so that the items' snake takes the longest sequences first and the CTAs' work
// evens out (measured on GB300 with 16 prompts of 512..8192 tokens: 1.13x against the
// order of cu_seqlens).  CTA-wide, after the previous kernel's writes are visible; the
// lengths are clamped as in decode, and the strict order makes perm a permutation
// whatever cu_seqlens holds.  scratch: B floats of shared memory that no copy uses yet.
__device__ __noinline__ void rank_sequences(const FwdParams& p, int B, float* scratch, uint16_t* perm) {
  for (int b = threadIdx.x; b < B; b += blockDim.x) {
    const int qs = min(max(__ldg(p.cu_q + b), 0), p.total_q);
    const int qe = min(max(__ldg(p.cu_q + b + 1), qs), p.total_q);
    const int ks = min(max(__ldg(p.cu_k + b), 0), p.total_k);
    const int ke = min(max(__ldg(p.cu_k + b + 1), ks), p.total_k);
    scratch[b] = static_cast<float>(qe - qs) * static_cast<float>(ke - ks);
  }
  __syncthreads();
  for (int b = threadIdx.x; b < B; b += blockDim.x) {
    const float w = scratch[b];
    int r = 0;
    for (int o = 0; o < B; ++o) {
      const float wo = scratch[o];
      r += (wo > w || (wo == w && o < b)) ? 1 : 0;
    }
    perm[r] = static_cast<uint16_t>(b);
  }
  fence_proxy_async_smem();  // the scratch's accesses before the TMA copies that overwrite it
  __syncthreads();
}

// kPacked: a launch over packed sequences (cu_q set), which may take them in the order of
// seq_perm; the other launches' code has no such step.
template <bool kPacked, int BN>
__device__ __forceinline__ Item decode(const FwdParams& p, int item, const uint16_t* seq_perm) {
  Item it;
  const int nqt = p.num_qtiles;
  const int unit = fast_div(item, p.dm_split, p.ds_split);
  it.split = item - unit * p.num_splits;
  // Head major: heads in order (their K/V stay in L2 while their tiles run).  Rank major:
  // tile rank r of every head, then rank r + 1; the host picks it for causal problems
  // whose K/V all fit in L2, where the snake of item_of over every head's longest tiles
  // first evens out the CTAs' work.  Either way a head's causal tiles go longest first.
  const int ua = fast_div(unit, p.dm_order, p.ds_order);
  const int ub = unit - ua * p.order_div;
  it.bh = p.rank_major ? ub : ua;
  int qtile = p.rank_major ? ua : ub;
  if (p.causal) qtile = nqt - 1 - qtile;
  it.b = fast_div(it.bh, p.dm_h, p.ds_h);
  it.hh = it.bh - it.b * p.H;
  it.q0 = qtile * kBM;
  it.q_base = 0;
  it.k_base = 0;
  it.Nq = p.Nq;
  it.Nk = p.Nk;
  it.bcoord = it.b;
  it.valid = true;
  if (p.cu_q) {
    if constexpr (kPacked) {
      if (p.seq_sort) {  // the unit's sequence is the one of its rank in decreasing work
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
    it.valid = it.q0 < it.Nq;
  }
  it.kv_len = it.Nk;
  if (p.lens) {
    const int L = __ldg(p.lens + it.b);
    it.kv_len = L < 0 ? 0 : (L > it.Nk ? it.Nk : L);
  }
  const int qlast = min(it.q0 + kBM - 1, it.Nq - 1);
  const int max_limit = row_key_limit(qlast, it.kv_len, it.Nq, it.Nk, p.causal);
  it.min_limit = row_key_limit(it.q0, it.kv_len, it.Nq, it.Nk, p.causal);
  const int nvis = max_limit > 0 ? (max_limit + BN - 1) / BN : 0;  // key blocks any row of the tile sees
  // without splits an item takes every visible block (its key count may be per sequence)
  it.jb0 = it.split * p.split_blocks;
  const int nsplit = p.num_splits > 1 ? max(0, min(nvis, it.jb0 + p.split_blocks) - it.jb0) : nvis;
  it.nblk = it.valid ? nsplit : 0;
  return it;
}

// The items of CTA c, in order: round r takes items r G .. r G + G - 1 (G = number of
// CTAs), forward in even rounds and backward in odd ones, so the long causal tiles at the
// front of each head spread evenly over the CTAs.
__device__ __forceinline__ int item_of(int r, int c, int G) { return r * G + ((r & 1) ? G - 1 - c : c); }

// kSoftPairs: of every 16 pairs of scores in a block with no masked key, this many take
// their exponential from exp2_poly2 instead of ex2.approx, to relieve the MUFU unit.
//
// The kernel is persistent: one CTA per SM walks its items.  The K/V ring, the score
// buffers and their barriers run on without a break from one item to the next, so the
// next tile's Q and first K/V blocks load and its first S product runs while the softmax
// warps finish the previous tile.  Q is reused under q_free (the last S product of a tile
// has read it); o~ is read out before the next tile's first P is handed over.  At d = 64 a
// tile's O is staged (swizzled) in the shared-memory V stage of its last key block, whose
// P V product has finished, and leaves by one TMA store; the softmax warps then hand that
// stage back to the producer (v_free) instead of the P V issuer.  At d = 128 each thread
// stores its row of O straight from registers.
template <int D, bool kStates, int kSoftPairs, bool kPacked, int BN = kBN>
__global__ void __launch_bounds__(kThreads, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmO,
                    const FwdParams p) {
  using C = FwdCfg<D, BN>;
  constexpr int kBN = BN;           // keys per block of this instantiation
  constexpr int kSBufs = C::kSBufs;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t sQ = sbase + C::kOffQ;
  const uint32_t sK = sbase + C::kOffK;
  const uint32_t sV = sbase + C::kOffV;
  const uint32_t bar0 = sbase + C::kOffBar;
  const uint32_t bar_q_full = bar0;
  const uint32_t bar_q_free = bar0 + 8u;   // the last S product of a tile has read Q
  auto bar_k_full = [&](int s) { return bar0 + 8u * (3 + s); };
  auto bar_v_full = [&](int s) { return bar0 + 8u * (3 + C::kStages + s); };
  auto bar_k_free = [&](int s) { return bar0 + 8u * (3 + 2 * C::kStages + s); };
  auto bar_v_free = [&](int s) { return bar0 + 8u * (3 + 3 * C::kStages + s); };
  auto bar_s_full = [&](int b) { return bar0 + 8u * (3 + 4 * C::kStages + b); };
  // pv_done[b] completes once per P_g V with g % 3 == b (it also frees score buffer b)
  auto bar_pv_done = [&](int b) { return bar0 + 8u * (3 + 4 * C::kStages + kSBufs + b); };
  // p_full[b]: the softmax warps have written P_g (and rescaled o~) for g % 3 == b
  auto bar_p_full = [&](int b) { return bar0 + 8u * (3 + 4 * C::kStages + 2 * kSBufs + b); };
  auto bar_drain = [&](int i) { return bar0 + 8u * (3 + 4 * C::kStages + 3 * kSBufs + i); };
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
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(bar_k_full(s), 1);
      mbar_init(bar_v_full(s), 1);
      mbar_init(bar_k_free(s), 1);
      mbar_init(bar_v_free(s), 1);
    }
    for (int i = 0; i < kSBufs; ++i) {
      mbar_init(bar_s_full(i), 1);
      mbar_init(bar_pv_done(i), 1);
      mbar_init(bar_p_full(i), 4);
    }
    mbar_init(bar_drain(0), 1);
    mbar_init(bar_drain(1), 1);
    *abort_flag = 0u;
    fence_mbar_init();
  }
  if (warp == kWarpPv) tmem_alloc<kTmemCols>(smem_u32(tmem_slot));
  if (warp == kWarpTma && lane == 0) {
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
    if (!kStates && C::kStageO) tma_prefetch_desc(&tmO);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // Everything above touched only shared and tensor memory and the kernel parameters; a
  // launch that overlaps the previous kernel's tail waits here for it to finish.
  griddep_wait();
  griddep_launch_dependents();
  uint16_t* seq_perm = reinterpret_cast<uint16_t*>(smem + C::kOffPerm);
  if constexpr (kPacked) {
    if (p.seq_sort) rank_sequences(p, p.BH / p.H, reinterpret_cast<float*>(smem + C::kOffQ), seq_perm);
  }

  if (warp == kWarpTma) {
    // ================================================================ producer
    if (lane == 0) {
      const uint64_t pol_kv = policy_evict_last();
      const uint64_t pol_q = policy_evict_first();
      int g = 0;   // key blocks loaded so far over all items: ring slot g % kStages
      int kq = 0;  // items with work so far: uses of the Q buffer
      // Stage st has a K (V) load in flight when bit st of k_live (v_live) is set; the bit of
      // k_par (v_par) is the phase parity that load completes.  Bit masks rather than arrays
      // indexed by the stage: a dynamically indexed array would live in local memory.
      uint32_t k_live = 0, k_par = 0, v_live = 0, v_par = 0;
      bool ok = true;
      for (int ri = 0; ok; ++ri) {
        const int item = item_of(ri, cta, G);
        if (item >= p.num_items) break;
        const Item it = decode<kPacked, kBN>(p, item, seq_perm);
        if (it.nblk == 0) continue;
        // the previous tile's Q must have been read by its last S product
        if (kq > 0 && !mbar_wait(bar_q_free, (kq - 1) & 1, wc, 13)) break;
        mbar_arrive_expect_tx(bar_q_full, C::kQBytes);
        for (int s = 0; s < C::kSub; ++s)
          tma_load_4d(sQ + s * C::kSubBytesQ, &tmQ, bar_q_full, s * 64, it.q_base + it.q0, it.hh, it.bcoord, pol_q);
        ++kq;
        for (int j = 0; j < it.nblk; ++j, ++g) {
          const int st = g % C::kStages;
          const uint32_t ph = (g / C::kStages) & 1;
          if (!mbar_wait(bar_k_free(st), ph ^ 1, wc, 1)) {
            ok = false;
            break;
          }
          const uint32_t bit = 1u << st;
          k_live &= ~bit;
          if (j != p.fault_block) {  // the test hook withholds one block: its k_full never completes
            mbar_arrive_expect_tx(bar_k_full(st), C::kKVBytes);
            for (int s = 0; s < C::kSub; ++s)
              tma_load_4d(sK + st * C::kKVBytes + s * C::kSubBytesKV, &tmK, bar_k_full(st), s * 64,
                          it.k_base + (it.jb0 + j) * kBN, it.hh, it.bcoord, pol_kv);
            k_live |= bit;
            k_par = (k_par & ~bit) | (ph << st);
          }
          if (!mbar_wait(bar_v_free(st), ph ^ 1, wc, 2)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(bar_v_full(st), C::kKVBytes);
          for (int s = 0; s < C::kSub; ++s)
            tma_load_4d(sV + st * C::kKVBytes + s * C::kSubBytesKV, &tmV, bar_v_full(st), s * 64,
                        it.k_base + (it.jb0 + j) * kBN, it.hh, it.bcoord, pol_kv);
          v_live |= bit;
          v_par = (v_par & ~bit) | (ph << st);
        }
      }
      // Let the copies still in flight land before this warp leaves (in a normal run they
      // were consumed long ago; after a failed wait nobody else will wait for them).
#pragma unroll
      for (int s = 0; s < C::kStages; ++s) {
        if ((k_live >> s) & 1u) mbar_wait_drain(bar_k_full(s), (k_par >> s) & 1u, p.timeout_ns);
        if ((v_live >> s) & 1u) mbar_wait_drain(bar_v_full(s), (v_par >> s) & 1u, p.timeout_ns);
      }
    }
  } else if (warp == kWarpPv || warp == kWarpS) {
    // ================================================================ MMA issuers
    if (lane == 0) {
      // Shared-memory descriptors: the high word (stride 1024 B, version 1, 128-byte
      // swizzle) is the same for every operand; the low word holds the start address
      // (>> 4) and the leading byte offset, so a k-step is one add to the low word.
      const uint32_t dhi = (1024u >> 4) | (1u << 14) | (2u << 29);
      int g = 0;   // key blocks over all items
      int kq = 0;  // items with work
      bool ok = true;
      if (warp == kWarpS) {
        const uint32_t qlo = (sQ >> 4) | (1u << 16);
        const uint32_t klo = (sK >> 4) | (1u << 16);
        for (int ri = 0; ok; ++ri) {
          const int item = item_of(ri, cta, G);
          if (item >= p.num_items) break;
          const Item it = decode<kPacked, kBN>(p, item, seq_perm);
          if (it.nblk == 0) continue;
          ok = mbar_wait(bar_q_full, kq & 1, wc, 3);
          for (int j = 0; ok && j < it.nblk; ++j, ++g) {
            const int st = g % C::kStages;
            const int bf = g % kSBufs;
            // buffer bf last held P_{g-3}: its P V product must have consumed it
            if (g >= kSBufs) ok = mbar_wait(bar_pv_done(bf), ((g - kSBufs) / kSBufs) & 1, wc, 4);
            ok = ok && mbar_wait(bar_k_full(st), (g / C::kStages) & 1, wc, 5);
            if (!ok) break;
            tc_fence_after();
            // S_g = Q K_g^T: 8 (d = 128) or 4 (d = 64) k-steps of 16
            const uint32_t blo = klo + st * (C::kKVBytes >> 4);
            const uint32_t dst = tmem + C::col_s(bf);
#pragma unroll
            for (int ks = 0; ks < D / 16; ++ks) {
              // k-step ks: 16 columns of d, in sub-tile ks / 4 of the Q and of the K tile
              const uint32_t offq = (ks / 4) * (C::kSubBytesQ >> 4) + (ks % 4) * 2;
              const uint32_t offk = (ks / 4) * (C::kSubBytesKV >> 4) + (ks % 4) * 2;
              mma_ss(dst, (static_cast<uint64_t>(dhi) << 32) | (qlo + offq),
                     (static_cast<uint64_t>(dhi) << 32) | (blo + offk), C::kIdescS, ks > 0 ? 1u : 0u);
            }
            mma_commit(bar_s_full(bf));
            mma_commit(bar_k_free(st));
          }
          if (!ok) break;
          mma_commit(bar_q_free);  // Q may be overwritten once this tile's products have read it
          ++kq;
        }
      } else {
        const uint32_t vlo = (sV >> 4) | (static_cast<uint32_t>(C::kSubBytesKV >> 4) << 16);
        for (int ri = 0; ok; ++ri) {
          const int item = item_of(ri, cta, G);
          if (item >= p.num_items) break;
          const Item it = decode<kPacked, kBN>(p, item, seq_perm);
          if (it.nblk == 0) continue;
          // The first product of a tile overwrites o~.  The softmax warps read the previous
          // tile's o~ out before they write this tile's first P, and P_0 is awaited below,
          // so that ordering needs no barrier of its own.
          for (int j = 0; ok && j < it.nblk; ++j, ++g) {
            const int st = g % C::kStages;
            // V_g has normally landed long before P_g is ready: check it first
            ok = mbar_wait(bar_v_full(st), (g / C::kStages) & 1, wc, 7) &&
                 mbar_wait_poll(bar_p_full(g % kSBufs), (g / kSBufs) & 1, wc, 6);
            if (!ok) break;
            tc_fence_after();
            // o~ += P_g V_g: 8 k-steps of 16 keys; A = P_g from tensor memory, B = V_g MN-major
            const uint32_t blo = vlo + st * (C::kKVBytes >> 4);
            const uint32_t a = tmem + C::col_s(g % kSBufs);
#pragma unroll
            for (int ks = 0; ks < kBN / 16; ++ks)
              mma_ts(tmem + C::kColO, a + ks * 8,
                     (static_cast<uint64_t>(dhi) << 32) | (blo + ks * (16 * 128 >> 4)), C::kIdescO,
                     (j > 0 || ks > 0) ? 1u : 0u);
            mma_commit(bar_pv_done(g % kSBufs));
            // The V stage of a tile's last block is handed back by the softmax warps instead:
            // they stage the tile's O in it for the TMA store
            if (kStates || !C::kStageO || j + 1 < it.nblk) mma_commit(bar_v_free(st));
          }
          ++kq;
        }
      }
      // every MMA this thread issued must finish before tensor memory is released (in a
      // normal run they have: the softmax warps consumed them)
      mma_commit(bar_drain(warp == kWarpS));
      mbar_wait_drain(bar_drain(warp == kWarpS), 0, p.timeout_ns);
    }
  } else {
    // ================================================================ softmax / epilogue
    const int r = threadIdx.x;  // 0..127: row within the tile = tensor-memory lane
    const uint32_t tl = tmem + (static_cast<uint32_t>(warp * 32) << 16);
    const float c = p.c;
    int g = 0;  // key blocks over all items: score buffer g % 3
    bool ok = true;
    for (int ri = 0; ok; ++ri) {
      const int item = item_of(ri, cta, G);
      if (item >= p.num_items) break;
      const Item it = decode<kPacked, kBN>(p, item, seq_perm);
      if (!it.valid) continue;  // a tile past the end of a shorter packed sequence
      const int row = it.q0 + r;
      const int limit = row_key_limit(row, it.kv_len, it.Nq, it.Nk, p.causal);
      const int nblk = it.nblk;
      float m = -INFINITY;  // running max, log2 domain
      float l = 0.f;        // running denominator
      // Checking a barrier costs a long round trip even when its phase completed long ago.
      // The two checks of every block are therefore issued early, as non-blocking tests
      // whose results are consumed later: s_full of the next block and pv_done of the
      // previous block, both before the last chunk of this block's exponentials (measured:
      // testing s_full before the first chunk instead is about 1.5 % slower, the next
      // block's scores being ready less often).  Only when a test says "not yet" does the
      // thread take the (bounded) wait.
      bool s_seen = false;  // s_full of block j already seen complete
      for (int j = 0; j < nblk; ++j) {
        const int gj = g + j;  // this block's index over all items
        const uint32_t colS = C::col_s(gj % kSBufs);
        // every lane of the warp takes the same branch: the tcgen05 loads below are warp-wide
        if (!__all_sync(0xffffffffu, s_seen))
          ok = __all_sync(0xffffffffu, mbar_wait(bar_s_full(gj % kSBufs), (gj / kSBufs) & 1, wc, 9));
        if (!ok) break;
        tc_fence_after();
        uint32_t sr[kBN];
#pragma unroll
        for (int q = 0; q < kBN / 32; ++q) tmem_ld32(tl + colS + q * 32, sr + q * 32);
        tmem_wait_ld();
        float s[kBN];
#pragma unroll
        for (int k = 0; k < kBN; ++k) s[k] = __uint_as_float(sr[k]);
        const int kb = (it.jb0 + j) * kBN;
        if (kb + kBN > it.min_limit) {
#pragma unroll
          for (int k = 0; k < kBN; ++k)
            if (kb + k >= limit) s[k] = -INFINITY;
        }
        // block max: eight independent chains of 3-input max over s[0..kBN)
        float a[8];
#pragma unroll
        for (int c8 = 0; c8 < 8; ++c8) a[c8] = fmaxf(s[2 * c8], s[2 * c8 + 1]);
#pragma unroll
        for (int k = 16; k < kBN; k += 16) {
#pragma unroll
          for (int c8 = 0; c8 < 8; ++c8) a[c8] = fmax3(a[c8], s[k + 2 * c8], s[k + 2 * c8 + 1]);
        }
        const float mx = fmaxf(fmaxf(fmax3(a[0], a[1], a[2]), fmax3(a[3], a[4], a[5])), fmaxf(a[6], a[7]));
        // the reference moves when the block max passes it by more than tau (tau = 0:
        // whenever the max rises, the pages' rule; a row that has seen no visible key stays
        // at -inf)
        const float mb = mx * c;
        const float m_new = (mb > m + p.tau) ? mb : m;
        const float m_ref = (m_new == -INFINITY) ? 0.f : m_new;
        const float alpha = ex2_approx(m - m_ref);
        // p = exp2(c*s - m_ref), summed in fp32, packed to bf16 and stored 32 keys at a time
        const float2 c2 = make_float2(c, c);
        const float2 nm2 = make_float2(-m_ref, -m_ref);
        float2 acc0 = make_float2(0.f, 0.f), acc1 = make_float2(0.f, 0.f);
        bool pv_seen = false;  // pv_done of block j - 1 seen complete
        auto exp_block = [&](auto soft_tag) {
          constexpr bool kSoft = decltype(soft_tag)::value;
#pragma unroll
          for (int q = 0; q < kBN / 32; ++q) {
            if (q == kBN / 32 - 1)
              s_seen = j + 1 < nblk && mbar_test_wait(bar_s_full((gj + 1) % kSBufs), ((gj + 1) / kSBufs) & 1);
            if (q == kBN / 32 - 1)
              pv_seen = j > 0 && mbar_test_wait(bar_pv_done((gj - 1) % kSBufs), ((gj - 1) / kSBufs) & 1);
            uint32_t pk[16];
#pragma unroll
            for (int k = 0; k < 16; ++k) {
              float2 x = __ffma2_rn(make_float2(s[q * 32 + 2 * k], s[q * 32 + 2 * k + 1]), c2, nm2);
              if (kSoft && (k * kSoftPairs) % 16 < kSoftPairs) {
                x = exp2_poly2(x);
              } else {
                x.x = ex2_approx(x.x);
                x.y = ex2_approx(x.y);
              }
              if (k & 1)
                acc1 = __fadd2_rn(acc1, x);
              else
                acc0 = __fadd2_rn(acc0, x);
              pk[k] = pack_bf16x2(x.x, x.y);
            }
            tmem_st16(tl + colS + q * 16, pk);
          }
        };
        // blocks with a masked key (-inf scores) keep every exponential on ex2.approx
        if (kSoftPairs > 0 && kb + kBN <= it.min_limit)
          exp_block(std::true_type{});
        else
          exp_block(std::false_type{});
        const float2 acc = __fadd2_rn(acc0, acc1);
        l = l * alpha + (acc.x + acc.y);
        m = m_new;
        if (j > 0 && !__all_sync(0xffffffffu, alpha == 1.f)) {
          // o~ may be touched only after the previous P V product has landed in it
          if (!__all_sync(0xffffffffu, pv_seen))
            ok = __all_sync(0xffffffffu,
                            mbar_wait(bar_pv_done((gj - 1) % kSBufs), ((gj - 1) / kSBufs) & 1, wc, 10));
          if (!ok) break;
          tc_fence_after();
          const float2 al2 = make_float2(alpha, alpha);
#pragma unroll
          for (int q = 0; q < D / 64; ++q) {
            uint32_t o[64];
            tmem_ld32(tl + C::kColO + q * 64, o);
            tmem_ld32(tl + C::kColO + q * 64 + 32, o + 32);
            tmem_wait_ld();
#pragma unroll
            for (int k = 0; k < 32; ++k) {
              float2 v = __fmul2_rn(make_float2(__uint_as_float(o[2 * k]), __uint_as_float(o[2 * k + 1])), al2);
              o[2 * k] = __float_as_uint(v.x);
              o[2 * k + 1] = __float_as_uint(v.y);
            }
            tmem_st32(tl + C::kColO + q * 64, o);
            tmem_st32(tl + C::kColO + q * 64 + 32, o + 32);
          }
        }
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_p_full(gj % kSBufs));
      }
      // ---- epilogue: one division by l; O and LSE out
      const int gl = g + nblk - 1;  // the tile's last block
      if (ok && nblk > 0) {
        // the last P V (also the last MMA of the tile) has landed in o~
        ok = __all_sync(0xffffffffu, mbar_wait(bar_pv_done(gl % kSBufs), (gl / kSBufs) & 1, wc, 11));
        tc_fence_after();
      }
      g += nblk;
      const bool store = row < it.Nq;
      if (!kStates && C::kStageO && nblk > 0) {
        // O through the V stage of the last block and one TMA store.  Every softmax warp
        // reaches this barrier once per tile with blocks, also after a failed wait (it left
        // the block loop early), so they all agree on giving up and leave together.
        const bool give_up = bar_sync_or(1, 128, !ok || *abort_flag != 0u);
        if (give_up) {
          ok = false;
          break;
        }
        const int st_last = gl % C::kStages;
        const uint32_t stage = sV + st_last * C::kKVBytes;
        uint8_t* orow = smem + (stage - sbase) + r * 128;
        // the last tile of a packed sequence would overrun into the next sequence under a
        // TMA store: its rows are stored one by one instead (the same for the whole CTA)
        const bool direct = p.cu_q != nullptr && it.q0 + kBM > it.Nq;
        uint4* gdst = reinterpret_cast<uint4*>(p.o + it.b * p.os_b + it.hh * p.os_h +
                                               (it.q_base + (store ? row : 0)) * p.os_r);
        const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll
        for (int q = 0; q < D / 32; ++q) {
          uint32_t o[32];
          tmem_ld32(tl + C::kColO + q * 32, o);
          tmem_wait_ld();
#pragma unroll
          for (int ch = 0; ch < 4; ++ch) {
            uint4 v;
            v.x = pack_bf16x2(__uint_as_float(o[ch * 8 + 0]) * inv, __uint_as_float(o[ch * 8 + 1]) * inv);
            v.y = pack_bf16x2(__uint_as_float(o[ch * 8 + 2]) * inv, __uint_as_float(o[ch * 8 + 3]) * inv);
            v.z = pack_bf16x2(__uint_as_float(o[ch * 8 + 4]) * inv, __uint_as_float(o[ch * 8 + 5]) * inv);
            v.w = pack_bf16x2(__uint_as_float(o[ch * 8 + 6]) * inv, __uint_as_float(o[ch * 8 + 7]) * inv);
            if (direct) {
              if (store) gdst[q * 4 + ch] = v;
            } else {
              // columns 32q .. 32q + 31 = four 16-byte chunks of sub-tile q / 2, chunk
              // (q % 2) * 4 + ch, 128-byte swizzle
              const int chunk = (q % 2) * 4 + ch;
              *reinterpret_cast<uint4*>(orow + (q / 2) * C::kSubBytesKV + ((chunk ^ (r & 7)) * 16)) = v;
            }
          }
        }
        if (store) {
          const float lse = l > 0.f ? (m + __log2f(l)) * 0.69314718055994531f : -INFINITY;
          const size_t li = p.cu_q ? static_cast<size_t>(it.hh) * p.total_q + it.q_base + row
                                   : static_cast<size_t>(it.bh) * p.Nq + row;
          p.lse[li] = lse;
        }
        fence_proxy_async_smem();
        bar_sync_named(1, 128);
        if (r == 0) {
          if (!direct) {
            for (int s = 0; s < C::kSub; ++s)
              tma_store_4d(&tmO, stage + s * C::kSubBytesKV, s * 64, it.q_base + it.q0, it.hh, it.bcoord);
            tma_store_commit();
            tma_store_wait_read();  // the stage may be loaded again once the store has read it
          }
          mbar_arrive(bar_v_free(st_last));
        }
        // o~ has been read out (tcgen05 loads waited above): the next tile's first P V
        // product, ordered after this thread's next arrival on p_full, may overwrite it
        tc_fence_before();
        continue;
      }
      if (!ok) break;
      if constexpr (kStates) {
        // the state of this split, undivided: o~ and l as accumulated, m back in natural-log
        // units of the scaled scores (m2 = c * max q.k, c = scale * log2 e, so m = m2 * ln 2)
        const size_t ridx = (static_cast<size_t>(it.split) * p.BH + it.bh) * p.Nq + (store ? row : 0);
        float4* dst = reinterpret_cast<float4*>(p.st_o + ridx * D);
#pragma unroll
        for (int q = 0; q < D / 32; ++q) {
          uint32_t o[32];
          if (nblk > 0) {  // warp-wide load: every lane takes part, tail rows then skip the store
            tmem_ld32(tl + C::kColO + q * 32, o);
            tmem_wait_ld();
          } else {
#pragma unroll
            for (int k = 0; k < 32; ++k) o[k] = 0u;
          }
          if (store) {
#pragma unroll
            for (int k = 0; k < 8; ++k)
              dst[q * 8 + k] = make_float4(__uint_as_float(o[4 * k]), __uint_as_float(o[4 * k + 1]),
                                           __uint_as_float(o[4 * k + 2]), __uint_as_float(o[4 * k + 3]));
          }
        }
        if (store) {
          p.st_m[ridx] = m * 0.69314718055994531f;  // -inf stays -inf for a row that saw no key
          p.st_l[ridx] = l;
        }
      } else {  // straight from registers (d = 128, or a tile with no visible key)
        const float inv = l > 0.f ? 1.f / l : 0.f;
        uint32_t* dst = reinterpret_cast<uint32_t*>(p.o + it.b * p.os_b + it.hh * p.os_h +
                                                    (it.q_base + (store ? row : 0)) * p.os_r);
        // The whole row of o~ in one round trip (one wait for all the loads), packed to bf16
        // in place, then stored 32 bytes at a time where O's alignment allows it: a 16-byte
        // store fills only half of a 32-byte sector (measured on GB300 against four
        // load-wait rounds and 16-byte stores: 1.005-1.008x on causal d = 128 shapes).
        uint32_t o[D];
        if (nblk > 0) {  // warp-wide loads: every lane takes part, tail rows then skip the store
#pragma unroll
          for (int q = 0; q < D / 32; ++q) tmem_ld32(tl + C::kColO + q * 32, o + q * 32);
          tmem_wait_ld();
        } else {
#pragma unroll
          for (int k = 0; k < D; ++k) o[k] = 0u;
        }
#pragma unroll
        for (int k = 0; k < D / 2; ++k)
          o[k] = pack_bf16x2(__uint_as_float(o[2 * k]) * inv, __uint_as_float(o[2 * k + 1]) * inv);
        if (store) {
          if (p.o_v8) {
#pragma unroll
            for (int k = 0; k < D / 16; ++k) st_global_v8(dst + 8 * k, o + 8 * k);
          } else {
#pragma unroll
            for (int k = 0; k < D / 8; ++k)
              reinterpret_cast<uint4*>(dst)[k] = make_uint4(o[4 * k], o[4 * k + 1], o[4 * k + 2], o[4 * k + 3]);
          }
        }
        if (store) {
          const float lse = l > 0.f ? (m + __log2f(l)) * 0.69314718055994531f : -INFINITY;
          // [B, H, Nq], or [H, total_q] for packed sequences
          const size_t li = p.cu_q ? static_cast<size_t>(it.hh) * p.total_q + it.q_base + row
                                   : static_cast<size_t>(it.bh) * p.Nq + row;
          p.lse[li] = lse;
        }
      }
      // o~ has been read out (tcgen05 loads waited above): the next tile's first P V product,
      // ordered after this thread's next arrival on p_full, may overwrite it
      tc_fence_before();
    }
  }

  if (!kStates && C::kStageO && threadIdx.x == 0) tma_store_wait_all();  // the last O tile is out
  tc_fence_before();
  __syncthreads();
  if (warp == kWarpPv) {
    tc_fence_after();
    // the base re-read from shared memory: keeping `tmem` live through every role's code
    // to here can cost a spill (and so local memory) in the register-limited roles
    tmem_dealloc<kTmemCols>(*reinterpret_cast<volatile uint32_t*>(tmem_slot));
  }
}

}  // namespace attn
