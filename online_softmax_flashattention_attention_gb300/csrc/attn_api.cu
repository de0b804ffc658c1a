// Host side of the C ABI declared in include/attn.h: argument checks, TMA tensor maps,
// the launch, the device status word and the host-buffer entry point.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cmath>
#include <cstddef>
#include <cstdarg>
#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <algorithm>
#include <atomic>
#include <mutex>
#include <utility>

#include "../../include/attn.h"
#include "attn_fwd_kernel.cuh"
#include "attn_fwd_pair_kernel.cuh"
#include "attn_merge_kernel.cuh"

namespace {

constexpr int kMaxDevices = 64;
constexpr unsigned long long kDefaultTimeoutNs = 2000000000ull;  // 2 s per bounded wait

thread_local char g_err[512] = "";

attn_status fail(attn_status st, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof(g_err), fmt, ap);
  va_end(ap);
  return st;
}

std::mutex g_mu;
uint32_t* g_status[kMaxDevices] = {};
// Device address of the allocation-free entry point's status word, per device (null until
// that entry point's first call on the device).
uint32_t* g_noalloc_addr[kMaxDevices] = {};
int g_sms[kMaxDevices] = {};
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

struct Workspace {
  void* base = nullptr;
  size_t bytes = 0;
};
Workspace g_ws[kMaxDevices];

attn_status get_device(int* dev) {
  if (cudaGetDevice(dev) != cudaSuccess || *dev < 0 || *dev >= kMaxDevices)
    return fail(ATTN_ERR_NO_DEVICE, "no current CUDA device");
  return ATTN_OK;
}

attn_status setup(int dev, uint32_t** status) {
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_encode) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
    if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !fn)
      return fail(ATTN_ERR_NO_DEVICE, "cuTensorMapEncodeTiled unavailable: %s", cudaGetErrorString(e));
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  }
  if (!g_status[dev]) {
    cudaDeviceProp prop;
    if (cudaGetDeviceProperties(&prop, dev) != cudaSuccess)
      return fail(ATTN_ERR_NO_DEVICE, "cudaGetDeviceProperties failed");
    if (prop.major != 10 || prop.minor != 3)
      return fail(ATTN_ERR_NO_DEVICE, "device %d is sm_%d%d; this library is built for sm_103a", dev, prop.major,
                  prop.minor);
    uint32_t* s = nullptr;
    if (cudaMalloc(&s, sizeof(uint32_t)) != cudaSuccess) return fail(ATTN_ERR_NO_DEVICE, "status word alloc failed");
    if (cudaMemset(s, 0, sizeof(uint32_t)) != cudaSuccess) return fail(ATTN_ERR_NO_DEVICE, "status word init failed");
    g_status[dev] = s;
    g_sms[dev] = prop.multiProcessorCount;
  }
  *status = g_status[dev];
  return ATTN_OK;
}

// SM count of a device, cached (several host threads may fill the same slot: they
// write the same value).
std::atomic<int> g_sm_cache[kMaxDevices];
int sm_count(int dev) {
  int n = g_sm_cache[dev].load(std::memory_order_relaxed);
  if (n <= 0) {
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 1;
    g_sm_cache[dev].store(n, std::memory_order_relaxed);
  }
  return n;
}

// attn_fwd_host's copy streams and events, one set per device, created on first use.
constexpr int kHostEvents = 64;  // event slots, reused round robin (more than any chunk count)
struct HostPipe {
  cudaStream_t in = nullptr, out = nullptr;
  cudaEvent_t ev_start = nullptr, ev_end = nullptr;
  cudaEvent_t ev_in[kHostEvents] = {}, ev_done[kHostEvents] = {};
};
HostPipe* g_pipe[kMaxDevices] = {};

attn_status host_pipe(int dev, HostPipe** out) {
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_pipe[dev]) {
    HostPipe* hp = new HostPipe;
    cudaError_t e = cudaStreamCreateWithFlags(&hp->in, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&hp->out, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&hp->ev_start, cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&hp->ev_end, cudaEventDisableTiming);
    for (int i = 0; i < kHostEvents && e == cudaSuccess; ++i) {
      e = cudaEventCreateWithFlags(&hp->ev_in[i], cudaEventDisableTiming);
      if (e == cudaSuccess) e = cudaEventCreateWithFlags(&hp->ev_done[i], cudaEventDisableTiming);
    }
    if (e != cudaSuccess) return fail(ATTN_ERR_LAUNCH, "copy streams / events: %s", cudaGetErrorString(e));
    g_pipe[dev] = hp;
  }
  *out = g_pipe[dev];
  return ATTN_OK;
}

// How many chunks attn_fwd_host cuts a problem into: about one per 32 MB of input, at
// least one per batch, at most 16 (plus one per extra batch) -- enough to overlap the
// copies with the forward, few enough that every chunk's grid still fills the GPU.
int host_chunks(int B, int H, size_t in_bytes) {
  const long long want = static_cast<long long>(in_bytes / (32u << 20));
  long long n = std::max<long long>(1, std::min<long long>(16, want));
  n = std::min<long long>(n, static_cast<long long>(B) * H);
  return static_cast<int>(std::max<long long>(n, B));
}
int nch_per_batch(int nch, int B) { return std::max(1, nch / std::max(1, B)); }

// Where the four tensors live.  Each is seen through a 4-D map (d, rows, heads,
// batches) with element strides (batch, head, row); d is contiguous.  Packed sequences
// use one batch and the per-sequence row offsets cu_q / cu_k.
struct Geometry {
  long long qs[3], ks[3], vs[3], os[3];  // element strides: batch, head, row
  long long q_rows = 0, k_rows = 0;      // rows of the maps
  int map_b = 1;                         // batches of the maps
  int grid_q = 0;                        // query rows the grid covers (longest sequence)
  const int32_t* cu_q = nullptr;
  const int32_t* cu_k = nullptr;
};

Geometry dense_geometry(int B, int H, int Nq, int Nk, int d) {
  Geometry g;
  const long long qb = static_cast<long long>(H) * Nq * d, kb = static_cast<long long>(H) * Nk * d;
  const long long q[3] = {qb, static_cast<long long>(Nq) * d, d};
  const long long k[3] = {kb, static_cast<long long>(Nk) * d, d};
  for (int i = 0; i < 3; ++i) {
    g.qs[i] = g.os[i] = q[i];
    g.ks[i] = g.vs[i] = k[i];
  }
  g.q_rows = Nq;
  g.k_rows = Nk;
  g.map_b = B;
  g.grid_q = Nq;
  return g;
}

// 4-D map (d, rows, H, B) over bf16 with element strides (batch, head, row), box
// (64, 128, 1, 1), 128-byte swizzle; rows past `rows` read as zero and are not stored.
attn_status make_map(CUtensorMap* map, const void* ptr, int d, long long rows, int H, int B, const long long* st,
                     int box_rows = attn::kBM) {
  cuuint64_t dims[4] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(rows), static_cast<cuuint64_t>(H),
                        static_cast<cuuint64_t>(B)};
  cuuint64_t strides[3] = {static_cast<cuuint64_t>(st[2]) * 2, static_cast<cuuint64_t>(st[1]) * 2,
                           static_cast<cuuint64_t>(st[0]) * 2};
  cuuint32_t box[4] = {64, static_cast<cuuint32_t>(box_rows), 1, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(ptr), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(ATTN_ERR_LAUNCH, "cuTensorMapEncodeTiled failed (%d)", static_cast<int>(r));
  return ATTN_OK;
}

// Limit of every bounded device-side wait: ATTN_WAIT_LIMIT_MS when set (> 0), else 2 s.
unsigned long long wait_limit_ns() {
  const char* v = std::getenv("ATTN_WAIT_LIMIT_MS");
  if (v && *v) {
    const long ms = std::strtol(v, nullptr, 10);
    if (ms > 0) return static_cast<unsigned long long>(ms) * 1000000ull;
  }
  return kDefaultTimeoutNs;
}

// Test hook: ATTN_TEST_WITHHOLD_K_BLOCK=j makes every CTA's producer skip the load of key
// block j, so the waits on it run out and the failure path can be exercised without a fault.
// It is honoured only while ATTN_ENABLE_TEST_HOOKS=1 is set as well, so that a stray
// variable in a user's environment cannot silently drop keys.
int fault_block() {
  const char* on = std::getenv("ATTN_ENABLE_TEST_HOOKS");
  if (!on || std::strcmp(on, "1") != 0) return -1;
  const char* v = std::getenv("ATTN_TEST_WITHHOLD_K_BLOCK");
  if (v && *v) return static_cast<int>(std::strtol(v, nullptr, 10));
  return -1;
}

bool misaligned(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) != 0; }

attn_status check_args(const void* Q, const void* K, const void* V, void* O, float* LSE, int B, int H, int Nq,
                       int Nk, int d, float scale) {
  if (B < 0 || H < 0 || Nq < 0 || Nk < 0)
    return fail(ATTN_ERR_BAD_SHAPE, "negative size (B=%d H=%d Nq=%d Nk=%d)", B, H, Nq, Nk);
  if (d != 64 && d != 128) return fail(ATTN_ERR_UNSUPPORTED_D, "d=%d; supported: 64, 128", d);
  const long long BH = static_cast<long long>(B) * H;
  const long long tiles = BH * ((Nq + attn::kBM - 1) / attn::kBM);
  if (BH > INT32_MAX || tiles > INT32_MAX || static_cast<long long>(Nq) * BH > INT32_MAX * 64ll)
    return fail(ATTN_ERR_BAD_SHAPE, "problem too large (B*H=%lld)", BH);
  if (!std::isfinite(scale) || !(scale > 0.f)) return fail(ATTN_ERR_BAD_ARG, "scale must be finite and > 0");
  if (BH == 0 || Nq == 0) return ATTN_OK;
  if (!Q || !O || !LSE) return fail(ATTN_ERR_NULLPTR, "Q, O and LSE must not be NULL");
  if (Nk > 0 && (!K || !V)) return fail(ATTN_ERR_NULLPTR, "K and V must not be NULL when Nk > 0");
  if (misaligned(Q) || misaligned(O) || (Nk > 0 && (misaligned(K) || misaligned(V))))
    return fail(ATTN_ERR_MISALIGNED, "Q, K, V and O must be 16-byte aligned");
  if (reinterpret_cast<uintptr_t>(LSE) & 3u) return fail(ATTN_ERR_MISALIGNED, "LSE must be 4-byte aligned");
  return ATTN_OK;
}

// Where a partial-state launch writes: o~ [S, BH, Nq, D], m and l [S, BH, Nq], all fp32.
struct StateOut {
  float* o = nullptr;
  float* m = nullptr;
  float* l = nullptr;
  int num_splits = 1;
};

// How many of every 16 score pairs of an unmasked block take the polynomial exponential
// (exp2_poly2) in ATTN_EXP2_MIXED mode, per head dimension: of the splits measured on
// GB300 (1 to 5 of 16) the least slow; every split was slower than ex2.approx alone, so
// the default mode is ATTN_EXP2_HARDWARE.  The macros let a build try other splits.
#ifndef ATTN_SOFT_PAIRS_D128
#define ATTN_SOFT_PAIRS_D128 1
#endif
#ifndef ATTN_SOFT_PAIRS_D64
#define ATTN_SOFT_PAIRS_D64 1
#endif
template <int D>
constexpr int kDefaultSoftPairs = (D == 128) ? ATTN_SOFT_PAIRS_D128 : ATTN_SOFT_PAIRS_D64;

// Per-call choices the options struct carries, resolved for the kernel.
struct Variant {
  float tau_log2 = 0.f;  // rescale threshold in log2 units
  bool soft = false;     // mixed exponentials (kDefaultSoftPairs) or ex2.approx only (default)
  int key_block = attn::kBN;  // keys per block: kBN, or kBNWide / kBNNarrow (d = 128 dense, O out)
};

// Sets max dynamic shared memory once per device for a kernel instantiation.
template <typename Kernel>
attn_status set_smem_attr(Kernel kernel, int bytes, int dev, bool* done) {
  std::lock_guard<std::mutex> lock(g_mu);
  if (!done[dev]) {
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e != cudaSuccess) return fail(ATTN_ERR_LAUNCH, "cudaFuncSetAttribute: %s", cudaGetErrorString(e));
    done[dev] = true;
  }
  return ATTN_OK;
}

// Tensor maps of Q, K, V (and O unless the launch writes partial states) and the kernel
// parameters every forward kernel shares.
template <int D, bool kStates>
attn_status make_launch(const void* Q, const void* K, const void* V, void* O, float* LSE, int B, int H, int Nq,
                        int Nk, float scale, int causal, const int32_t* lens, uint32_t* status, const StateOut& so,
                        const Variant& var, const Geometry& geo, CUtensorMap* mq, CUtensorMap* mk, CUtensorMap* mv,
                        CUtensorMap* mo, attn::FwdParams* pp, int kv_box_rows = attn::kBN) {
  const int BH = B * H;
  attn_status st;
  if ((st = make_map(mq, Q, D, geo.q_rows, H, geo.map_b, geo.qs)) != ATTN_OK) return st;
  if (kStates) {
    *mo = *mq;  // never used: the partial-state epilogue stores with plain writes
  } else if ((st = make_map(mo, O, D, geo.q_rows, H, geo.map_b, geo.os)) != ATTN_OK) {
    return st;
  }
  if (geo.k_rows > 0) {
    // K and V move a key block at a time: kv_box_rows rows per copy
    if ((st = make_map(mk, K, D, geo.k_rows, H, geo.map_b, geo.ks, kv_box_rows)) != ATTN_OK) return st;
    if ((st = make_map(mv, V, D, geo.k_rows, H, geo.map_b, geo.vs, kv_box_rows)) != ATTN_OK) return st;
  } else {  // never read: every row is fully masked
    *mk = *mq;
    *mv = *mq;
  }
  attn::FwdParams& p = *pp;
  p.BH = BH;
  p.H = H;
  p.Nq = Nq;
  p.Nk = Nk;
  p.num_qtiles = (geo.grid_q + attn::kBM - 1) / attn::kBM;
  p.causal = causal ? 1 : 0;
  p.rank_major = 0;
  p.order_div = p.num_qtiles;
  p.c = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
  p.lens = lens;
  p.lse = LSE;
  p.status = status;
  p.timeout_ns = wait_limit_ns();
  p.fault_block = fault_block();
  p.tau = var.tau_log2;
  const int nkb = (Nk + attn::kBN - 1) / attn::kBN;
  p.num_splits = kStates ? so.num_splits : 1;
  p.split_blocks = kStates ? std::max(1, (nkb + so.num_splits - 1) / so.num_splits) : std::max(1, nkb);
  p.st_o = so.o;
  p.st_m = so.m;
  p.st_l = so.l;
  p.cu_q = geo.cu_q;
  p.cu_k = geo.cu_k;
  p.seq_sort = (geo.cu_q && B > 1 && B <= attn::kMaxSortedSeqs) ? 1 : 0;  // read by the packed kernels only
  p.total_q = static_cast<int>(geo.q_rows);
  p.total_k = static_cast<int>(geo.k_rows);
  p.o = static_cast<__nv_bfloat16*>(O);
  p.os_b = geo.cu_q ? 0 : geo.os[0];  // packed sequences address rows from cu_q, not by batch
  p.os_h = geo.os[1];
  p.os_r = geo.os[2];
  // O's base and every row stride (bf16 elements) on 32 bytes: each row can be stored 32
  // bytes at a time
  p.o_v8 = ((reinterpret_cast<uintptr_t>(O) & 31) == 0 && (p.os_b * 2) % 32 == 0 && (p.os_h * 2) % 32 == 0 &&
            (p.os_r * 2) % 32 == 0) ? 1 : 0;
  p.num_items = static_cast<int>(static_cast<long long>(p.num_qtiles) * BH * p.num_splits);
  return ATTN_OK;
}

// Multiplier and shift that divide by d with one multiply-high, one add and one shift:
// n / d = (umulhi(m, n) + n) >> s for 0 <= n < 2^31 and 1 <= d < 2^31, with s = ceil(log2 d)
// and m = floor(2^32 (2^s - d) / d) + 1 (the round-up method for division by invariant
// integers; n + umulhi(m, n) stays below 2^32 because both terms are below 2^31).
void divisor(int d, uint32_t* m, uint32_t* s) {
  uint32_t l = 0;
  while ((1ull << l) < static_cast<unsigned long long>(d)) ++l;
  *m = static_cast<uint32_t>(((1ull << 32) * ((1ull << l) - static_cast<unsigned long long>(d))) / d + 1);
  *s = l;
}
void set_divisors(attn::FwdParams* p) {
  divisor(p->num_splits, &p->dm_split, &p->ds_split);
  divisor(p->order_div, &p->dm_order, &p->ds_order);
  divisor(p->H, &p->dm_h, &p->ds_h);
}

// Launches `kernel` with programmatic stream serialization: it may be scheduled on the SMs
// the previous kernel in `stream` has already left, run its prologue there (barriers,
// tensor-memory allocation, descriptor prefetch) and wait in griddep_wait() for that
// kernel to finish before it touches global memory.  Stream order is kept for everything
// the kernels read and write.
template <typename... Params, typename... Args>
cudaError_t launch_pdl(void (*kernel)(Params...), unsigned grid, unsigned block, size_t smem, cudaStream_t stream,
                       Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(block);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Causal problems whose K and V take at most this much run every head's longest tiles
// first (FwdParams::rank_major): with K/V of all heads in L2 at once, the order evens out
// the CTAs' work; above it, heads in order keep each head's K/V in L2 while it runs.
constexpr long long kRankMajorMaxKvBytes = 96ll << 20;

// K and V of every head, bytes.
long long kv_footprint(int B, int H, int Nk, int D) { return 4ll * B * H * Nk * D; }

// The shared-memory attribute of one instantiation of each forward kernel, set once per
// device (one flag per device and instantiation).
template <int D, bool kStates, int kSoft, bool kPacked, int BN = attn::kBN>
attn_status fwd_kernel_attr(int dev) {
  static bool attr_set[kMaxDevices] = {};
  return set_smem_attr(attn::attn_fwd_kernel<D, kStates, kSoft, kPacked, BN>, attn::FwdCfg<D, BN>::kSmemAlloc, dev,
                       attr_set);
}
template <int kSoft, bool kPacked>
attn_status pair_kernel_attr(int dev) {
  static bool attr_set[kMaxDevices] = {};
  return set_smem_attr(attn::attn_fwd_pair_kernel<kSoft, kPacked>, attn::PairCfg::kSmemAlloc, dev, attr_set);
}

template <int D, bool kStates, int kSoft, bool kPacked, int BN = attn::kBN>
attn_status launch_one(const void* Q, const void* K, const void* V, void* O, float* LSE, int B, int H, int Nq,
                       int Nk, float scale, int causal, const int32_t* lens, cudaStream_t stream, int dev,
                       uint32_t* status, const StateOut& so, const Variant& var, const Geometry& geo) {
  using C = attn::FwdCfg<D, BN>;
  auto kernel = attn::attn_fwd_kernel<D, kStates, kSoft, kPacked, BN>;
  attn_status st;
  if ((st = fwd_kernel_attr<D, kStates, kSoft, kPacked, BN>(dev)) != ATTN_OK) return st;
  CUtensorMap mq, mk, mv, mo;
  attn::FwdParams p;
  if ((st = make_launch<D, kStates>(Q, K, V, O, LSE, B, H, Nq, Nk, scale, causal, lens, status, so, var, geo, &mq,
                                    &mk, &mv, &mo, &p, BN)) != ATTN_OK)
    return st;
  if (!kStates && causal && !geo.cu_q && kv_footprint(B, H, Nk, D) <= kRankMajorMaxKvBytes) p.rank_major = 1;
  p.order_div = p.rank_major ? p.BH : p.num_qtiles;
  set_divisors(&p);
  // persistent: one CTA per SM (shared and tensor memory allow no second), each walking
  // its items
  const int sms = sm_count(dev);
  const unsigned grid = static_cast<unsigned>(std::min<long long>(p.num_items, sms > 0 ? sms : 1));
  // only packed-sequence launches use the sequence order's shared memory
  const int smem = p.seq_sort ? C::kSmemAlloc : C::kSmemAllocNoPerm;
  cudaError_t e = launch_pdl(kernel, grid, attn::kThreads, smem, stream, mq, mk, mv, mo, p);
  if (e != cudaSuccess) return fail(ATTN_ERR_LAUNCH, "kernel launch: %s", cudaGetErrorString(e));
  return ATTN_OK;
}

// d = 64, O and LSE out: two query tiles per CTA (attn_fwd_pair_kernel), when there are
// enough pairs of tiles to give every SM one.
template <int kSoft, bool kPacked>
attn_status launch_pair(const void* Q, const void* K, const void* V, void* O, float* LSE, int B, int H, int Nq,
                        int Nk, float scale, int causal, const int32_t* lens, cudaStream_t stream, int dev,
                        uint32_t* status, const Variant& var, const Geometry& geo) {
  using C = attn::PairCfg;
  auto kernel = attn::attn_fwd_pair_kernel<kSoft, kPacked>;
  attn_status st;
  if ((st = pair_kernel_attr<kSoft, kPacked>(dev)) != ATTN_OK) return st;
  CUtensorMap mq, mk, mv, mo;
  attn::FwdParams p;
  if ((st = make_launch<64, false>(Q, K, V, O, LSE, B, H, Nq, Nk, scale, causal, lens, status, StateOut{}, var, geo,
                                   &mq, &mk, &mv, &mo, &p)) != ATTN_OK)
    return st;
  p.num_items = static_cast<int>(static_cast<long long>((p.num_qtiles + 1) / 2) * p.BH);  // pairs of tiles
  if (causal && !geo.cu_q && kv_footprint(B, H, Nk, 64) <= kRankMajorMaxKvBytes) p.rank_major = 1;
  p.order_div = p.rank_major ? p.BH : (p.num_qtiles + 1) / 2;
  const int sms = sm_count(dev);
  const unsigned grid = static_cast<unsigned>(std::min<long long>(p.num_items, sms > 0 ? sms : 1));
  const int smem = p.seq_sort ? C::kSmemAlloc : C::kSmemAllocNoPerm;
  cudaError_t e = launch_pdl(kernel, grid, attn::kPairThreads, smem, stream, mq, mk, mv, p);
  if (e != cudaSuccess) return fail(ATTN_ERR_LAUNCH, "kernel launch: %s", cudaGetErrorString(e));
  return ATTN_OK;
}

// Whether a d = 64 forward takes the two-tile kernel (measured on GB300): with a causal
// mask, when every SM gets a pair of query tiles (with fewer, single tiles spread the
// unequal causal tiles over more SMs); without one, as soon as the pairs fill more than
// half the SMs (a single-tile grid would then need two rounds of equal tiles).
bool use_pair_kernel(int dev, int B, int H, const Geometry& geo, int causal) {
  const long long pairs = static_cast<long long>(B) * H * (((geo.grid_q + attn::kBM - 1) / attn::kBM + 1) / 2);
  return causal ? pairs >= sm_count(dev) : 2 * pairs > sm_count(dev);
}

// kPacked: packed sequences (geo.cu_q set), the kernels' instantiation that may rank them.
template <int D, bool kStates, bool kPacked>
attn_status launch_as(const void* Q, const void* K, const void* V, void* O, float* LSE, int B, int H, int Nq, int Nk,
                      float scale, int causal, const int32_t* lens, cudaStream_t stream, int dev, uint32_t* status,
                      const StateOut& so, const Variant& var, const Geometry& g) {
  if (var.key_block != attn::kBN) {  // the 192- and 64-key-block builds: d = 128, O out, not packed
    if constexpr (D == 128 && !kStates && !kPacked) {
      if (var.key_block == attn::kBNWide)
        return launch_one<128, false, 0, false, attn::kBNWide>(Q, K, V, O, LSE, B, H, Nq, Nk, scale, causal, lens,
                                                               stream, dev, status, so, var, g);
      return launch_one<128, false, 0, false, attn::kBNNarrow>(Q, K, V, O, LSE, B, H, Nq, Nk, scale, causal, lens,
                                                               stream, dev, status, so, var, g);
    }
    return fail(ATTN_ERR_BAD_ARG, "key_block=%d is available at d = 128 without packed sequences",
                var.key_block);
  }
  if constexpr (D == 64 && !kStates) {
    if (use_pair_kernel(dev, B, H, g, causal)) {
      if (var.soft)
        return launch_pair<kDefaultSoftPairs<64>, kPacked>(Q, K, V, O, LSE, B, H, Nq, Nk, scale, causal, lens,
                                                           stream, dev, status, var, g);
      return launch_pair<0, kPacked>(Q, K, V, O, LSE, B, H, Nq, Nk, scale, causal, lens, stream, dev, status, var,
                                     g);
    }
  }
  if (var.soft)
    return launch_one<D, kStates, kDefaultSoftPairs<D>, kPacked>(Q, K, V, O, LSE, B, H, Nq, Nk, scale, causal, lens,
                                                                 stream, dev, status, so, var, g);
  return launch_one<D, kStates, 0, kPacked>(Q, K, V, O, LSE, B, H, Nq, Nk, scale, causal, lens, stream, dev, status,
                                            so, var, g);
}

template <int D, bool kStates>
attn_status launch(const void* Q, const void* K, const void* V, void* O, float* LSE, int B, int H, int Nq, int Nk,
                   float scale, int causal, const int32_t* lens, cudaStream_t stream, int dev, uint32_t* status,
                   const StateOut& so = StateOut{}, const Variant& var = Variant{}, const Geometry* geo = nullptr) {
  const Geometry g = geo ? *geo : dense_geometry(B, H, Nq, Nk, D);
  if constexpr (!kStates) {
    if (g.cu_q)
      return launch_as<D, false, true>(Q, K, V, O, LSE, B, H, Nq, Nk, scale, causal, lens, stream, dev, status, so,
                                       var, g);
  }
  return launch_as<D, kStates, false>(Q, K, V, O, LSE, B, H, Nq, Nk, scale, causal, lens, stream, dev, status, so,
                                      var, g);
}

// Options -> kernel variant; NULL means the defaults.
attn_status resolve_options(const attn_options* opts, Variant* var) {
  *var = Variant{};
  if (!opts) return ATTN_OK;
  // the first fields are always there; key_block was added later and defaults when the
  // caller's struct ends before it
  const size_t base = offsetof(attn_options, key_block);
  if (opts->size < base)
    return fail(ATTN_ERR_BAD_ARG, "attn_options.size=%zu; expected at least %zu", opts->size, base);
  const float t = opts->rescale_threshold;
  if (!std::isfinite(t) || t < 0.f || t > 20.f)
    return fail(ATTN_ERR_BAD_ARG, "rescale_threshold=%g; must be in [0, 20]", static_cast<double>(t));
  if (opts->exp2_mode < ATTN_EXP2_DEFAULT || opts->exp2_mode > ATTN_EXP2_MIXED)
    return fail(ATTN_ERR_BAD_ARG, "exp2_mode=%d", opts->exp2_mode);
  var->tau_log2 = static_cast<float>(static_cast<double>(t) * 1.4426950408889634);
  var->soft = opts->exp2_mode == ATTN_EXP2_MIXED;
  if (opts->size >= base + sizeof(int)) {
    const int kb = opts->key_block;
    if (kb != 0 && kb != attn::kBN && kb != attn::kBNWide && kb != attn::kBNNarrow)
      return fail(ATTN_ERR_BAD_ARG, "key_block=%d; must be 0, %d, %d or %d", kb, attn::kBN, attn::kBNNarrow,
                  attn::kBNWide);
    if ((kb == attn::kBNWide || kb == attn::kBNNarrow) && var->soft)
      return fail(ATTN_ERR_BAD_ARG, "key_block=%d takes exp2_mode ATTN_EXP2_HARDWARE or DEFAULT", kb);
    var->key_block = kb == 0 ? attn::kBN : kb;
  }
  return ATTN_OK;
}

}  // namespace

extern "C" {

attn_status attn_fwd(const void* Q, const void* K, const void* V, void* O, float* LSE, int B, int H, int Nq, int Nk,
                     int d, float scale, int causal, const int32_t* key_padding_lens, void* stream) {
  g_err[0] = '\0';
  attn_status st = check_args(Q, K, V, O, LSE, B, H, Nq, Nk, d, scale);
  if (st != ATTN_OK) return st;
  if (static_cast<long long>(B) * H == 0 || Nq == 0) return ATTN_OK;
  int dev;
  if ((st = get_device(&dev)) != ATTN_OK) return st;
  uint32_t* status = nullptr;
  if ((st = setup(dev, &status)) != ATTN_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (d == 128)
    return launch<128, false>(Q, K, V, O, LSE, B, H, Nq, Nk, scale, causal, key_padding_lens, s, dev, status);
  return launch<64, false>(Q, K, V, O, LSE, B, H, Nq, Nk, scale, causal, key_padding_lens, s, dev, status);
}

attn_status attn_fwd_ex(const void* Q, const void* K, const void* V, void* O, float* LSE, int B, int H, int Nq,
                        int Nk, int d, float scale, int causal, const int32_t* key_padding_lens,
                        const attn_options* opts, void* stream) {
  g_err[0] = '\0';
  Variant var;
  attn_status st = resolve_options(opts, &var);
  if (st != ATTN_OK) return st;
  if ((st = check_args(Q, K, V, O, LSE, B, H, Nq, Nk, d, scale)) != ATTN_OK) return st;
  if (static_cast<long long>(B) * H == 0 || Nq == 0) return ATTN_OK;
  int dev;
  if ((st = get_device(&dev)) != ATTN_OK) return st;
  uint32_t* status = nullptr;
  if ((st = setup(dev, &status)) != ATTN_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (d == 128)
    return launch<128, false>(Q, K, V, O, LSE, B, H, Nq, Nk, scale, causal, key_padding_lens, s, dev, status,
                              StateOut{}, var);
  return launch<64, false>(Q, K, V, O, LSE, B, H, Nq, Nk, scale, causal, key_padding_lens, s, dev, status,
                           StateOut{}, var);
}

attn_status attn_fwd_strided(const void* Q, const void* K, const void* V, void* O, float* LSE, int B, int H, int Nq,
                             int Nk, int d, float scale, int causal, const int32_t* key_padding_lens,
                             const int64_t* q_strides, const int64_t* k_strides, const int64_t* v_strides,
                             const int64_t* o_strides, void* stream) {
  g_err[0] = '\0';
  attn_status st = check_args(Q, K, V, O, LSE, B, H, Nq, Nk, d, scale);
  if (st != ATTN_OK) return st;
  if (static_cast<long long>(B) * H == 0 || Nq == 0) return ATTN_OK;
  if (!q_strides || !k_strides || !v_strides || !o_strides) return fail(ATTN_ERR_NULLPTR, "stride arrays must not be NULL");
  Geometry g = dense_geometry(B, H, Nq, Nk, d);
  const int64_t* in[4] = {q_strides, k_strides, v_strides, o_strides};
  long long* out[4] = {g.qs, g.ks, g.vs, g.os};
  for (int t = 0; t < 4; ++t)
    for (int i = 0; i < 3; ++i) {
      const int64_t v = in[t][i];
      if (v <= 0 || (v & 7) != 0 || v >= (1ll << 38))
        return fail(ATTN_ERR_BAD_ARG, "stride %d of tensor %d is %lld; strides must be positive multiples of 8 "
                    "elements (16 bytes) below 2^38", i, t, static_cast<long long>(v));
      out[t][i] = v;
    }
  int dev;
  if ((st = get_device(&dev)) != ATTN_OK) return st;
  uint32_t* status = nullptr;
  if ((st = setup(dev, &status)) != ATTN_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (d == 128)
    return launch<128, false>(Q, K, V, O, LSE, B, H, Nq, Nk, scale, causal, key_padding_lens, s, dev, status,
                              StateOut{}, Variant{}, &g);
  return launch<64, false>(Q, K, V, O, LSE, B, H, Nq, Nk, scale, causal, key_padding_lens, s, dev, status,
                           StateOut{}, Variant{}, &g);
}

attn_status attn_fwd_varlen(const void* Q, const void* K, const void* V, void* O, float* LSE,
                            const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k, int B, int H, int max_seqlen_q,
                            int total_q, int total_k, int d, float scale, int causal, void* stream) {
  g_err[0] = '\0';
  if (B < 0 || H < 0 || max_seqlen_q < 0 || total_q < 0 || total_k < 0)
    return fail(ATTN_ERR_BAD_SHAPE, "negative size (B=%d H=%d max_seqlen_q=%d total_q=%d total_k=%d)", B, H,
                max_seqlen_q, total_q, total_k);
  if (d != 64 && d != 128) return fail(ATTN_ERR_UNSUPPORTED_D, "d=%d; supported: 64, 128", d);
  if (!std::isfinite(scale) || !(scale > 0.f)) return fail(ATTN_ERR_BAD_ARG, "scale must be finite and > 0");
  const long long tiles = static_cast<long long>(B) * H * ((max_seqlen_q + attn::kBM - 1) / attn::kBM);
  if (tiles > INT32_MAX || static_cast<long long>(total_q) * H * d > (1ll << 40))
    return fail(ATTN_ERR_BAD_SHAPE, "problem too large");
  if (static_cast<long long>(B) * H == 0 || max_seqlen_q == 0 || total_q == 0) return ATTN_OK;
  if (!Q || !O || !LSE || !cu_seqlens_q || !cu_seqlens_k)
    return fail(ATTN_ERR_NULLPTR, "Q, O, LSE and the cu_seqlens arrays must not be NULL");
  if (total_k > 0 && (!K || !V)) return fail(ATTN_ERR_NULLPTR, "K and V must not be NULL when total_k > 0");
  if (misaligned(Q) || misaligned(O) || misaligned(LSE) || (total_k > 0 && (misaligned(K) || misaligned(V))))
    return fail(ATTN_ERR_MISALIGNED, "pointers must be 16-byte aligned");
  Geometry g;
  const long long row = static_cast<long long>(H) * d;  // packed [total, H, d]
  const long long q[3] = {static_cast<long long>(total_q) * row, d, row};
  const long long k[3] = {static_cast<long long>(total_k > 0 ? total_k : 1) * row, d, row};
  for (int i = 0; i < 3; ++i) {
    g.qs[i] = g.os[i] = q[i];
    g.ks[i] = g.vs[i] = k[i];
  }
  g.q_rows = total_q;
  g.k_rows = total_k;
  g.map_b = 1;
  g.grid_q = max_seqlen_q;
  g.cu_q = cu_seqlens_q;
  g.cu_k = cu_seqlens_k;
  int dev;
  attn_status st;
  if ((st = get_device(&dev)) != ATTN_OK) return st;
  uint32_t* status = nullptr;
  if ((st = setup(dev, &status)) != ATTN_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // Nq / Nk of the parameters are unused for packed sequences (each CTA reads its own)
  if (d == 128)
    return launch<128, false>(Q, K, V, O, LSE, B, H, max_seqlen_q, 0, scale, causal, nullptr, s, dev, status,
                              StateOut{}, Variant{}, &g);
  return launch<64, false>(Q, K, V, O, LSE, B, H, max_seqlen_q, 0, scale, causal, nullptr, s, dev, status,
                           StateOut{}, Variant{}, &g);
}

attn_status attn_fwd_host(const void* Q, const void* K, const void* V, void* O, float* LSE, int B, int H, int Nq,
                          int Nk, int d, float scale, int causal, const int32_t* key_padding_lens, void* stream) {
  g_err[0] = '\0';
  attn_status st = check_args(Q, K, V, O, LSE, B, H, Nq, Nk, d, scale);
  if (st != ATTN_OK) return st;
  if (static_cast<long long>(B) * H == 0 || Nq == 0) return ATTN_OK;
  int dev;
  if ((st = get_device(&dev)) != ATTN_OK) return st;
  const size_t BH = static_cast<size_t>(B) * H;
  const size_t q_bytes = BH * Nq * d * 2, kv_bytes = BH * Nk * d * 2, lse_bytes = BH * Nq * 4;
  const size_t lens_bytes = key_padding_lens ? static_cast<size_t>(B) * 4 : 0;
  auto up = [](size_t x) { return (x + 255) & ~static_cast<size_t>(255); };
  const size_t need = 2 * up(q_bytes) + 2 * up(kv_bytes) + up(lse_bytes) + up(lens_bytes);
  Workspace& ws = g_ws[dev];
  {
    std::lock_guard<std::mutex> lock(g_mu);
    if (ws.bytes < need) {
      if (ws.base) cudaFree(ws.base);
      ws.base = nullptr;
      ws.bytes = 0;
      if (cudaMalloc(&ws.base, need) != cudaSuccess) return fail(ATTN_ERR_LAUNCH, "workspace alloc of %zu B failed", need);
      ws.bytes = need;
    }
  }
  uint8_t* w = static_cast<uint8_t*>(ws.base);
  uint8_t* dQ = w;
  uint8_t* dO = dQ + up(q_bytes);
  uint8_t* dK = dO + up(q_bytes);
  uint8_t* dV = dK + up(kv_bytes);
  float* dL = reinterpret_cast<float*>(dV + up(kv_bytes));
  int32_t* dlens = key_padding_lens ? reinterpret_cast<int32_t*>(reinterpret_cast<uint8_t*>(dL) + up(lse_bytes)) : nullptr;
  HostPipe* hp = nullptr;
  if ((st = host_pipe(dev, &hp)) != ATTN_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // The copies run on two streams of their own, overlapped with the forward on `stream`:
  // chunk i (a run of heads of one batch) is copied in, computed, and copied out while
  // chunk i + 1 is copied in.  Chunks start after the work already queued on `stream`,
  // and `stream` waits for the last copy out, so the call keeps stream order.
  const int nch = host_chunks(B, H, q_bytes + 2 * kv_bytes);
  cudaError_t e = cudaEventRecord(hp->ev_start, s);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(hp->in, hp->ev_start, 0);
  if (e == cudaSuccess && lens_bytes)
    e = cudaMemcpyAsync(dlens, key_padding_lens, lens_bytes, cudaMemcpyHostToDevice, hp->in);
  const size_t qh = static_cast<size_t>(Nq) * d * 2, kh = static_cast<size_t>(Nk) * d * 2;  // bytes per head
  int done = 0;
  for (int b = 0; b < B && e == cudaSuccess; ++b) {
    for (int h0 = 0; h0 < H && e == cudaSuccess; ++done) {
      const int hc = std::min(H - h0, (H + nch_per_batch(nch, B) - 1) / nch_per_batch(nch, B));
      const size_t bh0 = static_cast<size_t>(b) * H + h0;
      const int slot = done % kHostEvents;
      // the slot's events were last used kHostEvents chunks ago: their work is queued ahead
      e = cudaMemcpyAsync(dQ + bh0 * qh, static_cast<const uint8_t*>(Q) + bh0 * qh, hc * qh, cudaMemcpyHostToDevice,
                          hp->in);
      if (e == cudaSuccess && kh)
        e = cudaMemcpyAsync(dK + bh0 * kh, static_cast<const uint8_t*>(K) + bh0 * kh, hc * kh,
                            cudaMemcpyHostToDevice, hp->in);
      if (e == cudaSuccess && kh)
        e = cudaMemcpyAsync(dV + bh0 * kh, static_cast<const uint8_t*>(V) + bh0 * kh, hc * kh,
                            cudaMemcpyHostToDevice, hp->in);
      if (e == cudaSuccess) e = cudaEventRecord(hp->ev_in[slot], hp->in);
      if (e == cudaSuccess) e = cudaStreamWaitEvent(s, hp->ev_in[slot], 0);
      if (e != cudaSuccess) break;
      st = attn_fwd(dQ + bh0 * qh, kh ? dK + bh0 * kh : nullptr, kh ? dV + bh0 * kh : nullptr, dO + bh0 * qh,
                    dL + bh0 * Nq, 1, hc, Nq, Nk, d, scale, causal, dlens ? dlens + b : nullptr, stream);
      if (st != ATTN_OK) return st;
      e = cudaEventRecord(hp->ev_done[slot], s);
      if (e == cudaSuccess) e = cudaStreamWaitEvent(hp->out, hp->ev_done[slot], 0);
      if (e == cudaSuccess)
        e = cudaMemcpyAsync(static_cast<uint8_t*>(O) + bh0 * qh, dO + bh0 * qh, hc * qh, cudaMemcpyDeviceToHost,
                            hp->out);
      if (e == cudaSuccess)
        e = cudaMemcpyAsync(LSE + bh0 * Nq, dL + bh0 * Nq, static_cast<size_t>(hc) * Nq * 4, cudaMemcpyDeviceToHost,
                            hp->out);
      h0 += hc;
    }
  }
  if (e == cudaSuccess) e = cudaEventRecord(hp->ev_end, hp->out);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(s, hp->ev_end, 0);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return fail(ATTN_ERR_LAUNCH, "host-buffer pipeline: %s", cudaGetErrorString(e));
  return ATTN_OK;
}

attn_status attn_release_workspace(void) {
  int dev;
  attn_status st = get_device(&dev);
  if (st != ATTN_OK) return st;
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_ws[dev].base) cudaFree(g_ws[dev].base);
  g_ws[dev] = Workspace{};
  return ATTN_OK;
}

attn_status attn_status_sync(void* stream) {
  g_err[0] = '\0';
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail(ATTN_ERR_LAUNCH, "stream sync: %s", cudaGetErrorString(e));
  int dev;
  attn_status st = get_device(&dev);
  if (st != ATTN_OK) return st;
  // the status word of the allocating entry points, then the no-alloc entry point's one
  uint32_t* words[2] = {g_status[dev], g_noalloc_addr[dev]};
  uint32_t seen = 0;
  for (uint32_t* w : words) {
    if (!w) continue;
    uint32_t v = 0;
    if (cudaMemcpy(&v, w, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess)
      return fail(ATTN_ERR_LAUNCH, "status read failed");
    if (v) {  // cleared in `stream` order, so a later launch's report is not wiped
      cudaStream_t s = static_cast<cudaStream_t>(stream);
      if (cudaMemsetAsync(w, 0, sizeof(uint32_t), s) != cudaSuccess || cudaStreamSynchronize(s) != cudaSuccess)
        return fail(ATTN_ERR_LAUNCH, "status clear failed");
      seen |= v;
    }
  }
  if (seen) return fail(ATTN_ERR_TIMEOUT, "a bounded device wait ran out (status word 0x%x)", seen);
  return ATTN_OK;
}

const char* attn_last_error(void) { return g_err; }

int attn_version(void) { return 100; }

}  // extern "C"

// ---------------------------------------------------------------------------------------
// Allocation-free entry point.  Its device scratch is this fixed array: word 0 is the
// status word of the kernel's bounded waits.  Host code only ever uses the array's name
// through cudaGetSymbolAddress; the address it returns (per device) goes to the kernel.

namespace {

constexpr int kNoAllocScratchWords = 64;
constexpr size_t kNoAllocScratchBytes = kNoAllocScratchWords * sizeof(uint32_t);  // 256 B per device
static __device__ __align__(256) uint32_t g_noalloc_scratch[kNoAllocScratchWords];

// One-time set-up per device (that device current): kernel-facing address of the array,
// device check, the tensor-map encoder, and every kernel attribute and cached value a later
// call could otherwise set on first use (the shared-memory size of each forward kernel
// this entry point can launch, the SM count).  No allocation.
attn_status noalloc_setup(int dev, uint32_t** addr) {
  {
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_encode) {
      void* fn = nullptr;
      cudaDriverEntryPointQueryResult q;
      cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
      if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !fn)
        return fail(ATTN_ERR_NO_DEVICE, "cuTensorMapEncodeTiled unavailable: %s", cudaGetErrorString(e));
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
    if (g_noalloc_addr[dev]) {
      *addr = g_noalloc_addr[dev];
      return ATTN_OK;
    }
    cudaDeviceProp prop;
    if (cudaGetDeviceProperties(&prop, dev) != cudaSuccess)
      return fail(ATTN_ERR_NO_DEVICE, "cudaGetDeviceProperties failed");
    if (prop.major != 10 || prop.minor != 3)
      return fail(ATTN_ERR_NO_DEVICE, "device %d is sm_%d%d; this library is built for sm_103a", dev, prop.major,
                  prop.minor);
  }
  // set_smem_attr takes the lock itself
  attn_status st;
  if ((st = fwd_kernel_attr<128, false, 0, false>(dev)) != ATTN_OK) return st;
  if ((st = fwd_kernel_attr<64, false, 0, false>(dev)) != ATTN_OK) return st;
  if ((st = pair_kernel_attr<0, false>(dev)) != ATTN_OK) return st;
  sm_count(dev);
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_noalloc_addr[dev]) {
    void* p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || !p)
      return fail(ATTN_ERR_NO_DEVICE, "cudaGetSymbolAddress of the scratch array failed: %s", cudaGetErrorString(e));
    g_noalloc_addr[dev] = static_cast<uint32_t*>(p);
  }
  *addr = g_noalloc_addr[dev];
  return ATTN_OK;
}

}  // namespace

extern "C" attn_status attn_fwd_noalloc(const void* Q, const void* K, const void* V, void* O, float* LSE, int B,
                                        int H, int Nq, int Nk, int d, float scale, int causal,
                                        const int32_t* key_padding_lens, int check_status, void* stream) {
  g_err[0] = '\0';
  attn_status st = check_args(Q, K, V, O, LSE, B, H, Nq, Nk, d, scale);
  if (st != ATTN_OK) return st;
  if (static_cast<long long>(B) * H == 0 || Nq == 0) return ATTN_OK;
  const size_t need = sizeof(uint32_t);  // the forward kernel's only scratch: its status word
  if (need > kNoAllocScratchBytes)
    return fail(ATTN_ERR_BAD_SHAPE, "needs %zu B of scratch; the fixed array holds %zu B", need,
                kNoAllocScratchBytes);
  int dev;
  if ((st = get_device(&dev)) != ATTN_OK) return st;
  uint32_t* scratch = nullptr;
  if ((st = noalloc_setup(dev, &scratch)) != ATTN_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // The status word is an OR of every bounded wait that ran out since it was last read:
  // it starts at zero (the array is zero when the library's module loads) and is cleared
  // only where it is read, here with check_status or by attn_status_sync.
  st = (d == 128) ? launch<128, false>(Q, K, V, O, LSE, B, H, Nq, Nk, scale, causal, key_padding_lens, s, dev, scratch)
                  : launch<64, false>(Q, K, V, O, LSE, B, H, Nq, Nk, scale, causal, key_padding_lens, s, dev, scratch);
  if (st != ATTN_OK || !check_status) return st;
  uint32_t word = 0;
  cudaError_t e = cudaStreamSynchronize(s);
  if (e == cudaSuccess) e = cudaMemcpy(&word, scratch, sizeof(word), cudaMemcpyDeviceToHost);
  if (e == cudaSuccess && word) {
    e = cudaMemsetAsync(scratch, 0, need, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  }
  if (e != cudaSuccess) return fail(ATTN_ERR_LAUNCH, "reading the status word: %s", cudaGetErrorString(e));
  if (word) return fail(ATTN_ERR_TIMEOUT, "a bounded device wait ran out (status word 0x%x)", word);
  return ATTN_OK;
}

// ---------------------------------------------------------------------------------------
// Split-KV: partial states over key splits, and their merge.

namespace {

constexpr int kMaxSplits = 256;

size_t round256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

attn_status launch_merge(const float* o_st, const float* m_st, const float* l_st, int S, long long rows, int d,
                         void* O, float* LSE, cudaStream_t stream, int sms) {
  attn::MergeParams mp;
  mp.st_o = o_st;
  mp.st_m = m_st;
  mp.st_l = l_st;
  mp.S = S;
  mp.rows = rows;
  mp.O = static_cast<__nv_bfloat16*>(O);
  mp.lse = LSE;
  constexpr long long kRowsPerBlock = attn::kMergeThreads / 32;
  const long long want = (rows + kRowsPerBlock - 1) / kRowsPerBlock;
  const unsigned grid = static_cast<unsigned>(std::min<long long>(want, static_cast<long long>(sms) * 8));
  cudaError_t e = d == 128 ? launch_pdl(attn::attn_merge_kernel<128>, grid, attn::kMergeThreads, 0, stream, mp)
                           : launch_pdl(attn::attn_merge_kernel<64>, grid, attn::kMergeThreads, 0, stream, mp);
  if (e != cudaSuccess) return fail(ATTN_ERR_LAUNCH, "merge launch: %s", cudaGetErrorString(e));
  return ATTN_OK;
}

// The automatic split count: enough (unit, split) CTAs to fill the SMs once when the
// units alone do not, never more splits than key blocks / 4 (each split keeps at least
// four blocks of work to amortise its start-up) and never more than kMaxSplits.
int auto_splits(long long units, int nkb, int sms) {
  if (units <= 0 || units >= sms) return 1;
  long long s = sms / units;
  s = std::min<long long>(s, std::max(1, nkb / 4));
  s = std::min<long long>(s, kMaxSplits);
  return static_cast<int>(std::max<long long>(1, s));
}

}  // namespace

extern "C" {

attn_status attn_fwd_states(const void* Q, const void* K, const void* V, float* o_states, float* m_states,
                            float* l_states, int B, int H, int Nq, int Nk, int d, float scale, int causal,
                            const int32_t* key_padding_lens, int num_splits, void* stream) {
  g_err[0] = '\0';
  attn_status st = check_args(Q, K, V, o_states, m_states, B, H, Nq, Nk, d, scale);
  if (st != ATTN_OK) return st;
  if (num_splits < 1 || num_splits > kMaxSplits)
    return fail(ATTN_ERR_BAD_ARG, "num_splits=%d; must be in [1, %d]", num_splits, kMaxSplits);
  if (static_cast<long long>(B) * H == 0 || Nq == 0) return ATTN_OK;
  if (!l_states) return fail(ATTN_ERR_NULLPTR, "l_states must not be NULL");
  if (misaligned(l_states)) return fail(ATTN_ERR_MISALIGNED, "pointers must be 16-byte aligned");
  const long long units = static_cast<long long>(B) * H * ((Nq + attn::kBM - 1) / attn::kBM);
  if (units * num_splits > INT32_MAX) return fail(ATTN_ERR_BAD_SHAPE, "too many (tile, split) units");
  int dev;
  if ((st = get_device(&dev)) != ATTN_OK) return st;
  uint32_t* status = nullptr;
  if ((st = setup(dev, &status)) != ATTN_OK) return st;
  StateOut so;
  so.o = o_states;
  so.m = m_states;
  so.l = l_states;
  so.num_splits = num_splits;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (d == 128)
    return launch<128, true>(Q, K, V, nullptr, nullptr, B, H, Nq, Nk, scale, causal, key_padding_lens, s, dev, status,
                             so);
  return launch<64, true>(Q, K, V, nullptr, nullptr, B, H, Nq, Nk, scale, causal, key_padding_lens, s, dev, status,
                          so);
}

attn_status attn_merge_states(const float* o_states, const float* m_states, const float* l_states, int num_states,
                              long long rows, int d, void* O, float* LSE, void* stream) {
  g_err[0] = '\0';
  if (d != 64 && d != 128) return fail(ATTN_ERR_UNSUPPORTED_D, "d=%d; supported: 64, 128", d);
  if (num_states < 1) return fail(ATTN_ERR_BAD_ARG, "num_states=%d; must be >= 1", num_states);
  if (rows < 0) return fail(ATTN_ERR_BAD_SHAPE, "rows=%lld must be >= 0", rows);
  if (rows == 0) return ATTN_OK;
  if (!o_states || !m_states || !l_states || !O || !LSE)
    return fail(ATTN_ERR_NULLPTR, "state and output pointers must not be NULL");
  if (misaligned(o_states) || misaligned(O) || (reinterpret_cast<uintptr_t>(m_states) & 3u) ||
      (reinterpret_cast<uintptr_t>(l_states) & 3u) || (reinterpret_cast<uintptr_t>(LSE) & 3u))
    return fail(ATTN_ERR_MISALIGNED, "o_states and O must be 16-byte aligned, m, l and LSE 4-byte aligned");
  int dev;
  attn_status st = get_device(&dev);
  if (st != ATTN_OK) return st;
  uint32_t* status = nullptr;
  if ((st = setup(dev, &status)) != ATTN_OK) return st;
  return launch_merge(o_states, m_states, l_states, num_states, rows, d, O, LSE, static_cast<cudaStream_t>(stream),
                      g_sms[dev]);
}

size_t attn_splitkv_workspace_bytes(int B, int H, int Nq, int d, int num_splits) {
  if (B < 0 || H < 0 || Nq < 0 || (d != 64 && d != 128) || num_splits < 1 || num_splits > kMaxSplits) return 0;
  const size_t rows = static_cast<size_t>(B) * H * Nq * num_splits;
  return round256(rows * d * 4) + 2 * round256(rows * 4);
}

int attn_splitkv_splits(int B, int H, int Nq, int Nk) {
  if (B <= 0 || H <= 0 || Nq <= 0 || Nk < 0) return 1;
  int dev;
  if (get_device(&dev) != ATTN_OK) return 1;
  uint32_t* status = nullptr;
  if (setup(dev, &status) != ATTN_OK) return 1;
  const long long units = static_cast<long long>(B) * H * ((Nq + attn::kBM - 1) / attn::kBM);
  return auto_splits(units, (Nk + attn::kBN - 1) / attn::kBN, g_sms[dev]);
}

attn_status attn_fwd_splitkv(const void* Q, const void* K, const void* V, void* O, float* LSE, int B, int H, int Nq,
                             int Nk, int d, float scale, int causal, const int32_t* key_padding_lens, int num_splits,
                             void* workspace, size_t workspace_bytes, void* stream) {
  g_err[0] = '\0';
  attn_status st = check_args(Q, K, V, O, LSE, B, H, Nq, Nk, d, scale);
  if (st != ATTN_OK) return st;
  if (num_splits > kMaxSplits) return fail(ATTN_ERR_BAD_ARG, "num_splits=%d > %d", num_splits, kMaxSplits);
  if (static_cast<long long>(B) * H == 0 || Nq == 0) return ATTN_OK;
  const int S = num_splits >= 1 ? num_splits : attn_splitkv_splits(B, H, Nq, Nk);
  if (S == 1) return attn_fwd(Q, K, V, O, LSE, B, H, Nq, Nk, d, scale, causal, key_padding_lens, stream);
  const size_t need = attn_splitkv_workspace_bytes(B, H, Nq, d, S);
  if (!workspace) return fail(ATTN_ERR_NULLPTR, "workspace must not be NULL for %d splits", S);
  if (misaligned(workspace)) return fail(ATTN_ERR_MISALIGNED, "workspace must be 16-byte aligned");
  if (workspace_bytes < need)
    return fail(ATTN_ERR_BAD_ARG, "workspace of %zu B is smaller than the %zu B %d splits need", workspace_bytes,
                need, S);
  const size_t rows = static_cast<size_t>(B) * H * Nq;
  uint8_t* w = static_cast<uint8_t*>(workspace);
  float* o_st = reinterpret_cast<float*>(w);
  float* m_st = reinterpret_cast<float*>(w + round256(rows * S * d * 4));
  float* l_st = reinterpret_cast<float*>(w + round256(rows * S * d * 4) + round256(rows * S * 4));
  st = attn_fwd_states(Q, K, V, o_st, m_st, l_st, B, H, Nq, Nk, d, scale, causal, key_padding_lens, S, stream);
  if (st != ATTN_OK) return st;
  return attn_merge_states(o_st, m_st, l_st, S, static_cast<long long>(rows), d, O, LSE, stream);
}

}  // extern "C"
