/*
 * attn.h -- C ABI of the fused attention forward (online softmax) for GB300 (sm_103a).
 *
 * The operation is the exact attention forward
 *
 *     O = softmax(scale * Q K^T + mask) V,   LSE_i = ln sum_j exp(scale * q_i . k_j)  (visible j)
 *
 * computed block by block with the online-softmax recurrence (running max m,
 * running denominator l, unnormalised accumulator o~, rescale by
 * alpha = exp(m_old - m_new) when the max rises, one division o~/l at the end),
 * never materialising the Nq x Nk score matrix.
 * Sources: "2.2b: FlashAttention -- Online Softmax" (hf-cn0.pages.dev), sections
 * "The Complete Online Softmax Algorithm" and "Extending to Attention";
 * "FlashAttention math" (aicassindra.com), sections "What we must compute" and
 * "The block-wise update, and the full algorithm"; "Tiled attention: running
 * max softmax" (archcrux.com) for masked keys and fully masked rows.
 *
 * Conventions (the pages leave these open; this library fixes them):
 *  - Layout: Q [B,H,Nq,d], K and V [B,H,Nk,d], O [B,H,Nq,d]: row-major, contiguous,
 *    bf16.  LSE [B,H,Nq]: fp32, natural log of the sum over visible keys of
 *    exp(scale * q . k).
 *  - Mask: key j is visible to query i iff j < L_b (key padding; L_b = key_padding_lens[b]
 *    clamped to [0, Nk], or Nk when key_padding_lens is NULL) and, when causal != 0,
 *    j <= i + (Nk - Nq) (bottom-right aligned; j <= i when Nq == Nk).  Masked scores are
 *    -inf before the block maximum is taken.
 *  - A row with no visible key (fully masked, or Nk == 0) gets O = 0 and LSE = -inf,
 *    never 0/0.
 *  - d must be 64 or 128.  scale must be finite and > 0 (1/sqrt(d) is the usual value).
 *  - Q, K, V and O must be 16-byte aligned (TMA), LSE 4-byte aligned; the library does
 *    not check that they are device pointers.
 *
 * Ownership: the caller owns every buffer.  attn_fwd allocates no device memory per
 * call; the library keeps one small device status word per device, created on first use.
 * Streams: every kernel is launched with programmatic stream serialization, so it may be
 * scheduled while the previous kernel in the stream finishes; it touches no global
 * memory before that kernel has completed and its writes are visible, so stream order
 * holds for every buffer as with a plain launch.
 * Errors: every entry point returns an attn_status; no C++ exception crosses this ABI.
 * attn_last_error() gives a message for the calling thread's last failure.
 */
#ifndef ATTN_H_
#define ATTN_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  ATTN_OK = 0,
  ATTN_ERR_NULLPTR = -1,        /* a required pointer is NULL */
  ATTN_ERR_BAD_SHAPE = -2,      /* negative or too-large B, H, Nq, Nk */
  ATTN_ERR_UNSUPPORTED_D = -3,  /* d not in {64, 128} */
  ATTN_ERR_MISALIGNED = -4,     /* a pointer is not 16-byte aligned */
  ATTN_ERR_NO_DEVICE = -5,      /* no usable sm_103 device / CUDA runtime error at setup */
  ATTN_ERR_LAUNCH = -6,         /* kernel launch or copy failed (message in attn_last_error) */
  ATTN_ERR_TIMEOUT = -7,        /* a bounded device-side wait ran out (see attn_status_sync) */
  ATTN_ERR_BAD_ARG = -8         /* scale not finite or not > 0, or another bad scalar */
} attn_status;

/*
 * attn_fwd -- enqueue the attention forward on `stream`.
 *   Q, K, V   device bf16 inputs (layouts above).  K and V may be NULL when Nk == 0.
 *   O         device bf16 output [B,H,Nq,d];  LSE device fp32 output [B,H,Nq].
 *   B, H, Nq, Nk >= 0; a call with B*H*Nq == 0 does nothing and returns ATTN_OK.
 *   d         64 or 128.     scale   multiplies q . k before the softmax.
 *   causal    0 or nonzero (bottom-right aligned causal mask).
 *   key_padding_lens  device int32[B] or NULL (no padding).
 *   stream    a cudaStream_t, or NULL for the legacy default stream.
 * Asynchronous: returns after the launch.  Argument and launch errors are returned at
 * once; a device-side wait timeout is reported by attn_status_sync.
 * Environment, read at every launch (all entry points):
 *   ATTN_WAIT_LIMIT_MS          limit of each device-side wait in ms (default 2000).
 *   ATTN_TEST_WITHHOLD_K_BLOCK  test hook, honoured only while ATTN_ENABLE_TEST_HOOKS=1 is
 *                               also set: the loader skips key block j (0-based) of every
 *                               tile, so the waits on it run out; the call then reports
 *                               ATTN_ERR_TIMEOUT and O / LSE are not written.
 */
attn_status attn_fwd(const void* Q, const void* K, const void* V, void* O, float* LSE, int B, int H, int Nq,
                     int Nk, int d, float scale, int causal, const int32_t* key_padding_lens, void* stream);

/* Exponential evaluation modes (attn_options.exp2_mode). */
enum {
  ATTN_EXP2_DEFAULT = 0,   /* the library's choice (currently ATTN_EXP2_HARDWARE: measured fastest) */
  ATTN_EXP2_HARDWARE = 1,  /* every exp2 on the MUFU unit (ex2.approx) */
  ATTN_EXP2_MIXED = 2      /* in blocks without a masked key, 1 of every 16 pairs of scores takes
                              a degree-4 polynomial on the FMA pipe (relative error < 3e-6) */
};

/* Per-call choices for attn_fwd_ex.  Set size = sizeof(attn_options); zero the rest for
 * the defaults.  (An addition of this library; the pages fix neither choice.) */
typedef struct attn_options {
  size_t size;
  /* Lazy rescale: the running max m is moved (and l, o~ rescaled) only when a block's max
   * exceeds it by more than tau = this many natural-log units.  0 = the pages' rule
   * (rescale whenever the max rises).  The result is the same in exact arithmetic:
   * softmax is invariant to the reference ("FlashAttention math", "Safe softmax": any
   * constant m).  Range [0, 20].
   * Stability bound ("FlashAttention math", "Proof of numerical stability", restated for
   * a reference that may trail the max by up to tau): every score the recurrence meets
   * is at most m + tau, so every probability p = exp(s - m) <= e^tau (<= 4.9e8 at
   * * tau = 20, well inside the range of bf16 P and of fp32), the running sum
   * l <= Nk * e^tau and |o~| <= Nk * e^tau * max|V| (per column).  The result is finite
   * whenever Nk * e^tau * max|V| < FLT_MAX = 3.4e38 (at tau = 0 this is the plain fp32
   * accumulation bound Nk * max|V|); inputs beyond it may overflow o~ to inf and are
   * excluded.  Example: at tau = 20 and Nk = 2^20 keys, |V| must stay below 6.7e23. */
  float rescale_threshold;
  int exp2_mode;           /* ATTN_EXP2_* */
  /* Keys per block: 0 or 128 (the default), 64 or 192.  64 and 192 are available at
   * d = 128 for the dense layouts (attn_fwd_ex; not packed sequences, not split-KV states)
   * with exp2_mode DEFAULT or HARDWARE: the same recurrence over blocks of another size
   * ("FlashAttention math", "Proof of exactness": blocks of any size give the same result).
   * 192 keeps two score buffers in tensor memory instead of three, 64 three buffers of 64
   * columns and four K/V stages.  Both are measured slower than 128 on GB300; they let a
   * caller check that the result does not depend on the block size.  Any other value is
   * ATTN_ERR_BAD_ARG.  Callers built before this field existed pass a smaller size and get
   * the default. */
  int key_block;
} attn_options;

/*
 * attn_fwd_ex -- attn_fwd with options (opts may be NULL: the defaults, identical to
 * attn_fwd).  Errors: as attn_fwd, plus ATTN_ERR_BAD_ARG for a bad options struct.
 */
attn_status attn_fwd_ex(const void* Q, const void* K, const void* V, void* O, float* LSE, int B, int H, int Nq,
                        int Nk, int d, float scale, int causal, const int32_t* key_padding_lens,
                        const attn_options* opts, void* stream);

/*
 * attn_fwd_strided -- attn_fwd over tensors with any (batch, head, row) strides, e.g.
 * the [B, N, H, d] ("BSHD") layout: strides {N*H*d, d, H*d}.  (The pages fix no layout;
 * an addition of this library.)
 *   q_strides, k_strides, v_strides, o_strides: host int64[3] each, the element strides
 *   of the batch, head and row dimensions; element (b, h, i, x) of Q is at
 *   Q + b*q_strides[0] + h*q_strides[1] + i*q_strides[2] + x (d is contiguous).
 *   Every stride must be a positive multiple of 8 elements (16 bytes, for TMA) below
 *   2^38; the rows of O must not overlap.  LSE stays contiguous [B, H, Nq].
 *   Everything else as attn_fwd.  Errors: as attn_fwd, plus ATTN_ERR_BAD_ARG for a bad
 *   stride and ATTN_ERR_NULLPTR for a NULL stride array.
 */
attn_status attn_fwd_strided(const void* Q, const void* K, const void* V, void* O, float* LSE, int B, int H, int Nq,
                             int Nk, int d, float scale, int causal, const int32_t* key_padding_lens,
                             const int64_t* q_strides, const int64_t* k_strides, const int64_t* v_strides,
                             const int64_t* o_strides, void* stream);

/*
 * attn_fwd_varlen -- attention over B packed sequences of different lengths (an addition
 * of this library; the pages treat one sequence).
 *   Q, O  device bf16 [total_q, H, d]: sequence b is rows cu_seqlens_q[b] ..
 *         cu_seqlens_q[b+1] - 1.  K, V device bf16 [total_k, H, d], rows cu_seqlens_k[b] ..
 *   cu_seqlens_q, cu_seqlens_k  device int32[B + 1], non-decreasing from 0 to total_q /
 *         total_k (values are clamped to [0, total] on the device, so a bad array cannot
 *         make the kernel write outside O and LSE).
 *   max_seqlen_q  >= the longest query sequence (the grid covers that many rows; longer
 *         sequences are left partly unwritten).
 *   LSE   device fp32 [H, total_q].
 *   Masks per sequence: query i of sequence b (Nq_b rows, Nk_b keys) sees key j iff
 *   j < Nk_b and, when causal, j <= i + (Nk_b - Nq_b).  A sequence with no keys gets O = 0
 *   and LSE = -inf.  Asynchronous; timeouts through attn_status_sync.
 */
attn_status attn_fwd_varlen(const void* Q, const void* K, const void* V, void* O, float* LSE,
                            const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k, int B, int H, int max_seqlen_q,
                            int total_q, int total_k, int d, float scale, int causal, void* stream);

/*
 * attn_fwd_host -- the same operation on HOST buffers (pinned memory recommended).
 * Copies Q, K, V (and key_padding_lens, a host int32[B] or NULL) to the device, runs the
 * forward, copies O and LSE back and synchronises `stream` before it returns.  The copies
 * run on two streams of the library's own, overlapped with the forward on `stream`: the
 * heads are cut into chunks (runs of heads of one batch, about 32 MB of input each) and
 * chunk i is computed while chunk i + 1 is copied in and chunk i - 1 copied out.  The
 * work starts after what is already queued on `stream`.  Uses a per-device workspace
 * that grows to the largest problem seen and is kept until attn_release_workspace(); it
 * allocates only when a call needs more room (and creates its two streams once).
 */
attn_status attn_fwd_host(const void* Q, const void* K, const void* V, void* O, float* LSE, int B, int H,
                          int Nq, int Nk, int d, float scale, int causal, const int32_t* key_padding_lens,
                          void* stream);

/* Free the attn_fwd_host workspace of the current device. */
attn_status attn_release_workspace(void);

/* Synchronise `stream`, then read and clear the device status words of the current
 * device (the one the allocating entry points use and, once attn_fwd_noalloc has run
 * on the device, its fixed one): ATTN_ERR_TIMEOUT if a kernel's bounded wait ran out
 * since the last check.  Reads and clears with plain copies; allocates nothing. */
attn_status attn_status_sync(void* stream);

/* Message for the calling thread's last non-OK status ("" if none). */
const char* attn_last_error(void);

/* Library version, major * 10000 + minor * 100 + patch. */
int attn_version(void);

/*
 * attn_fwd_noalloc -- attn_fwd for callers that must not allocate device memory.
 * (An addition of this library; the source pages have no counterpart.)
 *
 * Who needs it: code that runs where cudaMalloc is off limits -- a process whose device
 * memory is handed out by someone else's pool or a fixed budget, a real-time or
 * embedded caller that may not allocate after start-up, or a plugin that must not
 * grow the host application's footprint.  attn_fwd itself allocates a 4-byte status
 * word with cudaMalloc on its first call on each device; this entry point never does.
 *
 * Same arguments and semantics as attn_fwd, plus check_status.  The caller still
 * passes every input and output buffer.  The only device scratch the kernel needs
 * (one 32-bit status word for its bounded waits) lives in a fixed array compiled into
 * the library: 256 bytes per device, held by every GPU that loads the library until
 * the process exits.  A call whose scratch need exceeds that size is rejected with
 * ATTN_ERR_BAD_SHAPE (the forward kernel needs 4 bytes, so today no call is).
 *
 *  - The first call on a device does one-time set-up with that device current: it
 *    looks up the array's device address (cudaGetSymbolAddress), sets the shared-memory
 *    attribute of every kernel this entry point can launch (d = 128, d = 64 with one
 *    and with two query tiles per CTA) and caches the SM count.  Make that first call
 *    before any stream capture.
 *  - Every call shares the array and it keeps the last call's contents.  Its status
 *    word is the OR of every bounded wait that ran out since the word was last read; it
 *    starts at zero and is cleared where it is read: by a call with check_status != 0
 *    and by attn_status_sync.  Calls that overlap on the GPU (different streams, or
 *    several host threads) share that word, so a timeout is reported to whichever of
 *    them reads it first; serialise them if you rely on the attribution.
 *  - check_status == 0: asynchronous, like attn_fwd; a device-side wait that runs out
 *    still ends the kernel, and attn_status_sync (on a stream ordered after the call)
 *    reports it later.  check_status != 0: the call synchronises `stream` and returns
 *    ATTN_ERR_TIMEOUT if a wait ran out since the word was last read.
 *  - It calls no cudaMalloc, cudaFree or other allocating routine, and its kernels use no
 *    local memory (which the driver would back on first launch).  Loading the library's
 *    device code onto a device takes device memory once per process, as for any CUDA
 *    library (the module image, which holds the fixed array): under CUDA's default lazy
 *    module loading that happens at the library's first call on the device, whichever
 *    entry point it is.  A caller whose device memory must not move after start-up makes
 *    one call at start-up (attn_status_sync(NULL) is enough) or sets
 *    CUDA_MODULE_LOADING=EAGER.
 */
attn_status attn_fwd_noalloc(const void* Q, const void* K, const void* V, void* O, float* LSE, int B, int H,
                             int Nq, int Nk, int d, float scale, int causal, const int32_t* key_padding_lens,
                             int check_status, void* stream);

/* ------------------------------------------------------------------------------------
 * Split-KV: the keys of every row are cut into splits, each split is absorbed into its
 * own running state, and the states are merged.
 *
 * A state is the triple the recurrence carries ("FlashAttention math", section "The
 * running state"): m = the largest visible scaled score scale * q . k_j of the split,
 * l = sum exp(s_j - m) and o~ = sum exp(s_j - m) v_j (unnormalised) over the split's
 * visible keys.  A split with no visible key for a row holds the initial state
 * m = -inf, l = 0, o~ = 0.  The pages let keys be absorbed in any order and in blocks of
 * any size (same page, "Proof of exactness"); states of disjoint key sets combine with
 * the rescaling identity (section "The rescaling identity, derived"): with
 * m = max_s m_s, l = sum_s exp(m_s - m) l_s and o~ = sum_s exp(m_s - m) o~_s.
 * This serves shapes with few query tiles and many keys (decoding, short prompts over
 * a long cache), where one CTA per query tile leaves most SMs idle; the same merge is
 * the exchange step of a key-sharded (context-parallel) forward.
 * ------------------------------------------------------------------------------------ */

/*
 * attn_fwd_states -- the partial states of num_splits key splits (1 <= num_splits <= 256).
 *   Split s covers keys [s * C, (s + 1) * C) intersected with [0, Nk), where
 *   C = 128 * ceil(ceil(Nk / 128) / num_splits); masks as for attn_fwd.
 *   Q, K, V, B, H, Nq, Nk, d, scale, causal, key_padding_lens, stream: as attn_fwd.
 *   o_states  device fp32 [num_splits, B, H, Nq, d]: o~.
 *   m_states  device fp32 [num_splits, B, H, Nq]: m (natural-log units; -inf = empty).
 *   l_states  device fp32 [num_splits, B, H, Nq]: l.
 *   All three 16-byte aligned.  Asynchronous; timeouts through attn_status_sync.
 *   Errors: as attn_fwd, plus ATTN_ERR_BAD_ARG for num_splits out of range.
 */
attn_status attn_fwd_states(const void* Q, const void* K, const void* V, float* o_states, float* m_states,
                            float* l_states, int B, int H, int Nq, int Nk, int d, float scale, int causal,
                            const int32_t* key_padding_lens, int num_splits, void* stream);

/*
 * attn_merge_states -- merge num_states >= 1 states per row and finish each row:
 *   O = o~ / l (bf16) and LSE = m + ln l, or O = 0 and LSE = -inf when every state of
 *   the row is empty.  rows = number of rows (B * H * Nq for attn_fwd_states' output).
 *   o_states fp32 [num_states, rows, d] (16-byte aligned), m_states and l_states fp32
 *   [num_states, rows], O bf16 [rows, d] (16-byte aligned), LSE fp32 [rows]; all device.
 *   The states may come from anywhere (another GPU's keys, a previous call).
 *   Asynchronous on `stream`.  Errors: NULLPTR, MISALIGNED, UNSUPPORTED_D, BAD_ARG
 *   (num_states < 1), BAD_SHAPE (rows < 0), LAUNCH.
 */
attn_status attn_merge_states(const float* o_states, const float* m_states, const float* l_states, int num_states,
                              long long rows, int d, void* O, float* LSE, void* stream);

/* Bytes of device workspace attn_fwd_splitkv needs for num_splits splits (0 for
 * invalid arguments): the three state arrays, each rounded up to 256 bytes. */
size_t attn_splitkv_workspace_bytes(int B, int H, int Nq, int d, int num_splits);

/* The split count attn_fwd_splitkv picks when given num_splits <= 0, on the current
 * device: 1 when the query tiles alone fill the SMs, else enough splits to fill them
 * once, at most one split per four key blocks and at most 256. */
int attn_splitkv_splits(int B, int H, int Nq, int Nk);

/*
 * attn_fwd_splitkv -- attn_fwd computed as attn_fwd_states + attn_merge_states.
 *   Same arguments and result as attn_fwd (within the same tolerance, not bitwise),
 *   plus num_splits (<= 0: attn_splitkv_splits' choice) and a caller-owned device
 *   workspace of at least attn_splitkv_workspace_bytes(B, H, Nq, d, splits) bytes,
 *   16-byte aligned.  With one split the call is attn_fwd and the workspace is unused.
 *   No allocation.  Asynchronous; ATTN_ERR_BAD_ARG if the workspace is too small.
 */
attn_status attn_fwd_splitkv(const void* Q, const void* K, const void* V, void* O, float* LSE, int B, int H, int Nq,
                             int Nk, int d, float scale, int causal, const int32_t* key_padding_lens, int num_splits,
                             void* workspace, size_t workspace_bytes, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* ATTN_H_ */
