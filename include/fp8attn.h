/*
 * fp8attn.h -- C ABI of the GB300 (sm_103a) causal prefill attention library
 * (libfp8attn.so).
 *
 * The operation is the causal forward ("prefill") attention with equal query
 * and key lengths that the article "Zyphra ZYFA: FP8 FlashAttention for AMD
 * MI355X, Up to 1.76x Faster" describes in "TL;DR" (causal forward attention in
 * FP8 e4m3 and BF16, head dim 128 and the MLA shape 192/128) and whose limits
 * "Breaking the FP8 Attention Bottleneck on AMD MI355X: How Zyphra ZYFA
 * Unleashes Performance" states in "Application Boundaries and Engineering
 * Decisions" (no decode, no paged KV cache, no variable-length batches):
 *
 *     out[b, i, h, :] = sum_{j <= i} softmax_j(scale * <q~[b,i,h,:], k~[b,j,g,:]>) v~[b,j,g,:]
 *
 * with g = floor(h * Hkv / Hq) (grouped-query head mapping), q~ = dq * q,
 * k~ = dk * k, v~ = dv * v the dequantized inputs and scale = 1/sqrt(Dqk)
 * (attn_fwd_ex / attn_fwd_full take any scale; with causal = 0 the sum runs
 * over all j < S; with ATTN_FLAG_DESCALE_PER_BKV the descales are per (batch,
 * kv head)).
 *
 * Four arithmetic paths compute it (the fourth, a diagnostic, through
 * attn_fwd_ex / attn_fwd_full only):
 *   - attn_fwd_fp8: the Lean-P path.  Each probability is an e4m3 code made by
 *     one multiply-add and an integer conversion ("Lean P: one multiply-add
 *     instead of an exponential"); each 64-key block of probabilities carries
 *     a power-of-two scale that the P.V product removes, and the row is
 *     divided by the sum of the rounded probabilities ("Per-block scaling and
 *     a rounded row sum").
 *   - attn_fwd_fp8_exact: the exact-softmax FP8 ablation (exact exponential,
 *     probabilities rounded to e4m3, row sum of the unrounded probabilities).
 *   - attn_fwd_bf16: exact softmax with BF16 inputs and probabilities.
 *   - ATTN_VARIANT_BLOCK_EXACT: Lean-P's block scale and rounded row sum, with
 *     each probability taken from the exponential unit and rounded to e4m3.
 * attn_quantize_fp8 turns bf16 or fp32 Q or K into the e4m3 codes and the
 * device descale these calls take, optionally after a Hadamard rotation.
 *
 * Layouts (all row-major, contiguous, "BSHD" as in flash_attn_func):
 *   q   [B, S, Hq,  Dqk]    k [B, S, Hkv, Dqk]    v [B, S, Hkv, Dv]
 *   out [B, S, Hq,  Dv]     bf16 (or fp32 through attn_fwd_ex)
 * FP8 inputs are OCP e4m3 bytes; descale_q/k/v point to ONE fp32 each in
 * DEVICE memory (per-tensor descales), so a call can be captured in a CUDA
 * graph.  BF16 inputs are bf16 values.
 *
 * Descales must be finite and greater than zero (a descale is amax/448 of
 * the tensor, 1 for an all-zero tensor).  They live on the device, so the
 * library cannot check them: with a zero, negative or non-finite descale the
 * kernels still run to completion without a fault, but the output (and the
 * LSE) is unspecified.  The Python binding rejects such values where it sees
 * them on the host.
 *
 * Non-finite codes: e4m3 has no infinities; a NaN code (0x7F, 0xFF) in q or k
 * makes that score NaN.  The Lean-P path gives such a key weight 0 (its
 * saturating multiply-add flushes NaN to 0 and the block maximum skips it);
 * the exact paths propagate the NaN to every row that sees the key.  A NaN in
 * v reaches every row whose weight on that key is non-zero.
 *
 * Supported: causal = 0 or 1, (Dqk, Dv) in {(128, 128), (192, 128)} for FP8 and
 * (128, 128) for BF16, any S >= 1, B >= 1, Hq % Hkv == 0.  Base addresses must
 * be 16-byte aligned.  The device must be sm_103 (GB300).
 *
 * Ownership and threading: the caller owns every buffer, including the
 * optional workspace of attn_fwd_full.  The library allocates no device
 * memory and keeps no global mutable state besides a per-device cache of
 * kernel attributes, a cache of split schedules and a call counter; calls on
 * different streams may run concurrently (each with its own workspace).
 * Calls are asynchronous on `stream` (a cudaStream_t, NULL = legacy default
 * stream); argument errors are returned synchronously before anything is
 * launched.
 */
#ifndef FP8ATTN_H
#define FP8ATTN_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

#define FP8ATTN_API_VERSION 9

/* Return codes of every entry point. */
typedef enum {
  ATTN_OK = 0,
  ATTN_ERR_INVALID_ARG = 1, /* null/misaligned pointer, bad size, Hq % Hkv != 0 */
  ATTN_ERR_UNSUPPORTED = 2, /* valid but not implemented: other head dims */
  ATTN_ERR_ARCH = 3,        /* current device is not sm_103 */
  ATTN_ERR_CUDA = 4,        /* a CUDA runtime/driver call failed (launch, tensor map) */
  ATTN_ERR_TIMEOUT = 5      /* a device-side bounded wait expired (see dev_status) */
} attn_status;

/* Arithmetic path selector for attn_fwd_ex. */
typedef enum {
  ATTN_VARIANT_LEANP = 0,     /* FP8 Lean-P (attn_fwd_fp8) */
  ATTN_VARIANT_EXACT_FP8 = 1, /* FP8 exact-softmax ablation (attn_fwd_fp8_exact) */
  ATTN_VARIANT_BF16 = 2,      /* BF16 exact softmax (attn_fwd_bf16) */
  /* FP8 diagnostic: Lean-P's 64-key power-of-two block scale and rounded row
   * sum, with each probability 2^(x/8 - e + T) taken from the exponential
   * unit and rounded to the nearest e4m3 instead of the Lean-P code.  It
   * differs from ATTN_VARIANT_LEANP in the code step alone, which isolates
   * what the one-multiply-add code costs in accuracy and saves in time
   * ("Zyphra ZYFA: FP8 FlashAttention for AMD MI355X", "Lean P" and
   * "Per-block scaling and a rounded row sum"). */
  ATTN_VARIANT_BLOCK_EXACT = 3,
  /* FP8 Lean-P with the code grid anchored at the row's running maximum m:
   * per 64-key block k = floor(lambda*(m - block max)) and the code
   * floor(8*lambda*(s - m) + 8k + 112 + 2^-6), clamped to [0, 126], with the
   * block scale 2^(-7-k); O and the rounded row sum are rescaled exactly by
   * 2^(lambda*(m_old - m_new)) whenever m grows (per 128-key tile).  The key
   * holding the maximum gets exactly the code of 2^7.  ATTN_VARIANT_LEANP
   * anchors the grid at integer log2 values instead (its reference moves only
   * by powers of two).  Both follow "Lean P: one multiply-add instead of an
   * exponential" and "Per-block scaling and a rounded row sum", which leave
   * the anchor of the power-of-two scale open. */
  ATTN_VARIANT_LEANP_A3 = 4
} attn_variant;

/* Output element type for attn_fwd_ex. */
typedef enum { ATTN_OUT_BF16 = 0, ATTN_OUT_F32 = 1 } attn_out_dtype;

/* attn_fwd_ex flags. */
#define ATTN_FLAG_NONE 0
/* Test hook: the load warp issues no copies, so every consumer's bounded wait
 * expires.  The kernel then sets *dev_status to ATTN_ERR_TIMEOUT and returns
 * with its tensor memory released.  Requires dev_status != NULL and uses a
 * short (about 0.2 s) wait limit. */
#define ATTN_FLAG_TEST_STALL_LOADS 1
/* The three descales hold B*Hkv values each, [B, Hkv] row-major: the Q heads
 * of kv head g in batch b use entry b*Hkv + g (the per-(batch, kv head)
 * descales of FP8 flash_attn_func); without the flag, one value each. */
#define ATTN_FLAG_DESCALE_PER_BKV 2
/* Test hook: run the work items in chunks of one (batch, kv head) each, the
 * order the library otherwise chooses only for problems whose K and V exceed
 * 256 MB (to keep the kv heads in flight inside L2).  The item order changes
 * no arithmetic, so the result is bitwise the same as without the flag. */
#define ATTN_FLAG_TEST_CHUNK_UNITS 4

/*
 * FP8 Lean-P causal prefill attention ("Lean P: one multiply-add instead of an
 * exponential", "Per-block scaling and a rounded row sum").
 *   q, k, v      device pointers to e4m3 bytes in the layouts above
 *   descale_*    device pointers to one fp32 each
 *   out          device pointer, bf16 [B, S, Hq, Dv]
 *   causal       1 (row i sees keys 0 .. i) or 0 (all keys)
 *   stream       cudaStream_t or NULL
 * Returns an attn_status.  A device-side wait expiry cannot be reported here
 * (nothing is read back); use attn_fwd_ex with dev_status to observe it.
 */
int attn_fwd_fp8(const void* q, const void* k, const void* v, const float* descale_q,
                 const float* descale_k, const float* descale_v, void* out, int B, int Hq,
                 int Hkv, int S, int Dqk, int Dv, int causal, void* stream);

/* FP8 exact-softmax ablation: p = 2^(log2(e) * (z - m)) from the hardware
 * exponential with a running max m per 128-key tile, P rounded to e4m3
 * (nearest even), row sum over the unrounded p (the "hardware exponential"
 * approach in the comparison table of "Zyphra ZYFA: FP8 FlashAttention for AMD
 * MI355X").  Arguments as attn_fwd_fp8. */
int attn_fwd_fp8_exact(const void* q, const void* k, const void* v, const float* descale_q,
                       const float* descale_k, const float* descale_v, void* out, int B,
                       int Hq, int Hkv, int S, int Dqk, int Dv, int causal, void* stream);

/* BF16 exact-softmax causal prefill attention ("TL;DR": BF16 kernels beside
 * the FP8 ones).  q, k, v, out are bf16 device pointers; Dqk = Dv = 128. */
int attn_fwd_bf16(const void* q, const void* k, const void* v, void* out, int B, int Hq, int Hkv,
                  int S, int Dqk, int Dv, int causal, void* stream);

/*
 * Extended entry point used by the tests and the benchmark.
 *   variant        attn_variant
 *   descale_*      device fp32 pointers (ignored for ATTN_VARIANT_BF16)
 *   out_dtype      attn_out_dtype; ATTN_OUT_F32 writes fp32 [B, S, Hq, Dv]
 *   softmax_scale  <= 0 selects 1/sqrt(Dqk)
 *   flags          ATTN_FLAG_* bits
 *   dev_status     NULL, or a device int the CALLER zeroes before the call;
 *                  the kernel stores ATTN_ERR_TIMEOUT there if a bounded wait
 *                  expired (the output is then undefined).  Read it after the
 *                  stream has synchronised.
 */
int attn_fwd_ex(int variant, const void* q, const void* k, const void* v, const float* descale_q,
                const float* descale_k, const float* descale_v, void* out, int out_dtype, int B,
                int Hq, int Hkv, int S, int Dqk, int Dv, int causal, float softmax_scale,
                int flags, int* dev_status, void* stream);

/* Static description of a status code (never NULL). */
const char* attn_status_string(int status);

/* Number of kernel launches one call makes (1 for every supported shape;
 * 0 when S == 0 or B == 0 is rejected).  Lets callers count launches. */
int attn_launches_per_call(void);

/*
 * The general entry point: attn_fwd_ex plus an optional log-sum-exp output,
 * for drop-in use behind a flash_attn_func-style interface ("Zyphra ZYFA: FP8
 * FlashAttention for AMD MI355X", "TL;DR").
 *   causal     1: row i sees keys 0 .. i; 0: every row sees all S keys
 *   flags      ATTN_FLAG_DESCALE_PER_BKV for [B, Hkv] descales (FP8 only);
 *              ATTN_FLAG_TEST_STALL_LOADS, ATTN_FLAG_TEST_CHUNK_UNITS as for
 *              attn_fwd_ex
 *   lse        NULL, or a device pointer to fp32 [B, Hq, S] (4-byte aligned):
 *              lse[b,h,i] = ln sum_j w_ij, the natural log of the row's own
 *              unnormalised weights (Lean-P: the rounded, scaled weights whose
 *              sum divides the output; exact paths: exp(z_ij) before rounding),
 *              z_ij = softmax_scale * descale_q * descale_k * <q_i, k_j>
 *   workspace, workspace_bytes
 *              NULL (and 0), or device memory of at least the size that
 *              attn_workspace_size reports for the same arguments, 256-byte
 *              aligned, owned by the caller and used by one call at a time
 *              (calls that overlap on the GPU need workspaces of their own).
 *              With it, problems with too few work items to fill every SM
 *              (few heads, short sequences) split their longest items along
 *              the keys into pieces that run on different SMs and are added up
 *              by the piece that finishes last, in a fixed order, so the result
 *              is the same on every call.  ATTN_VARIANT_LEANP and
 *              ATTN_VARIANT_BLOCK_EXACT: the codes depend on each 64-key block
 *              alone, so a split changes only the order of the fp32 sums.
 *              ATTN_VARIANT_BF16: each piece rounds its probabilities to bf16
 *              relative to its own running maximum, so a split result differs
 *              from whole items within the rounding of bf16.  The other
 *              variants always run whole items.  The memory needs no clearing: it holds
 *              partial results and counters tagged with a per-call number.
 *              Too small a workspace is an ATTN_ERR_INVALID_ARG; NULL runs
 *              every item whole, as attn_fwd_ex does.
 * Other arguments as attn_fwd_ex.  Returns an attn_status.
 */
int attn_fwd_full(int variant, const void* q, const void* k, const void* v,
                  const float* descale_q, const float* descale_k, const float* descale_v,
                  void* out, int out_dtype, float* lse, int B, int Hq, int Hkv, int S, int Dqk,
                  int Dv, int causal, float softmax_scale, int flags, int* dev_status,
                  void* workspace, size_t workspace_bytes, void* stream);

/*
 * Bytes of workspace attn_fwd_full uses for these arguments on the CURRENT
 * device (its SM count enters the schedule): 0 when the problem runs without
 * splitting (enough work items, a variant that does not split, or
 * ATTN_FLAG_TEST_CHUNK_UNITS), otherwise at most 128 MiB.  The split
 * schedule is chosen by a model of the kernel's time per key tile and per
 * work unit; it is cached per shape.  Returns an attn_status; *bytes is 0 on
 * error.
 */
int attn_workspace_size(int variant, int B, int Hq, int Hkv, int S, int Dqk, int Dv, int causal,
                        int flags, size_t* bytes);

/*
 * The split schedule that attn_fwd_full would choose for these arguments on
 * a GPU with `sms` SMs (>= 1), computed on the host without touching any
 * device: the items of query blocks >= *split_qb (256 query rows each) run
 * in *ns pieces, with *bytes of workspace; *ns = 1, *split_qb = 0 and
 * *bytes = 0 when the problem runs whole items.  For capacity planning and
 * for testing the schedule's choices.  This query has no counterpart in the
 * articles, and neither has the split schedule it describes.  Returns an
 * attn_status (ATTN_ERR_INVALID_ARG for invalid arguments, a NULL output
 * pointer or sms < 1); on error the non-NULL outputs hold the no-split
 * values.
 */
int attn_split_plan(int variant, int B, int Hq, int Hkv, int S, int Dqk, int Dv, int causal,
                    int flags, int sms, int* split_qb, int* ns, size_t* bytes);

/* Input element type for attn_quantize_fp8. */
typedef enum { ATTN_IN_BF16 = 0, ATTN_IN_F32 = 1 } attn_in_dtype;

/*
 * Per-tensor e4m3 quantisation of Q or K for attn_fwd_fp8, optionally after a
 * Hadamard rotation of every head vector ("Zyphra ZYFA: FP8 FlashAttention for
 * AMD MI355X", "How accurate is ZYFA's FP8 attention?": most FP8 error comes
 * from quantising the inputs, and rotating Q and K roughly halves it).  Q and
 * K must be rotated alike (both or neither): Q K^T is unchanged by a common
 * orthogonal rotation, V is never rotated.
 *   x          device pointer, [B, S, H, D] bf16 or fp32 (in_dtype), 16-byte
 *              aligned; finite values
 *   codes      device pointer, e4m3 [B, S, H, D], 16-byte aligned (written)
 *   descale    device pointer to one fp32 (written): dec(code) * descale
 *              approximates x (rotated: its orthonormal rotation)
 *   D          128 or 192
 *   hadamard   0: no rotation.  1: unnormalised Walsh-Hadamard transform of
 *              each head vector, in one block of 128 (D = 128) or in three
 *              blocks of 64 (D = 192); the normalisation 1/sqrt(block) goes
 *              into descale
 * Arithmetic (fp32 throughout): y = x or its transform (butterfly stages
 * h = 1, 2, 4, ...; pair (i, i+h) -> (y_i + y_{i+h}, y_i - y_{i+h})),
 * amax = max|y|, code = e4m3 round-to-nearest-even(y * 448/amax), saturated;
 * descale = (amax/448) * norm (amax = 0: norm).  Three kernel launches and one
 * 4-byte memset on `stream`; the descale word holds amax between them, so no
 * other memory is used.  Returns an attn_status.
 */
int attn_quantize_fp8(const void* x, int in_dtype, void* codes, float* descale, int B, int S,
                      int H, int D, int hadamard, void* stream);

/* Bytes of device scratch that attn_fwd_fp8_noalloc holds (32 MiB). */
#define ATTN_NOALLOC_SCRATCH_BYTES (32u * 1024u * 1024u)

/*
 * attn_fwd_fp8 for callers that cannot allocate device memory, with the split
 * schedule of attn_fwd_full.  (The articles have no counterpart: this is an
 * interface for callers of this library.)  Some callers may not call
 * cudaMalloc: a framework or runtime that owns every device allocation
 * through its own allocator, a serving loop that allows no allocation after
 * start-up (an allocation can synchronise the device and stall the other
 * streams), or code with a fixed memory budget.  They pass inputs and
 * outputs as for attn_fwd_fp8 (same arguments, same result as attn_fwd_full
 * with a workspace), and the scratch that the split schedule needs comes from
 * a file-scope device array of ATTN_NOALLOC_SCRATCH_BYTES inside the library,
 * which every GPU that loads the library holds until the process exits.
 * Nothing is allocated: no cudaMalloc, cudaFree or allocating library call.
 *   - The first call on each device looks up the array's device address
 *     (cudaGetSymbolAddress, with that device current); make that first call
 *     before any stream capture.
 *   - Every call shares the array, which keeps the last call's contents;
 *     nothing in it needs clearing (the schedule tags its counters per call).
 *     Calls that overlap on the GPU (on different streams) race on the array
 *     and give wrong results: order them on one stream.
 *   - A problem whose split schedule needs more than ATTN_NOALLOC_SCRATCH_BYTES
 *     (attn_workspace_size reports the size) is rejected with
 *     ATTN_ERR_UNSUPPORTED before anything is launched.
 * Returns an attn_status.
 */
int attn_fwd_fp8_noalloc(const void* q, const void* k, const void* v, const float* descale_q,
                         const float* descale_k, const float* descale_v, void* out, int B, int Hq,
                         int Hkv, int S, int Dqk, int Dv, int causal, void* stream);

/* Library ABI version (FP8ATTN_API_VERSION of the build). */
int attn_api_version(void);

/* Debug timeline (only in the debug library built with FA8_TIMELINE; the
 * release library returns ATTN_ERR_UNSUPPORTED without touching the device).
 * Copies the clock64 stamps that CTA 0 recorded into
 * host[0 .. min(capacity, 3072)), as [6][64][8] unsigned 64-bit values.  Its
 * first work item, per key tile j:
 *   [t][j][0..4]   softmax of query tile t, key tile j: before the wait for S,
 *                  S ready, S copied out (arrived), codes computed, P stored
 *   [2+t][j][0..2] P.V issuer for tile t: before the wait for P, P ready, P.V
 *                  issued;  [2+t][j][3..5] S issuer for tile t: before the
 *                  wait for S to be free, S free, S product issued
 * Every item (round r of CTA 0), at its boundaries:
 *   [4][r][0..6]   Q load issued, first K load issued, Q ready for the S
 *                  issuer, first S product issued, last S product issued,
 *                  first P.V product issued, last P.V product issued
 *   [5][r][4t+0..3] softmax of tile t: first S ready, last P.V complete
 *                  (epilogue start), O released, output stored
 * Unwritten entries are 0 (after a reset) or hold older launches' stamps.
 * With reset != 0 the device copy is zeroed afterwards.  Synchronous with
 * respect to the device; for profiling, not for production calls. */
int attn_debug_timeline(unsigned long long* host, int capacity, int reset);

#ifdef __cplusplus
}
#endif

#endif /* FP8ATTN_H */
