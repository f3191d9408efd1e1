/*
 * attnfuse — fused RoPE + variant attention for NVIDIA GB300 (sm_103a). C ABI.
 *
 * The operation is the one described in "AttnFuse: A Composable DSL for Compiling Attentions
 * to Fused GPU Kernels" (arXiv 2609.13612): rotary position embedding applied to Q and K tiles
 * on-chip (§4.1, NeoX half-split pairs (i, i+d/2)), score combinators applied to score tiles
 * (§3.1: scaled_dot_product, causal, sliding_window, full, block_sparse, alibi, additive_bias,
 * softmax), an online-softmax accumulation into O and the per-row log-sum-exp (§2, §4.4), the
 * three-kernel backward (§4.4), and split-KV decoding (§4.2).
 *
 * Definitions used by every call (0-based positions; query row m sits at position m, key n at
 * position n; decode query at q_pos):
 *   theta_i   = rope_theta^(-2i/d), i < d/2;  R_p rotates pair (x_i, x_{i+d/2}) by p*theta_i
 *   s_mn      = scale * <R_m q_m, R_n k_n>  [+ slope_h * (n - m)]  [+ bias(b, h, m, n)]
 *   allowed   = FULL: all; CAUSAL: n <= m; WINDOW: |m - n| < W (and n <= m if causal);
 *               BLOCK_SPARSE: (m / blk, n / blk) in the CSR layout (and n <= m if causal)
 *   LSE_m     = ln sum_{allowed n} exp(s_mn)        (natural log; -inf if no n is allowed)
 *   O_m       = sum_{allowed n} exp(s_mn - LSE_m) v_n              (0 if no n is allowed)
 *   GQA: query head h reads key/value head h / (Hq / Hkv).
 *
 * Conventions:
 *   - Every function returns an attnfuse_status and never throws or exits. On error,
 *     attnfuse_last_error() returns a thread-local message.
 *   - Every launch is asynchronous on the caller's stream. The library never allocates or
 *     frees device memory: the caller owns every pointer, including the workspace, whose size
 *     the *_workspace_size functions report.
 *   - Q, K, V, O, dO, dQ, dK, dV are bf16 with element strides (b, h, n, c); the last stride
 *     must be 1, the other strides multiples of 8 elements, pointers 16-byte aligned.
 *   - LSE tensors are fp32 contiguous [B, Hq, N] (decode: [B, Hq]).
 *   - Supported head dims: d in {64, 128}. Hq % Hkv == 0.
 *   - Kernels give up on any internal wait after a bounded time instead of hanging; the
 *     device status word then reads ATTNFUSE_ERR_TIMEOUT (see attnfuse_device_status).
 *   - The library looks up its device-side words (status word, decode scratch) once per device
 *     and keeps their addresses for the life of the process: it must not be used on a device
 *     after a cudaDeviceReset of that device.
 */
#ifndef ATTNFUSE_H_
#define ATTNFUSE_H_

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef int attnfuse_status;
#define ATTNFUSE_OK 0
#define ATTNFUSE_ERR_INVALID_ARG 1
#define ATTNFUSE_ERR_UNSUPPORTED 2
#define ATTNFUSE_ERR_WORKSPACE_TOO_SMALL 3
#define ATTNFUSE_ERR_CUDA 4
#define ATTNFUSE_ERR_TIMEOUT 5
#define ATTNFUSE_ERR_FP16_RANGE 6 /* device status: a rotated Q' / K' value saturated fp16 */

/* Where RoPE is applied (paper §4.1 "Fused RoPE" vs. the pre-rotation of Fig. 1a / §5.3).
 * In both rotating modes the rotation runs in fp32 and the rotated Q', K' are rounded to fp16
 * (not bf16) before the score MMA: fp16 keeps 3 more mantissa bits, which keeps the LSE within
 * 1e-3 of the exact value. fp16 saturates at +-65504, so these modes need |q|, |k| < 46000
 * (a rotation can grow one component by sqrt(2)); a call that saturates (or meets a
 * non-finite input) still completes, and sets ATTNFUSE_ERR_FP16_RANGE in the device status
 * word (attnfuse_device_status). ROPE_NONE feeds bf16 inputs unchanged. */
typedef enum {
  ATTNFUSE_ROPE_NONE = 0,      /* no rotation: plain scaled_dot_product */
  ATTNFUSE_ROPE_FUSED = 1,     /* rotate in the attention kernel: each Q tile once, in
                                  shared memory, as it lands (no Q' round trip). K: one pass
                                  writes K' to the workspace just before the forward (K is 1/g
                                  of Q's size); on the head-dim-64 one-CTA forward (one query
                                  head per KV head, N < 8192) the forward rotates each K tile
                                  once per call into a workspace copy shared through L2 (long
                                  sequences) or per CTA in shared memory (short ones) */
  ATTNFUSE_ROPE_PREROTATE = 2, /* separate rotate kernel writes Q', K' to the workspace, then
                                  attention runs without rotation (the paper's baseline) */
  ATTNFUSE_ROPE_AUTO = 3       /* the faster of FUSED and PREROTATE for this call's N, head dim
                                  and direction, by the crossover N* measured on GB300 (the
                                  paper's Rotation Calculus, §5.3); see attnfuse_rope_auto_mode.
                                  The result is identical to the mode chosen. Decode: FUSED. */
} attnfuse_rope_mode;

/* Flag OR-ed into rope_mode: the workspace already holds the (cos, sin) table, built by an
 * earlier call on the same workspace (or by attnfuse_rope_table) for the same d and rope_theta
 * and for at least N positions, so the call skips rebuilding it. The table depends on
 * positions only, so a caller reusing one workspace across layers or steps can build it once. */
#define ATTNFUSE_ROPE_REUSE_TABLE 0x100

/* Mask combinators (paper §3.1 causal / sliding_window / full / block_sparse). */
typedef enum {
  ATTNFUSE_MASK_FULL = 0,
  ATTNFUSE_MASK_CAUSAL = 1,
  ATTNFUSE_MASK_WINDOW = 2,
  ATTNFUSE_MASK_BLOCK_SPARSE = 3
} attnfuse_mask_kind;

/* Bias combinators (paper §3.1 alibi / additive_bias). */
typedef enum {
  ATTNFUSE_BIAS_NONE = 0,
  ATTNFUSE_BIAS_ALIBI = 1,
  ATTNFUSE_BIAS_ADDITIVE = 2
} attnfuse_bias_kind;

/* Normaliser combinators (paper §3.1 softmax / relu_attention). The pages name relu_attention
 * without defining it; this library reads it as ReLU attention divided by the sequence length:
 *   O_m = (1/N) sum_{allowed n} max(s_mn, 0) v_n.
 * It has no log-sum-exp (lse must be NULL) and no backward (attnfuse_bwd returns
 * ATTNFUSE_ERR_UNSUPPORTED); the forward supports it for head dims 64 and 128 with every mask,
 * bias and rope mode. */
typedef enum {
  ATTNFUSE_NORM_SOFTMAX = 0,
  ATTNFUSE_NORM_RELU = 1
} attnfuse_normalizer;

/* A variant: one mask combinator, an optional causal restriction, one bias combinator and the
 * row normaliser.
 * All pointers are device pointers owned by the caller; unused fields are ignored. */
typedef struct {
  int32_t mask;                /* attnfuse_mask_kind */
  int32_t causal;              /* non-zero: also require n <= m (WINDOW, BLOCK_SPARSE, FULL) */
  int32_t window;              /* W >= 1 for ATTNFUSE_MASK_WINDOW */
  int32_t bs_block;            /* block edge for BLOCK_SPARSE: 64 or 128 */
  const int32_t* bs_row_ptr;   /* CSR block layout (paper §4.3 BlockMask): [ceil(N/blk) + 1] */
  const int32_t* bs_col_idx;   /* active block columns per block row, any order, no repeats */
  int32_t bias;                /* attnfuse_bias_kind */
  int32_t add_bias_is_bf16;    /* additive bias element type: 1 = bf16, 0 = fp32 */
  const float* alibi_slopes;   /* [Hq] fp32, required for ATTNFUSE_BIAS_ALIBI */
  const void* add_bias;        /* additive bias, element (b, h, m, n) at add_bias_strides */
  int64_t add_bias_strides[4]; /* element strides; 0 broadcasts that dimension */
  uint8_t* tile_visits;        /* debug, nullable: [B, Hq, ceil(N/128), ceil(N/128)] bytes; the
                                  forward writes 1 for every (q-tile, kv-tile) it computes.
                                  The caller zeroes it first. */
  float* dbias;                /* backward output, nullable, ATTNFUSE_BIAS_ADDITIVE only: the
                                  gradient of the loss with respect to bias(b, h, m, n), i.e.
                                  dS_mn = P_mn (dP_mn - D_m), fp32, one element per (b, h, m, n)
                                  of [B, Hq, N, N] (no broadcast: sum over the dimensions the
                                  bias broadcasts to obtain its own gradient). Every element is
                                  written, 0 where (m, n) is masked. 4-byte aligned. */
  int64_t dbias_strides[4];    /* element strides of dbias: (b, h, m) any, n == 1 */
  int32_t normalizer;          /* attnfuse_normalizer: the row normaliser (0 = softmax) */
  uint8_t* bwd_dq_visits;      /* debug, nullable: [B, Hq, ceil(N/128), ceil(N/128)] bytes; the
                                  backward's dQ kernel writes 1 for every (query tile, key tile)
                                  it computes. The caller zeroes it first. */
  uint8_t* bwd_dkdv_visits;    /* debug, nullable: [B, Hq, ceil(N/64), ceil(N/128)] bytes; the
                                  dK/dV kernel writes 1 for every (64-row query block of head h,
                                  key tile) it computes. The caller zeroes it first. */
} attnfuse_variant;

/* Last error message of this thread (empty string if none). */
const char* attnfuse_last_error(void);

/* Library version as 10000*major + 100*minor + patch. */
int attnfuse_version(void);

/* Synchronise `stream`, then read (and if `clear`, reset) the device status word of the
 * current device: ATTNFUSE_OK; ATTNFUSE_ERR_TIMEOUT if a kernel gave up waiting; else
 * ATTNFUSE_ERR_FP16_RANGE if a forward in a rotating mode (FUSED or PREROTATE) produced a
 * rotated Q' or K' element of magnitude >= 65504 or not finite: the fp16 operand saturated
 * (or the input was not finite) and that call's scores are not to be trusted. */
attnfuse_status attnfuse_device_status(cudaStream_t stream, int clear, int* code);

/* ------------------------------------------------------------------------------------------
 * Forward (paper §4.1 fused RoPE, §2 online softmax, §3.1 combinators, §4.3 block skipping).
 * q: [B, Hq, N, d]; k, v: [B, Hkv, N, d]; out: [B, Hq, N, d]; lse: [B, Hq, N] or NULL.
 * variant: NULL means causal with no bias. Fully masked (q-tile, kv-tile) pairs are skipped.
 * ------------------------------------------------------------------------------------------ */
/* Workspace: NONE none; FUSED the (cos, sin) table, the rotated keys (fp16, B*Hkv*N*d*2
 * bytes) and one 32-bit flag per 64 keys (zeroed by every call with cudaMemsetAsync on
 * `stream`); PREROTATE the table, Q' and K'. */
attnfuse_status attnfuse_fwd_workspace_size(int B, int Hq, int Hkv, int N, int d,
                                            attnfuse_rope_mode rope_mode, size_t* bytes);

attnfuse_status attnfuse_fwd(const void* q, const int64_t q_strides[4], const void* k,
                             const int64_t k_strides[4], const void* v,
                             const int64_t v_strides[4], void* out, const int64_t o_strides[4],
                             float* lse, int B, int Hq, int Hkv, int N, int d, float scale,
                             float rope_theta, attnfuse_rope_mode rope_mode,
                             const attnfuse_variant* variant, void* workspace,
                             size_t workspace_bytes, cudaStream_t stream);

/* ------------------------------------------------------------------------------------------
 * Forward on host buffers. q, k, v, out and lse (lse may be NULL) are host pointers to
 * contiguous [B, H, N, d] bf16 arrays (lse: [B, Hq, N] fp32); page-locked memory (cudaHostAlloc
 * or cudaHostRegister) lets the copies run asynchronously. The batch is processed in chunks of
 * chunk_b elements through two device buffer sets, so the copy-in of chunk c+1, the forward of
 * chunk c and the copy-out of chunk c-1 overlap: the copies run on two streams the library
 * creates once per device, the forwards on `stream`, ordered by events. The call returns after
 * queueing; the results are in out / lse once `stream` has reached this point (the copy-ins
 * start after the work queued on `stream` before the call). Other arguments as attnfuse_fwd
 * (no ATTNFUSE_ROPE_REUSE_TABLE: the first chunk builds the table, the others reuse it). With
 * chunk_b = 1 and fewer than 8 batch elements, each element is further split into groups of
 * KV heads (with their query heads), halving while Hkv allows, until there are 8 chunks: the
 * work that cannot overlap (the first copy-in, the last forward and copy-out) shrinks with
 * the chunk. The variant's device arrays are indexed per chunk: an additive bias, the ALiBi
 * slopes and tile_visits are offset by the chunk's first batch element and head. workspace:
 * device memory of
 * attnfuse_fwd_host_workspace_size bytes (two chunk buffer sets and one forward workspace).
 * Calls on one device are serialised by a lock while they queue work.
 * ------------------------------------------------------------------------------------------ */
attnfuse_status attnfuse_fwd_host_workspace_size(int B, int Hq, int Hkv, int N, int d,
                                                 attnfuse_rope_mode rope_mode, int chunk_b,
                                                 size_t* bytes);

attnfuse_status attnfuse_fwd_host(const void* q, const void* k, const void* v, void* out,
                                  float* lse, int B, int Hq, int Hkv, int N, int d, float scale,
                                  float rope_theta, attnfuse_rope_mode rope_mode,
                                  const attnfuse_variant* variant, int chunk_b, void* workspace,
                                  size_t workspace_bytes, cudaStream_t stream);

/* ------------------------------------------------------------------------------------------
 * e4m3 (fp8) forward (paper §9.1 future work: low-precision attention), head dim 128.
 * q: [B, Hq, N, 128], k, v: [B, Hkv, N, 128], all e4m3 (OCP FP8 E4M3: 1 sign, 4 exponent bits
 * with bias 7, 3 mantissa bits, no infinities; S.1111.111 is NaN), one byte per element,
 * element strides multiples of 16, innermost stride 1, 16-byte aligned. The values the call
 * attends over are q_scale * q, k_scale * k and v_scale * v (per-tensor dequantisation scales,
 * positive and finite); out (bf16) and lse (fp32, or NULL) are as in attnfuse_fwd.
 * The scores S = Q K^T run on tcgen05 kind::f8f6f4 MMAs (exact products, fp32 accumulation);
 * q_scale * k_scale * scale is applied with the softmax scale. V is widened to bf16 (exact)
 * by one pass into the workspace before the forward, and P V runs as in the bf16 forward;
 * v_scale multiplies O. No RoPE: q and k are used as given (a caller with rotary positions
 * quantises the rotated tensors). variant: as attnfuse_fwd (all masks, ALiBi, additive bias,
 * both normalisers). Workspace: attnfuse_fwd_fp8_workspace_size bytes (the widened V,
 * B*Hkv*N*256 bytes).
 * Errors: ATTNFUSE_ERR_UNSUPPORTED for d != 128; ATTNFUSE_ERR_INVALID_ARG for bad pointers,
 * strides or scales; ATTNFUSE_ERR_WORKSPACE_TOO_SMALL.
 * ------------------------------------------------------------------------------------------ */
attnfuse_status attnfuse_fwd_fp8_workspace_size(int B, int Hq, int Hkv, int N, int d,
                                                size_t* bytes);

attnfuse_status attnfuse_fwd_fp8(const void* q, const int64_t q_strides[4], const void* k,
                                 const int64_t k_strides[4], const void* v,
                                 const int64_t v_strides[4], void* out, const int64_t o_strides[4],
                                 float* lse, int B, int Hq, int Hkv, int N, int d, float scale,
                                 float q_scale, float k_scale, float v_scale,
                                 const attnfuse_variant* variant, void* workspace,
                                 size_t workspace_bytes, cudaStream_t stream);

/* ------------------------------------------------------------------------------------------
 * Backward (paper §4.4): preprocess D = rowsum(dO * O), a dK/dV kernel and a dQ kernel, no
 * atomics. Gradients are with respect to the un-rotated q and k (the inverse rotation is
 * applied in the epilogues) and dk, dv are summed over each GQA group.
 * out and lse are the forward's outputs, computed with the same variant. Every variant of
 * the forward is supported (paper §4.3: both passes visit only the active tiles): causal,
 * sliding window, block-sparse (the dK/dV kernel reads the CSR layout transposed), ALiBi and
 * the additive bias, whose gradient is written to variant->dbias when that is non-NULL.
 * ROPE_PREROTATE rotates Q and K once into the workspace, ROPE_FUSED on chip; both give
 * bit-identical gradients. The recomputed scores use bf16-rounded rotated operands; workspace
 * holds the (cos, sin) table (rotating modes), D and, for ROPE_PREROTATE, Q' and K'.
 * ------------------------------------------------------------------------------------------ */
attnfuse_status attnfuse_bwd_workspace_size(int B, int Hq, int Hkv, int N, int d,
                                            attnfuse_rope_mode rope_mode, size_t* bytes);

attnfuse_status attnfuse_bwd(const void* q, const int64_t q_strides[4], const void* k,
                             const int64_t k_strides[4], const void* v,
                             const int64_t v_strides[4], const void* out,
                             const int64_t o_strides[4], const float* lse, const void* dout,
                             const int64_t do_strides[4], void* dq, const int64_t dq_strides[4],
                             void* dk, const int64_t dk_strides[4], void* dv,
                             const int64_t dv_strides[4], int B, int Hq, int Hkv, int N, int d,
                             float scale, float rope_theta, attnfuse_rope_mode rope_mode,
                             const attnfuse_variant* variant, void* workspace,
                             size_t workspace_bytes, cudaStream_t stream);

/* ------------------------------------------------------------------------------------------
 * Split-KV decode (paper §4.2): one query row per (b, h) at position q_pos against a cache of
 * L keys stored already rotated. Phase 1 computes partial (max, sum, acc) per KV chunk, phase
 * 2 merges the chunks through their log-sum-exp. rope_mode applies to q only (NONE or FUSED).
 * q: [B, Hq, d] (strides b, h, c); k_cache, v_cache: [B, Hkv, L, d]; out: [B, Hq, d];
 * lse: [B, Hq] or NULL. num_splits: number of KV chunks per (b, kv-head), 0 = automatic
 * (about two resident CTAs per SM); chunks are whole 128-key tiles, so fewer chunks than
 * requested are used when L / 128 < num_splits, and at most 512 are used. Requires Hq / Hkv <= 32. The q rotation
 * (FUSED) is rounded to bf16, the element type of the cache.
 * ------------------------------------------------------------------------------------------ */
attnfuse_status attnfuse_decode_workspace_size(int B, int Hq, int Hkv, int L, int d,
                                               int num_splits, size_t* bytes);

attnfuse_status attnfuse_decode(const void* q, const int64_t q_strides[3], const void* k_cache,
                                const int64_t k_strides[4], const void* v_cache,
                                const int64_t v_strides[4], void* out,
                                const int64_t o_strides[3], float* lse, int B, int Hq, int Hkv,
                                int L, int d, int q_pos, float scale, float rope_theta,
                                attnfuse_rope_mode rope_mode, int num_splits, void* workspace,
                                size_t workspace_bytes, cudaStream_t stream);

/* attnfuse_decode for callers that cannot allocate device memory. (The paper has no
 * counterpart; this is an interface choice of this library.)
 * Some callers have no way to provide a device workspace: a serving runtime whose device memory
 * is entirely pre-reserved by its own allocator, a host program without an allocator of its
 * own to hand out scratch buffers, or a latency-critical path where a cudaMalloc (which may
 * synchronise the device) is not allowed. This entry point takes the same arguments as
 * attnfuse_decode minus the workspace and keeps the split-KV partial results in one fixed
 * 4 MiB array compiled into the library (each GPU that loads the library holds it until the
 * process exits). It allocates and frees nothing; the caller still passes q, the caches, out
 * and lse.
 *   - Problems whose partials need more than 4 MiB (attnfuse_decode_workspace_size) are
 *     rejected with ATTNFUSE_ERR_WORKSPACE_TOO_SMALL and a message naming both sizes.
 *   - The first call on a device looks up the array's device address (cudaGetSymbolAddress)
 *     with that device current; make that first call before any stream capture. The address
 *     is kept for the life of the process: after a cudaDeviceReset of that device the array
 *     is reloaded elsewhere, so do not call this entry point on a device that was reset.
 *   - All calls share the array, which keeps the last call's contents (every value a call
 *     reads is written by that same call first). Calls that overlap on the GPU, on one or
 *     several streams, race on the array and must be serialised by the caller. */
attnfuse_status attnfuse_decode_noalloc(const void* q, const int64_t q_strides[3],
                                        const void* k_cache, const int64_t k_strides[4],
                                        const void* v_cache, const int64_t v_strides[4], void* out,
                                        const int64_t o_strides[3], float* lse, int B, int Hq,
                                        int Hkv, int L, int d, int q_pos, float scale,
                                        float rope_theta, attnfuse_rope_mode rope_mode,
                                        int num_splits, cudaStream_t stream);

/* Number of KV chunks attnfuse_decode uses for num_splits = 0 on the current device. */
attnfuse_status attnfuse_decode_auto_splits(int B, int Hkv, int L, int* num_splits);

/* ------------------------------------------------------------------------------------------
 * Pre-rotation alone (paper Fig. 1a / §5.3 T_pre): x_rot = R_n x for x of shape [B, H, N, d]
 * (row n at position n), written contiguously to `out`. Used by ATTNFUSE_ROPE_PREROTATE and
 * exposed for the fused-vs-pre-rotated crossover measurement. workspace holds the cos/sin
 * table: attnfuse_fwd_workspace_size(.., ATTNFUSE_ROPE_FUSED, ..) bytes.
 * ------------------------------------------------------------------------------------------ */
attnfuse_status attnfuse_rope_prerotate(const void* x, const int64_t x_strides[4], void* out,
                                        int B, int H, int N, int d, float rope_theta,
                                        void* workspace, size_t workspace_bytes,
                                        cudaStream_t stream);

/* The mode ATTNFUSE_ROPE_AUTO resolves to for sequence length N and head dim d, for the
 * forward (backward = 0) or the backward (backward = 1). Measured on GB300 with B*N = 16384
 * tokens, causal: fusion wins for head dim 64 below N ~ 1.85k (forward) and N ~ 260
 * (backward), and for the head-dim-128 forward below N ~ 15k; above those, and for the
 * head-dim-128 backward at every N, the pre-rotation pass is cheaper than rotating K tiles on
 * chip. The workspace size functions accept ATTNFUSE_ROPE_AUTO and size for the resolved mode. */
attnfuse_status attnfuse_rope_auto_mode(int N, int d, int backward, attnfuse_rope_mode* mode);

/* Build the (cos, sin) table that the rotating modes keep at the start of their workspace:
 * entry (p, i) = (cos, sin)(p * theta_i) for p < N, i < d/2, fp32 pairs, computed in-kernel
 * with the angle reduced in turns (exact product split) so large positions keep full accuracy.
 * table: at least attnfuse_fwd_workspace_size(.., ATTNFUSE_ROPE_FUSED, ..) bytes. */
attnfuse_status attnfuse_rope_table(void* table, size_t table_bytes, int N, int d,
                                    float rope_theta, cudaStream_t stream);

/* Debug: launch one kernel whose only wait can never complete, bounded by `limit_ns`
 * nanoseconds. The kernel then records ATTNFUSE_ERR_TIMEOUT in the device status word and
 * returns, leaving the context usable. Exercises the timeout path without faulting. */
attnfuse_status attnfuse_debug_wait_timeout(uint64_t limit_ns, cudaStream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* ATTNFUSE_H_ */
