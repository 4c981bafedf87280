/*
 * fdma.h -- C ABI of libfdma: FlashAttention-style tiled attention with a
 * dynamic 4D mask (dense, or FlashMask column row-ranges), a learnable 4D
 * bias, block skipping and a fused, GQA-summed dBias, for sm_103a (GB300).
 *
 * Operation (Flash-DMA README, "Key Features" and the Quick Start example;
 * Flash-DMA issue #73, "Project Progress"; FlashMask README, "Formulation"
 * and "Sparse computation"):
 *
 *   keep(b,g,i,j) = mask[b,g,i,j] != 0                          (FDMA_MASK_DENSE)
 *                 | !(colranges[b,g,j,0] <= i < colranges[b,g,j,1])  (FDMA_MASK_COLRANGES)
 *                 | 1                                           (FDMA_MASK_NONE)
 *                   and, with is_causal, j <= i
 *   S[b,h,i,j]    = scale * <q[b,i,h,:], k[b,j,g,:]> + bias[b,g,i,j]   if keep, else -inf
 *   O[b,i,h,:]    = sum_j softmax_j(S[b,h,i,:]) v[b,j,g,:]
 *   lse[b,h,i]    = log sum_j exp(S[b,h,i,j])           (natural log)
 *
 * where g = h / (Hq / Hkv) (query heads are grouped contiguously onto kv
 * heads).  A row with no kept key yields O = 0 and lse = -inf, and receives
 * and produces zero gradient.  The backward returns dQ, dK, dV and
 *   dBias[b,g,i,j] = sum_{h in group g} dS[b,h,i,j],  dS = P*(dP - rowsum(dO*O)),
 * which is exactly 0 wherever keep is false.
 *
 * Tiles are 128 (queries) x 128 (keys).  A tile with no kept element is
 * SKIPPED: its K, V, bias and mask are never loaded by the attention kernels.
 *
 * Conventions for every entry point
 *   - All data pointers are CUDA device pointers owned by the caller; the
 *     library never allocates, frees or retains them.  `workspace` is
 *     caller-allocated device memory of at least fdma_workspace_size() bytes.
 *   - Every call is asynchronous on `stream` (a cudaStream_t; NULL = legacy
 *     default stream) and keeps no state between calls, except that the
 *     classification written into the workspace by one call may be reused by
 *     a later call with the same mask (FDMA_FLAG_REUSE_CLASSIFICATION).
 *   - Argument errors are reported synchronously as a non-zero fdma_status;
 *     nothing is launched in that case.  Launch failures return
 *     FDMA_ERR_CUDA.  Kernel-side time-outs (a wait that exceeded its bound)
 *     are recorded in a device error word read by fdma_get_device_error().
 *   - No function throws or aborts.
 *   - Element types: q, k, v, out, dout, dq, dk, dv, mask, bias, dbias are
 *     bf16; lse is fp32; colranges is int32.
 */
#ifndef FDMA_H_
#define FDMA_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define FDMA_API __attribute__((visibility("default")))
#else
#define FDMA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  FDMA_OK = 0,
  FDMA_ERR_INVALID = 1,      /* bad argument (shape, pointer, stride, scale) */
  FDMA_ERR_UNSUPPORTED = 2,  /* valid but not implemented (head dim, alignment, strides) */
  FDMA_ERR_CUDA = 3,         /* a CUDA runtime call or launch failed */
  FDMA_ERR_TIMEOUT = 4,      /* a bounded in-kernel wait expired (see fdma_get_device_error) */
  FDMA_ERR_WORKSPACE = 5     /* workspace missing or smaller than fdma_workspace_size() */
} fdma_status;

typedef enum {
  FDMA_MASK_NONE = 0,
  FDMA_MASK_DENSE = 1,       /* bf16 (B,Hkv,Nq,Nk), nonzero = keep */
  FDMA_MASK_COLRANGES = 2,   /* int32 (B,Hkv,Nk,2): one masked query-row range per key column */
  FDMA_MASK_DENSE_U8 = 3,    /* uint8 / bool (B,Hkv,Nq,Nk), nonzero = keep */
  FDMA_MASK_COLRANGES2 = 4,  /* int32 (B,Hkv,Nk,4): two masked query-row ranges per key column */
  FDMA_MASK_BITS = 5         /* uint8 (B,Hkv,Nq,ceil(Nk/8)) bit-packed: bit (j & 7) of byte j >> 3 = keep */
} fdma_mask_kind;

/* flags */
#define FDMA_FLAG_REUSE_CLASSIFICATION 1u /* workspace already classified for this mask: skip the classifier */
#define FDMA_FLAG_NO_SKIP 2u              /* debug: treat every causally allowed tile as PARTIAL (no skipping) */
#define FDMA_FLAG_TEST_SHORT_WAIT 4u      /* test: in fdma_fwd / fdma_bwd the softmax (compute) warps first wait
                                             about 100 us on a barrier nothing arrives at; the wait expires,
                                             the kernel unwinds (its own copies and products drained, TMEM
                                             freed) and fdma_get_device_error() returns FDMA_ERR_TIMEOUT.
                                             The outputs are then incomplete.  Exercises the bounded-wait
                                             failure path without any fault. */

typedef struct fdma_args {
  /* problem size: batch, query length, key length, query heads, kv heads, head dim d of q and
     k.  With dv (below) = d: a multiple of 8 from 8 to 128, run on the 64- or 128-wide kernels
     with the missing columns read as zeros.  Also d = 192 with dv = 128 and d = 256 with
     dv = 256 (FlashMask README, "Performance", SM100 head-dim table): the forward on a one-head
     kernel, the backward on kernels that split the gradient columns into two parts (each
     recomputes S and dP; slower per flop than d <= 128).  Other values: FDMA_ERR_UNSUPPORTED. */
  int32_t B, Nq, Nk, Hq, Hkv, d;

  /* q (B,Nq,Hq,d), k (B,Nk,Hkv,d) and v (B,Nk,Hkv,dv); strides in ELEMENTS for (batch, seq,
     head); the head-dim axis is contiguous.  seq/head/batch strides * 2 bytes must be multiples
     of 16. */
  const void* q;
  int64_t q_stride[3];
  const void* k;
  int64_t k_stride[3];
  const void* v;
  int64_t v_stride[3];

  /* mask selection (fdma_mask_kind) */
  int32_t mask_kind;
  /* FDMA_MASK_DENSE: bf16 (B,Hkv,Nq,Nk), nonzero = keep (both signed zeros count as zero).
     FDMA_MASK_DENSE_U8: uint8 (or bool) (B,Hkv,Nq,Nk), nonzero = keep.
     Strides (batch, head, row) in elements, columns contiguous; every stride a multiple of 8
     elements (0 broadcasts a batch or head), base 16-byte aligned (else FDMA_ERR_UNSUPPORTED).
     FDMA_MASK_BITS: uint8 (B,Hkv,Nq,ceil(Nk/8)), one bit per key, least significant bit first
     (key j of row i is bit j & 7 of byte j >> 3); bits past Nk are ignored.  Strides (batch,
     head, row) in bytes, any alignment (0 broadcasts a batch or head). */
  const void* mask;
  int64_t mask_stride[3];
  /* FDMA_MASK_COLRANGES: int32 (B,Hkv,Nk,2): query rows [start,end) are MASKED for key
     column j (start >= end: none masked; values outside [0,Nq) are clamped by the test).
     FDMA_MASK_COLRANGES2: int32 (B,Hkv,Nk,4): rows [start1,end1) and [start2,end2) are
     masked (the union), each range read as above.
     cr_stride = (batch, head) strides in int32 elements; within one (batch, head) the
     (Nk, 2) or (Nk, 4) block is contiguous (key j at offset 2*j or 4*j). */
  const int32_t* colranges;
  int64_t cr_stride[2];

  /* optional bf16 bias (B,Hkv,Nq,Nk) (NULL = zero bias); strides (batch, head, row) in
     elements, each a multiple of 8 elements, base 16-byte aligned.  A batch or head stride
     of 0 broadcasts the bias over that axis (the row stride must be nonzero); dBias is
     still returned per (batch, kv head): sum it over a broadcast axis for the gradient of
     the broadcast tensor. */
  const void* bias;
  int64_t bias_stride[3];

  int32_t is_causal; /* 1: keep additionally requires j <= i + (Nk - Nq) (bottom-right aligned:
                        j <= i when Nq == Nk); 2: keep requires j <= i + q_offset (below); 0: no
                        causal rule; other values FDMA_ERR_INVALID.  Rows that see no key are
                        fully masked. */
  float scale;       /* multiplies Q K^T only; must be finite and > 0 */
  uint32_t flags;    /* FDMA_FLAG_* */

  void* workspace; /* device memory, >= fdma_workspace_size(args, for_bwd) bytes, 256-byte aligned */
  size_t workspace_bytes;

  /* is_causal == 2 only: the position of query row 0 in the key sequence, so that query row i
     sees keys j <= i + q_offset.  A slice of query rows [r0, r1) of a longer causal problem
     over the same keys is the problem on those rows with q_offset = r0 + (Nk - Nq_full) (context
     parallelism: each rank's rows against all keys).  |q_offset| <= 2^30, else
     FDMA_ERR_INVALID.  Ignored for is_causal 0 and 1. */
  int32_t q_offset;

  /* head dim of v, out and dout; 0 means dv = d (a zero-initialised struct keeps the equal
     head dims).  Negative: FDMA_ERR_INVALID.  Allowed pairs: see d above. */
  int32_t dv;
} fdma_args;

/* Bytes of workspace needed by fdma_classify_blocks / fdma_fwd (for_bwd = 0) or by
   fdma_bwd as well (for_bwd = 1).  Returns 0 when the shape in args is invalid. */
FDMA_API size_t fdma_workspace_size(const fdma_args* args, int for_bwd);

/* Block classification (Flash-DMA "Key Features": OR-reduction over each
   mask block; FlashMask "Sparse computation": fully masked / partially masked
   / unmasked).  Writes the per-tile classes into the workspace and, when
   block_map != NULL, also to block_map: int8 (B, Hkv, ceil(Nq/128), ceil(Nk/128)),
   contiguous, values 0 = SKIP (no kept element), 1 = PARTIAL, 2 = FULL (every
   in-bounds element kept).  Reads the dense mask once; reads no mask above
   the causal diagonal.  block_m and block_n must be 128. */
FDMA_API int fdma_classify_blocks(const fdma_args* args, int block_m, int block_n, int8_t* block_map, void* stream);

/* Forward.  Classifies (unless FDMA_FLAG_REUSE_CLASSIFICATION) and computes
   out: bf16 (B,Nq,Hq,dv) contiguous and lse: fp32 (B,Hq,Nq) contiguous.
   Precision: the softmax weights enter the P V product rounded to bf16, and both O and lse
   are normalised by the sum of those rounded weights (so the weights that produced O sum to
   exactly 1).  lse is therefore the log-sum-exp of the definition up to a relative error of
   the row sum of at most 2^-9: |lse - exact| <= ln(1 + 2^-9) ~ 1.95e-3, plus fp32 rounding.
   fdma_bwd expects this lse (it recomputes the same weights). */
FDMA_API int fdma_fwd(const fdma_args* args, void* out, float* lse, void* stream);

/* Backward.  out, dout: bf16 (B,Nq,Hq,dv) contiguous; lse as written by fdma_fwd.
   Outputs dq: bf16 (B,Nq,Hq,d), dk: bf16 (B,Nk,Hkv,d) and dv: bf16 (B,Nk,Hkv,dv) (summed over each
   group's query heads), dbias: bf16 (B,Hkv,Nq,Nk) (NULL: not computed; requires
   args->bias != NULL), all contiguous.  Every dbias element is written (zeros in
   skipped tiles and at masked positions).  Classifies unless
   FDMA_FLAG_REUSE_CLASSIFICATION.  Needs the for_bwd workspace size.
   Determinism: dk, dv and dbias are bitwise reproducible run to run (each is summed in a
   fixed order inside one CTA).  dq is not: every key tile adds its part to an fp32
   accumulator with atomic reductions whose order varies, so repeated calls can differ in
   the last bits of dq (well inside the bf16 rounding of the result). */
FDMA_API int fdma_bwd(const fdma_args* args, const void* out, const void* dout, const float* lse, void* dq, void* dk,
             void* dv, void* dbias, void* stream);

/* Forward without a caller-provided workspace, for callers that cannot allocate device
   memory when they call it (an allocator or memory-pool callback, a plugin handed only
   fixed buffers, a process whose device footprint must not grow after start-up).  The
   pages describe no such entry point; it has no counterpart there.
   Same operation, arguments and outputs as fdma_fwd (args->workspace and
   args->workspace_bytes are ignored, FDMA_FLAG_REUSE_CLASSIFICATION is ignored: every call
   classifies).  Its workspace is one 16 MiB array of device memory compiled into the
   library; every GPU that loads the library holds it until the process exits.  Problems
   whose forward workspace (fdma_workspace_size(args, 0)) exceeds 16 MiB -- roughly more than
   4095 tiles of 128 x 128 over B * Hkv -- are rejected with FDMA_ERR_WORKSPACE before
   anything is launched.  No memory is allocated: no cudaMalloc, cudaFree or allocating
   library call.  The first call on a device looks up the array's device address with that
   device current; make that first call before any stream capture.  All calls share the one
   array and each overwrites what the previous call left there (nothing in it needs to start
   at zero), so calls whose executions overlap on the GPU race with each other: order them
   on one stream or synchronize between them. */
FDMA_API int fdma_fwd_noalloc(const fdma_args* args, void* out, float* lse, void* stream);

/* Dynamic top-k mask (Flash-DMA README, "Quick Start" example: the sparse mask built from
   the bias before the attention call).  For every row (b, g, i) of bias, bf16 (B,Hkv,Nq,Nk):
     - if Nk <= keep_window: every key is kept;
     - else the keep_window keys of largest bias value are selected (equal values: the
       smaller key index first; +0 and -0 are equal), and a selected key is kept unless its
       bias equals the bf16 minimum (-3.3895e38).
   mask: (B,Hkv,Nq,Nk) contiguous, 1 where kept and 0 elsewhere, bf16 (mask_kind =
   FDMA_MASK_DENSE) or uint8 (FDMA_MASK_DENSE_U8).  bias_out (NULL: not written) receives the
   bias where kept and the bf16 minimum elsewhere, laid out with bias_stride (so bias_out ==
   bias rewrites the bias in place); with bias_out the strides must be nonzero and rows must
   not overlap.  bias_stride: elements between batches, kv heads and rows (keys contiguous;
   stride 0 broadcasts when bias_out is NULL).  Requirements: keep_window >= 1; Nk <= 65536
   and a multiple of 8, strides multiples of 8 and pointers 16-byte aligned, else
   FDMA_ERR_UNSUPPORTED.  Deterministic: the result does not depend on the launch. */
FDMA_API int fdma_topk_mask(const void* bias, const int64_t bias_stride[3], int B, int Hkv, int Nq, int Nk,
                            int keep_window, int mask_kind, void* mask, void* bias_out, void* stream);

/* Synchronizes `stream`, returns the first kernel-side error recorded since the last call
   (FDMA_OK if none) and clears it. */
FDMA_API int fdma_get_device_error(void* stream);

/* Static, human-readable name of a status code. */
FDMA_API const char* fdma_status_string(int status);

#ifdef __cplusplus
}
#endif

#endif /* FDMA_H_ */
