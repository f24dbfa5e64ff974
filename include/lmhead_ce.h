/*
 * lmhead_ce.h -- C ABI of the fused tied-LM-head + softcapped cross-entropy
 * library for B300 (sm_103a).
 *
 * The operation (notation: N rows, d model dim, V vocab, c softcap):
 *   z = h W^T                   tied LM head: W is the [V, d] embedding table
 *   s = c * tanh(z / c)         tanh logit softcap
 *   lse_i = ln sum_j exp(s_ij)  log-sum-exp over the vocabulary
 *   nll_i = lse_i - s_{i,t_i}   next-token negative log-likelihood
 *   bpb = sum nll / (ln 2 * sum bytes)       bits per byte
 *   dh = w G W,  dW (+)= w G^T h,  G_ij = (p_ij - [j == t_i]) (1 - (s_ij/c)^2),
 *   p_ij = exp(s_ij - lse_i), w = grad_scale.
 * Sources (page title, section):
 *   - "parameter-golf: ... Where Model Size Becomes the Game", "The Baseline
 *     Is a Map, Not the Destination": the step is logits = model(x);
 *     loss = criterion(logits, y); loss.backward().
 *   - "parameter-golf README", leaderboard row "Naive Baseline": tied
 *     embeddings (the head's W is the input embedding table).
 *   - "HYDRA Golf" site stack list ("fused softcapped CE kernel") and
 *     "parameter-golf README" leaderboard row "PR1736 + PolarNS + MIN_LR +
 *     SparseAttnGate + FusedCE + Warm-A TTT" ("fused softcapped CE").  The
 *     pages give no softcap formula; the tanh form above is used.
 *   - tproger news "OpenAI launched Parameter Golf", section "Rules and
 *     metric": bits per byte on FineWeb validation (bytes, not tokens).
 *   - "parameter-golf README", leaderboard row "Sliding Window Eval": stride
 *     64 sliding-window scoring, expressed here as a row mask.
 *   - "HYDRA Golf" site stack list: per-group int4 head ("LQER asymmetric
 *     int4, per-group compression"); this library reads it as symmetric,
 *     group 64 along d, fp16 scales (lmhead_ce_*_int4), and also offers the
 *     asymmetric form with integer zero points (lmce_qhead).
 *   - "parameter-golf README", leaderboard rows "Mixed Quant + Sliding Window
 *     Eval" (int8 embeddings), "VarLen Attention + Fused MLP + Multi-Phase
 *     Global SGD TTT" (int7 embeddings) and "fp16 Embed" (FP16 tied
 *     embedding): more storage formats of the tied table (lmce_qhead).
 *   - "parameter-golf README", leaderboard rows "SP8192 + CaseOps + ..."
 *     (byte-sidecar BPB accounting) and "CaseOps Tokenizer + ..." (validation
 *     byte sidecars); "HYDRA Golf" submission conditions (tokenizer-aware
 *     validation BPB): bytes per scored token from a per-id table
 *     (bpb_reduce_lut) or a per-row sidecar (bpb_reduce).
 *   - "parameter-golf README", leaderboard row "11L Partial RoPE + LN Scale +
 *     EMA + XSA4" (layerwise LN scale): the normalisation in front of the head,
 *     read as RMSNorm with an optional gain (lmhead_rmsnorm_*).
 *
 * Conventions for every entry point:
 *   - All pointers are DEVICE pointers unless a comment says host.  The caller
 *     owns every buffer; the library allocates nothing.
 *   - bf16 arrays are passed as uint16_t bit patterns (lmce_bf16).
 *   - h is [N, d] row-major with row stride ldh elements; W is [V, d]
 *     row-major (stride d).  Base addresses and row strides must be 16-byte
 *     aligned (ldh % 8 == 0).  d must be a multiple of 64 with d <= 512.
 *     N and V are arbitrary (>= 1); tails are handled inside the kernels.
 *   - targets are int64 in [0, V) on every unmasked row.
 *   - softcap c >= 0 and finite; c = 0 means no cap (s = z).  Up to
 *     lmce_softcap_max(V) the forward sums e^s with a fixed shift; c = 0 and
 *     larger caps take a running-maximum form of the same kernel.
 *   - row_mask (nullable) is [N] uint8: 0 = row not scored (nll = 0, lse = 0,
 *     dh row = 0, no contribution to dW or the bpb sums).
 *   - ws is a device workspace of at least lmce_workspace_bytes(...) bytes,
 *     16-byte aligned, zero-filled once by the caller (or by
 *     lmce_workspace_init) before its first use.  It carries a sticky device
 *     status word; concurrent calls must use distinct workspaces.
 *   - stream is a cudaStream_t (passed as void*; NULL = default stream).  All
 *     work is asynchronous on it; only lmce_status synchronises.
 *   - Return values: LMCE_OK, or an error detected on the host before any
 *     launch (nothing was enqueued), or LMCE_ECUDA for a launch failure.
 *     Errors found by the kernels (a target out of range, a bounded wait that
 *     expired) are reported later through lmce_status.
 */
#ifndef LMHEAD_CE_H_
#define LMHEAD_CE_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define LMCE_API __attribute__((visibility("default")))
#else
#define LMCE_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef uint16_t lmce_bf16; /* bfloat16 bit pattern */
typedef uint16_t lmce_f16;  /* IEEE binary16 bit pattern */

enum lmce_status_code {
  LMCE_OK = 0,
  LMCE_EINVAL = 1,   /* null pointer, bad shape or stride, misalignment, N or V < 1, short workspace */
  LMCE_ENOTSUP = 2,  /* d not a multiple of 64 or > 512, softcap negative or not finite, no sm_103 device */
  LMCE_ECUDA = 3,    /* CUDA runtime / launch failure; text via lmce_last_cuda_error() */
  LMCE_EDATA = 4,    /* device-detected: target outside [0, V) on a scored row; or sum of bytes == 0 */
  LMCE_ETIMEOUT = 5  /* device-detected: a bounded in-kernel wait expired (the kernel returned early) */
};

/* Workspace flags. */
#define LMCE_WS_MASKED 1u /* room for row-mask compaction (masked forward) */
#define LMCE_WS_INT4 2u   /* room for the dequantised bf16 copy of an int4 head */
#define LMCE_WS_EMBED 4u  /* room for lmhead_tied_embed_bwd (counting sort, piece sums) */
#define LMCE_WS_QHEAD 2u  /* room for the dequantised bf16 copy of any lmce_qhead (same as LMCE_WS_INT4) */
#define LMCE_WS_RMSNORM 8u /* room for the RMSNorm calls (normalised rows, their gradient, the gain's partials) */

/* Storage formats of a quantised (or fp16) tied table, for lmhead_ce_*_q. */
#define LMCE_QHEAD_INT4 1      /* symmetric int4: two's-complement nibbles, fp16 scale per group */
#define LMCE_QHEAD_INT4_ASYM 2 /* asymmetric int4: unsigned nibbles, fp16 scale and zero point per group */
#define LMCE_QHEAD_INT8_ROW 3  /* int8 codes (int7: |q| <= 63), one fp16 scale per row */
#define LMCE_QHEAD_FP16 4      /* fp16 table */

/* A quantised head [V, d].  Dequantisation is exact up to one RNE rounding
 * to bf16:
 *   INT4:      W[v,k] = bf16_rne(q * scales[v, k/group]), q in [-8, 7], element
 *              2m in the low nibble of byte m of codes [V, d/2];
 *   INT4_ASYM: W[v,k] = bf16_rne((q - zeros[v, k/group]) * scales[v, k/group]),
 *              q in [0, 15] (same packing), zeros [V, d/group] bytes in [0, 15];
 *   INT8_ROW:  W[v,k] = bf16_rne(q * scales[v]), codes [V, d] int8;
 *   FP16:      W[v,k] = bf16_rne(codes[v,k]), codes [V, d] fp16 (scales unused).
 * group (int4 formats) is a multiple of 16 dividing d.  codes are 8-byte
 * (int4) or 16-byte (int8, fp16) aligned device pointers; scales are device
 * fp16 arrays.  The struct itself is host memory, read during the call. */
typedef struct lmce_qhead {
  int format;
  int group;
  const void* codes;
  const lmce_f16* scales;
  const uint8_t* zeros;
} lmce_qhead;

/* Accumulator of the bits-per-byte sums (device memory for bpb_reduce). */
typedef struct lmce_bpb_acc {
  double sum_nll;      /* sum of nll over scored rows (nats) */
  long long sum_bytes; /* sum of bytes over scored rows */
  long long n_scored;  /* number of scored rows */
} lmce_bpb_acc;

/* Bytes of workspace needed for problems of up to N rows, V vocab, d dims,
 * for the uses named in flags (LMCE_WS_*). */
LMCE_API size_t lmce_workspace_bytes(int64_t N, int64_t V, int64_t d, unsigned flags);

/* Zero the workspace's status word (asynchronous on stream). */
LMCE_API int lmce_workspace_init(void* ws, size_t ws_bytes, void* stream);

/* Largest softcap of the fixed-shift forward for vocab V.  Up to it the
 * forward sums e^s without a running maximum (|s| < c bounds every term),
 * which stays in fp32 range while V e^c is finite and e^-c normal; larger
 * softcaps, and 0 (no cap), use a running maximum (slower epilogue). */
LMCE_API float lmce_softcap_max(int64_t V);

/* Forward.  Defining passages: see the header comment (tied head, tanh
 * softcap, log-sum-exp, next-token NLL).
 * Inputs: h [N, d] bf16 (row stride ldh), W [V, d] bf16, tgt [N] int64,
 * row_mask [N] uint8 or NULL, softcap c.
 * Outputs: nll [N] fp32; lse [N] fp32 or NULL (needed by the backward).
 * With a row mask only the scored rows are computed (they are compacted into
 * the workspace first); requires a workspace sized with LMCE_WS_MASKED. */
LMCE_API int lmhead_ce_fwd(const lmce_bf16* h, int64_t ldh, const lmce_bf16* W, int64_t N, int64_t V, int64_t d,
                  const int64_t* tgt, const uint8_t* row_mask, float softcap, float* nll, float* lse, void* ws,
                  size_t ws_bytes, void* stream);

/* Backward of L = grad_scale * sum over scored rows of nll_i.
 * Inputs as lmhead_ce_fwd plus lse [N] fp32 from the forward, and
 * optionally (nullable) nll [N] fp32 from the same forward call.  With nll
 * the target's p - 1 is taken as expm1(-nll) instead of e^{s_t - lse} - 1;
 * the latter loses its relative precision in fp32 as p_t -> 1 (s_t and lse
 * cancel), which matters for confident predictions.
 * Outputs (each nullable, at least one non-NULL):
 *   dh [N, d] bf16 (row stride ldh), overwritten; masked rows get 0.
 *   dW [V, d] fp32: accumulate_dW != 0 adds into it, else overwrites.
 * grad_scale: dL/dnll of each scored row (1/M for a mean over M rows). */
LMCE_API int lmhead_ce_bwd(const lmce_bf16* h, int64_t ldh, const lmce_bf16* W, int64_t N, int64_t V, int64_t d,
                  const int64_t* tgt, const uint8_t* row_mask, float softcap, const float* lse, const float* nll,
                  float grad_scale, lmce_bf16* dh, float* dW, int accumulate_dW, void* ws, size_t ws_bytes,
                  void* stream);

/* Forward and backward of one training step, for L = grad_scale * sum over
 * scored rows of nll_i (defining passages as lmhead_ce_fwd and
 * lmhead_ce_bwd).  Outputs: nll and lse [N] fp32 (both required); dh [N, d]
 * bf16 (row stride ldh, nullable); dW [V, d] fp32 (nullable;
 * accumulate_dW != 0 adds into it).
 * With dh requested and softcap <= 60 the forward and dh come from ONE pass
 * over the vocabulary: the row's normaliser is applied after the
 * accumulation (dh_i = -w/S_i sum_{j != t_i} e^{s_ij}(1 - tanh^2) W_j
 * + w (p_{i,t_i} - 1)(1 - tanh_{i,t_i}^2) W_{t_i}, S_i = sum_j e^{s_ij}),
 * which saves the separate forward's logit GEMM.  dW then takes a second
 * pass that reads lse and nll.  Masked rows are computed and zeroed in that pass
 * (no compaction), so a heavily masked batch is better served by
 * lmhead_ce_fwd + lmhead_ce_bwd.  Softcap 0 (no cap), softcaps above 60, or
 * dh == NULL run the forward and the backward passes separately.  Same
 * workspace and layout rules as lmhead_ce_bwd. */
LMCE_API int lmhead_ce_fwd_bwd(const lmce_bf16* h, int64_t ldh, const lmce_bf16* W, int64_t N, int64_t V, int64_t d,
                      const int64_t* tgt, const uint8_t* row_mask, float softcap, float grad_scale, float* nll,
                      float* lse, lmce_bf16* dh, float* dW, int accumulate_dW, void* ws, size_t ws_bytes,
                      void* stream);

/* Forward with the head stored as per-group int4 (symmetric, two's-complement
 * nibbles; element 2m of a row in the low nibble of byte m) with one fp16
 * scale per group of `group` elements along d.  Wq [V, d/2] uint8, scales
 * [V, d/group] fp16.  The head is dequantised on the device into the
 * workspace (W_deq = bf16_rne(q * scale), bit-exact) and the bf16 forward
 * runs on it.  Needs a workspace sized with LMCE_WS_INT4 (| LMCE_WS_MASKED
 * with a row mask).  group must divide d and be a multiple of 16. */
LMCE_API int lmhead_ce_fwd_int4(const lmce_bf16* h, int64_t ldh, const uint8_t* Wq, const lmce_f16* scales, int group,
                       int64_t N, int64_t V, int64_t d, const int64_t* tgt, const uint8_t* row_mask, float softcap,
                       float* nll, float* lse, void* ws, size_t ws_bytes, void* stream);

/* The same forward as lmhead_ce_fwd_int4 with the dequantisation inside the
 * forward kernel: the packed nibbles stream through the kernel's ring (a
 * quarter of the bf16 head's bytes) and converter warps write each stage's
 * bf16 tile (bf16_rne(q * scale), bit-exact, so nll and lse are bit for bit
 * those of lmhead_ce_fwd_int4).  Needs no room for a dequantised copy: the
 * workspace is lmce_workspace_bytes(N, V, d, row_mask ? LMCE_WS_MASKED : 0).
 * Wq must be 16-byte aligned.  lmhead_ce_fwd_int4 (dequantise once, then
 * the bf16 forward) is faster on large batches; this call saves the 2 V d
 * byte copy and its pass, which pays on small ones. */
LMCE_API int lmhead_ce_fwd_int4_inkernel(const lmce_bf16* h, int64_t ldh, const uint8_t* Wq, const lmce_f16* scales,
                                         int group, int64_t N, int64_t V, int64_t d, const int64_t* tgt,
                                         const uint8_t* row_mask, float softcap, float* nll, float* lse, void* ws,
                                         size_t ws_bytes, void* stream);

/* Backward for the int4 head: dh only (the quantised head is frozen).
 * Same layout rules as lmhead_ce_fwd_int4 and lmhead_ce_bwd. */
LMCE_API int lmhead_ce_bwd_int4(const lmce_bf16* h, int64_t ldh, const uint8_t* Wq, const lmce_f16* scales, int group,
                       int64_t N, int64_t V, int64_t d, const int64_t* tgt, const uint8_t* row_mask, float softcap,
                       const float* lse, const float* nll, float grad_scale, lmce_bf16* dh, void* ws,
                       size_t ws_bytes, void* stream);

/* Forward and dh for the int4 head in one call: the head is dequantised once
 * (as in lmhead_ce_fwd_int4) and, for softcap <= 60, nll, lse and dh come
 * from the single fused pass of lmhead_ce_fwd_bwd; above that the forward
 * and the dh backward run as two passes.  Equal, up to rounding order, to
 * lmhead_ce_fwd_int4 followed by lmhead_ce_bwd_int4.  nll, lse [N] fp32 and
 * dh (row stride ldh, 16-byte aligned) are required.  Needs a workspace
 * sized with LMCE_WS_INT4 (| LMCE_WS_MASKED with a row mask).  A target
 * outside [0, V) sets LMCE_EDATA in the status word and nll = NaN for that
 * row; its dh row stays finite but carries no meaning. */
LMCE_API int lmhead_ce_fwd_bwd_int4(const lmce_bf16* h, int64_t ldh, const uint8_t* Wq, const lmce_f16* scales,
                           int group, int64_t N, int64_t V, int64_t d, const int64_t* tgt,
                           const uint8_t* row_mask, float softcap, float grad_scale, float* nll, float* lse,
                           lmce_bf16* dh, void* ws, size_t ws_bytes, void* stream);

/* Gradient of the tied table through the input embedding.  With tied
 * embeddings W is also the input embedding table ("[AGENT TASK] OpenAI
 * Parameter Golf", architecture experiments table, row "Tied embeddings";
 * "parameter-golf README", leaderboard row "Naive Baseline":
 * TiedEmbeddings), so the table's gradient is the head's dW (from
 * lmhead_ce_bwd or lmhead_ce_fwd_bwd) plus, for every input position i, the
 * gradient g_i of the loss with respect to that position's embedding row:
 *   dW[ids[i], :] += g[i, :]   for i = 0 .. N-1.
 * Inputs: ids [N] int64 (the input tokens), g [N, d] bf16 with row stride
 * ldg elements (ldg % 8 == 0, 16-byte aligned).  dW [V, d] fp32 is added to.
 * Deterministic: each token's rows are summed in row order in fp32 (in
 * pieces of at most 32 rows, then groups of 16 pieces, each added in order),
 * then added to dW once, by an atomic add that flushes a subnormal operand or
 * result (below 2^-126 in magnitude) to zero.  A row whose id is outside
 * [0, V) is skipped and sets LMCE_EDATA in the status word.  Needs a workspace sized with LMCE_WS_EMBED; d as for the head
 * (a multiple of 64, at most 512). */
LMCE_API int lmhead_tied_embed_bwd(const int64_t* ids, const lmce_bf16* g, int64_t ldg, int64_t N, int64_t V,
                          int64_t d, float* dW, void* ws, size_t ws_bytes, void* stream);

/* Forward, dh backward and the training-side forward + dh for a quantised or
 * fp16 tied table (formats above).  The head is dequantised once per call
 * into the workspace (bit-exact), then the bf16 kernels run on it, exactly
 * as lmhead_ce_fwd / lmhead_ce_bwd (dh only; the stored head is frozen) /
 * lmhead_ce_fwd_bwd (dh, no dW).  Workspace: lmce_workspace_bytes(N, V, d,
 * LMCE_WS_QHEAD | (row_mask ? LMCE_WS_MASKED : 0)).  The int4 entry points
 * above are these calls with an LMCE_QHEAD_INT4 head. */
LMCE_API int lmhead_ce_fwd_q(const lmce_bf16* h, int64_t ldh, const lmce_qhead* head, int64_t N, int64_t V,
                             int64_t d, const int64_t* tgt, const uint8_t* row_mask, float softcap, float* nll,
                             float* lse, void* ws, size_t ws_bytes, void* stream);
LMCE_API int lmhead_ce_bwd_q(const lmce_bf16* h, int64_t ldh, const lmce_qhead* head, int64_t N, int64_t V,
                             int64_t d, const int64_t* tgt, const uint8_t* row_mask, float softcap, const float* lse,
                             const float* nll, float grad_scale, lmce_bf16* dh, void* ws, size_t ws_bytes,
                             void* stream);
LMCE_API int lmhead_ce_fwd_bwd_q(const lmce_bf16* h, int64_t ldh, const lmce_qhead* head, int64_t N, int64_t V,
                                 int64_t d, const int64_t* tgt, const uint8_t* row_mask, float softcap,
                                 float grad_scale, float* nll, float* lse, lmce_bf16* dh, void* ws, size_t ws_bytes,
                                 void* stream);
/* Dequantise a head into out [V, d] bf16 (the routine the calls above use;
 * exposed for bit-exactness tests). */
LMCE_API int lmhead_qhead_dequant(const lmce_qhead* head, int64_t V, int64_t d, lmce_bf16* out, void* stream);

/* RMSNorm in front of the head ("parameter-golf README", leaderboard row
 * "11L Partial RoPE + LN Scale + EMA + XSA4": layerwise LN scale):
 *   h_i = g * x_i * rinv_i,  rinv_i = 1 / sqrt(mean_k x_ik^2 + eps)
 * x [N, d] bf16 (row stride ldx), g [d] fp32 gain or NULL (no gain), eps >= 0.
 * lmhead_rmsnorm_fwd writes h [N, d] bf16 (row stride ldh) and rinv [N]
 * fp32 (the reciprocal RMS, computed in fp32).
 * lmhead_rmsnorm_bwd takes dh = dL/dh [N, d] bf16 and writes
 *   dx_i = rinv_i (g dh_i) - x_i rinv_i^3 / d * sum_k g_k dh_ik x_ik  (bf16)
 * and, if dg is not NULL, dg (+)= sum_i dh_i x_i rinv_i ([d] fp32, added
 * when accumulate_dg != 0), summed in a fixed order (deterministic); dg
 * needs a workspace of lmce_workspace_bytes(N, 1, d, LMCE_WS_RMSNORM).
 * Alignment as for h (16-byte bases, strides multiples of 8 elements). */
LMCE_API int lmhead_rmsnorm_fwd(const lmce_bf16* x, int64_t ldx, const float* g, float eps, int64_t N, int64_t d,
                                lmce_bf16* h, int64_t ldh, float* rinv, void* stream);
LMCE_API int lmhead_rmsnorm_bwd(const lmce_bf16* x, int64_t ldx, const float* g, const float* rinv,
                                const lmce_bf16* dh, int64_t lddh, int64_t N, int64_t d, lmce_bf16* dx, int64_t lddx,
                                float* dg, int accumulate_dg, void* ws, size_t ws_bytes, void* stream);
/* The head on RMSNorm'd hidden states in one call: lmhead_rmsnorm_fwd into
 * the workspace, then lmhead_ce_fwd (forward) or lmhead_ce_fwd_bwd (training
 * step: nll, lse, dW (+)= ... with the normalised rows, and dx / dg through
 * lmhead_rmsnorm_bwd; dx and dg nullable, dg needs dx; accumulate applies to
 * dW and dg).  Workspace: lmce_workspace_bytes(N, V, d, LMCE_WS_RMSNORM |
 * (row_mask ? LMCE_WS_MASKED : 0)). */
LMCE_API int lmhead_ce_fwd_rmsnorm(const lmce_bf16* x, int64_t ldx, const float* g, float eps, const lmce_bf16* W,
                                   int64_t N, int64_t V, int64_t d, const int64_t* tgt, const uint8_t* row_mask,
                                   float softcap, float* nll, float* lse, void* ws, size_t ws_bytes, void* stream);
LMCE_API int lmhead_ce_fwd_bwd_rmsnorm(const lmce_bf16* x, int64_t ldx, const float* g, float eps,
                                       const lmce_bf16* W, int64_t N, int64_t V, int64_t d, const int64_t* tgt,
                                       const uint8_t* row_mask, float softcap, float grad_scale, float* nll,
                                       float* lse, lmce_bf16* dx, int64_t lddx, float* dg, float* dW, int accumulate,
                                       void* ws, size_t ws_bytes, void* stream);

/* Bits-per-byte sums (tproger news, "Rules and metric").  Adds, over rows with
 * row_mask != 0 (all rows if NULL), sum nll (fp64), sum bytes and the row
 * count into *acc (device memory).  Deterministic: fixed grid, fixed
 * summation tree, one ordered update of *acc. */
LMCE_API int bpb_reduce(const float* nll, const int32_t* bytes, const uint8_t* row_mask, int64_t N, lmce_bpb_acc* acc,
               void* ws, size_t ws_bytes, void* stream);

/* As bpb_reduce, with the bytes of each scored row taken from the
 * tokenizer's per-id byte-length table: bytes_i = lut[tgt[i]] ("parameter-golf
 * README", leaderboard rows "SP8192 + CaseOps + ..." and "CaseOps Tokenizer +
 * ...": byte sidecars; "HYDRA Golf" submission conditions: tokenizer-aware
 * validation BPB).  tgt [N] int64, lut [V] int32 (device).  A scored row
 * whose target is outside [0, V) counts nothing and sets LMCE_EDATA in the
 * workspace status word (read with lmce_status). */
LMCE_API int bpb_reduce_lut(const float* nll, const int64_t* tgt, const int32_t* lut, int64_t V,
                            const uint8_t* row_mask, int64_t N, lmce_bpb_acc* acc, void* ws, size_t ws_bytes,
                            void* stream);

/* Host helper: *bpb_out = acc->sum_nll / (ln 2 * acc->sum_bytes).  acc is a
 * HOST copy.  Returns LMCE_EDATA when sum_bytes == 0. */
LMCE_API int lmce_bpb(const lmce_bpb_acc* acc, double* bpb_out);

/* Dequantise an int4 head into out [V, d] bf16 (the same device routine the
 * int4 entry points use; exposed for bit-exactness tests). */
LMCE_API int lmhead_int4_dequant(const uint8_t* Wq, const lmce_f16* scales, int64_t V, int64_t d, int group, lmce_bf16* out,
                        void* stream);

/* Forward that allocates nothing and takes no workspace.  For callers that
 * cannot give the library device memory: code whose host process owns every
 * byte of device memory through its own pool and forbids other allocations,
 * or code on a path where cudaMalloc's implicit device synchronisation is not
 * acceptable.  There is no counterpart of this call in the pages; it is the
 * same computation as lmhead_ce_fwd without a row mask.
 * The scratch (about 16.3 MiB) is a static device array of this library:
 * every GPU that loads the library holds it until the process exits, and
 * all calls on one device share it, so calls that overlap on the GPU (other
 * streams, other threads) race and must be serialised by the caller.
 * Limits: N <= 65536 and V <= 8192 (else LMCE_EINVAL); d as for
 * lmhead_ce_fwd; softcap in (0, lmce_softcap_max(V)] (the fixed-shift form;
 * else LMCE_ENOTSUP).  The first call on a device looks up the scratch's
 * device address (cudaGetSymbolAddress); make that first call before any
 * stream capture.  The status word of this scratch is not readable by the
 * caller, so errors found on the device show in the outputs: a target
 * outside [0, V) gives nll = NaN for that row, and a bounded wait that
 * expired gives nll = lse = NaN on every row (each call clears the status
 * word when it starts).
 * Arguments: as lmhead_ce_fwd (all pointers device pointers; stream is a
 * cudaStream_t). */
LMCE_API int lmhead_ce_fwd_noalloc(const lmce_bf16* h, int64_t ldh, const lmce_bf16* W, int64_t N, int64_t V,
                                   int64_t d, const int64_t* tgt, float softcap, float* nll, float* lse,
                                   void* stream);

/* Self-test of the bounded wait that every in-kernel wait of this library
 * uses: one thread waits on an mbarrier that receives its arrival only if
 * arrive != 0; if the wait exceeds limit_cycles SM clock cycles it sets
 * LMCE_ETIMEOUT in the workspace status word and the kernel returns (read
 * it with lmce_status).  Faults, traps and hangs nothing.  ws: a workspace
 * of at least 64 bytes.  (Not part of the pages' method: a failure-detection
 * check.) */
LMCE_API int lmce_wait_selftest(long long limit_cycles, int arrive, void* ws, size_t ws_bytes, void* stream);

/* Synchronise stream, then read and clear the workspace's device status
 * word.  *code receives LMCE_OK, LMCE_EDATA or LMCE_ETIMEOUT (the most
 * severe recorded).  Returns LMCE_ECUDA if the synchronisation fails. */
LMCE_API int lmce_status(void* ws, void* stream, int* code);

/* Text of the last CUDA error seen by this library (thread-local). */
LMCE_API const char* lmce_last_cuda_error(void);

/* Number of kernels this library has enqueued in this process so far (a
 * diagnostic counter; monotonically increasing, thread-safe). */
LMCE_API unsigned long long lmce_launch_count(void);

/* Short text for a status code. */
LMCE_API const char* lmce_strerror(int code);

#ifdef __cplusplus
}
#endif

#endif /* LMHEAD_CE_H_ */
