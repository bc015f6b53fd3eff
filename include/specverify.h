/*
 * specverify -- the verify step of speculative decoding on one GB300 (sm_103a).
 *
 * A C ABI with plain pointers and sizes.  Every array argument is a DEVICE pointer owned
 * by the caller unless marked "host".  Calls are asynchronous on the given CUDA stream
 * (a cudaStream_t passed as void*; NULL = the legacy default stream) and return 0 or a
 * negative SPEC_E_* code; argument errors are found on the host before anything is
 * launched, and a description is kept for spec_last_error() (per host thread).
 *
 * Sources the operations follow (pages of the write-ups, by title and section):
 *  [SD-Apple]  "Speculative Decoding on Apple Silicon: 119% Faster on Qwen3.8",
 *              "How speculative decoding works" (draft K tokens, one batched target
 *              pass, keep the agreeing prefix, correct the first mismatch) and "Why this
 *              needed a patch to mlx_lm at all" (a KV cache is rolled back by slicing
 *              the rejected entries off its end).
 *  [MTP-fixes] "Qwen3.5 and Qwen3.6 MTP head reaches 1.4x on Apple Silicon after three
 *              fixes", "The verify was wrong under sampling" (accept with probability
 *              min(1, p/q), resample from max(0, p - q) renormalised) and "Truncation
 *              has to match on both sides" (top-k 20 / top-p 0.95 on both p and q).
 *  [Draft]     "What is Speculative Decoding and How Does a Draft Model Work?", "#2"
 *              and "#3" (greedy acceptance; one target pass always emits >= 1 token).
 *
 * Readings of what the pages leave open (the same in the CPU oracle):
 *  - a full acceptance emits a bonus token from the last target row;
 *  - uniforms u[b][0..K-1] drive the acceptance tests u < P/Q, u[b][K] drives the one
 *    final draw (residual resample or bonus);
 *  - truncation = top-k on the raw logits (ties to the lower token id), softmax of
 *    logits/temperature over those k, then keep tokens while the mass before them is
 *    below top_p (the first always stays; top_p >= 1 keeps all k), renormalise;
 *  - the final draw is an inverse CDF over the support in ascending token id;
 *  - temperature 0 is greedy: argmax (lower id on ties), accept while equal;
 *  - draft_logits == NULL means deterministic drafts (q = one-hot at the draft token).
 */
#ifndef SPECVERIFY_H
#define SPECVERIFY_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Status codes. */
#define SPEC_OK          0
#define SPEC_E_INVAL   (-1)  /* bad argument (NULL pointer, size out of range, bad dtype) */
#define SPEC_E_NOMEM   (-2)  /* workspace too small, page pool exhausted, allocation failed */
#define SPEC_E_RANGE   (-3)  /* a size above a compiled or configured maximum */
#define SPEC_E_STATE   (-4)  /* call not valid in the current state (e.g. no weights) */
#define SPEC_E_TIMEOUT (-5)  /* a bounded device-side wait gave up (reported per sequence) */
#define SPEC_E_CUDA    (-6)  /* a CUDA runtime call failed */
#define SPEC_E_DRAFT   (-7)  /* a drafted token has q = 0 under its own truncated draft row */

/* Largest top_k of the one-pass selection (a warp-wide sorted list). */
#define SPEC_TOPK_MAX 32

/* Sampler; temperature 0 selects greedy acceptance.  top_k in [1, SPEC_TOPK_MAX] when
 * temperature > 0; top_p in [0, 1] (values >= 1 disable the nucleus cut). */
typedef struct {
    float temperature;
    int32_t top_k;
    float top_p;
} spec_sampling;

/* Description of the last error on this host thread ("" if none). */
const char* spec_last_error(void);

/* Library version string. */
const char* spec_version(void);

/* ------------------------------------------------------------------------------------
 * Fused verify on caller-provided logits  ([MTP-fixes] both sections; [Draft] "#2").
 *
 * One pass over every needed row of target_logits [B][K+1][V] and draft_logits
 * [B][K][V] (fp32, row-major, contiguous).  Per row: exact top-k selection (greedy:
 * argmax), temperature softmax over the top-k, top-p cut, renormalisation; per sequence
 * b with k_b = draft_len[b] (K if draft_len is NULL) drafts: the acceptance tests of
 * draft_tokens[b][0..k_b-1] in order, stopping at the first rejection, then the final
 * draw.  Rows past k_b are not read.
 *
 * Outputs (device): accepted_len[b] in [0, k_b]; next_token[b] = the correction or bonus
 * token; out_ids/out_probs [B][SPEC_TOPK_MAX] (may be NULL): the distribution the final
 * token was drawn from, ascending token id, padded with id -1 / prob 0; seq_status[b]
 * (may be NULL): SPEC_OK, SPEC_E_DRAFT (then accepted_len[b] = number accepted before the
 * illegal draft and next_token[b] = -1) or SPEC_E_TIMEOUT (outputs of b undefined).
 *
 * workspace: device scratch of at least spec_verify_logits_workspace_bytes(B, K, V)
 * bytes, 256-byte aligned, owned by the caller; its contents need no initialisation (the
 * call clears what must start at zero with cudaMemsetAsync on `stream`).  Two calls that
 * share a workspace must not overlap on the GPU.
 * Errors: SPEC_E_INVAL for NULL required pointers, B < 1, K < 0, V < 2, K > 64,
 * temperature < 0 or NaN, top_k outside [1, SPEC_TOPK_MAX] with temperature > 0;
 * SPEC_E_NOMEM if workspace_bytes is too small; SPEC_E_CUDA on a launch failure.
 * ---------------------------------------------------------------------------------- */
size_t spec_verify_logits_workspace_bytes(int B, int K, int V);

int spec_verify_logits(int B, int K, int V,
                       const float* target_logits, const float* draft_logits,
                       const int32_t* draft_tokens, const int32_t* draft_len,
                       const float* uniforms, const spec_sampling* sampling /* host */,
                       int32_t* accepted_len, int32_t* next_token,
                       int32_t* out_ids, float* out_probs, int32_t* seq_status,
                       void* workspace, size_t workspace_bytes, void* stream);

/* ------------------------------------------------------------------------------------
 * Sample one token from each of R rows of logits [R][V] (fp32) under the same
 * truncation, by inverse CDF over ascending token id with uniforms[r]; greedy (argmax)
 * when temperature == 0.  This is how a draft model's token is drawn from its truncated
 * distribution q ([MTP-fixes] "Truncation has to match on both sides").
 * out_tokens [R] (device).  Workspace rules as for spec_verify_logits.
 * ---------------------------------------------------------------------------------- */
size_t spec_sample_logits_workspace_bytes(int R, int V);

int spec_sample_logits(int R, int V, const float* logits, const float* uniforms,
                       const spec_sampling* sampling /* host */, int32_t* out_tokens,
                       void* workspace, size_t workspace_bytes, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* SPECVERIFY_H */
