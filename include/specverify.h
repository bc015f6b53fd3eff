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
 *  [OptiQ]     "Speculative decoding on Apple Silicon" (mlx-optiq docs), "N-gram lookup:
 *              any model" (draft what followed an earlier occurrence of the last tokens).
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
 * illegal draft and next_token[b] = -1), SPEC_E_INVAL (the row the final token comes from
 * has nothing to draw from -- sampling from a row without a finite logit; next_token[b]
 * = -1, out_ids of b all -1) or SPEC_E_TIMEOUT (outputs of b undefined).
 *
 * Logits are finite or -inf.  A row of -inf only: greedy takes its lowest id (the
 * argmax tie order); sampling has no distribution there (SPEC_E_INVAL above).  A NaN
 * entry makes that sequence's outputs unspecified, but its ids still lie in [0, V) or
 * are -1.
 * workspace: device scratch of at least spec_verify_logits_workspace_bytes(B, K, V)
 * bytes, 256-byte aligned, owned by the caller; its contents need no initialisation (the
 * call clears what must start at zero with cudaMemsetAsync on `stream`).  Two calls that
 * share a workspace must not overlap on the GPU.
 * Errors: SPEC_E_INVAL for NULL required pointers, B < 1, K < 0, V < 2, K > 64,
 * temperature < 0 or NaN, top_k outside [1, SPEC_TOPK_MAX] with temperature > 0;
 * SPEC_E_RANGE when the B (2K + 1) rows reach 2^30 or their logits 2^40 elements;
 * SPEC_E_NOMEM if workspace_bytes is too small; SPEC_E_CUDA on a launch failure.
 * spec_verify_logits_workspace_bytes returns 0 for sizes the call would reject.
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
 * spec_verify_logits without a caller workspace, for callers that cannot allocate
 * device memory: for example code that runs while a CUDA graph is being captured (where
 * cudaMalloc is not allowed), a serving loop that must not stall on the allocator,
 * or a host that owns a fixed device-memory budget and forbids new allocations.  No
 * counterpart on the pages: this is an interface convenience of this library.
 *
 * Same arguments and outputs as spec_verify_logits, minus the workspace.  The scratch is
 * one fixed array of spec_verify_logits_noalloc_max_bytes() (8 MiB) compiled into the
 * library, present on every GPU that loads it until the process exits; sizes whose
 * workspace (spec_verify_logits_workspace_bytes) exceeds it are rejected with
 * SPEC_E_RANGE.  The call allocates nothing: no cudaMalloc/cudaFree or allocating library
 * routine.  The first call on a device looks up the array's device address once
 * (cudaGetSymbolAddress, with that device current) and caches it: make that first call
 * before any stream capture.  The cached address (like the kernel attributes the
 * library sets once per device) belongs to the device's primary context: after
 * cudaDeviceReset on that device the library is not to be used again in the process.  Every call shares the one array (what must start at zero is
 * cleared on the stream at each call), so calls that overlap on the GPU -- on different
 * streams, or from several host threads -- race and must be serialised by the caller.
 * ---------------------------------------------------------------------------------- */
size_t spec_verify_logits_noalloc_max_bytes(void);

int spec_verify_logits_noalloc(int B, int K, int V,
                               const float* target_logits, const float* draft_logits,
                               const int32_t* draft_tokens, const int32_t* draft_len,
                               const float* uniforms, const spec_sampling* sampling /* host */,
                               int32_t* accepted_len, int32_t* next_token,
                               int32_t* out_ids, float* out_probs, int32_t* seq_status, void* stream);

/* ------------------------------------------------------------------------------------
 * Sample one token from each of R rows of logits [R][V] (fp32) under the same
 * truncation, by inverse CDF over ascending token id with uniforms[r]; greedy (argmax)
 * when temperature == 0.  This is how a draft model's token is drawn from its truncated
 * distribution q ([MTP-fixes] "Truncation has to match on both sides").
 * out_tokens [R] (device); -1 for a row without a finite logit when sampling.  Workspace
 * rules as for spec_verify_logits.
 * ---------------------------------------------------------------------------------- */
size_t spec_sample_logits_workspace_bytes(int R, int V);

int spec_sample_logits(int R, int V, const float* logits, const float* uniforms,
                       const spec_sampling* sampling /* host */, int32_t* out_tokens,
                       void* workspace, size_t workspace_bytes, void* stream);


/* ------------------------------------------------------------------------------------
 * Model context: the target decoder's verify pass, its paged KV cache and the trim.
 *
 * The decoder is the plain dense Llama/Qwen-style reading (the pages name the model
 * families but print no architecture): x = E[tok]; per layer h = RMSNorm(x),
 * q, k, v = h Wq^T, h Wk^T, h Wv^T, rotate-half RoPE on q and k at absolute positions,
 * causal GQA softmax attention (scale 1/sqrt(head_dim)), x += attn Wo^T,
 * x += (silu(RMSNorm(x) Wg^T) * (RMSNorm(x) Wu^T)) Wd^T; logits = RMSNorm(x) Wlm^T.
 * No biases, untied lm_head.  The residual stream is fp32; dtype sets the storage of
 * weights, GEMM inputs and the KV cache.
 *
 * KV cache ([SD-Apple] "Why this needed a patch"): paged, page_tokens = 16 tokens per
 * page, one block table per sequence slot, pages shared by all layers.  The sequence
 * lengths live on the device; a trim is an O(1) length update on the device (the pages
 * past the new length stay reserved and are reclaimed lazily by spec_seq_len /
 * spec_seq_reset).  Convention: before spec_verify the cache holds every committed token
 * of the sequence except the pending one (last_tokens[b]); the pass appends K+1 entries
 * (pending + drafts); keeping a+1 of them commits the pending token and the a accepted
 * drafts, and next_token[b] becomes the new pending token.
 * ---------------------------------------------------------------------------------- */
#define SPEC_F32  0
#define SPEC_BF16 1
#define SPEC_PAGE_TOKENS 16

typedef struct {
    int32_t n_layers, d_model, n_q_heads, n_kv_heads, head_dim, ffn_dim, vocab;
    float rope_theta, rms_eps;
    int32_t dtype;                 /* SPEC_F32 or SPEC_BF16 */
} spec_model_cfg;

typedef struct {
    int32_t max_batch;             /* sequence slots [0, max_batch) */
    int32_t max_ctx;               /* tokens per sequence, pending ones included */
    int32_t max_k;                 /* drafts per verify pass, <= 64 */
    int32_t num_pages;             /* KV pool pages; 0 = max_batch * ceil(max_ctx / 16) */
    int32_t prefill_chunk;         /* tokens per prefill pass; 0 = 128 */
} spec_ctx_limits;

typedef struct spec_ctx spec_ctx;

/* Create a context bound to `stream` (cudaStream_t as void*): allocates the KV pool,
 * activations and workspaces on the current device.  SPEC_E_INVAL on a bad shape
 * (head_dim a multiple of 32 and <= 256, d_model <= 8192, d_model / ffn_dim / heads*head_dim multiples of 8,
 * n_q_heads a multiple of n_kv_heads), SPEC_E_NOMEM when an allocation fails.
 * Concurrency: a tensor-core GEMM of more than 16 tokens whose tiles are shared by several
 * CTAs has those CTAs wait for one another's partial sums (bounded: SPEC_E_TIMEOUT after
 * 2 s), which needs all of its CTAs resident together.  The library's own launches are
 * serialised on the context's stream, so that always holds; passes of two contexts must
 * not run concurrently on different streams (their CTAs could hold the SMs the other's
 * waiting CTAs need until the bound runs out). */
int spec_create(const spec_model_cfg* cfg, const spec_ctx_limits* limits, void* stream, spec_ctx** out);

/* Load the weights.  names[i] is one of "embed" [V][d], "final_norm" [d], "lm_head" [V][d],
 * and per layer l "layers.<l>.attn_norm" [d], ".wq" [hq*hd][d], ".wk" [hkv*hd][d],
 * ".wv" [hkv*hd][d], ".wo" [d][hq*hd], ".ffn_norm" [d], ".wg" [F][d], ".wu" [F][d],
 * ".wd" [d][F]; dev_ptrs[i] a row-major device array of the model dtype, 16-byte aligned.
 * Missing names are SPEC_E_STATE at the first forward.
 * Ownership: float32 models borrow every array (never copied; the caller keeps them
 * alive).  bf16 models on the tensor-core path copy the matrices of the GEMMs (wq, wk, wv,
 * wo, wg, wu, wd, lm_head) once, when the last weight arrives, into a library-owned
 * tile-major buffer (the same bytes in the order the tensor cores consume them, so that
 * a pipeline stage is one contiguous copy) and never read the caller's GEMM matrices
 * again: the caller may free them after this call (spec_weights_copied returns 1), and
 * should, since a second resident copy of the weights is what to avoid ([MTP-fixes]
 * "Duplicate weights in unified memory").  "embed" and the norm gains stay borrowed.
 * Changes the caller makes to its GEMM matrices later are not seen.  SPEC_E_NOMEM when
 * the copy cannot be allocated. */
int spec_load_weights(spec_ctx* ctx, const char* const* names, const void* const* dev_ptrs, int n);

/* 1 when the context holds its own copy of the GEMM matrices (all weights loaded, bf16
 * tensor-core path), so that the caller's GEMM arrays are no longer read; else 0.
 * (No counterpart on the pages: weight ownership of this library.) */
int spec_weights_copied(const spec_ctx* ctx);

/* Ingest tokens[0..n) (device int32) of sequence slot seq_id after what it already holds
 * (chunks of prefill_chunk tokens, the same kernels as the verify pass).  When
 * out_last_logits (device fp32 [V]) is given it receives the logits after the last token.
 * Note the KV convention above: to start a generation, prefill the prompt without its
 * last token and pass that token as the pending one.  Token ids outside [0, V) are
 * embedded as token 0 (the ids are device data, so they are not checked on the host). */
int spec_prefill(spec_ctx* ctx, int seq_id, const int32_t* tokens, int n, float* out_last_logits);

/* The verify pass ([SD-Apple] "How speculative decoding works"; [Draft] "#2"):
 * one batched target forward over [last_tokens[b], draft_tokens[b][0..K)] for the B
 * sequence slots seq_ids[0..B) (HOST array), then the fused verify of
 * spec_verify_logits on the resulting logits (draft_logits [B][K][V] fp32 gives q;
 * NULL = deterministic drafts), then, when auto_trim != 0, the trim to len + a + 1.
 * With auto_trim == 0 the K+1 entries stay and spec_kv_trim does the trim later.
 * Outputs as spec_verify_logits; out_logits (device fp32 [B][K+1][V], may be NULL)
 * receives the target logits.  Greedy (temperature 0) with out_logits NULL on a bf16
 * model: the lm_head GEMM's epilogue keeps, per token, only each 128-row vocabulary
 * tile's largest logit (lowest id on ties) and a merge takes the rows' argmax from those
 * ([MTP-fixes] "Truncation has to match on both sides": the greedy rule needs the argmax
 * alone), so the [B][K+1][V] logits are never written; the outputs are those of the
 * full-logits path, bit for bit.  Ids outside [0, V) are embedded as token 0: a pending
 * token then reads as token 0, and such a draft can never be accepted.  SPEC_E_RANGE when
 * a sequence would exceed max_ctx, SPEC_E_NOMEM when the page pool is exhausted. */
int spec_verify(spec_ctx* ctx, int B, const int32_t* seq_ids, int K,
                const int32_t* last_tokens, const int32_t* draft_tokens, const int32_t* draft_len,
                const float* draft_logits, const float* uniforms, const spec_sampling* sampling,
                int32_t* accepted_len, int32_t* next_token, int32_t* out_ids, float* out_probs,
                int32_t* seq_status, float* out_logits, int auto_trim);

/* Single-token decode of B slots: spec_verify with K = 0 (the token is appended and the
 * next one is drawn from its logits with uniforms[b]).  The comparator of the verify pass.
 * uniforms (device fp32 [B]) is required, also when greedy (then unread).  A row without
 * a finite logit has no distribution to draw from: sampling then writes next_token[b] = -1
 * (no per-sequence status here; spec_verify with K = 0 reports it in seq_status). */
int spec_decode(spec_ctx* ctx, int B, const int32_t* seq_ids, const int32_t* tokens,
                const spec_sampling* sampling, const float* uniforms, int32_t* next_token,
                float* out_logits);

/* Draft K tokens with this (draft) model without returning to the host between them
 * ([SD-Apple] "The original result: Qwen3-8B": the draft's K passes are sequential, a
 * fixed cost per round that grows with K).  Runs the kernels of K spec_decode calls back
 * to back on the device: step i decodes row i's token and draws the next from its logits
 * (truncated as `sampling` says, inverse CDF with uniforms[b][i]; greedy at temperature
 * 0), which is the input of step i + 1.  The K steps are replayed from one CUDA graph per
 * (B, K, sampling, logits wanted), captured on first use.  tokens [B] (device int32): each
 * sequence's pending token; uniforms [B][K] (device fp32, required also when greedy);
 * out_tokens [B][K] (device int32): the drafts d_1..d_K; out_logits [B][K][V] (device
 * fp32, may be NULL): the logits each draft was drawn from (the draft rows of
 * spec_verify).  KV: appends the pending token and d_1..d_{K-1} (K entries), as K
 * spec_decode calls do; the same bits as those calls.  1 <= K <= max_k; errors as
 * spec_verify. */
int spec_draft(spec_ctx* ctx, int B, const int32_t* seq_ids, int K, const int32_t* tokens,
               const spec_sampling* sampling, const float* uniforms, int32_t* out_tokens, float* out_logits);

/* N-gram drafts on the device ([OptiQ] "N-gram lookup: any model": when the last tokens of
 * a sequence occurred earlier in it, draft what followed).  The context of slot
 * seq_ids[b] is its committed tokens (the positions its KV cache holds; the library
 * records each token id as it is embedded) followed by pending[b]: the same rule as
 * spec_ngram_draft on that context -- the longest suffix of max_match down to min_match
 * tokens (1 <= min_match <= max_match <= SPEC_NGRAM_MAX_MATCH) with an earlier
 * occurrence, its most recent occurrence, and the tokens that followed it.
 * drafts [B][n_draft] (device int32, 1 <= n_draft <= 64): the draft, then pending[b] in the
 * rows past it; draft_len [B] (device int32): min(n_draft, cap[b], tokens available), 0
 * when nothing matches; cap [B] (device int32) may be NULL.  pending [B] device.  Feeds
 * spec_verify (last_tokens = pending, draft_tokens = drafts with K = n_draft, draft_len)
 * without a host round trip.  Enqueued on the context's stream. */
int spec_ngram_draft_device(spec_ctx* ctx, int B, const int32_t* seq_ids, const int32_t* pending, int n_draft,
                            int min_match, int max_match, const int32_t* cap, int gated, int32_t* drafts,
                            int32_t* draft_len);

/* The draft-length gate on the device ([OptiQ] "N-gram lookup: any model": the length of a
 * step's draft follows how often recent drafts were accepted, against the timed cost of a
 * verify pass), per sequence slot, with the rule and arithmetic of spec_ngram_gate_* (host,
 * below): alpha = (S + 1) / (S + F + 2), S accepted draft tokens and F first rejections,
 * both multiplied by decay every round; n = the n <= min(n_max, available) with the largest
 * (1 + alpha + ... + alpha^n) / cost[n], the smaller n on ties.
 * config: n_max in [0, 64], cost [n_max + 1] (HOST doubles, > 0), decay in [0, 1]; resets
 * every slot's (S, F) to 0 (spec_seq_reset resets one slot).  Synchronous.
 * update: one round per sequence: drafted[b], accepted[b] (device int32 [B], e.g. the
 * draft_len given to spec_verify and its accepted_len).
 * choose: n_out[b] (device int32 [B]) for available[b] (device int32 [B]) tokens.
 * With gated != 0, spec_ngram_draft_device applies the gate to each sequence's available
 * continuation (the tokens its lookup found, at most n_draft) before cap.  SPEC_E_STATE
 * when the gate is used before config; enqueued on the context's stream. */
int spec_ngram_gate_device_config(spec_ctx* ctx, int n_max, const double* cost, double decay);
int spec_ngram_gate_device_update(spec_ctx* ctx, int B, const int32_t* seq_ids, const int32_t* drafted,
                                  const int32_t* accepted);
int spec_ngram_gate_device_choose(spec_ctx* ctx, int B, const int32_t* seq_ids, const int32_t* available,
                                  int32_t* n_out);

/* Trim after a verify pass run with auto_trim == 0: keep accepted_len[b] + 1 of the
 * K + 1 entries it appended (device O(1) length update).  accepted_len (device int32 [B])
 * is clamped to [0, K], so a trim never reaches below the entries the pass appended. */
int spec_kv_trim(spec_ctx* ctx, int B, const int32_t* seq_ids, int K, const int32_t* accepted_len);

/* Exact length of a slot (synchronises the context stream; reclaims pages past it).
 * Fails with SPEC_E_TIMEOUT as spec_sync does. */
int spec_seq_len(spec_ctx* ctx, int seq_id, int32_t* out_len);

/* Wait for the context's stream, then report the device-side status: SPEC_E_TIMEOUT when
 * a bounded wait inside a kernel (a tensor-core GEMM's pipeline barriers; each gives up
 * after 2 s) gave up since the context was created.  The
 * kernel then skipped the rest of its work, so results since then are unreliable; the
 * status is sticky and the context must be destroyed.  SPEC_E_CUDA on a stream error.
 * (No counterpart on the pages: the library's own failure reporting.) */
int spec_sync(spec_ctx* ctx);

/* Check of the failure path above: launch one bounded wait (the GEMM kernels' own wait
 * helper, with a budget of budget_ms milliseconds, 1..2000) on a barrier that nothing
 * completes.  The wait runs out, records SPEC_E_TIMEOUT in the context's device status
 * word and the kernel returns -- no copy in flight, no tensor memory held -- so the next
 * spec_sync returns SPEC_E_TIMEOUT and the context is spent, while the GPU and other
 * contexts stay usable.  bf16 tensor-core contexts only (SPEC_E_STATE otherwise).
 * (No counterpart on the pages: the library's own failure reporting.) */
int spec_check_wait_timeout(spec_ctx* ctx, int budget_ms);

/* Empty a slot and return its pages to the pool. */
int spec_seq_reset(spec_ctx* ctx, int seq_id);

/* Execution options (both on by default): SPEC_OPT_GRAPHS replays the decoder pass of a
 * (B, K) shape from a CUDA graph captured on first use; SPEC_OPT_PDL lets each GEMM start
 * (barrier set-up, first weight tiles) while the previous kernel finishes.  Neither
 * changes any result bit. */
#define SPEC_OPT_GRAPHS 1
#define SPEC_OPT_PDL    2
/* SPEC_OPT_L2_PREFETCH (value 0..64, default 0 = off): once a GEMM has issued all its loads,
 * each of its CTAs warms L2 with this many 64-column atoms (16 KB each) of the weights it
 * will stream first in the next GEMM of the pass.  Changes no result bit. */
#define SPEC_OPT_L2_PREFETCH 3
/* SPEC_OPT_ATTN_L2_AHEAD (0..64, default 0 = off): on long contexts, where one attention CTA
 * walks a run of 64-key splits, the K and V pages of the split this many splits ahead are
 * prefetched into L2 (bulk prefetch, no shared memory) while the current one is computed.
 * Changes no result bit (measured neutral on 2k-16k contexts). */
#define SPEC_OPT_ATTN_L2_AHEAD 7
/* SPEC_OPT_GEMM_MIN_FILL (percent, 0..101, default 80): a tensor-core GEMM with fewer output
 * tiles than SMs runs as a whole number of CTAs per tile when that keeps at least this share
 * of the SMs busy, else one CTA per SM over equal ranges that cross tile boundaries (101:
 * always the latter).  The split sets the order of the K sums, so it changes result bits
 * (within the rounding of fp32 accumulation), the same way for every token count. */
#define SPEC_OPT_GEMM_MIN_FILL 8
/* SPEC_OPT_GEMM_MAX_SPLIT (0..64, default 0 = no cap): the most CTAs that share one output
 * tile of a tensor-core GEMM with fewer tiles than SMs; with a cap the GEMM runs as that
 * whole number of CTAs per tile (1: one CTA per tile, no fix-up), whatever share of the
 * SMs stays busy.  Like SPEC_OPT_GEMM_MIN_FILL it sets the order of the K sums. */
#define SPEC_OPT_GEMM_MAX_SPLIT 9
int spec_set_option(spec_ctx* ctx, int option, int value);

/* Per-kernel-class timing of the context's passes with CUDA events recorded on its
 * stream around each launch (off by default; meant for a measurement pass).  Classes:
 * 0 QKV GEMM, 1 O GEMM, 2 gate/up GEMM, 3 down GEMM, 4 lm_head GEMM, 5 attention,
 * 6 fused verify, 7 other small kernels. */
#define SPEC_PROF_CLASSES 8
int spec_profile(spec_ctx* ctx, int enable);

/* Synchronise the context stream and return, per class, the summed event time (ms), the
 * number of launches and the algorithmic bytes those launches move (weights for the
 * GEMMs, KV pages read + written for attention, logits for the verify), accumulated since
 * the previous read; then reset.  Arrays of SPEC_PROF_CLASSES entries (host). */
int spec_profile_read(spec_ctx* ctx, double* ms, long long* launches, double* bytes);

/* ------------------------------------------------------------------------------------
 * Host-side n-gram drafter ([OptiQ] "Speculative decoding on Apple Silicon" (mlx-optiq
 * docs), "N-gram lookup: any model").  One object per sequence holds the sequence's
 * committed tokens (host memory) and an index of their m-grams for
 * m in [min_match, max_match].  A draft takes the longest m (max_match down to min_match,
 * at most length - 1) whose last-m-token suffix occurred earlier, and returns the tokens
 * that followed its most recent earlier occurrence, at most n_draft of them; no match
 * drafts nothing.  Host-only: no CUDA calls, no stream.
 *
 * spec_ngram_create: 1 <= min_match <= max_match <= SPEC_NGRAM_MAX_MATCH, else
 *   SPEC_E_INVAL; SPEC_E_NOMEM if the object cannot be allocated.  Destroy with
 *   spec_ngram_destroy (NULL is ignored).
 * spec_ngram_append: append n committed tokens (host array); SPEC_E_NOMEM when the index
 *   cannot grow (the object then holds a prefix of the tokens).
 * spec_ngram_draft: writes the draft to out (host, room for n_draft) and returns its
 *   length (>= 0), or a negative SPEC_E_* code.
 * spec_ngram_draft_batch: drafts for B objects at once into out_tokens (host [B][K],
 *   entries past out_len[b] set to 0) and out_len (host [B]) -- the draft_tokens/draft_len
 *   of one spec_verify call.
 * spec_ngram_length: number of tokens held, or SPEC_E_INVAL for NULL.
 * ---------------------------------------------------------------------------------- */
#define SPEC_NGRAM_MAX_MATCH 8

typedef struct spec_ngram spec_ngram;

int spec_ngram_create(int min_match, int max_match, spec_ngram** out);
int spec_ngram_append(spec_ngram* g, const int32_t* tokens, int n);
int spec_ngram_draft(const spec_ngram* g, int n_draft, int32_t* out);
int spec_ngram_draft_batch(spec_ngram* const* g, int B, int K, int32_t* out_tokens, int32_t* out_len);
int spec_ngram_length(const spec_ngram* g);
void spec_ngram_destroy(spec_ngram* g);

/* Draft-length gate ([OptiQ] "N-gram lookup: any model": the draft length follows how often
 * recent drafts were accepted, against a timed verification pass).  Reading: acceptance
 * alpha = (S + 1) / (S + F + 2) from decayed counts of accepted draft tokens S and first
 * rejections F (both multiplied by `decay` every round, drafts or not); a round drafts the
 * n <= min(n_max, available) maximising (1 + alpha + ... + alpha^n) / cost[n], the
 * smaller n on ties.  cost [n_max + 1] (host): the timed cost of a verify pass with n
 * drafted tokens, any positive unit.  Host-only.
 *
 * spec_ngram_gate_create: SPEC_E_INVAL for n_max outside [0, 1024], decay outside [0, 1]
 *   or a cost that is not finite and positive; SPEC_E_NOMEM if allocation fails.
 * spec_ngram_gate_choose: the draft length for a round whose drafter offers `available`
 *   tokens (>= 0), or SPEC_E_INVAL.
 * spec_ngram_gate_update: after the round: `drafted` tokens were verified and `accepted`
 *   of them kept (0 <= accepted <= drafted, else SPEC_E_INVAL).
 * spec_ngram_gate_acceptance: the current alpha (-1 for NULL). */
typedef struct spec_ngram_gate spec_ngram_gate;

int spec_ngram_gate_create(int n_max, const double* cost, double decay, spec_ngram_gate** out);
int spec_ngram_gate_choose(const spec_ngram_gate* g, int available);
int spec_ngram_gate_update(spec_ngram_gate* g, int drafted, int accepted);
double spec_ngram_gate_acceptance(const spec_ngram_gate* g);
void spec_ngram_gate_destroy(spec_ngram_gate* g);

/* Number of kernels the context launched since creation (for launch accounting). */
long long spec_kernel_launches(const spec_ctx* ctx);

void spec_destroy(spec_ctx* ctx);

#ifdef __cplusplus
}
#endif

#endif /* SPECVERIFY_H */
