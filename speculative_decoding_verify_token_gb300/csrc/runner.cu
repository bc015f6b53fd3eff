// Model context of the C ABI: the paged KV cache manager, the decoder pass and the
// verify / decode / prefill / trim entry points.
//
// One pass over B sequences x T tokens (token m = b*T + t):
//   embed -> per layer [RMSNorm -> QKV GEMM (+RoPE, +KV append) -> attention ->
//   O GEMM (+residual) -> RMSNorm -> gate/up GEMM (+SwiGLU) -> down GEMM (+residual)]
//   -> final RMSNorm -> lm_head GEMM (fp32 logits) -> fused verify -> length update.
// The verify pass is the pages' "one batched forward pass" of the target over the pending
// token and the K drafts ("Speculative Decoding on Apple Silicon...", "How speculative
// decoding works"); the trim is the slice of a plain KV cache ("Why this needed a patch
// to mlx_lm at all"), here an O(1) device-side length update.
#include <algorithm>
#include <cmath>
#include <cstring>
#include <string>

#include <cuda_bf16.h>

#include "epilogue.cuh"
#include "host_util.h"
#include "model.h"

namespace sv {

// fused verify entry shared with verify.cu (no workspace allocation, context workspace)
int verify_into(int B, int K, int V, const float* target, const float* draft, const int* draft_tokens,
                const int* draft_len, const float* u, const spec_sampling* s, int* accepted, int* next, int* out_ids,
                float* out_probs, int* status, void* ws, size_t ws_bytes, cudaStream_t st);
int verify_prepare();

static int cuda_fail(const char* what, cudaError_t e) {
    return set_error(SPEC_E_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

template <typename P>
static int dalloc(Ctx& c, P** p, size_t bytes, bool zero = false) {
    void* q = nullptr;
    if (bytes == 0) bytes = 256;
    cudaError_t e = cudaMalloc(&q, bytes);
    if (e != cudaSuccess) return set_error(SPEC_E_NOMEM, "cudaMalloc(%zu) failed: %s", bytes, cudaGetErrorString(e));
    c.allocs.push_back(q);
    if (zero) {
        e = cudaMemset(q, 0, bytes);
        if (e != cudaSuccess) return cuda_fail("cudaMemset", e);
    }
    *p = static_cast<P*>(q);
    return SPEC_OK;
}

static void drop_graphs(Ctx& c) {
    for (auto& g : c.graphs) cudaGraphExecDestroy(g.exec);
    c.graphs.clear();
    for (auto& g : c.draft_graphs) cudaGraphExecDestroy(g.exec);
    c.draft_graphs.clear();
}

static void free_all(Ctx& c) {
    drop_graphs(c);
    if (c.cap_stream) cudaStreamDestroy(c.cap_stream);
    c.cap_stream = nullptr;
    tc_destroy(c);
    for (auto& r : c.prof_recs) { cudaEventDestroy(r.a); cudaEventDestroy(r.b); }
    for (auto e : c.prof_pool) cudaEventDestroy(e);
    c.prof_recs.clear();
    c.prof_pool.clear();
    for (int i = 0; i < SLOT_RING; ++i)
        if (c.ring_ev[i]) cudaEventDestroy(c.ring_ev[i]);
    for (void* p : c.allocs) cudaFree(p);
    c.allocs.clear();
    if (c.h_block_table) cudaFreeHost(c.h_block_table);
    if (c.h_seq_ids) cudaFreeHost(c.h_seq_ids);
    c.h_block_table = nullptr;
    c.h_seq_ids = nullptr;
}

// ---- page management ------------------------------------------------------------------

static int reclaim(Ctx& c) {
    cudaError_t e = cudaStreamSynchronize(c.stream);
    if (e != cudaSuccess) return cuda_fail("cudaStreamSynchronize", e);
    std::vector<int> len(c.lim.max_batch);
    e = cudaMemcpy(len.data(), c.d_seq_len, sizeof(int) * len.size(), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail("cudaMemcpy", e);
    for (int s = 0; s < c.lim.max_batch; ++s) {
        c.len_hi[s] = len[s];
        const int keep = (len[s] + SPEC_PAGE_TOKENS - 1) / SPEC_PAGE_TOKENS;
        while (c.n_pages[s] > keep) {
            --c.n_pages[s];
            c.free_pages.push_back(c.h_block_table[(size_t)s * c.max_pages + c.n_pages[s]]);
        }
    }
    return SPEC_OK;
}

// Make sure the slots have pages for positions < len_hi + T; copies new table entries.
static int ensure_pages(Ctx& c, const int* slots, int B, int T) {
    for (int pass = 0; pass < 2; ++pass) {
        int need_total = 0;
        bool range_ok = true;
        for (int b = 0; b < B; ++b) {
            const int s = slots[b];
            const int need_len = c.len_hi[s] + T;
            if (need_len > c.lim.max_ctx) range_ok = false;
            const int need = (need_len + SPEC_PAGE_TOKENS - 1) / SPEC_PAGE_TOKENS;
            need_total += std::max(0, need - c.n_pages[s]);
        }
        if ((!range_ok || need_total > (int)c.free_pages.size()) && pass == 0) {
            int rc = reclaim(c);
            if (rc != SPEC_OK) return rc;
            continue;
        }
        if (!range_ok) return set_error(SPEC_E_RANGE, "a sequence would exceed max_ctx=%d", c.lim.max_ctx);
        if (need_total > (int)c.free_pages.size())
            return set_error(SPEC_E_NOMEM, "KV page pool exhausted (%d free, %d needed)", (int)c.free_pages.size(),
                             need_total);
        for (int b = 0; b < B; ++b) {
            const int s = slots[b];
            const int need = (c.len_hi[s] + T + SPEC_PAGE_TOKENS - 1) / SPEC_PAGE_TOKENS;
            const int first = c.n_pages[s];
            while (c.n_pages[s] < need) {
                c.h_block_table[(size_t)s * c.max_pages + c.n_pages[s]] = c.free_pages.back();
                c.free_pages.pop_back();
                ++c.n_pages[s];
            }
            if (c.n_pages[s] > first) {
                const size_t off = (size_t)s * c.max_pages + first;
                cudaError_t e = cudaMemcpyAsync(c.d_block_table + off, c.h_block_table + off,
                                                sizeof(int) * (c.n_pages[s] - first), cudaMemcpyHostToDevice, c.stream);
                if (e != cudaSuccess) return cuda_fail("block table copy", e);
            }
        }
        return SPEC_OK;
    }
    return SPEC_OK;
}

static int check_slots(const Ctx& c, const int* slots, int B) {
    if (B < 1 || B > c.lim.max_batch) return set_error(SPEC_E_INVAL, "B=%d outside [1, %d]", B, c.lim.max_batch);
    if (!slots) return set_error(SPEC_E_INVAL, "seq_ids is NULL");
    std::vector<char> seen(c.lim.max_batch, 0);
    for (int b = 0; b < B; ++b) {
        if (slots[b] < 0 || slots[b] >= c.lim.max_batch)
            return set_error(SPEC_E_INVAL, "seq_id %d outside [0, %d)", slots[b], c.lim.max_batch);
        if (seen[slots[b]]) return set_error(SPEC_E_INVAL, "seq_id %d repeated", slots[b]);
        seen[slots[b]] = 1;
    }
    return SPEC_OK;
}

// Copy slot ids to the device through an entry of a pinned staging ring; an entry is
// rewritten only after the event recorded behind its previous copy has completed.
static int upload_slots(Ctx& c, const int* slots, int B) {
    const int i = c.ring_pos;
    c.ring_pos = (c.ring_pos + 1) % SLOT_RING;
    cudaError_t e;
    if (c.ring_used[i]) {
        e = cudaEventSynchronize(c.ring_ev[i]);
        if (e != cudaSuccess) return cuda_fail("cudaEventSynchronize", e);
    }
    int* h = c.h_seq_ids + (size_t)i * c.lim.max_batch;
    std::memcpy(h, slots, sizeof(int) * B);
    e = cudaMemcpyAsync(c.d_seq_ids, h, sizeof(int) * B, cudaMemcpyHostToDevice, c.stream);
    if (e != cudaSuccess) return cuda_fail("seq id copy", e);
    e = cudaEventRecord(c.ring_ev[i], c.stream);
    if (e != cudaSuccess) return cuda_fail("cudaEventRecord", e);
    c.ring_used[i] = true;
    return SPEC_OK;
}

// ---- the decoder pass ---------------------------------------------------------------------

static cudaEvent_t prof_event(Ctx& c) {
    if (!c.prof_pool.empty()) {
        cudaEvent_t e = c.prof_pool.back();
        c.prof_pool.pop_back();
        return e;
    }
    cudaEvent_t e = nullptr;
    cudaEventCreate(&e);
    return e;
}

// Scoped timing of one launch (or a group of launches) of class `cls`.
struct ProfScope {
    Ctx& c;
    int cls;
    double bytes;
    cudaEvent_t a = nullptr;
    ProfScope(Ctx& c_, int cls_, double bytes_) : c(c_), cls(cls_), bytes(bytes_) {
        if (c.prof_on) {
            a = prof_event(c);
            cudaEventRecord(a, c.stream);
        }
    }
    ~ProfScope() {
        if (a) {
            cudaEvent_t b = prof_event(c);
            cudaEventRecord(b, c.stream);
            c.prof_recs.push_back({cls, a, b, bytes});
        }
    }
};

static double gemm_weight_bytes(const Ctx& c, int gid) {
    const spec_model_cfg& m = c.cfg;
    const double d = m.d_model, qd = (double)m.n_q_heads * m.head_dim, kvd = (double)m.n_kv_heads * m.head_dim;
    const double F = m.ffn_dim, V = m.vocab, es = c.esize;
    switch (gid) {
    case GEMM_QKV: return (qd + 2 * kvd) * d * es;
    case GEMM_O: return d * qd * es;
    case GEMM_GU: return 2 * F * d * es;
    case GEMM_DOWN: return d * F * es;
    default: return V * d * es;
    }
}

static inline void* layer_pool(const Ctx& c, void* pool, int l) {
    return static_cast<uint8_t*>(pool) + (size_t)l * c.layer_pool_elems * c.esize;
}

// One GEMM of the pass: on the tensor-core path over tokens [x_row0, x_row0 + e.M) of the
// pass's pass_M tokens (operand layout, see epilogue.cuh), on the SIMT path from X.
static int gemm(Ctx& c, int gid, int layer, const void* wa, const void* wb, const void* wc, int K, int n_pairs,
                const void* X, const EpiArgs& e, int pass_M, int x_row0 = 0) {
    ProfScope ps(c, gid, gemm_weight_bytes(c, gid));
    if (c.use_tc) {
        const int n = tc_gemm(c, gid, layer, x_row0, e.M, pass_M, e, c.stream);
        if (n < 0) return n;
        c.launches += n;
        return SPEC_OK;
    }
    launch_gemm_simt(c, wa, wb, wc, K, n_pairs, X, e, c.stream);
    c.launches += 1;
    return SPEC_OK;
}

// Forward of B x T tokens already in d_tokens for the slots in d_seq_ids.  logits_out gets
// every row ([B*T][V]) or, when last_only, the last row only ([V]); nullptr = no lm_head.
static int forward(Ctx& c, const int* slots, int B, int T, float* logits_out, bool last_only,
                   bool graph_mode = false, bool lm_amax = false) {
    const spec_model_cfg& m = c.cfg;
    const int M = B * T;
    const int d = m.d_model, hd = m.head_dim, hq = m.n_q_heads, hkv = m.n_kv_heads, F = m.ffn_dim;
    cudaStream_t st = c.stream;
    // the tensor-core path folds every RMSNorm into the GEMMs around it (see epilogue.cuh)
    const bool fused = c.use_tc;
    int max_after = 0;
    double kv_bytes = 0.0;    // keys + values read per layer (upper bound of the lengths) + written
    for (int b = 0; b < B; ++b) {
        max_after = std::max(max_after, c.len_hi[slots[b]] + T);
        kv_bytes += (double)(c.len_hi[slots[b]] + 2 * T) * 2.0 * hkv * hd * c.esize;
    }
    if (graph_mode) max_after = c.lim.max_ctx;   // the graph is replayed at any length

    // consumer / producer halves of the fused norm
    auto norm_in = [&](EpiArgs& e, const float* ssq, int row0) {
        if (!fused) return;
        e.ssq_in = ssq; e.n_ssq = d / 128; e.ssq_ld = c.Mmax; e.ssq_row0 = row0;
        e.norm_d = (float)d; e.eps = m.rms_eps;
    };
    auto norm_out = [&](EpiArgs& e, float* ssq, const void* g) {
        if (!fused) return;
        e.xg_out = c.Xn; e.g_next = g; e.ssq_out = ssq; e.ssq_ld = c.Mmax;
    };
    // split activations: the queries' lo halves follow the M hi rows; the GEMM operands
    // (normed rows, attention output, SwiGLU output) are in the operand layout of act_rows(M)
    // rows, lo halves act_rows(M) * 64 elements after the hi ones
    const size_t qlo = c.split ? (size_t)M * hq * hd : 0;
    const int sw = c.use_tc ? act_rows(M) : 0;
    const size_t act_lo = c.split ? (size_t)sw * 64 : 0;
    // the tensor-core attention (batched contexts) takes passes of up to 96 query rows per
    // (sequence, kv head), with the queries in its own layout; the KV pool is in the
    // swizzled layout on the tensor-core path (kv_off)
    const bool att_tc = c.use_tc && c.att_tc && attn_tc_fits(T * (hq / hkv));
    const int q_np = att_tc ? ((T * (hq / hkv) + 15) & ~15) : 0;
    EpiArgs eq{};
    eq.kind = EPI_QKV; eq.M = M; eq.q_out = c.Q; eq.block_table = c.d_block_table; eq.max_pages = c.max_pages;
    eq.tok_seq = c.d_tok_seq; eq.tok_pos = c.d_tok_pos; eq.rope = c.d_rope; eq.hq = hq; eq.hkv = hkv; eq.hd = hd;
    eq.kv_sw = c.use_tc ? 1 : 0; eq.num_pages = c.num_pages; eq.q_np = q_np; eq.q_T = T;
    norm_in(eq, c.ssq_a, 0);
    eq.lo_off = qlo;
    EpiArgs er{};
    er.kind = EPI_RESID; er.M = M; er.x = c.X; er.ldx = d;
    er.lo_off = act_lo; er.sw_rows = sw;
    EpiArgs es{};
    es.kind = EPI_SWIGLU; es.M = M; es.h_out = c.H; es.F = F;
    es.lo_off = act_lo; es.sw_rows = sw;
    norm_in(es, c.ssq_f, 0);
    AttnArgs aa{};
    aa.q = c.Q; aa.o = c.O; aa.block_table = c.d_block_table; aa.max_pages = c.max_pages; aa.seq_ids = c.d_seq_ids;
    aa.seq_len = c.d_seq_len; aa.T = T; aa.hq = hq; aa.hkv = hkv; aa.hd = hd; aa.scale = 1.0f / sqrtf((float)hd);
    aa.n_chunks = c.n_chunks; aa.part_o = c.part_o; aa.part_ml = c.part_ml;
    aa.split_keys = att_tc ? attn_tc_split_keys() : c.split_keys; aa.att_cnt = c.att_cnt;
    aa.kv_sw = eq.kv_sw; aa.num_pages = c.num_pages; aa.q_np = q_np; aa.err = tc_error_ptr(c);
    aa.q_lo_off = qlo; aa.o_lo_off = act_lo; aa.o_sw_rows = sw;
    aa.l2_ahead = c.attn_l2_ahead;

    int rc;
    launch_embed(c, M, T, st, fused);
    c.launches += 1;
    for (int l = 0; l < m.n_layers; ++l) {
        const LayerWeights& L = c.w.layers[l];
        if (!fused) {
            launch_rmsnorm(c, c.X, L.attn_norm, c.Xn, M, st);
            c.launches += 1;
        }
        eq.k_layer = layer_pool(c, c.k_pool, l);
        eq.v_layer = layer_pool(c, c.v_pool, l);
        if ((rc = gemm(c, GEMM_QKV, l, L.wq, L.wk, L.wv, d, (hq + 2 * hkv) * hd / 2, c.Xn, eq, M)) != SPEC_OK) return rc;
        aa.k_layer = eq.k_layer;
        aa.v_layer = eq.v_layer;
        {
            ProfScope ps(c, 5, kv_bytes);
            c.launches += launch_attention(c, aa, B, max_after, st);
        }
        norm_out(er, c.ssq_f, L.ffn_norm);
        if ((rc = gemm(c, GEMM_O, l, L.wo, nullptr, nullptr, hq * hd, d / 2, c.O, er, M)) != SPEC_OK) return rc;
        if (!fused) {
            launch_rmsnorm(c, c.X, L.ffn_norm, c.Xn, M, st);
            c.launches += 1;
        }
        if ((rc = gemm(c, GEMM_GU, l, L.wg, L.wu, nullptr, d, F, c.Xn, es, M)) != SPEC_OK) return rc;
        norm_out(er, c.ssq_a, l + 1 < m.n_layers ? c.w.layers[l + 1].attn_norm : c.w.final_norm);
        if ((rc = gemm(c, GEMM_DOWN, l, L.wd, nullptr, nullptr, F, d / 2, c.H, er, M)) != SPEC_OK) return rc;
    }
    if (logits_out != nullptr) {
        EpiArgs el{};
        el.kind = EPI_STORE; el.x = logits_out; el.ldx = m.vocab;
        if (fused) {
            // the last row alone: the launch covers its 16-row group (operand rows start on
            // a multiple of 16) and stores only that group's last row
            const int r0 = last_only ? ((M - 1) & ~15) : 0;
            el.M = M - r0;
            el.keep_last = last_only ? 1 : 0;
            if (lm_amax && !last_only) {    // per-tile argmax keys instead of the logits
                el.amax_out = c.d_lm_amax;
                el.amax_ld = m.vocab / 128;
            }
            norm_in(el, c.ssq_a, r0);
            if ((rc = gemm(c, GEMM_LM, -1, c.w.lm_head, nullptr, nullptr, d, m.vocab / 2, c.Xn, el, M, r0)) != SPEC_OK)
                return rc;
        } else {
            const int rows = last_only ? 1 : M;
            const size_t off = last_only ? (size_t)(M - 1) : 0;
            launch_rmsnorm(c, c.X + off * d, c.w.final_norm, static_cast<uint8_t*>(c.Xn) + off * d * c.esize, rows, st);
            c.launches += 1;
            el.M = rows;
            if ((rc = gemm(c, GEMM_LM, -1, c.w.lm_head, nullptr, nullptr, d, m.vocab / 2,
                           static_cast<uint8_t*>(c.Xn) + off * d * c.esize, el, M)) != SPEC_OK)
                return rc;
        }
    }
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail("decoder pass launch", e);
    return SPEC_OK;
}

// The decoder pass of B x T tokens through a CUDA graph captured once per (B, T) (logits
// to the internal buffer).  Falls back to eager launches while profiling.
static int forward_graph(Ctx& c, const int* slots, int B, int T, bool lm_amax = false) {
    GraphEntryLookup:
    for (auto& g : c.graphs) {
        if (g.B == B && g.T == T && g.amax == lm_amax) {
            cudaError_t e = cudaGraphLaunch(g.exec, c.stream);
            if (e != cudaSuccess) return cuda_fail("cudaGraphLaunch", e);
            c.launches += g.kernels;
            return SPEC_OK;
        }
    }
    // capture on the context's private stream (the caller's may be the legacy stream, which
    // cannot be captured); the graph is launched on the caller's stream
    cudaGraph_t graph = nullptr;
    cudaStream_t saved = c.stream;
    c.stream = c.cap_stream;
    cudaError_t e = cudaStreamBeginCapture(c.stream, cudaStreamCaptureModeThreadLocal);
    if (e != cudaSuccess) {
        c.stream = saved;
        return cuda_fail("cudaStreamBeginCapture", e);
    }
    const long long l0 = c.launches;
    const int rc = forward(c, slots, B, T, c.logits, false, true, lm_amax);
    const long long n = c.launches - l0;
    c.launches = l0;
    e = cudaStreamEndCapture(c.stream, &graph);
    c.stream = saved;
    if (rc != SPEC_OK) {
        if (graph) cudaGraphDestroy(graph);
        return rc;
    }
    if (e != cudaSuccess) return cuda_fail("cudaStreamEndCapture", e);
    cudaGraphExec_t exec = nullptr;
    e = cudaGraphInstantiate(&exec, graph, 0);
    cudaGraphDestroy(graph);
    if (e != cudaSuccess) return cuda_fail("cudaGraphInstantiate", e);
    c.graphs.push_back({B, T, lm_amax, exec, n});
    goto GraphEntryLookup;
}

// K decode steps of the draft model on the device: step i embeds row i of d_draft_tok,
// runs the decoder pass, samples each sequence's token from its truncated distribution
// with uniform d_draft_u[i][b] (greedy at temperature 0) into row i + 1, copies the step's
// logits to d_draft_logits[i] when wanted, and advances the lengths by one.  Exactly the
// kernels of K spec_decode calls, in the same order, so the drafts are the same bits.
static int draft_steps(Ctx& c, const int* slots, int B, int K, const spec_sampling* s, bool want_logits) {
    const int V = c.cfg.vocab;
    int rc;
    for (int i = 0; i < K; ++i) {
        cudaError_t e = cudaMemcpyAsync(c.d_tokens, c.d_draft_tok + (size_t)i * c.lim.max_batch, sizeof(int) * B,
                                        cudaMemcpyDeviceToDevice, c.stream);
        if (e != cudaSuccess) return cuda_fail("draft token copy", e);
        if ((rc = forward(c, slots, B, 1, c.logits, false, true)) != SPEC_OK) return rc;
        if (want_logits) {
            e = cudaMemcpyAsync(c.d_draft_logits + (size_t)i * c.lim.max_batch * V, c.logits, sizeof(float) * B * V,
                                cudaMemcpyDeviceToDevice, c.stream);
            if (e != cudaSuccess) return cuda_fail("draft logits copy", e);
        }
        rc = verify_into(B, 0, V, c.logits, nullptr, nullptr, nullptr, c.d_draft_u + (size_t)i * c.lim.max_batch, s,
                         c.d_draft_acc, c.d_draft_tok + (size_t)(i + 1) * c.lim.max_batch, nullptr, nullptr,
                         c.d_status_scratch, c.vws, c.vws_bytes, c.stream);
        if (rc != SPEC_OK) return rc;
        launch_advance_len(c.d_seq_ids, c.d_seq_len, B, 0, 1, nullptr, 0, c.stream);
        c.launches += 3;
    }
    cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? SPEC_OK : cuda_fail("draft step launch", e);
}

}  // namespace sv

using namespace sv;

extern "C" int spec_create(const spec_model_cfg* cfg, const spec_ctx_limits* limits, void* stream, spec_ctx** out) {
    clear_error();
    if (!cfg || !limits || !out) return set_error(SPEC_E_INVAL, "NULL argument");
    const spec_model_cfg& m = *cfg;
    if (m.n_layers < 1 || m.d_model < 8 || m.d_model % 8 || m.n_q_heads < 1 || m.n_kv_heads < 1 ||
        m.n_q_heads % m.n_kv_heads || m.head_dim < 32 || m.head_dim % 32 || m.head_dim > 256 ||
        (m.n_q_heads * m.head_dim) % 8 || m.ffn_dim < 8 || m.ffn_dim % 8 || m.vocab < 2 || m.vocab % 2 ||
        m.d_model > 8192 ||
        !(m.rope_theta > 0.0f) || !(m.rms_eps >= 0.0f) || (m.dtype != SPEC_F32 && m.dtype != SPEC_BF16))
        return set_error(SPEC_E_INVAL, "bad model shape");
    spec_ctx_limits lim = *limits;
    if (lim.max_batch < 1 || lim.max_ctx < 2 || lim.max_k < 0 || lim.max_k > 64)
        return set_error(SPEC_E_INVAL, "bad limits");
    if (lim.prefill_chunk <= 0) lim.prefill_chunk = 128;
    lim.prefill_chunk = std::min(lim.prefill_chunk, 256);
    const int max_pages = (lim.max_ctx + SPEC_PAGE_TOKENS - 1) / SPEC_PAGE_TOKENS;
    if (lim.num_pages <= 0) lim.num_pages = lim.max_batch * max_pages;

    spec_ctx* c = new spec_ctx();
    c->cfg = m;
    c->lim = lim;
    c->stream = static_cast<cudaStream_t>(stream);
    c->esize = m.dtype == SPEC_BF16 ? 2 : 4;
    cudaGetDevice(&c->device);
    cudaDeviceGetAttribute(&c->num_sms, cudaDevAttrMultiProcessorCount, c->device);
    c->num_pages = lim.num_pages;
    c->max_pages = max_pages;
    c->w.layers.resize(m.n_layers);
    c->Mmax = std::max(lim.max_batch * (lim.max_k + 1), lim.prefill_chunk);
    // batched contexts take the tensor-core attention (512-key splits); small batches keep
    // the 64-key mma.sync kernel, whose short splits fill the GPU at B = 1.  The choice is
    // fixed per context, so a token's bits never depend on the batch it shares a pass with.
    c->att_tc = lim.max_batch > 4;
    c->split_keys = attention_split_keys(m.head_dim, c->esize);
    c->n_chunks = (lim.max_ctx + c->split_keys - 1) / c->split_keys;
    const size_t qd = (size_t)m.n_q_heads * m.head_dim;
    c->layer_pool_elems = (size_t)lim.num_pages * m.n_kv_heads * SPEC_PAGE_TOKENS * m.head_dim;
    int rc = SPEC_OK;
    auto ok = [&](int r) { rc = r; return r == SPEC_OK; };
    const size_t halves = c->esize == 2 ? 2 : 1;    // bf16: hi and lo halves of the GEMM inputs
    if (!(ok(dalloc(*c, &c->k_pool, c->layer_pool_elems * m.n_layers * c->esize, true)) &&
          ok(dalloc(*c, &c->v_pool, c->layer_pool_elems * m.n_layers * c->esize, true)) &&
          ok(dalloc(*c, &c->d_block_table, sizeof(int) * (size_t)lim.max_batch * max_pages, true)) &&
          ok(dalloc(*c, &c->d_seq_len, sizeof(int) * lim.max_batch, true)) &&
          ok(dalloc(*c, &c->d_rope, sizeof(float2) * (size_t)lim.max_ctx * (m.head_dim / 2))) &&
          ok(dalloc(*c, &c->X, sizeof(float) * (size_t)c->Mmax * m.d_model, true)) &&
          ok(dalloc(*c, &c->Xn, halves * c->esize * act_rows(c->Mmax) * m.d_model, true)) &&
          // + the padding rows of the tensor-core attention's query layout (16 per sequence and kv head)
          ok(dalloc(*c, &c->Q, halves * c->esize * (c->Mmax * qd + (size_t)lim.max_batch * m.n_kv_heads * 16 * 128), true)) &&
          ok(dalloc(*c, &c->O, halves * c->esize * act_rows(c->Mmax) * qd, true)) &&
          ok(dalloc(*c, &c->H, halves * c->esize * act_rows(c->Mmax) * m.ffn_dim, true)) &&
          ok(dalloc(*c, &c->ssq_a, sizeof(float) * (size_t)c->Mmax * ((m.d_model + 127) / 128), true)) &&
          ok(dalloc(*c, &c->ssq_f, sizeof(float) * (size_t)c->Mmax * ((m.d_model + 127) / 128), true)) &&
          ok(dalloc(*c, &c->logits, sizeof(float) * (size_t)c->Mmax * m.vocab)) &&
          ok(dalloc(*c, &c->d_tokens, sizeof(int) * c->Mmax, true)) &&
          ok(dalloc(*c, &c->d_tok_seq, sizeof(int) * c->Mmax, true)) &&
          ok(dalloc(*c, &c->d_tok_pos, sizeof(int) * c->Mmax, true)) &&
          ok(dalloc(*c, &c->d_tok_log, sizeof(int) * (size_t)lim.max_batch * lim.max_ctx, true)) &&
          (m.dtype != SPEC_BF16 ||
           ok(dalloc(*c, &c->d_lm_amax, sizeof(unsigned long long) * (size_t)c->Mmax * (m.vocab / 128 + 1)))) &&
          ok(dalloc(*c, &c->d_seq_ids, sizeof(int) * lim.max_batch, true)) &&
          ok(dalloc(*c, &c->part_o, sizeof(float) * (size_t)c->Mmax * m.n_q_heads * c->n_chunks * m.head_dim)) &&
          ok(dalloc(*c, &c->part_ml, sizeof(float2) * (size_t)c->Mmax * m.n_q_heads * c->n_chunks)) &&
          ok(dalloc(*c, &c->att_cnt, sizeof(int) * (size_t)lim.max_batch * m.n_kv_heads, true)) &&
          ok(dalloc(*c, &c->d_status_scratch, sizeof(int) * lim.max_batch)))) {
        free_all(*c);
        delete c;
        return rc;
    }
    c->vws_bytes = 0;
    for (int b = 1; b <= lim.max_batch; ++b)
        for (int k = 0; k <= lim.max_k; ++k)
            c->vws_bytes = std::max(c->vws_bytes, spec_verify_logits_workspace_bytes(b, k, m.vocab));
    if (!ok(dalloc(*c, &c->vws, c->vws_bytes))) {
        free_all(*c);
        delete c;
        return rc;
    }
    if (cudaMallocHost(reinterpret_cast<void**>(&c->h_block_table), sizeof(int) * (size_t)lim.max_batch * max_pages) !=
            cudaSuccess ||
        cudaMallocHost(reinterpret_cast<void**>(&c->h_seq_ids), sizeof(int) * SLOT_RING * lim.max_batch) !=
            cudaSuccess) {
        free_all(*c);
        delete c;
        return set_error(SPEC_E_NOMEM, "cudaMallocHost failed");
    }
    std::memset(c->h_block_table, 0, sizeof(int) * (size_t)lim.max_batch * max_pages);
    for (int i = 0; i < SLOT_RING; ++i) {
        if (cudaEventCreateWithFlags(&c->ring_ev[i], cudaEventDisableTiming) != cudaSuccess) {
            free_all(*c);
            delete c;
            return set_error(SPEC_E_CUDA, "cudaEventCreate failed");
        }
    }
    c->free_pages.resize(lim.num_pages);
    for (int i = 0; i < lim.num_pages; ++i) c->free_pages[i] = lim.num_pages - 1 - i;
    c->n_pages.assign(lim.max_batch, 0);
    c->len_hi.assign(lim.max_batch, 0);
    if (cudaStreamCreateWithFlags(&c->cap_stream, cudaStreamNonBlocking) != cudaSuccess) {
        free_all(*c);
        delete c;
        return set_error(SPEC_E_CUDA, "cudaStreamCreate failed");
    }
    launch_rope_table(c->d_rope, lim.max_ctx, m.head_dim, (double)m.rope_theta, c->stream);
    if (attention_set_smem_limits(m.head_dim) != 0) {
        free_all(*c);
        delete c;
        return set_error(SPEC_E_CUDA, "attention shared-memory attribute");
    }
    cudaError_t e = cudaStreamSynchronize(c->stream);
    if (e != cudaSuccess) {
        free_all(*c);
        delete c;
        return cuda_fail("spec_create", e);
    }
    *out = c;
    return SPEC_OK;
}

extern "C" int spec_load_weights(spec_ctx* c, const char* const* names, const void* const* ptrs, int n) {
    clear_error();
    if (!c || (n > 0 && (!names || !ptrs))) return set_error(SPEC_E_INVAL, "NULL argument");
    for (int i = 0; i < n; ++i) {
        if (!names[i] || !ptrs[i]) return set_error(SPEC_E_INVAL, "NULL name or pointer at %d", i);
        if (reinterpret_cast<uintptr_t>(ptrs[i]) & 15) return set_error(SPEC_E_INVAL, "%s not 16-byte aligned", names[i]);
        const std::string s(names[i]);
        if (s == "embed") { c->w.embed = ptrs[i]; continue; }
        if (s == "final_norm") { c->w.final_norm = ptrs[i]; continue; }
        if (s == "lm_head") { c->w.lm_head = ptrs[i]; continue; }
        int l = -1;
        char field[32] = {0};
        if (std::sscanf(s.c_str(), "layers.%d.%31s", &l, field) != 2 || l < 0 || l >= c->cfg.n_layers)
            return set_error(SPEC_E_INVAL, "unknown weight name '%s'", names[i]);
        LayerWeights& L = c->w.layers[l];
        const std::string f(field);
        if (f == "attn_norm") L.attn_norm = ptrs[i];
        else if (f == "wq") L.wq = ptrs[i];
        else if (f == "wk") L.wk = ptrs[i];
        else if (f == "wv") L.wv = ptrs[i];
        else if (f == "wo") L.wo = ptrs[i];
        else if (f == "ffn_norm") L.ffn_norm = ptrs[i];
        else if (f == "wg") L.wg = ptrs[i];
        else if (f == "wu") L.wu = ptrs[i];
        else if (f == "wd") L.wd = ptrs[i];
        else return set_error(SPEC_E_INVAL, "unknown weight name '%s'", names[i]);
    }
    bool all = c->w.embed && c->w.final_norm && c->w.lm_head;
    for (const LayerWeights& L : c->w.layers)
        all = all && L.attn_norm && L.wq && L.wk && L.wv && L.wo && L.ffn_norm && L.wg && L.wu && L.wd;
    c->weights_ready = all;
    if (all && c->cfg.dtype == SPEC_BF16) {
        int rc = tc_create(*c);
        if (rc != SPEC_OK) return rc;
    }
    return SPEC_OK;
}

extern "C" int spec_weights_copied(const spec_ctx* c) { return c && c->use_tc ? 1 : 0; }

static int common_checks(spec_ctx* c) {
    if (!c) return set_error(SPEC_E_INVAL, "ctx is NULL");
    if (!c->weights_ready) return set_error(SPEC_E_STATE, "weights not (fully) loaded");
    return SPEC_OK;
}

extern "C" int spec_prefill(spec_ctx* c, int seq_id, const int32_t* tokens, int n, float* out_last_logits) {
    clear_error();
    int rc = common_checks(c);
    if (rc != SPEC_OK) return rc;
    if (seq_id < 0 || seq_id >= c->lim.max_batch) return set_error(SPEC_E_INVAL, "bad seq_id");
    if (n < 1 || !tokens) return set_error(SPEC_E_INVAL, "bad tokens");
    if ((rc = upload_slots(*c, &seq_id, 1)) != SPEC_OK) return rc;
    for (int p0 = 0; p0 < n; p0 += c->lim.prefill_chunk) {
        const int T = std::min(c->lim.prefill_chunk, n - p0);
        if ((rc = ensure_pages(*c, &seq_id, 1, T)) != SPEC_OK) return rc;
        cudaError_t e = cudaMemcpyAsync(c->d_tokens, tokens + p0, sizeof(int) * T, cudaMemcpyDeviceToDevice, c->stream);
        if (e != cudaSuccess) return cuda_fail("token copy", e);
        const bool last = p0 + T == n;
        if ((rc = forward(*c, &seq_id, 1, T, last ? out_last_logits : nullptr, true)) != SPEC_OK) return rc;
        launch_advance_len(c->d_seq_ids, c->d_seq_len, 1, 0, T, nullptr, 0, c->stream);
        c->launches += 1;
        c->len_hi[seq_id] += T;
    }
    cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? SPEC_OK : cuda_fail("spec_prefill", e);
}

extern "C" int spec_verify(spec_ctx* c, int B, const int32_t* seq_ids, int K, const int32_t* last_tokens,
                           const int32_t* draft_tokens, const int32_t* draft_len, const float* draft_logits,
                           const float* uniforms, const spec_sampling* sampling, int32_t* accepted_len,
                           int32_t* next_token, int32_t* out_ids, float* out_probs, int32_t* seq_status,
                           float* out_logits, int auto_trim) {
    clear_error();
    int rc = common_checks(c);
    if (rc != SPEC_OK) return rc;
    if ((rc = check_slots(*c, seq_ids, B)) != SPEC_OK) return rc;
    if (K < 0 || K > c->lim.max_k) return set_error(SPEC_E_INVAL, "K=%d outside [0, %d]", K, c->lim.max_k);
    if (!last_tokens || (K > 0 && !draft_tokens) || !uniforms || !sampling || !accepted_len || !next_token)
        return set_error(SPEC_E_INVAL, "NULL required pointer");
    if ((rc = upload_slots(*c, seq_ids, B)) != SPEC_OK) return rc;
    if ((rc = ensure_pages(*c, seq_ids, B, K + 1)) != SPEC_OK) return rc;
    launch_verify_tokens(last_tokens, draft_tokens, K, c->d_tokens, B, c->stream);
    c->launches += 1;
    // greedy without logits on the tensor-core path: the lm_head epilogue keeps only each
    // 128-row tile's argmax key per token, the [M][V] logits are never written
    const bool amax = c->use_tc && sampling->temperature == 0.0f && out_logits == nullptr && c->d_lm_amax;
    float* logits = out_logits ? out_logits : c->logits;
    if (amax) {
        if (c->use_graphs && !c->prof_on) rc = forward_graph(*c, seq_ids, B, K + 1, true);
        else rc = forward(*c, seq_ids, B, K + 1, c->logits, false, false, true);
        if (rc != SPEC_OK) return rc;
        {
            ProfScope psv(*c, 6, (double)B * (K + 1) * (c->cfg.vocab / 128) * 8.0);
            rc = launch_greedy_amax(c->d_lm_amax, c->cfg.vocab / 128, B, K, draft_tokens, draft_len, accepted_len,
                                    next_token, out_ids, out_probs, seq_status, c->stream);
        }
    } else if (c->use_graphs && !c->prof_on) {
        logits = c->logits;
        if ((rc = forward_graph(*c, seq_ids, B, K + 1)) != SPEC_OK) return rc;
        if (out_logits) {
            cudaError_t e = cudaMemcpyAsync(out_logits, c->logits, sizeof(float) * (size_t)B * (K + 1) * c->cfg.vocab,
                                            cudaMemcpyDeviceToDevice, c->stream);
            if (e != cudaSuccess) return cuda_fail("logits copy", e);
        }
    } else if ((rc = forward(*c, seq_ids, B, K + 1, logits, false)) != SPEC_OK) {
        return rc;
    }
    if (!amax) {
        ProfScope psv(*c, 6, (double)B * (K + 1) * c->cfg.vocab * 4.0 +
                                 (draft_logits && sampling->temperature > 0 ? (double)B * K * c->cfg.vocab * 4.0 : 0.0));
        rc = verify_into(B, K, c->cfg.vocab, logits, draft_logits, draft_tokens, draft_len, uniforms, sampling,
                         accepted_len, next_token, out_ids, out_probs, seq_status, c->vws, c->vws_bytes, c->stream);
    }
    if (rc != SPEC_OK) return rc;
    c->launches += 1;
    if (auto_trim) launch_advance_len(c->d_seq_ids, c->d_seq_len, B, 1, 0, accepted_len, K, c->stream);
    else launch_advance_len(c->d_seq_ids, c->d_seq_len, B, 0, K + 1, nullptr, K, c->stream);
    c->launches += 1;
    for (int b = 0; b < B; ++b) c->len_hi[seq_ids[b]] += K + 1;
    cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? SPEC_OK : cuda_fail("spec_verify", e);
}

extern "C" int spec_decode(spec_ctx* c, int B, const int32_t* seq_ids, const int32_t* tokens,
                           const spec_sampling* sampling, const float* uniforms, int32_t* next_token,
                           float* out_logits) {
    int rc = common_checks(c);
    if (rc != SPEC_OK) return rc;
    if (B < 1 || B > c->lim.max_batch) return set_error(SPEC_E_INVAL, "bad B");
    return spec_verify(c, B, seq_ids, 0, tokens, nullptr, nullptr, nullptr, uniforms, sampling,
                       c->d_status_scratch, next_token, nullptr, nullptr, nullptr, out_logits, 1);
}

extern "C" int spec_draft(spec_ctx* c, int B, const int32_t* seq_ids, int K, const int32_t* tokens,
                          const spec_sampling* sampling, const float* uniforms, int32_t* out_tokens,
                          float* out_logits) {
    clear_error();
    int rc = common_checks(c);
    if (rc != SPEC_OK) return rc;
    if ((rc = check_slots(*c, seq_ids, B)) != SPEC_OK) return rc;
    if (K < 1 || K > c->lim.max_k) return set_error(SPEC_E_INVAL, "K=%d outside [1, %d]", K, c->lim.max_k);
    if (!tokens || !sampling || !uniforms || !out_tokens) return set_error(SPEC_E_INVAL, "NULL required pointer");
    const int V = c->cfg.vocab, Bm = c->lim.max_batch;
    if (!c->d_draft_tok) {
        if ((rc = dalloc(*c, &c->d_draft_tok, sizeof(int) * (size_t)(c->lim.max_k + 1) * Bm, true)) != SPEC_OK ||
            (rc = dalloc(*c, &c->d_draft_u, sizeof(float) * (size_t)c->lim.max_k * Bm, true)) != SPEC_OK ||
            (rc = dalloc(*c, &c->d_draft_logits, sizeof(float) * (size_t)c->lim.max_k * Bm * V)) != SPEC_OK ||
            (rc = dalloc(*c, &c->d_draft_acc, sizeof(int) * (size_t)Bm)) != SPEC_OK)
            return rc;
    }
    if ((rc = upload_slots(*c, seq_ids, B)) != SPEC_OK) return rc;
    if ((rc = ensure_pages(*c, seq_ids, B, K)) != SPEC_OK) return rc;
    // inputs into the context's own buffers (a graph replays fixed addresses): the pending
    // tokens as row 0, the uniforms [B][K] as rows [K][max_batch]
    cudaError_t e = cudaMemcpyAsync(c->d_draft_tok, tokens, sizeof(int) * B, cudaMemcpyDeviceToDevice, c->stream);
    if (e != cudaSuccess) return cuda_fail("token copy", e);
    launch_transpose_f32(uniforms, K, c->d_draft_u, Bm, B, K, c->stream);
    const bool want_logits = out_logits != nullptr;
    const spec_sampling s = *sampling;
    if (!c->use_graphs || c->prof_on) {
        if ((rc = draft_steps(*c, seq_ids, B, K, &s, want_logits)) != SPEC_OK) return rc;
    } else {
        cudaGraphExec_t exec = nullptr;
        for (auto& g : c->draft_graphs)
            if (g.B == B && g.K == K && g.want_logits == (int)want_logits && g.temperature == s.temperature &&
                g.top_k == s.top_k && g.top_p == s.top_p) {
                exec = g.exec;
                c->launches += g.kernels;
                break;
            }
        if (!exec) {
            if ((rc = verify_prepare()) != SPEC_OK) return set_error(SPEC_E_CUDA, "verify kernel attributes");
            // capture on the context's private stream (the caller's may be the legacy stream)
            cudaGraph_t graph = nullptr;
            cudaStream_t saved = c->stream;
            c->stream = c->cap_stream;
            e = cudaStreamBeginCapture(c->stream, cudaStreamCaptureModeThreadLocal);
            if (e != cudaSuccess) {
                c->stream = saved;
                return cuda_fail("cudaStreamBeginCapture", e);
            }
            const long long l0 = c->launches;
            rc = draft_steps(*c, seq_ids, B, K, &s, want_logits);
            const long long n = c->launches - l0;
            e = cudaStreamEndCapture(c->stream, &graph);
            c->stream = saved;
            if (rc != SPEC_OK) {
                if (graph) cudaGraphDestroy(graph);
                return rc;
            }
            if (e != cudaSuccess) return cuda_fail("cudaStreamEndCapture", e);
            e = cudaGraphInstantiate(&exec, graph, 0);
            cudaGraphDestroy(graph);
            if (e != cudaSuccess) return cuda_fail("cudaGraphInstantiate", e);
            c->draft_graphs.push_back({B, K, s.top_k, (int)want_logits, s.temperature, s.top_p, exec, n});
        }
        e = cudaGraphLaunch(exec, c->stream);
        if (e != cudaSuccess) return cuda_fail("cudaGraphLaunch", e);
    }
    // outputs: token rows 1..K -> [B][K]; logits rows [K][max_batch][V] -> [B][K][V]
    launch_transpose_i32(c->d_draft_tok + Bm, Bm, out_tokens, K, K, B, c->stream);
    if (want_logits) {
        for (int i = 0; i < K; ++i) {
            e = cudaMemcpy2DAsync(out_logits + (size_t)i * V, sizeof(float) * (size_t)K * V,
                                  c->d_draft_logits + (size_t)i * Bm * V, sizeof(float) * (size_t)V,
                                  sizeof(float) * (size_t)V, B, cudaMemcpyDeviceToDevice, c->stream);
            if (e != cudaSuccess) return cuda_fail("draft logits copy", e);
        }
    }
    for (int b = 0; b < B; ++b) c->len_hi[seq_ids[b]] += K;
    c->launches += 2;
    e = cudaGetLastError();
    return e == cudaSuccess ? SPEC_OK : cuda_fail("spec_draft", e);
}

extern "C" int spec_ngram_draft_device(spec_ctx* c, int B, const int32_t* seq_ids, const int32_t* pending,
                                       int n_draft, int min_match, int max_match, const int32_t* cap, int gated,
                                       int32_t* drafts, int32_t* draft_len) {
    clear_error();
    if (!c) return set_error(SPEC_E_INVAL, "ctx is NULL");
    int rc = check_slots(*c, seq_ids, B);
    if (rc != SPEC_OK) return rc;
    if (!pending || !drafts || !draft_len) return set_error(SPEC_E_INVAL, "NULL required pointer");
    if (n_draft < 1 || n_draft > 64 || min_match < 1 || max_match < min_match || max_match > SPEC_NGRAM_MAX_MATCH)
        return set_error(SPEC_E_INVAL, "need 1 <= n_draft <= 64 and 1 <= min_match <= max_match <= %d",
                         SPEC_NGRAM_MAX_MATCH);
    if (gated && c->gate_nmax < 0) return set_error(SPEC_E_STATE, "the device gate is not configured");
    if ((rc = upload_slots(*c, seq_ids, B)) != SPEC_OK) return rc;
    launch_ngram_draft(*c, B, pending, n_draft, min_match, max_match, cap, drafts, draft_len, gated != 0, c->stream);
    c->launches += 1;
    const cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? SPEC_OK : cuda_fail("spec_ngram_draft_device", e);
}

extern "C" int spec_ngram_gate_device_config(spec_ctx* c, int n_max, const double* cost, double decay) {
    clear_error();
    if (!c) return set_error(SPEC_E_INVAL, "ctx is NULL");
    if (n_max < 0 || n_max > 64) return set_error(SPEC_E_INVAL, "n_max=%d outside [0, 64]", n_max);
    if (!cost) return set_error(SPEC_E_INVAL, "cost is NULL");
    if (!(decay >= 0.0 && decay <= 1.0)) return set_error(SPEC_E_INVAL, "decay outside [0, 1]");
    for (int n = 0; n <= n_max; ++n)
        if (!(cost[n] > 0.0) || !std::isfinite(cost[n])) return set_error(SPEC_E_INVAL, "cost[%d] must be > 0", n);
    if (!c->d_gate_sf) {
        int rc = dalloc(*c, &c->d_gate_sf, sizeof(double) * 2 * (size_t)c->lim.max_batch, true);
        if (rc == SPEC_OK) rc = dalloc(*c, &c->d_gate_cost, sizeof(double) * 65, true);
        if (rc != SPEC_OK) return rc;
    }
    cudaError_t e = cudaMemcpyAsync(c->d_gate_cost, cost, sizeof(double) * (n_max + 1), cudaMemcpyHostToDevice,
                                    c->stream);
    if (e == cudaSuccess) e = cudaMemsetAsync(c->d_gate_sf, 0, sizeof(double) * 2 * (size_t)c->lim.max_batch, c->stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize(c->stream);
    if (e != cudaSuccess) return cuda_fail("spec_ngram_gate_device_config", e);
    c->gate_nmax = n_max;
    c->gate_decay = decay;
    return SPEC_OK;
}

extern "C" int spec_ngram_gate_device_update(spec_ctx* c, int B, const int32_t* seq_ids, const int32_t* drafted,
                                             const int32_t* accepted) {
    clear_error();
    if (!c) return set_error(SPEC_E_INVAL, "ctx is NULL");
    int rc = check_slots(*c, seq_ids, B);
    if (rc != SPEC_OK) return rc;
    if (!drafted || !accepted) return set_error(SPEC_E_INVAL, "NULL required pointer");
    if (c->gate_nmax < 0) return set_error(SPEC_E_STATE, "the device gate is not configured");
    if ((rc = upload_slots(*c, seq_ids, B)) != SPEC_OK) return rc;
    launch_gate_update(*c, B, drafted, accepted, c->stream);
    c->launches += 1;
    const cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? SPEC_OK : cuda_fail("spec_ngram_gate_device_update", e);
}

extern "C" int spec_ngram_gate_device_choose(spec_ctx* c, int B, const int32_t* seq_ids, const int32_t* available,
                                             int32_t* n_out) {
    clear_error();
    if (!c) return set_error(SPEC_E_INVAL, "ctx is NULL");
    int rc = check_slots(*c, seq_ids, B);
    if (rc != SPEC_OK) return rc;
    if (!available || !n_out) return set_error(SPEC_E_INVAL, "NULL required pointer");
    if (c->gate_nmax < 0) return set_error(SPEC_E_STATE, "the device gate is not configured");
    if ((rc = upload_slots(*c, seq_ids, B)) != SPEC_OK) return rc;
    launch_gate_choose(*c, B, available, n_out, c->stream);
    c->launches += 1;
    const cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? SPEC_OK : cuda_fail("spec_ngram_gate_device_choose", e);
}

extern "C" int spec_kv_trim(spec_ctx* c, int B, const int32_t* seq_ids, int K, const int32_t* accepted_len) {
    clear_error();
    if (!c) return set_error(SPEC_E_INVAL, "ctx is NULL");
    int rc = check_slots(*c, seq_ids, B);
    if (rc != SPEC_OK) return rc;
    if (K < 0 || K > c->lim.max_k || !accepted_len) return set_error(SPEC_E_INVAL, "bad K or accepted_len");
    if ((rc = upload_slots(*c, seq_ids, B)) != SPEC_OK) return rc;
    launch_advance_len(c->d_seq_ids, c->d_seq_len, B, 2, 0, accepted_len, K, c->stream);
    c->launches += 1;
    cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? SPEC_OK : cuda_fail("spec_kv_trim", e);
}

// After the stream has been synchronised: SPEC_E_TIMEOUT when a bounded wait inside a
// tensor-core GEMM gave up since the context was created.  The device word stays set: the
// passes since then may hold wrong values, and so may the GEMMs' tile counters, so the
// context is not to be used again.
static int device_status(Ctx& c) {
    int word = 0;
    if (tc_error_word(c, &word) != SPEC_OK) return set_error(SPEC_E_CUDA, "reading the device error word failed");
    if (word != 0)
        return set_error(SPEC_E_TIMEOUT,
                         "a bounded wait on the device gave up (status %d); results since then are unreliable, "
                         "destroy the context", word);
    return SPEC_OK;
}

extern "C" int spec_sync(spec_ctx* c) {
    clear_error();
    if (!c) return set_error(SPEC_E_INVAL, "ctx is NULL");
    const cudaError_t e = cudaStreamSynchronize(c->stream);
    if (e != cudaSuccess) return cuda_fail("cudaStreamSynchronize", e);
    return device_status(*c);
}

extern "C" int spec_check_wait_timeout(spec_ctx* c, int budget_ms) {
    clear_error();
    if (!c) return set_error(SPEC_E_INVAL, "ctx is NULL");
    if (budget_ms < 1 || budget_ms > 2000) return set_error(SPEC_E_INVAL, "budget_ms=%d outside [1, 2000]", budget_ms);
    return tc_wait_probe(*c, budget_ms);
}

extern "C" int spec_seq_len(spec_ctx* c, int seq_id, int32_t* out_len) {
    clear_error();
    if (!c || !out_len || seq_id < 0 || seq_id >= c->lim.max_batch) return set_error(SPEC_E_INVAL, "bad argument");
    int rc = reclaim(*c);
    if (rc != SPEC_OK) return rc;
    if ((rc = device_status(*c)) != SPEC_OK) return rc;
    *out_len = c->len_hi[seq_id];
    return SPEC_OK;
}

extern "C" int spec_seq_reset(spec_ctx* c, int seq_id) {
    clear_error();
    if (!c || seq_id < 0 || seq_id >= c->lim.max_batch) return set_error(SPEC_E_INVAL, "bad argument");
    cudaError_t e = cudaStreamSynchronize(c->stream);
    if (e != cudaSuccess) return cuda_fail("cudaStreamSynchronize", e);
    e = cudaMemset(c->d_seq_len + seq_id, 0, sizeof(int));
    if (e == cudaSuccess && c->d_gate_sf) e = cudaMemset(c->d_gate_sf + 2 * (size_t)seq_id, 0, 2 * sizeof(double));
    if (e != cudaSuccess) return cuda_fail("cudaMemset", e);
    while (c->n_pages[seq_id] > 0) {
        --c->n_pages[seq_id];
        c->free_pages.push_back(c->h_block_table[(size_t)seq_id * c->max_pages + c->n_pages[seq_id]]);
    }
    c->len_hi[seq_id] = 0;
    return SPEC_OK;
}

extern "C" long long spec_kernel_launches(const spec_ctx* c) { return c ? c->launches : 0; }

extern "C" int spec_set_option(spec_ctx* c, int option, int value) {
    clear_error();
    if (!c) return set_error(SPEC_E_INVAL, "ctx is NULL");
    if (option == SPEC_OPT_GRAPHS) {
        c->use_graphs = value != 0;
    } else if (option == SPEC_OPT_PDL) {
        c->use_pdl = value != 0;
        drop_graphs(*c);
    } else if (option == SPEC_OPT_ATTN_L2_AHEAD) {
        if (value < 0 || value > 64) return set_error(SPEC_E_INVAL, "attention L2 prefetch distance must be in [0, 64]");
        c->attn_l2_ahead = value;
        drop_graphs(*c);
    } else if (option == SPEC_OPT_GEMM_MIN_FILL) {
        if (value < 0 || value > 101) return set_error(SPEC_E_INVAL, "GEMM fill must be in [0, 101] percent");
        c->gemm_min_fill = value;
        drop_graphs(*c);
    } else if (option == SPEC_OPT_GEMM_MAX_SPLIT) {
        if (value < 0 || value > 64) return set_error(SPEC_E_INVAL, "GEMM split cap must be in [0, 64]");
        c->gemm_max_split = value;
        drop_graphs(*c);
    } else if (option == SPEC_OPT_L2_PREFETCH) {
        if (value < 0 || value > 64) return set_error(SPEC_E_INVAL, "L2 prefetch atoms must be in [0, 64]");
        c->l2_prefetch_atoms = value;
        drop_graphs(*c);
    } else {
        return set_error(SPEC_E_INVAL, "unknown option %d", option);
    }
    return SPEC_OK;
}

extern "C" int spec_profile(spec_ctx* c, int enable) {
    clear_error();
    if (!c) return set_error(SPEC_E_INVAL, "ctx is NULL");
    c->prof_on = enable != 0;
    return SPEC_OK;
}

extern "C" int spec_profile_read(spec_ctx* c, double* ms, long long* launches, double* bytes) {
    clear_error();
    if (!c || !ms || !launches || !bytes) return set_error(SPEC_E_INVAL, "NULL argument");
    cudaError_t e = cudaStreamSynchronize(c->stream);
    if (e != cudaSuccess) return cuda_fail("cudaStreamSynchronize", e);
    for (int i = 0; i < SPEC_PROF_CLASSES; ++i) { ms[i] = 0.0; launches[i] = 0; bytes[i] = 0.0; }
    for (const auto& r : c->prof_recs) {
        float t = 0.0f;
        cudaEventElapsedTime(&t, r.a, r.b);
        ms[r.cls] += t;
        launches[r.cls] += 1;
        bytes[r.cls] += r.bytes;
        c->prof_pool.push_back(r.a);
        c->prof_pool.push_back(r.b);
    }
    c->prof_recs.clear();
    return SPEC_OK;
}

extern "C" void spec_destroy(spec_ctx* c) {
    if (!c) return;
    cudaStreamSynchronize(c->stream);
    free_all(*c);
    delete c;
}
