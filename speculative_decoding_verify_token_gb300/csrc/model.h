// The model context of the C ABI (spec_ctx) and the launchers of the decoder kernels.
#pragma once

#include <cuda_runtime.h>
#include <cstdint>
#include <string>
#include <vector>

#include "specverify.h"

namespace sv {

constexpr unsigned FULL_MASK = 0xffffffffu;

struct LayerWeights {
    const void *attn_norm = nullptr, *wq = nullptr, *wk = nullptr, *wv = nullptr, *wo = nullptr;
    const void *ffn_norm = nullptr, *wg = nullptr, *wu = nullptr, *wd = nullptr;
};

struct ModelWeights {
    const void *embed = nullptr, *final_norm = nullptr, *lm_head = nullptr;
    std::vector<LayerWeights> layers;
};

struct AttnArgs {
    const void* q;            // [M][hq][hd], or the tensor-core attention's layout (q_np > 0)
    void* o;                  // [M][hq * hd] at act_off(m, col, hq * hd, o_sw_rows)
    const void* k_layer;      // this layer's K pool (kv_off layout)
    const void* v_layer;
    const int* block_table;
    int max_pages;
    const int* seq_ids;       // [B] device
    const int* seq_len;       // [slots] device, length before this pass
    int T, hq, hkv, hd;
    float scale;
    int n_chunks;             // split capacity of the partial buffers
    int split_keys;           // keys per split (multiple of 16, fixed per context)
    float* part_o;            // [B][hkv][n_chunks][T*G][hd]
    float2* part_ml;          // [B][hkv][n_chunks][T*G]
    int* att_cnt;             // [slots * hkv] arrival counters, zero between passes
    size_t q_lo_off;          // split activations: elements from a query (output) value to
    size_t o_lo_off;          // its bf16 lo half; 0 = not split
    int l2_ahead;             // multi-split kernel: splits prefetched into L2 ahead of the copies
    int o_sw_rows;            // layout of o (the O GEMM's operand layout); 0 = row-major
    int kv_sw, num_pages;     // KV pool layout (kv_off)
    int q_np;                 // > 0: queries in q_att_off layout, tensor-core attention
    int* err;                 // device status word for a wait that gave up, or nullptr
};

struct TcGemm;   // tcgen05 GEMM plans (gemm_tc.cu)

// The five GEMMs of the decoder pass.
enum GemmId { GEMM_QKV = 0, GEMM_O = 1, GEMM_GU = 2, GEMM_DOWN = 3, GEMM_LM = 4 };
constexpr int SLOT_RING = 64;   // pinned staging entries for slot-id uploads

struct Ctx {
    spec_model_cfg cfg{};
    spec_ctx_limits lim{};
    cudaStream_t stream = nullptr;
    int esize = 4;
    int device = 0;
    int num_sms = 0;
    ModelWeights w;
    bool weights_ready = false;
    long long launches = 0;

    // paged KV
    int num_pages = 0, max_pages = 0;
    void* k_pool = nullptr;    // [L][P][hkv][16][hd]
    void* v_pool = nullptr;
    size_t layer_pool_elems = 0;
    int* d_block_table = nullptr;   // [slots][max_pages]
    int* h_block_table = nullptr;   // pinned mirror
    int* d_seq_len = nullptr;       // [slots]
    std::vector<int> free_pages;
    std::vector<int> n_pages;       // pages held per slot
    std::vector<int> len_hi;        // upper bound of each slot's device length
    float2* d_rope = nullptr;       // [max_ctx][hd/2]

    // activations
    int Mmax = 0;
    float* X = nullptr;             // [Mmax][d]
    // GEMM inputs and queries; bf16 models hold two halves, [2][Mmax][...] (hi, then the
    // lo remainders, used by the tensor-core path)
    void* Xn = nullptr;             // [Mmax][d]
    void* Q = nullptr;              // [Mmax][hq*hd]
    void* O = nullptr;              // [Mmax][hq*hd]
    void* H = nullptr;              // [Mmax][F]
    bool split = false;             // activations split into bf16 hi + lo (tensor-core path)
    // fused RMSNorm (tensor-core path): per-128-column-tile sums of squares of the residual
    // stream feeding the attention norm (a) and the FFN norm (f), [d/128][Mmax] each
    float* ssq_a = nullptr;
    float* ssq_f = nullptr;
    float* logits = nullptr;        // [Mmax][V]
    int* d_tokens = nullptr;        // [Mmax]
    int* d_tok_seq = nullptr;
    int* d_tok_pos = nullptr;
    int* d_tok_log = nullptr;       // [slots][max_ctx] token id at each position (n-gram context)
    unsigned long long* d_lm_amax = nullptr;   // [Mmax][vocab / 128] per-tile argmax keys (greedy, bf16)
    // draft-length gate on the device: per slot (S, F); cost[0..gate_nmax]; -1 = not configured
    double* d_gate_sf = nullptr;
    double* d_gate_cost = nullptr;
    double gate_decay = 0.9;
    int gate_nmax = -1;
    int* d_seq_ids = nullptr;       // [max_batch]
    int* h_seq_ids = nullptr;       // pinned staging ring [SLOT_RING][max_batch]
    cudaEvent_t ring_ev[SLOT_RING] = {};
    bool ring_used[SLOT_RING] = {};
    int ring_pos = 0;
    int n_chunks = 0;
    float* part_o = nullptr;
    float2* part_ml = nullptr;
    int* att_cnt = nullptr;
    int split_keys = 0;
    // verify
    void* vws = nullptr;
    size_t vws_bytes = 0;
    int* d_status_scratch = nullptr;
    // profiling (events around each launch of a class)
    bool prof_on = false;
    struct ProfRec { int cls; cudaEvent_t a, b; double bytes; };
    std::vector<ProfRec> prof_recs;
    std::vector<cudaEvent_t> prof_pool;
    // CUDA graphs of the decoder pass per (B, T); programmatic dependent launch
    bool use_graphs = true;
    bool use_pdl = true;
    int l2_prefetch_atoms = 0;             // next-GEMM weight atoms per CTA warmed into L2
    int gemm_min_fill = 80;                // percent of the SMs a whole-tile GEMM split must keep busy
    int gemm_max_split = 0;                // most CTAs per output tile (0: no cap)
    cudaStream_t cap_stream = nullptr;     // private stream the graphs are captured on
    struct GraphEntry { int B, T; bool amax; cudaGraphExec_t exec; long long kernels; };
    std::vector<GraphEntry> graphs;
    // device-resident drafting loop (spec_draft): tokens [max_k + 1][max_batch] (row i =
    // the input of step i), uniforms [max_k][max_batch], logits [max_k][max_batch][V], one
    // graph per (B, K, sampling, logits wanted)
    int* d_draft_tok = nullptr;
    float* d_draft_u = nullptr;
    float* d_draft_logits = nullptr;
    int* d_draft_acc = nullptr;
    struct DraftGraph { int B, K, top_k, want_logits; float temperature, top_p; cudaGraphExec_t exec; long long kernels; };
    std::vector<DraftGraph> draft_graphs;
    // tensor-core GEMM
    TcGemm* tc = nullptr;
    bool use_tc = false;
    bool att_tc = false;            // tensor-core attention for passes of <= 96 rows (max_batch > 4)
    int attn_l2_ahead = 0;                 // splits of K/V warmed in L2 ahead (long contexts)
    std::vector<void*> allocs;
};

// kernels
void launch_embed(const Ctx& c, int M, int T, cudaStream_t st, bool fused_norm);
void launch_rmsnorm(const Ctx& c, const float* X, const void* g, void* Xn, int M, cudaStream_t st);
void launch_rope_table(float2* table, int max_pos, int hd, double theta, cudaStream_t st);
void launch_verify_tokens(const int* last, const int* drafts, int K, int* tokens, int B, cudaStream_t st);
void launch_advance_len(const int* seq_ids, int* seq_len, int B, int mode, int add, const int* accepted, int K,
                        cudaStream_t st);
int launch_greedy_amax(const unsigned long long* keys, int n_tiles, int B, int K, const int32_t* draft_tokens,
                       const int32_t* draft_len, int32_t* accepted_len, int32_t* next_token, int32_t* out_ids,
                       float* out_probs, int32_t* seq_status, cudaStream_t st);
void launch_ngram_draft(const Ctx& c, int B, const int* pending, int n_draft, int min_match, int max_match,
                        const int* cap, int* drafts, int* draft_len, bool gated, cudaStream_t st);
void launch_gate_update(const Ctx& c, int B, const int* drafted, const int* accepted, cudaStream_t st);
void launch_gate_choose(const Ctx& c, int B, const int* available, int* n_out, cudaStream_t st);
// dst[c * ldd + r] = src[r * lds + c] for r < R, c < C (int32 / float32)
void launch_transpose_i32(const int* src, int lds, int* dst, int ldd, int R, int C, cudaStream_t st);
void launch_transpose_f32(const float* src, int lds, float* dst, int ldd, int R, int C, cudaStream_t st);
struct EpiArgs;
void launch_gemm_simt(const Ctx& c, const void* wa, const void* wb, const void* wc, int K, int n_pairs,
                      const void* X, const EpiArgs& e, cudaStream_t st);
int launch_attention(const Ctx& c, const AttnArgs& a, int B, int max_len_after, cudaStream_t st);
int attention_set_smem_limits(int hd);
int attention_split_keys(int hd, int esize);
// tensor-core attention (attn_tc.cu): passes of up to 96 query rows per (sequence, kv head)
int attn_tc_split_keys();                    // keys per split
bool attn_tc_fits(int rows);
int attn_tc_set_smem_limits();
void launch_attn_tc(bool pdl, const AttnArgs& a, int nsplit, int B, int sms, cudaStream_t st);

// tcgen05 GEMM (bf16 models)
int tc_create(Ctx& c);                       // tile-major weight copy + workspaces, after weights are loaded
void tc_destroy(Ctx& c);
// returns kernels launched, or a negative SPEC_E_* code; the GEMM reads tokens [x_row0,
// x_row0 + M) (x_row0 a multiple of 16) of its input in the operand layout of a pass of
// pass_M tokens
int tc_gemm(Ctx& c, int gemm_id, int layer, int x_row0, int M, int pass_M, const EpiArgs& e, cudaStream_t st);
bool tc_supported(const Ctx& c);
int tc_error_word(Ctx& c, int* out);          // device error word of the tensor-core GEMM (synchronous)
int* tc_error_ptr(Ctx& c);                    // that word's device address (nullptr without the plan)
int tc_wait_probe(Ctx& c, int budget_ms);     // one bounded wait that runs out (failure-path check)

}  // namespace sv

struct spec_ctx : public sv::Ctx {};
