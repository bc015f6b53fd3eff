// Persistent decoder pass for small token counts (M = B*T <= 32).
//
// One cooperative launch, one CTA per SM, runs the whole verify / decode forward: embed,
// then per layer the QKV GEMM (+RoPE, +paged KV append), the attention splits, their
// combine, the O GEMM (+residual), the gate/up GEMM (+SwiGLU) and the down GEMM
// (+residual), then the lm_head GEMM, with the RMSNorms folded into the GEMMs.  Each phase
// does exactly the work of the per-kernel pass -- the same stream-K partition of the
// (tile, K atom) space, the same tcgen05 MMA order, the same fixup order, the same
// attention splits and combine order -- so both passes give the same bits.
//
// What changes is the hand-off between phases.  A kernel boundary becomes a wait on
// counters in global memory that the producing phase bumps after each finished tile
// (release / acquire at GPU scope), and the weights never wait: one producer warp streams
// the weight tiles of the CTA's next K atoms into the shared-memory ring as soon as a slot
// frees, across phase boundaries, while a second producer warp adds the activation tiles
// once the phase's inputs are complete.  A decode or verify step of these models is
// weight streaming ("Speculative Decoding on Apple Silicon: 119% Faster on Qwen3.8",
// "How speculative decoding works"), so HBM keeps streaming through the boundaries.
//
// Every phase only starts its MMAs after the previous phase has finished completely (its
// activation inputs depend on all of it), which is what makes single buffers safe: no
// phase can overwrite a buffer that an earlier phase still reads.  All CTAs are resident
// (cooperative launch) and every wait points to an earlier phase, so no wait can cycle.
// Every wait is bounded by wall-clock time; on expiry the CTA records SPEC_E_TIMEOUT,
// stops, lets its copies in flight land, frees its tensor memory and exits.
#include <algorithm>
#include <vector>

#include "attn_mma.cuh"
#include "host_util.h"
#include "tc_common.cuh"

namespace sv {

constexpr int PF_THREADS = 224;      // warp 0 weights, 1 MMA, 2-5 epilogue + attention, 6 activations
constexpr int PF_MAX_NTOK = 32;
constexpr int PF_MAX_STAGES = 8;
constexpr int PF_SMEM_LIMIT = 232448;   // shared memory of one CTA (static + dynamic)
constexpr int PF_MAX_ATOMS = 4;

enum { CTR_EMBED = 0, CTR_EXIT = 1, CTR_LAYER0 = 2 };

#ifdef PF_TRACE
// Per-CTA, per-phase timeline of the last launch (profiling builds only): [cta][phase][
//  0 first weight stage issued, 1 last weight stage issued, 2 inputs complete (activation
//  producer), 3 first stage ready (MMA), 4 last MMA committed, 5 epilogue done,
//  6 attention start, 7 attention done, 8 combine done, then for the last fixup of the
//  phase: 9 accumulator ready, 10 ticket taken, 11 partials summed, 12 epilogue written,
//  13 released; 14 first attention item inputs ready, 15 first combine row inputs ready,
//  16 first combine row done]
constexpr int PF_TRACE_PH = 4 * 64 + 1;
constexpr int PF_TRACE_EV = 17;
__device__ unsigned long long g_pf_trace[160][PF_TRACE_PH][PF_TRACE_EV];
#define PF_STAMP(ph, i) g_pf_trace[blockIdx.x][(ph)][(i)] = globaltimer_ns()
__device__ __forceinline__ void g_pf_trace_put(int ph, int i, unsigned long long t) { g_pf_trace[blockIdx.x][ph][i] = t; }
#else
#define PF_STAMP(ph, i) ((void)0)
__device__ __forceinline__ void g_pf_trace_put(int, int, unsigned long long) {}
#endif

struct PfParams {
    const CUtensorMap* wmaps;   // [L][7] (q k v o g u d), then lm_head; device memory
    const CUtensorMap* xmaps;   // GEMM inputs Xn, O, H (16-row boxes); device memory
    const void* const* gains;   // [2L + 1]: attn_norm and ffn_norm of each layer, final_norm
    int L, d, hq, hkv, hd, F, V;
    int M, T, B, ntok;
    BRows br;                   // rows of the activation operand (split activations)
    int x_lo_row;               // first lo row of the split activations (= M)
    int stages, atoms, stage_bytes;
    int l2_ahead;               // weight atoms prefetched into L2 ahead of the ring
    EpiArgs eq, eo, es, ed, el;  // epilogues of QKV, O, gate/up, down, lm_head (layer fields set per phase)
    AttnArgs aa;
    size_t layer_pool_bytes;
    uint8_t* k_pool;
    uint8_t* v_pool;
    // embed
    const int* tokens;
    const __nv_bfloat16* embed;
    float* X;
    __nv_bfloat16* Xn;
    float* ssq_a;
    int ssq_ld;
    int* tok_seq;
    int* tok_pos;
    // hand-off counters: [0] embedded rows, [1] exit ticket, then per layer
    // [hkv QKV head groups][B x hkv attention splits][combined rows][O][gate/up][down] tiles
    unsigned* ctr;
    int ctr_stride, ctr_count;
    float* partial;             // [grid][2] x ntok/16 chunks of [4][128] float4 stream-K partial sums
    int* tile_cnt;              // [n_tile_cnt] fixup tickets, zero between launches
    int n_tile_cnt;
    int* err;
};

// ---- phases ---------------------------------------------------------------------------------
// phase ph < 4L: GEMM (ph & 3) of layer ph >> 2 (QKV, O, gate/up, down); ph = 4L: lm_head.

struct PhGeom {
    int gid, layer, n_tiles, KB, G;
    long long T;
    const CUtensorMap* w;
    const CUtensorMap* x;
};

__device__ __forceinline__ PhGeom ph_geom(const PfParams& P, int ph) {
    PhGeom g;
    if (ph == 4 * P.L) {
        g.gid = GEMM_LM; g.layer = -1; g.n_tiles = P.V / TC_BM; g.KB = P.d / TC_ATOM;
        g.w = P.wmaps + 7 * P.L; g.x = P.xmaps;
    } else {
        g.layer = ph >> 2;
        g.gid = ph & 3;
        const CUtensorMap* lw = P.wmaps + 7 * g.layer;
        switch (g.gid) {
        case GEMM_QKV: g.n_tiles = P.hq + 2 * P.hkv; g.KB = P.d / TC_ATOM; g.w = lw; g.x = P.xmaps; break;
        case GEMM_O: g.n_tiles = P.d / TC_BM; g.KB = P.hq * P.hd / TC_ATOM; g.w = lw + 3; g.x = P.xmaps + 1; break;
        case GEMM_GU: g.n_tiles = P.F / 64; g.KB = P.d / TC_ATOM; g.w = lw + 4; g.x = P.xmaps; break;
        default: g.n_tiles = P.d / TC_BM; g.KB = P.F / TC_ATOM; g.w = lw + 6; g.x = P.xmaps + 2; break;
        }
    }
    g.T = (long long)g.n_tiles * g.KB;
    g.G = (int)min((long long)gridDim.x, g.T);   // the per-kernel GEMM's grid: same partition
    return g;
}

__device__ __forceinline__ unsigned* ctr_layer(const PfParams& P, int l) {
    return P.ctr + CTR_LAYER0 + (size_t)l * P.ctr_stride;
}
__device__ __forceinline__ unsigned* ctr_qkv(const PfParams& P, int l, int j) { return ctr_layer(P, l) + j; }
__device__ __forceinline__ unsigned* ctr_att(const PfParams& P, int l, int b, int j) {
    return ctr_layer(P, l) + P.hkv + b * P.hkv + j;
}
__device__ __forceinline__ unsigned* ctr_comb(const PfParams& P, int l) { return ctr_layer(P, l) + P.hkv * (P.B + 1); }
__device__ __forceinline__ unsigned* ctr_o(const PfParams& P, int l) { return ctr_comb(P, l) + 1; }
__device__ __forceinline__ unsigned* ctr_gu(const PfParams& P, int l) { return ctr_comb(P, l) + 2; }
__device__ __forceinline__ unsigned* ctr_down(const PfParams& P, int l) { return ctr_comb(P, l) + 3; }

// What the activation operand of phase ph waits for.
__device__ __forceinline__ void ph_dep(const PfParams& P, int ph, const unsigned*& c, unsigned& target) {
    if (ph == 4 * P.L) {
        c = ctr_down(P, P.L - 1);
        target = (unsigned)(P.d / TC_BM);
        return;
    }
    const int l = ph >> 2;
    switch (ph & 3) {
    case GEMM_QKV:
        if (l == 0) { c = P.ctr + CTR_EMBED; target = (unsigned)P.M; }
        else { c = ctr_down(P, l - 1); target = (unsigned)(P.d / TC_BM); }
        break;
    case GEMM_O: c = ctr_comb(P, l); target = (unsigned)(P.M * P.hq); break;
    case GEMM_GU: c = ctr_o(P, l); target = (unsigned)(P.d / TC_BM); break;
    default: c = ctr_gu(P, l); target = (unsigned)(P.F / 64); break;
    }
}

// Counter bumped when tile `tile` of phase ph is finished (nullptr for the lm_head).
__device__ __forceinline__ unsigned* ph_done(const PfParams& P, int ph, int tile) {
    if (ph == 4 * P.L) return nullptr;
    const int l = ph >> 2;
    switch (ph & 3) {
    case GEMM_QKV: {
        const int j = tile < P.hq ? tile / (P.hq / P.hkv) : (tile < P.hq + P.hkv ? tile - P.hq : tile - P.hq - P.hkv);
        return ctr_qkv(P, l, j);
    }
    case GEMM_O: return ctr_o(P, l);
    case GEMM_GU: return ctr_gu(P, l);
    default: return ctr_down(P, l);
    }
}

__device__ __forceinline__ void ph_epi(const PfParams& P, int ph, EpiArgs& e) {
    if (ph == 4 * P.L) { e = P.el; return; }
    const int l = ph >> 2;
    switch (ph & 3) {
    case GEMM_QKV:
        e = P.eq;
        e.k_layer = P.k_pool + (size_t)l * P.layer_pool_bytes;
        e.v_layer = P.v_pool + (size_t)l * P.layer_pool_bytes;
        break;
    case GEMM_O: e = P.eo; e.g_next = P.gains[2 * l + 1]; break;
    case GEMM_GU: e = P.es; break;
    default: e = P.ed; e.g_next = P.gains[2 * l + 2]; break;
    }
}

// ---- bounded waits ----------------------------------------------------------------------------

__device__ __forceinline__ bool pf_expired(unsigned long long t0, volatile int* abort_flag, int* err) {
    if (*abort_flag) return true;
    if (globaltimer_ns() - t0 > WAIT_BUDGET_NS) {
        *abort_flag = 1;
        atomicExch(err, SPEC_E_TIMEOUT);
        return true;
    }
    return false;
}

__device__ __forceinline__ bool pf_bar_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag, int* err) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = globaltimer_ns();
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if (pf_expired(t0, abort_flag, err)) return false;
    }
}

__device__ __forceinline__ unsigned ld_acquire_u32(const unsigned* p) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ unsigned ld_relaxed_u32(const unsigned* p) {
    unsigned v;
    asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// Wait until *c >= target: relaxed polls with a short backoff (pollers must not crowd the
// weight stream out of the memory system), then one acquire.
__device__ __forceinline__ bool pf_ctr_wait(const unsigned* c, unsigned target, volatile int* abort_flag, int* err) {
    if (ld_acquire_u32(c) >= target) return true;
    const unsigned long long t0 = globaltimer_ns();
    unsigned ns = 32;
    while (true) {
        __nanosleep(ns);
        if (ld_relaxed_u32(c) >= target) {
            asm volatile("fence.acq_rel.gpu;" ::: "memory");
            return true;
        }
        if (ns < 256) ns <<= 1;
        if (pf_expired(t0, abort_flag, err)) return false;
    }
}

// Orders this thread's generic-proxy global writes with later async-proxy (TMA) reads.
__device__ __forceinline__ void fence_proxy_async_global() {
    asm volatile("fence.proxy.async.global;" ::: "memory");
}

// Publish: every writer has passed a barrier before; one thread releases at GPU scope
// (release is cumulative over the writes the barrier ordered before it).
__device__ __forceinline__ void release_bump(unsigned* c) {
    asm volatile("red.release.gpu.global.add.u32 [%0], 1;" :: "l"(c) : "memory");
}

// Fixup ticket: releases this CTA's partial sums, acquires those of the earlier arrivals.
__device__ __forceinline__ int ticket_acq_rel(int* c) {
    int old;
    asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], 1;" : "=r"(old) : "l"(c) : "memory");
    return old;
}

// Next weight atom of the CTA's walk over all phases (the L2 prefetch runs this many atoms
// ahead of the shared-memory ring).
struct AtomCursor {
    int ph = -1;
    PhGeom g;
    long long a = 0, s1 = 0;
    __device__ __forceinline__ void next_phase(const PfParams& P, int cta) {
        while (++ph <= 4 * P.L) {
            g = ph_geom(P, ph);
            if (cta >= g.G) continue;
            a = range_start(g.T, g.G, cta);
            s1 = range_start(g.T, g.G, cta + 1);
            if (a < s1) return;
        }
    }
    __device__ __forceinline__ bool valid(const PfParams& P) const { return ph <= 4 * P.L; }
    __device__ __forceinline__ void prefetch_one(const PfParams& P, int cta) {
        const int tile = (int)(a / g.KB), kt = (int)(a - (long long)tile * g.KB);
        const CUtensorMap *m0, *m1;
        int r0, r1;
        tile_rows_of(g.gid, g.w, P.hq, P.hkv, tile, m0, r0, m1, r1);
        tma_prefetch_l2(m0, kt * TC_ATOM, r0);
        tma_prefetch_l2(m1, kt * TC_ATOM, r1);
        if (++a >= s1) next_phase(P, cta);
    }
};

// ---- roles ------------------------------------------------------------------------------------

struct PfShared {
    uint64_t* full_a;
    uint64_t* full_b;
    uint64_t* empty_bar;
    uint64_t* accf;
    uint64_t* acce;
    volatile int* abort_flag;
    int* flag;                // scratch broadcast flag of the epilogue warps
    float* inv_s;
    float (*red)[TC_CW];
    float* xs;
    AttnSmem att;
    uint32_t base;
};

// Warp 0: weight tiles of every stage of every phase, in order; waits only for free slots.
__device__ __noinline__ long long pf_weights(const PfParams& P, const PfShared& sh) {
    const uint64_t pw = policy_evict_first();
    const int S = P.stages;
    const int cta = blockIdx.x;
    long long i = 0;
    long long loaded = 0, prefetched = 0;   // atoms
    AtomCursor pf;
    pf.next_phase(P, cta);
    for (int ph = 0; ph <= 4 * P.L; ++ph) {
        const PhGeom g = ph_geom(P, ph);
        if (cta >= g.G) continue;
        const long long s0 = range_start(g.T, g.G, cta), s1 = range_start(g.T, g.G, cta + 1);
        StageWalk w(s0, s1, g.KB, P.atoms);
        long long seg0 = s0;
        while (!w.done()) {
            int n, tile, kt;
            bool sf, sl;
            w.cur(n, tile, kt, sf, sl, seg0);
            // keep HBM busy while the ring waits: L2 prefetch of the atoms l2_ahead beyond
            loaded += n;
            while (P.l2_ahead > 0 && prefetched < loaded + P.l2_ahead && pf.valid(P)) {
                pf.prefetch_one(P, cta);
                ++prefetched;
            }
            const int s = (int)(i % S);
            if (!pf_bar_wait(smem_u32(&sh.empty_bar[s]), (uint32_t)(((i / S) & 1) ^ 1), sh.abort_flag, P.err))
                return i;
            const uint32_t fb = smem_u32(&sh.full_a[s]);
            if (w.g == s0) PF_STAMP(ph, 0);
            if (w.g + n >= s1) PF_STAMP(ph, 1);
            mbar_arrive_expect_tx(fb, (uint32_t)(n * TC_ATOM_A));
            const uint32_t a_dst = sh.base + (uint32_t)s * P.stage_bytes;
            const CUtensorMap *m0, *m1;
            int r0, r1;
            tile_rows_of(g.gid, g.w, P.hq, P.hkv, tile, m0, r0, m1, r1);
            for (int at = 0; at < n; ++at) {
                const int kc = (kt + at) * TC_ATOM;
                tma_load_2d(a_dst + at * TC_ATOM_A, m0, kc, r0, fb, pw);
                tma_load_2d(a_dst + at * TC_ATOM_A + TC_ATOM_A / 2, m1, kc, r1, fb, pw);
            }
            ++i;
            w.g += n;
            if (sl) seg0 = w.g;
        }
    }
    return i;
}

// Warp 6: activation tiles, each phase once its inputs are complete.
__device__ __noinline__ long long pf_activations(const PfParams& P, const PfShared& sh) {
    const uint64_t px = policy_evict_last();
    const int S = P.stages;
    const int cta = blockIdx.x;
    const uint32_t b_off = (uint32_t)(P.atoms * TC_ATOM_A);
    const uint32_t per_atom_b = (uint32_t)(P.br.nb * TC_ATOM * 2);
    long long i = 0;
    for (int ph = 0; ph <= 4 * P.L; ++ph) {
        const PhGeom g = ph_geom(P, ph);
        if (cta >= g.G) continue;
        const unsigned* dc;
        unsigned target;
        ph_dep(P, ph, dc, target);
        if (!pf_ctr_wait(dc, target, sh.abort_flag, P.err)) return i;
        PF_STAMP(ph, 2);
        fence_proxy_async_global();
        const long long s0 = range_start(g.T, g.G, cta), s1 = range_start(g.T, g.G, cta + 1);
        StageWalk w(s0, s1, g.KB, P.atoms);
        long long seg0 = s0;
        while (!w.done()) {
            int n, tile, kt;
            bool sf, sl;
            w.cur(n, tile, kt, sf, sl, seg0);
            const int s = (int)(i % S);
            if (!pf_bar_wait(smem_u32(&sh.empty_bar[s]), (uint32_t)(((i / S) & 1) ^ 1), sh.abort_flag, P.err))
                return i;
            const uint32_t fb = smem_u32(&sh.full_b[s]);
            mbar_arrive_expect_tx(fb, (uint32_t)n * per_atom_b);
            const uint32_t b_dst = sh.base + (uint32_t)s * P.stage_bytes + b_off;
            for (int at = 0; at < n; ++at) {
                const int kc = (kt + at) * TC_ATOM;
                const uint32_t b_at = b_dst + at * per_atom_b;
                for (int t = 0; t < P.br.nr0 / 16; ++t)
                    tma_load_2d(b_at + t * 2048, g.x, kc, P.br.b_row0 + t * 16, fb, px);
                if (P.br.b_row1 >= 0)
                    for (int t = 0; t < (P.br.nb - P.br.nr0) / 16; ++t)
                        tma_load_2d(b_at + (P.br.nr0 + t * 16) * 128, g.x, kc, P.br.b_row1 + t * 16, fb, px);
            }
            ++i;
            w.g += n;
            if (sl) seg0 = w.g;
        }
    }
    return i;
}

// Warp 1 (one thread): MMAs of every stage into the double-buffered TMEM accumulators.
__device__ __noinline__ long long pf_mma(const PfParams& P, const PfShared& sh, uint32_t tmem) {
    const int S = P.stages;
    const int cta = blockIdx.x;
    const int acc_cols = P.br.acc_stride;
    const uint32_t idesc = idesc_bf16(P.br.nb);     // at most 64 rows: one MMA
    const uint32_t b_off = (uint32_t)(P.atoms * TC_ATOM_A);
    long long i = 0;
    int si = 0;
    uint32_t d_tmem = tmem;
    for (int ph = 0; ph <= 4 * P.L; ++ph) {
        const PhGeom g = ph_geom(P, ph);
        if (cta >= g.G) continue;
        const long long s0 = range_start(g.T, g.G, cta), s1 = range_start(g.T, g.G, cta + 1);
        StageWalk w(s0, s1, g.KB, P.atoms);
        long long seg0 = s0;
        while (!w.done()) {
            int n, tile, kt;
            bool sf, sl;
            w.cur(n, tile, kt, sf, sl, seg0);
            const int buf = si & 1;
            if (sf) {
                if (!pf_bar_wait(smem_u32(&sh.acce[buf]), (uint32_t)(((si >> 1) & 1) ^ 1), sh.abort_flag, P.err))
                    return i;
                tc_fence_after();
                d_tmem = tmem + (uint32_t)(buf * acc_cols);
            }
            const int s = (int)(i % S);
            const uint32_t par = (uint32_t)((i / S) & 1);
            if (!pf_bar_wait(smem_u32(&sh.full_a[s]), par, sh.abort_flag, P.err) ||
                !pf_bar_wait(smem_u32(&sh.full_b[s]), par, sh.abort_flag, P.err))
                return i;
            tc_fence_after();
            if (w.g == s0) PF_STAMP(ph, 3);
            const uint32_t a_addr = sh.base + (uint32_t)s * P.stage_bytes;
            const uint64_t ad0 = smem_desc_sw128(a_addr), bd0 = smem_desc_sw128(a_addr + b_off);
            const uint64_t a_step = TC_ATOM_A >> 4, b_step = (uint64_t)(P.br.nb * TC_ATOM * 2) >> 4;
            for (int at = 0; at < n; ++at)
                mma_bf16_atom(d_tmem, ad0 + (uint64_t)at * a_step, bd0 + (uint64_t)at * b_step, idesc,
                              (!sf || at > 0) ? 1u : 0u);
            mma_commit(smem_u32(&sh.empty_bar[s]));
            ++i;
            w.g += n;
            if (w.g >= s1) PF_STAMP(ph, 4);
            if (sl) {
                mma_commit(smem_u32(&sh.accf[buf]));
                ++si;
                seg0 = w.g;
            }
        }
    }
    return i;
}

// Epilogue warps: one GEMM phase's accumulators (full tiles, or partial sums and the fixup
// of the last CTA of a tile), then the tile's completion count.  Returns false on abort.
__device__ __noinline__ bool pf_gemm_epilogue(const PfParams& P, const PfShared& sh, int ph, uint32_t tmem,
                                                 int& si) {
    const PhGeom g = ph_geom(P, ph);
    const int cta = blockIdx.x;
    if (cta >= g.G) return true;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int q = warp & 3;
    const int row = q * 32 + lane;
    const int etid = threadIdx.x - 64;
    EpiArgs e;
    ph_epi(P, ph, e);
    // the epilogue reads what earlier phases wrote (residual stream, sums of squares, token
    // positions): acquire the phase's inputs itself (already complete once its first
    // accumulator is ready, so this overlaps the MMAs)
    if (etid == 0) {
        const unsigned* dc;
        unsigned target;
        ph_dep(P, ph, dc, target);
        *sh.flag = pf_ctr_wait(dc, target, sh.abort_flag, P.err) ? 1 : 0;
    }
    epi_bar();
    if (!*sh.flag) return false;
    if (e.ssq_in != nullptr) {
        for (int m = etid; m < P.M; m += 128) {
            const float* src = e.ssq_in + e.ssq_row0 + m;
            float ss = 0.0f;
            for (int t = 0; t < e.n_ssq; ++t) ss += __ldcg(src + (size_t)t * e.ssq_ld);
            sh.inv_s[m] = 1.0f / sqrtf(ss / e.norm_d + e.eps);
        }
    }
    epi_bar();
    const long long T = g.T;
    const int G = g.G;
    const long long s0 = range_start(T, G, cta), s1 = range_start(T, G, cta + 1);
    long long gg = s0;
    while (gg < s1) {
        const int tile = (int)(gg / g.KB);
        const long long tile_k0 = (long long)tile * g.KB;
        const long long seg_end = min(s1, tile_k0 + g.KB);
        const bool full_tile = (gg == tile_k0) && (seg_end == tile_k0 + g.KB);
        const int buf = si & 1;
        const bool okw = pf_bar_wait(smem_u32(&sh.accf[buf]), (uint32_t)((si >> 1) & 1), sh.abort_flag, P.err);
        if (epi_any(okw ? 0 : 1)) return false;
        tc_fence_after();
        unsigned long long t_acc = 0;
#ifdef PF_TRACE
        t_acc = globaltimer_ns();
#endif
        const uint32_t taddr = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(buf * P.br.acc_stride);
        bool finished = false;
        if (full_tile) {
            for (int c0 = 0; c0 < P.ntok; c0 += TC_CW) {
                float v[16];
                acc_ld16(taddr, c0, P.br.lo_col, v);
                if (c0 + TC_CW >= P.ntok) {
                    tc_fence_before();
                    mbar_arrive(smem_u32(&sh.acce[buf]));
                }
#pragma unroll
                for (int j = 0; j < 16; ++j) sh.xs[row * TC_XPITCH + j] = v[j];
                epi_bar();
                epi_chunk(g.gid, P.M, e, sh.xs, sh.inv_s, sh.red, tile, c0, etid);
                epi_bar();
            }
            finished = true;
        } else {
            const int which = (s0 >= tile_k0) ? 0 : 1;
            for (int c0 = 0; c0 < P.ntok; c0 += TC_CW) {
                float v[16];
                acc_ld16(taddr, c0, P.br.lo_col, v);
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    *partial_f4(P.partial, cta, which, P.ntok, c0, j, row) =
                        make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
            }
            tc_fence_before();
            mbar_arrive(smem_u32(&sh.acce[buf]));
            const int c_lo = owner_cta(T, G, tile_k0);
            const int c_hi = owner_cta(T, G, tile_k0 + g.KB - 1);
            epi_bar();
            if (etid == 0) {
                const int prev = ticket_acq_rel(P.tile_cnt + tile);
                *sh.flag = (prev == c_hi - c_lo) ? 1 : 0;
            }
            epi_bar();
            if (*sh.flag) {
                if (etid == 0) { g_pf_trace_put(ph, 9, t_acc); PF_STAMP(ph, 10); }
                const int wc_lo = (range_start(T, G, c_lo) >= tile_k0) ? 0 : 1;
                for (int c0 = 0; c0 < P.ntok; c0 += TC_CW) {
                    float acc[16];
#pragma unroll
                    for (int j = 0; j < 16; ++j) acc[j] = 0.0f;
                    for (int cb = c_lo; cb <= c_hi; cb += 6) {
                        float4 part[6][4];
#pragma unroll
                        for (int u = 0; u < 6; ++u) {
                            const int cc = cb + u;
                            if (cc <= c_hi) {
                                const int wc = cc == c_lo ? wc_lo : 0;
#pragma unroll
                                for (int j = 0; j < 4; ++j)
                                    part[u][j] = __ldcg(partial_f4(P.partial, cc, wc, P.ntok, c0, j, row));
                            }
                        }
#pragma unroll
                        for (int u = 0; u < 6; ++u) {
                            if (cb + u <= c_hi) {
#pragma unroll
                                for (int j = 0; j < 4; ++j) {
                                    acc[4 * j] += part[u][j].x; acc[4 * j + 1] += part[u][j].y;
                                    acc[4 * j + 2] += part[u][j].z; acc[4 * j + 3] += part[u][j].w;
                                }
                            }
                        }
                    }
#pragma unroll
                    for (int j = 0; j < 16; ++j) sh.xs[row * TC_XPITCH + j] = acc[j];
                    epi_bar();
                    if (etid == 0 && c0 == 0) PF_STAMP(ph, 11);
                    epi_chunk(g.gid, P.M, e, sh.xs, sh.inv_s, sh.red, tile, c0, etid);
                    epi_bar();
                }
                if (etid == 0) { P.tile_cnt[tile] = 0; PF_STAMP(ph, 12); }
                finished = true;
            }
            epi_bar();     // every thread has read the flag before it is written again
        }
        if (finished) {
            unsigned* dc = ph_done(P, ph, tile);
            if (dc != nullptr) {
                fence_proxy_async_global();
                epi_bar();
                if (etid == 0) { release_bump(dc); if (!full_tile) PF_STAMP(ph, 13); }
            }
        }
        gg = seg_end;
        ++si;
    }
    if (etid == 0) PF_STAMP(ph, 5);
    return true;
}

// Embedding of the rows m = cta, cta + grid, ...: the embed kernel's arithmetic (a warp per
// 128-column tile), by the 4 epilogue warps.
__device__ __noinline__ void pf_embed(const PfParams& P) {
    const int etid = threadIdx.x - 64;
    const int wl = etid >> 5, lane = threadIdx.x & 31;
    for (int m = blockIdx.x; m < P.M; m += gridDim.x) {
        const int b = m / P.T, t = m - b * P.T;
        int tok = P.tokens[m];
        if (tok < 0 || tok >= P.V) tok = 0;
        if (etid == 0) {
            const int slot = P.aa.seq_ids[b];
            P.tok_seq[m] = slot;
            P.tok_pos[m] = P.aa.seq_len[slot] + t;
        }
        const __nv_bfloat16* row = P.embed + (size_t)tok * P.d;
        const __nv_bfloat16* gain = static_cast<const __nv_bfloat16*>(P.gains[0]);
        float* xr = P.X + (size_t)m * P.d;
        for (int tile = wl; tile < (P.d >> 7); tile += 4) {
            const int c = tile * 128 + lane * 4;
            const uint2 u = *reinterpret_cast<const uint2*>(row + c);
            const float4 v = make_float4(__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xffff0000u),
                                         __uint_as_float(u.y << 16), __uint_as_float(u.y & 0xffff0000u));
            *reinterpret_cast<float4*>(xr + c) = v;
            const uint2 gu = *reinterpret_cast<const uint2*>(gain + c);
            const float4 gg = make_float4(__uint_as_float(gu.x << 16), __uint_as_float(gu.x & 0xffff0000u),
                                          __uint_as_float(gu.y << 16), __uint_as_float(gu.y & 0xffff0000u));
            const float4 y = make_float4(v.x * gg.x, v.y * gg.y, v.z * gg.z, v.w * gg.w);
            __nv_bfloat162 h01 = __floats2bfloat162_rn(y.x, y.y);
            __nv_bfloat162 h23 = __floats2bfloat162_rn(y.z, y.w);
            uint2 o;
            o.x = *reinterpret_cast<uint32_t*>(&h01);
            o.y = *reinterpret_cast<uint32_t*>(&h23);
            *reinterpret_cast<uint2*>(P.Xn + (size_t)m * P.d + c) = o;
            if (P.br.lo_col) {   // bf16 remainders (split activations)
                const float2 f01 = __bfloat1622float2(h01), f23 = __bfloat1622float2(h23);
                __nv_bfloat162 l01 = __floats2bfloat162_rn(y.x - f01.x, y.y - f01.y);
                __nv_bfloat162 l23 = __floats2bfloat162_rn(y.z - f23.x, y.w - f23.y);
                o.x = *reinterpret_cast<uint32_t*>(&l01);
                o.y = *reinterpret_cast<uint32_t*>(&l23);
                *reinterpret_cast<uint2*>(P.Xn + (size_t)P.x_lo_row * P.d + (size_t)m * P.d + c) = o;
            }
            float sq = v.x * v.x;
            sq = fmaf(v.y, v.y, sq);
            sq = fmaf(v.z, v.z, sq);
            sq = fmaf(v.w, v.w, sq);
            sq = warp_sum(sq);
            if (lane == 0) P.ssq_a[(size_t)tile * P.ssq_ld + m] = sq;
        }
        fence_proxy_async_global();
        epi_bar();
        if (etid == 0) release_bump(P.ctr + CTR_EMBED);
    }
}

__device__ __forceinline__ int pf_nsplit(const PfParams& P, int b) {
    return (P.aa.seq_len[P.aa.seq_ids[b]] + P.T + MMA_SPLIT - 1) / MMA_SPLIT;
}

// Attention items (b, kv head j, split s) = cta, cta + grid, ... of layer l.
__device__ __noinline__ bool pf_attention(const PfParams& P, const PfShared& sh, int l) {
    const int etid = threadIdx.x - 64;
    AttnArgs a = P.aa;
    a.k_layer = P.k_pool + (size_t)l * P.layer_pool_bytes;
    a.v_layer = P.v_pool + (size_t)l * P.layer_pool_bytes;
    const unsigned group_tiles = (unsigned)(P.hq / P.hkv + 2);
    int total = 0;
    for (int b = 0; b < P.B; ++b) total += P.hkv * pf_nsplit(P, b);
    if (etid == 0) PF_STAMP(4 * l, 6);
    for (int it = blockIdx.x; it < total; it += gridDim.x) {
        int b = 0, rem = it, ns = 0;
        for (; b < P.B; ++b) {
            ns = pf_nsplit(P, b);
            if (rem < P.hkv * ns) break;
            rem -= P.hkv * ns;
        }
        const int j = rem / ns, s = rem - j * ns;
        const unsigned* dc = ctr_qkv(P, l, j);
        const bool ok = attn_mma_item(
            a, s, j, b, sh.att, etid, [] { epi_bar(); },
            [&]() -> bool {
                if (etid == 0) {
                    *sh.flag = pf_ctr_wait(dc, group_tiles, sh.abort_flag, P.err) ? 1 : 0;
                    if (it == (int)blockIdx.x) PF_STAMP(4 * l, 14);
                }
                epi_bar();
                return *sh.flag != 0;
            });
        if (!ok) return false;
        epi_bar();
        if (etid == 0) release_bump(ctr_att(P, l, b, j));
    }
    if (etid == 0) PF_STAMP(4 * l, 7);
    return true;
}

// Combine rows (b, j, r) = warp index, + 4 grid, ... of layer l.
__device__ __noinline__ bool pf_combine(const PfParams& P, const PfShared& sh, int l) {
    const int lane = threadIdx.x & 31;
    const int wl = (threadIdx.x >> 5) - 2;
    const int R = P.T * (P.hq / P.hkv);
    const int NR = P.B * P.hkv * R;
    int ok = 1;
    for (int rg = blockIdx.x * 4 + wl; rg < NR && ok; rg += gridDim.x * 4) {
        const int b = rg / (P.hkv * R);
        const int rem = rg - b * P.hkv * R;
        const int j = rem / R, r = rem - j * R;
        int got = 1;
        if (lane == 0) got = pf_ctr_wait(ctr_att(P, l, b, j), (unsigned)pf_nsplit(P, b), sh.abort_flag, P.err) ? 1 : 0;
        got = __shfl_sync(FULL, got, 0);
        if (!got) {
            ok = 0;
            break;
        }
        if (threadIdx.x == 64 && rg == (int)blockIdx.x * 4) PF_STAMP(4 * l, 15);
        attn_combine_row_dpl<__nv_bfloat16, 4>(P.aa, r, j, b, lane);     // head_dim 128
        fence_proxy_async_global();
        __syncwarp();
        if (lane == 0) release_bump(ctr_comb(P, l));
        if (threadIdx.x == 64 && rg == (int)blockIdx.x * 4) PF_STAMP(4 * l, 16);
    }
    const bool fail = epi_any(ok ? 0 : 1);
    if (threadIdx.x == 64) PF_STAMP(4 * l, 8);
    return !fail;
}

__global__ void __launch_bounds__(PF_THREADS, 1) pf_kernel(const __grid_constant__ PfParams P) {
    extern __shared__ uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t full_a[PF_MAX_STAGES], full_b[PF_MAX_STAGES], empty_bar[PF_MAX_STAGES];
    __shared__ __align__(8) uint64_t accf[2], acce[2], done_bar;
    __shared__ uint32_t tmem_sh;
    __shared__ int flag, last_cta;
    __shared__ volatile int abort_flag;
    __shared__ long long n_issued_a, n_issued_b, n_consumed;
    __shared__ float inv_s[PF_MAX_NTOK];
    __shared__ float red_s[4][TC_CW];
    __shared__ float wmax[4][MMA_RT], wsum[4][MMA_RT];

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t base = (smem_u32(smem_raw) + 1023u) & ~1023u;
    uint8_t* gbase = smem_raw + (base - smem_u32(smem_raw));
    PfShared sh;
    sh.full_a = full_a; sh.full_b = full_b; sh.empty_bar = empty_bar; sh.accf = accf; sh.acce = acce;
    sh.abort_flag = &abort_flag;
    sh.flag = &flag;
    sh.inv_s = inv_s;
    sh.red = red_s;
    sh.base = base;
    sh.xs = reinterpret_cast<float*>(gbase + (size_t)P.stages * P.stage_bytes);
    sh.att.Ks = reinterpret_cast<__nv_bfloat16*>(gbase + (size_t)P.stages * P.stage_bytes + TC_XBYTES);
    sh.att.Vs = sh.att.Ks + MMA_SPLIT * MMA_PITCH;
    sh.att.Qs = sh.att.Vs + MMA_SPLIT * MMA_PITCH;
    sh.att.Qlo = sh.att.Qs + MMA_RT * MMA_PITCH;
    sh.att.Ps = sh.att.Qlo + MMA_RT * MMA_PITCH;
    sh.att.wmax = wmax;
    sh.att.wsum = wsum;
    const int acc_cols = P.br.acc_stride;
    const uint32_t ncols = (uint32_t)max(32, 1 << (32 - __clz(2 * acc_cols - 1)));

    if (threadIdx.x == 0) {
        for (int s = 0; s < P.stages; ++s) {
            mbar_init(smem_u32(&full_a[s]), 1);
            mbar_init(smem_u32(&full_b[s]), 1);
            mbar_init(smem_u32(&empty_bar[s]), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(smem_u32(&accf[b]), 1);
            mbar_init(smem_u32(&acce[b]), 128);
        }
        mbar_init(smem_u32(&done_bar), 1);
        abort_flag = 0;
        n_issued_a = n_issued_b = n_consumed = 0;
        fence_barrier_init();
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                     :: "r"(smem_u32(&tmem_sh)), "r"(ncols) : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_sh;

    if (warp == 0) {
        if (lane == 0) n_issued_a = pf_weights(P, sh);
    } else if (warp == 1) {
        if (lane == 0) {
            n_consumed = pf_mma(P, sh, tmem);
            // no MMA may still write tensor memory when it is freed
            mma_commit(smem_u32(&done_bar));
            mbar_wait(smem_u32(&done_bar), 0);
        }
    } else if (warp == 6) {
        if (lane == 0) n_issued_b = pf_activations(P, sh);
    } else {
        int si = 0;
        pf_embed(P);
        bool ok = true;
        for (int l = 0; l < P.L && ok; ++l) {
            ok = pf_gemm_epilogue(P, sh, 4 * l + GEMM_QKV, tmem, si) && pf_attention(P, sh, l) &&
                 pf_combine(P, sh, l) && pf_gemm_epilogue(P, sh, 4 * l + GEMM_O, tmem, si) &&
                 pf_gemm_epilogue(P, sh, 4 * l + GEMM_GU, tmem, si) &&
                 pf_gemm_epilogue(P, sh, 4 * l + GEMM_DOWN, tmem, si);
        }
        if (ok) pf_gemm_epilogue(P, sh, 4 * P.L, tmem, si);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (abort_flag) {
        // copies issued for stages the MMA never consumed must land before the CTA exits
        const int S = P.stages;
        if (threadIdx.x == 0)
            for (long long k = n_consumed; k < n_issued_a; ++k)
                mbar_wait(smem_u32(&full_a[k % S]), (uint32_t)((k / S) & 1));
        if (threadIdx.x == 192)
            for (long long k = n_consumed; k < n_issued_b; ++k)
                mbar_wait(smem_u32(&full_b[k % S]), (uint32_t)((k / S) & 1));
        __syncthreads();
    }
    if (warp == 1)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" :: "r"(tmem), "r"(ncols) : "memory");
    // the last CTA out clears the hand-off counters (and, after an error, the fixup tickets)
    if (threadIdx.x == 0) {
        __threadfence();
        last_cta = atomicAdd(P.ctr + CTR_EXIT, 1u) == gridDim.x - 1 ? 1 : 0;
    }
    __syncthreads();
    if (last_cta) {
        __threadfence();
        for (int i = threadIdx.x; i < P.ctr_count; i += PF_THREADS) P.ctr[i] = 0;
        if (*reinterpret_cast<volatile int*>(P.err) != 0)
            for (int i = threadIdx.x; i < P.n_tile_cnt; i += PF_THREADS) P.tile_cnt[i] = 0;
    }
}

// ---- host side ----------------------------------------------------------------------------------

#ifdef PF_TRACE
extern "C" int spec_debug_pf_trace(unsigned long long* out, int* dims) {
    dims[0] = 160; dims[1] = PF_TRACE_PH; dims[2] = PF_TRACE_EV;
    return cudaMemcpyFromSymbol(out, g_pf_trace, sizeof(g_pf_trace)) == cudaSuccess ? 0 : -6;
}
#endif

struct PfPlan {
    CUtensorMap* wmaps = nullptr;    // device [7L + 1]
    CUtensorMap* xmaps = nullptr;    // device [3]
    const void** gains = nullptr;    // device [2L + 1]
    unsigned* ctr = nullptr;
    int ctr_stride = 0, ctr_count = 0;
    int static_smem = 0;
};

int tc_export(const Ctx& c, CUtensorMap* wmaps, CUtensorMap* xmaps, float** partial, int** tile_cnt, int* n_tile_cnt,
              int** err);

void pf_destroy(Ctx& c) {
    if (!c.pf) return;
    cudaFree(c.pf->wmaps);
    cudaFree(c.pf->xmaps);
    cudaFree(c.pf->gains);
    cudaFree(c.pf->ctr);
    delete c.pf;
    c.pf = nullptr;
}

// Plans the persistent pass (after tc_create); leaves c.pf null when the device cannot run
// it (no cooperative launch, or the CTA does not fit on an SM).
int pf_create(Ctx& c) {
    if (!c.use_tc || c.pf) return SPEC_OK;
    int coop = 0;
    if (cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, c.device) != cudaSuccess || !coop) return SPEC_OK;
    cudaFuncAttributes fa;
    if (cudaFuncGetAttributes(&fa, pf_kernel) != cudaSuccess) return SPEC_OK;
    const spec_model_cfg& m = c.cfg;
    const int L = m.n_layers;
    std::vector<CUtensorMap> w((size_t)7 * L + 1), x(3);
    float* partial;
    int *tile_cnt, n_tile_cnt, *err;
    int rc = tc_export(c, w.data(), x.data(), &partial, &tile_cnt, &n_tile_cnt, &err);
    if (rc != SPEC_OK) return rc;
    std::vector<const void*> g((size_t)2 * L + 1);
    for (int l = 0; l < L; ++l) {
        g[2 * l] = c.w.layers[l].attn_norm;
        g[2 * l + 1] = c.w.layers[l].ffn_norm;
    }
    g[2 * L] = c.w.final_norm;
    PfPlan* p = new PfPlan();
    p->ctr_stride = m.n_kv_heads * (c.lim.max_batch + 1) + 4;
    p->ctr_count = CTR_LAYER0 + L * p->ctr_stride;
    p->static_smem = (int)fa.sharedSizeBytes;
    bool ok = cudaMalloc(&p->wmaps, sizeof(CUtensorMap) * w.size()) == cudaSuccess &&
              cudaMalloc(&p->xmaps, sizeof(CUtensorMap) * x.size()) == cudaSuccess &&
              cudaMalloc(&p->gains, sizeof(void*) * g.size()) == cudaSuccess &&
              cudaMalloc(&p->ctr, sizeof(unsigned) * p->ctr_count) == cudaSuccess;
    ok = ok && cudaMemcpy(p->wmaps, w.data(), sizeof(CUtensorMap) * w.size(), cudaMemcpyHostToDevice) == cudaSuccess &&
         cudaMemcpy(p->xmaps, x.data(), sizeof(CUtensorMap) * x.size(), cudaMemcpyHostToDevice) == cudaSuccess &&
         cudaMemcpy(p->gains, g.data(), sizeof(void*) * g.size(), cudaMemcpyHostToDevice) == cudaSuccess &&
         cudaMemset(p->ctr, 0, sizeof(unsigned) * p->ctr_count) == cudaSuccess;
    const int dyn_max = PF_SMEM_LIMIT - p->static_smem;
    ok = ok && cudaFuncSetAttribute(pf_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, dyn_max) == cudaSuccess;
    int blocks = 0;
    ok = ok && cudaOccupancyMaxActiveBlocksPerMultiprocessor(&blocks, pf_kernel, PF_THREADS, dyn_max) == cudaSuccess &&
         blocks >= 1;
    c.pf = p;
    if (!ok) {
        cudaGetLastError();
        pf_destroy(c);
        return SPEC_OK;       // not an error: the per-kernel pass runs instead
    }
    return SPEC_OK;
}

bool pf_usable(const Ctx& c, int M) { return c.pf != nullptr && c.use_pf && M >= 1 && M <= PF_MAX_NTOK; }

int pf_launch(Ctx& c, int B, int T, const EpiArgs& eq, const EpiArgs& eo, const EpiArgs& es, const EpiArgs& ed,
              const EpiArgs& el, const AttnArgs& aa, cudaStream_t st) {
    const spec_model_cfg& m = c.cfg;
    PfPlan* pl = c.pf;
    PfParams P{};
    P.wmaps = pl->wmaps;
    P.xmaps = pl->xmaps;
    P.gains = pl->gains;
    P.L = m.n_layers; P.d = m.d_model; P.hq = m.n_q_heads; P.hkv = m.n_kv_heads; P.hd = m.head_dim;
    P.F = m.ffn_dim; P.V = m.vocab;
    P.M = B * T; P.T = T; P.B = B;
    P.ntok = (P.M + 15) & ~15;
    P.br = b_rows(c.split, P.M, 0, P.M);
    P.x_lo_row = P.M;
    const int per_atom = TC_ATOM_A + P.br.nb * TC_ATOM * 2;
    const int budget = PF_SMEM_LIMIT - pl->static_smem - 1024 - TC_XBYTES - (int)MMA_SMEM;
    P.atoms = std::max(1, std::min(PF_MAX_ATOMS, c.pf_atoms));
    while (P.atoms > 1 && budget / (P.atoms * per_atom) < 2) P.atoms >>= 1;
    P.stage_bytes = P.atoms * per_atom;
    P.l2_ahead = c.pf_l2_ahead;
    P.stages = std::min(PF_MAX_STAGES, budget / P.stage_bytes);
    if (P.stages < 2) return set_error(SPEC_E_RANGE, "persistent pass: stage does not fit in shared memory");
    P.eq = eq; P.eo = eo; P.es = es; P.ed = ed; P.el = el;
    P.aa = aa;
    P.layer_pool_bytes = c.layer_pool_elems * c.esize;
    P.k_pool = static_cast<uint8_t*>(c.k_pool);
    P.v_pool = static_cast<uint8_t*>(c.v_pool);
    P.tokens = c.d_tokens;
    P.embed = static_cast<const __nv_bfloat16*>(c.w.embed);
    P.X = c.X;
    P.Xn = static_cast<__nv_bfloat16*>(c.Xn);
    P.ssq_a = c.ssq_a;
    P.ssq_ld = c.Mmax;
    P.tok_seq = c.d_tok_seq;
    P.tok_pos = c.d_tok_pos;
    P.ctr = pl->ctr;
    P.ctr_stride = pl->ctr_stride;
    P.ctr_count = pl->ctr_count;
    int rc = tc_export(c, nullptr, nullptr, &P.partial, &P.tile_cnt, &P.n_tile_cnt, &P.err);
    if (rc != SPEC_OK) return rc;
    const size_t smem = 1024 + (size_t)P.stages * P.stage_bytes + TC_XBYTES + MMA_SMEM;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(c.num_sms);
    cfg.blockDim = dim3(PF_THREADS);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, pf_kernel, P);
    if (e != cudaSuccess) return set_error(SPEC_E_CUDA, "persistent pass launch: %s", cudaGetErrorString(e));
    return 1;
}

}  // namespace sv
