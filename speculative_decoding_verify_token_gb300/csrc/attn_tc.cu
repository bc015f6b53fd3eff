// Multi-query causal GQA attention over the paged KV cache on the 5th-generation tensor
// cores (tcgen05), for passes of up to 96 query rows per (sequence, kv head): the verify
// pass (T = K + 1 tokens x G query heads), single-token decode and the drafting loop
// ("What is Speculative Decoding and How Does a Draft Model Work?", section "#3": the K+1
// positions are scored in one target pass; "Speculative Decoding on Apple Silicon...",
// section "How speculative decoding works": one pass over the cache serves all of them).
//
// Work items are (512-key split, kv head, sequence), four 128-key tiles each, taken by
// persistent CTAs (one per SM) so that the K and V of later items stream in while earlier
// ones are in their softmax (used by contexts sized for batched serving; small batches keep
// the 64-key mma.sync kernel, whose many short splits fill the GPU at B = 1).  Per item:
//  * S^T = K Q^T with the keys as the MMA's M (128 rows, every row used) and the query rows
//    as N (the rows padded to np = 16..96): A = a K tile straight from the cache (the pool
//    is kept in the swizzled per-head layout, so a run of consecutive pages is one bulk
//    copy), B = the queries as bf16 hi + lo halves accumulated into the same columns;
//  * the split's S tiles stay in tensor memory; the softmax warps take the rows' maxima over
//    the whole split first (one thread per key, shuffles and a fixed cross-warp order),
//    then write P = 2^(s - m) per tile as bf16 hi + lo halves (the probabilities need
//    about 16 significant bits: rounded to bf16 alone they moved the logits of one
//    8B-width layer by up to 1e-2) into shared memory as the next MMA's B operand;
//  * O^T += V^T P^T with V^T as an MN-major A operand (the same V tile, read transposed
//    by the tensor core) and the output in tensor memory; no rescaling, since the maxima
//    are final before the first P;
//  * the split's (max, sum, unnormalised output) per row go to the partial buffers that
//    the combine kernel reduces in a fixed order.
// Across items: a ring of 32 KB K/V tile slots (3-6, as shared memory allows), two query
// buffers (a query buffer holds the item's P once its QK MMAs are done), and for up to 48
// rows two sets of S and O columns in tensor memory, so that QK of item n + 1 runs while
// the softmax of item n does; P V of item n then follows QK of item n + 1.
// Every row's arithmetic depends only on its own position and the split boundaries (fixed
// multiples of 512), not on np, T or the batch: a token gets the same bits decoded alone
// or verified with K drafts.
#include <cuda_bf16.h>
#include <algorithm>
#include <cmath>

#include "tc_common.cuh"

namespace sv {

constexpr int AT_TILE = 128;                    // keys per tile (the QK MMA's M)
constexpr int AT_TILES = 4;
constexpr int AT_SPLIT = AT_TILES * AT_TILE;    // keys per split (CTA)
constexpr int AT_SLOT_BYTES = 2 * AT_TILE * 128;   // two 64-dim halves of 128 keys x 128 B
constexpr int AT_THREADS = 320;                // loads, MMA, 8 softmax warps
constexpr int AT_MAX_ROWS = 96;
constexpr int AT_MAXC = 128;                    // most items per CTA (the grid grows beyond one CTA per SM)

int attn_tc_split_keys() { return AT_SPLIT; }
bool attn_tc_fits(int rows) { return rows >= 1 && rows <= AT_MAX_ROWS; }

// MN-major operand, 128-byte swizzle: 64-element rows of 128 B along the contiguous
// dimension; lbo = bytes between 64-element groups of that dimension, 8-row groups along
// the other dimension 1024 B apart.
__device__ __forceinline__ uint64_t smem_desc_mn_sw128(uint32_t addr, uint32_t lbo) {
    return (uint64_t)((addr >> 4) & 0x3FFFu) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
           ((uint64_t)(1024 >> 4) << 32) | ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

// kind::f16 instruction descriptor, M = 128, N = n, D f32, bf16 operands; a_mn: A MN-major.
__device__ __forceinline__ uint32_t idesc_bf16_m128(int n, bool a_mn) {
    return (1u << 4) | (1u << 7) | (1u << 10) | (a_mn ? (1u << 15) : 0u) | ((uint32_t)(n >> 3) << 17) |
           ((uint32_t)(128 >> 4) << 24);
}

// Barrier of the 256 softmax threads (named barrier 1), and the same with an OR of pred.
__device__ __forceinline__ void at_bar() { asm volatile("bar.sync 1, 256;" ::: "memory"); }
__device__ __forceinline__ int at_any(int pred) {
    int r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\tsetp.ne.b32 p, %1, 0;\n\t"
        "bar.red.or.pred q, 1, 256, p;\n\tselp.b32 %0, 1, 0, q;\n\t}"
        : "=r"(r) : "r"(pred) : "memory");
    return r;
}

// 8 columns of this warp's TMEM lane quarter, 32-bit each.
__device__ __forceinline__ void tmem_ld8(uint32_t taddr, float (&v)[8]) {
    uint32_t r[8];
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
                 : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = __uint_as_float(r[i]);
}

// 2^x by the SFU's approximation (ex2.approx: a few ulp of float32); +0 for x = -inf.
__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ void at_fail(const AttnArgs& a) {
    if (a.err) atomicExch(a.err, SPEC_E_TIMEOUT);
}

// Per row count: TMEM buffers for S and O (two while they fit, so that the scores of the
// next item are computed while the softmax works on this one), bytes of one Q buffer (the
// item's even P tiles go there once its scores are done; odd P tiles go to a third buffer
// of the same size), ring slots of 32 KB that fit the shared memory left.
template <int NP>
struct AtCfg {
    static constexpr int SBUF = NP <= 48 ? 2 : 1;
    static constexpr uint32_t QBYTES = 512u * NP;
    static constexpr int BUFCOLS = (AT_TILES + 1) * NP;
    static constexpr int CW = SBUF * BUFCOLS;
    static constexpr uint32_t NCOLS = CW <= 128 ? 128u : (CW <= 256 ? 256u : 512u);
    static constexpr int NS0 = (int)((232448u - 4096u - 1024u - 3u * QBYTES) / AT_SLOT_BYTES);
    static constexpr int NS = NS0 > 6 ? 6 : NS0;
    static constexpr int NK = NS / 2;                // K ring slots
    static constexpr int NV = NS - NK;               // V ring slots
    static constexpr size_t SMEM = 1024 + 3 * (size_t)QBYTES + (size_t)NS * AT_SLOT_BYTES;
};

// Persistent: CTA c takes items c, c + grid, ... of the (split, kv head, sequence) space
// (split fastest), skipping splits past a sequence's end.  Warp 0 = loads (per item its
// queries, its K tiles into the K ring, its V tiles into the V ring), warp 1 = MMA issuer
// (QK tiles and P V tiles each in item order, issued as their inputs arrive) and TMEM
// owner, warps 2-9 = softmax and output.
template <int NP>
__global__ void __launch_bounds__(AT_THREADS, 1) attn_tc_kernel(const __grid_constant__ AttnArgs a, int n_items,
                                                                int nsplit) {
    using C = AtCfg<NP>;
    extern __shared__ uint8_t at_smem[];
    __shared__ __align__(8) uint64_t k_full[C::NK], k_empty[C::NK], v_full[C::NV], v_empty[C::NV];
    __shared__ __align__(8) uint64_t q_full[2], q_free[2], s_full[C::SBUF], t_free[C::SBUF], o_full[C::SBUF];
    __shared__ __align__(8) uint64_t p_full[2], p_done[2], done_bar;     // per P buffer (tile parity)
    __shared__ uint32_t tmem_sh;
    __shared__ volatile int abort_flag;
    __shared__ int cand_l0[AT_MAXC];      // seq_len of this CTA's k-th item's sequence, -1 = split past its end
    __shared__ int cand_slot[AT_MAXC];
    __shared__ int page_cache[4][32];     // the loads warp's page lists of the last items (see there)
    __shared__ float red[4][NP];
    __shared__ float row_m[NP];           // the rows' maxima over the split (base-2 scaled scores)

    pdl_launch_dependents();
    const int G = a.hq / a.hkv;
    const int R = a.T * G;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int ncand = min(AT_MAXC, (n_items - (int)blockIdx.x + (int)gridDim.x - 1) / (int)gridDim.x);
    auto item_of = [&](int k, int& s, int& g, int& b) {
        const int it = (int)blockIdx.x + k * (int)gridDim.x;
        s = it % nsplit;
        const int r = it / nsplit;
        g = r % a.hkv;
        b = r / a.hkv;
    };
    for (int k = threadIdx.x; k < ncand; k += AT_THREADS) {
        int s, g, b;
        item_of(k, s, g, b);
        const int slot = a.seq_ids[b];
        const int L0 = a.seq_len[slot];
        cand_l0[k] = s * AT_SPLIT < L0 + a.T ? L0 : -1;
        cand_slot[k] = slot;
    }
    const uint32_t base = (smem_u32(at_smem) + 1023u) & ~1023u;
    uint8_t* gbase = at_smem + (base - smem_u32(at_smem));
    const uint32_t pbuf1 = base + 2 * C::QBYTES;    // odd P tiles
    const uint32_t ring = base + 3 * C::QBYTES;
    // zero the ring once: V rows past a split's keys are multiplied by P = 0 and must be finite
    for (int i = threadIdx.x; i < C::NS * AT_SLOT_BYTES / 16; i += AT_THREADS)
        reinterpret_cast<uint4*>(gbase + 3 * C::QBYTES)[i] = make_uint4(0, 0, 0, 0);
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    if (threadIdx.x == 0) {
        for (int i = 0; i < C::NK; ++i) {
            mbar_init(smem_u32(&k_full[i]), 1);
            mbar_init(smem_u32(&k_empty[i]), 1);
        }
        for (int i = 0; i < C::NV; ++i) {
            mbar_init(smem_u32(&v_full[i]), 1);
            mbar_init(smem_u32(&v_empty[i]), 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(smem_u32(&q_full[i]), 1);
            mbar_init(smem_u32(&q_free[i]), 1);
        }
        for (int i = 0; i < C::SBUF; ++i) {
            mbar_init(smem_u32(&s_full[i]), 1);
            mbar_init(smem_u32(&t_free[i]), 256);
            mbar_init(smem_u32(&o_full[i]), 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(smem_u32(&p_full[i]), 256);
            mbar_init(smem_u32(&p_done[i]), 1);
        }
        mbar_init(smem_u32(&done_bar), 1);
        abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                     :: "r"(smem_u32(&tmem_sh)), "r"(C::NCOLS) : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_sh;

    const uint32_t kring = ring, vring = ring + (uint32_t)C::NK * AT_SLOT_BYTES;
    if (warp == 0) {
        // ---- loads, the whole warp: two queues in item order, K tiles (each item's queries
        // first) and V tiles (an item's V after its K), each tile issued as soon as its ring
        // has a free slot, so that the next item's keys never wait for this item's values.
        // Lane p holds the p-th page of an item's split; the page lists of the last four
        // items the K queue reached are kept for the V queue. ----
        pdl_wait();
        const uint64_t pol = policy_evict_first();
        const size_t half_stride = (size_t)a.num_pages * 16 * 64;        // elements between halves
        uint32_t sk = 0, sv = 0;            // tiles issued into the K and V rings
        // one K or V tile (8 pages of 2 x 2 KB) into slot sl, runs of consecutive pages as
        // one bulk copy per 64-dim half
        auto issue_tile = [&](bool is_v, int sl, int g, int tile, int npg, int pg) {
            const int p_lo = tile * 8, np_t = min(npg, p_lo + 8) - p_lo;
            const uint32_t fb = smem_u32(is_v ? &v_full[sl] : &k_full[sl]);
            const uint32_t dst0 = (is_v ? vring : kring) + (uint32_t)sl * AT_SLOT_BYTES;
            const __nv_bfloat16* pool = static_cast<const __nv_bfloat16*>(is_v ? a.v_layer : a.k_layer) +
                                        (size_t)g * 2 * half_stride;
            if (lane == 0) mbar_arrive_expect_tx(fb, (uint32_t)np_t * 4096u);
            int prev = __shfl_sync(FULL_MASK, pg, p_lo);
            int first = prev, run_start = 0;
            for (int p = 1; p <= np_t; ++p) {
                const int cur = p < np_t ? __shfl_sync(FULL_MASK, pg, p_lo + p) : -2;
                if (cur != prev + 1) {          // a run of consecutive pages ends at p - 1
                    if (lane == 0)
                        for (int h = 0; h < 2; ++h)
                            bulk_g2s(dst0 + (uint32_t)h * (AT_SLOT_BYTES / 2) + (uint32_t)run_start * 2048u,
                                     pool + h * half_stride + (size_t)first * 16 * 64,
                                     (uint32_t)(p - run_start) * 2048u, fb, pol);
                    run_start = p;
                    first = cur;
                }
                prev = cur;
            }
        };
        auto next_nonempty = [&](int k) {
            while (k < ncand && cand_l0[k] < 0) ++k;
            return k;
        };
        struct Q {
            int k, n, t, nt, npg, g;
        };
        auto start = [&](Q& q, int k, int n) {
            q.k = k;
            q.n = n;
            q.t = 0;
            if (k < ncand) {
                int s, g, b;
                item_of(k, s, g, b);
                const int nkeys = min(AT_SPLIT, cand_l0[k] + a.T - s * AT_SPLIT);
                q.nt = (nkeys + AT_TILE - 1) / AT_TILE;
                q.npg = (nkeys + 15) >> 4;
                q.g = g;
            }
        };
        Q kq, vq;
        start(kq, next_nonempty(0), 0);
        start(vq, kq.k, 0);
        bool kq_qdone = false;
        int kq_pg = 0;
        if (kq.k < ncand) {                 // the first item's pages
            int s, g, b;
            item_of(kq.k, s, g, b);
            const int lp = s * (AT_SPLIT / 16) + lane;
            if (lane < kq.npg && lp < a.max_pages) kq_pg = a.block_table[(size_t)cand_slot[kq.k] * a.max_pages + lp];
            kq_pg = min(max(kq_pg, 0), a.num_pages - 1);
            page_cache[0][lane] = kq_pg;
        }
        int kdone = 0;                      // items whose K tiles are all issued
        bool ok = true;
        unsigned long long idle_since = globaltimer_ns();
        while (vq.k < ncand) {
            int act = 0;
            if (lane == 0) {
                if (abort_flag) {
                    act = -1;
                } else if (kq.k < ncand && !kq_qdone) {
                    if (kq.n < 2 || mbar_test(smem_u32(&q_free[kq.n & 1]), (uint32_t)(((kq.n >> 1) - 1) & 1))) act = 1;
                } else if (kq.k < ncand &&
                           (sk < (uint32_t)C::NK || mbar_test(smem_u32(&k_empty[sk % C::NK]), ((sk / C::NK) - 1) & 1))) {
                    act = 2;
                }
                if (act == 0 && vq.n < kdone &&
                    (sv < (uint32_t)C::NV || mbar_test(smem_u32(&v_empty[sv % C::NV]), ((sv / C::NV) - 1) & 1)))
                    act = 3;
                if (act == 0 && globaltimer_ns() - idle_since > WAIT_BUDGET_NS) act = -1;
            }
            act = __shfl_sync(FULL_MASK, act, 0);
            if (act < 0) {
                ok = false;
                break;
            }
            if (act == 0) continue;
            idle_since = globaltimer_ns();
            if (act == 1) {
                // the queries of the K queue's item (their buffer is free once P V of the item
                // two before has run)
                if (lane == 0) {
                    int s, g, b;
                    item_of(kq.k, s, g, b);
                    const int qb = kq.n & 1;
                    mbar_arrive_expect_tx(smem_u32(&q_full[qb]), C::QBYTES);
                    bulk_g2s(base + (uint32_t)qb * C::QBYTES,
                             static_cast<const __nv_bfloat16*>(a.q) + ((size_t)b * a.hkv + g) * (C::QBYTES / 2),
                             C::QBYTES, smem_u32(&q_full[qb]), pol);
                }
                kq_qdone = true;
            } else if (act == 2) {
                issue_tile(false, (int)(sk % C::NK), kq.g, kq.t, kq.npg, kq_pg);
                ++sk;
                if (++kq.t == kq.nt) {
                    ++kdone;
                    start(kq, next_nonempty(kq.k + 1), kq.n + 1);
                    kq_qdone = false;
                    if (kq.k < ncand) {
                        int s, g, b;
                        item_of(kq.k, s, g, b);
                        const int lp = s * (AT_SPLIT / 16) + lane;
                        int pg = 0;
                        if (lane < kq.npg && lp < a.max_pages) pg = a.block_table[(size_t)cand_slot[kq.k] * a.max_pages + lp];
                        kq_pg = min(max(pg, 0), a.num_pages - 1);
                        page_cache[kq.n & 3][lane] = kq_pg;
                    }
                }
            } else {
                issue_tile(true, (int)(sv % C::NV), vq.g, vq.t, vq.npg, page_cache[vq.n & 3][lane]);
                ++sv;
                if (++vq.t == vq.nt) start(vq, next_nonempty(vq.k + 1), vq.n + 1);
            }
        }
        if (lane == 0) {
            if (!ok) {
                abort_flag = 1;
                at_fail(a);
            }
            // no copy may still be landing when the CTA leaves
            for (uint32_t j = sk > (uint32_t)C::NK ? sk - C::NK : 0; j < sk; ++j)
                if (!mbar_wait(smem_u32(&k_full[j % C::NK]), (j / C::NK) & 1)) at_fail(a);
            for (uint32_t j = sv > (uint32_t)C::NV ? sv - C::NV : 0; j < sv; ++j)
                if (!mbar_wait(smem_u32(&v_full[j % C::NV]), (j / C::NV) & 1)) at_fail(a);
            const int nq = kq.n + (kq_qdone ? 1 : 0);
            for (int m = max(0, nq - 2); m < nq; ++m)
                if (!mbar_wait(smem_u32(&q_full[m & 1]), (uint32_t)((m >> 1) & 1))) at_fail(a);
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // ---- MMA issuer: two queues in item order, QK tiles and P V tiles, each tile
            // issued as soon as its inputs are there (polled, not waited on, so that a P V
            // tile waiting for its probabilities never holds up the next item's scores) ----
            pdl_wait();
            const uint32_t id_s = idesc_bf16_m128(NP, false);
            const uint32_t id_o = idesc_bf16_m128(NP, true);
            uint32_t sk = 0, sv = 0, pc0 = 0, pc1 = 0;      // P tiles consumed per buffer
            // QK queue: candidate index, item count, tile; P V queue likewise
            int qk_k = 0, qk_n = 0, qk_t = 0, qk_nt = 0;
            int pv_k = 0, pv_n = 0, pv_t = 0, pv_nt = 0;
            auto next_item = [&](int k, int& nt) -> int {        // first non-empty candidate >= k
                for (; k < ncand; ++k) {
                    const int L0 = cand_l0[k];
                    if (L0 < 0) continue;
                    int s, g, b;
                    item_of(k, s, g, b);
                    nt = (min(AT_SPLIT, L0 + a.T - s * AT_SPLIT) + AT_TILE - 1) / AT_TILE;
                    return k;
                }
                return ncand;
            };
            qk_k = next_item(0, qk_nt);
            pv_k = next_item(0, pv_nt);
            bool ok = true;
            unsigned long long idle_since = globaltimer_ns();
            while (ok && pv_k < ncand) {
                bool progressed = false;
                if (qk_k < ncand) {
                    const int buf = qk_n % C::SBUF, qb = qk_n & 1;
                    const int sl = (int)(sk % C::NK);
                    bool ready = true;
                    if (qk_t == 0) {
                        if (qk_n >= C::SBUF)
                            ready = mbar_test(smem_u32(&t_free[buf]), (uint32_t)(((qk_n / C::SBUF) - 1) & 1));
                        ready = ready && mbar_test(smem_u32(&q_full[qb]), (uint32_t)((qk_n >> 1) & 1));
                    }
                    ready = ready && mbar_test(smem_u32(&k_full[sl]), (sk / C::NK) & 1);
                    if (ready) {
                        tc_fence_after();
                        const uint32_t kb = kring + (uint32_t)sl * AT_SLOT_BYTES;
                        const uint32_t qbuf = base + (uint32_t)qb * C::QBYTES;
#pragma unroll
                        for (int lo = 0; lo < 2; ++lo)
#pragma unroll
                            for (int h = 0; h < 2; ++h)
                                mma_bf16_atom(tmem + (uint32_t)(buf * C::BUFCOLS + qk_t * NP),
                                              smem_desc_sw128(kb + (uint32_t)h * (AT_SLOT_BYTES / 2)),
                                              smem_desc_sw128(qbuf + (uint32_t)(lo * 2 + h) * NP * 128), id_s,
                                              (lo | h) ? 1u : 0u);
                        mma_commit(smem_u32(&k_empty[sl]));
                        ++sk;
                        if (++qk_t == qk_nt) {
                            mma_commit(smem_u32(&s_full[buf]));
                            qk_t = 0;
                            ++qk_n;
                            qk_k = next_item(qk_k + 1, qk_nt);
                        }
                        progressed = true;
                    }
                }
                if (pv_n < qk_n) {            // P of an item exists only after its scores
                    const int buf = pv_n % C::SBUF, qb = pv_n & 1;
                    const int sl = (int)(sv % C::NV);
                    const int pb = pv_t & 1;
                    if (mbar_test(smem_u32(&v_full[sl]), (sv / C::NV) & 1) &&
                        mbar_test(smem_u32(&p_full[pb]), (pb ? pc1 : pc0) & 1)) {
                        tc_fence_after();
                        const uint32_t vb = vring + (uint32_t)sl * AT_SLOT_BYTES;
                        const uint32_t pbuf = pb ? pbuf1 : base + (uint32_t)qb * C::QBYTES;
                        const uint32_t dcol = tmem + (uint32_t)(buf * C::BUFCOLS + AT_TILES * NP);
#pragma unroll
                        for (int lo = 0; lo < 2; ++lo)
#pragma unroll
                            for (int ks = 0; ks < AT_TILE / 16; ++ks)
                                mma_bf16(dcol, smem_desc_mn_sw128(vb + (uint32_t)ks * 2048u, AT_SLOT_BYTES / 2),
                                         smem_desc_sw128(pbuf + (uint32_t)(lo * 2 + (ks >> 2)) * NP * 128 +
                                                         (uint32_t)(ks & 3) * 32),
                                         id_o, (pv_t | lo | ks) ? 1u : 0u);
                        mma_commit(smem_u32(&v_empty[sl]));
                        mma_commit(smem_u32(&p_done[pb]));
                        ++sv;
                        if (pb) ++pc1; else ++pc0;
                        if (++pv_t == pv_nt) {
                            mma_commit(smem_u32(&o_full[buf]));
                            mma_commit(smem_u32(&q_free[qb]));
                            pv_t = 0;
                            ++pv_n;
                            pv_k = next_item(pv_k + 1, pv_nt);
                        }
                        progressed = true;
                    }
                }
                if (progressed) {
                    idle_since = globaltimer_ns();
                } else if (abort_flag || globaltimer_ns() - idle_since > WAIT_BUDGET_NS) {
                    ok = false;
                }
            }
            if (!ok) {
                abort_flag = 1;
                at_fail(a);
            }
            // nothing may still write tensor memory when it is freed
            mma_commit(smem_u32(&done_bar));
            mbar_wait(smem_u32(&done_bar), 0);
        }
    } else {
        // ---- softmax and output, warps 2-9: thread = key of a tile (S^T lanes), later dim
        // (O^T lanes); warps 2-5 take rows [0, NP/2), warps 6-9 rows [NP/2, NP), so that two
        // warps per scheduler hide each other's latency ----
        pdl_wait();
        constexpr int HR = NP / 2;                       // rows per warp group
        constexpr int NCH = HR / 8;                      // 8-column TMEM loads per group
        const int q4 = warp & 3;                         // TMEM lane quarter of this warp
        const int grp = (warp - 2) >> 2;
        const int etid = threadIdx.x - 64;               // 0 .. 255
        const int r0 = grp * HR;
        const int key = q4 * 32 + lane;                  // key of a tile / dim of the output
        const uint32_t tl = tmem + ((uint32_t)(q4 * 32) << 16);
        const float sl2 = a.scale * 1.4426950408889634f;
        const int atom = key >> 6, kc = key & 63;
        uint32_t pw0 = 0, pw1 = 0;          // P tiles written per buffer
        int n = 0;
        bool ok = true;
        // the output of an item is read out after the next item's maxima (its last P V has
        // finished by then), or at once when S and O are single-buffered
        bool o_pending = false;
        size_t o_pbase = 0;
        int o_buf = 0, o_n = 0;
        auto read_out = [&]() -> bool {
            const bool okw = !abort_flag && mbar_wait(smem_u32(&o_full[o_buf]), (uint32_t)((o_n / C::SBUF) & 1));
            if (at_any(okw ? 0 : 1)) return false;
            tc_fence_after();
#pragma unroll
            for (int ch = 0; ch < NCH; ++ch) {
                float v[8];
                tmem_ld8(tl + (uint32_t)(o_buf * C::BUFCOLS + AT_TILES * NP + r0 + ch * 8), v);
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    if (r0 + ch * 8 + e < R) a.part_o[(o_pbase + r0 + ch * 8 + e) * 128 + key] = v[e];
            }
            // the item's S and O columns are free for item o_n + SBUF
            tc_fence_before();
            mbar_arrive(smem_u32(&t_free[o_buf]));
            o_pending = false;
            return true;
        };
        for (int k = 0; ok && k < ncand; ++k) {
            const int L0 = cand_l0[k];
            if (L0 < 0) continue;
            int s, g, b;
            item_of(k, s, g, b);
            const int k0 = s * AT_SPLIT;
            const int nt = (min(AT_SPLIT, L0 + a.T - k0) + AT_TILE - 1) / AT_TILE;
            const int buf = n % C::SBUF, qb = n & 1;
            const uint32_t sbase = tl + (uint32_t)(buf * C::BUFCOLS + r0);
            // key kk (split-relative) is visible to row j = t * G + hh when kk <= L0 - k0 + t;
            // padding rows (j >= R) see none
            int lim[HR];
            {
                int t = r0 / G, hh = r0 - (r0 / G) * G;
#pragma unroll
                for (int jj = 0; jj < HR; ++jj) {
                    lim[jj] = r0 + jj < R ? L0 - k0 + t : -1;
                    if (++hh == G) { hh = 0; ++t; }
                }
            }
            bool okw = !abort_flag && mbar_wait(smem_u32(&s_full[buf]), (uint32_t)((n / C::SBUF) & 1));
            if (at_any(okw ? 0 : 1)) {
                ok = false;
                break;
            }
            tc_fence_after();
            // row maxima over the split: this thread's keys (one per tile), the warp
            // (butterfly), then the four lane quarters in a fixed order
            float mrow[HR];
#pragma unroll
            for (int jj = 0; jj < HR; ++jj) mrow[jj] = -INFINITY;
            for (int i = 0; i < nt; ++i) {
                const int kk = i * AT_TILE + key;
#pragma unroll
                for (int ch = 0; ch < NCH; ++ch) {
                    float v[8];
                    tmem_ld8(sbase + (uint32_t)(i * NP + ch * 8), v);
#pragma unroll
                    for (int e = 0; e < 8; ++e)
                        if (kk <= lim[ch * 8 + e]) mrow[ch * 8 + e] = fmaxf(mrow[ch * 8 + e], v[e] * sl2);
                }
            }
#pragma unroll
            for (int jj = 0; jj < HR; ++jj) {
                float m = mrow[jj];
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(FULL_MASK, m, o));
                if (lane == 0) red[q4][r0 + jj] = m;
            }
            at_bar();
            if (etid < NP) row_m[etid] = fmaxf(fmaxf(red[0][etid], red[1][etid]), fmaxf(red[2][etid], red[3][etid]));
#pragma unroll
            for (int jj = 0; jj < HR; ++jj) {
                const float m = fmaxf(fmaxf(red[0][r0 + jj], red[1][r0 + jj]), fmaxf(red[2][r0 + jj], red[3][r0 + jj]));
                mrow[jj] = m == -INFINITY ? 0.0f : m;
            }
            at_bar();
            if (o_pending && !read_out()) {
                ok = false;
                break;
            }
            // P = 2^(s - m) per tile, bf16 hi and lo, into the B operand of P V: even tiles
            // into this item's query buffer (its QK MMAs are complete), odd tiles into the
            // third buffer, so that a tile is written while P V runs on the one before
            float lsum[HR];
#pragma unroll
            for (int jj = 0; jj < HR; ++jj) lsum[jj] = 0.0f;
            for (int i = 0; i < nt; ++i) {
                const int pb = i & 1;
                const uint32_t pw = pb ? pw1 : pw0;
                if (pw > 0) {               // that buffer's previous tile must have been read
                    okw = !abort_flag && mbar_wait(smem_u32(&p_done[pb]), (pw - 1) & 1);
                    if (at_any(okw ? 0 : 1)) {
                        ok = false;
                        break;
                    }
                }
                uint8_t* pbuf = gbase + (pb ? 2 * C::QBYTES : qb * C::QBYTES);
                const int kk = i * AT_TILE + key;
#pragma unroll
                for (int ch = 0; ch < NCH; ++ch) {
                    float v[8];
                    tmem_ld8(sbase + (uint32_t)(i * NP + ch * 8), v);
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        const int jj = ch * 8 + e, j = r0 + jj;
                        const float p = kk <= lim[jj] ? fast_exp2(fmaf(v[e], sl2, -mrow[jj])) : 0.0f;
                        lsum[jj] += p;
                        const __nv_bfloat16 hi = __float2bfloat16_rn(p);
                        const __nv_bfloat16 lo = __float2bfloat16_rn(p - __bfloat162float(hi));
                        const uint32_t off = (uint32_t)j * 128 + ((uint32_t)(((kc >> 3) ^ (j & 7)) << 4) | ((kc & 7) << 1));
                        *reinterpret_cast<__nv_bfloat16*>(pbuf + (uint32_t)atom * NP * 128 + off) = hi;
                        *reinterpret_cast<__nv_bfloat16*>(pbuf + (uint32_t)(2 + atom) * NP * 128 + off) = lo;
                    }
                }
                // the generic-proxy writes of P must be visible to the tensor core
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                tc_fence_before();
                mbar_arrive(smem_u32(&p_full[pb]));
                if (pb) ++pw1; else ++pw0;
            }
            if (!ok) break;
            // row sums: warp butterfly, then the four lane quarters in a fixed order
#pragma unroll
            for (int jj = 0; jj < HR; ++jj) {
                float l = lsum[jj];
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) l += __shfl_xor_sync(FULL_MASK, l, o);
                if (lane == 0) red[q4][r0 + jj] = l;
            }
            at_bar();
            const size_t pbase = (((size_t)b * a.hkv + g) * a.n_chunks + s) * R;
            if (etid < R) {
                const float l = ((red[0][etid] + red[1][etid]) + red[2][etid]) + red[3][etid];
                a.part_ml[pbase + etid] = make_float2(row_m[etid], l);
            }
            o_pending = true;
            o_pbase = pbase;
            o_buf = buf;
            o_n = n;
            if (C::SBUF == 1 && !read_out()) {
                ok = false;
                break;
            }
            ++n;
        }
        if (ok && o_pending && !read_out()) ok = false;
        if (!ok && etid == 0) {
            abort_flag = 1;
            at_fail(a);
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" :: "r"(tmem), "r"(C::NCOLS) : "memory");
}

int attn_tc_set_smem_limits() {
    void* k[6] = {(void*)attn_tc_kernel<16>, (void*)attn_tc_kernel<32>, (void*)attn_tc_kernel<48>,
                  (void*)attn_tc_kernel<64>, (void*)attn_tc_kernel<80>, (void*)attn_tc_kernel<96>};
    const size_t sm[6] = {AtCfg<16>::SMEM, AtCfg<32>::SMEM, AtCfg<48>::SMEM, AtCfg<64>::SMEM, AtCfg<80>::SMEM,
                          AtCfg<96>::SMEM};
    for (int i = 0; i < 6; ++i)
        if (cudaFuncSetAttribute(k[i], cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm[i]) != cudaSuccess)
            return -1;
    return 0;
}

// Launch over nsplit 512-key splits; rows = T * G <= 96.
void launch_attn_tc(bool pdl, const AttnArgs& a, int nsplit, int B, int sms, cudaStream_t st) {
    const int np = (a.T * (a.hq / a.hkv) + 15) & ~15;
    const int n_items = nsplit * a.hkv * B;
    // one CTA per SM, more only when an SM would get more than AT_MAXC items
    const int grid = std::min(n_items, std::max(sms, (n_items + AT_MAXC - 1) / AT_MAXC));
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(AT_THREADS);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    switch (np) {
    case 16: cfg.dynamicSmemBytes = AtCfg<16>::SMEM; cudaLaunchKernelEx(&cfg, attn_tc_kernel<16>, a, n_items, nsplit); break;
    case 32: cfg.dynamicSmemBytes = AtCfg<32>::SMEM; cudaLaunchKernelEx(&cfg, attn_tc_kernel<32>, a, n_items, nsplit); break;
    case 48: cfg.dynamicSmemBytes = AtCfg<48>::SMEM; cudaLaunchKernelEx(&cfg, attn_tc_kernel<48>, a, n_items, nsplit); break;
    case 64: cfg.dynamicSmemBytes = AtCfg<64>::SMEM; cudaLaunchKernelEx(&cfg, attn_tc_kernel<64>, a, n_items, nsplit); break;
    case 80: cfg.dynamicSmemBytes = AtCfg<80>::SMEM; cudaLaunchKernelEx(&cfg, attn_tc_kernel<80>, a, n_items, nsplit); break;
    default: cfg.dynamicSmemBytes = AtCfg<96>::SMEM; cudaLaunchKernelEx(&cfg, attn_tc_kernel<96>, a, n_items, nsplit); break;
    }
}

}  // namespace sv
