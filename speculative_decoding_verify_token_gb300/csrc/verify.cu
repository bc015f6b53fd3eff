// Fused verify kernel: one streaming pass over the target (and draft) logits rows of a
// speculative-decoding verify step, then per-row truncation and per-sequence acceptance.
//
// What it computes follows "Qwen3.5 and Qwen3.6 MTP head reaches 1.4x on Apple Silicon
// after three fixes" ("The verify was wrong under sampling": accept with probability
// min(1, p/q), resample from max(0, p - q) renormalised; "Truncation has to match on both
// sides": top-k 20 / top-p 0.95 on p and q alike) and, at temperature 0, the greedy rule
// of "What is Speculative Decoding and How Does a Draft Model Work?" ("#2": keep drafts
// while they equal the target's choice, replace the first mismatch).
//
// GB300 design, two kernels:
//  * pass 1 streams every needed row once, with coalesced 16-byte streaming loads (two
//    blocks of 4 KB in flight per warp, 16 warps per SM), and writes for each 256-element
//    fine block its largest element with that element's id and its second largest element
//    (12 bytes per KB read); eight lanes own a fine block, so the reductions are 3-step
//    shuffles within the group;
//  * pass 2 (one CTA per sequence, one warp per row, launched programmatically dependent
//    on pass 1) ranks the fine blocks' maxima: tau, the k-th largest of the 32 lanes'
//    maxima, bounds the row's k-th largest element from below, the maxima >= tau are
//    merged into the row's top list, and only the blocks whose second largest element
//    reaches that list's k-th value can hold a further top-k element -- on random rows
//    about one row in four re-reads one fine block (1 KB).  Ties and adversarial rows stay
//    exact.  Pass 2 is a latency chain, so its orderings are rank selections (each entry
//    counts the entries that beat it over shared memory and goes to that place) rather
//    than bitonic sorts, whose 15 dependent shuffle stages cost about 1.5 us a sort;
//  * each row's truncated distribution is built from its list in shared memory, and warp 0
//    runs the sequence's acceptance scan and the final inverse-CDF draw.
#include <cstdio>
#include <cstring>
#include <cmath>
#include <algorithm>
#include <atomic>
#include <mutex>

#include "common.cuh"
#include "host_util.h"

namespace sv {

constexpr int LISTN = 32;
constexpr int VT_MAX_K = 64;
constexpr int VB = 1024;                             // elements per block (the pass-1 unit, coarse maxima)
constexpr int VB4 = VB / 4;                          // float4 per block
constexpr int VF = 256;                              // elements per fine block (fine maxima, pass-2 reads)
constexpr int NF = VB / VF;                          // fine blocks per block
constexpr int BM_THREADS = 256;                      // pass 1 CTA
#ifndef BM_CTAS_PER_SM
#define BM_CTAS_PER_SM 2                             // 16 warps per SM
#endif
constexpr int BM_INFLIGHT = 2;                       // blocks loaded at once per warp
// registers per pass-1 thread (two CTAs of 256 threads per SM)
#ifndef BM_MAXNREG
#define BM_MAXNREG 96
#endif
#ifndef BM_SMEM_CARVEOUT
#define BM_SMEM_CARVEOUT 13                         // per cent of L1 kept as shared memory
#endif
#ifndef BM_STATIC_PCT
#define BM_STATIC_PCT 90                             // share of pass-1 blocks in static sweeps
#endif
constexpr int RF_MAX_WARPS = 16;                     // pass 2: warps (rows in flight) per CTA
constexpr int RF_SAMPLE_WARPS = 4;                   // sample mode: rows per CTA
constexpr int RF_BPL = 5;                            // blocks' second values a lane holds per round
constexpr int RF_KPL = 2 * RF_BPL;                   // float4 of (maximum, id) pairs a lane holds per round
constexpr int RF_BATCH = 4;                          // fine blocks read again at once per warp
constexpr int RF_SEL_CAP = 64;                       // fine blocks listed before they are read again
// per-warp pool of (value, id) entries: the buffered candidates and, during a merge, the
// warp's list of LISTN behind them; merged before an append could overflow it (appends come
// 64 or 128 at a time)
constexpr int RF_CAND_CAP = 192;
// 4-byte words of shared memory per warp: the pool, the merge's output list, the fine
// blocks to read again
constexpr int RF_WARP_WORDS = 2 * RF_CAND_CAP + 2 * LISTN + RF_SEL_CAP;

enum { MODE_VERIFY = 0, MODE_SAMPLE = 1 };

struct VerifyParams {
    const float* target;        // [B][K+1][V] (verify) or [R][V] (sample)
    const float* draft;         // [B][K][V] or nullptr
    const int* draft_tokens;    // [B][K]
    const int* draft_len;       // [B] or nullptr
    const float* u;             // [B][K+1] (verify) or [R] (sample)
    int B, K, V;
    float temperature;
    int top_k;                  // effective k (1 when greedy)
    float top_p;
    int mode;
    int n_target_rows;          // B*(K+1) (verify) or R (sample)
    int n_rows;                 // + B*K draft rows when draft logits are given
    int nbb;                    // blocks per row (ceil(V / VB)); fine blocks NF * nbb
    int* accepted_len;
    int* next_token;
    int* out_ids;
    float* out_probs;
    int* seq_status;
    int* out_tokens;
    // workspace
    int* blk_next;              // pass-1 dynamic block counter
    float2* fk;                 // [n_rows][NF * nbb] fine block (maximum, id of an element at it)
    float* fm2;                 // [n_rows][NF * nbb] fine block second largest element
};

struct RowInfo {
    const float* ptr;
    int seq;        // sequence (verify) or row index (sample)
    int pos;        // position within the sequence's rows
    bool is_draft;
};

__device__ __forceinline__ int draft_count(const VerifyParams& p, int b) {
    if (p.draft_len == nullptr) return p.K;
    int k = p.draft_len[b];
    return k < 0 ? 0 : (k > p.K ? p.K : k);
}

__device__ __forceinline__ RowInfo row_info(const VerifyParams& p, int r) {
    RowInfo ri;
    if (p.mode == MODE_SAMPLE) {
        ri.ptr = p.target + (size_t)r * p.V; ri.seq = r; ri.pos = 0; ri.is_draft = false;
    } else if (r < p.n_target_rows) {
        ri.ptr = p.target + (size_t)r * p.V; ri.seq = r / (p.K + 1); ri.pos = r % (p.K + 1); ri.is_draft = false;
    } else {
        const int rr = r - p.n_target_rows;
        ri.ptr = p.draft + (size_t)rr * p.V; ri.seq = rr / p.K; ri.pos = rr % p.K; ri.is_draft = true;
    }
    return ri;
}

__device__ __forceinline__ bool row_needed(const VerifyParams& p, const RowInfo& ri) {
    if (p.mode == MODE_SAMPLE) return true;
    const int kb = draft_count(p, ri.seq);
    return ri.is_draft ? (ri.pos < kb) : (ri.pos <= kb);
}

// Row layout: [0, head) scalar, [head, head + body) 16-byte aligned body, then a scalar tail.
__device__ __forceinline__ void row_split(const float* ptr, int V, int& head, int& body) {
    const int mis = (int)((reinterpret_cast<uintptr_t>(ptr) >> 2) & 3);
    head = (4 - mis) & 3;
    if (head > V) head = V;
    body = ((V - head) / 4) * 4;
}

__device__ __forceinline__ float pick4(const float4& x, int c) {
    float r = x.x;
    r = (c == 1) ? x.y : r;
    r = (c == 2) ? x.z : r;
    r = (c == 3) ? x.w : r;
    return r;
}

// The warp's running list (lane j = j-th best under better(), padded with (-inf, SENT_ID))
// and the n candidates buffered in pool[0, n) become the best LISTN entries of their union.
// Each entry's place is the number of entries of the union that beat it: better() orders
// entries with distinct ids strictly, and every real entry has its own id (one element of
// the row), so the places are those of a sort of the union.  Padding is never placed; the
// output starts as padding, so no id can come from the list or the pool alone.  The counts
// read the pool as broadcast shared-memory loads with no dependence between them, where a
// bitonic sort is a chain of dependent shuffles.  A list that already holds entries (the
// merges after blocks are read again: a few candidates) is sorted, so entry j has j
// entries above it in the list; only the candidates are counted against it, and a
// candidate counts the list with one ballot.  Not inlined: it is reached from many unrolled
// sites, and one copy keeps the code in the instruction cache.
struct ListEntry { float v; int id; };
__device__ __noinline__ ListEntry merge_candidates(float lv, int lid, float2* pool, float2* outl, int n, int lane) {
    const float2 PAD = make_float2(-INFINITY, __int_as_float(SENT_ID));
    const unsigned real = __ballot_sync(FULL, lid != SENT_ID);
    outl[lane] = PAD;
    if (real != 0u && n <= 32) {
        __syncwarp();
        int cl = 0, lrank = 0;
        for (int i = 0; i < n; ++i) {
            const float2 c = pool[i];
            const int ic = __float_as_int(c.y);
            cl += better(c.x, ic, lv, lid) ? 1 : 0;
            const unsigned lb = __ballot_sync(FULL, lid != SENT_ID && better(lv, lid, c.x, ic));
            if (lane == i) lrank = __popc(lb);
        }
        const float2 me = lane < n ? pool[lane] : PAD;
        const int im = __float_as_int(me.y);
        int crank = lrank;
        if (lane < n) {
            for (int i = 0; i < n; ++i) {
                const float2 c = pool[i];
                crank += better(c.x, __float_as_int(c.y), me.x, im) ? 1 : 0;
            }
        }
        if (lid != SENT_ID && lane + cl < LISTN) outl[lane + cl] = make_float2(lv, __int_as_float(lid));
        if (lane < n && im != SENT_ID && crank < LISTN) outl[crank] = me;
        __syncwarp();
        const float2 r = outl[lane];
        __syncwarp();
        return ListEntry{r.x, __float_as_int(r.y)};
    }
    if (lid != SENT_ID) pool[n + __popc(real & ((1u << lane) - 1u))] = make_float2(lv, __int_as_float(lid));
    __syncwarp();
    const int P = n + __popc(real);
    for (int e0 = 0; e0 < P; e0 += 64) {
        const int ea = e0 + lane, eb = ea + 32;
        const float2 A = ea < P ? pool[ea] : PAD;
        const float2 Bq = eb < P ? pool[eb] : PAD;
        const int ia = __float_as_int(A.y), ib = __float_as_int(Bq.y);
        int ra = 0, rb = 0;
#pragma unroll 4
        for (int j = 0; j < P; ++j) {
            const float2 c = pool[j];
            const int ic = __float_as_int(c.y);
            ra += better(c.x, ic, A.x, ia) ? 1 : 0;
            rb += better(c.x, ic, Bq.x, ib) ? 1 : 0;
        }
        if (ia != SENT_ID && ra < LISTN) outl[ra] = A;
        if (ib != SENT_ID && rb < LISTN) outl[rb] = Bq;
    }
    __syncwarp();
    const float2 r = outl[lane];
    __syncwarp();
    return ListEntry{r.x, __float_as_int(r.y)};
}

__device__ __forceinline__ void flush_candidates(float& lv, int& lid, float2* pool, float2* outl, int n, int lane) {
    const ListEntry e = merge_candidates(lv, lid, pool, outl, n, lane);
    lv = e.v;
    lid = e.id;
}

// Truncated distribution of a merged row list (lane j = j-th best): lane j's (id, probability),
// id -1 where the entry is cut.
__device__ void row_dist(const VerifyParams& p, float lv, int lid, int lane, int& oid, float& op) {
    const int k = p.top_k;
    if (p.temperature == 0.0f) {
        oid = lane == 0 ? lid : -1;
        op = lane == 0 ? 1.0f : 0.0f;
    } else {
        const bool valid = lane < k && lid != SENT_ID;
        const float v0 = __shfl_sync(FULL, lv, 0);
        const float e = valid ? expf((lv - v0) / p.temperature) : 0.0f;
        const float S = warp_sum(e);
        const float pr = e / S;
        // exclusive prefix sum of pr in ranking order
        float incl = pr;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const float t = __shfl_up_sync(FULL, incl, o);
            if (lane >= o) incl += t;
        }
        const float before = incl - pr;
        const bool kept = valid && (lane == 0 || p.top_p >= 1.0f || before < p.top_p);
        const float S2 = warp_sum(kept ? e : 0.0f);
        oid = kept ? lid : -1;
        op = kept ? e / S2 : 0.0f;
    }
}

// Inverse CDF over ascending token id: (key, w) per lane, key = SENT_ID (weight 0) for
// empty lanes.  Returns the chosen token; sorts (key, w) ascending in place -- each entry
// goes to the number of entries before it (smaller key, or equal key on a lower lane), a
// permutation -- through the 64 entries of scratch.
__device__ int inverse_cdf_draw(int& key, float& w, float u, int lane, float& Z, float2* scratch) {
    scratch[lane] = make_float2(__int_as_float(key), w);
    __syncwarp();
    int rk = 0;
#pragma unroll
    for (int j = 0; j < 32; ++j) {
        const int o = __float_as_int(scratch[j].x);
        rk += (o < key || (o == key && j < lane)) ? 1 : 0;
    }
    scratch[32 + rk] = make_float2(__int_as_float(key), w);
    __syncwarp();
    const float2 srt = scratch[32 + lane];
    __syncwarp();
    key = __float_as_int(srt.x);
    w = srt.y;
    Z = warp_sum(key != SENT_ID ? w : 0.0f);
    float cum = key != SENT_ID ? w : 0.0f;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const float t = __shfl_up_sync(FULL, cum, o);
        if (lane >= o) cum += t;
    }
    const float target = u * Z;
    const unsigned sel = __ballot_sync(FULL, key != SENT_ID && cum > target);
    const unsigned valid = __ballot_sync(FULL, key != SENT_ID);
    if (valid == 0u) return -1;           // nothing to draw from: no finite logit in the row
    const int src = sel ? __ffs(sel) - 1 : 31 - __clz(valid);
    return __shfl_sync(FULL, key, src);
}

// Acceptance scan of one sequence on one warp, over its rows' truncated distributions in
// shared memory: target position i at list i, draft position i at list kb + 1 + i.
// sdt [K]: the sequence's draft tokens, su [K + 1]: its uniforms (copies in shared memory).
__device__ void finish_sequence(const VerifyParams& p, int b, int lane, const int* rid, const float* rp,
                                const int* sdt, const float* su, float2* scratch) {
    const int kb = draft_count(p, b);
    auto tl = [&](int i) { return i * LISTN + lane; };
    auto dl = [&](int i) { return (kb + 1 + i) * LISTN + lane; };
    const float* ub = su;
    int a = 0, next = -1, status = SPEC_OK;
    int okey = SENT_ID;
    float ow = 0.0f, oZ = 1.0f;
    if (p.temperature == 0.0f) {
        while (a < kb && sdt[a] == rid[a * LISTN]) ++a;
        next = rid[a * LISTN];
        okey = lane == 0 ? next : SENT_ID;
        ow = lane == 0 ? 1.0f : 0.0f;
    } else {
        const bool has_q = p.draft != nullptr;
        bool reject = false;
        a = kb;
        int d = -1;
        // the positions' P(d) and Q(d), SB positions per round with their loads issued
        // together; a list holds each id at most once, so the lane whose id is d (if any)
        // holds its probability.  The scan stops at the first reject.
        constexpr int SB = 4;
        bool done = false;
        for (int i0 = 0; i0 < kb && !done; i0 += SB) {
            float pd[SB], qd[SB];
            int dt[SB];
#pragma unroll
            for (int j = 0; j < SB; ++j) {
                const int i = i0 + j;
                pd[j] = 0.0f; qd[j] = 1.0f; dt[j] = -1;
                if (i < kb) {
                    dt[j] = sdt[i];
                    const unsigned mp = __ballot_sync(FULL, rid[tl(i)] == dt[j]);
                    pd[j] = mp ? rp[i * LISTN + __ffs(mp) - 1] : 0.0f;
                    if (has_q) {
                        const unsigned mq = __ballot_sync(FULL, rid[dl(i)] == dt[j]);
                        qd[j] = mq ? rp[(kb + 1 + i) * LISTN + __ffs(mq) - 1] : 0.0f;
                    }
                }
            }
            for (int j = 0; j < SB && i0 + j < kb; ++j) {
                d = dt[j];
                if (qd[j] == 0.0f) { status = SPEC_E_DRAFT; a = i0 + j; done = true; break; }
                const float ratio = pd[j] / qd[j];
                if (!(ub[i0 + j] < ratio)) { a = i0 + j; reject = true; done = true; break; }
            }
        }
        if (status == SPEC_OK) {
            const int pid = rid[tl(a)];
            const float pp = rp[tl(a)];
            float w = pid >= 0 ? pp : 0.0f;
            if (reject) {
                float qx = 0.0f;
                if (has_q) {
                    const int q0 = (kb + 1 + a) * LISTN;
#pragma unroll 8
                    for (int t = 0; t < LISTN; ++t) {
                        const int tid = rid[q0 + t];
                        if (tid >= 0 && tid == pid) qx = rp[q0 + t];
                    }
                } else {
                    qx = (pid == d) ? 1.0f : 0.0f;
                }
                float r = pid >= 0 ? fmaxf(pp - qx, 0.0f) : 0.0f;
                // residual empty (r >= 0, so a zero sum is no positive lane): fall back to P
                if (__ballot_sync(FULL, r > 0.0f) == 0u) r = w;
                w = r;
            }
            okey = (pid >= 0 && w > 0.0f) ? pid : SENT_ID;
            ow = okey != SENT_ID ? w : 0.0f;
            next = inverse_cdf_draw(okey, ow, ub[p.K], lane, oZ, scratch);
        }
    }
    if (status == SPEC_OK && (next < 0 || next == SENT_ID)) status = SPEC_E_INVAL;
    if (p.out_ids != nullptr) {
        const bool v = okey != SENT_ID && status == SPEC_OK;
        p.out_ids[(size_t)b * SPEC_TOPK_MAX + lane] = v ? okey : -1;
        p.out_probs[(size_t)b * SPEC_TOPK_MAX + lane] = v ? ow / oZ : 0.0f;
    }
    if (lane == 0) {
        p.accepted_len[b] = a;
        p.next_token[b] = status == SPEC_OK ? next : -1;
        if (p.seq_status) p.seq_status[b] = status;
    }
}



__device__ __forceinline__ float max4(const float4& x) { return fmaxf(fmaxf(x.x, x.y), fmaxf(x.z, x.w)); }

__device__ __forceinline__ float comp4(const float4& x, int c) {
    return c == 0 ? x.x : c == 1 ? x.y : c == 2 ? x.z : x.w;
}

// Fine blocks: fine block 4 b + g of block b is the 64 float4 of the block's lanes
// [8 g, 8 g + 8) in pass 1 -- body float4 b * VB4 + l + 32 u for l in that range and u in
// [0, 8).  A warp reading it again takes two of them per lane: l = 8 g + (lane & 7),
// u = (lane >> 3) + 4 h.
__device__ __forceinline__ int fine_float4(int fb, int lane, int h) {
    const int b = fb >> 2, g = fb & 3;
    return b * VB4 + 8 * g + (lane & 7) + 32 * ((lane >> 3) + 4 * h);
}

// Largest and second largest of four values (as a multiset: equal values count twice).
__device__ __forceinline__ void top2_4(const float4& v, float& t1, float& t2) {
    const float h1 = fmaxf(v.x, v.y), l1 = fminf(v.x, v.y);
    const float h2 = fmaxf(v.z, v.w), l2 = fminf(v.z, v.w);
    t1 = fmaxf(h1, h2);
    t2 = fmaxf(fminf(h1, h2), fmaxf(l1, l2));
}

// Maximum over the 8-lane group of the calling lane.
__device__ __forceinline__ float group8_max(float x) {
#pragma unroll
    for (int o = 1; o < 8; o <<= 1) x = fmaxf(x, __shfl_xor_sync(FULL, x, o));
    return x;
}

// (a1, a2) <- the top two of the multiset union of (a1, a2) and (b1, b2).
__device__ __forceinline__ void top2_merge(float& a1, float& a2, float b1, float b2) {
    a2 = fmaxf(fminf(a1, b1), fmaxf(a2, b2));
    a1 = fmaxf(a1, b1);
}

#ifdef VT_TRACE
// Per-row timeline of the last refine launch (profiling builds only): [row][0, 1 start,
// 2 tau, 3 candidates merged, 4 blocks read again, 5 row finished]
__device__ unsigned long long g_vt_trace[4096][6];
#define VT_STAMP(r, i) if (lane == 0 && (r) < 4096) g_vt_trace[r][i] = globaltimer_ns()
// pass 1: [CTA][0 start, 1 end]
__device__ unsigned long long g_vt_p1[1024][2];
#define VT_P1_STAMP(i) if (threadIdx.x == 0 && blockIdx.x < 1024) g_vt_p1[blockIdx.x][i] = globaltimer_ns()
extern "C" int spec_debug_vt_trace(unsigned long long* out) {
    if (cudaMemcpyFromSymbol(out, g_vt_trace, sizeof(g_vt_trace)) != cudaSuccess) return -6;
    return cudaMemcpyFromSymbol(out + 4096 * 6, g_vt_p1, sizeof(g_vt_p1)) == cudaSuccess ? 0 : -6;
}
#else
#define VT_STAMP(r, i) ((void)0)
#define VT_P1_STAMP(i) ((void)0)
#endif

// Pass 1: for every VF-element fine block of each needed row, its largest element with the
// id of one element at that value, and its second largest element (fine block 0 also covers
// the row's unaligned head and tail, at most 3 + 3 scalars).  A warp reads VB elements
// (four fine blocks) at a time, BM_INFLIGHT such blocks before reducing any of them; the
// last (100 - BM_STATIC_PCT) per cent of the blocks are handed out by a counter.
__global__ void __maxnreg__(BM_MAXNREG) vt_stats_kernel(const VerifyParams p) {
    pdl_launch_dependents();     // pass 2 may be scheduled now; it waits per row
    const int lane = threadIdx.x & 31;
    const long long nw = (long long)gridDim.x * (BM_THREADS / 32);
    const long long total = (long long)p.n_rows * p.nbb;
    const long long gw = (long long)blockIdx.x * (BM_THREADS / 32) + (threadIdx.x >> 5);
    // BM_STATIC_PCT per cent of the blocks in static sweeps over all warps, the rest in
    // pairs of consecutive blocks from a counter (SMs do not stream at the same rate)
    const long long sweep = nw * BM_INFLIGHT;
    const long long n_static = (total * BM_STATIC_PCT / 100) / sweep;
    const long long dyn0 = n_static * sweep;
    int nextb = 0;               // lane 0: the next dynamic grab, fetched one iteration ahead
    if (n_static == 0 && lane == 0) nextb = atomicAdd(p.blk_next, BM_INFLIGHT);
    VT_P1_STAMP(0);
    for (long long it = 0;; ++it) {
        long long w0, wstep;
        if (it < n_static) {
            w0 = gw + it * sweep;
            wstep = nw;
        } else {
            const int nb = __shfl_sync(FULL, nextb, 0);
            w0 = dyn0 + nb;
            wstep = 1;
            if (nb < 0 || w0 >= total) break;     // the counter starts at 0 (cleared by the host)
        }
        float4 x[BM_INFLIGHT][VB4 / 32];
        int row[BM_INFLIGHT], blk[BM_INFLIGHT];
        bool act[BM_INFLIGHT];
        const float* ptr[BM_INFLIGHT];
        int head[BM_INFLIGHT], body[BM_INFLIGHT];
#pragma unroll
        for (int j = 0; j < BM_INFLIGHT; ++j) {
            const long long w = w0 + j * wstep;
            act[j] = false;
            row[j] = 0; blk[j] = 0; ptr[j] = nullptr; head[j] = 0; body[j] = 0;
            if (w < total) {
                row[j] = (int)(w / p.nbb);
                blk[j] = (int)(w - (long long)row[j] * p.nbb);
                const RowInfo ri = row_info(p, row[j]);
                act[j] = row_needed(p, ri);
                ptr[j] = ri.ptr;
                row_split(ri.ptr, p.V, head[j], body[j]);
            }
            const int n4 = act[j] ? min(VB4, (body[j] >> 2) - blk[j] * VB4) : 0;
            const float4* src = reinterpret_cast<const float4*>(ptr[j] + head[j]) + (size_t)blk[j] * VB4;
#pragma unroll
            for (int u = 0; u < VB4 / 32; ++u) {
                const int idx = lane + 32 * u;
                x[j][u] = idx < n4 ? __ldcs(src + idx) : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
            }
        }
        if (lane == 0 && it + 1 >= n_static) nextb = atomicAdd(p.blk_next, BM_INFLIGHT);
#pragma unroll
        for (int j = 0; j < BM_INFLIGHT; ++j) {
            if (!act[j]) continue;      // uniform over the warp
            // fine block g = lanes [8 g, 8 g + 8), all eight of their float4 (fine_block_lanes)
            const int n4 = min(VB4, (body[j] >> 2) - blk[j] * VB4);
            const int g = lane >> 3;
            float a1 = -INFINITY, a2 = -INFINITY, hm[VB4 / 32];
#pragma unroll
            for (int u = 0; u < VB4 / 32; ++u) {
                float t1, t2;
                top2_4(x[j][u], t1, t2);
                hm[u] = t1;
                top2_merge(a1, a2, t1, t2);
            }
            float sh = -INFINITY, st = -INFINITY;               // block 0: head and tail scalars
            int tail0 = 0;
            if (blk[j] == 0) {
                tail0 = head[j] + body[j];
                if (lane < head[j]) sh = ptr[j][lane];
                if (lane < p.V - tail0) st = ptr[j][tail0 + lane];
                top2_merge(a1, a2, sh, -INFINITY);
                top2_merge(a1, a2, st, -INFINITY);
            }
            const float M1 = group8_max(a1);
            const unsigned eq = (__ballot_sync(FULL, a1 == M1) >> (8 * g)) & 0xffu;
            const int L = 8 * g + __ffs(eq) - 1;
            // the block's second largest: the other lanes' maxima and lane L's second
            const float M2 = group8_max(lane == L ? a2 : a1);
            // lane's first element (in id order: head, body, tail) equal to its maximum
            int id = SENT_ID;
            if (blk[j] == 0 && lane < p.V - tail0 && st == a1) id = tail0 + lane;
            {
                int uf = -1;
#pragma unroll
                for (int u = VB4 / 32 - 1; u >= 0; --u) uf = hm[u] == a1 ? u : uf;
                if (uf >= 0 && lane + 32 * uf < n4) {
                    float4 xv = x[j][0];
#pragma unroll
                    for (int u = 1; u < VB4 / 32; ++u) xv = uf == u ? x[j][u] : xv;
                    const int c = xv.x == a1 ? 0 : xv.y == a1 ? 1 : xv.z == a1 ? 2 : 3;
                    id = head[j] + 4 * (blk[j] * VB4 + lane + 32 * uf) + c;
                }
            }
            if (blk[j] == 0 && lane < head[j] && sh == a1) id = lane;
            const int idL = __shfl_sync(FULL, id, L);
            // lane 0 stores the four blocks' statistics (group leaders 0, 8, 16, 24)
            float r1[NF], r2[NF], rid[NF];
#pragma unroll
            for (int f = 0; f < NF; ++f) {
                r1[f] = __shfl_sync(FULL, M1, 8 * f);
                r2[f] = __shfl_sync(FULL, M2, 8 * f);
                rid[f] = __int_as_float(__shfl_sync(FULL, idL, 8 * f));
            }
            if (lane == 0) {
                static_assert(NF == 4, "a block's fine statistics are stored as float4s");
                const size_t fi = (size_t)row[j] * p.nbb * NF + (size_t)blk[j] * NF;
                float4* k4 = reinterpret_cast<float4*>(p.fk + fi);
                k4[0] = make_float4(r1[0], rid[0], r1[1], rid[1]);
                k4[1] = make_float4(r1[2], rid[2], r1[3], rid[3]);
                *reinterpret_cast<float4*>(p.fm2 + fi) = make_float4(r2[0], r2[1], r2[2], r2[3]);
            }
        }
    }
    VT_P1_STAMP(1);
}

// Append each lane's (v, id) for which c holds to the warp's buffer, in lane order (ballot
// + prefix count).
__device__ __forceinline__ void append_if(bool c, float v, int id, float2* pool, int& cnt, int lane) {
    const unsigned m = __ballot_sync(FULL, c);
    if (c) pool[cnt + __popc(m & ((1u << lane) - 1u))] = make_float2(v, __int_as_float(id));
    cnt += __popc(m);
}

// Append each lane's index x for which c holds to the warp's list, in lane order.
__device__ __forceinline__ void append_index(bool c, int x, int* list, int& n, int lane) {
    const unsigned m = __ballot_sync(FULL, c);
    if (c) list[n + __popc(m & ((1u << lane) - 1u))] = x;
    n += __popc(m);
}

// Read the n listed fine blocks of the row again, RF_BATCH at a time, and merge their
// elements >= tau2 -- all but the block's recorded maximum (already listed) -- into the
// warp's list (lv, lid).  pool/outl: the warp's candidate pool (empty on entry and exit)
// and merge output.
__device__ __forceinline__ void reread_blocks(const VerifyParams& p, const RowInfo& ri, int row, const int* sel,
                                              int n, float tau2, int head, int body, float& lv, int& lid,
                                              float2* pool, float2* outl, int lane) {
    const int n4_row = body >> 2;
    const float4* src = reinterpret_cast<const float4*>(ri.ptr + head);
    const size_t krow = (size_t)row * NF * p.nbb;
    int cnt = 0;
    for (int i0 = 0; i0 < n; i0 += RF_BATCH) {
        int fb[RF_BATCH], skip[RF_BATCH];
        float4 x[RF_BATCH][2];
#pragma unroll
        for (int j = 0; j < RF_BATCH; ++j) {
            fb[j] = i0 + j < n ? sel[i0 + j] : -1;
            skip[j] = fb[j] >= 0 ? __float_as_int(__ldcg(&p.fk[krow + fb[j]].y)) : SENT_ID;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int idx = fine_float4(fb[j], lane, h);
                x[j][h] = (fb[j] >= 0 && idx < n4_row)
                              ? __ldcs(src + idx) : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
            }
        }
#pragma unroll
        for (int j = 0; j < RF_BATCH; ++j) {
            if (fb[j] < 0) continue;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                if (cnt > RF_CAND_CAP - LISTN - 128) {
                    flush_candidates(lv, lid, pool, outl, cnt, lane);
                    cnt = 0;
                }
                const int idx = fine_float4(fb[j], lane, h);
                const int e = head + 4 * idx;
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const float v = comp4(x[j][h], c);
                    append_if(idx < n4_row && e + c != skip[j] && v >= tau2, v, e + c, pool, cnt, lane);
                }
            }
            if (fb[j] == 0) {      // the unaligned head and tail belong to fine block 0
                if (cnt > RF_CAND_CAP - LISTN - 64) {
                    flush_candidates(lv, lid, pool, outl, cnt, lane);
                    cnt = 0;
                }
                const int tail0 = head + body;
                const bool hok = lane < head, tok = lane < p.V - tail0;
                const float hv = hok ? ri.ptr[lane] : -INFINITY;
                const float tv = tok ? ri.ptr[tail0 + lane] : -INFINITY;
                append_if(hok && lane != skip[j] && hv >= tau2, hv, lane, pool, cnt, lane);
                append_if(tok && tail0 + lane != skip[j] && tv >= tau2, tv, tail0 + lane, pool, cnt, lane);
            }
        }
    }
    flush_candidates(lv, lid, pool, outl, cnt, lane);
}

// One row of pass 2 on one warp.  Candidates are the fine blocks' maxima:
// tau, the k-th largest of the 32 lanes' maxima over their shares of them, is at most the
// row's k-th largest element, so only blocks with a maximum >= tau can hold a top-k element
// at their maximum.  The top list of those candidates has k-th value tau2; any element other
// than a block's recorded maximum is at most the block's second largest value, so a block
// whose second value is below tau2 holds nothing else of the top k.  The few blocks whose
// second value reaches tau2 are read again and their other elements >= tau2 merged in.
// Returns lane j's entry of the row's top list (j-th best).
__device__ __forceinline__ ListEntry refine_row(const VerifyParams& p, int row, int lane, float2* pool,
                                                float2* outl, int* sel) {
    const RowInfo ri = row_info(p, row);
    VT_STAMP(row, 0);
    VT_STAMP(row, 1);
    const int k = p.top_k;
    const int nbb = p.nbb, nfb = NF * nbb;
    const int nq = nfb / 2;                                  // float4 = two (maximum, id) pairs
    const float4* kq = reinterpret_cast<const float4*>(p.fk + (size_t)row * nfb);
    const float4* m2q = reinterpret_cast<const float4*>(p.fm2 + (size_t)row * nfb);
    const float4 NEG = make_float4(-INFINITY, __int_as_float(SENT_ID), -INFINITY, __int_as_float(SENT_ID));
    // the first round of (maximum, id) pairs and second values, loaded together
    float4 kv[RF_KPL], mv[RF_BPL];
#pragma unroll
    for (int i = 0; i < RF_KPL; ++i) {
        const int q = lane + 32 * i;
        kv[i] = q < nq ? __ldcg(kq + q) : NEG;
    }
#pragma unroll
    for (int i = 0; i < RF_BPL; ++i) {
        const int b = lane + 32 * i;
        mv[i] = b < nbb ? __ldcg(m2q + b) : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
    }
    float lm = -INFINITY;
#pragma unroll
    for (int i = 0; i < RF_KPL; ++i) lm = fmaxf(lm, fmaxf(kv[i].x, kv[i].z));
    for (int q = lane + 32 * RF_KPL; q < nq; q += 32) {
        const float4 t = __ldcg(kq + q);
        lm = fmaxf(lm, fmaxf(t.x, t.z));
    }
    // tau: the k-th best lane maximum, from each lane's rank among the 32 (ties to the lower
    // lane, so the ranks are 0..31 once each)
    float* lmx = reinterpret_cast<float*>(outl);
    lmx[lane] = lm;
    __syncwarp();
    int rk = 0;
#pragma unroll
    for (int j = 0; j < 32; ++j) {
        const float o = lmx[j];
        rk += (o > lm || (o == lm && j < lane)) ? 1 : 0;
    }
    const unsigned at = __ballot_sync(FULL, rk == k - 1);
    const float tau = at ? lmx[__ffs(at) - 1] : -INFINITY;
    __syncwarp();
    VT_STAMP(row, 2);

    // candidates: the maxima >= tau
    float lv = -INFINITY;
    int lid = SENT_ID;
    int cnt = 0;
    for (int q0 = 0; q0 < nq; q0 += 32 * RF_KPL) {
        if (q0 > 0) {
#pragma unroll
            for (int i = 0; i < RF_KPL; ++i) {
                const int q = q0 + lane + 32 * i;
                kv[i] = q < nq ? __ldcg(kq + q) : NEG;
            }
        }
        // bit 2i / 2i+1: the lane's pair i.x / i.z is a candidate; each lane's place in the
        // pool is the candidates of the lanes below it, from ballots of the count's bits
        unsigned mb = 0;
#pragma unroll
        for (int i = 0; i < RF_KPL; ++i) {
            mb |= (__float_as_int(kv[i].y) != SENT_ID && kv[i].x >= tau ? 1u : 0u) << (2 * i);
            mb |= (__float_as_int(kv[i].w) != SENT_ID && kv[i].z >= tau ? 1u : 0u) << (2 * i + 1);
        }
        const int c = __popc(mb);
        const unsigned lt = (1u << lane) - 1u;
        int before = 0, total = 0;
#pragma unroll
        for (int bit = 0; bit < 5; ++bit) {                  // c <= 2 RF_KPL < 32
            const unsigned bm = __ballot_sync(FULL, (c >> bit) & 1);
            before += __popc(bm & lt) << bit;
            total += __popc(bm) << bit;
        }
        if (cnt > 0 && cnt + total > RF_CAND_CAP - LISTN) {
            flush_candidates(lv, lid, pool, outl, cnt, lane);
            cnt = 0;
        }
        if (total <= RF_CAND_CAP - LISTN) {
            int pos = cnt + before;
#pragma unroll
            for (int i = 0; i < RF_KPL; ++i) {
                if ((mb >> (2 * i)) & 1u) pool[pos++] = make_float2(kv[i].x, kv[i].y);
                if ((mb >> (2 * i + 1)) & 1u) pool[pos++] = make_float2(kv[i].z, kv[i].w);
            }
            cnt += total;
        } else {
            // more than a pool of candidates in one round (rows of many equal maxima): in turns
#pragma unroll
            for (int i = 0; i < RF_KPL; ++i) {
                if (cnt > RF_CAND_CAP - LISTN - 64) {
                    flush_candidates(lv, lid, pool, outl, cnt, lane);
                    cnt = 0;
                }
                append_if((mb >> (2 * i)) & 1u, kv[i].x, __float_as_int(kv[i].y), pool, cnt, lane);
                append_if((mb >> (2 * i + 1)) & 1u, kv[i].z, __float_as_int(kv[i].w), pool, cnt, lane);
            }
        }
    }
    flush_candidates(lv, lid, pool, outl, cnt, lane);
    cnt = 0;
    const float tau2 = __shfl_sync(FULL, lv, k - 1);
    VT_STAMP(row, 3);

    // blocks whose second value reaches tau2: read again, every element >= tau2 but the
    // recorded maximum joins the list.  Each lane keeps a bit per fine block of its share
    // (RF_BPL blocks of 4) and hands them out one per step into the warp's list.
    int head, body;
    row_split(ri.ptr, p.V, head, body);
    int n = 0;
    for (int b0 = 0; b0 < nbb; b0 += 32 * RF_BPL) {
        if (b0 > 0) {
#pragma unroll
            for (int i = 0; i < RF_BPL; ++i) {
                const int b = b0 + lane + 32 * i;
                mv[i] = b < nbb ? __ldcg(m2q + b) : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
            }
        }
        unsigned bits = 0;
#pragma unroll
        for (int i = 0; i < RF_BPL; ++i) {
            if (b0 + lane + 32 * i < nbb) {
                bits |= (mv[i].x >= tau2 ? 1u : 0u) << (4 * i);
                bits |= (mv[i].y >= tau2 ? 2u : 0u) << (4 * i);
                bits |= (mv[i].z >= tau2 ? 4u : 0u) << (4 * i);
                bits |= (mv[i].w >= tau2 ? 8u : 0u) << (4 * i);
            }
        }
        while (true) {
            const bool more = __any_sync(FULL, bits != 0);
            if (more) {
                int fbi = -1;
                if (bits) {
                    const int t = __ffs(bits) - 1;
                    bits &= bits - 1;
                    fbi = 4 * (b0 + lane + 32 * (t >> 2)) + (t & 3);
                }
                append_index(fbi >= 0, fbi, sel, n, lane);
            }
            const bool last = !more && b0 + 32 * RF_BPL >= nbb;
            if (n > RF_SEL_CAP - 32 || (last && n > 0)) {
                __syncwarp();
                reread_blocks(p, ri, row, sel, n, tau2, head, body, lv, lid, pool, outl, lane);
                n = 0;
            }
            if (!more) break;
        }
    }
    VT_STAMP(row, 4);
    return ListEntry{lv, lid};
}

// Pass 2.  Verify: one CTA per sequence, one warp per row of the sequence (rows beyond the
// CTA's warps are taken in turn); each row's truncated distribution goes to shared memory
// and warp 0 runs the sequence's acceptance scan there.  Sample: one warp per row, which
// draws its token itself.  Launched programmatically dependent on pass 1: the CTAs may be
// resident early, the statistics are read after pass 1 is done.
// Dynamic shared memory: per warp a pool of RF_CAND_CAP (value, id) entries, a merge output
// of LISTN and RF_SEL_CAP fine block indices, then (verify) the sequence's lists, ids then
// probabilities (room for 2K + 1 rows), its K draft tokens and K + 1 uniforms.
__global__ void __launch_bounds__(RF_MAX_WARPS * 32) vt_refine_kernel(const VerifyParams p) {
    extern __shared__ __align__(16) unsigned char rf_smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nwarps = blockDim.x >> 5;
    float2* pool = reinterpret_cast<float2*>(reinterpret_cast<float*>(rf_smem) + warp * RF_WARP_WORDS);
    float2* outl = pool + RF_CAND_CAP;
    int* sel = reinterpret_cast<int*>(outl + LISTN);
    // inputs (draft tokens, uniforms, draft lengths) are complete before pass 1 starts, so
    // they are read while it runs; pass 1's statistics only after pdl_wait()
    if (p.mode == MODE_SAMPLE) {
        const int row = blockIdx.x * nwarps + warp;
        const float ur = row < p.n_rows ? p.u[row] : 0.0f;
        pdl_wait();
        if (row >= p.n_rows) return;
        const ListEntry e = refine_row(p, row, lane, pool, outl, sel);
        int key;
        float w;
        row_dist(p, e.v, e.id, lane, key, w);
        if (key < 0 || !(w > 0.0f)) { key = SENT_ID; w = 0.0f; }     // as the verify scan: weight > 0
        float Z;
        const int tok = inverse_cdf_draw(key, w, ur, lane, Z, pool);
        if (lane == 0) p.out_tokens[row] = tok;
        VT_STAMP(row, 5);
        return;
    }
    const int b = blockIdx.x;
    const int kb = draft_count(p, b);
    const int nr = (kb + 1) + (p.draft != nullptr ? kb : 0);
    const int nr_max = (p.K + 1) + (p.draft != nullptr ? p.K : 0);
    int* rid = reinterpret_cast<int*>(rf_smem) + nwarps * RF_WARP_WORDS;
    float* rp = reinterpret_cast<float*>(rid + nr * LISTN);
    int* sdt = rid + 2 * nr_max * LISTN;
    float* su = reinterpret_cast<float*>(sdt + p.K);
    for (int t = threadIdx.x; t < 2 * p.K + 1; t += blockDim.x) {
        if (t < p.K) sdt[t] = t < kb ? p.draft_tokens[(size_t)b * p.K + t] : -1;
        else su[t - p.K] = p.u[(size_t)b * (p.K + 1) + (t - p.K)];
    }
    pdl_wait();
    for (int r = warp; r < nr; r += nwarps) {
        const int row = r <= kb ? b * (p.K + 1) + r : p.n_target_rows + b * p.K + (r - kb - 1);
        const ListEntry e = refine_row(p, row, lane, pool, outl, sel);
        row_dist(p, e.v, e.id, lane, rid[r * LISTN + lane], rp[r * LISTN + lane]);
        VT_STAMP(row, 5);
    }
    __syncthreads();
    if (warp == 0) finish_sequence(p, b, lane, rid, rp, sdt, su, pool);
}

// ---- host side ---------------------------------------------------------------------------

struct Plan {
    int n_rows, nbb;
    size_t off_blk, off_fk, off_fm2, total, counters_bytes;
};

static inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// largest pass-2 shared memory: RF_MAX_WARPS warps, the lists of 2 VT_MAX_K + 1 rows, the
// draft tokens and uniforms
constexpr int RF_SMEM_MAX = (RF_MAX_WARPS * RF_WARP_WORDS + 2 * (2 * VT_MAX_K + 1) * LISTN + 2 * VT_MAX_K + 1) * 4;

static Plan make_plan(int n_rows_max, int V) {
    Plan pl{};
    pl.n_rows = n_rows_max;
    pl.nbb = (V + VB - 1) / VB;
    size_t o = 0;
    pl.off_blk = o; o += 4;
    pl.counters_bytes = o;
    o = align256(o);
    pl.off_fk = o; o = align256(o + (size_t)n_rows_max * pl.nbb * NF * 8);
    pl.off_fm2 = o; o = align256(o + (size_t)n_rows_max * pl.nbb * NF * 4);
    pl.total = o;
    return pl;
}

// SM count of the current device; the first call on a device also sets pass 1's shared
// memory carveout (pass 1 uses none: a small carveout leaves L1, which holds its loads in
// flight, large -- a 100% carveout measured 15% slower) and pass 2's dynamic shared memory
// limit.
static int device_setup() {
    constexpr int MAX_DEV = 64;
    static std::atomic<int> sms[MAX_DEV];
    static std::mutex mu;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return -1;
    if (dev < MAX_DEV && sms[dev].load() > 0) return sms[dev].load();
    std::lock_guard<std::mutex> lock(mu);
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return -1;
    if (cudaFuncSetAttribute(vt_stats_kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                             BM_SMEM_CARVEOUT) != cudaSuccess ||
        cudaFuncSetAttribute(vt_refine_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, RF_SMEM_MAX) !=
            cudaSuccess)
        return -1;
    if (dev < MAX_DEV) sms[dev].store(n);
    return n;
}

// Attributes of the verify kernels on the current device, set before any stream capture.
int verify_prepare() { return device_setup() > 0 ? SPEC_OK : SPEC_E_CUDA; }

static int launch_verify(VerifyParams& prm, const Plan& pl, void* ws, cudaStream_t st) {
    uint8_t* w = static_cast<uint8_t*>(ws);
    prm.blk_next = reinterpret_cast<int*>(w + pl.off_blk);
    prm.fk = reinterpret_cast<float2*>(w + pl.off_fk);
    prm.fm2 = reinterpret_cast<float*>(w + pl.off_fm2);
    prm.nbb = pl.nbb;

    cudaError_t e = cudaMemsetAsync(ws, 0, pl.counters_bytes, st);
    if (e != cudaSuccess) return set_error(SPEC_E_CUDA, "cudaMemsetAsync: %s", cudaGetErrorString(e));
    const int nsm = device_setup();
    if (nsm <= 0) return set_error(SPEC_E_CUDA, "no CUDA device, or its verify kernel attributes could not be set");
    const long long blocks = (long long)prm.n_rows * pl.nbb;
    const long long warps_needed = (blocks + BM_INFLIGHT - 1) / BM_INFLIGHT;
    const int grid1 = (int)std::max(1LL, std::min((long long)nsm * BM_CTAS_PER_SM, (warps_needed + 7) / 8));
    vt_stats_kernel<<<grid1, BM_THREADS, 0, st>>>(prm);
    cudaLaunchConfig_t cfg = {};
    if (prm.mode == MODE_SAMPLE) {
        cfg.gridDim = dim3((prm.n_rows + RF_SAMPLE_WARPS - 1) / RF_SAMPLE_WARPS);
        cfg.blockDim = dim3(RF_SAMPLE_WARPS * 32);
        cfg.dynamicSmemBytes = (size_t)RF_SAMPLE_WARPS * RF_WARP_WORDS * 4;
    } else {
        const int nr_max = (prm.K + 1) + (prm.draft != nullptr ? prm.K : 0);
        const int nw = std::min(nr_max, RF_MAX_WARPS);
        cfg.gridDim = dim3(prm.B);
        cfg.blockDim = dim3(nw * 32);
        cfg.dynamicSmemBytes = ((size_t)nw * RF_WARP_WORDS + (size_t)2 * nr_max * LISTN + 2 * (size_t)prm.K + 1) * 4;
    }
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, vt_refine_kernel, prm);
    if (e != cudaSuccess) return set_error(SPEC_E_CUDA, "vt_refine_kernel launch: %s", cudaGetErrorString(e));
    e = cudaGetLastError();
    if (e != cudaSuccess) return set_error(SPEC_E_CUDA, "verify kernel launch: %s", cudaGetErrorString(e));
    return SPEC_OK;
}

static int check_sampling(const spec_sampling* s, int V, int& k_eff) {
    if (s == nullptr) return set_error(SPEC_E_INVAL, "sampling is NULL");
    if (!(s->temperature >= 0.0f) || std::isinf(s->temperature))
        return set_error(SPEC_E_INVAL, "temperature must be finite and >= 0");
    if (s->temperature == 0.0f) { k_eff = 1; return SPEC_OK; }
    if (s->top_k < 1 || s->top_k > SPEC_TOPK_MAX)
        return set_error(SPEC_E_INVAL, "top_k must be in [1, %d] when temperature > 0", SPEC_TOPK_MAX);
    if (!(s->top_p >= 0.0f)) return set_error(SPEC_E_INVAL, "top_p must be >= 0");
    k_eff = std::min(s->top_k, V);
    return SPEC_OK;
}


// The B (2K + 1) rows of a call (target and draft) are counted in int and their logits
// addressed with 40-bit offsets: both limits hold for any size the library is meant for.
static bool rows_fit(int B, int K, int V) {
    const long long rows = (long long)B * (2 * K + 1);
    return rows < (1LL << 30) && rows * (long long)V < (1LL << 40);
}

// Validation + launch of the fused verify (used by spec_verify_logits and spec_verify).
int verify_into(int B, int K, int V, const float* target_logits, const float* draft_logits,
                const int32_t* draft_tokens, const int32_t* draft_len, const float* uniforms,
                const spec_sampling* sampling, int32_t* accepted_len, int32_t* next_token, int32_t* out_ids,
                float* out_probs, int32_t* seq_status, void* workspace, size_t workspace_bytes, cudaStream_t st) {
    if (B < 1 || K < 0 || V < 2) return set_error(SPEC_E_INVAL, "bad sizes B=%d K=%d V=%d", B, K, V);
    if (K > VT_MAX_K) return set_error(SPEC_E_INVAL, "K=%d above the maximum %d", K, VT_MAX_K);
    if (!rows_fit(B, K, V)) return set_error(SPEC_E_RANGE, "logits too large");
    int k_eff = 1;
    int rc = check_sampling(sampling, V, k_eff);
    if (rc != SPEC_OK) return rc;
    if (!target_logits || !uniforms || !accepted_len || !next_token || !workspace)
        return set_error(SPEC_E_INVAL, "NULL required pointer");
    if (K > 0 && !draft_tokens) return set_error(SPEC_E_INVAL, "draft_tokens is NULL");
    if ((out_ids == nullptr) != (out_probs == nullptr))
        return set_error(SPEC_E_INVAL, "out_ids and out_probs must both be given or both be NULL");
    if (reinterpret_cast<uintptr_t>(workspace) & 255) return set_error(SPEC_E_INVAL, "workspace not 256-byte aligned");
    if ((reinterpret_cast<uintptr_t>(target_logits) & 3) || (reinterpret_cast<uintptr_t>(draft_logits) & 3))
        return set_error(SPEC_E_INVAL, "logits must be 4-byte aligned");
    const Plan pl = make_plan(B * (2 * K + 1), V);
    if (workspace_bytes < pl.total)
        return set_error(SPEC_E_NOMEM, "workspace %zu bytes < required %zu", workspace_bytes, pl.total);

    VerifyParams prm{};
    prm.target = target_logits;
    const bool sampling_mode = sampling->temperature != 0.0f;
    prm.draft = (sampling_mode && K > 0) ? draft_logits : nullptr;
    prm.draft_tokens = draft_tokens;
    prm.draft_len = draft_len;
    prm.u = uniforms;
    prm.B = B; prm.K = K; prm.V = V;
    prm.temperature = sampling->temperature;
    prm.top_k = k_eff;
    prm.top_p = sampling->top_p;
    prm.mode = MODE_VERIFY;
    prm.n_target_rows = B * (K + 1);
    prm.n_rows = prm.n_target_rows + (prm.draft ? B * K : 0);
    prm.accepted_len = accepted_len;
    prm.next_token = next_token;
    prm.out_ids = out_ids;
    prm.out_probs = out_probs;
    prm.seq_status = seq_status;
    prm.out_tokens = nullptr;
    return launch_verify(prm, pl, workspace, st);
}

}  // namespace sv

namespace sv {

// Greedy verify from the lm_head epilogue's per-tile argmax keys (amax_key, [M][n_tiles]):
// one CTA per sequence; its warps merge each needed row's keys (the row's largest logit,
// lowest id on ties: the argmax the top-k pass takes from the full logits), then warp 0
// applies the greedy rule (accept drafts while they equal the row's argmax).  Outputs as
// verify_into's greedy mode: out_ids[b][0] = next token with probability 1, the rest -1 / 0.
constexpr int GA_WARPS = 8;
__global__ void __launch_bounds__(GA_WARPS * 32) greedy_amax_kernel(
    const unsigned long long* __restrict__ keys, int n_tiles, int K, const int32_t* __restrict__ draft_tokens,
    const int32_t* __restrict__ draft_len, int32_t* accepted_len, int32_t* next_token, int32_t* out_ids,
    float* out_probs, int32_t* seq_status) {
    __shared__ int amax[VT_MAX_K + 1];
    const int b = blockIdx.x;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    int kb = K;
    if (draft_len != nullptr) kb = min(max(draft_len[b], 0), K);
    for (int i = warp; i <= kb; i += GA_WARPS) {
        const unsigned long long* row = keys + (size_t)(b * (K + 1) + i) * n_tiles;
        unsigned long long best = 0;
        for (int t = lane; t < n_tiles; t += 32) {
            const unsigned long long k = __ldcg(row + t);
            best = k > best ? k : best;
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const unsigned long long x = __shfl_xor_sync(FULL, best, o);
            best = x > best ? x : best;
        }
        if (lane == 0) amax[i] = (int)(0xFFFFFFFFu - (uint32_t)(best & 0xFFFFFFFFull));
    }
    __syncthreads();
    if (warp != 0) return;
    int a = 0;
    while (a < kb && draft_tokens[(size_t)b * K + a] == amax[a]) ++a;
    const int next = amax[a];
    if (out_ids != nullptr) {
        out_ids[(size_t)b * SPEC_TOPK_MAX + lane] = lane == 0 ? next : -1;
        out_probs[(size_t)b * SPEC_TOPK_MAX + lane] = lane == 0 ? 1.0f : 0.0f;
    }
    if (lane == 0) {
        accepted_len[b] = a;
        next_token[b] = next;
        if (seq_status) seq_status[b] = SPEC_OK;
    }
}

int launch_greedy_amax(const unsigned long long* keys, int n_tiles, int B, int K, const int32_t* draft_tokens,
                       const int32_t* draft_len, int32_t* accepted_len, int32_t* next_token, int32_t* out_ids,
                       float* out_probs, int32_t* seq_status, cudaStream_t st) {
    if (K < 0 || K > VT_MAX_K) return set_error(SPEC_E_INVAL, "K=%d outside [0, %d]", K, VT_MAX_K);
    if ((out_ids == nullptr) != (out_probs == nullptr))
        return set_error(SPEC_E_INVAL, "out_ids and out_probs must both be given or both be NULL");
    greedy_amax_kernel<<<B, GA_WARPS * 32, 0, st>>>(keys, n_tiles, K, draft_tokens, draft_len, accepted_len, next_token,
                                                   out_ids, out_probs, seq_status);
    const cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? SPEC_OK : set_error(SPEC_E_CUDA, "greedy_amax_kernel launch: %s", cudaGetErrorString(e));
}

}  // namespace sv

using namespace sv;

extern "C" size_t spec_verify_logits_workspace_bytes(int B, int K, int V) {
    if (B < 1 || K < 0 || V < 2 || K > VT_MAX_K || !rows_fit(B, K, V)) return 0;
    return make_plan(B * (2 * K + 1), V).total;
}

extern "C" int spec_verify_logits(int B, int K, int V, const float* target_logits, const float* draft_logits,
                                  const int32_t* draft_tokens, const int32_t* draft_len, const float* uniforms,
                                  const spec_sampling* sampling, int32_t* accepted_len, int32_t* next_token,
                                  int32_t* out_ids, float* out_probs, int32_t* seq_status, void* workspace,
                                  size_t workspace_bytes, void* stream) {
    clear_error();
    return verify_into(B, K, V, target_logits, draft_logits, draft_tokens, draft_len, uniforms, sampling,
                       accepted_len, next_token, out_ids, out_probs, seq_status, workspace, workspace_bytes,
                       static_cast<cudaStream_t>(stream));
}

extern "C" size_t spec_sample_logits_workspace_bytes(int R, int V) {
    if (R < 1 || V < 2) return 0;
    return make_plan(R, V).total;
}

extern "C" int spec_sample_logits(int R, int V, const float* logits, const float* uniforms,
                                  const spec_sampling* sampling, int32_t* out_tokens, void* workspace,
                                  size_t workspace_bytes, void* stream) {
    clear_error();
    if (R < 1 || V < 2) return set_error(SPEC_E_INVAL, "bad sizes R=%d V=%d", R, V);
    int k_eff = 1;
    int rc = check_sampling(sampling, V, k_eff);
    if (rc != SPEC_OK) return rc;
    if (!logits || !uniforms || !out_tokens || !workspace) return set_error(SPEC_E_INVAL, "NULL required pointer");
    if (reinterpret_cast<uintptr_t>(workspace) & 255) return set_error(SPEC_E_INVAL, "workspace not 256-byte aligned");
    if (reinterpret_cast<uintptr_t>(logits) & 3) return set_error(SPEC_E_INVAL, "logits must be 4-byte aligned");
    const Plan pl = make_plan(R, V);
    if (workspace_bytes < pl.total)
        return set_error(SPEC_E_NOMEM, "workspace %zu bytes < required %zu", workspace_bytes, pl.total);
    VerifyParams prm{};
    prm.target = logits;
    prm.u = uniforms;
    prm.B = R; prm.K = 0; prm.V = V;
    prm.temperature = sampling->temperature;
    prm.top_k = k_eff;
    prm.top_p = sampling->top_p;
    prm.mode = MODE_SAMPLE;
    prm.n_target_rows = R;
    prm.n_rows = R;
    prm.out_tokens = out_tokens;
    return launch_verify(prm, pl, workspace, static_cast<cudaStream_t>(stream));
}

// ---- allocation-free variant -------------------------------------------------------------
//
// Scratch for spec_verify_logits_noalloc: a fixed-size array that every GPU loading the
// library holds for the life of the process.  Host code may not pass `g_noalloc_scratch`
// to a kernel (on the host the name is only a stand-in); the device address is looked up
// once per device with cudaGetSymbolAddress and cached.
namespace sv {
constexpr size_t NOALLOC_SCRATCH_BYTES = 8u << 20;      // 8 MiB
static __device__ __align__(256) uint8_t g_noalloc_scratch[NOALLOC_SCRATCH_BYTES];
constexpr int NOALLOC_MAX_DEVICES = 64;
static void* g_noalloc_ptr[NOALLOC_MAX_DEVICES] = {};
static std::mutex g_noalloc_mu;

static int noalloc_scratch(void** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return set_error(SPEC_E_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
    if (dev < 0 || dev >= NOALLOC_MAX_DEVICES) return set_error(SPEC_E_RANGE, "device ordinal %d too large", dev);
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    if (g_noalloc_ptr[dev] == nullptr) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess || p == nullptr)
            return set_error(SPEC_E_CUDA, "cudaGetSymbolAddress: %s", cudaGetErrorString(e));
        g_noalloc_ptr[dev] = p;
    }
    *out = g_noalloc_ptr[dev];
    return SPEC_OK;
}
}  // namespace sv

extern "C" size_t spec_verify_logits_noalloc_max_bytes(void) { return sv::NOALLOC_SCRATCH_BYTES; }

extern "C" int spec_verify_logits_noalloc(int B, int K, int V, const float* target_logits, const float* draft_logits,
                                          const int32_t* draft_tokens, const int32_t* draft_len, const float* uniforms,
                                          const spec_sampling* sampling, int32_t* accepted_len, int32_t* next_token,
                                          int32_t* out_ids, float* out_probs, int32_t* seq_status, void* stream) {
    clear_error();
    const size_t need = spec_verify_logits_workspace_bytes(B, K, V);
    if (need == 0) {
        if (B < 1 || K < 0 || V < 2 || K > sv::VT_MAX_K) return set_error(SPEC_E_INVAL, "bad sizes B=%d K=%d V=%d", B, K, V);
        return set_error(SPEC_E_RANGE, "B=%d K=%d V=%d is above the built-in scratch of %zu bytes", B, K, V,
                         sv::NOALLOC_SCRATCH_BYTES);
    }
    if (need > sv::NOALLOC_SCRATCH_BYTES)
        return set_error(SPEC_E_RANGE, "B=%d K=%d V=%d needs %zu bytes of scratch, above the built-in %zu", B, K, V,
                         need, sv::NOALLOC_SCRATCH_BYTES);
    void* scratch = nullptr;
    const int rc = sv::noalloc_scratch(&scratch);
    if (rc != SPEC_OK) return rc;
    return sv::verify_into(B, K, V, target_logits, draft_logits, draft_tokens, draft_len, uniforms, sampling,
                           accepted_len, next_token, out_ids, out_probs, seq_status, scratch,
                           sv::NOALLOC_SCRATCH_BYTES, static_cast<cudaStream_t>(stream));
}
