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
// GB300 design:
//  * persistent grid of 3 CTAs x 8 warps per SM; every warp streams one (row, chunk) work
//    item at a time with coalesced 16-byte streaming loads, 8 in flight per lane (about
//    100 KB of HBM reads in flight per SM), handed out by a global atomic counter so the
//    warps stay balanced whatever B, K and V are (the index of the next item is fetched
//    one item ahead);
//  * each warp keeps an exact running top-k of its item as a warp-wide sorted list (one
//    entry per lane); the common path per 1024 elements is a lane maximum and one vote
//    against the running cut, which is the larger of the list's k-th value and a lower
//    bound of the row's k-th value shared by all chunks of the row (atomicMax on an
//    order-preserving integer key); the rare candidates go to a shared-memory buffer and
//    through a bitonic sort + merge 32 at a time;
//  * the last warp to finish a row (atomic arrival count, no spin-wait) merges the chunk
//    lists and builds the row's truncated distribution; the last row of a sequence runs
//    the acceptance scan and the final inverse-CDF draw on one warp.
#include <cstdio>
#include <cstring>
#include <cmath>
#include <algorithm>
#include <mutex>

#include "common.cuh"
#include "host_util.h"

namespace sv {

constexpr int VT_WARPS = 8;
constexpr int VT_THREADS = VT_WARPS * 32;
constexpr int VT_BLOCKS_PER_SM = 2;
constexpr int VS_UNROLL = 8;                         // 16-byte loads per lane per iteration (x2 in flight)
constexpr int VT_CHUNK_QUANTUM = 1024;               // chunk sizes are multiples of this
constexpr int LISTN = 32;
constexpr int VT_TARGET_ITEMS = 4096;
constexpr int VT_MAX_CHUNKS = 128;
constexpr int VT_MAX_K = 64;
// per-warp candidate buffer: a flush leaves < 32 entries and one iteration adds at most
// 32 * 4 * VS_UNROLL, so it never overflows
constexpr int VT_CAND_CAP = 32 + 32 * 4 * 8;

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
    int chunks;                 // chunks per row
    int chunk_elems;            // body elements per chunk (multiple of VT_CHUNK_QUANTUM)
    int n_items;                // n_rows * chunks
    int* accepted_len;
    int* next_token;
    int* out_ids;
    float* out_probs;
    int* seq_status;
    int* out_tokens;
    // workspace
    int* work;                  // [1] item counter
    int* row_cnt;               // [n_rows]
    int* seq_cnt;               // [B]
    unsigned* row_bound;        // [n_rows] order-preserving key of a lower bound of the row's k-th best
    float* cl_v;                // [n_rows][chunks][LISTN]
    int* cl_id;
    int* rd_n;                  // [n_rows]
    int* rd_id;                 // [n_rows][LISTN]
    float* rd_p;
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

// One round: every lane offers at most one candidate; sort them and merge into the list.
__device__ __forceinline__ void offer_round(float& lv, int& lid, bool has, float cv, int cid, int lane) {
    if (!has) { cv = -INFINITY; cid = SENT_ID; }
    warp_sort_desc(cv, cid, lane);
    warp_merge_desc(lv, lid, cv, cid, lane);
}

// Order-preserving map of floats to unsigned ints (for atomicMax); 0 means "no bound".
__device__ __forceinline__ unsigned float_key(float f) {
    const unsigned b = __float_as_uint(f);
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
__device__ __forceinline__ float key_float(unsigned k) {
    if (k == 0u) return -INFINITY;
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

// Sort + merge the warp's buffered candidates into its running list, 32 at a time.
__device__ __forceinline__ void flush_candidates(float& lv, int& lid, const float* cv, const int* ci, int n,
                                                 int lane) {
    __syncwarp();
    for (int base = 0; base < n; base += 32) {
        const bool has = base + lane < n;
        float v = has ? cv[base + lane] : -INFINITY;
        int id = has ? ci[base + lane] : SENT_ID;
        warp_sort_desc(v, id, lane);
        warp_merge_desc(lv, lid, v, id, lane);
    }
    __syncwarp();
}

// Truncated distribution of a merged row list (lane j = j-th best), written to rd_*.
__device__ void build_row_dist(const VerifyParams& p, int row, float lv, int lid, int lane) {
    const int k = p.top_k;
    int n;
    int oid;
    float op;
    if (p.temperature == 0.0f) {
        n = 1;
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
        n = __popc(__ballot_sync(FULL, kept));
        const float S2 = warp_sum(kept ? e : 0.0f);
        oid = kept ? lid : -1;
        op = kept ? e / S2 : 0.0f;
    }
    p.rd_id[(size_t)row * LISTN + lane] = oid;
    p.rd_p[(size_t)row * LISTN + lane] = op;
    if (lane == 0) p.rd_n[row] = n;
}

// Inverse CDF over ascending token id: (key, w) per lane, key = SENT_ID for empty lanes.
// Returns the chosen token; sorts (key, w) ascending in place.
__device__ int inverse_cdf_draw(int& key, float& w, float u, int lane, float& Z) {
    warp_sort_asc_key(key, w, lane);
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
    int src;
    if (sel) src = __ffs(sel) - 1;
    else src = valid ? 31 - __clz(valid) : 0;
    return __shfl_sync(FULL, key, src);
}

__device__ __forceinline__ int trow(const VerifyParams& p, int b, int i) { return b * (p.K + 1) + i; }
__device__ __forceinline__ int drow(const VerifyParams& p, int b, int i) { return p.n_target_rows + b * p.K + i; }

// Acceptance scan of one sequence on one warp.
__device__ void finish_sequence(const VerifyParams& p, int b, int lane) {
    const int kb = draft_count(p, b);
    const float* ub = p.u + (size_t)b * (p.K + 1);
    int a = 0, next = -1, status = SPEC_OK;
    int okey = SENT_ID;
    float ow = 0.0f, oZ = 1.0f;
    if (p.temperature == 0.0f) {
        while (a < kb && p.draft_tokens[(size_t)b * p.K + a] == __ldcg(p.rd_id + (size_t)trow(p, b, a) * LISTN)) ++a;
        next = __ldcg(p.rd_id + (size_t)trow(p, b, a) * LISTN);
        okey = lane == 0 ? next : SENT_ID;
        ow = lane == 0 ? 1.0f : 0.0f;
    } else {
        const bool has_q = p.draft != nullptr;
        bool reject = false;
        a = kb;
        int d = -1;
        for (int i = 0; i < kb; ++i) {
            d = p.draft_tokens[(size_t)b * p.K + i];
            const int pid = __ldcg(p.rd_id + (size_t)trow(p, b, i) * LISTN + lane);
            const float pp = __ldcg(p.rd_p + (size_t)trow(p, b, i) * LISTN + lane);
            const float pd = warp_max(pid == d ? pp : 0.0f);
            float qd = 1.0f;
            if (has_q) {
                const int qid = __ldcg(p.rd_id + (size_t)drow(p, b, i) * LISTN + lane);
                const float qp = __ldcg(p.rd_p + (size_t)drow(p, b, i) * LISTN + lane);
                qd = warp_max(qid == d ? qp : 0.0f);
            }
            if (qd == 0.0f) { status = SPEC_E_DRAFT; a = i; break; }
            const float ratio = pd / qd;
            if (!(ub[i] < ratio)) { a = i; reject = true; break; }
        }
        if (status == SPEC_OK) {
            const int prow = trow(p, b, a);
            const int pid = __ldcg(p.rd_id + (size_t)prow * LISTN + lane);
            const float pp = __ldcg(p.rd_p + (size_t)prow * LISTN + lane);
            float w = pid >= 0 ? pp : 0.0f;
            if (reject) {
                float qx = 0.0f;
                if (has_q) {
                    const int qid = __ldcg(p.rd_id + (size_t)drow(p, b, a) * LISTN + lane);
                    const float qp = __ldcg(p.rd_p + (size_t)drow(p, b, a) * LISTN + lane);
                    for (int t = 0; t < LISTN; ++t) {
                        const int tid = __shfl_sync(FULL, qid, t);
                        const float tp = __shfl_sync(FULL, qp, t);
                        if (tid >= 0 && tid == pid) qx = tp;
                    }
                } else {
                    qx = (pid == d) ? 1.0f : 0.0f;
                }
                float r = pid >= 0 ? fmaxf(pp - qx, 0.0f) : 0.0f;
                if (warp_sum(r) == 0.0f) r = w;      // residual empty: fall back to P
                w = r;
            }
            okey = (pid >= 0 && w > 0.0f) ? pid : SENT_ID;
            ow = okey != SENT_ID ? w : 0.0f;
            next = inverse_cdf_draw(okey, ow, ub[p.K], lane, oZ);
        }
    }
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

// The last chunk of a row: merge the chunk lists, build the distribution, then either
// sample (sample mode) or arrive on the sequence.
__device__ void finish_row(const VerifyParams& p, int row, int lane) {
    float lv = -INFINITY;
    int lid = SENT_ID;
    const size_t base = (size_t)row * p.chunks * LISTN;
    constexpr int BATCH = 8;
    for (int c0 = 0; c0 < p.chunks; c0 += BATCH) {
        float bv[BATCH];
        int bi[BATCH];
#pragma unroll
        for (int j = 0; j < BATCH; ++j) {
            const int c = c0 + j;
            if (c < p.chunks) {
                bv[j] = __ldcg(p.cl_v + base + (size_t)c * LISTN + lane);
                bi[j] = __ldcg(p.cl_id + base + (size_t)c * LISTN + lane);
            } else {
                bv[j] = -INFINITY; bi[j] = SENT_ID;
            }
        }
#pragma unroll
        for (int j = 0; j < BATCH; ++j)
            if (c0 + j < p.chunks) warp_merge_desc(lv, lid, bv[j], bi[j], lane);
    }
    build_row_dist(p, row, lv, lid, lane);

    if (p.mode == MODE_SAMPLE) {
        int key = __ldcg(p.rd_id + (size_t)row * LISTN + lane);
        float w = __ldcg(p.rd_p + (size_t)row * LISTN + lane);
        if (key < 0) { key = SENT_ID; w = 0.0f; }
        float Z;
        const int tok = inverse_cdf_draw(key, w, p.u[row], lane, Z);
        if (lane == 0) p.out_tokens[row] = tok;
        return;
    }
    const RowInfo ri = row_info(p, row);
    const int b = ri.seq;
    const int kb = draft_count(p, b);
    const int expected = (kb + 1) + (p.draft != nullptr && p.temperature != 0.0f ? kb : 0);
    __threadfence();
    __syncwarp();
    int prev = 0;
    if (lane == 0) prev = atomicAdd(p.seq_cnt + b, 1);
    prev = __shfl_sync(FULL, prev, 0);
    if (prev == expected - 1) {
        __threadfence();
        finish_sequence(p, b, lane);
    }
}


// One warp streams one (row, chunk) work item at a time: coalesced 16-byte streaming loads,
// two register tiles of VS_UNROLL float4 per lane so that the next 4 KB of the row is in
// flight while the current 4 KB is examined, 2 CTAs of 8 warps per SM.  Per 1024 elements
// the common path is a lane maximum (per float4 first) and one vote against the running
// cut; only the float4s whose maximum reaches the cut are looked at element by element.
struct TopkState {
    float lv, lb, published;
    int lid, ccount;
};

__device__ __forceinline__ void examine_tile(const VerifyParams& p, const float4 (&x)[VS_UNROLL], int i0, int s0,
                                             bool first, unsigned rb_key, unsigned* rb_ptr, TopkState& st,
                                             float* cbuf_v, int* cbuf_id, int* ccnt, int lane) {
    const int k = p.top_k;
    float mu[VS_UNROLL];
#pragma unroll
    for (int u = 0; u < VS_UNROLL; ++u) mu[u] = fmaxf(fmaxf(x[u].x, x[u].y), fmaxf(x[u].z, x[u].w));
    float mx = mu[0];
#pragma unroll
    for (int u = 1; u < VS_UNROLL; ++u) mx = fmaxf(mx, mu[u]);
    if (first) {
        // k distinct elements reach the k-th largest lane maximum: a lower bound of the
        // chunk's (and the row's) k-th best.
        float m = mx;
        int dummy = lane;
        warp_sort_desc(m, dummy, lane);
        st.lb = __shfl_sync(FULL, m, k - 1);
        if (lane == 0 && st.lb > -INFINITY) atomicMax(rb_ptr, float_key(st.lb));
        st.published = st.lb;
    }
    st.lb = fmaxf(st.lb, key_float(rb_key));
    const float cut = fmaxf(st.lb, __shfl_sync(FULL, st.lv, k - 1));
    if (__any_sync(FULL, mx >= cut)) {
        // value test only: an entry equal to the k-th value with a larger id is a harmless
        // extra for the exact merge
        if (mx >= cut) {
#pragma unroll
            for (int u = 0; u < VS_UNROLL; ++u) {
                if (mu[u] >= cut) {
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const float xc = pick4(x[u], q);
                        if (xc >= cut) {
                            const int pos = atomicAdd(ccnt, 1);
                            cbuf_v[pos] = xc;
                            cbuf_id[pos] = s0 + 4 * (i0 + lane + 32 * u) + q;
                        }
                    }
                }
            }
        }
        __syncwarp();
        st.ccount = *reinterpret_cast<volatile int*>(ccnt);
    }
    if (st.ccount >= 32 || (st.ccount > 0 && __shfl_sync(FULL, st.lid, k - 1) == SENT_ID)) {
        flush_candidates(st.lv, st.lid, cbuf_v, cbuf_id, st.ccount, lane);
        st.ccount = 0;
        if (lane == 0) *ccnt = 0;
        __syncwarp();
    }
    const float kth = __shfl_sync(FULL, st.lv, k - 1);
    if (kth > st.published) {
        if (lane == 0) atomicMax(rb_ptr, float_key(kth));
        st.published = kth;
        st.lb = fmaxf(st.lb, kth);
    }
}

__device__ __forceinline__ void load_tile(float4 (&x)[VS_UNROLL], const float4* src, int i0, int n4, int lane) {
#pragma unroll
    for (int u = 0; u < VS_UNROLL; ++u) {
        const int idx = i0 + lane + 32 * u;
        x[u] = idx < n4 ? __ldcs(src + idx) : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
    }
}

__global__ void __launch_bounds__(VT_THREADS, VT_BLOCKS_PER_SM) verify_kernel(const VerifyParams p) {
    __shared__ float cand_v[VT_WARPS][VT_CAND_CAP];
    __shared__ int cand_id[VT_WARPS][VT_CAND_CAP];
    __shared__ int ccnt_s[VT_WARPS];

    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    float* cbuf_v = cand_v[warp];
    int* cbuf_id = cand_id[warp];
    int* ccnt = &ccnt_s[warp];
    if (lane == 0) *ccnt = 0;
    __syncwarp();
    int pref = 0;
    if (lane == 0) pref = atomicAdd(p.work, 1);
    constexpr int STEP = 32 * VS_UNROLL;

    while (true) {
        // next needed work item (the index after it is fetched now and used next time)
        int it = 0;
        if (lane == 0) {
            it = pref;
            while (it < p.n_items && !row_needed(p, row_info(p, it / p.chunks))) it = atomicAdd(p.work, 1);
            if (it < p.n_items) pref = atomicAdd(p.work, 1);
        }
        it = __shfl_sync(FULL, it, 0);
        if (it >= p.n_items) break;
        const int row = it / p.chunks, c = it % p.chunks;
        const RowInfo ri = row_info(p, row);
        int head, body;
        row_split(ri.ptr, p.V, head, body);
        const int s0 = head + min(c * p.chunk_elems, body);
        const int s1 = head + min(body, (c + 1) * p.chunk_elems);
        const float4* src = reinterpret_cast<const float4*>(ri.ptr + s0);
        const int n4 = s1 > s0 ? (s1 - s0) >> 2 : 0;
        unsigned* rb_ptr = p.row_bound + row;

        TopkState st;
        st.lv = -INFINITY; st.lb = -INFINITY; st.published = -INFINITY; st.lid = SENT_ID; st.ccount = 0;
        float4 xa[VS_UNROLL], xb[VS_UNROLL];
        if (n4 > 0) load_tile(xa, src, 0, n4, lane);
        for (int i0 = 0; i0 < n4; i0 += 2 * STEP) {
            unsigned rb_key = *reinterpret_cast<volatile unsigned*>(rb_ptr);
            if (i0 + STEP < n4) load_tile(xb, src, i0 + STEP, n4, lane);
            examine_tile(p, xa, i0, s0, i0 == 0, rb_key, rb_ptr, st, cbuf_v, cbuf_id, ccnt, lane);
            if (i0 + STEP >= n4) break;
            rb_key = *reinterpret_cast<volatile unsigned*>(rb_ptr);
            if (i0 + 2 * STEP < n4) load_tile(xa, src, i0 + 2 * STEP, n4, lane);
            examine_tile(p, xb, i0 + STEP, s0, false, rb_key, rb_ptr, st, cbuf_v, cbuf_id, ccnt, lane);
        }
        float lv = st.lv;
        int lid = st.lid;
        if (st.ccount > 0) {
            flush_candidates(lv, lid, cbuf_v, cbuf_id, st.ccount, lane);
            if (lane == 0) *ccnt = 0;
            __syncwarp();
        }
        // scalar head / tail of the row
        const int tail0 = head + body, tail = p.V - tail0;
        if (c == 0 && head > 0) {
            const bool has = lane < head;
            offer_round(lv, lid, has, has ? ri.ptr[lane] : 0.0f, lane, lane);
        }
        if (c == p.chunks - 1 && tail > 0) {
            const bool has = lane < tail;
            offer_round(lv, lid, has, has ? ri.ptr[tail0 + lane] : 0.0f, tail0 + lane, lane);
        }
        // publish the chunk list; the last chunk of the row finishes it
        const size_t o = ((size_t)row * p.chunks + c) * LISTN + lane;
        p.cl_v[o] = lv;
        p.cl_id[o] = lid;
        __threadfence();
        __syncwarp();
        int prev = 0;
        if (lane == 0) prev = atomicAdd(p.row_cnt + row, 1);
        prev = __shfl_sync(FULL, prev, 0);
        if (prev == p.chunks - 1) {
            __threadfence();
            finish_row(p, row, lane);
        }
    }
}

// ---- host side ---------------------------------------------------------------------------

struct Plan {
    int n_rows, chunks, chunk_elems;
    size_t off_work, off_row, off_seq, off_rb, off_clv, off_clid, off_rdn, off_rdid, off_rdp, total, counters_bytes;
};

static inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

static Plan make_plan(int n_rows_max, int n_seq, int V) {
    Plan pl{};
    pl.n_rows = n_rows_max;
    const int per_row = std::max(1, (VT_TARGET_ITEMS + n_rows_max - 1) / n_rows_max);
    long long ch = ((long long)V + per_row - 1) / per_row;
    ch = ((ch + VT_CHUNK_QUANTUM - 1) / VT_CHUNK_QUANTUM) * VT_CHUNK_QUANTUM;
    if (ch < VT_CHUNK_QUANTUM) ch = VT_CHUNK_QUANTUM;
    long long chunks = ((long long)V + ch - 1) / ch;
    if (chunks > VT_MAX_CHUNKS) {
        chunks = VT_MAX_CHUNKS;
        ch = (((long long)V + chunks - 1) / chunks + VT_CHUNK_QUANTUM - 1) / VT_CHUNK_QUANTUM * VT_CHUNK_QUANTUM;
        chunks = ((long long)V + ch - 1) / ch;
    }
    pl.chunks = (int)chunks;
    pl.chunk_elems = (int)ch;
    size_t o = 0;
    pl.off_work = o; o += 4;
    pl.off_row = o; o += (size_t)n_rows_max * 4;
    pl.off_seq = o; o += (size_t)n_seq * 4;
    pl.off_rb = o; o += (size_t)n_rows_max * 4;
    pl.counters_bytes = o;
    o = align256(o);
    const size_t lists = (size_t)n_rows_max * pl.chunks * LISTN;
    pl.off_clv = o; o = align256(o + lists * 4);
    pl.off_clid = o; o = align256(o + lists * 4);
    pl.off_rdn = o; o = align256(o + (size_t)n_rows_max * 4);
    pl.off_rdid = o; o = align256(o + (size_t)n_rows_max * LISTN * 4);
    pl.off_rdp = o; o = align256(o + (size_t)n_rows_max * LISTN * 4);
    pl.total = o;
    return pl;
}

static int sm_count() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return -1;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return -1;
    return n;
}

static int launch_verify(VerifyParams& prm, const Plan& pl, void* ws, cudaStream_t st) {
    uint8_t* w = static_cast<uint8_t*>(ws);
    prm.work = reinterpret_cast<int*>(w + pl.off_work);
    prm.row_cnt = reinterpret_cast<int*>(w + pl.off_row);
    prm.seq_cnt = reinterpret_cast<int*>(w + pl.off_seq);
    prm.row_bound = reinterpret_cast<unsigned*>(w + pl.off_rb);
    prm.cl_v = reinterpret_cast<float*>(w + pl.off_clv);
    prm.cl_id = reinterpret_cast<int*>(w + pl.off_clid);
    prm.rd_n = reinterpret_cast<int*>(w + pl.off_rdn);
    prm.rd_id = reinterpret_cast<int*>(w + pl.off_rdid);
    prm.rd_p = reinterpret_cast<float*>(w + pl.off_rdp);
    prm.chunks = pl.chunks;
    prm.chunk_elems = pl.chunk_elems;
    prm.n_items = prm.n_rows * pl.chunks;

    cudaError_t e = cudaMemsetAsync(ws, 0, pl.counters_bytes, st);
    if (e != cudaSuccess) return set_error(SPEC_E_CUDA, "cudaMemsetAsync: %s", cudaGetErrorString(e));
    const int nsm = sm_count();
    if (nsm <= 0) return set_error(SPEC_E_CUDA, "no CUDA device");
    const int grid = std::max(1, std::min(nsm * VT_BLOCKS_PER_SM, (prm.n_items + VT_WARPS - 1) / VT_WARPS));
    verify_kernel<<<grid, VT_THREADS, 0, st>>>(prm);
    e = cudaGetLastError();
    if (e != cudaSuccess) return set_error(SPEC_E_CUDA, "verify_kernel launch: %s", cudaGetErrorString(e));
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


// Validation + launch of the fused verify (used by spec_verify_logits and spec_verify).
int verify_into(int B, int K, int V, const float* target_logits, const float* draft_logits,
                const int32_t* draft_tokens, const int32_t* draft_len, const float* uniforms,
                const spec_sampling* sampling, int32_t* accepted_len, int32_t* next_token, int32_t* out_ids,
                float* out_probs, int32_t* seq_status, void* workspace, size_t workspace_bytes, cudaStream_t st) {
    if (B < 1 || K < 0 || V < 2) return set_error(SPEC_E_INVAL, "bad sizes B=%d K=%d V=%d", B, K, V);
    if (K > VT_MAX_K) return set_error(SPEC_E_INVAL, "K=%d above the maximum %d", K, VT_MAX_K);
    if ((long long)B * (2 * K + 1) * (long long)V >= (1LL << 40))
        return set_error(SPEC_E_RANGE, "logits too large");
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
    const Plan pl = make_plan(B * (2 * K + 1), B, V);
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

using namespace sv;

extern "C" size_t spec_verify_logits_workspace_bytes(int B, int K, int V) {
    if (B < 1 || K < 0 || V < 2 || K > VT_MAX_K) return 0;
    return make_plan(B * (2 * K + 1), B, V).total;
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
    return make_plan(R, R, V).total;
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
    const Plan pl = make_plan(R, R, V);
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
    if (need == 0) return set_error(SPEC_E_INVAL, "bad sizes B=%d K=%d V=%d", B, K, V);
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
