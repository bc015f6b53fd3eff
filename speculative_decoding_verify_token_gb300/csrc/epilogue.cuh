// GEMM epilogues of the decoder layers, shared by the SIMT and the tcgen05 GEMMs.
//
// A GEMM computes acc[m][n] = sum_k X[m][k] W[n][k]; the epilogue consumes the two
// outputs of a row pair (n0, n1) of one token m:
//  * EPI_QKV    : the pair is (j, j + hd/2) of one head of the stacked [q; k; v] rows;
//                 rotate-half RoPE at the token's absolute position for q and k, then q
//                 goes to the Q buffer and k, v into the token's paged-KV slot;
//  * EPI_SWIGLU : the pair is (gate f, up f) -> H[m][f] = silu(gate) * up;
//  * EPI_RESID  : the pair is (2p, 2p + 1) -> X[m][n] += acc (fp32 residual stream);
//  * EPI_STORE  : the pair is (2p, 2p + 1) -> out[m][n] = acc (fp32 logits).
//
// Split activations (tensor-core path): a bf16 GEMM input x is stored as two bf16 halves,
// hi = bf16(x) and lo = bf16(x - hi), lo_off elements apart, and the GEMM accumulates
// W hi + W lo (about 16 significant bits of x instead of 8); the queries are split the same
// way for the attention.  lo_off = 0 stores hi only.
//
// Operand layout of the tensor-core GEMM inputs (act_off): a pass of M tokens is padded to
// Mp = act_rows(M) rows (8 up to 8 tokens, else a multiple of 16); per 64-column K atom the
// Mp hi rows, then the Mp lo rows, of
// 128 bytes each, every row's eight 16-byte chunks in the 128-byte swizzled order the
// tensor cores read (chunk j of row m at position j ^ (m % 8)).  The rows of one atom are
// then one contiguous run of global memory that lands in shared memory, by one bulk copy,
// exactly as the MMA descriptor expects, and the lo half of an element is Mp * 64 elements
// after its hi half.
//
// Fused RMSNorm (tensor-core GEMM only): RMSNorm(x) W^T = (x * g) W^T / rms(x), so a
// residual epilogue that also writes xg = bf16(x_new * g_next) and, per 128-column tile
// of x, the sum of x_new^2 lets the GEMM that consumes the normed row apply 1/rms(x) to
// its accumulators; no separate normalisation kernel runs.
#pragma once

#include <cuda_bf16.h>
#include <cstdint>

namespace sv {

enum EpiKind { EPI_QKV = 0, EPI_SWIGLU = 1, EPI_RESID = 2, EPI_STORE = 3 };

// Order-preserving 64-bit key of logit v at vocabulary id: the larger key is the larger
// value, and of equal values the lower id (the greedy argmax's tie order); -0 counts as +0.
__device__ __forceinline__ unsigned long long amax_key(float v, int id) {
    uint32_t u = v == 0.0f ? 0u : __float_as_uint(v);
    u = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
    return ((unsigned long long)u << 32) | (unsigned long long)(0xFFFFFFFFu - (uint32_t)id);
}

// Rows of the tensor-core operand layout for a pass (or a GEMM launch) of M tokens: a
// multiple of 8, so that a row's swizzle phase (row % 8) is the same counted from the start
// of the hi block, of the lo block or of any launch's first row.
__host__ __device__ __forceinline__ int act_rows(int M) { return M <= 8 ? 8 : (M + 15) & ~15; }

// Element offset of dimension d of key r (0..15) of KV page `page`, kv head h, in one
// layer's K (or V) pool: row-major [page][hkv][16][hd] when sw = 0; for the tensor-core
// attention (hd = 128) [hkv][2 halves of 64 dims][num_pages][16][64], every 128-byte key
// row of a half in the swizzled order the MMA reads (16-byte chunk j at j ^ (r % 8)), so
// that the keys of consecutive pages of one head and half are one contiguous run.
__host__ __device__ __forceinline__ size_t kv_off(int page, int h, int r, int d, int hkv, int hd, int num_pages,
                                                  int sw) {
    if (sw == 0) return (((size_t)page * hkv + h) * 16 + r) * hd + d;
    return ((((size_t)h * 2 + (d >> 6)) * num_pages + page) * 16 + r) * 64 +
           (size_t)(((((d & 63) >> 3) ^ (r & 7)) << 3) | (d & 7));
}

// Element offset of dimension d of query row r (r = t * G + hh: token t, query head hh of
// the group) of (sequence b, kv head g) in the tensor-core attention's query layout: per
// (b, g) the hi rows then the lo rows, each as two 64-dim halves of np rows of 128 bytes
// (swizzled as above); the lo half of a value is 2 * np * 64 elements after its hi half.
__host__ __device__ __forceinline__ size_t q_att_off(int b, int g, int r, int d, int hkv, int np) {
    return ((((size_t)b * hkv + g) * 4 + (d >> 6)) * np + r) * 64 + (size_t)(((((d & 63) >> 3) ^ (r & 7)) << 3) | (d & 7));
}

// Element offset of row m, column n of an activation with ld columns: row-major when
// sw_rows = 0, else the tensor-core operand layout of a pass padded to sw_rows rows.
__host__ __device__ __forceinline__ size_t act_off(int m, int n, int ld, int sw_rows) {
    if (sw_rows == 0) return (size_t)m * ld + n;
    return ((size_t)(n >> 6) * 2 * sw_rows + m) * 64 + (size_t)(((((n >> 3) & 7) ^ (m & 7)) << 3) | (n & 7));
}

struct EpiArgs {
    int kind;
    int M;
    // QKV
    void* q_out;                // [M][hq*hd], or the attention's query layout (q_np > 0)
    void* k_layer;              // this layer's K pool (kv_off layout)
    void* v_layer;
    int kv_sw, num_pages;       // KV pool layout (kv_off)
    int q_np, q_T;              // q_np > 0: queries in q_att_off layout of q_np rows, q_T tokens per sequence
    const int* block_table;     // [slots][max_pages]
    int max_pages;
    const int* tok_seq;         // [M] slot of token m
    const int* tok_pos;         // [M] absolute position of token m
    const float2* rope;         // [max_pos][hd/2] (cos, sin)
    int hq, hkv, hd;
    // SWIGLU
    void* h_out;                // [M][F] at act_off(m, f, F, sw_rows)
    int F;
    int sw_rows;                // layout of h_out and xg_out (act_off); 0 = row-major
    // RESID / STORE
    float* x;                   // [M][ldx]
    int ldx;
    int keep_last;              // STORE: 0 = every row; 1 = only the launch's last row, to row 0
    // STORE, tensor-core path: instead of the logits, per token m and 128-row tile t the key
    // of the tile's largest logit at amax_out[m * amax_ld + t] (see amax_key); nullptr = store
    unsigned long long* amax_out;
    int amax_ld;
    size_t lo_off;              // split activations: elements from a hi value to its lo half
    int m0;                     // token offset of this launch (rows m0 .. m0 + M - 1)
    // fused RMSNorm, producer side (RESID): xg_out = bf16(x_new * g_next), ssq_out[t][m] =
    // sum of x_new[m][n]^2 over the 128 columns n of tile t (fixed order)
    void* xg_out;               // [M][ldx] bf16 at act_off(m, n, ldx, sw_rows), or nullptr
    const void* g_next;         // [ldx] bf16
    float* ssq_out;             // [ldx / 128][ssq_ld]
    // consumer side: accumulators of token m are scaled by 1/sqrt(sum_t ssq_in[t][row0 + m]
    // / norm_d + eps), the tiles summed in order
    const float* ssq_in;        // [n_ssq][ssq_ld] or nullptr
    int n_ssq, ssq_ld, ssq_row0;
    float norm_d, eps;
};

template <typename T> __device__ __forceinline__ T from_f32(float v);
template <> __device__ __forceinline__ float from_f32<float>(float v) { return v; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float v) { return __float2bfloat16_rn(v); }

template <typename T> __device__ __forceinline__ float to_f32(T v);
template <> __device__ __forceinline__ float to_f32<float>(float v) { return v; }
template <> __device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 v) { return __bfloat162float(v); }

__device__ __forceinline__ float silu_f(float g) { return g / (1.0f + expf(-g)); }

// Store v at p, and its bf16 remainder at p + lo_off when lo_off != 0 (bf16 only).
template <typename T> __device__ __forceinline__ void store_split(T* p, size_t lo_off, float v);
template <> __device__ __forceinline__ void store_split<float>(float* p, size_t, float v) { *p = v; }
template <>
__device__ __forceinline__ void store_split<__nv_bfloat16>(__nv_bfloat16* p, size_t lo_off, float v) {
    const __nv_bfloat16 h = __float2bfloat16_rn(v);
    *p = h;
    if (lo_off) p[lo_off] = __float2bfloat16_rn(v - __bfloat162float(h));
}

// Row pair of pair index p for the QKV layout: head slot hs in [0, hq + 2 hkv), j < hd/2.
__device__ __forceinline__ void qkv_pair_rows(int p, int hd, int& hs, int& j) {
    const int half = hd >> 1;
    hs = p / half;
    j = p - hs * half;
}

// QKV epilogue of one token m (pass-wide index) and one rotate-half pair (j, j + hd/2) of
// head row hs: RoPE with (cos, sin) = cs for q and k heads, then the query store (hi/lo
// split) or the K/V append at position pos of KV page `page`.
template <typename T>
__device__ __forceinline__ void qkv_store(const EpiArgs& e, int m, int hs, int j, int pos, float2 cs, int page,
                                          float a0, float a1) {
    const int half = e.hd >> 1;
    if (hs < e.hq + e.hkv) {
        const float r0 = a0 * cs.x - a1 * cs.y;
        const float r1 = a1 * cs.x + a0 * cs.y;
        a0 = r0; a1 = r1;
    }
    if (hs < e.hq) {
        if (e.q_np > 0) {
            const int G = e.hq / e.hkv;
            const int b = m / e.q_T, t = m - b * e.q_T, g = hs / G, r = t * G + (hs - g * G);
            T* q = static_cast<T*>(e.q_out);
            const size_t lo = (size_t)2 * e.q_np * 64;
            store_split<T>(q + q_att_off(b, g, r, j, e.hkv, e.q_np), lo, a0);
            store_split<T>(q + q_att_off(b, g, r, j + half, e.hkv, e.q_np), lo, a1);
        } else {
            T* q = static_cast<T*>(e.q_out) + (size_t)m * e.hq * e.hd + (size_t)hs * e.hd;
            store_split<T>(q + j, e.lo_off, a0);
            store_split<T>(q + j + half, e.lo_off, a1);
        }
    } else {
        const bool is_k = hs < e.hq + e.hkv;
        const int kvh = is_k ? hs - e.hq : hs - e.hq - e.hkv;
        T* base = static_cast<T*>(is_k ? e.k_layer : e.v_layer);
        const int r = pos & 15;
        base[kv_off(page, kvh, r, j, e.hkv, e.hd, e.num_pages, e.kv_sw)] = from_f32<T>(a0);
        base[kv_off(page, kvh, r, j + half, e.hkv, e.hd, e.num_pages, e.kv_sw)] = from_f32<T>(a1);
    }
}

template <typename T>
__device__ __forceinline__ void epi_pair(const EpiArgs& e, int m_local, int p, float a0, float a1) {
    const int m = m_local + e.m0;
    switch (e.kind) {
    case EPI_QKV: {
        int hs, j;
        qkv_pair_rows(p, e.hd, hs, j);
        const int pos = e.tok_pos[m];
        const float2 cs = hs < e.hq + e.hkv ? e.rope[(size_t)pos * (e.hd >> 1) + j] : make_float2(1.0f, 0.0f);
        const int page = hs >= e.hq ? e.block_table[(size_t)e.tok_seq[m] * e.max_pages + (pos >> 4)] : 0;
        qkv_store<T>(e, m, hs, j, pos, cs, page, a0, a1);
        break;
    }
    case EPI_SWIGLU:
        store_split<T>(static_cast<T*>(e.h_out) + act_off(m, p, e.F, e.sw_rows), e.lo_off, silu_f(a0) * a1);
        break;
    case EPI_RESID: {
        float* x = e.x + (size_t)m * e.ldx + 2 * p;
        x[0] += a0;
        x[1] += a1;
        break;
    }
    default: {
        if (e.keep_last && m_local != e.M - 1) break;
        float* x = e.x + (size_t)(e.keep_last ? 0 : m) * e.ldx + 2 * p;
        x[0] = a0;
        x[1] = a1;
        break;
    }
    }
}

}  // namespace sv
