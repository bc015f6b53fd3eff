// Small kernels of the decoder pass: embedding gather (with per-token slot/position),
// RMSNorm, the RoPE table, the verify-pass token layout and the O(1) KV length updates.
#include <cuda_bf16.h>

#include "common.cuh"
#include "epilogue.cuh"
#include "model.h"

namespace sv {

// 4 consecutive elements of T as floats / stored from floats.
template <typename T> struct Quad;
template <> struct Quad<float> {
    __device__ __forceinline__ static float4 load(const float* p) { return *reinterpret_cast<const float4*>(p); }
    __device__ __forceinline__ static void store(float* p, float4 v) { *reinterpret_cast<float4*>(p) = v; }
};
template <> struct Quad<__nv_bfloat16> {
    __device__ __forceinline__ static float4 load(const __nv_bfloat16* p) {
        const uint2 u = *reinterpret_cast<const uint2*>(p);
        return make_float4(__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xffff0000u), __uint_as_float(u.y << 16),
                           __uint_as_float(u.y & 0xffff0000u));
    }
    __device__ __forceinline__ static void store(__nv_bfloat16* p, float4 v) {
        __nv_bfloat162 a = __floats2bfloat162_rn(v.x, v.y), b = __floats2bfloat162_rn(v.z, v.w);
        uint2 u;
        u.x = *reinterpret_cast<uint32_t*>(&a);
        u.y = *reinterpret_cast<uint32_t*>(&b);
        *reinterpret_cast<uint2*>(p) = u;
    }
};


// X[m][:] = E[tok[m]][:] in fp32; token m = b*T + t belongs to slot seq_ids[b] at
// position seq_len[slot] + t.  Ids outside [0, V) are embedded as token 0.  The token id
// (as given) is also recorded at tok_log[slot][position]: the slot's context for the
// on-device n-gram drafter.  With Xg set
// (fused RMSNorm of the tensor-core path) it also writes Xg[m] = bf16(X[m] * g), in the
// GEMM operand layout act_off(m, n, d, sw_rows), and, per 128-column tile t, ssq[t][m] =
// sum of X[m][n]^2 over the tile (one warp per tile).
template <typename T>
__global__ void embed_kernel(const int* __restrict__ tokens, const int* __restrict__ seq_ids,
                             const int* __restrict__ seq_len, int T_per_seq, const T* __restrict__ E,
                             float* __restrict__ X, int* __restrict__ tok_seq, int* __restrict__ tok_pos, int d,
                             int V, T* __restrict__ Xg, const T* __restrict__ g, float* __restrict__ ssq,
                             int ssq_ld, size_t lo_off, int sw_rows, int* __restrict__ tok_log, int max_ctx) {
    pdl_launch_dependents();
    const int m = blockIdx.x;
    const int b = m / T_per_seq;
    const int t = m - b * T_per_seq;
    const int raw = tokens[m];
    const int tok = (raw < 0 || raw >= V) ? 0 : raw;
    if (threadIdx.x == 0) {
        const int slot = seq_ids[b];
        const int pos = seq_len[slot] + t;
        tok_seq[m] = slot;
        tok_pos[m] = pos;
        if (pos < max_ctx) tok_log[(size_t)slot * max_ctx + pos] = raw;
    }
    const T* row = E + (size_t)tok * d;
    float* xr = X + (size_t)m * d;
    if (Xg == nullptr) {
        for (int i = threadIdx.x; i < (d >> 2); i += blockDim.x)
            reinterpret_cast<float4*>(xr)[i] = Quad<T>::load(row + 4 * i);
        return;
    }
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int tile = warp; tile < (d >> 7); tile += blockDim.x >> 5) {
        const int c = tile * 128 + lane * 4;
        const float4 v = Quad<T>::load(row + c);
        *reinterpret_cast<float4*>(xr + c) = v;
        const float4 gg = Quad<T>::load(g + c);
        const float4 y = make_float4(v.x * gg.x, v.y * gg.y, v.z * gg.z, v.w * gg.w);
        const size_t o = act_off(m, c, d, sw_rows);      // 4 columns inside one 16-byte chunk
        Quad<T>::store(Xg + o, y);
        if (lo_off) {      // bf16 remainder (split activations)
            const float4 h = make_float4(to_f32<T>(from_f32<T>(y.x)), to_f32<T>(from_f32<T>(y.y)),
                                         to_f32<T>(from_f32<T>(y.z)), to_f32<T>(from_f32<T>(y.w)));
            Quad<T>::store(Xg + lo_off + o, make_float4(y.x - h.x, y.y - h.y, y.z - h.z, y.w - h.w));
        }
        float sq = v.x * v.x;
        sq = fmaf(v.y, v.y, sq);
        sq = fmaf(v.z, v.z, sq);
        sq = fmaf(v.w, v.w, sq);
        sq = warp_sum(sq);
        if (lane == 0) ssq[(size_t)tile * ssq_ld + m] = sq;
    }
}

constexpr int NORM_THREADS = 256;
constexpr int NORM_VEC = 8;      // float4 per thread held in registers: d <= 8192

// Xn[m] = X[m] / sqrt(mean(X[m]^2) + eps) * g, stored in the model dtype.  All loads of a
// row are issued at once; the sum of squares is reduced in a fixed order (per thread, then
// warp butterfly, then warps in order), so a row's result does not depend on M.
template <typename T>
__global__ void __launch_bounds__(NORM_THREADS) rmsnorm_kernel(const float* __restrict__ X, const T* __restrict__ g,
                                                               T* __restrict__ Xn, int d, float eps) {
    pdl_launch_dependents();
    const int m = blockIdx.x;
    const int n4 = d >> 2;
    const float4* x4 = reinterpret_cast<const float4*>(X + (size_t)m * d);
    float4 v[NORM_VEC];
    float ss = 0.0f;
#pragma unroll
    for (int j = 0; j < NORM_VEC; ++j) {
        const int i = threadIdx.x + NORM_THREADS * j;
        v[j] = i < n4 ? x4[i] : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int j = 0; j < NORM_VEC; ++j) {
        ss = fmaf(v[j].x, v[j].x, ss);
        ss = fmaf(v[j].y, v[j].y, ss);
        ss = fmaf(v[j].z, v[j].z, ss);
        ss = fmaf(v[j].w, v[j].w, ss);
    }
    __shared__ float red[NORM_THREADS / 32];
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(FULL_MASK, ss, o);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
    __syncthreads();
    float tot = 0.0f;
#pragma unroll
    for (int w = 0; w < NORM_THREADS / 32; ++w) tot += red[w];
    const float inv = 1.0f / sqrtf(tot / (float)d + eps);
#pragma unroll
    for (int j = 0; j < NORM_VEC; ++j) {
        const int i = threadIdx.x + NORM_THREADS * j;
        if (i < n4) {
            const float4 gg = Quad<T>::load(g + 4 * i);
            Quad<T>::store(Xn + (size_t)m * d + 4 * i,
                           make_float4(v[j].x * inv * gg.x, v[j].y * inv * gg.y, v[j].z * inv * gg.z, v[j].w * inv * gg.w));
        }
    }
}

// table[pos][j] = (cos, sin)(pos * theta^(-2j/hd)), evaluated in double precision.
__global__ void rope_table_kernel(float2* table, int max_pos, int half, int hd, double theta) {
    const size_t n = (size_t)max_pos * half;
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x) {
        const int pos = (int)(i / half);
        const int j = (int)(i - (size_t)pos * half);
        const double inv_freq = pow(theta, -2.0 * j / hd);
        const double ang = (double)pos * inv_freq;
        table[i] = make_float2((float)cos(ang), (float)sin(ang));
    }
}

// tokens[b][0] = last[b], tokens[b][1..K] = drafts[b][0..K).
__global__ void verify_tokens_kernel(const int* __restrict__ last, const int* __restrict__ drafts, int K,
                                     int* __restrict__ tokens, int B) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= B * (K + 1)) return;
    const int b = i / (K + 1), t = i - b * (K + 1);
    tokens[i] = t == 0 ? last[b] : drafts[b * K + t - 1];
}

// mode 0: len[slot] += add; mode 1: len[slot] += accepted[b] + 1 (trim after a verify
// pass that has not advanced the length); mode 2: len[slot] -= K - accepted[b].
__global__ void advance_len_kernel(const int* __restrict__ seq_ids, int* __restrict__ seq_len, int B, int mode,
                                   int add, const int* __restrict__ accepted, int K) {
    const int b = blockIdx.x * blockDim.x + threadIdx.x;
    if (b >= B) return;
    const int slot = seq_ids[b];
    int a = accepted ? accepted[b] : 0;
    a = a < 0 ? 0 : (a > K ? K : a);
    if (mode == 0) seq_len[slot] += add;
    else if (mode == 1) seq_len[slot] += a + 1;
    else seq_len[slot] -= K - a;
}

// dst[c * ldd + r] = src[r * lds + c] for r < R, c < C.
template <typename E>
__global__ void transpose_kernel(const E* __restrict__ src, int lds, E* __restrict__ dst, int ldd, int R, int C) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= R * C) return;
    const int r = i / C, c = i - r * C;
    dst[(size_t)c * ldd + r] = src[(size_t)r * lds + c];
}

void launch_transpose_i32(const int* src, int lds, int* dst, int ldd, int R, int C, cudaStream_t st) {
    transpose_kernel<int><<<(R * C + 255) / 256, 256, 0, st>>>(src, lds, dst, ldd, R, C);
}

void launch_transpose_f32(const float* src, int lds, float* dst, int ldd, int R, int C, cudaStream_t st) {
    transpose_kernel<float><<<(R * C + 255) / 256, 256, 0, st>>>(src, lds, dst, ldd, R, C);
}

void launch_embed(const Ctx& c, int M, int T, cudaStream_t st, bool fused_norm) {
    const int sw_rows = fused_norm ? act_rows(M) : 0;
    if (c.cfg.dtype == SPEC_BF16) {
        using bf = __nv_bfloat16;
        embed_kernel<bf><<<M, 256, 0, st>>>(c.d_tokens, c.d_seq_ids, c.d_seq_len, T, static_cast<const bf*>(c.w.embed),
                                            c.X, c.d_tok_seq, c.d_tok_pos, c.cfg.d_model, c.cfg.vocab,
                                            fused_norm ? static_cast<bf*>(c.Xn) : nullptr,
                                            static_cast<const bf*>(c.w.layers[0].attn_norm), c.ssq_a, c.Mmax,
                                            c.split ? (size_t)sw_rows * 64 : 0, sw_rows, c.d_tok_log,
                                            c.lim.max_ctx);
    } else {
        embed_kernel<float><<<M, 256, 0, st>>>(c.d_tokens, c.d_seq_ids, c.d_seq_len, T,
                                               static_cast<const float*>(c.w.embed), c.X, c.d_tok_seq, c.d_tok_pos,
                                               c.cfg.d_model, c.cfg.vocab, nullptr, nullptr, nullptr, 0, 0, 0,
                                               c.d_tok_log, c.lim.max_ctx);
    }
}

void launch_rmsnorm(const Ctx& c, const float* X, const void* g, void* Xn, int M, cudaStream_t st) {
    const int threads = NORM_THREADS;
    if (c.cfg.dtype == SPEC_BF16)
        rmsnorm_kernel<__nv_bfloat16><<<M, threads, 0, st>>>(X, static_cast<const __nv_bfloat16*>(g),
                                                             static_cast<__nv_bfloat16*>(Xn), c.cfg.d_model,
                                                             c.cfg.rms_eps);
    else
        rmsnorm_kernel<float><<<M, threads, 0, st>>>(X, static_cast<const float*>(g), static_cast<float*>(Xn),
                                                     c.cfg.d_model, c.cfg.rms_eps);
}

void launch_rope_table(float2* table, int max_pos, int hd, double theta, cudaStream_t st) {
    rope_table_kernel<<<512, 256, 0, st>>>(table, max_pos, hd / 2, hd, theta);
}

void launch_verify_tokens(const int* last, const int* drafts, int K, int* tokens, int B, cudaStream_t st) {
    const int n = B * (K + 1);
    verify_tokens_kernel<<<(n + 255) / 256, 256, 0, st>>>(last, drafts, K, tokens, B);
}

// Draft-length gate ("Speculative decoding on Apple Silicon" (mlx-optiq docs), section
// "N-gram lookup: any model"): a drafted token is accepted with probability alpha =
// (S + 1) / (S + F + 2), S the accepted draft tokens and F the first rejections of the
// slot's recent rounds, both decayed every round; a round of n drafts is expected to emit
// E(n) = 1 + alpha + ... + alpha^n tokens at the timed cost cost[n], and the gate drafts the
// n <= min(n_max, available) with the largest E(n) / cost[n], the smaller n on ties.  The
// same double-precision arithmetic as the host gate (spec_ngram_gate_*).
__device__ int gate_choose(double S, double F, const double* cost, int n_max, int available) {
    const int lim = max(0, min(n_max, available));
    const double a = (S + 1.0) / (S + F + 2.0);
    double e = 1.0, pw = 1.0, best_v = 1.0 / cost[0];
    int best = 0;
    for (int n = 1; n <= lim; ++n) {
        pw *= a;
        e += pw;
        const double v = e / cost[n];
        if (v > best_v) {
            best_v = v;
            best = n;
        }
    }
    return best;
}

__global__ void gate_update_kernel(const int* __restrict__ seq_ids, int B, double* __restrict__ sf, double decay,
                                   const int* __restrict__ drafted, const int* __restrict__ accepted) {
    const int b = blockIdx.x * blockDim.x + threadIdx.x;
    if (b >= B) return;
    const int slot = seq_ids[b];
    double S = sf[2 * slot] * decay, F = sf[2 * slot + 1] * decay;
    const int d = drafted[b], acc = accepted[b];
    if (d > 0) {
        S += acc;
        if (acc < d) F += 1.0;
    }
    sf[2 * slot] = S;
    sf[2 * slot + 1] = F;
}

__global__ void gate_choose_kernel(const int* __restrict__ seq_ids, int B, const double* __restrict__ sf,
                                   const double* __restrict__ cost, int n_max, const int* __restrict__ available,
                                   int* __restrict__ n_out) {
    const int b = blockIdx.x * blockDim.x + threadIdx.x;
    if (b >= B) return;
    const int slot = seq_ids[b];
    n_out[b] = gate_choose(sf[2 * slot], sf[2 * slot + 1], cost, n_max, available[b]);
}

void launch_gate_update(const Ctx& c, int B, const int* drafted, const int* accepted, cudaStream_t st) {
    gate_update_kernel<<<(B + 127) / 128, 128, 0, st>>>(c.d_seq_ids, B, c.d_gate_sf, c.gate_decay, drafted, accepted);
}

void launch_gate_choose(const Ctx& c, int B, const int* available, int* n_out, cudaStream_t st) {
    gate_choose_kernel<<<(B + 127) / 128, 128, 0, st>>>(c.d_seq_ids, B, c.d_gate_sf, c.d_gate_cost, c.gate_nmax,
                                                       available, n_out);
}

// N-gram drafts of one sequence per CTA ("Speculative decoding on Apple Silicon"
// (mlx-optiq docs), section "N-gram lookup: any model").  The context is the slot's
// committed tokens tok_log[slot][0, L) (L = its length) followed by the pending token: n =
// L + 1 tokens.  For every earlier end position e <= n - 2, l(e) = the length of the common
// suffix of ctx[0, e] and the whole context, capped at min(max_match, n - 1); an
// occurrence of the context's last m tokens ends at e exactly when l(e) >= m.  The longest
// suffix with an earlier occurrence is m* = max l(e) (drafting needs m* >= min_match), and
// its most recent occurrence is the largest e with l(e) = m*: one max-reduction of
// (l(e), e).  The draft is ctx[e + 1, e + 1 + k), k = min(n_draft, n - 1 - e), then the
// gate's choice for those k available tokens when gate_sf is set, then cap; rows past
// draft_len[b] = k hold the pending token.  The rule of spec_ngram_draft (host) and of the
// oracle's lookup, as one scan.
constexpr int NG_THREADS = 256;
__global__ void __launch_bounds__(NG_THREADS) ngram_draft_kernel(const int* __restrict__ seq_ids,
                                                               const int* __restrict__ seq_len,
                                                               const int* __restrict__ tok_log, int max_ctx,
                                                               const int* __restrict__ pending, int n_draft,
                                                               int min_match, int max_match,
                                                               const int* __restrict__ cap, int* __restrict__ drafts,
                                                               int* __restrict__ draft_len,
                                                               const double* __restrict__ gate_sf,
                                                               const double* __restrict__ gate_cost, int gate_nmax) {
    __shared__ int tail[SPEC_NGRAM_MAX_MATCH];
    __shared__ unsigned long long red[NG_THREADS / 32];
    const int b = blockIdx.x;
    const int slot = seq_ids[b];
    const int L = min(seq_len[slot], max_ctx);
    const int n = L + 1;
    const int* ctx = tok_log + (size_t)slot * max_ctx;
    const int last = pending[b];
    const int mcap = min(max_match, n - 1);
    if (threadIdx.x < SPEC_NGRAM_MAX_MATCH) {
        const int j = threadIdx.x;
        tail[j] = j == 0 ? last : (j < n ? ctx[n - 1 - j] : 0);
    }
    __syncthreads();
    // key = l << 32 | e, maximised; 0 = no occurrence of at least min_match tokens
    unsigned long long key = 0;
    for (int e = threadIdx.x; e <= n - 2; e += NG_THREADS) {
        int l = 0;
        while (l < mcap && l <= e && ctx[e - l] == tail[l]) ++l;
        if (l >= min_match) {
            const unsigned long long k = ((unsigned long long)l << 32) | (unsigned)e;
            key = k > key ? k : key;
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const unsigned long long x = __shfl_xor_sync(FULL_MASK, key, o);
        key = x > key ? x : key;
    }
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = key;
    __syncthreads();
    if (threadIdx.x == 0) {
        unsigned long long k = 0;
        for (int w = 0; w < NG_THREADS / 32; ++w) k = red[w] > k ? red[w] : k;
        red[0] = k;
    }
    __syncthreads();
    key = red[0];
    int k = 0, e = -1;
    if (key != 0) {
        e = (int)(key & 0xffffffffu);
        k = min(n_draft, n - 1 - e);
    }
    if (gate_sf != nullptr) k = gate_choose(gate_sf[2 * slot], gate_sf[2 * slot + 1], gate_cost, gate_nmax, k);
    if (cap) k = max(0, min(k, cap[b]));
    for (int i = threadIdx.x; i < n_draft; i += NG_THREADS) {
        const int p = e + 1 + i;
        drafts[(size_t)b * n_draft + i] = i < k ? (p == n - 1 ? last : ctx[p]) : last;
    }
    if (threadIdx.x == 0) draft_len[b] = k;
}

void launch_ngram_draft(const Ctx& c, int B, const int* pending, int n_draft, int min_match, int max_match,
                        const int* cap, int* drafts, int* draft_len, bool gated, cudaStream_t st) {
    ngram_draft_kernel<<<B, NG_THREADS, 0, st>>>(c.d_seq_ids, c.d_seq_len, c.d_tok_log, c.lim.max_ctx, pending, n_draft,
                                                min_match, max_match, cap, drafts, draft_len,
                                                gated ? c.d_gate_sf : nullptr, c.d_gate_cost, c.gate_nmax);
}

void launch_advance_len(const int* seq_ids, int* seq_len, int B, int mode, int add, const int* accepted, int K,
                        cudaStream_t st) {
    advance_len_kernel<<<(B + 127) / 128, 128, 0, st>>>(seq_ids, seq_len, B, mode, add, accepted, K);
}

}  // namespace sv
