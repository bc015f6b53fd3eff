// Small kernels of the decoder pass: embedding gather (with per-token slot/position),
// RMSNorm, the RoPE table, the verify-pass token layout and the O(1) KV length updates.
#include <cuda_bf16.h>

#include "common.cuh"
#include "epilogue.cuh"
#include "model.h"

namespace sv {

// X[m][:] = E[tok[m]][:] in fp32; token m = b*T + t belongs to slot seq_ids[b] at
// position seq_len[slot] + t.  Ids outside [0, V) are embedded as token 0.
template <typename T>
__global__ void embed_kernel(const int* __restrict__ tokens, const int* __restrict__ seq_ids,
                             const int* __restrict__ seq_len, int T_per_seq, const T* __restrict__ E,
                             float* __restrict__ X, int* __restrict__ tok_seq, int* __restrict__ tok_pos, int d,
                             int V) {
    pdl_launch_dependents();
    const int m = blockIdx.x;
    const int b = m / T_per_seq;
    const int t = m - b * T_per_seq;
    int tok = tokens[m];
    if (tok < 0 || tok >= V) tok = 0;
    if (threadIdx.x == 0) {
        const int slot = seq_ids[b];
        tok_seq[m] = slot;
        tok_pos[m] = seq_len[slot] + t;
    }
    const T* row = E + (size_t)tok * d;
    for (int i = threadIdx.x; i < d; i += blockDim.x) X[(size_t)m * d + i] = to_f32<T>(row[i]);
}

// Xn[m] = X[m] / sqrt(mean(X[m]^2) + eps) * g, stored in the model dtype.
template <typename T>
__global__ void rmsnorm_kernel(const float* __restrict__ X, const T* __restrict__ g, T* __restrict__ Xn, int d,
                               float eps) {
    pdl_launch_dependents();
    const int m = blockIdx.x;
    const float* x = X + (size_t)m * d;
    float ss = 0.0f;
    for (int i = threadIdx.x; i < d; i += blockDim.x) ss += x[i] * x[i];
    __shared__ float red[32];
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(FULL_MASK, ss, o);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
    __syncthreads();
    if (threadIdx.x < 32) {
        float v = threadIdx.x < (blockDim.x >> 5) ? red[threadIdx.x] : 0.0f;
        for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(FULL_MASK, v, o);
        if (threadIdx.x == 0) red[0] = v;
    }
    __syncthreads();
    const float inv = 1.0f / sqrtf(red[0] / (float)d + eps);
    for (int i = threadIdx.x; i < d; i += blockDim.x)
        Xn[(size_t)m * d + i] = from_f32<T>(x[i] * inv * to_f32<T>(g[i]));
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

void launch_embed(const Ctx& c, int M, int T, cudaStream_t st) {
    if (c.cfg.dtype == SPEC_BF16)
        embed_kernel<__nv_bfloat16><<<M, 256, 0, st>>>(c.d_tokens, c.d_seq_ids, c.d_seq_len, T,
                                                       static_cast<const __nv_bfloat16*>(c.w.embed), c.X, c.d_tok_seq,
                                                       c.d_tok_pos, c.cfg.d_model, c.cfg.vocab);
    else
        embed_kernel<float><<<M, 256, 0, st>>>(c.d_tokens, c.d_seq_ids, c.d_seq_len, T,
                                               static_cast<const float*>(c.w.embed), c.X, c.d_tok_seq, c.d_tok_pos,
                                               c.cfg.d_model, c.cfg.vocab);
}

void launch_rmsnorm(const Ctx& c, const float* X, const void* g, void* Xn, int M, cudaStream_t st) {
    const int threads = c.cfg.d_model >= 1024 ? 512 : 256;
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

void launch_advance_len(const int* seq_ids, int* seq_len, int B, int mode, int add, const int* accepted, int K,
                        cudaStream_t st) {
    advance_len_kernel<<<(B + 127) / 128, 128, 0, st>>>(seq_ids, seq_len, B, mode, add, accepted, K);
}

}  // namespace sv
