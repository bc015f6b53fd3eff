// CUDA-core GEMM with the decoder epilogues: the fp32 path (exact fp32 arithmetic for the
// float32 configuration, where tensor cores would round to tf32).
//
// One warp owns one row pair (see epilogue.cuh) for all M tokens; lanes stride over K with
// 16-byte loads and the partial sums are combined by a fixed butterfly.  The arithmetic of
// an output element does not depend on M, so a token's logits are bit-identical whether it
// is decoded alone or verified together with K drafts.
#include <cuda_bf16.h>

#include "epilogue.cuh"
#include "model.h"

namespace sv {

template <typename T>
struct PairWeights {
    const T* a;      // QKV: Wq, SWIGLU: Wg, else W
    const T* b;      // QKV: Wk, SWIGLU: Wu
    const T* c;      // QKV: Wv
    int K;
    int n_pairs;
};

template <typename T>
__device__ __forceinline__ void pair_rows(int kind, const PairWeights<T>& w, const EpiArgs& e, int p, const T*& r0,
                                          const T*& r1) {
    const size_t K = (size_t)w.K;
    if (kind == EPI_QKV) {
        int hs, j;
        qkv_pair_rows(p, e.hd, hs, j);
        const T* base;
        int h;
        if (hs < e.hq) { base = w.a; h = hs; }
        else if (hs < e.hq + e.hkv) { base = w.b; h = hs - e.hq; }
        else { base = w.c; h = hs - e.hq - e.hkv; }
        r0 = base + ((size_t)h * e.hd + j) * K;
        r1 = r0 + (size_t)(e.hd >> 1) * K;
    } else if (kind == EPI_SWIGLU) {
        r0 = w.a + (size_t)p * K;
        r1 = w.b + (size_t)p * K;
    } else {
        r0 = w.a + (size_t)(2 * p) * K;
        r1 = r0 + K;
    }
}

template <typename T>
__device__ __forceinline__ void load_vec(const T* p, float (&v)[16 / sizeof(T)]);

template <>
__device__ __forceinline__ void load_vec<float>(const float* p, float (&v)[4]) {
    const float4 x = *reinterpret_cast<const float4*>(p);
    v[0] = x.x; v[1] = x.y; v[2] = x.z; v[3] = x.w;
}

template <>
__device__ __forceinline__ void load_vec<__nv_bfloat16>(const __nv_bfloat16* p, float (&v)[8]) {
    const uint4 x = *reinterpret_cast<const uint4*>(p);
    const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        v[2 * i] = __uint_as_float(w[i] << 16);
        v[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
}

constexpr int SIMT_MT = 8;
constexpr int SIMT_WARPS = 8;

template <typename T>
__global__ void __launch_bounds__(SIMT_WARPS * 32) gemm_simt_kernel(const PairWeights<T> w, const T* __restrict__ X,
                                                                     const EpiArgs e) {
    const int lane = threadIdx.x & 31;
    const int p = blockIdx.x * SIMT_WARPS + (threadIdx.x >> 5);
    if (p >= w.n_pairs) return;
    const T* r0;
    const T* r1;
    pair_rows<T>(e.kind, w, e, p, r0, r1);
    constexpr int VEC = 16 / sizeof(T);
    const int K = w.K;
    for (int m0 = 0; m0 < e.M; m0 += SIMT_MT) {
        float acc0[SIMT_MT], acc1[SIMT_MT];
#pragma unroll
        for (int i = 0; i < SIMT_MT; ++i) { acc0[i] = 0.0f; acc1[i] = 0.0f; }
        for (int k = lane * VEC; k < K; k += 32 * VEC) {
            float wa[VEC], wb[VEC];
            load_vec<T>(r0 + k, wa);
            load_vec<T>(r1 + k, wb);
#pragma unroll
            for (int i = 0; i < SIMT_MT; ++i) {
                if (m0 + i < e.M) {
                    float xv[VEC];
                    load_vec<T>(X + (size_t)(m0 + i) * K + k, xv);
#pragma unroll
                    for (int q = 0; q < VEC; ++q) {
                        acc0[i] = fmaf(xv[q], wa[q], acc0[i]);
                        acc1[i] = fmaf(xv[q], wb[q], acc1[i]);
                    }
                }
            }
        }
#pragma unroll
        for (int i = 0; i < SIMT_MT; ++i) {
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                acc0[i] += __shfl_xor_sync(FULL_MASK, acc0[i], o);
                acc1[i] += __shfl_xor_sync(FULL_MASK, acc1[i], o);
            }
        }
        float s0 = 0.0f, s1 = 0.0f;
#pragma unroll
        for (int i = 0; i < SIMT_MT; ++i)
            if (lane == i) { s0 = acc0[i]; s1 = acc1[i]; }
        if (lane < SIMT_MT && m0 + lane < e.M) epi_pair<T>(e, m0 + lane, p, s0, s1);
    }
}

// n_pairs: QKV (hq + 2 hkv) * hd / 2; SWIGLU F; RESID / STORE N / 2.
void launch_gemm_simt(const Ctx& c, const void* wa, const void* wb, const void* wc, int K, int n_pairs,
                      const void* X, const EpiArgs& e, cudaStream_t st) {
    const int grid = (n_pairs + SIMT_WARPS - 1) / SIMT_WARPS;
    if (c.cfg.dtype == SPEC_BF16) {
        PairWeights<__nv_bfloat16> w{static_cast<const __nv_bfloat16*>(wa), static_cast<const __nv_bfloat16*>(wb),
                                     static_cast<const __nv_bfloat16*>(wc), K, n_pairs};
        gemm_simt_kernel<__nv_bfloat16><<<grid, SIMT_WARPS * 32, 0, st>>>(w, static_cast<const __nv_bfloat16*>(X), e);
    } else {
        PairWeights<float> w{static_cast<const float*>(wa), static_cast<const float*>(wb),
                             static_cast<const float*>(wc), K, n_pairs};
        gemm_simt_kernel<float><<<grid, SIMT_WARPS * 32, 0, st>>>(w, static_cast<const float*>(X), e);
    }
}

}  // namespace sv
