// Paged causal GQA attention of a decoder pass over T new tokens per sequence.
//
// For each (sequence, kv head) the T*G query rows (T positions x G = hq/hkv query heads)
// share one pass over the sequence's KV pages.  The keys are split into chunks of 64
// absolute positions; chunk c of a row holds partial (max, sum, unnormalised output) over
// the keys in [64c, 64c + 64) that the row may see (key position <= row position).  The
// combine walks a row's chunks 0..pos/64 in order.  Every row is computed on its own with
// a fixed order of operations, so a token gets the same bits whether it is decoded alone
// (T = 1) or verified together with K drafts (T = K + 1).
#include <cuda_bf16.h>
#include <cmath>

#include "epilogue.cuh"
#include "model.h"

namespace sv {

constexpr int ATT_RT = 32;

template <typename T>
__global__ void __launch_bounds__(256) attn_partial_kernel(const AttnArgs a) {
    extern __shared__ float sm[];
    const int hd = a.hd, hdp = hd + 1;
    float* Ks = sm;                                   // [64][hd+1]
    float* Vs = Ks + ATT_CHUNK * hdp;                 // [64][hd]
    float* Qs = Vs + ATT_CHUNK * hd;                  // [RT][hd+1]
    float* Ss = Qs + ATT_RT * hdp;                    // [RT][65]

    const int c = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
    const int slot = a.seq_ids[b];
    const int L0 = a.seq_len[slot];
    const int Ltot = L0 + a.T;
    const int k0 = c * ATT_CHUNK;
    if (k0 >= Ltot) return;
    const int nk = min(ATT_CHUNK, Ltot - k0);
    const int G = a.hq / a.hkv;
    const int R = a.T * G;
    const T* kp = static_cast<const T*>(a.k_layer);
    const T* vp = static_cast<const T*>(a.v_layer);
    for (int i = threadIdx.x; i < nk * hd; i += blockDim.x) {
        const int key = i / hd, dd = i - key * hd;
        const int pos = k0 + key;
        const int page = a.block_table[(size_t)slot * a.max_pages + (pos >> 4)];
        const size_t off = (((size_t)page * a.hkv + g) * 16 + (pos & 15)) * hd + dd;
        Ks[key * hdp + dd] = to_f32<T>(kp[off]);
        Vs[key * hd + dd] = to_f32<T>(vp[off]);
    }
    const int t_first = max(0, k0 - L0);
    const T* Q = static_cast<const T*>(a.q);
    const size_t cbase = (((size_t)b * a.hkv + g) * a.n_chunks + c) * R;
    for (int rt = t_first * G; rt < R; rt += ATT_RT) {
        const int nr = min(ATT_RT, R - rt);
        __syncthreads();
        for (int i = threadIdx.x; i < nr * hd; i += blockDim.x) {
            const int ri = i / hd, dd = i - ri * hd;
            const int r = rt + ri, t = r / G, hh = r - t * G;
            const size_t m = (size_t)b * a.T + t;
            Qs[ri * hdp + dd] = to_f32<T>(Q[(m * a.hq + (size_t)g * G + hh) * hd + dd]);
        }
        __syncthreads();
        for (int i = threadIdx.x; i < nr * ATT_CHUNK; i += blockDim.x) {
            const int ri = i / ATT_CHUNK, key = i - ri * ATT_CHUNK;
            const int pos = L0 + (rt + ri) / G;
            float s = -INFINITY;
            if (key < nk && k0 + key <= pos) {
                const float* q = Qs + ri * hdp;
                const float* kk = Ks + key * hdp;
                float acc = 0.0f;
                for (int dd = 0; dd < hd; ++dd) acc = fmaf(q[dd], kk[dd], acc);
                s = acc * a.scale;
            }
            Ss[ri * (ATT_CHUNK + 1) + key] = s;
        }
        __syncthreads();
        const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
        for (int ri = warp; ri < nr; ri += blockDim.x >> 5) {
            float* srow = Ss + ri * (ATT_CHUNK + 1);
            const float s0 = srow[lane], s1 = srow[lane + 32];
            float mx = fmaxf(s0, s1);
            for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(FULL_MASK, mx, o));
            const float p0 = s0 == -INFINITY ? 0.0f : expf(s0 - mx);
            const float p1 = s1 == -INFINITY ? 0.0f : expf(s1 - mx);
            srow[lane] = p0;
            srow[lane + 32] = p1;
            float l = p0 + p1;
            for (int o = 16; o > 0; o >>= 1) l += __shfl_xor_sync(FULL_MASK, l, o);
            if (lane == 0) a.part_ml[cbase + rt + ri] = make_float2(mx, l);
        }
        __syncthreads();
        for (int i = threadIdx.x; i < nr * hd; i += blockDim.x) {
            const int ri = i / hd, dd = i - ri * hd;
            const int pos = L0 + (rt + ri) / G;
            const int lim = min(nk, pos - k0 + 1);
            const float* prow = Ss + ri * (ATT_CHUNK + 1);
            float acc = 0.0f;
            for (int key = 0; key < lim; ++key) acc = fmaf(prow[key], Vs[key * hd + dd], acc);
            a.part_o[(cbase + rt + ri) * hd + dd] = acc;
        }
    }
}

template <typename T>
__global__ void attn_combine_kernel(const AttnArgs a) {
    const int r = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
    const int G = a.hq / a.hkv;
    const int R = a.T * G;
    if (r >= R) return;
    const int slot = a.seq_ids[b];
    const int t = r / G, hh = r - t * G;
    const int pos = a.seq_len[slot] + t;
    const int nc = pos / ATT_CHUNK + 1;
    const size_t base = ((size_t)b * a.hkv + g) * a.n_chunks;
    float mt = -INFINITY;
    for (int c = 0; c < nc; ++c) mt = fmaxf(mt, a.part_ml[(base + c) * R + r].x);
    T* O = static_cast<T*>(a.o);
    const size_t m = (size_t)b * a.T + t;
    for (int dd = threadIdx.x; dd < a.hd; dd += blockDim.x) {
        float o = 0.0f, l = 0.0f;
        for (int c = 0; c < nc; ++c) {
            const float2 ml = a.part_ml[(base + c) * R + r];
            const float w = expf(ml.x - mt);
            o = fmaf(w, a.part_o[((base + c) * R + r) * a.hd + dd], o);
            l = fmaf(w, ml.y, l);
        }
        O[(m * a.hq + (size_t)g * G + hh) * a.hd + dd] = from_f32<T>(o / l);
    }
}

size_t attn_partial_smem(int hd) {
    return sizeof(float) * ((size_t)ATT_CHUNK * (hd + 1) + (size_t)ATT_CHUNK * hd + (size_t)ATT_RT * (hd + 1) +
                            (size_t)ATT_RT * (ATT_CHUNK + 1));
}

int launch_attention(const Ctx& c, const AttnArgs& a, int B, int max_len_after, cudaStream_t st) {
    const int chunks = (max_len_after + ATT_CHUNK - 1) / ATT_CHUNK;
    const size_t smem = attn_partial_smem(a.hd);
    const dim3 g1(chunks, a.hkv, B);
    const dim3 g2(a.T * (a.hq / a.hkv), a.hkv, B);
    if (c.cfg.dtype == SPEC_BF16) {
        attn_partial_kernel<__nv_bfloat16><<<g1, 256, smem, st>>>(a);
        attn_combine_kernel<__nv_bfloat16><<<g2, 128, 0, st>>>(a);
    } else {
        attn_partial_kernel<float><<<g1, 256, smem, st>>>(a);
        attn_combine_kernel<float><<<g2, 128, 0, st>>>(a);
    }
    return 2;
}

int attention_set_smem_limits(int hd) {
    const int smem = (int)attn_partial_smem(hd);
    if (cudaFuncSetAttribute(attn_partial_kernel<__nv_bfloat16>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) !=
            cudaSuccess ||
        cudaFuncSetAttribute(attn_partial_kernel<float>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) !=
            cudaSuccess)
        return -1;
    return 0;
}

}  // namespace sv
