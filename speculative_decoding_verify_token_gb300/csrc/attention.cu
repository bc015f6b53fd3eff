// Paged causal GQA attention of a decoder pass over T new tokens per sequence.
//
// For each (sequence, kv head) the T*G query rows (T positions x G = hq/hkv query heads)
// share one pass over the sequence's KV pages.  The keys are split at fixed absolute
// positions (SPLIT keys, a multiple of the 16-token page); one CTA per (split, kv head,
// sequence) loads all pages of its split with 1-D bulk copies on the TMA engine (each
// page-head block is a contiguous 16 x head_dim run) and computes, per visible row, the
// split's max, sum and unnormalised output.  The last CTA of a (sequence, kv head) to
// finish (atomic arrival count, no spin-wait) combines a row's splits 0..pos/SPLIT in
// order.  Every row is computed on its own in a fixed order of operations that depends
// only on its absolute position, so a token gets the same bits whether it is decoded
// alone (T = 1) or verified together with K drafts (T = K + 1).
#include <cuda_bf16.h>
#include <cmath>

#include "common.cuh"
#include "epilogue.cuh"
#include "model.h"

namespace sv {

constexpr int ATT_THREADS = 256;
constexpr int ATT_RT = 32;                     // query rows per tile
constexpr int ATT_KV_SMEM = 128 * 1024;        // K + V bytes of one split

constexpr int MMA_SPLIT = 64;                  // keys per split on the tensor-core path
constexpr int MMA_RT = 64;                     // query rows per tile (4 m16 tiles)
constexpr int MMA_PITCH = 136;                 // bf16 row pitch of K, V, Q in smem (272 B)
constexpr int MMA_PPITCH = 72;                 // bf16 row pitch of P (144 B)

static bool use_mma_path(int hd, int esize) { return hd == 128 && esize == 2; }

int attention_split_keys(int hd, int esize) {
    if (use_mma_path(hd, esize)) return MMA_SPLIT;
    int s = ATT_KV_SMEM / (2 * hd * esize);
    s = (s / 16) * 16;
    return s > 256 ? 256 : s;
}

template <typename T>
struct Vec16;   // 16 bytes of T as floats
template <>
struct Vec16<__nv_bfloat16> {
    static constexpr int N = 8;
    __device__ __forceinline__ static void load(const __nv_bfloat16* p, float* v) {
        const uint4 x = *reinterpret_cast<const uint4*>(p);
        const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            v[2 * i] = __uint_as_float(w[i] << 16);
            v[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
        }
    }
};
template <>
struct Vec16<float> {
    static constexpr int N = 4;
    __device__ __forceinline__ static void load(const float* p, float* v) {
        const float4 x = *reinterpret_cast<const float4*>(p);
        v[0] = x.x; v[1] = x.y; v[2] = x.z; v[3] = x.w;
    }
};

template <typename T>
__global__ void __launch_bounds__(ATT_THREADS, 1) attn_split_kernel(const AttnArgs a) {
    extern __shared__ __align__(128) uint8_t sm_raw[];
    __shared__ __align__(8) uint64_t bar;
    const int hd = a.hd, split = a.split_keys;
    T* Ks = reinterpret_cast<T*>(sm_raw);                               // [split][hd]
    T* Vs = Ks + (size_t)split * hd;                                    // [split][hd]
    float* Qs = reinterpret_cast<float*>(Vs + (size_t)split * hd);      // [RT][hd]
    float* Ss = Qs + (size_t)ATT_RT * hd;                               // [RT][split]

    pdl_launch_dependents();
    const int s = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
    const int slot = a.seq_ids[b];
    const int L0 = a.seq_len[slot];
    const int Ltot = L0 + a.T;
    const int k0 = s * split;
    if (k0 >= Ltot) return;
    const int nk = min(split, Ltot - k0);
    const int G = a.hq / a.hkv;
    const int R = a.T * G;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t bar_u = smem_u32(&bar);

    // ---- load the split's K and V pages (bulk copies, one mbarrier phase) ----
    const int npages = (nk + 15) >> 4;
    const uint32_t page_bytes = (uint32_t)(16 * hd * sizeof(T));
    if (threadIdx.x == 0) {
        mbar_init(bar_u, 1);
        fence_barrier_init();
        mbar_arrive_expect_tx(bar_u, 2u * page_bytes * (uint32_t)npages);
        const uint64_t pol = policy_evict_first();
        const T* kp = static_cast<const T*>(a.k_layer);
        const T* vp = static_cast<const T*>(a.v_layer);
        for (int pg = 0; pg < npages; ++pg) {
            const int page = a.block_table[(size_t)slot * a.max_pages + ((k0 >> 4) + pg)];
            const size_t off = ((size_t)page * a.hkv + g) * 16 * hd;
            bulk_g2s(smem_u32(Ks + (size_t)pg * 16 * hd), kp + off, page_bytes, bar_u, pol);
            bulk_g2s(smem_u32(Vs + (size_t)pg * 16 * hd), vp + off, page_bytes, bar_u, pol);
        }
    }
    const int t_first = max(0, k0 - L0);
    const T* Q = static_cast<const T*>(a.q);
    const size_t pbase = (((size_t)b * a.hkv + g) * a.n_chunks + s) * R;
    const int chunks16 = hd * (int)sizeof(T) / 16;          // 16-byte chunks per K row
    constexpr int VN = Vec16<T>::N;
    const int dpl = hd / 32;                                 // output dims per lane
    __syncthreads();
    bool ok = true;
    for (int rt = t_first * G; rt < R; rt += ATT_RT) {
        const int nr = min(ATT_RT, R - rt);
        __syncthreads();
        for (int i = threadIdx.x; i < nr * hd; i += ATT_THREADS) {
            const int ri = i / hd, dd = i - ri * hd;
            const int r = rt + ri, t = r / G, hh = r - t * G;
            const size_t m = (size_t)b * a.T + t;
            Qs[ri * hd + dd] = to_f32<T>(Q[(m * a.hq + (size_t)g * G + hh) * hd + dd]);
        }
        if (rt == t_first * G) ok = mbar_wait(bar_u, 0);     // the pages must have landed
        __syncthreads();
        if (!__syncthreads_and(ok)) break;
        // scores: warp per row, lane per key (keys lane + 32 i); each lane walks the
        // 16-byte chunks of its key row in a rotated order (conflict-free banks).
        for (int ri = warp; ri < nr; ri += ATT_THREADS / 32) {
            const int pos = L0 + (rt + ri) / G;
            const int lim = min(nk, pos - k0 + 1);
            const float* q = Qs + ri * hd;
            float* srow = Ss + (size_t)ri * split;
            for (int j = lane; j < split; j += 32) {
                float acc = -INFINITY;
                if (j < lim) {
                    acc = 0.0f;
                    const T* krow = Ks + (size_t)j * hd;
                    for (int c = 0; c < chunks16; ++c) {
                        const int cc = (c + lane) % chunks16;
                        float kv[VN];
                        Vec16<T>::load(krow + cc * VN, kv);
#pragma unroll
                        for (int e = 0; e < VN; ++e) acc = fmaf(q[cc * VN + e], kv[e], acc);
                    }
                    acc *= a.scale;
                }
                srow[j] = acc;
            }
            __syncwarp();
            float mx = -INFINITY;
            for (int j = lane; j < lim; j += 32) mx = fmaxf(mx, srow[j]);
            mx = warp_max(mx);
            float l = 0.0f;
            for (int j = lane; j < lim; j += 32) {
                const float p = expf(srow[j] - mx);
                srow[j] = p;
                l += p;
            }
            l = warp_sum(l);
            __syncwarp();
            float o[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) o[e] = 0.0f;
            for (int j = 0; j < lim; ++j) {
                const float p = srow[j];
                const T* vrow = Vs + (size_t)j * hd + lane * dpl;
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    if (e < dpl) o[e] = fmaf(p, to_f32<T>(vrow[e]), o[e]);
            }
            float* dst = a.part_o + (pbase + rt + ri) * hd + lane * dpl;
#pragma unroll
            for (int e = 0; e < 8; ++e)
                if (e < dpl) dst[e] = o[e];
            if (lane == 0) a.part_ml[pbase + rt + ri] = make_float2(mx * 1.4426950408889634f, l);
        }
    }
    if (!ok) mbar_wait(bar_u, 0);   // the copy never completed: one more bounded wait, then return
}


// ---- tensor-core path (bf16, head_dim 128): mma.sync m16n8k16 --------------------------------

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" :: "r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
    asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
}
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr));
}
__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
    asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
                 "{%0, %1, %2, %3};"
                 : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
                 : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&v);
}

// One CTA of 4 warps per (64-key split, kv head, sequence).  S = Q K^T with warp w owning
// keys [16w, 16w + 16); softmax statistics reduced in a fixed order; O = P V with warp w
// owning dims [32w, 32w + 32).  Rows are independent, so the bits do not depend on T.
__global__ void __launch_bounds__(128) attn_mma_kernel(const AttnArgs a) {
    extern __shared__ __align__(128) uint8_t sm_raw[];
    __shared__ float wmax[4][MMA_RT], wsum[4][MMA_RT];
    __nv_bfloat16* Ks = reinterpret_cast<__nv_bfloat16*>(sm_raw);
    __nv_bfloat16* Vs = Ks + MMA_SPLIT * MMA_PITCH;
    __nv_bfloat16* Qs = Vs + MMA_SPLIT * MMA_PITCH;
    __nv_bfloat16* Ps = Qs + MMA_RT * MMA_PITCH;

    pdl_launch_dependents();
    const int s = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
    const int slot = a.seq_ids[b];
    const int L0 = a.seq_len[slot];
    const int Ltot = L0 + a.T;
    const int k0 = s * MMA_SPLIT;
    if (k0 >= Ltot) return;
    const int nk = min(MMA_SPLIT, Ltot - k0);
    const int G = a.hq / a.hkv;
    const int R = a.T * G;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int gq = lane >> 2, tq = lane & 3;

    // K and V rows of the split (zero past the sequence end)
    const __nv_bfloat16* kp = static_cast<const __nv_bfloat16*>(a.k_layer);
    const __nv_bfloat16* vp = static_cast<const __nv_bfloat16*>(a.v_layer);
    for (int i = tid; i < MMA_SPLIT * 16; i += 128) {
        const int key = i >> 4, ch = i & 15;
        const uint32_t kd = smem_u32(Ks + key * MMA_PITCH + ch * 8);
        const uint32_t vd = smem_u32(Vs + key * MMA_PITCH + ch * 8);
        if (key < nk) {
            const int pos = k0 + key;
            const int page = a.block_table[(size_t)slot * a.max_pages + (pos >> 4)];
            const size_t off = (((size_t)page * a.hkv + g) * 16 + (pos & 15)) * 128 + ch * 8;
            cp_async16(kd, kp + off);
            cp_async16(vd, vp + off);
        } else {
            *reinterpret_cast<uint4*>(Ks + key * MMA_PITCH + ch * 8) = make_uint4(0, 0, 0, 0);
            *reinterpret_cast<uint4*>(Vs + key * MMA_PITCH + ch * 8) = make_uint4(0, 0, 0, 0);
        }
    }
    const int t_first = max(0, k0 - L0);
    const __nv_bfloat16* Q = static_cast<const __nv_bfloat16*>(a.q);
    const size_t pbase = (((size_t)b * a.hkv + g) * a.n_chunks + s) * R;
    const float sl2 = a.scale * 1.4426950408889634f;     // softmax in base 2
    for (int rt = t_first * G; rt < R; rt += MMA_RT) {
        const int nr = min(MMA_RT, R - rt);
        const int mtiles = (nr + 15) >> 4;
        __syncthreads();
        for (int i = tid; i < mtiles * 16 * 16; i += 128) {
            const int ri = i >> 4, ch = i & 15;
            if (ri < nr) {
                const int r = rt + ri, t = r / G, hh = r - t * G;
                const size_t m = (size_t)b * a.T + t;
                cp_async16(smem_u32(Qs + ri * MMA_PITCH + ch * 8), Q + (m * a.hq + (size_t)g * G + hh) * 128 + ch * 8);
            } else {
                *reinterpret_cast<uint4*>(Qs + ri * MMA_PITCH + ch * 8) = make_uint4(0, 0, 0, 0);
            }
        }
        cp_async_wait_all();
        __syncthreads();

        // ---- S = Q K^T for this warp's 16 keys ----
        float sacc[4][2][4];
#pragma unroll
        for (int mt = 0; mt < 4; ++mt)
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) sacc[mt][nt][e] = 0.0f;
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
            uint32_t b0, b1, b2, b3;
            {
                const int key = warp * 16 + (lane & 7) + (lane >> 4) * 8;
                const int dim = ks * 16 + ((lane >> 3) & 1) * 8;
                ldsm_x4(smem_u32(Ks + key * MMA_PITCH + dim), b0, b1, b2, b3);
            }
#pragma unroll
            for (int mt = 0; mt < 4; ++mt) {
                if (mt < mtiles) {
                    uint32_t a0, a1, a2, a3;
                    const int row = mt * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
                    const int col = ks * 16 + (lane >> 4) * 8;
                    ldsm_x4(smem_u32(Qs + row * MMA_PITCH + col), a0, a1, a2, a3);
                    mma16816(sacc[mt][0], a0, a1, a2, a3, b0, b1);
                    mma16816(sacc[mt][1], a0, a1, a2, a3, b2, b3);
                }
            }
        }
        // mask, per-warp row max
#pragma unroll
        for (int mt = 0; mt < 4; ++mt) {
            if (mt >= mtiles) continue;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int row = mt * 16 + gq + h * 8;
                const int pos = (row < nr) ? L0 + (rt + row) / G : -1;
                float mx = -INFINITY;
#pragma unroll
                for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const int key = warp * 16 + nt * 8 + 2 * tq + e;
                        float v = sacc[mt][nt][h * 2 + e] * sl2;
                        if (key >= nk || k0 + key > pos) v = -INFINITY;
                        sacc[mt][nt][h * 2 + e] = v;
                        mx = fmaxf(mx, v);
                    }
                mx = fmaxf(mx, __shfl_xor_sync(FULL, mx, 1));
                mx = fmaxf(mx, __shfl_xor_sync(FULL, mx, 2));
                if (tq == 0) wmax[warp][row] = mx;
            }
        }
        __syncthreads();
        // p = 2^(s - m), per-warp row sums, P to smem (bf16)
#pragma unroll
        for (int mt = 0; mt < 4; ++mt) {
            if (mt >= mtiles) continue;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int row = mt * 16 + gq + h * 8;
                float m = fmaxf(fmaxf(wmax[0][row], wmax[1][row]), fmaxf(wmax[2][row], wmax[3][row]));
                if (m == -INFINITY) m = 0.0f;
                float sum = 0.0f;
#pragma unroll
                for (int nt = 0; nt < 2; ++nt) {
                    const float p0 = exp2f(sacc[mt][nt][h * 2] - m);
                    const float p1 = exp2f(sacc[mt][nt][h * 2 + 1] - m);
                    sum += p0;
                    sum += p1;
                    *reinterpret_cast<uint32_t*>(Ps + row * MMA_PPITCH + warp * 16 + nt * 8 + 2 * tq) = pack_bf16(p0, p1);
                }
                sum += __shfl_xor_sync(FULL, sum, 1);
                sum += __shfl_xor_sync(FULL, sum, 2);
                if (tq == 0) wsum[warp][row] = sum;
            }
        }
        __syncthreads();
        // ---- O = P V for this warp's 32 dims ----
        float oacc[4][4][4];
#pragma unroll
        for (int mt = 0; mt < 4; ++mt)
#pragma unroll
            for (int nt = 0; nt < 4; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) oacc[mt][nt][e] = 0.0f;
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) {
            uint32_t v[8];
            {
                const int key = ks * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
                const int dim = warp * 32 + (lane >> 4) * 8;
                ldsm_x4_t(smem_u32(Vs + key * MMA_PITCH + dim), v[0], v[1], v[2], v[3]);
                ldsm_x4_t(smem_u32(Vs + key * MMA_PITCH + dim + 16), v[4], v[5], v[6], v[7]);
            }
#pragma unroll
            for (int mt = 0; mt < 4; ++mt) {
                if (mt < mtiles) {
                    uint32_t a0, a1, a2, a3;
                    const int row = mt * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
                    const int col = ks * 16 + (lane >> 4) * 8;
                    ldsm_x4(smem_u32(Ps + row * MMA_PPITCH + col), a0, a1, a2, a3);
                    mma16816(oacc[mt][0], a0, a1, a2, a3, v[0], v[1]);
                    mma16816(oacc[mt][1], a0, a1, a2, a3, v[2], v[3]);
                    mma16816(oacc[mt][2], a0, a1, a2, a3, v[4], v[5]);
                    mma16816(oacc[mt][3], a0, a1, a2, a3, v[6], v[7]);
                }
            }
        }
#pragma unroll
        for (int mt = 0; mt < 4; ++mt) {
            if (mt >= mtiles) continue;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int row = mt * 16 + gq + h * 8;
                if (row >= nr) continue;
                float* dst = a.part_o + (pbase + rt + row) * 128 + warp * 32 + 2 * tq;
#pragma unroll
                for (int nt = 0; nt < 4; ++nt)
                    *reinterpret_cast<float2*>(dst + nt * 8) = make_float2(oacc[mt][nt][h * 2], oacc[mt][nt][h * 2 + 1]);
                if (warp == 0 && tq == 0) {
                    const float m = fmaxf(fmaxf(wmax[0][row], wmax[1][row]), fmaxf(wmax[2][row], wmax[3][row]));
                    const float l = ((wsum[0][row] + wsum[1][row]) + wsum[2][row]) + wsum[3][row];
                    a.part_ml[pbase + rt + row] = make_float2(m, l);
                }
            }
        }
    }
}

// Combine of the splits of every query row: one warp per row; the row's splits
// 0..pos/SPLIT are reduced in a fixed order (lanes over splits for the max and the sum,
// then the output in split order), so the result depends only on the row's position.
template <typename T>
__global__ void __launch_bounds__(128) attn_combine_kernel(const AttnArgs a) {
    pdl_launch_dependents();
    pdl_wait();
    const int G = a.hq / a.hkv;
    const int R = a.T * G;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int r = blockIdx.x * 4 + warp;
    const int g = blockIdx.y, b = blockIdx.z;
    if (r >= R) return;
    const int slot = a.seq_ids[b];
    const int t = r / G, hh = r - t * G;
    const int ns = (a.seq_len[slot] + t) / a.split_keys + 1;
    const size_t cbase = ((size_t)b * a.hkv + g) * a.n_chunks;
    float mloc = -INFINITY;
    for (int c = lane; c < ns; c += 32) mloc = fmaxf(mloc, a.part_ml[(cbase + c) * R + r].x);
    const float mt = warp_max(mloc);
    float lloc = 0.0f;
    for (int c = lane; c < ns; c += 32) {
        const float2 ml = a.part_ml[(cbase + c) * R + r];
        lloc = fmaf(exp2f(ml.x - mt), ml.y, lloc);
    }
    const float l = warp_sum(lloc);
    const int dpl = a.hd / 32;
    float o[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) o[e] = 0.0f;
    for (int c0 = 0; c0 < ns; c0 += 8) {
        float w[8];
        float v[8][8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int c = c0 + u;
            w[u] = 0.0f;
            if (c < ns) {
                w[u] = exp2f(a.part_ml[(cbase + c) * R + r].x - mt);
                const float* src = a.part_o + ((cbase + c) * R + r) * a.hd + lane * dpl;
#pragma unroll
                for (int e = 0; e < 8; ++e) v[u][e] = e < dpl ? src[e] : 0.0f;
            }
        }
#pragma unroll
        for (int u = 0; u < 8; ++u)
            if (c0 + u < ns) {
#pragma unroll
                for (int e = 0; e < 8; ++e) o[e] = fmaf(w[u], v[u][e], o[e]);
            }
    }
    const size_t m = (size_t)b * a.T + t;
    T* dst = static_cast<T*>(a.o) + (m * a.hq + (size_t)g * G + hh) * a.hd + lane * dpl;
#pragma unroll
    for (int e = 0; e < 8; ++e)
        if (e < dpl) dst[e] = from_f32<T>(o[e] / l);
}

constexpr size_t MMA_SMEM = sizeof(__nv_bfloat16) * ((size_t)3 * 64 * MMA_PITCH + (size_t)MMA_RT * MMA_PPITCH);

size_t attn_smem(int hd, int esize) {
    const int split = attention_split_keys(hd, esize);
    return (size_t)2 * split * hd * esize + sizeof(float) * ((size_t)ATT_RT * hd + (size_t)ATT_RT * split);
}

int launch_attention(const Ctx& c, const AttnArgs& a, int B, int max_len_after, cudaStream_t st) {
    const int nsplit = (max_len_after + a.split_keys - 1) / a.split_keys;
    const int G = a.hq / a.hkv;
    const dim3 cgrid((a.T * G + 3) / 4, a.hkv, B);
    if (use_mma_path(a.hd, c.esize)) {
        attn_mma_kernel<<<dim3(nsplit, a.hkv, B), 128, MMA_SMEM, st>>>(a);
        attn_combine_kernel<__nv_bfloat16><<<cgrid, 128, 0, st>>>(a);
        return 2;
    }
    const size_t smem = attn_smem(a.hd, c.esize);
    const dim3 grid(nsplit, a.hkv, B);
    if (c.cfg.dtype == SPEC_BF16) {
        attn_split_kernel<__nv_bfloat16><<<grid, ATT_THREADS, smem, st>>>(a);
        attn_combine_kernel<__nv_bfloat16><<<cgrid, 128, 0, st>>>(a);
    } else {
        attn_split_kernel<float><<<grid, ATT_THREADS, smem, st>>>(a);
        attn_combine_kernel<float><<<cgrid, 128, 0, st>>>(a);
    }
    return 2;
}

int attention_set_smem_limits(int hd) {
    if (cudaFuncSetAttribute(attn_mma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)MMA_SMEM) !=
        cudaSuccess)
        return -1;
    if (cudaFuncSetAttribute(attn_split_kernel<__nv_bfloat16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)attn_smem(hd, 2)) != cudaSuccess ||
        cudaFuncSetAttribute(attn_split_kernel<float>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)attn_smem(hd, 4)) != cudaSuccess)
        return -1;
    return 0;
}

}  // namespace sv
