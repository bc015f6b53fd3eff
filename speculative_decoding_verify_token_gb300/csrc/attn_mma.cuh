// Device pieces of the tensor-core attention (bf16, head_dim 128, mma.sync m16n8k16): one
// (split, kv head, sequence) item over the paged KV cache, and the combine of one query
// row's splits.
#pragma once

#include <cuda_bf16.h>
#include <cmath>

#include "common.cuh"
#include "epilogue.cuh"
#include "model.h"

namespace sv {

constexpr int MMA_SPLIT = 64;                  // keys per split on the tensor-core path
constexpr int MMA_RT = 64;                     // query rows per tile (4 m16 tiles)
constexpr int MMA_PITCH = 136;                 // bf16 row pitch of K, V, Q in smem (272 B)
constexpr int MMA_PPITCH = 72;                 // bf16 row pitch of P (144 B)

// Shared memory of one attention item: K, V, Q, Q lo [64][MMA_PITCH] and P, P lo
// [64][MMA_PPITCH] bf16 (dynamic) and the per-warp row statistics.
struct AttnSmem {
    __nv_bfloat16 *Ks, *Vs, *Qs, *Qlo, *Ps, *Plo;     // Qlo, Plo: lo halves of split values
    float (*wmax)[MMA_RT];
    float (*wsum)[MMA_RT];
};
constexpr size_t MMA_SMEM = sizeof(__nv_bfloat16) * ((size_t)4 * 64 * MMA_PITCH + (size_t)2 * MMA_RT * MMA_PPITCH);

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

// The scores, softmax and P V of one tile of up to 64 query rows (rows rt .. rt + nr of the
// item, in Qs / Qlo rows 0 .. nr) against the nk keys in Ks / Vs starting at key k0, and the
// tile's per-split (max, sum, unnormalised output) for rows >= row_lo.  Each row's bits
// depend only on the row, the keys and the split, not on the other rows of the tile.
// The probabilities enter P V as bf16 hi + lo halves (Ps, Plo), like the split queries:
// rounded to bf16 alone (8 significant bits) they moved the logits of one 8B-width layer
// by up to 1e-2, which compounds over tens of layers.  Plo is written only after every
// warp has finished reading Ks, so it may alias Ks when the tile is the item's only one.
template <class Sync>
__device__ __forceinline__ void attn_mma_tile(const AttnArgs& a, const __nv_bfloat16* Ks, const __nv_bfloat16* Vs,
                                              const __nv_bfloat16* Qs, const __nv_bfloat16* Qlo, __nv_bfloat16* Ps,
                                              __nv_bfloat16* Plo,
                                              float (*wmax)[MMA_RT], float (*wsum)[MMA_RT], bool qsplit, int rt,
                                              int nr, int row_lo, int k0, int nk, int L0, int G, size_t pbase,
                                              float sl2, int tid, Sync sync) {
    const int warp = tid >> 5, lane = tid & 31;
    const int gq = lane >> 2, tq = lane & 3;
    const int mtiles = (nr + 15) >> 4;
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
                if (qsplit) {      // q_lo K^T into the same scores
                    ldsm_x4(smem_u32(Qlo + row * MMA_PITCH + col), a0, a1, a2, a3);
                    mma16816(sacc[mt][0], a0, a1, a2, a3, b0, b1);
                    mma16816(sacc[mt][1], a0, a1, a2, a3, b2, b3);
                }
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
    sync();
    // p = 2^(s - m), per-warp row sums, P to smem (bf16 hi and lo)
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
                const uint32_t hi = pack_bf16(p0, p1);
                const float2 hf = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&hi));
                *reinterpret_cast<uint32_t*>(Ps + row * MMA_PPITCH + warp * 16 + nt * 8 + 2 * tq) = hi;
                *reinterpret_cast<uint32_t*>(Plo + row * MMA_PPITCH + warp * 16 + nt * 8 + 2 * tq) =
                    pack_bf16(p0 - hf.x, p1 - hf.y);
            }
            sum += __shfl_xor_sync(FULL, sum, 1);
            sum += __shfl_xor_sync(FULL, sum, 2);
            if (tq == 0) wsum[warp][row] = sum;
        }
    }
    sync();
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
                ldsm_x4(smem_u32(Plo + row * MMA_PPITCH + col), a0, a1, a2, a3);
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

// One attention item: the 64-key split s of kv head g of sequence b, for all T*G query
// rows, by 128 threads (4 warps; tid in [0, 128)).  S = Q K^T with warp w owning keys
// [16w, 16w + 16); softmax statistics reduced in a fixed order; O = P V with warp w owning
// dims [32w, 32w + 32).  Rows are independent, so the bits do not depend on T.  sync() is
// a barrier of the 128 threads; dep_wait() (called by all of them) returns once the
// queries and this pass's keys may be read, false to give up.  The per-split (max, sum,
// unnormalised output) of every visible row goes to part_ml / part_o.
template <class Sync, class DepWait>
__device__ __forceinline__ bool attn_mma_item(const AttnArgs& a, int s, int g, int b, const AttnSmem& sm, int tid,
                                              Sync sync, DepWait dep_wait) {
    __nv_bfloat16* Ks = sm.Ks;
    __nv_bfloat16* Vs = sm.Vs;
    __nv_bfloat16* Qs = sm.Qs;
    __nv_bfloat16* Qlo = sm.Qlo;
    const bool qsplit = a.q_lo_off != 0;
    __nv_bfloat16* Ps = sm.Ps;
    float (*wmax)[MMA_RT] = sm.wmax;
    float (*wsum)[MMA_RT] = sm.wsum;
    const int slot = a.seq_ids[b];
    const int L0 = a.seq_len[slot];
    const int Ltot = L0 + a.T;
    const int k0 = s * MMA_SPLIT;
    if (k0 >= Ltot) return true;
    const int nk = min(MMA_SPLIT, Ltot - k0);
    const int G = a.hq / a.hkv;
    const int R = a.T * G;

    // K and V rows of the split (zero past the sequence end)
    const __nv_bfloat16* kp = static_cast<const __nv_bfloat16*>(a.k_layer);
    const __nv_bfloat16* vp = static_cast<const __nv_bfloat16*>(a.v_layer);
    // keys of earlier passes first; the keys of this pass (appended by the QKV GEMM) and
    // the queries only once dep_wait() has seen that GEMM's output
    const int n_old = max(0, min(nk, L0 - k0));
    for (int i = tid; i < MMA_SPLIT * 16; i += 128) {
        const int key = i >> 4, ch = i & 15;
        if (key < n_old) {
            const int pos = k0 + key;
            const int page = a.block_table[(size_t)slot * a.max_pages + (pos >> 4)];
            const size_t off = kv_off(page, g, pos & 15, ch * 8, a.hkv, 128, a.num_pages, a.kv_sw);
            cp_async16(smem_u32(Ks + key * MMA_PITCH + ch * 8), kp + off);
            cp_async16(smem_u32(Vs + key * MMA_PITCH + ch * 8), vp + off);
        } else if (key >= nk) {
            *reinterpret_cast<uint4*>(Ks + key * MMA_PITCH + ch * 8) = make_uint4(0, 0, 0, 0);
            *reinterpret_cast<uint4*>(Vs + key * MMA_PITCH + ch * 8) = make_uint4(0, 0, 0, 0);
        }
    }
    if (!dep_wait()) {
        cp_async_wait_all();     // let the copies already issued land before giving up
        return false;
    }
    for (int i = tid; i < MMA_SPLIT * 16; i += 128) {
        const int key = i >> 4, ch = i & 15;
        if (key >= n_old && key < nk) {
            const int pos = k0 + key;
            const int page = a.block_table[(size_t)slot * a.max_pages + (pos >> 4)];
            const size_t off = kv_off(page, g, pos & 15, ch * 8, a.hkv, 128, a.num_pages, a.kv_sw);
            cp_async16(smem_u32(Ks + key * MMA_PITCH + ch * 8), kp + off);
            cp_async16(smem_u32(Vs + key * MMA_PITCH + ch * 8), vp + off);
        }
    }
    const int t_first = max(0, k0 - L0);
    const __nv_bfloat16* Q = static_cast<const __nv_bfloat16*>(a.q);
    const size_t pbase = (((size_t)b * a.hkv + g) * a.n_chunks + s) * R;
    const float sl2 = a.scale * 1.4426950408889634f;     // softmax in base 2
    for (int rt = t_first * G; rt < R; rt += MMA_RT) {
        const int nr = min(MMA_RT, R - rt);
        const int mtiles = (nr + 15) >> 4;
        sync();
        for (int i = tid; i < mtiles * 16 * 16; i += 128) {
            const int ri = i >> 4, ch = i & 15;
            if (ri < nr) {
                const int r = rt + ri, t = r / G, hh = r - t * G;
                const size_t m = (size_t)b * a.T + t;
                const __nv_bfloat16* src = Q + (m * a.hq + (size_t)g * G + hh) * 128 + ch * 8;
                cp_async16(smem_u32(Qs + ri * MMA_PITCH + ch * 8), src);
                if (qsplit) cp_async16(smem_u32(Qlo + ri * MMA_PITCH + ch * 8), src + a.q_lo_off);
            } else {
                *reinterpret_cast<uint4*>(Qs + ri * MMA_PITCH + ch * 8) = make_uint4(0, 0, 0, 0);
                if (qsplit) *reinterpret_cast<uint4*>(Qlo + ri * MMA_PITCH + ch * 8) = make_uint4(0, 0, 0, 0);
            }
        }
        cp_async_wait_all();
        sync();

        attn_mma_tile(a, Ks, Vs, Qs, Qlo, Ps, sm.Plo, wmax, wsum, qsplit, rt, nr, 0, k0, nk, L0, G, pbase, sl2, tid,
                      sync);
    }
    return true;
}

template <typename T, int DPL>
__device__ __forceinline__ void attn_combine_row_dpl(const AttnArgs& a, int r, int g, int b, int lane) {
    const int G = a.hq / a.hkv;
    const int R = a.T * G;
    const int slot = a.seq_ids[b];
    const int t = r / G, hh = r - t * G;
    const int ns = (a.seq_len[slot] + t) / a.split_keys + 1;
    const size_t cbase = ((size_t)b * a.hkv + g) * a.n_chunks;
    // (max, sum) of splits lane, lane + 32, ...; the first 32 stay in registers and reach the
    // other lanes by shuffles, and the output loads of up to 16 splits are issued together
    float2 ml0 = make_float2(-INFINITY, 0.0f);
    if (lane < ns) ml0 = __ldcg(a.part_ml + (cbase + lane) * R + r);
    float mloc = ml0.x;
    for (int c = lane + 32; c < ns; c += 32) mloc = fmaxf(mloc, __ldcg(a.part_ml + (cbase + c) * R + r).x);
    const float mt = warp_max(mloc);
    float lloc = 0.0f;
    if (lane < ns) lloc = fmaf(exp2f(ml0.x - mt), ml0.y, lloc);
    for (int c = lane + 32; c < ns; c += 32) {
        const float2 ml = __ldcg(a.part_ml + (cbase + c) * R + r);
        lloc = fmaf(exp2f(ml.x - mt), ml.y, lloc);
    }
    const float l = warp_sum(lloc);
    float o[DPL];
#pragma unroll
    for (int e = 0; e < DPL; ++e) o[e] = 0.0f;
    constexpr int CG = 16;
    for (int c0 = 0; c0 < ns; c0 += CG) {
        float w[CG];
        float v[CG][DPL];
#pragma unroll
        for (int u = 0; u < CG; ++u) {
            const int c = c0 + u;
            w[u] = 0.0f;
            if (c < ns) {        // uniform over the warp
                const float mc = c < 32 ? __shfl_sync(FULL, ml0.x, c) : __ldcg(a.part_ml + (cbase + c) * R + r).x;
                w[u] = exp2f(mc - mt);
                const float* src = a.part_o + ((cbase + c) * R + r) * a.hd + lane * DPL;
#pragma unroll
                for (int e = 0; e < DPL; ++e) v[u][e] = __ldcg(src + e);
            }
        }
#pragma unroll
        for (int u = 0; u < CG; ++u)
            if (c0 + u < ns) {
#pragma unroll
                for (int e = 0; e < DPL; ++e) o[e] = fmaf(w[u], v[u][e], o[e]);
            }
    }
    const int m = b * a.T + t;
    const int col = ((g * G + hh) * a.hd) + lane * DPL;
#pragma unroll
    for (int e = 0; e < DPL; ++e)
        store_split<T>(static_cast<T*>(a.o) + act_off(m, col + e, a.hq * a.hd, a.o_sw_rows), a.o_lo_off, o[e] / l);
}

// head_dim 128 with the row's (max, sum) pairs staged in shared memory (mls: room for
// COMB_MAXC splits, per warp): the same arithmetic, in the same order, as the general
// version -- lanes over splits for the max and the sum, then the output in split order --
// with one 16-byte load per lane and split and CG splits' loads in flight.
constexpr int COMB_MAXC = 512;
template <typename T>
__device__ __forceinline__ void attn_combine_row_128(const AttnArgs& a, int r, int g, int b, int lane, float2* mls) {
    const int G = a.hq / a.hkv;
    const int R = a.T * G;
    const int slot = a.seq_ids[b];
    const int t = r / G, hh = r - t * G;
    const int ns = (a.seq_len[slot] + t) / a.split_keys + 1;
    const size_t cbase = ((size_t)b * a.hkv + g) * a.n_chunks;
    for (int c = lane; c < ns; c += 32) mls[c] = __ldcg(a.part_ml + (cbase + c) * R + r);
    __syncwarp();
    float mloc = -INFINITY;
    for (int c = lane; c < ns; c += 32) mloc = fmaxf(mloc, mls[c].x);
    const float mt = warp_max(mloc);
    float lloc = 0.0f;
    for (int c = lane; c < ns; c += 32) lloc = fmaf(exp2f(mls[c].x - mt), mls[c].y, lloc);
    const float l = warp_sum(lloc);
    __syncwarp();
    for (int c = lane; c < ns; c += 32) mls[c].x = exp2f(mls[c].x - mt);
    __syncwarp();
    float o0 = 0.0f, o1 = 0.0f, o2 = 0.0f, o3 = 0.0f;
    constexpr int CG = 16;
    const float4* src = reinterpret_cast<const float4*>(a.part_o + (cbase * R + r) * 128) + lane;
    const size_t cstride = (size_t)R * 128 / 4;      // float4 per split
    for (int c0 = 0; c0 < ns; c0 += CG) {
        float4 v[CG];
#pragma unroll
        for (int u = 0; u < CG; ++u)
            v[u] = c0 + u < ns ? __ldcg(src + (size_t)(c0 + u) * cstride) : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
#pragma unroll
        for (int u = 0; u < CG; ++u)
            if (c0 + u < ns) {        // uniform over the warp
                const float w = mls[c0 + u].x;
                o0 = fmaf(w, v[u].x, o0);
                o1 = fmaf(w, v[u].y, o1);
                o2 = fmaf(w, v[u].z, o2);
                o3 = fmaf(w, v[u].w, o3);
            }
    }
    __syncwarp();
    const int m = b * a.T + t;
    // four columns inside one 16-byte chunk of the operand layout
    T* dst = static_cast<T*>(a.o) + act_off(m, (g * G + hh) * 128 + lane * 4, a.hq * 128, a.o_sw_rows);
    store_split<T>(dst + 0, a.o_lo_off, o0 / l);
    store_split<T>(dst + 1, a.o_lo_off, o1 / l);
    store_split<T>(dst + 2, a.o_lo_off, o2 / l);
    store_split<T>(dst + 3, a.o_lo_off, o3 / l);
}

// Combine of the splits of one query row r of kv head g of sequence b, by one warp (lane =
// lane index): the row's splits 0..pos/SPLIT are reduced in a fixed order (lanes over
// splits for the max and the sum, then the output in split order), so the result depends
// only on the row's position.  head_dim = 32 * DPL.
template <typename T>
__device__ __forceinline__ void attn_combine_row(const AttnArgs& a, int r, int g, int b, int lane) {
    if (r >= a.T * (a.hq / a.hkv)) return;
    switch (a.hd / 32) {
    case 1: attn_combine_row_dpl<T, 1>(a, r, g, b, lane); break;
    case 2: attn_combine_row_dpl<T, 2>(a, r, g, b, lane); break;
    case 3: attn_combine_row_dpl<T, 3>(a, r, g, b, lane); break;
    case 4: attn_combine_row_dpl<T, 4>(a, r, g, b, lane); break;
    case 5: attn_combine_row_dpl<T, 5>(a, r, g, b, lane); break;
    case 6: attn_combine_row_dpl<T, 6>(a, r, g, b, lane); break;
    case 7: attn_combine_row_dpl<T, 7>(a, r, g, b, lane); break;
    default: attn_combine_row_dpl<T, 8>(a, r, g, b, lane); break;
    }
}

}  // namespace sv
