// Device pieces of the tcgen05 skinny GEMM: PTX wrappers (TMA tensor loads, tcgen05 MMA /
// commit / TMEM loads), the shared-memory and instruction descriptors, the stream-K
// partition of the (tile, K atom) space and the epilogue of one staged accumulator chunk.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>

#include "common.cuh"
#include "epilogue.cuh"
#include "model.h"

namespace sv {

constexpr int TC_THREADS = 192;
constexpr int TC_BM = 128;
constexpr int TC_ATOM = 64;                          // K elements per atom = accumulation unit
constexpr int TC_ATOM_A = TC_BM * TC_ATOM * 2;       // 16 KB: one 128-row x 64 A atom
constexpr int TC_MAX_NTOK = 256;                    // tokens of one launch (more: several launches)
constexpr int TC_MMA_NMAX = 256;                    // N of one tcgen05.mma (M = 128)
constexpr int TC_MAX_STAGES = 8;
constexpr int TC_CW = 16;                           // epilogue column chunk
constexpr int TC_XPITCH = TC_CW + 1;
constexpr int TC_XBYTES = TC_BM * TC_XPITCH * 4;
// ---- PTX wrappers --------------------------------------------------------------------------

__device__ __forceinline__ uint64_t policy_evict_last() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// K-major operand, 128-byte swizzle: rows of 128 B, 8-row atoms 1024 B apart.
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t addr) {
    return (uint64_t)((addr >> 4) & 0x3FFFu) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
           ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

// kind::f16 instruction descriptor: D fp32, A and B bf16, both K-major, M = 128, N = n.
__device__ __forceinline__ uint32_t idesc_bf16(int n) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(TC_BM >> 4) << 24);
}

__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}"
        :: "r"(d_tmem), "l"(a), "l"(b), "r"(idesc), "r"(acc) : "memory");
}

// The four MMAs of one 64-column K atom (K = 16 each; descriptors advance by 32 bytes = 2
// units), in one asm block so that the issuing thread spends as few instructions as
// possible between them: the weight stream waits on this thread.  acc = 0 starts a new
// accumulation with the first of them.
__device__ __forceinline__ void mma_bf16_atom(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "setp.eq.b32 q, %4, %4;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %5, %6, %3, q;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %7, %8, %3, q;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %9, %10, %3, q;\n\t}"
        :: "r"(d_tmem), "l"(a), "l"(b), "r"(idesc), "r"(acc), "l"(a + 2), "l"(b + 2), "l"(a + 4), "l"(b + 4),
           "l"(a + 6), "l"(b + 6)
        : "memory");
}

__device__ __forceinline__ void mma_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" :: "r"(bar) : "memory");
}

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void epi_bar() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

// Accumulator values of tokens c0 .. c0 + 15 in this thread's TMEM lane: the W x_hi
// products plus the W x_lo products lo_col columns further on (hi + lo, in that order).
// lo_col = 8 (at most 8 tokens, c0 = 0): hi and lo share the one 16-column group.
__device__ __forceinline__ void acc_ld16(uint32_t taddr, int c0, int lo_col, float (&v)[16]) {
    tmem_ld16(taddr + (uint32_t)c0, v);
    if (lo_col >= 16) {
        float w[16];
        tmem_ld16(taddr + (uint32_t)(c0 + lo_col), w);
#pragma unroll
        for (int j = 0; j < 16; ++j) v[j] += w[j];
    } else {
#pragma unroll
        for (int j = 0; j < 8; ++j) v[j] += v[j + 8];
    }
}

// Rows of the activation operand B of one launch over M tokens: its rows = act_rows(M) hi
// rows, then its rows lo rows (every K atom of the operand layout holds them in that
// order), so the MMA's N is 2 rows, a token's lo product sits `rows` columns after its hi
// product, and one accumulator buffer spans 2 rows TMEM columns.  (One MMA per K-step
// over both halves: accumulating the lo rows into the hi rows' columns instead takes two
// MMAs per K-step, which at 8 rows, N = 16, doubled the tensor pipe's instruction count
// and slowed the 8-token GEMMs by a quarter.)
struct BRows {
    int rows;         // hi (and lo) rows of the launch
    int nb;           // rows of B (the MMA N)
    int lo_col;       // see acc_ld16
    int acc_stride;   // TMEM columns per accumulator buffer
};
__host__ __device__ inline BRows b_rows(int M) {
    BRows r;
    r.rows = act_rows(M);
    r.nb = 2 * r.rows;
    r.lo_col = r.rows;
    r.acc_stride = 2 * r.rows;
    return r;
}

// 1 if any of the 128 epilogue threads passes pred != 0 (and a barrier among them).
__device__ __forceinline__ int epi_any(int pred) {
    int r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\tsetp.ne.b32 p, %1, 0;\n\t"
        "bar.red.or.pred q, 1, 128, p;\n\tselp.b32 %0, 1, 0, q;\n\t}"
        : "=r"(r) : "r"(pred) : "memory");
    return r;
}

// ---- tile geometry --------------------------------------------------------------------------

// Source of half h (rows 64h .. 64h + 63) of the 128 rows of GEMM tile `tile`: matrix `mat`
// of the GEMM's weight list, rows row0 .. row0 + 63.  QKV stacks q, k and v (one 128-row
// head per tile); gate/up puts the 64 gate rows of 64 outputs over the 64 up rows of the
// same outputs (the SwiGLU epilogue pairs them); the others take 128 consecutive rows.
__host__ __device__ inline void tile_half_rows(int gid, int hq, int hkv, int tile, int h, int& mat, int& row0) {
    if (gid == GEMM_QKV) {
        int t = tile, w = 0;
        if (t >= hq) { t -= hq; w = 1; if (t >= hkv) { t -= hkv; w = 2; } }
        mat = w;
        row0 = t * TC_BM + 64 * h;
    } else if (gid == GEMM_GU) {
        mat = h;
        row0 = tile * 64;
    } else {
        mat = 0;
        row0 = tile * TC_BM + 64 * h;
    }
}

__device__ __forceinline__ long long range_start(long long T, int G, int c) {
    return (long long)(((unsigned long long)c * (unsigned long long)T) / (unsigned)G);
}

// CTA whose k-block range contains k-block x.
__device__ __forceinline__ int owner_cta(long long T, int G, long long x) {
    int c = (int)(((x + 1) * G + T - 1) / T) - 1;
    while (c > 0 && range_start(T, G, c) > x) --c;
    while (c + 1 < G && range_start(T, G, c + 1) <= x) ++c;
    return c;
}

// Walk of a CTA's atom range in pipeline stages: a stage holds up to p.atoms consecutive
// atoms of one tile segment.  Producer and MMA issuer walk it identically.
struct StageWalk {
    long long g, s1;
    int KB, A;
    __device__ __forceinline__ StageWalk(long long s0_, long long s1_, int KB_, int A_)
        : g(s0_), s1(s1_), KB(KB_), A(A_) {}
    __device__ __forceinline__ bool done() const { return g >= s1; }
    // atoms of the current stage, its tile, its first atom within the tile, and whether it
    // starts / ends a segment
    __device__ __forceinline__ void cur(int& n, int& tile, int& k_in_tile, bool& seg_first, bool& seg_last,
                                        long long seg_start_of_g) const {
        tile = (int)(g / KB);
        k_in_tile = (int)(g - (long long)tile * KB);
        const long long seg_end = min(s1, (long long)(tile + 1) * KB);
        n = (int)min((long long)A, seg_end - g);
        seg_first = (g == seg_start_of_g);
        seg_last = (g + n == seg_end);
    }
};

// Stream-K partial sums of one (CTA, slot): ntok / 16 chunks of 16 token columns, each
// stored as [4 float4 columns][TC_BM rows], so that a warp's stores and loads of one float4
// column of a chunk (32 consecutive rows) are contiguous.  ntok is a multiple of 16.
__device__ __forceinline__ float4* partial_f4(float* base, int cta, int which, int ntok, int c0, int j, int row) {
    return reinterpret_cast<float4*>(base + (((size_t)cta * 2 + which) * ntok + c0) * TC_BM) + (size_t)j * TC_BM + row;
}

// Inputs of the epilogue of the first 16-column chunk of a tile (residual values and the
// next norm's gains; or per-token positions, RoPE pairs and KV pages), loaded before the
// accumulator is ready so that their latency is off the end of the GEMM.
struct EpiPre {
    float2 v[TC_CW / 2];    // RESID: x pairs; QKV: (cos, sin)
    int pos[TC_CW / 2], page[TC_CW / 2];
    float2 g;               // RESID: gains of the next norm
};

__device__ __forceinline__ void epi_preload(int M, const EpiArgs& e, int tile, int etid, EpiPre& pre) {
    const int i = etid & 63;
    const int half = etid >> 6;
    const int pidx = tile * 64 + i;
    if (e.kind == EPI_RESID && e.xg_out != nullptr) {
        const int n0 = 2 * pidx;
        pre.g = __bfloat1622float2(
            *reinterpret_cast<const __nv_bfloat162*>(static_cast<const __nv_bfloat16*>(e.g_next) + n0));
#pragma unroll
        for (int j = 0; j < TC_CW / 2; ++j) {
            const int m = half + 2 * j;
            pre.v[j] = m < M ? __ldcg(reinterpret_cast<const float2*>(e.x + (size_t)(m + e.m0) * e.ldx + n0))
                             : make_float2(0.0f, 0.0f);
        }
    } else if (e.kind == EPI_QKV) {
        int hs, jq;
        qkv_pair_rows(pidx, e.hd, hs, jq);
#pragma unroll
        for (int j = 0; j < TC_CW / 2; ++j) {
            const int m = half + 2 * j;
            pre.pos[j] = m < M ? e.tok_pos[m + e.m0] : 0;
        }
#pragma unroll
        for (int j = 0; j < TC_CW / 2; ++j) {
            const int m = half + 2 * j;
            pre.v[j] = (m < M && hs < e.hq + e.hkv) ? e.rope[(size_t)pre.pos[j] * (e.hd >> 1) + jq]
                                                   : make_float2(1.0f, 0.0f);
            pre.page[j] = (m < M && hs >= e.hq)
                              ? e.block_table[(size_t)e.tok_seq[m + e.m0] * e.max_pages + (pre.pos[j] >> 4)] : 0;
        }
    }
}

// Epilogue of one 16-column chunk staged in xs[128][17]: 64 row pairs x 16 tokens.
// inv_s[m] = 1/rms of token m when the GEMM consumes a normed row; red = [4 warps][16]
// scratch of the sums of squares when it produces one; pre = the chunk's inputs already
// loaded by epi_preload (chunk c0 = 0 only), or nullptr.
__device__ __forceinline__ void epi_chunk(int gid, int M, const EpiArgs& e, const float* xs, const float* inv_s,
                                          float (*red)[TC_CW], int tile, int c0, int etid,
                                          const EpiPre* pre = nullptr) {
    const int i = etid & 63;
    const int half = etid >> 6;
    const bool adjacent = (gid == GEMM_O || gid == GEMM_DOWN || gid == GEMM_LM);
    const int r0 = adjacent ? 2 * i : i;
    const int r1 = adjacent ? 2 * i + 1 : i + 64;
    const int pidx = tile * 64 + i;
    if (e.kind == EPI_RESID && e.xg_out != nullptr) {
        // x += acc; xg = bf16(x * g_next); per token, the tile's sum of x^2 (each warp's
        // 32 pairs by a butterfly, then the two warps of a half in order)
        const int n0 = 2 * pidx;
        float2 g;
        const int wq = (etid >> 5) & 1;
        // this thread's residual pairs of the chunk's tokens, loaded together (written by
        // other CTAs: not from L1)
        float2 xin[TC_CW / 2];
        if (pre != nullptr) {
            g = pre->g;
#pragma unroll
            for (int j = 0; j < TC_CW / 2; ++j) xin[j] = pre->v[j];
        } else {
            g = __bfloat1622float2(
                *reinterpret_cast<const __nv_bfloat162*>(static_cast<const __nv_bfloat16*>(e.g_next) + n0));
#pragma unroll
            for (int j = 0; j < TC_CW / 2; ++j) {
                const int m = c0 + half + 2 * j;
                xin[j] = m < M ? __ldcg(reinterpret_cast<const float2*>(e.x + (size_t)(m + e.m0) * e.ldx + n0))
                               : make_float2(0.0f, 0.0f);
            }
        }
#pragma unroll
        for (int j = 0; j < TC_CW / 2; ++j) {
            const int cc = half + 2 * j;
            const int m = c0 + cc;
            if (m >= M) break;        // uniform over a warp: a warp holds one half
            float2* x = reinterpret_cast<float2*>(e.x + (size_t)(m + e.m0) * e.ldx + n0);
            float2 xv = xin[j];
            xv.x += xs[r0 * TC_XPITCH + cc];
            xv.y += xs[r1 * TC_XPITCH + cc];
            *x = xv;
            const float y0 = xv.x * g.x, y1 = xv.y * g.y;
            __nv_bfloat16* xg = static_cast<__nv_bfloat16*>(e.xg_out) + act_off(m + e.m0, n0, e.ldx, e.sw_rows);
            const __nv_bfloat162 hi = __floats2bfloat162_rn(y0, y1);
            *reinterpret_cast<__nv_bfloat162*>(xg) = hi;
            if (e.lo_off) {
                const float2 hf = __bfloat1622float2(hi);
                *reinterpret_cast<__nv_bfloat162*>(xg + e.lo_off) = __floats2bfloat162_rn(y0 - hf.x, y1 - hf.y);
            }
            const float sq = warp_sum(fmaf(xv.x, xv.x, xv.y * xv.y));
            if ((etid & 31) == 0) red[half * 2 + wq][cc] = sq;
        }
        epi_bar();
        if (etid < TC_CW && c0 + etid < M) {
            const int h = etid & 1;
            e.ssq_out[(size_t)tile * e.ssq_ld + e.m0 + c0 + etid] = red[2 * h][etid] + red[2 * h + 1][etid];
        }
        return;
    }
    const bool scaled = e.ssq_in != nullptr;
    if (e.kind == EPI_STORE && e.amax_out != nullptr) {
        // the tile's largest logit per token (lowest id on ties) instead of the logits: this
        // thread's two adjacent rows, its warp (butterfly over keys), then the two warps of
        // the token's parity (rows 0-63, then 64-127)
        float v[TC_CW / 2][2];
#pragma unroll
        for (int j = 0; j < TC_CW / 2; ++j) {
            const int cc = half + 2 * j;
            const float sc = (scaled && c0 + cc < M) ? inv_s[c0 + cc] : 1.0f;
            v[j][0] = xs[r0 * TC_XPITCH + cc] * sc;
            v[j][1] = xs[r1 * TC_XPITCH + cc] * sc;
        }
        epi_bar();          // every thread has its values: xs can hold the warps' keys
        unsigned long long* wk = reinterpret_cast<unsigned long long*>(const_cast<float*>(xs));   // [4][TC_CW]
        const int wq = (etid >> 5) & 1;
        const int id0 = tile * TC_BM + r0;
#pragma unroll
        for (int j = 0; j < TC_CW / 2; ++j) {
            const unsigned long long k0 = amax_key(v[j][0], id0), k1 = amax_key(v[j][1], id0 + 1);
            unsigned long long k = k0 > k1 ? k0 : k1;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                const unsigned long long x = __shfl_xor_sync(FULL_MASK, k, o);
                k = x > k ? x : k;
            }
            if ((etid & 31) == 0) wk[(half * 2 + wq) * TC_CW + half + 2 * j] = k;
        }
        epi_bar();
        if (etid < TC_CW && c0 + etid < M) {
            const int h = etid & 1;
            const unsigned long long a = wk[(2 * h) * TC_CW + etid], b2 = wk[(2 * h + 1) * TC_CW + etid];
            e.amax_out[(size_t)(e.m0 + c0 + etid) * e.amax_ld + tile] = a > b2 ? a : b2;
        }
        return;
    }
    if (e.kind == EPI_QKV) {
        // the chunk's per-token inputs (position, RoPE pair, KV page) loaded together first
        int hs, jq;
        qkv_pair_rows(pidx, e.hd, hs, jq);
        int pos[TC_CW / 2], page[TC_CW / 2];
        float2 cs[TC_CW / 2];
        if (pre != nullptr) {
#pragma unroll
            for (int j = 0; j < TC_CW / 2; ++j) {
                pos[j] = pre->pos[j];
                cs[j] = pre->v[j];
                page[j] = pre->page[j];
            }
        } else {
#pragma unroll
            for (int j = 0; j < TC_CW / 2; ++j) {
                const int m = c0 + half + 2 * j;
                pos[j] = m < M ? e.tok_pos[m + e.m0] : 0;
            }
#pragma unroll
            for (int j = 0; j < TC_CW / 2; ++j) {
                const int m = c0 + half + 2 * j;
                cs[j] = (m < M && hs < e.hq + e.hkv) ? e.rope[(size_t)pos[j] * (e.hd >> 1) + jq]
                                                     : make_float2(1.0f, 0.0f);
                page[j] = (m < M && hs >= e.hq)
                              ? e.block_table[(size_t)e.tok_seq[m + e.m0] * e.max_pages + (pos[j] >> 4)] : 0;
            }
        }
#pragma unroll
        for (int j = 0; j < TC_CW / 2; ++j) {
            const int cc = half + 2 * j;
            const int m = c0 + cc;
            if (m >= M) break;
            float a0 = xs[r0 * TC_XPITCH + cc], a1 = xs[r1 * TC_XPITCH + cc];
            if (scaled) {
                const float s = inv_s[m];
                a0 *= s;
                a1 *= s;
            }
            qkv_store<__nv_bfloat16>(e, m + e.m0, hs, jq, pos[j], cs[j], page[j], a0, a1);
        }
        return;
    }
    for (int cc = half; cc < TC_CW; cc += 2) {
        const int m = c0 + cc;
        if (m >= M) break;
        float a0 = xs[r0 * TC_XPITCH + cc], a1 = xs[r1 * TC_XPITCH + cc];
        if (scaled) {
            const float s = inv_s[m];
            a0 *= s;
            a1 *= s;
        }
        epi_pair<__nv_bfloat16>(e, m, pidx, a0, a1);
    }
}

}  // namespace sv
