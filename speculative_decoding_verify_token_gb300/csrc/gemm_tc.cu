// Skinny bf16 GEMM of the verify pass on the 5th-generation tensor cores (tcgen05).
//
// Y[m][n] = sum_k X[m][k] W[n][k] with M = B*(K+1) tokens (<= 256) and weight matrices of
// 6-150 k rows: the work is streaming the weights through HBM ("most of that pass is spent
// moving weights through memory", "Speculative Decoding on Apple Silicon...", section
// "How speculative decoding works").  Design:
//  * swap-AB: a 128-row weight tile is the A operand, the tokens' hi and lo rows are the N
//    dimension (16..512, two MMAs above 256); the fp32 accumulator [128 x N] lives in
//    tensor memory, two of them while they fit its 512 columns (up to 128 tokens);
//  * the weights are re-laid out once, when they are loaded, tile-major: every (tile, K
//    atom) is the 16 KB A operand of one MMA atom, already in the 128-byte-swizzled order
//    the tensor cores read, so a ring stage of n consecutive atoms of a tile is ONE
//    contiguous bulk copy (cp.async.bulk) of n x 16 KB; a tensor-map box of 64 rows
//    instead makes 64 separate 128-byte row requests, and issuing the boxes of a stage
//    costs microseconds at the start of every GEMM;
//  * the activations (the B operand: hi rows, then lo rows) are written by the kernels that
//    produce them directly in the same swizzled order, K atom by K atom (the operand
//    layout, epilogue.cuh), so a stage's B is one bulk copy as well: a tensor-map load
//    of 16-row boxes moved about 37 GB/s per SM against 130-170 GB/s for one bulk copy of
//    the same bytes, which at 144 tokens (36 KB of B per 16 KB weight atom) made the
//    activations, not the weights, the limit; stages go into an mbarrier ring of up to 8
//    stages of up to four 64-column K atoms; weights are loaded evict-first, activations
//    evict-last (every CTA re-reads them);
//  * warp roles: warp 0 = TMA producer, warp 1 = tcgen05.mma issuer (one thread) and TMEM
//    owner, warps 2-5 = epilogue (tcgen05.ld of the 4 lane quarters);
//  * persistent stream-K: the (tile, k-block) space is cut into one contiguous range per
//    CTA; a tile shared by several CTAs is finished by the last one to arrive (atomic
//    ticket, no spin-wait), which adds the partial sums in CTA order.  With a whole number
//    s of CTAs per tile and more than 16 tokens, the s CTAs instead share the finishing
//    (each takes every s-th 16-token chunk, after a bounded wait for the others' partial
//    sums, adding them in the same order).  The split depends only on the weight shape and
//    the SM count, so a token's outputs are bit-identical for every M (a decode step and a
//    verify pass agree exactly);
//  * fused epilogues (RoPE + paged KV append, SwiGLU, residual add, fp32 logits) shared
//    with the CUDA-core GEMM, and a fused RMSNorm: the residual GEMMs also write
//    bf16(x * g) of the next norm and per-tile sums of squares, and the GEMM reading that
//    normed row scales its accumulators by 1/rms of the token.
#include <cuda.h>
#include <cuda_bf16.h>
#include <algorithm>

#include "host_util.h"
#include "tc_common.cuh"

namespace sv {

#ifndef TC_MAX_ATOMS
#define TC_MAX_ATOMS 4          // most 64-element K atoms (128-byte swizzle spans) per stage
#endif
#ifndef TC_MIN_STAGES
#define TC_MIN_STAGES 2         // fewest pipeline stages a launch may use (fewer, larger stages
#endif                          // measured faster at 144 tokens: 2 x 104 KB over 4 x 52 KB)
#ifndef TC_CTAS_PER_SM
#define TC_CTAS_PER_SM 1        // resident GEMM CTAs per SM (shared memory split between them)
#endif
// dynamic bytes per CTA: with one CTA per SM, three stages of four atoms at 16 tokens plus
// the staging tile and the alignment slack, leaving 1.5 KB of the 227 KB for static data
constexpr int TC_SMEM_MAX = TC_CTAS_PER_SM == 1 ? 230912 : 110 * 1024;

struct TcParams {
    const uint8_t* wt;        // this GEMM's tile-major weights: [n_tiles][KB] atoms of TC_ATOM_A bytes
    const uint8_t* x;         // the GEMM input in the operand layout of a pass of x_rows rows
    int x_rows;
    int gid;
    int n_tiles, KB;          // tiles; K atoms per tile (the stream-K unit)
    int ntok, M, x_row0;      // ntok = M rounded up to 16 (stride of the partial sums)
    int x_whole;              // the launch reads all x_rows rows: a stage's B is one copy
    BRows br;                 // rows of the activation operand (hi rows, then lo rows)
    int stages, stage_bytes;  // ring slots; bytes per slot
    int atoms;                // most atoms per stage (stages never cross a segment end)
    int hq, hkv;
    // L2 prefetch of the next GEMM's first weight atoms of this CTA's range (issued by the
    // producer once its own loads are all issued)
    const uint8_t* nwt;
    int n_ntiles, n_KB, n_atoms;       // n_atoms = 0: no prefetch
    float* partial;          // [grid][2] x ntok/16 chunks of [4][128] float4 (partial_f4)
    int* tile_cnt;           // [n_tiles], zero between launches
    int split_s;             // CTAs per tile of a whole-tile split (grid = n_tiles x split_s), else 0
    int* err;
    EpiArgs e;
};

#ifdef TC_TRACE
// Per-CTA timeline of the last launch of each GEMM kind (profiling builds only):
// [gid][cta][0 entry, 1 set-up done, 2 first stage ready, 3 last MMA issued,
//            4 last accumulator ready, 5 exit; split fix-up: 6 partials published,
//            7 all contributors published, 8 first own chunk done, 9 all own chunks done,
//            10 first own chunk's sums staged]
__device__ unsigned long long g_tc_trace[5][1024][12];
#define TC_STAMP(i) do { if (blockIdx.x < 1024) g_tc_trace[p.gid][blockIdx.x][i] = globaltimer_ns(); } while (0)
#else
#define TC_STAMP(i) ((void)0)
#endif

// The weights (A) of n consecutive K atoms kt .. kt + n - 1 of a tile: one bulk copy.
__device__ __forceinline__ void load_stage_a(const TcParams& p, int tile, int kt, int n, uint32_t a_dst, uint32_t fb,
                                             uint64_t pol) {
    bulk_g2s(a_dst, p.wt + ((size_t)tile * p.KB + kt) * TC_ATOM_A, (uint32_t)(n * TC_ATOM_A), fb, pol);
}

// The token rows (B) of the n K atoms kt .. kt + n - 1, already in the swizzled order the
// MMA reads (operand layout, epilogue.cuh): per atom the launch's ntok hi rows, then its
// ntok lo rows.  When the launch covers all rows of the pass, the atoms' blocks are
// contiguous in global memory as in shared memory and the stage's B is one bulk copy.
__device__ __forceinline__ void load_stage_b(const TcParams& p, int kt, int n, uint32_t b_dst, uint32_t fb,
                                             uint64_t pol) {
    const size_t blk = (size_t)p.x_rows * 128;                 // one atom's hi (or lo) rows
    const uint8_t* src = p.x + (size_t)kt * 2 * blk + (size_t)p.x_row0 * 128;
    const uint32_t rows_b = (uint32_t)p.br.rows * 128;
    if (p.x_whole) {
        bulk_g2s(b_dst, src, (uint32_t)n * 2 * rows_b, fb, pol);
        return;
    }
    for (int at = 0; at < n; ++at) {
        bulk_g2s(b_dst + (uint32_t)at * 2 * rows_b, src + (size_t)at * 2 * blk, rows_b, fb, pol);
        bulk_g2s(b_dst + (uint32_t)at * 2 * rows_b + rows_b, src + (size_t)at * 2 * blk + blk, rows_b, fb, pol);
    }
}

__global__ void __launch_bounds__(TC_THREADS, TC_CTAS_PER_SM) tc_gemm_kernel(const __grid_constant__ TcParams p) {
    extern __shared__ uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t full_bar[TC_MAX_STAGES], empty_bar[TC_MAX_STAGES];
    __shared__ __align__(8) uint64_t accf[2], acce[2], done_bar;
    __shared__ uint32_t tmem_sh;
    __shared__ int last_flag;
    __shared__ float inv_s[TC_MAX_NTOK];
    __shared__ float red_s[4][TC_CW];

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) TC_STAMP(0);
    const uint32_t base = (smem_u32(smem_raw) + 1023u) & ~1023u;
    float* xs = reinterpret_cast<float*>(smem_raw + (base - smem_u32(smem_raw)) + p.stages * p.stage_bytes);
    const int G = gridDim.x, cta = blockIdx.x;
    const long long T = (long long)p.n_tiles * p.KB;
    const long long s0 = range_start(T, G, cta), s1 = range_start(T, G, cta + 1);
    const int S = p.stages;
    // accumulator buffers of br.acc_stride columns: two while they fit the 512 TMEM columns
    const int acc_cols = p.br.acc_stride;
    const int nbuf = 2 * acc_cols <= 512 ? 2 : 1;
    const uint32_t ncols = (uint32_t)min(512, max(32, 1 << (32 - __clz(nbuf * acc_cols - 1))));

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(smem_u32(&full_bar[s]), 1);
            mbar_init(smem_u32(&empty_bar[s]), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(smem_u32(&accf[b]), 1);
            mbar_init(smem_u32(&acce[b]), 128);
        }
        mbar_init(smem_u32(&done_bar), 1);
        fence_barrier_init();
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                     :: "r"(smem_u32(&tmem_sh)), "r"(ncols) : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_sh;
    if (threadIdx.x == 0) TC_STAMP(1);
    pdl_launch_dependents();

    if (warp == 0) {
        if (lane == 0) {
            const uint64_t pw = policy_evict_first();
            const uint64_t px = policy_evict_last();
            // The first ring's worth of weight tiles does not depend on the previous kernel:
            // issue it before waiting for that kernel, then the activations.
            const uint32_t per_atom_tx = (uint32_t)(TC_ATOM_A + p.br.nb * TC_ATOM * 2);
            const uint32_t b_off = (uint32_t)(p.atoms * TC_ATOM_A);
            StageWalk w(s0, s1, p.KB, p.atoms);
            long long i = 0;
            long long seg0 = s0;
            for (; i < S && !w.done(); ++i) {
                int n, tile, kt;
                bool sf, sl;
                w.cur(n, tile, kt, sf, sl, seg0);
                const uint32_t fb = smem_u32(&full_bar[i]);
                mbar_arrive_expect_tx(fb, per_atom_tx * n);
                const uint32_t a_dst = base + (uint32_t)i * p.stage_bytes;
                load_stage_a(p, tile, kt, n, a_dst, fb, pw);
                w.g += n;
                if (sl) seg0 = w.g;
            }
            pdl_wait();
            {
                StageWalk w2(s0, s1, p.KB, p.atoms);
                long long sg = s0;
                for (long long j = 0; j < i; ++j) {
                    int n, tile, kt;
                    bool sf, sl;
                    w2.cur(n, tile, kt, sf, sl, sg);
                    load_stage_b(p, kt, n, base + (uint32_t)j * p.stage_bytes + b_off, smem_u32(&full_bar[j]), px);
                    w2.g += n;
                    if (sl) sg = w2.g;
                }
            }
            for (; !w.done(); ++i) {
                int n, tile, kt;
                bool sf, sl;
                w.cur(n, tile, kt, sf, sl, seg0);
                const int s = (int)(i % S);
                if (!mbar_wait(smem_u32(&empty_bar[s]), (uint32_t)(((i / S) & 1) ^ 1))) {
                    atomicExch(p.err, SPEC_E_TIMEOUT);
                    break;
                }
                const uint32_t fb = smem_u32(&full_bar[s]);
                mbar_arrive_expect_tx(fb, per_atom_tx * n);
                const uint32_t a_dst = base + (uint32_t)s * p.stage_bytes;
                load_stage_a(p, tile, kt, n, a_dst, fb, pw);
                load_stage_b(p, kt, n, a_dst + b_off, fb, px);
                w.g += n;
                if (sl) seg0 = w.g;
            }
            if (p.n_atoms > 0) {
                // warm L2 with the first atoms this CTA index will stream in the next GEMM,
                // so HBM keeps working while the kernels in between run
                // (the atoms of a range are contiguous in the tile-major layout)
                const long long T2 = (long long)p.n_ntiles * p.n_KB;
                const long long a0 = range_start(T2, G, cta);
                const long long a1 = min(range_start(T2, G, cta + 1), a0 + p.n_atoms);
                if (a1 > a0) bulk_prefetch_l2(p.nwt + (size_t)a0 * TC_ATOM_A, (uint32_t)((a1 - a0) * TC_ATOM_A));
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // one MMA of N = br.nb while that fits an instruction, else two (rows [0, 256)
            // and [256, nb) of B into the matching accumulator columns)
            const int nb = p.br.nb;
            const bool one = nb <= TC_MMA_NMAX;
            const uint32_t idesc = idesc_bf16(one ? nb : TC_MMA_NMAX);
            const uint32_t idesc1 = one ? 0u : idesc_bf16(nb - TC_MMA_NMAX);
            const uint64_t a_step = TC_ATOM_A >> 4, b_step = (uint64_t)(nb * TC_ATOM * 2) >> 4;
            const uint32_t b_off = (uint32_t)(p.atoms * TC_ATOM_A);
            StageWalk w(s0, s1, p.KB, p.atoms);
            long long i = 0, seg0 = s0;
            int si = 0;
            bool ok = true;
            uint32_t d_tmem = tmem;
            while (ok && !w.done()) {
                int n, tile, kt;
                bool sf, sl;
                w.cur(n, tile, kt, sf, sl, seg0);
                const int buf = si % nbuf;
                if (sf) {
                    if (!mbar_wait(smem_u32(&acce[buf]), (uint32_t)(((si / nbuf) & 1) ^ 1))) {
                        atomicExch(p.err, SPEC_E_TIMEOUT);
                        break;
                    }
                    tc_fence_after();
                    d_tmem = tmem + (uint32_t)(buf * acc_cols);
                }
                const int s = (int)(i % S);
                if (!mbar_wait(smem_u32(&full_bar[s]), (uint32_t)((i / S) & 1))) {
                    atomicExch(p.err, SPEC_E_TIMEOUT);
                    ok = false;
                    break;
                }
                if (i == 0) TC_STAMP(2);
                tc_fence_after();
                const uint32_t a_addr = base + (uint32_t)s * p.stage_bytes;
                // descriptors of atom 0; each further atom is TC_ATOM_A (A) and nb rows of 128 B
                // (B) further on (the address field counts 16-byte units)
                const uint64_t ad0 = smem_desc_sw128(a_addr);
                const uint64_t bd0 = smem_desc_sw128(a_addr + b_off);
                if (one) {
                    for (int at = 0; at < n; ++at)
                        mma_bf16_atom(d_tmem, ad0 + (uint64_t)at * a_step, bd0 + (uint64_t)at * b_step, idesc,
                                      (!sf || at > 0) ? 1u : 0u);
                } else {
                    // B rows [0, 256) into columns [0, 256), rows [256, nb) into [256, nb)
                    for (int at = 0; at < n; ++at) {
                        const uint64_t ad = ad0 + (uint64_t)at * a_step, bd = bd0 + (uint64_t)at * b_step;
                        mma_bf16_atom(d_tmem, ad, bd, idesc, (!sf || at > 0) ? 1u : 0u);
                        mma_bf16_atom(d_tmem + TC_MMA_NMAX, ad, bd + (uint64_t)((TC_MMA_NMAX * TC_ATOM * 2) >> 4),
                                      idesc1, (!sf || at > 0) ? 1u : 0u);
                    }
                }
                mma_commit(smem_u32(&empty_bar[s]));
                ++i;
                w.g += n;
                if (sl) {
                    mma_commit(smem_u32(&accf[buf]));
                    ++si;
                    seg0 = w.g;
                }
            }
            TC_STAMP(3);
            // make sure no MMA is still writing tensor memory before it is freed
            mma_commit(smem_u32(&done_bar));
            mbar_wait(smem_u32(&done_bar), 0);
        }
    } else {
        pdl_wait();     // outputs of the previous kernel may still be read by it until then
        const int q = warp & 3;
        const int row = q * 32 + lane;
        const int etid = threadIdx.x - 64;
        if (p.e.ssq_in != nullptr) {
            // 1/rms of every token of the launch, its tiles' sums of squares added in order
            for (int m = etid; m < p.M; m += 128) {
                const float* src = p.e.ssq_in + p.e.ssq_row0 + m;
                float ss = 0.0f;
                for (int t = 0; t < p.e.n_ssq; ++t) ss += __ldcg(src + (size_t)t * p.e.ssq_ld);
                inv_s[m] = 1.0f / sqrtf(ss / p.e.norm_d + p.e.eps);
            }
            epi_bar();
        }
        int si = 0;
        long long g = s0;
        while (g < s1) {
            const int tile = (int)(g / p.KB);
            const long long tile_k0 = (long long)tile * p.KB;
            const long long seg_end = min(s1, tile_k0 + p.KB);
            const bool full_tile = (g == tile_k0) && (seg_end == tile_k0 + p.KB);
            const int buf = si % nbuf;
            EpiPre pre;
            epi_preload(p.M, p.e, tile, etid, pre);
            // contributors of a split tile (CTA order), found before the accumulator is ready
            int c_lo = cta, c_hi = cta, wc_lo = 0;
            if (!full_tile) {
                c_lo = owner_cta(T, G, tile_k0);
                c_hi = owner_cta(T, G, tile_k0 + p.KB - 1);
                wc_lo = (range_start(T, G, c_lo) >= tile_k0) ? 0 : 1;
            }
            const bool okw = mbar_wait(smem_u32(&accf[buf]), (uint32_t)((si / nbuf) & 1));
            if (epi_any(okw ? 0 : 1)) {
                if (etid == 0) atomicExch(p.err, SPEC_E_TIMEOUT);
                break;
            }
            tc_fence_after();
            if (etid == 0 && seg_end == s1) TC_STAMP(4);
            const uint32_t taddr = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(buf * acc_cols);
            if (full_tile) {
                for (int c0 = 0; c0 < p.ntok; c0 += TC_CW) {
                    float v[16];
                    acc_ld16(taddr, c0, p.br.lo_col, v);
                    if (c0 + TC_CW >= p.ntok) {
                        tc_fence_before();
                        mbar_arrive(smem_u32(&acce[buf]));
                    }
#pragma unroll
                    for (int j = 0; j < 16; ++j) xs[row * TC_XPITCH + j] = v[j];
                    epi_bar();
                    epi_chunk(p.gid, p.M, p.e, xs, inv_s, red_s, tile, c0, etid, c0 == 0 ? &pre : nullptr);
                    epi_bar();
                }
            } else if (p.split_s > 1 && p.ntok > TC_CW) {
                // Whole-tile split of several 16-token chunks: each of the s contributors
                // finalizes the chunks ch with ch % s == its index.  It publishes its sums of
                // the other chunks, waits (bounded) until all s have published, then adds the
                // tile's sums of its own chunks in contributor order (its own from tensor
                // memory): the additions a single finalizer makes, spread over s CTAs.
                const int s = p.split_s, me = cta - c_lo;
                for (int c0 = 0, ch = 0; c0 < p.ntok; c0 += TC_CW, ++ch) {
                    if (ch % s == me) continue;
                    float v[16];
                    acc_ld16(taddr, c0, p.br.lo_col, v);
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        *partial_f4(p.partial, cta, 0, p.ntok, c0, j, row) =
                            make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
                }
                __threadfence();
                epi_bar();
                if (etid == 0) {
                    atomicAdd(p.tile_cnt + tile, 1);
                    TC_STAMP(6);
                    last_flag = wait_count_at_least(p.tile_cnt + tile, s) ? 1 : 0;
                    TC_STAMP(7);
                }
                epi_bar();
                if (!last_flag) {
                    if (etid == 0) atomicExch(p.err, SPEC_E_TIMEOUT);
                } else {
                    __threadfence();
                    for (int c0 = me * TC_CW; c0 < p.ntok; c0 += s * TC_CW) {
                        float acc[16];
#pragma unroll
                        for (int j = 0; j < 16; ++j) acc[j] = 0.0f;
                        for (int cc = c_lo; cc <= c_hi; ++cc) {
                            float v[16];
                            if (cc == cta) {
                                acc_ld16(taddr, c0, p.br.lo_col, v);
                            } else {
#pragma unroll
                                for (int j = 0; j < 4; ++j) {
                                    const float4 t4 = __ldcg(partial_f4(p.partial, cc, 0, p.ntok, c0, j, row));
                                    v[4 * j] = t4.x; v[4 * j + 1] = t4.y; v[4 * j + 2] = t4.z; v[4 * j + 3] = t4.w;
                                }
                            }
#pragma unroll
                            for (int j = 0; j < 16; ++j) acc[j] += v[j];
                        }
#pragma unroll
                        for (int j = 0; j < 16; ++j) xs[row * TC_XPITCH + j] = acc[j];
                        epi_bar();
                        if (etid == 0 && c0 == me * TC_CW) TC_STAMP(10);
                        epi_chunk(p.gid, p.M, p.e, xs, inv_s, red_s, tile, c0, etid, c0 == 0 ? &pre : nullptr);
                        epi_bar();
                        if (etid == 0 && c0 == me * TC_CW) TC_STAMP(8);
                    }
                }
                if (etid == 0) TC_STAMP(9);
                tc_fence_before();
                mbar_arrive(smem_u32(&acce[buf]));
                // every contributor has passed its wait once all s have arrived a second time
                if (etid == 0 && atomicAdd(p.tile_cnt + tile, 1) == 2 * s - 1) p.tile_cnt[tile] = 0;
            } else {
                const int which = (s0 >= tile_k0) ? 0 : 1;
                for (int c0 = 0; c0 < p.ntok; c0 += TC_CW) {
                    float v[16];
                    acc_ld16(taddr, c0, p.br.lo_col, v);
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        *partial_f4(p.partial, cta, which, p.ntok, c0, j, row) =
                            make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
                }
                tc_fence_before();
                mbar_arrive(smem_u32(&acce[buf]));
                __threadfence();
                epi_bar();
                if (etid == 0) {
                    const int prev = atomicAdd(p.tile_cnt + tile, 1);
                    last_flag = (prev == c_hi - c_lo) ? 1 : 0;
                }
                epi_bar();
                if (last_flag) {
                    __threadfence();
                    // contributors in CTA order; the first one's slot is 1 unless its range
                    // starts exactly at the tile, every later one starts inside the tile
                    for (int c0 = 0; c0 < p.ntok; c0 += TC_CW) {
                        float acc[16];
#pragma unroll
                        for (int j = 0; j < 16; ++j) acc[j] = 0.0f;
                        for (int cb = c_lo; cb <= c_hi; cb += 4) {
                            float4 part[4][4];
#pragma unroll
                            for (int u = 0; u < 4; ++u) {
                                const int cc = cb + u;
                                if (cc <= c_hi) {
                                    const int wc = cc == c_lo ? wc_lo : 0;
#pragma unroll
                                    for (int j = 0; j < 4; ++j)
                                        part[u][j] = __ldcg(partial_f4(p.partial, cc, wc, p.ntok, c0, j, row));
                                }
                            }
#pragma unroll
                            for (int u = 0; u < 4; ++u) {
                                if (cb + u <= c_hi) {
#pragma unroll
                                    for (int j = 0; j < 4; ++j) {
                                        acc[4 * j] += part[u][j].x; acc[4 * j + 1] += part[u][j].y;
                                        acc[4 * j + 2] += part[u][j].z; acc[4 * j + 3] += part[u][j].w;
                                    }
                                }
                            }
                        }
#pragma unroll
                        for (int j = 0; j < 16; ++j) xs[row * TC_XPITCH + j] = acc[j];
                        epi_bar();
                        epi_chunk(p.gid, p.M, p.e, xs, inv_s, red_s, tile, c0, etid, c0 == 0 ? &pre : nullptr);
                        epi_bar();
                    }
                    if (etid == 0) p.tile_cnt[tile] = 0;
                }
            }
            g = seg_end;
            ++si;
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (threadIdx.x == 0) TC_STAMP(5);
    if (warp == 1)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" :: "r"(tmem), "r"(ncols) : "memory");
}

// ---- host side ------------------------------------------------------------------------------

struct TcGemm {
    uint8_t* wt = nullptr;                 // tile-major weights of every GEMM
    std::vector<size_t> off;               // byte offset of GEMM (layer, gid) at 4 * layer + gid; lm_head last
    float* partial = nullptr;
    int* tile_cnt = nullptr;
    int* err = nullptr;
    int n_tile_cnt = 0;
    int grid = 0;
};

bool tc_supported(const Ctx& c) {
    const spec_model_cfg& m = c.cfg;
    return m.dtype == SPEC_BF16 && m.head_dim == 128 && m.d_model % 128 == 0 && m.vocab % 128 == 0 &&
           m.ffn_dim % 64 == 0 && (m.n_q_heads * m.head_dim) % 64 == 0;
}

// Weight bytes, tiles and K atoms per tile of GEMM `gid` (one layer; lm_head for GEMM_LM).
static void gemm_shape(const spec_model_cfg& m, int gid, int& n_tiles, int& KB) {
    const int d = m.d_model, qd = m.n_q_heads * m.head_dim, F = m.ffn_dim;
    switch (gid) {
    case GEMM_QKV: n_tiles = m.n_q_heads + 2 * m.n_kv_heads; KB = d / TC_ATOM; break;
    case GEMM_O: n_tiles = d / TC_BM; KB = qd / TC_ATOM; break;
    case GEMM_GU: n_tiles = F / 64; KB = d / TC_ATOM; break;
    case GEMM_DOWN: n_tiles = d / TC_BM; KB = F / TC_ATOM; break;
    default: n_tiles = m.vocab / TC_BM; KB = d / TC_ATOM; break;
    }
}

// Tile-major copy of one weight GEMM (see the file header): destination 16-byte chunk i =
// ((atom * 2 + half) * 64 + row) * 8 + chunk, atom = tile * KB + k, holds the source chunk
// chunk ^ (row % 8) of that row (the 128-byte swizzle of a K-major operand row).
struct RelayoutArgs {
    const __nv_bfloat16* src[3];   // the GEMM's weight matrices, row-major [rows][ld]
    int gid, hq, hkv, KB, ld;
    size_t n_chunks;
    uint8_t* dst;
};

__global__ void tc_relayout_kernel(const RelayoutArgs a) {
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < a.n_chunks; i += (size_t)gridDim.x * blockDim.x) {
        const int cd = (int)(i & 7);
        const int r = (int)((i >> 3) & 63);
        const int h = (int)((i >> 9) & 1);
        const size_t atom = i >> 10;
        const int tile = (int)(atom / a.KB), k = (int)(atom - (size_t)tile * a.KB);
        int mat, row0;
        tile_half_rows(a.gid, a.hq, a.hkv, tile, h, mat, row0);
        const int c = cd ^ (r & 7);
        *reinterpret_cast<uint4*>(a.dst + i * 16) =
            *reinterpret_cast<const uint4*>(a.src[mat] + (size_t)(row0 + r) * a.ld + (size_t)k * TC_ATOM + c * 8);
    }
}

int tc_create(Ctx& c) {
    c.use_tc = false;
    if (!tc_supported(c)) return SPEC_OK;
    const spec_model_cfg& m = c.cfg;
    TcGemm* t = new TcGemm();
    const uint64_t d = m.d_model, qd = (uint64_t)m.n_q_heads * m.head_dim, kvd = (uint64_t)m.n_kv_heads * m.head_dim,
                   F = m.ffn_dim, V = m.vocab;
    int rc = SPEC_OK;
    // tile-major weights: offsets of (layer, gid) at 4 * layer + gid, lm_head last
    const int L = m.n_layers;
    t->off.resize((size_t)4 * L + 1);
    size_t total = 0;
    for (int i = 0; i <= 4 * L; ++i) {
        int nt, kb;
        gemm_shape(m, i == 4 * L ? GEMM_LM : i % 4, nt, kb);
        t->off[i] = total;
        total += (size_t)nt * kb * TC_ATOM_A;
    }
    {
        void* w = nullptr;
        if (cudaMalloc(&w, total) != cudaSuccess) {
            delete t;
            return set_error(SPEC_E_NOMEM, "tile-major weight copy (%zu bytes) allocation failed", total);
        }
        t->wt = static_cast<uint8_t*>(w);
    }
    for (int i = 0; i <= 4 * L; ++i) {
        const int gid = i == 4 * L ? GEMM_LM : i % 4;
        RelayoutArgs a{};
        int nt, kb;
        gemm_shape(m, gid, nt, kb);
        a.gid = gid; a.hq = m.n_q_heads; a.hkv = m.n_kv_heads; a.KB = kb; a.ld = kb * TC_ATOM;
        a.n_chunks = (size_t)nt * kb * (TC_ATOM_A / 16);
        a.dst = t->wt + t->off[i];
        using bf = __nv_bfloat16;
        if (gid == GEMM_LM) {
            a.src[0] = static_cast<const bf*>(c.w.lm_head);
        } else {
            const LayerWeights& lw = c.w.layers[i / 4];
            switch (gid) {
            case GEMM_QKV:
                a.src[0] = static_cast<const bf*>(lw.wq); a.src[1] = static_cast<const bf*>(lw.wk);
                a.src[2] = static_cast<const bf*>(lw.wv);
                break;
            case GEMM_O: a.src[0] = static_cast<const bf*>(lw.wo); break;
            case GEMM_GU: a.src[0] = static_cast<const bf*>(lw.wg); a.src[1] = static_cast<const bf*>(lw.wu); break;
            default: a.src[0] = static_cast<const bf*>(lw.wd); break;
            }
        }
        tc_relayout_kernel<<<4 * c.num_sms, 256, 0, c.stream>>>(a);
    }
    if (cudaGetLastError() != cudaSuccess || cudaStreamSynchronize(c.stream) != cudaSuccess)
        rc = set_error(SPEC_E_CUDA, "weight re-layout failed");
    t->grid = c.num_sms;
    const int max_tiles = (int)std::max<uint64_t>({V / 128, F / 64, d / 128, qd / 128 + 2 * kvd / 128});
    if (rc == SPEC_OK) {
        void *a = nullptr, *b = nullptr, *e = nullptr;
        if (cudaMalloc(&a, sizeof(float) * (size_t)t->grid * 2 * TC_BM * ((c.Mmax + 15) & ~15)) != cudaSuccess ||
            cudaMalloc(&b, sizeof(int) * (size_t)max_tiles) != cudaSuccess ||
            cudaMalloc(&e, sizeof(int)) != cudaSuccess) {
            rc = set_error(SPEC_E_NOMEM, "tensor-core GEMM workspace allocation failed");
        } else {
            cudaMemset(b, 0, sizeof(int) * (size_t)max_tiles);
            cudaMemset(e, 0, sizeof(int));
        }
        t->partial = static_cast<float*>(a);
        t->tile_cnt = static_cast<int*>(b);
        t->n_tile_cnt = max_tiles;
        t->err = static_cast<int*>(e);
    }
    if (rc == SPEC_OK &&
        cudaFuncSetAttribute(tc_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, TC_SMEM_MAX) != cudaSuccess)
        rc = set_error(SPEC_E_CUDA, "cudaFuncSetAttribute(tc_gemm_kernel)");
    if (rc != SPEC_OK) {
        if (t->wt) cudaFree(t->wt);
        if (t->partial) cudaFree(t->partial);
        if (t->tile_cnt) cudaFree(t->tile_cnt);
        if (t->err) cudaFree(t->err);
        delete t;
        return rc;
    }
    c.tc = t;
    c.use_tc = true;
    c.split = true;
    return SPEC_OK;
}

void tc_destroy(Ctx& c) {
    if (!c.tc) return;
    cudaFree(c.tc->wt);
    cudaFree(c.tc->partial);
    cudaFree(c.tc->tile_cnt);
    cudaFree(c.tc->err);
    delete c.tc;
    c.tc = nullptr;
    c.use_tc = false;
    c.split = false;
}

#ifdef TC_TRACE
extern "C" int spec_debug_tc_trace(unsigned long long* out) {
    return cudaMemcpyFromSymbol(out, g_tc_trace, sizeof(g_tc_trace)) == cudaSuccess ? 0 : -6;
}
#endif

// One bounded wait, by the GEMM kernel's wait helper, on an mbarrier that nothing
// completes: no copy is in flight and no tensor memory is held, so when the budget runs out
// the thread records SPEC_E_TIMEOUT in the context's device status word, exactly as a GEMM
// wait that gave up would, and the kernel returns.
__global__ void wait_probe_kernel(int* err, unsigned long long budget_ns) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x != 0) return;
    mbar_init(smem_u32(&bar), 1);
    fence_barrier_init();
    if (!mbar_wait(smem_u32(&bar), 0, budget_ns)) atomicExch(err, SPEC_E_TIMEOUT);
}

int tc_wait_probe(Ctx& c, int budget_ms) {
    if (!c.tc) return set_error(SPEC_E_STATE, "no tensor-core GEMM plan (bf16 model with all weights loaded)");
    wait_probe_kernel<<<1, 32, 0, c.stream>>>(c.tc->err, (unsigned long long)budget_ms * 1000000ull);
    const cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? SPEC_OK : set_error(SPEC_E_CUDA, "wait_probe_kernel launch: %s", cudaGetErrorString(e));
}

int* tc_error_ptr(Ctx& c) { return c.tc ? c.tc->err : nullptr; }

int tc_error_word(Ctx& c, int* out) {
    if (!c.tc) { *out = 0; return SPEC_OK; }
    return cudaMemcpy(out, c.tc->err, sizeof(int), cudaMemcpyDeviceToHost) == cudaSuccess ? SPEC_OK : SPEC_E_CUDA;
}

// CTAs of a GEMM of n_tiles output tiles on `sms` SMs.  With fewer tiles than SMs, the grid
// is a whole number s of CTAs per tile (each CTA one s-th of a tile's K atoms, every tile
// finished by exactly s contributors, whose partial sums the last one reads in one batch)
// as long as that keeps at least min_fill percent of the SMs streaming; otherwise one CTA
// per SM with the (tile, atom) space cut into equal ranges across tile boundaries.  The
// choice depends only on the weight shape and the SM count, so a token's result bits do
// not depend on how many tokens share the launch.
static int gemm_grid(int n_tiles, int sms, int min_fill, int max_split) {
    if (n_tiles >= sms) return sms;
    if (max_split > 0) return n_tiles * std::min(max_split, sms / n_tiles);
    const int g = n_tiles * (sms / n_tiles);
    return 100 * g >= min_fill * sms ? g : sms;
}

static int tc_gemm_launch(Ctx& c, int gid, int layer, int x_row0, int M, int pass_M, const EpiArgs& e,
                          cudaStream_t st) {
    TcGemm* t = c.tc;
    const spec_model_cfg& m = c.cfg;
    if (M < 1 || M > TC_MAX_NTOK) return set_error(SPEC_E_RANGE, "GEMM with M=%d tokens (max %d)", M, TC_MAX_NTOK);
    TcParams p{};
    const int d = m.d_model, qd = m.n_q_heads * m.head_dim, F = m.ffn_dim;
    int Kdim = d;
    p.x = static_cast<const uint8_t*>(c.Xn);
    int KB = 0;
    gemm_shape(m, gid, p.n_tiles, KB);
    p.wt = t->wt + t->off[gid == GEMM_LM ? (size_t)4 * m.n_layers : (size_t)4 * layer + gid];
    if (gid == GEMM_O) {
        Kdim = qd;
        p.x = static_cast<const uint8_t*>(c.O);
    } else if (gid == GEMM_DOWN) {
        Kdim = F;
        p.x = static_cast<const uint8_t*>(c.H);
    }
    p.x_rows = act_rows(pass_M);
    p.x_row0 = x_row0;
    p.gid = gid;
    p.KB = Kdim / TC_ATOM;
    p.ntok = (M + 15) & ~15;
    p.M = M;
    p.br = b_rows(M);
    if (x_row0 % 8 != 0 || x_row0 + p.br.rows > p.x_rows)
        return set_error(SPEC_E_RANGE, "GEMM rows [%d, %d) outside the pass's %d operand rows", x_row0,
                         x_row0 + p.br.rows, p.x_rows);
    p.x_whole = (x_row0 == 0 && p.br.rows == p.x_rows) ? 1 : 0;
    // the widest stage (most K atoms) that still leaves TC_MIN_STAGES ring slots; the
    // stream-K split is in atoms, so this choice changes no result bit
    const int budget = TC_SMEM_MAX - 1024 - TC_XBYTES;
    const int per_atom = TC_ATOM_A + p.br.nb * TC_ATOM * 2;
    p.atoms = 1;
    for (int a = TC_MAX_ATOMS; a > 1; --a)
        if (budget / (a * per_atom) >= TC_MIN_STAGES) { p.atoms = a; break; }
    p.stage_bytes = p.atoms * per_atom;
    p.stages = std::min(TC_MAX_STAGES, budget / p.stage_bytes);
    if (p.stages < 2) return set_error(SPEC_E_RANGE, "GEMM stage does not fit in shared memory");
    p.hq = m.n_q_heads;
    p.hkv = m.n_kv_heads;
    p.partial = t->partial;
    p.tile_cnt = t->tile_cnt;
    p.err = t->err;
    p.e = e;
    // the next GEMM of the pass (QKV -> O -> gate/up -> down -> next layer's QKV or lm_head)
    p.n_atoms = 0;
    if (c.l2_prefetch_atoms > 0 && gid != GEMM_LM) {
        int ngid = gid + 1, nlayer = layer;
        if (gid == GEMM_DOWN) {
            ngid = layer + 1 < m.n_layers ? GEMM_QKV : GEMM_LM;
            nlayer = layer + 1 < m.n_layers ? layer + 1 : -1;
        }
        gemm_shape(m, ngid, p.n_ntiles, p.n_KB);
        p.nwt = t->wt + t->off[ngid == GEMM_LM ? (size_t)4 * m.n_layers : (size_t)4 * nlayer + ngid];
        p.n_atoms = c.l2_prefetch_atoms;
    }
    const long long T = (long long)p.n_tiles * p.KB;
    const int grid = (int)std::min<long long>(gemm_grid(p.n_tiles, t->grid, c.gemm_min_fill, c.gemm_max_split), T);
    // a whole number of CTAs per tile: CTA tile * s + i takes the i-th s-th of the tile's K
    p.split_s = (p.n_tiles < grid && grid % p.n_tiles == 0) ? grid / p.n_tiles : 0;
    const size_t smem = 1024 + (size_t)p.stages * p.stage_bytes + TC_XBYTES;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(TC_THREADS);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = c.use_pdl ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t err = cudaLaunchKernelEx(&cfg, tc_gemm_kernel, p);
    if (err != cudaSuccess) return set_error(SPEC_E_CUDA, "tc_gemm_kernel launch: %s", cudaGetErrorString(err));
    return 1;
}

// More tokens than one launch holds run as launches over equal chunks of whole 16-token
// groups (each streams the weights again); every token sees the same arithmetic as in a
// single launch, so the results do not depend on the split.
int tc_gemm(Ctx& c, int gid, int layer, int x_row0, int M, int pass_M, const EpiArgs& e, cudaStream_t st) {
    if (M <= TC_MAX_NTOK) return tc_gemm_launch(c, gid, layer, x_row0, M, pass_M, e, st);
    const int n = (M + TC_MAX_NTOK - 1) / TC_MAX_NTOK;
    int launched = 0, m0 = 0;
    for (int i = 0; i < n; ++i) {
        const int rest = M - m0, parts = n - i;
        const int chunk = std::min(rest, (((rest + parts - 1) / parts) + 15) & ~15);
        EpiArgs ec = e;
        ec.M = chunk;
        ec.m0 = e.m0 + m0;
        if (ec.ssq_in) ec.ssq_row0 = e.ssq_row0 + m0;
        const int r = tc_gemm_launch(c, gid, layer, x_row0 + m0, chunk, pass_M, ec, st);
        if (r < 0) return r;
        launched += r;
        m0 += chunk;
    }
    return launched;
}

}  // namespace sv
