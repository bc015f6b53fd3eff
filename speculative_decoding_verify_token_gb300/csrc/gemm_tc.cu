// Skinny bf16 GEMM of the verify pass on the 5th-generation tensor cores (tcgen05).
//
// Y[m][n] = sum_k X[m][k] W[n][k] with M = B*(K+1) tokens (<= 256) and weight matrices of
// 6-150 k rows: the work is streaming the weights through HBM ("most of that pass is spent
// moving weights through memory", "Speculative Decoding on Apple Silicon...", section
// "How speculative decoding works").  Design:
//  * swap-AB: a 128-row weight tile is the A operand, the tokens are the N dimension
//    (16..256); the fp32 accumulator [128 x N] lives in tensor memory;
//  * operands arrive by TMA (cp.async.bulk.tensor, 128-byte swizzle) into an mbarrier ring
//    of up to 8 stages of 64 k-elements; weights are loaded evict-first, activations
//    evict-last (every CTA re-reads them);
//  * warp roles: warp 0 = TMA producer, warp 1 = tcgen05.mma issuer (one thread) and TMEM
//    owner, warps 2-5 = epilogue (tcgen05.ld of the 4 lane quarters);
//  * persistent stream-K: the (tile, k-block) space is cut into one contiguous range per
//    CTA; a tile shared by several CTAs is finished by the last one to arrive (atomic
//    ticket, no spin-wait), which adds the partial sums in CTA order.  The split depends
//    only on the weight shape and the SM count, so a token's outputs are bit-identical for
//    every M (a decode step and a verify pass agree exactly);
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
#define TC_MIN_STAGES 3         // fewest pipeline stages a launch may use
#endif
#ifndef TC_CTAS_PER_SM
#define TC_CTAS_PER_SM 1        // resident GEMM CTAs per SM (shared memory split between them)
#endif
// dynamic bytes per CTA: with one CTA per SM, three stages of four atoms at 16 tokens plus
// the staging tile and the alignment slack, leaving 1.5 KB of the 227 KB for static data
constexpr int TC_SMEM_MAX = TC_CTAS_PER_SM == 1 ? 230912 : 110 * 1024;

struct TcParams {
    CUtensorMap wmap[3];
    CUtensorMap xmap;
    int gid;
    int n_tiles, KB;          // tiles; K atoms per tile (the stream-K unit)
    int ntok, M, x_row0;      // ntok = M rounded up to 16 (stride of the partial sums)
    BRows br;                 // rows of the activation operand (split activations)
    int stages, stage_bytes;  // ring slots; bytes per slot
    int atoms;                // most atoms per stage (stages never cross a segment end)
    int hq, hkv;
    // L2 prefetch of the next GEMM's first weight atoms of this CTA's range (issued by the
    // producer once its own loads are all issued)
    CUtensorMap nwmap[3];
    int ngid, n_ntiles, n_KB, n_atoms;       // n_atoms = 0: no prefetch
    float* partial;          // [grid][2] x ntok/16 chunks of [4][128] float4 (partial_f4)
    int* tile_cnt;           // [n_tiles], zero between launches
    int* err;
    EpiArgs e;
};

#ifdef TC_TRACE
// Per-CTA timeline of the last launch of each GEMM kind (profiling builds only):
// [gid][cta][0 entry, 1 set-up done, 2 first stage ready, 3 last MMA issued,
//            4 last accumulator ready, 5 exit]
__device__ unsigned long long g_tc_trace[5][1024][6];
#define TC_STAMP(i) g_tc_trace[p.gid][blockIdx.x][i] = globaltimer_ns()
#else
#define TC_STAMP(i) ((void)0)
#endif

__device__ __forceinline__ void tile_rows(const TcParams& p, int tile, const CUtensorMap*& m0, int& r0,
                                          const CUtensorMap*& m1, int& r1) {
    tile_rows_of(p.gid, p.wmap, p.hq, p.hkv, tile, m0, r0, m1, r1);
}

// One K atom of a stage: the tile's 128 weight rows as two 64-row boxes (A) and the token
// rows in boxes of 16 (B), at K coordinate kc.
__device__ __forceinline__ void load_atom_a(const TcParams& p, int tile, int kc, uint32_t a_dst, uint32_t fb,
                                            uint64_t pol) {
    const CUtensorMap *m0, *m1;
    int r0, r1;
    tile_rows(p, tile, m0, r0, m1, r1);
    tma_load_2d(a_dst, m0, kc, r0, fb, pol);
    tma_load_2d(a_dst + TC_ATOM_A / 2, m1, kc, r1, fb, pol);
}

__device__ __forceinline__ void load_atom_b(const TcParams& p, int kc, uint32_t b_dst, uint32_t fb, uint64_t pol) {
    for (int t = 0; t < p.br.nr0 / 16; ++t) tma_load_2d(b_dst + t * 2048, &p.xmap, kc, p.br.b_row0 + t * 16, fb, pol);
    if (p.br.b_row1 >= 0)
        for (int t = 0; t < (p.br.nb - p.br.nr0) / 16; ++t)
            tma_load_2d(b_dst + (p.br.nr0 + t * 16) * 128, &p.xmap, kc, p.br.b_row1 + t * 16, fb, pol);
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
        asm volatile("prefetch.tensormap [%0];" :: "l"(reinterpret_cast<uint64_t>(&p.wmap[0])) : "memory");
        asm volatile("prefetch.tensormap [%0];" :: "l"(reinterpret_cast<uint64_t>(&p.xmap)) : "memory");
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
                for (int at = 0; at < n; ++at) load_atom_a(p, tile, (kt + at) * TC_ATOM, a_dst + at * TC_ATOM_A, fb, pw);
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
                    const uint32_t b_dst = base + (uint32_t)j * p.stage_bytes + b_off;
                    for (int at = 0; at < n; ++at)
                        load_atom_b(p, (kt + at) * TC_ATOM, b_dst + at * p.br.nb * TC_ATOM * 2, smem_u32(&full_bar[j]),
                                    px);
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
                for (int at = 0; at < n; ++at) {
                    load_atom_a(p, tile, (kt + at) * TC_ATOM, a_dst + at * TC_ATOM_A, fb, pw);
                    load_atom_b(p, (kt + at) * TC_ATOM, a_dst + b_off + at * p.br.nb * TC_ATOM * 2, fb, px);
                }
                w.g += n;
                if (sl) seg0 = w.g;
            }
            if (p.n_atoms > 0) {
                // warm L2 with the first atoms this CTA index will stream in the next GEMM,
                // so HBM keeps working while the kernels in between run
                const long long T2 = (long long)p.n_ntiles * p.n_KB;
                const long long a0 = range_start(T2, G, cta);
                const long long a1 = min(range_start(T2, G, cta + 1), a0 + p.n_atoms);
                for (long long g = a0; g < a1; ++g) {
                    const int tile = (int)(g / p.n_KB), kt = (int)(g % p.n_KB);
                    const CUtensorMap *m0, *m1;
                    int r0, r1;
                    tile_rows_of(p.ngid, p.nwmap, p.hq, p.hkv, tile, m0, r0, m1, r1);
                    tma_prefetch_l2(m0, kt * TC_ATOM, r0);
                    tma_prefetch_l2(m1, kt * TC_ATOM, r1);
                }
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
                    epi_chunk(p.gid, p.M, p.e, xs, inv_s, red_s, tile, c0, etid);
                    epi_bar();
                }
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
                const int c_lo = owner_cta(T, G, tile_k0);
                const int c_hi = owner_cta(T, G, tile_k0 + p.KB - 1);
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
                    const int wc_lo = (range_start(T, G, c_lo) >= tile_k0) ? 0 : 1;
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
                        epi_chunk(p.gid, p.M, p.e, xs, inv_s, red_s, tile, c0, etid);
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

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

struct TcLayerMaps {
    CUtensorMap q, k, v, o, g, u, d;
};

struct TcGemm {
    std::vector<TcLayerMaps> layers;
    CUtensorMap lm;
    CUtensorMap xn, xo, xh;
    float* partial = nullptr;
    int* tile_cnt = nullptr;
    int* err = nullptr;
    int n_tile_cnt = 0;
    int grid = 0;
};

static EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static bool tried = false;
    if (!tried) {
        tried = true;
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(f);
    }
    return fn;
}

// bf16 row-major [rows][cols], box = 64 columns (128 B, the swizzle span) x box_rows rows.
static int make_map(CUtensorMap* m, const void* ptr, uint64_t rows, uint64_t cols, uint32_t box_rows) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return set_error(SPEC_E_CUDA, "cuTensorMapEncodeTiled unavailable");
    const cuuint64_t dims[2] = {cols, rows};
    const cuuint64_t strides[1] = {cols * 2};
    const cuuint32_t box[2] = {64, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    const CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box, estr,
                           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return set_error(SPEC_E_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
    return SPEC_OK;
}

bool tc_supported(const Ctx& c) {
    const spec_model_cfg& m = c.cfg;
    return m.dtype == SPEC_BF16 && m.head_dim == 128 && m.d_model % 128 == 0 && m.vocab % 128 == 0 &&
           m.ffn_dim % 64 == 0 && (m.n_q_heads * m.head_dim) % 64 == 0 && encode_fn();
}

int tc_create(Ctx& c) {
    c.use_tc = false;
    if (!tc_supported(c)) return SPEC_OK;
    const spec_model_cfg& m = c.cfg;
    TcGemm* t = new TcGemm();
    const uint64_t d = m.d_model, qd = (uint64_t)m.n_q_heads * m.head_dim, kvd = (uint64_t)m.n_kv_heads * m.head_dim,
                   F = m.ffn_dim, V = m.vocab;
    int rc = SPEC_OK;
    t->layers.resize(m.n_layers);
    for (int l = 0; l < m.n_layers && rc == SPEC_OK; ++l) {
        const LayerWeights& L = c.w.layers[l];
        TcLayerMaps& M = t->layers[l];
        if ((rc = make_map(&M.q, L.wq, qd, d, 64)) || (rc = make_map(&M.k, L.wk, kvd, d, 64)) ||
            (rc = make_map(&M.v, L.wv, kvd, d, 64)) || (rc = make_map(&M.o, L.wo, d, qd, 64)) ||
            (rc = make_map(&M.g, L.wg, F, d, 64)) || (rc = make_map(&M.u, L.wu, F, d, 64)) ||
            (rc = make_map(&M.d, L.wd, d, F, 64)))
            break;
    }
    if (rc == SPEC_OK) rc = make_map(&t->lm, c.w.lm_head, V, d, 64);
    // GEMM inputs as [2][Mmax][cols]: bf16 hi rows, then the lo remainders
    if (rc == SPEC_OK) rc = make_map(&t->xn, c.Xn, 2 * (uint64_t)c.Mmax, d, 16);
    if (rc == SPEC_OK) rc = make_map(&t->xo, c.O, 2 * (uint64_t)c.Mmax, qd, 16);
    if (rc == SPEC_OK) rc = make_map(&t->xh, c.H, 2 * (uint64_t)c.Mmax, F, 16);
    t->grid = c.num_sms * TC_CTAS_PER_SM;
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

// Tensor maps and workspace of the context's GEMMs for the persistent pass: wmaps [7L + 1]
// (q k v o g u d per layer, then lm_head) and xmaps [3] (Xn, O, H); either may be null.
int tc_export(const Ctx& c, CUtensorMap* wmaps, CUtensorMap* xmaps, float** partial, int** tile_cnt, int* n_tile_cnt,
              int** err) {
    const TcGemm* t = c.tc;
    if (!t) return set_error(SPEC_E_STATE, "tensor-core GEMM not planned");
    const spec_model_cfg& m = c.cfg;
    if (wmaps) {
        for (int l = 0; l < m.n_layers; ++l) {
            const TcLayerMaps& L = t->layers[l];
            CUtensorMap* w = wmaps + (size_t)7 * l;
            w[0] = L.q; w[1] = L.k; w[2] = L.v; w[3] = L.o; w[4] = L.g; w[5] = L.u; w[6] = L.d;
        }
        wmaps[(size_t)7 * m.n_layers] = t->lm;
    }
    if (xmaps) {
        xmaps[0] = t->xn;
        xmaps[1] = t->xo;
        xmaps[2] = t->xh;
    }
    *partial = t->partial;
    *tile_cnt = t->tile_cnt;
    *n_tile_cnt = t->n_tile_cnt;
    *err = t->err;
    return SPEC_OK;
}

int tc_error_word(Ctx& c, int* out) {
    if (!c.tc) { *out = 0; return SPEC_OK; }
    return cudaMemcpy(out, c.tc->err, sizeof(int), cudaMemcpyDeviceToHost) == cudaSuccess ? SPEC_OK : SPEC_E_CUDA;
}

// Weight maps, tile count and K atoms per tile of GEMM `gid` of `layer`.
static void gemm_geometry(const Ctx& c, int gid, int layer, CUtensorMap* maps, int& n_tiles, int& KB) {
    const TcGemm* t = c.tc;
    const spec_model_cfg& m = c.cfg;
    const int d = m.d_model, qd = m.n_q_heads * m.head_dim, F = m.ffn_dim;
    switch (gid) {
    case GEMM_QKV:
        maps[0] = t->layers[layer].q; maps[1] = t->layers[layer].k; maps[2] = t->layers[layer].v;
        n_tiles = m.n_q_heads + 2 * m.n_kv_heads; KB = d / TC_ATOM;
        break;
    case GEMM_O: maps[0] = t->layers[layer].o; n_tiles = d / TC_BM; KB = qd / TC_ATOM; break;
    case GEMM_GU:
        maps[0] = t->layers[layer].g; maps[1] = t->layers[layer].u; n_tiles = F / 64; KB = d / TC_ATOM;
        break;
    case GEMM_DOWN: maps[0] = t->layers[layer].d; n_tiles = d / TC_BM; KB = F / TC_ATOM; break;
    default: maps[0] = t->lm; n_tiles = m.vocab / TC_BM; KB = d / TC_ATOM; break;
    }
}

static int tc_gemm_launch(Ctx& c, int gid, int layer, const void* X, int M, int pass_M, const EpiArgs& e,
                          cudaStream_t st) {
    TcGemm* t = c.tc;
    const spec_model_cfg& m = c.cfg;
    if (M < 1 || M > TC_MAX_NTOK) return set_error(SPEC_E_RANGE, "GEMM with M=%d tokens (max %d)", M, TC_MAX_NTOK);
    TcParams p{};
    const int d = m.d_model, qd = m.n_q_heads * m.head_dim, F = m.ffn_dim;
    int Kdim = d;
    const CUtensorMap* xm = &t->xn;
    const uint8_t* xbase = static_cast<const uint8_t*>(c.Xn);
    switch (gid) {
    case GEMM_QKV:
        p.wmap[0] = t->layers[layer].q; p.wmap[1] = t->layers[layer].k; p.wmap[2] = t->layers[layer].v;
        p.n_tiles = m.n_q_heads + 2 * m.n_kv_heads;
        break;
    case GEMM_O:
        p.wmap[0] = t->layers[layer].o; p.n_tiles = d / TC_BM; Kdim = qd; xm = &t->xo;
        xbase = static_cast<const uint8_t*>(c.O);
        break;
    case GEMM_GU:
        p.wmap[0] = t->layers[layer].g; p.wmap[1] = t->layers[layer].u; p.n_tiles = F / 64;
        break;
    case GEMM_DOWN:
        p.wmap[0] = t->layers[layer].d; p.n_tiles = d / TC_BM; Kdim = F; xm = &t->xh;
        xbase = static_cast<const uint8_t*>(c.H);
        break;
    default:
        p.wmap[0] = t->lm; p.n_tiles = m.vocab / TC_BM;
        break;
    }
    const size_t off = static_cast<const uint8_t*>(X) - xbase;
    p.x_row0 = (int)(off / ((size_t)Kdim * 2));
    p.xmap = *xm;
    p.gid = gid;
    p.KB = Kdim / TC_ATOM;
    p.ntok = (M + 15) & ~15;
    p.M = M;
    // the widest stage (most K atoms) that still leaves TC_MIN_STAGES ring slots; the
    // stream-K split is in atoms, so this choice changes no result bit
    const int budget = TC_SMEM_MAX - 1024 - TC_XBYTES;
    p.br = b_rows(c.split, M, p.x_row0, pass_M);
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
        gemm_geometry(c, ngid, nlayer, p.nwmap, p.n_ntiles, p.n_KB);
        p.ngid = ngid;
        p.n_atoms = c.l2_prefetch_atoms;
    }
    const long long T = (long long)p.n_tiles * p.KB;
    const int grid = (int)std::min<long long>(t->grid, T);
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
int tc_gemm(Ctx& c, int gid, int layer, const void* X, int M, int pass_M, const EpiArgs& e, cudaStream_t st) {
    if (M <= TC_MAX_NTOK) return tc_gemm_launch(c, gid, layer, X, M, pass_M, e, st);
    const spec_model_cfg& m = c.cfg;
    const int Kdim = gid == GEMM_O ? m.n_q_heads * m.head_dim : (gid == GEMM_DOWN ? m.ffn_dim : m.d_model);
    const int n = (M + TC_MAX_NTOK - 1) / TC_MAX_NTOK;
    int launched = 0, m0 = 0;
    for (int i = 0; i < n; ++i) {
        const int rest = M - m0, parts = n - i;
        const int chunk = std::min(rest, (((rest + parts - 1) / parts) + 15) & ~15);
        EpiArgs ec = e;
        ec.M = chunk;
        ec.m0 = e.m0 + m0;
        if (ec.ssq_in) ec.ssq_row0 = e.ssq_row0 + m0;
        const int r = tc_gemm_launch(c, gid, layer, static_cast<const uint8_t*>(X) + (size_t)m0 * Kdim * 2, chunk, pass_M,
                                     ec, st);
        if (r < 0) return r;
        launched += r;
        m0 += chunk;
    }
    return launched;
}

}  // namespace sv
