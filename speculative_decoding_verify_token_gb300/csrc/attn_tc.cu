// Multi-query causal GQA attention over the paged KV cache on the 5th-generation tensor
// cores (tcgen05), for passes of up to 96 query rows per (sequence, kv head): the verify
// pass (T = K + 1 tokens x G query heads), single-token decode and the drafting loop
// ("What is Speculative Decoding and How Does a Draft Model Work?", section "#3": the K+1
// positions are scored in one target pass; "Speculative Decoding on Apple Silicon...",
// section "How speculative decoding works": one pass over the cache serves all of them).
//
// One CTA per (512-key split, kv head, sequence), four 128-key tiles (used by contexts
// sized for batched serving; small batches keep the 64-key mma.sync kernel, whose many
// short splits fill the GPU at B = 1):
//  * S^T = K Q^T with the keys as the MMA's M (128 rows, every row used) and the query rows
//    as N (the rows padded to np = 16..96): A = a K tile straight from the cache (the pool
//    is kept in the swizzled per-head layout, so a run of consecutive pages is one bulk
//    copy), B = the queries as bf16 hi + lo halves accumulated into the same columns;
//  * the split's S tiles stay in tensor memory; the softmax warps take the rows' maxima over
//    the whole split first (one thread per key, shuffles and a fixed cross-warp order),
//    then write P = 2^(s - m) per tile as bf16 hi + lo halves (the probabilities need
//    about 16 significant bits: rounded to bf16 alone they moved the logits of one
//    8B-width layer by up to 1e-2) into shared memory as the next MMA's B operand;
//  * O^T += V^T P^T with V^T as an MN-major A operand (the same V tile, read transposed
//    by the tensor core) and the output in tensor memory; no rescaling, since the maxima
//    are final before the first P;
//  * the split's (max, sum, unnormalised output) per row go to the partial buffers that
//    the combine kernel reduces in a fixed order.
// Every row's arithmetic depends only on its own position and the split boundaries (fixed
// multiples of 512), not on np, T or the batch: a token gets the same bits decoded alone
// or verified with K drafts.
#include <cuda_bf16.h>
#include <algorithm>
#include <cmath>

#include "tc_common.cuh"

namespace sv {

constexpr int AT_TILE = 128;                    // keys per tile (the QK MMA's M)
constexpr int AT_TILES = 4;
constexpr int AT_SPLIT = AT_TILES * AT_TILE;    // keys per split (CTA)
constexpr int AT_SLOTS = 2;                     // ring slots of one K or V tile
constexpr int AT_SLOT_BYTES = 2 * AT_TILE * 128;   // two 64-dim halves of 128 keys x 128 B
constexpr int AT_THREADS = 192;
constexpr int AT_MAX_ROWS = 96;

int attn_tc_split_keys() { return AT_SPLIT; }
bool attn_tc_fits(int rows) { return rows >= 1 && rows <= AT_MAX_ROWS; }

// MN-major operand, 128-byte swizzle: 64-element rows of 128 B along the contiguous
// dimension; lbo = bytes between 64-element groups of that dimension, 8-row groups along
// the other dimension 1024 B apart.
__device__ __forceinline__ uint64_t smem_desc_mn_sw128(uint32_t addr, uint32_t lbo) {
    return (uint64_t)((addr >> 4) & 0x3FFFu) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
           ((uint64_t)(1024 >> 4) << 32) | ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

// kind::f16 instruction descriptor, M = 128, N = n, D f32, bf16 operands; a_mn: A MN-major.
__device__ __forceinline__ uint32_t idesc_bf16_m128(int n, bool a_mn) {
    return (1u << 4) | (1u << 7) | (1u << 10) | (a_mn ? (1u << 15) : 0u) | ((uint32_t)(n >> 3) << 17) |
           ((uint32_t)(128 >> 4) << 24);
}

__device__ __forceinline__ void at_fail(const AttnArgs& a) {
    if (a.err) atomicExch(a.err, SPEC_E_TIMEOUT);
}

template <int NP>
__global__ void __launch_bounds__(AT_THREADS, NP <= 48 ? 2 : 1) attn_tc_kernel(const __grid_constant__ AttnArgs a) {
    extern __shared__ uint8_t at_smem[];
    __shared__ __align__(8) uint64_t full_bar[AT_SLOTS], empty_bar[AT_SLOTS];
    __shared__ __align__(8) uint64_t q_bar, s_bar, p_bar, pe_bar, o_bar, done_bar;
    __shared__ uint32_t tmem_sh;
    __shared__ int pages[AT_SPLIT / 16];
    __shared__ int row_lim[NP];                 // last visible key of each row, relative to the split
    __shared__ float red[4][NP];
    __shared__ float row_m[NP];                 // the rows' maxima over the split (base-2 scaled scores)
    constexpr uint32_t QBYTES = 512u * NP;      // Q (hi, lo) x 2 halves x NP rows x 128 B; later P
    constexpr int CW = (AT_TILES + 1) * NP;     // S tiles + O
    constexpr uint32_t NCOLS = CW <= 32 ? 32u : (CW <= 64 ? 64u : (CW <= 128 ? 128u : (CW <= 256 ? 256u : 512u)));

    pdl_launch_dependents();
    const int s = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
    const int slot = a.seq_ids[b];
    const int L0 = a.seq_len[slot];
    const int Ltot = L0 + a.T;
    const int k0 = s * AT_SPLIT;
    if (k0 >= Ltot) return;                     // uniform over the CTA, before any barrier
    const int nkeys = min(AT_SPLIT, Ltot - k0);
    const int nt = (nkeys + AT_TILE - 1) / AT_TILE;
    const int npg = (nkeys + 15) >> 4;
    const int G = a.hq / a.hkv;
    const int R = a.T * G;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t base = (smem_u32(at_smem) + 1023u) & ~1023u;
    uint8_t* gbase = at_smem + (base - smem_u32(at_smem));
    const uint32_t qbuf = base;
    const uint32_t ring = base + QBYTES;

    // zero the ring (V rows past the split's keys are multiplied by P = 0 and must be
    // finite), the page list and the rows' visibility limits
    for (int i = threadIdx.x; i < AT_SLOTS * AT_SLOT_BYTES / 16; i += AT_THREADS)
        reinterpret_cast<uint4*>(gbase + QBYTES)[i] = make_uint4(0, 0, 0, 0);
    if (threadIdx.x < AT_SPLIT / 16) {
        const int lp = (k0 >> 4) + threadIdx.x;
        int pg = 0;
        if (threadIdx.x < npg && lp < a.max_pages) pg = a.block_table[(size_t)slot * a.max_pages + lp];
        pages[threadIdx.x] = min(max(pg, 0), a.num_pages - 1);
    }
    if (threadIdx.x < NP) {
        const int j = threadIdx.x;
        row_lim[j] = j < R ? L0 + j / G - k0 : -1;     // keys k (split-relative) <= row_lim are visible
    }
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    if (threadIdx.x == 0) {
        for (int i = 0; i < AT_SLOTS; ++i) {
            mbar_init(smem_u32(&full_bar[i]), 1);
            mbar_init(smem_u32(&empty_bar[i]), 1);
        }
        mbar_init(smem_u32(&q_bar), 1);
        mbar_init(smem_u32(&s_bar), 1);
        mbar_init(smem_u32(&p_bar), 128);
        mbar_init(smem_u32(&pe_bar), 1);
        mbar_init(smem_u32(&o_bar), 1);
        mbar_init(smem_u32(&done_bar), 1);
        fence_barrier_init();
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                     :: "r"(smem_u32(&tmem_sh)), "r"(NCOLS) : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_sh;

    if (warp == 0) {
        if (lane == 0) {
            // ---- producer: K tiles 0..nt-1, then V tiles 0..nt-1, through the ring ----
            const uint64_t pol = policy_evict_first();
            const int n_stage = 2 * nt;
            const size_t half_stride = (size_t)a.num_pages * 16 * 64;      // elements between halves
            auto issue = [&](int j) -> bool {
                const int sl = j % AT_SLOTS;
                if (j >= AT_SLOTS && !mbar_wait(smem_u32(&empty_bar[sl]), (uint32_t)(((j / AT_SLOTS) - 1) & 1))) {
                    at_fail(a);
                    return false;
                }
                const bool is_v = j >= nt;
                const int tile = is_v ? j - nt : j;
                const __nv_bfloat16* pool = static_cast<const __nv_bfloat16*>(is_v ? a.v_layer : a.k_layer) +
                                            (size_t)g * 2 * half_stride;
                const int p_lo = tile * 8, p_hi = min(npg, p_lo + 8);
                const uint32_t fb = smem_u32(&full_bar[sl]);
                mbar_arrive_expect_tx(fb, (uint32_t)(p_hi - p_lo) * 4096u);
                const uint32_t dst0 = ring + (uint32_t)sl * AT_SLOT_BYTES;
                for (int p = p_lo; p < p_hi;) {
                    int q = p + 1;
                    while (q < p_hi && pages[q] == pages[q - 1] + 1) ++q;     // a run of consecutive pages
                    for (int h = 0; h < 2; ++h)
                        bulk_g2s(dst0 + (uint32_t)h * (AT_SLOT_BYTES / 2) + (uint32_t)(p - p_lo) * 2048u,
                                 pool + h * half_stride + (size_t)pages[p] * 16 * 64, (uint32_t)(q - p) * 2048u, fb,
                                 pol);
                    p = q;
                }
                return true;
            };
            // tiles holding only keys of earlier passes do not depend on the QKV GEMM
            int j = 0;
            bool ok = true;
            auto old_keys = [&](int jj) {
                const int tile = jj >= nt ? jj - nt : jj;
                return k0 + (tile + 1) * AT_TILE <= L0;
            };
            while (j < min(AT_SLOTS, n_stage) && old_keys(j)) ok = issue(j++) && ok;
            pdl_wait();
            mbar_arrive_expect_tx(smem_u32(&q_bar), QBYTES);
            bulk_g2s(qbuf, static_cast<const __nv_bfloat16*>(a.q) + ((size_t)b * a.hkv + g) * (QBYTES / 2), QBYTES,
                     smem_u32(&q_bar), pol);
            for (; ok && j < n_stage; ++j) ok = issue(j);
            // no copy may still be landing when the CTA leaves
            for (int jj = max(0, j - AT_SLOTS); jj < j; ++jj)
                if (!mbar_wait(smem_u32(&full_bar[jj % AT_SLOTS]), (uint32_t)((jj / AT_SLOTS) & 1))) at_fail(a);
            if (!mbar_wait(smem_u32(&q_bar), 0)) at_fail(a);
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // ---- MMA issuer ----
            pdl_wait();
            const uint32_t id_s = idesc_bf16_m128(NP, false);
            const uint32_t id_o = idesc_bf16_m128(NP, true);
            bool ok = mbar_wait(smem_u32(&q_bar), 0);
            if (ok) tc_fence_after();
            for (int i = 0; ok && i < nt; ++i) {
                const int sl = i % AT_SLOTS;
                if (!(ok = mbar_wait(smem_u32(&full_bar[sl]), (uint32_t)((i / AT_SLOTS) & 1)))) break;
                tc_fence_after();
                const uint32_t kb = ring + (uint32_t)sl * AT_SLOT_BYTES;
#pragma unroll
                for (int lo = 0; lo < 2; ++lo)
#pragma unroll
                    for (int h = 0; h < 2; ++h)
                        mma_bf16_atom(tmem + (uint32_t)(i * NP), smem_desc_sw128(kb + (uint32_t)h * (AT_SLOT_BYTES / 2)),
                                      smem_desc_sw128(qbuf + (uint32_t)(lo * 2 + h) * NP * 128), id_s,
                                      (lo | h) ? 1u : 0u);
                mma_commit(smem_u32(&empty_bar[sl]));
            }
            if (ok) mma_commit(smem_u32(&s_bar));
            for (int i = 0; ok && i < nt; ++i) {
                const int jj = nt + i, sl = jj % AT_SLOTS;
                if (!(ok = mbar_wait(smem_u32(&full_bar[sl]), (uint32_t)((jj / AT_SLOTS) & 1)))) break;
                if (!(ok = mbar_wait(smem_u32(&p_bar), (uint32_t)(i & 1)))) break;
                tc_fence_after();
                const uint32_t vb = ring + (uint32_t)sl * AT_SLOT_BYTES;
#pragma unroll
                for (int lo = 0; lo < 2; ++lo)
#pragma unroll
                    for (int ks = 0; ks < AT_TILE / 16; ++ks)
                        mma_bf16(tmem + (uint32_t)(AT_TILES * NP), smem_desc_mn_sw128(vb + (uint32_t)ks * 2048u,
                                                                                       AT_SLOT_BYTES / 2),
                                 smem_desc_sw128(qbuf + (uint32_t)(lo * 2 + (ks >> 2)) * NP * 128 + (uint32_t)(ks & 3) * 32),
                                 id_o, (i | lo | ks) ? 1u : 0u);
                mma_commit(smem_u32(&empty_bar[sl]));
                mma_commit(smem_u32(&pe_bar));
            }
            if (ok) mma_commit(smem_u32(&o_bar));
            if (!ok) at_fail(a);
            // nothing may still write tensor memory when it is freed
            mma_commit(smem_u32(&done_bar));
            mbar_wait(smem_u32(&done_bar), 0);
        }
    } else {
        // ---- softmax and output: thread = key (S^T lanes) and then dim (O^T lanes) ----
        pdl_wait();
        const int q4 = warp & 3;                        // TMEM lane quarter of this warp
        const int etid = threadIdx.x - 64;
        const int key = q4 * 32 + lane;                 // key of the tile / dim of the output
        const uint32_t tl = tmem + ((uint32_t)(q4 * 32) << 16);
        const float sl2 = a.scale * 1.4426950408889634f;
        bool ok = mbar_wait(smem_u32(&s_bar), 0);
        if (epi_any(ok ? 0 : 1)) {
            if (etid == 0) at_fail(a);
        } else {
            tc_fence_after();
            // row maxima over the split: this thread's keys (one per tile), then the warp
            // (butterfly), then the four warps in a fixed order
#pragma unroll
            for (int c0 = 0; c0 < NP; c0 += 16) {
                float mx[16];
#pragma unroll
                for (int jj = 0; jj < 16; ++jj) mx[jj] = -INFINITY;
                for (int i = 0; i < nt; ++i) {
                    float v[16];
                    tmem_ld16(tl + (uint32_t)(i * NP + c0), v);
                    const int kk = i * AT_TILE + key;
#pragma unroll
                    for (int jj = 0; jj < 16; ++jj)
                        if (kk <= row_lim[c0 + jj]) mx[jj] = fmaxf(mx[jj], v[jj] * sl2);
                }
#pragma unroll
                for (int jj = 0; jj < 16; ++jj) {
                    float m = mx[jj];
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(FULL_MASK, m, o));
                    if (lane == 0) red[q4][c0 + jj] = m;
                }
            }
            epi_bar();
            if (etid < NP) row_m[etid] = fmaxf(fmaxf(red[0][etid], red[1][etid]), fmaxf(red[2][etid], red[3][etid]));
            epi_bar();
            // P = 2^(s - m) per tile, bf16 hi and lo, into the B operand of P V (it
            // overwrites the queries, whose MMAs are complete); row sums per thread
            float lsum[NP];
#pragma unroll
            for (int jj = 0; jj < NP; ++jj) lsum[jj] = 0.0f;
            const int atom = key >> 6, kc = key & 63;
            uint8_t* pbuf = gbase;
            for (int i = 0; i < nt; ++i) {
                if (i > 0) {
                    ok = mbar_wait(smem_u32(&pe_bar), (uint32_t)((i - 1) & 1));
                    if (epi_any(ok ? 0 : 1)) {
                        if (etid == 0) at_fail(a);
                        break;
                    }
                }
                const int kk = i * AT_TILE + key;
#pragma unroll
                for (int c0 = 0; c0 < NP; c0 += 16) {
                    float v[16];
                    tmem_ld16(tl + (uint32_t)(i * NP + c0), v);
#pragma unroll
                    for (int jj = 0; jj < 16; ++jj) {
                        const int j = c0 + jj;
                        const float rm = row_m[j];
                        const float m = rm == -INFINITY ? 0.0f : rm;
                        const float p = kk <= row_lim[j] ? exp2f(v[jj] * sl2 - m) : 0.0f;
                        lsum[j] += p;
                        const __nv_bfloat16 hi = __float2bfloat16_rn(p);
                        const __nv_bfloat16 lo = __float2bfloat16_rn(p - __bfloat162float(hi));
                        const uint32_t off = (uint32_t)j * 128 + ((uint32_t)(((kc >> 3) ^ (j & 7)) << 4) | ((kc & 7) << 1));
                        *reinterpret_cast<__nv_bfloat16*>(pbuf + (uint32_t)(0 * 2 + atom) * NP * 128 + off) = hi;
                        *reinterpret_cast<__nv_bfloat16*>(pbuf + (uint32_t)(1 * 2 + atom) * NP * 128 + off) = lo;
                    }
                }
                // the generic-proxy writes of P must be visible to the tensor core
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                tc_fence_before();
                mbar_arrive(smem_u32(&p_bar));
            }
            if (ok) {
                // row sums: warp butterfly, then the four warps in a fixed order
#pragma unroll
                for (int jj = 0; jj < NP; ++jj) {
                    float l = lsum[jj];
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1) l += __shfl_xor_sync(FULL_MASK, l, o);
                    if (lane == 0) red[q4][jj] = l;
                }
                epi_bar();
                const size_t pbase = (((size_t)b * a.hkv + g) * a.n_chunks + s) * R;
                if (etid < R) {
                    const float l = ((red[0][etid] + red[1][etid]) + red[2][etid]) + red[3][etid];
                    a.part_ml[pbase + etid] = make_float2(row_m[etid], l);
                }
                ok = mbar_wait(smem_u32(&o_bar), 0);
                if (epi_any(ok ? 0 : 1)) {
                    if (etid == 0) at_fail(a);
                } else {
                    tc_fence_after();
#pragma unroll
                    for (int c0 = 0; c0 < NP; c0 += 16) {
                        float v[16];
                        tmem_ld16(tl + (uint32_t)(AT_TILES * NP + c0), v);
#pragma unroll
                        for (int jj = 0; jj < 16; ++jj)
                            if (c0 + jj < R) a.part_o[(pbase + c0 + jj) * 128 + key] = v[jj];
                    }
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" :: "r"(tmem), "r"(NCOLS) : "memory");
}

static size_t attn_tc_smem(int np) {
    // 1 KB alignment slack + Q/P + the ring; above 48 rows one CTA per SM
    const size_t s = 1024 + 512 * (size_t)np + (size_t)AT_SLOTS * AT_SLOT_BYTES;
    return np <= 48 ? s : std::max<size_t>(s, 120 * 1024);
}

int attn_tc_set_smem_limits() {
    const int np[6] = {16, 32, 48, 64, 80, 96};
    void* k[6] = {(void*)attn_tc_kernel<16>, (void*)attn_tc_kernel<32>, (void*)attn_tc_kernel<48>,
                  (void*)attn_tc_kernel<64>, (void*)attn_tc_kernel<80>, (void*)attn_tc_kernel<96>};
    for (int i = 0; i < 6; ++i)
        if (cudaFuncSetAttribute(k[i], cudaFuncAttributeMaxDynamicSharedMemorySize, (int)attn_tc_smem(np[i])) !=
            cudaSuccess)
            return -1;
    return 0;
}



// Launch over nsplit 512-key splits; rows = T * G <= 96.
void launch_attn_tc(bool pdl, const AttnArgs& a, int nsplit, int B, cudaStream_t st) {
    const int np = (a.T * (a.hq / a.hkv) + 15) & ~15;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(nsplit, a.hkv, B);
    cfg.blockDim = dim3(AT_THREADS);
    cfg.dynamicSmemBytes = attn_tc_smem(np);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    switch (np) {
    case 16: cudaLaunchKernelEx(&cfg, attn_tc_kernel<16>, a); break;
    case 32: cudaLaunchKernelEx(&cfg, attn_tc_kernel<32>, a); break;
    case 48: cudaLaunchKernelEx(&cfg, attn_tc_kernel<48>, a); break;
    case 64: cudaLaunchKernelEx(&cfg, attn_tc_kernel<64>, a); break;
    case 80: cudaLaunchKernelEx(&cfg, attn_tc_kernel<80>, a); break;
    default: cudaLaunchKernelEx(&cfg, attn_tc_kernel<96>, a); break;
    }
}

}  // namespace sv
