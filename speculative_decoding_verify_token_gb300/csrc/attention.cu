// Paged causal GQA attention of a decoder pass over T new tokens per sequence.
//
// Passes of at most 96 query rows per (sequence, kv head) of batched contexts (max_batch >
// 4) on the tensor-core GEMM path run the tcgen05 kernel of attn_tc.cu (512-key splits);
// the kernels below serve small batches, longer passes (prefill chunks), other head dims
// and float32 models.
//
// For each (sequence, kv head) the T*G query rows (T positions x G = hq/hkv query heads)
// share one pass over the sequence's KV pages.  The keys are split at fixed absolute
// positions (64-key splits on the tensor-core path, a multiple of the 16-token page):
//  * attn_mma_kernel: one CTA per (split, kv head, sequence); it copies the split's keys and
//    values with 16-byte cp.async -- the keys of earlier passes before it waits for the QKV
//    GEMM (programmatic launch), this pass's keys and the queries after -- and writes the
//    split's per-row max, sum and unnormalised output (mma.sync bf16, queries and
//    probabilities as bf16 hi + lo);
//  * attn_mma_multi_kernel (long contexts): one CTA per run of consecutive splits, with the
//    same per-split arithmetic and K/V double-buffered;
//  * a combine kernel per row then reduces the row's splits 0..pos/64 in a fixed order
//    (attn_combine128_kernel up to 512 splits, attn_combine_kernel beyond).
// Every row is computed on its own in a fixed order of operations that depends only on
// its absolute position, so a token gets the same bits whether it is decoded alone
// (T = 1) or verified together with K drafts (T = K + 1).  The SIMT kernels (float32
// models, other head dims) follow the same split / combine structure with bulk copies.
#include <cuda_bf16.h>
#include <cmath>

#include "attn_mma.cuh"

namespace sv {

constexpr int ATT_THREADS = 256;
constexpr int ATT_RT = 32;                     // query rows per tile
constexpr int ATT_KV_SMEM = 128 * 1024;        // K + V bytes of one split
#ifndef ATT_MULTI_MIN
#define ATT_MULTI_MIN 4                        // fewest splits per CTA worth the multi-split kernel
#endif


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


// ---- tensor-core path (bf16, head_dim 128) ---------------------------------------------------

// One CTA of 4 warps per (64-key split, kv head, sequence).
__global__ void __launch_bounds__(128) attn_mma_kernel(const AttnArgs a) {
    extern __shared__ __align__(128) uint8_t sm_raw[];
    __shared__ float wmax[4][MMA_RT], wsum[4][MMA_RT];
    pdl_launch_dependents();
    AttnSmem sm;
    sm.Ks = reinterpret_cast<__nv_bfloat16*>(sm_raw);
    sm.Vs = sm.Ks + MMA_SPLIT * MMA_PITCH;
    sm.Qs = sm.Vs + MMA_SPLIT * MMA_PITCH;
    sm.Qlo = sm.Qs + MMA_RT * MMA_PITCH;
    sm.Ps = sm.Qlo + MMA_RT * MMA_PITCH;
    sm.Plo = sm.Ps + MMA_RT * MMA_PPITCH;
    sm.wmax = wmax;
    sm.wsum = wsum;
    // keys of earlier passes load before the wait for the QKV GEMM (programmatic launch)
    attn_mma_item(a, blockIdx.x, blockIdx.y, blockIdx.z, sm, threadIdx.x, [] { __syncthreads(); },
                  [] { pdl_wait(); return true; });
}

// Long contexts: one CTA of 4 warps per run of `spc` consecutive 64-key splits of a (kv head,
// sequence), for items whose T*G query rows fit one 64-row tile.  The queries are loaded
// once; K and V of the next split stream into the other half of a double buffer while the
// current split is computed by the same per-tile code as attn_mma_kernel, so every split's
// partial (and hence every output bit) is the same as with one CTA per split -- only the
// number of CTAs, and the per-CTA overhead, change.  Rows a split fully masks (positions
// below its first key) are not written; the combine never reads them.
constexpr size_t MMA_MULTI_SMEM =
    sizeof(__nv_bfloat16) * ((size_t)4 * MMA_SPLIT * MMA_PITCH + (size_t)2 * MMA_RT * MMA_PITCH +
                             (size_t)MMA_RT * MMA_PPITCH);

__device__ __forceinline__ void attn_load_split(const AttnArgs& a, int slot, int g, int k0, int nk,
                                                __nv_bfloat16* Ks, __nv_bfloat16* Vs, int tid) {
    const __nv_bfloat16* kp = static_cast<const __nv_bfloat16*>(a.k_layer);
    const __nv_bfloat16* vp = static_cast<const __nv_bfloat16*>(a.v_layer);
    for (int i = tid; i < MMA_SPLIT * 16; i += 128) {
        const int key = i >> 4, ch = i & 15;
        if (key < nk) {
            const int pos = k0 + key;
            const int page = a.block_table[(size_t)slot * a.max_pages + (pos >> 4)];
            const size_t off = kv_off(page, g, pos & 15, ch * 8, a.hkv, 128, a.num_pages, a.kv_sw);
            cp_async16(smem_u32(Ks + key * MMA_PITCH + ch * 8), kp + off);
            cp_async16(smem_u32(Vs + key * MMA_PITCH + ch * 8), vp + off);
        } else {
            *reinterpret_cast<uint4*>(Ks + key * MMA_PITCH + ch * 8) = make_uint4(0, 0, 0, 0);
            *reinterpret_cast<uint4*>(Vs + key * MMA_PITCH + ch * 8) = make_uint4(0, 0, 0, 0);
        }
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
}

// Warm L2 with the K and V pages of split s (four 16-token pages of each, 4 KB apiece: one
// run, or two 2 KB halves in the tensor-core layout).
__device__ __forceinline__ void attn_prefetch_split(const AttnArgs& a, int slot, int g, int s, int Ltot) {
    const __nv_bfloat16* kp = static_cast<const __nv_bfloat16*>(a.k_layer);
    const __nv_bfloat16* vp = static_cast<const __nv_bfloat16*>(a.v_layer);
    for (int pos = s * MMA_SPLIT; pos < min(Ltot, (s + 1) * MMA_SPLIT); pos += 16) {
        const int page = a.block_table[(size_t)slot * a.max_pages + (pos >> 4)];
        for (int h = 0; h < (a.kv_sw ? 2 : 1); ++h) {
            const size_t off = kv_off(page, g, 0, h * 64, a.hkv, 128, a.num_pages, a.kv_sw);
            const uint32_t bytes = a.kv_sw ? 2048u : 4096u;
            asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" :: "l"(kp + off), "r"(bytes) : "memory");
            asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" :: "l"(vp + off), "r"(bytes) : "memory");
        }
    }
}

__global__ void __launch_bounds__(128) attn_mma_multi_kernel(const AttnArgs a, int spc) {
    extern __shared__ __align__(128) uint8_t sm_raw[];
    __shared__ float wmax[4][MMA_RT], wsum[4][MMA_RT];
    pdl_launch_dependents();
    __nv_bfloat16* Kb = reinterpret_cast<__nv_bfloat16*>(sm_raw);          // [2][K, V][64][PITCH]
    __nv_bfloat16* Qs = Kb + 4 * MMA_SPLIT * MMA_PITCH;
    __nv_bfloat16* Qlo = Qs + MMA_RT * MMA_PITCH;
    __nv_bfloat16* Ps = Qlo + MMA_RT * MMA_PITCH;
    const int tid = threadIdx.x;
    const int g = blockIdx.y, b = blockIdx.z;
    const int slot = a.seq_ids[b];
    const int L0 = a.seq_len[slot];
    const int Ltot = L0 + a.T;
    const int s_begin = blockIdx.x * spc;
    const int s_end = min(s_begin + spc, (Ltot + MMA_SPLIT - 1) / MMA_SPLIT);
    if (s_begin >= s_end) return;
    const int G = a.hq / a.hkv;
    const int R = a.T * G;            // <= MMA_RT (checked by the host)
    const bool qsplit = a.q_lo_off != 0;
    const __nv_bfloat16* Q = static_cast<const __nv_bfloat16*>(a.q);
    for (int i = tid; i < MMA_RT * 16; i += 128) {
        const int ri = i >> 4, ch = i & 15;
        if (ri < R) {
            const int t = ri / G, hh = ri - t * G;
            const size_t m = (size_t)b * a.T + t;
            const __nv_bfloat16* src = Q + (m * a.hq + (size_t)g * G + hh) * 128 + ch * 8;
            cp_async16(smem_u32(Qs + ri * MMA_PITCH + ch * 8), src);
            if (qsplit) cp_async16(smem_u32(Qlo + ri * MMA_PITCH + ch * 8), src + a.q_lo_off);
        } else {
            *reinterpret_cast<uint4*>(Qs + ri * MMA_PITCH + ch * 8) = make_uint4(0, 0, 0, 0);
            if (qsplit) *reinterpret_cast<uint4*>(Qlo + ri * MMA_PITCH + ch * 8) = make_uint4(0, 0, 0, 0);
        }
    }
    auto kbuf = [&](int s) { return Kb + (size_t)(s & 1) * 2 * MMA_SPLIT * MMA_PITCH; };
    const int ahead = a.l2_ahead;
    if (tid == 0)
        for (int s = s_begin + 1; s < min(s_end, s_begin + 1 + ahead); ++s) attn_prefetch_split(a, slot, g, s, Ltot);
    {
        const int k0 = s_begin * MMA_SPLIT;
        attn_load_split(a, slot, g, k0, min(MMA_SPLIT, Ltot - k0), kbuf(s_begin), kbuf(s_begin) + MMA_SPLIT * MMA_PITCH,
                        tid);        // commits the queries too
    }
    const float sl2 = a.scale * 1.4426950408889634f;
    for (int s = s_begin; s < s_end; ++s) {
        if (tid == 0 && ahead > 0 && s + 1 + ahead < s_end) attn_prefetch_split(a, slot, g, s + 1 + ahead, Ltot);
        if (s + 1 < s_end) {
            const int k1 = (s + 1) * MMA_SPLIT;
            attn_load_split(a, slot, g, k1, min(MMA_SPLIT, Ltot - k1), kbuf(s + 1),
                            kbuf(s + 1) + MMA_SPLIT * MMA_PITCH, tid);
            asm volatile("cp.async.wait_group 1;" ::: "memory");
        } else {
            asm volatile("cp.async.wait_group 0;" ::: "memory");
        }
        __syncthreads();
        const int k0 = s * MMA_SPLIT;
        const int nk = min(MMA_SPLIT, Ltot - k0);
        const size_t pbase = (((size_t)b * a.hkv + g) * a.n_chunks + s) * R;
        // one row tile per item here (R <= MMA_RT), so the split's keys are dead once its
        // scores are taken and the probabilities' lo halves go in their place
        attn_mma_tile(a, kbuf(s), kbuf(s) + MMA_SPLIT * MMA_PITCH, Qs, Qlo, Ps, kbuf(s), wmax, wsum, qsplit, 0, R,
                      max(0, k0 - L0) * G, k0, nk, L0, G, pbase, sl2, tid, [] { __syncthreads(); });
        __syncthreads();             // this half of the buffer is refilled two splits on
    }
}

// One warp per query row.
template <typename T>
__global__ void __launch_bounds__(128) attn_combine_kernel(const AttnArgs a) {
    pdl_launch_dependents();
    pdl_wait();
    attn_combine_row<T>(a, blockIdx.x * 4 + (threadIdx.x >> 5), blockIdx.y, blockIdx.z, threadIdx.x & 31);
}

// head_dim 128 with at most COMB_MAXC splits: the vectorised combine (same bits), with few
// enough registers for six CTAs (24 warps) per SM.
template <typename T>
__global__ void __launch_bounds__(128, 6) attn_combine128_kernel(const AttnArgs a) {
    __shared__ float2 mls[4][COMB_MAXC];
    pdl_launch_dependents();
    pdl_wait();
    const int warp = threadIdx.x >> 5;
    const int r = blockIdx.x * 4 + warp;
    if (r >= a.T * (a.hq / a.hkv)) return;
    attn_combine_row_128<T>(a, r, blockIdx.y, blockIdx.z, threadIdx.x & 31, mls[warp]);
}

size_t attn_smem(int hd, int esize) {
    const int split = attention_split_keys(hd, esize);
    return (size_t)2 * split * hd * esize + sizeof(float) * ((size_t)ATT_RT * hd + (size_t)ATT_RT * split);
}

// Launch with programmatic stream serialization when pdl is set: the kernel may start
// while the previous one finishes and waits for it (griddepcontrol.wait) where it first
// reads that kernel's outputs.
template <typename... Args>
static void launch_pdl(bool pdl, void (*kernel)(Args...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                       Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaLaunchKernelEx(&cfg, kernel, args...);
}

int launch_attention(const Ctx& c, const AttnArgs& a, int B, int max_len_after, cudaStream_t st) {
    const int nsplit = (max_len_after + a.split_keys - 1) / a.split_keys;
    const int G = a.hq / a.hkv;
    const dim3 cgrid((a.T * G + 3) / 4, a.hkv, B);
    if (a.q_np > 0) {
        // tensor-core attention and the vectorised combine, both launched early (the
        // combine waits for the attention's partials with griddepcontrol.wait)
        launch_attn_tc(c.use_pdl, a, nsplit, B, c.num_sms > 0 ? c.num_sms : 148, st);
        if (nsplit <= COMB_MAXC)
            launch_pdl(c.use_pdl, attn_combine128_kernel<__nv_bfloat16>, cgrid, dim3(128), 0, st, a);
        else
            launch_pdl(c.use_pdl, attn_combine_kernel<__nv_bfloat16>, cgrid, dim3(128), 0, st, a);
        return 2;
    }
    if (use_mma_path(a.hd, c.esize)) {
        // splits per CTA: one while the items fill about four waves of the GPU, more for
        // long contexts (at least ATT_MULTI_MIN), so that each CTA streams a run of keys
        const long long items = (long long)nsplit * a.hkv * B;
        const long long target = 4LL * 2 * (c.num_sms > 0 ? c.num_sms : 152);
        int spc = (int)std::min<long long>(nsplit, (items + target - 1) / target);
        if (a.T * G > MMA_RT || spc < ATT_MULTI_MIN) spc = 1;
        if (spc == 1) {
            launch_pdl(c.use_pdl, attn_mma_kernel, dim3(nsplit, a.hkv, B), dim3(128), MMA_SMEM, st, a);
        } else {
            attn_mma_multi_kernel<<<dim3((nsplit + spc - 1) / spc, a.hkv, B), 128, MMA_MULTI_SMEM, st>>>(a, spc);
        }
        if (a.n_chunks <= COMB_MAXC)
            attn_combine128_kernel<__nv_bfloat16><<<cgrid, 128, 0, st>>>(a);
        else
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
    if (attn_tc_set_smem_limits() != 0) return -1;
    if (cudaFuncSetAttribute(attn_mma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)MMA_SMEM) !=
            cudaSuccess ||
        cudaFuncSetAttribute(attn_mma_multi_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)MMA_MULTI_SMEM) != cudaSuccess)
        return -1;
    if (cudaFuncSetAttribute(attn_split_kernel<__nv_bfloat16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)attn_smem(hd, 2)) != cudaSuccess ||
        cudaFuncSetAttribute(attn_split_kernel<float>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)attn_smem(hd, 4)) != cudaSuccess)
        return -1;
    return 0;
}

}  // namespace sv
