// Combine kernel ("Kernel B"): merges the per-split partials of one
// (sequence, query head) row,
//     m = max_i m_i,  w_i = exp(m_i - m),  out = sum_i w_i acc_i / sum_i w_i l_i
// ("Attention at 128k: Split Over Context", §2; aprender issue 3725 design
// note §2). A neutral partial (l = 0) gets weight 0 and its acc is not used
// (an empty split of the MLA kernel leaves it unwritten).
//
// For a context-parallel step the partials of several ranks are merged the
// same way: the (rank, split) pairs of a row are one list.
//
// One CTA per (query head, sequence, 128 value columns); 8 warps. Each warp
// loads the acc vectors of its own splits (s = warp, warp + 8, ...) first,
// then computes m and l over all splits itself (lanes stride the splits, warp
// shuffles reduce), so the only block-wide step is the final sum of the 8
// warps' vectors. Launched with programmatic stream serialization: the CTAs
// may start while the split kernel drains and wait in griddepcontrol.wait.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <type_traits>

#include "internal.h"
#include "merge.cuh"
#include "ptx.cuh"

namespace skv {

constexpr int kCombineThreads = 256;
constexpr int kCombineWarps = kCombineThreads / 32;
constexpr int kCombineCols = 128;   // value columns per CTA (one float4 per lane)
constexpr int kCombinePrefetch = 10; // acc vectors per lane loaded before the weights
                                     // (all of them for up to 80 splits)

template <typename OT> __device__ __forceinline__ void store1(OT *p, float v);
template <> __device__ __forceinline__ void store1<float>(float *p, float v) { *p = v; }
template <> __device__ __forceinline__ void store1<__half>(__half *p, float v)
{
    *p = __float2half_rn(v);
}
template <> __device__ __forceinline__ void store1<__nv_bfloat16>(__nv_bfloat16 *p, float v)
{
    *p = __float2bfloat16_rn(v);
}

// Merge the partials of row h of sequence b over the 128 value columns of
// block z. Every warp takes part; warp 0 returns the normalised result of its
// lane's four columns (the other warps' return values are not used). Ends with
// the block barrier that makes part[] reusable.
__device__ __forceinline__ float4 merge_columns(const CombineParams &p, int h, int b, int z,
                                                float4 (*part)[32])
{
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int S = p.n_splits[b];
    const int SR = S * p.n_ranks;                            // (rank, split) pairs
    const size_t slot0 = (size_t)p.split_base[b];
    const int col = z * kCombineCols + lane * 4;
    const bool live = col < p.v_dim;
    // pair i = r * S + s: rank r's split s (a division only with several ranks)
    const float2 *ml0 = p.ml + slot0 * p.n_heads + h;
    const float *acc0 = p.acc + (slot0 * p.n_heads + h) * p.v_dim + (live ? col : 0);
    const size_t acc_step = (size_t)p.n_heads * p.v_dim;
    auto ml_of = [&](int i) {
        if (p.n_ranks == 1) return __ldg(ml0 + (size_t)i * p.n_heads);
        const int r = i / S;
        return __ldg(ml0 + r * p.rank_ml + (size_t)(i - r * S) * p.n_heads);
    };
    auto acc_of = [&](int i) {
        const float *a = acc0 + (size_t)i * acc_step;
        if (p.n_ranks > 1) {
            const int r = i / S;
            a = acc0 + r * p.rank_acc + (size_t)(i - r * S) * acc_step;
        }
        return __ldg(reinterpret_cast<const float4 *>(a));
    };

    // acc vectors of this warp's first pairs, in flight while m and l are formed
    float4 pv[kCombinePrefetch];
#pragma unroll
    for (int i = 0; i < kCombinePrefetch; ++i) {
        const int sp = warp + kCombineWarps * i;
        pv[i] = (live && sp < SR) ? acc_of(sp) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    // m = max_i m_i and l = sum_i e^{m_i - m} l_i, by every warp for itself, in
    // one pass: each lane merges its pairs online, then the lanes merge theirs
    // pairwise with the same rescaling (every lane ends with the same M and L)
    float M = kNeutralM, L = 0.f;
#pragma unroll 4
    for (int sp = lane; sp < SR; sp += 32) {
        const float2 x = ml_of(sp);
        if (x.x > M) {
            L = fmaf(L, ex2((M - x.x) * kLog2e), x.y);
            M = x.x;
        } else {
            L = fmaf(x.y, ex2((x.x - M) * kLog2e), L);
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float Mo = __shfl_xor_sync(0xffffffffu, M, o);
        const float Lo = __shfl_xor_sync(0xffffffffu, L, o);
        const float Mn = fmaxf(M, Mo);
        L = L * ex2((M - Mn) * kLog2e) + Lo * ex2((Mo - Mn) * kLog2e);
        M = Mn;
    }

    float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int i = 0; i < kCombinePrefetch; ++i) {
        const int sp = warp + kCombineWarps * i;
        if (sp < SR) {
            const float2 x = ml_of(sp);
            if (x.y > 0.f) fma4(a, ex2((x.x - M) * kLog2e), pv[i]);
        }
    }
    for (int sp = warp + kCombineWarps * kCombinePrefetch; sp < SR; sp += kCombineWarps) {
        const float2 x = ml_of(sp);
        if (live && x.y > 0.f) fma4(a, ex2((x.x - M) * kLog2e), acc_of(sp));
    }
    part[warp][lane] = a;
    __syncthreads();
    float4 t = make_float4(0.f, 0.f, 0.f, 0.f);
    if (warp == 0 && live) {
        t = part[0][lane];
#pragma unroll
        for (int w = 1; w < kCombineWarps; ++w) {
            const float4 u = part[w][lane];
            t.x += u.x; t.y += u.y; t.z += u.z; t.w += u.w;
        }
        const float inv = 1.f / L;
        t.x *= inv; t.y *= inv; t.z *= inv; t.w *= inv;
    }
    return t;
}

template <typename OT>
__global__ void __launch_bounds__(kCombineThreads)
    combine_kernel(const __grid_constant__ CombineParams p)
{
    __shared__ __align__(16) float4 part[kCombineWarps][32];

    griddep_wait();

    const int h = blockIdx.x, b = blockIdx.y;
    const int lane = threadIdx.x & 31;
    const float4 t = merge_columns(p, h, b, blockIdx.z, part);
    const int col = blockIdx.z * kCombineCols + lane * 4;
    if (threadIdx.x < 32 && col < p.v_dim) {
        OT *out = reinterpret_cast<OT *>(p.out) + ((size_t)b * p.n_heads + h) * p.v_dim + col;
        store4<OT>(out, t);
    }
}

// ---------------------------------------------------------------------------
// The same merge with the partials staged in shared memory, for one rank's
// partials and a v_dim that is a multiple of 128: bulk copies bring each
// split's 512-byte block of the CTA's 128 columns (one mbarrier for all of
// them) while warp 0 forms the weights w_s = e^{m_s - m} / sum_i e^{m_i - m} l_i
// from the (m, l) pairs (w_s = 0 for a neutral partial, whose block is never
// used); then warp w sums w_s acc_s over the splits w, w + 8, ... from shared
// memory and warp 0 adds the 8 sums in a fixed order. The copies are issued
// right after griddepcontrol.wait, so the CTA waits for one round trip.
constexpr int kStagedMaxSplits = 256;

// A stage: [max_splits blocks of 512 B][max_splits weights][8 x 32 float4
// sums], and an mbarrier and a flag (right after it, or elsewhere)
struct Stage {
    unsigned char *blk;
    float *wts;
    float4 *red;
    uint64_t *bar;
    volatile int *flag;
};

__host__ __device__ constexpr int staged_wts_bytes(int max_splits)
{
    return (max_splits * 4 + 15) / 16 * 16;
}

// bytes of the blocks, weights and sums (the mbarrier and flag apart)
__host__ __device__ constexpr int staged_area_bytes(int max_splits)
{
    return max_splits * kCombineCols * 4 + staged_wts_bytes(max_splits) + kCombineWarps * 32 * 16;
}

static int combine_staged_smem_bytes(int max_splits)
{
    return staged_area_bytes(max_splits) + 16;
}

// the blocks, weights and sums at base; the mbarrier and the flag at bar
__device__ __forceinline__ Stage stage_in(unsigned char *base, int max_splits, uint64_t *bar)
{
    Stage st;
    st.blk = base;
    st.wts = reinterpret_cast<float *>(base + (size_t)max_splits * kCombineCols * 4);
    st.red = reinterpret_cast<float4 *>(base + (size_t)max_splits * kCombineCols * 4 +
                                        staged_wts_bytes(max_splits));
    st.bar = bar;
    st.flag = reinterpret_cast<volatile int *>(bar + 1);
    return st;
}

__device__ __forceinline__ Stage stage_at(unsigned char *base, int max_splits)
{
    return stage_in(base, max_splits,
                    reinterpret_cast<uint64_t *>(base + staged_area_bytes(max_splits)));
}

// Thread 0 sets the stage's mbarrier up; the caller syncs the block before use.
__device__ __forceinline__ void stage_init(const Stage &st)
{
    if (threadIdx.x == 0) {
        mbar_init(st.bar, 1);
        fence_mbar_init();
    }
}

// The merge of row h of sequence b over the 128 columns of block z, after
// griddepcontrol.wait. Warp 0 gets the normalised result of its lane's four
// columns; *ok (the same in every thread) is false when the wait for the
// blocks ran out (recorded in the status word; the result is then zero), as
// it does when `load` is false (a test hook: no copy is issued). Every thread
// of the block calls it; it ends with a block barrier.
__device__ __forceinline__ float4 staged_merge(const CombineParams &p, int h, int b, int z,
                                               const Stage &st, bool load, bool *ok)
{
    constexpr int BLK = kCombineCols * 4;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int S = p.n_splits[b];
    const size_t slot0 = (size_t)p.split_base[b];
    fence_proxy_async_global(); // the split kernel's partials, for the bulk copies

    if (threadIdx.x == 0 && load) mbar_arrive_expect_tx(st.bar, (uint32_t)(S * BLK));
    __syncthreads(); // the expected bytes are set before any copy completes
    if (load)
        for (int s = threadIdx.x; s < S; s += kCombineThreads)
            bulk_load_g2s(st.blk + (size_t)s * BLK,
                          p.acc + ((slot0 + s) * p.n_heads + h) * p.v_dim + z * kCombineCols, BLK,
                          st.bar);
    if (warp == 0) {
        // m = max_i m_i, l = sum_i e^{m_i - m} l_i: the lanes merge their splits
        // online (all pairs of up to 128 splits in flight at once), then pairwise
        constexpr int WB = 4;
        const float2 *ml = p.ml + slot0 * p.n_heads + h;
        float2 x[WB];
        float M = kNeutralM, L = 0.f;
        for (int s0 = 0; s0 < S; s0 += 32 * WB) {
#pragma unroll
            for (int i = 0; i < WB; ++i) {
                const int s = s0 + 32 * i + lane;
                x[i] = s < S ? __ldg(ml + (size_t)s * p.n_heads) : make_float2(kNeutralM, 0.f);
            }
#pragma unroll
            for (int i = 0; i < WB; ++i) {
                if (x[i].y > 0.f) {
                    const float mn = fmaxf(M, x[i].x);
                    L = L * ex2((M - mn) * kLog2e) + x[i].y * ex2((x[i].x - mn) * kLog2e);
                    M = mn;
                }
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float Mo = __shfl_xor_sync(0xffffffffu, M, o);
            const float Lo = __shfl_xor_sync(0xffffffffu, L, o);
            const float mn = fmaxf(M, Mo);
            L = L * ex2((M - mn) * kLog2e) + Lo * ex2((Mo - mn) * kLog2e);
            M = mn;
        }
        const float inv = L > 0.f ? 1.f / L : 0.f;
        if (S <= 32 * WB) { // the pairs are still in registers
#pragma unroll
            for (int i = 0; i < WB; ++i) {
                const int s = 32 * i + lane;
                if (s < S) st.wts[s] = x[i].y > 0.f ? ex2((x[i].x - M) * kLog2e) * inv : 0.f;
            }
        } else {
            for (int s = lane; s < S; s += 32) {
                const float2 y = __ldg(ml + (size_t)s * p.n_heads);
                st.wts[s] = y.y > 0.f ? ex2((y.x - M) * kLog2e) * inv : 0.f;
            }
        }
    }
    if (threadIdx.x == 0) {
        // a wait that runs out (or copies never requested, the test hook)
        // leaves this CTA's result zero and records the timeout
        volatile int never = 0;
        const bool done = load && mbar_wait_bounded(st.bar, 0, p.timeout_ns, &never);
        if (!done) {
            atomicCAS(p.status, 0, kStatusTimeoutCombine);
            // copies still in flight land before the CTA's memory is released
            if (load) (void)mbar_wait_bounded(st.bar, 0, p.timeout_ns, &never);
        }
        *st.flag = done ? 1 : 0;
    }
    __syncthreads(); // also publishes the weights
    *ok = *st.flag != 0;
    float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
    if (*ok) {
        volatile int never = 0;
        (void)mbar_wait_bounded(st.bar, 0, p.timeout_ns, &never); // complete: this thread's view
#pragma unroll 4
        for (int s = warp; s < S; s += kCombineWarps) {
            const float w = st.wts[s];
            const float4 v = reinterpret_cast<const float4 *>(st.blk + (size_t)s * BLK)[lane];
            if (w > 0.f) fma4(a, w, v);
        }
    }
    st.red[warp * 32 + lane] = a;
    __syncthreads();
    float4 t = make_float4(0.f, 0.f, 0.f, 0.f);
    if (warp == 0) {
        t = st.red[lane];
#pragma unroll
        for (int w = 1; w < kCombineWarps; ++w) {
            const float4 u = st.red[w * 32 + lane];
            t.x += u.x;
            t.y += u.y;
            t.z += u.z;
            t.w += u.w;
        }
    }
    __syncthreads(); // the stage may be reused
    return t;
}

template <typename OT>
__global__ void __launch_bounds__(kCombineThreads)
    combine_staged_kernel(const __grid_constant__ CombineParams p, int max_splits)
{
    extern __shared__ __align__(128) unsigned char dsm[];
    const Stage st = stage_at(dsm, max_splits);
    stage_init(st);
    __syncthreads();

    griddep_wait();

    bool ok;
    const float4 t = staged_merge(p, blockIdx.x, blockIdx.y, blockIdx.z, st,
                                  !(p.flags & DA_FLAG_TEST_NO_TMA), &ok);
    if (ok && threadIdx.x < 32) {
        OT *out = reinterpret_cast<OT *>(p.out) + ((size_t)blockIdx.y * p.n_heads + blockIdx.x) * p.v_dim +
                  blockIdx.z * kCombineCols + threadIdx.x * 4;
        store4<OT>(out, t);
    }
}

// ---------------------------------------------------------------------------
// Combine fused with the per-head output projection (the MLA value
// up-projection wv_b): out[b][h][e] = sum_c W[h][e][c] merged[b][h][c]. The
// projection is a function of the merged result, not of any one partial, so it
// runs after the merge and never per split ("The Kernel Level" / PR #49
// write-up: the output projection moves into the combine).
//
// A cluster of Z = ceil(v_dim / 128) CTAs serves one (row, sequence); CTA z
// merges the columns [128 z, 128 z + 128) as the combine does, projects them
// with its slice W[h][:][128 z ...] (held in shared memory) into out_dim
// partial sums, and the cluster adds the Z partial vectors through distributed
// shared memory in a fixed order (bit-reproducible). Where the combine stages
// the partials (one rank, whole 128-column blocks), the slice shares their
// shared memory: its rows are asked into L2 as the CTA starts and copied in by
// bulk copies once the merge is done, so the CTA holds max(slice, stage)
// rather than both. Otherwise the slice is copied in before
// griddepcontrol.wait and the partials are read with plain loads.
// asks for `bytes` (multiple of 16, address 16-byte aligned) of global memory
// to be brought into L2, without waiting for them
__device__ __forceinline__ void bulk_prefetch_l2(const void *src, uint32_t bytes)
{
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

template <typename WT> struct WLoad;
template <> struct WLoad<float> {
    static __device__ __forceinline__ float4 get(const unsigned char *row, int c)
    {
        return *reinterpret_cast<const float4 *>(row + c * 4);
    }
};
template <> struct WLoad<__nv_bfloat16> {
    static __device__ __forceinline__ float4 get(const unsigned char *row, int c)
    {
        const uint2 u = *reinterpret_cast<const uint2 *>(row + c * 2);
        return make_float4(__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xffff0000u),
                           __uint_as_float(u.y << 16), __uint_as_float(u.y & 0xffff0000u));
    }
};

// [region: the W slice [out_dim][128], or the staged partials, whichever is
// larger][partial outputs [out_dim]][slice mbarrier | stage mbarrier, flag]
__host__ __device__ constexpr int proj_region_bytes(int es, int out_dim, int max_splits)
{
    return ((out_dim * kCombineCols * es > staged_area_bytes(max_splits)
                 ? out_dim * kCombineCols * es
                 : staged_area_bytes(max_splits)) + 15) / 16 * 16;
}

static int combine_proj_smem_bytes(int w_dtype, int out_dim, int max_splits)
{
    const int es = w_dtype == DA_BF16 ? 2 : 4;
    return proj_region_bytes(es, out_dim, max_splits) + ((out_dim * 4 + 15) / 16) * 16 + 32;
}

template <typename OT, typename WT>
__global__ void __launch_bounds__(kCombineThreads)
    combine_proj_kernel(const __grid_constant__ CombineParams p, int max_splits)
{
    __shared__ __align__(16) float4 part[kCombineWarps][32];
    __shared__ __align__(16) float merged[kCombineCols];
    extern __shared__ __align__(128) unsigned char dsm[];
    constexpr int ES = sizeof(WT);
    const int rb = proj_region_bytes(ES, p.out_dim, max_splits);
    unsigned char *wsl = dsm;                                           // [out_dim][128] WT
    float *po = reinterpret_cast<float *>(dsm + rb);
    uint64_t *bar = reinterpret_cast<uint64_t *>(dsm + rb + ((p.out_dim * 4 + 15) / 16) * 16);
    const bool staged = max_splits > 0;
    const Stage st = stage_in(dsm, max_splits, bar + 1);

    const int h = blockIdx.x, b = blockIdx.y, z = blockIdx.z, Z = gridDim.z;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int c0 = z * kCombineCols;
    const int ncols = min(kCombineCols, p.v_dim - c0);
    const uint32_t row_bytes = (uint32_t)(ncols * ES);
    const bool load_w = !(p.flags & DA_FLAG_TEST_NO_TMA);
    const unsigned char *w0 = static_cast<const unsigned char *>(p.w) +
                              ((size_t)(h % p.w_heads) * p.w_head_stride + c0) * ES;
    auto copy_slice = [&]() {
        if (threadIdx.x == 0 && load_w) mbar_arrive_expect_tx(bar, row_bytes * p.out_dim);
        if (load_w)
            for (int e = threadIdx.x; e < p.out_dim; e += kCombineThreads)
                bulk_load_g2s(wsl + (size_t)e * kCombineCols * ES,
                              w0 + (size_t)e * p.w_row_stride * ES, row_bytes, bar);
    };

    if (threadIdx.x == 0) {
        mbar_init(bar, 1);
        if (staged) stage_init(st);
        fence_mbar_init();
    }
    __syncthreads();
    if (!staged) {
        copy_slice();
    } else if (load_w) {
        for (int e = threadIdx.x; e < p.out_dim; e += kCombineThreads)
            bulk_prefetch_l2(w0 + (size_t)e * p.w_row_stride * ES, row_bytes);
    }

    griddep_wait();

    float4 t;
    if (staged) {
        bool ok; // a timed-out wait leaves t zero and is recorded; the cluster still meets below
        t = staged_merge(p, h, b, z, st, true, &ok);
        // the staged blocks are read; the slice's bulk copies may overwrite them
        fence_proxy_async_smem();
        __syncthreads();
        copy_slice();
    } else {
        t = merge_columns(p, h, b, z, part);
    }
    if (warp == 0) reinterpret_cast<float4 *>(merged)[lane] = t; // zeros past v_dim
    __syncthreads();

    // every thread waits for the slice; a wait that runs out (or a slice never
    // requested, the test hook) leaves this CTA's partial sums at zero and
    // records the timeout, and the cluster still meets at both barriers
    bool have_w = load_w;
    if (have_w) {
        volatile int never = 0;
        have_w = mbar_wait_bounded(bar, 0, p.timeout_ns, &never);
    }
    if (!have_w && threadIdx.x == 0) atomicCAS(p.status, 0, kStatusTimeoutProj);

    // partial projection: warp w takes rows w, w + 8, ...; lane l its 4 columns
    const bool live = lane * 4 < ncols;
    const float4 m4 = reinterpret_cast<const float4 *>(merged)[lane];
    for (int e = warp; e < p.out_dim; e += kCombineWarps) {
        float v = 0.f;
        if (have_w && live) {
            const float4 w4 = WLoad<WT>::get(wsl + (size_t)e * kCombineCols * ES, lane * 4);
            v = fmaf(w4.x, m4.x, fmaf(w4.y, m4.y, fmaf(w4.z, m4.z, w4.w * m4.w)));
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
        if (lane == 0) po[e] = v;
    }
    __syncthreads();
    cluster_sync_all(); // every CTA's po is written and visible in the cluster

    // CTA z adds the Z partial vectors for its share of the out_dim rows
    const int per = (p.out_dim + Z - 1) / Z;
    const int e = z * per + (int)threadIdx.x;
    if ((int)threadIdx.x < per && e < p.out_dim) {
        const uint32_t a = smem_u32(po + e);
        float sum = 0.f;
        for (int r = 0; r < Z; ++r) sum += ld_cluster_f32(map_to_rank(a, r));
        OT *out = reinterpret_cast<OT *>(p.out) + ((size_t)b * p.n_heads + h) * p.out_dim + e;
        store1<OT>(out, sum);
    }
    cluster_sync_all(); // the peers have read this CTA's po
    if (!have_w && load_w) {
        // copies still in flight must land before the CTA's memory is released
        volatile int never = 0;
        (void)mbar_wait_bounded(bar, 0, p.timeout_ns, &never);
    }
}

template <typename OT>
static cudaError_t launch_staged(cudaLaunchConfig_t &cfg, const CombineParams &p, int max_splits)
{
    const int smem = combine_staged_smem_bytes(max_splits);
    cudaError_t e = cudaFuncSetAttribute(combine_staged_kernel<OT>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    cfg.dynamicSmemBytes = smem;
    return cudaLaunchKernelEx(&cfg, combine_staged_kernel<OT>, p, max_splits);
}

cudaError_t launch_combine(int out_dtype, int v_dim, const CombineParams &p, int grid_x,
                           int grid_y, cudaStream_t stream, bool pdl)
{
    if (v_dim % 4 != 0) return cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid_x, grid_y, (v_dim + kCombineCols - 1) / kCombineCols);
    cfg.blockDim = dim3(kCombineThreads, 1, 1);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    int max_splits = 0;
    for (int b = 0; b < p.batch; ++b) max_splits = p.n_splits[b] > max_splits ? p.n_splits[b] : max_splits;
    // one rank's partials in whole 128-column blocks: staged in shared memory
    if (p.n_ranks == 1 && v_dim % kCombineCols == 0 && max_splits <= kStagedMaxSplits &&
        !(p.flags & DA_FLAG_COMBINE_LOADS)) {
        switch (out_dtype) {
        case DA_F32: return launch_staged<float>(cfg, p, max_splits);
        case DA_F16: return launch_staged<__half>(cfg, p, max_splits);
        case DA_BF16: return launch_staged<__nv_bfloat16>(cfg, p, max_splits);
        default: return cudaErrorInvalidValue;
        }
    }
    switch (out_dtype) {
    case DA_F32: return cudaLaunchKernelEx(&cfg, combine_kernel<float>, p);
    case DA_F16: return cudaLaunchKernelEx(&cfg, combine_kernel<__half>, p);
    case DA_BF16: return cudaLaunchKernelEx(&cfg, combine_kernel<__nv_bfloat16>, p);
    default: return cudaErrorInvalidValue;
    }
}

template <typename OT, typename WT>
cudaError_t launch_proj_t(const CombineParams &p, int grid_x, int grid_y, cudaStream_t stream,
                          bool pdl)
{
    // the partials staged (sharing the slice's shared memory) for one rank's
    // partials in whole 128-column blocks
    int max_splits = 0;
    for (int b = 0; b < p.batch; ++b) max_splits = p.n_splits[b] > max_splits ? p.n_splits[b] : max_splits;
    if (!(p.n_ranks == 1 && p.v_dim % kCombineCols == 0 && max_splits <= kStagedMaxSplits &&
          !(p.flags & DA_FLAG_COMBINE_LOADS)))
        max_splits = 0;
    const int smem = combine_proj_smem_bytes(std::is_same<WT, float>::value ? DA_F32 : DA_BF16,
                                             p.out_dim, max_splits);
    cudaError_t e = cudaFuncSetAttribute(combine_proj_kernel<OT, WT>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    const int Z = (p.v_dim + kCombineCols - 1) / kCombineCols;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid_x, grid_y, Z);
    cfg.blockDim = dim3(kCombineThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 1;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = Z;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 2 : 1;
    return cudaLaunchKernelEx(&cfg, combine_proj_kernel<OT, WT>, p, max_splits);
}

cudaError_t launch_combine_proj(int out_dtype, int w_dtype, const CombineParams &p, int grid_x,
                                int grid_y, cudaStream_t stream, bool pdl)
{
    const int Z = (p.v_dim + kCombineCols - 1) / kCombineCols;
    if (p.v_dim % 8 != 0 || Z > 8 || p.out_dim < 1 || p.out_dim > kProjMaxOut)
        return cudaErrorInvalidValue;
    const bool bf = w_dtype == DA_BF16;
    if (!bf && w_dtype != DA_F32) return cudaErrorInvalidValue;
    switch (out_dtype) {
    case DA_F32: return bf ? launch_proj_t<float, __nv_bfloat16>(p, grid_x, grid_y, stream, pdl)
                           : launch_proj_t<float, float>(p, grid_x, grid_y, stream, pdl);
    case DA_F16: return bf ? launch_proj_t<__half, __nv_bfloat16>(p, grid_x, grid_y, stream, pdl)
                           : launch_proj_t<__half, float>(p, grid_x, grid_y, stream, pdl);
    case DA_BF16:
        return bf ? launch_proj_t<__nv_bfloat16, __nv_bfloat16>(p, grid_x, grid_y, stream, pdl)
                  : launch_proj_t<__nv_bfloat16, float>(p, grid_x, grid_y, stream, pdl);
    default: return cudaErrorInvalidValue;
    }
}

} // namespace skv
