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

#include "internal.h"
#include "ptx.cuh"

namespace skv {

constexpr int kCombineThreads = 256;
constexpr int kCombineWarps = kCombineThreads / 32;
constexpr int kCombineCols = 128;   // value columns per CTA (one float4 per lane)
constexpr int kCombinePrefetch = 8; // acc vectors per lane loaded before the weights

template <typename OT> __device__ __forceinline__ void store4(OT *p, float4 v);
template <> __device__ __forceinline__ void store4<float>(float *p, float4 v)
{
    *reinterpret_cast<float4 *>(p) = v;
}
template <> __device__ __forceinline__ void store4<__half>(__half *p, float4 v)
{
    __half2 a = __floats2half2_rn(v.x, v.y), b = __floats2half2_rn(v.z, v.w);
    uint2 u;
    u.x = *reinterpret_cast<uint32_t *>(&a);
    u.y = *reinterpret_cast<uint32_t *>(&b);
    *reinterpret_cast<uint2 *>(p) = u;
}
template <> __device__ __forceinline__ void store4<__nv_bfloat16>(__nv_bfloat16 *p, float4 v)
{
    __nv_bfloat162 a = __floats2bfloat162_rn(v.x, v.y), b = __floats2bfloat162_rn(v.z, v.w);
    uint2 u;
    u.x = *reinterpret_cast<uint32_t *>(&a);
    u.y = *reinterpret_cast<uint32_t *>(&b);
    *reinterpret_cast<uint2 *>(p) = u;
}

__device__ __forceinline__ void fma4(float4 &a, float w, const float4 &v)
{
    a.x = fmaf(w, v.x, a.x);
    a.y = fmaf(w, v.y, a.y);
    a.z = fmaf(w, v.z, a.z);
    a.w = fmaf(w, v.w, a.w);
}

template <typename OT>
__global__ void __launch_bounds__(kCombineThreads)
    combine_kernel(const __grid_constant__ CombineParams p)
{
    __shared__ __align__(16) float4 part[kCombineWarps][32];

    griddep_wait();

    const int h = blockIdx.x, b = blockIdx.y;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int S = p.n_splits[b];
    const int SR = S * p.n_ranks;                            // (rank, split) pairs
    const size_t slot0 = (size_t)p.split_base[b];
    const int col = blockIdx.z * kCombineCols + lane * 4;
    const bool live = col < p.v_dim;
    // pair i = r * S + s: rank r's split s
    auto ml_of = [&](int i) {
        const int r = i / S;
        return __ldg(p.ml + r * p.rank_ml + (slot0 + (i - r * S)) * p.n_heads + h);
    };
    auto acc_of = [&](int i) {
        const int r = i / S;
        return __ldg(reinterpret_cast<const float4 *>(
            p.acc + r * p.rank_acc + ((slot0 + (i - r * S)) * p.n_heads + h) * p.v_dim + col));
    };

    // acc vectors of this warp's first pairs, in flight while m and l are formed
    float4 pv[kCombinePrefetch];
#pragma unroll
    for (int i = 0; i < kCombinePrefetch; ++i) {
        const int sp = warp + kCombineWarps * i;
        pv[i] = (live && sp < SR) ? acc_of(sp) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    // m = max_i m_i and l = sum_i e^{m_i - m} l_i, by every warp for itself
    float M = kNeutralM;
    for (int sp = lane; sp < SR; sp += 32) M = fmaxf(M, ml_of(sp).x);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    float L = 0.f;
    for (int sp = lane; sp < SR; sp += 32) {
        const float2 x = ml_of(sp);
        L = fmaf(x.y, ex2((x.x - M) * kLog2e), L);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) L += __shfl_xor_sync(0xffffffffu, L, o);

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
    if (warp == 0 && live) {
        float4 t = part[0][lane];
#pragma unroll
        for (int w = 1; w < kCombineWarps; ++w) {
            const float4 u = part[w][lane];
            t.x += u.x; t.y += u.y; t.z += u.z; t.w += u.w;
        }
        const float inv = 1.f / L;
        t.x *= inv; t.y *= inv; t.z *= inv; t.w *= inv;
        OT *out = reinterpret_cast<OT *>(p.out) + ((size_t)b * p.n_heads + h) * p.v_dim + col;
        store4<OT>(out, t);
    }
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
    switch (out_dtype) {
    case DA_F32: return cudaLaunchKernelEx(&cfg, combine_kernel<float>, p);
    case DA_F16: return cudaLaunchKernelEx(&cfg, combine_kernel<__half>, p);
    case DA_BF16: return cudaLaunchKernelEx(&cfg, combine_kernel<__nv_bfloat16>, p);
    default: return cudaErrorInvalidValue;
    }
}

} // namespace skv
