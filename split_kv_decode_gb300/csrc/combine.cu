// Combine kernel ("Kernel B"): merges the per-split partials of one
// (sequence, query head) row,
//     m = max_i m_i,  w_i = exp(m_i - m),  out = sum_i w_i acc_i / sum_i w_i l_i
// ("Attention at 128k: Split Over Context", §2; aprender issue 3725 design
// note §2). A neutral partial (l = 0, m = -1e30) gets weight 0.
//
// One CTA per (query head, sequence). Threads are laid out as Dv/4 lanes over
// the value width (float4 each) times NG groups over the splits; the groups'
// sums meet in shared memory. Launched with programmatic stream
// serialization: the CTAs may start while the split kernel drains and wait in
// griddepcontrol.wait until its partials are visible.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "internal.h"
#include "ptx.cuh"

namespace skv {

constexpr int kCombineThreads = 256;
constexpr int kCombineWChunk = 1024; // split weights staged per pass

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

__device__ __forceinline__ float block_reduce(float v, bool is_max, float *red)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float x = __shfl_xor_sync(0xffffffffu, v, o);
        v = is_max ? fmaxf(v, x) : v + x;
    }
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    __syncthreads();
    if (lane == 0) red[warp] = v;
    __syncthreads();
    v = red[0];
    for (int w = 1; w < (int)(blockDim.x >> 5); ++w) v = is_max ? fmaxf(v, red[w]) : v + red[w];
    return v;
}

template <typename OT>
__global__ void __launch_bounds__(kCombineThreads)
    combine_kernel(const __grid_constant__ CombineParams p)
{
    __shared__ float wts[kCombineWChunk];
    __shared__ float red[kCombineThreads / 32];
    __shared__ __align__(16) float part[kCombineThreads * 4];

    griddep_wait();

    const int h = blockIdx.x, b = blockIdx.y;
    const int S = p.n_splits[b];
    const size_t slot0 = (size_t)p.split_base[b];
    const int nlane = p.v_dim / 4;                  // threads across the value width
    const int ng = kCombineThreads / nlane;         // groups across the splits
    const int e4 = threadIdx.x % nlane, g = threadIdx.x / nlane;

    // pass 1: m = max_i m_i
    float mx = kNeutralM;
    for (int i = threadIdx.x; i < S; i += blockDim.x)
        mx = fmaxf(mx, p.ml[(slot0 + i) * p.n_heads + h].x);
    const float M = block_reduce(mx, true, red);

    // pass 2: weights, the merged l, and the weighted sum of acc
    float lsum = 0.f;
    float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int c0 = 0; c0 < S; c0 += kCombineWChunk) {
        const int cn = min(kCombineWChunk, S - c0);
        __syncthreads();
        for (int i = threadIdx.x; i < cn; i += blockDim.x) {
            const float2 x = p.ml[(slot0 + c0 + i) * p.n_heads + h];
            const float w = ex2((x.x - M) * kLog2e);
            wts[i] = w;
            lsum += w * x.y;
        }
        __syncthreads();
        if (g < ng) {
            for (int i = g; i < cn; i += ng) {
                const float w = wts[i];
                const float4 v = *reinterpret_cast<const float4 *>(
                    p.acc + ((slot0 + c0 + i) * p.n_heads + h) * p.v_dim + e4 * 4);
                a.x = fmaf(w, v.x, a.x);
                a.y = fmaf(w, v.y, a.y);
                a.z = fmaf(w, v.z, a.z);
                a.w = fmaf(w, v.w, a.w);
            }
        }
    }
    const float L = block_reduce(lsum, false, red);
    reinterpret_cast<float4 *>(part)[threadIdx.x] = a;
    __syncthreads();
    if (threadIdx.x < nlane) {
        float4 t = reinterpret_cast<float4 *>(part)[threadIdx.x];
        for (int gg = 1; gg < ng; ++gg) {
            const float4 u = reinterpret_cast<float4 *>(part)[gg * nlane + threadIdx.x];
            t.x += u.x; t.y += u.y; t.z += u.z; t.w += u.w;
        }
        const float inv = 1.f / L;
        t.x *= inv; t.y *= inv; t.z *= inv; t.w *= inv;
        OT *out = reinterpret_cast<OT *>(p.out) + ((size_t)b * p.n_heads + h) * p.v_dim;
        store4<OT>(out + threadIdx.x * 4, t);
    }
}

cudaError_t launch_combine(int out_dtype, int v_dim, const CombineParams &p, int grid_x,
                           int grid_y, cudaStream_t stream, bool pdl)
{
    if (v_dim % 4 != 0 || v_dim / 4 > kCombineThreads) return cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid_x, grid_y, 1);
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
