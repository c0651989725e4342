// The merge of split partials, for the combine kernel and for split kernels
// that merge their own partials (no second launch), plus the arrival counters
// those split kernels use to find out when every partial of a group is in.
//
// Merge ("Attention at 128k: Split Over Context", §2; aprender issue 3725
// design note §2): for one (sequence, row),
//     m = max_i m_i,  w_i = exp(m_i - m),  out = sum_i w_i acc_i / sum_i w_i l_i,
// where a neutral partial (l = 0) gets weight 0 and its acc is not read.
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "internal.h"
#include "ptx.cuh"

namespace skv {

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

// One warp merges the S partials of row `row` of the slots slot0 .. slot0+S-1
// over the 128 value columns [col0, col0 + 128), a float4 per lane, and stores
// the normalised result at out_row + col0 in the output type. The partials were
// written by other CTAs of the same launch, so they are read through L2 (.cg),
// after the arrival that made them visible.
__device__ __forceinline__ void warp_merge_row(const float2 *ml, const float *acc, size_t slot0,
                                               int S, int n_rows, int row, int v_dim, int col0,
                                               void *out_row, int out_dtype)
{
    const int lane = threadIdx.x & 31;
    const int col = col0 + lane * 4;
    const bool live = col < v_dim;
    // m = max_i m_i and l = sum_i e^{m_i - m} l_i: each lane merges its splits
    // online, then the lanes merge theirs pairwise (all lanes end equal)
    float M = kNeutralM, L = 0.f;
    for (int s = lane; s < S; s += 32) {
        const float2 x = __ldcg(ml + (slot0 + s) * n_rows + row);
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
    // sum_i w_i acc_i, eight splits' loads in flight at a time
    float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
    const float4 *acc4 = reinterpret_cast<const float4 *>(acc);
    const size_t stride = (size_t)n_rows * v_dim / 4;    // float4s between slots
    const size_t base = ((slot0 * n_rows + row) * (size_t)v_dim + (live ? col : col0)) / 4;
    for (int s0 = 0; s0 < S; s0 += 8) {
        float2 x[8];
        float4 v[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int s = min(s0 + i, S - 1);
            x[i] = __ldcg(ml + (slot0 + s) * n_rows + row);
            v[i] = __ldcg(acc4 + base + (size_t)s * stride);
        }
#pragma unroll
        for (int i = 0; i < 8; ++i)
            if (s0 + i < S && x[i].y > 0.f) fma4(a, ex2((x[i].x - M) * kLog2e), v[i]);
    }
    if (!live) return;
    const float inv = 1.f / L;
    a.x *= inv;
    a.y *= inv;
    a.z *= inv;
    a.w *= inv;
    switch (out_dtype) {
    case DA_F32: store4<float>(static_cast<float *>(out_row) + col, a); break;
    case DA_F16: store4<__half>(static_cast<__half *>(out_row) + col, a); break;
    default: store4<__nv_bfloat16>(static_cast<__nv_bfloat16 *>(out_row) + col, a); break;
    }
}

// One warp merges the S partials of one float4 of row `row` (value columns
// [4*c4, 4*c4 + 4)) and stores the normalised result at out_row + 4*c4: the
// lanes take the splits (all of them in flight at once for S <= 32), each
// lane merges its splits online and the lanes merge pairwise. The partials
// were written by other CTAs of the same launch and are read through L2.
__device__ __forceinline__ void warp_merge_float4(const float2 *ml, const float *acc, size_t slot0,
                                                  int S, int n_rows, int row, int v_dim, int c4,
                                                  void *out_row, int out_dtype)
{
    const int lane = threadIdx.x & 31;
    float M = kNeutralM, L = 0.f;
    float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
    const float4 *acc4 = reinterpret_cast<const float4 *>(acc);
    for (int s = lane; s < S; s += 32) {
        const size_t r = (slot0 + s) * n_rows + row;
        const float2 x = __ldcg(ml + r);
        const float4 v = __ldcg(acc4 + r * (v_dim / 4) + c4);
        if (x.y > 0.f) {
            const float mn = fmaxf(M, x.x);
            const float f0 = ex2((M - mn) * kLog2e), f1 = ex2((x.x - mn) * kLog2e);
            a.x = a.x * f0 + v.x * f1;
            a.y = a.y * f0 + v.y * f1;
            a.z = a.z * f0 + v.z * f1;
            a.w = a.w * f0 + v.w * f1;
            L = L * f0 + x.y * f1;
            M = mn;
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float Mo = __shfl_xor_sync(0xffffffffu, M, o);
        const float Lo = __shfl_xor_sync(0xffffffffu, L, o);
        const float ax = __shfl_xor_sync(0xffffffffu, a.x, o);
        const float ay = __shfl_xor_sync(0xffffffffu, a.y, o);
        const float az = __shfl_xor_sync(0xffffffffu, a.z, o);
        const float aw = __shfl_xor_sync(0xffffffffu, a.w, o);
        const float mn = fmaxf(M, Mo);
        const float f0 = ex2((M - mn) * kLog2e), f1 = ex2((Mo - mn) * kLog2e);
        a.x = a.x * f0 + ax * f1;
        a.y = a.y * f0 + ay * f1;
        a.z = a.z * f0 + az * f1;
        a.w = a.w * f0 + aw * f1;
        L = L * f0 + Lo * f1;
        M = mn;
    }
    if (lane != 0) return;
    const float inv = 1.f / L;
    a.x *= inv;
    a.y *= inv;
    a.z *= inv;
    a.w *= inv;
    switch (out_dtype) {
    case DA_F32: store4<float>(static_cast<float *>(out_row) + 4 * c4, a); break;
    case DA_F16: store4<__half>(static_cast<__half *>(out_row) + 4 * c4, a); break;
    default: store4<__nv_bfloat16>(static_cast<__nv_bfloat16 *>(out_row) + 4 * c4, a); break;
    }
}

// Output row `row` of sequence b in the [B][rows][v_dim] output.
__device__ __forceinline__ void *out_row_ptr(const FusedOut &f, int b, int rows, int row,
                                             int v_dim)
{
    const size_t es = f.out_dtype == DA_F32 ? 4 : 2;
    return static_cast<unsigned char *>(f.out) + ((size_t)b * rows + row) * v_dim * es;
}

// One arrival on a counter that the library zeroes at the start of every call
// (a memset on the same stream): returns the count including this arrival. One
// atomic add per arrival, so arrivals that come together do not retry.
__device__ __forceinline__ uint32_t arrive(uint32_t *ctr) { return atomicAdd(ctr, 1u) + 1u; }

} // namespace skv
