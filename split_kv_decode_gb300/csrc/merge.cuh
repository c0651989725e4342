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

// One warp merges the S partials of C consecutive float4s of row `row` (value
// columns [4*c4, 4*(c4 + C))) and stores the normalised result at
// out_row + 4*c4. Lane sl*C + c takes float4 c4 + c of the splits sl,
// sl + 32/C, sl + 2*32/C, ..., NB of them in flight at a time; each lane merges
// its splits online, then the 32/C lanes of each float4 merge pairwise, so a
// unit costs one round trip to L2 for up to NB*32/C splits. The partials were
// written by other CTAs of the same launch and are read through L2.
template <int C, int NB>
__device__ __forceinline__ void warp_merge_cols(const float2 *ml, const float *acc, size_t slot0,
                                                int S, int n_rows, int row, int v_dim, int c4,
                                                void *out_row, int out_dtype)
{
    static_assert(C == 1 || C == 2 || C == 4 || C == 8 || C == 16, "C divides 32");
    constexpr int SL = 32 / C;
    const int lane = threadIdx.x & 31, c = lane % C, sl = lane / C;
    const int V4 = v_dim / 4;
    const bool live = c4 + c < V4;
    const float4 *acc4 = reinterpret_cast<const float4 *>(acc);
    float M = kNeutralM, L = 0.f;
    float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int s0 = sl; s0 < S; s0 += SL * NB) {
        float2 x[NB];
        float4 v[NB];
#pragma unroll
        for (int i = 0; i < NB; ++i) {
            const int s = s0 + i * SL;
            x[i] = make_float2(kNeutralM, 0.f);
            v[i] = make_float4(0.f, 0.f, 0.f, 0.f);
            if (s < S) {
                const size_t r = (slot0 + s) * n_rows + row;
                x[i] = __ldcg(ml + r);
                if (live) v[i] = __ldcg(acc4 + r * V4 + c4 + c);
            }
        }
#pragma unroll
        for (int i = 0; i < NB; ++i) {
            if (x[i].y > 0.f) { // a neutral partial (l = 0) takes no part
                const float mn = fmaxf(M, x[i].x);
                const float f0 = ex2((M - mn) * kLog2e), f1 = ex2((x[i].x - mn) * kLog2e);
                a.x = a.x * f0 + v[i].x * f1;
                a.y = a.y * f0 + v[i].y * f1;
                a.z = a.z * f0 + v[i].z * f1;
                a.w = a.w * f0 + v[i].w * f1;
                L = L * f0 + x[i].y * f1;
                M = mn;
            }
        }
    }
#pragma unroll
    for (int o = C; o < 32; o <<= 1) {
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
    if (sl != 0 || !live) return;
    const float inv = 1.f / L;
    a.x *= inv;
    a.y *= inv;
    a.z *= inv;
    a.w *= inv;
    void *dst = static_cast<unsigned char *>(out_row) +
                (size_t)4 * (c4 + c) * (out_dtype == DA_F32 ? 4 : 2);
    switch (out_dtype) {
    case DA_F32: store4<float>(static_cast<float *>(dst), a); break;
    case DA_F16: store4<__half>(static_cast<__half *>(dst), a); break;
    default: store4<__nv_bfloat16>(static_cast<__nv_bfloat16 *>(dst), a); break;
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
