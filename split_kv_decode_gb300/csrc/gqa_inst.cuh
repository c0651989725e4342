// Instantiation and launch of the GQA split kernel for one storage type.
// Included by gqa_f32.cu / gqa_f16.cu / gqa_bf16.cu so the three storage
// types compile in parallel.
#pragma once
#include "gqa_split.cuh"

namespace skv {

constexpr int pow2_floor(int x) { return x < 2 ? 1 : 2 * pow2_floor(x / 2); }
constexpr int cmin(int a, int b) { return a < b ? a : b; }

// Tile geometry of one (storage bytes, head_dim, group) instantiation.
//
// The consumers are latency-bound (shuffle and shared-load chains per tile),
// so more consumer warps per SM help as long as their registers fit:
//   * preferred: 11 consumer warps + 1 producer (12 warps per SM, 3 per
//     sub-partition: a 168-register ceiling); used when the estimated
//     register need 2*G*EPL (q, acc) + P*G (partial dots) + 64 fits with at
//     least 2 rows per warp and a stage of at most 48 KB;
//   * otherwise 7 consumer warps + 1 producer (8 warps: 255-register ceiling)
//     with rows per warp P under a 176-float budget and a stage of at most
//     64 KB;
//   * then as many stages (2..6) as fit in 180 KB of shared memory.
// P (rows per warp per tile) is a power of two.
// Rows of 256 bytes (D = 128 in a 16-bit type) are read by half-warps, two rows
// at a time (LPR = 16 lanes per row, 16-byte loads): twice the q and acc
// registers per lane (EPL = D / LPR) but half the dot registers per row, so
// it is used for G <= 4 only.
constexpr int gqa_reg_est(int PH, int G, int EPL) { return 2 * G * EPL + PH * G + 64; }

template <int ES, int D, int G> struct GqaGeom {
    static constexpr int LPR = (D * ES == 256 && G <= 4) ? 16 : 32;
    static constexpr int RPW = 32 / LPR;
    static constexpr int EPL = D / LPR;
    static constexpr int B11 = (168 - 64 - 2 * G * EPL) / G; // dot registers per head
    static constexpr int P11 = pow2_floor(cmin(B11 > 0 ? RPW * B11 : 0, 49152 / (2 * 11 * D * ES)));
    static constexpr bool WIDE = B11 >= 2 && P11 >= 2 * RPW && (P11 * G) % 4 == 0;
    static constexpr int NCW = WIDE ? 11 : 7;
    static constexpr int P =
        WIDE ? P11 : pow2_floor(cmin(65536 / (2 * 7 * D * ES), RPW * ((176 - 2 * G * EPL) / G)));
    static constexpr int T = P * NCW;
    static constexpr int STAGE = 2 * T * D * ES;
    static constexpr int NST = cmin(6, 184320 / STAGE);
    static_assert(NST >= 2, "at least two stages");
    static_assert(P % RPW == 0, "whole row steps");
    // a paged tile that spans a block end is T / gcd(T, block_size) boxes, at
    // most T / gcd(T, 16) = NCW when P <= 16: one per lane of the producer warp
    static_assert(P <= 16 && NCW <= 32, "paged boxes per tile");
    static_assert(!WIDE || gqa_reg_est(P / RPW, G, EPL) <= 168, "register estimate");
};

template <typename DT, int D, int G> struct GqaInst {
    using Geo = GqaGeom<sizeof(DT), D, G>;
    using Ker = GqaKernel<DT, D, G, Geo::T, Geo::NCW, Geo::NST, Geo::LPR>;
    static void config(GqaConfig *c)
    {
        c->tile = Geo::T;
        c->ctas_per_sm = 1;
        c->smem_bytes = Ker::SMEM_ALLOC;
        c->threads = Ker::THREADS;
    }
    static cudaError_t launch(int grid, cudaStream_t st, const GqaMaps &maps,
                              const SplitParams &p)
    {
        auto *fn = gqa_split_kernel<DT, D, G, Geo::T, Geo::NCW, Geo::NST, Geo::LPR>;
        cudaError_t e =
            cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, Ker::SMEM_ALLOC);
        if (e != cudaSuccess) return e;
        fn<<<grid, Ker::THREADS, Ker::SMEM_ALLOC, st>>>(maps, p);
        return cudaGetLastError();
    }
};

// Calls F::template run<GqaInst<DT, D, G>>() for a supported (D, G); false if unsupported.
template <typename DT, typename F> bool gqa_visit(int D, int G, F &&f)
{
#define SKV_CASE(d, g)                                                                           \
    if (D == d && G == g) {                                                                      \
        f(GqaInst<DT, d, g>{});                                                                  \
        return true;                                                                             \
    }
    SKV_CASE(256, 1) SKV_CASE(256, 2) SKV_CASE(256, 3) SKV_CASE(256, 4) SKV_CASE(256, 5)
    SKV_CASE(256, 6) SKV_CASE(256, 7) SKV_CASE(256, 8)
    SKV_CASE(128, 1) SKV_CASE(128, 2) SKV_CASE(128, 3) SKV_CASE(128, 4) SKV_CASE(128, 5)
    SKV_CASE(128, 6) SKV_CASE(128, 7) SKV_CASE(128, 8)
#undef SKV_CASE
    return false;
}

template <typename DT> bool gqa_config_dt(int D, int G, GqaConfig *cfg)
{
    return gqa_visit<DT>(D, G, [&](auto inst) { decltype(inst)::config(cfg); });
}

template <typename DT>
cudaError_t gqa_launch_dt(int D, int G, int grid, cudaStream_t st, const GqaMaps &maps,
                          const SplitParams &p)
{
    cudaError_t err = cudaErrorInvalidValue;
    gqa_visit<DT>(D, G, [&](auto inst) { err = decltype(inst)::launch(grid, st, maps, p); });
    return err;
}

} // namespace skv
