// Instantiation and launch of the GQA split kernel for one storage type.
// Included by gqa_f32.cu / gqa_f16.cu / gqa_bf16.cu so the three storage
// types compile in parallel.
#pragma once
#include "gqa_split.cuh"

namespace skv {

constexpr int pow2_floor(int x) { return x < 2 ? 1 : 2 * pow2_floor(x / 2); }
constexpr int cmin(int a, int b) { return a < b ? a : b; }

// Tile geometry of one (storage bytes, head_dim, group) instantiation:
//   * 7 consumer warps and one producer warp (8 warps: two per SM
//     sub-partition, so the 255-register ceiling applies), one CTA per SM;
//   * rows per warp per tile P: a power of two, at most a 64 KB stage
//     (K tile + V tile) and within the register budget below; then as many
//     stages as fit in 192 KB;
//   * register budget per consumer lane: q and acc (2*G*EPL floats) plus the
//     P*G partial dots must stay under 176 floats.
template <int ES, int D, int G> struct GqaGeom {
    static constexpr int NCW = 7;
    static constexpr int EPL = D / 32;
    static constexpr int T_STAGE = 32768 / (D * ES);
    static constexpr int P = pow2_floor(cmin(T_STAGE / NCW, (176 - 2 * G * EPL) / G));
    static constexpr int T = P * NCW;
    static constexpr int NST = 196608 / (2 * T * D * ES);
};

template <typename DT, int D, int G> struct GqaInst {
    using Geo = GqaGeom<sizeof(DT), D, G>;
    using Ker = GqaKernel<DT, D, G, Geo::T, Geo::NCW, Geo::NST>;
    static void config(GqaConfig *c)
    {
        c->tile = Geo::T;
        c->ctas_per_sm = 1;
        c->smem_bytes = Ker::SMEM_ALLOC;
        c->threads = Ker::THREADS;
    }
    static cudaError_t launch(int grid, cudaStream_t st, const CUtensorMap &km,
                              const CUtensorMap &vm, const SplitParams &p)
    {
        auto *fn = gqa_split_kernel<DT, D, G, Geo::T, Geo::NCW, Geo::NST>;
        cudaError_t e =
            cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, Ker::SMEM_ALLOC);
        if (e != cudaSuccess) return e;
        fn<<<grid, Ker::THREADS, Ker::SMEM_ALLOC, st>>>(km, vm, p);
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
    SKV_CASE(256, 1) SKV_CASE(256, 2) SKV_CASE(256, 4) SKV_CASE(256, 6) SKV_CASE(256, 8)
    SKV_CASE(128, 1) SKV_CASE(128, 2) SKV_CASE(128, 4) SKV_CASE(128, 6) SKV_CASE(128, 8)
#undef SKV_CASE
    return false;
}

template <typename DT> bool gqa_config_dt(int D, int G, GqaConfig *cfg)
{
    return gqa_visit<DT>(D, G, [&](auto inst) { decltype(inst)::config(cfg); });
}

template <typename DT>
cudaError_t gqa_launch_dt(int D, int G, int grid, cudaStream_t st, const CUtensorMap &km,
                          const CUtensorMap &vm, const SplitParams &p)
{
    cudaError_t err = cudaErrorInvalidValue;
    gqa_visit<DT>(D, G, [&](auto inst) { err = decltype(inst)::launch(grid, st, km, vm, p); });
    return err;
}

} // namespace skv
