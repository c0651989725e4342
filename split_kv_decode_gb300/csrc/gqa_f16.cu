// GQA split kernel instantiations for f16 KV storage.
#include "gqa_inst.cuh"

namespace skv {

bool gqa_config_f16(int D, int G, GqaConfig *cfg) { return gqa_config_dt<__half>(D, G, cfg); }

cudaError_t gqa_launch_f16(int D, int G, int grid, cudaStream_t st, const GqaMaps &maps,
                        const SplitParams &p)
{
    return gqa_launch_dt<__half>(D, G, grid, st, maps, p);
}

} // namespace skv
