// GQA split kernel instantiations for f32 KV storage.
#include "gqa_inst.cuh"

namespace skv {

bool gqa_config_f32(int D, int G, GqaConfig *cfg) { return gqa_config_dt<float>(D, G, cfg); }

cudaError_t gqa_launch_f32(int D, int G, int grid, cudaStream_t st, const GqaMaps &maps,
                        const SplitParams &p)
{
    return gqa_launch_dt<float>(D, G, grid, st, maps, p);
}

} // namespace skv
