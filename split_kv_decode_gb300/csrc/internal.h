// Internal declarations shared by the host side of the library (api.cpp,
// plan.cpp) and the kernel translation units. Not part of the C ABI.
#pragma once
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "split_kv_decode.h"

namespace skv {

// Workspace layout (all offsets from the workspace base, bytes):
//   [0, 256)                status header: int32 status word at offset 0
//   [256, 256 + ml_bytes)   float2 (m, l) per (slot, query head)
//   then                    float acc[slot][n_heads][v_dim]
//   then                    uint32 arrival counters, zeroed by the library at the
//                           start of a call that uses them: one per (sequence,
//                           KV head) group, at least two
// A slot is one split of one sequence: slot = split_base[b] + s.
constexpr int64_t kWsHeader = 256;

inline int64_t ws_ml_offset() { return kWsHeader; }
inline int64_t ws_acc_offset(int64_t total_splits, int n_heads)
{
    int64_t ml = total_splits * n_heads * 8;
    return kWsHeader + ((ml + 255) / 256) * 256;
}
inline int64_t ws_ctr_offset(int64_t total_splits, int n_heads, int v_dim)
{
    const int64_t t = ws_acc_offset(total_splits, n_heads) + total_splits * n_heads * v_dim * 4;
    return (t + 255) / 256 * 256;
}
inline int64_t ws_counters(int batch, int n_kv_heads)
{
    const int64_t n = (int64_t)batch * n_kv_heads;
    return n < 2 ? 2 : n;
}
// rounded to 256 bytes, so that workspaces placed back to back (one per rank
// of a context-parallel step) keep every region aligned
inline int64_t ws_total(int64_t total_splits, int n_heads, int v_dim, int64_t n_counters)
{
    return ws_ctr_offset(total_splits, n_heads, v_dim) + (n_counters * 4 + 255) / 256 * 256;
}

// A split kernel that merges its own partials (no combine launch): the last
// partial of a (sequence, KV head) group to arrive merges the group's rows
// (GQA kernels); every CTA merges a share of the rows once all CTAs have
// arrived (MLA tensor-core kernel).
struct FusedOut {
    void *out;                   // [B][rows][v_dim] in out_dtype
    uint32_t *ctr;               // arrival counters (workspace tail), zero at launch
    int32_t out_dtype;           // DA_F32 / DA_F16 / DA_BF16
    int32_t on;                  // 0: partials only (a combine launch merges them)
};

// Status word codes written by kernels (low byte = da_status_t, next byte = kernel).
constexpr int kStatusTimeoutGqa = DA_ETIMEOUT | (DA_KERNEL_GQA_TMA << 8);
constexpr int kStatusTimeoutMla = DA_ETIMEOUT | (DA_KERNEL_MLA_TC << 8);
constexpr int kStatusTimeoutTc = DA_ETIMEOUT | (DA_KERNEL_GQA_TC << 8);
constexpr int kStatusTimeoutProj = DA_ETIMEOUT | (15 << 8); // combine with the projection
constexpr int kStatusTimeoutCombine = DA_ETIMEOUT | (14 << 8); // staged combine

// Per-launch description of the work items shared by the split kernels.
struct ItemTable {
    int32_t batch;
    int32_t n_items;
    int32_t n_kv_heads;
    int32_t row_groups;      // SIMT GQA kernel: the rows of a (sequence, KV head, split)
                             // are cut into this many groups, one work item each (1 elsewhere)
    int32_t seq_lens[DA_MAX_BATCH];
    int32_t chunk[DA_MAX_BATCH];
    int32_t split_base[DA_MAX_BATCH + 1];
};

struct SplitParams {
    const float *q;          // [B][q_len][hq][Dk]
    float2 *ml;              // workspace (m, l) per (slot, row)
    float *acc;              // workspace acc per (slot, row, Dv)
    int *status;             // workspace status word
    int32_t n_heads;         // rows per sequence: q_len * hq (query token, head)
    int32_t q_len;           // query tokens per sequence (causal among them)
    int32_t hq;              // query heads per token
    float scale_log2;        // scale * log2(e)
    uint64_t timeout_ns;
    int32_t flags;
    // Optional, read on the device (so that one captured launch serves changing
    // contexts): current lengths (each clamped to [1, items.seq_lens[b]]), and
    // a block table for paged caches. NULL: the plan's lengths / contiguous caches.
    FusedOut fused;
    const int32_t *dev_lens;
    const int32_t *block_table; // [batch][max_blocks] pool block of each block_size positions
    int32_t max_blocks;
    int32_t block_size;
    int32_t oob_block;       // a block coordinate past the pool: TMA fills zeros there
    int32_t box_rows;        // paged: gcd(tile, block_size), so no box of box_rows rows
                             // that starts at a multiple of box_rows spans two blocks
    ItemTable items;
};

struct MlaParams {
    const float *q;          // [B][Hq][576]
    const void *cache;       // latent rows (f32, f16 or bf16): element (b, pos, d) at
                             // b*batch_stride + pos*pos_stride + d (elements)
    int64_t pos_stride;      // elements between positions (>= 576)
    int64_t batch_stride;    // elements between sequences
    float2 *ml;              // workspace (m, l) per (slot, head)
    float *acc;              // workspace acc per (slot, head, 512)
    int *status;             // workspace status word
    int32_t n_heads;         // rows per sequence: q_len * hq (query token, head), token-major
    int32_t q_len;           // query tokens per sequence (causal among them)
    int32_t hq;              // query heads per token
    float scale_log2;        // scale * log2(e)
    uint64_t timeout_ns;
    int32_t flags;
    // Optional, as for the GQA kernel: current lengths read on the device, and
    // a block table over a pool of latent rows (row (block, slot) at
    // cache + block * block_stride + slot * pos_stride).
    const int32_t *dev_lens;
    const int32_t *block_table;
    int32_t max_blocks;
    int32_t block_size;
    int64_t block_stride;
    // Which kernel serves a sequence, decided on the device from its current
    // length L (the plan's, or the one read from dev_lens): the f32 kernel when
    // L < exact_below, else the tensor-core kernel. Each kernel skips the other's
    // sequences entirely (it writes nothing for them).
    int32_t exact_below;
    int32_t reset_status;    // the exact kernel runs alone in this call: it clears the status word
    FusedOut fused;
    ItemTable items;         // n_kv_heads = 1
};

// MLA tensor-core split kernel: rows per CTA = rows / 2 (a 2-CTA cluster
// shares every tile); supported rows (heads x q_len): 32, 64, 96, 128; an f32,
// f16 or bf16 latent cache (kv_dtype).
bool mla_supported_heads(int n_heads);
int mla_smem_bytes(int n_heads);
cudaError_t launch_mla_split(int grid, cudaStream_t stream, const MlaParams &p, int kv_dtype);
// 2-CTA clusters of the MLA tensor-core kernel the current device holds at once
// (0 if unknown): its merge without a combine launch needs every cluster resident.
int mla_max_clusters(int n_heads);
// Split kernel in f32 on the CUDA cores (f32_split.cu): MLA sequences below the
// exactness threshold. One CTA per (work item, group of 32 rows): grid =
// n_items * f32_split_groups(rows per item).
struct F32Params {
    const float *q;          // [B][q_len][hq][DK]
    const float *k, *v;      // f32 caches; for MLA v == k (values: the first DV columns)
    int64_t k_pos_stride, k_head_stride, k_batch_stride, k_block_stride; // elements
    int64_t v_pos_stride, v_head_stride, v_batch_stride, v_block_stride;
    float2 *ml;
    float *acc;
    int *status;
    int32_t n_heads;         // rows per sequence: q_len * hq
    int32_t q_len;
    int32_t hq;
    float scale_log2;
    int32_t flags;
    int32_t exact_below;     // sequences at or past this current length are skipped
    int32_t reset_status;    // this kernel runs alone in the call: it clears the status word
    const int32_t *dev_lens;
    const int32_t *block_table;
    int32_t max_blocks;
    int32_t block_size;
    ItemTable items;
};
int f32_split_groups(int rows_per_item);
cudaError_t launch_f32_split(int head_dim, int v_dim, bool shared_kv, int grid,
                             cudaStream_t stream, const F32Params &p);

struct CombineParams {
    const float2 *ml;
    const float *acc;
    void *out;
    int32_t n_heads;
    int32_t v_dim;
    int32_t batch;
    // partials of n_ranks ranks that ran the same plan, workspaces back to back:
    // rank r's (m, l) at ml + r * rank_ml, its acc at acc + r * rank_acc
    int32_t n_ranks;
    int64_t rank_ml;
    int64_t rank_acc;
    // the per-head output projection of combine_proj_kernel: out row e of row h
    // is sum_c w[(h % w_heads) * w_head_stride + e * w_row_stride + c] * merged[c]
    const void *w;
    int64_t w_head_stride;
    int64_t w_row_stride;
    int32_t out_dim;
    int32_t w_heads;
    int *status;             // workspace status word (a timed-out weight load)
    uint64_t timeout_ns;
    int32_t flags;
    int32_t n_splits[DA_MAX_BATCH];
    int32_t split_base[DA_MAX_BATCH];
};

// Tensor-core GQA kernel (gqa_tc.cu): tiles of tc_tile(D) positions;
// shared-memory layout for head_dim D and R rows per item (the same on host
// and device). 64-position tiles beat 32-position ones with twice the stages
// (117 against 179 us for 8 rows at D = 256): the per-tile hand-offs, not the
// ring depth, set the pace.
__host__ __device__ constexpr int tc_tile(int) { return 64; }
constexpr int kTcMaxStages = 6;
constexpr int kTcBarriers = 32;
constexpr int kTcSmemMax = 232448;
struct TcLayout {
    int chunk_bytes;  // one 64-column chunk of a tile: tc_tile(D) rows of 128 B
    int tile_bytes;   // K (or V) tile: D / 64 chunks
    int stage_bytes;  // K + V
    int rpad, npv;    // rows rounded up to 8 (Q rows written), to 16 (PV N)
    int qch;          // one 64-column chunk of Q: rpad rows of 128 B
    int pslot;        // one P buffer: npv rows of 128 B
    int nst;          // stages
    int q_off, stage_off, p_off, bar_off, misc_off, alpha_off, used;
};
__host__ __device__ inline TcLayout tc_layout(int D, int R)
{
    TcLayout L;
    L.chunk_bytes = tc_tile(D) * 128;
    L.tile_bytes = (D / 64) * L.chunk_bytes;
    L.stage_bytes = 2 * L.tile_bytes;
    L.rpad = (R + 7) / 8 * 8;
    L.npv = (R + 15) / 16 * 16;
    L.qch = L.rpad * 128;
    L.pslot = L.npv * 128;
    // Q comes first: the 128-row MMA reads 128 rows from the start of every Q
    // chunk, so past the last one it reads into the first stage (rows whose
    // scores nobody reads)
    L.q_off = 0;
    const int qbytes = (D / 64) * L.qch;
    const int stages_off = (qbytes + 1023) / 1024 * 1024;
    const int rest = 2 * L.pslot + kTcBarriers * 8 + 16 + 128 * 4 + 1024;
    int nst = (kTcSmemMax - stages_off - rest) / L.stage_bytes;
    L.nst = nst > kTcMaxStages ? kTcMaxStages : nst;
    L.stage_off = stages_off;
    L.p_off = stages_off + L.nst * L.stage_bytes;
    L.bar_off = L.p_off + 2 * L.pslot;
    L.misc_off = L.bar_off + kTcBarriers * 8;
    L.alpha_off = L.misc_off + 16;
    L.used = L.alpha_off + 128 * 4;
    return L;
}
cudaError_t launch_gqa_tc(int kv_dtype, int head_dim, int grid, cudaStream_t st,
                          const CUtensorMap &km, const CUtensorMap &vm, const SplitParams &p);

// TMA maps of the SIMT GQA kernel: k and v copy a whole tile of T rows; for a
// paged pool kb and vb copy box_rows rows, the boxes of a tile that spans a
// block end (contiguous caches: left zero, unused).
struct GqaMaps {
    CUtensorMap k, v, kb, vb;
};
// Static configuration of a GQA instantiation (tile rows, CTAs per SM, smem).
struct GqaConfig {
    int tile;
    int ctas_per_sm;
    int smem_bytes;
    int threads;
};
bool gqa_config(int kv_dtype, int head_dim, int group, GqaConfig *cfg);

cudaError_t launch_combine(int out_dtype, int v_dim, const CombineParams &p, int grid_x,
                           int grid_y, cudaStream_t stream, bool pdl);
// combine fused with the per-head output projection: clusters of ceil(v_dim /
// 128) CTAs (at most 8), each merging 128 columns and projecting them
constexpr int kProjMaxOut = 256;
constexpr int kProjMaxVdim = 1024;
cudaError_t launch_combine_proj(int out_dtype, int w_dtype, const CombineParams &p, int grid_x,
                                int grid_y, cudaStream_t stream, bool pdl);

} // namespace skv
