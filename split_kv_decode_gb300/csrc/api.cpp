// C ABI of libsplitkv.so: argument validation, planning, TMA descriptors,
// launches with a per-phase launch guard, and the short form's per-device
// workspace.
//
// Launch guard: every launch is followed by cudaGetLastError(), and a failure
// is reported with the phase that raised it ("Attention at 128k" §5.3: poll
// per phase so a bad launch is reported where it happened, not at some later
// collective).
#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <numeric>
#include <mutex>
#include <string>
#include <vector>

#include "internal.h"
#include "plan_internal.h"

namespace skv {

bool gqa_config_f32(int D, int G, GqaConfig *cfg);
bool gqa_config_f16(int D, int G, GqaConfig *cfg);
bool gqa_config_bf16(int D, int G, GqaConfig *cfg);
cudaError_t gqa_launch_f32(int D, int G, int grid, cudaStream_t st,
                           const GqaMaps &maps, const SplitParams &p);
cudaError_t gqa_launch_f16(int D, int G, int grid, cudaStream_t st,
                           const GqaMaps &maps, const SplitParams &p);
cudaError_t gqa_launch_bf16(int D, int G, int grid, cudaStream_t st,
                           const GqaMaps &maps, const SplitParams &p);

namespace {

thread_local std::string g_err;

int fail(int code, const char *phase, const char *fmt, ...)
{
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    g_err = std::string(phase) + ": " + buf;
    return code;
}

int dtype_size(int dt)
{
    switch (dt) {
    case DA_F32: return 4;
    case DA_F16:
    case DA_BF16: return 2;
    default: return 0;
    }
}

const char *dtype_name(int dt)
{
    switch (dt) {
    case DA_F32: return "f32";
    case DA_F16: return "f16";
    case DA_BF16: return "bf16";
    default: return "?";
    }
}

bool gqa_config_any(int dt, int D, int G, GqaConfig *cfg)
{
    switch (dt) {
    case DA_F32: return gqa_config_f32(D, G, cfg);
    case DA_F16: return gqa_config_f16(D, G, cfg);
    case DA_BF16: return gqa_config_bf16(D, G, cfg);
    default: return false;
    }
}

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

// query tokens per sequence, and rows (query token, head) of the workspace and out
int q_len_of(const da_args_t *a) { return a->q_len > 1 ? a->q_len : 1; }
int rows_of(const da_args_t *a) { return a->n_heads * q_len_of(a); }

int check_args(const da_args_t *a)
{
    if (!a) return fail(DA_EINVAL, "args", "args is NULL");
    if (a->batch < 1 || a->batch > DA_MAX_BATCH)
        return fail(DA_EINVAL, "args", "batch %d outside [1, %d]", a->batch, DA_MAX_BATCH);
    if (a->n_heads < 1 || a->n_kv_heads < 1)
        return fail(DA_EINVAL, "args", "n_heads %d / n_kv_heads %d must be >= 1", a->n_heads,
                    a->n_kv_heads);
    if (a->n_heads % a->n_kv_heads)
        return fail(DA_EINVAL, "args", "n_heads %d is not a multiple of n_kv_heads %d",
                    a->n_heads, a->n_kv_heads);
    if (a->head_dim < 1 || a->v_dim < 1 || a->v_dim > 1024)
        return fail(DA_EINVAL, "args", "head_dim %d / v_dim %d out of range", a->head_dim,
                    a->v_dim);
    if (a->capacity < 1) return fail(DA_EINVAL, "args", "capacity %d < 1", a->capacity);
    if (!dtype_size(a->kv_dtype)) return fail(DA_EINVAL, "args", "kv_dtype %d", a->kv_dtype);
    if (!dtype_size(a->out_dtype)) return fail(DA_EINVAL, "args", "out_dtype %d", a->out_dtype);
    if (!std::isfinite(a->scale)) return fail(DA_EINVAL, "args", "scale is not finite");
    if (a->k_pos_stride < 1 || a->k_head_stride < 1 || a->v_pos_stride < 1 ||
        a->v_head_stride < 1 || a->k_batch_stride < 0 || a->v_batch_stride < 0)
        return fail(DA_EINVAL, "args", "cache strides must be positive");
    if (a->batch > 1 && (a->k_batch_stride < 1 || a->v_batch_stride < 1))
        return fail(DA_EINVAL, "args", "batch strides must be positive when batch > 1");
    if (a->force_splits < 0) return fail(DA_EINVAL, "args", "force_splits < 0");
    if (a->timeout_us < 0) return fail(DA_EINVAL, "args", "timeout_us < 0");
    if (a->q_len < 0 || a->q_len > 64) return fail(DA_EINVAL, "args", "q_len %d outside [0, 64]", a->q_len);
    if ((a->flags & DA_FLAG_MLA_SIMT) && (a->flags & DA_FLAG_MLA_TC))
        return fail(DA_EINVAL, "args", "DA_FLAG_MLA_SIMT and DA_FLAG_MLA_TC exclude each other");
    return DA_OK;
}

// Does a split + combine call let the split kernel merge its own partials?
// Only when the caller asks for one launch (and never for a split-only call).
bool want_fuse(const da_args_t *a)
{
    return (a->flags & DA_FLAG_ONE_LAUNCH) && !(a->flags & DA_FLAG_NO_COMBINE);
}

// MLA: sequences shorter than this (current length) run on the f32
// CUDA-core kernel, the others on the tensor-core kernel
int mla_exact_below(const da_args_t *a)
{
    if (a->kv_dtype != DA_F32) return 0; // 16-bit caches: the stored values are the operands
    if (a->flags & DA_FLAG_MLA_SIMT) return INT32_MAX;
    if (a->flags & DA_FLAG_MLA_TC) return 0;
    return DA_MLA_EXACT_BELOW;
}

struct KernelChoice {
    int kernel;
    int tile;        // planner quantum: chunks are multiples of it
    int ctas_per_sm;
    int cluster;     // CTAs that share one work item
    int row_groups = 1; // SIMT GQA kernel: work items per (sequence, KV head, split)
};

// Rows of a (sequence, KV head) group that one SIMT work item holds when the
// group has more than 8: the largest divisor of the group's rows up to 8.
int simt_rows_per_item(int rows)
{
    for (int g = 8; g > 1; --g)
        if (rows % g == 0) return g;
    return 1;
}

// Work items per (sequence, KV head, split) on the SIMT kernel: more than one
// for an f32 cache whose groups hold 9 to 128 rows (16-bit caches take such
// groups on the tensor cores)
int simt_row_groups(const da_args_t *a)
{
    const int G = a->n_heads / a->n_kv_heads * (a->q_len > 1 ? a->q_len : 1);
    if (a->kv_dtype == DA_F32 && (a->head_dim == 128 || a->head_dim == 256) && G > 8 &&
        G <= 128)
        return G / simt_rows_per_item(G);
    return 1;
}

int select_kernel(const da_args_t *a, KernelChoice *kc)
{
    // the GQA kernel serves the q_len tokens of a group as extra rows
    const int G = a->n_heads / a->n_kv_heads * q_len_of(a);
    const int es = dtype_size(a->kv_dtype);
    if (a->head_dim == 576 && a->v_dim == 512 && a->n_kv_heads == 1) {
        // the rows of an item are (query token, head) pairs, like heads of MQA
        if (!mla_supported_heads(rows_of(a)))
            return fail(DA_EUNSUPPORTED, "plan",
                        "the MLA kernel serves 32, 64, 96 or 128 query rows (heads x q_len; "
                        "got %d)",
                        rows_of(a));
        if (a->k_pos_stride < 576 || (a->k_pos_stride * es) % 16 ||
            (a->batch > 1 && (a->k_batch_stride * es) % 16))
            return fail(DA_EUNSUPPORTED, "plan",
                        "MLA latent rows need >= 576 elements and 16-byte aligned strides");
        if ((a->flags & DA_FLAG_MLA_SIMT) && a->kv_dtype != DA_F32)
            return fail(DA_EUNSUPPORTED, "plan",
                        "DA_FLAG_MLA_SIMT: the f32 CUDA-core MLA kernel reads an f32 cache");
        if (a->v_pos_stride != a->k_pos_stride || (a->batch > 1 && a->v_batch_stride != a->k_batch_stride))
            return fail(DA_EUNSUPPORTED, "plan",
                        "MLA values must be the first 512 columns of the key rows (same strides)");
        kc->kernel = DA_KERNEL_MLA_TC;
        kc->tile = 16;
        kc->ctas_per_sm = 1;
        kc->cluster = 2;
        return DA_OK;
    }
    if (a->head_dim != a->v_dim)
        return fail(DA_EUNSUPPORTED, "plan", "GQA kernel needs v_dim == head_dim (got %d, %d)",
                    a->head_dim, a->v_dim);
    const int64_t st[6] = {a->k_pos_stride, a->k_head_stride, a->v_pos_stride,
                           a->v_head_stride, a->batch > 1 ? a->k_batch_stride : 0,
                           a->batch > 1 ? a->v_batch_stride : 0};
    for (int i = 0; i < 6; ++i)
        if ((st[i] * es) % 16)
            return fail(DA_EUNSUPPORTED, "plan",
                        "cache strides must be multiples of 16 bytes for TMA tiles");
    // many rows per item on a 16-bit cache: the tensor-core kernel
    const bool tc_shape = es == 2 && (a->head_dim == 128 || a->head_dim == 256) && G >= 8 &&
                          G <= 128;
    if (tc_shape && !(G == 8 && (a->flags & DA_FLAG_GQA_SIMT))) {
        kc->kernel = DA_KERNEL_GQA_TC;
        kc->tile = tc_tile(a->head_dim);
        kc->ctas_per_sm = 1;
        kc->cluster = 1;
        return DA_OK;
    }
    // more rows per group than the SIMT kernel holds (an f32 cache): the group's
    // rows are cut into row groups of up to 8, one work item each; the items of a
    // slice run side by side, so the slice is read from HBM once and from L2 again
    kc->row_groups = simt_row_groups(a);
    const int g = G / kc->row_groups;
    GqaConfig cfg;
    if (!gqa_config_any(a->kv_dtype, a->head_dim, g, &cfg))
        return fail(DA_EUNSUPPORTED, "plan",
                    "no GQA kernel for head_dim %d, group %d (heads per KV head x q_len), "
                    "%s KV (head_dim 128 or 256; group 1 to 128)",
                    a->head_dim, G, dtype_name(a->kv_dtype));
    kc->kernel = DA_KERNEL_GQA_TMA;
    kc->tile = cfg.tile;
    kc->ctas_per_sm = cfg.ctas_per_sm;
    kc->cluster = 1;
    return DA_OK;
}

// ---- TMA descriptors ----------------------------------------------------------
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn()
{
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

CUtensorMapDataType tma_dtype(int dt)
{
    switch (dt) {
    case DA_F16: return CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    case DA_BF16: return CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    default: return CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
    }
}

// 4-D map over (d, kv head, position, batch) with box (box_d, 1, rows, 1):
// box_d = D unswizzled (SIMT kernel), or 64 columns landing 128-byte-swizzled
// (tensor-core kernel, sw128 = true).
int encode_cache_map(CUtensorMap *map, const void *base, int dt, int D, int hkv, int cap,
                     int batch, int64_t head_st, int64_t pos_st, int64_t batch_st, int rows,
                     bool sw128 = false)
{
    EncodeTiledFn enc = encode_fn();
    if (!enc) return fail(DA_ECUDA, "tma", "cuTensorMapEncodeTiled is unavailable");
    const int es = dtype_size(dt);
    if (batch == 1) batch_st = pos_st * cap;
    cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)hkv, (cuuint64_t)cap, (cuuint64_t)batch};
    cuuint64_t strides[3] = {(cuuint64_t)(head_st * es), (cuuint64_t)(pos_st * es),
                             (cuuint64_t)(batch_st * es)};
    cuuint32_t box[4] = {(cuuint32_t)(sw128 ? 64 : D), 1, (cuuint32_t)rows, 1};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    CUresult r = enc(map, tma_dtype(dt), 4, const_cast<void *>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE,
                     sw128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        return fail(DA_EUNSUPPORTED, "tma", "cuTensorMapEncodeTiled rejected the cache layout (%d)",
                    (int)r);
    return DA_OK;
}

// 4-D map over a paged pool (d, kv head, slot in block, block) with box
// (D, 1, rows, 1); slots past block_size and blocks past num_blocks read zeros.
int encode_pool_map(CUtensorMap *map, const void *base, int dt, int D, int hkv, int block_size,
                    int num_blocks, int64_t head_st, int64_t pos_st, int64_t block_st, int rows,
                    bool sw128 = false)
{
    EncodeTiledFn enc = encode_fn();
    if (!enc) return fail(DA_ECUDA, "tma", "cuTensorMapEncodeTiled is unavailable");
    const int es = dtype_size(dt);
    cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)hkv, (cuuint64_t)block_size,
                          (cuuint64_t)num_blocks};
    cuuint64_t strides[3] = {(cuuint64_t)(head_st * es), (cuuint64_t)(pos_st * es),
                             (cuuint64_t)(block_st * es)};
    cuuint32_t box[4] = {(cuuint32_t)(sw128 ? 64 : D), 1, (cuuint32_t)rows, 1};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    CUresult r = enc(map, tma_dtype(dt), 4, const_cast<void *>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE,
                     sw128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        return fail(DA_EUNSUPPORTED, "tma", "cuTensorMapEncodeTiled rejected the paged pool (%d)",
                    (int)r);
    return DA_OK;
}

int check_plan(const da_args_t *a, const da_plan_t *pl, KernelChoice *kc)
{
    if (!pl) return fail(DA_EINVAL, "args", "plan is NULL");
    int rc = select_kernel(a, kc);
    if (rc) return rc;
    if (pl->batch != a->batch || pl->kernel != kc->kernel || pl->tile != kc->tile)
        return fail(DA_EINVAL, "plan", "plan was made for other arguments");
    int64_t base = 0, items = 0;
    for (int b = 0; b < a->batch; ++b) {
        const int L = pl->seq_lens[b];
        if (L < q_len_of(a) || L > a->capacity)
            return fail(DA_EINVAL, "plan", "seq_lens[%d] = %d outside [q_len %d, capacity %d]",
                        b, L, q_len_of(a), a->capacity);
        if (pl->chunk[b] < 1 || pl->n_splits[b] != ceil_div(L, pl->chunk[b]) ||
            pl->split_base[b] != base)
            return fail(DA_EINVAL, "plan", "inconsistent split table at b = %d", b);
        base += pl->n_splits[b];
        items += (int64_t)pl->n_splits[b] * a->n_kv_heads * kc->row_groups;
    }
    if (pl->total_splits != base || pl->n_items != items || pl->grid < kc->cluster ||
        pl->grid > items * kc->cluster || pl->grid % kc->cluster)
        return fail(DA_EINVAL, "plan", "inconsistent plan totals");
    if (pl->workspace_bytes != ws_total(pl->total_splits, rows_of(a), a->v_dim,
                                        ws_counters(a->batch, a->n_kv_heads)))
        return fail(DA_EINVAL, "plan", "inconsistent workspace size");
    return DA_OK;
}

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// SMs of the current device (0 if the query fails)
int device_sms()
{
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
        (void)cudaGetLastError();
        return 0;
    }
    return n;
}

// the split kernel's grid; the test hook DA_FLAG_TEST_BAD_LAUNCH asks for an
// empty one, which the runtime refuses before anything runs
int split_grid(const da_args_t *a, const da_plan_t *pl)
{
    return (a->flags & DA_FLAG_TEST_BAD_LAUNCH) ? 0 : pl->grid;
}

FusedOut fused_out(const da_args_t *a, const da_plan_t *pl, void *ws, void *out)
{
    FusedOut f;
    std::memset(&f, 0, sizeof f);
    f.ctr = reinterpret_cast<uint32_t *>(static_cast<uint8_t *>(ws) +
                                         ws_ctr_offset(pl->total_splits, rows_of(a), a->v_dim));
    f.out = out;
    f.out_dtype = a->out_dtype;
    return f;
}

// The arrival counters start every call at zero: one memset on the stream,
// before the split kernel that counts on them.
int zero_counters(const da_args_t *a, const da_plan_t *pl, const FusedOut &f, cudaStream_t st)
{
    const cudaError_t e =
        cudaMemsetAsync(f.ctr, 0, (size_t)ws_counters(a->batch, a->n_kv_heads) * 4, st);
    if (e != cudaSuccess) return fail(DA_ELAUNCH, "split", "counter reset: %s", cudaGetErrorString(e));
    (void)pl;
    return DA_OK;
}

// Parameters of the f32 CUDA-core split kernel (f32 caches only).
F32Params f32_params(const da_args_t *a, const da_plan_t *pl, const float *q, const void *k,
                     const void *v, void *ws, const da_dev_t *dev)
{
    F32Params f;
    std::memset(&f, 0, sizeof f);
    uint8_t *w = static_cast<uint8_t *>(ws);
    f.q = q;
    f.k = static_cast<const float *>(k);
    f.v = static_cast<const float *>(v);
    f.k_pos_stride = a->k_pos_stride;
    f.k_head_stride = a->k_head_stride;
    f.k_batch_stride = a->batch > 1 ? a->k_batch_stride : 0;
    f.v_pos_stride = a->v_pos_stride;
    f.v_head_stride = a->v_head_stride;
    f.v_batch_stride = a->batch > 1 ? a->v_batch_stride : 0;
    f.ml = reinterpret_cast<float2 *>(w + ws_ml_offset());
    f.acc = reinterpret_cast<float *>(w + ws_acc_offset(pl->total_splits, rows_of(a)));
    f.status = reinterpret_cast<int *>(w);
    f.n_heads = rows_of(a);
    f.q_len = q_len_of(a);
    f.hq = a->n_heads;
    f.scale_log2 = a->scale * 1.4426950408889634f;
    f.flags = a->flags;
    f.exact_below = INT32_MAX;
    f.reset_status = 1;
    f.items.batch = a->batch;
    f.items.n_items = pl->n_items;
    f.items.n_kv_heads = a->n_kv_heads;
    for (int b = 0; b < a->batch; ++b) {
        f.items.seq_lens[b] = pl->seq_lens[b];
        f.items.chunk[b] = pl->chunk[b];
        f.items.split_base[b] = pl->split_base[b];
    }
    f.items.split_base[a->batch] = pl->total_splits;
    if (dev) {
        f.dev_lens = dev->seq_lens;
        if (dev->block_table) {
            f.block_table = dev->block_table;
            f.max_blocks = dev->max_blocks_per_seq;
            f.block_size = dev->block_size;
            f.k_block_stride = dev->k_block_stride;
            f.v_block_stride = dev->v_block_stride;
        }
    }
    return f;
}

int launch_mla(const da_args_t *a, const da_plan_t *pl, const float *q, const void *k,
               const void *v, void *ws, cudaStream_t st, const da_dev_t *dev, void *out,
               bool want_fuse, bool *fused)
{
    (void)v; // the same buffer as k (checked with the arguments)
    MlaParams p;
    std::memset(&p, 0, sizeof p);
    uint8_t *w = static_cast<uint8_t *>(ws);
    p.q = q;
    p.cache = k;
    p.pos_stride = a->k_pos_stride;
    p.batch_stride = a->batch > 1 ? a->k_batch_stride : 0;
    p.ml = reinterpret_cast<float2 *>(w + ws_ml_offset());
    p.acc = reinterpret_cast<float *>(w + ws_acc_offset(pl->total_splits, rows_of(a)));
    p.status = reinterpret_cast<int *>(w);
    p.n_heads = rows_of(a);
    p.q_len = q_len_of(a);
    p.hq = a->n_heads;
    p.scale_log2 = a->scale * 1.4426950408889634f;
    p.timeout_ns = (uint64_t)(a->timeout_us > 0 ? a->timeout_us : 2000000) * 1000ull;
    p.flags = a->flags;
    p.items.batch = a->batch;
    p.items.n_items = pl->n_items;
    p.items.n_kv_heads = 1;
    for (int b = 0; b < a->batch; ++b) {
        p.items.seq_lens[b] = pl->seq_lens[b];
        p.items.chunk[b] = pl->chunk[b];
        p.items.split_base[b] = pl->split_base[b];
    }
    p.items.split_base[a->batch] = pl->total_splits;
    if (dev) {
        p.dev_lens = dev->seq_lens;
        if (dev->block_table) {
            p.block_table = dev->block_table;
            p.max_blocks = dev->max_blocks_per_seq;
            p.block_size = dev->block_size;
            p.block_stride = dev->k_block_stride;
        }
    }
    // each sequence on one of the two kernels, chosen on the device from its
    // current length; both write their partials into the same workspace for
    // the one combine. A kernel is launched if any sequence may need it:
    // lengths read on the device can be anything from q_len to the plan's.
    p.exact_below = mla_exact_below(a);
    bool any_exact = false, any_tc = false;
    for (int b = 0; b < a->batch; ++b) {
        const int L = pl->seq_lens[b];
        any_tc |= L >= p.exact_below;
        any_exact |= (p.dev_lens ? q_len_of(a) : L) < p.exact_below;
    }
    // the tensor-core kernel merges its own partials when it serves every
    // sequence and the GPU holds all its clusters at once (its grid-wide
    // arrival count must not wait on a cluster that cannot start)
    p.fused = fused_out(a, pl, ws, out);
    p.fused.on = want_fuse && !any_exact && pl->grid / 2 <= mla_max_clusters(rows_of(a));
    *fused = p.fused.on != 0;
    if (p.fused.on) {
        const int rc = zero_counters(a, pl, p.fused, st);
        if (rc) return rc;
    }
    if (any_tc) {
        cudaError_t e = launch_mla_split(split_grid(a, pl), st, p, a->kv_dtype);
        if (e != cudaSuccess) return fail(DA_ELAUNCH, "split", "%s", cudaGetErrorString(e));
    }
    if (any_exact) {
        F32Params f = f32_params(a, pl, q, k, k, ws, dev);
        f.exact_below = p.exact_below;
        f.reset_status = any_tc ? 0 : 1;
        const int grid = (a->flags & DA_FLAG_TEST_BAD_LAUNCH)
                             ? 0
                             : pl->n_items * f32_split_groups(rows_of(a));
        cudaError_t e = launch_f32_split(576, 512, true, grid, st, f);
        if (e != cudaSuccess) return fail(DA_ELAUNCH, "split", "%s", cudaGetErrorString(e));
    }
    return DA_OK;
}

// Launches the split kernel(s). want_fuse: the kernels may merge their own
// partials into `out` (no combine launch); *fused says whether they will.
int launch_split(const da_args_t *a, const da_plan_t *pl, const float *q, const void *k,
                 const void *v, void *ws, cudaStream_t st, const da_dev_t *dev, void *out,
                 bool want_fuse, bool *fused)
{
    *fused = false;
    if (pl->kernel == DA_KERNEL_MLA_TC)
        return launch_mla(a, pl, q, k, v, ws, st, dev, out, want_fuse, fused);

    SplitParams p;
    std::memset(&p, 0, sizeof p);
    uint8_t *w = static_cast<uint8_t *>(ws);
    p.q = q;
    p.ml = reinterpret_cast<float2 *>(w + ws_ml_offset());
    p.acc = reinterpret_cast<float *>(w + ws_acc_offset(pl->total_splits, rows_of(a)));
    p.status = reinterpret_cast<int *>(w);
    p.n_heads = rows_of(a);
    p.q_len = q_len_of(a);
    p.hq = a->n_heads;
    p.scale_log2 = a->scale * 1.4426950408889634f;
    p.timeout_ns = (uint64_t)(a->timeout_us > 0 ? a->timeout_us : 2000000) * 1000ull;
    p.flags = a->flags;
    p.items.batch = a->batch;
    p.items.n_items = pl->n_items;
    p.items.n_kv_heads = a->n_kv_heads;
    for (int b = 0; b < a->batch; ++b) {
        p.items.seq_lens[b] = pl->seq_lens[b];
        p.items.chunk[b] = pl->chunk[b];
        p.items.split_base[b] = pl->split_base[b];
    }
    p.items.split_base[a->batch] = pl->total_splits;
    const bool tc = pl->kernel == DA_KERNEL_GQA_TC;
    // Both GQA kernels merge with every CTA of the launch waiting for its
    // groups, so they fuse only when the whole grid is resident at once (the
    // plan's CTAs per SM on this device's SMs); otherwise the combine launch
    // merges.
    const bool fuse = want_fuse && pl->grid <= device_sms() * pl->ctas_per_sm;
    p.fused = fused_out(a, pl, ws, out);
    p.fused.on = fuse;
    *fused = fuse;
    if (fuse) {
        const int rc = zero_counters(a, pl, p.fused, st);
        if (rc) return rc;
    }

    GqaMaps m;
    std::memset(&m, 0, sizeof m);
    int rc;
    if (dev && dev->block_table) {
        p.block_table = dev->block_table;
        p.max_blocks = dev->max_blocks_per_seq;
        p.block_size = dev->block_size;
        p.oob_block = dev->num_blocks;
        // Tiles run across block ends. The tensor-core kernel copies every tile
        // as boxes of box_rows rows, which never span a block. The SIMT kernel
        // copies a tile that lies in one block as one box of T rows (maps k, v)
        // and one that spans a block end as boxes of box_rows rows (maps kb, vb).
        p.box_rows = std::gcd(pl->tile, dev->block_size);
        auto pool = [&](CUtensorMap *km, CUtensorMap *vm, int rows) {
            int r = encode_pool_map(km, k, a->kv_dtype, a->head_dim, a->n_kv_heads,
                                    dev->block_size, dev->num_blocks, a->k_head_stride,
                                    a->k_pos_stride, dev->k_block_stride, rows, tc);
            if (r) return r;
            return encode_pool_map(vm, v, a->kv_dtype, a->v_dim, a->n_kv_heads, dev->block_size,
                                   dev->num_blocks, a->v_head_stride, a->v_pos_stride,
                                   dev->v_block_stride, rows, tc);
        };
        if ((rc = pool(&m.k, &m.v, tc ? p.box_rows : pl->tile))) return rc;
        if (!tc && (rc = pool(&m.kb, &m.vb, p.box_rows))) return rc;
    } else {
        rc = encode_cache_map(&m.k, k, a->kv_dtype, a->head_dim, a->n_kv_heads, a->capacity,
                              a->batch, a->k_head_stride, a->k_pos_stride, a->k_batch_stride,
                              pl->tile, tc);
        if (rc) return rc;
        rc = encode_cache_map(&m.v, v, a->kv_dtype, a->v_dim, a->n_kv_heads, a->capacity,
                              a->batch, a->v_head_stride, a->v_pos_stride, a->v_batch_stride,
                              pl->tile, tc);
        if (rc) return rc;
    }
    if (dev) p.dev_lens = dev->seq_lens;
    if (tc) {
        const cudaError_t e =
            launch_gqa_tc(a->kv_dtype, a->head_dim, split_grid(a, pl), st, m.k, m.v, p);
        if (e != cudaSuccess) return fail(DA_ELAUNCH, "split", "%s", cudaGetErrorString(e));
        return DA_OK;
    }

    p.items.row_groups = simt_row_groups(a);
    const int G = a->n_heads / a->n_kv_heads * q_len_of(a) / p.items.row_groups;
    cudaError_t e;
    switch (a->kv_dtype) {
    case DA_F32: e = gqa_launch_f32(a->head_dim, G, split_grid(a, pl), st, m, p); break;
    case DA_F16: e = gqa_launch_f16(a->head_dim, G, split_grid(a, pl), st, m, p); break;
    default: e = gqa_launch_bf16(a->head_dim, G, split_grid(a, pl), st, m, p); break;
    }
    if (e != cudaSuccess) return fail(DA_ELAUNCH, "split", "%s", cudaGetErrorString(e));
    return DA_OK;
}

// the projection's weights: element type, width, strides and alignment
int check_proj(const da_args_t *a, const da_proj_t *pj, da_proj_t *norm)
{
    if (!pj || !pj->w) return fail(DA_EINVAL, "args", "proj or proj->w is NULL");
    if (pj->w_dtype != DA_F32 && pj->w_dtype != DA_BF16)
        return fail(DA_EUNSUPPORTED, "args", "projection weights must be f32 or bf16");
    if (pj->out_dim < 1 || pj->out_dim > kProjMaxOut)
        return fail(DA_EUNSUPPORTED, "args", "projection out_dim %d outside [1, %d]", pj->out_dim,
                    kProjMaxOut);
    if (a->v_dim % 8 || a->v_dim > kProjMaxVdim)
        return fail(DA_EUNSUPPORTED, "args",
                    "a projected v_dim must be a multiple of 8 and at most %d", kProjMaxVdim);
    *norm = *pj;
    if (!norm->row_stride) norm->row_stride = a->v_dim;
    if (!norm->head_stride) norm->head_stride = (int64_t)pj->out_dim * norm->row_stride;
    const int es = dtype_size(pj->w_dtype);
    if (!aligned(pj->w, 16) || (norm->row_stride * es) % 16 || (norm->head_stride * es) % 16)
        return fail(DA_EINVAL, "args",
                    "projection weights and their strides must be 16-byte aligned");
    if (norm->row_stride < a->v_dim || norm->head_stride < 0)
        return fail(DA_EINVAL, "args", "projection row_stride %lld < v_dim %d",
                    (long long)norm->row_stride, a->v_dim);
    return DA_OK;
}

int launch_combine_phase(const da_args_t *a, const da_plan_t *pl, const void *ws, void *out,
                         cudaStream_t st, int n_ranks = 1, const da_proj_t *proj = nullptr)
{
    CombineParams c;
    std::memset(&c, 0, sizeof c);
    c.n_ranks = n_ranks;
    c.rank_ml = pl->workspace_bytes / 8; // float2 elements between ranks' workspaces
    c.rank_acc = pl->workspace_bytes / 4;
    const uint8_t *w = static_cast<const uint8_t *>(ws);
    c.ml = reinterpret_cast<const float2 *>(w + ws_ml_offset());
    c.acc = reinterpret_cast<const float *>(w + ws_acc_offset(pl->total_splits, rows_of(a)));
    c.out = out;
    c.n_heads = rows_of(a);
    c.v_dim = a->v_dim;
    c.batch = a->batch;
    for (int b = 0; b < a->batch; ++b) {
        c.n_splits[b] = pl->n_splits[b];
        c.split_base[b] = pl->split_base[b];
    }
    cudaError_t e;
    c.status = reinterpret_cast<int *>(const_cast<uint8_t *>(w));
    c.timeout_ns = (uint64_t)(a->timeout_us > 0 ? a->timeout_us : 2000000) * 1000ull;
    c.flags = a->flags;
    if (proj) {
        c.w = proj->w;
        c.w_head_stride = proj->head_stride;
        c.w_row_stride = proj->row_stride;
        c.out_dim = proj->out_dim;
        c.w_heads = a->n_heads;
        e = launch_combine_proj(a->out_dtype, proj->w_dtype, c, rows_of(a), a->batch, st, true);
    } else {
        e = launch_combine(a->out_dtype, a->v_dim, c, rows_of(a), a->batch, st, true);
    }
    if (e == cudaSuccess) e = cudaGetLastError();
    if (e != cudaSuccess) return fail(DA_ELAUNCH, "combine", "%s", cudaGetErrorString(e));
    return DA_OK;
}

int check_buffers(int kernel, const float *q, const void *k, const void *v, const void *out)
{
    if (!q || !k || !v || !out) return fail(DA_EINVAL, "args", "a tensor pointer is NULL");
    if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(out, 16))
        return fail(DA_EINVAL, "args", "q, caches and out must be 16-byte aligned");
    if (kernel == DA_KERNEL_MLA_TC && k != v)
        return fail(DA_EUNSUPPORTED, "args",
                    "MLA values must be the first 512 columns of the key rows: pass the same "
                    "buffer as k_cache and v_cache");
    return DA_OK;
}

// short form: one workspace per device
std::mutex g_ws_mu;
std::vector<std::pair<void *, size_t>> g_ws;

} // namespace

// Lets other translation units of the library report through
// decode_attn_last_error().
int set_error(int code, const char *phase, const char *msg) { return fail(code, phase, "%s", msg); }

} // namespace skv

using namespace skv;

extern "C" {

int decode_attn_plan(const da_args_t *a, const int32_t *lens, int num_sms, da_plan_t *plan)
{
    int rc = check_args(a);
    if (rc) return rc;
    if (!lens || !plan) return fail(DA_EINVAL, "args", "seq_lens or plan is NULL");
    for (int b = 0; b < a->batch; ++b)
        if (lens[b] < q_len_of(a) || lens[b] > a->capacity)
            return fail(DA_EINVAL, "args", "seq_lens[%d] = %d outside [q_len %d, capacity %d]",
                        b, lens[b], q_len_of(a), a->capacity);
    KernelChoice kc;
    rc = select_kernel(a, &kc);
    if (rc) return rc;
    if (num_sms <= 0) {
        int dev = 0;
        cudaError_t e = cudaGetDevice(&dev);
        if (e == cudaSuccess)
            e = cudaDeviceGetAttribute(&num_sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess)
            return fail(DA_ECUDA, "plan", "SM count query failed: %s", cudaGetErrorString(e));
    }
    PlanOut po;
    int slots = std::max(1, num_sms * kc.ctas_per_sm / kc.cluster);
    if (kc.kernel == DA_KERNEL_MLA_TC) {
        // every sequence on the f32 kernel: its CTAs serve (item, group of 32
        // rows), one per SM, so the items fill the SMs divided by the groups
        bool all_exact = true;
        for (int b = 0; b < a->batch; ++b) all_exact &= lens[b] < mla_exact_below(a);
        if (all_exact) slots = std::max(1, num_sms / f32_split_groups(rows_of(a)));
    }

    const int prc = plan_splits(lens, a->batch, a->n_kv_heads * kc.row_groups, kc.tile, slots,
                                a->force_splits, 1 << 22, &po);
    if (prc == 1) return fail(DA_EINVAL, "plan", "invalid lengths");
    if (prc == 2) return fail(DA_EUNSUPPORTED, "plan", "too many work items");
    std::memset(plan, 0, sizeof *plan);
    plan->kernel = kc.kernel;
    plan->num_sms = num_sms;
    plan->ctas_per_sm = kc.ctas_per_sm;
    plan->tile = kc.tile;
    // the split kernel's CTAs (for MLA, the tensor-core kernel's clusters, one
    // CTA per SM, even when every sequence runs on the f32 kernel)
    plan->grid = (int32_t)std::min<int64_t>(
                     po.n_items, std::max(1, num_sms * kc.ctas_per_sm / kc.cluster)) *
                 kc.cluster;
    plan->n_items = po.n_items;
    plan->batch = a->batch;
    int64_t base = 0;
    int32_t mx = 0;
    for (int b = 0; b < a->batch; ++b) {
        plan->seq_lens[b] = lens[b];
        plan->chunk[b] = po.chunk[b];
        plan->n_splits[b] = po.n_splits[b];
        plan->split_base[b] = (int32_t)base;
        base += po.n_splits[b];
        if (po.n_splits[b] > mx) mx = po.n_splits[b];
    }
    plan->total_splits = (int32_t)base;
    plan->max_splits = mx;
    plan->workspace_bytes = ws_total(base, rows_of(a), a->v_dim, ws_counters(a->batch, a->n_kv_heads));
    plan->est_cost = po.est_cost;
    return DA_OK;
}

int64_t decode_attn_workspace_bytes(const da_plan_t *plan)
{
    return plan ? plan->workspace_bytes : 0;
}

int decode_attn_splitk_ex(const da_args_t *a, const da_plan_t *plan, const float *q,
                          const void *k, const void *v, void *out, void *ws, size_t ws_bytes,
                          da_stream_t stream)
{
    int rc = check_args(a);
    if (rc) return rc;
    KernelChoice kc;
    rc = check_plan(a, plan, &kc);
    if (rc) return rc;
    rc = check_buffers(kc.kernel, q, k, v, out);
    if (rc) return rc;
    if (!ws || !aligned(ws, 256))
        return fail(DA_EINVAL, "args", "workspace must be non-NULL and 256-byte aligned");
    if ((int64_t)ws_bytes < plan->workspace_bytes)
        return fail(DA_ENOSPACE, "args", "workspace %zu bytes < %lld needed", ws_bytes,
                    (long long)plan->workspace_bytes);
    cudaError_t pre = cudaGetLastError();
    if (pre != cudaSuccess)
        return fail(DA_ECUDA, "before split", "pending CUDA error: %s", cudaGetErrorString(pre));
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    bool fused = false;
    rc = launch_split(a, plan, q, k, v, ws, st, nullptr, out, want_fuse(a), &fused);
    if (rc) return rc;
    if (fused || (a->flags & DA_FLAG_NO_COMBINE)) return DA_OK;
    return launch_combine_phase(a, plan, ws, out, st);
}

int decode_attn_splitk_dev(const da_args_t *a, const da_plan_t *plan, const da_dev_t *dev,
                           const float *q, const void *k, const void *v, void *out, void *ws,
                           size_t ws_bytes, da_stream_t stream)
{
    int rc = check_args(a);
    if (rc) return rc;
    if (!dev) return fail(DA_EINVAL, "args", "dev is NULL");
    KernelChoice kc;
    rc = check_plan(a, plan, &kc);
    if (rc) return rc;
    if (kc.kernel == DA_KERNEL_MLA_TC && dev->block_table &&
        (dev->v_block_stride != dev->k_block_stride ||
         (dev->k_block_stride * dtype_size(a->kv_dtype)) % 16))
        return fail(DA_EUNSUPPORTED, "args",
                    "MLA latent pools: one pool for keys and values (equal block strides, "
                    "16-byte multiples)");
    rc = check_buffers(kc.kernel, q, k, v, out);
    if (rc) return rc;
    if (dev->seq_lens && !aligned(dev->seq_lens, 4))
        return fail(DA_EINVAL, "args", "dev->seq_lens must be 4-byte aligned");
    if (dev->block_table) {
        const int es = dtype_size(a->kv_dtype);
        if (!aligned(dev->block_table, 4))
            return fail(DA_EINVAL, "args", "dev->block_table must be 4-byte aligned");
        if (dev->block_size < 16 || dev->block_size % 16)
            return fail(DA_EUNSUPPORTED, "args", "block_size %d: a positive multiple of 16",
                        dev->block_size);
        if (dev->max_blocks_per_seq < 1 || dev->num_blocks < 1)
            return fail(DA_EINVAL, "args", "max_blocks_per_seq and num_blocks must be >= 1");
        if ((dev->k_block_stride * es) % 16 || (dev->v_block_stride * es) % 16 ||
            dev->k_block_stride < (int64_t)dev->block_size * a->k_pos_stride ||
            dev->v_block_stride < (int64_t)dev->block_size * a->v_pos_stride)
            return fail(DA_EUNSUPPORTED, "args",
                        "block strides must hold block_size positions and be multiples of 16 "
                        "bytes");
        for (int b = 0; b < a->batch; ++b)
            if ((int64_t)plan->seq_lens[b] > (int64_t)dev->max_blocks_per_seq * dev->block_size)
                return fail(DA_EINVAL, "args",
                            "seq_lens[%d] = %d exceeds max_blocks_per_seq x block_size", b,
                            plan->seq_lens[b]);
        // the GQA kernels copy a paged tile in boxes of multiples of gcd(tile,
        // block_size) rows that start at multiples of that height, so a split
        // must start at one
        if (kc.kernel != DA_KERNEL_MLA_TC) {
            const int h = std::gcd(plan->tile, dev->block_size);
            for (int b = 0; b < a->batch; ++b)
                if (plan->chunk[b] % h)
                    return fail(DA_EINVAL, "plan",
                                "chunk[%d] = %d: paged caches need chunks that are multiples "
                                "of %d",
                                b, plan->chunk[b], h);
        }
    }
    if (!ws || !aligned(ws, 256))
        return fail(DA_EINVAL, "args", "workspace must be non-NULL and 256-byte aligned");
    if ((int64_t)ws_bytes < plan->workspace_bytes)
        return fail(DA_ENOSPACE, "args", "workspace %zu bytes < %lld needed", ws_bytes,
                    (long long)plan->workspace_bytes);
    cudaError_t pre = cudaGetLastError();
    if (pre != cudaSuccess)
        return fail(DA_ECUDA, "before split", "pending CUDA error: %s", cudaGetErrorString(pre));
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    bool fused = false;
    rc = launch_split(a, plan, q, k, v, ws, st, dev, out, want_fuse(a), &fused);
    if (rc) return rc;
    if (fused || (a->flags & DA_FLAG_NO_COMBINE)) return DA_OK;
    return launch_combine_phase(a, plan, ws, out, st);
}

int decode_attn_combine_ranks(const da_args_t *a, const da_plan_t *plan, const void *ws,
                              int n_ranks, void *out, da_stream_t stream)
{
    int rc = check_args(a);
    if (rc) return rc;
    KernelChoice kc;
    rc = check_plan(a, plan, &kc);
    if (rc) return rc;
    if (n_ranks < 1 || n_ranks > 4096)
        return fail(DA_EINVAL, "args", "n_ranks %d outside [1, 4096]", n_ranks);
    if (!ws || !aligned(ws, 256)) return fail(DA_EINVAL, "args", "workspaces misaligned or NULL");
    if (!out || !aligned(out, 16)) return fail(DA_EINVAL, "args", "out misaligned or NULL");
    cudaError_t pre = cudaGetLastError();
    if (pre != cudaSuccess)
        return fail(DA_ECUDA, "before combine", "pending CUDA error: %s",
                    cudaGetErrorString(pre));
    return launch_combine_phase(a, plan, ws, out, reinterpret_cast<cudaStream_t>(stream),
                                n_ranks);
}

int decode_attn_combine_proj(const da_args_t *a, const da_plan_t *plan, const da_proj_t *proj,
                             const void *ws, int n_ranks, void *out, da_stream_t stream)
{
    int rc = check_args(a);
    if (rc) return rc;
    KernelChoice kc;
    rc = check_plan(a, plan, &kc);
    if (rc) return rc;
    da_proj_t pj;
    rc = check_proj(a, proj, &pj);
    if (rc) return rc;
    if (n_ranks < 1 || n_ranks > 4096)
        return fail(DA_EINVAL, "args", "n_ranks %d outside [1, 4096]", n_ranks);
    if (!ws || !aligned(ws, 256)) return fail(DA_EINVAL, "args", "workspaces misaligned or NULL");
    if (!out || !aligned(out, 16)) return fail(DA_EINVAL, "args", "out misaligned or NULL");
    cudaError_t pre = cudaGetLastError();
    if (pre != cudaSuccess)
        return fail(DA_ECUDA, "before combine", "pending CUDA error: %s",
                    cudaGetErrorString(pre));
    return launch_combine_phase(a, plan, ws, out, reinterpret_cast<cudaStream_t>(stream),
                                n_ranks, &pj);
}

int decode_attn_splitk_proj(const da_args_t *a, const da_plan_t *plan, const da_proj_t *proj,
                            const float *q, const void *k, const void *v, void *out, void *ws,
                            size_t ws_bytes, da_stream_t stream)
{
    int rc = check_args(a);
    if (rc) return rc;
    KernelChoice kc;
    rc = check_plan(a, plan, &kc);
    if (rc) return rc;
    da_proj_t pj;
    rc = check_proj(a, proj, &pj);
    if (rc) return rc;
    rc = check_buffers(kc.kernel, q, k, v, out);
    if (rc) return rc;
    if (!ws || !aligned(ws, 256))
        return fail(DA_EINVAL, "args", "workspace must be non-NULL and 256-byte aligned");
    if ((int64_t)ws_bytes < plan->workspace_bytes)
        return fail(DA_ENOSPACE, "args", "workspace %zu bytes < %lld needed", ws_bytes,
                    (long long)plan->workspace_bytes);
    cudaError_t pre = cudaGetLastError();
    if (pre != cudaSuccess)
        return fail(DA_ECUDA, "before split", "pending CUDA error: %s", cudaGetErrorString(pre));
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    bool fused = false; // the projection runs in its own combine launch
    rc = launch_split(a, plan, q, k, v, ws, st, nullptr, out, false, &fused);
    if (rc) return rc;
    return launch_combine_phase(a, plan, ws, out, st, 1, &pj);
}

int decode_attn_combine(const da_args_t *a, const da_plan_t *plan, const void *ws, void *out,
                        da_stream_t stream)
{
    int rc = check_args(a);
    if (rc) return rc;
    KernelChoice kc;
    rc = check_plan(a, plan, &kc);
    if (rc) return rc;
    if (!ws || !aligned(ws, 256)) return fail(DA_EINVAL, "args", "workspace misaligned or NULL");
    if (!out || !aligned(out, 16)) return fail(DA_EINVAL, "args", "out misaligned or NULL");
    cudaError_t pre = cudaGetLastError();
    if (pre != cudaSuccess)
        return fail(DA_ECUDA, "before combine", "pending CUDA error: %s",
                    cudaGetErrorString(pre));
    return launch_combine_phase(a, plan, ws, out, reinterpret_cast<cudaStream_t>(stream));
}

int decode_attn_splitk(const float *q, const float *k, const float *v, const int32_t *seq_lens,
                       int n_heads, int n_kv_heads, int head_dim, float scale, float *out,
                       da_stream_t stream)
{
    if (!seq_lens) return fail(DA_EINVAL, "args", "seq_lens is NULL");
    if (n_kv_heads < 1 || head_dim < 1)
        return fail(DA_EINVAL, "args", "n_kv_heads %d / head_dim %d must be >= 1", n_kv_heads,
                    head_dim);
    const int L = seq_lens[0];
    da_args_t a;
    std::memset(&a, 0, sizeof a);
    a.batch = 1;
    a.n_heads = n_heads;
    a.n_kv_heads = n_kv_heads;
    a.head_dim = head_dim;
    a.v_dim = head_dim;
    a.capacity = L;
    a.k_pos_stride = a.v_pos_stride = (int64_t)n_kv_heads * head_dim;
    a.k_head_stride = a.v_head_stride = head_dim;
    a.k_batch_stride = a.v_batch_stride = (int64_t)L * n_kv_heads * head_dim;
    a.kv_dtype = DA_F32;
    a.out_dtype = DA_F32;
    a.scale = scale;
    da_plan_t plan;
    int rc = decode_attn_plan(&a, seq_lens, 0, &plan);
    if (rc) return rc;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail(DA_ECUDA, "workspace", "%s", cudaGetErrorString(e));
    // The lock is held until the launches are enqueued, so another thread
    // cannot free (to grow) or release this workspace between the lookup and
    // the launches; cudaFree then waits for the kernels already enqueued.
    std::lock_guard<std::mutex> lk(g_ws_mu);
    if ((int)g_ws.size() <= dev) g_ws.resize(dev + 1, {nullptr, 0});
    auto &slot = g_ws[dev];
    if (slot.second < (size_t)plan.workspace_bytes) {
        if (slot.first) cudaFree(slot.first);
        slot = {nullptr, 0};
        size_t want = (size_t)plan.workspace_bytes * 2;
        e = cudaMalloc(&slot.first, want);
        if (e != cudaSuccess)
            return fail(DA_ECUDA, "workspace", "cudaMalloc of %zu bytes: %s", want,
                        cudaGetErrorString(e));
        slot.second = want;
    }
    return decode_attn_splitk_ex(&a, &plan, q, k, v, out, slot.first,
                                 (size_t)plan.workspace_bytes, stream);
}

int decode_attn_device_status(void *ws, da_stream_t stream)
{
    if (!ws) return fail(DA_EINVAL, "args", "workspace is NULL");
    cudaError_t e = cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return fail(DA_ECUDA, "sync", "%s", cudaGetErrorString(e));
    int v = 0;
    e = cudaMemcpy(&v, ws, sizeof v, cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return fail(DA_ECUDA, "status", "%s", cudaGetErrorString(e));
    if (v == 0) return DA_OK;
    const int zero = 0;
    cudaMemcpy(ws, &zero, sizeof zero, cudaMemcpyHostToDevice);
    const int code = v & 0xff, kernel = (v >> 8) & 0xff;
    if (code == DA_ETIMEOUT)
        return fail(DA_ETIMEOUT,
                    kernel == DA_KERNEL_MLA_TC   ? "split (mla)"
                    : kernel == DA_KERNEL_GQA_TC ? "split (gqa, tensor cores)"
                    : kernel == (kStatusTimeoutProj >> 8) ? "combine (projection)"
                    : kernel == (kStatusTimeoutCombine >> 8) ? "combine"
                                                          : "split (gqa)",
                    "a bounded in-kernel wait ran out");
    return fail(DA_ECUDA, "status", "unexpected status word 0x%x", v);
}

const char *decode_attn_last_error(void) { return g_err.c_str(); }

void decode_attn_release(void)
{
    std::lock_guard<std::mutex> lk(g_ws_mu);
    int cur = 0;
    cudaGetDevice(&cur);
    for (size_t d = 0; d < g_ws.size(); ++d)
        if (g_ws[d].first) {
            cudaSetDevice((int)d);
            cudaFree(g_ws[d].first);
            g_ws[d] = {nullptr, 0};
        }
    cudaSetDevice(cur);
}

const char *decode_attn_version(void)
{
    return "split_kv_decode_gb300 0.2 (sm_103a: SIMT and tcgen05 GQA, tcgen05 MLA, combine with projection)";
}

} // extern "C"
