/*
 * split_kv_decode.h -- C ABI of the split-KV decode-attention library
 * (libsplitkv.so, GB300 / sm_103a).
 *
 * The operation: one query token per sequence attends over a long KV cache,
 *     out[b,h,:] = softmax(q[b,h,:] . K[b,0:L_b,kv,:]^T * scale) . V[b,0:L_b,kv,:]
 * with kv = h / G, G = n_heads / n_kv_heads (GQA; MQA/MLA when n_kv_heads = 1),
 * computed split over context ("flash-decoding"): every (sequence, KV head,
 * split) work item streams one contiguous slice of K/V once for all G query
 * heads that share it, keeps the online-softmax state (m, l, acc) on chip,
 * and writes one un-normalised partial per query head; a combine kernel
 * merges the partials by rescaling with exp(m_i - m).
 *   - Split over context, contiguous slices, neutral empty slices, per-device
 *     scratch, launch guard: "Attention at 128k: Split Over Context, Split
 *     Over Heads" (jared-hpc.com, Part 4 Lecture 06), sections 2 and 5.3.
 *   - Kernel A / Kernel B pair, raw device pointers plus a storage tag,
 *     caller-owned partials, split count chosen on the host from L:
 *     aprender issue 3725 design note, sections 2 and 3.
 *   - Partial triple and LSE merge; MLA absorbed decode as 96..128 heads
 *     over one 576-wide latent; plan/run separation: "The Kernel Level:
 *     Attention and MoE" (llm-serving.xyz lecture 07), sections "Decode
 *     Starves the SMs" and "A kernel alone is not a serving system".
 *
 * Conventions for every call:
 *   - All tensor pointers are DEVICE pointers of the current CUDA device,
 *     owned by the caller; the library never frees them.
 *   - q is float32 [batch][n_heads][head_dim] (with q_len > 1:
 *     [batch][q_len][n_heads][head_dim]), contiguous.
 *   - K/V element (b, pos, kv, d) lives at base + b*batch_stride +
 *     pos*pos_stride + kv*head_stride + d (strides in ELEMENTS). For MLA pass
 *     the same buffer as k_cache and v_cache with v_dim < head_dim: the
 *     values are the first v_dim columns of each latent row.
 *   - out is [batch][n_heads][v_dim], contiguous, of type out_dtype.
 *   - Work is enqueued on `stream` (a cudaStream_t; NULL = legacy default
 *     stream). No call below synchronises or allocates, except where its
 *     comment says so.
 *   - Every call returns a da_status_t. On failure a thread-local message
 *     naming the phase ("args", "plan", "split", "combine", ...) is
 *     available from decode_attn_last_error().
 */
#ifndef SPLIT_KV_DECODE_H
#define SPLIT_KV_DECODE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *da_stream_t; /* same type as cudaStream_t */

typedef enum { DA_F32 = 0, DA_F16 = 1, DA_BF16 = 2 } da_dtype_t;

typedef enum {
    DA_OK = 0,
    DA_EINVAL = 1,       /* an argument is out of range or inconsistent            */
    DA_EUNSUPPORTED = 2, /* valid, but no kernel here serves it (reason in message) */
    DA_ENOSPACE = 3,     /* workspace smaller than decode_attn_workspace_bytes()   */
    DA_ELAUNCH = 4,      /* a kernel launch failed; the message names the phase    */
    DA_ETIMEOUT = 5,     /* a bounded in-kernel wait ran out (see device_status)   */
    DA_ECUDA = 6         /* another CUDA runtime error                             */
} da_status_t;

#define DA_MAX_BATCH 256

/* da_args_t.flags */
#define DA_FLAG_NO_COMBINE 0x1   /* decode_attn_splitk_ex runs the split kernel only */
#define DA_FLAG_GQA_SIMT 0x2     /* for 16-bit caches with 8 rows per work item (see
                                    DA_KERNEL_GQA_TC), use the SIMT kernel instead  */
#define DA_FLAG_NO_CAUSAL 0x4    /* with q_len > 1: every new token sees every
                                    position of the (slice of the) cache, for a
                                    slice that lies wholly before the new tokens,
                                    e.g. every rank but the last of a
                                    context-parallel step                          */
#define DA_FLAG_MLA_SIMT 0x8     /* MLA shape: every sequence on the f32 CUDA-core
                                    kernel (see DA_MLA_EXACT_BELOW)                  */
#define DA_FLAG_MLA_TC 0x10      /* MLA shape: every sequence on the tensor-core
                                    kernel, whose operands are bf16 (see
                                    DA_MLA_EXACT_BELOW)                              */
#define DA_FLAG_ONE_LAUNCH 0x20  /* the split kernel merges its own partials (no
                                    combine launch). GQA kernels (SIMT and tensor
                                    cores): once a CTA has written all its items,
                                    each item merges a share of its (sequence, KV
                                    head) group after waiting for the group's last
                                    arrival; MLA tensor-core kernel: once all CTAs
                                    have finished, each stages its share of the
                                    rows in shared memory and merges it. Only when
                                    the plan's grid (the MLA kernel's clusters) is
                                    resident at once, else the combine launch
                                    merges. A memset of the workspace's arrival
                                    counters precedes the launch. The waits assume
                                    the launch is not sharing the SMs with kernels
                                    of other streams; if it is, they may run out
                                    (DA_ETIMEOUT in the status word). Measured on
                                    GB300 slower than the default two launches on
                                    every benchmarked workload (by 1 to 8 us on
                                    one sequence, more on batches), so it is an
                                    option, not the default                        */
#define DA_FLAG_COMBINE_LOADS 0x40 /* the combine kernel reads the partials with
                                    plain loads instead of staging them in shared
                                    memory by bulk copies (kept for comparison;
                                    partials of several ranks, a v_dim that is not
                                    a multiple of 128 or more than 256 splits of a
                                    sequence always take this form)                */
#define DA_FLAG_TEST_NO_TMA 0x100 /* test hook: the producer issues no copy, so every
                                     consumer wait runs out after timeout_us and the
                                     kernel reports DA_ETIMEOUT through device_status;
                                     the staged combine (and the projection) issues
                                     none either and reports its own timeout when
                                     no earlier one is recorded                      */
#define DA_FLAG_TEST_BAD_LAUNCH 0x200 /* test hook: the split kernel is launched with an
                                     empty grid, which the runtime refuses before
                                     anything runs (a launch error that does not stick
                                     to the context): the call returns DA_ELAUNCH and
                                     the message names the "split" phase             */

/*
 * MLA sequences shorter than this many positions run on an f32 CUDA-core
 * kernel, longer ones on the tensor-core kernel. The choice is made on the
 * device from the current length (the plan's, or the one decode_attn_splitk_dev
 * reads), so a captured launch follows a context that grows past it.
 * The tensor-core kernel rounds q, the latent rows and the probabilities to
 * bf16 and accumulates in f32. Over thousands of attended positions those
 * rounding errors average out: on caches drawn like the MLA workload (N(0,
 * 0.5) latents, N(0, 1) queries), max|err| stays below 1e-4 of max|V| from
 * about 1000 positions up. With few positions a single value row's rounding
 * (up to 2^-9 of it) reaches the output, so short sequences take the f32
 * kernel, which keeps every operand in f32 (within 2e-4 of max|V| at any
 * length; the work there is small). Attention peaked on a few positions of a
 * long context shows the bf16 rounding the same way: callers who need the f32
 * bound there set DA_FLAG_MLA_SIMT. DA_FLAG_MLA_TC sends everything to the
 * tensor cores.
 */
#define DA_MLA_EXACT_BELOW 2048

/* Kernels the planner can choose (da_plan_t.kernel). */
#define DA_KERNEL_GQA_TMA 1 /* SIMT split kernel, TMA-staged K/V tiles (GQA, MQA) */
#define DA_KERNEL_MLA_TC 2  /* MLA (576/512 latent): the tcgen05/TMEM split kernel,
                               and the f32 CUDA-core one for sequences shorter
                               than DA_MLA_EXACT_BELOW                          */
#define DA_KERNEL_GQA_TC 3  /* tcgen05/TMEM split kernel for GQA/MQA work items of
                               8 to 128 query rows ((n_heads / n_kv_heads) * q_len),
                               f16 or bf16 caches, head_dim 128 or 256; q and the
                               probabilities are rounded to the cache type         */


typedef struct {
    int32_t batch;       /* 1 .. DA_MAX_BATCH                                  */
    int32_t n_heads;     /* query heads                                        */
    int32_t n_kv_heads;  /* KV heads; n_heads % n_kv_heads == 0                */
    int32_t head_dim;    /* q/K width: 128 or 256 (GQA), 576 (MLA)             */
    int32_t v_dim;       /* V width: == head_dim (GQA), 512 (MLA)              */
    int32_t capacity;    /* positions allocated per sequence; seq_lens <= it   */
    int64_t k_batch_stride, k_pos_stride, k_head_stride; /* elements            */
    int64_t v_batch_stride, v_pos_stride, v_head_stride; /* elements            */
    int32_t kv_dtype;    /* da_dtype_t of the cache                            */
    int32_t out_dtype;   /* da_dtype_t of out (DA_F32, DA_F16 or DA_BF16)      */
    float scale;         /* score scale, usually 1/sqrt(head_dim)              */
    int32_t force_splits;/* 0: heuristic; n > 0: n splits per sequence (capped
                            so that no split is empty)                         */
    int32_t flags;       /* DA_FLAG_*                                          */
    int32_t timeout_us;  /* bound on every in-kernel wait; 0 = 2 000 000 us    */
    int32_t q_len;       /* query tokens per sequence; 0 or 1: one. With q_len
                            > 1, q is [batch][q_len][n_heads][head_dim] and out
                            [batch][q_len][n_heads][v_dim]; token i sits at
                            position L - q_len + i and attends to positions
                            0 .. L - q_len + i (causal among the new tokens,
                            whose K/V rows are in the cache: the causal query
                            tile of "Decoder Block 6: Online Attention, the
                            Capstone", Lesson). The rows of a work item are
                            (n_heads / n_kv_heads) * q_len (token, head)
                            pairs: 1 to 8 (SIMT GQA kernel; 9 to 128 on an
                            f32 cache, cut into row groups of up to 8, one
                            work item each), 8 to 128 (tensor-core GQA
                            kernel, 16-bit caches), or 32, 64, 96 or 128
                            (MLA). Every seq_len >= q_len; at most 64.        */
} da_args_t;

/* A host-side plan (plan/run separation): which kernel, how the context is
 * cut, and how many CTAs run. Pure host data; decode_attn_plan fills it. */
typedef struct {
    int32_t kernel;                     /* DA_KERNEL_*                                  */
    int32_t num_sms;                    /* SMs the plan was made for                    */
    int32_t ctas_per_sm;                /* resident split CTAs per SM                   */
    int32_t tile;                       /* positions per staged tile                    */
    int32_t grid;                       /* split-kernel CTAs (persistent)               */
    int32_t n_items;                    /* work items: (sequence, KV head, split),
                                           and per row group on an f32 cache with
                                           more than 8 rows per KV head             */
    int32_t total_splits;               /* sum over b of n_splits[b]                    */
    int32_t max_splits;                 /* max over b of n_splits[b]                    */
    int32_t batch;
    int32_t seq_lens[DA_MAX_BATCH];     /* copied from the caller                       */
    int32_t chunk[DA_MAX_BATCH];        /* positions per split of sequence b            */
    int32_t n_splits[DA_MAX_BATCH];     /* ceil(seq_lens[b] / chunk[b]); none empty     */
    int32_t split_base[DA_MAX_BATCH];   /* prefix sum of n_splits                       */
    int64_t workspace_bytes;            /* bytes decode_attn_splitk_ex needs            */
    int64_t est_cost;                   /* planner's makespan estimate (positions)      */
} da_plan_t;

/*
 * decode_attn_plan -- choose the kernel and the split of the context.
 * Pure host code: the plan step of the plan/run split described in "The
 * Kernel Level", where the host looks at the lengths of the batch and fixes
 * how the work is partitioned and balanced before anything runs.
 * The split count follows aprender issue 3725 §2 (chunk = ceil(L / S),
 * n_splits = ceil(L / chunk), so no split is ever empty) with the budget taken
 * on the product (sequences x KV heads x splits), as "Attention at 128k"
 * §5.1 asks, so that every SM gets equal work.
 *   args           shapes, strides, dtypes (validated here)
 *   seq_lens_host  HOST int32[args->batch], each in [1, args->capacity]
 *   num_sms        SM count to plan for; <= 0 queries the current device
 *   plan           out
 * Returns DA_OK, DA_EINVAL, DA_EUNSUPPORTED, or DA_ECUDA (device query).
 */
int decode_attn_plan(const da_args_t *args, const int32_t *seq_lens_host, int num_sms,
                     da_plan_t *plan);

/* Workspace bytes the plan needs (partials + a small status header). */
int64_t decode_attn_workspace_bytes(const da_plan_t *plan);

/*
 * decode_attn_splitk_ex -- run the split kernel and (unless
 * DA_FLAG_NO_COMBINE) the combine kernel on `stream`.
 * Split kernel (the plan's choice, da_plan_t.kernel): Kernel A of aprender
 * issue 3725 §2 re-designed for sm_103a (DA_KERNEL_GQA_TMA); for work items
 * of 8 to 128 query rows on a 16-bit cache the same item on tensor cores
 * (DA_KERNEL_GQA_TC); for MLA the heads-batched kernel of "Attention at 128k"
 * §4 on tensor cores (DA_KERNEL_MLA_TC). Partials (m, l, acc) are written per
 * (query row, split), acc left un-normalised; empty slices are neutral
 * (l = 0, m = -1e30).
 *   workspace   DEVICE memory, >= plan->workspace_bytes, 256-byte aligned,
 *               caller-owned (per device; "Attention at 128k" §2 explains why
 *               one pointer must never serve two devices). Contents need no
 *               initialisation.
 * Validation before any launch: DA_EINVAL / DA_EUNSUPPORTED / DA_ENOSPACE.
 * The MLA shape (head_dim 576, v_dim 512, one KV head) needs an f32, f16 or
 * bf16 latent cache, 32, 64, 96 or 128 query rows (heads x q_len), and
 * k_cache == v_cache; otherwise DA_EUNSUPPORTED.
 * A failed launch: DA_ELAUNCH, message names the phase ("split"/"combine").
 * Asynchronous: a timed-out wait inside the kernel is reported later by
 * decode_attn_device_status().
 */
int decode_attn_splitk_ex(const da_args_t *args, const da_plan_t *plan, const float *q,
                          const void *k_cache, const void *v_cache, void *out,
                          void *workspace, size_t workspace_bytes, da_stream_t stream);

/*
 * decode_attn_combine -- merge the partials in `workspace` into out:
 *   m = max_i m_i, w_i = exp(m_i - m), out = sum_i w_i acc_i / sum_i w_i l_i
 * ("Attention at 128k" §2; aprender issue 3725 §2, Kernel B). One CTA per
 * (sequence, query head). Reads what decode_attn_splitk_ex (with
 * DA_FLAG_NO_COMBINE) left for the same args and plan.
 */
int decode_attn_combine(const da_args_t *args, const da_plan_t *plan, const void *workspace,
                        void *out, da_stream_t stream);

/*
 * decode_attn_combine_ranks -- the combine of a context-parallel step (DCP:
 * "The Kernel Level: Attention and MoE", the split-KV section: the same merge
 * across GPUs that hold slices of the context). n_ranks ranks each ran
 * decode_attn_splitk_dev with DA_FLAG_NO_COMBINE and the SAME plan on their
 * own slice of every sequence (the plan made for the longest slice, the slice
 * lengths in seq_lens); `workspaces` holds their workspaces back to back, rank
 * r at r * plan->workspace_bytes (e.g. after an all-gather). Merges, for every
 * (sequence, query head), the partials of all ranks and splits:
 *   m = max m_ri, out = sum e^{m_ri - m} acc_ri / sum e^{m_ri - m} l_ri.
 * n_ranks = 1 is decode_attn_combine. One kernel launch on `stream`.
 */
int decode_attn_combine_ranks(const da_args_t *args, const da_plan_t *plan,
                              const void *workspaces, int n_ranks, void *out,
                              da_stream_t stream);

/*
 * da_proj_t -- a per-head output projection applied to the merged attention
 * output: out[b][h][e] = sum_c W[h][e][c] * attn[b][h][c], e < out_dim,
 * c < v_dim. For MLA this is the value up-projection wv_b, which maps a head's
 * merged 512-wide latent to its value head; it is a function of the merged
 * result, not of any one split, so it runs in the combine ("Attention at 128k"
 * §2, the PR #49 decisions: the output projection moves into the combine).
 * With q_len > 1 every token of a head uses that head's W. Caller-owned device
 * memory, read only.
 */
typedef struct da_proj_t {
    const void *w;        /* DEVICE: element (h, e, c) at h*head_stride + e*row_stride
                             + c, 16-byte aligned                                   */
    int32_t w_dtype;      /* DA_F32 or DA_BF16                                    */
    int32_t out_dim;      /* projected width per head, 1 .. 256                    */
    int64_t head_stride;  /* elements between heads' matrices; 0: out_dim*row_stride
                             (byte size a multiple of 16)                          */
    int64_t row_stride;   /* elements between rows of one head; 0: v_dim (>= v_dim,
                             byte size a multiple of 16)                           */
} da_proj_t;

/*
 * decode_attn_combine_proj -- decode_attn_combine_ranks followed, in the same
 * kernel, by the projection `proj`: out is [batch][q_len][n_heads][out_dim]
 * in args->out_dtype. The merge is the one of decode_attn_combine_ranks
 * (n_ranks = 1: decode_attn_combine); v_dim must be a multiple of 8 and at
 * most 1024. One launch of clusters of ceil(v_dim / 128) CTAs per (sequence,
 * query head); the weights are fetched while the split kernel drains. A
 * weight load that does not finish within args->timeout_us sets the status
 * word of the first workspace (decode_attn_device_status: "combine
 * (projection)") and leaves that part of out undefined. Errors as
 * decode_attn_combine, plus DA_EUNSUPPORTED for a weight type, out_dim or
 * v_dim outside the above and DA_EINVAL for misaligned weights.
 */
int decode_attn_combine_proj(const da_args_t *args, const da_plan_t *plan,
                             const da_proj_t *proj, const void *workspaces, int n_ranks,
                             void *out, da_stream_t stream);

/*
 * decode_attn_splitk_proj -- decode_attn_splitk_ex whose combine is
 * decode_attn_combine_proj: the split kernel, then the merge with the
 * projection, two launches on `stream`; out is [batch][q_len][n_heads]
 * [out_dim]. DA_FLAG_NO_COMBINE is ignored.
 */
int decode_attn_splitk_proj(const da_args_t *args, const da_plan_t *plan, const da_proj_t *proj,
                            const float *q, const void *k_cache, const void *v_cache, void *out,
                            void *workspace, size_t workspace_bytes, da_stream_t stream);

/*
 * decode_attn_splitk -- the short form: batch 1, f32 q/K/V/out,
 * v_dim = head_dim, caches laid out [seq_len][n_kv_heads][head_dim]
 * contiguous, scale given.
 *   seq_lens  HOST int32[1]: the context length L (>= 1)
 * Plans on the host and runs split + combine on `stream` using a workspace
 * the library owns, one per device ("Attention at 128k" §2: per-device
 * scratch). The first call on a device, and a call that needs a larger
 * workspace than before, allocates it with cudaMalloc (which synchronises);
 * decode_attn_release() frees them.
 * Every short-form call on a device shares that one workspace. The library
 * holds a lock while it enqueues, so no call launches on a workspace that
 * another thread is replacing. But calls whose kernels overlap on the GPU
 * (several streams, or several threads) race on the workspace's contents:
 * serialise them, or give each stream its own workspace through
 * decode_attn_splitk_ex.
 */
int decode_attn_splitk(const float *q, const float *k_cache, const float *v_cache,
                       const int32_t *seq_lens, int n_heads, int n_kv_heads, int head_dim,
                       float scale, float *out, da_stream_t stream);

/*
 * decode_attn_device_status -- synchronise `stream`, then read and clear the
 * status word at the start of `workspace` that the split kernel sets when a
 * bounded wait runs out. Returns DA_OK, DA_ETIMEOUT (message names the
 * kernel), or DA_ECUDA if the synchronisation itself failed.
 */
int decode_attn_device_status(void *workspace, da_stream_t stream);

/*
 * decode_attn_splitk_noalloc -- decode_attn_splitk_ex for callers that cannot
 * allocate device memory. The pages have no counterpart to it.
 *
 * Some callers cannot call cudaMalloc: code that runs while the device must
 * not synchronise (cudaMalloc can), hosts whose memory manager owns all device
 * memory and forbids raw allocations, and plugins that get no allocator handle.
 * This entry point takes no workspace: the partials live in a file-scope
 * device array of 16 MiB inside the library, which every GPU that loads the
 * library keeps until the process exits. It calls no cudaMalloc, cudaFree or
 * other allocating routine.
 *   - Same arguments and behaviour as decode_attn_splitk_ex minus the
 *     workspace; the caller still passes q, the caches and out.
 *   - Returns DA_ENOSPACE, with a message naming the limit, when
 *     plan->workspace_bytes exceeds 16 MiB (at most 16 MiB / (4 * (v_dim + 2))
 *     (query head, split) partials).
 *   - The first call on a device looks the array up once with
 *     cudaGetSymbolAddress (with that device current); make that first call
 *     before any stream capture.
 *   - Every call on a device shares the one array, which keeps the last call's
 *     contents: calls that overlap on the GPU (other streams, other threads)
 *     race and corrupt each other's partials. Serialise them.
 *   - DA_FLAG_NO_COMBINE is refused (DA_EINVAL): the partials would stay in
 *     the private array, where no later call could combine them.
 *   - Treat the output of this entry point as unchecked for in-kernel
 *     timeouts. A bounded wait that runs out sets a status word inside the
 *     private array, which the host cannot read and the next call clears; the
 *     output of such a call is wrong and nothing reports it. Callers that need
 *     that check use decode_attn_splitk_ex with a workspace and
 *     decode_attn_device_status.
 */
int decode_attn_splitk_noalloc(const da_args_t *args, const da_plan_t *plan, const float *q,
                               const void *k_cache, const void *v_cache, void *out,
                               da_stream_t stream);

/*
 * Device-side lengths and paged caches for decode_attn_splitk_dev.
 * "The Kernel Level: Attention and MoE" (llm-serving.xyz lecture 07), sections
 * "A kernel alone is not a serving system" and the CUDA-graph section: the
 * kernel indexes K/V through a block table, and the step is captured once and
 * replayed, so everything that changes per step lives in device memory.
 *   seq_lens      DEVICE int32[batch], the current length of every sequence,
 *                 read by the kernel; each is clamped to [1, plan->seq_lens[b]]
 *                 (make the plan for the largest lengths the launch will see).
 *                 NULL: the plan's lengths. It must not change while a call
 *                 that reads it is in flight.
 *   block_table   DEVICE int32[batch * max_blocks_per_seq], or NULL for the
 *                 contiguous caches of da_args_t. Entry [b][i] is the pool block
 *                 that holds positions [i * block_size, (i + 1) * block_size)
 *                 of sequence b. Entries past a sequence's length may be loaded,
 *                 and the GQA kernels may copy rows of the blocks they name by TMA
 *                 for positions they then mask (any value is safe there: TMA reads
 *                 zeros outside the pool); no result depends on them.
 *                 With a table, k_cache / v_cache point at pools whose element
 *                 (block, slot, kv, d) is at base + block * *_block_stride +
 *                 slot * *_pos_stride + kv * *_head_stride + d (elements);
 *                 capacity and the batch strides of da_args_t are not used for
 *                 addressing (capacity must still cover every length).
 *   block_size    positions per block: a positive multiple of 16. Tiles run
 *                 across block ends, so every block size streams whole tiles:
 *                 the SIMT GQA kernel copies a tile that lies in one block as one
 *                 TMA box and one that spans a block end as boxes of
 *                 gcd(tile, block_size) rows, the tensor-core GQA kernel every
 *                 tile as boxes of gcd(64, block_size) rows; boxes start at
 *                 multiples of their height, so the plan's chunks must be
 *                 multiples of gcd(tile, block_size) (the planner's are
 *                 multiples of the tile; DA_EINVAL otherwise). The MLA kernel
 *                 looks up every row.
 *   num_blocks    blocks in each pool; table entries must be < num_blocks.
 *   k_block_stride, v_block_stride  elements between blocks (16-byte multiples,
 *                 at least block_size * pos_stride).
 */
typedef struct {
    const int32_t *seq_lens;
    const int32_t *block_table;
    int32_t max_blocks_per_seq;
    int32_t block_size;
    int32_t num_blocks;
    int32_t reserved;           /* 0 */
    int64_t k_block_stride;
    int64_t v_block_stride;
} da_dev_t;

/*
 * decode_attn_splitk_dev -- decode_attn_splitk_ex with lengths read on the
 * device and, optionally, paged K/V caches (da_dev_t). It makes no host-side
 * decision that depends on the current lengths, so a launch captured in a CUDA
 * graph stays valid while the lengths grow up to the plan's. Splits that start
 * past a sequence's current length write neutral partials (l = 0). Both
 * kernels: for the MLA shape the pool holds the latent rows once (k_cache ==
 * v_cache, equal block strides). Validation before any launch as in
 * decode_attn_splitk_ex, plus the da_dev_t rules above (DA_EINVAL /
 * DA_EUNSUPPORTED).
 */
int decode_attn_splitk_dev(const da_args_t *args, const da_plan_t *plan, const da_dev_t *dev,
                           const float *q, const void *k_cache, const void *v_cache, void *out,
                           void *workspace, size_t workspace_bytes, da_stream_t stream);

/* Thread-local description of the last failure on this thread ("" if none). */
const char *decode_attn_last_error(void);

/* Frees the short form's per-device workspaces (synchronises each device). */
void decode_attn_release(void);

/* Library version string. */
const char *decode_attn_version(void);

#ifdef __cplusplus
}
#endif

#endif /* SPLIT_KV_DECODE_H */
