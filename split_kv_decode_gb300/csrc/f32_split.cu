// Split kernel in f32 on the CUDA cores, for MLA work items over an f32
// latent cache, sm_103a.
//
// It serves MLA as MQA, whose rows outnumber what the warp-per-row SIMT kernel
// holds in registers (the template also takes separate K and V caches of one
// width; the library instantiates the MLA shape only):
//   * MLA as MQA: every query row attends over one shared 576-wide latent row
//     per position, and the values are the first 512 columns of the same rows
//     ("Attention at 128k", §1.1 and §4; "The Kernel Level", absorbed MLA
//     decode). The tensor-core MLA kernel rounds q, the latent rows and the
//     probabilities to bf16; with few attended positions a single value row's
//     rounding (up to 2^-9 of it) shows in the output, so the library sends
//     sequences whose current length is below DA_MLA_EXACT_BELOW here (and any
//     sequence when the caller asks for it). The choice is made on the device,
//     from the same length both kernels read, so a captured launch follows a
//     context that grows past the threshold.
// Every operand is f32: the scores and the weighted sum carry f32 rounding only.
//
// Work split: one CTA per (work item, group of 32 rows); a work item is a
// contiguous slice of one sequence's context for one KV head ("Attention at
// 128k" §2). The CTA walks its slice in tiles of 32 positions, K (and V) rows
// double-buffered in shared memory by cp.async. A lane owns one row of the
// group in every warp, and warp c owns two slices of the work:
//   * columns [c DK/8, (c+1) DK/8) of the QK product: its q slice stays in
//     registers, each key row is read as broadcast 128-bit loads, and the
//     eight warps' partial dot products are summed through shared memory;
//   * value columns [c DV/8, (c+1) DV/8) of the PV product, accumulated in
//     registers across the whole slice.
// Every warp runs the online softmax (m, l) of its lane's row over the tile
// (KL07's recurrence; the same inputs in the same order, so all eight copies
// agree bit for bit), which leaves each warp the probabilities and the
// rescale factor of exactly the rows it accumulates: no broadcast is needed.
// The item's partial (m, l, acc[DV]) per row goes to the workspace in the
// layout the combine kernel reads, like every other split kernel.
//
// There is no wait on another role or CTA here (only __syncthreads and
// cp.async groups of the CTA itself), so no bounded wait is needed. Rows of a
// group past the item's rows compute on zero q and are not written.
#include <climits>
#include <cstdint>

#include "internal.h"
#include "ptx.cuh"

namespace skv {
namespace {

constexpr int kRows = 32;  // rows per CTA, one per lane
constexpr int kTP = 32;    // positions per staged tile
constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;

template <int DK, int DV, bool SHARED> struct Shape {
    static constexpr int DS = DK / kWarps;                     // QK columns per warp
    static constexpr int ES = DV / kWarps;                     // value columns per warp
    static constexpr int KROW = DK * 4, VROW = SHARED ? 0 : DV * 4; // bytes per staged row
    static constexpr int TILE = kTP * (KROW + VROW);           // one buffer (K tile, V tile)
    static constexpr int PIECES = TILE / 16;                   // 16-byte cp.async pieces
    static constexpr int SMR = kWarps * kTP * kRows * 4;       // partial dot products
    static constexpr int SMEM = 2 * TILE + SMR;
    static_assert(DS % 8 == 0 && ES % 4 == 0, "slices of float4");
    static_assert(PIECES % kThreads == 0, "whole cp.async rounds");
    static_assert(!SHARED || DV <= DK, "values are a prefix of the key row");
    static_assert(SMEM <= 232448, "shared memory");
};

__device__ __forceinline__ void cp_async16(uint32_t saddr, const void *g)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(saddr), "l"(g) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N> __device__ __forceinline__ void cp_async_wait()
{
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

template <int DK, int DV, bool SHARED>
__global__ void __launch_bounds__(kThreads, 1) f32_split_kernel(const __grid_constant__ F32Params p)
{
    using S = Shape<DK, DV, SHARED>;
    extern __shared__ __align__(16) uint8_t sm[];
    float *R = reinterpret_cast<float *>(sm + 2 * S::TILE); // [warp][position][row]
    const uint32_t sbase = smem_u32(sm);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const ItemTable &it = p.items;
    const int hkv = it.n_kv_heads;
    const int rows_item = p.n_heads / hkv;        // (token, head) rows of a work item
    const int Gh = p.hq / hkv;                    // query heads per KV head
    const int n_groups = (rows_item + kRows - 1) / kRows;
    const int item = blockIdx.x / n_groups, group = blockIdx.x % n_groups;
    if (p.reset_status && blockIdx.x == 0 && threadIdx.x == 0) *p.status = 0;

    // item -> (sequence, KV head, split, positions [p0, p1)); items run over
    // (sequence, split, KV head) like the other split kernels
    const int t = item / hkv, kvh = item - t * hkv;
    int lo = 0, hi = it.batch - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (it.split_base[mid] <= t) lo = mid;
        else hi = mid - 1;
    }
    const int b = lo;
    int L = it.seq_lens[b];
    if (p.dev_lens) L = max(p.q_len, min(__ldg(p.dev_lens + b), L));
    if (L >= p.exact_below) return; // the tensor-core MLA kernel serves this sequence
    const int s = t - it.split_base[b];
    const int p0 = s * it.chunk[b];
    const int p1 = min(L, p0 + it.chunk[b]);
    // this lane's row of the item: token j / Gh, head kvh * Gh + j % Gh
    const int j = group * kRows + lane;
    const bool row_ok = j < rows_item;
    const int token = row_ok ? j / Gh : 0;
    const int row = token * p.hq + kvh * Gh + (row_ok ? j - token * Gh : 0); // row of the sequence
    const size_t rowg = ((size_t)it.split_base[b] + s) * p.n_heads + row;
    if (p1 <= p0) { // a split past the current length: neutral partial
        if (warp == 0 && row_ok) p.ml[rowg] = make_float2(kNeutralM, 0.f);
        return;
    }
    // this row's token sees positions below lim (causal among the new tokens)
    const int lim = (p.flags & DA_FLAG_NO_CAUSAL) ? (INT_MAX >> 1) : L - p.q_len + 1 + token;

    auto key_row = [&](int pos, const float *base, int64_t pos_st, int64_t head_st,
                       int64_t batch_st, int64_t block_st) -> const float * {
        if (p.block_table) {
            const int idx = pos / p.block_size;
            const int blk = __ldg(p.block_table + (size_t)b * p.max_blocks + idx);
            return base + (size_t)blk * block_st + (size_t)(pos - idx * p.block_size) * pos_st +
                   (size_t)kvh * head_st;
        }
        return base + (size_t)b * batch_st + (size_t)pos * pos_st + (size_t)kvh * head_st;
    };
    // tile t -> buffer: the K rows (and the V rows) of positions [p0 + 32t, +32);
    // rows past the slice repeat its last row (finite; their probabilities are
    // zero)
    auto load_tile = [&](int tt, int buf) {
        const int base = p0 + tt * kTP;
        const uint32_t dst = sbase + buf * S::TILE;
        for (int i = threadIdx.x; i < S::PIECES; i += kThreads) {
            const int byte = i * 16;
            const float *src;
            if (SHARED || byte < kTP * S::KROW) {
                const int pos = min(base + byte / S::KROW, p1 - 1);
                src = key_row(pos, p.k, p.k_pos_stride, p.k_head_stride, p.k_batch_stride,
                              p.k_block_stride) + (byte % S::KROW) / 4;
            } else {
                constexpr int VROW = SHARED ? 1 : S::VROW; // (never 0 here)
                const int vb = byte - kTP * S::KROW;
                const int pos = min(base + vb / VROW, p1 - 1);
                src = key_row(pos, p.v, p.v_pos_stride, p.v_head_stride, p.v_batch_stride,
                              p.v_block_stride) + (vb % VROW) / 4;
            }
            cp_async16(dst + byte, src);
        }
        cp_async_commit();
    };
    load_tile(0, 0);

    // this lane's row of q, columns of this warp's QK slice, in registers with
    // scale * log2(e) folded in; as pairs, for the paired FMA (two f32 FMAs per
    // instruction, each rounded as fmaf)
    float2 qr[S::DS / 2];
    {
        const float4 *qs = reinterpret_cast<const float4 *>(
            p.q + ((size_t)b * p.n_heads + row) * DK + warp * S::DS);
        const float f = row_ok ? p.scale_log2 : 0.f;
#pragma unroll
        for (int i = 0; i < S::DS / 4; ++i) {
            const float4 v = __ldg(qs + i);
            qr[2 * i] = make_float2(v.x * f, v.y * f);
            qr[2 * i + 1] = make_float2(v.z * f, v.w * f);
        }
    }

    float2 o[S::ES / 2]; // O[row][ES warp + e], unnormalised, as pairs of columns
#pragma unroll
    for (int e = 0; e < S::ES / 2; ++e) o[e] = make_float2(0.f, 0.f);
    float m = -INFINITY, l = 0.f;
    const int ntiles = (p1 - p0 + kTP - 1) / kTP;

    for (int tt = 0; tt < ntiles; ++tt) {
        const int buf = tt & 1;
        if (tt + 1 < ntiles) {
            load_tile(tt + 1, buf ^ 1);
            cp_async_wait<1>();
        } else {
            cp_async_wait<0>();
        }
        __syncthreads(); // tile tt is in shared memory for every thread
        const float *Kt = reinterpret_cast<const float *>(sm + buf * S::TILE);
        const float *Vt = SHARED ? Kt : Kt + kTP * DK;
        constexpr int VSTRIDE = SHARED ? DK : DV; // floats between staged value rows

        // partial scores over this warp's columns, four positions at a time
        // (eight independent accumulator pairs, so the FMAs do not wait on each
        // other)
#pragma unroll 1
        for (int j0 = 0; j0 < kTP; j0 += 4) {
            float2 acc[4][2];
#pragma unroll
            for (int u = 0; u < 4; ++u) acc[u][0] = acc[u][1] = make_float2(0.f, 0.f);
#pragma unroll
            for (int i = 0; i < S::DS / 4; ++i) {
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const float4 k4 =
                        reinterpret_cast<const float4 *>(Kt + (j0 + u) * DK + warp * S::DS)[i];
                    acc[u][0] = __ffma2_rn(qr[2 * i], make_float2(k4.x, k4.y), acc[u][0]);
                    acc[u][1] = __ffma2_rn(qr[2 * i + 1], make_float2(k4.z, k4.w), acc[u][1]);
                }
            }
#pragma unroll
            for (int u = 0; u < 4; ++u)
                R[(warp * kTP + j0 + u) * kRows + lane] =
                    (acc[u][0].x + acc[u][1].x) + (acc[u][0].y + acc[u][1].y);
        }
        __syncthreads();
        // full scores of positions [4 warp, 4 warp + 4): the eight slices summed
        // in a fixed order, written over slice 0 (no other warp reads these
        // positions of slice 0)
#pragma unroll
        for (int q = 0; q < kTP / kWarps; ++q) {
            const int jj = warp * (kTP / kWarps) + q;
            float sum = 0.f;
#pragma unroll
            for (int c = 0; c < kWarps; ++c) sum += R[(c * kTP + jj) * kRows + lane];
            R[jj * kRows + lane] = sum;
        }
        __syncthreads();

        // online softmax of this lane's row over the tile
        const int nvalid = max(0, min(kTP, min(p1, lim) - (p0 + tt * kTP)));
        float tmax = -INFINITY;
#pragma unroll
        for (int jj = 0; jj < kTP; ++jj)
            if (jj < nvalid) tmax = fmaxf(tmax, R[jj * kRows + lane]);
        const float mn = fmaxf(m, tmax);
        if (mn != m) { // the running max moved: rescale (m = -inf: nothing held yet)
            const float alpha = (m == -INFINITY) ? 0.f : ex2(m - mn);
            l *= alpha;
#pragma unroll
            for (int e = 0; e < S::ES / 2; ++e) {
                o[e].x *= alpha;
                o[e].y *= alpha;
            }
            m = mn;
        }
        // O[row][this warp's value columns] += sum_j p_j V[j][.], with p_j formed
        // from the tile's scores as it goes (they stay in shared memory)
#pragma unroll(DK > 256 ? 1 : 4)
        for (int jj = 0; jj < kTP; ++jj) {
            const float pjj = (jj < nvalid) ? ex2(R[jj * kRows + lane] - m) : 0.f;
            l += pjj;
            const float4 *vr = reinterpret_cast<const float4 *>(Vt + jj * VSTRIDE + warp * S::ES);
            const float2 pp = make_float2(pjj, pjj);
#pragma unroll
            for (int i = 0; i < S::ES / 4; ++i) {
                const float4 v = vr[i];
                o[2 * i] = __ffma2_rn(pp, make_float2(v.x, v.y), o[2 * i]);
                o[2 * i + 1] = __ffma2_rn(pp, make_float2(v.z, v.w), o[2 * i + 1]);
            }
        }
        __syncthreads(); // before the next round overwrites this buffer and R
    }

    if (row_ok) {
        float4 *dst = reinterpret_cast<float4 *>(p.acc + rowg * DV + warp * S::ES);
#pragma unroll
        for (int i = 0; i < S::ES / 4; ++i)
            dst[i] = make_float4(o[2 * i].x, o[2 * i].y, o[2 * i + 1].x, o[2 * i + 1].y);
        if (warp == 0) p.ml[rowg] = make_float2(l > 0.f ? m * kLn2 : kNeutralM, l);
    }
    griddep_launch_dependents();
}

template <int DK, int DV, bool SHARED>
cudaError_t launch_t(int grid, cudaStream_t st, const F32Params &p)
{
    using S = Shape<DK, DV, SHARED>;
    auto *fn = f32_split_kernel<DK, DV, SHARED>;
    cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, S::SMEM);
    if (e != cudaSuccess) return e;
    fn<<<grid, kThreads, S::SMEM, st>>>(p);
    return cudaGetLastError();
}

} // namespace

int f32_split_groups(int rows_per_item) { return (rows_per_item + kRows - 1) / kRows; }

cudaError_t launch_f32_split(int head_dim, int v_dim, bool shared_kv, int grid, cudaStream_t st,
                             const F32Params &p)
{
    if (shared_kv && head_dim == 576 && v_dim == 512) return launch_t<576, 512, true>(grid, st, p);
    return cudaErrorInvalidValue;
}

} // namespace skv
