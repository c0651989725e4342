// MLA-as-MQA split kernel in f32 on the CUDA cores, sm_103a.
//
// The same product as the tensor-core MLA kernel -- every query row attends
// over one shared 576-wide latent row per position, and the values are the
// first 512 columns of the same rows ("Attention at 128k", §1.1 and §4; "The
// Kernel Level", absorbed MLA decode) -- but with every operand kept in f32:
// q, the latent rows and the probabilities are never rounded to a 16-bit type.
// The tensor-core kernel rounds all three to bf16, and with few attended
// positions a single value row's rounding (up to 2^-9 of it) shows in the
// output directly; here the scores and the weighted sum carry f32 rounding
// only. The library sends sequences whose current length is below
// DA_MLA_EXACT_BELOW positions here (where the work is small enough for the
// CUDA cores), and any sequence when the caller asks for it; the choice is
// made on the device, from the same length both kernels read, so a captured
// launch follows a context that grows past the threshold.
//
// Work split: one CTA per (work item, group of 32 query rows); a work item is
// a contiguous slice of one sequence's context ("Attention at 128k" §2). The
// CTA walks its slice in tiles of 32 latent rows, double-buffered in shared
// memory by cp.async. A lane owns one query row (lane = row of the group) in
// every warp, and warp c owns two slices of the work:
//   * columns [72c, 72c + 72) of the QK product: its q slice stays in
//     registers, each latent row is read as broadcast 128-bit loads, and the
//     eight warps' partial dot products are summed through shared memory;
//   * value columns [64c, 64c + 64) of the PV product, accumulated in
//     registers across the whole slice.
// Every warp runs the online softmax (m, l) of its lane's row over the tile
// (KL07's recurrence; the same inputs in the same order, so all eight copies
// agree bit for bit), which leaves each warp the probabilities and the
// rescale factor of exactly the rows it accumulates: no broadcast is needed.
// The item's partial (m, l, acc[512]) per row goes to the workspace in the
// layout the combine kernel reads, like every other split kernel.
//
// There is no wait on another role or CTA here (only __syncthreads and
// cp.async groups of the CTA itself), so no bounded wait is needed.
#include <climits>
#include <cstdint>

#include "internal.h"
#include "ptx.cuh"

namespace skv {
namespace {

constexpr int kDk = 576;
constexpr int kDv = 512;
constexpr int kRows = 32;                           // query rows per CTA, one per lane
constexpr int kTP = 32;                             // latent rows per staged tile
constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr int kDSlice = kDk / kWarps;               // 72 QK columns per warp
constexpr int kESlice = kDv / kWarps;               // 64 value columns per warp
constexpr int kRowChunks = kDk * 4 / 16;            // 144 16-byte pieces per latent row
constexpr int kTileBytes = kTP * kDk * 4;           // 73,728
constexpr int kPieces = kTileBytes / 16 / kThreads; // 18 cp.async per thread per tile
constexpr int kSmR = kWarps * kTP * kRows * 4;      // partial dot products, 32 KB
constexpr int kSmem = 2 * kTileBytes + kSmR;        // 180,224
static_assert(kDSlice % 4 == 0 && kESlice % 4 == 0, "slices of float4");
static_assert(kTileBytes % (16 * kThreads) == 0, "whole cp.async rounds");

__device__ __forceinline__ void cp_async16(uint32_t saddr, const void *g)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(saddr), "l"(g) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N> __device__ __forceinline__ void cp_async_wait()
{
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__global__ void __launch_bounds__(kThreads, 1) mla_exact_kernel(const __grid_constant__ MlaParams p)
{
    extern __shared__ __align__(16) uint8_t sm[];
    float *R = reinterpret_cast<float *>(sm + 2 * kTileBytes); // [warp][position][row]
    const uint32_t sbase = smem_u32(sm);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n_groups = (p.n_heads + kRows - 1) / kRows;
    const int item = blockIdx.x / n_groups, group = blockIdx.x % n_groups;
    const ItemTable &it = p.items;
    if (p.reset_status && blockIdx.x == 0 && threadIdx.x == 0) *p.status = 0;

    // item -> (sequence, split, positions [p0, p1))
    int lo = 0, hi = it.batch - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (it.split_base[mid] <= item) lo = mid;
        else hi = mid - 1;
    }
    const int b = lo;
    int L = it.seq_lens[b];
    if (p.dev_lens) L = max(p.q_len, min(__ldg(p.dev_lens + b), L));
    if (L >= p.exact_below) return; // the tensor-core kernel serves this sequence
    const int s = item - it.split_base[b];
    const int p0 = s * it.chunk[b];
    const int p1 = min(L, p0 + it.chunk[b]);
    const int row = group * kRows + lane;
    const bool row_ok = row < p.n_heads;
    const size_t rowg = ((size_t)it.split_base[b] + s) * p.n_heads + row;
    if (p1 <= p0) { // a split past the current length: neutral partial
        if (warp == 0 && row_ok) p.ml[rowg] = make_float2(kNeutralM, 0.f);
        return;
    }
    // this row's token sees positions below lim (causal among the new tokens)
    const int lim = (p.flags & DA_FLAG_NO_CAUSAL) ? (INT_MAX >> 1)
                                                   : L - p.q_len + 1 + row / p.hq;

    const float *cache = static_cast<const float *>(p.cache); // an f32 cache
    auto row_src = [&](int pos) -> const float * {
        if (p.block_table) {
            const int idx = pos / p.block_size;
            const int blk = __ldg(p.block_table + (size_t)b * p.max_blocks + idx);
            return cache + (size_t)blk * p.block_stride +
                   (size_t)(pos - idx * p.block_size) * p.pos_stride;
        }
        return cache + (size_t)b * p.batch_stride + (size_t)pos * p.pos_stride;
    };
    // tile t -> buffer: rows past the slice repeat its last row (finite; their
    // probabilities are zero)
    auto load_tile = [&](int t, int buf) {
        const int base = p0 + t * kTP;
        const uint32_t dst = sbase + buf * kTileBytes;
#pragma unroll 6
        for (int i = 0; i < kPieces; ++i) {
            const int c = threadIdx.x + i * kThreads; // 16-byte piece of the tile
            const int r = c / kRowChunks, col = c - r * kRowChunks;
            cp_async16(dst + c * 16, row_src(min(base + r, p1 - 1)) + col * 4);
        }
        cp_async_commit();
    };
    load_tile(0, 0);

    // this lane's row of q, columns of this warp's QK slice, in registers with
    // scale * log2(e) folded in
    float4 qr[kDSlice / 4];
    {
        const float4 *qs = reinterpret_cast<const float4 *>(
            p.q + ((size_t)b * p.n_heads + (row_ok ? row : 0)) * kDk + warp * kDSlice);
#pragma unroll
        for (int i = 0; i < kDSlice / 4; ++i) {
            float4 v = __ldg(qs + i);
            const float f = row_ok ? p.scale_log2 : 0.f;
            qr[i] = make_float4(v.x * f, v.y * f, v.z * f, v.w * f);
        }
    }

    float o[kESlice]; // O[row][64 warp + e], unnormalised
#pragma unroll
    for (int e = 0; e < kESlice; ++e) o[e] = 0.f;
    float m = -INFINITY, l = 0.f;
    const int ntiles = (p1 - p0 + kTP - 1) / kTP;

    for (int t = 0; t < ntiles; ++t) {
        const int buf = t & 1;
        if (t + 1 < ntiles) {
            load_tile(t + 1, buf ^ 1);
            cp_async_wait<1>();
        } else {
            cp_async_wait<0>();
        }
        __syncthreads(); // tile t is in shared memory for every thread
        const float *K = reinterpret_cast<const float *>(sm + buf * kTileBytes);

        // partial scores over this warp's 72 columns, every position of the tile
#pragma unroll 2
        for (int j = 0; j < kTP; ++j) {
            const float4 *kr = reinterpret_cast<const float4 *>(K + j * kDk + warp * kDSlice);
            float a0 = 0.f, a1 = 0.f;
#pragma unroll
            for (int i = 0; i < kDSlice / 4; i += 2) {
                const float4 k0 = kr[i], k1 = kr[i + 1];
                a0 = fmaf(qr[i].x, k0.x, a0);
                a0 = fmaf(qr[i].y, k0.y, a0);
                a0 = fmaf(qr[i].z, k0.z, a0);
                a0 = fmaf(qr[i].w, k0.w, a0);
                a1 = fmaf(qr[i + 1].x, k1.x, a1);
                a1 = fmaf(qr[i + 1].y, k1.y, a1);
                a1 = fmaf(qr[i + 1].z, k1.z, a1);
                a1 = fmaf(qr[i + 1].w, k1.w, a1);
            }
            R[(warp * kTP + j) * kRows + lane] = a0 + a1;
        }
        __syncthreads();
        // full scores of positions [4 warp, 4 warp + 4): the eight slices summed
        // in a fixed order, written over slice 0 (no other warp reads these
        // positions of slice 0)
#pragma unroll
        for (int jj = 0; jj < kTP / kWarps; ++jj) {
            const int j = warp * (kTP / kWarps) + jj;
            float sum = 0.f;
#pragma unroll
            for (int c = 0; c < kWarps; ++c) sum += R[(c * kTP + j) * kRows + lane];
            R[j * kRows + lane] = sum;
        }
        __syncthreads();

        // online softmax of this lane's row over the tile
        const int nvalid = max(0, min(kTP, min(p1, lim) - (p0 + t * kTP)));
        float pj[kTP];
        float tmax = -INFINITY;
#pragma unroll
        for (int j = 0; j < kTP; ++j) {
            pj[j] = R[j * kRows + lane];
            if (j < nvalid) tmax = fmaxf(tmax, pj[j]);
        }
        const float mn = fmaxf(m, tmax);
        if (mn != m) { // the running max moved: rescale (m = -inf: nothing held yet)
            const float alpha = (m == -INFINITY) ? 0.f : ex2(m - mn);
            l *= alpha;
#pragma unroll
            for (int e = 0; e < kESlice; ++e) o[e] *= alpha;
            m = mn;
        }
#pragma unroll
        for (int j = 0; j < kTP; ++j) {
            pj[j] = (j < nvalid) ? ex2(pj[j] - m) : 0.f;
            l += pj[j];
        }
        // O[row][this warp's 64 columns] += sum_j p_j V[j][.]
#pragma unroll
        for (int j = 0; j < kTP; ++j) {
            const float4 *vr = reinterpret_cast<const float4 *>(K + j * kDk + warp * kESlice);
#pragma unroll
            for (int i = 0; i < kESlice / 4; ++i) {
                const float4 v = vr[i];
                o[4 * i + 0] = fmaf(pj[j], v.x, o[4 * i + 0]);
                o[4 * i + 1] = fmaf(pj[j], v.y, o[4 * i + 1]);
                o[4 * i + 2] = fmaf(pj[j], v.z, o[4 * i + 2]);
                o[4 * i + 3] = fmaf(pj[j], v.w, o[4 * i + 3]);
            }
        }
        __syncthreads(); // before the next round overwrites this buffer and R
    }

    if (row_ok) {
        float4 *dst = reinterpret_cast<float4 *>(p.acc + rowg * kDv + warp * kESlice);
#pragma unroll
        for (int i = 0; i < kESlice / 4; ++i)
            dst[i] = make_float4(o[4 * i], o[4 * i + 1], o[4 * i + 2], o[4 * i + 3]);
        if (warp == 0) p.ml[rowg] = make_float2(l > 0.f ? m * kLn2 : kNeutralM, l);
    }
    griddep_launch_dependents();
}

} // namespace

int mla_exact_groups(int rows) { return (rows + kRows - 1) / kRows; }

cudaError_t launch_mla_exact(int grid, cudaStream_t st, const MlaParams &p)
{
    cudaError_t e = cudaFuncSetAttribute(mla_exact_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
    if (e != cudaSuccess) return e;
    mla_exact_kernel<<<grid, kThreads, kSmem, st>>>(p);
    return cudaGetLastError();
}

} // namespace skv
