// MLA-as-MQA split kernel on tcgen05 tensor cores, sm_103a.
//
// Multi-head latent attention at decode is MQA: every query head attends over
// one shared 576-wide latent row per position (512 latent + 64 rope columns),
// and the values are the first 512 columns of the same rows ("Attention at
// 128k", §1.1 and §4; "The Kernel Level", absorbed MLA decode). With 96 heads
// against one shared latent, every tile is a real dense contraction:
//     S[h][pos]  = sum_d Q[h][d] * K[pos][d]          (M = heads, N = 64 positions, K = 576)
//     O^T[e][h] += sum_pos V[pos][e] * P[h][pos]      (M = 512 in 4 blocks of 128, N = heads)
// Both products run on the tensor cores (bf16 operands, f32 accumulation in
// TMEM), and each latent byte is read from HBM once for all heads.
//
// Work split: a cluster of two CTAs (on two SMs) takes a work item, a
// contiguous slice of one sequence's context (split over context, "Attention at
// 128k" §2), and walks it in tiles of 64 positions. CTA r:
//   * converts rows [32r, 32r + 32) of every tile from f32 to bf16 into its own
//     shared memory and ships them to the peer CTA with bulk shared-memory
//     copies, so every row is read from HBM once and converted once;
//   * owns query rows [r*N, r*N + N), N = rows / 2 (a row is a query head, or
//     with several new tokens per sequence a (token, head) pair, token-major,
//     whose token sees the positions up to its own): their bf16 Q (scale and
//     log2 e folded in), S and O^T in its TMEM, and their partials.
// The tile buffer is double-buffered (two slots of nine 64-column chunks,
// 128-byte-swizzled, K-major), so the converters fill tile t+1 while the
// tensor core and the softmax work on tile t. A chunk is the B operand of the
// QK product (64 positions x 64 columns) and, read MN-major, half an M block
// of the PV product (64 value columns x 64 positions).
//
// Roles (14 warps):
//   warps 0-3   softmax and epilogue. S uses the 64-row TMEM layout, in which
//               head h sits in lane 32*(h/16) + h%16; so thread (w, l < 16) owns
//               head 16w + l: its 64 scores, running max m and sum l stay in
//               registers, and its probability row is one 128-byte row of P.
//               All 128 threads (one per TMEM lane) read O^T in the epilogue.
//   warps 4-11  converters: 4 rows each; a whole tile row (nine 64-column chunks)
//               of 128-bit loads in flight per lane.
//               They only store and arrive on a barrier: no proxy fence, so
//               their loads stay in flight across tiles.
//   warp 12     TMEM allocation and the one thread that issues the MMAs; it
//               polls both products and issues whichever is ready: QK(t+1)
//               once the tile is in, PV(t) once P(t) is written.
//   warp 13     publisher: once the converters have stored a tile half, it
//               makes the stores visible to the async proxy (one fence per
//               tile, on the synchronisation path from the stores to the
//               tensor core and to the bulk copies), ships the half to the peer
//               CTA as nine 4 KB bulk copies and releases the tile to the MMA.
// Q has N real rows; the 64-row MMA reads 64 rows from each Q chunk, so rows
// N..63 alias the next chunk (or slack). Those rows give S rows that no thread
// reads.
//
// The running max is moved lazily: a head's reference m changes only when a
// tile holds a score above m + 8 (log2 units), so P <= 2^8 and l, O^T cannot
// overflow, and O^T (whose column h spans all lanes) is rescaled only then.
// Any reference gives the same partial after normalisation.
#include <atomic>
#include <climits>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "internal.h"
#include "merge.cuh"
#include "ptx.cuh"

namespace skv {
namespace {

constexpr int kDk = 576;
constexpr int kDv = 512;
constexpr int kTile = 64;                         // positions per tile = QK N
constexpr int kChunks = 9;                        // 64-column chunks of a latent row
constexpr int kChunkBytes = kTile * 128;          // 8 KB
constexpr int kSlotBytes = kChunks * kChunkBytes; // 72 KB
constexpr int kSoftWarps = 4;
constexpr int kConvWarps = 8;
constexpr int kRowsPerConv = 32 / kConvWarps;     // rows of the half-tile per converter warp
constexpr int kMmaWarp = kSoftWarps + kConvWarps;
constexpr int kPubWarp = kMmaWarp + 1;
constexpr int kThreads = (kPubWarp + 1) * 32;
constexpr float kTau = 8.f;                       // lazy-rescale threshold (log2 units)
constexpr int kGroups = 3;                        // a tile is released to the MMA in 3 chunk groups
constexpr int kGroupChunks = kChunks / kGroups;
constexpr int kPeerTx = kGroupChunks * kConvWarps * kRowsPerConv * 128; // bytes the peer ships per group

// P of a tile (N rows of 64 positions, 128 B each) lives in the tile's own
// slot, over its last chunk (the 64 rope columns): that chunk is read by the
// tile's QK product and, for this CTA's rows, by the bulk copy to the peer. The
// softmax writes P once the QK products of both CTAs are done (the peer's waited
// for the copy), and the slot is refilled only after both CTAs' PV products of
// the tile are done.
constexpr int kPChunk = kChunks - 1;

template <int N> struct Layout {
    static constexpr int TILE = 0;                          // 2 slots x 72 KB
    static constexpr int QCH = N * 128;                     // one Q chunk (N rows)
    static constexpr int Q = TILE + 2 * kSlotBytes;
    static constexpr int QEND = Q + kChunks * QCH + (kTile * 128 - QCH); // 64-row reads stay inside
    static constexpr int BAR = (QEND + 15) / 16 * 16;
    static constexpr int NBAR = 28;
    static constexpr int MISC = BAR + NBAR * 8;             // tmem base, abort flag
    static constexpr int ALPHA = (MISC + 16 + 15) / 16 * 16; // float alpha[N]
    static constexpr int USED = ALPHA + N * 4;
    static constexpr int ALLOC = USED + 1024;
    static constexpr int O_COL = 128;                       // O^T block j at O_COL + j*N
    static constexpr int TMEM_COLS = O_COL + 4 * N <= 256 ? 256 : 512;
    static_assert(N % 16 == 0 && N >= 16 && N <= 64, "heads per CTA");
    static_assert(QCH % 1024 == 0 && Q % 1024 == 0, "swizzle atoms");
    static_assert(ALLOC <= 232448, "shared memory");
};

// barrier indices (slot-indexed ones take +slot)
// B_FULL + kGroups*slot + g: chunk group g of the slot's tile is in (both halves);
// B_CONV + kGroups*slot + g: this CTA's converters have stored their rows of group g
constexpr int B_FULL = 0, B_EMPTY = 6, B_SFULL = 8, B_SFREE = 10, B_PFULL = 12, B_PFREE = 14,
              B_PVDONE = 16, B_OREADY = 17, B_OFREE = 18, B_QFULL = 19, B_QFREE = 20,
              B_DRAIN = 21, B_CONV = 22;

// byte offset of (row, byte) in a region of 128-byte rows with 128-byte swizzle
__device__ __forceinline__ uint32_t sw128(uint32_t row, uint32_t byte)
{
    return (row >> 3) * 1024 + (row & 7) * 128 + ((((byte >> 4) ^ row) & 7) << 4) + (byte & 15);
}

// The cache's element type CT and the MMA operand type: an f32 or bf16 cache
// feeds bf16 operands (q and P rounded to bf16), an f16 cache f16 operands.
template <typename CT> struct Operand {
    static constexpr bool kF16 = false;
    static __device__ __forceinline__ uint32_t pack(float a, float b)
    {
        __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
        return *reinterpret_cast<uint32_t *>(&h);
    }
};
template <> struct Operand<__half> {
    static constexpr bool kF16 = true;
    static __device__ __forceinline__ uint32_t pack(float a, float b)
    {
        __half2 h = __floats2half2_rn(a, b);
        return *reinterpret_cast<uint32_t *>(&h);
    }
};

__device__ __forceinline__ bool bar_or(int id, int threads, bool pred)
{
    uint32_t r;
    asm volatile("{\n\t.reg .pred p, q;\n\t"
                 "setp.ne.u32 p, %1, 0;\n\t"
                 "bar.red.or.pred q, %2, %3, p;\n\t"
                 "selp.u32 %0, 1, 0, q;\n\t}"
                 : "=r"(r)
                 : "r"((uint32_t)pred), "r"(id), "r"(threads)
                 : "memory");
    return r != 0;
}

struct Item {
    int b, s, p0, p1, ntiles, L; // L: the length the item's sequence attends over
    bool skip;                   // the exact f32 kernel serves this sequence
};

// item -> (sequence, split, positions [p0, p1), tiles). With lengths read on
// the device a split may start past its sequence's current end: an empty item.
__device__ __forceinline__ Item get_item(const MlaParams &p, int item)
{
    const ItemTable &it = p.items;
    Item x;
    int lo = 0, hi = it.batch - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (it.split_base[mid] <= item) lo = mid;
        else hi = mid - 1;
    }
    x.b = lo;
    x.s = item - it.split_base[lo];
    x.p0 = x.s * it.chunk[lo];
    int L = it.seq_lens[lo];
    if (p.dev_lens) L = max(p.q_len, min(__ldg(p.dev_lens + lo), L));
    x.L = L;
    x.p1 = min(L, x.p0 + it.chunk[lo]);
    x.skip = L < p.exact_below;
    x.ntiles = (x.p1 > x.p0 && !x.skip) ? (x.p1 - x.p0 + kTile - 1) / kTile : 0;
    return x;
}

// The (item, tile, chunk) units of a cluster's work, in order; gt counts tiles.
// Empty items have no tiles and are skipped.
struct Cursor {
    int item, t, c, gt;
    Item x;
    bool done;
    __device__ __forceinline__ void seek(const MlaParams &p, int stride)
    {
        for (;;) {
            done = item >= p.items.n_items;
            if (done) return;
            x = get_item(p, item);
            if (x.ntiles > 0) return;
            item += stride;
        }
    }
    __device__ __forceinline__ void start(const MlaParams &p, int first, int stride)
    {
        item = first;
        t = 0;
        c = 0;
        gt = 0;
        seek(p, stride);
    }
    __device__ __forceinline__ void next(const MlaParams &p, int stride)
    {
        if (++c == kChunks) {
            c = 0;
            ++gt;
            if (++t == x.ntiles) {
                t = 0;
                item += stride;
                seek(p, stride);
            }
        }
    }
    __device__ __forceinline__ void next_tile(const MlaParams &p, int stride)
    {
        c = kChunks - 1;
        next(p, stride);
    }
};

__device__ __forceinline__ void raise_abort(volatile int *abort_flag, uint32_t abort_peer,
                                            int *status)
{
    if (!*abort_flag) {
        *abort_flag = 1;
        st_cluster_u32(abort_peer, 1u);
        atomicCAS(status, 0, kStatusTimeoutMla);
    }
}

// The merge without a combine launch, once every CTA of the launch has written
// its partials. CTA c takes the (sequence, row, 128 value columns) units c,
// c + gridDim.x, ... and stages them in its tile slots, idle by now: bulk
// copies bring each split's 512-byte block of a unit, as many units per pass
// as fit, while warp k forms the weights w_s = e^{m_s - m} / sum_i e^{m_i - m} l_i
// of the pass's unit k from the (m, l) pairs (w_s = 0 for a neutral partial,
// whose block is never used). The warps then share out each unit's splits, sum
// w_s acc_s from shared memory and add their sums in a fixed order. A unit with
// more splits than the stage holds is merged from L2 by eight warps instead.
constexpr int kNW = kThreads / 32;
constexpr int kStageBytes = 2 * kSlotBytes;                 // the two tile slots
constexpr int kSBarOff = kStageBytes - 64;                  // staging mbarrier, pass header
constexpr int kRedOff = kSBarOff - kNW * 32 * 16;           // per-warp sums, float4 per lane
constexpr int kTabOff = kRedOff - 256;                      // the pass's unit table
constexpr int kPassUnits = 8;
constexpr int kBlk = 128 * 4;                               // bytes of one split's block

struct PassUnit {
    int b, row, z, S, off; // off: the unit's first block in the stage
};
static_assert(kPassUnits * sizeof(PassUnit) <= 256 && kPassUnits <= kNW, "pass table");
static_assert(kRedOff % 16 == 0 && kTabOff % 16 == 0, "staging alignment");

__device__ __noinline__ void mla_merge_staged(const MlaParams &p, uint8_t *sm)
{
    constexpr int CU = kDv / 128;
    const ItemTable &it = p.items;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int rows = p.n_heads, units = it.batch * rows * CU;
    uint64_t *sbar = reinterpret_cast<uint64_t *>(sm + kSBarOff);
    volatile int *hdr = reinterpret_cast<volatile int *>(sm + kSBarOff + 16); // nu, nb, next, ok
    PassUnit *tab = reinterpret_cast<PassUnit *>(sm + kTabOff);
    float4 *red = reinterpret_cast<float4 *>(sm + kRedOff);
    volatile int never = 0;
    // the tile slots' generic and tensor-core accesses, and the acquire of the
    // partials, before the bulk copies
    fence_proxy_async_smem();
    fence_proxy_async_global();
    __syncthreads();
    if (threadIdx.x == 0) {
        mbar_init(sbar, 1);
        fence_mbar_init();
    }
    __syncthreads();
    uint32_t phase = 0;
    for (int u = blockIdx.x; u < units;) {
        if (threadIdx.x == 0) {
            int nu = 0, nb = 0, v = u;
            while (v < units && nu < kPassUnits) {
                const int b = v / (rows * CU), r = v - b * (rows * CU);
                const int S = it.split_base[b + 1] - it.split_base[b];
                if ((nb + S) * (kBlk + 4) > kTabOff) break;
                tab[nu] = PassUnit{b, r / CU, r % CU, S, nb};
                nb += S;
                ++nu;
                v += gridDim.x;
            }
            hdr[0] = nu;
            hdr[1] = nb;
            hdr[2] = v;
            if (nu > 0) mbar_arrive_expect_tx(sbar, (uint32_t)(nb * kBlk));
        }
        __syncthreads();
        const int nu = hdr[0], nb = hdr[1], next = hdr[2];
        if (nu == 0) {
            // more splits than the stage holds: from L2, a warp per 16 columns
            const int b = u / (rows * CU), r = u - b * (rows * CU), row = r / CU;
            if (warp < 8)
                warp_merge_cols<4, 10>(p.ml, p.acc, (size_t)it.split_base[b],
                                       it.split_base[b + 1] - it.split_base[b], rows, row, kDv,
                                       (r % CU) * 32 + warp * 4, out_row_ptr(p.fused, b, rows, row, kDv),
                                       p.fused.out_dtype);
            __syncthreads(); // the header is read before it is rewritten
            u += gridDim.x;
            continue;
        }
        // block j of the pass: split j - off of the unit it falls in
        for (int j = threadIdx.x; j < nb; j += kThreads) {
            int k = 0;
            while (k + 1 < nu && tab[k + 1].off <= j) ++k;
            const PassUnit t = tab[k];
            const float *src = p.acc +
                               (((size_t)it.split_base[t.b] + (j - t.off)) * rows + t.row) * kDv +
                               t.z * 128;
            bulk_load_g2s(sm + (size_t)j * kBlk, src, kBlk, sbar);
        }
        float *wts = reinterpret_cast<float *>(sm + (size_t)nb * kBlk);
        if (warp < nu) {
            const PassUnit t = tab[warp];
            const float2 *ml = p.ml + (size_t)it.split_base[t.b] * rows + t.row;
            constexpr int WB = 4; // pairs per lane in flight at once: 128 splits per round trip
            float2 x[WB];
            float M = kNeutralM, L = 0.f;
            for (int s0 = 0; s0 < t.S; s0 += 32 * WB) {
#pragma unroll
                for (int i = 0; i < WB; ++i) {
                    const int s = s0 + 32 * i + lane;
                    x[i] = s < t.S ? __ldcg(ml + (size_t)s * rows) : make_float2(kNeutralM, 0.f);
                }
#pragma unroll
                for (int i = 0; i < WB; ++i) {
                    if (x[i].y > 0.f) {
                        const float mn = fmaxf(M, x[i].x);
                        L = L * ex2((M - mn) * kLog2e) + x[i].y * ex2((x[i].x - mn) * kLog2e);
                        M = mn;
                    }
                }
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                const float Mo = __shfl_xor_sync(0xffffffffu, M, o);
                const float Lo = __shfl_xor_sync(0xffffffffu, L, o);
                const float mn = fmaxf(M, Mo);
                L = L * ex2((M - mn) * kLog2e) + Lo * ex2((Mo - mn) * kLog2e);
                M = mn;
            }
            const float inv = L > 0.f ? 1.f / L : 0.f;
            if (t.S <= 32 * WB) { // the pairs are still in registers
#pragma unroll
                for (int i = 0; i < WB; ++i) {
                    const int s = 32 * i + lane;
                    if (s < t.S)
                        wts[t.off + s] = x[i].y > 0.f ? ex2((x[i].x - M) * kLog2e) * inv : 0.f;
                }
            } else {
                for (int s = lane; s < t.S; s += 32) {
                    const float2 y = __ldcg(ml + (size_t)s * rows);
                    wts[t.off + s] = y.y > 0.f ? ex2((y.x - M) * kLog2e) * inv : 0.f;
                }
            }
        }
        if (threadIdx.x == 0) {
            const bool ok = mbar_wait_bounded(sbar, phase, p.timeout_ns, &never);
            if (!ok) {
                atomicCAS(p.status, 0, kStatusTimeoutMla);
                // copies still in flight land before the CTA's memory is released
                (void)mbar_wait_bounded(sbar, phase, p.timeout_ns, &never);
            }
            hdr[3] = ok ? 1 : 0;
        }
        __syncthreads(); // also publishes the weights
        if (!hdr[3]) break;
        (void)mbar_wait_bounded(sbar, phase, p.timeout_ns, &never); // complete: this thread's view
        phase ^= 1u;
        {
            // warp w sums unit w % nu over the splits w / nu, w / nu + G, ...
            const int k = warp % nu, g = warp / nu, G = (kNW - 1 - k) / nu + 1;
            const PassUnit t = tab[k];
            float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 4
            for (int s = g; s < t.S; s += G) {
                const float w = wts[t.off + s];
                const float4 v = reinterpret_cast<const float4 *>(sm + (size_t)(t.off + s) * kBlk)[lane];
                if (w > 0.f) fma4(a, w, v);
            }
            red[warp * 32 + lane] = a;
        }
        __syncthreads();
        if (warp < nu) {
            const PassUnit t = tab[warp];
            float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
            for (int w = warp; w < kNW; w += nu) {
                const float4 v = red[w * 32 + lane];
                o.x += v.x;
                o.y += v.y;
                o.z += v.z;
                o.w += v.w;
            }
            unsigned char *dst = static_cast<unsigned char *>(out_row_ptr(p.fused, t.b, rows, t.row, kDv));
            const int col = t.z * 128 + lane * 4;
            switch (p.fused.out_dtype) {
            case DA_F32: store4<float>(reinterpret_cast<float *>(dst) + col, o); break;
            case DA_F16: store4<__half>(reinterpret_cast<__half *>(dst) + col, o); break;
            default: store4<__nv_bfloat16>(reinterpret_cast<__nv_bfloat16 *>(dst) + col, o); break;
            }
        }
        if (next >= units) break;
        // the stage, the table and the sums are rewritten by the next pass
        fence_proxy_async_smem();
        __syncthreads();
        u = next;
    }
}

template <int N, typename CT>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    mla_split_kernel(const __grid_constant__ MlaParams p)
{
    using LY = Layout<N>;
    using OP = Operand<CT>;
    constexpr bool kWide = sizeof(CT) == 4; // an f32 cache: 32 bytes per lane and chunk
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *bar = reinterpret_cast<uint64_t *>(sm + LY::BAR);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + LY::MISC);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(sm + LY::MISC + 4);
    float *alpha_sm = reinterpret_cast<float *>(sm + LY::ALPHA);
    const uint32_t sm_base = smem_u32(sm);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank(), peer = rank ^ 1u;
    const int cluster = blockIdx.x >> 1, nclusters = gridDim.x >> 1;
    const ItemTable &it = p.items;
    const int hbase = (int)rank * N;
    const uint32_t abort_peer = map_to_rank(smem_u32((const void *)abort_flag), peer);
    volatile int never = 0;

    if (threadIdx.x == 0) {
        for (int s = 0; s < 2; ++s) {
            for (int g = 0; g < kGroups; ++g) {
                mbar_init(bar + B_FULL + kGroups * s + g, 1);
                mbar_init(bar + B_CONV + kGroups * s + g, kConvWarps);
            }
            mbar_init(bar + B_EMPTY + s, 2);
            mbar_init(bar + B_SFULL + s, 2); // both CTAs' QK products (see kPChunk)
            mbar_init(bar + B_SFREE + s, kSoftWarps);
            mbar_init(bar + B_PFULL + s, kSoftWarps);
            mbar_init(bar + B_PFREE + s, 1);
        }
        mbar_init(bar + B_PVDONE, 1);
        mbar_init(bar + B_OREADY, 1);
        mbar_init(bar + B_OFREE, kSoftWarps);
        mbar_init(bar + B_QFULL, kConvWarps);
        mbar_init(bar + B_QFREE, 1);
        mbar_init(bar + B_DRAIN, 1);
        *abort_flag = 0;
        if (blockIdx.x == 0) *p.status = 0;
        fence_mbar_init();
    }
    if (warp == kMmaWarp) tmem_alloc(tmem_slot, LY::TMEM_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    cluster_sync_all(); // both CTAs' barriers exist before any remote arrival
    const uint32_t tmem = *tmem_slot;

    if (warp >= kSoftWarps && warp < kMmaWarp) {
        // =============================== converters ===============================
        const int cw = warp - kSoftWarps;
        const uint32_t row0 = rank * 32 + cw * kRowsPerConv; // this warp's rows of every tile
        const int trow = lane >> 3, q8 = lane & 7;            // this lane's row and 8 columns
        // f32 cache: lane q8 takes floats [4*q8, 4*q8 + 4) and [32 + 4*q8, 36 + 4*q8)
        // of each 64-column chunk, so each load instruction reads whole 128-byte
        // halves of 4 rows; 16-bit cache: elements [8*q8, 8*q8 + 8), whole 128-byte
        // rows, stored as they are
        const uint32_t off_lo = sw128(row0 + trow, q8 * (kWide ? 8 : 16));
        const uint32_t off_hi = sw128(row0 + trow, 64 + q8 * 8);
        uint32_t eph = 0, qph = 0;
        bool ok = true;
        // A whole tile of this lane's row (9 chunks) is in flight in registers:
        // the loads of tile t+1 go out as the stores of tile t free the registers,
        // and the unrolled body has no branch. Rows past the item's end are
        // loaded from its last row and stored as zeros (the cache may hold
        // anything there; the zero rows keep the PV product finite).
        constexpr int kLd = kWide ? 2 : 1;      // 16-byte loads per lane and chunk
        constexpr int kChunkV4 = 64 * (int)sizeof(CT) / 16; // 16-byte units per chunk of a row
        float4 ld[kChunks][kLd];
        const CT *cache = static_cast<const CT *>(p.cache);
        auto row_src = [&](const Cursor &u) {
            const int pos = min(u.x.p0 + u.t * kTile + (int)row0 + trow, u.x.p1 - 1);
            if (p.block_table) { // paged: the row's block from the table
                const int idx = pos / p.block_size;
                const int blk = __ldg(p.block_table + (size_t)u.x.b * p.max_blocks + idx);
                return reinterpret_cast<const float4 *>(
                    cache + (size_t)blk * p.block_stride +
                    (size_t)(pos - idx * p.block_size) * p.pos_stride) + q8;
            }
            return reinterpret_cast<const float4 *>(cache + (size_t)u.x.b * p.batch_stride +
                                                    (size_t)pos * p.pos_stride) + q8;
        };
        Cursor cur;
        cur.start(p, cluster, nclusters);
        if (!cur.done) {
            const float4 *src = row_src(cur);
#pragma unroll
            for (int c = 0; c < kChunks; ++c)
#pragma unroll
                for (int i = 0; i < kLd; ++i) ld[c][i] = ldg_stream_v4(src + kChunkV4 * c + 8 * i);
        }
        while (!cur.done) {
            Cursor nxt = cur;
            nxt.next_tile(p, nclusters);
            const int slot = cur.gt & 1;
            if (cur.t == 0) {
                // a new item: this CTA's heads of q (scale and log2 e folded in),
                // once the previous item's QK products are done with Q
                if (!mbar_wait_bounded(bar + B_QFREE, qph ^ 1u, p.timeout_ns, abort_flag)) {
                    ok = false;
                    break;
                }
                qph ^= 1u;
                const float *qb = p.q + ((size_t)cur.x.b * p.n_heads + hbase) * kDk;
                for (int task = cw * 32 + lane; task < N * 72; task += kConvWarps * 32) {
                    const int h = task / 72, g = task % 72, c = g >> 3, j = g & 7;
                    const float4 a = __ldg(reinterpret_cast<const float4 *>(qb + h * kDk + g * 8));
                    const float4 b = __ldg(reinterpret_cast<const float4 *>(qb + h * kDk + g * 8 + 4));
                    const float sc = p.scale_log2;
                    sts_v4(sm_base + LY::Q + c * LY::QCH + sw128(h, j * 16),
                           OP::pack(a.x * sc, a.y * sc), OP::pack(a.z * sc, a.w * sc),
                           OP::pack(b.x * sc, b.y * sc), OP::pack(b.z * sc, b.w * sc));
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar + B_QFULL);
            }
            // the slot is free once both CTAs' MMAs are done with its last tile
            if (!mbar_wait_bounded(bar + B_EMPTY + slot, ((eph >> slot) & 1u) ^ 1u, p.timeout_ns,
                                   abort_flag)) {
                ok = false;
                break;
            }
            eph ^= 1u << slot;
            const bool valid = cur.x.p0 + cur.t * kTile + (int)row0 + trow < cur.x.p1;
            // after the last tile the loads re-read this tile's row (never used)
            const float4 *nsrc = nxt.done ? row_src(cur) : row_src(nxt);
            const uint32_t tile = sm_base + LY::TILE + slot * kSlotBytes;
            // (under DA_FLAG_TEST_NO_TMA the publisher ships nothing; the
            // converters run unchanged)
#pragma unroll
            for (int c = 0; c < kChunks; ++c) {
                if constexpr (kWide) {
                    const uint32_t a0 = OP::pack(ld[c][0].x, ld[c][0].y);
                    const uint32_t a1 = OP::pack(ld[c][0].z, ld[c][0].w);
                    const uint32_t b0 = OP::pack(ld[c][1].x, ld[c][1].y);
                    const uint32_t b1 = OP::pack(ld[c][1].z, ld[c][1].w);
                    sts_v2(tile + c * kChunkBytes + off_lo, valid ? a0 : 0u, valid ? a1 : 0u);
                    sts_v2(tile + c * kChunkBytes + off_hi, valid ? b0 : 0u, valid ? b1 : 0u);
                } else {
                    const float4 v = ld[c][0];
                    sts_v4(tile + c * kChunkBytes + off_lo, valid ? __float_as_uint(v.x) : 0u,
                           valid ? __float_as_uint(v.y) : 0u, valid ? __float_as_uint(v.z) : 0u,
                           valid ? __float_as_uint(v.w) : 0u);
                }
#pragma unroll
                for (int i = 0; i < kLd; ++i) ld[c][i] = ldg_stream_v4(nsrc + kChunkV4 * c + 8 * i);
                if (c % kGroupChunks == kGroupChunks - 1) {
                    __syncwarp();
                    if (lane == 0) mbar_arrive(bar + B_CONV + kGroups * slot + c / kGroupChunks);
                }
            }
            cur = nxt;
        }
        if (!ok) raise_abort(abort_flag, abort_peer, p.status);
        // every commit (local and the peer's) aimed at this CTA's empty barriers
        // has landed once each slot has been released once more
        const uint64_t lim = *abort_flag ? 1000000ull : p.timeout_ns;
        for (int s = 0; s < 2; ++s)
            (void)mbar_wait_bounded(bar + B_EMPTY + s, ((eph >> s) & 1u) ^ 1u, lim, &never);
    } else if (warp == kMmaWarp) {
        // ============================ MMA issue (1 thread) ============================
        if (lane == 0) {
            constexpr uint32_t IDESC_QK = idesc_f16kind(64, kTile, 0, 0, !OP::kF16);
            constexpr uint32_t IDESC_PV = idesc_f16kind(128, N, 1, 0, !OP::kF16);
            uint32_t fph = 0, sph = 0, pph = 0, oph = 0, qph = 0;
            bool ok = true, q_ready = false;
            int qg = 0; // next chunk group of the current QK tile
            // Two cursors over this cluster's tiles: the next QK product and the
            // next PV product (never ahead of the QK cursor). Each turn issues
            // whichever is ready, so PV(t) goes out as soon as P(t) is written
            // and QK(t+1) as soon as the tile is in, in either order.
            Cursor qk, pv;
            qk.start(p, cluster, nclusters);
            pv.start(p, cluster, nclusters);
            int items_pv = 0;
            uint64_t last = global_ns();
            while (!pv.done) {
                bool progress = false;
                if (pv.gt < qk.gt) {
                    // O^T += V^T . P^T once P is written (and, at an item's first
                    // tile, once the previous item's epilogue has read O^T)
                    const int slot = pv.gt & 1;
                    const bool first = pv.t == 0;
                    if (mbar_test(bar + B_PFULL + slot, (pph >> slot) & 1u) &&
                        (!first || items_pv == 0 || mbar_test(bar + B_OFREE, oph))) {
                        pph ^= 1u << slot;
                        if (first && items_pv > 0) oph ^= 1u;
                        if (first) ++items_pv;
                        tc_fence_after();
                        const uint64_t vd = smem_desc_sw128(sm_base + LY::TILE + slot * kSlotBytes,
                                                            kChunkBytes, 1024);
                        const uint64_t pd = smem_desc_sw128(
                            sm_base + LY::TILE + slot * kSlotBytes + kPChunk * kChunkBytes, 16, 1024);
#pragma unroll
                        for (int j = 0; j < 4; ++j)
#pragma unroll
                            for (int k = 0; k < 4; ++k)
                                tc_mma_bf16(tmem + LY::O_COL + j * N,
                                            vd + (uint64_t)((2 * j * kChunkBytes + k * 2048) >> 4),
                                            pd + (uint64_t)((k * 32) >> 4), IDESC_PV,
                                            (first && k == 0) ? 0u : 1u);
                        tc_commit_mc(bar + B_EMPTY + slot, 3);
                        tc_commit(bar + B_PFREE + slot);
                        tc_commit(bar + B_PVDONE);
                        if (pv.t == pv.x.ntiles - 1) tc_commit(bar + B_OREADY);
                        progress = true;
                        pv.next_tile(p, nclusters);
                    }
                }
                if (!qk.done) {
                    // S = Q . K_tile^T once Q of the item is in, the tile is full
                    // and the softmax has released this S slot
                    const int slot = qk.gt & 1;
                    if (!q_ready && mbar_test(bar + B_QFULL, qph)) {
                        qph ^= 1u;
                        q_ready = true;
                    }
                    const int fb = kGroups * slot + qg;
                    if (q_ready && mbar_test(bar + B_FULL + fb, (fph >> fb) & 1u) &&
                        (qg > 0 || mbar_test(bar + B_SFREE + slot, ((sph >> slot) & 1u) ^ 1u))) {
                        fph ^= 1u << fb;
                        if (qg == 0) sph ^= 1u << slot;
                        tc_fence_after();
                        // descriptors advance by adding (byte offset >> 4) to the start field
                        const int c0 = qg * kGroupChunks;
                        const uint64_t qd =
                            smem_desc_sw128(sm_base + LY::Q + c0 * LY::QCH, 16, 1024);
                        const uint64_t kd = smem_desc_sw128(
                            sm_base + LY::TILE + slot * kSlotBytes + c0 * kChunkBytes, 16, 1024);
#pragma unroll
                        for (int c = 0; c < kGroupChunks; ++c)
#pragma unroll
                            for (int k = 0; k < 4; ++k)
                                tc_mma_bf16(tmem + slot * kTile,
                                            qd + (uint64_t)((c * LY::QCH + k * 32) >> 4),
                                            kd + (uint64_t)((c * kChunkBytes + k * 32) >> 4),
                                            IDESC_QK, (qg | c | k) != 0 ? 1u : 0u);
                        progress = true;
                        if (++qg == kGroups) {
                            qg = 0;
                            // to both CTAs: P overwrites the tile's last chunk only
                            // once the peer has its copy of this CTA's rows too (the
                            // peer's QK waited for them), so the outgoing bulk copy
                            // has read them
                            tc_commit_mc(bar + B_SFULL + slot, 3);
                            if (qk.t == qk.x.ntiles - 1) {
                                tc_commit(bar + B_QFREE);
                                q_ready = false;
                            }
                            qk.next_tile(p, nclusters);
                        }
                    }
                }
                // no sleep between polls: the thread issues as soon as a product is
                // ready (a 32 ns sleep here cost 2 us per launch)
                if (progress) {
                    last = global_ns();
                } else if (*abort_flag || global_ns() - last > p.timeout_ns) {
                    ok = false;
                    break;
                }
            }
            if (!ok) raise_abort(abort_flag, abort_peer, p.status);
            // no MMA may be in flight when TMEM is freed
            tc_commit(bar + B_DRAIN);
            (void)mbar_wait_bounded(bar + B_DRAIN, 0, p.timeout_ns, &never);
        }
        __syncwarp();
    } else if (warp == kPubWarp) {
        // ======================= publisher (1 thread per CTA) =======================
        if (lane == 0 && !(p.flags & DA_FLAG_TEST_NO_TMA)) {
            uint32_t cph = 0;
            bool ok = true;
            int gt = 0;
            for (int item = cluster; ok && item < it.n_items; item += nclusters) {
                const Item x = get_item(p, item);
                for (int t = 0; t < x.ntiles; ++t, ++gt) {
                    const int slot = gt & 1;
                    for (int g = 0; g < kGroups && ok; ++g) {
                        const int fb = kGroups * slot + g;
                        if (!mbar_wait_bounded(bar + B_CONV + fb, (cph >> fb) & 1u, p.timeout_ns,
                                               abort_flag)) {
                            ok = false;
                            break;
                        }
                        cph ^= 1u << fb;
                        // the converters' stores, acquired through B_CONV, become visible
                        // to the async proxy (the bulk copies here, the MMAs after B_FULL)
                        fence_proxy_async_smem();
                        const uint32_t half = LY::TILE + slot * kSlotBytes + rank * 32 * 128;
                        const uint32_t peer_full = map_to_rank(smem_u32(bar + B_FULL + fb), peer);
#pragma unroll
                        for (int c = g * kGroupChunks; c < (g + 1) * kGroupChunks; ++c) {
                            const uint32_t src = sm_base + half + c * kChunkBytes;
                            bulk_copy_to_cta(map_to_rank(src, peer), src, 32 * 128, peer_full);
                        }
                        mbar_arrive_expect_tx(bar + B_FULL + fb, kPeerTx);
                    }
                    if (!ok) break;
                }
            }
            if (!ok) raise_abort(abort_flag, abort_peer, p.status);
        }
        __syncwarp();
    } else {
        // ========================= softmax and epilogue (warps 0-3) ========================
        const int tid = threadIdx.x;            // TMEM lane of the epilogue rows
        const int h = 16 * warp + lane;         // head of this lane in the 64-row S layout
        const bool owner = lane < 16 && h < N;
        const uint32_t tl = tmem + ((uint32_t)(warp * 32) << 16);
        uint32_t sph = 0, ppf = 0, oph = 0;
        int gt = 0;
        bool ab = false;
        for (int item = cluster; !ab && item < it.n_items; item += nclusters) {
            const Item x = get_item(p, item);
            if (x.ntiles == 0) { // an empty item: a neutral partial, no MMA took part
                if (x.skip) continue; // the exact kernel writes this item's partials
                const size_t row0 = ((size_t)it.split_base[x.b] + x.s) * p.n_heads + hbase;
                if (owner) p.ml[row0 + h] = make_float2(kNeutralM, 0.f);
                continue;
            }
            float m = -INFINITY, l = 0.f;
            // this row's token sees positions below lim (causal among the new
            // tokens; with one token, every position of the item)
            const int lim = (p.flags & DA_FLAG_NO_CAUSAL) ? (INT_MAX >> 1)
                                                          : x.L - p.q_len + 1 + (hbase + h) / p.hq;
            for (int t = 0; t < x.ntiles; ++t, ++gt) {
                const int slot = gt & 1;
                bool okw = mbar_wait_bounded(bar + B_SFULL + slot, (sph >> slot) & 1u,
                                             p.timeout_ns, abort_flag);
                if (bar_or(2, 128, !okw)) {
                    ab = true;
                    break;
                }
                sph ^= 1u << slot;
                tc_fence_after();
                const int nvalid = max(0, min(kTile, min(x.p1, lim) - (x.p0 + t * kTile)));
                const uint32_t scol = tl + slot * kTile;
                // this thread's head: its 64 scores (one TMEM round trip) and
                // their max over the valid positions
                float sc[kTile];
#pragma unroll
                for (int g = 0; g < 4; ++g) tmem_ld16(scol + 16 * g, sc + 16 * g);
                tmem_wait_ld();
                float tm = -INFINITY;
#pragma unroll
                for (int i = 0; i < kTile; ++i)
                    if (i < nvalid) tm = fmaxf(tm, sc[i]);
                const bool ex = owner && tm > m + kTau;
                if (bar_or(2, 128, ex)) {
                    // move the reference of the heads that outgrew it; rescale l and O^T
                    const float mn = ex ? tm : m;
                    const float alpha = (mn == m) ? 1.f : (m == -INFINITY ? 0.f : ex2(m - mn));
                    if (owner) alpha_sm[h] = alpha;
                    l *= alpha;
                    m = mn;
                    if (t > 0) {
                        // PV(t-1) is done with O^T before it is rescaled
                        okw = mbar_wait_bounded(bar + B_PVDONE, (uint32_t)(gt - 1) & 1u,
                                                p.timeout_ns, abort_flag);
                        named_bar_sync(2, 128);
                        if (bar_or(2, 128, !okw)) {
                            ab = true;
                            break;
                        }
                        tc_fence_after();
#pragma unroll
                        for (int j = 0; j < 4; ++j)
#pragma unroll
                            for (int g = 0; g < N / 16; ++g) {
                                float o[16];
                                tmem_ld16(tl + LY::O_COL + j * N + 16 * g, o);
                                tmem_wait_ld();
#pragma unroll
                                for (int i = 0; i < 16; ++i) o[i] *= alpha_sm[16 * g + i];
                                tmem_st16(tl + LY::O_COL + j * N + 16 * g, o);
                            }
                        tmem_wait_st();
                    }
                    named_bar_sync(2, 128); // alpha_sm is read before it is rewritten
                    // the scores are not held across this rare path: read them again
#pragma unroll
                    for (int g = 0; g < 4; ++g) tmem_ld16(scol + 16 * g, sc + 16 * g);
                    tmem_wait_ld();
                }
                // P row of this head: 2^(s - m) in bf16, once PV(t-2) is done with the slot
                okw = mbar_wait_bounded(bar + B_PFREE + slot, ((ppf >> slot) & 1u) ^ 1u,
                                        p.timeout_ns, abort_flag);
                if (bar_or(2, 128, !okw)) {
                    ab = true;
                    break;
                }
                ppf ^= 1u << slot;
                const uint32_t prow = sm_base + LY::TILE + slot * kSlotBytes + kPChunk * kChunkBytes;
                if (owner) {
#pragma unroll
                    for (int g = 0; g < 4; ++g) {
                        uint32_t w[8];
#pragma unroll
                        for (int i = 0; i < 16; i += 2) {
                            const float p0 = (16 * g + i < nvalid) ? ex2(sc[16 * g + i] - m) : 0.f;
                            const float p1 =
                                (16 * g + i + 1 < nvalid) ? ex2(sc[16 * g + i + 1] - m) : 0.f;
                            l += p0 + p1;
                            w[i >> 1] = OP::pack(p0, p1);
                        }
                        sts_v4(prow + sw128(h, 32 * g), w[0], w[1], w[2], w[3]);
                        sts_v4(prow + sw128(h, 32 * g + 16), w[4], w[5], w[6], w[7]);
                    }
                }
                tc_fence_before();
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(bar + B_SFREE + slot);
                    mbar_arrive(bar + B_PFULL + slot);
                }
            }
            if (ab) break;
            // ------------------------------- epilogue -------------------------------
            bool okw = mbar_wait_bounded(bar + B_OREADY, oph, p.timeout_ns, abort_flag);
            if (bar_or(2, 128, !okw)) break;
            oph ^= 1u;
            tc_fence_after();
            const size_t slot_id = (size_t)it.split_base[x.b] + x.s;
            const size_t row0 = slot_id * p.n_heads + hbase;
#pragma unroll
            for (int j = 0; j < 4; ++j)
#pragma unroll
                for (int g = 0; g < N / 16; ++g) {
                    float o[16];
                    tmem_ld16(tl + LY::O_COL + j * N + 16 * g, o);
                    tmem_wait_ld();
#pragma unroll
                    for (int i = 0; i < 16; ++i)
                        p.acc[(row0 + 16 * g + i) * kDv + 128 * j + tid] = o[i];
                }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar + B_OFREE);
            if (owner) p.ml[row0 + h] = make_float2(l > 0.f ? m * kLn2 : kNeutralM, l);
        }
    }

    // ---------------------------------- teardown ----------------------------------
    tc_fence_before();
    __syncthreads();
    if (*abort_flag) {
        // let copies already in flight from the peer land before the cluster exits
        const uint64_t t0 = global_ns();
        while (global_ns() - t0 < 200000ull) {
        }
    }
    cluster_sync_all();
    tc_fence_after();
    if (warp == kMmaWarp) tmem_dealloc(tmem, LY::TMEM_COLS);

    if (p.fused.on) {
        // The merge without a combine launch: once every CTA of the launch has
        // written its partials (a grid-wide arrival count; the library fuses
        // only when the GPU holds all the launch's clusters at once), every warp
        // of the grid merges a share of the units.
        volatile int *go = abort_flag + 1;
        uint32_t *arrived = p.fused.ctr;
        __threadfence(); // this thread's partial writes, before the arrival
        __syncthreads();
        if (threadIdx.x == 0) {
            (void)arrive(arrived);
            const uint64_t t0 = global_ns();
            bool ok = true;
            while (*reinterpret_cast<volatile uint32_t *>(arrived) < gridDim.x) {
                if (global_ns() - t0 > p.timeout_ns) {
                    ok = false;
                    atomicCAS(p.status, 0, kStatusTimeoutMla);
                    break;
                }
                __nanosleep(100);
            }
            __threadfence();
            *go = ok && *reinterpret_cast<volatile int *>(p.status) == 0;
        }
        __syncthreads();
        if (*go) mla_merge_staged(p, sm);
    }
    if (threadIdx.x == 0) griddep_launch_dependents();
}

} // namespace

bool mla_supported_heads(int n_heads)
{
    return n_heads == 32 || n_heads == 64 || n_heads == 96 || n_heads == 128;
}

int mla_smem_bytes(int n_heads)
{
    switch (n_heads) {
    case 32: return Layout<16>::ALLOC;
    case 64: return Layout<32>::ALLOC;
    case 96: return Layout<48>::ALLOC;
    case 128: return Layout<64>::ALLOC;
    default: return 0;
    }
}

template <int N, typename CT>
static cudaError_t launch_n(int grid, cudaStream_t st, const MlaParams &p)
{
    auto *fn = mla_split_kernel<N, CT>;
    cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         Layout<N>::ALLOC);
    if (e != cudaSuccess) return e;
    fn<<<grid, kThreads, Layout<N>::ALLOC, st>>>(p);
    return cudaGetLastError();
}

template <int N> static cudaError_t launch_dt(int kv_dtype, int grid, cudaStream_t st,
                                             const MlaParams &p)
{
    switch (kv_dtype) {
    case DA_F32: return launch_n<N, float>(grid, st, p);
    case DA_F16: return launch_n<N, __half>(grid, st, p);
    case DA_BF16: return launch_n<N, __nv_bfloat16>(grid, st, p);
    default: return cudaErrorInvalidValue;
    }
}

// How many of the kernel's 2-CTA clusters the current device holds at once
// (cached per device and row count; 0 if the query fails).
template <int N> static int max_clusters_n()
{
    constexpr int kDevs = 64;
    static std::atomic<int> cache[kDevs]; // 0: not asked yet; -1: the query failed
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kDevs) return 0;
    if (cache[dev] == 0) {
        auto *fn = mla_split_kernel<N, float>; // the same resources for every cache type
        int n = -1;
        if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 Layout<N>::ALLOC) == cudaSuccess) {
            cudaLaunchConfig_t cfg = {};
            cfg.gridDim = dim3(2);
            cfg.blockDim = dim3(kThreads);
            cfg.dynamicSmemBytes = Layout<N>::ALLOC;
            cudaLaunchAttribute at[1];
            at[0].id = cudaLaunchAttributeClusterDimension;
            at[0].val.clusterDim.x = 2;
            at[0].val.clusterDim.y = 1;
            at[0].val.clusterDim.z = 1;
            cfg.attrs = at;
            cfg.numAttrs = 1;
            if (cudaOccupancyMaxActiveClusters(&n, (void *)fn, &cfg) != cudaSuccess || n < 1) n = -1;
        }
        (void)cudaGetLastError();
        cache[dev].store(n);
    }
    const int n = cache[dev].load();
    return n > 0 ? n : 0;
}

int mla_max_clusters(int n_heads)
{
    switch (n_heads) {
    case 32: return max_clusters_n<16>();
    case 64: return max_clusters_n<32>();
    case 96: return max_clusters_n<48>();
    case 128: return max_clusters_n<64>();
    default: return 0;
    }
}

cudaError_t launch_mla_split(int grid, cudaStream_t st, const MlaParams &p, int kv_dtype)
{
    switch (p.n_heads) {
    case 32: return launch_dt<16>(kv_dtype, grid, st, p);
    case 64: return launch_dt<32>(kv_dtype, grid, st, p);
    case 96: return launch_dt<48>(kv_dtype, grid, st, p);
    case 128: return launch_dt<64>(kv_dtype, grid, st, p);
    default: return cudaErrorInvalidValue;
    }
}

} // namespace skv
