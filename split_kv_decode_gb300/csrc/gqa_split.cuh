// GQA / MQA split kernel ("Kernel A"), sm_103a.
//
// One persistent CTA per SM walks a static round-robin list of work items.
// An item is (sequence b, KV head, split s): a contiguous slice
// [s*chunk, min(L, (s+1)*chunk)) of that KV head's cache, read once for all
// G query heads of the group ("Attention at 128k: Split Over Context", §2:
// contiguous slices; aprender issue 3725 design note §2: one block per
// (KV head, split) serving all G heads).
//
// Warp roles:
//   warp NCW (producer, one lane) streams the slice's K and V tiles of T rows
//     into an NST-stage shared-memory ring with TMA tensor copies; each stage
//     has a "full" mbarrier (transaction bytes) and an "empty" mbarrier
//     (one arrival per consumer warp).
//   warps 0..NCW-1 (consumers) each own P = T/NCW rows of every tile. A warp
//     reads a row with 128-bit shared loads spread over its 32 lanes, forms
//     the G dot products against q (held in registers), and reduces the P*G
//     partial dots across lanes with a transpose-reduce (each shuffle step
//     halves the number of live values per lane). Every warp keeps its own
//     online-softmax state (running max m, per-lane partial sums of l, and
//     acc[G][D] in registers), following the recurrence of "The Kernel
//     Level", section "But Softmax Wants the Whole Row".
// At the end of an item the NCW warp states are merged with the same
// rescaling as the combine (m = max m_w, weights e^{m_w - m}) by a pairwise
// tree through shared memory, and one un-normalised partial (m, l, acc[D]) per
// query head is written.
//
// Scores are kept in base-2 units: q is pre-multiplied by scale*log2(e) so
// that e^{s - m} = 2^{s2 - m2}; the stored m is converted back to natural
// units. Positions past the slice (or past the sequence) are masked to -inf
// before the max and skipped in the PV update, so whatever the cache holds
// there (never-written memory, NaN) cannot leak in.
#pragma once
#include <climits>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "internal.h"
#include "merge.cuh"
#include "ptx.cuh"

namespace skv {

// ---- storage conversion: one chunk of EPC elements (16 or 8 bytes) -----------
template <typename DT, int EPC> struct Chunk;

template <> struct Chunk<float, 4> {
    static __device__ __forceinline__ void load(const float *p, float *f)
    {
        float4 x = *reinterpret_cast<const float4 *>(p);
        f[0] = x.x; f[1] = x.y; f[2] = x.z; f[3] = x.w;
    }
};

__device__ __forceinline__ void h2_to_f(uint32_t w, float &a, float &b)
{
    __half2 h = *reinterpret_cast<__half2 *>(&w);
    float2 f = __half22float2(h);
    a = f.x;
    b = f.y;
}

__device__ __forceinline__ void bf2_to_f(uint32_t w, float &a, float &b)
{
    a = __uint_as_float(w << 16);
    b = __uint_as_float(w & 0xffff0000u);
}

template <> struct Chunk<__half, 8> {
    static __device__ __forceinline__ void load(const __half *p, float *f)
    {
        uint4 x = *reinterpret_cast<const uint4 *>(p);
        h2_to_f(x.x, f[0], f[1]); h2_to_f(x.y, f[2], f[3]);
        h2_to_f(x.z, f[4], f[5]); h2_to_f(x.w, f[6], f[7]);
    }
};
template <> struct Chunk<__half, 4> {
    static __device__ __forceinline__ void load(const __half *p, float *f)
    {
        uint2 x = *reinterpret_cast<const uint2 *>(p);
        h2_to_f(x.x, f[0], f[1]); h2_to_f(x.y, f[2], f[3]);
    }
};
template <> struct Chunk<__nv_bfloat16, 8> {
    static __device__ __forceinline__ void load(const __nv_bfloat16 *p, float *f)
    {
        uint4 x = *reinterpret_cast<const uint4 *>(p);
        bf2_to_f(x.x, f[0], f[1]); bf2_to_f(x.y, f[2], f[3]);
        bf2_to_f(x.z, f[4], f[5]); bf2_to_f(x.w, f[6], f[7]);
    }
};
template <> struct Chunk<__nv_bfloat16, 4> {
    static __device__ __forceinline__ void load(const __nv_bfloat16 *p, float *f)
    {
        uint2 x = *reinterpret_cast<const uint2 *>(p);
        bf2_to_f(x.x, f[0], f[1]); bf2_to_f(x.y, f[2], f[3]);
    }
};

// ---- transpose-reduce of N per-lane values over the 32 lanes of a warp ------
// While N is even, each step keeps one half of the values and sends the other
// half to the partner lane (lane ^ MASK), halving N; once N is odd the
// remaining steps are plain butterflies. Afterwards a lane holds
// tr_out<N,16>() totals whose original indices are tr_base(lane) + r.
template <int N, int MASK> __host__ __device__ constexpr int tr_out()
{
    if constexpr (MASK == 0) return N;
    else if constexpr (N % 2 == 0 && N > 1) return tr_out<N / 2, MASK / 2>();
    else return tr_out<N, MASK / 2>();
}

template <int N, int MASK> __device__ __forceinline__ int tr_base(int lane)
{
    if constexpr (MASK == 0) return 0;
    else if constexpr (N % 2 == 0 && N > 1)
        return ((lane & MASK) ? N / 2 : 0) + tr_base<N / 2, MASK / 2>(lane);
    else return tr_base<N, MASK / 2>(lane);
}

// true for exactly one lane among those holding the same totals
template <int N, int MASK> __device__ __forceinline__ bool tr_writer(int lane)
{
    if constexpr (MASK == 0) return true;
    else if constexpr (N % 2 == 0 && N > 1) return tr_writer<N / 2, MASK / 2>(lane);
    else return ((lane & MASK) == 0) && tr_writer<N, MASK / 2>(lane);
}

template <int N, int MASK> __device__ __forceinline__ void tr_reduce(float *v, int lane)
{
    if constexpr (MASK > 0) {
        if constexpr (N % 2 == 0 && N > 1) {
            const bool up = (lane & MASK) != 0;
#pragma unroll
            for (int i = 0; i < N / 2; ++i) {
                float send = up ? v[i] : v[i + N / 2];
                float keep = up ? v[i + N / 2] : v[i];
                v[i] = keep + __shfl_xor_sync(0xffffffffu, send, MASK);
            }
            tr_reduce<N / 2, MASK / 2>(v, lane);
        } else {
#pragma unroll
            for (int i = 0; i < N; ++i) v[i] += __shfl_xor_sync(0xffffffffu, v[i], MASK);
            tr_reduce<N, MASK / 2>(v, lane);
        }
    }
}

__device__ __forceinline__ bool named_bar_or(int id, int threads, bool pred)
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

// item -> (b, kv head, split[, row group]); the row groups of a (b, kv head,
// split) are consecutive items, so the CTAs that read the same slice run at
// the same time (the later reads are L2 hits)
__device__ __forceinline__ void decode_item(const ItemTable &it, int item, int &b, int &kvh,
                                            int &s, int &rg)
{
    const int rgs = it.row_groups > 1 ? it.row_groups : 1;
    const int u = item / rgs;
    rg = item - u * rgs;
    const int t = u / it.n_kv_heads;
    kvh = u - t * it.n_kv_heads;
    int lo = 0, hi = it.batch - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (it.split_base[mid] <= t) lo = mid;
        else hi = mid - 1;
    }
    b = lo;
    s = t - it.split_base[lo];
}

__device__ __forceinline__ void decode_item(const ItemTable &it, int item, int &b, int &kvh,
                                            int &s)
{
    int rg;
    decode_item(it, item, b, kvh, s, rg);
}

// the length an item of sequence b attends over: the plan's, or the current
// length read on the device, kept within [q_len, the plan's]
__device__ __forceinline__ int item_len(const SplitParams &p, int b)
{
    const int L = p.items.seq_lens[b];
    return p.dev_lens ? max(p.q_len, min(__ldg(p.dev_lens + b), L)) : L;
}

// A tile is T rows, cut only at the item's end: in a paged cache tiles run
// across block ends like in a contiguous one (the producers copy such tiles
// piecewise, each piece from its own block).
template <int T> __device__ __forceinline__ int tile_end(int t0, int p1) { return min(t0 + T, p1); }

template <int X> __host__ __device__ constexpr int align_up(int v) { return (v + X - 1) / X * X; }

// LPR (lanes per row) is 32, or 16 when a row is only 256 bytes (D = 128 in a
// 16-bit type): then the two half-warps read two rows at once, each lane with
// one 16-byte load per row, and the dot products reduce over 16 lanes.
template <typename DT, int D, int G, int T, int NCW, int NST, int LPR> struct GqaKernel {
    static constexpr int ES = sizeof(DT);
    static constexpr int RPW = 32 / LPR;                     // rows a warp reads at once
    static constexpr int EPL = D / LPR;                      // elements per lane per row
    static constexpr int CB = (EPL * ES < 16) ? EPL * ES : 16; // bytes per chunk load
    static constexpr int EPC = CB / ES;                      // elements per chunk
    static constexpr int NCH = EPL / EPC;                    // chunks per lane per row
    static constexpr int P = T / NCW;                        // rows per warp per tile
    static constexpr int PH = P / RPW;                       // row steps per tile
    static constexpr int NV = P * G;                         // dots per warp per tile
    static constexpr int NVL = PH * G;                       // dots per lane group per tile
    static constexpr int R = tr_out<NVL, LPR / 2>();
    static constexpr int R2 = (NV + 31) / 32;
    static constexpr int TILE_BYTES = T * D * ES;
    static constexpr int STAGE_BYTES = 2 * TILE_BYTES;
    static constexpr int THREADS = (NCW + 1) * 32;
    static constexpr int CONSUMERS = NCW * 32;
    // shared memory layout (offsets from a 1024-byte aligned base)
    static constexpr int OFF_BAR = NST * STAGE_BYTES;
    static constexpr int OFF_ABORT = OFF_BAR + 2 * NST * 8;
    static constexpr int WARP_SCR = align_up<4>(2 * NV + 2 * G); // floats: sc, pscr, mw, aw
    static constexpr int OFF_WARP = align_up<16>(OFF_ABORT + 16);
    static constexpr int OFF_ML = align_up<16>(OFF_WARP + NCW * WARP_SCR * 4);
    // merge tree: at distance d the warps w = d (mod 2d) pass their sums to
    // w - d through slot w / (2d); even and odd levels use separate slot sets
    static constexpr int tree_slots(int d) { return NCW > d ? (NCW - d + 2 * d - 1) / (2 * d) : 0; }
    static constexpr int cmax(int a, int b) { return a > b ? a : b; }
    static constexpr int TREE_EVEN = cmax(tree_slots(1), cmax(tree_slots(4), tree_slots(16)));
    static constexpr int TREE_ODD = cmax(tree_slots(2), tree_slots(8));
    static constexpr int OFF_TREE = align_up<16>(OFF_ML + NCW * G * 8);
    static constexpr int SMEM_USED = OFF_TREE + (TREE_EVEN + TREE_ODD) * G * D * 4;
    static constexpr int SMEM_ALLOC = SMEM_USED + 1024;      // slack for the 1024 alignment
    static_assert(D % LPR == 0 && NCH * EPC == EPL && (LPR == 32 || LPR == 16), "row split");
    static_assert(P % RPW == 0, "rows per warp split into lane groups");
    static_assert(T % NCW == 0 && NV % 4 == 0, "tile split");
    static_assert(T <= 256 && D <= 256, "TMA box limits");
    static_assert(SMEM_ALLOC <= 232448, "shared memory budget");
    static_assert(WARP_SCR % 4 == 0 && NV % 4 == 0, "16-byte aligned per-warp scratch");
    static_assert(TILE_BYTES % 128 == 0, "TMA destination alignment");
    static_assert(NCW * G * D * 4 <= NST * STAGE_BYTES, "flat merge slots in the stage ring");
};

// The SIMT kernel's merge without a combine launch (DA_FLAG_ONE_LAUNCH), run
// once all of a CTA's items are written: each of its items merges a share of
// its (sequence, KV head) group. The group's (row, 16 value columns) units are
// cut into as many shares as the group has items, and item k of the group
// (split s, row group rg: k = s * row groups + rg) takes share k, one warp per
// unit, after waiting (bounded) for the group's last arrival. The library fuses only when
// every CTA of the launch is resident at once, so no wait depends on a CTA
// that has not started; a CTA waits only after all its own arrivals, so none
// depends on another's wait. Kept out of line: the kernel's main loop keeps
// its own register allocation.
template <int D, int NCW>
__device__ __noinline__ void fused_merge_shares(const SplitParams &p, volatile int *abort_flag)
{
    const ItemTable &it = p.items;
    const int warp = threadIdx.x >> 5;
    const int Gh = p.hq / it.n_kv_heads;
    const int rows_grp = Gh * p.q_len;
    auto row_off = [&](int jf) { return p.q_len == 1 ? jf : (jf / Gh) * p.hq + jf % Gh; };
    volatile int *go = abort_flag + 1; // the header's spare word
    const int rgs = it.row_groups > 1 ? it.row_groups : 1;
    for (int item = blockIdx.x; item < it.n_items; item += gridDim.x) {
        int b, kvh, s, rg;
        decode_item(it, item, b, kvh, s, rg);
        const int S = it.split_base[b + 1] - it.split_base[b];
        const uint32_t n = (uint32_t)(S * rgs);
        if (threadIdx.x == 0) {
            const volatile uint32_t *ctr = p.fused.ctr + (size_t)b * it.n_kv_heads + kvh;
            const uint64_t t0 = global_ns();
            bool ok = true;
            while (*ctr < n) {
                if (*abort_flag || global_ns() - t0 > p.timeout_ns) {
                    ok = false;
                    *abort_flag = 1;
                    atomicCAS(p.status, 0, kStatusTimeoutGqa);
                    break;
                }
                __nanosleep(64);
            }
            *go = ok ? 1 : 0;
        }
        named_bar_sync(1, NCW * 32);
        if (!*go) break;
        __threadfence(); // the group's partials, before they are read
        constexpr int C = 4, CU = D / (4 * C); // float4s per unit, units per row
        const int U = rows_grp * CU, k = s * rgs + rg;
        const int u0 = (int)((int64_t)k * U / (int64_t)n);
        const int u1 = (int)((int64_t)(k + 1) * U / (int64_t)n);
        for (int u = u0 + warp; u < u1; u += NCW) {
            const int row = kvh * Gh + row_off(u / CU);
            warp_merge_cols<C, 8>(p.ml, p.acc, (size_t)it.split_base[b], S, p.n_heads, row, D,
                                  (u % CU) * C, out_row_ptr(p.fused, b, p.n_heads, row, D),
                                  p.fused.out_dtype);
        }
        named_bar_sync(1, NCW * 32); // *go is read before it is rewritten
    }
}

template <typename DT, int D, int G, int T, int NCW, int NST, int LPR>
__global__ void __launch_bounds__((NCW + 1) * 32, 1)
    gqa_split_kernel(const __grid_constant__ GqaMaps maps, const __grid_constant__ SplitParams p)
{
    using K = GqaKernel<DT, D, G, T, NCW, NST, LPR>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + K::OFF_BAR);
    uint64_t *empty = full + NST;
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + K::OFF_ABORT);
    float2 *sm_ml = reinterpret_cast<float2 *>(smem + K::OFF_ML);
    float *sm_tree = reinterpret_cast<float *>(smem + K::OFF_TREE);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const ItemTable &it = p.items;

    // The producer sets the stage barriers up and goes straight on to its first
    // copies; the consumers wait for the set-up on named barrier 2 (after loading
    // their first q), so the copies start without a CTA-wide barrier in front.
    if (warp == NCW && lane == 0) {
        for (int s = 0; s < NST; ++s) {
            mbar_init(full + s, 1);
            mbar_init(empty + s, NCW);
        }
        *abort_flag = 0;
        if (blockIdx.x == 0) *p.status = 0;
        fence_mbar_init();
    }

    if (warp == NCW) {
        __syncwarp();
        named_bar_arrive(2, K::CONSUMERS + 32);
        // ------------------------------- producer -------------------------------
        // Lane 0 waits on the stage barriers and issues the copies. For paged
        // caches the whole warp walks the items and tiles: the lanes hold a
        // window of 32 consecutive block-table entries of the current sequence
        // (one coalesced load). A tile whose rows lie in one block is one TMA box
        // of T rows; a tile that spans a block end is T / box_rows short boxes. So
        // tiles run across blocks as in a contiguous cache and every stage
        // carries a full tile. For contiguous caches lane 0 walks alone.
        const bool paged = p.block_table != nullptr;
        if (!paged && lane != 0) return;
        const unsigned mask = paged ? 0xffffffffu : 1u;
        if (lane == 0) {
            tma_prefetch_map(&maps.k);
            tma_prefetch_map(&maps.v);
            if (paged) {
                tma_prefetch_map(&maps.kb);
                tma_prefetch_map(&maps.vb);
            }
        }
        const uint64_t pol = l2_evict_first_policy();
        int last_parity[NST];
#pragma unroll
        for (int s = 0; s < NST; ++s) last_parity[s] = -1;
        int stage = 0;
        uint32_t phase = 0;
        bool ok = true;
        int win_b = -1, win_lo = 0;
        int32_t win_entry = 0;
        // paged: tile and block lengths in units of the box height
        const int hrows = paged ? p.box_rows : 1;
        const int tile_u = T / hrows, block_u = paged ? p.block_size / hrows : 1;
        for (int item = blockIdx.x; ok && item < it.n_items; item += gridDim.x) {
            int b, kvh, s;
            decode_item(it, item, b, kvh, s);
            const int Lb = item_len(p, b);
            const int p0 = s * it.chunk[b];
            const int p1 = min(Lb, p0 + it.chunk[b]);
            // paged: block index and slot of the tile start (slot in units of
            // h = box_rows), advanced without divisions: the producer's time per
            // tile is on the copy path
            const int bs = p.block_size;
            int bi = paged ? p0 / bs : 0, su = paged ? (p0 - bi * bs) / hrows : 0;
            for (int t0 = p0, t1; t0 < p1; t0 = t1) {
                t1 = tile_end<T>(t0, p1);
                bool got = true;
                if (lane == 0)
                    got = mbar_wait_bounded(empty + stage, phase ^ 1u, p.timeout_ns, abort_flag);
                if (!__shfl_sync(mask, got, 0)) {
                    ok = false;
                    break;
                }
                if (!(p.flags & DA_FLAG_TEST_NO_TMA)) {
                    uint8_t *dst = smem + stage * K::STAGE_BYTES;
                    if (paged) {
                        // the window covers the kSpan blocks from bi, as many as a
                        // tile can touch (blocks hold 16 or more positions)
                        constexpr int kSpan = (T + 14) / 16 + 1;
                        static_assert(kSpan <= 32, "window of 32 table entries");
                        if (b != win_b || bi < win_lo || bi + kSpan > win_lo + 32) {
                            win_b = b;
                            win_lo = bi;
                            win_entry = (bi + lane < p.max_blocks)
                                            ? p.block_table[(size_t)b * p.max_blocks + bi + lane]
                                            : p.oob_block;
                        }
                        const int so = su * hrows;
                        if (so + (t1 - t0) <= bs) {
                            // the tile's rows lie in one block: one box of T rows at
                            // (slot in block, block); rows of the box past the block
                            // lie past the item's end and read as zeros
                            const int blk = __shfl_sync(0xffffffffu, win_entry, bi - win_lo);
                            if (lane == 0) {
                                mbar_arrive_expect_tx(full + stage, K::STAGE_BYTES);
                                tma_load_4d(dst, &maps.k, full + stage, 0, kvh, so, blk, pol);
                                tma_load_4d(dst + K::TILE_BYTES, &maps.v, full + stage, 0, kvh,
                                            so, blk, pol);
                            }
                        } else {
                            // the tile spans a block end: it is copied as T / h boxes
                            // of h = box_rows rows (h divides T and block_size, so no
                            // box spans a block), lane i copying box i from the block
                            // that holds it; every lane walks the blocks' shares of the
                            // tile (the block comes by shuffle), so the boxes go out
                            // in one warp instruction
                            int br = -1, bslot = 0, bblk = 0;
                            for (int ru = 0, nb = 0, blki = bi, s0 = su; ru < tile_u;
                                 ++blki, s0 = 0) {
                                const int len = min(tile_u - ru, block_u - s0);
                                const int blk = __shfl_sync(0xffffffffu, win_entry, blki - win_lo);
                                const int i = lane - nb;
                                if (i >= 0 && i < len) {
                                    br = ru + i;
                                    bslot = (s0 + i) * hrows;
                                    bblk = blk;
                                }
                                nb += len;
                                ru += len;
                            }
                            if (lane == 0) mbar_arrive_expect_tx(full + stage, K::STAGE_BYTES);
                            __syncwarp();
                            if (br >= 0) {
                                const int off = br * hrows * D * K::ES;
                                tma_load_4d(dst + off, &maps.kb, full + stage, 0, kvh, bslot, bblk,
                                            pol);
                                tma_load_4d(dst + K::TILE_BYTES + off, &maps.vb, full + stage, 0,
                                            kvh, bslot, bblk, pol);
                            }
                        }
                        for (su += tile_u; su >= block_u; su -= block_u) ++bi;
                    } else if (lane == 0) { // contiguous: one box at (position, sequence)
                        mbar_arrive_expect_tx(full + stage, K::STAGE_BYTES);
                        tma_load_4d(dst, &maps.k, full + stage, 0, kvh, t0, b, pol);
                        tma_load_4d(dst + K::TILE_BYTES, &maps.v, full + stage, 0, kvh, t0, b, pol);
                    }
#pragma unroll
                    for (int x = 0; x < NST; ++x)
                        if (x == stage) last_parity[x] = (int)phase;
                }
                if (++stage == NST) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
        }
        if (lane == 0) {
            if (!ok) {
                *abort_flag = 1;
                atomicCAS(p.status, 0, kStatusTimeoutGqa);
            }
            // Nothing may be in flight when the CTA exits: wait (bounded) for the
            // last copy issued into every stage.
            volatile int never = 0;
#pragma unroll
            for (int s = 0; s < NST; ++s)
                if (last_parity[s] >= 0)
                    (void)mbar_wait_bounded(full + s, (uint32_t)last_parity[s], p.timeout_ns,
                                            &never);
        }
        return;
    }

    // --------------------------------- consumers ---------------------------------
    float *scr = reinterpret_cast<float *>(smem + K::OFF_WARP) + warp * K::WARP_SCR;
    float *sc = scr;               // [NV] scores (log2 units), masked
    float *pscr = scr + K::NV;     // [NV] probabilities
    float *mw = pscr + K::NV;      // [G] running max of this warp
    float *aw = mw + G;            // [G] last rescale factors
    const int half = lane / LPR, sub = lane % LPR; // lane group (row of a step) and lane in it
    const int tbase = tr_base<K::NVL, LPR / 2>(lane);
    const bool twriter = tr_writer<K::NVL, LPR / 2>(lane);

    // The rows of a (sequence, KV head) group are (query token, head) pairs:
    // row jf is token jf / Gh and head kvh * Gh + jf % Gh of that token, Gh =
    // heads per KV head. A work item holds G of them: rows [rg G, rg G + G) of
    // its row group rg (all of them when there is one group). Offsets of row jf
    // from the (sequence, group) base, in q and workspace rows:
    const int Gh = p.hq / it.n_kv_heads;
    const int rows_grp = Gh * p.q_len; // rows of a (sequence, KV head) group
    auto row_off = [&](int jf) { return p.q_len == 1 ? jf : (jf / Gh) * p.hq + jf % Gh; };
    // the token of each (step, row) value this lane writes after the reduce;
    // constant over an item's tiles, so the causal test in the tile loop is an add
    int tok_r[K::R];
    auto set_tokens = [&](int rg) {
#pragma unroll
        for (int r = 0; r < K::R; ++r) tok_r[r] = (rg * G + (tbase + r) % G) / Gh;
    };

    // q for the G rows of an item's group, pre-scaled into log2 units. The
    // next item's q is loaded right after the last tile of the current one,
    // so the load overlaps the merge.
    float q[G][K::EPL];
    auto load_q = [&](int item) {
        int qb_b, qb_kvh, qb_s, qb_rg;
        decode_item(it, item, qb_b, qb_kvh, qb_s, qb_rg);
        const float *qb = p.q + ((size_t)qb_b * p.n_heads + (size_t)qb_kvh * Gh) * D;
#pragma unroll
        for (int h = 0; h < G; ++h)
#pragma unroll
            for (int c = 0; c < K::NCH; ++c)
#pragma unroll
                for (int e = 0; e < K::EPC; e += 4) {
                    float4 x = *reinterpret_cast<const float4 *>(
                        qb + (size_t)row_off(qb_rg * G + h) * D + (c * LPR + sub) * K::EPC + e);
                    q[h][c * K::EPC + e + 0] = x.x * p.scale_log2;
                    q[h][c * K::EPC + e + 1] = x.y * p.scale_log2;
                    q[h][c * K::EPC + e + 2] = x.z * p.scale_log2;
                    q[h][c * K::EPC + e + 3] = x.w * p.scale_log2;
                }
    };
    if (blockIdx.x < it.n_items) load_q(blockIdx.x);
    named_bar_sync(2, K::CONSUMERS + 32); // the producer's barrier set-up

    int stage = 0;
    uint32_t phase = 0;
    for (int item = blockIdx.x; item < it.n_items; item += gridDim.x) {
        int b, kvh, s, rg;
        decode_item(it, item, b, kvh, s, rg);
        set_tokens(rg);
        const int jg = rg * G; // the item's first row of its (sequence, KV head) group
        const int p0 = s * it.chunk[b];
        const int Lb = item_len(p, b);
        const int p1 = min(Lb, p0 + it.chunk[b]); // p1 <= p0: an empty item
        // token i of q_len sees positions below lim0 + i (causal among the new
        // tokens); with one token lim0 = Lb and no tile reaches past it, and a
        // slice before the new tokens (DA_FLAG_NO_CAUSAL) has no limit
        const int lim0 = (p.flags & DA_FLAG_NO_CAUSAL) ? (INT_MAX >> 1) : Lb - p.q_len + 1;

        float acc[G][K::EPL];
        float m[G];
#pragma unroll
        for (int h = 0; h < G; ++h) {
            m[h] = kNeutralM;
#pragma unroll
            for (int e = 0; e < K::EPL; ++e) acc[h][e] = 0.f;
        }
        float l_lane[K::R2];
#pragma unroll
        for (int k = 0; k < K::R2; ++k) l_lane[k] = 0.f;
        if (lane < G) mw[lane] = kNeutralM;
        __syncwarp();

        bool aborted = false;
        for (int t0 = p0, t1; t0 < p1; t0 = t1) {
            t1 = tile_end<T>(t0, p1);
            if (!mbar_wait_bounded(full + stage, phase, p.timeout_ns, abort_flag)) {
                aborted = true;
                break;
            }
            const DT *Kt = reinterpret_cast<const DT *>(smem + stage * K::STAGE_BYTES) +
                           warp * K::P * D;
            const DT *Vt = reinterpret_cast<const DT *>(smem + stage * K::STAGE_BYTES +
                                                        K::TILE_BYTES) +
                           warp * K::P * D;
            const int valid = min(t1 - t0 - warp * K::P, K::P);
            if (valid > 0) {
                // ---- scores: P rows x G heads, partial over this lane's elements;
                // step r2 reads row r2 * RPW + half
                float dv[K::NVL];
#pragma unroll
                for (int i = 0; i < K::NVL; ++i) dv[i] = 0.f;
#pragma unroll
                for (int r2 = 0; r2 < K::PH; ++r2)
#pragma unroll
                    for (int c = 0; c < K::NCH; ++c) {
                        float kf[K::EPC];
                        Chunk<DT, K::EPC>::load(
                            Kt + (r2 * K::RPW + half) * D + (c * LPR + sub) * K::EPC, kf);
#pragma unroll
                        for (int h = 0; h < G; ++h)
#pragma unroll
                            for (int e = 0; e < K::EPC; ++e)
                                dv[r2 * G + h] = fmaf(q[h][c * K::EPC + e], kf[e], dv[r2 * G + h]);
                    }
                tr_reduce<K::NVL, LPR / 2>(dv, lane);
                if (t1 <= lim0) {
#pragma unroll
                    for (int r = 0; r < K::R; ++r) {
                        const int idx = tbase + r;                   // (step, row) of this group
                        const int row = (idx / G) * K::RPW + half;
                        const float sv = (row < valid) ? dv[r] : -INFINITY;
                        if (twriter) sc[row * G + idx % G] = sv;
                    }
                } else { // a tile that reaches the new tokens (rare): the causal limit too
#pragma unroll
                    for (int r = 0; r < K::R; ++r) {
                        const int idx = tbase + r;
                        const int row = (idx / G) * K::RPW + half;
                        const bool live =
                            row < valid && t0 + warp * K::P + row < lim0 + tok_r[r];
                        const float sv = live ? dv[r] : -INFINITY;
                        if (twriter) sc[row * G + idx % G] = sv;
                    }
                }
                __syncwarp();
                // ---- running max per head (every lane computes it redundantly)
                float tmax[G];
#pragma unroll
                for (int h = 0; h < G; ++h) tmax[h] = -INFINITY;
#pragma unroll
                for (int i = 0; i < K::NV / 4; ++i) {
                    const float4 x = reinterpret_cast<const float4 *>(sc)[i];
                    tmax[(4 * i + 0) % G] = fmaxf(tmax[(4 * i + 0) % G], x.x);
                    tmax[(4 * i + 1) % G] = fmaxf(tmax[(4 * i + 1) % G], x.y);
                    tmax[(4 * i + 2) % G] = fmaxf(tmax[(4 * i + 2) % G], x.z);
                    tmax[(4 * i + 3) % G] = fmaxf(tmax[(4 * i + 3) % G], x.w);
                }
                bool changed = false;
#pragma unroll
                for (int h = 0; h < G; ++h) changed |= tmax[h] > m[h];
                if (changed) { // warp-uniform: every lane holds the same m and tmax
#pragma unroll
                    for (int h = 0; h < G; ++h) {
                        const float mn = fmaxf(m[h], tmax[h]);
                        const float alpha = ex2(m[h] - mn);
                        m[h] = mn;
#pragma unroll
                        for (int e = 0; e < K::EPL; ++e) acc[h][e] *= alpha;
                        if (lane == h) {
                            mw[h] = mn;
                            aw[h] = alpha;
                        }
                    }
                    __syncwarp();
#pragma unroll
                    for (int k = 0; k < K::R2; ++k) {
                        const int idx = lane + 32 * k;
                        if (idx < K::NV) l_lane[k] *= aw[idx % G];
                    }
                }
                // ---- probabilities, one (row, head) pair per lane
#pragma unroll
                for (int k = 0; k < K::R2; ++k) {
                    const int idx = lane + 32 * k;
                    if (idx < K::NV) {
                        const float pv = ex2(sc[idx] - mw[idx % G]);
                        pscr[idx] = pv;
                        l_lane[k] += pv;
                    }
                }
                __syncwarp();
                // ---- acc += p * v over the valid rows (each lane group its own rows)
#pragma unroll
                for (int r2 = 0; r2 < K::PH; ++r2) {
                    const int r = r2 * K::RPW + half;
                    if (r < valid) {
                        float pw[G];
                        if constexpr (G % 4 == 0) {
#pragma unroll
                            for (int h = 0; h < G; h += 4) {
                                const float4 x =
                                    *reinterpret_cast<const float4 *>(pscr + r * G + h);
                                pw[h] = x.x; pw[h + 1] = x.y; pw[h + 2] = x.z; pw[h + 3] = x.w;
                            }
                        } else if constexpr (G % 2 == 0) {
#pragma unroll
                            for (int h = 0; h < G; h += 2) {
                                const float2 x =
                                    *reinterpret_cast<const float2 *>(pscr + r * G + h);
                                pw[h] = x.x; pw[h + 1] = x.y;
                            }
                        } else {
#pragma unroll
                            for (int h = 0; h < G; ++h) pw[h] = pscr[r * G + h];
                        }
#pragma unroll
                        for (int c = 0; c < K::NCH; ++c) {
                            float vf[K::EPC];
                            Chunk<DT, K::EPC>::load(Vt + r * D + (c * LPR + sub) * K::EPC, vf);
#pragma unroll
                            for (int h = 0; h < G; ++h)
#pragma unroll
                                for (int e = 0; e < K::EPC; ++e)
                                    acc[h][c * K::EPC + e] =
                                        fmaf(pw[h], vf[e], acc[h][c * K::EPC + e]);
                        }
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(empty + stage);
            if (++stage == NST) {
                stage = 0;
                phase ^= 1u;
            }
        }
        if (aborted) {
            *abort_flag = 1;
            atomicCAS(p.status, 0, kStatusTimeoutGqa);
        }
        // Barrier A (always taken): the OR makes the abort decision uniform.
        if (named_bar_or(1, K::CONSUMERS, aborted || *abort_flag)) break;
        if (item + (int)gridDim.x < it.n_items) load_q(item + gridDim.x);
        if constexpr (K::RPW == 2) {
            // the two lane groups hold the same value columns for different rows
#pragma unroll
            for (int h = 0; h < G; ++h)
#pragma unroll
                for (int e = 0; e < K::EPL; ++e)
                    acc[h][e] += __shfl_xor_sync(0xffffffffu, acc[h][e], 16);
        }

        // ---- merge the NCW warp states of this item ----
        // per-warp l per head from the per-lane partial sums
#pragma unroll
        for (int k = 0; k < K::R2; ++k) {
            const int idx = lane + 32 * k;
            if (idx < K::NV) pscr[idx] = l_lane[k];
        }
        __syncwarp();
        if (lane < G) {
            float lw = 0.f;
#pragma unroll
            for (int r = 0; r < K::P; ++r) lw += pscr[r * G + lane];
            sm_ml[warp * G + lane] = make_float2(mw[lane], lw);
        }
        named_bar_sync(1, K::CONSUMERS); // B
        // lane h < G forms the item's max and sum for head h over the warps
        float Mh = kNeutralM, Lh = 0.f;
        if (lane < G) {
#pragma unroll
            for (int w = 0; w < NCW; ++w) Mh = fmaxf(Mh, sm_ml[w * G + lane].x);
#pragma unroll
            for (int w = 0; w < NCW; ++w) {
                const float2 x = sm_ml[w * G + lane];
                Lh += x.y * ex2(x.x - Mh);
            }
        }
        {
            // every warp rescales its acc to the common max of the item ...
#pragma unroll
            for (int h = 0; h < G; ++h) {
                const float f = ex2(m[h] - __shfl_sync(0xffffffffu, Mh, h));
#pragma unroll
                for (int e = 0; e < K::EPL; ++e) acc[h][e] *= f;
            }
            // ... and the warps are summed in a fixed order, so the merged partial
            // does not depend on timing (bit-reproducible). A CTA's last item finds
            // the stage ring idle (every copy has landed and been consumed): all
            // warps store their acc there and every consumer thread sums one
            // float4 of the item over the warps and writes it. Earlier items,
            // whose next tiles may be landing in the ring, sum through a pairwise
            // tree of slots into warp 0, which writes the partial.
        }
        const size_t slot_id = (size_t)it.split_base[b] + s;
        const size_t row0 = slot_id * p.n_heads + (size_t)kvh * Gh;
        if (item + (int)gridDim.x >= it.n_items) {
            float *flat = reinterpret_cast<float *>(smem);
            if (half == 0) {
#pragma unroll
                for (int h = 0; h < G; ++h)
#pragma unroll
                    for (int c = 0; c < K::NCH; ++c)
#pragma unroll
                        for (int e = 0; e < K::EPC; e += 4)
                            *reinterpret_cast<float4 *>(flat + (warp * G + h) * D +
                                                        (c * LPR + sub) * K::EPC + e) =
                                make_float4(acc[h][c * K::EPC + e], acc[h][c * K::EPC + e + 1],
                                            acc[h][c * K::EPC + e + 2], acc[h][c * K::EPC + e + 3]);
            }
            named_bar_sync(1, K::CONSUMERS);
            const float4 *flat4 = reinterpret_cast<const float4 *>(flat);
            for (int i = threadIdx.x; i < G * D / 4; i += K::CONSUMERS) {
                float4 y = flat4[i];
#pragma unroll
                for (int w = 1; w < NCW; ++w) {
                    const float4 z = flat4[w * (G * D / 4) + i];
                    y.x += z.x;
                    y.y += z.y;
                    y.z += z.z;
                    y.w += z.w;
                }
                const int h = i / (D / 4);
                *reinterpret_cast<float4 *>(p.acc + (row0 + row_off(jg + h)) * D +
                                            (i - h * (D / 4)) * 4) = y;
            }
            if (warp == 0 && lane < G)
                p.ml[row0 + row_off(jg + lane)] = make_float2(Lh > 0.f ? Mh * kLn2 : kNeutralM, Lh);
        } else {
#pragma unroll
            for (int d = 1, lvl = 0; d < NCW; d *= 2, ++lvl) {
                float *set = sm_tree + ((lvl & 1) ? K::TREE_EVEN : 0) * G * D;
                float *slot = set + (warp / (2 * d)) * G * D;
                if (warp % (2 * d) == d && half == 0) {
#pragma unroll
                    for (int h = 0; h < G; ++h)
#pragma unroll
                        for (int c = 0; c < K::NCH; ++c)
#pragma unroll
                            for (int e = 0; e < K::EPC; e += 4)
                                *reinterpret_cast<float4 *>(slot + h * D + (c * LPR + sub) * K::EPC + e) =
                                    make_float4(acc[h][c * K::EPC + e], acc[h][c * K::EPC + e + 1],
                                                acc[h][c * K::EPC + e + 2], acc[h][c * K::EPC + e + 3]);
                }
                named_bar_sync(1, K::CONSUMERS);
                if (warp % (2 * d) == 0 && warp + d < NCW && half == 0) {
#pragma unroll
                    for (int h = 0; h < G; ++h)
#pragma unroll
                        for (int c = 0; c < K::NCH; ++c)
#pragma unroll
                            for (int e = 0; e < K::EPC; e += 4) {
                                const float4 y = *reinterpret_cast<const float4 *>(
                                    slot + h * D + (c * LPR + sub) * K::EPC + e);
                                acc[h][c * K::EPC + e] += y.x;
                                acc[h][c * K::EPC + e + 1] += y.y;
                                acc[h][c * K::EPC + e + 2] += y.z;
                                acc[h][c * K::EPC + e + 3] += y.w;
                            }
                }
            }
            // warp 0 writes the partial: acc from its registers, (m, l) per head
            if (warp == 0) {
                if (half == 0) {
                    float *dst = p.acc + row0 * D;
#pragma unroll
                    for (int h = 0; h < G; ++h)
#pragma unroll
                        for (int c = 0; c < K::NCH; ++c)
#pragma unroll
                            for (int e = 0; e < K::EPC; e += 4)
                                *reinterpret_cast<float4 *>(dst + (size_t)row_off(jg + h) * D +
                                                            (c * LPR + sub) * K::EPC + e) =
                                    make_float4(acc[h][c * K::EPC + e], acc[h][c * K::EPC + e + 1],
                                                acc[h][c * K::EPC + e + 2], acc[h][c * K::EPC + e + 3]);
                }
                if (lane < G)
                    p.ml[row0 + row_off(jg + lane)] =
                        make_float2(Lh > 0.f ? Mh * kLn2 : kNeutralM, Lh);
            }
        }
        if (p.fused.on) {
            // the merge without a combine launch: every writer publishes its share
            // of the partial, then one arrival on the group's counter
            __threadfence();
            named_bar_sync(1, K::CONSUMERS);
            if (threadIdx.x == 0) (void)arrive(p.fused.ctr + (size_t)b * it.n_kv_heads + kvh);
        }
    }
    // the consumer warps take the same decision (a barrier-wide or of the flag)
    if (p.fused.on && !named_bar_or(1, K::CONSUMERS, *abort_flag != 0))
        fused_merge_shares<D, NCW>(p, abort_flag);
    if (threadIdx.x == 0) griddep_launch_dependents();
}

} // namespace skv
