// GQA / MQA split kernel on tcgen05 tensor cores, for work items with many
// query rows, sm_103a.
//
// An item is (sequence b, KV head, split s), as for the SIMT kernel, but its
// rows are R = (query heads per KV head) x q_len (query token, head) pairs,
// 8 <= R <= 128: a group of heads sharing a KV head, and for several new
// tokens per sequence every token of the group ("Decoder Block 6: Online
// Attention, the Capstone", Lesson: a tile of query rows consumes each staged
// K/V tile once). With that many rows each tile is a small dense contraction,
//     S[r][pos]  = sum_d Q[r][d] K[pos][d]          (M = 128 rows, N = 64 positions, K = D)
//     O^T[e][r] += sum_pos V[pos][e] P[r][pos]      (M = 128 value columns per block, N = R)
// and both run on the tensor cores (16-bit operands of the cache's own type,
// f32 accumulation in TMEM), so the SIMT issue rate no longer bounds the
// kernel: the K/V stream does.
//
// Data path: a producer warp copies each 64-position tile of K and of V with
// TMA in 64-column boxes that land 128-byte-swizzled (the layout the MMA
// reads), into a ring of stages; there is no conversion and no register
// staging. Q (scale * log2 e folded in, rounded to the cache type) is written
// once per item into the same swizzled K-major layout at the start of shared
// memory; rows R.. of the 128-row MMA read past a Q chunk into the next one
// (past the last, into the first stage) and give S rows that no thread reads.
//
// Roles (6 warps, one CTA per SM):
//   warps 0-3  softmax and epilogue: thread r owns row r (TMEM lane r of S):
//              its 64 scores per tile (one TMEM round trip), running max m and
//              sum l in registers, its probability row of P; causal limit
//              among the new tokens; the lazy rescale of the MLA kernel
//              (reference max moved only by more than 8 in log2 units). In
//              the epilogue thread e reads value column e of O^T.
//   warp 4     TMA producer (one lane; the whole warp for paged caches, as in
//              the SIMT kernel: a tile is copied as boxes that each lie in one
//              block, so tiles span blocks).
//   warp 5     TMEM owner and the one thread that issues the MMAs; it polls
//              QK(t+1) (tile in, S slot free) and PV(t) (P written) and
//              issues whichever is ready.
// Every wait is bounded; a wait that runs out sets the status word and the
// CTA drains and returns.
#include <climits>
#include <type_traits>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "gqa_split.cuh"
#include "internal.h"
#include "merge.cuh"
#include "ptx.cuh"

namespace skv {
namespace {

constexpr int kTcThreads = 192;
constexpr int kTcProd = 4;  // producer warp
constexpr int kTcMma = 5;   // MMA warp
constexpr float kTcTau = 8.f;
constexpr int kTcOCol = 128; // O^T block j at kTcOCol + j * npv (after two S slots of T <= 64)

// barrier indices
constexpr int TB_FULL = 0, TB_EMPTY = kTcMaxStages, TB_SFULL = 2 * kTcMaxStages,
              TB_SFREE = TB_SFULL + 2, TB_PFULL = TB_SFREE + 2, TB_PFREE = TB_PFULL + 2,
              TB_PVDONE = TB_PFREE + 2, TB_OREADY = TB_PVDONE + 1, TB_OFREE = TB_OREADY + 1,
              TB_QFULL = TB_OFREE + 1, TB_QFREE = TB_QFULL + 1, TB_DRAIN = TB_QFREE + 1,
              TB_N = TB_DRAIN + 1;
static_assert(TB_N <= kTcBarriers, "barrier count");

// byte offset of (row, byte) in a region of 128-byte rows with 128-byte swizzle
// (the pattern TMA's 128-byte swizzle writes)
__device__ __forceinline__ uint32_t tsw(uint32_t row, uint32_t byte)
{
    return (row >> 3) * 1024 + (row & 7) * 128 + ((((byte >> 4) ^ row) & 7) << 4) + (byte & 15);
}

template <typename DT> __device__ __forceinline__ uint32_t pack2(float a, float b);
template <> __device__ __forceinline__ uint32_t pack2<__half>(float a, float b)
{
    __half2 h = __floats2half2_rn(a, b);
    return *reinterpret_cast<uint32_t *>(&h);
}
template <> __device__ __forceinline__ uint32_t pack2<__nv_bfloat16>(float a, float b)
{
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t *>(&h);
}

__device__ __forceinline__ bool tc_bar_or(bool pred)
{
    uint32_t r;
    asm volatile("{\n\t.reg .pred p, q;\n\t"
                 "setp.ne.u32 p, %1, 0;\n\t"
                 "bar.red.or.pred q, 1, 128, p;\n\t"
                 "selp.u32 %0, 1, 0, q;\n\t}"
                 : "=r"(r)
                 : "r"((uint32_t)pred)
                 : "memory");
    return r != 0;
}

// The (item, tile) sequence of a CTA, the same for every role: items
// blockIdx.x, blockIdx.x + gridDim.x, ...; an item's tiles are T positions,
// the last one cut at the item's end (block ends of a paged cache do not cut
// tiles: the producer copies a tile box by box); items without positions
// (device lengths shorter than the plan's) have no tiles and are skipped.
template <int T> struct Walk {
    int item, b, kvh, s, p0, p1, t0, t1, gt;
    bool done, first;
    __device__ __forceinline__ void load_item(const SplitParams &p)
    {
        for (;;) {
            done = item >= p.items.n_items;
            if (done) return;
            decode_item(p.items, item, b, kvh, s);
            p0 = s * p.items.chunk[b];
            p1 = min(item_len(p, b), p0 + p.items.chunk[b]);
            if (p1 > p0) break;
            item += gridDim.x;
        }
        t0 = p0;
        t1 = tile_end<T>(t0, p1);
        first = true;
    }
    __device__ __forceinline__ void start(const SplitParams &p)
    {
        item = blockIdx.x;
        gt = 0;
        load_item(p);
    }
    __device__ __forceinline__ bool last() const { return t1 >= p1; }
    __device__ __forceinline__ void next(const SplitParams &p)
    {
        ++gt;
        if (t1 >= p1) {
            item += gridDim.x;
            load_item(p);
        } else {
            t0 = t1;
            t1 = tile_end<T>(t0, p1);
            first = false;
        }
    }
};

// The merge without a combine launch, run by the four softmax warps of every
// CTA once all its own partials are written and counted: for each of its items
// the CTA waits (bounded) until every split of the item's (sequence, KV head)
// group has arrived, then merges share s (the item's split) of the group's
// (row, 16 value columns) units into out. The library fuses only when the
// whole grid is resident at once, so no wait depends on a CTA that has not
// started, and a CTA waits only after its own arrivals.
template <int D>
__device__ __noinline__ void tc_merge_shares(const SplitParams &p, volatile int *abort_flag)
{
    constexpr int C = 4, CU = D / (4 * C); // float4s per unit, units per row
    const ItemTable &it = p.items;
    const int warp = threadIdx.x >> 5;
    const int Gh = p.hq / it.n_kv_heads;
    const int U = Gh * p.q_len * CU;
    volatile int *go = abort_flag + 1;
    for (int item = blockIdx.x; item < it.n_items; item += gridDim.x) {
        int b, kvh, s;
        decode_item(it, item, b, kvh, s);
        const int S = it.split_base[b + 1] - it.split_base[b];
        if (threadIdx.x == 0) {
            const volatile uint32_t *ctr = p.fused.ctr + (size_t)b * it.n_kv_heads + kvh;
            const uint64_t t0 = global_ns();
            bool ok = true;
            while (*ctr < (uint32_t)S) {
                if (*abort_flag || global_ns() - t0 > p.timeout_ns) {
                    ok = false;
                    *abort_flag = 1;
                    atomicCAS(p.status, 0, kStatusTimeoutTc);
                    break;
                }
                __nanosleep(64);
            }
            *go = ok ? 1 : 0;
        }
        named_bar_sync(1, 128);
        if (!*go) break;
        __threadfence(); // the group's partials, before they are read
        const int u0 = (int)((int64_t)s * U / S), u1 = (int)((int64_t)(s + 1) * U / S);
        for (int u = u0 + warp; u < u1; u += 4) {
            const int rr = u / CU, tk = rr / Gh;
            const int row = kvh * Gh + tk * p.hq + (rr - tk * Gh);
            warp_merge_cols<C, 8>(p.ml, p.acc, (size_t)it.split_base[b], S, p.n_heads, row, D,
                                  (u - rr * CU) * C, out_row_ptr(p.fused, b, p.n_heads, row, D),
                                  p.fused.out_dtype);
        }
        named_bar_sync(1, 128); // *go is read before it is rewritten
    }
}

template <typename DT, int D>
__global__ void __launch_bounds__(kTcThreads, 1)
    gqa_tc_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                  const __grid_constant__ SplitParams p)
{
    constexpr int T = tc_tile(D); // positions per tile: QK N, PV K
    constexpr int NCH = D / 64;   // 64-column chunks of a row
    constexpr int NBLK = D / 128; // 128-column blocks of O^T
    const int R = p.n_heads / p.items.n_kv_heads; // rows of an item
    const int Gh = p.hq / p.items.n_kv_heads;     // query heads per KV head
    const TcLayout L = tc_layout(D, R);

    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sb = smem_u32(sm);
    uint64_t *bar = reinterpret_cast<uint64_t *>(sm + L.bar_off);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + L.misc_off);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(sm + L.misc_off + 4);
    float *alpha_sm = reinterpret_cast<float *>(sm + L.alpha_off);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int NST = L.nst;
    volatile int never = 0;

    if (threadIdx.x == 0) {
        for (int s = 0; s < NST; ++s) {
            mbar_init(bar + TB_FULL + s, 1);
            mbar_init(bar + TB_EMPTY + s, 1);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(bar + TB_SFULL + s, 1);
            mbar_init(bar + TB_SFREE + s, 4);
            mbar_init(bar + TB_PFULL + s, 4);
            mbar_init(bar + TB_PFREE + s, 1);
        }
        mbar_init(bar + TB_PVDONE, 1);
        mbar_init(bar + TB_OREADY, 1);
        mbar_init(bar + TB_OFREE, 4);
        mbar_init(bar + TB_QFULL, 4);
        mbar_init(bar + TB_QFREE, 1);
        mbar_init(bar + TB_DRAIN, 1);
        *abort_flag = 0;
        if (blockIdx.x == 0) *p.status = 0;
        fence_mbar_init();
    }
    if (warp == kTcMma) tmem_alloc(tmem_slot, 512);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == kTcProd) {
        // =============================== TMA producer ===============================
        const bool paged = p.block_table != nullptr;
        if (paged || lane == 0) {
            const unsigned mask = paged ? 0xffffffffu : 1u;
            if (lane == 0) {
                tma_prefetch_map(&kmap);
                tma_prefetch_map(&vmap);
            }
            const uint64_t pol = l2_evict_first_policy();
            uint32_t eph = 0;
            int win_b = -1, win_lo = 0;
            int32_t win_entry = 0;
            bool ok = true;
            Walk<T> w;
            for (w.start(p); !w.done; w.next(p)) {
                const int st = w.gt % NST;
                // a stage's first use finds its barrier's previous phase complete
                bool got = true;
                if (lane == 0)
                    got = mbar_wait_bounded(bar + TB_EMPTY + st, ((eph >> st) & 1u) ^ 1u,
                                            p.timeout_ns, abort_flag);
                eph ^= 1u << st;
                if (!__shfl_sync(mask, got, 0)) {
                    ok = false;
                    break;
                }
                if (p.flags & DA_FLAG_TEST_NO_TMA) continue;
                uint8_t *dst = sm + L.stage_off + st * L.stage_bytes;
                if (paged) {
                    // box j holds rows [t0 + j*h, t0 + (j+1)*h) of every 64-column
                    // chunk, h = box_rows (16, 32 or 64: a divisor of the tile and of
                    // block_size), so no box spans two blocks and a tile spans blocks
                    // freely; h * 128 bytes is a multiple of the 1024-byte swizzle
                    // atom, so the boxes land in the layout one 64-row box would give
                    const int bs = p.block_size, h = p.box_rows, nbox = T / h;
                    const int lo = w.t0 / bs, hi = (w.t0 + T - 1) / bs;
                    if (w.b != win_b || lo < win_lo || hi >= win_lo + 32) {
                        win_b = w.b;
                        win_lo = lo;
                        win_entry = (lo + lane < p.max_blocks)
                                        ? p.block_table[(size_t)w.b * p.max_blocks + lo + lane]
                                        : p.oob_block;
                    }
                    const int pos = w.t0 + min(lane, nbox - 1) * h;
                    const int idx = pos / bs;
                    const int blk = __shfl_sync(0xffffffffu, win_entry, idx - win_lo);
                    if (lane == 0) mbar_arrive_expect_tx(bar + TB_FULL + st, L.stage_bytes);
                    __syncwarp();
                    if (lane < nbox) {
                        // rows of a box past the pool read as zeros
#pragma unroll
                        for (int c = 0; c < NCH; ++c) {
                            const int off = c * L.chunk_bytes + lane * h * 128;
                            tma_load_4d(dst + off, &kmap, bar + TB_FULL + st, c * 64, w.kvh,
                                        pos - idx * bs, blk, pol);
                            tma_load_4d(dst + L.tile_bytes + off, &vmap, bar + TB_FULL + st,
                                        c * 64, w.kvh, pos - idx * bs, blk, pol);
                        }
                    }
                } else if (lane == 0) {
                    // contiguous: one box per chunk at (position, sequence); rows past
                    // the cache read as zeros
                    mbar_arrive_expect_tx(bar + TB_FULL + st, L.stage_bytes);
#pragma unroll
                    for (int c = 0; c < NCH; ++c) {
                        tma_load_4d(dst + c * L.chunk_bytes, &kmap, bar + TB_FULL + st, c * 64,
                                    w.kvh, w.t0, w.b, pol);
                        tma_load_4d(dst + L.tile_bytes + c * L.chunk_bytes, &vmap,
                                    bar + TB_FULL + st, c * 64, w.kvh, w.t0, w.b, pol);
                    }
                }
            }
            if (!ok && lane == 0) {
                *abort_flag = 1;
                atomicCAS(p.status, 0, kStatusTimeoutTc);
            }
        }
    } else if (warp == kTcMma) {
        // ============================ MMA issue (1 thread) ============================
        if (lane == 0) {
            constexpr bool BF = sizeof(DT) == 2 && !std::is_same<DT, __half>::value;
            const uint32_t idesc_qk = idesc_f16kind(128, T, 0, 0, BF);
            const uint32_t idesc_pv = idesc_f16kind(128, L.npv, 1, 0, BF);
            uint32_t fph = 0, sph = 0, pph = 0, qph = 0, oph = 0;
            bool ok = true, q_ready = false;
            int items_pv = 0;
            Walk<T> qk, pv;
            qk.start(p);
            pv.start(p);
            uint64_t last = global_ns();
            while (!pv.done) {
                bool progress = false;
                if (pv.gt < qk.gt) {
                    // O^T += V^T . P^T once P(t) is written (and, at an item's first
                    // tile, once the previous item's epilogue has read O^T)
                    const int ps = pv.gt & 1, st = pv.gt % NST;
                    if (mbar_test(bar + TB_PFULL + ps, (pph >> ps) & 1u) &&
                        (!pv.first || items_pv == 0 || mbar_test(bar + TB_OFREE, oph))) {
                        pph ^= 1u << ps;
                        if (pv.first && items_pv > 0) oph ^= 1u;
                        if (pv.first) ++items_pv;
                        tc_fence_after();
                        const uint32_t vt = sb + L.stage_off + st * L.stage_bytes + L.tile_bytes;
                        const uint64_t vd = smem_desc_sw128(vt, L.chunk_bytes, 1024);
                        const uint64_t pd = smem_desc_sw128(sb + L.p_off + ps * L.pslot, 16, 1024);
#pragma unroll
                        for (int j = 0; j < NBLK; ++j)
#pragma unroll
                            for (int k = 0; k < T / 16; ++k)
                                tc_mma_bf16(tmem + kTcOCol + j * L.npv,
                                            vd + (uint64_t)((2 * j * L.chunk_bytes + k * 2048) >> 4),
                                            pd + (uint64_t)((k * 32) >> 4), idesc_pv,
                                            (pv.first && k == 0) ? 0u : 1u);
                        tc_commit(bar + TB_EMPTY + st);
                        tc_commit(bar + TB_PFREE + ps);
                        tc_commit(bar + TB_PVDONE);
                        if (pv.last()) tc_commit(bar + TB_OREADY);
                        progress = true;
                        pv.next(p);
                    }
                }
                if (!qk.done) {
                    // S = Q . K_tile^T once Q of the item is in, the tile is full and
                    // the softmax has released this S slot
                    const int ss = qk.gt & 1, st = qk.gt % NST;
                    if (!q_ready && mbar_test(bar + TB_QFULL, qph)) {
                        qph ^= 1u;
                        q_ready = true;
                    }
                    if (q_ready && mbar_test(bar + TB_FULL + st, (fph >> st) & 1u) &&
                        mbar_test(bar + TB_SFREE + ss, ((sph >> ss) & 1u) ^ 1u)) {
                        fph ^= 1u << st;
                        sph ^= 1u << ss;
                        tc_fence_after();
                        const uint64_t qd = smem_desc_sw128(sb + L.q_off, 16, 1024);
                        const uint64_t kd = smem_desc_sw128(sb + L.stage_off + st * L.stage_bytes, 16, 1024);
#pragma unroll
                        for (int c = 0; c < NCH; ++c)
#pragma unroll
                            for (int k = 0; k < 4; ++k)
                                tc_mma_bf16(tmem + ss * T,
                                            qd + (uint64_t)((c * L.qch + k * 32) >> 4),
                                            kd + (uint64_t)((c * L.chunk_bytes + k * 32) >> 4),
                                            idesc_qk, (c | k) != 0 ? 1u : 0u);
                        tc_commit(bar + TB_SFULL + ss);
                        if (qk.last()) {
                            tc_commit(bar + TB_QFREE);
                            q_ready = false;
                        }
                        progress = true;
                        qk.next(p);
                    }
                }
                if (progress) {
                    last = global_ns();
                } else {
                    if (*abort_flag || global_ns() - last > p.timeout_ns) {
                        ok = false;
                        break;
                    }
                    __nanosleep(32);
                }
            }
            if (!ok && !*abort_flag) {
                *abort_flag = 1;
                atomicCAS(p.status, 0, kStatusTimeoutTc);
            }
            // no MMA may be in flight when TMEM is freed
            tc_commit(bar + TB_DRAIN);
            (void)mbar_wait_bounded(bar + TB_DRAIN, 0, p.timeout_ns, &never);
        }
        __syncwarp();
    } else {
        // ========================= softmax and epilogue (warps 0-3) ========================
        const int r = threadIdx.x;          // row of S (TMEM lane), value column in the epilogue
        const bool owner = r < R;
        const int token = r / Gh, g = r - (r / Gh) * Gh;
        const int row_off = owner ? token * p.hq + g : 0; // + kvh * Gh per item
        const uint32_t tl = tmem + ((uint32_t)(warp * 32) << 16);
        uint32_t sph = 0, pfp = 0, qfp = 0, oph = 0;
        bool ab = false;
        int items = 0, gt = 0;
        // After an item's partial is written: the four warps publish their
        // writes, then one arrival on the item's (sequence, KV head) group.
        auto arrive_group = [&](int b, int kvh) {
            __threadfence();
            named_bar_sync(1, 128);
            if (threadIdx.x == 0) (void)arrive(p.fused.ctr + (size_t)b * p.items.n_kv_heads + kvh);
        };
        for (int item = blockIdx.x; !ab && item < p.items.n_items; item += gridDim.x) {
            int b, kvh, s;
            decode_item(p.items, item, b, kvh, s);
            const int Lb = item_len(p, b);
            const int p0 = s * p.items.chunk[b];
            const int p1 = min(Lb, p0 + p.items.chunk[b]);
            const size_t slot_id = (size_t)p.items.split_base[b] + s;
            const size_t wrow = slot_id * p.n_heads + (size_t)kvh * Gh + row_off;
            if (p1 <= p0) { // an empty item: a neutral partial, no MMA took part
                if (owner) p.ml[wrow] = make_float2(kNeutralM, 0.f);
                if (p.fused.on) arrive_group(b, kvh);
                continue;
            }
            // ---- Q of this item's rows, once the previous item's QK is done with Q
            if (items > 0) {
                const bool okw =
                    mbar_wait_bounded(bar + TB_QFREE, qfp, p.timeout_ns, abort_flag);
                if (tc_bar_or(!okw)) break;
                qfp ^= 1u;
            }
            // the item's q rows [rpad][D], scaled and rounded to the cache type, in
            // the swizzled layout (rows past R zero): the four warps take 8-column
            // units, four per thread in flight, so q arrives in one round trip
            {
                constexpr int U8 = D / 8; // 8-column units of a row
                const int units = L.rpad * U8;
                const float sc = p.scale_log2;
                for (int u0 = threadIdx.x; u0 < units; u0 += 4 * 128) {
                    float4 qa[4], qb[4];
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const int u = u0 + i * 128, rr = u / U8;
                        qa[i] = qb[i] = make_float4(0.f, 0.f, 0.f, 0.f);
                        if (u < units && rr < R) {
                            const int tk = rr / Gh;
                            const float *qr = p.q +
                                              ((size_t)(b * p.q_len + tk) * p.hq +
                                               (size_t)kvh * Gh + (rr - tk * Gh)) * D +
                                              (u - rr * U8) * 8;
                            qa[i] = __ldg(reinterpret_cast<const float4 *>(qr));
                            qb[i] = __ldg(reinterpret_cast<const float4 *>(qr + 4));
                        }
                    }
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const int u = u0 + i * 128;
                        if (u < units) {
                            const int rr = u / U8, j8 = u - rr * U8;
                            sts_v4(sb + L.q_off + (j8 >> 3) * L.qch + tsw(rr, (j8 & 7) * 16),
                                   pack2<DT>(qa[i].x * sc, qa[i].y * sc),
                                   pack2<DT>(qa[i].z * sc, qa[i].w * sc),
                                   pack2<DT>(qb[i].x * sc, qb[i].y * sc),
                                   pack2<DT>(qb[i].z * sc, qb[i].w * sc));
                        }
                    }
                }
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar + TB_QFULL);
            ++items;

            // ---- tiles
            // token i of q_len sees positions below lim0 + i (causal among the new
            // tokens); with one token every position of the item is visible
            const int lim =
                (p.flags & DA_FLAG_NO_CAUSAL) ? (INT_MAX >> 1) : Lb - p.q_len + 1 + token;
            float m = -INFINITY, l = 0.f;
            bool firsttile = true;
            for (int t0 = p0, t1; t0 < p1; t0 = t1, ++gt, firsttile = false) {
                t1 = tile_end<T>(t0, p1);
                const int ss = gt & 1;
                // S(t) is in, and PV(t-2) is done with this P slot; the outcome of
                // both waits joins the rescale vote below (one block-wide vote per
                // tile in the common case)
                bool okw = mbar_wait_bounded(bar + TB_SFULL + ss, (sph >> ss) & 1u, p.timeout_ns,
                                             abort_flag);
                okw = okw && mbar_wait_bounded(bar + TB_PFREE + ss, ((pfp >> ss) & 1u) ^ 1u,
                                               p.timeout_ns, abort_flag);
                sph ^= 1u << ss;
                pfp ^= 1u << ss;
                tc_fence_after();
                if (t1 - t0 < T) {
                    // a short tile: the V rows past it hold whatever the cache (or
                    // the pool) has there; zero them, as 0 * NaN would reach O^T.
                    // (The K rows past it only give scores that are masked.)
                    const int tv = t1 - t0;
                    const uint32_t vt = sb + L.stage_off + (gt % NST) * L.stage_bytes + L.tile_bytes;
                    for (int i = r; i < (T - tv) * NCH * 8; i += 128) {
                        const int row = tv + i / (NCH * 8), rem = i % (NCH * 8);
                        sts_v4(vt + (rem >> 3) * L.chunk_bytes + tsw(row, (rem & 7) * 16), 0u, 0u,
                               0u, 0u);
                    }
                }
                const int nv = max(0, min(t1, lim) - t0); // visible positions of this row
                float sc[T];
#pragma unroll
                for (int q4 = 0; q4 < T / 16; ++q4) tmem_ld16(tl + ss * T + 16 * q4, sc + 16 * q4);
                tmem_wait_ld();
                float tm = -INFINITY;
#pragma unroll
                for (int i = 0; i < T; ++i)
                    if (i < nv) tm = fmaxf(tm, sc[i]);
                const bool ex = owner && tm > m + kTcTau;
                if (tc_bar_or(ex || !okw)) {
                    if (tc_bar_or(!okw)) { // a wait ran out somewhere: leave together
                        ab = true;
                        break;
                    }
                    // move the reference of the rows that outgrew it; rescale l and O^T
                    const float mn = ex ? tm : m;
                    const float alpha = (mn == m) ? 1.f : (m == -INFINITY ? 0.f : ex2(m - mn));
                    alpha_sm[r] = alpha;
                    l *= alpha;
                    m = mn;
                    if (!firsttile) {
                        // PV(t-1) is done with O^T before it is rescaled
                        okw = mbar_wait_bounded(bar + TB_PVDONE, (uint32_t)(gt - 1) & 1u,
                                                p.timeout_ns, abort_flag);
                        named_bar_sync(1, 128);
                        if (tc_bar_or(!okw)) {
                            ab = true;
                            break;
                        }
                        tc_fence_after();
                        for (int j = 0; j < NBLK; ++j)
                            for (int g16 = 0; g16 < L.npv / 16; ++g16) {
                                float o[16];
                                tmem_ld16(tl + kTcOCol + j * L.npv + 16 * g16, o);
                                tmem_wait_ld();
#pragma unroll
                                for (int i = 0; i < 16; ++i) o[i] *= alpha_sm[16 * g16 + i];
                                tmem_st16(tl + kTcOCol + j * L.npv + 16 * g16, o);
                            }
                        tmem_wait_st();
                    }
                    named_bar_sync(1, 128); // alpha_sm is read before it is rewritten
#pragma unroll
                    for (int q4 = 0; q4 < T / 16; ++q4)
                        tmem_ld16(tl + ss * T + 16 * q4, sc + 16 * q4);
                    tmem_wait_ld();
                }
                // P row: 2^(s - m) in the cache type
                if (r < L.npv) {
                    const uint32_t prow = sb + L.p_off + ss * L.pslot;
#pragma unroll
                    for (int q4 = 0; q4 < T / 16; ++q4) {
                        uint32_t w8[8];
#pragma unroll
                        for (int i = 0; i < 16; i += 2) {
                            const int c = 16 * q4 + i;
                            const float a0 = (owner && c < nv) ? ex2(sc[c] - m) : 0.f;
                            const float a1 = (owner && c + 1 < nv) ? ex2(sc[c + 1] - m) : 0.f;
                            l += a0 + a1;
                            w8[i >> 1] = pack2<DT>(a0, a1);
                        }
                        sts_v4(prow + tsw(r, 32 * q4), w8[0], w8[1], w8[2], w8[3]);
                        sts_v4(prow + tsw(r, 32 * q4 + 16), w8[4], w8[5], w8[6], w8[7]);
                    }
                }
                tc_fence_before();
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(bar + TB_SFREE + ss);
                    mbar_arrive(bar + TB_PFULL + ss);
                }
            }
            if (ab) break;
            // ------------------------------- epilogue -------------------------------
            const bool okw = mbar_wait_bounded(bar + TB_OREADY, oph, p.timeout_ns, abort_flag);
            if (tc_bar_or(!okw)) break;
            oph ^= 1u;
            tc_fence_after();
            // each row's partial row, from its owner thread (the scratch of the
            // rescale factors is free here), so the store loop has no division
            int *wrow_sm = reinterpret_cast<int *>(alpha_sm);
            wrow_sm[r] = owner ? (int)wrow : 0;
            named_bar_sync(1, 128);
            for (int j = 0; j < NBLK; ++j)
                for (int g16 = 0; g16 < L.npv / 16; ++g16) {
                    float o[16];
                    tmem_ld16(tl + kTcOCol + j * L.npv + 16 * g16, o);
                    tmem_wait_ld();
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        const int rr = 16 * g16 + i;
                        if (rr < R) p.acc[(size_t)wrow_sm[rr] * D + 128 * j + r] = o[i];
                    }
                }
            named_bar_sync(1, 128); // the table is read before the scratch is reused
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar + TB_OFREE);
            if (owner) p.ml[wrow] = make_float2(l > 0.f ? m * kLn2 : kNeutralM, l);
            if (p.fused.on) arrive_group(b, kvh);
        }
        if (ab && threadIdx.x == 0 && !*abort_flag) {
            *abort_flag = 1;
            atomicCAS(p.status, 0, kStatusTimeoutTc);
        }
        // the four warps take the same decision (a barrier-wide or of the flag)
        if (p.fused.on && !tc_bar_or(*abort_flag != 0)) tc_merge_shares<D>(p, abort_flag);
    }

    // ---------------------------------- teardown ----------------------------------
    tc_fence_before();
    __syncthreads();
    if (*abort_flag) {
        // let copies already in flight land before the CTA exits
        const uint64_t t0 = global_ns();
        while (global_ns() - t0 < 200000ull) {
        }
    }
    tc_fence_after();
    if (warp == kTcMma) tmem_dealloc(tmem, 512);
    if (threadIdx.x == 0) griddep_launch_dependents();
}

template <typename DT, int D>
cudaError_t launch_t(int grid, cudaStream_t st, const CUtensorMap &km, const CUtensorMap &vm,
                     const SplitParams &p, int smem)
{
    auto *fn = gqa_tc_kernel<DT, D>;
    cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    fn<<<grid, kTcThreads, smem, st>>>(km, vm, p);
    return cudaGetLastError();
}

} // namespace

cudaError_t launch_gqa_tc(int kv_dtype, int head_dim, int grid, cudaStream_t st,
                          const CUtensorMap &km, const CUtensorMap &vm, const SplitParams &p)
{
    const int R = p.n_heads / p.items.n_kv_heads;
    const TcLayout L = tc_layout(head_dim, R);
    if (L.nst < 2) return cudaErrorInvalidValue;
    const int smem = L.used + 1024;
    if (kv_dtype == DA_F16) {
        if (head_dim == 128) return launch_t<__half, 128>(grid, st, km, vm, p, smem);
        if (head_dim == 256) return launch_t<__half, 256>(grid, st, km, vm, p, smem);
    } else if (kv_dtype == DA_BF16) {
        if (head_dim == 128) return launch_t<__nv_bfloat16, 128>(grid, st, km, vm, p, smem);
        if (head_dim == 256) return launch_t<__nv_bfloat16, 256>(grid, st, km, vm, p, smem);
    }
    return cudaErrorInvalidValue;
}

} // namespace skv
