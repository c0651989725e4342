// MLA-as-MQA split kernel on tcgen05 tensor cores, sm_103a.
//
// Multi-head latent attention at decode is MQA: every query head attends over
// one shared 576-wide latent row per position (512 latent + 64 rope columns),
// and the values are the first 512 columns of the same rows ("Attention at
// 128k", §1.1 and §4; "The Kernel Level", absorbed MLA decode). With 96 heads
// against one shared latent the per-tile work is a real dense contraction:
//     S^T[pos][h] = sum_d K[pos][d] * Q[h][d]        (M = 128 positions, K = 576)
//     O^T[e][h]  += sum_pos V[pos][e] * P[pos][h]     (M = 512 in 4 blocks of 128)
// so both products run on the tensor cores (bf16 operands, f32 accumulation
// in TMEM), and each latent byte is read from HBM once for all heads.
//
// Work split: a cluster of two CTAs (on two SMs) takes a work item, a
// contiguous slice of one sequence's context (split over context, "Attention at
// 128k" §2). Both CTAs walk the slice in tiles of 128 positions. CTA r:
//   * converts rows [64r, 64r + 64) of every tile from f32 to bf16 into its own
//     shared memory and ships them to the peer CTA with a bulk shared-memory copy,
//     so the tile is read from HBM once and converted once;
//   * owns query heads [r*N, r*N + N), N = n_heads / 2: their bf16 Q (scale and
//     log2 e folded in), their S^T and O^T in its TMEM, their partials.
// Roles inside a CTA (9 warps: three per SM sub-partition at most, so a
// thread may hold up to 168 registers):
//   warps 0-3  softmax and epilogue: thread p owns TMEM lane p (tile position p);
//   warps 4-7  converters (f32 -> bf16 with 128-bit loads, 3 chunks in flight),
//              16 rows (two swizzle atoms) of the CTA's half-tile each;
//   warp 8     TMEM allocation and the single thread that issues the MMAs.
// The tile buffer is 9 chunks of [128 positions][64 columns] bf16 in the
// 128-byte-swizzled K-major layout: each chunk is an A operand of the QK
// product (positions x 64 columns of K) and, read MN-major, half an M block of
// the PV product (64 value columns x positions). A chunk is freed (for the next
// tile) as soon as both CTAs' MMAs are done with it, so conversion of tile t+1
// overlaps the softmax and PV of tile t.
//
// Softmax in the transposed layout: a head's scores lie across the 128 lanes,
// so the exact per-tile max would need a cross-lane reduction per head. The
// running reference max m of each head is instead kept lazily: it is set from
// the first tile of an item and only moved (with the rescale of l and of the
// head's O^T column) when a score exceeds it by more than 2^8. Any reference
// value gives the same partial after normalisation; bounding the exponent keeps
// every 2^(s - m) <= 256, so nothing overflows.
#include <cuda_bf16.h>

#include "internal.h"
#include "ptx.cuh"

namespace skv {
namespace {

constexpr int kDk = 576;
constexpr int kDv = 512;
constexpr int kTile = 128;               // positions per tile = MMA M
constexpr int kChunks = 9;               // 64-column chunks of a latent row (8 value + rope)
constexpr int kChunkBytes = kTile * 128; // 16 KB
constexpr int kSoftWarps = 4;
constexpr int kConvWarps = 4;
constexpr int kMmaWarp = kSoftWarps + kConvWarps;
constexpr int kThreads = (kMmaWarp + 1) * 32;
constexpr int kPF = 3;                   // converter chunks in flight
constexpr float kTau = 8.f;              // lazy-rescale threshold (log2 units)
constexpr int kRope = 8;                 // index of the rope chunk

// chunk processed at step ci of a tile: the rope chunk first (it is freed as
// soon as QK is done), then the value chunks in order
__device__ __forceinline__ int chunk_at(int ci) { return ci == 0 ? kRope : ci - 1; }

__host__ __device__ constexpr int tmem_cols_for(int N)
{
    return 5 * N <= 32 ? 32 : 5 * N <= 64 ? 64 : 5 * N <= 128 ? 128 : 5 * N <= 256 ? 256 : 512;
}

template <int N> struct Layout {
    static constexpr int KV = 0;                            // 9 x 16 KB tile chunks
    static constexpr int QCH = N * 128;                     // bytes of one Q chunk
    static constexpr int Q = KV + kChunks * kChunkBytes;    // 9 Q chunks
    static constexpr int PT = Q + kChunks * QCH;            // P^T: 2 sub-chunks of 64 positions
    static constexpr int BAR = PT + 2 * QCH;
    static constexpr int NBAR = 27;
    static constexpr int MISC = BAR + NBAR * 8;             // tmem base, abort flag
    static constexpr int MREF = (MISC + 16 + 15) / 16 * 16; // float m_ref[N]
    static constexpr int SCR = MREF + N * 4;                // float scratch[4][N]
    static constexpr int USED = SCR + kSoftWarps * N * 4;
    static constexpr int ALLOC = USED + 1024;
    static constexpr int TMEM_COLS = tmem_cols_for(N);
    static constexpr int S_COL = 0;
    static constexpr int O_COL = N;                         // O^T block j at O_COL + j*N
    static_assert(N % 16 == 0 && N >= 16 && N <= 48, "heads per CTA");
    static_assert(QCH % 1024 == 0 && Q % 1024 == 0 && PT % 1024 == 0, "swizzle atoms");
    static_assert(ALLOC <= 232448, "shared memory");
};

// barrier indices
constexpr int B_FULL = 0, B_EMPTY = 9, B_SFULL = 18, B_SFREE = 19, B_PFULL = 20, B_PFREE = 21,
              B_OREADY = 22, B_OFREE = 23, B_DRAIN = 24, B_QFULL = 25, B_QFREE = 26;

// byte offset of (row, byte) in a region of 128-byte rows with 128-byte swizzle
__device__ __forceinline__ uint32_t sw128(uint32_t row, uint32_t byte)
{
    return (row >> 3) * 1024 + (row & 7) * 128 + ((((byte >> 4) ^ row) & 7) << 4) + (byte & 15);
}

__device__ __forceinline__ uint32_t pack_bf16(float a, float b)
{
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t *>(&h);
}

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
    int b, s, p0, p1, ntiles;
};

__device__ __forceinline__ Item get_item(const ItemTable &it, int item)
{
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
    x.p1 = min(it.seq_lens[lo], x.p0 + it.chunk[lo]);
    x.ntiles = (x.p1 - x.p0 + kTile - 1) / kTile;
    return x;
}

// Sequence of (item, tile, chunk) units one converter walks through.
struct Cursor {
    int item, t, ci;
    Item x;
    bool done;
    __device__ __forceinline__ void start(const ItemTable &it, int first)
    {
        item = first;
        t = 0;
        ci = 0;
        done = item >= it.n_items;
        if (!done) x = get_item(it, item);
    }
    __device__ __forceinline__ void next(const ItemTable &it, int stride)
    {
        if (++ci == kChunks) {
            ci = 0;
            if (++t == x.ntiles) {
                t = 0;
                item += stride;
                done = item >= it.n_items;
                if (!done) x = get_item(it, item);
            }
        }
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

template <int N>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    mla_split_kernel(const __grid_constant__ MlaParams p)
{
    using LY = Layout<N>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *bar = reinterpret_cast<uint64_t *>(sm + LY::BAR);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + LY::MISC);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(sm + LY::MISC + 4);
    float *m_ref = reinterpret_cast<float *>(sm + LY::MREF);
    float *scr = reinterpret_cast<float *>(sm + LY::SCR);
    const uint32_t sm_base = smem_u32(sm);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank(), peer = rank ^ 1u;
    const int cluster = blockIdx.x >> 1, nclusters = gridDim.x >> 1;
    const ItemTable &it = p.items;
    const int hbase = (int)rank * N;
    const uint32_t abort_peer = map_to_rank(smem_u32((const void *)abort_flag), peer);
    volatile int never = 0;

    if (threadIdx.x == 0) {
        for (int c = 0; c < kChunks; ++c) {
            mbar_init(bar + B_FULL + c, kConvWarps);
            mbar_init(bar + B_EMPTY + c, 2);
        }
        mbar_init(bar + B_SFULL, 1);
        mbar_init(bar + B_SFREE, kSoftWarps);
        mbar_init(bar + B_PFULL, kSoftWarps);
        mbar_init(bar + B_PFREE, 1);
        mbar_init(bar + B_OREADY, 1);
        mbar_init(bar + B_OFREE, kSoftWarps);
        mbar_init(bar + B_DRAIN, 1);
        mbar_init(bar + B_QFULL, kConvWarps);
        mbar_init(bar + B_QFREE, 1);
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
        const uint32_t row0 = rank * 64 + cw * 16; // this warp's 16 rows of every tile
        uint32_t eph = 0;                         // per-chunk empty parity bits
        uint32_t qph = 0;                         // q_free parity
        bool ok = true;
        const bool no_copy = (p.flags & DA_FLAG_TEST_NO_TMA) != 0;
        float4 ld[kPF][4][2];
        Cursor ahead, cur;
        ahead.start(it, cluster);
        cur.start(it, cluster);
        auto issue = [&](const Cursor &u, float4 (&r)[4][2]) {
            const int c = chunk_at(u.ci);
            const float *base = p.cache + (size_t)u.x.b * p.batch_stride;
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const int task = lane + 32 * k, row = task >> 3, q8 = task & 7;
                const int pos = u.x.p0 + u.t * kTile + (int)row0 + row;
                if (pos < u.x.p1) {
                    const float4 *src = reinterpret_cast<const float4 *>(
                        base + (size_t)pos * p.pos_stride + c * 64 + q8 * 8);
                    r[k][0] = __ldg(src);
                    r[k][1] = __ldg(src + 1);
                } else {
                    r[k][0] = r[k][1] = make_float4(0.f, 0.f, 0.f, 0.f);
                }
            }
        };
#pragma unroll
        for (int k = 0; k < kPF - 1; ++k)
            if (!ahead.done) {
                issue(ahead, ld[k]);
                ahead.next(it, nclusters);
            }
        while (ok && !cur.done) {
#pragma unroll
            for (int u = 0; u < kPF; ++u) {
                if (!ok || cur.done) break;
                if (!ahead.done) {
                    issue(ahead, ld[(u + kPF - 1) % kPF]);
                    ahead.next(it, nclusters);
                }
                if (cur.t == 0 && cur.ci == 0) {
                    // a new item: this CTA's heads of q (scale and log2 e folded in),
                    // once the previous item's QK products are done with Q
                    if (!mbar_wait_bounded(bar + B_QFREE, qph ^ 1u, p.timeout_ns, abort_flag)) {
                        ok = false;
                        break;
                    }
                    qph ^= 1u;
                    const float *qb = p.q + ((size_t)cur.x.b * p.n_heads + hbase) * kDk;
                    for (int task = cw * 32 + lane; task < N * 72; task += kConvWarps * 32) {
                        const int h = task / 72, q8 = task % 72, c = q8 >> 3, j = q8 & 7;
                        const float4 a = __ldg(reinterpret_cast<const float4 *>(qb + h * kDk + q8 * 8));
                        const float4 b = __ldg(reinterpret_cast<const float4 *>(qb + h * kDk + q8 * 8 + 4));
                        const float sc = p.scale_log2;
                        uint4 v;
                        v.x = pack_bf16(a.x * sc, a.y * sc);
                        v.y = pack_bf16(a.z * sc, a.w * sc);
                        v.z = pack_bf16(b.x * sc, b.y * sc);
                        v.w = pack_bf16(b.z * sc, b.w * sc);
                        *reinterpret_cast<uint4 *>(sm + LY::Q + c * LY::QCH + sw128(h, j * 16)) = v;
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(bar + B_QFULL);
                }
                const int c = chunk_at(cur.ci);
                uint4 pk[4];
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const float4 a = ld[u][k][0], b = ld[u][k][1];
                    pk[k].x = pack_bf16(a.x, a.y);
                    pk[k].y = pack_bf16(a.z, a.w);
                    pk[k].z = pack_bf16(b.x, b.y);
                    pk[k].w = pack_bf16(b.z, b.w);
                }
                if (!mbar_wait_bounded(bar + B_EMPTY + c, ((eph >> c) & 1u) ^ 1u, p.timeout_ns,
                                       abort_flag)) {
                    ok = false;
                    break;
                }
                eph ^= 1u << c;
                if (!no_copy) {
                    uint8_t *chunk = sm + LY::KV + c * kChunkBytes;
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const int task = lane + 32 * k, row = task >> 3, q8 = task & 7;
                        *reinterpret_cast<uint4 *>(chunk + sw128(row0 + row, q8 * 16)) = pk[k];
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        const uint32_t src = sm_base + LY::KV + c * kChunkBytes + row0 * 128;
                        bulk_copy_to_cta(map_to_rank(src, peer), src, 2048,
                                         map_to_rank(smem_u32(bar + B_FULL + c), peer));
                        if (cw == 0) mbar_arrive_expect_tx(bar + B_FULL + c, 8 * 1024);
                        else mbar_arrive(bar + B_FULL + c);
                    }
                }
                cur.next(it, nclusters);
            }
        }
        if (!ok) raise_abort(abort_flag, abort_peer, p.status);
        // every commit (local and the peer's) that targets this CTA's empty
        // barriers has landed once each chunk has been released once more
        const uint64_t lim = *abort_flag ? 1000000ull : p.timeout_ns;
        for (int c = 0; c < kChunks; ++c)
            (void)mbar_wait_bounded(bar + B_EMPTY + c, ((eph >> c) & 1u) ^ 1u, lim, &never);
    } else if (warp == kMmaWarp) {
        // ============================ MMA issue (1 thread) ============================
        if (lane == 0) {
            constexpr uint32_t IDESC_QK = idesc_bf16_f32(kTile, N, 0, 0);
            constexpr uint32_t IDESC_PV = idesc_bf16_f32(kTile, N, 1, 0);
            uint32_t fph = 0, sph = 0, pph = 0, oph = 0, qph = 0;
            bool ok = true, first_item = true;
            for (int item = cluster; ok && item < it.n_items; item += nclusters) {
                const Item x = get_item(it, item);
                if (!mbar_wait_bounded(bar + B_QFULL, qph, p.timeout_ns, abort_flag)) {
                    ok = false;
                    break;
                }
                qph ^= 1u;
                for (int t = 0; ok && t < x.ntiles; ++t) {
                    // S^T = K_tile . Q^T (wait until the softmax has read the previous S^T)
                    if (!mbar_wait_bounded(bar + B_SFREE, sph ^ 1u, p.timeout_ns, abort_flag)) {
                        ok = false;
                        break;
                    }
                    sph ^= 1u;
                    for (int ci = 0; ci < kChunks; ++ci) {
                        const int c = chunk_at(ci);
                        if (!mbar_wait_bounded(bar + B_FULL + c, (fph >> c) & 1u, p.timeout_ns,
                                               abort_flag)) {
                            ok = false;
                            break;
                        }
                        fph ^= 1u << c;
                        tc_fence_after();
                        const uint32_t a0 = sm_base + LY::KV + c * kChunkBytes;
                        const uint32_t b0 = sm_base + LY::Q + c * LY::QCH;
#pragma unroll
                        for (int k = 0; k < 4; ++k)
                            tc_mma_bf16(tmem + LY::S_COL, smem_desc_sw128(a0 + k * 32, 16, 1024),
                                        smem_desc_sw128(b0 + k * 32, 16, 1024), IDESC_QK,
                                        (ci | k) != 0);
                        if (c == kRope) tc_commit_mc(bar + B_EMPTY + kRope, 3);
                    }
                    if (!ok) break;
                    tc_commit(bar + B_SFULL);
                    if (t == x.ntiles - 1) tc_commit(bar + B_QFREE);
                    // O^T += V^T . P^T once the softmax has written P^T
                    if (!mbar_wait_bounded(bar + B_PFULL, pph, p.timeout_ns, abort_flag)) {
                        ok = false;
                        break;
                    }
                    pph ^= 1u;
                    if (t == 0 && !first_item) {
                        // the epilogue of the previous item has read O^T
                        if (!mbar_wait_bounded(bar + B_OFREE, oph, p.timeout_ns, abort_flag)) {
                            ok = false;
                            break;
                        }
                        oph ^= 1u;
                    }
                    tc_fence_after();
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const uint32_t a0 = sm_base + LY::KV + (2 * j) * kChunkBytes;
#pragma unroll
                        for (int k = 0; k < 8; ++k) {
                            const uint32_t bk = sm_base + LY::PT + (k >> 2) * LY::QCH + (k & 3) * 32;
                            tc_mma_bf16(tmem + LY::O_COL + j * N,
                                        smem_desc_sw128(a0 + k * 2048, kChunkBytes, 1024),
                                        smem_desc_sw128(bk, 16, 1024), IDESC_PV,
                                        (t > 0 || k > 0) ? 1u : 0u);
                        }
                        tc_commit_mc(bar + B_EMPTY + 2 * j, 3);
                        tc_commit_mc(bar + B_EMPTY + 2 * j + 1, 3);
                    }
                    tc_commit(bar + B_PFREE);
                }
                if (!ok) break;
                tc_commit(bar + B_OREADY);
                first_item = false;
            }
            if (!ok) raise_abort(abort_flag, abort_peer, p.status);
            // no MMA may be in flight when TMEM is freed
            tc_commit(bar + B_DRAIN);
            (void)mbar_wait_bounded(bar + B_DRAIN, 0, p.timeout_ns, &never);
        }
        __syncwarp();
    } else {
        // ========================= softmax and epilogue (warps 0-3) ========================
        const int tid = threadIdx.x; // 0..127 = TMEM lane = tile position
        const uint32_t tl = tmem + ((uint32_t)(warp * 32) << 16);
        uint32_t sph = 0, pph = 0, oph = 0;
        for (int item = cluster; item < it.n_items; item += nclusters) {
            const Item x = get_item(it, item);
            float l[N];
#pragma unroll
            for (int h = 0; h < N; ++h) l[h] = 0.f;
            if (tid < N) m_ref[tid] = -INFINITY;
            named_bar_sync(2, 128);
            bool ab = false;
            for (int t = 0; t < x.ntiles; ++t) {
                bool okw = mbar_wait_bounded(bar + B_SFULL, sph, p.timeout_ns, abort_flag);
                if (bar_or(2, 128, !okw)) {
                    ab = true;
                    break;
                }
                sph ^= 1u;
                tc_fence_after();
                const int pos = x.p0 + t * kTile + tid;
                const bool valid = pos < x.p1;
                // pass 1: does any score outgrow its head's reference max?
                bool ex = false;
#pragma unroll
                for (int g = 0; g < N / 16; ++g) {
                    float sg[16];
                    tmem_ld16(tl + LY::S_COL + 16 * g, sg);
                    tmem_wait_ld();
#pragma unroll
                    for (int i = 0; i < 16; ++i) ex |= valid && sg[i] > m_ref[16 * g + i] + kTau;
                }
                okw = mbar_wait_bounded(bar + B_PFREE, pph ^ 1u, p.timeout_ns, abort_flag);
                if (bar_or(2, 128, !okw)) {
                    ab = true;
                    break;
                }
                pph ^= 1u;
                if (bar_or(2, 128, ex)) {
                    // move the reference max of the heads that outgrew it
#pragma unroll
                    for (int g = 0; g < N / 16; ++g) {
                        float sg[16];
                        tmem_ld16(tl + LY::S_COL + 16 * g, sg);
                        tmem_wait_ld();
#pragma unroll
                        for (int i = 0; i < 16; ++i) {
                            float v = valid ? sg[i] : -INFINITY;
#pragma unroll
                            for (int o = 16; o > 0; o >>= 1)
                                v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
                            if (lane == 0) scr[warp * N + 16 * g + i] = v;
                        }
                    }
                    named_bar_sync(2, 128);
#pragma unroll
                    for (int g = 0; g < N / 16; ++g) {
                        float alpha[16];
#pragma unroll
                        for (int i = 0; i < 16; ++i) {
                            const int h = 16 * g + i;
                            const float tm = fmaxf(fmaxf(scr[h], scr[N + h]),
                                                   fmaxf(scr[2 * N + h], scr[3 * N + h]));
                            const float mo = m_ref[h];
                            const float mn = tm > mo + kTau ? tm : mo;
                            alpha[i] = (mn == mo) ? 1.f : (mo == -INFINITY ? 0.f : ex2(mo - mn));
                            l[h] *= alpha[i];
                        }
                        if (t > 0) {
#pragma unroll
                            for (int j = 0; j < 4; ++j) {
                                float o[16];
                                tmem_ld16(tl + LY::O_COL + j * N + 16 * g, o);
                                tmem_wait_ld();
#pragma unroll
                                for (int i = 0; i < 16; ++i) o[i] *= alpha[i];
                                tmem_st16(tl + LY::O_COL + j * N + 16 * g, o);
                            }
                            tmem_wait_st();
                        }
                    }
                    named_bar_sync(2, 128); // every thread has used the old m_ref
                    if (tid < N) {
                        const float tm = fmaxf(fmaxf(scr[tid], scr[N + tid]),
                                               fmaxf(scr[2 * N + tid], scr[3 * N + tid]));
                        if (tm > m_ref[tid] + kTau) m_ref[tid] = tm;
                    }
                    named_bar_sync(2, 128);
                }
                // pass 2: P^T[h][pos] = 2^(s - m_ref) in bf16, K-major (positions contiguous)
                uint8_t *pt = sm + LY::PT + (tid >> 6) * LY::QCH;
                const uint32_t pb = (uint32_t)(tid & 63) * 2;
#pragma unroll
                for (int g = 0; g < N / 16; ++g) {
                    float sg[16];
                    tmem_ld16(tl + LY::S_COL + 16 * g, sg);
                    tmem_wait_ld();
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        const int h = 16 * g + i;
                        const float pv = valid ? ex2(sg[i] - m_ref[h]) : 0.f;
                        l[h] += pv;
                        *reinterpret_cast<__nv_bfloat16 *>(pt + sw128(h, pb)) =
                            __float2bfloat16_rn(pv);
                    }
                }
                tc_fence_before();
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(bar + B_SFREE);
                    mbar_arrive(bar + B_PFULL);
                }
            }
            if (ab) break;
            // ------------------------------- epilogue -------------------------------
            bool okw = mbar_wait_bounded(bar + B_OREADY, oph, p.timeout_ns, abort_flag);
            if (bar_or(2, 128, !okw)) break;
            oph ^= 1u;
            tc_fence_after();
#pragma unroll
            for (int h = 0; h < N; ++h) {
                float v = l[h];
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
                if (lane == 0) scr[warp * N + h] = v;
            }
            const size_t slot = (size_t)it.split_base[x.b] + x.s;
            const size_t row0 = slot * p.n_heads + hbase;
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
            named_bar_sync(2, 128);
            if (tid < N) {
                const float L = scr[tid] + scr[N + tid] + scr[2 * N + tid] + scr[3 * N + tid];
                p.ml[row0 + tid] = make_float2(L > 0.f ? m_ref[tid] * kLn2 : kNeutralM, L);
            }
            named_bar_sync(2, 128);
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
    if (threadIdx.x == 0) griddep_launch_dependents();
}

} // namespace

bool mla_supported_heads(int n_heads) { return n_heads == 32 || n_heads == 64 || n_heads == 96; }

int mla_smem_bytes(int n_heads)
{
    switch (n_heads) {
    case 32: return Layout<16>::ALLOC;
    case 64: return Layout<32>::ALLOC;
    case 96: return Layout<48>::ALLOC;
    default: return 0;
    }
}

template <int N> static cudaError_t launch_n(int grid, cudaStream_t st, const MlaParams &p)
{
    auto *fn = mla_split_kernel<N>;
    cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         Layout<N>::ALLOC);
    if (e != cudaSuccess) return e;
    fn<<<grid, kThreads, Layout<N>::ALLOC, st>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_mla_split(int grid, cudaStream_t st, const MlaParams &p)
{
    switch (p.n_heads) {
    case 32: return launch_n<16>(grid, st, p);
    case 64: return launch_n<32>(grid, st, p);
    case 96: return launch_n<48>(grid, st, p);
    default: return cudaErrorInvalidValue;
    }
}

} // namespace skv
