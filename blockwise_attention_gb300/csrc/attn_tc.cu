// Tensor-core attention kernel for sm_103a (bf16 Q/K/V, head dim 64 or 128).
//
// Persistent CTAs (one per SM) take work items = (query tile of 128 rows,
// batch item, head), claimed one at a time from a launch-wide counter in
// heaviest-first order (or dealt round-robin when no counter is given).  For each item the query tile stays resident in shared
// memory while the key tiles of its walk arrive in ring order; every tile is
// folded into a running (row max, denominator, weighted sum) that is rescaled
// to the new maximum, never added or averaged (brunomaga "Improving numerical
// stability"; llm-systems "Circulate K/V blocks with Ring").
//
// Roles (256 threads):
//   warp 0      TMA producer: Q tile, then K and V tiles into two stage rings
//               (128B-swizzled boxes of 64 columns x 128 rows); K of tile j is
//               issued before V of tile j - 1.
//   warp 1      owns TMEM (512 columns) and issues tcgen05.mma from one thread:
//               S = Q K^T (A, B from shared memory, fp32 accumulate in TMEM),
//               O += P V (A = P from TMEM, B = V from shared memory).
//   warps 4..7  softmax: thread t owns query row t (TMEM lane t).  Reads S,
//               applies scale and exclusions, updates (m, l), writes P (bf16)
//               to TMEM, rescales O when the row maximum grows by more than
//               2^8, and at the end normalises O and stores out / lse.
//   warps 2..3  idle.
// S has three buffers and PV runs two tiles behind QK: QK(j+1) and QK(j+2)
// are computed while the softmax works on tile j, so three tiles are in
// flight between the tensor pipe and the softmax.  P(j) (bf16, 64 columns) is
// written over the S buffer it was computed from; QK(j+3), the next writer of
// that buffer, is issued after PV(j), and the tensor pipe executes in issue
// order.  K stages are released when their QK completes, V stages when their
// PV completes.
//
// TMEM columns: S0 [0,128) S1 [128,256) S2 [256,384) O [384,384+D).
//
// The producer passes each claimed item (index, key-tile count) to the MMA
// thread and the softmax warps through a two-slot ring (ITEM_FULL / ITEM_EMPTY).
//
// Every mbarrier wait is bounded (globaltimer); on expiry the CTA records
// BA_ERR_TIMEOUT in the error word, drains its outstanding copies and MMAs
// (with bounded waits), frees TMEM and returns.
#include <cuda.h>
#include <cuda_bf16.h>

#include "epilogue.cuh"
#include "tc_ptx.cuh"

namespace ba {
namespace {

template <int D>
struct Cfg {
    static constexpr int NBOX = D / 64;            // 64-column boxes per tile
    static constexpr int BOX_BYTES = TILE * 128;   // 128 rows x 128 bytes
    static constexpr int TILE_BYTES = NBOX * BOX_BYTES;
    // One K stage and one V stage per S buffer: tile j uses K stage, V stage
    // and S buffer j % 3, so the S_FULL commit of QK(j) also frees K stage
    // j % 3 and the PV_DONE commit of PV(j) frees V stage j % 3.
    static constexpr int NSB = 3;                  // S buffers in TMEM
    static constexpr int KS = NSB;                 // K stages
    static constexpr int VS = NSB;                 // V stages
    static constexpr int TIR = 16;                 // key-tile description ring (power of two)
    static constexpr int Q_OFF = 0;
    static constexpr int K_OFF = TILE_BYTES;
    static constexpr int V_OFF = K_OFF + KS * TILE_BYTES;
    static constexpr int BAR_OFF = V_OFF + VS * TILE_BYTES;
    enum {
        B_QFULL = 0,
        B_QEMPTY,
        B_KFULL,
        B_VFULL = B_KFULL + KS,
        B_SFULL = B_VFULL + VS,     // QK(j) complete: S ready, K stage j % 3 free
        B_PFULL = B_SFULL + NSB,
        B_PVDONE = B_PFULL + NSB,   // PV(j) complete: V stage j % 3 free, O may be rescaled
        B_OFULL = B_PVDONE + NSB,
        B_OEMPTY,
        B_DRAIN,
        B_ITEMFULL,
        B_ITEMEMPTY = B_ITEMFULL + 2,
        NBAR = B_ITEMEMPTY + 2
    };
    // [0] tmem base, [1] abort, [2..3] item key tiles, [4..5] item index (by item parity)
    static constexpr int MISC_OFF = BAR_OFF + NBAR * 8;
    // TIR x {global position, len | class << 16, tile sequence number + 1, unused}
    static constexpr int TI_OFF = MISC_OFF + 32;
    static constexpr int SMEM_BYTES = TI_OFF + TIR * 16 + 1024;  // + slack to align the base to 1 KB
    static constexpr uint32_t S_COL = 0;     // S buffer b at S_COL + 128 b; P over its first 64 columns
    static constexpr uint32_t O_COL = 384;
    static constexpr uint32_t TMEM_COLS = 512;
    // Instruction descriptors (kind::f16): D fp32 (bits 4-5 = 1), A and B
    // bf16 (bits 7-9, 10-12 = 1), B major bit 16 (0 = K-major, 1 = MN-major),
    // N >> 3 at bits 17-22, M >> 4 at bits 24-28.
    static constexpr uint32_t IDESC_QK =
        (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(TILE >> 3) << 17) | ((uint32_t)(TILE >> 4) << 24);
    static constexpr uint32_t IDESC_PV = (1u << 4) | (1u << 7) | (1u << 10) | (1u << 16) |
                                         ((uint32_t)(D >> 3) << 17) | ((uint32_t)(TILE >> 4) << 24);
};

// 32 bytes of an exclusion mask (1 = excluded) starting at p, of which the
// first n are meaningful, applied to s[0..31].
__device__ __forceinline__ void mask_bytes(const uint8_t *p, int n, float *s) {
    uint32_t w[8];
    if (n >= 32 && (reinterpret_cast<uintptr_t>(p) & 15) == 0) {
        const uint4 a = __ldg(reinterpret_cast<const uint4 *>(p));
        const uint4 b = __ldg(reinterpret_cast<const uint4 *>(p + 16));
        w[0] = a.x; w[1] = a.y; w[2] = a.z; w[3] = a.w;
        w[4] = b.x; w[5] = b.y; w[6] = b.z; w[7] = b.w;
    } else {
#pragma unroll
        for (int k = 0; k < 8; ++k) w[k] = 0;
#pragma unroll
        for (int i = 0; i < 32; ++i)
            if (i < n) w[i >> 2] |= (uint32_t)__ldg(p + i) << (8 * (i & 3));
    }
#pragma unroll
    for (int i = 0; i < 32; ++i)
        if ((w[i >> 2] >> (8 * (i & 3))) & 0xffu) s[i] = -INFINITY;
}

// Exclusions of keys [c0, c0 + 32) of key tile kt for the query at global
// position qpos: past the tile end, causal future, key padding, attn_mask.
__device__ __forceinline__ void mask_chunk(const Geom &g, int b, long long qpos, bool row_valid, const KTile &kt,
                                           int c0, float *s) {
    const long long diag = qpos - kt.pos0;   // key j lies in the future when j > diag
#pragma unroll
    for (int i = 0; i < 32; ++i) {
        const int j = c0 + i;
        if (j >= kt.len || (g.causal && j > diag)) s[i] = -INFINITY;
    }
    const int n = kt.len - c0;
    if (!row_valid || n <= 0) return;
    if (g.kpm) mask_bytes(g.kpm + b * g.kpm_ld + kt.pos0 + c0, n, s);
    if (g.am) mask_bytes(g.am + qpos * g.am_ld + kt.pos0 + c0, n, s);
}

// ----------------------------------------------------------------------------
// Kernel
// ----------------------------------------------------------------------------

template <int D>
__global__ void __launch_bounds__(256, 1)
    attn_tc_kernel(const AttnArgs a, const __grid_constant__ CUtensorMap tq,
                   const __grid_constant__ CUtensorMap tk, const __grid_constant__ CUtensorMap tv) {
    using C = Cfg<D>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_base = smem_u32(smem_raw);
    const uint32_t base = (raw_base + 1023u) & ~1023u;
    uint8_t *gbase = smem_raw + (base - raw_base);
    const uint32_t sQ = base + C::Q_OFF, sK = base + C::K_OFF, sV = base + C::V_OFF;
    const uint32_t bars = base + C::BAR_OFF;
    auto bar = [&](int i) { return bars + 8u * (uint32_t)i; };
    volatile uint32_t *misc = reinterpret_cast<volatile uint32_t *>(gbase + C::MISC_OFF);
    volatile uint32_t *tinfo = reinterpret_cast<volatile uint32_t *>(gbase + C::TI_OFF);
    const uint32_t sTI = base + C::TI_OFF;
    volatile int *abort = reinterpret_cast<volatile int *>(gbase + C::MISC_OFF + 4);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const Geom &g = a.g;
    const uint64_t lim = a.wait_limit_ns;

    if (threadIdx.x == 0) {
        mbar_init(bar(C::B_QFULL), 1);
        mbar_init(bar(C::B_QEMPTY), 1);
        for (int i = 0; i < C::KS; ++i) mbar_init(bar(C::B_KFULL + i), 1);
        for (int i = 0; i < C::VS; ++i) mbar_init(bar(C::B_VFULL + i), 1);
        for (int i = 0; i < C::NSB; ++i) {
            mbar_init(bar(C::B_SFULL + i), 1);
            mbar_init(bar(C::B_PFULL + i), 128);
            mbar_init(bar(C::B_PVDONE + i), 1);
        }
        mbar_init(bar(C::B_OFULL), 1);
        mbar_init(bar(C::B_OEMPTY), 128);
        mbar_init(bar(C::B_DRAIN), 1);
        for (int i = 0; i < 2; ++i) {
            mbar_init(bar(C::B_ITEMFULL + i), 1);
            mbar_init(bar(C::B_ITEMEMPTY + i), 1 + 4);   // MMA warp + one lane per softmax warp
        }
        for (int i = 0; i < C::TIR; ++i) tinfo[4 * i + 2] = 0xffffffffu;   // no tile yet
        misc[1] = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         base + C::MISC_OFF),
                     "r"(C::TMEM_COLS)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    if (warp == 0 && lane == 0) {
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tq)) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tk)) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tv)) : "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = misc[0];

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            uint32_t kfill = 0, vfill = 0, qfills = 0, it_local = 0;
            bool ok = true;
            // Items are claimed from the launch's counter in index order (heaviest
            // first under causal masking), so an SM takes its next item when it runs
            // out of work; without a counter they are dealt round-robin by CTA.
            int w = a.sched ? (int)atomicAdd(a.sched, 1u) : (int)blockIdx.x;
            for (;; ++it_local) {
                // Publish (item, key tiles) in slot it & 1 for the MMA thread and the
                // softmax warps; the slot's previous item (it - 2) has been read by all.
                const uint32_t sl = it_local & 1;
                if (it_local >= 2 &&
                    !mbar_wait(bar(C::B_ITEMEMPTY + sl), ((it_local >> 1) - 1) & 1, abort, a.err, lim)) {
                    ok = false;
                    break;
                }
                if (w >= g.n_items) {
                    misc[4 + sl] = 0xffffffffu;   // end of work
                    mbar_arrive(bar(C::B_ITEMFULL + sl));
                    break;
                }
                const QTile qt = work_item(g, w);
                misc[4 + sl] = (uint32_t)w;
                misc[2 + sl] = (uint32_t)kwalk_count(g, qt);
                mbar_arrive(bar(C::B_ITEMFULL + sl));
                if (it_local > 0 && !mbar_wait(bar(C::B_QEMPTY), (it_local - 1) & 1, abort, a.err, lim)) {
                    ok = false;
                    break;
                }
                mbar_arrive_expect_tx(bar(C::B_QFULL), C::TILE_BYTES);
                for (int bx = 0; bx < C::NBOX; ++bx)
                    tma_load_4d(sQ + bx * C::BOX_BYTES, &tq, bx * 64, qt.row0, qt.h, qt.b, bar(C::B_QFULL));
                ++qfills;
                KWalk wk;
                kwalk_begin(g, qt, wk);
                KTile kt;
                int prev_row = -1;   // k/v row of the tile whose V is still to be loaded
                for (;;) {
                    const bool more = kwalk_next(g, qt, wk, kt);
                    if (more) {
                        const uint32_t st = kfill % C::KS, use = kfill / C::KS;
                        if (use > 0 && !mbar_wait(bar(C::B_SFULL + st), (use - 1) & 1, abort, a.err, lim)) {
                            ok = false;
                            break;
                        }
                        // Describe tile kfill for the softmax warps in slot kfill % TIR.  QK of
                        // tile kfill - 3 has completed (the wait above), so the softmax has
                        // finished tile kfill - 6 (QK(j) is issued after PV(j - 3)) and has
                        // read every description older than that, including this slot's last.
                        {
                            const uint32_t e = (kfill % C::TIR) * 4;
                            tinfo[e] = (uint32_t)kt.pos0;
                            tinfo[e + 1] = (uint32_t)kt.len | ((uint32_t)kt.cls << 16);
                            st_release_shared(sTI + e * 4 + 8, kfill + 1);
                        }
                        mbar_arrive_expect_tx(bar(C::B_KFULL + st), C::TILE_BYTES);
                        for (int bx = 0; bx < C::NBOX; ++bx)
                            tma_load_4d(sK + st * C::TILE_BYTES + bx * C::BOX_BYTES, &tk, bx * 64, kt.row0, qt.h,
                                        qt.b, bar(C::B_KFULL + st));
                        ++kfill;
                    }
                    if (prev_row >= 0) {
                        const uint32_t st = vfill % C::VS, use = vfill / C::VS;
                        if (use > 0 && !mbar_wait(bar(C::B_PVDONE + st), (use - 1) & 1, abort, a.err, lim)) {
                            ok = false;
                            break;
                        }
                        mbar_arrive_expect_tx(bar(C::B_VFULL + st), C::TILE_BYTES);
                        for (int bx = 0; bx < C::NBOX; ++bx)
                            tma_load_4d(sV + st * C::TILE_BYTES + bx * C::BOX_BYTES, &tv, bx * 64, prev_row, qt.h,
                                        qt.b, bar(C::B_VFULL + st));
                        ++vfill;
                    }
                    if (!more) break;
                    prev_row = kt.row0;
                }
                if (!ok) break;
                w = a.sched ? (int)atomicAdd(a.sched, 1u) : w + (int)gridDim.x;
            }
            if (!ok) {
                // Let the copies already issued land before the CTA exits.
                volatile int never = 0;
                const uint64_t lim2 = 200000000ull;
                if (qfills > 0) mbar_wait(bar(C::B_QFULL), (qfills - 1) & 1, &never, nullptr, lim2);
                for (uint32_t i = 0; i < (uint32_t)C::KS && i < kfill; ++i) {
                    const uint32_t last = kfill - 1 - i;
                    mbar_wait(bar(C::B_KFULL + last % C::KS), (last / C::KS) & 1, &never, nullptr, lim2);
                }
                for (uint32_t i = 0; i < (uint32_t)C::VS && i < vfill; ++i) {
                    const uint32_t last = vfill - 1 - i;
                    mbar_wait(bar(C::B_VFULL + last % C::VS), (last / C::VS) & 1, &never, nullptr, lim2);
                }
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        // Per key tile j: QK(j) -> S[j % 3] once K(j) has landed, and PV(j - 2)
        // once the softmax has written P(j - 2) and V(j - 2) has landed.  QK(j)
        // overwrites the buffer that held P(j - 3), which PV(j - 3), issued just
        // before, has read: the tensor pipe executes in issue order, so no
        // separate "S free" barrier is needed.
        // The whole warp runs this loop converged (waits, counters, descriptors);
        // each MMA and commit is issued by one elected lane.
        {
            uint32_t it_local = 0;
            uint32_t qb = 0, qph = 0;   // buffer / stage index and phase of the next QK
            uint32_t pb = 0, pph = 0;   // buffer / stage index and phase of the next PV
            bool ok = true;
            const uint64_t qdesc0 = sdesc(sQ, 16, 1024);            // K-major, 128B swizzle
            const uint64_t kdesc0 = sdesc(sK, 16, 1024);
            const uint64_t vdesc0 = sdesc(sV, C::BOX_BYTES, 1024);   // MN-major
            // descriptor start-address fields advance by bytes / 16
            constexpr uint32_t STAGE16 = C::TILE_BYTES >> 4;
            auto qk = [&]() -> bool {
                if (!warp_wait(bar(C::B_KFULL + qb), qph, abort, a.err, lim)) return false;
                const uint64_t kd = kdesc0 + (uint64_t)(qb * STAGE16);
                const uint32_t sd = tmem + C::S_COL + qb * 128;
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint64_t off = (uint64_t)(((kk >> 2) * C::BOX_BYTES + (kk & 3) * 32) >> 4);
                    mma_ss_one(sd, qdesc0 + off, kd + off, C::IDESC_QK, kk > 0 ? 1u : 0u);
                }
                mma_commit_one(bar(C::B_SFULL + qb));
                qb = qb == C::NSB - 1 ? 0 : qb + 1;
                qph ^= qb == 0;
                return true;
            };
            auto pv = [&](bool first) -> bool {
                if (!warp_wait(bar(C::B_PFULL + pb), pph, abort, a.err, lim)) return false;
                if (!warp_wait(bar(C::B_VFULL + pb), pph, abort, a.err, lim)) return false;
                tc_fence_after();   // P was written by the softmax warps' tcgen05.st
                const uint64_t vd = vdesc0 + (uint64_t)(pb * STAGE16);
                const uint32_t pa = tmem + C::S_COL + pb * 128;
#pragma unroll
                for (int kk = 0; kk < TILE / 16; ++kk)
                    mma_ts_one(tmem + C::O_COL, pa + kk * 8, vd + (uint64_t)((kk * 2048) >> 4), C::IDESC_PV,
                               (first && kk == 0) ? 0u : 1u);
                mma_commit_one(bar(C::B_PVDONE + pb));
                pb = pb == C::NSB - 1 ? 0 : pb + 1;
                pph ^= pb == 0;
                return true;
            };
            for (;; ++it_local) {
                const uint32_t sl = it_local & 1;
                if (!warp_wait(bar(C::B_ITEMFULL + sl), (it_local >> 1) & 1, abort, a.err, lim)) {
                    ok = false;
                    break;
                }
                const uint32_t item = misc[4 + sl], n = misc[2 + sl];
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(C::B_ITEMEMPTY + sl));
                if (item == 0xffffffffu) break;
                if (!warp_wait(bar(C::B_QFULL), it_local & 1, abort, a.err, lim)) {
                    ok = false;
                    break;
                }
                // QK(0), QK(1); Q_EMPTY is committed right after the item's last QK.
                if (n == 0) mma_commit_one(bar(C::B_QEMPTY));
                if (n >= 1 && !(ok = qk())) break;
                if (n == 1) mma_commit_one(bar(C::B_QEMPTY));
                if (n >= 2 && !(ok = qk())) break;
                if (n == 2) mma_commit_one(bar(C::B_QEMPTY));
                // O of the previous item must have been read out before this item's
                // first PV writes O (and before O_FULL): waited once per item, so
                // the O_FULL / O_EMPTY phases never run two ahead of their waiters.
                if (it_local > 0 && !(ok = warp_wait(bar(C::B_OEMPTY), (it_local - 1) & 1, abort, a.err, lim)))
                    break;
                for (uint32_t t = 2; t < n; ++t) {
                    if (!(ok = qk())) break;
                    if (t + 1 == n) mma_commit_one(bar(C::B_QEMPTY));
                    if (!(ok = pv(t == 2))) break;
                }
                if (!ok) break;
                if (n >= 2 && !(ok = pv(n == 2))) break;
                if (n >= 1 && !(ok = pv(n == 1))) break;
                mma_commit_one(bar(C::B_OFULL));
            }
            if (!ok) {
                // Wait for the MMAs already issued before TMEM is released.
                volatile int never = 0;
                mma_commit_one(bar(C::B_DRAIN));
                warp_wait(bar(C::B_DRAIN), 0, &never, nullptr, 200000000ull);
            }
        }
        __syncwarp();
    } else if (warp >= 4) {
        // ------------------------------------------------------------ softmax / epilogue
        const int row = (warp & 3) * 32 + lane;
        const uint32_t lane_addr = ((uint32_t)((warp & 3) * 32) << 16);
        const float sl2 = a.scale_log2;
        uint32_t it_local = 0;
        uint32_t sb = 0, sph = 0;   // S buffer and phase of the next tile
        uint32_t pvb = 0, pvph = 0; // S buffer and phase of the previous tile (valid once n > 0)
        uint32_t tcnt = 0;          // key tiles described so far (ring position)
        bool ok = true;
        for (;; ++it_local) {
            const uint32_t sl = it_local & 1;
            if (!warp_wait(bar(C::B_ITEMFULL + sl), (it_local >> 1) & 1, abort, a.err, lim)) {
                ok = false;
                break;
            }
            const uint32_t item = misc[4 + sl], n_tiles = misc[2 + sl];
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(C::B_ITEMEMPTY + sl));
            if (item == 0xffffffffu) break;
            const QTile qt = work_item(g, (int)item);
            const long long qpos = qt.pos0 + row;
            float m_ref = -INFINITY, l = 0.f;
            int n = 0;
            for (uint32_t j = 0; j < n_tiles; ++j) {
                if (!warp_wait(bar(C::B_SFULL + sb), sph, abort, a.err, lim)) {
                    ok = false;
                    break;
                }
                // The producer walked the tiles; take this one's position, length and
                // class (written before K of the tile was loaded, so normally present).
                KTile kt;
                {
                    const uint32_t e = (tcnt % C::TIR) * 4;
                    if (!warp_wait_seq(sTI + e * 4 + 8, tcnt + 1, abort, a.err, lim)) {
                        ok = false;
                        break;
                    }
                    const uint32_t dx = tinfo[e], dy = tinfo[e + 1];
                    ++tcnt;
                    kt.pos0 = (long long)dx;
                    kt.len = (int)(dy & 0xffffu);
                    kt.cls = (int)(dy >> 16);
                }
                tc_fence_after();
                float s[TILE];
                {
                    uint32_t r[TILE];
#pragma unroll
                    for (int c = 0; c < TILE / 32; ++c)
                        tmem_ld32(tmem + lane_addr + C::S_COL + sb * 128 + c * 32,
                                  *reinterpret_cast<uint32_t(*)[32]>(&r[c * 32]));
                    tmem_wait_ld();
#pragma unroll
                    for (int j = 0; j < TILE; ++j) s[j] = __uint_as_float(r[j]);
                }

                if (kt.cls == BA_TILE_PARTIAL || kt.len < TILE) {
                    const bool row_valid = row < qt.len;   // rows past the tile end are never stored
#pragma unroll
                    for (int c = 0; c < TILE / 32; ++c) mask_chunk(g, qt.b, qpos, row_valid, kt, c * 32, &s[c * 32]);
                }
                // p = 2^(s * scale * log2(e) - m) with m the running reference maximum,
                // computed before this tile's maximum is known: the lazy rule keeps m
                // unless the tile's maximum exceeds it by more than 2^8, so the tile
                // maximum (ALU pipe) and the exponentials (MUFU / FMA pipes) run side by
                // side, and only a row whose maximum did move redoes its exponentials.
                // Arguments two lanes at a time, sums in four two-lane accumulators.
                float sc[8];
                uint32_t pk[TILE / 2];
                auto exp_tile = [&](float m_use) {
#pragma unroll
                    for (int k = 0; k < 8; ++k) sc[k] = 0.f;
#pragma unroll
                    for (int j = 0; j < TILE / 2; ++j) {
                        float x0, x1;
                        ffma2_bc(s[2 * j], s[2 * j + 1], sl2, -m_use, x0, x1);
                        const float p0 = fast_exp2(x0);
                        const float p1 = fast_exp2(x1);
                        fadd2_acc(sc[2 * (j & 3)], sc[2 * (j & 3) + 1], p0, p1);
                        pk[j] = pack_bf16(p0, p1);
                    }
                };
                exp_tile(m_ref == -INFINITY ? 0.f : m_ref);
                // row maximum: 8 independent chains of three-input maxima, then a tree
                float mc[8];
#pragma unroll
                for (int k = 0; k < 8; ++k) mc[k] = fmaxf(s[k], s[8 + k]);
#pragma unroll
                for (int j = 16; j < TILE; j += 16) {
#pragma unroll
                    for (int k = 0; k < 8; ++k) mc[k] = fmax3(mc[k], s[j + k], s[j + 8 + k]);
                }
                const float mx = fmaxf(fmax3(mc[0], mc[1], mc[2]), fmax3(fmax3(mc[3], mc[4], mc[5]), mc[6], mc[7]));
                const float m_new = fmaxf(m_ref, mx * sl2);
                const bool resc = m_new > m_ref + 8.0f;   // true when m_ref = -inf and m_new finite
                float alpha = 1.f;
                if (__any_sync(0xffffffffu, resc)) {
                    if (resc) {
                        alpha = fast_exp2(m_ref - m_new);
                        m_ref = m_new;
                    }
                    exp_tile(m_ref == -INFINITY ? 0.f : m_ref);   // rows that kept m repeat the same values
                }
                const float sum = ((sc[0] + sc[1]) + (sc[2] + sc[3])) + ((sc[4] + sc[5]) + (sc[6] + sc[7]));
                l = l * alpha + sum;

                // P over the first 64 columns of the S buffer just read
#pragma unroll
                for (int c = 0; c < TILE / 64; ++c)
                    tmem_st32(tmem + lane_addr + C::S_COL + sb * 128 + c * 32,
                              *reinterpret_cast<const uint32_t(*)[32]>(&pk[c * 32]));
                if (__any_sync(0xffffffffu, resc) && n > 0) {
                    // O may be rescaled once PV of the previous tile has completed
                    if (!warp_wait(bar(C::B_PVDONE + pvb), pvph, abort, a.err, lim)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
#pragma unroll
                    for (int c = 0; c < D / 32; ++c) {
                        uint32_t r[32];
                        tmem_ld32(tmem + lane_addr + C::O_COL + c * 32, r);
                        tmem_wait_ld();
#pragma unroll
                        for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * alpha);
                        tmem_st32(tmem + lane_addr + C::O_COL + c * 32, r);
                    }
                }
                tmem_wait_st();
                tc_fence_before();
                mbar_arrive(bar(C::B_PFULL + sb));
                pvb = sb;
                pvph = sph;
                sb = sb == C::NSB - 1 ? 0 : sb + 1;
                sph ^= sb == 0;
                ++n;
            }
            if (!ok) break;
            // epilogue
            if (!warp_wait(bar(C::B_OFULL), it_local & 1, abort, a.err, lim)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const bool valid = row < qt.len;
            const long long row_flat = ((long long)qt.b * g.H + qt.h) * a.rows + qt.row0 + row;
            const float acc_l = (a.acc_lse != nullptr && valid) ? a.acc_lse[row_flat] : -INFINITY;
            const RowFinal f = row_final(m_ref, n > 0 ? l : 0.f, acc_l);
#pragma unroll
            for (int c = 0; c < D / 32; ++c) {
                uint32_t r[32];
                float o[32];
                if (n > 0) {
                    tmem_ld32(tmem + lane_addr + C::O_COL + c * 32, r);
                    tmem_wait_ld();
#pragma unroll
                    for (int i = 0; i < 32; ++i) o[i] = __uint_as_float(r[i]);
                } else {
#pragma unroll
                    for (int i = 0; i < 32; ++i) o[i] = 0.f;
                }
                if (valid) store_row_chunk(a, row_flat, c * 32, o, 32, f);
            }
            if (valid) a.lse[row_flat] = f.lse;
            tc_fence_before();
            mbar_arrive(bar(C::B_OEMPTY));
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) {
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(C::TMEM_COLS)
                     : "memory");
    }
}

template <int D>
int launch_d(const AttnArgs &a, const TmaMaps &m, int num_sms, cudaStream_t s) {
    using C = Cfg<D>;
    static_assert(C::SMEM_BYTES <= 232448, "shared memory budget");
    cudaError_t e = cudaFuncSetAttribute(attn_tc_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         C::SMEM_BYTES);
    if (e != cudaSuccess) return BA_ERR_CUDA;
    int grid = a.g.n_items < num_sms ? a.g.n_items : num_sms;
    attn_tc_kernel<D><<<grid, 256, C::SMEM_BYTES, s>>>(a, m.q, m.k, m.v);
    return cudaGetLastError() == cudaSuccess ? BA_OK : BA_ERR_CUDA;
}

}  // namespace

bool tc_supported(int dtype, int d) { return dtype == BA_BF16 && (d == 64 || d == 128); }

size_t tc_smem_bytes(int d) { return d == 128 ? Cfg<128>::SMEM_BYTES : Cfg<64>::SMEM_BYTES; }

int launch_attn_tc(const AttnArgs &a, const TmaMaps &m, int num_sms, cudaStream_t s) {
    if (a.g.n_items == 0) return BA_OK;
    if (a.g.d == 128) return launch_d<128>(a, m, num_sms, s);
    if (a.g.d == 64) return launch_d<64>(a, m, num_sms, s);
    return BA_ERR_SHAPE;
}

}  // namespace ba
