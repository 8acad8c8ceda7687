// Tensor-core attention kernel for sm_103a (bf16 Q/K/V, head dim 64 or 128).
//
// Persistent CTAs (one per SM) take work items = (pair of adjacent query tiles
// of 128 rows, batch item, head), claimed one at a time from a launch-wide
// counter in heaviest-first order (or dealt round-robin when no counter is
// given).  The two query tiles stay resident in shared memory and share every
// key / value tile of their walk, which arrives in ring order; each tile is
// folded into a running (row max, denominator, weighted sum) per row that is
// rescaled to the new maximum, never added or averaged (brunomaga "Improving
// numerical stability"; llm-systems "Circulate K/V blocks with Ring").
//
// Roles (320 threads, ten warps):
//   warp 0      TMA producer: both Q tiles, then K and V tiles into two stage
//               rings (128B-swizzled boxes of 64 columns x 128 rows); K of tile
//               j is issued before V of tile j - 1.  It also claims the items
//               and describes every key tile for the softmax warps.
//   warp 1      owns TMEM (512 columns) and issues tcgen05.mma, one elected
//               lane per instruction: S_x = Q_x K^T (A, B from shared memory,
//               fp32 accumulate in TMEM) and O_x += P_x V (A = P_x from TMEM).
//   warps 2..5  softmax group 0 (query tile 0), warps 6..9 softmax group 1
//               (query tile 1): thread t of a group owns row t of its tile
//               (TMEM lane t; warp w reaches lanes 32 (w % 4) .. + 31).  Reads
//               S_x, applies scale and exclusions, takes the row maximum,
//               updates (m, l), writes P_x (bf16) over S_x, rescales O_x when the
//               row maximum grows by more than 2^8, and at the end normalises O_x
//               and stores out / lse.  Ten warps leave 168 registers a thread:
//               the 128 scores of a row stay in registers, the probabilities go
//               to TMEM 32 keys at a time.
// Ping-pong: per key tile j the MMA warp issues PV_0(j), QK_0(j+1), PV_1(j),
// QK_1(j+1).  While group 0 works on S_0(j+1) the tensor pipe runs the
// products of group 1, and the other way round, so the softmax of one group
// hides under the products of the other, and each K / V tile brought in from
// L2 serves 256 query rows.  P_x(j) is written over the S_x columns it was
// computed from; QK_x(j+1), the next writer of S_x, is issued after PV_x(j),
// and the tensor pipe executes in issue order.
//
// TMEM columns: S_0 [0,128) S_1 [128,256) O_0 [256,256+D) O_1 [256+D,256+2D).
//
// The producer passes each claimed item (index, key-tile count) to the MMA
// warp and the softmax warps through a two-slot ring (ITEM_FULL / ITEM_EMPTY).
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

// ST: the layout has the output staging region (instantiations that store
// full tiles by TMA); without it the shared-memory carve-out stays smaller,
// which leaves more L1 for the long-walk kernel's spill slots.
template <int D, bool ST>
struct Cfg {
    static constexpr int NBOX = D / 64;            // 64-column boxes per tile
    static constexpr int BOX_BYTES = TILE * 128;   // 128 rows x 128 bytes
    static constexpr int TILE_BYTES = NBOX * BOX_BYTES;
    static constexpr int KS = D == 128 ? 2 : 3;    // K stages
    static constexpr int VS = KS;                  // V stages
    static constexpr int TIR = 16;                 // key-tile description ring (power of two)
    static constexpr int Q_OFF = 0;                // query tile x at Q_OFF + x * TILE_BYTES
    static constexpr int K_OFF = 2 * TILE_BYTES;
    static constexpr int V_OFF = K_OFF + KS * TILE_BYTES;
    // Output staging: 32 rows x 64 columns (bf16, 128B swizzle) per softmax warp,
    // warp q of group x at OST_OFF + (4 x + q) * OST_WARP; a TMA store writes them out.
    static constexpr int OST_WARP = 32 * 128;
    static constexpr int OST_OFF = V_OFF + VS * TILE_BYTES;
    static constexpr int BAR_OFF = OST_OFF + (ST ? 8 * OST_WARP : 0);
    enum {
        B_QFULL = 0,
        B_QEMPTY,
        B_KFULL,
        B_KEMPTY = B_KFULL + KS,     // QK_0(j) and QK_1(j) complete: K stage free
        B_VFULL = B_KEMPTY + KS,
        B_VEMPTY = B_VFULL + VS,     // PV_0(j) and PV_1(j) complete: V stage free
        B_SFULL = B_VEMPTY + VS,     // [x]: QK_x complete
        B_PFULL = B_SFULL + 2,       // [2 x + h]: P_x of keys [64 h, 64 h + 64) stored by group x (128 arrivals)
        B_PVDONE = B_PFULL + 4,      // [x]: PV_x complete (O_x may be rescaled)
        B_OFULL = B_PVDONE + 2,      // [x]: the item's last PV_x complete
        B_OEMPTY = B_OFULL + 2,      // [x]: group x has read O_x out (128 arrivals)
        B_DRAIN = B_OEMPTY + 2,
        B_ITEMFULL,
        B_ITEMEMPTY = B_ITEMFULL + 2,
        NBAR = B_ITEMEMPTY + 2
    };
    // [0] tmem base, [1] abort, [2..3] item key tiles, [4..5] item index (by item parity)
    static constexpr int MISC_OFF = BAR_OFF + NBAR * 8;
    // TIR x {global position, len | class0 << 16 | class1 << 20, tile sequence number + 1, unused}
    static constexpr int TI_OFF = MISC_OFF + 32;
    static constexpr int SMEM_USED = TI_OFF + TIR * 16 + 1024;   // + slack to align the base to 1 KB
    // At least 120 KB, so that one CTA occupies an SM: each CTA allocates all
    // 512 TMEM columns, and a second one would wait inside tcgen05.alloc.
    static constexpr int SMEM_BYTES = SMEM_USED > 120 * 1024 ? SMEM_USED : 120 * 1024;
    static constexpr uint32_t S_COL = 0;           // S_x at S_COL + 128 x; P_x over its first 64 columns
    static constexpr uint32_t O_COL = 256;         // O_x at O_COL + D x
    static constexpr uint32_t TMEM_COLS = 512;
    static constexpr int THREADS = 320;
    // Instruction descriptors (kind::f16): D fp32 (bits 4-5 = 1), A and B
    // bf16 (bits 7-9, 10-12 = 1), B major bit 16 (0 = K-major, 1 = MN-major),
    // N >> 3 at bits 17-22, M >> 4 at bits 24-28.
    static constexpr uint32_t IDESC_QK =
        (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(TILE >> 3) << 17) | ((uint32_t)(TILE >> 4) << 24);
    static constexpr uint32_t IDESC_PV = (1u << 4) | (1u << 7) | (1u << 10) | (1u << 16) |
                                         ((uint32_t)(D >> 3) << 17) | ((uint32_t)(TILE >> 4) << 24);
};

// 32 bits of an exclusion mask (1 = excluded, one byte per key) starting at p,
// of which the first n are meaningful; bit i set when byte i is nonzero.
__device__ __forceinline__ uint32_t excl_bits(const uint8_t *p, int n) {
    uint32_t w[8];
    if (n >= 32 && (reinterpret_cast<uintptr_t>(p) & 15) == 0) {
        const uint4 a = __ldg(reinterpret_cast<const uint4 *>(p));
        const uint4 b = __ldg(reinterpret_cast<const uint4 *>(p + 16));
        w[0] = a.x; w[1] = a.y; w[2] = a.z; w[3] = a.w;
        w[4] = b.x; w[5] = b.y; w[6] = b.z; w[7] = b.w;
    } else {
        for (int k = 0; k < 8; ++k) w[k] = 0;
        for (int i = 0; i < 32 && i < n; ++i) w[i >> 2] |= (uint32_t)__ldg(p + i) << (8 * (i & 3));
    }
    uint32_t m = 0;
#pragma unroll
    for (int i = 0; i < 32; ++i)
        if ((w[i >> 2] >> (8 * (i & 3))) & 0xffu) m |= 1u << i;
    return m;
}

// Keys [c0, c0 + 32) of key tile kt that the query at global position qpos
// may see (bit i for key c0 + i): inside the tile, not in the causal future,
// not padded, not forbidden by attn_mask.  Out of line: it runs on PARTIAL
// tiles only, and inlined into the softmax loop its registers and code sat
// beside the 128 scores of every tile.
__device__ __noinline__ uint32_t keep_bits(const Geom &g, int b, long long qpos, bool row_valid, long long kpos0,
                                           int klen, int c0) {
    const int n = klen - c0;
    if (n <= 0) return 0u;
    uint32_t m = n >= 32 ? 0xffffffffu : (1u << n) - 1u;
    if (g.causal) {
        const long long lim = qpos - kpos0 - c0;   // key c0 + i lies in the future when i > lim
        if (lim < 0) return 0u;
        if (lim < 31) m &= (2u << lim) - 1u;
    }
    if (!row_valid) return m;   // rows past the tile end are never stored; their mask rows may not exist
    if (g.kpm) m &= ~excl_bits(g.kpm + b * g.kpm_ld + kpos0 + c0, n);
    if (g.am) m &= ~excl_bits(g.am + qpos * g.am_ld + kpos0 + c0, n);
    return m;
}

// The keys of key tile kt (positions kpos0 .. kpos0 + klen - 1) that the query
// at global position qpos may see, as four 32-bit masks (bit i of m[c] for key
// 32 c + i): inside the tile, not in the causal future, not padded, not
// forbidden by attn_mask.  Every mask byte the tile needs is loaded before any
// is used (up to sixteen independent 16-byte loads), so the call costs about
// one load latency, and it is made before the tile's scores are waited for.
// The kernels that use it (PF: launches with masks, striped ranks, or short
// walks, where PARTIAL tiles are a sizeable share) trade this for a slightly
// different hot loop, measured about 1 % slower on the 64K prefill, whose
// walks are long and nearly all FULL.
struct Keep4 {
    uint32_t m[4];
};

__device__ __noinline__ Keep4 keep_bits4(const Geom &g, int b, long long qpos, bool row_valid, long long kpos0,
                                         int klen) {
    Keep4 r;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        const int n = klen - 32 * c;
        uint32_t m = n <= 0 ? 0u : (n >= 32 ? 0xffffffffu : (1u << n) - 1u);
        if (g.causal) {
            const long long lim = qpos - kpos0 - 32 * c;   // key 32 c + i lies in the future when i > lim
            if (lim < 0) m = 0u;
            else if (lim < 31) m &= (2u << lim) - 1u;
        }
        r.m[c] = m;
    }
    if (!row_valid) return r;   // rows past the tile end are never stored; their mask rows may not exist
    uint32_t ek[4] = {0u, 0u, 0u, 0u}, ea[4] = {0u, 0u, 0u, 0u};
    if (g.kpm) {
        const uint8_t *p = g.kpm + b * g.kpm_ld + kpos0;
#pragma unroll
        for (int c = 0; c < 4; ++c)
            if (klen > 32 * c) ek[c] = excl_bits(p + 32 * c, klen - 32 * c);
    }
    if (g.am) {
        const uint8_t *p = g.am + qpos * g.am_ld + kpos0;
#pragma unroll
        for (int c = 0; c < 4; ++c)
            if (klen > 32 * c) ea[c] = excl_bits(p + 32 * c, klen - 32 * c);
    }
#pragma unroll
    for (int c = 0; c < 4; ++c) r.m[c] &= ~(ek[c] | ea[c]);
    return r;
}

// ----------------------------------------------------------------------------
// Kernel
// ----------------------------------------------------------------------------

template <int D, bool S, bool PF>
__global__ void __launch_bounds__(320, 1)
    attn_tc_kernel(const AttnArgs a, const __grid_constant__ CUtensorMap tq,
                   const __grid_constant__ CUtensorMap tk, const __grid_constant__ CUtensorMap tv,
                   const __grid_constant__ CUtensorMap to) {
    using C = Cfg<D, PF>;
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
        for (int i = 0; i < C::KS; ++i) {
            mbar_init(bar(C::B_KFULL + i), 1);
            mbar_init(bar(C::B_KEMPTY + i), 1);
        }
        for (int i = 0; i < C::VS; ++i) {
            mbar_init(bar(C::B_VFULL + i), 1);
            mbar_init(bar(C::B_VEMPTY + i), 1);
        }
        for (int i = 0; i < 4; ++i) mbar_init(bar(C::B_PFULL + i), 128);
        for (int x = 0; x < 2; ++x) {
            mbar_init(bar(C::B_SFULL + x), 1);
            mbar_init(bar(C::B_PVDONE + x), 1);
            mbar_init(bar(C::B_OFULL + x), 1);
            mbar_init(bar(C::B_OEMPTY + x), 128);
        }
        mbar_init(bar(C::B_DRAIN), 1);
        for (int i = 0; i < 2; ++i) {
            mbar_init(bar(C::B_ITEMFULL + i), 1);
            mbar_init(bar(C::B_ITEMEMPTY + i), 1 + 8);   // MMA warp + one lane per softmax warp
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
    // A CTA that holds all 512 TMEM columns holds them from column 0, so the
    // TMEM addresses below are compile-time constants (which keeps the MMA issue
    // on the uniform datapath).  Any other base is reported through the error
    // word and nothing runs.
    const uint32_t tmem_base = misc[0];
    constexpr uint32_t tmem = 0u;

    if (tmem_base != 0u) {
        if (threadIdx.x == 0) atomicOr(a.err, ERR_TIMEOUT_BIT);
    } else if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            uint32_t kfill = 0, vfill = 0, qfills = 0, it_local = 0;
            bool ok = true;
            // Items are claimed from the launch's counter in index order (heaviest
            // first under causal masking), so an SM takes its next item when it runs
            // out of work; without a counter they are dealt round-robin by CTA.
            int w = a.sched ? (int)atomicAdd(a.sched, 1u) : (int)blockIdx.x;
            for (;; ++it_local) {
                // Publish (item, key tiles | second tile present << 31) in slot it & 1 for
                // the MMA warp and the softmax warps; the slot's previous item (it - 2)
                // has been read by all.
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
                const QPair p = work_pair<S>(g, w);
                const bool has1 = p.q1.len > 0;
                misc[4 + sl] = (uint32_t)w;
                misc[2 + sl] = (uint32_t)pair_count<S>(g, p) | (has1 ? 0x80000000u : 0u);
                mbar_arrive(bar(C::B_ITEMFULL + sl));
                if (it_local > 0 && !mbar_wait(bar(C::B_QEMPTY), (it_local - 1) & 1, abort, a.err, lim)) {
                    ok = false;
                    break;
                }
                mbar_arrive_expect_tx(bar(C::B_QFULL), (has1 ? 2 : 1) * C::TILE_BYTES);
                for (int bx = 0; bx < C::NBOX; ++bx)
                    tma_load_rows<S>(sQ + bx * C::BOX_BYTES, &tq, g, bx * 64, p.q0.row0, p.q0.h, p.q0.b, bar(C::B_QFULL));
                if (has1)
                    for (int bx = 0; bx < C::NBOX; ++bx)
                        tma_load_rows<S>(sQ + C::TILE_BYTES + bx * C::BOX_BYTES, &tq, g, bx * 64, p.q1.row0, p.q0.h,
                                      p.q0.b, bar(C::B_QFULL));
                ++qfills;
                KWalk wk;
                kwalk_begin<S>(g, p.span, wk);
                KTile kt;
                int c0, c1;
                int prev_row = -1;   // k/v row of the tile whose V is still to be loaded
                for (;;) {
                    const bool more = pair_next<S>(g, p, wk, kt, c0, c1);
                    // V of the previous tile first: its products come before this tile's scores
                    if (prev_row >= 0) {
                        const uint32_t st = vfill % C::VS, use = vfill / C::VS;
                        if (use > 0 && !mbar_wait(bar(C::B_VEMPTY + st), (use - 1) & 1, abort, a.err, lim)) {
                            ok = false;
                            break;
                        }
                        mbar_arrive_expect_tx(bar(C::B_VFULL + st), C::TILE_BYTES);
                        for (int bx = 0; bx < C::NBOX; ++bx)
                            tma_load_rows<S>(sV + st * C::TILE_BYTES + bx * C::BOX_BYTES, &tv, g, bx * 64, prev_row,
                                          p.q0.h, p.q0.b, bar(C::B_VFULL + st));
                        ++vfill;
                    }
                    if (more) {
                        const uint32_t st = kfill % C::KS, use = kfill / C::KS;
                        if (use > 0 && !mbar_wait(bar(C::B_KEMPTY + st), (use - 1) & 1, abort, a.err, lim)) {
                            ok = false;
                            break;
                        }
                        // Describe tile kfill in slot kfill % TIR.  Both products of tile
                        // kfill - KS have completed (the wait above), and QK_x(j) is issued
                        // after PV_x(j - 1): each group has read every description up to
                        // kfill - KS - 1, including this slot's last (TIR > KS + 1).
                        {
                            const uint32_t e = (kfill % C::TIR) * 4;
                            tinfo[e] = (uint32_t)kt.pos0;
                            tinfo[e + 1] = (uint32_t)kt.len | ((uint32_t)c0 << 16) | ((uint32_t)c1 << 20);
                            st_release_shared(sTI + e * 4 + 8, kfill + 1);
                        }
                        mbar_arrive_expect_tx(bar(C::B_KFULL + st), C::TILE_BYTES);
                        for (int bx = 0; bx < C::NBOX; ++bx)
                            tma_load_rows<S>(sK + st * C::TILE_BYTES + bx * C::BOX_BYTES, &tk, g, bx * 64, kt.row0,
                                          p.q0.h, p.q0.b, bar(C::B_KFULL + st));
                        ++kfill;
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
        // Per item: QK_0(0), QK_1(0); then for each key tile j: PV_0(j) once group 0
        // has written P_0(j), QK_0(j+1) into S_0 (over P_0(j), which PV_0(j), issued
        // just before, has read: the tensor pipe executes in issue order), and the
        // same for group 1.  The whole warp runs this loop converged (waits,
        // counters, descriptors); each MMA and commit is issued by one elected lane.
        {
            uint32_t it_local = 0;
            uint32_t kst = 0, kph = 0;   // K stage and phase of the next QK
            uint32_t vst = 0, vph = 0;   // V stage and phase of the next PV
            uint32_t pc[2] = {0, 0};     // PV_x issued so far (P_FULL[x] phases)
            uint32_t oc[2] = {0, 0};     // items finished by group x (O_EMPTY[x] phases)
            bool ok = true;
            const uint64_t qdesc0 = sdesc(sQ, 16, 1024);            // K-major, 128B swizzle
            const uint64_t kdesc0 = sdesc(sK, 16, 1024);
            const uint64_t vdesc0 = sdesc(sV, C::BOX_BYTES, 1024);   // MN-major
            // descriptor start-address fields advance by bytes / 16
            constexpr uint32_t STAGE16 = C::TILE_BYTES >> 4;
            auto qk = [&](int x) {
                const uint64_t qd = qdesc0 + (uint64_t)(x * STAGE16);
                const uint64_t kd = kdesc0 + (uint64_t)(kst * STAGE16);
                const uint32_t sd = tmem + C::S_COL + x * 128;
                // Short-walk instantiations issue four MMAs per election (8K -0.7 %, striped
                // 8K -2 %); the long-walk one keeps one election per MMA (64K +0.3 % batched).
                if constexpr (PF) {
#pragma unroll
                    for (int k4 = 0; k4 < D / 64; ++k4) {   // one 64-column box: four MMAs of K = 16
                        uint64_t ad[4], bd[4];
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            const uint64_t off = (uint64_t)((k4 * C::BOX_BYTES + i * 32) >> 4);
                            ad[i] = qd + off;
                            bd[i] = kd + off;
                        }
                        mma_ss_4(sd, ad, bd, C::IDESC_QK, k4 > 0 ? 1u : 0u);
                    }
                } else {
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {
                        const uint64_t off = (uint64_t)(((kk >> 2) * C::BOX_BYTES + (kk & 3) * 32) >> 4);
                        mma_ss_one(sd, qd + off, kd + off, C::IDESC_QK, kk > 0 ? 1u : 0u);
                    }
                }
                mma_commit_one(bar(C::B_SFULL + x));
            };
            // P_x arrives in two halves of 64 keys: the products of the first half run
            // while group x computes the exponentials of the second.
            auto pv = [&](int x, bool first) -> bool {
                const uint64_t vd = vdesc0 + (uint64_t)(vst * STAGE16);
                const uint32_t pa = tmem + C::S_COL + x * 128;
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    if (!warp_wait(bar(C::B_PFULL + 2 * x + h), pc[x] & 1, abort, a.err, lim)) return false;
                    tc_fence_after();   // P was written by the softmax warps' tcgen05.st
                    if constexpr (PF) {
                        uint32_t at[4];
                        uint64_t bd[4];
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            const int kk = 4 * h + i;
                            at[i] = pa + kk * 8;
                            bd[i] = vd + (uint64_t)((kk * 2048) >> 4);
                        }
                        mma_ts_4(tmem + C::O_COL + x * D, at, bd, C::IDESC_PV, (first && h == 0) ? 0u : 1u);
                    } else {
#pragma unroll
                        for (int kk = 4 * h; kk < 4 * h + 4; ++kk)
                            mma_ts_one(tmem + C::O_COL + x * D, pa + kk * 8, vd + (uint64_t)((kk * 2048) >> 4),
                                       C::IDESC_PV, (first && kk == 0) ? 0u : 1u);
                    }
                }
                ++pc[x];
                mma_commit_one(bar(C::B_PVDONE + x));
                return true;
            };
            auto next_k = [&]() {
                kst = kst == C::KS - 1 ? 0 : kst + 1;
                kph ^= kst == 0;
            };
            // O_x of group x's previous item must have been read out before this
            // item's first PV_x writes O_x (and before O_FULL[x]): waited once per item.
            auto o_free = [&](int x) -> bool {
                return oc[x] == 0 || warp_wait(bar(C::B_OEMPTY + x), (oc[x] - 1) & 1, abort, a.err, lim);
            };
            for (;; ++it_local) {
                const uint32_t sl = it_local & 1;
                if (!warp_wait(bar(C::B_ITEMFULL + sl), (it_local >> 1) & 1, abort, a.err, lim)) {
                    ok = false;
                    break;
                }
                const uint32_t item = misc[4 + sl], nn = misc[2 + sl];
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(C::B_ITEMEMPTY + sl));
                if (item == 0xffffffffu) break;
                const uint32_t n = nn & 0x7fffffffu;
                const int ng = (nn >> 31) ? 2 : 1;   // query tiles in the pair
                if (!warp_wait(bar(C::B_QFULL), it_local & 1, abort, a.err, lim)) {
                    ok = false;
                    break;
                }
                if (n == 0) {
                    mma_commit_one(bar(C::B_QEMPTY));
                    for (int x = 0; x < ng && ok; ++x) {
                        if (!(ok = o_free(x))) break;
                        mma_commit_one(bar(C::B_OFULL + x));
                        ++oc[x];
                    }
                    if (!ok) break;
                    continue;
                }
                // tile 0: both QKs, then the K stage and (one tile) Q are released
                if (!(ok = warp_wait(bar(C::B_KFULL + kst), kph, abort, a.err, lim))) break;
                for (int x = 0; x < ng; ++x) qk(x);
                mma_commit_one(bar(C::B_KEMPTY + kst));
                if (n == 1) mma_commit_one(bar(C::B_QEMPTY));
                next_k();
                for (uint32_t j = 0; j < n && ok; ++j) {
                    const bool last = j + 1 == n;
                    if (!(ok = warp_wait(bar(C::B_VFULL + vst), vph, abort, a.err, lim))) break;
                    for (int x = 0; x < ng; ++x) {
                        if (j == 0 && !(ok = o_free(x))) break;
                        if (!(ok = pv(x, j == 0))) break;
                        if (last) {
                            mma_commit_one(bar(C::B_OFULL + x));
                        } else {
                            if (x == 0 && !(ok = warp_wait(bar(C::B_KFULL + kst), kph, abort, a.err, lim))) break;
                            qk(x);
                        }
                    }
                    if (!ok) break;
                    mma_commit_one(bar(C::B_VEMPTY + vst));   // V(j) free once PV_0(j), PV_1(j) complete
                    vst = vst == C::VS - 1 ? 0 : vst + 1;
                    vph ^= vst == 0;
                    if (!last) {
                        mma_commit_one(bar(C::B_KEMPTY + kst));   // K(j+1) free once QK_0(j+1), QK_1(j+1) complete
                        if (j + 2 == n) mma_commit_one(bar(C::B_QEMPTY));
                        next_k();
                    }
                }
                if (!ok) break;
                for (int x = 0; x < ng; ++x) ++oc[x];
            }
            if (!ok) {
                // Wait for the MMAs already issued before TMEM is released.
                volatile int never = 0;
                mma_commit_one(bar(C::B_DRAIN));
                warp_wait(bar(C::B_DRAIN), 0, &never, nullptr, 200000000ull);
            }
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ softmax / epilogue
        const int x = (warp - 2) >> 2;                 // group: query tile of the pair
        const int quad = warp & 3;                     // TMEM lanes 32 quad .. + 31
        const int row = quad * 32 + lane;
        const uint32_t lane_addr = (uint32_t)(quad * 32) << 16;
        const uint32_t scol = C::S_COL + (uint32_t)x * 128, ocol = C::O_COL + (uint32_t)x * D;
        const float sl2 = a.scale_log2;
        uint32_t sx = 0;     // S_x completions seen (S_FULL[x] phases)
        uint32_t tx = 0;     // P_x tiles stored (the previous one's PV_x is PV_DONE[x] phase tx - 1)
        uint32_t ox = 0;     // items finished (O_FULL[x] phases)
        uint32_t tcnt = 0;   // key tiles described so far (ring position)
        bool ok = true;
        for (uint32_t it_local = 0;; ++it_local) {
            const uint32_t sl = it_local & 1;
            if (!warp_wait(bar(C::B_ITEMFULL + sl), (it_local >> 1) & 1, abort, a.err, lim)) {
                ok = false;
                break;
            }
            const uint32_t item = misc[4 + sl], nn = misc[2 + sl];
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(C::B_ITEMEMPTY + sl));
            if (item == 0xffffffffu) break;
            const uint32_t n_tiles = nn & 0x7fffffffu;
            if (x == 1 && !(nn >> 31)) {   // the pair holds one tile: nothing for group 1
                tcnt += n_tiles;
                continue;
            }
            const QPair pr = work_pair<S>(g, (int)item);
            const QTile qt = x ? pr.q1 : pr.q0;
            const long long qpos = qt.pos0 + row;
            float m_ref = -INFINITY, l = 0.f;
            int n = 0;
            for (uint32_t j = 0; j < n_tiles; ++j) {
                // The producer walked the tiles; take this one's position, length and
                // class (written before K of the tile was loaded, so normally present,
                // and read before the scores arrive).
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
                    kt.cls = (int)((dy >> (16 + 4 * x)) & 15u);
                }
                // FULL tiles need no predicate; PARTIAL ones, and tiles EMPTY for this
                // group's rows (seen only by the other tile of the pair), are masked.
                const bool masked = kt.cls != BA_TILE_FULL || kt.len < TILE;
                Keep4 keep;
                if constexpr (PF) {
                    if (masked) keep = keep_bits4(g, qt.b, qpos, row < qt.len, kt.pos0, kt.len);
                }
                if (!warp_wait(bar(C::B_SFULL + x), sx & 1, abort, a.err, lim)) {
                    ok = false;
                    break;
                }
                ++sx;
                tc_fence_after();
                float s[TILE];
                {
                    uint32_t r[TILE];
#pragma unroll
                    for (int c = 0; c < TILE / 32; ++c)
                        tmem_ld32(tmem + lane_addr + scol + c * 32, *reinterpret_cast<uint32_t(*)[32]>(&r[c * 32]));
                    tmem_wait_ld();
#pragma unroll
                    for (int j2 = 0; j2 < TILE; ++j2) s[j2] = __uint_as_float(r[j2]);
                }

                if (masked) {
#pragma unroll
                    for (int c = 0; c < TILE / 32; ++c) {
                        uint32_t kb;
                        if constexpr (PF) {
                            kb = keep.m[c];
                        } else {
                            kb = keep_bits(g, qt.b, qpos, row < qt.len, kt.pos0, kt.len, c * 32);
                        }
#pragma unroll
                        for (int i = 0; i < 32; ++i)
                            if (!((kb >> i) & 1u)) s[c * 32 + i] = -INFINITY;
                    }
                }
                // Row maximum first (8 independent chains of three-input maxima, then a
                // tree).  The reference maximum m moves only when the tile's maximum
                // exceeds it by more than 2^8 (lazy rule: the sums and O keep their scale
                // otherwise; p stays below 2^8).
                float mc[8];
#pragma unroll
                for (int k = 0; k < 8; ++k) mc[k] = fmaxf(s[k], s[8 + k]);
#pragma unroll
                for (int j2 = 16; j2 < TILE; j2 += 16) {
#pragma unroll
                    for (int k = 0; k < 8; ++k) mc[k] = fmax3(mc[k], s[j2 + k], s[j2 + 8 + k]);
                }
                const float mx = fmaxf(fmax3(mc[0], mc[1], mc[2]), fmax3(fmax3(mc[3], mc[4], mc[5]), mc[6], mc[7]));
                const float m_new = fmaxf(m_ref, mx * sl2);
                const bool resc = m_new > m_ref + 8.0f;   // true when m_ref = -inf and m_new finite
                float alpha = 1.f;
                if (resc) {
                    alpha = fast_exp2(m_ref - m_new);   // 0 when m_ref = -inf
                    m_ref = m_new;
                }
                // O must be rescaled (rarely, when m moved) before this tile's first
                // PV_x is issued; P is handed to the MMA warp in two halves of 64 keys,
                // the first as soon as it is stored when no rescale is due, so that its
                // products run while the second half's exponentials are computed.
                const bool rescale_o = __any_sync(0xffffffffu, resc) && n > 0;
                // p = 2^(s * scale * log2(e) - m), arguments two lanes at a time, sums in
                // four two-lane accumulators; P (bf16) goes over the S columns already
                // read, 16 columns (32 keys) at a time.
                const float m_use = m_ref == -INFINITY ? 0.f : m_ref;
                float sc[8];
#pragma unroll
                for (int k = 0; k < 8; ++k) sc[k] = 0.f;
#pragma unroll
                for (int c = 0; c < TILE / 32; ++c) {
                    uint32_t pk[16];
#pragma unroll
                    for (int j2 = 0; j2 < 16; ++j2) {
                        float x0, x1;
                        ffma2_bc(s[32 * c + 2 * j2], s[32 * c + 2 * j2 + 1], sl2, -m_use, x0, x1);
                        const float p0 = fast_exp2(x0);
                        const float p1 = fast_exp2(x1);
                        fadd2_acc(sc[2 * (j2 & 3)], sc[2 * (j2 & 3) + 1], p0, p1);
                        pk[j2] = pack_bf16(p0, p1);
                    }
                    tmem_st16(tmem + lane_addr + scol + c * 16, pk);
                    if (c == 1 && !rescale_o) {
                        tmem_wait_st();
                        tc_fence_before();
                        mbar_arrive(bar(C::B_PFULL + 2 * x));
                    }
                }
                const float sum = ((sc[0] + sc[1]) + (sc[2] + sc[3])) + ((sc[4] + sc[5]) + (sc[6] + sc[7]));
                l = l * alpha + sum;
                if (rescale_o) {
                    // once the previous tile's PV_x has completed
                    if (!warp_wait(bar(C::B_PVDONE + x), (tx - 1) & 1, abort, a.err, lim)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
#pragma unroll
                    for (int c = 0; c < D / 32; ++c) {
                        uint32_t r[32];
                        tmem_ld32(tmem + lane_addr + ocol + c * 32, r);
                        tmem_wait_ld();
#pragma unroll
                        for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * alpha);
                        tmem_st32(tmem + lane_addr + ocol + c * 32, r);
                    }
                }
                tmem_wait_st();
                tc_fence_before();
                if (rescale_o) mbar_arrive(bar(C::B_PFULL + 2 * x));
                mbar_arrive(bar(C::B_PFULL + 2 * x + 1));
                ++tx;
                ++n;
            }
            if (!ok) break;
            // epilogue
            if (!warp_wait(bar(C::B_OFULL + x), ox & 1, abort, a.err, lim)) {
                ok = false;
                break;
            }
            ++ox;
            tc_fence_after();
            const bool valid = row < qt.len;
            const long long row_flat = ((long long)qt.b * g.H + qt.h) * a.rows + out_row<S>(g, qt, row);
            const float acc_l = (a.acc_lse != nullptr && valid) ? a.acc_lse[row_flat] : -INFINITY;
            const RowFinal f = row_final(m_ref, n > 0 ? l : 0.f, acc_l);
            // (the instantiations for long walks keep the per-row stores: there the
            // item boundary is rare and the staging code costs registers in the loop)
            if (PF && a.tma_out && qt.len == TILE) {
                // Full tile, bf16 output, no partial to merge: each warp stages its
                // 32 rows, 64 columns at a time, in shared memory (128B swizzle: the
                // 16-byte unit u of row r at unit u ^ (r & 7)) and writes them with one
                // TMA store, so that the global writes are whole lines and the warp
                // does not wait for them.
                const uint32_t ost = base + C::OST_OFF + (uint32_t)(4 * x + quad) * C::OST_WARP;
                const uint32_t orow = ost + (uint32_t)lane * 128u;
#pragma unroll
                for (int bx = 0; bx < C::NBOX; ++bx) {
                    // the staging rows are free once the previous store has read them
                    if (lane == 0) bulk_wait_read();
                    __syncwarp();
#pragma unroll
                    for (int c = 2 * bx; c < 2 * bx + 2; ++c) {
                        uint32_t r[32];
                        if (n > 0) {
                            tmem_ld32(tmem + lane_addr + ocol + c * 32, r);
                            tmem_wait_ld();
                        } else {
#pragma unroll
                            for (int i = 0; i < 32; ++i) r[i] = 0u;
                        }
#pragma unroll
                        for (int u4 = 0; u4 < 4; ++u4) {
                            uint32_t w[4];
#pragma unroll
                            for (int k = 0; k < 4; ++k)
                                w[k] = pack_bf16(f.wb * (__uint_as_float(r[8 * u4 + 2 * k]) * f.inv_l),
                                                 f.wb * (__uint_as_float(r[8 * u4 + 2 * k + 1]) * f.inv_l));
                            const uint32_t u = (uint32_t)(4 * (c & 1) + u4);
                            st_shared_v4(orow + ((u ^ (uint32_t)(lane & 7)) << 4), w);
                        }
                    }
                    fence_proxy_async_shared();
                    __syncwarp();
                    if (lane == 0) {
                        if constexpr (S)
                            tma_store_5d(&to, ost, bx * 64, qt.rank, (int)qt.pos0 + 32 * quad, qt.h, qt.b);
                        else
                            tma_store_4d(&to, ost, bx * 64, qt.row0 + 32 * quad, qt.h, qt.b);
                        bulk_commit();
                    }
                }
            } else {
#pragma unroll
                for (int c = 0; c < D / 32; ++c) {
                    uint32_t r[32];
                    float o[32];
                    if (n > 0) {
                        tmem_ld32(tmem + lane_addr + ocol + c * 32, r);
                        tmem_wait_ld();
#pragma unroll
                        for (int i = 0; i < 32; ++i) o[i] = __uint_as_float(r[i]);
                    } else {
#pragma unroll
                        for (int i = 0; i < 32; ++i) o[i] = 0.f;
                    }
                    if (valid) store_row_chunk(a, row_flat, c * 32, o, 32, f);
                }
            }
            if (valid) a.lse[row_flat] = f.lse;
            tc_fence_before();
            mbar_arrive(bar(C::B_OEMPTY + x));
        }
        if constexpr (PF) {
            // the output stores this warp issued have finished before the CTA exits
            if (lane == 0) bulk_wait_all();
            __syncwarp();
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) {
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(C::TMEM_COLS)
                     : "memory");
    }
}

template <int D, bool S, bool PF>
int launch_dpf(const AttnArgs &a, const TmaMaps &m, int num_sms, cudaStream_t s) {
    using C = Cfg<D, PF>;
    static_assert(C::SMEM_BYTES <= 232448, "shared memory budget");
    cudaError_t e = cudaFuncSetAttribute(attn_tc_kernel<D, S, PF>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         C::SMEM_BYTES);
    if (e != cudaSuccess) return BA_ERR_CUDA;
    int grid = a.g.n_items < num_sms ? a.g.n_items : num_sms;
    attn_tc_kernel<D, S, PF><<<grid, C::THREADS, C::SMEM_BYTES, s>>>(a, m.q, m.k, m.v, m.o);
    return cudaGetLastError() == cudaSuccess ? BA_OK : BA_ERR_CUDA;
}

// Masks are prefetched (keep_bits4 before the scores are waited for) when
// PARTIAL tiles are a sizeable share of the walks: with masks, with striped
// ranks (a diagonal in every block), or when a head has fewer than 256 key
// tiles (T < 32K: the causal diagonal tiles are one in about 17 of a walk
// or more).
template <int D, bool S>
int launch_d(const AttnArgs &a, const TmaMaps &m, int num_sms, cudaStream_t s) {
    if constexpr (S) {
        return launch_dpf<D, S, true>(a, m, num_sms, s);
    } else {
        const bool pf = a.g.kpm != nullptr || a.g.am != nullptr || a.g.n_ktiles < 256;
        return pf ? launch_dpf<D, S, true>(a, m, num_sms, s) : launch_dpf<D, S, false>(a, m, num_sms, s);
    }
}

}  // namespace

bool tc_supported(int dtype, int d) { return dtype == BA_BF16 && (d == 64 || d == 128); }

size_t tc_smem_bytes(int d) { return d == 128 ? Cfg<128, true>::SMEM_BYTES : Cfg<64, true>::SMEM_BYTES; }

int launch_attn_tc(const AttnArgs &a, const TmaMaps &m, int num_sms, cudaStream_t s) {
    // The kernel's unit of work is a pair of query tiles (work_pair).
    AttnArgs ap = a;
    ap.g.n_items = n_pairs(a.g) * a.g.B * a.g.H;
    ap.g.tail_levels = pair_tail_levels(a.g, num_sms);
    if (ap.g.n_items == 0 || a.g.n_qtiles == 0) return BA_OK;
    if (a.g.striped) {
        if (a.g.d == 128) return launch_d<128, true>(ap, m, num_sms, s);
        if (a.g.d == 64) return launch_d<64, true>(ap, m, num_sms, s);
        return BA_ERR_SHAPE;
    }
    if (a.g.d == 128) return launch_d<128, false>(ap, m, num_sms, s);
    if (a.g.d == 64) return launch_d<64, false>(ap, m, num_sms, s);
    return BA_ERR_SHAPE;
}

}  // namespace ba
