// Attention backward on the tensor cores (tcgen05, bf16 inputs, d = 64 / 128).
//
// The gradients of "Sequence/context parallelism" (brunomaga), section "Ring
// Attention", backward pass: with p_ij = exp(scale q_i . k_j - LSE_i) from the
// saved LSE of the whole row and D_i = dout_i . out_i,
//   dV_j = sum_i p_ij dout_i,  ds_ij = p_ij (dout_i . v_j - D_i),
//   dK_j = scale sum_i ds_ij q_i,  dQ_i = scale sum_j ds_ij k_j.
// Two kernels, no atomics (every output row is written by one CTA):
//
// bwd_dkdv_tc_kernel: one CTA per 128-key tile of one (b, h).  K and V of the
//   tile stay in shared memory; the query tiles that see them stream through a
//   two-stage ring (Q, dout, and the rows' LSE and D).  Per query tile:
//     S^T  = K Q^T     (8 MMAs, fp32 into TMEM)
//     dP^T = V dout^T  (8 MMAs)
//     the elementwise warps form P^T and dS^T (bf16) over those TMEM columns
//     dV  += P^T dout  (A = P^T from TMEM, B = dout MN-major)
//     dK  += dS^T Q    (A = dS^T from TMEM, B = Q MN-major)
// bwd_dq_tc_kernel: one CTA per 128-row query tile; key tiles stream:
//     S = Q K^T, dP = dout V^T, dS (bf16) over S, dQ += dS K.
// Seven products per (query tile, key tile) against the five of the gradient
// itself: S and dP are formed in both kernels, which is what keeps dQ free of
// atomics.  The scale is applied to dK and dQ in the epilogues.
//
// Roles (384 threads): warp 0 TMA producer (and the LSE / D rows, loaded by its
// 32 lanes), warp 1 TMEM owner and MMA issuer (converged, one elected lane per
// instruction), two elementwise + epilogue groups: warps 4..7 take half 0 and
// warps 8..11 half 1 of every partner tile (thread t of a group owns TMEM lane
// t; two warps per sub-partition share the elementwise work of a tile), and
// split the epilogue (dK/dV: dV rows / dK rows; dQ: the two column halves).
// Warps 2..3 idle (the groups must start on a warpgroup boundary).
// Every mbarrier wait is bounded, as in the forward kernel.
#include "internal.h"
#include "tc_ptx.cuh"

namespace ba {
namespace {

template <int D>
struct BCfg {
    static constexpr int NBOX = D / 64;
    static constexpr int BOX_BYTES = TILE * 128;          // 128 rows x 128 bytes
    static constexpr int TILE_BYTES = NBOX * BOX_BYTES;   // one 128-row tile of one tensor
    static constexpr int NST = 2;                         // streamed stages
    static constexpr int RES_OFF = 0;                     // resident pair: R0, R1
    static constexpr int STG_OFF = 2 * TILE_BYTES;
    static constexpr int VEC_OFF = 2 * TILE_BYTES;        // within a stage: 128 LSE (log2 units) + 128 D
    static constexpr int STG_BYTES = 2 * TILE_BYTES + 1024;
    static constexpr int BAR_OFF = STG_OFF + NST * STG_BYTES;
    // RES_FULL / RES_EMPTY: the resident pair of the current item loaded / no longer read.
    // S_FULL[h], P_FULL[h]: half h (64 query / key columns) of the tile's scores and products.
    // ACC_FULL / ACC_EMPTY: the item's accumulators complete / read out by the epilogue.
    // ITEM_FULL[s] / ITEM_EMPTY[s]: the two-slot ring of claimed items.
    enum {
        B_RES = 0,
        B_RESE,
        B_FULL,
        B_EMPTY = B_FULL + NST,
        B_SFULL = B_EMPTY + NST,
        B_PFULL = B_SFULL + 2,
        B_ACCF = B_PFULL + 2,
        B_ACCE,
        B_DRAIN,
        B_ITEMF,
        B_ITEME = B_ITEMF + 2,
        NBAR = B_ITEME + 2
    };
    static constexpr int MISC_OFF = BAR_OFF + NBAR * 8;   // [0] tmem base, [1] abort, [4..5] item by slot
    // At least 120 KB, so that one CTA occupies an SM: each CTA allocates all
    // 512 TMEM columns, and a second one would wait inside tcgen05.alloc.
    static constexpr int SMEM_USED = MISC_OFF + 32 + 1024;   // misc words [0..5], + slack to align the base to 1 KB
    static constexpr int SMEM_BYTES = SMEM_USED > 120 * 1024 ? SMEM_USED : 120 * 1024;
    static constexpr uint32_t S_COL = 0, DP_COL = 128, ACC0_COL = 256, ACC1_COL = 256 + D;
    static constexpr uint32_t TMEM_COLS = 512;
    // kind::f16, fp32 accumulate, bf16 A and B, N >> 3 at 17, M >> 4 at 24
    // Half a tile: 64 rows of the streamed operand (N of the score products, K of the
    // gradient products), 8 KB into each 128B-swizzled box.
    static constexpr int HALF = TILE / 2;
    static constexpr int HALF_BYTES = HALF * 128;
    static constexpr uint32_t IDESC_SS = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(HALF >> 3) << 17) |
                                         ((uint32_t)(TILE >> 4) << 24);   // M = 128, N = 64
    static constexpr uint32_t IDESC_TS = (1u << 4) | (1u << 7) | (1u << 10) | (1u << 16) |
                                         ((uint32_t)(D >> 3) << 17) | ((uint32_t)(TILE >> 4) << 24);
};

// A 128-row tile of one side with the global position of its first row.
struct BTile {
    long long row0;
    int len;
    long long pos0;
    int chunk;
};

__device__ __forceinline__ BTile btile(const BwdArgs &a, int t, bool is_q) {
    BTile x;
    if (!a.ring) {
        const int L = is_q ? a.Lq : a.Lk;
        x.row0 = (long long)t * TILE;
        x.len = min(TILE, L - (int)x.row0);
        x.pos0 = x.row0 + (is_q ? a.q_off : a.k_off);
        x.chunk = 0;
    } else {
        const int per = (a.CL + TILE - 1) / TILE;
        x.chunk = t / per;
        const int r = (t % per) * TILE;
        x.row0 = (long long)x.chunk * a.CL + r;
        x.len = min(TILE, a.CL - r);
        x.pos0 = x.row0;
    }
    return x;
}

__device__ __forceinline__ int n_tiles_side(const BwdArgs &a, bool is_q) {
    if (a.ring) return a.NC * ((a.CL + TILE - 1) / TILE);
    return ((is_q ? a.Lq : a.Lk) + TILE - 1) / TILE;
}

// Work item w of a persistent backward kernel -> (own tile, b * H + h).  Items are
// grouped by heads_per_group (b, h) pairs so that concurrently running CTAs share
// the streamed side in L2; within a group they come heaviest first under causal
// masking: the earliest key tiles (dK/dV: every later query sees them), the latest
// query tiles (dQ: they see every earlier key).
__device__ __forceinline__ void bwd_item(const BwdArgs &a, int w, int n_side, bool own_is_q, int &tile, int &bh) {
    const int BH = a.B * a.H, G = a.heads_per_group > 0 ? a.heads_per_group : 1;
    const int per_group = G * n_side;
    const int grp = w / per_group, rem = w % per_group;
    const int g_heads = BH - grp * G < G ? BH - grp * G : G;   // last group may be short
    const int lvl = rem / g_heads;
    bh = grp * G + rem % g_heads;
    tile = own_is_q ? n_side - 1 - lvl : lvl;
}

// Walk over the partner tiles of an own tile: the rows of the other side that
// the covered ring steps pair it with (block mode: the whole other side), cut
// into 128-row tiles, with causal clipping.  Every role of a CTA runs the same
// walk.
struct PWalk {
    int step, span;
    long long row, row_end, dpos;
    bool open;
};

__device__ __forceinline__ bool pwalk_span(const BwdArgs &a, const BTile &own, bool own_is_key, PWalk &w) {
    // set [row, row_end) to span `w.span` of step `w.step`; false when the walk is over
    for (;;) {
        const int nsteps = a.ring ? a.s_end - a.s_begin : 1;
        if (w.step >= nsteps) return false;
        long long r0, r1, dpos;
        if (!a.ring) {
            if (w.span > 0) {
                ++w.step;
                w.span = 0;
                continue;
            }
            r0 = 0;
            r1 = own_is_key ? a.Lq : a.Lk;
            dpos = own_is_key ? a.q_off : a.k_off;
        } else {
            const int nsp = a.zigzag ? 2 : 1;
            if (w.span >= nsp) {
                ++w.step;
                w.span = 0;
                continue;
            }
            const int me = !a.zigzag ? own.chunk : (own.chunk < a.P ? own.chunk : 2 * a.P - 1 - own.chunk);
            const int s = a.s_begin + w.step;
            // keys of rank src meet the queries of rank (src + s) mod P;
            // queries of rank r meet the keys of rank (r - s) mod P
            const int other = own_is_key ? (me + s) % a.P : ((me - s) % a.P + a.P) % a.P;
            const int c = w.span == 0 ? other : 2 * a.P - 1 - other;
            r0 = (long long)c * a.CL;
            r1 = r0 + a.CL;
            dpos = 0;
        }
        if (a.causal) {
            if (own_is_key) {   // queries before the first key see none of the tile
                const long long lo = own.pos0 - dpos;
                if (r0 < lo) r0 = lo;
            } else {            // keys after the last query are seen by none of it
                const long long hi = own.pos0 + own.len - dpos;
                if (r1 > hi) r1 = hi;
            }
        }
        w.row = r0;
        w.row_end = r1;
        w.dpos = dpos;
        if (r0 < r1) return true;
        ++w.span;
    }
}

__device__ __forceinline__ void pwalk_begin(const BwdArgs &a, const BTile &own, bool own_is_key, PWalk &w) {
    w.step = 0;
    w.span = 0;
    w.open = pwalk_span(a, own, own_is_key, w);
}

// Next partner tile into p; false at the end.
__device__ __forceinline__ bool pwalk_next(const BwdArgs &a, const BTile &own, bool own_is_key, PWalk &w,
                                           BTile &p) {
    while (w.open) {
        if (w.row < w.row_end) {
            p.row0 = w.row;
            p.len = (int)min((long long)TILE, w.row_end - w.row);
            p.pos0 = w.row + w.dpos;
            p.chunk = 0;
            w.row += TILE;
            return true;
        }
        ++w.span;
        w.open = pwalk_span(a, own, own_is_key, w);
    }
    return false;
}

__device__ __forceinline__ bool bexcluded(const BwdArgs &a, int b, long long qp, long long kp) {
    if (a.causal && kp > qp) return true;
    if (a.kpm && a.kpm[b * a.kpm_ld + kp]) return true;
    if (a.am && a.am[qp * a.am_ld + kp]) return true;
    return false;
}

// Visibility of 32 pairs as a bit mask (bit i: pair i is kept), for the tiles
// that need exclusions.  Kept out of line: inlined into the unrolled elementwise
// loops it made them too large for the instruction cache.
// Key fixed (dK/dV kernel): queries q0 + i, i < 32, of which the first n exist.
__device__ __noinline__ uint32_t keep_bits_queries(const BwdArgs &a, int b, long long q0, int n, long long kp,
                                                   bool kvalid) {
    uint32_t m = 0;
    if (!kvalid) return 0;
    for (int i = 0; i < 32 && i < n; ++i)
        if (!bexcluded(a, b, q0 + i, kp)) m |= 1u << i;
    return m;
}
// Query fixed (dQ kernel): keys k0 + i, i < 32, of which the first n exist.
__device__ __noinline__ uint32_t keep_bits_keys(const BwdArgs &a, int b, long long qp, bool qvalid, long long k0,
                                                int n) {
    uint32_t m = 0;
    if (!qvalid) return 0;
    for (int i = 0; i < 32 && i < n; ++i)
        if (!bexcluded(a, b, qp, k0 + i)) m |= 1u << i;
    return m;
}

// Four consecutive floats of shared memory (16-byte aligned address).
__device__ __forceinline__ float4 lds4(uint32_t saddr) {
    float4 v;
    asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(saddr));
    return v;
}

// Common prologue: barriers, TMEM, tensor-map prefetch.  Returns the TMEM base.
template <int D>
__device__ __forceinline__ uint32_t bwd_prologue(uint32_t bars, volatile uint32_t *misc, uint32_t misc_addr,
                                                 int full_count, const CUtensorMap *m0, const CUtensorMap *m1,
                                                 const CUtensorMap *m2, const CUtensorMap *m3) {
    using C = BCfg<D>;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    auto bar = [&](int i) { return bars + 8u * (uint32_t)i; };
    if (threadIdx.x == 0) {
        mbar_init(bar(C::B_RES), 1);
        mbar_init(bar(C::B_RESE), 1);
        for (int i = 0; i < C::NST; ++i) {
            mbar_init(bar(C::B_FULL + i), full_count);
            mbar_init(bar(C::B_EMPTY + i), 1);
        }
        for (int hh = 0; hh < 2; ++hh) {
            mbar_init(bar(C::B_SFULL + hh), 1);
            mbar_init(bar(C::B_PFULL + hh), 128);
        }
        mbar_init(bar(C::B_ACCF), 1);
        mbar_init(bar(C::B_ACCE), 256);   // every elementwise thread (both groups) after its epilogue
        mbar_init(bar(C::B_DRAIN), 1);
        for (int i = 0; i < 2; ++i) {
            mbar_init(bar(C::B_ITEMF + i), 1);
            mbar_init(bar(C::B_ITEME + i), 1 + 8);   // MMA warp + one lane per elementwise warp
        }
        misc[1] = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(misc_addr),
                     "r"(C::TMEM_COLS)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    if (warp == 0 && lane == 0) {
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(m0)) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(m1)) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(m2)) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(m3)) : "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    return misc[0];
}

// 128 rows of one tensor (all its 64-column boxes) at row `row0` of (b, h).
template <int D>
__device__ __forceinline__ void tma_tile(uint32_t dst, const CUtensorMap *map, long long row0, int h, int b,
                                         uint32_t bar) {
    using C = BCfg<D>;
#pragma unroll
    for (int bx = 0; bx < C::NBOX; ++bx) tma_load_4d(dst + bx * C::BOX_BYTES, map, bx * 64, (int)row0, h, b, bar);
}

// The elementwise warps' epilogue: D fp32 columns of one TMEM lane to a global
// row.  Every lane of the warp executes the (warp-collective) TMEM loads; only
// lanes with a valid row store.
template <int D>
__device__ __forceinline__ void store_acc_row(uint32_t taddr, float *dst, float mul, bool acc, bool valid,
                                              int c_begin = 0, int c_end = D / 32) {
#pragma unroll
    for (int c = 0; c < D / 32; ++c) {
        if (c < c_begin || c >= c_end) continue;
        uint32_t r[32];
        tmem_ld32(taddr + c * 32, r);
        tmem_wait_ld();
        if (!valid) continue;
        float4 *o = reinterpret_cast<float4 *>(dst + c * 32);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            float4 v = make_float4(__uint_as_float(r[4 * i]) * mul, __uint_as_float(r[4 * i + 1]) * mul,
                                   __uint_as_float(r[4 * i + 2]) * mul, __uint_as_float(r[4 * i + 3]) * mul);
            if (acc) {
                const float4 old = o[i];
                v.x += old.x;
                v.y += old.y;
                v.z += old.z;
                v.w += old.w;
            }
            o[i] = v;
        }
    }
}

// ---------------------------------------------------------------------------
// dK, dV
// ---------------------------------------------------------------------------

template <int D>
__global__ void __launch_bounds__(384, 1)
    bwd_dkdv_tc_kernel(const BwdArgs a, const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                       const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap tdo) {
    using C = BCfg<D>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_base = smem_u32(smem_raw);
    const uint32_t base = (raw_base + 1023u) & ~1023u;
    uint8_t *gbase = smem_raw + (base - raw_base);
    const uint32_t bars = base + C::BAR_OFF;
    auto bar = [&](int i) { return bars + 8u * (uint32_t)i; };
    volatile uint32_t *misc = reinterpret_cast<volatile uint32_t *>(gbase + C::MISC_OFF);
    volatile int *abort = reinterpret_cast<volatile int *>(gbase + C::MISC_OFF + 4);
    const uint32_t sK = base + C::RES_OFF, sV = sK + C::TILE_BYTES;
    auto stage = [&](int st) { return base + C::STG_OFF + (uint32_t)st * C::STG_BYTES; };
    auto vec = [&](int st) {
        return reinterpret_cast<float *>(gbase + C::STG_OFF + st * C::STG_BYTES + C::VEC_OFF);
    };

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const long long q_rows = a.ring ? a.T : a.Lq;
    const int n_side = n_tiles_side(a, false), n_items = n_side * a.B * a.H;
    const uint64_t lim = a.wait_limit_ns;
    const uint32_t tmem = bwd_prologue<D>(bars, misc, base + C::MISC_OFF, 32, &tq, &tk, &tv, &tdo);

    if (warp == 0) {
        // ------------------------------------------------------------ producer (all lanes)
        // Claims key tiles (items) from the launch's counter, publishes them, loads the
        // item's resident K / V once the previous item's score products are done with
        // them, then streams the query tiles of its walk (Q, dout, and the rows' LSE / D).
        bool ok = true;
        uint32_t fills = 0, loads = 0;
        int w = 0;
        if (lane == 0) w = (int)atomicAdd(a.sched, 1u);
        w = __shfl_sync(0xffffffffu, w, 0);
        for (uint32_t it = 0;; ++it) {
            const uint32_t sl = it & 1;
            if (it >= 2 && !warp_wait(bar(C::B_ITEME + sl), ((it >> 1) - 1) & 1, abort, a.err, lim)) {
                ok = false;
                break;
            }
            if (w >= n_items) {
                if (lane == 0) misc[4 + sl] = 0xffffffffu;   // end of work
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(C::B_ITEMF + sl));
                break;
            }
            int ktile, bh;
            bwd_item(a, w, n_side, false, ktile, bh);
            const int b = bh / a.H, h = bh % a.H;
            const BTile kt = btile(a, ktile, false);
            if (lane == 0) misc[4 + sl] = (uint32_t)w;
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(C::B_ITEMF + sl));
            if (it > 0 && !warp_wait(bar(C::B_RESE), (it - 1) & 1, abort, a.err, lim)) {
                ok = false;
                break;
            }
            if (lane == 0) {
                mbar_arrive_expect_tx(bar(C::B_RES), 2 * C::TILE_BYTES);
                tma_tile<D>(sK, &tk, kt.row0, h, b, bar(C::B_RES));
                tma_tile<D>(sV, &tv, kt.row0, h, b, bar(C::B_RES));
            }
            ++loads;
            PWalk pw;
            pwalk_begin(a, kt, true, pw);
            BTile pt;
            while (ok && pwalk_next(a, kt, true, pw, pt)) {
                const int st = fills % C::NST;
                const uint32_t use = fills / C::NST;
                if (use > 0 && !warp_wait(bar(C::B_EMPTY + st), (use - 1) & 1, abort, a.err, lim)) {
                    ok = false;
                    break;
                }
                float *lse2 = vec(st), *dd = lse2 + TILE;
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int c = lane * 4 + i;
                    float L = -INFINITY, Dv = 0.f;
                    if (c < pt.len) {
                        const long long row = (long long)bh * q_rows + pt.row0 + c;
                        L = a.lse[row];
                        Dv = a.D[row];
                    }
                    // -LSE in log2 units; -inf makes p = exp2(x + nlse2) exactly 0 for rows
                    // past the tile and rows without keys
                    lse2[c] = L == -INFINITY ? -INFINITY : -L * 1.4426950408889634f;
                    dd[c] = Dv;
                }
                if (lane == 0) {
                    mbar_arrive_expect_tx(bar(C::B_FULL + st), 2 * C::TILE_BYTES);
                    tma_tile<D>(stage(st), &tq, pt.row0, h, b, bar(C::B_FULL + st));
                    tma_tile<D>(stage(st) + C::TILE_BYTES, &tdo, pt.row0, h, b, bar(C::B_FULL + st));
                } else {
                    mbar_arrive(bar(C::B_FULL + st));
                }
                ++fills;
            }
            if (!ok) break;
            if (lane == 0) w = (int)atomicAdd(a.sched, 1u);
            w = __shfl_sync(0xffffffffu, w, 0);
        }
        if (!ok && lane == 0) {
            // Let the copies already issued land before the CTA exits.
            volatile int never = 0;
            if (loads > 0) mbar_wait(bar(C::B_RES), (loads - 1) & 1, &never, nullptr, 200000000ull);
            for (uint32_t i = 0; i < (uint32_t)C::NST && i < fills; ++i) {
                const uint32_t last = fills - 1 - i;
                mbar_wait(bar(C::B_FULL + last % C::NST), (last / C::NST) & 1, &never, nullptr, 200000000ull);
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer (converged)
        // Each query tile is taken in two halves of 64 queries.  Per tile t:
        // dV, dK += half 0 (once the elementwise warps stored its P^T, dS^T), then the
        // next tile's half-0 scores, then dV, dK += half 1, then the next tile's
        // half-1 scores: the scores of one half are computed while the elementwise
        // warps work on the other.  Half h of S^T / dP^T lives in columns
        // [64 h, 64 h + 64) of its region and its bf16 P^T / dS^T in the first 32 of
        // them, so the next tile's half 0 never touches what half 1 still needs.
        // Across items: RES_EMPTY is committed after an item's last score products
        // (the producer may then load the next item's K / V), ACC_FULL after its last
        // gradient products, and an item's first gradient products wait for ACC_EMPTY
        // of the previous one (its epilogue has read the accumulators).
        bool ok = true;
        const uint64_t kdesc = sdesc(sK, 16, 1024), vdesc = sdesc(sV, 16, 1024);   // K-major A operands
        // S^T_h = K Q_h^T and dP^T_h = V dout_h^T (fp32 into TMEM) for the tile in stage st
        auto scores = [&](int st, int hh) {
            const uint32_t sQ = stage(st) + hh * C::HALF_BYTES, sDO = stage(st) + C::TILE_BYTES + hh * C::HALF_BYTES;
            const uint64_t qk = sdesc(sQ, 16, 1024), dok = sdesc(sDO, 16, 1024);   // K-major B operands
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
                const uint64_t off = (uint64_t)(((kk >> 2) * C::BOX_BYTES + (kk & 3) * 32) >> 4);
                mma_ss_one(tmem + C::S_COL + hh * C::HALF, kdesc + off, qk + off, C::IDESC_SS, kk > 0 ? 1u : 0u);
            }
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
                const uint64_t off = (uint64_t)(((kk >> 2) * C::BOX_BYTES + (kk & 3) * 32) >> 4);
                mma_ss_one(tmem + C::DP_COL + hh * C::HALF, vdesc + off, dok + off, C::IDESC_SS, kk > 0 ? 1u : 0u);
            }
            mma_commit_one(bar(C::B_SFULL + hh));
        };
        // dV += P^T_h dout_h and dK += dS^T_h q_h for the tile in stage st
        auto grads = [&](int st, int hh, uint32_t t, bool first) -> bool {
            if (!warp_wait(bar(C::B_PFULL + hh), t & 1, abort, a.err, lim)) return false;
            tc_fence_after();   // P^T and dS^T were written by the elementwise warps' tcgen05.st
            const uint32_t sQ = stage(st), sDO = stage(st) + C::TILE_BYTES;
            const uint64_t don = sdesc(sDO, C::BOX_BYTES, 1024), qn = sdesc(sQ, C::BOX_BYTES, 1024);   // MN-major B
#pragma unroll
            for (int kk = 0; kk < C::HALF / 16; ++kk)
                mma_ts_one(tmem + C::ACC0_COL, tmem + C::S_COL + hh * C::HALF + kk * 8,
                           don + (uint64_t)((hh * C::HALF_BYTES + kk * 2048) >> 4), C::IDESC_TS,
                           (first && kk == 0) ? 0u : 1u);   // dV += P^T dout
#pragma unroll
            for (int kk = 0; kk < C::HALF / 16; ++kk)
                mma_ts_one(tmem + C::ACC1_COL, tmem + C::DP_COL + hh * C::HALF + kk * 8,
                           qn + (uint64_t)((hh * C::HALF_BYTES + kk * 2048) >> 4), C::IDESC_TS,
                           (first && kk == 0) ? 0u : 1u);   // dK += dS^T q
            return true;
        };
        uint32_t t = 0;   // query tiles so far, over all items (stage and barrier phases)
        for (uint32_t it = 0;; ++it) {
            const uint32_t sl = it & 1;
            if (!warp_wait(bar(C::B_ITEMF + sl), (it >> 1) & 1, abort, a.err, lim)) {
                ok = false;
                break;
            }
            const uint32_t w = misc[4 + sl];
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(C::B_ITEME + sl));
            if (w == 0xffffffffu) break;
            int ktile, bh;
            bwd_item(a, (int)w, n_side, false, ktile, bh);
            const BTile kt = btile(a, ktile, false);
            if (!warp_wait(bar(C::B_RES), it & 1, abort, a.err, lim)) {
                ok = false;
                break;
            }
            PWalk pw;
            pwalk_begin(a, kt, true, pw);
            BTile pt;
            bool have = pwalk_next(a, kt, true, pw, pt);
            if (!have) {
                // no query sees this key tile: the accumulators are not touched
                mma_commit_one(bar(C::B_RESE));
                if (it > 0 && !(ok = warp_wait(bar(C::B_ACCE), (it - 1) & 1, abort, a.err, lim))) break;
                mma_commit_one(bar(C::B_ACCF));
                continue;
            }
            if (!(ok = warp_wait(bar(C::B_FULL + t % C::NST), (t / C::NST) & 1, abort, a.err, lim))) break;
            scores(t % C::NST, 0);
            scores(t % C::NST, 1);
            bool first = true;
            while (have) {
                const int st = t % C::NST, stn = (t + 1) % C::NST;
                const bool more = pwalk_next(a, kt, true, pw, pt);
                if (!more) mma_commit_one(bar(C::B_RESE));   // the item's last score products are issued
                if (first && it > 0 && !(ok = warp_wait(bar(C::B_ACCE), (it - 1) & 1, abort, a.err, lim))) break;
                if (!(ok = grads(st, 0, t, first))) break;
                first = false;
                if (more) {
                    if (!(ok = warp_wait(bar(C::B_FULL + stn), ((t + 1) / C::NST) & 1, abort, a.err, lim))) break;
                    scores(stn, 0);
                }
                if (!(ok = grads(st, 1, t, false))) break;
                mma_commit_one(bar(C::B_EMPTY + st));
                if (more) scores(stn, 1);
                ++t;
                have = more;
            }
            if (!ok) break;
            mma_commit_one(bar(C::B_ACCF));
        }
        if (!ok) {
            volatile int never = 0;
            mma_commit_one(bar(C::B_DRAIN));
            warp_wait(bar(C::B_DRAIN), 0, &never, nullptr, 200000000ull);
        }
        __syncwarp();
    } else if (warp >= 4) {
        // ------------------------------------------------------------ elementwise + epilogue
        const int j = (warp & 3) * 32 + lane;               // key row of the tile (TMEM lane)
        const uint32_t lane_addr = (uint32_t)((warp & 3) * 32) << 16;
        const int grp = (warp - 4) >> 2;                    // group: half grp of every partner tile
        const float sl2 = a.scale * 1.4426950408889634f;
        bool ok = true;
        uint32_t t = 0;   // query tiles so far, over all items
        for (uint32_t it = 0;; ++it) {
            const uint32_t sl = it & 1;
            if (!warp_wait(bar(C::B_ITEMF + sl), (it >> 1) & 1, abort, a.err, lim)) {
                ok = false;
                break;
            }
            const uint32_t w = misc[4 + sl];
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(C::B_ITEME + sl));
            if (w == 0xffffffffu) break;
            int ktile, bh;
            bwd_item(a, (int)w, n_side, false, ktile, bh);
            const int b = bh / a.H;
            const BTile kt = btile(a, ktile, false);
            const bool jvalid = j < kt.len;
            const long long kp = kt.pos0 + j;
            uint32_t n_done = 0;   // query tiles of this item (the same for every lane)
            PWalk pw;
            pwalk_begin(a, kt, true, pw);
            BTile pt;
            while (ok && pwalk_next(a, kt, true, pw, pt)) {
                const int st = t % C::NST;
                const uint32_t s_nlse = smem_u32(vec(st)), s_dd = s_nlse + TILE * 4;   // -LSE log2 units, D
                const bool full = kt.len == TILE && pt.len == TILE && !a.kpm && !a.am &&
                                  (!a.causal || kt.pos0 + TILE - 1 <= pt.pos0);
#pragma unroll 1
                for (int c = 2 * grp; c < 2 * grp + 2; ++c) {
                    const int hh = c >> 1;   // half of the tile: queries [64 hh, 64 hh + 64)
                    if ((c & 1) == 0) {
                        if (!warp_wait(bar(C::B_SFULL + hh), t & 1, abort, a.err, lim)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                    }
                    uint32_t rs[32], rd[32];
                    tmem_ld32(tmem + lane_addr + C::S_COL + c * 32, rs);
                    tmem_ld32(tmem + lane_addr + C::DP_COL + c * 32, rd);
                    tmem_wait_ld();
                    const uint32_t keep =
                        full ? 0xffffffffu
                             : keep_bits_queries(a, b, pt.pos0 + c * 32, pt.len - c * 32, kp, jvalid);
                    uint32_t pp[16], pd[16];
#pragma unroll
                    for (int q4 = 0; q4 < 8; ++q4) {
                        const float4 nl = lds4(s_nlse + (c * 32 + q4 * 4) * 4);
                        const float4 d4 = lds4(s_dd + (c * 32 + q4 * 4) * 4);
                        const float nlv[4] = {nl.x, nl.y, nl.z, nl.w}, ddv[4] = {d4.x, d4.y, d4.z, d4.w};
                        float pv[4], dv[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const int i = q4 * 4 + e;
                            float p = fast_exp2(fmaf(__uint_as_float(rs[i]), sl2, nlv[e]));
                            p = (keep >> i) & 1u ? p : 0.f;   // columns past the partner tile are never kept
                            pv[e] = p;
                            dv[e] = p * (__uint_as_float(rd[i]) - ddv[e]);
                        }
                        pp[q4 * 2] = pack_bf16(pv[0], pv[1]);
                        pp[q4 * 2 + 1] = pack_bf16(pv[2], pv[3]);
                        pd[q4 * 2] = pack_bf16(dv[0], dv[1]);
                        pd[q4 * 2 + 1] = pack_bf16(dv[2], dv[3]);
                    }
                    // P^T / dS^T of these 32 queries into 16 columns of this half that the
                    // earlier chunk of the half has read
                    const uint32_t pcol = hh * C::HALF + (c & 1) * 16;
                    tmem_st16(tmem + lane_addr + C::S_COL + pcol, pp);
                    tmem_st16(tmem + lane_addr + C::DP_COL + pcol, pd);
                    if (c & 1) {
                        tmem_wait_st();
                        tc_fence_before();
                        mbar_arrive(bar(C::B_PFULL + hh));
                    }
                }
                if (!ok) break;
                ++t;
                ++n_done;
            }
            if (!ok) break;
            // epilogue of the item: the accumulators to dV / dK rows, then hand them back
            if (!warp_wait(bar(C::B_ACCF), it & 1, abort, a.err, lim)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const long long row = ((long long)bh * (a.ring ? a.T : a.Lk) + kt.row0 + j) * D;
            // group 0 writes the dV rows, group 1 the dK rows
            if (n_done > 0) {   // the same for every lane: the TMEM loads below stay warp-collective
                if (grp == 0)
                    store_acc_row<D>(tmem + lane_addr + C::ACC0_COL, a.dv + row, 1.f, a.accumulate != 0, jvalid);
                else
                    store_acc_row<D>(tmem + lane_addr + C::ACC1_COL, a.dk + row, a.scale, a.accumulate != 0, jvalid);
            } else if (jvalid && !a.accumulate) {
                float *dst = grp == 0 ? a.dv : a.dk;
                for (int c = 0; c < D; ++c) dst[row + c] = 0.f;
            }
            tc_fence_before();
            mbar_arrive(bar(C::B_ACCE));
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(C::TMEM_COLS)
                     : "memory");
}

// ---------------------------------------------------------------------------
// dQ
// ---------------------------------------------------------------------------

template <int D>
__global__ void __launch_bounds__(384, 1)
    bwd_dq_tc_kernel(const BwdArgs a, const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                     const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap tdo) {
    using C = BCfg<D>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_base = smem_u32(smem_raw);
    const uint32_t base = (raw_base + 1023u) & ~1023u;
    uint8_t *gbase = smem_raw + (base - raw_base);
    const uint32_t bars = base + C::BAR_OFF;
    auto bar = [&](int i) { return bars + 8u * (uint32_t)i; };
    volatile uint32_t *misc = reinterpret_cast<volatile uint32_t *>(gbase + C::MISC_OFF);
    volatile int *abort = reinterpret_cast<volatile int *>(gbase + C::MISC_OFF + 4);
    const uint32_t sQ = base + C::RES_OFF, sDO = sQ + C::TILE_BYTES;
    auto stage = [&](int st) { return base + C::STG_OFF + (uint32_t)st * C::STG_BYTES; };

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const long long q_rows = a.ring ? a.T : a.Lq;
    const int n_side = n_tiles_side(a, true), n_items = n_side * a.B * a.H;
    const uint64_t lim = a.wait_limit_ns;
    const uint32_t tmem = bwd_prologue<D>(bars, misc, base + C::MISC_OFF, 1, &tq, &tk, &tv, &tdo);

    if (warp == 0) {
        // ------------------------------------------------------------ producer (one lane)
        // Claims query tiles (items), publishes them, loads the item's resident Q / dout
        // once the previous item's score products are done with them, then streams the
        // K / V tiles of its walk.
        if (lane == 0) {
            bool ok = true;
            uint32_t fills = 0, loads = 0;
            int w = (int)atomicAdd(a.sched + 1, 1u);
            for (uint32_t it = 0;; ++it) {
                const uint32_t sl = it & 1;
                if (it >= 2 && !mbar_wait(bar(C::B_ITEME + sl), ((it >> 1) - 1) & 1, abort, a.err, lim)) {
                    ok = false;
                    break;
                }
                if (w >= n_items) {
                    misc[4 + sl] = 0xffffffffu;   // end of work
                    mbar_arrive(bar(C::B_ITEMF + sl));
                    break;
                }
                int qtile, bh;
                bwd_item(a, w, n_side, true, qtile, bh);
                const int b = bh / a.H, h = bh % a.H;
                const BTile qt = btile(a, qtile, true);
                misc[4 + sl] = (uint32_t)w;
                mbar_arrive(bar(C::B_ITEMF + sl));
                if (it > 0 && !mbar_wait(bar(C::B_RESE), (it - 1) & 1, abort, a.err, lim)) {
                    ok = false;
                    break;
                }
                mbar_arrive_expect_tx(bar(C::B_RES), 2 * C::TILE_BYTES);
                tma_tile<D>(sQ, &tq, qt.row0, h, b, bar(C::B_RES));
                tma_tile<D>(sDO, &tdo, qt.row0, h, b, bar(C::B_RES));
                ++loads;
                PWalk pw;
                pwalk_begin(a, qt, false, pw);
                BTile pt;
                while (pwalk_next(a, qt, false, pw, pt)) {
                    const int st = fills % C::NST;
                    const uint32_t use = fills / C::NST;
                    if (use > 0 && !mbar_wait(bar(C::B_EMPTY + st), (use - 1) & 1, abort, a.err, lim)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(bar(C::B_FULL + st), 2 * C::TILE_BYTES);
                    tma_tile<D>(stage(st), &tk, pt.row0, h, b, bar(C::B_FULL + st));
                    tma_tile<D>(stage(st) + C::TILE_BYTES, &tv, pt.row0, h, b, bar(C::B_FULL + st));
                    ++fills;
                }
                if (!ok) break;
                w = (int)atomicAdd(a.sched + 1, 1u);
            }
            if (!ok) {
                // Let the copies already issued land before the CTA exits.
                volatile int never = 0;
                if (loads > 0) mbar_wait(bar(C::B_RES), (loads - 1) & 1, &never, nullptr, 200000000ull);
                for (uint32_t i = 0; i < (uint32_t)C::NST && i < fills; ++i) {
                    const uint32_t last = fills - 1 - i;
                    mbar_wait(bar(C::B_FULL + last % C::NST), (last / C::NST) & 1, &never, nullptr, 200000000ull);
                }
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer (converged)
        // Each key tile is taken in two halves of 64 keys, in the order of the dK/dV
        // kernel: dQ += half 0, the next tile's half-0 scores, dQ += half 1, the next
        // tile's half-1 scores.  Half h of S / dP lives in columns [64 h, 64 h + 64)
        // of its region and its bf16 dS in the first 32 of them.  Across items as in
        // the dK/dV kernel (RES_EMPTY, ACC_FULL, ACC_EMPTY).
        bool ok = true;
        const uint64_t qdesc = sdesc(sQ, 16, 1024), dodesc = sdesc(sDO, 16, 1024);   // K-major A operands
        // S_h = Q K_h^T and dP_h = dout V_h^T for the tile in stage st
        auto scores = [&](int st, int hh) {
            const uint32_t sK = stage(st) + hh * C::HALF_BYTES, sV = stage(st) + C::TILE_BYTES + hh * C::HALF_BYTES;
            const uint64_t kk_ = sdesc(sK, 16, 1024), vk = sdesc(sV, 16, 1024);   // K-major B operands
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
                const uint64_t off = (uint64_t)(((kk >> 2) * C::BOX_BYTES + (kk & 3) * 32) >> 4);
                mma_ss_one(tmem + C::S_COL + hh * C::HALF, qdesc + off, kk_ + off, C::IDESC_SS, kk > 0 ? 1u : 0u);
            }
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
                const uint64_t off = (uint64_t)(((kk >> 2) * C::BOX_BYTES + (kk & 3) * 32) >> 4);
                mma_ss_one(tmem + C::DP_COL + hh * C::HALF, dodesc + off, vk + off, C::IDESC_SS, kk > 0 ? 1u : 0u);
            }
            mma_commit_one(bar(C::B_SFULL + hh));
        };
        // dQ += dS_h K_h for the tile in stage st
        auto grads = [&](int st, int hh, uint32_t t, bool first) -> bool {
            if (!warp_wait(bar(C::B_PFULL + hh), t & 1, abort, a.err, lim)) return false;
            tc_fence_after();   // dS was written by the elementwise warps' tcgen05.st
            const uint64_t kn = sdesc(stage(st), C::BOX_BYTES, 1024);   // K as the MN-major B operand
#pragma unroll
            for (int kk = 0; kk < C::HALF / 16; ++kk)
                mma_ts_one(tmem + C::ACC0_COL, tmem + C::S_COL + hh * C::HALF + kk * 8,
                           kn + (uint64_t)((hh * C::HALF_BYTES + kk * 2048) >> 4), C::IDESC_TS,
                           (first && kk == 0) ? 0u : 1u);   // dQ += dS K
            return true;
        };
        uint32_t t = 0;   // key tiles so far, over all items
        for (uint32_t it = 0;; ++it) {
            const uint32_t sl = it & 1;
            if (!warp_wait(bar(C::B_ITEMF + sl), (it >> 1) & 1, abort, a.err, lim)) {
                ok = false;
                break;
            }
            const uint32_t w = misc[4 + sl];
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(C::B_ITEME + sl));
            if (w == 0xffffffffu) break;
            int qtile, bh;
            bwd_item(a, (int)w, n_side, true, qtile, bh);
            const BTile qt = btile(a, qtile, true);
            if (!warp_wait(bar(C::B_RES), it & 1, abort, a.err, lim)) {
                ok = false;
                break;
            }
            PWalk pw;
            pwalk_begin(a, qt, false, pw);
            BTile pt;
            bool have = pwalk_next(a, qt, false, pw, pt);
            if (!have) {
                mma_commit_one(bar(C::B_RESE));
                if (it > 0 && !(ok = warp_wait(bar(C::B_ACCE), (it - 1) & 1, abort, a.err, lim))) break;
                mma_commit_one(bar(C::B_ACCF));
                continue;
            }
            if (!(ok = warp_wait(bar(C::B_FULL + t % C::NST), (t / C::NST) & 1, abort, a.err, lim))) break;
            scores(t % C::NST, 0);
            scores(t % C::NST, 1);
            bool first = true;
            while (have) {
                const int st = t % C::NST, stn = (t + 1) % C::NST;
                const bool more = pwalk_next(a, qt, false, pw, pt);
                if (!more) mma_commit_one(bar(C::B_RESE));   // the item's last score products are issued
                if (first && it > 0 && !(ok = warp_wait(bar(C::B_ACCE), (it - 1) & 1, abort, a.err, lim))) break;
                if (!(ok = grads(st, 0, t, first))) break;
                first = false;
                if (more) {
                    if (!(ok = warp_wait(bar(C::B_FULL + stn), ((t + 1) / C::NST) & 1, abort, a.err, lim))) break;
                    scores(stn, 0);
                }
                if (!(ok = grads(st, 1, t, false))) break;
                mma_commit_one(bar(C::B_EMPTY + st));
                if (more) scores(stn, 1);
                ++t;
                have = more;
            }
            if (!ok) break;
            mma_commit_one(bar(C::B_ACCF));
        }
        if (!ok) {
            volatile int never = 0;
            mma_commit_one(bar(C::B_DRAIN));
            warp_wait(bar(C::B_DRAIN), 0, &never, nullptr, 200000000ull);
        }
        __syncwarp();
    } else if (warp >= 4) {
        // ------------------------------------------------------------ elementwise + epilogue
        const int i = (warp & 3) * 32 + lane;               // query row of the tile (TMEM lane)
        const uint32_t lane_addr = (uint32_t)((warp & 3) * 32) << 16;
        const int grp = (warp - 4) >> 2;                    // group: half grp of every partner tile
        const float sl2 = a.scale * 1.4426950408889634f;
        bool ok = true;
        uint32_t t = 0;   // key tiles so far, over all items
        for (uint32_t it = 0;; ++it) {
            const uint32_t sl = it & 1;
            if (!warp_wait(bar(C::B_ITEMF + sl), (it >> 1) & 1, abort, a.err, lim)) {
                ok = false;
                break;
            }
            const uint32_t w = misc[4 + sl];
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(C::B_ITEME + sl));
            if (w == 0xffffffffu) break;
            int qtile, bh;
            bwd_item(a, (int)w, n_side, true, qtile, bh);
            const int b = bh / a.H;
            const BTile qt = btile(a, qtile, true);
            const bool ivalid = i < qt.len;
            const long long qp = qt.pos0 + i;
            float nlse2 = -INFINITY, Dv = 0.f;   // -LSE in log2 units (-inf: p = 0)
            if (ivalid) {
                const long long row = (long long)bh * q_rows + qt.row0 + i;
                const float L = a.lse[row];
                nlse2 = L == -INFINITY ? -INFINITY : -L * 1.4426950408889634f;
                Dv = a.D[row];
            }
            uint32_t n_done = 0;   // key tiles of this item (the same for every lane)
            PWalk pw;
            pwalk_begin(a, qt, false, pw);
            BTile pt;
            while (ok && pwalk_next(a, qt, false, pw, pt)) {
                const bool full = qt.len == TILE && pt.len == TILE && !a.kpm && !a.am &&
                                  (!a.causal || pt.pos0 + TILE - 1 <= qt.pos0);
#pragma unroll 1
                for (int c = 2 * grp; c < 2 * grp + 2; ++c) {
                    const int hh = c >> 1;   // half of the tile: keys [64 hh, 64 hh + 64)
                    if ((c & 1) == 0) {
                        if (!warp_wait(bar(C::B_SFULL + hh), t & 1, abort, a.err, lim)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                    }
                    uint32_t rs[32], rd[32];
                    tmem_ld32(tmem + lane_addr + C::S_COL + c * 32, rs);
                    tmem_ld32(tmem + lane_addr + C::DP_COL + c * 32, rd);
                    tmem_wait_ld();
                    const uint32_t keep =
                        full ? 0xffffffffu : keep_bits_keys(a, b, qp, ivalid, pt.pos0 + c * 32, pt.len - c * 32);
                    uint32_t pd[16];
#pragma unroll
                    for (int k2 = 0; k2 < 16; ++k2) {
                        float dv[2];
#pragma unroll
                        for (int e = 0; e < 2; ++e) {
                            const int k = 2 * k2 + e;
                            float p = fast_exp2(fmaf(__uint_as_float(rs[k]), sl2, nlse2));
                            p = (keep >> k) & 1u ? p : 0.f;
                            dv[e] = p * (__uint_as_float(rd[k]) - Dv);
                        }
                        pd[k2] = pack_bf16(dv[0], dv[1]);
                    }
                    // dS of these 32 keys into 16 columns of this half that the earlier
                    // chunk of the half has read
                    tmem_st16(tmem + lane_addr + C::S_COL + hh * C::HALF + (c & 1) * 16, pd);
                    if (c & 1) {
                        tmem_wait_st();
                        tc_fence_before();
                        mbar_arrive(bar(C::B_PFULL + hh));
                    }
                }
                if (!ok) break;
                ++t;
                ++n_done;
            }
            if (!ok) break;
            // epilogue of the item: the accumulator to dQ rows, then hand it back
            if (!warp_wait(bar(C::B_ACCF), it & 1, abort, a.err, lim)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const long long row = ((long long)bh * q_rows + qt.row0 + i) * D;
            // group g writes columns [g D/2, g D/2 + D/2) of the dQ rows
            if (n_done > 0)   // uniform: the TMEM loads stay warp-collective
                store_acc_row<D>(tmem + lane_addr + C::ACC0_COL, a.dq + row, a.scale, a.accumulate != 0, ivalid,
                                 grp * (D / 64), grp * (D / 64) + D / 64);
            else if (ivalid && !a.accumulate)
                for (int c = grp * (D / 2); c < grp * (D / 2) + D / 2; ++c) a.dq[row + c] = 0.f;
            tc_fence_before();
            mbar_arrive(bar(C::B_ACCE));
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(C::TMEM_COLS)
                     : "memory");
}

template <int D>
int launch_bwd_tc_d(const BwdArgs &a, const BwdMaps &m, int num_sms, cudaStream_t s) {
    using C = BCfg<D>;
    static_assert(C::SMEM_BYTES <= 232448, "shared memory budget");
    if (cudaFuncSetAttribute(bwd_dkdv_tc_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES) !=
            cudaSuccess ||
        cudaFuncSetAttribute(bwd_dq_tc_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES) !=
            cudaSuccess)
        return BA_ERR_CUDA;
    // CTAs claim (own tile, b, h) items from a zeroed counter, heaviest first.  Short
    // walks (fewer than 256 tiles per head): one persistent CTA per SM, the next item's
    // first score products overlapping the previous item's epilogue.  Long walks: one
    // CTA per item (each claims one and exits), which measured faster there.
    if (cudaMemsetAsync(a.sched, 0, 2 * sizeof(unsigned), s) != cudaSuccess) return BA_ERR_CUDA;
    const long long BH = (long long)a.B * a.H;
    const long long n_kt = a.ring ? (long long)a.NC * ((a.CL + TILE - 1) / TILE) : (a.Lk + TILE - 1) / TILE;
    const long long n_qt = a.ring ? (long long)a.NC * ((a.CL + TILE - 1) / TILE) : (a.Lq + TILE - 1) / TILE;
    if (n_kt * BH > 0x7fffffffLL || n_qt * BH > 0x7fffffffLL) return BA_ERR_SHAPE;
    const bool persistent = n_kt < 256 && n_qt < 256;
    const long long cap = persistent ? num_sms : 0x7fffffffLL;
    const int g_kv = (int)(n_kt * BH < cap ? n_kt * BH : cap);
    const int g_q = (int)(n_qt * BH < cap ? n_qt * BH : cap);
    if (g_kv > 0) bwd_dkdv_tc_kernel<D><<<g_kv, 384, C::SMEM_BYTES, s>>>(a, m.q, m.k, m.v, m.dout);
    if (g_q > 0) bwd_dq_tc_kernel<D><<<g_q, 384, C::SMEM_BYTES, s>>>(a, m.q, m.k, m.v, m.dout);
    return cudaGetLastError() == cudaSuccess ? BA_OK : BA_ERR_CUDA;
}

}  // namespace

bool bwd_tc_supported(int dtype, int d) { return dtype == BA_BF16 && (d == 64 || d == 128); }

// D pre-pass, then the dK/dV and dQ tensor-core kernels.
int launch_attn_bwd_tc(const BwdArgs &a, const BwdMaps &m, int num_sms, cudaStream_t s) {
    if ((long long)a.B * a.H == 0) return BA_OK;
    int rc = launch_bwd_pre(a, num_sms, s);
    if (rc) return rc;
    if (a.d == 128) return launch_bwd_tc_d<128>(a, m, num_sms, s);
    if (a.d == 64) return launch_bwd_tc_d<64>(a, m, num_sms, s);
    return BA_ERR_SHAPE;
}

}  // namespace ba
