// Shared device-side pieces of libblockattn: the work geometry (which query
// tiles exist, which key tiles each of them visits and in what order), the
// tile classes of the combined exclusion mask, and bounded mbarrier waits.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "blockattn.h"

namespace ba {

constexpr int TILE = 128;               // query rows and keys per tile
constexpr unsigned ERR_TIMEOUT_BIT = 1u;
constexpr float LOG2E = 1.4426950408889634f;
constexpr float LN2 = 0.6931471805599453f;

// ---------------------------------------------------------------------------
// Geometry
// ---------------------------------------------------------------------------
//
// Block mode (attn_block_fwd): query rows [0, Lq) of the q tensor are global
// positions q_off + i; keys [0, Lk) of k/v are global positions k_off + j.
// Tiles are cut every 128 rows from the block origin.
//
// Ring mode (ring_attn_fwd): q, k, v are (B, H, T, d) in global order.  T is
// cut into NC equal chunks of CL tokens (NC = P contiguous, 2P zigzag); rank r
// owns chunk r (contiguous) or chunks r and 2P-1-r (zigzag, local order as
// listed).  Tiles are cut every 128 tokens from each chunk start, so a chunk
// whose length is not a multiple of 128 ends in a ragged tile.  A query tile
// of rank r visits, for ring steps s in [s_begin, s_end), the key tiles of the
// chunks of rank (r - s) mod P in that rank's local order.
//
// Striped ring (striped = 1; brunomaga "When to use Ulysses and Ring
// attention" names Striped Attention): rank r owns the tokens t = r + P u,
// u = 0 .. CL-1 (NC = P, CL = T / P).  The walk then runs over "rows" in rank
// order, R = r CL + u, whose token is r + P u (row_token below): the tensor
// maps address the rows of a rank as a strided view, and out / lse are stored
// at the tokens.  Causality needs no global position: key (rank c, local u')
// is visible to query (rank r, local u) iff c + P u' <= r + P u, i.e. iff
// u' <= u when c <= r and u' < u when c > r.  So the walk's positions are
// local indices, a query at u and a key at u' + [c > r]: the block of every
// (rank, step) pair is the lower triangle with its diagonal (c <= r) or
// without it (c > r), and "key position <= query position" holds as in the
// other partitions.  Masks are indexed by token and are not taken here.
//
// The geometry functions below take the striped choice as a template
// parameter S (instantiated from g.striped by the launching code), so that the
// kernels of the other partitions compile without it.
struct Geom {
    int B, H, d;
    int ring;
    int striped;
    // block mode
    int Lq, Lk;
    long long q_off, k_off;
    // ring mode
    int T, P, zigzag, CL, NC, s_begin, s_end;
    // derived
    int nqt_pc, nkt_pc;      // tiles per q chunk / per k chunk
    int n_qtiles, n_ktiles;  // per (b, h)
    int heads_per_group;     // (b, h) pairs interleaved per group of work items
    int tail_levels;         // lightest query-tile levels dealt last, across all heads (0: none)
    int n_items;             // n_qtiles * B * H
    int causal;
    const uint8_t *kpm;
    long long kpm_ld;
    const uint8_t *am;
    long long am_ld;
    const int8_t *cls;       // (B, n_qtiles, n_ktiles) classes, or nullptr (causal only)
};

struct QTile {
    int g;              // q tile id within (b, h): 0 .. n_qtiles-1
    int row0, len;      // first row in the q tensor, valid rows (1..128)
    long long pos0;     // global position of the first row
    int rank;           // owning rank (ring mode)
    int b, h;
};

struct KTile {
    int idx;            // key tile id within (b, h): 0 .. n_ktiles-1
    int row0, len;      // first row in the k/v tensors, valid keys (1..128)
    long long pos0;     // global position of the first key
    int cls;            // BA_TILE_*
};

__host__ __device__ inline int ceil_div(int a, int b) { return (a + b - 1) / b; }

// Owner rank of chunk c.
__host__ __device__ inline int chunk_owner(const Geom &g, int c) {
    if (!g.zigzag) return c;
    return c < g.P ? c : 2 * g.P - 1 - c;
}

// Query tile with id qg (0 .. n_qtiles-1) of head (b, h).
template <bool S>
__host__ __device__ inline QTile q_tile(const Geom &g, int qg, int b, int h) {
    QTile t;
    t.g = qg;
    t.b = b;
    t.h = h;
    if (g.ring) {
        int c = qg / g.nqt_pc, i = qg % g.nqt_pc;
        t.row0 = c * g.CL + i * TILE;
        int end = (c + 1) * g.CL;
        t.len = (t.row0 + TILE < end ? t.row0 + TILE : end) - t.row0;
        t.pos0 = S ? i * TILE : t.row0;   // striped: local index within the rank
        t.rank = chunk_owner(g, c);
    } else {
        t.row0 = qg * TILE;
        t.len = (t.row0 + TILE < g.Lq ? t.row0 + TILE : g.Lq) - t.row0;
        t.pos0 = g.q_off + t.row0;
        t.rank = 0;
    }
    return t;
}

// Key tile with id kg (0 .. n_ktiles-1), geometry only (class not set).
__host__ __device__ inline KTile k_tile_by_id(const Geom &g, int kg) {
    KTile t;
    t.idx = kg;
    t.cls = BA_TILE_PARTIAL;
    if (g.ring) {
        int c = kg / g.nkt_pc, i = kg % g.nkt_pc;
        t.row0 = c * g.CL + i * TILE;
        int end = (c + 1) * g.CL;
        t.len = (t.row0 + TILE < end ? t.row0 + TILE : end) - t.row0;
        t.pos0 = t.row0;
    } else {
        t.row0 = kg * TILE;
        t.len = (t.row0 + TILE < g.Lk ? t.row0 + TILE : g.Lk) - t.row0;
        t.pos0 = g.k_off + t.row0;
    }
    return t;
}

// Incremental walk over the key tiles a query tile visits, in ring order,
// with EMPTY tiles skipped.  Every role of a kernel runs the same walk, so they
// agree on the sequence without communicating.  Without a class map, causal
// EMPTY tiles are skipped chunk-wise (a key tile, and every later tile of its
// chunk, is EMPTY once its first key lies after the query tile's last row).
// The state is kept in 32-bit integers and advanced by additions: the walk
// runs on the single MMA-issuing thread, where its latency is on the critical
// path of every tile.
struct KWalk {
    int row;        // first k/v row of the next tile
    int chunk_end;  // end row of the current chunk
    int idx;        // tile id of the next tile (class-map column)
    int s, ci, src; // ring step, chunk of the source rank, source rank
    int q_last;     // global position of the query tile's last row
    int q_first;    // global position of the query tile's first row
    int pos_off;    // global position = row + pos_off
    int qrank;      // rank of the query tile (ring mode)
};

// Position of the first key of chunk c for a query tile of rank qrank: its
// global position, or in the striped ring its local index 0 shifted by one
// when the key's rank follows the query's (see Geom).
template <bool S>
__host__ __device__ __forceinline__ int chunk_pos0(const Geom &g, int c, int qrank) {
    return S ? (c > qrank ? 1 : 0) : c * g.CL;
}

template <bool S>
__host__ __device__ __forceinline__ void kwalk_set_chunk(const Geom &g, KWalk &w, int c) {
    w.row = c * g.CL;
    w.chunk_end = w.row + g.CL;
    w.idx = c * g.nkt_pc;
    w.pos_off = chunk_pos0<S>(g, c, w.qrank) - w.row;
}

template <bool S>
__host__ __device__ __forceinline__ void kwalk_begin(const Geom &g, const QTile &q, KWalk &w) {
    w.q_first = (int)q.pos0;
    w.q_last = (int)q.pos0 + q.len - 1;
    w.ci = 0;
    w.qrank = q.rank;
    if (g.ring) {
        w.pos_off = 0;
        w.s = g.s_begin;
        w.src = ((q.rank - w.s) % g.P + g.P) % g.P;
        if (w.s < g.s_end) {
            kwalk_set_chunk<S>(g, w, w.src);
        } else {
            w.row = w.chunk_end = 0;   // empty step range: the walk is over
            w.ci = 1;
            w.s = g.s_end;
        }
    } else {
        w.pos_off = (int)g.k_off;
        w.s = 0;
        w.src = 0;
        w.row = 0;
        w.chunk_end = g.Lk;
        w.idx = 0;
    }
}

// Moves to the next chunk of the walk; false when the walk is over.
template <bool S>
__host__ __device__ __forceinline__ bool kwalk_next_chunk(const Geom &g, KWalk &w) {
    if (!g.ring) return false;
    if (g.zigzag && w.ci == 0) {
        w.ci = 1;
        kwalk_set_chunk<S>(g, w, 2 * g.P - 1 - w.src);
        return true;
    }
    w.ci = 0;
    if (++w.s >= g.s_end) return false;
    w.src = w.src == 0 ? g.P - 1 : w.src - 1;
    kwalk_set_chunk<S>(g, w, w.src);
    return true;
}

// Next non-EMPTY key tile of the walk into k; false at the end.
template <bool S>
__host__ __device__ __forceinline__ bool kwalk_next(const Geom &g, const QTile &q, KWalk &w, KTile &k) {
    for (;;) {
        if (w.row >= w.chunk_end) {
            if (!kwalk_next_chunk<S>(g, w)) return false;
            continue;
        }
        const int row = w.row;
        const int pos = row + w.pos_off;
        const int rem = w.chunk_end - row;
        k.row0 = row;
        k.len = rem < TILE ? rem : TILE;
        k.pos0 = pos;
        k.idx = w.idx;
        w.row = row + TILE;
        ++w.idx;
        if (g.cls) {
            k.cls = g.cls[((long long)q.b * g.n_qtiles + q.g) * g.n_ktiles + k.idx];
            if (k.cls == BA_TILE_EMPTY) continue;
            return true;
        }
        if (g.causal) {
            if (pos > w.q_last) {          // this and the rest of the chunk lie in the future
                w.row = w.chunk_end;
                continue;
            }
            k.cls = pos + k.len - 1 <= w.q_first ? BA_TILE_FULL : BA_TILE_PARTIAL;
        } else {
            k.cls = BA_TILE_FULL;
        }
        if (k.cls == BA_TILE_FULL && (g.kpm || g.am)) k.cls = BA_TILE_PARTIAL;   // masks need predicates
        return true;
    }
}

// Number of key tiles kwalk_next yields for query tile q.  Without a class map
// this is a sum over the walk's chunks (a chunk contributes its tiles that start
// at or before q's last row under causal masking, all of them otherwise), so it
// costs a few operations per chunk instead of a walk over every tile.
template <bool S>
__host__ __device__ inline int kwalk_count(const Geom &g, const QTile &q) {
    if (g.cls) {
        KWalk w;
        kwalk_begin<S>(g, q, w);
        KTile k;
        int n = 0;
        while (kwalk_next<S>(g, q, w, k)) ++n;
        return n;
    }
    const long long q_last = q.pos0 + q.len - 1;
    auto chunk_tiles = [&](long long first_pos, int len) -> int {
        const int tiles = (len + TILE - 1) / TILE;
        if (!g.causal) return tiles;
        if (first_pos > q_last) return 0;
        const long long upto = (q_last - first_pos) / TILE + 1;   // tiles starting at or before q_last
        return upto < tiles ? (int)upto : tiles;
    };
    if (!g.ring) return chunk_tiles(g.k_off, g.Lk);
    int n = 0;
    int src = ((q.rank - g.s_begin) % g.P + g.P) % g.P;
    for (int s = g.s_begin; s < g.s_end; ++s) {
        n += chunk_tiles(chunk_pos0<S>(g, src, q.rank), g.CL);
        if (g.zigzag) n += chunk_tiles(chunk_pos0<S>(g, 2 * g.P - 1 - src, q.rank), g.CL);
        src = src == 0 ? g.P - 1 : src - 1;
    }
    return n;
}

// Token of row R of a ring tensor: R itself, or r + P u for row R = r CL + u
// of the striped ring.
template <bool S>
__host__ __device__ __forceinline__ long long row_token(const Geom &g, long long R) {
    if (!S) return R;
    const long long r = R / g.CL;
    return r + (long long)g.P * (R - r * g.CL);
}

// Row of out / lse (token order) for row `row` of query tile q.
template <bool S>
__host__ __device__ __forceinline__ long long out_row(const Geom &g, const QTile &q, int row) {
    return S ? q.rank + (long long)g.P * (q.pos0 + row) : (long long)q.row0 + row;
}

// Work item w -> (q tile, b, h).  Items are grouped by heads_per_group (b, h)
// pairs so that concurrently running CTAs share K/V in L2; within a group the
// query tiles come heaviest first under causal masking (latest positions).
template <bool S>
__host__ __device__ inline QTile work_item(const Geom &g, int w) {
    int BH = g.B * g.H;
    int G = g.heads_per_group;
    int per_group = G * g.n_qtiles;
    int grp = w / per_group;
    int rem = w % per_group;
    int g_heads = BH - grp * G < G ? BH - grp * G : G;   // last group may be short
    int qi = rem / g_heads;
    int bh = grp * G + rem % g_heads;
    int qg = g.causal ? g.n_qtiles - 1 - qi : qi;
    return q_tile<S>(g, qg, bh / g.H, bh % g.H);
}

// Is key position kp excluded for query position qp of batch item b?
__device__ inline bool excluded(const Geom &g, int b, long long qp, long long kp) {
    if (g.causal && kp > qp) return true;
    if (g.kpm && g.kpm[b * g.kpm_ld + kp]) return true;
    if (g.am && g.am[qp * g.am_ld + kp]) return true;
    return false;
}

// ---------------------------------------------------------------------------
// Pairs of query tiles (the tensor-core kernel's unit of work)
// ----------------------------------------------------------------------------
//
// The unit of work is a pair of adjacent query tiles of one chunk (ring mode)
// or of the block: tiles 2i and 2i + 1 of the chunk; when the chunk has an odd
// number of tiles its last pair holds one tile.  The two tiles cover
// consecutive positions, so the pair's key walk is the walk of the 256-row span
// that covers both; each key tile of it carries one class per tile (a tile that
// only the second query tile sees is EMPTY for the first, whose rows then see
// no key in it).

struct QPair {
    QTile q0, q1;    // q1.len == 0 when the pair holds one tile
    QTile span;      // both tiles as one query range (walk geometry)
};

__host__ __device__ inline int pairs_per_chunk(const Geom &g) {
    const int per = g.ring ? g.nqt_pc : g.n_qtiles;
    return (per + 1) / 2;
}

// Pairs per (b, h).
__host__ __device__ inline int n_pairs(const Geom &g) {
    return (g.ring ? g.NC : 1) * pairs_per_chunk(g);
}

// Work item w -> pair.  Pairs are dealt heaviest first under causal masking
// (latest positions), in two phases.  Phase 1 holds every level but the
// g.tail_levels lightest of each (b, h): grouped by heads_per_group (b, h) so
// that concurrently running CTAs share K/V in L2.  Phase 2 deals the lightest
// levels of all heads, heaviest first: the items claimed last are the smallest
// of the launch, so the CTAs finish within about one small item of each other.
template <bool S>
__host__ __device__ inline QPair work_pair(const Geom &g, int w) {
    const int BH = g.B * g.H, G = g.heads_per_group, np = n_pairs(g);
    const int tail = g.tail_levels < np ? g.tail_levels : np;
    const int heavy = np - tail;
    int pi, bh;
    if (w < heavy * BH) {
        const int per_group = G * heavy;
        const int grp = w / per_group, rem = w % per_group;
        const int g_heads = BH - grp * G < G ? BH - grp * G : G;   // last group may be short
        pi = rem / g_heads;
        bh = grp * G + rem % g_heads;
    } else {
        const int w2 = w - heavy * BH;
        pi = heavy + w2 / BH;
        bh = w2 % BH;
    }
    const int ppc = pairs_per_chunk(g), per = g.ring ? g.nqt_pc : g.n_qtiles;
    int c, i;
    if (S && g.causal) {
        // a query at local index u of rank r sees P u + r + 1 keys: deal the
        // levels of all ranks together, last level and last rank first
        c = g.NC - 1 - pi % g.NC;
        i = ppc - 1 - pi / g.NC;
    } else {
        const int pg = g.causal ? np - 1 - pi : pi;
        c = pg / ppc;
        i = pg % ppc;
    }
    const int b = bh / g.H, h = bh % g.H;
    QPair p;
    p.q0 = q_tile<S>(g, c * per + 2 * i, b, h);
    if (2 * i + 1 < per) {
        p.q1 = q_tile<S>(g, c * per + 2 * i + 1, b, h);
    } else {
        p.q1 = p.q0;
        p.q1.len = 0;
    }
    p.span = p.q0;
    p.span.len = p.q0.len + p.q1.len;
    return p;
}

// Next key tile of the pair's walk that one of its query tiles sees, with the
// class for each (c1 = EMPTY when the pair holds one tile); false at the end.
template <bool S>
__host__ __device__ __forceinline__ bool pair_next(const Geom &g, const QPair &p, KWalk &w, KTile &k, int &c0,
                                              int &c1) {
    const int q0_last = (int)p.q0.pos0 + p.q0.len - 1;
    const bool has1 = p.q1.len > 0;
    for (;;) {
        if (w.row >= w.chunk_end) {
            if (!kwalk_next_chunk<S>(g, w)) return false;
            continue;
        }
        const int row = w.row;
        const int pos = row + w.pos_off;
        const int rem = w.chunk_end - row;
        k.row0 = row;
        k.len = rem < TILE ? rem : TILE;
        k.pos0 = pos;
        k.idx = w.idx;
        w.row = row + TILE;
        ++w.idx;
        if (g.cls) {
            const int8_t *m = g.cls + ((long long)p.q0.b * g.n_qtiles + p.q0.g) * g.n_ktiles + k.idx;
            c0 = m[0];
            c1 = has1 ? m[g.n_ktiles] : BA_TILE_EMPTY;
            if (c0 == BA_TILE_EMPTY && c1 == BA_TILE_EMPTY) continue;
            return true;
        }
        if (g.causal) {
            if (pos > w.q_last) {          // this and the rest of the chunk lie in the future of both
                w.row = w.chunk_end;
                continue;
            }
            const int k_last = pos + k.len - 1;
            c0 = pos > q0_last ? BA_TILE_EMPTY : (k_last <= (int)p.q0.pos0 ? BA_TILE_FULL : BA_TILE_PARTIAL);
            c1 = !has1 ? BA_TILE_EMPTY : (k_last <= (int)p.q1.pos0 ? BA_TILE_FULL : BA_TILE_PARTIAL);
        } else {
            c0 = BA_TILE_FULL;
            c1 = has1 ? BA_TILE_FULL : BA_TILE_EMPTY;
        }
        if (g.kpm || g.am) {   // masks need predicates
            if (c0 == BA_TILE_FULL) c0 = BA_TILE_PARTIAL;
            if (c1 == BA_TILE_FULL) c1 = BA_TILE_PARTIAL;
        }
        return true;
    }
}

// Number of key tiles pair_next yields for pair p.
template <bool S>
__host__ __device__ inline int pair_count(const Geom &g, const QPair &p) {
    if (!g.cls) return kwalk_count<S>(g, p.span);   // the span's walk: both tiles see a tile the span sees
    KWalk w;
    kwalk_begin<S>(g, p.span, w);
    KTile k;
    int c0, c1, n = 0;
    while (pair_next<S>(g, p, w, k, c0, c1)) ++n;
    return n;
}

// Lightest levels dealt last (work_pair's phase 2) for a launch on num_sms SMs:
// under causal masking, when each SM gets fewer than 32 items, enough of them to
// give each SM about four small items at the end of the launch.  With many items
// per SM the heaviest-first order of each head group already ends on small items,
// and keeping the groups whole keeps their K/V in L2.
__host__ __device__ inline int pair_tail_levels(const Geom &g, int num_sms) {
    const int np = n_pairs(g), BH = g.B * g.H;
    if (!g.causal || BH <= 0 || (long long)np * BH >= 32LL * num_sms) return 0;
    const int want = (4 * num_sms + BH - 1) / BH;
    return want < np ? want : np;
}

// ---------------------------------------------------------------------------
// mbarrier helpers with bounded waits
// ---------------------------------------------------------------------------

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Wait until the phase with the given parity of barrier `bar` has completed.
// Gives up (returns false) when *abort is set by another role, or after
// limit_ns nanoseconds, in which case it sets *abort and the error word.
__device__ __forceinline__ bool mbar_test_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int *abort,
                                          unsigned *err, uint64_t limit_ns) {
    if (mbar_test_wait(bar, parity)) return true;   // already complete: no suspend
    if (mbar_try_wait(bar, parity)) return true;
    uint64_t t0 = global_timer_ns();
    for (uint32_t n = 1;; ++n) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((n & 63) == 0) {
            if (*abort) return false;
            if (global_timer_ns() - t0 > limit_ns) {
                *abort = 1;
                if (err) atomicOr(err, ERR_TIMEOUT_BIT);
                return false;
            }
        }
    }
}

}  // namespace ba
