// Attention backward on the CUDA cores (fp32 arithmetic, bf16 or fp32 inputs).
//
// The backward pass of "Sequence/context parallelism" (brunomaga), section
// "Ring Attention": every (query block, key block) pair contributes
//   dV_j += p_ij dout_i,  dp_ij = dout_i . v_j,  ds_ij = p_ij (dp_ij - D_i),
//   dQ_i += scale ds_ij k_j,  dK_j += scale ds_ij q_i,
// with p_ij = exp(scale q_i . k_j - LSE_i) from the saved LSE of the whole row
// and D_i = dout_i . out_i from the saved output.  dQ accumulates where the
// query block lives; dK and dV accumulate with their key block (on the page
// they travel around the ring with K and V).  On one GPU the emulated ranks are
// token ranges, so "travelling" is indexing: a key tile gathers the
// contributions of every query range that sees it.
//
// Kernels:
//   bwd_pre_kernel    D_i = dout_i . out_i, one warp per row.
//   bwd_dkdv_kernel   one block per 64-key tile of one (b, h): dK, dV in
//                     registers, query rows streamed in chunks of 16.
//   bwd_dq_kernel     one block per 64-row query tile: dQ in registers, key
//                     rows streamed in chunks of 16.
// Both main kernels recompute the scores and p from q, k and LSE, so neither
// needs atomics; each output row is written by exactly one block.
#include <cuda_bf16.h>

#include "internal.h"

namespace ba {
namespace {

constexpr int BT = 64;    // rows of the tile a block owns
constexpr int BC = 16;    // rows of the partner chunk streamed through shared memory
constexpr int NTH = 256;  // threads per block

__device__ __forceinline__ float ld_elem(const void *base, int dtype, long long idx) {
    if (dtype == BA_BF16) return __bfloat162float(static_cast<const __nv_bfloat16 *>(base)[idx]);
    return static_cast<const float *>(base)[idx];
}

__device__ __forceinline__ long long elem_index(const TensorRef &t, int b, int h, long long row, int c) {
    return (long long)b * t.sB + (long long)h * t.sH + row * t.sT + c;
}

// ---------------------------------------------------------------------------
// D_i = dout_i . out_i
// ---------------------------------------------------------------------------

__global__ void __launch_bounds__(256) bwd_pre_kernel(const BwdArgs a, long long rows_per_bh) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const long long n_rows = (long long)a.B * a.H * rows_per_bh;
    for (long long r = (long long)blockIdx.x * 8 + warp; r < n_rows; r += (long long)gridDim.x * 8) {
        const long long bh = r / rows_per_bh, row = r % rows_per_bh;
        const int b = (int)(bh / a.H), h = (int)(bh % a.H);
        float acc = 0.f;
        for (int c = lane; c < a.d; c += 32)
            acc += ld_elem(a.dout.p, a.dtype, elem_index(a.dout, b, h, row, c)) *
                   ld_elem(a.out.p, a.dtype, elem_index(a.out, b, h, row, c));
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
        if (lane == 0) a.D[r] = acc;
    }
}

// ---------------------------------------------------------------------------
// Tiles and partner ranges
// ---------------------------------------------------------------------------

// A tile of up to BT rows of one side, with the global position of its first row.
struct Tile {
    long long row0;   // first row in the tensor
    int len;          // rows (1..BT)
    long long pos0;   // global position of row0
    int chunk;        // ring chunk holding it (ring mode)
};

struct Span {
    long long row0, row1;   // [row0, row1) rows of the partner tensor
    long long pos0;         // global position of row0
};

__device__ __forceinline__ int chunk_owner_rank(const BwdArgs &a, int c) {
    return !a.zigzag ? c : (c < a.P ? c : 2 * a.P - 1 - c);
}

// Tile t of one side (q side when is_q, else k side).
__device__ __forceinline__ Tile make_tile(const BwdArgs &a, int t, bool is_q) {
    Tile x;
    if (!a.ring) {
        const int L = is_q ? a.Lq : a.Lk;
        x.row0 = (long long)t * BT;
        x.len = min(BT, L - (int)x.row0);
        x.pos0 = x.row0 + (is_q ? a.q_off : a.k_off);
        x.chunk = 0;
    } else {
        const int per = (a.CL + BT - 1) / BT;
        x.chunk = t / per;
        const int r = (t % per) * BT;
        x.row0 = (long long)x.chunk * a.CL + r;
        x.len = min(BT, a.CL - r);
        x.pos0 = x.row0;
    }
    return x;
}

// The partner spans of a tile: every contiguous range of the other side that
// the covered ring steps pair it with (block mode: the whole other side).
// Returns the number of spans (at most 2 per step).
__device__ __forceinline__ int partner_spans(const BwdArgs &a, const Tile &x, bool x_is_q, int step, Span *sp) {
    if (!a.ring) {
        sp[0].row0 = 0;
        sp[0].row1 = x_is_q ? a.Lk : a.Lq;
        sp[0].pos0 = x_is_q ? a.k_off : a.q_off;
        return 1;
    }
    const int me = chunk_owner_rank(a, x.chunk);
    // queries of rank r meet keys of rank (r - s) mod P; keys of rank src meet
    // queries of rank (src + s) mod P
    const int other = x_is_q ? ((me - step) % a.P + a.P) % a.P : (me + step) % a.P;
    int n = 0;
    sp[n].row0 = (long long)other * a.CL;
    sp[n].row1 = sp[n].row0 + a.CL;
    sp[n].pos0 = sp[n].row0;
    ++n;
    if (a.zigzag) {
        const int c2 = 2 * a.P - 1 - other;
        sp[n].row0 = (long long)c2 * a.CL;
        sp[n].row1 = sp[n].row0 + a.CL;
        sp[n].pos0 = sp[n].row0;
        ++n;
    }
    return n;
}

__device__ __forceinline__ bool is_excluded(const BwdArgs &a, int b, long long qp, long long kp) {
    if (a.causal && kp > qp) return true;
    if (a.kpm && a.kpm[b * a.kpm_ld + kp]) return true;
    if (a.am && a.am[qp * a.am_ld + kp]) return true;
    return false;
}

// ---------------------------------------------------------------------------
// dK, dV: one block per key tile
// ---------------------------------------------------------------------------

// Shared memory (floats): K[BT][d+1], V[BT][d+1], Q[BC][d+1], G[BC][d+1] (dout),
// P[BC][BT+1], dS[BC][BT+1], lse[BC], D[BC].  The +1 pads put the rows of a
// tile in different banks.
__host__ __device__ inline size_t dkdv_smem_bytes(int d) {
    return sizeof(float) * ((size_t)2 * BT * (d + 1) + (size_t)2 * BC * (d + 1) + (size_t)2 * BC * (BT + 1) + 2 * BC);
}

template <int D>
__global__ void __launch_bounds__(NTH) bwd_dkdv_kernel(const BwdArgs a) {
    extern __shared__ float smf[];
    constexpr int LD = D + 1;
    float *Ks = smf, *Vs = Ks + BT * LD, *Qs = Vs + BT * LD, *Gs = Qs + BC * LD;
    float *Ps = Gs + BC * LD, *Ss = Ps + BC * (BT + 1), *lse_s = Ss + BC * (BT + 1), *D_s = lse_s + BC;
    const int t = threadIdx.x;
    const int bh = blockIdx.y, b = bh / a.H, h = bh % a.H;
    const Tile kt = make_tile(a, blockIdx.x, false);
    const long long q_rows = a.ring ? a.T : a.Lq;

    for (int e = t; e < BT * D; e += NTH) {
        const int j = e / D, c = e % D;
        float kv = 0.f, vv = 0.f;
        if (j < kt.len) {
            kv = ld_elem(a.k.p, a.dtype, elem_index(a.k, b, h, kt.row0 + j, c));
            vv = ld_elem(a.v.p, a.dtype, elem_index(a.v, b, h, kt.row0 + j, c));
        }
        Ks[j * LD + c] = kv;
        Vs[j * LD + c] = vv;
    }

    // accumulators: key jo = t / 4, columns c = (t % 4) + 4 m
    constexpr int NCOL = D / 4;
    const int jo = t >> 2, co = t & 3;
    float dk[NCOL], dv[NCOL];
#pragma unroll
    for (int m = 0; m < NCOL; ++m) dk[m] = dv[m] = 0.f;
    // score entries: query i = t / 16, keys j = (t % 16) + 16 r
    const int si = t >> 4, sj = t & 15;
    const float sl2 = a.scale * 1.4426950408889634f;
    const long long k_last = kt.pos0 + kt.len - 1;

    const int steps = a.ring ? a.s_end - a.s_begin : 1;
    for (int st = 0; st < steps; ++st) {
        Span sp[2];
        const int nsp = partner_spans(a, kt, false, a.ring ? a.s_begin + st : 0, sp);
        for (int si_ = 0; si_ < nsp; ++si_) {
            long long r0 = sp[si_].row0;
            const long long r1 = sp[si_].row1, dpos = sp[si_].pos0 - sp[si_].row0;
            // causal: queries before the tile's first key see none of it
            if (a.causal && r0 + dpos < kt.pos0) r0 = kt.pos0 - dpos;
            for (long long q0 = r0; q0 < r1; q0 += BC) {
                const int qn = (int)min((long long)BC, r1 - q0);
                __syncthreads();   // previous chunk fully consumed
                for (int e = t; e < BC * D; e += NTH) {
                    const int i = e / D, c = e % D;
                    float qv = 0.f, gv = 0.f;
                    if (i < qn) {
                        qv = ld_elem(a.q.p, a.dtype, elem_index(a.q, b, h, q0 + i, c));
                        gv = ld_elem(a.dout.p, a.dtype, elem_index(a.dout, b, h, q0 + i, c));
                    }
                    Qs[i * LD + c] = qv;
                    Gs[i * LD + c] = gv;
                }
                if (t < BC) {
                    const long long row = (long long)bh * q_rows + q0 + t;
                    lse_s[t] = t < qn ? a.lse[row] : -INFINITY;
                    D_s[t] = t < qn ? a.D[row] : 0.f;
                }
                __syncthreads();
                // p and ds of (query si, keys sj + 16 r)
                {
                    float s4[4] = {0.f, 0.f, 0.f, 0.f}, g4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 8
                    for (int c = 0; c < D; ++c) {
                        const float qv = Qs[si * LD + c], gv = Gs[si * LD + c];
#pragma unroll
                        for (int r = 0; r < 4; ++r) {
                            s4[r] = fmaf(qv, Ks[(sj + 16 * r) * LD + c], s4[r]);
                            g4[r] = fmaf(gv, Vs[(sj + 16 * r) * LD + c], g4[r]);
                        }
                    }
                    const long long qp = q0 + dpos + si;
                    const float L = lse_s[si];
#pragma unroll
                    for (int r = 0; r < 4; ++r) {
                        const int j = sj + 16 * r;
                        float p = 0.f, ds = 0.f;
                        if (si < qn && j < kt.len && L != -INFINITY && !is_excluded(a, b, qp, kt.pos0 + j)) {
                            p = exp2f(fmaf(s4[r], sl2, -L * 1.4426950408889634f));
                            ds = p * (g4[r] - D_s[si]);
                        }
                        Ps[si * (BT + 1) + j] = p;
                        Ss[si * (BT + 1) + j] = ds;
                    }
                }
                __syncthreads();
                // dV += p^T dout, dK += scale ds^T q
#pragma unroll 4
                for (int i = 0; i < qn; ++i) {
                    const float p = Ps[i * (BT + 1) + jo], ds = Ss[i * (BT + 1) + jo];
#pragma unroll
                    for (int m = 0; m < NCOL; ++m) {
                        const int c = co + 4 * m;
                        dv[m] = fmaf(p, Gs[i * LD + c], dv[m]);
                        dk[m] = fmaf(ds, Qs[i * LD + c], dk[m]);
                    }
                }
                (void)k_last;
            }
        }
    }
    if (jo < kt.len) {
        const long long row = ((long long)bh * (a.ring ? a.T : a.Lk) + kt.row0 + jo) * D;
#pragma unroll
        for (int m = 0; m < NCOL; ++m) {
            const int c = co + 4 * m;
            const float gk = dk[m] * a.scale, gv = dv[m];
            a.dk[row + c] = a.accumulate ? a.dk[row + c] + gk : gk;
            a.dv[row + c] = a.accumulate ? a.dv[row + c] + gv : gv;
        }
    }
}

// ---------------------------------------------------------------------------
// dQ: one block per query tile
// ---------------------------------------------------------------------------

// Shared memory (floats): Q[BT][d+1], G[BT][d+1], K[BC][d+1], V[BC][d+1],
// dS[BT][BC+1], lse[BT], D[BT].
__host__ __device__ inline size_t dq_smem_bytes(int d) {
    return sizeof(float) * ((size_t)2 * BT * (d + 1) + (size_t)2 * BC * (d + 1) + (size_t)BT * (BC + 1) + 2 * BT);
}

template <int D>
__global__ void __launch_bounds__(NTH) bwd_dq_kernel(const BwdArgs a) {
    extern __shared__ float smf[];
    constexpr int LD = D + 1;
    float *Qs = smf, *Gs = Qs + BT * LD, *Ks = Gs + BT * LD, *Vs = Ks + BC * LD;
    float *Ss = Vs + BC * LD, *lse_s = Ss + BT * (BC + 1), *D_s = lse_s + BT;
    const int t = threadIdx.x;
    const int bh = blockIdx.y, b = bh / a.H, h = bh % a.H;
    const Tile qt = make_tile(a, blockIdx.x, true);
    const long long q_rows = a.ring ? a.T : a.Lq;

    for (int e = t; e < BT * D; e += NTH) {
        const int i = e / D, c = e % D;
        float qv = 0.f, gv = 0.f;
        if (i < qt.len) {
            qv = ld_elem(a.q.p, a.dtype, elem_index(a.q, b, h, qt.row0 + i, c));
            gv = ld_elem(a.dout.p, a.dtype, elem_index(a.dout, b, h, qt.row0 + i, c));
        }
        Qs[i * LD + c] = qv;
        Gs[i * LD + c] = gv;
    }
    if (t < BT) {
        const long long row = (long long)bh * q_rows + qt.row0 + t;
        lse_s[t] = t < qt.len ? a.lse[row] : -INFINITY;
        D_s[t] = t < qt.len ? a.D[row] : 0.f;
    }

    constexpr int NCOL = D / 4;
    const int io = t >> 2, co = t & 3;
    float dq[NCOL];
#pragma unroll
    for (int m = 0; m < NCOL; ++m) dq[m] = 0.f;
    // score entries: key j = t % 16, queries i = (t / 16) + 16 r
    const int sj = t & 15, si = t >> 4;
    const float sl2 = a.scale * 1.4426950408889634f;
    const long long q_last = qt.pos0 + qt.len - 1;

    const int steps = a.ring ? a.s_end - a.s_begin : 1;
    for (int st = 0; st < steps; ++st) {
        Span sp[2];
        const int nsp = partner_spans(a, qt, true, a.ring ? a.s_begin + st : 0, sp);
        for (int s_ = 0; s_ < nsp; ++s_) {
            const long long r0 = sp[s_].row0, dpos = sp[s_].pos0 - sp[s_].row0;
            long long r1 = sp[s_].row1;
            // causal: keys after the tile's last query are seen by none of it
            if (a.causal && r1 + dpos > q_last + 1) r1 = q_last + 1 - dpos;
            for (long long k0 = r0; k0 < r1; k0 += BC) {
                const int kn = (int)min((long long)BC, r1 - k0);
                __syncthreads();
                for (int e = t; e < BC * D; e += NTH) {
                    const int j = e / D, c = e % D;
                    float kv = 0.f, vv = 0.f;
                    if (j < kn) {
                        kv = ld_elem(a.k.p, a.dtype, elem_index(a.k, b, h, k0 + j, c));
                        vv = ld_elem(a.v.p, a.dtype, elem_index(a.v, b, h, k0 + j, c));
                    }
                    Ks[j * LD + c] = kv;
                    Vs[j * LD + c] = vv;
                }
                __syncthreads();
                {
                    float s4[4] = {0.f, 0.f, 0.f, 0.f}, g4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 8
                    for (int c = 0; c < D; ++c) {
                        const float kv = Ks[sj * LD + c], vv = Vs[sj * LD + c];
#pragma unroll
                        for (int r = 0; r < 4; ++r) {
                            s4[r] = fmaf(Qs[(si + 16 * r) * LD + c], kv, s4[r]);
                            g4[r] = fmaf(Gs[(si + 16 * r) * LD + c], vv, g4[r]);
                        }
                    }
                    const long long kp = k0 + dpos + sj;
#pragma unroll
                    for (int r = 0; r < 4; ++r) {
                        const int i = si + 16 * r;
                        const float L = lse_s[i];
                        float ds = 0.f;
                        if (sj < kn && i < qt.len && L != -INFINITY && !is_excluded(a, b, qt.pos0 + i, kp)) {
                            const float p = exp2f(fmaf(s4[r], sl2, -L * 1.4426950408889634f));
                            ds = p * (g4[r] - D_s[i]);
                        }
                        Ss[i * (BC + 1) + sj] = ds;
                    }
                }
                __syncthreads();
#pragma unroll 4
                for (int j = 0; j < kn; ++j) {
                    const float ds = Ss[io * (BC + 1) + j];
#pragma unroll
                    for (int m = 0; m < NCOL; ++m) dq[m] = fmaf(ds, Ks[j * LD + co + 4 * m], dq[m]);
                }
            }
        }
    }
    if (io < qt.len) {
        const long long row = ((long long)bh * q_rows + qt.row0 + io) * D;
#pragma unroll
        for (int m = 0; m < NCOL; ++m) {
            const int c = co + 4 * m;
            const float g = dq[m] * a.scale;
            a.dq[row + c] = a.accumulate ? a.dq[row + c] + g : g;
        }
    }
}

template <int D>
int launch_d(const BwdArgs &a, int n_qt, int n_kt, cudaStream_t s) {
    const size_t s1 = dkdv_smem_bytes(D), s2 = dq_smem_bytes(D);
    if (cudaFuncSetAttribute(bwd_dkdv_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)s1) !=
            cudaSuccess ||
        cudaFuncSetAttribute(bwd_dq_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)s2) != cudaSuccess)
        return BA_ERR_CUDA;
    const int BH = a.B * a.H;
    if (n_kt > 0) bwd_dkdv_kernel<D><<<dim3(n_kt, BH), NTH, s1, s>>>(a);
    if (n_qt > 0) bwd_dq_kernel<D><<<dim3(n_qt, BH), NTH, s2, s>>>(a);
    return cudaGetLastError() == cudaSuccess ? BA_OK : BA_ERR_CUDA;
}

}  // namespace

// D_i = dout_i . out_i for every query row into a.D.
int launch_bwd_pre(const BwdArgs &a, int num_sms, cudaStream_t s) {
    const long long q_rows = a.ring ? a.T : a.Lq;
    const long long warps = (long long)a.B * a.H * q_rows;
    if (warps == 0) return BA_OK;
    long long blocks = (warps + 7) / 8;
    if (blocks > 8LL * num_sms) blocks = 8LL * num_sms;
    bwd_pre_kernel<<<(int)blocks, 256, 0, s>>>(a, q_rows);
    return cudaGetLastError() == cudaSuccess ? BA_OK : BA_ERR_CUDA;
}

// D = rowsum(dout * out), then dK/dV and dQ.  a.D must hold B*H*rows floats.
int launch_attn_bwd(const BwdArgs &a, int num_sms, cudaStream_t s) {
    const int BH = a.B * a.H;
    if (BH == 0) return BA_OK;
    if (BH > 65535) return BA_ERR_SHAPE;
    const int n_qt = a.ring ? a.NC * ((a.CL + BT - 1) / BT) : (a.Lq + BT - 1) / BT;
    const int n_kt = a.ring ? a.NC * ((a.CL + BT - 1) / BT) : (a.Lk + BT - 1) / BT;
    {
        const int rc = launch_bwd_pre(a, num_sms, s);
        if (rc) return rc;
    }
    switch (a.d) {
        case 16: return launch_d<16>(a, n_qt, n_kt, s);
        case 32: return launch_d<32>(a, n_qt, n_kt, s);
        case 64: return launch_d<64>(a, n_qt, n_kt, s);
        case 128: return launch_d<128>(a, n_qt, n_kt, s);
        default: return BA_ERR_SHAPE;
    }
}

}  // namespace ba
