// CUDA-core attention kernel: fp32 arithmetic throughout, for fp32 inputs
// (whose 1e-4 output tolerance the bf16 tensor-core path cannot meet) and for
// bf16 inputs with head dimension 16 or 32.
//
// One CTA of 128 threads per query tile, one thread per query row.  The CTA
// walks the tile's key tiles in ring order (the same walk as the tensor-core
// kernel), stages 32 keys of K and V at a time in shared memory as fp32, and
// keeps the running (max, denominator, weighted sum) of its row in registers.
// Each 32-key group is folded in with the rescale-to-the-new-maximum update
// (brunomaga "Improving numerical stability").
#include <cuda_bf16.h>

#include "epilogue.cuh"

namespace ba {
namespace {

constexpr int SUB = 32;  // keys staged per round

template <typename T>
__device__ __forceinline__ float to_f32(T x);
template <>
__device__ __forceinline__ float to_f32<float>(float x) { return x; }
template <>
__device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 x) { return __bfloat162float(x); }

template <int D, typename Tin, bool S>
__global__ void __launch_bounds__(TILE) attn_simt_kernel(const AttnArgs a) {
    __shared__ float Ks[SUB][D + 1];
    __shared__ float Vs[SUB][D];
    const Geom &g = a.g;
    const QTile qt = work_item<S>(g, blockIdx.x);
    const int r = threadIdx.x;
    const bool valid = r < qt.len;
    const long long qpos = qt.pos0 + r;
    const Tin *qb = static_cast<const Tin *>(a.q) + qt.b * a.qsB + qt.h * a.qsH;
    const Tin *kb = static_cast<const Tin *>(a.k) + qt.b * a.ksB + qt.h * a.ksH;
    const Tin *vb = static_cast<const Tin *>(a.v) + qt.b * a.vsB + qt.h * a.vsH;

    float q[D], o[D];
#pragma unroll
    for (int c = 0; c < D; ++c) {
        q[c] = valid ? to_f32(qb[row_token<S>(g, qt.row0 + r) * a.qsT + c]) : 0.f;
        o[c] = 0.f;
    }
    float m = -INFINITY, l = 0.f;   // running max (log2 units) and denominator

    KWalk wk;
    kwalk_begin<S>(g, qt, wk);
    KTile kt;
    while (kwalk_next<S>(g, qt, wk, kt)) {
        for (int s0 = 0; s0 < kt.len; s0 += SUB) {
            __syncthreads();
            for (int e = threadIdx.x; e < SUB * D; e += blockDim.x) {
                int j = e / D, c = e % D;
                bool in = s0 + j < kt.len;
                const long long row = row_token<S>(g, kt.row0 + s0 + j);
                Ks[j][c] = in ? to_f32(kb[row * a.ksT + c]) : 0.f;
                Vs[j][c] = in ? to_f32(vb[row * a.vsT + c]) : 0.f;
            }
            __syncthreads();
            if (!valid) continue;
            float x[SUB];
            float mx = -INFINITY;
#pragma unroll 4
            for (int j = 0; j < SUB; ++j) {
                int kj = s0 + j;
                bool ok = kj < kt.len &&
                          (kt.cls == BA_TILE_FULL || !excluded(g, qt.b, qpos, kt.pos0 + kj));
                float dot = 0.f;
#pragma unroll
                for (int c = 0; c < D; ++c) dot = fmaf(q[c], Ks[j][c], dot);
                x[j] = ok ? dot * a.scale_log2 : -INFINITY;
                mx = fmaxf(mx, x[j]);
            }
            float m_new = fmaxf(m, mx);
            if (m_new == -INFINITY) continue;      // nothing visible yet
            float alpha = exp2f(m - m_new);        // 0 when m == -inf
            l *= alpha;
#pragma unroll
            for (int c = 0; c < D; ++c) o[c] *= alpha;
            for (int j = 0; j < SUB; ++j) {
                float p = exp2f(x[j] - m_new);     // 0 for excluded keys
                l += p;
#pragma unroll
                for (int c = 0; c < D; ++c) o[c] = fmaf(p, Vs[j][c], o[c]);
            }
            m = m_new;
        }
    }
    if (!valid) return;
    const long long row_flat = ((long long)qt.b * g.H + qt.h) * a.rows + out_row<S>(g, qt, r);
    const float acc_l = a.acc_lse ? a.acc_lse[row_flat] : -INFINITY;
    const RowFinal f = row_final(m, l, acc_l);
#pragma unroll
    for (int c0 = 0; c0 < D; c0 += 32) {
        constexpr int N = D < 32 ? D : 32;
        store_row_chunk(a, row_flat, c0, o + c0, N, f);
    }
    a.lse[row_flat] = f.lse;
}

template <int D, bool S>
int launch_ds(const AttnArgs &a, cudaStream_t s) {
    dim3 grid(a.g.n_items);
    if (a.dtype == BA_F32)
        attn_simt_kernel<D, float, S><<<grid, TILE, 0, s>>>(a);
    else
        attn_simt_kernel<D, __nv_bfloat16, S><<<grid, TILE, 0, s>>>(a);
    return cudaGetLastError() == cudaSuccess ? BA_OK : BA_ERR_CUDA;
}

template <int D>
int launch_d(const AttnArgs &a, cudaStream_t s) {
    return a.g.striped ? launch_ds<D, true>(a, s) : launch_ds<D, false>(a, s);
}

}  // namespace

int launch_attn_simt(const AttnArgs &a, cudaStream_t s) {
    if (a.g.n_items == 0) return BA_OK;
    switch (a.g.d) {
        case 16: return launch_d<16>(a, s);
        case 32: return launch_d<32>(a, s);
        case 64: return launch_d<64>(a, s);
        case 128: return launch_d<128>(a, s);
        default: return BA_ERR_SHAPE;
    }
}

}  // namespace ba
