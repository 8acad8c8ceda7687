// Decode attention against a long KV cache, split along the keys.
//
// Decode processes one query token per sequence and shards the KV cache rather
// than the input tokens ("Sequence/context parallelism" (brunomaga), the note
// on the inference decode step); a sequence's cache grows as tokens arrive
// ("Transformers and Attention" (ai.engineer), item #57 on KV-cache allocation).  The cache of one
// (b, h) is cut into key splits; each split yields a partial attention (O, LSE)
// over its keys, and the partials are merged by the LSE rule, never added or
// averaged (brunomaga, "Circulate K/V blocks with Ring": the merge of
// accumulate_out_and_lse, here over all splits at once, which is the same
// associative merge taken pairwise).
//
// decode_split_kernel: one CTA per (split, b, h).  A group of LPK lanes owns one
//   key at a time, each lane 16 bytes of the row (8 bf16 or 4 fp32); four keys
//   per group are loaded before they are used, so that every SM keeps tens of
//   KB of K/V in flight.  Each group keeps an online (m, l, o); the groups of
//   the CTA are merged in shared memory into the split's (O / l, LSE).
// decode_combine_kernel: one warp per (b, h): LSE-merge of the splits.
// Both are bound by HBM: every cached K and V byte up to the sequence length is
// read once.
#include <cuda_bf16.h>

#include <cstdint>

#include "internal.h"

namespace ba {
namespace {

constexpr int DEC_THREADS = 128;
constexpr int DEC_UNROLL = 4;

template <typename T>
struct Vec16;   // 16 bytes of T, unpacked to fp32
template <>
struct Vec16<__nv_bfloat16> {
    static constexpr int N = 8;
    __device__ __forceinline__ static void load(const void *p, float (&x)[8]) {
        const uint4 u = __ldg(reinterpret_cast<const uint4 *>(p));
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            x[2 * i] = __uint_as_float(w[i] << 16);
            x[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
        }
    }
};
template <>
struct Vec16<float> {
    static constexpr int N = 4;
    __device__ __forceinline__ static void load(const void *p, float (&x)[4]) {
        const float4 u = __ldg(reinterpret_cast<const float4 *>(p));
        x[0] = u.x;
        x[1] = u.y;
        x[2] = u.z;
        x[3] = u.w;
    }
};

template <typename T, int D>
__global__ void __launch_bounds__(DEC_THREADS) decode_split_kernel(const DecodeArgs a) {
    constexpr int EPL = Vec16<T>::N;     // elements per lane
    constexpr int LPK = D / EPL;         // lanes per key (2..32)
    constexpr int GROUPS = DEC_THREADS / LPK;
    constexpr int GPW = 32 / LPK;                 // key groups per warp
    constexpr int WARPS = DEC_THREADS / 32;
    __shared__ float sm_o[GROUPS][D];
    __shared__ float sm_m[GROUPS], sm_l[GROUPS];

    const int split = blockIdx.x, bh = blockIdx.y, b = bh / a.H, h = bh % a.H;
    const int len = a.lengths ? min(max(a.lengths[b], 0), a.S) : a.S;
    const int k0 = split * a.split_len, k1 = min(len, k0 + a.split_len);
    const int grp = threadIdx.x / LPK, gl = threadIdx.x % LPK;
    const int warp = threadIdx.x / 32, gw = (threadIdx.x % 32) / LPK;
    const float sl2 = a.scale * 1.4426950408889634f;

    float q[EPL];
    {
        const T *qp = static_cast<const T *>(a.q) + (long long)b * a.qsB + (long long)h * a.qsH;
        Vec16<T>::load(qp + gl * EPL, q);
    }
    const T *kb = static_cast<const T *>(a.k) + (long long)b * a.ksB + (long long)h * a.ksH;
    const T *vb = static_cast<const T *>(a.v) + (long long)b * a.vsB + (long long)h * a.vsH;

    float m = -INFINITY, l = 0.f, o[EPL];
#pragma unroll
    for (int e = 0; e < EPL; ++e) o[e] = 0.f;

    // The loop runs on a warp-uniform key base (the shuffles below span the
    // warp); keys past the split end are masked, their loads clamped in range.
    for (int jb = k0 + warp * GPW * DEC_UNROLL; jb < k1; jb += WARPS * GPW * DEC_UNROLL) {
        const int j0 = jb + gw * DEC_UNROLL;
        float kx[DEC_UNROLL][EPL], vx[DEC_UNROLL][EPL];
#pragma unroll
        for (int u = 0; u < DEC_UNROLL; ++u) {
            const int j = min(j0 + u, k1 - 1);   // clamp: a lane never reads past the valid keys
            Vec16<T>::load(kb + (long long)j * a.ksT + gl * EPL, kx[u]);
            Vec16<T>::load(vb + (long long)j * a.vsT + gl * EPL, vx[u]);
        }
        float s[DEC_UNROLL];
#pragma unroll
        for (int u = 0; u < DEC_UNROLL; ++u) {
            float acc = 0.f;
#pragma unroll
            for (int e = 0; e < EPL; ++e) acc = fmaf(q[e], kx[u][e], acc);
#pragma unroll
            for (int off = LPK / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off, LPK);
            s[u] = j0 + u < k1 ? acc * sl2 : -INFINITY;   // log2 units
        }
        float mx = s[0];
#pragma unroll
        for (int u = 1; u < DEC_UNROLL; ++u) mx = fmaxf(mx, s[u]);
        const float m_new = fmaxf(m, mx);
        const float alpha = m == -INFINITY ? 0.f : exp2f(m - m_new);
        l *= alpha;
#pragma unroll
        for (int e = 0; e < EPL; ++e) o[e] *= alpha;
#pragma unroll
        for (int u = 0; u < DEC_UNROLL; ++u) {
            const float p = s[u] == -INFINITY ? 0.f : exp2f(s[u] - m_new);
            l += p;
#pragma unroll
            for (int e = 0; e < EPL; ++e) o[e] = fmaf(p, vx[u][e], o[e]);
        }
        m = m_new;
    }
    // merge the groups of the CTA
#pragma unroll
    for (int e = 0; e < EPL; ++e) sm_o[grp][gl * EPL + e] = o[e];
    if (gl == 0) {
        sm_m[grp] = m;
        sm_l[grp] = l;
    }
    __syncthreads();
    const long long prow = (long long)bh * a.n_splits + split;
    for (int c = threadIdx.x; c < D; c += DEC_THREADS) {
        float M = -INFINITY;
        for (int g = 0; g < GROUPS; ++g) M = fmaxf(M, sm_m[g]);
        float L = 0.f, acc = 0.f;
        if (M != -INFINITY) {
            for (int g = 0; g < GROUPS; ++g) {
                const float w = sm_m[g] == -INFINITY ? 0.f : exp2f(sm_m[g] - M);
                L += w * sm_l[g];
                acc += w * sm_o[g][c];
            }
        }
        a.part_o[prow * D + c] = L > 0.f ? acc / L : 0.f;
        if (c == 0) a.part_lse[prow] = L > 0.f ? (M + log2f(L)) * 0.6931471805599453f : -INFINITY;
    }
}

// LSE merge of the splits of one (b, h): L = log sum_s e^{L_s},
// O = sum_s e^{L_s - L} O_s; splits with L_s = -inf carry no keys.
template <int D>
__global__ void __launch_bounds__(256) decode_combine_kernel(const DecodeArgs a) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const long long bh = (long long)blockIdx.x * 8 + warp;
    if (bh >= (long long)a.B * a.H) return;
    const float *pl = a.part_lse + bh * a.n_splits;
    float M = -INFINITY;
    for (int s = 0; s < a.n_splits; ++s) M = fmaxf(M, pl[s]);
    float sum = 0.f;
    if (M != -INFINITY)
        for (int s = 0; s < a.n_splits; ++s) sum += pl[s] == -INFINITY ? 0.f : expf(pl[s] - M);
    const float L = M == -INFINITY ? -INFINITY : M + logf(sum);
    for (int c = lane; c < D; c += 32) {
        float acc = 0.f;
        if (L != -INFINITY)
            for (int s = 0; s < a.n_splits; ++s)
                if (pl[s] != -INFINITY) acc += expf(pl[s] - L) * a.part_o[(bh * a.n_splits + s) * D + c];
        const long long oi = bh * D + c;
        if (a.out_dtype == BA_BF16)
            static_cast<__nv_bfloat16 *>(a.out)[oi] = __float2bfloat16_rn(acc);
        else
            static_cast<float *>(a.out)[oi] = acc;
    }
    if (lane == 0) a.lse[bh] = L;
}

template <typename T, int D>
int launch_td(const DecodeArgs &a, cudaStream_t s) {
    decode_split_kernel<T, D><<<dim3(a.n_splits, a.B * a.H), DEC_THREADS, 0, s>>>(a);
    if (cudaGetLastError() != cudaSuccess) return BA_ERR_CUDA;
    const long long rows = (long long)a.B * a.H;
    decode_combine_kernel<D><<<(int)((rows + 7) / 8), 256, 0, s>>>(a);
    return cudaGetLastError() == cudaSuccess ? BA_OK : BA_ERR_CUDA;
}

template <typename T>
int launch_t(const DecodeArgs &a, cudaStream_t s) {
    switch (a.d) {
        case 16: return launch_td<T, 16>(a, s);
        case 32: return launch_td<T, 32>(a, s);
        case 64: return launch_td<T, 64>(a, s);
        case 128: return launch_td<T, 128>(a, s);
        default: return BA_ERR_SHAPE;
    }
}

}  // namespace

int launch_decode(const DecodeArgs &a, cudaStream_t s) {
    if ((long long)a.B * a.H == 0) return BA_OK;
    if (a.B * a.H > 65535 || a.n_splits < 1) return BA_ERR_SHAPE;
    return a.dtype == BA_BF16 ? launch_t<__nv_bfloat16>(a, s) : launch_t<float>(a, s);
}

}  // namespace ba
