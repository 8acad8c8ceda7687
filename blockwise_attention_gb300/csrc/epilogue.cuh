// Row epilogue shared by the attention kernels: normalise the running
// weighted sum, optionally merge it with an fp32 partial attention already in
// memory (LSE rule), and store out / lse.
#pragma once

#include <cuda_bf16.h>

#include "internal.h"

namespace ba {

// LSE merge weights of an accumulated partial (La) and a new block (Lb),
// natural log: L = M + log(e^(La-M) + e^(Lb-M)), wa = e^(La-L), wb = e^(Lb-L).
// A side with -inf carries no keys and gets weight 0.
__device__ __forceinline__ void merge_weights(float La, float Lb, float &wa, float &wb, float &L) {
    if (Lb == -INFINITY) {
        wa = La == -INFINITY ? 0.f : 1.f;   // both empty: no key at all, out = 0
        wb = 0.f;
        L = La;
        return;
    }
    if (La == -INFINITY) {
        wa = 0.f;
        wb = 1.f;
        L = Lb;
        return;
    }
    float M = fmaxf(La, Lb);
    L = M + logf(expf(La - M) + expf(Lb - M));
    wa = expf(La - L);
    wb = expf(Lb - L);
}

// Per-row finalisation state computed once from (m, l) of the online softmax.
struct RowFinal {
    float wa, wb;   // weights of the accumulator row and of (o / l)
    float inv_l;    // 1 / l (0 when the block saw no key)
    float lse;      // merged natural-log LSE to store
};

// m2: running maximum in log2 units of scaled scores; l: running denominator
// relative to 2^m2.  acc_lse: accumulator LSE or -inf when there is none.
__device__ __forceinline__ RowFinal row_final(float m2, float l, float acc_lse) {
    RowFinal f;
    float Lb = -INFINITY;
    f.inv_l = 0.f;
    if (l > 0.f) {
        Lb = (m2 + log2f(l)) * LN2;
        f.inv_l = 1.f / l;
    }
    merge_weights(acc_lse, Lb, f.wa, f.wb, f.lse);
    return f;
}

// Store n (multiple of 8) consecutive output values of row `row_flat`
// starting at column c0: out = wa * acc + wb * inv_l * o.
__device__ __forceinline__ void store_row_chunk(const AttnArgs &a, long long row_flat, int c0,
                                                const float *o, int n, const RowFinal &f) {
    const int d = a.g.d;
    float vals[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) {
        if (i < n) vals[i] = f.wb * (o[i] * f.inv_l);
    }
    if (a.acc_o != nullptr && f.wa != 0.f) {
        const float4 *src = reinterpret_cast<const float4 *>(a.acc_o + row_flat * d + c0);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            if (4 * i < n) {
                float4 t = src[i];
                vals[4 * i + 0] += f.wa * t.x;
                vals[4 * i + 1] += f.wa * t.y;
                vals[4 * i + 2] += f.wa * t.z;
                vals[4 * i + 3] += f.wa * t.w;
            }
        }
    }
    if (a.out_dtype == BA_BF16) {
        uint4 *dst = reinterpret_cast<uint4 *>(static_cast<__nv_bfloat16 *>(a.out) + row_flat * d + c0);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            if (8 * i < n) {
                uint4 u;
                __nv_bfloat162 p0 = __floats2bfloat162_rn(vals[8 * i + 0], vals[8 * i + 1]);
                __nv_bfloat162 p1 = __floats2bfloat162_rn(vals[8 * i + 2], vals[8 * i + 3]);
                __nv_bfloat162 p2 = __floats2bfloat162_rn(vals[8 * i + 4], vals[8 * i + 5]);
                __nv_bfloat162 p3 = __floats2bfloat162_rn(vals[8 * i + 6], vals[8 * i + 7]);
                u.x = *reinterpret_cast<uint32_t *>(&p0);
                u.y = *reinterpret_cast<uint32_t *>(&p1);
                u.z = *reinterpret_cast<uint32_t *>(&p2);
                u.w = *reinterpret_cast<uint32_t *>(&p3);
                dst[i] = u;
            }
        }
    } else {
        float4 *dst = reinterpret_cast<float4 *>(static_cast<float *>(a.out) + row_flat * d + c0);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            if (4 * i < n) dst[i] = make_float4(vals[4 * i], vals[4 * i + 1], vals[4 * i + 2], vals[4 * i + 3]);
        }
    }
}

}  // namespace ba
