// Ulysses all-to-all on one GPU ("Sequence/context parallelism" (brunomaga),
// section "Ulysses sequence parallelism"; "Change token partitions into head
// partitions with Ulysses").
//
// P emulated ranks.  Token-split side: rank r holds tokens [r T/P, (r+1) T/P)
// of every head, stacked as one contiguous (P, H, B, T/P, d) array.  Head-split
// side: rank r holds heads [r H/P, (r+1) H/P) for every token; here it is any
// strided (B, H, T, d) view, which covers the stacked (P, H/P, B, T, d) array
// (sH = B T d, sB = T d, sT = d) as well as the contiguous (B, H, T, d) output
// of the attention kernel.  The exchange is a permutation of whole d-rows:
// token-split row (r, h, b, tl) <-> head-side row (b, h, t = r T/P + tl).  It
// is bound by HBM (each byte read once and written once).  When the head side
// keeps consecutive tokens in consecutive rows (sT = d, true of both layouts
// above), the rows of one (r, h, b) for a run of tokens are a contiguous span on
// both sides: a block copies one span of up to 64 rows, with its index
// arithmetic done once, in 16-byte vectors when sizes and addresses allow.
#include <cuda_runtime.h>

#include <cstdint>

#include "internal.h"

namespace ba {
namespace {

template <typename U>
__global__ void __launch_bounds__(256) a2a_kernel(const UlyssesArgs a) {
    const long long vec_per_row = a.row_bytes / (long long)sizeof(U);
    const long long n_rows = (long long)a.P * a.H * a.B * a.Tl;
    const long long total = n_rows * vec_per_row;
    const long long stride = (long long)gridDim.x * blockDim.x;
    for (long long v = (long long)blockIdx.x * blockDim.x + threadIdx.x; v < total; v += stride) {
        const long long n = v / vec_per_row, col = v % vec_per_row;
        // token-split row n = ((r * H + h) * B + b) * Tl + tl
        const long long tl = n % a.Tl;
        long long rest = n / a.Tl;
        const long long b = rest % a.B;
        rest /= a.B;
        const long long h = rest % a.H;
        const long long r = rest / a.H;
        const long long t = r * a.Tl + tl;
        const long long head_off = (b * a.sB + h * a.sH + t * a.sT) * a.elem_bytes;   // bytes
        const long long tok_off = n * a.row_bytes;
        const U *src;
        U *dst;
        if (a.to_head) {
            src = reinterpret_cast<const U *>(static_cast<const uint8_t *>(a.tok) + tok_off);
            dst = reinterpret_cast<U *>(static_cast<uint8_t *>(a.head) + head_off);
        } else {
            src = reinterpret_cast<const U *>(static_cast<const uint8_t *>(a.head) + head_off);
            dst = reinterpret_cast<U *>(static_cast<uint8_t *>(a.tok) + tok_off);
        }
        dst[col] = src[col];
    }
}

constexpr int SPAN_ROWS = 64;

// One block per span: (r, h, b) and up to SPAN_ROWS consecutive local tokens.
template <typename U>
__global__ void __launch_bounds__(256) a2a_span_kernel(const UlyssesArgs a, int spans_per_rhb) {
    const long long sid = blockIdx.x;
    const long long rhb = sid / spans_per_rhb;
    const int tl0 = (int)(sid % spans_per_rhb) * SPAN_ROWS;
    const int rows = min(SPAN_ROWS, a.Tl - tl0);
    const long long b = rhb % a.B, h = (rhb / a.B) % a.H, r = rhb / ((long long)a.B * a.H);
    const long long tok_off = (rhb * a.Tl + tl0) * a.row_bytes;
    const long long head_off = (b * a.sB + h * a.sH + (r * a.Tl + tl0) * a.sT) * a.elem_bytes;
    const uint8_t *src;
    uint8_t *dst;
    if (a.to_head) {
        src = static_cast<const uint8_t *>(a.tok) + tok_off;
        dst = static_cast<uint8_t *>(a.head) + head_off;
    } else {
        src = static_cast<const uint8_t *>(a.head) + head_off;
        dst = static_cast<uint8_t *>(a.tok) + tok_off;
    }
    const int n = (int)(rows * a.row_bytes / (long long)sizeof(U));
    const U *s = reinterpret_cast<const U *>(src);
    U *d = reinterpret_cast<U *>(dst);
    for (int i = threadIdx.x; i < n; i += blockDim.x) d[i] = s[i];
}

template <typename U>
int launch_span(const UlyssesArgs &a, cudaStream_t s) {
    const int spans_per = (a.Tl + SPAN_ROWS - 1) / SPAN_ROWS;
    const long long blocks = (long long)a.P * a.H * a.B * spans_per;
    if (blocks > 0x7fffffffLL) return BA_ERR_SHAPE;
    a2a_span_kernel<U><<<(unsigned)blocks, 256, 0, s>>>(a, spans_per);
    return cudaGetLastError() == cudaSuccess ? BA_OK : BA_ERR_CUDA;
}

template <typename U>
int launch_u(const UlyssesArgs &a, int num_sms, cudaStream_t s) {
    const long long total = (long long)a.P * a.H * a.B * a.Tl * (a.row_bytes / (long long)sizeof(U));
    long long blocks = (total + 255) / 256;
    const long long cap = (long long)num_sms * 8;   // 8 resident blocks of 256 per SM
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    a2a_kernel<U><<<(int)blocks, 256, 0, s>>>(a);
    return cudaGetLastError() == cudaSuccess ? BA_OK : BA_ERR_CUDA;
}

bool aligned(const UlyssesArgs &a, long long unit) {
    const uintptr_t p1 = reinterpret_cast<uintptr_t>(a.tok), p2 = reinterpret_cast<uintptr_t>(a.head);
    return a.row_bytes % unit == 0 && p1 % unit == 0 && p2 % unit == 0 && (a.sB * a.elem_bytes) % unit == 0 &&
           (a.sH * a.elem_bytes) % unit == 0 && (a.sT * a.elem_bytes) % unit == 0;
}

}  // namespace

int launch_ulysses_a2a(const UlyssesArgs &a, int num_sms, cudaStream_t s) {
    if ((long long)a.P * a.H * a.B * a.Tl == 0 || a.row_bytes == 0) return BA_OK;
    if (a.sT * a.elem_bytes == a.row_bytes) {   // consecutive tokens in consecutive rows
        if (aligned(a, 16)) return launch_span<uint4>(a, s);
        if (aligned(a, 4)) return launch_span<uint32_t>(a, s);
        if (aligned(a, 2)) return launch_span<uint16_t>(a, s);
        return launch_span<uint8_t>(a, s);
    }
    if (aligned(a, 16)) return launch_u<uint4>(a, num_sms, s);
    if (aligned(a, 4)) return launch_u<uint32_t>(a, num_sms, s);
    if (aligned(a, 2)) return launch_u<uint16_t>(a, num_sms, s);
    return launch_u<uint8_t>(a, num_sms, s);
}

}  // namespace ba
