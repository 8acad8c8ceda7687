// C-ABI entry points of libblockattn.so (declared in include/blockattn.h):
// argument checks, geometry set-up, workspace carving, TMA descriptors and
// kernel dispatch, plus the bandwidth-bound kernels (LSE merge, RoPE, tile
// classes) and the host-side index maps.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cudaTypedefs.h>

#include <cmath>
#include <cstring>
#include <mutex>

#include "internal.h"

using namespace ba;

namespace {

// ---------------------------------------------------------------------------
// device error word (one per device, lives as long as the module)
// ---------------------------------------------------------------------------
__device__ unsigned g_err_word;

// Fixed scratch of attn_block_fwd_noalloc: the tile-class map, for callers that
// cannot allocate.  Present on every device that loads the library.
static __device__ __align__(256) int8_t g_noalloc_classes[BA_NOALLOC_MAX_CLASS_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
unsigned *g_err_ptr[kMaxDevices];
int g_num_sms[kMaxDevices];
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

int current_device() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return -1;
    return dev < kMaxDevices ? dev : -1;
}

// Per-device set-up, done once with the device current: the address of the
// error word and the SM count.
int device_setup(int dev) {
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_err_ptr[dev]) return BA_OK;
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_err_word) != cudaSuccess) return BA_ERR_CUDA;
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return BA_ERR_CUDA;
    g_num_sms[dev] = sms;
    g_err_ptr[dev] = static_cast<unsigned *>(p);
    return BA_OK;
}

// Device address of g_noalloc_classes on device `dev` (which must be current),
// looked up on the first call on that device.  Host code may not use the
// array's name as a device pointer: it names a host-side stand-in.
int8_t *g_noalloc_ptr[kMaxDevices];

int noalloc_scratch(int dev, int8_t **out) {
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_noalloc_ptr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_classes) != cudaSuccess || p == nullptr) return BA_ERR_CUDA;
        g_noalloc_ptr[dev] = static_cast<int8_t *>(p);
    }
    *out = g_noalloc_ptr[dev];
    return BA_OK;
}

int get_encoder() {
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_encode) return BA_OK;
    void *fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess || fn == nullptr)
        return BA_ERR_CUDA;
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    return BA_OK;
}

constexpr unsigned long long kWaitLimitNs = 4000000000ull;  // 4 s: far beyond any legitimate wait

size_t elem_size(int dtype) { return dtype == BA_F32 ? 4 : 2; }

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// Workspace block at the front of every attention workspace: one 32-bit item
// counter per kernel launch of the call, zeroed on the stream before them.
size_t sched_bytes(int launches) { return align256((size_t)4 * (size_t)(launches > 0 ? launches : 1)); }

int zero_sched(void *p, int launches, cudaStream_t s) {
    return cudaMemsetAsync(p, 0, (size_t)4 * (size_t)launches, s) == cudaSuccess ? BA_OK : BA_ERR_CUDA;
}

bool valid_dtype(int t) { return t == BA_F32 || t == BA_BF16; }
bool valid_d(int d) { return d == 16 || d == 32 || d == 64 || d == 128; }

// (B, H, rows, d) bf16 tensor map: 4-D, box 64 columns x box_rows rows, 128B swizzle.
int encode_map(CUtensorMap *m, const void *base, int d, long long rows, int H, int B, long long sT, long long sH,
               long long sB, int box_rows = TILE) {
    cuuint64_t dims[4] = {(cuuint64_t)d, (cuuint64_t)rows, (cuuint64_t)H, (cuuint64_t)B};
    cuuint64_t strides[3] = {(cuuint64_t)sT * 2, (cuuint64_t)sH * 2, (cuuint64_t)sB * 2};
    cuuint32_t box[4] = {64, (cuuint32_t)box_rows, 1, 1};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(base), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? BA_OK : BA_ERR_CUDA;
}

// Striped ring: the (B, H, T, d) tensor seen as {d, P, T/P, H, B}, token
// r + P u at coordinates (r, u), so that a box {64, 1, 128, 1, 1} loads 128
// consecutive tokens of rank r (a stride of P rows) into the same shared-memory
// layout as the 4-D box (box_rows consecutive tokens of the rank for the stores).
int encode_map_striped(CUtensorMap *m, const void *base, int d, int P, long long T, int H, int B, long long sT,
                       long long sH, long long sB, int box_rows = TILE) {
    cuuint64_t dims[5] = {(cuuint64_t)d, (cuuint64_t)P, (cuuint64_t)(T / P), (cuuint64_t)H, (cuuint64_t)B};
    cuuint64_t strides[4] = {(cuuint64_t)sT * 2, (cuuint64_t)sT * 2 * P, (cuuint64_t)sH * 2, (cuuint64_t)sB * 2};
    cuuint32_t box[5] = {64, 1, (cuuint32_t)box_rows, 1, 1};
    cuuint32_t estr[5] = {1, 1, 1, 1, 1};
    CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void *>(base), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? BA_OK : BA_ERR_CUDA;
}

// TMA needs 16-byte aligned bases and byte strides; B or H of 1 may carry any stride.
bool tma_ok(const ba_tensor &t, int B, int H) {
    auto al = [](long long s) { return (s * 2) % 16 == 0 && s >= 0; };
    if (reinterpret_cast<uintptr_t>(t.ptr) % 16) return false;
    if (!al(t.sT)) return false;
    if (H > 1 && !al(t.sH)) return false;
    if (B > 1 && !al(t.sB)) return false;
    return true;
}

ba_tensor fix_unit_strides(ba_tensor t, int B, int H, int rows, int d) {
    // A size-1 axis may have any stride; give it a legal one for TMA.
    if (H <= 1) t.sH = (long long)rows * t.sT > 0 ? (long long)rows * t.sT : d;
    if (B <= 1) t.sB = (long long)H * t.sH > 0 ? (long long)H * t.sH : d;
    return t;
}

int heads_per_group(int B, int H, long long keys, int d, int dtype) {
    const double per_head = 2.0 * (double)keys * d * elem_size(dtype);
    long long G = (long long)(48.0 * 1024 * 1024 / (per_head > 1 ? per_head : 1));
    if (G < 1) G = 1;
    if (G > (long long)B * H) G = (long long)B * H;
    return (int)(G < 1 ? 1 : G);
}

// ---------------------------------------------------------------------------
// small kernels
// ---------------------------------------------------------------------------

// Exclusion bytes (nonzero = excluded) of keys [j0, j0 + 16) of a mask row,
// of which the first n exist: one 16-byte load when they all exist and the
// row is aligned, byte loads otherwise.
__device__ __forceinline__ uint4 mask16(const uint8_t *p, int n) {
    if (n >= 16 && (reinterpret_cast<uintptr_t>(p) & 15) == 0) return __ldg(reinterpret_cast<const uint4 *>(p));
    uint32_t w[4] = {0u, 0u, 0u, 0u};
    for (int i = 0; i < 16 && i < n; ++i) w[i >> 2] |= (uint32_t)__ldg(p + i) << (8 * (i & 3));
    return make_uint4(w[0], w[1], w[2], w[3]);
}

// Class of every (b, q tile, k tile) of the walk geometry: one CTA per tile
// pair, one thread per query row, which reads its key-padding and attn_mask
// bytes 16 keys at a time.  (Masks are never taken with striped ranks, so the
// positions are the tokens.)
__global__ void tile_class_kernel(const Geom g, int8_t *cls) {
    const int kg = blockIdx.x, qg = blockIdx.y, b = blockIdx.z;
    const QTile q = q_tile<false>(g, qg, b, 0);
    const KTile k = k_tile_by_id(g, kg);
    const int i = threadIdx.x;
    int any = 0, all = 1;
    if (i < q.len) {
        const long long qp = q.pos0 + i;
        const uint8_t *kr = g.kpm ? g.kpm + b * g.kpm_ld + k.pos0 : nullptr;
        const uint8_t *ar = g.am ? g.am + qp * g.am_ld + k.pos0 : nullptr;
        const long long lim = g.causal ? qp - k.pos0 : (long long)TILE;   // keys j > lim lie in the future
        for (int j0 = 0; j0 < k.len; j0 += 16) {
            const int n = k.len - j0;
            const uint4 ek = kr ? mask16(kr + j0, n) : make_uint4(0u, 0u, 0u, 0u);
            const uint4 ea = ar ? mask16(ar + j0, n) : make_uint4(0u, 0u, 0u, 0u);
            const uint32_t e[4] = {ek.x | ea.x, ek.y | ea.y, ek.z | ea.z, ek.w | ea.w};
#pragma unroll
            for (int jj = 0; jj < 16; ++jj) {
                if (jj >= n) break;
                const bool vis = ((e[jj >> 2] >> (8 * (jj & 3))) & 0xffu) == 0u && j0 + jj <= lim;
                any |= vis;
                all &= vis;
            }
        }
    }
    any = __syncthreads_or(any);
    all = __syncthreads_and(all);
    if (i == 0) cls[((long long)b * g.n_qtiles + qg) * g.n_ktiles + kg] =
        (int8_t)(!any ? BA_TILE_EMPTY : (all ? BA_TILE_FULL : BA_TILE_PARTIAL));
}

// LSE merge weights (natural log) of one row: a <- wa a + wb b, lse <- L.
// Returns false when b carries no keys and a stays as it is.
__device__ __forceinline__ bool merge_row_weights(float A, float Bv, float &wa, float &wb, float &L) {
    if (Bv == -INFINITY) {
        if (A != -INFINITY) return false;   // nothing to fold in: a unchanged
        wa = wb = 0.f;                      // neither side saw a key: out = 0, lse = -inf
        L = -INFINITY;
        return true;
    }
    if (A == -INFINITY) {
        wa = 0.f;
        wb = 1.f;
        L = Bv;
        return true;
    }
    const float M = fmaxf(A, Bv);
    L = M + logf(expf(A - M) + expf(Bv - M));
    wa = expf(A - L);
    wb = expf(Bv - L);
    return true;
}

// a <- merge(a, b) for rows of d <= 128 columns, d a multiple of 4 and 16-byte
// aligned rows: one warp per row, lane c holding columns 4c .. 4c+3; each warp
// takes two rows per iteration and issues all four loads of both (LSEs and
// rows) before it computes, so that the loads of a row do not wait for its
// weights.  Streaming loads and stores: every byte is touched once.
__global__ void __launch_bounds__(256) merge_vec_kernel(float4 *__restrict__ oa, float *__restrict__ la,
                                                        const float4 *__restrict__ ob,
                                                        const float *__restrict__ lb, long long rows, int nv) {
    const int lane = threadIdx.x & 31;
    const long long warps = (long long)gridDim.x * (blockDim.x >> 5);
    const long long w0 = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    const bool col = lane < nv;
    for (long long r0 = w0; r0 < rows; r0 += 2 * warps) {
        const long long rr[2] = {r0, r0 + warps};
        float A[2], Bv[2];
        float4 x[2], y[2];
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const bool in = rr[u] < rows;
            A[u] = in ? __ldcs(la + rr[u]) : 0.f;
            Bv[u] = in ? __ldcs(lb + rr[u]) : 0.f;
            x[u] = in && col ? __ldcs(oa + rr[u] * nv + lane) : make_float4(0.f, 0.f, 0.f, 0.f);
            y[u] = in && col ? __ldcs(ob + rr[u] * nv + lane) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            if (rr[u] >= rows) continue;
            float wa, wb, L;
            if (!merge_row_weights(A[u], Bv[u], wa, wb, L)) continue;
            if (col) {
                float4 o;
                // a side of weight 0 contributes 0 whatever its row holds
                o.x = (wa != 0.f ? wa * x[u].x : 0.f) + wb * y[u].x;
                o.y = (wa != 0.f ? wa * x[u].y : 0.f) + wb * y[u].y;
                o.z = (wa != 0.f ? wa * x[u].z : 0.f) + wb * y[u].z;
                o.w = (wa != 0.f ? wa * x[u].w : 0.f) + wb * y[u].w;
                __stcs(oa + rr[u] * nv + lane, o);
            }
            if (lane == 0) la[rr[u]] = L;
        }
    }
}

// a <- merge(a, b), any d: one warp per row.
__global__ void merge_kernel(float *__restrict__ oa, float *__restrict__ la, const float *__restrict__ ob,
                             const float *__restrict__ lb, long long rows, int d) {
    const int lane = threadIdx.x & 31;
    const long long warps = (long long)gridDim.x * (blockDim.x >> 5);
    for (long long r = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); r < rows; r += warps) {
        float wa, wb, L;
        if (!merge_row_weights(la[r], lb[r], wa, wb, L)) continue;
        float *pa = oa + r * d;
        const float *pb = ob + r * d;
        for (int c = lane; c < d; c += 32) pa[c] = (wa != 0.f ? wa * pa[c] : 0.f) + wb * pb[c];
        if (lane == 0) la[r] = L;
    }
}

struct Thetas {
    double th[64];
};

// Up to two tensors rotated by one launch (Q and K share the angles).
struct RopeArgs {
    const void *x[2];
    long long sB[2], sH[2], sT[2];
    void *y[2];
    int n;
    int B, H, T, d;
    const int32_t *positions;
    double pos_scale;       // Position Interpolation: angle = (position * pos_scale) * theta
    unsigned *err;          // device error word (bounded waits of the bulk-copy kernel)
    unsigned long long wait_limit_ns;
    Thetas th;
    float4 tab[128];   // (cos hi, cos lo, sin hi, sin lo) of n pi / 64, n = 0 .. 127 (sincos_ff)
};

// fp64 -> bf16 with one rounding (ties to even): truncate to fp32, make the
// result's last bit sticky when inexact (round-to-odd), then round to bf16.
__device__ __forceinline__ __nv_bfloat16 round_bf16_from_f64(double y) {
    float f = __double2float_rz(y);
    if ((double)f != y && isfinite(f)) f = __uint_as_float(__float_as_uint(f) | 1u);
    return __float2bfloat16_rn(f);
}

// Error-free sum of two floats (Knuth): a + b = s + e exactly.
__device__ __forceinline__ void two_sum(float a, float b, float &s, float &e) {
    s = __fadd_rn(a, b);
    const float bb = __fsub_rn(s, a);
    e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb));
}

// A value split into four floats of at most 16 significant bits each, so that
// the product of any piece with a bfloat16 value (8 significant bits) is exact
// in fp32 (split4_ff builds one from a float-float).
struct Split4 {
    float k[4];
};

// x0 * c - x1 * s (or x0 * s + x1 * c with the roles passed in) for bfloat16
// x0, x1, rounded once to bfloat16.  Level-1 and level-2 products are exact
// and summed with error-free transforms; the rest carries < 2^-47 |x|.
__device__ __forceinline__ uint16_t rot_bf16(float x0, const Split4 &a, float x1, const Split4 &b) {
    // y = x0 * a - x1 * b
    float h1, l1, h2, l2;
    two_sum(__fmul_rn(x0, a.k[0]), -__fmul_rn(x1, b.k[0]), h1, l1);
    two_sum(__fmul_rn(x0, a.k[1]), -__fmul_rn(x1, b.k[1]), h2, l2);
    const float t3 = __fsub_rn(__fmul_rn(x0, a.k[2]), __fmul_rn(x1, b.k[2]));
    const float t4 = __fsub_rn(__fmul_rn(x0, a.k[3]), __fmul_rn(x1, b.k[3]));
    float s, e;
    two_sum(h1, h2, s, e);
    const float small = __fadd_rn(__fadd_rn(__fadd_rn(l1, l2), __fadd_rn(t3, t4)), e);
    float hi, lo;
    two_sum(s, small, hi, lo);               // hi + lo = value, |lo| <= ulp(hi) / 2
    // Round hi + lo to bfloat16: only when hi sits exactly on a bfloat16
    // midpoint does lo decide the direction.
    const uint32_t u = __float_as_uint(hi);
    uint32_t bits;
    if ((u & 0xFFFFu) == 0x8000u && lo != 0.f) {
        const bool away = (lo > 0.f) == (hi > 0.f);
        bits = away ? (u + 0x8000u) >> 16 : u >> 16;
    } else {
        bits = __bfloat16_as_ushort(__float2bfloat16_rn(hi));
    }
    return (uint16_t)bits;
}

// A float-float value hi + lo (|lo| at most about 2^-24 |hi|): 48 significant
// bits carried by the fp32 pipe, which runs far faster than the fp64 one.
struct FF {
    float hi, lo;
};

// x y: the product of the high parts split exactly by an fma, plus the cross
// terms (relative error about 2^-47).
__device__ __forceinline__ FF ff_mul(FF x, FF y) {
    const float p = x.hi * y.hi;
    const float e = fmaf(x.hi, y.hi, -p);
    return FF{p, fmaf(x.hi, y.lo, fmaf(x.lo, y.hi, e))};
}

// x + y: Knuth's two-sum of the high parts plus the low parts, renormalised.
__device__ __forceinline__ FF ff_add(FF x, FF y) {
    const float s = x.hi + y.hi;
    const float bb = s - x.hi;
    const float e = (x.hi - (s - bb)) + (y.hi - bb);
    const float l = e + (x.lo + y.lo);
    const float h = s + l;
    return FF{h, l - (h - s)};
}

__device__ __forceinline__ FF ff_neg(FF x) { return FF{-x.hi, -x.lo}; }

// sin and cos of an fp64 angle a to about 2^-48 absolute, table-driven (Tang's
// method).  In fp64 only the reduction: a = n pi/64 + r, |r| <= pi/128, with
// pi/64 split into pieces of 27, 27 and 24 significant bits (n * piece exact
// for |n| < 2^23); r goes to float-float, the third piece's product folded
// into its low part.  Then in float-float on the fp32 pipe: the Taylor series
// of sin r and cos r (the r^3/3! and r^2/2! terms carried with their rounding
// errors, r^5/5!, r^7/7!, r^4/4!, r^6/6! in fp32, the next terms below 2^-60),
// and the angle sum with the table entries cos, sin (n pi / 64), n mod 128.
// Angles of 2^19 and beyond take sincos() in fp64.
__device__ __forceinline__ void sincos_ff(double a, const float4 *tab, FF &sn, FF &cs) {
    constexpr double K = 0x1.45f306dc9c883p+4;        // 64 / pi
    constexpr double Q1 = 0x1.921fb54000000p-5;       // pi / 64 = Q1 + Q2 + Q3 (+ 5e-28)
    constexpr double Q2 = 0x1.10b4612000000p-35;
    constexpr float Q3 = -0x1.676734p-65f;
    constexpr float K6 = 0x1.555556p-3f;              // 1/6 = K6 + K6E (+ 2^-52)
    constexpr float K6E = -0x1.555556p-28f;
    if (!(fabs(a) < 524288.0)) {
        double sv, cv;
        sincos(a, &sv, &cv);
        const float sh = __double2float_rn(sv), ch = __double2float_rn(cv);
        sn = FF{sh, __double2float_rn(sv - (double)sh)};
        cs = FF{ch, __double2float_rn(cv - (double)ch)};
        return;
    }
    const double nd = rint(a * K);
    double r = fma(-nd, Q1, a);
    r = fma(-nd, Q2, r);
    const int n = (int)nd;
    const float rh = __double2float_rn(r);
    const float rl = fmaf(-(float)n, Q3, __double2float_rn(r - (double)rh));
    const float p = rh * rh, pe = fmaf(rh, rh, -p);     // rh^2 = p + pe exactly
    // sin r = r - r^3/6 + r^5/120 - r^7/5040
    const float c3 = p * rh, c3e = fmaf(p, rh, -c3);     // rh^3 = c3 + c3e + pe rh
    const float l3 = c3e + fmaf(pe, rh, 3.f * p * rl);   // with the 3 rh^2 rl term of r^3
    const float t3h = c3 * K6, t3e = fmaf(c3, K6, -t3h);
    const float t3l = t3e + fmaf(c3, K6E, l3 * K6);      // r^3 / 6 = t3h + t3l
    const float t57 = rh * p * p * fmaf(p, -1.f / 5040.f, 1.f / 120.f);
    const float s1 = rh - t3h, s1e = (rh - s1) - t3h;    // exact (|rh| >= |t3h|)
    const FF sin_r{s1, ((s1e + rl) - t3l) + t57};
    // cos r = 1 - r^2/2 + r^4/24 - r^6/720
    const float t2h = 0.5f * p, t2l = 0.5f * fmaf(2.f * rh, rl, pe);
    const float t46 = p * p * fmaf(p, -1.f / 720.f, 1.f / 24.f);
    const float c1 = 1.f - t2h, c1e = (1.f - c1) - t2h;  // exact
    const FF cos_r{c1, (c1e - t2l) + t46};
    const float4 t = tab[n & 127];                       // (cos hi, cos lo, sin hi, sin lo) of (n mod 128) pi/64
    const FF tc{t.x, t.y}, ts{t.z, t.w};
    cs = ff_add(ff_mul(tc, cos_r), ff_neg(ff_mul(ts, sin_r)));
    sn = ff_add(ff_mul(ts, cos_r), ff_mul(tc, sin_r));
}

// c = hi + lo with hi of 16 significant bits (its product with a bfloat16 is
// exact in fp32) and lo the fp32 rounding of the rest (|lo| < 2^-15 |c|).
__device__ __forceinline__ void split_hi_lo(FF c, float &hi, float &lo) {
    hi = __uint_as_float(__float_as_uint(c.hi) & 0xFFFFFF00u);
    lo = (c.hi - hi) + c.lo;
}

// c as four pieces of at most 16 significant bits whose sum is exactly
// c.hi + c.lo, so that each product with a bfloat16 is exact in fp32.
__device__ __forceinline__ Split4 split4_ff(FF c) {
    Split4 r;
    r.k[0] = __uint_as_float(__float_as_uint(c.hi) & 0xFFFFFF00u);
    r.k[1] = c.hi - r.k[0];
    r.k[2] = __uint_as_float(__float_as_uint(c.lo) & 0xFFFFFF00u);
    r.k[3] = c.lo - r.k[2];
    return r;
}

// Two fp32 lanes per instruction (sm_100 f32x2 forms), each lane an IEEE
// operation rounded to nearest.
__device__ __forceinline__ float2 mul2(float2 a, float2 b) {
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rd;\n\tmov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
        "mul.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y) : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
}
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) {
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\tmov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
        "mov.b64 rc, {%6, %7};\n\tfma.rn.f32x2 rd, ra, rb, rc;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y) : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
    return d;
}
__device__ __forceinline__ float2 add2(float2 a, float2 b) {
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rd;\n\tmov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
        "add.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y) : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
}

__device__ __forceinline__ uint32_t bf16x2_rn(float2 v) {
    __nv_bfloat162 p = __floats2bfloat162_rn(v.x, v.y);   // .x (low half) = v.x
    return *reinterpret_cast<uint32_t *>(&p);
}

// The split cos and sin of one pair's angle, arranged for the two-lane forms:
// lane 0 computes x0 c - x1 s, lane 1 computes x0 s + x1 c.
struct RopeRowPair {
    float2 hi;     // (c_hi,  s_hi)
    float2 hi_r;   // (-s_hi, c_hi)
    float2 lo;     // (c_lo,  s_lo)
    float2 lo_r;   // (-s_lo, c_lo)
};

// One output pair of bfloat16 inputs (x0, x1), packed as two bfloat16.  The
// rotation runs in fp32 on the split cos / sin: y = h + t with h = x0 c_hi -
// x1 s_hi (the products exact, one rounding) and t the low-part terms.  Its
// error is below E = 2^-22 |y| + 2^-36 (|x0| + |x1|) (the roundings of h and
// y, 2^-24 each, and 2^-37 |x| for the low parts and the split), see the
// exact path.  The packed result is safe when y - E' and y + E' (E' = E +
// 2^-22 |y| covering their own rounding) round to the same bfloat16: every
// value between them, the exact rotation included, rounds there as well
// (Ziv's rounding test).  Returns false when the test cannot decide.
__device__ __forceinline__ bool rot_fast2(float x0, float x1, const RopeRowPair &k, uint32_t &packed) {
    const float2 xx0 = make_float2(x0, x0), xx1 = make_float2(x1, x1);
    const float2 h = fma2(xx0, k.hi, mul2(xx1, k.hi_r));
    const float2 t = fma2(xx0, k.lo, mul2(xx1, k.lo_r));
    const float2 y = add2(h, t);
    const float a = fmaf(0x1p-36f, fabsf(x0) + fabsf(x1), 0x1p-126f);   // absolute term (and denormals)
    const float2 ay = make_float2(fabsf(y.x), fabsf(y.y));
    const float2 e = fma2(ay, make_float2(0x1p-21f, 0x1p-21f), make_float2(a, a));
    const uint32_t up = bf16x2_rn(add2(y, e));
    const uint32_t dn = bf16x2_rn(add2(y, make_float2(-e.x, -e.y)));
    packed = up;
    return up == dn;
}

// The four pairs 4 c0 .. 4 c0 + 3 at position t: cos and sin of their angles
// (float-float), split for the fast path (k) and kept whole for the exact one.
__device__ __forceinline__ void rope_setup(const RopeArgs &a, const float4 *tab, long long t, int c0,
                                           RopeRowPair (&k)[4], float4 (&exact)[4][256]) {
    const double m = (a.positions ? (double)a.positions[t] : (double)t) * a.pos_scale;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        FF cs, sn;
        sincos_ff(m * a.th.th[c0 + i], tab, sn, cs);
        float ch, cl, sh, sl;
        split_hi_lo(cs, ch, cl);
        split_hi_lo(sn, sh, sl);
        k[i].hi = make_float2(ch, sh);
        k[i].hi_r = make_float2(-sh, ch);
        k[i].lo = make_float2(cl, sl);
        k[i].lo_r = make_float2(-sl, cl);
        exact[i][threadIdx.x] = make_float4(cs.hi, cs.lo, sn.hi, sn.lo);
    }
}

// Rotate four bfloat16 pairs (one 16-byte word) by the fast path, falling back
// to the exact rotation for a pair whose rounding the test cannot decide.
__device__ __forceinline__ uint4 rope_rotate(const uint32_t (&w)[4], const RopeRowPair (&k)[4],
                                             const float4 (&exact)[4][256]) {
    uint32_t out[4];
    bool ok[4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
        ok[i] = rot_fast2(__uint_as_float(w[i] << 16), __uint_as_float(w[i] & 0xFFFF0000u), k[i], out[i]);
    if (!(ok[0] && ok[1] && ok[2] && ok[3])) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            if (ok[i]) continue;
            const float x0 = __uint_as_float(w[i] << 16), x1 = __uint_as_float(w[i] & 0xFFFF0000u);
            const float4 e = exact[i][threadIdx.x];
            const Split4 c4 = split4_ff(FF{e.x, e.y}), s4 = split4_ff(FF{e.z, e.w});
            Split4 nc4;
#pragma unroll
            for (int j = 0; j < 4; ++j) nc4.k[j] = -c4.k[j];
            out[i] = (uint32_t)rot_bf16(x0, c4, x1, s4) |                // x0 cos - x1 sin
                     ((uint32_t)rot_bf16(x0, s4, x1, nc4) << 16);       // x0 sin - x1 (-cos)
        }
    }
    return make_uint4(out[0], out[1], out[2], out[3]);
}

// Rows [r_begin, r_end) of the (tensor, b, h) list given to a CTA (blockIdx.y).
__device__ __forceinline__ void rope_rows(const RopeArgs &a, int &r_begin, int &r_end) {
    const int rows = a.n * a.B * a.H;
    const int per = (rows + gridDim.y - 1) / gridDim.y;
    r_begin = blockIdx.y * per;
    r_end = r_begin + per < rows ? r_begin + per : rows;
}

// bfloat16 with d a multiple of 8.  A CTA of 256 threads covers TP = 2048 / d
// positions x d columns; thread (t, g) owns the four pairs 4g .. 4g+3 at
// position t.  It computes their angles' cos and sin once (float-float,
// table-driven) and rotates those pairs in every row of the CTA's share of the
// (tensor, b, h) rows, four rows' 16-byte loads in flight at a time.  The
// rotation runs in fp32 with a rounding test; the rare coordinate the test
// cannot decide is recomputed exactly (rot_bf16), so every output is the exact
// rotation rounded once to bfloat16.  (Strided rows; contiguous ones take the
// bulk-copy kernel below.)
template <bool VEC>
__global__ void __launch_bounds__(256, 3) rope_bf16_kernel(const RopeArgs a) {
    __shared__ float4 tab[128];
    __shared__ float4 exact[4][256];   // float-float (cos, sin) of each thread's pairs, for the exact path
    if (threadIdx.x < 128) tab[threadIdx.x] = a.tab[threadIdx.x];
    __syncthreads();
    const int G = a.d / 8;
    const int TP = 256 / G;
    const int tl = threadIdx.x / G, grp = threadIdx.x % G;
    const long long t = (long long)blockIdx.x * TP + tl;
    if (tl >= TP || t >= a.T) return;
    const int c0 = grp * 4;
    RopeRowPair k[4];
    rope_setup(a, tab, t, c0, k, exact);
    int r_begin, r_end;
    rope_rows(a, r_begin, r_end);
    constexpr int U = 4;
    for (int r0 = r_begin; r0 < r_end; r0 += U) {
        uint32_t w[U][4];
        __nv_bfloat16 *py[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int r = r0 + u;
            py[u] = nullptr;
            if (r >= r_end) continue;
            const int ti = r / (a.B * a.H), bh = r % (a.B * a.H), b = bh / a.H, h = bh % a.H;
            const __nv_bfloat16 *px = static_cast<const __nv_bfloat16 *>(a.x[ti]) + b * a.sB[ti] +
                                      h * a.sH[ti] + t * a.sT[ti] + 2 * c0;
            py[u] = static_cast<__nv_bfloat16 *>(a.y[ti]) + ((long long)bh * a.T + t) * a.d + 2 * c0;
            if (VEC) {
                const uint4 v = __ldcs(reinterpret_cast<const uint4 *>(px));
                w[u][0] = v.x; w[u][1] = v.y; w[u][2] = v.z; w[u][3] = v.w;
            } else {
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    w[u][i] = (uint32_t)__bfloat16_as_ushort(px[2 * i]) |
                              ((uint32_t)__bfloat16_as_ushort(px[2 * i + 1]) << 16);
            }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            if (py[u] == nullptr) continue;
            *reinterpret_cast<uint4 *>(py[u]) = rope_rotate(w[u], k, exact);
        }
    }
}

// bfloat16, d a multiple of 8, contiguous rows (sT = d): the CTA's positions
// are one contiguous block of TP d 2 = 4096 bytes in every row, which one
// thread streams into a ring of ROPE_RING shared-memory slots with bulk copies
// (cp.async.bulk, completion counted on a "full" mbarrier per slot), ROPE_RING
// rows ahead of the rotation.  Each thread reads its 16 bytes of a slot,
// rotates them as in rope_bf16_kernel and stores the result; each warp then
// signals the slot's "empty" mbarrier, and the streaming thread refills the
// slot once all eight warps have.  Many rows' bytes are in flight per CTA
// without registers held for them, and no block-wide barrier is taken per
// row.  Every wait is bounded: on expiry the thread records the timeout and
// stops (the streaming thread first lets its copies in flight land).
constexpr int ROPE_RING = 12;   // 48 KB of slots (even: rows go two by two); three CTAs an SM keep 144 KB in flight
__global__ void __launch_bounds__(256, 3) rope_bf16_bulk_kernel(const RopeArgs a) {
    __shared__ float4 tab[128];
    __shared__ float4 exact[4][256];
    extern __shared__ __align__(128) uint4 ring_mem[];   // ROPE_RING slots of 256 16-byte words
    uint4(*ring)[256] = reinterpret_cast<uint4(*)[256]>(ring_mem);
    __shared__ __align__(8) uint64_t full[ROPE_RING], empty[ROPE_RING];
    __shared__ int abort_flag;
    if (threadIdx.x < 128) tab[threadIdx.x] = a.tab[threadIdx.x];
    if (threadIdx.x == 0) {
        for (int i = 0; i < ROPE_RING; ++i) {
            mbar_init(smem_u32(&full[i]), 1);
            mbar_init(smem_u32(&empty[i]), 8);   // one arrival per warp
        }
        abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    const int G = a.d / 8;
    const int TP = 256 / G;
    const int tl = threadIdx.x / G, grp = threadIdx.x % G;
    const long long t0 = (long long)blockIdx.x * TP;
    const long long t = t0 + tl;
    const bool valid = tl < TP && t < a.T;   // (256 = TP G exactly when d divides 2048)
    const int tp = a.T - t0 < TP ? (int)(a.T - t0) : TP;   // positions of this block
    const uint32_t bytes = (uint32_t)tp * (uint32_t)a.d * 2u;
    int r_begin, r_end;
    rope_rows(a, r_begin, r_end);
    const int BH = a.B * a.H;
    // row r = (tensor ti, b, h): positions t0 .. t0 + tp - 1 of head (b, h)
    auto src = [&](int r) -> const void * {
        const int ti = r / BH, bh = r % BH, b = bh / a.H, h = bh % a.H;
        return static_cast<const __nv_bfloat16 *>(a.x[ti]) + b * a.sB[ti] + h * a.sH[ti] + t0 * a.sT[ti];
    };
    auto issue = [&](int slot, int r) {
        const uint32_t bar = smem_u32(&full[slot]);
        mbar_arrive_expect_tx(bar, bytes);
        asm volatile(
            "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                smem_u32(&ring[slot][0])),
            "l"(src(r)), "r"(bytes), "r"(bar)
            : "memory");
    };
    int issued = 0;   // rows issued (thread 0)
    if (threadIdx.x == 0)
        for (; issued < ROPE_RING && r_begin + issued < r_end; ++issued) issue(issued, r_begin + issued);
    RopeRowPair k[4];
    if (valid) rope_setup(a, tab, t, grp * 4, k, exact);
    // output row pointer, advanced row by row: (ti, bh) of row r_begin, then bh + 1 ...
    int ti = r_begin / BH, bh = r_begin % BH;
    const long long step = (long long)a.T * a.d;
    __nv_bfloat16 *py = static_cast<__nv_bfloat16 *>(a.y[ti]) + ((long long)bh * a.T + t) * a.d + grp * 8;
    auto advance = [&]() {   // py to the next row
        if (++bh == BH) {
            bh = 0;
            ++ti;
            py = static_cast<__nv_bfloat16 *>(a.y[ti < a.n ? ti : 0]) + (long long)t * a.d + grp * 8;
        } else {
            py += step;
        }
    };
    // refill slot with row r_begin + issued (= the row ROPE_RING after the one just read)
    // once every warp has read it; false when the wait expired
    auto refill = [&](int slot, uint32_t ph) -> bool {
        if (issued >= r_end - r_begin) return true;
        if (!mbar_wait(smem_u32(&empty[slot]), ph, &abort_flag, a.err, a.wait_limit_ns)) return false;
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");   // generic reads before the copy's writes
        issue(slot, r_begin + issued);
        ++issued;
        return true;
    };
    // two rows (two slots) per iteration: their rotations are independent work
    const int nrows = r_end - r_begin;
    for (int i = 0; i < nrows; i += 2) {
        const bool two = i + 1 < nrows;
        const int s0 = i % ROPE_RING, s1 = (i + 1) % ROPE_RING;   // ROPE_RING is even
        const uint32_t ph0 = (uint32_t)(i / ROPE_RING) & 1u, ph1 = (uint32_t)((i + 1) / ROPE_RING) & 1u;
        // warp-uniform verdicts, so that a warp leaves the loop whole
        bool got = mbar_wait(smem_u32(&full[s0]), ph0, &abort_flag, a.err, a.wait_limit_ns);
        if (got && two) got = mbar_wait(smem_u32(&full[s1]), ph1, &abort_flag, a.err, a.wait_limit_ns);
        if (!__all_sync(0xffffffffu, got)) break;
        __nv_bfloat16 *py0 = py;
        advance();
        __nv_bfloat16 *py1 = py;
        if (two) advance();
        if (valid) {
            const uint4 v0 = ring[s0][threadIdx.x];
            const uint4 v1 = two ? ring[s1][threadIdx.x] : v0;
            const uint32_t w0[4] = {v0.x, v0.y, v0.z, v0.w}, w1[4] = {v1.x, v1.y, v1.z, v1.w};
            const uint4 o0 = rope_rotate(w0, k, exact);
            const uint4 o1 = rope_rotate(w1, k, exact);
            __stcs(reinterpret_cast<uint4 *>(py0), o0);
            if (two) __stcs(reinterpret_cast<uint4 *>(py1), o1);
        }
        __syncwarp();
        if ((threadIdx.x & 31) == 0) {
            mbar_arrive(smem_u32(&empty[s0]));
            if (two) mbar_arrive(smem_u32(&empty[s1]));
        }
        bool stop = false;
        if (threadIdx.x == 0) stop = !refill(s0, ph0) || (two && !refill(s1, ph1));
        if (__any_sync(0xffffffffu, stop)) break;
    }
    if (threadIdx.x == 0 && abort_flag) {
        // let the copies still in flight land before the CTA exits
        volatile int never = 0;
        for (int j = 0; j < ROPE_RING; ++j) {
            const int n_use = (issued - j + ROPE_RING - 1) / ROPE_RING;   // fills of slot j
            if (j < issued && n_use > 0)
                mbar_wait(smem_u32(&full[j]), (uint32_t)(n_use - 1) & 1u, &never, nullptr, 200000000ull);
        }
    }
}

// float32 (and any layout): fp64 arithmetic, one thread per (position, pair).
__global__ void rope_f32_kernel(const RopeArgs a) {
    const int half = a.d / 2;
    const long long n = (long long)a.T * half;
    for (long long e = (long long)blockIdx.x * blockDim.x + threadIdx.x; e < n;
         e += (long long)gridDim.x * blockDim.x) {
        const int t = (int)(e / half), c = (int)(e % half);
        const double m = (a.positions ? (double)a.positions[t] : (double)t) * a.pos_scale;
        double sn, cs;
        sincos(m * a.th.th[c], &sn, &cs);
        for (int ti = 0; ti < a.n; ++ti) {
            const float *xb = static_cast<const float *>(a.x[ti]);
            float *yb = static_cast<float *>(a.y[ti]);
            for (int b = 0; b < a.B; ++b) {
                for (int h = 0; h < a.H; ++h) {
                    const float *px = xb + b * a.sB[ti] + h * a.sH[ti] + (long long)t * a.sT[ti] + 2 * c;
                    const double x0 = px[0], x1 = px[1];
                    const double y0 = __dsub_rn(__dmul_rn(x0, cs), __dmul_rn(x1, sn));
                    const double y1 = __dadd_rn(__dmul_rn(x0, sn), __dmul_rn(x1, cs));
                    float *py = yb + (((long long)b * a.H + h) * a.T + t) * a.d + 2 * c;
                    py[0] = __double2float_rn(y0);
                    py[1] = __double2float_rn(y1);
                }
            }
        }
    }
}

// bfloat16 with a head dimension that is not a multiple of 8: fp64, per pair.
__global__ void rope_bf16_pair_kernel(const RopeArgs a) {
    const int half = a.d / 2;
    const long long n = (long long)a.T * half;
    for (long long e = (long long)blockIdx.x * blockDim.x + threadIdx.x; e < n;
         e += (long long)gridDim.x * blockDim.x) {
        const int t = (int)(e / half), c = (int)(e % half);
        const double m = (a.positions ? (double)a.positions[t] : (double)t) * a.pos_scale;
        double sn, cs;
        sincos(m * a.th.th[c], &sn, &cs);
        for (int ti = 0; ti < a.n; ++ti) {
            const __nv_bfloat16 *xb = static_cast<const __nv_bfloat16 *>(a.x[ti]);
            __nv_bfloat16 *yb = static_cast<__nv_bfloat16 *>(a.y[ti]);
            for (int b = 0; b < a.B; ++b) {
                for (int h = 0; h < a.H; ++h) {
                    const __nv_bfloat16 *px = xb + b * a.sB[ti] + h * a.sH[ti] + (long long)t * a.sT[ti] + 2 * c;
                    const double x0 = __bfloat162float(px[0]), x1 = __bfloat162float(px[1]);
                    const double y0 = __dsub_rn(__dmul_rn(x0, cs), __dmul_rn(x1, sn));
                    const double y1 = __dadd_rn(__dmul_rn(x0, sn), __dmul_rn(x1, cs));
                    __nv_bfloat16 *py = yb + (((long long)b * a.H + h) * a.T + t) * a.d + 2 * c;
                    py[0] = round_bf16_from_f64(y0);
                    py[1] = round_bf16_from_f64(y1);
                }
            }
        }
    }
}

// Waits on an mbarrier nothing completes; the bounded wait gives up and
// records a timeout.
__global__ void wait_timeout_kernel(unsigned *err, unsigned long long limit_ns) {
    __shared__ __align__(8) uint64_t barrier_word;
    __shared__ int abort_flag;
    const uint32_t bar = smem_u32(&barrier_word);
    if (threadIdx.x == 0) {
        abort_flag = 0;
        mbar_init(bar, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    if (threadIdx.x == 0) mbar_wait(bar, 0, &abort_flag, err, limit_ns);
    __syncthreads();
}

// ---------------------------------------------------------------------------
// shared host helpers
// ---------------------------------------------------------------------------

// Stream-ordered scratch: caller's buffer, or cudaMallocAsync'd and freed on
// the stream when the call is done.
struct Scratch {
    void *ptr = nullptr;
    bool owned = false;
    cudaStream_t s = nullptr;
    int acquire(void *ws, size_t ws_bytes, size_t need, cudaStream_t stream) {
        s = stream;
        if (need == 0) return BA_OK;
        if (ws) {
            if (reinterpret_cast<uintptr_t>(ws) & 255) return BA_ERR_ARG;
            if (ws_bytes < need) return BA_ERR_WORKSPACE;
            ptr = ws;
            return BA_OK;
        }
        if (cudaMallocAsync(&ptr, need, stream) != cudaSuccess) return BA_ERR_CUDA;
        owned = true;
        return BA_OK;
    }
    ~Scratch() {
        if (owned && ptr) cudaFreeAsync(ptr, s);
    }
};

int run_tile_classes(const Geom &g, int8_t *cls, cudaStream_t s) {
    if (g.n_qtiles == 0 || g.n_ktiles == 0 || g.B == 0) return BA_OK;
    if (g.n_qtiles > 65535 || g.B > 65535) return BA_ERR_SHAPE;
    dim3 grid(g.n_ktiles, g.n_qtiles, g.B);
    tile_class_kernel<<<grid, TILE, 0, s>>>(g, cls);
    return cudaGetLastError() == cudaSuccess ? BA_OK : BA_ERR_CUDA;
}

// Rotate one or two (B, H, T, d) tensors (x2 / y2 may be null) into contiguous outputs.
int launch_rope(const ba_tensor &x, const ba_tensor *x2, int B, int H, int T, int d, int dtype,
                const int32_t *pos, float base, float pos_scale, void *y, void *y2, cudaStream_t s) {
    RopeArgs a;
    std::memset(&a, 0, sizeof a);
    for (int c = 0; c < d / 2; ++c) a.th.th[c] = std::pow((double)base, -(double)(2 * c) / (double)d);
    a.n = x2 ? 2 : 1;
    const ba_tensor *xs[2] = {&x, x2};
    void *ys[2] = {y, y2};
    bool vec = dtype == BA_BF16 && d % 8 == 0;
    for (int i = 0; i < a.n; ++i) {
        a.x[i] = xs[i]->ptr;
        a.sB[i] = xs[i]->sB;
        a.sH[i] = xs[i]->sH;
        a.sT[i] = xs[i]->sT;
        a.y[i] = ys[i];
        vec = vec && reinterpret_cast<uintptr_t>(a.x[i]) % 16 == 0 && reinterpret_cast<uintptr_t>(a.y[i]) % 16 == 0 &&
              a.sT[i] % 8 == 0 && (H <= 1 || a.sH[i] % 8 == 0) && (B <= 1 || a.sB[i] % 8 == 0);
    }
    a.B = B;
    a.H = H;
    a.T = T;
    a.d = d;
    a.positions = pos;
    a.pos_scale = pos_scale > 0.f ? (double)pos_scale : 1.0;   // a float times an int32 is exact in fp64
    {
        const int dev = current_device();
        a.err = dev >= 0 ? g_err_ptr[dev] : nullptr;
        a.wait_limit_ns = kWaitLimitNs;
    }
    if ((long long)T * d == 0 || B == 0 || H == 0) return BA_OK;
    const int threads = 256;
    if (dtype == BA_BF16 && d % 8 == 0) {
        // the table of sincos_ff: cos, sin (n pi / 64) as float-float, from the first
        // quadrant by symmetry
        const long double pi = 3.14159265358979323846264338327950288L;
        for (int n = 0; n < 128; ++n) {
            const int q = n / 32, m = n % 32;   // angle = q pi/2 + m pi/64
            long double c = cosl(pi * m / 64), sv = sinl(pi * m / 64);
            if (m == 0) {
                c = 1;
                sv = 0;
            }
            for (int i = 0; i < q; ++i) {   // rotate by pi/2: (c, s) -> (-s, c)
                const long double t = c;
                c = -sv;
                sv = t;
            }
            const float ch = (float)c, sh = (float)sv;
            a.tab[n] = make_float4(ch, (float)(c - ch), sh, (float)(sv - sh));
        }
        const int per_cta = 2048 / d;                       // positions per CTA
        const long long gx = ((long long)T + per_cta - 1) / per_cta;
        const long long rows = (long long)a.n * B * H;
        const int dev = current_device();
        const long long want = 8LL * (dev >= 0 && g_num_sms[dev] > 0 ? g_num_sms[dev] : 152);
        long long gy = (want + gx - 1) / gx;                // split the rows when positions are few
        if (gy > rows) gy = rows;
        if (gy > 65535) gy = 65535;
        if (gy < 1) gy = 1;
        if (gx > 0x7fffffffLL) return BA_ERR_SHAPE;
        const dim3 grid((unsigned)gx, (unsigned)gy);
        bool rows_contiguous = vec;
        for (int i = 0; i < a.n; ++i) rows_contiguous = rows_contiguous && a.sT[i] == d;
        if (rows_contiguous) {
            const int ring_bytes = ROPE_RING * 256 * 16;
            if (cudaFuncSetAttribute(rope_bf16_bulk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, ring_bytes) !=
                cudaSuccess)
                return BA_ERR_CUDA;
            rope_bf16_bulk_kernel<<<grid, threads, ring_bytes, s>>>(a);
        }
        else if (vec)
            rope_bf16_kernel<true><<<grid, threads, 0, s>>>(a);
        else
            rope_bf16_kernel<false><<<grid, threads, 0, s>>>(a);
        return cudaGetLastError() == cudaSuccess ? BA_OK : BA_ERR_CUDA;
    }
    const long long per = d / 2;
    long long blocks = ((long long)T * per + threads - 1) / threads;
    if (blocks > 1 << 20) blocks = 1 << 20;
    if (dtype == BA_F32)
        rope_f32_kernel<<<(unsigned)blocks, threads, 0, s>>>(a);
    else
        rope_bf16_pair_kernel<<<(unsigned)blocks, threads, 0, s>>>(a);
    return cudaGetLastError() == cudaSuccess ? BA_OK : BA_ERR_CUDA;
}

// Launch the attention kernel that matches dtype and d.
int run_attention(AttnArgs &a, int dev, int nrows_q, int nrows_k, cudaStream_t s) {
    if (!tc_supported(a.dtype, a.g.d) || nrows_k == 0 || nrows_q == 0) return launch_attn_simt(a, s);
    int rc = get_encoder();
    if (rc) return rc;
    TmaMaps m;
    std::memset(&m, 0, sizeof m);
    const int B = a.g.B, H = a.g.H, d = a.g.d;
    // Full tiles of a bf16 output with nothing to merge are written by TMA stores
    // (boxes of 32 rows, one per softmax warp); out is (B, H, rows, d) contiguous.
    const long long osT = d, osH = a.rows * (long long)d, osB = osH * H;
    a.tma_out = a.out_dtype == BA_BF16 && a.acc_o == nullptr && reinterpret_cast<uintptr_t>(a.out) % 16 == 0;
    if (a.g.striped) {
        const int P = a.g.P;
        if ((rc = encode_map_striped(&m.q, a.q, d, P, nrows_q, H, B, a.qsT, a.qsH, a.qsB))) return rc;
        if ((rc = encode_map_striped(&m.k, a.k, d, P, nrows_k, H, B, a.ksT, a.ksH, a.ksB))) return rc;
        if ((rc = encode_map_striped(&m.v, a.v, d, P, nrows_k, H, B, a.vsT, a.vsH, a.vsB))) return rc;
        if (a.tma_out && encode_map_striped(&m.o, a.out, d, P, a.rows, H, B, osT, osH, osB, 32)) a.tma_out = 0;
        return launch_attn_tc(a, m, g_num_sms[dev], s);
    }
    if ((rc = encode_map(&m.q, a.q, d, nrows_q, H, B, a.qsT, a.qsH, a.qsB))) return rc;
    if ((rc = encode_map(&m.k, a.k, d, nrows_k, H, B, a.ksT, a.ksH, a.ksB))) return rc;
    if ((rc = encode_map(&m.v, a.v, d, nrows_k, H, B, a.vsT, a.vsH, a.vsB))) return rc;
    if (a.tma_out && encode_map(&m.o, a.out, d, a.rows, H, B, osT, osH, osB, 32)) a.tma_out = 0;
    return launch_attn_tc(a, m, g_num_sms[dev], s);
}

int check_tensor(const ba_tensor &t) { return t.ptr ? BA_OK : BA_ERR_ARG; }

}  // namespace

// ===========================================================================
// C ABI
// ===========================================================================

extern "C" {

const char *ba_strerror(int code) {
    switch (code) {
        case BA_OK: return "ok";
        case BA_ERR_ARG: return "invalid argument";
        case BA_ERR_SHAPE: return "unsupported shape";
        case BA_ERR_CUDA: return "CUDA error";
        case BA_ERR_TIMEOUT: return "device wait timed out";
        case BA_ERR_UNSUPPORTED: return "unsupported combination";
        case BA_ERR_WORKSPACE: return "workspace too small";
        case BA_ERR_NOALLOC_LIMIT: return "tile-class map larger than the fixed no-allocation scratch";
        default: return "unknown error";
    }
}

int ba_pair_schedule(int B, int H, int T, int P, int partition, int causal, int num_sms, int32_t *items,
                     int64_t capacity) {
    if (B < 0 || H < 0 || T < 0 || P < 1 || num_sms < 1 || capacity < 0) return BA_ERR_ARG;
    if (partition != BA_PART_CONTIGUOUS && partition != BA_PART_ZIGZAG && partition != BA_PART_STRIPED)
        return BA_ERR_ARG;
    const int NC = partition == BA_PART_ZIGZAG ? 2 * P : P;
    if (T % NC) return BA_ERR_SHAPE;
    if ((long long)B * H == 0 || T == 0) return 0;
    // the geometry ring_attn_fwd builds for a fused launch without masks (d = 128, bf16)
    Geom g;
    std::memset(&g, 0, sizeof g);
    g.B = B;
    g.H = H;
    g.d = 128;
    g.ring = 1;
    g.striped = partition == BA_PART_STRIPED;
    g.T = T;
    g.P = P;
    g.zigzag = partition == BA_PART_ZIGZAG;
    g.NC = NC;
    g.CL = T / NC;
    g.nqt_pc = g.nkt_pc = ceil_div(g.CL, TILE);
    g.n_qtiles = g.n_ktiles = NC * g.nqt_pc;
    g.heads_per_group = heads_per_group(B, H, T, 128, BA_BF16);
    g.causal = causal != 0;
    g.s_begin = 0;
    g.s_end = P;
    const long long n = (long long)n_pairs(g) * B * H;
    if (n > 0x7fffffffLL) return BA_ERR_SHAPE;
    g.n_items = (int)n;
    g.tail_levels = pair_tail_levels(g, num_sms);
    const int heavy_items = (n_pairs(g) - g.tail_levels) * B * H;
    for (long long w = 0; items && w < n && w < capacity; ++w) {
        const QPair p = g.striped ? work_pair<true>(g, (int)w) : work_pair<false>(g, (int)w);
        int32_t *o = items + 8 * w;
        o[0] = p.q0.b;
        o[1] = p.q0.h;
        o[2] = p.q0.row0;
        o[3] = p.q0.len;
        o[4] = p.q1.row0;
        o[5] = p.q1.len;
        o[6] = g.striped ? pair_count<true>(g, p) : pair_count<false>(g, p);
        o[7] = w < heavy_items ? 0 : 1;
    }
    return (int)n;
}

int ba_index_maps(int T, int P, int partition, int32_t *tok_of, int32_t *schedule) {
    if (T < 0 || P < 1) return BA_ERR_ARG;
    if (partition != BA_PART_CONTIGUOUS && partition != BA_PART_ZIGZAG && partition != BA_PART_STRIPED)
        return BA_ERR_ARG;
    const int NC = partition == BA_PART_ZIGZAG ? 2 * P : P;
    if (T % NC) return BA_ERR_SHAPE;
    const int CL = T / NC, per = T / P;
    if (tok_of) {
        for (int r = 0; r < P; ++r) {
            // chunks of rank r in its local order
            const int c0 = r, c1 = 2 * P - 1 - r;
            for (int t = 0; t < per; ++t) {
                int tok;
                if (partition == BA_PART_CONTIGUOUS)
                    tok = r * CL + t;
                else if (partition == BA_PART_STRIPED)
                    tok = t * P + r;
                else
                    tok = t < CL ? c0 * CL + t : c1 * CL + (t - CL);
                tok_of[(long long)r * per + t] = tok;
            }
        }
    }
    if (schedule) {
        for (int r = 0; r < P; ++r)
            for (int s = 0; s < P; ++s) schedule[r * P + s] = ((r - s) % P + P) % P;
    }
    return BA_OK;
}

int ba_sync_status(ba_stream_t stream) {
    const int dev = current_device();
    if (dev < 0) return BA_ERR_CUDA;
    int rc = device_setup(dev);
    if (rc) return rc;
    if (cudaStreamSynchronize(stream) != cudaSuccess) return BA_ERR_CUDA;
    unsigned w = 0;
    if (cudaMemcpy(&w, g_err_ptr[dev], sizeof w, cudaMemcpyDeviceToHost) != cudaSuccess) return BA_ERR_CUDA;
    if (w) {
        const unsigned zero = 0;
        if (cudaMemcpy(g_err_ptr[dev], &zero, sizeof zero, cudaMemcpyHostToDevice) != cudaSuccess)
            return BA_ERR_CUDA;
        return BA_ERR_TIMEOUT;
    }
    return BA_OK;
}

int ba_debug_wait_timeout(int64_t timeout_ns, ba_stream_t stream) {
    const int dev = current_device();
    if (dev < 0) return BA_ERR_CUDA;
    int rc = device_setup(dev);
    if (rc) return rc;
    if (timeout_ns < 0) return BA_ERR_ARG;
    if (timeout_ns > 2000000000LL) timeout_ns = 2000000000LL;
    wait_timeout_kernel<<<1, 32, 0, stream>>>(g_err_ptr[dev], (unsigned long long)timeout_ns);
    return cudaGetLastError() == cudaSuccess ? BA_OK : BA_ERR_CUDA;
}

int attn_merge(float *out_a, float *lse_a, const float *out_b, const float *lse_b, int64_t rows, int d,
               ba_stream_t stream) {
    if (!out_a || !lse_a || !out_b || !lse_b || rows < 0 || d < 1) return BA_ERR_ARG;
    if (rows == 0) return BA_OK;
    const int dev = current_device();
    if (dev < 0) return BA_ERR_CUDA;
    int rc = device_setup(dev);
    if (rc) return rc;
    long long blocks = (rows + 7) / 8;
    const long long cap = (long long)g_num_sms[dev] * 8;   // eight resident 256-thread CTAs per SM
    if (blocks > cap) blocks = cap;
    const bool vec = (d & 3) == 0 && d <= 128 && (reinterpret_cast<uintptr_t>(out_a) & 15) == 0 &&
                     (reinterpret_cast<uintptr_t>(out_b) & 15) == 0;
    if (vec)
        merge_vec_kernel<<<(unsigned)blocks, 256, 0, stream>>>(reinterpret_cast<float4 *>(out_a), lse_a,
                                                                reinterpret_cast<const float4 *>(out_b), lse_b,
                                                                rows, d / 4);
    else
        merge_kernel<<<(unsigned)blocks, 256, 0, stream>>>(out_a, lse_a, out_b, lse_b, rows, d);
    return cudaGetLastError() == cudaSuccess ? BA_OK : BA_ERR_CUDA;
}

int rope_apply(ba_tensor x, ba_tensor x2, int B, int H, int T, int d, int dtype, const int32_t *positions,
               float base, float pos_scale, void *y, void *y2, ba_stream_t stream) {
    if (B < 0 || H < 0 || T < 0 || d < 2 || (d & 1) || d > 128 || !valid_dtype(dtype) || !(base > 0.f))
        return BA_ERR_ARG;
    if (pos_scale < 0.f || !(pos_scale == pos_scale)) return BA_ERR_ARG;
    const bool two = x2.ptr != nullptr || y2 != nullptr;
    if ((long long)B * H * T > 0 && (!x.ptr || !y || (two && (!x2.ptr || !y2)))) return BA_ERR_ARG;
    const int dev = current_device();
    if (dev < 0) return BA_ERR_CUDA;
    int rc = device_setup(dev);
    if (rc) return rc;
    return launch_rope(x, two ? &x2 : nullptr, B, H, T, d, dtype, positions, base, pos_scale, y,
                       two ? y2 : nullptr, stream);
}

int ba_tile_classes(int B, int Lq, int Lk, int64_t q_off, int64_t k_off, const uint8_t *key_padding_mask,
                    int64_t kpm_ld, const uint8_t *attn_mask, int64_t am_ld, int causal, int8_t *classes,
                    ba_stream_t stream) {
    if (B < 0 || Lq < 0 || Lk < 0 || q_off < 0 || k_off < 0 || !classes) return BA_ERR_ARG;
    const int dev = current_device();
    if (dev < 0) return BA_ERR_CUDA;
    int rc = device_setup(dev);
    if (rc) return rc;
    Geom g;
    std::memset(&g, 0, sizeof g);
    g.B = B;
    g.H = 1;
    g.Lq = Lq;
    g.Lk = Lk;
    g.q_off = q_off;
    g.k_off = k_off;
    g.nqt_pc = g.n_qtiles = ceil_div(Lq, TILE);
    g.nkt_pc = g.n_ktiles = ceil_div(Lk, TILE);
    g.causal = causal != 0;
    g.kpm = key_padding_mask;
    g.kpm_ld = kpm_ld;
    g.am = attn_mask;
    g.am_ld = am_ld;
    return run_tile_classes(g, classes, stream);
}

size_t attn_block_fwd_workspace_size(int B, int Lq, int Lk, int has_masks) {
    if (B < 0 || Lq < 0 || Lk < 0) return 0;
    size_t bytes = sched_bytes(1);
    if (has_masks) bytes += align256((size_t)B * ceil_div(Lq, TILE) * ceil_div(Lk, TILE));
    return bytes;
}

int attn_block_fwd(ba_tensor q, ba_tensor k, ba_tensor v, int B, int H, int Lq, int Lk, int d, int dtype,
                   int64_t q_off, int64_t k_off, const uint8_t *key_padding_mask, int64_t kpm_ld,
                   const uint8_t *attn_mask, int64_t am_ld, int causal, float scale, void *out, int out_dtype,
                   float *lse, int accumulate, void *workspace, size_t workspace_bytes, ba_stream_t stream) {
    if (B < 0 || H < 0 || Lq < 0 || Lk < 0 || q_off < 0 || k_off < 0 || !valid_dtype(dtype)) return BA_ERR_ARG;
    const bool rows_exist = (long long)B * H * Lq > 0;
    if (rows_exist && (check_tensor(q) || !out || !lse)) return BA_ERR_ARG;
    if (rows_exist && Lk > 0 && (check_tensor(k) || check_tensor(v))) return BA_ERR_ARG;
    if (!valid_d(d)) return BA_ERR_SHAPE;
    if (out_dtype != BA_F32 && out_dtype != dtype) return BA_ERR_ARG;
    if (accumulate && out_dtype != BA_F32) return BA_ERR_ARG;
    if ((key_padding_mask && kpm_ld < k_off + Lk) || (attn_mask && am_ld < k_off + Lk)) return BA_ERR_ARG;
    if (B == 0 || H == 0 || Lq == 0) return BA_OK;
    const int dev = current_device();
    if (dev < 0) return BA_ERR_CUDA;
    int rc = device_setup(dev);
    if (rc) return rc;
    const bool tc = tc_supported(dtype, d) && Lk > 0;
    q = fix_unit_strides(q, B, H, Lq, d);
    k = fix_unit_strides(k, B, H, Lk, d);
    v = fix_unit_strides(v, B, H, Lk, d);
    if (tc && (!tma_ok(q, B, H) || !tma_ok(k, B, H) || !tma_ok(v, B, H))) return BA_ERR_ARG;

    AttnArgs a;
    std::memset(&a, 0, sizeof a);
    Geom &g = a.g;
    g.B = B;
    g.H = H;
    g.d = d;
    g.Lq = Lq;
    g.Lk = Lk;
    g.q_off = q_off;
    g.k_off = k_off;
    g.nqt_pc = g.n_qtiles = ceil_div(Lq, TILE);
    g.nkt_pc = g.n_ktiles = ceil_div(Lk, TILE);
    g.heads_per_group = heads_per_group(B, H, Lk, d, dtype);
    g.n_items = g.n_qtiles * B * H;
    g.causal = causal != 0;
    g.kpm = key_padding_mask;
    g.kpm_ld = kpm_ld;
    g.am = attn_mask;
    g.am_ld = am_ld;

    const bool masks = key_padding_mask || attn_mask;
    Scratch ws;
    if ((rc = ws.acquire(workspace, workspace_bytes, attn_block_fwd_workspace_size(B, Lq, Lk, masks), stream)))
        return rc;
    uint8_t *wp = static_cast<uint8_t *>(ws.ptr);
    a.sched = reinterpret_cast<unsigned *>(wp);
    if ((rc = zero_sched(wp, 1, stream))) return rc;
    wp += sched_bytes(1);
    if (masks) {
        g.cls = reinterpret_cast<const int8_t *>(wp);
        if ((rc = run_tile_classes(g, reinterpret_cast<int8_t *>(wp), stream))) return rc;
    }
    a.q = q.ptr;
    a.k = k.ptr;
    a.v = v.ptr;
    a.qsB = q.sB; a.qsH = q.sH; a.qsT = q.sT;
    a.ksB = k.sB; a.ksH = k.sH; a.ksT = k.sT;
    a.vsB = v.sB; a.vsH = v.sH; a.vsT = v.sT;
    a.dtype = dtype;
    const float sc = scale > 0.f ? scale : (float)(1.0 / std::sqrt((double)d));
    a.scale_log2 = sc * LOG2E;
    a.out = out;
    a.out_dtype = out_dtype;
    a.lse = lse;
    a.rows = Lq;
    a.acc_o = accumulate ? static_cast<const float *>(out) : nullptr;
    a.acc_lse = accumulate ? lse : nullptr;
    a.err = g_err_ptr[dev];
    a.wait_limit_ns = kWaitLimitNs;
    return run_attention(a, dev, Lq, Lk, stream);
}

size_t ring_attn_fwd_workspace_size(int B, int H, int T, int d, int dtype, int P, int partition, int mode,
                                    int has_masks, int rope, int out_dtype) {
    if (P < 1 || T < 0) return 0;
    const int NC = partition == BA_PART_ZIGZAG ? 2 * P : P;
    if (NC == 0 || T % NC) return 0;
    const int CL = T / NC;
    const size_t nt = (size_t)NC * ceil_div(CL, TILE);
    size_t bytes = sched_bytes(mode == BA_MODE_STEPWISE ? P : 1);
    if (has_masks) bytes += align256((size_t)B * nt * nt);
    const size_t tensor = (size_t)B * H * T * d;
    if (rope) bytes += 2 * align256(tensor * elem_size(dtype));
    if (mode == BA_MODE_STEPWISE && P > 1 && out_dtype != BA_F32) bytes += align256(tensor * 4);
    return bytes;
}

int ring_attn_fwd(ba_tensor q, ba_tensor k, ba_tensor v, int B, int H, int T, int d, int dtype, int P, int partition,
                  int mode, const uint8_t *key_padding_mask, int64_t kpm_ld, const uint8_t *attn_mask, int64_t am_ld,
                  int causal, float scale, int rope, float rope_base, void *out, int out_dtype, float *lse,
                  int32_t *index_maps_out, void *workspace, size_t workspace_bytes, ba_stream_t stream) {
    if (B < 0 || H < 0 || T < 0 || P < 1 || !valid_dtype(dtype)) return BA_ERR_ARG;
    if ((long long)B * H * T > 0 && (check_tensor(q) || check_tensor(k) || check_tensor(v) || !out || !lse))
        return BA_ERR_ARG;
    if (partition != BA_PART_CONTIGUOUS && partition != BA_PART_ZIGZAG && partition != BA_PART_STRIPED)
        return BA_ERR_ARG;
    // striped: masks are indexed by token, and a rank's tokens are not a range of them
    if (partition == BA_PART_STRIPED && (key_padding_mask || attn_mask)) return BA_ERR_UNSUPPORTED;
    if (mode != BA_MODE_STEPWISE && mode != BA_MODE_FUSED) return BA_ERR_ARG;
    if (out_dtype != BA_F32 && out_dtype != dtype) return BA_ERR_ARG;
    if (!valid_d(d)) return BA_ERR_SHAPE;
    if (rope && ((d & 1) || !(rope_base > 0.f))) return BA_ERR_ARG;
    if ((key_padding_mask && kpm_ld < T) || (attn_mask && am_ld < T)) return BA_ERR_ARG;
    const int NC = partition == BA_PART_ZIGZAG ? 2 * P : P;
    if (T % NC) return BA_ERR_SHAPE;
    if (index_maps_out) {
        int rc = ba_index_maps(T, P, partition, index_maps_out, index_maps_out + T);
        if (rc) return rc;
    }
    if (B == 0 || H == 0 || T == 0) return BA_OK;
    const int dev = current_device();
    if (dev < 0) return BA_ERR_CUDA;
    int rc = device_setup(dev);
    if (rc) return rc;
    const bool tc = tc_supported(dtype, d);
    q = fix_unit_strides(q, B, H, T, d);
    k = fix_unit_strides(k, B, H, T, d);
    v = fix_unit_strides(v, B, H, T, d);
    if (tc && !tma_ok(v, B, H)) return BA_ERR_ARG;
    if (tc && !rope && (!tma_ok(q, B, H) || !tma_ok(k, B, H))) return BA_ERR_ARG;

    const bool masks = key_padding_mask || attn_mask;
    Scratch ws;
    const size_t need = ring_attn_fwd_workspace_size(B, H, T, d, dtype, P, partition, mode, masks, rope, out_dtype);
    if ((rc = ws.acquire(workspace, workspace_bytes, need, stream))) return rc;
    uint8_t *wp = static_cast<uint8_t *>(ws.ptr);
    const int launches = mode == BA_MODE_STEPWISE ? P : 1;
    unsigned *sched = reinterpret_cast<unsigned *>(wp);
    if ((rc = zero_sched(wp, launches, stream))) return rc;
    wp += sched_bytes(launches);

    AttnArgs a;
    std::memset(&a, 0, sizeof a);
    Geom &g = a.g;
    g.B = B;
    g.H = H;
    g.d = d;
    g.ring = 1;
    g.striped = partition == BA_PART_STRIPED;
    g.T = T;
    g.P = P;
    g.zigzag = partition == BA_PART_ZIGZAG;
    g.NC = NC;
    g.CL = T / NC;
    g.nqt_pc = g.nkt_pc = ceil_div(g.CL, TILE);
    g.n_qtiles = g.n_ktiles = NC * g.nqt_pc;
    g.heads_per_group = heads_per_group(B, H, T, d, dtype);
    g.n_items = g.n_qtiles * B * H;
    g.causal = causal != 0;
    g.kpm = key_padding_mask;
    g.kpm_ld = kpm_ld;
    g.am = attn_mask;
    g.am_ld = am_ld;
    g.s_begin = 0;
    g.s_end = P;

    if (masks) {
        g.cls = reinterpret_cast<const int8_t *>(wp);
        if ((rc = run_tile_classes(g, reinterpret_cast<int8_t *>(wp), stream))) return rc;
        wp += align256((size_t)B * g.n_qtiles * g.n_ktiles);
    }
    const size_t tensor = (size_t)B * H * T * d;
    if (rope) {
        void *qr = wp;
        wp += align256(tensor * elem_size(dtype));
        void *kr = wp;
        wp += align256(tensor * elem_size(dtype));
        if ((rc = launch_rope(q, &k, B, H, T, d, dtype, nullptr, rope_base, 1.f, qr, kr, stream))) return rc;
        const long long sT = d, sH = (long long)T * d, sB = (long long)H * T * d;
        q = ba_tensor{qr, sB, sH, sT};
        k = ba_tensor{kr, sB, sH, sT};
    }
    a.q = q.ptr;
    a.k = k.ptr;
    a.v = v.ptr;
    a.qsB = q.sB; a.qsH = q.sH; a.qsT = q.sT;
    a.ksB = k.sB; a.ksH = k.sH; a.ksT = k.sT;
    a.vsB = v.sB; a.vsH = v.sH; a.vsT = v.sT;
    a.dtype = dtype;
    const float sc = scale > 0.f ? scale : (float)(1.0 / std::sqrt((double)d));
    a.scale_log2 = sc * LOG2E;
    a.lse = lse;
    a.rows = T;
    a.err = g_err_ptr[dev];
    a.wait_limit_ns = kWaitLimitNs;

    if (mode == BA_MODE_FUSED || P == 1) {
        a.sched = sched;
        a.out = out;
        a.out_dtype = out_dtype;
        return run_attention(a, dev, T, T, stream);
    }
    // Step-wise: one launch per ring step, each folding the step's block into
    // the fp32 (out, lse) accumulator; the last step writes the final dtype.
    float *acc = out_dtype == BA_F32 ? static_cast<float *>(out) : reinterpret_cast<float *>(wp);
    for (int s = 0; s < P; ++s) {
        g.s_begin = s;
        g.s_end = s + 1;
        a.sched = sched + s;
        a.acc_o = s > 0 ? acc : nullptr;
        a.acc_lse = s > 0 ? lse : nullptr;
        const bool last = s == P - 1;
        a.out = last ? out : acc;
        a.out_dtype = last ? out_dtype : BA_F32;
        if ((rc = run_attention(a, dev, T, T, stream))) return rc;
    }
    return BA_OK;
}

// ---------------------------------------------------------------------------
// Backward
// ---------------------------------------------------------------------------

namespace {

ba::TensorRef tref(const ba_tensor &t) { return ba::TensorRef{t.ptr, t.sB, t.sH, t.sT}; }

// The tensor-core backward for bf16 with d in {64, 128} when every operand can
// be read by TMA; the CUDA-core kernels otherwise.
int run_bwd(ba::BwdArgs &a, ba_tensor q, ba_tensor k, ba_tensor v, ba_tensor dout, long long q_rows,
            long long k_rows, int dev, cudaStream_t s) {
    a.err = g_err_ptr[dev];
    a.wait_limit_ns = kWaitLimitNs;
    auto al16 = [](const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; };   // float4 epilogues
    if (ba::bwd_tc_supported(a.dtype, a.d) && q_rows > 0 && k_rows > 0 && tma_ok(q, a.B, a.H) &&
        tma_ok(k, a.B, a.H) && tma_ok(v, a.B, a.H) && tma_ok(dout, a.B, a.H) && al16(a.dq) && al16(a.dk) &&
        al16(a.dv)) {
        int rc = get_encoder();
        if (rc) return rc;
        ba::BwdMaps m;
        if ((rc = encode_map(&m.q, q.ptr, a.d, q_rows, a.H, a.B, q.sT, q.sH, q.sB))) return rc;
        if ((rc = encode_map(&m.dout, dout.ptr, a.d, q_rows, a.H, a.B, dout.sT, dout.sH, dout.sB))) return rc;
        if ((rc = encode_map(&m.k, k.ptr, a.d, k_rows, a.H, a.B, k.sT, k.sH, k.sB))) return rc;
        if ((rc = encode_map(&m.v, v.ptr, a.d, k_rows, a.H, a.B, v.sT, v.sH, v.sB))) return rc;
        return ba::launch_attn_bwd_tc(a, m, g_num_sms[dev], s);
    }
    return ba::launch_attn_bwd(a, g_num_sms[dev], s);
}

int check_bwd_common(ba_tensor q, ba_tensor k, ba_tensor v, ba_tensor out, ba_tensor dout, const float *lse,
                     int B, int H, int Lq, int Lk, int d, int dtype, const float *dq, const float *dk,
                     const float *dv) {
    if (B < 0 || H < 0 || Lq < 0 || Lk < 0 || !valid_dtype(dtype)) return BA_ERR_ARG;
    if (!valid_d(d)) return BA_ERR_SHAPE;
    const bool qrows = (long long)B * H * Lq > 0, krows = (long long)B * H * Lk > 0;
    if (qrows && (check_tensor(q) || check_tensor(out) || check_tensor(dout) || !lse || !dq)) return BA_ERR_ARG;
    if (krows && (check_tensor(k) || check_tensor(v) || !dk || !dv)) return BA_ERR_ARG;
    return BA_OK;
}

}  // namespace

// 256 bytes of item counters for the persistent tensor-core kernels, then D.
size_t attn_block_bwd_workspace_size(int B, int H, int Lq) {
    if (B < 0 || H < 0 || Lq < 0) return 0;
    return 256 + align256((size_t)4 * (size_t)B * (size_t)H * (size_t)Lq);
}

int attn_block_bwd(ba_tensor q, ba_tensor k, ba_tensor v, ba_tensor out, ba_tensor dout, const float *lse, int B,
                   int H, int Lq, int Lk, int d, int dtype, int64_t q_off, int64_t k_off,
                   const uint8_t *key_padding_mask, int64_t kpm_ld, const uint8_t *attn_mask, int64_t am_ld,
                   int causal, float scale, float *dq, float *dk, float *dv, int accumulate, void *workspace,
                   size_t workspace_bytes, ba_stream_t stream) {
    int rc = check_bwd_common(q, k, v, out, dout, lse, B, H, Lq, Lk, d, dtype, dq, dk, dv);
    if (rc) return rc;
    if (q_off < 0 || k_off < 0) return BA_ERR_ARG;
    if ((key_padding_mask && kpm_ld < k_off + Lk) || (attn_mask && am_ld < k_off + Lk)) return BA_ERR_ARG;
    if (B == 0 || H == 0 || (Lq == 0 && Lk == 0)) return BA_OK;
    const int dev = current_device();
    if (dev < 0) return BA_ERR_CUDA;
    if ((rc = device_setup(dev))) return rc;
    Scratch ws;
    if ((rc = ws.acquire(workspace, workspace_bytes, attn_block_bwd_workspace_size(B, H, Lq), stream))) return rc;
    ba::BwdArgs a;
    std::memset(&a, 0, sizeof a);
    a.B = B;
    a.H = H;
    a.d = d;
    a.dtype = dtype;
    a.ring = 0;
    a.Lq = Lq;
    a.Lk = Lk;
    a.q_off = q_off;
    a.k_off = k_off;
    a.causal = causal != 0;
    a.kpm = key_padding_mask;
    a.kpm_ld = kpm_ld;
    a.am = attn_mask;
    a.am_ld = am_ld;
    q = fix_unit_strides(q, B, H, Lq, d);
    out = fix_unit_strides(out, B, H, Lq, d);
    dout = fix_unit_strides(dout, B, H, Lq, d);
    k = fix_unit_strides(k, B, H, Lk, d);
    v = fix_unit_strides(v, B, H, Lk, d);
    a.q = tref(q);
    a.out = tref(out);
    a.dout = tref(dout);
    a.k = tref(k);
    a.v = tref(v);
    a.lse = lse;
    a.sched = static_cast<unsigned *>(ws.ptr);
    a.D = reinterpret_cast<float *>(static_cast<uint8_t *>(ws.ptr) + 256);
    a.heads_per_group = heads_per_group(B, H, Lq > Lk ? Lq : Lk, d, dtype);
    a.scale = scale > 0.f ? scale : (float)(1.0 / std::sqrt((double)d));
    a.dq = dq;
    a.dk = dk;
    a.dv = dv;
    a.accumulate = accumulate != 0;
    return run_bwd(a, q, k, v, dout, Lq, Lk, dev, stream);
}

size_t ring_attn_bwd_workspace_size(int B, int H, int T) { return attn_block_bwd_workspace_size(B, H, T); }

int ring_attn_bwd(ba_tensor q, ba_tensor k, ba_tensor v, ba_tensor out, ba_tensor dout, const float *lse, int B,
                  int H, int T, int d, int dtype, int P, int partition, int mode, const uint8_t *key_padding_mask,
                  int64_t kpm_ld, const uint8_t *attn_mask, int64_t am_ld, int causal, float scale, float *dq,
                  float *dk, float *dv, void *workspace, size_t workspace_bytes, ba_stream_t stream) {
    int rc = check_bwd_common(q, k, v, out, dout, lse, B, H, T, T, d, dtype, dq, dk, dv);
    if (rc) return rc;
    if (P < 1) return BA_ERR_ARG;
    if (partition == BA_PART_STRIPED) return BA_ERR_UNSUPPORTED;   // tokens of a rank are not a position range
    if (partition != BA_PART_CONTIGUOUS && partition != BA_PART_ZIGZAG) return BA_ERR_ARG;
    if (mode != BA_MODE_STEPWISE && mode != BA_MODE_FUSED) return BA_ERR_ARG;
    if ((key_padding_mask && kpm_ld < T) || (attn_mask && am_ld < T)) return BA_ERR_ARG;
    const int NC = partition == BA_PART_ZIGZAG ? 2 * P : P;
    if (T % NC) return BA_ERR_SHAPE;
    if (B == 0 || H == 0 || T == 0) return BA_OK;
    const int dev = current_device();
    if (dev < 0) return BA_ERR_CUDA;
    if ((rc = device_setup(dev))) return rc;
    Scratch ws;
    if ((rc = ws.acquire(workspace, workspace_bytes, ring_attn_bwd_workspace_size(B, H, T), stream))) return rc;
    ba::BwdArgs a;
    std::memset(&a, 0, sizeof a);
    a.B = B;
    a.H = H;
    a.d = d;
    a.dtype = dtype;
    a.ring = 1;
    a.T = T;
    a.P = P;
    a.zigzag = partition == BA_PART_ZIGZAG;
    a.NC = NC;
    a.CL = T / NC;
    a.causal = causal != 0;
    a.kpm = key_padding_mask;
    a.kpm_ld = kpm_ld;
    a.am = attn_mask;
    a.am_ld = am_ld;
    q = fix_unit_strides(q, B, H, T, d);
    out = fix_unit_strides(out, B, H, T, d);
    dout = fix_unit_strides(dout, B, H, T, d);
    k = fix_unit_strides(k, B, H, T, d);
    v = fix_unit_strides(v, B, H, T, d);
    a.q = tref(q);
    a.out = tref(out);
    a.dout = tref(dout);
    a.k = tref(k);
    a.v = tref(v);
    a.lse = lse;
    a.sched = static_cast<unsigned *>(ws.ptr);
    a.D = reinterpret_cast<float *>(static_cast<uint8_t *>(ws.ptr) + 256);
    a.heads_per_group = heads_per_group(B, H, T, d, dtype);
    a.scale = scale > 0.f ? scale : (float)(1.0 / std::sqrt((double)d));
    a.dq = dq;
    a.dk = dk;
    a.dv = dv;
    if (mode == BA_MODE_FUSED || P == 1) {
        a.s_begin = 0;
        a.s_end = P;
        a.accumulate = 0;
        return run_bwd(a, q, k, v, dout, T, T, dev, stream);
    }
    // Step-wise, as on the page: step s pairs the queries of rank r with the
    // K/V block of rank (r - s) mod P; dQ accumulates in place and dK / dV
    // accumulate at their block's rows (the page rotates them with K and V).
    for (int s = 0; s < P; ++s) {
        a.s_begin = s;
        a.s_end = s + 1;
        a.accumulate = s > 0;
        if ((rc = run_bwd(a, q, k, v, dout, T, T, dev, stream))) return rc;
    }
    return BA_OK;
}

// ---------------------------------------------------------------------------
// Ulysses
// ---------------------------------------------------------------------------

int ulysses_all_to_all(const void *src, void *dst, int P, int H, int B, int T, int d, int elem_bytes, int direction,
                       ba_stream_t stream) {
    if (P < 1 || H < 0 || B < 0 || T < 0 || d < 1) return BA_ERR_ARG;
    if (elem_bytes != 1 && elem_bytes != 2 && elem_bytes != 4 && elem_bytes != 8) return BA_ERR_ARG;
    if (direction != BA_A2A_TOKEN_TO_HEAD && direction != BA_A2A_HEAD_TO_TOKEN) return BA_ERR_ARG;
    if (H % P || T % P) return BA_ERR_SHAPE;
    if ((long long)H * B * T == 0) return BA_OK;
    if (!src || !dst) return BA_ERR_ARG;
    const int dev = current_device();
    if (dev < 0) return BA_ERR_CUDA;
    int rc = device_setup(dev);
    if (rc) return rc;
    ba::UlyssesArgs u;
    u.P = P;
    u.H = H;
    u.B = B;
    u.Tl = T / P;
    u.elem_bytes = elem_bytes;
    u.row_bytes = (long long)d * elem_bytes;
    // head side: the stacked (P, H/P, B, T, d) array, i.e. (B, H, T, d) with sH = B T d
    u.sT = d;
    u.sB = (long long)T * d;
    u.sH = (long long)B * T * d;
    u.to_head = direction == BA_A2A_TOKEN_TO_HEAD;
    u.tok = u.to_head ? const_cast<void *>(src) : dst;
    u.head = u.to_head ? dst : const_cast<void *>(src);
    return ba::launch_ulysses_a2a(u, g_num_sms[dev], stream);
}

size_t ulysses_attn_fwd_workspace_size(int P, int H, int B, int T, int d, int dtype, int has_masks) {
    if (P < 1 || H < 0 || B < 0 || T < 0 || d < 1 || !valid_dtype(dtype)) return 0;
    const size_t tensor = (size_t)B * H * T * d * elem_size(dtype);
    return 4 * align256(tensor) + align256((size_t)B * H * T * 4) +
           ring_attn_fwd_workspace_size(B, H, T, d, dtype, 1, BA_PART_CONTIGUOUS, BA_MODE_FUSED, has_masks, 0, dtype);
}

int ulysses_attn_fwd(const void *q_tok, const void *k_tok, const void *v_tok, int P, int H, int B, int T, int d,
                     int dtype, const uint8_t *key_padding_mask, int64_t kpm_ld, const uint8_t *attn_mask,
                     int64_t am_ld, int causal, float scale, void *out_tok, float *lse_tok, void *workspace,
                     size_t workspace_bytes, ba_stream_t stream) {
    if (P < 1 || H < 0 || B < 0 || T < 0 || !valid_dtype(dtype)) return BA_ERR_ARG;
    if (!valid_d(d)) return BA_ERR_SHAPE;
    if (H % P || T % P) return BA_ERR_SHAPE;
    if ((key_padding_mask && kpm_ld < T) || (attn_mask && am_ld < T)) return BA_ERR_ARG;
    if ((long long)B * H * T == 0) return BA_OK;
    if (!q_tok || !k_tok || !v_tok || !out_tok || !lse_tok) return BA_ERR_ARG;
    const int dev = current_device();
    if (dev < 0) return BA_ERR_CUDA;
    int rc = device_setup(dev);
    if (rc) return rc;
    const bool masks = key_padding_mask || attn_mask;
    Scratch ws;
    const size_t need = ulysses_attn_fwd_workspace_size(P, H, B, T, d, dtype, masks);
    if ((rc = ws.acquire(workspace, workspace_bytes, need, stream))) return rc;
    uint8_t *wp = static_cast<uint8_t *>(ws.ptr);
    const size_t eb = elem_size(dtype), tensor = (size_t)B * H * T * d * eb;
    void *qh = wp, *kh = wp + align256(tensor), *vh = wp + 2 * align256(tensor), *oh = wp + 3 * align256(tensor);
    float *lh = reinterpret_cast<float *>(wp + 4 * align256(tensor));
    uint8_t *aws = wp + 4 * align256(tensor) + align256((size_t)B * H * T * 4);
    const size_t aws_bytes = need - (size_t)(aws - wp);
    // 1. first all-to-all: token-split -> head-split (P, H/P, B, T, d) for q, k, v
    const void *srcs[3] = {q_tok, k_tok, v_tok};
    void *dsts[3] = {qh, kh, vh};
    for (int i = 0; i < 3; ++i)
        if ((rc = ulysses_all_to_all(srcs[i], dsts[i], P, H, B, T, d, (int)eb, BA_A2A_TOKEN_TO_HEAD, stream)))
            return rc;
    // 2. attention over the full context of every head: the head-split array is a
    //    (B, H, T, d) view with sB = T d, sH = B T d (one launch for all ranks)
    const int64_t sB = (int64_t)T * d, sH = (int64_t)B * T * d, sT = d;
    rc = ring_attn_fwd(ba_tensor{qh, sB, sH, sT}, ba_tensor{kh, sB, sH, sT}, ba_tensor{vh, sB, sH, sT}, B, H, T, d,
                       dtype, 1, BA_PART_CONTIGUOUS, BA_MODE_FUSED, key_padding_mask, kpm_ld, attn_mask, am_ld,
                       causal, scale, 0, 0.f, oh, dtype, lh, nullptr, aws, aws_bytes, stream);
    if (rc) return rc;
    // 3. reverse all-to-all of out (B, H, T, d) and lse (B, H, T) into token-split arrays
    ba::UlyssesArgs u;
    u.P = P;
    u.H = H;
    u.B = B;
    u.Tl = T / P;
    u.to_head = 0;
    u.tok = out_tok;
    u.head = oh;
    u.elem_bytes = (int)eb;
    u.row_bytes = (long long)d * eb;
    u.sT = d;
    u.sH = (long long)T * d;
    u.sB = (long long)H * T * d;
    if ((rc = ba::launch_ulysses_a2a(u, g_num_sms[dev], stream))) return rc;
    u.tok = lse_tok;
    u.head = lh;
    u.elem_bytes = 4;
    u.row_bytes = 4;
    u.sT = 1;
    u.sH = T;
    u.sB = (long long)H * T;
    return ba::launch_ulysses_a2a(u, g_num_sms[dev], stream);
}

// ---------------------------------------------------------------------------
// Decode with a split KV cache
// ---------------------------------------------------------------------------

namespace {

int decode_splits(int B, int H, int S, int num_splits, int num_sms) {
    if (num_splits > 0) return num_splits < S ? num_splits : (S > 0 ? S : 1);
    const long long bh = (long long)B * H > 0 ? (long long)B * H : 1;
    long long n = (4LL * num_sms + bh - 1) / bh;   // about four CTAs per SM
    const long long cap = (S + 63) / 64 > 0 ? (S + 63) / 64 : 1;   // at least 64 keys per split
    if (n > cap) n = cap;
    if (n < 1) n = 1;
    return (int)n;
}

bool rows16(const void *p, long long sB, long long sH, long long sT, size_t eb) {
    return (reinterpret_cast<uintptr_t>(p) & 15) == 0 && (sB * (long long)eb) % 16 == 0 &&
           (sH * (long long)eb) % 16 == 0 && (sT * (long long)eb) % 16 == 0;
}

}  // namespace

size_t attn_decode_workspace_size(int B, int H, int S, int d, int num_splits) {
    if (B < 0 || H < 0 || S < 0 || d < 1) return 0;
    const int n = decode_splits(B, H, S, num_splits, 152);
    const int dev = current_device();
    const int n_dev = dev >= 0 && g_num_sms[dev] > 0 ? decode_splits(B, H, S, num_splits, g_num_sms[dev]) : n;
    const int nn = n > n_dev ? n : n_dev;
    return align256((size_t)B * H * nn * d * 4) + align256((size_t)B * H * nn * 4);
}

int attn_decode_fwd(ba_tensor q, ba_tensor k, ba_tensor v, int B, int H, int S, int d, int dtype,
                    const int32_t *lengths, int num_splits, float scale, void *out, int out_dtype, float *lse,
                    void *workspace, size_t workspace_bytes, ba_stream_t stream) {
    if (B < 0 || H < 0 || S < 0 || num_splits < 0 || !valid_dtype(dtype)) return BA_ERR_ARG;
    if (!valid_d(d)) return BA_ERR_SHAPE;
    if (out_dtype != BA_F32 && out_dtype != dtype) return BA_ERR_ARG;
    if ((long long)B * H == 0) return BA_OK;
    if (check_tensor(q) || !out || !lse || (S > 0 && (check_tensor(k) || check_tensor(v)))) return BA_ERR_ARG;
    const size_t eb = elem_size(dtype);
    q = fix_unit_strides(q, B, H, 1, d);
    k = fix_unit_strides(k, B, H, S, d);
    v = fix_unit_strides(v, B, H, S, d);
    if (!rows16(q.ptr, q.sB, q.sH, d, eb) || (S > 0 && (!rows16(k.ptr, k.sB, k.sH, k.sT, eb) ||
                                                         !rows16(v.ptr, v.sB, v.sH, v.sT, eb))))
        return BA_ERR_ARG;   // the kernel reads 16-byte vectors of every row
    const int dev = current_device();
    if (dev < 0) return BA_ERR_CUDA;
    int rc = device_setup(dev);
    if (rc) return rc;
    ba::DecodeArgs a;
    std::memset(&a, 0, sizeof a);
    a.B = B;
    a.H = H;
    a.S = S;
    a.d = d;
    a.dtype = dtype;
    a.q = q.ptr;
    a.qsB = q.sB;
    a.qsH = q.sH;
    a.k = k.ptr;
    a.ksB = k.sB;
    a.ksH = k.sH;
    a.ksT = k.sT;
    a.v = v.ptr;
    a.vsB = v.sB;
    a.vsH = v.sH;
    a.vsT = v.sT;
    a.lengths = lengths;
    a.scale = scale > 0.f ? scale : (float)(1.0 / std::sqrt((double)d));
    a.n_splits = decode_splits(B, H, S, num_splits, g_num_sms[dev]);
    a.split_len = S > 0 ? (S + a.n_splits - 1) / a.n_splits : 1;
    Scratch ws;
    const size_t need = align256((size_t)B * H * a.n_splits * d * 4) + align256((size_t)B * H * a.n_splits * 4);
    if ((rc = ws.acquire(workspace, workspace_bytes, need, stream))) return rc;
    a.part_o = static_cast<float *>(ws.ptr);
    a.part_lse = reinterpret_cast<float *>(static_cast<uint8_t *>(ws.ptr) +
                                           align256((size_t)B * H * a.n_splits * d * 4));
    a.out = out;
    a.out_dtype = out_dtype;
    a.lse = lse;
    return ba::launch_decode(a, stream);
}

// Same work as attn_block_fwd, with the tile-class map in the library's fixed
// device array instead of a workspace: nothing is allocated.
int attn_block_fwd_noalloc(ba_tensor q, ba_tensor k, ba_tensor v, int B, int H, int Lq, int Lk, int d, int dtype,
                           int64_t q_off, int64_t k_off, const uint8_t *key_padding_mask, int64_t kpm_ld,
                           const uint8_t *attn_mask, int64_t am_ld, int causal, float scale, void *out,
                           int out_dtype, float *lse, int accumulate, ba_stream_t stream) {
    if (B < 0 || H < 0 || Lq < 0 || Lk < 0 || q_off < 0 || k_off < 0 || !valid_dtype(dtype)) return BA_ERR_ARG;
    const bool rows_exist = (long long)B * H * Lq > 0;
    if (rows_exist && (check_tensor(q) || !out || !lse)) return BA_ERR_ARG;
    if (rows_exist && Lk > 0 && (check_tensor(k) || check_tensor(v))) return BA_ERR_ARG;
    if (!valid_d(d)) return BA_ERR_SHAPE;
    if (out_dtype != BA_F32 && out_dtype != dtype) return BA_ERR_ARG;
    if (accumulate && out_dtype != BA_F32) return BA_ERR_ARG;
    if ((key_padding_mask && kpm_ld < k_off + Lk) || (attn_mask && am_ld < k_off + Lk)) return BA_ERR_ARG;
    const bool masks = key_padding_mask || attn_mask;
    const size_t class_bytes = (size_t)B * ceil_div(Lq, TILE) * ceil_div(Lk, TILE);
    if (masks && class_bytes > (size_t)BA_NOALLOC_MAX_CLASS_BYTES) return BA_ERR_NOALLOC_LIMIT;
    if (B == 0 || H == 0 || Lq == 0) return BA_OK;
    const int dev = current_device();
    if (dev < 0) return BA_ERR_CUDA;
    int rc = device_setup(dev);
    if (rc) return rc;
    int8_t *classes = nullptr;
    if (masks && (rc = noalloc_scratch(dev, &classes))) return rc;
    const bool tc = tc_supported(dtype, d) && Lk > 0;
    q = fix_unit_strides(q, B, H, Lq, d);
    k = fix_unit_strides(k, B, H, Lk, d);
    v = fix_unit_strides(v, B, H, Lk, d);
    if (tc && (!tma_ok(q, B, H) || !tma_ok(k, B, H) || !tma_ok(v, B, H))) return BA_ERR_ARG;

    AttnArgs a;
    std::memset(&a, 0, sizeof a);
    Geom &g = a.g;
    g.B = B;
    g.H = H;
    g.d = d;
    g.Lq = Lq;
    g.Lk = Lk;
    g.q_off = q_off;
    g.k_off = k_off;
    g.nqt_pc = g.n_qtiles = ceil_div(Lq, TILE);
    g.nkt_pc = g.n_ktiles = ceil_div(Lk, TILE);
    g.heads_per_group = heads_per_group(B, H, Lk, d, dtype);
    g.n_items = g.n_qtiles * B * H;
    g.causal = causal != 0;
    g.kpm = key_padding_mask;
    g.kpm_ld = kpm_ld;
    g.am = attn_mask;
    g.am_ld = am_ld;
    if (masks) {
        // every entry the attention kernel reads is written here first
        g.cls = classes;
        if ((rc = run_tile_classes(g, classes, stream))) return rc;
    }
    a.q = q.ptr;
    a.k = k.ptr;
    a.v = v.ptr;
    a.qsB = q.sB; a.qsH = q.sH; a.qsT = q.sT;
    a.ksB = k.sB; a.ksH = k.sH; a.ksT = k.sT;
    a.vsB = v.sB; a.vsH = v.sH; a.vsT = v.sT;
    a.dtype = dtype;
    const float sc = scale > 0.f ? scale : (float)(1.0 / std::sqrt((double)d));
    a.scale_log2 = sc * LOG2E;
    a.out = out;
    a.out_dtype = out_dtype;
    a.lse = lse;
    a.rows = Lq;
    a.acc_o = accumulate ? static_cast<const float *>(out) : nullptr;
    a.acc_lse = accumulate ? lse : nullptr;
    a.err = g_err_ptr[dev];
    a.wait_limit_ns = kWaitLimitNs;
    return run_attention(a, dev, Lq, Lk, stream);
}

}  // extern "C"
