// Host-side interface between the C-ABI entry points (api.cu) and the kernel
// translation units.  Not part of the public ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include "common.cuh"

namespace ba {

// Arguments of one attention launch (block or ring geometry).
struct AttnArgs {
    Geom g;
    const void *q, *k, *v;               // base pointers, dtype `dtype`
    long long qsB, qsH, qsT;             // element strides (d contiguous)
    long long ksB, ksH, ksT;
    long long vsB, vsH, vsT;
    int dtype;                           // BA_F32 / BA_BF16
    float scale_log2;                    // softmax scale * log2(e)
    void *out;                           // (B, H, rows, d) contiguous, out_dtype
    int out_dtype;
    int tma_out;                         // tensor-core kernel: full tiles stored by TMA (map `o`)
    float *lse;                          // (B, H, rows) natural-log LSE
    long long rows;                      // rows of out/lse per (b, h): Lq or T
    const float *acc_o;                  // nullable fp32 (B, H, rows, d) partial to merge with
    const float *acc_lse;                // nullable fp32 (B, H, rows)
    unsigned *err;                       // device error word
    unsigned *sched;                     // nullable zeroed item counter (dynamic scheduling); null = round-robin
    unsigned long long wait_limit_ns;    // bounded-wait limit
};

// A (B, H, rows, d) tensor with element strides, d contiguous.
struct TensorRef {
    const void *p;
    long long sB, sH, sT;
};

// Arguments of the attention backward (block or ring geometry).  Rows of
// q/out/dout and of k/v are positions - off in block mode and token positions
// in ring mode (global token order).
struct BwdArgs {
    int B, H, d, dtype;
    int ring;                            // 0: one block (Lq x Lk at q_off / k_off)
    int Lq, Lk;
    long long q_off, k_off;
    int T, P, zigzag, CL, NC, s_begin, s_end;   // ring geometry and the steps to cover
    int causal;
    const uint8_t *kpm;
    long long kpm_ld;
    const uint8_t *am;
    long long am_ld;
    TensorRef q, k, v, out, dout;
    const float *lse;                    // (B, H, Lq) natural-log LSE of the whole row
    float *D;                            // (B, H, Lq) dout . out, written by the pre-pass
    float scale;
    float *dq, *dk, *dv;                 // fp32 (B, H, L, d) contiguous
    int accumulate;                      // add into dq / dk / dv instead of overwriting
    unsigned *err;                       // device error word (tensor-core kernels)
    unsigned long long wait_limit_ns;    // bounded-wait limit (tensor-core kernels)
    unsigned *sched;                     // 2 zeroed item counters (dK/dV kernel, dQ kernel), tensor-core kernels
    int heads_per_group;                 // (b, h) pairs whose items run side by side (L2 reuse)
};

// TMA descriptors of q, k, v and dout for the tensor-core backward.
struct BwdMaps {
    CUtensorMap q, k, v, dout;
};

int launch_attn_bwd(const BwdArgs &a, int num_sms, cudaStream_t s);
int launch_bwd_pre(const BwdArgs &a, int num_sms, cudaStream_t s);
bool bwd_tc_supported(int dtype, int d);
int launch_attn_bwd_tc(const BwdArgs &a, const BwdMaps &m, int num_sms, cudaStream_t s);

// One Ulysses exchange: the token-split stacked array (P, H, B, Tl, d),
// contiguous, against a strided (B, H, T = P Tl, d) view of the head side.
struct UlyssesArgs {
    void *tok;                // token-split array
    void *head;               // head-side view base
    long long sB, sH, sT;     // head-side element strides (d contiguous)
    int P, H, B, Tl;
    long long row_bytes;      // d * elem_bytes
    int elem_bytes;
    int to_head;              // 1: token-split -> head side, 0: head side -> token-split
};

int launch_ulysses_a2a(const UlyssesArgs &a, int num_sms, cudaStream_t s);

// Decode attention of one query per (b, h) against a KV cache, in key splits.
struct DecodeArgs {
    int B, H, S, d, dtype;
    const void *q, *k, *v;               // q: (B, H, 1, d); k, v: (B, H, S, d), element strides
    long long qsB, qsH;
    long long ksB, ksH, ksT, vsB, vsH, vsT;
    const int32_t *lengths;              // (B) valid cache lengths, or nullptr = S
    float scale;
    int split_len, n_splits;
    float *part_o, *part_lse;            // (B*H, n_splits, d), (B*H, n_splits) fp32 partials
    void *out;                           // (B, H, 1, d) contiguous, out_dtype
    int out_dtype;
    float *lse;                          // (B, H, 1)
};

int launch_decode(const DecodeArgs &a, cudaStream_t s);

// TMA descriptors of Q, K, V (loads) and out (stores, boxes of 32 rows) for
// the tensor-core kernel.
struct TmaMaps {
    CUtensorMap q, k, v, o;
};

int launch_attn_simt(const AttnArgs &a, cudaStream_t s);
int launch_attn_tc(const AttnArgs &a, const TmaMaps &maps, int num_sms, cudaStream_t s);
bool tc_supported(int dtype, int d);
size_t tc_smem_bytes(int d);

}  // namespace ba
