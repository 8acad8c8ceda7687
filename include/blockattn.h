/*
 * blockattn.h -- C ABI of libblockattn.so: blockwise multi-head scaled-dot-
 * product attention with the Ring-Attention online-softmax (LSE) merge,
 * hand-written for NVIDIA GB300 (sm_103a).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Tensor arguments are DEVICE pointers owned by the caller.  The library
 *    never frees caller memory and never keeps a pointer after a call returns.
 *  - Q, K, V use the layout (B, H, T, d): `ba_tensor` carries the base pointer
 *    and element strides of the B, H and T axes; the d axis is contiguous.
 *    Outputs are contiguous: out (B, H, L, d), lse (B, H, L).
 *  - Masks are uint8 with 1 = EXCLUDED, indexed at GLOBAL token positions:
 *      key_padding_mask[b * kpm_ld + key_pos]      (B rows, >= total keys)
 *      attn_mask[query_pos * am_ld + key_pos]      (>= total queries rows)
 *    The library receives only the pointer and the row stride, so it cannot
 *    see how many rows a mask has: the caller must pass a key-padding mask
 *    with at least B rows and an attn_mask with a row for every global query
 *    position of the call (q_off + Lq rows for a block, T for a ring), each
 *    row covering every global key position the call reads.  A shorter mask
 *    is read past its end.  (The Python binding checks the shapes.)
 *    A pair (i, j) takes part iff it is not excluded by causality (j > i,
 *    when causal != 0), by the key padding of its batch item, or by attn_mask:
 *    the exclusions are OR-combined ("PyTorch MultiheadAttention", item #2 of
 *    ai.engineer "Transformers and Attention"; causal = diagonal + lower
 *    triangle, item #24 "PyTorch scaled_dot_product_attention").
 *  - lse is the NATURAL-log log-sum-exp of the scaled scores of a row,
 *    LSE_i = log sum_j exp(s_ij), s_ij = scale * q_i . k_j ("Ring Attention"
 *    and "Improving numerical stability" on brunomaga "Sequence/context
 *    parallelism").  A row with no visible key gets out = 0 and lse = -inf.
 *  - Every call is asynchronous on `stream` and returns BA_OK or a negative
 *    error code (ba_strerror names it).  Argument errors are detected on the
 *    host before anything is launched.  A device-side wait that exceeds its
 *    time limit is reported by ba_sync_status() as BA_ERR_TIMEOUT; kernels
 *    never trap.
 *  - Scratch: entry points that need scratch take (workspace, workspace_bytes).
 *    workspace == NULL makes the library allocate it stream-ordered
 *    (cudaMallocAsync) and free it on the same stream before returning;
 *    the *_workspace_size() queries give the bytes a caller should pass.
 *    A caller's workspace must start on a 256-byte boundary (BA_ERR_ARG
 *    otherwise) and is used only by this call's launches on `stream`.  Its
 *    first 256 bytes (more for many ring steps) hold the zeroed item
 *    counters from which the attention kernel's CTAs claim work, heaviest
 *    query tiles first, so that every SM stays busy to the end.
 *  - bf16 inputs with d in {64, 128} run on the tcgen05 tensor-core kernel
 *    (TMA-staged tiles, TMEM accumulators); fp32 inputs, and bf16 with other d
 *    in {16, 32}, run on a CUDA-core kernel that keeps fp32 arithmetic.
 */
#ifndef BLOCKATTN_H
#define BLOCKATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *ba_stream_t; /* a cudaStream_t; NULL = legacy default stream */

enum {
    BA_OK = 0,
    BA_ERR_ARG = -1,         /* bad pointer, size, flag or alignment */
    BA_ERR_SHAPE = -2,       /* sizes not supported (d, T vs P, ...) */
    BA_ERR_CUDA = -3,        /* a CUDA runtime/driver call failed */
    BA_ERR_TIMEOUT = -4,     /* a bounded device-side wait expired */
    BA_ERR_UNSUPPORTED = -5, /* combination not implemented */
    BA_ERR_WORKSPACE = -6,   /* workspace smaller than required */
    BA_ERR_NOALLOC_LIMIT = -7 /* larger than the fixed scratch of attn_block_fwd_noalloc */
};

enum { BA_F32 = 0, BA_BF16 = 1 };
/* Token partitions over P ranks: contiguous blocks, zigzag (2P chunks, rank r
 * holds chunks r and 2P-1-r), and striped (token t on rank t mod P, rank r
 * holding r, r+P, r+2P, ... in that order; brunomaga "When to use Ulysses and
 * Ring attention" names Striped Attention).  ring_attn_fwd takes striped
 * partitions without masks (masks are indexed by token, and a striped rank's
 * tokens are not a range: BA_ERR_UNSUPPORTED with a mask); ring_attn_bwd
 * returns BA_ERR_UNSUPPORTED for them. */
enum { BA_PART_CONTIGUOUS = 0, BA_PART_ZIGZAG = 1, BA_PART_STRIPED = 2 };
enum { BA_MODE_STEPWISE = 0, BA_MODE_FUSED = 1 };
enum { BA_TILE_EMPTY = 0, BA_TILE_FULL = 1, BA_TILE_PARTIAL = 2 };

/* Strided (B, H, T, d) tensor: element (b, h, t, c) is at
 * ptr + b*sB + h*sH + t*sT + c (in elements of the tensor's dtype). */
typedef struct {
    const void *ptr;
    int64_t sB, sH, sT;
} ba_tensor;

/*
 * attn_block_fwd -- one block of attention: the queries of q against the keys
 * and values of k, v, with per-row LSE.  This is the per-step kernel of the
 * ring loop (brunomaga "Implementation": each step computes the block output
 * and the per-row LSE of the local queries against the current K/V block).
 *
 *  q: (B, H, Lq, d); local row i is global query position q_off + i.
 *  k, v: (B, H, Lk, d); local key j is global key position k_off + j.
 *  dtype: BA_F32 or BA_BF16 (q, k, v share it).  d: 16, 32, 64 or 128.
 *  key_padding_mask / attn_mask: NULL or as in the conventions above; their
 *    lds are in elements and must cover the global positions used.
 *  causal: exclude key positions greater than the query position (global).
 *  scale: > 0, or <= 0 for 1/sqrt(d).
 *  out: (B, H, Lq, d) contiguous, out_dtype = BA_F32 or dtype.
 *  lse: (B, H, Lq) fp32 contiguous.
 *  accumulate: 0 = overwrite (out, lse); 1 = (out, lse) already hold a partial
 *    attention of the same rows over other keys (fp32 out required; out = 0,
 *    lse = -inf means "nothing yet") and the block is merged into it with the
 *    LSE rule: L = log(e^La + e^Lb), O = e^(La-L) Oa + e^(Lb-L) Ob.
 *  workspace: see conventions; attn_block_fwd_workspace_size() bytes.
 * Errors: BA_ERR_ARG (NULL q/k/v/out/lse, negative sizes, accumulate with a
 * non-fp32 out, misaligned TMA strides), BA_ERR_SHAPE (unsupported d).
 */
size_t attn_block_fwd_workspace_size(int B, int Lq, int Lk, int has_masks);
int attn_block_fwd(ba_tensor q, ba_tensor k, ba_tensor v,
                   int B, int H, int Lq, int Lk, int d, int dtype,
                   int64_t q_off, int64_t k_off,
                   const uint8_t *key_padding_mask, int64_t kpm_ld,
                   const uint8_t *attn_mask, int64_t am_ld,
                   int causal, float scale,
                   void *out, int out_dtype, float *lse, int accumulate,
                   void *workspace, size_t workspace_bytes, ba_stream_t stream);

/*
 * attn_merge -- a <- merge(a, b) for two partial attentions of the same rows
 * over disjoint key sets: with M = max(La, Lb), L = M + log(e^(La-M) + e^(Lb-M))
 * and O = e^(La-L) Oa + e^(Lb-L) Ob; a side with lse = -inf contributes nothing.
 * This is accumulate_out_and_lse of brunomaga "Implementation"; the outputs of
 * blocks are never added or averaged (llm-systems "CP: Split Long Contexts
 * Across GPUs", "Circulate K/V blocks with Ring").
 *  out_a (rows, d), lse_a (rows): fp32, updated in place.
 *  out_b (rows, d), lse_b (rows): fp32, read only.  d >= 1.
 */
int attn_merge(float *out_a, float *lse_a, const float *out_b, const float *lse_b,
               int64_t rows, int d, ba_stream_t stream);

/*
 * ring_attn_fwd -- Ring Attention over P context-parallel ranks emulated on
 * one GPU (llm-systems "Circulate K/V blocks with Ring"; brunomaga
 * "Distributed algorithm").  The T tokens are split into P ranks
 * (partition = BA_PART_CONTIGUOUS: P equal time blocks; BA_PART_ZIGZAG: 2P
 * equal chunks, rank r owning chunks r and 2P-1-r, llm-systems "Balance the
 * workload in causal attention"; BA_PART_STRIPED: rank r owns the tokens
 * r + P u, and under causal masking its block against the K/V of rank c is a
 * lower triangle over local indices, with the diagonal when c <= r and
 * without it when c > r).  Every rank keeps its queries resident; at
 * ring step s = 0..P-1 it folds in the K/V block of rank (r - s) mod P (local
 * block first, then the previous rank's, ...).  Positions and masks stay the
 * global ones.  There is no inter-GPU traffic: each rank's "received" block is
 * the partition already resident in this GPU's memory.
 *
 *  q, k, v: (B, H, T, d), dtype as for attn_block_fwd.
 *  mode: BA_MODE_FUSED = one persistent launch, each query tile walks the
 *    whole ring in-kernel with the running (max, denominator, weighted sum);
 *    BA_MODE_STEPWISE = one launch per ring step, each merging its block
 *    into an fp32 (out, lse) accumulator (the page's loop, step by step).
 *  rope != 0: Q and K are first rotated (see rope_apply, positions 0..T-1,
 *    base rope_base) into workspace copies; the caller's q, k are unchanged.
 *  out: (B, H, T, d) in global token order, out_dtype BA_F32 or dtype.
 *  lse: (B, H, T) fp32.
 *  index_maps_out: NULL, or host int32[T + P*P] receiving the partition
 *    (rank-major token ids, P x T/P) followed by the schedule src[r][s].
 * Errors: BA_ERR_SHAPE when T is not divisible by P (contiguous, striped) or
 * 2P (zigzag), or d is unsupported; BA_ERR_UNSUPPORTED for a striped
 * partition with a mask; BA_ERR_ARG as for attn_block_fwd.
 */
size_t ring_attn_fwd_workspace_size(int B, int H, int T, int d, int dtype, int P,
                                    int partition, int mode, int has_masks, int rope,
                                    int out_dtype);
int ring_attn_fwd(ba_tensor q, ba_tensor k, ba_tensor v,
                  int B, int H, int T, int d, int dtype,
                  int P, int partition, int mode,
                  const uint8_t *key_padding_mask, int64_t kpm_ld,
                  const uint8_t *attn_mask, int64_t am_ld,
                  int causal, float scale, int rope, float rope_base,
                  void *out, int out_dtype, float *lse, int32_t *index_maps_out,
                  void *workspace, size_t workspace_bytes, ba_stream_t stream);

/*
 * attn_block_bwd -- gradients of one attention block ("Sequence/context
 * parallelism" (brunomaga), section "Ring Attention", backward pass): with
 * p_ij = exp(scale q_i . k_j - lse_i) over the visible pairs and
 * D_i = dout_i . out_i,
 *   dV_j = sum_i p_ij dout_i,   ds_ij = p_ij (dout_i . v_j - D_i),
 *   dQ_i = scale sum_j ds_ij k_j,   dK_j = scale sum_i ds_ij q_i.
 * out and lse are the forward results of the WHOLE rows (all keys, not just
 * this block), as the page's per-step backward uses them; the blocks' dQ, dK,
 * dV then add up to the gradients of the full attention.
 *  q, out, dout: (B, H, Lq, d); k, v: (B, H, Lk, d); strides and dtype as
 *    for attn_block_fwd (q, k, v, out, dout share the dtype).
 *  lse: (B, H, Lq) fp32 natural log, -inf for rows that see no key.
 *  q_off, k_off, masks, causal, scale: as for attn_block_fwd.
 *  dq: (B, H, Lq, d), dk, dv: (B, H, Lk, d), fp32 contiguous, caller-owned.
 *  accumulate: 0 = overwrite dq, dk, dv; 1 = add this block's gradients.
 *  workspace: attn_block_bwd_workspace_size() bytes, 256-byte aligned, owned by
 *    the caller (or NULL: allocated and freed on the stream): the D_i vector
 *    (fp32 per row).
 * bf16 with d = 64 or 128, TMA-legal strides and 16-byte aligned dq / dk / dv
 * run on the tensor cores (tcgen05; P and dS rounded to bf16 for the
 * products, fp32 accumulation); everything else runs on the CUDA cores in fp32.
 * Errors: BA_ERR_ARG (NULL pointers for non-empty sides, negative sizes or
 * offsets, masks not covering the global positions), BA_ERR_SHAPE (d not in
 * {16, 32, 64, 128}).
 */
size_t attn_block_bwd_workspace_size(int B, int H, int Lq);
int attn_block_bwd(ba_tensor q, ba_tensor k, ba_tensor v, ba_tensor out, ba_tensor dout,
                   const float *lse, int B, int H, int Lq, int Lk, int d, int dtype,
                   int64_t q_off, int64_t k_off,
                   const uint8_t *key_padding_mask, int64_t kpm_ld,
                   const uint8_t *attn_mask, int64_t am_ld,
                   int causal, float scale,
                   float *dq, float *dk, float *dv, int accumulate,
                   void *workspace, size_t workspace_bytes, ba_stream_t stream);

/*
 * ring_attn_bwd -- the backward pass of Ring Attention over P emulated ranks
 * ("Sequence/context parallelism" (brunomaga), section "Ring Attention",
 * backward): at step s rank r pairs its queries with the K/V block of rank
 * (r - s) mod P; dQ accumulates at the queries, and dK / dV accumulate with
 * their K/V block (the page rotates them around the ring with K and V, so
 * after P steps each rank holds the gradients of its own block).  On one GPU
 * the ranks are the token ranges of the partition, so a block's dK / dV rows
 * collect the contributions of every rank's queries in place.
 *  q, k, v, out, dout: (B, H, T, d) in global token order; lse: (B, H, T).
 *  mode: BA_MODE_FUSED = every step in one launch pair; BA_MODE_STEPWISE =
 *    one launch pair per ring step, accumulating, as on the page.
 *  dq, dk, dv: (B, H, T, d) fp32 contiguous, overwritten.
 *  workspace: ring_attn_bwd_workspace_size() bytes.
 * Errors: as attn_block_bwd, plus BA_ERR_SHAPE when T is not divisible by P
 * (contiguous) or 2P (zigzag).
 */
size_t ring_attn_bwd_workspace_size(int B, int H, int T);
int ring_attn_bwd(ba_tensor q, ba_tensor k, ba_tensor v, ba_tensor out, ba_tensor dout,
                  const float *lse, int B, int H, int T, int d, int dtype,
                  int P, int partition, int mode,
                  const uint8_t *key_padding_mask, int64_t kpm_ld,
                  const uint8_t *attn_mask, int64_t am_ld,
                  int causal, float scale,
                  float *dq, float *dk, float *dv,
                  void *workspace, size_t workspace_bytes, ba_stream_t stream);

/*
 * Ulysses ("Sequence/context parallelism" (brunomaga), section "Ulysses
 * sequence parallelism"; "Change token partitions into head partitions with
 * Ulysses"): P ranks first hold token shards, an all-to-all turns them into
 * head shards holding the full context of H/P heads each, attention runs
 * unchanged per head, and a reverse all-to-all returns the output to token
 * shards.  On one GPU the ranks' buffers are stacked along a leading P axis.
 *
 * ulysses_all_to_all -- one exchange of whole d-rows (a permutation, exact):
 *  BA_A2A_TOKEN_TO_HEAD: src (P, H, B, T/P, d) -> dst (P, H/P, B, T, d), where
 *    rank r of dst holds heads [r H/P, (r+1) H/P) for tokens 0..T-1 in order;
 *  BA_A2A_HEAD_TO_TOKEN: the inverse.
 *  Both arrays contiguous, elem_bytes in {1, 2, 4, 8}, caller-owned, must not
 *  overlap.  Errors: BA_ERR_SHAPE unless P divides H and T; BA_ERR_ARG for bad
 *  sizes, direction or NULL pointers.
 */
#define BA_A2A_TOKEN_TO_HEAD 0
#define BA_A2A_HEAD_TO_TOKEN 1
int ulysses_all_to_all(const void *src, void *dst, int P, int H, int B, int T, int d,
                       int elem_bytes, int direction, ba_stream_t stream);

/*
 * ulysses_attn_fwd -- Ulysses attention over P emulated ranks: the first
 * all-to-all of q, k, v, one attention launch over every head's full context
 * (the tensor-core kernel for bf16 d in {64, 128}), and the reverse all-to-all
 * of out and lse.
 *  q_tok, k_tok, v_tok: (P, H, B, T/P, d) contiguous token shards, dtype.
 *  masks, causal, scale: as for ring_attn_fwd (global token positions).
 *  out_tok: (P, H, B, T/P, d) contiguous, dtype; lse_tok: (P, H, B, T/P) fp32.
 *  workspace: ulysses_attn_fwd_workspace_size() bytes (head-split q, k, v and
 *    out, lse, and the attention's own scratch).
 * Errors: BA_ERR_SHAPE unless P divides H and T and d is supported; BA_ERR_ARG
 * as for ring_attn_fwd.
 */
size_t ulysses_attn_fwd_workspace_size(int P, int H, int B, int T, int d, int dtype, int has_masks);
int ulysses_attn_fwd(const void *q_tok, const void *k_tok, const void *v_tok,
                     int P, int H, int B, int T, int d, int dtype,
                     const uint8_t *key_padding_mask, int64_t kpm_ld,
                     const uint8_t *attn_mask, int64_t am_ld,
                     int causal, float scale, void *out_tok, float *lse_tok,
                     void *workspace, size_t workspace_bytes, ba_stream_t stream);

/*
 * attn_decode_fwd -- decode attention: one query token per (b, h) against a KV
 * cache, split along the keys.  Decode processes one token at a time and
 * shards the KV cache rather than the input tokens ("Sequence/context
 * parallelism" (brunomaga), the note on the inference decode step); each split
 * gives a partial (O, LSE) over its keys and the partials are merged by the LSE
 * rule of attn_merge (an associative merge; here all splits at once).
 *  q: (B, H, 1, d); k_cache, v_cache: (B, H, S, d) with element strides, every
 *    row starting on a 16-byte boundary (BA_ERR_ARG otherwise).
 *  lengths: NULL, or device int32[B]: keys [0, lengths[b]) of sequence b are
 *    valid (clamped to [0, S]); a sequence of length 0 gets out = 0, lse = -inf.
 *  num_splits: 0 = chosen by the library (about four CTAs per SM, at least 64
 *    keys per split), else the number of key splits.
 *  out: (B, H, 1, d) contiguous, out_dtype BA_F32 or dtype; lse: (B, H, 1) fp32.
 *  workspace: attn_decode_workspace_size() bytes (fp32 partials).
 * Bound by HBM: every valid K and V byte is read once.
 */
size_t attn_decode_workspace_size(int B, int H, int S, int d, int num_splits);
int attn_decode_fwd(ba_tensor q, ba_tensor k_cache, ba_tensor v_cache,
                    int B, int H, int S, int d, int dtype,
                    const int32_t *lengths, int num_splits, float scale,
                    void *out, int out_dtype, float *lse,
                    void *workspace, size_t workspace_bytes, ba_stream_t stream);

/*
 * rope_apply -- rotary position embedding ("RoFormer", item #4 of ai.engineer
 * "Transformers and Attention"): split each d-vector into coordinate pairs
 * (2c, 2c+1) and rotate pair c by the angle m * base^(-2c/d), m the token
 * position: (x0, x1) -> (x0 cos - x1 sin, x0 sin + x1 cos).  The result equals
 * the rotation evaluated in fp64 and rounded once (ties to even) to the
 * tensor dtype (bf16 uses exact fp32 products of 16-bit pieces of the fp64
 * cos/sin, summed with error-free transforms).
 *  x: (B, H, T, d) strided input; y: (B, H, T, d) contiguous output of the
 *  same dtype (may not alias x).  x2 / y2: an optional second tensor of the
 *  same shape rotated by the same launch (e.g. K next to Q); pass
 *  x2.ptr = NULL and y2 = NULL for one tensor.  positions: NULL (position of
 *  row t is t) or device int32[T].  d must be even and <= 128 (else BA_ERR_ARG).
 *  pos_scale: Position Interpolation ("Extending Context Window of Large
 *  Language Models via Position Interpolation", item #59): the position index
 *  is multiplied by pos_scale (e.g. original / extended window) before the
 *  angle is formed, m' = m * pos_scale in fp64 (exact); 0 or 1 = plain RoPE,
 *  negative or NaN = BA_ERR_ARG.
 */
int rope_apply(ba_tensor x, ba_tensor x2, int B, int H, int T, int d, int dtype,
               const int32_t *positions, float base, float pos_scale, void *y, void *y2,
               ba_stream_t stream);

/*
 * ba_tile_classes -- class of each 128 x 128 tile of the combined exclusion
 * mask for the block rows [q_off, q_off+Lq) x keys [k_off, k_off+Lk), tiles
 * counted from the block origin: BA_TILE_EMPTY (no visible pair), FULL (all
 * pairs visible) or PARTIAL.  classes: device int8 (B, ceil(Lq/128),
 * ceil(Lk/128)).  The attention kernels skip EMPTY tiles and apply per-element
 * predicates on PARTIAL ones.
 */
int ba_tile_classes(int B, int Lq, int Lk, int64_t q_off, int64_t k_off,
                    const uint8_t *key_padding_mask, int64_t kpm_ld,
                    const uint8_t *attn_mask, int64_t am_ld, int causal,
                    int8_t *classes, ba_stream_t stream);

/*
 * ba_index_maps -- host, exact integers: the emulated ranks' token ownership
 * tok_of[r * (T/P) + t] (rank r's t-th local token, in its local order) and
 * the ring schedule schedule[r * P + s] = (r - s) mod P.  Same partitions and
 * order as ring_attn_fwd.  Returns BA_ERR_SHAPE for indivisible T.
 */
int ba_index_maps(int T, int P, int partition, int32_t *tok_of, int32_t *schedule);

/*
 * ba_pair_schedule -- host, exact integers: the work items of the tensor-core
 * forward kernel for a ring_attn_fwd launch without masks (causal or not) over
 * B x H heads of T tokens, P ranks, on num_sms SMs, in the order the kernel
 * deals them.  An item is a pair of adjacent 128-row query tiles of one chunk
 * (a chunk with an odd tile count ends in a one-tile pair) with the key tiles
 * its walk visits.  items (nullable): capacity rows of 8 int32, item w at
 * items[8 w ..]: b, h, first query row of tile 0, its rows, first query row of
 * tile 1, its rows (0: no second tile), key tiles visited, phase (0: grouped
 * by heads, heaviest first; 1: the lightest levels of all heads, dealt last).
 * Returns the number of items (every item is written when capacity allows),
 * or BA_ERR_SHAPE for indivisible T, BA_ERR_ARG for bad sizes.  Computed by
 * the same functions the kernel uses; for tests and inspection.
 */
int ba_pair_schedule(int B, int H, int T, int P, int partition, int causal, int num_sms,
                     int32_t *items, int64_t capacity);

/*
 * attn_block_fwd_noalloc -- attn_block_fwd for callers that cannot allocate
 * device memory.  The pages have no counterpart; this is a library-level
 * variant.  Some hosts own every device allocation themselves (for example a
 * framework that plans all buffers ahead of execution and forbids allocation
 * while it runs, or a process that works under a hard memory budget), so they
 * can neither pass a workspace nor let the library call cudaMalloc.  This
 * entry point takes the same arguments as attn_block_fwd minus the workspace
 * and performs no allocation of any kind: the one piece of scratch
 * attn_block_fwd needs -- the tile-class map built when a key-padding mask or
 * attn_mask is given, B * ceil(Lq/128) * ceil(Lk/128) bytes -- lives in a
 * fixed device array of BA_NOALLOC_MAX_CLASS_BYTES bytes inside the library,
 * present on every GPU that loads the library until the process exits.
 *  - Inputs and outputs are the caller's, exactly as for attn_block_fwd.
 *  - A call whose tile-class map would exceed BA_NOALLOC_MAX_CLASS_BYTES
 *    returns BA_ERR_NOALLOC_LIMIT before launching anything.
 *  - The first call on a device looks up the array's device address on that
 *    device (cudaGetSymbolAddress); make that first call before any stream
 *    capture.  The address is kept for the rest of the process, so a
 *    cudaDeviceReset() of that device after the first call is not supported
 *    (the reset unloads the module and the kept address would be stale; the
 *    library's timeout flag is looked up and kept the same way).
 *  - All calls on a GPU share that GPU's array, and it keeps the last call's
 *    contents.  Every entry a call reads is first written by that call, so
 *    nothing needs clearing; but calls that overlap on the same GPU (for
 *    example on two streams) race on it when they use masks: serialise them.
 */
#define BA_NOALLOC_MAX_CLASS_BYTES (1 << 20)
int attn_block_fwd_noalloc(ba_tensor q, ba_tensor k, ba_tensor v,
                           int B, int H, int Lq, int Lk, int d, int dtype,
                           int64_t q_off, int64_t k_off,
                           const uint8_t *key_padding_mask, int64_t kpm_ld,
                           const uint8_t *attn_mask, int64_t am_ld,
                           int causal, float scale,
                           void *out, int out_dtype, float *lse, int accumulate,
                           ba_stream_t stream);

/* Synchronise `stream` and report whether any kernel launched by this library
 * on the current device since the previous call gave up a bounded device wait
 * (BA_ERR_TIMEOUT), or a CUDA error occurred (BA_ERR_CUDA).  Clears the flag. */
int ba_sync_status(ba_stream_t stream);

/* Test hook for the bounded-wait path: launches one CTA that waits on an
 * mbarrier nothing will complete, giving up after `timeout_ns` nanoseconds
 * (capped at 2e9) and recording BA_ERR_TIMEOUT for ba_sync_status. */
int ba_debug_wait_timeout(int64_t timeout_ns, ba_stream_t stream);

const char *ba_strerror(int code);

#ifdef __cplusplus
}
#endif
#endif /* BLOCKATTN_H */
