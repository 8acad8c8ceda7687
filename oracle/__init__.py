"""ORACLE -- test infrastructure only.

A plain, slow, obviously correct CPU statement of what the blockwise / ring
attention path computes, in fp64.  Only ``tests/``, ``__graft_entry__.smoke()``
and the benchmark's CPU-baseline leg may import it; the product package never
does, and it shares no code with the CUDA library (the two meet only in the
seeded input generators of ``blockwise_attention_gb300.workloads``).

Parts and the passages they follow:

* ``attention``: fp64 scaled-dot-product attention with the causal,
  key-padding and attn_mask exclusions OR-combined, plus the per-row natural-log
  LSE ("Attention Is All You Need" #22 and #15 sec. 3.2.1, "PyTorch
  scaled_dot_product_attention" #24 and "PyTorch MultiheadAttention" #2 on the
  ai.engineer "Transformers and Attention" page; "Ring Attention" and
  "Improving numerical stability" on the brunomaga sequence-parallelism page).
  C code in ``attention.c``.
* ``rope``: rotation of coordinate pairs by positional angles ("RoFormer" #4),
  fp64, rounded once to the storage type.  C code in ``attention.c``.
* ``merge``: the LSE merge of two partial attentions over disjoint key sets
  (brunomaga "Improving numerical stability": rescale both sides to the new
  maximum; LSE property).  Never adds or averages the outputs (llm-systems
  "Circulate K/V blocks with Ring").
* ``partition``, ``schedule``, ``tile_classes``: the emulated ranks' token
  ownership (contiguous; zigzag of llm-systems "Balance the workload in causal
  attention"), the ring order (llm-systems "Circulate K/V blocks with Ring";
  brunomaga "Distributed algorithm") and the EMPTY/FULL/PARTIAL class of each
  128 x 128 tile of the combined exclusion mask.

Every function here is pinned by ``tests/test_oracle*.py`` against what the
pages and the mathematics fix (worked example, closed forms, invariants, brute
force, a library routine), never against the CUDA path.
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")
_SRC = os.path.join(_HERE, "attention.c")
_lib = None

EMPTY, FULL, PARTIAL = 0, 1, 2


def build(force: bool = False) -> str:
    """Compile the C oracle with gcc (no fused multiply-add)."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math",
                               "-shared", "-fPIC", "-pthread", _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB_PATH)
        i64, f64, vp = ctypes.c_int64, ctypes.c_double, ctypes.c_void_p
        lib.oracle_attention.restype = ctypes.c_int
        lib.oracle_attention.argtypes = [vp, vp, vp, i64, i64, i64, i64, i64, i64, i64,
                                         vp, i64, vp, i64, ctypes.c_int, f64, vp, i64, vp, vp,
                                         ctypes.c_int]
        lib.oracle_attention_bwd.restype = ctypes.c_int
        lib.oracle_attention_bwd.argtypes = [vp, vp, vp, vp, i64, i64, i64, i64, i64, i64, i64,
                                             vp, i64, vp, i64, ctypes.c_int, f64, vp, vp, vp, vp, vp,
                                             ctypes.c_int]
        lib.oracle_rope.restype = ctypes.c_int
        lib.oracle_rope.argtypes = [vp, i64, i64, i64, vp, f64, f64, ctypes.c_int, vp, vp]
        lib.oracle_round_bf16.restype = ctypes.c_float
        lib.oracle_round_bf16.argtypes = [f64]
        _lib = lib
    return _lib


def _f32(x) -> np.ndarray:
    if hasattr(x, "detach"):  # torch tensor
        x = x.detach().to("cpu").float().numpy()
    return np.ascontiguousarray(x, dtype=np.float32)


def _u8(x) -> Optional[np.ndarray]:
    if x is None:
        return None
    if hasattr(x, "detach"):
        x = x.detach().to("cpu").numpy()
    return np.ascontiguousarray(x, dtype=np.uint8)


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def default_threads() -> int:
    return max(1, len(os.sched_getaffinity(0)))


def attention(q, k, v, *, causal=False, kpm=None, am=None, scale=None, q_pos0=0, k_pos0=0,
              rows=None, nthreads=None):
    """fp64 attention of q (B,H,L,d) against k, v (B,H,S,d).

    kpm: (B, >=k_pos0+S) 1 = excluded key, indexed at GLOBAL key positions.
    am:  (>=q_pos0+L, >=k_pos0+S) 1 = excluded pair, at global positions.
    rows: optional int array of flat row ids ((b*H + h)*L + i).
    Returns (out (n, d) float64, lse (n,) float64) with n = len(rows) or B*H*L
    (reshape to (B,H,L,d) / (B,H,L) for the full case).
    """
    lib = _load()
    q, k, v = _f32(q), _f32(k), _f32(v)
    B, H, L, d = q.shape
    S = k.shape[2]
    assert k.shape == (B, H, S, d) and v.shape == (B, H, S, d)
    kpm, am = _u8(kpm), _u8(am)
    # masks are indexed at global positions: they must cover every position used
    if kpm is not None and (kpm.shape[0] < B or kpm.shape[1] < k_pos0 + S):
        raise ValueError("key_padding_mask does not cover the key positions")
    if am is not None and (am.shape[0] < q_pos0 + L or am.shape[1] < k_pos0 + S):
        raise ValueError("attn_mask does not cover the (query, key) positions")
    if rows is not None:
        rows = np.ascontiguousarray(rows, dtype=np.int64)
        n = rows.size
    else:
        n = B * H * L
    out = np.zeros((n, d), dtype=np.float64)
    lse = np.zeros((n,), dtype=np.float64)
    rc = lib.oracle_attention(_ptr(q), _ptr(k), _ptr(v), B, H, L, S, d, q_pos0, k_pos0,
                              _ptr(kpm), 0 if kpm is None else kpm.shape[1],
                              _ptr(am), 0 if am is None else am.shape[1],
                              int(bool(causal)), 0.0 if scale is None else float(scale),
                              _ptr(rows), n, _ptr(out), _ptr(lse),
                              nthreads or default_threads())
    if rc != 0:
        raise ValueError("oracle_attention: bad arguments")
    if rows is None:
        return out.reshape(B, H, L, d), lse.reshape(B, H, L)
    return out, lse


def attention_bwd(q, k, v, dout, *, causal=False, kpm=None, am=None, scale=None, q_pos0=0, k_pos0=0,
                  nthreads=None):
    """fp64 gradients of attention(q, k, v) contracted with dout (same shape as out).

    Masks and positions as for attention().  Returns (dq, dk, dv, out, lse) as
    float64 arrays of shapes (B,H,L,d), (B,H,S,d), (B,H,S,d), (B,H,L,d), (B,H,L).
    """
    lib = _load()
    q, k, v, dout = _f32(q), _f32(k), _f32(v), _f32(dout)
    B, H, L, d = q.shape
    S = k.shape[2]
    assert k.shape == (B, H, S, d) and v.shape == (B, H, S, d) and dout.shape == q.shape
    kpm, am = _u8(kpm), _u8(am)
    if kpm is not None and (kpm.shape[0] < B or kpm.shape[1] < k_pos0 + S):
        raise ValueError("key_padding_mask does not cover the key positions")
    if am is not None and (am.shape[0] < q_pos0 + L or am.shape[1] < k_pos0 + S):
        raise ValueError("attn_mask does not cover the (query, key) positions")
    dq = np.zeros((B, H, L, d), dtype=np.float64)
    dk = np.zeros((B, H, S, d), dtype=np.float64)
    dv = np.zeros((B, H, S, d), dtype=np.float64)
    out = np.zeros((B, H, L, d), dtype=np.float64)
    lse = np.zeros((B, H, L), dtype=np.float64)
    rc = lib.oracle_attention_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(dout), B, H, L, S, d, q_pos0, k_pos0,
                                  _ptr(kpm), 0 if kpm is None else kpm.shape[1],
                                  _ptr(am), 0 if am is None else am.shape[1],
                                  int(bool(causal)), 0.0 if scale is None else float(scale),
                                  _ptr(dq), _ptr(dk), _ptr(dv), _ptr(out), _ptr(lse),
                                  nthreads or default_threads())
    if rc != 0:
        raise ValueError("oracle_attention_bwd: bad arguments")
    return dq, dk, dv, out, lse


def ulysses_token_to_head(x_tok: np.ndarray, P: int) -> np.ndarray:
    """The first Ulysses all-to-all ("Sequence/context parallelism" (brunomaga),
    section "Ulysses sequence parallelism"; "Change token partitions into head
    partitions with Ulysses"): rank r holds tokens [r T/P, (r+1) T/P) of every
    head, as x_tok[r] of shape (H, B, T/P, d); afterwards rank r holds heads
    [r H/P, (r+1) H/P) for all T tokens, as (H/P, B, T, d).  Written as the
    exchange itself: rank r receives, from every rank s, s's tokens of r's heads,
    and places them at s's token range."""
    P_, H, B, Tl, d = x_tok.shape
    assert P_ == P and H % P == 0
    hl = H // P
    out = np.empty((P, hl, B, Tl * P, d), dtype=x_tok.dtype)
    for r in range(P):          # receiving rank
        for s in range(P):      # sending rank
            out[r, :, :, s * Tl:(s + 1) * Tl, :] = x_tok[s, r * hl:(r + 1) * hl, :, :, :]
    return out


def ulysses_head_to_token(x_head: np.ndarray, P: int) -> np.ndarray:
    """The second (reverse) Ulysses all-to-all: rank r holds heads
    [r H/P, (r+1) H/P) for all T tokens, as (H/P, B, T, d); afterwards rank r
    holds tokens [r T/P, (r+1) T/P) of every head, as (H, B, T/P, d)."""
    P_, hl, B, T, d = x_head.shape
    assert P_ == P and T % P == 0
    Tl = T // P
    out = np.empty((P, hl * P, B, Tl, d), dtype=x_head.dtype)
    for r in range(P):          # receiving rank (token range)
        for s in range(P):      # sending rank (head range)
            out[r, s * hl:(s + 1) * hl, :, :, :] = x_head[s, :, :, r * Tl:(r + 1) * Tl, :]
    return out


def rope(x, base=10000.0, positions=None, round_to="bf16", pos_scale=1.0):
    """Rotate coordinate pairs of x (..., T, d).  round_to: "bf16", "f32" or None
    (None returns the unrounded float64 rotation).  pos_scale multiplies the
    position index before the angle is formed (Position Interpolation)."""
    lib = _load()
    xa = _f32(x)
    shape = xa.shape
    T, d = shape[-2], shape[-1]
    BH = int(np.prod(shape[:-2])) if len(shape) > 2 else 1
    pos = None if positions is None else np.ascontiguousarray(positions, dtype=np.int64)
    if round_to is None:
        y = np.zeros(shape, dtype=np.float64)
        rc = lib.oracle_rope(_ptr(xa), BH, T, d, _ptr(pos), float(base), float(pos_scale), 0, _ptr(y), None)
    else:
        y = np.zeros(shape, dtype=np.float32)
        rc = lib.oracle_rope(_ptr(xa), BH, T, d, _ptr(pos), float(base), float(pos_scale),
                             2 if round_to == "bf16" else 1, None, _ptr(y))
    if rc != 0:
        raise ValueError("oracle_rope: bad arguments")
    return y


def round_bf16(x: float) -> float:
    """Nearest bfloat16 value of a double (ties to even)."""
    return float(_load().oracle_round_bf16(float(x)))


def merge(out_a, lse_a, out_b, lse_b):
    """LSE merge of two partial attentions of the same rows over disjoint keys.

    Both sides are rescaled to the common maximum M = max(L_a, L_b):
    L = M + log(exp(L_a - M) + exp(L_b - M)), O = exp(L_a - L) O_a + exp(L_b - L) O_b.
    A side with L = -inf (no visible key) contributes nothing.
    """
    oa = np.asarray(out_a, dtype=np.float64)
    ob = np.asarray(out_b, dtype=np.float64)
    la = np.asarray(lse_a, dtype=np.float64)
    lb = np.asarray(lse_b, dtype=np.float64)
    out = np.zeros(np.broadcast_shapes(oa.shape, ob.shape), dtype=np.float64)
    lse = np.full(np.broadcast_shapes(la.shape, lb.shape), -np.inf)
    for idx in np.ndindex(lse.shape):
        a, b = la[idx], lb[idx]
        if a == -np.inf and b == -np.inf:
            continue
        if b == -np.inf:
            out[idx], lse[idx] = oa[idx], a
            continue
        if a == -np.inf:
            out[idx], lse[idx] = ob[idx], b
            continue
        m = max(a, b)
        L = m + math.log(math.exp(a - m) + math.exp(b - m))
        out[idx] = math.exp(a - L) * oa[idx] + math.exp(b - L) * ob[idx]
        lse[idx] = L
    return out, lse


# ---------------------------------------------------------------------------
# index maps (exact integers)
# ---------------------------------------------------------------------------

def partition(T: int, P: int, kind: str) -> np.ndarray:
    """Token ids owned by each emulated rank, (P, T//P), in the rank's local order.

    contiguous: rank r holds the r-th of P equal time blocks.
    zigzag: the sequence is cut into 2P equal chunks; rank r holds chunk r
    followed by chunk 2P-1-r (early and late tokens paired).
    striped: token t belongs to rank t mod P, in order (rank r holds r, r+P,
    r+2P, ...): the pages name Striped Attention as a permutation that
    balances causal work; round-robin stripes of one token are the reading
    taken here.
    """
    tok = np.zeros((P, T // P), dtype=np.int32)
    if kind == "contiguous":
        assert T % P == 0
        n = T // P
        for r in range(P):
            for t in range(n):
                tok[r, t] = r * n + t
    elif kind == "zigzag":
        assert T % (2 * P) == 0
        c = T // (2 * P)
        for r in range(P):
            for t in range(c):
                tok[r, t] = r * c + t
                tok[r, c + t] = (2 * P - 1 - r) * c + t
    elif kind == "striped":
        assert T % P == 0
        for r in range(P):
            for t in range(T // P):
                tok[r, t] = t * P + r
    else:
        raise ValueError(kind)
    return tok


def schedule(P: int) -> np.ndarray:
    """Ring order: at step s rank r works on the K/V block of rank (r - s) mod P
    (each step every rank passes its block to the next rank)."""
    src = np.zeros((P, P), dtype=np.int32)
    for r in range(P):
        for s in range(P):
            src[r, s] = (r - s) % P
    return src


def is_visible(b, i, j, causal, kpm, am) -> bool:
    """Combined exclusions at global positions i (query), j (key)."""
    if causal and j > i:
        return False
    if kpm is not None and kpm[b][j]:
        return False
    if am is not None and am[i][j]:
        return False
    return True


def tile_classes(B, Lq, Lk, q_off=0, k_off=0, causal=False, kpm=None, am=None, tile=128):
    """Class of every (b, q-tile, k-tile) of the block rows [q_off, q_off+Lq) x keys
    [k_off, k_off+Lk), tiles of `tile` starting at the block origin.
    EMPTY: no visible pair; FULL: every pair visible; PARTIAL otherwise.
    Plain loops over every pair (small sizes only)."""
    kpm = None if kpm is None else np.asarray(kpm)
    am = None if am is None else np.asarray(am)
    nqt = -(-Lq // tile)
    nkt = -(-Lk // tile)
    cls = np.zeros((B, nqt, nkt), dtype=np.int8)
    for b in range(B):
        for qt in range(nqt):
            for kt in range(nkt):
                n_vis = n_all = 0
                for i in range(qt * tile, min(Lq, (qt + 1) * tile)):
                    for j in range(kt * tile, min(Lk, (kt + 1) * tile)):
                        n_all += 1
                        n_vis += is_visible(b, q_off + i, k_off + j, causal, kpm, am)
                cls[b, qt, kt] = EMPTY if n_vis == 0 else (FULL if n_vis == n_all else PARTIAL)
    return cls
