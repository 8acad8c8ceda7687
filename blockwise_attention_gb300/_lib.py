"""Build and load libblockattn.so (CUDA, sm_103a) and bind its C ABI.

The binding only marshals arguments: torch tensors become device pointers and
element strides, outputs and workspace are allocated with torch, and every
step of the computation runs in the library's kernels.  There is no other
implementation behind these functions; if the library cannot be built or
loaded they raise.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from concurrent.futures import ThreadPoolExecutor

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
_ROOT = os.path.dirname(_PKG)
_CSRC = os.path.join(_PKG, "csrc")
_BUILD = os.path.join(_PKG, "_build")
LIB_PATH = os.path.join(_BUILD, "libblockattn.so")
_SOURCES = ["api.cu", "attn_simt.cu", "attn_tc.cu", "attn_bwd.cu", "attn_bwd_tc.cu", "ulysses.cu", "decode.cu"]
_HEADERS = ["common.cuh", "internal.h", "epilogue.cuh", "tc_ptx.cuh"]
ARCH_FLAGS = ["-gencode", "arch=compute_103a,code=sm_103a"]

BA_OK, BA_ERR_ARG, BA_ERR_SHAPE, BA_ERR_CUDA, BA_ERR_TIMEOUT, BA_ERR_UNSUPPORTED, BA_ERR_WORKSPACE = \
    0, -1, -2, -3, -4, -5, -6
BA_ERR_NOALLOC_LIMIT = -7
BA_NOALLOC_MAX_CLASS_BYTES = 1 << 20
BA_F32, BA_BF16 = 0, 1
PARTITIONS = {"contiguous": 0, "zigzag": 1, "striped": 2}
MODES = {"stepwise": 0, "fused": 1}
BA_TILE_EMPTY, BA_TILE_FULL, BA_TILE_PARTIAL = 0, 1, 2

_lib = None


class BlockAttnError(RuntimeError):
    def __init__(self, fn, code):
        msg = _lib.ba_strerror(code).decode() if _lib is not None else str(code)
        super().__init__(f"{fn} failed: {msg} ({code})")
        self.code = code


def _nvcc():
    for c in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", "nvcc"):
        if c and (os.path.isabs(c) and os.path.exists(c) or not os.path.isabs(c)):
            return c
    return "nvcc"


def _stale() -> bool:
    if not os.path.exists(LIB_PATH):
        return True
    t = os.path.getmtime(LIB_PATH)
    deps = [os.path.join(_CSRC, f) for f in _SOURCES + _HEADERS]
    deps.append(os.path.join(_ROOT, "include", "blockattn.h"))
    return any(os.path.getmtime(p) > t for p in deps)


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile the CUDA sources for sm_103a (in parallel) and link the shared library."""
    if not force and not _stale():
        return LIB_PATH
    os.makedirs(_BUILD, exist_ok=True)
    nvcc = _nvcc()
    common = [nvcc, *ARCH_FLAGS, "-lineinfo", "-O3", "-std=c++17", "-Xcompiler", "-fPIC",
              "-I", os.path.join(_ROOT, "include")]

    def compile_one(src):
        obj = os.path.join(_BUILD, src.replace(".cu", ".o"))
        cmd = common + ["-c", os.path.join(_CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stderr}")
        if verbose and r.stderr:
            print(r.stderr)
        return obj

    with ThreadPoolExecutor(len(_SOURCES)) as ex:
        objs = list(ex.map(compile_one, _SOURCES))
    tmp = LIB_PATH + f".tmp{os.getpid()}"
    r = subprocess.run([nvcc, *ARCH_FLAGS, "-shared", "-o", tmp, *objs], capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stderr}")
    os.replace(tmp, LIB_PATH)
    return LIB_PATH


class ba_tensor(ctypes.Structure):
    _fields_ = [("ptr", ctypes.c_void_p), ("sB", ctypes.c_int64), ("sH", ctypes.c_int64),
                ("sT", ctypes.c_int64)]


EXPORTED = ["attn_block_fwd", "attn_block_fwd_workspace_size", "attn_merge", "ring_attn_fwd",
            "ring_attn_fwd_workspace_size", "rope_apply", "ba_tile_classes", "ba_index_maps",
            "ba_sync_status", "ba_debug_wait_timeout", "ba_strerror", "attn_block_fwd_noalloc",
            "attn_block_bwd", "attn_block_bwd_workspace_size", "ring_attn_bwd", "ring_attn_bwd_workspace_size",
            "ulysses_all_to_all", "ulysses_attn_fwd", "ulysses_attn_fwd_workspace_size",
            "attn_decode_fwd", "attn_decode_workspace_size", "ba_pair_schedule"]


def load(path: str | None = None):
    """Load the library (building it first when needed) and declare signatures."""
    global _lib
    if _lib is not None:
        return _lib
    if path is None:
        path = build()
    lib = ctypes.CDLL(path)
    i, i64, sz, vp, f = ctypes.c_int, ctypes.c_int64, ctypes.c_size_t, ctypes.c_void_p, ctypes.c_float
    T = ba_tensor
    lib.ba_strerror.restype = ctypes.c_char_p
    lib.ba_strerror.argtypes = [i]
    lib.attn_block_fwd_workspace_size.restype = sz
    lib.attn_block_fwd_workspace_size.argtypes = [i, i, i, i]
    lib.attn_block_fwd.restype = i
    lib.attn_block_fwd.argtypes = [T, T, T, i, i, i, i, i, i, i64, i64, vp, i64, vp, i64, i, f, vp, i, vp, i,
                                   vp, sz, vp]
    lib.attn_block_fwd_noalloc.restype = i
    lib.attn_block_fwd_noalloc.argtypes = [T, T, T, i, i, i, i, i, i, i64, i64, vp, i64, vp, i64, i, f, vp, i, vp,
                                           i, vp]
    lib.attn_merge.restype = i
    lib.attn_merge.argtypes = [vp, vp, vp, vp, i64, i, vp]
    lib.ring_attn_fwd_workspace_size.restype = sz
    lib.ring_attn_fwd_workspace_size.argtypes = [i, i, i, i, i, i, i, i, i, i, i]
    lib.ring_attn_fwd.restype = i
    lib.ring_attn_fwd.argtypes = [T, T, T, i, i, i, i, i, i, i, i, vp, i64, vp, i64, i, f, i, f, vp, i, vp, vp,
                                  vp, sz, vp]
    lib.rope_apply.restype = i
    lib.rope_apply.argtypes = [T, T, i, i, i, i, i, vp, f, f, vp, vp, vp]
    lib.ba_tile_classes.restype = i
    lib.ba_tile_classes.argtypes = [i, i, i, i64, i64, vp, i64, vp, i64, i, vp, vp]
    lib.ba_index_maps.restype = i
    lib.ba_index_maps.argtypes = [i, i, i, vp, vp]
    lib.ba_pair_schedule.restype = i
    lib.ba_pair_schedule.argtypes = [i, i, i, i, i, i, i, vp, ctypes.c_int64]
    lib.ba_sync_status.restype = i
    lib.ba_sync_status.argtypes = [vp]
    lib.ba_debug_wait_timeout.restype = i
    lib.ba_debug_wait_timeout.argtypes = [i64, vp]
    lib.attn_block_bwd_workspace_size.restype = sz
    lib.attn_block_bwd_workspace_size.argtypes = [i, i, i]
    lib.attn_block_bwd.restype = i
    lib.attn_block_bwd.argtypes = [T, T, T, T, T, vp, i, i, i, i, i, i, i64, i64, vp, i64, vp, i64, i, f,
                                   vp, vp, vp, i, vp, sz, vp]
    lib.ring_attn_bwd_workspace_size.restype = sz
    lib.ring_attn_bwd_workspace_size.argtypes = [i, i, i]
    lib.ring_attn_bwd.restype = i
    lib.ring_attn_bwd.argtypes = [T, T, T, T, T, vp, i, i, i, i, i, i, i, i, vp, i64, vp, i64, i, f,
                                  vp, vp, vp, vp, sz, vp]
    lib.ulysses_all_to_all.restype = i
    lib.ulysses_all_to_all.argtypes = [vp, vp, i, i, i, i, i, i, i, vp]
    lib.ulysses_attn_fwd_workspace_size.restype = sz
    lib.ulysses_attn_fwd_workspace_size.argtypes = [i, i, i, i, i, i, i]
    lib.ulysses_attn_fwd.restype = i
    lib.ulysses_attn_fwd.argtypes = [vp, vp, vp, i, i, i, i, i, i, vp, i64, vp, i64, i, f, vp, vp, vp, sz, vp]
    lib.attn_decode_workspace_size.restype = sz
    lib.attn_decode_workspace_size.argtypes = [i, i, i, i, i]
    lib.attn_decode_fwd.restype = i
    lib.attn_decode_fwd.argtypes = [T, T, T, i, i, i, i, i, vp, i, f, vp, i, vp, vp, sz, vp]
    _lib = lib
    return lib


def _check(fn, rc):
    if rc != BA_OK:
        raise BlockAttnError(fn, rc)


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _dtype_code(t: torch.dtype) -> int:
    if t == torch.float32:
        return BA_F32
    if t == torch.bfloat16:
        return BA_BF16
    raise TypeError(f"unsupported dtype {t}")


def _tensor(x: torch.Tensor) -> ba_tensor:
    if x.dim() != 4 or x.stride(-1) != 1:
        raise ValueError("expected a (B, H, T, d) tensor with a contiguous last axis")
    if not x.is_cuda:
        raise ValueError("expected a CUDA tensor")
    return ba_tensor(x.data_ptr(), x.stride(0), x.stride(1), x.stride(2))


def _mask(m, rows, cols, name="mask"):
    """(pointer, ld) of a 2-D uint8 mask.  The library indexes masks at global
    positions and sees only the pointer and the row stride, so the binding
    checks here that the mask covers every row (batch item for the key-padding
    mask, query position for attn_mask) and every key position a launch reads."""
    if m is None:
        return None, 0
    if m.dtype != torch.uint8 or m.dim() != 2 or m.stride(1) != 1:
        raise ValueError("masks are 2-D uint8 CUDA tensors with a contiguous last axis")
    if m.shape[0] < rows or m.shape[1] < cols:
        raise ValueError(f"{name} of shape {tuple(m.shape)} does not cover the ({rows}, {cols}) "
                         f"rows and key positions the call reads")
    if m.shape[0] > 1 and m.stride(0) < cols:
        raise ValueError(f"{name} rows overlap (stride {m.stride(0)} < {cols} key positions)")
    if not m.is_cuda:
        raise ValueError("masks are 2-D uint8 CUDA tensors with a contiguous last axis")
    return ctypes.c_void_p(m.data_ptr()), m.stride(0)


def _masks(key_padding_mask, attn_mask, B, q_rows, k_cols):
    """Both masks of a call whose queries reach global position q_rows - 1 and
    whose keys reach k_cols - 1."""
    kpm, kpm_ld = _mask(key_padding_mask, B, k_cols, "key_padding_mask")
    am, am_ld = _mask(attn_mask, q_rows, k_cols, "attn_mask")
    return kpm, kpm_ld, am, am_ld


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _check_out(out, lse, shape):
    """Outputs are written as contiguous (B, H, L, d) and (B, H, L) buffers."""
    if tuple(out.shape) != tuple(shape) or not out.is_contiguous() or not out.is_cuda:
        raise ValueError(f"out must be a contiguous CUDA tensor of shape {tuple(shape)}")
    if tuple(lse.shape) != tuple(shape[:3]) or not lse.is_contiguous() or lse.dtype != torch.float32:
        raise ValueError(f"lse must be a contiguous float32 CUDA tensor of shape {tuple(shape[:3])}")


def attn_block_fwd(q, k, v, *, q_off=0, k_off=0, key_padding_mask=None, attn_mask=None, causal=False,
                   scale=None, out=None, out_dtype=None, lse=None, accumulate=False, workspace=None,
                   stream=None):
    """One attention block with per-row natural-log LSE; see include/blockattn.h."""
    lib = load()
    B, H, Lq, d = q.shape
    Lk = k.shape[2]
    dt = _dtype_code(q.dtype)
    if out_dtype is None:
        out_dtype = out.dtype if out is not None else q.dtype
    if out is None:
        out = torch.empty((B, H, Lq, d), dtype=out_dtype, device=q.device)
    if lse is None:
        lse = torch.empty((B, H, Lq), dtype=torch.float32, device=q.device)
    _check_out(out, lse, (B, H, Lq, d))
    kpm, kpm_ld, am, am_ld = _masks(key_padding_mask, attn_mask, B, q_off + Lq, k_off + Lk)
    need = lib.attn_block_fwd_workspace_size(B, Lq, Lk, int(kpm is not None or am is not None))
    if workspace is None and need:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    rc = lib.attn_block_fwd(_tensor(q), _tensor(k), _tensor(v), B, H, Lq, Lk, d, dt, q_off, k_off, kpm, kpm_ld,
                            am, am_ld, int(bool(causal)), 0.0 if scale is None else float(scale),
                            _ptr(out), _dtype_code(out.dtype), _ptr(lse), int(bool(accumulate)),
                            _ptr(workspace), 0 if workspace is None else workspace.numel(), _stream(stream))
    _check("attn_block_fwd", rc)
    return out, lse


def attn_block_fwd_noalloc(q, k, v, out, lse, *, q_off=0, k_off=0, key_padding_mask=None, attn_mask=None,
                           causal=False, scale=None, accumulate=False, stream=None):
    """attn_block_fwd for callers that cannot allocate device memory: the caller
    passes out and lse, and the library allocates nothing (its tile-class scratch
    is a fixed device array of BA_NOALLOC_MAX_CLASS_BYTES).  Returns (out, lse)."""
    lib = load()
    B, H, Lq, d = q.shape
    Lk = k.shape[2]
    _check_out(out, lse, (B, H, Lq, d))
    kpm, kpm_ld, am, am_ld = _masks(key_padding_mask, attn_mask, B, q_off + Lq, k_off + Lk)
    rc = lib.attn_block_fwd_noalloc(_tensor(q), _tensor(k), _tensor(v), B, H, Lq, Lk, d, _dtype_code(q.dtype),
                                    q_off, k_off, kpm, kpm_ld, am, am_ld, int(bool(causal)),
                                    0.0 if scale is None else float(scale), _ptr(out), _dtype_code(out.dtype),
                                    _ptr(lse), int(bool(accumulate)), _stream(stream))
    _check("attn_block_fwd_noalloc", rc)
    return out, lse


def attn_merge(out_a, lse_a, out_b, lse_b, stream=None):
    """In place: (out_a, lse_a) <- LSE merge of (out_a, lse_a) and (out_b, lse_b)."""
    lib = load()
    for t in (out_a, lse_a, out_b, lse_b):
        if t.dtype != torch.float32 or not t.is_contiguous() or not t.is_cuda:
            raise ValueError("attn_merge takes contiguous fp32 CUDA tensors")
    d = out_a.shape[-1]
    rows = lse_a.numel()
    if out_a.numel() != rows * d or out_b.numel() != rows * d or lse_b.numel() != rows:
        raise ValueError("shape mismatch")
    _check("attn_merge", lib.attn_merge(_ptr(out_a), _ptr(lse_a), _ptr(out_b), _ptr(lse_b), rows, d,
                                        _stream(stream)))
    return out_a, lse_a


def ring_attn_fwd_workspace_size(B, H, T, d, dtype, P, partition="contiguous", mode="fused", has_masks=False,
                                 rope=False, out_dtype=None):
    lib = load()
    dt = _dtype_code(dtype)
    odt = dt if out_dtype is None else _dtype_code(out_dtype)
    return lib.ring_attn_fwd_workspace_size(B, H, T, d, dt, P, PARTITIONS[partition], MODES[mode],
                                            int(bool(has_masks)), int(bool(rope)), odt)


def ring_attn_fwd(q, k, v, *, P, partition="contiguous", mode="fused", key_padding_mask=None, attn_mask=None,
                  causal=False, scale=None, rope=False, rope_base=10000.0, out=None, out_dtype=None, lse=None,
                  return_index_maps=False, workspace=None, stream=None):
    """Ring Attention over P emulated ranks; see include/blockattn.h.
    Returns (out, lse) or (out, lse, tok_of (P, T/P), schedule (P, P))."""
    lib = load()
    B, H, T, d = q.shape
    dt = _dtype_code(q.dtype)
    if out_dtype is None:
        out_dtype = out.dtype if out is not None else q.dtype
    if out is None:
        out = torch.empty((B, H, T, d), dtype=out_dtype, device=q.device)
    if lse is None:
        lse = torch.empty((B, H, T), dtype=torch.float32, device=q.device)
    _check_out(out, lse, (B, H, T, d))
    kpm, kpm_ld, am, am_ld = _masks(key_padding_mask, attn_mask, B, T, T)
    masks = kpm is not None or am is not None
    need = ring_attn_fwd_workspace_size(B, H, T, d, q.dtype, P, partition, mode, masks, rope, out.dtype)
    if workspace is None and need:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    maps = None
    if return_index_maps:
        maps = (ctypes.c_int32 * (T + P * P))()
    rc = lib.ring_attn_fwd(_tensor(q), _tensor(k), _tensor(v), B, H, T, d, dt, P, PARTITIONS[partition],
                           MODES[mode], kpm, kpm_ld, am, am_ld, int(bool(causal)),
                           0.0 if scale is None else float(scale), int(bool(rope)), float(rope_base),
                           _ptr(out), _dtype_code(out.dtype), _ptr(lse),
                           None if maps is None else ctypes.cast(maps, ctypes.c_void_p),
                           _ptr(workspace), 0 if workspace is None else workspace.numel(), _stream(stream))
    _check("ring_attn_fwd", rc)
    if return_index_maps:
        import numpy as np
        arr = np.ctypeslib.as_array(maps).copy()
        return out, lse, arr[:T].reshape(P, T // P), arr[T:].reshape(P, P)
    return out, lse


def _grads(B, H, Lq, Lk, d, device, dq, dk, dv):
    shapes = ((dq, (B, H, Lq, d)), (dk, (B, H, Lk, d)), (dv, (B, H, Lk, d)))
    res = []
    for t, shape in shapes:
        if t is None:
            t = torch.empty(shape, dtype=torch.float32, device=device)
        elif t.dtype != torch.float32 or not t.is_contiguous() or tuple(t.shape) != shape or not t.is_cuda:
            raise ValueError(f"gradient buffers must be contiguous fp32 CUDA tensors of shape {shape}")
        res.append(t)
    return res


def _check_bwd_inputs(q, out, dout, lse):
    if out.dtype != q.dtype or dout.dtype != q.dtype:
        raise TypeError("out and dout must have the dtype of q")
    if out.shape != q.shape or dout.shape != q.shape:
        raise ValueError("out and dout must have the shape of q")
    if lse.dtype != torch.float32 or not lse.is_contiguous() or tuple(lse.shape) != tuple(q.shape[:3]):
        raise ValueError("lse must be a contiguous fp32 tensor of shape (B, H, L)")


def attn_block_bwd(q, k, v, out, dout, lse, *, q_off=0, k_off=0, key_padding_mask=None, attn_mask=None,
                   causal=False, scale=None, dq=None, dk=None, dv=None, accumulate=False, workspace=None,
                   stream=None):
    """Gradients (dq, dk, dv) (fp32) of one attention block given the forward
    out and lse of the whole rows; see include/blockattn.h."""
    lib = load()
    B, H, Lq, d = q.shape
    Lk = k.shape[2]
    _check_bwd_inputs(q, out, dout, lse)
    dq, dk, dv = _grads(B, H, Lq, Lk, d, q.device, dq, dk, dv)
    kpm, kpm_ld, am, am_ld = _masks(key_padding_mask, attn_mask, B, q_off + Lq, k_off + Lk)
    need = lib.attn_block_bwd_workspace_size(B, H, Lq)
    if workspace is None and need:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    rc = lib.attn_block_bwd(_tensor(q), _tensor(k), _tensor(v), _tensor(out), _tensor(dout), _ptr(lse), B, H, Lq,
                            Lk, d, _dtype_code(q.dtype), q_off, k_off, kpm, kpm_ld, am, am_ld, int(bool(causal)),
                            0.0 if scale is None else float(scale), _ptr(dq), _ptr(dk), _ptr(dv),
                            int(bool(accumulate)), _ptr(workspace), 0 if workspace is None else workspace.numel(),
                            _stream(stream))
    _check("attn_block_bwd", rc)
    return dq, dk, dv


def ring_attn_bwd(q, k, v, out, dout, lse, *, P, partition="contiguous", mode="fused", key_padding_mask=None,
                  attn_mask=None, causal=False, scale=None, dq=None, dk=None, dv=None, workspace=None,
                  stream=None):
    """Ring Attention backward over P emulated ranks: (dq, dk, dv) fp32 in global
    token order; see include/blockattn.h."""
    lib = load()
    B, H, T, d = q.shape
    _check_bwd_inputs(q, out, dout, lse)
    dq, dk, dv = _grads(B, H, T, T, d, q.device, dq, dk, dv)
    kpm, kpm_ld, am, am_ld = _masks(key_padding_mask, attn_mask, B, T, T)
    need = lib.ring_attn_bwd_workspace_size(B, H, T)
    if workspace is None and need:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    rc = lib.ring_attn_bwd(_tensor(q), _tensor(k), _tensor(v), _tensor(out), _tensor(dout), _ptr(lse), B, H, T, d,
                           _dtype_code(q.dtype), P, PARTITIONS[partition], MODES[mode], kpm, kpm_ld, am, am_ld,
                           int(bool(causal)), 0.0 if scale is None else float(scale), _ptr(dq), _ptr(dk),
                           _ptr(dv), _ptr(workspace), 0 if workspace is None else workspace.numel(),
                           _stream(stream))
    _check("ring_attn_bwd", rc)
    return dq, dk, dv


A2A = {"token_to_head": 0, "head_to_token": 1}


def ulysses_all_to_all(x, P, direction, *, out=None, stream=None):
    """One Ulysses exchange of a contiguous stacked array: token_to_head takes
    (P, H, B, T/P, d) to (P, H/P, B, T, d); head_to_token is the inverse."""
    lib = load()
    if not x.is_contiguous() or not x.is_cuda:
        raise ValueError("ulysses_all_to_all takes a contiguous CUDA tensor")
    if direction == "token_to_head":
        P_, H, B, Tl, d = x.shape
        shape, T = (P, H // P, B, Tl * P, d), Tl * P
    elif direction == "head_to_token":
        P_, hl, B, T, d = x.shape
        H = hl * P
        shape = (P, H, B, T // P, d)
    else:
        raise ValueError(direction)
    if P_ != P:
        raise ValueError("leading axis must be P")
    if out is None:
        out = torch.empty(shape, dtype=x.dtype, device=x.device)
    elif tuple(out.shape) != shape or out.dtype != x.dtype or not out.is_contiguous():
        raise ValueError(f"out must be a contiguous tensor of shape {shape}")
    rc = lib.ulysses_all_to_all(_ptr(x), _ptr(out), P, H, B, T, d, x.element_size(), A2A[direction],
                                _stream(stream))
    _check("ulysses_all_to_all", rc)
    return out


def ulysses_attn_fwd(q_tok, k_tok, v_tok, *, key_padding_mask=None, attn_mask=None, causal=False, scale=None,
                     out=None, lse=None, workspace=None, stream=None):
    """Ulysses attention over P emulated ranks from token shards (P, H, B, T/P, d):
    returns (out (P, H, B, T/P, d), lse (P, H, B, T/P) fp32); see include/blockattn.h."""
    lib = load()
    for t in (q_tok, k_tok, v_tok):
        if not t.is_contiguous() or not t.is_cuda or t.shape != q_tok.shape or t.dtype != q_tok.dtype:
            raise ValueError("q_tok, k_tok, v_tok must be contiguous CUDA tensors of one shape and dtype")
    P, H, B, Tl, d = q_tok.shape
    T = P * Tl
    if out is None:
        out = torch.empty_like(q_tok)
    if lse is None:
        lse = torch.empty((P, H, B, Tl), dtype=torch.float32, device=q_tok.device)
    if tuple(out.shape) != tuple(q_tok.shape) or out.dtype != q_tok.dtype or not out.is_contiguous():
        raise ValueError("out must be contiguous, of the shape and dtype of q_tok")
    if tuple(lse.shape) != (P, H, B, Tl) or lse.dtype != torch.float32 or not lse.is_contiguous():
        raise ValueError("lse must be a contiguous fp32 tensor of shape (P, H, B, T/P)")
    kpm, kpm_ld, am, am_ld = _masks(key_padding_mask, attn_mask, B, T, T)
    dt = _dtype_code(q_tok.dtype)
    need = lib.ulysses_attn_fwd_workspace_size(P, H, B, T, d, dt, int(kpm is not None or am is not None))
    if workspace is None and need:
        workspace = torch.empty(need, dtype=torch.uint8, device=q_tok.device)
    rc = lib.ulysses_attn_fwd(_ptr(q_tok), _ptr(k_tok), _ptr(v_tok), P, H, B, T, d, dt, kpm, kpm_ld, am, am_ld,
                              int(bool(causal)), 0.0 if scale is None else float(scale), _ptr(out), _ptr(lse),
                              _ptr(workspace), 0 if workspace is None else workspace.numel(), _stream(stream))
    _check("ulysses_attn_fwd", rc)
    return out, lse


def attn_decode_fwd(q, k_cache, v_cache, *, lengths=None, num_splits=0, scale=None, out=None, out_dtype=None,
                    lse=None, workspace=None, stream=None):
    """Decode attention of q (B, H, 1, d) against k_cache, v_cache (B, H, S, d),
    split along the keys and merged by the LSE rule; lengths: int32 (B) CUDA
    tensor of valid cache lengths or None.  Returns (out, lse)."""
    lib = load()
    B, H, one, d = q.shape
    if one != 1:
        raise ValueError("decode takes one query per (b, h): q of shape (B, H, 1, d)")
    S = k_cache.shape[2]
    if out_dtype is None:
        out_dtype = out.dtype if out is not None else q.dtype
    if out is None:
        out = torch.empty((B, H, 1, d), dtype=out_dtype, device=q.device)
    if lse is None:
        lse = torch.empty((B, H, 1), dtype=torch.float32, device=q.device)
    _check_out(out, lse, (B, H, 1, d))
    if lengths is not None and (lengths.dtype != torch.int32 or not lengths.is_cuda or lengths.numel() != B):
        raise ValueError("lengths must be an int32 CUDA tensor of B entries")
    need = lib.attn_decode_workspace_size(B, H, S, d, int(num_splits))
    if workspace is None and need:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    rc = lib.attn_decode_fwd(_tensor(q), _tensor(k_cache), _tensor(v_cache), B, H, S, d, _dtype_code(q.dtype),
                             _ptr(lengths), int(num_splits), 0.0 if scale is None else float(scale), _ptr(out),
                             _dtype_code(out.dtype), _ptr(lse), _ptr(workspace),
                             0 if workspace is None else workspace.numel(), _stream(stream))
    _check("attn_decode_fwd", rc)
    return out, lse


def rope_apply(x, *, x2=None, base=10000.0, positions=None, pos_scale=1.0, out=None, out2=None, stream=None):
    """Rotary position embedding of x (B, H, T, d) into a contiguous output; with
    x2 given, rotates x2 by the same launch and returns (y, y2).  pos_scale is
    the Position Interpolation factor applied to the position index."""
    lib = load()
    B, H, T, d = x.shape
    if out is None:
        out = torch.empty((B, H, T, d), dtype=x.dtype, device=x.device)
    if x2 is not None:
        if x2.shape != x.shape or x2.dtype != x.dtype:
            raise ValueError("x2 must match x")
        if out2 is None:
            out2 = torch.empty((B, H, T, d), dtype=x.dtype, device=x.device)
    if positions is not None and (positions.dtype != torch.int32 or not positions.is_cuda):
        raise ValueError("positions: int32 CUDA tensor")
    t2 = _tensor(x2) if x2 is not None else ba_tensor(None, 0, 0, 0)
    _check("rope_apply", lib.rope_apply(_tensor(x), t2, B, H, T, d, _dtype_code(x.dtype), _ptr(positions),
                                        float(base), float(pos_scale), _ptr(out), _ptr(out2), _stream(stream)))
    return out if x2 is None else (out, out2)


def tile_classes(B, Lq, Lk, *, q_off=0, k_off=0, key_padding_mask=None, attn_mask=None, causal=False,
                 device="cuda", stream=None):
    """int8 (B, ceil(Lq/128), ceil(Lk/128)) tile classes computed on the device."""
    lib = load()
    out = torch.empty((B, -(-Lq // 128), -(-Lk // 128)), dtype=torch.int8, device=device)
    kpm, kpm_ld, am, am_ld = _masks(key_padding_mask, attn_mask, B, q_off + Lq, k_off + Lk)
    _check("ba_tile_classes", lib.ba_tile_classes(B, Lq, Lk, q_off, k_off, kpm, kpm_ld, am, am_ld,
                                                  int(bool(causal)), _ptr(out), _stream(stream)))
    return out


def index_maps(T, P, partition="contiguous"):
    """Host, exact: (tok_of (P, T/P) int32, schedule (P, P) int32)."""
    import numpy as np
    lib = load()
    tok = np.zeros(T, dtype=np.int32)
    sch = np.zeros(P * P, dtype=np.int32)
    _check("ba_index_maps", lib.ba_index_maps(T, P, PARTITIONS[partition], tok.ctypes.data_as(ctypes.c_void_p),
                                              sch.ctypes.data_as(ctypes.c_void_p)))
    return tok.reshape(P, T // P), sch.reshape(P, P)


def pair_schedule(B, H, T, P, partition="zigzag", causal=True, num_sms=152):
    """Host, exact: the tensor-core forward kernel's work items for a ring_attn_fwd
    launch without masks, in dealing order, as an (n, 8) int32 array of
    (b, h, tile-0 row0, tile-0 rows, tile-1 row0, tile-1 rows, key tiles, phase)."""
    import numpy as np
    lib = load()
    n = lib.ba_pair_schedule(B, H, T, P, PARTITIONS[partition], int(causal), num_sms, None, 0)
    _check("ba_pair_schedule", min(n, 0))
    items = np.zeros((max(n, 0), 8), dtype=np.int32)
    if n > 0:
        _check("ba_pair_schedule", min(lib.ba_pair_schedule(B, H, T, P, PARTITIONS[partition], int(causal), num_sms,
                                                            items.ctypes.data_as(ctypes.c_void_p), n), 0))
    return items


def sync_status(stream=None) -> int:
    """Synchronise and return BA_OK, or BA_ERR_TIMEOUT when a bounded device wait expired."""
    return load().ba_sync_status(_stream(stream))


def debug_wait_timeout(timeout_ns: int, stream=None):
    _check("ba_debug_wait_timeout", load().ba_debug_wait_timeout(int(timeout_ns), _stream(stream)))
