"""The C-ABI library builds, loads and exports every declared entry point; the
host-side index maps agree bit for bit with the oracle; bad arguments are
rejected on the host before anything reaches a GPU.  No GPU needed."""
import ctypes
import os
import re

import numpy as np
import pytest

import oracle
import blockwise_attention_gb300 as ba
from blockwise_attention_gb300 import _lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    src = open(os.path.join(ROOT, "include", "blockattn.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[a-z_0-9]+\s*\*?\s*([a-z_0-9]+)\s*\(", src, flags=re.M)
    return sorted(set(names))


def test_library_exports_every_declared_symbol():
    lib = ba.load()
    names = declared_functions()
    assert len(names) >= 10
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == set(_lib.EXPORTED)


def test_strerror():
    lib = ba.load()
    assert lib.ba_strerror(0) == b"ok"
    assert lib.ba_strerror(-4) == b"device wait timed out"


@pytest.mark.parametrize("T,P,kind", [(8, 4, "contiguous"), (8, 2, "zigzag"), (8, 2, "contiguous"),
                                      (8, 2, "striped"), (8192, 8, "striped"), (12, 3, "striped"),
                                      (1024, 4, "contiguous"), (8192, 8, "zigzag"), (65536, 16, "zigzag"),
                                      (512, 2, "contiguous"), (1000, 4, "zigzag"), (96, 3, "zigzag"),
                                      (7, 1, "contiguous")])
def test_index_maps_bit_exact(T, P, kind):
    tok, sch = ba.index_maps(T, P, kind)
    assert np.array_equal(tok, oracle.partition(T, P, kind))
    assert np.array_equal(sch, oracle.schedule(P))


def test_index_maps_rejects_indivisible():
    lib = ba.load()
    buf = (ctypes.c_int32 * 64)()
    assert lib.ba_index_maps(10, 4, 0, buf, buf) == _lib.BA_ERR_SHAPE
    assert lib.ba_index_maps(12, 4, 1, buf, buf) == _lib.BA_ERR_SHAPE
    assert lib.ba_index_maps(8, 0, 0, buf, buf) == _lib.BA_ERR_ARG


def test_argument_errors_are_host_side():
    lib = ba.load()
    T0 = _lib.ba_tensor(None, 0, 0, 0)
    T1 = _lib.ba_tensor(16, 1 << 20, 1 << 14, 64)
    dummy = ctypes.c_void_p(16)
    # NULL q
    assert lib.attn_block_fwd(T0, T1, T1, 1, 1, 8, 8, 64, 1, 0, 0, None, 0, None, 0, 0, 0.0, dummy, 1, dummy, 0,
                              None, 0, None) == _lib.BA_ERR_ARG
    # unsupported head dimension
    assert lib.attn_block_fwd(T1, T1, T1, 1, 1, 8, 8, 48, 1, 0, 0, None, 0, None, 0, 0, 0.0, dummy, 1, dummy, 0,
                              None, 0, None) == _lib.BA_ERR_SHAPE
    # accumulate needs an fp32 output
    assert lib.attn_block_fwd(T1, T1, T1, 1, 1, 8, 8, 64, 1, 0, 0, None, 0, None, 0, 0, 0.0, dummy, 1, dummy, 1,
                              None, 0, None) == _lib.BA_ERR_ARG
    # ring: T not divisible by 2P for zigzag
    assert lib.ring_attn_fwd(T1, T1, T1, 1, 1, 12, 64, 1, 4, 1, 1, None, 0, None, 0, 1, 0.0, 0, 1e4, dummy, 1,
                             dummy, None, None, 0, None) == _lib.BA_ERR_SHAPE
    # ring: odd d with rope
    assert lib.rope_apply(T1, T0, 1, 1, 8, 7, 1, None, 1e4, 1.0, dummy, None, None) == _lib.BA_ERR_ARG
    # negative Position Interpolation scale
    assert lib.rope_apply(T1, T0, 1, 1, 8, 8, 1, None, 1e4, -0.5, dummy, None, None) == _lib.BA_ERR_ARG
    # striped partitions take no masks (masks are indexed by token); T must divide by P
    assert lib.ring_attn_fwd(T1, T1, T1, 1, 1, 16, 64, 1, 4, 2, 1, dummy, 16, None, 0, 1, 0.0, 0, 1e4, dummy, 1,
                             dummy, None, None, 0, None) == _lib.BA_ERR_UNSUPPORTED
    assert lib.ring_attn_fwd(T1, T1, T1, 1, 1, 18, 64, 1, 4, 2, 1, None, 0, None, 0, 1, 0.0, 0, 1e4, dummy, 1,
                             dummy, None, None, 0, None) == _lib.BA_ERR_SHAPE
    # the striped backward is not built
    assert lib.ring_attn_bwd(T1, T1, T1, T1, T1, dummy, 1, 1, 16, 64, 1, 4, 2, 1, None, 0, None, 0, 1, 0.0,
                             dummy, dummy, dummy, None, 0, None) == _lib.BA_ERR_UNSUPPORTED
    assert lib.attn_merge(None, dummy, dummy, dummy, 4, 4, None) == _lib.BA_ERR_ARG
    # backward: NULL out, unsupported d, T not divisible by 2P, masks not covering positions
    assert lib.attn_block_bwd(T1, T1, T1, T0, T1, dummy, 1, 1, 8, 8, 64, 1, 0, 0, None, 0, None, 0, 0, 0.0,
                              dummy, dummy, dummy, 0, None, 0, None) == _lib.BA_ERR_ARG
    assert lib.attn_block_bwd(T1, T1, T1, T1, T1, dummy, 1, 1, 8, 8, 48, 1, 0, 0, None, 0, None, 0, 0, 0.0,
                              dummy, dummy, dummy, 0, None, 0, None) == _lib.BA_ERR_SHAPE
    assert lib.attn_block_bwd(T1, T1, T1, T1, T1, dummy, 1, 1, 8, 8, 64, 1, 0, 4, dummy, 8, None, 0, 0, 0.0,
                              dummy, dummy, dummy, 0, None, 0, None) == _lib.BA_ERR_ARG
    assert lib.ring_attn_bwd(T1, T1, T1, T1, T1, dummy, 1, 1, 12, 64, 1, 4, 1, 1, None, 0, None, 0, 1, 0.0,
                             dummy, dummy, dummy, None, 0, None) == _lib.BA_ERR_SHAPE


def test_workspace_sizes():
    # rope copies of q and k for the 64K config: 2 x 268M bf16 elements
    n = ba.ring_attn_fwd_workspace_size(1, 32, 65536, 128, __import__("torch").bfloat16, 16, "zigzag", "fused",
                                        False, True)
    # plus the 256-byte block of item counters (one per launch) at the front
    assert n == 256 + 2 * 32 * 65536 * 128 * 2
    assert ba.ring_attn_fwd_workspace_size(1, 32, 65536, 128, __import__("torch").bfloat16, 16, "zigzag",
                                           "fused", False, False) == 256
    # step-wise: one counter per ring step (64 steps -> 256 bytes, 65 -> 512)
    assert ba.ring_attn_fwd_workspace_size(1, 1, 128 * 64, 64, __import__("torch").float32, 64, "contiguous",
                                           "stepwise", False, False) == 256
    assert ba.ring_attn_fwd_workspace_size(1, 1, 128 * 65, 64, __import__("torch").float32, 65, "contiguous",
                                           "stepwise", False, False) == 512


def test_masks_must_cover_the_positions_read():
    """The C ABI sees only a mask's pointer and row stride; the binding rejects a
    mask with too few rows or key positions before any launch (a local (Lq, Lk)
    attn_mask passed with q_off > 0 is the easy way to get this wrong)."""
    import torch
    kpm = torch.zeros((2, 100), dtype=torch.uint8)
    with pytest.raises(ValueError, match="does not cover"):
        _lib._masks(kpm, None, 3, 10, 100)            # fewer rows than batch items
    with pytest.raises(ValueError, match="does not cover"):
        _lib._masks(kpm, None, 2, 10, 101)            # fewer key positions than k_off + Lk
    am = torch.zeros((64, 128), dtype=torch.uint8)
    with pytest.raises(ValueError, match="does not cover"):
        _lib._masks(None, am, 1, 32 + 64, 128)        # local (Lq, Lk) mask with q_off = 32
    with pytest.raises(ValueError, match="overlap"):
        _lib._masks(None, torch.zeros((4, 256), dtype=torch.uint8)[:, :100].as_strided((8, 100), (50, 1)),
                    1, 8, 100)
    # shapes that cover everything pass the coverage checks (and stop only at the
    # device check, since these are host tensors)
    with pytest.raises(ValueError, match="CUDA"):
        _lib._masks(kpm, am, 2, 64, 100)
