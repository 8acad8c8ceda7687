"""GPU parity of the attention backward (attn_block_bwd, ring_attn_bwd) against
the fp64 gradient oracle.  The forward results the backward consumes (out, lse)
come from the library's own forward, as in a training step.

Tolerance: the largest absolute error of each gradient, divided by that
gradient's largest magnitude.  fp32 inputs: 1e-4 (fp32 accumulation over at
most a few thousand terms).  bf16 inputs: 2e-2, because the forward output the
backward reads is rounded to bf16 (relative 2^-9) and enters every
ds = p (dout . v - dout . out)."""
import math

import numpy as np
import pytest
import torch

import oracle
import blockwise_attention_gb300 as ba

pytestmark = pytest.mark.gpu

TOL = {"bf16": 2e-2, "f32": 1e-4}
DT = {"bf16": torch.bfloat16, "f32": torch.float32}


def rand(shape, dtype, seed, std=1.0):
    g = torch.Generator(device="cuda").manual_seed(seed)
    return (torch.randn(shape, generator=g, device="cuda") * std).to(dtype)


def check(grads, refs, dt, label):
    for name, g, r in zip(("dq", "dk", "dv"), grads, refs):
        g = g.detach().cpu().numpy().astype(np.float64)
        assert np.isfinite(g).all(), f"{label} {name}: non-finite"
        scale = max(float(np.abs(r).max()), 1e-30)
        err = float(np.abs(g - r).max()) / scale
        print({"label": label, "grad": name, "rel_max_err": err})
        assert err <= TOL[dt], (label, name, err)


@pytest.mark.parametrize("dt,d", [("bf16", 128), ("bf16", 64), ("f32", 128), ("f32", 64), ("f32", 32),
                                  ("bf16", 16)])
@pytest.mark.parametrize("causal", [False, True])
def test_block_backward_ragged_offsets(dt, d, causal):
    B, H, Lq, Lk = 2, 2, 300, 333
    q_off, k_off = 40, 0
    q, k, v = rand((B, H, Lq, d), DT[dt], 1, 0.5), rand((B, H, Lk, d), DT[dt], 2, 0.5), rand((B, H, Lk, d), DT[dt], 3)
    g = rand((B, H, Lq, d), DT[dt], 4)
    out, lse = ba.attn_block_fwd(q, k, v, q_off=q_off, k_off=k_off, causal=causal)
    grads = ba.attn_block_bwd(q, k, v, out, g, lse, q_off=q_off, k_off=k_off, causal=causal)
    refs = oracle.attention_bwd(q.float().cpu(), k.float().cpu(), v.float().cpu(), g.float().cpu(), causal=causal,
                                q_pos0=q_off, k_pos0=k_off)[:3]
    check(grads, refs, dt, f"block {dt} d={d} causal={causal}")


def test_block_backward_masks_at_offsets():
    B, H, Lq, Lk, q_off, k_off, d = 2, 2, 200, 260, 100, 60, 64
    q, k, v = rand((B, H, Lq, d), torch.float32, 10), rand((B, H, Lk, d), torch.float32, 11), \
        rand((B, H, Lk, d), torch.float32, 12)
    g = rand((B, H, Lq, d), torch.float32, 13)
    rng = np.random.default_rng(3)
    kpm = (rng.random((B, k_off + Lk)) < 0.2).astype(np.uint8)
    am = (rng.random((q_off + Lq, k_off + Lk)) < 0.3).astype(np.uint8)
    am[q_off + 5, :] = 1   # a row that sees nothing
    kpm_t, am_t = torch.from_numpy(kpm).cuda(), torch.from_numpy(am).cuda()
    out, lse = ba.attn_block_fwd(q, k, v, q_off=q_off, k_off=k_off, key_padding_mask=kpm_t, attn_mask=am_t,
                                 causal=True)
    grads = ba.attn_block_bwd(q, k, v, out, g, lse, q_off=q_off, k_off=k_off, key_padding_mask=kpm_t,
                              attn_mask=am_t, causal=True)
    refs = oracle.attention_bwd(q.cpu(), k.cpu(), v.cpu(), g.cpu(), causal=True, kpm=kpm, am=am, q_pos0=q_off,
                                k_pos0=k_off)[:3]
    check(grads, refs, "f32", "block masks")
    assert torch.all(grads[0][:, :, 5] == 0)


def test_key_blocks_add_up_to_the_full_gradient():
    """The page's per-step backward: each key block's gradients with the whole
    rows' out and lse; dq accumulates over the blocks, each block owns its dk, dv."""
    B, H, L, d = 1, 2, 260, 64
    q, k, v = (rand((B, H, L, d), torch.float32, 20 + i) for i in range(3))
    g = rand((B, H, L, d), torch.float32, 23)
    out, lse = ba.ring_attn_fwd(q, k, v, P=1, causal=True, out_dtype=torch.float32)
    cut = 97
    dq = torch.zeros_like(q)
    dk = torch.empty_like(k)
    dv = torch.empty_like(v)
    for k0, k1 in ((cut, L), (0, cut)):   # any order
        dk_b = torch.zeros((B, H, k1 - k0, d), device="cuda")
        dv_b = torch.zeros_like(dk_b)
        ba.attn_block_bwd(q, k[:, :, k0:k1].contiguous(), v[:, :, k0:k1].contiguous(), out, g, lse, k_off=k0,
                          causal=True, dq=dq, dk=dk_b, dv=dv_b, accumulate=True)
        dk[:, :, k0:k1] = dk_b
        dv[:, :, k0:k1] = dv_b
    refs = oracle.attention_bwd(q.cpu(), k.cpu(), v.cpu(), g.cpu(), causal=True)[:3]
    check((dq, dk, dv), refs, "f32", "key blocks")


@pytest.mark.parametrize("T,P,part", [(1000, 4, "zigzag"), (1000, 4, "contiguous"), (384, 3, "zigzag"),
                                      (512, 1, "contiguous"), (96, 2, "zigzag")])
@pytest.mark.parametrize("mode", ["fused", "stepwise"])
def test_ring_backward(T, P, part, mode):
    B, H, d = 1, 2, 128
    q, k, v = rand((B, H, T, d), torch.bfloat16, 30, 0.5), rand((B, H, T, d), torch.bfloat16, 31, 0.5), \
        rand((B, H, T, d), torch.bfloat16, 32)
    g = rand((B, H, T, d), torch.bfloat16, 33)
    out, lse = ba.ring_attn_fwd(q, k, v, P=P, partition=part, causal=True)
    grads = ba.ring_attn_bwd(q, k, v, out, g, lse, P=P, partition=part, mode=mode, causal=True)
    refs = oracle.attention_bwd(q.float().cpu(), k.float().cpu(), v.float().cpu(), g.float().cpu(),
                                causal=True)[:3]
    check(grads, refs, "bf16", f"ring T={T} P={P} {part} {mode}")


def test_ring_backward_fp32_stepwise_equals_fused():
    """Both ring modes cover every (query, key) pair once; in fp32 they agree with
    the oracle to 1e-4 and with each other to rounding of the summation order."""
    B, H, T, d, P = 2, 2, 640, 64, 4
    q, k, v = (rand((B, H, T, d), torch.float32, 40 + i) for i in range(3))
    g = rand((B, H, T, d), torch.float32, 43)
    out, lse = ba.ring_attn_fwd(q, k, v, P=P, partition="zigzag", causal=True)
    fused = ba.ring_attn_bwd(q, k, v, out, g, lse, P=P, partition="zigzag", mode="fused", causal=True)
    step = ba.ring_attn_bwd(q, k, v, out, g, lse, P=P, partition="zigzag", mode="stepwise", causal=True)
    refs = oracle.attention_bwd(q.cpu(), k.cpu(), v.cpu(), g.cpu(), causal=True)[:3]
    check(fused, refs, "f32", "ring fp32 fused")
    check(step, refs, "f32", "ring fp32 stepwise")
