"""attn_block_fwd_noalloc, the entry point for callers that cannot allocate
device memory (hosts that own every device allocation, or run under a hard
memory budget): same results as attn_block_fwd on two calls in a row, and a
clear error beyond its fixed scratch.  Kept in a file that pytest collects
last; it passes alone in a fresh process and after the other tests."""
import math

import numpy as np
import pytest
import torch

import oracle
import blockwise_attention_gb300 as ba
from blockwise_attention_gb300 import _lib
from tests.parity import TOL_LSE, TOL_OUT, compare

pytestmark = pytest.mark.gpu


def _inputs(B, H, Lq, Lk, d, seed, dtype=torch.bfloat16):
    g = torch.Generator(device="cuda").manual_seed(seed)
    q = torch.randn((B, H, Lq, d), generator=g, device="cuda").to(dtype)
    k = torch.randn((B, H, Lk, d), generator=g, device="cuda").to(dtype)
    v = torch.randn((B, H, Lk, d), generator=g, device="cuda").to(dtype)
    rng = np.random.default_rng(seed)
    kpm = np.zeros((B, Lk), np.uint8)
    for b in range(B):
        kpm[b, rng.integers(Lk // 2, Lk + 1):] = 1
    # attn_mask rows are global query positions q_off + i with q_off = Lk - Lq
    am = (rng.random((Lk, Lk)) < 0.2).astype(np.uint8)
    am[:, 200:330] = 1          # a fully excluded key band: EMPTY tiles
    am[Lk - Lq + 7, :] = 1      # local row 7 sees nothing
    return q, k, v, torch.from_numpy(kpm).cuda(), torch.from_numpy(am).cuda()


def _check_same(out_n, lse_n, out_r, lse_r, dt="bf16"):
    o_n, o_r = out_n.float().cpu().numpy(), out_r.float().cpu().numpy()
    l_n, l_r = lse_n.cpu().numpy(), lse_r.cpu().numpy()
    fin = np.isfinite(l_r)
    assert np.array_equal(fin, np.isfinite(l_n))
    assert np.max(np.abs(o_n - o_r)) <= TOL_OUT[dt]
    assert np.max(np.abs(l_n[fin] - l_r[fin])) <= TOL_LSE


def _oracle(q, k, v, **kw):
    return oracle.attention(q.float().cpu(), k.float().cpu(), v.float().cpu(), **kw)


def test_noalloc_matches_attn_block_fwd_on_two_calls():
    # two calls in a row with different shapes: the second call's tile-class map is
    # smaller and differently laid out, so stale entries from the first would show
    for (B, H, Lq, Lk, causal, seed) in [(3, 4, 400, 520, True, 11), (2, 2, 300, 333, False, 12)]:
        q, k, v, kpm, am = _inputs(B, H, Lq, Lk, 128, seed)
        out_r, lse_r = ba.attn_block_fwd(q, k, v, q_off=Lk - Lq, key_padding_mask=kpm, attn_mask=am,
                                         causal=causal)
        out_n = torch.empty_like(out_r)
        lse_n = torch.empty_like(lse_r)
        ba.attn_block_fwd_noalloc(q, k, v, out_n, lse_n, q_off=Lk - Lq, key_padding_mask=kpm, attn_mask=am,
                                  causal=causal)
        torch.cuda.synchronize()
        assert ba.sync_status() == 0
        _check_same(out_n, lse_n, out_r, lse_r)
        assert torch.all(lse_n[:, :, 7] == -math.inf)
        # and against the fp64 oracle on the same inputs
        o_ref, l_ref = _oracle(q, k, v, causal=causal, kpm=kpm.cpu().numpy(), am=am.cpu().numpy(),
                               q_pos0=Lk - Lq)
        compare(out_n, lse_n, o_ref, l_ref, "bf16", f"noalloc B={B} Lq={Lq} Lk={Lk} causal={causal}")


@pytest.mark.parametrize("dt,d", [("f32", 64), ("bf16", 32), ("f32", 16)])
def test_noalloc_cuda_core_path(dt, d):
    """fp32 inputs and bf16 with d = 32 run on the CUDA-core kernel, which reads
    the same fixed tile-class array; two calls in a row, masked then masked
    with other shapes, against attn_block_fwd and the oracle."""
    dtype = torch.float32 if dt == "f32" else torch.bfloat16
    for (B, H, Lq, Lk, causal, seed) in [(2, 3, 260, 390, True, 21), (3, 2, 140, 333, False, 22)]:
        q, k, v, kpm, am = _inputs(B, H, Lq, Lk, d, seed, dtype)
        out_r, lse_r = ba.attn_block_fwd(q, k, v, q_off=Lk - Lq, key_padding_mask=kpm, attn_mask=am,
                                         causal=causal, out_dtype=torch.float32)
        out_n = torch.empty_like(out_r)
        lse_n = torch.empty_like(lse_r)
        ba.attn_block_fwd_noalloc(q, k, v, out_n, lse_n, q_off=Lk - Lq, key_padding_mask=kpm, attn_mask=am,
                                  causal=causal)
        torch.cuda.synchronize()
        assert ba.sync_status() == 0
        _check_same(out_n, lse_n, out_r, lse_r, dt)
        o_ref, l_ref = _oracle(q, k, v, causal=causal, kpm=kpm.cpu().numpy(), am=am.cpu().numpy(),
                               q_pos0=Lk - Lq)
        compare(out_n, lse_n, o_ref, l_ref, dt, f"noalloc {dt} d={d} causal={causal}")


def test_noalloc_without_masks_and_accumulate():
    """Causal without masks (no class map: the kernel deals work items
    round-robin), then a second key block merged into the first with
    accumulate=1 into an fp32 out; both against attn_block_fwd and the oracle."""
    B, H, Lq, d = 2, 4, 384, 128
    q, k, v, _, _ = _inputs(B, H, Lq, 700, d, 31)
    k0, v0, k1, v1 = k[:, :, :316], v[:, :, :316], k[:, :, 316:], v[:, :, 316:]
    q_off = 700 - Lq
    out_r, lse_r = ba.attn_block_fwd(q, k0, v0, q_off=q_off, causal=True, out_dtype=torch.float32)
    out_n = torch.empty_like(out_r)
    lse_n = torch.empty_like(lse_r)
    ba.attn_block_fwd_noalloc(q, k0, v0, out_n, lse_n, q_off=q_off, causal=True)
    torch.cuda.synchronize()
    _check_same(out_n, lse_n, out_r, lse_r)
    ba.attn_block_fwd(q, k1, v1, q_off=q_off, k_off=316, causal=True, out=out_r, lse=lse_r, accumulate=True)
    ba.attn_block_fwd_noalloc(q, k1, v1, out_n, lse_n, q_off=q_off, k_off=316, causal=True, accumulate=True)
    torch.cuda.synchronize()
    assert ba.sync_status() == 0
    _check_same(out_n, lse_n, out_r, lse_r)
    o_ref, l_ref = _oracle(q, k, v, causal=True, q_pos0=q_off)
    compare(out_n, lse_n, o_ref, l_ref, "bf16", "noalloc causal + accumulate")


def test_noalloc_rejects_sizes_beyond_its_scratch():
    # 70 x 128 x 128 tile pairs = 1,146,880 class bytes > 1 MiB
    B, H, L, d = 70, 1, 128 * 128, 64
    assert B * (L // 128) * (L // 128) > _lib.BA_NOALLOC_MAX_CLASS_BYTES
    q = torch.zeros((1, 1, 8, d), dtype=torch.bfloat16, device="cuda")
    kpm = torch.zeros((B, L), dtype=torch.uint8, device="cuda")
    lib = ba.load()
    t = _lib.ba_tensor(q.data_ptr(), 0, 0, d)
    rc = lib.attn_block_fwd_noalloc(t, t, t, B, H, L, L, d, _lib.BA_BF16, 0, 0, _lib.ctypes.c_void_p(kpm.data_ptr()),
                                    L, None, 0, 0, 0.0, _lib.ctypes.c_void_p(q.data_ptr()), _lib.BA_BF16,
                                    _lib.ctypes.c_void_p(q.data_ptr()), 0, None)
    assert rc == _lib.BA_ERR_NOALLOC_LIMIT
    assert b"no-allocation" in lib.ba_strerror(rc)
