"""GPU edge cases of the C ABI against the oracle: ragged tails, partial chunks,
blocks at offsets, accumulate mode and merge, fully masked rows, strided
(B, T, H, d) inputs, P = 1, empty inputs, bit-exact RoPE and tile classes,
and the bounded-wait error path."""
import math

import numpy as np
import pytest
import torch

import oracle
import blockwise_attention_gb300 as ba
from tests.parity import compare

pytestmark = pytest.mark.gpu


def rand(shape, dtype, seed, std=1.0):
    g = torch.Generator(device="cuda").manual_seed(seed)
    return (torch.randn(shape, generator=g, device="cuda") * std).to(dtype)


DT = {"bf16": torch.bfloat16, "f32": torch.float32}


@pytest.mark.parametrize("dt,d", [("bf16", 128), ("bf16", 64), ("bf16", 32), ("bf16", 16), ("f32", 64),
                                  ("f32", 128)])
@pytest.mark.parametrize("causal", [False, True])
def test_block_ragged_offsets(dt, d, causal):
    """Lq, Lk not multiples of 128; the block sits at global offsets."""
    B, H, Lq, Lk = 2, 3, 300, 333
    q, k, v = rand((B, H, Lq, d), DT[dt], 1), rand((B, H, Lk, d), DT[dt], 2), rand((B, H, Lk, d), DT[dt], 3)
    q_off, k_off = 40, 0  # queries 40..339 against keys 0..332
    out, lse = ba.attn_block_fwd(q, k, v, q_off=q_off, k_off=k_off, causal=causal, out_dtype=torch.float32)
    o_ref, l_ref = oracle.attention(q.float().cpu(), k.float().cpu(), v.float().cpu(), causal=causal,
                                    q_pos0=q_off, k_pos0=k_off)
    compare(out, lse, o_ref, l_ref, dt, f"block {dt} d={d} causal={causal}")


@pytest.mark.parametrize("dt,d", [("bf16", 128), ("bf16", 64), ("f32", 64)])
@pytest.mark.parametrize("causal", [False, True])
def test_block_masks_at_offsets(dt, d, causal):
    """attn_block_fwd with key padding and attn_mask indexed at global positions."""
    B, H, Lq, Lk, q_off, k_off = 2, 3, 260, 300, 140, 100
    q, k, v = rand((B, H, Lq, d), DT[dt], 60), rand((B, H, Lk, d), DT[dt], 61), rand((B, H, Lk, d), DT[dt], 62)
    rng = np.random.default_rng(1)
    kpm = (rng.random((B, k_off + Lk)) < 0.2).astype(np.uint8)
    am = (rng.random((q_off + Lq, k_off + Lk)) < 0.3).astype(np.uint8)
    am[q_off + 9, :] = 1                   # local row 9 sees nothing
    am[:, k_off + 128:k_off + 256] = 1     # an EMPTY key tile
    kpm_t, am_t = torch.from_numpy(kpm).cuda(), torch.from_numpy(am).cuda()
    out, lse = ba.attn_block_fwd(q, k, v, q_off=q_off, k_off=k_off, key_padding_mask=kpm_t, attn_mask=am_t,
                                 causal=causal, out_dtype=torch.float32)
    o_ref, l_ref = oracle.attention(q.float().cpu(), k.float().cpu(), v.float().cpu(), causal=causal, kpm=kpm,
                                    am=am, q_pos0=q_off, k_pos0=k_off)
    compare(out, lse, o_ref, l_ref, dt, f"block masks {dt} d={d} causal={causal}")
    assert torch.all(lse[:, :, 9] == -math.inf)


@pytest.mark.parametrize("T,P,part", [(1000, 4, "zigzag"), (1000, 4, "contiguous"), (384, 3, "zigzag"),
                                      (640, 1, "contiguous"), (96, 2, "zigzag")])
@pytest.mark.parametrize("mode", ["fused", "stepwise"])
def test_ring_ragged_chunks(T, P, part, mode):
    B, H, d = 1, 2, 128
    q, k, v = rand((B, H, T, d), torch.bfloat16, 4), rand((B, H, T, d), torch.bfloat16, 5), \
        rand((B, H, T, d), torch.bfloat16, 6)
    out, lse = ba.ring_attn_fwd(q, k, v, P=P, partition=part, mode=mode, causal=True)
    o_ref, l_ref = oracle.attention(q.float().cpu(), k.float().cpu(), v.float().cpu(), causal=True)
    compare(out, lse, o_ref, l_ref, "bf16", f"ring T={T} P={P} {part} {mode}")


@pytest.mark.parametrize("dt", ["bf16", "f32"])
def test_accumulate_over_key_blocks_and_merge(dt):
    """Keys in three blocks folded with accumulate=1, and two halves merged with
    attn_merge, both equal attention over all keys."""
    B, H, L, S, d = 2, 2, 200, 390, 64
    q, k, v = rand((B, H, L, d), DT[dt], 7), rand((B, H, S, d), DT[dt], 8), rand((B, H, S, d), DT[dt], 9)
    o_ref, l_ref = oracle.attention(q.float().cpu(), k.float().cpu(), v.float().cpu(), causal=True, q_pos0=S - L)
    out = torch.zeros((B, H, L, d), dtype=torch.float32, device="cuda")
    lse = torch.full((B, H, L), -math.inf, device="cuda")
    for a, b in [(0, 130), (130, 131), (131, 390)]:   # includes a single-key block
        ba.attn_block_fwd(q, k[:, :, a:b], v[:, :, a:b], q_off=S - L, k_off=a, causal=True, out=out, lse=lse,
                          accumulate=True)
    compare(out, lse, o_ref, l_ref, dt, f"accumulate {dt}")
    oa, la = ba.attn_block_fwd(q, k[:, :, :256], v[:, :, :256], q_off=S - L, causal=True, out_dtype=torch.float32)
    ob, lb = ba.attn_block_fwd(q, k[:, :, 256:], v[:, :, 256:], q_off=S - L, k_off=256, causal=True,
                               out_dtype=torch.float32)
    ba.attn_merge(oa, la, ob, lb)
    compare(oa, la, o_ref, l_ref, dt, f"merge {dt}")


def test_merge_kernel_against_oracle_merge():
    g = torch.Generator(device="cuda").manual_seed(3)
    rows, d = 5000, 128
    oa = torch.randn((rows, d), generator=g, device="cuda")
    ob = torch.randn((rows, d), generator=g, device="cuda")
    la = torch.randn((rows,), generator=g, device="cuda") * 5
    lb = torch.randn((rows,), generator=g, device="cuda") * 5
    la[::7] = -math.inf
    lb[::11] = -math.inf
    ref_o, ref_l = oracle.merge(oa.cpu().numpy(), la.cpu().numpy(), ob.cpu().numpy(), lb.cpu().numpy())
    ba.attn_merge(oa, la, ob, lb)
    l = la.cpu().numpy()
    fin = np.isfinite(ref_l)
    assert np.array_equal(fin, np.isfinite(l))
    assert np.max(np.abs(l[fin] - ref_l[fin])) < 1e-5
    assert np.max(np.abs(oa.cpu().numpy() - ref_o)) < 1e-5


@pytest.mark.parametrize("dt,d", [("bf16", 128), ("bf16", 64), ("f32", 32)])
def test_fully_masked_rows_and_masks(dt, d):
    B, H, T = 2, 2, 300
    q, k, v = rand((B, H, T, d), DT[dt], 10), rand((B, H, T, d), DT[dt], 11), rand((B, H, T, d), DT[dt], 12)
    rng = np.random.default_rng(0)
    am = (rng.random((T, T)) < 0.3).astype(np.uint8)
    am[5, :] = 1          # row 5 sees nothing
    am[200:260, :] = 1    # a band of rows that see nothing
    am[:, 130:256] = 1    # a fully excluded key tile
    kpm = np.zeros((B, T), np.uint8)
    kpm[1, 150:] = 1
    am_t, kpm_t = torch.from_numpy(am).cuda(), torch.from_numpy(kpm).cuda()
    out, lse = ba.ring_attn_fwd(q, k, v, P=2, partition="contiguous", attn_mask=am_t, key_padding_mask=kpm_t,
                                out_dtype=torch.float32)
    o_ref, l_ref = oracle.attention(q.float().cpu(), k.float().cpu(), v.float().cpu(), kpm=kpm, am=am)
    compare(out, lse, o_ref, l_ref, dt, f"masks {dt} d={d}")
    assert torch.all(out[:, :, 5] == 0) and torch.all(lse[:, :, 5] == -math.inf)
    cls = ba.tile_classes(B, T, T, key_padding_mask=kpm_t, attn_mask=am_t, causal=True).cpu().numpy()
    assert np.array_equal(cls, oracle.tile_classes(B, T, T, kpm=kpm, am=am, causal=True))


def test_strided_flash_layout():
    """Q/K/V handed over as (B, T, H, d) storage viewed as (B, H, T, d)."""
    B, T, H, d = 2, 520, 4, 128
    base = [rand((B, T, H, d), torch.bfloat16, 20 + i) for i in range(3)]
    q, k, v = [x.permute(0, 2, 1, 3) for x in base]
    assert not q.is_contiguous()
    out, lse = ba.ring_attn_fwd(q, k, v, P=4, partition="zigzag", causal=True)
    o_ref, l_ref = oracle.attention(q.float().cpu(), k.float().cpu(), v.float().cpu(), causal=True)
    compare(out, lse, o_ref, l_ref, "bf16", "strided")


def test_empty_inputs():
    q = torch.empty((1, 2, 0, 64), dtype=torch.bfloat16, device="cuda")
    out, lse = ba.ring_attn_fwd(q, q, q, P=1)
    assert out.numel() == 0 and lse.numel() == 0
    q = rand((1, 1, 8, 64), torch.bfloat16, 30)
    kz = torch.empty((1, 1, 0, 64), dtype=torch.bfloat16, device="cuda")
    out, lse = ba.attn_block_fwd(q, kz, kz, out_dtype=torch.float32)
    assert torch.all(out == 0) and torch.all(lse == -math.inf)


@pytest.mark.parametrize("dt,d", [("bf16", 128), ("bf16", 64), ("bf16", 16), ("bf16", 6), ("f32", 128),
                                  ("f32", 10)])
def test_rope_bit_exact(dt, d):
    B, H, T = 2, 3, 777
    x = rand((B, H, T, d), DT[dt], 40)
    x2 = rand((B, H, T, d), DT[dt], 41, std=3.0)
    y = ba.rope_apply(x, base=10000.0)
    ref = oracle.rope(x.float().cpu(), base=10000.0, round_to=dt)
    assert np.array_equal(y.float().cpu().numpy(), ref)
    pos = torch.arange(T, dtype=torch.int32, device="cuda") * 37 + 5
    y1, y2 = ba.rope_apply(x, x2=x2, base=500000.0, positions=pos)
    for xi, yi in ((x, y1), (x2, y2)):
        ref2 = oracle.rope(xi.float().cpu(), base=500000.0, positions=pos.cpu().numpy(), round_to=dt)
        assert np.array_equal(yi.float().cpu().numpy(), ref2)


def test_rope_strided_and_large_positions():
    """Strided (B, T, H, d) input; positions up to 2^20, where angles are large."""
    B, T, H, d = 1, 300, 4, 128
    base = rand((B, T, H, d), torch.bfloat16, 42)
    x = base.permute(0, 2, 1, 3)
    pos = torch.randint(0, 1 << 20, (T,), dtype=torch.int32, device="cuda")
    y = ba.rope_apply(x, base=10000.0, positions=pos)
    ref = oracle.rope(x.float().cpu(), base=10000.0, positions=pos.cpu().numpy(), round_to="bf16")
    assert np.array_equal(y.float().cpu().numpy(), ref)


def test_bounded_wait_reports_timeout():
    assert ba.sync_status() == 0
    ba.debug_wait_timeout(50_000_000)   # 50 ms on an mbarrier nothing completes
    assert ba.sync_status() == -4       # BA_ERR_TIMEOUT, context still usable
    assert ba.sync_status() == 0
    q = rand((1, 1, 128, 64), torch.bfloat16, 50)
    out, lse = ba.ring_attn_fwd(q, q, q, P=1)
    torch.cuda.synchronize()
    assert torch.isfinite(out.float()).all()


@pytest.mark.parametrize("mode", ["fused", "stepwise"])
def test_workspace_reuse_and_alignment(mode):
    """A caller's workspace holds the item counters the kernel claims work from:
    they are re-zeroed by every call, so one buffer serves call after call, and a
    workspace off a 256-byte boundary is refused before anything is launched."""
    B, H, T, d, P = 1, 3, 1024, 128, 4
    need = ba.ring_attn_fwd_workspace_size(B, H, T, d, torch.bfloat16, P, "zigzag", mode)
    assert need >= 256
    ws = torch.empty(need + 512, dtype=torch.uint8, device="cuda")
    ws.fill_(0xA5)   # counters start from garbage: the call must clear them
    for seed in (70, 80):
        q, k, v = (rand((B, H, T, d), torch.bfloat16, seed + i) for i in range(3))
        out, lse = ba.ring_attn_fwd(q, k, v, P=P, partition="zigzag", mode=mode, causal=True, workspace=ws)
        o_ref, l_ref = oracle.attention(q.float().cpu(), k.float().cpu(), v.float().cpu(), causal=True)
        compare(out, lse, o_ref, l_ref, "bf16", f"workspace reuse {mode} seed={seed}")
    with pytest.raises(ba.BlockAttnError):
        ba.ring_attn_fwd(q, k, v, P=P, partition="zigzag", mode=mode, causal=True, workspace=ws[16:])
    out, lse = ba.attn_block_fwd(q, k, v, causal=True, workspace=ws, out_dtype=torch.float32)
    o_ref, l_ref = oracle.attention(q.float().cpu(), k.float().cpu(), v.float().cpu(), causal=True)
    compare(out, lse, o_ref, l_ref, "bf16", "block with caller workspace")


@pytest.mark.parametrize("dt,d", [("bf16", 128), ("bf16", 6), ("f32", 64)])
@pytest.mark.parametrize("scale", [0.25, float(np.float32(0.3)), 0.125])
def test_rope_position_interpolation_bit_exact(dt, d, scale):
    """Position Interpolation: the position index times pos_scale before the angle;
    bit-exact against the fp64 oracle rounded once (the scale as the ABI's fp32)."""
    B, H, T = 2, 3, 500
    x = rand((B, H, T, d), DT[dt], 60)
    pos = torch.arange(T, dtype=torch.int32, device="cuda") * 8 + 3
    y = ba.rope_apply(x, base=10000.0, positions=pos, pos_scale=scale)
    ref = oracle.rope(x.float().cpu(), base=10000.0, positions=pos.cpu().numpy(), round_to=dt, pos_scale=scale)
    assert np.array_equal(y.float().cpu().numpy(), ref)
    # scale 1/4 at positions 4m reproduces plain RoPE at m
    m = torch.arange(T, dtype=torch.int32, device="cuda")
    assert torch.equal(ba.rope_apply(x, positions=4 * m, pos_scale=0.25), ba.rope_apply(x, positions=m))


@pytest.mark.parametrize("d", [128, 64])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("ring", [False, True])
def test_growing_scores_rescale(d, causal, ring):
    """Scores that grow along the keys: the running maximum of a row moves by far
    more than the kernel's lazy threshold (2^8 in exp2 units) several times after
    the row's first key tile, so O and the sums are rescaled mid-row (the pages'
    online softmax: every new maximum rescales the weighted sum already held)."""
    B, H, T = 1, 2, 1024
    g = torch.Generator(device="cpu").manual_seed(77)
    q = torch.randn((B, H, T, d), generator=g) * 0.5
    k = torch.randn((B, H, T, d), generator=g) * 0.5
    v = torch.randn((B, H, T, d), generator=g)
    # a common direction that later keys follow more and more: the scores of the
    # last row run from about 0 to 14 (natural-log units) along the keys
    q[..., 0] = 4.0
    k[..., 0] = torch.linspace(0.0, 3.5 * math.sqrt(d), T).view(1, 1, T)
    q, k, v = (x.to(torch.bfloat16).cuda() for x in (q, k, v))
    if ring:
        out, lse = ba.ring_attn_fwd(q, k, v, P=4, partition="zigzag", causal=causal, out_dtype=torch.float32)
    else:
        out, lse = ba.attn_block_fwd(q, k, v, causal=causal, out_dtype=torch.float32)
    o_ref, l_ref = oracle.attention(q.float().cpu(), k.float().cpu(), v.float().cpu(), causal=causal)
    # the last row's maximum grows by more than twice the threshold across its tiles
    s_last = (q.float()[0, 0, -1] @ k.float()[0, 0].T) / math.sqrt(d) * 1.4426950408889634
    assert float(s_last[-128:].max() - s_last[:128].max()) > 2 * 8.0
    compare(out, lse, o_ref, l_ref, "bf16", f"growing scores d={d} causal={causal} ring={ring}")


# Score levels (exp2 units) of the keys of tile t, half h (64 keys each), for
# rescale_inside_tile: each places a jump where one branch of the tensor-core
# kernel's lazy rescale runs.  With the reference maximum m of the row taken on
# the first tile, a later half whose scores sit near m passes on the sum of its
# p; a half whose scores are 10 above m moves m (more than 2^8 above it), and
# one 4 above m has a sum of p over 2^8 but moves nothing.
LEVELS = {
    "first_half": lambda t, h: 10.0 * t,            # the jump at the start of each tile
    "second_half": lambda t, h: 10.0 * (t + h),     # the jump in the middle of each tile
    "sum_only_first": lambda t, h: 4.0 * t,
    "sum_only_second": lambda t, h: 4.0 * (t + h),
}


@pytest.mark.parametrize("case", sorted(LEVELS))
@pytest.mark.parametrize("d", [128, 64])
@pytest.mark.parametrize("causal", [False, True])
def test_rescale_inside_tile(case, d, causal):
    """Online softmax (brunomaga "Improving numerical stability"): the running
    maximum of a row moves inside a key tile, in its first or its second half of
    64 keys, or a half's probabilities sum past 2^8 with the maximum unmoved.
    The output must match the oracle whichever way the kernel splits the tile."""
    B, H, T = 1, 2, 384
    g = torch.Generator(device="cpu").manual_seed(91)
    q = torch.randn((B, H, T, d), generator=g) * 0.5
    k = torch.randn((B, H, T, d), generator=g) * 0.5
    v = torch.randn((B, H, T, d), generator=g)
    per_unit = 4.0 / math.sqrt(d) * 1.4426950408889634   # exp2 units of score per unit of k[..., 0]
    q[..., 0] = 4.0
    lev = torch.tensor([LEVELS[case](j // 128, (j % 128) // 64) for j in range(T)])
    k[..., 0] = (lev / per_unit).view(1, 1, T)
    q, k, v = (x.to(torch.bfloat16).cuda() for x in (q, k, v))
    out, lse = ba.attn_block_fwd(q, k, v, causal=causal, out_dtype=torch.float32)
    o_ref, l_ref = oracle.attention(q.float().cpu(), k.float().cpu(), v.float().cpu(), causal=causal)
    compare(out, lse, o_ref, l_ref, "bf16", f"rescale inside tile {case} d={d} causal={causal}")
