"""Striped partitions (rank r holds tokens r, r + P, r + 2P, ...; Striped
Attention, named in brunomaga "When to use Ulysses and Ring attention") through
ring_attn_fwd against the fp64 oracle.  The partition and the ring order do not
change the result: every configuration must reach plain attention over the
whole sequence, in both ring modes, on the tensor-core path (bf16, d = 64 / 128)
and on the CUDA-core path (fp32, bf16 d = 32)."""
import numpy as np
import pytest
import torch

import oracle
import blockwise_attention_gb300 as ba
from blockwise_attention_gb300.workloads import WORKLOADS, make_inputs
from tests.parity import compare, oracle_ring_reference, sample_rows

pytestmark = pytest.mark.gpu


def rand(shape, dtype, seed, std=1.0):
    g = torch.Generator(device="cuda").manual_seed(seed)
    return (torch.randn(shape, generator=g, device="cuda") * std).to(dtype)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("mode", ["fused", "stepwise"])
def test_tiny_ring_f32_striped(causal, mode):
    w = WORKLOADS["tiny_ring_f32"].replace(causal=causal, partition="striped")
    inp = make_inputs(w, "cuda")
    out, lse, tok, sch = ba.ring_attn_fwd(inp.q, inp.k, inp.v, P=w.P, partition="striped", mode=mode,
                                          causal=causal, return_index_maps=True)
    assert np.array_equal(tok, oracle.partition(w.T, w.P, "striped"))
    assert tok[1].tolist() == [1, 5]
    assert sch[0].tolist() == [0, 3, 2, 1]
    o_ref, l_ref = oracle_ring_reference(inp, w)
    compare(out, lse, o_ref, l_ref, "f32", f"tiny striped causal={causal} {mode}")


@pytest.mark.parametrize("mode", ["fused", "stepwise"])
def test_striped_prefill_8k(mode):
    """The 8K prefill workload (B=4, H=16, d=128, causal) over P=8 striped ranks."""
    w = WORKLOADS["zigzag_prefill_8k"].replace(partition="striped")
    inp = make_inputs(w, "cuda")
    out, lse = ba.ring_attn_fwd(inp.q, inp.k, inp.v, P=w.P, partition="striped", mode=mode, causal=True)
    heads = [(0, 1), (1, 9), (2, 14), (3, 0)]
    rows_r = sample_rows(len(heads), 1, w.T, [(i, 0) for i in range(len(heads))], 256, w.T // w.P, seed=3)
    # rows next to every rank boundary of the striping: tokens r + P u for the first and last u
    o_ref, l_ref = oracle_ring_reference(inp, w, rows=rows_r, heads=heads)
    sel = torch.from_numpy(rows_r).cuda()
    sel_o = torch.stack([out[b, h] for b, h in heads]).reshape(-1, w.d)[sel]
    sel_l = torch.stack([lse[b, h] for b, h in heads]).reshape(-1)[sel]
    compare(sel_o, sel_l, o_ref, l_ref, "bf16", f"striped_prefill_8k {mode}")
    # the same bits as the zigzag partition would be too strong (sums run in another
    # order); the two partitions must agree to the bf16 tolerance on every row
    out_z, lse_z = ba.ring_attn_fwd(inp.q, inp.k, inp.v, P=w.P, partition="zigzag", mode="fused", causal=True)
    assert torch.max(torch.abs(out.float() - out_z.float())).item() <= 2e-2
    assert torch.max(torch.abs(lse - lse_z)).item() <= 1e-5


@pytest.mark.parametrize("T,P,d,causal", [(1000, 4, 128, True), (1000, 4, 64, True), (384, 3, 128, False),
                                          (96, 2, 128, True), (2048, 16, 64, True), (640, 1, 128, True)])
@pytest.mark.parametrize("mode", ["fused", "stepwise"])
def test_striped_ragged(T, P, d, causal, mode):
    """Ranks whose token count is not a multiple of 128 (ragged last tiles), P that
    is not a power of two, P = 1, and ranks of 128 tokens."""
    B, H = 2, 2
    q, k, v = (rand((B, H, T, d), torch.bfloat16, 40 + i) for i in range(3))
    out, lse = ba.ring_attn_fwd(q, k, v, P=P, partition="striped", mode=mode, causal=causal)
    o_ref, l_ref = oracle.attention(q.float().cpu(), k.float().cpu(), v.float().cpu(), causal=causal)
    compare(out, lse, o_ref, l_ref, "bf16", f"striped T={T} P={P} d={d} causal={causal} {mode}")


@pytest.mark.parametrize("dt,d", [("f32", 64), ("bf16", 32), ("f32", 16)])
def test_striped_cuda_core_path(dt, d):
    B, H, T, P = 1, 3, 600, 5
    dtype = torch.float32 if dt == "f32" else torch.bfloat16
    q, k, v = (rand((B, H, T, d), dtype, 50 + i) for i in range(3))
    for mode in ("fused", "stepwise"):
        out, lse = ba.ring_attn_fwd(q, k, v, P=P, partition="striped", mode=mode, causal=True,
                                    out_dtype=torch.float32)
        o_ref, l_ref = oracle.attention(q.float().cpu(), k.float().cpu(), v.float().cpu(), causal=True)
        compare(out, lse, o_ref, l_ref, dt, f"striped {dt} d={d} {mode}")


def test_striped_rope_and_strided_inputs():
    """RoPE inside the call (rotated copies addressed through the striped view),
    and Q/K/V handed over as (B, T, H, d) storage."""
    B, T, H, d, P = 2, 1024, 4, 128, 4
    base = [rand((B, T, H, d), torch.bfloat16, 60 + i) for i in range(3)]
    q, k, v = [x.permute(0, 2, 1, 3) for x in base]
    out, lse = ba.ring_attn_fwd(q, k, v, P=P, partition="striped", causal=True, rope=True, rope_base=10000.0)
    qr = torch.from_numpy(oracle.rope(q.float().cpu(), base=10000.0, round_to="bf16"))
    kr = torch.from_numpy(oracle.rope(k.float().cpu(), base=10000.0, round_to="bf16"))
    o_ref, l_ref = oracle.attention(qr, kr, v.float().cpu(), causal=True)
    compare(out, lse, o_ref, l_ref, "bf16", "striped rope strided")
    out2, lse2 = ba.ring_attn_fwd(q, k, v, P=P, partition="striped", causal=False)
    o_ref, l_ref = oracle.attention(q.float().cpu(), k.float().cpu(), v.float().cpu(), causal=False)
    compare(out2, lse2, o_ref, l_ref, "bf16", "striped strided non-causal")


def test_striped_refuses_masks():
    B, H, T, d = 1, 1, 256, 64
    q = rand((B, H, T, d), torch.bfloat16, 70)
    kpm = torch.zeros((B, T), dtype=torch.uint8, device="cuda")
    with pytest.raises(ba.BlockAttnError) as e:
        ba.ring_attn_fwd(q, q, q, P=2, partition="striped", key_padding_mask=kpm)
    assert e.value.code == -5
