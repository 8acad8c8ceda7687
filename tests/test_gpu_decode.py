"""GPU parity of decode attention with a split KV cache (attn_decode_fwd): one
query per (b, h) against a ragged cache, checked against the oracle (plain
attention with the cache lengths as key padding), and against folding
attn_merge pairwise over per-split partial attentions."""
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


def kpm_from(lengths, S):
    kpm = np.zeros((len(lengths), S), np.uint8)
    for b, n in enumerate(lengths):
        kpm[b, max(0, min(n, S)):] = 1
    return kpm


@pytest.mark.parametrize("dt,d", [("bf16", 128), ("bf16", 64), ("f32", 64), ("bf16", 16), ("f32", 128)])
@pytest.mark.parametrize("splits", [0, 1, 7])
def test_decode_against_oracle(dt, d, splits):
    dtype = torch.bfloat16 if dt == "bf16" else torch.float32
    B, H, S = 4, 3, 5000
    lengths = [5000, 1, 3333, 0]
    q = rand((B, H, 1, d), dtype, 1)
    k, v = rand((B, H, S, d), dtype, 2), rand((B, H, S, d), dtype, 3)
    lens = torch.tensor(lengths, dtype=torch.int32, device="cuda")
    out, lse = ba.attn_decode_fwd(q, k, v, lengths=lens, num_splits=splits, out_dtype=torch.float32)
    o_ref, l_ref = oracle.attention(q.float().cpu(), k.float().cpu(), v.float().cpu(), kpm=kpm_from(lengths, S))
    compare(out, lse, o_ref, l_ref, "f32" if dt == "f32" else "bf16", f"decode {dt} d={d} splits={splits}")
    assert torch.all(lse[3] == -float("inf")) and torch.all(out[3] == 0)


def test_decode_strided_cache_and_bf16_out():
    """A cache held as (B, S, H, d) storage and viewed as (B, H, S, d)."""
    B, H, S, d = 2, 4, 3000, 128
    kb, vb = rand((B, S, H, d), torch.bfloat16, 4), rand((B, S, H, d), torch.bfloat16, 5)
    k, v = kb.permute(0, 2, 1, 3), vb.permute(0, 2, 1, 3)
    q = rand((B, H, 1, d), torch.bfloat16, 6)
    out, lse = ba.attn_decode_fwd(q, k, v)
    o_ref, l_ref = oracle.attention(q.float().cpu(), k.float().cpu(), v.float().cpu())
    compare(out, lse, o_ref, l_ref, "bf16", "decode strided")


def test_pairwise_attn_merge_of_splits_equals_decode():
    """The decode combine is the LSE merge of attn_merge applied to all splits at
    once: folding attn_merge over per-split attn_block_fwd partials agrees."""
    B, H, S, d, n = 2, 2, 2000, 64, 5
    q = rand((B, H, 1, d), torch.float32, 7)
    k, v = rand((B, H, S, d), torch.float32, 8), rand((B, H, S, d), torch.float32, 9)
    out, lse = ba.attn_decode_fwd(q, k, v, num_splits=n, out_dtype=torch.float32)
    cut = [round(S * i / n) for i in range(n + 1)]
    acc_o, acc_l = None, None
    for i in range(n):
        o_i, l_i = ba.attn_block_fwd(q, k[:, :, cut[i]:cut[i + 1]].contiguous(), v[:, :, cut[i]:cut[i + 1]].contiguous(),
                                     out_dtype=torch.float32)
        if acc_o is None:
            acc_o, acc_l = o_i.clone(), l_i.clone()
        else:
            ba.attn_merge(acc_o, acc_l, o_i, l_i)
    assert torch.allclose(acc_o, out, atol=1e-5, rtol=0) and torch.allclose(acc_l, lse, atol=1e-5, rtol=0)
    o_ref, l_ref = oracle.attention(q.cpu(), k.cpu(), v.cpu())
    compare(out, lse, o_ref, l_ref, "f32", "decode vs merged splits")


def test_decode_full_size_sampled():
    """The decode measurement workload: B=8, H=32, a 65536-slot bf16 cache with
    lengths drawn in [32768, 65536]; four (b, h) pairs against the oracle."""
    from blockwise_attention_gb300.workloads import make_decode_inputs
    inp = make_decode_inputs("cuda")
    out, lse = ba.attn_decode_fwd(inp.q, inp.k, inp.v, lengths=inp.lengths, out_dtype=torch.float32)
    lengths = inp.lengths.cpu().tolist()
    for b, h in ((0, 0), (3, 17), (5, 31), (7, 8)):
        sl = (slice(b, b + 1), slice(h, h + 1))
        o_ref, l_ref = oracle.attention(inp.q[sl].float().cpu(), inp.k[sl].float().cpu(), inp.v[sl].float().cpu(),
                                        kpm=kpm_from([lengths[b]], inp.k.shape[2]))
        compare(out[sl], lse[sl], o_ref, l_ref, "bf16", f"decode full b={b} h={h}")
