"""GPU checks of the Ulysses path: the all-to-all exchanges are bit-exact
permutations (compared with the oracle's layout maps), and Ulysses attention
equals plain attention (oracle) within the forward tolerances."""
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


def to_tok(x, P):
    """(B, H, T, d) -> token shards (P, H, B, T/P, d) (test-side reshaping)."""
    B, H, T, d = x.shape
    return x.permute(1, 0, 2, 3).reshape(H, B, P, T // P, d).permute(2, 0, 1, 3, 4).contiguous()


def from_tok(x):
    """(P, H, B, T/P, d) -> (B, H, T, d)."""
    P, H, B, Tl, d = x.shape
    return x.permute(1, 2, 0, 3, 4).reshape(H, B, P * Tl, d).permute(1, 0, 2, 3).contiguous()


@pytest.mark.parametrize("P,H,B,T,d,dtype", [(4, 8, 2, 64, 128, torch.bfloat16), (2, 2, 1, 4, 1, torch.float32),
                                             (3, 6, 2, 27, 3, torch.bfloat16), (8, 16, 1, 256, 64, torch.float32),
                                             (1, 5, 3, 10, 16, torch.bfloat16)])
def test_all_to_all_bit_exact(P, H, B, T, d, dtype):
    x = rand((P, H, B, T // P, d), dtype, 1)
    y = ba.ulysses_all_to_all(x, P, "token_to_head")
    ref = oracle.ulysses_token_to_head(x.float().cpu().numpy(), P)
    assert np.array_equal(y.float().cpu().numpy(), ref)
    z = ba.ulysses_all_to_all(y, P, "head_to_token")
    assert torch.equal(z, x)


@pytest.mark.parametrize("dt,d", [("bf16", 128), ("bf16", 64), ("f32", 64)])
@pytest.mark.parametrize("masks", ["causal", "pad_band"])
def test_ulysses_attention_equals_plain_attention(dt, d, masks):
    dtype = torch.bfloat16 if dt == "bf16" else torch.float32
    P, B, H, T = 4, 2, 8, 512
    q, k, v = (rand((B, H, T, d), dtype, 10 + i, 0.5) for i in range(3))
    kw, okw = {}, {}
    if masks == "causal":
        kw["causal"] = okw["causal"] = True
    else:
        lens = [T - 37, T - 200]
        kpm = torch.zeros((B, T), dtype=torch.uint8)
        for b, n in enumerate(lens):
            kpm[b, n:] = 1
        i = torch.arange(T).view(-1, 1)
        j = torch.arange(T).view(1, -1)
        am = (((i - j).abs() > 64) & (i != 0) & (j != 0)).to(torch.uint8)
        kw.update(key_padding_mask=kpm.cuda(), attn_mask=am.cuda())
        okw.update(kpm=kpm.numpy(), am=am.numpy())
    out_tok, lse_tok = ba.ulysses_attn_fwd(to_tok(q, P), to_tok(k, P), to_tok(v, P), **kw)
    out, lse = from_tok(out_tok), from_tok(lse_tok.unsqueeze(-1)).squeeze(-1)
    o_ref, l_ref = oracle.attention(q.float().cpu(), k.float().cpu(), v.float().cpu(), **okw)
    compare(out, lse, o_ref, l_ref, dt, f"ulysses {dt} d={d} {masks}")


def test_ulysses_full_size_8k_sampled():
    """The 8K causal configuration (B=4, H=16, T=8192, d=128, bf16) over P=8 ranks:
    the exchange is checked bit for bit on one tensor, the output on sampled rows."""
    from blockwise_attention_gb300.workloads import WORKLOADS, make_inputs
    from tests.parity import sample_rows
    w = WORKLOADS["zigzag_prefill_8k"]
    inp = make_inputs(w, "cuda")
    P = 8
    qt, kt, vt = to_tok(inp.q, P), to_tok(inp.k, P), to_tok(inp.v, P)
    qh = ba.ulysses_all_to_all(qt, P, "token_to_head")
    assert np.array_equal(qh.float().cpu().numpy(), oracle.ulysses_token_to_head(qt.float().cpu().numpy(), P))
    out_tok, lse_tok = ba.ulysses_attn_fwd(qt, kt, vt, causal=True)
    out, lse = from_tok(out_tok), from_tok(lse_tok.unsqueeze(-1)).squeeze(-1)
    heads = [(0, 0), (3, 15), (1, 7)]
    rows = sample_rows(w.B, w.H, w.T, heads, per_head=48, chunk=1024, seed=3)
    o_ref, l_ref = oracle.attention(inp.q.float().cpu(), inp.k.float().cpu(), inp.v.float().cpu(), causal=True,
                                    rows=rows)
    o = out.reshape(-1, w.d)[torch.from_numpy(rows).cuda()]
    l = lse.reshape(-1)[torch.from_numpy(rows).cuda()]
    compare(o, l, o_ref, l_ref, "bf16", "ulysses 8K sampled")
