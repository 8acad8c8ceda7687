"""Pins of the Ulysses layout oracle: the pages' worked example, the round trip,
and the placement of every labelled element (its head and token survive the
exchange), plus the composition with attention: attention computed per rank on
the head-split layout and sent back equals attention on the unpartitioned
tensors.  Sources: "Sequence/context parallelism" (brunomaga), section
"Ulysses sequence parallelism" (the (H, B, T/P, E) <-> (H/P, B, T, E) view
swap), and "Change token partitions into head partitions with Ulysses"."""
import numpy as np
import pytest

import oracle


def labelled(P, H, B, T, d):
    """x_tok[r, h, b, tl, e] = code of (h, b, global token, e), exact in float64."""
    Tl = T // P
    x = np.empty((P, H, B, Tl, d))
    for r in range(P):
        for h in range(H):
            for b in range(B):
                for tl in range(Tl):
                    for e in range(d):
                        x[r, h, b, tl, e] = ((h * 100 + b) * 10000 + r * Tl + tl) * 10 + e
    return x


def test_page_example_two_gpus_two_heads_four_tokens():
    """After the first all-to-all GPU 0 holds h0 for t0..t3 and GPU 1 holds h1 for
    the same four tokens; the reverse exchange sends t2..t3 of h0 back to GPU 1
    and t0..t1 of h1 back to GPU 0."""
    P, H, B, T, d = 2, 2, 1, 4, 1
    x = labelled(P, H, B, T, d)
    y = oracle.ulysses_token_to_head(x, P)
    assert y.shape == (2, 1, 1, 4, 1)
    code = lambda h, t: (h * 100 * 10000 + t) * 10
    assert [y[0, 0, 0, t, 0] for t in range(4)] == [code(0, t) for t in range(4)]
    assert [y[1, 0, 0, t, 0] for t in range(4)] == [code(1, t) for t in range(4)]
    z = oracle.ulysses_head_to_token(y, P)
    assert z[1, 0, 0, 0, 0] == code(0, 2) and z[1, 0, 0, 1, 0] == code(0, 3)   # h0, t2..t3 on GPU 1
    assert z[0, 1, 0, 0, 0] == code(1, 0) and z[0, 1, 0, 1, 0] == code(1, 1)   # h1, t0..t1 on GPU 0


@pytest.mark.parametrize("P,H,B,T,d", [(2, 4, 2, 6, 3), (4, 8, 1, 8, 2), (1, 3, 2, 5, 2), (3, 6, 2, 9, 1)])
def test_every_element_lands_at_its_head_and_token(P, H, B, T, d):
    x = labelled(P, H, B, T, d)
    y = oracle.ulysses_token_to_head(x, P)
    hl = H // P
    for r in range(P):
        for j in range(hl):
            for b in range(B):
                for t in range(T):
                    for e in range(d):
                        h = r * hl + j
                        assert y[r, j, b, t, e] == ((h * 100 + b) * 10000 + t) * 10 + e
    np.testing.assert_array_equal(oracle.ulysses_head_to_token(y, P), x)


def test_attention_on_the_head_split_layout_is_the_plain_attention():
    P, H, B, T, d = 2, 4, 2, 8, 4
    rng = np.random.default_rng(5)
    full = [rng.standard_normal((B, H, T, d)).astype(np.float32) for _ in range(3)]
    # token-split shards (P, H, B, T/P, d) of each tensor
    tok = [np.ascontiguousarray(x.transpose(1, 0, 2, 3).reshape(H, B, P, T // P, d).transpose(2, 0, 1, 3, 4))
           for x in full]
    heads = [oracle.ulysses_token_to_head(x, P) for x in tok]
    outs = []
    for r in range(P):
        q, k, v = (np.ascontiguousarray(x[r].transpose(1, 0, 2, 3)) for x in heads)   # (B, H/P, T, d)
        o, _ = oracle.attention(q, k, v, causal=True)
        outs.append(o.transpose(1, 0, 2, 3))                                           # (H/P, B, T, d)
    back = oracle.ulysses_head_to_token(np.stack(outs), P)                             # (P, H, B, T/P, d)
    o_full, _ = oracle.attention(*full, causal=True)
    o_tok = o_full.transpose(1, 0, 2, 3).reshape(H, B, P, T // P, d).transpose(2, 0, 1, 3, 4)
    np.testing.assert_array_equal(back, o_tok)
