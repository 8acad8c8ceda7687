"""Pins of the fp64 attention-gradient oracle against facts it does not compute
itself: central finite differences of the (separately pinned) forward oracle,
the softmax invariants of the gradients, and exact zeros the masking implies.

The backward pass the pages describe ("Sequence/context parallelism"
(brunomaga), section "Ring Attention", backward) sums per-block gradients that
use the saved out and LSE of the whole row; their sum is the gradient of the
attention function, which is what the oracle states and these tests pin."""
import numpy as np
import pytest

import oracle


def dyadic(rng, shape, step=2.0 ** -8, lim=2.0):
    """Random values on a 2^-8 grid in [-lim, lim]: exact in fp32, and so are x +- 2^-12."""
    n = int(lim / step)
    return (rng.integers(-n, n + 1, size=shape) * step).astype(np.float32)


def loss(q, k, v, g, **kw):
    out, _ = oracle.attention(q, k, v, **kw)
    return float(np.sum(out * g.astype(np.float64)))


CASES = [
    dict(),
    dict(causal=True, q_pos0=3, k_pos0=1),
    dict(kpm="pad", am="rand", causal=True, q_pos0=2, k_pos0=0),
]


@pytest.mark.parametrize("case", range(len(CASES)))
def test_gradients_match_central_differences(case):
    rng = np.random.default_rng(100 + case)
    B, H, L, S, d = 1, 2, 4, 5, 3
    q, k, v = dyadic(rng, (B, H, L, d)), dyadic(rng, (B, H, S, d)), dyadic(rng, (B, H, S, d))
    g = dyadic(rng, (B, H, L, d))
    kw = dict(CASES[case])
    if kw.get("kpm") == "pad":
        kpm = np.zeros((B, kw.get("k_pos0", 0) + S), np.uint8)
        kpm[0, -1] = 1
        kw["kpm"] = kpm
    if kw.get("am") == "rand":
        am = (rng.random((kw.get("q_pos0", 0) + L, kw.get("k_pos0", 0) + S)) < 0.3).astype(np.uint8)
        kw["am"] = am
    dq, dk, dv, _, _ = oracle.attention_bwd(q, k, v, g, **kw)
    h = 2.0 ** -12
    for name, x, grad in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        for idx in np.ndindex(x.shape):
            xp, xm = x.copy(), x.copy()
            xp[idx] += h
            xm[idx] -= h
            args_p = {"q": q, "k": k, "v": v}
            args_m = {"q": q, "k": k, "v": v}
            args_p[name], args_m[name] = xp, xm
            fd = (loss(args_p["q"], args_p["k"], args_p["v"], g, **kw) -
                  loss(args_m["q"], args_m["k"], args_m["v"], g, **kw)) / (2 * h)
            assert abs(fd - grad[idx]) <= 1e-6 + 1e-5 * abs(grad[idx]), (name, idx, fd, grad[idx])


def test_softmax_invariants():
    """Sum over keys of dK is 0 (shifting every key by one vector shifts each
    row's scores by a constant); sum of dV over keys equals the sum of dout over
    rows that see a key (each row's weights sum to 1)."""
    rng = np.random.default_rng(7)
    B, H, L, S, d = 2, 3, 9, 11, 5
    q = rng.standard_normal((B, H, L, d)).astype(np.float32)
    k = rng.standard_normal((B, H, S, d)).astype(np.float32)
    v = rng.standard_normal((B, H, S, d)).astype(np.float32)
    g = rng.standard_normal((B, H, L, d)).astype(np.float32)
    kpm = np.zeros((B, S), np.uint8)
    kpm[1, 7:] = 1
    dq, dk, dv, _, lse = oracle.attention_bwd(q, k, v, g, causal=True, kpm=kpm, q_pos0=2)
    scale_ref = np.abs(dk).max()
    assert np.abs(dk.sum(axis=2)).max() <= 1e-12 * max(1.0, scale_ref) * S
    seen = np.isfinite(lse)[..., None]
    np.testing.assert_allclose(dv.sum(axis=2), (g.astype(np.float64) * seen).sum(axis=2), atol=1e-12, rtol=0)
    # padded keys get no gradient at all
    assert np.all(dk[1, :, 7:] == 0) and np.all(dv[1, :, 7:] == 0)


def test_single_visible_key_rows_have_zero_dq():
    """Causal row 0 sees only key 0: its weight is exactly 1, so dS = 0 and dQ of
    that row is exactly 0, while dV of key 0 receives that row's dout."""
    rng = np.random.default_rng(8)
    B, H, L, d = 1, 1, 6, 4
    q, k, v = (rng.standard_normal((B, H, L, d)).astype(np.float32) for _ in range(3))
    g = rng.standard_normal((B, H, L, d)).astype(np.float32)
    dq, dk, dv, out, _ = oracle.attention_bwd(q, k, v, g, causal=True)
    assert np.all(dq[0, 0, 0] == 0)
    np.testing.assert_array_equal(out[0, 0, 0], v[0, 0, 0].astype(np.float64))


def test_fully_masked_row_contributes_nothing():
    rng = np.random.default_rng(9)
    B, H, L, S, d = 1, 1, 4, 4, 3
    q, k, v = (rng.standard_normal((B, H, n, d)).astype(np.float32) for n in (L, S, S))
    g = rng.standard_normal((B, H, L, d)).astype(np.float32)
    am = np.zeros((L, S), np.uint8)
    am[2, :] = 1
    dq, dk, dv, out, lse = oracle.attention_bwd(q, k, v, g, am=am)
    assert lse[0, 0, 2] == -np.inf and np.all(out[0, 0, 2] == 0) and np.all(dq[0, 0, 2] == 0)
    g2 = g.copy()
    g2[0, 0, 2] = 100.0   # the masked row's dout must not matter
    _, dk2, dv2, _, _ = oracle.attention_bwd(q, k, v, g2, am=am)
    np.testing.assert_array_equal(dk, dk2)
    np.testing.assert_array_equal(dv, dv2)
