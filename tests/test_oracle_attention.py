"""Pins of the fp64 attention oracle against what the pages and the mathematics
fix: the worked example, closed forms, invariants, brute force and a library
routine.  No GPU, no CUDA library."""
import math

import numpy as np
import pytest
import torch

import oracle
from tests.conftest import golden


def rnd(*shape, seed=0, scale=1.0):
    return np.random.default_rng(seed).standard_normal(shape).astype(np.float32) * np.float32(scale)


def brute_force(q, k, v, scale, visible):
    """Independent float64 Python loops: materialise the L x S score matrix,
    exponentiate the visible entries, normalise each row, weight V."""
    L, d = q.shape
    S = k.shape[0]
    out = [[0.0] * d for _ in range(L)]
    lse = [0.0] * L
    for i in range(L):
        sc = []
        for j in range(S):
            sc.append(sum(float(q[i][c]) * float(k[j][c]) for c in range(d)) * scale)
        vis = [j for j in range(S) if visible(i, j)]
        if not vis:
            lse[i] = -math.inf
            continue
        mx = max(sc[j] for j in vis)
        z = sum(math.exp(sc[j] - mx) for j in vis)
        lse[i] = mx + math.log(z)
        for j in vis:
            w = math.exp(sc[j] - mx) / z
            for c in range(d):
                out[i][c] += w * float(v[j][c])
    return np.array(out), np.array(lse)


def test_worked_example_l103():
    g = golden("sdpa_worked_example.json")
    # one query with zero scores against two keys: q = 0 makes every score 0
    q = np.zeros((1, 1, 1, 2), np.float32)
    k = rnd(1, 1, 2, 2, seed=3)
    v = np.array(g["values"], np.float32).reshape(1, 1, 2, 2)
    o, lse = oracle.attention(q, k, v)
    assert np.allclose(o[0, 0, 0], g["all_visible"]["output"], atol=1e-15)
    assert np.isclose(lse[0, 0, 0], math.log(2.0), atol=1e-15)
    # exclude the second source: with key padding and, separately, with attn_mask
    kpm = np.array([[0, 1]], np.uint8)
    o2, lse2 = oracle.attention(q, k, v, kpm=kpm)
    assert np.allclose(o2[0, 0, 0], g["second_source_excluded"]["output"], atol=1e-15)
    assert lse2[0, 0, 0] == 0.0  # single visible key with score 0
    am = np.array([[0, 1]], np.uint8)
    o3, _ = oracle.attention(q, k, v, am=am)
    assert np.array_equal(o3, o2)


@pytest.mark.parametrize("causal", [False, True])
def test_brute_force_tiny(causal):
    rng = np.random.default_rng(7)
    for trial in range(6):
        L = S = int(rng.integers(1, 7))
        d = int(rng.integers(1, 5))
        q, k, v = rnd(1, 1, L, d, seed=trial), rnd(1, 1, S, d, seed=trial + 10), rnd(1, 1, S, d, seed=trial + 20)
        kpm = (rng.random((1, S)) < 0.3).astype(np.uint8)
        am = (rng.random((L, S)) < 0.3).astype(np.uint8)
        o, lse = oracle.attention(q, k, v, causal=causal, kpm=kpm, am=am)

        def visible(i, j):
            return not ((causal and j > i) or kpm[0][j] or am[i][j])

        ob, lb = brute_force(q[0, 0], k[0, 0], v[0, 0], 1.0 / math.sqrt(d), visible)
        assert np.allclose(o[0, 0], ob, atol=1e-12, rtol=0)
        fin = np.isfinite(lb)
        assert np.array_equal(fin, np.isfinite(lse[0, 0]))
        assert np.allclose(lse[0, 0][fin], lb[fin], atol=1e-12, rtol=0)
        assert np.all(o[0, 0][~fin] == 0.0)


def test_matches_torch_sdpa_float64():
    """General case against a library routine: torch SDPA in float64 on CPU with a
    boolean 'allowed' mask (SDPA's polarity is True = take part)."""
    B, H, L, d = 2, 3, 37, 16
    q, k, v = rnd(B, H, L, d, seed=1), rnd(B, H, L, d, seed=2), rnd(B, H, L, d, seed=3)
    rng = np.random.default_rng(5)
    lengths = rng.integers(5, L + 1, size=B)
    kpm = (np.arange(L)[None, :] >= lengths[:, None]).astype(np.uint8)
    am = (rng.random((L, L)) < 0.4).astype(np.uint8)
    am[:, 0] = 0  # key 0 always allowed so no row is empty (SDPA returns NaN there)
    for causal in (False, True):
        o, lse = oracle.attention(q, k, v, causal=causal, kpm=kpm, am=am)
        allowed = ~(kpm[:, None, None, :].astype(bool) | am[None, None].astype(bool))
        if causal:
            allowed = allowed & np.tril(np.ones((L, L), bool))[None, None]
        ref = torch.nn.functional.scaled_dot_product_attention(
            torch.from_numpy(q).double(), torch.from_numpy(k).double(), torch.from_numpy(v).double(),
            attn_mask=torch.from_numpy(np.broadcast_to(allowed, (B, 1, L, L)).copy()))
        assert np.allclose(o, ref.numpy(), atol=1e-12, rtol=0)
        # LSE against torch.logsumexp of the masked scaled scores
        s = torch.einsum("bhid,bhjd->bhij", torch.from_numpy(q).double(), torch.from_numpy(k).double())
        s = s / math.sqrt(d)
        s = s.masked_fill(~torch.from_numpy(np.broadcast_to(allowed, (B, 1, L, L)).copy()), -math.inf)
        assert np.allclose(lse, torch.logsumexp(s, dim=-1).numpy(), atol=1e-12, rtol=0)


def test_rows_sum_to_one():
    """Softmax weights are nonnegative and sum to one: with V = 1 every output is 1."""
    B, H, L, d = 1, 2, 50, 8
    q, k = rnd(B, H, L, d, seed=4, scale=3.0), rnd(B, H, L, d, seed=5, scale=3.0)
    v = np.ones((B, H, L, d), np.float32)
    for causal in (False, True):
        o, _ = oracle.attention(q, k, v, causal=causal)
        assert np.allclose(o, 1.0, atol=1e-13)


def test_single_visible_key_and_causal_row0():
    B, H, L, d = 1, 1, 9, 4
    q, k, v = rnd(B, H, L, d, seed=6), rnd(B, H, L, d, seed=7), rnd(B, H, L, d, seed=8)
    kpm = np.ones((1, L), np.uint8)
    kpm[0, 4] = 0  # only key 4 visible
    o, lse = oracle.attention(q, k, v, kpm=kpm)
    assert np.allclose(o[0, 0], np.broadcast_to(v[0, 0, 4], (L, d)), atol=1e-15)
    scores = (q[0, 0].astype(np.float64) @ k[0, 0, 4].astype(np.float64)) / 2.0
    assert np.allclose(lse[0, 0], scores, atol=1e-14)
    # causal: row 0 sees only key 0, so O_0 = V_0 and LSE_0 = its score
    o, lse = oracle.attention(q, k, v, causal=True)
    assert np.allclose(o[0, 0, 0], v[0, 0, 0], atol=1e-15)
    assert np.isclose(lse[0, 0, 0], float(q[0, 0, 0].astype(np.float64) @ k[0, 0, 0].astype(np.float64)) / 2.0)


def test_equal_scores_give_mean_of_visible():
    B, H, L, d = 2, 1, 12, 5
    q = np.zeros((B, H, L, d), np.float32)
    k, v = rnd(B, H, L, d, seed=9), rnd(B, H, L, d, seed=10)
    kpm = np.zeros((B, L), np.uint8)
    kpm[1, 7:] = 1
    o, lse = oracle.attention(q, k, v, causal=True, kpm=kpm)
    for b in range(B):
        for i in range(L):
            vis = [j for j in range(i + 1) if not kpm[b, j]]
            assert np.allclose(o[b, 0, i], v[b, 0, vis].astype(np.float64).mean(0), atol=1e-14)
            assert np.isclose(lse[b, 0, i], math.log(len(vis)), atol=1e-14)


def test_fully_masked_row_is_zero_with_minus_inf_lse():
    q, k, v = rnd(1, 1, 3, 4, seed=11), rnd(1, 1, 3, 4, seed=12), rnd(1, 1, 3, 4, seed=13)
    am = np.zeros((3, 3), np.uint8)
    am[1, :] = 1
    o, lse = oracle.attention(q, k, v, am=am)
    assert lse[0, 0, 1] == -np.inf and np.all(o[0, 0, 1] == 0.0)
    assert np.isfinite(lse[0, 0, [0, 2]]).all()


def test_masked_positions_get_zero_weight():
    """Changing K or V at excluded positions leaves the result bit-for-bit unchanged."""
    B, H, L, d = 2, 2, 40, 8
    q, k, v = rnd(B, H, L, d, seed=14), rnd(B, H, L, d, seed=15), rnd(B, H, L, d, seed=16)
    kpm = np.zeros((B, L), np.uint8)
    kpm[0, 30:] = 1
    kpm[1, 17:] = 1
    o, lse = oracle.attention(q, k, v, causal=True, kpm=kpm)
    k2, v2 = k.copy(), v.copy()
    k2[0, :, 30:] = 1e3
    v2[0, :, 30:] = -7e4
    k2[1, :, 17:] = -2e3
    v2[1, :, 17:] = np.nan
    o2, lse2 = oracle.attention(q, k2, v2, causal=True, kpm=kpm)
    assert np.array_equal(o, o2) and np.array_equal(lse, lse2)


def test_exclusions_combine_as_or():
    """key_padding_mask and attn_mask together == one attn_mask holding their union."""
    B, H, L, d = 3, 2, 33, 8
    q, k, v = rnd(B, H, L, d, seed=17), rnd(B, H, L, d, seed=18), rnd(B, H, L, d, seed=19)
    rng = np.random.default_rng(3)
    kpm = (rng.random((B, L)) < 0.25).astype(np.uint8)
    am = (rng.random((L, L)) < 0.25).astype(np.uint8)
    o, lse = oracle.attention(q, k, v, causal=True, kpm=kpm, am=am)
    for b in range(B):
        union = (am | kpm[b][None, :]).astype(np.uint8)
        causal_mask = np.triu(np.ones((L, L), np.uint8), 1)
        ob, lb = oracle.attention(q[b:b + 1], k[b:b + 1], v[b:b + 1], am=union | causal_mask)
        assert np.array_equal(o[b:b + 1], ob) and np.array_equal(lse[b:b + 1], lb)


def test_causal_prefix_invariance():
    """Appending tokens leaves the earlier rows' outputs unchanged."""
    B, H, L, d = 1, 2, 30, 8
    q, k, v = rnd(B, H, L + 9, d, seed=20), rnd(B, H, L + 9, d, seed=21), rnd(B, H, L + 9, d, seed=22)
    o_long, l_long = oracle.attention(q, k, v, causal=True)
    o_short, l_short = oracle.attention(q[:, :, :L], k[:, :, :L], v[:, :, :L], causal=True)
    assert np.array_equal(o_long[:, :, :L], o_short) and np.array_equal(l_long[:, :, :L], l_short)


def test_permutation_equivariance():
    B, H, L, d = 1, 2, 25, 8
    q, k, v = rnd(B, H, L, d, seed=23), rnd(B, H, L, d, seed=24), rnd(B, H, L, d, seed=25)
    o, lse = oracle.attention(q, k, v)
    perm = np.random.default_rng(1).permutation(L)
    o_kv, l_kv = oracle.attention(q, k[:, :, perm], v[:, :, perm])
    assert np.allclose(o_kv, o, atol=1e-13) and np.allclose(l_kv, lse, atol=1e-13)
    o_q, l_q = oracle.attention(q[:, :, perm], k, v)
    assert np.allclose(o_q, o[:, :, perm], atol=1e-15) and np.allclose(l_q, lse[:, :, perm], atol=1e-15)


def test_scale_is_one_over_sqrt_d():
    """Scores are divided by sqrt(d): scale=1 on q/sqrt(d) gives the default result.
    q is drawn so that q/sqrt(d) is exact (d = 16 -> divide by 4)."""
    B, H, L, d = 1, 1, 20, 16
    q, k, v = rnd(B, H, L, d, seed=26), rnd(B, H, L, d, seed=27), rnd(B, H, L, d, seed=28)
    o, lse = oracle.attention(q, k, v, causal=True)
    o1, l1 = oracle.attention(q / np.float32(4.0), k, v, causal=True, scale=1.0)
    assert np.allclose(o, o1, atol=1e-14) and np.allclose(lse, l1, atol=1e-14)
    # and the statistical fact behind it: unit-variance dot products have variance ~d
    a, b = rnd(20000, 64, seed=40).astype(np.float64), rnd(20000, 64, seed=41).astype(np.float64)
    assert abs(np.var((a * b).sum(1)) / 64 - 1.0) < 0.05


def test_merge_of_any_split_equals_unsplit():
    """Taking the keys in blocks and merging with LSE gives the unsplit result,
    for random cut points and any merge order; plain averaging does not."""
    B, H, L, S, d = 2, 2, 21, 64, 8
    q, k, v = rnd(B, H, L, d, seed=29), rnd(B, H, S, d, seed=30), rnd(B, H, S, d, seed=31)
    kpm = np.zeros((B, S), np.uint8)
    kpm[1, 50:] = 1
    o_full, l_full = oracle.attention(q, k, v, kpm=kpm, q_pos0=S - L, causal=True)
    rng = np.random.default_rng(2)
    for trial in range(4):
        cuts = np.sort(rng.choice(np.arange(1, S), size=4, replace=False))
        bounds = [0, *cuts.tolist(), S]
        parts = []
        for a, b in zip(bounds[:-1], bounds[1:]):
            parts.append(oracle.attention(q, k[:, :, a:b], v[:, :, a:b], kpm=kpm, k_pos0=a,
                                          q_pos0=S - L, causal=True))
        order = rng.permutation(len(parts))
        o, l = parts[order[0]]
        for p in order[1:]:
            o, l = oracle.merge(o, l, *parts[p])
        assert np.allclose(o, o_full, atol=1e-13) and np.allclose(l, l_full, atol=1e-13)
    # averaging the block outputs is not attention over the union
    o_a, l_a = oracle.attention(q, k[:, :, :32], v[:, :, :32], kpm=kpm)
    o_b, l_b = oracle.attention(q, k[:, :, 32:], v[:, :, 32:], kpm=kpm, k_pos0=32)
    o_u, _ = oracle.attention(q, k, v, kpm=kpm)
    assert not np.allclose((o_a + o_b) / 2, o_u, atol=1e-3)
    assert not np.allclose(o_a + o_b, o_u, atol=1e-3)


def test_merge_with_empty_is_identity():
    o = rnd(5, 4, seed=32).astype(np.float64)
    l = rnd(5, seed=33).astype(np.float64)
    z = np.zeros_like(o)
    ninf = np.full(5, -np.inf)
    om, lm = oracle.merge(o, l, z, ninf)
    assert np.array_equal(om, o) and np.array_equal(lm, l)
    om, lm = oracle.merge(z, ninf, o, l)
    assert np.array_equal(om, o) and np.array_equal(lm, l)


def test_row_subset_matches_full():
    B, H, L, d = 2, 3, 17, 8
    q, k, v = rnd(B, H, L, d, seed=34), rnd(B, H, L, d, seed=35), rnd(B, H, L, d, seed=36)
    o, lse = oracle.attention(q, k, v, causal=True)
    rows = np.array([0, 5, 16, 17, 50, B * H * L - 1])
    os_, ls = oracle.attention(q, k, v, causal=True, rows=rows)
    assert np.array_equal(os_, o.reshape(-1, d)[rows]) and np.array_equal(ls, lse.reshape(-1)[rows])
