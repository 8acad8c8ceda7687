"""Host checks of the tensor-core forward kernel's work items (ba_pair_schedule,
computed by the functions the kernel itself runs): every query tile of every
head is dealt exactly once, the two tiles of an item are adjacent in one chunk,
each item's key-tile count equals a brute-force count over the walk (the ring
steps visit every chunk once; causal masking drops key tiles that start after
the pair's last query), and items come heaviest first, the lightest levels
last.  No GPU is needed."""
import math

import numpy as np
import pytest

import blockwise_attention_gb300 as ba

CASES = [
    # B, H, T, P, partition, causal, SMs
    (4, 16, 8192, 8, "zigzag", True, 152),      # 8K prefill shapes: 13.5 items per SM, light levels last
    (1, 32, 65536, 16, "zigzag", True, 152),    # 64K prefill shapes: grouped order only
    (2, 3, 1000, 4, "zigzag", True, 152),       # 125-token chunks: one ragged tile each
    (2, 3, 1000, 4, "contiguous", False, 152),  # bidirectional
    (1, 2, 384, 3, "zigzag", True, 4),          # 64-token chunks, few SMs
    (3, 5, 2560, 2, "contiguous", True, 16),    # 10 tiles per chunk
    (4, 16, 8192, 8, "striped", True, 152),     # 8K prefill shapes, striped ranks
    (2, 3, 1000, 4, "striped", True, 152),      # 250-token ranks: one ragged tile each
    (1, 2, 384, 3, "striped", True, 4),         # 128-token ranks
    (2, 2, 1024, 4, "striped", False, 16),      # bidirectional
]


def query_tiles(T, P, partition):
    """(row0, rows) of every 128-row query tile: tiles are cut from each chunk start.
    Rows are token positions, except for striped ranks, whose rows are in rank
    order: row c * cl + u holds token c + P * u."""
    nc = 2 * P if partition == "zigzag" else P
    cl = T // nc
    return [(c * cl + r, min(128, cl - r)) for c in range(nc) for r in range(0, cl, 128)], cl


def tile_visible(T, P, partition, q_row0, q_rows, k_row0, k_rows):
    """Does any key of the key tile precede or equal any query of the query tile
    (causal), by the tokens themselves?"""
    if partition != "striped":
        return k_row0 <= q_row0 + q_rows - 1
    cl = T // P
    tok = lambda R: (R // cl) + P * (R % cl)   # noqa: E731
    q_last = max(tok(R) for R in range(q_row0, q_row0 + q_rows))
    k_first = min(tok(R) for R in range(k_row0, k_row0 + k_rows))
    return k_first <= q_last


@pytest.mark.parametrize("B,H,T,P,part,causal,sms", CASES)
def test_pair_schedule(B, H, T, P, part, causal, sms):
    items = ba.pair_schedule(B, H, T, P, part, causal, sms)
    tiles, cl = query_tiles(T, P, part)
    n_tiles_per_chunk = math.ceil(cl / 128)
    assert items.shape == (B * H * math.ceil(n_tiles_per_chunk / 2) * (T // cl), 8)

    # every (b, h, query tile) exactly once
    dealt = []
    for b, h, r0, n0, r1, n1, _, _ in items:
        dealt.append((b, h, r0, n0))
        if n1 > 0:
            dealt.append((b, h, r1, n1))
            # the second tile follows the first within its chunk
            assert r1 == r0 + 128 and n0 == 128 and r0 // cl == r1 // cl
    expect = sorted((b, h, r, n) for b in range(B) for h in range(H) for r, n in tiles)
    assert sorted(tuple(int(x) for x in d) for d in dealt) == expect

    # key tiles of each item's walk, by brute force over all key tiles
    seen = {}
    for b, h, r0, n0, r1, n1, nk, _ in items:
        span = (r0, (r1 + n1 - r0) if n1 > 0 else n0)   # the pair's rows
        if span not in seen:
            seen[span] = sum(1 for k0, kn in tiles if not causal or tile_visible(T, P, part, *span, k0, kn))
        assert nk == seen[span]

    # heaviest first: within the grouped phase the key counts of one head never grow;
    # the last phase holds the lightest items of the launch, heaviest first
    phase = items[:, 7]
    assert np.all(np.diff(phase) >= 0)   # phase 0, then phase 1
    heavy, light = items[phase == 0], items[phase == 1]
    for b in range(B):
        for h in range(H):
            nk = heavy[(heavy[:, 0] == b) & (heavy[:, 1] == h), 6]
            assert np.all(np.diff(nk) <= 0)
    if causal and len(light):
        assert light[:, 6].max() <= heavy[:, 6].min() if len(heavy) else True
        assert np.all(np.diff(light[:, 6]) <= 0)
    if not causal:
        assert len(light) == 0 and np.all(items[:, 6] == len(tiles))


def test_pair_schedule_light_phase_rule():
    """The light phase exists only when the SMs get few items each: the 8K prefill
    shapes (2048 items on 152 SMs) deal their lightest levels last, the 64K shapes
    (8192 items) keep the grouped order throughout."""
    assert (ba.pair_schedule(4, 16, 8192, 8, "zigzag", True, 152)[:, 7] == 1).any()
    assert not (ba.pair_schedule(1, 32, 65536, 16, "zigzag", True, 152)[:, 7] == 1).any()


def test_pair_schedule_errors():
    with pytest.raises(ba.BlockAttnError):
        ba.pair_schedule(1, 1, 1000, 3, "zigzag", True, 152)      # T not divisible by 2P
    assert ba.pair_schedule(0, 4, 1024, 2, "zigzag", True, 152).shape == (0, 8)
