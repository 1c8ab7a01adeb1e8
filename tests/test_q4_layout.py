"""The LOCKS_DTYPE_Q4 byte layout of include/locks.h as the test side packs
it (tests/helpers.pack_q4 / unpack_q4), checked on the CPU: every code and
scale has its own byte, the pieces one scan lane reads are adjacent, and
packing round-trips."""

import numpy as np
import pytest

from tests.helpers import (_q4_coef_position, _q4_scale_order, _q4_word_position, pack_q4, q4_block_bytes,
                           unpack_q4)


@pytest.mark.parametrize("r", [2, 4, 6, 8])
@pytest.mark.parametrize("P", [16, 64])
def test_positions_are_permutations(r, P):
    assert sorted(_q4_word_position(m) for m in range(16)) == list(range(16))
    pos = [_q4_coef_position(i, j, r, P) for i in range(P) for j in range(r)]
    assert sorted(pos) == list(range(P * r))
    order = _q4_scale_order(r)
    assert len(order) == 2 * r + 1 and len(set(order)) == 2 * r + 1 and order[-1] == ("smu", 0)


@pytest.mark.parametrize("r", [2, 8])
@pytest.mark.parametrize("P", [16, 64])
def test_lane_pieces_are_adjacent(r, P):
    """Lane (g, c) of a scan warp reads basis words 4c .. 4c+3 of row g (the
    elements 32 s + 8 c .. +7, s = 0..3), the codes of tokens g + 8 t for
    columns 2c and 2c + 1 (t = 0 .. P/8 - 1), and the four scales of column
    pair c: each a contiguous range starting on a 4-byte boundary."""
    for c in range(4):
        words = [_q4_word_position(4 * s + c) for s in range(4)]
        assert words == list(range(4 * c, 4 * c + 4))
    for g in range(8):
        for c in range(r // 2):
            bytes_ = [_q4_coef_position(g + 8 * t, 2 * c + e, r, P) for t in range(P // 8) for e in range(2)]
            assert bytes_ == list(range(bytes_[0], bytes_[0] + 2 * (P // 8))) and bytes_[0] % 4 == 0
    order = _q4_scale_order(r)
    for c in range(r // 2):
        assert order[4 * c:4 * c + 4] == [("sv", 2 * c), ("sv", 2 * c + 1), ("sc", 2 * c), ("sc", 2 * c + 1)]


@pytest.mark.parametrize("r", [2, 4, 6, 8])
@pytest.mark.parametrize("P", [16, 64])
def test_pack_round_trip(r, P):
    rng = np.random.default_rng(r * 100 + P)
    qs = dict(vq=rng.integers(-7, 8, (r, 128)), sv=rng.random(r), cq=rng.integers(-127, 128, (P, r)),
              sc=rng.random(r), muq=rng.integers(-127, 128, 128), smu=0.25)
    buf = pack_q4(qs, r)
    assert buf.shape == (q4_block_bytes(r, P),)
    back = unpack_q4(buf, r, P)
    for key in ("vq", "cq", "muq"):
        assert np.array_equal(np.asarray(qs[key]), back[key]), key
    for key in ("sv", "sc"):
        assert np.allclose(np.asarray(qs[key], dtype=np.float32), back[key]), key
    assert back["smu"] == 0.25
