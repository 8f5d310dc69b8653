"""Hand-worked quantisation tiles (tests/golden/hand_tiles.json) against the oracle.

Each fixture carries its own derivation and the passages it follows; the
values were worked out by hand from those rules, not produced by any code.
"""
import json
import os

import numpy as np
import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
with open(os.path.join(HERE, "golden", "hand_tiles.json")) as f:
    TILES = json.load(f)["tiles"]


def _tile_bits(t):
    x = np.full(128, t.get("fill", 0.0), np.float32)
    for k, v in t["values"].items():
        x[int(k)] = v
    u = x.view(np.uint32)
    assert np.all((u & 0xFFFF) == 0), "fixture values must be exact BF16"
    return (u >> 16).astype(np.uint16).reshape(1, 128)


@pytest.mark.parametrize("t", TILES, ids=[t["name"] for t in TILES])
def test_hand_tile(oracle, t):
    q, sa = oracle.quant_act(_tile_bits(t), pow2=(t["mode"] == "pow2"))
    assert float(sa[0, 0]) == float.fromhex(t["scale"])
    for pos, code in t["codes"].items():
        assert int(q[0, int(pos)]) == int(code, 16), (pos, hex(q[0, int(pos)]))
    # the same tile read as a 128x1 column and as a 128x128 block row
    qT, sT = oracle.quant_act_T(np.ascontiguousarray(_tile_bits(t).T), pow2=(t["mode"] == "pow2"))
    assert np.array_equal(qT, q) and np.array_equal(sT, sa)
