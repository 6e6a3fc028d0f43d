"""Pins for the oracle's shard plan and owner lookup (CPU only).

Shard plan: "Sharded GEMM与Backprop：行、列、内维三种切分", section Python 参考实现
(numpy array_split per axis) and section 手动走一遍 (K=5, parts=2 -> 3/2, and
parts larger than the dimension gives empty shards)."""
import json
import os

import numpy as np
import pytest

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_worked_split(orc):
    g = json.load(open(os.path.join(GOLDEN, "worked_split.json")))
    off = orc.plan_shards(g["K"], g["parts"])
    assert list(np.diff(off)) == g["inner_split_sizes"]
    assert list(off) == [0, 3, 5]


@pytest.mark.parametrize("dim", range(0, 65))
def test_plan_matches_array_split(orc, dim):
    x = np.arange(dim)
    for parts in range(1, 81):
        off = orc.plan_shards(dim, parts)
        sizes = [len(c) for c in np.array_split(x, parts)]
        assert list(np.diff(off)) == sizes
        assert off[0] == 0 and off[-1] == dim
        # sizes differ by at most one, larger shards first, parts > dim gives
        # exactly parts - dim empty shards
        d = np.diff(off)
        assert d.max() - d.min() <= 1 and np.all(np.diff(d) <= 0)
        if parts > dim:
            assert int((d == 0).sum()) == parts - dim


def test_plan_rejects_bad_parts(orc):
    with pytest.raises(ValueError, match="partition"):
        orc.plan_shards(5, 0)


def test_owner_brute_force(orc):
    rng = np.random.default_rng(1)
    for _ in range(200):
        V = int(rng.integers(1, 50))
        P = int(rng.integers(1, 60))
        off = orc.plan_shards(V, P)
        for y in range(V):
            owners = [r for r in range(P) if off[r] <= y < off[r + 1]]
            assert len(owners) == 1            # half-open intervals: unique owner
            assert orc.owner(y, off) == owners[0]
            assert off[owners[0] + 1] > off[owners[0]]   # never an empty shard
        assert orc.owner(V, off) == -1
