"""The partition an attention launch chooses (host logic, no GPU): key-sequence
splits x output-column shares per (query tile, K/V head), merged in one
cluster or by the combine kernel.  Proposition A.1 of "Reflex: Real-Time VLA
Control through Streaming Inference" (§III "Core formulas") makes every
choice exact; these tests pin which one the cost model takes for the
workloads' shapes and check the limits every choice must respect."""
import numpy as np
import pytest

from tests._util import ensure_built

# Clusters of c CTAs (231 KB of shared memory each) a GB300 holds at once:
# measured 23 of 6, 15 of 8, 8 of 12 and 7 of 16; the other sizes follow the
# same GPC packing.
GB300_CAP = [0, 152, 76, 48, 38, 28, 23, 19, 15, 15, 14, 8, 8, 7, 7, 7, 7]
SMS, MAX_SPLITS = 152, 64


@pytest.fixture(scope="module")
def rx():
    try:
        ensure_built()
    except RuntimeError as e:  # pragma: no cover
        pytest.skip("cannot build librx.so here: %s" % e)
    from partitioned_kv_cache_gb300 import rx as m
    return m


def choose(rx, t_max, units, D=256, splits=0, dparts=0, max_splits=MAX_SPLITS, cap=GB300_CAP):
    return rx.choose_partition(t_max, units, D, SMS, max_splits, cap, splits, dparts)


@pytest.mark.parametrize("name,t_max,units,want", [
    # 51 tokens x 8 heads = 4 query tiles; key tiles = pinned + window + dynamic
    ("c2: 48 + 4x256 + 51 keys", 1 + 16 + 1, 4, (12, 2, True)),
    ("c3: 64 + 8x256 + 51 keys", 1 + 32 + 1, 4, (12, 2, True)),
    ("c4: 256 + 32x256 + 51 keys", 4 + 128 + 1, 4, (27, 1, False)),
    ("c5: c3 + 16 language tails of 32", 1 + 32 + 8, 5, (16, 1, True)),
    ("1024-token suffix over c3's keys", 1 + 32 + 16, 64, (2, 1, True)),
    ("2048-token suffix over c4's keys", 4 + 128 + 32, 128, (1, 1, False)),
])
def test_workload_partitions(rx, name, t_max, units, want):
    assert choose(rx, t_max, units) == want, name


def test_forced_values_are_kept_and_clamped(rx):
    assert choose(rx, 34, 4, splits=1) == (1, 4, False)        # dparts still chosen
    assert choose(rx, 34, 4, dparts=1)[1] == 1
    assert choose(rx, 18, 4, splits=20, dparts=1) == (18, 1, False)   # clamped to the key tiles
    assert choose(rx, 133, 4, splits=24, dparts=1) == (24, 1, False)  # beyond a cluster: combine kernel
    assert choose(rx, 133, 4, max_splits=8) == (8, 2, True)     # the workspace holds 8 splits
    # The allocation-free entry point's 8 MiB scratch holds 30 splits of c4's
    # 408 query rows: the same 27 as the cache's workspace.
    assert choose(rx, 133, 4, max_splits=30) == (27, 1, False)


def test_out_of_range_sizes_are_refused(rx):
    for kw in (dict(t_max=0, units=4), dict(t_max=34, units=0), dict(t_max=1 << 25, units=4),
               dict(t_max=34, units=1 << 25)):
        with pytest.raises(rx.RxError):
            choose(rx, **kw)


def test_invalid_column_split_is_refused(rx):
    with pytest.raises(rx.RxError):
        choose(rx, 34, 4, D=128, dparts=4)                      # 32-column shares
    with pytest.raises(rx.RxError):
        choose(rx, 34, 4, dparts=3)


def test_every_choice_respects_the_limits(rx):
    g = np.random.default_rng(7)
    for _ in range(400):
        D = int(g.choice([64, 128, 256]))
        t_max = int(g.integers(1, 300))
        units = int(g.integers(1, 160))
        max_splits = int(g.choice([1, 8, 16, 64]))
        sp, dp, fused = choose(rx, t_max, units, D=D, max_splits=max_splits)
        assert 1 <= sp <= min(t_max, max_splits)
        assert dp in (1, 2, 4) and D // dp >= 64
        assert fused == (2 <= sp <= 16 and GB300_CAP[sp] >= 1)
        if fused:                       # all clusters of the grid resident at once
            assert units * dp <= GB300_CAP[sp]
        elif sp > 1:                    # the unclustered grid stays within 3/4 of the SMs
            assert dp == 1 and units * sp <= 3 * SMS // 4
        else:
            assert units * dp <= SMS or (units > SMS and dp == 1)
