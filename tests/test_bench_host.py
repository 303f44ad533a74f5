"""Host helpers of bench.py that need no GPU."""
import numpy as np

import bench


def test_spread_is_p10_median_p90():
    ms = list(np.arange(1.0, 11.0))          # 1..10
    got = bench._spread(ms[::-1])
    assert got == {"p10": 1.9, "median": 5.5, "p90": 9.1}
    assert bench._spread([2.5]) == {"p10": 2.5, "median": 2.5, "p90": 2.5}


def test_split_partition_only_for_two_launches():
    assert bench._split_partition(0, 30000, 1) == 0
    assert bench._split_partition(0, 30000, 2) == 512
    assert bench._split_partition(256, 30000, 2) == 256
