"""The stream-K partition of the quantised GEMMs, through the library's host view of it
(pf_streamk_plan_host: the device code's own plan functions compiled for the host): every
k-block of every tile belongs to exactly one unit, in contiguous ranges; a skewed plan gives
its last units the stated k-blocks fewer; a unit runs its partial segments first (the
shorter of two ahead) and its whole tiles after, in k order; no unit has more than two
partial segments, and their scratch slots differ; owner() is the inverse of the ranges."""
import itertools

import numpy as np
import pytest

from quantized_transformer_prefill_q1_gb300 import pf

SHAPES = [(2, 24, 64, 76), (2, 16, 64, 76), (2, 96, 64, 76), (2, 16, 192, 76), (1, 5, 2, 7),
          (3, 1, 27, 38), (1, 1, 1, 1), (4, 7, 64, 152), (2, 2, 192, 76), (1, 594, 64, 152)]
SKEWS = [(0, 0), (26, 5), (26, 3), (36, 3), (20, 4), (76, 3), (10, 1000)]


@pytest.mark.parametrize("n_mt,n_nt,kbt,ctas", SHAPES)
@pytest.mark.parametrize("late_units,late_kb", SKEWS)
def test_partition(n_mt, n_nt, kbt, ctas, late_units, late_kb):
    total = n_mt * n_nt * kbt
    w = np.arange(total, dtype=np.int64)
    begins, segs, owners = pf.pf_streamk_plan_host(n_mt, n_nt, kbt, ctas, late_units, late_kb, 8, w)
    assert begins[0] == 0 and begins[-1] == total
    sizes = np.diff(begins)
    assert np.all(sizes >= 1)
    # owner(w) is the unit whose range holds w
    np.testing.assert_array_equal(owners, np.searchsorted(begins, w, side="right") - 1)
    # the skew: applied only while the late units are a minority; late ranges are shorter
    skewed = late_units > 0 and late_kb > 0 and 2 * late_units <= ctas and total // ctas > 1
    even = total // ctas
    if not skewed:
        assert sizes.max() - sizes.min() <= 1
    else:
        dk = min(late_kb, total // ctas - 1)
        early, late = sizes[: ctas - late_units], sizes[ctas - late_units:]
        assert early.max() - early.min() <= 1 and late.max() - late.min() <= 1
        assert abs(int(round(early.mean() - late.mean())) - dk) <= 1
        assert early.min() >= even
    covered = np.zeros(total, np.int32)
    for c in range(ctas):
        s = [tuple(x) for x in segs[c] if x[0] >= 0]
        assert 1 <= len(s) <= 8
        kbs = []
        for tile, kb0, nkb, slot in s:
            assert 0 <= kb0 and nkb >= 1 and kb0 + nkb <= kbt
            kbs.extend(tile * kbt + kb0 + i for i in range(nkb))
        assert sorted(kbs) == list(range(begins[c], begins[c + 1]))
        covered[kbs] += 1
        parts = [x for x in s if x[2] < kbt]
        assert len(parts) <= 2
        # partial segments first, the shorter of two ahead, then whole tiles in k order
        assert all(x[2] < kbt for x in s[: len(parts)])
        if len(parts) == 2:
            assert parts[0][2] <= parts[1][2]
            assert parts[0][3] != parts[1][3]
        whole = [x[0] for x in s[len(parts):]]
        assert whole == sorted(whole)
        assert all(x[3] == -1 for x in s[len(parts):])
    assert np.all(covered == 1)


def test_bad_sizes():
    with pytest.raises(pf.PfError) as e:
        pf.pf_streamk_plan_host(1, 1, 4, 5)  # more units than k-blocks
    assert e.value.status == 2
    with pytest.raises(pf.PfError):
        pf.pf_streamk_plan_host(1, 0, 4, 1)
