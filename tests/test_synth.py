"""The synthetic proving-key stand-ins reproduce the statistics the GATHER_CU page prints
for js_1x1_d8 ... js_16x16_d32 (mean row length x n = nnz, empty rows, longest row), and
their draws are valid field elements, distinct sorted columns and a seeded, repeatable
stream."""
import numpy as np
import pytest

from bn254_scalar_field_gb300 import synth
from oracle import fr_int as F

# domain: (A mean, A empty, A max, B mean, B empty, B max), as printed on the page
PAGE_STATS = {
    12: (2.31, 732, 65, 3.70, 737, 64),
    14: (1.51, 6224, 67, 2.34, 6231, 66),
    17: (1.13, 60696, 79, 1.70, 60715, 78),
    18: (1.13, 121848, 95, 1.69, 121883, 94),
}


@pytest.mark.parametrize("log_n", sorted(PAGE_STATS))
def test_row_statistics_match_page(log_n):
    n = 1 << log_n
    A, B, w = synth.problem(log_n)
    for (rp, col, val), (mean, empty, mx) in ((A, PAGE_STATS[log_n][:3]),
                                              (B, PAGE_STATS[log_n][3:])):
        lens = np.diff(rp.astype(np.int64))
        assert rp.shape == (n + 1,) and rp[0] == 0 and rp[-1] == col.shape[0]
        assert round(col.shape[0] / n, 2) == mean
        assert int((lens == 0).sum()) == empty
        assert int(lens.max()) == mx
        assert val.shape == (col.shape[0], 8)
        # distinct sorted columns within each row, all below n_wires
        rows = np.repeat(np.arange(n), lens)
        same = rows[1:] == rows[:-1]
        assert np.all(col[1:][same] > col[:-1][same])
        assert int(col.max()) < w.shape[0]
    frac = synth.CONFIGS[log_n]["frac01"]
    small = (w == 0).all(1) | (w == synth.MONT_ONE_LIMBS).all(1)
    assert abs(small.mean() - frac) < 0.02
    assert np.array_equal(w[0], synth.MONT_ONE_LIMBS)


def test_uniform_fr_is_canonical_and_repeatable():
    x = synth.uniform_fr(synth.SplitMix64(5), 4000)
    vals = F.array_to_ints(x)
    assert all(v < F.R_MOD for v in vals)
    assert len(set(vals)) == len(vals)
    assert max(vals) > F.R_MOD * 0.99  # covers the whole range, top limb included
    y = synth.uniform_fr(synth.SplitMix64(5), 4000)
    assert np.array_equal(x, y)


def test_splitmix64_reference_values():
    # splitmix64 seeded with 0: first outputs of the published generator
    out = synth.SplitMix64(0).u64(3)
    assert [int(v) for v in out] == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]
