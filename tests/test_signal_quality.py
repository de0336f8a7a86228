"""Host statistics of the signal-quality analysis (no GPU)."""
import numpy as np
import pytest
from scipy import stats

from demand_paged_kv_gqa_b300 import signal_quality as sq


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_spearman_matches_scipy_with_ties(seed):
    rng = np.random.default_rng(seed)
    x = rng.integers(-5, 6, size=200)          # many ties
    y = 0.5 * x + rng.integers(-4, 5, size=200)
    assert sq.spearman(x, y) == pytest.approx(stats.spearmanr(x, y).statistic, abs=1e-12)


def test_rank_average_ties():
    assert sq.rank_average([3, 1, 3, 2]).tolist() == [3.5, 1.0, 3.5, 2.0]


def test_statistics_pairs_follow_consecutive_boundaries():
    # request 7: Delta 5 then demand 10 -> 14 (+4, agree), Delta -2 then 14 -> 9 (-5, agree),
    # Delta 3 then 9 -> 9 (0: not a sign pair); request 8: a single boundary, no pair
    tr = {7: [(5, 10), (-2, 14), (3, 9), (0, 9)], 8: [(4, 100)]}
    x, y = sq.pairs_from_traces(tr)
    assert x.tolist() == [5, -2, 3] and y.tolist() == [4, -5, 0]
    st = sq.statistics(tr)
    assert st["pairs"] == 3 and st["sign_pairs"] == 2 and st["sign_agreement"] == 1.0
    assert st["spearman_rho"] == pytest.approx(stats.spearmanr(x, y).statistic)
