"""The stored spread of the chained backward statistics (tests/golden/
stat_spread.json, written by tests/golden/make_stat_spread.py from the oracle
alone) is what the oracle gives now, and the GPU tests' bounds for chained s
and s' follow from it (CPU, about 40 s)."""
import pytest

from tests import _util
from tests.golden import make_stat_spread


@pytest.fixture(scope="module")
def fresh():
    return make_stat_spread.compute()


def test_stored_spread_is_reproduced_by_the_oracle(fresh):
    stored = _util.stat_spread()
    for wl, stats in (("llama8b_block", ("s1", "s")), ("llama1b_mlp_bwd", ("s",))):
        assert stored[wl]["rows"] == fresh[wl]["rows"]
        for k in stats:
            # numpy's fp64 products may sum in another order on another BLAS,
            # which can move a truncation decision: a few percent at most
            assert fresh[wl][k] == pytest.approx(stored[wl][k], rel=0.05), (wl, k)


def test_chained_bounds_follow_from_the_spread():
    st = _util.stat_spread()
    for wl, k in (("llama8b_block", "s1"), ("llama8b_block", "s"), ("llama1b_mlp_bwd", "s")):
        tol = _util.chained_stat_tol(wl, k)
        assert tol == max(_util.TOL_F32, _util.CHAIN_MARGIN * st[wl][k])
        # the spread is a fraction of the bound it implies, never the bound itself
        assert st[wl][k] <= tol / _util.CHAIN_MARGIN
