"""Parity with the fp64 oracle on seeded random shapes: token counts, hidden
sizes (multiples of 8), vocabulary sizes, ignore fractions, target
distributions and chunk sizes drawn per case, on all four tile shapes, one
handle per shape reused across the cases (workspace growth, cached tile
orders, changing tensor maps)."""
import numpy as np
import pytest

import oracle
import workloads
from flce_testing import assert_parity, run

pytestmark = pytest.mark.gpu

SHAPES = ("single", "pair", "quad", "wide")


@pytest.fixture(scope="module")
def handles():
    from linear_cross_entropy_token_gb300 import FLCE
    hs = {c: FLCE("bf16", 0, hbm_budget_bytes=2 << 30, cta=c) for c in SHAPES}
    yield hs
    for h in hs.values():
        h.close()


def _case(i):
    g = np.random.default_rng(7000 + i)
    N = int(g.integers(1, 3000))
    H = 8 * int(g.integers(1, 97))
    V = int(g.integers(1, 20000))
    ign = float(g.choice([0.0, 0.05, 0.3]))
    chunk = int(g.choice([0, 64, 128, 384, 1000]))
    targets = "zipf" if i % 2 else "uniform"
    return N, H, V, ign, chunk, targets


@pytest.mark.parametrize("i", range(30))
def test_random_case(handles, i):
    N, H, V, ign, chunk, targets = _case(i)
    w = workloads.generate(workloads.custom(N, H, V, "bf16", targets=targets, ignore_frac=ign,
                                            seed=i))
    ref = oracle.flce_reference(w.x_f64(), w.W_f64(), w.t, w.ignore_index)
    res = run(handles[SHAPES[i % len(SHAPES)]], w, chunk=chunk)
    assert_parity(res, ref, "bf16", token_rtol=1e-3)
