"""Parity with the fp64 oracle on seeded random shapes: token counts, hidden
sizes (multiples of 8), vocabulary sizes, ignore fractions, target
distributions and chunk sizes drawn per case, rotating over the tile shapes (the
default picks wide or pair tiles per GEMM; wide tiles also with the dx and dW
GEMMs in one dynamically scheduled launch), one
handle per shape reused across the cases (workspace growth, cached tile
orders, changing tensor maps)."""
import numpy as np
import pytest

import oracle
import workloads
from flce_testing import assert_parity, run

pytestmark = pytest.mark.gpu

SHAPES = ("single", "pair", "wide", "auto", "wide-one_launch")


@pytest.fixture(scope="module")
def handles():
    from linear_cross_entropy_token_gb300 import FLCE
    hs = {}
    for c in SHAPES:
        cta, _, backward = c.partition("-")
        hs[c] = FLCE("bf16", 0, hbm_budget_bytes=2 << 30, cta=cta, backward=backward or "auto")
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


@pytest.fixture(scope="module")
def slab_handles():
    """Slab-mode handles with a 2 MiB budget, so that most random shapes
    run several vocabulary slabs per chunk."""
    from linear_cross_entropy_token_gb300 import FLCE
    hs = {c: FLCE("bf16", 0, hbm_budget_bytes=2 << 20, cta=c, dlogits_mode="slabs") for c in ("wide", "single")}
    yield hs
    for h in hs.values():
        h.close()


@pytest.mark.parametrize("i", range(12))
def test_random_case_slabs(slab_handles, i):
    from linear_cross_entropy_token_gb300 import FlceError
    N, H, V, ign, chunk, targets = _case(100 + i)
    w = workloads.generate(workloads.custom(N, H, V, "bf16", targets=targets, ignore_frac=ign,
                                            seed=100 + i))
    h = slab_handles["wide" if i % 2 else "single"]
    try:
        res = run(h, w, chunk=chunk)
    except FlceError as e:       # an explicit chunk too long for the 2 MiB budget
        assert e.status_name == "FLCE_ERR_BUDGET" and chunk > 0
        res = run(h, w)
    ref = oracle.flce_reference(w.x_f64(), w.W_f64(), w.t, w.ignore_index)
    assert_parity(res, ref, "bf16", token_rtol=1e-3)
