"""The C-ABI library: it loads, exports every function include/flce.h declares,
and its host-only logic (the token-chunk planner) does what it states. No
compute call runs here."""
import ctypes
import os

import pytest

from linear_cross_entropy_token_gb300 import build as flce_build
from linear_cross_entropy_token_gb300 import flce


@pytest.fixture(scope="module")
def lib():
    flce_build.build()
    return flce.load()


def test_exports_every_declared_function(lib):
    names = flce.header_functions()
    assert len(names) >= 18
    for n in names:
        assert hasattr(lib, n), f"libflce.so does not export {n}"


def test_abi_version_and_status_strings(lib):
    assert lib.flce_abi_version() == 5
    assert lib.flce_status_string(0) == b"FLCE_OK"
    assert lib.flce_status_string(4) == b"FLCE_ERR_BAD_TARGET"
    assert lib.flce_kernel_name(1) == b"gemm_logits_lse"
    assert lib.flce_kernel_name(99) == b"?"
    for k, name in enumerate(flce.KERNEL_KINDS):
        assert lib.flce_kernel_name(k).decode() == name


def test_library_is_built_for_sm103a_only():
    """build() compiles one -gencode, for compute capability 10.3."""
    assert flce_build.ARCH == ["-gencode", "arch=compute_103a,code=sm_103a"]


@pytest.mark.skipif(os.environ.get("CUDA_VISIBLE_DEVICES") is None and
                    __import__("torch").cuda.is_available(), reason="a GPU is present")
def test_create_without_gpu_is_unsupported(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    cfg = flce.make_config("bf16", 0)
    h = ctypes.c_void_p()
    st = lib.flce_create(ctypes.byref(h), ctypes.byref(cfg))
    assert st == 2 and not h.value   # FLCE_ERR_UNSUPPORTED, no handle
    with pytest.raises(flce.FlceError):
        flce.FLCE("bf16", 0)


def test_null_handle_calls_fail_cleanly(lib):
    loss = ctypes.c_float()
    assert lib.flce_forward_backward(None, None, None, None, 1, 8, 8, -100, 0, ctypes.byref(loss),
                                     None, None, None) == 1
    assert lib.flce_launch_count(None) == 0
    assert lib.flce_workspace_bytes(None, 16, 8, 8, 0) == 0
    assert lib.flce_last_error(None) == b"null handle"
    lib.flce_destroy(None)


# ---------------------------------------------------------------- planner

GiB = 1 << 30


def test_plan_llama3_default_budget():
    p = flce.plan(16384, 4096, 128256, "bf16")
    assert p["chunk"] == 4096 and p["num_chunks"] == 4
    assert p["vocab_tiles"] == 2004 and p["ldv"] == 128256   # a partial per 64 columns
    assert p["logits_bytes"] == 4096 * 128256 * 2
    assert p["workspace_bytes"] <= int(1.25 * GiB)
    # wide CTA-pair tiles for all three GEMMs at this shape (long reductions)
    assert (p["tile_m"], p["tile_n"], p["tile_n_dx"], p["tile_n_dw"]) == (256, 512, 512, 512)
    # dx and dW in one dynamically scheduled launch: the long dx units need
    # no split, the short dW units fill in behind them
    assert (p["backward_one_launch"], p["dx_splits"]) == (1, 1)
    sep = flce.plan(16384, 4096, 128256, "bf16", backward="separate")
    assert sep["dx_splits"] == 4        # 128 wide dx tiles on 76 SM pairs: 4 splits fill the waves
    q = flce.plan(16384, 4096, 128256, "bf16", cta="pair")
    assert (q["tile_n"], q["dx_splits"]) == (256, 2)   # 256 tiles of 256 x 256: 2 splits


def test_plan_long_context_stays_O_CV():
    p = flce.plan(131072, 4096, 128256, "bf16")
    full_logits = 131072 * 128256 * 2
    assert p["num_chunks"] * p["chunk"] >= 131072
    assert p["workspace_bytes"] <= int(1.25 * GiB) < full_logits / 20
    assert p["chunk"] % 128 == 0


def test_plan_explicit_chunk_and_budget():
    p = flce.plan(256, 128, 4096, "fp32", chunk=64)
    # the fp32 dx GEMM (64 x 128 output, two 64 x 64 tiles) splits its 4096-deep
    # reduction 32 ways to fill the SMs; its partials sit in the workspace
    assert (p["chunk"], p["num_chunks"], p["dx_splits"]) == (64, 4, 32)
    assert p["logits_bytes"] == 64 * 4096 * 4
    assert p["workspace_bytes"] >= p["logits_bytes"] + 32 * 64 * 128 * 4
    # a large output needs no split
    assert flce.plan(4096, 4096, 32000, "fp32")["dx_splits"] == 1
    p = flce.plan(16384, 4096, 151936, "bf16", chunk=8192, hbm_budget_bytes=4 * GiB)
    assert p["chunk"] == 8192 and p["num_chunks"] == 2
    with pytest.raises(flce.FlceError) as e:
        flce.plan(16384, 4096, 151936, "bf16", chunk=8192)   # 2.5 GB > default 1.25 GiB
    assert e.value.status_name == "FLCE_ERR_BUDGET"
    with pytest.raises(flce.FlceError) as e:
        flce.plan(16384, 4096, 151936, "bf16", hbm_budget_bytes=1 << 20)
    assert e.value.status_name == "FLCE_ERR_BUDGET"


def test_plan_small_and_ragged():
    p = flce.plan(2048, 1024, 32000, "bf16")
    assert p["chunk"] == 2048 and p["num_chunks"] == 1
    p = flce.plan(1000, 64, 4099, "bf16", chunk=300)
    assert (p["chunk"], p["num_chunks"], p["ldv"], p["vocab_tiles"]) == (300, 4, 4160, 65)
    p = flce.plan(50, 64, 100, "bf16")
    assert p["chunk"] == 50 and p["num_chunks"] == 1
    p = flce.plan(0, 64, 100, "bf16")
    assert p["chunk"] == 0 and p["num_chunks"] == 0


def test_plan_balances_chunks():
    for N in (5000, 16384, 40000, 131072):
        p = flce.plan(N, 4096, 128256, "bf16")
        last = N - (p["num_chunks"] - 1) * p["chunk"]
        assert 0 < last <= p["chunk"]
        # no chunk is more than one 128-token tile longer than an even split
        assert p["chunk"] - N / p["num_chunks"] < 128


def test_plan_slabs_bounded_in_V():
    """SLABS: the chunk buffer holds one vocabulary slab (a multiple of 512
    columns, at most 256 MiB and what the budget leaves), so the workspace
    no longer grows with V."""
    p = flce.plan(16384, 4096, 128256, "bf16", dlogits_mode="slabs")
    vs = p["vocab_slab"]
    assert vs % 512 == 0 and p["chunk"] * vs * 2 <= 256 << 20
    assert p["ldv"] == vs and p["logits_bytes"] == p["chunk"] * vs * 2
    assert p["dx_splits"] == 1
    # 256-row x 512-column tiles on 76 SM pairs: the slab is narrowed from
    # 32768 to 29184 columns, where the dlogits GEMM (16 x 57 tiles) and the
    # dW GEMM (114 x 8 tiles) both run 912 units, 12 full waves of 76
    assert (p["chunk"], vs) == (4096, 29184)
    inplace = flce.plan(16384, 4096, 128256, "bf16")
    assert p["workspace_bytes"] < inplace["workspace_bytes"] / 3
    # doubling V changes only the per-token log-sum-exp partials
    q = flce.plan(16384, 4096, 256512, "bf16", dlogits_mode="slabs", chunk=p["chunk"])
    assert q["vocab_slab"] == vs
    assert q["workspace_bytes"] - p["workspace_bytes"] <= p["chunk"] * 8 * (q["vocab_tiles"] - p["vocab_tiles"]) + 4096
    # small budgets shorten the chunk before they narrow the slab below 8192
    for mib, chunk, slab in ((128, 3328, 11776), (64, 1920, 9216), (24, 640, 11264)):
        r = flce.plan(16384, 4096, 128256, "bf16", dlogits_mode="slabs", hbm_budget_bytes=mib << 20)
        assert (r["chunk"], r["vocab_slab"]) == (chunk, slab)
        assert r["workspace_bytes"] <= mib << 20
    # an explicit chunk above 4096 tokens is clamped to 4096
    assert flce.plan(16384, 4096, 128256, "bf16", dlogits_mode="slabs", chunk=16384)["chunk"] == 4096
    with pytest.raises(flce.FlceError) as e:
        flce.plan(16384, 4096, 128256, "bf16", dlogits_mode="slabs", hbm_budget_bytes=64 << 20, chunk=4096)
    assert e.value.status_name == "FLCE_ERR_BUDGET"
    # a vocabulary narrower than the slab room is one slab
    s = flce.plan(2048, 1024, 4000, "bf16", dlogits_mode="slabs")
    assert s["vocab_slab"] == 4000 and s["ldv"] == 4032
    # fp32: the same walk on the CUDA-core path, 4-byte buffer entries
    f = flce.plan(256, 128, 4096, "fp32", chunk=64, dlogits_mode="slabs", hbm_budget_bytes=300 << 10)
    assert (f["chunk"], f["vocab_slab"], f["dx_splits"]) == (64, 1024, 1)
    assert f["logits_bytes"] == 64 * 1024 * 4 and f["workspace_bytes"] <= 300 << 10


def test_plan_rejects_bad_sizes():
    for args in ((-1, 8, 8), (8, 0, 8), (8, 8, 0)):
        with pytest.raises(flce.FlceError) as e:
            flce.plan(*args)
        assert e.value.status_name == "FLCE_ERR_INVALID_ARG"


def test_plan_invariants_over_extreme_shapes():
    """Every plan the SLABS and in-place planners return covers all tokens,
    fits its budget, keeps 64-column-aligned rows and a slab that is V or a
    multiple of 512; a budget too small is the only refusal."""
    import itertools
    for N, H, V, budget, dt, cta, mode in itertools.product(
            [1, 100, 16384, 131072], [8, 4096, 16384], [1, 300, 4099, 262147],
            [0, 32 << 20, 8 << 30], ["bf16", "fp32"], ["auto", "single"], ["slabs", "inplace"]):
        if dt == "fp32" and cta != "auto":
            continue
        try:
            p = flce.plan(N, H, V, dt, hbm_budget_bytes=budget, dlogits_mode=mode, cta=cta)
        except flce.FlceError as e:
            assert e.status_name == "FLCE_ERR_BUDGET", (N, H, V, budget, dt, cta, mode)
            continue
        vs = p["vocab_slab"]
        assert vs == V or (mode == "slabs" and vs % 512 == 0 and vs < V)
        assert p["workspace_bytes"] <= (budget or int(1.25 * GiB))
        assert p["num_chunks"] * p["chunk"] >= N > (p["num_chunks"] - 1) * p["chunk"]
        assert p["ldv"] % 64 == 0 and p["ldv"] >= vs
        assert p["dlogits"] == mode


def test_backward_launch_invariants_over_shapes():
    """The backward fields of every plan agree with one another: a plan that
    runs the dx and dW GEMMs in one launch runs them on one tile shape and
    puts nothing on the second stream; only CTA-pair bf16 plans in the
    in-place and recompute modes take either form; the dx split stays within
    1..8; and the default takes one launch exactly where dW runs wide."""
    import itertools
    for N, H, V, cta, backward, mode in itertools.product(
            [1, 300, 2048, 16384], [8, 256, 1024, 4096], [300, 4099, 32000, 151936],
            ["auto", "single", "pair", "wide"], ["auto", "separate", "one_launch"],
            ["inplace", "recompute", "slabs"]):
        p = flce.plan(N, H, V, cta=cta, backward=backward, dlogits_mode=mode,
                      hbm_budget_bytes=4 * GiB)
        one, beside = p["backward_one_launch"], p["dw_beside_dx"]
        assert one in (0, 1) and beside in (0, 1) and not (one and beside)
        assert 1 <= p["dx_splits"] <= 8
        if one:
            assert p["tile_n_dx"] == p["tile_n_dw"]
        if cta == "single" or mode == "slabs" or backward == "separate":
            assert one == 0, (N, H, V, cta, backward, mode)
        if cta == "single" or mode == "slabs":
            assert beside == 0
        if backward == "one_launch" and cta != "single" and mode != "slabs":
            assert one == 1
        if backward == "auto" and cta in ("auto", "wide") and mode != "slabs":
            assert one == (1 if p["tile_n_dw"] == 512 else 0), (N, H, V, cta, mode, p)


def test_plan_reports_the_mode_it_runs():
    """AUTO resolves to INPLACE; an fp32 handle runs RECOMPUTE in place."""
    assert flce.plan(4096, 1024, 32000)["dlogits"] == "inplace"
    assert flce.plan(4096, 1024, 32000, dlogits_mode="recompute")["dlogits"] == "recompute"
    assert flce.plan(4096, 1024, 32000, dtype="fp32", dlogits_mode="recompute")["dlogits"] == "inplace"
    assert flce.plan(4096, 1024, 32000, dlogits_mode="slabs")["dlogits"] == "slabs"


def test_plan_refuses_a_tile_shape_that_does_not_exist(lib):
    cfg = flce.make_config("bf16", 0)
    cfg.cta_pair = 3
    p = flce.Plan()
    assert lib.flce_make_plan(ctypes.byref(cfg), 1024, 256, 1000, 0, 0, ctypes.byref(p)) == 1


def test_plan_picks_tile_shapes_per_gemm():
    """The default handle times wide (256 x 512) against pair (256 x 256)
    tiles per GEMM with a model and takes pair tiles only where they win by
    more than 5%: where a wide tile would waste half its columns (H = 256:
    dx and dW), or leave a short dx launch with too few units; the logits
    GEMM stays wide. An explicit tile shape applies to every GEMM."""
    p = flce.plan(2048, 1024, 32000)
    assert (p["tile_n"], p["tile_n_dx"], p["tile_n_dw"]) == (512, 512, 512)
    n = flce.plan(2048, 256, 32000)
    assert (n["tile_n"], n["tile_n_dx"], n["tile_n_dw"], n["dx_splits"]) == (512, 256, 256, 8)
    q = flce.plan(2048, 1024, 32000, cta="wide")
    assert (q["tile_n"], q["tile_n_dx"], q["tile_n_dw"]) == (512, 512, 512)
    r = flce.plan(2048, 1024, 32000, cta="pair")
    assert (r["tile_n"], r["tile_n_dx"], r["tile_n_dw"]) == (256, 256, 256)
    # the slab walk keeps the wide tiles its slab sizing assumes
    s = flce.plan(16384, 4096, 128256, dlogits_mode="slabs")
    assert (s["tile_n"], s["tile_n_dx"], s["tile_n_dw"]) == (512, 512, 512)
    # wide dx and dW GEMMs share one dynamically scheduled launch by default;
    # separate launches put the small shape's 64-unit dx launch beside dW,
    # not the Llama-3 shape's 512-unit one; single-CTA tiles do neither
    assert (p["backward_one_launch"], p["dw_beside_dx"]) == (1, 0)
    # one launch of 48 dx units (16 tiles x 3 splits) and 250 dW units: three
    # splits keep the longest dx unit under the launch's work per SM pair
    assert p["dx_splits"] == 3
    assert (q["backward_one_launch"], r["backward_one_launch"], n["backward_one_launch"]) == (1, 0, 0)
    sep = flce.plan(2048, 1024, 32000, backward="separate")
    assert (sep["backward_one_launch"], sep["dw_beside_dx"]) == (0, 1)
    assert flce.plan(16384, 4096, 128256, backward="separate")["dw_beside_dx"] == 0
    assert flce.plan(16384, 4096, 128256)["backward_one_launch"] == 1
    one = flce.plan(2048, 256, 32000, backward="one_launch")   # one launch on dx's pair tiles
    assert (one["backward_one_launch"], one["tile_n_dx"], one["tile_n_dw"]) == (1, 256, 256)
    single = flce.plan(2048, 1024, 32000, cta="single", backward="one_launch")
    assert (single["backward_one_launch"], single["dw_beside_dx"]) == (0, 0)
    assert flce.plan(16384, 4096, 128256, dlogits_mode="slabs")["backward_one_launch"] == 0
