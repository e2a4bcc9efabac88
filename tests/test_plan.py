"""Host-side kernel selection (lr_plan_info, no device): which carry protocol
each shape plans.  The GPU parity tests pick their shapes to run every
protocol; these checks pin that the shapes they name really take them, and
the bounds between the protocols.  CPU only."""
import pytest

import linear_recurrence_scan_chunked_gb300 as lrs


@pytest.fixture(scope="module", autouse=True)
def lib():
    lrs.build()
    return lrs.load()


def plan(op, dtype, vec, T, B, D):
    return lrs.plan_info(op, dtype, vec, T, B * D)


@pytest.mark.parametrize("op", ["scan_fwd", "scan_bwd"])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_scans_up_to_2048_steps_take_the_cluster_kernel(op, dtype):
    for vec in (True, False):
        for T, ch in ((1, 1), (128, 1), (129, 2), (1024, 8), (1025, 9), (2048, 16)):
            p = plan(op, dtype, vec, T, 4, 256)
            assert p == {"protocol": "cluster", "tma": False, "tile_rows": 128, "n_chunks": ch}, (T, p)
    # the tiny-scan configuration, and many channel tiles of one chunk
    assert plan(op, dtype, True, 1024, 4, 256)["protocol"] == "cluster"
    assert plan(op, dtype, True, 64, 40, 1000)["protocol"] == "cluster"
    # ragged channel tiles on the vector path
    assert plan(op, dtype, True, 300, 1, 20)["protocol"] == "cluster"
    assert plan(op, dtype, True, 1000, 3, 12)["protocol"] == "cluster"
    # one step more: the scans' other protocols
    assert plan(op, dtype, True, 2049, 4, 256)["protocol"] != "cluster"


def test_the_scans_other_protocols_on_the_parity_shapes():
    # look-back past the cluster kernel (TMA tiles of 32 fp32 rows)
    assert plan("scan_fwd", "f32", True, 2100, 2, 256) == {"protocol": "look", "tma": True,
                                                            "tile_rows": 32, "n_chunks": 66}
    assert plan("scan_bwd", "f32", True, 2100, 2, 256)["protocol"] == "look"
    assert plan("scan_fwd", "f32", True, 3001, 2, 100)["protocol"] == "look"
    # strip (chain protocol on TMA tiles, 135 channel tiles of 128), and the
    # strip case of the allocation-free entry's test and of smoke
    for T, B, D, dt in ((2100, 33, 520, "f32"), (2100, 16, 1024, "bf16"), (2100, 16, 1024, "f32")):
        p = plan("scan_fwd", dt, True, T, B, D)
        assert (p["protocol"], p["tma"]) == ("chain", True), (T, B, D, dt)
    # register chain: the scalar path
    p = plan("scan_fwd", "f32", False, 2100, 3, 7)
    assert (p["protocol"], p["tma"]) == ("chain", False)
    # past the look-back budget (n_chunks^2 * channel tiles): the TMA chain
    p = plan("scan_fwd", "f32", True, 4097, 2, 128)
    assert (p["protocol"], p["tma"]) == ("chain", True)
    # long and narrow: walkers (the million-step configuration)
    assert plan("scan_fwd", "f32", True, 1 << 20, 1, 128)["protocol"] == "walk"
    assert plan("scan_fwd", "f32", True, 20000, 1, 128)["protocol"] == "walk"
    # the large-batch configuration: wide, the strip kernel
    p = plan("scan_fwd", "bf16", True, 8192, 16, 4096)
    assert (p["protocol"], p["tma"]) == ("chain", True)


@pytest.mark.parametrize("op", ["sru_fwd", "sru_bwd", "lstm_fwd", "lstm_bwd", "deer", "deer_bwd",
                                "deer_ode"])
def test_the_cells_and_deer_never_take_the_cluster_kernel(op):
    for T, B, D in ((1, 1, 4), (64, 1, 128), (300, 2, 256), (1024, 4, 256), (64, 40, 1000)):
        for vec in (True, False):
            assert plan(op, "f32", vec, T, B, D)["protocol"] != "cluster", (op, T, B, D, vec)


def test_the_deer_and_sru_configurations():
    p = plan("deer", "f32", True, 65536, 4, 256)
    assert (p["protocol"], p["tma"]) == ("walk", True)  # segmented walker, one-pass iterations
    p = plan("sru_fwd", "f32", True, 2048, 32, 1024)
    assert (p["protocol"], p["tma"]) == ("chain", True)  # strip kernel


def test_argument_errors():
    for args in (("scan_fwd", "f16", True, 10, 10), ("scan_fwd", "f32", True, 0, 10),
                 ("scan_fwd", "f32", True, 10, 0), ("scan_fwd", "f32", True, -1, 10)):
        with pytest.raises(ValueError):
            lrs.plan_info(*args)
    lib = lrs.load()
    assert lib.lr_plan_info(9, 0, 1, 10, 10, None, None, None, None) == lrs.LR_ERR_INVALID_ARG
    assert lib.lr_plan_info(-1, 0, 1, 10, 10, None, None, None, None) == lrs.LR_ERR_INVALID_ARG
    assert lib.lr_plan_info(0, 0, 1, 10, 10, None, None, None, None) == lrs.LR_OK
