"""The library's host planner (oop_out_prod_plan), with no GPU: which kernels
an OUT_PROD call enqueues on a 152-SM GB300.  The launchers take their
decisions from the same functions, and the GPU tests check the launch counts
of real calls.

The expected schedules are the winners of timings on a GB300 with both tile
schedules forced (median of 20 calls after an L2 flush, microseconds, data-
parallel / stream-K); near ties are left out."""

import pytest

import ggml_out_prod_gb300 as op

F32, Q8, Q4 = 0, 8, 2
SMS = 152


@pytest.fixture(scope="module", autouse=True)
def built():
    op.build()
    op.lib()
    op.oop_debug_set_tc_schedule(0)
    yield
    op.oop_debug_set_tc_schedule(0)


def plan(a_type, ne_a, ne_b, **kw):
    return op.out_prod_plan(a_type, ne_a, ne_b, kw.pop("sms", SMS), **kw)


def dense(t, m, k, n, slices=1):
    return t, (m, k, 1, 1), (n, k, slices, 1)


# (a_type, ne_a, ne_b), measured data-parallel / stream-K in microseconds
# (128 x 128 tiles; stream-K runs the full waves as whole tiles first)
DATA_PARALLEL_WINS = [
    ((F32, (128, 512, 4, 1), (128, 512, 16, 1)), (36.9, 42.0)),    # grouped heads, 1 sequence
    ((F32, (128, 512, 4, 2), (128, 512, 16, 2)), (38.9, 46.1)),    # grouped heads, 2 sequences
    (dense(Q8, 1536, 1536, 1024), (65.5, 76.8)),
]
STREAM_K_WINS = [
    (dense(Q8, 512, 4096, 256), (135.1, 44.0)),
    (dense(F32, 256, 2048, 96), (79.9, 46.0)),
    (dense(F32, 512, 1024, 192), (49.2, 39.9)),
    (dense(F32, 128, 8192, 128), (253.9, 62.4)),
    (dense(Q8, 1024, 2048, 512), (77.8, 54.3)),
    (dense(F32, 256, 512, 128), (38.8, 33.9)),
    (dense(Q8, 1024, 1024, 256), (51.2, 42.0)),
    (dense(F32, 128, 2048, 96), (79.9, 44.0)),
    (dense(Q8, 2048, 2048, 384), (79.8, 62.5)),
    (dense(F32, 640, 4096, 192), (135.2, 48.1)),
    (dense(Q8, 1536, 1536, 256), (63.5, 48.1)),
    (dense(Q8, 5120, 5120, 1024), (475.1, 369.7)),
    (dense(Q8, 5120, 17408, 1024), (1520.6, 1152.0)),
    (dense(Q8, 17408, 5120, 1024), (1231.9, 1160.2)),
]


@pytest.mark.parametrize("shape,times", DATA_PARALLEL_WINS)
def test_schedule_data_parallel_where_it_measured_faster(shape, times):
    assert times[0] < times[1]
    p = plan(*shape)
    assert p["kernel"] == op.KERNEL_TC_DATA_PARALLEL and p["ctas"] == 0 and p["launches"] == 2


@pytest.mark.parametrize("shape,times", STREAM_K_WINS)
def test_schedule_stream_k_where_it_measured_faster(shape, times):
    assert times[1] < times[0]
    p = plan(*shape)
    assert p["kernel"] == op.KERNEL_TC_STREAM_K and p["launches"] == 3
    assert 1 <= p["ctas"] <= SMS


@pytest.mark.parametrize("m,k", [(5120, 5120), (5120, 17408), (17408, 5120)])
def test_headline_shapes_take_stream_k(m, k):
    """320 / 320 / 1088 tiles: 2.1, 2.1 and 7.2 waves, the last ones 11%,
    11% and 16% full; stream-K runs the full waves as whole tiles and splits
    only the 16 / 16 / 24 tail tiles."""
    for t in (Q8, Q4):
        p = plan(*dense(t, m, k, 1024))
        assert p["kernel"] == op.KERNEL_TC_STREAM_K and p["ctas"] == SMS


def test_whole_waves_stay_data_parallel():
    # 304 tiles = two full waves: nothing to split, even when stream-K is forced
    shape = dense(Q8, 128 * 38, 4096, 1024)
    assert plan(*shape)["kernel"] == op.KERNEL_TC_DATA_PARALLEL
    try:
        op.oop_debug_set_tc_schedule(2)
        assert plan(*shape)["kernel"] == op.KERNEL_TC_DATA_PARALLEL
    finally:
        op.oop_debug_set_tc_schedule(0)


def test_minimum_workspace_and_forced_schedules():
    shape = dense(F32, 128, 8192, 128)
    need = op.oop_out_prod_workspace_min_size(*shape)
    assert plan(*shape, workspace_bytes=need)["kernel"] == op.KERNEL_TC_DATA_PARALLEL
    assert op.oop_out_prod_plan(*shape, 0, SMS, need - 256)[0] == op.ERR_WORKSPACE
    try:
        op.oop_debug_set_tc_schedule(1)
        assert plan(*shape)["kernel"] == op.KERNEL_TC_DATA_PARALLEL
        op.oop_debug_set_tc_schedule(2)
        p = plan(*dense(Q8, 5120, 5120, 1024))
        assert p["kernel"] == op.KERNEL_TC_STREAM_K and p["ctas"] == SMS
    finally:
        op.oop_debug_set_tc_schedule(0)


def test_stream_k_ctas_never_exceed_the_iterations():
    # one tile of one k-block: at most one CTA
    p = plan(*dense(F32, 100, 20, 50))
    assert p["ctas"] in (0, 1)
    p = plan(*dense(F32, 128, 2048, 96))          # 64 iterations
    assert p["ctas"] == 64


def test_path_choice():
    assert plan(F32, (256, 512, 1, 1), (8, 512, 1, 1))["path"] == op.PATH_SKINNY
    assert plan(F32, (256, 512, 1, 1), (32, 512, 1, 1))["path"] == op.PATH_SKINNY
    assert plan(F32, (256, 512, 1, 1), (33, 512, 1, 1))["path"] == op.PATH_TCGEN05
    assert plan(Q8, (256, 512, 1, 1), (8, 512, 1, 1))["path"] == op.PATH_TCGEN05
    assert plan(Q4, (256, 512, 1, 1), (8, 512, 1, 1))["path"] == op.PATH_TCGEN05
    p = plan(Q8, (256, 512, 1, 1), (8, 512, 1, 1), path=op.PATH_SIMT)
    assert p["kernel"] == op.KERNEL_SIMT and p["launches"] == 1
    assert op.oop_out_prod_plan(Q8, (256, 512, 1, 1), (8, 512, 1, 1), op.PATH_SKINNY, SMS, 0)[0] \
        == op.ERR_PATH


@pytest.mark.parametrize("ne_a,ne_b,kernel,item_m", [
    # a single LoRA gradient: 20 items of 128 m, too few for the persistent form
    ((2560, 512, 1, 1), (8, 512, 1, 1), op.KERNEL_SKINNY, 0),
    ((2560, 512, 1, 1), (24, 512, 1, 1), op.KERNEL_SKINNY, 0),
    # 64 gradients: 1280 items of 128 m (rank 24: 109 us at 128 m, 150 us at 64)
    ((2560, 512, 64, 1), (8, 512, 64, 1), op.KERNEL_SKINNY_TMA, 128),
    ((2560, 512, 64, 1), (24, 512, 64, 1), op.KERNEL_SKINNY_TMA, 128),
    # N = 28, 32: 64-wide items (four m per lane do not fit in the registers)
    ((2560, 512, 64, 1), (28, 512, 64, 1), op.KERNEL_SKINNY_TMA, 64),
    ((2560, 512, 64, 1), (32, 512, 64, 1), op.KERNEL_SKINNY_TMA, 64),
    # rank 24 with 256 items of 128 m but 512 of 64: 64-wide (230 us against
    # 320 us for the register kernel)
    ((4096, 4096, 8, 1), (24, 4096, 8, 1), op.KERNEL_SKINNY_TMA, 64),
    ((1000, 130, 20, 1), (24, 130, 20, 1), op.KERNEL_SKINNY_TMA, 64),
    # N = 16 has no 64-wide fallback: 160 items of 128 m -> register kernel
    ((1000, 130, 20, 1), (16, 130, 20, 1), op.KERNEL_SKINNY, 0),
    ((1000, 300, 40, 1), (8, 300, 40, 1), op.KERNEL_SKINNY_TMA, 128),
    # the TMA form needs N % 4 == 0 and M % 4 == 0
    ((2560, 512, 64, 1), (6, 512, 64, 1), op.KERNEL_SKINNY, 0),
    ((2562, 512, 64, 1), (8, 512, 64, 1), op.KERNEL_SKINNY, 0),
])
def test_skinny_kernel_choice(ne_a, ne_b, kernel, item_m):
    p = plan(F32, ne_a, ne_b)
    assert p["path"] == op.PATH_SKINNY and p["launches"] == 1
    assert (p["kernel"], p["item_m"]) == (kernel, item_m)


def test_skinny_threshold_follows_the_sm_count():
    """Two items per SM: 160 items of 128 m take the persistent form on an
    80-SM part and not on 152 SMs."""
    shape = (F32, (2560, 512, 8, 1), (8, 512, 8, 1))
    assert plan(*shape, sms=80)["kernel"] == op.KERNEL_SKINNY_TMA
    assert plan(*shape, sms=SMS)["kernel"] == op.KERNEL_SKINNY


def test_empty_and_k_zero():
    p = plan(F32, (256, 512, 1, 1), (0, 512, 1, 1))
    assert p == {"path": 0, "kernel": op.KERNEL_NONE, "item_m": 0, "ctas": 0, "launches": 0}
    p = plan(Q8, (256, 0, 1, 1), (64, 0, 1, 1))
    assert p["kernel"] == op.KERNEL_NONE and p["launches"] == 0 and p["path"] == op.PATH_TCGEN05


def test_argument_errors():
    assert op.oop_out_prod_plan(F32, (256, 512, 1, 1), (8, 512, 1, 1), 0, 0, 0)[0] == op.ERR_DEVICE
    assert op.oop_out_prod_plan(F32, (256, 512, 1, 1), (8, 511, 1, 1), 0, SMS, 0)[0] == op.ERR_SHAPE
    assert op.oop_out_prod_plan(F32, (256, 512, 3, 1), (8, 512, 4, 1), 0, SMS, 0)[0] \
        == op.ERR_BROADCAST
    assert op.oop_out_prod_plan(F32, (256, 512, 1, 1), (8, 512, 1, 1), 9, SMS, 0)[0] == op.ERR_PATH
    L = op.lib()
    assert L.oop_out_prod_plan(F32, op._ne((256, 512, 1, 1)), op._ne((8, 512, 1, 1)), 0, SMS, 0,
                               None) == op.ERR_NULL
