"""The library's size queries on CPU (pure host code): the invariants their
documentation states, on shapes of every kind the workloads use."""

import pytest

import ggml_out_prod_gb300 as op

F32, Q8, Q4, BF16 = 0, 8, 2, 30
SLOT = 2 * 128 * 128 * 4           # two 128 x 128 fp32 partial tiles per stream-K CTA

SHAPES = [
    (F32, (256, 512, 1, 1), (8, 512, 1, 1)),
    (F32, (2560, 512, 64, 1), (24, 512, 64, 1)),
    (F32, (128, 512, 4, 2), (128, 512, 16, 2)),
    (Q8, (5120, 5120, 1, 1), (1024, 5120, 1, 1)),
    (Q4, (17408, 5120, 1, 1), (1024, 5120, 1, 1)),
    (F32, (200, 301, 2, 1), (70, 301, 4, 3)),
    (F32, (128, 8192, 1, 1), (128, 8192, 1, 1)),
]


def _bytes(a_type, ne_a, ne_b):
    m, k, a2, a3 = ne_a
    n, _, b2, b3 = ne_b
    a = {F32: 4 * m, Q8: m // 32 * 34, Q4: m // 32 * 18}[a_type] * k * a2 * a3
    return a, 4 * n * k * b2 * b3, 4 * m * n * b2 * b3


@pytest.fixture(scope="module", autouse=True)
def built():
    op.build()
    op.lib()


@pytest.mark.parametrize("a_type,ne_a,ne_b", SHAPES)
def test_workspace_sizes(a_type, ne_a, ne_b):
    full = op.oop_out_prod_workspace_size(a_type, ne_a, ne_b)
    least = op.oop_out_prod_workspace_min_size(a_type, ne_a, ne_b)
    n, k, b2, b3 = ne_b
    assert full % 256 == 0 and least % 256 == 0
    # the minimum holds the TF32 split of src1: hi and lo words of every element
    assert least >= 2 * 4 * n * k * b2 * b3
    assert least < 2 * 4 * n * (k + 4) * b2 * b3 + 2 * 256
    # the rest holds two partial tiles for each of at most 160 stream-K CTAs
    assert (full - least) % SLOT == 0 and 1 <= (full - least) // SLOT <= 160


def _host_chunks(a_type, ne_a, ne_b):
    # the host entry's k chunks: one slice, not the skinny-N f32 case, >= 256 rows each
    single = ne_a[2] * ne_a[3] == 1 and ne_b[2] * ne_b[3] == 1
    if not single or (a_type == F32 and ne_b[0] <= 32):
        return 1
    return max(1, min(4, ne_a[1] // 256))


@pytest.mark.parametrize("a_type,ne_a,ne_b", SHAPES)
def test_host_buffer_holds_every_tensor(a_type, ne_a, ne_b):
    a, b, dst = _bytes(a_type, ne_a, ne_b)
    ws = op.oop_out_prod_workspace_size(a_type, ne_a, ne_b)
    total = op.oop_out_prod_host_buffer_size(a_type, ne_a, ne_b)
    parts = (_host_chunks(a_type, ne_a, ne_b) - 1) * -(-dst // 256) * 256
    assert total % 256 == 0
    assert a + b + dst + ws + parts <= total <= a + b + dst + ws + parts + 4 * 255


@pytest.mark.parametrize("a_type,ne_a,ne_b", [
    (F32, (256, 512, 1, 1), (8, 511, 1, 1)),       # K mismatch
    (Q8, (100, 64, 1, 1), (64, 64, 1, 1)),         # quantised M not a multiple of 32
    (F32, (256, 512, 3, 1), (8, 512, 4, 1)),       # no exact broadcast
    (9, (256, 512, 1, 1), (8, 512, 1, 1)),         # q8_1: not a src0 type
    (12, (128, 512, 1, 1), (8, 512, 1, 1)),        # q4_K needs M % 256
    (F32, (256, -1, 1, 1), (8, -1, 1, 1)),         # negative size
])
def test_invalid_shapes_size_zero(a_type, ne_a, ne_b):
    assert op.oop_out_prod_workspace_size(a_type, ne_a, ne_b) == 0
    assert op.oop_out_prod_workspace_min_size(a_type, ne_a, ne_b) == 0
    assert op.oop_out_prod_host_buffer_size(a_type, ne_a, ne_b) == 0


def test_mul_mat_id_back_workspace():
    ne_w, ne_ids = (2048, 768, 32), (8, 512)
    for wt in (F32, BF16):
        ws = op.oop_mul_mat_id_back_workspace_size(wt, ne_w, ne_ids)
        # at least the TF32 split (hi and lo) of every routed slot's g row
        assert ws >= 2 * 4 * 768 * 8 * 512
    assert op.oop_mul_mat_id_back_workspace_size(9, ne_w, ne_ids) == 0      # q8_1: no
    assert op.oop_mul_mat_id_back_workspace_size(Q8, ne_w, ne_ids) > 0     # every other type
    assert op.oop_mul_mat_id_back_workspace_size(F32, (2048, 768, 6145), ne_ids) == 0
    assert op.oop_mul_mat_id_back_workspace_size(F32, ne_w, (0, 512)) == 0


@pytest.mark.parametrize("a_type,ne_a,ne_b", [
    (F32, (256, 0, 1, 1), (8, 0, 1, 1)),          # skinny-N shape, empty sum
    (Q8, (512, 0, 1, 1), (300, 0, 1, 1)),         # tensor-core shape, empty sum
    (F32, (128, 0, 2, 1), (70, 0, 4, 3)),         # broadcast, empty sum
])
def test_host_buffer_empty_sum(a_type, ne_a, ne_b):
    """K == 0 is a valid call (dst is zero-filled, then copied out): the host
    entry still needs room for dst, although no workspace."""
    assert op.oop_out_prod_workspace_min_size(a_type, ne_a, ne_b) == 0
    _, _, dst = _bytes(a_type, ne_a, ne_b)
    total = op.oop_out_prod_host_buffer_size(a_type, ne_a, ne_b)
    assert dst <= total <= dst + 4 * 255


def test_expert_weight_grad_workspace():
    ne_x, ne_dy = (2048, 8, 512), (768, 8, 512)
    ws = op.oop_mul_mat_id_weight_grad_workspace_size(ne_x, ne_dy, 32)
    # the gathered x rows and the split of dy for every routed slot, with up
    # to one k-block of padding per expert
    rows = 8 * 512 + 32 * 32
    assert ws >= 4 * rows * 2048 + 2 * 4 * 768 * rows
    assert op.oop_mul_mat_id_weight_grad_workspace_size(ne_x, ne_dy, 0) == 0
    assert op.oop_mul_mat_id_weight_grad_workspace_size((2048, 3, 512), ne_dy, 32) == 0  # 8 % 3
    assert op.oop_mul_mat_id_weight_grad_workspace_size(ne_x, (768, 8, 511), 32) == 0
