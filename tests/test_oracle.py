"""Pins of the CPU oracle against facts that do not come from the oracle.

Each test names what fixes the expected value: numpy's own binary16/bfloat16
conversions, exact integer arithmetic, the rank-one closed form, linearity,
explicit replication of src0 slices (numpy's repeat), numpy float64 matmul,
finite differences of the forward product, printed values from the pages
(golden fixtures), and a planted defect (fp16 staging) that must fail the
acceptance gate.  All run on the CPU.
"""

import json
import os

import numpy as np
import pytest

import synth

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _gold(name):
    with open(os.path.join(GOLD, name)) as f:
        return json.load(f)


def _gate(dst, f64, ab):
    """The acceptance bound: |x - exact| <= 2e-6 * sum_k |a*b|."""
    return np.abs(dst.astype(np.float64) - f64) <= 2e-6 * ab


# --------------------------------------------------------------------------
# generator
# --------------------------------------------------------------------------

def test_splitmix64_published_vector():
    g = _gold("splitmix64.json")
    got = synth.splitmix64(g["seed"], 0, 3)
    assert [int(x) for x in got] == [int(h, 16) for h in g["outputs_hex"]]


def test_normals_are_standard():
    x = synth.normal(123, 200000).astype(np.float64)
    assert abs(x.mean()) < 0.01 and abs(x.std() - 1.0) < 0.01
    assert np.all(np.isfinite(x))


def test_outliers_exact_count_and_range():
    x = np.zeros(100000, np.float32)
    synth.add_outliers(x, 5)
    nz = x[x != 0]
    assert nz.size == 200
    assert np.all(np.abs(nz) >= 6.6e4) and np.all(np.abs(nz) <= 1.5e5)
    assert 0 < (nz > 0).sum() < 200


def test_routing_distinct():
    ids = synth.routing_ids(9, 32, 8, 512)
    assert ids.shape == (512, 8)
    assert ids.min() >= 0 and ids.max() < 32
    for row in ids:
        assert len(set(row.tolist())) == 8


# --------------------------------------------------------------------------
# scalar decoders against numpy
# --------------------------------------------------------------------------

def test_half_decoder_all_patterns(orc):
    pats = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = pats.view(np.float16).astype(np.float64)
    got = np.array([orc.half_to_double(int(p)) for p in pats])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    # signed zero is kept
    assert np.signbit(orc.half_to_double(0x8000))


def test_bf16_decoder_all_patterns(orc):
    pats = np.arange(65536, dtype=np.uint32)
    ref = (pats << 16).astype(np.uint32).view(np.float32).astype(np.float64)
    got = np.array([orc.bf16_to_double(int(p)) for p in pats])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


def test_round_to_half_matches_numpy(orc):
    rng = np.random.default_rng(0)
    xs = np.concatenate([
        rng.normal(size=3000) * 10.0 ** rng.integers(-9, 6, size=3000),
        [65504.0, 65519.99, 65520.0, 65536.0, 131273.0, 6.0e-8, 2.98e-8, 3.0e-8,
         6.1e-5, 1.0 + 2.0 ** -11, 1.0 + 3 * 2.0 ** -11, -0.0, 0.0],
    ])
    for x in xs:
        assert orc.round_to_half(x) == float(np.float16(x)) or (
            np.isinf(orc.round_to_half(x)) and np.isinf(np.float16(x)))


def test_half_staging_golden(orc):
    g = _gold("half_staging.json")
    assert orc.round_to_half(g["half_max"]) == g["half_max"]
    for x in g["overflow_examples"]:
        assert np.isinf(orc.round_to_half(x))
    for x in g["finite_examples"]:
        assert np.isfinite(orc.round_to_half(x))


# --------------------------------------------------------------------------
# dequantisation
# --------------------------------------------------------------------------

def test_q8_0_every_int8_value(orc):
    blocks = np.zeros((8, 34), np.uint8)
    blocks[:, 0:2] = np.array([0x00, 0x3C], np.uint8)        # d = 1.0
    q = np.arange(-128, 128, dtype=np.int8).reshape(8, 32)
    blocks[:, 2:] = q.view(np.uint8)
    got = orc.dequant_row(synth.TYPE_Q8_0, blocks.reshape(-1), 256)
    assert np.array_equal(got, np.arange(-128, 128, dtype=np.float64))


@pytest.mark.parametrize("dbits", [0x3C00, 0x0001, 0x03FF, 0x7BFF, 0x8000, 0xB555, 0x2E66])
def test_q8_0_scales(orc, dbits):
    rng = np.random.default_rng(dbits)
    q = rng.integers(-127, 128, size=32).astype(np.int8)
    blk = np.zeros(34, np.uint8)
    blk[0:2] = np.array([dbits & 0xFF, dbits >> 8], np.uint8)
    blk[2:] = q.view(np.uint8)
    d = np.array([dbits], np.uint16).view(np.float16).astype(np.float64)[0]
    got = orc.dequant_row(synth.TYPE_Q8_0, blk, 32)
    assert np.array_equal(got, d * q.astype(np.float64))


def test_q4_0_golden_block(orc):
    g = _gold("q4_0_block.json")
    blk = np.frombuffer(bytes.fromhex(g["block_hex"]), np.uint8)
    got = orc.dequant_row(synth.TYPE_Q4_0, blk, 32)
    assert np.array_equal(got, np.array(g["elements"]))


def test_q4_0_every_nibble(orc):
    for v in range(16):
        blk = np.zeros(18, np.uint8)
        blk[0:2] = np.array([0x00, 0x3C], np.uint8)          # d = 1.0
        blk[2:] = v | (v << 4)
        got = orc.dequant_row(synth.TYPE_Q4_0, blk, 32)
        assert np.all(got == v - 8)


@pytest.mark.parametrize("tid,std", [(synth.TYPE_Q8_0, 0.02), (synth.TYPE_Q4_0, 0.02),
                                     (synth.TYPE_Q8_0, 3.0), (synth.TYPE_Q4_0, 3.0)])
def test_quant_round_trip(orc, tid, std):
    x = synth.normal(77, 64 * 256, std=std).reshape(64, 256)
    qb = synth.quantize_q8_0(x) if tid == synth.TYPE_Q8_0 else synth.quantize_q4_0(x)
    bs = 34 if tid == synth.TYPE_Q8_0 else 18
    for r in range(64):
        deq = orc.dequant_row(tid, qb[r], 256)
        blocks = qb[r].reshape(8, bs)
        d = np.abs(blocks[:, 0:2].copy().view(np.float16).astype(np.float64)).reshape(8)
        err = np.abs(deq - x[r].astype(np.float64)).reshape(8, 32)
        # q8_0: half a step; q4_0: its codes span [-8, 7] steps while the data
        # spans +-8, so the far side can clamp by one step.  Plus the scale's
        # own rounding carried by the largest code.
        step = 0.5 if tid == synth.TYPE_Q8_0 else 1.0
        lim = d[:, None] * (step + 128 * 2.0 ** -11) + 1e-30
        assert np.all(err <= lim)
    if tid == synth.TYPE_Q8_0:
        # requantising the dequantised values reproduces the bytes exactly
        deq_all = np.stack([orc.dequant_row(tid, qb[r], 256) for r in range(64)])
        assert np.array_equal(synth.quantize_q8_0(deq_all.astype(np.float32)), qb)


# --------------------------------------------------------------------------
# OUT_PROD
# --------------------------------------------------------------------------

def _int_inputs(rng, ne_a, ne_b, lim=8):
    a = rng.integers(-lim, lim + 1, size=(ne_a[3], ne_a[2], ne_a[1], ne_a[0])).astype(np.float32)
    b = rng.integers(-lim, lim + 1, size=(ne_b[3], ne_b[2], ne_b[1], ne_b[0])).astype(np.float32)
    return a, b


def _exact_int(a, b, ne_a, ne_b):
    """Integer reference: numpy int64 einsum over src0 slices replicated with
    np.repeat (slice i2 reads src0 slice i2 // dps2, i3 // dps3)."""
    dps2, dps3 = ne_b[2] // ne_a[2], ne_b[3] // ne_a[3]
    ai = np.repeat(np.repeat(a.astype(np.int64), dps2, axis=1), dps3, axis=0)
    bi = b.astype(np.int64)
    return np.einsum("xykm,xykn->xynm", ai, bi)


@pytest.mark.parametrize("ne_a,ne_b", [
    ((7, 5, 1, 1), (3, 5, 1, 1)),
    ((33, 64, 2, 1), (17, 64, 6, 1)),
    ((16, 9, 1, 2), (5, 9, 3, 4)),
    ((40, 1, 1, 1), (1, 1, 1, 1)),
])
def test_out_prod_integer_exact(orc, ne_a, ne_b):
    rng = np.random.default_rng(sum(ne_a) * 31 + sum(ne_b))
    a, b = _int_inputs(rng, ne_a, ne_b)
    r = orc.out_prod(a, synth.TYPE_F32, b, ne_a, ne_b)
    exact = _exact_int(a, b, ne_a, ne_b)
    assert np.array_equal(r["f64"], exact.astype(np.float64))
    assert np.array_equal(r["dst"], exact.astype(np.float32))
    assert np.array_equal(r["abs"], np.abs(
        np.einsum("xykm,xykn->xykmn",
                  np.repeat(np.repeat(a.astype(np.int64), ne_b[2] // ne_a[2], 1),
                            ne_b[3] // ne_a[3], 0), b.astype(np.int64))).sum(2)
        .transpose(0, 1, 3, 2).astype(np.float64))


@pytest.mark.parametrize("tid", [synth.TYPE_Q8_0, synth.TYPE_Q4_0])
def test_out_prod_quant_integer_exact(orc, tid):
    """Quantised src0 with d = 1: the dequantised weights are the integer codes."""
    rng = np.random.default_rng(tid)
    M, K, N = 64, 12, 5
    if tid == synth.TYPE_Q8_0:
        q = rng.integers(-127, 128, size=(K, M)).astype(np.int8)
        blk = np.zeros((K, M // 32, 34), np.uint8)
        blk[..., 0:2] = np.array([0x00, 0x3C], np.uint8)
        blk[..., 2:] = q.reshape(K, M // 32, 32).view(np.uint8)
        vals = q.astype(np.int64)
    else:
        v = rng.integers(0, 16, size=(K, M)).astype(np.uint8)
        blk = np.zeros((K, M // 32, 18), np.uint8)
        blk[..., 0:2] = np.array([0x00, 0x3C], np.uint8)
        vb = v.reshape(K, M // 32, 32)
        blk[..., 2:] = vb[..., :16] | (vb[..., 16:] << 4)
        vals = v.astype(np.int64) - 8
    a = blk.reshape(1, 1, K, -1)
    b = rng.integers(-9, 10, size=(1, 1, K, N)).astype(np.float32)
    r = orc.out_prod(a, tid, b, (M, K, 1, 1), (N, K, 1, 1))
    exact = np.einsum("km,kn->nm", vals, b[0, 0].astype(np.int64))
    assert np.array_equal(r["f64"][0, 0], exact.astype(np.float64))


def test_out_prod_rank_one_closed_form(orc):
    a = synth.normal(1, 300).reshape(1, 1, 1, 300)
    b = synth.normal(2, 19).reshape(1, 1, 1, 19) * np.float32(1e5)
    r = orc.out_prod(a, synth.TYPE_F32, b, (300, 1, 1, 1), (19, 1, 1, 1))
    outer = np.outer(b[0, 0, 0].astype(np.float64), a[0, 0, 0].astype(np.float64))
    assert np.array_equal(r["f64"][0, 0], outer)          # one exact product each
    assert np.array_equal(r["dst"][0, 0], outer.astype(np.float32))


def test_out_prod_matches_numpy_f64(orc):
    ne_a, ne_b = (70, 130, 2, 1), (37, 130, 4, 1)
    a = synth.make_a(synth.TYPE_F32, ne_a, 3)
    b = synth.make_b(ne_b, 4, std=100.0, outliers=True)
    r = orc.out_prod(a, synth.TYPE_F32, b, ne_a, ne_b)
    ar = np.repeat(a.astype(np.float64), 2, axis=1)
    ref = np.einsum("xykm,xykn->xynm", ar, b.astype(np.float64))
    assert np.all(np.abs(r["f64"] - ref) <= 1e-13 * r["abs"])
    assert np.all(_gate(r["dst"], ref, r["abs"]))


def test_out_prod_linearity(orc):
    ne_a, ne_b = (48, 40, 1, 1), (9, 40, 1, 1)
    rng = np.random.default_rng(5)
    # values on a 2^-10 grid, so alpha*a1 + beta*a2 is exact in f32
    a1 = (rng.integers(-2048, 2048, size=(1, 1, 40, 48)) / 1024.0).astype(np.float32)
    a2 = (rng.integers(-2048, 2048, size=(1, 1, 40, 48)) / 1024.0).astype(np.float32)
    b = synth.make_b(ne_b, 6, std=1e3, outliers=True)
    al, be = np.float32(4.0), np.float32(-0.5)
    lhs = orc.out_prod(al * a1 + be * a2, synth.TYPE_F32, b, ne_a, ne_b)
    r1 = orc.out_prod(a1, synth.TYPE_F32, b, ne_a, ne_b)
    r2 = orc.out_prod(a2, synth.TYPE_F32, b, ne_a, ne_b)
    rhs = 4.0 * r1["f64"] - 0.5 * r2["f64"]
    bound = 1e-13 * (4.0 * r1["abs"] + 0.5 * r2["abs"])
    assert np.all(np.abs(lhs["f64"] - rhs) <= bound)
    # and in b
    b1 = (rng.integers(-4096, 4096, size=(1, 1, 40, 9)) / 8.0).astype(np.float32)
    b2 = (rng.integers(-4096, 4096, size=(1, 1, 40, 9)) / 8.0).astype(np.float32)
    a = synth.make_a(synth.TYPE_F32, ne_a, 7)
    lhs = orc.out_prod(a, synth.TYPE_F32, 2.0 * b1 + 0.25 * b2, ne_a, ne_b)
    r1 = orc.out_prod(a, synth.TYPE_F32, b1, ne_a, ne_b)
    r2 = orc.out_prod(a, synth.TYPE_F32, b2, ne_a, ne_b)
    rhs = 2.0 * r1["f64"] + 0.25 * r2["f64"]
    assert np.all(np.abs(lhs["f64"] - rhs) <= 1e-13 * (2.0 * r1["abs"] + 0.25 * r2["abs"]))


@pytest.mark.parametrize("tid", [synth.TYPE_F32, synth.TYPE_Q8_0, synth.TYPE_Q4_0])
@pytest.mark.parametrize("ne_a,ne_b", [((64, 24, 4, 1), (10, 24, 16, 1)),
                                       ((64, 24, 2, 2), (10, 24, 4, 4))])
def test_broadcast_equals_replication(orc, tid, ne_a, ne_b):
    a = synth.make_a(tid, ne_a, 8)
    b = synth.make_b(ne_b, 9, outliers=True)
    dps2, dps3 = ne_b[2] // ne_a[2], ne_b[3] // ne_a[3]
    rep = np.repeat(np.repeat(a, dps2, axis=1), dps3, axis=0)
    ne_rep = (ne_a[0], ne_a[1], ne_b[2], ne_b[3])
    r1 = orc.out_prod(a, tid, b, ne_a, ne_b)
    r2 = orc.out_prod(rep, tid, b, ne_rep, ne_b)
    assert np.array_equal(r1["f64"], r2["f64"])
    assert np.array_equal(r1["dst"], r2["dst"])


def test_shape_contract_golden(orc):
    for c in _gold("shape_contract.json")["cases"]:
        ne_a, ne_b = tuple(c["ne_a"]), tuple(c["ne_b"])
        M, K = 2, ne_a[1]
        a_small = np.ones((ne_a[3], ne_a[2], ne_a[1], M), np.float32)
        b_small = np.ones((ne_b[3], ne_b[2], ne_b[1], 1), np.float32)
        na = (M,) + ne_a[1:]
        nb = (1,) + ne_b[1:]
        if c["ok"]:
            r = orc.out_prod(a_small, synth.TYPE_F32, b_small, na, nb)
            assert r["dst"].shape == (c["ne_dst"][3], c["ne_dst"][2], 1, M)
            assert np.all(r["dst"] == K)
        else:
            with pytest.raises(ValueError):
                orc.out_prod(a_small, synth.TYPE_F32, b_small, na, nb)


def test_empty_sum_is_zero(orc):
    a = np.zeros((1, 1, 0, 32), np.float32)
    b = np.zeros((1, 1, 0, 3), np.float32)
    r = orc.out_prod(a, synth.TYPE_F32, b, (32, 0, 1, 1), (3, 0, 1, 1))
    assert np.array_equal(r["dst"], np.zeros((1, 1, 3, 32), np.float32))


def test_at_matches_whole(orc):
    ne_a, ne_b = (96, 33, 2, 1), (11, 33, 4, 1)
    a = synth.make_a(synth.TYPE_Q8_0, ne_a, 12, std=0.02)
    b = synth.make_b(ne_b, 13, std=1e3, outliers=True)
    whole = orc.out_prod(a, synth.TYPE_Q8_0, b, ne_a, ne_b)
    rng = np.random.default_rng(1)
    coords = np.stack([rng.integers(0, 96, 200), rng.integers(0, 11, 200),
                       rng.integers(0, 4, 200), np.zeros(200, np.int64)], 1)
    val, ab = orc.out_prod_at(a, synth.TYPE_Q8_0, b, ne_a, ne_b, coords)
    ref = whole["f64"][coords[:, 3], coords[:, 2], coords[:, 1], coords[:, 0]]
    assert np.array_equal(val, ref)


# --------------------------------------------------------------------------
# the overflow gate catches fp16 staging (planted defect, on the CPU)
# --------------------------------------------------------------------------

@pytest.mark.parametrize("tid", [synth.TYPE_F32, synth.TYPE_Q8_0])
def test_fp16_staging_fails_gate(orc, tid):
    ne_a, ne_b = (64, 256, 1, 1), (24, 256, 1, 1)
    a = synth.make_a(tid, ne_a, 14, std=1.0)
    b = synth.make_b(ne_b, 15, std=100.0, outliers=True)
    good = orc.out_prod(a, tid, b, ne_a, ne_b)
    bad = orc.out_prod_fp16_staged(a, tid, b, ne_a, ne_b)
    assert np.all(_gate(good["dst"], good["f64"], good["abs"]))
    assert not np.all(np.isfinite(bad))             # the Inf/NaN symptom
    finite = np.isfinite(bad)
    ok = _gate(np.where(finite, bad, 0), good["f64"], good["abs"]) & finite
    assert ok.mean() < 0.5                          # and the rounding symptom


# --------------------------------------------------------------------------
# MUL_MAT_ID_BACK
# --------------------------------------------------------------------------

def test_mmid_one_hot_equals_dense(orc):
    """All slots routed to expert e: dx[:, i, :] = out_prod(W_e, g[:, i, :]^T)."""
    K, N, E, n_used, T = 40, 24, 5, 3, 7
    W = synth.normal(20, K * N * E).reshape(E, N, K)
    g = synth.normal(21, N * n_used * T).reshape(T, n_used, N)
    e = 3
    ids = np.full((T, n_used), e, np.int32)
    r = orc.mul_mat_id_back(W, synth.TYPE_F32, ids, g, (K, N, E))
    for i in range(n_used):
        bT = np.ascontiguousarray(g[:, i, :].T).reshape(1, 1, N, T)   # b[n=t, k=r]
        a = W[e].reshape(1, 1, N, K)                                 # a[m=k, k=r]
        op = orc.out_prod(a, synth.TYPE_F32, bT, (K, N, 1, 1), (T, N, 1, 1))
        assert np.array_equal(op["f64"][0, 0], r["f64"][:, i, :])


@pytest.mark.parametrize("wt", [synth.TYPE_F32, synth.TYPE_BF16])
def test_mmid_matches_numpy(orc, wt):
    K, N, E, n_used, T = 64, 48, 6, 4, 9
    W = synth.normal(22, K * N * E, std=0.02).reshape(E, N, K)
    Wd = W.astype(np.float64)
    if wt == synth.TYPE_BF16:
        W = synth.to_bf16_bits(W)
        Wd = (W.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    ids = synth.routing_ids(23, E, n_used, T)
    g = synth.normal(24, N * n_used * T).reshape(T, n_used, N)
    r = orc.mul_mat_id_back(W, wt, ids, g, (K, N, E))
    ref = np.einsum("tirk,tir->tik", Wd[ids], g.astype(np.float64))
    assert np.all(np.abs(r["f64"] - ref) <= 1e-13 * r["abs"])
    coords = np.array([[0, 0, 0], [63, 3, 8], [17, 2, 4]])
    val, _ = orc.mul_mat_id_back_at(W, wt, ids, g, (K, N, E), coords)
    assert np.array_equal(val, r["f64"][coords[:, 2], coords[:, 1], coords[:, 0]])


def test_mmid_rejects_bad_id(orc):
    W = np.zeros((2, 3, 4), np.float32)
    g = np.zeros((1, 1, 3), np.float32)
    with pytest.raises(ValueError):
        orc.mul_mat_id_back(W, synth.TYPE_F32, np.array([[2]], np.int32), g, (4, 3, 2))


# --------------------------------------------------------------------------
# the backward of MUL_MAT through OUT_PROD, by finite differences
# ("metal: OUT_PROD multiplies in float staging", scope paragraph:
#  src0's gradient is out_prod(src1, grad), src1's is out_prod(src0, grad^T))
# --------------------------------------------------------------------------

def test_finite_difference_of_forward(orc):
    K, R, T = 12, 7, 5
    rng = np.random.default_rng(11)
    W = rng.normal(size=(R, K))          # ggml {K, R}
    x = rng.normal(size=(T, K))          # ggml {K, T}
    G = rng.normal(size=(T, R))          # upstream gradient {R, T}

    def loss(Wm, xm):
        return float((orc.mul_mat(Wm, xm) * G).sum())

    # d/dx = out_prod(W, G^T): a = W {K (m), R (k)}, b[n=t, k=r] = G^T
    gx = orc.out_prod(W.astype(np.float32), synth.TYPE_F32,
                      np.ascontiguousarray(G.T).astype(np.float32),
                      (K, R, 1, 1), (T, R, 1, 1))["f64"][0, 0]
    # d/dW = out_prod(x, G): a = x {K (m), T (k)}, b = G {R (n), T (k)}
    gw = orc.out_prod(x.astype(np.float32), synth.TYPE_F32, G.astype(np.float32),
                      (K, T, 1, 1), (R, T, 1, 1))["f64"][0, 0]
    Wf = W.astype(np.float32).astype(np.float64)
    xf = x.astype(np.float32).astype(np.float64)
    Gf = G.astype(np.float32).astype(np.float64)
    G[:] = Gf
    for t in range(T):
        for k in range(K):
            xp, xm = xf.copy(), xf.copy()
            xp[t, k] += 1.0
            xm[t, k] -= 1.0
            fd = (loss(Wf, xp) - loss(Wf, xm)) / 2.0
            assert abs(fd - gx[t, k]) <= 1e-12 * (1 + abs(fd))
    for r in range(R):
        for k in range(K):
            Wp, Wm = Wf.copy(), Wf.copy()
            Wp[r, k] += 1.0
            Wm[r, k] -= 1.0
            fd = (loss(Wp, xf) - loss(Wm, xf)) / 2.0
            assert abs(fd - gw[r, k]) <= 1e-12 * (1 + abs(fd))


# --------------------------------------------------------------------------
# src1 as a strided view, and the MUL_MAT backward pair
# ("metal: OUT_PROD multiplies in float staging", scope paragraph: the
#  gradient of src1 is out_prod(src0, grad^T), a transposed view of grad)
# --------------------------------------------------------------------------

def _views(rng):
    """(name, src1 view) pairs: a transpose, padded rows, a slice step, a
    zero stride (one row read for every n)."""
    base = rng.normal(size=(2, 3, 40, 30)).astype(np.float32) * np.float32(100)
    return [
        ("transposed", np.swapaxes(base, 2, 3)),                  # (2, 3, 30, 40): k fastest
        ("padded rows", base[:, :, :, 3:20]),                     # row stride 30, N = 17
        ("every other slice", base[:, ::2]),
        ("broadcast row", np.broadcast_to(base[:, :, :, :1], (2, 3, 40, 9))),
    ]


def test_strided_equals_contiguous(orc):
    rng = np.random.default_rng(21)
    for name, v in _views(rng):
        ne_b, nb = orc.view_ne_nb(v)
        ne_a = (48, ne_b[1], 1, ne_b[3])
        a = synth.make_a(synth.TYPE_F32, ne_a, 120)
        r1 = orc.out_prod_strided(a, synth.TYPE_F32, v, ne_a)
        r2 = orc.out_prod(a, synth.TYPE_F32, np.ascontiguousarray(v), ne_a, ne_b)
        for key in ("dst", "f64", "abs"):
            assert np.array_equal(r1[key], r2[key]), f"{name} {key}"


def test_strided_integer_exact(orc):
    """Small-integer inputs through a transposed view equal an int64 einsum of
    the transposed integers (every sum exact)."""
    rng = np.random.default_rng(22)
    M, K, N = 40, 33, 19
    a = rng.integers(-8, 9, size=(1, 1, K, M)).astype(np.float32)
    g = rng.integers(-8, 9, size=(1, 1, N, K)).astype(np.float32)   # g[n, k] row-major
    v = np.swapaxes(g, 2, 3)                                          # b[k][n] view of g
    r = orc.out_prod_strided(a, synth.TYPE_F32, v, (M, K, 1, 1))
    exact = np.einsum("km,nk->nm", a[0, 0].astype(np.int64), g[0, 0].astype(np.int64))
    assert np.array_equal(r["f64"][0, 0], exact.astype(np.float64))


def _forward_f64(W, x, ne_w, ne_x):
    """y[r,t,i2,i3] = sum_k W[k,r,i2/dps2,i3/dps3] x[k,t,i2,i3], in numpy."""
    d2, d3 = ne_x[2] // ne_w[2], ne_x[3] // ne_w[3]
    Wr = np.repeat(np.repeat(W, d2, axis=1), d3, axis=0)      # (ne13, ne12, R, K)
    return np.einsum("abrk,abtk->abtr", Wr, x)


@pytest.mark.parametrize("ne_w,ne_x", [
    ((9, 6, 1, 1), (9, 5, 1, 1)),
    ((8, 5, 2, 1), (8, 4, 4, 1)),      # dps2 = 2: dW sums over adjacent slices
    ((7, 4, 2, 1), (7, 3, 4, 2)),      # dps2 = 2, dps3 = 2: groups not adjacent
])
def test_mul_mat_back_finite_differences(orc, ne_w, ne_x):
    """The loss L = sum(y * G) is linear in W and in x, so a central
    difference with step 1 in fp64 is the gradient up to rounding."""
    rng = np.random.default_rng(sum(ne_w) + 7 * sum(ne_x))
    K, R, w2, w3 = ne_w
    _, T, x2, x3 = ne_x
    W = rng.normal(size=(w3, w2, R, K)).astype(np.float32)
    x = rng.normal(size=(x3, x2, T, K)).astype(np.float32)
    G = rng.normal(size=(x3, x2, T, R)).astype(np.float32)
    Wd, xd, Gd = (v.astype(np.float64) for v in (W, x, G))
    out = orc.mul_mat_back(W, synth.TYPE_F32, x, G, ne_w)

    def loss(Wm, xm):
        return float((_forward_f64(Wm, xm, ne_w, ne_x) * Gd).sum())

    for idx in np.ndindex(xd.shape):
        xp, xm = xd.copy(), xd.copy()
        xp[idx] += 1.0
        xm[idx] -= 1.0
        fd = (loss(Wd, xp) - loss(Wd, xm)) / 2.0
        assert abs(fd - out["dx"]["f64"][idx]) <= 1e-12 * (1 + abs(fd)), idx
    for idx in np.ndindex(Wd.shape):
        Wp, Wm = Wd.copy(), Wd.copy()
        Wp[idx] += 1.0
        Wm[idx] -= 1.0
        fd = (loss(Wp, xd) - loss(Wm, xd)) / 2.0
        assert abs(fd - out["dW"]["f64"][idx]) <= 1e-12 * (1 + abs(fd)), idx


@pytest.mark.parametrize("tid", [synth.TYPE_F32, synth.TYPE_Q8_0, synth.TYPE_Q4_0])
def test_mul_mat_back_dx_is_out_prod_of_transposed_grad(orc, tid):
    """dx = OUT_PROD(W, dy^T) with the same products in the same order: bit
    for bit, for quantised W too."""
    ne_w, ne_x = (64, 24, 2, 1), (64, 10, 4, 1)
    W = synth.make_a(tid, ne_w, 121, std=0.02)
    x = synth.make_b((64, 10, 4, 1), 122)
    dy = synth.make_b((24, 10, 4, 1), 123, std=1e3, outliers=True)
    out = orc.mul_mat_back(W, tid, x, dy, ne_w)
    ref = orc.out_prod_strided(W, tid, np.swapaxes(dy, 2, 3), ne_w)
    for key in ("dst", "f64", "abs"):
        assert np.array_equal(out["dx"][key], ref[key]), key


@pytest.mark.parametrize("ne_w,ne_x", [
    ((48, 12, 1, 1), (48, 20, 1, 1)),
    ((48, 12, 2, 1), (48, 20, 6, 1)),        # dps2 = 3, adjacent slices
    ((48, 12, 1, 2), (48, 20, 3, 4)),        # ne02 = 1, dps3 = 2: adjacent too
])
def test_mul_mat_back_dw_is_out_prod_over_grouped_slices(orc, ne_w, ne_x):
    """Where each broadcast group of slices is adjacent in memory (dps3 = 1 or
    ne02 = 1), dW = OUT_PROD(x, dy) over the group's rows taken as one longer
    reduction: bit for bit (the same products in the same order)."""
    K, R, w2, w3 = ne_w
    _, T, x2, x3 = ne_x
    x = synth.make_b((K, T, x2, x3), 124)
    dy = synth.make_b((R, T, x2, x3), 125, std=1e3, outliers=True)
    W = synth.make_a(synth.TYPE_F32, ne_w, 126)
    out = orc.mul_mat_back(W, synth.TYPE_F32, x, dy, ne_w)
    group = (x2 // w2) * (x3 // w3)
    ref = orc.out_prod(x.reshape(w3, w2, group * T, K), synth.TYPE_F32,
                       dy.reshape(w3, w2, group * T, R), (K, group * T, w2, w3),
                       (R, group * T, w2, w3))
    for key in ("dst", "f64", "abs"):
        assert np.array_equal(out["dW"][key], ref[key]), key


# --------------------------------------------------------------------------
# the other src0 types ("Metal kernel_mul_mat_id_back", first bullet: out_prod's
# instantiation set; q4_K: "metal: OUT_PROD multiplies in float staging",
# answer (2)).  The oracle's decoders and synth's quantisers are separate
# implementations of each block layout; these pins tie them together on data
# that makes a misplaced bit, nibble or scale index show up as a gross error.
# --------------------------------------------------------------------------

_LEVELS = {synth.TYPE_Q4_0: 15, synth.TYPE_Q4_1: 15, synth.TYPE_Q5_0: 31,
           synth.TYPE_Q5_1: 31, synth.TYPE_Q8_0: 254, synth.TYPE_Q2_K: 3,
           synth.TYPE_Q3_K: 7, synth.TYPE_Q4_K: 15, synth.TYPE_Q5_K: 31,
           synth.TYPE_Q6_K: 63}
_SUB = {synth.TYPE_Q2_K: 16, synth.TYPE_Q3_K: 16, synth.TYPE_Q6_K: 16}


def _graded(rows, ne0, sub, seed, offset, grades=8):
    """Normals whose consecutive `sub`-element groups are scaled by
    2^(i % grades) (and, with `offset`, shifted by a group-dependent amount)."""
    x = synth.normal(seed, rows * ne0).reshape(rows, ne0).astype(np.float64)
    g = np.arange(ne0) // sub
    x *= 2.0 ** (g % grades)
    if offset:
        x += 0.5 * (2.0 ** (g % grades)) * ((g % 3) - 1)
    return x.astype(np.float32)


@pytest.mark.parametrize("tid", sorted(_LEVELS))
def test_quantiser_decoder_round_trip(orc, tid):
    """dequant(quant(x)) stays within about one code step of x in every group
    of elements that shares a scale; a decoder reading the wrong scale, nibble
    or bit would be off by the magnitude of another group (2x to 128x)."""
    qk, _ = synth.BLOCK[tid]
    sub = _SUB.get(tid, 32)
    ne0, rows = 2 * 256, 6
    # a K-quant's sub-block scales are 6-bit (4-bit for q2_K) multiples of one
    # super-block scale, so its groups may differ by 8x at most
    grades = 4 if qk == 256 else 8
    for offset in (False, True):
        x = _graded(rows, ne0, sub, 140 + tid, offset, grades)
        q = synth.quantize(tid, x)
        deq = np.stack([orc.dequant_row(tid, q[r], ne0) for r in range(rows)])
        xs = x.astype(np.float64).reshape(rows, -1, sub)
        ds = deq.reshape(rows, -1, sub)
        span = np.maximum(xs.max(axis=2), 0) - np.minimum(xs.min(axis=2), 0)
        # one code step of the group, widened for the binary16 / 6-bit scale
        # rounding; a group's neighbours differ from it by a factor of 2 or more
        err = np.abs(ds - xs).max(axis=2)
        ratio = float((err / np.maximum(span / _LEVELS[tid], 1e-30)).max())
        assert ratio <= 1.25, (tid, offset, ratio)


@pytest.mark.parametrize("tid", sorted(_LEVELS))
def test_decoder_scales_with_the_block_scales(orc, tid):
    """Multiplying every binary16 scale field of a block by 2 (exponent + 1)
    doubles every decoded element (the scales multiply every term)."""
    qk, nbytes = synth.BLOCK[tid]
    x = _graded(2, 256, _SUB.get(tid, 32), 150 + tid, True, 4)
    q = synth.quantize(tid, x).reshape(-1, nbytes).copy()
    fields = {synth.TYPE_Q4_0: [0], synth.TYPE_Q4_1: [0, 2], synth.TYPE_Q5_0: [0],
              synth.TYPE_Q5_1: [0, 2], synth.TYPE_Q8_0: [0], synth.TYPE_Q2_K: [80, 82],
              synth.TYPE_Q3_K: [108], synth.TYPE_Q4_K: [0, 2], synth.TYPE_Q5_K: [0, 2],
              synth.TYPE_Q6_K: [208]}[tid]
    before = np.stack([orc.dequant_row(tid, b, qk) for b in q])
    q2 = q.copy()
    for off in fields:
        h = q2[:, off:off + 2].copy().view(np.uint16)[:, 0]
        exp = (h >> 10) & 31
        assert np.all((exp > 0) & (exp < 30)), "normal scales only"
        q2[:, off:off + 2] = (h + (1 << 10)).astype(np.uint16).view(np.uint8).reshape(-1, 2)
    after = np.stack([orc.dequant_row(tid, b, qk) for b in q2])
    assert np.array_equal(after, 2 * before)


@pytest.mark.parametrize("tid", [synth.TYPE_F16, synth.TYPE_BF16])
def test_plain_16bit_types_out_prod(orc, tid):
    """f16 / bf16 src0: OUT_PROD equals numpy's float64 product of numpy's own
    decoding of the 16-bit patterns."""
    ne_a, ne_b = (40, 33, 1, 1), (9, 33, 1, 1)
    x = synth.normal(160, 40 * 33).reshape(1, 1, 33, 40)
    bits = synth.quantize(tid, x)
    if tid == synth.TYPE_F16:
        vals = bits.view(np.float16).astype(np.float64)
    else:
        vals = (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    b = synth.make_b(ne_b, 161)
    r = orc.out_prod(bits, tid, b, ne_a, ne_b)
    ref = np.einsum("km,kn->nm", vals[0, 0], b[0, 0].astype(np.float64))
    assert np.all(np.abs(r["f64"][0, 0] - ref) <= 1e-13 * r["abs"][0, 0])


@pytest.mark.parametrize("wt", [synth.TYPE_F16, synth.TYPE_Q8_0, synth.TYPE_Q4_1, synth.TYPE_Q5_0,
                                synth.TYPE_Q2_K, synth.TYPE_Q4_K, synth.TYPE_Q6_K])
def test_mmid_one_hot_equals_dense_every_weight_type(orc, wt):
    """Expert weights of every type ("Metal kernel_mul_mat_id_back", first
    bullet): with all slots routed to expert e, dx[:, i, :] equals OUT_PROD of
    that expert's rows (the same bytes as a src0) and g^T, bit for bit."""
    qk = synth.BLOCK.get(wt, (1, 2))[0]
    K, N, E, n_used, T = (256 if qk == 256 else 64), 24, 4, 2, 6
    x = synth.normal(22, K * N * E, std=0.1).reshape(E, N, K)
    W = synth.quantize(wt, x)                       # rows (e, r) of K elements
    W = W.reshape(E, N, -1).view(np.uint8) if wt == synth.TYPE_F16 else W.reshape(E, N, -1)
    g = synth.normal(23, N * n_used * T).reshape(T, n_used, N)
    for e in (0, 3):
        ids = np.full((T, n_used), e, np.int32)
        r = orc.mul_mat_id_back(W, wt, ids, g, (K, N, E))
        for i in range(n_used):
            bT = np.ascontiguousarray(g[:, i, :].T).reshape(1, 1, N, T)
            op = orc.out_prod(W[e].reshape(1, 1, N, -1), wt, bT, (K, N, 1, 1), (T, N, 1, 1))
            assert np.array_equal(op["f64"][0, 0], r["f64"][:, i, :])


# --------------------------------------------------------------------------
# the expert-weight gradient of MUL_MAT_ID (the op whose input gradient is
# MUL_MAT_ID_BACK; "Metal kernel_mul_mat_id_back" is proven with the
# gradient check of MUL_MAT_ID)
# --------------------------------------------------------------------------

def _moe_inputs(seed, K, N, E, n_used, n_x, T):
    x = synth.normal(seed, T * n_x * K).reshape(T, n_x, K)
    dy = synth.normal(seed + 1, T * n_used * N).reshape(T, n_used, N)
    ids = synth.routing_ids(seed + 2, E, n_used, T)
    return x, ids, dy


@pytest.mark.parametrize("n_x", [1, 3])
def test_expert_weight_grad_finite_differences(orc, n_x):
    """L = sum(y * G) with y[r,i,t] = sum_k W[k,r,ids[i,t]] x[k, i % n_x, t] is
    linear in W: central differences of a numpy forward give dW."""
    K, N, E, n_used, T = 5, 4, 4, 3, 6
    x, ids, G = _moe_inputs(180, K, N, E, n_used, n_x, T)
    out = orc.mul_mat_id_weight_grad(x, ids, G, E)
    W = np.random.default_rng(7).normal(size=(E, N, K))
    xd, Gd = x.astype(np.float64), G.astype(np.float64)

    def loss(Wm):
        y = np.einsum("tirk,tik->tir", Wm[ids], xd[:, np.arange(n_used) % n_x, :])
        return float((y * Gd).sum())

    for idx in np.ndindex(W.shape):
        Wp, Wm = W.copy(), W.copy()
        Wp[idx] += 1.0
        Wm[idx] -= 1.0
        fd = (loss(Wp) - loss(Wm)) / 2.0
        assert abs(fd - out["f64"][idx]) <= 1e-12 * (1 + abs(fd)), idx


def test_expert_weight_grad_sums_to_dense(orc):
    """Summed over experts, the gradient is the dense weight gradient over
    every slot: OUT_PROD(x, dy) with all slots as one reduction."""
    K, N, E, n_used, T = 40, 24, 6, 4, 30
    x, ids, dy = _moe_inputs(182, K, N, E, n_used, n_used, T)
    out = orc.mul_mat_id_weight_grad(x, ids, dy, E)
    dense = orc.out_prod(x.reshape(1, 1, T * n_used, K), synth.TYPE_F32,
                         dy.reshape(1, 1, T * n_used, N), (K, T * n_used, 1, 1),
                         (N, T * n_used, 1, 1))
    total = out["f64"].sum(axis=0)
    assert np.all(np.abs(total - dense["f64"][0, 0]) <= 1e-12 * dense["abs"][0, 0])
    assert np.allclose(out["abs"].sum(axis=0), dense["abs"][0, 0], rtol=1e-12, atol=0)


def test_expert_weight_grad_one_hot(orc):
    """All slots routed to expert e: dW[:, :, e] is OUT_PROD(x, dy) over all
    slots, bit for bit; every other expert's gradient is zero."""
    K, N, E, n_used, T = 32, 20, 3, 2, 9
    x, _, dy = _moe_inputs(184, K, N, E, n_used, 1, T)
    ids = np.full((T, n_used), 1, np.int32)
    out = orc.mul_mat_id_weight_grad(x, ids, dy, E)
    xs = np.repeat(x, n_used, axis=1)                        # every slot's row
    dense = orc.out_prod(xs.reshape(1, 1, T * n_used, K), synth.TYPE_F32,
                         dy.reshape(1, 1, T * n_used, N), (K, T * n_used, 1, 1),
                         (N, T * n_used, 1, 1))
    assert np.array_equal(out["f64"][1], dense["f64"][0, 0])
    assert not out["f64"][0].any() and not out["f64"][2].any()
