"""Pins for the oracle: checks of oracle/ against facts fixed outside it.

Each test ties an oracle function to something other than the oracle itself:
the byte accounting the pages print (tests/golden/page_accounting.txt),
IEEE binary16 conversion as numpy implements it, closed-form quantization
cases, exact rational arithmetic, brute-force fp64 products computed
element by element with numpy, and algebraic invariants.  They are chosen so
that a plausible slip in the oracle (a wrong rounding mode, 1/d taken from
the fp16 scale, a transposed operand, a dropped block, a sign error, a wrong
byte order) fails at least one of them.
"""
import os

import numpy as np
import pytest

import oracle
import q8_synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _page_facts():
    facts = {}
    with open(os.path.join(GOLDEN, "page_accounting.txt")) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                k, v = line.split()
                facts[k] = int(v)
    return facts


def _blocks_from(d16, q):
    """Assemble 34-byte blocks from scale bits and quants (byte layout only)."""
    d16 = np.asarray(d16, dtype=np.uint16)
    q = np.asarray(q, dtype=np.int8)
    rows, nb = d16.shape
    b = np.zeros((rows, nb, 34), dtype=np.uint8)
    b[:, :, 0] = d16 & 0xFF
    b[:, :, 1] = d16 >> 8
    b[:, :, 2:] = q.view(np.uint8)
    return b.reshape(rows, nb * 34)


def _round_half_away(v):
    return np.sign(v) * np.floor(np.abs(v) + 0.5)


# --------------------------------------------------------------------------
# byte accounting printed on the pages
# --------------------------------------------------------------------------

def test_block_and_tile_accounting_matches_pages():
    facts = _page_facts()
    c = oracle.constants()
    assert c["qk"] == facts["block_values"] == 32
    # a block = one fp16 scale + 32 int8 quants
    assert c["block_bytes"] == facts["scale_bytes"] + facts["block_values"]
    assert c["ember_tile_bytes"] == facts["tile_bytes"]
    # "exactly the encoded size of 16 ordinary Q8_0 blocks"
    assert facts["tile_bytes"] == facts["tile_rows"] * c["block_bytes"]
    x = q8_synth.normal_np((3, 96), 1.0, 7)
    assert oracle.quantize(x).nbytes == 3 * 3 * 34


def test_ember_tile_layout_and_round_trip():
    facts = _page_facts()
    rng = np.random.default_rng(11)
    blocks = rng.integers(0, 256, size=(16, 34), dtype=np.uint8)
    tile = oracle.ember_tile_pack(blocks)
    assert tile.nbytes == facts["tile_bytes"]
    # packing only moves bytes: same multiset of bytes, and it inverts
    assert np.array_equal(np.sort(tile), np.sort(blocks.ravel()))
    assert np.array_equal(oracle.ember_tile_unpack(tile), blocks)
    # the figure: group g holds rows 0..15, coordinates 4g..4g+3 each
    g_bytes = facts["tile_rows"] * facts["tile_group_values"]
    for g in range(facts["tile_groups"]):
        grp = tile[g * g_bytes:(g + 1) * g_bytes].reshape(16, 4)
        assert np.array_equal(grp, blocks[:, 2 + 4 * g:2 + 4 * g + 4])
    # then the 16 scales in row order
    sc = tile[facts["tile_groups"] * g_bytes:].reshape(16, 2)
    assert np.array_equal(sc, blocks[:, 0:2])


# --------------------------------------------------------------------------
# binary16 conversion: IEEE round-to-nearest-even as numpy implements it
# --------------------------------------------------------------------------

def test_f16_decode_exhaustive_vs_numpy():
    h = np.arange(65536, dtype=np.uint16)
    ours = oracle.f16_bits_to_f32(h)
    ref = h.view(np.float16).astype(np.float32)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan].view(np.uint32), ref[~nan].view(np.uint32))


def test_f16_encode_vs_numpy():
    rng = np.random.default_rng(3)
    mags = np.exp2(rng.uniform(-30, 17, size=20000)).astype(np.float32)
    signs = np.where(rng.random(20000) < 0.5, -1, 1).astype(np.float32)
    x = mags * signs
    special = np.array([
        0.0, -0.0, 1.0, 65504.0, 65519.996, 65520.0, 1e9, -1e9,
        2.0**-24, 2.0**-25, 3 * 2.0**-26, 2.0**-25 * 1.0000001, 2.0**-14,
        2.0**-14 - 2.0**-25, 1 + 2.0**-11, 1 + 3 * 2.0**-11, 1 - 2.0**-12,
        2047.5, 2049.0, 2051.0, 1e-40, np.inf, -np.inf,
    ], dtype=np.float32)
    x = np.concatenate([x, special])
    ours = oracle.f32_to_f16_bits(x)
    with np.errstate(over="ignore"):
        ref = x.astype(np.float16).view(np.uint16)
    assert np.array_equal(ours, ref)
    assert oracle.f16_bits_to_f32(oracle.f32_to_f16_bits(np.float32(np.nan))) != \
        oracle.f16_bits_to_f32(oracle.f32_to_f16_bits(np.float32(np.nan)))


# --------------------------------------------------------------------------
# quantization: closed forms
# --------------------------------------------------------------------------

def test_quantize_unit_scale_ties_away_from_zero():
    # amax = 127 gives d = 127/127 = 1 exactly, 1/d = 1, so q = round(x) with
    # ties away from zero; 0.49999997 (the float just below 0.5) goes to 0.
    vals = [127.0, 2.5, -2.5, 0.49999997, 0.5, -0.5, 1.5, -1.5, 126.5,
            -126.5, 0.0, -0.0, 3.49999976, 100.25, -7.75, 64.5]
    x = np.zeros(32, dtype=np.float32)
    x[:len(vals)] = vals
    d16, q = oracle.split_blocks(oracle.quantize(x), 32)
    assert d16[0, 0] == 0x3C00  # 1.0
    expect = [127, 3, -3, 0, 1, -1, 2, -2, 127, -127, 0, 0, 3, 100, -8, 65]
    assert q[0, 0, :len(vals)].tolist() == expect
    assert not q[0, 0, len(vals):].any()


def test_quantize_block_with_overflowing_reciprocal():
    # amax = 1e-40 (subnormal): d = amax/127 is below 2^-128, so 1/d
    # overflows to inf; every nonzero value then maps to +-inf before the
    # clamp, i.e. to +-127, zeros (0 * inf) stay 0, and the scale rounds to
    # binary16 zero
    x = np.zeros(32, dtype=np.float32)
    x[:5] = [-1e-40, 1e-40, 0.0, -0.0, -3e-45]
    d16, q = oracle.split_blocks(oracle.quantize(x), 32)
    assert d16[0, 0] == 0
    assert q[0, 0, :5].tolist() == [-127, 127, 0, 0, -127]
    assert not q[0, 0, 5:].any()


def test_quantize_zero_constant_and_one_hot_blocks():
    z = oracle.quantize(np.zeros((1, 64), np.float32))
    assert not z.any()  # d = 0 and every q = 0: all 34 bytes zero, twice
    for c, dbits in ((127.0, 0x3C00), (-254.0, 0x4000), (63.5, 0x3800)):
        d16, q = oracle.split_blocks(oracle.quantize(np.full(32, c, np.float32)), 32)
        assert d16[0, 0] == dbits
        assert (q == (127 if c > 0 else -127)).all()
    x = np.zeros(32, np.float32)
    x[9] = -3.0
    d16, q = oracle.split_blocks(oracle.quantize(x), 32)
    assert q[0, 0, 9] == -127 and np.count_nonzero(q) == 1
    assert d16[0, 0] == np.float16(np.float32(3.0) / np.float32(127.0)).view(np.uint16)


def test_quantize_matches_exact_rounding_of_x_over_fp32_d():
    # q must be x/d rounded half away from zero, where d is the fp32 value of
    # amax/127 (not its fp16 copy).  x/d is evaluated exactly enough in fp64;
    # only values within 1e-5 of a rounding tie are excused (the single fp32
    # products x*(1/d) may land on either side there).
    x = q8_synth.normal_np((64, 32 * 16), 1.0, 5)
    x[0, :32] *= np.float32(1e-3)
    x[1, :32] *= np.float32(3e4)
    K = x.shape[1]
    d16, q = oracle.split_blocks(oracle.quantize(x), K)
    xb = x.reshape(64, -1, 32).astype(np.float64)
    amax = np.abs(x.reshape(64, -1, 32)).max(axis=2)
    d32 = (amax / np.float32(127.0)).astype(np.float32).astype(np.float64)
    ratio = xb / d32[:, :, None]
    frac = np.abs(np.abs(ratio) - np.floor(np.abs(ratio)) - 0.5)
    ok = frac > 1e-5
    expect = _round_half_away(ratio)
    assert np.array_equal(q[ok].astype(np.float64), expect[ok])
    assert ok.mean() > 0.999
    # |q| <= 127, never -128; the largest |x| of a block maps to +-127
    assert np.abs(q.astype(np.int32)).max() <= 127
    arg = np.abs(xb).argmax(axis=2)
    qmax = np.take_along_axis(q.astype(np.int32), arg[:, :, None], 2)[:, :, 0]
    assert (np.abs(qmax) == 127).all()
    # stored scale = fp16 (round to nearest even) of fp32 amax/127
    ref16 = (amax / np.float32(127.0)).astype(np.float32).astype(np.float16).view(np.uint16)
    assert np.array_equal(d16, ref16)


def test_dequantization_error_bounds():
    # |x - q*d| <= d/2 up to the fp32 rounding of 1/d and of x*(1/d)
    # (relative 3*2^-24 on |x/d| <= 127); against the stored fp16 scale
    # the bound widens by 127*|d - d16|.
    x = q8_synth.normal_np((128, 32 * 8), 1.0, 9).astype(np.float32)
    K = x.shape[1]
    d16, q = oracle.split_blocks(oracle.quantize(x), K)
    amax = np.abs(x.reshape(128, -1, 32)).max(axis=2)
    d = (amax / np.float32(127.0)).astype(np.float64)
    xb = x.reshape(128, -1, 32).astype(np.float64)
    err = np.abs(xb - q.astype(np.float64) * d[:, :, None])
    assert (err <= d[:, :, None] * (0.5 + 127 * 3 * 2.0**-24)).all()
    dh = d16.view(np.float16).astype(np.float64)
    err16 = np.abs(xb - q.astype(np.float64) * dh[:, :, None])
    assert (err16 <= (d * (0.5 + 127 * 3 * 2.0**-24) + 127 * np.abs(d - dh))[:, :, None] + 1e-30).all()


def test_quantize_symmetries():
    x = q8_synth.normal_np((8, 128), 1.0, 13)
    d0, q0 = oracle.split_blocks(oracle.quantize(x), 128)
    d1, q1 = oracle.split_blocks(oracle.quantize(-x), 128)
    assert np.array_equal(d0, d1) and np.array_equal(q0, -q1)
    # scaling by a power of two is exact in fp32: same quants, scale x 2^3
    d2, q2 = oracle.split_blocks(oracle.quantize(x * np.float32(8.0)), 128)
    assert np.array_equal(q0, q2)
    assert np.array_equal(d2.view(np.float16).astype(np.float64),
                          d0.view(np.float16).astype(np.float64) * 8.0)


# --------------------------------------------------------------------------
# block dots and the product: brute force
# --------------------------------------------------------------------------

def _dequant(blocks, K):
    d16, q = oracle.split_blocks(blocks, K)
    d = d16.view(np.float16).astype(np.float64)
    return (q.astype(np.float64) * d[:, :, None]).reshape(d.shape[0], K)


@pytest.mark.parametrize("N,K,M", [(5, 96, 3), (7, 32, 1), (16, 128, 4), (3, 160, 2)])
def test_block_dots_and_gemm_brute_force(N, K, M):
    W = oracle.quantize(q8_synth.normal_np((N, K), 0.02, 100 + N))
    A = oracle.quantize(q8_synth.normal_np((M, K), 1.0, 200 + M))
    isum = oracle.block_dots(W, A, K)
    _, qw = oracle.split_blocks(W, K)
    _, qa = oracle.split_blocks(A, K)
    ref = np.einsum("nbi,mbi->mnb", qw.astype(np.int64), qa.astype(np.int64))
    assert np.array_equal(isum.astype(np.int64), ref)
    # element-by-element fp64 product of the dequantized matrices
    y, S = oracle.gemm(W, A, K)
    yb = _dequant(A, K) @ _dequant(W, K).T
    assert y.shape == (M, N)
    assert np.allclose(y, yb, rtol=0, atol=1e-12 * (S.max() + 1e-300))
    assert (S >= np.abs(y) - 1e-15).all()


def test_block_dot_extremes_and_int32_bound():
    K = 64
    x = np.ones((1, K), np.float32)
    Wp = oracle.quantize(x)
    An = oracle.quantize(-x)
    assert oracle.block_dots(Wp, Wp, K)[0, 0].tolist() == [32 * 127 * 127] * 2
    assert oracle.block_dots(Wp, An, K)[0, 0].tolist() == [-516128] * 2
    W = oracle.quantize(q8_synth.normal_np((64, 256), 0.02, 1))
    A = oracle.quantize(q8_synth.normal_np((4, 256), 1.0, 2))
    assert np.abs(oracle.block_dots(W, A, 256)).max() <= 516128


def test_gemm_identity_like_weights():
    # Row n of W is one-hot at coordinate i_n of every block with value 127,
    # so d_w = 1 and q_w = 127 there: y[m][n] = 127 * sum_b q_a[m][b][i_n] * d_a[m][b].
    K, N, M = 96, 6, 2
    x = np.zeros((N, K), np.float32)
    idx = [0, 5, 31, 7, 16, 30]
    for n, i in enumerate(idx):
        x[n, i::32] = 127.0
    W = oracle.quantize(x)
    A = oracle.quantize(q8_synth.normal_np((M, K), 1.0, 21))
    y, S = oracle.gemm(W, A, K)
    d16, qa = oracle.split_blocks(A, K)
    da = d16.view(np.float16).astype(np.float64)
    for n, i in enumerate(idx):
        exp = 127.0 * (qa[:, :, i].astype(np.float64) * da).sum(axis=1)
        assert np.allclose(y[:, n], exp, rtol=1e-14, atol=0)


def test_gemm_nonnegative_terms_give_S_equal_y_and_fused_composition():
    K, N, M = 64, 4, 3
    W = oracle.quantize(np.abs(q8_synth.normal_np((N, K), 0.02, 31)))
    x = np.abs(q8_synth.normal_np((M, K), 1.0, 32))
    A = oracle.quantize(x)
    y, S = oracle.gemm(W, A, K)
    assert np.array_equal(y, S)
    yf, Sf, Af = oracle.quant_gemm(W, x, K)
    assert np.array_equal(Af, A) and np.array_equal(yf, y) and np.array_equal(Sf, S)


def test_golden_small_case_reproduces():
    """The stored small case (written by tests/golden/make_golden.py, which calls
    only oracle/) still reproduces: guards the oracle against silent drift."""
    import json
    with open(os.path.join(GOLDEN, "small_case.json")) as f:
        g = json.load(f)
    W = oracle.quantize(q8_synth.weights(g["N"], g["K"], g["seed_w"]).numpy())
    x = q8_synth.activations(g["M"], g["K"], g["seed_x"]).numpy()
    A = oracle.quantize(x)
    assert W.tobytes().hex() == g["W_blocks_hex"]
    assert A.tobytes().hex() == g["A_blocks_hex"]
    isum = oracle.block_dots(W, A, g["K"])
    assert isum.ravel().tolist() == g["isum"]
    y, S = oracle.gemm(W, A, g["K"])
    assert np.array_equal(y.ravel(), np.array(g["y"], dtype=np.float64))
