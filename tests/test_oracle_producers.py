"""Pins of the oracle's fused producers (CPU only): the residual add + RMSNorm
+ quantization and the SwiGLU + quantization that emit the next GEMM's int8
input ("Ferro" README, "How the iGPU path is fast", item 3).

The pages give no arithmetic for these fusions; the readings (pairwise sum
of squares, ms = s / K, r = 1 / sqrt(ms + eps), y = (h * r) * gamma; silu(g)
= g / (1 + e^-g) with a fixed single-precision e^x) are pinned here against
things other than the oracle: values derived by hand, math.exp / fp64
numpy, numpy's float32 arithmetic, closed forms and invariances.
"""
import math

import numpy as np
import pytest

import oracle

ULP = 2.0 ** -23


def _dequant(blocks, K):
    d, q = oracle.split_blocks(blocks, K)
    return q.astype(np.float64) * oracle.f16_bits_to_f32(d).astype(np.float64)[..., None]


# ---- pairwise sum ----------------------------------------------------------------

def test_pairwise_sum_small_integers_exact():
    rng = np.random.default_rng(0)
    for n in (1, 2, 3, 7, 64, 1000, 3072):
        v = rng.integers(-1000, 1000, size=n)
        assert oracle.pairwise_sum(v.astype(np.float32)) == float(v.sum())


def test_pairwise_sum_tree_order_and_zero_padding_by_hand():
    e = 2.0 ** -24
    # (1 + 0) + (e + e) = 1 + 2^-23; left to right would give 1 (each 1 + e
    # is a tie that rounds to even, i.e. back to 1)
    assert oracle.pairwise_sum([1.0, 0.0, e, e]) == 1.0 + 2 * e
    # three values are padded to four leaves: (e + e) + (1 + 0) = 1 + 2^-23,
    # whereas e + (e + 1) would round to 1
    assert oracle.pairwise_sum([e, e, 1.0]) == 1.0 + 2 * e
    assert oracle.pairwise_sum([1.0, e]) == 1.0


def test_pairwise_sum_close_to_exact_sum():
    rng = np.random.default_rng(1)
    for n in (5, 96, 2048, 5000):
        v = rng.standard_normal(n).astype(np.float32) ** 2
        exact = math.fsum(float(a) for a in v)
        depth = math.ceil(math.log2(n)) + 1
        assert abs(oracle.pairwise_sum(v) - exact) <= depth * 2.0 ** -24 * exact


# ---- e^x and silu ------------------------------------------------------------------

def test_exp_against_math_exp():
    x = np.linspace(-87.0, 88.0, 400_001, dtype=np.float32)
    e = oracle.exp_f32(x).astype(np.float64)
    ref = np.exp(x.astype(np.float64))
    rel = np.abs(e - ref) / ref
    assert ref.min() >= 2.0 ** -126  # the whole domain has normal results
    assert rel.max() <= 3 * ULP
    assert oracle.exp_f32(np.float32(0.0)) == 1.0


def test_exp_domain_ends():
    e = oracle.exp_f32(np.array([88.0001, 100.0, np.inf, -87.0001, -200.0, -np.inf], dtype=np.float32))
    assert np.isinf(e[:3]).all() and (e[:3] > 0).all()
    assert (e[3:] == 0.0).all()


def test_silu_values():
    g = np.linspace(-20.0, 20.0, 20_001, dtype=np.float32)
    s = oracle.silu_f32(g).astype(np.float64)
    gd = g.astype(np.float64)
    ref = gd / (1.0 + np.exp(-gd))
    nz = np.abs(ref) > 1e-30
    assert (np.abs(s - ref)[nz] / np.abs(ref[nz])).max() <= 6 * ULP
    # silu(g) - silu(-g) = g (sigma(g) + sigma(-g) = 1)
    odd = s - oracle.silu_f32(-g).astype(np.float64)
    assert np.abs(odd - gd).max() <= 8 * ULP * np.abs(gd).max()
    assert oracle.silu_f32(np.float32(0.0)) == 0.0
    big = np.array([88.5, 1000.0], dtype=np.float32)
    assert np.array_equal(oracle.silu_f32(big), big)              # e^-g = 0
    neg = oracle.silu_f32(np.array([-88.5, -1000.0], dtype=np.float32))
    assert (neg == 0.0).all() and np.signbit(neg).all()            # g / inf = -0


# ---- residual + RMSNorm + quantization ---------------------------------------------

def test_residual_add_is_float32_addition():
    rng = np.random.default_rng(2)
    x = rng.standard_normal((3, 96)).astype(np.float32)
    d = rng.standard_normal((3, 96)).astype(np.float32)
    h, _ = oracle.residual_rmsnorm_quantize(x, d, np.ones(96, np.float32), 1e-5)
    assert np.array_equal(h, x + d)
    h0, _ = oracle.residual_rmsnorm_quantize(x, None, np.ones(96, np.float32), 1e-5)
    assert np.array_equal(h0, x)


@pytest.mark.parametrize("K", [32, 96, 2048])
def test_rmsnorm_constant_row_closed_form(K):
    # h = +-2^j everywhere: ms = 4^j, r = 2^-j exactly (eps far below an ulp
    # of ms), y = +-1, so every block has d = 1/127 and q = +-127
    for c in (4.0, -0.25):
        x = np.full((1, K), c, dtype=np.float32)
        _, b = oracle.residual_rmsnorm_quantize(x, None, np.ones(K, np.float32), 1e-12)
        d, q = oracle.split_blocks(b, K)
        assert (q == (127 if c > 0 else -127)).all()
        assert (d == oracle.f32_to_f16_bits(np.float32(1.0) / np.float32(127.0))).all()


def test_rmsnorm_scale_invariance_exact():
    rng = np.random.default_rng(3)
    x = rng.standard_normal((4, 3072)).astype(np.float32)
    g = (1.0 + 0.1 * rng.standard_normal(3072)).astype(np.float32)
    _, b1 = oracle.residual_rmsnorm_quantize(x, None, g, 1e-30)
    _, b2 = oracle.residual_rmsnorm_quantize(np.float32(8.0) * x, None, g, 1e-30)
    assert np.array_equal(b1, b2)


@pytest.mark.parametrize("K,eps", [(2048, 1e-5), (96, 0.5), (8192, 1e-6)])
def test_rmsnorm_against_fp64(K, eps):
    rng = np.random.default_rng(K)
    M = 3
    x = rng.standard_normal((M, K)).astype(np.float32)
    d = (0.5 * rng.standard_normal((M, K))).astype(np.float32)
    g = (1.0 + 0.2 * rng.standard_normal(K)).astype(np.float32)
    h, b = oracle.residual_rmsnorm_quantize(x, d, g, eps)
    h64 = (x + d).astype(np.float64)
    y64 = h64 / np.sqrt((h64 ** 2).mean(axis=1, keepdims=True) + eps) * g.astype(np.float64)
    deq = _dequant(b, K).reshape(M, K)
    amax = np.abs(y64).reshape(M, K // 32, 32).max(axis=2)
    bound = 0.5625 * amax / 127.0 + 16 * ULP * amax
    err = np.abs(deq - y64).reshape(M, K // 32, 32).max(axis=2)
    assert (err <= bound).all()


# ---- SwiGLU + quantization ----------------------------------------------------------

def test_swiglu_zero_up_gives_zero_blocks():
    gu = np.zeros((2, 128), dtype=np.float32)
    gu[:, :64] = np.random.default_rng(4).standard_normal((2, 64))
    b = oracle.swiglu_quantize(gu, 64)
    assert not b.any()


def test_swiglu_large_gate_is_plain_product():
    # gate >= 88: e^-gate = 0 and silu(gate) = gate exactly, so h = gate * up
    rng = np.random.default_rng(5)
    F = 96
    g = (100.0 + rng.random((3, F)) * 50).astype(np.float32)
    u = rng.standard_normal((3, F)).astype(np.float32)
    b = oracle.swiglu_quantize(np.concatenate([g, u], axis=1), F)
    assert np.array_equal(b, oracle.quantize(g * u))


def test_swiglu_against_fp64():
    rng = np.random.default_rng(6)
    M, F = 4, 8192
    gu = (2.0 * rng.standard_normal((M, 2 * F))).astype(np.float32)
    b = oracle.swiglu_quantize(gu, F)
    g = gu[:, :F].astype(np.float64)
    u = gu[:, F:].astype(np.float64)
    h64 = g / (1.0 + np.exp(-g)) * u
    deq = _dequant(b, F).reshape(M, F)
    amax = np.abs(h64).reshape(M, F // 32, 32).max(axis=2)
    err = np.abs(deq - h64).reshape(M, F // 32, 32).max(axis=2)
    assert (err <= 0.5625 * amax / 127.0 + 16 * ULP * amax).all()
