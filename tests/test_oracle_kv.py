"""Pins for the oracle's int8 KV cache codec (oracle.kv_quantize /
oracle.kv_dequantize): checks against facts fixed outside the oracle.

- the byte accounting the pages print for the int8 cache
  (tests/golden/kv_accounting.txt);
- the codebook: the quants of a 32-value block equal those of the
  activation quantizer (pinned on its own in test_oracle_pins.py), the
  stored scale equals amax / 127 as numpy's IEEE single-precision division
  gives it, unrounded;
- closed forms: a block with amax = 127 has scale exactly 1 (quants are the
  values rounded half away from zero), zero and constant blocks;
- dequantization: numpy's single-precision product q * d, and the error
  bound |x - x'| <= d/2 (plus the rounding of x = q*d and of 1/d);
- slot addressing: scatter then gather returns the rows, slots not named
  keep what they held, slots outside the cache are skipped.

A slip such as the scale stored as binary16, 1/d taken from a rounded
scale, ties to even, a scale per 16 or 64 values, a transposed slot index or
a dequantization by division fails at least one of them.
"""
import os

import numpy as np
import pytest

import oracle
import q8_synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _facts():
    facts = {}
    with open(os.path.join(GOLDEN, "kv_accounting.txt")) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                k, v = line.split()
                facts[k] = int(v)
    return facts


def _round_half_away(v):
    v = np.asarray(v, dtype=np.float64)  # v + 0.5 exact in fp64 for these values
    return np.sign(v) * np.floor(np.abs(v) + 0.5)


def test_kv_accounting_matches_pages():
    f = _facts()
    c = oracle.constants()
    assert c["kv_block_bytes"] == f["kv_scale_values"] + f["kv_scale_bytes"] == 36
    # f32 holds 4 bytes per value: the int8 cache is 36/128 of it, f16 64/128
    f32_block = 4 * f["kv_scale_values"]
    assert f["kv_f32_mb"] * c["kv_block_bytes"] == f["kv_int8_mb"] * f32_block
    assert f["kv_f32_mb"] * 2 * f["kv_scale_values"] == f["kv_f16_mb"] * f32_block
    # the oracle's planes hold exactly that many bytes
    cap, D = 7, 96
    q, d = oracle.kv_quantize(np.zeros((cap, D), np.float32), cap)
    assert q.nbytes + d.nbytes == cap * (D // 32) * c["kv_block_bytes"]
    assert q.shape == (cap, D) and d.shape == (cap, D // 32)


@pytest.mark.parametrize("std", [1.0, 0.02, 1e-30, 3e4])
def test_kv_codes_are_the_q8_codebook_with_the_fp32_scale(std):
    rows, D = 40, 256
    x = q8_synth.normal_np((rows, D), std, 11)
    x[3, 32:64] = 0.0                    # a zero block
    x[5, :32] = np.float32(std)          # a constant block
    q, d = oracle.kv_quantize(x, rows)
    blocks = oracle.quantize(x)          # the activation quantizer (pinned on its own)
    d16, qa = oracle.split_blocks(blocks, D)
    assert np.array_equal(q.reshape(rows, D // 32, 32), qa)
    amax = np.abs(x.reshape(rows, D // 32, 32)).max(axis=2)
    d_ref = (amax.astype(np.float32) / np.float32(127.0)).astype(np.float32)
    assert np.array_equal(d.view(np.uint32), d_ref.view(np.uint32))
    # rounding the fp32 scale to binary16 gives the activation block's scale
    assert np.array_equal(d.astype(np.float16).view(np.uint16), d16)


def test_kv_unit_scale_ties_and_closed_forms():
    v = np.zeros(32, np.float32)
    v[0] = 127.0
    v[1:9] = [2.5, -2.5, 0.5, -0.5, 1.49999988, -3.5, 0.49999997, 126.5]
    q, d = oracle.kv_quantize(v[None, :], 1)
    assert d[0, 0] == 1.0
    assert np.array_equal(q[0], _round_half_away(v).astype(np.int8))
    assert list(q[0, :9]) == [127, 3, -3, 1, -1, 1, -4, 0, 127]
    assert np.array_equal(oracle.kv_dequantize(q, d)[0], q[0].astype(np.float32))
    # zero block: scale 0, codes 0, values 0
    q, d = oracle.kv_quantize(np.zeros((1, 32), np.float32), 1)
    assert d[0, 0] == 0.0 and not q.any() and not oracle.kv_dequantize(q, d).any()
    # constant block c: every code 127, value 127 * fl(c / 127)
    for c in (1.0, -0.3, 1e-20, 5e3):
        q, d = oracle.kv_quantize(np.full((1, 32), c, np.float32), 1)
        dc = np.float32(np.float32(abs(c)) / np.float32(127.0))
        assert d[0, 0] == dc
        assert (q[0] == (127 if c > 0 else -127)).all()
        assert (oracle.kv_dequantize(q, d)[0] == np.float32(q[0, 0]) * dc).all()
    # one-hot block: a single +-127
    v = np.zeros((1, 32), np.float32)
    v[0, 17] = -0.75
    q, d = oracle.kv_quantize(v, 1)
    assert q[0, 17] == -127 and np.count_nonzero(q) == 1


def test_kv_dequantize_is_the_single_precision_product_and_error_bound():
    rows, D = 64, 512
    x = q8_synth.normal_np((rows, D), 1.0, 12) * np.exp(q8_synth.normal_np((rows, 1), 3.0, 13))
    x = x.astype(np.float32)
    q, d = oracle.kv_quantize(x, rows)
    y = oracle.kv_dequantize(q, d)
    dd = np.repeat(d, 32, axis=1)
    assert np.array_equal(y.view(np.uint32), (q.astype(np.float32) * dd).view(np.uint32))
    # |x - q d| <= d/2 (1 + 2^-22) for the exact product; the stored value adds
    # the product's own rounding (half an ulp of |y|)
    err = np.abs(x.astype(np.float64) - y.astype(np.float64))
    bound = dd.astype(np.float64) / 2 * (1 + 2.0 ** -22) + np.abs(y.astype(np.float64)) * 2.0 ** -24
    assert (err <= bound).all()
    # and the bound is nearly reached (a scale per 32 values, not finer)
    assert (err / dd).max() > 0.45


def test_kv_slots_scatter_gather_and_untouched_slots():
    D, cap = 128, 50
    rng = np.random.default_rng(14)
    x = q8_synth.normal_np((20, D), 1.0, 15)
    slots = rng.permutation(cap)[:20].astype(np.int32)
    sentinel_q = np.full((cap, D), 99, np.int8)
    sentinel_d = np.full((cap, D // 32), -7.0, np.float32)
    q, d = oracle.kv_quantize(x, cap, slots=slots, cache=(sentinel_q, sentinel_d))
    # each row lands in its slot exactly as a row quantized alone
    q1, d1 = oracle.kv_quantize(x, 20)
    assert np.array_equal(q[slots], q1) and np.array_equal(d[slots], d1)
    others = np.setdiff1d(np.arange(cap), slots)
    assert (q[others] == 99).all() and (d[others] == -7.0).all()
    # gathering by the same slots returns the rows' dequantized values
    assert np.array_equal(oracle.kv_dequantize(q, d, slots=slots), oracle.kv_dequantize(q1, d1))
    # a slot outside the cache is skipped (written nowhere, read as zero)
    bad = slots.copy()
    bad[3], bad[7] = cap, -1
    q2, d2 = oracle.kv_quantize(x, cap, slots=bad)
    assert not q2[slots[3]].any() and not q2[slots[7]].any()
    out = oracle.kv_dequantize(q1, d1, slots=np.array([0, 20, -1, 19], np.int32))
    assert out[1].sum() == 0 and out[2].sum() == 0 and np.array_equal(out[3], oracle.kv_dequantize(q1, d1)[19])
