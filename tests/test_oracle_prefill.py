"""Pins of the oracle's prefill summation order (CPU only).

The prefill tile GEMM keeps, per output, one fixed single-precision order
("Ferro" README, "Exactness contract": prefill rows take the tile GEMM and a
row's result does not depend on how many rows share the launch or how the
prompt is sliced).  The reading: blocks in order, in segments of 16; inside
a segment sigma = fma(isum_b, d_w d_a, sigma) from +0; the segment sums of
the first ceil(nseg/2) segments (low half) and of the rest (high half) each
added in order from +0; y = Y_lo + Y_hi.  Pinned here by values derived by
hand (which fail for another segment length, a plain running sum, one
sequential sum over all segments, or a separately rounded product), by
single-rounding results computed exactly in fp64, and by the error bound
against the fp64 product.
"""
import math

import numpy as np
import pytest

import oracle
import q8_synth

U = 2.0 ** -24


def _block(d: float, q) -> np.ndarray:
    b = np.zeros(34, dtype=np.uint8)
    b[:2] = np.frombuffer(np.float16(d).tobytes(), dtype=np.uint8)
    qq = np.zeros(32, dtype=np.int8)
    qq[: len(q)] = q
    b[2:] = qq.view(np.uint8)
    return b


def _rows(blocks_per_row):
    return np.stack([np.concatenate(r) for r in blocks_per_row])


def test_segment_structure_by_hand():
    # W row: block 0 has isum 4 * 64 * 64 = 2^14 against the activation
    # block below and scales 32 * 32 -> term 2^24; blocks 1..15 give 1 each
    # (same segment as 2^24: each 2^24 + 1 is a tie that rounds back to
    # 2^24), blocks 16..31 give 1 each (sigma = 16), block 32 gives 1.
    # Order with segments of 16: Y = 2^24, then 2^24 + 16 (exact), then
    # 2^24 + 17 -> tie between 2^24 + 16 and 2^24 + 18, even significand:
    # 2^24 + 16.  Segments of 8 give 2^24 + 24, a running sum 2^24, the
    # exact sum 2^24 + 32.
    nb = 33
    w = [_block(32.0, [64, 64, 64, 64])] + [_block(1.0, [1]) for _ in range(nb - 1)]
    a = [_block(32.0, [64, 64, 64, 64])] + [_block(1.0, [1]) for _ in range(nb - 1)]
    W, A = _rows([w]), _rows([a])
    y = oracle.gemm_prefill_order(W, A, 32 * nb)
    assert y[0, 0] == np.float32(2.0 ** 24 + 16)
    assert oracle.gemm_prefill_order(W, A, 32 * nb, seg=8)[0, 0] == np.float32(2.0 ** 24 + 24)
    assert oracle.gemm_prefill_order(W, A, 32 * nb, seg=nb)[0, 0] == np.float32(2.0 ** 24)
    y64, _ = oracle.gemm(W, A, 32 * nb)
    assert y64[0, 0] == 2.0 ** 24 + 32


def test_halves_by_hand():
    # four segments of 16 blocks: segment 0 sums to 2^24 (block 0 as above,
    # its other blocks zero), segments 1, 2, 3 to 1 each.  Low half = the
    # first two segments: Y_lo = 2^24 + 1, a tie that rounds to 2^24; high
    # half Y_hi = 1 + 1 = 2; y = 2^24 + 2 (exact).  One sequential sum over
    # the four segments gives 2^24 (every + 1 is a tie back to 2^24); the
    # exact sum is 2^24 + 3.
    nb = 64
    w = [_block(32.0, [64, 64, 64, 64])] + [_block(0.0, []) for _ in range(nb - 1)]
    a = [_block(32.0, [64, 64, 64, 64])] + [_block(0.0, []) for _ in range(nb - 1)]
    for j in (16, 32, 48):
        w[j] = _block(1.0, [1])
        a[j] = _block(1.0, [1])
    W, A = _rows([w]), _rows([a])
    assert oracle.gemm_prefill_order(W, A, 32 * nb)[0, 0] == np.float32(2.0 ** 24 + 2)
    # one segment of all 64 blocks: a running fma sum, 2^24
    assert oracle.gemm_prefill_order(W, A, 32 * nb, seg=nb)[0, 0] == np.float32(2.0 ** 24)
    y64, _ = oracle.gemm(W, A, 32 * nb)
    assert y64[0, 0] == 2.0 ** 24 + 3
    # three segments (K = 48 blocks): low half = two segments, high half the
    # third alone: Y_lo = 2^24 (tie), Y_hi = 1, y = 2^24 + 1 -> tie -> 2^24
    W3, A3 = _rows([w[:48]]), _rows([a[:48]])
    assert oracle.gemm_prefill_order(W3, A3, 32 * 48)[0, 0] == np.float32(2.0 ** 24)


def _fused_case():
    # two blocks in one segment: t0 = 1 exactly, then isum1 * s1 with s1
    # = dw * da carrying 21 significant bits, so the product is inexact in
    # fp32.  Search for a case where one rounding of (t0 + isum1 s1) and two
    # roundings (product first) disagree; both are computed from exact fp64
    # values (every quantity here fits 53 bits).
    for dw_k in range(1, 200):
        dw = 1.0 + dw_k * 2.0 ** -10
        for da_k in range(1, 64):
            da = 1.0 + da_k * 2.0 ** -10
            for isum in range(3001, 4064, 7):
                s = dw * da  # exact in fp64 and in fp32 (22 bits)
                exact = isum * s + 1.0
                one = np.float32(exact)
                two = np.float32(np.float32(isum * s) + np.float32(1.0))
                if one != two:
                    return dw, da, isum, one, two
    raise AssertionError("no case found")


def test_fma_rounds_once():
    dw, da, isum, one, two = _fused_case()
    # isum from 127-valued quants against ones, remainder in one lane
    qw = [127] * (isum // 127) + [isum % 127]
    assert sum(qw) == isum and len(qw) <= 32
    W = _rows([[_block(1.0, [1]), _block(dw, qw)]])
    A = _rows([[_block(1.0, [1]), _block(da, [1] * len(qw))]])
    y = oracle.gemm_prefill_order(W, A, 64)
    assert y[0, 0] == one and y[0, 0] != two


def test_single_block_is_the_rounded_product():
    rng = np.random.default_rng(7)
    for _ in range(200):
        q1 = rng.integers(-127, 128, size=32)
        q2 = rng.integers(-127, 128, size=32)
        d1 = float(np.float16(rng.uniform(1e-4, 2.0)))
        d2 = float(np.float16(rng.uniform(1e-4, 2.0)))
        W, A = _rows([[_block(d1, q1)]]), _rows([[_block(d2, q2)]])
        isum = int(np.dot(q1, q2))
        y = oracle.gemm_prefill_order(W, A, 32)[0, 0]
        assert y == np.float32(isum * (d1 * d2))  # one rounding of an exact fp64 value


@pytest.mark.parametrize("K", [32, 512, 2048, 8192, 65536])
def test_error_bound_against_fp64(K):
    rng_seed = q8_synth.derive_seed("pf-pin", K)
    N, M = (3, 2) if K == 65536 else (6, 5)
    w = q8_synth.normal_np((N, K), 0.02, rng_seed)
    x = q8_synth.normal_np((M, K), 1.0, rng_seed + 1)
    W, A = oracle.quantize(w), oracle.quantize(x)
    y = oracle.gemm_prefill_order(W, A, K).astype(np.float64)
    y64, S = oracle.gemm(W, A, K)
    nb = K // 32
    bound = (17 + math.ceil(nb / 16)) * U * S
    assert (np.abs(y - y64) <= bound).all()
    assert (bound <= 1e-5 * S).all()


def test_error_bound_same_sign_terms():
    # every term positive: the running sums grow to S, the worst case for
    # the sequential parts of the order
    K = 65536
    rng = np.random.default_rng(11)
    w = np.abs(rng.standard_normal((2, K))).astype(np.float32)
    x = np.abs(rng.standard_normal((1, K))).astype(np.float32)
    W, A = oracle.quantize(w), oracle.quantize(x)
    y = oracle.gemm_prefill_order(W, A, K).astype(np.float64)
    y64, S = oracle.gemm(W, A, K)
    assert (np.abs(y - y64) <= (17 + 128) * U * S).all()


def test_rows_are_independent_of_the_batch():
    K = 1024
    w = q8_synth.normal_np((7, K), 0.02, q8_synth.derive_seed("pf-ind", 0))
    x = q8_synth.normal_np((9, K), 1.0, q8_synth.derive_seed("pf-ind", 1))
    W, A = oracle.quantize(w), oracle.quantize(x)
    y = oracle.gemm_prefill_order(W, A, K)
    for m in (0, 4, 8):
        assert np.array_equal(oracle.gemm_prefill_order(W, A[m:m + 1], K)[0], y[m])
