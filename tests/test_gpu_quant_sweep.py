"""GPU quantization swept over every significand of the block maximum.

The quantizer computes d = amax/127 and 1/d with division-free, correctly
rounded methods (checked on the host in test_quant_arith.py); this sweep
checks the device code itself through the public calls: 2^23 blocks whose
amax takes every float significand in [1, 2) (so d = amax/127 takes about
every value of its binade), the other 31 values of each block uniform in
(-amax, amax), plus blocks at the extreme exponents (subnormal amax, subnormal
d, amax near the top of the range).  The stored blocks must equal the
oracle's byte for byte (the quantization rule of "Q8_0 block quantization",
block format and scale rule).  The fused GEMV's staging quantizes with the same
functions spread over 8 lanes per block; its published activation blocks are
checked the same way on a sample of the sweep."""
import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def q8():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    import q8_block_quantized_gb300 as q8mod
    return q8mod


def _blocks_with_amax(amax: np.ndarray, seed: int) -> np.ndarray:
    """Blocks (rows of 32) whose largest magnitude is exactly amax[b]."""
    rng = np.random.default_rng(seed)
    nb = amax.size
    u = (rng.random((nb, 32), dtype=np.float32) * np.float32(2.0) - np.float32(1.0))
    x = u * amax[:, None]  # |RN(amax * u)| <= amax for |u| < 1
    pos = np.arange(nb) % 32
    sign = np.where(np.arange(nb) % 2 == 0, np.float32(1.0), np.float32(-1.0))
    x[np.arange(nb), pos] = amax * sign
    return x


def _check_quantize(q8, x2d: np.ndarray):
    rows, K = x2d.shape
    want = oracle.quantize(x2d)
    xd = torch.from_numpy(x2d).cuda()
    out = q8.empty_blocks(rows, K, "cuda")
    q8.q8_quantize_act(xd, out)
    torch.cuda.synchronize()
    got = out.cpu().numpy()
    bad = np.nonzero((got != want).reshape(rows, -1, 34).any(axis=2))
    assert bad[0].size == 0, "first differing block (row, block): %s" % ((bad[0][0], bad[1][0]),)


def test_every_significand_of_amax(q8):
    nb = 1 << 23
    amax = (np.uint32(127 << 23) | np.arange(nb, dtype=np.uint32)).view(np.float32)  # [1, 2)
    x = _blocks_with_amax(amax, seed=1)
    _check_quantize(q8, x.reshape(2048, -1))


@pytest.mark.parametrize("exp", [-149, -140, -126, -121, -119, -118, 0, 60, 120, 127])
def test_extreme_exponents(q8, exp):
    nb = 1 << 18
    rng = np.random.default_rng(exp + 1000)
    if exp == -149:  # any subnormal amax
        bits = rng.integers(1, 1 << 23, nb, dtype=np.uint32)
    elif exp < -126:  # subnormal amax with its leading bit at 2^exp
        bits = rng.integers(1 << (exp + 149), 1 << (exp + 150), nb, dtype=np.uint32)
    else:
        bits = np.uint32((exp + 127) << 23) | rng.integers(0, 1 << 23, nb, dtype=np.uint32)
    amax = bits.view(np.float32)
    x = _blocks_with_amax(amax, seed=exp + 2000)
    _check_quantize(q8, x.reshape(256, -1))


@pytest.mark.parametrize("exp", [0, -149, -126, -121, 120])
def test_fused_staging_publishes_the_same_blocks(q8, exp):
    # M = 16 rows of K = 65536 (2048 blocks each); the fused call quantizes
    # in its staging and publishes the blocks through A_out.  exp 0: amax
    # every 256th significand of [1, 2); otherwise random significands at
    # that exponent (subnormal amax at -149)
    M, K, N = 16, 65536, 128
    nb = M * K // 32
    if exp == 0:
        bits = np.uint32(127 << 23) | (np.arange(nb, dtype=np.uint32) * 256)
    else:
        rng = np.random.default_rng(exp + 3000)
        lo = 1 if exp == -149 else 0
        bits = (np.uint32(0 if exp == -149 else (exp + 127) << 23)
                | rng.integers(lo, 1 << 23, nb, dtype=np.uint32))
    x = _blocks_with_amax(bits.view(np.float32), seed=exp + 4000).reshape(M, K)
    want = oracle.quantize(x)
    W = q8.pack_weights_f32(torch.randn(N, K, device="cuda") * 0.02)
    y = torch.empty(M, N, device="cuda")
    A_out = q8.empty_blocks(M, K, "cuda")
    ws = q8.new_workspace(N, K, M)
    q8.q8_fused_quant_gemm(W, N, K, torch.from_numpy(x).cuda(), M, y, A_blocks_out=A_out,
                           workspace=ws)
    torch.cuda.synchronize()
    assert np.array_equal(A_out.cpu().numpy(), want)
    assert q8.q8_device_error() == 0
