"""q8_gemm_noalloc: the GEMV for callers that cannot allocate device memory.

Such callers (for example a plugin whose host application owns the device's
memory, or a latency-critical loop that must not call cudaMalloc) cannot
hand q8_gemm a workspace; q8_gemm_noalloc uses scratch built into the library
instead.  These tests call it through the C ABI, twice in a row on shapes that
split along K (so the built-in scratch is used and reused), and check each
result against q8_gemm with a caller-allocated workspace: within the parity
tolerance used everywhere (|dy| <= 1e-5 * sum|terms| + 1e-6, sum|terms| from
the oracle) and, because both run the same reduction order, bit for bit.

Shapes of more than 32 rows run as several launches that reuse the scratch
one after the other; Q8_FLAG_PDL is covered too.

This file is collected last so a run that stops at the first failure has
already run every other test; it passes alone in a fresh process too.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import q8_synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def q8():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    import q8_block_quantized_gb300 as q8mod
    return q8mod


def _case(q8, N, K, M, seed):
    w = q8_synth.weights(N, K, q8_synth.derive_seed("na-w", N, K, seed))
    x = q8_synth.activations(M, K, q8_synth.derive_seed("na-x", M, K, seed))
    Wb = oracle.quantize(w.numpy())
    Ab = oracle.quantize(x.numpy())
    y_or, S = oracle.gemm(Wb, Ab, K)
    W = q8.pack_weights_f32(w.cuda())
    A = torch.from_numpy(Ab).cuda()
    return W, A, y_or, S


def _noalloc_raw(q8, W, N, K, A, M, y, flags=0):
    # straight through the C ABI with raw pointers
    st = q8.lib().q8_gemm_noalloc(ctypes.c_void_p(W.data_ptr()), N, K,
                                  ctypes.c_void_p(A.data_ptr()), M,
                                  ctypes.c_void_p(y.data_ptr()), flags,
                                  ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0, q8.lib().q8_strerror(st).decode()


# (N, K, M, whether the shape splits along K and so uses the scratch)
SHAPES = [(256, 8192, 16, True), (300, 4096, 16, True), (300, 4096, 40, True),
          (512, 2048, 1, False), (2048, 2048, 3, False)]


@pytest.mark.parametrize("N,K,M,split", SHAPES)
@pytest.mark.parametrize("flags", [0, 1])  # plain, and Q8_FLAG_PDL
def test_noalloc_matches_gemm_twice(q8, N, K, M, split, flags):
    assert (q8.q8_workspace_bytes(N, K, M) > 0) == split
    assert q8.q8_workspace_bytes(N, K, M) <= q8.NOALLOC_SCRATCH_BYTES
    results = []
    for call in range(2):  # two calls in a row reuse the same built-in scratch
        W, A, y_or, S = _case(q8, N, K, M, seed=call)
        ws = q8.new_workspace(N, K, M)
        y_ref = torch.full((M, N), float("nan"), device="cuda")
        q8.q8_gemm(W, N, K, A, M, y_ref, workspace=ws)
        y = torch.full((M, N), float("nan"), device="cuda")
        _noalloc_raw(q8, W, N, K, A, M, y, flags)
        torch.cuda.synchronize()
        # the oracle's fp64 product, within the parity tolerance
        err = (y.double().cpu().numpy() - y_or)
        assert (np.abs(err) <= 1e-5 * S + 1e-6).all(), (N, K, M, call, np.abs(err).max())
        # and bit for bit the call with a caller-allocated workspace
        assert torch.equal(y, y_ref)
        results.append(y)
    assert not torch.equal(results[0], results[1])  # different inputs, fresh results
    assert q8.q8_device_error() == 0


def test_noalloc_uses_scratch_for_split_shapes(q8):
    # the shapes above that split along K do need scratch, and it fits
    assert 0 < q8.q8_workspace_bytes(256, 8192, 16) <= q8.NOALLOC_SCRATCH_BYTES


def test_noalloc_rejects_shapes_beyond_scratch(q8):
    # a split shape whose partials exceed the built-in scratch: refused with
    # Q8_ESCRATCH before anything is enqueued (the first candidate the
    # planner splits that far)
    cands = [(4096, 65536, 64), (16384, 262144, 16), (16384, 1 << 20, 64)]
    big = [(N, K, M) for N, K, M in cands
           if q8.q8_workspace_bytes(N, K, M) > q8.NOALLOC_SCRATCH_BYTES]
    assert big, "no candidate shape needs more than the built-in scratch"
    N, K, M = big[0]
    W = torch.empty(16, dtype=torch.uint8, device="cuda")  # never read
    A = torch.empty(16, dtype=torch.uint8, device="cuda")
    y = torch.empty(16, dtype=torch.float32, device="cuda")
    st = q8.lib().q8_gemm_noalloc(ctypes.c_void_p(W.data_ptr()), N, K,
                                  ctypes.c_void_p(A.data_ptr()), M,
                                  ctypes.c_void_p(y.data_ptr()), 0, None)
    assert st == -8
    assert "scratch" in q8.lib().q8_strerror(st).decode()


def test_noalloc_stages_in_every_cta_when_the_images_do_not_fit(q8):
    # 64 rows (two launches of 32) at K = 32768: the activations staged once
    # per call would need more than the built-in scratch, the split's partial
    # sums alone fit -- the call stages its activations in every CTA instead
    # and computes the same bits as q8_gemm with a full workspace
    N, K, M = 256, 32768, 64
    assert q8.q8_workspace_bytes(N, K, M) > q8.NOALLOC_SCRATCH_BYTES
    W, A, y_or, S = _case(q8, N, K, M, seed=7)
    ws = q8.new_workspace(N, K, M)
    y_ref = torch.full((M, N), float("nan"), device="cuda")
    q8.q8_gemm(W, N, K, A, M, y_ref, workspace=ws)
    y = torch.full((M, N), float("nan"), device="cuda")
    _noalloc_raw(q8, W, N, K, A, M, y)
    torch.cuda.synchronize()
    err = (y.double().cpu().numpy() - y_or)
    assert (np.abs(err) <= 1e-5 * S + 1e-6).all(), np.abs(err).max()
    assert torch.equal(y, y_ref)
    assert q8.q8_device_error() == 0
