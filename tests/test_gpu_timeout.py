"""The decode GEMV's failure path, exercised without any fault.

Every wait of the GEMV kernels on their copy ring is bounded; a wait that
gives up sets a bit in the device error word, the kernel stops issuing,
lets the copies it issued land and returns.  The test hook
q8_set_wait_limit_ns shortens those waits to 1 ns, so the first wait that
cannot be satisfied at once gives up (the producer's first wait for a free
stage, while the consumers are still staging activations).  Nothing here
faults, traps or hangs: the kernel simply returns early.  The test checks
that the error is reported with the GEMV's role bits, that the drain of
copies in flight succeeded (its bound stays 2 s), and that the next call on
the same context gives the correct bits again.
"""
import pytest
import torch

import q8_synth

pytestmark = pytest.mark.gpu

DEV = "cuda"
ETIMEOUT_STATUS = 7  # -Q8_ETIMEOUT
ROLE_PRODUCER, ROLE_CONSUMER, ROLE_DRAIN = 1, 2, 4


@pytest.fixture(scope="module")
def q8():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    import q8_block_quantized_gb300 as q8mod
    assert q8mod.q8_device_error() == 0
    return q8mod


@pytest.fixture(scope="module")
def big(q8):
    # 608 tiles of 128 rows: four units of 8 rounds per CTA, so the three-stage
    # ring must be refilled and the producer has to wait for free stages
    N, K = 77824, 2048
    W = q8.pack_weights_f32(q8_synth.weights(N, K, q8_synth.derive_seed("timeout", N, K), DEV))
    torch.cuda.synchronize()
    return N, K, W


@pytest.mark.parametrize("M", [1, 4, 16])
def test_shortened_wait_reports_timeout_and_next_call_is_correct(q8, big, M):
    N, K, W = big
    x = q8_synth.activations(M, K, q8_synth.derive_seed("timeout-x", M), DEV)
    ws = q8.new_workspace(N, K, M)
    y_ref = torch.empty(M, N, device=DEV)
    q8.q8_fused_quant_gemm(W, N, K, x, M, y_ref, workspace=ws)
    assert q8.q8_device_error() == 0

    y = torch.full((M, N), 7.0, device=DEV)
    q8.q8_set_wait_limit_ns(1)
    try:
        q8.q8_fused_quant_gemm(W, N, K, x, M, y, workspace=ws)
        code = q8.q8_device_error()  # waits for the device
    finally:
        q8.q8_set_wait_limit_ns(0)
    assert code >> 8 == ETIMEOUT_STATUS, hex(code)
    roles = code & 0xFF
    assert roles & (ROLE_PRODUCER | ROLE_CONSUMER), hex(code)
    assert not roles & ROLE_DRAIN, "a copy in flight did not land within the drain's bound"
    assert not roles & ~(ROLE_PRODUCER | ROLE_CONSUMER), hex(code)

    # the context is usable and the workspace tickets are intact after a
    # re-zeroing (the documented recovery after a reported failure)
    if ws is not None:
        ws.zero_()
    y2 = torch.empty(M, N, device=DEV)
    q8.q8_fused_quant_gemm(W, N, K, x, M, y2, workspace=ws)
    assert q8.q8_device_error() == 0
    assert torch.equal(y2, y_ref)


@pytest.mark.parametrize("M", [16, 40])
def test_shortened_wait_on_k_split_shapes(q8, M):
    # 16 virtual tiles of 128 rows, K split 8 ways: the splits of a tile run
    # as one cluster and combine through distributed shared memory.  A
    # failed wait must not stop a CTA from signalling the others, and no CTA
    # may leave while another still reads its shared memory: the call ends,
    # reports the timeout without a drain failure, and the next call is right.
    N, K = 2048, 8192
    W = q8.pack_weights_f32(q8_synth.weights(N, K, q8_synth.derive_seed("timeout-split", N, K), DEV))
    x = q8_synth.activations(M, K, q8_synth.derive_seed("timeout-split-x", M), DEV)
    ws = q8.new_workspace(N, K, M)
    y_ref = torch.empty(M, N, device=DEV)
    q8.q8_fused_quant_gemm(W, N, K, x, M, y_ref, workspace=ws)
    assert q8.q8_device_error() == 0
    y = torch.empty(M, N, device=DEV)
    q8.q8_set_wait_limit_ns(1)
    try:
        q8.q8_fused_quant_gemm(W, N, K, x, M, y, workspace=ws)
        code = q8.q8_device_error()
    finally:
        q8.q8_set_wait_limit_ns(0)
    assert code >> 8 == ETIMEOUT_STATUS, hex(code)
    roles = code & 0xFF
    assert roles & (ROLE_PRODUCER | ROLE_CONSUMER), hex(code)
    assert not roles & ~(ROLE_PRODUCER | ROLE_CONSUMER), hex(code)
    if ws is not None:
        ws.zero_()
    y2 = torch.empty(M, N, device=DEV)
    q8.q8_fused_quant_gemm(W, N, K, x, M, y2, workspace=ws)
    assert q8.q8_device_error() == 0
    assert torch.equal(y2, y_ref)
