"""Determinism of the GPU path ("Ember: packed Q8 decode", the measurement
paragraphs: a deterministic run is checked by hashing its output; "Ferrule":
results independent of the memory backing).

- The projection stack replayed twice, and built a second time from the same
  seeds, gives the same SHA-256 digest of all its outputs.
- q8_gemm and q8_gemm_prefill give the same bits whatever the (documented)
  alignment of their buffers: activation blocks at 2-byte offsets, y at
  4-byte offsets, W and the workspaces at other 16-byte-aligned addresses.
"""
import hashlib

import numpy as np
import pytest
import torch

import q8_synth

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module")
def q8():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    import q8_block_quantized_gb300 as q8mod
    return q8mod


def _digest(t: torch.Tensor) -> str:
    return hashlib.sha256(t.detach().cpu().numpy().tobytes()).hexdigest()


@pytest.mark.parametrize("M", [1, 4])
def test_stack_digest_is_stable(q8, M):
    from q8_block_quantized_gb300.stack import Q8Stack
    st = Q8Stack(q8_synth.LLAMA_1B, M=M, mode="fused", layers=2)
    g = st.capture()
    g.replay()
    torch.cuda.synchronize()
    d1 = _digest(st.y_all)
    st.y_all.fill_(float("nan"))
    g.replay()
    torch.cuda.synchronize()
    assert _digest(st.y_all) == d1
    st2 = Q8Stack(q8_synth.LLAMA_1B, M=M, mode="fused", layers=2)
    st2.step()
    torch.cuda.synchronize()
    assert _digest(st2.y_all) == d1
    assert q8.q8_device_error() == 0


def _at(buf: torch.Tensor, offset: int, nbytes: int) -> torch.Tensor:
    return buf[offset:offset + nbytes]


def test_gemm_bits_do_not_depend_on_buffer_addresses(q8):
    N, K, M = 3072, 2048, 4
    w = q8_synth.weights(N, K, q8_synth.derive_seed("det-w"), DEV)
    x = q8_synth.activations(M, K, q8_synth.derive_seed("det-x"), DEV)
    W0 = q8.pack_weights_f32(w)
    A0 = q8.empty_blocks(M, K)
    q8.q8_quantize_act(x, A0)
    wbytes, abytes = W0.numel(), A0.numel()
    ref = None
    for w_off, a_off, y_off in ((0, 0, 0), (16, 2, 4), (48, 34, 12), (4096, 6, 8)):
        Wbuf = torch.zeros(wbytes + w_off, dtype=torch.uint8, device=DEV)
        W = _at(Wbuf, w_off, wbytes)
        W.copy_(W0)
        Abuf = torch.zeros(abytes + a_off, dtype=torch.uint8, device=DEV)
        A = _at(Abuf, a_off, abytes).view(M, -1)
        A.copy_(A0)
        ybuf = torch.full((M * N + y_off // 4,), float("nan"), device=DEV)
        y = ybuf[y_off // 4:].view(M, N)
        q8.q8_gemm(W, N, K, A, M, y, workspace=q8.new_workspace(N, K, M))
        torch.cuda.synchronize()
        if ref is None:
            ref = y.clone()
        else:
            assert torch.equal(y.view(torch.int32), ref.view(torch.int32)), (w_off, a_off, y_off)
    assert q8.q8_device_error() == 0


def test_prefill_bits_do_not_depend_on_buffer_addresses(q8):
    N, K, M = 1000, 1568, 130
    w = q8_synth.weights(N, K, q8_synth.derive_seed("det-pw"), DEV)
    x = q8_synth.activations(M, K, q8_synth.derive_seed("det-px"), DEV)
    W0 = q8.pack_weights_f32(w)
    A0 = q8.empty_blocks(M, K)
    q8.q8_quantize_act(x, A0)
    wbytes, abytes = W0.numel(), A0.numel()
    wsb = q8.q8_prefill_workspace_bytes(K, M)
    ref = None
    for w_off, a_off, y_off, ws_off in ((0, 0, 0, 0), (16, 2, 4, 16), (96, 34, 8, 4096)):
        Wbuf = torch.zeros(wbytes + w_off, dtype=torch.uint8, device=DEV)
        W = _at(Wbuf, w_off, wbytes)
        W.copy_(W0)
        Abuf = torch.zeros(abytes + a_off, dtype=torch.uint8, device=DEV)
        A = _at(Abuf, a_off, abytes).view(M, -1)
        A.copy_(A0)
        ybuf = torch.full((M * N + y_off // 4,), float("nan"), device=DEV)
        y = ybuf[y_off // 4:].view(M, N)
        wsbuf = torch.full((wsb + ws_off,), 0xA5, dtype=torch.uint8, device=DEV)
        q8.q8_gemm_prefill(W, N, K, A, M, y, _at(wsbuf, ws_off, wsb))
        torch.cuda.synchronize()
        if ref is None:
            ref = y.clone()
            assert not np.isnan(ref.cpu().numpy()).any()
        else:
            assert torch.equal(y.view(torch.int32), ref.view(torch.int32)), (w_off, a_off, y_off, ws_off)
    assert q8.q8_device_error() == 0
