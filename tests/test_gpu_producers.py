"""Parity of the fused producers with the oracle, through the C ABI: the
residual add + RMSNorm + quantization and SwiGLU + quantization ("Ferro"
README, "How the iGPU path is fast", item 3).  Both emit Q8_0 blocks, which
must equal the oracle's bit for bit, as must the residual stream h_out.
"""
import numpy as np
import pytest
import torch

import oracle
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


def _normal(shape, std, *seed):
    return q8_synth.normal_np(shape, std, q8_synth.derive_seed("prod", *seed))


@pytest.mark.parametrize("M,K", [(1, 32), (3, 96), (2, 512), (1, 2048), (5, 3072), (64, 2048),
                                 (2, 8192), (3, 16416), (1024, 2048)])
@pytest.mark.parametrize("mode", ["x", "x+delta", "inplace"])
def test_rmsnorm_quantize_matches_oracle(q8, M, K, mode):
    x = _normal((M, K), 1.0, "x", M, K)
    delta = _normal((M, K), 0.7, "d", M, K) if mode != "x" else None
    gamma = (1.0 + _normal((K,), 0.3, "g", K)).astype(np.float32)
    eps = 1e-5 if K != 96 else 0.5
    if M >= 3:
        x[1] = 0.0           # a zero row: y = 0, zero blocks
        if delta is not None:
            delta[1] = 0.0
        x[2, : K // 2] *= 1e3  # a wide dynamic range inside a row
    h_ref, b_ref = oracle.residual_rmsnorm_quantize(x, delta, gamma, eps)
    xd = torch.from_numpy(x).to(DEV)
    dd = None if delta is None else torch.from_numpy(delta).to(DEV)
    gd = torch.from_numpy(gamma).to(DEV)
    out = torch.full((M, (K // 32) * 34), 0xAB, dtype=torch.uint8, device=DEV)
    if mode == "inplace":
        q8.q8_residual_rmsnorm_quantize(xd, gd, eps, out, delta=dd, h_out=xd)
        h = xd
    else:
        h = torch.full((M, K), float("nan"), device=DEV)
        q8.q8_residual_rmsnorm_quantize(xd, gd, eps, out, delta=dd, h_out=h)
    torch.cuda.synchronize()
    assert np.array_equal(out.cpu().numpy(), b_ref)
    assert np.array_equal(h.cpu().numpy(), h_ref)
    if mode == "x":  # without h_out the kernel recomputes h for the second pass
        out2 = torch.zeros_like(out)
        q8.q8_residual_rmsnorm_quantize(torch.from_numpy(x).to(DEV), gd, eps, out2)
        torch.cuda.synchronize()
        assert np.array_equal(out2.cpu().numpy(), b_ref)


@pytest.mark.parametrize("M,F", [(1, 32), (5, 96), (1, 8192), (64, 8192), (1024, 2048), (3, 11008)])
def test_swiglu_quantize_matches_oracle(q8, M, F):
    gu = _normal((M, 2 * F), 2.0, "gu", M, F)
    if M >= 5:
        # gate values across e^-g's whole domain and its ends
        n = min(F, 4096)
        gu[0, :n] = np.linspace(-100.0, 100.0, n, dtype=np.float32)
        gu[1, :n] = np.linspace(-88.5, -86.5, n, dtype=np.float32)
        gu[2, :n] = np.linspace(86.5, 88.5, n, dtype=np.float32)
        gu[3, F:] = 0.0  # up = 0: zero blocks
    ref = oracle.swiglu_quantize(gu, F)
    out = torch.full((M, (F // 32) * 34), 0xCD, dtype=torch.uint8, device=DEV)
    q8.q8_swiglu_quantize(torch.from_numpy(gu).to(DEV), out)
    torch.cuda.synchronize()
    assert np.array_equal(out.cpu().numpy(), ref)


def test_producers_feed_the_gemv_and_chain_with_pdl(q8):
    # residual + norm -> q8_gemm (gate/up) -> SwiGLU -> q8_gemm (down), as a
    # graph with programmatic dependent launch, against the oracle chain
    M, K, F = 2, 2048, 8192
    x = _normal((M, K), 1.0, "cx")
    delta = _normal((M, K), 0.5, "cd")
    gamma = (1.0 + _normal((K,), 0.2, "cg")).astype(np.float32)
    w_gu = q8_synth.weights(2 * F, K, q8_synth.derive_seed("cwgu"), DEV)
    w_dn = q8_synth.weights(K, F, q8_synth.derive_seed("cwdn"), DEV)
    Wgu, Wdn = q8.pack_weights_f32(w_gu), q8.pack_weights_f32(w_dn)
    xd, dd, gd = (torch.from_numpy(a).to(DEV) for a in (x, delta, gamma))
    A1 = q8.empty_blocks(M, K)
    y1 = torch.empty((M, 2 * F), device=DEV)
    A2 = q8.empty_blocks(M, F)
    y2 = torch.empty((M, K), device=DEV)
    h = torch.empty((M, K), device=DEV)
    ws1, ws2 = q8.new_workspace(2 * F, K, M), q8.new_workspace(K, F, M)

    def step():
        q8.q8_residual_rmsnorm_quantize(xd, gd, 1e-5, A1, delta=dd, h_out=h, flags=q8.FLAG_PDL)
        q8.q8_gemm(Wgu, 2 * F, K, A1, M, y1, workspace=ws1, flags=q8.FLAG_PDL)
        q8.q8_swiglu_quantize(y1, A2, flags=q8.FLAG_PDL)
        q8.q8_gemm(Wdn, K, F, A2, M, y2, workspace=ws2, flags=q8.FLAG_PDL)

    step()
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        step()
    y2.fill_(float("nan"))
    g.replay()
    torch.cuda.synchronize()
    h_ref, A1_ref = oracle.residual_rmsnorm_quantize(x, delta, gamma, 1e-5)
    assert np.array_equal(A1.cpu().numpy(), A1_ref) and np.array_equal(h.cpu().numpy(), h_ref)
    # the GEMV's output is checked against the oracle within tolerance; the
    # SwiGLU input is the GPU's own y1 (its bits are the GEMV's), so A2 is exact
    Wb_gu = oracle.quantize(w_gu.cpu().numpy())
    y1_ref, S1 = oracle.gemm(Wb_gu, A1_ref, K)
    assert (np.abs(y1.double().cpu().numpy() - y1_ref) <= 1e-5 * S1 + 1e-6).all()
    A2_ref = oracle.swiglu_quantize(y1.cpu().numpy(), F)
    assert np.array_equal(A2.cpu().numpy(), A2_ref)
    y2_ref, S2 = oracle.gemm(oracle.quantize(w_dn.cpu().numpy()), A2_ref, F)
    assert (np.abs(y2.double().cpu().numpy() - y2_ref) <= 1e-5 * S2 + 1e-6).all()
    assert q8.q8_device_error() == 0


@pytest.mark.parametrize("F,K,M", [(8192, 2048, 1), (8192, 2048, 3), (4864, 3072, 16), (8192, 2048, 33),
                                   (2496, 512, 5)])
def test_swiglu_epilogue_gemv(q8, F, K, M):
    # gate/up GEMV with SwiGLU in its epilogue: equal, bit for bit, to
    # SwiGLU + quantization of the plain GEMV's outputs on the same W
    gate = q8_synth.weights(F, K, q8_synth.derive_seed("sw-g", F, K), DEV)
    up = q8_synth.weights(F, K, q8_synth.derive_seed("sw-u", F, K), DEV)
    W = q8.pack_weights_f32(q8.interleave_gate_up(gate, up))
    x = q8_synth.activations(M, K, q8_synth.derive_seed("sw-x", M, K), DEV)
    A = q8.empty_blocks(M, K)
    q8.q8_quantize_act(x, A)
    out = torch.full((M, (F // 32) * 34), 0xEE, dtype=torch.uint8, device=DEV)
    q8.q8_gemm_swiglu(W, F, K, A, M, out)
    outf = torch.zeros_like(out)
    q8.q8_fused_quant_gemm_swiglu(W, F, K, x, M, outf, flags=q8.FLAG_PDL)
    y = torch.empty((M, 2 * F), dtype=torch.float32, device=DEV)
    q8.q8_gemm(W, 2 * F, K, A, M, y, workspace=q8.new_workspace(2 * F, K, M))
    torch.cuda.synchronize()
    G = q8.q8_packed_tile_rows(2 * F) // 2
    yg = y.view(M, F // G, 2, G)
    gu = torch.cat([yg[:, :, 0, :].reshape(M, F), yg[:, :, 1, :].reshape(M, F)], dim=1)
    ref = oracle.swiglu_quantize(gu.cpu().numpy(), F)
    assert np.array_equal(out.cpu().numpy(), ref)
    assert np.array_equal(outf.cpu().numpy(), ref)
    # the GEMV part against the oracle on sampled rows of the interleaved matrix
    rows = np.array([0, G - 1, G, 2 * G, 2 * F - 1])
    w_rows = q8.interleave_gate_up(gate, up)[torch.from_numpy(rows).to(DEV)].cpu().numpy()
    y_ref, S_ref = oracle.gemm(oracle.quantize(w_rows), A.cpu().numpy(), K)
    err = np.abs(y[:, torch.from_numpy(rows).to(DEV)].double().cpu().numpy() - y_ref)
    assert (err <= 1e-5 * S_ref + 1e-6).all()
    assert q8.q8_device_error() == 0


def test_swiglu_epilogue_gemv_shape_errors(q8):
    dummy = torch.zeros(64, dtype=torch.uint8, device=DEV)
    xd = torch.zeros(64, dtype=torch.float32, device=DEV)
    for F, K, M in ((2432, 512, 1),       # 32-row tiles: no epilogue layout
                    (8192 + 32, 512, 1),  # F not a multiple of the group
                    (8192, 65536, 16)):   # would split along K
        with pytest.raises(q8.Q8Error) as e:
            q8._check("q8_gemm_swiglu", q8.lib().q8_gemm_swiglu(dummy.data_ptr(), F, K, dummy.data_ptr(), M,
                                                                dummy.data_ptr(), 0, None))
        assert e.value.status == -2
    with pytest.raises(q8.Q8Error) as e:
        q8._check("q8_fused_quant_gemm_swiglu", q8.lib().q8_fused_quant_gemm_swiglu(
            dummy.data_ptr(), 8192, 2048, xd.data_ptr(), 1, dummy.data_ptr(), 2, None))
    assert e.value.status == -1  # the tcgen05 option is not offered here
