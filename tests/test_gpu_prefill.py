"""Parity of the prefill tile GEMM (q8_gemm_prefill, q8_fused_quant_gemm_prefill)
with the oracle, through the C ABI.

The GPU result must equal, bit for bit, the oracle's statement of the fixed
prefill order (oracle.gemm_prefill_order, pinned in test_oracle_prefill.py),
lie within the library tolerance of the fp64 product, and give every row
the same bits whatever M is, wherever the row sits and however the rows are
sliced ("Ferro" README, "Exactness contract").
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


def _case(q8, N, K, M, tag):
    w = q8_synth.weights(N, K, q8_synth.derive_seed("pf-w", tag, N, K), DEV)
    x = q8_synth.activations(M, K, q8_synth.derive_seed("pf-x", tag, M, K), DEV)
    Wb = q8.empty_blocks(N, K)
    q8.q8_quantize_act(w, Wb)
    W = q8.empty_packed(N, K)
    q8.q8_repack_weights(Wb, N, K, W)
    A = q8.empty_blocks(M, K)
    q8.q8_quantize_act(x, A)
    return w, x, Wb, W, A


def _prefill(q8, W, N, K, A, M, flags=0):
    y = torch.full((M, N), float("nan"), device=DEV)
    ws = q8.new_prefill_workspace(K, M)
    q8.q8_gemm_prefill(W, N, K, A, M, y, ws, flags=flags)
    return y


# (N, K, M): weight tiles of 128, 64, 32 and 16 rows; ragged N (a last tile
# of 8 rows), ragged K (a last chunk of 5 blocks, K not a multiple of 256),
# ragged M, one segment (K < 512), segments cut inside a chunk
CASES = [
    (256, 2048, 130),
    (16384, 2048, 64),
    (3072, 2048, 200),
    (2048, 8192, 128),
    (8192, 1024, 16),
    (1000, 416, 5),
    (300, 96, 1),
    (600, 1568, 257),
    (4096, 2048, 300),
    (256, 65536, 130),  # K = Q8_MAX_PREFILL_K: 128 segments
    (1001, 416, 33),    # last weight tile of 9 rows: chunk copies with a ragged tail copied by hand
]


@pytest.mark.parametrize("N,K,M", CASES)
def test_prefill_bitwise_equals_oracle_order(q8, N, K, M):
    _, _, Wb, W, A = _case(q8, N, K, M, "eq")
    y = _prefill(q8, W, N, K, A, M)
    torch.cuda.synchronize()
    Wn, An = Wb.cpu().numpy(), A.cpu().numpy()
    ref = oracle.gemm_prefill_order(Wn, An, K)
    got = y.cpu().numpy()
    assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))
    # and within the library tolerance of the fp64 product
    y64, S = oracle.gemm(Wn, An, K)
    assert (np.abs(got.astype(np.float64) - y64) <= 1e-5 * S + 1e-6).all()
    assert q8.q8_device_error() == 0


def test_prefill_subnormal_and_zero_scales(q8):
    # activation rows scaled down so their block scales (amax / 127) are
    # binary16 subnormals, zero rows (d = 0), and weight rows likewise: the
    # scale products must stay exact
    N, K, M = 256, 1024, 130
    w = q8_synth.weights(N, K, q8_synth.derive_seed("pf-sub-w"), DEV)
    x = q8_synth.activations(M, K, q8_synth.derive_seed("pf-sub-x"), DEV)
    x[0:40] *= 1e-4
    x[40:50] *= 1e-7
    x[50] = 0.0
    w[0:30] *= 1e-3
    w[31] = 0.0
    Wb = q8.empty_blocks(N, K)
    q8.q8_quantize_act(w, Wb)
    W = q8.empty_packed(N, K)
    q8.q8_repack_weights(Wb, N, K, W)
    A = q8.empty_blocks(M, K)
    q8.q8_quantize_act(x, A)
    y = _prefill(q8, W, N, K, A, M)
    torch.cuda.synchronize()
    An = A.cpu().numpy()
    d16 = An.reshape(M, K // 32, 34)[:, :, :2].copy().view(np.uint16)
    assert ((d16 & 0x7C00) == 0).sum() > 1000  # many subnormal (or zero) scales
    ref = oracle.gemm_prefill_order(Wb.cpu().numpy(), An, K)
    assert np.array_equal(y.cpu().numpy().view(np.uint32), ref.view(np.uint32))
    assert q8.q8_device_error() == 0


# N = 2048: every launch below splits its tiles along K over two CTAs;
# N = 4096: the full prompt (96 tiles) does not, its slices do -- the bits
# are the same either way
@pytest.mark.parametrize("N", [2048, 4096])
def test_prefill_rows_do_not_depend_on_the_launch(q8, N):
    K, M = 2048, 300
    _, _, _, W, A = _case(q8, N, K, M, "inv")
    y = _prefill(q8, W, N, K, A, M)
    # slices of the prompt (cut inside a 128-row tile), single rows, and a
    # shuffled row order all give the same bits per row
    for lo, hi in ((0, 100), (100, 129), (129, 300), (77, 78), (299, 300)):
        ys = _prefill(q8, W, N, K, A[lo:hi].contiguous(), hi - lo)
        assert torch.equal(ys.view(torch.int32), y[lo:hi].view(torch.int32)), (lo, hi)
    perm = torch.from_numpy(np.random.default_rng(3).permutation(M)).to(DEV)
    yp = _prefill(q8, W, N, K, A[perm].contiguous(), M)
    assert torch.equal(yp.view(torch.int32), y[perm].view(torch.int32))
    assert q8.q8_device_error() == 0


def test_fused_prefill_equals_quantize_then_prefill(q8):
    N, K, M = 3072, 2048, 140
    _, x, _, W, A = _case(q8, N, K, M, "fused")
    y = _prefill(q8, W, N, K, A, M)
    yf = torch.full_like(y, float("nan"))
    ws = q8.new_prefill_workspace(K, M)
    q8.q8_fused_quant_gemm_prefill(W, N, K, x, M, yf, ws, flags=q8.FLAG_PDL)
    A_out = torch.zeros_like(A)
    yf2 = torch.full_like(y, float("nan"))
    # with A_blocks_out the blocks of x need no room in the workspace
    pk = (M * (K // 32) * 34 + 15) // 16 * 16
    q8.q8_fused_quant_gemm_prefill(W, N, K, x, M, yf2, ws[: ws.numel() - pk], A_blocks_out=A_out)
    torch.cuda.synchronize()
    assert torch.equal(yf.view(torch.int32), y.view(torch.int32))
    assert torch.equal(yf2.view(torch.int32), y.view(torch.int32))
    assert torch.equal(A_out, A)
    assert q8.q8_device_error() == 0


def test_prefill_graph_with_pdl(q8):
    # pack + GEMM captured in a CUDA graph with programmatic dependent launch
    N, K, M = 2048, 2048, 128
    _, _, Wb, W, A = _case(q8, N, K, M, "graph")
    y = torch.empty((M, N), device=DEV)
    ws = q8.new_prefill_workspace(K, M)
    q8.q8_gemm_prefill(W, N, K, A, M, y, ws, flags=q8.FLAG_PDL)
    torch.cuda.synchronize()
    ref = y.clone()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        q8.q8_gemm_prefill(W, N, K, A, M, y, ws, flags=q8.FLAG_PDL)
    y.fill_(float("nan"))
    g.replay()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(y.view(torch.int32), ref.view(torch.int32))
    assert q8.q8_device_error() == 0


def test_prefill_full_size_sampled(q8):
    # the LM head shape (128256 x 2048) at 512 rows: sampled outputs against
    # the oracle's order, which it computes one by one
    N, K, M = 128256, 2048, 512
    _, _, Wb, W, A = _case(q8, N, K, M, "head")
    y = _prefill(q8, W, N, K, A, M)
    torch.cuda.synchronize()
    rng = np.random.default_rng(5)
    rows = np.unique(np.concatenate([rng.integers(0, N, 40), [0, 127, 128, N - 1]]))
    ms = np.unique(np.concatenate([rng.integers(0, M, 6), [0, 127, 128, M - 1]]))
    Wn = Wb[torch.from_numpy(rows).to(DEV)].cpu().numpy()
    An = A[torch.from_numpy(ms).to(DEV)].cpu().numpy()
    ref = oracle.gemm_prefill_order(Wn, An, K)
    got = y[torch.from_numpy(ms).to(DEV)][:, torch.from_numpy(rows).to(DEV)].cpu().numpy()
    assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))
    assert not np.isnan(y.cpu().numpy()).any()
    assert q8.q8_device_error() == 0


def test_prefill_argument_errors(q8):
    N, K, M = 256, 2048, 4
    _, _, _, W, A = _case(q8, N, K, M, "err")
    y = torch.empty((M, N), device=DEV)
    ws = q8.new_prefill_workspace(K, M)
    lib = q8.lib()
    s = torch.cuda.current_stream().cuda_stream
    # workspace one byte short of the split flags (4096 bytes) and the packed activations
    need = 4096 + (ws.numel() - 4096) // 2
    assert lib.q8_gemm_prefill(W.data_ptr(), N, K, A.data_ptr(), M, y.data_ptr(), ws.data_ptr(), need - 1, 0,
                               s) == -6
    assert lib.q8_gemm_prefill(W.data_ptr(), N, K, A.data_ptr(), M, y.data_ptr(), ws.data_ptr(), need, 0, s) == 0
    # the fused call without A_blocks_out needs the whole workspace
    x = torch.zeros((M, K), device=DEV)
    assert lib.q8_fused_quant_gemm_prefill(W.data_ptr(), N, K, x.data_ptr(), M, y.data_ptr(), None,
                                           ws.data_ptr(), need, 0, s) == -6
    torch.cuda.synchronize()
    assert q8.q8_device_error() == 0
