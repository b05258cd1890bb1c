"""Parity of the CUDA path with the oracle, through the C ABI.

Bit-exact: activation quantization (every call site), weight quantization,
repack/unpack, per-block int32 dots, and the GEMV output when every scale is
exactly 1 (then y is an exact integer sum).  Within tolerance:
|y_gpu - y| <= 1e-5 * sum|terms| + 1e-6 with the oracle in fp64.  Bitwise:
batch invariance (a row alone == the same row among others, in any position,
at any M), fused == quantize + GEMV, PDL launch == plain launch, and the same
row of W gives the same bits whatever the matrix's N (different K-splits).
"""
import numpy as np
import pytest
import torch

import oracle
import q8_synth

pytestmark = pytest.mark.gpu

TOL_REL, TOL_ABS = 1e-5, 1e-6


@pytest.fixture(scope="module")
def q8():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    import q8_block_quantized_gb300 as q8mod
    return q8mod


DEV = "cuda"


def _case(N, K, M, seed):
    w = q8_synth.weights(N, K, q8_synth.derive_seed("w", N, K, seed))
    x = q8_synth.activations(M, K, q8_synth.derive_seed("x", M, K, seed))
    return w, x


def _gpu_pack(q8, w):
    return q8.pack_weights_f32(w.to(DEV))


def _run_gemm(q8, W, N, K, A, M, flags=0):
    y = torch.full((M, N), float("nan"), dtype=torch.float32, device=DEV)
    ws = q8.new_workspace(N, K, M)
    q8.q8_gemm(W, N, K, A, M, y, workspace=ws, flags=flags)
    return y


def _run_fused(q8, W, N, K, x, M, flags=0, want_A=False):
    y = torch.full((M, N), float("nan"), dtype=torch.float32, device=DEV)
    A = q8.empty_blocks(M, K) if want_A else None
    ws = q8.new_workspace(N, K, M)
    q8.q8_fused_quant_gemm(W, N, K, x, M, y, A_blocks_out=A, workspace=ws, flags=flags)
    return y, A


def _assert_within_tol(y_gpu, y_ref, S_ref):
    yg = y_gpu.double().cpu().numpy()
    err = np.abs(yg - y_ref)
    tol = TOL_REL * S_ref + TOL_ABS
    bad = err > tol
    assert not bad.any(), "max err %g at %s (tol %g)" % (err.max(), np.argwhere(bad)[:3], tol.max())


# ---------------------------------------------------------------------------
# quantization
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("M,K", [(1, 32), (3, 96), (64, 2048), (17, 8192), (1000, 160)])
def test_quantize_act_bit_exact(q8, M, K):
    x = q8_synth.activations(M, K, 1000 + M + K)
    ref = oracle.quantize(x.numpy())
    out = q8.empty_blocks(M, K)
    q8.q8_quantize_act(x.to(DEV), out)
    assert np.array_equal(out.cpu().numpy(), ref)


def test_quantize_special_blocks_bit_exact(q8):
    rows = []
    z = np.zeros(32, np.float32)
    rows.append(z)                                   # all zero
    t = z.copy(); t[:8] = [127.0, 2.5, -2.5, 0.49999997, 0.5, -0.5, 126.5, -126.5]
    rows.append(t)                                   # d = 1, ties
    rows.append(np.full(32, -3.0, np.float32))       # constant
    oh = z.copy(); oh[17] = 1e-3; rows.append(oh)    # one-hot, small
    rows.append(np.full(32, 6.0e-8, np.float32))     # d16 subnormal
    rows.append(np.full(32, 65504.0 * 100, np.float32))  # large d
    tiny = q8_synth.normal_np(32, 1e-20, 5); rows.append(tiny)
    x = np.concatenate(rows).reshape(1, -1).astype(np.float32)
    K = x.shape[1]
    ref = oracle.quantize(x)
    out = q8.empty_blocks(1, K)
    q8.q8_quantize_act(torch.from_numpy(x).to(DEV), out)
    assert np.array_equal(out.cpu().numpy(), ref)


def test_weight_quantize_repack_round_trip(q8):
    for N, K in [(1, 32), (130, 96), (300, 2048), (257, 40 * 32), (128, 256)]:
        w = q8_synth.weights(N, K, N * 7 + K)
        ref = oracle.quantize(w.numpy())
        W = _gpu_pack(q8, w)
        assert W.numel() == q8.q8_packed_bytes(N, K) == ref.nbytes
        back = q8.empty_blocks(N, K)
        q8.q8_unpack_weights(W, N, K, back)
        assert np.array_equal(back.cpu().numpy(), ref)
        # the packed layout only moves bytes
        assert np.array_equal(np.sort(W.cpu().numpy()), np.sort(ref.ravel()))


@pytest.mark.parametrize("N,K", [(131, 11 * 32), (3000, 5 * 32), (9000, 17 * 32), (20000, 96),
                                 (40000, 64), (80000, 32), (160000, 32)])
def test_packed_layout_matches_header_description(q8, N, K):
    # the byte positions stated in q8.h, for ragged tiles and chunks and
    # every tile height
    R = q8.q8_packed_tile_rows(N)
    exp_R = next((c for c in (16, 32, 64) if -(-N // c) <= 152), 128)
    assert R == exp_R
    nb = K // 32
    rng = np.random.default_rng(4)
    blocks = rng.integers(0, 256, size=(N, nb * 34), dtype=np.uint8)
    src = torch.from_numpy(blocks).to(DEV)
    W = q8.empty_packed(N, K)
    q8.q8_repack_weights(src, N, K, W)
    P = W.cpu().numpy()
    for n in sorted(set([0, 5, R - 1, R, N - 1, N - 2, N // 2])):
        for b in sorted(set([0, nb - 1, nb // 2, min(9, nb - 1)])):
            t, i = divmod(n, R)
            r = min(R, N - R * t)
            c, j = divmod(b, 8)
            kb = min(8, nb - 8 * c)
            base = R * t * nb * 34 + r * 8 * c * 34
            blk = blocks[n, b * 34:(b + 1) * 34]
            for h in range(2):
                off = base + ((2 * j + h) * r + i) * 16
                assert np.array_equal(P[off:off + 16], blk[2 + 16 * h:2 + 16 * h + 16])
            so = base + kb * r * 32 + (j * r + i) * 2
            assert np.array_equal(P[so:so + 2], blk[0:2])


# ---------------------------------------------------------------------------
# dots and the product
# ---------------------------------------------------------------------------

def test_block_dots_bit_exact(q8):
    for N, K, M in [(37, 96, 3), (300, 512, 16), (129, 8192, 2)]:
        w, x = _case(N, K, M, 1)
        Wb = oracle.quantize(w.numpy())
        Ab = oracle.quantize(x.numpy())
        ref = oracle.block_dots(Wb, Ab, K)
        W = _gpu_pack(q8, w)
        A = torch.from_numpy(Ab).to(DEV)
        isum = torch.empty((M, N, K // 32), dtype=torch.int32, device=DEV)
        q8.q8_block_dots(W, N, K, A, M, isum)
        assert np.array_equal(isum.cpu().numpy(), ref)


GEMM_SHAPES = [
    (1, 32, 1), (37, 96, 3), (128, 256, 1), (129, 160, 2), (300, 2048, 1), (300, 2048, 5),
    (1000, 2048, 8), (513, 8192, 1), (256, 3072, 16), (2048, 2048, 1), (700, 1024, 17),
    (260, 512, 33), (130, 2048, 64), (3, 32 * 37, 4),
]


@pytest.mark.parametrize("N,K,M", GEMM_SHAPES)
def test_gemm_within_tolerance(q8, N, K, M):
    w, x = _case(N, K, M, 2)
    Wb = oracle.quantize(w.numpy())
    Ab = oracle.quantize(x.numpy())
    y_ref, S_ref = oracle.gemm(Wb, Ab, K)
    W = _gpu_pack(q8, w)
    A = torch.from_numpy(Ab).to(DEV)
    y = _run_gemm(q8, W, N, K, A, M)
    _assert_within_tol(y, y_ref, S_ref)
    # fused path: same bits, and its A_blocks_out is the oracle's quantization
    yf, Af = _run_fused(q8, W, N, K, x.to(DEV), M, want_A=True)
    assert torch.equal(y, yf)
    assert np.array_equal(Af.cpu().numpy(), Ab)


def _unit_blocks(rng, rows, K):
    """Integer values in [-127, 127] with a 127 in every block: every scale is
    exactly 1 and the quants are the values themselves."""
    v = rng.integers(-127, 128, size=(rows, K)).astype(np.float32)
    v[:, ::32] = 127.0
    return v


# Each decode path computes its own block dots: the DP4A path (1-4 rows),
# the fp16 mma.sync tile kernel (5-8 rows), the virtual-tile kernel (9-64
# rows, in passes of up to 32) and, with Q8_FLAG_TCGEN05, tcgen05 MMAs (16-row
# passes on 128-row tiles).  With unit scales and activation row m zero
# except block b(m), y[m][n] is that row's exact int32 dot for block b(m):
# every path's dot is compared bit for bit with the oracle's, at every block
# position of a chunk and on every tile height.
@pytest.mark.parametrize("M", [1, 2, 4, 8, 12, 16, 32, 64])
@pytest.mark.parametrize("N", [40, 300, 2048, 16384])
def test_decode_block_dots_exact_on_every_path(q8, M, N):
    K = 512  # two chunks of 8 blocks
    NB = K // 32
    rng = np.random.default_rng(N * 100 + M)
    w = _unit_blocks(rng, N, K)
    x = _unit_blocks(rng, M, K)
    sel = np.arange(M) % NB
    for m in range(M):
        keep = np.zeros(K, dtype=bool)
        keep[sel[m] * 32:(sel[m] + 1) * 32] = True
        x[m, ~keep] = 0.0  # zero blocks: scale 0, quants 0, terms exactly 0
    Wb, Ab = oracle.quantize(w), oracle.quantize(x)
    isum = oracle.block_dots(Wb, Ab, K)  # [M][N][NB]
    expect = isum[np.arange(M), :, sel].astype(np.float32)  # [M][N]
    W = _gpu_pack(q8, torch.from_numpy(w))
    A = torch.from_numpy(Ab).to(DEV)
    y = _run_gemm(q8, W, N, K, A, M)
    assert np.array_equal(y.cpu().numpy(), expect)
    yf, _ = _run_fused(q8, W, N, K, torch.from_numpy(x).to(DEV), M)
    assert np.array_equal(yf.cpu().numpy(), expect)
    if M >= 9 and N % 128 == 0 and q8.q8_packed_tile_rows(N) == 128:
        yt = _run_gemm(q8, W, N, K, A, M, flags=q8.FLAG_TCGEN05)
        assert np.array_equal(yt.cpu().numpy(), expect)


@pytest.mark.parametrize("M", [4, 8, 16, 64])
def test_gemm_exact_integer_sum_with_unit_scales(q8, M):
    # every block has amax = 127, so every scale is exactly 1 and
    # y = sum_b isum_b exactly (partial sums stay below 2^24 here)
    N, K = 260, 2048
    rng = np.random.default_rng(8 + M)
    w, x = _unit_blocks(rng, N, K), _unit_blocks(rng, M, K)
    Wb, Ab = oracle.quantize(w), oracle.quantize(x)
    isum = oracle.block_dots(Wb, Ab, K).astype(np.int64).sum(axis=2)
    assert np.abs(isum).max() < 2**24
    W = _gpu_pack(q8, torch.from_numpy(w))
    y = _run_gemm(q8, W, N, K, torch.from_numpy(Ab).to(DEV), M)
    assert np.array_equal(y.cpu().numpy().astype(np.int64), isum)
    yf, _ = _run_fused(q8, W, N, K, torch.from_numpy(x).to(DEV), M)
    assert np.array_equal(yf.cpu().numpy().astype(np.int64), isum)


@pytest.mark.parametrize("M", [1, 3, 8, 16, 40])
def test_gemm_zero_and_subnormal_scale_blocks(q8, M):
    # blocks whose binary16 scale is 0 or subnormal (amax below 127 * 2^-14),
    # in W and in the activations, among ordinary ones: products of two
    # subnormal binary16 scales are still exact normal fp32 values
    N, K = 300, 1024
    rng = np.random.default_rng(20 + M)
    w = (rng.standard_normal((N, K)) * q8_synth.WEIGHT_STD).astype(np.float32)
    x = rng.standard_normal((M, K)).astype(np.float32)
    nb = K // 32
    for arr, rows in ((w, N), (x, M)):
        kind = rng.integers(0, 4, size=(rows, nb))  # 0 zero, 1 subnormal, 2 tiny subnormal, 3 ordinary
        for r in range(rows):
            for b in range(nb):
                blk = arr[r, b * 32:(b + 1) * 32]
                if kind[r, b] == 0:
                    blk[:] = 0.0
                elif kind[r, b] == 1:
                    blk *= np.float32(1e-4) / np.abs(blk).max()
                elif kind[r, b] == 2:
                    blk *= np.float32(3e-7) / np.abs(blk).max()
    Wb, Ab = oracle.quantize(w), oracle.quantize(x)
    d16, _ = oracle.split_blocks(Wb, K)
    assert ((d16 & 0x7C00) == 0).any() and ((d16 != 0) & ((d16 & 0x7C00) == 0)).any()
    y_ref, S_ref = oracle.gemm(Wb, Ab, K)
    W = _gpu_pack(q8, torch.from_numpy(w))
    y = _run_gemm(q8, W, N, K, torch.from_numpy(Ab).to(DEV), M)
    _assert_within_tol(y, y_ref, S_ref)
    yf, Af = _run_fused(q8, W, N, K, torch.from_numpy(x).to(DEV), M, want_A=True)
    assert np.array_equal(Af.cpu().numpy(), Ab)
    assert torch.equal(yf, y)
    # the row decoded alone has the same bits
    y1 = _run_gemm(q8, W, N, K, torch.from_numpy(Ab[-1:].copy()).to(DEV), 1)
    assert torch.equal(y1[0], y[-1])


# ---------------------------------------------------------------------------
# batch invariance and order invariance (bitwise)
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("N,K", [(2048, 2048), (3072, 2048), (2048, 8192), (700, 3072),
                                 (5120, 3072), (16384, 3072), (3072, 8192)])  # the 3B shapes too
def test_batch_invariance_shuffled_rows(q8, N, K):
    Mmax = 64
    w, x = _case(N, K, Mmax, 3)
    W = _gpu_pack(q8, w)
    xd = x.to(DEV)
    A_all = q8.empty_blocks(Mmax, K)
    q8.q8_quantize_act(xd, A_all)
    solo = torch.empty((Mmax, N), dtype=torch.float32, device=DEV)
    for m in range(Mmax):
        solo[m:m + 1] = _run_gemm(q8, W, N, K, A_all[m:m + 1].contiguous(), 1)
    gen = torch.Generator().manual_seed(N + K)
    for M in (1, 2, 3, 4, 8, 16, 32, 64):
        perm = torch.randperm(Mmax, generator=gen)[:M]
        A = A_all[perm.to(DEV)].contiguous()
        y = _run_gemm(q8, W, N, K, A, M)
        assert torch.equal(y, solo[perm.to(DEV)]), "M=%d" % M
        yf, _ = _run_fused(q8, W, N, K, xd[perm.to(DEV)].contiguous(), M)
        assert torch.equal(yf, solo[perm.to(DEV)]), "fused M=%d" % M


def test_row_result_independent_of_matrix_height(q8):
    # the first rows of W give the same bits whether W has 130 rows (no split
    # along K) or 128256 rows: the plans differ, the reduction order does not
    K, M = 2048, 3
    w, x = _case(4096, K, M, 4)
    A = q8.empty_blocks(M, K)
    q8.q8_quantize_act(x.to(DEV), A)
    ys = []
    for N in (130, 1000, 4096):
        W = _gpu_pack(q8, w[:N].contiguous())
        ys.append(_run_gemm(q8, W, N, K, A, M)[:, :130])
    assert torch.equal(ys[0], ys[1]) and torch.equal(ys[0], ys[2])


def test_pdl_flag_same_bits(q8):
    N, K, M = 1000, 2048, 4
    w, x = _case(N, K, M, 5)
    W = _gpu_pack(q8, w)
    xd = x.to(DEV)
    A = q8.empty_blocks(M, K)
    q8.q8_quantize_act(xd, A, flags=q8.FLAG_PDL)
    y0 = _run_gemm(q8, W, N, K, A, M)
    y1 = _run_gemm(q8, W, N, K, A, M, flags=q8.FLAG_PDL)
    yf, _ = _run_fused(q8, W, N, K, xd, M, flags=q8.FLAG_PDL)
    torch.cuda.synchronize()
    assert torch.equal(y0, y1) and torch.equal(y0, yf)


def test_workspace_left_zero_and_reusable(q8):
    N, K, M = 256, 8192, 16
    w, x = _case(N, K, M, 6)
    W = _gpu_pack(q8, w)
    A = q8.empty_blocks(M, K)
    q8.q8_quantize_act(x.to(DEV), A)
    ws = q8.new_workspace(N, K, M)
    assert ws is not None  # this shape is split along K
    y = torch.empty((M, N), dtype=torch.float32, device=DEV)
    outs = []
    for _ in range(3):  # noqa: B007
        q8.q8_gemm(W, N, K, A, M, y, workspace=ws)
        outs.append(y.clone())
    torch.cuda.synchronize()
    assert torch.equal(outs[0], outs[1]) and torch.equal(outs[0], outs[2])
    assert int(ws[:16384].view(torch.int32).abs().sum()) == 0


def test_workspace_shared_across_shapes(q8):
    # one workspace serves calls of different shapes in sequence (tickets
    # live in a fixed prefix that partials never touch)
    K, M = 2048, 16
    shapes = [(256, 8192), (512, 2048), (2048, 2048), (300, 4096), (256, 8192)]
    need = max(q8.q8_workspace_bytes(N, K_, M) for N, K_ in shapes)
    ws = torch.zeros(need, dtype=torch.uint8, device=DEV)
    for N, K_ in shapes:
        w, x = _case(N, K_, M, 9)
        W = _gpu_pack(q8, w)
        A = q8.empty_blocks(M, K_)
        q8.q8_quantize_act(x.to(DEV), A)
        y = torch.empty((M, N), dtype=torch.float32, device=DEV)
        q8.q8_gemm(W, N, K_, A, M, y, workspace=ws)
        own = _run_gemm(q8, W, N, K_, A, M)
        assert torch.equal(y, own), (N, K_)


def test_host_errors_raise(q8):
    N, K, M = 256, 8192, 1
    W = q8.empty_packed(N, K)
    A = q8.empty_blocks(M, K)
    y = torch.empty((M, N), dtype=torch.float32, device=DEV)
    with pytest.raises(q8.Q8Error) as e:
        q8.q8_gemm(W, N, K, A, M, y, workspace=None)   # needs a workspace
    assert e.value.status == -6
    with pytest.raises(q8.Q8Error) as e:
        q8.q8_gemm(W, N, K + 1, A, M, y)
    assert e.value.status == -2
    with pytest.raises(q8.Q8Error):
        q8.q8_gemm(W[1:], N, K, A, M, y)                 # misaligned W
    assert q8.q8_device_error() == 0


@pytest.mark.parametrize("N,K", [(10000, 2080), (16384, 3072), (12800, 8192)])
@pytest.mark.parametrize("M", [9, 16, 33, 64])
def test_tcgen05_flag_gives_the_same_bits(q8, N, K, M):
    # Q8_FLAG_TCGEN05: 128-row tiles with 9-16 rows per pass take the tcgen05
    # kernel (ragged last tile, ragged last chunk, split K, several passes)
    assert q8.q8_packed_tile_rows(N) == 128
    w, x = _case(N, K, M, 21)
    W = _gpu_pack(q8, w)
    Ab = oracle.quantize(x.numpy())
    A = torch.from_numpy(Ab).to(DEV)
    xd = x.to(DEV)
    ws = q8.new_workspace(N, K, M)
    outs = {}
    for flags in (0, q8.FLAG_TCGEN05, q8.FLAG_TCGEN05 | q8.FLAG_PDL):
        y = torch.full((M, N), float("nan"), dtype=torch.float32, device=DEV)
        q8.q8_gemm(W, N, K, A, M, y, workspace=ws, flags=flags)
        yf = torch.full((M, N), float("nan"), dtype=torch.float32, device=DEV)
        q8.q8_fused_quant_gemm(W, N, K, xd, M, yf, workspace=ws, flags=flags)
        outs[flags] = (y, yf)
    torch.cuda.synchronize()
    base = outs[0][0]
    for y, yf in outs.values():
        assert torch.equal(y, base) and torch.equal(yf, base)
    if N * K <= 30_000_000:
        y_ref, S_ref = oracle.gemm(oracle.quantize(w.numpy()), Ab, K)
        _assert_within_tol(outs[q8.FLAG_TCGEN05][0], y_ref, S_ref)
    if ws is not None:  # split along K: the tickets are left zero
        assert not ws[:16384].any()
    assert q8.q8_device_error() == 0


@pytest.mark.parametrize("N,K,M", [(300, 512, 65), (2048, 2048, 200), (1000, 3072, 1000)])
def test_prefill_rows_equal_decode_rows(q8, N, K, M):
    # more than 16 rows run as 16-row passes through the same kernels: every
    # row of a prefill batch is bitwise the row computed alone (M = 1)
    w, x = _case(N, K, M, 31)
    W = _gpu_pack(q8, w)
    Ab = oracle.quantize(x.numpy())
    A = torch.from_numpy(Ab).to(DEV)
    y = torch.full((M, N), float("nan"), dtype=torch.float32, device=DEV)
    q8.q8_gemm(W, N, K, A, M, y, workspace=q8.new_workspace(N, K, M))
    yf = torch.full((M, N), float("nan"), dtype=torch.float32, device=DEV)
    q8.q8_fused_quant_gemm(W, N, K, x.to(DEV), M, yf, workspace=q8.new_workspace(N, K, M))
    torch.cuda.synchronize()
    assert torch.equal(y, yf)
    ws1 = q8.new_workspace(N, K, 1)
    for m in (0, 17, M // 2, M - 1):
        y1 = torch.empty((1, N), dtype=torch.float32, device=DEV)
        q8.q8_gemm(W, N, K, A[m:m + 1].contiguous(), 1, y1, workspace=ws1)
        torch.cuda.synchronize()
        assert torch.equal(y1[0], y[m]), m
    if M * N * K <= 700_000_000:
        y_ref, S_ref = oracle.gemm(oracle.quantize(w.numpy()), Ab, K)
        _assert_within_tol(y, y_ref, S_ref)
    assert q8.q8_device_error() == 0


@pytest.mark.parametrize("N,K,M", [(20_000_000, 32, 1), (20_000_000, 32, 3), (16, 1 << 20, 1), (40, 1 << 20, 5)])
def test_extreme_shapes_sampled_against_oracle(q8, N, K, M):
    # a very tall matrix (row and tile offsets past 2^31 bytes) and a very
    # wide one (deep splits along K): sampled rows against the oracle, and
    # the fused path bitwise equal to quantize + GEMV
    gen = torch.Generator(device=DEV)
    gen.manual_seed(N + K + M)
    w = torch.randn((N, K), generator=gen, device=DEV) * q8_synth.WEIGHT_STD
    x = torch.randn((M, K), generator=gen, device=DEV)
    W = q8.pack_weights_f32(w)
    A = q8.empty_blocks(M, K)
    q8.q8_quantize_act(x, A)
    ws = q8.new_workspace(N, K, M)
    y = torch.empty((M, N), dtype=torch.float32, device=DEV)
    q8.q8_gemm(W, N, K, A, M, y, workspace=ws)
    yf = torch.empty((M, N), dtype=torch.float32, device=DEV)
    q8.q8_fused_quant_gemm(W, N, K, x, M, yf, workspace=ws)
    torch.cuda.synchronize()
    assert torch.equal(y, yf)
    rows = np.unique(np.concatenate([[0, 1, N // 2, N - 1], np.random.default_rng(N).integers(0, N, 60)]))
    Wb = oracle.quantize(w[torch.from_numpy(rows).to(DEV)].cpu().numpy())
    Ab = A.cpu().numpy()
    assert np.array_equal(Ab, oracle.quantize(x.cpu().numpy()))
    y_ref, S_ref = oracle.gemm(Wb, Ab, K)
    err = np.abs(y[:, torch.from_numpy(rows).to(DEV)].double().cpu().numpy() - y_ref)
    assert (err <= TOL_REL * S_ref + TOL_ABS).all(), err.max()
    if ws is not None:
        assert not ws[:16384].any()
    del w, W
    torch.cuda.empty_cache()
    assert q8.q8_device_error() == 0


# A single virtual tile (N <= 128) split along K into S = K / 256 units: the
# S CTAs of the tile form one thread-block cluster (S <= 8) and combine
# their values through distributed shared memory; S = 12 takes the
# workspace and tickets.  Every row equals the row decoded alone (the
# one-row kernel, its own split and merge) bit for bit, and the oracle's
# product within tolerance; fused and unfused calls, and one launch of 32
# rows plus one of 8 (M = 40).
@pytest.mark.parametrize("S", [2, 3, 5, 7, 8, 12])
@pytest.mark.parametrize("M", [9, 16, 40])
def test_k_split_combine_every_split_count(q8, S, M):
    N, K = 100, 256 * S
    w, x = _case(N, K, M, 31 + S)
    W = _gpu_pack(q8, w)
    Wb = oracle.quantize(w.numpy())
    Ab = oracle.quantize(x.numpy())
    A = torch.from_numpy(Ab).to(DEV)
    y = _run_gemm(q8, W, N, K, A, M)
    yf, _ = _run_fused(q8, W, N, K, x.to(DEV), M)
    torch.cuda.synchronize()
    assert torch.equal(y, yf)
    y_ref, S_ref = oracle.gemm(Wb, Ab, K)
    _assert_within_tol(y, y_ref, S_ref)
    for m in (0, M // 2, M - 1):
        solo = _run_gemm(q8, W, N, K, A[m:m + 1].contiguous(), 1)
        assert torch.equal(y[m:m + 1], solo), m
    assert q8.q8_device_error() == 0
