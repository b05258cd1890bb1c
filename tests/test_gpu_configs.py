"""Parity at the full workload sizes, in the benchmark's launch configuration
(the projection stack captured in a CUDA graph, calls chained with
programmatic dependent launch), on sampled outputs the oracle computes one by
one:

1. one 2048x2048 GEMV, M = 1;
2. one Llama-3.2-1B layer (QKV 3072x2048, O, gate/up 16384x2048, down
   2048x8192), M = 1;
3. the LM head 128256x2048 at M = 1 and 8;
4. the 16-layer 1B stack + head at M = 1, 4, 8, 16, with a shuffled-row
   batch-invariance check;
5. the 28-layer 3B stack + head at M = 1, 16, 32, 64.

For each projection the oracle gets the fp32 weight rows of a random sample
of output rows and the fp32 inputs, quantizes them itself, and must agree
bit for bit on the quantized weights and within the tolerance on y.
"""
import numpy as np
import pytest
import torch

import oracle
import q8_synth

pytestmark = pytest.mark.gpu

SAMPLE_ROWS = 24


@pytest.fixture(scope="module")
def q8():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    import q8_block_quantized_gb300 as q8mod
    return q8mod


def _check_stack(q8, st, rng, sample_layers=None):
    from q8_block_quantized_gb300.stack import Q8Stack  # noqa: F401
    outs = st.outputs()
    ins = st.inputs()
    projs = {p.name: p for p in st.shape.layer_projs()}
    projs["lm_head"] = st.shape.head()
    keys = sorted(outs)
    if sample_layers is not None:
        keys = [k for k in keys if k[0] in sample_layers or k[1] == "lm_head"]
    for (li, name) in keys:
        p = projs[name]
        rows = np.sort(rng.choice(p.N, size=min(SAMPLE_ROWS, p.N), replace=False))
        w32 = st.weights_f32(li, p)
        w_rows = w32[torch.from_numpy(rows).to(w32.device)].cpu().numpy()
        del w32
        Wb = oracle.quantize(w_rows)
        # the GPU's own quantized weights for those rows (unpacked), bit-exact
        back = q8.empty_blocks(p.N, p.K)
        q8.q8_unpack_weights(st.weights[(li, name)], p.N, p.K, back)
        assert np.array_equal(back[torch.from_numpy(rows).to(back.device)].cpu().numpy(), Wb), (li, name)
        x = ins[(li, name)].cpu().numpy()
        y_ref, S_ref = oracle.gemm(Wb, oracle.quantize(x), p.K)
        yg = outs[(li, name)][:, torch.from_numpy(rows).to(back.device)].double().cpu().numpy()
        err = np.abs(yg - y_ref)
        assert (err <= 1e-5 * S_ref + 1e-6).all(), (li, name, err.max())


def _run_graph(st):
    g = st.capture()
    g.replay()
    torch.cuda.synchronize()
    return g


def test_config1_single_gemv(q8):
    N = K = 2048
    w = q8_synth.weights(N, K, 0, "cuda")
    x = q8_synth.activations(1, K, 0, "cuda")
    W = q8.pack_weights_f32(w)
    y = torch.empty((1, N), dtype=torch.float32, device="cuda")
    ws = q8.new_workspace(N, K, 1)
    q8.q8_fused_quant_gemm(W, N, K, x, 1, y, workspace=ws, flags=q8.FLAG_PDL)
    torch.cuda.synchronize()
    Wb = oracle.quantize(w.cpu().numpy())
    y_ref, S_ref = oracle.gemm(Wb, oracle.quantize(x.cpu().numpy()), K)
    assert (np.abs(y.double().cpu().numpy() - y_ref) <= 1e-5 * S_ref + 1e-6).all()


def test_config2_one_1b_layer(q8):
    from q8_block_quantized_gb300.stack import Q8Stack
    for mode in ("shared", "fused", "unfused"):
        st = Q8Stack(q8_synth.LLAMA_1B, M=1, layers=1, mode=mode)
        _run_graph(st)
        _check_stack(q8, st, np.random.default_rng(2))


def test_config3_lm_head(q8):
    from q8_block_quantized_gb300.stack import Q8Stack
    base = Q8Stack(q8_synth.LLAMA_1B, M=1, layers=0)
    _run_graph(base)
    _check_stack(q8, base, np.random.default_rng(3))
    st8 = Q8Stack(q8_synth.LLAMA_1B, M=8, layers=0, shared_weights=base.weights)
    _run_graph(st8)
    _check_stack(q8, st8, np.random.default_rng(4))


def _shuffle_invariance(st):
    """Permute the rows of every input; every output must permute bitwise."""
    ref = {k: v.clone() for k, v in st.outputs().items()}
    perm = torch.randperm(st.M, generator=torch.Generator().manual_seed(st.M)).cuda()
    for x in st.inputs().values():
        x.copy_(x[perm].clone())
    st.step()
    torch.cuda.synchronize()
    for k, v in st.outputs().items():
        assert torch.equal(v, ref[k][perm]), k


def _solo_rows_match(st, base_weights, rows):
    """Row m of an M-row step equals the same input run alone (M = 1)."""
    from q8_block_quantized_gb300.stack import Q8Stack
    solo = Q8Stack(st.shape, M=1, layers=st.n_layers, shared_weights=base_weights)
    ins, outs = st.inputs(), st.outputs()
    for m in rows:
        for k, x in solo.inputs().items():
            x.copy_(ins[k][m:m + 1])
        solo.step()
        torch.cuda.synchronize()
        for k, y in solo.outputs().items():
            assert torch.equal(y, outs[k][m:m + 1]), (m, k)


def test_config4_1b_stack(q8):
    from q8_block_quantized_gb300.stack import Q8Stack
    base = Q8Stack(q8_synth.LLAMA_1B, M=1)
    _run_graph(base)
    _check_stack(q8, base, np.random.default_rng(5), sample_layers={0, 7, 15})
    for M in (4, 8, 16):
        st = Q8Stack(q8_synth.LLAMA_1B, M=M, shared_weights=base.weights)
        _run_graph(st)
        _check_stack(q8, st, np.random.default_rng(6 + M), sample_layers={0, 15})
        if M == 16:
            _solo_rows_match(st, base.weights, rows=[0, 9, 15])
        _shuffle_invariance(st)
        del st
    torch.cuda.empty_cache()


def test_config5_3b_stack(q8):
    from q8_block_quantized_gb300.stack import Q8Stack
    base = Q8Stack(q8_synth.LLAMA_3B, M=1)
    _run_graph(base)
    _check_stack(q8, base, np.random.default_rng(7), sample_layers={0, 27})
    for M in (16, 32, 64):
        st = Q8Stack(q8_synth.LLAMA_3B, M=M, shared_weights=base.weights)
        _run_graph(st)
        _check_stack(q8, st, np.random.default_rng(8 + M), sample_layers={13})
        if M == 64:
            _solo_rows_match(st, base.weights, rows=[0, 63])
        _shuffle_invariance(st)
        del st
    assert q8.q8_device_error() == 0
