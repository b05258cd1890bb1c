"""A decode step over a synthetic Q8_0 projection stack, made of libq8 calls.

The step is the per-token work of the projections of a Llama-3.2-style
decoder ("Ember: packed Q8 decode" measures this model family): for every
layer, one activation quantization shared by Q/K/V (one concatenated N =
q + 2*kv GEMV), the O projection, one quantization shared by gate/up (one
N = 2*ffn GEMV), the down projection; then the LM head.  Single-consumer
inputs (O, down, head) go through the fused quantize+GEMV call.

Inputs are independent seeded N(0, 1) rows per projection input (no norms,
attention or residuals between projections), weights seeded N(0, 0.02).
Everything here is allocation and call sequencing; all arithmetic is in
libq8's kernels.  The step can be captured once into a CUDA graph and
replayed; consecutive calls are chained with programmatic dependent launch.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import torch

import q8_synth
from . import (FLAG_PDL, FLAG_TCGEN05, empty_blocks, pack_weights_f32, q8_fused_quant_gemm,
               q8_fused_quant_gemm_prefill, q8_gemm, q8_prefill_workspace_bytes, q8_quantize_act,
               q8_workspace_bytes)

# "prefill": every projection through the prefill tile GEMM (quantize, pack,
# tile GEMM per call) instead of the decode GEMV
MODES = ("shared", "fused", "unfused", "prefill")


@dataclass
class Call:
    kind: str            # "quant", "gemm", "fused", "prefill"
    proj: str
    layer: int
    N: int = 0
    K: int = 0
    W: torch.Tensor | None = None
    x: torch.Tensor | None = None        # fp32 input view
    A: torch.Tensor | None = None        # activation blocks
    y: torch.Tensor | None = None        # output view


@dataclass
class Q8Stack:
    shape: q8_synth.StackShape
    M: int
    mode: str = "fused"
    layers: int | None = None
    seed: int = 0
    pdl: bool = True
    tcgen05: bool = False                # Q8_FLAG_TCGEN05 on every GEMV call
    device: str = "cuda"
    shared_weights: dict | None = None   # reuse another stack's packed weights
    include_head: bool = True            # False: the layers' projections only
    calls: list = field(default_factory=list)

    def __post_init__(self):
        if self.mode not in MODES:
            raise ValueError("mode must be one of %s" % (MODES,))
        L = self.shape.layers if self.layers is None else self.layers
        self.n_layers = L
        projs = self.shape.layer_projs()
        head = self.shape.head()
        dev = torch.device(self.device)
        entries = [(li, p) for li in range(L) for p in projs] + ([(L, head)] if self.include_head else [])
        # one flat fp32 input buffer and one flat output buffer per step
        self.x_all = torch.empty(self.M * sum(p.K for _, p in entries), dtype=torch.float32,
                                 device=dev)
        self.y_all = torch.empty(self.M * sum(p.N for _, p in entries), dtype=torch.float32,
                                 device=dev)
        self.weights = {}
        xo = yo = 0
        ws_need = 0
        pf_need = 0
        calls = []
        for li, p in entries:
            if self.shared_weights is not None:
                W = self.shared_weights[(li, p.name)]
            else:
                w32 = self.weights_f32(li, p)
                W = pack_weights_f32(w32)
                del w32
            self.weights[(li, p.name)] = W
            x = self.x_all[xo:xo + self.M * p.K].view(self.M, p.K)
            xo += self.M * p.K
            y = self.y_all[yo:yo + self.M * p.N].view(self.M, p.N)
            yo += self.M * p.N
            shared_input = p.name in ("qkv", "gate_up")
            if self.mode == "prefill":
                pf_need = max(pf_need, q8_prefill_workspace_bytes(p.K, self.M))
                calls.append(Call("prefill", p.name, li, p.N, p.K, W=W, x=x, y=y))
                continue
            ws_need = max(ws_need, q8_workspace_bytes(p.N, p.K, self.M))
            if self.mode == "fused" or (self.mode == "shared" and not shared_input):
                calls.append(Call("fused", p.name, li, p.N, p.K, W=W, x=x, y=y))
            else:
                A = empty_blocks(self.M, p.K, dev)
                calls.append(Call("quant", p.name, li, 0, p.K, x=x, A=A))
                calls.append(Call("gemm", p.name, li, p.N, p.K, W=W, A=A, y=y))
        self.calls = calls
        self.workspace = (torch.zeros(ws_need, dtype=torch.uint8, device=dev)
                          if ws_need else None)
        self.pf_workspace = (torch.empty(pf_need, dtype=torch.uint8, device=dev)
                             if pf_need else None)
        self.refill_inputs(step=0)
        torch.cuda.synchronize()

    def weights_f32(self, layer: int, p: q8_synth.Proj) -> torch.Tensor:
        """The fp32 weights (before quantization) of one projection, regenerated
        from its seed."""
        seed_w = q8_synth.derive_seed(self.shape.name, self.seed, layer, p.name, "w")
        return q8_synth.weights(p.N, p.K, seed_w, torch.device(self.device))

    # -- inputs ------------------------------------------------------------------
    def refill_inputs(self, step: int):
        seed = q8_synth.derive_seed(self.shape.name, self.seed, "x", step)
        self.x_all.copy_(q8_synth.normal_torch((self.x_all.numel(),), 1.0, seed, self.x_all.device))

    # -- the step -------------------------------------------------------------------
    def step(self, stream=None):
        flags = FLAG_PDL if self.pdl else 0
        gflags = flags | (FLAG_TCGEN05 if self.tcgen05 else 0)
        ws = self.workspace
        for c in self.calls:
            if c.kind == "quant":
                q8_quantize_act(c.x, c.A, flags=flags, stream=stream)
            elif c.kind == "prefill":
                q8_fused_quant_gemm_prefill(c.W, c.N, c.K, c.x, self.M, c.y, self.pf_workspace, flags=flags,
                                            stream=stream)
            elif c.kind == "gemm":
                q8_gemm(c.W, c.N, c.K, c.A, self.M, c.y, workspace=ws, flags=gflags, stream=stream)
            else:
                q8_fused_quant_gemm(c.W, c.N, c.K, c.x, self.M, c.y, workspace=ws, flags=gflags,
                                    stream=stream)

    def capture(self) -> torch.cuda.CUDAGraph:
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            self.step()  # warm: plans, function attributes
        torch.cuda.current_stream().wait_stream(s)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            self.step()
        torch.cuda.synchronize()
        return g

    # -- accounting -------------------------------------------------------------------
    def launches_per_step(self) -> int:
        n = 0
        for c in self.calls:
            if c.kind == "quant":
                n += 1
            elif c.kind == "prefill":
                n += 3  # quantize, pack, tile GEMM
            else:
                n += (self.M + 15) // 16
        return n

    def mac_per_step(self) -> int:
        """Multiply-accumulates of one step: M * sum of N * K."""
        return self.M * sum(c.N * c.K for c in self.calls if c.kind != "quant")

    def weight_bytes(self) -> int:
        return sum(W.numel() for W in self.weights.values())

    def bytes_per_step(self) -> int:
        """Algorithmic bytes of one step: packed weights + fp32 inputs + fp32 outputs.
        Quantized activation blocks are intermediates and not counted."""
        return self.weight_bytes() + 4 * self.x_all.numel() + 4 * self.y_all.numel()

    def outputs(self):
        """(layer, proj) -> output view [M][N]."""
        return {(c.layer, c.proj): c.y for c in self.calls if c.y is not None}

    def inputs(self):
        """(layer, proj) -> fp32 input view [M][K] (the shared input for qkv/gate_up)."""
        return {(c.layer, c.proj): c.x for c in self.calls if c.x is not None}
