"""Python binding of libq8 (the C ABI in include/q8.h).

Argument marshalling only: every step of the computation runs in the CUDA
kernels of ``libq8.so``.  PyTorch supplies device memory and streams.  The
functions carry the C names; tensors are passed by their data pointers after
dtype/device/contiguity checks, and a non-zero status raises ``Q8Error``.

The library must have been built (``q8_block_quantized_gb300.build.build()``
or ``__graft_entry__.build()``); importing the binding without it raises.
There is no fallback of any kind.
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libq8.so")

QK = 32
BLOCK_BYTES = 34
MAX_M = 4096
MAX_DOTS_M = 64
MAX_TILE_ROWS = 128
CHUNK_BLOCKS = 8
FLAG_PDL = 1
FLAG_TCGEN05 = 2
PREFILL_TILE_ROWS = 128
PREFILL_SEGMENT = 16
MAX_PREFILL_K = 65536
MAX_KV_D = 1 << 24
KV_BLOCK_BYTES = 36

STATUS = {0: "Q8_OK", -1: "Q8_EINVAL", -2: "Q8_ESHAPE", -3: "Q8_EALIGN", -4: "Q8_EDEVICE",
          -5: "Q8_ECUDA", -6: "Q8_EWORKSPACE", -7: "Q8_ETIMEOUT", -8: "Q8_ESCRATCH"}
NOALLOC_SCRATCH_BYTES = 4 << 20

# Every function q8.h declares, with its ctypes signature.
_vp, _i64, _int, _u, _sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_uint, ctypes.c_size_t
SIGNATURES = {
    "q8_strerror": (ctypes.c_char_p, [_int]),
    "q8_abi_version": (_int, []),
    "q8_blocks_bytes": (_sz, [_i64, _i64]),
    "q8_packed_bytes": (_sz, [_i64, _i64]),
    "q8_packed_tile_rows": (_int, [_i64]),
    "q8_workspace_bytes": (_sz, [_i64, _i64, _int]),
    "q8_quantize_act": (_int, [_vp, _i64, _i64, _vp, _u, _vp]),
    "q8_residual_rmsnorm_quantize": (_int, [_vp, _vp, _vp, ctypes.c_float, _i64, _i64, _vp, _vp, _u, _vp]),
    "q8_swiglu_quantize": (_int, [_vp, _i64, _i64, _vp, _u, _vp]),
    "q8_repack_weights": (_int, [_vp, _i64, _i64, _vp, _vp]),
    "q8_gemm": (_int, [_vp, _i64, _i64, _vp, _int, _vp, _vp, _sz, _u, _vp]),
    "q8_fused_quant_gemm": (_int, [_vp, _i64, _i64, _vp, _int, _vp, _vp, _vp, _sz, _u, _vp]),
    "q8_gemm_noalloc": (_int, [_vp, _i64, _i64, _vp, _int, _vp, _u, _vp]),
    "q8_gemm_swiglu": (_int, [_vp, _i64, _i64, _vp, _int, _vp, _u, _vp]),
    "q8_fused_quant_gemm_swiglu": (_int, [_vp, _i64, _i64, _vp, _int, _vp, _u, _vp]),
    "q8_prefill_workspace_bytes": (_sz, [_i64, _int]),
    "q8_gemm_prefill": (_int, [_vp, _i64, _i64, _vp, _int, _vp, _vp, _sz, _u, _vp]),
    "q8_fused_quant_gemm_prefill": (_int, [_vp, _i64, _i64, _vp, _int, _vp, _vp, _vp, _sz, _u, _vp]),
    "q8_kv_cache_bytes": (_sz, [_i64, _i64]),
    "q8_kv_quantize": (_int, [_vp, _i64, _i64, _vp, _i64, _vp, _vp, _u, _vp]),
    "q8_kv_dequantize": (_int, [_vp, _vp, _i64, _i64, _vp, _i64, _vp, _u, _vp]),
    "q8_unpack_weights": (_int, [_vp, _i64, _i64, _vp, _vp]),
    "q8_block_dots": (_int, [_vp, _i64, _i64, _vp, _int, _vp, _vp]),
    "q8_device_error": (_int, [ctypes.POINTER(ctypes.c_uint)]),
    "q8_device_info": (_int, [ctypes.POINTER(_int), ctypes.POINTER(_int), ctypes.POINTER(_int)]),
    "q8_set_wait_limit_ns": (_int, [ctypes.c_uint64]),
}

_lib = None


class Q8Error(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        msg = lib().q8_strerror(status).decode()
        super().__init__("%s returned %d (%s)" % (fn, status, msg))


def lib() -> ctypes.CDLL:
    """The loaded libq8.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError("libq8.so is not built (%s); run "
                               "q8_block_quantized_gb300.build.build()" % LIB_PATH)
        handle = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            f = getattr(handle, name)
            f.restype = res
            f.argtypes = args
        _lib = handle
    return _lib


def _check(fn: str, status: int) -> None:
    if status != 0:
        raise Q8Error(fn, status)


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _dev(t: torch.Tensor, dtype, name: str) -> int:
    if not isinstance(t, torch.Tensor):
        raise TypeError("%s must be a torch.Tensor" % name)
    if t.device.type != "cuda" or t.dtype != dtype or not t.is_contiguous():
        raise ValueError("%s must be a contiguous %s CUDA tensor (got %s %s)"
                         % (name, dtype, t.dtype, t.device))
    return t.data_ptr()


def _opt(t, dtype, name):
    return None if t is None else _dev(t, dtype, name)


# ---- sizes ------------------------------------------------------------------

def q8_blocks_bytes(rows: int, K: int) -> int:
    return int(lib().q8_blocks_bytes(rows, K))


def q8_packed_bytes(N: int, K: int) -> int:
    return int(lib().q8_packed_bytes(N, K))


def q8_packed_tile_rows(N: int) -> int:
    return int(lib().q8_packed_tile_rows(N))


def q8_workspace_bytes(N: int, K: int, M: int) -> int:
    return int(lib().q8_workspace_bytes(N, K, M))


# ---- the four calls ----------------------------------------------------------

def q8_quantize_act(x: torch.Tensor, out_blocks: torch.Tensor, flags: int = 0, stream=None):
    M, K = x.shape
    _check("q8_quantize_act", lib().q8_quantize_act(
        _dev(x, torch.float32, "x"), M, K, _dev(out_blocks, torch.uint8, "out_blocks"),
        flags, _stream(stream)))
    return out_blocks


def q8_residual_rmsnorm_quantize(x: torch.Tensor, gamma: torch.Tensor, eps: float,
                                 out_blocks: torch.Tensor, delta: torch.Tensor | None = None,
                                 h_out: torch.Tensor | None = None, flags: int = 0, stream=None):
    """h = x + delta; out_blocks = quantized RMSNorm(h) * gamma (see q8.h)."""
    M, K = x.shape
    _check("q8_residual_rmsnorm_quantize", lib().q8_residual_rmsnorm_quantize(
        _dev(x, torch.float32, "x"), _opt(delta, torch.float32, "delta"),
        _dev(gamma, torch.float32, "gamma"), float(eps), M, K,
        _opt(h_out, torch.float32, "h_out"), _dev(out_blocks, torch.uint8, "out_blocks"),
        flags, _stream(stream)))
    return out_blocks


def q8_swiglu_quantize(gate_up: torch.Tensor, out_blocks: torch.Tensor, flags: int = 0,
                       stream=None):
    """out_blocks = quantized silu(gate) * up, gate_up = [M][2F] (see q8.h)."""
    M, F2 = gate_up.shape
    _check("q8_swiglu_quantize", lib().q8_swiglu_quantize(
        _dev(gate_up, torch.float32, "gate_up"), M, F2 // 2,
        _dev(out_blocks, torch.uint8, "out_blocks"), flags, _stream(stream)))
    return out_blocks


def q8_repack_weights(src_blocks: torch.Tensor, N: int, K: int, dst: torch.Tensor, stream=None):
    _check("q8_repack_weights", lib().q8_repack_weights(
        _dev(src_blocks, torch.uint8, "src_blocks"), N, K, _dev(dst, torch.uint8, "dst"),
        _stream(stream)))
    return dst


def q8_gemm(W: torch.Tensor, N: int, K: int, A_blocks: torch.Tensor, M: int, y: torch.Tensor,
            workspace: torch.Tensor | None = None, flags: int = 0, stream=None):
    ws = _opt(workspace, torch.uint8, "workspace")
    _check("q8_gemm", lib().q8_gemm(
        _dev(W, torch.uint8, "W"), N, K, _dev(A_blocks, torch.uint8, "A_blocks"), M,
        _dev(y, torch.float32, "y"), ws, 0 if workspace is None else workspace.numel(),
        flags, _stream(stream)))
    return y


def q8_fused_quant_gemm(W: torch.Tensor, N: int, K: int, x: torch.Tensor, M: int, y: torch.Tensor,
                        A_blocks_out: torch.Tensor | None = None,
                        workspace: torch.Tensor | None = None, flags: int = 0, stream=None):
    ws = _opt(workspace, torch.uint8, "workspace")
    _check("q8_fused_quant_gemm", lib().q8_fused_quant_gemm(
        _dev(W, torch.uint8, "W"), N, K, _dev(x, torch.float32, "x"), M,
        _dev(y, torch.float32, "y"), _opt(A_blocks_out, torch.uint8, "A_blocks_out"), ws,
        0 if workspace is None else workspace.numel(), flags, _stream(stream)))
    return y


def q8_prefill_workspace_bytes(K: int, M: int) -> int:
    return lib().q8_prefill_workspace_bytes(K, M)


def q8_gemm_prefill(W: torch.Tensor, N: int, K: int, A_blocks: torch.Tensor, M: int, y: torch.Tensor,
                    workspace: torch.Tensor, flags: int = 0, stream=None):
    _check("q8_gemm_prefill", lib().q8_gemm_prefill(
        _dev(W, torch.uint8, "W"), N, K, _dev(A_blocks, torch.uint8, "A_blocks"), M,
        _dev(y, torch.float32, "y"), _dev(workspace, torch.uint8, "workspace"), workspace.numel(),
        flags, _stream(stream)))
    return y


def q8_fused_quant_gemm_prefill(W: torch.Tensor, N: int, K: int, x: torch.Tensor, M: int, y: torch.Tensor,
                                workspace: torch.Tensor, A_blocks_out: torch.Tensor | None = None,
                                flags: int = 0, stream=None):
    _check("q8_fused_quant_gemm_prefill", lib().q8_fused_quant_gemm_prefill(
        _dev(W, torch.uint8, "W"), N, K, _dev(x, torch.float32, "x"), M,
        _dev(y, torch.float32, "y"), _opt(A_blocks_out, torch.uint8, "A_blocks_out"),
        _dev(workspace, torch.uint8, "workspace"), workspace.numel(), flags, _stream(stream)))
    return y


def q8_gemm_noalloc(W: torch.Tensor, N: int, K: int, A_blocks: torch.Tensor, M: int,
                    y: torch.Tensor, flags: int = 0, stream=None):
    """q8_gemm for callers that cannot allocate: split-K scratch is the
    library's built-in array (shared by all calls; do not overlap calls)."""
    _check("q8_gemm_noalloc", lib().q8_gemm_noalloc(
        _dev(W, torch.uint8, "W"), N, K, _dev(A_blocks, torch.uint8, "A_blocks"), M,
        _dev(y, torch.float32, "y"), flags, _stream(stream)))
    return y


def q8_gemm_swiglu(W: torch.Tensor, F: int, K: int, A_blocks: torch.Tensor, M: int,
                   out_blocks: torch.Tensor, flags: int = 0, stream=None):
    """The gate/up GEMV with SwiGLU in its epilogue (W rows interleaved, see
    interleave_gate_up): out_blocks = quantized silu(gate) * up."""
    _check("q8_gemm_swiglu", lib().q8_gemm_swiglu(
        _dev(W, torch.uint8, "W"), F, K, _dev(A_blocks, torch.uint8, "A_blocks"), M,
        _dev(out_blocks, torch.uint8, "out_blocks"), flags, _stream(stream)))
    return out_blocks


def q8_fused_quant_gemm_swiglu(W: torch.Tensor, F: int, K: int, x: torch.Tensor, M: int,
                               out_blocks: torch.Tensor, flags: int = 0, stream=None):
    _check("q8_fused_quant_gemm_swiglu", lib().q8_fused_quant_gemm_swiglu(
        _dev(W, torch.uint8, "W"), F, K, _dev(x, torch.float32, "x"), M,
        _dev(out_blocks, torch.uint8, "out_blocks"), flags, _stream(stream)))
    return out_blocks


def interleave_gate_up(gate: torch.Tensor, up: torch.Tensor) -> torch.Tensor:
    """[F][K] gate and up rows -> the [2F][K] row order q8_gemm_swiglu expects:
    groups of G = q8_packed_tile_rows(2F) / 2 gate rows, each followed by the
    up rows of the same indices (a copy; no arithmetic)."""
    F, K = gate.shape
    G = q8_packed_tile_rows(2 * F) // 2
    if G < 32 or F % G:
        raise ValueError("F = %d has no SwiGLU epilogue layout (group %d)" % (F, G))
    return torch.stack([gate.reshape(F // G, G, K), up.reshape(F // G, G, K)], dim=1).reshape(2 * F, K)


# ---- int8 KV cache codec ---------------------------------------------------------

def q8_kv_cache_bytes(capacity: int, D: int) -> int:
    return int(lib().q8_kv_cache_bytes(capacity, D))


def q8_kv_quantize(x: torch.Tensor, cache_q: torch.Tensor, cache_d: torch.Tensor,
                   slots: torch.Tensor | None = None, flags: int = 0, stream=None):
    """Write K/V rows x [rows][D] into cache slots (slots: int32 [rows], or
    None for slot = row) as int8 quants cache_q [capacity][D] and fp32 scales
    cache_d [capacity][D/32] (see q8.h)."""
    rows, D = x.shape
    capacity = cache_q.shape[0]
    if cache_q.shape != (capacity, D) or cache_d.shape != (capacity, D // QK):
        raise ValueError("cache planes must be [capacity][D] int8 and [capacity][D/32] fp32")
    _check("q8_kv_quantize", lib().q8_kv_quantize(
        _dev(x, torch.float32, "x"), rows, D, _opt(slots, torch.int32, "slots"), capacity,
        _dev(cache_q, torch.int8, "cache_q"), _dev(cache_d, torch.float32, "cache_d"),
        flags, _stream(stream)))
    return cache_q, cache_d


def q8_kv_dequantize(cache_q: torch.Tensor, cache_d: torch.Tensor, out: torch.Tensor,
                     slots: torch.Tensor | None = None, flags: int = 0, stream=None):
    """out [rows][D] fp32 = the dequantized cache slots slots[r] (slot r when
    slots is None)."""
    capacity, D = cache_q.shape
    rows = out.shape[0]
    if cache_d.shape != (capacity, D // QK) or out.shape != (rows, D):
        raise ValueError("shapes: cache_q [capacity][D], cache_d [capacity][D/32], out [rows][D]")
    _check("q8_kv_dequantize", lib().q8_kv_dequantize(
        _dev(cache_q, torch.int8, "cache_q"), _dev(cache_d, torch.float32, "cache_d"), capacity, D,
        _opt(slots, torch.int32, "slots"), rows, _dev(out, torch.float32, "out"), flags, _stream(stream)))
    return out


# ---- test hooks ----------------------------------------------------------------

def q8_unpack_weights(packed: torch.Tensor, N: int, K: int, dst_blocks: torch.Tensor, stream=None):
    _check("q8_unpack_weights", lib().q8_unpack_weights(
        _dev(packed, torch.uint8, "packed"), N, K, _dev(dst_blocks, torch.uint8, "dst_blocks"),
        _stream(stream)))
    return dst_blocks


def q8_block_dots(W: torch.Tensor, N: int, K: int, A_blocks: torch.Tensor, M: int,
                  isum: torch.Tensor, stream=None):
    _check("q8_block_dots", lib().q8_block_dots(
        _dev(W, torch.uint8, "W"), N, K, _dev(A_blocks, torch.uint8, "A_blocks"), M,
        _dev(isum, torch.int32, "isum"), _stream(stream)))
    return isum


def q8_device_error() -> int:
    code = ctypes.c_uint(0)
    _check("q8_device_error", lib().q8_device_error(ctypes.byref(code)))
    return code.value


def q8_set_wait_limit_ns(ns: int) -> None:
    """Test hook: limit of the GEMV ring waits for later launches (0 = 2 s)."""
    _check("q8_set_wait_limit_ns", lib().q8_set_wait_limit_ns(int(ns)))


def q8_device_info():
    sm, ma, mi = ctypes.c_int(), ctypes.c_int(), ctypes.c_int()
    _check("q8_device_info", lib().q8_device_info(ctypes.byref(sm), ctypes.byref(ma), ctypes.byref(mi)))
    return sm.value, ma.value, mi.value


# ---- conveniences (allocation through torch; no arithmetic) --------------------

def empty_blocks(rows: int, K: int, device="cuda") -> torch.Tensor:
    return torch.empty((rows, (K // QK) * BLOCK_BYTES), dtype=torch.uint8, device=device)


def empty_packed(N: int, K: int, device="cuda") -> torch.Tensor:
    return torch.empty(q8_packed_bytes(N, K), dtype=torch.uint8, device=device)


def new_workspace(N: int, K: int, M: int, device="cuda") -> torch.Tensor | None:
    n = q8_workspace_bytes(N, K, M)
    return torch.zeros(n, dtype=torch.uint8, device=device) if n else None


def new_prefill_workspace(K: int, M: int, device="cuda") -> torch.Tensor:
    return torch.empty(q8_prefill_workspace_bytes(K, M), dtype=torch.uint8, device=device)


def pack_weights_f32(w: torch.Tensor, stream=None) -> torch.Tensor:
    """fp32 [N][K] weights on the device -> packed Q8_0 (quantize, then repack)."""
    N, K = w.shape
    blocks = empty_blocks(N, K, w.device)
    q8_quantize_act(w, blocks, stream=stream)
    packed = empty_packed(N, K, w.device)
    q8_repack_weights(blocks, N, K, packed, stream=stream)
    return packed
