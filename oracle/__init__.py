"""The oracle: a plain CPU restatement of the Q8_0 block-quantized product.

TEST INFRASTRUCTURE ONLY.  Only the test suite, ``__graft_entry__.smoke()``
and the benchmark's CPU-baseline leg may import this package.  It shares no
code with the CUDA library (``q8_block_quantized_gb300``) and imports nothing
from it; the library never imports this package.

The arithmetic lives in ``q8_oracle.c`` (plain C99, built with gcc at
``-O2 -ffp-contract=off``); this module only builds that file and passes numpy
arrays to it.  Each C function cites the page passage it follows:

* "Ferro" README, "How the iGPU path is fast", item 1: Q8_0 weights, per-32
  activation blocks, int8 dot products.
* "Ember: packed Q8 decode", the row-contiguous source figure (a block is a
  scale followed by 32 quants) and the packed 16-row tile figure (544 bytes
  per 16 blocks).
* "Ferro" README, "How the iGPU path is fast", item 3: fused producers (the
  residual add and the norm, SwiGLU) that emit the next GEMM's int8 input.
* "Ferro" README, "Exactness, scheduling and operations (LM serving)", item
  "KV cache": K/V rows as int8 with one fp32 scale per 32 values.

Every function is pinned by ``tests/test_oracle_pins.py``; none is
"parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "q8_oracle.c")
_LIB = os.path.join(_HERE, "libq8oracle.so")
_lock = threading.Lock()
_lib = None

QK = 32
BLOCK_BYTES = 34
EMBER_TILE_BYTES = 544

_CFLAGS = ["-std=c99", "-O2", "-ffp-contract=off", "-fno-fast-math",
           "-fPIC", "-shared", "-Wall", "-Wextra"]


def build(force: bool = False) -> str:
    """Compile q8_oracle.c into libq8oracle.so next to it (gcc, portable C)."""
    stale = (not os.path.exists(_LIB)
             or os.path.getmtime(_LIB) < os.path.getmtime(_SRC))
    if force or stale:
        tmp = _LIB + ".tmp.%d" % os.getpid()
        subprocess.run(["gcc", *_CFLAGS, "-o", tmp, _SRC, "-lm"], check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        u8p = ctypes.POINTER(ctypes.c_uint8)
        f32p = ctypes.POINTER(ctypes.c_float)
        f64p = ctypes.POINTER(ctypes.c_double)
        i32p = ctypes.POINTER(ctypes.c_int32)
        i64 = ctypes.c_int64
        lib.q8o_f32_to_f16.argtypes = [ctypes.c_float]
        lib.q8o_f32_to_f16.restype = ctypes.c_uint16
        lib.q8o_f16_to_f32.argtypes = [ctypes.c_uint16]
        lib.q8o_f16_to_f32.restype = ctypes.c_float
        lib.q8o_quantize_block.argtypes = [f32p, u8p]
        lib.q8o_quantize_rows.argtypes = [f32p, i64, i64, u8p]
        lib.q8o_block_dots.argtypes = [u8p, i64, i64, u8p, i64, i32p]
        lib.q8o_gemm.argtypes = [u8p, i64, i64, u8p, i64, f64p, f64p]
        lib.q8o_quant_gemm.argtypes = [u8p, i64, i64, f32p, i64, u8p, f64p, f64p]
        lib.q8o_gemm_prefill_order.argtypes = [u8p, i64, i64, u8p, i64, i64, f32p]
        lib.q8o_ember_tile_pack.argtypes = [u8p, u8p]
        lib.q8o_pairwise_sum.argtypes = [f32p, i64]
        lib.q8o_pairwise_sum.restype = ctypes.c_float
        lib.q8o_exp_array.argtypes = [f32p, i64, f32p]
        lib.q8o_silu_array.argtypes = [f32p, i64, f32p]
        lib.q8o_residual_rmsnorm_quantize.argtypes = [f32p, f32p, f32p, ctypes.c_float, i64, i64,
                                                      f32p, u8p]
        lib.q8o_swiglu_quantize.argtypes = [f32p, i64, i64, u8p]
        lib.q8o_ember_tile_unpack.argtypes = [u8p, u8p]
        i8p = ctypes.POINTER(ctypes.c_int8)
        lib.q8o_kv_quantize.argtypes = [f32p, i64, i64, i32p, i64, i8p, f32p]
        lib.q8o_kv_dequantize.argtypes = [i8p, f32p, i64, i64, i32p, i64, f32p]
        for name in ("q8o_qk", "q8o_block_bytes", "q8o_ember_tile_bytes", "q8o_kv_block_bytes"):
            getattr(lib, name).restype = ctypes.c_int
        _lib = lib
        return lib


def _ptr(a: np.ndarray, ctype):
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def _f32(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.float32)


def _u8(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.uint8)


def constants() -> dict:
    lib = _load()
    return {"qk": lib.q8o_qk(), "block_bytes": lib.q8o_block_bytes(),
            "ember_tile_bytes": lib.q8o_ember_tile_bytes(),
            "kv_block_bytes": lib.q8o_kv_block_bytes()}


def f32_to_f16_bits(x) -> np.ndarray:
    """binary32 -> binary16 bit patterns, round to nearest even (elementwise)."""
    lib = _load()
    flat = _f32(x).ravel()
    out = np.empty(flat.shape, dtype=np.uint16)
    for i, v in enumerate(flat):
        out[i] = lib.q8o_f32_to_f16(float(v))
    return out.reshape(np.shape(x))


def f16_bits_to_f32(h) -> np.ndarray:
    lib = _load()
    flat = np.ascontiguousarray(h, dtype=np.uint16).ravel()
    out = np.empty(flat.shape, dtype=np.float32)
    for i, v in enumerate(flat):
        out[i] = lib.q8o_f16_to_f32(int(v))
    return out.reshape(np.shape(h))


def quantize(x) -> np.ndarray:
    """fp32 [rows][K] -> uint8 [rows][K/32*34] Q8_0 blocks."""
    lib = _load()
    x = _f32(x)
    if x.ndim == 1:
        x = x.reshape(1, -1)
    rows, K = x.shape
    if K % QK:
        raise ValueError("K must be a multiple of 32")
    out = np.zeros((rows, (K // QK) * BLOCK_BYTES), dtype=np.uint8)
    lib.q8o_quantize_rows(_ptr(x, ctypes.c_float), rows, K, _ptr(out, ctypes.c_uint8))
    return out


def block_dots(W, A, K: int) -> np.ndarray:
    """Exact per-block int32 dots: isum[m][n][b]."""
    lib = _load()
    W, A = _u8(W), _u8(A)
    nb = K // QK
    N = W.size // (nb * BLOCK_BYTES)
    M = A.size // (nb * BLOCK_BYTES)
    isum = np.zeros((M, N, nb), dtype=np.int32)
    lib.q8o_block_dots(_ptr(W, ctypes.c_uint8), N, K, _ptr(A, ctypes.c_uint8), M,
                       _ptr(isum, ctypes.c_int32))
    return isum


def gemm(W, A, K: int):
    """(y, S): fp64 outputs [M][N] and the sum of |terms| per output."""
    lib = _load()
    W, A = _u8(W), _u8(A)
    nb = K // QK
    N = W.size // (nb * BLOCK_BYTES)
    M = A.size // (nb * BLOCK_BYTES)
    y = np.zeros((M, N), dtype=np.float64)
    S = np.zeros((M, N), dtype=np.float64)
    lib.q8o_gemm(_ptr(W, ctypes.c_uint8), N, K, _ptr(A, ctypes.c_uint8), M,
                 _ptr(y, ctypes.c_double), _ptr(S, ctypes.c_double))
    return y, S


def gemm_prefill_order(W, A, K: int, seg: int = 16) -> np.ndarray:
    """float32 [M][N]: the prefill product in its fixed single-precision
    order (fma through segments of `seg` blocks; the segment sums of the
    first ceil(nseg/2) segments and of the rest each added in order; then the
    two halves added); see q8o_gemm_prefill_order."""
    lib = _load()
    W, A = _u8(W), _u8(A)
    nb = K // QK
    N = W.size // (nb * BLOCK_BYTES)
    M = A.size // (nb * BLOCK_BYTES)
    y = np.zeros((M, N), dtype=np.float32)
    lib.q8o_gemm_prefill_order(_ptr(W, ctypes.c_uint8), N, K, _ptr(A, ctypes.c_uint8), M, seg,
                               _ptr(y, ctypes.c_float))
    return y


def quant_gemm(W, x, K: int):
    """Fused form: quantize fp32 activations x [M][K], then the product.
    Returns (y, S, A_blocks)."""
    lib = _load()
    W, x = _u8(W), _f32(x)
    if x.ndim == 1:
        x = x.reshape(1, -1)
    nb = K // QK
    N = W.size // (nb * BLOCK_BYTES)
    M = x.shape[0]
    A = np.zeros((M, nb * BLOCK_BYTES), dtype=np.uint8)
    y = np.zeros((M, N), dtype=np.float64)
    S = np.zeros((M, N), dtype=np.float64)
    lib.q8o_quant_gemm(_ptr(W, ctypes.c_uint8), N, K, _ptr(x, ctypes.c_float), M,
                       _ptr(A, ctypes.c_uint8), _ptr(y, ctypes.c_double),
                       _ptr(S, ctypes.c_double))
    return y, S, A


def pairwise_sum(v) -> float:
    """Single-precision pairwise (tree) sum, zero-padded to a power of two."""
    v = _f32(v).ravel()
    return float(_load().q8o_pairwise_sum(_ptr(v, ctypes.c_float), v.size))


def exp_f32(x) -> np.ndarray:
    """The fixed single-precision e^x of the fused producers (elementwise)."""
    x = _f32(x)
    out = np.empty_like(x)
    _load().q8o_exp_array(_ptr(x.ravel(), ctypes.c_float), x.size, _ptr(out.ravel(), ctypes.c_float))
    return out


def silu_f32(x) -> np.ndarray:
    """silu(g) = g / (1 + e^-g) in single precision (elementwise)."""
    x = _f32(x)
    out = np.empty_like(x)
    _load().q8o_silu_array(_ptr(x.ravel(), ctypes.c_float), x.size, _ptr(out.ravel(), ctypes.c_float))
    return out


def residual_rmsnorm_quantize(x, delta, gamma, eps: float):
    """h = x + delta (delta may be None), y = RMSNorm(h) * gamma, quantized.
    Returns (h [M][K] float32, blocks uint8 [M][K/32*34])."""
    lib = _load()
    x = _f32(x)
    if x.ndim == 1:
        x = x.reshape(1, -1)
    M, K = x.shape
    if K % QK:
        raise ValueError("K must be a multiple of 32")
    d = None if delta is None else _f32(delta).reshape(M, K)
    g = _f32(gamma).reshape(K)
    h = np.zeros((M, K), dtype=np.float32)
    out = np.zeros((M, (K // QK) * BLOCK_BYTES), dtype=np.uint8)
    lib.q8o_residual_rmsnorm_quantize(_ptr(x, ctypes.c_float),
                                      None if d is None else _ptr(d, ctypes.c_float),
                                      _ptr(g, ctypes.c_float), float(eps), M, K,
                                      _ptr(h, ctypes.c_float), _ptr(out, ctypes.c_uint8))
    return h, out


def swiglu_quantize(gu, F: int) -> np.ndarray:
    """gu [M][2F] (gate | up) -> blocks of silu(gate) * up, uint8 [M][F/32*34]."""
    gu = _f32(gu)
    if gu.ndim == 1:
        gu = gu.reshape(1, -1)
    M = gu.shape[0]
    if gu.shape[1] != 2 * F or F % QK:
        raise ValueError("gu must be [M][2F] with F a multiple of 32")
    out = np.zeros((M, (F // QK) * BLOCK_BYTES), dtype=np.uint8)
    _load().q8o_swiglu_quantize(_ptr(gu, ctypes.c_float), M, F, _ptr(out, ctypes.c_uint8))
    return out


def ember_tile_pack(blocks16) -> np.ndarray:
    """16 row-contiguous blocks (uint8 [16][34]) -> one 544-byte Ember record."""
    lib = _load()
    src = _u8(blocks16).reshape(16 * BLOCK_BYTES)
    out = np.zeros(EMBER_TILE_BYTES, dtype=np.uint8)
    lib.q8o_ember_tile_pack(_ptr(src, ctypes.c_uint8), _ptr(out, ctypes.c_uint8))
    return out


def ember_tile_unpack(tile) -> np.ndarray:
    lib = _load()
    src = _u8(tile).reshape(EMBER_TILE_BYTES)
    out = np.zeros((16, BLOCK_BYTES), dtype=np.uint8)
    lib.q8o_ember_tile_unpack(_ptr(src, ctypes.c_uint8), _ptr(out, ctypes.c_uint8))
    return out


def kv_quantize(x, capacity: int, slots=None, cache=None):
    """K/V rows x [rows][D] fp32 written into an int8 cache of `capacity`
    slots: returns (q int8 [capacity][D], d fp32 [capacity][D/32]).  Row r
    goes to slot slots[r] (slot r when slots is None); a slot outside
    [0, capacity) is skipped.  `cache` = (q, d) arrays updated in place
    (new zeroed arrays when None)."""
    lib = _load()
    x = _f32(x)
    if x.ndim == 1:
        x = x.reshape(1, -1)
    rows, D = x.shape
    if D % QK:
        raise ValueError("D must be a multiple of 32")
    if cache is None:
        q = np.zeros((capacity, D), dtype=np.int8)
        d = np.zeros((capacity, D // QK), dtype=np.float32)
    else:
        q, d = cache
        assert q.dtype == np.int8 and d.dtype == np.float32 and q.flags["C_CONTIGUOUS"] and d.flags["C_CONTIGUOUS"]
        assert q.shape == (capacity, D) and d.shape == (capacity, D // QK)
    sl = None if slots is None else np.ascontiguousarray(slots, dtype=np.int32)
    if sl is not None and sl.size != rows:
        raise ValueError("one slot per row")
    lib.q8o_kv_quantize(_ptr(x, ctypes.c_float), rows, D,
                        None if sl is None else _ptr(sl, ctypes.c_int32), capacity,
                        _ptr(q, ctypes.c_int8), _ptr(d, ctypes.c_float))
    return q, d


def kv_dequantize(q, d, slots=None, rows=None) -> np.ndarray:
    """Read rows back from an int8 cache (q [capacity][D], d [capacity][D/32]):
    out[r] = q[slot] * d[slot] per 32-value block, fp32; rows whose slot is
    outside the cache stay zero."""
    lib = _load()
    q = np.ascontiguousarray(q, dtype=np.int8)
    d = _f32(d)
    capacity, D = q.shape
    sl = None if slots is None else np.ascontiguousarray(slots, dtype=np.int32)
    n = capacity if sl is None else sl.size
    if rows is not None:
        n = rows
    out = np.zeros((n, D), dtype=np.float32)
    lib.q8o_kv_dequantize(_ptr(q, ctypes.c_int8), _ptr(d, ctypes.c_float), capacity, D,
                          None if sl is None else _ptr(sl, ctypes.c_int32), n, _ptr(out, ctypes.c_float))
    return out


# --- byte views of a block array (no arithmetic): scale bits and quants -------

def split_blocks(blocks, K: int):
    """uint8 [rows][K/32*34] -> (d16 bits uint16 [rows][K/32], q int8 [rows][K/32][32])."""
    b = _u8(blocks)
    rows = b.size // ((K // QK) * BLOCK_BYTES)
    b = b.reshape(rows, K // QK, BLOCK_BYTES)
    d16 = b[:, :, 0].astype(np.uint16) | (b[:, :, 1].astype(np.uint16) << 8)
    q = b[:, :, 2:].view(np.int8)
    return d16, q
