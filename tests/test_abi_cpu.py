"""CPU checks of the C ABI: libq8.so builds, loads, exports every function
include/q8.h declares, the binding covers exactly those, and host-side
argument checks reject bad calls before anything touches a device."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    names = []
    for fn in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if fn.endswith(".h"):
            with open(os.path.join(ROOT, "include", fn)) as f:
                names += re.findall(r"^Q8_API\s+[\w\s\*]*?\b(q8_\w+)\s*\(", f.read(), re.M)
    return names


@pytest.fixture(scope="module")
def lib():
    from q8_block_quantized_gb300 import build
    build.build()
    import q8_block_quantized_gb300 as q8
    return q8.lib()


def test_header_declares_the_four_calls():
    d = set(_declared())
    for name in ("q8_quantize_act", "q8_repack_weights", "q8_gemm", "q8_fused_quant_gemm"):
        assert name in d


def test_every_declared_symbol_is_exported(lib):
    names = _declared()
    assert len(names) >= 10
    for name in names:
        assert hasattr(lib, name), name


def test_binding_signatures_match_header(lib):
    import q8_block_quantized_gb300 as q8
    assert set(q8.SIGNATURES) == set(_declared())


def test_sizes_and_strings(lib):
    import q8_block_quantized_gb300 as q8
    assert q8.q8_blocks_bytes(3, 96) == 3 * 3 * 34
    assert q8.q8_packed_bytes(128256, 2048) == 128256 * 64 * 34
    assert q8.q8_packed_bytes(7, 33) == 0
    assert q8.q8_blocks_bytes(0, 32) == 0
    assert lib.q8_abi_version() == 1
    for code in (0, -1, -2, -3, -4, -5, -6, -7, -8):
        assert lib.q8_strerror(code).decode().startswith(q8.STATUS[code])


def test_host_argument_checks_reject_before_any_device_work(lib):
    # every case fails in the host-side checks, which run before the device
    # is queried; no GPU is needed
    fake = ctypes.c_void_p(0x10000)      # 16-byte aligned, never dereferenced
    odd = ctypes.c_void_p(0x10001)
    y = ctypes.c_void_p(0x20000)
    g = lib.q8_gemm
    assert g(None, 8, 64, fake, 1, y, None, 0, 0, None) == -1          # null W
    assert g(fake, 8, 64, None, 1, y, None, 0, 0, None) == -1          # null A
    assert g(fake, 8, 64, fake, 1, y, None, 0, 4, None) == -1          # unknown flag
    assert g(fake, 8, 63, fake, 1, y, None, 0, 0, None) == -2          # K % 32
    assert g(fake, 8, 0, fake, 1, y, None, 0, 0, None) == -2           # K = 0
    assert g(fake, 0, 64, fake, 1, y, None, 0, 0, None) == -2          # N = 0
    assert g(fake, 8, 64, fake, 0, y, None, 0, 0, None) == -2          # M = 0
    assert g(fake, 8, 64, fake, 4097, y, None, 0, 0, None) == -2       # M > Q8_MAX_M
    assert lib.q8_block_dots(fake, 8, 64, fake, 65, fake, None) == -2  # M > Q8_MAX_DOTS_M
    assert g(odd, 8, 64, fake, 1, y, None, 0, 0, None) == -3           # W misaligned
    assert g(fake, 8, 64, odd, 1, y, None, 0, 0, None) == -3           # A misaligned
    f = lib.q8_fused_quant_gemm
    assert f(fake, 8, 64, None, 1, y, None, None, 0, 0, None) == -1
    assert f(fake, 8, 64, odd, 1, y, None, None, 0, 0, None) == -3
    assert f(fake, 8, 64, fake, 1, y, odd, None, 0, 0, None) == -3
    q = lib.q8_quantize_act
    assert q(None, 1, 64, fake, 0, None) == -1
    assert q(fake, 1, 48, fake, 0, None) == -2
    assert q(fake, -1, 64, fake, 0, None) == -2
    assert q(odd, 1, 64, fake, 0, None) == -3
    r = lib.q8_repack_weights
    assert r(fake, 8, 64, None, None) == -1
    assert r(fake, 8, 64, ctypes.c_void_p(0x10008), None) == -3        # dst 8-aligned only
    assert r(fake, 8, 40, fake, None) == -2
    assert lib.q8_block_dots(fake, 8, 64, fake, 1, odd, None) == -3
    assert lib.q8_unpack_weights(fake, 8, 64, None, None) == -1
    assert lib.q8_gemm_noalloc(fake, 8, 64, fake, 1, y, 2, None) == -1   # only Q8_FLAG_PDL there
    n = lib.q8_residual_rmsnorm_quantize
    assert n(None, None, fake, 1e-5, 1, 64, None, fake, 0, None) == -1          # null x
    assert n(fake, None, None, 1e-5, 1, 64, None, fake, 0, None) == -1          # null gamma
    assert n(fake, None, fake, 0.0, 1, 64, None, fake, 0, None) == -1           # eps = 0
    assert n(fake, None, fake, float("nan"), 1, 64, None, fake, 0, None) == -1  # eps NaN
    assert n(fake, None, fake, float("inf"), 1, 64, None, fake, 0, None) == -1  # eps inf
    assert n(fake, None, fake, 1e-5, 1, 48, None, fake, 0, None) == -2          # K % 32
    assert n(fake, None, fake, 1e-5, 0, 64, None, fake, 0, None) == -2          # M = 0
    assert n(fake, None, fake, 1e-5, 1, (1 << 24) + 32, None, fake, 0, None) == -2  # K too large
    eight = ctypes.c_void_p(0x10008)
    assert n(eight, None, fake, 1e-5, 1, 64, None, fake, 0, None) == -3         # x 8-aligned only
    assert n(fake, eight, fake, 1e-5, 1, 64, None, fake, 0, None) == -3         # delta
    assert n(fake, None, fake, 1e-5, 1, 64, eight, fake, 0, None) == -3         # h_out
    assert n(fake, None, fake, 1e-5, 1, 64, None, odd, 0, None) == -3           # out odd
    e = lib.q8_gemm_swiglu
    assert e(None, 64, 64, fake, 1, fake, 0, None) == -1                        # null W
    assert e(fake, 64, 64, None, 1, fake, 0, None) == -1                        # null A
    assert e(fake, 64, 64, fake, 1, fake, 2, None) == -1                        # tcgen05 not offered
    assert e(fake, 48, 64, fake, 1, fake, 0, None) == -2                        # F % 32
    assert e(fake, 64, 64, fake, 0, fake, 0, None) == -2                        # M = 0
    assert e(fake, 64, 64, fake, 1, odd, 0, None) == -2                         # 16-row tiles: no layout
    assert lib.q8_fused_quant_gemm_swiglu(fake, 8192, 64, None, 1, fake, 0, None) == -1
    pf = lib.q8_gemm_prefill
    big = 1 << 20
    assert pf(None, 64, 64, fake, 1, y, fake, big, 0, None) == -1              # null W
    assert pf(fake, 64, 64, None, 1, y, fake, big, 0, None) == -1              # null A
    assert pf(fake, 64, 64, fake, 1, None, fake, big, 0, None) == -1           # null y
    assert pf(fake, 64, 64, fake, 1, y, fake, big, 2, None) == -1              # only Q8_FLAG_PDL
    assert pf(fake, 64, 48, fake, 1, y, fake, big, 0, None) == -2              # K % 32
    assert pf(fake, 64, 65536 + 32, fake, 1, y, fake, big, 0, None) == -2      # K > Q8_MAX_PREFILL_K
    assert pf(fake, 0, 64, fake, 1, y, fake, big, 0, None) == -2               # N = 0
    assert pf(fake, 64, 64, fake, 0, y, fake, big, 0, None) == -2              # M = 0
    assert pf(fake, (1 << 31) - 1, 64, fake, (1 << 31) - 1, y, fake, big, 0, None) == -2  # > 2^31 tiles
    assert pf(odd, 64, 64, fake, 1, y, fake, big, 0, None) == -3               # W misaligned
    assert pf(fake, 64, 64, odd, 1, y, fake, big, 0, None) == -3               # A misaligned
    assert pf(fake, 64, 64, fake, 1, y, eight, big, 0, None) == -3             # workspace 8-aligned
    assert pf(fake, 64, 64, fake, 3, y, None, big, 0, None) == -6              # no workspace
    assert pf(fake, 64, 64, fake, 3, y, fake, 4096 + 208 - 1, 0, None) == -6   # one byte short (flags + packed)
    fq = lib.q8_fused_quant_gemm_prefill
    assert fq(fake, 64, 64, None, 1, y, None, fake, big, 0, None) == -1        # null x
    assert fq(fake, 64, 64, fake, 1, y, odd, fake, big, 0, None) == -3         # A_blocks_out odd
    assert fq(fake, 64, 64, fake, 3, y, None, fake, 4096 + 2 * 208 - 1, 0, None) == -6  # x's blocks need room too
    assert lib.q8_prefill_workspace_bytes(64, 3) == 4096 + 2 * 208             # split flags + 3*2*34 = 204 -> 208, twice
    assert lib.q8_prefill_workspace_bytes(65536 + 32, 3) == 0
    assert lib.q8_prefill_workspace_bytes(64, 0) == 0
    s = lib.q8_swiglu_quantize
    assert s(None, 1, 64, fake, 0, None) == -1
    assert s(fake, 1, 64, fake, 2, None) == -1                                  # unknown flag
    assert s(fake, 1, 48, fake, 0, None) == -2
    assert s(fake, 0, 64, fake, 0, None) == -2
    assert s(eight, 1, 64, fake, 0, None) == -3
    assert s(fake, 1, 64, odd, 0, None) == -3
    kq = lib.q8_kv_quantize
    assert kq(None, 1, 64, None, 4, fake, fake, 0, None) == -1                  # null x
    assert kq(fake, 1, 64, None, 4, None, fake, 0, None) == -1                  # null quant plane
    assert kq(fake, 1, 64, None, 4, fake, None, 0, None) == -1                  # null scale plane
    assert kq(fake, 1, 64, None, 4, fake, fake, 2, None) == -1                  # unknown flag
    assert kq(fake, 1, 48, None, 4, fake, fake, 0, None) == -2                  # D % 32
    assert kq(fake, 0, 64, None, 4, fake, fake, 0, None) == -2                  # rows = 0
    assert kq(fake, 1, 64, None, 0, fake, fake, 0, None) == -2                  # capacity = 0
    assert kq(fake, 1, (1 << 24) + 32, None, 4, fake, fake, 0, None) == -2      # D > Q8_MAX_KV_D
    assert kq(eight, 1, 64, None, 4, fake, fake, 0, None) == -3                 # x 8-aligned only
    assert kq(fake, 1, 64, odd, 4, fake, fake, 0, None) == -3                   # slots odd
    assert kq(fake, 1, 64, None, 4, ctypes.c_void_p(0x10002), fake, 0, None) == -3
    kd = lib.q8_kv_dequantize
    assert kd(fake, fake, 4, 64, None, 1, None, 0, None) == -1                  # null out
    assert kd(fake, fake, 4, 64, None, 1, eight, 0, None) == -3                 # out 8-aligned only
    assert kd(fake, fake, 4, 40, None, 1, fake, 0, None) == -2
    assert kd(fake, odd, 4, 64, None, 1, fake, 0, None) == -3                   # scales odd
    assert lib.q8_kv_cache_bytes(4096, 512) == 4096 * 16 * 36
    assert lib.q8_kv_cache_bytes(0, 512) == 0 and lib.q8_kv_cache_bytes(4, 40) == 0


def test_no_device_means_an_error_not_a_fallback(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    fake = ctypes.c_void_p(0x10000)
    st = lib.q8_gemm(fake, 8, 64, fake, 1, fake, None, 0, 0, None)
    assert st in (-5, -4)
    assert lib.q8_workspace_bytes(2048, 2048, 1) == 0
