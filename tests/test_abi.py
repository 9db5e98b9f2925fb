"""The C ABI without a GPU: the library loads, exports every function the
header declares, and rejects bad arguments before touching the device."""
import ctypes

import pytest

from fp8_fine_grained_17_b300 import fp8bs

EXPECTED = {"fp8bs_quantize_act_1x128", "fp8bs_quantize_weight_128x128", "fp8bs_gemm",
            "fp8bs_grouped_gemm", "fp8bs_gemm_tiled", "fp8bs_grouped_gemm_tiled",
            "fp8bs_norm_quantize_act_1x128", "fp8bs_gemm_bf16_act", "fp8bs_grouped_gemm_bf16_act",
            "fp8bs_quantize_act_and_weight", "fp8bs_quantize_act_1x128_pow2",
            "fp8bs_quantize_weight_128x128_pow2",
            "fp8bs_status_string", "fp8bs_last_device_error"}


def test_header_declares_the_boundary():
    assert EXPECTED <= set(fp8bs.header_symbols())


def test_library_exports_every_header_symbol():
    L = fp8bs.lib()
    for name in fp8bs.header_symbols():
        assert hasattr(L, name), name


def test_status_strings():
    assert fp8bs.status_string(0) == "ok"
    assert "timed out" in fp8bs.status_string(4)
    assert fp8bs.status_string(99) == "unknown status"


# Fake, 16-byte aligned, never dereferenced addresses: every call below is
# rejected (or is a no-op) before any CUDA call.
P = 0x10000


def test_quantize_argument_checks():
    L = fp8bs.lib()
    f = L.fp8bs_quantize_act_1x128
    assert f(P, -1, 128, 128, P, 128, P, None) == fp8bs.ERR_INVALID_ARG
    assert f(P, 4, 100, 128, P, 128, P, None) == fp8bs.ERR_UNSUPPORTED
    assert f(P, 0, 128, 128, P, 128, P, None) == fp8bs.OK          # empty: no-op
    assert f(None, 4, 128, 128, P, 128, P, None) == fp8bs.ERR_INVALID_ARG
    assert f(P, 4, 128, 64, P, 128, P, None) == fp8bs.ERR_INVALID_ARG   # ldx < K
    assert f(P + 8, 4, 128, 128, P, 128, P, None) == fp8bs.ERR_INVALID_ARG  # misaligned
    assert f(P, 4, 128, 132, P, 128, P, None) == fp8bs.ERR_INVALID_ARG  # row not 16B aligned
    g = L.fp8bs_quantize_weight_128x128
    assert g(P, 4, 130, 130, P, 130, P, None) == fp8bs.ERR_UNSUPPORTED
    assert g(P, 0, 128, 128, P, 128, P, None) == fp8bs.OK
    assert g(P, 4, 128, 128, None, 128, P, None) == fp8bs.ERR_INVALID_ARG


def test_gemm_argument_checks():
    f = fp8bs.lib().fp8bs_gemm
    assert f(P, P, P, P, P, 0, 4, 200, 128, 200, None) == fp8bs.ERR_UNSUPPORTED   # N % 128
    assert f(P, P, P, P, P, 0, 4, 128, 100, 128, None) == fp8bs.ERR_UNSUPPORTED   # K % 128
    assert f(P, P, P, P, P, 0, -4, 128, 128, 128, None) == fp8bs.ERR_INVALID_ARG
    assert f(P, P, P, P, P, 0, 0, 128, 128, 128, None) == fp8bs.OK               # M = 0
    assert f(P, P, P, P, None, 0, 4, 128, 128, 128, None) == fp8bs.ERR_INVALID_ARG
    assert f(P, P, P, P, P, 7, 4, 128, 128, 128, None) == fp8bs.ERR_INVALID_ARG   # dtype
    assert f(P, P, P, P, P, 0, 4, 128, 128, 100, None) == fp8bs.ERR_INVALID_ARG   # ldc < N
    assert f(P, P, P, P, P, 1, 4, 128, 128, 132, None) == fp8bs.ERR_INVALID_ARG   # bf16 row align
    assert f(P, P + 1, P, P, P, 0, 4, 128, 128, 128, None) == fp8bs.ERR_INVALID_ARG


def test_grouped_argument_checks():
    f = fp8bs.lib().fp8bs_grouped_gemm
    assert f(P, P, P, 0, 10, P, P, P, 0, 128, 128, 128, None) == fp8bs.ERR_INVALID_ARG   # E = 0
    assert f(P, P, P, 513, 10, P, P, P, 0, 128, 128, 128, None) == fp8bs.ERR_UNSUPPORTED
    assert f(P, P, None, 2, 10, P, P, P, 0, 128, 128, 128, None) == fp8bs.ERR_INVALID_ARG
    assert f(P, P, P, 2, 0, P, P, P, 0, 128, 128, 128, None) == fp8bs.OK                 # no rows
    assert f(P, P, P + 2, 2, 10, P, P, P, 0, 128, 128, 128, None) == fp8bs.ERR_INVALID_ARG


def test_tile_argument_checks():
    L = fp8bs.lib()
    f = L.fp8bs_gemm_tiled
    assert f(P, P, P, P, P, 0, 4, 128, 128, 128, 9, None) == fp8bs.ERR_INVALID_ARG     # unknown tile
    assert f(P, P, P, P, P, 0, 4, 384, 128, 384, fp8bs.TILE_PAIR_256x256, None) == fp8bs.ERR_INVALID_ARG
    assert f(P, P, P, P, P, 0, 0, 512, 128, 512, fp8bs.TILE_PAIR_256x256, None) == fp8bs.OK
    g = L.fp8bs_grouped_gemm_tiled
    assert g(P, P, P, 2, 10, P, P, P, 0, 128, 128, 128, -1, None) == fp8bs.ERR_INVALID_ARG
    assert g(P, P, P, 2, 0, P, P, P, 0, 256, 128, 256, fp8bs.TILE_PAIR_256x128, None) == fp8bs.OK


def test_norm_argument_checks():
    f = fp8bs.lib().fp8bs_norm_quantize_act_1x128
    R, L_ = fp8bs.NORM_RMS, fp8bs.NORM_LAYER
    assert f(P, 0, 128, 128, P, None, R, 1e-6, P, 128, P, None, None, None) == fp8bs.OK      # M = 0
    assert f(P, -1, 128, 128, P, None, R, 1e-6, P, 128, P, None, None, None) == fp8bs.ERR_INVALID_ARG
    assert f(P, 4, 100, 128, P, None, R, 1e-6, P, 128, P, None, None, None) == fp8bs.ERR_UNSUPPORTED
    assert f(P, 4, 65536 + 128, 65536 + 128, P, None, R, 1e-6, P, 65536 + 128, P, None, None,
             None) == fp8bs.ERR_UNSUPPORTED                                                 # K too large
    assert f(P, 4, 0, 0, P, None, R, 1e-6, P, 0, P, None, None, None) == fp8bs.ERR_INVALID_ARG  # K = 0
    assert f(P, 4, 128, 128, P, None, 2, 1e-6, P, 128, P, None, None, None) == fp8bs.ERR_INVALID_ARG  # kind
    assert f(P, 4, 128, 128, P, None, L_, -1.0, P, 128, P, None, None, None) == fp8bs.ERR_INVALID_ARG  # eps
    assert f(P, 4, 128, 128, P, None, L_, float("nan"), P, 128, P, None, None,
             None) == fp8bs.ERR_INVALID_ARG
    assert f(P, 4, 128, 128, None, None, R, 1e-6, P, 128, P, None, None, None) == fp8bs.ERR_INVALID_ARG  # gamma
    assert f(P, 4, 128, 128, P, P + 8, R, 1e-6, P, 128, P, None, None, None) == fp8bs.ERR_INVALID_ARG  # beta align
    assert f(P, 4, 128, 128, P, None, R, 1e-6, P, 128, P, P + 2, None, None) == fp8bs.ERR_INVALID_ARG  # mean align
    assert f(P, 4, 128, 120, P, None, R, 1e-6, P, 128, P, None, None, None) == fp8bs.ERR_INVALID_ARG  # ldx < K


def test_bf16_act_gemm_argument_checks():
    f = fp8bs.lib().fp8bs_gemm_bf16_act
    assert f(P, 128, P, P, P, 1, 0, 256, 128, 256, None) == fp8bs.OK                   # M = 0
    assert f(P, 128, P, P, P, 1, -1, 256, 128, 256, None) == fp8bs.ERR_INVALID_ARG
    assert f(P, 128, P, P, P, 1, 4, 200, 128, 200, None) == fp8bs.ERR_UNSUPPORTED     # N % 128
    assert f(P, 100, P, P, P, 1, 4, 256, 100, 256, None) == fp8bs.ERR_UNSUPPORTED     # K % 128
    assert f(P, 120, P, P, P, 1, 4, 256, 128, 256, None) == fp8bs.ERR_INVALID_ARG     # lda < K
    assert f(P, 132, P, P, P, 1, 4, 256, 128, 256, None) == fp8bs.ERR_INVALID_ARG     # row not 16B
    assert f(P + 8, 128, P, P, P, 1, 4, 256, 128, 256, None) == fp8bs.ERR_INVALID_ARG  # misaligned
    assert f(None, 128, P, P, P, 1, 4, 256, 128, 256, None) == fp8bs.ERR_INVALID_ARG
    assert f(P, 128, P, None, P, 1, 4, 256, 128, 256, None) == fp8bs.ERR_INVALID_ARG  # sw
    g = fp8bs.lib().fp8bs_grouped_gemm_bf16_act
    assert g(P, 128, P, 2, 0, P, P, P, 1, 256, 128, 256, None) == fp8bs.OK             # no rows
    assert g(P, 128, P, 0, 10, P, P, P, 1, 256, 128, 256, None) == fp8bs.ERR_INVALID_ARG
    assert g(P, 128, P, 513, 10, P, P, P, 1, 256, 128, 256, None) == fp8bs.ERR_UNSUPPORTED
    assert g(P, 128, P + 2, 2, 10, P, P, P, 1, 256, 128, 256, None) == fp8bs.ERR_INVALID_ARG


def test_pair_quantize_argument_checks():
    f = fp8bs.lib().fp8bs_quantize_act_and_weight
    assert f(P, 0, 128, 128, P, 128, P, P, 0, 128, 128, P, 128, P, None) == fp8bs.OK       # both empty
    assert f(P, -1, 128, 128, P, 128, P, P, 4, 128, 128, P, 128, P, None) == fp8bs.ERR_INVALID_ARG
    assert f(P, 4, 100, 128, P, 128, P, P, 4, 128, 128, P, 128, P, None) == fp8bs.ERR_UNSUPPORTED
    assert f(P, 4, 128, 128, P, 128, P, P, 4, 130, 130, P, 130, P, None) == fp8bs.ERR_UNSUPPORTED
    assert f(None, 4, 128, 128, P, 128, P, P, 4, 128, 128, P, 128, P, None) == fp8bs.ERR_INVALID_ARG
    assert f(P, 4, 128, 128, P, 128, P, P, 4, 128, 128, None, 128, P, None) == fp8bs.ERR_INVALID_ARG
    assert f(P, 4, 128, 120, P, 128, P, P, 4, 128, 128, P, 128, P, None) == fp8bs.ERR_INVALID_ARG
    assert f(P, 4, 128, 128, P, 128, P + 2, P, 4, 128, 128, P, 128, P, None) == fp8bs.ERR_INVALID_ARG


def test_pow2_quantize_argument_checks():
    L = fp8bs.lib()
    for f in (L.fp8bs_quantize_act_1x128_pow2, L.fp8bs_quantize_weight_128x128_pow2):
        assert f(P, 0, 128, 128, P, 128, P, None) == fp8bs.OK
        assert f(P, -1, 128, 128, P, 128, P, None) == fp8bs.ERR_INVALID_ARG
        assert f(P, 4, 100, 128, P, 128, P, None) == fp8bs.ERR_UNSUPPORTED
        assert f(None, 4, 128, 128, P, 128, P, None) == fp8bs.ERR_INVALID_ARG
        assert f(P + 8, 4, 128, 128, P, 128, P, None) == fp8bs.ERR_INVALID_ARG
