"""Failure detection on the GPU without a fault.

Every wait of the GEMM kernels is bounded. The test-only injection makes the
producer of the first CTA leave out the copies of one K chunk and shortens
the waits to 20 ms, so the waits for that chunk run out (a barrier that
nothing completes). The kernel must report FP8BS_ERR_TIMEOUT through
fp8bs_last_device_error, write nothing outside C, finish every other tile
correctly, and leave the device usable: the next normal call is correct."""
import time

import numpy as np
import pytest
import torch

from fp8_fine_grained_17_b300 import fp8bs
from fp8_fine_grained_17_b300 import workloads as wl
from helpers import check_gemm, gpu_quant_act, gpu_quant_weight, to_dev_bf16

pytestmark = pytest.mark.gpu

M, N, K = 256, 512, 1024          # 8 K chunks; every CTA takes one tile
STALL_CHUNK = 3
WAIT_NS = 20_000_000
SENTINEL = -5.0

# Rows and columns of the tile the first CTA (or CTA pair) owns.
FIRST_TILE = {
    fp8bs.TILE_128x256: (128, 256),
    fp8bs.TILE_128x128: (128, 128),
    fp8bs.TILE_PAIR_256x256: (256, 256),
    fp8bs.TILE_PAIR_256x128: (256, 128),
    "fused": (128, 256),
}
CASES = [(t, torch.float32) for t in FIRST_TILE] + [
    (t, torch.bfloat16) for t in (fp8bs.TILE_PAIR_256x256, fp8bs.TILE_PAIR_256x128)]


def _inputs():
    rng = np.random.default_rng(99)
    a = wl.bf16_bits(rng.standard_normal((M, K)).astype(np.float32))
    w = wl.bf16_bits((rng.standard_normal((N, K)) * 0.02).astype(np.float32))
    return a, w


def _launch(tile, a_bits, qa, sa, qw, sw, c):
    if tile == "fused":
        fp8bs.fp8bs_gemm_bf16_act(to_dev_bf16(a_bits), qw, sw, c)
    else:
        fp8bs.fp8bs_gemm(qa, sa, qw, sw, c, None, tile)


@pytest.mark.parametrize("tile,out", CASES)
def test_stalled_chunk_times_out_and_device_recovers(orc, tile, out):
    """One CTA's producer leaves a chunk's copies out: its waits give up,
    the launch reports TIMEOUT, nothing outside C is written, every other
    tile is correct (bf16 output of a pair: written by TMA stores, which the
    CTAs wait for before they exit) and the next launch is correct."""
    a_bits, w_bits = _inputs()
    qa, sa = gpu_quant_act(a_bits)
    qw, sw = gpu_quant_weight(w_bits)
    C_or, B = orc.gemm(*orc.quantize_act_1x128(a_bits), *orc.quantize_weight_128x128(w_bits))
    assert fp8bs.fp8bs_last_device_error() == fp8bs.OK

    # Output inside a guarded buffer: a row above, a row below, 64 columns right.
    buf = torch.full((M + 2, N + 64), SENTINEL, dtype=out, device="cuda")
    c = buf[1:M + 1, :N]
    fp8bs.fp8bs_test_inject_stall(STALL_CHUNK, WAIT_NS)
    try:
        t0 = time.perf_counter()
        _launch(tile, a_bits, qa, sa, qw, sw, c)
        status = fp8bs.fp8bs_last_device_error()
        elapsed = time.perf_counter() - t0
    finally:
        fp8bs.fp8bs_test_inject_stall(-1, 0)
    assert status == fp8bs.ERR_TIMEOUT, fp8bs.status_string(status)
    assert elapsed < 5.0, f"the stalled launch took {elapsed:.2f} s"
    assert fp8bs.fp8bs_last_device_error() == fp8bs.OK        # cleared by the read

    # Nothing outside C was written.
    assert torch.all(buf[0] == SENTINEL) and torch.all(buf[M + 1] == SENTINEL)
    assert torch.all(buf[:, N:] == SENTINEL)
    # Every tile except the first CTA's is complete and correct.
    tr, tc = FIRST_TILE[tile]
    got = c.float().cpu().numpy().astype(np.float64)
    mask = np.ones((M, N), bool)
    mask[:tr, :tc] = False
    tol = 2e-5 * B + 1e-6
    if out == torch.bfloat16:
        tol = tol + np.abs(C_or) * 2.0 ** -8
    assert np.all(np.abs(got - C_or)[mask] <= tol[mask])

    # The device is usable: the same call without the injection is correct.
    c2 = torch.full((M, N), SENTINEL, dtype=out, device="cuda")
    _launch(tile, a_bits, qa, sa, qw, sw, c2)
    assert fp8bs.fp8bs_last_device_error() == fp8bs.OK
    check_gemm(c2, C_or, B, out == torch.bfloat16)


def test_injection_arguments_checked():
    assert fp8bs.lib().fp8bs_test_inject_stall(0, 10) == fp8bs.ERR_INVALID_ARG
    assert fp8bs.lib().fp8bs_test_inject_stall(1 << 40, WAIT_NS) == fp8bs.ERR_INVALID_ARG
    assert fp8bs.lib().fp8bs_test_inject_stall(-1, 0) == fp8bs.OK


@pytest.mark.parametrize("out", [torch.float32, torch.bfloat16])
def test_stall_in_a_launch_that_splits_its_last_wave(orc, out):
    """The same injection in a launch that hands partial tiles over through a
    workspace: 4096 x 1280 x 4096 on CTA pairs is 80 tiles on 74 pairs, so the
    last 6 tiles are each split into 2 K ranges (units 0-11). Unit 0 takes tile
    0 and then owns tile 74 (rows 2560-2815, columns 1024-1279); its stalled
    chunk in tile 0 leaves both unfinished, while unit 1 still hands its range of
    tile 74 over. TIMEOUT is reported, nothing outside C is written, every
    other tile is correct, and the next launch with the same workspace (a new
    epoch, so the stale flag cannot match) is correct."""
    M_, N_, K_ = 4096, 1280, 4096
    tile = fp8bs.TILE_PAIR_256x256
    rng = np.random.default_rng(123)
    a_bits = wl.bf16_bits(rng.standard_normal((M_, K_)).astype(np.float32))
    w_bits = wl.bf16_bits((rng.standard_normal((N_, K_)) * 0.02).astype(np.float32))
    qa, sa = gpu_quant_act(a_bits)
    qw, sw = gpu_quant_weight(w_bits)
    C_or, B = orc.gemm(*orc.quantize_act_1x128(a_bits), *orc.quantize_weight_128x128(w_bits))
    nbytes = fp8bs.fp8bs_gemm_workspace_size(M_, N_, K_, tile)
    assert nbytes > 0, "this shape is meant to split its last wave"
    ws = torch.zeros(nbytes, dtype=torch.uint8, device="cuda")
    assert fp8bs.fp8bs_last_device_error() == fp8bs.OK

    buf = torch.full((M_ + 2, N_ + 64), SENTINEL, dtype=out, device="cuda")
    c = buf[1:M_ + 1, :N_]
    fp8bs.fp8bs_test_inject_stall(STALL_CHUNK, WAIT_NS)
    try:
        t0 = time.perf_counter()
        fp8bs.fp8bs_gemm_ws(qa, sa, qw, sw, c, ws, None, tile)
        status = fp8bs.fp8bs_last_device_error()
        elapsed = time.perf_counter() - t0
    finally:
        fp8bs.fp8bs_test_inject_stall(-1, 0)
    assert status == fp8bs.ERR_TIMEOUT, fp8bs.status_string(status)
    assert elapsed < 5.0, f"the stalled launch took {elapsed:.2f} s"
    assert fp8bs.fp8bs_last_device_error() == fp8bs.OK

    assert torch.all(buf[0] == SENTINEL) and torch.all(buf[M_ + 1] == SENTINEL)
    assert torch.all(buf[:, N_:] == SENTINEL)
    got = c.float().cpu().numpy().astype(np.float64)
    mask = np.ones((M_, N_), bool)
    mask[0:256, 0:256] = False            # tile 0
    mask[2560:2816, 1024:1280] = False    # tile 74, owned by unit 0
    tol = 2e-5 * B + 1e-6
    if out == torch.bfloat16:
        tol = tol + np.abs(C_or) * 2.0 ** -8
    assert np.all(np.abs(got - C_or)[mask] <= tol[mask])

    c2 = torch.full((M_, N_), SENTINEL, dtype=out, device="cuda")
    fp8bs.fp8bs_gemm_ws(qa, sa, qw, sw, c2, ws, None, tile)
    assert fp8bs.fp8bs_last_device_error() == fp8bs.OK
    check_gemm(c2, C_or, B, out == torch.bfloat16)
