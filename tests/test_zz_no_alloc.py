"""The allocation-free GEMM entry point (fp8bs_gemm_noalloc).

It exists for callers that cannot allocate device memory where they call the
GEMM (an allocator callback that must not re-enter the allocator, a plug-in
that may not own device memory): its workspace is a fixed array in the
library's own device memory, shared by every call on the device. Checked
here through the C ABI: two calls in a row give the output of the
workspace-taking entry point fp8bs_gemm_ws (bit for bit: same split, same
sums) and are within the oracle's bound; a shape whose split needs more than
the fixed array is refused before anything runs. This file is collected last
so that a run stopping at its first failure has run every other test."""
import ctypes

import numpy as np
import pytest
import torch

from fp8_fine_grained_17_b300 import fp8bs
from fp8_fine_grained_17_b300 import workloads as wl
from helpers import check_gemm, gpu_quant_act, gpu_quant_weight

pytestmark = pytest.mark.gpu


def _call_noalloc(qa, sa, qw, sw, c, tile):
    """Straight through the C entry point (no Python-side allocation)."""
    M, K = qa.shape
    N = qw.shape[0]
    return fp8bs.lib().fp8bs_gemm_noalloc(
        qa.data_ptr(), sa.data_ptr(), qw.data_ptr(), sw.data_ptr(), c.data_ptr(), fp8bs.OUT_BF16,
        M, N, K, c.stride(0), int(tile), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


@pytest.mark.parametrize("M,N,K,tile", [(2048, 3328, 4096, fp8bs.TILE_PAIR_256x256),
                                        (1024, 5888, 4096, fp8bs.TILE_128x256)])
def test_noalloc_matches_workspace_entry_point_twice(orc, M, N, K, tile):
    rng = np.random.default_rng(M + N + 17)
    a = wl.bf16_bits(rng.standard_normal((M, K)).astype(np.float32))
    w = wl.bf16_bits((rng.standard_normal((N, K)) * 0.02).astype(np.float32))
    qa, sa = gpu_quant_act(a)
    qw, sw = gpu_quant_weight(w)
    need = fp8bs.fp8bs_gemm_workspace_size(M, N, K, tile)
    assert 0 < need <= fp8bs.NOALLOC_SCRATCH_BYTES, "the shape is meant to use the scratch"
    ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
    ref = fp8bs.gemm_ws(qa, sa, qw, sw, ws, torch.bfloat16, tile=tile)
    assert fp8bs.fp8bs_last_device_error() == fp8bs.OK
    C_or, B = orc.gemm(*orc.quantize_act_1x128(a), *orc.quantize_weight_128x128(w))
    check_gemm(ref, C_or, B, True)
    for call in range(2):
        c = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
        assert _call_noalloc(qa, sa, qw, sw, c, tile) == fp8bs.OK
        assert fp8bs.fp8bs_last_device_error() == fp8bs.OK
        check_gemm(c, C_or, B, True)
        assert torch.equal(c.view(torch.int16), ref.view(torch.int16)), f"call {call}"


def test_noalloc_without_split_matches_plain_gemm():
    # A shape that does not split uses no scratch: exactly fp8bs_gemm.
    g = torch.Generator(device="cuda")
    g.manual_seed(5)
    M, N, K = 512, 1024, 1024
    qa = torch.randint(0, 0x7E, (M, K), dtype=torch.uint8, device="cuda", generator=g)
    qw = torch.randint(0, 0x7E, (N, K), dtype=torch.uint8, device="cuda", generator=g)
    sa = torch.rand((M, K // 128), device="cuda", generator=g) * 1e-2
    sw = torch.rand((N // 128, K // 128), device="cuda", generator=g) * 1e-2
    assert fp8bs.fp8bs_gemm_workspace_size(M, N, K) == 0
    c = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    for _ in range(2):
        assert _call_noalloc(qa, sa, qw, sw, c, fp8bs.TILE_AUTO) == fp8bs.OK
        assert fp8bs.fp8bs_last_device_error() == fp8bs.OK
        assert torch.equal(c, fp8bs.gemm(qa, sa, qw, sw, torch.bfloat16))


def test_noalloc_rejects_a_split_larger_than_the_scratch():
    # 896 x 39680 x 6144 with 128x256 tiles: 1085 tiles on 148 CTAs leave 49
    # tiles, cut in 3 pieces: 98 partial tiles of 128 KB, more than 12 MiB.
    # Refused before any launch (real-size operands all the same).
    M, N, K, tile = 896, 39680, 6144, fp8bs.TILE_128x256
    need = fp8bs.fp8bs_gemm_workspace_size(M, N, K, tile)
    if need <= fp8bs.NOALLOC_SCRATCH_BYTES:
        pytest.skip(f"on this GPU the split needs only {need} bytes")
    qa = torch.zeros((M, K), dtype=torch.uint8, device="cuda")
    sa = torch.ones((M, K // 128), dtype=torch.float32, device="cuda")
    qw = torch.zeros((N, K), dtype=torch.uint8, device="cuda")
    sw = torch.ones((N // 128, K // 128), dtype=torch.float32, device="cuda")
    c = torch.full((M, N), 3.0, dtype=torch.bfloat16, device="cuda")
    assert _call_noalloc(qa, sa, qw, sw, c, tile) == fp8bs.ERR_UNSUPPORTED
    torch.cuda.synchronize()
    assert torch.all(c == 3.0).item()
