"""GEMMs with the 1x128 activation quantization inside the kernel.

Two checks: parity with the float64 oracle (the oracle's 1x128 quantizer
followed by its GEMM, the statement of the problem's bound), and bit-identity
with the unfused GPU path (quantizer kernel, then the 128 x 256 GEMM): the
fused kernel must use the same codes and scales and the same promotion order."""
import numpy as np
import pytest
import torch

from fp8_fine_grained_17_b300 import fp8bs
from fp8_fine_grained_17_b300 import workloads as wl
from helpers import check_gemm, gpu_quant_weight, to_dev_bf16

pytestmark = pytest.mark.gpu


def _dense(M, N, K, seed, outliers=None):
    rng = np.random.default_rng(seed)
    a, _ = wl.activations(rng, M, K, outliers)
    w = wl.weights(rng, N, K)
    return a, w


def _unfused(a_dev, qw, sw, out):
    qa, sa = fp8bs.quantize_act(a_dev)
    return fp8bs.gemm(qa, sa, qw, sw, out, tile=fp8bs.TILE_128x256)


@pytest.mark.parametrize("M,N,K", [
    (1, 256, 128), (5, 256, 256), (127, 512, 384), (129, 384, 512), (300, 640, 1024),
    (513, 256, 640), (128, 256, 4096), (640, 1280, 1152),
])
@pytest.mark.parametrize("out", [torch.float32, torch.bfloat16])
def test_fused_matches_oracle_and_unfused(orc, M, N, K, out):
    a_bits, w_bits = _dense(M, N, K, seed=M * 7 + N + K, outliers=50.0)
    a = to_dev_bf16(a_bits)
    qw, sw = gpu_quant_weight(w_bits)
    c = fp8bs.gemm_bf16_act(a, qw, sw, out)
    torch.cuda.synchronize()
    assert fp8bs.fp8bs_last_device_error() == fp8bs.OK
    ref = _unfused(a, qw, sw, out)
    assert torch.equal(c.view(torch.int32 if out == torch.float32 else torch.int16),
                       ref.view(torch.int32 if out == torch.float32 else torch.int16))
    qa_o, sa_o = orc.quantize_act_1x128(a_bits)
    qw_o, sw_o = orc.quantize_weight_128x128(w_bits)
    C_or, B = orc.gemm(qa_o, sa_o, qw_o, sw_o)
    check_gemm(c, C_or, B, out == torch.bfloat16)


def _random_fused_cases(n=8, seed=5):
    rng = np.random.default_rng(seed)
    return [(int(rng.choice([1, 63, 128, 257, 700, 1500])), 128 * int(rng.integers(1, 17)),
             128 * int(rng.choice([1, 3, 10, 24])),
             torch.bfloat16 if rng.random() < 0.6 else torch.float32) for _ in range(n)]


@pytest.mark.parametrize("M,N,K,out", _random_fused_cases())
def test_fused_random_shapes(orc, M, N, K, out):
    """Seeded shapes through the same two checks."""
    test_fused_matches_oracle_and_unfused(orc, M, N, K, out)


def test_fused_strided_activations(orc):
    M, N, K = 200, 512, 768
    a_bits, w_bits = _dense(M, N, K, seed=11)
    buf = torch.zeros((M, K + 64), dtype=torch.bfloat16, device="cuda")
    buf[:, :K] = to_dev_bf16(a_bits)
    a = buf[:, :K]
    qw, sw = gpu_quant_weight(w_bits)
    c = fp8bs.gemm_bf16_act(a, qw, sw, torch.float32)
    ref = _unfused(a.contiguous(), qw, sw, torch.float32)
    assert torch.equal(c, ref)
    qa_o, sa_o = orc.quantize_act_1x128(a_bits)
    qw_o, sw_o = orc.quantize_weight_128x128(w_bits)
    C_or, B = orc.gemm(qa_o, sa_o, qw_o, sw_o)
    check_gemm(c, C_or, B, False)


def test_fused_zero_and_tiny_groups(orc):
    # All-zero groups (scale 1) and groups with amax below 2^-100 (the exact
    # division path of the codec) inside the kernel.
    M, N, K = 64, 256, 512
    a_bits, w_bits = _dense(M, N, K, seed=12)
    a = wl.bits_to_f32(a_bits).copy()
    a[:8, :] = 0.0
    a[8:16, 128:256] *= np.float32(2.0 ** -110)
    a_bits = wl.bf16_bits(a)
    dev = to_dev_bf16(a_bits)
    qw, sw = gpu_quant_weight(w_bits)
    c = fp8bs.gemm_bf16_act(dev, qw, sw, torch.float32)
    assert torch.equal(c, _unfused(dev, qw, sw, torch.float32))
    qa_o, sa_o = orc.quantize_act_1x128(a_bits)
    qw_o, sw_o = orc.quantize_weight_128x128(w_bits)
    C_or, B = orc.gemm(qa_o, sa_o, qw_o, sw_o)
    check_gemm(c, C_or, B, False)


@pytest.mark.parametrize("counts,N,K", [
    ([3, 0, 5, 1], 256, 256),
    ([130, 1, 0, 257, 64], 384, 512),
    ([0, 128, 0], 640, 256),
])
def test_fused_grouped(orc, counts, N, K):
    d = wl.moe(seed=sum(counts) + N + 5, N=N, K=K, counts=counts)
    E = len(counts)
    a = to_dev_bf16(d.a_bits)
    qw, sw = gpu_quant_weight(d.w_bits.reshape(E * N, K))
    qw, sw = qw.view(E, N, K), sw.view(E, N // 128, K // 128)
    off = torch.from_numpy(d.offsets).cuda()
    c = fp8bs.grouped_gemm_bf16_act(a, off, qw, sw, torch.bfloat16)
    assert fp8bs.fp8bs_last_device_error() == fp8bs.OK
    qa, sa = fp8bs.quantize_act(a)
    ref = fp8bs.grouped_gemm(qa, sa, off, qw, sw, torch.bfloat16, tile=fp8bs.TILE_128x256)
    assert torch.equal(c.view(torch.int16), ref.view(torch.int16))
    qa_o, sa_o = orc.quantize_act_1x128(d.a_bits)
    q_o, s_o = orc.quantize_weight_128x128(d.w_bits.reshape(E * N, K))
    C_or, B = orc.grouped_gemm(qa_o, sa_o, d.offsets, q_o.reshape(E, N, K), s_o.reshape(E, N // 128, K // 128))
    check_gemm(c, C_or, B, True)


@pytest.mark.slow
def test_fused_full_size(orc):
    # The benchmarked GEMM, 4096 x 4096 x 7168, bf16 out: every output
    # element against the float64 oracle (the oracle's quantizers, then its
    # GEMM) and bit for bit against the unfused GPU path.
    d = wl.cfg3(0)
    a = to_dev_bf16(d.a_bits)
    qw, sw = gpu_quant_weight(d.w_bits)
    c = fp8bs.gemm_bf16_act(a, qw, sw, torch.bfloat16)
    ref = _unfused(a, qw, sw, torch.bfloat16)
    assert fp8bs.fp8bs_last_device_error() == fp8bs.OK
    assert torch.equal(c.view(torch.int16), ref.view(torch.int16))
    qa_o, sa_o = orc.quantize_act_1x128(d.a_bits)
    qw_o, sw_o = orc.quantize_weight_128x128(d.w_bits)
    C_or, B = orc.gemm(qa_o, sa_o, qw_o, sw_o)
    check_gemm(c, C_or, B, True)


@pytest.mark.slow
def test_fused_moe_workload(orc):
    # The MoE workload (32 experts, N=4096, K=7168, seeded top-8 routing of
    # 8192 tokens): every output element against the float64 oracle and bit
    # for bit against the unfused GPU path.
    d = wl.moe(seed=0)
    E, N, K = 32, 4096, 7168
    a = to_dev_bf16(d.a_bits)
    qw, sw = gpu_quant_weight(d.w_bits.reshape(E * N, K))
    qw, sw = qw.view(E, N, K), sw.view(E, N // 128, K // 128)
    off = torch.from_numpy(d.offsets).cuda()
    c = fp8bs.grouped_gemm_bf16_act(a, off, qw, sw, torch.bfloat16)
    qa, sa = fp8bs.quantize_act(a)
    ref = fp8bs.grouped_gemm(qa, sa, off, qw, sw, torch.bfloat16, tile=fp8bs.TILE_128x256)
    assert fp8bs.fp8bs_last_device_error() == fp8bs.OK
    assert torch.equal(c.view(torch.int16), ref.view(torch.int16))
    del qa, sa, qw, sw, ref
    qa_o, sa_o = orc.quantize_act_1x128(d.a_bits)
    qw_o, sw_o = orc.quantize_weight_128x128(d.w_bits.reshape(E * N, K))
    C_or, B = orc.grouped_gemm(qa_o, sa_o, d.offsets, qw_o.reshape(E, N, K), sw_o.reshape(E, N // 128, K // 128))
    check_gemm(c, C_or, B, True)
