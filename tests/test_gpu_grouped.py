"""GPU parity of the grouped (MoE up-projection) GEMM against the oracle."""
import numpy as np
import pytest
import torch

from fp8_fine_grained_17_b300 import fp8bs
from fp8_fine_grained_17_b300 import workloads as wl
from helpers import check_codes, check_gemm, gpu_quant_act, gpu_quant_weight

pytestmark = pytest.mark.gpu


def _quant_experts(orc, w_bits, check=True):
    """Per-expert weight quantization on the GPU as one [E*N, K] call."""
    E, N, K = w_bits.shape
    qw, sw = gpu_quant_weight(w_bits.reshape(E * N, K))
    if check:
        q_o, s_o = orc.quantize_weight_128x128(w_bits.reshape(E * N, K))
        check_codes(qw, sw, q_o, s_o)
    return qw.view(E, N, K), sw.view(E, N // 128, K // 128)


@pytest.mark.parametrize("counts,N,K", [
    ([3, 0, 5, 1], 128, 256),
    ([0, 0, 0, 200], 256, 384),
    ([130, 1, 0, 257, 64], 384, 512),
    ([1], 128, 128),
    ([0, 128, 0], 640, 256),
])
@pytest.mark.parametrize("out", [torch.float32, torch.bfloat16])
def test_grouped_small(orc, counts, N, K, out):
    d = wl.moe(seed=sum(counts) + N, N=N, K=K, counts=counts)
    qa, sa = gpu_quant_act(d.a_bits)
    qa_o, sa_o = orc.quantize_act_1x128(d.a_bits)
    check_codes(qa, sa, qa_o, sa_o)
    qw, sw = _quant_experts(orc, d.w_bits)
    off = torch.from_numpy(d.offsets).cuda()
    c = fp8bs.grouped_gemm(qa, sa, off, qw, sw, out)
    assert fp8bs.fp8bs_last_device_error() == fp8bs.OK
    E, N, K = d.w_bits.shape
    q_o, s_o = orc.quantize_weight_128x128(d.w_bits.reshape(E * N, K))
    C_or, B = orc.grouped_gemm(qa_o, sa_o, d.offsets, q_o.reshape(E, N, K),
                               s_o.reshape(E, N // 128, K // 128))
    check_gemm(c, C_or, B, out == torch.bfloat16)


@pytest.mark.parametrize("tile", [fp8bs.TILE_AUTO, fp8bs.TILE_PAIR_256x256])
@pytest.mark.parametrize("out", [torch.float32, torch.bfloat16])
def test_rows_outside_experts_untouched(orc, tile, out):
    """offsets[E] < total_M: trailing rows are not written. With bf16
    output a pair stores whole 32-row boxes by TMA and writes a box that runs
    past an expert's end (rows 64-95 and 102-133 here) row by row."""
    d = wl.moe(seed=9, N=256, K=256, counts=[70, 40])
    extra = 30
    a_bits = np.concatenate([d.a_bits, d.a_bits[:extra]])
    qa, sa = gpu_quant_act(a_bits)
    qw, sw = _quant_experts(orc, d.w_bits, check=False)
    c = torch.full((a_bits.shape[0], 256), 5.0, dtype=out, device="cuda")
    fp8bs.fp8bs_grouped_gemm(qa, sa, torch.from_numpy(d.offsets).cuda(), qw, sw, c, tile=tile)
    torch.cuda.synchronize()
    assert fp8bs.fp8bs_last_device_error() == fp8bs.OK
    assert torch.all(c[110:] == 5.0)
    q_o, s_o = orc.quantize_act_1x128(a_bits[:110])
    wq, ws = orc.quantize_weight_128x128(d.w_bits.reshape(-1, 256))
    C_or, B = orc.grouped_gemm(q_o, s_o, d.offsets, wq.reshape(2, 256, 256), ws.reshape(2, 2, 2))
    check_gemm(c[:110], C_or, B, out == torch.bfloat16)


def test_bad_offsets_reported(orc):
    """Decreasing offsets: nothing is written and the device error says so."""
    d = wl.moe(seed=10, N=128, K=128, counts=[10, 10])
    qa, sa = gpu_quant_act(d.a_bits)
    qw, sw = _quant_experts(orc, d.w_bits, check=False)
    c = torch.full((20, 128), 2.0, dtype=torch.float32, device="cuda")
    bad = torch.tensor([0, 15, 12], dtype=torch.int32, device="cuda")
    fp8bs.fp8bs_grouped_gemm(qa, sa, bad, qw, sw, c)
    assert fp8bs.fp8bs_last_device_error() == fp8bs.ERR_INVALID_ARG
    assert torch.all(c == 2.0)
    assert fp8bs.fp8bs_last_device_error() == fp8bs.OK      # cleared by the read


@pytest.mark.slow
@pytest.mark.parametrize("n_tokens", [wl.N_TOKENS, 256])
def test_moe_full_workload(orc, n_tokens):
    """32 experts, N=4096, K=7168, rows from the seeded top-8 router over
    8192 tokens (prefill) or 256 (a decode batch: a few rows per expert).
    Every code and scale of both quantizations against the oracle, then every
    output element of the grouped GEMM against the float64 oracle."""
    d = wl.moe(seed=0, counts=wl.moe_routing(0, n_tokens=n_tokens))
    E, N, K = d.w_bits.shape
    qa, sa = gpu_quant_act(d.a_bits)
    qw, sw = gpu_quant_weight(d.w_bits.reshape(E * N, K))
    off = torch.from_numpy(d.offsets).cuda()
    c = fp8bs.grouped_gemm(qa, sa, off, qw.view(E, N, K), sw.view(E, N // 128, K // 128))
    assert fp8bs.fp8bs_last_device_error() == fp8bs.OK
    qa_o, sa_o = orc.quantize_act_1x128(d.a_bits)
    check_codes(qa, sa, qa_o, sa_o)
    del qa, sa
    qw_o, sw_o = orc.quantize_weight_128x128(d.w_bits.reshape(E * N, K))
    check_codes(qw, sw, qw_o, sw_o)
    del qw, sw
    C_or, B = orc.grouped_gemm(qa_o, sa_o, d.offsets, qw_o.reshape(E, N, K),
                               sw_o.reshape(E, N // 128, K // 128))
    worst = check_gemm(c, C_or, B, True)
    print(f"moe {n_tokens} tokens ({int(d.offsets[-1])} rows): worst err/tol {worst:.3g}")


@pytest.mark.parametrize("tile", [fp8bs.TILE_128x256, fp8bs.TILE_128x128,
                                  fp8bs.TILE_PAIR_256x256, fp8bs.TILE_PAIR_256x128])
@pytest.mark.parametrize("out", [torch.float32, torch.bfloat16])
def test_grouped_every_tile(orc, tile, out):
    """Empty, single-row and multi-tile experts through every tile shape;
    the expert ends (300, 301, 430) fall inside 32-row store boxes."""
    counts = [0, 300, 1, 129, 0, 520]
    d = wl.moe(seed=11, N=512, K=384, counts=counts)
    qa, sa = gpu_quant_act(d.a_bits)
    qw, sw = _quant_experts(orc, d.w_bits, check=False)
    off = torch.from_numpy(d.offsets).cuda()
    c = fp8bs.grouped_gemm(qa, sa, off, qw, sw, out, tile=tile)
    assert fp8bs.fp8bs_last_device_error() == fp8bs.OK
    E, N, K = d.w_bits.shape
    qa_o, sa_o = orc.quantize_act_1x128(d.a_bits)
    q_o, s_o = orc.quantize_weight_128x128(d.w_bits.reshape(E * N, K))
    C_or, B = orc.grouped_gemm(qa_o, sa_o, d.offsets, q_o.reshape(E, N, K),
                               s_o.reshape(E, N // 128, K // 128))
    check_gemm(c, C_or, B, out == torch.bfloat16)


@pytest.mark.parametrize("fused", [False, True])
def test_grouped_max_experts(orc, fused):
    """The largest expert count the library takes (512), most experts empty or
    with a handful of rows, a few with several m-tiles; quantized operands
    and, separately, the kernel with the activation quantization inside."""
    rng = np.random.default_rng(77)
    counts = rng.choice([0, 0, 1, 2, 3], size=512)
    counts[[5, 300, 511]] = [130, 257, 64]
    N, K = 256, 256
    d = wl.moe(seed=77, N=N, K=K, counts=counts)
    E = 512
    qw, sw = _quant_experts(orc, d.w_bits, check=False)
    off = torch.from_numpy(d.offsets).cuda()
    if fused:
        c = fp8bs.grouped_gemm_bf16_act(wl.bits_to_torch(d.a_bits).cuda(), off, qw, sw, torch.float32)
    else:
        qa, sa = gpu_quant_act(d.a_bits)
        c = fp8bs.grouped_gemm(qa, sa, off, qw, sw, torch.float32)
    assert fp8bs.fp8bs_last_device_error() == fp8bs.OK
    qa_o, sa_o = orc.quantize_act_1x128(d.a_bits)
    q_o, s_o = orc.quantize_weight_128x128(d.w_bits.reshape(E * N, K))
    C_or, B = orc.grouped_gemm(qa_o, sa_o, d.offsets, q_o.reshape(E, N, K), s_o.reshape(E, N // 128, K // 128))
    check_gemm(c, C_or, B, False)


def _random_grouped_cases(n=16, seed=77):
    """Seeded expert row counts (empty experts included), tiles, output types
    and trailing rows outside every expert."""
    rng = np.random.default_rng(seed)
    tiles = [fp8bs.TILE_AUTO, fp8bs.TILE_128x256, fp8bs.TILE_128x128, fp8bs.TILE_PAIR_256x256,
             fp8bs.TILE_PAIR_256x128]
    cases = []
    for i in range(n):
        tile = tiles[i % len(tiles)]
        E = int(rng.integers(1, 9))
        counts = [int(x) if rng.random() > 0.2 else 0 for x in rng.integers(1, 400, size=E)]
        if sum(counts) == 0:
            counts[-1] = int(rng.integers(1, 400))
        nb = int(rng.integers(1, 7))
        if tile == fp8bs.TILE_PAIR_256x256 and nb % 2:
            nb += 1
        K = 128 * int(rng.choice([1, 3, 8, 16]))
        out = torch.bfloat16 if rng.random() < 0.6 else torch.float32
        extra = int(rng.choice([0, 0, 31, 100]))
        cases.append((tuple(counts), 128 * nb, K, tile, out, extra))
    return cases


@pytest.mark.parametrize("counts,N,K,tile,out,extra", _random_grouped_cases())
def test_random_grouped_against_oracle(orc, counts, N, K, tile, out, extra):
    """Every element of the experts' rows against the oracle; rows after the
    last expert keep their values; the same bits as the 128x128 tile."""
    d = wl.moe(seed=sum(counts) + N + K, N=N, K=K, counts=list(counts))
    total = int(d.offsets[-1])
    a_bits = d.a_bits if extra == 0 else np.concatenate([d.a_bits, d.a_bits[:1].repeat(extra, axis=0)])
    qa, sa = gpu_quant_act(a_bits)
    qw, sw = _quant_experts(orc, d.w_bits, check=False)
    off = torch.from_numpy(d.offsets).cuda()
    c = torch.full((total + extra, N), -3.0, dtype=out, device="cuda")
    fp8bs.fp8bs_grouped_gemm(qa, sa, off, qw, sw, c, None, tile)
    torch.cuda.synchronize()
    assert fp8bs.fp8bs_last_device_error() == fp8bs.OK
    E = len(counts)
    q_o, s_o = orc.quantize_act_1x128(a_bits[:total])
    wq, ws = orc.quantize_weight_128x128(d.w_bits.reshape(E * N, K))
    C_or, B = orc.grouped_gemm(q_o, s_o, d.offsets, wq.reshape(E, N, K), ws.reshape(E, N // 128, K // 128))
    check_gemm(c[:total], C_or, B, out == torch.bfloat16)
    assert torch.all(c[total:] == -3.0)
    ref = fp8bs.grouped_gemm(qa, sa, off, qw, sw, out, tile=fp8bs.TILE_128x128)
    assert torch.equal(c[:total], ref[:total])
