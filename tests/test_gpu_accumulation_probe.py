"""How many bits the FP8 tensor-core accumulation keeps inside one 128-K chunk
on this GPU (outputs only).

The pages report that H800's FP8 MMA keeps about 14 bits when accumulating,
which is why partial sums are promoted to FP32 at a fixed K interval ("How
Google Is Changing How We Method Deepseek", paragraph on limited
accumulation bit width; "personal notes concerning the deepseek core
readings", paragraph on accumulation precision). Here each probe row r holds
one product 2^8 (16 x 16) and 31 products 2^-s (s = r), either in the same
32-wide K block as the big one (one MMA instruction) or in the next block
(a later MMA into the same TMEM accumulator). With unit scales the GEMM's
FP32 output is the chunk's raw tensor-core partial. Any binary32 summation
order gives exactly 256 + 31 * 2^-s for s <= 15, so a partial that differs
from it there shows the accumulator keeping fewer bits. Measured on B300: exact
for every s < 16 (23 bits below the big product), in one MMA and across MMAs,
i.e. binary32-grade; at 24 bits below, the partial is truncated (15 instead of
the round-to-nearest 16 units). The assertion is that binary32-grade
profile; the promotion interval (one 128-K chunk) is then set by the scale
groups alone."""
import numpy as np
import pytest
import torch

from fp8_fine_grained_17_b300 import fp8bs

pytestmark = pytest.mark.gpu


def _code_pow2(e: int) -> int:
    """E4M3 code of 2^e (normal for e >= -6, subnormal m * 2^-9 below)."""
    return ((e + 7) << 3) if e >= -6 else (1 << (e + 9))


def _probe(same_block: bool):
    """Output (r, n), r, n = 0..9, sums 16*16 + 31 * (2^-r * 2^-n): the
    small-product exponent is s = r + n (0..18)."""
    M, N, K = 128, 128, 128
    qa = np.zeros((M, K), np.uint8)
    qw = np.zeros((N, K), np.uint8)
    lo, hi = (1, 32) if same_block else (32, 63)
    for i in range(10):
        qa[i, 0] = _code_pow2(4)
        qw[i, 0] = _code_pow2(4)
        qa[i, lo:hi] = _code_pow2(-i)
        qw[i, lo:hi] = _code_pow2(-i)
    sa = torch.ones((M, K // 128), dtype=torch.float32, device="cuda")
    sw = torch.ones((N // 128, K // 128), dtype=torch.float32, device="cuda")
    c = fp8bs.gemm(torch.from_numpy(qa).cuda(), sa, torch.from_numpy(qw).cuda(), sw, torch.float32)
    assert fp8bs.fp8bs_last_device_error() == fp8bs.OK
    got = c[:10, :10].double().cpu().numpy()
    r, n = np.meshgrid(np.arange(10), np.arange(10), indexing="ij")
    S = r + n
    exact = 256.0 + 31.0 * np.exp2(-S.astype(np.float64))
    return S.ravel(), got.ravel(), exact.ravel()


@pytest.mark.parametrize("same_block", [True, False])
def test_accumulation_bits(same_block, capsys):
    S, got, exact = _probe(same_block)
    exact_at = {int(s): bool(np.all(got[S == s] == exact[S == s])) for s in np.unique(S)}
    first_loss = next((s for s, ok in sorted(exact_at.items()) if not ok), None)
    with capsys.disabled():
        where = "one MMA (same 32-wide K block)" if same_block else "two MMAs (next K block)"
        msg = f"\n{where}: 256 + 31*2^-s exact for s < {first_loss}" if first_loss is not None \
            else f"\n{where}: exact for every s <= 18"
        if first_loss is not None:
            i = int(np.flatnonzero(S == first_loss)[0])
            msg += (f"; at s = {first_loss} ({8 + first_loss} bits below the big product) "
                    f"got {got[i]!r}, exact {exact[i]!r}")
        print(msg)
    assert all(exact_at[s] for s in exact_at if s <= 15)
