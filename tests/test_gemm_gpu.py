"""The tensor-core GEMM (sc_gemm_bf16) against exact products.

Inputs are dyadic (A on a 1/8 grid, B on a 1/64 grid, both in [-1, 1]): every
product is a multiple of 2^-9 and every partial sum of these sizes stays far
below 2^15, so FP32 accumulation is exact in any order.  The FP64 product
(numpy) is therefore the exact result: the FP32 outputs must match it bit for
bit, the bf16 output must be its round-to-nearest-even, and the reduce-add
mode must give C + A B exactly.  Shapes cover both layouts of each operand,
ragged edges in M, N and K, more tiles than SMs (each CTA cycling through both
tensor-memory accumulators) and a long K.
"""

import itertools

import numpy as np
import pytest
import torch

import precision_off_policy_gb300 as sc

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _library():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    sc.build()
    sc.lib()


def _dyadic(shape, denom, lim, gen):
    k = torch.randint(-lim, lim + 1, shape, generator=gen)
    return (k.double() / denom)


def _padded(x, dtype, fill=0.0):
    """x on the device in rows padded past a 16-byte boundary (the tensor
    copies' row alignment) by 16 more bytes, as a view of its first columns;
    the padding holds `fill`."""
    rows, cols = x.shape
    per = 16 // torch.empty((), dtype=dtype).element_size()
    buf = torch.full((rows, (cols + per - 1) // per * per + per), fill, dtype=dtype)
    buf[:, :cols] = x.to(dtype)
    return buf.cuda()[:, :cols]


def _run(M, N, K, a_kmajor, b_kmajor, c_mode, seed=0):
    gen = torch.Generator().manual_seed(seed + 1000 * M + N + 7 * K)
    A = _dyadic((M, K), 8, 8, gen)          # exact in bf16
    B = _dyadic((K, N), 64, 64, gen)
    a = _padded(A if a_kmajor else A.T, torch.bfloat16, 3.0)
    b = _padded(B.T if b_kmajor else B, torch.bfloat16, 3.0)
    exact = (A.numpy() @ B.numpy())          # FP64: exact for these inputs
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    if c_mode == sc.GEMM_BF16:
        c = _padded(torch.zeros(M, N), torch.bfloat16, 7.0)
        c.fill_(7.0)
        sc.sc_gemm_bf16(a, b, c, a_kmajor, b_kmajor, c_mode, status=status)
        want = torch.from_numpy(exact).float().to(torch.bfloat16)
        got = c.cpu()
        assert torch.equal(got.view(torch.int16), want.view(torch.int16)), \
            f"bf16 mismatch: {(got.float() - want.float()).abs().max()}"
    else:
        c0 = _dyadic((M, N), 4, 8, gen)
        c = _padded(c0 if c_mode == sc.GEMM_FP32_ADD else torch.full((M, N), 7.0), torch.float32, 7.0)
        sc.sc_gemm_bf16(a, b, c, a_kmajor, b_kmajor, c_mode, status=status)
        want = exact + (c0.numpy() if c_mode == sc.GEMM_FP32_ADD else 0.0)
        got = c.cpu().double().numpy()
        assert np.array_equal(got, want), f"FP32 mismatch: {np.abs(got - want).max()}"
    pad = c.as_strided((M, c.stride(0)), (c.stride(0), 1))[:, N:]
    assert torch.all(pad == 7.0), "the row padding past N is not written"
    torch.cuda.synchronize()
    assert int(status.item()) == 0


@pytest.mark.parametrize("a_kmajor,b_kmajor", list(itertools.product([True, False], repeat=2)))
@pytest.mark.parametrize("c_mode", [sc.GEMM_BF16, sc.GEMM_FP32, sc.GEMM_FP32_ADD])
def test_layouts_and_output_modes_with_ragged_edges(a_kmajor, b_kmajor, c_mode):
    _run(200, 300, 136, a_kmajor, b_kmajor, c_mode)


@pytest.mark.parametrize("M,N,K", [(1, 1, 1), (128, 256, 64), (129, 257, 65), (64, 8, 8), (8, 64, 200)])
def test_small_and_exact_tile_shapes(M, N, K):
    _run(M, N, K, True, True, sc.GEMM_BF16)
    _run(M, N, K, False, False, sc.GEMM_FP32)


@pytest.mark.parametrize("a_kmajor,b_kmajor", [(True, True), (True, False), (False, False)])
def test_more_tiles_than_sms(a_kmajor, b_kmajor):
    # 32 x 16 = 512 output tiles: every CTA takes several, alternating between
    # its two accumulators
    _run(4096, 4096, 192, a_kmajor, b_kmajor, sc.GEMM_BF16)


def test_long_inner_dimension():
    # the LM head's dH product has K = V = 151936
    _run(128, 256, 151936, True, False, sc.GEMM_FP32)


def test_back_to_back_calls_reuse_nothing_stale():
    for seed in range(3):
        _run(300, 520, 128, True, True, sc.GEMM_FP32_ADD, seed=seed)
