"""GPU unit test of the fifth-generation tensor-core primitives (TMEM
allocation, the 128-byte-swizzled K-major shared-memory descriptor, the
kind::f16 instruction descriptor, the MMA chain, its mbarrier commit and the
TMEM loads) through the one-block product export of libcf.so.

Small-integer operands make every product and sum exact in fp32, so the
result is compared bit for bit with a host matmul: a wrong row, column or k
index anywhere in the layout changes some element.
"""
import pytest
import torch

from attention_block_gb300 import binding

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _need_cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    binding.lib()


DT = {"f16": (binding.CF_F16, torch.float16), "bf16": (binding.CF_BF16, torch.bfloat16)}


def _run(dt, n, k, a, b, a_mn=False):
    code, _ = DT[dt]
    d = torch.full((128, n), float("nan"), device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    assert binding.cf_test_tc05_gemm(code, n, k, a, b, d, err, a_mn=a_mn) == binding.CF_OK
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    return d


@pytest.mark.parametrize("dt", ["f16", "bf16"])
@pytest.mark.parametrize("n,k", [(16, 64), (64, 64), (64, 256), (128, 128), (256, 256)])
def test_integer_product_is_exact(dt, n, k):
    _, tt = DT[dt]
    g = torch.Generator().manual_seed(n * 7 + k)
    a = torch.randint(-8, 9, (128, k), generator=g).to(tt)
    b = torch.randint(-8, 9, (n, k), generator=g).to(tt)
    d = _run(dt, n, k, a.cuda(), b.cuda())
    ref = (a.double() @ b.double().T).float()
    assert torch.equal(d.cpu(), ref)


@pytest.mark.parametrize("dt", ["f16", "bf16"])
@pytest.mark.parametrize("n,k", [(32, 64), (64, 128), (128, 64), (256, 192)])
def test_m_major_a_integer_product_is_exact(dt, n, k):
    """A read as the transpose of a [k, 128] weight tile held in two swizzled
    64-column boxes (the transposed projections' operand)."""
    _, tt = DT[dt]
    g = torch.Generator().manual_seed(n * 13 + k)
    w = torch.randint(-8, 9, (k, 128), generator=g).to(tt)
    b = torch.randint(-8, 9, (n, k), generator=g).to(tt)
    d = _run(dt, n, k, w.cuda(), b.cuda(), a_mn=True)
    ref = (w.double().T @ b.double().T).float()
    assert torch.equal(d.cpu(), ref)


@pytest.mark.parametrize("dt", ["f16", "bf16"])
def test_normal_operands_match_fp32_matmul(dt):
    _, tt = DT[dt]
    g = torch.Generator().manual_seed(11)
    a = torch.randn(128, 192, generator=g).to(tt)
    b = torch.randn(96, 192, generator=g).to(tt)
    d = _run(dt, 96, 192, a.cuda(), b.cuda()).cpu().double()
    ref = a.double() @ b.double().T
    assert (d - ref).abs().max().item() <= 1e-4 * ref.abs().max().item() + 1e-5


def test_argument_errors():
    a = torch.zeros(128, 64, dtype=torch.float16, device="cuda")
    d = torch.zeros(128, 64, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    for n, k in ((8, 64), (24, 64), (272, 64), (64, 48), (256, 1024)):
        assert binding.cf_test_tc05_gemm(binding.CF_F16, n, k, a, a, d, err) == \
            binding.CF_ERR_INVALID_ARG, (n, k)
    assert binding.cf_test_tc05_gemm(binding.CF_F32, 64, 64, a, a, d, err) == \
        binding.CF_ERR_INVALID_ARG
