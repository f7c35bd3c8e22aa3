"""The measurement copy (rlca_measure_copy) that the bench's copy ceilings come from:
every output element is the sum of the inputs and flag bytes at that element, for fp32
and 16-bit inputs, every launch shape and ragged sizes, so the ceiling moves every byte
it claims to move."""
import pytest
import torch

import segmented_associative_scan_gb300 as rlca

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _device(cuda_device):
    rlca.build()
    rlca.lib()


def _expected(inputs, flags, dtype):
    acc = torch.zeros_like(inputs[0], dtype=torch.float64)
    for x in inputs:
        # 16-bit inputs are widened as bf16 bit patterns (the copy only needs to use them).
        if x.dtype != torch.float32:
            x = x.view(torch.int16).to(torch.int32).bitwise_and(0xffff).bitwise_left_shift(16) \
                 .view(torch.float32)
        acc += x.double()
    for f in flags:
        acc += f.double()
    return acc


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16, torch.float16])
@pytest.mark.parametrize("chunks", [1, 2, 4])
@pytest.mark.parametrize("n", [1, 7, 256, 1000, 4096 * 3 + 5, 1 << 20])
@pytest.mark.parametrize("n_in,n_flags,n_out", [(1, 1, 1), (2, 2, 2), (4, 0, 1), (3, 1, 4)])
def test_copy_streams_every_element(dtype, chunks, n, n_in, n_flags, n_out):
    g = torch.Generator(device="cuda").manual_seed(n + 7 * n_in)
    dev = "cuda:0"
    inputs = [torch.randn(n, device=dev, generator=g).to(dtype) for _ in range(n_in)]
    flags = [torch.randint(0, 3, (n,), device=dev, dtype=torch.uint8, generator=g)
             for _ in range(n_flags)]
    outputs = [torch.full((n,), float("nan"), device=dev) for _ in range(n_out)]
    rlca.measure_copy(inputs, flags, outputs, chunks=chunks)
    torch.cuda.synchronize()
    want = _expected(inputs, flags, dtype)
    for o in outputs:
        assert torch.allclose(o.double(), want, rtol=1e-6, atol=1e-5)
