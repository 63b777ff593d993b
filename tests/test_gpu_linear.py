"""The tcgen05 projection GEMM (kv4_linear_bf16) against a float32 matmul of the same
bf16 inputs: every output within one bf16 rounding of the float32 result (plus the
float32 summation-order difference), on decode, ragged and prefill shapes."""
import pytest
import torch

from int8_hybrid_paged_gb300 import build as kbuild
from int8_hybrid_paged_gb300 import kv4

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    kbuild.build()
    kv4.load()
    torch.backends.cuda.matmul.allow_tf32 = False


def _inputs(M, N, K, seed):
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    x = torch.randn((M, K), generator=g, device="cuda", dtype=torch.float32).to(torch.bfloat16)
    w = (torch.randn((N, K), generator=g, device="cuda", dtype=torch.float32) / K ** 0.5).to(torch.bfloat16)
    return x, w


@pytest.mark.parametrize("M,N,K", [(1, 128, 64), (300, 256, 128), (129, 384, 576),
                                   (64, 1024, 512), (100, 384, 256), (128, 128, 128),   # split-K clusters
                                   (256, 6144, 4096), (2048, 1024, 4096),
                                   (1300, 6144, 320), (4096, 6144, 4096)])   # 256-wide tiles
def test_linear_matches_float32_matmul(M, N, K):
    x, w = _inputs(M, N, K, seed=M + N + K)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    y = kv4.kv4_linear_bf16(x, w, err=err)
    ref = x.float() @ w.float().t()
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    got = y.float()
    scale = (x.float().abs() @ w.float().abs().t())                 # sum of |products|
    bound = 2.0 ** -8 * ref.abs() + 2.0 ** -20 * scale + 1e-30
    bad = (got - ref).abs() > bound
    assert not bad.any(), f"{int(bad.sum())} of {bad.numel()} outputs off, worst {(got - ref).abs().max().item()}"


def test_rejects_unsupported_shapes():
    x, w = _inputs(4, 128, 64, seed=1)
    with pytest.raises(kv4.KV4Error):
        kv4.kv4_linear_bf16(x, w[:100].contiguous())               # N not a multiple of 128
    with pytest.raises(kv4.KV4Error):
        kv4.kv4_linear_bf16(x[:, :32].contiguous(), w[:, :32].contiguous())   # K not a multiple of 64
