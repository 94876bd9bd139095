"""The automatic entry points reuse the plan and encoded parameters of a repeated launch (same
context, shape, pointers and workspace).  A reuse must compute what a fresh launch computes: new
contents of the same buffers, other shapes on the same pointers, other workspaces, more distinct
launches than the cache holds, and stream-K plans (whose flags carry a stamp drawn anew for every
launch, so a repeated launch must never accept the previous one's flags)."""
import pytest

from gpu_helpers import assert_parity, from_dev_bits, require_gpu, to_dev, torch

from dense_fp16_gemm_03_gb300 import gemm as G
from dense_fp16_gemm_03_gb300 import inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def _fill(dst, X):
    dst.copy_(to_dev(X))


def test_repeated_launch_sees_new_contents():
    M, N, K = 300, 520, 1088
    a = torch.empty((M, K), dtype=torch.float16, device="cuda")
    b = torch.empty((N, K), dtype=torch.float16, device="cuda")
    c = torch.empty((M, N), dtype=torch.float16, device="cuda")
    for seed in range(4):
        A, B = inputs.make_operands(M, N, K, "eighths", seed=seed)
        _fill(a, A)
        _fill(b, B)
        c.fill_(float("nan"))
        G.gemm_f16_nt(a, b, c)
        assert G.gemm_f16_take_device_error()[0] == G.GEMM_OK
        assert_parity(from_dev_bits(c), A, B, exact=True)


def test_same_pointers_other_shapes():
    """Leading rows of one allocation: same pointers, different M (and N), different plans."""
    big_a = torch.empty((1024, 2048), dtype=torch.float16, device="cuda")
    big_b = torch.empty((1024, 2048), dtype=torch.float16, device="cuda")
    big_c = torch.empty((1024 * 1024,), dtype=torch.float16, device="cuda")
    for (M, N, K) in [(256, 256, 2048), (1000, 1024, 2048), (256, 256, 2048), (129, 512, 2048), (1000, 1024, 2048)]:
        A, B = inputs.make_operands(M, N, K, "eighths", seed=M + N)
        a, b = big_a[:M], big_b[:N]
        _fill(a, A)
        _fill(b, B)
        c = big_c[:M * N].view(M, N)
        c.fill_(float("nan"))
        G.gemm_f16_nt(a, b, c)
        assert G.gemm_f16_take_device_error()[0] == G.GEMM_OK
        assert_parity(from_dev_bits(c), A, B, exact=True)


def test_stream_k_repeats_and_workspaces():
    """100 x 20000 x 4104 plans a stream-K tail: back-to-back launches on one workspace, with new
    operands each time, then on a second workspace, then the first again."""
    M, N, K = 100, 20000, 4104
    plan = G.gemm_f16_nt_plan(M, N, K)
    ws_bytes = G.gemm_f16_nt_workspace_size(M, N, K)
    assert ws_bytes > 0
    ws1 = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    ws2 = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    a = torch.empty((M, K), dtype=torch.float16, device="cuda")
    b = torch.empty((N, K), dtype=torch.float16, device="cuda")
    c = torch.empty((M, N), dtype=torch.float16, device="cuda")
    for i, ws in enumerate((ws1, ws1, ws1, ws2, ws1)):
        A, B = inputs.make_operands(M, N, K, "eighths", seed=100 + i)
        _fill(a, A)
        _fill(b, B)
        c.fill_(float("nan"))
        G.gemm_f16_nt_ws(a, b, c, ws)
        assert G.gemm_f16_take_device_error()[0] == G.GEMM_OK
        assert_parity(from_dev_bits(c), A, B, exact=True)
    assert plan.stream_k == 1 or plan.split_k > 1


def test_more_launches_than_the_cache_holds():
    shapes = [(128, 64, 64), (256, 256, 256), (300, 520, 136), (512, 512, 1024), (200, 1000, 3000), (96, 2056, 264)]
    bufs = []
    for (M, N, K) in shapes:
        A, B = inputs.make_operands(M, N, K, "eighths", seed=M * 3 + K)
        bufs.append((A, B, to_dev(A), to_dev(B), torch.empty((M, N), dtype=torch.float16, device="cuda")))
    for _ in range(3):
        for (A, B, a, b, c) in bufs:
            c.fill_(float("nan"))
            G.gemm_f16_nt(a, b, c)
            assert G.gemm_f16_take_device_error()[0] == G.GEMM_OK
            assert_parity(from_dev_bits(c), A, B, exact=True)


def test_other_streams_reuse_the_launch():
    """The stream is not part of the key: the same launch on two streams, one after the other."""
    M, N, K = 256, 512, 2048
    A, B = inputs.make_operands(M, N, K, "eighths", seed=3)
    a, b = to_dev(A), to_dev(B)
    c = torch.empty((M, N), dtype=torch.float16, device="cuda")
    for s in (torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.current_stream()):
        c.fill_(float("nan"))
        torch.cuda.synchronize()
        G.gemm_f16_nt(a, b, c, stream=s)
        s.synchronize()
        assert G.gemm_f16_take_device_error(s)[0] == G.GEMM_OK
        assert_parity(from_dev_bits(c), A, B, exact=True)
