"""Split-K against the CPU oracle: every (tile, part) is computed on its own
and published as fp32, and a second kernel adds a tile's parts in part order
and rounds once to fp16.  With operands in {-8..8}/8 every part and every sum
is exact, so the result must match the oracle bit for bit; real-valued
operands must meet |c_gpu - c_ref| <= 1e-3 * sum|a*b| + ulp16(c_ref).  The
shapes include ragged edges, tiles of 128 and 256 columns on one CTA, a CTA
pair and a multicast cluster, and more (tile, part) units than clusters, so
that clusters walk several units.
"""
import numpy as np
import pytest

from gpu_helpers import assert_parity, from_dev_bits, require_gpu, run_gpu, to_dev, torch

from dense_fp16_gemm_03_gb300 import gemm as G
from dense_fp16_gemm_03_gb300 import inputs

pytestmark = pytest.mark.gpu

SPLIT_VARIANTS = [0, 1, 2, 3, 4, 11, 12, 18]   # fp16 C, B [N,K], whole 64-column chunks, no operand swap
SHAPES = [(129, 264, 2048), (300, 520, 4096), (640, 1032, 520), (1000, 1000, 1000), (2304, 2304, 1024),
          (3000, 5000, 512), (8, 64, 8192)]


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


@pytest.mark.parametrize("shape", SHAPES)
@pytest.mark.parametrize("variant", SPLIT_VARIANTS)
def test_split_k_exact(shape, variant):
    M, N, K = shape
    plan = G.gemm_f16_nt_plan_ex(M, N, K, variant, 0, 2)
    assert plan.split_k >= 2 and plan.stream_k == 0 and plan.workspace_bytes > 0
    A, B = inputs.make_operands(M, N, K, "eighths", seed=5 * M + N + K)
    assert_parity(run_gpu(A, B, variant=variant, stream_k=2), A, B, exact=True)


@pytest.mark.parametrize("shape", [(777, 1000, 1536), (256, 256, 65536), (512, 512, 16384)])
def test_split_k_real_valued(shape):
    M, N, K = shape
    A, B = inputs.make_operands(M, N, K, "normal", seed=M + K)
    assert_parity(run_gpu(A, B, variant=2, stream_k=2), A, B)


def test_automatic_plan_uses_split_k_for_long_k():
    """A lone 256 x 256 tile with K = 65536: the automatic plan splits its K and the workspace entry
    point runs it (exact on integer-valued operands)."""
    M, N, K = 256, 256, 65536
    p = G.gemm_f16_nt_plan(M, N, K)
    assert p.split_k > 1
    A, B = inputs.make_operands(M, N, K, "eighths", seed=17)
    assert_parity(run_gpu(A, B, use_ws_entry=True), A, B, exact=True)


def test_split_k_guard_bands_and_reused_workspace():
    """The reduction writes C only inside [0,M) x [0,N); one workspace serves back-to-back launches
    with different operands."""
    M, N, K = 300, 520, 4096
    guard = 4096
    buf = torch.full((guard + M * N + guard,), float("nan"), dtype=torch.float16, device="cuda")
    c = buf[guard:guard + M * N].view(M, N)
    plan = G.gemm_f16_nt_plan_ex(M, N, K, 2, 0, 2)
    ws = torch.full((int(plan.workspace_bytes),), 0x7F, dtype=torch.uint8, device="cuda")
    for seed in (1, 2):
        A, B = inputs.make_operands(M, N, K, "eighths", seed=seed)
        G.gemm_f16_nt_run(plan, to_dev(A), to_dev(B), c, ws)
        assert G.gemm_f16_take_device_error()[0] == G.GEMM_OK
        assert torch.isnan(buf[:guard]).all() and torch.isnan(buf[guard + M * N:]).all()
        assert_parity(from_dev_bits(c), A, B, exact=True)


def test_split_k_refused_where_unsupported():
    """Split-K needs fp16 C with B [N,K], tiles of whole 64-column chunks up to 256 columns and no
    operand swap; every other variant refuses it."""
    for v in range(G.gemm_f16_variant_count()):
        info = G.gemm_f16_variant_info(v)
        capable = (info["layout"] == 0 and not info["swapped"] and info["block_n"] % 64 == 0
                   and info["block_n"] <= 256 and info["k_split"] == 1)
        if capable:
            assert G.gemm_f16_nt_plan_ex(1000, 1000, 1000, v, 0, 2).split_k >= 2
        else:
            with pytest.raises(G.GemmError):
                G.gemm_f16_nt_plan_ex(1000, 1000, 1000, v, 0, 2)
