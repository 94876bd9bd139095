"""K split across a cluster (the variants whose k_split is > 1): the CTAs of a cluster share every
128 x block_n tile, each accumulating one run of its K blocks, then trade fp32 partials through
distributed shared memory and each adds up and stores its share of the columns.

Integer-valued operands ({-8..8}/8) keep every partial sum exact in fp32 however K is grouped, so
the product must equal the oracle's bit for bit: for K-block counts that split unevenly or leave
some CTAs of the cluster no K block at all, for ragged edges, for clusters that walk several tiles
(each partner slot reused, the slots handed back between tiles) and for every raster width.
Real-valued operands must meet the element-wise tolerance."""
import numpy as np
import pytest

from gpu_helpers import assert_parity, from_dev_bits, require_gpu, run_gpu, to_dev, torch

import oracle
from dense_fp16_gemm_03_gb300 import gemm as G
from dense_fp16_gemm_03_gb300 import inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def _k_split_variants():
    return [v for v in range(G.gemm_f16_variant_count()) if G.gemm_f16_variant_info(v)["k_split"] > 1]


def test_k_split_variants_exist():
    ks = {G.gemm_f16_variant_info(v)["k_split"] for v in _k_split_variants()}
    assert ks == {2, 4}


# K blocks of 64: 1, 2 and 3 blocks leave CTAs of a four-CTA cluster empty; 10 and 17 split unevenly
@pytest.mark.parametrize("shape", [(1, 8, 8), (128, 64, 64), (256, 256, 128), (256, 256, 192), (129, 264, 72),
                                   (300, 520, 136), (256, 512, 640), (1000, 1000, 1088), (96, 2056, 264),
                                   (128, 64, 4096)])
def test_k_split_exact(shape):
    M, N, K = shape
    A, B = inputs.make_operands(M, N, K, "eighths", seed=M + 3 * N + 11 * K)
    for v in _k_split_variants():
        assert_parity(run_gpu(A, B, variant=v), A, B, exact=True)


@pytest.mark.parametrize("clusters", [1, 2, 3, 7])
def test_k_split_clusters_walking_several_tiles(clusters):
    """A grid of few clusters: each walks many tiles, so the partners' slots in every CTA are refilled
    tile after tile, each time only after the CTA has handed them back."""
    M, N, K = 1000, 2056, 520
    A, B = inputs.make_operands(M, N, K, "eighths", seed=clusters + 40)
    ref, _ = oracle.gemm_nt(A, B)
    a, b = to_dev(A), to_dev(B)
    for v in _k_split_variants():
        plan = G.gemm_f16_nt_plan_ex(M, N, K, v, 0, 0)
        assert plan.num_tiles > clusters * 4
        plan.grid = int(clusters * plan.cluster)
        c = torch.full((M, N), float("nan"), dtype=torch.float16, device="cuda")
        G.gemm_f16_nt_run(plan, a, b, c)
        assert G.gemm_f16_take_device_error()[0] == G.GEMM_OK
        got = from_dev_bits(c)
        bad = np.argwhere(got != ref)
        assert bad.size == 0, "variant %d, %d clusters: first mismatch at %s" % (v, clusters, tuple(bad[0]))


@pytest.mark.parametrize("width", [1, 3, 8])
def test_k_split_raster_width(width):
    A, B = inputs.make_operands(700, 1800, 256, "eighths", seed=width)
    for v in _k_split_variants():
        assert_parity(run_gpu(A, B, variant=v, raster_width=width), A, B, exact=True)


@pytest.mark.parametrize("shape", [(777, 1000, 1536), (512, 512, 4096), (129, 264, 72)])
@pytest.mark.parametrize("dist", ["normal", "uniform"])
def test_k_split_tolerance(shape, dist):
    M, N, K = shape
    A, B = inputs.make_operands(M, N, K, dist, seed=M + N + K)
    for v in _k_split_variants():
        assert_parity(run_gpu(A, B, variant=v), A, B)


def test_k_split_rotated_walk_exact():
    """A rotated K walk, then split: each CTA sums a different run of K blocks, the product is the same."""
    M, N, K = 300, 520, 4096
    A, B = inputs.make_operands(M, N, K, "eighths", seed=9)
    a, b = to_dev(A), to_dev(B)
    for v in _k_split_variants():
        plan = G.gemm_f16_nt_plan_ex(M, N, K, v, 0, 0)
        plan.k_rotate = 1
        c = torch.full((M, N), float("nan"), dtype=torch.float16, device="cuda")
        G.gemm_f16_nt_run(plan, a, b, c)
        assert G.gemm_f16_take_device_error()[0] == G.GEMM_OK
        assert_parity(from_dev_bits(c), A, B, exact=True)


def test_k_split_refuses_tails_and_split_k():
    """The cluster already shares each tile's K blocks: a stream-K tail or split-K is refused, at
    planning and when a hand-edited plan asks for one."""
    M, N, K = 1000, 1000, 4096
    a = torch.zeros((M, K), dtype=torch.float16, device="cuda")
    b = torch.zeros((N, K), dtype=torch.float16, device="cuda")
    c = torch.zeros((M, N), dtype=torch.float16, device="cuda")
    for v in _k_split_variants():
        for stream_k in (1, 2):
            with pytest.raises(G.GemmError):
                G.gemm_f16_nt_plan_ex(M, N, K, v, 0, stream_k)
        plan = G.gemm_f16_nt_plan_ex(M, N, K, v, 0, 0)
        plan.stream_k = 1
        with pytest.raises(G.GemmError) as e:
            G.gemm_f16_nt_run(plan, a, b, c)
        assert e.value.status == G.GEMM_ERR_INVALID_ARG
