"""Parity of the CUDA path (through the C ABI) with the CPU oracle.

Integer-valued operands ({-8..8}/8) make every partial sum exact in fp32
and in double, so the GPU must match the oracle bit for bit there; real-
valued operands must meet |gpu - oracle| <= 1e-3 * sum|a*b| + ulp16(oracle)
element by element.  Sizes span several tiles and ragged tails; the five
configured workloads are checked entirely, every element of C, at their
real sizes (the 8192^3 product through both entry points and through every
launch shape of the pipeline ablation ladder).
"""
import numpy as np
import pytest

from gpu_helpers import assert_parity, from_dev_bits, num_sms, require_gpu, run_gpu, to_dev, torch

import oracle
from dense_fp16_gemm_03_gb300 import gemm as G
from dense_fp16_gemm_03_gb300 import inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def _variants():
    """The compiled variants of this layout (B [N,K], fp16 C)."""
    return [v for v in range(G.gemm_f16_variant_count()) if G.gemm_f16_variant_info(v)["layout"] == 0]


def _tail_variants():
    """Those that can run a stream-K tail (all but the K-split clusters, which share every tile's K)."""
    return [v for v in _variants() if G.gemm_f16_variant_info(v)["k_split"] == 1]


# ------------------------------------------------------------------ small

@pytest.mark.parametrize("variant", [0, 1, 2, 3, 4, 5, 11, 12, 13, 14, 15, 16, 17, 18, 19, 20, 21, 22])
def test_square_256_exact_every_variant(variant):
    w = inputs.BY_NAME["square_256"]
    A, B = inputs.workload_operands(w)
    c = run_gpu(A, B, variant=variant)
    assert_parity(c, A, B, exact=True)


def test_day78_lcg_operands_256():
    A, B = inputs.lcg_eighths(256, 256, 256)
    assert_parity(run_gpu(A, B), A, B, exact=True)


RAGGED = [(1, 8, 8), (3, 8, 16), (129, 264, 72), (128, 256, 64), (257, 136, 200), (300, 520, 136),
          (640, 1032, 520), (1000, 1000, 1000), (96, 2056, 264), (300, 872, 200)]


@pytest.mark.parametrize("shape", RAGGED)
@pytest.mark.parametrize("variant", [0, 1, 2, 3, 4, 5, 11, 12, 13, 14, 15, 16, 17, 18, 19, 20, 21, 22])
def test_ragged_exact(shape, variant):
    M, N, K = shape
    A, B = inputs.make_operands(M, N, K, "eighths", seed=M + 7 * N + 13 * K)
    assert_parity(run_gpu(A, B, variant=variant), A, B, exact=True)


@pytest.mark.parametrize("shape", [(129, 264, 72), (777, 1000, 1536), (1024, 1024, 4096)])
@pytest.mark.parametrize("dist", ["normal", "uniform"])
def test_real_valued_tolerance(shape, dist):
    M, N, K = shape
    A, B = inputs.make_operands(M, N, K, dist, seed=M * N + K)
    for v in _variants():
        assert_parity(run_gpu(A, B, variant=v), A, B)


@pytest.mark.parametrize("width", [1, 2, 3, 5, 8, 64])
def test_raster_width_does_not_change_results(width):
    """The raster only reorders tiles: every width gives the oracle's product, bit for bit."""
    A, B = inputs.make_operands(700, 1800, 256, "eighths", seed=5)
    ref, _ = oracle.gemm_nt(A, B)
    for v in _variants():
        got = run_gpu(A, B, variant=v, raster_width=width)
        bad = np.argwhere(got != ref)
        assert bad.size == 0, "variant %d width %d: first mismatch at %s" % (v, width, tuple(bad[0]))


@pytest.mark.parametrize("variant", [8, 9, 10, 2, 4, 15])
def test_one_tile_per_cluster_grid(variant):
    """The ablation ladder's non-persistent launches: a plan whose grid is overridden to one tile per
    cluster (every cluster walks exactly one tile) gives the oracle's product bit for bit."""
    M, N, K = 1000, 2056, 520
    A, B = inputs.make_operands(M, N, K, "eighths", seed=variant + 100)
    plan = G.gemm_f16_nt_plan_ex(M, N, K, variant, 1, 0)
    plan.grid = int(plan.num_tiles * plan.cluster)
    c = torch.full((M, N), float("nan"), dtype=torch.float16, device="cuda")
    G.gemm_f16_nt_run(plan, to_dev(A), to_dev(B), c)
    assert G.gemm_f16_take_device_error()[0] == G.GEMM_OK
    assert_parity(from_dev_bits(c), A, B, exact=True)


# -------------------------------------------------------------- stream-K

SK_SHAPES = [(640, 1032, 520), (1000, 1000, 1000), (300, 520, 4096), (128, 256, 8192), (2304, 2304, 1024),
             (129, 264, 72), (3000, 5000, 512)]


@pytest.mark.parametrize("shape", SK_SHAPES)
@pytest.mark.parametrize("variant", [0, 1, 2, 3, 4, 5, 11, 12, 13, 14, 15, 16, 17, 18])
def test_stream_k_exact(shape, variant):
    """Split tiles are summed from fp32 partials; on integer-valued operands
    every partial and every sum is exact, so the result is still bit-exact."""
    M, N, K = shape
    A, B = inputs.make_operands(M, N, K, "eighths", seed=3 * M + N + K)
    assert_parity(run_gpu(A, B, variant=variant, stream_k=1), A, B, exact=True)


@pytest.mark.parametrize("variant", [1, 13])
def test_stream_k_tail_past_one_wave_exact(variant):
    """A few more tiles than clusters (one row of them, K in 33 blocks, the last ragged): the automatic
    tail spreads every tile over all clusters, each taking a little over one tile, so nearly every
    tile is split in two and finished by the cluster that holds its first K block."""
    M, N, K = 100, 128 * (num_sms() + 6), 2056
    plan = G.gemm_f16_nt_plan_ex(M, N, K, variant, 0, -1)
    assert plan.stream_k == 1 and plan.dp_tiles == 0 and plan.num_tiles > plan.grid // plan.cluster
    A, B = inputs.make_operands(M, N, K, "eighths", seed=N + variant)
    assert_parity(run_gpu(A, B, variant=variant, stream_k=-1), A, B, exact=True)


@pytest.mark.parametrize("variant", [15, 16, 17])
def test_wide_tail_after_whole_waves_exact(variant):
    """Wide tiles keep every whole wave data-parallel and split only the partial last wave over all
    clusters: one whole wave plus a partial one (ragged edges, K in 40 blocks), bit for bit."""
    M, N, K = 256 * 13, 5000, 2560
    plan = G.gemm_f16_nt_plan_ex(M, N, K, variant, 0, 1)
    slots = plan.grid // plan.cluster
    assert plan.stream_k == 1 and plan.dp_tiles > 0 and plan.dp_tiles % slots == 0
    assert 0 < plan.num_tiles - plan.dp_tiles < slots
    A, B = inputs.make_operands(M, N, K, "eighths", seed=variant + 7)
    assert_parity(run_gpu(A, B, variant=variant, stream_k=1), A, B, exact=True)


@pytest.mark.parametrize("shape", [(777, 1000, 1536), (1024, 1024, 4096), (128, 2048, 16384)])
def test_stream_k_tolerance(shape):
    M, N, K = shape
    A, B = inputs.make_operands(M, N, K, "normal", seed=M + K)
    for v in _tail_variants():
        assert_parity(run_gpu(A, B, variant=v, stream_k=1), A, B)


@pytest.mark.parametrize("fill", [0x00, 0x01, 0xFF])
def test_stream_k_reused_and_dirty_workspace(fill):
    """Stream-K flags carry per-launch stamps: a workspace full of leftovers or
    of an earlier launch's flags must not let an owner read stale partials."""
    M, N, K = 1000, 1000, 1000
    A, B = inputs.make_operands(M, N, K, "eighths", seed=fill + 1)
    A2, B2 = inputs.make_operands(M, N, K, "eighths", seed=fill + 2)
    for v in (1, 2, 4, 15):
        plan = G.gemm_f16_nt_plan_ex(M, N, K, v, 0, 1)
        assert plan.stream_k == 1
        ws = torch.full((int(plan.workspace_bytes),), fill, dtype=torch.uint8, device="cuda")
        for (X, Y) in ((A, B), (A2, B2), (A, B)):      # back to back on one workspace
            c = torch.full((M, N), float("nan"), dtype=torch.float16, device="cuda")
            G.gemm_f16_nt_run(plan, to_dev(X), to_dev(Y), c, ws)
            assert G.gemm_f16_take_device_error()[0] == G.GEMM_OK
            assert_parity(from_dev_bits(c), X, Y, exact=True)


def test_stream_k_plan_shape():
    sms = num_sms()
    p = G.gemm_f16_nt_plan_ex(4096, 4096, 4096, 2, 0, 1)
    assert p.stream_k == 1 and p.workspace_bytes > 0
    assert p.sk_iters == (p.num_tiles - p.dp_tiles) * p.k_blocks
    assert p.dp_tiles % (p.grid // p.cluster) == 0


def test_workspace_entry_point_rejects_small_workspace():
    M, N, K = 1000, 1000, 8192
    need = G.gemm_f16_nt_workspace_size(M, N, K)
    assert need > 0                               # the automatic plan splits K here (few tiles)
    a = torch.zeros((M, K), dtype=torch.float16, device="cuda")
    b = torch.zeros((N, K), dtype=torch.float16, device="cuda")
    c = torch.zeros((M, N), dtype=torch.float16, device="cuda")
    small = torch.empty(need - 256, dtype=torch.uint8, device="cuda")
    st = G.lib().gemm_f16_nt_ws(M, N, K, a.data_ptr(), b.data_ptr(), c.data_ptr(), small.data_ptr(), need - 256,
                                torch.cuda.current_stream().cuda_stream)
    assert st == G.GEMM_ERR_WORKSPACE


@pytest.mark.parametrize("shape", [(128, 2048, 4096), (1000, 1000, 1000), (300, 520, 4096)])
def test_k_rotation_exact(shape):
    """A rotated K walk only reorders the fp32 sums: integer-valued products stay bit-exact."""
    M, N, K = shape
    A, B = inputs.make_operands(M, N, K, "eighths", seed=M + 5 * N)
    a, b = to_dev(A), to_dev(B)
    for v in _variants():
        plan = G.gemm_f16_nt_plan_ex(M, N, K, v, 0, 0)
        for rot in (0, 1):
            plan.k_rotate = rot
            c = torch.full((M, N), float("nan"), dtype=torch.float16, device="cuda")
            G.gemm_f16_nt_run(plan, a, b, c)
            assert G.gemm_f16_take_device_error()[0] == G.GEMM_OK
            assert_parity(from_dev_bits(c), A, B, exact=True)


# ------------------------------------------------------ structured operands

@pytest.mark.parametrize("n", [128, 200, 256, 520])
def test_identity_and_permutation(n):
    rng = np.random.Generator(np.random.PCG64(n))
    B = rng.standard_normal((n, n)).astype(np.float16)
    for v in _variants():
        c = run_gpu(inputs.identity(n), B, variant=v)          # = B^T exactly
        assert np.array_equal(oracle.f16_to_f64(c), B.T.astype(np.float64))
        P, p = inputs.permutation(n, seed=n + 1)
        c = run_gpu(P, B, variant=v)                            # C[i, j] = B[j, p[i]]
        assert np.array_equal(oracle.f16_to_f64(c), B[:, p].T.astype(np.float64))
        c = run_gpu(B, inputs.identity(n), variant=v)          # = B exactly
        assert np.array_equal(oracle.f16_to_f64(c), B.astype(np.float64))


@pytest.mark.parametrize("shape", [(129, 264, 72), (256, 512, 640), (300, 8, 4096)])
def test_rank1_closed_form(shape):
    M, N, K = shape
    A, B, (u, w, v) = inputs.rank1(M, N, K, seed=K)
    expect = (np.outer(u, w) * float(np.sum(v * v))).astype(np.float16).view(np.uint16)
    for var in _variants():
        assert np.array_equal(run_gpu(A, B, variant=var), expect)


# ----------------------------------------------------------------- edges

def test_empty_and_zero_k():
    a = torch.zeros((0, 64), dtype=torch.float16, device="cuda")
    b = torch.zeros((16, 64), dtype=torch.float16, device="cuda")
    c = torch.empty((0, 16), dtype=torch.float16, device="cuda")
    G.gemm_f16_nt(a, b, c)
    a = torch.randn((40, 0), device="cuda").half()
    b = torch.randn((24, 0), device="cuda").half()
    c = torch.full((40, 24), 7.0, dtype=torch.float16, device="cuda")
    G.gemm_f16_nt(a, b, c)                                      # empty sum: C := 0
    torch.cuda.synchronize()
    assert torch.count_nonzero(c).item() == 0


def test_guard_bands_untouched():
    M, N, K = 300, 520, 136
    A, B = inputs.make_operands(M, N, K, "eighths", seed=9)
    guard = 4096
    buf = torch.full((guard + M * N + guard,), float("nan"), dtype=torch.float16, device="cuda")
    c = buf[guard:guard + M * N].view(M, N)
    G.gemm_f16_nt(to_dev(A), to_dev(B), c)
    torch.cuda.synchronize()
    assert torch.isnan(buf[:guard]).all() and torch.isnan(buf[guard + M * N:]).all()
    assert_parity(from_dev_bits(c), A, B, exact=True)


def test_misaligned_pointer_rejected_without_launch():
    a = torch.zeros(64 * 64 + 8, dtype=torch.float16, device="cuda")
    b = torch.zeros((64, 64), dtype=torch.float16, device="cuda")
    c = torch.full((64, 64), 3.0, dtype=torch.float16, device="cuda")
    st = G.lib().gemm_f16_nt(64, 64, 64, a.data_ptr() + 2, b.data_ptr(), c.data_ptr(),
                             torch.cuda.current_stream().cuda_stream)
    assert st == G.GEMM_ERR_ALIGNMENT
    torch.cuda.synchronize()
    assert (c == 3.0).all()


def test_side_stream_and_host_entry_point():
    M, N, K = 384, 640, 320
    A, B = inputs.make_operands(M, N, K, "eighths", seed=21)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        c = run_gpu(A, B, stream=s)
    assert_parity(c, A, B, exact=True)
    a_h = torch.from_numpy(A.view(np.int16)).view(torch.float16).pin_memory()
    b_h = torch.from_numpy(B.view(np.int16)).view(torch.float16).pin_memory()
    c_h = torch.empty((M, N), dtype=torch.float16).pin_memory()
    a_d = torch.empty((M, K), dtype=torch.float16, device="cuda")
    b_d = torch.empty((N, K), dtype=torch.float16, device="cuda")
    c_d = torch.empty((M, N), dtype=torch.float16, device="cuda")
    G.gemm_f16_nt_host(a_h, b_h, c_h, a_d, b_d, c_d, stream=s)
    s.synchronize()
    assert_parity(c_h.view(torch.int16).numpy().view(np.uint16), A, B, exact=True)
    ws = torch.empty(max(256, G.gemm_f16_nt_workspace_size(M, N, K)), dtype=torch.uint8, device="cuda")
    c_h.zero_()
    G.gemm_f16_nt_host(a_h, b_h, c_h, a_d, b_d, c_d, ws, stream=s)
    s.synchronize()
    assert_parity(c_h.view(torch.int16).numpy().view(np.uint16), A, B, exact=True)


@pytest.mark.parametrize("shape", [(2048, 1032, 520), (3000, 520, 264), (4096, 1024, 512), (8192, 264, 136)])
@pytest.mark.parametrize("use_ws", [False, True])
def test_host_entry_point_chunked(shape, use_ws):
    """From 2048 rows on, the host-buffer entry point moves A and C through in row chunks on two
    copy streams beside the GEMMs (ragged last chunk included); back-to-back calls with different
    operands on one stream must not overwrite device buffers a previous call still reads, and the
    caller's stream must continue only after the last copy out."""
    M, N, K = shape
    s = torch.cuda.Stream()
    a_d = torch.empty((M, K), dtype=torch.float16, device="cuda")
    b_d = torch.empty((N, K), dtype=torch.float16, device="cuda")
    c_d = torch.empty((M, N), dtype=torch.float16, device="cuda")
    ws = None
    if use_ws:
        ws = torch.empty(max(256, G.gemm_f16_nt_workspace_size(M, N, K)), dtype=torch.uint8, device="cuda")
    pairs, outs = [], []
    for seed in (31, 32, 33):
        A, B = inputs.make_operands(M, N, K, "eighths", seed=seed + M)
        a_h = torch.from_numpy(A.view(np.int16)).view(torch.float16).pin_memory()
        b_h = torch.from_numpy(B.view(np.int16)).view(torch.float16).pin_memory()
        c_h = torch.full((M, N), float("nan"), dtype=torch.float16).pin_memory()
        pairs.append((A, B, a_h, b_h))                                   # host buffers live until the sync
        outs.append(c_h)
        G.gemm_f16_nt_host(a_h, b_h, c_h, a_d, b_d, c_d, ws, stream=s)     # no sync between calls
    with torch.cuda.stream(s):
        c_dev_copy = c_d.clone()                                          # ordered after the last call
    s.synchronize()
    assert G.gemm_f16_take_device_error()[0] == G.GEMM_OK
    for (A, B, _, _), c_h in zip(pairs, outs):
        assert_parity(c_h.view(torch.int16).numpy().view(np.uint16), A, B, exact=True)
    assert torch.equal(c_dev_copy.cpu().view(torch.int16), outs[-1].view(torch.int16))


def test_plan_matches_device():
    p = G.gemm_f16_nt_plan(8192, 8192, 8192)
    assert p.num_sms == num_sms()
    assert G.gemm_f16_nt_workspace_size(8192, 8192, 8192) == p.workspace_bytes
    if p.stream_k:
        assert p.workspace_bytes >= p.grid * (p.block_m // p.cta_group) * p.block_n * 4


def test_host_planner_reproduces_device_plans():
    """On a 152-SM GB300 the device measures 76 co-resident clusters of two CTAs and 36 of four; the
    host planner given those counts must produce the device's own automatic plans."""
    if num_sms() != 152:
        pytest.skip("the cluster table below is GB300's")
    clusters = [{1: 152, 2: 76, 4: 36}[G.gemm_f16_variant_info(v)["cluster"]]
                for v in range(G.gemm_f16_variant_count())]
    for w in inputs.WORKLOADS:
        dev = G.gemm_f16_nt_plan(w.M, w.N, w.K).as_dict()
        host = G.gemm_f16_nt_plan_for_clusters(w.M, w.N, w.K, 152, clusters).as_dict()
        assert dev == host, w.name


# ------------------------------------------------------- full workloads

def _full(name):
    w = inputs.BY_NAME[name]
    A, B = inputs.workload_operands(w)
    return w, A, B


@pytest.mark.parametrize("use_ws", [False, True])
@pytest.mark.parametrize("name", ["square_256", "ragged_3000x5000x4096"])
def test_integer_workloads_bit_exact(name, use_ws):
    w, A, B = _full(name)
    assert_parity(run_gpu(A, B, use_ws_entry=use_ws), A, B, exact=True)


@pytest.mark.parametrize("use_ws", [False, True])
@pytest.mark.parametrize("name", ["square_4096", "skinny_128x16384x16384"])
def test_real_workloads_full_tolerance(name, use_ws):
    w, A, B = _full(name)
    assert_parity(run_gpu(A, B, use_ws_entry=use_ws), A, B)


@pytest.fixture(scope="module")
def square_8192():
    """The 8192^3 workload and the oracle's whole product (about half a minute on 16 host cores)."""
    w, A, B = _full("square_8192")
    ref, absum = oracle.gemm_nt(A, B)
    return w, A, B, ref, absum


def _assert_full_parity(c_bits, ref, absum, what):
    """Every element within the bound.  Elements whose bits equal the oracle's pass by definition,
    so the bound is evaluated only where the bits differ (the same verdict, much faster)."""
    flat, rflat = c_bits.ravel(), ref.ravel()
    diff = np.flatnonzero(flat != rflat)
    rep = oracle.check_parity(flat[diff], rflat[diff], absum.ravel()[diff])
    assert rep.ok, "%s: %r (first failure at flat index %s)" % (
        what, rep, None if rep.first is None else int(diff[rep.first[0]]))
    assert not np.isnan(oracle.f16_to_f64(flat)).any(), what
    return diff.size


@pytest.mark.parametrize("use_ws", [False, True])
def test_square_8192_full(square_8192, use_ws):
    """All 67,108,864 elements of the headline product, through both entry points."""
    w, A, B, ref, absum = square_8192
    _assert_full_parity(run_gpu(A, B, use_ws_entry=use_ws), ref, absum, "use_ws=%s" % use_ws)


def test_square_8192_full_ablation_launches(square_8192):
    """Every rung of the pipeline ablation ladder (bench.py --ablation) computes the whole 8192^3
    product within the bound, including the rungs that launch one tile per cluster."""
    import bench
    w, A, B, ref, absum = square_8192
    a, b = to_dev(A), to_dev(B)
    for label, _, variant, raster, one_tile in bench.ABLATION:
        plan = G.gemm_f16_nt_plan_ex(w.M, w.N, w.K, variant, raster, 0)
        if one_tile:
            plan.grid = int(plan.num_tiles * plan.cluster)
        c = torch.full((w.M, w.N), float("nan"), dtype=torch.float16, device="cuda")
        G.gemm_f16_nt_run(plan, a, b, c)
        st, code = G.gemm_f16_take_device_error()
        assert st == G.GEMM_OK, "%s: device error word 0x%x" % (label, code)
        _assert_full_parity(from_dev_bits(c), ref, absum, label)
