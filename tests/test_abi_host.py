"""Host-side checks of the C-ABI library that need no GPU: it loads, exports
every declared symbol, validates arguments before touching a device, plans
deterministically, and its scheduler arithmetic (raster map, fast division)
is exact.  The scheduler functions checked here are the same inline code
the kernel runs."""
import ctypes
import math
import os
import re

import numpy as np
import pytest

from dense_fp16_gemm_03_gb300 import build as pkg_build
from dense_fp16_gemm_03_gb300 import gemm as G
from dense_fp16_gemm_03_gb300 import inputs

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    pkg_build.build()
    return G.lib()


TRACE_BLOCK = re.compile(r"#ifdef GEMM_F16_PHASE_TRACE\n(.*?)#endif", re.S)


def _declared_functions(trace_build=False):
    """Functions the header declares for the product build (or, trace_build, only those of the trace build)."""
    text = open(os.path.join(ROOT, "include", "gemm_f16.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    blocks = TRACE_BLOCK.findall(text)
    text = " ".join(blocks) if trace_build else TRACE_BLOCK.sub("", text)
    return sorted(set(re.findall(r"\b(gemm_\w+)\s*\(", text)))


def test_every_declared_symbol_is_exported(L):
    names = _declared_functions()
    assert len(names) >= 14
    for name in names:
        assert hasattr(L, name), name
    assert set(names) == set(G.EXPORTED)


def test_trace_entry_only_in_trace_build(L):
    # the phase-trace setter is declared for the GEMM_F16_PHASE_TRACE build alone; the product
    # library neither exports it nor carries the stamps
    assert _declared_functions(trace_build=True) == ["gemm_f16_trace_set"]
    assert not hasattr(L, "gemm_f16_trace_set")


def test_static_scratch_size_matches_header(L):
    text = open(os.path.join(ROOT, "include", "gemm_f16.h")).read()
    m = re.search(r"#define GEMM_F16_STATIC_SCRATCH_BYTES \((\d+)u \* 1024u \* 1024u\)", text)
    assert m and int(m.group(1)) * 1024 * 1024 == G.STATIC_SCRATCH_BYTES


def test_status_strings(L):
    for s in range(9):
        assert G.status_string(s).startswith("GEMM_")
        assert L.gemm_status_string(s) == L.gemm_f16_status_string(s)
    assert "unknown" in G.status_string(99)


def test_variant_table(L):
    n = G.gemm_f16_variant_count()
    assert n >= 2
    for v in range(n):
        info = G.gemm_f16_variant_info(v)
        assert info["cta_group"] in (1, 2)
        assert info["block_n"] % 32 == 0 and 32 <= info["block_n"] <= 512
        assert info["smem_bytes"] <= 232448
        assert info["layout"] in (0, 1) and info["cluster"] in (1, 2, 4)
    with pytest.raises(G.GemmError):
        G.gemm_f16_variant_info(n)


def test_fast_divmod_brute_force(L):
    rng = np.random.Generator(np.random.PCG64(0))
    divisors = list(range(1, 300)) + [int(x) for x in rng.integers(1, 2 ** 32, size=200)] + [
        2 ** 31, 2 ** 31 + 1, 2 ** 32 - 1, 65535, 65536, 65537]
    numerators = [0, 1, 2, 2 ** 31 - 1, 2 ** 31, 2 ** 32 - 1] + [int(x) for x in rng.integers(0, 2 ** 32, size=60)]
    for d in divisors:
        for n in numerators + [d - 1, d, d + 1, 2 * d - 1, (2 ** 32 - 1) // d * d]:
            if not 0 <= n < 2 ** 32:
                continue
            q, r = G.gemm_f16_fast_divmod(d, n)
            assert (q, r) == divmod(n, d), (d, n)
    with pytest.raises(G.GemmError):
        G.gemm_f16_fast_divmod(0, 5)


def _reference_raster(tiles_m, tiles_n, width, t):
    """Grouped raster, written out independently: groups of `width`
    N-columns (the last one narrower), row-major (N fastest) inside."""
    width = max(1, min(width, tiles_n))
    group = t // (width * tiles_m)
    n_first = group * width
    w = min(width, tiles_n - n_first)
    r = t - group * width * tiles_m
    return r // w, n_first + r % w


@pytest.mark.parametrize("tiles_m,tiles_n", [(1, 1), (1, 64), (64, 1), (7, 5), (13, 29), (32, 32), (24, 20), (2, 2),
                                             (64, 32), (3, 17)])
@pytest.mark.parametrize("width", [1, 2, 3, 4, 8, 16, 100])
def test_raster_is_a_bijection_and_grouped(L, tiles_m, tiles_n, width):
    seen = set()
    for t in range(tiles_m * tiles_n):
        mb, nb = G.gemm_f16_raster_coord(tiles_m, tiles_n, width, t)
        assert 0 <= mb < tiles_m and 0 <= nb < tiles_n
        assert (mb, nb) == _reference_raster(tiles_m, tiles_n, width, t)
        seen.add((mb, nb))
    assert len(seen) == tiles_m * tiles_n


def test_raster_width_one_is_plain_row_major(L):
    for t in range(5 * 7):
        # width 1: each group is one N-column, walked down M
        assert G.gemm_f16_raster_coord(5, 7, 1, t) == (t % 5, t // 5)


def test_plan_for_shapes(L):
    p = G.gemm_f16_nt_plan_for(8192, 8192, 8192, 148, stream_k=0)
    assert p.block_k == 64 and p.k_blocks == 128
    assert p.tiles_m * p.block_m >= 8192 and p.tiles_n * p.block_n >= 8192
    assert p.num_tiles == p.tiles_m * p.tiles_n
    assert p.grid % p.cluster == 0 and p.grid <= 148
    assert p.workspace_bytes == 0
    r = G.gemm_f16_nt_plan_for(3000, 5000, 4096, 148, stream_k=0)
    assert r.tiles_m == -(-3000 // r.block_m) and r.tiles_n == -(-5000 // r.block_n)
    for v in range(G.gemm_f16_variant_count()):
        q = G.gemm_f16_nt_plan_for(128, 16384, 16384, 148, variant=v, raster_width=4, stream_k=0)
        assert q.variant == v and q.raster_width == min(4, q.tiles_n)
        assert q.grid // q.cluster <= q.num_tiles


@pytest.mark.parametrize("m,n,k,status", [
    (-1, 8, 8, G.GEMM_ERR_INVALID_ARG),
    (8, 12, 8, G.GEMM_ERR_UNSUPPORTED_SHAPE),      # n % 8
    (8, 8, 12, G.GEMM_ERR_UNSUPPORTED_SHAPE),      # k % 8
    (2 ** 31, 8, 8, G.GEMM_ERR_UNSUPPORTED_SHAPE),
])
def test_plan_rejects_bad_shapes(L, m, n, k, status):
    p = G.Plan()
    assert L.gemm_f16_nt_plan_for(m, n, k, 148, 0, -1, 0, 0, ctypes.byref(p)) == status
    assert L.gemm_f16_nn_f32(m, n, k, 1 << 20, 1 << 20, 1 << 20, None) == status


def test_argument_errors_before_any_device_call(L):
    """Pointer and shape validation happens on the host before any CUDA call."""
    good = 1 << 20
    assert L.gemm_f16_nt(8, 8, 8, None, good, good, None) == G.GEMM_ERR_INVALID_ARG
    assert L.gemm_f16_nt(8, 8, 8, good, good, None, None) == G.GEMM_ERR_INVALID_ARG
    assert L.gemm_f16_nt(8, 8, 8, good + 2, good, good, None) == G.GEMM_ERR_ALIGNMENT
    assert L.gemm_f16_nt(8, 8, 8, good, good + 8, good, None) == G.GEMM_ERR_ALIGNMENT
    assert L.gemm_f16_nt(8, 8, 8, good, good, good + 4, None) == G.GEMM_ERR_ALIGNMENT
    assert L.gemm_f16_nt(8, 12, 8, good, good, good, None) == G.GEMM_ERR_UNSUPPORTED_SHAPE
    assert L.gemm_f16_nt(8, 8, 10, good, good, good, None) == G.GEMM_ERR_UNSUPPORTED_SHAPE
    assert L.gemm_f16_nt(-3, 8, 8, good, good, good, None) == G.GEMM_ERR_INVALID_ARG
    # empty output: a no-op that needs no pointers at all
    assert L.gemm_f16_nt(0, 8, 8, None, None, None, None) == G.GEMM_OK
    assert L.gemm_f16_nt(8, 0, 8, None, None, None, None) == G.GEMM_OK
    assert L.gemm_f16_nt_run(None, good, good, good, None, 0, None) == G.GEMM_ERR_INVALID_ARG


def test_no_cuda_device_is_an_error_not_a_crash(L):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    good = 1 << 20
    st = L.gemm_f16_nt(128, 128, 64, good, good, good, None)
    assert st == G.GEMM_ERR_CUDA
    p = G.Plan()
    assert L.gemm_f16_nt_plan(128, 128, 64, ctypes.byref(p)) == G.GEMM_ERR_CUDA


@pytest.mark.parametrize("shape", [(4096, 4096, 4096), (3000, 5000, 4096), (128, 16384, 16384), (8192, 8192, 8192),
                                   (1000, 1000, 1000), (128, 256, 8192)])
@pytest.mark.parametrize("variant", [0, 1, 2, 3, 4, 5, 11, 12, 13, 14, 15, 16, 17, 18])
def test_stream_k_plan_invariants(L, shape, variant):
    m, n, k = shape
    for sms in (148, 152):
        p = G.gemm_f16_nt_plan_for(m, n, k, sms, 0, variant, 0, 1)
        workers = p.grid // p.cluster
        if p.stream_k:
            assert p.sk_iters == (p.num_tiles - p.dp_tiles) * p.k_blocks
            assert p.sk_iters >= workers and p.dp_tiles % workers == 0
            assert p.num_tiles - p.dp_tiles <= 2 * workers            # at most two waves are split
            if G.gemm_f16_variant_info(variant)["block_n"] > 256:     # wide tiles: only a partial last wave
                assert p.num_tiles - p.dp_tiles < workers
            bn = G.gemm_f16_variant_info(variant)["block_n"]        # one CTA's partial tile is 128 x bn
            assert p.workspace_bytes >= p.grid * 128 * bn * 4 + p.grid * 8
            slots = sms // p.cluster
            if p.dp_tiles > 0:                                        # after whole waves: every cluster
                assert workers == slots
            else:                                                     # few tiles: sized against the fix-up
                assert workers == min(slots, max(1, int(p.num_tiles * math.sqrt(0.18 * p.k_blocks) + 0.5)))
                # the tail gives each cluster num_tiles / workers tiles: fewer than the most any
                # cluster would run data-parallel (a second, partial wave counts whole)
                dp_waves = -(-p.num_tiles // min(p.num_tiles, slots))
                assert p.num_tiles < dp_waves * workers
        else:                                                         # too little work to split
            assert p.workspace_bytes == 0 and p.dp_tiles == p.num_tiles
        q = G.gemm_f16_nt_plan_for(m, n, k, sms, 0, variant, 0, 0)
        assert q.stream_k == 0 and q.workspace_bytes == 0 and q.dp_tiles == q.num_tiles


@pytest.mark.parametrize("tiles_over_slots,expect_tail", [
    (5, True),        # a few tiles past one wave: each cluster takes a little over one tile
    (152, False),     # exactly two waves: whole tiles already balance
    (0, False),       # exactly one wave
    (100, True),      # a second wave two-thirds full
])
def test_forced_tail_only_when_it_shortens_the_longest_cluster(L, tiles_over_slots, expect_tail):
    """Variant 1 (128 x 128 tiles, 152 slots on 152 SMs) over one strip of B rows: a forced stream-K
    tail is kept exactly when it gives some cluster less work than the data-parallel waves would."""
    tiles = 152 + tiles_over_slots
    p = G.gemm_f16_nt_plan_for(128, 128 * tiles, 4096, 152, 0, 1, 0, 1)
    assert p.num_tiles == tiles
    slots = 152
    full_waves = tiles // slots
    dp = (full_waves - 1) * slots if full_waves >= 1 else 0
    left = tiles - dp
    assert bool(p.stream_k) == expect_tail
    if p.stream_k:
        workers = p.grid // p.cluster
        assert p.dp_tiles == dp and left < -(-left // min(left, slots)) * workers
    else:
        assert p.dp_tiles == tiles and p.workspace_bytes == 0


def _gb300_clusters():
    """Co-resident clusters per variant on a 152-SM GB300 (measured: 76 clusters of two CTAs, 36 of
    four; single CTAs one per SM)."""
    return [{1: 152, 2: 76, 4: 36}[G.gemm_f16_variant_info(v)["cluster"]] for v in range(G.gemm_f16_variant_count())]


def test_gb300_plans_of_the_configured_workloads(L):
    """The host planner with GB300's cluster counts gives the plans the device runs (seen in the bench
    lines), and the committed DRAM-traffic captures were taken on exactly those plans."""
    import json
    expect = {
        "square_256": (22, 0, 0, 0),
        "square_4096": (15, 0, 0, 0),
        "square_8192": (15, 0, 0, 0),
        "ragged_3000x5000x4096": (16, 0, 0, 0),
        "skinny_128x16384x16384": (13, 0, 0, 1),
    }
    rec = json.load(open(os.path.join(os.path.dirname(__file__), "..", "profiles", "dram_traffic.json")))
    for name, (variant, stream_k, split_k, k_rotate) in expect.items():
        w = inputs.BY_NAME[name]
        p = G.gemm_f16_nt_plan_for_clusters(w.M, w.N, w.K, 152, _gb300_clusters())
        assert (p.variant, p.stream_k, p.split_k, p.k_rotate) == (variant, stream_k, split_k, k_rotate), name
        captured = rec["workloads"].get(name)
        if captured is not None:
            assert all(getattr(p, k) == v for k, v in captured["plan"].items()), name


def test_cluster_counts_steer_the_tile_choice(L):
    """3000 x 5000 x 4096: with 38 clusters of four (152 / 4) two multicast pairs with a stream-K tail
    are estimated cheapest; with GB300's 36 the 256 x 448 tile is."""
    clusters = _gb300_clusters()
    assert G.gemm_f16_nt_plan_for_clusters(3000, 5000, 4096, 152, clusters).variant == 16
    ideal = [152 // G.gemm_f16_variant_info(v)["cluster"] for v in range(G.gemm_f16_variant_count())]
    p = G.gemm_f16_nt_plan_for_clusters(3000, 5000, 4096, 152, ideal)
    assert (p.variant, p.stream_k) == (4, 1)
    assert p.as_dict() == G.gemm_f16_nt_plan_for(3000, 5000, 4096, 152).as_dict()


def test_plan_for_clusters_argument_errors(L):
    n_var = G.gemm_f16_variant_count()
    p = G.Plan()
    good = (ctypes.c_int32 * n_var)(*_gb300_clusters())
    assert L.gemm_f16_nt_plan_for_clusters(256, 256, 256, 152, None, n_var, -1, 0, -1, ctypes.byref(p)) == \
        G.GEMM_ERR_INVALID_ARG
    assert L.gemm_f16_nt_plan_for_clusters(256, 256, 256, 152, good, n_var - 1, -1, 0, -1, ctypes.byref(p)) == \
        G.GEMM_ERR_INVALID_ARG
    bad = (ctypes.c_int32 * n_var)(*([0] + _gb300_clusters()[1:]))
    assert L.gemm_f16_nt_plan_for_clusters(256, 256, 256, 152, bad, n_var, -1, 0, -1, ctypes.byref(p)) == \
        G.GEMM_ERR_INVALID_ARG
    assert L.gemm_f16_nt_plan_for_clusters(256, 256, 256, 152, good, n_var, -1, 0, -1, ctypes.byref(p)) == G.GEMM_OK


def _segments(p):
    """The kernel's segment walk for every cluster, written out independently."""
    workers = p.grid // p.cluster
    out = {}
    for w in range(workers):
        segs = [(t, 0, p.k_blocks) for t in range(w, p.dp_tiles, workers)]
        b, e = w * p.sk_iters // workers, (w + 1) * p.sk_iters // workers
        it = b
        while it < e:
            u, lo = divmod(it, p.k_blocks)
            hi = min(p.k_blocks, lo + (e - it))
            segs.append((p.dp_tiles + u, lo, hi))
            it += hi - lo
        out[w] = segs
    return out


@pytest.mark.parametrize("shape", [(4096, 4096, 4096), (3000, 5000, 4096), (128, 16384, 16384), (128, 256, 8192),
                                   (100, 20000, 8192), (128, 24576, 8192)])
def test_stream_k_covers_every_k_block_once(L, shape):
    m, n, k = shape
    for variant in range(G.gemm_f16_variant_count()):
        if G.gemm_f16_variant_info(variant)["k_split"] > 1:
            # a K-split cluster already shares every tile's K blocks: no stream-K tail, no split-K
            for stream_k in (1, 2):
                with pytest.raises(G.GemmError):
                    G.gemm_f16_nt_plan_for(m, n, k, 152, 0, variant, 0, stream_k)
            continue
        p = G.gemm_f16_nt_plan_for(m, n, k, 152, 0, variant, 0, 1)
        if not p.stream_k:
            continue
        cover = {}
        owners = {}
        for w, segs in _segments(p).items():
            n_dp = sum(1 for (t, _, _) in segs if t < p.dp_tiles)
            for i, (t, lo, hi) in enumerate(segs):
                for kb in range(lo, hi):
                    assert (t, kb) not in cover
                    cover[(t, kb)] = w
                if lo == 0 and hi < p.k_blocks:
                    owners[t] = w
                    assert i == len(segs) - 1                         # an owning segment ends its range
                if lo > 0:
                    assert i == n_dp                                  # a publishing segment starts the stream-K range
        assert len(cover) == p.num_tiles * p.k_blocks
        for t, w in owners.items():                                   # contributors come after the owner
            assert all(cover[(t, kb)] >= w for kb in range(p.k_blocks))


def test_layout_of_plans(L):
    for v in range(G.gemm_f16_variant_count()):
        info = G.gemm_f16_variant_info(v)
        p = G.gemm_f16_nt_plan_for(1000, 1000, 1000, 152, 0, v, 0, 0)
        assert p.layout == info["layout"] and p.cluster == info["cluster"]
    assert G.gemm_f16_nt_plan_for(8192, 8192, 8192, 152).layout == 0     # automatic plans are NT


def test_nn_argument_errors(L):
    good = 1 << 20
    assert L.gemm_f16_nn_f32(8, 8, 8, None, good, good, None) == G.GEMM_ERR_INVALID_ARG
    assert L.gemm_f16_nn_f32(8, 8, 8, good, good, good + 4, None) == G.GEMM_ERR_ALIGNMENT
    assert L.gemm_f16_nn_f32(0, 8, 8, None, None, None, None) == G.GEMM_OK


def test_k_rotation_rule(L):
    skinny = G.gemm_f16_nt_plan_for(128, 16384, 16384, 152)
    assert skinny.k_rotate == 1 and skinny.stream_k == 0      # one row of tiles: no strip is shared
    big = G.gemm_f16_nt_plan_for(8192, 8192, 8192, 152)
    assert big.k_rotate == 0                                   # strips shared by neighbouring tiles


@pytest.mark.parametrize("shape,variant,stream_k,split", [
    ((8192, 8192, 8192), 15, 0, False),    # 256 x 512 pair tiles: least data per flop, 96% of the waves busy
    ((6144, 6144, 6144), 15, 0, False),
    ((4096, 8192, 4096), 16, 0, False),    # 256 x 448 tiles fill exactly 4 waves; 256 x 512 ones 84% of theirs
    ((3000, 5000, 4096), 4, 1, False),     # with 38 clusters of four, multicast pairs and a stream-K tail
                                           # (3.3 waves) edge out 144 tiles of 256 x 448 (95% of 2 waves);
                                           # GB300 fits 36, and there the 256 x 448 tile wins
    ((256, 256, 256), 22, 0, False),       # latency-bound: sixteen single-CTA 128 x 32 tiles (3.00 us against 3.21
                                           # for 128 x 64, 3.89 for 128 x 128, 5.74 for one 256 x 256 pair tile)
    ((2048, 1024, 256), 1, 0, False),      # 128 x 64 tiles would need a second wave: 128 x 128
    ((1024, 1024, 448), 18, 0, False),     # 7 K blocks: no stream-K tail (it took 9.05 us against 4.6)
    ((128, 2048, 256), 22, 0, False),      # a strip of rows with short K
    ((256, 256, 512), 22, 0, False),       # mid-size, 8 K blocks: the smallest single-CTA tile in one wave
    ((1024, 1024, 256), 18, 0, False),     # 128 x 32 tiles would need a second wave: 128 x 64
    ((1024, 1024, 1024), 18, 0, False),    # (1024^3: 6.91 us against 13.09 for multicast pairs with split K)
    ((1536, 1536, 1536), 1, 0, False),     # 128 x 64 tiles would need two waves: 128 x 128
    ((2048, 2048, 2048), 0, 0, False),     # 128 x 256 (13.30 us against 15.42)
    ((128, 16384, 16384), 13, 0, False),   # M <= 128, B rows for 64 of 76 pairs: swapped pair tiles, rotated
    ((100, 20000, 8192), 13, 1, False),    # 79 pair tiles for 76 pairs: a stream-K tail, not a second wave
    ((128, 8192, 8192), 1, 0, True),       # 32 pair tiles would idle most pairs: 128 x 128 tiles, K split
    ((256, 256, 1 << 20), 2, 0, True),     # one tile, long K: split-K over every cluster
    ((512, 512, 65536), 4, 0, True),
    ((200, 1000, 3000), 19, 0, False),     # few tiles, 47 K blocks: each tile's K shared by a cluster of four
    ((256, 256, 8192), 1, 0, True),        # four 128 x 128 tiles, 128 K blocks: split-K (unsplit it ran on two SMs)
    ((512, 256, 16384), 1, 0, True),       # 8 tiles x 256 K blocks: 128 x 128 tiles with split-K
    ((512, 512, 32768), 4, 0, True),       # 16 tiles x 512 K blocks: past 4096, multicast pairs with split-K
    ((512, 512, 1024), 20, 0, False),      # 16 K blocks, tiles for half the pairs: K split over CTA pairs
    ((1024, 1024, 2048), 21, 0, False),    # 32 K blocks, 128 x 128 tiles for 64 of 76 pairs: K split in two
    ((4096, 4096, 4096), 4, 1, False),     # whole waves in front: a stream-K tail over every cluster
])
def test_auto_variant_choices(L, shape, variant, stream_k, split):
    """The automatic plan's tile choice on a 152-SM part with every variant's full complement of
    clusters (the measured cases its cost estimates were fitted to)."""
    p = G.gemm_f16_nt_plan_for(*shape, 152)
    assert (p.variant, p.stream_k, p.split_k > 1) == (variant, stream_k, split)
