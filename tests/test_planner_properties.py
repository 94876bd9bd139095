"""Seeded random shapes through the host planner (pure host code, no GPU):
every plan it makes, automatic or forced, must be one the kernels can run
correctly and one the launch-time validation accepts.

For each plan: whole clusters, never more clusters than are resident (a
stream-K tail's owners wait for contributors), a workspace of exactly the
size its layout needs, and -- walked out independently of the kernel -- a
segment schedule that covers every K block of every tile exactly once, in
which a tile split by a stream-K tail is finished by the cluster holding
its first K block as that cluster's last segment, with every contributor
after it (so nobody waits on a waiter).  Split-K plans cut each tile into
parts of at least one K block that add up to the tile."""
import math

import numpy as np
import pytest

from dense_fp16_gemm_03_gb300 import build as pkg_build
from dense_fp16_gemm_03_gb300 import gemm as G


@pytest.fixture(scope="module")
def L():
    pkg_build.build()
    return G.lib()


def _clusters():
    return [{1: 152, 2: 76, 4: 36}[G.gemm_f16_variant_info(v)["cluster"]] for v in range(G.gemm_f16_variant_count())]


def _round_up(x, a):
    return (x + a - 1) // a * a


def _check_plan(p, m, n, k, clusters):
    info = G.gemm_f16_variant_info(p.variant)
    cs = info["cluster"]
    assert p.cluster == cs and p.grid >= cs and p.grid % cs == 0
    workers = p.grid // cs
    slots = clusters[p.variant]
    assert workers <= slots
    assert p.k_blocks == -(-k // 64)
    if p.split_k > 1:
        assert p.stream_k == 0 and p.dp_tiles == p.num_tiles and p.sk_iters == 0 and p.k_rotate == 0
        assert p.split_k <= p.k_blocks and workers <= p.num_tiles * p.split_k
        assert p.workspace_bytes == _round_up(p.num_tiles * p.split_k * cs * 128 * info["block_n"] * 4, 256)
        bounds = [s * p.k_blocks // p.split_k for s in range(p.split_k + 1)]
        assert bounds[0] == 0 and bounds[-1] == p.k_blocks
        assert all(bounds[i + 1] > bounds[i] for i in range(p.split_k))     # no empty part
        return
    if p.stream_k == 0:
        assert p.dp_tiles == p.num_tiles and p.sk_iters == 0 and p.workspace_bytes == 0
        assert workers <= max(1, p.num_tiles)
        return
    assert p.sk_iters == (p.num_tiles - p.dp_tiles) * p.k_blocks and p.sk_iters >= workers
    assert p.workspace_bytes == _round_up(p.grid * 128 * info["block_n"] * 4, 256) + _round_up(p.grid * 8, 256)
    # the segment walk, written out independently of the kernel: data-parallel tiles t < dp_tiles go to
    # cluster t mod workers whole; the stream-K iterations are cut into equal contiguous ranges
    intervals, owner = {}, {}
    for w in range(workers):
        b, e = w * p.sk_iters // workers, (w + 1) * p.sk_iters // workers
        it, segs = b, []
        while it < e:
            u, lo = divmod(it, p.k_blocks)
            hi = min(p.k_blocks, lo + (e - it))
            segs.append((p.dp_tiles + u, lo, hi))
            it += hi - lo
        for i, (t, lo, hi) in enumerate(segs):
            intervals.setdefault(t, []).append((lo, hi, w))
            if lo == 0 and hi < p.k_blocks:
                owner[t] = w
                assert i == len(segs) - 1            # an owning segment is its cluster's last
            if lo > 0:
                assert i == 0                        # a publishing segment is its range's first
    # every tail tile's K blocks exactly once: its intervals, sorted, tile [0, k_blocks)
    assert set(intervals) == set(range(p.dp_tiles, p.num_tiles))
    for t, iv in intervals.items():
        iv.sort()
        assert iv[0][0] == 0 and iv[-1][1] == p.k_blocks
        assert all(iv[i][1] == iv[i + 1][0] for i in range(len(iv) - 1))
        if t in owner:                               # contributors come after the owner
            assert all(w >= owner[t] for (_, _, w) in iv)


def test_random_plans_are_runnable(L):
    rng = np.random.Generator(np.random.PCG64(4242))
    clusters = _clusters()
    n_var = G.gemm_f16_variant_count()
    nt = [v for v in range(n_var) if G.gemm_f16_variant_info(v)["layout"] == 0]
    checked = 0
    for _ in range(2500):
        m = int(rng.integers(1, 20000)) if rng.random() < 0.7 else int(rng.integers(1, 300))
        n = 8 * int(rng.integers(1, 3000))
        k = 8 * int(rng.integers(1, 9000))
        variant = -1 if rng.random() < 0.4 else int(rng.choice(nt))
        stream_k = int(rng.choice([-1, 0, 1, 2]))
        try:
            p = G.gemm_f16_nt_plan_for_clusters(m, n, k, 152, clusters, variant, int(rng.integers(0, 9)), stream_k)
        except G.GemmError as e:
            # only a split requested of a variant without split K is refused, and a stream-K tail of a
            # variant whose clusters split every tile's K blocks
            k_split = variant >= 0 and G.gemm_f16_variant_info(variant)["k_split"] > 1
            assert e.status == G.GEMM_ERR_INVALID_ARG and (stream_k == 2 or (stream_k == 1 and k_split))
            continue
        assert (p.m, p.n, p.k) == (m, n, k)
        _check_plan(p, m, n, k, clusters)
        checked += 1
    assert checked > 2000
