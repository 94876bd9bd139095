"""The library keeps per-device host state (the kernels' shared-memory
attribute and cluster counts, the device error word's address, the
allocation-free entry point's scratch address) for the CUDA context it was
made in.  After cudaDeviceReset the primary context, the loaded module and
every such address are new; the next call must notice and make the state
again instead of handing a kernel a stale address.

Checked in a child process that drives the CUDA runtime directly (no torch,
whose own state a reset would invalidate): products through gemm_f16_nt and
gemm_f16_nt_noalloc, a reset, fresh buffers, the same products again, each
compared with the CPU oracle.  cudaDeviceReset ends only this child's own
context.
"""
import os
import subprocess
import sys
import textwrap

import pytest

from gpu_helpers import require_gpu

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = textwrap.dedent(r'''
    import ctypes, sys
    import numpy as np
    sys.path.insert(0, ROOT)
    import oracle
    from dense_fp16_gemm_03_gb300 import gemm as G, inputs

    L = G.lib()
    rt = ctypes.CDLL("libcudart.so.13")        # the runtime the library is linked against
    vp = ctypes.c_void_p
    rt.cudaMalloc.argtypes = [ctypes.POINTER(vp), ctypes.c_size_t]
    rt.cudaFree.argtypes = [vp]
    rt.cudaMemcpy.argtypes = [vp, vp, ctypes.c_size_t, ctypes.c_int]
    H2D, D2H = 1, 2

    def ok(e, what):
        if e != 0:
            raise SystemExit("%s failed: cuda error %d" % (what, e))

    def run(fn_name, A, B):
        M, K = A.shape
        N = B.shape[0]
        ptrs = []
        for arr in (A, B):
            p = vp()
            ok(rt.cudaMalloc(ctypes.byref(p), arr.nbytes), "cudaMalloc")
            ok(rt.cudaMemcpy(p, arr.ctypes.data_as(vp), arr.nbytes, H2D), "cudaMemcpy")
            ptrs.append(p)
        c = vp()
        ok(rt.cudaMalloc(ctypes.byref(c), M * N * 2), "cudaMalloc")
        st = getattr(L, fn_name)(M, N, K, ptrs[0], ptrs[1], c, None)
        if st != 0:
            raise SystemExit("%s returned %s" % (fn_name, G.status_string(st)))
        code = ctypes.c_uint32()
        st = L.gemm_f16_take_device_error(None, ctypes.byref(code))
        if st != 0:
            raise SystemExit("device error word 0x%x after %s" % (code.value, fn_name))
        out = np.empty((M, N), dtype=np.uint16)
        ok(rt.cudaMemcpy(out.ctypes.data_as(vp), c, M * N * 2, D2H), "cudaMemcpy")
        for p in ptrs + [c]:
            ok(rt.cudaFree(p), "cudaFree")
        ref, _ = oracle.gemm_nt(A, B)
        if not np.array_equal(out, ref):
            raise SystemExit("%s differs from the oracle (%d elements)" % (fn_name, int((out != ref).sum())))

    # 100 x 20000 x 4104 needs scratch (a stream-K tail): the allocation-free form uses the static array
    A1, B1 = inputs.make_operands(100, 20000, 4104, "eighths", seed=3)
    A2, B2 = inputs.make_operands(300, 520, 264, "eighths", seed=4)
    for round_ in range(2):
        run("gemm_f16_nt_noalloc", A1, B1)
        run("gemm_f16_nt", A2, B2)
        if round_ == 0:
            ok(rt.cudaDeviceReset(), "cudaDeviceReset")
    print("context reset ok")
''').replace("ROOT", repr(ROOT))


def test_state_is_remade_after_device_reset():
    require_gpu()
    r = subprocess.run([sys.executable, "-c", CHILD], capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-2000:]
    assert "context reset ok" in r.stdout
