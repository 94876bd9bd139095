"""ctypes binding of the C ABI in include/gemm_f16.h (same entry-point names).

Argument marshalling only: every step of the product runs in the CUDA
library.  A missing library raises at load time; there is no fallback.
Device buffers are torch tensors (or raw integer device addresses); streams
are torch.cuda.Stream objects, raw cudaStream_t integers, or None for the
current torch stream.
"""
import ctypes
import os

from . import build as _build

GEMM_OK = 0
GEMM_ERR_INVALID_ARG = 1
GEMM_ERR_ALIGNMENT = 2
GEMM_ERR_UNSUPPORTED_SHAPE = 3
GEMM_ERR_ARCH = 4
GEMM_ERR_WORKSPACE = 5
GEMM_ERR_LAUNCH = 6
GEMM_ERR_TIMEOUT = 7
GEMM_ERR_CUDA = 8

LIB_PATH = _build.LIB

# size of the scratch array built into the library (GEMM_F16_STATIC_SCRATCH_BYTES)
STATIC_SCRATCH_BYTES = 20 * 1024 * 1024


class GemmError(RuntimeError):
    def __init__(self, status, where):
        self.status = status
        super().__init__("%s: %s" % (where, status_string(status)))


class Plan(ctypes.Structure):
    """Mirror of gemm_f16_plan_t."""
    _fields_ = [
        ("variant", ctypes.c_int32),
        ("cta_group", ctypes.c_int32),
        ("block_m", ctypes.c_int32),
        ("block_n", ctypes.c_int32),
        ("block_k", ctypes.c_int32),
        ("stages", ctypes.c_int32),
        ("raster_width", ctypes.c_int32),
        ("stream_k", ctypes.c_int32),
        ("layout", ctypes.c_int32),
        ("k_rotate", ctypes.c_int32),
        ("m", ctypes.c_int64),
        ("n", ctypes.c_int64),
        ("k", ctypes.c_int64),
        ("tiles_m", ctypes.c_int64),
        ("tiles_n", ctypes.c_int64),
        ("num_tiles", ctypes.c_int64),
        ("k_blocks", ctypes.c_int64),
        ("dp_tiles", ctypes.c_int64),
        ("sk_iters", ctypes.c_int64),
        ("grid", ctypes.c_int32),
        ("cluster", ctypes.c_int32),
        ("smem_bytes", ctypes.c_int32),
        ("num_sms", ctypes.c_int32),
        ("workspace_bytes", ctypes.c_uint64),
        ("split_k", ctypes.c_int32),
    ]

    def as_dict(self):
        return {name: getattr(self, name) for name, _ in self._fields_}

    def __repr__(self):
        return "Plan(%s)" % ", ".join("%s=%s" % kv for kv in self.as_dict().items())


# every symbol the public header declares
EXPORTED = [
    "gemm_f16_status_string", "gemm_status_string", "gemm_f16_variant_count", "gemm_f16_variant_info",
    "gemm_f16_nt_plan", "gemm_f16_nt_plan_for", "gemm_f16_nt_plan_for_clusters", "gemm_f16_nt_plan_ex",
    "gemm_f16_nt_workspace_size",
    "gemm_f16_nt", "gemm_f16_nt_ws", "gemm_f16_nt_run", "gemm_f16_nt_host",
    "gemm_f16_take_device_error", "gemm_f16_raster_coord", "gemm_f16_fast_divmod",
    "gemm_f16_nt_run_stall_test", "gemm_f16_nt_noalloc",
    "gemm_f16_nn_f32", "gemm_f16_nn_f32_ws", "gemm_f16_nn_f32_plan_ex",
]

_lib = None


def lib():
    """Load libgemm_f16.so (built in-tree by build.py); raise if it is missing."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError("libgemm_f16.so is not built (%s); run __graft_entry__.build()" % LIB_PATH)
    L = ctypes.CDLL(LIB_PATH)
    i32, i64, u32, vp = ctypes.c_int32, ctypes.c_int64, ctypes.c_uint32, ctypes.c_void_p
    pi32, pi64, pu32 = ctypes.POINTER(i32), ctypes.POINTER(i64), ctypes.POINTER(u32)
    P = ctypes.POINTER(Plan)
    sig = {
        "gemm_f16_status_string": (ctypes.c_char_p, [ctypes.c_int]),
        "gemm_status_string": (ctypes.c_char_p, [ctypes.c_int]),
        "gemm_f16_variant_count": (i32, []),
        "gemm_f16_variant_info": (ctypes.c_int, [i32, pi32, pi32, pi32, pi32, pi32, pi32, pi32, pi32]),
        "gemm_f16_nt_plan": (ctypes.c_int, [i64, i64, i64, P]),
        "gemm_f16_nt_plan_for": (ctypes.c_int, [i64, i64, i64, i32, i32, i32, i32, i32, P]),
        "gemm_f16_nt_plan_for_clusters": (ctypes.c_int, [i64, i64, i64, i32, pi32, i32, i32, i32, i32, P]),
        "gemm_f16_nt_plan_ex": (ctypes.c_int, [i64, i64, i64, i32, i32, i32, P]),
        "gemm_f16_nt_workspace_size": (ctypes.c_int, [i64, i64, i64, ctypes.POINTER(ctypes.c_size_t)]),
        "gemm_f16_nt": (ctypes.c_int, [i64, i64, i64, vp, vp, vp, vp]),
        "gemm_f16_nt_ws": (ctypes.c_int, [i64, i64, i64, vp, vp, vp, vp, ctypes.c_size_t, vp]),
        "gemm_f16_nt_run": (ctypes.c_int, [P, vp, vp, vp, vp, ctypes.c_size_t, vp]),
        "gemm_f16_nt_host": (ctypes.c_int, [i64, i64, i64, vp, vp, vp, vp, vp, vp, vp, ctypes.c_size_t, vp]),
        "gemm_f16_take_device_error": (ctypes.c_int, [vp, pu32]),
        "gemm_f16_raster_coord": (ctypes.c_int, [i64, i64, i32, i64, pi64, pi64]),
        "gemm_f16_fast_divmod": (ctypes.c_int, [u32, u32, pu32, pu32]),
        "gemm_f16_nt_run_stall_test": (ctypes.c_int, [P, vp, vp, vp, u32, ctypes.c_longlong, vp]),
        "gemm_f16_nt_noalloc": (ctypes.c_int, [i64, i64, i64, vp, vp, vp, vp]),
        "gemm_f16_nn_f32": (ctypes.c_int, [i64, i64, i64, vp, vp, vp, vp]),
        "gemm_f16_nn_f32_ws": (ctypes.c_int, [i64, i64, i64, vp, vp, vp, vp, ctypes.c_size_t, vp]),
        "gemm_f16_nn_f32_plan_ex": (ctypes.c_int, [i64, i64, i64, i32, i32, i32, P]),
    }
    for name, (res, args) in sig.items():
        f = getattr(L, name)
        f.restype = res
        f.argtypes = args
    _lib = L
    return L


def status_string(status):
    return lib().gemm_f16_status_string(int(status)).decode()


def _check(status, where):
    if status != GEMM_OK:
        raise GemmError(status, where)


_torch = None


def _tm():
    """torch, imported once (the binding works without it for plain integer addresses)."""
    global _torch
    if _torch is None:
        import torch
        _torch = torch
    return _torch


def _ptr(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(stream):
    if stream is None:
        return _tm().cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


# ----------------------------------------------------------------- queries

def gemm_f16_variant_count():
    return int(lib().gemm_f16_variant_count())


def gemm_f16_variant_info(variant):
    cg, bn, st, sm, cl, lay, sw, ks = (ctypes.c_int32() for _ in range(8))
    _check(lib().gemm_f16_variant_info(variant, ctypes.byref(cg), ctypes.byref(bn), ctypes.byref(st),
                                       ctypes.byref(sm), ctypes.byref(cl), ctypes.byref(lay), ctypes.byref(sw),
                                       ctypes.byref(ks)),
           "gemm_f16_variant_info")
    return {"cta_group": cg.value, "block_n": bn.value, "stages": st.value, "smem_bytes": sm.value,
            "cluster": cl.value, "layout": lay.value, "swapped": sw.value, "k_split": ks.value}


def gemm_f16_nt_plan(m, n, k):
    p = Plan()
    _check(lib().gemm_f16_nt_plan(m, n, k, ctypes.byref(p)), "gemm_f16_nt_plan")
    return p


def gemm_f16_nt_plan_for(m, n, k, num_sms, max_clusters=0, variant=-1, raster_width=0, stream_k=-1):
    """stream_k: -1 automatic, 0 data-parallel only, 1 stream-K tail."""
    p = Plan()
    _check(lib().gemm_f16_nt_plan_for(m, n, k, num_sms, max_clusters, variant, raster_width, stream_k,
                                      ctypes.byref(p)), "gemm_f16_nt_plan_for")
    return p


def gemm_f16_nt_plan_for_clusters(m, n, k, num_sms, clusters_by_variant, variant=-1, raster_width=0, stream_k=-1):
    """Host-only plan with the co-resident cluster count of every variant given (one entry per variant)."""
    table = (ctypes.c_int32 * len(clusters_by_variant))(*clusters_by_variant)
    p = Plan()
    _check(lib().gemm_f16_nt_plan_for_clusters(m, n, k, num_sms, table, len(clusters_by_variant), variant,
                                               raster_width, stream_k, ctypes.byref(p)),
           "gemm_f16_nt_plan_for_clusters")
    return p


def gemm_f16_nt_plan_ex(m, n, k, variant=-1, raster_width=0, stream_k=-1):
    """Plan for the current device with optional overrides (negative/zero = automatic)."""
    p = Plan()
    _check(lib().gemm_f16_nt_plan_ex(m, n, k, variant, raster_width, stream_k, ctypes.byref(p)),
           "gemm_f16_nt_plan_ex")
    return p


def workspace_for(plan, device="cuda"):
    """A torch uint8 buffer of the plan's workspace size (None if it needs none)."""
    if plan.workspace_bytes == 0:
        return None
    import torch
    return torch.empty(int(plan.workspace_bytes), dtype=torch.uint8, device=device)


def gemm_f16_nt_workspace_size(m, n, k):
    b = ctypes.c_size_t()
    _check(lib().gemm_f16_nt_workspace_size(m, n, k, ctypes.byref(b)), "gemm_f16_nt_workspace_size")
    return b.value


# ------------------------------------------------------------------ launches

def _shape(a, b):
    sa, sb = a.shape, b.shape
    if len(sa) != 2 or len(sb) != 2 or sa[1] != sb[1]:
        raise ValueError("a must be [M,K] and b [N,K]")
    f16 = _tm().float16
    if (a.dtype is not f16 or b.dtype is not f16 or not (a.is_cuda and b.is_cuda)
            or not (a.is_contiguous() and b.is_contiguous())):
        raise ValueError("operands must be contiguous float16 CUDA tensors")
    return sa[0], sb[0], sa[1]


def _check_matrix(t, rows, cols, dtype_name, what):
    """A device buffer given as a tensor must be a contiguous CUDA matrix of the expected shape and
    dtype (the C ABI sees only its address).  Raw integer addresses are the caller's responsibility."""
    if t is None or isinstance(t, int):
        return
    if (t.shape != (rows, cols) or t.dtype is not getattr(_tm(), dtype_name) or not t.is_cuda
            or not t.is_contiguous()):
        raise ValueError("%s must be a contiguous %s CUDA tensor of shape [%d, %d]" % (what, dtype_name, rows, cols))


def gemm_f16_nt(a, b, c=None, stream=None):
    """C = A . B^T for contiguous fp16 CUDA tensors A [M,K], B [N,K]; returns C [M,N]."""
    m, n, k = _shape(a, b)
    if c is None:
        torch = _tm()
        c = torch.empty((m, n), dtype=torch.float16, device=a.device)
    else:
        _check_matrix(c, m, n, "float16", "c")
    _check(lib().gemm_f16_nt(m, n, k, _ptr(a), _ptr(b), _ptr(c), _stream(stream)), "gemm_f16_nt")
    return c


def gemm_f16_nt_ws(a, b, c, workspace, stream=None):
    m, n, k = _shape(a, b)
    _check_matrix(c, m, n, "float16", "c")
    ws_bytes = 0 if workspace is None else workspace.nbytes
    _check(lib().gemm_f16_nt_ws(m, n, k, _ptr(a), _ptr(b), _ptr(c), _ptr(workspace), ws_bytes,
                                _stream(stream)), "gemm_f16_nt_ws")
    return c


def gemm_f16_nt_run(plan, a, b, c, workspace=None, stream=None):
    m, n, k = int(plan.m), int(plan.n), int(plan.k)
    _check_matrix(a, m, k, "float16", "a")
    if plan.layout == 0:
        _check_matrix(b, n, k, "float16", "b")
        _check_matrix(c, m, n, "float16", "c")
    else:
        _check_matrix(b, k, n, "float16", "b")
        _check_matrix(c, m, n, "float32", "d")
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib().gemm_f16_nt_run(ctypes.byref(plan), _ptr(a), _ptr(b), _ptr(c), _ptr(workspace), ws_bytes,
                                 _stream(stream)), "gemm_f16_nt_run")
    return c


def gemm_f16_nt_noalloc(a, b, c, stream=None):
    """C = A . B^T with the library's built-in scratch array (allocates nothing).

    For callers that may not allocate device memory; calls must not overlap
    on the GPU (they share the one scratch array).  Make the first call on a
    device before any stream capture.
    """
    m, n, k = _shape(a, b)
    if c is None:
        raise ValueError("c must be a contiguous float16 [M,N] CUDA tensor")
    _check_matrix(c, m, n, "float16", "c")
    _check(lib().gemm_f16_nt_noalloc(m, n, k, _ptr(a), _ptr(b), _ptr(c), _stream(stream)), "gemm_f16_nt_noalloc")
    return c


def _shape_kn(a, b_kn):
    if a.dim() != 2 or b_kn.dim() != 2 or a.shape[1] != b_kn.shape[0]:
        raise ValueError("a must be [M,K] and b [K,N]")
    import torch
    for t in (a, b_kn):
        if t.dtype != torch.float16 or not t.is_contiguous() or not t.is_cuda:
            raise ValueError("operands must be contiguous float16 CUDA tensors")
    return a.shape[0], b_kn.shape[1], a.shape[1]


def gemm_f16_nn_f32(a, b_kn, d=None, stream=None):
    """D = A . B for fp16 A [M,K] and B [K,N] (both row-major); D [M,N] float32."""
    import torch
    m, n, k = _shape_kn(a, b_kn)
    if d is None:
        d = torch.empty((m, n), dtype=torch.float32, device=a.device)
    elif tuple(d.shape) != (m, n) or d.dtype != torch.float32 or not d.is_contiguous():
        raise ValueError("d must be a contiguous float32 [M,N] tensor")
    _check(lib().gemm_f16_nn_f32(m, n, k, _ptr(a), _ptr(b_kn), _ptr(d), _stream(stream)), "gemm_f16_nn_f32")
    return d


def gemm_f16_nn_f32_ws(a, b_kn, d, workspace, stream=None):
    m, n, k = _shape_kn(a, b_kn)
    _check_matrix(d, m, n, "float32", "d")
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib().gemm_f16_nn_f32_ws(m, n, k, _ptr(a), _ptr(b_kn), _ptr(d), _ptr(workspace), ws_bytes,
                                    _stream(stream)), "gemm_f16_nn_f32_ws")
    return d


def gemm_f16_nn_f32_plan_ex(m, n, k, variant=-1, raster_width=0, stream_k=-1):
    p = Plan()
    _check(lib().gemm_f16_nn_f32_plan_ex(m, n, k, variant, raster_width, stream_k, ctypes.byref(p)),
           "gemm_f16_nn_f32_plan_ex")
    return p


def gemm_f16_nt_host(a_host, b_host, c_host, a_dev, b_dev, c_dev, workspace=None, stream=None):
    """End-to-end call on host tensors (pinned for asynchronous copies) and device buffers of the same
    shapes; every host and device matrix is checked before the call."""
    m, k = a_host.shape
    n = b_host.shape[0]
    for t, rows, cols, what in ((a_host, m, k, "a_host"), (b_host, n, k, "b_host"), (c_host, m, n, "c_host")):
        if (tuple(t.shape) != (rows, cols) or str(t.dtype) != "torch.float16" or not t.is_contiguous()
                or t.is_cuda):
            raise ValueError("%s must be a contiguous float16 host tensor of shape [%d, %d]" % (what, rows, cols))
    _check_matrix(a_dev, m, k, "float16", "a_dev")
    _check_matrix(b_dev, n, k, "float16", "b_dev")
    _check_matrix(c_dev, m, n, "float16", "c_dev")
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib().gemm_f16_nt_host(m, n, k, _ptr(a_host), _ptr(b_host), _ptr(c_host), _ptr(a_dev), _ptr(b_dev),
                                  _ptr(c_dev), _ptr(workspace), ws_bytes, _stream(stream)), "gemm_f16_nt_host")
    return c_host


def gemm_f16_take_device_error(stream=None):
    """(status, code): GEMM_ERR_TIMEOUT with the recorded code if a kernel gave up a wait."""
    code = ctypes.c_uint32()
    st = lib().gemm_f16_take_device_error(_stream(stream), ctypes.byref(code))
    return st, code.value


def gemm_f16_nt_run_stall_test(plan, a, b, c, skip_fill, wait_limit_cycles, stream=None):
    m, n, k = int(plan.m), int(plan.n), int(plan.k)
    _check_matrix(a, m, k, "float16", "a")
    _check_matrix(b, n, k, "float16", "b")
    _check_matrix(c, m, n, "float16", "c")
    return lib().gemm_f16_nt_run_stall_test(ctypes.byref(plan), _ptr(a), _ptr(b), _ptr(c), skip_fill,
                                            wait_limit_cycles, _stream(stream))


# ------------------------------------------------------ scheduler arithmetic

def gemm_f16_raster_coord(tiles_m, tiles_n, raster_width, tile):
    mb, nb = ctypes.c_int64(), ctypes.c_int64()
    _check(lib().gemm_f16_raster_coord(tiles_m, tiles_n, raster_width, tile, ctypes.byref(mb), ctypes.byref(nb)),
           "gemm_f16_raster_coord")
    return mb.value, nb.value


def gemm_f16_fast_divmod(d, n):
    q, r = ctypes.c_uint32(), ctypes.c_uint32()
    _check(lib().gemm_f16_fast_divmod(d, n, ctypes.byref(q), ctypes.byref(r)), "gemm_f16_fast_divmod")
    return q.value, r.value
