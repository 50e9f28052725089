"""ctypes binding of ``libdmuon.so`` (argument marshalling only).

Every function here has the name of the C entry point it wraps
(``include/dmuon.h``) and does nothing but convert arguments and raise
``DmuonError`` on a non-zero status.  All arithmetic runs in the library's
CUDA kernels; there is no fallback: if the library is missing, loading it
raises.
"""

from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libdmuon.so")

DMUON_OK = 0
DMUON_ERR_INVALID_ARG = 1
DMUON_ERR_RANK_LT2 = 2
DMUON_ERR_SHAPE = 3
DMUON_ERR_DTYPE = 4
DMUON_ERR_CUDA = 5
DMUON_ERR_TIMEOUT = 6
DMUON_ERR_NOMEM = 7
DMUON_ERR_UNSUPPORTED = 8

DMUON_DTYPE_F32 = 0
DMUON_DTYPE_BF16 = 1

DMUON_FLAG_NESTEROV = 1
DMUON_FLAG_FP32_NS = 2

EXPORTED = (
    "dmuon_status_string", "dmuon_last_error", "dmuon_lpt_assign", "dmuon_context_create",
    "dmuon_context_destroy", "dmuon_muon_step", "dmuon_adamw_step", "dmuon_sync",
    "dmuon_selftest_wait_timeout", "dmuon_set_tuning", "dmuon_kernel_launches", "dmuon_profile",
    "dmuon_profile_read", "dmuon_muon_step_noalloc", "dmuon_lpt_assign_layered", "dmuon_step_host",
    "dmuon_muon_step_noalloc_sync", "dmuon_profile_host_timeline", "dmuon_context_set_tuning",
)

KERNEL_KINDS = ("momentum", "norm", "ns_gram", "ns_poly", "ns_combine", "update", "adamw")


class DmuonError(RuntimeError):
    def __init__(self, status, message):
        super().__init__(f"dmuon status {status}: {message}")
        self.status = status


class DmuonMatrix(ctypes.Structure):
    _fields_ = [
        ("rank", ctypes.c_int32),
        ("grad_dtype", ctypes.c_int32),
        ("shape", ctypes.c_int64 * 4),
        ("master", ctypes.c_void_p),
        ("momentum", ctypes.c_void_p),
        ("grad", ctypes.c_void_p),
        ("param_bf16", ctypes.c_void_p),
    ]


class DmuonVector(ctypes.Structure):
    _fields_ = [
        ("numel", ctypes.c_int64),
        ("grad_dtype", ctypes.c_int32),
        ("reserved", ctypes.c_int32),
        ("master", ctypes.c_void_p),
        ("exp_avg", ctypes.c_void_p),
        ("exp_avg_sq", ctypes.c_void_p),
        ("grad", ctypes.c_void_p),
        ("param_bf16", ctypes.c_void_p),
    ]


class DmuonHostIO(ctypes.Structure):
    _fields_ = [("grad_host", ctypes.c_void_p), ("param_host", ctypes.c_void_p)]


class DmuonMuonHparams(ctypes.Structure):
    _fields_ = [
        ("lr", ctypes.c_float), ("momentum", ctypes.c_float), ("wd", ctypes.c_float),
        ("ns_steps", ctypes.c_int32), ("a", ctypes.c_float), ("b", ctypes.c_float), ("c", ctypes.c_float),
        ("flags", ctypes.c_uint32),
    ]


class DmuonAdamwHparams(ctypes.Structure):
    _fields_ = [
        ("lr", ctypes.c_float), ("beta1", ctypes.c_float), ("beta2", ctypes.c_float), ("eps", ctypes.c_float),
        ("wd", ctypes.c_float), ("reserved", ctypes.c_int32), ("step", ctypes.c_int64),
    ]


_lib = None


def load_library(path=LIB_PATH):
    """Load the library once and declare every signature.  Raises if absent."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(
            f"{path} is missing: build it first (python -c 'import __graft_entry__ as g; g.build()')")
    lib = ctypes.CDLL(path)
    vp, i32, i64, f32 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float
    sig = {
        "dmuon_status_string": (ctypes.c_char_p, [ctypes.c_int]),
        "dmuon_last_error": (ctypes.c_char_p, []),
        "dmuon_lpt_assign": (ctypes.c_int, [ctypes.POINTER(i64), i32, i32, ctypes.POINTER(i32),
                                            ctypes.POINTER(i64)]),
        "dmuon_lpt_assign_layered": (ctypes.c_int, [ctypes.POINTER(i64), ctypes.POINTER(i32), i32, i32, i64,
                                                    ctypes.POINTER(i32), ctypes.POINTER(i64)]),
        "dmuon_context_create": (ctypes.c_int, [ctypes.POINTER(vp), i32]),
        "dmuon_context_destroy": (ctypes.c_int, [vp]),
        "dmuon_muon_step": (ctypes.c_int, [vp, ctypes.POINTER(DmuonMatrix), i32, f32, f32, f32, i32,
                                           f32, f32, f32, ctypes.c_uint32, vp]),
        "dmuon_adamw_step": (ctypes.c_int, [vp, ctypes.POINTER(DmuonVector), i32, f32, f32, f32, f32,
                                            f32, i64, vp]),
        "dmuon_sync": (ctypes.c_int, [vp, vp]),
        "dmuon_selftest_wait_timeout": (ctypes.c_int, [vp, i32, vp]),
        "dmuon_set_tuning": (ctypes.c_int, [i32, i32]),
        "dmuon_context_set_tuning": (ctypes.c_int, [vp, i32, i32]),
        "dmuon_kernel_launches": (i64, [vp]),
        "dmuon_profile": (ctypes.c_int, [vp, i32]),
        "dmuon_profile_read": (ctypes.c_int, [vp, ctypes.POINTER(ctypes.c_double), ctypes.POINTER(i64)]),
        "dmuon_muon_step_noalloc": (ctypes.c_int, [ctypes.POINTER(DmuonMatrix), f32, f32, f32, i32, f32, f32,
                                                   f32, ctypes.c_uint32, vp]),
        "dmuon_muon_step_noalloc_sync": (ctypes.c_int, [vp]),
        "dmuon_profile_host_timeline": (ctypes.c_int, [vp, ctypes.POINTER(ctypes.c_double), i32,
                                                       ctypes.POINTER(i32)]),
        "dmuon_step_host": (ctypes.c_int, [vp, ctypes.POINTER(DmuonMatrix), ctypes.POINTER(DmuonHostIO), i32,
                                           ctypes.POINTER(DmuonMuonHparams), ctypes.POINTER(DmuonVector),
                                           ctypes.POINTER(DmuonHostIO), i32, ctypes.POINTER(DmuonAdamwHparams),
                                           i32, vp]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def _check(status):
    if status != DMUON_OK:
        lib = load_library()
        raise DmuonError(status, lib.dmuon_last_error().decode(errors="replace"))


def _stream_handle(stream):
    if stream is None:
        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, torch.cuda.Stream):
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _grad_dtype(t):
    if t.dtype == torch.bfloat16:
        return DMUON_DTYPE_BF16
    if t.dtype == torch.float32:
        return DMUON_DTYPE_F32
    return -1


# ------------------------------------------------------------------ wrappers

def dmuon_status_string(status):
    return load_library().dmuon_status_string(int(status)).decode()


def dmuon_lpt_assign(sizes, n_slots):
    """LPT assignment of int64 ``sizes`` to ``n_slots`` slots: (slots, loads)."""
    lib = load_library()
    n = len(sizes)
    arr = (ctypes.c_int64 * max(n, 1))(*[int(s) for s in sizes])
    out = (ctypes.c_int32 * max(n, 1))()
    loads = (ctypes.c_int64 * max(int(n_slots), 1))()
    _check(lib.dmuon_lpt_assign(arr, n, int(n_slots), out, loads))
    return [out[i] for i in range(n)], [loads[i] for i in range(int(n_slots))]


def dmuon_lpt_assign_layered(sizes, layers, n_slots, small_threshold=5_000_000):
    """Layer-aware LPT (same-layer distinct slots, small items of a layer
    merged): (slots, loads)."""
    lib = load_library()
    n = len(sizes)
    if len(layers) != n:
        raise ValueError("one layer id per item")
    arr = (ctypes.c_int64 * max(n, 1))(*[int(s) for s in sizes])
    lay = (ctypes.c_int32 * max(n, 1))(*[int(x) for x in layers])
    out = (ctypes.c_int32 * max(n, 1))()
    loads = (ctypes.c_int64 * max(int(n_slots), 1))()
    _check(lib.dmuon_lpt_assign_layered(arr, lay, n, int(n_slots), int(small_threshold), out, loads))
    return [out[i] for i in range(n)], [loads[i] for i in range(int(n_slots))]


def dmuon_context_create(device=0):
    lib = load_library()
    h = ctypes.c_void_p()
    _check(lib.dmuon_context_create(ctypes.byref(h), int(device)))
    return h


def dmuon_context_destroy(ctx):
    _check(load_library().dmuon_context_destroy(ctx))


def matrix_desc(master, momentum, grad, param_bf16=None, shape=None):
    """DmuonMatrix for contiguous torch tensors (no checks beyond dtype/shape)."""
    d = DmuonMatrix()
    shp = tuple(shape if shape is not None else master.shape)
    d.rank = len(shp)
    for i, s in enumerate(shp[:4]):
        d.shape[i] = int(s)
    d.grad_dtype = _grad_dtype(grad)
    d.master = _ptr(master)
    d.momentum = _ptr(momentum)
    d.grad = _ptr(grad)
    d.param_bf16 = _ptr(param_bf16)
    return d


def vector_desc(master, exp_avg, exp_avg_sq, grad, param_bf16=None):
    d = DmuonVector()
    d.numel = master.numel()
    d.grad_dtype = _grad_dtype(grad)
    d.master = _ptr(master)
    d.exp_avg = _ptr(exp_avg)
    d.exp_avg_sq = _ptr(exp_avg_sq)
    d.grad = _ptr(grad)
    d.param_bf16 = _ptr(param_bf16)
    return d


def descriptor_array(descs, cls):
    arr = (cls * max(len(descs), 1))()
    for i, d in enumerate(descs):
        arr[i] = d
    return arr


def dmuon_muon_step(ctx, mats, lr, momentum, wd, ns_steps, a, b, c, flags=DMUON_FLAG_NESTEROV,
                    stream=None):
    """``mats``: a list of DmuonMatrix or a ctypes array of them."""
    lib = load_library()
    if isinstance(mats, (list, tuple)):
        n = len(mats)
        mats = descriptor_array(mats, DmuonMatrix)
    else:
        n = len(mats)
    _check(lib.dmuon_muon_step(ctx, mats, n, float(lr), float(momentum), float(wd), int(ns_steps),
                               float(a), float(b), float(c), int(flags), _stream_handle(stream)))


def dmuon_adamw_step(ctx, vecs, lr, beta1, beta2, eps, wd, step, stream=None):
    lib = load_library()
    if isinstance(vecs, (list, tuple)):
        n = len(vecs)
        vecs = descriptor_array(vecs, DmuonVector)
    else:
        n = len(vecs)
    _check(lib.dmuon_adamw_step(ctx, vecs, n, float(lr), float(beta1), float(beta2), float(eps),
                                float(wd), int(step), _stream_handle(stream)))


def dmuon_sync(ctx, stream=None):
    _check(load_library().dmuon_sync(ctx, _stream_handle(stream)))


def dmuon_selftest_wait_timeout(ctx, timeout_us, stream=None):
    _check(load_library().dmuon_selftest_wait_timeout(ctx, int(timeout_us), _stream_handle(stream)))


def dmuon_set_tuning(key, value):
    """Process-wide default of one tuning key (contexts created later copy it)."""
    _check(load_library().dmuon_set_tuning(int(key), int(value)))


def dmuon_context_set_tuning(ctx, key, value):
    """One tuning key of one context."""
    _check(load_library().dmuon_context_set_tuning(ctx, int(key), int(value)))


def dmuon_kernel_launches(ctx):
    return int(load_library().dmuon_kernel_launches(ctx))


def dmuon_profile(ctx, enable):
    _check(load_library().dmuon_profile(ctx, 1 if enable else 0))


def dmuon_profile_read(ctx):
    """{kind: (total device ms, launches)} since the previous read."""
    n = len(KERNEL_KINDS)
    ms = (ctypes.c_double * n)()
    cnt = (ctypes.c_int64 * n)()
    _check(load_library().dmuon_profile_read(ctx, ms, cnt))
    return {k: (ms[i], cnt[i]) for i, k in enumerate(KERNEL_KINDS)}


def dmuon_profile_host_timeline(ctx):
    """Timeline of the last host-buffer step made while profiling (ms since
    its start): {"h2d_done", "end", "groups": [(h2d_done, compute_done,
    d2h_done), ...]}, or None if none was recorded."""
    lib = load_library()
    n = ctypes.c_int32()
    cap = 2 + 3 * 64
    buf = (ctypes.c_double * cap)()
    _check(lib.dmuon_profile_host_timeline(ctx, buf, cap, ctypes.byref(n)))
    if n.value == 0:
        return None
    return {"h2d_done": buf[0], "end": buf[1],
            "groups": [tuple(buf[2 + 3 * g + k] for k in range(3)) for g in range(n.value)]}


def dmuon_muon_step_noalloc(mat, lr, momentum, wd, ns_steps, a, b, c, flags=DMUON_FLAG_NESTEROV,
                            stream=None):
    """Muon step of one tensor with all scratch in the library's static device
    array (no device allocation).  ``mat`` is one DmuonMatrix."""
    _check(load_library().dmuon_muon_step_noalloc(
        ctypes.byref(mat), float(lr), float(momentum), float(wd), int(ns_steps), float(a), float(b),
        float(c), int(flags), _stream_handle(stream)))


def dmuon_muon_step_noalloc_sync(stream=None):
    """Wait for ``stream``; raise DmuonError(DMUON_ERR_TIMEOUT) if a bounded
    device-side wait of the allocation-free entry point ran out."""
    _check(load_library().dmuon_muon_step_noalloc_sync(_stream_handle(stream)))


def muon_hparams(lr, momentum, wd, ns_steps=5, a=3.4445, b=-4.7750, c=2.0315, nesterov=True, fp32_ns=False):
    flags = (DMUON_FLAG_NESTEROV if nesterov else 0) | (DMUON_FLAG_FP32_NS if fp32_ns else 0)
    return DmuonMuonHparams(float(lr), float(momentum), float(wd), int(ns_steps), float(a), float(b), float(c),
                            flags)


def adamw_hparams(lr, beta1, beta2, eps, wd, step):
    return DmuonAdamwHparams(float(lr), float(beta1), float(beta2), float(eps), float(wd), 0, int(step))


def dmuon_step_host(ctx, mats, mat_io, muon, vecs=None, vec_io=None, adamw=None, n_groups=8, stream=None):
    """``mats``/``vecs``: ctypes arrays (or lists) of DmuonMatrix/DmuonVector;
    ``mat_io``/``vec_io``: matching arrays of DmuonHostIO; ``muon``/``adamw``:
    DmuonMuonHparams/DmuonAdamwHparams (or None when the list is empty)."""
    lib = load_library()
    vecs = [] if vecs is None else vecs
    vec_io = [] if vec_io is None else vec_io
    n_m, n_v = len(mats), len(vecs)
    if len(mat_io) != n_m or len(vec_io) != n_v:
        raise ValueError("one host io entry per tensor")
    if isinstance(mats, (list, tuple)):
        mats = descriptor_array(mats, DmuonMatrix)
    if isinstance(mat_io, (list, tuple)):
        mat_io = descriptor_array(mat_io, DmuonHostIO)
    if isinstance(vecs, (list, tuple)):
        vecs = descriptor_array(vecs, DmuonVector)
    if isinstance(vec_io, (list, tuple)):
        vec_io = descriptor_array(vec_io, DmuonHostIO)
    _check(lib.dmuon_step_host(ctx, mats, mat_io, n_m, ctypes.byref(muon) if muon is not None else None,
                               vecs, vec_io, n_v, ctypes.byref(adamw) if adamw is not None else None,
                               int(n_groups), _stream_handle(stream)))
