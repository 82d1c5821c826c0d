"""GB300 (sm_103a) TN GEMM: C = A @ B.T with fp16/bf16 (fp32 accumulate) and int8->int32.

A thin ctypes binding over the C ABI of ``libgemm_gb300.so`` (declared in
``include/gemm.h``), with the same function names.  It only marshals
arguments: every step of the GEMM runs in the library's CUDA kernels.  If the
library is missing or cannot load, every call raises; nothing here computes a
result on the CPU or through another library.
"""
from __future__ import annotations

import ctypes
import functools
import os
import threading

from ._build import LIB_PATH, build_pycall
from ._build import build_library as _build_cuda_library

__all__ = [
    "GEMM_F16", "GEMM_BF16", "GEMM_I8_I32", "GEMM_LAYOUT_TN", "GEMM_LAYOUT_NN", "GEMM_LAYOUT_TT",
    "GEMM_LAYOUT_NT", "LAYOUTS", "GemmError", "Plan",
    "build_library", "gemm_plan_create", "gemm_plan_create_with_config", "gemm_run",
    "gemm_run_bias_act", "ACTIVATIONS", "tma_intensity_run", "TMA_MODES",
    "gemm_plan_check", "gemm_plan_destroy", "gemm_plan_get_config", "gemm_plan_get_launch",
    "gemm_plan_set_timeout",
    "gemm_plan_set_wait_test",
    "gemm_select_config", "gemm_tile_coords", "gemm_workspace_bytes", "gemm_status_string",
    "gemm_abi_version", "gemm_launch_empty", "gemm_run_splitk_noalloc", "gemm_noalloc_check",
    "gemm_noalloc_set_wait_test", "gemm_probe_mma_rate", "library", "DTYPES",
]

GEMM_F16, GEMM_BF16, GEMM_I8_I32 = 0, 1, 2
GEMM_LAYOUT_TN, GEMM_LAYOUT_NN, GEMM_LAYOUT_TT, GEMM_LAYOUT_NT = 0, 1, 2, 3
LAYOUTS = {"TN": GEMM_LAYOUT_TN, "NN": GEMM_LAYOUT_NN, "TT": GEMM_LAYOUT_TT, "NT": GEMM_LAYOUT_NT}
DTYPES = {"f16": GEMM_F16, "bf16": GEMM_BF16, "i8": GEMM_I8_I32}

STATUS_NAMES = {
    0: "GEMM_OK", 1: "GEMM_ERR_INVALID_ARG", 2: "GEMM_ERR_UNSUPPORTED", 3: "GEMM_ERR_ALIGNMENT",
    4: "GEMM_ERR_NO_DEVICE", 5: "GEMM_ERR_ARCH", 6: "GEMM_ERR_OOM", 7: "GEMM_ERR_TENSORMAP",
    8: "GEMM_ERR_LAUNCH", 9: "GEMM_ERR_DEVICE_TIMEOUT", 10: "GEMM_ERR_CUDA",
    11: "GEMM_ERR_SCRATCH_LIMIT",
}


class GemmError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        self.name = STATUS_NAMES.get(status, str(status))
        super().__init__("%s%s" % (what + ": " if what else "", gemm_status_string(status)))


class gemm_config_t(ctypes.Structure):
    _fields_ = [("block_n", ctypes.c_int32), ("stages", ctypes.c_int32),
                ("split_k", ctypes.c_int32), ("raster_group", ctypes.c_int32),
                ("max_ctas", ctypes.c_int32), ("split_mode", ctypes.c_int32),
                ("cta_pair", ctypes.c_int32), ("direct_store", ctypes.c_int32),
                ("multicast", ctypes.c_int32), ("l2_prefetch", ctypes.c_int32),
                ("kblocks_per_stage", ctypes.c_int32)]

    def as_dict(self):
        return {f: int(getattr(self, f)) for f, _ in self._fields_}


_lock = threading.Lock()
_lib = None
_pycall = None   # CPython entry points for gemm_run / gemm_launch_empty, when built


def build_library(force: bool = False, verbose: bool = False, ptxas_info: bool = False) -> str:
    """Build libgemm_gb300.so (nvcc, sm_103a) if stale, and the CPython entry points
    for the per-call functions (gcc); return the library's path."""
    path = _build_cuda_library(force=force, verbose=verbose, ptxas_info=ptxas_info)
    build_pycall(force=force)
    return path


def library() -> ctypes.CDLL:
    """The loaded C-ABI library (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError("libgemm_gb300.so is not built (run "
                                   "dense_gemm_hgemm_gb300.build_library())")
            lib = ctypes.CDLL(LIB_PATH)
            i64, i32, vp = ctypes.c_int64, ctypes.c_int32, ctypes.c_void_p
            cfgp = ctypes.POINTER(gemm_config_t)
            sig = {
                "gemm_plan_create": ([i64, i64, i64, i32, i32, ctypes.POINTER(vp)], i32),
                "gemm_plan_create_with_config": ([i64, i64, i64, i32, i32, cfgp,
                                                  ctypes.POINTER(vp)], i32),
                "gemm_run": ([vp, vp, vp, vp, vp], i32),
                "gemm_run_bias_act": ([vp, vp, vp, vp, vp, i32, vp], i32),
                "gemm_plan_check": ([vp, vp], i32),
                "gemm_plan_destroy": ([vp], i32),
                "gemm_plan_get_config": ([vp, cfgp], i32),
                "gemm_plan_get_launch": ([vp, ctypes.POINTER(i32), ctypes.POINTER(i32),
                                          ctypes.POINTER(i32)], i32),
                "gemm_plan_set_timeout": ([vp, ctypes.c_uint64], i32),
                "gemm_plan_set_wait_test": ([vp, ctypes.c_uint32], i32),
                "gemm_select_config": ([i64, i64, i64, i32, i32, cfgp], i32),
                "gemm_tile_coords": ([i64, i64, i32, i64, ctypes.POINTER(i64),
                                      ctypes.POINTER(i64)], i32),
                "gemm_workspace_bytes": ([i64, i64, i64, i32, cfgp, ctypes.POINTER(ctypes.c_size_t)], i32),
                "gemm_status_string": ([i32], ctypes.c_char_p),
                "gemm_abi_version": ([], i32),
                "gemm_launch_empty": ([i32, vp], i32),
                "gemm_run_splitk_noalloc": ([i64, i64, i64, i32, i32, vp, vp, vp, vp], i32),
                "gemm_noalloc_check": ([vp], i32),
                "gemm_noalloc_set_wait_test": ([ctypes.c_uint32, ctypes.c_uint64], i32),
                "gemm_probe_mma_rate": ([i32, i32, vp, vp, vp, vp], i32),
                "tma_intensity_run": ([i32, i32, ctypes.c_float, ctypes.c_float, vp, vp, i64, i32,
                                       vp, vp], i32),
            }
            for name, (args, res) in sig.items():
                fn = getattr(lib, name)
                fn.argtypes = args
                fn.restype = res
            global _pycall
            try:
                from . import _gemm_pycall as pc
                addr = lambda f: ctypes.cast(f, ctypes.c_void_p).value
                pc.set_targets(addr(lib.gemm_run), addr(lib.gemm_launch_empty))
                _pycall = pc
            except ImportError:
                _pycall = None
            _lib = lib
    return _lib


def _check(status: int, what: str):
    if status != 0:
        raise GemmError(status, what)


def _dtype_code(dtype) -> int:
    return DTYPES[dtype] if isinstance(dtype, str) else int(dtype)


def _ptr(x) -> int | None:
    """Device address of a torch tensor (or an int address)."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _config(cfg) -> gemm_config_t:
    if isinstance(cfg, gemm_config_t):
        return cfg
    c = gemm_config_t()
    c.block_n = int(cfg.get("block_n", 128))
    c.stages = int(cfg.get("stages", 0))
    c.split_k = int(cfg.get("split_k", 1))
    c.raster_group = int(cfg.get("raster_group", 16))
    c.max_ctas = int(cfg.get("max_ctas", 0))
    c.split_mode = int(cfg.get("split_mode", 0))
    c.cta_pair = int(cfg.get("cta_pair", 0))
    c.direct_store = int(cfg.get("direct_store", 0))
    c.multicast = int(cfg.get("multicast", 0))
    c.l2_prefetch = int(cfg.get("l2_prefetch", 0))
    c.kblocks_per_stage = int(cfg.get("kblocks_per_stage", 0))
    return c


def gemm_status_string(status: int) -> str:
    return library().gemm_status_string(int(status)).decode()


def gemm_abi_version() -> int:
    return int(library().gemm_abi_version())


def gemm_launch_empty(grid: int, stream=None) -> None:
    if library() is not None and _pycall is not None:
        _check(_pycall.launch_empty(int(grid), _stream(stream) or 0), "gemm_launch_empty")
        return
    _check(library().gemm_launch_empty(int(grid), _stream(stream)), "gemm_launch_empty")


def gemm_run_splitk_noalloc(M: int, N: int, K: int, dtype, split_k: int, A, B, C,
                            stream=None) -> None:
    """Split-K C = A @ B.T that allocates no device memory: its scratch is a fixed
    16 MiB array inside the library (for callers that may not allocate; see
    include/gemm.h for the size limit and the sharing rules)."""
    _check(library().gemm_run_splitk_noalloc(M, N, K, _dtype_code(dtype), int(split_k), _ptr(A),
                                             _ptr(B), _ptr(C), _stream(stream)),
           "gemm_run_splitk_noalloc")


def gemm_noalloc_check(stream=None) -> None:
    """Synchronise `stream`; raise GemmError(GEMM_ERR_DEVICE_TIMEOUT) if a no-alloc call
    since the last check gave up on a wait (the record is cleared by this call)."""
    _check(library().gemm_noalloc_check(_stream(stream)), "gemm_noalloc_check")


def gemm_noalloc_set_wait_test(extra_bytes: int, timeout_ns: int = 0) -> None:
    """Failure-test hook of the no-alloc path (process-wide): ring slots wait for
    `extra_bytes` that never arrive; 0 restores normal operation."""
    _check(library().gemm_noalloc_set_wait_test(int(extra_bytes), int(timeout_ns)),
           "gemm_noalloc_set_wait_test")


def gemm_probe_mma_rate(grid: int, iters: int, cycles, ns, error_word, stream=None) -> None:
    """Back-to-back tcgen05.mma (M=128, N=256, K=16) issue-rate probe: per CTA, SM cycles
    and ns from the first issue to completion (see include/gemm_probe.h)."""
    _check(library().gemm_probe_mma_rate(int(grid), int(iters), _ptr(cycles), _ptr(ns),
                                         _ptr(error_word), _stream(stream)), "gemm_probe_mma_rate")


TMA_MODES = {"sync": 0, "bulk1d": 1, "tensor2d": 2, "pipe2": 3}


def tma_intensity_run(mode, fma_iters: int, a: float, b: float, x, y, cols: int = 2048,
                      error_word=None, stream=None) -> None:
    """The TMA load-mode x FMA-intensity experiment (see include/tma_intensity.h)."""
    m = TMA_MODES[mode] if isinstance(mode, str) else int(mode)
    _check(library().tma_intensity_run(m, int(fma_iters), float(a), float(b), _ptr(x), _ptr(y),
                                       x.numel() if hasattr(x, "numel") else int(x), int(cols),
                                       _ptr(error_word), _stream(stream)), "tma_intensity_run")


def gemm_plan_create(M: int, N: int, K: int, dtype="f16", layout: int = GEMM_LAYOUT_TN) -> int:
    h = ctypes.c_void_p()
    _check(library().gemm_plan_create(M, N, K, _dtype_code(dtype), layout, ctypes.byref(h)),
           "gemm_plan_create")
    return h.value


def gemm_plan_create_with_config(M, N, K, dtype, config, layout: int = GEMM_LAYOUT_TN) -> int:
    h = ctypes.c_void_p()
    c = _config(config)
    _check(library().gemm_plan_create_with_config(M, N, K, _dtype_code(dtype), layout,
                                                  ctypes.byref(c), ctypes.byref(h)),
           "gemm_plan_create_with_config")
    return h.value


def gemm_run(plan: int, A, B, C, stream=None) -> None:
    lib = library()
    if _pycall is not None:
        _check(_pycall.run(plan or 0, _ptr(A) or 0, _ptr(B) or 0, _ptr(C) or 0,
                           _stream(stream) or 0), "gemm_run")
        return
    _check(lib.gemm_run(plan, _ptr(A), _ptr(B), _ptr(C), _stream(stream)), "gemm_run")


ACT_NONE, ACT_RELU, ACT_GELU, ACT_SILU = 0, 1, 2, 3
ACTIVATIONS = {"none": ACT_NONE, "relu": ACT_RELU, "gelu": ACT_GELU, "silu": ACT_SILU}


def gemm_run_bias_act(plan: int, A, B, C, bias=None, act=ACT_NONE, stream=None) -> None:
    """C = act(A @ B.T + bias) with the bias (N fp32 values or None) and activation fused."""
    a = ACTIVATIONS[act] if isinstance(act, str) else int(act)
    _check(library().gemm_run_bias_act(plan, _ptr(A), _ptr(B), _ptr(C), _ptr(bias), a,
                                       _stream(stream)), "gemm_run_bias_act")


def gemm_plan_check(plan: int, stream=None) -> None:
    _check(library().gemm_plan_check(plan, _stream(stream)), "gemm_plan_check")


def gemm_plan_destroy(plan: int) -> None:
    _check(library().gemm_plan_destroy(plan), "gemm_plan_destroy")


def gemm_plan_get_config(plan: int) -> dict:
    c = gemm_config_t()
    _check(library().gemm_plan_get_config(plan, ctypes.byref(c)), "gemm_plan_get_config")
    return c.as_dict()


def gemm_plan_get_launch(plan: int) -> dict:
    """{"grid", "cluster", "max_active_clusters"} of the plan's GEMM kernel launch."""
    g, c, n = ctypes.c_int32(), ctypes.c_int32(), ctypes.c_int32()
    _check(library().gemm_plan_get_launch(plan, ctypes.byref(g), ctypes.byref(c), ctypes.byref(n)),
           "gemm_plan_get_launch")
    return {"grid": g.value, "cluster": c.value, "max_active_clusters": n.value}


def gemm_plan_set_timeout(plan: int, ns: int) -> None:
    _check(library().gemm_plan_set_timeout(plan, int(ns)), "gemm_plan_set_timeout")


def gemm_plan_set_wait_test(plan: int, extra_bytes: int) -> None:
    _check(library().gemm_plan_set_wait_test(plan, int(extra_bytes)), "gemm_plan_set_wait_test")


def gemm_select_config(M, N, K, dtype, num_sms: int) -> dict:
    c = gemm_config_t()
    _check(library().gemm_select_config(M, N, K, _dtype_code(dtype), num_sms, ctypes.byref(c)),
           "gemm_select_config")
    return c.as_dict()


def gemm_tile_coords(m_blocks: int, n_blocks: int, raster_group: int, tile: int):
    m = ctypes.c_int64()
    n = ctypes.c_int64()
    _check(library().gemm_tile_coords(m_blocks, n_blocks, raster_group, tile, ctypes.byref(m),
                                      ctypes.byref(n)), "gemm_tile_coords")
    return m.value, n.value


def gemm_workspace_bytes(M, N, K, dtype, config) -> int:
    b = ctypes.c_size_t()
    c = _config(config)
    _check(library().gemm_workspace_bytes(M, N, K, _dtype_code(dtype), ctypes.byref(c),
                                          ctypes.byref(b)), "gemm_workspace_bytes")
    return int(b.value)


def _plan_run(box, A, B, C, stream=None, bias=None, act=ACT_NONE) -> None:
    """Plan.run for the plan handle in box[0] (None once the plan is closed)."""
    handle = box[0]
    if bias is not None or act not in (ACT_NONE, "none"):
        gemm_run_bias_act(handle, A, B, C, bias, act, stream)
        return
    pc = _pycall
    if pc is None:
        gemm_run(handle, A, B, C, stream)
        return
    try:   # tensors and a stream object
        st = pc.run(handle or 0, A.data_ptr(), B.data_ptr(), C.data_ptr(), stream.cuda_stream)
    except AttributeError:   # addresses or a stream handle given as ints, or no stream
        st = pc.run(handle or 0, _ptr(A) or 0, _ptr(B) or 0, _ptr(C) or 0, _stream(stream) or 0)
    if st:
        raise GemmError(st, "gemm_run")


class Plan:
    """Owning wrapper of a plan handle: ``with Plan(M, N, K, "f16") as p: p.run(A, B, C)``.

    ``run(A, B, C, stream)`` with tensors and a stream object, the per-call form of
    a serving loop, goes straight to gemm_run through a C-level runner bound to the
    plan (argument marshalling only); every other form takes the general path."""

    def __init__(self, M: int, N: int, K: int, dtype="f16", config=None, layout=GEMM_LAYOUT_TN):
        self.M, self.N, self.K, self.dtype = M, N, K, dtype
        lay = LAYOUTS[layout] if isinstance(layout, str) else int(layout)
        self.handle = (gemm_plan_create(M, N, K, dtype, lay) if config is None
                       else gemm_plan_create_with_config(M, N, K, dtype, config, lay))
        self._box = [self.handle]
        runner = getattr(_pycall, "Runner", None)
        if runner is not None:   # an instance attribute: shadows the method below
            self.run = runner(self._box, functools.partial(_plan_run, self._box))

    @property
    def config(self) -> dict:
        return gemm_plan_get_config(self.handle)

    @property
    def launch(self) -> dict:
        return gemm_plan_get_launch(self.handle)

    def run(self, A, B, C, stream=None, bias=None, act=ACT_NONE) -> None:
        """C = A @ B.T (optionally act(A @ B.T + bias)) on `stream`."""
        _plan_run(self._box, A, B, C, stream, bias, act)

    def check(self, stream=None) -> None:
        gemm_plan_check(self.handle, stream)

    def set_timeout(self, ns: int) -> None:
        gemm_plan_set_timeout(self.handle, ns)

    def set_wait_test(self, extra_bytes: int) -> None:
        gemm_plan_set_wait_test(self.handle, extra_bytes)

    def close(self) -> None:
        if self.handle:
            self._box[0] = None   # the runner falls back to the general path, which refuses
            gemm_plan_destroy(self.handle)
            self.handle = None

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
