"""Python binding of libgemm_f32 (FP32 GEMM C = A*B on GB300, sm_103a).

Argument marshalling only: every step of the computation runs in the CUDA
library's kernels.  The functions carry the C-ABI's names (include/gemm_f32.h)
and take plain integers for pointers and streams; ``Plan`` adds a small
convenience layer that accepts torch CUDA tensors (PyTorch supplies device
memory and streams, nothing else).

The library is loaded on first use.  There is no fallback: if libgemm_f32.so
is missing or cannot be loaded, every call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libgemm_f32.so")

OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_CUDA, ERR_TIMEOUT, ERR_OOM = range(6)
VARIANT_AUTO, VARIANT_SIMT, VARIANT_TCGEN05, VARIANT_SHORT_M, VARIANT_SHORT_N = 0, 1, 2, 3, 4
STATUS_NAMES = {0: "OK", 1: "INVALID_ARG", 2: "UNSUPPORTED", 3: "CUDA", 4: "TIMEOUT", 5: "OOM"}

EXPORTED = ("gemm_f32_opts_init", "gemm_f32_plan", "gemm_f32_plan_ex", "gemm_f32_run",
            "gemm_f32_run_host", "gemm_f32_check", "gemm_f32_plan_destroy",
            "gemm_f32_plan_describe", "gemm_f32_plan_workspace_bytes", "gemm_f32_status_string",
            "gemm_f32_version", "gemm_f32_plan_kernel_launches", "gemm_f32_trace_enable",
            "gemm_f32_trace_read", "gemm_f32_run_splitk_noalloc", "gemm_f32_plan_batched")


class GemmError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: GEMM_F32_{'ERR_' if status else ''}{STATUS_NAMES.get(status, status)}")
        self.status = status


class Opts(ctypes.Structure):
    """Mirror of gemm_f32_opts."""
    _fields_ = [("variant", ctypes.c_int32), ("tile_m", ctypes.c_int32), ("tile_n", ctypes.c_int32),
                ("stages", ctypes.c_int32), ("split_k", ctypes.c_int32), ("tf32_terms", ctypes.c_int32),
                ("wait_timeout_cycles", ctypes.c_int64), ("debug_withhold_stage", ctypes.c_int32),
                ("separate_syncs", ctypes.c_int32), ("operand_split", ctypes.c_int32),
                ("tile_group", ctypes.c_int32), ("tile_k", ctypes.c_int32), ("host_panels", ctypes.c_int32),
                ("split_reduce", ctypes.c_int32), ("k_slices", ctypes.c_int32),
                ("host_col_blocks", ctypes.c_int32), ("simt_fragments", ctypes.c_int32)]


_lock = threading.Lock()
_lib = None


def load(path: str | None = None):
    """Load libgemm_f32.so (built by software_pipelined_gb300.build)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        p = path or LIB_PATH
        if not os.path.exists(p):
            raise RuntimeError(f"libgemm_f32.so not built ({p}); run software_pipelined_gb300.build.build()")
        lib = ctypes.CDLL(p)
        i64, vp, st = ctypes.c_int64, ctypes.c_void_p, ctypes.c_int
        lib.gemm_f32_opts_init.argtypes = [ctypes.POINTER(Opts)]
        lib.gemm_f32_opts_init.restype = st
        lib.gemm_f32_plan.argtypes = [i64, i64, i64, i64, i64, i64, ctypes.POINTER(vp)]
        lib.gemm_f32_plan.restype = st
        lib.gemm_f32_plan_ex.argtypes = [i64, i64, i64, i64, i64, i64, ctypes.POINTER(Opts),
                                         ctypes.POINTER(vp)]
        lib.gemm_f32_plan_ex.restype = st
        lib.gemm_f32_run.argtypes = [vp, vp, vp, vp, vp]
        lib.gemm_f32_run.restype = st
        lib.gemm_f32_run_host.argtypes = [vp, vp, vp, vp, vp]
        lib.gemm_f32_run_host.restype = st
        lib.gemm_f32_check.argtypes = [vp, vp]
        lib.gemm_f32_check.restype = st
        lib.gemm_f32_plan_destroy.argtypes = [vp]
        lib.gemm_f32_plan_destroy.restype = None
        lib.gemm_f32_plan_describe.argtypes = [vp, ctypes.c_char_p, ctypes.c_size_t]
        lib.gemm_f32_plan_describe.restype = st
        lib.gemm_f32_plan_workspace_bytes.argtypes = [vp]
        lib.gemm_f32_plan_workspace_bytes.restype = ctypes.c_size_t
        lib.gemm_f32_status_string.argtypes = [st]
        lib.gemm_f32_status_string.restype = ctypes.c_char_p
        lib.gemm_f32_version.argtypes = []
        lib.gemm_f32_version.restype = st
        lib.gemm_f32_plan_kernel_launches.argtypes = [vp]
        lib.gemm_f32_plan_kernel_launches.restype = st
        lib.gemm_f32_trace_enable.argtypes = [vp, st]
        lib.gemm_f32_trace_enable.restype = st
        lib.gemm_f32_trace_read.argtypes = [vp, ctypes.POINTER(ctypes.c_float), st, ctypes.POINTER(st)]
        lib.gemm_f32_trace_read.restype = st
        lib.gemm_f32_run_splitk_noalloc.argtypes = [i64, i64, i64, i64, i64, i64, vp, vp, vp,
                                                    ctypes.c_int32, vp]
        lib.gemm_f32_run_splitk_noalloc.restype = st
        lib.gemm_f32_plan_batched.argtypes = [i64, i64, i64, i64, i64, i64, i64, i64, i64, i64,
                                              ctypes.POINTER(Opts), ctypes.POINTER(vp)]
        lib.gemm_f32_plan_batched.restype = st
        _lib = lib
        return lib


# ---------------------------------------------------------------------------
# C-ABI names (plain integers for pointers, plan handles and streams).
# ---------------------------------------------------------------------------

def gemm_f32_opts_init() -> Opts:
    o = Opts()
    load().gemm_f32_opts_init(ctypes.byref(o))
    return o


def gemm_f32_plan(M, N, K, lda, ldb, ldc):
    """Returns (status, plan_handle_int_or_None)."""
    h = ctypes.c_void_p()
    s = load().gemm_f32_plan(M, N, K, lda, ldb, ldc, ctypes.byref(h))
    return s, h.value


def gemm_f32_plan_ex(M, N, K, lda, ldb, ldc, opts: Opts | None):
    h = ctypes.c_void_p()
    s = load().gemm_f32_plan_ex(M, N, K, lda, ldb, ldc, ctypes.byref(opts) if opts is not None else None,
                                ctypes.byref(h))
    return s, h.value


def gemm_f32_plan_batched(M, N, K, lda, ldb, ldc, batch, stride_a, stride_b, stride_c, opts: Opts | None):
    h = ctypes.c_void_p()
    s = load().gemm_f32_plan_batched(M, N, K, lda, ldb, ldc, batch, stride_a, stride_b, stride_c,
                                     ctypes.byref(opts) if opts is not None else None, ctypes.byref(h))
    return s, h.value


def gemm_f32_run(plan, A, B, C, stream=0) -> int:
    return load().gemm_f32_run(plan, A, B, C, stream)


def gemm_f32_run_host(plan, A, B, C, stream=0) -> int:
    return load().gemm_f32_run_host(plan, A, B, C, stream)


def gemm_f32_check(plan, stream=0) -> int:
    return load().gemm_f32_check(plan, stream)


def gemm_f32_plan_destroy(plan) -> None:
    load().gemm_f32_plan_destroy(plan)


def gemm_f32_plan_describe(plan) -> tuple[int, str]:
    buf = ctypes.create_string_buffer(512)
    s = load().gemm_f32_plan_describe(plan, buf, len(buf))
    return s, buf.value.decode()


def gemm_f32_plan_workspace_bytes(plan) -> int:
    return int(load().gemm_f32_plan_workspace_bytes(plan))


def gemm_f32_plan_kernel_launches(plan) -> int:
    return int(load().gemm_f32_plan_kernel_launches(plan))


def gemm_f32_trace_enable(plan, capacity: int) -> int:
    return load().gemm_f32_trace_enable(plan, capacity)


def gemm_f32_trace_read(plan, max_runs: int):
    """Returns (status, list of (split_ms, main_ms, reduce_ms) per recorded run)."""
    buf = (ctypes.c_float * (3 * max(max_runs, 1)))()
    n = ctypes.c_int(0)
    s = load().gemm_f32_trace_read(plan, buf, max_runs, ctypes.byref(n))
    return s, [(buf[3 * i], buf[3 * i + 1], buf[3 * i + 2]) for i in range(n.value)]


def gemm_f32_run_splitk_noalloc(M, N, K, lda, ldb, ldc, A, B, C, split_k, stream=0) -> int:
    """Split-K GEMM whose scratch is the library's fixed device array: no
    allocation at all (see the header for the size limit and the sharing rule)."""
    return load().gemm_f32_run_splitk_noalloc(M, N, K, lda, ldb, ldc, A, B, C, split_k, stream)


def gemm_f32_status_string(s: int) -> str:
    return load().gemm_f32_status_string(s).decode()


def gemm_f32_version() -> int:
    return int(load().gemm_f32_version())


# ---------------------------------------------------------------------------
# Convenience wrapper over torch tensors.
# ---------------------------------------------------------------------------

def _ld(t, rows, cols):
    """Leading dimension (elements) of a row-major 2-D tensor view."""
    if t.dim() != 2:
        raise ValueError("expected a 2-D tensor")
    if cols > 1 and t.stride(1) != 1:
        raise ValueError("inner stride must be 1 (row-major)")
    return t.stride(0) if rows > 1 else max(cols, 1)


class Plan:
    """A gemm_f32 plan for fixed shapes and leading dimensions."""

    def __init__(self, M, N, K, lda=None, ldb=None, ldc=None, *, variant=VARIANT_AUTO, tile_m=0,
                 tile_n=0, stages=0, split_k=0, tf32_terms=0, wait_timeout_cycles=0,
                 debug_withhold_stage=0, separate_syncs=0, operand_split=0, tile_group=0, tile_k=0, host_panels=0,
                 split_reduce=0, k_slices=0, host_col_blocks=0, simt_fragments=0, batch=None,
                 stride_a=0, stride_b=0, stride_c=0):
        self.M, self.N, self.K = int(M), int(N), int(K)
        self.lda = int(lda if lda is not None else max(K, 1))
        self.ldb = int(ldb if ldb is not None else max(N, 1))
        self.ldc = int(ldc if ldc is not None else max(N, 1))
        o = gemm_f32_opts_init()
        o.variant, o.tile_m, o.tile_n, o.stages, o.split_k = variant, tile_m, tile_n, stages, split_k
        o.tf32_terms, o.wait_timeout_cycles = tf32_terms, wait_timeout_cycles
        o.debug_withhold_stage = debug_withhold_stage
        o.separate_syncs = separate_syncs
        o.operand_split = operand_split
        o.tile_group = tile_group
        o.tile_k = tile_k
        o.host_panels = host_panels
        o.split_reduce = split_reduce
        o.k_slices = k_slices
        o.host_col_blocks = host_col_blocks
        o.simt_fragments = simt_fragments
        if batch is None:
            s, h = gemm_f32_plan_ex(self.M, self.N, self.K, self.lda, self.ldb, self.ldc, o)
        else:
            s, h = gemm_f32_plan_batched(self.M, self.N, self.K, self.lda, self.ldb, self.ldc, int(batch),
                                         int(stride_a), int(stride_b), int(stride_c), o)
        if s != OK:
            raise GemmError(s, "gemm_f32_plan_ex" if batch is None else "gemm_f32_plan_batched")
        self.handle = h

    def describe(self) -> str:
        return gemm_f32_plan_describe(self.handle)[1]

    @property
    def workspace_bytes(self) -> int:
        return gemm_f32_plan_workspace_bytes(self.handle)

    @property
    def kernel_launches(self) -> int:
        return gemm_f32_plan_kernel_launches(self.handle)

    def trace_enable(self, capacity: int) -> None:
        s = gemm_f32_trace_enable(self.handle, capacity)
        if s != OK:
            raise GemmError(s, "gemm_f32_trace_enable")

    def trace_read(self, max_runs: int):
        s, runs = gemm_f32_trace_read(self.handle, max_runs)
        if s != OK:
            raise GemmError(s, "gemm_f32_trace_read")
        return runs

    def run_ptr(self, A: int, B: int, C: int, stream: int = 0) -> int:
        return gemm_f32_run(self.handle, A, B, C, stream)

    def run(self, A, B, C, stream=None):
        """C = A @ B for torch float32 CUDA tensors (row-major views)."""
        import torch
        for name, t in (("A", A), ("B", B), ("C", C)):
            if t.dtype != torch.float32 or not t.is_cuda:
                raise TypeError(f"{name} must be a float32 CUDA tensor")
        if tuple(A.shape) != (self.M, self.K) or tuple(B.shape) != (self.K, self.N) or \
                tuple(C.shape) != (self.M, self.N):
            raise ValueError("tensor shapes do not match the plan")
        if _ld(A, self.M, self.K) != self.lda or _ld(B, self.K, self.N) != self.ldb or \
                _ld(C, self.M, self.N) != self.ldc:
            raise ValueError("leading dimensions do not match the plan")
        st = stream if stream is not None else torch.cuda.current_stream()
        s = gemm_f32_run(self.handle, A.data_ptr(), B.data_ptr(), C.data_ptr(), st.cuda_stream)
        if s != OK:
            raise GemmError(s, "gemm_f32_run")
        return C

    def run_host(self, A_ptr: int, B_ptr: int, C_ptr: int, stream: int = 0) -> int:
        return gemm_f32_run_host(self.handle, A_ptr, B_ptr, C_ptr, stream)

    def check(self, stream=None) -> int:
        if stream is None:
            import torch
            stream = torch.cuda.current_stream().cuda_stream
        return gemm_f32_check(self.handle, stream)

    def close(self):
        if getattr(self, "handle", None):
            gemm_f32_plan_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()


def matmul(A, B, out=None, **plan_kwargs):
    """C = A @ B (torch float32 CUDA tensors) through a one-off plan."""
    import torch
    M, K = A.shape
    N = B.shape[1]
    C = out if out is not None else torch.empty((M, N), dtype=torch.float32, device=A.device)
    with Plan(M, N, K, _ld(A, M, K), _ld(B, K, N), _ld(C, M, N), **plan_kwargs) as p:
        p.run(A, B, C)
        torch.cuda.current_stream().synchronize()
    return C
