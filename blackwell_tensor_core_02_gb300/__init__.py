"""GB300 (sm_103a) fp16 GEMM  D = A·Bᵀ  — Python binding of the C ABI.

Argument marshalling only: every step of the computation runs in the CUDA
library ``_build/libgemm_f16.so`` (see ``include/gemm_f16.h``). PyTorch only
supplies device memory and streams. There is no fallback: if the library
cannot be built or loaded, every call raises.

    import torch, blackwell_tensor_core_02_gb300 as g
    A = torch.randn(4096, 4096, device="cuda", dtype=torch.float16)
    B = torch.randn(4096, 4096, device="cuda", dtype=torch.float16)   # N×K
    D = g.gemm_f16_nt(A, B)                                          # M×N = A @ B.T
"""
from __future__ import annotations

import ctypes
import threading

from . import build as _build

__all__ = [
    "GemmError", "Options", "load", "gemm_f16_nt", "gemm_f16_nt_ptr", "gemm_f16_nt_supported",
    "gemm_f16_nt_host", "HostPipeline", "workspace_size", "WorkItem", "last_device_status", "status_string", "schedule", "cta_origin", "pipeline_trace", "STATUS",
]

STATUS = {
    0: "GEMM_OK", -1: "GEMM_ERR_INVALID_ARG", -2: "GEMM_ERR_UNSUPPORTED_SHAPE", -3: "GEMM_ERR_MISALIGNED",
    -4: "GEMM_ERR_NO_DEVICE", -5: "GEMM_ERR_ARCH", -6: "GEMM_ERR_LAUNCH", -7: "GEMM_ERR_DEVICE_TIMEOUT",
    -8: "GEMM_ERR_CUDA", -9: "GEMM_ERR_SCRATCH_LIMIT", -10: "GEMM_ERR_DEVICE_BOUNDS",
}


class GemmError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {status_string(code)} ({code})")


class WorkItem(ctypes.Structure):
    """Mirror of ``gemm_f16_work_item``."""
    _fields_ = [(n, ctypes.c_int64) for n in ("m_idx", "n_idx", "n_off", "n_len", "slice", "kt_begin", "kt_end")]


class LaunchInfo(ctypes.Structure):
    """Mirror of ``gemm_f16_launch_info``."""
    _fields_ = [("cta_group", ctypes.c_int32), ("consumers", ctypes.c_int32), ("block_n", ctypes.c_int32),
                ("split_k", ctypes.c_int32), ("block_m", ctypes.c_int32), ("stages", ctypes.c_int32),
                ("clusters", ctypes.c_int64), ("work_items", ctypes.c_int64), ("workspace_bytes", ctypes.c_int64),
                ("cluster_k", ctypes.c_int32)]


class Options(ctypes.Structure):
    """Mirror of ``gemm_f16_options`` (zero fields mean defaults)."""
    _fields_ = [("cta_group", ctypes.c_int32), ("max_clusters", ctypes.c_int32),
                ("raster_group", ctypes.c_int32), ("debug_flags", ctypes.c_int32), ("timeout_ns", ctypes.c_int64),
                ("overlap_launch", ctypes.c_int32), ("consumers", ctypes.c_int32), ("block_n", ctypes.c_int32),
                ("block_m", ctypes.c_int32), ("cluster_k", ctypes.c_int32)]


_lock = threading.Lock()
_lib: ctypes.CDLL | None = None


def _declare(lib: ctypes.CDLL) -> ctypes.CDLL:
    """Argument and result types of every C entry point."""
    vp, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32
    i64p, i32p = ctypes.POINTER(ctypes.c_int64), ctypes.POINTER(ctypes.c_int32)
    lib.gemm_f16_nt.argtypes = [vp, vp, vp, i64, i64, i64, vp]
    lib.gemm_f16_nt.restype = ctypes.c_int
    lib.gemm_f16_nt_ex.argtypes = [vp, vp, vp, i64, i64, i64, vp, ctypes.POINTER(Options)]
    lib.gemm_f16_nt_ex.restype = ctypes.c_int
    lib.gemm_f16_nt_supported.argtypes = [i64, i64, i64]
    lib.gemm_f16_nt_supported.restype = ctypes.c_int
    lib.gemm_f16_last_device_status.argtypes = [vp, ctypes.POINTER(ctypes.c_uint64)]
    lib.gemm_f16_last_device_status.restype = ctypes.c_int
    lib.gemm_f16_status_string.argtypes = [ctypes.c_int]
    lib.gemm_f16_status_string.restype = ctypes.c_char_p
    lib.gemm_f16_nt_schedule.argtypes = [i64, i64, i64, i32, i32, i32, i32, i32, i32, i64, i64, i64,
                                         ctypes.POINTER(WorkItem)]
    lib.gemm_f16_nt_schedule.restype = ctypes.c_int
    lib.gemm_f16_nt_cta_origin.argtypes = [i32, i32, i32, i32, i64, i64, i64, i64, i32, i64p, i64p, i64p, i64p]
    lib.gemm_f16_nt_cta_origin.restype = ctypes.c_int
    lib.gemm_f16_nt_host.argtypes = [vp, vp, vp, i64, i64, i64, vp, vp, vp, vp, ctypes.POINTER(Options)]
    lib.gemm_f16_nt_host.restype = ctypes.c_int
    lib.gemm_f16_nt_ws.argtypes = [vp, vp, vp, i64, i64, i64, vp, i64, vp, ctypes.POINTER(Options)]
    lib.gemm_f16_nt_ws.restype = ctypes.c_int
    lib.gemm_f16_nt_workspace_size.argtypes = [i64, i64, i64, ctypes.POINTER(Options)]
    lib.gemm_f16_nt_workspace_size.restype = ctypes.c_int64
    lib.gemm_f16_nt_static_ws.argtypes = [vp, vp, vp, i64, i64, i64, vp, ctypes.POINTER(Options)]
    lib.gemm_f16_nt_static_ws.restype = ctypes.c_int
    lib.gemm_f16_nt_describe.argtypes = [i64, i64, i64, ctypes.POINTER(Options), i32, ctypes.POINTER(LaunchInfo)]
    lib.gemm_f16_nt_describe.restype = ctypes.c_int
    lib.gemm_f16_pipeline_trace.argtypes = [i32, i32, i32, i32p, i32p]
    lib.gemm_f16_pipeline_trace.restype = ctypes.c_int
    lib.gemm_f16_co_resident.argtypes = [i32p, i32]
    lib.gemm_f16_co_resident.restype = ctypes.c_int
    lib.gemm_f16_nt_describe_for.argtypes = [i64, i64, i64, ctypes.POINTER(Options), i32, i32p, i32,
                                             ctypes.POINTER(LaunchInfo)]
    lib.gemm_f16_nt_describe_for.restype = ctypes.c_int
    return lib


def load() -> ctypes.CDLL:
    """Build (if stale) and load the CUDA library; raise if that is impossible."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        _lib = _declare(ctypes.CDLL(_build.build()))
        return _lib


_checked: ctypes.CDLL | None = None


def load_checked() -> ctypes.CDLL:
    """The checked build of the same library (device range checks compiled in; for tests).
    It is a separate shared object with its own device code and status word."""
    global _checked
    with _lock:
        if _checked is None:
            _checked = _declare(ctypes.CDLL(_build.build(checked=True)))
        return _checked


def status_string(code: int) -> str:
    return load().gemm_f16_status_string(int(code)).decode()


def gemm_f16_nt_supported(M: int, N: int, K: int) -> bool:
    return bool(load().gemm_f16_nt_supported(M, N, K))


def _stream_handle(stream) -> int | None:
    if stream is None:
        import torch

        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def gemm_f16_nt_ptr(A_ptr: int, B_ptr: int, D_ptr: int, M: int, N: int, K: int, stream: int | None = 0,
                    options: Options | None = None, workspace_ptr: int | None = None, workspace_bytes: int = 0) -> int:
    """Raw C-ABI call with device pointers; returns the status code (no raise).

    With a workspace the call goes through ``gemm_f16_nt_ws`` (split-K allowed)."""
    lib = load()
    if workspace_ptr is not None:
        return lib.gemm_f16_nt_ws(A_ptr, B_ptr, D_ptr, M, N, K, workspace_ptr, workspace_bytes, stream,
                                  ctypes.byref(options) if options is not None else None)
    if options is None:
        return lib.gemm_f16_nt(A_ptr, B_ptr, D_ptr, M, N, K, stream)
    return lib.gemm_f16_nt_ex(A_ptr, B_ptr, D_ptr, M, N, K, stream, ctypes.byref(options))


def workspace_size(M: int, N: int, K: int, options: Options | None = None) -> int:
    """Bytes of split-K workspace gemm_f16_nt_ws would use on the current device (0: no split)."""
    rc = load().gemm_f16_nt_workspace_size(M, N, K, ctypes.byref(options) if options is not None else None)
    if rc < 0:
        raise GemmError(int(rc), "gemm_f16_nt_workspace_size")
    return int(rc)


_workspaces: dict = {}


def _workspace_for(nbytes: int, device, stream):
    """A cached device buffer of at least `nbytes` for this device and stream (torch's allocator)."""
    import torch

    key = (device.index if device.index is not None else torch.cuda.current_device(), stream)
    buf = _workspaces.get(key)
    if buf is None or buf.numel() < nbytes:
        # Allocate on the stream that uses the buffer: torch's caching allocator then hands
        # this memory (or the smaller buffer it replaces) to later allocations only in that
        # stream's order, after the GEMMs already queued there.
        s = torch.cuda.ExternalStream(stream, device=device) if stream else torch.cuda.default_stream(device)
        with torch.cuda.stream(s):
            buf = torch.empty(max(nbytes, 1 << 20), dtype=torch.uint8, device=device)
        _workspaces[key] = buf
    return buf


def gemm_f16_nt(A, B, D=None, *, stream=None, options: Options | None = None, workspace=True):
    """D = A·Bᵀ for fp16 CUDA tensors A (M×K) and B (N×K); returns D (M×N).

    With ``workspace=True`` (default) a cached device buffer per device and
    stream is passed, so that few-tile problems may split their K-loop
    (``gemm_f16_nt_ws``); ``False`` calls ``gemm_f16_nt_ex`` without one; a
    uint8 CUDA tensor uses that buffer.
    """
    import torch

    if A.dtype != torch.float16 or B.dtype != torch.float16:
        raise TypeError("A and B must be torch.float16")
    if A.dim() != 2 or B.dim() != 2 or A.shape[1] != B.shape[1]:
        raise ValueError(f"expected A (M×K) and B (N×K), got {tuple(A.shape)} and {tuple(B.shape)}")
    if not (A.is_cuda and B.is_cuda) or not (A.is_contiguous() and B.is_contiguous()):
        raise ValueError("A and B must be contiguous CUDA tensors")
    M, K = A.shape
    N = B.shape[0]
    if D is None:
        D = torch.empty((M, N), dtype=torch.float16, device=A.device)
    elif D.dtype != torch.float16 or tuple(D.shape) != (M, N) or not D.is_contiguous() or not D.is_cuda:
        raise ValueError("D must be a contiguous fp16 CUDA tensor of shape (M, N)")
    with torch.cuda.device(A.device):
        sh = _stream_handle(stream)
        ws_ptr, ws_bytes = None, 0
        if workspace is True:
            need = workspace_size(M, N, K, options)
            if need > 0:
                buf = _workspace_for(need, A.device, sh)
                ws_ptr, ws_bytes = buf.data_ptr(), buf.numel()
        elif workspace is not False and workspace is not None:
            ws_ptr, ws_bytes = workspace.data_ptr(), workspace.numel() * workspace.element_size()
        rc = gemm_f16_nt_ptr(A.data_ptr(), B.data_ptr(), D.data_ptr(), M, N, K, sh, options, ws_ptr, ws_bytes)
    if rc != 0:
        raise GemmError(rc, "gemm_f16_nt")
    return D


def gemm_f16_nt_host(A_host, B_host, D_host=None, *, device=None, stream=None, A_dev=None, B_dev=None,
                     D_dev=None, options: Options | None = None):
    """End-to-end call on HOST fp16 tensors through the C entry point ``gemm_f16_nt_host``: the
    copy of A and B into device buffers, the GEMM and the copy of D back, all enqueued on one
    stream.  Pass pinned host tensors for asynchronous copies and (optionally) reusable device
    buffers. Returns the host D after the stream has finished.
    """
    import torch

    dev = torch.device(device or "cuda")
    s = stream or torch.cuda.current_stream(dev)
    M, K = A_host.shape
    N = B_host.shape[0]
    with torch.cuda.stream(s):
        A_dev = A_dev if A_dev is not None else torch.empty((M, K), dtype=torch.float16, device=dev)
        B_dev = B_dev if B_dev is not None else torch.empty((N, K), dtype=torch.float16, device=dev)
        D_dev = D_dev if D_dev is not None else torch.empty((M, N), dtype=torch.float16, device=dev)
    if D_host is None:
        D_host = torch.empty((M, N), dtype=torch.float16, pin_memory=True)
    _host_call(A_host, B_host, D_host, A_dev, B_dev, D_dev, s, options)
    s.synchronize()
    return D_host


def _host_call(A_host, B_host, D_host, A_dev, B_dev, D_dev, stream, options=None) -> None:
    """One ``gemm_f16_nt_host`` call (checks dtypes, shapes and contiguity; raises on a status)."""
    import torch

    M, K = A_host.shape
    N = B_host.shape[0]
    for t, shape, host in ((A_host, (M, K), True), (B_host, (N, K), True), (D_host, (M, N), True),
                           (A_dev, (M, K), False), (B_dev, (N, K), False), (D_dev, (M, N), False)):
        if t.dtype != torch.float16 or tuple(t.shape) != shape or not t.is_contiguous() or t.is_cuda == host:
            raise ValueError("host and device operands must be contiguous fp16 tensors of matching shapes")
    rc = load().gemm_f16_nt_host(A_host.data_ptr(), B_host.data_ptr(), D_host.data_ptr(), M, N, K,
                                 A_dev.data_ptr(), B_dev.data_ptr(), D_dev.data_ptr(), stream.cuda_stream,
                                 ctypes.byref(options) if options is not None else None)
    if rc != 0:
        raise GemmError(rc, "gemm_f16_nt_host")


class HostPipeline:
    """GEMMs on HOST fp16 tensors with the copies overlapped: D_i = A_i·B_iᵀ.

    Each step is one ``gemm_f16_nt_host`` call (copy-in, GEMM, copy-out enqueued on one
    stream).  Device buffers and streams come in `depth` slots; step i uses slot i % depth,
    so step i+1's copy-in and step i-1's copy-out run while step i's GEMM does.  A slot's
    stream orders its own steps, so a slot's buffers are reused only after its previous
    copy-out.  Pass pinned host tensors, and read a D_host only after synchronize().
    """

    def __init__(self, M: int, N: int, K: int, *, device=None, depth: int = 3):
        import torch

        self.dev = torch.device(device or "cuda")
        self.M, self.N, self.K = M, N, K
        self.depth = depth
        self.streams = [torch.cuda.Stream(self.dev) for _ in range(depth)]
        mk = lambda *shape: torch.empty(shape, dtype=torch.float16, device=self.dev)  # noqa: E731
        self.A = [mk(M, K) for _ in range(depth)]
        self.B = [mk(N, K) for _ in range(depth)]
        self.D = [mk(M, N) for _ in range(depth)]
        self.i = 0

    def submit(self, A_host, B_host, D_host) -> None:
        """Queue one step: copy A_host, B_host in, compute, copy D out into D_host."""
        j = self.i % self.depth
        self.i += 1
        _host_call(A_host, B_host, D_host, self.A[j], self.B[j], self.D[j], self.streams[j])

    def record_start(self):
        """An event, on every slot's stream, before the next submit (for timing): the first slot's."""
        import torch

        e = torch.cuda.Event(enable_timing=True)
        e.record(self.streams[self.i % self.depth])
        for k in range(1, self.depth):
            self.streams[(self.i + k) % self.depth].wait_event(e)
        return e

    def record_end(self):
        """An event after everything submitted so far (for timing): all slots joined on one stream."""
        import torch

        last = self.streams[(self.i - 1) % self.depth]
        for s in self.streams:
            if s is not last:
                ev = torch.cuda.Event()
                ev.record(s)
                last.wait_event(ev)
        e = torch.cuda.Event(enable_timing=True)
        e.record(last)
        return e

    def synchronize(self) -> None:
        for s in self.streams:
            s.synchronize()


def last_device_status(stream=None) -> tuple[int, int]:
    """(status, info) of the device status word, after synchronising `stream`; clears it."""
    info = ctypes.c_uint64(0)
    rc = load().gemm_f16_last_device_status(_stream_handle(stream), ctypes.byref(info))
    return rc, info.value


def schedule(M: int, N: int, cta_group: int, raster_group: int, num_clusters: int, cluster_id: int,
             it: int, K: int = 4096, consumers: int = 1, split_k: int = 0, block_n: int = 256,
             block_m: int = 128):
    """The iter-th work item of one cluster as (m_idx, n_idx, n_off, n_len, slice, kt_begin, kt_end),
    or None when it has no more."""
    w = WorkItem()
    rc = load().gemm_f16_nt_schedule(M, N, K, cta_group, consumers, block_n, block_m, raster_group, split_k,
                                     num_clusters, cluster_id, it, ctypes.byref(w))
    if rc < 0:
        raise GemmError(rc, "gemm_f16_nt_schedule")
    return tuple(getattr(w, f) for f, _ in WorkItem._fields_) if rc == 1 else None


def cta_origin(cta_group: int, m_idx: int, n_idx: int, rank: int, n_off: int = 0, n_len: int = 256,
               consumers: int = 1, block_n: int = 256, block_m: int = 128) -> dict:
    """Rows/columns CTA `rank` of a work item loads and writes (see the C header)."""
    out = [ctypes.c_int64() for _ in range(4)]
    rc = load().gemm_f16_nt_cta_origin(cta_group, consumers, block_n, block_m, m_idx, n_idx, n_off, n_len, rank,
                                       *[ctypes.byref(o) for o in out])
    if rc != 0:
        raise GemmError(rc, "gemm_f16_nt_cta_origin")
    return dict(zip(("a_row", "b_row", "d_row", "d_col"), (o.value for o in out)))


def describe(M: int, N: int, K: int, options: Options | None = None, with_workspace: bool = False) -> dict:
    """The kernel configuration a call would launch for this shape on the current device (see the C header)."""
    info = LaunchInfo()
    rc = load().gemm_f16_nt_describe(M, N, K, ctypes.byref(options) if options is not None else None,
                                     1 if with_workspace else 0, ctypes.byref(info))
    if rc != 0:
        raise GemmError(rc, "gemm_f16_nt_describe")
    return {f: getattr(info, f) for f, _ in LaunchInfo._fields_}


CONFIG_KINDS = 11  # GEMM_F16_CONFIG_KINDS


def co_resident() -> list[int]:
    """Co-resident clusters of each kernel configuration on the current device (see the C header)."""
    buf = (ctypes.c_int32 * CONFIG_KINDS)()
    rc = load().gemm_f16_co_resident(buf, CONFIG_KINDS)
    if rc != 0:
        raise GemmError(rc, "gemm_f16_co_resident")
    return list(buf)


def describe_for(M: int, N: int, K: int, co_resident_counts, options: Options | None = None,
                 with_workspace: bool = False) -> dict:
    """The configuration a call would launch on a device with these co-resident counts (pure host)."""
    counts = (ctypes.c_int32 * len(co_resident_counts))(*co_resident_counts)
    info = LaunchInfo()
    rc = load().gemm_f16_nt_describe_for(M, N, K, ctypes.byref(options) if options is not None else None,
                                         1 if with_workspace else 0, counts, len(co_resident_counts),
                                         ctypes.byref(info))
    if rc != 0:
        raise GemmError(rc, "gemm_f16_nt_describe_for")
    return {f: getattr(info, f) for f, _ in LaunchInfo._fields_}


def pipeline_trace(depth: int, initial_phase: int, steps: int) -> list[tuple[int, int]]:
    """The (stage, phase) a ring's PipelineState shows before each of `steps` advances."""
    st = (ctypes.c_int32 * max(steps, 1))()
    ph = (ctypes.c_int32 * max(steps, 1))()
    rc = load().gemm_f16_pipeline_trace(depth, initial_phase, steps, st, ph)
    if rc != 0:
        raise GemmError(rc, "gemm_f16_pipeline_trace")
    return [(st[i], ph[i]) for i in range(steps)]
