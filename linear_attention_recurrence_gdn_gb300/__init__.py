"""GB300-native Gated DeltaNet (GDN) recurrence: Python binding of ``libgdn.so``.

The functions here carry the names of the C entry points declared in ``include/gdn.h`` and
only marshal arguments: tensors become device pointers and sizes, the current torch stream
becomes the ``cudaStream_t``, and every step of the computation runs in the library's CUDA
kernels.  There is no fallback: if ``libgdn.so`` is missing, or the call is rejected, the
function raises.

Computed (logicaffeine ``codegen_cuda::gdn``, module description and "The fusion"): per
value head and token, ``u = S k^``, ``S = alpha S + beta (v - alpha u) k^T``, ``o = S q^``,
``y = rmsnorm(o * silu(z)) * GN``, with ``k^``, ``q^`` l2-normalised and ``q^`` scaled by
``1/sqrt(Dk)`` (torch_to_nnef ``gated_delta``, native_gdn_reject_reason) and
``alpha = exp(log_decay)``.
"""
from __future__ import annotations

import ctypes
import os

import torch

from . import build as _build

LIBRARY = _build.LIBRARY

GDN_F32, GDN_BF16, GDN_F16 = 0, 1, 2
GDN_FLAG_SCAN_TMEM = 1          # gdn_params.flags: tensor-memory chunked scan where it applies
GDN_FLAG_HOST_IO = 2            # gdn_params.flags: decode inputs and y in pinned host memory
GDN_FLAG_SCAN_BLOCK16 = 4       # gdn_params.flags: the 16-token block scan kernel for every shape
GDN_FLAG_SCAN_CHUNKED = 8       # gdn_params.flags: the chunked scan kernel wherever it applies
_DTYPE_CODE = {torch.float32: GDN_F32, torch.bfloat16: GDN_BF16, torch.float16: GDN_F16}

GDN_OK = 0
GDN_ERR_NULL_PTR = -1
GDN_ERR_BAD_SHAPE = -2
GDN_ERR_UNSUPPORTED_DIM = -3
GDN_ERR_BAD_DTYPE = -4
GDN_ERR_MISALIGNED = -5
GDN_ERR_ALIASING = -6
GDN_ERR_BAD_ARG = -7
GDN_ERR_CUDA = -8
GDN_ERR_TIMEOUT = -9

GDN_SCAN_SPLIT_NOALLOC_MAX_BYTES = 16 << 20   # fixed scratch of gdn_scan_split_noalloc

# Symbols declared in include/gdn.h (checked by the tests against the header).
EXPORTED = ("gdn_decode_step", "gdn_scan", "gdn_scan_split", "gdn_scan_split_workspace",
            "gdn_scan_split_noalloc", "gdn_reject_reason", "gdn_status_string",
            "gdn_last_error", "gdn_device_status", "gdn_selftest_wait_timeout",
            "gdn_selftest_scan_wait_limit", "gdn_version")


class GdnParams(ctypes.Structure):
    """ctypes mirror of ``gdn_params`` in include/gdn.h."""
    _fields_ = [
        ("B", ctypes.c_int32), ("S", ctypes.c_int32), ("Hk", ctypes.c_int32),
        ("Hv", ctypes.c_int32), ("Dk", ctypes.c_int32), ("Dv", ctypes.c_int32),
        ("head_major", ctypes.c_int32), ("act_dtype", ctypes.c_int32),
        ("gate_dtype", ctypes.c_int32), ("flags", ctypes.c_int32),
        ("q", ctypes.c_void_p), ("k", ctypes.c_void_p), ("v", ctypes.c_void_p),
        ("log_decay", ctypes.c_void_p), ("beta", ctypes.c_void_p), ("z", ctypes.c_void_p),
        ("gn", ctypes.c_void_p), ("s0", ctypes.c_void_p),
        ("state", ctypes.c_void_p), ("y", ctypes.c_void_p),
        ("qk_eps", ctypes.c_float), ("norm_eps", ctypes.c_float),
    ]


class GdnError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(message)
        self.status = status


_lib = None


def library(path: str | None = None) -> ctypes.CDLL:
    """Load ``libgdn.so`` (raises if it has not been built)."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or LIBRARY
    if not os.path.exists(p):
        raise RuntimeError(f"{p} is missing: build it first (python -c 'import "
                           "__graft_entry__ as g; g.build()'); there is no fallback path")
    lib = ctypes.CDLL(p)
    P = ctypes.POINTER(GdnParams)
    lib.gdn_decode_step.argtypes = [P, ctypes.c_void_p]
    lib.gdn_decode_step.restype = ctypes.c_int
    lib.gdn_scan.argtypes = [P, ctypes.c_void_p]
    lib.gdn_scan.restype = ctypes.c_int
    lib.gdn_scan_split.argtypes = [P, ctypes.c_int, ctypes.c_void_p, ctypes.c_size_t,
                                   ctypes.c_void_p]
    lib.gdn_scan_split.restype = ctypes.c_int
    lib.gdn_scan_split_workspace.argtypes = [P, ctypes.c_int]
    lib.gdn_scan_split_workspace.restype = ctypes.c_size_t
    lib.gdn_scan_split_noalloc.argtypes = [P, ctypes.c_int, ctypes.c_void_p]
    lib.gdn_scan_split_noalloc.restype = ctypes.c_int
    lib.gdn_reject_reason.argtypes = [P, ctypes.c_int]
    lib.gdn_reject_reason.restype = ctypes.c_char_p
    lib.gdn_status_string.argtypes = [ctypes.c_int]
    lib.gdn_status_string.restype = ctypes.c_char_p
    lib.gdn_last_error.argtypes = []
    lib.gdn_last_error.restype = ctypes.c_char_p
    lib.gdn_device_status.argtypes = [ctypes.c_void_p]
    lib.gdn_device_status.restype = ctypes.c_int
    lib.gdn_selftest_wait_timeout.argtypes = [ctypes.c_void_p, ctypes.c_double]
    lib.gdn_selftest_wait_timeout.restype = ctypes.c_int
    lib.gdn_selftest_scan_wait_limit.argtypes = [ctypes.c_void_p, ctypes.c_double]
    lib.gdn_selftest_scan_wait_limit.restype = ctypes.c_int
    lib.gdn_version.argtypes = []
    lib.gdn_version.restype = ctypes.c_int
    if path is None:
        _lib = lib
    return lib


def _ptr(t) -> int | None:
    return None if t is None else t.data_ptr()


def make_params(q, k, v, log_decay, beta, state, y, *, z=None, gn=None, s0=None,
                head_major=False, qk_eps=1e-6, norm_eps=1e-6, flags=0) -> GdnParams:
    """Fill a :class:`GdnParams` from tensors (shapes read per ``head_major``).

    Tensors must be contiguous; nothing is copied or converted here.
    """
    for name, t in (("q", q), ("k", k), ("v", v), ("log_decay", log_decay), ("beta", beta),
                    ("state", state), ("y", y), ("z", z), ("gn", gn), ("s0", s0)):
        if t is not None and not t.is_contiguous():
            raise GdnError(GDN_ERR_BAD_ARG, f"{name} must be contiguous (no implicit copies)")
    if q.dim() != 4 or v.dim() != 4 or state.dim() != 4:
        raise GdnError(GDN_ERR_BAD_SHAPE, "q, k, v must be 4-D and state [B,Hv,Dv,Dk]")
    if head_major:
        B, Hk, S, Dk = q.shape
        Hv, Dv = v.shape[1], v.shape[3]
        expect_v = (B, Hv, S, Dv)
        expect_g = (B, Hv, S)
    else:
        B, S, Hk, Dk = q.shape
        Hv, Dv = v.shape[2], v.shape[3]
        expect_v = (B, S, Hv, Dv)
        expect_g = (B, S, Hv)
    checks = [("k", k, tuple(q.shape)), ("v", v, expect_v), ("y", y, expect_v),
              ("log_decay", log_decay, expect_g), ("beta", beta, expect_g),
              ("state", state, (B, Hv, Dv, Dk))]
    if z is not None:
        checks.append(("z", z, expect_v))
    if gn is not None:
        checks.append(("gn", gn, (Dv,)))
    if s0 is not None:
        checks.append(("s0", s0, (B, Hv, Dv, Dk)))
    for name, t, shape in checks:
        if tuple(t.shape) != tuple(shape):
            raise GdnError(GDN_ERR_BAD_SHAPE, f"{name} has shape {tuple(t.shape)}, expected {shape}")
    act = _DTYPE_CODE.get(q.dtype)
    gate = _DTYPE_CODE.get(log_decay.dtype)
    if act is None or gate is None:
        raise GdnError(GDN_ERR_BAD_DTYPE, "q and log_decay must be float32, bfloat16 or float16")
    for name, t in (("k", k), ("v", v), ("z", z)):
        if t is not None and t.dtype != q.dtype:
            raise GdnError(GDN_ERR_BAD_DTYPE, f"{name} must have q's dtype")
    if beta.dtype != log_decay.dtype:
        raise GdnError(GDN_ERR_BAD_DTYPE, "beta must have log_decay's dtype")
    for name, t in (("state", state), ("y", y), ("gn", gn), ("s0", s0)):
        if t is not None and t.dtype != torch.float32:
            raise GdnError(GDN_ERR_BAD_DTYPE, f"{name} must be float32")
    return GdnParams(B=B, S=S, Hk=Hk, Hv=Hv, Dk=Dk, Dv=Dv, head_major=int(bool(head_major)),
                     act_dtype=act, gate_dtype=gate, flags=int(flags),
                     q=_ptr(q), k=_ptr(k), v=_ptr(v), log_decay=_ptr(log_decay),
                     beta=_ptr(beta), z=_ptr(z), gn=_ptr(gn), s0=_ptr(s0),
                     state=_ptr(state), y=_ptr(y), qk_eps=qk_eps, norm_eps=norm_eps)


def _stream_handle(stream, device) -> int:
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _raise(lib, status: int, params: GdnParams, is_decode: int):
    if status == GDN_OK:
        return
    text = lib.gdn_status_string(status).decode()
    reason = lib.gdn_reject_reason(ctypes.byref(params), is_decode)
    detail = reason.decode() if reason else lib.gdn_last_error().decode()
    raise GdnError(status, f"{text}: {detail}")


def _require_cuda(*tensors):
    for t in tensors:
        if t is not None and not t.is_cuda:
            raise GdnError(GDN_ERR_BAD_ARG, "all tensors must be CUDA tensors (no CPU path)")


def _require_device_addressable(*tensors):
    # GDN_FLAG_HOST_IO operands: CUDA tensors, or pinned host tensors (mapped into the
    # device's address space); the kernel reads and writes them, nothing runs on the CPU
    for t in tensors:
        if t is not None and not t.is_cuda and not t.is_pinned():
            raise GdnError(GDN_ERR_BAD_ARG,
                           "host_io operands must be CUDA tensors or pinned host tensors")


def gdn_decode_step(q, k, v, log_decay, beta, state, y=None, *, z=None, gn=None,
                    head_major=False, qk_eps=1e-6, norm_eps=1e-6, stream=None, host_io=False):
    """One decode token (S == 1); ``state`` [B,Hv,Dv,Dk] f32 is updated in place.

    Returns ``y`` (allocated with v's shape in f32 if not given: on v's device, or pinned
    host memory when v is a host tensor).  ``host_io=True`` sets GDN_FLAG_HOST_IO: q, k, v,
    z, the gates and y may then be pinned host tensors, which the kernel reads and writes
    directly (state and gn stay CUDA tensors).  The result is ready when the stream is.
    """
    if host_io:
        _require_device_addressable(q, k, v, log_decay, beta, y, z)
        _require_cuda(state, gn)
    else:
        _require_cuda(q, k, v, log_decay, beta, state, y, z, gn)
    if y is None:
        y = (torch.empty(v.shape, dtype=torch.float32, device=v.device) if v.is_cuda
             else torch.empty(v.shape, dtype=torch.float32).pin_memory())
    prm = make_params(q, k, v, log_decay, beta, state, y, z=z, gn=gn, head_major=head_major,
                      qk_eps=qk_eps, norm_eps=norm_eps, flags=GDN_FLAG_HOST_IO if host_io else 0)
    lib = library()
    st = lib.gdn_decode_step(ctypes.byref(prm), _stream_handle(stream, state.device))
    _raise(lib, st, prm, 1)
    return y


def gdn_scan(q, k, v, log_decay, beta, state=None, y=None, *, s0=None, z=None, gn=None,
             head_major=False, qk_eps=1e-6, norm_eps=1e-6, stream=None, tmem=False,
             block16=False, chunked=False):
    """The recurrence over the time axis from ``s0`` (None = zeros).

    Returns ``(y, state)``; ``state`` may be ``s0`` itself (in-place resume).  ``tmem=True``
    sets GDN_FLAG_SCAN_TMEM (the 32-token look-ahead tensor-memory kernel where it applies);
    ``block16=True`` sets GDN_FLAG_SCAN_BLOCK16 (the 16-token block kernel for every shape),
    ``chunked=True`` GDN_FLAG_SCAN_CHUNKED (the chunked kernel wherever it applies).
    """
    _require_cuda(q, k, v, log_decay, beta, state, y, z, gn, s0)
    if head_major:
        B, Hk, S, Dk = q.shape
        Hv, Dv = v.shape[1], v.shape[3]
    else:
        B, S, Hk, Dk = q.shape
        Hv, Dv = v.shape[2], v.shape[3]
    if y is None:
        y = torch.empty(v.shape, dtype=torch.float32, device=v.device)
    if state is None:
        state = torch.empty((B, Hv, Dv, Dk), dtype=torch.float32, device=v.device)
    prm = make_params(q, k, v, log_decay, beta, state, y, z=z, gn=gn, s0=s0,
                      head_major=head_major, qk_eps=qk_eps, norm_eps=norm_eps,
                      flags=(GDN_FLAG_SCAN_TMEM if tmem else 0) |
                      (GDN_FLAG_SCAN_BLOCK16 if block16 else 0) |
                      (GDN_FLAG_SCAN_CHUNKED if chunked else 0))
    lib = library()
    st = lib.gdn_scan(ctypes.byref(prm), _stream_handle(stream, v.device))
    _raise(lib, st, prm, 0)
    return y, state


def gdn_scan_split(q, k, v, log_decay, beta, state=None, y=None, *, segments, s0=None, z=None,
                   gn=None, head_major=False, qk_eps=1e-6, norm_eps=1e-6, stream=None,
                   workspace=None):
    """``gdn_scan`` with the sequence cut into ``segments`` ranges run in parallel (for batches
    with few heads).  Returns ``(y, state)`` like ``gdn_scan``.  ``workspace``: a CUDA tensor of
    at least ``gdn_scan_split_workspace`` bytes (allocated here when None).
    """
    _require_cuda(q, k, v, log_decay, beta, state, y, z, gn, s0, workspace)
    if head_major:
        B, Hk, S, Dk = q.shape
        Hv, Dv = v.shape[1], v.shape[3]
    else:
        B, S, Hk, Dk = q.shape
        Hv, Dv = v.shape[2], v.shape[3]
    if y is None:
        y = torch.empty(v.shape, dtype=torch.float32, device=v.device)
    if state is None:
        state = torch.empty((B, Hv, Dv, Dk), dtype=torch.float32, device=v.device)
    prm = make_params(q, k, v, log_decay, beta, state, y, z=z, gn=gn, s0=s0,
                      head_major=head_major, qk_eps=qk_eps, norm_eps=norm_eps)
    lib = library()
    need = lib.gdn_scan_split_workspace(ctypes.byref(prm), int(segments))
    own_workspace = workspace is None
    if own_workspace:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=v.device)
    nbytes = workspace.numel() * workspace.element_size()
    st = lib.gdn_scan_split(ctypes.byref(prm), int(segments), _ptr(workspace), nbytes,
                            _stream_handle(stream, v.device))
    _raise(lib, st, prm, 0)
    if own_workspace and stream is not None:
        # the kernels use the workspace on `stream`, not on the current stream it was
        # allocated on: keep the caching allocator from reusing it before `stream` is done
        workspace.record_stream(stream if isinstance(stream, torch.cuda.Stream)
                                else torch.cuda.ExternalStream(int(stream), device=v.device))
    return y, state


def gdn_scan_split_noalloc(q, k, v, log_decay, beta, state, y, *, segments, s0=None, z=None,
                           gn=None, head_major=False, qk_eps=1e-6, norm_eps=1e-6, stream=None):
    """``gdn_scan_split`` for callers that cannot allocate device memory: the C entry point
    takes its scratch from a fixed array inside the library (at most
    ``GDN_SCAN_SPLIT_NOALLOC_MAX_BYTES``) and allocates nothing.  ``state`` and ``y`` are the
    caller's output tensors (required here).  Calls that overlap on the GPU share that array
    and race: keep them on one stream.  Returns ``(y, state)``.
    """
    _require_cuda(q, k, v, log_decay, beta, state, y, z, gn, s0)
    prm = make_params(q, k, v, log_decay, beta, state, y, z=z, gn=gn, s0=s0,
                      head_major=head_major, qk_eps=qk_eps, norm_eps=norm_eps)
    lib = library()
    st = lib.gdn_scan_split_noalloc(ctypes.byref(prm), int(segments),
                                    _stream_handle(stream, v.device))
    _raise(lib, st, prm, 0)
    return y, state


def gdn_scan_split_workspace(params: GdnParams, segments: int) -> int:
    return library().gdn_scan_split_workspace(ctypes.byref(params), int(segments))


def gdn_reject_reason(params: GdnParams, is_decode: bool) -> str | None:
    r = library().gdn_reject_reason(ctypes.byref(params), int(bool(is_decode)))
    return None if r is None else r.decode()


def gdn_status_string(status: int) -> str:
    return library().gdn_status_string(status).decode()


def gdn_last_error() -> str:
    return library().gdn_last_error().decode()


def gdn_device_status(stream=None, device=None) -> int:
    """GDN_OK, or GDN_ERR_TIMEOUT if a kernel abandoned work since the last check."""
    return library().gdn_device_status(_stream_handle(stream, device))


def gdn_selftest_wait_timeout(limit_ms: float = 1.0, stream=None, device=None) -> int:
    """Launch the test hook whose bounded mbarrier wait runs out after ``limit_ms``."""
    return library().gdn_selftest_wait_timeout(_stream_handle(stream, device), float(limit_ms))


def gdn_selftest_scan_wait_limit(limit_us: float, stream=None, device=None) -> int:
    """Set the first-attempt limit of the chunked scan kernel's waits (0 = the default)."""
    return library().gdn_selftest_scan_wait_limit(_stream_handle(stream, device), float(limit_us))


def gdn_version() -> int:
    return library().gdn_version()


class HostDecodeStep:
    """A decode step fed from pinned host memory and returning y to it, with no copies.

    The step's inputs (q, k, v, z, log_decay, beta) sit in one pinned host buffer (views in
    :attr:`host`, each input 256-byte aligned) and y in pinned :attr:`y_host`.  :meth:`run`
    is one C-ABI call with GDN_FLAG_HOST_IO, whose kernel reads each head's inputs from host
    memory and writes y there, and one wait on an event recorded behind it.  Write a step's
    inputs into :attr:`host` before calling :meth:`run`.

    ``like`` holds tensors with the step's shapes and dtypes (S == 1, per ``head_major``);
    ``z`` and ``gn`` are both given or both omitted (raw o).  ``state`` (updated in place) and
    ``gn`` are CUDA tensors; the object keeps them alive (its parameter block holds their
    device addresses).  Steps run on ``stream`` (default: the current stream of ``state``'s
    device when the stepper is made) unless :meth:`run` names another.
    """

    NAMES = ("q", "k", "v", "z", "log_decay", "beta")

    def __init__(self, like: dict, state, gn=None, *, head_major=False, qk_eps=1e-6,
                 norm_eps=1e-6, stream: torch.cuda.Stream | None = None):
        _require_cuda(state, gn)
        self.state, self.gn = state, gn
        names = [n for n in self.NAMES if like.get(n) is not None]
        offs, off = {}, 0
        for n in names:
            offs[n] = off
            off += (like[n].numel() * like[n].element_size() + 255) // 256 * 256
        self._h_buf = torch.empty(off, dtype=torch.uint8).pin_memory()

        def view(n):
            nbytes = like[n].numel() * like[n].element_size()
            return self._h_buf[offs[n]:offs[n] + nbytes].view(like[n].dtype).view(like[n].shape)

        self.host = {n: view(n) for n in names}
        self.y_host = torch.empty(like["v"].shape, dtype=torch.float32).pin_memory()
        self.h2d_bytes = sum(like[n].numel() * like[n].element_size() for n in names)
        self.d2h_bytes = self.y_host.numel() * 4
        h = self.host
        self._params = make_params(h["q"], h["k"], h["v"], h["log_decay"], h["beta"], state,
                                   self.y_host, z=h.get("z"), gn=gn, head_major=head_major,
                                   qk_eps=qk_eps, norm_eps=norm_eps, flags=GDN_FLAG_HOST_IO)
        self._lib = library()
        self._device = state.device
        # the stream the steps run on unless run() names another (default: the current
        # stream of state's device when the stepper is made); its handle and the parameter
        # block's address are kept, so a step costs one C call and one event wait
        self._stream = stream if stream is not None else torch.cuda.current_stream(self._device)
        self._handle = self._stream.cuda_stream
        self._pref = ctypes.byref(self._params)
        self._done = torch.cuda.Event()

    def run(self, sync: bool = True, stream: torch.cuda.Stream | None = None):
        """One step on ``stream`` (a torch CUDA stream; default: the stepper's stream); returns
        :attr:`y_host`, valid once the stream has completed (``sync=True`` waits here)."""
        s = stream if stream is not None else self._stream
        st = self._lib.gdn_decode_step(self._pref, s.cuda_stream if stream is not None else self._handle)
        if st != GDN_OK:
            _raise(self._lib, st, self._params, 1)
        if sync:
            # an event recorded behind the step and waited on
            self._done.record(s)
            self._done.synchronize()
        return self.y_host
