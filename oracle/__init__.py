"""fp64 oracle for the Gated DeltaNet recurrence -- TEST INFRASTRUCTURE ONLY.

Only the test-suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py``
may import this package.  The CUDA library never calls it, and it shares no code with the
CUDA library.

Two independent implementations live here:

* ``gdn_oracle.c`` (loaded through :func:`run`): plain C, double precision, the literal
  three-pass recurrence of the logicaffeine ``codegen_cuda::gdn`` page (module description),
  or, with ``mode="fused"``, the single-pass identity of that page's "The fusion" section.
* :mod:`oracle.closed_form_decimal`: a 50-digit ``decimal`` brute force of the same
  recurrence written in its closed matrix form, for tiny shapes.  It pins the C oracle.

This module only marshals arrays: every input is widened exactly to float64 and handed to
the C code; nothing here computes any part of the method.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import tempfile

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(_HERE, "gdn_oracle.c")
LIBRARY = os.path.join(_HERE, "libgdn_oracle.so")

# gcc flags: no FMA contraction so x86 and Arm hosts give the same bits.
CFLAGS = ["-std=c99", "-O2", "-ffp-contract=off", "-fPIC", "-shared", "-Wall", "-Wextra"]


def compile_oracle(source: str = SOURCE, output: str = LIBRARY) -> str:
    """Compile the C oracle into a shared library (atomically replaces ``output``)."""
    out_dir = os.path.dirname(os.path.abspath(output))
    fd, tmp = tempfile.mkstemp(suffix=".so", dir=out_dir)
    os.close(fd)
    cmd = ["gcc", *CFLAGS, "-I", _HERE, "-o", tmp, source, "-lpthread", "-lm"]
    try:
        subprocess.run(cmd, check=True, capture_output=True, text=True)
    except subprocess.CalledProcessError as e:  # pragma: no cover - build failure path
        os.unlink(tmp)
        raise RuntimeError(f"oracle build failed:\n{' '.join(cmd)}\n{e.stderr}") from e
    os.replace(tmp, output)
    return output


class _Args(ctypes.Structure):
    _fields_ = [
        ("B", ctypes.c_int32), ("S", ctypes.c_int32), ("Hk", ctypes.c_int32),
        ("Hv", ctypes.c_int32), ("Dk", ctypes.c_int32), ("Dv", ctypes.c_int32),
        ("head_major", ctypes.c_int32), ("mode", ctypes.c_int32),
        ("q", ctypes.c_void_p), ("k", ctypes.c_void_p),
        ("v", ctypes.c_void_p), ("z", ctypes.c_void_p),
        ("g", ctypes.c_void_p), ("beta", ctypes.c_void_p),
        ("gn", ctypes.c_void_p), ("s0", ctypes.c_void_p),
        ("y", ctypes.c_void_p), ("state", ctypes.c_void_p),
        ("qk_eps", ctypes.c_double), ("norm_eps", ctypes.c_double),
        ("heads", ctypes.c_void_p), ("n_heads", ctypes.c_int64),
        ("threads", ctypes.c_int32), ("reserved", ctypes.c_int32),
    ]


_loaded: dict[str, ctypes.CDLL] = {}


def load(path: str | None = None) -> ctypes.CDLL:
    """Load (building first if needed) an oracle shared library."""
    path = path or LIBRARY
    if path in _loaded:
        return _loaded[path]
    if path == LIBRARY and (not os.path.exists(LIBRARY)
                            or os.path.getmtime(LIBRARY) < os.path.getmtime(SOURCE)):
        compile_oracle()
    lib = ctypes.CDLL(path)
    lib.oracle_gdn_run.argtypes = [ctypes.POINTER(_Args)]
    lib.oracle_gdn_run.restype = ctypes.c_int
    _loaded[path] = lib
    return lib


def _f64(x):
    """Exact widening of a tensor / array to a contiguous float64 numpy array."""
    if x is None:
        return None
    if hasattr(x, "detach"):  # torch tensor (bf16 has no numpy dtype: widen in torch)
        import torch
        return np.ascontiguousarray(x.detach().cpu().to(torch.float64).numpy())
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(a):
    return None if a is None else a.ctypes.data


def run(q, k, v, log_decay, beta, *, z=None, gn=None, s0=None, head_major=False,
        qk_eps=1e-6, norm_eps=1e-6, mode="literal", heads=None, threads=1,
        library: str | None = None):
    """Run the oracle.  Returns ``(y, state)`` as float64 numpy arrays.

    Shapes: ``head_major=False``: q,k ``[B,S,Hk,Dk]``, v,z ``[B,S,Hv,Dv]``,
    log_decay,beta ``[B,S,Hv]``; ``head_major=True``: ``[B,H,S,W]`` / ``[B,H,S]``.
    ``s0`` is ``[B,Hv,Dv,Dk]`` or None (zeros).  ``heads`` optionally restricts the
    computation to a list of flattened heads ``b*Hv+hv`` (other entries stay NaN).
    """
    lib = load(library)
    q64, k64, v64 = _f64(q), _f64(k), _f64(v)
    g64, b64 = _f64(log_decay), _f64(beta)
    z64, gn64, s064 = _f64(z), _f64(gn), _f64(s0)
    if q64.ndim != 4 or v64.ndim != 4:
        raise ValueError("q,k,v must be 4-D")
    if head_major:
        B, Hk, S, Dk = q64.shape
        _, Hv, _, Dv = v64.shape
    else:
        B, S, Hk, Dk = q64.shape
        _, _, Hv, Dv = v64.shape
    if k64.shape != q64.shape:
        raise ValueError("q and k shapes differ")
    y = np.full(v64.shape, np.nan)
    state = np.full((B, Hv, Dv, Dk), np.nan)
    heads_arr = None
    if heads is not None:
        heads_arr = np.ascontiguousarray(np.asarray(heads, dtype=np.int64))
    a = _Args(B=B, S=S, Hk=Hk, Hv=Hv, Dk=Dk, Dv=Dv, head_major=int(bool(head_major)),
              mode={"literal": 0, "fused": 1}[mode],
              q=_ptr(q64), k=_ptr(k64), v=_ptr(v64), z=_ptr(z64), g=_ptr(g64),
              beta=_ptr(b64), gn=_ptr(gn64), s0=_ptr(s064), y=_ptr(y), state=_ptr(state),
              qk_eps=float(qk_eps), norm_eps=float(norm_eps),
              heads=_ptr(heads_arr), n_heads=0 if heads_arr is None else len(heads_arr),
              threads=int(threads))
    rc = lib.oracle_gdn_run(ctypes.byref(a))
    if rc != 0:
        raise ValueError(f"oracle_gdn_run rejected its arguments (code {rc})")
    return y, state
