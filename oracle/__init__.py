"""CPU oracle for the selective-scan forward pass (TEST INFRASTRUCTURE ONLY).

Only the tests, the smoke check and the CPU-baseline leg of the benchmark may
import this package.  The product library never loads it, and it shares no
code with the CUDA path.  The arithmetic lives in ``ss_oracle.c`` (plain C,
double precision, sequential in time); this module compiles it with gcc and
marshals numpy arrays to it.

Functions and the passages they follow:
  * ``Oracle.fwd``      -- the sequential definition of the scan: the Russian
    task spec "Реализовать selective scan (Mamba)", Этап 1 steps 3-4;
    "Mamba CUDA 实现解析" eq (4)-(7); the Blelloch article's section 4.1.
  * ``Oracle.combine``  -- the associative operator of "Mamba CUDA 实现解析",
    eq (10).
  * ``Oracle.bwd``      -- the exact derivative of ``fwd`` in reverse mode (the
    backward that the Russian task spec asks to verify with gradcheck, Этап 3
    step 4 and section 5; the Blelloch article, section 5.3).
  * ``Oracle.ssd``      -- the Mamba-2 recurrence with one scalar decay per head
    (the Mamba-2 cuTile news page, "Технические детали оптимизации"), run
    sequentially per (batch, head).

Parity status: pinned.  The pins (closed forms, the unrolled sum of eq (8) by
brute force, composition under eq (10)-(12), special cases) live in
``tests/oracle_pins.py`` and run with ``pytest -m "not gpu"``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from pathlib import Path

import numpy as np

ORACLE_DIR = Path(__file__).resolve().parent
SOURCE = ORACLE_DIR / "ss_oracle.c"
LIBRARY = ORACLE_DIR / "libss_oracle.so"

DTYPES = {"f32": 0, "bf16": 1}
GCC_FLAGS = ["-O2", "-std=c11", "-fPIC", "-shared", "-pthread", "-fno-fast-math"]


def build(source: Path | str = SOURCE, output: Path | str = LIBRARY,
          force: bool = False) -> Path:
    """Compile the oracle's C source into a shared library with gcc."""
    source, output = Path(source), Path(output)
    if (not force and output.exists()
            and output.stat().st_mtime >= source.stat().st_mtime):
        return output
    tmp = output.with_suffix(".so.tmp")
    cmd = ["gcc", *GCC_FLAGS, str(source), "-o", str(tmp), "-lm"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"oracle build failed:\n{' '.join(cmd)}\n{r.stderr}")
    os.replace(tmp, output)
    return output


def _as_input(x, dtype: str):
    """Return a C-contiguous numpy view of an input in the oracle's encoding.

    f32 inputs are float32 arrays; bf16 inputs are passed as their uint16 bit
    patterns.  torch tensors (CPU) are accepted and converted without copies
    of the values' meaning.
    """
    if x is None:
        return None
    try:
        import torch
        if isinstance(x, torch.Tensor):
            x = x.detach().cpu().contiguous()
            if x.dtype == torch.bfloat16:
                return x.view(torch.int16).numpy().view(np.uint16)
            return x.numpy()
    except ImportError:  # pragma: no cover
        pass
    x = np.ascontiguousarray(x)
    if dtype == "bf16" and x.dtype != np.uint16:
        raise TypeError("bf16 inputs must be passed as uint16 bit patterns or torch bf16")
    if dtype == "f32" and x.dtype != np.float32:
        raise TypeError("f32 inputs must be float32")
    return x


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


class Oracle:
    """ctypes handle on one compiled oracle library."""

    def __init__(self, library: Path | str | None = None):
        path = Path(library) if library is not None else build()
        self.path = path
        lib = ctypes.CDLL(str(path))
        lib.ss_oracle_fwd.restype = ctypes.c_int
        lib.ss_oracle_fwd.argtypes = [ctypes.c_void_p] * 8 + [
            ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
            ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
            ctypes.c_int, ctypes.c_int]
        lib.ss_oracle_fwd_pc.restype = ctypes.c_int
        lib.ss_oracle_fwd_pc.argtypes = list(lib.ss_oracle_fwd.argtypes)
        lib.ss_oracle_bwd.restype = ctypes.c_int
        lib.ss_oracle_bwd.argtypes = [ctypes.c_void_p] * 8 + [ctypes.c_int] + \
            [ctypes.c_void_p] * 12 + [ctypes.c_int64] * 4 + [ctypes.c_int, ctypes.c_int]
        lib.ss_oracle_ssd.restype = ctypes.c_int
        lib.ss_oracle_ssd.argtypes = [ctypes.c_void_p] * 7 + [ctypes.c_int] + \
            [ctypes.c_void_p] * 2 + [ctypes.c_int64] * 6 + [ctypes.c_int, ctypes.c_int]
        lib.ss_oracle_ssd_h0.restype = ctypes.c_int
        lib.ss_oracle_ssd_h0.argtypes = [ctypes.c_void_p] * 7 + [ctypes.c_int] + \
            [ctypes.c_void_p] * 3 + [ctypes.c_int64] * 6 + [ctypes.c_int, ctypes.c_int]
        lib.ss_oracle_combine.restype = None
        lib.ss_oracle_combine.argtypes = [ctypes.c_void_p] * 6 + [ctypes.c_int64]
        self.lib = lib

    def fwd(self, u, delta, A, B, C, D=None, z=None, delta_bias=None,
            delta_softplus=True, h0=None, dtype: str = "f32",
            nthreads: int | None = None, bc_per_channel: bool = False):
        """Sequential fp64 forward; returns (y [b,d,L], last_state [b,d,N]).

        bc_per_channel: B and C are [b,d,N,L], one row per channel (the task
        spec's kernel sketch layout), instead of [b,N,L]."""
        u_, dl_, B_, C_, z_ = (_as_input(t, dtype) for t in (u, delta, B, C, z))
        A_ = _as_input(A, "f32")
        D_ = _as_input(D, "f32")
        bias_ = _as_input(delta_bias, "f32")
        batch, dim, seqlen = u_.shape
        dstate = A_.shape[1]
        bc_shape = (batch, dim, dstate, seqlen) if bc_per_channel else (batch, dstate, seqlen)
        for name, arr, shape in (("delta", dl_, (batch, dim, seqlen)),
                                 ("A", A_, (dim, dstate)),
                                 ("B", B_, bc_shape),
                                 ("C", C_, bc_shape)):
            if tuple(arr.shape) != shape:
                raise ValueError(f"{name} has shape {arr.shape}, expected {shape}")
        if z_ is not None and tuple(z_.shape) != (batch, dim, seqlen):
            raise ValueError("z has the wrong shape")
        h0_ = None
        if h0 is not None:
            h0_ = np.ascontiguousarray(h0, dtype=np.float64)
            if h0_.shape != (batch, dim, dstate):
                raise ValueError("h0 has the wrong shape")
        y = np.empty((batch, dim, seqlen), dtype=np.float64)
        last = np.empty((batch, dim, dstate), dtype=np.float64)
        nt = nthreads if nthreads is not None else (os.cpu_count() or 1)
        fn = self.lib.ss_oracle_fwd_pc if bc_per_channel else self.lib.ss_oracle_fwd
        rc = fn(
            _ptr(u_), _ptr(dl_), _ptr(A_), _ptr(B_), _ptr(C_), _ptr(D_), _ptr(z_),
            _ptr(bias_), int(bool(delta_softplus)), _ptr(h0_), _ptr(y), _ptr(last),
            batch, dim, dstate, seqlen, DTYPES[dtype], nt)
        if rc != 0:
            raise RuntimeError(f"ss_oracle_fwd failed with status {rc}")
        return y, last

    def bwd(self, u, delta, A, B, C, D=None, z=None, delta_bias=None, delta_softplus=True,
            h0=None, dy=None, dlast=None, dtype: str = "f32", nthreads: int | None = None):
        """Reverse-mode derivative of ``fwd`` for a loss with gradient dy on y
        (and dlast on last_state); returns a dict of fp64 gradients: du,
        ddelta, dA, dB, dC, dD, dz, dbias, dh0 (None for absent inputs)."""
        u_, dl_, B_, C_, z_, dy_ = (_as_input(t, dtype) for t in (u, delta, B, C, z, dy))
        A_ = _as_input(A, "f32")
        D_ = _as_input(D, "f32")
        bias_ = _as_input(delta_bias, "f32")
        batch, dim, seqlen = u_.shape
        dstate = A_.shape[1]
        if dy_ is None or tuple(dy_.shape) != (batch, dim, seqlen):
            raise ValueError("dy must have the shape of y")
        h0_ = None if h0 is None else np.ascontiguousarray(h0, dtype=np.float64)
        dl_last = None if dlast is None else np.ascontiguousarray(dlast, dtype=np.float64)
        for name, arr in (("h0", h0_), ("dlast", dl_last)):
            if arr is not None and arr.shape != (batch, dim, dstate):
                raise ValueError(f"{name} has the wrong shape")
        f64 = np.float64
        out = {
            "du": np.empty((batch, dim, seqlen), f64), "ddelta": np.empty((batch, dim, seqlen), f64),
            "dA": np.empty((dim, dstate), f64), "dB": np.empty((batch, dstate, seqlen), f64),
            "dC": np.empty((batch, dstate, seqlen), f64),
            "dD": np.empty(dim, f64) if D_ is not None else None,
            "dz": np.empty((batch, dim, seqlen), f64) if z_ is not None else None,
            "dbias": np.empty(dim, f64) if bias_ is not None else None,
            "dh0": np.empty((batch, dim, dstate), f64) if h0_ is not None else None,
        }
        nt = nthreads if nthreads is not None else (os.cpu_count() or 1)
        rc = self.lib.ss_oracle_bwd(
            _ptr(u_), _ptr(dl_), _ptr(A_), _ptr(B_), _ptr(C_), _ptr(D_), _ptr(z_), _ptr(bias_),
            int(bool(delta_softplus)), _ptr(h0_), _ptr(dy_), _ptr(dl_last),
            *(_ptr(out[k]) for k in ("du", "ddelta", "dA", "dB", "dC", "dD", "dz", "dbias", "dh0")),
            batch, dim, dstate, seqlen, DTYPES[dtype], nt)
        if rc != 0:
            raise RuntimeError(f"ss_oracle_bwd failed with status {rc}")
        return out

    def ssd(self, x, dt, A, B, C, D=None, dt_bias=None, dt_softplus=True,
            dtype: str = "f32", nthreads: int | None = None, initial_state=None):
        """Sequential fp64 Mamba-2 forward; returns (y [b,L,H,P], final_state [b,H,P,N]).

        x [b,L,H,P], dt [b,L,H], A [H], B and C [b,L,G,N], D and dt_bias [H];
        initial_state [b,H,P,N] is the state before step 0 (default zero)."""
        x_, dt_, B_, C_ = (_as_input(t, dtype) for t in (x, dt, B, C))
        A_, D_, bias_ = (_as_input(t, "f32") for t in (A, D, dt_bias))
        batch, seqlen, nheads, headdim = x_.shape
        ngroups, dstate = B_.shape[2], B_.shape[3]
        for name, arr, shape in (("dt", dt_, (batch, seqlen, nheads)), ("A", A_, (nheads,)),
                                 ("B", B_, (batch, seqlen, ngroups, dstate)),
                                 ("C", C_, (batch, seqlen, ngroups, dstate)),
                                 ("D", D_, (nheads,)), ("dt_bias", bias_, (nheads,))):
            if arr is not None and tuple(arr.shape) != shape:
                raise ValueError(f"{name} has shape {arr.shape}, expected {shape}")
        h0 = None
        if initial_state is not None:
            h0 = np.ascontiguousarray(initial_state, dtype=np.float64)
            if h0.shape != (batch, nheads, headdim, dstate):
                raise ValueError("initial_state has the wrong shape")
        y = np.empty((batch, seqlen, nheads, headdim), dtype=np.float64)
        final = np.empty((batch, nheads, headdim, dstate), dtype=np.float64)
        nt = nthreads if nthreads is not None else (os.cpu_count() or 1)
        rc = self.lib.ss_oracle_ssd_h0(
            _ptr(x_), _ptr(dt_), _ptr(A_), _ptr(B_), _ptr(C_), _ptr(D_), _ptr(bias_),
            int(bool(dt_softplus)), _ptr(h0), _ptr(y), _ptr(final),
            batch, seqlen, nheads, headdim, ngroups, dstate, DTYPES[dtype], nt)
        if rc != 0:
            raise RuntimeError(f"ss_oracle_ssd failed with status {rc}")
        return y, final

    def combine(self, a1, v1, a2, c2):
        """Elementwise (a1, v1) (+) (a2, c2) of eq (10); returns (a, v)."""
        arrs = [np.ascontiguousarray(x, dtype=np.float64) for x in (a1, v1, a2, c2)]
        shape = np.broadcast_shapes(*(x.shape for x in arrs))
        arrs = [np.ascontiguousarray(np.broadcast_to(x, shape)) for x in arrs]
        a_out = np.empty(shape, dtype=np.float64)
        v_out = np.empty(shape, dtype=np.float64)
        self.lib.ss_oracle_combine(*(_ptr(x) for x in arrs), _ptr(a_out), _ptr(v_out),
                                   int(np.prod(shape)))
        return a_out, v_out


_DEFAULT: Oracle | None = None


def default() -> Oracle:
    """The oracle built from this directory's source (compiled on first use)."""
    global _DEFAULT
    if _DEFAULT is None:
        _DEFAULT = Oracle()
    return _DEFAULT
