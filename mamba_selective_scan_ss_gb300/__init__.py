"""GB300-native Mamba selective-scan forward: Python binding of the C ABI.

This module only marshals arguments to ``libss_selective_scan.so`` (see
``include/ss_selective_scan.h``); every step of the computation runs in the
library's CUDA kernels.  If the library has not been built, the functions
raise: there is no fallback implementation.

Low-level names mirror the C ABI exactly (raw device pointers as ints):
    ss_selective_scan_fwd, ss_selective_scan_fwd_h0, ss_selective_state_update,
    ss_selective_scan_bwd, ss_selective_scan_bwd_h0, ss_selective_scan_fwd_pc,
    ss_selective_scan_fwd_pc_h0, ss_selective_scan_fwd_host, ss_mamba2_fwd, ss_mamba2_fwd_h0,
    ss_status_string, ss_selective_scan_check, ss_selective_scan_plan,
    ss_selective_scan_fwd_noalloc
plus convenience wrappers for torch CUDA tensors:
    selective_scan_fwd(u, delta, A, B, C, D=None, z=None, delta_bias=None,
                       delta_softplus=True, h0=None, ...)
    selective_state_update(state, x, dt, A, B, C, D=None, z=None, dt_bias=None,
                           dt_softplus=True, y=None)
    selective_scan_bwd(u, delta, A, B, C, D, z, delta_bias, delta_softplus, dy,
                       dlast_state=None, h0=None)
    mamba2_fwd(x, dt, A, B, C, D=None, dt_bias=None, dt_softplus=True, ...)
"""
from __future__ import annotations

import contextlib
import ctypes
from pathlib import Path

__all__ = [
    "SS_F32", "SS_BF16", "SS_OK", "SS_ERR_INVALID_ARGUMENT", "SS_ERR_UNSUPPORTED",
    "SS_ERR_CUDA", "SS_ERR_TIMEOUT", "SS_ERR_SCRATCH_LIMIT", "SelectiveScanError", "library_path", "load_library",
    "ss_selective_scan_fwd", "ss_status_string", "ss_selective_scan_check",
    "ss_selective_scan_plan", "ss_selective_scan_fwd_noalloc", "ss_selective_scan_fwd_h0",
    "ss_selective_state_update", "ss_selective_scan_bwd", "ss_selective_scan_bwd_h0",
    "ss_selective_scan_fwd_pc", "ss_selective_scan_fwd_pc_h0", "ss_selective_scan_fwd_host",
    "ss_mamba2_fwd", "ss_mamba2_fwd_h0", "selective_scan_fwd", "test_hooks",
    "selective_state_update", "selective_scan_bwd", "mamba2_fwd", "selective_scan_fwd_host",
]

SS_F32, SS_BF16 = 0, 1
(SS_OK, SS_ERR_INVALID_ARGUMENT, SS_ERR_UNSUPPORTED, SS_ERR_CUDA, SS_ERR_TIMEOUT,
 SS_ERR_SCRATCH_LIMIT) = range(6)

_PKG = Path(__file__).resolve().parent
_LIBS: dict = {}
_USE_TEST_BUILD = False


class SelectiveScanError(RuntimeError):
    def __init__(self, status: int, what: str = "ss_selective_scan_fwd"):
        self.status = status
        super().__init__(f"{what} failed: {ss_status_string(status)}")


def library_path(test_build: bool = False) -> Path:
    """Path of the shipped library (or of its test build, which adds the
    plan overrides and the unit-skipping hook that the tests drive through
    SS_NCHUNKS, SS_CTAS_PER_SM, SS_MAMBA2_ROWS and SS_TEST_SKIP_UNITS)."""
    return _PKG / ("libss_selective_scan_test.so" if test_build else "libss_selective_scan.so")


def _declare(lib):
    vp, i64 = ctypes.c_void_p, ctypes.c_int64
    lib.ss_selective_scan_fwd.restype = ctypes.c_int
    lib.ss_selective_scan_fwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, ctypes.c_int,
                                          vp, vp, i64, i64, i64, i64, ctypes.c_int, vp]
    lib.ss_status_string.restype = ctypes.c_char_p
    lib.ss_status_string.argtypes = [ctypes.c_int]
    lib.ss_selective_scan_check.restype = ctypes.c_int
    lib.ss_selective_scan_check.argtypes = [vp]
    lib.ss_selective_scan_fwd_noalloc.restype = ctypes.c_int
    lib.ss_selective_scan_fwd_noalloc.argtypes = list(lib.ss_selective_scan_fwd.argtypes)
    lib.ss_selective_scan_fwd_h0.restype = ctypes.c_int
    lib.ss_selective_scan_fwd_h0.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, ctypes.c_int,
                                             vp, vp, vp, i64, i64, i64, i64, ctypes.c_int, vp]
    lib.ss_selective_state_update.restype = ctypes.c_int
    lib.ss_selective_state_update.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp,
                                              ctypes.c_int, vp, i64, i64, i64,
                                              ctypes.c_int, vp]
    lib.ss_selective_scan_fwd_pc.restype = ctypes.c_int
    lib.ss_selective_scan_fwd_pc.argtypes = list(lib.ss_selective_scan_fwd.argtypes)
    lib.ss_selective_scan_fwd_pc_h0.restype = ctypes.c_int
    lib.ss_selective_scan_fwd_pc_h0.argtypes = list(lib.ss_selective_scan_fwd_h0.argtypes)
    lib.ss_selective_scan_fwd_host.restype = ctypes.c_int
    lib.ss_selective_scan_fwd_host.argtypes = list(lib.ss_selective_scan_fwd_h0.argtypes)
    lib.ss_selective_scan_bwd.restype = ctypes.c_int
    lib.ss_selective_scan_bwd.argtypes = [vp] * 8 + [ctypes.c_int] + [vp] * 10 + \
        [i64, i64, i64, i64, ctypes.c_int, vp]
    lib.ss_selective_scan_bwd_h0.restype = ctypes.c_int
    lib.ss_selective_scan_bwd_h0.argtypes = [vp] * 8 + [ctypes.c_int] + [vp] * 12 + \
        [i64, i64, i64, i64, ctypes.c_int, vp]
    lib.ss_mamba2_fwd.restype = ctypes.c_int
    lib.ss_mamba2_fwd.argtypes = [vp] * 7 + [ctypes.c_int, vp, vp] + [i64] * 6 + \
        [ctypes.c_int, vp]
    lib.ss_mamba2_fwd_h0.restype = ctypes.c_int
    lib.ss_mamba2_fwd_h0.argtypes = [vp] * 7 + [ctypes.c_int, vp, vp, vp] + [i64] * 6 + \
        [ctypes.c_int, vp]
    lib.ss_selective_scan_plan.restype = ctypes.c_int
    lib.ss_selective_scan_plan.argtypes = [i64, i64, i64, i64, ctypes.c_int, ctypes.c_int,
                                           ctypes.c_int, ctypes.POINTER(_Plan)]


def load_library(test_build: bool | None = None):
    """Load the native library (raises if it was not built).

    By default the shipped library; inside ``with test_hooks():`` (or with
    test_build=True) its test build.
    """
    tb = _USE_TEST_BUILD if test_build is None else bool(test_build)
    if tb not in _LIBS:
        path = library_path(tb)
        if not path.exists():
            raise RuntimeError(
                f"{path.name} is missing: build it with __graft_entry__.build() "
                "(the selective scan has no non-CUDA implementation)")
        lib = ctypes.CDLL(str(path))
        _declare(lib)
        _LIBS[tb] = lib
    return _LIBS[tb]


@contextlib.contextmanager
def test_hooks():
    """Route every call made inside the block to the test build of the
    library, which honours SS_NCHUNKS / SS_CTAS_PER_SM (plan overrides),
    SS_MAMBA2_ROWS (the Mamba-2 tensor-core shape on the general path) and
    SS_TEST_SKIP_UNITS (units never handed out, so that device waits run out).
    The shipped library reads no environment variable."""
    global _USE_TEST_BUILD
    prev = _USE_TEST_BUILD
    _USE_TEST_BUILD = True
    try:
        yield load_library()
    finally:
        _USE_TEST_BUILD = prev


class _Plan(ctypes.Structure):
    _fields_ = [(name, ctypes.c_int64) for name in
                ("nchunks", "chunk_len", "state_groups", "ctas", "kernel_launches",
                 "scratch_bytes", "vector_path")]


def ss_selective_scan_plan(batch, dim, dstate, seqlen, dtype, aligned16, sm_count) -> dict:
    """Launch plan of one call (host-only): chunks, launches, scratch bytes."""
    plan = _Plan()
    status = load_library().ss_selective_scan_plan(batch, dim, dstate, seqlen, int(dtype),
                                                   int(bool(aligned16)), sm_count,
                                                   ctypes.byref(plan))
    if status != SS_OK:
        raise SelectiveScanError(status, "ss_selective_scan_plan")
    return {name: getattr(plan, name) for name, _ in _Plan._fields_}


def ss_selective_scan_fwd(u, delta, A, B, C, D, z, delta_bias, delta_softplus, y, last_state,
                          batch, dim, dstate, seqlen, dtype, stream) -> int:
    """Direct call of the C entry point; pointers are ints (0/None = NULL)."""
    return load_library().ss_selective_scan_fwd(
        u, delta, A, B, C, D, z, delta_bias, int(delta_softplus), y, last_state,
        batch, dim, dstate, seqlen, int(dtype), stream)


def ss_selective_scan_fwd_noalloc(u, delta, A, B, C, D, z, delta_bias, delta_softplus, y,
                                  last_state, batch, dim, dstate, seqlen, dtype, stream) -> int:
    """The forward for callers that cannot allocate device memory during a call.

    Same arguments as ``ss_selective_scan_fwd``; the library uses its own fixed
    16 MiB device buffer instead of allocating scratch, so calls that overlap
    on the GPU must not be issued (they would share that buffer).
    """
    return load_library().ss_selective_scan_fwd_noalloc(
        u, delta, A, B, C, D, z, delta_bias, int(delta_softplus), y, last_state,
        batch, dim, dstate, seqlen, int(dtype), stream)


def ss_selective_scan_fwd_h0(u, delta, A, B, C, D, z, delta_bias, delta_softplus, h0, y,
                             last_state, batch, dim, dstate, seqlen, dtype, stream) -> int:
    """The forward started from state h0 (fp32 [batch, dim, dstate], 0/None = zero)."""
    return load_library().ss_selective_scan_fwd_h0(
        u, delta, A, B, C, D, z, delta_bias, int(delta_softplus), h0, y, last_state,
        batch, dim, dstate, seqlen, int(dtype), stream)


def ss_selective_state_update(state, x, dt, A, B, C, D, z, dt_bias, dt_softplus, y,
                              batch, dim, dstate, dtype, stream) -> int:
    """One decode step; state (fp32 [batch, dim, dstate]) is updated in place."""
    return load_library().ss_selective_state_update(
        state, x, dt, A, B, C, D, z, dt_bias, int(dt_softplus), y, batch, dim, dstate,
        int(dtype), stream)


def ss_selective_scan_fwd_pc(u, delta, A, B, C, D, z, delta_bias, delta_softplus, y, last_state,
                             batch, dim, dstate, seqlen, dtype, stream) -> int:
    """The forward with B and C per channel ([batch, dim, dstate, seqlen])."""
    return load_library().ss_selective_scan_fwd_pc(
        u, delta, A, B, C, D, z, delta_bias, int(delta_softplus), y, last_state,
        batch, dim, dstate, seqlen, int(dtype), stream)


def ss_selective_scan_fwd_pc_h0(u, delta, A, B, C, D, z, delta_bias, delta_softplus, h0, y,
                                last_state, batch, dim, dstate, seqlen, dtype, stream) -> int:
    """The per-channel forward started from state h0 (fp32 [batch, dim, dstate])."""
    return load_library().ss_selective_scan_fwd_pc_h0(
        u, delta, A, B, C, D, z, delta_bias, int(delta_softplus), h0, y, last_state,
        batch, dim, dstate, seqlen, int(dtype), stream)


def ss_selective_scan_fwd_host(u, delta, A, B, C, D, z, delta_bias, delta_softplus, h0, y,
                               last_state, batch, dim, dstate, seqlen, dtype, stream) -> int:
    """The forward on host arrays (pointers are host addresses); synchronous."""
    return load_library().ss_selective_scan_fwd_host(
        u, delta, A, B, C, D, z, delta_bias, int(delta_softplus), h0, y, last_state,
        batch, dim, dstate, seqlen, int(dtype), stream)


def ss_selective_scan_bwd(u, delta, A, B, C, D, z, delta_bias, delta_softplus, dy, dlast_state,
                          du, ddelta, dA, dB, dC, dD, dz, dbias, batch, dim, dstate, seqlen,
                          dtype, stream) -> int:
    """Direct call of the backward entry point; pointers are ints (0/None = NULL)."""
    return load_library().ss_selective_scan_bwd(
        u, delta, A, B, C, D, z, delta_bias, int(delta_softplus), dy, dlast_state, du, ddelta,
        dA, dB, dC, dD, dz, dbias, batch, dim, dstate, seqlen, int(dtype), stream)


def ss_selective_scan_bwd_h0(u, delta, A, B, C, D, z, delta_bias, delta_softplus, h0, dy,
                             dlast_state, du, ddelta, dA, dB, dC, dD, dz, dbias, dh0, batch,
                             dim, dstate, seqlen, dtype, stream) -> int:
    """The backward from initial state h0, with dh0 (its gradient)."""
    return load_library().ss_selective_scan_bwd_h0(
        u, delta, A, B, C, D, z, delta_bias, int(delta_softplus), h0, dy, dlast_state, du, ddelta,
        dA, dB, dC, dD, dz, dbias, dh0, batch, dim, dstate, seqlen, int(dtype), stream)


def ss_mamba2_fwd(x, dt, A, B, C, D, dt_bias, dt_softplus, y, final_state, batch, seqlen,
                  nheads, headdim, ngroups, dstate, dtype, stream) -> int:
    """The Mamba-2 forward (scalar decay per head) on the tensor cores."""
    return load_library().ss_mamba2_fwd(
        x, dt, A, B, C, D, dt_bias, int(dt_softplus), y, final_state, batch, seqlen, nheads,
        headdim, ngroups, dstate, int(dtype), stream)

def ss_mamba2_fwd_h0(x, dt, A, B, C, D, dt_bias, dt_softplus, initial_state, y, final_state,
                     batch, seqlen, nheads, headdim, ngroups, dstate, dtype, stream) -> int:
    """The Mamba-2 forward from a given state (fp32 [batch, nheads, headdim, dstate])."""
    return load_library().ss_mamba2_fwd_h0(
        x, dt, A, B, C, D, dt_bias, int(dt_softplus), initial_state, y, final_state, batch,
        seqlen, nheads, headdim, ngroups, dstate, int(dtype), stream)


def ss_status_string(status: int) -> str:
    return load_library().ss_status_string(int(status)).decode()


def ss_selective_scan_check(stream=None) -> int:
    return load_library().ss_selective_scan_check(stream)


def _ptr(t):
    return None if t is None else t.data_ptr()


def _io_dtype(t):
    import torch

    if t.dtype == torch.float32:
        return SS_F32
    if t.dtype == torch.bfloat16:
        return SS_BF16
    raise TypeError(f"unsupported dtype {t.dtype}")


def _check_tensors(ref, io, fp32):
    import torch

    for name, t in io:
        if t is not None and t.dtype != ref.dtype:
            raise TypeError(f"{name} must have dtype {ref.dtype}")
    for name, t in fp32:
        if t is not None and t.dtype != torch.float32:
            raise TypeError(f"{name} must be float32")
    for _, t in (*io, *fp32):
        if t is not None and (not t.is_cuda or not t.is_contiguous()):
            raise ValueError("all tensors must be contiguous CUDA tensors")


def _stream(stream, device):
    import torch

    if stream is None:
        return torch.cuda.current_stream(device).cuda_stream
    return stream if isinstance(stream, int) else stream.cuda_stream


def selective_scan_fwd(u, delta, A, B, C, D=None, z=None, delta_bias=None,
                       delta_softplus: bool = True, return_last_state: bool = True,
                       y=None, last_state=None, stream=None, h0=None):
    """Run the forward on torch CUDA tensors in the ABI layouts.

    u, delta, z: [batch, dim, seqlen]; B, C: [batch, dstate, seqlen] (or
    [batch, dim, dstate, seqlen]: one row per channel, ss_selective_scan_fwd_pc); A:
    [dim, dstate] fp32; D, delta_bias: [dim] fp32.  u, delta, B, C, z share one
    dtype (float32 or bfloat16), which is also y's dtype.  Returns y, or
    (y, last_state) with last_state [batch, dim, dstate] fp32.  Outputs are
    allocated with torch unless given.  h0 (fp32 [batch, dim, dstate]) is the
    state before step 0 (default zero); last_state may be h0 itself.  Runs on
    ``stream`` (a torch.cuda.Stream or a raw cudaStream_t int), default
    torch's current stream.
    """
    import torch

    dt = _io_dtype(u)
    _check_tensors(u, (("u", u), ("delta", delta), ("B", B), ("C", C), ("z", z)),
                   (("A", A), ("D", D), ("delta_bias", delta_bias), ("h0", h0)))
    batch, dim, seqlen = u.shape
    dstate = A.shape[1]
    if y is None:
        y = torch.empty_like(u)
    if last_state is None and return_last_state:
        last_state = torch.empty((batch, dim, dstate), device=u.device, dtype=torch.float32)
    s = _stream(stream, u.device)
    args = (_ptr(u), _ptr(delta), _ptr(A), _ptr(B), _ptr(C), _ptr(D), _ptr(z), _ptr(delta_bias),
            delta_softplus)
    outs = (_ptr(y), _ptr(last_state) if return_last_state else None,
            batch, dim, dstate, seqlen, dt, s)
    per_channel = B.dim() == 4
    if per_channel:
        if h0 is None:
            status = ss_selective_scan_fwd_pc(*args, *outs)
        else:
            status = ss_selective_scan_fwd_pc_h0(*args, _ptr(h0), *outs)
    elif h0 is None:
        status = ss_selective_scan_fwd(*args, *outs)
    else:
        status = ss_selective_scan_fwd_h0(*args, _ptr(h0), *outs)
    if status != SS_OK:
        what = ("_pc" if per_channel else "") + ("" if h0 is None else "_h0")
        raise SelectiveScanError(status, "ss_selective_scan_fwd" + what)
    return (y, last_state) if return_last_state else y


def selective_scan_fwd_host(u, delta, A, B, C, D=None, z=None, delta_bias=None,
                            delta_softplus: bool = True, h0=None, y=None, last_state=None,
                            stream=None):
    """The forward on CPU torch tensors (pinned for overlapped copies), through
    ss_selective_scan_fwd_host: same layouts and dtypes as selective_scan_fwd;
    returns (y, last_state) as CPU tensors once they are complete.  The copies
    and the scan run on ``stream`` (default torch's current stream) and two
    streams of the call's own."""
    import torch

    for name, t in (("u", u), ("delta", delta), ("A", A), ("B", B), ("C", C), ("D", D),
                    ("z", z), ("delta_bias", delta_bias), ("h0", h0)):
        if t is not None and (t.is_cuda or not t.is_contiguous()):
            raise ValueError(f"{name} must be a contiguous CPU tensor")
    dt = _io_dtype(u)
    for name, t in (("delta", delta), ("B", B), ("C", C), ("z", z)):
        if t is not None and t.dtype != u.dtype:
            raise TypeError(f"{name} must have dtype {u.dtype}")
    for name, t in (("A", A), ("D", D), ("delta_bias", delta_bias), ("h0", h0)):
        if t is not None and t.dtype != torch.float32:
            raise TypeError(f"{name} must be float32")
    batch, dim, seqlen = u.shape
    dstate = A.shape[1]
    if y is None:
        y = torch.empty(u.shape, dtype=u.dtype, pin_memory=u.is_pinned())
    if last_state is None:
        last_state = torch.empty((batch, dim, dstate), dtype=torch.float32,
                                 pin_memory=u.is_pinned())
    s = _stream(stream, torch.device("cuda", torch.cuda.current_device()))
    status = ss_selective_scan_fwd_host(
        _ptr(u), _ptr(delta), _ptr(A), _ptr(B), _ptr(C), _ptr(D), _ptr(z), _ptr(delta_bias),
        delta_softplus, _ptr(h0), _ptr(y), _ptr(last_state), batch, dim, dstate, seqlen, dt, s)
    if status != SS_OK:
        raise SelectiveScanError(status, "ss_selective_scan_fwd_host")
    return y, last_state


def selective_state_update(state, x, dt, A, B, C, D=None, z=None, dt_bias=None,
                           dt_softplus: bool = True, y=None, stream=None):
    """One decode step on torch CUDA tensors; ``state`` is updated in place.

    state: [batch, dim, dstate] fp32; x, dt, z: [batch, dim]; B, C: [batch,
    dstate]; A: [dim, dstate] fp32; D, dt_bias: [dim] fp32.  x, dt, B, C, z
    share one dtype (float32 or bfloat16), which is also y's.  Returns y.
    """
    import torch

    io = _io_dtype(x)
    _check_tensors(x, (("x", x), ("dt", dt), ("B", B), ("C", C), ("z", z)),
                   (("state", state), ("A", A), ("D", D), ("dt_bias", dt_bias)))
    batch, dim = x.shape
    dstate = A.shape[1]
    if y is None:
        y = torch.empty_like(x)
    status = ss_selective_state_update(
        _ptr(state), _ptr(x), _ptr(dt), _ptr(A), _ptr(B), _ptr(C), _ptr(D), _ptr(z),
        _ptr(dt_bias), dt_softplus, _ptr(y), batch, dim, dstate, io, _stream(stream, x.device))
    if status != SS_OK:
        raise SelectiveScanError(status, "ss_selective_state_update")
    return y


def selective_scan_bwd(u, delta, A, B, C, D=None, z=None, delta_bias=None,
                       delta_softplus: bool = True, dy=None, dlast_state=None, stream=None,
                       h0=None):
    """Gradients of the forward on torch CUDA tensors.

    Returns a dict: du, ddelta (and dz) in the I/O dtype; dA [dim, dstate],
    dB, dC [batch, dstate, seqlen], dD, dbias [dim] in float32 (None for an
    absent input); with h0 (float32 [batch, dim, dstate], the forward's
    initial state, default zero) also dh0 of the same shape.  dy has y's
    shape and dtype; dlast_state (float32 [batch, dim, dstate]) is the
    gradient of last_state, default zero.
    """
    import torch

    io = _io_dtype(u)
    _check_tensors(u, (("u", u), ("delta", delta), ("B", B), ("C", C), ("z", z), ("dy", dy)),
                   (("A", A), ("D", D), ("delta_bias", delta_bias), ("dlast_state", dlast_state)))
    batch, dim, seqlen = u.shape
    dstate = A.shape[1]
    f32 = dict(device=u.device, dtype=torch.float32)
    g = {"du": torch.empty_like(u), "ddelta": torch.empty_like(u),
         "dA": torch.empty((dim, dstate), **f32),
         "dB": torch.empty((batch, dstate, seqlen), **f32),
         "dC": torch.empty((batch, dstate, seqlen), **f32),
         "dD": torch.empty((dim,), **f32) if D is not None else None,
         "dz": torch.empty_like(u) if z is not None else None,
         "dbias": torch.empty((dim,), **f32) if delta_bias is not None else None,
         "dh0": torch.empty((batch, dim, dstate), **f32) if h0 is not None else None}
    if h0 is not None:
        _check_tensors(u, (), (("h0", h0),))
    status = ss_selective_scan_bwd_h0(
        _ptr(u), _ptr(delta), _ptr(A), _ptr(B), _ptr(C), _ptr(D), _ptr(z), _ptr(delta_bias),
        delta_softplus, _ptr(h0), _ptr(dy), _ptr(dlast_state),
        *(_ptr(g[k]) for k in ("du", "ddelta", "dA", "dB", "dC", "dD", "dz", "dbias", "dh0")),
        batch, dim, dstate, seqlen, io, _stream(stream, u.device))
    if status != SS_OK:
        raise SelectiveScanError(status, "ss_selective_scan_bwd")
    return g


def mamba2_fwd(x, dt, A, B, C, D=None, dt_bias=None, dt_softplus: bool = True,
               return_final_state: bool = True, y=None, final_state=None, stream=None,
               initial_state=None):
    """The Mamba-2 forward on torch CUDA tensors (ss_mamba2_fwd).

    x: [batch, seqlen, nheads, headdim] bf16; dt: [batch, seqlen, nheads] bf16;
    A, D, dt_bias: [nheads] fp32; B, C: [batch, seqlen, ngroups, dstate] bf16.
    Returns y (like x), or (y, final_state) with final_state [batch, nheads,
    headdim, dstate] fp32.  initial_state (fp32, like final_state) is the state
    before step 0 (default zero, ss_mamba2_fwd_h0); final_state may be it.
    """
    import torch

    io = _io_dtype(x)
    _check_tensors(x, (("x", x), ("dt", dt), ("B", B), ("C", C)),
                   (("A", A), ("D", D), ("dt_bias", dt_bias), ("initial_state", initial_state)))
    batch, seqlen, nheads, headdim = x.shape
    ngroups, dstate = B.shape[2], B.shape[3]
    if y is None:
        y = torch.empty_like(x)
    if final_state is None and return_final_state:
        final_state = torch.empty((batch, nheads, headdim, dstate), device=x.device,
                                  dtype=torch.float32)
    status = ss_mamba2_fwd_h0(_ptr(x), _ptr(dt), _ptr(A), _ptr(B), _ptr(C), _ptr(D),
                              _ptr(dt_bias), dt_softplus, _ptr(initial_state), _ptr(y),
                              _ptr(final_state) if return_final_state else None,
                              batch, seqlen, nheads, headdim, ngroups, dstate, io,
                              _stream(stream, x.device))
    if status != SS_OK:
        raise SelectiveScanError(status, "ss_mamba2_fwd_h0")
    return (y, final_state) if return_final_state else y
