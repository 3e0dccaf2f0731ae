"""The no-allocation entry point against the regular one, through the C ABI.

ss_selective_scan_fwd_noalloc serves callers that cannot allocate device
memory during a call (a caching allocator they must not bypass, a real-time
path without allocator calls, a host that owns all device memory up front).
It runs the same kernel with its scratch in a fixed device buffer of the
library.  Each case calls it twice in a row, so the second call also shows
that state left in the shared buffer by the first one does not leak into
the result.  Problems whose carries would not fit the buffer run with fewer
chunks; those cases are also checked against the CPU oracle.  This file is
collected last on purpose.
"""
import os
import subprocess
import sys
from pathlib import Path

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import mamba_selective_scan_ss_gb300 as ss
from mamba_selective_scan_ss_gb300 import _build
import oracle
from mamba_selective_scan_ss_gb300.inputs import WORKLOADS, ScanWorkload, make_inputs

pytestmark = pytest.mark.gpu

TOL = {"f32": (1e-5, 1e-4), "bf16": (1e-2, 1e-2)}


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    _build.build_all()
    ss.load_library()


def _ptrs(d, y, st):
    def pt(t):
        return None if t is None else t.data_ptr()
    return [pt(d["u"]), pt(d["delta"]), pt(d["A"]), pt(d["B"]), pt(d["C"]), pt(d["D"]),
            pt(d["z"]), pt(d["delta_bias"]), int(d["delta_softplus"]), y.data_ptr(),
            st.data_ptr()]


def _call(fn, w, d):
    y = torch.empty_like(d["u"])
    st = torch.empty((w.batch, w.dim, w.dstate), device="cuda", dtype=torch.float32)
    dt = ss.SS_F32 if w.dtype == "f32" else ss.SS_BF16
    status = fn(*_ptrs(d, y, st), w.batch, w.dim, w.dstate, w.seqlen, dt,
                torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    return status, y, st


def _close(got, ref, dtype, what):
    atol, rtol = TOL[dtype]
    g = got.float().cpu().numpy().astype(np.float64)
    r = ref.float().cpu().numpy().astype(np.float64)
    err = np.abs(g - r)
    assert np.all(err <= atol + rtol * np.abs(r)), f"{what}: max |err| {err.max():.3e}"


CASES = [
    WORKLOADS["0"],
    ScanWorkload("bf16-b2-d640-n16-L2048", 2, 640, 16, 2048, "bf16", seed=21),
    ScanWorkload("f32-b1-d256-n16-L8192-slow", 1, 256, 16, 8192, "f32", seed=22,
                 dt_lo=1e-4, dt_hi=1e-2),
    ScanWorkload("bf16-b4-d2560-n16-L1024", 4, 2560, 16, 1024, "bf16", seed=23),
    ScanWorkload("f32-b2-d96-n40-L512", 2, 96, 40, 512, "f32", seed=24),
    ScanWorkload("bf16-b1-d64-n8-L4096-noz", 1, 64, 8, 4096, "bf16", has_z=False, seed=25),
]


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_noalloc_matches_regular_entry_point_twice(w):
    d = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in make_inputs(w).items()}
    status, y_ref, st_ref = _call(ss.ss_selective_scan_fwd, w, d)
    assert status == ss.SS_OK
    for attempt in range(2):
        status, y, st = _call(ss.ss_selective_scan_fwd_noalloc, w, d)
        assert status == ss.SS_OK, ss.ss_status_string(status)
        assert ss.ss_selective_scan_check(None) == ss.SS_OK
        _close(y, y_ref, w.dtype, f"{w.name} y (call {attempt + 1})")
        _close(st, st_ref, w.dtype, f"{w.name} last_state (call {attempt + 1})")


# fewer chunks than the regular plan: the carries of 32 decoupled chunks (21 MB)
# and of 8 chained chunks (31 MB) do not fit the 16 MiB buffer
LOWERED = [
    ScanWorkload("bf16-b1-d3584-n16-L16384-decoupled", 1, 3584, 16, 16384, "bf16", seed=28,
                 dt_lo=1e-4, dt_hi=1e-2),
    ScanWorkload("bf16-b4-d5120-n16-L2048-chained", 4, 5120, 16, 2048, "bf16", seed=29),
]


@pytest.mark.parametrize("w", LOWERED, ids=lambda w: w.name)
def test_noalloc_with_fewer_chunks_matches_oracle(w):
    inp = make_inputs(w)
    d = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    status, y_ref, st_ref = _call(ss.ss_selective_scan_fwd, w, d)
    assert status == ss.SS_OK
    for attempt in range(2):
        status, y, st = _call(ss.ss_selective_scan_fwd_noalloc, w, d)
        assert status == ss.SS_OK, ss.ss_status_string(status)
        assert ss.ss_selective_scan_check(None) == ss.SS_OK
        _close(y, y_ref, w.dtype, f"{w.name} y (call {attempt + 1})")
        _close(st, st_ref, w.dtype, f"{w.name} last_state (call {attempt + 1})")
    # sampled channels of every batch row, whole sequences, against the oracle
    ch = sorted({0, 1, 63, 64, w.dim // 2, w.dim - 1})
    sub = dict(inp)
    for k in ("u", "delta", "z"):
        sub[k] = inp[k][:, ch].contiguous()
    for k in ("A", "D", "delta_bias"):
        sub[k] = inp[k][ch].contiguous()
    yo, so = oracle.default().fwd(sub["u"], sub["delta"], sub["A"], sub["B"], sub["C"], sub["D"],
                                  sub["z"], sub["delta_bias"], True, dtype=w.dtype)
    _close(y[:, ch], torch.from_numpy(yo), w.dtype, f"{w.name} y vs oracle")
    _close(st[:, ch], torch.from_numpy(so), w.dtype, f"{w.name} last_state vs oracle")


# A child process without torch: the library's own CUDA runtime (test build)
# allocates, resets the device and allocates again.  Before the call after the
# reset, the buffer address the entry point will use is compared with a fresh
# lookup in the new context; the call runs only if they agree.
_RESET_CHILD = r"""
import ctypes, sys
import numpy as np
sys.path.insert(0, sys.argv[1])
import mamba_selective_scan_ss_gb300 as ss
lib = ss.load_library(test_build=True)
vp = ctypes.c_void_p
lib.ss_test_malloc.argtypes = [ctypes.POINTER(vp), ctypes.c_size_t]
lib.ss_test_free.argtypes = [vp]
lib.ss_test_memcpy.argtypes = [vp, vp, ctypes.c_size_t]
lib.ss_test_noalloc_addresses.argtypes = [ctypes.POINTER(vp), ctypes.POINTER(vp)]
b, d, n, L = 2, 256, 16, 1024
rng = np.random.default_rng(7)
host = {
    "u": rng.standard_normal((b, d, L), dtype=np.float32),
    "delta": rng.standard_normal((b, d, L), dtype=np.float32),
    "A": -np.tile(np.arange(1, n + 1, dtype=np.float32), (d, 1)),
    "B": rng.standard_normal((b, n, L), dtype=np.float32),
    "C": rng.standard_normal((b, n, L), dtype=np.float32),
    "D": rng.standard_normal(d, dtype=np.float32),
    "z": rng.standard_normal((b, d, L), dtype=np.float32),
    "bias": np.full(d, -4.0, dtype=np.float32),
}
def upload():
    dev = {}
    for k, v in host.items():
        p = vp()
        assert lib.ss_test_malloc(ctypes.byref(p), v.nbytes) == 0
        assert lib.ss_test_memcpy(p, v.ctypes.data, v.nbytes) == 0
        dev[k] = p
    for k, nbytes in (("y", b * d * L * 4), ("st", b * d * n * 4)):
        p = vp()
        assert lib.ss_test_malloc(ctypes.byref(p), nbytes) == 0
        dev[k] = p
    return dev
def run(fn, dev):
    st = fn(dev["u"], dev["delta"], dev["A"], dev["B"], dev["C"], dev["D"], dev["z"], dev["bias"],
            1, dev["y"], dev["st"], b, d, n, L, ss.SS_F32, None)
    assert st == ss.SS_OK, st
    y = np.empty((b, d, L), np.float32)
    assert lib.ss_test_memcpy(y.ctypes.data, dev["y"], y.nbytes) == 0
    return y
def addresses():
    used, fresh = vp(), vp()
    assert lib.ss_test_noalloc_addresses(ctypes.byref(used), ctypes.byref(fresh)) == 0
    return used.value, fresh.value
dev = upload()
y_before = run(lib.ss_selective_scan_fwd_noalloc, dev)
used, fresh = addresses()
assert used == fresh, (used, fresh)
assert lib.ss_test_device_reset() == 0
dev = upload()                      # the new context: buffers allocated again
used, fresh = addresses()
assert used == fresh, ("stale buffer address after the reset", used, fresh)
y_after = run(lib.ss_selective_scan_fwd_noalloc, dev)
y_regular = run(lib.ss_selective_scan_fwd, dev)
assert lib.ss_selective_scan_check(None) == ss.SS_OK
tol = 1e-5 + 1e-4 * np.abs(y_regular)
assert np.all(np.abs(y_after - y_regular) <= tol), "after reset"
assert np.all(np.abs(y_before - y_regular) <= tol), "before reset"
print("reset ok")
"""


def test_noalloc_after_device_reset():
    repo = Path(__file__).resolve().parent.parent
    out = subprocess.run([sys.executable, "-c", _RESET_CHILD, str(repo)], capture_output=True,
                         text=True, timeout=300, env=dict(os.environ))
    assert out.returncode == 0 and "reset ok" in out.stdout, out.stdout + out.stderr


def test_noalloc_rejects_what_does_not_fit():
    # 32 states need a float32 partial read-out of batch*dim*seqlen (32 MiB here),
    # more than the fixed buffer holds: refused before anything is launched
    w = ScanWorkload("f32-b1-d2048-n32-L4096", 1, 2048, 32, 4096, "f32", seed=26)
    d = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in make_inputs(w).items()}
    status, y, _ = _call(ss.ss_selective_scan_fwd_noalloc, w, d)
    assert status == ss.SS_ERR_SCRATCH_LIMIT
    assert ss.ss_status_string(status) == "SS_ERR_SCRATCH_LIMIT"
    # and a misaligned row start is refused too (vector path only)
    w2 = ScanWorkload("f32-b1-d8-n16-L30", 1, 8, 16, 30, "f32", seed=27)
    d2 = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in make_inputs(w2).items()}
    status, _, _ = _call(ss.ss_selective_scan_fwd_noalloc, w2, d2)
    assert status == ss.SS_ERR_UNSUPPORTED
