"""The no-allocation entry point against the regular one, through the C ABI.

ss_selective_scan_fwd_noalloc serves callers that cannot allocate device
memory during a call (a caching allocator they must not bypass, a real-time
path without allocator calls, a host that owns all device memory up front).
It runs the same kernel with its scratch in a fixed device buffer of the
library.  Each case calls it twice in a row, so the second call also shows
that state left in the shared buffer by the first one does not leak into
the result.  This file is collected last on purpose.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import mamba_selective_scan_ss_gb300 as ss
from mamba_selective_scan_ss_gb300 import _build
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
