"""Bounded device-side waits: a wait that runs out is reported and the context
stays usable.

Units of the scheduled kernel wait for the states their predecessors publish,
with at most 2^20 polls per wait.  The host test hook SS_TEST_SKIP_UNITS
starts each launch's ticket counter past the first units, so those units are
never run and their successors wait on flags that nothing sets.  The wait
gives up (a fraction of a second), the kernel sets the device error word,
uses a zero carry and finishes; ss_selective_scan_check then returns
SS_ERR_TIMEOUT once and clears the word.  Nothing faults, traps or hangs.  A
normal call afterwards must still match the oracle.
"""
import time

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import mamba_selective_scan_ss_gb300 as ss
import oracle
from mamba_selective_scan_ss_gb300 import _build
from mamba_selective_scan_ss_gb300.inputs import ScanWorkload, make_inputs

pytestmark = pytest.mark.gpu

ATOL, RTOL = 1e-5, 1e-4


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    _build.build_all()
    ss.load_library()


def _run(inp):
    d = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    y, last = ss.selective_scan_fwd(d["u"], d["delta"], d["A"], d["B"], d["C"], d["D"], d["z"],
                                    d["delta_bias"], d["delta_softplus"])
    return y, last


@pytest.mark.parametrize("mode", ["decoupled", "chained"])
def test_wait_that_runs_out_is_reported(test_build, monkeypatch, mode):
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    monkeypatch.setenv("SS_NCHUNKS", "2")
    if mode == "decoupled":
        # one row tile, two chunks: the second chunk's look-back waits on the first
        w = ScanWorkload("timeout-decoupled-b1-d64-n16-L256-f32", 1, 64, 16, 256, "f32",
                         has_z=True, seed=11)
    else:
        # as many row tiles as CTAs: chunk 1 of tile 0 waits for chunk 0's end state
        monkeypatch.setenv("SS_CTAS_PER_SM", "1")
        w = ScanWorkload(f"timeout-chained-b1-d{64 * sms}-n16-L128-f32", 1, 64 * sms, 16, 128,
                         "f32", has_z=True, seed=12)
    plan = ss.ss_selective_scan_plan(w.batch, w.dim, w.dstate, w.seqlen, ss.SS_F32, 1, sms)
    assert plan["vector_path"] == 1 and plan["nchunks"] == 2
    assert plan["ctas"] == (2 if mode == "decoupled" else sms)
    inp = make_inputs(w)
    assert ss.ss_selective_scan_check(None) == ss.SS_OK

    monkeypatch.setenv("SS_TEST_SKIP_UNITS", "1")
    t0 = time.monotonic()
    _run(inp)
    status = ss.ss_selective_scan_check(None)
    elapsed = time.monotonic() - t0
    assert status == ss.SS_ERR_TIMEOUT, ss.ss_status_string(status)
    assert elapsed < 30.0
    assert ss.ss_selective_scan_check(None) == ss.SS_OK  # reported once, then cleared

    monkeypatch.delenv("SS_TEST_SKIP_UNITS")
    y, last = _run(inp)
    torch.cuda.synchronize()
    assert ss.ss_selective_scan_check(None) == ss.SS_OK
    y_ref, last_ref = oracle.default().fwd(inp["u"], inp["delta"], inp["A"], inp["B"], inp["C"],
                                           inp["D"], inp["z"], inp["delta_bias"],
                                           inp["delta_softplus"], dtype=w.dtype)
    for got, ref, what in ((y, y_ref, "y"), (last, last_ref, "last_state")):
        g = got.float().cpu().numpy().astype(np.float64)
        err = np.abs(g - ref)
        assert np.all(err <= ATOL + RTOL * np.abs(ref)), f"{what}: max |err| {err.max():.3e}"
