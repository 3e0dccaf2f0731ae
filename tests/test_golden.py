"""Stored expected values (tests/golden/, written by tests/golden/make_golden.py
with the seeded input generators and the oracle only).

On the CPU the oracle must reproduce its stored results exactly: a change in
its arithmetic shows up here and the fixtures have to be regenerated on
purpose.  On the GPU the CUDA path is held to the forward's tolerances against
the same numbers (fp32: |err| <= 1e-5 + 1e-4 |ref|; the backward per tensor
against its own scale, as in test_bwd_gpu).
"""
import json
from pathlib import Path

import numpy as np
import pytest

import oracle

GOLDEN = Path(__file__).resolve().parent / "golden"
CASES = sorted(p.stem for p in GOLDEN.glob("*.json"))


def load(name):
    return json.loads((GOLDEN / f"{name}.json").read_text())


def f32(v):
    return None if v is None else np.asarray(v, dtype=np.float32)


def run_oracle(case):
    orc = oracle.default()
    i = case["inputs"]
    if case["kind"] == "forward":
        h0 = None if case["h0"] is None else np.asarray(case["h0"])
        y, last = orc.fwd(f32(i["u"]), f32(i["delta"]), f32(i["A"]), f32(i["B"]), f32(i["C"]),
                          f32(i["D"]), f32(i["z"]), f32(i["delta_bias"]), i["delta_softplus"],
                          h0=h0, dtype="f32")
        return {"y": y, "last_state": last}
    if case["kind"] == "backward":
        g = orc.bwd(f32(i["u"]), f32(i["delta"]), f32(i["A"]), f32(i["B"]), f32(i["C"]),
                    f32(i["D"]), f32(i["z"]), f32(i["delta_bias"]), i["delta_softplus"],
                    dy=f32(case["dy"]), dtype="f32")
        return {k: v for k, v in g.items() if v is not None}
    y, fin = orc.ssd(f32(i["x"]), f32(i["dt"]), f32(i["A"]), f32(i["B"]), f32(i["C"]),
                     f32(i["D"]), f32(i["dt_bias"]), i["dt_softplus"], dtype="f32")
    return {"y": y, "final_state": fin}


def stored(case):
    if case["kind"] == "backward":
        return {k: np.asarray(v) for k, v in case["grads"].items() if v is not None}
    keys = ("y", "last_state") if case["kind"] == "forward" else ("y", "final_state")
    return {k: np.asarray(case[k]) for k in keys}


@pytest.mark.parametrize("name", CASES)
def test_oracle_reproduces_its_stored_results(name):
    case = load(name)
    assert case["citation"]
    got, want = run_oracle(case), stored(case)
    assert set(got) == set(want)
    for k in want:
        assert np.array_equal(np.asarray(got[k]), want[k]), f"{name}: {k} changed"


@pytest.mark.gpu
@pytest.mark.parametrize("name", CASES)
def test_cuda_path_matches_the_stored_results(name):
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import mamba_selective_scan_ss_gb300 as ss
    from mamba_selective_scan_ss_gb300 import _build
    _build.build_all()
    ss.load_library()
    case = load(name)
    i = case["inputs"]
    dev = lambda v: None if v is None else torch.tensor(np.asarray(v, dtype=np.float32)).cuda()
    want = stored(case)
    if case["kind"] == "forward":
        y, last = ss.selective_scan_fwd(dev(i["u"]), dev(i["delta"]), dev(i["A"]), dev(i["B"]),
                                        dev(i["C"]), dev(i["D"]), dev(i["z"]),
                                        dev(i["delta_bias"]), i["delta_softplus"],
                                        h0=dev(case["h0"]))
        got = {"y": y, "last_state": last}
    elif case["kind"] == "backward":
        g = ss.selective_scan_bwd(dev(i["u"]), dev(i["delta"]), dev(i["A"]), dev(i["B"]),
                                  dev(i["C"]), dev(i["D"]), dev(i["z"]), dev(i["delta_bias"]),
                                  i["delta_softplus"], dy=dev(case["dy"]))
        got = {k: v for k, v in g.items() if k in want}
    else:
        y, fin = ss.mamba2_fwd(dev(i["x"]), dev(i["dt"]), dev(i["A"]), dev(i["B"]), dev(i["C"]),
                               dev(i["D"]), dev(i["dt_bias"]), i["dt_softplus"])
        got = {"y": y, "final_state": fin}
    torch.cuda.synchronize()
    for k, ref in want.items():
        g = got[k].float().cpu().numpy().astype(np.float64)
        if case["kind"] == "backward":
            bound = 1e-4 * np.abs(ref) + 1e-5 * np.abs(ref).max()
        else:
            bound = 1e-5 + 1e-4 * np.abs(ref)
        err = np.abs(g - ref)
        assert np.all(err <= bound), f"{name} {k}: max |err|/bound {np.max(err / bound):.3g}"
