"""The forward on host arrays (ss_selective_scan_fwd_host) through the C ABI.

The call works in pieces with copies and scans overlapped: slices of the
batch, or, for a single sequence, segments of about 4096 steps scanned from
the state the previous one left.  Its results are held to the forward's tolerances against the
oracle, and to the same tolerances against the device entry point (one call
over the whole sequence); pinned and pageable host memory both work.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import mamba_selective_scan_ss_gb300 as ss
import oracle
from mamba_selective_scan_ss_gb300 import _build
from mamba_selective_scan_ss_gb300.inputs import ScanWorkload, make_inputs

pytestmark = pytest.mark.gpu

TOL = {"f32": (1e-5, 1e-4), "bf16": (1e-2, 1e-2)}


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    _build.build_all()
    ss.load_library()


@pytest.fixture(scope="module")
def orc():
    return oracle.default()


def close(got, ref, dtype, what):
    atol, rtol = TOL[dtype]
    g = got.float().numpy().astype(np.float64) if isinstance(got, torch.Tensor) else got
    r = ref.float().cpu().numpy().astype(np.float64) if isinstance(ref, torch.Tensor) else ref
    err = np.abs(g - r)
    bound = atol + rtol * np.abs(r)
    assert np.all(err <= bound), f"{what}: max |err|/bound {np.max(err / bound):.3g}"


def host(inp, pinned):
    return {k: (v.pin_memory() if (pinned and isinstance(v, torch.Tensor)) else v)
            for k, v in inp.items()}


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("shape", [(1, 64, 16, 9000), (1, 33, 16, 12300), (1, 40, 16, 300),
                                   (3, 40, 16, 300), (11, 24, 16, 130)])
def test_host_forward_matches_the_oracle(orc, dtype, shape):
    """One sequence in two segments (9000 steps: 4544 + 4456, the second
    ragged), in three (12300: 4160 x 2 + 3980) and in one (300); batches in
    three slices of one and in six slices of two (the last of one)."""
    b, d, n, L = shape
    w = ScanWorkload(f"host-b{b}-d{d}-n{n}-L{L}-{dtype}", b, d, n, L, dtype, seed=L)
    inp = make_inputs(w)
    h = host(inp, pinned=True)
    y, last = ss.selective_scan_fwd_host(h["u"], h["delta"], h["A"], h["B"], h["C"], h["D"],
                                         h["z"], h["delta_bias"], True)
    y_ref, last_ref = orc.fwd(inp["u"], inp["delta"], inp["A"], inp["B"], inp["C"], inp["D"],
                              inp["z"], inp["delta_bias"], True, dtype=dtype)
    close(y, y_ref, dtype, "y")
    close(last, last_ref, dtype, "last_state")


@pytest.mark.parametrize("pinned", [True, False])
def test_host_forward_equals_the_device_call(pinned):
    """Against one device call over the whole sequence, from a given state,
    with the state updated in place in host memory."""
    w = ScanWorkload("host-vs-dev-b3-d96-n16-L8300-f32", 3, 96, 16, 8300, "f32", seed=3)
    inp = make_inputs(w)
    g = torch.Generator().manual_seed(4)
    h0 = torch.randn((w.batch, w.dim, w.dstate), generator=g)
    d = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    y_dev, last_dev = ss.selective_scan_fwd(d["u"], d["delta"], d["A"], d["B"], d["C"], d["D"],
                                            d["z"], d["delta_bias"], True, h0=h0.cuda())
    torch.cuda.synchronize()
    h = host(inp, pinned)
    state = h0.clone().pin_memory() if pinned else h0.clone()
    y, last = ss.selective_scan_fwd_host(h["u"], h["delta"], h["A"], h["B"], h["C"], h["D"],
                                         h["z"], h["delta_bias"], True, h0=state,
                                         last_state=state)
    assert last.data_ptr() == state.data_ptr()
    close(y, y_dev, "f32", "y")
    close(last, last_dev, "f32", "last_state")


def test_host_single_sequence_from_a_state_in_place():
    """A single sequence in two segments chained through the state, from a
    given state updated in place, against one device call."""
    w = ScanWorkload("host-seq-b1-d128-n16-L8300-f32", 1, 128, 16, 8300, "f32", seed=6)
    inp = make_inputs(w)
    g = torch.Generator().manual_seed(7)
    h0 = torch.randn((w.batch, w.dim, w.dstate), generator=g)
    d = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    y_dev, last_dev = ss.selective_scan_fwd(d["u"], d["delta"], d["A"], d["B"], d["C"], d["D"],
                                            d["z"], d["delta_bias"], True, h0=h0.cuda())
    torch.cuda.synchronize()
    h = host(inp, True)
    state = h0.clone().pin_memory()
    y, last = ss.selective_scan_fwd_host(h["u"], h["delta"], h["A"], h["B"], h["C"], h["D"],
                                         h["z"], h["delta_bias"], True, h0=state,
                                         last_state=state)
    close(y, y_dev, "f32", "y")
    close(last, last_dev, "f32", "last_state")


def test_host_forward_validates_before_copying():
    w = ScanWorkload("host-bad-b1-d8-n16-L64-f32", 1, 8, 16, 64, "f32", seed=5)
    inp = make_inputs(w)
    y = torch.empty_like(inp["u"])
    st = ss.ss_selective_scan_fwd_host(inp["u"].data_ptr(), inp["delta"].data_ptr(),
                                       inp["A"].data_ptr(), inp["B"].data_ptr(),
                                       inp["C"].data_ptr(), None, None, None, 1, None,
                                       inp["u"].data_ptr(), None, 1, 8, 16, 64, ss.SS_F32, None)
    assert st == ss.SS_ERR_INVALID_ARGUMENT  # y over u
    st = ss.ss_selective_scan_fwd_host(inp["u"].data_ptr(), inp["delta"].data_ptr(),
                                       inp["A"].data_ptr(), inp["B"].data_ptr(),
                                       inp["C"].data_ptr(), None, None, None, 1, None,
                                       y.data_ptr(), None, 1, 8, 257, 64, ss.SS_F32, None)
    assert st == ss.SS_ERR_UNSUPPORTED
