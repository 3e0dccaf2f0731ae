"""The general Mamba-2 path (ss_mamba2_fwd for any head dim, up to 256 states,
fp32 or bf16 I/O) against the fp64 oracle, through the C ABI.

Every call that is not bf16 with head dim 64 and 128 states runs each head
group as one selective scan over its heads' channels (fp32 arithmetic, bf16
only where y is stored), so it is held to the forward's tolerances, element
by element: fp32 I/O |err| <= 1e-5 + 1e-4*|ref|, bf16 I/O
|err| <= 1e-2*(1 + |ref|), on y and on the final state.  The test build can
send the tensor-core shape down the same path (SS_MAMBA2_ROWS), which gives
that shape an implementation that meets the bf16 element bound too.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import mamba_selective_scan_ss_gb300 as ss
import oracle
from mamba_selective_scan_ss_gb300 import _build
from mamba_selective_scan_ss_gb300.inputs import Mamba2Workload, make_mamba2_inputs

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
    g = got.float().cpu().numpy().astype(np.float64)
    err = np.abs(g - ref)
    bound = atol + rtol * np.abs(ref)
    assert np.all(err <= bound), f"{what}: max |err|/bound {np.max(err / bound):.3g}"


def W(b, L, H, P, G, N, dtype="f32", seed=0, **kw):
    return Mamba2Workload(f"m2r-b{b}-L{L}-h{H}-p{P}-g{G}-n{N}-{dtype}", b, L, H, P, G, N, dtype,
                          seed=seed, **kw)


def run_case(orc, w, softplus=True, h0=None, in_place=False):
    inp = make_mamba2_inputs(w)
    if not softplus:
        inp["dt"] = (inp["dt"].float().abs() * 0.05 + 1e-3).to(inp["dt"].dtype)
        inp["dt_bias"] = None
    d = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    h0_d = None if h0 is None else h0.clone().cuda()
    y, s = ss.mamba2_fwd(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], d["dt_bias"], softplus,
                         initial_state=h0_d, final_state=h0_d if in_place else None)
    torch.cuda.synchronize()
    assert ss.ss_selective_scan_check(None) == ss.SS_OK
    if in_place:
        assert s.data_ptr() == h0_d.data_ptr()
    ref_y, ref_s = orc.ssd(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"], inp["D"],
                           inp["dt_bias"], softplus, dtype=w.dtype,
                           initial_state=None if h0 is None else h0.double().numpy())
    close(y, ref_y, w.dtype, "y")
    close(s, ref_s, w.dtype, "final state")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("shape", [(2, 100, 4, 32, 2, 16), (1, 257, 6, 24, 3, 64),
                                   (2, 64, 2, 64, 1, 256), (1, 33, 3, 8, 1, 200),
                                   (1, 1, 2, 16, 1, 7), (2, 130, 2, 64, 1, 128)])
def test_general_shapes(orc, dtype, shape):
    """Head dims 8-64, 7-256 states, one to three groups, ragged and aligned
    lengths; fp32 I/O, and bf16 I/O off the tensor-core shape (the last case
    is that shape in fp32)."""
    run_case(orc, W(*shape, dtype=dtype, seed=sum(shape)))


@pytest.mark.parametrize("opts", [dict(has_D=False), dict(has_bias=False)])
def test_optional_inputs(orc, opts):
    run_case(orc, W(2, 90, 4, 16, 2, 32, seed=91, **opts))


def test_without_softplus(orc):
    run_case(orc, W(2, 80, 2, 32, 1, 48, "bf16", seed=92), softplus=False)


@pytest.mark.parametrize("G", [1, 2])
def test_from_initial_state(orc, G):
    w = W(2, 120, 4, 16, G, 24, seed=93 + G)
    g = torch.Generator().manual_seed(94 + G)
    h0 = torch.randn((w.batch, w.nheads, w.headdim, w.dstate), generator=g) * 0.5
    run_case(orc, w, h0=h0)


@pytest.mark.parametrize("G", [1, 3])
def test_initial_state_in_place(orc, G):
    w = W(1, 70, 3, 16, G, 16, "bf16", seed=95 + G)
    g = torch.Generator().manual_seed(96 + G)
    h0 = torch.randn((w.batch, w.nheads, w.headdim, w.dstate), generator=g) * 0.5
    run_case(orc, w, h0=h0, in_place=True)


@pytest.mark.parametrize("L", [300, 2048])
def test_tensor_core_shape_on_the_scan_path_meets_the_bf16_bound(test_build, orc, monkeypatch, L):
    """bf16, head dim 64, 128 states sent down the general path (test build):
    every element within 1e-2 (1 + |ref|), unlike the tensor-core kernel's
    bf16 operands (see test_mamba2_gpu)."""
    monkeypatch.setenv("SS_MAMBA2_ROWS", "1")
    run_case(orc, W(1, L, 4, 64, 2, 128, "bf16", seed=97))
