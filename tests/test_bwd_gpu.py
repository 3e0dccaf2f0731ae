"""Backward pass against the oracle's backward, through the C ABI.

ss_selective_scan_bwd returns the gradients of every input; the oracle's
ss_oracle_bwd (pinned by finite differences of the pinned forward) gives the
same in fp64 from the same inputs.  Gradients of shared inputs are sums over
many terms (dB, dC over the channels of a batch row, dA, dD and dbias over
batch and time), so each tensor is compared against its own scale:
  |err| <= RTOL * |ref| + ATOL * max|ref|
with fp32 RTOL 1e-4, ATOL 1e-5 for fp32 outputs; du, ddelta and dz are rounded
to the I/O dtype, so bf16 I/O adds the bf16 rounding, 1e-2 * |ref|.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import mamba_selective_scan_ss_gb300 as ss
import oracle
from mamba_selective_scan_ss_gb300 import _build
from mamba_selective_scan_ss_gb300.inputs import WORKLOADS, ScanWorkload, make_inputs

pytestmark = pytest.mark.gpu

RTOL, ATOL = 1e-4, 1e-5


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    _build.build_all()
    ss.load_library()


@pytest.fixture(scope="module")
def orc():
    return oracle.default()


def W(b, d, n, L, dtype="f32", seed=0, **kw):
    return ScanWorkload(f"bwd-b{b}-d{d}-n{n}-L{L}-{dtype}", b, d, n, L, dtype, seed=seed, **kw)


def grad_inputs(w, seed, with_dlast):
    g = torch.Generator().manual_seed(seed)
    io = torch.float32 if w.dtype == "f32" else torch.bfloat16
    dy = torch.randn((w.batch, w.dim, w.seqlen), generator=g).to(io)
    dlast = torch.randn((w.batch, w.dim, w.dstate), generator=g) if with_dlast else None
    return dy, dlast


def compare(got, ref, name, dtype):
    g = got.float().cpu().numpy().astype(np.float64)
    scale = float(np.max(np.abs(ref))) if ref.size else 0.0
    io_rounded = name in ("du", "ddelta", "dz") and dtype == "bf16"
    rtol = 1e-2 if io_rounded else RTOL
    bound = rtol * np.abs(ref) + ATOL * max(scale, 1e-30)
    err = np.abs(g - ref)
    assert np.all(err <= bound), (f"{name}: max |err|/bound {np.max(err / bound):.3g} "
                                  f"(max |err| {err.max():.3e}, scale {scale:.3e})")


def run_case(orc, w, seed=5, with_dlast=False, softplus=True, with_h0=False):
    inp = make_inputs(w)
    dy, dlast = grad_inputs(w, seed, with_dlast)
    if not softplus:
        inp["delta"] = (inp["delta"].float().abs() * 0.05).to(inp["delta"].dtype)
        inp["delta_bias"] = None
    h0 = None
    if with_h0:
        h0 = torch.randn((w.batch, w.dim, w.dstate), generator=torch.Generator().manual_seed(seed + 1))
    d = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    got = ss.selective_scan_bwd(d["u"], d["delta"], d["A"], d["B"], d["C"], d["D"], d["z"],
                                d["delta_bias"], softplus, dy=dy.cuda(),
                                dlast_state=None if dlast is None else dlast.cuda(),
                                h0=None if h0 is None else h0.cuda())
    torch.cuda.synchronize()
    ref = orc.bwd(inp["u"], inp["delta"], inp["A"], inp["B"], inp["C"], inp["D"], inp["z"],
                  inp["delta_bias"], softplus, dy=dy,
                  h0=None if h0 is None else h0.double().numpy(),
                  dlast=None if dlast is None else dlast.double().numpy(), dtype=w.dtype)
    for name in ("du", "ddelta", "dA", "dB", "dC", "dD", "dz", "dbias", "dh0"):
        if ref[name] is None:
            assert got[name] is None, name
            continue
        compare(got[name], ref[name], name, w.dtype)
    return got


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("shape", [(2, 64, 16, 64), (1, 70, 16, 37), (3, 5, 16, 200),
                                   (2, 130, 16, 1024), (2, 40, 16, 1), (1, 40, 16, 7),
                                   (1, 40, 16, 8), (1, 40, 16, 9), (1, 1, 16, 100)])
def test_backward_matches_oracle(orc, dtype, shape):
    run_case(orc, W(*shape, dtype=dtype, seed=71))


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("with_h0", [False, True])
def test_backward_96_row_ctas(orc, dtype, with_h0):
    """2 x 5120 rows: 160 CTAs of 64 rows would put two on some SMs of a 152-SM
    GPU, 108 CTAs of 96 rows one on each, so the launch takes 96-row CTAs (the
    last tile of each batch row 32 rows short, the last block of steps 4 short);
    every gradient against the oracle."""
    run_case(orc, W(2, 5120, 16, 100, dtype=dtype, seed=73), with_h0=with_h0, with_dlast=with_h0)


@pytest.mark.parametrize("dstate", [1, 2, 4, 7, 8, 12, 16, 17, 24, 32, 33, 64])
def test_backward_dstate(orc, dstate):
    """Up to 16 states in one group; above, groups of 16 whose row sums
    (d(dt), du, the gate's pre-activation) are carried from group to group."""
    run_case(orc, W(2, 40, dstate, 96, seed=72))


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("shape", [(2, 64, 16, 64), (1, 70, 16, 37), (2, 40, 16, 300),
                                   (2, 33, 40, 120), (1, 20, 5, 9), (1, 8, 256, 40)])
def test_backward_from_initial_state(orc, dtype, shape):
    """ss_selective_scan_bwd_h0: h0 enters the recompute (and dA through the
    first decay), and dh0 = exp(dt_0 A) g_0 comes back."""
    run_case(orc, W(*shape, dtype=dtype, seed=79), with_dlast=True, with_h0=True)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("opts", [dict(has_z=False), dict(has_D=False), dict(has_bias=False),
                                  dict(has_z=False, has_D=False, has_bias=False)])
def test_backward_optional_inputs(orc, dtype, opts):
    run_case(orc, W(2, 33, 16, 80, dtype=dtype, seed=73, **opts))


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_backward_without_softplus_and_with_state_gradient(orc, dtype):
    run_case(orc, W(2, 48, 16, 72, dtype=dtype, seed=74), with_dlast=True, softplus=False)
    run_case(orc, W(1, 64, 16, 300, dtype=dtype, seed=75), with_dlast=True)


def test_backward_full_size_sampled_batch_row(orc):
    """The Mamba-2.8B-shaped layer (batch 8, dim 5120, 16 states, seqlen 2048,
    bf16 I/O, z gate) in the benchmark's launch: 640 CTAs of 64 rows, 256
    checkpointed blocks per row.  One batch row is checked whole against the
    oracle run on that row alone: du, ddelta and dz of its 5120 channels, and
    dB, dC, which sum over exactly those channels.  dA, dD and dbias sum over
    every batch row and step of one channel, so sampled channels are checked
    with the oracle run on those channels of all eight batch rows (which also
    gives their du, ddelta and dz in every row)."""
    w = WORKLOADS["2"]
    inp = make_inputs(w)
    dy, _ = grad_inputs(w, 91, False)
    d = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    got = ss.selective_scan_bwd(d["u"], d["delta"], d["A"], d["B"], d["C"], d["D"], d["z"],
                                d["delta_bias"], True, dy=dy.cuda())
    torch.cuda.synchronize()
    b = 5
    row = {k: (inp[k][b:b + 1].contiguous() if k in ("u", "delta", "B", "C", "z") else inp[k])
           for k in inp}
    ref = orc.bwd(row["u"], row["delta"], row["A"], row["B"], row["C"], row["D"], row["z"],
                  row["delta_bias"], True, dy=dy[b:b + 1].contiguous(), dtype=w.dtype)
    for name in ("du", "ddelta", "dz", "dB", "dC"):
        compare(got[name][b:b + 1], ref[name], name, w.dtype)
    ch = [0, 1, 2047, 2048, 4095, 5119]
    cols = {k: (inp[k][:, ch].contiguous() if k in ("u", "delta", "z") else
                inp[k][ch].contiguous() if k in ("A", "D", "delta_bias") else inp[k])
            for k in inp}
    ref = orc.bwd(cols["u"], cols["delta"], cols["A"], cols["B"], cols["C"], cols["D"],
                  cols["z"], cols["delta_bias"], True, dy=dy[:, ch].contiguous(), dtype=w.dtype)
    for name in ("dA", "dD", "dbias"):
        compare(got[name][ch], ref[name], name, w.dtype)
    for name in ("du", "ddelta", "dz"):
        compare(got[name][:, ch], ref[name], name, w.dtype)


def test_backward_is_deterministic():
    w = W(4, 200, 16, 512, dtype="bf16", seed=76)
    inp = make_inputs(w)
    dy, _ = grad_inputs(w, 77, False)
    d = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    runs = [ss.selective_scan_bwd(d["u"], d["delta"], d["A"], d["B"], d["C"], d["D"], d["z"],
                                  d["delta_bias"], True, dy=dy.cuda()) for _ in range(2)]
    torch.cuda.synchronize()
    for name in runs[0]:
        if runs[0][name] is not None:
            assert torch.equal(runs[0][name], runs[1][name]), name


def test_backward_rejects_more_than_256_states():
    w = W(1, 8, 257, 16, seed=78)
    inp = make_inputs(w)
    d = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    with pytest.raises(ss.SelectiveScanError):
        ss.selective_scan_bwd(d["u"], d["delta"], d["A"], d["B"], d["C"], d["D"], d["z"],
                              d["delta_bias"], True, dy=torch.zeros_like(d["u"]))
