"""Initial state and decode step against the oracle, through the C ABI.

ss_selective_scan_fwd_h0 runs the forward from a given state and
ss_selective_state_update runs one token with the state updated in place.
The oracle evaluates both as its sequential forward from h0 (seqlen 1 for a
decode step).  Tolerances are those of the forward: fp32 I/O
|err| <= 1e-5 + 1e-4*|ref|, bf16 I/O |err| <= 1e-2*(1 + |ref|), on y and on
the state, plus the part of the fp32 rounding that the initial state itself
carries (see h0_slack).
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import mamba_selective_scan_ss_gb300 as ss
import oracle
from mamba_selective_scan_ss_gb300 import _build
from mamba_selective_scan_ss_gb300.inputs import (DecodeWorkload, ScanWorkload,
                                                  make_decode_inputs, make_inputs)

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


def close(got, ref, dtype, what, slack=0.0):
    atol, rtol = TOL[dtype]
    g = got.float().cpu().numpy().astype(np.float64) if isinstance(got, torch.Tensor) else got
    err = np.abs(g - ref)
    bound = atol + rtol * np.abs(ref) + slack
    assert np.all(err <= bound), f"{what}: max |err|/bound {np.max(err / bound):.3g}"


# Relative error per step of an fp32 state update with the approximate ex2:
# about 2^-22 for the exponential (the kernels' decays come from the MUFU
# instruction ex2.approx.ftz.f32, accurate to about 22 bits over the argument
# range a decay takes, plus the rounding of its fp32 argument dt * A * log2(e))
# and 2^-23 for the products and sums, rounded up to one bound per step.
STEP_EPS = 2.0 ** -21


def h0_slack(inp, h0):
    """Rounding carried by the initial state, as (slack on y [b,d,L], on last_state [b,d,N]).

    The part of h_t that comes from h0 is h0_n * prod_{s<=t} a_s with
    a_s = exp(dt_s * A_n); in fp32 every factor adds up to STEP_EPS of
    relative error, so after t steps that part is off by at most
    t * STEP_EPS * |h0_n| * exp(A_n * sum_{s<=t} dt_s), and y_t by that times
    |C_{n,t}| summed over n.  A state that starts at zero carries none of it.
    """
    def f64(t):
        return t.double().numpy()
    x = f64(inp["delta"]) + (f64(inp["delta_bias"])[None, :, None]
                             if inp["delta_bias"] is not None else 0.0)
    dt = np.maximum(x, 0) + np.log1p(np.exp(-np.abs(x))) if inp["delta_softplus"] else x
    cum = np.cumsum(dt, axis=-1)                                    # [b,d,L]
    A = f64(inp["A"])                                               # [d,N]
    steps = np.arange(1, dt.shape[-1] + 1)
    carried = np.abs(h0.double().numpy())[..., None] * np.exp(A[None, :, :, None] * cum[:, :, None, :])
    slack_state = STEP_EPS * steps * carried                        # [b,d,N,L]
    y = np.einsum("bdnl,bnl->bdl", slack_state, np.abs(f64(inp["C"])))
    return y, slack_state[..., -1]


@pytest.mark.parametrize("seqlen", [4, 1])
def test_decay_factor_error(seqlen):
    """The per-step error STEP_EPS assumes for the decay a = exp(dt A): read
    a back through the C ABI (state 1 before step 0, no input, dt = 0 after
    the first step) on the vector path (seqlen 4) and the scalar path
    (seqlen 1), and bound its relative error against exp(dt A) in fp64 of
    the same fp32 dt and A.  The exponent dt A log2(e) is itself rounded in
    fp32 (relative 2^-23 of |x|, x = dt A log2 e), so the bound is
    2^-22 (1 + |x|), and within STEP_EPS where |x| <= 1 (a >= 1/2; a
    stronger decay shrinks the state it carries, and its error with it)."""
    b, d, n = 1, 256, 16
    g = torch.Generator().manual_seed(71)
    dt0 = torch.exp(torch.rand((d,), generator=g) * 8.0 - 7.0)          # e^-7 .. e^1
    A = -(torch.rand((d, n), generator=g) * 3.0 + 0.01)                  # -3.01 .. -0.01
    delta = torch.zeros((b, d, seqlen))
    delta[:, :, 0] = dt0
    u = torch.zeros((b, d, seqlen))
    B = torch.zeros((b, n, seqlen))
    C = torch.zeros((b, n, seqlen))
    h0 = torch.ones((b, d, n))
    _, last = ss.selective_scan_fwd(u.cuda(), delta.cuda(), A.cuda(), B.cuda(), C.cuda(),
                                    None, None, None, False, h0=h0.cuda())
    torch.cuda.synchronize()
    got = last.cpu().double().numpy()[0]                                 # [d, n]
    x = dt0.double().numpy()[:, None] * A.double().numpy()               # natural-log exponent
    exact = np.exp(x)
    rel = np.abs(got - exact) / exact
    x2 = np.abs(x) / np.log(2.0)
    print(f"[decay] seqlen {seqlen}: max rel error {rel.max():.3g} "
          f"({np.log2(rel.max()):.1f} in log2); |x| <= 1: {rel[x2 <= 1].max():.3g}")
    assert np.all(rel <= 2.0 ** -22 * (1.0 + x2)), f"max ratio {np.max(rel / (2.0 ** -22 * (1 + x2))):.3g}"
    assert rel[x2 <= 1].max() <= STEP_EPS


def dev(inp):
    return {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}


def random_state(w, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randn((w.batch, w.dim, w.dstate), generator=g, dtype=torch.float32)


def oracle_fwd(orc, inp, dtype, h0):
    return orc.fwd(inp["u"], inp["delta"], inp["A"], inp["B"], inp["C"], inp["D"], inp["z"],
                   inp["delta_bias"], inp["delta_softplus"], h0=h0.double().numpy(),
                   dtype=dtype)


def W(b, d, n, L, dtype="f32", seed=0, **kw):
    return ScanWorkload(f"b{b}-d{d}-n{n}-L{L}-{dtype}", b, d, n, L, dtype, seed=seed, **kw)


# (shape, forced chunk count or None): chained and decoupled vector paths,
# whole rows, the scalar path (seqlen not a multiple of the vector), state
# groups (dstate > 16) and the 4- and 8-state kernels
H0_CASES = [
    ((4, 640, 16, 512), None), ((1, 64, 16, 1024), None), ((2, 96, 16, 256), 1),
    ((1, 64, 16, 1024), 5), ((2, 40, 16, 37), None), ((1, 64, 16, 999), 3),
    ((2, 70, 33, 320), None), ((1, 30, 4, 256), 3), ((2, 50, 8, 200), 2),
]


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("shape,nchunks", H0_CASES)
def test_forward_from_initial_state(test_build, orc, monkeypatch, dtype, shape, nchunks):
    if nchunks:
        monkeypatch.setenv("SS_NCHUNKS", str(nchunks))
    w = W(*shape, dtype=dtype, seed=31)
    inp = make_inputs(w)
    h0 = random_state(w, 32)
    d = dev(inp)
    y, last = ss.selective_scan_fwd(d["u"], d["delta"], d["A"], d["B"], d["C"], d["D"], d["z"],
                                    d["delta_bias"], True, h0=h0.cuda())
    torch.cuda.synchronize()
    assert ss.ss_selective_scan_check(None) == ss.SS_OK
    y_ref, last_ref = oracle_fwd(orc, inp, dtype, h0)
    sy, ss_ = h0_slack(inp, h0)
    close(y, y_ref, dtype, "y", sy)
    close(last, last_ref, dtype, "last_state", ss_)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("shape,nchunks", [((4, 640, 16, 512), 4), ((1, 64, 16, 2048), 9),
                                           ((2, 40, 16, 301), 3), ((1, 64, 16, 256), 1),
                                           ((1, 40, 24, 512), 4)])
def test_state_updated_in_place(test_build, orc, monkeypatch, dtype, shape, nchunks):
    """last_state may be h0 itself: every chunk must still start from the old state."""
    monkeypatch.setenv("SS_NCHUNKS", str(nchunks))
    w = W(*shape, dtype=dtype, seed=33)
    inp = make_inputs(w)
    h0 = random_state(w, 34)
    d = dev(inp)
    state = h0.cuda()
    y, last = ss.selective_scan_fwd(d["u"], d["delta"], d["A"], d["B"], d["C"], d["D"], d["z"],
                                    d["delta_bias"], True, h0=state, last_state=state)
    torch.cuda.synchronize()
    assert last.data_ptr() == state.data_ptr()
    y_ref, last_ref = oracle_fwd(orc, inp, dtype, h0)
    sy, ss_ = h0_slack(inp, h0)
    close(y, y_ref, dtype, "y", sy)
    close(state, last_ref, dtype, "state", ss_)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_chained_calls_equal_one_call(orc, dtype):
    """Two calls chained through the state equal one call over both segments."""
    w = W(2, 96, 16, 1024, dtype=dtype, seed=35)
    inp = make_inputs(w)
    d = dev(inp)
    y_all, last_all = ss.selective_scan_fwd(d["u"], d["delta"], d["A"], d["B"], d["C"], d["D"],
                                            d["z"], d["delta_bias"], True)
    cut = 384

    def seg(t, lo, hi):
        return t[..., lo:hi].contiguous()

    y1, s1 = ss.selective_scan_fwd(seg(d["u"], 0, cut), seg(d["delta"], 0, cut), d["A"],
                                   seg(d["B"], 0, cut), seg(d["C"], 0, cut), d["D"],
                                   seg(d["z"], 0, cut), d["delta_bias"], True)
    y2, s2 = ss.selective_scan_fwd(seg(d["u"], cut, None), seg(d["delta"], cut, None), d["A"],
                                   seg(d["B"], cut, None), seg(d["C"], cut, None), d["D"],
                                   seg(d["z"], cut, None), d["delta_bias"], True, h0=s1)
    torch.cuda.synchronize()
    y_ref, last_ref = orc.fwd(inp["u"], inp["delta"], inp["A"], inp["B"], inp["C"], inp["D"],
                              inp["z"], inp["delta_bias"], True, dtype=dtype)
    close(torch.cat([y1, y2], dim=-1), y_ref, dtype, "y of the chained calls")
    close(s2, last_ref, dtype, "state after the chained calls")
    close(y_all, y_ref, dtype, "y of one call")
    close(last_all, last_ref, dtype, "state of one call")


def decode_inputs(b, d, n, dtype, seed, *, z=True, D=True, bias=True):
    """One token and a state from the seeded decode recipe of inputs.py."""
    w = DecodeWorkload(f"decode-b{b}-d{d}-n{n}-{dtype}", b, d, n, dtype, has_z=z, has_D=D,
                       has_bias=bias, seed=seed)
    t = make_decode_inputs(w)
    t.pop("dt_softplus")
    return t


def oracle_step(orc, t, dtype, softplus=True):
    def col(v):
        return None if v is None else v.unsqueeze(-1).contiguous()
    y, last = orc.fwd(col(t["x"]), col(t["dt"]), t["A"], col(t["B"]), col(t["C"]), t["D"],
                      col(t["z"]), t["dt_bias"], softplus, h0=t["state"].double().numpy(),
                      dtype=dtype)
    return y[..., 0], last


def run_step(t, softplus=True):
    d = {k: (None if v is None else v.cuda()) for k, v in t.items()}
    y = ss.selective_state_update(d["state"], d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"],
                                  d["z"], d["dt_bias"], softplus)
    torch.cuda.synchronize()
    return y, d["state"]


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("dstate", [1, 3, 4, 5, 8, 16, 17, 33, 64, 100, 128, 129, 256])
def test_decode_step(orc, dtype, dstate):
    t = decode_inputs(3, 70, dstate, dtype, seed=40 + dstate)
    y, state = run_step(t)
    y_ref, state_ref = oracle_step(orc, t, dtype)
    close(y, y_ref, dtype, "y")
    close(state, state_ref, dtype, "state")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("opts", [dict(z=False), dict(D=False), dict(bias=False),
                                  dict(z=False, D=False, bias=False), dict(softplus=False)])
def test_decode_step_optional_inputs(orc, dtype, opts):
    opts = dict(opts)
    softplus = opts.pop("softplus", True)
    t = decode_inputs(2, 33, 16, dtype, seed=60, **opts)
    if not softplus:
        # without softplus dt = dt_raw + bias: keep it a small positive step
        t["dt"] = (t["dt"].float().abs() * 0.05).to(t["dt"].dtype)
        t["dt_bias"] = None
    y, state = run_step(t, softplus)
    y_ref, state_ref = oracle_step(orc, t, dtype, softplus)
    close(y, y_ref, dtype, "y")
    close(state, state_ref, dtype, "state")


def test_decode_large_batch(orc):
    """Many rows, 16 states: rows cross blocks and warps in every position."""
    t = decode_inputs(64, 517, 16, "bf16", seed=61)
    y, state = run_step(t)
    y_ref, state_ref = oracle_step(orc, t, "bf16")
    close(y, y_ref, "bf16", "y")
    close(state, state_ref, "bf16", "state")


@pytest.mark.parametrize("dstate", [4, 5])
def test_decode_more_batch_rows_than_one_grid_axis(orc, dstate):
    """batch above 65535 takes several launches over the batch rows."""
    t = decode_inputs(70001, 3, dstate, "f32", seed=64)
    y, state = run_step(t)
    y_ref, state_ref = oracle_step(orc, t, "f32")
    close(y, y_ref, "f32", "y")
    close(state, state_ref, "f32", "state")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_decode_loop_equals_forward(orc, dtype):
    """T decode steps from h0 equal the forward from h0 over the same T tokens."""
    w = W(2, 48, 16, 24, dtype=dtype, seed=62)
    inp = make_inputs(w)
    h0 = random_state(w, 63)
    state = h0.cuda()
    d = dev(inp)
    ys = []
    for step in range(w.seqlen):
        def tok(v):
            return None if v is None else v[..., step].contiguous()
        ys.append(ss.selective_state_update(state, tok(d["u"]), tok(d["delta"]), d["A"],
                                            tok(d["B"]), tok(d["C"]), d["D"], tok(d["z"]),
                                            d["delta_bias"], True))
    torch.cuda.synchronize()
    y_ref, last_ref = oracle_fwd(orc, inp, dtype, h0)
    sy, ss_ = h0_slack(inp, h0)
    close(torch.stack(ys, dim=-1), y_ref, dtype, "y of the decode loop", sy)
    close(state, last_ref, dtype, "state after the decode loop", ss_)
    y_f, last_f = ss.selective_scan_fwd(d["u"], d["delta"], d["A"], d["B"], d["C"], d["D"],
                                        d["z"], d["delta_bias"], True, h0=h0.cuda())
    torch.cuda.synchronize()
    close(y_f, y_ref, dtype, "y of the forward", sy)
    close(last_f, last_ref, dtype, "state of the forward", ss_)
