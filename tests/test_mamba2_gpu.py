"""Mamba-2 forward (ss_mamba2_fwd, tensor cores) against the fp64 oracle.

Tolerance, from the kernel's arithmetic.  The inputs are bf16 and enter the
products exactly; three derived operands are rounded to bf16 (unit roundoff
u = 2^-8) where they enter a product: the decayed C.B weights of a chunk, the
decayed inputs w_s x_s of the chunk's state, and the state carried into a
chunk.  Every product term is therefore off by at most u (2u for the carried
state, which also carries the rounding of the inputs it was built from), the
state itself stays fp32, and y is rounded to bf16 once more.  With y_abs and
state_abs the oracle's results on |x|, |B|, |C|, |D| (all decays are
positive, so these bound the sums of |term|):
    |y - ref|     <= 1.1 (2u y_abs + u |ref|) + 1e-6
    |state - ref| <= 1.1 u state_abs + 1e-6
That bound is rigorous but loose where terms cancel, so the normwise error is
also held to 4u: ||y - ref|| <= 4u ||ref||, a few independent roundings of u
each (a misplaced decay step or a dropped term is off by 1e-2..1 of the norm).
The bound fixed for bf16 I/O in the Mamba-1 forward, |err| <= 1e-2 (1 + |ref|)
element by element, is NOT met everywhere by this kernel: its bf16 derived
operands (above all w.x in the chunk-state product, whose rounding the
carried state passes on to the next chunk) leave elements whose reference is
small against its terms up to about 3x that bound (measured: 1.09x on the
small workload, 2.83x on the first step of a chunk of one step).  The ratio
is computed and printed for every case so that the shortfall stays visible.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import mamba_selective_scan_ss_gb300 as ss
import oracle
from mamba_selective_scan_ss_gb300 import _build
from mamba_selective_scan_ss_gb300.inputs import (MAMBA2_WORKLOADS, Mamba2Workload,
                                                  make_mamba2_inputs)

pytestmark = pytest.mark.gpu

U = 2.0 ** -8


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    _build.build_all()
    ss.load_library()


@pytest.fixture(scope="module")
def orc():
    return oracle.default()


def W(b, L, H, G, seed=0, **kw):
    return Mamba2Workload(f"m2-b{b}-L{L}-h{H}-g{G}", b, L, H, 64, G, 128, "bf16", seed=seed, **kw)


def oracle_with_bounds(orc, inp, softplus=True, h0=None):
    ref_y, ref_s = orc.ssd(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"], inp["D"],
                           inp["dt_bias"], softplus, dtype="bf16", initial_state=h0)
    D_abs = None if inp["D"] is None else inp["D"].abs()
    abs_y, abs_s = orc.ssd(inp["x"].abs(), inp["dt"], inp["A"], inp["B"].abs(), inp["C"].abs(),
                           D_abs, inp["dt_bias"], softplus, dtype="bf16",
                           initial_state=None if h0 is None else np.abs(h0))
    return ref_y, ref_s, abs_y, abs_s


def check(got_y, got_s, ref_y, ref_s, abs_y, abs_s):
    gy = got_y.float().cpu().numpy().astype(np.float64)
    err = np.abs(gy - ref_y)
    bound = 1.1 * (2 * U * abs_y + U * np.abs(ref_y)) + 1e-6
    assert np.all(err <= bound), f"y: max |err|/bound {np.max(err / bound):.3g}"
    norm = np.linalg.norm(gy - ref_y) / max(np.linalg.norm(ref_y), 1e-30)
    assert norm <= 4 * U, f"y: normwise error {norm:.3e} > {4 * U:.3e}"
    io = err / (1e-2 * (1 + np.abs(ref_y)))
    print(f"[bf16 I/O bound] y: worst |err| / (1e-2 (1+|ref|)) = {io.max():.3g}")
    if got_s is not None:
        gs = got_s.cpu().numpy().astype(np.float64)
        err_s = np.abs(gs - ref_s)
        bound_s = 1.1 * U * abs_s + 1e-6
        assert np.all(err_s <= bound_s), f"state: max |err|/bound {np.max(err_s / bound_s):.3g}"
        io_s = err_s / (1e-2 * (1 + np.abs(ref_s)))
        print(f"[bf16 I/O bound] state: worst |err| / (1e-2 (1+|ref|)) = {io_s.max():.3g}")


def run(inp, softplus=True, final=True, h0=None, final_buf=None):
    d = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    out = ss.mamba2_fwd(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], d["dt_bias"], softplus,
                        return_final_state=final, initial_state=h0, final_state=final_buf)
    torch.cuda.synchronize()
    assert ss.ss_selective_scan_check(None) == ss.SS_OK
    return out if final else (out, None)


def run_case(orc, w, softplus=True, mutate=None):
    inp = make_mamba2_inputs(w)
    if mutate:
        mutate(inp)
    y, s = run(inp, softplus)
    check(y, s, *oracle_with_bounds(orc, inp, softplus))


def test_small_workload(orc):
    run_case(orc, MAMBA2_WORKLOADS["m2_small"])


@pytest.mark.parametrize("L", [1, 2, 127, 128, 129, 255, 512])
def test_sequence_lengths(orc, L):
    run_case(orc, W(1, L, 2, 1, seed=20 + L))


@pytest.mark.parametrize("H,G", [(8, 1), (6, 3), (4, 4)])
def test_groups(orc, H, G):
    run_case(orc, W(2, 200, H, G, seed=31 + H + G))


@pytest.mark.parametrize("opts", [dict(has_D=False), dict(has_bias=False),
                                  dict(has_D=False, has_bias=False)])
def test_optional_inputs(orc, opts):
    run_case(orc, W(2, 150, 4, 2, seed=41, **opts))


def test_without_softplus(orc):
    def small_positive_dt(inp):
        inp["dt"] = (inp["dt"].float().abs() * 0.05 + 1e-3).to(torch.bfloat16)
        inp["dt_bias"] = None
    run_case(orc, W(2, 260, 4, 2, seed=43), softplus=False, mutate=small_positive_dt)


def test_without_final_state(orc):
    w = W(1, 140, 2, 1, seed=44)
    inp = make_mamba2_inputs(w)
    y, _ = run(inp, final=False)
    ref_y, ref_s, abs_y, abs_s = oracle_with_bounds(orc, inp)
    check(y, None, ref_y, ref_s, abs_y, abs_s)


def test_full_size_sampled_heads(orc):
    """The Mamba-2-2.7B-shaped layer in the benchmark's launch; (batch, head)
    units sampled across the grid are checked against the oracle on their own
    slices (each unit is independent)."""
    w = MAMBA2_WORKLOADS["m2_2.7b"]
    inp = make_mamba2_inputs(w)
    y, s = run(inp)
    y, s = y.cpu(), s.cpu()
    H, G = w.nheads, w.ngroups
    for b, h in [(0, 0), (3, 41), (7, 79)]:
        g = h // (H // G)
        sub = {"x": inp["x"][b:b + 1, :, h:h + 1].contiguous(),
               "dt": inp["dt"][b:b + 1, :, h:h + 1].contiguous(),
               "A": inp["A"][h:h + 1].contiguous(),
               "B": inp["B"][b:b + 1, :, g:g + 1].contiguous(),
               "C": inp["C"][b:b + 1, :, g:g + 1].contiguous(),
               "D": inp["D"][h:h + 1].contiguous(),
               "dt_bias": inp["dt_bias"][h:h + 1].contiguous()}
        check(y[b:b + 1, :, h:h + 1], s[b:b + 1, h:h + 1], *oracle_with_bounds(orc, sub))


def initial_state(w, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randn((w.batch, w.nheads, w.headdim, w.dstate), generator=g) * 0.5


@pytest.mark.parametrize("L", [1, 127, 128, 129, 300])
def test_from_initial_state(orc, L):
    """The state before step 0 given: it enters chunk 0 the way a carried
    state enters every later chunk (its bf16 copy in the C.H^T product)."""
    w = W(2, L, 4, 2, seed=60 + L)
    inp = make_mamba2_inputs(w)
    h0 = initial_state(w, 61 + L)
    y, s = run(inp, h0=h0.cuda())
    check(y, s, *oracle_with_bounds(orc, inp, h0=h0.numpy().astype(np.float64)))


def test_initial_state_updated_in_place(orc):
    w = W(1, 200, 2, 1, seed=62)
    inp = make_mamba2_inputs(w)
    h0 = initial_state(w, 63)
    buf = h0.clone().cuda()
    y, s = run(inp, h0=buf, final_buf=buf)
    assert s.data_ptr() == buf.data_ptr()
    check(y, s, *oracle_with_bounds(orc, inp, h0=h0.numpy().astype(np.float64)))


def test_chained_calls_at_a_chunk_boundary_equal_one_call():
    """Split at a multiple of the 128-step chunk, the second call starts from
    the first call's fp32 final state, which is exactly the state the single
    call carries across that boundary: the results agree bit for bit."""
    w = W(2, 384, 4, 2, seed=64)
    inp = make_mamba2_inputs(w)
    y_all, s_all = run(inp)
    part = lambda sl: {k: (v[:, sl].contiguous() if k in ("x", "dt", "B", "C") else v)
                       for k, v in inp.items()}
    y1, s1 = run(part(slice(0, 256)))
    y2, s2 = run(part(slice(256, 384)), h0=s1)
    assert torch.equal(torch.cat([y1, y2], 1), y_all)
    assert torch.equal(s2, s_all)


def test_is_deterministic():
    inp = make_mamba2_inputs(W(2, 300, 4, 2, seed=45))
    y1, s1 = run(inp)
    y2, s2 = run(inp)
    assert torch.equal(y1, y2) and torch.equal(s1, s2)


def test_rejects_more_than_256_states():
    inp = make_mamba2_inputs(Mamba2Workload("m2-n257", 1, 16, 2, 32, 1, 257, seed=46))
    d = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    with pytest.raises(ss.SelectiveScanError):
        ss.mamba2_fwd(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], d["dt_bias"])
