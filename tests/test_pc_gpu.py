"""Forward with B and C per channel against the oracle, through the C ABI.

ss_selective_scan_fwd_pc takes B and C as [batch, dim, dstate, seqlen] (one
row per channel); the oracle's forward reads the same layout
(bc_per_channel).  Tolerances are those of the forward: fp32 I/O
|err| <= 1e-5 + 1e-4*|ref|, bf16 I/O |err| <= 1e-2*(1 + |ref|), on y and
last_state.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import mamba_selective_scan_ss_gb300 as ss
import oracle
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


@pytest.fixture(scope="module")
def orc():
    return oracle.default()


def close(got, ref, dtype, what):
    atol, rtol = TOL[dtype]
    g = got.float().cpu().numpy().astype(np.float64)
    err = np.abs(g - ref)
    bound = atol + rtol * np.abs(ref)
    assert np.all(err <= bound), f"{what}: max |err|/bound {np.max(err / bound):.3g}"


def check(orc, w):
    inp = make_inputs(w)
    if not w.softplus:
        # without softplus dt = delta + bias must stay positive: shift delta
        inp["delta"] = (inp["delta"].float().abs() * 0.05 + 0.01).to(inp["delta"].dtype)
        inp["delta_bias"] = None
    d = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    y, last = ss.selective_scan_fwd(d["u"], d["delta"], d["A"], d["B"], d["C"], d["D"], d["z"],
                                    d["delta_bias"], d["delta_softplus"])
    torch.cuda.synchronize()
    y_ref, last_ref = orc.fwd(inp["u"], inp["delta"], inp["A"], inp["B"], inp["C"], inp["D"],
                              inp["z"], inp["delta_bias"], inp["delta_softplus"],
                              dtype=w.dtype, bc_per_channel=True)
    close(y, y_ref, w.dtype, "y")
    close(last, last_ref, w.dtype, "last_state")


def W(b, d, n, L, dtype="f32", **kw):
    return ScanWorkload(f"pc-b{b}-d{d}-n{n}-L{L}-{dtype}", b, d, n, L, dtype,
                        bc_per_channel=True, seed=kw.pop("seed", 81), **kw)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("shape", [(2, 33, 16, 64), (1, 5, 16, 37), (3, 70, 16, 200),
                                   (1, 1, 16, 1), (2, 300, 16, 24)])
def test_per_channel_forward(orc, dtype, shape):
    check(orc, W(*shape, dtype=dtype))


@pytest.mark.parametrize("dstate", [1, 3, 4, 5, 8, 12, 17, 32, 64, 100, 128,
                                    129, 160, 200, 256])
def test_per_channel_dstate(orc, dstate):
    """Up to 128 states a row's lanes sit in one warp; above, a row takes two
    warps whose read-outs meet in shared memory."""
    check(orc, W(2, 9, dstate, 40, seed=82))


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("dstate", [16, 200])
def test_per_channel_vector_path_wide_rows(orc, dtype, dstate):
    """Vector path (seqlen a multiple of 32 bytes of steps) with 64-lane rows
    and a ragged last CTA (3 * 7 rows)."""
    check(orc, W(3, 7, dstate, 96, dtype=dtype, seed=86))


def check_h0(orc, w, in_place=False):
    inp = make_inputs(w)
    g = torch.Generator().manual_seed(w.seed + 1)
    h0 = torch.randn((w.batch, w.dim, w.dstate), generator=g, dtype=torch.float32)
    d = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    h0_d = h0.cuda()
    last_buf = h0_d if in_place else None
    y, last = ss.selective_scan_fwd(d["u"], d["delta"], d["A"], d["B"], d["C"], d["D"], d["z"],
                                    d["delta_bias"], d["delta_softplus"], h0=h0_d,
                                    last_state=last_buf)
    torch.cuda.synchronize()
    y_ref, last_ref = orc.fwd(inp["u"], inp["delta"], inp["A"], inp["B"], inp["C"], inp["D"],
                              inp["z"], inp["delta_bias"], inp["delta_softplus"],
                              h0=h0.numpy(), dtype=w.dtype, bc_per_channel=True)
    close(y, y_ref, w.dtype, "y")
    close(last, last_ref, w.dtype, "last_state")
    if in_place:
        assert last.data_ptr() == h0_d.data_ptr()


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("shape", [(2, 33, 16, 64), (1, 5, 7, 37), (2, 6, 200, 48)])
def test_per_channel_from_initial_state(orc, dtype, shape):
    check_h0(orc, W(*shape, dtype=dtype, seed=87))


def test_per_channel_state_updated_in_place(orc):
    check_h0(orc, W(2, 10, 16, 32, seed=88), in_place=True)


def test_per_channel_chained_calls_equal_one_call():
    """Two calls, the second from the first's last state, give the result of
    one call over the whole sequence."""
    w = W(2, 12, 16, 128, seed=89)
    inp = make_inputs(w)
    d = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    args = lambda sl, ks: [d[k][..., sl].contiguous() if d[k] is not None else None for k in ks]
    y_all, s_all = ss.selective_scan_fwd(d["u"], d["delta"], d["A"], d["B"], d["C"], d["D"],
                                         d["z"], d["delta_bias"], True)
    half = slice(0, 64), slice(64, 128)
    ys, state = [], None
    for sl in half:
        u, dl, B, C, z = args(sl, ("u", "delta", "B", "C", "z"))
        y, state = ss.selective_scan_fwd(u, dl, d["A"], B, C, d["D"], z, d["delta_bias"], True,
                                         h0=state)
        ys.append(y)
    torch.cuda.synchronize()
    atol, rtol = TOL["f32"]
    assert torch.allclose(torch.cat(ys, -1), y_all, atol=atol, rtol=rtol)
    assert torch.allclose(state, s_all, atol=atol, rtol=rtol)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("opts", [dict(has_z=False), dict(has_D=False), dict(has_bias=False),
                                  dict(softplus=False)])
def test_per_channel_optional_inputs(orc, dtype, opts):
    check(orc, W(2, 20, 16, 48, dtype=dtype, seed=83, **opts))


def test_per_channel_with_shared_rows_equals_shared_layout():
    """Every channel given its batch row's B/C: the shared-layout forward's result."""
    w = ScanWorkload("pc-shared-b2-d40-n16-L64-f32", 2, 40, 16, 64, "f32", seed=84)
    inp = make_inputs(w)
    d = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    y_s, s_s = ss.selective_scan_fwd(d["u"], d["delta"], d["A"], d["B"], d["C"], d["D"], d["z"],
                                     d["delta_bias"], True)
    Bp = d["B"][:, None].expand(-1, w.dim, -1, -1).contiguous()
    Cp = d["C"][:, None].expand(-1, w.dim, -1, -1).contiguous()
    y_p, s_p = ss.selective_scan_fwd(d["u"], d["delta"], d["A"], Bp, Cp, d["D"], d["z"],
                                     d["delta_bias"], True)
    torch.cuda.synchronize()
    atol, rtol = TOL["f32"]
    assert torch.allclose(y_p, y_s, atol=atol, rtol=rtol)
    assert torch.allclose(s_p, s_s, atol=atol, rtol=rtol)


def test_per_channel_full_size_sampled_rows(orc):
    """The benchmark's per-channel workload (batch 8, dim 5120, 16 states,
    seqlen 512, bf16 I/O, z gate) in its launch: rows are independent, so
    blocks of 64 channels at the start, middle and end of the grid are checked
    against the oracle run on those rows alone."""
    w = WORKLOADS["pc_2"]
    inp = make_inputs(w)
    d = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    y, last = ss.selective_scan_fwd(d["u"], d["delta"], d["A"], d["B"], d["C"], d["D"], d["z"],
                                    d["delta_bias"], d["delta_softplus"])
    torch.cuda.synchronize()
    y, last = y.cpu(), last.cpu()
    for b, c0 in [(0, 0), (3, 2560), (7, w.dim - 64)]:
        rows = slice(c0, c0 + 64)
        sub = {k: inp[k][b:b + 1, rows].contiguous() for k in ("u", "delta", "z", "B", "C")}
        sub.update({k: inp[k][rows].contiguous() for k in ("A", "D", "delta_bias")})
        y_ref, last_ref = orc.fwd(sub["u"], sub["delta"], sub["A"], sub["B"], sub["C"], sub["D"],
                                  sub["z"], sub["delta_bias"], inp["delta_softplus"],
                                  dtype=w.dtype, bc_per_channel=True)
        close(y[b:b + 1, rows], y_ref, w.dtype, f"y rows {b},{c0}")
        close(last[b:b + 1, rows], last_ref, w.dtype, f"last_state rows {b},{c0}")


def test_per_channel_rejects_more_than_256_states():
    w = W(1, 2, 257, 8, seed=85)
    inp = make_inputs(w)
    d = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    with pytest.raises(ss.SelectiveScanError):
        ss.selective_scan_fwd(d["u"], d["delta"], d["A"], d["B"], d["C"], d["D"], d["z"],
                              d["delta_bias"], True)
