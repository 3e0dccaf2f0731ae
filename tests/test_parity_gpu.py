"""CUDA path against the CPU oracle, element by element, through the C ABI.

Tolerances are those fixed for the method's outputs: for fp32 I/O
|err| <= 1e-5 + 1e-4*|ref|, for bf16 I/O |err| <= 1e-2*(1 + |ref|), applied to
both y and last_state.  Small cases compare every element; the full-size
workloads, run in the benchmark's launch configuration, compare sampled
channel rows that the oracle evaluates one by one.
"""
import os

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


def to_dev(inp):
    return {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}


def run_gpu(inp, **kw):
    d = to_dev(inp)
    y, last = ss.selective_scan_fwd(d["u"], d["delta"], d["A"], d["B"], d["C"], d["D"], d["z"],
                                    d["delta_bias"], d["delta_softplus"], **kw)
    torch.cuda.synchronize()
    assert ss.ss_selective_scan_check(None) == ss.SS_OK
    return y.float().cpu().numpy().astype(np.float64), last.cpu().numpy().astype(np.float64)


def run_oracle(orc, inp, dtype):
    return orc.fwd(inp["u"], inp["delta"], inp["A"], inp["B"], inp["C"], inp["D"], inp["z"],
                   inp["delta_bias"], inp["delta_softplus"], dtype=dtype)


def assert_close(got, ref, dtype, what):
    atol, rtol = TOL[dtype]
    err = np.abs(got - ref)
    bound = atol + rtol * np.abs(ref)
    bad = ~(err <= bound)
    if bad.any():
        i = np.unravel_index(np.argmax(np.where(bad, err / bound, 0)), err.shape)
        raise AssertionError(f"{what}: {bad.sum()}/{bad.size} out of tolerance; worst at {i}: "
                             f"got {got[i]!r} ref {ref[i]!r} (|err| {err[i]:.3e} > {bound[i]:.3e})")


def check(orc, w: ScanWorkload, inp=None, **kw):
    inp = inp if inp is not None else make_inputs(w)
    y, last = run_gpu(inp, **kw)
    y_ref, last_ref = run_oracle(orc, inp, w.dtype)
    assert_close(y, y_ref, w.dtype, f"{w.name} y")
    assert_close(last, last_ref, w.dtype, f"{w.name} last_state")


def W(b, d, n, L, dtype="f32", **kw):
    return ScanWorkload(f"b{b}-d{d}-n{n}-L{L}-{dtype}", b, d, n, L, dtype, **kw)


# ---- the tiny workload and the task spec's test sizes (batch, dim, seqlen) ----
def test_tiny_workload(orc):
    check(orc, WORKLOADS["0"])


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("b,d,L", [(2, 4, 8), (1, 32, 256), (8, 128, 64)])
def test_task_spec_sizes(orc, dtype, b, d, L):
    check(orc, W(b, d, 16, L, dtype, seed=b * 1000 + L))


# ---- degenerate and edge cases ----
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("shape", [(1, 1, 16, 1), (3, 1, 16, 40), (2, 5, 16, 1), (1, 1, 1, 1),
                                   (1, 130, 16, 67), (2, 129, 16, 1000), (1, 7, 16, 8)])
def test_edge_shapes(orc, dtype, shape):
    check(orc, W(*shape, dtype, seed=sum(shape)))


@pytest.mark.parametrize("dstate", [1, 2, 3, 4, 5, 7, 8, 9, 12, 16, 17, 24, 32, 33, 64, 100, 256])
def test_dstate(orc, dstate):
    check(orc, W(2, 20, dstate, 96, seed=dstate))


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("opts", [dict(has_z=False), dict(has_D=False), dict(has_bias=False),
                                  dict(softplus=False, dt_lo=1e-2, dt_hi=1e-1),
                                  dict(has_z=False, has_D=False, has_bias=False)])
def test_optional_inputs(orc, dtype, opts):
    w = W(2, 48, 16, 200, dtype, seed=7, **opts)
    inp = make_inputs(w)
    if not w.softplus:
        # without softplus dt = delta + bias must stay positive: shift delta
        inp["delta"] = (inp["delta"].float().abs() * 0.05 + 0.01).to(inp["delta"].dtype)
        inp["delta_bias"] = None
    check(orc, w, inp)


# ---- dt = softplus(delta + bias) over its whole range ----
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("seqlen", [1, 64])
def test_softplus_sweep(orc, dtype, seqlen):
    """delta + bias swept over [-20, 20] across channels, so dt runs from 2e-9
    to 20 through the kernel's softplus: seqlen 1 is the closed form of a
    single step (the scalar path), seqlen 64 the vector path's polynomial."""
    w = W(1, 4096, 16, seqlen, dtype, seed=41)
    inp = make_inputs(w)
    inp["delta_bias"] = torch.linspace(-20.0, 20.0, w.dim, dtype=torch.float32)
    inp["delta"] = (0.01 * inp["delta"].float()).to(inp["delta"].dtype)
    check(orc, w, inp)


# ---- sequence split into chunks joined by the eq (10) operator ----
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("nchunks", [2, 3, 7, 16])
@pytest.mark.parametrize("L,dstate", [(1000, 16), (4096, 16), (777, 33), (640, 8)])
def test_chunked_sequence(test_build, orc, monkeypatch, dtype, nchunks, L, dstate):
    monkeypatch.setenv("SS_NCHUNKS", str(nchunks))
    check(orc, W(2, 70, dstate, L, dtype, seed=nchunks + L, dt_lo=1e-4, dt_hi=1e-2))


# ---- the ticketed scheduler in each of its modes ----
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("ctas_per_sm,shape,nchunks", [
    (1, (4, 2560, 16, 1024), 4),   # more row tiles than CTAs: chained chunks
    (2, (2, 5120, 16, 1024), 8),   # fewer tiles than CTAs: decoupled, long look-backs
    (4, (1, 256, 16, 4096), 32),   # few tiles, many chunks: decoupled look-back
])
def test_scheduler_modes(test_build, orc, monkeypatch, dtype, ctas_per_sm, shape, nchunks):
    monkeypatch.setenv("SS_CTAS_PER_SM", str(ctas_per_sm))
    monkeypatch.setenv("SS_NCHUNKS", str(nchunks))
    w = W(*shape, dtype, seed=ctas_per_sm * 7 + nchunks, dt_lo=1e-4, dt_hi=1e-2)
    inp = make_inputs(w)
    y, last = run_gpu(inp)
    rows = sample_rows(w, 64, seed=5)
    ref = oracle_rows(orc, inp, w, rows)
    yf = y.reshape(-1, w.seqlen)
    sf = last.reshape(-1, w.dstate)
    for r in sorted(ref):
        assert_close(yf[r], ref[r][0], dtype, f"row {r} y")
        assert_close(sf[r], ref[r][1], dtype, f"row {r} state")


# ---- unaligned rows take the scalar path ----
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_unaligned_rows(orc, dtype):
    w = W(2, 33, 16, 128, dtype, seed=5)
    inp = make_inputs(w)
    # shift u/delta/z by one element inside a larger buffer: 16-byte alignment is lost
    for k in ("u", "delta", "z"):
        t = inp[k]
        big = torch.zeros(t.numel() + 1, dtype=t.dtype)
        big[1:] = t.reshape(-1)
        inp[k] = big[1:].view(t.shape)
    d = to_dev(inp)
    for k in ("u", "delta", "z"):
        base = torch.zeros(d[k].numel() + 1, dtype=d[k].dtype, device="cuda")
        base[1:] = d[k].reshape(-1)
        d[k] = base[1:].view(d[k].shape)
        assert d[k].data_ptr() % 16 != 0
    y, last = ss.selective_scan_fwd(d["u"], d["delta"], d["A"], d["B"], d["C"], d["D"], d["z"],
                                    d["delta_bias"], True)
    torch.cuda.synchronize()
    y_ref, last_ref = run_oracle(orc, inp, dtype)
    assert_close(y.float().cpu().numpy().astype(np.float64), y_ref, dtype, "unaligned y")
    assert_close(last.cpu().numpy().astype(np.float64), last_ref, dtype, "unaligned state")


# ---- bounds: guard bands around every output stay untouched ----
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("shape", [(2, 130, 16, 200), (1, 3, 5, 37)])
def test_guard_bands(test_build, orc, monkeypatch, dtype, shape):
    monkeypatch.setenv("SS_NCHUNKS", "3")
    w = W(*shape, dtype, seed=11)
    inp = make_inputs(w)
    d = to_dev(inp)
    pad = 4096
    io = d["u"].dtype
    ybuf = torch.full((d["u"].numel() + 2 * pad,), 7.0, dtype=io, device="cuda")
    sbuf = torch.full((w.batch * w.dim * w.dstate + 2 * pad,), 9.0, dtype=torch.float32,
                      device="cuda")
    y = ybuf[pad:pad + d["u"].numel()].view(d["u"].shape)
    st = sbuf[pad:pad + w.batch * w.dim * w.dstate].view(w.batch, w.dim, w.dstate)
    ss.selective_scan_fwd(d["u"], d["delta"], d["A"], d["B"], d["C"], d["D"], d["z"],
                          d["delta_bias"], True, y=y, last_state=st)
    torch.cuda.synchronize()
    for buf, val in ((ybuf, 7.0), (sbuf, 9.0)):
        assert torch.all(buf[:pad] == val) and torch.all(buf[-pad:] == val)
    y_ref, last_ref = run_oracle(orc, inp, dtype)
    assert_close(y.float().cpu().numpy().astype(np.float64), y_ref, dtype, "guarded y")
    assert_close(st.cpu().numpy().astype(np.float64), last_ref, dtype, "guarded state")


def test_deterministic():
    w = W(2, 300, 16, 3000, "bf16", seed=3)
    d = to_dev(make_inputs(w))
    outs = []
    for _ in range(2):
        y, st = ss.selective_scan_fwd(d["u"], d["delta"], d["A"], d["B"], d["C"], d["D"],
                                      d["z"], d["delta_bias"], True)
        torch.cuda.synchronize()
        outs.append((y.clone(), st.clone()))
    assert torch.equal(outs[0][0], outs[1][0]) and torch.equal(outs[0][1], outs[1][1])


def test_invalid_arguments_write_nothing():
    w = W(1, 4, 16, 32, seed=1)
    d = to_dev(make_inputs(w))
    y = torch.full_like(d["u"], 3.0)
    p = [d["u"].data_ptr(), d["delta"].data_ptr(), d["A"].data_ptr(), d["B"].data_ptr(),
         d["C"].data_ptr(), d["D"].data_ptr(), d["z"].data_ptr(), d["delta_bias"].data_ptr()]
    for bad in (dict(batch=0), dict(seqlen=0), dict(dstate=300)):
        kw = dict(batch=1, dim=4, dstate=16, seqlen=32)
        kw.update(bad)
        status = ss.ss_selective_scan_fwd(*p, 1, y.data_ptr(), None, kw["batch"], kw["dim"],
                                          kw["dstate"], kw["seqlen"], ss.SS_F32, None)
        assert status in (ss.SS_ERR_INVALID_ARGUMENT, ss.SS_ERR_UNSUPPORTED)
    # y aliasing u is refused
    status = ss.ss_selective_scan_fwd(*p, 1, d["u"].data_ptr(), None, 1, 4, 16, 32, ss.SS_F32,
                                      None)
    assert status == ss.SS_ERR_INVALID_ARGUMENT
    torch.cuda.synchronize()
    assert torch.all(y == 3.0)


# ---- full-size workloads in the benchmark's launch configuration: sampled rows ----
def sample_rows(w, count, seed):
    rng = np.random.default_rng(seed)
    rows = rng.choice(w.batch * w.dim, size=min(count, w.batch * w.dim), replace=False)
    rows = np.union1d(rows, [0, w.batch * w.dim - 1])
    return rows


def oracle_rows(orc, inp, w, rows):
    """Oracle on a subset of (batch, channel) rows; returns {row: (y, state)}."""
    out = {}
    by_batch = {}
    for r in rows:
        by_batch.setdefault(int(r) // w.dim, []).append(int(r) % w.dim)
    for b, ds in by_batch.items():
        ds = np.array(sorted(ds))
        sub = {
            "u": inp["u"][b:b + 1, ds], "delta": inp["delta"][b:b + 1, ds],
            "A": inp["A"][ds], "B": inp["B"][b:b + 1], "C": inp["C"][b:b + 1],
            "D": inp["D"][ds] if inp["D"] is not None else None,
            "z": inp["z"][b:b + 1, ds] if inp["z"] is not None else None,
            "delta_bias": inp["delta_bias"][ds] if inp["delta_bias"] is not None else None,
            "delta_softplus": inp["delta_softplus"],
        }
        y, st = run_oracle(orc, sub, w.dtype)
        for i, dd in enumerate(ds):
            out[b * w.dim + int(dd)] = (y[0, i], st[0, i])
    return out


@pytest.mark.parametrize("key", ["1", "2", "3", "4_256", "4_1024", "4_4096", "4_16384"])
def test_full_size_workload_sampled(orc, key):
    w = WORKLOADS[key]
    inp = make_inputs(w)
    d = to_dev(inp)
    y, st = ss.selective_scan_fwd(d["u"], d["delta"], d["A"], d["B"], d["C"], d["D"], d["z"],
                                  d["delta_bias"], True)
    torch.cuda.synchronize()
    assert ss.ss_selective_scan_check(None) == ss.SS_OK
    count = 48 if w.seqlen <= 4096 else 12
    rows = sample_rows(w, count, seed=int(w.seed) + 99)
    ref = oracle_rows(orc, inp, w, rows)
    yf = y.view(-1, w.seqlen)
    sf = st.view(-1, w.dstate)
    idx = torch.tensor(sorted(ref), dtype=torch.long, device="cuda")
    y_rows = yf[idx].float().cpu().numpy().astype(np.float64)
    s_rows = sf[idx].cpu().numpy().astype(np.float64)
    for i, r in enumerate(sorted(ref)):
        assert_close(y_rows[i], ref[r][0], w.dtype, f"{w.name} row {r} y")
        assert_close(s_rows[i], ref[r][1], w.dtype, f"{w.name} row {r} state")
    # every output is finite
    assert torch.isfinite(y.float()).all()


# Ragged rows of a size that takes the padded vector path (seqlen not a
# multiple of the 16-byte vector, rows x steps >= 2^16): the rows are copied
# into aligned, padded rows whose extra steps leave the state unchanged
# (dt = 0 there), the vector path runs on them and y is copied back.
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("shape", [(4, 512, 16, 1023), (2, 300, 16, 509), (1, 256, 32, 777)])
def test_ragged_rows_on_the_padded_vector_path(orc, dtype, shape):
    b, d, n, L = shape
    check(orc, ScanWorkload(f"ragged-b{b}-d{d}-n{n}-L{L}-{dtype}", b, d, n, L, dtype,
                            seed=L + d))


def _no_softplus_inputs(w, bias_value):
    """dt = delta + bias > 0 without the softplus, with a bias present."""
    inp = make_inputs(w)
    bias = torch.full((w.dim,), bias_value, dtype=torch.float32)
    delta = inp["delta"].float().abs() * 0.05 + 0.01
    inp["delta"] = delta.to(inp["delta"].dtype)
    inp["delta_bias"] = bias
    return inp


def test_ragged_rows_padded_without_softplus_fp32(orc):
    """No softplus, fp32: the padding's delta is -bias, which cancels the bias
    exactly, so the padded steps leave the state as it is."""
    w = ScanWorkload("ragged-nosp-b2-d300-n16-L511-f32", 2, 300, 16, 511, "f32",
                     softplus=False, seed=7)
    check(orc, w, _no_softplus_inputs(w, 0.37))


def test_ragged_rows_bf16_without_softplus_stay_scalar(orc):
    """bf16 without softplus and with a bias cannot pad exactly (-0.37 is not a
    bf16 value): the scalar path runs, and matches the oracle."""
    w = ScanWorkload("ragged-nosp-b2-d300-n16-L511-bf16", 2, 300, 16, 511, "bf16",
                     softplus=False, seed=8)
    check(orc, w, _no_softplus_inputs(w, 0.37))
