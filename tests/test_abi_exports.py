"""The C-ABI library builds, loads and exports every symbol its header declares;
host-side argument validation rejects bad calls before touching the device.
CPU only: no call here reaches a kernel or the CUDA runtime."""
import ctypes
import re
import subprocess
from pathlib import Path

import pytest

from mamba_selective_scan_ss_gb300 import _build
import mamba_selective_scan_ss_gb300 as ss

HEADER = Path(__file__).resolve().parent.parent / "include" / "ss_selective_scan.h"


@pytest.fixture(scope="module")
def lib():
    _build.build_all()
    return ss.load_library()


def declared_functions():
    text = HEADER.read_text()
    return sorted(set(re.findall(r"SS_API\s+[\w\s\*]+?\b(ss_\w+)\s*\(", text)))


def test_header_declares_the_entry_points():
    assert declared_functions() == ["ss_mamba2_fwd", "ss_mamba2_fwd_h0", "ss_selective_scan_bwd",
                                    "ss_selective_scan_bwd_h0", "ss_selective_scan_check",
                                    "ss_selective_scan_fwd",
                                    "ss_selective_scan_fwd_h0", "ss_selective_scan_fwd_host",
                                    "ss_selective_scan_fwd_noalloc",
                                    "ss_selective_scan_fwd_pc", "ss_selective_scan_fwd_pc_h0",
                                    "ss_selective_scan_plan", "ss_selective_state_update",
                                    "ss_status_string"]


def test_library_exports_every_declared_symbol(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", str(ss.library_path())],
                         capture_output=True, text=True, check=True).stdout
    exported = set(re.findall(r"\bT (ss_\w+)", out))
    for name in declared_functions():
        assert name in exported, name
        assert hasattr(lib, name)


def test_shipped_library_has_no_test_hooks(lib):
    """The tuning overrides and the unit-skipping hook live only in the test
    build: the shipped library neither names their variables nor exports the
    hook's kernel."""
    shipped = ss.library_path().read_bytes()
    for name in (b"SS_TEST_SKIP_UNITS", b"SS_NCHUNKS", b"SS_CTAS_PER_SM", b"SS_MAMBA2_ROWS",
                 b"ss_set_ticket"):
        assert name not in shipped, name
    test = ss.library_path(test_build=True).read_bytes()
    assert b"SS_TEST_SKIP_UNITS" in test and b"SS_NCHUNKS" in test


def test_status_strings(lib):
    assert ss.ss_status_string(ss.SS_OK) == "SS_OK"
    assert ss.ss_status_string(ss.SS_ERR_TIMEOUT) == "SS_ERR_TIMEOUT"
    assert ss.ss_status_string(99) == "SS_UNKNOWN_STATUS"


def _fake_ptrs():
    # host buffers stand in for device pointers: validation never dereferences them
    bufs = [ctypes.create_string_buffer(4096) for _ in range(11)]
    return bufs, [ctypes.addressof(b) for b in bufs]


def test_validation_rejects_bad_arguments(lib):
    bufs, p = _fake_ptrs()
    u, dl, A, B, C, D, z, bias, y, st, _ = p
    ok = dict(u=u, delta=dl, A=A, B=B, C=C, D=D, z=z, delta_bias=bias, delta_softplus=1,
              y=y, last_state=st, batch=1, dim=2, dstate=4, seqlen=8, dtype=ss.SS_F32,
              stream=None)

    def call(**kw):
        a = dict(ok, **kw)
        return ss.ss_selective_scan_fwd(**a)

    assert call(u=None) == ss.SS_ERR_INVALID_ARGUMENT
    assert call(B=None) == ss.SS_ERR_INVALID_ARGUMENT
    assert call(y=None) == ss.SS_ERR_INVALID_ARGUMENT
    assert call(batch=0) == ss.SS_ERR_INVALID_ARGUMENT       # batch=0: refused, no crash
    assert call(seqlen=0) == ss.SS_ERR_INVALID_ARGUMENT
    assert call(dim=-3) == ss.SS_ERR_INVALID_ARGUMENT
    assert call(dstate=257) == ss.SS_ERR_UNSUPPORTED
    assert call(dtype=7) == ss.SS_ERR_UNSUPPORTED
    assert call(batch=1 << 40, dim=1 << 30) == ss.SS_ERR_UNSUPPORTED   # overflows int64
    assert call(y=u) == ss.SS_ERR_INVALID_ARGUMENT           # output aliases an input
    assert call(y=u + 16) == ss.SS_ERR_INVALID_ARGUMENT      # partial overlap
    assert call(last_state=dl) == ss.SS_ERR_INVALID_ARGUMENT
    assert call(last_state=y) == ss.SS_ERR_INVALID_ARGUMENT
    assert call(u=u + 1) == ss.SS_ERR_INVALID_ARGUMENT       # misaligned fp32 pointer
    assert call(A=A + 2) == ss.SS_ERR_INVALID_ARGUMENT
    assert call(u=u + 1, dtype=ss.SS_BF16) == ss.SS_ERR_INVALID_ARGUMENT  # odd bf16 address


def test_validation_of_the_initial_state_entry_point(lib):
    bufs, p = _fake_ptrs()
    u, dl, A, B, C, D, z, bias, y, st, h0 = p
    ok = dict(u=u, delta=dl, A=A, B=B, C=C, D=D, z=z, delta_bias=bias, delta_softplus=1, h0=h0,
              y=y, last_state=st, batch=1, dim=2, dstate=4, seqlen=8, dtype=ss.SS_F32,
              stream=None)

    def call(**kw):
        return ss.ss_selective_scan_fwd_h0(**dict(ok, **kw))

    assert call(u=None) == ss.SS_ERR_INVALID_ARGUMENT
    assert call(h0=h0 + 2) == ss.SS_ERR_INVALID_ARGUMENT       # misaligned fp32 state
    assert call(y=h0) == ss.SS_ERR_INVALID_ARGUMENT            # output over the initial state
    assert call(last_state=h0 + 4) == ss.SS_ERR_INVALID_ARGUMENT  # partial overlap (not in place)
    assert call(last_state=u) == ss.SS_ERR_INVALID_ARGUMENT
    assert call(dstate=300) == ss.SS_ERR_UNSUPPORTED
    assert call(seqlen=0) == ss.SS_ERR_INVALID_ARGUMENT


def test_validation_of_the_decode_step(lib):
    bufs, p = _fake_ptrs()
    state, x, dt, A, B, C, D, z, bias, y, _ = p
    ok = dict(state=state, x=x, dt=dt, A=A, B=B, C=C, D=D, z=z, dt_bias=bias, dt_softplus=1,
              y=y, batch=2, dim=3, dstate=4, dtype=ss.SS_F32, stream=None)

    def call(**kw):
        return ss.ss_selective_state_update(**dict(ok, **kw))

    assert call(state=None) == ss.SS_ERR_INVALID_ARGUMENT
    assert call(C=None) == ss.SS_ERR_INVALID_ARGUMENT
    assert call(batch=0) == ss.SS_ERR_INVALID_ARGUMENT
    assert call(dstate=257) == ss.SS_ERR_UNSUPPORTED
    assert call(dtype=5) == ss.SS_ERR_UNSUPPORTED
    assert call(batch=1 << 40, dim=1 << 30) == ss.SS_ERR_UNSUPPORTED
    assert call(y=x) == ss.SS_ERR_INVALID_ARGUMENT             # output over an input
    assert call(state=B) == ss.SS_ERR_INVALID_ARGUMENT         # state over an input
    assert call(y=state + 8) == ss.SS_ERR_INVALID_ARGUMENT     # output over the state
    assert call(state=state + 2) == ss.SS_ERR_INVALID_ARGUMENT  # misaligned fp32 state
    assert call(x=x + 1, dtype=ss.SS_BF16) == ss.SS_ERR_INVALID_ARGUMENT


def test_validation_of_the_backward(lib):
    bufs = [ctypes.create_string_buffer(4096) for _ in range(19)]
    p = [ctypes.addressof(b) for b in bufs]
    names = ["u", "delta", "A", "B", "C", "D", "z", "delta_bias", "dy", "dlast_state", "du",
             "ddelta", "dA", "dB", "dC", "dD", "dz", "dbias"]
    ok = dict(zip(names, p), delta_softplus=1, batch=1, dim=2, dstate=4, seqlen=8,
              dtype=ss.SS_F32, stream=None)

    def call(**kw):
        return ss.ss_selective_scan_bwd(**dict(ok, **kw))

    assert call(dy=None) == ss.SS_ERR_INVALID_ARGUMENT
    assert call(dB=None) == ss.SS_ERR_INVALID_ARGUMENT
    assert call(dz=None) == ss.SS_ERR_INVALID_ARGUMENT          # z given, dz missing
    assert call(dstate=257) == ss.SS_ERR_UNSUPPORTED            # backward: dstate <= 256
    assert call(seqlen=0) == ss.SS_ERR_INVALID_ARGUMENT
    assert call(dtype=3) == ss.SS_ERR_UNSUPPORTED
    assert call(du=ok["u"]) == ss.SS_ERR_INVALID_ARGUMENT       # output over an input
    assert call(dC=ok["dB"] + 8) == ss.SS_ERR_INVALID_ARGUMENT  # two outputs overlap
    assert call(dA=ok["dA"] + 2) == ss.SS_ERR_INVALID_ARGUMENT  # misaligned fp32 output

    # the initial-state variant: h0 is an input, dh0 an output
    extra = [ctypes.create_string_buffer(4096) for _ in range(2)]
    h0, dh0 = (ctypes.addressof(b) for b in extra)

    def call_h0(**kw):
        args = dict(ok, h0=h0, dh0=dh0)
        args.update(kw)
        return ss.ss_selective_scan_bwd_h0(**args)

    assert call_h0(dh0=ok["u"]) == ss.SS_ERR_INVALID_ARGUMENT   # dh0 over an input
    assert call_h0(dh0=ok["dA"]) == ss.SS_ERR_INVALID_ARGUMENT  # dh0 over another output
    assert call_h0(du=h0) == ss.SS_ERR_INVALID_ARGUMENT         # an output over h0
    assert call_h0(h0=h0 + 2) == ss.SS_ERR_INVALID_ARGUMENT     # misaligned h0
    assert call_h0(dstate=257) == ss.SS_ERR_UNSUPPORTED



def test_validation_of_the_mamba2_forward(lib):
    bufs = [ctypes.create_string_buffer(4096) for _ in range(10)]
    p = [ctypes.addressof(b) for b in bufs]
    names = ["x", "dt", "A", "B", "C", "D", "dt_bias", "y", "final_state"]
    ok = dict(zip(names, p), dt_softplus=1, batch=1, seqlen=8, nheads=2, headdim=64,
              ngroups=1, dstate=128, dtype=ss.SS_BF16, stream=None)

    def call(**kw):
        return ss.ss_mamba2_fwd(**dict(ok, **kw))

    assert call(x=None) == ss.SS_ERR_INVALID_ARGUMENT
    assert call(y=None) == ss.SS_ERR_INVALID_ARGUMENT
    assert call(seqlen=0) == ss.SS_ERR_INVALID_ARGUMENT
    assert call(nheads=3, ngroups=2) == ss.SS_ERR_INVALID_ARGUMENT  # heads not a multiple of groups
    assert call(dtype=7) == ss.SS_ERR_UNSUPPORTED
    assert call(dstate=257) == ss.SS_ERR_UNSUPPORTED                # at most 256 states
    assert call(headdim=32, dstate=257) == ss.SS_ERR_UNSUPPORTED    # on the general path too
    assert call(dtype=ss.SS_F32, dstate=300) == ss.SS_ERR_UNSUPPORTED
    assert call(x=ok["x"] + 1) == ss.SS_ERR_INVALID_ARGUMENT        # not aligned to its element
    assert call(dtype=ss.SS_F32, B=ok["B"] + 2) == ss.SS_ERR_INVALID_ARGUMENT
    assert call(y=ok["x"]) == ss.SS_ERR_INVALID_ARGUMENT            # output over an input
    assert call(final_state=ok["y"]) == ss.SS_ERR_INVALID_ARGUMENT  # outputs overlap

def test_plan_is_host_only_and_consistent(lib, monkeypatch):
    monkeypatch.delenv("SS_NCHUNKS", raising=False)
    monkeypatch.delenv("SS_CTAS_PER_SM", raising=False)
    # vector path: one scheduled launch per call, chunks joined inside the kernel
    p = ss.ss_selective_scan_plan(8, 5120, 16, 2048, ss.SS_BF16, True, 152)
    assert p["state_groups"] == 1 and p["vector_path"] == 1 and p["kernel_launches"] == 1
    assert p["nchunks"] >= 1 and p["ctas"] <= 152 * 8
    # few rows and a long sequence: many chunks, still one launch
    p = ss.ss_selective_scan_plan(1, 2048, 16, 65536, ss.SS_BF16, True, 152)
    assert p["nchunks"] > 1 and p["kernel_launches"] == 1
    assert p["chunk_len"] % 64 == 0 and (p["nchunks"] - 1) * p["chunk_len"] < 65536
    assert p["scratch_bytes"] > 0
    # dstate above 16 runs in state groups, one launch per group
    p = ss.ss_selective_scan_plan(2, 64, 40, 256, ss.SS_F32, True, 152)
    assert p["state_groups"] == 3 and p["kernel_launches"] == 3
    # misaligned pointers or odd lengths take the scalar path (aggregate + carry + main)
    p = ss.ss_selective_scan_plan(2, 64, 16, 250, ss.SS_BF16, True, 152)
    assert p["vector_path"] == 0
    assert ss.ss_selective_scan_plan(2, 64, 16, 256, ss.SS_BF16, False, 152)["vector_path"] == 0
    monkeypatch.setenv("SS_NCHUNKS", "4")
    # the shipped library reads no environment variable: the plan is unchanged
    plain = ss.ss_selective_scan_plan(2, 64, 16, 1024, ss.SS_F32, True, 152)
    monkeypatch.delenv("SS_NCHUNKS")
    assert plain == ss.ss_selective_scan_plan(2, 64, 16, 1024, ss.SS_F32, True, 152)
    # the test build honours the override, on both paths
    monkeypatch.setenv("SS_NCHUNKS", "4")
    with ss.test_hooks():
        p = ss.ss_selective_scan_plan(2, 64, 16, 1024, ss.SS_F32, False, 152)
        assert p["nchunks"] == 4 and p["kernel_launches"] == 3
        assert p["scratch_bytes"] == 3 * 128 * 16 * 8 + 4 * 128 * 16 * 4
        assert ss.ss_selective_scan_plan(2, 64, 16, 1024, ss.SS_F32, True, 152)["nchunks"] == 4
    with pytest.raises(ss.SelectiveScanError):
        ss.ss_selective_scan_plan(0, 64, 16, 1024, ss.SS_F32, True, 152)
    with pytest.raises(ss.SelectiveScanError):
        ss.ss_selective_scan_plan(1, 64, 300, 1024, ss.SS_F32, True, 152)
