"""Host-side plan of ss_selective_scan_fwd_noalloc (CPU only, no CUDA call).

The no-allocation entry point keeps the regular plan but lowers the chunk
count to the largest one whose carries fit its fixed 16 MiB buffer.  The test
build of the library exposes that plan (ss_test_noalloc_plan), so the choice
can be checked without a GPU."""
import ctypes

import pytest

import mamba_selective_scan_ss_gb300 as ss
from mamba_selective_scan_ss_gb300 import _build

LIMIT = 16 << 20
REC_BYTES = 64 * 16 * 12  # per chunk and 64-channel row tile: 16 states x (8 + 4) bytes


@pytest.fixture(scope="module")
def tlib():
    _build.build_all()
    lib = ss.load_library(test_build=True)
    i64 = ctypes.c_int64
    lib.ss_test_noalloc_plan.restype = ctypes.c_int
    lib.ss_test_noalloc_plan.argtypes = [i64, i64, i64, i64, ctypes.c_int, ctypes.c_int,
                                         ctypes.POINTER(ss._Plan)]
    return lib


def noalloc_plan(lib, b, d, n, L, dt, sms=152):
    p = ss._Plan()
    st = lib.ss_test_noalloc_plan(b, d, n, L, dt, sms, ctypes.byref(p))
    return st, {k: getattr(p, k) for k, _ in ss._Plan._fields_}


@pytest.mark.parametrize("shape", [
    (8, 5120, 16, 2048, ss.SS_BF16),    # chained chunks (load balance only): 8 -> fewer
    (1, 3584, 16, 16384, ss.SS_BF16),   # decoupled look-back over many chunks: 32 -> 24
    (16, 1536, 16, 16384, ss.SS_F32),   # the fp32 sequence sweep at L = 16384
])
def test_chunks_lowered_to_the_largest_count_that_fits(tlib, shape):
    b, d, n, L, dt = shape
    with ss.test_hooks():
        regular = ss.ss_selective_scan_plan(b, d, n, L, dt, True, 152)
    assert regular["scratch_bytes"] > LIMIT          # the regular plan would not fit
    st, p = noalloc_plan(tlib, b, d, n, L, dt)
    assert st == ss.SS_OK
    assert 1 < p["nchunks"] < regular["nchunks"]
    assert p["scratch_bytes"] <= LIMIT
    assert p["chunk_len"] % 64 == 0 and (p["nchunks"] - 1) * p["chunk_len"] < L <= \
        p["nchunks"] * p["chunk_len"]
    # one chunk more would not fit: the records alone would pass the limit
    tiles = b * ((d + 63) // 64)
    assert (p["nchunks"] + 1) * tiles * REC_BYTES > LIMIT - 128 - (p["nchunks"] + 1) * tiles * 4


def test_small_problem_keeps_the_regular_plan(tlib):
    with ss.test_hooks():
        regular = ss.ss_selective_scan_plan(1, 256, 16, 8192, ss.SS_F32, True, 152)
    st, p = noalloc_plan(tlib, 1, 256, 16, 8192, ss.SS_F32)
    assert st == ss.SS_OK and p["nchunks"] == regular["nchunks"]


def test_what_cannot_fit_is_refused(tlib):
    # dstate 32: the fp32 partial read-out of batch*dim*seqlen (32 MiB) alone
    st, _ = noalloc_plan(tlib, 1, 2048, 32, 4096, ss.SS_F32)
    assert st == ss.SS_ERR_SCRATCH_LIMIT
