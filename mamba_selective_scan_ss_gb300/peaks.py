"""Loader for the unit-throughput microbenchmarks (libss_peaks.so).

The roofline of the selective-scan forward kernel needs the per-SM rates of
the MUFU ex2 unit and of the FP32 FMA pipe, which are measured here on the
device at hand rather than taken from a data sheet, and the shared-memory load
rates that bound how fast B and C reach the lanes.
"""
from __future__ import annotations

import ctypes
from pathlib import Path

_LIB = None

PROBES = {
    "ex2": 0,             # MUFU ex2 results
    "ffma": 1,            # scalar FP32 FMA lane-ops
    "ffma2": 2,           # packed f32x2 FMA lane-ops
    "update_scalar": 3,   # selective-scan state updates, scalar FP32 body
    "update_packed": 4,   # selective-scan state updates, the scan kernel's f32x2 lane layout
    "update_mix": 5,      # pipe mix of one update (2 FFMA2 + 1 ex2), nothing else
    "lds128_bcast": 6,    # 16-byte shared-memory loads, every lane the same address
    "lds128_distinct": 7,  # 16-byte shared-memory loads, each lane its own address
    "lds32_bcast": 8,     # 4-byte shared-memory loads, every lane the same address
}

DEFAULT_ITERS = {"ex2": 20000, "ffma": 40000, "ffma2": 20000,
                 "update_scalar": 4000, "update_packed": 500, "update_mix": 20000,
                 "lds128_bcast": 20000, "lds128_distinct": 20000, "lds32_bcast": 20000}


def _lib():
    global _LIB
    if _LIB is None:
        path = Path(__file__).resolve().parent / "libss_peaks.so"
        if not path.exists():
            raise RuntimeError(f"{path.name} is not built; run __graft_entry__.build()")
        lib = ctypes.CDLL(str(path))
        lib.ss_peaks_measure.restype = ctypes.c_int
        lib.ss_peaks_measure.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                         ctypes.c_int, ctypes.POINTER(ctypes.c_double)]
        _LIB = lib
    return _LIB


def measure(probe: str, iters: int | None = None, blocks_per_sm: int = 4,
            threads: int = 256) -> dict:
    """Run one probe; returns rates over the GPU and per clock per SM."""
    res = (ctypes.c_double * 5)()
    it = iters if iters is not None else DEFAULT_ITERS[probe]
    rc = _lib().ss_peaks_measure(PROBES[probe], it, blocks_per_sm, threads, res)
    if rc != 0:
        raise RuntimeError(f"peaks probe {probe} failed with CUDA error {rc}")
    return {"probe": probe, "per_s": res[0], "per_clk_per_sm": res[1],
            "sm_mhz": res[2], "sms": int(res[3]), "ms": res[4],
            "blocks_per_sm": blocks_per_sm, "threads": threads}


def main() -> None:
    """Print every probe as one JSON line, at 1, 2 and 8 warps per scheduler
    for the update probes (occupancy scaling of the update body)."""
    import json

    runs = [("ex2", 4, 256), ("ffma", 4, 256), ("ffma2", 4, 256),
            ("lds128_bcast", 4, 256), ("lds128_distinct", 4, 256), ("lds32_bcast", 4, 256)]
    for probe in ("update_mix", "update_packed", "update_scalar"):
        runs += [(probe, 2, 64), (probe, 4, 64), (probe, 4, 256)]
    for probe, bps, thr in runs:
        r = measure(probe, blocks_per_sm=bps, threads=thr)
        r["warps_per_scheduler"] = bps * thr / 32 / 4
        print(json.dumps(r), flush=True)


if __name__ == "__main__":
    main()
