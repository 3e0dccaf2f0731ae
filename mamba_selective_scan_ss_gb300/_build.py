"""In-tree build of the native libraries (nvcc for sm_103a, gcc for host C).

Every library is rebuilt only when the hash of its sources and flags changes;
the hash is kept in a ``.stamp`` file beside the library.  Libraries are
compiled in parallel so a cold build stays within a few tens of seconds.
"""
from __future__ import annotations

import hashlib
import os
import shutil
import subprocess
from dataclasses import dataclass, field
from pathlib import Path

PKG_DIR = Path(__file__).resolve().parent
CSRC = PKG_DIR / "csrc"
REPO_ROOT = PKG_DIR.parent
INCLUDE = REPO_ROOT / "include"

ARCH_FLAGS = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_COMMON = [
    *ARCH_FLAGS,
    "-O3",
    "-lineinfo",
    "-std=c++17",
    "-Xcompiler", "-fPIC",
    "-Xcompiler", "-fvisibility=hidden",
    "-shared",
]


@dataclass
class NativeLib:
    name: str                     # output file name, e.g. libss_selective_scan.so
    sources: list[Path]
    deps: list[Path] = field(default_factory=list)   # headers that trigger a rebuild
    extra: list[str] = field(default_factory=list)
    compiler: str = "nvcc"

    @property
    def path(self) -> Path:
        return PKG_DIR / self.name

    def command(self) -> list[str]:
        if self.compiler == "nvcc":
            return ["nvcc", *NVCC_COMMON, f"-I{INCLUDE}", *self.extra,
                    *map(str, self.sources), "-o", str(self.path)]
        raise ValueError(self.compiler)

    def digest(self) -> str:
        h = hashlib.sha256()
        h.update(" ".join(self.command()).encode())
        for p in [*self.sources, *self.deps]:
            h.update(p.read_bytes())
        return h.hexdigest()


def _kernel_headers() -> list[Path]:
    return sorted(CSRC.glob("*.cuh")) + sorted(INCLUDE.glob("*.h"))


def libraries() -> list[NativeLib]:
    libs = [NativeLib("libss_peaks.so", [CSRC / "peaks.cu"])]
    api = CSRC / "ss_api.cu"
    if api.exists():
        libs.insert(0, NativeLib(
            "libss_selective_scan.so",
            [api],
            deps=_kernel_headers(),
            extra=["-DSS_BUILDING_LIBRARY", "-Xptxas", "-warn-spills"],
        ))
        # the same sources with the test hooks (plan overrides, skipped units)
        # compiled in: loaded only by the tests that force scheduling modes or
        # make a device wait run out
        libs.insert(1, NativeLib(
            "libss_selective_scan_test.so",
            [api],
            deps=_kernel_headers(),
            extra=["-DSS_BUILDING_LIBRARY", "-DSS_TEST_HOOKS"],
        ))
    return libs


def build_all(verbose: bool = False, force: bool = False) -> list[Path]:
    """Compile every native library of the package; returns their paths."""
    if shutil.which("nvcc") is None:
        raise RuntimeError("nvcc not found on PATH: cannot build the CUDA libraries")
    procs = []
    for lib in libraries():
        stamp = lib.path.with_suffix(".stamp")
        dig = lib.digest()
        if (not force and lib.path.exists() and stamp.exists()
                and stamp.read_text().strip() == dig):
            continue
        cmd = lib.command()
        if verbose:
            print(" ".join(cmd), flush=True)
        tmp_out = lib.path.with_suffix(".so.tmp")
        cmd[-1] = str(tmp_out)
        procs.append((lib, stamp, dig, tmp_out,
                      subprocess.Popen(cmd, stdout=subprocess.PIPE,
                                       stderr=subprocess.STDOUT, text=True)))
    errors = []
    for lib, stamp, dig, tmp_out, p in procs:
        out, _ = p.communicate()
        if p.returncode != 0:
            errors.append(f"{lib.name}:\n{out}")
            continue
        if verbose and out.strip():
            print(out, flush=True)
        os.replace(tmp_out, lib.path)
        stamp.write_text(dig + "\n")
    if errors:
        raise RuntimeError("native build failed:\n" + "\n".join(errors))
    return [lib.path for lib in libraries()]
