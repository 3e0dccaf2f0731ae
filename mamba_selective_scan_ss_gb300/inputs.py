"""Seeded synthetic inputs for the selective-scan forward workloads.

This module only draws random tensors in the layouts of the C ABI; it holds
none of the scan's arithmetic.  Both the CUDA path and the CPU oracle are fed
from here, so that they see bit-identical inputs.

Workload shapes (batch, dim, dstate, seqlen) and value distributions:
  * u, delta_raw, z ~ N(0, 1), layout [batch, dim, seqlen]
  * per-channel step size dt ~ LogUniform[lo, hi] and delta_bias = log(expm1(dt)),
    i.e. the inverse of softplus, so softplus(0 + delta_bias) = dt
  * A[d, n] = -(n + 1)                       (the real diagonal init of Mamba)
  * B, C ~ N(0, 1), layout [batch, dstate, seqlen], shared by all channels
    (bc_per_channel workloads: [batch, dim, dstate, seqlen], one row per channel)
  * D ~ N(0, 1), layout [dim]
Draw order is u, delta_raw, dt, B, C, D, z from one torch CPU generator seeded
with the workload's seed.  For bf16 workloads u, delta_raw, B, C and z are
rounded to bf16 (round to nearest even) before either side sees them; A, D,
delta_bias stay fp32.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, replace

import torch


@dataclass(frozen=True)
class ScanWorkload:
    name: str
    batch: int
    dim: int
    dstate: int
    seqlen: int
    dtype: str = "f32"            # "f32" or "bf16": type of u, delta, B, C, z, y
    has_z: bool = True
    has_D: bool = True
    has_bias: bool = True
    softplus: bool = True
    dt_lo: float = 1e-3
    dt_hi: float = 1e-1
    seed: int = 0
    bc_per_channel: bool = False  # B, C [batch, dim, dstate, seqlen] instead of shared

    @property
    def updates(self) -> int:
        """State updates of one forward pass: batch * dim * seqlen * dstate."""
        return self.batch * self.dim * self.seqlen * self.dstate

    @property
    def elt(self) -> int:
        return 4 if self.dtype == "f32" else 2

    def algorithmic_bytes(self) -> int:
        """Bytes one forward pass must move at least once through HBM.

        u, delta, (z) in and y out are [b, d, L]; B and C are [b, N, L];
        A is [d, N]; D and delta_bias [d]; last_state [b, d, N] fp32 out.
        """
        bdl = self.batch * self.dim * self.seqlen
        streams = 3 + (1 if self.has_z else 0)          # u, delta, y (+ z)
        b = streams * bdl * self.elt
        b += 2 * self.batch * self.dstate * self.seqlen * self.elt * (
            self.dim if self.bc_per_channel else 1)
        b += 4 * self.dim * self.dstate
        b += 4 * self.dim * (int(self.has_D) + int(self.has_bias))
        b += 4 * self.batch * self.dim * self.dstate
        return b

    def with_(self, **kw) -> "ScanWorkload":
        return replace(self, **kw)


def _cfg4(L: int) -> ScanWorkload:
    return ScanWorkload(f"seqlen-sweep-b16-d1536-n16-L{L}-f32", 16, 1536, 16, L, "f32",
                        has_z=True, seed=4)


WORKLOADS = {
    "0": ScanWorkload("tiny-b2-d16-n16-L128-f32", 2, 16, 16, 128, "f32",
                      has_z=False, seed=0),
    "1": ScanWorkload("mamba130m-layer-b2-d1536-n16-L2048-f32", 2, 1536, 16, 2048, "f32",
                      has_z=True, seed=1),
    "2": ScanWorkload("mamba2.8b-layer-b8-d5120-n16-L2048-bf16", 8, 5120, 16, 2048, "bf16",
                      has_z=True, seed=2),
    "3": ScanWorkload("long-seq-b1-d2048-n16-L65536-bf16", 1, 2048, 16, 65536, "bf16",
                      has_z=True, dt_lo=1e-4, dt_hi=1e-2, seed=3),
    "4_256": _cfg4(256),
    "4_1024": _cfg4(1024),
    "4_4096": _cfg4(4096),
    "4_16384": _cfg4(16384),
    # per-channel B/C (one row per channel): a Mamba-2.8B-shaped layer at L=512
    "pc_2": ScanWorkload("per-channel-bc-b8-d5120-n16-L512-bf16", 8, 5120, 16, 512, "bf16",
                         has_z=True, seed=9, bc_per_channel=True),
}


def make_inputs(w: ScanWorkload) -> dict:
    """Draw one workload's inputs on the CPU (torch tensors, ABI layout)."""
    g = torch.Generator(device="cpu")
    g.manual_seed(w.seed)
    b, d, n, L = w.batch, w.dim, w.dstate, w.seqlen
    io = torch.float32 if w.dtype == "f32" else torch.bfloat16

    u = torch.randn((b, d, L), generator=g, dtype=torch.float32)
    delta = torch.randn((b, d, L), generator=g, dtype=torch.float32)
    lo, hi = math.log(w.dt_lo), math.log(w.dt_hi)
    dt = torch.exp(torch.rand((d,), generator=g, dtype=torch.float64) * (hi - lo) + lo)
    bc_shape = (b, d, n, L) if w.bc_per_channel else (b, n, L)
    Bm = torch.randn(bc_shape, generator=g, dtype=torch.float32)
    Cm = torch.randn(bc_shape, generator=g, dtype=torch.float32)
    D = torch.randn((d,), generator=g, dtype=torch.float32)
    z = torch.randn((b, d, L), generator=g, dtype=torch.float32) if w.has_z else None

    A = -torch.arange(1, n + 1, dtype=torch.float32).repeat(d, 1).contiguous()
    bias = torch.log(torch.expm1(dt)).to(torch.float32)

    out = {
        "u": u.to(io).contiguous(),
        "delta": delta.to(io).contiguous(),
        "A": A,
        "B": Bm.to(io).contiguous(),
        "C": Cm.to(io).contiguous(),
        "D": D if w.has_D else None,
        "z": z.to(io).contiguous() if z is not None else None,
        "delta_bias": bias if w.has_bias else None,
        "delta_softplus": bool(w.softplus),
    }
    return out


# ---- decode step: one token from a given state -------------------------------
@dataclass(frozen=True)
class DecodeWorkload:
    name: str
    batch: int
    dim: int
    dstate: int
    dtype: str = "bf16"
    has_z: bool = True
    has_D: bool = True
    has_bias: bool = True
    seed: int = 0

    @property
    def updates(self) -> int:
        """State updates of one step: batch * dim * dstate."""
        return self.batch * self.dim * self.dstate

    @property
    def elt(self) -> int:
        return 4 if self.dtype == "f32" else 2

    def algorithmic_bytes(self) -> int:
        """State read and written once; x, dt, z read and y written once; B, C,
        A, D and the bias read once."""
        rows = self.batch * self.dim
        streams = 3 + int(self.has_z)
        b = 8 * rows * self.dstate
        b += streams * rows * self.elt
        b += 2 * self.batch * self.dstate * self.elt
        b += 4 * self.dim * self.dstate
        b += 4 * self.dim * (int(self.has_D) + int(self.has_bias))
        return b


DECODE_WORKLOADS = {
    # one token of a Mamba-2.8B-shaped layer (dim 5120) for 64 sequences
    "decode_64": DecodeWorkload("decode-b64-d5120-n16-bf16", 64, 5120, 16, "bf16", seed=7),
    "decode_256": DecodeWorkload("decode-b256-d5120-n16-bf16", 256, 5120, 16, "bf16", seed=8),
}


def make_decode_inputs(w: DecodeWorkload) -> dict:
    """One token's inputs and a state, on the CPU, in the C ABI layouts.

    The forward's recipe restricted to one step: x, dt_raw, z ~ N(0, 1) [b, d];
    dt ~ LogUniform[1e-3, 1e-1] per channel and dt_bias = log(expm1(dt));
    A[d, n] = -(n + 1); B, C ~ N(0, 1) [b, N]; D ~ N(0, 1) [d]; the state
    ~ N(0, 1) [b, d, N] fp32.  Draw order x, dt_raw, dt, B, C, D, z, state.
    bf16 workloads round x, dt_raw, B, C and z to bf16 before either side sees
    them.
    """
    g = torch.Generator(device="cpu")
    g.manual_seed(w.seed)
    b, d, n = w.batch, w.dim, w.dstate
    io = torch.float32 if w.dtype == "f32" else torch.bfloat16
    x = torch.randn((b, d), generator=g, dtype=torch.float32)
    dt_raw = torch.randn((b, d), generator=g, dtype=torch.float32)
    lo, hi = math.log(1e-3), math.log(1e-1)
    dt = torch.exp(torch.rand((d,), generator=g, dtype=torch.float64) * (hi - lo) + lo)
    Bm = torch.randn((b, n), generator=g, dtype=torch.float32)
    Cm = torch.randn((b, n), generator=g, dtype=torch.float32)
    D = torch.randn((d,), generator=g, dtype=torch.float32)
    z = torch.randn((b, d), generator=g, dtype=torch.float32)
    state = torch.randn((b, d, n), generator=g, dtype=torch.float32)
    A = -torch.arange(1, n + 1, dtype=torch.float32).repeat(d, 1).contiguous()
    bias = torch.log(torch.expm1(dt)).to(torch.float32)
    return {
        "state": state,
        "x": x.to(io).contiguous(),
        "dt": dt_raw.to(io).contiguous(),
        "A": A,
        "B": Bm.to(io).contiguous(),
        "C": Cm.to(io).contiguous(),
        "D": D if w.has_D else None,
        "z": z.to(io).contiguous() if w.has_z else None,
        "dt_bias": bias if w.has_bias else None,
        "dt_softplus": True,
    }


# ---------------------------------------------------------------- Mamba-2
@dataclass(frozen=True)
class Mamba2Workload:
    """A Mamba-2 forward (one scalar decay per head): x [b, L, H, P], dt
    [b, L, H], B and C [b, L, G, N], A, D and dt_bias [H]."""
    name: str
    batch: int
    seqlen: int
    nheads: int
    headdim: int
    ngroups: int
    dstate: int
    dtype: str = "bf16"
    has_D: bool = True
    has_bias: bool = True
    seed: int = 0

    @property
    def updates(self) -> int:
        """State updates of one call: batch * seqlen * nheads * headdim * dstate."""
        return self.batch * self.seqlen * self.nheads * self.headdim * self.dstate

    @property
    def elt(self) -> int:
        return 4 if self.dtype == "f32" else 2

    def algorithmic_bytes(self) -> int:
        """x, dt, B, C read once, y written once, the final state written once,
        A, D and the bias read once."""
        tok = self.batch * self.seqlen
        b = 2 * tok * self.nheads * self.headdim * self.elt     # x, y
        b += tok * self.nheads * self.elt                       # dt
        b += 2 * tok * self.ngroups * self.dstate * self.elt    # B, C
        b += 4 * self.batch * self.nheads * self.headdim * self.dstate  # final state
        b += 4 * self.nheads * (1 + int(self.has_D) + int(self.has_bias))
        return b

    def chunk_flops(self, chunk: int) -> int:
        """Multiply-add flops of the chunked evaluation with chunks of ``chunk``
        steps: per (batch, chunk, group) C B^T; per (batch, chunk, head) the
        masked product with x, the read-out of the incoming state and the
        chunk's own state."""
        nch = -(-self.seqlen // chunk)
        q, p, n = chunk, self.headdim, self.dstate
        per_head = 2 * q * q * p + 2 * q * n * p + 2 * q * n * p
        per_group = 2 * q * q * n
        return self.batch * nch * (self.nheads * per_head + self.ngroups * per_group)


MAMBA2_WORKLOADS = {
    # a Mamba-2-2.7B-shaped layer: d_inner 5120 = 80 heads of 64, 128 states, one group
    "m2_2.7b": Mamba2Workload("mamba2-2.7b-layer-b8-L2048-h80-p64-n128-bf16", 8, 2048, 80, 64, 1,
                              128, "bf16", seed=12),
    # small case the oracle finishes in seconds: three chunks (the last ragged), two groups
    "m2_small": Mamba2Workload("mamba2-small-b2-L300-h4-p64-n128-g2-bf16", 2, 300, 4, 64, 2, 128,
                               "bf16", seed=11),
}


def make_mamba2_inputs(w: Mamba2Workload) -> dict:
    """Draw a Mamba-2 workload's inputs on the CPU (torch tensors, ABI layouts).

    x, dt_raw ~ N(0, 1); per-head step dt ~ LogUniform[1e-3, 1e-1] and dt_bias =
    log(expm1(dt)); A[h] = -U[1, 16] (the Mamba-2 initialisation range);
    B, C ~ N(0, 1) [b, L, G, N]; D ~ N(0, 1) [H].  Draw order x, dt_raw, dt, A,
    B, C, D.  bf16 workloads round x, dt_raw, B and C to bf16.
    """
    g = torch.Generator(device="cpu")
    g.manual_seed(w.seed)
    b, L, H, P, G, N = w.batch, w.seqlen, w.nheads, w.headdim, w.ngroups, w.dstate
    io = torch.float32 if w.dtype == "f32" else torch.bfloat16
    x = torch.randn((b, L, H, P), generator=g, dtype=torch.float32)
    dt_raw = torch.randn((b, L, H), generator=g, dtype=torch.float32)
    lo, hi = math.log(1e-3), math.log(1e-1)
    dt = torch.exp(torch.rand((H,), generator=g, dtype=torch.float64) * (hi - lo) + lo)
    A = -(1.0 + 15.0 * torch.rand((H,), generator=g, dtype=torch.float32))
    Bm = torch.randn((b, L, G, N), generator=g, dtype=torch.float32)
    Cm = torch.randn((b, L, G, N), generator=g, dtype=torch.float32)
    D = torch.randn((H,), generator=g, dtype=torch.float32)
    bias = torch.log(torch.expm1(dt)).to(torch.float32)
    return {
        "x": x.to(io).contiguous(),
        "dt": dt_raw.to(io).contiguous(),
        "A": A.contiguous(),
        "B": Bm.to(io).contiguous(),
        "C": Cm.to(io).contiguous(),
        "D": D if w.has_D else None,
        "dt_bias": bias if w.has_bias else None,
        "dt_softplus": True,
    }
