"""Write the stored expected values under tests/golden/ (test infrastructure).

Each fixture holds small seeded inputs and the fp64 oracle's results for them,
so that the tests can check the oracle against its stored results (a change in
its arithmetic shows up as a diff that has to be regenerated on purpose) and
the CUDA path against the same numbers.  Only the seeded input generators and
oracle/ are used here.  Run from the repository root:

    python tests/golden/make_golden.py
"""
import json
import sys
from pathlib import Path

import numpy as np

HERE = Path(__file__).resolve().parent
sys.path.insert(0, str(HERE.parent.parent))

import oracle  # noqa: E402
from mamba_selective_scan_ss_gb300.inputs import (Mamba2Workload, ScanWorkload,  # noqa: E402
                                                  make_inputs, make_mamba2_inputs)


def arr(t):
    return None if t is None else np.asarray(t, dtype=np.float64).tolist()


def inputs_of(inp):
    return {k: (arr(v.double().numpy()) if hasattr(v, "double") else v) for k, v in inp.items()}


def forward_case(name, w, cite, h0=None):
    orc = oracle.default()
    inp = make_inputs(w)
    y, last = orc.fwd(inp["u"], inp["delta"], inp["A"], inp["B"], inp["C"], inp["D"], inp["z"],
                      inp["delta_bias"], inp["delta_softplus"], h0=h0, dtype="f32")
    out = {"kind": "forward", "citation": cite, "inputs": inputs_of(inp),
           "h0": arr(h0), "y": arr(y), "last_state": arr(last)}
    (HERE / f"{name}.json").write_text(json.dumps(out, indent=0) + "\n")


def backward_case(name, w, cite):
    orc = oracle.default()
    inp = make_inputs(w)
    rng = np.random.default_rng(5)
    dy = rng.standard_normal((w.batch, w.dim, w.seqlen))
    g = orc.bwd(inp["u"], inp["delta"], inp["A"], inp["B"], inp["C"], inp["D"], inp["z"],
                inp["delta_bias"], inp["delta_softplus"], dy=dy.astype(np.float32), dtype="f32")
    out = {"kind": "backward", "citation": cite, "inputs": inputs_of(inp),
           "dy": arr(dy.astype(np.float32)), "grads": {k: arr(v) for k, v in g.items()}}
    (HERE / f"{name}.json").write_text(json.dumps(out, indent=0) + "\n")


def mamba2_case(name, w, cite):
    orc = oracle.default()
    inp = make_mamba2_inputs(w)
    y, fin = orc.ssd(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"], inp["D"],
                     inp["dt_bias"], inp["dt_softplus"], dtype="f32")
    out = {"kind": "mamba2", "citation": cite, "inputs": inputs_of(inp), "y": arr(y),
           "final_state": arr(fin)}
    (HERE / f"{name}.json").write_text(json.dumps(out, indent=0) + "\n")


SCAN = ('"Mamba CUDA 实现解析" eq (4)-(7) (the selective-scan recurrence and read-out) with the '
        'task spec\'s skip D*u and silu(z) gate ("ТЕХНИЧЕСКОЕ ЗАДАНИЕ: Реализовать selective '
        'scan (Mamba)", Этап 1)')

if __name__ == "__main__":
    forward_case("forward_b1_d4_n4_L16_f32", ScanWorkload("g-fwd", 1, 4, 4, 16, "f32", seed=101),
                 SCAN)
    h0 = np.random.default_rng(6).standard_normal((1, 3, 4))
    forward_case("forward_h0_b1_d3_n4_L9_f32", ScanWorkload("g-fwd-h0", 1, 3, 4, 9, "f32", seed=102),
                 SCAN + "; from a given state h0 (the sequential form of the Blelloch article, "
                 "section 1)", h0=h0)
    backward_case("backward_b1_d2_n4_L6_f32", ScanWorkload("g-bwd", 1, 2, 4, 6, "f32", seed=103),
                  "the chain rule through " + SCAN + " (gradients the task spec asks to check by "
                  "gradcheck, Этап 3 step 4)")
    mamba2_case("mamba2_b1_L5_h2_p2_n3_f32", Mamba2Workload("g-m2", 1, 5, 2, 2, 1, 3, "f32",
                                                            seed=104),
                "the per-head recurrence of the Mamba-2 cuTile news page (section on the "
                "technical details of the optimisation)")
    print("written")
