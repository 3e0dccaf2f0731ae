"""Pins of the CPU oracle against what the pages and the mathematics fix.

Every pin takes an ``oracle.Oracle`` and raises AssertionError if the oracle
disagrees with an independent statement of the result: a closed form, the
unrolled sum of "Mamba CUDA 实现解析" eq (8) evaluated by brute force, the
prefix formulation of eq (10)-(12), a special case that reduces to a library
routine, or an exact invariance.  None of them re-evaluates the oracle's own
recurrence.  ``tests/test_oracle_mutants.py`` runs the same battery against
mutated copies of the oracle to show that each plausible mistake fails at
least one pin.
"""
from __future__ import annotations

import numpy as np

RTOL = 1e-12     # fp64 closed forms against the fp64 oracle
ATOL = 1e-13


def _rand_problem(rng, b, d, n, L, *, z=True, D=True, bias=True, a_scale=1.0):
    """Small random fp32 problem with dt in a moderate range."""
    f = np.float32
    u = rng.standard_normal((b, d, L)).astype(f)
    delta = (rng.standard_normal((b, d, L)) * 0.5).astype(f)
    A = (-rng.uniform(0.2, 2.0, (d, n)) * a_scale).astype(f)
    B = rng.standard_normal((b, n, L)).astype(f)
    C = rng.standard_normal((b, n, L)).astype(f)
    Dv = rng.standard_normal(d).astype(f) if D else None
    zv = rng.standard_normal((b, d, L)).astype(f) if z else None
    bias_v = (rng.standard_normal(d) * 0.5 - 1.0).astype(f) if bias else None
    return dict(u=u, delta=delta, A=A, B=B, C=C, D=Dv, z=zv, delta_bias=bias_v)


def _softplus(x):
    # library form: log(exp(0) + exp(x))
    return np.logaddexp(0.0, x)


def _silu(z):
    # z * sigmoid(z) with sigmoid from its tanh identity
    return z * 0.5 * (1.0 + np.tanh(0.5 * z))


def _dt(p, softplus):
    x = p["delta"].astype(np.float64)
    if p["delta_bias"] is not None:
        x = x + p["delta_bias"].astype(np.float64)[None, :, None]
    return _softplus(x) if softplus else x


def _readout(p, h_all, softplus=True):
    """y from states h_all [b,d,L,N]: y = sum_n C h + D u, then the gate."""
    C = p["C"].astype(np.float64)                       # [b,N,L]
    y = np.einsum("bdtn,bnt->bdt", h_all, C)
    u = p["u"].astype(np.float64)
    if p["D"] is not None:
        y = y + p["D"].astype(np.float64)[None, :, None] * u
    if p["z"] is not None:
        y = y * _silu(p["z"].astype(np.float64))
    return y


def _close(got, want, rtol=RTOL, atol=ATOL, what=""):
    got, want = np.asarray(got), np.asarray(want)
    assert got.shape == want.shape, f"{what}: shape {got.shape} != {want.shape}"
    err = np.abs(got - want)
    tol = atol + rtol * np.abs(want)
    bad = err > tol
    assert not bad.any(), (f"{what}: {bad.sum()} of {bad.size} elements off, "
                           f"max err {err.max():.3e}")


# --------------------------------------------------------------------------
# Q1: brute force of the unrolled form, eq (8) of "Mamba CUDA 实现解析":
#   v_k = a_k...a_1 v_0 + sum_{j=1..k} (prod_{m=j+1..k} a_m) b_j u_j
# with a_m = exp(dt_m A), b_j = dt_j B_j (eq (5)-(6)); every product is formed
# explicitly, O(L^2 N), no recursion.
def pin_unrolled_sum(orc, seed=11):
    rng = np.random.default_rng(seed)
    for softplus in (True, False):
        for opts in (dict(), dict(z=False), dict(D=False, bias=False)):
            b, d, n, L = 2, 3, 4, 7
            p = _rand_problem(rng, b, d, n, L, **opts)
            h0 = rng.standard_normal((b, d, n))
            dt = _dt(p, softplus)                                   # [b,d,L]
            A = p["A"].astype(np.float64)                           # [d,N]
            a = np.exp(dt[..., None] * A[None, :, None, :])         # [b,d,L,N]
            Bt = np.transpose(p["B"].astype(np.float64), (0, 2, 1))  # [b,L,N]
            bu = dt[..., None] * Bt[:, None, :, :] * p["u"].astype(np.float64)[..., None]
            h_all = np.zeros((b, d, L, n))
            for k in range(L):
                total = np.ones((b, d, n))
                for m in range(0, k + 1):
                    total = total * a[:, :, m, :]
                acc = total * h0
                for j in range(0, k + 1):
                    prod = np.ones((b, d, n))
                    for m in range(j + 1, k + 1):
                        prod = prod * a[:, :, m, :]
                    acc = acc + prod * bu[:, :, j, :]
                h_all[:, :, k, :] = acc
            y_want = _readout(p, h_all)
            y, last = orc.fwd(**p, delta_softplus=softplus, h0=h0)
            _close(y, y_want, rtol=1e-11, atol=1e-12, what="eq(8) y")
            _close(last, h_all[:, :, -1, :], rtol=1e-11, atol=1e-12, what="eq(8) state")


# Q2: A = 0 makes every a_k = 1, so the state is a plain cumulative sum of
# dt*B*u (a textbook prefix sum, numpy.cumsum).
def pin_zero_A_is_cumsum(orc, seed=12):
    rng = np.random.default_rng(seed)
    b, d, n, L = 2, 3, 5, 33
    for softplus in (True, False):
        p = _rand_problem(rng, b, d, n, L)
        p["A"] = np.zeros_like(p["A"])
        dt = _dt(p, softplus)
        Bt = np.transpose(p["B"].astype(np.float64), (0, 2, 1))
        inc = dt[..., None] * Bt[:, None] * p["u"].astype(np.float64)[..., None]
        h_all = np.cumsum(inc, axis=2)
        y, last = orc.fwd(**p, delta_softplus=softplus)
        _close(y, _readout(p, h_all), rtol=1e-11, atol=1e-11, what="A=0 y")
        _close(last, h_all[:, :, -1], rtol=1e-11, atol=1e-11, what="A=0 state")


# Q3: inputs constant in time give constant a and c, and the closed geometric
# series h_k = c (1 - a^k) / (1 - a) (k = 1..L), y_k = sum_n C_n h_k + D u.
def pin_constant_inputs_geometric(orc):
    b, d, n, L = 1, 2, 3, 50
    f = np.float32
    u = np.full((b, d, L), 0.75, f)
    delta = np.full((b, d, L), -1.25, f)
    A = np.array([[-0.5, -1.0, -3.0], [-0.25, -2.0, -0.125]], f)
    Bv = np.array([0.5, -1.5, 2.0], f)
    Cv = np.array([1.25, 0.5, -0.75], f)
    B = np.repeat(Bv[None, :, None], L, axis=2).astype(f)
    C = np.repeat(Cv[None, :, None], L, axis=2).astype(f)
    Dv = np.array([0.3, -0.7], f)
    bias = np.array([0.5, -0.5], f)
    y, last = orc.fwd(u, delta, A, B, C, D=Dv, delta_bias=bias, delta_softplus=True)
    k = np.arange(1, L + 1, dtype=np.float64)
    for dd in range(d):
        dt = float(_softplus(np.float64(-1.25) + np.float64(bias[dd])))
        a = np.exp(dt * A[dd].astype(np.float64))                 # [N]
        c = dt * Bv.astype(np.float64) * 0.75
        h = c[None, :] * (1.0 - a[None, :] ** k[:, None]) / (1.0 - a[None, :])
        yk = h @ Cv.astype(np.float64) + float(Dv[dd]) * 0.75
        _close(y[0, dd], yk, rtol=1e-12, atol=1e-13, what="geometric y")
        _close(last[0, dd], h[-1], rtol=1e-12, atol=1e-13, what="geometric state")


# Q4a: eq (10) is associative ("Mamba CUDA 实现解析", the proof after eq (10)).
# Small integers make every product exact in fp64, so equality is exact.
def pin_combine_associative(orc, seed=14):
    rng = np.random.default_rng(seed)
    a1, v1, a2, c2, a3, c3 = (rng.integers(-9, 10, 4096).astype(np.float64) for _ in range(6))
    l_a, l_v = orc.combine(a1, v1, a2, c2)
    left = orc.combine(l_a, l_v, a3, c3)
    r_a, r_v = orc.combine(a2, c2, a3, c3)
    right = orc.combine(a1, v1, r_a, r_v)
    assert np.array_equal(left[0], right[0]) and np.array_equal(left[1], right[1])
    # and the operator itself, entry by entry, on the right-hand side of eq (10)
    assert np.array_equal(l_a, a2 * a1) and np.array_equal(l_v, a2 * v1 + c2)
    # identity element (1, 0)
    one, zero = np.ones(4), np.zeros(4)
    ia, iv = orc.combine(one, zero, a1[:4], c2[:4])
    assert np.array_equal(ia, a1[:4]) and np.array_equal(iv, c2[:4])


# Q4b: eq (11)-(12): the state at the end of the sequence is the second
# component of s_0 (+) E_1 (+) ... (+) E_K for any split into chunks, where E_k
# is the chunk's own (product of a, state reached from zero).  The chunk's
# product of a is read off the oracle as its response to h0 = 1 with u = 0.
# The outputs of a chunk run from the true carry equal the full run's outputs.
def pin_chunked_prefix(orc, seed=15):
    rng = np.random.default_rng(seed)
    b, d, n, L = 2, 3, 4, 64
    p = _rand_problem(rng, b, d, n, L)
    y_full, last_full = orc.fwd(**p)
    for cuts in ([17], [5, 40], [1, 2, 63], [20, 21, 22, 50]):
        bounds = [0, *cuts, L]
        s_a = np.ones((b, d, n))
        s_v = np.zeros((b, d, n))
        for lo, hi in zip(bounds[:-1], bounds[1:]):
            q = {k: (v[..., lo:hi].copy() if (isinstance(v, np.ndarray) and v.ndim == 3) else v)
                 for k, v in p.items()}
            # the chunk from the true carry reproduces the full run's outputs
            y_c, last_c = orc.fwd(**q, h0=s_v)
            _close(y_c, y_full[..., lo:hi], rtol=1e-12, atol=1e-13, what="chunk y")
            # E_k = (prod a, state from zero)
            _, e_v = orc.fwd(**q)
            q0 = dict(q, u=np.zeros_like(q["u"]))
            _, e_a = orc.fwd(**q0, h0=np.ones((b, d, n)))
            s_a, s_v = orc.combine(s_a, s_v, e_a, e_v)
            _close(s_v, last_c, rtol=1e-12, atol=1e-13, what="prefix vs carry")
        _close(s_v, last_full, rtol=1e-12, atol=1e-13, what="prefix state")
    # the product of a over the whole sequence is exp(A * sum dt)
    q0 = dict(p, u=np.zeros_like(p["u"]))
    _, pa = orc.fwd(**q0, h0=np.ones((b, d, n)))
    want = np.exp(_dt(p, True).sum(axis=2)[..., None] * p["A"].astype(np.float64)[None])
    _close(pa, want, rtol=1e-12, atol=1e-300, what="prod a")


# Q5: seqlen = 1 from a zero state: y = (dt u sum_n B_n C_n + D u) silu(z),
# last_state = dt u B.
def pin_single_step(orc, seed=16):
    rng = np.random.default_rng(seed)
    b, d, n = 3, 4, 6
    p = _rand_problem(rng, b, d, n, 1)
    dt = _dt(p, True)[..., 0]
    u = p["u"].astype(np.float64)[..., 0]
    Bv = p["B"].astype(np.float64)[..., 0]
    Cv = p["C"].astype(np.float64)[..., 0]
    bc = (Bv * Cv).sum(axis=1)                                   # [b]
    y_want = (dt * u * bc[:, None] + p["D"].astype(np.float64)[None] * u)
    y_want = y_want * _silu(p["z"].astype(np.float64)[..., 0])
    state_want = (dt * u)[..., None] * Bv[:, None, :]
    y, last = orc.fwd(**p)
    _close(y[..., 0], y_want, what="L=1 y")
    _close(last, state_want, what="L=1 state")


# Q6: dim = 1, N = 1, no D, no z, no bias, softplus off is the per-(b,d)
# thread loop sketched in "Реализовать selective scan (Mamba)", Этап 2
# (state = exp(delta*A)*state + delta*B*u; y = C*state), with B and C of the
# single channel.
def pin_task_spec_sketch(orc, seed=17):
    rng = np.random.default_rng(seed)
    b, L = 3, 40
    u = rng.standard_normal((b, 1, L)).astype(np.float32)
    delta = rng.uniform(0.01, 0.5, (b, 1, L)).astype(np.float32)
    A = np.array([[-0.8]], np.float32)
    B = rng.standard_normal((b, 1, L)).astype(np.float32)
    C = rng.standard_normal((b, 1, L)).astype(np.float32)
    y, last = orc.fwd(u, delta, A, B, C, delta_softplus=False)
    for bi in range(b):
        state = 0.0
        for t in range(L):
            dA = np.exp(float(delta[bi, 0, t]) * float(A[0, 0]))
            dB = float(delta[bi, 0, t]) * float(B[bi, 0, t])
            state = dA * state + dB * float(u[bi, 0, t])
            assert abs(y[bi, 0, t] - float(C[bi, 0, t]) * state) <= 1e-13 + 1e-12 * abs(state)
        assert abs(last[bi, 0, 0] - state) <= 1e-13 + 1e-12 * abs(state)


# Q7: A -> -inf makes a = 0: no memory, h_t = dt_t u_t B_t.
def pin_no_memory(orc, seed=18):
    rng = np.random.default_rng(seed)
    b, d, n, L = 2, 3, 4, 25
    p = _rand_problem(rng, b, d, n, L)
    p["A"] = np.full_like(p["A"], -1e30)
    dt = _dt(p, True)
    Bt = np.transpose(p["B"].astype(np.float64), (0, 2, 1))
    h_all = dt[..., None] * Bt[:, None] * p["u"].astype(np.float64)[..., None]
    y, last = orc.fwd(**p)
    _close(y, _readout(p, h_all), what="a=0 y")
    _close(last, h_all[:, :, -1], what="a=0 state")


# Q8: B = 0 leaves the state at zero, so y = D u silu(z) and last_state = 0;
# C = 0 gives the same y with a non-zero state.
def pin_zero_B_or_C(orc, seed=19):
    rng = np.random.default_rng(seed)
    b, d, n, L = 2, 3, 4, 30
    p = _rand_problem(rng, b, d, n, L)
    skip = (p["D"].astype(np.float64)[None, :, None] * p["u"].astype(np.float64)
            * _silu(p["z"].astype(np.float64)))
    y, last = orc.fwd(**dict(p, B=np.zeros_like(p["B"])))
    _close(y, skip, what="B=0 y")
    assert np.all(last == 0.0)
    y, last = orc.fwd(**dict(p, C=np.zeros_like(p["C"])))
    _close(y, skip, what="C=0 y")
    assert np.any(last != 0.0)


# Exact invariances: scaling u by 2 scales the state and the pre-gate output
# by exactly 2 (dt does not depend on u); permuting channels permutes the
# outputs when A, D and the bias are permuted with them; batches only see
# their own B and C.
def pin_invariances(orc, seed=20):
    rng = np.random.default_rng(seed)
    b, d, n, L = 3, 5, 4, 20
    p = _rand_problem(rng, b, d, n, L, z=False)
    y1, s1 = orc.fwd(**p)
    y2, s2 = orc.fwd(**dict(p, u=(p["u"] * np.float32(2.0))))
    assert np.array_equal(y2, 2.0 * y1) and np.array_equal(s2, 2.0 * s1)
    perm = rng.permutation(d)
    q = dict(p, u=p["u"][:, perm].copy(), delta=p["delta"][:, perm].copy(),
             A=p["A"][perm].copy(), D=p["D"][perm].copy(),
             delta_bias=p["delta_bias"][perm].copy())
    yp, sp = orc.fwd(**q)
    assert np.array_equal(yp, y1[:, perm]) and np.array_equal(sp, s1[:, perm])
    bperm = rng.permutation(b)
    q = dict(p, u=p["u"][bperm].copy(), delta=p["delta"][bperm].copy(),
             B=p["B"][bperm].copy(), C=p["C"][bperm].copy())
    yb, sb = orc.fwd(**q)
    assert np.array_equal(yb, y1[bperm]) and np.array_equal(sb, s1[bperm])


# bf16 inputs are widened exactly: the oracle fed bf16 bit patterns agrees
# bit for bit with the oracle fed the same values as fp32 (torch's own
# bf16 -> fp32 conversion).
def pin_bf16_widening(orc, seed=21):
    import torch
    g = torch.Generator().manual_seed(seed)
    b, d, n, L = 2, 3, 4, 16
    t = {k: torch.randn(s, generator=g) for k, s in
         (("u", (b, d, L)), ("delta", (b, d, L)), ("B", (b, n, L)), ("C", (b, n, L)),
          ("z", (b, d, L)))}
    A = -torch.rand((d, n), generator=g) - 0.1
    D = torch.randn(d, generator=g)
    bias = torch.randn(d, generator=g) - 2.0
    t16 = {k: v.to(torch.bfloat16) for k, v in t.items()}
    t32 = {k: v.to(torch.float32) for k, v in t16.items()}
    ya, sa = orc.fwd(**t16, A=A, D=D, delta_bias=bias, dtype="bf16")
    yb, sb = orc.fwd(**t32, A=A, D=D, delta_bias=bias, dtype="f32")
    assert np.array_equal(ya, yb) and np.array_equal(sa, sb)


# --------------------------------------------------------------------------
# The backward against finite differences of the forward.  The task spec asks
# for the gradients to be verified with gradcheck (Этап 3 step 4, section 5);
# here every gradient the oracle's backward returns is compared with central
# differences of the oracle's forward (itself pinned above) for the loss
# sum(dy * y) + sum(dlast * last_state).  Inputs are fp32, so each one is
# moved to the neighbouring fp32 values v +- e (e a power of two, exact), and
# two step sizes are combined by Richardson extrapolation, which leaves an
# O(e^4) truncation error (about 1e-9 here); h0 is fp64 and moved the same way.
def _fd_loss(orc, p, dy, dlast, softplus):
    y, last = orc.fwd(**p, delta_softplus=softplus)
    return float(np.sum(dy.astype(np.float64) * y) + np.sum(dlast * last))


def _fd_grad(orc, p, key, idx, dy, dlast, softplus):
    base = p[key]
    def at(delta):
        q = dict(p)
        arr = base.copy()
        arr[idx] = base[idx] + delta
        q[key] = arr
        return _fd_loss(orc, q, dy, dlast, softplus), float(arr[idx]) - float(base[idx])

    def central(e):
        lp, sp = at(e)
        lm, sm = at(-e)
        return (lp - lm) / (sp - sm)

    e = 2.0 ** -7
    return (4.0 * central(e / 2) - central(e)) / 3.0


def pin_backward_finite_differences(orc, seed=22):
    rng = np.random.default_rng(seed)
    for softplus, z, D, bias in ((True, True, True, True), (False, False, False, False),
                                 (True, False, True, False)):
        b, d, n, L = 2, 2, 3, 4
        p = _rand_problem(rng, b, d, n, L, z=z, D=D, bias=bias)
        if not softplus:  # a positive step without softplus
            p["delta"] = np.abs(p["delta"]).astype(np.float32) + np.float32(0.05)
            p["delta_bias"] = None
        p["h0"] = rng.standard_normal((b, d, n))
        dy = rng.standard_normal((b, d, L)).astype(np.float32)
        dlast = rng.standard_normal((b, d, n))
        g = orc.bwd(**p, delta_softplus=softplus, dy=dy, dlast=dlast)
        names = {"u": "du", "delta": "ddelta", "A": "dA", "B": "dB", "C": "dC", "D": "dD",
                 "z": "dz", "delta_bias": "dbias", "h0": "dh0"}
        for key, gname in names.items():
            if p.get(key) is None:
                assert g[gname] is None, f"{gname} returned for an absent input"
                continue
            fd = np.array([_fd_grad(orc, p, key, idx, dy, dlast, softplus)
                           for idx in np.ndindex(p[key].shape)]).reshape(p[key].shape)
            _close(g[gname], fd, rtol=1e-6, atol=1e-7, what=f"{gname} (softplus={softplus})")


# --------------------------------------------------------------------------
# Euler's identity for the backward: with the step sizes fixed, the loss
#   L = sum dy * y + sum dlast * last_state = sum dy' * y' + sum dlast * h_L
# (dy' = dy silu(z), y' the output before the gate) is linear in u, in B, in
# C and in D, so the gradient dotted with its own input gives back that part
# of the loss exactly:
#   sum u du = L,  sum B dB = sum dy' (C.h) + sum dlast h_L,
#   sum C dC = sum dy' (C.h),  sum D dD = sum dy' D u.
# The right-hand sides come from the forward (pinned above) run without the
# gate and without D; a wrong sign, index or missing term in du, dB, dC or dD
# breaks the equality.
def pin_backward_euler_identities(orc, seed=27):
    rng = np.random.default_rng(seed)
    for softplus, z, D, with_dlast in ((True, True, True, True), (False, False, True, False),
                                       (True, True, False, True)):
        b, d, n, L = 2, 3, 4, 6
        p = _rand_problem(rng, b, d, n, L, z=z, D=D)
        if not softplus:
            p["delta"] = np.abs(p["delta"]).astype(np.float32) + np.float32(0.05)
            p["delta_bias"] = None
        dy = rng.standard_normal((b, d, L)).astype(np.float32)
        dlast = rng.standard_normal((b, d, n)) if with_dlast else None
        g = orc.bwd(**p, delta_softplus=softplus, dy=dy, dlast=dlast)
        bare = dict(p, z=None, D=None)
        ch, h_L = orc.fwd(**bare, delta_softplus=softplus)   # C.h and the last state
        dyp = dy.astype(np.float64)
        if p["z"] is not None:
            dyp = dyp * _silu(p["z"].astype(np.float64))
        u = p["u"].astype(np.float64)
        du_part = (np.sum(dyp * u * p["D"].astype(np.float64)[None, :, None])
                   if p["D"] is not None else 0.0)
        last = float(np.sum(dlast * h_L)) if dlast is not None else 0.0
        lin = float(np.sum(dyp * ch))
        tag = f"(softplus={softplus}, z={z}, D={D}, dlast={with_dlast})"
        _close(np.sum(u * g["du"]), lin + du_part + last, rtol=1e-10, atol=1e-12,
               what=f"sum u du {tag}")
        _close(np.sum(p["B"].astype(np.float64) * g["dB"]), lin + last, rtol=1e-10,
               atol=1e-12, what=f"sum B dB {tag}")
        _close(np.sum(p["C"].astype(np.float64) * g["dC"]), lin, rtol=1e-10, atol=1e-12,
               what=f"sum C dC {tag}")
        if p["D"] is not None:
            _close(np.sum(p["D"].astype(np.float64) * g["dD"]), du_part, rtol=1e-10,
                   atol=1e-12, what=f"sum D dD {tag}")


# --------------------------------------------------------------------------
# Per-channel B/C (the task spec's kernel sketch keeps B and C per [b,d,t]):
# with every channel given the same rows the result equals the shared layout
# bit for bit, and every channel equals the shared-layout oracle run alone on
# that channel (batch 1, dim 1) with its own rows, bit for bit.
def pin_per_channel_bc(orc, seed=23):
    rng = np.random.default_rng(seed)
    b, d, n, L = 2, 3, 4, 7
    p = _rand_problem(rng, b, d, n, L)
    y_s, s_s = orc.fwd(**p)
    q = dict(p)
    q["B"] = np.ascontiguousarray(np.broadcast_to(p["B"][:, None], (b, d, n, L)))
    q["C"] = np.ascontiguousarray(np.broadcast_to(p["C"][:, None], (b, d, n, L)))
    y_b, s_b = orc.fwd(**q, bc_per_channel=True)
    assert np.array_equal(y_b, y_s) and np.array_equal(s_b, s_s), "broadcast rows differ"
    q["B"] = rng.standard_normal((b, d, n, L)).astype(np.float32)
    q["C"] = rng.standard_normal((b, d, n, L)).astype(np.float32)
    y_pc, s_pc = orc.fwd(**q, bc_per_channel=True)
    for bi in range(b):
        for di in range(d):
            one = {k: (None if v is None else v) for k, v in q.items()}
            one["u"] = q["u"][bi:bi + 1, di:di + 1].copy()
            one["delta"] = q["delta"][bi:bi + 1, di:di + 1].copy()
            one["z"] = q["z"][bi:bi + 1, di:di + 1].copy()
            one["A"] = q["A"][di:di + 1].copy()
            one["D"] = q["D"][di:di + 1].copy()
            one["delta_bias"] = q["delta_bias"][di:di + 1].copy()
            one["B"] = q["B"][bi, di][None].copy()
            one["C"] = q["C"][bi, di][None].copy()
            y1, s1 = orc.fwd(**one)
            assert np.array_equal(y1[0, 0], y_pc[bi, di]), f"channel ({bi},{di}) y"
            assert np.array_equal(s1[0, 0], s_pc[bi, di]), f"channel ({bi},{di}) state"


# --------------------------------------------------------------------------
# Mamba-2 (one scalar decay per head; the Mamba-2 cuTile news page,
# "Технические детали оптимизации"):  h_t = exp(A dt_t) h_{t-1} + dt_t B_t x_t,
# y_t = C_t . h_t + D x_t, per (batch, head), B and C shared by a group of heads.
def _ssd_problem(rng, b, L, H, P, G, N, *, D=True, bias=True):
    f = np.float32
    return dict(
        x=rng.standard_normal((b, L, H, P)).astype(f),
        dt=(rng.standard_normal((b, L, H)) * 0.5).astype(f),
        A=(-rng.uniform(0.3, 2.0, H)).astype(f),
        B=rng.standard_normal((b, L, G, N)).astype(f),
        C=rng.standard_normal((b, L, G, N)).astype(f),
        D=rng.standard_normal(H).astype(f) if D else None,
        dt_bias=(rng.standard_normal(H) * 0.5 - 1.0).astype(f) if bias else None)


def _ssd_dt(p, softplus):
    x = p["dt"].astype(np.float64)
    if p["dt_bias"] is not None:
        x = x + p["dt_bias"].astype(np.float64)[None, None, :]
    return _softplus(x) if softplus else x


# The quadratic ("dual") form of the same recurrence: with cum_t = sum_{r<=t} A dt_r,
#   y_t = sum_{s<=t} (C_t . B_s) exp(cum_t - cum_s) dt_s x_s + D x_t
#   h_L = sum_s exp(cum_{L-1} - cum_s) dt_s x_s B_s^T
# evaluated by brute force over every (t, s) pair under an explicit causal mask.
def pin_ssd_quadratic_form(orc, seed=24):
    rng = np.random.default_rng(seed)
    cases = [(2, 9, 4, 3, 2, 5, True, True), (1, 6, 3, 2, 1, 4, False, True),
             (1, 1, 2, 2, 2, 3, True, False), (2, 12, 6, 2, 3, 2, True, True)]
    for b, L, H, P, G, N, softplus, with_d in cases:
        p = _ssd_problem(rng, b, L, H, P, G, N, D=with_d)
        dt = _ssd_dt(p, softplus)                                   # [b,L,H]
        cum = np.cumsum(dt * p["A"].astype(np.float64)[None, None, :], axis=1)
        grp = np.arange(H) // (H // G)
        Bh = p["B"].astype(np.float64)[:, :, grp, :]                # [b,L,H,N]
        Ch = p["C"].astype(np.float64)[:, :, grp, :]
        x = p["x"].astype(np.float64)
        cb = np.einsum("bthn,bshn->bhts", Ch, Bh)
        ct = cum.transpose(0, 2, 1)                                 # [b,H,L]
        causal = np.tril(np.ones((L, L), dtype=bool))
        seg = np.where(causal, ct[:, :, :, None] - ct[:, :, None, :], 0.0)
        w = np.where(causal, np.exp(seg), 0.0) * cb * dt.transpose(0, 2, 1)[:, :, None, :]
        y = np.einsum("bhts,bshp->bthp", w, x)
        if with_d:
            y = y + p["D"].astype(np.float64)[None, None, :, None] * x
        wl = np.exp(cum[:, -1:, :] - cum) * dt                      # [b,L,H]
        final = np.einsum("bsh,bshp,bshn->bhpn", wl, x, Bh)
        y_o, f_o = orc.ssd(**p, dt_softplus=softplus)
        _close(y_o, y, rtol=1e-11, atol=1e-12, what="ssd quadratic form y")
        _close(f_o, final, rtol=1e-11, atol=1e-12, what="ssd quadratic form state")


# A head of the Mamba-2 recurrence is the Mamba-1 scan (already pinned above)
# with the head's P channels as the scan's channels, A[d,n] = A_h for every
# state, dt the same for every channel, and B, C the head group's rows.
def pin_ssd_is_mamba1_with_scalar_decay(orc, seed=25):
    rng = np.random.default_rng(seed)
    b, L, H, P, G, N = 2, 11, 4, 3, 2, 5
    for softplus in (True, False):
        p = _ssd_problem(rng, b, L, H, P, G, N)
        y_o, f_o = orc.ssd(**p, dt_softplus=softplus)
        for h in range(H):
            g = h // (H // G)
            q = dict(u=np.ascontiguousarray(p["x"][:, :, h, :].transpose(0, 2, 1)),
                     delta=np.ascontiguousarray(np.broadcast_to(
                         p["dt"][:, None, :, h], (b, P, L))),
                     A=np.full((P, N), p["A"][h], np.float32),
                     B=np.ascontiguousarray(p["B"][:, :, g, :].transpose(0, 2, 1)),
                     C=np.ascontiguousarray(p["C"][:, :, g, :].transpose(0, 2, 1)),
                     D=np.full(P, p["D"][h], np.float32), z=None,
                     delta_bias=np.full(P, p["dt_bias"][h], np.float32))
            y1, s1 = orc.fwd(**q, delta_softplus=softplus)
            _close(y_o[:, :, h, :], y1.transpose(0, 2, 1), rtol=1e-14, atol=1e-15,
                   what=f"ssd head {h} y")
            _close(f_o[:, h], s1, rtol=1e-14, atol=1e-15, what=f"ssd head {h} state")


# The page's chunked evaluation ("jump formula"): the state after a chunk is the
# incoming state decayed over the chunk plus the chunk's own state from zero,
# and each output of the chunk adds C_t . (exp(cum_t) h_in) to its zero-state
# output, cum_t the decay accumulated inside the chunk up to t.
def pin_ssd_jump_formula(orc, seed=26):
    rng = np.random.default_rng(seed)
    b, L, H, P, G, N, L1 = 2, 13, 4, 2, 2, 3, 5
    p = _ssd_problem(rng, b, L, H, P, G, N)
    y_all, f_all = orc.ssd(**p)
    part = lambda sl: {k: (np.ascontiguousarray(v[:, sl]) if k in ("x", "dt", "B", "C") else v)
                       for k, v in p.items()}
    y1, f1 = orc.ssd(**part(slice(0, L1)))
    p2 = part(slice(L1, L))
    y2, f2 = orc.ssd(**p2)
    cum2 = np.cumsum(_ssd_dt(p2, True) * p["A"].astype(np.float64)[None, None, :], axis=1)
    grp = np.arange(H) // (H // G)
    C2 = p2["C"].astype(np.float64)[:, :, grp, :]                     # [b,L2,H,N]
    carry = np.einsum("bthn,bth,bhpn->bthp", C2, np.exp(cum2), f1)
    _close(y_all[:, :L1], y1, rtol=1e-13, atol=1e-14, what="ssd first chunk")
    _close(y_all[:, L1:], y2 + carry, rtol=1e-11, atol=1e-12, what="ssd second chunk y")
    _close(f_all, np.exp(cum2[:, -1])[:, :, None, None] * f1 + f2, rtol=1e-11, atol=1e-12,
           what="ssd state after both chunks")


# A given state h0 before step 0 is the state a preceding segment of the
# sequence left: the second part run from the first part's final state equals
# the tail of one run over the whole sequence.  With x = 0 nothing enters the
# state, which only decays: h_t = exp(cum_t) h0 and y_t = C_t . h_t (closed form).
def pin_ssd_initial_state(orc, seed=28):
    rng = np.random.default_rng(seed)
    b, L, H, P, G, N, L1 = 2, 11, 4, 2, 2, 3, 4
    p = _ssd_problem(rng, b, L, H, P, G, N)
    y_all, f_all = orc.ssd(**p)
    part = lambda sl: {k: (np.ascontiguousarray(v[:, sl]) if k in ("x", "dt", "B", "C") else v)
                       for k, v in p.items()}
    _, f1 = orc.ssd(**part(slice(0, L1)))
    y2, f2 = orc.ssd(**part(slice(L1, L)), initial_state=f1)
    _close(y2, y_all[:, L1:], rtol=1e-12, atol=1e-13, what="ssd continued from a state: y")
    _close(f2, f_all, rtol=1e-12, atol=1e-13, what="ssd continued from a state: final state")

    q = dict(p, x=np.zeros_like(p["x"]))
    h0 = rng.standard_normal((b, H, P, N))
    y0, f0 = orc.ssd(**q, initial_state=h0)
    cum = np.cumsum(_ssd_dt(q, True) * q["A"].astype(np.float64)[None, None, :], axis=1)
    grp = np.arange(H) // (H // G)
    Ch = q["C"].astype(np.float64)[:, :, grp, :]                     # [b,L,H,N]
    y_cf = np.einsum("bthn,bth,bhpn->bthp", Ch, np.exp(cum), h0)
    _close(y0, y_cf, rtol=1e-12, atol=1e-13, what="ssd decay of h0 alone: y")
    _close(f0, np.exp(cum[:, -1])[:, :, None, None] * h0, rtol=1e-12, atol=1e-13,
           what="ssd decay of h0 alone: final state")


ALL_PINS = [
    pin_unrolled_sum,
    pin_zero_A_is_cumsum,
    pin_constant_inputs_geometric,
    pin_combine_associative,
    pin_chunked_prefix,
    pin_single_step,
    pin_task_spec_sketch,
    pin_no_memory,
    pin_zero_B_or_C,
    pin_invariances,
    pin_bf16_widening,
    pin_backward_finite_differences,
    pin_backward_euler_identities,
    pin_per_channel_bc,
    pin_ssd_quadratic_form,
    pin_ssd_is_mamba1_with_scalar_decay,
    pin_ssd_jump_formula,
    pin_ssd_initial_state,
]
