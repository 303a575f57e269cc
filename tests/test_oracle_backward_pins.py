"""Pins of the oracle's backward (gradients with respect to x, W and b).

Each pin compares the oracle with something other than itself:

* ``torch.autograd`` through the independent float64 composite
  (``tests/composite.py``: permute/addmm/gelu/complex rotation/transpose);
* central finite differences of the oracle's own forward, which is pinned
  separately (``test_oracle_pins.py``);
* the activation derivatives against mpmath at 50 digits (numerical
  differentiation of the closed forms);
* invariants: the gradient rotation preserves each pair's norm, and the
  sampled-row / sampled-column modes equal the full evaluation.

``test_planted_backward_mistake_is_caught`` plants each backward mistake of
``oracle.BWD_MUTATIONS`` and checks that some pin fails.
"""
from __future__ import annotations

import numpy as np
import pytest

import fpsynth
import oracle
from tests.composite import composite_backward
from tests.test_oracle_pins import SMALL, _close

A = fpsynth
W_ = fpsynth.Workload

# every feature of the forward, on shapes the composite differentiates quickly
BWD_CASES = {
    "tiny_fp32": SMALL["tiny_fp32"],
    "walrus_small": SMALL["walrus_small"],
    "bert_ff_small": SMALL["bert_ff_small"],
    "llm_rope_small": SMALL["llm_rope_small"],
    "silu_rope_f32": SMALL["silu_rope_f32"],
    "gqa_partial_rope": SMALL["gqa_partial_rope"],
    "relu2_f32": SMALL["relu2_f32"],
    "k_transposed": SMALL["k_transposed"],
    "gelu_tanh_f32": W_("gelu_tanh_f32", (2, 6, 16), 2, 1, 16, 32, 2, 8, A.ACT_GELU_TANH,
                        10000.0, True, "f32", 15),
    "gqa_full_rope_kt": W_("gqa_full_rope_kt", (2, 5, 32), 2, 1, 32, 16, 4, 8, A.ACT_GELU_ERF,
                           1000.0, True, "f32", 16, n_query_groups=2, k_transposed=True),
}


def _kw(w, inp):
    return dict(channel_dim=w.channel_dim, n_batch_dims=w.n_batch_dims, C=w.C, F=w.F,
                heads=w.heads, head_dim=w.head_dim, act=w.act, rope_base=w.rope_base,
                pos=inp.get("pos"), groups=w.n_query_groups, rope_n_elem=w.rope_n_elem,
                k_transposed=w.k_transposed, rope_cos=inp.get("rope_cos"),
                rope_sin=inp.get("rope_sin"))


def _autograd(w, inp, grads):
    g64 = {k: fpsynth.as_float64(v, w.dtype) for k, v in grads.items()}
    return composite_backward(fpsynth.as_float64(inp["x"], w.dtype),
                              fpsynth.as_float64(inp["W"], w.dtype),
                              fpsynth.as_float64(inp["b"], w.dtype), g64, **_kw(w, inp))


def _obwd(w, inp, grads, mutate=0, **kw):
    return oracle.backward_workload(w, inp, grads, mutate=mutate, threads=2, **kw)


# ---------------------------------------------------------------- pins

def pin_autograd(mutate=0):
    """Library cross-check: torch.autograd of sum(g * composite(x, W, b))."""
    bad = []
    for name, w in BWD_CASES.items():
        inp = fpsynth.make_inputs(w)
        if w.rope_base > 0:
            inp["pos"] = (np.arange(w.T, dtype=np.int32) * 5 + 3) % 89
        grads = fpsynth.make_grads(w)
        got = _obwd(w, inp, grads, mutate)
        ref = _autograd(w, inp, grads)
        for k in ("dx", "dW"):
            if not _close(got[k], ref[k], rtol=1e-10, atol=1e-10):
                bad.append(f"autograd:{name}:{k}")
        if w.bias and not _close(got["db"], ref["db"], rtol=1e-10, atol=1e-10):
            bad.append(f"autograd:{name}:db")
    # caller cos/sin tables (random, as in the rope_one_entry listing's test)
    w = SMALL["gqa_partial_rope"].scaled(name="table_bwd", rope_n_elem=6)
    inp = fpsynth.make_inputs(w)
    rng = np.random.default_rng(4)
    inp["rope_cos"] = rng.standard_normal((w.T, 6))
    inp["rope_sin"] = rng.standard_normal((w.T, 6))
    grads = fpsynth.make_grads(w)
    got = _obwd(w, inp, grads, mutate)
    ref = _autograd(w, inp, grads)
    for k in ("dx", "dW"):
        if not _close(got[k], ref[k], rtol=1e-10, atol=1e-10):
            bad.append(f"autograd:tables:{k}")
    return bad


def pin_finite_differences(mutate=0):
    """Brute force: central differences of sum(g * forward) on a tiny f32 case
    with every block (GELU ff, rotated q/k, v), for entries of x, W and b."""
    w = W_("fd_case", (1, 3, 8), 2, 1, 8, 8, 2, 4, A.ACT_GELU_ERF, 10000.0, True, "f32", 17)
    inp = fpsynth.make_inputs(w)
    grads = fpsynth.make_grads(w)
    g64 = {k: fpsynth.as_float64(v, "f32") for k, v in grads.items()}
    got = _obwd(w, inp, grads, mutate)

    def loss(x, W, b):
        out = oracle.forward(x, W, b, channel_dim=2, n_batch_dims=1, C=w.C, F=w.F,
                             heads=w.heads, head_dim=w.head_dim, act=w.act,
                             rope_base=w.rope_base, dtype="f32", threads=1)
        return sum(float((out[k] * g64[k]).sum()) for k in ("ff", "q", "k", "v"))

    bad = []
    h = np.float32(2.0 ** -7)
    probes = [("x", (0, 1, 3)), ("x", (0, 2, 0)), ("W", (2, 5)), ("W", (7, 10)), ("W", (4, 21)),
              ("b", (3,)), ("b", (13,)), ("b", (22,))]
    for name, idx in probes:
        arrs = {"x": inp["x"].copy(), "W": inp["W"].copy(), "b": inp["b"].copy()}
        a0 = arrs[name][idx]
        arrs[name][idx] = a0 + h
        up = loss(arrs["x"], arrs["W"], arrs["b"])
        arrs[name][idx] = a0 - h
        dn = loss(arrs["x"], arrs["W"], arrs["b"])
        fd = (up - dn) / (2.0 * float(h))
        if name == "x":
            an = got["dx"][idx[1], idx[2]]
        elif name == "W":
            an = got["dW"][idx]
        else:
            an = got["db"][idx]
        if abs(fd - an) > 1e-4 * max(1.0, abs(an)):
            bad.append(f"fd:{name}{idx}: fd {fd:.6g} analytic {an:.6g}")
    return bad


def _single_column_grad(values, act, mutate=0):
    """C = 1, F = 1, x = 1, W = y, g = 1: db = act'(y), one token per value."""
    n = len(values)
    x = np.ones((1, n, 1), dtype=np.float32)
    W = np.ones((1, 1), dtype=np.float32)
    b = None
    out = []
    for v in values:
        W[0, 0] = np.float32(v)
        r = oracle.backward(x[:, :1], W, b, {"ff": np.ones((1, 1), np.float32)}, channel_dim=2,
                            n_batch_dims=1, C=1, F=1, heads=0, head_dim=0, act=act,
                            rope_base=0.0, dtype="f32", threads=1, mutate=mutate)
        out.append(r["db"][0])
    return np.array(out)


def pin_activation_derivatives(mutate=0):
    """act'(y) against mpmath's numerical derivative of the closed forms (50 digits)."""
    mp = pytest.importorskip("mpmath")
    mp.mp.dps = 50
    pts = [-6.0, -2.5, -1.0, -0.25, 0.0, 0.125, 0.75, 1.5, 3.0, 7.0]
    forms = {
        1: lambda y: y / 2 * (1 + mp.erf(y / mp.sqrt(2))),
        2: lambda y: y / 2 * (1 + mp.tanh(mp.sqrt(2 / mp.pi) * (y + mp.mpf("0.044715") * y ** 3))),
        3: lambda y: y / (1 + mp.exp(-y)),
        4: lambda y: max(y, 0) ** 2,
    }
    bad = []
    for act, f in forms.items():
        ref = [float(mp.diff(f, mp.mpf(v))) if not (act == 4 and v == 0.0) else 0.0 for v in pts]
        got = _single_column_grad(pts, act, mutate)
        if not _close(got, ref, rtol=1e-13, atol=1e-14):
            bad.append(f"act_deriv:{act}")
    return bad


def pin_rotation_transpose_norm(mutate=0):
    """Invariant: with the computed (cos, sin) the gradient rotation is
    orthogonal, so each rotated pair keeps the norm of its upstream gradient
    (act none, no bias, one token: G's q/k entries are the rotated gradient)."""
    w = W_("rot_norm", (1, 4, 16), 2, 1, 16, 0, 2, 8, A.ACT_NONE, 10000.0, False, "f32", 18)
    inp = fpsynth.make_inputs(w)
    grads = fpsynth.make_grads(w)
    cols = list(range(w.N))
    bad = []
    # db over one token is that token's G row; use a one-token view per position
    for t in range(w.T):
        wt = w.scaled(name="rot_norm_t", x_shape=(1, 1, 16))
        it = {"x": inp["x"][:, t:t + 1].copy(), "W": inp["W"], "b": None,
              "pos": np.array([t * 37 + 1], dtype=np.int32)}
        gt = {"ff": None, "q": grads["q"][:, t:t + 1].copy(), "k": grads["k"][:, t:t + 1].copy(),
              "v": grads["v"][:, t:t + 1].copy()}
        G = _obwd(wt, it, gt, mutate, cols=cols)["db"]
        for blk, g in (("q", gt["q"]), ("k", gt["k"])):
            off = 0 if blk == "q" else w.C
            for hh in range(w.heads):
                u = G[off + hh * 8: off + hh * 8 + 8]
                gg = g[hh, 0].astype(np.float64)
                for i in range(4):
                    if abs(np.hypot(u[i], u[i + 4]) - np.hypot(gg[i], gg[i + 4])) > 1e-12:
                        bad.append(f"rot_norm:{blk}:h{hh}:t{t}:i{i}")
        if not _close(G[2 * w.C:], gt["v"][:, 0].reshape(-1).astype(np.float64), rtol=0, atol=0):
            bad.append(f"rot_norm:v:t{t}")
    return bad


def pin_sampled_match_full(mutate=0):
    """Consistency: dx of sampled rows and dW/db of sampled columns equal the full evaluation."""
    bad = []
    for name in ("walrus_small", "gqa_partial_rope", "k_transposed"):
        w = BWD_CASES[name]
        inp = fpsynth.make_inputs(w)
        grads = fpsynth.make_grads(w)
        full = _obwd(w, inp, grads, mutate)
        rows = [0, w.M // 2, w.M - 1]
        cols = [0, w.N // 3, w.N - 1]
        r = _obwd(w, inp, grads, mutate, rows=rows)
        c = _obwd(w, inp, grads, mutate, cols=cols)
        if not _close(r["dx"], full["dx"][rows], rtol=1e-13, atol=1e-13):
            bad.append(f"rows:{name}")
        if not _close(c["dW"], full["dW"][:, cols], rtol=1e-12, atol=1e-12):
            bad.append(f"cols:{name}:dW")
        if not _close(c["db"], full["db"][cols], rtol=1e-12, atol=1e-12):
            bad.append(f"cols:{name}:db")
    return bad


PINS = [pin_autograd, pin_finite_differences, pin_activation_derivatives,
        pin_rotation_transpose_norm, pin_sampled_match_full]


@pytest.mark.parametrize("pin", PINS, ids=lambda p: p.__name__)
def test_backward_pins_hold(pin):
    assert pin(0) == []


@pytest.mark.parametrize("mutation", sorted(oracle.BWD_MUTATIONS), ids=str)
def test_planted_backward_mistake_is_caught(mutation):
    mid = oracle.BWD_MUTATIONS[mutation]
    caught = {p.__name__: b for p in PINS if (b := p(mid))}
    assert caught, f"planted mistake '{mutation}' passed every pin"


def test_backward_rejects_bad_samples():
    w = BWD_CASES["walrus_small"]
    inp = fpsynth.make_inputs(w)
    grads = fpsynth.make_grads(w)
    with pytest.raises(ValueError):
        _obwd(w, inp, grads, cols=[w.N])
    with pytest.raises(ValueError):
        _obwd(w, inp, grads, rows=[w.M])
    with pytest.raises(ValueError):
        _obwd(w, inp, {**grads, "q": None})
