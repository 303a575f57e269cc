"""Pins of the CPU oracle to things other than itself (no GPU needed).

Each ``pin_*`` function checks the oracle against one independent source —
a library routine (torch float64 composite), a closed form evaluated in
mpmath, a hand-worked fixture under ``tests/golden/``, or an invariant that
the pages' operation must satisfy — and returns a list of failure strings.
``test_pins_hold`` runs them on the real oracle; ``test_planted_mistake_is_caught``
plants each mistake of the oracle's mutation list and requires that at least
one pin fails.
"""
from __future__ import annotations

import json
import math
import os

import numpy as np
import pytest

import fpsynth
import oracle
from tests.composite import composite

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _load(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _close(a, b, rtol=1e-12, atol=1e-12):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    if a.shape != b.shape:
        return False
    return bool(np.all(np.abs(a - b) <= atol + rtol * np.abs(b)))


# Small versions of every workload family: same axes/roles, a few tiles of tokens.
SMALL = {
    "tiny_fp32": fpsynth.WORKLOADS["tiny_fp32"],
    "walrus_small": fpsynth.WORKLOADS["walrus_bf16"].scaled(
        name="walrus_small", x_shape=(2, 3, 32, 4, 4, 1), C=32, F=64, heads=2, head_dim=16),
    "bert_ff_small": fpsynth.WORKLOADS["bert_ff_bf16"].scaled(
        name="bert_ff_small", x_shape=(2, 5, 24), C=24, F=40),
    "bert_qkv_small": fpsynth.WORKLOADS["bert_qkv_bf16"].scaled(
        name="bert_qkv_small", x_shape=(3, 7, 24), C=24, heads=3, head_dim=8),
    "llm_rope_small": fpsynth.WORKLOADS["llm_qkv_rope_bf16"].scaled(
        name="llm_rope_small", x_shape=(2, 9, 32), C=32, heads=2, head_dim=16),
    "unet_small": fpsynth.WORKLOADS["unet_qkv_bf16"].scaled(
        name="unet_small", x_shape=(2, 16, 3, 5), C=16, heads=2, head_dim=8),
    "silu_rope_f32": fpsynth.Workload("silu_rope_f32", (3, 12, 2, 2), 1, 1, 12, 20, 2, 6,
                                      fpsynth.ACT_SILU, 500.0, True, "f32", 11),
    "gqa_partial_rope": fpsynth.Workload("gqa_partial_rope", (2, 6, 32), 2, 1, 32, 0, 4, 8,
                                         fpsynth.ACT_NONE, 10000.0, False, "bf16", 12,
                                         rope_n_elem=4, n_query_groups=2),
    "relu2_f32": fpsynth.Workload("relu2_f32", (2, 7, 16), 2, 1, 16, 24, 2, 8,
                                  fpsynth.ACT_RELU2, 0.0, True, "f32", 13),
    "k_transposed": fpsynth.Workload("k_transposed", (2, 5, 24), 2, 1, 24, 0, 3, 8,
                                     fpsynth.ACT_NONE, 10000.0, True, "f32", 14,
                                     k_transposed=True),
}


def _oracle(w, inp, mutate=0, **kw):
    return oracle.forward_workload(w, inp, mutate=mutate, threads=2, **kw)


def _composite(w, inp):
    return composite(fpsynth.as_float64(inp["x"], w.dtype), fpsynth.as_float64(inp["W"], w.dtype),
                     fpsynth.as_float64(inp["b"], w.dtype), channel_dim=w.channel_dim,
                     n_batch_dims=w.n_batch_dims, C=w.C, F=w.F, heads=w.heads,
                     head_dim=w.head_dim, act=w.act, rope_base=w.rope_base, pos=inp.get("pos"),
                     groups=w.n_query_groups, rope_n_elem=w.rope_n_elem,
                     k_transposed=w.k_transposed, rope_cos=inp.get("rope_cos"),
                     rope_sin=inp.get("rope_sin"))


# ---------------------------------------------------------------- pins

def pin_composite(mutate=0):
    """Library cross-check: torch float64 permute/addmm/gelu/complex-rotation/transpose."""
    bad = []
    for name, w in SMALL.items():
        inp = fpsynth.make_inputs(w)
        if w.rope_base > 0:
            # explicit, non-trivial positions shared by all batch elements
            inp["pos"] = (np.arange(w.T, dtype=np.int32) * 3 + 5) % 97
        got = _oracle(w, inp, mutate)
        ref = _composite(w, inp)
        for k in ("ff", "q", "k", "v"):
            if not _close(got[k], ref[k], rtol=1e-11, atol=1e-11):
                bad.append(f"composite:{name}:{k}")
        if w.rope_base > 0:
            got = _oracle(w, {**inp, "pos": None}, mutate)
            ref = _composite(w, {**inp, "pos": None})
            for k in ("q", "k"):
                if not _close(got[k], ref[k], rtol=1e-11, atol=1e-11):
                    bad.append(f"composite-defaultpos:{name}:{k}")
    return bad


def pin_hand_linear(mutate=0):
    g = _load("hand_linear.json")
    bad = []
    xt = np.array(g["x_tokens_by_channels"], dtype=np.float32)  # [T, C]
    W = np.array(g["W"], dtype=np.float32)
    b = np.array(g["b"], dtype=np.float32)
    for dtype in ("f32", "bf16"):
        conv = (lambda a: fpsynth.f32_to_bf16_bits(a)) if dtype == "bf16" else (lambda a: a)
        for layout in ("row_major", "channels_first"):
            if layout == "row_major":
                x, cd = xt[None], 2  # [1, T, C]
            else:
                x, cd = np.ascontiguousarray(xt.T)[None], 1  # [1, C, T]
            out = oracle.forward(conv(x), conv(W), conv(b), channel_dim=cd, n_batch_dims=1,
                                 C=g["C"], F=g["F"], heads=g["heads"], head_dim=g["head_dim"],
                                 act=g["act"], rope_base=g["rope_base"], dtype=dtype,
                                 mutate=mutate, threads=1)
            for k in ("ff", "q", "k", "v"):
                if not _close(out[k], g["expect"][k], rtol=0, atol=0):
                    bad.append(f"hand_linear:{dtype}:{layout}:{k}")
    return bad


def pin_hand_scatter(mutate=0):
    g = _load("hand_scatter.json")
    x = np.array(g["x_btc"], dtype=np.float32)
    C = g["C"]
    W = np.concatenate([np.eye(C, dtype=np.float32)] * 3, axis=1)
    out = oracle.forward(x, W, None, channel_dim=2, n_batch_dims=1, C=C, F=0, heads=g["heads"],
                         head_dim=g["head_dim"], act=0, rope_base=0.0, dtype="f32",
                         mutate=mutate, threads=1)
    bad = []
    for k in ("q", "k", "v"):
        if not _close(out[k], g["expect_q"], rtol=0, atol=0):
            bad.append(f"hand_scatter:{k}")
    return bad


def pin_quarter_turn(mutate=0):
    mp = pytest.importorskip("mpmath")
    g = _load("rope_quarter_turn.json")
    x = np.array(g["x_tokens"], dtype=np.float32)[None]  # [1, T, 4]
    hd = g["head_dim"]
    W = np.concatenate([np.eye(hd, dtype=np.float32)] * 3, axis=1)
    base = 4.0 / math.pi ** 2
    pos = np.array(g["pos"], dtype=np.int32)
    out = oracle.forward(x, W, None, channel_dim=2, n_batch_dims=1, C=hd, F=0, heads=1,
                         head_dim=hd, act=0, rope_base=base, dtype="f32", pos=pos,
                         mutate=mutate, threads=1)
    bad = []
    for k in ("q", "k"):
        o = out[k][0]
        if not _close(o[:, 1], g["expect_lane1"], atol=1e-12):
            bad.append(f"quarter:{k}:lane1")
        if not _close(o[:, 3], g["expect_lane3"], atol=1e-12):
            bad.append(f"quarter:{k}:lane3")
        for t, p in enumerate(g["pos"]):
            a, c = float(x[0, t, 0]), float(x[0, t, 2])
            e0 = float(a * mp.cos(p) - c * mp.sin(p))
            e2 = float(c * mp.cos(p) + a * mp.sin(p))
            if not (_close(o[t, 0], e0, atol=1e-12) and _close(o[t, 2], e2, atol=1e-12)):
                bad.append(f"quarter:{k}:lanes02:t{t}")
    if not _close(out["v"][0], x[0], rtol=0, atol=0):
        bad.append("quarter:v-rotated")
    return bad


def _single_column(values, act, dtype="f32", mutate=0):
    """ff = act(x * 1): C = 1, F = 1, a [1, M, 1] input."""
    x = np.array(values, dtype=np.float32).reshape(1, -1, 1)
    W = np.ones((1, 1), dtype=np.float32)
    out = oracle.forward(x, W, None, channel_dim=2, n_batch_dims=1, C=1, F=1, heads=0,
                         head_dim=0, act=act, rope_base=0.0, dtype=dtype, mutate=mutate,
                         threads=1)
    return out["ff"][:, 0]


PTS = [-6.0, -3.5, -1.25, -0.5, -0.125, 0.0, 0.0625, 0.375, 1.0, 2.5, 4.0, 9.0]


def pin_activation_closed_forms(mutate=0):
    """GELU (erf, tanh) and SiLU against mpmath at 50 digits, plus identities."""
    mp = pytest.importorskip("mpmath")
    mp.mp.dps = 50
    bad = []
    ys = [mp.mpf(v) for v in PTS]
    erf_ref = [float(y / 2 * (1 + mp.erf(y / mp.sqrt(2)))) for y in ys]
    tanh_ref = [float(y / 2 * (1 + mp.tanh(mp.sqrt(2 / mp.pi) * (y + mp.mpf("0.044715") * y ** 3))))
                for y in ys]
    silu_ref = [float(y / (1 + mp.exp(-y))) for y in ys]
    relu2_ref = [float(max(y, 0) ** 2) for y in ys]
    for act, ref, nm in ((1, erf_ref, "gelu"), (2, tanh_ref, "gelu_tanh"), (3, silu_ref, "silu"),
                         (4, relu2_ref, "relu2")):
        got = _single_column(PTS, act, mutate=mutate)
        # absolute floor: 1 + erf(y/sqrt 2) cancels for y << 0 (error ~ulp(1)*|y|)
        if not _close(got, ref, rtol=1e-14, atol=1e-15):
            bad.append(f"closed_form:{nm}")
    # GELU(y) - GELU(-y) = y for the exact (erf) form: Phi(y) + Phi(-y) = 1
    g_pos = _single_column(PTS, 1, mutate=mutate)
    g_neg = _single_column([-v for v in PTS], 1, mutate=mutate)
    if not _close(g_pos - g_neg, PTS, atol=1e-14):
        bad.append("gelu_odd_identity")
    return bad


def pin_linear_is_unsplit_gemm(mutate=0):
    """Invariant 1: with no activation and no rotation, the split outputs, put
    back side by side per token, equal one GEMM x W + b (numpy matmul on the
    permuted activation)."""
    bad = []
    for name in ("walrus_small", "bert_qkv_small", "unet_small"):
        w = SMALL[name].scaled(act=0, rope_base=0.0)
        inp = fpsynth.make_inputs(w)
        x = fpsynth.as_float64(inp["x"], w.dtype)
        perm = [a for a in range(x.ndim) if a != w.channel_dim] + [w.channel_dim]
        X = np.transpose(x, perm).reshape(w.M, w.C)
        Y = X @ fpsynth.as_float64(inp["W"], w.dtype)
        if inp["b"] is not None:
            Y = Y + fpsynth.as_float64(inp["b"], w.dtype)
        rows = list(range(w.M))
        out = _oracle(w, inp, mutate, rows=rows)
        cat = np.concatenate([out["ff"], out["q"], out["k"], out["v"]], axis=1)
        if not _close(cat, Y, rtol=1e-12, atol=1e-12):
            bad.append(f"unsplit:{name}")
    return bad


def _rope_case():
    w = SMALL["llm_rope_small"]
    return w, fpsynth.make_inputs(w)


def pin_rope_position_zero_identity(mutate=0):
    """Invariant 2: at position 0 the rotation is the identity."""
    w, inp = _rope_case()
    on = _oracle(w, {**inp, "pos": np.zeros(w.T, np.int32)}, mutate)
    off = _oracle(w.scaled(rope_base=0.0), inp, mutate)
    return [] if all(_close(on[k], off[k], rtol=1e-15, atol=0) for k in "qkv") else ["pos0"]


def pin_rope_pair_norm(mutate=0):
    """Invariant 3: each rotated pair (i, i + hd/2) keeps its Euclidean norm."""
    w, inp = _rope_case()
    on = _oracle(w, inp, mutate)
    off = _oracle(w.scaled(rope_base=0.0), inp, mutate)
    h = w.head_dim // 2
    bad = []
    for k in ("q", "k", "v"):
        n_on = on[k][..., :h] ** 2 + on[k][..., h:] ** 2
        n_off = off[k][..., :h] ** 2 + off[k][..., h:] ** 2
        if not _close(n_on, n_off, rtol=1e-12, atol=1e-12):
            bad.append(f"pairnorm:{k}")
        if k == "v" and not _close(on[k], off[k], rtol=0, atol=0):
            bad.append("v-rotated")
    # the rotation must actually move something at p > 0
    if _close(on["q"], off["q"], rtol=1e-9, atol=1e-9):
        bad.append("rope-noop")
    return bad


def pin_rope_relative_position(mutate=0):
    """Invariant 4: q(t1) . k(t2) after rotation depends only on pos[t1] - pos[t2]."""
    w, inp = _rope_case()
    pos = np.array([(7 * t) % 23 for t in range(w.T)], dtype=np.int32)
    a = _oracle(w, {**inp, "pos": pos}, mutate)
    b = _oracle(w, {**inp, "pos": pos + 1000}, mutate)
    bad = []
    for o in (a, b):
        o["dots"] = np.einsum("htd,hsd->hts", o["q"], o["k"])
    if not _close(a["dots"], b["dots"], rtol=1e-9, atol=1e-9):
        bad.append("relpos")
    # and the shift does change the vectors themselves (not a trivial pass)
    if _close(a["q"], b["q"], rtol=1e-6, atol=1e-6):
        bad.append("relpos-trivial")
    return bad


def pin_rows_match_full(mutate=0):
    """The sampled-rows mode reports the same values as the full scatter."""
    bad = []
    for name in ("walrus_small", "gqa_partial_rope"):
        w = SMALL[name]
        inp = fpsynth.make_inputs(w)
        full = _oracle(w, inp, mutate)
        rows = [0, w.M - 1, w.T, 5 % w.M]
        part = _oracle(w, inp, mutate, rows=rows)
        nkv = w.n_query_groups or w.heads
        for r, m in enumerate(rows):
            bb, t = divmod(m, w.T)
            if w.F and not _close(part["ff"][r], full["ff"][m], rtol=0, atol=0):
                bad.append(f"rows:{name}:ff")
            for hh in range(w.heads):
                if not _close(part["q"][r, hh * w.head_dim:(hh + 1) * w.head_dim],
                              full["q"][bb * w.heads + hh, t], rtol=0, atol=0):
                    bad.append(f"rows:{name}:q")
            for g in range(nkv):
                for k in ("k", "v"):
                    if not _close(part[k][r, g * w.head_dim:(g + 1) * w.head_dim],
                                  full[k][bb * nkv + g, t], rtol=0, atol=0):
                        bad.append(f"rows:{name}:{k}")
    return bad


def pin_strided_view(mutate=0):
    """A channels-first logical view of a channels-last buffer (non-contiguous
    strides) gives the same result as the contiguous copy."""
    w = SMALL["unet_small"]
    inp = fpsynth.make_inputs(w)
    x = inp["x"]  # [B, C, H, W] contiguous
    buf = np.ascontiguousarray(np.transpose(x, (0, 2, 3, 1)))  # [B, H, W, C]
    B, C, H, Wd = x.shape
    strides = (H * Wd * C, 1, Wd * C, C)
    a = _oracle(w, inp, mutate)
    b = oracle.forward(x, inp["W"], inp["b"], channel_dim=1, n_batch_dims=1, C=w.C, F=w.F,
                       heads=w.heads, head_dim=w.head_dim, act=w.act, rope_base=w.rope_base,
                       dtype=w.dtype, x_base=buf, x_strides=strides, mutate=mutate, threads=2)
    return [] if all(_close(a[k], b[k], rtol=0, atol=0) for k in "qkv") else ["strided"]


def _table_case(seed=3):
    w = SMALL["gqa_partial_rope"].scaled(name="table_case", rope_n_elem=6)
    inp = fpsynth.make_inputs(w)
    rng = np.random.default_rng(seed)
    n = w.rope_n_elem
    inp["rope_cos"] = rng.standard_normal((w.T, n))
    inp["rope_sin"] = rng.standard_normal((w.T, n))
    return w, inp


def pin_rope_table_forms(mutate=0):
    """Caller cos/sin tables (the rope_one_entry listing's inputs, random as in
    its test): the torch elementwise form, two exact special tables, linearity
    in (cos, sin), and agreement with the computed angles when the table holds
    them."""
    bad = []
    w, inp = _table_case()
    got = _oracle(w, inp, mutate)
    ref = _composite(w, inp)
    for k in ("q", "k", "v"):
        if not _close(got[k], ref[k], rtol=1e-12, atol=1e-12):
            bad.append(f"table-composite:{k}")
    n, h = w.rope_n_elem, w.rope_n_elem // 2
    plain = _oracle(w.scaled(rope_base=0.0), {**inp, "rope_cos": None, "rope_sin": None}, mutate)
    # cos = 1, sin = 0: identity; cos = 0, sin = 1: the rotated vector cat(-x2, x1), exactly
    ident = _oracle(w, {**inp, "rope_cos": np.ones((w.T, n)), "rope_sin": np.zeros((w.T, n))},
                    mutate)
    quarter = _oracle(w, {**inp, "rope_cos": np.zeros((w.T, n)), "rope_sin": np.ones((w.T, n))},
                      mutate)
    for k in ("q", "k"):
        if not _close(ident[k], plain[k], rtol=0, atol=0):
            bad.append(f"table-identity:{k}")
        want = plain[k].copy()
        want[..., :h] = -plain[k][..., h:n]
        want[..., h:n] = plain[k][..., :h]
        if not _close(quarter[k], want, rtol=0, atol=0):
            bad.append(f"table-quarter:{k}")
    # linearity: the rotated lanes are linear in (cos, sin) jointly
    rng = np.random.default_rng(9)
    c2, s2 = rng.standard_normal((w.T, n)), rng.standard_normal((w.T, n))
    o2 = _oracle(w, {**inp, "rope_cos": c2, "rope_sin": s2}, mutate)
    o12 = _oracle(w, {**inp, "rope_cos": inp["rope_cos"] + c2, "rope_sin": inp["rope_sin"] + s2},
                  mutate)
    for k in ("q", "k"):
        if not _close(o12[k][..., :n], got[k][..., :n] + o2[k][..., :n], rtol=1e-12, atol=1e-12):
            bad.append(f"table-linear:{k}")
    # a table holding cos/sin of the default angles reproduces the computed path
    wf = w.scaled(rope_n_elem=0)
    nf = wf.head_dim
    ang = np.arange(wf.T)[:, None] * wf.rope_base ** (-2.0 * np.arange(nf // 2) / nf)[None, :]
    ang = np.concatenate([ang, ang], axis=1)
    tab = _oracle(wf, {**inp, "rope_cos": np.cos(ang), "rope_sin": np.sin(ang)}, mutate)
    comp = _oracle(wf, {**inp, "rope_cos": None, "rope_sin": None}, mutate)
    for k in ("q", "k"):
        if not _close(tab[k], comp[k], rtol=1e-12, atol=1e-12):
            bad.append(f"table-vs-angles:{k}")
    return bad


PINS = [pin_composite, pin_hand_linear, pin_hand_scatter, pin_quarter_turn,
        pin_activation_closed_forms, pin_linear_is_unsplit_gemm, pin_rope_position_zero_identity,
        pin_rope_pair_norm, pin_rope_relative_position, pin_rows_match_full, pin_strided_view,
        pin_rope_table_forms]


@pytest.mark.parametrize("pin", PINS, ids=lambda p: p.__name__)
def test_pins_hold(pin):
    assert pin(0) == []


@pytest.mark.parametrize("mutation", sorted(oracle.MUTATIONS), ids=str)
def test_planted_mistake_is_caught(mutation):
    mid = oracle.MUTATIONS[mutation]
    caught = {}
    for pin in PINS:
        bad = pin(mid)
        if bad:
            caught[pin.__name__] = bad
    assert caught, f"planted mistake '{mutation}' passed every pin"


def test_rejects_bad_arguments():
    x = np.zeros((1, 4, 8), np.float32)
    W = np.zeros((8, 24), np.float32)
    with pytest.raises(ValueError):
        oracle.forward(x, W, None, channel_dim=2, n_batch_dims=1, C=7, F=0, heads=2, head_dim=4,
                       act=0, rope_base=0.0, dtype="f32")
    with pytest.raises(ValueError):  # odd head size
        oracle.forward(x, W, None, channel_dim=2, n_batch_dims=1, C=8, F=0, heads=8, head_dim=1,
                       act=0, rope_base=0.0, dtype="f32")
