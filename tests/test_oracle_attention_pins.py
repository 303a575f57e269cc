"""Pins of the attention oracle (attn_oracle.c) to things other than itself.

Each ``pin_*`` checks ``oracle.attention`` against one independent source: a
torch float64 composite of softmax(scale q k^T) v (library routines), closed
forms (a zero query averages the values; a single key returns its value), a
hand-worked fixture, invariants of softmax attention (joint permutation of
keys and values, a common shift of every key's score) and the chunking
property the page relies on (the result does not depend on the chunk sizes).
``test_planted_attention_mistake_is_caught`` plants each mistake of the
oracle's mutation list and requires that at least one pin fails.
"""
from __future__ import annotations

import json
import os

import numpy as np
import pytest
import torch

import fpsynth
import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _draw(shape, seed, stream, dtype, sd=1.0):
    n = int(np.prod(shape))
    vals = fpsynth.normal(seed, stream, n) * sd
    a = vals.astype(np.float32)
    return (fpsynth.f32_to_bf16_bits(a) if dtype == "bf16" else a).reshape(shape)


def _wide(a, dtype):
    return torch.from_numpy(fpsynth.as_float64(a, dtype))


CASES = [  # (BH, Tq, Tk, hd, dtype, k_transposed)
    (2, 37, 53, 16, "f32", False),
    (3, 20, 130, 64, "bf16", True),
    (1, 129, 7, 32, "bf16", False),
]


def _case(BH, Tq, Tk, hd, dtype, kt, seed=5):
    q = _draw((BH, Tq, hd), seed, 11, dtype)
    k = _draw((BH, hd, Tk) if kt else (BH, Tk, hd), seed, 12, dtype)
    v = _draw((BH, Tk, hd), seed, 13, dtype)
    return q, k, v


def _torch_ref(q, k, v, dtype, kt, scale=None):
    qt, kk, vt = _wide(q, dtype), _wide(k, dtype), _wide(v, dtype)
    kT = kk if kt else kk.transpose(1, 2)
    hd = qt.shape[-1]
    s = (qt @ kT) * (hd ** -0.5 if scale is None else scale)
    return (torch.softmax(s, dim=-1) @ vt).numpy()


def pin_torch_composite(mutate=0):
    bad = []
    for BH, Tq, Tk, hd, dt, kt in CASES:
        q, k, v = _case(BH, Tq, Tk, hd, dt, kt)
        got = oracle.attention(q, k, v, dtype=dt, k_transposed=kt, q_chunk=16, kv_chunk=24,
                               mutate=mutate)
        ref = _torch_ref(q, k, v, dt, kt)
        if not np.allclose(got, ref, rtol=1e-10, atol=1e-12):
            bad.append(f"torch composite {BH, Tq, Tk, hd, dt, kt}: {np.abs(got - ref).max():.3e}")
    return bad


def pin_chunk_size_invariance(mutate=0):
    bad = []
    q, k, v = _case(2, 33, 47, 16, "f32", True)
    base = oracle.attention(q, k, v, dtype="f32", k_transposed=True, mutate=mutate)
    for qc, kc in ((1, 1), (3, 5), (7, 17), (33, 46), (64, 64)):
        got = oracle.attention(q, k, v, dtype="f32", k_transposed=True, q_chunk=qc, kv_chunk=kc,
                               mutate=mutate)
        if not np.allclose(got, base, rtol=1e-12, atol=1e-13):
            bad.append(f"chunks {qc},{kc}: {np.abs(got - base).max():.3e}")
    return bad


def pin_closed_forms(mutate=0):
    bad = []
    BH, Tk, hd = 2, 9, 8
    _, k, v = _case(BH, 4, Tk, hd, "f32", False)
    vw = fpsynth.as_float64(v, "f32")
    # a zero query scores every key equally: the output is the mean of the values
    q0 = np.zeros((BH, 4, hd), np.float32)
    got = oracle.attention(q0, k, v, dtype="f32", kv_chunk=4, mutate=mutate)
    if not np.allclose(got, np.broadcast_to(vw.mean(axis=1, keepdims=True), got.shape),
                       rtol=1e-13, atol=1e-14):
        bad.append("zero query is not the mean of the values")
    # one key: every query returns its value
    q, k1, v1 = _case(BH, 5, 1, hd, "f32", False)
    got = oracle.attention(q, k1, v1, dtype="f32", mutate=mutate)
    if not np.allclose(got, np.broadcast_to(fpsynth.as_float64(v1, "f32"), got.shape),
                       rtol=1e-14, atol=1e-15):
        bad.append("a single key does not return its value")
    # hand-worked fixture
    d = json.load(open(os.path.join(GOLDEN, "attn_hand.json")))
    qh = np.array(d["q"], np.float32)
    kh = np.array([[[0.0], [np.log(4.0)]]], np.float32)
    vh = np.array(d["v"], np.float32)
    got = oracle.attention(qh, kh, vh, dtype="f32", scale=d["scale"], kv_chunk=1, mutate=mutate)
    if not np.allclose(got, np.array(d["expect"]), rtol=0, atol=1e-6):
        bad.append(f"hand fixture: {got.ravel()} vs {np.array(d['expect']).ravel()}")
    return bad


def pin_invariants(mutate=0):
    bad = []
    q, k, v = _case(2, 11, 19, 16, "f32", False)
    base = oracle.attention(q, k, v, dtype="f32", kv_chunk=6, mutate=mutate)
    # keys and values permuted together
    perm = np.random.default_rng(3).permutation(19)
    got = oracle.attention(q, np.ascontiguousarray(k[:, perm]), np.ascontiguousarray(v[:, perm]),
                           dtype="f32", kv_chunk=6, mutate=mutate)
    if not np.allclose(got, base, rtol=1e-12, atol=1e-13):
        bad.append("joint key/value permutation changed the output")
    # a vector u added to every key shifts all scores of a query row by q.u
    u = np.array([0.5] * 8 + [-0.25] * 8, np.float32)
    got = oracle.attention(q, (k + u).astype(np.float32), v, dtype="f32", kv_chunk=6,
                           mutate=mutate)
    ref = _torch_ref(q, (k + u).astype(np.float32), v, "f32", False)
    if not np.allclose(got, ref, rtol=1e-10, atol=1e-12) or \
            not np.allclose(got, _torch_ref(q, k, v, "f32", False), rtol=1e-4, atol=1e-5):
        bad.append("a common shift of each row's scores changed the output")
    return bad


PINS = [pin_torch_composite, pin_chunk_size_invariance, pin_closed_forms, pin_invariants]


@pytest.mark.parametrize("pin", PINS, ids=lambda f: f.__name__)
def test_attention_pins_hold(pin):
    assert pin() == []


@pytest.mark.parametrize("name", sorted(oracle.ATTN_MUTATIONS))
def test_planted_attention_mistake_is_caught(name):
    code = oracle.ATTN_MUTATIONS[name]
    caught = [p.__name__ for p in PINS if p(mutate=code)]
    assert caught, f"no pin caught the planted mistake {name}"
