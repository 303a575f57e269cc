"""fp_forward_noalloc against fp_forward, through the C ABI (needs a GB300).

fp_forward_noalloc is for callers that may not allocate device memory, such as
a plug-in inside a framework that owns every device byte through its own pool,
or a serving process with a fixed memory budget set at start-up. It keeps the
kernels' scratch (status words, rotary table) in a static device array. Here
its outputs must match the plan-based entry point on two calls in a row; the
second call has other positions and another sequence length, so a table left
over from the first call would show up as a mismatch.

This file sorts last so a run that stops at the first failure has already run
every other test; it also passes on its own in a fresh process.
"""
import numpy as np
import pytest
import torch

import ff_input_projection_gb300 as fpx
import fpsynth
import oracle
from tests.gpu_util import assert_close, host, run, to_device

pytestmark = pytest.mark.gpu

FIRST = fpsynth.Workload("noalloc_walrus", (2, 3, 64, 16, 16, 1), 2, 1, 64, 128, 2, 32,
                         fpsynth.ACT_GELU_ERF, 10000.0, True, "bf16", 61)
SECOND = fpsynth.Workload("noalloc_llm", (2, 333, 256), 2, 1, 256, 0, 2, 128, fpsynth.ACT_NONE,
                          500.0, False, "bf16", 62)


def _noalloc(w, inp, pos):
    x, W, b = (to_device(inp[k], w.dtype) for k in ("x", "W", "b"))
    pos_t = None if pos is None else torch.from_numpy(pos.astype(np.int32)).cuda()
    Bb, T = w.Bb, w.T
    dt = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    ff = torch.empty((Bb * T, w.F), dtype=dt, device="cuda") if w.F else None
    kvh = w.n_query_groups or w.heads
    qkv = [torch.empty((Bb * nh, T, w.head_dim), dtype=dt, device="cuda")
           for nh in (w.heads, kvh, kvh)] if w.heads else [None] * 3
    cfg = fpx.fp_config(w.C, w.F, w.heads, w.head_dim, w.n_query_groups, w.rope_n_elem, w.act,
                        w.rope_base, int(w.k_transposed))
    L = fpx.make_layout(x.shape, x.stride(), w.channel_dim, w.n_batch_dims,
                        fpx.FP_BF16 if w.dtype == "bf16" else fpx.FP_F32)
    p = lambda t: None if t is None else t.data_ptr()
    st = fpx.fp_forward_noalloc(cfg, x.data_ptr(), L, W.data_ptr(), p(b), p(pos_t), p(ff),
                                p(qkv[0]), p(qkv[1]), p(qkv[2]),
                                torch.cuda.current_stream().cuda_stream)
    assert st == fpx.FP_OK, fpx.fp_last_error()
    torch.cuda.synchronize()
    return dict(zip(("ff", "q", "k", "v"), (ff, *qkv)))


def test_noalloc_matches_fp_forward_two_calls(cuda_ok):
    cases = [(FIRST, (np.arange(FIRST.T) * 7 + 11) % 5000), (SECOND, None)]
    for w, pos in cases:
        inp = fpsynth.make_inputs(w)
        ref = run(w, inp, pos=pos)
        got = _noalloc(w, inp, pos)
        # the oracle too, so the check does not rest on the other entry point alone
        ref_o = oracle.forward_workload(w, dict(inp, pos=pos))
        for k in ("ff", "q", "k", "v"):
            if ref[k] is None:
                assert got[k] is None
                continue
            assert_close(host(got[k]), host(ref[k]), w.dtype, f"{w.name}:{k}")
            assert_close(host(got[k]), ref_o[k], w.dtype, f"{w.name}:{k} (oracle)")
        # the status words of the static array: nothing went wrong, and reading
        # them allocates nothing either
        assert fpx.fp_get_device_status(None, torch.cuda.current_stream().cuda_stream) == \
            fpx.FP_OK, fpx.fp_last_error()


def test_noalloc_leaves_free_device_memory_unchanged(cuda_ok):
    """After a first call has loaded the kernels, a call with another sequence
    length and other positions changes the device's free memory by nothing."""
    w = FIRST
    inp = fpsynth.make_inputs(w)
    _noalloc(w, inp, None)  # loads the kernel variants this configuration uses
    w2 = w.scaled(name="noalloc_walrus_2", x_shape=(2, 5, 64, 16, 16, 1))
    inp2 = fpsynth.make_inputs(w2)
    pos2 = (np.arange(w2.T) * 3 + 5) % 7000
    x, W, b = (to_device(inp2[k], w2.dtype) for k in ("x", "W", "b"))
    pos_t = torch.from_numpy(pos2.astype(np.int32)).cuda()
    ff = torch.empty((w2.Bb * w2.T, w2.F), dtype=torch.bfloat16, device="cuda")
    qkv = [torch.empty((w2.Bb * w2.heads, w2.T, w2.head_dim), dtype=torch.bfloat16,
                       device="cuda") for _ in range(3)]
    cfg = fpx.fp_config(w2.C, w2.F, w2.heads, w2.head_dim, 0, 0, w2.act, w2.rope_base, 0)
    L = fpx.make_layout(x.shape, x.stride(), w2.channel_dim, w2.n_batch_dims, fpx.FP_BF16)
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    st = fpx.fp_forward_noalloc(cfg, x.data_ptr(), L, W.data_ptr(), b.data_ptr(), pos_t.data_ptr(),
                                ff.data_ptr(), *[t.data_ptr() for t in qkv],
                                torch.cuda.current_stream().cuda_stream)
    assert st == fpx.FP_OK, fpx.fp_last_error()
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0, (free0, free1)
    ref = oracle.forward_workload(w2, dict(inp2, pos=pos2))
    for k, o in zip(("ff", "q", "k", "v"), [ff] + qkv):
        assert_close(host(o), ref[k], "bf16", f"noalloc second call:{k}")


def test_noalloc_rejects_a_table_beyond_its_maximum(cuda_ok):
    # T * rotated-half = 8200 * 64 > 524288 table entries
    C, T = 128, 8200
    x = torch.zeros((1, T, C), dtype=torch.bfloat16, device="cuda")
    W = torch.zeros((C, 3 * C), dtype=torch.bfloat16, device="cuda")
    outs = [torch.empty((1, T, C), dtype=torch.bfloat16, device="cuda") for _ in range(3)]
    cfg = fpx.fp_config(C, 0, 1, C, 0, 0, 0, 10000.0)
    L = fpx.make_layout(x.shape, x.stride(), 2, 1, fpx.FP_BF16)
    st = fpx.fp_forward_noalloc(cfg, x.data_ptr(), L, W.data_ptr(), None, None, None,
                                *[o.data_ptr() for o in outs], None)
    assert st == fpx.FP_ERR_INVALID_ARG
    assert "at most 524288" in fpx.fp_last_error()
