"""Device-side failure detection without a GPU fault.

Every mbarrier wait in the tensor-core kernel is bounded. A test hook makes
one CTA withhold its first operand stage, so the MMA thread's wait runs out:
the kernel records FP_ERR_TIMEOUT in the plan's status word, the other roles
and CTAs stop, in-flight copies drain, TMEM is freed and the launch returns.
The context must stay usable: the next launch is correct.
"""
import pytest

import ff_input_projection_gb300 as fpx
import fpsynth
import oracle
from tests.gpu_util import assert_close, host, run, to_device

pytestmark = pytest.mark.gpu

CASE = fpsynth.Workload("fault_case", (2, 3, 64, 16, 16, 1), 2, 1, 64, 128, 2, 32,
                        fpsynth.ACT_GELU_ERF, 10000.0, True, "bf16", 51)


def test_timeout_is_reported_and_context_survives(cuda_ok):
    import torch
    w = CASE
    inp = fpsynth.make_inputs(w)
    proj = fpx.FusedProjection(w.C, w.F, w.heads, w.head_dim, w.act, w.rope_base)
    proj.set_option(fpx.FP_OPT_WAIT_LIMIT_NS, 200_000_000)  # 0.2 s
    proj.set_option(fpx.FP_OPT_INJECT_STALL, 1)
    x, W, b = (to_device(inp[k], w.dtype) for k in ("x", "W", "b"))
    proj.forward(x, W, b, None, channel_dim=w.channel_dim)
    torch.cuda.synchronize()
    assert proj.device_status() == fpx.FP_ERR_TIMEOUT
    # status was cleared by the read; the hook is one-shot; the GPU still works
    assert proj.device_status() == fpx.FP_OK
    ref = oracle.forward_workload(w, inp)
    out = run(w, inp, proj=proj)
    for k in ("ff", "q", "k", "v"):
        assert_close(host(out[k]), ref[k], w.dtype, f"after-timeout:{k}")


def test_backward_timeout_is_reported_and_context_survives(cuda_ok):
    """The same hook in the backward's first tensor-core GEMM (the ff gradient)."""
    import torch
    from tests.test_gpu_backward import run_backward
    w = CASE
    inp = fpsynth.make_inputs(w)
    grads = fpsynth.make_grads(w)
    proj = fpx.FusedProjection(w.C, w.F, w.heads, w.head_dim, w.act, w.rope_base)
    proj.set_option(fpx.FP_OPT_WAIT_LIMIT_NS, 200_000_000)  # 0.2 s
    proj.set_option(fpx.FP_OPT_INJECT_STALL, 1)
    x, W, b = (to_device(inp[k], w.dtype) for k in ("x", "W", "b"))
    g = tuple(to_device(grads[k], w.dtype) for k in ("ff", "q", "k", "v"))
    proj.backward(x, W, b, g, channel_dim=w.channel_dim)
    torch.cuda.synchronize()
    assert proj.device_status() == fpx.FP_ERR_TIMEOUT
    assert proj.device_status() == fpx.FP_OK
    dx, dW, db = run_backward(w, inp, grads, proj=proj)
    ref = oracle.backward_workload(w, inp, grads)
    assert_close(dx, ref["dx"], "bf16", "after-timeout:dx")
    assert_close(dW, ref["dW"], "bf16", "after-timeout:dW")
