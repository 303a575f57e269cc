"""Harder GPU checks of the forward, through the C ABI (needs a GB300).

* Persistent grids capped at 2 and 4 CTAs, so every CTA runs many tiles: both
  TMEM accumulators and their barrier phases are compared element by element.
* FP_OPT_BOUNDS_CHECK: with the check on, results are unchanged and nothing is
  reported; in its test mode (extents halved) the stores past the middle of
  each buffer are reported and never made.
* Guard bands: each output sits between two bands of a sentinel value, which
  must be untouched after the call (no kernel writes outside its outputs).
* 192-column tensor-core tiles (FP_OPT_TILE_N): forced on small shapes that
  cover ragged column tails, whole and straddled heads, the bias MMA and the
  pre-transposed k; identical bits to 256-column tiles and to the oracle.
* Scratch grown in stream order on one stream and used from others, and a
  forward captured into a CUDA graph on a stream other than the one that built
  the rotary table.
"""
import numpy as np
import pytest
import torch

import ff_input_projection_gb300 as fpx
import fpsynth
import oracle
from tests.gpu_util import assert_close, host, nan_outputs, out_shapes, run, to_device

pytestmark = pytest.mark.gpu

W_ = fpsynth.Workload
A = fpsynth

MULTI_TILE = [
    W_("mt_walrus", (2, 3, 64, 16, 16, 1), 2, 1, 64, 192, 2, 32, A.ACT_GELU_ERF, 10000.0, True,
       "bf16", 91),
    W_("mt_bert_qkv", (3, 177, 192), 2, 1, 192, 0, 3, 64, A.ACT_NONE, 0.0, True, "bf16", 92),
    W_("mt_llm_rope", (2, 300, 256), 2, 1, 256, 256, 2, 128, A.ACT_SILU, 10000.0, False, "bf16",
       93),
]


@pytest.mark.parametrize("max_ctas", [2, 4])
@pytest.mark.parametrize("cluster", [1, 2])
@pytest.mark.parametrize("w", MULTI_TILE, ids=lambda w: w.name)
def test_many_tiles_per_cta(w, cluster, max_ctas, cuda_ok):
    inp = fpsynth.make_inputs(w)
    proj = fpx.FusedProjection(w.C, w.F, w.heads, w.head_dim, w.act, w.rope_base)
    proj.set_option(fpx.FP_OPT_CLUSTER, cluster)
    proj.set_option(fpx.FP_OPT_MAX_CTAS, max_ctas)
    out = run(w, inp, proj=proj)
    ref = oracle.forward_workload(w, inp)
    for k in ("ff", "q", "k", "v"):
        if out[k] is not None:
            assert_close(host(out[k]), ref[k], w.dtype, f"{w.name}/{cluster}/{max_ctas}:{k}")


TILE192 = [
    # ff only, N = 1000: five full tiles of 192 and a 40-column tail
    W_("t192_ff_ragged", (3, 200, 256), 2, 1, 256, 1000, 0, 0, A.ACT_GELU_ERF, 0.0, True, "bf16",
       81),
    # q|k|v of 64-wide heads (three heads per tile) after a 192-column ff block
    W_("t192_ff_qkv", (2, 150, 256), 2, 1, 256, 192, 4, 64, A.ACT_SILU, 0.0, True, "bf16", 82),
    # 128-wide heads straddle the 192-column tiles; grouped k/v
    W_("t192_hd128_gqa", (2, 130, 512), 2, 1, 512, 0, 4, 128, A.ACT_NONE, 0.0, False, "bf16", 83,
       n_query_groups=2),
    # channels-first x (the A operand MN-major) and k pre-transposed: one tile
    W_("t192_nchw_kt", (2, 64, 12, 20), 1, 1, 64, 0, 1, 64, A.ACT_NONE, 0.0, True, "bf16", 84,
       k_transposed=True),
]


@pytest.mark.parametrize("max_ctas", [0, 4])
@pytest.mark.parametrize("w", TILE192, ids=lambda w: w.name)
def test_tile_192_matches_256(w, max_ctas, cuda_ok):
    inp = fpsynth.make_inputs(w)
    outs = []
    for tile_n in (256, 192):
        proj = _proj(w)
        proj.set_option(fpx.FP_OPT_TILE_N, tile_n)
        if max_ctas:
            proj.set_option(fpx.FP_OPT_MAX_CTAS, max_ctas)
        outs.append(run(w, inp, proj=proj))
        assert proj.device_status() == fpx.FP_OK, fpx.fp_last_error()
    ref = oracle.forward_workload(w, inp)
    for k in ("ff", "q", "k", "v"):
        if outs[0][k] is not None:
            assert torch.equal(outs[0][k], outs[1][k]), f"{w.name}:{k}"
            assert_close(host(outs[1][k]), ref[k], w.dtype, f"{w.name}/192:{k}")


# workloads whose stores are (partly) addressed by the kernels themselves
DIRECT = [
    W_("bc_short_seq_tc", (7, 20, 128), 2, 1, 128, 128, 2, 64, A.ACT_GELU_ERF, 10000.0, True,
       "bf16", 94),
    W_("bc_kt_bf16", (2, 3, 64, 8, 16, 1), 2, 1, 64, 64, 2, 32, A.ACT_GELU_ERF, 10000.0, True,
       "bf16", 95, k_transposed=True),
    W_("bc_ragged", (2, 3, 64, 10, 20, 1), 2, 1, 64, 128, 2, 32, A.ACT_GELU_ERF, 10000.0, True,
       "bf16", 96),
    W_("bc_simt_bf16", (2, 64, 5, 7), 1, 1, 64, 64, 2, 32, A.ACT_GELU_ERF, 10000.0, True, "bf16",
       97),
    W_("bc_simt_f32", (3, 50, 48), 2, 1, 48, 96, 3, 16, A.ACT_GELU_ERF, 10000.0, True, "f32", 98,
       k_transposed=True),
]
# tensor-core ff tiles, all rows valid: every store is the kernel-addressed
# warp-wide block copy out of the staging buffer
BLOCKS = W_("bc_blocks_tc", (4, 256, 128), 2, 1, 128, 640, 0, 0, A.ACT_GELU_ERF, 0.0, True,
            "bf16", 99)
DIRECT.append(BLOCKS)
SIMT_ONLY = [w for w in DIRECT if w.name.startswith("bc_simt")]


def _proj(w):
    return fpx.FusedProjection(w.C, w.F, w.heads, w.head_dim, w.act, w.rope_base,
                               w.n_query_groups, w.rope_n_elem, w.k_transposed)


@pytest.mark.parametrize("w", DIRECT, ids=lambda w: w.name)
def test_bounds_check_passes_correct_stores(w, cuda_ok):
    inp = fpsynth.make_inputs(w)
    proj = _proj(w)
    proj.set_option(fpx.FP_OPT_BOUNDS_CHECK, 1)
    out = run(w, inp, proj=proj)  # also asserts the device status is FP_OK
    ref = oracle.forward_workload(w, inp)
    for k in ("ff", "q", "k", "v"):
        if out[k] is not None:
            assert_close(host(out[k]), ref[k], w.dtype, f"{w.name}:{k}")


@pytest.mark.parametrize("w", SIMT_ONLY + [BLOCKS], ids=lambda w: w.name)
def test_bounds_check_stops_and_reports_stores_past_the_extent(w, cuda_ok):
    """Test mode: every extent is halved, so stores into the second half of a
    buffer count as out of bounds. They must be skipped (the NaN fill stays)
    and reported; the first half is still the right answer."""
    inp = fpsynth.make_inputs(w)
    proj = _proj(w)
    proj.set_option(fpx.FP_OPT_BOUNDS_CHECK, 2)
    x, W, b = (to_device(inp[k], w.dtype) for k in ("x", "W", "b"))
    out = proj.forward(x, W, b, None, channel_dim=w.channel_dim, n_batch_dims=w.n_batch_dims,
                       out=nan_outputs(proj, w))
    torch.cuda.synchronize()
    assert proj.device_status() == fpx.FP_ERR_DEVICE_BOUNDS
    assert proj.device_status() == fpx.FP_OK  # reported once, then cleared
    ref = oracle.forward_workload(w, inp)
    for k, o in zip(("ff", "q", "k", "v"), out):
        if o is None:
            continue
        flat = host(o).reshape(-1)
        r = ref[k].reshape(-1)
        half = flat.size // 2
        assert np.isnan(flat[half:]).all(), k
        rms = float(np.sqrt(np.mean(r ** 2)))
        assert_close(flat[:half], r[:half], w.dtype, f"{w.name}:{k}", rms=rms)


GUARD = 4096  # elements of sentinel before and after each output


@pytest.mark.parametrize("w", DIRECT + [A.WORKLOADS["gqa_rope_toy_bf16"], MULTI_TILE[2]],
                         ids=lambda w: w.name)
def test_guard_bands_around_outputs_stay_untouched(w, cuda_ok):
    inp = fpsynth.make_inputs(w)
    proj = _proj(w)
    dt = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    sentinel = 1234.5
    bufs, views = [], []
    for s in out_shapes(proj, w):
        if s is None:
            bufs.append(None)
            views.append(None)
            continue
        n = int(np.prod(s))
        buf = torch.full((n + 2 * GUARD,), sentinel, dtype=dt, device="cuda")
        buf[GUARD:GUARD + n] = float("nan")
        bufs.append(buf)
        views.append(buf[GUARD:GUARD + n].view(s))
    x, W, b = (to_device(inp[k], w.dtype) for k in ("x", "W", "b"))
    out = proj.forward(x, W, b, None, channel_dim=w.channel_dim, n_batch_dims=w.n_batch_dims,
                       out=tuple(views))
    torch.cuda.synchronize()
    assert proj.device_status() == fpx.FP_OK, fpx.fp_last_error()
    ref = oracle.forward_workload(w, inp)
    for k, buf, o in zip(("ff", "q", "k", "v"), bufs, out):
        if buf is None:
            continue
        assert (buf[:GUARD] == sentinel).all() and (buf[-GUARD:] == sentinel).all(), k
        assert_close(host(o), ref[k], w.dtype, f"{w.name}:{k}")


def test_scratch_growth_across_streams_and_graph_capture(cuda_ok):
    """The plan's scratch grows in stream order on the stream of the call that
    needs it; calls on other streams are ordered after it, and a forward
    captured on yet another stream waits on the table as an external event."""
    short = W_("grow_short", (2, 300, 256), 2, 1, 256, 0, 2, 128, A.ACT_NONE, 10000.0, False,
               "bf16", 99)
    long_ = short.scaled(name="grow_long", x_shape=(2, 1000, 256))
    proj = _proj(short)
    s1, s2, s3 = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()

    def fwd(w, stream):
        inp = fpsynth.make_inputs(w)
        x, W = to_device(inp["x"], "bf16"), to_device(inp["W"], "bf16")
        with torch.cuda.stream(stream):
            out = proj.forward(x, W, None, None, channel_dim=2, out=nan_outputs(proj, w))
        return inp, out

    checks = [(short, s1), (long_, s2), (short, s1), (long_, s3)]
    for w, st in checks:
        inp, out = fwd(w, st)
        torch.cuda.synchronize()
        assert proj.device_status() == fpx.FP_OK, fpx.fp_last_error()
        ref = oracle.forward_workload(w, inp)
        for k, o in zip(("ff", "q", "k", "v"), out):
            if o is not None:
                assert_close(host(o), ref[k], "bf16", f"{w.name}:{k}")
    # captured on a stream that never ran this plan (the table was built on s3)
    inp = fpsynth.make_inputs(long_)
    x, W = to_device(inp["x"], "bf16"), to_device(inp["W"], "bf16")
    outs = nan_outputs(proj, long_)
    g = torch.cuda.CUDAGraph()
    cap = torch.cuda.Stream()
    with torch.cuda.graph(g, stream=cap):
        proj.forward(x, W, None, None, channel_dim=2, out=outs, stream=cap.cuda_stream)
    g.replay()
    torch.cuda.synchronize()
    assert proj.device_status() == fpx.FP_OK, fpx.fp_last_error()
    ref = oracle.forward_workload(long_, inp)
    for k, o in zip(("ff", "q", "k", "v"), outs):
        if o is not None:
            assert_close(host(o), ref[k], "bf16", f"captured:{k}")
