"""fp_attention against the CPU oracle, through the C ABI (needs a GB300).

The attention consumes the projection's outputs in the [batch*heads, tokens,
head_dim] layout of memory-efficient-attention issue #7. Small cases compare
every output element (one and several key chunks, ragged chunk tails, both k
layouts, head_dim 64 and 128, grouped-query heads, peaky softmax rows); the
UNet attention configuration (4096 tokens, 5 heads, batch 2) is fed by
fp_forward with k emitted pre-transposed and compared in full. Launches whose
query blocks leave the last wave of SMs partly idle split those blocks' keys
over several CTAs and merge the partial results in a second launch; one case
fills exactly one wave and is not split. Tolerance: the bf16 rule,
|d| <= max(1e-2 |ref|, 2e-2 rms(ref)).
"""
import numpy as np
import pytest
import torch

import ff_input_projection_gb300 as fpx
import fpsynth
import oracle
from tests.gpu_util import assert_close, host, run, to_device

pytestmark = pytest.mark.gpu

# (name, batch, heads, kv_heads, head_dim, T_q, T_k, k_transposed, q scale, softmax scale)
CASES = [
    ("kt_two_chunks", 2, 2, 2, 64, 200, 200, True, 1.0, 0.0),
    ("plain_k", 2, 2, 2, 64, 150, 264, False, 1.0, 0.0),
    ("one_key_chunk", 1, 3, 3, 64, 130, 72, True, 1.0, 0.0),
    ("one_key_chunk_odd", 1, 3, 3, 64, 130, 77, False, 1.0, 0.0),
    ("hd128", 1, 2, 2, 128, 129, 296, True, 1.0, 0.0),
    ("hd128_plain", 2, 1, 1, 128, 64, 129, False, 1.0, 0.0),
    ("single_query", 1, 2, 2, 64, 1, 512, True, 1.0, 0.0),
    ("grouped_query", 2, 4, 2, 64, 100, 136, True, 1.0, 0.0),
    ("peaky_rows", 1, 2, 2, 64, 128, 640, True, 6.0, 0.0),
    ("custom_scale", 1, 1, 1, 64, 96, 256, False, 1.0, 0.5),
    # one block over 8 key chunks, the last ragged: 8 splits of one chunk each
    ("many_splits_ragged", 1, 1, 1, 64, 128, 1000, True, 1.0, 0.0),
    ("many_splits_hd128", 1, 1, 1, 128, 70, 904, False, 2.0, 0.0),
]


def _bits(shape, seed, stream, sd=1.0):
    vals = fpsynth.normal(seed, stream, int(np.prod(shape))) * sd
    return fpsynth.f32_to_bf16_bits(vals.astype(np.float32)).reshape(shape)


@pytest.mark.parametrize("case", CASES, ids=lambda c: c[0])
def test_attention_small_full_compare(case, cuda_ok):
    name, B, H, KV, hd, Tq, Tk, kt, qs, scale = case
    seed = 200 + CASES.index(case)
    q = _bits((B * H, Tq, hd), seed, 1, qs)
    k = _bits((B * KV, hd, Tk) if kt else (B * KV, Tk, hd), seed, 2)
    v = _bits((B * KV, Tk, hd), seed, 3)
    proj = fpx.FusedProjection(H * hd, 0, H, hd, "none", 0.0, KV if KV != H else 0, 0, kt)
    qd, kd, vd = (to_device(a, "bf16") for a in (q, k, v))
    out = torch.full((B * H, Tq, hd), float("nan"), dtype=torch.bfloat16, device="cuda")
    proj.attention(qd, kd, vd, batch=B, scale=scale, out=out)
    torch.cuda.synchronize()
    assert proj.device_status() == fpx.FP_OK, fpx.fp_last_error()
    # the oracle takes each query head's own k/v head
    zkv = np.array([(z // H) * KV + (z % H) // (H // KV) for z in range(B * H)])
    ref = oracle.attention(q, np.ascontiguousarray(k[zkv]), np.ascontiguousarray(v[zkv]),
                           dtype="bf16", k_transposed=kt, scale=scale if scale > 0 else None,
                           q_chunk=37, kv_chunk=50)
    assert_close(host(out), ref, "bf16", name)
    nkb = (Tk + 127) // 128
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    blocks = B * H * ((Tq + 127) // 128)
    split = blocks % sms != 0 and nkb >= 2 and min(nkb, sms // (blocks % sms)) >= 2
    assert proj.last_launch_count == (2 if split else 1)


def test_attention_whole_wave_is_not_split(cuda_ok):
    """As many query blocks as SMs: one wave, every block over all its keys in
    one CTA (one launch), against the oracle."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    B, H, hd, Tq, Tk = 1, sms, 64, 100, 384
    q = _bits((B * H, Tq, hd), 301, 1)
    k = _bits((B * H, hd, Tk), 301, 2)
    v = _bits((B * H, Tk, hd), 301, 3)
    proj = fpx.FusedProjection(H * hd, 0, H, hd, "none", 0.0, 0, 0, True)
    out = torch.full((B * H, Tq, hd), float("nan"), dtype=torch.bfloat16, device="cuda")
    proj.attention(*(to_device(a, "bf16") for a in (q, k, v)), batch=B, out=out)
    torch.cuda.synchronize()
    assert proj.device_status() == fpx.FP_OK, fpx.fp_last_error()
    assert proj.last_launch_count == 1
    ref = oracle.attention(q, k, v, dtype="bf16", k_transposed=True, q_chunk=64, kv_chunk=100)
    assert_close(host(out), ref, "bf16", "whole wave")


def test_attention_on_unet_projection_outputs(cuda_ok):
    """The diffusion-UNet attention projection (x NCHW [2, 320, 64, 64], 5 heads
    x 64) with k emitted pre-transposed, then attention over its outputs: every
    element against the oracle evaluated on the same q, k^T, v."""
    w = fpsynth.WORKLOADS["unet_qkv_bf16"].scaled(k_transposed=True)
    inp = fpsynth.make_inputs(w)
    proj = fpx.FusedProjection(w.C, w.F, w.heads, w.head_dim, w.act, w.rope_base, 0, 0, True)
    out = run(w, inp, proj=proj)
    q, kT, v = out["q"], out["k"], out["v"]
    assert tuple(kT.shape) == (w.Bb * w.heads, w.head_dim, w.T)
    att = torch.full_like(q, float("nan"))
    proj.attention(q, kT, v, batch=w.Bb, out=att)
    torch.cuda.synchronize()
    assert proj.device_status() == fpx.FP_OK, fpx.fp_last_error()
    bits = lambda t: t.cpu().view(torch.int16).numpy().view(np.uint16)
    ref = oracle.attention(bits(q), bits(kT), bits(v), dtype="bf16", k_transposed=True,
                           q_chunk=512, kv_chunk=1024)
    assert_close(host(att), ref, "bf16", "unet attention")


def test_attention_rejects_on_host(cuda_ok):
    proj = fpx.FusedProjection(96, 0, 3, 32, "none", 0.0)
    t = torch.zeros((3, 10, 32), dtype=torch.bfloat16, device="cuda")
    st = fpx.fp_attention(proj.plan, t.data_ptr(), t.data_ptr(), t.data_ptr(),
                          torch.empty_like(t).data_ptr(), 1, 10, 10, 0.0, None)
    assert st == fpx.FP_ERR_UNSUPPORTED_LAYOUT  # head_dim 32
    proj2 = fpx.FusedProjection(128, 0, 2, 64, "none", 0.0, 0, 0, True)
    u = torch.zeros((2, 64, 12), dtype=torch.bfloat16, device="cuda")
    st = fpx.fp_attention(proj2.plan, u.data_ptr(), u.data_ptr(), u.data_ptr(),
                          torch.empty_like(u).data_ptr(), 1, 12, 12, 0.0, None)
    assert st == fpx.FP_ERR_UNSUPPORTED_LAYOUT  # pre-transposed k with T_k % 8 != 0
    st = fpx.fp_attention(proj2.plan, u.data_ptr(), u.data_ptr(), u.data_ptr(), u.data_ptr(),
                          1, 16, 16, 0.0, None)
    assert st == fpx.FP_ERR_INVALID_ARG  # out overlaps the inputs


@pytest.mark.parametrize("hd,kt", [(128, False), (64, True)])
def test_attention_persistent_many_units(hd, kt, cuda_ok):
    """320 query blocks (B 2 x 5 heads x 4096 queries) on one CTA per SM: each
    CTA walks several whole blocks (alternating TMEM output buffers, the q
    buffer refilled between units) and then key ranges of the split tail;
    every element against the oracle."""
    B, H, Tq, Tk = 2, 5, 4096, 512
    q = _bits((B * H, Tq, hd), 320 + hd, 1)
    k = _bits((B * H, hd, Tk) if kt else (B * H, Tk, hd), 320 + hd, 2)
    v = _bits((B * H, Tk, hd), 320 + hd, 3)
    proj = fpx.FusedProjection(H * hd, 0, H, hd, "none", 0.0, 0, 0, kt)
    out = torch.full((B * H, Tq, hd), float("nan"), dtype=torch.bfloat16, device="cuda")
    proj.attention(*(to_device(a, "bf16") for a in (q, k, v)), batch=B, out=out)
    torch.cuda.synchronize()
    assert proj.device_status() == fpx.FP_OK, fpx.fp_last_error()
    ref = oracle.attention(q, k, v, dtype="bf16", k_transposed=kt, q_chunk=1024, kv_chunk=256)
    assert_close(host(out), ref, "bf16", f"persistent hd{hd}")
