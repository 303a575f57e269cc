"""The C ABI without a GPU: the library loads, exports what include/fp.h declares,
and rejects bad arguments on the host before any CUDA call."""
import ctypes
import os
import re

import pytest

import ff_input_projection_gb300 as fpx
from ff_input_projection_gb300 import _build

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "fp.h")


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return fpx.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(fp_[a-z_]+)\s*\(", text)))


def test_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert set(names) == set(fpx.EXPORTS), names
    for n in names:
        assert hasattr(lib, n), n


def test_status_strings(lib):
    for code in range(8):
        s = fpx.fp_status_string(code)
        assert s and s != "unknown status"
    assert fpx.fp_status_string(99) == "unknown status"


@pytest.mark.parametrize("args", [
    (0, 64, 2, 16, 0, 0.0),      # C = 0
    (32, 64, 2, 15, 0, 0.0),     # odd head_dim
    (32, 64, 3, 16, 0, 0.0),     # heads * head_dim != C
    (32, 40, 2, 16, 0, 0.0),     # ff_hidden not a multiple of head_dim
    (32, 0, 0, 0, 0, 0.0),       # nothing to compute
    (32, 64, 2, 16, 9, 0.0),     # unknown activation
    (32, 64, 2, 16, 5, 0.0),     # unknown activation
    (512, 0, 2, 256, 0, 10000.0),  # rotary with head_dim > 128
    (32, -1, 2, 16, 0, 0.0),     # negative ff_hidden
])
def test_create_rejects(lib, args):
    st, h = fpx.fp_create(*args)
    assert st == fpx.FP_ERR_INVALID_ARG and h is None
    assert fpx.fp_last_error()


def _plan(C=64, F=64, heads=4, hd=16, act=1, rope=0.0):
    st, h = fpx.fp_create(C, F, heads, hd, act, rope)
    assert st == fpx.FP_OK, fpx.fp_last_error()
    return h


# fake, 16-byte-aligned device addresses: the checks below must reject the call
# before anything dereferences them
X, WP, BP, O1, O2, O3, O4 = (0x10000000 + i * 0x1000000 for i in range(7))


def _cf_layout(dtype=fpx.FP_BF16, B=2, C=64, H=8, W=8):
    return fpx.make_layout([B, C, H, W], [C * H * W, H * W, W, 1], 1, 1, dtype)


def test_forward_rejects_on_host(lib):
    h = _plan()
    L = _cf_layout()
    fwd = lambda **kw: fpx.fp_forward(h, kw.get("x", X), kw.get("L", L), kw.get("W", WP),
                                      kw.get("b", BP), None, kw.get("ff", O1), kw.get("q", O2),
                                      kw.get("k", O3), kw.get("v", O4), None)
    assert fwd(x=None) == fpx.FP_ERR_INVALID_ARG
    assert fwd(W=None) == fpx.FP_ERR_INVALID_ARG
    assert fwd(ff=None) == fpx.FP_ERR_INVALID_ARG  # F > 0 needs out_ff
    assert fwd(k=None) == fpx.FP_ERR_INVALID_ARG
    assert fwd(x=X + 2) == fpx.FP_ERR_MISALIGNED
    assert fwd(b=BP + 8) == fpx.FP_ERR_MISALIGNED
    assert fwd(q=O1) == fpx.FP_ERR_INVALID_ARG       # outputs alias
    assert fwd(v=X) == fpx.FP_ERR_INVALID_ARG        # output aliases input
    bad = _cf_layout(C=32)
    assert fwd(L=bad) == fpx.FP_ERR_INVALID_ARG      # channel count
    L2 = _cf_layout()
    L2.channel_dim = 7
    assert fwd(L=L2) == fpx.FP_ERR_INVALID_ARG
    L3 = _cf_layout()
    L3.dtype = 5
    assert fwd(L=L3) == fpx.FP_ERR_INVALID_ARG
    L4 = _cf_layout()
    L4.sizes[2] = -1
    assert fwd(L=L4) == fpx.FP_ERR_INVALID_ARG
    L5 = _cf_layout()
    L5.n_batch_dims = 4
    assert fwd(L=L5) == fpx.FP_ERR_INVALID_ARG
    fpx.fp_destroy(h)


def test_forward_host_rejects_on_host(lib):
    """The host-buffer entry point runs fp_forward's argument checks on the
    caller's pointers first, and takes only page-locked host memory: plain
    addresses (here, with no GPU, nothing is page-locked) are refused before
    any copy or launch."""
    h = _plan()
    L = _cf_layout()
    host = lambda **kw: fpx.fp_forward_host(h, kw.get("x", X), kw.get("L", L), WP, BP, None,
                                            kw.get("ff", O1), O2, O3, O4, None)
    assert fpx.fp_forward_host(None, X, L, WP, BP, None, O1, O2, O3, O4, None) == \
        fpx.FP_ERR_INVALID_ARG
    assert host(x=None) == fpx.FP_ERR_INVALID_ARG
    assert host(ff=None) == fpx.FP_ERR_INVALID_ARG     # F > 0 needs out_ff
    assert host(x=X + 2) == fpx.FP_ERR_MISALIGNED
    assert host(ff=X) == fpx.FP_ERR_INVALID_ARG        # output aliases input
    assert host(L=_cf_layout(C=32)) == fpx.FP_ERR_INVALID_ARG
    assert host() == fpx.FP_ERR_INVALID_ARG            # not page-locked host memory
    assert "page-locked" in fpx.fp_last_error()
    E = fpx.make_layout([0, 64, 8, 8], [4096, 64, 8, 1], 1, 1, fpx.FP_BF16)
    assert host(L=E) == fpx.FP_OK                      # no tokens: nothing to copy
    assert fpx.fp_last_launch_count(h) == 0
    fpx.fp_destroy(h)


def test_backward_host_rejects_on_host(lib):
    """fp_backward_host: fp_backward's checks first, then a dense x and
    page-locked host memory, all before anything is enqueued."""
    h = _plan()
    L = _cf_layout()
    G = (O1, O2, O3, O4)
    DX, DW, DB = 0x30000000, 0x31000000, 0x32000000
    bh = lambda **kw: fpx.fp_backward_host(h, kw.get("x", X), kw.get("L", L), WP, BP, None,
                                           *kw.get("g", G), kw.get("dx", DX), kw.get("dW", DW),
                                           DB, None)
    assert fpx.fp_backward_host(None, X, L, WP, BP, None, *G, DX, DW, DB, None) == \
        fpx.FP_ERR_INVALID_ARG
    assert bh(x=None) == fpx.FP_ERR_INVALID_ARG
    assert bh(g=(None, O2, O3, O4)) == fpx.FP_ERR_INVALID_ARG   # F > 0 needs g_ff
    assert bh(dW=None) == fpx.FP_ERR_INVALID_ARG
    assert bh(L=_cf_layout(dtype=fpx.FP_F32)) == fpx.FP_ERR_UNSUPPORTED_LAYOUT
    padded = fpx.make_layout([2, 64, 8, 8], [64 * 80, 80, 8, 1], 1, 1, fpx.FP_BF16)
    assert bh(L=padded) == fpx.FP_ERR_UNSUPPORTED_LAYOUT        # not dense
    assert bh() == fpx.FP_ERR_INVALID_ARG                       # not page-locked
    assert "page-locked" in fpx.fp_last_error()
    fpx.fp_destroy(h)


@pytest.mark.parametrize("kw", [
    dict(n_query_groups=3),                 # heads % groups
    dict(rope_n_elem=5),                    # odd
    dict(rope_n_elem=20),                   # > head_dim
    dict(n_query_groups=-1),
])
def test_create_ex_rejects(lib, kw):
    base = dict(C=64, ff_hidden=0, heads=4, head_dim=16, n_query_groups=2, rope_n_elem=0,
                act=0, rope_base=10000.0)
    base.update(kw)
    st, h = fpx.fp_create_ex(fpx.fp_config(**base))
    assert st == fpx.FP_ERR_INVALID_ARG and h is None


def test_create_ex_grouped_query(lib):
    cfg = fpx.fp_config(C=512, ff_hidden=0, heads=16, head_dim=32, n_query_groups=4,
                        rope_n_elem=8, act=0, rope_base=10000.0)
    st, h = fpx.fp_create_ex(cfg)
    assert st == fpx.FP_OK
    fpx.fp_destroy(h)


def test_backward_rejects_on_host(lib):
    """fp_backward's argument checks run on the host, before any CUDA call."""
    h = _plan()  # C 64, F 64, 4 heads of 16: N = 256
    L = _cf_layout()  # 2 x 64 tokens
    st, need = fpx.fp_backward_workspace_size(h, L)
    assert st == fpx.FP_OK and need == 128 * 256 * 2  # G [M, N] bf16, 256-byte rounded
    DX, DW, DB, WS = (0x30000000 + i * 0x1000000 for i in range(4))

    def bwd(plan=h, L=L, dx=DX, dW=DW, ws=WS, wsb=need):
        return fpx.fp_backward(plan, X, L, WP, BP, None, O1, O2, O3, O4, dx, dW, DB, ws, wsb, None)

    assert bwd(plan=None) == fpx.FP_ERR_INVALID_ARG
    assert bwd(dx=None) == fpx.FP_ERR_INVALID_ARG
    assert bwd(dW=None) == fpx.FP_ERR_INVALID_ARG
    assert bwd(dx=DX + 2) == fpx.FP_ERR_MISALIGNED
    assert bwd(ws=WS + 16) == fpx.FP_ERR_MISALIGNED       # workspace wants 256 bytes
    assert bwd(wsb=need - 256) == fpx.FP_ERR_INVALID_ARG  # workspace too small
    assert "workspace" in fpx.fp_last_error()
    assert bwd(L=_cf_layout(dtype=fpx.FP_F32)) == fpx.FP_ERR_UNSUPPORTED_LAYOUT
    st, _ = fpx.fp_backward_workspace_size(None, L)
    assert st == fpx.FP_ERR_INVALID_ARG
    E = fpx.make_layout([0, 64, 8, 8], [4096, 64, 8, 1], 1, 1, fpx.FP_BF16)
    st, need0 = fpx.fp_backward_workspace_size(h, E)
    assert st == fpx.FP_OK and need0 == 0
    assert bwd(L=E, dW=None) == fpx.FP_ERR_INVALID_ARG  # dW is written even with no tokens
    fpx.fp_destroy(h)


def test_empty_input_is_a_no_op(lib):
    h = _plan()
    L = fpx.make_layout([0, 64, 8, 8], [4096, 64, 8, 1], 1, 1, fpx.FP_BF16)
    assert fpx.fp_forward(h, X, L, WP, BP, None, O1, O2, O3, O4, None) == fpx.FP_OK
    assert fpx.fp_last_launch_count(h) == 0
    fpx.fp_destroy(h)


def test_options_and_status_without_device(lib):
    h = _plan()
    assert fpx.fp_set_option(h, fpx.FP_OPT_GROUP_M, 0) == fpx.FP_ERR_INVALID_ARG
    assert fpx.fp_set_option(h, fpx.FP_OPT_GROUP_M, 16) == fpx.FP_OK
    assert fpx.fp_set_option(h, fpx.FP_OPT_WAIT_LIMIT_NS, -5) == fpx.FP_ERR_INVALID_ARG
    assert fpx.fp_set_option(h, 77, 1) == fpx.FP_ERR_INVALID_ARG
    for v, want in ((-1, fpx.FP_ERR_INVALID_ARG), (3, fpx.FP_ERR_INVALID_ARG), (0, fpx.FP_OK),
                    (1, fpx.FP_OK), (2, fpx.FP_OK)):
        assert fpx.fp_set_option(h, fpx.FP_OPT_BOUNDS_CHECK, v) == want, v
    for v, want in ((128, fpx.FP_ERR_INVALID_ARG), (-1, fpx.FP_ERR_INVALID_ARG),
                    (192, fpx.FP_OK), (256, fpx.FP_OK), (0, fpx.FP_OK)):
        assert fpx.fp_set_option(h, fpx.FP_OPT_TILE_N, v) == want, v
    # no device state yet: nothing to report, no CUDA call made
    assert fpx.fp_get_device_status(h, None) == fpx.FP_OK
    fpx.fp_destroy(h)
    fpx.fp_destroy(None)


def test_wrapper_raises(lib):
    with pytest.raises(fpx.FpError):
        fpx.FusedProjection(30, 0, 4, 8)


def test_binding_has_no_fallback(monkeypatch, tmp_path):
    # a missing library is an error, never a silent substitute
    monkeypatch.setattr(fpx, "_lib", None)
    monkeypatch.setattr(_build, "LIB", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError):
        fpx.load()


def test_wrapper_checks_buffer_sizes(lib):
    """The C ABI gets raw pointers, so the torch wrapper checks sizes on the
    host: a weight with the wrong column count (e.g. a grouped-query weight
    given to a plan built without groups) is rejected before any launch."""
    import torch
    proj = fpx.FusedProjection(512, 0, 16, 32, "none", 10000.0)  # blocked q|k|v: N = 1536
    x = torch.zeros((2, 8, 512), dtype=torch.bfloat16)
    W_gqa = torch.zeros((512, 768), dtype=torch.bfloat16)       # grouped-query width
    with pytest.raises(ValueError):
        proj.forward(x, W_gqa, None, None, channel_dim=2)
    W = torch.zeros((512, 1536), dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        proj.forward(x, W, torch.zeros(10, dtype=torch.bfloat16), None, channel_dim=2)
    with pytest.raises(ValueError):
        proj.forward(x, W, None, torch.zeros(8, dtype=torch.int64), channel_dim=2)
    with pytest.raises(ValueError):
        proj.forward(x, W.float(), None, None, channel_dim=2)
    proj.close()


def test_host_wrappers_check_buffers(lib):
    """The host-buffer wrappers take only page-locked CPU activations,
    gradients and results, contiguous where the library copies byte ranges,
    and a weight on the GPU; each mismatch raises before the C ABI is called
    (without a GPU nothing here can be page-locked or on the device)."""
    import torch
    proj = fpx.FusedProjection(64, 64, 4, 16, "gelu", 0.0)
    x = torch.zeros((2, 8, 64), dtype=torch.bfloat16)           # pageable
    W = torch.zeros((64, 256), dtype=torch.bfloat16)            # CPU, not CUDA
    with pytest.raises(ValueError):
        proj.forward_host(x, W, None, None, channel_dim=2)
    grads = (torch.zeros((16, 64), dtype=torch.bfloat16),) + \
        tuple(torch.zeros((8, 8, 16), dtype=torch.bfloat16) for _ in range(3))
    with pytest.raises(ValueError):
        proj.backward_host(x, W, None, grads, channel_dim=2)
    with pytest.raises(ValueError):
        proj.backward_host(x.transpose(1, 2), W, None, grads, channel_dim=1)
    proj.close()
