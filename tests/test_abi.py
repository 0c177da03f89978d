"""CPU checks of the C-ABI library: it loads without a GPU, exports every
symbol the header declares, and rejects bad arguments on the host."""
import ctypes
import os
import re

import pytest

from transformer_decoder_layer_llama_gb300 import api, synth

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include",
                      "llama_layer.h")


def declared_symbols():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(ll_[a-z0-9_]+)\s*\(", text)))


def test_every_declared_symbol_is_exported():
    names = declared_symbols()
    assert len(names) >= 10, names
    for n in names:
        assert hasattr(api.lib, n), n
    assert set(names) == set(api.EXPORTED)


def test_strerror_names_codes():
    assert api.lib.ll_strerror(0) == b"ok"
    assert b"workspace" in api.lib.ll_strerror(api.LL_ERR_WORKSPACE)


def test_sizes_are_host_arithmetic():
    c = api.make_config(synth.DIMS_7B, 4096)
    n = api.packed_weights_size(c)
    w = (12288 * 4096 + 4096 * 4096 + 2 * 11008 * 4096 + 4096 * 11008) * 2
    assert w <= n < w + 4096 * 64 * 8 + 1 << 20
    assert api.workspace_size(c, 2048, 16) > 6 * 2048 * 4096 * 2
    bad = api.make_config(synth.LayerDims(4096, 32, 32, 96, 11008, 128), 4096)
    assert api.packed_weights_size(bad) == 0          # head_dim 96 unsupported
    assert api.workspace_size(c, 0, 16) == 0


def test_step_by_step_workspace_is_the_fused_one_plus_its_intermediates():
    c = api.make_config(synth.DIMS_7B, 4096)
    T, mb = 64, 32
    fused = api.workspace_size(c, T, mb)
    assert api.lib.ll_workspace_size_mode(ctypes.byref(c), T, mb, api.LL_MODE_FUSED) == fused
    step = api.workspace_size(c, T, mb, api.LL_MODE_STEP_BY_STEP)
    nqkv, H, I = 12288, 4096, 11008
    extra = T * (nqkv + 1 + H + 2 * I + H) * 4
    assert extra <= step - fused < extra + 6 * 256
    assert api.lib.ll_workspace_size_mode(ctypes.byref(c), T, mb, 2) == 0
    cp, sp = api.ll_checkpoints(), api.ll_step_checkpoints()
    assert api.lib.ll_workspace_checkpoints(ctypes.byref(c), T, mb, ctypes.byref(cp)) == 0
    assert api.lib.ll_workspace_step_checkpoints(ctypes.byref(c), T, mb, ctypes.byref(sp)) == 0
    assert fused <= sp.qkv < sp.slots < sp.o_proj < sp.gate_up < sp.down < step
    assert sp.down + T * H * 4 <= step and cp.a < fused


def test_host_validation_returns_codes_without_launching():
    c = api.make_config(synth.DIMS_TINY, 128)
    pool = api.ll_kv_pool(0, 0, 0)
    null = ctypes.c_void_p(0)
    rc = api.lib.ll_layer_prefill(ctypes.byref(c), null, null, null, 1, 1, ctypes.byref(pool), null,
                                  1, null, null, 0, null, null)
    assert rc == api.LL_ERR_INVALID_ARG
    rc = api.lib.ll_reshape_and_cache(null, null, null, 1, 2, 64, 16, ctypes.byref(pool), null, null)
    assert rc == api.LL_ERR_INVALID_ARG
    gqa17 = api.make_config(synth.LayerDims(256, 34, 2, 64, 688, 16), 128)   # group of 17 heads
    assert api.lib.ll_layer_decode_step(ctypes.byref(gqa17), null, null, ctypes.byref(pool), null,
                                        1, null, 1, null, null, 0, null, null) == api.LL_ERR_UNSUPPORTED
    assert api.lib.ll_linear(null, null, null, 1, 16, 16, null, 0, null, null) == api.LL_ERR_INVALID_ARG


def test_python_binding_refuses_cpu_tensors():
    import torch
    c = api.make_config(synth.DIMS_TINY, 128)
    x = torch.zeros(4, 256, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        api.linear(x, torch.zeros(16, 256, dtype=torch.bfloat16))


def test_workspace_checkpoints_lie_inside_the_workspace():
    """The fused layer's checkpoints (one region per kernel output) are disjoint,
    16-byte aligned, hold max_tokens rows each, and fit the workspace size."""
    for name in ("tiny_gqa", "llama2_7b_decode", "llama70b_gqa_decode"):
        d = synth.WORKLOADS[name].dims
        cfg = api.make_config(d, max_position=4096)
        T, mb = 96, 40
        total = api.workspace_size(cfg, T, mb)
        out = api.ll_checkpoints()
        assert api.lib.ll_workspace_checkpoints(ctypes.byref(cfg), T, mb, ctypes.byref(out)) == 0
        nq = d.n_heads * d.head_dim
        widths = {"x_hat": d.hidden * 2, "q": nq * 2, "o": nq * 2, "h": d.hidden * 4,
                  "h_hat": d.hidden * 2, "a": d.intermediate * 2}
        spans = sorted((getattr(out, k), getattr(out, k) + T * w) for k, w in widths.items())
        for (a0, a1), (b0, _) in zip(spans, spans[1:]):
            assert a1 <= b0
        assert all(a0 % 16 == 0 for a0, _ in spans)
        assert spans[-1][1] <= total
        assert api.lib.ll_workspace_checkpoints(ctypes.byref(cfg), 0, mb, ctypes.byref(out)) == api.LL_ERR_INVALID_ARG
