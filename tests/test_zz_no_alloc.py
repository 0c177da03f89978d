"""The non-allocating decode-attention entry point, called through the C ABI.

ll_paged_attention_decode_noalloc serves callers that only own the buffers
they pass in (for example a plugin handed its input and output tensors by a
host framework that offers no workspace): it keeps its split partials in a
fixed array inside the library.  Two calls in a row (different shapes, the
second reusing the array the first left behind) must give the same result as
ll_paged_attention_decode with a caller workspace.  This file is collected
last on purpose.
"""
import ctypes
import math

import pytest
import torch

from oracle import llama_layer as O
from tests.helpers import assert_close, bits, f64
from transformer_decoder_layer_llama_gb300 import synth

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    from transformer_decoder_layer_llama_gb300 import api


def _case(B, Hq, Hkv, d, bs, lo, hi, seed):
    dims = synth.LayerDims(Hq * d, Hq, Hkv, d, 64, bs)
    ctx = synth.make_context_lens(B, lo, hi, seed=seed)
    table, nb = synth.make_block_table(ctx.tolist(), bs, seed=seed, extra_blocks=2)
    kp, vp = synth.make_pool(nb, dims, seed=seed)
    q = synth.normal_bf16((B, Hq, d), 1.0, seed=seed, tag="q")
    return [t.cuda() for t in (q, kp, vp, table, ctx)]


def _noalloc_via_abi(q, kp, vp, table, ctx, scale, out=None, status=None):
    B, Hq, d = q.shape
    out = torch.empty_like(q) if out is None else out
    status = torch.zeros(1, dtype=torch.int32, device="cuda") if status is None else status
    pool = api.ll_kv_pool(kp.data_ptr(), vp.data_ptr(), kp.shape[0])
    rc = api.lib.ll_paged_attention_decode_noalloc(
        ctypes.c_void_p(q.data_ptr()), ctypes.byref(pool), ctypes.c_void_p(table.data_ptr()),
        table.shape[1], ctypes.c_void_p(ctx.data_ptr()), B, Hq, kp.shape[1], d, kp.shape[2],
        scale, ctypes.c_void_p(out.data_ptr()), ctypes.c_void_p(status.data_ptr()),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == api.LL_OK, api.lib.ll_last_error()
    return out, status


def test_noalloc_matches_workspace_entry_two_calls():
    cases = [(4, 16, 2, 128, 128, 700, 3000, 5), (3, 8, 8, 64, 16, 1, 300, 6)]
    for B, Hq, Hkv, d, bs, lo, hi, seed in cases:
        q, kp, vp, table, ctx = _case(B, Hq, Hkv, d, bs, lo, hi, seed)
        scale = 1 / math.sqrt(d)
        ref = api.paged_attention_decode(q, kp, vp, table, ctx, scale)
        got, status = _noalloc_via_abi(q, kp, vp, table, ctx, scale)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        assert_close(f64(got), f64(ref), f"noalloc B{B} Hq{Hq} d{d}")


def _scratch_bytes(B, Hq, d, max_blocks, bs):
    """What the call needs of the fixed array: per split row the float32 partial output and
    (m, l), plus one 16-byte dispatch-order entry, and a 16-byte pad."""
    rows = B * Hq * -(-max_blocks * bs // 1024)
    return rows * ((d + 2) * 4 + 16) + 16


def test_noalloc_nine_splits_near_the_array_limit():
    """A block table 71 blocks wide (9 splits of 1024 keys) over 430 sequences x 16 heads:
    the scratch need sits just under the 32 MiB array, the dispatch-order table (built for
    8 or more splits) lands at its end.  Two sequences are 9 splits long, the rest short.
    Checked against the oracle and the workspace entry point, twice in a row, and the
    device's free memory does not move across the second call."""
    B, Hq, Hkv, d, bs, width = 430, 16, 2, 128, 128, 71
    need = _scratch_bytes(B, Hq, d, width, bs)
    assert 32 * 2 ** 20 - 600_000 < need <= 32 * 2 ** 20
    dims = synth.LayerDims(Hq * d, Hq, Hkv, d, 64, bs)
    ctx = synth.make_context_lens(B, 1, 200, seed=8)
    ctx[3], ctx[200] = 9000, 8193
    table, nb = synth.make_block_table(ctx.tolist(), bs, seed=8, extra_blocks=2, width=width)
    kp, vp = synth.make_pool(nb, dims, seed=8)
    q = synth.normal_bf16((B, Hq, d), 1.0, seed=8, tag="q")
    qd, kpd, vpd, td, cd = (t.cuda() for t in (q, kp, vp, table, ctx))
    scale = 1 / math.sqrt(d)
    ref = O.paged_attention_decode(f64(q), bits(kp), bits(vp), table.numpy(), ctx.numpy(), scale)
    ws_ref = api.paged_attention_decode(qd, kpd, vpd, td, cd, scale)
    got1, st1 = _noalloc_via_abi(qd, kpd, vpd, td, cd, scale)
    out2, st2 = torch.empty_like(qd), torch.zeros(1, dtype=torch.int32, device="cuda")
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    got2, _ = _noalloc_via_abi(qd, kpd, vpd, td, cd, scale, out=out2, status=st2)
    torch.cuda.synchronize()
    free1 = torch.cuda.mem_get_info()[0]
    assert int(st1.item()) == 0 and int(st2.item()) == 0
    assert free1 >= free0, (free0, free1)
    for got in (got1, got2):
        assert_close(f64(got), ref, "noalloc, 9 splits, against the oracle")
        assert_close(f64(got), f64(ws_ref), "noalloc, 9 splits, against the workspace entry point")


def test_noalloc_rejects_sizes_beyond_its_array():
    q, kp, vp, table, ctx = _case(2, 16, 2, 128, 128, 100, 200, 7)
    big = torch.zeros((4096, 4096), dtype=torch.int32, device="cuda")   # 4096 rows x 512K keys
    qb = torch.zeros((4096, 16, 128), dtype=torch.bfloat16, device="cuda")
    ctxb = torch.ones(4096, dtype=torch.int32, device="cuda")
    pool = api.ll_kv_pool(kp.data_ptr(), vp.data_ptr(), kp.shape[0])
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    rc = api.lib.ll_paged_attention_decode_noalloc(
        ctypes.c_void_p(qb.data_ptr()), ctypes.byref(pool), ctypes.c_void_p(big.data_ptr()), 4096,
        ctypes.c_void_p(ctxb.data_ptr()), 4096, 16, 2, 128, 128, 0.1,
        ctypes.c_void_p(qb.data_ptr()), ctypes.c_void_p(status.data_ptr()), None)
    assert rc == api.LL_ERR_UNSUPPORTED
    assert b"scratch" in api.lib.ll_last_error()
