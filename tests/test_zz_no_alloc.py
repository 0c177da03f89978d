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

from tests.helpers import assert_close, f64
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


def _noalloc_via_abi(q, kp, vp, table, ctx, scale):
    B, Hq, d = q.shape
    out = torch.empty_like(q)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
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
