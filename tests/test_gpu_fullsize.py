"""GPU parity at the full sizes of the named workloads, in the launch
configuration bench.py times (same entry points, same shapes).

* Llama-2-7B layer prefill, one sequence of 2048 tokens: every output element
  and the cache contents against the oracle.
* Llama-2-7B layer decode step, batch 64, context ~U[512, 4096].
* 70B-shaped GQA layer decode step, batch 16, context ~U[4096, 32768]
  (several 1024-key splits per sequence).

Layer outputs use the two-tier check of tests/helpers.py (the per-element
bound on all but a small fraction, a derived hard bound on every element);
the cache writes are checked slot by slot.
"""
import numpy as np
import pytest
import torch

from oracle import llama_layer as O
from tests.helpers import assert_close, assert_close_fullsize, bits, f64
from transformer_decoder_layer_llama_gb300 import synth

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    from transformer_decoder_layer_llama_gb300 import api
DEV = "cuda"


def _weights(wl, seed):
    W = synth.make_weights(wl.dims, wl.w_std, seed=seed)
    Wn = {k: f64(v) for k, v in W.items()}
    return W, Wn


def test_llama2_7b_prefill_full():
    wl = synth.WORKLOADS["llama2_7b_prefill"]
    d, B, S = wl.dims, wl.batch, wl.prefill_len
    W, Wn = _weights(wl, 11)
    x = synth.make_x(B * S, d.hidden, seed=12)
    table, nb = synth.make_block_table([S] * B, d.block_size, seed=13, extra_blocks=2)
    kp, vp = synth.make_pool(nb, d, seed=14, fill="sentinel")
    pos = synth.prefill_positions(B, S)
    cfg = api.make_config(d, S)
    packed = api.pack_weights(cfg, {k: v.to(DEV) for k, v in W.items()})
    kpd, vpd = kp.to(DEV), vp.to(DEV)
    status = api.new_status()
    y = api.layer_prefill(cfg, packed, x.to(DEV), pos.to(DEV), B, S, kpd, vpd, table.to(DEV),
                          status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    ko, vo = bits(kp), bits(vp)
    y_ref = O.layer_prefill(d, Wn, f64(x), pos.numpy(), B, S, ko, vo, table.numpy())
    assert_close_fullsize(f64(y), y_ref, "7B prefill y")
    kg, vg = bits(kpd), bits(vpd)
    np.testing.assert_array_equal(kg == 0xC480, ko == 0xC480)
    assert_close(O.bf16_value(kg), O.bf16_value(ko), "7B K cache")
    assert_close(O.bf16_value(vg), O.bf16_value(vo), "7B V cache")


@pytest.mark.parametrize("name", ["llama2_7b_decode", "llama70b_gqa_decode"])
def test_decode_step_full(name):
    wl = synth.WORKLOADS[name]
    d, B = wl.dims, wl.batch
    W, Wn = _weights(wl, 21)
    ctx = synth.make_context_lens(B, wl.ctx_lo, wl.ctx_hi, seed=22)
    ctx[0], ctx[-1] = wl.ctx_lo, wl.ctx_hi          # both ends of the range
    table, nb = synth.make_block_table(ctx.tolist(), d.block_size, seed=23, extra_blocks=2)
    kp, vp = synth.make_pool(nb, d, seed=24)
    x = synth.make_x(B, d.hidden, seed=25)
    cfg = api.make_config(d, int(ctx.max()))
    packed = api.pack_weights(cfg, {k: v.to(DEV) for k, v in W.items()})
    kpd, vpd = kp.to(DEV), vp.to(DEV)
    status = api.new_status()
    y = api.layer_decode_step(cfg, packed, x.to(DEV), kpd, vpd, table.to(DEV), ctx.to(DEV),
                              status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    ko, vo = bits(kp), bits(vp)
    want = {}
    y_ref = O.layer_decode_step(d, Wn, f64(x), ko, vo, table.numpy(), ctx.numpy(), want=want)
    assert_close_fullsize(f64(y), y_ref, f"{name} y")
    # the appended K/V rows: same slots, values within tolerance; everything else untouched
    kg, vg = bits(kpd), bits(vpd)
    changed = np.any(kg != bits(kp), axis=(1, 3)) | np.any(ko != bits(kp), axis=(1, 3))
    blk, off = np.nonzero(changed)
    assert len(blk) <= B
    assert_close(O.bf16_value(kg[blk, :, off]), O.bf16_value(ko[blk, :, off]), f"{name} new K")
    assert_close(O.bf16_value(vg[blk, :, off]), O.bf16_value(vo[blk, :, off]), f"{name} new V")
    mask = np.ones(kg.shape[0], bool)
    mask[np.unique(blk)] = False
    np.testing.assert_array_equal(kg[mask], ko[mask])
