"""The step-by-step execution mode (page "ATB fused-operator matrix and KV-cache
management", section on the engineering limits of fusion granularity): every
operator of the chain as its own kernel, every intermediate kept.

* Each operator's output against the oracle's value of that operator, including
  the ones the fused kernels never write out: q/k/v before RoPE, o W_o^T before
  the residual add, gate and up before SiLU * up, a W_down^T before the residual.
* Fused against step-by-step on the same inputs: the element-wise arithmetic of
  the two modes is the same code, so every shared intermediate, the cache and
  the output must agree bit for bit (tiny workload and the full 7B sizes).
"""
import numpy as np
import pytest
import torch

from oracle import llama_layer as O
from tests.helpers import assert_close, bits, f64
from transformer_decoder_layer_llama_gb300 import synth

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    from transformer_decoder_layer_llama_gb300 import api
DEV = "cuda"


def _unpack_qkv(qkv, d):
    """The QKV Linear output in the packed column order -> element order."""
    Hq, Hkv, hd = d.n_heads, d.n_kv_heads, d.head_dim
    T = qkv.shape[0]
    qk = qkv[:, :(Hq + Hkv) * hd].reshape(T, Hq + Hkv, hd // 2, 2)
    qk = np.concatenate([qk[..., 0], qk[..., 1]], axis=-1).reshape(T, -1)
    return np.concatenate([qk, qkv[:, (Hq + Hkv) * hd:]], axis=1)


def _tiny(seed, S, B, steps):
    wl = synth.WORKLOADS["tiny_gqa"]
    d = wl.dims
    W = synth.make_weights(d, wl.w_std, seed=seed)
    table, nb = synth.make_block_table([S + steps] * B, d.block_size, seed=seed + 3, extra_blocks=3)
    kp, vp = synth.make_pool(nb, d, seed=seed + 4, fill="sentinel")
    cfg = api.make_config(d, max_position=S + steps + 1)
    packed = api.pack_weights(cfg, {k: v.to(DEV) for k, v in W.items()})
    return d, W, {k: f64(v) for k, v in W.items()}, table, kp, vp, cfg, packed


@pytest.mark.parametrize("phase", ["prefill", "decode"])
def test_step_by_step_every_operator_against_oracle(phase):
    B, S = 2, 40
    d, W, Wn, table, kp, vp, cfg, packed = _tiny(101, S, B, 1)
    kpd, vpd, td = kp.to(DEV), vp.to(DEV), table.to(DEV)
    ko, vo = bits(kp), bits(vp)
    mode = api.LL_MODE_STEP_BY_STEP
    want = {}
    status = api.new_status()
    if phase == "prefill":
        T = B * S
        x = synth.make_x(T, d.hidden, seed=102)
        pos = synth.prefill_positions(B, S)
        ws = api.new_workspace(cfg, T, table.shape[1], mode=mode)
        y = api.layer_prefill(cfg, packed, x.to(DEV), pos.to(DEV), B, S, kpd, vpd, td, workspace=ws,
                              status=status, mode=mode)
        y_ref = O.layer_prefill(d, Wn, f64(x), pos.numpy(), B, S, ko, vo, table.numpy(), want=want)
    else:
        x0 = synth.make_x(B * S, d.hidden, seed=103)
        pos = synth.prefill_positions(B, S)
        api.layer_prefill(cfg, packed, x0.to(DEV), pos.to(DEV), B, S, kpd, vpd, td, mode=mode)
        O.layer_prefill(d, Wn, f64(x0), pos.numpy(), B, S, ko, vo, table.numpy())
        T = B
        x = synth.make_x(B, d.hidden, seed=104)
        ctx = torch.full((B,), S + 1, dtype=torch.int32)
        ws = api.new_workspace(cfg, T, table.shape[1], mode=mode)
        y = api.layer_decode_step(cfg, packed, x.to(DEV), kpd, vpd, td, ctx.to(DEV), workspace=ws,
                                  status=status, mode=mode)
        y_ref = O.layer_decode_step(d, Wn, f64(x), ko, vo, table.numpy(), ctx.numpy(), want=want)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    cp = api.checkpoints(cfg, ws, T, table.shape[1], T)
    sp = api.step_checkpoints(cfg, ws, T, table.shape[1], T)
    gu = f64(sp["gate_up"])
    got = {
        "x_hat": f64(cp["x_hat"]), "qkv": _unpack_qkv(f64(sp["qkv"]), d), "q": f64(cp["q"]),
        "k": f64(sp["k"]), "v": f64(sp["v"]), "o": f64(cp["o"]), "o_proj": f64(sp["o_proj"]),
        "h": f64(cp["h"]), "h_hat": f64(cp["h_hat"]), "gate": gu[:, 0::2], "up": gu[:, 1::2],
        "a": f64(cp["a"]), "down": f64(sp["down"]), "y": f64(y),
    }
    ref = {
        "x_hat": want["xh"], "qkv": want["qkv"], "q": want["q"].reshape(T, -1), "k": want["k"].reshape(T, -1),
        "v": want["v"].reshape(T, -1), "o": want["o"].reshape(T, -1), "o_proj": want["o_proj"], "h": want["h"],
        "h_hat": want["hh"], "gate": want["gate"], "up": want["up"], "a": want["a"], "down": want["down"],
        "y": y_ref,
    }
    for name in got:
        assert_close(got[name], ref[name], f"step-by-step {phase} {name}")
    np.testing.assert_array_equal(sp["slots"].cpu().numpy(), want["slots"])
    # the pool: the same slots written as the oracle's, values within the bound
    kg = bits(kpd)
    np.testing.assert_array_equal(kg == 0xC480, ko == 0xC480)
    assert_close(O.bf16_value(kg), O.bf16_value(ko), f"step-by-step {phase} K cache")


def _both_modes(run):
    """run(mode) -> (y, workspace, pools); returns both modes' results."""
    return run(api.LL_MODE_FUSED), run(api.LL_MODE_STEP_BY_STEP)


def _assert_same(fused, step, cfg, T, max_blocks, what):
    (yf, wsf, poolsf), (ys, wss, poolss) = fused, step
    torch.cuda.synchronize()
    assert torch.equal(yf, ys), f"{what}: y differs (max |diff| {(yf.float() - ys.float()).abs().max().item()})"
    cf = api.checkpoints(cfg, wsf, T, max_blocks, T)
    cs = api.checkpoints(cfg, wss, T, max_blocks, T)
    for name in cf:
        assert torch.equal(cf[name], cs[name]), f"{what}: checkpoint {name} differs"
    for pf, ps in zip(poolsf, poolss):
        assert torch.equal(pf, ps), f"{what}: KV pool differs"


@pytest.mark.parametrize("phase", ["prefill", "decode"])
def test_fused_equals_step_by_step_tiny(phase):
    B, S = 3, 37
    d, W, Wn, table, kp, vp, cfg, packed = _tiny(111, S, B, 1)
    td = table.to(DEV)
    x = synth.make_x(B * S, d.hidden, seed=112).to(DEV)
    pos = synth.prefill_positions(B, S).to(DEV)
    xd = synth.make_x(B, d.hidden, seed=113).to(DEV)
    ctx = torch.full((B,), S + 1, dtype=torch.int32, device=DEV)

    def run(mode):
        kpd, vpd = kp.to(DEV), vp.to(DEV)
        T = B * S if phase == "prefill" else B
        ws = api.new_workspace(cfg, T, table.shape[1], mode=mode)
        if phase == "prefill":
            y = api.layer_prefill(cfg, packed, x, pos, B, S, kpd, vpd, td, workspace=ws, mode=mode)
        else:
            api.layer_prefill(cfg, packed, x, pos, B, S, kpd, vpd, td, mode=mode)
            y = api.layer_decode_step(cfg, packed, xd, kpd, vpd, td, ctx, workspace=ws, mode=mode)
        return y, ws, (kpd, vpd)

    T = B * S if phase == "prefill" else B
    _assert_same(*_both_modes(run), cfg, T, table.shape[1], f"tiny {phase}")


@pytest.mark.parametrize("name", ["llama2_7b_prefill", "llama2_7b_decode", "llama70b_gqa_decode"])
def test_fused_equals_step_by_step_full_size(name):
    wl = synth.WORKLOADS[name]
    d = wl.dims
    W = synth.make_weights(d, wl.w_std, seed=121)
    if wl.prefill_len:
        B, S = wl.batch, wl.prefill_len
        T = B * S
        table, nb = synth.make_block_table([S] * B, d.block_size, seed=122, extra_blocks=2)
        cfg = api.make_config(d, S)
        pos = synth.prefill_positions(B, S).to(DEV)
        ctx = None
    else:
        B = T = wl.batch
        ctx_h = synth.make_context_lens(B, wl.ctx_lo, wl.ctx_hi, seed=122)
        table, nb = synth.make_block_table(ctx_h.tolist(), d.block_size, seed=123, extra_blocks=2)
        cfg = api.make_config(d, int(ctx_h.max()))
        ctx = ctx_h.to(DEV)
    packed = api.pack_weights(cfg, {k: v.to(DEV) for k, v in W.items()})
    x = synth.make_x(T, d.hidden, seed=124).to(DEV)
    td = table.to(DEV)
    kp, vp = synth.make_pool(nb, d, seed=125)
    kp, vp = kp.to(DEV), vp.to(DEV)

    def run(mode):
        kpd, vpd = kp.clone(), vp.clone()
        ws = api.new_workspace(cfg, T, table.shape[1], mode=mode)
        if ctx is None:
            y = api.layer_prefill(cfg, packed, x, pos, B, S, kpd, vpd, td, workspace=ws, mode=mode)
        else:
            y = api.layer_decode_step(cfg, packed, x, kpd, vpd, td, ctx, workspace=ws, mode=mode)
        return y, ws, (kpd, vpd)

    _assert_same(*_both_modes(run), cfg, T, table.shape[1], name)


def test_step_by_step_rejects_unknown_mode():
    d, W, Wn, table, kp, vp, cfg, packed = _tiny(131, 8, 1, 0)
    with pytest.raises(api.LayerError):
        api.layer_prefill(cfg, packed, synth.make_x(8, d.hidden, seed=1).to(DEV),
                          synth.prefill_positions(1, 8).to(DEV), 1, 8, kp.to(DEV), vp.to(DEV), table.to(DEV),
                          workspace=api.new_workspace(cfg, 8, table.shape[1]), mode=7)
