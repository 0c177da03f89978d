"""How far a correct BF16 tensor-core implementation of the layer drifts from the oracle.

This is a CPU model of the arithmetic the CUDA path performs -- float32
accumulation of BF16 operands, BF16 rounding of every MatMul operand and of the
KV cache, a float32 residual stream, attention probabilities carried with about
16 bits -- written in plain PyTorch float32 (it shares no code with the CUDA
library and is not the oracle).  Comparing it with the float64 oracle shows the
spread that the oracle/GPU comparison must tolerate: rare 1-ulp differences in
the rounding of a BF16 operand (the model and the oracle round values that
differ in their last float32 bits) move the next MatMul's output slightly,
which flips further roundings downstream.  At the 7B prefill size this cascade
alone leaves a small fraction of output elements outside the per-element bound
1e-2 + 1e-2*|ref|, whatever the summation order.

Run:  python tests/tolerance_model.py llama2_7b_decode [llama2_7b_prefill llama2_7b_decode_int8kv ...]
"""
import math
import os
import sys

import numpy as np
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

from oracle import llama_layer as O  # noqa: E402
from transformer_decoder_layer_llama_gb300 import synth  # noqa: E402

BF = torch.bfloat16


def _b(t):
    return t.to(BF).float()


def _rope32(u, pos, theta, d):
    half = d // 2
    inv = theta ** (-(2.0 * np.arange(half)) / d)
    ang = np.asarray(pos, np.float64)[:, None] * inv[None, :]
    c = torch.from_numpy(np.cos(ang)).float()[:, None, :]
    s = torch.from_numpy(np.sin(ang)).float()[:, None, :]
    u1, u2 = u[..., :half], u[..., half:]
    return torch.cat([u1 * c - u2 * s, u2 * c + u1 * s], -1)


def _quant32(rows):
    """INT8 codes (as float32) and float32 scales of rows [..., d]: absmax / 127, nearest code."""
    amax = rows.abs().amax(-1)
    scale = amax / 127.0
    safe = torch.where(scale > 0, scale, torch.ones_like(scale))
    return torch.round(rows / safe[..., None]).clamp(-127, 127), scale


def model_layer(d, W, x, pos, seqs, Kc, Vc, q8=None, p_fp16=True):
    """float32/BF16 model of one layer call; Kc/Vc: per-sequence contiguous caches
    [Hkv, capacity, head_dim] (float32 holding BF16 values), updated in place.
    q8: for an INT8 cache, per-sequence (K codes, K scales, V codes, V scales) float32
    [Hkv, capacity(, head_dim)], updated in place; attention then runs as the INT8 kernel
    does: scores from the codes times the K scale, each probability times its key's V scale
    entering P V as two FP16 parts under an exponent base at the largest such weight
    (p_fp16), or exactly."""
    Hq, Hkv, dh = d.n_heads, d.n_kv_heads, d.head_dim
    G = Hq // Hkv
    T = x.shape[0]
    xf = x.float()
    r = 1 / torch.sqrt((xf * xf).mean(1, keepdim=True) + d.rms_eps)
    xh = _b(xf * r * W["g_attn"])
    qkv = xh @ W["w_qkv"].float().T
    q = _b(_rope32(qkv[:, :Hq * dh].reshape(T, Hq, dh), pos, d.rope_theta, dh))
    k = _b(_rope32(qkv[:, Hq * dh:(Hq + Hkv) * dh].reshape(T, Hkv, dh), pos, d.rope_theta, dh))
    v = _b(qkv[:, (Hq + Hkv) * dh:].reshape(T, Hkv, dh))
    if q8 is None:
        for t in range(T):
            Kc[seqs[t]][:, pos[t]] = k[t]
            Vc[seqs[t]][:, pos[t]] = v[t]
    else:
        for t in range(T):
            kc, ks, vc, vs = q8[seqs[t]]
            kc[:, pos[t]], ks[:, pos[t]] = _quant32(k[t])
            vc[:, pos[t]], vs[:, pos[t]] = _quant32(v[t])
    o = torch.zeros(T, Hq, dh)
    sl2 = (1 / math.sqrt(dh)) * 1.4426950408889634
    for t in range(T):
        n = pos[t] + 1
        if q8 is not None:
            kc, ks, vc, vs = (c[:, :n] for c in q8[seqs[t]])
            for h in range(Hq):
                s = (kc[h // G] @ q[t, h]) * ks[h // G] * sl2
                p = torch.exp2(s - s.max())
                if p_fp16:
                    # base at the largest weight p * v_scale; the weight in two FP16 parts
                    lw = s + torch.log2(vs[h // G]).clamp(min=-40)
                    p = torch.exp2(s - lw.max())
                    pv = p * vs[h // G]
                    hi = pv.half().float()
                    pv = hi + (pv - hi).half().float()
                else:
                    pv = p * vs[h // G]
                o[t, h] = (pv @ vc[h // G]) / p.sum()
            continue
        K, V = Kc[seqs[t]][:, :n], Vc[seqs[t]][:, :n]
        for h in range(Hq):
            s = (K[h // G] @ q[t, h]) * sl2
            p = torch.exp2(s - s.max())
            ph = _b(p)
            pl = _b(p - ph)
            o[t, h] = ((ph @ V[h // G]) + (pl @ V[h // G])) / p.sum()
    o = _b(o)
    h1 = xf + o.reshape(T, -1) @ W["w_o"].float().T
    r2 = 1 / torch.sqrt((h1 * h1).mean(1, keepdim=True) + d.rms_eps)
    hh = _b(h1 * r2 * W["g_ffn"])
    a = _b(torch.nn.functional.silu(hh @ W["w_gate"].float().T) * (hh @ W["w_up"].float().T))
    return _b(h1 + a @ W["w_down"].float().T)


def spread(name, seed=21, p_fp16=True):
    q8 = name.endswith("_int8kv")
    wl = synth.WORKLOADS[name.replace("_int8kv", "")]
    d = wl.dims
    W = synth.make_weights(d, wl.w_std, seed)
    Wn = {k: v.float().numpy().astype(np.float64) for k, v in W.items()}
    bits = lambda t: t.contiguous().view(torch.int16).numpy().view(np.uint16).copy()
    if wl.prefill_len:
        B, S = wl.batch, wl.prefill_len
        T = B * S
        table, nb = synth.make_block_table([S] * B, d.block_size, seed + 2, extra_blocks=2)
        kp, vp = synth.make_pool(nb, d, seed + 3, fill="sentinel")
        x = synth.make_x(T, d.hidden, seed + 4)
        pos = synth.prefill_positions(B, S).tolist()
        seqs = [t // S for t in range(T)]
        Kc = [torch.zeros(d.n_kv_heads, S, d.head_dim) for _ in range(B)]
        Vc = [torch.zeros(d.n_kv_heads, S, d.head_dim) for _ in range(B)]
        ref = O.layer_prefill(d, Wn, x.float().numpy().astype(np.float64), np.array(pos), B, S,
                              bits(kp), bits(vp), table.numpy())
    else:
        B = wl.batch
        ctx = synth.make_context_lens(B, wl.ctx_lo, wl.ctx_hi, seed + 1)
        table, nb = synth.make_block_table(ctx.tolist(), d.block_size, seed + 2, extra_blocks=2)
        x = synth.make_x(B, d.hidden, seed + 4)
        pos = (ctx - 1).tolist()
        seqs = list(range(B))
        if q8:
            kc, vc, ks, vs = synth.make_pool_q8(nb, d, seed + 3)
            ko, vo = O.QuantPool(kc.numpy().copy(), ks.numpy().copy()), O.QuantPool(vc.numpy().copy(), vs.numpy().copy())

            def gather(t, i):
                blocks = table[i, :-(-int(ctx[i]) // d.block_size)].long()
                return torch.cat(list(t[blocks].float()), dim=1)
            quant = [tuple(gather(t, i) for t in (kc, ks, vc, vs)) for i in range(B)]
            Kc = Vc = None
        else:
            kp, vp = synth.make_pool(nb, d, seed + 3)
            ko, vo = bits(kp), bits(vp)
            Kc = [torch.from_numpy(O.gather_cache(ko, table[i].numpy(), int(ctx[i]))).float() for i in range(B)]
            Vc = [torch.from_numpy(O.gather_cache(vo, table[i].numpy(), int(ctx[i]))).float() for i in range(B)]
            quant = None
        ref = O.layer_decode_step(d, Wn, x.float().numpy().astype(np.float64), ko, vo, table.numpy(),
                                  ctx.numpy())
    y = model_layer(d, W, x, pos, seqs, Kc, Vc, q8=quant if not wl.prefill_len else None,
                    p_fp16=p_fp16).double().numpy()
    err = np.abs(y - ref)
    tol = 1e-2 + 1e-2 * np.abs(ref)
    return {"workload": name + ("" if not q8 or p_fp16 else " (exact P)"), "elements": int(err.size), "rms_err": float(np.sqrt((err ** 2).mean())),
            "max_err": float(err.max()), "worst_over_tol": float((err / tol).max()),
            "frac_outside": float((err > tol).mean())}


if __name__ == "__main__":
    torch.set_num_threads(os.cpu_count() or 1)
    for n in sys.argv[1:] or ["llama2_7b_decode"]:
        print(spread(n), flush=True)
        if n.endswith("_int8kv"):
            print(spread(n, p_fp16=False), flush=True)
