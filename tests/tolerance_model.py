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

Run:  python tests/tolerance_model.py llama2_7b_decode [llama2_7b_prefill ...]
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


def model_layer(d, W, x, pos, seqs, Kc, Vc):
    """float32/BF16 model of one layer call; Kc/Vc: per-sequence contiguous caches
    [Hkv, capacity, head_dim] (float32 holding BF16 values), updated in place."""
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
    for t in range(T):
        Kc[seqs[t]][:, pos[t]] = k[t]
        Vc[seqs[t]][:, pos[t]] = v[t]
    o = torch.zeros(T, Hq, dh)
    sl2 = (1 / math.sqrt(dh)) * 1.4426950408889634
    for t in range(T):
        n = pos[t] + 1
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


def spread(name, seed=21):
    wl = synth.WORKLOADS[name]
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
        kp, vp = synth.make_pool(nb, d, seed + 3)
        x = synth.make_x(B, d.hidden, seed + 4)
        ko, vo = bits(kp), bits(vp)
        Kc = [torch.from_numpy(O.gather_cache(ko, table[i].numpy(), int(ctx[i]))).float() for i in range(B)]
        Vc = [torch.from_numpy(O.gather_cache(vo, table[i].numpy(), int(ctx[i]))).float() for i in range(B)]
        pos = (ctx - 1).tolist()
        seqs = list(range(B))
        ref = O.layer_decode_step(d, Wn, x.float().numpy().astype(np.float64), ko, vo, table.numpy(),
                                  ctx.numpy())
    y = model_layer(d, W, x, pos, seqs, Kc, Vc).double().numpy()
    err = np.abs(y - ref)
    tol = 1e-2 + 1e-2 * np.abs(ref)
    return {"workload": name, "elements": int(err.size), "rms_err": float(np.sqrt((err ** 2).mean())),
            "max_err": float(err.max()), "worst_over_tol": float((err / tol).max()),
            "frac_outside": float((err > tol).mean())}


if __name__ == "__main__":
    torch.set_num_threads(os.cpu_count() or 1)
    for n in sys.argv[1:] or ["llama2_7b_decode"]:
        print(spread(n), flush=True)
