"""The seeded input generators: deterministic, and independent between tensors."""
import numpy as np
import torch

from transformer_decoder_layer_llama_gb300 import synth


def test_same_seed_same_bytes():
    a = synth.make_weights(synth.DIMS_TINY, 0.02, seed=3)
    b = synth.make_weights(synth.DIMS_TINY, 0.02, seed=3)
    for k in a:
        assert torch.equal(a[k], b[k])


def test_streams_do_not_alias_across_tensors_or_seeds():
    # an input drawn with any small seed must not repeat a weight row of any small seed
    d = synth.DIMS_TINY
    rows = []
    for s in range(8):
        W = synth.make_weights(d, 1.0, seed=s)
        rows += [W[k][:4].float() for k in ("w_qkv", "w_gate", "w_up")]
        rows.append(W["w_down"][:4, :256].float())
    rows = torch.cat(rows)
    for s in range(40):
        x = synth.make_x(4, d.hidden, seed=s).float()
        c = (x @ rows.T) / (x.norm(dim=1, keepdim=True) * rows.norm(dim=1)[None])
        assert c.abs().max() < 0.5, s


def test_block_table_is_a_partial_permutation():
    t, nb = synth.make_block_table([5, 40, 17], 16, seed=1, extra_blocks=3)
    used = t[t >= 0].numpy()
    assert nb == 1 + 3 + 2 + 3 and len(np.unique(used)) == len(used) == 6
    assert (t[0, 1:] == -1).all() and (t[1, :3] >= 0).all()


def test_slot_mapping_distinct_with_skips():
    s = synth.make_slot_mapping(50, 64, seed=2, n_skip=5).numpy()
    assert (s == -1).sum() == 5
    v = s[s >= 0]
    assert len(np.unique(v)) == len(v) and v.max() < 64
