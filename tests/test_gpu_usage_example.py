"""The usage example a user starts from (the same lines as the README's): a 7B
layer prefill of 2048 tokens into a fresh paged pool, then one decode step, through
the Python binding (GPU)."""
import pytest
import torch


@pytest.mark.gpu
def test_usage_example_runs():
    from transformer_decoder_layer_llama_gb300 import api, synth

    d = synth.LayerDims(hidden=4096, n_heads=32, n_kv_heads=32, head_dim=128,
                        intermediate=11008, block_size=128)
    cfg = api.make_config(d, max_position=8192)
    W = {k: v.cuda() for k, v in synth.make_weights(d, 0.02, seed=0).items()}
    packed = api.pack_weights(cfg, W)
    k_pool = torch.zeros(64, 32, 128, 128, dtype=torch.bfloat16, device="cuda")
    v_pool = torch.zeros_like(k_pool)
    table = torch.arange(17, dtype=torch.int32, device="cuda").view(1, 17)
    x = torch.randn(2048, 4096, device="cuda").bfloat16()
    pos = torch.arange(2048, dtype=torch.int32, device="cuda")
    y = api.layer_prefill(cfg, packed, x, pos, 1, 2048, k_pool, v_pool, table)
    ctx = torch.tensor([2049], dtype=torch.int32, device="cuda")
    y1 = api.layer_decode_step(cfg, packed, torch.randn(1, 4096, device="cuda").bfloat16(),
                               k_pool, v_pool, table, ctx)
    torch.cuda.synchronize()
    assert y.shape == (2048, 4096) and y1.shape == (1, 4096)
    assert torch.isfinite(y.float()).all() and torch.isfinite(y1.float()).all()
    # the prefill wrote the 2048 positions of blocks 0-15 and the decode step position 2048
    assert bool((k_pool[:16].float().abs().sum(dim=(1, 2, 3)) > 0).all())
    assert float(k_pool[16, :, 0].float().abs().sum()) > 0
    assert float(k_pool[16, :, 1:].float().abs().sum()) == 0
