"""CPU checks of the seeded input generators that the tests, the bench and
the smoke run share: reproducible per seed, the stated distributions, and
group sizes that always sum to the row count."""
import numpy as np
import pytest
import torch

from grouped_gemm_top_gb300 import synth


def test_same_seed_same_draws():
    a = synth.make_normal_bf16((300, 64), 11)
    b = synth.make_normal_bf16((300, 64), 11)
    assert torch.equal(a, b)
    assert not torch.equal(a, synth.make_normal_bf16((300, 64), 12))


def test_normal_draws_have_the_stated_moments():
    x = synth.make_normal_bf16((512, 512), 3, std=0.02).float()
    assert abs(x.mean().item()) < 1e-3
    assert abs(x.std().item() - 0.02) < 1e-3
    z = synth.make_logits(4096, 64, seed=5)
    assert z.dtype == torch.float32 and abs(z.mean().item()) < 0.01 and abs(z.std().item() - 1.0) < 0.01


def test_zipf_bias_is_a_permuted_log_rank():
    E, s = 64, 1.2
    bias = synth.zipf_bias(E, s, seed=0)
    ranks = np.exp(-bias.astype(np.float64) / s)
    assert np.allclose(np.sort(ranks), np.arange(1, E + 1), rtol=1e-5)
    logits = synth.make_logits(8, E, seed=0, zipf_s=s) - synth.make_logits(8, E, seed=0)
    assert np.allclose(logits.numpy(), np.broadcast_to(bias, (8, E)), atol=1e-6)


@pytest.mark.parametrize("G,M,alpha", [(8, 16384, 0.3), (256, 65536, 0.3), (64, 1000, 1.0), (5, 0, 0.3)])
def test_dirichlet_group_sizes_sum_to_m(G, M, alpha):
    m = synth.dirichlet_group_sizes(G, M, alpha, seed=2)
    assert m.shape == (G,) and m.dtype == np.int64 and (m >= 0).all() and int(m.sum()) == M
    assert np.array_equal(m, synth.dirichlet_group_sizes(G, M, alpha, seed=2))


def test_layer_inputs_shapes_and_shared_experts_last():
    inp = synth.make_layer_inputs(16, 128, 4, 64, n_shared=1)
    assert inp["logits"].shape == (16, 4) and inp["x"].shape == (16, 128) and inp["dout"].shape == (16, 128)
    assert inp["W1"].shape == (5, 128, 128) and inp["W2"].shape == (5, 64, 128)
    # the routed experts' weights do not depend on the number of shared experts
    base = synth.make_layer_inputs(16, 128, 4, 64)
    assert torch.equal(inp["W1"][:4], base["W1"]) and torch.equal(inp["W2"][:4], base["W2"])
