"""The seeded input recipe: determinism and the stated shapes/distributions."""
import torch

import fa_inputs as inp


def test_same_seed_same_tensors():
    a = inp.dense(1, 2, 33, 64, seed=4, causal=True)
    b = inp.dense(1, 2, 33, 64, seed=4, causal=True)
    assert torch.equal(a.q, b.q) and torch.equal(a.k, b.k) and torch.equal(a.v, b.v)
    c = inp.dense(1, 2, 33, 64, seed=5, causal=True)
    assert not torch.equal(a.q, c.q)


def test_config_shapes():
    c1 = inp.config1()
    assert c1.q.dtype == torch.float32 and tuple(c1.q.shape) == (1, 1, 256, 64)
    assert c1.scale == 1 / 8 and not c1.causal
    c2 = inp.config2()
    assert c2.q.dtype == torch.bfloat16 and tuple(c2.q.shape) == (4, 16, 2048, 128)
    assert c2.causal


def test_varlen_lengths_recipe():
    for D in (64, 128):
        c = inp.config5(D)
        lens = c.meta["lens"]
        assert sum(lens) == 65536 == c.q.shape[0]
        assert all(1 <= n <= 8192 for n in lens)
        assert c.cu_seqlens[0] == 0 and c.cu_seqlens[-1] == 65536
        assert tuple(c.q.shape[1:]) == (16, D)
    # the same seed draws the same lengths at both head dims
    assert inp.config5(64).meta["lens"] == inp.config5(128).meta["lens"]


def test_decode_lengths_recipe():
    g = torch.Generator().manual_seed(4)
    lens = torch.randint(1024, 32769, (64,), generator=g).tolist()
    c = inp.decode(2, 1, 64, seed=4, num_splits=16, lens=[3, 7])
    assert c.cu_seqlens_k.tolist() == [0, 3, 10] and tuple(c.k_cache.shape) == (10, 1, 64)
    assert all(1024 <= n <= 32768 for n in lens)


def test_config3_scores_are_large():
    # std 3 for q and k: scaled scores have std ~ 9 (128 products of variance 81)
    c = inp.dense(1, 1, 64, 128, seed=3, causal=True, qk_std=3.0)
    s = (c.q.float() @ c.k.float().transpose(-1, -2)) * c.scale
    assert 6.0 < float(s.std()) < 12.0
