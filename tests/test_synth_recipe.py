"""The seeded input generator follows the stated recipe: Qwen3-4B-like heads,
Q and V ~ N(0, 1), a per-channel key mean ~ N(0, std 2) with 4 outlier
channels per KV head (mean and noise x 20), per-tensor scales that keep
every block scale in range, the page/tail split of the hybrid cache, and the
batch's log-uniform lengths."""
import numpy as np
import torch

from nvfp4_kv_cache_bd_gb300 import synth


def sylvester(n=128):
    h = np.array([[1.0]])
    while h.shape[0] < n:
        h = np.block([[h, h], [h, -h]])
    return h / np.sqrt(n)


def test_key_mean_has_four_outliers_per_head():
    mu, mask = synth.key_mean(8, 0)
    assert mu.shape == (8, 128) and mask.shape == (8, 128)
    assert mask.sum(dim=1).tolist() == [4] * 8
    normal = mu[~mask]
    assert 1.8 < float(normal.std()) < 2.2 and abs(float(normal.mean())) < 0.3
    ratio = float(mu[mask].abs().mean()) / float(normal.abs().mean())
    assert 8.0 < ratio < 40.0


def test_keys_and_values_follow_the_recipe():
    mu, mask = synth.key_mean(8, 3)
    k, v = synth.keys_values(4096, 8, 3, mu=mu, mask=mask)
    assert k.dtype == torch.bfloat16 and v.dtype == torch.bfloat16 and k.shape == (4096, 8, 128)
    noise = k.float() - mu.unsqueeze(0)
    m = mask.unsqueeze(0).expand_as(noise)
    assert 0.95 < float(noise[~m].std()) < 1.05
    assert 18.0 < float(noise[m].std()) < 22.0
    assert 0.97 < float(v.float().std()) < 1.03 and abs(float(v.float().mean())) < 0.01
    q = synth.query(2, 32, 3)
    assert q.shape == (2, 32, 128) and 0.9 < float(q.float().std()) < 1.1


def test_generator_is_seeded():
    a = synth.keys_values(64, 8, 5)
    b = synth.keys_values(64, 8, 5)
    c = synth.keys_values(64, 8, 6)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])
    assert not torch.equal(a[0], c[0])
    assert torch.equal(synth.query(1, 32, 5), synth.query(1, 32, 5))


def test_gscales_bound_every_transformed_key_and_value():
    mu, mask = synth.key_mean(8, 1)
    k, v = synth.keys_values(512, 8, 1, mu=mu, mask=mask)
    gk, gv = synth.gscales(k, v, mu, True, True)
    assert gv == np.float32(float(v.float().abs().max()) / 2688.0)
    # centered and rotated keys: every coordinate stays within 2688 * g_K
    x = (k.double() - mu.double().unsqueeze(0)).numpy().reshape(-1, 128)
    y = x @ sylvester().T
    assert np.abs(y).max() <= 2688.0 * gk * (1 + 1e-6)
    # without rotation the bound is the plain maximum
    gk2, _ = synth.gscales(k, v, mu, False, True)
    assert np.isclose(2688.0 * gk2, np.abs(x).max(), rtol=1e-6)


def test_split_tokens_matches_the_workloads():
    assert synth.split_tokens(4096) == (16, 31, 112)
    assert synth.split_tokens(32768) == (16, 255, 112)
    assert synth.split_tokens(131072) == (16, 1023, 112)
    assert synth.split_tokens(0) == (0, 0, 0)
    assert synth.split_tokens(16) == (16, 0, 0)
    assert synth.split_tokens(143) == (16, 0, 127)
    assert synth.split_tokens(144) == (16, 1, 0)


def test_batch_lengths_are_log_uniform_and_seeded():
    lens = synth.log_uniform_lengths(32, 1024, 65536, 0)
    assert lens == synth.log_uniform_lengths(32, 1024, 65536, 0)
    assert len(lens) == 32 and all(1024 <= x <= 65536 for x in lens)
    assert sum(lens) == 417192     # the batch the benchmark reports
    logs = np.log(np.array(synth.log_uniform_lengths(4096, 1024, 65536, 1), dtype=np.float64))
    # log-uniform: the logs are uniform on [ln 1024, ln 65536]
    u = (logs - np.log(1024)) / (np.log(65536) - np.log(1024))
    assert abs(u.mean() - 0.5) < 0.02 and abs(u.var() - 1 / 12) < 0.01


def test_page_permutation_is_a_permutation():
    p = synth.page_permutation(1023, 0)
    assert p.dtype == torch.int32 and sorted(p.tolist()) == list(range(1023))
    assert not torch.equal(p, torch.arange(1023, dtype=torch.int32))
