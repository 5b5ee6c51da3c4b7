"""The seeded input generators: deterministic, thread-count independent, and
drawing what the recipe says."""
import numpy as np
import pytest
import torch

import workloads


def test_deterministic_and_thread_independent():
    s = workloads.custom(300, 96, 1000, dtype="bf16", ignore_frac=0.1, seed=3)
    a = workloads.generate(s, threads=1)
    b = workloads.generate(s, threads=4)
    np.testing.assert_array_equal(a.x, b.x)
    np.testing.assert_array_equal(a.W, b.W)
    np.testing.assert_array_equal(a.t, b.t)
    c = workloads.generate(workloads.custom(300, 96, 1000, dtype="bf16", ignore_frac=0.1, seed=4))
    assert not np.array_equal(a.W, c.W)


def test_blocks_cross_block_boundary(monkeypatch):
    monkeypatch.setattr(workloads, "BLOCK", 1000)
    s = workloads.custom(37, 64, 50, dtype="fp32")
    a = workloads.generate(s, threads=1)
    b = workloads.generate(s, threads=3)
    np.testing.assert_array_equal(a.x, b.x)
    # block 1 of x starts at flat element 1000 with its own stream
    g = workloads._stream(0, 0, 1)
    np.testing.assert_array_equal(a.x.reshape(-1)[1000:1010], g.standard_normal(10, dtype=np.float32))


def test_bf16_rounding_is_round_to_nearest_even():
    g = np.random.default_rng(0)
    f = (g.standard_normal(100000) * 10.0 ** g.integers(-8, 8, 100000)).astype(np.float32)
    # exact ties: low 16 bits = 0x8000
    ties = (g.integers(0, 0x7F00, 1000, dtype=np.uint32) << np.uint32(16)) | np.uint32(0x8000)  # finite only
    f = np.concatenate([f, ties.view(np.float32)])
    out = np.empty(f.shape, np.uint16)
    workloads.round_f32_to_bf16_bits(f.copy(), out)
    ref = torch.from_numpy(f).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(out, ref)
    back = workloads.bf16_bits_to_f32(out)
    np.testing.assert_array_equal(back, torch.from_numpy(f).to(torch.bfloat16).float().numpy())


def test_value_distributions():
    w = workloads.make("small_bf16", N=4096, V=5000, H=256)
    x = w.x_f64()
    W = w.W_f64()
    assert abs(x.mean()) < 0.01 and abs(x.std() - 1.0) < 0.01
    assert abs(W.std() - 0.02) < 0.0005
    assert (w.t == -100).sum() == 4096 // 10
    tv = w.t[w.t != -100]
    assert tv.min() >= 0 and tv.max() < 5000


def test_zipf_targets_and_exact_ignore_count():
    s = workloads.spec("llama3_bf16", N=20000, H=8)
    t = workloads.make_targets(s)
    assert (t == -100).sum() == 20000 // 20
    tv = t[t != -100]
    assert tv.min() >= 0 and tv.max() < s.V
    # P(k=1) = 1/H_{V,1.1}; the generalized harmonic number for V=128256
    k = np.arange(1, s.V + 1, dtype=np.float64)
    p1 = 1.0 / np.sum(k ** -1.1)
    frac0 = np.mean(tv == 0)
    assert abs(frac0 - p1) < 4 * np.sqrt(p1 * (1 - p1) / len(tv))
    # rank order: token 0 more frequent than token 1 more frequent than token 9
    c = np.bincount(tv, minlength=10)
    assert c[0] > c[1] > c[9]


def test_named_configs_shapes():
    c = workloads.CONFIGS
    assert (c["tiny_fp32"].N, c["tiny_fp32"].H, c["tiny_fp32"].V, c["tiny_fp32"].chunk) == (256, 128, 4096, 64)
    assert (c["small_bf16"].N, c["small_bf16"].H, c["small_bf16"].V) == (2048, 1024, 32000)
    assert (c["llama3_bf16"].N, c["llama3_bf16"].H, c["llama3_bf16"].V) == (16384, 4096, 128256)
    assert (c["qwen3_bf16"].V, c["long_bf16"].N) == (151936, 131072)
    assert workloads.QWEN3_CHUNKS == (1024, 2048, 4096, 8192)


@pytest.mark.parametrize("name", ["tiny_fp32", "small_bf16"])
def test_small_configs_generate(name):
    w = workloads.make(name)
    assert w.x.shape == (w.N, w.H) and w.W.shape == (w.V, w.H) and w.t.shape == (w.N,)
    assert w.x.dtype == (np.float32 if w.spec.dtype == "fp32" else np.uint16)
