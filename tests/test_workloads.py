"""The seeded input generator: determinism, formats and routing recipe (CPU only)."""
import numpy as np

from workloads import configs, gen


def test_normal_is_deterministic_and_thread_independent(monkeypatch):
    a = gen.normal16((3, 1), (3, gen.CHUNK // 2 + 5), 0.02, "f16")
    monkeypatch.setattr(gen, "_threads", lambda: 1)
    b = gen.normal16((3, 1), (3, gen.CHUNK // 2 + 5), 0.02, "f16")
    assert a.dtype == np.float16 and np.array_equal(a.view(np.uint16), b.view(np.uint16))
    assert abs(float(a.astype(np.float64).std()) - 0.02) < 1e-3
    c = gen.normal16((3, 2), (3, 100), 0.02, "f16")
    assert not np.array_equal(a[:, :100], c)


def test_bf16_storage_is_rne_of_float32():
    x = np.array([1.0, 1 + 2 ** -8, 1 + 3 * 2 ** -8, -3.0, 2 ** -10], dtype=np.float32)
    bits = gen.f32_to_bf16_bits(x)
    assert bits.tolist() == [0x3F80, 0x3F80, 0x3F82, 0xC040, 0x3A80]
    assert gen.bf16_bits_to_f32(bits).tolist() == [1.0, 1.0, 1 + 2 ** -6, -3.0, 2 ** -10]


def test_integers_are_exact_in_both_formats():
    for dt in gen.DTYPES:
        v = gen.to_f32(gen.integers16(4, (1000,), -2, 2, dt), dt)
        assert set(np.unique(v).tolist()) <= {-2.0, -1.0, 0.0, 1.0, 2.0}


def test_routing_recipe():
    ids, w = gen.routing(5, 4096, 8, 2)
    assert ids.shape == (4096, 2) and ids.dtype == np.int32
    assert np.all(ids[:, 0] != ids[:, 1])
    assert np.allclose(w.sum(axis=1), 1.0, atol=1e-6) and np.all(w[:, 0] >= w[:, 1])
    counts = np.bincount(ids.reshape(-1), minlength=8)
    assert counts[0] == counts.max() and counts[0] > 2 * counts[7]   # Zipf-skewed load
    ids2, _ = gen.routing(5, 64, 8, 2, force_empty=(3,))
    assert not np.any(ids2 == 3)


def test_config_shapes():
    c = configs.small(configs.CONFIGS["rs_mlp1"], M=64, N=32, K=128)
    As, Bs = configs.rs_inputs(c)
    assert [a.shape for a in As] == [(64, 16)] * 8 and [b.shape for b in Bs] == [(16, 32)] * 8
    c = configs.small(configs.CONFIGS["ag_mlp0"], M=64, N=64, K=32)
    xs, ws = configs.ag_inputs(c)
    assert [x.shape for x in xs] == [(8, 32)] * 8 and [w.shape for w in ws] == [(32, 8)] * 8
    m = configs.small(configs.CONFIGS["moe"], T=16, H=8, F=16)
    d = configs.moe_inputs(m)
    assert d["w1_shards"][0].shape == (8, 8, 2) and d["w2_shards"][0].shape == (8, 2, 8)
    assert d["h_shards"][0].shape == (32, 2) and d["x_shards"][0].dtype == np.uint16
