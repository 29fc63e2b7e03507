"""The seeded input generator: published test vectors, determinism, recipes."""
import ctypes

import numpy as np

import datagen
from datagen import workloads
from conftest import golden


def test_splitmix64_and_fnv_vectors():
    g = golden("splitmix64.json")
    lib = datagen._load()
    got = [lib.gen_draw(0, i) for i in range(3)]
    assert got == [int(h, 16) for h in g["splitmix64_state0"]]
    lib.gen_fnv1a64.restype = ctypes.c_uint64
    lib.gen_fnv1a64.argtypes = [ctypes.c_char_p]
    for s, h in g["fnv1a64"].items():
        assert lib.gen_fnv1a64(s.encode()) == int(h, 16)


def test_normal_moments_and_thread_independence():
    a = datagen.normal(7, "t", (2_000_001,), "f64")
    assert abs(a.mean()) < 3e-3 and abs(a.std() - 1) < 3e-3
    # a prefix drawn alone equals the same prefix of a long (threaded) fill
    b = datagen.normal(7, "t", (1001,), "f64")
    assert np.array_equal(a[:1001], b)
    c = datagen.normal(7, "t", (2_000_001,), "f32")
    assert np.array_equal(c, a.astype(np.float32))


def test_bf16_rounding_nearest_even():
    # 1 + 2^-8 is a tie between 1 and 1 + 2^-7: rounds to even (1.0)
    x = np.array([1.0 + 2**-8, 1.0 + 3 * 2**-8, -2.5, 1e-40], np.float32)
    b = datagen.f32_to_bf16_bits(x)
    back = datagen.bf16_bits_to_f32(b)
    assert back[0] == 1.0 and back[1] == 1.0 + 2**-6 and back[2] == -2.5
    z = datagen.normal(3, "r", (100_000,), "bf16")
    f = datagen.normal(3, "r", (100_000,), "f32")
    assert np.array_equal(z, datagen.f32_to_bf16_bits(f))


def test_labels_exact_ignore_count():
    lab = datagen.labels(0, "x", 256, 1024, 0.05)
    assert (lab == -100).sum() == round(0.05 * 256)
    v = lab[lab != -100]
    assert v.min() >= 0 and v.max() < 1024
    lab2 = datagen.labels(3, "y", 8192, 128256, 0.10)
    assert (lab2 == -100).sum() == 819
    assert np.array_equal(lab2, datagen.labels(3, "y", 8192, 128256, 0.10))


def test_streams_keyed_by_name():
    a = datagen.normal(0, "a", (64,), "f32")
    b = datagen.normal(0, "b", (64,), "f32")
    c = datagen.normal(1, "a", (64,), "f32")
    assert not np.array_equal(a, b) and not np.array_equal(a, c)


def test_workload_recipes():
    t = workloads.tiny("f32")
    assert t["rmsnorm"].spec("x").shape == (256, 256)
    assert t["rope"].spec("q").shape == (2, 128, 4, 64)
    assert t["swiglu"].spec("gate").shape == (256, 688)
    assert t["linear_ce"].spec("W").shape == (1024, 256) and t["linear_ce"].spec("W").std == 0.02
    w = t["rmsnorm"].make("w")
    assert abs(w.mean() - 1) < 0.05 and 0.05 < w.std() < 0.15
    r = workloads.rmsnorm_rope_llama3()
    assert r["rope"].spec("k").shape == (4, 8192, 8, 128)
    q = workloads.qwen_chain(512)
    assert q["linear_ce"].params["V"] == 151936
