"""The seeded input generator follows its published definitions."""
import numpy as np

from bwd_qwen3_layer_gb300 import synth

G = 0x9E3779B97F4A7C15


def test_splitmix64_reference_outputs():
    # first three outputs of splitmix64 started from state 0
    assert synth._mix_int(G) == 0xE220A8397B1DCDAF
    assert synth._mix_int(2 * G) == 0x6E789E6AA1B965F4
    assert synth._mix_int(3 * G) == 0x06C45D188009454F
    # the vectorised finaliser agrees with the scalar one
    idx = np.arange(1, 6, dtype=np.uint64)
    z = synth._mix_arr(idx * np.uint64(G))
    assert [int(x) for x in z] == [synth._mix_int(i * G) for i in range(1, 6)]


def test_fnv1a64_reference_outputs():
    assert synth.fnv1a64("") == 0xCBF29CE484222325
    assert synth.fnv1a64("a") == 0xAF63DC4C8601EC8C


def test_streams_are_counter_based_and_distributed():
    a = synth.uniform(3, "x", 1000)
    b = synth.uniform(3, "x", 400, start=600)
    assert np.array_equal(a[600:], b)
    assert not np.array_equal(a, synth.uniform(4, "x", 1000))
    n = synth.normal(0, "n", (200_000,))
    assert abs(n.mean()) < 0.01 and abs(n.std() - 1) < 0.01
    r = synth.randint(0, "r", (100_000,), 7)
    assert r.min() == 0 and r.max() == 6
    assert np.all(np.abs(np.bincount(r) / 1e5 - 1 / 7) < 0.01)


def test_round_bf16():
    x = np.array([1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -9, -3.14159, 65504.0, 1e-30])
    y = synth.round_bf16(x)
    assert y[0] == 1.0
    assert y[1] == 1.0                  # tie -> even
    assert y[2] == 1.0 + 2 ** -7        # above half -> up
    assert abs(y[3] + 3.14159) < 2 ** -7 * 4
    # result is representable: low 16 bits of the fp32 pattern are zero
    assert np.all(y.astype(np.float32).view(np.uint32) & 0xFFFF == 0)
