"""The seeded input generator: determinism, counter addressing, bf16 rounding."""
import math

import numpy as np
import pytest
import torch

import synth


def test_splitmix64_first_outputs_match_the_published_sequence():
    """SplitMix64 seeded with 0 starts 0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4,
    0x06C45D188009454F (the reference sequence of the generator's authors)."""
    # with key(stream) replaced by a 0 state, bits(c) is the c-th output
    with np.errstate(over="ignore"):
        c = np.arange(3, dtype=np.uint64)
        out = synth._mix(np.uint64(0) + (c + np.uint64(1)) * synth.GOLDEN)
    assert [int(x) for x in out] == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]


def test_streams_are_deterministic_and_counter_addressed():
    a = synth.normal(7, 5000)
    b = synth.normal(7, 5000)
    np.testing.assert_array_equal(a, b)
    # any window can be produced on its own
    np.testing.assert_array_equal(synth.normal(7, 100, start=1234), a[1234:1334])
    assert not np.array_equal(synth.normal(8, 100), a[:100])


def test_chunking_does_not_change_values(monkeypatch):
    a = synth.tensor(3, (3, 1000), "bf16")
    monkeypatch.setattr(synth, "CHUNK", 97)
    b = synth.tensor(3, (3, 1000), "bf16")
    np.testing.assert_array_equal(a, b)


def test_normal_moments():
    x = synth.normal(1, 1 << 20)
    assert abs(x.mean()) < 5e-3
    assert abs(x.std() - 1.0) < 5e-3
    # fourth moment of a standard normal is 3
    assert abs((x ** 4).mean() - 3.0) < 0.05


def test_bf16_rounding_is_round_to_nearest_even():
    rng = np.random.default_rng(0)
    x = (rng.standard_normal(100000) * np.exp(rng.uniform(-20, 20, 100000))).astype(np.float32)
    # exact ties: 1 + 2^-8 rounds down to 1 (even), 1 + 3 * 2^-8 rounds up
    x = np.concatenate([x, np.float32([1 + 2 ** -8, 1 + 3 * 2 ** -8, -(1 + 2 ** -8)])])
    ours = synth.round_to_bf16(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).to(torch.float32).numpy()
    np.testing.assert_array_equal(ours, ref)
    assert ours[-3] == 1.0 and ours[-2] == 1 + 2 ** -6 and ours[-1] == -1.0


def test_workload_shapes_and_counts():
    w = synth.WORKLOADS["multihead"]
    assert w.shape == (4, 32, 4096, 128)
    assert w.flops == 4 * 4 * 32 * 4096 ** 2 * 128
    assert w.scale == pytest.approx(1 / math.sqrt(128))
    c = synth.WORKLOADS["causal"]
    assert c.causal and c.flops == 2 * 32 * 16384 ** 2 * 128
    p = synth.WORKLOADS["peaked"]
    assert p.qk_mult == 4.0 and p.dtype == "bf16"
    assert synth.WORKLOADS["large_d"].dtype == "fp32"


def test_peaked_inputs_are_four_times_bf16_values():
    w = synth.WORKLOADS["peaked"].scaled(H=1, N=64)
    q, k, v = w.inputs()
    base = synth.tensor(3 * w.seed, w.shape, "bf16")
    np.testing.assert_array_equal(q, 4.0 * base)
    np.testing.assert_array_equal(synth.round_to_bf16(q), q)
    np.testing.assert_array_equal(synth.round_to_bf16(v), v)
