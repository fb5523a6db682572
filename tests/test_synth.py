"""The seeded input generator: SplitMix64 against its published first output,
distribution sanity, bf16 round-to-nearest-even against torch's conversion,
and the subnormal planting recipe."""
import math

import numpy as np
import torch

from implicit_gemm_conv2d_gb300 import synth


def test_splitmix64_first_output_from_state_zero():
    # SplitMix64 (Steele, Lea & Flood 2014) started from state 0 first returns
    # 0xE220A8397B1DCDAF; the counter form mixes state + GAMMA.
    z = synth._mix(np.array([synth.GAMMA], dtype=np.uint64))[0]
    assert int(z) == 0xE220A8397B1DCDAF


def test_counter_form_matches_sequential_generator():
    def seq(state, n):
        out = []
        for _ in range(n):
            state = (state + 0x9E3779B97F4A7C15) & (2**64 - 1)
            z = state
            z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & (2**64 - 1)
            z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & (2**64 - 1)
            out.append(z ^ (z >> 31))
        return out
    s0 = int(synth.stream_state(synth.SEED, 3))
    assert [int(v) for v in synth.splitmix64(synth.SEED, 3, 0, 50)] == seq(s0, 50)
    assert [int(v) for v in synth.splitmix64(synth.SEED, 3, 17, 5)] == seq(s0, 22)[17:]


def test_determinism_and_streams_differ():
    a = synth.conv_inputs(4, 3, 5, 11, 15, 5, 3)
    b = synth.conv_inputs(4, 3, 5, 11, 15, 5, 3)
    for k in a:
        assert a[k].tobytes() == b[k].tobytes()
    assert not np.array_equal(a["x"].reshape(-1)[:60], a["dy"].reshape(-1)[:60])


def test_bias_is_optional_and_its_own_stream():
    base = synth.conv_inputs(4, 3, 5, 11, 15, 5, 3)
    withb = synth.conv_inputs(4, 3, 5, 11, 15, 5, 3, need=("x", "w", "dy", "bias"))
    assert "bias" not in base and withb["bias"].shape == (5,)
    for k in base:  # asking for the bias changes none of the other tensors
        assert base[k].tobytes() == withb[k].tobytes()
    a = 1 / math.sqrt(3 * 25)
    assert np.all(np.abs(withb["bias"]) < a)
    assert not np.array_equal(withb["bias"], withb["w"].reshape(-1)[:5])
    bf = synth.conv_inputs(4, 3, 5, 11, 15, 5, 3, dtype="bf16", need=("bias",))["bias"]
    assert np.array_equal(bf, synth.to_dtype_values(withb["bias"].astype(np.float64), "bf16"))


def test_distributions():
    n = 1 << 20
    x = synth.normal(synth.SEED, 1, n)
    assert abs(x.mean()) < 5e-3 and abs(x.std() - 1) < 5e-3
    a = 1 / math.sqrt(59 * 25)
    w = synth.uniform_pm(synth.SEED, 2, n, a)
    assert w.min() >= -a and w.max() < a
    assert abs(w.mean()) < 2e-3 * a * 10 and abs(w.std() - a / math.sqrt(3)) < 1e-3 * a


def test_bf16_rounding_matches_torch():
    rng = np.random.default_rng(0)
    v = np.concatenate([rng.standard_normal(100000).astype(np.float32) * 10.0 ** rng.integers(-30, 30, 100000),
                        np.array([1.0 + 2**-8, 1.0 + 3 * 2**-8, -(1.0 + 2**-8), 3.4e38, 1e-40, -0.0],
                                 dtype=np.float32)]).astype(np.float32)
    ours = synth.round_bf16_bits(v)
    ref = torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)
    # ties go to even: 1 + 2^-8 sits halfway between 1 and 1 + 2^-7
    assert synth.bf16_bits_to_f32(synth.round_bf16_bits(np.array([1.0 + 2**-8], np.float32)))[0] == 1.0


def test_bf16_inputs_are_bf16_exact():
    d = synth.conv_inputs(2, 3, 4, 5, 5, 3, 1, dtype="bf16")
    for v in d.values():
        assert np.array_equal(synth.bf16_bits_to_f32(synth.round_bf16_bits(v)), v)


def test_subnormal_planting():
    d = synth.conv_inputs(64, 8, 4, 5, 5, 3, 1, subnormal=True)
    x = d["x"]
    tiny = (x != 0) & (np.abs(x) < np.float32(2.0**-126))
    frac = tiny.mean()
    assert 0.007 < frac < 0.013
    e = np.log2(np.abs(x[tiny]).astype(np.float64))
    assert np.all(e == np.round(e)) and e.min() >= -149 and e.max() < -127


def test_scale_is_exact_power_of_two():
    a = synth.conv_inputs(2, 3, 4, 5, 5, 3, 1)
    b = synth.conv_inputs(2, 3, 4, 5, 5, 3, 1, scale=0.125)
    assert np.array_equal(a["x"] * np.float32(0.125), b["x"])
    assert np.array_equal(a["dy"], b["dy"])
