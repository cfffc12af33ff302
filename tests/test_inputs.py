"""The seeded input recipe shared by both sides: 16-bit rounding, exact widening, the
seed rule and the shapes and scale of every workload.  Parity cannot catch a mistake
here (both sides would see the same wrong bits), so the recipe is pinned on its own."""

import numpy as np
import pytest
import torch

from exact_tiled_attention_27_gb300 import inputs as I


def _torch_bits(x32, dtype):
    t = torch.from_numpy(np.ascontiguousarray(x32, dtype=np.float32))
    t = t.to(torch.bfloat16 if dtype == "bf16" else torch.float16)
    return t.view(torch.int16).numpy().view(np.uint16)


def test_bf16_rounding_hand_values():
    one = np.float32(1.0)
    ulp = np.float32(2.0 ** -7)        # bf16 spacing just above 1
    vals = np.array([one, one + ulp / 2, one + 3 * ulp / 2, one + ulp / 4, one + 3 * ulp / 4,
                     -(one + ulp / 2), np.float32(3.0), np.float32(-0.0)], dtype=np.float32)
    want = np.array([0x3F80, 0x3F80, 0x3F82, 0x3F80, 0x3F81, 0xBF80, 0x4040, 0x8000], dtype=np.uint16)
    # ties go to the even mantissa: 1 + ulp/2 -> 1, 1 + 3 ulp/2 -> 1 + 2 ulp
    assert np.array_equal(I._round_f32_to_bf16_bits(vals), want)


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_rounding_matches_torch(dtype):
    rng = np.random.default_rng(5)
    x = (rng.standard_normal(200_000) * np.exp2(rng.integers(-20, 12, 200_000))).astype(np.float32)
    # exact ties for bf16: the low 16 bits are 0x8000
    ties = (rng.integers(0, 2 ** 15, 1000, dtype=np.uint32) << 16) | np.uint32(0x8000)
    x = np.concatenate([x, ties.view(np.float32)[np.isfinite(ties.view(np.float32))]])
    with np.errstate(over="ignore"):                   # beyond the fp16 range both give +-inf
        assert np.array_equal(I.f64_to_bits(x.astype(np.float64), dtype), _torch_bits(x, dtype))


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_widening_is_exact_and_round_trips(dtype):
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    with np.errstate(invalid="ignore"):                # the NaN patterns, excluded below
        x = I.bits_to_f64(bits, dtype)
    finite = np.isfinite(x)
    assert np.array_equal(I.f64_to_bits(x[finite], dtype), bits[finite])
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16 if dtype == "bf16" else torch.float16)
    ref = ref.double().numpy()
    assert np.array_equal(x[finite], ref[finite])


def test_draws_are_deterministic_and_distinct():
    a = I.gaussian_bits((4, 1000), 1234)
    assert np.array_equal(a, I.gaussian_bits((4, 1000), 1234))
    assert not np.array_equal(a, I.gaussian_bits((4, 1000), 1235))


def test_seed_rule_gives_every_tensor_of_every_workload_its_own_stream():
    seen = {}
    for name, w in I.WORKLOADS.items():
        for t in ("q", "k", "v", "do"):
            s = I.seed_for(w["index"], w.get("length_index", 0), t)
            key = (name.replace("_causal", "").replace("_full", ""), t)   # causal/full pairs share inputs
            assert seen.setdefault(s, key) == key, f"{name}.{t} reuses seed {s} of {seen[s]}"
    for name, w in I.EXTRA_WORKLOADS.items():
        for t in ("q", "k", "v", "do"):
            s = I.seed_for(w["index"], 0, t)
            assert s not in seen, f"{name}.{t} reuses seed {s}"
            seen[s] = (name, t)


@pytest.mark.parametrize("mult", [1.0, 3.0])
def test_gaussian_scale_and_dO_unscaled(mult):
    c = I.make_case(2, 4, 2048, 64, "bf16", True, mult=mult, workload_index=9)
    n = c.q.size
    for name in ("q", "k", "v"):
        x = c.f64(name)
        assert abs(x.mean()) < 5 * mult / np.sqrt(n)
        assert abs(x.std() / mult - 1.0) < 0.01
    do = c.f64("do")
    assert abs(do.std() - 1.0) < 0.01                 # dO is N(0, 1) whatever the input multiplier
    assert c.scale == 64 ** -0.5


def test_workload_table_matches_the_stated_configs():
    W = I.WORKLOADS
    assert (W["c1_tiny"]["B"], W["c1_tiny"]["H"], W["c1_tiny"]["N"], W["c1_tiny"]["d"]) == (1, 1, 256, 64)
    assert (W["c2_gpt2s"]["B"], W["c2_gpt2s"]["H"], W["c2_gpt2s"]["N"]) == (8, 12, 1024)
    assert W["c4a_long"]["dtype"] == W["c4b_long_d128"]["dtype"] == "fp16"
    for n in I.SWEEP_N:
        for m in ("causal", "full"):
            w = W[f"c5_n{n}_{m}"]
            assert w["B"] * w["N"] == 65536 and w["H"] == 16 and w["mult"] == 3.0 and w["dtype"] == "bf16"
            assert w["causal"] == (m == "causal")
