"""The seeded input generators: determinism, exact bf16 rounding, target
recipes, and the pages' printed memory figures."""

import json
import math
import os

import numpy as np
import torch

import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "page_memory_figures.json")


def test_splitmix64_matches_sequential_definition():
    # Sequential splitmix64 written with Python integers.
    def seq(seed, n):
        out, x = [], seed
        for _ in range(n):
            x = (x + 0x9E3779B97F4A7C15) & 0xFFFFFFFFFFFFFFFF
            z = x
            z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & 0xFFFFFFFFFFFFFFFF
            z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & 0xFFFFFFFFFFFFFFFF
            out.append(z ^ (z >> 31))
        return out
    for seed in (0, 1, 0xDEADBEEF12345678):
        ref = seq(seed, 20)
        got = synth.splitmix64(seed, 20)
        assert [int(v) for v in got] == ref
        assert [int(v) for v in synth.splitmix64(seed, 5, start=7)] == ref[7:12]
    # Published first output for seed 0 of the reference generator.
    assert int(synth.splitmix64(0, 1)[0]) == 0xE220A8397B1DCDAF


def test_bf16_rounding_is_round_to_nearest_even():
    # fp32-exact inputs: torch's fp32 -> bf16 cast is RNE, so both must agree.
    x = np.random.default_rng(0).standard_normal(100000).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(synth.f64_to_bf16_bits(x.astype(np.float64)), ref)
    # Midpoints: 1 + 2^-8 lies halfway between 1 and 1 + 2^-7 -> even (1.0).
    one = 0x3F80
    assert synth.f64_to_bf16_bits(np.array([1 + 2.0 ** -8]))[0] == one
    assert synth.f64_to_bf16_bits(np.array([1 + 3 * 2.0 ** -8]))[0] == one + 2
    # Just above the midpoint in fp64 (not representable in fp32): rounds up,
    # which a double rounding through fp32 would get wrong.
    assert synth.f64_to_bf16_bits(np.array([1 + 2.0 ** -8 + 2.0 ** -40]))[0] == one + 1
    assert synth.f64_to_bf16_bits(np.array([-1.0]))[0] == 0xBF80
    back = synth.bf16_bits_to_f64(synth.f64_to_bf16_bits(np.array([0.1, -3.5, 1e-3])))
    assert np.allclose(back, [0.1, -3.5, 1e-3], rtol=2 ** -8)


def test_normals_are_seeded_and_have_the_requested_spread():
    a = synth.normal_bf16(7, (300, 64), 0.25)
    b = synth.normal_bf16(7, (300, 64), 0.25)
    c = synth.normal_bf16(8, (300, 64), 0.25)
    assert np.array_equal(a, b) and not np.array_equal(a, c)
    x = synth.bf16_bits_to_f64(a)
    assert abs(x.mean()) < 0.01 and abs(x.std() - 0.25) < 0.005


def test_zipf_rank_one_frequency():
    v, s, n = 5000, 1.1, 200000
    y = synth.zipf_targets(3, n, v, s)
    assert y.min() >= 0 and y.max() < v
    hv = sum(r ** -s for r in range(1, v + 1))
    p1 = 1.0 / hv
    assert abs(np.mean(y == 0) - p1) < 4 * math.sqrt(p1 * (1 - p1) / n)
    assert np.mean(y == 0) > np.mean(y == 1) > np.mean(y == 9)


def test_ignore_count_is_exact():
    y = np.arange(1000, dtype=np.int64)
    for frac, k in ((0.05, 50), (0.02, 20), (0.1, 100), (0.0, 0)):
        z = synth.apply_ignore(y, 11, frac)
        assert np.sum(z == synth.IGNORE_INDEX) == k
        keep = z != synth.IGNORE_INDEX
        assert np.array_equal(z[keep], y[keep])


def test_top16_targets_pick_large_scores():
    h = synth.normal_bf16(1, (64, 32), 1.0)
    w = synth.normal_bf16(2, (500, 32), math.sqrt(9 / 32))
    y = synth.topk_targets(5, h, w, 16, 0.8)
    s = synth.bf16_bits_to_f64(h) @ synth.bf16_bits_to_f64(w).T
    rank = np.array([(s[i] > s[i, y[i]]).sum() for i in range(64)])
    assert np.mean(rank < 16) > 0.6
    assert np.array_equal(y, synth.topk_targets(5, h, w, 16, 0.8))


def test_tiny_workload_recipe():
    wl = synth.WORKLOADS["tiny"]
    inp = synth.make_inputs(wl, seed=0)
    assert inp["H"].shape == (256, 128) and inp["W"].shape == (4096, 128)
    assert inp["H"].dtype == np.uint16
    assert np.sum(inp["y"] == -100) == 13
    w = synth.bf16_bits_to_f64(inp["W"])
    assert abs(w.std() - 1 / math.sqrt(128)) < 0.002
    again = synth.make_inputs(wl, seed=0)
    assert all(np.array_equal(inp[k], again[k]) for k in ("H", "W", "y"))


def test_page_memory_figures():
    figs = json.load(open(GOLDEN))["figures"]
    by_id = {f["id"]: f for f in figs}
    wl = synth.WORKLOADS
    assert round(wl["long128k_head"].logits_bytes_bf16() / 2 ** 30, 2) == by_id["gravity16b_128k_logits"]["value"]
    assert round(wl["gravity16b_head"].logits_bytes_bf16() / 2 ** 30, 2) == by_id["gravity16b_8k_logits"]["value"]
    f = by_id["rows8192_vocab128000_logits"]
    w128 = wl["llama3_8b_head"].scaled(vocab=f["vocab"])
    assert round(w128.logits_bytes_bf16() / 2 ** 30, 2) == f["value"]
    f = by_id["gemma2_2b_gradient_lower_bound"]
    assert round(wl["gemma2_2b_head"].grad_bytes_bf16() / 2 ** 20) == f["value"]


def test_shared_component_workload():
    base = synth.Workload("b", 600, 64, 100, 1.0, "uniform", 0.0)
    shared = synth.Workload("s", 600, 64, 100, 1.0, "uniform", 0.0, h_shared=2.0)
    a = synth.make_inputs(base, seed=4)
    b = synth.make_inputs(shared, seed=4)
    # W and y come from their own streams; without a shared component H is unchanged.
    assert np.array_equal(a["W"], b["W"]) and np.array_equal(a["y"], b["y"])
    assert np.array_equal(synth.make_inputs(base, seed=4)["H"], a["H"])
    ha = synth.bf16_bits_to_f64(a["H"])
    hb = synth.bf16_bits_to_f64(b["H"])
    shift = hb.mean(axis=0) - ha.mean(axis=0)
    # The shift has norm h_shared * sqrt(D); the two means differ only by it
    # (up to one bf16 rounding per element).
    assert abs(np.linalg.norm(shift) - 2.0 * math.sqrt(64)) < 0.1
    assert np.max(np.abs((hb - ha) - shift[None, :])) < 2.0 ** -6 * (np.max(np.abs(hb)) + 1)
