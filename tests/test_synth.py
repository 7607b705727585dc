"""Host-side checks of the seeded input generator (no GPU)."""

import numpy as np
import pytest

from synth import workloads as wl


def test_bf16_rounding_matches_torch():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(0)
    x = np.concatenate([
        rng.standard_normal(20000).astype(np.float32) * np.float32(3.0),
        np.array([0.0, -0.0, 1.0, 1.00390625, 1.01171875, -2.5, 3.3e38, 1e-40], np.float32),
    ])
    want = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(wl.f32_to_bf16_bits(x), want)
    back = wl.bf16_bits_to_f32(want)
    assert np.array_equal(back, torch.from_numpy(want.view(np.int16)).view(torch.bfloat16).float().numpy())


def test_logits_grid_and_range():
    z = wl.logits_f32(wl.raw_words(0, 0, wl.TAG_VERIFY, 0, 100000))
    assert z.dtype == np.float32
    assert z.min() >= -8.0 and z.max() < 8.0
    scaled = (z.astype(np.float64) + 8.0) * 2 ** 20
    assert np.array_equal(scaled, np.round(scaled))


def test_streams_are_deterministic_and_independent():
    a = wl.raw_words(0, 0, wl.TAG_TREE, 3, 64)
    b = wl.raw_words(0, 0, wl.TAG_TREE, 3, 64)
    c = wl.raw_words(0, 1, wl.TAG_TREE, 3, 64)
    d = wl.raw_words(0, 0, wl.TAG_HIDDEN, 3, 64)
    assert np.array_equal(a, b)
    assert not np.array_equal(a, c) and not np.array_equal(a, d)


def test_normal_bf16_moments():
    bits = wl.normal_bf16_bits(wl.raw_words(0, 0, wl.TAG_W, 0, 400000), 0.02)
    x = wl.bf16_bits_to_f32(bits).astype(np.float64)
    assert abs(x.mean()) < 2e-4
    assert abs(x.std() - 0.02) < 4e-4
    assert np.abs(x).max() < 0.02 * 3.47  # Irwin-Hall(4) support is +-sqrt(12)


def test_w_head_rows_are_consistent_with_full_matrix():
    w = wl.Workload(wl.get_config("toy_v4096_h256"))
    full = w.w_head()
    assert full.shape == (4096, 256) and full.dtype == np.uint16
    assert np.array_equal(w.w_head_rows(250, 777), full[250:777])
    assert np.array_equal(w.w_head_rows(4095, 4096), full[4095:])


def test_zipf_ids_range_and_skew():
    V = 1000
    ids = wl.zipf_ids(V, 1.1, wl.unit_f64(wl.raw_words(0, 0, wl.TAG_PROMPT, 9, 50000)))
    assert ids.min() >= 0 and ids.max() < V
    counts = np.bincount(ids, minlength=V)
    assert counts[0] > counts[1] > counts[5] > counts[100]


def test_toy_workload_shapes():
    cfg = wl.get_config("toy_v4096_h256")
    w = wl.Workload(cfg)
    p = w.prompt(0)
    assert p.shape == (256,) and p.dtype == np.int32 and 0 <= p.min() and p.max() < cfg.V
    t = w.trees(0)
    assert t.shape == (16, 16) and t.min() >= 0 and t.max() < cfg.V
    assert w.prefill_logits(0).shape == (256, 4096)
    assert w.verify_logits(0, 3).shape == (16, 4096)
    rows = {w.verify_row(0, s) for s in range(16)}
    assert rows <= set(range(16)) and len(rows) > 1
    assert w.hiddens(0, 2).shape == (16, 256)


def test_self_copy_prompt_locality():
    cfg = wl.get_config("llama3_8b_v128256_h4096")
    p = wl.Workload(cfg).prompt(0)
    # with 60% self-copies the prompt has far fewer distinct ids than positions
    assert len(np.unique(p)) < 0.6 * len(p)


def test_batched_prompt_lengths():
    cfg = wl.get_config("batched16_v128256_h4096")
    w = wl.Workload(cfg)
    lens = [w.prompt_len(b) for b in range(cfg.batch)]
    assert all(512 <= L <= 4096 for L in lens) and len(set(lens)) > 1
