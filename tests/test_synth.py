"""The seeded input generator: determinism, shapes and the stated distributions."""
import numpy as np

import synth


def test_bf16_rounding_and_widening():
    x = np.array([1.0, 1.00390625, 1.001953125, 1.005859375, -2.5, 3.0e-39], dtype=np.float32)
    b = synth.f32_to_bf16_bits(x)
    # bf16 step at 1.0 is 2^-7: 1 + 2^-8 is a tie (-> even, 1.0), 1 + 2^-9 rounds down,
    # 1 + 3*2^-9 rounds up
    assert list(synth.bf16_bits_to_f32(b)[:5]) == [1.0, 1.0, 1.0, 1.0078125, -2.5]


def test_tiny_deterministic_and_shaped():
    a, b = synth.make_tiny(), synth.make_tiny()
    assert np.array_equal(a.hidden_gen, b.hidden_gen) and np.array_equal(a.head.W, b.head.W)
    assert a.hidden_gen.shape == (64, 128) and a.head.W.shape == (1000, 128)
    assert a.token_ids.min() >= 0 and a.token_ids.max() < 1000
    assert a.mask.sum() == 48 and list(a.seq_offsets) == [0, 16, 32, 48, 64]
    assert a.mask.reshape(4, 16)[:, :4].sum() == 0
    diff = synth.bf16_bits_to_f32(a.hidden_train) - synth.bf16_bits_to_f32(a.hidden_gen)
    rows = a.meta["shifted_rows"]
    assert len(rows) == 2 and np.all(a.mask[rows] == 1)
    assert abs(np.mean(diff[rows]) - 0.5) < 0.05
    other = np.setdiff1d(np.arange(64), rows)
    assert 0.07 < np.std(diff[other]) < 0.13


def test_distributions():
    b = synth.make_custom(T=256, d=512, V=4096, tag="dist")
    W = synth.bf16_bits_to_f32(b.head.W)
    assert abs(np.std(W) - 2 / np.sqrt(512)) < 0.01 * 2 / np.sqrt(512) * 5
    g = synth.bf16_bits_to_f32(b.head.gamma)
    assert abs(np.mean(g) - 1) < 0.05 and abs(np.std(g) - np.sqrt(0.05)) < 0.03
    h = synth.bf16_bits_to_f32(b.hidden_gen)
    assert abs(np.std(h) - 1) < 0.01
    # Zipf: the most frequent id accounts for a large share
    _, counts = np.unique(b.token_ids, return_counts=True)
    assert counts.max() > 0.05 * b.T


def test_qwen3_8b_prefix_structure_small():
    head = synth.Head(d=64, V=100, W=np.zeros((100, 64), np.uint16),
                      gamma=np.zeros(64, np.uint16), vocab_perm=np.arange(100))
    head.d = 64
    b = synth.make_qwen3_8b(samples=3, prefix=5, response=7, head=head)
    L = 12
    for s in range(1, 3):
        assert np.array_equal(b.hidden_gen[s * L:s * L + 5], b.hidden_gen[:5])
        assert np.array_equal(b.hidden_train[s * L:s * L + 5], b.hidden_train[:5])
        assert np.array_equal(b.token_ids[s * L:s * L + 5], b.token_ids[:5])
        assert not np.array_equal(b.hidden_gen[s * L + 5:(s + 1) * L], b.hidden_gen[5:L])
    assert b.mask.reshape(3, L)[:, 5:].all() and not b.mask.reshape(3, L)[:, :5].any()


def test_sweep_plan_small():
    head = synth.make_custom(T=1, d=64, V=300, tag="sw").head
    plan = synth.make_sweep(Ms=(1, 7, 50), n_targets=40, head=head)
    for M, batches in plan.batches.items():
        seen = np.concatenate([bt["target_idx"] for bt in batches])
        assert sorted(seen.tolist()) == list(range(40))
        for bt in batches:
            assert bt["hidden"].shape == (M, 64)
            assert np.array_equal(bt["hidden"][bt["target_pos"]], plan.targets_hidden[bt["target_idx"]])
            assert np.array_equal(bt["ids"][bt["target_pos"]], plan.targets_ids[bt["target_idx"]])
