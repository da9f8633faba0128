"""CPU tests of the seeded input recipe: block b of tensor t is drawn from
numpy.random.default_rng([seed, t, b]), so the values do not depend on how
many threads draw the blocks, and both sides of every comparison read the
same cast values."""
import numpy as np

from sequence_tensor_transformer_gb300 import synth

SHAPE = (5, synth.BLOCK // 2 + 7)  # two full blocks and a ragged third


def test_draw_does_not_depend_on_the_thread_count(monkeypatch):
    monkeypatch.setattr(synth, "_threads", lambda: 1)
    one = synth.draw(SHAPE, 0.5, 1.0, "bf16", 3, 17)
    monkeypatch.setattr(synth, "_threads", lambda: 3)
    three = synth.draw(SHAPE, 0.5, 1.0, "bf16", 3, 17)
    assert np.array_equal(one, three)


def test_blocks_follow_their_counter_based_seeds():
    n = int(np.prod(SHAPE))
    got = synth.draw(SHAPE, 1.0, 0.0, "fp32", 11, 4).reshape(-1)
    for b in range((n + synth.BLOCK - 1) // synth.BLOCK):
        lo, hi = b * synth.BLOCK, min(n, (b + 1) * synth.BLOCK)
        ref = np.random.default_rng([11, 4, b]).standard_normal(hi - lo).astype(np.float32)
        assert np.array_equal(got[lo:hi], ref), b


def test_tensor_ids_and_seeds_give_independent_draws():
    a = synth.draw((1000,), 1.0, 0.0, "fp32", 0, 1)
    assert not np.array_equal(a, synth.draw((1000,), 1.0, 0.0, "fp32", 0, 2))
    assert not np.array_equal(a, synth.draw((1000,), 1.0, 0.0, "fp32", 1, 1))
    # the workloads' tensors use distinct ids: x and the partials differ
    inp = synth.boundary_inputs(synth.TINY_FP32)
    assert not np.array_equal(inp["x"], inp["partials"][0])
