"""Properties of the seeded input generator (shared by both sides)."""
import numpy as np

from combine_topk_ids_rank_gb300 import synth


def test_uniform_ids_distinct_and_in_range():
    ids = synth.topk_ids(0, 4, 300, 64, 8)
    assert ids.dtype == np.int32 and ids.shape == (4, 300, 8)
    assert ids.min() >= 0 and ids.max() < 64
    for row in ids.reshape(-1, 8):
        assert len(set(row.tolist())) == 8
    # roughly uniform expert usage
    counts = np.bincount(ids.ravel(), minlength=64)
    assert counts.min() > 0.6 * counts.mean() and counts.max() < 1.4 * counts.mean()


def test_zipf_first_draw_follows_popularity():
    E, s = 256, 1.2
    ids = synth.topk_ids(1, 2, 20000, E, 8, "zipf", s)
    p = np.arange(1, E + 1, dtype=np.float64) ** -s
    p /= p.sum()
    first = np.bincount(ids[:, :, 0].ravel(), minlength=E) / ids[:, :, 0].size
    # the first draw is a plain draw from p; compare the head of the distribution
    for e in range(5):
        se = np.sqrt(p[e] * (1 - p[e]) / ids[:, :, 0].size)
        assert abs(first[e] - p[e]) < 5 * se
    for row in ids.reshape(-1, 8)[:2000]:
        assert len(set(row.tolist())) == 8


def test_weights_are_softmax_rows():
    w = synth.topk_weights(0, 3, 50, 8)
    assert w.dtype == np.float32
    assert np.all(w > 0)
    assert np.allclose(w.sum(axis=-1), 1.0, atol=1e-6)


def test_prefix_property_for_ladder_rungs():
    a = synth.topk_ids(0, 8, 64, 256, 8)
    b = synth.topk_ids(0, 8, 16, 256, 8)
    assert np.array_equal(a[:, :16], b)
    xa = synth.per_rank_rows(0, synth.X, 2, 32, 40)
    xb = synth.per_rank_rows(0, synth.X, 2, 8, 40)
    assert np.array_equal(xa[:, :8], xb)


def test_expert_out_planes_independent_of_extent():
    counts = np.array([[3, 0], [5, 2]])
    a = synth.expert_out_planes(0, 2, 8, 16, counts)
    b = synth.expert_out_planes(0, 2, 6, 16, np.minimum(counts, 2))
    for d in range(2):
        for s in range(2):
            n = min(counts[d, s], 2)
            assert np.array_equal(a[d, s, :n], b[d, s, :n])


def test_normal_payload_statistics():
    x = synth.per_rank_rows(0, synth.X, 2, 64, 512)
    v = (x.astype(np.uint32) << 16).view(np.float32)
    assert abs(v.mean()) < 0.02 and abs(v.std() - 1.0) < 0.02
    g = (synth.gamma(0, 4096).astype(np.uint32) << 16).view(np.float32)
    assert abs(g.mean() - 1.0) < 0.01 and abs(g.std() - 0.1) < 0.01
