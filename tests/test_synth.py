"""The seeded input generator: the same bits however a range is requested
(whole batch, one head, any start position), so that the GPU side and the
oracle side, which request the same tokens in different pieces, see the same
inputs."""
import numpy as np

from long_context_kv_gb300 import synth


def test_one_head_equals_the_batched_draw():
    sc = synth.channel_scale(5, 3, 128)
    K = synth.keys(5, 2, 3, 0, 5000, 128, sc)
    V = synth.values(5, 2, 3, 0, 5000, 128)
    for b in range(2):
        for h in range(3):
            assert np.array_equal(K[b, h], synth.key_rows(5, b, h, 0, 5000, 128, sc))
            assert np.array_equal(V[b, h], synth.value_rows(5, b, h, 0, 5000, 128))


def test_any_position_range_is_a_slice_of_the_whole():
    sc = synth.channel_scale(6, 1, 128)
    whole = synth.keys(6, 1, 1, 0, 9000, 128, sc)
    for t0, t1 in [(0, 1), (4095, 4097), (100, 8999), (8192, 9000)]:
        assert np.array_equal(synth.keys(6, 1, 1, t0, t1, 128, sc)[0, 0], whole[0, 0, t0:t1])


def test_streams_are_distinct_and_seeded():
    sc = synth.channel_scale(7, 2, 128)
    a = synth.key_rows(7, 0, 0, 0, 64, 128, sc)
    assert not np.array_equal(a, synth.key_rows(7, 0, 1, 0, 64, 128, sc))
    assert not np.array_equal(a, synth.key_rows(8, 0, 0, 0, 64, 128, sc))
    assert np.array_equal(a, synth.key_rows(7, 0, 0, 0, 64, 128, sc))
    # drift: zero rate gives the undrifted keys; the offset grows linearly in t
    assert np.array_equal(synth.drift_keys(7, 2, 2, 3, 128, sc, rate=0.0), synth.decode_keys(7, 2, 2, 3, 128, sc))
    m1 = synth.drift_offset(7, 2, 128, sc, 256)
    m2 = synth.drift_offset(7, 2, 128, sc, 512)
    np.testing.assert_allclose(m2, 2 * m1, rtol=1e-6)
    np.testing.assert_allclose(np.abs(m1), 0.02 * sc, rtol=1e-6)


def test_query_walk_keeps_the_norm_and_sets_the_cosine():
    q = synth.queries_from_keys(3, synth.keys(3, 2, 4, 0, 1, 128, synth.channel_scale(3, 4, 128))[:, :, 0], 0.5, 0)
    assert np.array_equal(synth.query_walk(3, q, 1.0, 5), q)
    for corr in (0.0, 0.5, 0.9, 0.99):
        nxt = synth.query_walk(3, q, corr, 5)
        cos = np.sum(nxt * q, -1) / (np.linalg.norm(nxt, axis=-1) * np.linalg.norm(q, axis=-1))
        # the noise has q's norm and is nearly orthogonal to it in 128 dimensions
        assert np.all(np.abs(cos - corr) < 0.3 * np.sqrt(1 - corr * corr) + 1e-6)
        np.testing.assert_allclose(np.linalg.norm(nxt, axis=-1), np.linalg.norm(q, axis=-1), rtol=0.3)
    assert not np.array_equal(synth.query_walk(3, q, 0.5, 5), synth.query_walk(3, q, 0.5, 6))
