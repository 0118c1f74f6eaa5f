"""The seeded input generator: determinism, index independence, moments."""
import numpy as np

import synthetic
from synthetic import workloads


def test_values_are_a_function_of_the_index():
    full = synthetic.grads(7, 3, 1e-2, n=5000, outlier_frac=0.01, outlier_mult=100.0)
    idx = np.array([0, 1, 17, 4096, 4999])
    part = synthetic.grads(7, 3, 1e-2, idx=idx, outlier_frac=0.01, outlier_mult=100.0)
    assert part.tobytes() == full[idx].tobytes()


def test_steps_seeds_streams_differ():
    a = synthetic.grads(7, 1, 1e-3, n=64)
    assert not np.array_equal(a, synthetic.grads(7, 2, 1e-3, n=64))
    assert not np.array_equal(a, synthetic.grads(8, 1, 1e-3, n=64))
    assert not np.array_equal(a, synthetic.draw(7, synthetic.STREAM_W, 1, 1e-3, n=64))


def test_hash_matches_reference_splitmix64():
    # SplitMix64 with state 0: first outputs of the published generator.
    outs, state = [], 0
    for _ in range(3):
        state = (state + synthetic.GOLDEN) & synthetic.MASK64
        outs.append(synthetic.mix64_int(state))
    assert outs == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]
    got = synthetic.hash_words(0, np.arange(3))
    assert [int(x) for x in got] == outs


def test_moments_and_outliers():
    n = 1 << 20
    g = synthetic.grads(7, 1, 1e-3, n=n)
    assert abs(g.mean()) < 1e-5 and abs(g.std() - 1e-3) < 1e-5
    assert np.abs(g).max() <= 1e-3 * 3.47
    h = synthetic.grads(7, 1, 1e-3, n=n, outlier_frac=0.001, outlier_mult=1000.0)
    frac = np.mean(h != g)
    assert 0.0008 < frac < 0.0012
    assert np.allclose(h[h != g], g[h != g] * np.float32(1000.0), rtol=0, atol=0)


def test_gpt_110m_table():
    t = workloads.gpt_110m_tensors()
    assert len(t) == 196 and sum(k for _, k in t) == 110_418_432
    off, num = workloads.offset_table(t)
    assert off[0] == 0 and all(o + k == o2 for o, k, o2 in zip(off, num, off[1:]))
    assert all(k % 4 == 0 for k in num)
