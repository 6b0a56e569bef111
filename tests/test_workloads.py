"""The synthetic-input recipes: determinism and the id-list structure."""
import numpy as np

from sparse_selected_attention_gb300 import workloads as wl


def test_generator_is_deterministic_and_seeded():
    a = wl.random_u64(5, 1, 1000)
    b = wl.random_u64(5, 1, 1000)
    c = wl.random_u64(6, 1, 1000)
    d = wl.random_u64(5, 2, 1000)
    assert np.array_equal(a, b) and not np.array_equal(a, c) and not np.array_equal(a, d)
    # SplitMix64 reference value: seed 0 of the original generator emits
    # 0xE220A8397B1DCDAF first; our stream key is a SplitMix64 output too, so
    # check the mixer on that published first output instead.
    z = np.array([0x9E3779B97F4A7C15], dtype=np.uint64)
    assert int(wl._mix(z)[0]) == 0xE220A8397B1DCDAF


def test_distributions():
    u = wl.uniform(5, 3, (200000,))
    assert 0.0 <= u.min() and u.max() < 1.0 and abs(u.mean() - 0.5) < 0.005
    n = wl.normal(5, 4, (200000,))
    assert abs(n.mean()) < 0.01 and abs(n.std() - 1.0) < 0.01
    c = wl.make_cache(20000, seed=5)
    assert c.kq.min() == -127 and c.kq.max() == 127 and c.kq.dtype == np.int8
    assert c.ksc.dtype == np.float16 and float(c.ksc.min()) >= 0.00099 and float(c.ksc.max()) <= 0.02001


def test_decode_ids_structure():
    ids = wl.decode_ids(8, 30000)
    for t in range(8):
        p = 30000 + t
        row = ids[t]
        cells = row[row >= 0]
        assert len(cells) == 321 and np.all(row[321:] == -1)
        assert np.all(np.diff(cells) > 0) and cells[0] == 0 and cells[-1] == p
        assert np.array_equal(cells[:64], np.arange(64)) and np.array_equal(cells[64:], np.arange(p - 256, p + 1))
    tiny = wl.decode_ids(1, 320)[0]
    assert np.array_equal(tiny[:321], np.arange(321)) and np.all(tiny[321:] == -1)
    small = wl.decode_ids(1, 10)[0]
    assert np.array_equal(small[:11], np.arange(11)) and np.all(small[11:] == -1)


def test_even_ids_structure():
    for pos0 in (0, 30000):
        ids = wl.even_ids(1984, pos0)
        for t in (0, 1, 63, 64, 1000, 1983):
            p = pos0 + t
            row = ids[t]
            k = min(p + 1, 2048)
            cells = row[:k]
            assert np.all(row[k:] == -1)
            assert np.all(np.diff(cells) > 0) and cells[0] == 0 and cells[-1] == p and cells.max() <= p
            assert len(np.unique(cells)) == k
    wide = wl.even_ids(3, 30000, width=2112, select=2051)
    assert np.all(np.sum(wide >= 0, axis=1) == 2051)
    assert np.all(wide[:, 2048:2051] >= 0) and np.all(wide[:, 2051:] == -1)


def test_edge_modes():
    q = wl.queries_f16(14, seed=5)
    e1 = wl.edge_signed_zero(q)
    assert np.all(e1[0] == 0) and not np.signbit(e1[0]).any()
    assert np.all(e1[3] == 0) and np.signbit(e1[3]).all()
    assert np.array_equal(e1[1], q[1])
    cache = wl.make_cache(100, seed=5)
    e2, c2 = wl.edge_cancellation(q, cache)
    assert np.array_equal(c2.kq[:, 64:], c2.kq[:, :64]) and np.array_equal(c2.ksc[:, 2:], c2.ksc[:, :2])
    assert not np.array_equal(cache.kq[:, 64:], cache.kq[:, :64])
    d = e2[5, :, 64:].astype(np.float32) + e2[5, :, :64].astype(np.float32)
    assert np.abs(d).max() < 0.01
    assert np.array_equal(e2[4], q[4])
