"""The seeded input generators: SplitMix64 against a pure-Python restatement of
its published definition (Steele, Lea, Flood, OOPSLA 2014), counter-based
addressing, threaded fills and the value ranges of each kind."""
import numpy as np

import synth

M64 = (1 << 64) - 1


def splitmix64_py(seed, count):
    state, out = seed & M64, []
    for _ in range(count):
        state = (state + 0x9E3779B97F4A7C15) & M64
        z = state
        z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & M64
        z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & M64
        out.append(z ^ (z >> 31))
    return out


def test_raw_stream_matches_definition():
    for seed in (0, 1234, 1241, M64):
        got = synth.fill(synth.RAW64, seed, 300).tolist()
        assert got == splitmix64_py(seed, 300)


def test_counter_addressing_and_threads():
    n = (1 << 21) + 37                     # large enough to split across threads
    a = synth.fill(synth.UNIF_F32, 99, n, lo=-3.0, hi=5.0)
    for start in (0, 1, 12345, n - 10):
        b = synth.fill(synth.UNIF_F32, 99, 10, start=start, lo=-3.0, hi=5.0)
        assert np.array_equal(a[start:start + 10], b)
    idx = [0, 7, 1 << 20, n - 1]
    assert np.array_equal(synth.at(synth.UNIF_F32, 99, idx, lo=-3.0, hi=5.0), a[idx])


def test_uniform_f32_formula_and_range():
    z = np.array(splitmix64_py(5, 1000), dtype=np.uint64)
    u = (z >> np.uint64(40)).astype(np.float32) * np.float32(2.0 ** -24)
    want = np.float32(-1e3) + np.float32(2e3) * u
    got = synth.fill(synth.UNIF_F32, 5, 1000, lo=-1e3, hi=1e3)
    assert np.array_equal(got, want)
    big = synth.fill(synth.UNIF_F32, 6, 1 << 20, lo=-1.0, hi=1.0)
    assert big.min() >= -1.0 and big.max() < 1.0


def test_int_and_bits_and_counts():
    v = synth.fill(synth.UNIF_I32, 3, 1 << 18, lo_i=-2 ** 30, hi_i=2 ** 30)
    assert v.min() >= -2 ** 30 and v.max() <= 2 ** 30
    z = np.array(splitmix64_py(3, 50), dtype=object)
    want = [-2 ** 30 + ((int(x) >> 11) % (2 ** 31 + 1)) for x in z]
    assert v[:50].tolist() == want
    b = synth.fill(synth.BITS16, 3, 50)
    assert b.tolist() == [int(x) >> 48 for x in z]
    c = synth.a2av_send_counts(0, 16)
    assert c.dtype == np.int32 and c.min() >= 0 and c.max() <= 2047


def test_normal_moments():
    x = synth.fill(synth.NORM_F32, 11, 1 << 20).astype(np.float64)
    assert abs(x.mean()) < 5e-3 and abs(x.std() - 1.0) < 5e-3
    assert np.all(np.isfinite(x))


def test_workload_slices_and_samples():
    w = synth.TreduceWorkload("t", 3, synth.DT_BF16, 7, 9, 12, 5, 8, ("normal", 0, 1),
                              ["sum"], src_pad=0x7FD5)
    s = w.slice(2)
    assert s.shape == (7, 12)
    assert np.all(s[5:, :] == 0x7FD5) and np.all(s[:, 8:] == 0x7FD5)
    ii, jj = np.array([0, 4, 2]), np.array([0, 7, 3])
    assert np.array_equal(w.sample(2, ii, jj), s[ii, jj])
    assert w.algorithmic_bytes() == 4 * 2 * 5 * 8


def test_a2av_rows():
    n, tr, size = 4, 10, 6
    x = synth.a2av_input(1, n, tr, size)
    for row in (0, 3, 7, 9):
        assert np.array_equal(synth.a2av_input_row(1, row, n, tr, size), x[row])
    assert x[5, 0] == 1 and x[5, 1] == 2 and x[5, 2] == 1     # mr = 2: row 5 = (d 2, i 1)
