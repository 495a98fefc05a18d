"""The seeded input generator: known-answer splitmix64, determinism, slicing, distributions."""
import numpy as np

import seeded_inputs as si


def test_splitmix64_known_answer():
    # Published splitmix64 outputs for seed 1234567.
    want = [6457827717110365317, 3203168211198807973, 9817491932198370423,
            4593380528125082431, 16408922859458223821]
    assert [int(v) for v in si.splitmix64(1234567, 0, 5)] == want


def test_counter_slices_agree():
    full = si.splitmix64(99, 0, 1000)
    assert np.array_equal(full[300:700], si.splitmix64(99, 300, 400))
    d = si.Dist("normal", 0.0, 1.0)
    assert np.array_equal(si.draw_f16(d, 5, 0, 1000)[200:600], si.draw_f16(d, 5, 200, 400))


def test_workload_shapes_and_determinism():
    w = si.WORKLOADS["ktile_grid_256x256x512"]
    A, B = w.operands()
    A2, B2 = w.operands()
    assert A.shape == (256, 512) and B.shape == (256, 512)
    assert A.dtype == np.float16 and B.dtype == np.float16
    assert np.array_equal(A.view(np.uint16), A2.view(np.uint16))
    assert np.array_equal(B.view(np.uint16), B2.view(np.uint16))
    # B continues the stream after A
    assert np.array_equal(B.reshape(-1), si.draw_f16(w.b, w.seed, 256 * 512, 256 * 512))
    assert not np.array_equal(A.view(np.uint16), B.view(np.uint16))


def test_distributions():
    u = si.draw_f16(si.Dist("uniform", -1, 1), 3, 0, 1 << 18).astype(np.float64)
    assert u.min() >= -1 and u.max() <= 1
    assert abs(u.mean()) < 0.01 and abs(u.var() - 1 / 3) < 0.01
    z = si.draw_f16(si.Dist("normal", 0.0, 0.02), 4, 0, 1 << 18).astype(np.float64)
    assert abs(z.mean()) < 1e-3 and abs(z.std() - 0.02) < 5e-4
    # the fp16 values are exactly the RNE rounding of the underlying doubles
    d = si.Dist("uniform", -1, 1)
    raw = d.draw_f64(7, 0, 4096)
    assert np.array_equal(si.draw_f16(d, 7, 0, 4096), raw.astype(np.float16))


def test_headline_metadata():
    w = si.WORKLOADS[si.HEADLINE]
    assert (w.M, w.N, w.K) == (4096, 4096, 4096)
    assert w.flop == 2 * 4096 ** 3
    assert si.WORKLOAD_ORDER[0] == "single_tile_128x128x64"
