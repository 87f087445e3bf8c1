"""The input generator: Philox-4x32-10 known answers, C vs NumPy twin, moments."""
import numpy as np

import ragen


def test_philox_known_answers():
    # known-answer vectors of the Random123 distribution for philox4x32 with 10 rounds
    assert ragen.philox4x32_10([0, 0, 0, 0], [0, 0]).tolist() == [
        0x6627E8D5, 0xE169C58D, 0xBC57AC4C, 0x9B00DBD8]
    assert ragen.philox4x32_10([0xFFFFFFFF] * 4, [0xFFFFFFFF] * 2).tolist() == [
        0x408F276D, 0x41C83B0E, 0xA20BC7C6, 0x6D5451FD]
    assert ragen.philox4x32_10([0x243F6A88, 0x85A308D3, 0x13198A2E, 0x03707344],
                               [0xA4093822, 0x299F31D0]).tolist() == [
        0xD16CFE09, 0x94FDCCEB, 0x5001E420, 0x24126EA1]
    np_out = ragen.philox4x32_10_np(np.array([[0x243F6A88, 0x85A308D3, 0x13198A2E, 0x03707344]],
                                             dtype=np.uint32), (0xA4093822, 0x299F31D0))
    assert np_out[0].tolist() == [0xD16CFE09, 0x94FDCCEB, 0x5001E420, 0x24126EA1]


def test_c_and_numpy_twins_agree_bitwise():
    for seed, tid, start, n in [(0, 0, 0, 4096), (3000, 2, 12345, 777), (1000, 1, 2**33 + 3, 65)]:
        a = ragen.normal_f32(seed, tid, n, start=start)
        b = ragen.normal_f32_numpy(seed, tid, n, start=start)
        assert np.array_equal(a.view(np.uint32), b.view(np.uint32))
        assert np.array_equal(ragen.normal_bf16(seed, tid, n, start=start),
                              ragen.f32_to_bf16_bits_numpy(b))


def test_subsets_are_consistent():
    full = ragen.normal_bf16(7, 1, 10 * 64)
    rows = [0, 3, 9, 4]
    sub = ragen.normal_bf16_rows(7, 1, rows, 64)
    assert np.array_equal(sub, full.reshape(10, 64)[rows])
    assert np.array_equal(ragen.normal_bf16(7, 1, 100, start=37), full[37:137])


def test_moments():
    x = ragen.normal_f32(1000, 0, 1 << 20).astype(np.float64)
    assert abs(x.mean()) < 5e-3 and abs(x.var() - 1) < 1e-2
    assert abs((x ** 3).mean()) < 2e-2 and abs((x ** 4).mean() - 3) < 5e-2
