"""The seeded input generator: Philox known answers, determinism, row
addressability and the structure each workload promises."""
import numpy as np
import pytest

import workloads as wk


def test_philox_known_answers():
    # Known-answer vectors published with the Random123 library for
    # Philox4x32 with 10 rounds (Salmon et al., SC'11).
    cases = [
        ([0, 0, 0, 0], [0, 0], [0x6627E8D5, 0xE169C58D, 0xBC57AC4C, 0x9B00DBD8]),
        ([0xFFFFFFFF] * 4, [0xFFFFFFFF] * 2, [0x408F276D, 0x41C83B0E, 0xA20BC7C6, 0x6D5451FD]),
        ([0x243F6A88, 0x85A308D3, 0x13198A2E, 0x03707344], [0xA4093822, 0x299F31D0],
         [0xD16CFE09, 0x94FDCCEB, 0x5001E420, 0x24126EA1]),
    ]
    for ctr, key, want in cases:
        assert wk.philox4x32_10(ctr, key).tolist() == want


def test_rows_regenerate_independently():
    wl = wk.WORKLOADS["ragged"].with_(rows=8, width=2048)
    full, starts, ends = wk.make_all(wl)
    again = wk.make_rows(wl, [5, 2], starts, ends)
    assert np.array_equal(again.view(np.uint32), full[[5, 2]].view(np.uint32))
    assert np.array_equal(wk.make_all(wl)[0].view(np.uint32), full.view(np.uint32))


def test_normal_moments():
    wl = wk.WORKLOADS["tiny"]
    x, _, _ = wk.make_all(wl)
    assert abs(float(x.mean())) < 0.02 and abs(float(x.std()) - 1.0) < 0.02


@pytest.mark.parametrize("name", list(wk.WORKLOADS))
def test_bounds_shapes_and_ranges(name):
    wl = wk.WORKLOADS[name]
    starts, ends = wk.bounds(wl)
    assert ends.dtype == np.int32 and len(ends) == wl.n_bounds
    if name == "tiny":
        assert ends.min() >= 1 and ends.max() <= 4096
    elif name == "decode_short":
        assert ends.min() >= 128 and ends.max() <= 2048
    elif name == "decode_1m":
        assert len(ends) == 48 and ends.min() >= 2 and ends.max() <= 16385
        assert 300 < np.median(ends) < 1200
    elif name == "prefill_1m":
        assert ends[0] == 1_046_273 and ends[-1] == 1_048_320
    elif name == "ragged":
        assert starts.min() >= 0 and starts.max() <= 512
        W, B = wl.width, wl.block_size
        for v in [0, 1, 1023, 1024, 1025, W, W + 1, W + 7, W + B + 3]:
            assert v in ends.tolist()


def test_ragged_ties_and_neg_inf():
    wl = wk.WORKLOADS["ragged"].with_(rows=16)
    x, starts, ends = wk.make_all(wl)
    logical = x[:, 0::2]
    frac_ninf = float(np.isneginf(logical).mean())
    assert 0.0005 < frac_ninf < 0.002
    # exact ties: the row with the longest live span repeats far more values
    # than independent float32 normals would (about 1 % of its columns)
    live = np.minimum(ends.astype(np.int64), wl.width) - starts
    r = int(np.argmax(live))
    row = logical[r, starts[r]:starts[r] + live[r]]
    _, counts = np.unique(row[np.isfinite(row)], return_counts=True)
    assert (counts - 1).sum() > 0.005 * live[r]
    # the interleaved slots hold finite filler
    assert np.isfinite(x[:, 1::2]).all()


def test_prefill_spikes_planted():
    wl = wk.WORKLOADS["prefill_1m"]
    starts, ends = wk.bounds(wl)
    x = wk.make_rows(wl, [0, 2047], starts, ends)
    for i, r in enumerate([0, 2047]):
        big = np.nonzero(x[i] >= 6.0)[0]
        assert 60 <= len(big) <= 64 + 2  # 64 spikes (collisions rare), few natural +6 sigma
        assert big.max() < ends[r]
