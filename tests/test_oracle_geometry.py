"""Pins of the oracle's split geometry to the examples the pages print, plus
the invariants every geometry must satisfy."""
import itertools
import json
import os

import pytest

import oracle
from oracle.geometry import ceil_div


def _cases(golden_dir):
    with open(os.path.join(golden_dir, "geometry_examples.json")) as f:
        return json.load(f)["cases"]


def test_printed_examples(golden_dir):
    for c in _cases(golden_dir):
        a = c["args"]
        n, chunk = oracle.split_geometry(a["cap"], a["units"], a["wave"], a["granule"],
                                         a["min_chunk"], a["max_splits"], a["mode"], a["override"])
        assert n == c["expect"]["num_splits"], c["name"]
        assert chunk == c["expect"]["chunk"], c["name"]
        if "grid" in c["expect"]:
            assert n * a["units"] == c["expect"]["grid"], c["name"]


def test_wave_rule_granule_16_keeps_the_printed_examples(golden_dir):
    for c in _cases(golden_dir):
        a = dict(c["args"])
        if a["mode"] != oracle.MODE_WAVE:
            continue
        a["granule"] = 16
        n, chunk = oracle.split_geometry(**a)
        assert (n, chunk) == (c["expect"]["num_splits"], c["expect"]["chunk"])


@pytest.mark.parametrize("mode", [oracle.MODE_WAVE, oracle.MODE_POW2_TILES])
def test_invariants(mode):
    caps = [1, 15, 16, 17, 63, 64, 65, 127, 128, 129, 509, 2048, 2112, 4096, 8192, 100000]
    units = [1, 2, 16, 32, 128, 1000]
    waves = [1, 152, 304, 608, 1216]
    granules = [16, 64] if mode == oracle.MODE_POW2_TILES else [1, 16]
    for cap, u, w, g, ov in itertools.product(caps, units, waves, granules, [0, 1, 3, 256]):
        n, chunk = oracle.split_geometry(cap, u, w, g, 128, 32, mode, ov)
        assert 1 <= n <= 32
        assert chunk % g == 0 and chunk >= g
        assert n * chunk >= cap, "every candidate reaches the merge"
        assert (n - 1) * chunk < cap, "no launched split is empty by construction"


def test_pow2_rule_fits_one_wave():
    for cap, u, w in itertools.product([64, 640, 2048, 8192, 32768], [1, 2, 8, 16, 64],
                                       [152, 304, 396, 608]):
        n, chunk = oracle.split_geometry(cap, u, w, 64, 64, 32, oracle.MODE_POW2_TILES, 0)
        tiles = ceil_div(cap, 64)
        tps = chunk // 64
        assert tps & (tps - 1) == 0 or n == 32 or n * u <= w
        if n < 32 and u <= w:
            assert n * u <= w


def test_geometry_never_depends_on_live_length():
    # the function has no live-length argument: same inputs, same answer
    a = oracle.split_geometry(8192, 128, 608, 16, 128, 32, oracle.MODE_WAVE)
    b = oracle.split_geometry(8192, 128, 608, 16, 128, 32, oracle.MODE_WAVE)
    assert a == b


def test_rejects_bad_arguments():
    with pytest.raises(ValueError):
        oracle.split_geometry(100, 0, 10, 1, 1, 32, 0)
    with pytest.raises(ValueError):
        oracle.split_geometry(100, 1, 10, 1, 1, 32, 7)
