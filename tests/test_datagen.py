"""The seeded input generator (no GPU)."""
import os

import numpy as np
import pytest

import datagen

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_splitmix64_published_outputs():
    rows = []
    with open(os.path.join(GOLDEN, "splitmix64.txt")) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if line:
                i, v = line.split()
                rows.append((int(i), int(v, 16)))
    out = datagen.raw64(0, len(rows))
    for i, v in rows:
        assert int(out[i]) == v


def test_counter_based_and_deterministic():
    a = datagen.raw64(5, 100)
    b = datagen.raw64(5, 60, offset=40)
    assert np.array_equal(a[40:], b)
    assert not np.array_equal(datagen.raw64(6, 100), a)


def test_uniform_exact_in_fp32_and_in_range():
    u = datagen.uniform(1001, (4096,))
    assert np.all((u > -1) & (u < 1))
    assert np.array_equal(u.astype(np.float32).astype(np.float64), u)
    assert abs(u.mean()) < 0.05
    assert abs(u.var() - 1.0 / 3.0) < 0.02


def test_normal_moments():
    x = datagen.normal(1004, (200000,))
    assert abs(x.mean()) < 0.01
    assert abs(x.std() - 1.0) < 0.01


def test_small_ints_range():
    v = datagen.small_ints(9, (10000,), -8, 8)
    assert v.min() == -8 and v.max() == 8
    assert np.array_equal(v, np.round(v))


def test_bf16_round_to_nearest_even():
    # value -> expected bf16 bits, fixed by RNE on the 16 dropped bits
    cases = {
        1.0: 0x3F80,
        1.0 + 2 ** -8: 0x3F80,          # tie, rounds to even mantissa 0
        1.0 + 3 * 2 ** -8: 0x3F82,      # tie, rounds up to even mantissa 2
        1.0 + 1.5 * 2 ** -8: 0x3F81,    # above the tie
        -2.0: 0xC000,
        0.0: 0x0000,
    }
    for v, want in cases.items():
        assert int(datagen.to_bf16_bits(np.array([v]))[0]) == want


def test_bf16_rounding_matches_ml_dtypes():
    ml_dtypes = pytest.importorskip("ml_dtypes")
    x = datagen.uniform(77, (50000,)).astype(np.float32) * np.float32(3.7)
    ours = datagen.f32_to_bf16_bits(x)
    theirs = x.astype(ml_dtypes.bfloat16).view(np.uint16)
    assert np.array_equal(ours, theirs)


def test_seed_convention():
    assert datagen.seed_for(3, datagen.ROLE_A) == 3001
    assert datagen.seed_for(3, datagen.ROLE_BIAS) == 3004


def test_operand_streams_match_their_recorded_digests():
    """The first 4096 stored values of every operand stream the bench and the
    tests draw are unchanged (tests/golden/datagen_digests.txt)."""
    import importlib.util

    spec = importlib.util.spec_from_file_location(
        "make_datagen_digests", os.path.join(GOLDEN, "make_datagen_digests.py"))
    mk = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mk)
    import hashlib

    n_u = n_n = 0
    with open(os.path.join(GOLDEN, "datagen_digests.txt")) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            kind, seed, payload = line.rstrip("\n").split("|")[:3]
            if kind == "U":
                recipe, digest = payload, line.split("|")[3]
                got = hashlib.sha256(mk.uniform_bits(int(seed), recipe)).hexdigest()
                assert got == digest, line
                n_u += 1
            else:
                want = np.array([float(v) for v in payload.split()])
                got = datagen.normal(int(seed), (len(want),))
                np.testing.assert_allclose(got, want, rtol=1e-13, atol=0)
                n_n += 1
    assert n_u == len(mk.UNIFORM_STREAMS) and n_n == len(mk.NORMAL_STREAMS)
