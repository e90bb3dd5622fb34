"""The CPU oracle against its pins (no GPU)."""
import json
import os

import numpy as np
import pytest

import oracle
from oracle.chunk_table import SENTINEL, build_chunk_table, cdiv, nt_max_bound

import oracle_pins as P

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


@pytest.fixture(scope="module")
def lib():
    return oracle.load_library()


@pytest.mark.parametrize("pin", P.ALL_PINS, ids=lambda f: f.__name__)
def test_oracle_pin(lib, pin):
    pin(lib)


def test_chunked_form_matches_dk_ne_dv(lib):
    rng = np.random.default_rng(21)
    c = P.rand_case(rng, 130, 2, 2, 12, 20, lengths=[64, 66])
    o1, f1 = P.run(lib, c)
    from oracle.chunked import chunked_forward
    o2, f2 = chunked_forward(c["q"], c["k"], c["v"], c["g"], c["beta"], c["scale"],
                             c["initial_state"], c["cu_seqlens"])
    assert P.rel(o1, o2) < 1e-12 and P.rel(f1, f2) < 1e-12


def test_oracle_rejects_bad_arguments(lib):
    rng = np.random.default_rng(1)
    c = P.rand_case(rng, 10, 2, 3, 4, 4)           # Hv not a multiple of H
    with pytest.raises(ValueError):
        P.run(lib, c)
    c = P.rand_case(rng, 10, 1, 1, 4, 4)
    with pytest.raises(ValueError):
        P.run(lib, c, cu_seqlens=np.array([0, 6, 4]))
    with pytest.raises(ValueError):
        P.run(lib, c, cu_seqlens=np.array([0, 11]))


def test_oracle_thread_count_does_not_change_results(lib):
    rng = np.random.default_rng(2)
    c = P.rand_case(rng, 90, 2, 4, 16, 16, lengths=[40, 50])
    a = oracle.recurrent_forward(c["q"], c["k"], c["v"], c["g"], c["beta"], c["scale"],
                                 c["initial_state"], c["cu_seqlens"], nthreads=1, lib=lib)
    b = oracle.recurrent_forward(c["q"], c["k"], c["v"], c["g"], c["beta"], c["scale"],
                                 c["initial_state"], c["cu_seqlens"], nthreads=4, lib=lib)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


# ------------------------------------------------------------------ chunk table
def test_chunk_table_definition():
    cu = [0, 5, 5, 69, 200, 200]
    table, offs, total = build_chunk_table(cu, nt_max=12)
    assert total == 1 + 0 + 1 + 3 + 0 == offs[-1]
    assert offs == [0, 1, 1, 2, 5, 5]
    assert table[:5] == [[0, 0], [2, 0], [3, 0], [3, 1], [3, 2]]
    assert all(r == [SENTINEL, SENTINEL] for r in table[5:])


def test_chunk_table_bound_is_tight():
    """31 one-token sequences plus one of 4065 tokens fill NT_max exactly."""
    lengths = [1] * 31 + [4096 - 31]
    cu = np.concatenate([[0], np.cumsum(lengths)])
    nt_max = nt_max_bound(4096, 32)
    table, offs, total = build_chunk_table(cu, nt_max)
    assert nt_max == 95 and total == 95
    assert all(r[0] >= 0 for r in table)


def test_rfc_memory_figure_pins_nt_max():
    """The RFC's resident-memory example implies NT_max = 95 for (4096, 32)."""
    with open(os.path.join(GOLDEN, "rfc_static_bound.json")) as f:
        g = json.load(f)
    nt = nt_max_bound(g["T_max"], g["N_max"], g["chunk_size"])
    assert g["state_bytes_per_head_per_chunk"] == g["dk"] * g["dv"] * 4
    total_mb = nt * g["H"] * g["state_bytes_per_head_per_chunk"] / 2 ** 20
    assert abs(total_mb - g["approx_resident_MB"]) < 1.0
    assert nt == 95


@pytest.mark.parametrize("seed", range(20))
def test_chunk_table_never_exceeds_bound(seed):
    rng = np.random.default_rng(seed)
    n = int(rng.integers(1, 33))
    cuts = np.sort(rng.integers(0, 4097, size=n - 1))
    cu = np.concatenate([[0], cuts, [int(rng.integers(cuts[-1] if n > 1 else 0, 4097))]])
    _, offs, total = build_chunk_table(cu, nt_max_bound(4096, 32))
    assert total <= nt_max_bound(4096, 32)
    assert total == sum(cdiv(int(b - a), 64) for a, b in zip(cu[:-1], cu[1:]))


@pytest.mark.parametrize("pin", P.BACKWARD_PINS, ids=lambda f: f.__name__)
def test_backward_pin(lib, pin):
    pin(lib)


def test_backward_is_independent_of_thread_count(lib):
    rng = np.random.default_rng(24)
    c = P.rand_case(rng, 140, 2, 4, 8, 8, lengths=[70, 70])
    do = rng.standard_normal(c["v"].shape)
    a = oracle.recurrent_backward(c["q"], c["k"], c["v"], c["g"], c["beta"], c["scale"],
                                  c["initial_state"], c["cu_seqlens"], do, None, nthreads=1)
    b = oracle.recurrent_backward(c["q"], c["k"], c["v"], c["g"], c["beta"], c["scale"],
                                  c["initial_state"], c["cu_seqlens"], do, None, nthreads=3)
    for key in a:
        assert np.array_equal(a[key], b[key]), key
