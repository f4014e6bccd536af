"""The native step composer (moe_compose_prefill) against the oracle's prefill chunking, call
for call, and its argument checks.  Host-only: no GPU."""
import ctypes

import numpy as np
import pytest

import oracle


@pytest.fixture(scope="module")
def pkg():
    import decode_batches_gb300 as m
    from decode_batches_gb300 import build
    build.build()
    m.load_library()
    return m


def test_composer_matches_the_oracle(pkg):
    rng = np.random.default_rng(7)
    cases = [(0, 20000, q, True, 4096) for q in (128, 512, 1024, 2048, 4096, 8192)]
    cases += [(81920, 8478, 2048, True, cap) for cap in (4096, 3072, 2560)]
    cases += [(1539, 12288, 2048, False, 4096), (5, 0, 64, True, 4096), (4095, 1, 1, True, 4096)]
    for _ in range(300):
        cases.append((int(rng.integers(0, 1 << 33)), int(rng.integers(0, 50000)),
                      int(rng.choice([1, 3, 128, 2048, 5000, 8192])), bool(rng.integers(0, 2)),
                      int(rng.choice([1, 100, 2560, 4096, 65536]))))
    for start, n, q, active, cap in cases:
        got = pkg.compose_prefill(start, n, q, active, cap)
        want = oracle.prefill_calls(start, n, q, active, cap)
        assert [(p, c) for p, c, _ in got] == want, (start, n, q, active, cap)
        pieces = [piece for _, _, piece in got]
        assert pieces == sorted(pieces) and (not pieces or pieces[0] == 0)


def test_composer_piece_index_follows_the_server_pieces(pkg):
    got = pkg.compose_prefill(1539, 6144, 2048, True)
    assert [(c, piece) for _, c, piece in got] == [(2048, 0), (509, 1), (1539, 1), (2048, 2)]


def test_composer_partial_output_and_argument_checks(pkg):
    lib = pkg.load_library()
    total = ctypes.c_int64(-1)
    arr = (pkg.PrefillCall * 2)()
    assert lib.moe_compose_prefill(1539, 12288, 2048, 1, 4096, arr, 2, ctypes.byref(total)) == 0
    assert total.value == 9 and (arr[0].n, arr[1].n) == (2048, 509)
    bad = [(-1, 10, 2048, 1, 4096), (0, -1, 2048, 1, 4096), (0, 10, 0, 1, 4096), (0, 10, 2048, 1, 0)]
    for args in bad:
        assert lib.moe_compose_prefill(*args, None, 0, ctypes.byref(total)) == pkg.MOE_ERR_INVALID_ARG
        assert lib.moe_last_error()
    assert lib.moe_compose_prefill(0, 10, 2048, 1, 4096, None, 0, None) == pkg.MOE_ERR_INVALID_ARG
    assert lib.moe_compose_prefill(0, 10, 2048, 1, 4096, None, 3, ctypes.byref(total)) == pkg.MOE_ERR_INVALID_ARG
