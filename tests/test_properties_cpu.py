"""Randomised property checks (CPU only; skipped where hypothesis is not installed).

* the oracle's zigzag maps, single sequence and micro-batch, on random shapes:
  permutations, their inverses, 1/D of every sequence per rank, equal causal work;
* the library's closed-form cost model against the oracle's brute-force count on
  random layer shapes and micro-batches, for every scheme.
"""
import numpy as np
import pytest

hypothesis = pytest.importorskip("hypothesis")
from hypothesis import given, settings, strategies as st  # noqa: E402

import oracle  # noqa: E402
from oracle import cost_sim  # noqa: E402

tsp = pytest.importorskip("folded_tensor_sequence_tsp_gb300")
B = tsp._binding


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import os
    if not os.path.exists(B.library_path()):
        import __graft_entry__
        __graft_entry__.build()
    B.load_library()


@settings(max_examples=60, deadline=None)
@given(D=st.integers(1, 9), chunk=st.integers(1, 12), batch=st.integers(1, 4))
def test_zigzag_maps_on_random_shapes(D, chunk, batch):
    S = 2 * D * chunk
    T = S // D
    fwd = oracle.zigzag_forward_index(S, D)
    assert sorted(fwd.tolist()) == list(range(S))
    inv = oracle.zigzag_inverse_index(S, D)
    assert (inv[fwd] == np.arange(S)).all()
    pairs = oracle.causal_pairs_per_rank(S, D)
    assert (pairs == pairs[0]).all() and pairs.sum() == S * (S + 1) // 2
    fb = oracle.zigzag_forward_index_batched(S, D, batch)
    assert sorted(fb.tolist()) == list(range(batch * S))
    for b in range(batch):
        rows = fb[b * S:(b + 1) * S]
        # sequence b sits in block (r, b) of the rank-major layout, in the single-
        # sequence local order
        r, l = rows // (batch * T), rows % T
        assert ((rows // T) % batch == b).all()
        assert np.array_equal(r * T + l, fwd)


SCHEMES = ["dp", "tp", "sp", "tsp", "tp_sp"]


@settings(max_examples=40, deadline=None)
@given(scheme=st.sampled_from(SCHEMES), D=st.sampled_from([1, 2, 4]),
       heads=st.sampled_from([2, 4, 8]), d=st.sampled_from([2, 4]), f_per=st.integers(1, 6),
       chunk=st.integers(1, 6), batch=st.integers(1, 3), tp=st.sampled_from([1, 2]))
def test_cost_model_equals_brute_force_on_random_shapes(scheme, D, heads, d, f_per, chunk, batch, tp):
    H, F, S = heads * d, 4 * f_per, 2 * 4 * chunk
    if scheme == "dp":
        D = 1
    if scheme == "tp_sp":
        if D % tp or heads % tp or F % tp or S % (2 * (D // tp)):
            return
    elif heads % D or F % D or S % (2 * D):
        return
    got = B.tsp_cost_model_batched(scheme, D, S, batch, H, heads, F, tp=tp if scheme == "tp_sp" else 0)
    want = cost_sim.simulate(scheme, D, S, H, heads, F, tp=tp if scheme == "tp_sp" else 0, batch=batch)
    for k, v in want.items():
        assert got[k] == pytest.approx(v, rel=1e-12, abs=1e-9), (k, got[k], v)
