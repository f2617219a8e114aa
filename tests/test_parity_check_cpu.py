"""The GPU tests' tolerance check rejects kernel-like defects (CPU only).

The check (gpu_util.assert_close) holds every element within 3e-2 plus half a
bf16 ulp of the oracle's stored-precision layer, plus that layer's own largest
distance from the exact one in the element's row, and the relative Frobenius
error against the exact layer within 1e-2. Here a flawless bf16 implementation is
stood in for by the stored-precision layer rounded to bf16; it must pass, and
copies of it with a planted defect must fail: a 128x128 tile off by 0.05, one
row's causal mask shifted by one key (the mistake planted in a copy of the
oracle's attention), a whole query tile's mask shifted, one output row taken
from its neighbour.
"""
import math

import numpy as np
import pytest

import oracle
import tsp_inputs
from gpu_util import RECORDS, assert_close, half_ulp_bf16, stored_layer

D, S, H, HEADS, F = 2, 256, 256, 4, 688     # the tiny workload's shape


@pytest.fixture(scope="module")
def case():
    cfg = tsp_inputs.LayerConfig("t", D, S, H, HEADS, F, 1234)
    b = tsp_inputs.layer_inputs(cfg)
    x = oracle.widen_bf16(b["x"])
    W = {k: oracle.widen_bf16(v) for k, v in b.items() if k != "x"}
    exact = oracle.layer_forward(x, W, HEADS)
    st = stored_layer(x, W, HEADS)
    return x, W, exact, st


def _check(got, exact, ref):
    n = len(RECORDS)
    try:
        assert_close(got, exact, "checker: planted", ref=ref)
    finally:
        del RECORDS[n:]


def _rejected(got, exact, ref):
    with pytest.raises(AssertionError):
        _check(got, exact, ref)


def _masked_layer(x, W, shift_rows):
    """The stored-precision layer with the causal mask of `shift_rows` moved one key
    later (each of those queries also sees the key right after it): a planted
    mistake in a copy of the oracle's attention head."""
    def head(q, k, v, q_pos, k_pos, store=None):
        d = q.shape[1]
        s = (q @ k.T) / math.sqrt(d)
        lim = np.asarray(q_pos)[:, None] + np.isin(np.asarray(q_pos), shift_rows)[:, None]
        s = np.where(np.asarray(k_pos)[None, :] <= lim, s, -np.inf)
        p = np.exp(s - s.max(1, keepdims=True))
        return ((p if store is None else store(p)) @ v) / p.sum(1, keepdims=True)
    saved = oracle.tsp_oracle.causal_attention_head
    oracle.tsp_oracle.causal_attention_head = head
    try:
        return stored_layer(x, W, HEADS)
    finally:
        oracle.tsp_oracle.causal_attention_head = saved


def test_flawless_output_passes(case):
    _, _, exact, st = case
    for key in ("attn", "out"):
        _check(oracle.round_bf16(st[key]), exact[key], st[key])


def test_output_rounding_alone_can_exceed_3e_2():
    # why the element bound carries half a bf16 ulp: from |y| = 8 on, the nearest
    # bf16 value can be more than 3e-2 away
    y = np.array([8.0 + 2 ** -5 - 1e-9, 34.0 + 0.12])
    err = np.abs(oracle.round_bf16(y) - y)
    assert (err > 3e-2).all() and (err <= half_ulp_bf16(y)).all()


def test_tile_off_by_005_is_rejected(case):
    _, _, exact, st = case
    got = oracle.round_bf16(st["out"])
    got[128:256, 128:256] += 0.05
    _rejected(got, exact["out"], st["out"])


def test_one_rows_mask_shift_is_rejected(case):
    x, W, exact, st = case
    bad = _masked_layer(x, W, [1])
    got = oracle.round_bf16(bad["out"])
    assert not np.array_equal(got[1], oracle.round_bf16(st["out"][1]))
    _rejected(got, exact["out"], st["out"])


def test_query_tile_mask_shift_is_rejected(case):
    x, W, exact, st = case
    bad = _masked_layer(x, W, np.arange(128))
    _rejected(oracle.round_bf16(bad["attn"]), exact["attn"], st["attn"])
    _rejected(oracle.round_bf16(bad["out"]), exact["out"], st["out"])


def test_late_rows_mask_shift_is_rejected_when_the_key_matters():
    # A row that sees 200 keys moves by O(1/200) when one more key comes in, below
    # any 3e-2 bound, unless that key dominates its scores. Here key 201 is query
    # 200's best match (scores of std ~9, as in the GPU sharp-score attention test),
    # so a mask that lets row 200 see key 201 changes the row by O(1).
    rng = np.random.default_rng(5)
    q, k = (oracle.round_bf16(rng.standard_normal((S, 64)) * 3) for _ in range(2))
    k[201] = q[200]
    v = oracle.round_bf16(rng.standard_normal((S, 64)))
    pos = np.arange(S)
    want = oracle.causal_attention_head(q, k, v, pos, pos)
    lim = pos.copy()
    lim[200] += 1
    s = np.where(pos[None, :] <= lim[:, None], q @ k.T / 8.0, -np.inf)
    p = np.exp(s - s.max(1, keepdims=True))
    bad = oracle.round_bf16((p @ v) / p.sum(1, keepdims=True))
    _check(oracle.round_bf16(want), want, want)
    _rejected(bad, want, want)


def test_row_from_its_neighbour_is_rejected(case):
    _, _, exact, st = case
    got = oracle.round_bf16(st["out"])
    got[77] = got[78]
    _rejected(got, exact["out"], st["out"])


def test_realistic_accumulation_noise_passes(case):
    # fp32-accumulation-sized noise (1e-3 rms) on top of a flawless result passes
    _, _, exact, st = case
    noise = np.random.default_rng(6).standard_normal(st["out"].shape) * 1e-3
    _check(oracle.round_bf16(st["out"] + noise), exact["out"], st["out"])
