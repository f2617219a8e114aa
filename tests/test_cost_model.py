"""The per-device cost model of [TSP] s3 (memory, communication, FLOPs of DP, TP,
SP, TP+SP and TSP), CPU only.

The library's closed forms (tsp_cost_model, host code) are checked element for
element against the oracle's brute-force count (oracle/cost_sim.py), which builds
explicit per-device ownership sets and steps every collective chunk by chunk. The
page's qualitative claims are then checked on the model, and the TSP figures are
tied to what the library's plan actually allocates.
"""
import pytest

import tsp_inputs
from oracle import cost_sim

tsp = pytest.importorskip("folded_tensor_sequence_tsp_gb300")
B = tsp._binding

FIELDS = ("devices", "weight_elems", "weight_inflight_elems", "act_elems", "act_inflight_elems",
          "comm_weight_elems", "comm_act_elems", "flops")

# small layers the brute-force count finishes quickly; S is a multiple of 2D (zigzag)
SHAPES = [
    dict(S=96, H=32, heads=8, F=48),
    dict(S=64, H=16, heads=4, F=40),
    dict(S=128, H=64, heads=8, F=16),
]


def _cases():
    for shp in SHAPES:
        for D in (1, 2, 4):
            if shp["heads"] % D or shp["F"] % D or shp["S"] % (2 * D):
                continue
            yield ("dp", D, 0, shp)
            yield ("tp", D, 0, shp)
            yield ("sp", D, 0, shp)
            yield ("tsp", D, 0, shp)
            for tp in (2, 4):
                sg = D // tp if D % tp == 0 else 0
                if sg >= 1 and shp["heads"] % tp == 0 and shp["F"] % tp == 0 and shp["S"] % (2 * sg) == 0:
                    yield ("tp_sp", D, tp, shp)
    shp = SHAPES[0]
    for scheme, tp in (("tsp", 0), ("tp", 0), ("sp", 0), ("tp_sp", 2), ("tp_sp", 4)):
        yield (scheme, 8, tp, shp)


CASES = list(_cases())


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import os
    if not os.path.exists(B.library_path()):
        import __graft_entry__
        __graft_entry__.build()
    B.load_library()


@pytest.mark.parametrize("scheme,D,tp,shp", CASES,
                         ids=[f"{c[0]}-D{c[1]}-tp{c[2]}-S{c[3]['S']}H{c[3]['H']}F{c[3]['F']}" for c in CASES])
def test_model_equals_brute_force_count(scheme, D, tp, shp):
    got = B.tsp_cost_model(scheme, D, shp["S"], shp["H"], shp["heads"], shp["F"], tp=tp)
    want = cost_sim.simulate(scheme, D, shp["S"], shp["H"], shp["heads"], shp["F"], tp=tp)
    for k in FIELDS:
        assert got[k] == pytest.approx(want[k], rel=1e-12, abs=1e-9), (k, got[k], want[k])


def _reduce_scatter_only(n, g):
    import numpy as np
    recv = np.zeros(g, dtype=np.int64)
    chunks = [len(c) for c in np.array_split(np.arange(n), g)]
    for step in range(g - 1):
        for i in range(g):
            recv[(i + 1) % g] += chunks[(i - step) % g]
    return recv


def _allgather_with_own_block(blocks):
    import numpy as np
    return np.full(len(blocks), sum(blocks), dtype=np.int64)


@pytest.mark.parametrize("name,patch", [
    ("all-reduce without its all-gather half", ("_ring_allreduce", _reduce_scatter_only)),
    ("all-gather counting the device's own block", ("_ring_allgather", _allgather_with_own_block)),
    ("zigzag groups replaced by contiguous halves",
     ("_tokens", lambda S, r, G: __import__("numpy").arange(r * S // G, (r + 1) * S // G))),
])
def test_hand_example_catches_a_planted_mistake(monkeypatch, name, patch):
    """A plausible mistake planted in the brute-force count breaks the hand-worked
    example (or the balance check that every device gets the same counts)."""
    monkeypatch.setattr(cost_sim, patch[0], patch[1])
    caught = False
    for scheme, want in _hand_table():
        D = 1 if scheme == "dp" else 2
        try:
            sim = cost_sim.simulate(scheme, D, 8, 4, 2, 4)
        except ValueError:
            caught = True
            continue
        if any(sim[k] != want[k] for k in FIELDS):
            caught = True
    assert caught, name


def _model(scheme, D, cfg, tp=0):
    return B.tsp_cost_model(scheme, D, cfg.S, cfg.hidden, cfg.heads, cfg.ffn, tp=tp)


@pytest.mark.parametrize("name", ["small", "7b-16k", "7b-64k", "7b-128k"])
def test_only_tsp_divides_weights_and_activations_by_D(name):
    """[TSP] s3, memory: TSP is the scheme that cuts both the weight-proportional and
    the activation memory by 1/D on D devices; TP leaves activations (x, h)
    replicated, SP leaves the weights replicated, and a tp x (D/tp) TP+SP grid
    divides them by tp and D/tp only."""
    cfg = tsp_inputs.config_by_name(name)
    D = cfg.D
    dp = _model("dp", 1, cfg)
    tspm = _model("tsp", D, cfg)
    assert tspm["weight_elems"] == pytest.approx(dp["weight_elems"] / D)
    assert tspm["act_elems"] == pytest.approx(dp["act_elems"] / D)
    tpm, spm = _model("tp", D, cfg), _model("sp", D, cfg)
    assert tpm["act_elems"] > dp["act_elems"] / D
    assert spm["weight_elems"] == dp["weight_elems"]
    for tp in (2, D // 2):
        g = _model("tp_sp", D, cfg, tp=tp)
        assert g["weight_elems"] > dp["weight_elems"] / D or g["act_elems"] > dp["act_elems"] / D
    # the lowest per-device memory of the five, counting what is in flight
    total = lambda m: m["weight_elems"] + m["weight_inflight_elems"] + m["act_elems"] + m["act_inflight_elems"]
    others = [tpm, spm] + [_model("tp_sp", D, cfg, tp=t) for t in (2, 4)]
    assert all(total(tspm) < total(m) for m in others)


def test_tsp_communication_trade_off():
    """[TSP] s3, communication: TSP moves weights, which TP and TP+SP do not; its
    activation traffic is the K/V all-gather only, so for long sequences it
    receives less than TP (crossover at S = 2H + 1.5F for the same D)."""
    H, heads, F, D = 4096, 32, 11008, 8
    cross = 2 * H + 1.5 * F
    tot = lambda m: m["comm_weight_elems"] + m["comm_act_elems"]
    for S in (4096, 16384):
        t = B.tsp_cost_model("tsp", D, S, H, heads, F)
        p = B.tsp_cost_model("tp", D, S, H, heads, F)
        assert t["comm_weight_elems"] > 0 and p["comm_weight_elems"] == 0
        assert tot(t) > tot(p)
    for S in (32768, 65536, 131072):
        t = B.tsp_cost_model("tsp", D, S, H, heads, F)
        p = B.tsp_cost_model("tp", D, S, H, heads, F)
        assert tot(t) < tot(p)
        assert S > cross
    # the weight share of TSP's traffic falls as S grows
    shares = [B.tsp_cost_model("tsp", D, S, H, heads, F) for S in (16384, 65536, 131072)]
    fr = [m["comm_weight_elems"] / tot(m) for m in shares]
    assert fr[0] > fr[1] > fr[2]


@pytest.mark.parametrize("scheme,tp", [("tp", 0), ("sp", 0), ("tp_sp", 2), ("tsp", 0)])
def test_same_per_device_flops(scheme, tp):
    """[TSP] s3, FLOPs: TSP keeps the per-device FLOPs of TP and SP (the layer's / D)."""
    cfg = tsp_inputs.config_by_name("7b-64k")
    m = _model(scheme, cfg.D, cfg, tp=tp)
    assert m["flops"] == pytest.approx(B.tsp_cost_model("dp", 1, cfg.S, cfg.hidden, cfg.heads,
                                                        cfg.ffn)["flops"] / cfg.D)


@pytest.mark.parametrize("name", ["small", "7b-64k"])
def test_tsp_model_matches_the_plan_allocations(name):
    """The library's TSP plan holds, per logical rank, exactly the model's resident
    weight shard (the packed buffer / D, less the zero rows and columns that pad an
    MLP shard to a multiple of 64) and one head group's gathered K/V (the
    natural-order K and V buffers of one shard)."""
    cfg = tsp_inputs.config_by_name(name)
    plan = B.tsp_plan(cfg.D, cfg.S, cfg.hidden, cfg.heads, cfg.ffn)
    i = plan.info
    m = _model("tsp", cfg.D, cfg)
    pad = 3 * cfg.hidden * (i.shard_ffn_padded - i.shard_ffn)  # W1, W3 rows and W2 columns
    assert i.wpack_elems / cfg.D - pad == m["weight_elems"]
    assert 2 * cfg.S * i.shard_hidden == m["act_inflight_elems"]
    # the per-rank layer input of the sharded layout: T rows of H
    assert i.T * cfg.hidden == m["act_elems"] * cfg.hidden / (6 * cfg.hidden + 3 * cfg.ffn)


def test_rejects_shapes_that_do_not_divide():
    with pytest.raises(B.TSPError):
        B.tsp_cost_model("tsp", 3, 96, 32, 8, 48)
    with pytest.raises(B.TSPError):
        B.tsp_cost_model("tp_sp", 8, 96, 32, 8, 48, tp=3)


def _hand_table():
    import os
    path = os.path.join(os.path.dirname(__file__), "golden", "cost_model_hand_D2.txt")
    rows = []
    with open(path) as fh:
        for ln in fh:
            if ln.strip() and not ln.startswith("#"):
                parts = ln.split()
                rows.append((parts[0], dict(zip(FIELDS, (float(v) for v in parts[1:])))))
    return rows


@pytest.mark.parametrize("scheme,want", _hand_table(), ids=lambda v: v if isinstance(v, str) else "")
def test_hand_worked_example(scheme, want):
    """The brute-force count and the closed forms both give the hand-worked values
    (tests/golden/cost_model_hand_D2.txt) for a 2-device layer small enough to
    count on paper."""
    D = 1 if scheme == "dp" else 2
    sim = cost_sim.simulate(scheme, D, 8, 4, 2, 4)
    got = B.tsp_cost_model(scheme, D, 8, 4, 2, 4)
    for k in FIELDS:
        assert sim[k] == want[k], ("simulator", k, sim[k], want[k])
        assert got[k] == want[k], ("model", k, got[k], want[k])


# ------------------------------------------------------- micro-batches ([TSP] s4)

BATCH_CASES = [c for c in CASES if c[3] is SHAPES[1] or (c[1] == 8)]


@pytest.mark.parametrize("batch", [2, 3])
@pytest.mark.parametrize("scheme,D,tp,shp", BATCH_CASES,
                         ids=[f"{c[0]}-D{c[1]}-tp{c[2]}-S{c[3]['S']}" for c in BATCH_CASES])
def test_batched_model_equals_brute_force_count(scheme, D, tp, shp, batch):
    got = B.tsp_cost_model_batched(scheme, D, shp["S"], batch, shp["H"], shp["heads"], shp["F"], tp=tp)
    want = cost_sim.simulate(scheme, D, shp["S"], shp["H"], shp["heads"], shp["F"], tp=tp, batch=batch)
    for k in FIELDS:
        assert got[k] == pytest.approx(want[k], rel=1e-12, abs=1e-9), (k, got[k], want[k])
    one = B.tsp_cost_model(scheme, D, shp["S"], shp["H"], shp["heads"], shp["F"], tp=tp)
    assert got["weight_elems"] == one["weight_elems"]          # weights serve the batch once
    assert got["comm_weight_elems"] == one["comm_weight_elems"]


@pytest.mark.parametrize("scheme,D,tp", [("dp", 1, 0), ("tp", 4, 0), ("sp", 4, 0),
                                         ("tp_sp", 4, 2), ("tsp", 4, 0)])
def test_max_micro_batch_equals_brute_force_search(scheme, D, tp):
    shp = SHAPES[1]
    for layers in (1, 3):
        for budget in (1e3, 2e4, 6.5e4, 1.3e5, 4e5):
            got = B.tsp_cost_max_batch(scheme, D, shp["S"], shp["H"], shp["heads"], shp["F"],
                                       layers, budget, tp=tp)
            want = cost_sim.max_micro_batch(scheme, D, shp["S"], shp["H"], shp["heads"], shp["F"],
                                            budget, layers=layers, tp=tp)
            assert got == want, (layers, budget, got, want)


def test_max_micro_batch_boundaries():
    shp = SHAPES[0]
    c = cost_sim.simulate("tsp", 4, shp["S"], shp["H"], shp["heads"], shp["F"], batch=5)
    exact = 2 * cost_sim.memory_elems(c, layers=2)       # exactly five sequences fit
    args = ("tsp", 4, shp["S"], shp["H"], shp["heads"], shp["F"], 2)
    assert B.tsp_cost_max_batch(*args, exact) == 5
    assert B.tsp_cost_max_batch(*args, exact - 1) == 4
    assert B.tsp_cost_max_batch(*args, 0.0) == 0
    with pytest.raises(B.TSPError):
        B.tsp_cost_max_batch(*args[:-1], 0, 1e9)             # layers < 1
    with pytest.raises(B.TSPError):
        B.tsp_cost_model_batched("tsp", 4, shp["S"], 0, shp["H"], shp["heads"], shp["F"])


def test_tsp_admits_the_largest_micro_batch():
    """[TSP] s4: the smaller per-device footprint lets TSP take larger micro-batches.
    A 32-layer 7B-shaped model on D = 8 devices of 288 GB: TSP's largest micro-batch
    is at least that of TP, SP and TP+SP at 16K and 64K tokens, and above TP's."""
    for S in (16384, 65536):
        m = {s: B.tsp_cost_max_batch(s, 8, S, 4096, 32, 11008, 32, 288e9, tp=tp)
             for s, tp in (("tp", 0), ("sp", 0), ("tp_sp", 2), ("tsp", 0))}
        assert m["tsp"] >= max(m.values()) and m["tsp"] > m["tp"], (S, m)
        assert m["tsp"] >= 1
