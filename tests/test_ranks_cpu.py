"""The TSP schedule across ranks (folded_tensor_sequence_tsp_gb300.ranks) on the CPU.

The schedule is the page's ("Folding Tensor and Sequence Parallelism for
Memory-Efficient Transformer Training & Inference", s2 Methodology): a broadcast
of each packed attention shard, local projections, a K/V all-gather along the
sequence, attention of each rank's zigzag queries and local accumulation; then the
MLP shards around a ring with local accumulation and no all-reduce. Here every
step's compute is the float64 oracle's (test infrastructure), so these tests check
the schedule and the exchanges themselves: that each rank receives the right shard
and K/V at the right step and that the composition is the plain layer. Two gloo
processes run it with real collectives; the message sizes are checked against the
library's cost model. The CUDA steps are checked on the GPU (test_gpu_ranks.py).
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import oracle
import tsp_inputs
from folded_tensor_sequence_tsp_gb300 import ranks as R


class OracleRankCompute:
    """The rank-local steps by the float64 oracle. A shard's attention part is the
    flattened [Wq_k; Wk_k; Wv_k] rows and W_O,k columns, its MLP part the W1_k, W3_k
    rows and W2_k columns (float64 CPU tensors)."""

    act_dtype = torch.float64

    def __init__(self, D, S, H, heads, F, B=1):
        self.D, self.S, self.H, self.heads, self.F, self.B = D, S, H, heads, F, B
        self.T, self.Hd, self.Fd = S // D, H // D, F // D

    def shards(self, W, k):
        Hd, Fd = self.Hd, self.Fd
        c, f = slice(k * Hd, (k + 1) * Hd), slice(k * Fd, (k + 1) * Fd)
        att = np.concatenate([W["Wq"][c].ravel(), W["Wk"][c].ravel(), W["Wv"][c].ravel(),
                              W["Wo"][:, c].ravel()])
        mlp = np.concatenate([W["W1"][f].ravel(), W["W3"][f].ravel(), W["W2"][:, f].ravel()])
        return torch.from_numpy(att), torch.from_numpy(mlp)

    def _attn(self, shard):
        a, H, Hd = shard.numpy(), self.H, self.Hd
        n = Hd * H
        return (a[:n].reshape(Hd, H), a[n:2 * n].reshape(Hd, H), a[2 * n:3 * n].reshape(Hd, H),
                a[3 * n:].reshape(H, Hd))

    def begin(self, r, xs_r):
        return {"r": r, "x": xs_r.numpy(), "pos": oracle.rank_positions(self.S, self.D)[r]}

    def attention_project(self, st, k, attn_shard, kv_r):
        Wq, Wk, Wv, _ = self._attn(attn_shard)
        st["q"] = st["x"] @ Wq.T
        kv_r.copy_(torch.from_numpy(np.concatenate([st["x"] @ Wk.T, st["x"] @ Wv.T], axis=1)))

    def attention_finish(self, st, k, attn_shard, kv_all):
        # a micro-batch: rank rows [B][T], gathered K|V [D][B][T][2H/D]; one sequence's
        # queries see only that sequence's keys
        _, _, _, Wo = self._attn(attn_shard)
        B, T = self.B, self.T
        kv = kv_all.numpy().reshape(self.D, B, T, 2 * self.Hd)
        o = np.empty((B * T, self.Hd))
        for b in range(B):
            K = oracle.unshard_tokens(kv[:, b, :, :self.Hd], self.D)
            V = oracle.unshard_tokens(kv[:, b, :, self.Hd:], self.D)
            o[b * T:(b + 1) * T] = oracle.multihead_causal_attention(
                st["q"][b * T:(b + 1) * T], K, V, self.heads // self.D, q_pos=st["pos"],
                k_pos=np.arange(self.S))
        st["acc"] = (st["x"] if k == 0 else st["acc"]) + o @ Wo.T
        if k == self.D - 1:
            st["h"] = st["acc"].copy()

    def mlp_step(self, st, t, mlp_shard):
        m, H, Fd = mlp_shard.numpy(), self.H, self.Fd
        W1, W3, W2 = (m[:Fd * H].reshape(Fd, H), m[Fd * H:2 * Fd * H].reshape(Fd, H),
                      m[2 * Fd * H:].reshape(H, Fd))
        st["acc"] = st["acc"] + oracle.swiglu_mlp(st["h"], W1, W3, W2)

    def output(self, st):
        return torch.from_numpy(st["acc"])


def _problem(D, S, H, heads, F, seed):
    cfg = tsp_inputs.LayerConfig("t", D, S, H, heads, F, seed)
    b = tsp_inputs.layer_inputs(cfg)
    x = oracle.widen_bf16(b["x"])
    W = {k: oracle.widen_bf16(v) for k, v in b.items() if k != "x"}
    return x, W


def _run_local(D, S, H, heads, F, seed):
    x, W = _problem(D, S, H, heads, F, seed)
    comp = OracleRankCompute(D, S, H, heads, F)
    xs = oracle.shard_tokens(x, D)
    sh = {r: comp.shards(W, r) for r in range(D)}
    out = R.layer_forward_ranks(D, S // D, H // D, range(D), {r: torch.from_numpy(xs[r]) for r in range(D)},
                                {r: sh[r][0] for r in range(D)}, {r: sh[r][1] for r in range(D)},
                                R.LocalExchange(D), comp)
    return x, W, oracle.unshard_tokens(np.stack([out[r].numpy() for r in range(D)]), D)


@pytest.mark.parametrize("D", [1, 2, 3, 4])
def test_schedule_with_local_exchange_is_the_plain_layer(D):
    S, heads, F = 24 * D, 2 * D, 24 * D
    H = 8 * heads
    x, W, got = _run_local(D, S, H, heads, F, 70 + D)
    want = oracle.layer_forward(x, W, heads)["out"]
    assert np.abs(got - want).max() <= 1e-12 * max(1.0, np.abs(want).max())


def _batch_problem(D, S, H, heads, F, B, seed):
    """B sequences of one layer (same weights): x [B][S][H] float64 and the weights."""
    xs, W = [], None
    for b in range(B):
        x, Wb = _problem(D, S, H, heads, F, seed + 101 * b)
        xs.append(x)
        W = W or Wb
    return np.stack(xs), W


def _rank_rows(x, D, r):
    """Rank r's rows of a micro-batch: its zigzag tokens of every sequence, [B*T][H]."""
    return np.concatenate([oracle.shard_tokens(x[b], D)[r] for b in range(x.shape[0])])


@pytest.mark.parametrize("D,B", [(2, 2), (3, 3)])
def test_micro_batch_schedule_with_local_exchange(D, B):
    """A micro-batch through the same schedule: rank r holds its T tokens of every
    sequence, K|V are gathered as [D][B][T][2H/D], and every sequence's rows equal the
    plain layer of that sequence alone."""
    S, heads, F = 24 * D, 2 * D, 24 * D
    H = 8 * heads
    x, W = _batch_problem(D, S, H, heads, F, B, 300 + D)
    comp = OracleRankCompute(D, S, H, heads, F, B)
    sh = {r: comp.shards(W, r) for r in range(D)}
    out = R.layer_forward_ranks(D, B * (S // D), H // D, range(D),
                                {r: torch.from_numpy(_rank_rows(x, D, r)) for r in range(D)},
                                {r: sh[r][0] for r in range(D)}, {r: sh[r][1] for r in range(D)},
                                R.LocalExchange(D), comp)
    T = S // D
    for b in range(B):
        got = oracle.unshard_tokens(np.stack([out[r].numpy()[b * T:(b + 1) * T] for r in range(D)]), D)
        want = oracle.layer_forward(x[b], W, heads)["out"]
        assert np.abs(got - want).max() <= 1e-12 * max(1.0, np.abs(want).max()), b


def test_a_ring_that_skips_a_rank_is_caught(monkeypatch):
    """A ring shift that takes the parts from rank r + 2 instead of r + 1 makes ranks
    see some MLP shards twice and others never: the check above would fail."""
    def skip_one(self, send, recv):
        for r, t in recv.items():
            t.copy_(send[(r + 2) % self.D])
        return R._Done()
    monkeypatch.setattr(R.LocalExchange, "ring_shift", skip_one)
    D, S, H, heads, F = 4, 64, 32, 4, 64
    x, W, got = _run_local(D, S, H, heads, F, 79)
    want = oracle.layer_forward(x, W, heads)["out"]
    assert np.abs(got - want).max() > 1e-3


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _gloo_rank(rank, world, port, shape, results):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        D, S, H, heads, F, seed = shape
        x, W = _problem(D, S, H, heads, F, seed)
        comp = OracleRankCompute(D, S, H, heads, F)
        att, mlp = comp.shards(W, rank)            # this rank owns shard `rank` only
        xs_r = torch.from_numpy(np.ascontiguousarray(oracle.shard_tokens(x, D)[rank]))
        ex = R.TorchDistExchange()
        out = R.layer_forward_ranks(D, S // D, H // D, [rank], {rank: xs_r}, {rank: att},
                                    {rank: mlp}, ex, comp)[rank].numpy()
        pos = oracle.rank_positions(S, D)[rank]
        want = oracle.layer_forward(x, W, heads, rows=np.sort(pos))["out"]
        want = want[np.argsort(np.argsort(pos))]   # back to the rank's local order
        results[rank] = (float(np.abs(out - want).max()), float(np.abs(want).max()),
                         dict(ex.recv_bytes))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_run_the_layer():
    """Two processes, one rank each, real broadcast / all-gather / ring send-receive
    (gloo) on the tiny workload's shape: each rank's rows equal the plain layer's."""
    shape = (2, 256, 256, 4, 688, 1234)
    port = _free_port()
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        results = m.dict()
        procs = [ctx.Process(target=_gloo_rank, args=(r, 2, port, shape, results)) for r in range(2)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(300)
            assert p.exitcode == 0
        res = dict(results)
    for r in (0, 1):
        err, scale, recv = res[r]
        assert err <= 1e-12 * max(1.0, scale), (r, err)
        # one shard's attention part, K/V of the other rank for 2 shards, one MLP part
        H, F, T = 256, 688, 128
        assert recv["broadcast"] == 8 * (4 * H * H // 2)
        assert recv["all_gather"] == 8 * 2 * (T * 2 * H // 2)
        assert recv["ring"] == 8 * (3 * H * F // 2)


def _gloo_batch_rank(rank, world, port, shape, results):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        D, S, H, heads, F, B, seed = shape
        x, W = _batch_problem(D, S, H, heads, F, B, seed)
        comp = OracleRankCompute(D, S, H, heads, F, B)
        att, mlp = comp.shards(W, rank)
        xs_r = torch.from_numpy(np.ascontiguousarray(_rank_rows(x, D, rank)))
        ex = R.TorchDistExchange()
        out = R.layer_forward_ranks(D, B * (S // D), H // D, [rank], {rank: xs_r}, {rank: att},
                                    {rank: mlp}, ex, comp)[rank].numpy()
        pos = oracle.rank_positions(S, D)[rank]
        T = S // D
        err = 0.0
        for b in range(B):
            want = oracle.layer_forward(x[b], W, heads, rows=np.sort(pos))["out"]
            want = want[np.argsort(np.argsort(pos))]
            err = max(err, float(np.abs(out[b * T:(b + 1) * T] - want).max()) /
                      max(1.0, float(np.abs(want).max())))
        results[rank] = (err, dict(ex.recv_bytes))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_run_a_micro_batch():
    """Two processes through gloo with a micro-batch of 3 sequences: each rank's rows of
    each sequence equal that sequence's plain layer; the K/V all-gather carries B times
    one sequence's bytes, the weight messages are unchanged."""
    D, S, H, heads, F, B = 2, 64, 32, 4, 64, 3
    port = _free_port()
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        results = m.dict()
        procs = [ctx.Process(target=_gloo_batch_rank, args=(r, 2, port, (D, S, H, heads, F, B, 505),
                                                            results)) for r in range(2)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(300)
            assert p.exitcode == 0
        res = dict(results)
    T = S // D
    for r in (0, 1):
        err, recv = res[r]
        assert err <= 1e-12, (r, err)
        assert recv["broadcast"] == 8 * (4 * H * H // 2)
        assert recv["all_gather"] == 8 * 2 * (B * T * 2 * H // 2)
        assert recv["ring"] == 8 * (3 * H * F // 2)


@pytest.mark.parametrize("shape", [(2, 256, 256, 4, 512), (4, 1024, 512, 8, 2048),
                                   (2, 256, 256, 4, 688), (3, 1152, 384, 6, 600)],
                         ids=["D2-F256", "D4", "tiny-padded", "d3-padded"])
def test_message_sizes_match_the_cost_model(shape):
    """Bytes each rank receives in one layer forward with the library's shard layout
    (bf16): (D-1) attention parts, (D-1)/D of the K/V of every shard, (D-1) MLP parts.
    The cost model counts (D-1)/D of the unpadded parameters and 2(D-1)/D S H K/V
    elements; the MLP parts carry zero padding up to Fp (and the W13 tiles up to a
    multiple of 128), which the layout adds on top."""
    import folded_tensor_sequence_tsp_gb300 as tsp
    D, S, H, heads, F = shape
    plan = tsp.tsp_plan(D, S, H, heads, F)
    a_bytes, m_bytes = tsp.tsp_rank_shard_bytes(plan)
    i = plan.info
    Fp = i.shard_ffn_padded
    Fq = (Fp + 127) // 128 * 128
    assert a_bytes == 2 * 4 * H * (H // D)
    assert m_bytes == 2 * (2 * Fq * H + H * Fp)

    class Nothing:
        act_dtype = torch.bfloat16

        def begin(self, r, x):
            return None

        def attention_project(self, *a):
            pass

        def attention_finish(self, *a):
            pass

        def mlp_step(self, *a):
            pass

        def output(self, st):
            return None

    ex = R.LocalExchange(D)
    T = S // D
    z = lambda n: torch.zeros(n, dtype=torch.bfloat16)
    R.layer_forward_ranks(D, T, H // D, range(D), {r: z((T, H)) for r in range(D)},
                          {r: z(a_bytes // 2) for r in range(D)},
                          {r: z(m_bytes // 2) for r in range(D)}, ex, Nothing())
    per_rank = {k: v / D for k, v in ex.recv_bytes.items()}
    cost = tsp.tsp_cost_model("tsp", D, S, H, heads, F)
    P_attn, P_mlp = 4 * H * H, 3 * H * F
    # the cost model's weight traffic split into its attention and MLP shares
    assert cost["comm_weight_elems"] == pytest.approx((D - 1) / D * (P_attn + P_mlp))
    assert per_rank["broadcast"] == pytest.approx(2 * (D - 1) / D * P_attn)
    assert per_rank["all_gather"] == pytest.approx(2 * cost["comm_act_elems"])
    assert per_rank["ring"] == pytest.approx((D - 1) * m_bytes)
    if Fq == Fp == F // D:   # no padding: exactly the cost model's MLP share
        assert per_rank["ring"] == pytest.approx(2 * (D - 1) / D * P_mlp)
    else:
        assert per_rank["ring"] > 2 * (D - 1) / D * P_mlp
