"""The rank-local calls of the TSP layer (one rank's tokens, one weight shard per
call) on the GPU, through the C ABI.

Steps against the single-GPU path and the oracle: the rank's Q/K/V projection and
attention give the all-rank steps' rows of that rank bit for bit, the K/V gather
from the all-gathered K|V rows is the zigzag inverse bit for bit, and the whole
schedule (broadcast of attention shards, K/V all-gather, local accumulation, MLP
ring with local accumulation) reproduces the layer: every rank driven from this
process with buffer hand-offs, and two processes on this GPU exchanging through
gloo. The page's schedule is multi-device; here the ranks share one GPU, and no
kernel waits on another rank's kernel (the exchanges are between launches).
"""
import os
import socket

import numpy as np
import pytest
import torch

import oracle
import tsp_inputs
from gpu_util import Layer, assert_close, bits, dev, f64, rand_bits, stored_layer

tsp = pytest.importorskip("folded_tensor_sequence_tsp_gb300")
pytestmark = pytest.mark.gpu

SHAPES = {
    "tiny": (2, 256, 256, 4, 688),
    "ragged": (2, 200, 128, 2, 96),       # T = 100: partial tiles everywhere
    "d3": (3, 1152, 384, 6, 600),         # odd D, padded MLP shards (Fp 256, Fq 256)
    "d1": (1, 384, 256, 2, 512),
    "hd128": (2, 512, 512, 4, 1024),
    "small": (4, 4096, 1024, 16, 2816),   # Fp = 704: W13 tiles padded to 768
}


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    tsp.load_library()


def _shards(L):
    from folded_tensor_sequence_tsp_gb300 import ranks as R
    W = {k: L.d[k] for k in ("Wq", "Wk", "Wv", "Wo", "W1", "W3", "W2")}
    return R.pack_rank_shards(L.plan, W, range(L.info.D))


@pytest.mark.parametrize("name", list(SHAPES))
def test_rank_steps_match_the_all_rank_steps(name):
    """tsp_rank_qkv and tsp_rank_attention of rank r give rows r*T .. (r+1)*T - 1 of
    the all-rank Q/K/V projection and attention bit for bit (the same products and
    the same per-row softmax); tsp_rank_kv_gather is the zigzag inverse."""
    L = Layer(*SHAPES[name], seed=51)
    i = L.info
    D, T, S, Hd = i.D, i.T, i.S, i.shard_hidden
    sh = _shards(L)
    xs = L.sharded_x()
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    q_all, kn, vn = (torch.empty((S, Hd), dtype=torch.bfloat16, device="cuda") for _ in range(3))
    o_all = L.act()
    for k in sorted({0, D - 1}):
        tsp.tsp_qkv_projection_gathered(L.plan, k, xs, L.wpack, q_all, kn, vn, L.ws)
        tsp.tsp_causal_attention_q(L.plan, k, q_all, kn, vn, o_all, L.ws)
        kv_all = torch.empty((D, T, 2 * Hd), dtype=torch.bfloat16, device="cuda")
        qs = []
        for r in range(D):
            q_r = torch.empty((T, Hd), dtype=torch.bfloat16, device="cuda")
            tsp.tsp_rank_qkv(L.plan, xs[r * T:(r + 1) * T], sh[k][0], q_r, kv_all[r], ws)
            qs.append(q_r)
        kn_r, vn_r = torch.empty_like(kn), torch.empty_like(vn)
        tsp.tsp_rank_kv_gather(L.plan, kv_all, kn_r, vn_r)
        assert torch.equal(kn_r.view(torch.int16), kn.view(torch.int16)), k
        assert torch.equal(vn_r.view(torch.int16), vn.view(torch.int16)), k
        for r in range(D):
            assert torch.equal(qs[r].view(torch.int16), q_all[r * T:(r + 1) * T].view(torch.int16))
            o_r = torch.full((T, Hd), float("nan"), dtype=torch.bfloat16, device="cuda")
            tsp.tsp_rank_attention(L.plan, r, qs[r], kn_r, vn_r, o_r, ws)
            want = o_all[r * T:(r + 1) * T, k * Hd:(k + 1) * Hd].contiguous()
            assert torch.equal(o_r.view(torch.int16), want.view(torch.int16)), (k, r)
    assert tsp.tsp_device_status(ws) == tsp.TSP_OK
    L.check_status()


def test_rank_kv_gather_is_the_zigzag_inverse():
    L = Layer(*SHAPES["d3"], seed=52, names=["x"])
    i = L.info
    kv_bits = rand_bits((i.D, i.T, 2 * i.shard_hidden), 53)
    kn = torch.empty((i.S, i.shard_hidden), dtype=torch.bfloat16, device="cuda")
    vn = torch.empty_like(kn)
    tsp.tsp_rank_kv_gather(L.plan, dev(kv_bits), kn, vn)
    Hd = i.shard_hidden
    assert np.array_equal(bits(kn), oracle.unshard_tokens(kv_bits[:, :, :Hd], i.D))
    assert np.array_equal(bits(vn), oracle.unshard_tokens(kv_bits[:, :, Hd:], i.D))


@pytest.mark.parametrize("name", list(SHAPES))
def test_rank_schedule_reproduces_the_layer(name):
    """Every rank driven from this process (buffer hand-offs for the broadcast, the
    all-gather and the ring): the layer output against the oracle, and against
    tsp_layer_fwd (the same products; only the fp32 summation of the shards' partial
    outputs differs)."""
    from folded_tensor_sequence_tsp_gb300 import ranks as R
    L = Layer(*SHAPES[name], seed=54)
    i = L.info
    D, T = i.D, i.T
    sh = _shards(L)
    xs = L.sharded_x()
    comp = R.CudaRankCompute(L.plan)
    out = R.layer_forward_ranks(D, T, i.shard_hidden, range(D),
                                {r: xs[r * T:(r + 1) * T] for r in range(D)},
                                {r: sh[r][0] for r in range(D)}, {r: sh[r][1] for r in range(D)},
                                R.LocalExchange(D), comp)
    torch.cuda.synchronize()
    comp.check()
    got = torch.cat([out[r] for r in range(D)])
    layer = L.act()
    tsp.tsp_layer_fwd(L.plan, xs, L.wpack, layer, L.ws)
    L.check_status()
    nat = lambda t: f64(L.unshard(t))
    ref = oracle.layer_forward(L.f("x"), L.weights64(), i.heads)["out"]
    st = stored_layer(L.f("x"), L.weights64(), i.heads)["out"]
    assert_close(nat(got), ref, f"ranks {name} out", ref=st)
    assert_close(nat(got), nat(layer), f"ranks {name} vs tsp_layer_fwd")


@pytest.mark.parametrize("shape,batch", [((2, 256, 256, 4, 688), 3), ((4, 4096, 1024, 16, 2816), 2)],
                         ids=["tiny-b3", "small-b2"])
def test_rank_schedule_micro_batch(shape, batch):
    """A micro-batch through the rank-local path (rank r holds its rows of every
    sequence): each sequence's output against the oracle, and all of it against
    tsp_layer_fwd of the same batched plan."""
    from folded_tensor_sequence_tsp_gb300 import ranks as R
    L = Layer(*shape, seed=55, batch=batch)
    i = L.info
    D, H = i.D, i.hidden
    rows = batch * i.T
    sh = _shards(L)
    xs = L.sharded_x().view(-1, H)
    comp = R.CudaRankCompute(L.plan)
    out = R.layer_forward_ranks(D, rows, i.shard_hidden, range(D),
                                {r: xs[r * rows:(r + 1) * rows] for r in range(D)},
                                {r: sh[r][0] for r in range(D)}, {r: sh[r][1] for r in range(D)},
                                R.LocalExchange(D), comp)
    torch.cuda.synchronize()
    comp.check()
    got = torch.cat([out[r] for r in range(D)]).view(L.d["x"].shape)
    layer = L.act()
    tsp.tsp_layer_fwd(L.plan, xs, L.wpack, layer, L.ws)
    L.check_status()
    nat = lambda t: f64(L.unshard(t.reshape(L.d["x"].shape).contiguous()))
    x = L.f("x")
    W = L.weights64()
    ref = oracle.layer_forward_batched(x, W, i.heads)["out"]
    st = oracle.layer_forward_batched(x, W, i.heads, store=oracle.round_bf16)["out"]
    g = nat(got)
    for b in range(batch):
        assert_close(g[b], ref[b], f"ranks batch {shape[0]}x{shape[1]} seq {b}", ref=st[b])
    assert_close(g.reshape(-1, H), nat(layer).reshape(-1, H), f"ranks batch {batch} vs tsp_layer_fwd")


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _gpu_rank(rank, world, port, shape, results):
    """One rank per process on the one GPU: its own tokens and its own shard; the
    broadcast, all-gather and ring go through gloo via host memory."""
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    sys.path[:0] = [root, os.path.join(root, "tests")]
    import folded_tensor_sequence_tsp_gb300 as t
    from folded_tensor_sequence_tsp_gb300 import ranks as R
    torch.cuda.set_device(0)
    t.load_library()
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        D, S, H, heads, F, seed = shape
        cfg = tsp_inputs.LayerConfig("t", D, S, H, heads, F, seed)
        b = tsp_inputs.layer_inputs(cfg)
        to = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).cuda()
        plan = t.tsp_plan(D, S, H, heads, F)
        W = {k: to(v) for k, v in b.items() if k != "x"}
        att, mlp = R.pack_rank_shards(plan, W, [rank])[rank]
        T = S // D
        xs_r = to(oracle.shard_tokens(b["x"], D)[rank])
        comp = R.CudaRankCompute(plan)
        out = R.layer_forward_ranks(D, T, H // D, [rank], {rank: xs_r}, {rank: att}, {rank: mlp},
                                    R.TorchDistExchange(stage_host=True), comp)[rank]
        torch.cuda.synchronize()
        comp.check()
        results[rank] = out.view(torch.int16).cpu().numpy().view(np.uint16)
    finally:
        dist.destroy_process_group()


def test_two_processes_exchange_through_gloo():
    """Two ranks in two processes on this GPU, gloo collectives through host memory:
    the outputs assembled from both ranks match the oracle, and the ranks' output
    bits equal the single-process schedule's."""
    import torch.multiprocessing as mp
    from folded_tensor_sequence_tsp_gb300 import ranks as R
    shape = (2, 256, 256, 4, 688, 1234)
    D, S, H, heads, F, seed = shape
    port = _free_port()
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        results = m.dict()
        procs = [ctx.Process(target=_gpu_rank, args=(r, 2, port, shape, results)) for r in range(2)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(300)
            assert p.exitcode == 0
        res = dict(results)
    got = np.concatenate([res[0], res[1]]).reshape(D, S // D, H)
    L = Layer(D, S, H, heads, F, seed=seed)
    sh = _shards(L)
    xs = L.sharded_x()
    T = S // D
    one = R.layer_forward_ranks(D, T, H // D, range(D), {r: xs[r * T:(r + 1) * T] for r in range(D)},
                                {r: sh[r][0] for r in range(D)}, {r: sh[r][1] for r in range(D)},
                                R.LocalExchange(D), R.CudaRankCompute(L.plan))
    for r in range(D):
        assert np.array_equal(got[r], bits(one[r])), r
    x = L.f("x")
    ref = oracle.layer_forward(x, L.weights64(), heads)["out"]
    st = stored_layer(x, L.weights64(), heads)["out"]
    assert_close(oracle.unshard_tokens(oracle.widen_bf16(got), D), ref, "ranks gloo 2 processes",
                 ref=st)


@pytest.mark.slow
def test_rank_steps_at_the_7b_shape():
    """At the 7B shape and 16K tokens (the benchmark's launch sizes for one rank): the
    rank-local Q/K/V projection, K/V gather and attention of the first and the last
    rank give the all-rank steps' rows bit for bit, for the first and the last shard."""
    cfg = tsp_inputs.config_by_name("7b-16k")
    L = Layer(cfg.D, cfg.S, cfg.hidden, cfg.heads, cfg.ffn, seed=cfg.seed)
    i = L.info
    D, T, S, Hd = i.D, i.T, i.S, i.shard_hidden
    sh = _shards(L)
    xs = L.sharded_x()
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    q_all, kn, vn = (torch.empty((S, Hd), dtype=torch.bfloat16, device="cuda") for _ in range(3))
    o_all = L.act()
    kv_all = torch.empty((D, T, 2 * Hd), dtype=torch.bfloat16, device="cuda")
    for k in (0, D - 1):
        tsp.tsp_qkv_projection_gathered(L.plan, k, xs, L.wpack, q_all, kn, vn, L.ws)
        tsp.tsp_causal_attention_q(L.plan, k, q_all, kn, vn, o_all, L.ws)
        qs = {}
        for r in range(D):
            q_r = torch.empty((T, Hd), dtype=torch.bfloat16, device="cuda")
            tsp.tsp_rank_qkv(L.plan, xs[r * T:(r + 1) * T], sh[k][0], q_r, kv_all[r], ws)
            qs[r] = q_r
        kn_r, vn_r = torch.empty_like(kn), torch.empty_like(vn)
        tsp.tsp_rank_kv_gather(L.plan, kv_all, kn_r, vn_r)
        assert torch.equal(kn_r.view(torch.int16), kn.view(torch.int16)), k
        assert torch.equal(vn_r.view(torch.int16), vn.view(torch.int16)), k
        for r in (0, D - 1):
            assert torch.equal(qs[r].view(torch.int16), q_all[r * T:(r + 1) * T].view(torch.int16))
            o_r = torch.full((T, Hd), float("nan"), dtype=torch.bfloat16, device="cuda")
            tsp.tsp_rank_attention(L.plan, r, qs[r], kn_r, vn_r, o_r, ws)
            want = o_all[r * T:(r + 1) * T, k * Hd:(k + 1) * Hd].contiguous()
            assert torch.equal(o_r.view(torch.int16), want.view(torch.int16)), (k, r)
    assert tsp.tsp_device_status(ws) == tsp.TSP_OK
    L.check_status()
