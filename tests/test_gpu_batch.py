"""Micro-batches of several sequences on the CUDA path against the float64 oracle.

The page credits TSP's smaller per-device footprint with room for larger
micro-batches ("Folding Tensor and Sequence Parallelism for Memory-Efficient
Transformer Training & Inference", section 4, scalability). A micro-batch plan
holds B independent sequences; every rank owns its zigzag chunks of each of them
(rank-major [D, B, S/D, H]). Checked here: the index map and the shard/unshard
copies bit for bit, the blocks and the layer against the oracle on every
sequence, the batched call bit-identical to one call per sequence, the
7B-shaped layer at 4 x 16K tokens on sampled rows of every sequence, and the
backward: per-sequence input gradients and weight gradients summed over the
micro-batch, against the oracle and against one call per sequence.
"""
import numpy as np
import pytest
import torch

import oracle
import tsp_inputs
from gpu_util import (Layer, assert_close, assert_close_grad, bits, dev, f64, rand_bits,
                      stored_layer, stored_mlp)

tsp = pytest.importorskip("folded_tensor_sequence_tsp_gb300")
pytestmark = pytest.mark.gpu

SHAPES = {
    "tiny-b3": ((2, 256, 256, 4, 688), 3),
    "d3-b2": ((3, 1152, 384, 6, 600), 2),
    "hd128-b2": ((2, 512, 512, 4, 1024), 2),
    "small-b2": ((4, 4096, 1024, 16, 2816), 2),
}


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    tsp.load_library()


def _unshard(L, t):
    """Sharded [D*B*T, H] -> natural [B, S, H]."""
    out = torch.empty_like(t)
    tsp.tsp_unshard(L.plan, t, out)
    return out.view(L.info.batch, L.info.S, L.info.hidden)


def test_index_and_shard_bit_exact():
    for D, S, B in ((2, 256, 3), (3, 1152, 2), (8, 16384, 4), (1, 256, 5)):
        plan = tsp.tsp_plan_batched(D, S, B, 64 * D, D, D)
        fwd = torch.empty(B * S, dtype=torch.int32, device="cuda")
        inv = torch.empty(B * S, dtype=torch.int32, device="cuda")
        tsp.tsp_shard_index(plan, fwd, inv)
        want = oracle.zigzag_forward_index_batched(S, D, B)
        assert np.array_equal(fwd.cpu().numpy(), want), (D, S, B)
        winv = np.empty_like(want)
        winv[want] = np.arange(B * S)
        assert np.array_equal(inv.cpu().numpy(), winv), (D, S, B)
        H = 64 * D
        xb = tsp_inputs.normal_bf16_bits((B, S, H), 1.0, 77, 3)
        x = dev(xb)
        xs = torch.empty_like(x)
        tsp.tsp_shard(plan, x, xs)
        want_s = oracle.shard_tokens_batched(xb, D)
        assert np.array_equal(bits(xs).reshape(want_s.shape), want_s), (D, S, B)
        back = torch.empty_like(x)
        tsp.tsp_unshard(plan, xs, back)
        assert np.array_equal(bits(back), xb)


@pytest.mark.parametrize("name", list(SHAPES))
def test_batched_layer_matches_oracle(name):
    shape, batch = SHAPES[name]
    L = Layer(*shape, seed=21, batch=batch)
    xs = L.sharded_x()
    attn, mlp, out = L.act(), L.act(), L.act()
    tsp.tsp_attention_fwd(L.plan, xs, L.wpack, attn, L.ws)
    tsp.tsp_mlp_fwd(L.plan, xs, L.wpack, mlp, L.ws)
    tsp.tsp_layer_fwd(L.plan, xs, L.wpack, out, L.ws)
    L.check_status()
    W = L.weights64()
    x = L.f("x")
    ref = oracle.layer_forward_batched(x, W, L.info.heads)
    st = oracle.layer_forward_batched(x, W, L.info.heads, store=oracle.round_bf16)
    got_attn, got_mlp, got_out = (f64(_unshard(L, t)) for t in (attn, mlp, out))
    for b in range(batch):
        assert_close(got_attn[b], ref["attn"][b], f"batch {name} seq {b} attn", ref=st["attn"][b])
        want = oracle.swiglu_mlp(x[b], W["W1"], W["W3"], W["W2"])
        assert_close(got_mlp[b], want, f"batch {name} seq {b} mlp", ref=stored_mlp(x[b], W))
        assert_close(got_out[b], ref["out"][b], f"batch {name} seq {b} out", ref=st["out"][b])


@pytest.mark.parametrize("name", ["tiny-b3", "small-b2"])
def test_batched_call_equals_one_call_per_sequence(name):
    """Each output row depends only on its own sequence and takes the same K order
    and key tiles either way, so the micro-batch gives the single-sequence bits."""
    shape, batch = SHAPES[name]
    L = Layer(*shape, seed=22, batch=batch)
    out = L.act()
    tsp.tsp_layer_fwd(L.plan, L.sharded_x(), L.wpack, out, L.ws)
    L.check_status()
    got = bits(_unshard(L, out))
    one = tsp.tsp_plan(*shape)
    ws = torch.empty(tsp.tsp_workspace_bytes(one), dtype=torch.uint8, device="cuda")
    tsp.tsp_workspace_init(one, ws)
    for b in range(batch):
        x = L.d["x"][b].contiguous()
        xs, o, nat = torch.empty_like(x), torch.empty_like(x), torch.empty_like(x)
        tsp.tsp_shard(one, x, xs)
        tsp.tsp_layer_fwd(one, xs, L.wpack, o, ws)
        tsp.tsp_unshard(one, o, nat)
        assert tsp.tsp_device_status(ws) == tsp.TSP_OK
        assert np.array_equal(bits(nat), got[b]), f"sequence {b}"


def test_batched_host_entry_point_matches_device_path():
    shape, batch = SHAPES["d3-b2"]
    L = Layer(*shape, seed=23, batch=batch)
    out = L.act()
    tsp.tsp_layer_fwd(L.plan, L.sharded_x(), L.wpack, out, L.ws)
    want = bits(_unshard(L, out))
    x_host = torch.from_numpy(L.bits["x"].view(np.int16).copy()).view(torch.bfloat16).pin_memory()
    out_host = torch.full_like(x_host, float("nan")).pin_memory()
    tsp.tsp_layer_fwd_host(L.plan, x_host, L.wpack, out_host, L.ws)
    torch.cuda.current_stream().synchronize()
    L.check_status()
    assert np.array_equal(out_host.view(torch.int16).numpy().view(np.uint16), want)


@pytest.mark.slow
def test_7b_16k_micro_batch_of_4_sampled_rows():
    """The 7B-shaped layer on 4 sequences of 16K tokens (65,536 rows, the launch
    configuration the benchmark's micro-batch workload times), 64 sampled rows of
    every sequence against the oracle."""
    cfg = tsp_inputs.config_by_name("7b-16k")
    batch = 4
    L = Layer(cfg.D, cfg.S, cfg.hidden, cfg.heads, cfg.ffn, seed=cfg.seed, batch=batch)
    xs = L.sharded_x()
    out = L.act()
    tsp.tsp_layer_fwd(L.plan, xs, L.wpack, out, L.ws)
    L.check_status()
    nat = _unshard(L, out)
    W = L.weights64()
    x = L.f("x")
    for b in range(batch):
        rows = tsp_inputs.sample_rows(cfg.S, 64, cfg.seed + b)
        got = f64(nat[b][torch.from_numpy(rows).cuda()])
        ref = oracle.layer_forward(x[b], W, cfg.heads, rows=rows)
        st = stored_layer(x[b], W, cfg.heads, rows=rows)
        assert_close(got, ref["out"], f"7b-16k x4 seq {b} out rows", ref=st["out"])


# ---------------------------------------------------------------- backward

def _batched_dout(L, seed):
    b = rand_bits((L.info.tokens, L.info.hidden), seed)
    return b.reshape(L.info.batch, L.info.S, L.info.hidden), dev(b)


@pytest.mark.parametrize("name", list(SHAPES))
def test_batched_layer_backward_matches_oracle(name):
    shape, batch = SHAPES[name]
    L = Layer(*shape, seed=24, batch=batch)
    ws = L.bwd_workspace()
    g_bits, g_dev = _batched_dout(L, 25)
    dxs = L.act()
    dwpack = torch.zeros(L.info.wpack_elems, dtype=torch.float32, device="cuda")
    tsp.tsp_layer_bwd(L.plan, L.sharded_x(), L.wpack, L.shard(g_dev), dxs, dwpack, ws)
    L.check_status()
    got = L.grads(dwpack)
    args = (L.f("x"), L.weights64(), L.info.heads, oracle.widen_bf16(g_bits))
    ref = oracle.layer_backward_batched(*args)
    st = oracle.layer_backward_batched(*args, store=oracle.round_bf16)
    dx = f64(_unshard(L, dxs))
    for b in range(batch):
        assert_close_grad(dx[b], ref["dx"][b], f"batch bwd {name} seq {b} dx", ref=st["dx"][b])
    for k in ("dWq", "dWk", "dWv", "dWo", "dW1", "dW3", "dW2"):
        assert_close_grad(got[k], ref[k], f"batch bwd {name} {k}", ref=st[k], bf16_out=False)


@pytest.mark.parametrize("name", ["tiny-b3", "small-b2"])
def test_batched_backward_equals_one_call_per_sequence(name):
    """Input gradients are row-wise and per sequence: bit-identical to one backward
    per sequence. Weight gradients sum every sequence's tokens in one K loop, so
    they equal the sum of the per-sequence gradients up to fp32 summation order."""
    shape, batch = SHAPES[name]
    L = Layer(*shape, seed=26, batch=batch)
    ws = L.bwd_workspace()
    _, g_dev = _batched_dout(L, 27)
    dxs = L.act()
    dwpack = torch.zeros(L.info.wpack_elems, dtype=torch.float32, device="cuda")
    tsp.tsp_layer_bwd(L.plan, L.sharded_x(), L.wpack, L.shard(g_dev), dxs, dwpack, ws)
    L.check_status()
    got_dx = bits(_unshard(L, dxs))
    one = tsp.tsp_plan(*shape)
    ws1 = torch.empty(tsp.tsp_bwd_workspace_bytes(one), dtype=torch.uint8, device="cuda")
    tsp.tsp_workspace_init(one, ws1)
    S, H = L.info.S, L.info.hidden
    dsum = torch.zeros_like(dwpack)
    for b in range(batch):
        x = L.d["x"][b].contiguous()
        g = g_dev[b * S:(b + 1) * S].contiguous()
        xs, gs, dx1, nat = (torch.empty_like(x) for _ in range(4))
        tsp.tsp_shard(one, x, xs)
        tsp.tsp_shard(one, g, gs)
        dw1 = torch.zeros_like(dwpack)
        tsp.tsp_layer_bwd(one, xs, L.wpack, gs, dx1, dw1, ws1)
        tsp.tsp_unshard(one, dx1, nat)
        assert tsp.tsp_device_status(ws1) == tsp.TSP_OK
        assert np.array_equal(bits(nat), got_dx[b]), f"sequence {b} dx"
        dsum += dw1
    want = dsum.double().cpu().numpy()
    have = dwpack.double().cpu().numpy()
    assert_close_grad(have, want, f"batch bwd {name} packed weight gradients", bf16_out=False)


def test_batched_training_pair_equals_layer_fwd_and_bwd():
    shape, batch = SHAPES["d3-b2"]
    L = Layer(*shape, seed=28, batch=batch)
    ws = L.bwd_workspace()
    _, g_dev = _batched_dout(L, 29)
    xs, dout = L.sharded_x(), L.shard(g_dev)
    out_ref, out_tr = L.act(), L.act()
    tsp.tsp_layer_fwd(L.plan, xs, L.wpack, out_ref, ws)
    saved = torch.full((tsp.tsp_saved_bytes(L.plan),), 0xFF, dtype=torch.uint8, device="cuda")
    tsp.tsp_layer_fwd_train(L.plan, xs, L.wpack, out_tr, saved, ws)
    assert torch.equal(out_ref.view(torch.int16), out_tr.view(torch.int16))
    dxs_ref, dxs_sv = L.act(), L.act()
    dw_ref = torch.zeros(L.info.wpack_elems, dtype=torch.float32, device="cuda")
    dw_sv = torch.full_like(dw_ref, float("nan"))
    tsp.tsp_layer_bwd(L.plan, xs, L.wpack, dout, dxs_ref, dw_ref, ws)
    tsp.tsp_layer_bwd_saved(L.plan, xs, L.wpack, saved, dout, dxs_sv, dw_sv, ws)
    L.check_status()
    assert torch.equal(dxs_ref.view(torch.int16), dxs_sv.view(torch.int16))
    assert torch.equal(dw_ref, dw_sv)
