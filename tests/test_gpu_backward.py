"""Parity of the backward pass against the float64 oracle's chain rule.

Inputs are the seeded layer inputs plus a seeded output gradient (N(0,1), bf16).
Data gradients are compared in natural token order, weight gradients after
unpacking from the packed fp32 layout. Bound (gpu_util.assert_close_grad):
relative Frobenius <= 1e-2 against the exact oracle, and every element within
3e-2 x (the gradient's rms) of the oracle's stored-precision gradient, plus half
a bf16 ulp for the bf16 data gradients, plus that reference's own distance from
the exact gradient in the element's row.
"""
import numpy as np
import pytest
import torch

import oracle
import tsp_inputs
from gpu_util import Layer, assert_close_grad, bf16_round, dev, f64, rand_bits

tsp = pytest.importorskip("folded_tensor_sequence_tsp_gb300")
pytestmark = pytest.mark.gpu

SHAPES = {
    "tiny": (2, 256, 256, 4, 688),
    "ragged": (2, 200, 128, 2, 96),
    "d3": (3, 1152, 384, 6, 600),
    "small": (4, 4096, 1024, 16, 2816),
    "S2": (1, 2, 64, 1, 8),
}


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    tsp.load_library()


def _dout(L, seed):
    b = rand_bits((L.info.S, L.info.hidden), seed)
    return b, dev(b)


@pytest.mark.parametrize("name", list(SHAPES))
def test_mlp_backward_matches_oracle(name):
    L = Layer(*SHAPES[name], seed=21)
    ws = L.bwd_workspace()
    g_bits, g_dev = _dout(L, 22)
    hs, dmlp = L.sharded_x(), L.shard(g_dev)
    dhs = L.act()
    dwpack = torch.zeros(L.info.wpack_elems, dtype=torch.float32, device="cuda")
    tsp.tsp_mlp_bwd(L.plan, hs, L.wpack, dmlp, dhs, dwpack, ws)
    L.check_status()
    got = L.grads(dwpack)
    W = L.weights64()
    args = (L.f("x"), W["W1"], W["W3"], W["W2"], oracle.widen_bf16(g_bits))
    ref = oracle.swiglu_mlp_backward(*args)
    st = oracle.swiglu_mlp_backward(*args, store=bf16_round)
    assert_close_grad(f64(L.unshard(dhs)), ref["dh"], f"mlp bwd {name} dh", ref=st["dh"])
    for k in ("dW1", "dW3", "dW2"):
        assert_close_grad(got[k], ref[k], f"mlp bwd {name} {k}", ref=st[k], bf16_out=False)
    # the attention sections of dwpack are left alone
    i = L.info
    assert not dwpack[: i.wpack_w13].any()


def test_mlp_backward_padding_gradients_are_zero():
    """Padded ffn rows/columns of the packed weights get exactly zero gradient."""
    L = Layer(*SHAPES["tiny"], seed=23)  # F/D = 344 padded to 384
    ws = L.bwd_workspace()
    _, g_dev = _dout(L, 24)
    dhs = L.act()
    dwpack = torch.full((L.info.wpack_elems,), float("nan"), dtype=torch.float32, device="cuda")
    tsp.tsp_mlp_bwd(L.plan, L.sharded_x(), L.wpack, L.shard(g_dev), dhs, dwpack, ws)
    L.check_status()
    i = L.info
    H, NF, Fp, Fd = i.hidden, i.ffn_padded, i.shard_ffn_padded, i.shard_ffn
    w13 = dwpack[i.wpack_w13: i.wpack_w13 + 2 * NF * H].view(NF // 128, 256, H).cpu()
    w2 = dwpack[i.wpack_w2: i.wpack_w2 + H * NF].view(H, NF).cpu()
    fp = torch.arange(NF)
    pad = (fp % Fp) >= Fd
    assert pad.any()
    g13 = w13.view(NF // 128, 2, 128, H)
    pad13 = pad.view(NF // 128, 1, 128).expand(NF // 128, 2, 128)
    assert torch.isfinite(w13).all() and torch.isfinite(w2).all()
    assert (g13[pad13] == 0).all() and (g13[~pad13] != 0).any()
    assert (w2[:, pad] == 0).all()


def test_unpack_weight_grads_inverts_the_packing():
    """Packing bf16 weights, widening to fp32 and unpacking returns the weights."""
    L = Layer(*SHAPES["d3"], seed=25)
    packed32 = L.wpack.float()
    back = L.grads(packed32)
    for k in ("Wq", "Wk", "Wv", "Wo", "W1", "W3", "W2"):
        assert np.array_equal(back["d" + k], L.f(k)), k


# ---------------------------------------------------------------- attention

ATT_SHAPES = {
    "tiny": (2, 256, 256, 4, 688),        # zigzag chunk 64: tiles mix chunks
    "ragged": (2, 200, 128, 2, 96),       # partial last tile
    "d3": (3, 1152, 384, 6, 600),
    "hd128": (2, 512, 512, 4, 1024),      # chunk 128: contiguous tiles, head_dim 128
    "small": (4, 4096, 1024, 16, 2816),
}


def _attention_step(L, k, seed):
    """Synthetic Q (sharded rows), K, V (natural rows), dO (sharded rows) for shard k;
    GPU forward-with-lse then backward. Returns the inputs' bits and dqkv."""
    i = L.info
    S, Hd, H = i.S, i.shard_hidden, i.hidden
    qb, kb, vb = (rand_bits((S, Hd), seed + j) for j in range(3))
    dob = rand_bits((S, H), seed + 3)
    q, kn, vn, do = dev(qb), dev(kb), dev(vb), dev(dob)
    hpr = i.heads // i.D
    o = torch.zeros((S, H), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(hpr * i.stat_stride, dtype=torch.float32, device="cuda")
    delta = torch.empty_like(lse)
    dqkv = torch.zeros((S, 3 * H), dtype=torch.bfloat16, device="cuda")
    tsp.tsp_causal_attention_lse(L.plan, k, q, kn, vn, o, lse, L.ws)
    tsp.tsp_causal_attention_bwd(L.plan, k, q, kn, vn, o, do, lse, delta, dqkv, L.ws)
    L.check_status()
    return (qb, kb, vb, dob), dqkv


@pytest.mark.parametrize("name", list(ATT_SHAPES))
def test_attention_step_backward_matches_oracle(name):
    L = Layer(*ATT_SHAPES[name], seed=31, names=["x"])
    i = L.info
    S, D, Hd, d = i.S, i.D, i.shard_hidden, i.head_dim
    k = D - 1
    (qb, kb, vb, dob), dqkv = _attention_step(L, k, 32)
    q, kk, v, do = (oracle.widen_bf16(b) for b in (qb, kb, vb, dob))
    q_pos = oracle.rank_positions(S, D).reshape(-1)
    k_pos = np.arange(S)
    zig = oracle.zigzag_forward_index(S, D)  # sharded row of each token
    got = f64(dqkv)
    base = 3 * Hd * k
    for j in range(i.heads // D):
        c = slice(j * d, (j + 1) * d)
        args = (q[:, c], kk[:, c], v[:, c], q_pos, k_pos,
                do[:, k * Hd + j * d: k * Hd + (j + 1) * d])
        dq, dk, dv = oracle.causal_attention_head_backward(*args)
        rq, rk, rv = oracle.causal_attention_head_backward(*args, o_round=bf16_round,
                                                           store=bf16_round)
        assert_close_grad(got[:, base + j * d: base + (j + 1) * d], dq,
                          f"attn step bwd {name} dq head {j}", ref=rq)
        assert_close_grad(got[zig, base + Hd + j * d: base + Hd + (j + 1) * d], dk,
                          f"attn step bwd {name} dk head {j}", ref=rk)
        assert_close_grad(got[zig, base + 2 * Hd + j * d: base + 2 * Hd + (j + 1) * d], dv,
                          f"attn step bwd {name} dv head {j}", ref=rv)
    # other shards' columns are untouched
    other = np.ones(3 * i.hidden, bool)
    other[base: base + 3 * Hd] = False
    assert not got[:, other].any()


@pytest.mark.parametrize("name", ["tiny", "ragged", "d3", "hd128", "small"])
def test_attention_block_backward_matches_oracle(name):
    L = Layer(*ATT_SHAPES[name], seed=33)
    ws = L.bwd_workspace()
    g_bits, g_dev = _dout(L, 34)
    dxs = L.act()
    dwpack = torch.zeros(L.info.wpack_elems, dtype=torch.float32, device="cuda")
    tsp.tsp_attention_bwd(L.plan, L.sharded_x(), L.wpack, L.shard(g_dev), dxs, dwpack, ws)
    L.check_status()
    got = L.grads(dwpack)
    W = L.weights64()
    args = (L.f("x"), W["Wq"], W["Wk"], W["Wv"], W["Wo"], L.info.heads, oracle.widen_bf16(g_bits))
    ref = oracle.attention_block_backward(*args)
    st = oracle.attention_block_backward(*args, store=bf16_round)
    assert_close_grad(f64(L.unshard(dxs)), ref["dx"], f"attn bwd {name} dx", ref=st["dx"])
    for k in ("dWq", "dWk", "dWv", "dWo"):
        assert_close_grad(got[k], ref[k], f"attn bwd {name} {k}", ref=st[k], bf16_out=False)
    assert not dwpack[L.info.wpack_w13:].any()  # MLP sections untouched


# ---------------------------------------------------------------- whole layer

@pytest.mark.parametrize("name", ["tiny", "ragged", "d3", "hd128", "small"])
def test_layer_backward_matches_oracle(name):
    L = Layer(*ATT_SHAPES[name], seed=35)
    ws = L.bwd_workspace()
    g_bits, g_dev = _dout(L, 36)
    dxs = L.act()
    dwpack = torch.zeros(L.info.wpack_elems, dtype=torch.float32, device="cuda")
    tsp.tsp_layer_bwd(L.plan, L.sharded_x(), L.wpack, L.shard(g_dev), dxs, dwpack, ws)
    L.check_status()
    got = L.grads(dwpack)
    args = (L.f("x"), L.weights64(), L.info.heads, oracle.widen_bf16(g_bits))
    ref = oracle.layer_backward(*args)
    st = oracle.layer_backward(*args, store=bf16_round)
    assert_close_grad(f64(L.unshard(dxs)), ref["dx"], f"layer bwd {name} dx", ref=st["dx"])
    for k in ("dWq", "dWk", "dWv", "dWo", "dW1", "dW3", "dW2"):
        assert_close_grad(got[k], ref[k], f"layer bwd {name} {k}", ref=st[k], bf16_out=False)


def test_layer_backward_is_the_same_for_every_D():
    """The sharded backward computes the plain layer's gradients for D = 1, 2, 4, 8."""
    S, H, heads, F = 1024, 512, 8, 1024
    outs = {}
    for D in (1, 2, 4, 8):
        L = Layer(D, S, H, heads, F, seed=37)
        ws = L.bwd_workspace()
        g_bits, g_dev = _dout(L, 38)
        dxs = L.act()
        dwpack = torch.zeros(L.info.wpack_elems, dtype=torch.float32, device="cuda")
        tsp.tsp_layer_bwd(L.plan, L.sharded_x(), L.wpack, L.shard(g_dev), dxs, dwpack, ws)
        L.check_status()
        outs[D] = dict(L.grads(dwpack), dx=f64(L.unshard(dxs)))
    args = (L.f("x"), L.weights64(), heads, oracle.widen_bf16(g_bits))
    ref = oracle.layer_backward(*args)
    st = oracle.layer_backward(*args, store=bf16_round)
    for D, g in outs.items():
        for k, want in ref.items():
            assert_close_grad(g[k], want, f"bwd every D: D={D} {k}", ref=st[k],
                              bf16_out=(k == "dx"))


def test_layer_backward_is_deterministic():
    L = Layer(*ATT_SHAPES["small"], seed=39)
    ws = L.bwd_workspace()
    _, g_dev = _dout(L, 40)
    xs, dout = L.sharded_x(), L.shard(g_dev)
    res = []
    for _ in range(2):
        dxs = L.act()
        dwpack = torch.zeros(L.info.wpack_elems, dtype=torch.float32, device="cuda")
        tsp.tsp_layer_bwd(L.plan, xs, L.wpack, dout, dxs, dwpack, ws)
        res.append((dxs.view(torch.int16).clone(), dwpack.clone()))
    L.check_status()
    assert torch.equal(res[0][0], res[1][0]) and torch.equal(res[0][1], res[1][1])


@pytest.mark.parametrize("name", ["tiny", "ragged", "d3", "hd128", "small"])
def test_training_pair_equals_layer_fwd_and_bwd(name):
    """tsp_layer_fwd_train gives tsp_layer_fwd's output bit for bit and keeps o and
    the row statistics; tsp_layer_bwd_saved then gives tsp_layer_bwd's gradients bit
    for bit without running the attention forward again. The kept lse equals the
    forward attention step's lse, and o the attention block's output before W_O."""
    L = Layer(*ATT_SHAPES[name], seed=41)
    ws = L.bwd_workspace()
    _, g_dev = _dout(L, 42)
    xs, dout = L.sharded_x(), L.shard(g_dev)
    out_ref, out_tr = L.act(), L.act()
    tsp.tsp_layer_fwd(L.plan, xs, L.wpack, out_ref, ws)
    saved = torch.full((tsp.tsp_saved_bytes(L.plan),), 0xFF, dtype=torch.uint8, device="cuda")
    tsp.tsp_layer_fwd_train(L.plan, xs, L.wpack, out_tr, saved, ws)
    L.check_status()
    assert torch.equal(out_ref.view(torch.int16), out_tr.view(torch.int16))
    # the kept o: the attention output before W_O, rank-major rows
    i = L.info
    o_kept = saved[: i.S * i.hidden * 2].view(torch.bfloat16).view(i.S, i.hidden)
    lse_off = (i.S * i.hidden * 2 + 255) // 256 * 256
    lse_kept = saved[lse_off: lse_off + i.heads * i.stat_stride * 4].view(torch.float32)
    hpr = i.heads // i.D
    q = torch.empty((i.S, i.shard_hidden), dtype=torch.bfloat16, device="cuda")
    kn, vn = torch.empty_like(q), torch.empty_like(q)
    o = L.act()
    lse = torch.empty(hpr * i.stat_stride, dtype=torch.float32, device="cuda")
    for k in range(i.D):
        tsp.tsp_qkv_projection_gathered(L.plan, k, xs, L.wpack, q, kn, vn, ws)
        tsp.tsp_causal_attention_lse(L.plan, k, q, kn, vn, o, lse, ws)
        seg = lse_kept[k * hpr * i.stat_stride:(k + 1) * hpr * i.stat_stride].view(hpr, i.stat_stride)
        assert torch.equal(seg[:, :i.S], lse.view(hpr, i.stat_stride)[:, :i.S]), k
    L.check_status()
    assert torch.equal(o_kept.view(torch.int16), o.view(torch.int16))
    # backward from the kept activations
    dxs_ref, dxs_sv = L.act(), L.act()
    dw_ref = torch.zeros(i.wpack_elems, dtype=torch.float32, device="cuda")
    dw_sv = torch.full_like(dw_ref, float("nan"))
    tsp.tsp_layer_bwd(L.plan, xs, L.wpack, dout, dxs_ref, dw_ref, ws)
    tsp.tsp_layer_bwd_saved(L.plan, xs, L.wpack, saved, dout, dxs_sv, dw_sv, ws)
    L.check_status()
    assert torch.equal(dxs_ref.view(torch.int16), dxs_sv.view(torch.int16))
    assert torch.equal(dw_ref, dw_sv)


# ---------------------------------------------------------------- 7B shapes, sampled

@pytest.mark.slow
def test_7b_mlp_backward_sampled():
    """MLP backward at the 7B shape and 64K tokens (the benchmark's launch): 256
    sampled rows of dh and 16 sampled ffn indices of dW1, dW3 (rows) and dW2
    (columns), each computed by the oracle over every token."""
    cfg = tsp_inputs.config_by_name("7b-64k")
    L = Layer(cfg.D, cfg.S, cfg.hidden, cfg.heads, cfg.ffn, seed=cfg.seed)
    ws = L.bwd_workspace()
    g_bits, g_dev = _dout(L, 41)
    dhs = L.act()
    dwpack = torch.zeros(L.info.wpack_elems, dtype=torch.float32, device="cuda")
    tsp.tsp_mlp_bwd(L.plan, L.sharded_x(), L.wpack, L.shard(g_dev), dhs, dwpack, ws)
    L.check_status()
    rows = tsp_inputs.sample_rows(cfg.S, 256, cfg.seed)
    got_dh = f64(L.unshard(dhs)[torch.from_numpy(rows).cuda()])
    got = L.grads(dwpack)
    del dhs, dwpack, ws
    cols = np.sort(np.random.default_rng(cfg.seed).choice(cfg.ffn, 16, replace=False))
    W = L.weights64()
    args = (L.f("x"), W["W1"], W["W3"], W["W2"], oracle.widen_bf16(g_bits))
    ref = oracle.swiglu_mlp_backward(*args, rows=rows, ffn_cols=cols)
    st = oracle.swiglu_mlp_backward(*args, rows=rows, ffn_cols=cols, store=bf16_round)
    assert_close_grad(got_dh, ref["dh"], "7b-64k mlp bwd dh rows", ref=st["dh"])
    assert_close_grad(got["dW1"][cols], ref["dW1"], "7b-64k mlp bwd dW1 rows", ref=st["dW1"],
                      bf16_out=False)
    assert_close_grad(got["dW3"][cols], ref["dW3"], "7b-64k mlp bwd dW3 rows", ref=st["dW3"],
                      bf16_out=False)
    # dW2 columns: the oracle returns [H, cols]; rows of the check are W2's rows
    assert_close_grad(got["dW2"][:, cols], ref["dW2"], "7b-64k mlp bwd dW2 columns",
                      ref=st["dW2"], bf16_out=False)


@pytest.mark.slow
def test_7b_attention_step_backward_sampled():
    """Attention backward of one shard (4 heads of 128) at 64K tokens: dq of 256
    sampled query rows for every head, dk/dv of 256 sampled key rows for head 0 (the
    oracle visits every query for those)."""
    cfg = tsp_inputs.config_by_name("7b-64k")
    L = Layer(cfg.D, cfg.S, cfg.hidden, cfg.heads, cfg.ffn, seed=cfg.seed, names=["x"])
    i = L.info
    S, D, Hd, d = i.S, i.D, i.shard_hidden, i.head_dim
    k = D - 1
    (qb, kb, vb, dob), dqkv = _attention_step(L, k, 42)
    q_rows = tsp_inputs.sample_rows(S, 256, cfg.seed)  # sharded rows
    k_rows = tsp_inputs.sample_rows(S, 256, cfg.seed + 1)  # key positions
    zig = oracle.zigzag_forward_index(S, D)
    base = 3 * Hd * k
    got_q = f64(dqkv[torch.from_numpy(q_rows).cuda(), base: base + Hd])
    kz = torch.from_numpy(zig[k_rows]).cuda()
    got_k = f64(dqkv[kz, base + Hd: base + Hd + d])
    got_v = f64(dqkv[kz, base + 2 * Hd: base + 2 * Hd + d])
    del dqkv
    q, kk, v, do = (oracle.widen_bf16(b) for b in (qb, kb, vb, dob))
    q_pos = oracle.rank_positions(S, D).reshape(-1)
    k_pos = np.arange(S)
    for j in range(i.heads // D):
        c = slice(j * d, (j + 1) * d)
        dO = do[:, k * Hd + j * d: k * Hd + (j + 1) * d]
        # dq of a query needs that query's own softmax row only
        args = (q[q_rows, c], kk[:, c], v[:, c], q_pos[q_rows], k_pos, dO[q_rows])
        dq = oracle.causal_attention_head_backward(*args)[0]
        rq = oracle.causal_attention_head_backward(*args, o_round=bf16_round, store=bf16_round)[0]
        assert_close_grad(got_q[:, c], dq, f"7b-64k attn bwd dq head {j}", ref=rq)
    # dk, dv of head 0: every query that sees the sampled keys
    c = slice(0, d)
    dO = do[:, k * Hd: k * Hd + d]
    args = (q[:, c], kk[:, c], v[:, c], q_pos, k_pos, dO, q_rows[:1], k_rows)
    _, dk, dv = oracle.causal_attention_head_backward_rows(*args, q_block=2048)
    _, rk, rv = oracle.causal_attention_head_backward_rows(*args, q_block=2048, o_round=bf16_round,
                                                           store=bf16_round)
    assert_close_grad(got_k, dk, "7b-64k attn bwd dk head 0", ref=rk)
    assert_close_grad(got_v, dv, "7b-64k attn bwd dv head 0", ref=rv)


@pytest.mark.parametrize("name", ["tiny", "small"])
def test_training_step_replays_from_a_cuda_graph(name):
    """The training pair (tsp_layer_fwd_train + tsp_layer_bwd_saved) enqueues only
    kernels on the caller's stream, so one training step can be captured into a CUDA
    graph; replays give the eager output and gradients bit for bit."""
    L = Layer(*ATT_SHAPES[name], seed=43)
    ws = L.bwd_workspace()
    _, g_dev = _dout(L, 44)
    xs, dout = L.sharded_x(), L.shard(g_dev)
    i = L.info
    saved = torch.empty(tsp.tsp_saved_bytes(L.plan), dtype=torch.uint8, device="cuda")
    out_e, dxs_e = L.act(), L.act()
    dw_e = torch.empty(i.wpack_elems, dtype=torch.float32, device="cuda")
    tsp.tsp_layer_fwd_train(L.plan, xs, L.wpack, out_e, saved, ws)
    tsp.tsp_layer_bwd_saved(L.plan, xs, L.wpack, saved, dout, dxs_e, dw_e, ws)
    torch.cuda.synchronize()
    out_g, dxs_g = L.act(), L.act()
    dw_g = torch.empty_like(dw_e)
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            tsp.tsp_layer_fwd_train(L.plan, xs, L.wpack, out_g, saved, ws)
            tsp.tsp_layer_bwd_saved(L.plan, xs, L.wpack, saved, dout, dxs_g, dw_g, ws)
    torch.cuda.current_stream().wait_stream(s)
    for _ in range(2):
        out_g.zero_()
        dxs_g.zero_()
        dw_g.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(out_e.view(torch.int16), out_g.view(torch.int16))
        assert torch.equal(dxs_e.view(torch.int16), dxs_g.view(torch.int16))
        assert torch.equal(dw_e, dw_g)
    L.check_status()
