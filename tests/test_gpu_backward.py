"""Parity of the backward pass against the float64 oracle's chain rule.

Inputs are the seeded layer inputs plus a seeded output gradient (N(0,1), bf16).
Data gradients are compared in natural token order, weight gradients after
unpacking from the packed fp32 layout. Bound: relative Frobenius <= 1e-2 and each
element within 3e-2 x (the gradient's rms) x row scale + 2^-7 |ref|
(gpu_util.grad_tolerance).
"""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import Layer, assert_close_grad, dev, f64, rand_bits

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
    ref = oracle.swiglu_mlp_backward(L.f("x"), W["W1"], W["W3"], W["W2"],
                                     oracle.widen_bf16(g_bits))
    assert_close_grad(f64(L.unshard(dhs)), ref["dh"], f"{name} dh")
    for k in ("dW1", "dW3", "dW2"):
        assert_close_grad(got[k], ref[k], f"{name} {k}")
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
