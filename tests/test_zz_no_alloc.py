"""tsp_mlp_fwd_noalloc: the MLP block for callers that cannot allocate device memory.

Such callers (code running inside an allocator or memory-pool callback, plug-ins of
an application that owns all device memory, runtimes that forbid allocation after
start-up) pass inputs and outputs only; the scratch lives in a static device buffer
of the library. The no-alloc call launches the same two products with the same ring
order as tsp_mlp_fwd, so its output must equal tsp_mlp_fwd's bit for bit; both are
also held to the oracle's bound. This file is collected last so that a run stopping
at its first failure has already run every other test; it also passes alone in a
fresh process.
"""
import numpy as np
import pytest
import torch

import oracle
import tsp_inputs
from gpu_util import Layer, assert_close, dev, f64, rand_bits, stored_mlp

tsp = pytest.importorskip("folded_tensor_sequence_tsp_gb300")
pytestmark = pytest.mark.gpu

# the static buffer: 32 MiB, of which the first 256 bytes hold the status word
SCRATCH_BYTES = (32 << 20) - 256


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    tsp.load_library()


def _both(L, hs):
    """(tsp_mlp_fwd output, tsp_mlp_fwd_noalloc output) for the same input."""
    want = L.act()
    tsp.tsp_mlp_fwd(L.plan, hs, L.wpack, want, L.ws)
    got = torch.full_like(want, float("nan"))
    tsp.tsp_mlp_fwd_noalloc(L.plan, hs, L.wpack, got)
    torch.cuda.synchronize()
    L.check_status()
    return want, got


def _against_oracle(L, h_bits, out, name, rows=None):
    """The MLP is row-wise, so the oracle runs on the input rows in their sharded order."""
    h = oracle.widen_bf16(h_bits if rows is None else h_bits[rows])
    got = f64(out) if rows is None else f64(out)[rows]
    W = L.weights64()
    exact = oracle.swiglu_mlp(h, W["W1"], W["W3"], W["W2"])
    assert_close(got, exact, name, ref=stored_mlp(h, W))


def test_noalloc_mlp_matches_workspace_path_on_two_calls():
    L = Layer(4, 4096, 1024, 16, 2816, seed=17)  # G = 4096 x 2816 bf16 = 22 MiB
    for seed in (101, 102):  # two calls in a row; the second sees the first call's scratch
        h_bits = rand_bits((4096, 1024), seed)
        want, got = _both(L, dev(h_bits))
        assert torch.equal(got.view(torch.int16), want.view(torch.int16)), seed
        _against_oracle(L, h_bits, got, f"noalloc small call {seed - 100}")


def test_later_calls_reserve_no_device_memory():
    """After the first call on the device (which may make the driver reserve the
    static buffer), further calls leave the free device memory unchanged."""
    L = Layer(2, 1024, 512, 8, 1024, seed=19)
    hs = dev(rand_bits((1024, 512), 103))
    out = L.act()
    tsp.tsp_mlp_fwd_noalloc(L.plan, hs, L.wpack, out)
    torch.cuda.synchronize()
    before = torch.cuda.mem_get_info()[0]
    for _ in range(3):
        tsp.tsp_mlp_fwd_noalloc(L.plan, hs, L.wpack, out)
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] == before


def test_noalloc_largest_scratch_that_fits():
    """8188 tokens x 2048 padded ffn columns x 2 bytes = 33,538,048 bytes: the largest
    G of this hidden/ffn grid that fits the 32 MiB - 256 bytes of the buffer. The
    last 128-row tile is partial (T = 4094)."""
    D, S, H, heads, F = 2, 8188, 512, 8, 2048
    L = Layer(D, S, H, heads, F, seed=20)
    assert L.info.tokens * L.info.ffn_padded * 2 <= SCRATCH_BYTES
    assert L.info.tokens * (L.info.ffn_padded + 128) * 2 > SCRATCH_BYTES
    h_bits = rand_bits((S, H), 104)
    want, got = _both(L, dev(h_bits))
    assert torch.equal(got.view(torch.int16), want.view(torch.int16))
    rows = np.sort(np.random.default_rng(20).choice(S, 512, replace=False))
    rows[-1] = S - 1
    _against_oracle(L, h_bits, got, "noalloc largest G (sampled rows)", rows=rows)


def test_noalloc_micro_batch():
    """A micro-batch of 2 sequences (rank-major [D][B][T][H] rows): the ring order of
    the down projection walks each rank's B*T rows, as in tsp_mlp_fwd."""
    L = Layer(2, 2048, 512, 8, 1024, seed=21, batch=2)
    h_bits = rand_bits((L.info.tokens, 512), 105)
    want, got = _both(L, dev(h_bits))
    assert torch.equal(got.view(torch.int16), want.view(torch.int16))
    _against_oracle(L, h_bits, got, "noalloc micro-batch of 2")


def test_noalloc_rejects_shapes_beyond_its_buffer():
    L = Layer(8, 16384, 512, 8, 1024, seed=18, names=["x"])  # G = 16384 x 1024 x 2 = 32 MiB
    out = torch.empty_like(L.d["x"])
    wpack = torch.empty(L.info.wpack_elems, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(tsp.TSPError) as e:
        tsp.tsp_mlp_fwd_noalloc(L.plan, L.d["x"], wpack, out)
    assert e.value.status == tsp.TSP_ERR_UNSUPPORTED
    assert "static buffer" in str(e.value)
