"""tsp_mlp_fwd_noalloc: the MLP block for callers that cannot allocate device memory.

Such callers (code running inside an allocator or memory-pool callback, plug-ins of
an application that owns all device memory, runtimes that forbid allocation after
start-up) pass inputs and outputs only; the scratch lives in a static device buffer
of the library. This file is collected last so that a run stopping at its first
failure has already run every other test; it also passes alone in a fresh process.
"""
import pytest
import torch

from gpu_util import Layer, assert_close, dev, f64, rand_bits

tsp = pytest.importorskip("folded_tensor_sequence_tsp_gb300")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    tsp.load_library()


def test_noalloc_mlp_matches_workspace_path_on_two_calls():
    L = Layer(4, 4096, 1024, 16, 2816, seed=17)  # G = 4096 x 2816 bf16 = 22 MiB
    inputs = [dev(rand_bits((4096, 1024), s)) for s in (101, 102)]
    for hs in inputs:  # two calls in a row; the second sees the first call's scratch
        want = L.act()
        tsp.tsp_mlp_fwd(L.plan, hs, L.wpack, want, L.ws)
        got = torch.full_like(want, float("nan"))
        tsp.tsp_mlp_fwd_noalloc(L.plan, hs, L.wpack, got)
        torch.cuda.synchronize()
        assert_close(f64(got), f64(want), "noalloc vs workspace")
    L.check_status()


def test_noalloc_rejects_shapes_beyond_its_buffer():
    L = Layer(8, 16384, 512, 8, 1024, seed=18, names=["x"])  # G = 16384 x 1024 x 2 = 32 MiB
    out = torch.empty_like(L.d["x"])
    wpack = torch.empty(L.info.wpack_elems, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(tsp.TSPError) as e:
        tsp.tsp_mlp_fwd_noalloc(L.plan, L.d["x"], wpack, out)
    assert e.value.status == tsp.TSP_ERR_UNSUPPORTED
    assert "static buffer" in str(e.value)
