"""Failure detection without a GPU fault: a bounded device wait gives up, records
TSP_ERR_TIMEOUT in the workspace status word, and the context stays usable."""
import pytest
import torch

from gpu_util import Layer

tsp = pytest.importorskip("folded_tensor_sequence_tsp_gb300")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    tsp.load_library()


def test_wait_that_runs_out_reports_timeout_and_context_survives():
    L = Layer(2, 256, 256, 4, 688, seed=1)
    assert tsp.tsp_device_status(L.ws) == tsp.TSP_OK
    tsp.tsp_wait_selftest(L.ws, 20_000_000)  # 20 ms on a barrier nothing arrives at
    assert tsp.tsp_device_status(L.ws) == tsp.TSP_ERR_TIMEOUT
    assert "site 8" in tsp.tsp_last_error()
    assert tsp.tsp_device_status(L.ws) == tsp.TSP_OK  # read-and-clear
    # the same context still runs the layer
    xs = L.sharded_x()
    out = L.act()
    tsp.tsp_layer_fwd(L.plan, xs, L.wpack, out, L.ws)
    assert tsp.tsp_device_status(L.ws) == tsp.TSP_OK
    assert torch.isfinite(out.float()).all()


def test_errors_from_a_gpu_process_are_reported_not_raised_in_c():
    L = Layer(2, 256, 256, 4, 688, seed=1)
    qkv = torch.empty((L.info.S, 3 * L.info.shard_hidden), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(tsp.TSPError) as e:
        tsp.tsp_qkv_projection(L.plan, 5, L.d["x"], L.wpack, qkv, L.ws)
    assert e.value.status == tsp.TSP_ERR_INVALID_ARG
