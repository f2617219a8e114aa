"""Helpers shared by the GPU parity tests: moving seeded bf16 bit patterns to the
device and back, and the tolerance check of floating-point outputs.

The bound (bf16 inputs and weights, fp32 accumulation), for every checked output:
  * relative Frobenius error ||got - exact||_F / ||exact||_F <= 1e-2 against the
    exact float64 oracle, and
  * every element of row i within 3e-2 + h(ref) + delta_i of a reference `ref`:
      - h(ref) is half the spacing of bfloat16 values at |ref| for an output stored
        in bf16 (0 for an fp32 output): an output rounded to bf16 cannot be nearer
        than that to any value, and from |y| = 8 on h alone exceeds 3e-2;
      - `ref` is the exact oracle, or the oracle's stored-precision result (the
        same float64 computation with every value a bf16-in / fp32-accumulate
        implementation hands from one product to the next rounded to bf16:
        oracle.layer_forward(..., store=oracle.round_bf16) and the backward's
        counterpart);
      - delta_i = max_j |ref_ij - exact_ij| is how far that stored-precision
        result itself lies from the exact one in row i (0 when ref is exact),
        computed by the oracle alone. Two results that both round the same
        intermediates to bf16 - the oracle's and the kernel's - can lie apart by
        that much: where the kernel's inputs to a rounding differ from the
        oracle's in the last bits (the kernel's P is rounded to bf16, its sums run
        in another order), the bf16 value flips to the neighbouring one. At the
        7B shape the first token's MLP input h flips in 6% of its elements, and
        its output moves by 0.1 in exact arithmetic (delta = 0.11), while typical
        rows have delta of 0.02-0.035 and small shapes 1e-3.
Gradients take the same rule with 3e-2 times the gradient's rms as the absolute
part (the layer outputs' 3e-2 is for activations of rms 1).

Every check records the literal figures against the exact oracle (max |err| and
the number of elements above the absolute bound) and the largest delta_i it
allowed; tests/conftest.py prints them at the end of the session.
"""
import numpy as np
import torch

import oracle
import tsp_inputs

REL_FRO = 1e-2
MAX_ABS = 3e-2

# (name, elements, rel_fro, max|got-exact|, elements above atol vs exact, atol,
#  largest delta_i, max over elements of |got-ref| - bound, rows, rows whose
#  delta_i exceeds atol)  -- one per check, printed by the session summary
RECORDS = []


def dev(bits: np.ndarray) -> torch.Tensor:
    """uint16 bf16 bit patterns -> bf16 CUDA tensor (same bits)."""
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def f64(t: torch.Tensor) -> np.ndarray:
    return oracle.widen_bf16(bits(t))


def half_ulp_bf16(a):
    """Half the spacing of bfloat16 values at |a|: 2^(e-8) for a leading bit of
    weight 2^e, and 2^-134 below the normal range."""
    _, e = np.frexp(np.asarray(a, dtype=np.float64))
    return np.ldexp(1.0, np.maximum(e, -125) - 9)


def errors(got: np.ndarray, want: np.ndarray):
    err = got - want
    rel = float(np.linalg.norm(err) / max(np.linalg.norm(want), 1e-30))
    return rel, float(np.abs(err).max()) if err.size else 0.0


def row_delta(ref, exact):
    """delta_i = max_j |ref_ij - exact_ij| per row (axis 0), shaped to broadcast."""
    if ref is exact or ref.size == 0:
        return 0.0
    d = np.abs(ref - exact)
    if d.ndim < 2:
        return float(d.max())
    return d.reshape(d.shape[0], -1).max(axis=1).reshape((d.shape[0],) + (1,) * (d.ndim - 1))


def assert_close(got, exact, name="", ref=None, atol=MAX_ABS, bf16_out=True,
                 rel_fro=REL_FRO):
    """The bound of this module: rel. Frobenius vs `exact` <= rel_fro, and every
    element within atol + (half a bf16 ulp of |ref| if bf16_out) + delta_i of `ref`
    (default: `exact`, delta = 0). Returns (rel_fro, max |got - exact|)."""
    got = np.asarray(got, dtype=np.float64)
    exact = np.asarray(exact, dtype=np.float64)
    ref = exact if ref is None else np.asarray(ref, dtype=np.float64)
    assert got.shape == exact.shape == ref.shape, (name, got.shape, exact.shape, ref.shape)
    assert np.isfinite(got).all(), f"{name}: non-finite values"
    rel, mx = errors(got, exact)
    n_over = int((np.abs(got - exact) > atol).sum())
    delta = row_delta(ref, exact)
    margin, where = -atol, ""
    if got.size:
        bound = atol + (half_ulp_bf16(ref) if bf16_out else 0.0) + delta
        ex = np.abs(got - ref) - bound
        k = np.unravel_index(int(np.argmax(ex)), ex.shape)
        margin = float(ex[k])
        where = (f" at {tuple(int(i) for i in k)}: ref={ref[k]:.5f} exact={exact[k]:.5f} "
                 f"got={got[k]:.5f} bound={float(np.broadcast_to(bound, ex.shape)[k]):.4f}")
    rows = got.shape[0] if got.ndim else 1
    wide = int((np.asarray(delta) > atol).sum()) if np.ndim(delta) else int(delta > atol)
    RECORDS.append((name, int(got.size), rel, mx, n_over, float(atol),
                    float(np.max(delta)), margin, rows, wide))
    assert rel <= rel_fro and margin <= 0.0, (
        f"{name}: rel_fro={rel:.3e} (<= {rel_fro:g}) max_abs vs exact={mx:.3e} "
        f"({n_over} of {got.size} above {atol:.3g}); worst excess over the bound "
        f"{margin:.3e}{where}")
    return rel, mx


def assert_close_grad(got, exact, name="", ref=None, bf16_out=True):
    """assert_close for a gradient: the absolute part is 3e-2 times the gradient's
    rms (the layer outputs' bound, for activations of rms 1, taken relative to the
    gradient's own size, so that weight gradients - sums over all tokens - are held
    to the same relative accuracy). `ref` as in assert_close: the oracle's
    stored-precision gradient (oracle.layer_backward(..., store=oracle.round_bf16)
    and the block and head backwards' `store`)."""
    exact = np.asarray(exact, dtype=np.float64)
    rms = float(np.sqrt((exact ** 2).mean())) if exact.size else 1.0
    return assert_close(got, exact, name, ref=ref, atol=MAX_ABS * max(rms, 1e-30),
                        bf16_out=bf16_out)


def bf16_round(x):
    """Round float64 values to bfloat16 (nearest, ties to even)."""
    return oracle.round_bf16(x)


def stored_layer(x, W, heads, rows=None):
    """The oracle's layer at bf16 storage precision (see the module docstring)."""
    return oracle.layer_forward(x, W, heads, rows=rows, store=oracle.round_bf16)


def stored_mlp(h, W):
    """The oracle's MLP block with G rounded to bf16 before W2 (h is already bf16)."""
    return oracle.swiglu_mlp(h, W["W1"], W["W3"], W["W2"], store=oracle.round_bf16)


def rand_bits(shape, seed, std=1.0):
    return tsp_inputs.normal_bf16_bits(shape, std, seed, 42)


class Layer:
    """Seeded inputs of one layer shape on the device plus their float64 copies."""

    def __init__(self, D, S, H, heads, F, seed=7, names=None, batch=1):
        import folded_tensor_sequence_tsp_gb300 as tsp
        self.cfg = tsp_inputs.LayerConfig("t", D, S, H, heads, F, seed)
        self.bits = tsp_inputs.layer_inputs(self.cfg, names=names, batch=batch)
        self.plan = (tsp.tsp_plan(D, S, H, heads, F) if batch == 1
                     else tsp.tsp_plan_batched(D, S, batch, H, heads, F))
        self.info = self.plan.info
        self.ws = torch.empty(tsp.tsp_workspace_bytes(self.plan), dtype=torch.uint8, device="cuda")
        tsp.tsp_workspace_init(self.plan, self.ws)
        self.d = {k: dev(v) for k, v in self.bits.items()}
        self.wpack = None
        if names is None or "W2" in names:
            self.wpack = torch.empty(tsp.tsp_packed_weight_bytes(self.plan) // 2,
                                     dtype=torch.bfloat16, device="cuda")
            tsp.tsp_pack_weights(self.plan, *(self.d[k] for k in
                                              ("Wq", "Wk", "Wv", "Wo", "W1", "W3", "W2")),
                                 self.wpack)
        self._f64 = {}

    def f(self, k):
        if k not in self._f64:
            self._f64[k] = oracle.widen_bf16(self.bits[k])
        return self._f64[k]

    def weights64(self):
        return {k: self.f(k) for k in ("Wq", "Wk", "Wv", "Wo", "W1", "W3", "W2")}

    def sharded_x(self):
        import folded_tensor_sequence_tsp_gb300 as tsp
        xs = torch.empty_like(self.d["x"])
        tsp.tsp_shard(self.plan, self.d["x"], xs)
        return xs

    def act(self):
        return torch.empty((self.info.tokens, self.info.hidden), dtype=torch.bfloat16,
                           device="cuda")

    def bwd_workspace(self):
        import folded_tensor_sequence_tsp_gb300 as tsp
        ws = torch.empty(tsp.tsp_bwd_workspace_bytes(self.plan), dtype=torch.uint8, device="cuda")
        tsp.tsp_workspace_init(self.plan, ws)
        self.ws = ws  # check_status reads this workspace's status word from now on
        return ws

    def shard(self, t):
        import folded_tensor_sequence_tsp_gb300 as tsp
        out = torch.empty_like(t)
        tsp.tsp_shard(self.plan, t, out)
        return out

    def unshard(self, t):
        import folded_tensor_sequence_tsp_gb300 as tsp
        out = torch.empty_like(t)
        tsp.tsp_unshard(self.plan, t, out)
        return out

    def grads(self, dwpack):
        """Packed fp32 weight gradients -> dict of float64 arrays (nn.Linear layout)."""
        import folded_tensor_sequence_tsp_gb300 as tsp
        H, F = self.info.hidden, self.info.ffn
        out = {k: torch.empty(shape, dtype=torch.float32, device="cuda") for k, shape in (
            ("dWq", (H, H)), ("dWk", (H, H)), ("dWv", (H, H)), ("dWo", (H, H)),
            ("dW1", (F, H)), ("dW3", (F, H)), ("dW2", (H, F)))}
        tsp.tsp_unpack_weight_grads(self.plan, dwpack, **out)
        return {k: v.cpu().numpy().astype(np.float64) for k, v in out.items()}

    def check_status(self):
        import folded_tensor_sequence_tsp_gb300 as tsp
        assert tsp.tsp_device_status(self.ws) == tsp.TSP_OK, tsp.tsp_last_error()
