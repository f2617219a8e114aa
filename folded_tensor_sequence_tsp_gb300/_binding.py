"""Thin ctypes binding of libtsp.so (declared in include/tsp.h).

Argument marshalling only: each function checks the tensors it is given (device,
dtype, contiguity, size - the C ABI takes raw pointers and cannot check sizes),
passes their pointers and the current CUDA stream, and raises TSPError on a
non-OK status. Every step of the computation runs in the library's kernels; if
the library is not built, loading fails loudly.
"""
from __future__ import annotations

import ctypes
import os
import re

import torch

from . import build as _build

__all__ = [
    "TSPError", "PlanInfo", "Plan", "load_library", "library_path", "declared_functions",
    "TSP_OK", "TSP_ERR_INVALID_ARG", "TSP_ERR_UNSUPPORTED", "TSP_ERR_CUDA", "TSP_ERR_TIMEOUT",
    "tsp_plan", "tsp_plan_batched", "tsp_get_plan_info", "tsp_workspace_bytes", "tsp_packed_weight_bytes",
    "tsp_workspace_init", "tsp_pack_weights", "tsp_shard_index", "tsp_shard", "tsp_unshard",
    "tsp_attention_fwd", "tsp_mlp_fwd", "tsp_mlp_fwd_noalloc", "tsp_layer_fwd", "tsp_layer_fwd_host",
    "tsp_qkv_projection", "tsp_qkv_projection_gathered", "tsp_kv_allgather",
    "tsp_causal_attention", "tsp_causal_attention_q", "tsp_o_projection",
    "tsp_swiglu_gate_up", "tsp_swiglu_down", "tsp_device_status", "tsp_wait_selftest",
    "tsp_last_error", "tsp_bwd_workspace_bytes", "tsp_mlp_bwd", "tsp_unpack_weight_grads",
    "tsp_attention_bwd", "tsp_layer_bwd", "tsp_causal_attention_lse", "tsp_causal_attention_bwd",
    "SCHEMES", "tsp_cost_model", "tsp_cost_model_batched", "tsp_cost_max_batch", "tsp_saved_bytes", "tsp_layer_fwd_train", "tsp_layer_bwd_saved",
    "tsp_rank_shard_bytes", "tsp_pack_rank_shard", "tsp_rank_qkv", "tsp_rank_kv_gather",
    "tsp_rank_attention", "tsp_rank_o_accumulate", "tsp_rank_mlp_step",
]

TSP_OK, TSP_ERR_INVALID_ARG, TSP_ERR_UNSUPPORTED, TSP_ERR_CUDA, TSP_ERR_TIMEOUT = range(5)
_NAMES = {0: "TSP_OK", 1: "TSP_ERR_INVALID_ARG", 2: "TSP_ERR_UNSUPPORTED", 3: "TSP_ERR_CUDA",
          4: "TSP_ERR_TIMEOUT"}

HEADER = os.path.join(_build.ROOT, "include", "tsp.h")


class TSPError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{_NAMES.get(status, status)}: {message}")
        self.status = status


class PlanInfo(ctypes.Structure):
    _fields_ = [
        ("D", ctypes.c_int), ("S", ctypes.c_int64), ("hidden", ctypes.c_int),
        ("heads", ctypes.c_int), ("head_dim", ctypes.c_int), ("ffn", ctypes.c_int),
        ("T", ctypes.c_int64), ("C", ctypes.c_int64), ("shard_hidden", ctypes.c_int),
        ("shard_ffn", ctypes.c_int), ("shard_ffn_padded", ctypes.c_int),
        ("ffn_padded", ctypes.c_int), ("wpack_qkv", ctypes.c_size_t),
        ("wpack_o", ctypes.c_size_t), ("wpack_w13", ctypes.c_size_t),
        ("wpack_w2", ctypes.c_size_t), ("wpack_elems", ctypes.c_size_t),
        ("workspace_bytes", ctypes.c_size_t), ("bwd_workspace_bytes", ctypes.c_size_t),
        ("stat_stride", ctypes.c_int64), ("batch", ctypes.c_int), ("tokens", ctypes.c_int64),
        ("attention_group", ctypes.c_int),
    ]

    def as_dict(self):
        return {k: getattr(self, k) for k, _ in self._fields_}


class Cost(ctypes.Structure):
    _fields_ = [
        ("devices", ctypes.c_int), ("weight_elems", ctypes.c_double),
        ("weight_inflight_elems", ctypes.c_double), ("act_elems", ctypes.c_double),
        ("act_inflight_elems", ctypes.c_double), ("comm_weight_elems", ctypes.c_double),
        ("comm_act_elems", ctypes.c_double), ("flops", ctypes.c_double),
    ]


SCHEMES = {"dp": 0, "tp": 1, "sp": 2, "tp_sp": 3, "tsp": 4}

_lib = None
_P = ctypes.c_void_p
_I = ctypes.c_int
_SIGS = {
    "tsp_plan": (_I, [_I, ctypes.c_int64, _I, _I, _I, ctypes.POINTER(_P)]),
    "tsp_plan_batched": (_I, [_I, ctypes.c_int64, _I, _I, _I, _I, ctypes.POINTER(_P)]),
    "tsp_plan_destroy": (None, [_P]),
    "tsp_get_plan_info": (_I, [_P, ctypes.POINTER(PlanInfo)]),
    "tsp_workspace_bytes": (ctypes.c_size_t, [_P]),
    "tsp_packed_weight_bytes": (ctypes.c_size_t, [_P]),
    "tsp_workspace_init": (_I, [_P, _P, _P]),
    "tsp_pack_weights": (_I, [_P] * 9 + [_P]),
    "tsp_shard_index": (_I, [_P, _P, _P, _P]),
    "tsp_shard": (_I, [_P, _P, _P, _P]),
    "tsp_unshard": (_I, [_P, _P, _P, _P]),
    "tsp_attention_fwd": (_I, [_P] * 6),
    "tsp_mlp_fwd": (_I, [_P] * 6),
    "tsp_mlp_fwd_noalloc": (_I, [_P] * 5),
    "tsp_layer_fwd": (_I, [_P] * 6),
    "tsp_layer_fwd_host": (_I, [_P] * 6),
    "tsp_qkv_projection": (_I, [_P, _I, _P, _P, _P, _P, _P]),
    "tsp_kv_allgather": (_I, [_P] * 5),
    "tsp_qkv_projection_gathered": (_I, [_P, _I] + [_P] * 7),
    "tsp_causal_attention_q": (_I, [_P, _I] + [_P] * 6),
    "tsp_causal_attention": (_I, [_P, _I, _P, _P, _P, _P, _P, _P]),
    "tsp_o_projection": (_I, [_P] * 8),
    "tsp_swiglu_gate_up": (_I, [_P] * 6),
    "tsp_swiglu_down": (_I, [_P] * 8),
    "tsp_device_status": (_I, [_P, _P]),
    "tsp_wait_selftest": (_I, [_P, ctypes.c_uint64, _P]),
    "tsp_last_error": (ctypes.c_char_p, []),
    "tsp_bwd_workspace_bytes": (ctypes.c_size_t, [_P]),
    "tsp_mlp_bwd": (_I, [_P] * 8),
    "tsp_unpack_weight_grads": (_I, [_P] * 10),
    "tsp_attention_bwd": (_I, [_P] * 8),
    "tsp_layer_bwd": (_I, [_P] * 8),
    "tsp_causal_attention_lse": (_I, [_P, _I] + [_P] * 7),
    "tsp_causal_attention_bwd": (_I, [_P, _I] + [_P] * 10),
    "tsp_cost_model": (_I, [_I, _I, _I, ctypes.c_int64, _I, _I, _I, ctypes.POINTER(Cost)]),
    "tsp_cost_model_batched": (_I, [_I, _I, _I, ctypes.c_int64, _I, _I, _I, _I,
                                    ctypes.POINTER(Cost)]),
    "tsp_cost_max_batch": (_I, [_I, _I, _I, ctypes.c_int64, _I, _I, _I, _I, ctypes.c_double,
                                ctypes.POINTER(ctypes.c_int64)]),
    "tsp_saved_bytes": (ctypes.c_size_t, [_P]),
    "tsp_layer_fwd_train": (_I, [_P] * 7),
    "tsp_layer_bwd_saved": (_I, [_P] * 9),
    "tsp_rank_shard_bytes": (_I, [_P, ctypes.POINTER(ctypes.c_size_t), ctypes.POINTER(ctypes.c_size_t)]),
    "tsp_pack_rank_shard": (_I, [_P, _I] + [_P] * 10),
    "tsp_rank_qkv": (_I, [_P] * 7),
    "tsp_rank_kv_gather": (_I, [_P] * 5),
    "tsp_rank_attention": (_I, [_P, _I] + [_P] * 6),
    "tsp_rank_o_accumulate": (_I, [_P, _P, _P, _P, _I, _P, _P, _P, _P]),
    "tsp_rank_mlp_step": (_I, [_P] * 9),
}


def library_path() -> str:
    return _build.LIB


def declared_functions() -> list:
    """Names of the functions include/tsp.h declares."""
    with open(HEADER) as fh:
        text = fh.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(tsp_[a-z0-9_]+)\s*\(", text)))


def load_library():
    """Load libtsp.so (built by __graft_entry__.build()); raise if it is missing."""
    global _lib
    if _lib is not None:
        return _lib
    path = library_path()
    if not os.path.exists(path):
        raise RuntimeError(f"libtsp.so is not built ({path}); run __graft_entry__.build() "
                           "or python -m folded_tensor_sequence_tsp_gb300.build")
    lib = ctypes.CDLL(path)
    for name, (res, args) in _SIGS.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def tsp_last_error() -> str:
    return load_library().tsp_last_error().decode()


def _check(status: int, name: str):
    if status != TSP_OK:
        raise TSPError(status, f"{name}: {tsp_last_error()}")


def _stream(stream):
    if stream is None:
        return _P(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, torch.cuda.Stream):
        return _P(stream.cuda_stream)
    return _P(int(stream))


def _dev(t, name, numel=None, dtype=torch.bfloat16, optional=False):
    """Pointer of a contiguous CUDA tensor of `dtype` with at least `numel` elements."""
    if t is None:
        if optional:
            return _P(None)
        raise ValueError(f"{name} is required")
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if numel is not None and t.numel() < numel:
        raise ValueError(f"{name} holds {t.numel()} elements, needs {numel}")
    return _P(t.data_ptr())


def _host(t, name, numel):
    if not isinstance(t, torch.Tensor) or t.is_cuda or t.dtype != torch.bfloat16:
        raise ValueError(f"{name} must be a bfloat16 CPU tensor")
    if not t.is_contiguous() or t.numel() < numel:
        raise ValueError(f"{name} must be contiguous with {numel} elements")
    return _P(t.data_ptr())


class Plan:
    """Owns a tsp_plan_t handle."""

    def __init__(self, handle, lib):
        self._h = handle
        self._lib = lib
        info = PlanInfo()
        _check(lib.tsp_get_plan_info(handle, ctypes.byref(info)), "tsp_get_plan_info")
        self.info = info

    @property
    def handle(self):
        return self._h

    def __del__(self):
        if getattr(self, "_h", None) and self._lib is not None:
            self._lib.tsp_plan_destroy(self._h)
            self._h = None

    # shapes used by the checks below
    @property
    def act_elems(self):
        return self.info.tokens * self.info.hidden


def tsp_plan(D: int, S: int, hidden: int, heads: int, ffn: int) -> Plan:
    lib = load_library()
    h = _P()
    _check(lib.tsp_plan(D, S, hidden, heads, ffn, ctypes.byref(h)), "tsp_plan")
    return Plan(h, lib)


def tsp_plan_batched(D: int, S: int, batch: int, hidden: int, heads: int, ffn: int) -> Plan:
    """Plan for a micro-batch of `batch` sequences of S tokens (layout [D, B, S/D, H])."""
    lib = load_library()
    h = _P()
    _check(lib.tsp_plan_batched(D, S, batch, hidden, heads, ffn, ctypes.byref(h)),
           "tsp_plan_batched")
    return Plan(h, lib)


def tsp_get_plan_info(plan: Plan) -> dict:
    return plan.info.as_dict()


def tsp_workspace_bytes(plan: Plan) -> int:
    return load_library().tsp_workspace_bytes(plan.handle)


def tsp_packed_weight_bytes(plan: Plan) -> int:
    return load_library().tsp_packed_weight_bytes(plan.handle)


def _ws(plan, ws):
    return _dev(ws, "ws", tsp_workspace_bytes(plan), dtype=torch.uint8)


def _ws_status(ws):
    """Workspace of a single-step call: only its 256-byte status word is used."""
    return _dev(ws, "ws", 256, dtype=torch.uint8)


def tsp_workspace_init(plan, ws, stream=None):
    _check(load_library().tsp_workspace_init(plan.handle, _ws(plan, ws), _stream(stream)),
           "tsp_workspace_init")


def tsp_pack_weights(plan, Wq, Wk, Wv, Wo, W1, W3, W2, wpack, stream=None):
    i = plan.info
    H, F = i.hidden, i.ffn
    args = [_dev(Wq, "Wq", H * H), _dev(Wk, "Wk", H * H), _dev(Wv, "Wv", H * H),
            _dev(Wo, "Wo", H * H), _dev(W1, "W1", F * H), _dev(W3, "W3", F * H),
            _dev(W2, "W2", H * F), _dev(wpack, "wpack", i.wpack_elems)]
    _check(load_library().tsp_pack_weights(plan.handle, *args, _stream(stream)), "tsp_pack_weights")


def tsp_shard_index(plan, fwd, inv, stream=None):
    S = plan.info.tokens
    _check(load_library().tsp_shard_index(
        plan.handle, _dev(fwd, "fwd", S, torch.int32, optional=True),
        _dev(inv, "inv", S, torch.int32, optional=True), _stream(stream)), "tsp_shard_index")


def tsp_shard(plan, x, xs, stream=None):
    n = plan.act_elems
    _check(load_library().tsp_shard(plan.handle, _dev(x, "x", n), _dev(xs, "xs", n),
                                    _stream(stream)), "tsp_shard")


def tsp_unshard(plan, xs, x, stream=None):
    n = plan.act_elems
    _check(load_library().tsp_unshard(plan.handle, _dev(xs, "xs", n), _dev(x, "x", n),
                                      _stream(stream)), "tsp_unshard")


def _block(fn_name, plan, a, wpack, out, ws, stream):
    n = plan.act_elems
    fn = getattr(load_library(), fn_name)
    _check(fn(plan.handle, _dev(a, "input", n), _dev(wpack, "wpack", plan.info.wpack_elems),
              _dev(out, "out", n), _ws(plan, ws), _stream(stream)), fn_name)


def tsp_attention_fwd(plan, xs, wpack, attn, ws, stream=None):
    _block("tsp_attention_fwd", plan, xs, wpack, attn, ws, stream)


def tsp_mlp_fwd(plan, hs, wpack, mlp, ws, stream=None):
    _block("tsp_mlp_fwd", plan, hs, wpack, mlp, ws, stream)


def tsp_mlp_fwd_noalloc(plan, hs, wpack, mlp, stream=None):
    """tsp_mlp_fwd without a workspace, for callers that cannot allocate device memory
    (scratch in the library's static device buffer; see include/tsp.h)."""
    n = plan.act_elems
    _check(load_library().tsp_mlp_fwd_noalloc(
        plan.handle, _dev(hs, "hs", n), _dev(wpack, "wpack", plan.info.wpack_elems),
        _dev(mlp, "mlp", n), _stream(stream)), "tsp_mlp_fwd_noalloc")


def tsp_layer_fwd(plan, xs, wpack, out, ws, stream=None):
    _block("tsp_layer_fwd", plan, xs, wpack, out, ws, stream)


def tsp_layer_fwd_host(plan, x_host, wpack, out_host, ws, stream=None):
    n = plan.act_elems
    _check(load_library().tsp_layer_fwd_host(
        plan.handle, _host(x_host, "x_host", n), _dev(wpack, "wpack", plan.info.wpack_elems),
        _host(out_host, "out_host", n), _ws(plan, ws), _stream(stream)), "tsp_layer_fwd_host")


def tsp_qkv_projection(plan, shard, xs, wpack, qkv, ws, stream=None):
    i = plan.info
    _check(load_library().tsp_qkv_projection(
        plan.handle, int(shard), _dev(xs, "xs", plan.act_elems),
        _dev(wpack, "wpack", i.wpack_elems), _dev(qkv, "qkv", i.tokens * 3 * i.shard_hidden),
        _ws_status(ws), _stream(stream)), "tsp_qkv_projection")


def tsp_qkv_projection_gathered(plan, shard, xs, wpack, q, kn, vn, ws, stream=None):
    i = plan.info
    n = i.tokens * i.shard_hidden
    _check(load_library().tsp_qkv_projection_gathered(
        plan.handle, int(shard), _dev(xs, "xs", plan.act_elems),
        _dev(wpack, "wpack", i.wpack_elems), _dev(q, "q", n), _dev(kn, "kn", n),
        _dev(vn, "vn", n), _ws_status(ws), _stream(stream)), "tsp_qkv_projection_gathered")


def tsp_causal_attention_q(plan, shard, q, kn, vn, o, ws, stream=None):
    i = plan.info
    n = i.tokens * i.shard_hidden
    _check(load_library().tsp_causal_attention_q(
        plan.handle, int(shard), _dev(q, "q", n), _dev(kn, "kn", n), _dev(vn, "vn", n),
        _dev(o, "o", plan.act_elems), _ws_status(ws), _stream(stream)), "tsp_causal_attention_q")


def tsp_kv_allgather(plan, qkv, kn, vn, stream=None):
    i = plan.info
    n = i.tokens * i.shard_hidden
    _check(load_library().tsp_kv_allgather(
        plan.handle, _dev(qkv, "qkv", 3 * n), _dev(kn, "kn", n), _dev(vn, "vn", n),
        _stream(stream)), "tsp_kv_allgather")


def tsp_causal_attention(plan, shard, qkv, kn, vn, o, ws, stream=None):
    i = plan.info
    n = i.tokens * i.shard_hidden
    _check(load_library().tsp_causal_attention(
        plan.handle, int(shard), _dev(qkv, "qkv", 3 * n), _dev(kn, "kn", n), _dev(vn, "vn", n),
        _dev(o, "o", plan.act_elems), _ws_status(ws), _stream(stream)), "tsp_causal_attention")


def tsp_o_projection(plan, o, wpack, residual, out, ws, stream=None, out32=None):
    n = plan.act_elems
    _check(load_library().tsp_o_projection(
        plan.handle, _dev(o, "o", n), _dev(wpack, "wpack", plan.info.wpack_elems),
        _dev(residual, "residual", n, optional=True), _dev(out, "out", n),
        _dev(out32, "out32", n, torch.float32, optional=True), _ws_status(ws),
        _stream(stream)), "tsp_o_projection")


def tsp_swiglu_gate_up(plan, hs, wpack, g, ws, stream=None):
    i = plan.info
    _check(load_library().tsp_swiglu_gate_up(
        plan.handle, _dev(hs, "hs", plan.act_elems), _dev(wpack, "wpack", i.wpack_elems),
        _dev(g, "g", i.tokens * i.ffn_padded), _ws_status(ws), _stream(stream)), "tsp_swiglu_gate_up")


def tsp_swiglu_down(plan, g, wpack, residual, out, ws, stream=None, residual32=None):
    i = plan.info
    n = plan.act_elems
    _check(load_library().tsp_swiglu_down(
        plan.handle, _dev(g, "g", i.tokens * i.ffn_padded), _dev(wpack, "wpack", i.wpack_elems),
        _dev(residual, "residual", n, optional=True),
        _dev(residual32, "residual32", n, torch.float32, optional=True), _dev(out, "out", n),
        _ws_status(ws), _stream(stream)), "tsp_swiglu_down")


def tsp_device_status(ws, stream=None) -> int:
    """Synchronise the stream; return (and clear) the workspace status code."""
    return load_library().tsp_device_status(_dev(ws, "ws", 256, dtype=torch.uint8),
                                            _stream(stream))


def tsp_wait_selftest(ws, limit_ns: int, stream=None):
    _check(load_library().tsp_wait_selftest(_dev(ws, "ws", 256, dtype=torch.uint8),
                                            int(limit_ns), _stream(stream)), "tsp_wait_selftest")


# ------------------------------------------------------------------ backward

def tsp_bwd_workspace_bytes(plan: Plan) -> int:
    return load_library().tsp_bwd_workspace_bytes(plan.handle)


def _ws_bwd(plan, ws):
    return _dev(ws, "ws", tsp_bwd_workspace_bytes(plan), dtype=torch.uint8)


def tsp_mlp_bwd(plan, hs, wpack, dmlp, dhs, dwpack, ws, stream=None):
    """Backward of tsp_mlp_fwd: dhs (bf16, sharded) and the W1/W3/W2 sections of the
    packed fp32 weight gradient dwpack."""
    n = plan.act_elems
    i = plan.info
    _check(load_library().tsp_mlp_bwd(
        plan.handle, _dev(hs, "hs", n), _dev(wpack, "wpack", i.wpack_elems),
        _dev(dmlp, "dmlp", n), _dev(dhs, "dhs", n),
        _dev(dwpack, "dwpack", i.wpack_elems, torch.float32), _ws_bwd(plan, ws),
        _stream(stream)), "tsp_mlp_bwd")


def tsp_unpack_weight_grads(plan, dwpack, dWq=None, dWk=None, dWv=None, dWo=None, dW1=None,
                            dW3=None, dW2=None, stream=None):
    i = plan.info
    H, F = i.hidden, i.ffn
    f32 = torch.float32
    _check(load_library().tsp_unpack_weight_grads(
        plan.handle, _dev(dwpack, "dwpack", i.wpack_elems, f32),
        _dev(dWq, "dWq", H * H, f32, optional=True), _dev(dWk, "dWk", H * H, f32, optional=True),
        _dev(dWv, "dWv", H * H, f32, optional=True), _dev(dWo, "dWo", H * H, f32, optional=True),
        _dev(dW1, "dW1", F * H, f32, optional=True), _dev(dW3, "dW3", F * H, f32, optional=True),
        _dev(dW2, "dW2", H * F, f32, optional=True), _stream(stream)), "tsp_unpack_weight_grads")


def _bwd_block(fn_name, plan, a, wpack, g, dx, dwpack, ws, stream):
    n = plan.act_elems
    i = plan.info
    _check(getattr(load_library(), fn_name)(
        plan.handle, _dev(a, "input", n), _dev(wpack, "wpack", i.wpack_elems),
        _dev(g, "output gradient", n), _dev(dx, "input gradient", n),
        _dev(dwpack, "dwpack", i.wpack_elems, torch.float32), _ws_bwd(plan, ws),
        _stream(stream)), fn_name)


def tsp_attention_bwd(plan, xs, wpack, dattn, dxs, dwpack, ws, stream=None):
    """Backward of tsp_attention_fwd: dxs and the W_Q/W_K/W_V/W_O sections of dwpack."""
    _bwd_block("tsp_attention_bwd", plan, xs, wpack, dattn, dxs, dwpack, ws, stream)


def tsp_layer_bwd(plan, xs, wpack, dout, dxs, dwpack, ws, stream=None):
    """Backward of tsp_layer_fwd: dxs and every section of dwpack."""
    _bwd_block("tsp_layer_bwd", plan, xs, wpack, dout, dxs, dwpack, ws, stream)


def tsp_saved_bytes(plan: Plan) -> int:
    return load_library().tsp_saved_bytes(plan.handle)


def tsp_layer_fwd_train(plan, xs, wpack, out, saved, ws, stream=None):
    """tsp_layer_fwd that also keeps the attention output and row statistics in
    `saved` (a uint8 buffer of tsp_saved_bytes) for tsp_layer_bwd_saved."""
    n = plan.act_elems
    _check(load_library().tsp_layer_fwd_train(
        plan.handle, _dev(xs, "xs", n), _dev(wpack, "wpack", plan.info.wpack_elems),
        _dev(out, "out", n), _dev(saved, "saved", tsp_saved_bytes(plan), dtype=torch.uint8),
        _ws(plan, ws), _stream(stream)), "tsp_layer_fwd_train")


def tsp_layer_bwd_saved(plan, xs, wpack, saved, dout, dxs, dwpack, ws, stream=None):
    """tsp_layer_bwd using the `saved` of tsp_layer_fwd_train (no attention forward)."""
    n = plan.act_elems
    i = plan.info
    _check(load_library().tsp_layer_bwd_saved(
        plan.handle, _dev(xs, "xs", n), _dev(wpack, "wpack", i.wpack_elems),
        _dev(saved, "saved", tsp_saved_bytes(plan), dtype=torch.uint8),
        _dev(dout, "dout", n), _dev(dxs, "dxs", n),
        _dev(dwpack, "dwpack", i.wpack_elems, torch.float32), _ws_bwd(plan, ws),
        _stream(stream)), "tsp_layer_bwd_saved")


def tsp_causal_attention_lse(plan, shard, q, kn, vn, o, lse, ws, stream=None):
    i = plan.info
    n = i.tokens * i.shard_hidden
    nstat = (i.heads // i.D) * i.stat_stride
    _check(load_library().tsp_causal_attention_lse(
        plan.handle, int(shard), _dev(q, "q", n), _dev(kn, "kn", n), _dev(vn, "vn", n),
        _dev(o, "o", plan.act_elems), _dev(lse, "lse", nstat, torch.float32), _ws_status(ws),
        _stream(stream)), "tsp_causal_attention_lse")


def tsp_causal_attention_bwd(plan, shard, q, kn, vn, o, dout, lse, delta, dqkv, ws, stream=None):
    i = plan.info
    n = i.tokens * i.shard_hidden
    nstat = (i.heads // i.D) * i.stat_stride
    _check(load_library().tsp_causal_attention_bwd(
        plan.handle, int(shard), _dev(q, "q", n), _dev(kn, "kn", n), _dev(vn, "vn", n),
        _dev(o, "o", plan.act_elems), _dev(dout, "dout", plan.act_elems),
        _dev(lse, "lse", nstat, torch.float32), _dev(delta, "delta", nstat, torch.float32),
        _dev(dqkv, "dqkv", 3 * plan.act_elems), _ws_status(ws), _stream(stream)),
        "tsp_causal_attention_bwd")


def tsp_cost_model(scheme: str, D: int, S: int, hidden: int, heads: int, ffn: int, tp: int = 0) -> dict:
    """Per-device memory (elements), communication (elements received) and FLOPs of
    one layer forward under `scheme` (dp, tp, sp, tp_sp with a tp x D/tp grid, tsp)."""
    c = Cost()
    _check(load_library().tsp_cost_model(SCHEMES[scheme], D, tp, S, hidden, heads, ffn,
                                         ctypes.byref(c)), "tsp_cost_model")
    return {k: getattr(c, k) for k, _ in Cost._fields_}


def tsp_cost_model_batched(scheme: str, D: int, S: int, batch: int, hidden: int, heads: int,
                           ffn: int, tp: int = 0) -> dict:
    """tsp_cost_model for a micro-batch of `batch` sequences of S tokens."""
    c = Cost()
    _check(load_library().tsp_cost_model_batched(SCHEMES[scheme], D, tp, S, batch, hidden, heads,
                                                 ffn, ctypes.byref(c)), "tsp_cost_model_batched")
    return {k: getattr(c, k) for k, _ in Cost._fields_}


def tsp_cost_max_batch(scheme: str, D: int, S: int, hidden: int, heads: int, ffn: int,
                       layers: int, mem_bytes: float, tp: int = 0) -> int:
    """Largest micro-batch of S-token sequences whose per-device bf16 footprint for
    `layers` layers fits in mem_bytes under `scheme` (0 if one sequence does not)."""
    out = ctypes.c_int64()
    _check(load_library().tsp_cost_max_batch(SCHEMES[scheme], D, tp, S, hidden, heads, ffn,
                                             layers, float(mem_bytes), ctypes.byref(out)),
           "tsp_cost_max_batch")
    return int(out.value)


# ------------------------------------------------------------ rank-local steps

def tsp_rank_shard_bytes(plan: Plan):
    """(attention part, MLP part) bytes of one rank's weight shard."""
    a, m = ctypes.c_size_t(), ctypes.c_size_t()
    _check(load_library().tsp_rank_shard_bytes(plan.handle, ctypes.byref(a), ctypes.byref(m)),
           "tsp_rank_shard_bytes")
    return a.value, m.value


def tsp_pack_rank_shard(plan, k, Wq, Wk, Wv, Wo, W1, W3, W2, attn_shard, mlp_shard, stream=None):
    i = plan.info
    H, F = i.hidden, i.ffn
    a, m = tsp_rank_shard_bytes(plan)
    _check(load_library().tsp_pack_rank_shard(
        plan.handle, int(k), _dev(Wq, "Wq", H * H), _dev(Wk, "Wk", H * H), _dev(Wv, "Wv", H * H),
        _dev(Wo, "Wo", H * H), _dev(W1, "W1", F * H), _dev(W3, "W3", F * H), _dev(W2, "W2", H * F),
        _dev(attn_shard, "attn_shard", a // 2), _dev(mlp_shard, "mlp_shard", m // 2),
        _stream(stream)), "tsp_pack_rank_shard")


def _rank_rows(plan):
    """Rows one rank holds: its T tokens of every sequence of the micro-batch."""
    i = plan.info
    return i.batch * i.T


def tsp_rank_qkv(plan, xs_r, attn_shard, q_r, kv_r, ws, stream=None):
    i = plan.info
    n, Hd = _rank_rows(plan), i.shard_hidden
    _check(load_library().tsp_rank_qkv(
        plan.handle, _dev(xs_r, "xs_r", n * i.hidden),
        _dev(attn_shard, "attn_shard", tsp_rank_shard_bytes(plan)[0] // 2),
        _dev(q_r, "q_r", n * Hd), _dev(kv_r, "kv_r", 2 * n * Hd), _ws_status(ws),
        _stream(stream)), "tsp_rank_qkv")


def tsp_rank_kv_gather(plan, kv_all, kn, vn, stream=None):
    i = plan.info
    n = i.tokens * i.shard_hidden
    _check(load_library().tsp_rank_kv_gather(
        plan.handle, _dev(kv_all, "kv_all", 2 * n), _dev(kn, "kn", n), _dev(vn, "vn", n),
        _stream(stream)), "tsp_rank_kv_gather")


def tsp_rank_attention(plan, r, q_r, kn, vn, o_r, ws, stream=None):
    i = plan.info
    n, nr = i.tokens * i.shard_hidden, _rank_rows(plan) * i.shard_hidden
    _check(load_library().tsp_rank_attention(
        plan.handle, int(r), _dev(q_r, "q_r", nr), _dev(kn, "kn", n), _dev(vn, "vn", n),
        _dev(o_r, "o_r", nr), _ws_status(ws), _stream(stream)), "tsp_rank_attention")


def tsp_rank_o_accumulate(plan, o_r, attn_shard, residual, acc_r, h_r, ws, stream=None):
    """acc_r = residual + o_r W_O,k^T (fp32), h_r = bf16(acc_r). residual: bf16 x_r or
    fp32 (acc_r itself)."""
    i = plan.info
    rows = _rank_rows(plan)
    n = rows * i.hidden
    f32 = residual is not None and residual.dtype == torch.float32
    _check(load_library().tsp_rank_o_accumulate(
        plan.handle, _dev(o_r, "o_r", rows * i.shard_hidden),
        _dev(attn_shard, "attn_shard", tsp_rank_shard_bytes(plan)[0] // 2),
        _dev(residual, "residual", n, torch.float32 if f32 else torch.bfloat16), int(f32),
        _dev(acc_r, "acc_r", n, torch.float32), _dev(h_r, "h_r", n), _ws_status(ws),
        _stream(stream)), "tsp_rank_o_accumulate")


def tsp_rank_mlp_step(plan, h_r, mlp_shard, residual32, acc_r, out_r, g_r, ws, stream=None):
    i = plan.info
    rows = _rank_rows(plan)
    n = rows * i.hidden
    fq = (i.shard_ffn_padded + 127) // 128 * 128
    _check(load_library().tsp_rank_mlp_step(
        plan.handle, _dev(h_r, "h_r", n),
        _dev(mlp_shard, "mlp_shard", tsp_rank_shard_bytes(plan)[1] // 2),
        _dev(residual32, "residual32", n, torch.float32), _dev(acc_r, "acc_r", n, torch.float32),
        _dev(out_r, "out_r", n), _dev(g_r, "g_r", rows * fq), _ws_status(ws), _stream(stream)),
        "tsp_rank_mlp_step")
