"""The C-ABI library without a GPU: it loads, exports every declared symbol, and its
host logic (plan validation, derived sizes, argument checks) behaves. No compute
call is made here."""
import ctypes
import os
import subprocess

import pytest

import tsp_inputs

tsp = pytest.importorskip("folded_tensor_sequence_tsp_gb300")
B = tsp._binding


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(B.library_path()):
        import __graft_entry__
        __graft_entry__.build()
    return B.load_library()


def test_library_exports_every_declared_function(lib):
    declared = B.declared_functions()
    assert len(declared) >= 20
    out = subprocess.run(["nm", "-D", "--defined-only", B.library_path()], capture_output=True,
                         text=True, check=True).stdout
    exported = {ln.split()[-1] for ln in out.splitlines() if " T " in ln}
    missing = [f for f in declared if f not in exported]
    assert not missing, missing
    for f in declared:
        assert hasattr(lib, f)
    # the binding wraps every declared call under the same name
    for f in declared:
        if f not in ("tsp_plan_destroy",):
            assert hasattr(tsp, f), f


@pytest.mark.parametrize("cfg", tsp_inputs.CONFIGS, ids=lambda c: c.name)
def test_plan_sizes(lib, cfg):
    p = tsp.tsp_plan(cfg.D, cfg.S, cfg.hidden, cfg.heads, cfg.ffn)
    i = p.info
    assert (i.D, i.S, i.hidden, i.heads, i.ffn) == (cfg.D, cfg.S, cfg.hidden, cfg.heads, cfg.ffn)
    assert i.head_dim == cfg.head_dim and i.T == cfg.S // cfg.D and i.C == cfg.S // (2 * cfg.D)
    assert i.shard_hidden * cfg.D == cfg.hidden and i.shard_ffn * cfg.D == cfg.ffn
    Fp = i.shard_ffn_padded
    assert Fp >= i.shard_ffn and Fp % 64 == 0 and (cfg.D * Fp) % 128 == 0
    assert Fp - i.shard_ffn < 128
    assert i.ffn_padded == cfg.D * Fp
    H = cfg.hidden
    assert i.wpack_qkv == 0 and i.wpack_o == 3 * H * H and i.wpack_w13 == 4 * H * H
    assert i.wpack_w2 == 4 * H * H + 2 * i.ffn_padded * H
    assert i.wpack_elems == i.wpack_w2 + H * i.ffn_padded
    assert tsp.tsp_packed_weight_bytes(p) == 2 * i.wpack_elems
    ws = tsp.tsp_workspace_bytes(p)
    assert ws == i.workspace_bytes and ws % 256 == 0
    # workspace holds at least: status, Q|K|V of the shards of one attention launch,
    # O, h, G, two staging buffers
    S, G = cfg.S, i.attention_group
    assert G >= 1 and cfg.D % G == 0
    need = 256 + 2 * S * ((max(3, G) + 2 * G) * i.shard_hidden + 2 * H + i.ffn_padded + 2 * H) \
        + 4 * S * H
    assert need <= ws <= need + 256 * 10
    # G: the fewest shards per attention launch that give 512 two-tile CTAs
    ctas = -(-cfg.S // 256) * (cfg.heads // cfg.D)
    want = next((g for g in range(1, cfg.D + 1) if cfg.D % g == 0 and ctas * g >= 512), cfg.D)
    assert G == want


@pytest.mark.parametrize("args,code", [
    ((0, 256, 256, 4, 688), B.TSP_ERR_UNSUPPORTED),       # D < 1
    ((3, 256, 256, 4, 688), B.TSP_ERR_UNSUPPORTED),       # S % 2D
    ((2, 256, 256, 3, 688), B.TSP_ERR_UNSUPPORTED),       # hidden % heads
    ((2, 256, 256, 8, 688), B.TSP_ERR_UNSUPPORTED),       # head_dim 32
    ((4, 256, 192, 3, 688), B.TSP_ERR_UNSUPPORTED),       # heads % D
    ((2, 256, 256, 4, 687), B.TSP_ERR_UNSUPPORTED),       # ffn % D
    ((2, 2, 256, 4, 688), B.TSP_ERR_UNSUPPORTED),         # S < 2D
    ((2, 0, 256, 4, 688), B.TSP_ERR_UNSUPPORTED),         # empty sequence
    ((2, -4, 256, 4, 688), B.TSP_ERR_UNSUPPORTED),        # negative length
    ((2, 256, 0, 4, 688), B.TSP_ERR_UNSUPPORTED),         # no hidden width
    ((2, 256, 256, 4, 0), B.TSP_ERR_UNSUPPORTED),         # no ffn
    ((2, 1 << 27, 256, 4, 688), B.TSP_ERR_UNSUPPORTED),   # S too large
    ((65, 130, 64 * 65, 65, 65), B.TSP_ERR_UNSUPPORTED),  # D > 64
])
def test_plan_rejects_unsupported_shapes(lib, args, code):
    h = ctypes.c_void_p()
    assert lib.tsp_plan(*args, ctypes.byref(h)) == code
    assert not h.value
    assert B.tsp_last_error().startswith("tsp_plan")
    with pytest.raises(B.TSPError) as e:
        tsp.tsp_plan(*args)
    assert e.value.status == code


def test_plan_accepts_edge_shapes(lib):
    for args in [(1, 2, 64, 1, 1), (1, 200, 128, 2, 96), (64, 128, 4096, 64, 64),
                 (3, 1152, 384, 6, 600), (8, 131072, 4096, 32, 11008)]:
        p = tsp.tsp_plan(*args)
        assert p.info.D == args[0]


def test_null_and_misaligned_arguments_are_rejected_before_launch(lib):
    p = tsp.tsp_plan(2, 256, 256, 4, 688)
    h = p.handle
    ws = ctypes.c_void_p(1 << 20)  # never dereferenced: validation fails first
    assert lib.tsp_layer_fwd(h, None, ctypes.c_void_p(4096), ctypes.c_void_p(8192), ws, None) \
        == B.TSP_ERR_INVALID_ARG
    assert "null" in B.tsp_last_error()
    assert lib.tsp_layer_fwd(h, ctypes.c_void_p(4100), ctypes.c_void_p(4096),
                             ctypes.c_void_p(8192), ws, None) == B.TSP_ERR_INVALID_ARG
    assert "aligned" in B.tsp_last_error()
    assert lib.tsp_layer_fwd(h, ctypes.c_void_p(4096), ctypes.c_void_p(8192),
                             ctypes.c_void_p(4096), ws, None) == B.TSP_ERR_INVALID_ARG
    assert "alias" in B.tsp_last_error()
    assert lib.tsp_layer_fwd(h, ctypes.c_void_p(4096), ctypes.c_void_p(8192),
                             ctypes.c_void_p(12288), ctypes.c_void_p((1 << 20) + 16), None) \
        == B.TSP_ERR_INVALID_ARG
    assert "256-byte" in B.tsp_last_error()
    assert lib.tsp_qkv_projection(h, 2, ctypes.c_void_p(4096), ctypes.c_void_p(8192),
                                  ctypes.c_void_p(12288), ws, None) == B.TSP_ERR_INVALID_ARG
    assert "shard" in B.tsp_last_error()
    assert lib.tsp_causal_attention(h, -1, ctypes.c_void_p(4096), ctypes.c_void_p(8192),
                                    ctypes.c_void_p(12288), ctypes.c_void_p(16384), ws, None) \
        == B.TSP_ERR_INVALID_ARG
    assert lib.tsp_layer_fwd(None, ctypes.c_void_p(4096), ctypes.c_void_p(8192),
                             ctypes.c_void_p(12288), ws, None) == B.TSP_ERR_INVALID_ARG
    assert lib.tsp_wait_selftest(ws, 0, None) == B.TSP_ERR_INVALID_ARG
    assert lib.tsp_workspace_bytes(None) == 0


def test_binding_checks_tensor_sizes_without_calling_the_library(lib):
    import torch
    p = tsp.tsp_plan(2, 256, 256, 4, 688)
    small = torch.empty(10, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        tsp.tsp_layer_fwd(p, small, small, small, small)


def test_batched_plan_sizes_and_limits(lib):
    """A micro-batch plan: B*S rows everywhere, same weights, backward refused."""
    one = tsp.tsp_plan(4, 4096, 1024, 16, 2816)
    for batch in (1, 2, 3, 8):
        p = tsp.tsp_plan_batched(4, 4096, batch, 1024, 16, 2816)
        i = p.info
        assert i.batch == batch and i.tokens == batch * 4096 and i.S == 4096
        assert i.T == 1024 and i.C == 512
        assert i.wpack_elems == one.info.wpack_elems          # weights do not grow
        assert i.stat_stride == batch * 4096
        # every activation buffer grows with the micro-batch (the attention of fewer
        # shards per launch fills the GPU once the micro-batch adds CTAs)
        assert i.workspace_bytes >= batch * (one.info.workspace_bytes - 256) * \
            (3 + 2 * i.attention_group) / (3 + 2 * one.info.attention_group) * 0.9
        assert i.attention_group <= one.info.attention_group
        assert p.act_elems == batch * 4096 * 1024
    assert tsp.tsp_plan_batched(2, 256, 1, 256, 4, 688).info.tokens == 256
    h = ctypes.c_void_p()
    # T = S/D must be a multiple of 128 for B > 1; batch >= 1; B*S <= 2^26
    assert lib.tsp_plan_batched(2, 200, 2, 256, 4, 688, ctypes.byref(h)) == B.TSP_ERR_UNSUPPORTED
    assert "128" in B.tsp_last_error()
    assert lib.tsp_plan_batched(2, 200, 1, 256, 4, 688, ctypes.byref(h)) == B.TSP_OK
    lib.tsp_plan_destroy(h)
    assert lib.tsp_plan_batched(2, 256, 0, 256, 4, 688, ctypes.byref(h)) == B.TSP_ERR_UNSUPPORTED
    assert lib.tsp_plan_batched(8, 1 << 23, 16, 4096, 32, 11008,
                                ctypes.byref(h)) == B.TSP_ERR_UNSUPPORTED
    # the saved activations of the training pair and the backward workspace grow
    # with the micro-batch too
    p2 = tsp.tsp_plan_batched(4, 4096, 2, 1024, 16, 2816)
    assert tsp.tsp_saved_bytes(p2) >= 2 * 4096 * 1024 * 2 + 16 * 2 * 4096 * 4
    assert tsp.tsp_bwd_workspace_bytes(p2) > 2 * (tsp.tsp_bwd_workspace_bytes(one) - 256 * 40)


def test_header_is_plain_c_and_the_binding_matches_its_structs(tmp_path):
    """include/tsp.h compiles as C99 and C++, and the ctypes structures of the binding
    have the C structures' size and field offsets (a mismatch would corrupt every
    plan-info read)."""
    import shutil
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("no C compiler")
    inc = os.path.dirname(B.HEADER)
    fields = {"tsp_plan_info": [f for f, _ in B.PlanInfo._fields_],
              "tsp_cost": [f for f, _ in B.Cost._fields_]}
    lines = ['#include <stddef.h>', '#include <stdio.h>', '#include "tsp.h"', "int main(void) {"]
    for st, fs in fields.items():
        lines.append(f'  printf("{st} size %zu\\n", sizeof({st}));')
        for f in fs:
            lines.append(f'  printf("{st} {f} %zu\\n", offsetof({st}, {f}));')
    lines += ["  return 0;", "}"]
    src = tmp_path / "layout.c"
    src.write_text("\n".join(lines) + "\n")
    exe = tmp_path / "layout"
    subprocess.run([gcc, "-std=c99", "-Wall", "-Werror", "-I", inc, str(src), "-o", str(exe)],
                   check=True, capture_output=True)
    subprocess.run(["g++", "-fsyntax-only", "-x", "c++", "-I", inc, B.HEADER], check=True,
                   capture_output=True)
    got = {}
    for ln in subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout.splitlines():
        st, f, v = ln.split()
        got[(st, f)] = int(v)
    for st, cls in (("tsp_plan_info", B.PlanInfo), ("tsp_cost", B.Cost)):
        assert got[(st, "size")] == ctypes.sizeof(cls), st
        for f, _ in cls._fields_:
            assert got[(st, f)] == getattr(cls, f).offset, (st, f)


def test_library_links_and_plans_from_c(tmp_path, lib):
    """A plain C program includes tsp.h, links libtsp.so and makes the host-only calls
    (plan, plan info, sizes, cost model, error message) without a GPU."""
    import shutil
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("no C compiler")
    src = tmp_path / "use.c"
    src.write_text(r'''
#include <stdio.h>
#include "tsp.h"
int main(void) {
  tsp_plan_t plan = 0;
  if (tsp_plan(8, 65536, 4096, 32, 11008, &plan) != TSP_OK) return 1;
  tsp_plan_info info;
  if (tsp_get_plan_info(plan, &info) != TSP_OK) return 2;
  printf("%d %lld %zu %zu %d\n", info.D, (long long)info.T, tsp_workspace_bytes(plan),
         tsp_packed_weight_bytes(plan), info.attention_group);
  tsp_plan_destroy(plan);
  tsp_plan_t bad = 0;
  if (tsp_plan(3, 256, 256, 4, 688, &bad) != TSP_ERR_UNSUPPORTED || bad) return 3;
  printf("%s\n", tsp_last_error());
  tsp_cost c;
  if (tsp_cost_model(TSP_SCHEME_TSP, 8, 0, 65536, 4096, 32, 11008, &c) != TSP_OK) return 4;
  printf("%d %.0f\n", c.devices, c.weight_elems);
  return 0;
}
''')
    exe = tmp_path / "use"
    libdir = os.path.dirname(B.library_path())
    subprocess.run([gcc, "-std=c99", "-Wall", "-Werror", "-I", os.path.dirname(B.HEADER), str(src),
                    "-L", libdir, "-ltsp", "-Wl,-rpath," + libdir, "-o", str(exe)],
                   check=True, capture_output=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout.split("\n")
    p = tsp.tsp_plan(8, 65536, 4096, 32, 11008)
    D, T, ws, wp, G = out[0].split()
    assert (int(D), int(T), int(ws), int(wp), int(G)) == (
        8, 8192, tsp.tsp_workspace_bytes(p), tsp.tsp_packed_weight_bytes(p), p.info.attention_group)
    assert out[1].startswith("tsp_plan")
    devices, welems = out[2].split()
    assert int(devices) == 8 and float(welems) == (4 * 4096 * 4096 + 3 * 4096 * 11008) / 8


@pytest.mark.parametrize("shape", [(2, 256, 256, 4, 688), (2, 200, 128, 2, 96),
                                   (3, 1152, 384, 6, 600), (4, 4096, 1024, 16, 2816)],
                         ids=["tiny", "ragged", "d3", "small"])
def test_rank_calls_pass_their_host_checks(lib, shape):
    """Without a GPU the rank-local calls get as far as the tensor-map encoding (the
    first driver call) and no further: every host-side argument check of the call and
    of the kernels it launches accepts the shapes the schedule uses. The pointers are
    aligned placeholders that nothing dereferences here; the test never runs where a
    CUDA device is present."""
    import torch
    if torch.cuda.is_available():
        pytest.skip("placeholder pointers must never reach a GPU")
    p = tsp.tsp_plan(*shape)
    h = p.handle
    P = lambda i: ctypes.c_void_p(1 << (24 + i))   # distinct 16 MiB-aligned placeholders
    ws = P(0)
    calls = {
        "tsp_rank_qkv": lambda: lib.tsp_rank_qkv(h, P(1), P(2), P(3), P(4), ws, None),
        "tsp_rank_attention": lambda: lib.tsp_rank_attention(h, shape[0] - 1, P(1), P(2), P(3),
                                                             P(4), ws, None),
        "tsp_rank_o_accumulate bf16": lambda: lib.tsp_rank_o_accumulate(h, P(1), P(2), P(3), 0,
                                                                        P(4), P(5), ws, None),
        "tsp_rank_o_accumulate fp32": lambda: lib.tsp_rank_o_accumulate(h, P(1), P(2), P(4), 1,
                                                                        P(4), P(5), ws, None),
        "tsp_rank_mlp_step": lambda: lib.tsp_rank_mlp_step(h, P(1), P(2), P(4), P(4), P(5), P(6),
                                                           ws, None),
    }
    for name, call in calls.items():
        st = call()
        msg = B.tsp_last_error()
        assert st == B.TSP_ERR_CUDA and "cuTensorMapEncodeTiled" in msg, (name, st, msg)
    assert lib.tsp_rank_attention(h, shape[0], P(1), P(2), P(3), P(4), ws, None) \
        == B.TSP_ERR_INVALID_ARG
    a, m = tsp.tsp_rank_shard_bytes(p)
    i = p.info
    Fq = (i.shard_ffn_padded + 127) // 128 * 128
    assert a == 2 * 4 * i.hidden * i.shard_hidden
    assert m == 2 * (2 * Fq * i.hidden + i.hidden * i.shard_ffn_padded)


def test_rank_calls_pass_their_host_checks_with_a_micro_batch(lib):
    """The same for a micro-batch of two sequences (a micro-batch plan has S/D a
    multiple of 128, so each rank's rows of every sequence are whole 128-row tiles)."""
    import torch
    if torch.cuda.is_available():
        pytest.skip("placeholder pointers must never reach a GPU")
    p = tsp.tsp_plan_batched(2, 256, 2, 256, 4, 688)
    h = p.handle
    P = lambda i: ctypes.c_void_p(1 << (24 + i))
    ws = P(0)
    for st in (lib.tsp_rank_qkv(h, P(1), P(2), P(3), P(4), ws, None),
               lib.tsp_rank_attention(h, 1, P(1), P(2), P(3), P(4), ws, None),
               lib.tsp_rank_o_accumulate(h, P(1), P(2), P(4), 1, P(4), P(5), ws, None),
               lib.tsp_rank_mlp_step(h, P(1), P(2), P(4), P(4), P(5), P(6), ws, None)):
        assert st == B.TSP_ERR_CUDA and "cuTensorMapEncodeTiled" in B.tsp_last_error()
