"""Pins of the oracle to facts fixed outside of itself (CPU only).

Each check is written as a function of the implementation under test so that the
mutation tests at the bottom can plant a mistake in a copy of the oracle (on the
CPU) and show that some pin catches it.

Sources of the pins: hand-worked examples under tests/golden/, closed forms,
special cases that reduce to library routines (torch's scaled_dot_product_attention
and silu, which the oracle does not use), brute force on tiny inputs, and the
invariants stated on the page "Folding Tensor and Sequence Parallelism for
Memory-Efficient Transformer Training & Inference": 1/D of parameters and tokens
per rank (s2 "Unified sharding"), zigzag balancing of causal work (s2, attention
bullets), equal per-device FLOPs, i.e. the sharded layer equals the plain one
(s3 "Theoretical analysis").
"""
import math
import os
import types

import numpy as np
import pytest
import torch

import oracle
import tsp_inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read_golden(name):
    rows = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, vals = line.split(":")
            rows[key.strip()] = [float(v) for v in vals.split()]
    return rows


def _rand(shape, seed, scale=1.0):
    return np.random.default_rng(seed).standard_normal(shape) * scale


def _rand_weights(H, F, seed, scale=0.3):
    rng = np.random.default_rng(seed)
    W = {k: rng.standard_normal((H, H)) * scale for k in ("Wq", "Wk", "Wv", "Wo")}
    W["W1"] = rng.standard_normal((F, H)) * scale
    W["W3"] = rng.standard_normal((F, H)) * scale
    W["W2"] = rng.standard_normal((H, F)) * scale
    return W


def oracle_plain_layer(x, W, heads):
    """The single-sequence plain layer, which the pins above tie to torch's routines;
    the batched pins compare against it, never against a mutant."""
    return oracle.layer_forward(x, W, heads)


# ---------------------------------------------------------------- pin checks

def check_zigzag_golden(o):
    for name, S, D in (("zigzag_S16_D4.txt", 16, 4), ("zigzag_S8_D2.txt", 8, 2)):
        g = _read_golden(name)
        pos = o.rank_positions(S, D)
        for r in range(D):
            assert pos[r].tolist() == [int(v) for v in g[str(r)]], (name, r)


def check_zigzag_bruteforce(o):
    # Build the rank token lists by slicing the sequence into 2D chunks directly.
    for S, D in ((16, 4), (64, 2), (96, 3), (256, 8), (512, 1)):
        C = S // (2 * D)
        chunks = [list(range(c * C, (c + 1) * C)) for c in range(2 * D)]
        want = [chunks[r] + chunks[2 * D - 1 - r] for r in range(D)]
        assert o.rank_positions(S, D).tolist() == want, (S, D)
        fwd = o.zigzag_forward_index(S, D)
        assert sorted(fwd.tolist()) == list(range(S))       # a permutation
        inv = o.zigzag_inverse_index(S, D)
        assert (inv[fwd] == np.arange(S)).all()


def check_zigzag_balance(o):
    # Rank r's queries sit in chunks r and 2D-1-r; a query at position p sees p+1
    # keys, so each rank sees C^2 (2D-1) + C (C+1) pairs: the same for every r.
    for cfg in tsp_inputs.CONFIGS:
        S, D, C = cfg.S, cfg.D, cfg.chunk
        pairs = o.causal_pairs_per_rank(S, D)
        assert (pairs == C * C * (2 * D - 1) + C * (C + 1)).all(), cfg.name
        assert pairs.sum() == S * (S + 1) // 2


def check_shard_roundtrip(o):
    x = _rand((48, 5), 1)
    for D in (1, 2, 3, 4, 6, 8):
        if 48 % (2 * D):
            continue
        xs = o.shard_tokens(x, D)
        assert xs.shape == (D, 48 // D, 5)
        pos = o.rank_positions(48, D)
        assert np.array_equal(xs, x[pos])                    # rank r, row l = token pos[r,l]
        assert np.array_equal(o.unshard_tokens(xs, D), x)
    assert np.array_equal(o.shard_tokens(x, 1)[0], x)       # D = 1: identity


def check_attention_hand_example(o):
    g = _read_golden("attention_hand_example.txt")
    q = np.array([[1.0, 0, 0, 0], [0, 2.0, 0, 0]])
    v = np.array([[1.0, 0, 0, 0], [0, 1.0, 0, 0]])
    out = o.causal_attention_head(q, q.copy(), v, np.arange(2), np.arange(2))
    assert np.allclose(out[0], g["o0"], rtol=0, atol=1e-15)
    assert np.allclose(out[1], g["o1"], rtol=0, atol=1e-15)


def check_attention_vs_sdpa(o):
    # torch's causal scaled_dot_product_attention (float64, CPU) is an independent
    # implementation of the same definition.
    S, heads, d = 37, 3, 8
    q, k, v = (_rand((S, heads * d), s) for s in (2, 3, 4))
    got = o.multihead_causal_attention(q, k, v, heads)
    t = lambda a: torch.from_numpy(a).view(S, heads, d).transpose(0, 1)
    want = torch.nn.functional.scaled_dot_product_attention(t(q), t(k), t(v), is_causal=True)
    want = want.transpose(0, 1).reshape(S, heads * d).numpy()
    assert np.abs(got - want).max() < 1e-12


def check_attention_closed_forms(o):
    S, d = 19, 6
    k, v = _rand((S, d), 5), _rand((S, d), 6)
    # all-zero queries: equal scores, so row i is the mean of v_0..v_i
    out = o.causal_attention_head(np.zeros((S, d)), k, v, np.arange(S), np.arange(S))
    prefix_mean = np.cumsum(v, axis=0) / np.arange(1, S + 1)[:, None]
    assert np.abs(out - prefix_mean).max() < 1e-13
    # query 0 sees only key 0
    q = _rand((S, d), 7)
    out = o.causal_attention_head(q, k, v, np.arange(S), np.arange(S))
    assert np.abs(out[0] - v[0]).max() < 1e-15
    # one dominant key among the visible ones: the output is that key's value
    q = np.zeros((1, d)); q[0, 0] = 1.0
    kk = np.zeros((S, d)); kk[11, 0] = 1e4
    out = o.causal_attention_head(q, kk, v, np.array([15]), np.arange(S))
    assert np.abs(out[0] - v[11]).max() < 1e-12
    # the same dominant key is invisible to an earlier query
    out = o.causal_attention_head(q, kk, v, np.array([9]), np.arange(S))
    assert np.abs(out[0] - v[:10].mean(0)).max() < 1e-13


def check_attention_positions(o):
    # Queries in zigzag order with their global positions give the natural-order
    # result permuted the same way.
    S, D, heads, d = 32, 4, 2, 4
    q, k, v = (_rand((S, heads * d), s) for s in (8, 9, 10))
    nat = o.multihead_causal_attention(q, k, v, heads)
    pos = o.rank_positions(S, D).reshape(-1)
    zz = o.multihead_causal_attention(q[pos], k, v, heads, q_pos=pos, k_pos=np.arange(S))
    assert np.abs(zz - nat[pos]).max() < 1e-13


def check_silu_and_mlp(o):
    assert o.silu(np.array(0.0)) == 0.0
    assert abs(o.silu(np.array(1.0)) - 1.0 / (1.0 + math.exp(-1.0))) < 1e-16
    # hand example H = F = 1: h=2, W1=1, W3=3, W2=0.5 -> 0.5 * silu(2) * 6
    got = o.swiglu_mlp(np.array([[2.0]]), np.array([[1.0]]), np.array([[3.0]]), np.array([[0.5]]))
    assert abs(got[0, 0] - 3.0 * 2.0 / (1.0 + math.exp(-2.0))) < 1e-14
    # against torch's silu (float64): SwiGLU(h) = (silu(h W1^T) * h W3^T) W2^T
    h = _rand((7, 6), 11); W1 = _rand((5, 6), 12); W3 = _rand((5, 6), 13); W2 = _rand((6, 5), 14)
    th = torch.from_numpy
    want = (torch.nn.functional.silu(th(h) @ th(W1).T) * (th(h) @ th(W3).T)) @ th(W2).T
    assert np.abs(o.swiglu_mlp(h, W1, W3, W2) - want.numpy()).max() < 1e-12
    # zero-padded ffn columns contribute nothing (silu(0) * 0 = 0)
    W1p = np.vstack([W1, np.zeros((3, 6))]); W3p = np.vstack([W3, np.zeros((3, 6))])
    W2p = np.hstack([W2, _rand((6, 3), 15)])
    assert np.abs(o.swiglu_mlp(h, W1p, W3p, W2p) - want.numpy()).max() < 1e-12


def check_layer_vs_torch(o):
    # The plain layer against a composition of torch library routines.
    S, H, heads, F = 24, 16, 4, 12
    x = _rand((S, H), 20)
    W = _rand_weights(H, F, 21)
    got = o.layer_forward(x, W, heads)
    th = {k: torch.from_numpy(v) for k, v in W.items()}
    tx = torch.from_numpy(x)
    d = H // heads
    sp = lambda a: a.view(S, heads, d).transpose(0, 1)
    att = torch.nn.functional.scaled_dot_product_attention(
        sp(tx @ th["Wq"].T), sp(tx @ th["Wk"].T), sp(tx @ th["Wv"].T), is_causal=True)
    attn = att.transpose(0, 1).reshape(S, H) @ th["Wo"].T
    h = tx + attn
    mlp = (torch.nn.functional.silu(h @ th["W1"].T) * (h @ th["W3"].T)) @ th["W2"].T
    assert np.abs(got["attn"] - attn.numpy()).max() < 1e-12
    assert np.abs(got["out"] - (h + mlp).numpy()).max() < 1e-12
    # residual structure: Wo = 0 gives h = x; W2 = 0 gives out = h
    W0 = dict(W, Wo=np.zeros_like(W["Wo"]), W2=np.zeros_like(W["W2"]))
    r = o.layer_forward(x, W0, heads)
    assert np.array_equal(r["h"], x) and np.array_equal(r["out"], r["h"])


def check_sampled_rows(o):
    S, H, heads, F = 40, 16, 2, 8
    x = _rand((S, H), 30)
    W = _rand_weights(H, F, 31)
    full = o.layer_forward(x, W, heads)
    rows = np.array([0, 3, 17, 39])
    part = o.layer_forward(x, W, heads, rows=rows)
    for key in ("attn", "h", "mlp", "out"):
        assert np.abs(part[key] - full[key][rows]).max() < 1e-12, key


def check_tsp_equals_plain(o):
    # Equal per-device FLOPs means the sharded schedules compute the plain layer:
    # the TSP output is the same for every D, and D = 1 is the plain layer.
    S, H, heads, F = 64, 32, 8, 48
    x = _rand((S, H), 40)
    W = _rand_weights(H, F, 41)
    plain = o.layer_forward(x, W, heads)
    for D in (1, 2, 4, 8):
        tsp = o.tsp_layer_forward(x, W, heads, D)
        for key in ("attn", "h", "mlp", "out"):
            err = np.abs(tsp[key] - plain[key]).max() / np.abs(plain[key]).max()
            assert err < 1e-12, (D, key, err)


def check_rank_counts(o):
    for cfg in tsp_inputs.CONFIGS:
        H, F, D, S = cfg.hidden, cfg.ffn, cfg.D, cfg.S
        total = 4 * H * H + 3 * H * F       # Wq, Wk, Wv, Wo, W1, W3, W2 element counts
        assert o.rank_parameter_count(H, F, D) * D == total
        assert o.rank_activation_count(S, H, D) * D == S * H
    assert o.layer_flops(4, 2, 3) == 8 * 4 * 4 + 6 * 4 * 2 * 3 + 2 * 2 * 4 * 5


def check_zigzag_batched_golden(o):
    # Rank-major micro-batch layout [D][B][S/D], hand-worked (tests/golden).
    g = _read_golden("zigzag_batched_S8_D2_B2.txt")
    fwd = o.zigzag_forward_index_batched(8, 2, 2)
    inv = np.empty_like(fwd)
    inv[fwd] = np.arange(16)
    for r in range(2):
        for b in range(2):
            blk = inv[(r * 2 + b) * 4:(r * 2 + b + 1) * 4]
            assert blk.tolist() == [int(v) for v in g[f"{r}.{b}"]], (r, b)


def check_zigzag_batched_layout(o):
    for S, D, B in ((16, 4, 3), (64, 2, 2), (96, 3, 5), (48, 1, 2)):
        T = S // D
        fwd = o.zigzag_forward_index_batched(S, D, B)
        assert sorted(fwd.tolist()) == list(range(B * S))          # a permutation
        # every rank holds exactly T tokens of every sequence, at the same positions
        # as the single-sequence map (1/D of each sequence's tokens per rank)
        single = o.rank_positions(S, D)
        for b in range(B):
            rows = fwd[b * S:(b + 1) * S]
            rank = rows // (B * T)
            assert (np.bincount(rank, minlength=D) == T).all()
            assert ((rows // T) % B == b).all()
            for r in range(D):
                mine = np.sort(np.flatnonzero(rank == r))
                assert mine.tolist() == sorted(single[r].tolist())
        assert np.array_equal(o.zigzag_forward_index_batched(S, D, 1),
                              o.zigzag_forward_index(S, D))            # B = 1
        x = _rand((B, S, 3), 60)
        xs = o.shard_tokens_batched(x, D)
        assert xs.shape == (D, B, T, 3)
        for r in range(D):
            for b in range(B):
                assert np.array_equal(xs[r, b], x[b][single[r]])
        assert np.array_equal(o.unshard_tokens_batched(xs, D), x)


def check_tsp_batched_equals_plain(o):
    # A micro-batch through the TSP schedules gives each sequence's plain layer.
    S, H, heads, F, B = 32, 16, 4, 24, 3
    x = _rand((B, S, H), 61)
    W = _rand_weights(H, F, 62)
    plain = [oracle_plain_layer(x[b], W, heads) for b in range(B)]
    batched = o.layer_forward_batched(x, W, heads)
    for D in (1, 2, 4):
        tsp = o.tsp_layer_forward_batched(x, W, heads, D)
        for key in ("attn", "h", "mlp", "out"):
            for b in range(B):
                want = plain[b][key]
                scale = np.abs(want).max()
                assert np.abs(tsp[key][b] - want).max() / scale < 1e-12, (D, key, b)
                assert np.abs(batched[key][b] - want).max() / scale < 1e-12, (key, b)


def check_batched_sequences_independent(o):
    # Changing one sequence of the micro-batch leaves the others' outputs unchanged
    # (no attention across sequences, per-token MLP).
    S, H, heads, F, B, D = 16, 8, 2, 8, 3, 2
    x = _rand((B, S, H), 63)
    W = _rand_weights(H, F, 64)
    a = o.tsp_layer_forward_batched(x, W, heads, D)
    y = x.copy()
    y[1] = _rand((S, H), 65)
    c = o.tsp_layer_forward_batched(y, W, heads, D)
    for b in (0, 2):
        assert np.array_equal(a["out"][b], c["out"][b]), b
    assert not np.allclose(a["out"][1], c["out"][1])


def check_qkv_projection_shard(o):
    # The local projections of broadcast iteration k are x times the rows of heads
    # group k of W_Q, W_K and W_V ([TSP] s2, attention layers: a packed shard per
    # iteration). Pinned to torch's linear on the whole matrices, read per head:
    # the Q | K | V blocks of shard k are heads k*h/D .. (k+1)*h/D - 1 of the full
    # projections, in that order, and the shards together cover every head once.
    S, heads, d = 11, 8, 4
    H = heads * d
    x = _rand((S, H), 90)
    Wq, Wk, Wv = (_rand((H, H), s, 0.3) for s in (91, 92, 93))
    tx = torch.from_numpy(x)
    full = {n: torch.nn.functional.linear(tx, torch.from_numpy(w)).view(S, heads, d).numpy()
            for n, w in (("q", Wq), ("k", Wk), ("v", Wv))}
    for D in (1, 2, 4, 8):
        hpr = heads // D
        seen = np.zeros(heads, int)
        for k in range(D):
            got = o.qkv_projection_shard(x, Wq, Wk, Wv, k, D)
            assert got.shape == (S, 3 * H // D)
            blocks = got.reshape(S, 3, hpr, d)
            for b, n in enumerate("qkv"):
                want = full[n][:, k * hpr:(k + 1) * hpr]
                assert np.abs(blocks[:, b] - want).max() < 1e-12, (D, k, n)
            seen[k * hpr:(k + 1) * hpr] += 1
        assert (seen == 1).all()


def check_round_bf16(o):
    # Against torch's float32 -> bfloat16 conversion (round to nearest even) on
    # values float32 holds exactly, exact ties among them.
    v = np.random.default_rng(94).standard_normal(20000).astype(np.float32) * 5
    v[:8] = [1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -1.0 - 2 ** -8, 0.0, 2.0 ** -130,
             -(2.0 ** -128) * 1.5, 255.5 * 2 ** -7, 3.0e38]
    want = torch.from_numpy(v).to(torch.bfloat16).double().numpy()
    assert np.array_equal(o.round_bf16(v.astype(np.float64)), want)
    # float64 values that float32 cannot hold: the result is a bfloat16 value and no
    # bfloat16 value is nearer (brute force over the two neighbours of its bit
    # pattern); on a tie the pattern is even.
    a = np.random.default_rng(95).standard_normal(20000) * np.exp2(
        np.random.default_rng(96).integers(-20, 20, 20000))
    r = o.round_bf16(a)
    bits = (r.astype(np.float32).view(np.uint32) >> 16).astype(np.int64)
    assert np.array_equal(o.widen_bf16(bits.astype(np.uint16)), r)     # on the grid
    for nb in (bits - 1, bits + 1):
        other = o.widen_bf16((nb & 0xFFFF).astype(np.uint16))
        da, db = np.abs(a - r), np.abs(a - other)
        assert (da <= db).all()
        assert (bits[da == db] % 2 == 0).all()


def check_stored_layer_vs_torch(o):
    # The stored-precision layer (store = round_bf16) against a torch composition
    # that casts to bfloat16 at the same points: Q, K, V, the softmax weights before
    # P V (exp(s - max), unnormalised; the normalising sum unrounded), the attention
    # output before W_O, the MLP input and the gated activation.
    S, H, heads, F = 24, 16, 4, 12
    x = _rand((S, H), 97)
    W = _rand_weights(H, F, 98)
    got = o.layer_forward(x, W, heads, store=o.round_bf16)
    th = {k: torch.from_numpy(v) for k, v in W.items()}
    tx = torch.from_numpy(x)
    b = lambda t: t.to(torch.bfloat16).to(torch.float64)
    d = H // heads
    sp = lambda a: a.view(S, heads, d).transpose(0, 1)
    q, k, v = sp(b(tx @ th["Wq"].T)), sp(b(tx @ th["Wk"].T)), sp(b(tx @ th["Wv"].T))
    sc = (q @ k.transpose(1, 2) / math.sqrt(d)).masked_fill(
        ~torch.ones(S, S, dtype=torch.bool).tril(), float("-inf"))
    e = torch.exp(sc - sc.amax(dim=-1, keepdim=True))
    att = (b(e) @ v) / e.sum(dim=-1, keepdim=True)
    attn = b(att.transpose(0, 1).reshape(S, H)) @ th["Wo"].T
    h = tx + attn
    hb = b(h)
    g = b(torch.nn.functional.silu(hb @ th["W1"].T) * (hb @ th["W3"].T))
    out = h + g @ th["W2"].T
    assert np.abs(got["attn"] - attn.numpy()).max() < 1e-12
    assert np.abs(got["h"] - h.numpy()).max() < 1e-12
    assert np.abs(got["out"] - out.numpy()).max() < 1e-12
    # the identity as `store` is the exact layer; rounding moves it by little
    exact = o.layer_forward(x, W, heads)
    same = o.layer_forward(x, W, heads, store=lambda a: a)
    for key in exact:
        assert np.array_equal(same[key], exact[key]), key
    assert 0 < np.abs(got["out"] - exact["out"]).max() < 0.05 * np.abs(exact["out"]).max()
    # sampled rows of the stored layer are the full stored layer's rows
    rows = np.array([0, 5, 23])
    part = o.layer_forward(x, W, heads, rows=rows, store=o.round_bf16)
    assert np.abs(part["out"] - got["out"][rows]).max() < 1e-12


PINS = [check_zigzag_golden, check_zigzag_bruteforce, check_zigzag_balance,
        check_shard_roundtrip, check_attention_hand_example, check_attention_vs_sdpa,
        check_attention_closed_forms, check_attention_positions, check_silu_and_mlp,
        check_layer_vs_torch, check_sampled_rows, check_tsp_equals_plain, check_rank_counts,
        check_zigzag_batched_golden, check_zigzag_batched_layout, check_tsp_batched_equals_plain,
        check_batched_sequences_independent, check_qkv_projection_shard, check_round_bf16,
        check_stored_layer_vs_torch]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_oracle_pin(pin):
    pin(oracle)


# ------------------------------------------------- planted mistakes (CPU only)

def _mutant(**overrides):
    """A copy of the oracle namespace with some functions replaced."""
    ns = types.SimpleNamespace(**{k: getattr(oracle, k) for k in oracle.__all__})
    for k, v in overrides.items():
        setattr(ns, k, v)
    return ns


def _attn_head_mutant(scale=None, strict=False, shift=0):
    def f(q, k, v, q_pos, k_pos):
        d = q.shape[1]
        s = (q @ k.T) / (scale(d) if scale else math.sqrt(d))
        kp = np.asarray(k_pos)[None, :] + shift
        vis = kp < np.asarray(q_pos)[:, None] if strict else kp <= np.asarray(q_pos)[:, None]
        vis[:, 0] |= ~vis.any(1)          # keep rows non-empty so the maths stays finite
        s = np.where(vis, s, -np.inf)
        p = np.exp(s - s.max(1, keepdims=True))
        return (p @ v) / p.sum(1, keepdims=True)
    return f


def _one_long_sequence(x, W, heads, D):
    """Mistake: the micro-batch treated as one sequence of B*S tokens (later sequences
    attend to earlier ones)."""
    B, S, H = x.shape
    r = oracle.tsp_layer_forward(x.reshape(B * S, H), W, heads, D)
    return {k: v.reshape(B, S, H) for k, v in r.items()}


def _qkv_shifted(x, Wq, Wk, Wv, k, D):
    """Mistake: the heads group of shard k starts one head late (wraps at the end)."""
    heads = 8 if Wq.shape[0] % 8 == 0 else 1
    d = Wq.shape[0] // heads
    roll = lambda w: np.roll(w, -d, axis=0)
    return oracle.qkv_projection_shard(x, roll(Wq), roll(Wk), roll(Wv), k, D)


def _round_ties_away(a):
    """Mistake: halves rounded away from zero instead of to even."""
    a = np.asarray(a, dtype=np.float64)
    _, e = np.frexp(a)
    step = np.ldexp(1.0, np.maximum(e, -125) - 8)
    return np.sign(a) * np.floor(np.abs(a) / step + 0.5) * step


def _stored_layer_mutant(residual_rounded=False, round_g=True):
    def f(x, W, heads, rows=None, store=None):
        if store is None:
            return oracle.layer_forward(x, W, heads, rows=rows)
        attn = oracle.attention_block(x, W["Wq"], W["Wk"], W["Wv"], W["Wo"], heads, rows=rows,
                                      store=store)
        xr = x if rows is None else x[np.asarray(rows)]
        h = xr + attn
        hb = store(h)
        mlp = oracle.swiglu_mlp(hb, W["W1"], W["W3"], W["W2"], store=store if round_g else None)
        base = hb if residual_rounded else h
        return {"attn": attn, "h": h, "mlp": mlp, "out": base + mlp}
    return f


def _run_pins(o):
    failed = 0
    for pin in PINS:
        try:
            pin(o)
        except (AssertionError, ValueError, IndexError):
            failed += 1
    return failed


MUTANTS = {
    "scale 1/d": dict(causal_attention_head=_attn_head_mutant(scale=lambda d: d)),
    "no scale": dict(causal_attention_head=_attn_head_mutant(scale=lambda d: 1.0)),
    "mask excludes diagonal": dict(causal_attention_head=_attn_head_mutant(strict=True)),
    "mask off by one": dict(causal_attention_head=_attn_head_mutant(shift=-1)),
    "silu sign": dict(silu=lambda z: z / (1.0 + np.exp(z))),
    "swiglu gate/up swapped": dict(
        swiglu_mlp=lambda h, W1, W3, W2: ((h @ W1.T) * oracle.silu(h @ W3.T)) @ W2.T),
    "zigzag without fold": dict(rank_positions=lambda S, D: np.arange(S).reshape(D, S // D)),
    "pairs dropped +1": dict(causal_pairs_per_rank=lambda S, D: np.bincount(
        oracle.zigzag_owner(S, D)[0], weights=np.arange(S), minlength=D).astype(np.int64)),
    "micro-batch sequence-major": dict(zigzag_forward_index_batched=lambda S, D, B: (
        np.arange(B)[:, None] * S + oracle.zigzag_forward_index(S, D)[None, :]).reshape(-1)),
    "micro-batch as one sequence": dict(tsp_layer_forward_batched=_one_long_sequence),
    "qkv blocks K|Q|V": dict(qkv_projection_shard=lambda x, Wq, Wk, Wv, k, D: (
        oracle.qkv_projection_shard(x, Wk, Wq, Wv, k, D))),
    "qkv heads group off by one head": dict(qkv_projection_shard=_qkv_shifted),
    "qkv shard of W^T": dict(qkv_projection_shard=lambda x, Wq, Wk, Wv, k, D: (
        oracle.qkv_projection_shard(x, Wq.T, Wk.T, Wv.T, k, D))),
    "bf16 rounding truncates": dict(round_bf16=lambda a: oracle.widen_bf16(
        (np.asarray(a, np.float32).view(np.uint32) >> 16).astype(np.uint16))),
    "bf16 rounding ties away": dict(round_bf16=_round_ties_away),
    "stored h in the residual": dict(layer_forward=_stored_layer_mutant(residual_rounded=True)),
    "stored layer skips G": dict(layer_forward=_stored_layer_mutant(round_g=False)),
}


@pytest.mark.parametrize("name", list(MUTANTS))
def test_planted_mistake_is_caught(name):
    assert _run_pins(_mutant(**MUTANTS[name])) >= 1, f"no pin caught mutant {name!r}"


def test_mutant_in_layer_is_caught():
    """A mistake planted inside the layer (a transposed W_O) fails the torch pin."""
    def bad_attention_block(x, Wq, Wk, Wv, Wo, heads, rows=None):
        return oracle.attention_block(x, Wq, Wk, Wv, Wo.T, heads, rows)

    def bad_layer(x, W, heads, rows=None):
        attn = bad_attention_block(x, W["Wq"], W["Wk"], W["Wv"], W["Wo"], heads, rows)
        xr = x if rows is None else x[np.asarray(rows)]
        h = xr + attn
        mlp = oracle.swiglu_mlp(h, W["W1"], W["W3"], W["W2"])
        return {"attn": attn, "h": h, "mlp": mlp, "out": h + mlp}

    with pytest.raises(AssertionError):
        check_layer_vs_torch(_mutant(layer_forward=bad_layer))


# ------------------------------------------------------- the input generator

def test_bf16_rounding_matches_torch():
    v = np.random.default_rng(50).standard_normal(100000).astype(np.float32) * 3
    v[:4] = [1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -1.0 - 2 ** -8, 0.0]   # exact ties
    ours = tsp_inputs.bf16_bits_from_f32(v)
    theirs = torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, theirs)
    assert np.array_equal(oracle.widen_bf16(ours), torch.from_numpy(v).to(torch.bfloat16).double().numpy())


def test_generator_statistics_and_determinism():
    cfg = tsp_inputs.config_by_name("tiny")
    a = tsp_inputs.layer_inputs(cfg)
    b = tsp_inputs.layer_inputs(cfg)
    assert all(np.array_equal(a[k], b[k]) for k in a)
    x = oracle.widen_bf16(a["x"]); w = oracle.widen_bf16(a["W1"])
    assert a["x"].shape == (256, 256) and a["W1"].shape == (688, 256) and a["W2"].shape == (256, 688)
    assert abs(x.mean()) < 0.02 and abs(x.std() - 1) < 0.02
    assert abs(w.std() - 0.02) < 0.001
    assert not np.array_equal(a["Wq"], a["Wk"])
    rows = tsp_inputs.sample_rows(131072, 256, 7)
    assert rows[0] == 0 and rows[-1] == 131071 and len(rows) == 256
