"""Oracle for the TSP layer, forward and backward. TEST INFRASTRUCTURE ONLY.

A plain, slow, float64 NumPy restatement of what one transformer layer computes
under Folding Tensor and Sequence Parallelism (TSP). Only the test suite, the
package smoke check and the benchmark's CPU-baseline / reference legs may import
this module; the library never does. It shares no code with the CUDA path: the
only thing both sides take from elsewhere is the seeded input generator, which
holds none of the method's arithmetic.

Source, cited below as [TSP]: the summary page "Folding Tensor and Sequence
Parallelism for Memory-Efficient Transformer Training & Inference"
(gist.science, paper 2604.26294), sections 1 (Problem statement),
2 (Methodology) and 3 (Contributions).

What the page fixes, and what this module writes out:
  * each of D ranks holds 1/D of the parameters and 1/D of the sequence tokens
    ([TSP] s2, "Unified sharding");
  * attention runs a broadcast schedule over packed W_Q/W_K/W_V/W_O shards:
    local projections on each rank's own tokens, an all-gather of K/V along the
    sequence, then FlashAttention ([TSP] s2, "Attention layers");
  * zigzag partitioning balances causal attention work ([TSP] s2, same bullet list);
  * the gated MLP runs a ring schedule over W1/W2/W3 shards and each rank
    accumulates its partial outputs locally, with no all-reduce
    ([TSP] s2, "Gated MLP layers");
  * per-device FLOPs equal those of tensor/sequence parallelism ([TSP] s3,
    "Theoretical analysis" - FLOPs), i.e. the sharded layer computes the plain
    layer's result.

Readings taken where the page is silent (each is listed in the design notes):
  * no normalisation, no positional encoding, no dropout; a micro-batch is B
    independent sequences (each rank owns its zigzag chunks of every sequence);
  * softmax scale 1/sqrt(head_dim); causal mask j <= i over global positions,
    diagonal included;
  * W1 = gate (through SiLU), W3 = up, W2 = down; silu(z) = z / (1 + e^-z);
  * a layer is  h = x + Attn(x),  out = h + MLP(h); the block functions return
    the block outputs without the residual;
  * zigzag: the sequence is cut into 2D equal chunks of C = S/(2D) tokens and
    rank r owns chunks r and 2D-1-r, in that local order;
  * attention weight shard k = heads [k*h/D, (k+1)*h/D): the matching rows of
    W_Q, W_K, W_V and columns of W_O; MLP shard k = ffn slice [k*F/D, (k+1)*F/D):
    rows of W1, W3 and columns of W2;
  * broadcast iteration k uses shard k; at ring step t rank r holds shard
    (r + t) mod D;
  * the O projection is reduced like the MLP: each rank accumulates its partial
    products over k locally.

Everything is computed in float64 from the bfloat16 bit patterns of the inputs.
"""
from __future__ import annotations

import math

import numpy as np

__all__ = [
    "widen_bf16",
    "round_bf16",
    "zigzag_owner",
    "zigzag_forward_index",
    "zigzag_inverse_index",
    "shard_tokens",
    "unshard_tokens",
    "rank_positions",
    "causal_attention_head",
    "multihead_causal_attention",
    "attention_block",
    "silu",
    "swiglu_gate",
    "swiglu_mlp",
    "qkv_projection_shard",
    "layer_forward",
    "tsp_layer_forward",
    "zigzag_forward_index_batched",
    "shard_tokens_batched",
    "unshard_tokens_batched",
    "layer_forward_batched",
    "tsp_layer_forward_batched",
    "silu_grad",
    "causal_attention_head_backward",
    "causal_attention_head_backward_rows",
    "swiglu_mlp_backward",
    "attention_block_backward",
    "layer_backward",
    "layer_backward_batched",
    "tsp_layer_backward",
    "causal_pairs_per_rank",
    "layer_flops",
    "rank_parameter_count",
    "rank_activation_count",
]


def widen_bf16(bits: np.ndarray) -> np.ndarray:
    """bfloat16 bit patterns (uint16) -> float64 values (exact widening)."""
    b = np.ascontiguousarray(bits).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32).astype(np.float64)


BF16_MAX = (2.0 - 2.0 ** -7) * 2.0 ** 127


def round_bf16(a) -> np.ndarray:
    """The bfloat16 value nearest to each element, ties to the even significand.

    bfloat16 keeps 8 significant bits and float32's exponent range, so a value
    whose leading bit has weight 2^e is rounded to a multiple of 2^(e-7); below
    the normal range (e < -126) the spacing stays 2^-133. Rounded straight from
    float64 (no intermediate float32). Used only for the stored-precision variant
    of the layer (`store=round_bf16` below): the values a bf16-in / fp32-accumulate
    implementation hands from one product to the next are bf16.
    """
    a = np.asarray(a, dtype=np.float64)
    _, e = np.frexp(a)                      # a = m 2^e, 1/2 <= |m| < 1: leading bit 2^(e-1)
    step = np.ldexp(1.0, np.maximum(e, -125) - 8)
    r = np.round(a / step) * step           # np.round: halves go to the even integer
    return np.where(np.abs(r) > BF16_MAX, np.copysign(np.inf, a), r)


# --------------------------------------------------------------------------
# Zigzag sequence partitioning  ([TSP] s2, "Attention layers", last bullet)
# --------------------------------------------------------------------------

def zigzag_owner(S: int, D: int):
    """Rank and rank-local index of every global token position.

    The sequence is cut into 2D chunks of C = S/(2D) tokens. Chunk c < D goes to
    rank c (local rows 0..C-1); chunk c >= D goes to rank 2D-1-c (local rows
    C..2C-1). Returns (rank[S], local[S]) as int64 arrays.
    """
    if S % (2 * D):
        raise ValueError("S must be a multiple of 2D")
    C = S // (2 * D)
    t = np.arange(S, dtype=np.int64)
    chunk, off = t // C, t % C
    first = chunk < D
    rank = np.where(first, chunk, 2 * D - 1 - chunk)
    local = np.where(first, off, C + off)
    return rank, local


def zigzag_forward_index(S: int, D: int) -> np.ndarray:
    """fwd[t] = row of global token t in the rank-major [D, S/D] layout."""
    rank, local = zigzag_owner(S, D)
    return rank * (S // D) + local


def zigzag_inverse_index(S: int, D: int) -> np.ndarray:
    """inv[row] = global position of row `row` of the rank-major layout."""
    fwd = zigzag_forward_index(S, D)
    inv = np.empty_like(fwd)
    inv[fwd] = np.arange(S, dtype=np.int64)
    return inv


def shard_tokens(x: np.ndarray, D: int) -> np.ndarray:
    """[S, ...] natural order -> [D, S/D, ...]: rank r's tokens in local order."""
    S = x.shape[0]
    out = np.empty_like(x)
    out[zigzag_forward_index(S, D)] = x
    return out.reshape((D, S // D) + x.shape[1:])


def unshard_tokens(xs: np.ndarray, D: int) -> np.ndarray:
    """Inverse of shard_tokens: [D, S/D, ...] -> [S, ...] in natural order."""
    S = xs.shape[0] * xs.shape[1]
    flat = xs.reshape((S,) + xs.shape[2:])
    return flat[zigzag_forward_index(S, D)]


def rank_positions(S: int, D: int) -> np.ndarray:
    """[D, S/D]: global position of each rank's local token."""
    return zigzag_inverse_index(S, D).reshape(D, S // D)


# --------------------------------------------------------------------------
# Causal attention  ([TSP] s2, "Attention layers": FlashAttention over the
# gathered K/V; FlashAttention computes exact softmax attention)
# --------------------------------------------------------------------------

def causal_attention_head(q, k, v, q_pos, k_pos, store=None) -> np.ndarray:
    """One head: out_i = sum_j p_ij v_j / sum_j p_ij over keys with k_pos[j] <= q_pos[i].

    p_ij = exp(s_ij - max_j s_ij), s_ij = q_i . k_j / sqrt(d). q: [nq, d],
    k, v: [nk, d], positions int arrays. float64 throughout. With `store` (e.g.
    round_bf16) the weights p_ij pass through it before the product with v (the sum
    in the denominator stays unrounded), as when P is handed to the P V product in
    bf16.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    d = q.shape[1]
    s = (q @ k.T) / math.sqrt(d)
    visible = np.asarray(k_pos)[None, :] <= np.asarray(q_pos)[:, None]
    s = np.where(visible, s, -np.inf)
    m = s.max(axis=1, keepdims=True)
    p = np.exp(s - m)
    return ((p if store is None else store(p)) @ v) / p.sum(axis=1, keepdims=True)


def multihead_causal_attention(q, k, v, heads: int, q_pos=None, k_pos=None,
                               q_block: int = 1024, store=None) -> np.ndarray:
    """Split the H columns into `heads` heads of d = H/heads and attend per head.

    q: [nq, H], k, v: [nk, H]; positions default to 0..n-1. Queries are taken in
    blocks of `q_block` rows only to bound the score matrix's memory. `store` as in
    causal_attention_head.
    """
    nq, H = q.shape
    nk = k.shape[0]
    d = H // heads
    q_pos = np.arange(nq) if q_pos is None else np.asarray(q_pos)
    k_pos = np.arange(nk) if k_pos is None else np.asarray(k_pos)
    out = np.empty((nq, H), dtype=np.float64)
    for j in range(heads):
        c = slice(j * d, (j + 1) * d)
        for lo in range(0, nq, q_block):
            r = slice(lo, min(nq, lo + q_block))
            out[r, c] = causal_attention_head(q[r, c], k[:, c], v[:, c], q_pos[r], k_pos, store)
    return out


def attention_block(x, Wq, Wk, Wv, Wo, heads: int, rows=None, store=None) -> np.ndarray:
    """Causal multi-head self-attention of a plain (unsharded) layer, no residual.

    Attn(x) = concat_j softmax(Q_j K_j^T / sqrt(d) + causal) V_j  W_O^T with
    Q = x W_Q^T, K = x W_K^T, V = x W_V^T. All inputs float64 arrays.
    With `rows` (sorted positions) only those output rows are computed; K/V are
    projected for positions 0..max(rows), one head at a time.
    With `store` (a function of an array, e.g. round_bf16), the values one product
    hands to the next are passed through it: Q, K and V, the softmax weights P before
    P V, and the per-head attention output before W_O. Without it everything stays
    float64.
    """
    st = (lambda a: a) if store is None else store
    S, H = x.shape
    d = H // heads
    if rows is None:
        rows = np.arange(S)
    rows = np.asarray(rows, dtype=np.int64)
    kmax = int(rows.max()) + 1
    xk = x[:kmax]
    xq = x[rows]
    o = np.empty((rows.size, H), dtype=np.float64)
    for j in range(heads):
        c = slice(j * d, (j + 1) * d)
        qh = st(xq @ Wq[c].T)
        kh = st(xk @ Wk[c].T)
        vh = st(xk @ Wv[c].T)
        for lo in range(0, rows.size, 1024):
            r = slice(lo, min(rows.size, lo + 1024))
            o[r, c] = causal_attention_head(qh[r], kh, vh, rows[r], np.arange(kmax), store)
    return st(o) @ Wo.T


# --------------------------------------------------------------------------
# Gated MLP  ([TSP] s2, "Gated MLP layers": weights W1, W2, W3)
# --------------------------------------------------------------------------

def silu(z):
    """SiLU(z) = z * sigmoid(z) = z / (1 + exp(-z))."""
    return z / (1.0 + np.exp(-z))


def swiglu_gate(h, W1, W3) -> np.ndarray:
    """Gated activation G = silu(h W1^T) * (h W3^T)."""
    return silu(h @ W1.T) * (h @ W3.T)


def swiglu_mlp(h, W1, W3, W2, store=None) -> np.ndarray:
    """MLP(h) = (silu(h W1^T) * (h W3^T)) W2^T, no residual.

    With `store`, the gated activation G is passed through it before W2 (the value
    the first product hands to the second)."""
    G = swiglu_gate(h, W1, W3)
    return (G if store is None else store(G)) @ W2.T


def qkv_projection_shard(x, Wq, Wk, Wv, k: int, D: int) -> np.ndarray:
    """Local projections of broadcast iteration k ([TSP] s2, attention layers).

    x times the rows of heads group k ([k H/D, (k+1) H/D)) of W_Q, W_K and W_V;
    returns [n, 3H/D] laid out as Q | K | V.
    """
    Hd = Wq.shape[0] // D
    c = slice(k * Hd, (k + 1) * Hd)
    return np.concatenate([x @ Wq[c].T, x @ Wk[c].T, x @ Wv[c].T], axis=1)


# --------------------------------------------------------------------------
# Whole layer, plain and TSP-sharded
# --------------------------------------------------------------------------

def layer_forward(x, W: dict, heads: int, rows=None, store=None) -> dict:
    """Plain layer: h = x + Attn(x); out = h + MLP(h). float64 arrays in and out.

    W holds Wq, Wk, Wv, Wo, W1, W3, W2 (float64, [out, in]). With `rows` only those
    token rows are returned (attention still sees every earlier token).
    Returns {"attn", "h", "mlp", "out"} for the requested rows.

    With `store` (e.g. round_bf16) the layer is evaluated at a stated storage
    precision: every value handed from one product to the next goes through it
    (Q, K, V, the attention output before W_O, the MLP's input h and the gated
    activation G), while sums, the softmax and both residual adds stay float64.
    This is the bf16-in / fp32-accumulate layer with exact accumulation. Without
    `store` the layer is exact.
    """
    if store is None:
        attn = attention_block(x, W["Wq"], W["Wk"], W["Wv"], W["Wo"], heads, rows=rows)
    else:
        attn = attention_block(x, W["Wq"], W["Wk"], W["Wv"], W["Wo"], heads, rows=rows,
                               store=store)
    xr = x if rows is None else x[np.asarray(rows)]
    h = xr + attn
    if store is None:
        mlp = swiglu_mlp(h, W["W1"], W["W3"], W["W2"])
    else:
        mlp = swiglu_mlp(store(h), W["W1"], W["W3"], W["W2"], store=store)
    return {"attn": attn, "h": h, "mlp": mlp, "out": h + mlp}


def tsp_layer_forward(x, W: dict, heads: int, D: int) -> dict:
    """The same layer computed rank by rank under TSP's schedules ([TSP] s2).

    Rank r holds its zigzag token shard xs[r] ([S/D, H]). Attention: for each
    broadcast iteration k, every rank projects its own tokens with shard k's
    W_Q/W_K/W_V rows, K/V of all ranks are gathered along the sequence into
    natural order, each rank attends its queries (by global position) to the full
    K/V, and accumulates O_rk W_O,k^T locally. MLP: at ring step t rank r holds
    shard k = (r + t) mod D and adds silu(h_r W1_k^T) * (h_r W3_k^T) W2_k^T to its
    local accumulator; there is no all-reduce. Results are unsharded at the end
    and returned like layer_forward's (natural order).
    """
    S, H = x.shape
    F = W["W1"].shape[0]
    if heads % D or F % D or S % (2 * D):
        raise ValueError("TSP needs heads % D == 0, ffn % D == 0 and S % 2D == 0")
    hpr, Hd, Fd, T = heads // D, H // D, F // D, S // D
    xs = shard_tokens(x, D)
    pos = rank_positions(S, D)
    every = np.arange(S)

    acc = np.zeros((D, T, H))
    for k in range(D):                      # broadcast iteration: shard k goes to all
        c = slice(k * Hd, (k + 1) * Hd)
        Wq_k, Wk_k, Wv_k, Wo_k = W["Wq"][c], W["Wk"][c], W["Wv"][c], W["Wo"][:, c]
        q = [xs[r] @ Wq_k.T for r in range(D)]          # local projections
        k_all = unshard_tokens(np.stack([xs[r] @ Wk_k.T for r in range(D)]), D)
        v_all = unshard_tokens(np.stack([xs[r] @ Wv_k.T for r in range(D)]), D)
        for r in range(D):
            o = multihead_causal_attention(q[r], k_all, v_all, hpr, pos[r], every)
            acc[r] += o @ Wo_k.T                         # local accumulation over k
    hs = xs + acc

    acc2 = np.zeros((D, T, H))
    for t in range(D):                      # ring step
        for r in range(D):
            k = (r + t) % D
            f = slice(k * Fd, (k + 1) * Fd)
            g = silu(hs[r] @ W["W1"][f].T) * (hs[r] @ W["W3"][f].T)
            acc2[r] += g @ W["W2"][:, f].T
    outs = hs + acc2
    return {"attn": unshard_tokens(acc, D), "h": unshard_tokens(hs, D),
            "mlp": unshard_tokens(acc2, D), "out": unshard_tokens(outs, D)}


# --------------------------------------------------------------------------
# Micro-batches  ([TSP] s4, scalability: the smaller per-device footprint lets a
# device take larger micro-batches). A micro-batch is B independent sequences of
# S tokens each. Every rank owns its two zigzag chunks of EACH sequence, so rank
# r's local activations are [B, S/D, H] (sequence-major) and the rank-major
# layout of the micro-batch is [D, B, S/D, H]. Tokens of different sequences
# never attend to each other; the MLP is per token.
# --------------------------------------------------------------------------

def zigzag_forward_index_batched(S: int, D: int, B: int) -> np.ndarray:
    """fwd[b*S + t] = row of token t of sequence b in the rank-major [D, B, S/D] layout.

    Token t of sequence b sits on rank r at local row l (the single-sequence zigzag
    map), i.e. at row (r*B + b)*(S/D) + l.
    """
    rank, local = zigzag_owner(S, D)
    T = S // D
    seq = np.arange(B, dtype=np.int64)[:, None]
    return ((rank[None, :] * B + seq) * T + local[None, :]).reshape(-1)


def shard_tokens_batched(x: np.ndarray, D: int) -> np.ndarray:
    """[B, S, ...] natural order -> [D, B, S/D, ...]: rank r's rows of every sequence."""
    B, S = x.shape[:2]
    rest = x.shape[2:]
    out = np.empty((B * S,) + rest, dtype=x.dtype)
    out[zigzag_forward_index_batched(S, D, B)] = x.reshape((B * S,) + rest)
    return out.reshape((D, B, S // D) + rest)


def unshard_tokens_batched(xs: np.ndarray, D: int) -> np.ndarray:
    """Inverse of shard_tokens_batched: [D, B, S/D, ...] -> [B, S, ...]."""
    B, T = xs.shape[1], xs.shape[2]
    rest = xs.shape[3:]
    flat = xs.reshape((D * B * T,) + rest)
    return flat[zigzag_forward_index_batched(D * T, D, B)].reshape((B, D * T) + rest)


def layer_forward_batched(x, W: dict, heads: int, rows=None, store=None) -> dict:
    """The plain layer on each sequence of a micro-batch x [B, S, H] on its own.

    Returns layer_forward's dict with a leading batch axis ([B, S or len(rows), H]).
    `store` as in layer_forward.
    """
    res = [layer_forward(x[b], W, heads, rows=rows, store=store) for b in range(x.shape[0])]
    return {key: np.stack([r[key] for r in res]) for key in res[0]}


def tsp_layer_forward_batched(x, W: dict, heads: int, D: int) -> dict:
    """tsp_layer_forward for a micro-batch x [B, S, H], rank by rank.

    Rank r holds xs[r] = [B, S/D, H], its zigzag chunks of every sequence. In
    broadcast iteration k every rank projects all of its rows with shard k; the
    K/V rows of every rank are gathered per sequence into natural order, and rank
    r's queries of sequence b attend (by global position) to sequence b's keys only;
    each rank accumulates O_rk W_O,k^T locally. The MLP ring passes shard
    (r + t) mod D to rank r at step t for all of its B*S/D rows at once, with local
    accumulation and no all-reduce. Returns [B, S, H] arrays in natural order.
    """
    B, S, H = x.shape
    F = W["W1"].shape[0]
    if heads % D or F % D or S % (2 * D):
        raise ValueError("TSP needs heads % D == 0, ffn % D == 0 and S % 2D == 0")
    hpr, Hd, Fd = heads // D, H // D, F // D
    xs = shard_tokens_batched(x, D)                     # [D, B, T, H]
    pos = rank_positions(S, D)
    every = np.arange(S)

    acc = np.zeros(xs.shape)
    for k in range(D):                      # broadcast iteration: shard k goes to all
        c = slice(k * Hd, (k + 1) * Hd)
        Wo_k = W["Wo"][:, c]
        q = xs @ W["Wq"][c].T                            # local projections, [D, B, T, Hd]
        k_all = unshard_tokens_batched(xs @ W["Wk"][c].T, D)   # [B, S, Hd] per sequence
        v_all = unshard_tokens_batched(xs @ W["Wv"][c].T, D)
        for r in range(D):
            for b in range(B):
                o = multihead_causal_attention(q[r, b], k_all[b], v_all[b], hpr, pos[r], every)
                acc[r, b] += o @ Wo_k.T                  # local accumulation over k
    hs = xs + acc

    acc2 = np.zeros(xs.shape)
    for t in range(D):                      # ring step
        for r in range(D):
            k = (r + t) % D
            f = slice(k * Fd, (k + 1) * Fd)
            g = silu(hs[r] @ W["W1"][f].T) * (hs[r] @ W["W3"][f].T)
            acc2[r] += g @ W["W2"][:, f].T
    outs = hs + acc2
    return {"attn": unshard_tokens_batched(acc, D), "h": unshard_tokens_batched(hs, D),
            "mlp": unshard_tokens_batched(acc2, D), "out": unshard_tokens_batched(outs, D)}


# --------------------------------------------------------------------------
# Backward pass  ([TSP] title: training; the page describes the forward
# schedules only, so the backward is the chain rule of the same layer, and its
# sharded restatement runs the forward schedules in reverse)
# --------------------------------------------------------------------------

def silu_grad(z):
    """d silu / dz = s (1 + z (1 - s)), s = sigmoid(z)."""
    s = 1.0 / (1.0 + np.exp(-z))
    return s * (1.0 + z * (1.0 - s))


def causal_attention_head_backward(q, k, v, q_pos, k_pos, do, o_round=None, store=None):
    """Gradients (dq, dk, dv) of one head of causal_attention_head for output grad do.

    With P the softmax weights and O = P v: dv = P^T do, dP = do v^T,
    dS = P * (dP - Delta), dq = dS k / sqrt(d), dk = dS^T q / sqrt(d), where
    Delta_i = rowsum(dP_i * P_i), which equals rowsum(do_i * O_i).
    With `o_round` (a function of an array), Delta is rowsum(do * o_round(O)): the
    gradient obtained from a rounded copy of the output, such as the bf16 output a
    kernel stores and reads back.
    With `store` (e.g. round_bf16), the two values the products take from the
    element-wise step pass through it: P before dv = P^T do, and dS before dq and dk;
    and the output whose rounded copy forms Delta is the stored forward's
    (causal_attention_head with the same `store`: P rounded before P v).
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    do = np.asarray(do, dtype=np.float64)
    d = q.shape[1]
    s = (q @ k.T) / math.sqrt(d)
    visible = np.asarray(k_pos)[None, :] <= np.asarray(q_pos)[:, None]
    s = np.where(visible, s, -np.inf)
    e = np.exp(s - s.max(axis=1, keepdims=True))
    l = e.sum(axis=1, keepdims=True)
    p = e / l
    dv = (p if store is None else store(p)).T @ do
    dp = do @ v.T
    if o_round is None:
        delta = (dp * p).sum(axis=1, keepdims=True)
    else:
        o = ((e if store is None else store(e)) @ v) / l
        delta = (do * o_round(o)).sum(axis=1, keepdims=True)
    ds = p * (dp - delta)
    if store is not None:
        ds = store(ds)
    dq = ds @ k / math.sqrt(d)
    dk = ds.T @ q / math.sqrt(d)
    return dq, dk, dv


def causal_attention_head_backward_rows(q, k, v, q_pos, k_pos, do, q_rows, k_rows,
                                        q_block: int = 1024, o_round=None, store=None):
    """dq of the query rows q_rows and (dk, dv) of the key rows k_rows of one head.

    The same quantities as causal_attention_head_backward, for sequences whose full
    score matrix does not fit: dq_i depends on query i's own softmax only; dk_j and
    dv_j sum over every query that sees key j, so all queries are visited, `q_block`
    rows at a time, each with its softmax over all of its visible keys. `o_round` and
    `store` as in causal_attention_head_backward.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    do = np.asarray(do, dtype=np.float64)
    q_pos, k_pos = np.asarray(q_pos), np.asarray(k_pos)
    q_rows, k_rows = np.asarray(q_rows), np.asarray(k_rows)
    d = q.shape[1]
    dq = causal_attention_head_backward(q[q_rows], k, v, q_pos[q_rows], k_pos, do[q_rows],
                                        o_round, store)[0]
    dk = np.zeros((k_rows.size, d))
    dv = np.zeros((k_rows.size, d))
    for lo in range(0, q.shape[0], q_block):
        r = slice(lo, min(q.shape[0], lo + q_block))
        s = (q[r] @ k.T) / math.sqrt(d)
        visible = k_pos[None, :] <= q_pos[r, None]
        s = np.where(visible, s, -np.inf)
        e = np.exp(s - s.max(axis=1, keepdims=True))
        l = e.sum(axis=1, keepdims=True)
        p = e / l
        dp = do[r] @ v.T
        if o_round is None:
            delta = (dp * p).sum(axis=1, keepdims=True)
        else:
            o = ((e if store is None else store(e)) @ v) / l
            delta = (do[r] * o_round(o)).sum(axis=1, keepdims=True)
        ds = p * (dp - delta)
        if store is not None:
            ds, p = store(ds), store(p)
        dk += ds[:, k_rows].T @ q[r] / math.sqrt(d)
        dv += p[:, k_rows].T @ do[r]
    return dq, dk, dv


def swiglu_mlp_backward(h, W1, W3, W2, dmlp, rows=None, ffn_cols=None, store=None) -> dict:
    """Gradients of MLP(h) = G W2^T, G = silu(A1) * A3, A1 = h W1^T, A3 = h W3^T,
    for the output gradient dmlp (the block alone, no residual):

        dW2 = dmlp^T G       dG = dmlp W2
        dA1 = dG * A3 * silu'(A1)          dA3 = dG * silu(A1)
        dW1 = dA1^T h        dW3 = dA3^T h        dh = dA1 W1 + dA3 W3

    Returns {"dh", "dW1", "dW3", "dW2"}. With `rows`, dh holds those token rows only
    (each needs every ffn column of its own row); with `ffn_cols`, dW1 and dW3 hold
    those rows and dW2 those columns only (each needs every token).
    With `store` (e.g. round_bf16), the values handed from one product to the next
    pass through it: the kept pre-activations A1 and A3 (dA1 and dA3 are formed from
    the stored ones), G before dW2, and dA1, dA3 before the products that take them.
    """
    h = np.asarray(h, dtype=np.float64)
    dmlp = np.asarray(dmlp, dtype=np.float64)
    st = (lambda a: a) if store is None else store
    r = slice(None) if rows is None else np.asarray(rows)
    c = slice(None) if ffn_cols is None else np.asarray(ffn_cols)
    A1, A3 = h[r] @ W1.T, h[r] @ W3.T
    A1s, A3s = st(A1), st(A3)
    dG = dmlp[r] @ W2
    out = {"dh": st(dG * A3s * silu_grad(A1s)) @ W1 + st(dG * silu(A1s)) @ W3}
    A1, A3 = h @ W1[c].T, h @ W3[c].T
    A1s, A3s = st(A1), st(A3)
    dG = dmlp @ W2[:, c]
    out["dW2"] = dmlp.T @ st(silu(A1) * A3)
    out["dW1"] = st(dG * A3s * silu_grad(A1s)).T @ h
    out["dW3"] = st(dG * silu(A1s)).T @ h
    return out


def attention_block_backward(x, Wq, Wk, Wv, Wo, heads: int, dattn, store=None) -> dict:
    """Gradients of attention_block (no residual) for the output gradient dattn.

    With Q = x Wq^T, K = x Wk^T, V = x Wv^T, O the per-head causal attention and
    Attn = O Wo^T: dWo = dattn^T O, dO = dattn Wo, the per-head attention backward
    gives dQ, dK, dV, then dWq = dQ^T x (likewise K, V) and
    dx = dQ Wq + dK Wk + dV Wv. Returns {"dx", "dWq", "dWk", "dWv", "dWo"}.
    With `store` (e.g. round_bf16), the values handed between products pass through
    it: Q, K, V and O (as attention_block stores them: P rounded before P V), dO,
    the per-head P and dS (Delta formed from the stored O), and dQ, dK, dV.
    """
    S, H = x.shape
    d = H // heads
    st = (lambda a: a) if store is None else store
    Q, K, V = st(x @ Wq.T), st(x @ Wk.T), st(x @ Wv.T)
    O = st(multihead_causal_attention(Q, K, V, heads, store=store))
    g = {"dWo": dattn.T @ O}
    dO = st(dattn @ Wo)
    dQ, dK, dV = np.zeros_like(Q), np.zeros_like(K), np.zeros_like(V)
    pos = np.arange(S)
    for j in range(heads):
        c = slice(j * d, (j + 1) * d)
        dQ[:, c], dK[:, c], dV[:, c] = causal_attention_head_backward(
            Q[:, c], K[:, c], V[:, c], pos, pos, dO[:, c], o_round=store, store=store)
    dQ, dK, dV = st(dQ), st(dK), st(dV)
    g["dWq"], g["dWk"], g["dWv"] = dQ.T @ x, dK.T @ x, dV.T @ x
    g["dx"] = dQ @ Wq + dK @ Wk + dV @ Wv
    return g


def layer_backward(x, W: dict, heads: int, dout, store=None) -> dict:
    """Gradients of out = h + MLP(h), h = x + Attn(x), for the output gradient dout.

    The residual paths add the identity: dh = dout + (MLP backward of dout) and
    dx = dh + (attention backward of dh). Returns {"dx", "dWq", "dWk", "dWv",
    "dWo", "dW1", "dW3", "dW2"} (float64, the shapes of x and of the weights).
    With `store` (e.g. round_bf16), the forward values are those of
    layer_forward(..., store=store), the MLP backward takes the stored h, the
    attention backward the stored dh, and each block stores as its own backward
    says; both residual sums stay float64.
    """
    Wq, Wk, Wv, Wo = W["Wq"], W["Wk"], W["Wv"], W["Wo"]
    if store is None:
        h = x + attention_block(x, Wq, Wk, Wv, Wo, heads)
        m = swiglu_mlp_backward(h, W["W1"], W["W3"], W["W2"], dout)
        dh = dout + m["dh"]
        a = attention_block_backward(x, Wq, Wk, Wv, Wo, heads, dh)
    else:
        h = x + attention_block(x, Wq, Wk, Wv, Wo, heads, store=store)
        m = swiglu_mlp_backward(store(h), W["W1"], W["W3"], W["W2"], dout, store=store)
        dh = dout + m["dh"]
        a = attention_block_backward(x, Wq, Wk, Wv, Wo, heads, store(dh), store=store)
    g = {"dW1": m["dW1"], "dW3": m["dW3"], "dW2": m["dW2"]}
    for n in ("dWq", "dWk", "dWv", "dWo"):
        g[n] = a[n]
    g["dx"] = dh + a["dx"]
    return g


def layer_backward_batched(x, W: dict, heads: int, dout, store=None) -> dict:
    """Gradients of the sum over a micro-batch x [B, S, H] for dout [B, S, H].

    The sequences are independent: each sequence's input gradient is its own
    layer_backward's, and a weight gradient is the sum of the sequences' weight
    gradients. Returns layer_backward's keys, "dx" with a leading batch axis.
    `store` as in layer_backward.
    """
    res = [layer_backward(x[b], W, heads, dout[b], store=store) for b in range(x.shape[0])]
    g = {k: sum(r[k] for r in res) for k in res[0] if k != "dx"}
    g["dx"] = np.stack([r["dx"] for r in res])
    return g


def tsp_layer_backward(x, W: dict, heads: int, D: int, dout) -> dict:
    """layer_backward computed rank by rank, the forward schedules run in reverse.

    MLP, ring: at step t rank r holds shard k = (r + t) mod D with its partial
    weight gradients; it adds its own tokens' contributions (dW2_k += dout_r^T G_rk,
    dW1_k += dA1_rk^T h_r, dW3_k += dA3_rk^T h_r) and accumulates dh_r locally.
    Attention, broadcast iteration k: every rank computes dO_rk = dh_r Wo_k and
    dWo_k += dh_r^T O_rk; the attention backward of its queries yields dQ_rk and
    contributions to dK_k, dV_k at every key position, which are summed at the
    key's owner (the reverse of the K/V all-gather); then dx_r and the W_Q/W_K/W_V
    shard gradients. Returns the same dict as layer_backward (natural order).
    """
    S, H = x.shape
    F = W["W1"].shape[0]
    hpr, Hd, Fd, T = heads // D, H // D, F // D, S // D
    d = H // heads
    xs = shard_tokens(x, D)
    dos = shard_tokens(dout, D)
    pos = rank_positions(S, D)
    every = np.arange(S)
    # forward activations of every rank (recomputed)
    Qs, Ks, Vs, Os = {}, {}, {}, {}
    hs = xs.copy()
    for k in range(D):
        c = slice(k * Hd, (k + 1) * Hd)
        for r in range(D):
            Qs[r, k] = xs[r] @ W["Wq"][c].T
        K_all = unshard_tokens(np.stack([xs[r] @ W["Wk"][c].T for r in range(D)]), D)
        V_all = unshard_tokens(np.stack([xs[r] @ W["Wv"][c].T for r in range(D)]), D)
        Ks[k], Vs[k] = K_all, V_all
        for r in range(D):
            Os[r, k] = multihead_causal_attention(Qs[r, k], K_all, V_all, hpr, pos[r], every)
            hs[r] = hs[r] + Os[r, k] @ W["Wo"][:, c].T
    g = {n: np.zeros_like(W[n[1:]]) for n in ("dWq", "dWk", "dWv", "dWo", "dW1", "dW3", "dW2")}
    # MLP backward, ring schedule
    dhs = dos.copy()
    for t in range(D):
        for r in range(D):
            k = (r + t) % D
            f = slice(k * Fd, (k + 1) * Fd)
            A1, A3 = hs[r] @ W["W1"][f].T, hs[r] @ W["W3"][f].T
            G = silu(A1) * A3
            dG = dos[r] @ W["W2"][:, f]
            dA1 = dG * A3 * silu_grad(A1)
            dA3 = dG * silu(A1)
            g["dW2"][:, f] += dos[r].T @ G
            g["dW1"][f] += dA1.T @ hs[r]
            g["dW3"][f] += dA3.T @ hs[r]
            dhs[r] = dhs[r] + dA1 @ W["W1"][f] + dA3 @ W["W3"][f]
    # attention backward, broadcast schedule
    dxs = dhs.copy()
    for k in range(D):
        c = slice(k * Hd, (k + 1) * Hd)
        dK_nat, dV_nat = np.zeros((S, Hd)), np.zeros((S, Hd))
        dQ = {}
        for r in range(D):
            dO = dhs[r] @ W["Wo"][:, c]
            g["dWo"][:, c] += dhs[r].T @ Os[r, k]
            dQ[r] = np.zeros((T, Hd))
            for j in range(hpr):
                cc = slice(j * d, (j + 1) * d)
                dq, dk, dv = causal_attention_head_backward(
                    Qs[r, k][:, cc], Ks[k][:, cc], Vs[k][:, cc], pos[r], every, dO[:, cc])
                dQ[r][:, cc] = dq
                dK_nat[:, cc] += dk      # summed at the key's owner
                dV_nat[:, cc] += dv
        dKs, dVs = shard_tokens(dK_nat, D), shard_tokens(dV_nat, D)
        for r in range(D):
            dxs[r] = dxs[r] + dQ[r] @ W["Wq"][c] + dKs[r] @ W["Wk"][c] + dVs[r] @ W["Wv"][c]
            g["dWq"][c] += dQ[r].T @ xs[r]
            g["dWk"][c] += dKs[r].T @ xs[r]
            g["dWv"][c] += dVs[r].T @ xs[r]
    g["dx"] = unshard_tokens(dxs, D)
    return g


# --------------------------------------------------------------------------
# Counting  ([TSP] s2 "Unified sharding"; s3 memory and FLOPs analysis)
# --------------------------------------------------------------------------

def causal_pairs_per_rank(S: int, D: int) -> np.ndarray:
    """Number of visible (query, key) pairs of each rank's queries, by brute count."""
    rank, _ = zigzag_owner(S, D)
    keys_seen = np.arange(S, dtype=np.int64) + 1   # query at position p sees p+1 keys
    return np.bincount(rank, weights=keys_seen, minlength=D).astype(np.int64)


def layer_flops(S: int, H: int, F: int) -> int:
    """Algorithmic FLOPs of one layer forward (multiply-add = 2 FLOPs).

    Q/K/V/O projections 4 * 2SH^2, SwiGLU 3 * 2SHF, causal attention
    2 * (QK^T and PV) * d * (S(S+1)/2 pairs) * heads = 2HS(S+1).
    """
    return 8 * S * H * H + 6 * S * H * F + 2 * H * S * (S + 1)


def rank_parameter_count(H: int, F: int, D: int) -> int:
    """Parameters one rank holds: 1/D of W_Q, W_K, W_V, W_O, W1, W2, W3."""
    total = 4 * H * H + 3 * H * F
    if total % D:
        raise ValueError("parameters do not split evenly")
    return total // D


def rank_activation_count(S: int, H: int, D: int) -> int:
    """Layer-input activations one rank holds: its S/D tokens times H."""
    return (S // D) * H
