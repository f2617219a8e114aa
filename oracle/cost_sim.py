"""Brute-force count of per-device memory, communication and FLOPs of one layer
under DP, TP, SP, TP+SP and TSP. TEST INFRASTRUCTURE ONLY.

The page "Folding Tensor and Sequence Parallelism for Memory-Efficient
Transformer Training & Inference" (section 3, theoretical analysis) compares TSP
with DP, TP, SP and TP+SP on memory, communication and FLOPs in words only. This
module does not evaluate formulas: it builds, for every device, the explicit set
of weight elements and activation elements the device holds under each scheme's
sharding rules, and it steps every collective (ring all-reduce, ring all-gather,
broadcast, the TSP weight ring) chunk by chunk, adding up what each device
receives. Only the tests may import it; the library never does. It shares no
code with the library's closed-form model.

Sharding rules (the same readings as the rest of this repository):
  * weight shard g of G: heads [g h/G, (g+1) h/G) -> rows of W_Q, W_K, W_V and
    columns of W_O; ffn slice [g F/G, (g+1) F/G) -> rows of W1, W3, columns of W2;
  * token group r of G: the zigzag chunks r and 2G-1-r ([TSP] s2);
  * activations per token: x and h (boundary), q, k, v, o (head columns) and
    a1, a3, g (ffn columns);
  * TP keeps x and h on every device of its group; TP+SP uses a tp x (D/tp) grid,
    device d = sigma * tp + g with weight shard g and token group sigma;
  * a micro-batch of B sequences ([TSP] s4, scalability): every sequence is split
    the same way, so a device holds its tokens of each sequence; the weights (and
    the weight traffic of TSP) serve the whole micro-batch once.
"""
from __future__ import annotations

import numpy as np

from .tsp_oracle import zigzag_owner

SCHEMES = ("dp", "tp", "sp", "tp_sp", "tsp")


def _weight_shard(name, H, F, heads, g, G):
    """Boolean mask of weight shard g of G of one matrix (nn.Linear layout)."""
    d = H // heads
    hh = slice(g * (heads // G) * d, (g + 1) * (heads // G) * d)
    ff = slice(g * (F // G), (g + 1) * (F // G))
    shapes = {"Wq": (H, H), "Wk": (H, H), "Wv": (H, H), "Wo": (H, H),
              "W1": (F, H), "W3": (F, H), "W2": (H, F)}
    m = np.zeros(shapes[name], dtype=bool)
    if name in ("Wq", "Wk", "Wv"):
        m[hh, :] = True
    elif name == "Wo":
        m[:, hh] = True
    elif name in ("W1", "W3"):
        m[ff, :] = True
    else:
        m[:, ff] = True
    return m


ATT = ("Wq", "Wk", "Wv", "Wo")
MLP = ("W1", "W3", "W2")


def _shard_elems(names, H, F, heads, g, G):
    return sum(int(_weight_shard(n, H, F, heads, g, G).sum()) for n in names)


def _tokens(S, r, G):
    """Token indices of zigzag group r of G."""
    if G == 1:
        return np.arange(S)
    owner, _ = zigzag_owner(S, G)
    return np.nonzero(owner == r)[0]


def _ring_allreduce(n, g):
    """Elements each device of a g-device ring receives in an all-reduce of n
    elements: g-1 reduce-scatter steps then g-1 all-gather steps, one chunk each."""
    recv = np.zeros(g, dtype=np.int64)
    chunks = [len(c) for c in np.array_split(np.arange(n), g)]
    for step in range(g - 1):          # reduce-scatter
        for i in range(g):
            recv[(i + 1) % g] += chunks[(i - step) % g]
    for step in range(g - 1):          # all-gather
        for i in range(g):
            recv[(i + 1) % g] += chunks[(i + 1 - step) % g]
    return recv


def _ring_allgather(blocks):
    """Elements each device receives when every device's block goes around the ring."""
    g = len(blocks)
    recv = np.zeros(g, dtype=np.int64)
    for step in range(g - 1):
        for i in range(g):
            recv[(i + 1) % g] += blocks[(i - step) % g]
    return recv


def _visible_pairs(tokens):
    """Causal (query, key) pairs of the given query tokens (position p sees p + 1)."""
    return int(sum(int(t) + 1 for t in tokens))


def simulate(scheme, D, S, H, heads, F, tp=0, batch=1):
    """Per-device counts of one layer forward of a micro-batch of `batch` sequences;
    every device of a balanced layout gets the same numbers, which are returned (a
    ValueError if they differ)."""
    d_head = H // heads
    P_all = 4 * H * H + 3 * H * F
    per = []
    if scheme == "dp":
        devices = [dict(wg=(0, 1), tg=(0, 1), inner=(0, 1))]
    elif scheme == "tp":
        devices = [dict(wg=(d, D), tg=(0, 1), inner=(d, D)) for d in range(D)]
    elif scheme == "sp":
        devices = [dict(wg=(0, 1), tg=(d, D), inner=(0, 1)) for d in range(D)]
    elif scheme == "tp_sp":
        sg = D // tp
        devices = [dict(wg=(d % tp, tp), tg=(d // tp, sg), inner=(d % tp, tp)) for d in range(D)]
    elif scheme == "tsp":
        devices = [dict(wg=(d, D), tg=(d, D), inner=(0, 1)) for d in range(D)]
    else:
        raise ValueError(scheme)

    n_dev = len(devices)
    for d, dv in enumerate(devices):
        g, G = dv["wg"]
        r, R = dv["tg"]
        ig, IG = dv["inner"]
        toks = _tokens(S, r, R)          # this device's positions in each sequence
        ntok = batch * len(toks)         # ... over every sequence of the micro-batch
        # resident weights: the device's own shard
        weights = _shard_elems(ATT + MLP, H, F, heads, g, G)
        # activations: boundary tensors x, h on all columns of the device's tokens;
        # inner tensors on the device's token rows and its head / ffn columns
        head_cols = int(_weight_shard("Wo", H, F, heads, ig, IG)[0].sum())
        ffn_cols = int(_weight_shard("W2", H, F, heads, ig, IG)[0].sum())
        acts = ntok * (2 * H) + ntok * (4 * head_cols + 3 * ffn_cols)
        c = dict(devices=n_dev, weight_elems=weights, weight_inflight_elems=0, act_elems=acts,
                 act_inflight_elems=0, comm_weight_elems=0, comm_act_elems=0, flops=0)
        # every activation collective runs once per sequence of the micro-batch
        if scheme == "tp":
            ar = sum(int(_ring_allreduce(S * H, D)[d]) for _ in range(batch))
            c["comm_act_elems"] = 2 * ar
        elif scheme == "sp":
            blocks = [len(_tokens(S, q, D)) * 2 * H for q in range(D)]
            c["comm_act_elems"] = sum(int(_ring_allgather(blocks)[d]) for _ in range(batch))
            c["act_inflight_elems"] = batch * sum(blocks)
        elif scheme == "tp_sp":
            sg = D // tp
            grp_tokens = len(toks)
            kv_cols = 2 * (H // tp)
            blocks = [len(_tokens(S, q, sg)) * kv_cols for q in range(sg)]
            for _ in range(batch):
                c["comm_act_elems"] += 2 * int(_ring_allreduce(grp_tokens * H, tp)[g])
                c["comm_act_elems"] += int(_ring_allgather(blocks)[r])
            c["act_inflight_elems"] = batch * sum(blocks)
        elif scheme == "tsp":
            # attention: broadcast iteration k sends shard k to every other device;
            # each iteration all-gathers head group k's K/V of every device's tokens
            kv_cols = 2 * (H // D)
            att_in, kv_in, kv_buf = 0, 0, 0
            for k in range(D):
                if k != d:
                    att_in += _shard_elems(ATT, H, F, heads, k, D)   # once per micro-batch
                blocks = [len(_tokens(S, q, D)) * kv_cols for q in range(D)]
                kv_in += sum(int(_ring_allgather(blocks)[d]) for _ in range(batch))
                kv_buf = max(kv_buf, batch * sum(blocks))
            # MLP ring: at step t = 1..D-1 device d receives shard (d + t) mod D
            ring_in = sum(_shard_elems(MLP, H, F, heads, (d + t) % D, D) for t in range(1, D))
            c["comm_weight_elems"] = att_in + ring_in
            c["comm_act_elems"] = kv_in
            c["act_inflight_elems"] = kv_buf
            if D > 1:
                held = [_shard_elems(ATT, H, F, heads, k, D) for k in range(D) if k != d]
                held += [_shard_elems(MLP, H, F, heads, (d + t) % D, D) for t in range(1, D)]
                c["weight_inflight_elems"] = max(held)
        # FLOPs: 2 per multiply-add of the device's token rows with the weight
        # elements it applies to them, plus 4 per head dimension per visible pair
        if scheme == "tsp":
            applied = P_all  # every shard passes by every device
            pair_width = H
        else:
            applied = weights
            pair_width = head_cols
        c["flops"] = 2 * ntok * applied + 4 * pair_width * batch * _visible_pairs(toks)
        assert pair_width % d_head == 0
        per.append(c)
    first = per[0]
    for c in per[1:]:
        if c != first:
            raise ValueError(f"{scheme}: devices differ: {first} vs {c}")
    return first


def memory_elems(c, layers=1):
    """Elements one device holds for `layers` layers of counts c: every layer's
    resident weights and activations, and one layer's in-flight buffers at a time."""
    return (layers * (c["weight_elems"] + c["act_elems"])
            + c["weight_inflight_elems"] + c["act_inflight_elems"])


def max_micro_batch(scheme, D, S, H, heads, F, mem_bytes, layers=1, tp=0, limit=4096):
    """Largest micro-batch whose bf16 footprint (memory_elems x 2 bytes) fits in
    mem_bytes, found by simulating B = 1, 2, ... (0 if even one sequence does not fit)."""
    best = 0
    for b in range(1, limit + 1):
        if 2 * memory_elems(simulate(scheme, D, S, H, heads, F, tp=tp, batch=b), layers) > mem_bytes:
            break
        best = b
    return best
