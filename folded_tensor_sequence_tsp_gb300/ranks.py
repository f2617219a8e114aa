"""The TSP layer forward across ranks: the schedule of "Folding Tensor and Sequence
Parallelism for Memory-Efficient Transformer Training & Inference", section 2
(Methodology), over the library's rank-local calls.

Each of D ranks holds its T = S/D zigzag tokens and one weight shard, split in the
part that is broadcast (attention: packed W_Q/W_K/W_V rows and W_O columns of one
heads group) and the part that travels around the ring (the W1/W3/W2 slice of the
gated MLP). One layer forward is:

  attention, broadcast iteration k = 0 .. D-1
    the owner of shard k broadcasts its attention part to every rank;
    every rank projects its own tokens (tsp_rank_qkv);
    K/V are all-gathered along the sequence (every rank's [T][2H/D] rows);
    every rank runs its queries against the full K/V (tsp_rank_kv_gather,
    tsp_rank_attention) and accumulates its O-projection partial locally
    (tsp_rank_o_accumulate);
  MLP, ring step t = 0 .. D-1
    rank r holds the MLP part of shard (r + t) mod D, adds its SwiGLU partial to
    its local accumulator (tsp_rank_mlp_step) while the parts move one rank along
    the ring (rank r sends to r - 1 and receives from r + 1); no all-reduce.

The exchanges go through an Exchange object:
  * TorchDistExchange: one rank per process over torch.distributed. With the NCCL
    backend the CUDA buffers are sent as they are; with a host backend (gloo) they
    are staged through host memory. Every received shard and K/V block lands in a
    local buffer before a kernel reads it.
  * LocalExchange: every rank in this process (for example all D ranks on one GPU),
    the exchanges being copies between the ranks' buffers.
The compute goes through a RankCompute object; CudaRankCompute calls the library.
Every rank computes exactly its own rows, so the layer output of rank r equals
tsp_layer_fwd's rows of rank r up to fp32 summation order.
"""
from __future__ import annotations

import torch

from . import _binding as B


# ----------------------------------------------------------------- exchanges

class _Done:
    def wait(self):
        return None


class _Pending:
    """Completion of asynchronous torch.distributed work, then an optional copy-back."""

    def __init__(self, works, after=None):
        self.works, self.after = works, after

    def wait(self):
        for w in self.works:
            if w is not None:
                w.wait()
        if self.after is not None:
            self.after()
            self.after = None


class LocalExchange:
    """Every rank lives in this process: the broadcast, the all-gather and the ring
    shift are copies between the ranks' buffers (on the current stream for CUDA
    tensors, so they are ordered with the kernels that read them)."""

    def __init__(self, D: int):
        self.D = D
        self.recv_bytes = {"broadcast": 0, "all_gather": 0, "ring": 0}

    def broadcast(self, bufs: dict, src: int):
        for r, t in bufs.items():
            if r != src:
                t.copy_(bufs[src])
                self.recv_bytes["broadcast"] += t.numel() * t.element_size()
        return _Done()

    def all_gather(self, outs: dict, ins: dict):
        for r, out in outs.items():
            for j in range(self.D):
                out[j].copy_(ins[j])
                if j != r:
                    self.recv_bytes["all_gather"] += ins[j].numel() * ins[j].element_size()
        return _Done()

    def ring_shift(self, send: dict, recv: dict):
        for r, t in recv.items():
            t.copy_(send[(r + 1) % self.D])
            self.recv_bytes["ring"] += t.numel() * t.element_size()
        return _Done()


class TorchDistExchange:
    """One rank per process over torch.distributed (rank = the process group rank).

    `stage_host`: move CUDA buffers through host memory around each operation (for a
    host-only backend such as gloo). Without it the buffers are handed to the backend
    as they are (NCCL with CUDA buffers)."""

    def __init__(self, group=None, stage_host: bool = False):
        import torch.distributed as dist
        self.dist = dist
        self.group = group
        self.rank = dist.get_rank(group)
        self.D = dist.get_world_size(group)
        self.stage_host = stage_host
        self.recv_bytes = {"broadcast": 0, "all_gather": 0, "ring": 0}

    def _peer(self, r):
        return r if self.group is None else self.dist.get_global_rank(self.group, r)

    def _staged(self, t):
        if self.stage_host and t.is_cuda:
            return t.detach().to("cpu"), True
        return t, False

    def broadcast(self, bufs: dict, src: int):
        (r, t), = bufs.items()
        h, staged = self._staged(t)
        w = self.dist.broadcast(h, self._peer(src), group=self.group, async_op=True)
        if r != src:
            self.recv_bytes["broadcast"] += t.numel() * t.element_size()
        return _Pending([w], (lambda: t.copy_(h)) if staged and r != src else None)

    def all_gather(self, outs: dict, ins: dict):
        (r, out), = outs.items()
        h_in, staged = self._staged(ins[r])
        h_out = torch.empty(out.shape, dtype=out.dtype) if staged else out
        w = self.dist.all_gather([h_out[j] for j in range(self.D)], h_in, group=self.group,
                                 async_op=True)
        self.recv_bytes["all_gather"] += (self.D - 1) * ins[r].numel() * ins[r].element_size()
        return _Pending([w], (lambda: out.copy_(h_out)) if staged else None)

    def ring_shift(self, send: dict, recv: dict):
        (r, s), = send.items()
        t = recv[r]
        h_s, staged = self._staged(s)
        h_r = torch.empty(t.shape, dtype=t.dtype) if staged else t
        ws = [self.dist.isend(h_s, self._peer((r - 1) % self.D), group=self.group),
              self.dist.irecv(h_r, self._peer((r + 1) % self.D), group=self.group)]
        self.recv_bytes["ring"] += t.numel() * t.element_size()
        return _Pending(ws, (lambda: t.copy_(h_r)) if staged else None)


# ------------------------------------------------------------------- compute

class CudaRankCompute:
    """The rank-local library calls on CUDA buffers of one device (bf16 activations,
    fp32 accumulators). One object serves every rank that this process drives on
    the current device."""

    act_dtype = torch.bfloat16

    def __init__(self, plan):
        self.plan = plan
        i = plan.info
        # rows of one rank (its T tokens of every sequence of the micro-batch) and of
        # the natural-order K/V (every token of every sequence)
        self.D, self.S, self.T, self.H, self.Hd = i.D, i.tokens, i.batch * i.T, i.hidden, i.shard_hidden
        self.Fq = (i.shard_ffn_padded + 127) // 128 * 128
        self.device = torch.device("cuda", torch.cuda.current_device())
        self.ws = torch.zeros(256, dtype=torch.uint8, device=self.device)

    def shard_numel(self):
        a, m = B.tsp_rank_shard_bytes(self.plan)
        return a // 2, m // 2

    def begin(self, r, xs_r):
        e = lambda *shape, dt=torch.bfloat16: torch.empty(shape, dtype=dt, device=self.device)
        T, H, Hd, S = self.T, self.H, self.Hd, self.S
        return {"r": r, "x": xs_r, "q": e(T, Hd), "kn": e(S, Hd), "vn": e(S, Hd), "o": e(T, Hd),
                "acc": e(T, H, dt=torch.float32), "h": e(T, H), "g": e(T, self.Fq),
                "out": e(T, H)}

    def attention_project(self, st, k, attn_shard, kv_r):
        B.tsp_rank_qkv(self.plan, st["x"], attn_shard, st["q"], kv_r, self.ws)

    def attention_finish(self, st, k, attn_shard, kv_all):
        B.tsp_rank_kv_gather(self.plan, kv_all, st["kn"], st["vn"])
        B.tsp_rank_attention(self.plan, st["r"], st["q"], st["kn"], st["vn"], st["o"], self.ws)
        res = st["x"] if k == 0 else st["acc"]
        B.tsp_rank_o_accumulate(self.plan, st["o"], attn_shard, res, st["acc"], st["h"], self.ws)

    def mlp_step(self, st, t, mlp_shard):
        B.tsp_rank_mlp_step(self.plan, st["h"], mlp_shard, st["acc"], st["acc"], st["out"],
                            st["g"], self.ws)

    def output(self, st):
        return st["out"]

    def check(self):
        status = B.tsp_device_status(self.ws)
        if status != B.TSP_OK:
            raise B.TSPError(status, B.tsp_last_error())


# ------------------------------------------------------------------ schedule

def layer_forward_ranks(D: int, T: int, hd: int, ranks, xs: dict, attn_shards: dict,
                        mlp_shards: dict, exchange, compute) -> dict:
    """One layer forward of the ranks `ranks` (the ranks this process drives: all D
    for a LocalExchange, its own rank for a TorchDistExchange).

    xs[r]: rank r's zigzag tokens [T][H] (T: its rows, B S/D for a micro-batch of B
    sequences, [B][S/D][H]); attn_shards[r], mlp_shards[r]: the two parts of weight
    shard r (tsp_rank_shard_bytes layout for CudaRankCompute); hd = H/D.
    Returns {r: rank r's layer output [T][H]}. The MLP part circulates in a second
    buffer so that the caller's shards are left as they were. Transfers overlap the
    compute: the broadcast of attention shard k + 1 is in flight during iteration k,
    and the ring shift for MLP step t + 1 during step t.
    """
    ranks = list(ranks)
    like = next(iter(xs.values()))
    state = {r: compute.begin(r, xs[r]) for r in ranks}
    kv = {r: torch.empty((T, 2 * hd), dtype=compute.act_dtype, device=like.device) for r in ranks}
    kv_all = {r: torch.empty((D, T, 2 * hd), dtype=compute.act_dtype, device=like.device)
              for r in ranks}
    # two receive buffers: the broadcast of shard k + 1 is in flight while iteration k
    # computes (a rank's own shard is sent from where it lies)
    recv = [{r: torch.empty_like(attn_shards[r]) for r in ranks} for _ in range(2)]

    def start_broadcast(k):
        bufs = {r: attn_shards[r] if r == k else recv[k % 2][r] for r in ranks}
        return bufs, exchange.broadcast(bufs, src=k)

    nxt_b = start_broadcast(0)
    for k in range(D):  # broadcast iteration k: shard k's attention part to every rank
        cur, pending = nxt_b
        pending.wait()
        if k + 1 < D:
            nxt_b = start_broadcast(k + 1)
        for r in ranks:
            compute.attention_project(state[r], k, cur[r], kv[r])
        exchange.all_gather(kv_all, kv).wait()
        for r in ranks:
            compute.attention_finish(state[r], k, cur[r], kv_all[r])
    cur = {r: mlp_shards[r].clone() for r in ranks}
    nxt = {r: torch.empty_like(mlp_shards[r]) for r in ranks}
    for t in range(D):  # ring step t: rank r holds shard (r + t) mod D
        shift = exchange.ring_shift(cur, nxt) if t + 1 < D else None  # overlaps the step
        for r in ranks:
            compute.mlp_step(state[r], t, cur[r])
        if shift is not None:
            shift.wait()
            cur, nxt = nxt, cur
    return {r: compute.output(state[r]) for r in ranks}


def pack_rank_shards(plan, W: dict, ranks):
    """{r: (attention part, MLP part)} of weight shard r, laid out on the current CUDA
    device from the natural bf16 weights W (Wq, Wk, Wv, Wo, W1, W3, W2)."""
    a, m = B.tsp_rank_shard_bytes(plan)
    out = {}
    for r in ranks:
        att = torch.empty(a // 2, dtype=torch.bfloat16, device="cuda")
        mlp = torch.empty(m // 2, dtype=torch.bfloat16, device="cuda")
        B.tsp_pack_rank_shard(plan, r, W["Wq"], W["Wk"], W["Wv"], W["Wo"], W["W1"], W["W3"],
                              W["W2"], att, mlp)
        out[r] = (att, mlp)
    return out
