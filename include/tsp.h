/*
 * tsp.h - C ABI of the GB300 (sm_103a) forward of one Folding Tensor and
 * Sequence Parallelism (TSP) transformer layer, all D logical ranks on one GPU.
 *
 * Source of the method, cited below as [TSP]: the summary page "Folding Tensor and
 * Sequence Parallelism for Memory-Efficient Transformer Training & Inference"
 * (gist.science, paper 2604.26294). Section numbers refer to that page:
 * s1 Problem statement, s2 Methodology, s3 Contributions, s4 Results.
 *
 * What the library computes (a layer without normalisation or positional encoding):
 *     h   = x + Attn(x)        Attn: causal multi-head softmax attention, scale 1/sqrt(d)
 *     out = h + MLP(h)         MLP(h) = (silu(h W1^T) * (h W3^T)) W2^T
 * with the tokens of the sequence and the weights split over D ranks as [TSP] s2
 * describes: each rank owns 1/D of the tokens (zigzag chunks) and 1/D of the
 * weights; attention iterates over packed W_Q/W_K/W_V/W_O shards (broadcast
 * schedule), gathers K/V along the sequence and runs causal attention of each
 * rank's queries against the full K/V; the gated MLP streams W1/W3/W2 shards in
 * ring order and accumulates each rank's partial outputs locally, without an
 * all-reduce. On one GPU a "broadcast" or a "ring hand-off" is a read of a shard
 * in place, and the all-gather is a gather kernel into natural token order.
 *
 * Conventions shared by every entry point
 *   - Element type: bfloat16, passed as its 16-bit pattern (tsp_bf16). Arithmetic
 *     on tensor cores accumulates in fp32; intermediates stored in HBM (Q, K, V, P,
 *     O, h, G) are rounded to bf16 with round-to-nearest-even.
 *   - Pointers are DEVICE pointers unless the name ends in _host. The caller owns
 *     every buffer; the library allocates no device memory in any call below.
 *   - `stream` is a cudaStream_t passed as void* (NULL = the legacy default
 *     stream). All device work is enqueued asynchronously on it; calls return
 *     once the work is enqueued.
 *   - Activations in the "sharded" layout are rank-major [D, T, H] with
 *     T = S/D: rank r's rows are its zigzag tokens in local order (chunk r, then
 *     chunk 2D-1-r, chunk length C = S/(2D)). A plan for a micro-batch of B
 *     sequences (tsp_plan_batched) uses [D, B, T, H] instead.
 *   - Status is returned synchronously. Argument and shape problems return
 *     TSP_ERR_INVALID_ARG / TSP_ERR_UNSUPPORTED before anything is launched; a
 *     launch failure returns TSP_ERR_CUDA. Device-side waits are bounded: a wait
 *     that gives up records TSP_ERR_TIMEOUT in the workspace status word, which
 *     tsp_device_status() reports. tsp_last_error() returns a message for the
 *     last failing call of the calling thread. No C++ exception crosses the ABI.
 */
#ifndef TSP_H_
#define TSP_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef uint16_t tsp_bf16; /* bfloat16 bit pattern */

typedef enum tsp_status {
  TSP_OK = 0,
  TSP_ERR_INVALID_ARG = 1, /* null pointer, bad index, misaligned buffer        */
  TSP_ERR_UNSUPPORTED = 2, /* shape outside the supported set (see tsp_plan)    */
  TSP_ERR_CUDA = 3,        /* a CUDA runtime/driver call or a launch failed     */
  TSP_ERR_TIMEOUT = 4      /* a bounded device wait gave up (tsp_device_status) */
} tsp_status;

typedef struct tsp_plan_s* tsp_plan_t; /* opaque, library-owned, immutable */

/* Derived sizes of a plan (all element counts unless named _bytes). */
typedef struct tsp_plan_info {
  int D;            /* logical ranks = shards                                  */
  int64_t S;        /* tokens                                                  */
  int hidden;       /* H                                                       */
  int heads;        /* attention heads h                                       */
  int head_dim;     /* d = H / h                                               */
  int ffn;          /* F                                                       */
  int64_t T;        /* tokens per rank, S / D                                  */
  int64_t C;        /* zigzag chunk, S / (2D)                                  */
  int shard_hidden; /* H / D: width of one attention weight shard (h/D heads)  */
  int shard_ffn;    /* F / D: width of one MLP weight shard                    */
  int shard_ffn_padded; /* Fp >= F/D: stored width of one MLP shard (zero rows) */
  int ffn_padded;   /* NF = D * Fp: width of the gated activation G            */
  /* packed weight buffer (elements from its start) */
  size_t wpack_qkv;   /* [D][3H/D][H]: shard k = rows of W_Q, W_K, W_V of heads group k */
  size_t wpack_o;     /* [H][H]: W_O; shard k = columns [k H/D, (k+1) H/D)             */
  size_t wpack_w13;   /* [NF/128][256][H]: per 128 padded ffn columns, 128 W1 rows then 128 W3 rows */
  size_t wpack_w2;    /* [H][NF]: W2, shard k = columns [k Fp, (k+1) Fp), zero padded  */
  size_t wpack_elems; /* total elements of the packed buffer                          */
  size_t workspace_bytes;     /* tsp_workspace_bytes(plan)     */
  size_t bwd_workspace_bytes; /* tsp_bwd_workspace_bytes(plan) */
  int64_t stat_stride;        /* row stride of per-head row statistics (lse, delta): tokens rounded up to 128 */
  int batch;                  /* B: sequences of the micro-batch (1 for tsp_plan)  */
  int64_t tokens;             /* N = B * S: rows of every activation buffer        */
  int attention_group;        /* shards whose attention runs in one launch in the
                                 *_fwd calls: the fewest (a divisor of D) that give
                                 512 two-tile CTAs, so a short sequence still fills
                                 the GPU; their Q/K/V share the workspace           */
} tsp_plan_info;

/*
 * tsp_plan - validate a layer shape and derive sizes. Makes no CUDA call.
 *   D      logical ranks (shards) >= 1          [TSP] s2, "Unified sharding"
 *   S      tokens (batch 1)                     [TSP] s2
 *   hidden H, heads h: head_dim d = H/h must be 64 or 128
 *   ffn    F, the SwiGLU inner width
 * Supported iff S % (2D) == 0 (zigzag chunks), heads % D == 0 (whole heads per
 * attention shard), ffn % D == 0, H % 64 == 0, 1 <= D <= 64 and
 * 2D <= S <= 2^26; otherwise TSP_ERR_UNSUPPORTED. *out receives a plan that
 * the caller releases with tsp_plan_destroy.
 */
tsp_status tsp_plan(int D, int64_t S, int hidden, int heads, int ffn, tsp_plan_t* out);

/*
 * tsp_plan_batched - a plan for a micro-batch of `batch` independent sequences of S
 * tokens each ([TSP] s4: the smaller per-device footprint of TSP admits larger
 * micro-batches). Every rank owns its two zigzag chunks of EACH sequence, so the
 * sharded layout of every activation becomes rank-major [D][B][T][H]: rank r's rows
 * of sequence b are rows (r*B + b)*T .. (r*B + b)*T + T-1, in the single-sequence
 * local order. Natural (unsharded) buffers are [B][S][H]. Queries attend only to
 * the keys of their own sequence; the projections and the MLP run over all
 * N = B*S rows at once (one weight-shard pass serves the whole micro-batch).
 * Every entry point takes such a plan; in the buffer sizes stated below, read
 * N = B*S rows where a size says S or D*T (the lse / delta statistics hold
 * stat_stride >= N entries per head). The backward calls return the gradients of
 * the sum over the micro-batch: input gradients per sequence, weight gradients
 * summed over every sequence's tokens. Supported iff tsp_plan's conditions hold,
 * batch >= 1, batch * S <= 2^26 and, for batch > 1, T = S/D is a multiple of 128
 * (a 128-row query tile of the attention kernels never spans two ranks' blocks).
 * tsp_plan(D, S, ...) is tsp_plan_batched(D, S, 1, ...).
 */
tsp_status tsp_plan_batched(int D, int64_t S, int batch, int hidden, int heads, int ffn,
                            tsp_plan_t* out);
void tsp_plan_destroy(tsp_plan_t plan);
tsp_status tsp_get_plan_info(tsp_plan_t plan, tsp_plan_info* info);
/* Bytes of the caller-allocated workspace every *_fwd call below needs (256-byte
 * aligned). Its first 256 bytes hold the device status word. */
size_t tsp_workspace_bytes(tsp_plan_t plan);
/* Bytes of the packed weight buffer (tsp_plan_info.wpack_elems bf16 elements). */
size_t tsp_packed_weight_bytes(tsp_plan_t plan);

/*
 * tsp_workspace_init - zero the workspace status word (enqueued on stream).
 * Call once after allocating a workspace.
 */
tsp_status tsp_workspace_init(tsp_plan_t plan, void* ws, void* stream);

/*
 * tsp_pack_weights - build the packed, shard-major weight buffer ([TSP] s2:
 * packed W_Q/W_K/W_V/W_O shards for attention; W1/W2/W3 shards for the ring).
 * Inputs use the nn.Linear layout [out, in]: Wq/Wk/Wv/Wo [H][H], W1/W3 [F][H],
 * W2 [H][F]. wpack must hold tsp_packed_weight_bytes(plan) bytes. Padded ffn
 * columns are written as zero. Run once per weight set.
 */
tsp_status tsp_pack_weights(tsp_plan_t plan, const tsp_bf16* Wq, const tsp_bf16* Wk,
                            const tsp_bf16* Wv, const tsp_bf16* Wo, const tsp_bf16* W1,
                            const tsp_bf16* W3, const tsp_bf16* W2, tsp_bf16* wpack,
                            void* stream);

/*
 * tsp_shard_index - the zigzag map ([TSP] s2, zigzag partitioning that balances
 * causal attention work). fwd[t] = r*T + l for global token t owned by rank r at
 * local row l; inv[r*T + l] = t. Both int32 [S]. Either pointer may be NULL.
 * With a micro-batch (tsp_plan_batched): fwd[b*S + t] = (r*B + b)*T + l and inv its
 * inverse, both int32 [B*S].
 */
tsp_status tsp_shard_index(tsp_plan_t plan, int32_t* fwd, int32_t* inv, void* stream);

/* tsp_shard: x [S][H] natural order -> xs [D][T][H] zigzag rank-major
 * (micro-batch: x [B][S][H] -> xs [D][B][T][H]).
 * tsp_unshard: the inverse. Buffers must not overlap. */
tsp_status tsp_shard(tsp_plan_t plan, const tsp_bf16* x, tsp_bf16* xs, void* stream);
tsp_status tsp_unshard(tsp_plan_t plan, const tsp_bf16* xs, tsp_bf16* x, void* stream);

/*
 * tsp_attention_fwd - attention block of every rank, no residual ([TSP] s2,
 * attention layers: broadcast schedule over packed shards, local Q/K/V
 * projections, K/V all-gather, FlashAttention over zigzag query chunks).
 *   xs   [D][T][H] sharded layer input
 *   attn [D][T][H] sharded output Attn(x)
 * attn may not alias xs or ws.
 */
tsp_status tsp_attention_fwd(tsp_plan_t plan, const tsp_bf16* xs, const tsp_bf16* wpack,
                             tsp_bf16* attn, void* ws, void* stream);

/*
 * tsp_mlp_fwd - gated MLP of every rank, no residual ([TSP] s2, gated MLP layers:
 * W1/W3/W2 shards circulate in a ring; each rank accumulates its partial outputs
 * locally, with no all-reduce). hs and mlp are [D][T][H] sharded.
 */
tsp_status tsp_mlp_fwd(tsp_plan_t plan, const tsp_bf16* hs, const tsp_bf16* wpack,
                       tsp_bf16* mlp, void* ws, void* stream);

/*
 * tsp_layer_fwd - the whole layer on sharded activations:
 *   out = h + MLP(h), h = xs + Attn(xs); xs and out [D][T][H]. out may not alias xs.
 */
tsp_status tsp_layer_fwd(tsp_plan_t plan, const tsp_bf16* xs, const tsp_bf16* wpack,
                         tsp_bf16* out, void* ws, void* stream);

/*
 * tsp_layer_fwd_host - the whole layer from and to HOST memory in natural token
 * order: x_host [S][H] in, out_host [S][H] out. A page-locked input (pinned or
 * registered, i.e. mapped into the device address space) comes in rank by rank:
 * the copy engine moves each rank's rows (two runs of C natural rows per sequence)
 * to their sharded rows on a library-owned non-blocking stream of the device
 * (created on first use, kept until exit), while `stream` runs the Q/K/V products on
 * the ranks already in: of every shard when the padded ffn is at least 2 H (their
 * Q/K/V then live in workspace buffers that are idle until the O projection), else
 * of the first attention group. A page-locked output comes back
 * rank by rank: the down projection runs
 * per rank on `stream`, and each rank's rows are copied to out_host by the copy
 * engine on that stream while the next ranks compute; `stream` then waits for the
 * last copy. Both need S/D % 128 == 0; otherwise the zigzag shard / unshard kernels
 * read and write the mapped buffers directly, the copy and the permutation in one
 * pass.
 * The result is the same bit for bit either way. Pageable buffers are staged
 * through cudaMemcpyAsync and the workspace. The call returns once the work is
 * enqueued: synchronise `stream` before reading out_host.
 * The library-owned copy stream is one per device, shared by every caller and
 * thread: concurrent tsp_layer_fwd_host calls on different caller streams
 * serialise their host-link copies on it, and a call made while another thread
 * captures a CUDA graph that touches that stream disturbs the capture. Capture
 * tsp_layer_fwd (device buffers) rather than this call.
 */
tsp_status tsp_layer_fwd_host(tsp_plan_t plan, const tsp_bf16* x_host, const tsp_bf16* wpack,
                              tsp_bf16* out_host, void* ws, void* stream);

/*
 * tsp_mlp_fwd_noalloc - tsp_mlp_fwd for callers that cannot allocate device
 * memory. The page has no counterpart: this entry point exists for library users.
 * Some callers cannot call cudaMalloc (or any allocating routine, torch's included)
 * where they run the layer: code inside a custom allocator or memory-pool callback,
 * plug-ins of an application that owns every device allocation, runtimes that
 * forbid allocation after start-up. They still pass hs, wpack and mlp ([D][T][H]
 * as for tsp_mlp_fwd) but no workspace: the gated activation G and the status word
 * of the bounded device waits live in one static device array of 32 MiB inside the
 * library, which a device holds from the first call there until the process exits.
 * Limit: tokens (B x S) x ffn_padded x 2 bytes <= 32 MiB - 256 (e.g. S = 4096 with hidden 1024
 * and ffn 2816); larger shapes return TSP_ERR_UNSUPPORTED with a message.
 * The call allocates nothing (no cudaMalloc/cudaFree, no allocating library call)
 * once the array is in place on the device. Set-up: the first call on a device (in
 * each CUDA context) looks the array's device address up with cudaGetSymbolAddress,
 * with that device current. CUDA loads a library's device code lazily by default,
 * so that first lookup is also when the driver reserves the 32 MiB on the device:
 * make the first call at start-up, where reserving device memory is still allowed,
 * and before any stream capture. Later calls in the same context reserve nothing
 * (the free device memory does not change). Every call shares the array and the
 * array keeps the last call's contents (the call clears the status word itself;
 * G is overwritten in full): calls that overlap on the GPU (other streams, other
 * threads) race on it and must be serialised by the caller. A device wait that
 * gives up leaves mlp undefined; this variant has no status query (use tsp_mlp_fwd
 * with a workspace and tsp_device_status when that report is needed).
 */
tsp_status tsp_mlp_fwd_noalloc(tsp_plan_t plan, const tsp_bf16* hs, const tsp_bf16* wpack,
                               tsp_bf16* mlp, void* stream);

/* ---------------------------------------------------------------------------
 * Single steps of the hot path. The *_fwd calls above are compositions of these.
 * In these calls `ws` only provides the status word of the bounded device waits:
 * 256 bytes (256-byte aligned, zeroed once) are enough.
 * ------------------------------------------------------------------------- */

/*
 * tsp_qkv_projection - step "local projections" of broadcast iteration k
 * ([TSP] s2, attention layers): every rank multiplies its own tokens by shard k
 * of W_Q/W_K/W_V. qkv [D*T][3H/D]: columns [0,H/D) Q, [H/D,2H/D) K,
 * [2H/D,3H/D) V of heads group k (head-major, d columns per head), rows in the
 * sharded (zigzag) order.
 */
tsp_status tsp_qkv_projection(tsp_plan_t plan, int shard, const tsp_bf16* xs,
                              const tsp_bf16* wpack, tsp_bf16* qkv, void* ws, void* stream);

/*
 * tsp_kv_allgather - step "All-Gather of K/V along the sequence" ([TSP] s2):
 * gathers the K and V columns of every rank's qkv rows into natural token order:
 * kn[t] = K row of token t, vn[t] = V row of token t; kn, vn [S][H/D].
 */
tsp_status tsp_kv_allgather(tsp_plan_t plan, const tsp_bf16* qkv, tsp_bf16* kn, tsp_bf16* vn,
                            void* stream);

/*
 * tsp_qkv_projection_gathered - the local projections of broadcast iteration k with
 * the K/V all-gather fused into the GEMM epilogue (the two steps above in one
 * pass, bit-identical to them): Q rows stay in the sharded order in q [D*T][H/D]
 * (head-major, d columns per head); the K and V rows of every rank are written at
 * their natural token positions in kn, vn [S][H/D]. tsp_attention_fwd and
 * tsp_layer_fwd use this step.
 */
tsp_status tsp_qkv_projection_gathered(tsp_plan_t plan, int shard, const tsp_bf16* xs,
                                       const tsp_bf16* wpack, tsp_bf16* q, tsp_bf16* kn,
                                       tsp_bf16* vn, void* ws, void* stream);

/*
 * tsp_causal_attention - step "FlashAttention" for heads group k ([TSP] s2): every
 * query row of qkv (zigzag row, global position from the zigzag map) attends to
 * kn/vn rows 0..position. Writes o[row][k*H/D + j*d + c] for the h/D heads j of
 * the group; o is [D*T][H] (sharded rows). Scale 1/sqrt(d).
 */
tsp_status tsp_causal_attention(tsp_plan_t plan, int shard, const tsp_bf16* qkv,
                                const tsp_bf16* kn, const tsp_bf16* vn, tsp_bf16* o,
                                void* ws, void* stream);

/* tsp_causal_attention_q - the same step with Q from the q [D*T][H/D] buffer of
 * tsp_qkv_projection_gathered instead of the Q columns of a Q|K|V buffer. */
tsp_status tsp_causal_attention_q(tsp_plan_t plan, int shard, const tsp_bf16* q,
                                  const tsp_bf16* kn, const tsp_bf16* vn, tsp_bf16* o,
                                  void* ws, void* stream);

/*
 * tsp_o_projection - O projection with local accumulation over the attention
 * shards: out = o * W_O^T (+ residual if not NULL). The K-loop of the product walks
 * the shards k = 0..D-1 in broadcast order and accumulates in fp32 on chip.
 * o, residual, out [D*T][H] bf16. If out32 is not NULL (it needs a residual), the
 * fp32 value of out is also written there ([D*T][H] float), which is how
 * tsp_layer_fwd keeps h = x + Attn(x) in fp32 for the MLP's residual.
 */
tsp_status tsp_o_projection(tsp_plan_t plan, const tsp_bf16* o, const tsp_bf16* wpack,
                            const tsp_bf16* residual, tsp_bf16* out, float* out32, void* ws,
                            void* stream);

/*
 * tsp_swiglu_gate_up - G = silu(hs W1^T) * (hs W3^T) for every MLP shard:
 * g [D*T][NF], shard k in columns [k Fp, (k+1) Fp) (padded columns are 0).
 */
tsp_status tsp_swiglu_gate_up(tsp_plan_t plan, const tsp_bf16* hs, const tsp_bf16* wpack,
                              tsp_bf16* g, void* ws, void* stream);

/*
 * tsp_swiglu_down - out = G W2^T (+ residual) with the ring order of [TSP] s2: for
 * rows of rank r the K-loop takes shard (r + t) mod D at step t = 0..D-1 and
 * accumulates the partial outputs locally in fp32 (no all-reduce). The residual is
 * residual32 ([D*T][H] float) if not NULL, else residual ([D*T][H] bf16) if not
 * NULL, else none.
 */
tsp_status tsp_swiglu_down(tsp_plan_t plan, const tsp_bf16* g, const tsp_bf16* wpack,
                           const tsp_bf16* residual, const float* residual32, tsp_bf16* out,
                           void* ws, void* stream);

/* ---------------------------------------------------------------------------
 * Rank-local steps: the layer forward as one of D devices computes it ([TSP] s2,
 * Methodology: "Attention layers" and "Gated MLP layers"), for running the D
 * ranks on D devices (or several ranks on one). Rank r holds its T = S/D tokens
 * xs_r [T][H] (zigzag chunks r and 2D-1-r, in that order) and weight shard r. The
 * exchanges between the calls are the caller's (a collective library across
 * devices; buffer copies between ranks on one device):
 *   attention, broadcast iteration k = 0..D-1:
 *     the owner of shard k broadcasts its attention part;
 *     tsp_rank_qkv            (every rank, its own tokens)
 *     all-gather of every rank's kv_r [T][2H/D] into kv_all [D][T][2H/D] (rank order)
 *     tsp_rank_kv_gather      (K, V in natural token order)
 *     tsp_rank_attention      (the rank's queries against the full K/V)
 *     tsp_rank_o_accumulate   (acc_r += o_r W_O,k^T; residual x_r at k = 0)
 *   MLP, ring step t = 0..D-1: rank r holds MLP part of shard (r + t) mod D;
 *     tsp_rank_mlp_step       (acc_r += SwiGLU_k(h_r) W2_k^T; residual h32_r at t = 0)
 *     then every rank sends its MLP part to rank r - 1 and receives from r + 1.
 * No all-reduce anywhere: each rank accumulates its own rows. The result equals
 * tsp_layer_fwd's rows of rank r up to fp32 summation order (each shard's partial
 * product is added to an fp32 accumulator in HBM instead of one K loop in tensor
 * memory). A micro-batch plan (tsp_plan_batched, B sequences) is supported when
 * S/D % 128 == 0 (TSP_ERR_UNSUPPORTED otherwise): rank r then holds its T tokens of
 * every sequence, [B][T] rows wherever [T] is written below, kv_all is
 * [D][B][T][2H/D] and kn, vn are [B][S][H/D].
 * `ws` provides the status word only (256 bytes, as for the single steps). All
 * buffers are the caller's, 16-byte aligned; calls are asynchronous on `stream`.
 * ------------------------------------------------------------------------- */

/*
 * tsp_rank_shard_bytes - bytes of the two parts of one rank's weight shard k:
 *   attention part (broadcast): Wqkv_k [3H/D][H] (Q, K, V rows of heads group k:
 *     heads k*h/D .. (k+1)*h/D - 1), then W_O,k [H][H/D] (those heads' columns of W_O);
 *   MLP part (ring): W13_k [Fq/128][256][H] (per 128 padded ffn columns of slice
 *     k*F/D .., 128 W1 rows then the matching 128 W3 rows), then W2_k [H][Fp]
 *     (the slice's columns of W2). Fp = shard_ffn_padded, Fq = Fp rounded up to
 *     128; padded rows and columns are zero (silu(0) * 0 = 0 keeps it exact).
 */
tsp_status tsp_rank_shard_bytes(tsp_plan_t plan, size_t* attn_bytes, size_t* mlp_bytes);

/*
 * tsp_pack_rank_shard - lay out shard k from the natural weights (nn.Linear
 * layout [out][in], as tsp_pack_weights) into attn_shard and mlp_shard. Only shard
 * k's rows and columns are read.
 */
tsp_status tsp_pack_rank_shard(tsp_plan_t plan, int k, const tsp_bf16* Wq, const tsp_bf16* Wk,
                               const tsp_bf16* Wv, const tsp_bf16* Wo, const tsp_bf16* W1,
                               const tsp_bf16* W3, const tsp_bf16* W2, tsp_bf16* attn_shard,
                               tsp_bf16* mlp_shard, void* stream);

/*
 * tsp_rank_qkv - local projections of one rank with attention shard k ([TSP] s2):
 * q_r [T][H/D] = xs_r Wq_k^T; kv_r [T][2H/D] = (xs_r Wk_k^T | xs_r Wv_k^T) per row,
 * the rank's contribution to the K/V all-gather. bf16 out, fp32 accumulation.
 */
tsp_status tsp_rank_qkv(tsp_plan_t plan, const tsp_bf16* xs_r, const tsp_bf16* attn_shard,
                        tsp_bf16* q_r, tsp_bf16* kv_r, void* ws, void* stream);

/*
 * tsp_rank_kv_gather - K/V "all-gathered along the sequence" ([TSP] s2): kv_all
 * [D][T][2H/D] (every rank's kv_r in rank order) -> kn, vn [S][H/D] in natural
 * token order (the zigzag inverse). Bit-exact copy.
 */
tsp_status tsp_rank_kv_gather(tsp_plan_t plan, const tsp_bf16* kv_all, tsp_bf16* kn,
                              tsp_bf16* vn, void* stream);

/*
 * tsp_rank_attention - causal attention of rank r's queries (global positions of
 * its zigzag chunks) against the full K/V: o_r [T][H/D] for the h/D heads of the
 * current shard (head j at columns j*d). Scale 1/sqrt(d), key t visible iff
 * t <= position. q_r as tsp_rank_qkv wrote it.
 */
tsp_status tsp_rank_attention(tsp_plan_t plan, int r, const tsp_bf16* q_r, const tsp_bf16* kn,
                              const tsp_bf16* vn, tsp_bf16* o_r, void* ws, void* stream);

/*
 * tsp_rank_o_accumulate - local accumulation of the O projection ([TSP] s2, read
 * like the MLP's): acc_r [T][H] fp32 = residual + o_r W_O,k^T, and h_r = bf16(acc_r).
 * residual: x_r (bf16, residual_f32 = 0) at the first broadcast iteration, then
 * acc_r itself (fp32, residual_f32 = 1; in place). After the last iteration acc_r
 * is h = x + Attn(x) in fp32 and h_r its bf16 value (the MLP input).
 */
tsp_status tsp_rank_o_accumulate(tsp_plan_t plan, const tsp_bf16* o_r, const tsp_bf16* attn_shard,
                                 const void* residual, int residual_f32, float* acc_r,
                                 tsp_bf16* h_r, void* ws, void* stream);

/*
 * tsp_rank_mlp_step - one ring step of the gated MLP ([TSP] s2, local accumulation,
 * no all-reduce): g_r [T][Fq] bf16 = silu(h_r W1_k^T) * (h_r W3_k^T) (scratch), then
 * acc_r [T][H] fp32 = residual32 + g_r W2_k^T and out_r = bf16(acc_r). residual32:
 * the fp32 h of tsp_rank_o_accumulate at step 0, then acc_r itself (in place).
 * After the last step out_r is the layer output of rank r's rows.
 */
tsp_status tsp_rank_mlp_step(tsp_plan_t plan, const tsp_bf16* h_r, const tsp_bf16* mlp_shard,
                             const float* residual32, float* acc_r, tsp_bf16* out_r,
                             tsp_bf16* g_r, void* ws, void* stream);

/* ---------------------------------------------------------------------------
 * Backward pass. [TSP] (title, s1) is about training but the page describes the
 * forward schedules only; the backward is the chain rule of the same layer under
 * those schedules run in reverse: the MLP's ring (rank r at step t holds shard
 * (r + t) mod D and accumulates its dh locally) and the attention's broadcast
 * iterations (per shard: dO, the attention backward, whose K/V gradients are
 * summed at the key's owner - the reverse of the all-gather - then dx).
 *   - Weight gradients are fp32 in the PACKED layout of tsp_pack_weights:
 *     dwpack holds tsp_plan_info.wpack_elems floats, each section at the same
 *     element offset as in wpack, padded ffn entries written as zero.
 *     tsp_unpack_weight_grads converts them to the nn.Linear layout.
 *   - The backward calls recompute the forward activations they need from their
 *     inputs (no state is kept between calls) and need a workspace of
 *     tsp_bwd_workspace_bytes(plan) bytes (it extends the forward's workspace).
 *   - Data gradients (bf16) are [D][T][H] sharded like the activations.
 * ------------------------------------------------------------------------- */

/* Bytes of the workspace the *_bwd calls need (256-byte aligned). */
size_t tsp_bwd_workspace_bytes(tsp_plan_t plan);

/*
 * tsp_mlp_bwd - backward of tsp_mlp_fwd (no residual) for the output gradient
 * dmlp [D][T][H]: dhs [D][T][H] = dMLP/dh^T dmlp, and the W1, W3, W2 gradients
 * written into their sections of dwpack (the attention sections are untouched):
 *   A1|A3 = hs W13^T and G = silu(A1) A3 are recomputed (one GEMM, both saved),
 *   dW2 = dmlp^T G, dG = dmlp W2 -> dA1 = dG A3 silu'(A1), dA3 = dG silu(A1) (GEMM
 *   epilogue), dhs = dA1 W1 + dA3 W3 (K loop in ring order), dW1|dW3 = dA13^T hs.
 * dhs may not alias hs or dmlp.
 */
tsp_status tsp_mlp_bwd(tsp_plan_t plan, const tsp_bf16* hs, const tsp_bf16* wpack,
                       const tsp_bf16* dmlp, tsp_bf16* dhs, float* dwpack, void* ws,
                       void* stream);

/*
 * tsp_attention_bwd - backward of tsp_attention_fwd (no residual) for the output
 * gradient dattn [D][T][H]: dxs [D][T][H] and the W_Q, W_K, W_V, W_O gradients in
 * their sections of dwpack (the MLP sections are untouched). Per broadcast
 * iteration k the forward is recomputed (Q/K/V of shard k with the K/V gather, the
 * attention with each row's log-sum-exp); then dO = dattn W_O, dW_O = dattn^T O,
 * Delta = rowsum(dO * O), the attention backward of shard k's heads (dK/dV summed
 * over every rank's queries, written at the key owner's rows), and finally
 * dxs = dQKV W_QKV (K loop over the shards in broadcast order) and
 * dW_QKV = dQKV^T xs. dxs may not alias xs or dattn.
 */
tsp_status tsp_attention_bwd(tsp_plan_t plan, const tsp_bf16* xs, const tsp_bf16* wpack,
                             const tsp_bf16* dattn, tsp_bf16* dxs, float* dwpack, void* ws,
                             void* stream);

/*
 * tsp_layer_bwd - backward of tsp_layer_fwd for the output gradient dout [D][T][H]:
 *   dh  = dout + MLP backward of dout at h (h = xs + Attn(xs), recomputed),
 *   dxs = dh + attention backward of dh,
 * and every weight gradient in dwpack. dh is kept in fp32 for the residual and
 * rounded to bf16 once, as the operand of the attention backward's products.
 * dxs may not alias xs or dout.
 */
tsp_status tsp_layer_bwd(tsp_plan_t plan, const tsp_bf16* xs, const tsp_bf16* wpack,
                         const tsp_bf16* dout, tsp_bf16* dxs, float* dwpack, void* ws,
                         void* stream);

/*
 * Training pair: a forward that keeps the attention's output and row statistics,
 * and a backward that uses them instead of running the attention forward again
 * (the backward still recomputes the cheap projections: Q/K/V of every shard and h).
 *
 * tsp_saved_bytes - bytes of the caller buffer `saved` of the pair: o, the attention
 *   output before W_O, [D][T][H] bf16 (sharded rows, shard k's heads in columns
 *   [k H/D, (k+1) H/D)), then, at the next 256-byte boundary, lse [heads][stat_stride]
 *   fp32, the base-2 log-sum-exp of every head and row (tsp_causal_attention_lse).
 * tsp_layer_fwd_train - tsp_layer_fwd (bit-identical out) that also fills `saved`.
 * tsp_layer_bwd_saved - tsp_layer_bwd (bit-identical dxs and dwpack) for the same xs,
 *   wpack and the `saved` of tsp_layer_fwd_train; needs a tsp_bwd_workspace_bytes
 *   workspace. dxs may not alias xs or dout.
 */
size_t tsp_saved_bytes(tsp_plan_t plan);
tsp_status tsp_layer_fwd_train(tsp_plan_t plan, const tsp_bf16* xs, const tsp_bf16* wpack,
                               tsp_bf16* out, void* saved, void* ws, void* stream);
tsp_status tsp_layer_bwd_saved(tsp_plan_t plan, const tsp_bf16* xs, const tsp_bf16* wpack,
                               const void* saved, const tsp_bf16* dout, tsp_bf16* dxs,
                               float* dwpack, void* ws, void* stream);

/*
 * tsp_causal_attention_lse - tsp_causal_attention_q that also writes, for each of
 * shard k's heads j and query row r, lse[j * stat_stride + r] = log2 of the softmax
 * denominator of the row in the base-2 domain of the scaled scores, i.e. the
 * softmax weight of key t is exp2(q.k_t * log2(e)/sqrt(d) - lse). lse is
 * [H/(D d)][stat_stride] float (tsp_plan_info.stat_stride).
 */
tsp_status tsp_causal_attention_lse(tsp_plan_t plan, int shard, const tsp_bf16* q,
                                    const tsp_bf16* kn, const tsp_bf16* vn, tsp_bf16* o,
                                    float* lse, void* ws, void* stream);

/*
 * tsp_causal_attention_bwd - backward of the attention step of shard k. Inputs: q
 * [D*T][H/D] (sharded rows), kn, vn [S][H/D] (natural rows), o and dout [D*T][H]
 * (shard k's columns [k H/D, (k+1) H/D) are read), lse from
 * tsp_causal_attention_lse. Writes delta [H/(D d)][stat_stride] = rowsum(dout * o)
 * per head and row, and dQ | dK | dV of the shard's heads into columns
 * [3k H/D, 3(k+1) H/D) of dqkv [D*T][3H] (sharded rows; the dK/dV row of key t is
 * the zigzag row of t and sums the contributions of every rank's queries).
 */
tsp_status tsp_causal_attention_bwd(tsp_plan_t plan, int shard, const tsp_bf16* q,
                                    const tsp_bf16* kn, const tsp_bf16* vn, const tsp_bf16* o,
                                    const tsp_bf16* dout, const float* lse, float* delta,
                                    tsp_bf16* dqkv, void* ws, void* stream);

/*
 * tsp_unpack_weight_grads - packed fp32 weight gradients -> nn.Linear layout fp32:
 * dWq/dWk/dWv/dWo [H][H], dW1/dW3 [F][H], dW2 [H][F]. Any output may be NULL
 * (not written).
 */
tsp_status tsp_unpack_weight_grads(tsp_plan_t plan, const float* dwpack, float* dWq, float* dWk,
                                   float* dWv, float* dWo, float* dW1, float* dW3, float* dW2,
                                   void* stream);

/* ---------------------------------------------------------------------------
 * Cost model ([TSP] s3, theoretical analysis: memory, communication and FLOPs of
 * TSP against DP, TP, SP and TP+SP). The page states the comparison in words
 * only; these closed forms are written from each scheme's sharding rules for the
 * layer this library computes (batch 1, S tokens), per device and per layer:
 *   TSP_SCHEME_DP     the whole layer on one device (replicas take other sequences)
 *   TSP_SCHEME_TP     weights split over D devices by heads / ffn columns, the
 *                     layer input and residual (x, h) replicated, two ring
 *                     all-reduces of S x H (attention and MLP outputs)
 *   TSP_SCHEME_SP     tokens split over D devices, weights replicated, K/V
 *                     all-gathered over the sequence
 *   TSP_SCHEME_TP_SP  a tp x (D/tp) grid: weights split over tp, tokens over D/tp;
 *                     all-reduces in each tp group, K/V all-gathers across groups
 *   TSP_SCHEME_TSP    weights and tokens split over the same D devices; attention
 *                     shards broadcast, MLP shards passed around a ring, K/V
 *                     all-gathered per head group, no all-reduce
 * Activation elements per token: x and h (2H) plus q, k, v, o, a1, a3, g (4H + 3F).
 * Communication: elements one device receives in one forward, with ring
 * collectives (all-reduce of n over g devices: 2 (g-1)/g n; all-gather: (g-1)/g n).
 * FLOPs: 8SH^2 + 6SHF + 2HS(S+1) per layer (causal attention), divided evenly.
 * Makes no CUDA call. Shapes must divide evenly (heads, ffn by the weight split, S
 * by the token split), else TSP_ERR_UNSUPPORTED; tp is read for TP_SP only.
 * ------------------------------------------------------------------------- */
typedef enum tsp_scheme {
  TSP_SCHEME_DP = 0,
  TSP_SCHEME_TP = 1,
  TSP_SCHEME_SP = 2,
  TSP_SCHEME_TP_SP = 3,
  TSP_SCHEME_TSP = 4
} tsp_scheme;

typedef struct tsp_cost {
  int devices;                  /* devices one copy of the layer spans                    */
  double weight_elems;          /* resident weight elements per device                    */
  double weight_inflight_elems; /* received weight elements held at once (TSP: one shard) */
  double act_elems;             /* activation elements per device                         */
  double act_inflight_elems;    /* gathered K/V held during attention                     */
  double comm_weight_elems;     /* weight elements received per device per forward        */
  double comm_act_elems;        /* activation elements received per device per forward    */
  double flops;                 /* forward FLOPs per device                               */
} tsp_cost;

tsp_status tsp_cost_model(int scheme, int D, int tp, int64_t S, int hidden, int heads, int ffn,
                          tsp_cost* out);

/*
 * tsp_cost_model_batched - the same model for a micro-batch of `batch` sequences of
 * S tokens ([TSP] s4, scalability: TSP's smaller per-device footprint lets a device
 * take larger micro-batches). Every sequence is split like the single one, so
 * act_elems, act_inflight_elems, comm_act_elems and flops are `batch` times those
 * of tsp_cost_model; the weight terms (and TSP's weight traffic, which one pass of
 * the shards serves for the whole micro-batch) do not change. batch >= 1, else
 * TSP_ERR_INVALID_ARG. tsp_cost_model is batch 1.
 */
tsp_status tsp_cost_model_batched(int scheme, int D, int tp, int64_t S, int batch, int hidden,
                                  int heads, int ffn, tsp_cost* out);

/*
 * tsp_cost_max_batch - the largest micro-batch B whose bf16 footprint on one device
 * fits in mem_bytes under `scheme` for a model of `layers` such layers:
 *   bytes(B) = 2 * (layers * (weight_elems + B * act_elems)
 *                   + weight_inflight_elems + B * act_inflight_elems)
 * (every layer keeps its weights and activations, as training does; one layer's
 * received shard and gathered K/V exist at a time), with the batch-1 terms of
 * tsp_cost_model. *out = 0 if one sequence does not fit. layers >= 1 and a finite
 * mem_bytes >= 0, else TSP_ERR_INVALID_ARG; shape errors as tsp_cost_model.
 */
tsp_status tsp_cost_max_batch(int scheme, int D, int tp, int64_t S, int hidden, int heads,
                              int ffn, int layers, double mem_bytes, int64_t* out);

/*
 * tsp_device_status - synchronise `stream`, then read and clear the workspace
 * status word. Returns TSP_OK, TSP_ERR_TIMEOUT (a bounded device wait gave up; the
 * outputs of the affected call are undefined), TSP_ERR_UNSUPPORTED (a kernel whose
 * shared-memory layout fills the 227 KB limit found its dynamic shared memory at a
 * base that left no room, and returned without computing) or TSP_ERR_CUDA.
 */
tsp_status tsp_device_status(void* ws, void* stream);

/*
 * tsp_wait_selftest - launch one block that waits on a barrier nothing will
 * arrive at, with a bound of `limit_ns` nanoseconds; the kernel gives up, records
 * TSP_ERR_TIMEOUT in the status word and returns. Exercises the failure path of
 * the bounded waits without faulting or hanging the GPU.
 */
tsp_status tsp_wait_selftest(void* ws, uint64_t limit_ns, void* stream);

/* Message of the last failing call on this thread ("" if none). */
const char* tsp_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* TSP_H_ */
