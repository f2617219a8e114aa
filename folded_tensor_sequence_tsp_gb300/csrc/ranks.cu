// ranks.cu - the TSP layer forward as one rank computes it: the rank-local steps.
//
// "Folding Tensor and Sequence Parallelism for Memory-Efficient Transformer
// Training & Inference", section 2 (Methodology): each of D devices holds 1/D of
// the tokens (zigzag chunks r and 2D-1-r) and 1/D of the weights. Attention
// layers: at broadcast iteration k, the device that owns packed attention shard k
// (its W_Q/W_K/W_V rows and W_O columns) broadcasts it; every device projects its
// own tokens, K/V are all-gathered along the sequence, FlashAttention runs the
// device's queries against the full K/V, and the device accumulates its partial
// O-projection output locally. Gated MLP layers: the W1/W3/W2 shards travel around
// a ring; at step t device r holds shard (r + t) mod D and adds its SwiGLU partial
// output to a local accumulator, with no all-reduce.
//
// These calls are the compute of one device between those exchanges. The exchanges
// themselves (broadcast, all-gather, ring send/receive) are the caller's: a
// collective library across devices, or plain buffer hand-offs when several ranks
// share a device. Each call works on one rank's T rows and one weight shard held
// in its own buffer (the shard as it is sent), so no call reads another rank's
// memory. The kernels are the single-GPU path's: the tcgen05 GEMM (with a
// row-major K order over one shard and an fp32 accumulator read and written in
// place) and the attention kernel restricted to the rank's query rows.
#include "tsp_device.cuh"
#include "tsp_internal.h"

namespace tsp {
namespace {

// Elements of the two parts of one rank's weight shard (see tsp_rank_shard_bytes):
//   attention: Wqkv_k [3 Hd][H] (Q rows of heads group k, then K, then V), W_O,k [H][Hd]
//   MLP:       W13_k [Fq/128][256][H] (per 128 padded ffn columns: 128 W1 rows, then
//              the matching 128 W3 rows), W2_k [H][Fp]
// Fp is the shard's padded ffn width (a multiple of 64) and Fq = Fp rounded up to 128,
// so that every 256-row tile of W13_k holds matching gate and up rows.
struct ShardLayout {
  int64_t Fq;
  int64_t attn_elems, o_off;
  int64_t mlp_elems, w2_off;
};

ShardLayout shard_layout(const Plan& p) {
  ShardLayout l;
  l.Fq = (p.Fp + 127) / 128 * 128;
  l.o_off = 3LL * p.Hd * p.H;
  l.attn_elems = l.o_off + (int64_t)p.H * p.Hd;
  l.w2_off = 2LL * l.Fq * p.H;
  l.mlp_elems = l.w2_off + (int64_t)p.H * p.Fp;
  return l;
}

struct RankPackArgs {
  const uint16_t *Wq, *Wk, *Wv, *Wo, *W1, *W3, *W2;
  uint16_t *attn, *mlp;
  int64_t H, F, Hd, Fd, Fp, Fq, k;
  int64_t attn_elems, o_off, mlp_elems, w2_off;
};

// One element of shard k per thread (a one-time layout, not on the hot path).
__global__ void rank_pack_kernel(RankPackArgs a) {
  const int64_t total = a.attn_elems + a.mlp_elems;
  for (int64_t e = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; e < total;
       e += (int64_t)gridDim.x * blockDim.x) {
    if (e < a.attn_elems) {
      uint16_t v;
      if (e < a.o_off) {  // Wqkv_k
        const int64_t row = e / a.H, col = e - row * a.H;
        const int64_t sec = row / a.Hd, j = row - sec * a.Hd;
        const uint16_t* W = sec == 0 ? a.Wq : (sec == 1 ? a.Wk : a.Wv);
        v = W[(a.k * a.Hd + j) * a.H + col];
      } else {  // W_O columns of heads group k
        const int64_t x = e - a.o_off, row = x / a.Hd, c = x - row * a.Hd;
        v = a.Wo[row * a.H + a.k * a.Hd + c];
      }
      a.attn[e] = v;
    } else {
      const int64_t x = e - a.attn_elems;
      uint16_t v = 0;
      if (x < a.w2_off) {  // W13_k, interleaved per 128 padded columns
        const int64_t g = x / (256 * a.H), rem = x - g * 256 * a.H;
        const int64_t rr = rem / a.H, col = rem - rr * a.H;
        const int64_t f = g * 128 + (rr & 127);
        if (f < a.Fd) v = (rr < 128 ? a.W1 : a.W3)[(a.k * a.Fd + f) * a.H + col];
      } else {  // W2_k: columns k Fd .. of W2, zero padded to Fp
        const int64_t y = x - a.w2_off, row = y / a.Fp, f = y - row * a.Fp;
        if (f < a.Fd) v = a.W2[row * a.F + a.k * a.Fd + f];
      }
      a.mlp[x] = v;
    }
  }
}

tsp_status rank_check(tsp_plan_t plan, const char* what) {
  TSP_TRY(tsp_check_plan(plan));
  // a rank's rows of every sequence of a micro-batch ([B][T]) go through the 128-row
  // tiles together, as in the all-rank path
  if (plan->p.B > 1 && plan->p.T % 128)
    return fail(TSP_ERR_UNSUPPORTED, std::string(what) + ": a micro-batch needs S/D % 128 == 0");
  return TSP_OK;
}

}  // namespace
}  // namespace tsp

using namespace tsp;

extern "C" {

tsp_status tsp_rank_shard_bytes(tsp_plan_t plan, size_t* attn_bytes, size_t* mlp_bytes) {
  TSP_TRY(rank_check(plan, "tsp_rank_shard_bytes"));
  if (!attn_bytes || !mlp_bytes) return fail(TSP_ERR_INVALID_ARG, "tsp_rank_shard_bytes: null output");
  const ShardLayout l = shard_layout(plan->p);
  *attn_bytes = (size_t)l.attn_elems * 2;
  *mlp_bytes = (size_t)l.mlp_elems * 2;
  return TSP_OK;
}

tsp_status tsp_pack_rank_shard(tsp_plan_t plan, int k, const tsp_bf16* Wq, const tsp_bf16* Wk,
                               const tsp_bf16* Wv, const tsp_bf16* Wo, const tsp_bf16* W1,
                               const tsp_bf16* W3, const tsp_bf16* W2, tsp_bf16* attn_shard,
                               tsp_bf16* mlp_shard, void* stream) {
  TSP_TRY(rank_check(plan, "tsp_pack_rank_shard"));
  TSP_TRY(check_ptrs({Wq, Wk, Wv, Wo, W1, W3, W2, attn_shard, mlp_shard}, "tsp_pack_rank_shard"));
  const Plan& p = plan->p;
  if (k < 0 || k >= p.D) return fail(TSP_ERR_INVALID_ARG, "tsp_pack_rank_shard: shard out of range");
  const ShardLayout l = shard_layout(p);
  RankPackArgs a;
  a.Wq = reinterpret_cast<const uint16_t*>(Wq);
  a.Wk = reinterpret_cast<const uint16_t*>(Wk);
  a.Wv = reinterpret_cast<const uint16_t*>(Wv);
  a.Wo = reinterpret_cast<const uint16_t*>(Wo);
  a.W1 = reinterpret_cast<const uint16_t*>(W1);
  a.W3 = reinterpret_cast<const uint16_t*>(W3);
  a.W2 = reinterpret_cast<const uint16_t*>(W2);
  a.attn = reinterpret_cast<uint16_t*>(attn_shard);
  a.mlp = reinterpret_cast<uint16_t*>(mlp_shard);
  a.H = p.H;
  a.F = p.F;
  a.Hd = p.Hd;
  a.Fd = p.Fd;
  a.Fp = p.Fp;
  a.Fq = l.Fq;
  a.k = k;
  a.attn_elems = l.attn_elems;
  a.o_off = l.o_off;
  a.mlp_elems = l.mlp_elems;
  a.w2_off = l.w2_off;
  const int64_t total = l.attn_elems + l.mlp_elems;
  int64_t blocks = (total + 255) / 256;
  const int64_t cap = 8LL * sm_count();
  if (blocks > cap) blocks = cap;
  rank_pack_kernel<<<(unsigned)blocks, 256, 0, static_cast<cudaStream_t>(stream)>>>(a);
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? TSP_OK : cuda_fail(e, "tsp_pack_rank_shard: launch");
}

tsp_status tsp_rank_qkv(tsp_plan_t plan, const tsp_bf16* xs_r, const tsp_bf16* attn_shard,
                        tsp_bf16* q_r, tsp_bf16* kv_r, void* ws, void* stream) {
  TSP_TRY(rank_check(plan, "tsp_rank_qkv"));
  TSP_TRY(check_ptrs({xs_r, attn_shard, q_r, kv_r}, "tsp_rank_qkv"));
  TSP_TRY(check_ws(ws, "tsp_rank_qkv"));
  const Plan& p = plan->p;
  GemmCall c{};
  c.epi = EPI_QKV_SPLIT;
  c.A = xs_r;
  c.lda = p.H;
  c.M = (int64_t)p.B * p.T;  // the rank's rows of every sequence
  c.B = attn_shard;
  c.ldb = p.H;
  c.b_rows = 3LL * p.Hd;
  c.b_row0 = 0;
  c.N = 3LL * p.Hd;
  c.K = p.H;
  c.C = q_r;
  c.ldc = p.Hd;
  // K and V rows side by side in kv_r [T][2 Hd], in the rank's own row order: the
  // epilogue's zigzag row placement with one rank (chunks of T/2) is the identity
  c.split_k = kv_r;
  c.split_v = reinterpret_cast<uint16_t*>(kv_r) + p.Hd;
  c.split_ld = 2LL * p.Hd;
  c.split_hd = p.Hd;
  c.zz_C = p.T / 2;
  c.zz_T = p.T;
  c.zz_D = 1;
  c.zz_B = p.B;
  c.status = status_of(ws);
  return launch_gemm(c, static_cast<cudaStream_t>(stream));
}

tsp_status tsp_rank_kv_gather(tsp_plan_t plan, const tsp_bf16* kv_all, tsp_bf16* kn,
                              tsp_bf16* vn, void* stream) {
  TSP_TRY(rank_check(plan, "tsp_rank_kv_gather"));
  TSP_TRY(check_ptrs({kv_all, kn, vn}, "tsp_rank_kv_gather"));
  return launch_kv_gather_kv(plan->p, kv_all, kn, vn, static_cast<cudaStream_t>(stream));
}

tsp_status tsp_rank_attention(tsp_plan_t plan, int r, const tsp_bf16* q_r, const tsp_bf16* kn,
                              const tsp_bf16* vn, tsp_bf16* o_r, void* ws, void* stream) {
  TSP_TRY(rank_check(plan, "tsp_rank_attention"));
  TSP_TRY(check_ptrs({q_r, kn, vn, o_r}, "tsp_rank_attention"));
  TSP_TRY(check_ws(ws, "tsp_rank_attention"));
  const Plan& p = plan->p;
  if (r < 0 || r >= p.D) return fail(TSP_ERR_INVALID_ARG, "tsp_rank_attention: rank out of range");
  AttentionCall a{};
  a.qkv = q_r;
  a.ld_qkv = p.Hd;
  a.kn = kn;
  a.vn = vn;
  a.ld_kv = p.Hd;
  a.o = o_r;
  a.ld_o = p.Hd;
  a.o_col0 = 0;
  a.S = p.S;
  a.T = p.T;
  a.C = p.C;
  a.D = p.D;
  a.B = p.B;
  a.heads = p.hpr;
  a.d = p.d;
  a.status = status_of(ws);
  a.q_row0 = (int64_t)r * p.T;  // rank r's rows of each sequence's rank-major layout
  a.q_rows = p.T;
  return launch_attention(a, static_cast<cudaStream_t>(stream));
}

tsp_status tsp_rank_o_accumulate(tsp_plan_t plan, const tsp_bf16* o_r, const tsp_bf16* attn_shard,
                                 const void* residual, int residual_f32, float* acc_r,
                                 tsp_bf16* h_r, void* ws, void* stream) {
  TSP_TRY(rank_check(plan, "tsp_rank_o_accumulate"));
  TSP_TRY(check_ptrs({o_r, attn_shard, residual, acc_r, h_r}, "tsp_rank_o_accumulate"));
  TSP_TRY(check_ws(ws, "tsp_rank_o_accumulate"));
  const Plan& p = plan->p;
  GemmCall c{};
  c.epi = EPI_RESIDUAL;
  c.A = o_r;
  c.lda = p.Hd;
  c.M = (int64_t)p.B * p.T;
  c.B = static_cast<const uint16_t*>(static_cast<const void*>(attn_shard)) + shard_layout(p).o_off;
  c.ldb = p.Hd;
  c.b_rows = p.H;
  c.b_row0 = 0;
  c.N = p.H;
  c.K = p.Hd;
  c.C = h_r;
  c.ldc = p.H;
  c.R = residual;
  c.ldr = p.H;
  c.residual_f32 = residual_f32 ? 1 : 0;
  c.C32 = acc_r;
  c.status = status_of(ws);
  return launch_gemm(c, static_cast<cudaStream_t>(stream));
}

tsp_status tsp_rank_mlp_step(tsp_plan_t plan, const tsp_bf16* h_r, const tsp_bf16* mlp_shard,
                             const float* residual32, float* acc_r, tsp_bf16* out_r,
                             tsp_bf16* g_r, void* ws, void* stream) {
  TSP_TRY(rank_check(plan, "tsp_rank_mlp_step"));
  TSP_TRY(check_ptrs({h_r, mlp_shard, residual32, acc_r, out_r, g_r}, "tsp_rank_mlp_step"));
  TSP_TRY(check_ws(ws, "tsp_rank_mlp_step"));
  const Plan& p = plan->p;
  const ShardLayout l = shard_layout(p);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const uint16_t* w = static_cast<const uint16_t*>(static_cast<const void*>(mlp_shard));
  GemmCall up{};  // G_r = silu(h_r W1_k^T) * (h_r W3_k^T), [T][Fq] (padded columns 0)
  up.epi = EPI_SWIGLU;
  up.A = h_r;
  up.lda = p.H;
  up.M = (int64_t)p.B * p.T;
  up.B = w;
  up.ldb = p.H;
  up.b_rows = 2 * l.Fq;
  up.b_row0 = 0;
  up.N = 2 * l.Fq;
  up.K = p.H;
  up.C = g_r;
  up.ldc = l.Fq;
  up.status = status_of(ws);
  TSP_TRY(launch_gemm(up, s));
  GemmCall down{};  // acc_r = residual32 + G_r W2_k^T; out_r = bf16(acc_r)
  down.epi = EPI_RESIDUAL;
  down.A = g_r;
  down.lda = l.Fq;
  down.M = (int64_t)p.B * p.T;
  down.B = w + l.w2_off;
  down.ldb = p.Fp;
  down.b_rows = p.H;
  down.b_row0 = 0;
  down.N = p.H;
  down.K = p.Fp;
  down.C = out_r;
  down.ldc = p.H;
  down.R = residual32;
  down.ldr = p.H;
  down.residual_f32 = 1;
  down.C32 = acc_r;
  down.status = status_of(ws);
  return launch_gemm(down, s);
}

}  // extern "C"
