// backward.cu - the C ABI of the TSP layer backward (declared in include/tsp.h).
//
// "Folding Tensor and Sequence Parallelism for Memory-Efficient Transformer Training
// & Inference" targets training but describes only the forward schedules (section
// 2); the backward here is the chain rule of the same layer run under those
// schedules in reverse:
//   MLP, ring: rank r at ring step t holds shard k = (r + t) mod D, forms its own
//     dG, dA1|dA3 for that shard, adds the shard's term of dh_r locally (the K loop
//     of the dh product starts at rank r's shard and wraps around) and its tokens'
//     contribution to the shard's weight gradients; on one GPU the contributions
//     of all ranks are the K (token) dimension of one weight-gradient product.
//   attention, broadcast: per shard k, dO = dh W_O (columns of shard k), the
//     attention backward of every rank's queries, whose K/V gradients land at the
//     key's owner (the reverse of the all-gather), then dx and the shard's weight
//     gradients.
// A micro-batch runs every product over all B*S rows: the weight gradients sum the
// tokens of every sequence, the attention backward keeps each sequence to itself.
// Weight gradients are fp32, in the packed layout of the weights (a float array of
// wpack_elems), so each shard's gradient is contiguous like the shard itself.
#include "tsp_device.cuh"
#include "tsp_internal.h"

namespace tsp {
namespace {

// ------------------------------------------------------------------ GEMM steps

// A13 = hs W13^T (W13's packed column order) and G = silu(A1) * A3.
tsp_status swiglu_gate_up_save(const Plan& p, const void* hs, const void* wpack, void* g,
                               void* a13, void* ws, cudaStream_t s) {
  GemmCall c{};
  c.epi = EPI_SWIGLU_SAVE;
  c.A = hs;
  c.lda = p.H;
  c.M = p.N;
  c.B = static_cast<const uint16_t*>(wpack) + p.wp_w13;
  c.ldb = p.H;
  c.b_rows = 2LL * p.NF;
  c.N = 2LL * p.NF;
  c.K = p.H;
  c.C = g;
  c.ldc = p.NF;
  c.C2 = a13;
  c.ldc2 = 2LL * p.NF;
  c.status = status_of(ws);
  return launch_gemm(c, s);
}

// dG = dmlp W2 (all shards' columns), turned into dA1|dA3 by the epilogue, in place
// over the pre-activations A1|A3.
tsp_status swiglu_dgate(const Plan& p, const void* dmlp, const void* wpack, void* a13, void* ws,
                        cudaStream_t s) {
  GemmCall c{};
  c.epi = EPI_SWIGLU_BWD;
  c.A = dmlp;
  c.lda = p.H;
  c.M = p.N;
  c.B = static_cast<const uint16_t*>(wpack) + p.wp_w2;  // [H][NF] = [K][N]
  c.ldb = p.NF;
  c.b_rows = p.NF;
  c.b_mn = 1;
  c.N = p.NF;
  c.K = p.H;
  c.C = a13;
  c.ldc = 2LL * p.NF;
  c.C2 = a13;
  c.ldc2 = 2LL * p.NF;
  c.status = status_of(ws);
  return launch_gemm(c, s);
}

// dhs = dA13 W13 (+ residual, bf16; out32 = the fp32 value) with the ring K order.
tsp_status swiglu_dinput(const Plan& p, const void* da13, const void* wpack, const void* residual,
                         void* out, void* out32, void* ws, cudaStream_t s) {
  GemmCall c{};
  c.epi = residual ? EPI_RESIDUAL : EPI_STORE;
  c.A = da13;
  c.lda = 2LL * p.NF;
  c.M = p.N;
  c.B = static_cast<const uint16_t*>(wpack) + p.wp_w13;  // [2NF][H] = [K][N]
  c.ldb = p.H;
  c.b_rows = p.H;
  c.b_mn = 1;
  c.N = p.H;
  c.K = 2LL * p.NF;
  c.C = out;
  c.ldc = p.H;
  c.R = residual;
  c.ldr = p.H;
  c.C32 = out32;
  c.ring_rows = (int64_t)p.B * p.T;  // rank r's rows of every sequence
  c.ring_kblocks = 2LL * p.Fp / 64;
  c.status = status_of(ws);
  return launch_gemm(c, s);
}

// Weight gradient dW[M][N] = A^T B over the N = B*S tokens of the micro-batch:
// A [N][M], B [N][N] (both token-major, i.e. MN-major operands), fp32 out with row
// stride ldc.
tsp_status weight_grad(const Plan& p, const void* A, int64_t M, const void* B, int64_t N,
                       float* dW, int64_t ldc, void* ws, cudaStream_t s) {
  GemmCall c{};
  c.epi = EPI_STORE_F32;
  c.A = A;
  c.lda = M;
  c.M = M;
  c.a_mn = 1;
  c.B = B;
  c.ldb = N;
  c.b_rows = N;
  c.b_mn = 1;
  c.N = N;
  c.K = p.N;
  c.C32 = dW;
  c.ldc = ldc;
  c.status = status_of(ws);
  return launch_gemm(c, s);
}

// MLP backward of dmlp at hs: dhs (bf16; + residual and fp32 copy when given) and
// the W1/W3/W2 gradients in dwpack.
tsp_status mlp_backward(const Plan& p, const void* hs, const void* wpack, const void* dmlp,
                        const void* residual, void* dhs, void* dhs32, float* dwpack, void* ws,
                        cudaStream_t s) {
  NvtxRange range("tsp MLP backward (ring in reverse)");
  void* g = at<void>(ws, p.ws.g);
  void* a13 = at<void>(ws, p.ws.a13);
  TSP_TRY(swiglu_gate_up_save(p, hs, wpack, g, a13, ws, s));
  TSP_TRY(weight_grad(p, dmlp, p.H, g, p.NF, dwpack + p.wp_w2, p.NF, ws, s));  // dW2 = dmlp^T G
  TSP_TRY(swiglu_dgate(p, dmlp, wpack, a13, ws, s));
  TSP_TRY(swiglu_dinput(p, a13, wpack, residual, dhs, dhs32, ws, s));
  return weight_grad(p, a13, 2LL * p.NF, hs, p.H, dwpack + p.wp_w13, p.H, ws, s);  // dW13
}

// ------------------------------------------------------------------ attention

// dO = dattn W_O (every shard's columns), bf16.
tsp_status o_projection_dgrad(const Plan& p, const void* dattn, const void* wpack, void* dob,
                              void* ws, cudaStream_t s) {
  GemmCall c{};
  c.epi = EPI_STORE;
  c.A = dattn;
  c.lda = p.H;
  c.M = p.N;
  c.B = static_cast<const uint16_t*>(wpack) + p.wp_o;  // [H][H] = [K][N]
  c.ldb = p.H;
  c.b_rows = p.H;
  c.b_mn = 1;
  c.N = p.H;
  c.K = p.H;
  c.C = dob;
  c.ldc = p.H;
  c.status = status_of(ws);
  return launch_gemm(c, s);
}

// dxs = dQKV W_QKV (+ fp32 residual): K loop over the shards in broadcast order.
tsp_status qkv_dgrad(const Plan& p, const void* dqkv, const void* wpack, const float* residual32,
                     void* dxs, void* ws, cudaStream_t s) {
  GemmCall c{};
  c.epi = residual32 ? EPI_RESIDUAL : EPI_STORE;
  c.A = dqkv;
  c.lda = 3LL * p.H;
  c.M = p.N;
  c.B = static_cast<const uint16_t*>(wpack) + p.wp_qkv;  // [3H][H] = [K][N]
  c.ldb = p.H;
  c.b_rows = p.H;
  c.b_mn = 1;
  c.N = p.H;
  c.K = 3LL * p.H;
  c.C = dxs;
  c.ldc = p.H;
  c.R = residual32;
  c.ldr = p.H;
  c.residual_f32 = residual32 ? 1 : 0;
  c.status = status_of(ws);
  return launch_gemm(c, s);
}

// Attention backward of shard k's heads: dQ, dK, dV into the shard's columns of dqkv;
// lse and delta hold the rows of the shard's heads.
tsp_status attention_shard_backward(const Plan& p, int k, const void* q, const void* kn,
                                    const void* vn, const void* dob, const float* lse,
                                    const float* delta, void* dqkv, void* ws, cudaStream_t s) {
  AttentionBwdCall a{};
  a.q = q;
  a.ld_q = p.Hd;
  a.k = kn;
  a.v = vn;
  a.ld_kv = p.Hd;
  a.dout = dob;
  a.ld_do = p.H;
  a.do_col0 = (int64_t)k * p.Hd;
  a.lse = lse;
  a.delta = delta;
  a.ld_stat = p.ld_stat;
  uint16_t* base = static_cast<uint16_t*>(dqkv) + (int64_t)k * 3 * p.Hd;
  a.dq = base;
  a.dk = base + p.Hd;
  a.dv = base + 2 * p.Hd;
  a.ld_dqkv = 3LL * p.H;
  a.S = p.S;
  a.T = p.T;
  a.C = p.C;
  a.D = p.D;
  a.B = p.B;
  a.heads = p.hpr;
  a.d = p.d;
  a.status = status_of(ws);
  return launch_attention_bwd(a, s);
}

// The attention forward again, keeping every shard's Q, K, V and, when o is not
// NULL, the attention output before W_O (sharded rows) and each row's lse. With
// o == NULL only the projections run (a training forward kept o and lse).
tsp_status attention_recompute(const Plan& p, const void* xs, const void* wpack, void* ws,
                               cudaStream_t s, void* o, float* lse) {
  uint16_t* qa = at<uint16_t>(ws, p.ws.qa);
  uint16_t* ka = at<uint16_t>(ws, p.ws.ka);
  uint16_t* va = at<uint16_t>(ws, p.ws.va);
  const int64_t shard = p.N * p.Hd;
  for (int k = 0; k < p.D; ++k) {
    NvtxRange range("tsp attention recompute shard %d of %d", k, p.D);
    TSP_TRY(qkv_projection_gathered(p, k, xs, wpack, qa + k * shard, ka + k * shard,
                                    va + k * shard, ws, s));
    if (o)
      TSP_TRY(causal_attention(p, k, qa + k * shard, p.Hd, ka + k * shard, va + k * shard, o, ws,
                               s, lse + (int64_t)k * p.hpr * p.ld_stat));
  }
  return TSP_OK;
}

// Layout of the activations a training forward keeps (byte offsets, 256-aligned):
// o [N][H] bf16, then lse [heads][ld_stat] fp32.
size_t saved_lse_offset(const Plan& p) { return ((size_t)p.N * p.H * 2 + 255) & ~(size_t)255; }
size_t saved_bytes(const Plan& p) {
  return saved_lse_offset(p) + (((size_t)p.heads * p.ld_stat * 4 + 255) & ~(size_t)255);
}

// Backward of the attention block for dattn (bf16), after every shard's Q/K/V are in
// the workspace: dxs = (dAttn/dx)^T dattn (+ residual32), and the W_Q/W_K/W_V/W_O
// gradients. o is the attention output before W_O and lse the rows' log-sum-exp
// ([heads][ld_stat]), either recomputed into the workspace or kept by a training
// forward.
tsp_status attention_backward(const Plan& p, const void* xs, const void* wpack, const void* dattn,
                              const float* residual32, void* dxs, float* dwpack, void* ws,
                              cudaStream_t s, const void* o, const float* lse) {
  const uint16_t* qa = at<uint16_t>(ws, p.ws.qa);
  const uint16_t* ka = at<uint16_t>(ws, p.ws.ka);
  const uint16_t* va = at<uint16_t>(ws, p.ws.va);
  void* dob = at<void>(ws, p.ws.dob);
  void* dqkv = at<void>(ws, p.ws.dqkv);
  float* delta = at<float>(ws, p.ws.delta);
  TSP_TRY(o_projection_dgrad(p, dattn, wpack, dob, ws, s));
  TSP_TRY(weight_grad(p, dattn, p.H, o, p.H, dwpack + p.wp_o, p.H, ws, s));  // dWo = dattn^T o
  TSP_TRY(launch_attention_delta(o, dob, p.H, p.heads, p.d, p.N, delta, p.ld_stat, s));
  const int64_t shard = p.N * p.Hd;
  for (int k = 0; k < p.D; ++k) {  // broadcast iteration k, in reverse
    NvtxRange range("tsp attention backward shard %d of %d", k, p.D);
    TSP_TRY(attention_shard_backward(p, k, qa + k * shard, ka + k * shard, va + k * shard, dob,
                                     lse + (int64_t)k * p.hpr * p.ld_stat,
                                     delta + (int64_t)k * p.hpr * p.ld_stat, dqkv, ws, s));
  }
  TSP_TRY(qkv_dgrad(p, dqkv, wpack, residual32, dxs, ws, s));
  return weight_grad(p, dqkv, 3LL * p.H, xs, p.H, dwpack + p.wp_qkv, p.H, ws, s);  // dW_QKV
}

// The layer backward once Q/K/V of every shard are in the workspace and o / lse are
// available: h = x + o W_O^T, dh = dout + MLP backward, dxs = dh + attention backward.
tsp_status layer_backward_from(const Plan& p, const void* xs, const void* wpack, const void* dout,
                               void* dxs, float* dwpack, void* ws, cudaStream_t s, const void* o,
                               const float* lse) {
  void* h = at<void>(ws, p.ws.h);
  float* h32 = at<float>(ws, p.ws.h32);
  void* dh = at<void>(ws, p.ws.dh);
  float* dh32 = at<float>(ws, p.ws.dh32);
  TSP_TRY(o_projection(p, o, wpack, xs, h, h32, ws, s));
  // dh = dout + MLP backward of dout at h (fp32, and bf16 for the products below)
  TSP_TRY(mlp_backward(p, h, wpack, dout, dout, dh, dh32, dwpack, ws, s));
  // dx = dh + attention backward of dh
  return attention_backward(p, xs, wpack, dh, dh32, dxs, dwpack, ws, s, o, lse);
}

}  // namespace
}  // namespace tsp

using namespace tsp;

extern "C" {

size_t tsp_bwd_workspace_bytes(tsp_plan_t plan) { return plan ? plan->p.ws.total_bwd : 0; }

tsp_status tsp_mlp_bwd(tsp_plan_t plan, const tsp_bf16* hs, const tsp_bf16* wpack,
                       const tsp_bf16* dmlp, tsp_bf16* dhs, float* dwpack, void* ws,
                       void* stream) {
  TSP_TRY(tsp_check_plan(plan));
  TSP_TRY(check_ptrs({hs, wpack, dmlp, dhs, dwpack}, "tsp_mlp_bwd"));
  TSP_TRY(check_ws(ws, "tsp_mlp_bwd"));
  if (dhs == hs || dhs == dmlp) return fail(TSP_ERR_INVALID_ARG, "tsp_mlp_bwd: dhs aliases an input");
  return mlp_backward(plan->p, hs, wpack, dmlp, nullptr, dhs, nullptr, dwpack, ws,
                      static_cast<cudaStream_t>(stream));
}

tsp_status tsp_attention_bwd(tsp_plan_t plan, const tsp_bf16* xs, const tsp_bf16* wpack,
                             const tsp_bf16* dattn, tsp_bf16* dxs, float* dwpack, void* ws,
                             void* stream) {
  TSP_TRY(tsp_check_plan(plan));
  TSP_TRY(check_ptrs({xs, wpack, dattn, dxs, dwpack}, "tsp_attention_bwd"));
  TSP_TRY(check_ws(ws, "tsp_attention_bwd"));
  if (dxs == xs || dxs == dattn) return fail(TSP_ERR_INVALID_ARG, "tsp_attention_bwd: dxs aliases an input");
  const Plan& p = plan->p;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  void* o = at<void>(ws, p.ws.o);
  float* lse = at<float>(ws, p.ws.lse);
  TSP_TRY(attention_recompute(p, xs, wpack, ws, s, o, lse));
  return attention_backward(p, xs, wpack, dattn, nullptr, dxs, dwpack, ws, s, o, lse);
}

tsp_status tsp_layer_bwd(tsp_plan_t plan, const tsp_bf16* xs, const tsp_bf16* wpack,
                         const tsp_bf16* dout, tsp_bf16* dxs, float* dwpack, void* ws,
                         void* stream) {
  TSP_TRY(tsp_check_plan(plan));
  TSP_TRY(check_ptrs({xs, wpack, dout, dxs, dwpack}, "tsp_layer_bwd"));
  TSP_TRY(check_ws(ws, "tsp_layer_bwd"));
  if (dxs == xs || dxs == dout) return fail(TSP_ERR_INVALID_ARG, "tsp_layer_bwd: dxs aliases an input");
  const Plan& p = plan->p;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  void* o = at<void>(ws, p.ws.o);
  float* lse = at<float>(ws, p.ws.lse);
  // forward recompute: every shard's Q/K/V, lse and o
  TSP_TRY(attention_recompute(p, xs, wpack, ws, s, o, lse));
  return layer_backward_from(p, xs, wpack, dout, dxs, dwpack, ws, s, o, lse);
}

size_t tsp_saved_bytes(tsp_plan_t plan) { return plan ? saved_bytes(plan->p) : 0; }

tsp_status tsp_layer_fwd_train(tsp_plan_t plan, const tsp_bf16* xs, const tsp_bf16* wpack,
                               tsp_bf16* out, void* saved, void* ws, void* stream) {
  TSP_TRY(tsp_check_plan(plan));
  TSP_TRY(check_ptrs({xs, wpack, out, saved}, "tsp_layer_fwd_train"));
  TSP_TRY(check_ws(ws, "tsp_layer_fwd_train"));
  if (out == xs) return fail(TSP_ERR_INVALID_ARG, "tsp_layer_fwd_train: out aliases xs");
  const Plan& p = plan->p;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  void* o = saved;
  float* lse = at<float>(saved, saved_lse_offset(p));
  // the layer forward's steps, with o and each row's lse landing in `saved`
  TSP_TRY(attention_shards(p, xs, wpack, o, ws, s, lse));
  void* h = at<void>(ws, p.ws.h);
  void* h32 = at<void>(ws, p.ws.h32);
  TSP_TRY(o_projection(p, o, wpack, xs, h, h32, ws, s));
  return mlp_block(p, h, wpack, h32, 1, out, ws, s);
}

tsp_status tsp_layer_bwd_saved(tsp_plan_t plan, const tsp_bf16* xs, const tsp_bf16* wpack,
                               const void* saved, const tsp_bf16* dout, tsp_bf16* dxs,
                               float* dwpack, void* ws, void* stream) {
  TSP_TRY(tsp_check_plan(plan));
  TSP_TRY(check_ptrs({xs, wpack, saved, dout, dxs, dwpack}, "tsp_layer_bwd_saved"));
  TSP_TRY(check_ws(ws, "tsp_layer_bwd_saved"));
  if (dxs == xs || dxs == dout) return fail(TSP_ERR_INVALID_ARG, "tsp_layer_bwd_saved: dxs aliases an input");
  const Plan& p = plan->p;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const void* o = saved;
  const float* lse = at<float>(const_cast<void*>(saved), saved_lse_offset(p));
  // only the projections are recomputed: Q/K/V of every shard, then h
  TSP_TRY(attention_recompute(p, xs, wpack, ws, s, nullptr, nullptr));
  return layer_backward_from(p, xs, wpack, dout, dxs, dwpack, ws, s, o, lse);
}

tsp_status tsp_causal_attention_lse(tsp_plan_t plan, int shard, const tsp_bf16* q,
                                    const tsp_bf16* kn, const tsp_bf16* vn, tsp_bf16* o,
                                    float* lse, void* ws, void* stream) {
  TSP_TRY(tsp_check_plan(plan));
  TSP_TRY(check_ptrs({q, kn, vn, o, lse}, "tsp_causal_attention_lse"));
  TSP_TRY(check_ws(ws, "tsp_causal_attention_lse"));
  if (shard < 0 || shard >= plan->p.D)
    return fail(TSP_ERR_INVALID_ARG, "tsp_causal_attention_lse: shard out of range");
  const Plan& p = plan->p;
  return causal_attention(p, shard, q, p.Hd, kn, vn, o, ws, static_cast<cudaStream_t>(stream), lse);
}

tsp_status tsp_causal_attention_bwd(tsp_plan_t plan, int shard, const tsp_bf16* q,
                                    const tsp_bf16* kn, const tsp_bf16* vn, const tsp_bf16* o,
                                    const tsp_bf16* dout, const float* lse, float* delta,
                                    tsp_bf16* dqkv, void* ws, void* stream) {
  TSP_TRY(tsp_check_plan(plan));
  TSP_TRY(check_ptrs({q, kn, vn, o, dout, lse, delta, dqkv}, "tsp_causal_attention_bwd"));
  TSP_TRY(check_ws(ws, "tsp_causal_attention_bwd"));
  if (shard < 0 || shard >= plan->p.D)
    return fail(TSP_ERR_INVALID_ARG, "tsp_causal_attention_bwd: shard out of range");
  const Plan& p = plan->p;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int64_t col = (int64_t)shard * p.Hd;
  TSP_TRY(launch_attention_delta(static_cast<const uint16_t*>(o) + col,
                                 static_cast<const uint16_t*>(dout) + col, p.H, p.hpr, p.d, p.N,
                                 delta, p.ld_stat, s));
  return attention_shard_backward(p, shard, q, kn, vn, dout, lse, delta, dqkv, ws, s);
}

tsp_status tsp_unpack_weight_grads(tsp_plan_t plan, const float* dwpack, float* dWq, float* dWk,
                                   float* dWv, float* dWo, float* dW1, float* dW3, float* dW2,
                                   void* stream) {
  TSP_TRY(tsp_check_plan(plan));
  TSP_TRY(check_ptrs({dwpack}, "tsp_unpack_weight_grads"));
  return launch_unpack_grads(plan->p, dwpack, dWq, dWk, dWv, dWo, dW1, dW3, dW2,
                             static_cast<cudaStream_t>(stream));
}

}  // extern "C"
