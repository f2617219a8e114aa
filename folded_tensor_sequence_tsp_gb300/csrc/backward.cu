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
  c.M = p.S;
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
  c.M = p.S;
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
  c.M = p.S;
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
  c.ring_rows = p.T;
  c.ring_kblocks = 2LL * p.Fp / 64;
  c.status = status_of(ws);
  return launch_gemm(c, s);
}

// Weight gradient dW[M][N] = A^T B over the S tokens: A [S][M], B [S][N] (both
// token-major, i.e. MN-major operands), fp32 out with row stride ldc.
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
  c.K = p.S;
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
  void* g = at<void>(ws, p.ws.g);
  void* a13 = at<void>(ws, p.ws.a13);
  TSP_TRY(swiglu_gate_up_save(p, hs, wpack, g, a13, ws, s));
  TSP_TRY(weight_grad(p, dmlp, p.H, g, p.NF, dwpack + p.wp_w2, p.NF, ws, s));  // dW2 = dmlp^T G
  TSP_TRY(swiglu_dgate(p, dmlp, wpack, a13, ws, s));
  TSP_TRY(swiglu_dinput(p, a13, wpack, residual, dhs, dhs32, ws, s));
  return weight_grad(p, a13, 2LL * p.NF, hs, p.H, dwpack + p.wp_w13, p.H, ws, s);  // dW13
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

tsp_status tsp_unpack_weight_grads(tsp_plan_t plan, const float* dwpack, float* dWq, float* dWk,
                                   float* dWv, float* dWo, float* dW1, float* dW3, float* dW2,
                                   void* stream) {
  TSP_TRY(tsp_check_plan(plan));
  TSP_TRY(check_ptrs({dwpack}, "tsp_unpack_weight_grads"));
  return launch_unpack_grads(plan->p, dwpack, dWq, dWk, dWv, dWo, dW1, dW3, dW2,
                             static_cast<cudaStream_t>(stream));
}

}  // extern "C"
