// tsp_internal.h - host-side plan object and the launchers of the kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>
#include <stddef.h>
#include <stdio.h>
#include <stdint.h>

#include <initializer_list>
#include <string>

#include "../../include/tsp.h"

namespace tsp {

struct DevStatus;

// Layout of the caller's workspace (byte offsets, each 256-byte aligned). N = B*S
// rows: every token of the micro-batch.
struct WorkspaceLayout {
  size_t status;   // DevStatus
  size_t qkv;      // [N][max(3, G_att) H/D] Q|K|V of the current attention shard, or the Q
                   //   of the G_att shards of one attention launch (sharded rows)
  size_t kn, vn;   // [N][G_att H/D] K and V of those shards in natural token order
  size_t o;        // [N][H]   attention output before the O projection (sharded rows)
  size_t h;        // [N][H]   h = x + Attn(x) (sharded rows), bf16: input of the MLP
  size_t h32;      // [N][H]   the same h in fp32: the residual of the MLP block
  size_t g;        // [N][NF]  gated activation (sharded rows)
  size_t stage_in, stage_out;  // [N][H] natural-order staging for tsp_layer_fwd_host
  size_t total;
  // backward calls only (after `total`):
  size_t a13;      // [S][2NF] SwiGLU pre-activations A1|A3 (W13's packed column order),
                   //          overwritten in place by their gradients dA1|dA3
  size_t dh32;     // [S][H]   fp32 gradient of h (dout + MLP backward)
  size_t dh;       // [S][H]   the same in bf16 (operand of the attention backward)
  size_t dob;      // [S][H]   gradient of the attention output before W_O
  size_t lse;      // [heads][S] fp32 log-sum-exp (natural log) of each query row
  size_t delta;    // [heads][S] fp32 rowsum(dO * O) of each query row
  size_t qa;       // [D][S][H/D] Q of every shard (sharded rows)
  size_t ka, va;   // [D][S][H/D] K, V of every shard (natural rows)
  size_t dqkv;     // [S][3H]  dQ|dK|dV of shard k at columns [3k H/D, 3(k+1) H/D), sharded rows
  size_t total_bwd;
};

struct Plan {
  int D;
  int64_t S;  // tokens of one sequence
  int B;      // sequences of the micro-batch (rank-major layout [D][B][T][H])
  int64_t N;  // B * S: rows of every GEMM and of the activation buffers
  int H, heads, d, F;
  int64_t T, C;
  int Hd;   // H / D
  int hpr;  // heads / D
  int Fd;   // F / D
  int Fp;   // padded shard width of the MLP
  int NF;   // D * Fp
  int G_att;  // shards whose attention runs in one launch (divides D)
  int64_t ld_stat;  // row stride of the per-head row statistics (N rounded up to 128)
  size_t wp_qkv, wp_o, wp_w13, wp_w2, wp_elems;
  WorkspaceLayout ws;
};

// Raise a kernel's dynamic shared-memory limit to `bytes`, once per (kernel, device):
// the setting lasts for the context, so later launches make no driver call here
// (which also keeps a stream capture free of it).
tsp_status ensure_smem_limit(const void* kernel, int bytes, const char* what);

// Thread-local error message for tsp_last_error.
void set_error(const std::string& msg);
tsp_status fail(tsp_status code, const std::string& msg);
tsp_status cuda_fail(cudaError_t err, const char* what);

#define TSP_TRY(expr)              \
  do {                             \
    tsp_status st_ = (expr);       \
    if (st_ != TSP_OK) return st_; \
  } while (0)

inline size_t align256(size_t v) { return (v + 255) & ~static_cast<size_t>(255); }
inline bool al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline bool al256(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 255u) == 0; }
inline DevStatus* status_of(void* ws) { return static_cast<DevStatus*>(ws); }
template <class T>
T* at(void* ws, size_t off) {
  return reinterpret_cast<T*>(static_cast<uint8_t*>(ws) + off);
}

// Argument checks of the C entry points (they set the error message).
inline tsp_status check_ptrs(std::initializer_list<const void*> ptrs, const char* what) {
  for (const void* q : ptrs) {
    if (!q) return fail(TSP_ERR_INVALID_ARG, std::string(what) + ": null pointer");
    if (!al16(q)) return fail(TSP_ERR_INVALID_ARG, std::string(what) + ": pointer not 16-byte aligned");
  }
  return TSP_OK;
}
inline tsp_status check_ws(void* ws, const char* what) {
  if (!ws) return fail(TSP_ERR_INVALID_ARG, std::string(what) + ": null workspace");
  if (!al256(ws)) return fail(TSP_ERR_INVALID_ARG, std::string(what) + ": workspace not 256-byte aligned");
  return TSP_OK;
}

// cuTensorMapEncodeTiled through the runtime's driver entry point (no libcuda link).
// 2D bf16 map: inner dimension `inner` elements (contiguous), `outer` rows,
// `row_stride_bytes` between rows, box {box_inner, box_outer}, 128-byte swizzle,
// out-of-bounds elements read as zero.
tsp_status make_tmap_2d_bf16(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer,
                             uint64_t row_stride_bytes, uint32_t box_inner, uint32_t box_outer);

int sm_count();                     // of the current device (cached per device)
unsigned long long wait_limit_ns();  // bound of the device-side waits

// ---------------------------------------------------------------- launchers
// C[M][N] = A[M][K] * B[N][K]^T with the epilogues below. A rows have stride lda
// elements; B is rows [b_row0, b_row0 + N) of a [b_rows][K] matrix (stride ldb).
enum GemmEpilogue {
  EPI_STORE = 0,        // C = bf16(acc)
  EPI_RESIDUAL = 1,     // C = bf16(acc + R)
  EPI_SWIGLU = 2,       // C = bf16(silu(gate) * up) of each 256-column tile
  EPI_QKV_SPLIT = 3,    // Q | K | V columns split (see split_* below)
  EPI_STORE_F32 = 4,    // C32 = acc in fp32 (weight gradients)
  EPI_SWIGLU_SAVE = 5,  // EPI_SWIGLU, and the raw pre-activations to C2 (same columns)
  EPI_SWIGLU_BWD = 6,   // acc = dG [.. x NF]; A1|A3 read from C2; dA1|dA3 to C (C2's order)
};

struct GemmCall {
  int epi;
  // A: [M][K] (K-major) or, with a_mn, [K][M]; row stride lda elements.
  // B: rows [b_row0, b_row0 + N) of a [b_rows][K] matrix, or with b_mn columns
  // [b_row0, b_row0 + N) of a [K][b_rows] matrix; row stride ldb elements.
  const void* A; int64_t lda; int64_t M; int a_mn;
  const void* B; int64_t ldb; int64_t b_rows; int64_t b_row0; int b_mn;
  void* C2; int64_t ldc2;      // EPI_SWIGLU_SAVE / EPI_SWIGLU_BWD pre-activations
  int64_t N;  // columns of the product (for EPI_SWIGLU: 2x the output columns)
  int64_t K;
  void* C; int64_t ldc;
  const void* R; int64_t ldr;  // residual (EPI_RESIDUAL): bf16, or fp32 if residual_f32
  int residual_f32;
  void* C32;                   // optional fp32 copy of the output (EPI_RESIDUAL), row stride ldc;
                               // with an fp32 residual it may be the residual itself (in place)
  // EPI_QKV_SPLIT: the N = 3 n split_hd columns are Q | K | V of n shards in turn (shard j's
  // columns land at offset j split_hd of each destination); Q rows go to C (ldc),
  // K and V rows to split_k / split_v (row stride split_ld) at the natural token
  // position of the sharded row (zigzag chunk zz_C, tokens per rank zz_T, zz_D ranks,
  // zz_B sequences: sharded row (r*zz_B + b)*zz_T + l -> natural row b*S + pos(r, l))
  void* split_k; void* split_v; int64_t split_ld; int64_t split_hd;
  int64_t zz_C, zz_T; int zz_D; int zz_B;
  int64_t zz_row0;             // sharded row of A's first row (a product over part of the rows)
  int64_t ring_rows;           // rows per rank for the ring K order, 0 = natural order
  int64_t ring_kblocks;        // 64-wide K blocks per shard
  int ring_rank0;              // rank of the launch's first row (ring order)
  DevStatus* status;
};
tsp_status launch_gemm(const GemmCall& call, cudaStream_t stream);

// Rows of qkv, o and lse are the sharded rows of a micro-batch of B sequences
// ([D][B][T] rank-major); kn/vn rows are natural rows b*S + t. B = 0 means 1.
struct AttentionCall {
  const void* qkv; int64_t ld_qkv;   // Q at columns [j*d, (j+1)*d) for head j of the group
  const void* kn; const void* vn; int64_t ld_kv;
  void* o; int64_t ld_o; int64_t o_col0;
  float* lse; int64_t ld_lse;  // optional [heads][ld_lse] log-sum-exp (base 2) per row
  int64_t S; int64_t T; int64_t C; int D; int B;
  int heads;  // heads in this call
  int d;
  DevStatus* status;
  // q_rows > 0: only the sharded query rows [q_row0, q_row0 + q_rows) of the (single)
  // sequence, e.g. one rank's T rows; qkv, o and lse then hold those rows from row 0
  int64_t q_row0, q_rows;
};
tsp_status launch_attention(const AttentionCall& call, cudaStream_t stream);

// Attention backward of the heads of one shard (all ranks' queries).
//   q [S][ld_q] (sharded rows), k, v [S][ld_kv] (natural rows), head j at columns j*d;
//   dout [S][ld_do] (sharded rows), head j at columns do_col0 + j*d;
//   lse, delta [heads][ld_stat] fp32 per sharded row (lse from the forward, base 2;
//   delta = rowsum(dO * O));
//   dq, dk, dv [S][ld_dqkv] bf16 written at sharded rows, head j at columns j*d of
//   each pointer (dK/dV rows at the sharded row of their key position).
struct AttentionBwdCall {
  const void* q; int64_t ld_q;
  const void* k; const void* v; int64_t ld_kv;
  const void* dout; int64_t ld_do; int64_t do_col0;
  const float* lse; const float* delta; int64_t ld_stat;
  void* dq; void* dk; void* dv; int64_t ld_dqkv;
  int64_t S, T, C; int D;
  int B;  // sequences of the micro-batch ([D][B][T] sharded rows, K/V rows b*S + t); 0 = 1
  int heads, d;
  DevStatus* status;
};
tsp_status launch_attention_bwd(const AttentionBwdCall& call, cudaStream_t stream);
// delta[j][r] = sum_c dout[r][j*d + c] * o[r][j*d + c] for heads j < heads, rows r < S
tsp_status launch_attention_delta(const void* o, const void* dout, int64_t ld, int heads, int d,
                                  int64_t S, float* delta, int64_t ld_stat, cudaStream_t stream);

tsp_status launch_zigzag_index(const Plan& p, int32_t* fwd, int32_t* inv, cudaStream_t s);
tsp_status launch_zigzag_rows(const Plan& p, const void* src, void* dst, int64_t width,
                              bool to_sharded, cudaStream_t s);
tsp_status launch_kv_gather(const Plan& p, const void* qkv, void* kn, void* vn, cudaStream_t s);
// the same from K|V rows ([D][B][T][2 H/D], K then V per row) to natural order
tsp_status launch_kv_gather_kv(const Plan& p, const void* kv, void* kn, void* vn, cudaStream_t s);
tsp_status launch_pack_weights(const Plan& p, const void* Wq, const void* Wk, const void* Wv,
                               const void* Wo, const void* W1, const void* W3, const void* W2,
                               void* wpack, cudaStream_t s);
tsp_status launch_unpack_grads(const Plan& p, const float* dwpack, float* dWq, float* dWk,
                               float* dWv, float* dWo, float* dW1, float* dW3, float* dW2,
                               cudaStream_t s);
tsp_status launch_wait_selftest(DevStatus* st, unsigned long long limit_ns, cudaStream_t s);

// Steps of the forward (api.cu), shared with the backward orchestration.
tsp_status qkv_projection_gathered(const Plan& p, int k, const void* xs, const void* wpack,
                                   void* q, void* kn, void* vn, void* ws, cudaStream_t s);
// Q/K/V projections and attention of every shard (G_att shards per attention launch),
// o (and lse when not NULL: [heads][ld_stat]) written for every head.
tsp_status attention_shards(const Plan& p, const void* xs, const void* wpack, void* o, void* ws,
                            cudaStream_t s, float* lse, bool first_group_projected = false);
// lse (optional): [heads/D][ld_stat], the rows of shard k's heads.
tsp_status causal_attention(const Plan& p, int k, const void* qkv, int64_t ld_q, const void* kn,
                            const void* vn, void* o, void* ws, cudaStream_t s,
                            float* lse = nullptr);
tsp_status o_projection(const Plan& p, const void* o, const void* wpack, const void* residual,
                        void* out, void* out32, void* ws, cudaStream_t s);
tsp_status attention_block(const Plan& p, const void* xs, const void* wpack, const void* residual,
                           void* out, void* out32, void* ws, cudaStream_t s);
// G = SwiGLU(hs) then out = G W2^T (+ residual, fp32 when residual_f32) in ring order.
tsp_status mlp_block(const Plan& p, const void* hs, const void* wpack, const void* residual,
                     int residual_f32, void* out, void* ws, cudaStream_t s);

// An NVTX range around the host-side enqueue of one step of the schedules (a
// broadcast iteration's projection and attention, the O projection, the MLP ring),
// so that a trace tool shows which shard step issued which kernels. NVTX3 is
// header-only: without a tool attached a range costs a few nanoseconds.
class NvtxRange {
 public:
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  NvtxRange(const char* fmt, int a, int b) {
    char buf[96];
    snprintf(buf, sizeof buf, fmt, a, b);
    nvtxRangePushA(buf);
  }
  ~NvtxRange() { nvtxRangePop(); }
  NvtxRange(const NvtxRange&) = delete;
  NvtxRange& operator=(const NvtxRange&) = delete;
};

}  // namespace tsp

struct tsp_plan_s {
  tsp::Plan p;
};

inline tsp_status tsp_check_plan(tsp_plan_t plan) {
  return plan ? TSP_OK : tsp::fail(TSP_ERR_INVALID_ARG, "null plan");
}
