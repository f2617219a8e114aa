// tsp_internal.h - host-side plan object and the launchers of the kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <string>

#include "../../include/tsp.h"

namespace tsp {

struct DevStatus;

// Layout of the caller's workspace (byte offsets, each 256-byte aligned).
struct WorkspaceLayout {
  size_t status;   // DevStatus
  size_t qkv;      // [S][3H/D] Q|K|V of the current attention shard (sharded rows)
  size_t kn, vn;   // [S][H/D] K and V of the current shard in natural token order
  size_t o;        // [S][H]   attention output before the O projection (sharded rows)
  size_t h;        // [S][H]   h = x + Attn(x) (sharded rows), bf16: input of the MLP
  size_t h32;      // [S][H]   the same h in fp32: the residual of the MLP block
  size_t g;        // [S][NF]  gated activation (sharded rows)
  size_t stage_in, stage_out;  // [S][H] natural-order staging for tsp_layer_fwd_host
  size_t total;
};

struct Plan {
  int D;
  int64_t S;
  int H, heads, d, F;
  int64_t T, C;
  int Hd;   // H / D
  int hpr;  // heads / D
  int Fd;   // F / D
  int Fp;   // padded shard width of the MLP
  int NF;   // D * Fp
  size_t wp_qkv, wp_o, wp_w13, wp_w2, wp_elems;
  WorkspaceLayout ws;
};

// Thread-local error message for tsp_last_error.
void set_error(const std::string& msg);
tsp_status fail(tsp_status code, const std::string& msg);
tsp_status cuda_fail(cudaError_t err, const char* what);

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
enum GemmEpilogue { EPI_STORE = 0, EPI_RESIDUAL = 1, EPI_SWIGLU = 2, EPI_QKV_SPLIT = 3 };

struct GemmCall {
  int epi;
  const void* A; int64_t lda; int64_t M;
  const void* B; int64_t ldb; int64_t b_rows; int64_t b_row0;
  int64_t N;  // columns of the product (for EPI_SWIGLU: 2x the output columns)
  int64_t K;
  void* C; int64_t ldc;
  const void* R; int64_t ldr;  // residual (EPI_RESIDUAL): bf16, or fp32 if residual_f32
  int residual_f32;
  void* C32;                   // optional fp32 copy of the output (EPI_RESIDUAL, bf16 residual), row stride ldc
  // EPI_QKV_SPLIT: the N = 3 split_hd columns are Q | K | V; Q rows go to C (ldc),
  // K and V rows to split_k / split_v (row stride split_ld) at the natural token
  // position of the sharded row (zigzag chunk zz_C, tokens per rank zz_T, zz_D ranks)
  void* split_k; void* split_v; int64_t split_ld; int64_t split_hd;
  int64_t zz_C, zz_T; int zz_D;
  int64_t ring_rows;           // rows per rank for the ring K order, 0 = natural order
  int64_t ring_kblocks;        // 64-wide K blocks per shard
  DevStatus* status;
};
tsp_status launch_gemm(const GemmCall& call, cudaStream_t stream);

struct AttentionCall {
  const void* qkv; int64_t ld_qkv;   // Q at columns [j*d, (j+1)*d) for head j of the group
  const void* kn; const void* vn; int64_t ld_kv;
  void* o; int64_t ld_o; int64_t o_col0;
  int64_t S; int64_t T; int64_t C; int D;
  int heads;  // heads in this call
  int d;
  DevStatus* status;
};
tsp_status launch_attention(const AttentionCall& call, cudaStream_t stream);

tsp_status launch_zigzag_index(const Plan& p, int32_t* fwd, int32_t* inv, cudaStream_t s);
tsp_status launch_zigzag_rows(const Plan& p, const void* src, void* dst, int64_t width,
                              bool to_sharded, cudaStream_t s);
tsp_status launch_kv_gather(const Plan& p, const void* qkv, void* kn, void* vn, cudaStream_t s);
tsp_status launch_pack_weights(const Plan& p, const void* Wq, const void* Wk, const void* Wv,
                               const void* Wo, const void* W1, const void* W3, const void* W2,
                               void* wpack, cudaStream_t s);
tsp_status launch_wait_selftest(DevStatus* st, unsigned long long limit_ns, cudaStream_t s);

}  // namespace tsp
