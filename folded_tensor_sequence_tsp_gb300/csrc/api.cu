// api.cu - the C ABI of the TSP layer forward (declared in include/tsp.h).
//
// Host orchestration of the schedules of "Folding Tensor and Sequence Parallelism
// for Memory-Efficient Transformer Training & Inference", section 2:
//   attention  broadcast schedule: for shard k = 0..D-1 every rank projects its own
//              tokens with shard k's W_Q/W_K/W_V (one GEMM over all ranks' rows),
//              K/V are gathered along the sequence into natural order, causal
//              attention runs for the h/D heads of the shard; the O projection then
//              accumulates the shards' partial products on chip (its K loop walks
//              the shards in broadcast order).
//   MLP        ring schedule: the gate/up GEMM produces every shard's gated
//              activation; the down GEMM accumulates, for rank r's rows, shard
//              (r + t) mod D at step t in the on-chip accumulator (no all-reduce).
// On one GPU the broadcast and the ring hand-off are reads of a shard in place.
#include <cudaTypedefs.h>

#include <cstdio>
#include <cstdlib>
#include <mutex>
#include <new>
#include <set>
#include <string>
#include <tuple>

#include "tsp_device.cuh"
#include "tsp_internal.h"

namespace tsp {

namespace {
thread_local std::string g_last_error;


typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  });
  return fn;
}

}  // namespace

void set_error(const std::string& msg) { g_last_error = msg; }

tsp_status fail(tsp_status code, const std::string& msg) {
  g_last_error = msg;
  return code;
}

tsp_status ensure_smem_limit(const void* kernel, int bytes, const char* what) {
  static std::mutex mu;
  static std::set<std::tuple<const void*, int, int>> done;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, what);
  const auto key = std::make_tuple(kernel, dev, bytes);
  {
    std::lock_guard<std::mutex> lock(mu);
    if (done.count(key)) return TSP_OK;
  }
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e != cudaSuccess) return cuda_fail(e, what);
  std::lock_guard<std::mutex> lock(mu);
  done.insert(key);
  return TSP_OK;
}

tsp_status cuda_fail(cudaError_t err, const char* what) {
  g_last_error = std::string(what) + ": " + cudaGetErrorString(err);
  return TSP_ERR_CUDA;
}

tsp_status make_tmap_2d_bf16(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer,
                             uint64_t row_stride_bytes, uint32_t box_inner, uint32_t box_outer) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return fail(TSP_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {row_stride_bytes};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    char buf[160];
    snprintf(buf, sizeof buf, "cuTensorMapEncodeTiled failed (%d) for %llux%llu stride %llu",
             (int)r, (unsigned long long)inner, (unsigned long long)outer,
             (unsigned long long)row_stride_bytes);
    return fail(TSP_ERR_CUDA, buf);
  }
  return TSP_OK;
}

int sm_count() {
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 1;
  if (!cached[dev]) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
      n = 1;
    cached[dev] = n;
  }
  return cached[dev];
}

unsigned long long wait_limit_ns() {
  static unsigned long long v = [] {
    const char* e = getenv("TSP_WAIT_LIMIT_NS");
    unsigned long long x = e ? strtoull(e, nullptr, 10) : 0ull;
    return x ? x : 4000000000ull;  // 4 s: far above any legitimate wait
  }();
  return v;
}

// ------------------------------------------------------------------ steps

tsp_status qkv_projection(const Plan& p, int k, const void* xs, const void* wpack, void* qkv,
                          void* ws, cudaStream_t s) {
  GemmCall c{};
  c.epi = EPI_STORE;
  c.A = xs;
  c.lda = p.H;
  c.M = p.N;
  c.B = static_cast<const uint16_t*>(wpack) + p.wp_qkv;
  c.ldb = p.H;
  c.b_rows = 3LL * p.H;
  c.b_row0 = (int64_t)k * 3 * p.Hd;
  c.N = 3LL * p.Hd;
  c.K = p.H;
  c.C = qkv;
  c.ldc = 3LL * p.Hd;
  c.status = status_of(ws);
  return launch_gemm(c, s);
}

// Q/K/V projection of shards k .. k + n - 1 (one product: their packed rows are
// consecutive) with the K/V all-gather fused into the epilogue: Q rows stay in
// sharded order in q [S][ld]; K and V rows land at their natural token positions in
// kn, vn [S][ld] (ld >= n H/D elements; shard k + j's H/D columns start at column
// j H/D of each).
tsp_status qkv_projection_gathered(const Plan& p, int k, int n, const void* xs, const void* wpack,
                                   void* q, void* kn, void* vn, int64_t ld, void* ws,
                                   cudaStream_t s) {
  GemmCall c{};
  c.epi = EPI_QKV_SPLIT;
  c.A = xs;
  c.lda = p.H;
  c.M = p.N;
  c.B = static_cast<const uint16_t*>(wpack) + p.wp_qkv;
  c.ldb = p.H;
  c.b_rows = 3LL * p.H;
  c.b_row0 = (int64_t)k * 3 * p.Hd;
  c.N = 3LL * n * p.Hd;
  c.K = p.H;
  c.C = q;
  c.ldc = ld;
  c.split_k = kn;
  c.split_v = vn;
  c.split_ld = ld;
  c.split_hd = p.Hd;
  c.zz_C = p.C;
  c.zz_T = p.T;
  c.zz_D = p.D;
  c.zz_B = p.B;
  c.status = status_of(ws);
  return launch_gemm(c, s);
}

tsp_status qkv_projection_gathered(const Plan& p, int k, const void* xs, const void* wpack,
                                   void* q, void* kn, void* vn, void* ws, cudaStream_t s) {
  return qkv_projection_gathered(p, k, 1, xs, wpack, q, kn, vn, p.Hd, ws, s);
}

// Attention of the heads of shards k .. k + n - 1 in one launch: q holds their Q
// columns (row stride ld_q: 3H/D for the Q|K|V buffer of tsp_qkv_projection, n H/D
// for the Q buffer of the gathered projection), kn / vn their K / V columns (row
// stride ld_kv); o receives columns [k H/D, (k + n) H/D).
tsp_status causal_attention_shards(const Plan& p, int k, int n, const void* qkv, int64_t ld_q,
                                   const void* kn, const void* vn, int64_t ld_kv, void* o,
                                   void* ws, cudaStream_t s, float* lse) {
  AttentionCall a{};
  a.lse = lse;
  a.ld_lse = p.ld_stat;
  a.qkv = qkv;
  a.ld_qkv = ld_q;
  a.kn = kn;
  a.vn = vn;
  a.ld_kv = ld_kv;
  a.o = o;
  a.ld_o = p.H;
  a.o_col0 = (int64_t)k * p.Hd;
  a.S = p.S;
  a.T = p.T;
  a.C = p.C;
  a.D = p.D;
  a.B = p.B;
  a.heads = n * p.hpr;
  a.d = p.d;
  a.status = status_of(ws);
  return launch_attention(a, s);
}

tsp_status causal_attention(const Plan& p, int k, const void* qkv, int64_t ld_q, const void* kn,
                            const void* vn, void* o, void* ws, cudaStream_t s, float* lse) {
  return causal_attention_shards(p, k, 1, qkv, ld_q, kn, vn, p.Hd, o, ws, s, lse);
}

// The broadcast iterations of the attention block up to O (before W_O): per shard k
// the local projections with the fused K/V all-gather, then causal attention. The
// attention of p.G_att consecutive shards runs as one launch (their Q/K/V side by side
// in the workspace) when one shard alone would not fill the GPU with CTAs; each
// head's result is the same bit for bit. lse (optional) as for causal_attention.
tsp_status attention_shards(const Plan& p, const void* xs, const void* wpack, void* o, void* ws,
                            cudaStream_t s, float* lse, bool first_group_projected) {
  uint16_t* q = at<uint16_t>(ws, p.ws.qkv);
  uint16_t* kn = at<uint16_t>(ws, p.ws.kn);
  uint16_t* vn = at<uint16_t>(ws, p.ws.vn);
  const int G = p.G_att;
  const int64_t ld = (int64_t)G * p.Hd;
  for (int k = 0; k < p.D; k += G) {  // broadcast iterations k .. k + G - 1
    NvtxRange range("tsp attention shards %d..%d", k, k + G - 1);
    // local projections of the G shards (one product), K/V all-gather in the epilogue
    // (the first group's may already be in the workspace: tsp_layer_fwd_host)
    if (k > 0 || !first_group_projected)
      TSP_TRY(qkv_projection_gathered(p, k, G, xs, wpack, q, kn, vn, ld, ws, s));
    TSP_TRY(causal_attention_shards(p, k, G, q, ld, kn, vn, ld, o, ws, s,
                                    lse ? lse + (int64_t)k * p.hpr * p.ld_stat : nullptr));
  }
  return TSP_OK;
}

// out = o W_O^T (+ residual, bf16); with out32 also the fp32 value of out.
tsp_status o_projection(const Plan& p, const void* o, const void* wpack, const void* residual,
                        void* out, void* out32, void* ws, cudaStream_t s) {
  NvtxRange range("tsp O projection (shards accumulated)");
  GemmCall c{};
  c.epi = residual ? EPI_RESIDUAL : EPI_STORE;
  c.A = o;
  c.lda = p.H;
  c.M = p.N;
  c.B = static_cast<const uint16_t*>(wpack) + p.wp_o;
  c.ldb = p.H;
  c.b_rows = p.H;
  c.b_row0 = 0;
  c.N = p.H;
  c.K = p.H;
  c.C = out;
  c.ldc = p.H;
  c.R = residual;
  c.ldr = p.H;
  c.C32 = out32;
  c.status = status_of(ws);
  return launch_gemm(c, s);
}

tsp_status swiglu_gate_up(const Plan& p, const void* hs, const void* wpack, void* g, void* ws,
                          cudaStream_t s) {
  GemmCall c{};
  c.epi = EPI_SWIGLU;
  c.A = hs;
  c.lda = p.H;
  c.M = p.N;
  c.B = static_cast<const uint16_t*>(wpack) + p.wp_w13;
  c.ldb = p.H;
  c.b_rows = 2LL * p.NF;
  c.b_row0 = 0;
  c.N = 2LL * p.NF;
  c.K = p.H;
  c.C = g;
  c.ldc = p.NF;
  c.status = status_of(ws);
  return launch_gemm(c, s);
}

// out = G W2^T (+ residual: bf16, or fp32 when residual_f32) in ring order.
tsp_status swiglu_down(const Plan& p, const void* g, const void* wpack, const void* residual,
                       int residual_f32, void* out, void* ws, cudaStream_t s) {
  GemmCall c{};
  c.epi = residual ? EPI_RESIDUAL : EPI_STORE;
  c.A = g;
  c.lda = p.NF;
  c.M = p.N;
  c.B = static_cast<const uint16_t*>(wpack) + p.wp_w2;
  c.ldb = p.NF;
  c.b_rows = p.H;
  c.b_row0 = 0;
  c.N = p.H;
  c.K = p.NF;
  c.C = out;
  c.ldc = p.H;
  c.R = residual;
  c.ldr = p.H;
  c.residual_f32 = residual_f32;
  c.ring_rows = (int64_t)p.B * p.T;  // rank r's rows of every sequence
  c.ring_kblocks = p.Fp / 64;
  c.status = status_of(ws);
  return launch_gemm(c, s);
}

tsp_status attention_block(const Plan& p, const void* xs, const void* wpack, const void* residual,
                           void* out, void* out32, void* ws, cudaStream_t s) {
  void* o = at<void>(ws, p.ws.o);
  TSP_TRY(attention_shards(p, xs, wpack, o, ws, s, nullptr));
  return o_projection(p, o, wpack, residual, out, out32, ws, s);
}

tsp_status mlp_block(const Plan& p, const void* hs, const void* wpack, const void* residual,
                     int residual_f32, void* out, void* ws, cudaStream_t s) {
  NvtxRange range("tsp MLP ring (gate/up, down in ring order)");
  void* g = at<void>(ws, p.ws.g);
  TSP_TRY(swiglu_gate_up(p, hs, wpack, g, ws, s));
  return swiglu_down(p, g, wpack, residual, residual_f32, out, ws, s);
}

// Down projection of rank r's rows only (rows [r B T, (r+1) B T), every sequence of the
// micro-batch), with the fp32 residual; the ring order starts at shard r as in the
// whole-layer launch. When T is a multiple of the 128-row tile, every row block and
// K order is the whole-layer launch's, so the result is the same bit for bit.
tsp_status swiglu_down_rank(const Plan& p, int r, const void* g, const void* wpack,
                            const float* residual32, void* out, void* ws, cudaStream_t s) {
  const int64_t rows = (int64_t)p.B * p.T, r0 = (int64_t)r * rows;
  GemmCall c{};
  c.epi = EPI_RESIDUAL;
  c.A = static_cast<const uint16_t*>(g) + r0 * p.NF;
  c.lda = p.NF;
  c.M = rows;
  c.B = static_cast<const uint16_t*>(wpack) + p.wp_w2;
  c.ldb = p.NF;
  c.b_rows = p.H;
  c.b_row0 = 0;
  c.N = p.H;
  c.K = p.NF;
  c.C = static_cast<uint16_t*>(out) + r0 * p.H;
  c.ldc = p.H;
  c.R = residual32 + r0 * p.H;
  c.ldr = p.H;
  c.residual_f32 = 1;
  c.ring_rows = rows;
  c.ring_rank0 = r;
  c.ring_kblocks = p.Fp / 64;
  c.status = status_of(ws);
  return launch_gemm(c, s);
}

// The Q/K/V product of shards 0 .. n - 1 for rank r's rows only (rows [r B T, (r+1) B T)),
// into q, kn, vn (row stride ld, shard j's columns at j H/D); K/V rows land at their
// natural positions. Every output element takes the same K loop as in the product over
// all rows.
tsp_status qkv_rank(const Plan& p, int r, int n, const void* xs, const void* wpack, void* q,
                    void* kn, void* vn, int64_t ld, void* ws, cudaStream_t s) {
  const int64_t rows = (int64_t)p.B * p.T, r0 = (int64_t)r * rows;
  GemmCall c{};
  c.epi = EPI_QKV_SPLIT;
  c.A = static_cast<const uint16_t*>(xs) + r0 * p.H;
  c.lda = p.H;
  c.M = rows;
  c.B = static_cast<const uint16_t*>(wpack) + p.wp_qkv;
  c.ldb = p.H;
  c.b_rows = 3LL * p.H;
  c.b_row0 = 0;
  c.N = 3LL * n * p.Hd;
  c.K = p.H;
  c.C = static_cast<uint16_t*>(q) + r0 * ld;
  c.ldc = ld;
  c.split_k = kn;
  c.split_v = vn;
  c.split_ld = ld;
  c.split_hd = p.Hd;
  c.zz_C = p.C;
  c.zz_T = p.T;
  c.zz_D = p.D;
  c.zz_B = p.B;
  c.zz_row0 = r0;
  c.status = status_of(ws);
  return launch_gemm(c, s);
}

// A non-blocking stream per device for the host-link copies of tsp_layer_fwd_host,
// created on first use and kept for the life of the process.
tsp_status copy_stream(cudaStream_t* out) {
  static std::mutex mu;
  static cudaStream_t streams[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "copy stream: cudaGetDevice");
  if (dev < 0 || dev >= 64) return fail(TSP_ERR_UNSUPPORTED, "copy stream: device index >= 64");
  std::lock_guard<std::mutex> lock(mu);
  if (!streams[dev]) {
    e = cudaStreamCreateWithFlags(&streams[dev], cudaStreamNonBlocking);
    if (e != cudaSuccess) return cuda_fail(e, "copy stream: cudaStreamCreateWithFlags");
  }
  *out = streams[dev];
  return TSP_OK;
}

// The MLP of tsp_layer_fwd_host with its way back to pinned host memory overlapped:
// G for every row, then per rank r the down projection of r's rows on `s` while the
// copy engine moves the previous ranks' output rows to out_host on a side stream.
// Rank r's rows of sequence b are two runs of C natural rows (chunks r and 2D-1-r),
// so each goes back with one cudaMemcpyAsync. `s` waits for the last copy.
tsp_status mlp_block_to_host(const Plan& p, const void* hs, const void* wpack,
                             const float* residual32, void* out_dev_rows, tsp_bf16* out_host,
                             void* ws, cudaStream_t s) {
  void* g = at<void>(ws, p.ws.g);
  TSP_TRY(swiglu_gate_up(p, hs, wpack, g, ws, s));
  cudaStream_t s2 = nullptr;
  TSP_TRY(copy_stream(&s2));
  cudaEvent_t ready = nullptr, copied = nullptr;
  cudaError_t e = cudaEventCreateWithFlags(&ready, cudaEventDisableTiming);
  if (e == cudaSuccess) e = cudaEventCreateWithFlags(&copied, cudaEventDisableTiming);
  tsp_status st = TSP_OK;
  if (e != cudaSuccess) st = cuda_fail(e, "tsp_layer_fwd_host: cudaEventCreate");
  const size_t run_bytes = (size_t)p.C * p.H * 2;
  const uint16_t* src = static_cast<const uint16_t*>(out_dev_rows);
  for (int r = 0; st == TSP_OK && r < p.D; ++r) {
    st = swiglu_down_rank(p, r, g, wpack, residual32, out_dev_rows, ws, s);
    if (st != TSP_OK) break;
    // the copies of rank r start once its rows are written (a wait on an event uses
    // the record made just before it, so one event serves every rank)
    e = cudaEventRecord(ready, s);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(s2, ready, 0);
    for (int b = 0; e == cudaSuccess && b < p.B; ++b) {
      const int64_t row = ((int64_t)r * p.B + b) * p.T;  // first sharded row of (r, b)
      const int64_t nat0 = (int64_t)b * p.S + (int64_t)r * p.C;
      const int64_t nat1 = (int64_t)b * p.S + (int64_t)(2 * p.D - 1 - r) * p.C;
      e = cudaMemcpyAsync(out_host + nat0 * p.H, src + row * p.H, run_bytes,
                          cudaMemcpyDeviceToHost, s2);
      if (e == cudaSuccess)
        e = cudaMemcpyAsync(out_host + nat1 * p.H, src + (row + p.C) * p.H, run_bytes,
                            cudaMemcpyDeviceToHost, s2);
    }
    if (e != cudaSuccess) st = cuda_fail(e, "tsp_layer_fwd_host: copy out");
  }
  // the caller's stream goes on only after every copy enqueued above
  if (copied) {
    e = cudaEventRecord(copied, s2);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(s, copied, 0);
    if (e != cudaSuccess && st == TSP_OK) st = cuda_fail(e, "tsp_layer_fwd_host: join");
  }
  if (ready) cudaEventDestroy(ready);
  if (copied) cudaEventDestroy(copied);
  return st;
}

// The way in of tsp_layer_fwd_host, overlapped: rank by rank, the copy engine moves
// the rank's rows of x (two runs of C natural rows per sequence) from pinned host
// memory to their sharded rows in xs on the copy stream, and `s` runs the Q/K/V
// product of shards 0 .. n - 1 on those rows (into q, kn, vn with row stride ld) while
// the next ranks' rows arrive.
tsp_status shard_in_with_qkv(const Plan& p, const tsp_bf16* x_host, void* xs, const void* wpack,
                             int n, void* q, void* kn, void* vn, int64_t ld, void* ws,
                             cudaStream_t s) {
  cudaStream_t s2 = nullptr;
  TSP_TRY(copy_stream(&s2));
  cudaEvent_t start = nullptr, ready = nullptr;
  cudaError_t e = cudaEventCreateWithFlags(&start, cudaEventDisableTiming);
  if (e == cudaSuccess) e = cudaEventCreateWithFlags(&ready, cudaEventDisableTiming);
  // the copies overwrite xs only after the work enqueued on `s` before this call
  if (e == cudaSuccess) e = cudaEventRecord(start, s);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(s2, start, 0);
  tsp_status st = e == cudaSuccess ? TSP_OK : cuda_fail(e, "tsp_layer_fwd_host: copy-in events");
  const size_t run_bytes = (size_t)p.C * p.H * 2;
  uint16_t* dst = static_cast<uint16_t*>(xs);
  for (int r = 0; st == TSP_OK && r < p.D; ++r) {
    for (int b = 0; e == cudaSuccess && b < p.B; ++b) {
      const int64_t row = ((int64_t)r * p.B + b) * p.T;  // first sharded row of (r, b)
      const int64_t nat0 = (int64_t)b * p.S + (int64_t)r * p.C;
      const int64_t nat1 = (int64_t)b * p.S + (int64_t)(2 * p.D - 1 - r) * p.C;
      e = cudaMemcpyAsync(dst + row * p.H, x_host + nat0 * p.H, run_bytes, cudaMemcpyHostToDevice,
                          s2);
      if (e == cudaSuccess)
        e = cudaMemcpyAsync(dst + (row + p.C) * p.H, x_host + nat1 * p.H, run_bytes,
                            cudaMemcpyHostToDevice, s2);
    }
    if (e == cudaSuccess) e = cudaEventRecord(ready, s2);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(s, ready, 0);
    if (e != cudaSuccess) {
      st = cuda_fail(e, "tsp_layer_fwd_host: copy in");
      break;
    }
    st = qkv_rank(p, r, n, xs, wpack, q, kn, vn, ld, ws, s);
  }
  if (st != TSP_OK && ready) {
    // on a failure part way, `stream` still waits for the copies already enqueued, so
    // none of them writes xs after the call has returned its error
    if (cudaEventRecord(ready, s2) == cudaSuccess) cudaStreamWaitEvent(s, ready, 0);
  }
  if (start) cudaEventDestroy(start);
  if (ready) cudaEventDestroy(ready);
  return st;
}

// Device-side alias of a page-locked (pinned or registered) host buffer, or NULL if
// the runtime does not map it (pageable memory).
const void* mapped_host_alias(const void* host) {
  cudaPointerAttributes attr;
  cudaError_t e = cudaPointerGetAttributes(&attr, host);
  if (e != cudaSuccess) {
    cudaGetLastError();  // clear the sticky-free error of an unknown pointer
    return nullptr;
  }
  if (attr.type != cudaMemoryTypeHost || attr.devicePointer == nullptr) return nullptr;
  if (reinterpret_cast<uintptr_t>(attr.devicePointer) & 15u) return nullptr;
  return attr.devicePointer;
}

}  // namespace tsp

using namespace tsp;

#define TSP_GUARD_BEGIN try {
#define TSP_GUARD_END                                                   \
  }                                                                     \
  catch (const std::bad_alloc&) {                                       \
    return fail(TSP_ERR_INVALID_ARG, "host allocation failed");         \
  }                                                                     \
  catch (...) {                                                         \
    return fail(TSP_ERR_INVALID_ARG, "unexpected host exception");      \
  }

extern "C" {

tsp_status tsp_plan(int D, int64_t S, int hidden, int heads, int ffn, tsp_plan_t* out) {
  return tsp_plan_batched(D, S, 1, hidden, heads, ffn, out);
}

tsp_status tsp_plan_batched(int D, int64_t S, int batch, int hidden, int heads, int ffn,
                            tsp_plan_t* out) {
  TSP_GUARD_BEGIN
  if (!out) return fail(TSP_ERR_INVALID_ARG, "tsp_plan: null output");
  *out = nullptr;
  if (D < 1 || D > 64) return fail(TSP_ERR_UNSUPPORTED, "tsp_plan: D must be in [1, 64]");
  if (S < 2LL * D || S > (1LL << 26) || S % (2LL * D))
    return fail(TSP_ERR_UNSUPPORTED, "tsp_plan: S must be a multiple of 2D in [2D, 2^26]");
  if (batch < 1 || (int64_t)batch * S > (1LL << 26))
    return fail(TSP_ERR_UNSUPPORTED, "tsp_plan: batch must be >= 1 with batch * S <= 2^26");
  if (batch > 1 && (S / D) % 128)
    return fail(TSP_ERR_UNSUPPORTED,
                "tsp_plan: a micro-batch of several sequences needs S/D % 128 == 0");
  if (heads < 1 || hidden < 1 || hidden % heads)
    return fail(TSP_ERR_UNSUPPORTED, "tsp_plan: hidden must be a multiple of heads");
  const int d = hidden / heads;
  if (d != 64 && d != 128) return fail(TSP_ERR_UNSUPPORTED, "tsp_plan: head_dim must be 64 or 128");
  if (heads % D) return fail(TSP_ERR_UNSUPPORTED, "tsp_plan: heads must be a multiple of D");
  if (hidden % 64 || hidden > 32768) return fail(TSP_ERR_UNSUPPORTED, "tsp_plan: hidden must be a multiple of 64, <= 32768");
  if (ffn < D || ffn % D || ffn > (1 << 20)) return fail(TSP_ERR_UNSUPPORTED, "tsp_plan: ffn must be a positive multiple of D");

  Plan p{};
  p.D = D;
  p.S = S;
  p.B = batch;
  p.N = (int64_t)batch * S;
  p.H = hidden;
  p.heads = heads;
  p.d = d;
  p.F = ffn;
  p.T = S / D;
  p.C = S / (2LL * D);
  p.Hd = hidden / D;
  p.hpr = heads / D;
  p.Fd = ffn / D;
  p.Fp = (p.Fd + 63) / 64 * 64;
  if ((long long)D * p.Fp % 128) p.Fp = (p.Fd + 127) / 128 * 128;
  p.NF = D * p.Fp;
  p.ld_stat = (p.N + 127) / 128 * 128;
  {
    // shards per attention launch: the fewest that give 512 CTAs (two 128-row query
    // tiles each; about 3.4 per SM on 152 SMs), so that short sequences do not leave
    // most SMs idle in the launch's tail; 1 for long sequences
    const int64_t ctas = (S + 255) / 256 * (int64_t)(heads / D) * batch;
    int G = D;
    for (int g = 1; g <= D; ++g)
      if (D % g == 0 && ctas * g >= 512) {
        G = g;
        break;
      }
    p.G_att = G;
  }

  const size_t H = hidden;
  p.wp_qkv = 0;
  p.wp_o = 3 * H * H;
  p.wp_w13 = p.wp_o + H * H;
  p.wp_w2 = p.wp_w13 + 2 * (size_t)p.NF * H;
  p.wp_elems = p.wp_w2 + H * (size_t)p.NF;

  const size_t Sz = (size_t)p.N;  // rows of the activation buffers
  size_t off = 0;
  auto take = [&](size_t bytes) {
    size_t o = off;
    off = align256(off + bytes);
    return o;
  };
  p.ws.status = take(256);
  p.ws.qkv = take(Sz * (size_t)(p.G_att > 3 ? p.G_att : 3) * p.Hd * 2);
  p.ws.kn = take(Sz * (size_t)p.G_att * p.Hd * 2);
  p.ws.vn = take(Sz * (size_t)p.G_att * p.Hd * 2);
  p.ws.o = take(Sz * H * 2);
  p.ws.h = take(Sz * H * 2);
  p.ws.h32 = take(Sz * H * 4);
  p.ws.g = take(Sz * p.NF * 2);
  p.ws.stage_in = take(Sz * H * 2);
  p.ws.stage_out = take(Sz * H * 2);
  p.ws.total = off;
  p.ws.a13 = take(Sz * 2 * p.NF * 2);
  p.ws.dh32 = take(Sz * H * 4);
  p.ws.dh = take(Sz * H * 2);
  p.ws.dob = take(Sz * H * 2);
  p.ws.lse = take((size_t)heads * p.ld_stat * 4);
  p.ws.delta = take((size_t)heads * p.ld_stat * 4);
  p.ws.qa = take(Sz * H * 2);
  p.ws.ka = take(Sz * H * 2);
  p.ws.va = take(Sz * H * 2);
  p.ws.dqkv = take(Sz * 3 * H * 2);
  p.ws.total_bwd = off;

  tsp_plan_s* obj = new tsp_plan_s;
  obj->p = p;
  *out = obj;
  return TSP_OK;
  TSP_GUARD_END
}

void tsp_plan_destroy(tsp_plan_t plan) { delete plan; }

tsp_status tsp_get_plan_info(tsp_plan_t plan, tsp_plan_info* info) {
  TSP_TRY(tsp_check_plan(plan));
  if (!info) return fail(TSP_ERR_INVALID_ARG, "tsp_get_plan_info: null info");
  const Plan& p = plan->p;
  info->D = p.D;
  info->S = p.S;
  info->batch = p.B;
  info->tokens = p.N;
  info->attention_group = p.G_att;
  info->hidden = p.H;
  info->heads = p.heads;
  info->head_dim = p.d;
  info->ffn = p.F;
  info->T = p.T;
  info->C = p.C;
  info->shard_hidden = p.Hd;
  info->shard_ffn = p.Fd;
  info->shard_ffn_padded = p.Fp;
  info->ffn_padded = p.NF;
  info->wpack_qkv = p.wp_qkv;
  info->wpack_o = p.wp_o;
  info->wpack_w13 = p.wp_w13;
  info->wpack_w2 = p.wp_w2;
  info->wpack_elems = p.wp_elems;
  info->workspace_bytes = p.ws.total;
  info->bwd_workspace_bytes = p.ws.total_bwd;
  info->stat_stride = p.ld_stat;
  return TSP_OK;
}

size_t tsp_workspace_bytes(tsp_plan_t plan) { return plan ? plan->p.ws.total : 0; }

size_t tsp_packed_weight_bytes(tsp_plan_t plan) { return plan ? plan->p.wp_elems * 2 : 0; }

tsp_status tsp_workspace_init(tsp_plan_t plan, void* ws, void* stream) {
  TSP_TRY(tsp_check_plan(plan));
  TSP_TRY(check_ws(ws, "tsp_workspace_init"));
  cudaError_t e = cudaMemsetAsync(ws, 0, 256, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? TSP_OK : cuda_fail(e, "tsp_workspace_init");
}

tsp_status tsp_pack_weights(tsp_plan_t plan, const tsp_bf16* Wq, const tsp_bf16* Wk,
                            const tsp_bf16* Wv, const tsp_bf16* Wo, const tsp_bf16* W1,
                            const tsp_bf16* W3, const tsp_bf16* W2, tsp_bf16* wpack,
                            void* stream) {
  TSP_TRY(tsp_check_plan(plan));
  TSP_TRY(check_ptrs({Wq, Wk, Wv, Wo, W1, W3, W2, wpack}, "tsp_pack_weights"));
  return launch_pack_weights(plan->p, Wq, Wk, Wv, Wo, W1, W3, W2, wpack,
                             static_cast<cudaStream_t>(stream));
}

tsp_status tsp_shard_index(tsp_plan_t plan, int32_t* fwd, int32_t* inv, void* stream) {
  TSP_TRY(tsp_check_plan(plan));
  if (!fwd && !inv) return TSP_OK;
  return launch_zigzag_index(plan->p, fwd, inv, static_cast<cudaStream_t>(stream));
}

tsp_status tsp_shard(tsp_plan_t plan, const tsp_bf16* x, tsp_bf16* xs, void* stream) {
  TSP_TRY(tsp_check_plan(plan));
  TSP_TRY(check_ptrs({x, xs}, "tsp_shard"));
  if (x == xs) return fail(TSP_ERR_INVALID_ARG, "tsp_shard: buffers overlap");
  return launch_zigzag_rows(plan->p, x, xs, plan->p.H, true, static_cast<cudaStream_t>(stream));
}

tsp_status tsp_unshard(tsp_plan_t plan, const tsp_bf16* xs, tsp_bf16* x, void* stream) {
  TSP_TRY(tsp_check_plan(plan));
  TSP_TRY(check_ptrs({x, xs}, "tsp_unshard"));
  if (x == xs) return fail(TSP_ERR_INVALID_ARG, "tsp_unshard: buffers overlap");
  return launch_zigzag_rows(plan->p, xs, x, plan->p.H, false, static_cast<cudaStream_t>(stream));
}

tsp_status tsp_attention_fwd(tsp_plan_t plan, const tsp_bf16* xs, const tsp_bf16* wpack,
                             tsp_bf16* attn, void* ws, void* stream) {
  TSP_TRY(tsp_check_plan(plan));
  TSP_TRY(check_ptrs({xs, wpack, attn}, "tsp_attention_fwd"));
  TSP_TRY(check_ws(ws, "tsp_attention_fwd"));
  if (attn == xs) return fail(TSP_ERR_INVALID_ARG, "tsp_attention_fwd: attn aliases xs");
  return attention_block(plan->p, xs, wpack, nullptr, attn, nullptr, ws,
                         static_cast<cudaStream_t>(stream));
}

tsp_status tsp_mlp_fwd(tsp_plan_t plan, const tsp_bf16* hs, const tsp_bf16* wpack, tsp_bf16* mlp,
                       void* ws, void* stream) {
  TSP_TRY(tsp_check_plan(plan));
  TSP_TRY(check_ptrs({hs, wpack, mlp}, "tsp_mlp_fwd"));
  TSP_TRY(check_ws(ws, "tsp_mlp_fwd"));
  if (mlp == hs) return fail(TSP_ERR_INVALID_ARG, "tsp_mlp_fwd: mlp aliases hs");
  return mlp_block(plan->p, hs, wpack, nullptr, 0, mlp, ws, static_cast<cudaStream_t>(stream));
}

tsp_status tsp_layer_fwd(tsp_plan_t plan, const tsp_bf16* xs, const tsp_bf16* wpack,
                         tsp_bf16* out, void* ws, void* stream) {
  TSP_TRY(tsp_check_plan(plan));
  TSP_TRY(check_ptrs({xs, wpack, out}, "tsp_layer_fwd"));
  TSP_TRY(check_ws(ws, "tsp_layer_fwd"));
  if (out == xs) return fail(TSP_ERR_INVALID_ARG, "tsp_layer_fwd: out aliases xs");
  const Plan& p = plan->p;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  void* h = at<void>(ws, p.ws.h);
  void* h32 = at<void>(ws, p.ws.h32);
  // h = x + Attn(x), kept in bf16 (the MLP's input) and in fp32 (its residual), so
  // that out = h + MLP(h) is rounded to bf16 once
  TSP_TRY(attention_block(p, xs, wpack, xs, h, h32, ws, s));
  return mlp_block(p, h, wpack, h32, 1, out, ws, s);
}

tsp_status tsp_layer_fwd_host(tsp_plan_t plan, const tsp_bf16* x_host, const tsp_bf16* wpack,
                              tsp_bf16* out_host, void* ws, void* stream) {
  TSP_TRY(tsp_check_plan(plan));
  if (!x_host || !out_host) return fail(TSP_ERR_INVALID_ARG, "tsp_layer_fwd_host: null host buffer");
  TSP_TRY(check_ptrs({wpack}, "tsp_layer_fwd_host"));
  TSP_TRY(check_ws(ws, "tsp_layer_fwd_host"));
  const Plan& p = plan->p;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const size_t bytes = (size_t)p.N * p.H * 2;
  void* a = at<void>(ws, p.ws.stage_in);
  void* b = at<void>(ws, p.ws.stage_out);
  // Page-locked host memory (mapped into the device address space) moves rank by rank
  // through the copy engine, overlapped with the products, when every rank's rows are
  // whole 128-row tiles; otherwise the zigzag kernels read and write it directly (the
  // copy and the permutation in one pass over the host link). Other host memory goes
  // through staging copies.
  const void* x_dev = mapped_host_alias(x_host);
  void* out_dev = const_cast<void*>(mapped_host_alias(out_host));
  // rank-by-rank overlap needs whole 128-row tiles per rank (then the bits are those of
  // the products over all rows)
  const bool by_rank = p.T % 128 == 0;
  void* o = at<void>(ws, p.ws.o);
  void* h = at<void>(ws, p.ws.h);
  float* h32 = at<float>(ws, p.ws.h32);
  bool projected = false;
  // Q/K/V of every shard fit in buffers that are idle until the O projection (G and
  // the fp32 h) when the padded ffn is at least twice the hidden width
  const bool all_shards = x_dev && by_rank && (int64_t)p.NF >= 2LL * p.H;
  if (all_shards) {
    // b = shard(x) by the copy engine, rank by rank, under the Q/K/V products of every
    // shard; then the attention of every group from those buffers
    uint16_t* qa = at<uint16_t>(ws, p.ws.g);
    uint16_t* ka = qa + (size_t)p.N * p.H;
    uint16_t* va = at<uint16_t>(ws, p.ws.h32);
    TSP_TRY(shard_in_with_qkv(p, x_host, b, wpack, p.D, qa, ka, va, p.H, ws, s));
    for (int k = 0; k < p.D; k += p.G_att)
      TSP_TRY(causal_attention_shards(p, k, p.G_att, qa + (size_t)k * p.Hd, p.H,
                                      ka + (size_t)k * p.Hd, va + (size_t)k * p.Hd, p.H, o,
                                      ws, s, nullptr));
  } else if (x_dev && by_rank) {
    // b = shard(x) by the copy engine, rank by rank, under the first group's Q/K/V
    const int64_t ld = (int64_t)p.G_att * p.Hd;
    TSP_TRY(shard_in_with_qkv(p, x_host, b, wpack, p.G_att, at<void>(ws, p.ws.qkv),
                              at<void>(ws, p.ws.kn), at<void>(ws, p.ws.vn), ld, ws, s));
    projected = true;
  } else if (x_dev) {
    TSP_TRY(launch_zigzag_rows(p, x_dev, b, p.H, true, s));  // b = shard(x), read from host
  } else {
    cudaError_t e = cudaMemcpyAsync(a, x_host, bytes, cudaMemcpyHostToDevice, s);
    if (e != cudaSuccess) return cuda_fail(e, "tsp_layer_fwd_host: copy in");
    TSP_TRY(launch_zigzag_rows(p, a, b, p.H, true, s));  // b = shard(x)
  }
  // h = x + Attn(x), in bf16 and fp32 (the steps of tsp_layer_fwd)
  if (!all_shards) TSP_TRY(attention_shards(p, b, wpack, o, ws, s, nullptr, projected));
  TSP_TRY(o_projection(p, o, wpack, b, h, h32, ws, s));
  if (out_dev && by_rank) {
    // the MLP, whose output rows go back to the pinned host buffer rank by rank while
    // the next rank's down projection runs
    return mlp_block_to_host(p, h, wpack, h32, a, out_host, ws, s);
  }
  TSP_TRY(mlp_block(p, h, wpack, h32, 1, a, ws, s));  // a = layer(b)
  if (out_dev) {
    TSP_TRY(launch_zigzag_rows(p, a, out_dev, p.H, false, s));  // unshard into host memory
  } else {
    TSP_TRY(launch_zigzag_rows(p, a, b, p.H, false, s));  // b = unshard(a)
    cudaError_t e = cudaMemcpyAsync(out_host, b, bytes, cudaMemcpyDeviceToHost, s);
    if (e != cudaSuccess) return cuda_fail(e, "tsp_layer_fwd_host: copy out");
  }
  return TSP_OK;
}

tsp_status tsp_qkv_projection(tsp_plan_t plan, int shard, const tsp_bf16* xs,
                              const tsp_bf16* wpack, tsp_bf16* qkv, void* ws, void* stream) {
  TSP_TRY(tsp_check_plan(plan));
  TSP_TRY(check_ptrs({xs, wpack, qkv}, "tsp_qkv_projection"));
  TSP_TRY(check_ws(ws, "tsp_qkv_projection"));
  if (shard < 0 || shard >= plan->p.D) return fail(TSP_ERR_INVALID_ARG, "tsp_qkv_projection: shard out of range");
  return qkv_projection(plan->p, shard, xs, wpack, qkv, ws, static_cast<cudaStream_t>(stream));
}

tsp_status tsp_qkv_projection_gathered(tsp_plan_t plan, int shard, const tsp_bf16* xs,
                                       const tsp_bf16* wpack, tsp_bf16* q, tsp_bf16* kn,
                                       tsp_bf16* vn, void* ws, void* stream) {
  TSP_TRY(tsp_check_plan(plan));
  TSP_TRY(check_ptrs({xs, wpack, q, kn, vn}, "tsp_qkv_projection_gathered"));
  TSP_TRY(check_ws(ws, "tsp_qkv_projection_gathered"));
  if (shard < 0 || shard >= plan->p.D)
    return fail(TSP_ERR_INVALID_ARG, "tsp_qkv_projection_gathered: shard out of range");
  return qkv_projection_gathered(plan->p, shard, xs, wpack, q, kn, vn, ws,
                                 static_cast<cudaStream_t>(stream));
}

tsp_status tsp_causal_attention_q(tsp_plan_t plan, int shard, const tsp_bf16* q,
                                  const tsp_bf16* kn, const tsp_bf16* vn, tsp_bf16* o, void* ws,
                                  void* stream) {
  TSP_TRY(tsp_check_plan(plan));
  TSP_TRY(check_ptrs({q, kn, vn, o}, "tsp_causal_attention_q"));
  TSP_TRY(check_ws(ws, "tsp_causal_attention_q"));
  if (shard < 0 || shard >= plan->p.D)
    return fail(TSP_ERR_INVALID_ARG, "tsp_causal_attention_q: shard out of range");
  return causal_attention(plan->p, shard, q, plan->p.Hd, kn, vn, o, ws,
                          static_cast<cudaStream_t>(stream));
}

tsp_status tsp_kv_allgather(tsp_plan_t plan, const tsp_bf16* qkv, tsp_bf16* kn, tsp_bf16* vn,
                            void* stream) {
  TSP_TRY(tsp_check_plan(plan));
  TSP_TRY(check_ptrs({qkv, kn, vn}, "tsp_kv_allgather"));
  return launch_kv_gather(plan->p, qkv, kn, vn, static_cast<cudaStream_t>(stream));
}

tsp_status tsp_causal_attention(tsp_plan_t plan, int shard, const tsp_bf16* qkv,
                                const tsp_bf16* kn, const tsp_bf16* vn, tsp_bf16* o, void* ws,
                                void* stream) {
  TSP_TRY(tsp_check_plan(plan));
  TSP_TRY(check_ptrs({qkv, kn, vn, o}, "tsp_causal_attention"));
  TSP_TRY(check_ws(ws, "tsp_causal_attention"));
  if (shard < 0 || shard >= plan->p.D) return fail(TSP_ERR_INVALID_ARG, "tsp_causal_attention: shard out of range");
  return causal_attention(plan->p, shard, qkv, 3LL * plan->p.Hd, kn, vn, o, ws,
                          static_cast<cudaStream_t>(stream));
}

tsp_status tsp_o_projection(tsp_plan_t plan, const tsp_bf16* o, const tsp_bf16* wpack,
                            const tsp_bf16* residual, tsp_bf16* out, float* out32, void* ws,
                            void* stream) {
  TSP_TRY(tsp_check_plan(plan));
  TSP_TRY(check_ptrs({o, wpack, out}, "tsp_o_projection"));
  TSP_TRY(check_ws(ws, "tsp_o_projection"));
  if (residual && !al16(residual)) return fail(TSP_ERR_INVALID_ARG, "tsp_o_projection: residual not 16-byte aligned");
  if (out32 && !residual) return fail(TSP_ERR_INVALID_ARG, "tsp_o_projection: out32 needs a residual");
  if (out32 && !al16(out32)) return fail(TSP_ERR_INVALID_ARG, "tsp_o_projection: out32 not 16-byte aligned");
  return o_projection(plan->p, o, wpack, residual, out, out32, ws,
                      static_cast<cudaStream_t>(stream));
}

tsp_status tsp_swiglu_gate_up(tsp_plan_t plan, const tsp_bf16* hs, const tsp_bf16* wpack,
                              tsp_bf16* g, void* ws, void* stream) {
  TSP_TRY(tsp_check_plan(plan));
  TSP_TRY(check_ptrs({hs, wpack, g}, "tsp_swiglu_gate_up"));
  TSP_TRY(check_ws(ws, "tsp_swiglu_gate_up"));
  return swiglu_gate_up(plan->p, hs, wpack, g, ws, static_cast<cudaStream_t>(stream));
}

tsp_status tsp_swiglu_down(tsp_plan_t plan, const tsp_bf16* g, const tsp_bf16* wpack,
                           const tsp_bf16* residual, const float* residual32, tsp_bf16* out,
                           void* ws, void* stream) {
  TSP_TRY(tsp_check_plan(plan));
  TSP_TRY(check_ptrs({g, wpack, out}, "tsp_swiglu_down"));
  TSP_TRY(check_ws(ws, "tsp_swiglu_down"));
  if (residual && !al16(residual)) return fail(TSP_ERR_INVALID_ARG, "tsp_swiglu_down: residual not 16-byte aligned");
  if (residual32 && !al16(residual32)) return fail(TSP_ERR_INVALID_ARG, "tsp_swiglu_down: residual32 not 16-byte aligned");
  const void* r = residual32 ? static_cast<const void*>(residual32) : residual;
  return swiglu_down(plan->p, g, wpack, r, residual32 ? 1 : 0, out, ws,
                     static_cast<cudaStream_t>(stream));
}

tsp_status tsp_device_status(void* ws, void* stream) {
  TSP_TRY(check_ws(ws, "tsp_device_status"));
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  DevStatus st{};
  cudaError_t e = cudaMemcpyAsync(&st, ws, sizeof st, cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(e, "tsp_device_status");
  if (st.code == 0) return TSP_OK;
  e = cudaMemsetAsync(ws, 0, sizeof st, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(e, "tsp_device_status: clear");
  char buf[160];
  snprintf(buf, sizeof buf, "device wait gave up (site %u, block %u, thread %u)", st.site, st.block,
           st.thread);
  return fail(st.code == TSP_ERR_TIMEOUT ? TSP_ERR_TIMEOUT : TSP_ERR_CUDA, buf);
}

tsp_status tsp_wait_selftest(void* ws, uint64_t limit_ns, void* stream) {
  TSP_TRY(check_ws(ws, "tsp_wait_selftest"));
  if (limit_ns == 0 || limit_ns > 10000000000ull)
    return fail(TSP_ERR_INVALID_ARG, "tsp_wait_selftest: limit must be in (0, 10 s]");
  return launch_wait_selftest(status_of(ws), limit_ns, static_cast<cudaStream_t>(stream));
}

const char* tsp_last_error(void) { return g_last_error.c_str(); }

}  // extern "C"
