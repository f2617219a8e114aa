// noalloc.cu - tsp_mlp_fwd_noalloc: the gated MLP block without a caller workspace.
//
// Some callers cannot call cudaMalloc (or any allocating routine) at the point
// where they run the layer: code inside a custom allocator or a memory-pool
// callback, plug-ins of a host application that owns every device allocation, or
// runtimes that forbid allocation after start-up. They can still pass their inputs
// and outputs, but not the workspace tsp_mlp_fwd needs for the gated activation G.
// This entry point keeps that scratch (and the device status word of the bounded
// waits) in one file-scope device array of fixed size instead.
#include <cstdio>
#include <mutex>

#include "tsp_device.cuh"
#include "tsp_internal.h"

namespace {

// 32 MiB: the status word (first 256 bytes) and G = [tokens][ffn_padded] bf16.
constexpr size_t kNoallocScratchBytes = 32ull << 20;
constexpr size_t kNoallocStatusBytes = 256;

}  // namespace

// Every GPU that loads this library holds this array until the process exits.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocScratchBytes];

namespace {

std::mutex g_noalloc_mutex;
void* g_noalloc_addr[64] = {};  // device address of g_noalloc_scratch, per device

// Device address of the scratch array on the current device. The first call on a
// device looks it up (cudaGetSymbolAddress, with that device current); later calls
// reuse it.
tsp_status noalloc_scratch(void** out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return tsp::cuda_fail(e, "tsp_mlp_fwd_noalloc: cudaGetDevice");
  if (dev < 0 || dev >= 64) return tsp::fail(TSP_ERR_UNSUPPORTED, "tsp_mlp_fwd_noalloc: device index >= 64");
  std::lock_guard<std::mutex> lock(g_noalloc_mutex);
  if (!g_noalloc_addr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return tsp::cuda_fail(e, "tsp_mlp_fwd_noalloc: cudaGetSymbolAddress");
    g_noalloc_addr[dev] = p;
  }
  *out = g_noalloc_addr[dev];
  return TSP_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" tsp_status tsp_mlp_fwd_noalloc(tsp_plan_t plan, const tsp_bf16* hs,
                                          const tsp_bf16* wpack, tsp_bf16* mlp, void* stream) {
  tsp_plan_info info;
  tsp_status st = tsp_get_plan_info(plan, &info);
  if (st != TSP_OK) return st;
  if (!hs || !wpack || !mlp) return tsp::fail(TSP_ERR_INVALID_ARG, "tsp_mlp_fwd_noalloc: null pointer");
  if (!aligned16(hs) || !aligned16(wpack) || !aligned16(mlp))
    return tsp::fail(TSP_ERR_INVALID_ARG, "tsp_mlp_fwd_noalloc: pointer not 16-byte aligned");
  if (static_cast<const void*>(mlp) == static_cast<const void*>(hs))
    return tsp::fail(TSP_ERR_INVALID_ARG, "tsp_mlp_fwd_noalloc: mlp aliases hs");
  const size_t g_bytes = (size_t)info.tokens * (size_t)info.ffn_padded * 2;
  if (g_bytes > kNoallocScratchBytes - kNoallocStatusBytes) {
    char buf[200];
    snprintf(buf, sizeof buf,
             "tsp_mlp_fwd_noalloc: this shape needs %zu bytes of scratch (tokens x ffn_padded x 2), "
             "more than the %zu available in the static buffer; use tsp_mlp_fwd with a workspace",
             g_bytes, kNoallocScratchBytes - kNoallocStatusBytes);
    return tsp::fail(TSP_ERR_UNSUPPORTED, buf);
  }
  void* base = nullptr;
  st = noalloc_scratch(&base);
  if (st != TSP_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  tsp::DevStatus* status = static_cast<tsp::DevStatus*>(base);
  void* g = static_cast<unsigned char*>(base) + kNoallocStatusBytes;

  // The array keeps the previous call's contents: the status word must start at zero;
  // G is fully overwritten by the gate/up product.
  cudaError_t e = cudaMemsetAsync(status, 0, sizeof(tsp::DevStatus), s);
  if (e != cudaSuccess) return tsp::cuda_fail(e, "tsp_mlp_fwd_noalloc: clear status");

  const uint16_t* w = static_cast<const uint16_t*>(static_cast<const void*>(wpack));
  tsp::GemmCall up{};
  up.epi = tsp::EPI_SWIGLU;
  up.A = hs;
  up.lda = info.hidden;
  up.M = info.tokens;
  up.B = w + info.wpack_w13;
  up.ldb = info.hidden;
  up.b_rows = 2LL * info.ffn_padded;
  up.b_row0 = 0;
  up.N = 2LL * info.ffn_padded;
  up.K = info.hidden;
  up.C = g;
  up.ldc = info.ffn_padded;
  up.status = status;
  st = tsp::launch_gemm(up, s);
  if (st != TSP_OK) return st;

  tsp::GemmCall down{};
  down.epi = tsp::EPI_STORE;
  down.A = g;
  down.lda = info.ffn_padded;
  down.M = info.tokens;
  down.B = w + info.wpack_w2;
  down.ldb = info.ffn_padded;
  down.b_rows = info.hidden;
  down.b_row0 = 0;
  down.N = info.hidden;
  down.K = info.ffn_padded;
  down.C = mlp;
  down.ldc = info.hidden;
  down.ring_rows = (int64_t)info.batch * info.T;
  down.ring_kblocks = info.shard_ffn_padded / 64;
  down.status = status;
  return tsp::launch_gemm(down, s);
}
