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

// Every GPU on which this array is first used holds it until the process exits.
// CUDA loads a library's device code lazily by default (CUDA_MODULE_LOADING=LAZY):
// the driver reserves this array on a device when the first tsp_mlp_fwd_noalloc
// call there looks its address up, not when the library is loaded. With eager
// loading it is reserved on every device the process initialises.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocScratchBytes];

namespace {

typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long*);

// Unique id of the calling thread's current CUDA context (cuCtxGetId, fetched through
// the runtime's driver entry point), or 0 when it cannot be had. A context made
// after cudaDeviceReset, or another context on the same device, has another id.
unsigned long long current_context_id() {
  static CtxGetCurrentFn get_current = nullptr;
  static CtxGetIdFn get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<CtxGetCurrentFn>(p);
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<CtxGetIdFn>(p);
  });
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (!get_current || !get_id || get_current(&ctx) != CUDA_SUCCESS || !ctx ||
      get_id(ctx, &id) != CUDA_SUCCESS)
    return 0;
  return id;
}

struct ScratchAddr {
  unsigned long long ctx_id;  // context the address belongs to
  void* addr;                 // device address of g_noalloc_scratch in that context
};

std::mutex g_noalloc_mutex;
ScratchAddr g_noalloc_addr[64] = {};  // per device

// Device address of the scratch array in the current device's current context. The
// first call in a context looks it up (cudaGetSymbolAddress, with that device
// current); later calls in the same context reuse it. A new context (after
// cudaDeviceReset, or a context the caller made) is looked up again, so no call
// passes an address of a context that no longer exists.
tsp_status noalloc_scratch(void** out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return tsp::cuda_fail(e, "tsp_mlp_fwd_noalloc: cudaGetDevice");
  if (dev < 0 || dev >= 64) return tsp::fail(TSP_ERR_UNSUPPORTED, "tsp_mlp_fwd_noalloc: device index >= 64");
  const unsigned long long ctx = current_context_id();
  std::lock_guard<std::mutex> lock(g_noalloc_mutex);
  ScratchAddr& c = g_noalloc_addr[dev];
  if (!c.addr || ctx == 0 || c.ctx_id != ctx) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return tsp::cuda_fail(e, "tsp_mlp_fwd_noalloc: cudaGetSymbolAddress");
    // the runtime made its context current if there was none: key by that one
    c.ctx_id = ctx ? ctx : current_context_id();
    c.addr = p;
  }
  *out = c.addr;
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
