// zigzag.cu - the data-movement kernels of the TSP layer on sm_103a.
//
// Zigzag partitioning ("Folding Tensor and Sequence Parallelism for
// Memory-Efficient Transformer Training & Inference", section 2, attention
// layers): the S tokens are cut into 2D chunks of C = S/(2D); rank r owns chunk r
// (local rows 0..C-1) and chunk 2D-1-r (local rows C..2C-1), which gives every rank
// the same causal attention work. Token t therefore sits at row
//     zig(t) = r*T + l   (T = S/D)
// of the rank-major [D][T][...] layout. A micro-batch of B sequences (section 4,
// scalability: larger micro-batches) keeps every rank's rows of all sequences
// together: token t of sequence b (natural row b*S + t) sits at row
//     (r*B + b)*T + l   of the rank-major [D][B][T][...] layout.
//
// K/V all-gather along the sequence (same section): every rank's K and V columns
// of the current attention shard are gathered into one natural-order buffer.
//
// All of these are pure copies bound by HBM bandwidth: 16-byte vector loads and
// stores, one CTA per row (or a warp per row), grid sized in multiples of the SM
// count, several 16-byte loads in flight per thread.
#include "tsp_device.cuh"
#include "tsp_internal.h"

namespace tsp {
namespace {

struct Zig {
  long long C, T;
  int D, B;
  // sharded row of natural row n = b*S + t (S = D*T)
  __device__ __forceinline__ long long row_of(long long n) const {
    const long long b = n / (T * D);
    const long long t = n - b * (T * D);
    const long long c = t / C;
    const long long o = t - c * C;
    const long long r = c < D ? c : 2 * D - 1 - c;
    return (r * B + b) * T + (c < D ? o : C + o);
  }
};

// S here (and in the kernels below) is the number of natural rows: B * tokens.
__global__ void zigzag_index_kernel(int32_t* __restrict__ fwd, int32_t* __restrict__ inv,
                                    long long S, Zig z) {
  for (long long t = blockIdx.x * (long long)blockDim.x + threadIdx.x; t < S;
       t += (long long)gridDim.x * blockDim.x) {
    const long long row = z.row_of(t);
    if (fwd) fwd[t] = (int32_t)row;
    if (inv) inv[row] = (int32_t)t;
  }
}

// Copy whole rows of `vpr` 16-byte vectors: natural row t <-> sharded row zig(t).
template <int UNROLL>
__global__ void __launch_bounds__(256) zigzag_rows_kernel(const uint4* __restrict__ src,
                                                          uint4* __restrict__ dst, long long S,
                                                          int vpr, int to_sharded, Zig z) {
  for (long long t = blockIdx.x; t < S; t += gridDim.x) {
    const long long zr = z.row_of(t);
    const long long s_row = to_sharded ? t : zr;
    const long long d_row = to_sharded ? zr : t;
    const uint4* s = src + s_row * vpr;
    uint4* d = dst + d_row * vpr;
    for (int v0 = threadIdx.x; v0 < vpr; v0 += 256 * UNROLL) {
      uint4 buf[UNROLL];
#pragma unroll
      for (int u = 0; u < UNROLL; ++u) {
        const int v = v0 + u * 256;
        if (v < vpr) buf[u] = __ldcs(s + v);
      }
#pragma unroll
      for (int u = 0; u < UNROLL; ++u) {
        const int v = v0 + u * 256;
        if (v < vpr) __stcs(d + v, buf[u]);
      }
    }
  }
}

// kn[t] = qkv[zig(t)][Hd : 2Hd], vn[t] = qkv[zig(t)][2Hd : 3Hd]; one warp per token.
// Source rows hold K at vector column k_off and V at v_off, src_vec vectors apart
// (Q|K|V rows of a shard's projection: 3 vec_hd, vec_hd, 2 vec_hd; the K|V rows a
// rank contributes to the all-gather: 2 vec_hd, 0, vec_hd).
__global__ void __launch_bounds__(256) kv_gather_kernel(const uint4* __restrict__ qkv,
                                                        uint4* __restrict__ kn,
                                                        uint4* __restrict__ vn, long long S,
                                                        int vec_hd, Zig z, int src_vec,
                                                        int k_off, int v_off) {
  const int lane = threadIdx.x & 31;
  const long long warps = (long long)gridDim.x * (blockDim.x >> 5);
  for (long long t = blockIdx.x * (long long)(blockDim.x >> 5) + (threadIdx.x >> 5); t < S;
       t += warps) {
    const uint4* src = qkv + z.row_of(t) * (long long)src_vec;
    uint4* dk = kn + t * vec_hd;
    uint4* dv = vn + t * vec_hd;
    for (int v = lane; v < vec_hd; v += 64) {
      const bool second = v + 32 < vec_hd;
      const uint4 k0 = __ldcs(src + k_off + v);
      const uint4 v0 = __ldcs(src + v_off + v);
      uint4 k1, v1;
      if (second) {
        k1 = __ldcs(src + k_off + v + 32);
        v1 = __ldcs(src + v_off + v + 32);
      }
      dk[v] = k0;
      dv[v] = v0;
      if (second) {
        dk[v + 32] = k1;
        dv[v + 32] = v1;
      }
    }
  }
}

// ---------------------------------------------------------------- packing
// One-time layout of the weights (element-wise; not on the hot path).
struct PackArgs {
  const uint16_t *Wq, *Wk, *Wv, *Wo, *W1, *W3, *W2;
  uint16_t* out;
  int H, D, Hd, Fd, Fp, NF;
  long long n_qkv, n_o, n_w13, n_w2;  // element counts of the sections
};

__global__ void pack_weights_kernel(PackArgs a) {
  const long long total = a.n_qkv + a.n_o + a.n_w13 + a.n_w2;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total;
       i += (long long)gridDim.x * blockDim.x) {
    long long e = i;
    uint16_t v = 0;
    if (e < a.n_qkv) {
      // [D][3Hd][H]: shard k, local row j -> Wq/Wk/Wv row k*Hd + j % Hd
      const long long row = e / a.H, col = e - row * a.H;
      const long long k = row / (3LL * a.Hd), j = row - k * 3LL * a.Hd;
      const int part = (int)(j / a.Hd);
      const long long src_row = k * a.Hd + (j - (long long)part * a.Hd);
      const uint16_t* W = part == 0 ? a.Wq : (part == 1 ? a.Wk : a.Wv);
      v = W[src_row * a.H + col];
    } else if ((e -= a.n_qkv) < a.n_o) {
      v = a.Wo[e];  // [H][H] natural layout; shard k = columns [k Hd, (k+1) Hd)
    } else if ((e -= a.n_o) < a.n_w13) {
      // [NF/128][256][H]: rows 0..127 of group g are W1 rows of padded ffn index
      // 128g + j, rows 128..255 the W3 rows of the same indices
      const long long row = e / a.H, col = e - row * a.H;
      const long long g = row / 256, j = row - g * 256;
      const long long fp = g * 128 + (j & 127);
      const long long k = fp / a.Fp, loc = fp - k * a.Fp;
      if (loc < a.Fd) {
        const uint16_t* W = j < 128 ? a.W1 : a.W3;
        v = W[(k * a.Fd + loc) * a.H + col];
      }
    } else {
      e -= a.n_w13;
      // [H][NF]: column fp of shard k = fp / Fp -> W2 column k*Fd + fp % Fp (or zero)
      const long long row = e / a.NF, fp = e - row * a.NF;
      const long long k = fp / a.Fp, loc = fp - k * a.Fp;
      if (loc < a.Fd) v = a.W2[row * (long long)(a.D * a.Fd) + k * a.Fd + loc];
    }
    a.out[i] = v;
  }
}

// Weight gradients from the packed layout (fp32) to nn.Linear layout (fp32): each
// natural element reads its packed position (the inverse of pack_weights_kernel's
// map; padded ffn columns are dropped). Outputs that are NULL are skipped.
struct UnpackArgs {
  const float* in;
  float *dWq, *dWk, *dWv, *dWo, *dW1, *dW3, *dW2;
  int H, D, Hd, Fd, Fp, NF, F;
  long long wp_o, wp_w13, wp_w2;
};

__global__ void unpack_grads_kernel(UnpackArgs a) {
  const long long HH = (long long)a.H * a.H, FH = (long long)a.F * a.H;
  const long long total = 4 * HH + 3 * FH;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total;
       i += (long long)gridDim.x * blockDim.x) {
    long long e = i;
    if (e < 3 * HH) {  // dWq, dWk, dWv: row of heads group k -> packed row k*3Hd + part*Hd + j
      const int part = (int)(e / HH);
      e -= part * HH;
      float* out = part == 0 ? a.dWq : (part == 1 ? a.dWk : a.dWv);
      if (!out) continue;
      const long long row = e / a.H, col = e - row * a.H;
      const long long k = row / a.Hd, j = row - k * a.Hd;
      out[e] = a.in[((k * 3 + part) * a.Hd + j) * a.H + col];
    } else if ((e -= 3 * HH) < HH) {
      if (a.dWo) a.dWo[e] = a.in[a.wp_o + e];
    } else if ((e -= HH) < 2 * FH) {  // dW1, dW3: ffn row f -> padded index fp -> group row
      const int part = (int)(e / FH);
      e -= part * FH;
      float* out = part == 0 ? a.dW1 : a.dW3;
      if (!out) continue;
      const long long f = e / a.H, col = e - f * a.H;
      const long long k = f / a.Fd, fp = k * a.Fp + (f - k * a.Fd);
      const long long prow = (fp / 128) * 256 + part * 128 + (fp & 127);
      out[e] = a.in[a.wp_w13 + prow * a.H + col];
    } else {
      e -= 2 * FH;  // dW2 [H][F]: column f -> packed column fp
      if (!a.dW2) continue;
      const long long row = e / a.F, f = e - row * a.F;
      const long long k = f / a.Fd, fp = k * a.Fp + (f - k * a.Fd);
      a.dW2[e] = a.in[a.wp_w2 + row * a.NF + fp];
    }
  }
}

// One thread waits on a barrier that nothing arrives at, with a time bound.
__global__ void wait_selftest_kernel(DevStatus* st, unsigned long long limit_ns) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    WaitBound wb{st, limit_ns, &abort_flag};
    mbar_wait(&bar, 0, wb, SITE_SELFTEST);
  }
}

int grid_for(long long work_items, int per_sm) {
  const long long cap = (long long)sm_count() * per_sm;
  long long g = work_items < cap ? work_items : cap;
  return (int)(g < 1 ? 1 : g);
}

tsp_status check_launch(const char* what) {
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? TSP_OK : cuda_fail(e, what);
}

}  // namespace

tsp_status launch_zigzag_index(const Plan& p, int32_t* fwd, int32_t* inv, cudaStream_t s) {
  Zig z{p.C, p.T, p.D, p.B};
  zigzag_index_kernel<<<grid_for((p.N + 255) / 256, 8), 256, 0, s>>>(fwd, inv, p.N, z);
  return check_launch("zigzag index launch");
}

tsp_status launch_zigzag_rows(const Plan& p, const void* src, void* dst, int64_t width,
                              bool to_sharded, cudaStream_t s) {
  if ((width * 2) % 16) return fail(TSP_ERR_UNSUPPORTED, "zigzag rows: row bytes % 16 != 0");
  Zig z{p.C, p.T, p.D, p.B};
  const int vpr = (int)(width * 2 / 16);
  zigzag_rows_kernel<4><<<grid_for(p.N, 8), 256, 0, s>>>(static_cast<const uint4*>(src),
                                                          static_cast<uint4*>(dst), p.N, vpr,
                                                          to_sharded ? 1 : 0, z);
  return check_launch("zigzag rows launch");
}

tsp_status launch_kv_gather(const Plan& p, const void* qkv, void* kn, void* vn, cudaStream_t s) {
  Zig z{p.C, p.T, p.D, p.B};
  const int vec_hd = p.Hd * 2 / 16;
  kv_gather_kernel<<<grid_for((p.N + 7) / 8, 16), 256, 0, s>>>(
      static_cast<const uint4*>(qkv), static_cast<uint4*>(kn), static_cast<uint4*>(vn), p.N,
      vec_hd, z, 3 * vec_hd, vec_hd, 2 * vec_hd);
  return check_launch("kv gather launch");
}

tsp_status launch_kv_gather_kv(const Plan& p, const void* kv, void* kn, void* vn, cudaStream_t s) {
  Zig z{p.C, p.T, p.D, p.B};
  const int vec_hd = p.Hd * 2 / 16;
  kv_gather_kernel<<<grid_for((p.N + 7) / 8, 16), 256, 0, s>>>(
      static_cast<const uint4*>(kv), static_cast<uint4*>(kn), static_cast<uint4*>(vn), p.N,
      vec_hd, z, 2 * vec_hd, 0, vec_hd);
  return check_launch("kv gather launch");
}

tsp_status launch_pack_weights(const Plan& p, const void* Wq, const void* Wk, const void* Wv,
                               const void* Wo, const void* W1, const void* W3, const void* W2,
                               void* wpack, cudaStream_t s) {
  PackArgs a;
  a.Wq = static_cast<const uint16_t*>(Wq);
  a.Wk = static_cast<const uint16_t*>(Wk);
  a.Wv = static_cast<const uint16_t*>(Wv);
  a.Wo = static_cast<const uint16_t*>(Wo);
  a.W1 = static_cast<const uint16_t*>(W1);
  a.W3 = static_cast<const uint16_t*>(W3);
  a.W2 = static_cast<const uint16_t*>(W2);
  a.out = static_cast<uint16_t*>(wpack);
  a.H = p.H;
  a.D = p.D;
  a.Hd = p.Hd;
  a.Fd = p.Fd;
  a.Fp = p.Fp;
  a.NF = p.NF;
  a.n_qkv = (long long)3 * p.H * p.H;
  a.n_o = (long long)p.H * p.H;
  a.n_w13 = (long long)2 * p.NF * p.H;
  a.n_w2 = (long long)p.H * p.NF;
  const long long total = a.n_qkv + a.n_o + a.n_w13 + a.n_w2;
  pack_weights_kernel<<<grid_for((total + 255) / 256, 16), 256, 0, s>>>(a);
  return check_launch("pack weights launch");
}

tsp_status launch_unpack_grads(const Plan& p, const float* dwpack, float* dWq, float* dWk,
                               float* dWv, float* dWo, float* dW1, float* dW3, float* dW2,
                               cudaStream_t s) {
  UnpackArgs a;
  a.in = dwpack;
  a.dWq = dWq;
  a.dWk = dWk;
  a.dWv = dWv;
  a.dWo = dWo;
  a.dW1 = dW1;
  a.dW3 = dW3;
  a.dW2 = dW2;
  a.H = p.H;
  a.D = p.D;
  a.Hd = p.Hd;
  a.Fd = p.Fd;
  a.Fp = p.Fp;
  a.NF = p.NF;
  a.F = p.F;
  a.wp_o = (long long)p.wp_o;
  a.wp_w13 = (long long)p.wp_w13;
  a.wp_w2 = (long long)p.wp_w2;
  const long long total = 4LL * p.H * p.H + 3LL * p.F * p.H;
  unpack_grads_kernel<<<grid_for((total + 255) / 256, 16), 256, 0, s>>>(a);
  return check_launch("unpack weight gradients launch");
}

tsp_status launch_wait_selftest(DevStatus* st, unsigned long long limit_ns, cudaStream_t s) {
  wait_selftest_kernel<<<1, 32, 0, s>>>(st, limit_ns);
  return check_launch("wait selftest launch");
}

}  // namespace tsp
