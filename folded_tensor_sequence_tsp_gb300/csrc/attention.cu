// attention.cu - causal attention of zigzag query chunks against the gathered K/V
// ("Folding Tensor and Sequence Parallelism for Memory-Efficient Transformer
// Training & Inference", section 2, attention layers: FlashAttention after the
// K/V all-gather, zigzag partitioning for causal balance).
//
// Each CTA takes 128 query rows of one head (8 warps x 16 rows). A row r of the
// rank-major [D][T] layout holds the token at global position pos(r) (zigzag map);
// it attends to K/V rows 0..pos(r) of the natural-order gathered buffers. K/V tiles
// of 64 rows are streamed through a double-buffered, XOR-swizzled shared-memory
// ring with cp.async; S = Q K^T and O += P V run on mma.sync m16n8k16 (bf16 in,
// fp32 accumulate); softmax is online in base 2 with the row max and sum kept in
// registers and reduced across the 4 lanes of a row with warp shuffles. Only K/V
// tiles that reach past the smallest query position of a warp need the mask;
// tiles past its largest position are skipped.
//
// When the zigzag chunk is a multiple of 128 tokens every 128-row tile lies inside
// one chunk; CTAs then take tiles in decreasing natural position so the longest
// (latest) tiles start first.
#include "tsp_device.cuh"
#include "tsp_internal.h"

namespace tsp {
namespace {

constexpr int ATT_BM = 128;
constexpr int ATT_BN = 64;
constexpr int ATT_WARPS = 8;
constexpr int ATT_THREADS = ATT_WARPS * 32;

struct AttParams {
  const __nv_bfloat16* qkv;
  long long ld_qkv;
  const __nv_bfloat16* kn;
  const __nv_bfloat16* vn;
  long long ld_kv;
  __nv_bfloat16* o;
  long long ld_o;
  long long o_col0;
  long long S, T, C;
  int D;
  int heads;
  int natural_order;  // 1: CTAs walk 128-token tiles in decreasing position
  float scale_log2;   // log2(e) / sqrt(d)
};

__device__ __forceinline__ long long zig_row(long long t, long long C, long long T, int D) {
  const long long c = t / C, o = t - c * C;
  return c < D ? c * T + o : (2 * D - 1 - c) * T + C + o;
}

__device__ __forceinline__ long long row_pos(long long r, long long C, long long T, int D) {
  const long long rank = r / T, l = r - rank * T;
  return l < C ? rank * C + l : (2 * D - 1 - rank) * C + (l - C);
}

// Byte offset of 16-byte chunk `ch` of row `row` in a swizzled tile of HD columns.
template <int HD>
__device__ __forceinline__ uint32_t swz(int row, int ch) {
  return (uint32_t)(row * (HD * 2) + ((ch ^ (row & 7)) << 4));
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, bool valid) {
  const int n = valid ? 16 : 0;
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(n)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                          uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ void mma16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Load `rows` rows of HD bf16 (row stride ld elements) starting at global row
// `first` (rows at or beyond `limit` are zero-filled) into a swizzled tile.
template <int HD>
__device__ __forceinline__ void load_tile(uint32_t s_base, const __nv_bfloat16* g, long long ld,
                                          long long first, long long limit, int rows) {
  constexpr int CH = HD / 8;
  for (int i = threadIdx.x; i < rows * CH; i += ATT_THREADS) {
    const int r = i / CH, ch = i - r * CH;
    const long long gr = first + r;
    const bool ok = gr < limit;
    const __nv_bfloat16* src = g + (ok ? gr : 0) * ld + ch * 8;
    cp_async16(s_base + swz<HD>(r, ch), src, ok);
  }
}

template <int HD>
__global__ void __launch_bounds__(ATT_THREADS, 1) attention_mma_kernel(const AttParams p) {
  extern __shared__ __align__(128) uint8_t smem[];
  const uint32_t sQ = smem_addr(smem);
  const uint32_t sK0 = sQ + ATT_BM * HD * 2;
  const uint32_t sV0 = sK0 + 2 * ATT_BN * HD * 2;
  constexpr uint32_t KV_BYTES = ATT_BN * HD * 2;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int head = blockIdx.x % p.heads;
  const long long tile = blockIdx.x / p.heads;
  const long long nq_tiles = (p.S + ATT_BM - 1) / ATT_BM;

  // first sharded row of this CTA's 128 query rows
  long long row0;
  if (p.natural_order) {
    const long long nat_tile = nq_tiles - 1 - tile;
    row0 = zig_row(nat_tile * ATT_BM, p.C, p.T, p.D);
  } else {
    row0 = tile * ATT_BM;
  }

  // position range of this warp's 16 rows and of the whole CTA
  __shared__ long long s_wmax[ATT_WARPS];
  long long w_min = p.S, w_max = -1;
  const int g = lane >> 2, t4 = lane & 3;
  const long long my_r0 = row0 + warp * 16 + g, my_r1 = my_r0 + 8;
  const long long pos0 = my_r0 < p.S ? row_pos(my_r0, p.C, p.T, p.D) : -1;
  const long long pos1 = my_r1 < p.S ? row_pos(my_r1, p.C, p.T, p.D) : -1;
  {
    long long mn = min(pos0 < 0 ? p.S : pos0, pos1 < 0 ? p.S : pos1);
    long long mx = max(pos0, pos1);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      mn = min(mn, __shfl_xor_sync(0xffffffffu, mn, o));
      mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    }
    w_min = mn;
    w_max = mx;
  }
  if (lane == 0) s_wmax[warp] = w_max;
  __syncthreads();
  long long cta_max = 0;
#pragma unroll
  for (int w = 0; w < ATT_WARPS; ++w) cta_max = max(cta_max, s_wmax[w]);

  const __nv_bfloat16* Kg = p.kn + head * HD;
  const __nv_bfloat16* Vg = p.vn + head * HD;
  const int nkv = (int)(cta_max / ATT_BN) + 1;

  // Q tile and the first K/V tile
  load_tile<HD>(sQ, p.qkv + head * HD, p.ld_qkv, row0, p.S, ATT_BM);
  cp_async_commit();
  load_tile<HD>(sK0, Kg, p.ld_kv, 0, p.S, ATT_BN);
  load_tile<HD>(sV0, Vg, p.ld_kv, 0, p.S, ATT_BN);
  cp_async_commit();
  cp_async_wait<1>();
  __syncthreads();

  // Q fragments of this warp's 16 rows (A operand), kept in registers
  uint32_t qf[HD / 16][4];
#pragma unroll
  for (int ks = 0; ks < HD / 16; ++ks) {
    const int r = warp * 16 + (lane & 15);
    const int ch = ks * 2 + (lane >> 4);
    ldsm_x4(sQ + swz<HD>(r, ch), qf[ks][0], qf[ks][1], qf[ks][2], qf[ks][3]);
  }

  float oacc[HD / 8][4];
#pragma unroll
  for (int i = 0; i < HD / 8; ++i) oacc[i][0] = oacc[i][1] = oacc[i][2] = oacc[i][3] = 0.f;
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;

  for (int j = 0; j < nkv; ++j) {
    if (j + 1 < nkv) {
      const uint32_t nb = (uint32_t)((j + 1) & 1) * KV_BYTES;
      load_tile<HD>(sK0 + nb, Kg, p.ld_kv, (long long)(j + 1) * ATT_BN, p.S, ATT_BN);
      load_tile<HD>(sV0 + nb, Vg, p.ld_kv, (long long)(j + 1) * ATT_BN, p.S, ATT_BN);
    }
    cp_async_commit();
    cp_async_wait<1>();
    __syncthreads();

    const long long kv0 = (long long)j * ATT_BN;
    if (kv0 <= w_max) {
      const uint32_t sK = sK0 + (uint32_t)(j & 1) * KV_BYTES;
      const uint32_t sV = sV0 + (uint32_t)(j & 1) * KV_BYTES;
      float s[ATT_BN / 8][4];
#pragma unroll
      for (int n = 0; n < ATT_BN / 8; ++n) s[n][0] = s[n][1] = s[n][2] = s[n][3] = 0.f;
#pragma unroll
      for (int ks = 0; ks < HD / 16; ++ks) {
#pragma unroll
        for (int nb = 0; nb < ATT_BN / 16; ++nb) {
          const int r = nb * 16 + (lane & 7) + ((lane >> 4) << 3);
          const int ch = ks * 2 + ((lane >> 3) & 1);
          uint32_t b0, b1, b2, b3;
          ldsm_x4(sK + swz<HD>(r, ch), b0, b1, b2, b3);
          mma16816(s[2 * nb], qf[ks], b0, b1);
          mma16816(s[2 * nb + 1], qf[ks], b2, b3);
        }
      }
      // scale into base 2 and mask keys past each row's position
      const bool need_mask = kv0 + ATT_BN - 1 > w_min;
#pragma unroll
      for (int n = 0; n < ATT_BN / 8; ++n) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          float v = s[n][e] * p.scale_log2;
          if (need_mask) {
            const long long kpos = kv0 + n * 8 + 2 * t4 + (e & 1);
            const long long qpos = (e < 2) ? pos0 : pos1;
            if (kpos > qpos) v = -INFINITY;
          }
          s[n][e] = v;
        }
      }
      float mx0 = m0, mx1 = m1;
#pragma unroll
      for (int n = 0; n < ATT_BN / 8; ++n) {
        mx0 = fmaxf(mx0, fmaxf(s[n][0], s[n][1]));
        mx1 = fmaxf(mx1, fmaxf(s[n][2], s[n][3]));
      }
#pragma unroll
      for (int o = 1; o <= 2; o <<= 1) {
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, o));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, o));
      }
      // rows with nothing visible yet keep a finite reference so exp2 gives 0
      const float ref0 = mx0 == -INFINITY ? 0.f : mx0;
      const float ref1 = mx1 == -INFINITY ? 0.f : mx1;
      const float c0 = ex2(m0 - ref0), c1 = ex2(m1 - ref1);
      m0 = mx0;
      m1 = mx1;
      float rs0 = 0.f, rs1 = 0.f;
      uint32_t pf[ATT_BN / 16][4];
#pragma unroll
      for (int n = 0; n < ATT_BN / 8; ++n) {
        const float p0 = ex2(s[n][0] - ref0), p1 = ex2(s[n][1] - ref0);
        const float p2 = ex2(s[n][2] - ref1), p3 = ex2(s[n][3] - ref1);
        rs0 += p0 + p1;
        rs1 += p2 + p3;
        pf[n >> 1][(n & 1) * 2 + 0] = pack_bf16x2(p0, p1);
        pf[n >> 1][(n & 1) * 2 + 1] = pack_bf16x2(p2, p3);
      }
      l0 = l0 * c0 + rs0;
      l1 = l1 * c1 + rs1;
#pragma unroll
      for (int i = 0; i < HD / 8; ++i) {
        oacc[i][0] *= c0;
        oacc[i][1] *= c0;
        oacc[i][2] *= c1;
        oacc[i][3] *= c1;
      }
      // O += P V; P fragments reuse the S accumulator layout as the A operand
#pragma unroll
      for (int ks = 0; ks < ATT_BN / 16; ++ks) {
        const uint32_t a[4] = {pf[ks][0], pf[ks][1], pf[ks][2], pf[ks][3]};
#pragma unroll
        for (int db = 0; db < HD / 16; ++db) {
          const int r = ks * 16 + (lane & 7) + (((lane >> 3) & 1) << 3);
          const int ch = db * 2 + (lane >> 4);
          uint32_t b0, b1, b2, b3;
          ldsm_x4_t(sV + swz<HD>(r, ch), b0, b1, b2, b3);
          mma16816(oacc[2 * db], a, b0, b1);
          mma16816(oacc[2 * db + 1], a, b2, b3);
        }
      }
    }
    __syncthreads();
  }

  // normalise and store O rows (bf16)
  l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
  l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
  const float inv0 = l0 > 0.f ? 1.f / l0 : 0.f;
  const float inv1 = l1 > 0.f ? 1.f / l1 : 0.f;
  __nv_bfloat16* o0 = p.o + my_r0 * p.ld_o + p.o_col0 + head * HD;
  __nv_bfloat16* o1 = p.o + my_r1 * p.ld_o + p.o_col0 + head * HD;
#pragma unroll
  for (int i = 0; i < HD / 8; ++i) {
    const int col = i * 8 + 2 * t4;
    if (my_r0 < p.S)
      *reinterpret_cast<uint32_t*>(o0 + col) = pack_bf16x2(oacc[i][0] * inv0, oacc[i][1] * inv0);
    if (my_r1 < p.S)
      *reinterpret_cast<uint32_t*>(o1 + col) = pack_bf16x2(oacc[i][2] * inv1, oacc[i][3] * inv1);
  }
}

template <int HD>
tsp_status launch_hd(const AttParams& p, cudaStream_t stream) {
  const size_t smem = (size_t)ATT_BM * HD * 2 + 4ull * ATT_BN * HD * 2;
  auto kernel = attention_mma_kernel<HD>;
  cudaError_t e =
      cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return cuda_fail(e, "attention: cudaFuncSetAttribute");
  const long long blocks = ((p.S + ATT_BM - 1) / ATT_BM) * p.heads;
  kernel<<<(unsigned)blocks, ATT_THREADS, smem, stream>>>(p);
  e = cudaGetLastError();
  return e == cudaSuccess ? TSP_OK : cuda_fail(e, "attention: launch");
}

}  // namespace

tsp_status launch_attention(const AttentionCall& c, cudaStream_t stream) {
  if (c.d != 64 && c.d != 128) return fail(TSP_ERR_UNSUPPORTED, "attention: head_dim 64 or 128");
  AttParams p;
  p.qkv = static_cast<const __nv_bfloat16*>(c.qkv);
  p.ld_qkv = c.ld_qkv;
  p.kn = static_cast<const __nv_bfloat16*>(c.kn);
  p.vn = static_cast<const __nv_bfloat16*>(c.vn);
  p.ld_kv = c.ld_kv;
  p.o = static_cast<__nv_bfloat16*>(c.o);
  p.ld_o = c.ld_o;
  p.o_col0 = c.o_col0;
  p.S = c.S;
  p.T = c.T;
  p.C = c.C;
  p.D = c.D;
  p.heads = c.heads;
  p.natural_order = (c.C % ATT_BM == 0) ? 1 : 0;
  p.scale_log2 = 1.4426950408889634f / sqrtf((float)c.d);
  return c.d == 64 ? launch_hd<64>(p, stream) : launch_hd<128>(p, stream);
}

}  // namespace tsp
