// gemm_tcgen05.cu - the dense bf16 contractions of the TSP layer on sm_103a:
//   * Q/K/V projection of one attention shard   (local projections of a broadcast
//     iteration, "Folding Tensor and Sequence Parallelism for Memory-Efficient
//     Transformer Training & Inference", section 2, attention layers),
//   * O projection accumulated over the shards,
//   * SwiGLU gate/up product with the gating fused into the epilogue,
//   * SwiGLU down product accumulated over the MLP shards in ring order
//     (same page, section 2, gated MLP layers: local accumulation, no all-reduce).
//
// C[M][N] = A[M][K] * B[N][K]^T, A and B bf16 K-major, fp32 accumulation in tensor
// memory. One persistent CTA per SM walks output tiles of 128 x 256:
//   warp 0      TMA producer: 64-wide K slices of A and B into a 4-stage ring of
//               128B-swizzled shared-memory buffers (mbarrier transaction counts)
//   warp 1      allocates 512 TMEM columns (two 128x256 fp32 accumulators) and one
//               lane issues tcgen05.mma (M=128, N=256, K=16) and tcgen05.commit
//   warps 2..5  epilogue: tcgen05.ld of the accumulator rows (one row per thread),
//               fused residual add or SiLU gating, bf16 rounding, global stores;
//               the second accumulator lets the epilogue of a tile overlap the
//               main loop of the next.
// Ring order: with ring_rows > 0 the K loop of a tile whose rows belong to rank
// r = ring_rank0 + m0 / ring_rows starts at K block r * ring_kblocks and wraps
// around (ring_rank0: the rank of the launch's first row), so rank r
// takes MLP shard (r + t) mod D at step t, and the partial products of the shards
// are summed in the on-chip accumulator.
#include "tsp_device.cuh"
#include "tsp_internal.h"

namespace tsp {
namespace {

constexpr int BM = 128;
constexpr int BN = 256;
constexpr int BK = 64;
constexpr int STAGES = 4;
constexpr int THREADS = 192;
constexpr uint32_t A_BYTES = BM * BK * 2;
constexpr uint32_t B_BYTES = BN * BK * 2;
constexpr uint32_t STAGE_BYTES = A_BYTES + B_BYTES;
constexpr uint32_t TMEM_COLS = 2 * BN;
constexpr size_t SMEM_BYTES = 1024 + (size_t)STAGES * STAGE_BYTES + 256;

// Epilogue variants of the kernel.
enum Kind {
  K_STORE = 0,          // C = bf16(acc)
  K_RES_BF16 = 1,       // C = bf16(acc + R), R bf16
  K_SWIGLU = 2,         // C = bf16(silu(acc_gate) * acc_up)
  K_RES_BF16_OUT32 = 3, // C = bf16(acc + R), C32 = acc + R (fp32), R bf16
  K_RES_F32 = 4,        // C = bf16(acc + R), R fp32
  K_QKV_SPLIT = 5,      // Q|K|V columns: Q to C (sharded rows), K and V to natural rows
  K_STORE_F32 = 6,      // C32 = acc (fp32): weight gradients
  K_SWIGLU_SAVE = 7,    // as K_SWIGLU, and the pre-activations (A1|A3 tiles) to C2
  K_SWIGLU_BWD = 8,     // acc = dG; with A1/A3 from C2: dA1|dA3 to C in C2's packed order
  K_RES_F32_OUT32 = 9,  // C = bf16(acc + R), C32 = acc + R (fp32), R fp32 (may be C32:
                        // each element is read, then written, by one thread)
};

struct GemmParams {
  int M, N, K;
  int b_row0;
  __nv_bfloat16* C;
  long long ldc;
  const void* R;   // residual: bf16 or fp32 depending on the variant
  long long ldr;
  float* C32;      // fp32 copy of the output (K_RES_BF16_OUT32)
  // K_QKV_SPLIT: column sections of width split_hd (Q, K, V); K and V rows go to the
  // natural token position of the sharded row (zigzag inverse with chunk zz_C, T zz_T)
  __nv_bfloat16* split_k;
  __nv_bfloat16* split_v;
  long long split_ld;
  int split_hd;
  long long zz_C, zz_T;
  int zz_D, zz_B;
  long long zz_row0;  // sharded row of the launch's first row (a launch over part of the rows)
  __nv_bfloat16* C2;  // K_SWIGLU_SAVE: pre-activations out; K_SWIGLU_BWD: pre-activations in
  long long ldc2;
  int ring_rows;
  int ring_kblocks;
  int ring_rank0;
  int group_m;  // tile order: group_m row blocks walk down each column block in turn
  int wide;     // every epilogue pointer and row stride is 32-byte aligned: 32-byte accesses
  DevStatus* status;
  unsigned long long limit_ns;
};

// Tile t of the persistent walk -> (row block, column block). Consecutive tiles
// take group_m row blocks down one column block, then the next column block, so the
// group's A rows stay in L2 while each B column block is fetched once per group
// (group_m = 1 is the plain row-major walk).
__device__ __forceinline__ void tile_coords(int tile, int numM, int numN, int group_m, int& mt,
                                            int& nt) {
  const int span = group_m * numN;
  const int g = tile / span, r = tile - g * span;
  const int m_first = g * group_m;
  const int gm = min(group_m, numM - m_first);
  mt = m_first + r % gm;
  nt = r / gm;
}

// 32-byte global accesses: eight 32-bit words per thread, one whole L2 sector per
// access, so a row segment takes half the instructions and half the L2 sector writes
// of 16-byte accesses (two of which would each write half of the same sector). Every
// address must be 32-byte aligned: the launcher enables them (GemmParams::wide) only
// when every epilogue pointer and row stride is.
__device__ __forceinline__ void st_v8(void* ptr, const uint32_t (&w)[8]) {
  asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(ptr), "r"(w[0]),
               "r"(w[1]), "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7])
               : "memory");
}
__device__ __forceinline__ void ld_nc_v8(const void* ptr, uint32_t (&w)[8]) {
  asm volatile("ld.global.nc.v8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
               : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3]), "=r"(w[4]), "=r"(w[5]),
                 "=r"(w[6]), "=r"(w[7])
               : "l"(ptr));
}
__device__ __forceinline__ void ld_cs_v8(const void* ptr, uint32_t (&w)[8]) {
  asm volatile("ld.global.cs.v8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
               : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3]), "=r"(w[4]), "=r"(w[5]),
                 "=r"(w[6]), "=r"(w[7])
               : "l"(ptr));
}

// 32 fp32 values -> 32 bf16 (RNE) at dst (64 bytes).
__device__ __forceinline__ void store_row32(__nv_bfloat16* dst, const float (&f)[32], bool wide) {
  if (wide) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      uint32_t w[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) w[e] = pack_bf16x2(f[16 * h + 2 * e], f[16 * h + 2 * e + 1]);
      st_v8(dst + 16 * h, w);
    }
    return;
  }
  uint4* d = reinterpret_cast<uint4*>(dst);
#pragma unroll
  for (int v = 0; v < 4; ++v) {
    uint4 w;
    w.x = pack_bf16x2(f[8 * v + 0], f[8 * v + 1]);
    w.y = pack_bf16x2(f[8 * v + 2], f[8 * v + 3]);
    w.z = pack_bf16x2(f[8 * v + 4], f[8 * v + 5]);
    w.w = pack_bf16x2(f[8 * v + 6], f[8 * v + 7]);
    d[v] = w;
  }
}

// 32 fp32 values at dst (128 bytes).
__device__ __forceinline__ void store_row32_f32(float* dst, const float (&f)[32], bool wide) {
  if (wide) {
#pragma unroll
    for (int h = 0; h < 4; ++h) {
      uint32_t w[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) w[e] = __float_as_uint(f[8 * h + e]);
      st_v8(dst + 8 * h, w);
    }
    return;
  }
  float4* c4 = reinterpret_cast<float4*>(dst);
#pragma unroll
  for (int w = 0; w < 8; ++w) c4[w] = make_float4(f[4 * w + 0], f[4 * w + 1], f[4 * w + 2], f[4 * w + 3]);
}

// f += 32 bf16 values at src (64 bytes, read through the non-coherent path).
__device__ __forceinline__ void add_row32_bf16(float (&f)[32], const __nv_bfloat16* src, bool wide) {
  uint32_t u[16];
  if (wide) {
    uint32_t a[8], b[8];
    ld_nc_v8(src, a);
    ld_nc_v8(src + 16, b);
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      u[e] = a[e];
      u[8 + e] = b[e];
    }
  } else {
    const uint4* r4 = reinterpret_cast<const uint4*>(src);
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      const uint4 rv = __ldg(r4 + w);
      u[4 * w + 0] = rv.x;
      u[4 * w + 1] = rv.y;
      u[4 * w + 2] = rv.z;
      u[4 * w + 3] = rv.w;
    }
  }
#pragma unroll
  for (int e = 0; e < 16; ++e) {
    f[2 * e] += bf16_lo(u[e]);
    f[2 * e + 1] += bf16_hi(u[e]);
  }
}

// f += 32 fp32 values at src (128 bytes, streamed: read once).
__device__ __forceinline__ void add_row32_f32(float (&f)[32], const float* src, bool wide) {
  if (wide) {
#pragma unroll
    for (int h = 0; h < 4; ++h) {
      uint32_t a[8];
      ld_cs_v8(src + 8 * h, a);
#pragma unroll
      for (int e = 0; e < 8; ++e) f[8 * h + e] += __uint_as_float(a[e]);
    }
    return;
  }
  const float4* r4 = reinterpret_cast<const float4*>(src);
#pragma unroll
  for (int w = 0; w < 8; ++w) {
    const float4 rv = __ldcs(r4 + w);
    f[4 * w + 0] += rv.x;
    f[4 * w + 1] += rv.y;
    f[4 * w + 2] += rv.z;
    f[4 * w + 3] += rv.w;
  }
}

// A_MN / B_MN: operand stored MN-major, i.e. as a [K][M] (or [K][N]) matrix with
// M (N) contiguous; its tiles arrive as 64-element x 64-row TMA boxes (8 KB each,
// the 64-element blocks 8 KB apart, 8-row groups 1 KB apart) and a 16-wide K step
// is 2 KB. K-major operands arrive as [rows][64] boxes and step 32 B in K.
template <int EPI, bool A_MN, bool B_MN>
__global__ void __launch_bounds__(THREADS, 1)
    gemm_bf16_tcgen05(const __grid_constant__ CUtensorMap tmA,
                      const __grid_constant__ CUtensorMap tmB, const GemmParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + STAGES * A_BYTES;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + STAGES * STAGE_BYTES);
  uint64_t* full = bars;                  // [STAGES] TMA landed
  uint64_t* empty = bars + STAGES;        // [STAGES] MMAs reading the stage are done
  uint64_t* acc_full = bars + 2 * STAGES; // [2] accumulator complete
  uint64_t* acc_empty = acc_full + 2;     // [2] epilogue drained the accumulator
  uint64_t* drain = acc_empty + 2;        // [1] every MMA issued has completed
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int numM = (p.M + BM - 1) / BM;
  const int numN = (p.N + BN - 1) / BN;
  const int numTiles = numM * numN;
  const int nkb = (p.K + BK - 1) / BK;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&acc_full[a], 1);
      mbar_init(&acc_empty[a], 4);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  WaitBound wb{p.status, p.limit_ns, abort_flag};

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------------ producer
      int stage = 0;
      uint32_t phase = 0;
      int last_parity[STAGES];
#pragma unroll
      for (int s = 0; s < STAGES; ++s) last_parity[s] = -1;
      const uint64_t keep = l2_policy_evict_last();
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < numTiles; tile += gridDim.x) {
        int mt, nt;
        tile_coords(tile, numM, numN, p.group_m, mt, nt);
        const int m0 = mt * BM, n0 = nt * BN;
        int kb = 0;
        if (p.ring_rows > 0)
          kb = (int)(((long long)(p.ring_rank0 + m0 / p.ring_rows) * p.ring_kblocks) % nkb);
        for (int i = 0; i < nkb; ++i) {
          if (!mbar_wait(&empty[stage], phase ^ 1u, wb, SITE_GEMM_PRODUCER)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&full[stage], STAGE_BYTES);
          if constexpr (A_MN) {
#pragma unroll
            for (int b = 0; b < BM / 64; ++b)
              tma_load_2d(sA + stage * A_BYTES + b * 8192, &tmA, &full[stage], m0 + 64 * b, kb * BK);
          } else {
            tma_load_2d(sA + stage * A_BYTES, &tmA, &full[stage], kb * BK, m0);
          }
          if constexpr (B_MN) {
#pragma unroll
            for (int b = 0; b < BN / 64; ++b)
              tma_load_2d_hint(sB + stage * B_BYTES + b * 8192, &tmB, &full[stage],
                               p.b_row0 + n0 + 64 * b, kb * BK, keep);
          } else {
            tma_load_2d_hint(sB + stage * B_BYTES, &tmB, &full[stage], kb * BK, p.b_row0 + n0, keep);
          }
          last_parity[stage] = (int)phase;
          if (++kb == nkb) kb = 0;
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      // Do not leave while a TMA copy into this CTA's shared memory is in flight.
      WaitBound wd{p.status, p.limit_ns, nullptr};
      for (int s = 0; s < STAGES; ++s)
        if (last_parity[s] >= 0) mbar_wait(&full[s], (uint32_t)last_parity[s], wd, SITE_DRAIN);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ------------------------------------------------------------ MMA issuer
      const uint32_t idesc = make_idesc_bf16(BM, BN, B_MN, A_MN);
      constexpr uint32_t A_STEP = A_MN ? (2048u >> 4) : (32u >> 4);  // one 16-wide K step
      constexpr uint32_t B_STEP = B_MN ? (2048u >> 4) : (32u >> 4);
      // base descriptors of stage 0, built once; stages and K steps add offsets
      const uint64_t da0 = make_sdesc_sw128(smem_addr(sA), A_MN ? 8192 : 16, 1024);
      const uint64_t db0 = make_sdesc_sw128(smem_addr(sB), B_MN ? 8192 : 16, 1024);
      const uint32_t da_lo = (uint32_t)da0, da_hi = (uint32_t)(da0 >> 32);
      const uint32_t db_lo = (uint32_t)db0, db_hi = (uint32_t)(db0 >> 32);
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < numTiles; tile += gridDim.x) {
        if (!mbar_wait(&acc_empty[acc], acc_phase ^ 1u, wb, SITE_GEMM_MMA)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN);
        for (int i = 0; i < nkb; ++i) {
          if (!mbar_wait(&full[stage], phase, wb, SITE_GEMM_MMA)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_lo = da_lo + (uint32_t)stage * (A_BYTES >> 4);
          const uint32_t b_lo = db_lo + (uint32_t)stage * (B_BYTES >> 4);
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk)
            mma_ss_w(d_tmem, a_lo + kk * A_STEP, da_hi, b_lo + kk * B_STEP, db_hi, idesc,
                     (i | kk) != 0 ? 1u : 0u);
          mma_commit(&empty[stage]);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        mma_commit(&acc_full[acc]);
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1u;
      }
      // Every MMA issued above completes before TMEM is released.
      mma_commit(drain);
      WaitBound wd{p.status, p.limit_ns, nullptr};
      mbar_wait(drain, 0, wd, SITE_DRAIN);
    }
  } else {
    // -------------------------------------------------------------- epilogue
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    const int r_in_tile = q * 32 + lane;
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int tile = blockIdx.x; tile < numTiles; tile += gridDim.x) {
      int mt, nt;
      tile_coords(tile, numM, numN, p.group_m, mt, nt);
      if (!mbar_wait(&acc_full[acc], acc_phase, wb, SITE_GEMM_EPILOGUE)) break;
      tc_fence_after();
      const long long row = (long long)mt * BM + r_in_tile;
      const bool row_ok = row < p.M;
      const uint32_t tbase = tmem_base + (uint32_t)(acc * BN) + ((uint32_t)(q * 32) << 16);
      long long nat = 0;  // natural token position of this row (K_QKV_SPLIT)
      if constexpr (EPI == K_QKV_SPLIT) {
        // sharded row (rank*B + b)*T + l of a micro-batch -> natural row b*S + pos
        const long long arow = row + p.zz_row0;
        const long long rb = arow / p.zz_T, l = arow - rb * p.zz_T;
        const long long rank = rb / p.zz_B, b = rb - rank * p.zz_B;
        nat = b * (p.zz_T * p.zz_D) +
              (l < p.zz_C ? rank * p.zz_C + l : (2 * p.zz_D - 1 - rank) * p.zz_C + (l - p.zz_C));
      }
      if constexpr (EPI == K_SWIGLU || EPI == K_SWIGLU_SAVE) {
        // columns [0,128) of the tile are gate rows (W1), [128,256) up rows (W3)
        const int half_n = p.N >> 1;
#pragma unroll 1
        for (int c = 0; c < BN / 2; c += 32) {
          const int ocol = nt * (BN / 2) + c;
          if (ocol >= half_n) break;
          uint32_t gv[32], uv[32];
          tmem_ld32(tbase + c, gv);
          tmem_ld32(tbase + BN / 2 + c, uv);
          tmem_ld_wait();
          if (row_ok) {
            float f[32];
#pragma unroll
            for (int j = 0; j < 32; ++j) {
              const float g = __uint_as_float(gv[j]);
              const float u = __uint_as_float(uv[j]);
              f[j] = g / (1.0f + __expf(-g)) * u;
            }
            store_row32(p.C + row * p.ldc + ocol, f, p.wide);
            if constexpr (EPI == K_SWIGLU_SAVE) {
              float a1[32], a3[32];
#pragma unroll
              for (int j = 0; j < 32; ++j) {
                a1[j] = __uint_as_float(gv[j]);
                a3[j] = __uint_as_float(uv[j]);
              }
              store_row32(p.C2 + row * p.ldc2 + nt * BN + c, a1, p.wide);
              store_row32(p.C2 + row * p.ldc2 + nt * BN + BN / 2 + c, a3, p.wide);
            }
          }
        }
      } else {
#pragma unroll 1
        for (int c = 0; c < BN; c += 32) {
          const int col = nt * BN + c;
          if (col >= p.N) break;
          uint32_t v[32];
          tmem_ld32(tbase + c, v);
          tmem_ld_wait();
          if (row_ok) {
            float f[32];
#pragma unroll
            for (int j = 0; j < 32; ++j) f[j] = __uint_as_float(v[j]);
            if constexpr (EPI == K_RES_BF16 || EPI == K_RES_BF16_OUT32)
              add_row32_bf16(f, static_cast<const __nv_bfloat16*>(p.R) + row * p.ldr + col, p.wide);
            if constexpr (EPI == K_RES_F32 || EPI == K_RES_F32_OUT32)
              add_row32_f32(f, static_cast<const float*>(p.R) + row * p.ldr + col, p.wide);
            if constexpr (EPI == K_RES_BF16_OUT32 || EPI == K_RES_F32_OUT32)
              store_row32_f32(p.C32 + row * p.ldc + col, f, p.wide);
            if constexpr (EPI == K_STORE_F32) {
              store_row32_f32(p.C32 + row * p.ldc + col, f, p.wide);
            } else if constexpr (EPI == K_SWIGLU_BWD) {
              // f = dG for padded ffn columns col..col+31 (one 128-column group g);
              // silu'(a) = s (1 + a (1 - s)), s = sigmoid(a)
              const int g = col / (BN / 2), j0 = col - g * (BN / 2);
              const long long c1 = (long long)g * BN + j0, c3 = c1 + BN / 2;
              // C may alias C2: each element is read, then written, by this thread alone
              const uint4* a1p = reinterpret_cast<const uint4*>(p.C2 + row * p.ldc2 + c1);
              const uint4* a3p = reinterpret_cast<const uint4*>(p.C2 + row * p.ldc2 + c3);
              float d1[32], d3[32];
#pragma unroll
              for (int w = 0; w < 4; ++w) {
                const uint4 x1 = a1p[w], x3 = a3p[w];
                const uint32_t u1[4] = {x1.x, x1.y, x1.z, x1.w}, u3[4] = {x3.x, x3.y, x3.z, x3.w};
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                  const float a1 = (e & 1) ? bf16_hi(u1[e >> 1]) : bf16_lo(u1[e >> 1]);
                  const float a3 = (e & 1) ? bf16_hi(u3[e >> 1]) : bf16_lo(u3[e >> 1]);
                  const float sg = 1.0f / (1.0f + __expf(-a1));
                  const float dg = f[8 * w + e];
                  d1[8 * w + e] = dg * a3 * sg * (1.0f + a1 * (1.0f - sg));
                  d3[8 * w + e] = dg * a1 * sg;
                }
              }
              store_row32(p.C + row * p.ldc + c1, d1, p.wide);
              store_row32(p.C + row * p.ldc + c3, d3, p.wide);
            } else if constexpr (EPI == K_QKV_SPLIT) {
              // a 32-column chunk never straddles sections (split_hd % 32 == 0); the
              // sections go Q, K, V for each of the N / (3 split_hd) shards in turn,
              // and shard j's columns land at offset j * split_hd of each destination
              const int sec = col / p.split_hd;
              const int part = sec % 3;
              const int lc = (sec / 3) * p.split_hd + (col - sec * p.split_hd);
              if (part == 0)
                store_row32(p.C + row * p.ldc + lc, f, p.wide);
              else
                store_row32((part == 1 ? p.split_k : p.split_v) + nat * p.split_ld + lc, f, p.wide);
            } else {
              store_row32(p.C + row * p.ldc + col, f, p.wide);
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acc_empty[acc]);
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1u;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

bool aligned16(const void* ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15u) == 0; }

template <int EPI, bool A_MN, bool B_MN>
tsp_status launch_epi(const CUtensorMap& ta, const CUtensorMap& tb, const GemmParams& p, int grid,
                      cudaStream_t stream) {
  auto kernel = gemm_bf16_tcgen05<EPI, A_MN, B_MN>;
  TSP_TRY(ensure_smem_limit(reinterpret_cast<const void*>(kernel), (int)SMEM_BYTES,
                            "gemm: cudaFuncSetAttribute"));
  kernel<<<grid, THREADS, SMEM_BYTES, stream>>>(ta, tb, p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "gemm: launch");
  return TSP_OK;
}

}  // namespace

tsp_status launch_gemm(const GemmCall& c, cudaStream_t stream) {
  if (!c.A || !c.B || !(c.C || c.epi == EPI_STORE_F32) || !c.status)
    return fail(TSP_ERR_INVALID_ARG, "gemm: null pointer");
  if (c.M <= 0 || c.N <= 0 || c.K <= 0) return fail(TSP_ERR_INVALID_ARG, "gemm: empty shape");
  // a ragged last K block reads zeros past the end of K (TMA out-of-bounds fill)
  if (c.ring_rows > 0 && c.K % BK)
    return fail(TSP_ERR_UNSUPPORTED, "gemm: ring order needs K to be a multiple of 64");
  if (c.epi == EPI_SWIGLU ? (c.N % 64) : (c.N % 32))
    return fail(TSP_ERR_UNSUPPORTED, "gemm: N must be a multiple of 32 (64 for SwiGLU)");
  if (c.b_row0 < 0 || c.b_row0 + c.N > c.b_rows)
    return fail(TSP_ERR_INVALID_ARG, "gemm: B row range out of bounds");
  if (!aligned16(c.A) || !aligned16(c.B) || (c.C && !aligned16(c.C)) || (c.R && !aligned16(c.R)) ||
      (c.C32 && !aligned16(c.C32)) || (c.lda % 8) || (c.ldb % 8) || (c.ldc % 8) ||
      (c.R && (c.ldr % 8)))
    return fail(TSP_ERR_INVALID_ARG, "gemm: buffers and row strides must be 16-byte aligned");
  if (c.epi == EPI_RESIDUAL && !c.R) return fail(TSP_ERR_INVALID_ARG, "gemm: residual missing");
  if (c.epi == EPI_STORE_F32 && (!c.C32 || !aligned16(c.C32) || (c.ldc % 4)))
    return fail(TSP_ERR_INVALID_ARG, "gemm: fp32 output missing or misaligned");
  if ((c.epi == EPI_SWIGLU_SAVE || c.epi == EPI_SWIGLU_BWD) &&
      (!c.C2 || !aligned16(c.C2) || (c.ldc2 % 8) || c.N % 128))
    return fail(TSP_ERR_INVALID_ARG, "gemm: SwiGLU pre-activation buffer missing or misaligned");
  if (c.C32 && c.epi != EPI_STORE_F32 && c.epi != EPI_RESIDUAL)
    return fail(TSP_ERR_INVALID_ARG, "gemm: an fp32 copy of the output needs the residual epilogue");
  if (c.C32 && c.residual_f32 && (c.a_mn || c.b_mn))
    return fail(TSP_ERR_INVALID_ARG, "gemm: fp32 residual with an fp32 output: K-major operands only");
  if (c.epi == EPI_QKV_SPLIT &&
      (!c.split_k || !c.split_v || c.split_hd <= 0 || c.split_hd % 32 || c.N % (3 * c.split_hd) ||
       c.ldc < c.N / 3 || c.split_ld < c.N / 3 || (c.split_ld % 8) || !aligned16(c.split_k) ||
       !aligned16(c.split_v) || c.zz_C <= 0 || c.zz_T != 2 * c.zz_C || c.zz_D <= 0 ||
       c.zz_row0 < 0 || c.zz_row0 + c.M > c.zz_T * c.zz_D * (c.zz_B > 0 ? c.zz_B : 1)))
    return fail(TSP_ERR_INVALID_ARG, "gemm: bad Q/K/V split arguments");
  if (c.M > (1ll << 30) || c.N > (1ll << 30) || c.K > (1ll << 30) || c.b_rows > (1ll << 30))
    return fail(TSP_ERR_UNSUPPORTED, "gemm: dimension too large");
  if (c.ring_rows > 0 && (c.ring_kblocks <= 0))
    return fail(TSP_ERR_INVALID_ARG, "gemm: ring order needs ring_kblocks > 0");

  CUtensorMap ta, tb;
  // K-major operands: [rows][K] with boxes of 64 K-elements; MN-major operands:
  // [K][rows] with boxes of 64 elements x 64 K-rows
  tsp_status st = c.a_mn ? make_tmap_2d_bf16(&ta, c.A, (uint64_t)c.M, (uint64_t)c.K,
                                             (uint64_t)c.lda * 2, 64, 64)
                         : make_tmap_2d_bf16(&ta, c.A, (uint64_t)c.K, (uint64_t)c.M,
                                             (uint64_t)c.lda * 2, BK, BM);
  if (st != TSP_OK) return st;
  st = c.b_mn ? make_tmap_2d_bf16(&tb, c.B, (uint64_t)c.b_rows, (uint64_t)c.K,
                                  (uint64_t)c.ldb * 2, 64, 64)
              : make_tmap_2d_bf16(&tb, c.B, (uint64_t)c.K, (uint64_t)c.b_rows,
                                  (uint64_t)c.ldb * 2, BK, BN);
  if (st != TSP_OK) return st;

  GemmParams p;
  p.M = (int)c.M;
  p.N = (int)c.N;
  p.K = (int)c.K;
  p.b_row0 = (int)c.b_row0;
  p.C = static_cast<__nv_bfloat16*>(c.C);
  p.ldc = c.ldc;
  p.R = c.R;
  p.ldr = c.ldr;
  p.C32 = static_cast<float*>(c.C32);
  p.split_k = static_cast<__nv_bfloat16*>(c.split_k);
  p.split_v = static_cast<__nv_bfloat16*>(c.split_v);
  p.split_ld = c.split_ld;
  p.split_hd = (int)c.split_hd;
  p.zz_C = c.zz_C;
  p.zz_T = c.zz_T;
  p.zz_D = c.zz_D;
  p.zz_B = c.zz_B > 0 ? c.zz_B : 1;
  p.zz_row0 = c.zz_row0;
  p.C2 = static_cast<__nv_bfloat16*>(c.C2);
  p.ldc2 = c.ldc2;
  p.ring_rows = (int)c.ring_rows;
  p.ring_kblocks = (int)c.ring_kblocks;
  p.ring_rank0 = c.ring_rank0;
  // Tile order. If B fits easily in the 129 MB L2 (<= 48 MB), walk row-major: A is
  // read once and B stays cached. Otherwise group about 32 MB of A row blocks
  // (128 x K bf16 each) so each B column block is fetched once per group: the
  // SwiGLU gate/up weights (184 MB at the 7B shape) read 28.6 GB from DRAM per 64K
  // launch in row-major order, and the grouped walk runs 17% faster.
  {
    const long long b_bytes = c.N * c.K * 2;
    const long long row_block_bytes = (long long)BM * c.K * 2;
    long long g = b_bytes <= (48ll << 20) ? 1 : (32ll << 20) / row_block_bytes;
    p.group_m = (int)(g < 1 ? 1 : g);
  }
  {
    // 32-byte epilogue accesses need every pointer and row stride the epilogue
    // touches to be 32-byte aligned (columns move in steps of 32 elements)
    auto al32 = [](const void* q) { return (reinterpret_cast<uintptr_t>(q) & 31u) == 0; };
    bool w = true;
    if (c.C) w = w && al32(c.C) && (c.ldc * 2) % 32 == 0;
    if (c.C32) w = w && al32(c.C32) && (c.ldc * 4) % 32 == 0;
    if (c.C2) w = w && al32(c.C2) && (c.ldc2 * 2) % 32 == 0;
    if (c.R) w = w && al32(c.R) && (c.ldr * (c.residual_f32 ? 4 : 2)) % 32 == 0;
    if (c.epi == EPI_QKV_SPLIT)
      w = w && al32(c.split_k) && al32(c.split_v) && (c.split_ld * 2) % 32 == 0;
    p.wide = w ? 1 : 0;
  }
  p.status = c.status;
  p.limit_ns = wait_limit_ns();

  const long long tiles = ((c.M + BM - 1) / BM) * ((c.N + BN - 1) / BN);
  const int grid = (int)(tiles < sm_count() ? tiles : sm_count());
  const int majors = (c.a_mn ? 2 : 0) + (c.b_mn ? 1 : 0);
  if (majors == 0) {  // forward products
    switch (c.epi) {
      case EPI_STORE: return launch_epi<K_STORE, false, false>(ta, tb, p, grid, stream);
      case EPI_SWIGLU: return launch_epi<K_SWIGLU, false, false>(ta, tb, p, grid, stream);
      case EPI_SWIGLU_SAVE: return launch_epi<K_SWIGLU_SAVE, false, false>(ta, tb, p, grid, stream);
      case EPI_QKV_SPLIT: return launch_epi<K_QKV_SPLIT, false, false>(ta, tb, p, grid, stream);
      case EPI_RESIDUAL:
        if (c.residual_f32 && c.C32)
          return launch_epi<K_RES_F32_OUT32, false, false>(ta, tb, p, grid, stream);
        if (c.residual_f32) return launch_epi<K_RES_F32, false, false>(ta, tb, p, grid, stream);
        if (c.C32) return launch_epi<K_RES_BF16_OUT32, false, false>(ta, tb, p, grid, stream);
        return launch_epi<K_RES_BF16, false, false>(ta, tb, p, grid, stream);
      default: break;
    }
  } else if (majors == 1) {  // data gradients: B MN-major
    switch (c.epi) {
      case EPI_STORE: return launch_epi<K_STORE, false, true>(ta, tb, p, grid, stream);
      case EPI_SWIGLU_BWD: return launch_epi<K_SWIGLU_BWD, false, true>(ta, tb, p, grid, stream);
      case EPI_RESIDUAL:
        if (c.residual_f32) return launch_epi<K_RES_F32, false, true>(ta, tb, p, grid, stream);
        if (c.C32) return launch_epi<K_RES_BF16_OUT32, false, true>(ta, tb, p, grid, stream);
        return launch_epi<K_RES_BF16, false, true>(ta, tb, p, grid, stream);
      default: break;
    }
  } else if (majors == 3) {  // weight gradients: both MN-major, fp32 out
    if (c.epi == EPI_STORE_F32) return launch_epi<K_STORE_F32, true, true>(ta, tb, p, grid, stream);
  }
  return fail(TSP_ERR_INVALID_ARG, "gemm: unsupported epilogue / operand layout combination");
}

}  // namespace tsp
