// attention.cu - causal attention of zigzag query rows against the gathered K/V
// ("Folding Tensor and Sequence Parallelism for Memory-Efficient Transformer
// Training & Inference", section 2, attention layers: FlashAttention after the
// K/V all-gather; zigzag partitioning for causal balance).
//
// One CTA computes 128 query rows of one head on the 5th-generation tensor cores:
//   warp 0      TMA: the Q tile once, then K and V tiles of 128 keys into two
//               3-stage rings of 128B-swizzled shared-memory buffers, in the order
//               the MMAs consume them (K_0, then K_{j+1} before V_j); a K slot frees
//               as soon as its S MMA completes, a V slot when its PV MMA completes
//   warp 1      allocates 512 TMEM columns; one lane issues
//                 S_j  = Q K_j^T          tcgen05.mma, A and B from shared memory
//                 O   += P_j V_j          tcgen05.mma, A (= P) from tensor memory,
//                                          B (= V) MN-major from shared memory
//               with S_{j+1} issued before O += P_j V_j, so the tensor core works
//               on the next scores while the softmax of the current tile runs
//   warps 2..5  softmax, one query row per thread (TMEM lane = row): tcgen05.ld of
//               the S row, mask by global position, row max, exp2, row sum, bf16
//               P written back to TMEM with tcgen05.st; then the epilogue. The four
//               TMEM loads of a row are in flight together, and the row max and sum
//               use 8 independent partial accumulators (one warp per SM sub-partition
//               has no other warp to hide a 128-long dependency chain behind).
// TMEM columns: S0 [0,128) S1 [128,256) O [256,256+d) P0 [384,448) P1 [448,512).
//
// Online softmax in base 2 (scores pre-scaled by log2(e)/sqrt(d)). Each row keeps a
// reference maximum m and sum l; m only moves (and O and l are rescaled) when the
// tile maximum exceeds it by more than 8, so P = exp2(s - m) <= 256 and most tiles
// never touch O. The result is exact softmax: out = O / l at the end.
//
// Query row r of the rank-major layout is the token at global position pos(r) of
// the zigzag map; key t is visible iff t <= pos(r). CTAs of one head run before
// the next head (K/V of a head stay in L2 across its CTAs) and, when the zigzag
// chunk is a multiple of 128 tokens, take query tiles in decreasing position, so
// the longest tiles start first.
#include "tsp_device.cuh"
#include "tsp_internal.h"

namespace tsp {
namespace {

constexpr int QT = 128;      // query rows per CTA
constexpr int KT = 128;      // keys per tile
constexpr int KSTAGES = 3;   // K ring depth (a K slot frees when its S MMA completes)
constexpr int VSTAGES = 3;   // V ring depth (a V slot frees when its PV MMA completes)
constexpr int THREADS = 192;
constexpr uint32_t BOX_BYTES = 128 * 128;  // one TMA box: 128 rows x 64 bf16
constexpr uint32_t TM_S0 = 0, TM_S1 = 128, TM_O = 256, TM_P0 = 384, TM_P1 = 448;
constexpr uint32_t TMEM_COLS = 512;
constexpr float RESCALE_THRESHOLD = 8.0f;  // log2 units

template <int HD>
struct Geometry {
  static constexpr int BOXES = HD / 64;                 // 64-column boxes per row block
  static constexpr uint32_t Q_BYTES = QT * HD * 2;
  static constexpr uint32_t K_BYTES = KT * HD * 2;
  static constexpr size_t USED = 1024 + Q_BYTES + (size_t)(KSTAGES + VSTAGES) * K_BYTES + 256;
  // The CTA allocates all 512 TMEM columns, so it must be alone on its SM: ask for
  // more than half of the SM's 228 KB of shared memory.
  static constexpr size_t SMEM = USED > 120 * 1024 ? USED : 120 * 1024;
};

struct AttParams {
  __nv_bfloat16* o;
  long long ld_o;
  long long o_col0;
  long long S, T, C;
  int D;
  int heads;
  int q_tiles;
  int natural_order;
  float scale_log2;
  DevStatus* status;
  unsigned long long limit_ns;
};

__device__ __forceinline__ long long zig_row(long long t, long long C, long long T, int D) {
  const long long c = t / C, o = t - c * C;
  return c < D ? c * T + o : (2 * D - 1 - c) * T + C + o;
}

__device__ __forceinline__ long long row_pos(long long r, long long C, long long T, int D) {
  const long long rank = r / T, l = r - rank * T;
  return l < C ? rank * C + l : (2 * D - 1 - rank) * C + (l - C);
}

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

template <int HD>
__global__ void __launch_bounds__(THREADS, 1)
    attention_tcgen05_kernel(const __grid_constant__ CUtensorMap tmQ,
                             const __grid_constant__ CUtensorMap tmK,
                             const __grid_constant__ CUtensorMap tmV, const AttParams p) {
  using G = Geometry<HD>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sQ = smem;
  uint8_t* sK = smem + G::Q_BYTES;             // KSTAGES x K_BYTES
  uint8_t* sV = sK + KSTAGES * G::K_BYTES;     // VSTAGES x K_BYTES
  uint64_t* bars = reinterpret_cast<uint64_t*>(sV + VSTAGES * G::K_BYTES);
  uint64_t* q_full = bars;                     // [1]
  uint64_t* k_full = bars + 1;                 // [KSTAGES]
  uint64_t* k_empty = k_full + KSTAGES;        // [KSTAGES]
  uint64_t* v_full = k_empty + KSTAGES;        // [VSTAGES]
  uint64_t* v_empty = v_full + VSTAGES;        // [VSTAGES]
  uint64_t* s_full = v_empty + VSTAGES;        // [2] S_j ready in TMEM
  uint64_t* p_full = s_full + 2;          // [2] P_j written to TMEM (4 softmax warps)
  uint64_t* o_done = p_full + 2;          // [2] O += P_j V_j completed
  uint64_t* drain = o_done + 2;           // [1]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int head = blockIdx.x / p.q_tiles;
  const int tile = blockIdx.x - head * p.q_tiles;
  long long row0;
  if (p.natural_order) {
    row0 = zig_row((long long)(p.q_tiles - 1 - tile) * QT, p.C, p.T, p.D);
  } else {
    row0 = (long long)tile * QT;
  }
  // keys needed by this CTA: 0 .. largest position among its rows
  long long max_pos;
  if (p.natural_order) {
    max_pos = row_pos(row0 + QT - 1, p.C, p.T, p.D);
  } else {
    max_pos = 0;
    const long long last = min(row0 + QT, p.S);
    for (long long r = row0; r < last; ++r) max_pos = max(max_pos, row_pos(r, p.C, p.T, p.D));
  }
  const int n_tiles = (int)(max_pos / KT) + 1;
  const int col_q = head * HD;  // Q columns inside qkv; K/V columns inside kn/vn

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int s = 0; s < KSTAGES; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&k_empty[s], 1);
    }
    for (int s = 0; s < VSTAGES; ++s) {
      mbar_init(&v_full[s], 1);
      mbar_init(&v_empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&s_full[b], 1);
      mbar_init(&p_full[b], 4);
      mbar_init(&o_done[b], 1);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  WaitBound wb{p.status, p.limit_ns, abort_flag};

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------------ TMA producer
      mbar_arrive_expect_tx(q_full, G::Q_BYTES);
#pragma unroll
      for (int b = 0; b < G::BOXES; ++b)
        tma_load_2d(sQ + b * BOX_BYTES, &tmQ, q_full, col_q + 64 * b, (int)row0);
      // loads in the order the MMA warp consumes them: K_0, then K_{j+1}, V_j
      int k_last[KSTAGES], v_last[VSTAGES];
#pragma unroll
      for (int t = 0; t < KSTAGES; ++t) k_last[t] = -1;
#pragma unroll
      for (int t = 0; t < VSTAGES; ++t) v_last[t] = -1;
      auto load_k = [&](int j) {
        const int st = j % KSTAGES;
        const uint32_t ph = (uint32_t)((j / KSTAGES) & 1);
        if (!mbar_wait(&k_empty[st], ph ^ 1u, wb, SITE_ATT_PRODUCER)) return false;
        mbar_arrive_expect_tx(&k_full[st], G::K_BYTES);
#pragma unroll
        for (int b = 0; b < G::BOXES; ++b)
          tma_load_2d(sK + st * G::K_BYTES + b * BOX_BYTES, &tmK, &k_full[st], col_q + 64 * b,
                      j * KT);
        k_last[st] = (int)ph;
        return true;
      };
      auto load_v = [&](int j) {
        const int st = j % VSTAGES;
        const uint32_t ph = (uint32_t)((j / VSTAGES) & 1);
        if (!mbar_wait(&v_empty[st], ph ^ 1u, wb, SITE_ATT_PRODUCER)) return false;
        mbar_arrive_expect_tx(&v_full[st], G::K_BYTES);
#pragma unroll
        for (int b = 0; b < G::BOXES; ++b)
          tma_load_2d(sV + st * G::K_BYTES + b * BOX_BYTES, &tmV, &v_full[st], col_q + 64 * b,
                      j * KT);
        v_last[st] = (int)ph;
        return true;
      };
      bool ok = load_k(0);
      for (int j = 0; ok && j < n_tiles; ++j) {
        if (j + 1 < n_tiles) ok = load_k(j + 1);
        if (ok) ok = load_v(j);
      }
      WaitBound wd{p.status, p.limit_ns, nullptr};
      mbar_wait(q_full, 0, wd, SITE_DRAIN);
      for (int t = 0; t < KSTAGES; ++t)
        if (k_last[t] >= 0) mbar_wait(&k_full[t], (uint32_t)k_last[t], wd, SITE_DRAIN);
      for (int t = 0; t < VSTAGES; ++t)
        if (v_last[t] >= 0) mbar_wait(&v_full[t], (uint32_t)v_last[t], wd, SITE_DRAIN);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ------------------------------------------------------------ MMA issuer
      const uint32_t idesc_s = make_idesc_bf16(QT, KT, false);
      const uint32_t idesc_o = make_idesc_bf16(QT, HD, true);
      const uint32_t q_addr = smem_addr(sQ);
      auto issue_s = [&](int j) {
        const uint32_t k_addr = smem_addr(sK + (j % KSTAGES) * G::K_BYTES);
        const uint32_t d_tmem = tmem + ((j & 1) ? TM_S1 : TM_S0);
#pragma unroll
        for (int kk = 0; kk < HD / 16; ++kk) {
          const uint32_t off = (uint32_t)((kk >> 2) * BOX_BYTES + (kk & 3) * 32);
          mma_ss(d_tmem, make_sdesc_sw128(q_addr + off, 16, 1024),
                 make_sdesc_sw128(k_addr + off, 16, 1024), idesc_s, kk > 0 ? 1u : 0u);
        }
        mma_commit(&s_full[j & 1]);
        mma_commit(&k_empty[j % KSTAGES]);
      };
      bool ok = mbar_wait(q_full, 0, wb, SITE_ATT_MMA);
      if (ok) ok = mbar_wait(&k_full[0], 0, wb, SITE_ATT_MMA);
      if (ok) {
        tc_fence_after();
        issue_s(0);
      }
      for (int j = 0; ok && j < n_tiles; ++j) {
        if (j + 1 < n_tiles) {
          const int st = (j + 1) % KSTAGES;
          if (!mbar_wait(&k_full[st], (uint32_t)(((j + 1) / KSTAGES) & 1), wb, SITE_ATT_MMA)) break;
          tc_fence_after();
          issue_s(j + 1);
        }
        if (!mbar_wait(&p_full[j & 1], (uint32_t)((j >> 1) & 1), wb, SITE_ATT_MMA)) break;
        if (!mbar_wait(&v_full[j % VSTAGES], (uint32_t)((j / VSTAGES) & 1), wb, SITE_ATT_MMA)) break;
        tc_fence_after();
        const uint32_t v_addr = smem_addr(sV + (j % VSTAGES) * G::K_BYTES);
        const uint32_t p_tmem = tmem + ((j & 1) ? TM_P1 : TM_P0);
#pragma unroll
        for (int kk = 0; kk < KT / 16; ++kk) {
          // B = V: 16 keys (rows) x HD columns, MN-major: 64-column blocks BOX_BYTES
          // apart, 8-row groups 1024 B apart; A = P: 16 keys = 8 packed columns
          mma_ts(tmem + TM_O, p_tmem + (uint32_t)(kk * 8),
                 make_sdesc_sw128(v_addr + (uint32_t)(kk * 2048), BOX_BYTES, 1024), idesc_o,
                 (j > 0 || kk > 0) ? 1u : 0u);
        }
        mma_commit(&o_done[j & 1]);
        mma_commit(&v_empty[j % VSTAGES]);
      }
      mma_commit(drain);
      WaitBound wd{p.status, p.limit_ns, nullptr};
      mbar_wait(drain, 0, wd, SITE_DRAIN);
    }
  } else {
    // -------------------------------------------------------------- softmax
    const int q = warp & 3;
    const int r_local = q * 32 + lane;
    const long long grow = row0 + r_local;
    const bool row_ok = grow < p.S;
    const long long pos = row_ok ? row_pos(grow, p.C, p.T, p.D) : -1;
    const uint32_t lane_base = tmem + ((uint32_t)(q * 32) << 16);
    float m_ref = -INFINITY;  // reference maximum (scaled, log2 units)
    float l = 0.f;
    bool ok = true;
    // every lane waits; the warp goes on only if all lanes saw the phase complete
    auto warp_wait = [&](uint64_t* bar, uint32_t parity) {
      const bool mine = mbar_wait(bar, parity, wb, SITE_ATT_SOFTMAX);
      return __all_sync(0xffffffffu, mine) != 0;
    };
    for (int j = 0; j < n_tiles; ++j) {
      if (!warp_wait(&s_full[j & 1], (uint32_t)((j >> 1) & 1))) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t s_tmem = lane_base + ((j & 1) ? TM_S1 : TM_S0);
      // raw scores of this row: four TMEM loads in flight, one wait
      float sc[KT];
      {
        uint32_t ra[32], rb[32], rc[32], rd[32];
        tmem_ld32(s_tmem + 0, ra);
        tmem_ld32(s_tmem + 32, rb);
        tmem_ld32(s_tmem + 64, rc);
        tmem_ld32(s_tmem + 96, rd);
        tmem_ld_wait();
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          sc[e] = __uint_as_float(ra[e]);
          sc[32 + e] = __uint_as_float(rb[e]);
          sc[64 + e] = __uint_as_float(rc[e]);
          sc[96 + e] = __uint_as_float(rd[e]);
        }
      }
      const long long kv0 = (long long)j * KT;
      if (kv0 + KT - 1 > pos) {
#pragma unroll
        for (int e = 0; e < KT; ++e)
          if (kv0 + e > pos) sc[e] = -INFINITY;
      }
      // row maximum with 8 independent partial maxima (short dependency chains)
      float m8[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) m8[e] = sc[e];
#pragma unroll
      for (int e = 8; e < KT; ++e) m8[e & 7] = fmaxf(m8[e & 7], sc[e]);
      const float mraw = fmaxf(fmaxf(fmaxf(m8[0], m8[1]), fmaxf(m8[2], m8[3])),
                               fmaxf(fmaxf(m8[4], m8[5]), fmaxf(m8[6], m8[7])));
      const float mx = mraw * p.scale_log2;  // scale > 0 keeps the order
      // move the reference only when the tile maximum outgrows it by the threshold
      float factor = 1.f;
      const bool rescale = mx > m_ref + RESCALE_THRESHOLD;
      if (rescale) {
        factor = ex2(m_ref - mx);  // 0 when m_ref is still -inf
        m_ref = mx;
      }
      const float neg_ref = m_ref == -INFINITY ? 0.f : -m_ref;
      l *= factor;
      if (j > 0 && __any_sync(0xffffffffu, rescale && factor != 1.f)) {
        // O holds P_0..P_{j-1} V; wait for the last of those products, then rescale
        if (!warp_wait(&o_done[(j - 1) & 1], (uint32_t)(((j - 1) >> 1) & 1))) {
          ok = false;
          break;
        }
        tc_fence_after();
#pragma unroll
        for (int c = 0; c < HD; c += 16) {
          uint32_t r[16];
          tmem_ld16(lane_base + TM_O + c, r);
          tmem_ld_wait();
#pragma unroll
          for (int e = 0; e < 16; ++e) r[e] = __float_as_uint(__uint_as_float(r[e]) * factor);
          tmem_st16(lane_base + TM_O + c, r);
        }
      }
      // P_j goes to the buffer P_{j-2} used: its product must have completed
      if (j >= 2) {
        if (!warp_wait(&o_done[j & 1], (uint32_t)(((j - 2) >> 1) & 1))) {
          ok = false;
          break;
        }
      }
      const uint32_t p_tmem = lane_base + ((j & 1) ? TM_P1 : TM_P0);
      float sum8[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) sum8[e] = 0.f;
#pragma unroll
      for (int c = 0; c < KT; c += 32) {
        uint32_t r[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const float p0 = ex2(fmaf(sc[c + 2 * e], p.scale_log2, neg_ref));
          const float p1 = ex2(fmaf(sc[c + 2 * e + 1], p.scale_log2, neg_ref));
          sum8[e & 7] += p0 + p1;
          r[e] = pack_bf16x2(p0, p1);
        }
        tmem_st16(p_tmem + (uint32_t)(c / 2), r);
      }
      const float sum = ((sum8[0] + sum8[1]) + (sum8[2] + sum8[3])) +
                        ((sum8[4] + sum8[5]) + (sum8[6] + sum8[7]));
      l += sum;
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&p_full[j & 1]);
    }
    // ------------------------------------------------------------ epilogue
    if (ok && warp_wait(&o_done[(n_tiles - 1) & 1], (uint32_t)(((n_tiles - 1) >> 1) & 1))) {
      tc_fence_after();
      const float inv = l > 0.f ? 1.f / l : 0.f;
      __nv_bfloat16* dst = p.o + grow * p.ld_o + p.o_col0 + col_q;
#pragma unroll
      for (int c = 0; c < HD; c += 32) {
        uint32_t r[32];
        tmem_ld32(lane_base + TM_O + c, r);
        tmem_ld_wait();
        if (row_ok) {
          uint4* d4 = reinterpret_cast<uint4*>(dst + c);
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            uint4 w;
            w.x = pack_bf16x2(__uint_as_float(r[8 * v + 0]) * inv, __uint_as_float(r[8 * v + 1]) * inv);
            w.y = pack_bf16x2(__uint_as_float(r[8 * v + 2]) * inv, __uint_as_float(r[8 * v + 3]) * inv);
            w.z = pack_bf16x2(__uint_as_float(r[8 * v + 4]) * inv, __uint_as_float(r[8 * v + 5]) * inv);
            w.w = pack_bf16x2(__uint_as_float(r[8 * v + 6]) * inv, __uint_as_float(r[8 * v + 7]) * inv);
            d4[v] = w;
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

template <int HD>
tsp_status launch_hd(const AttentionCall& c, const AttParams& p, cudaStream_t stream) {
  CUtensorMap tq, tk, tv;
  tsp_status st = make_tmap_2d_bf16(&tq, c.qkv, (uint64_t)c.ld_qkv, (uint64_t)c.S,
                                    (uint64_t)c.ld_qkv * 2, 64, QT);
  if (st != TSP_OK) return st;
  st = make_tmap_2d_bf16(&tk, c.kn, (uint64_t)c.ld_kv, (uint64_t)c.S, (uint64_t)c.ld_kv * 2, 64, KT);
  if (st != TSP_OK) return st;
  st = make_tmap_2d_bf16(&tv, c.vn, (uint64_t)c.ld_kv, (uint64_t)c.S, (uint64_t)c.ld_kv * 2, 64, KT);
  if (st != TSP_OK) return st;
  auto kernel = attention_tcgen05_kernel<HD>;
  const size_t smem = Geometry<HD>::SMEM;
  cudaError_t e =
      cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return cuda_fail(e, "attention: cudaFuncSetAttribute");
  const long long blocks = (long long)p.q_tiles * p.heads;
  kernel<<<(unsigned)blocks, THREADS, smem, stream>>>(tq, tk, tv, p);
  e = cudaGetLastError();
  return e == cudaSuccess ? TSP_OK : cuda_fail(e, "attention: launch");
}

}  // namespace

tsp_status launch_attention(const AttentionCall& c, cudaStream_t stream) {
  if (c.d != 64 && c.d != 128) return fail(TSP_ERR_UNSUPPORTED, "attention: head_dim 64 or 128");
  if (!c.qkv || !c.kn || !c.vn || !c.o || !c.status)
    return fail(TSP_ERR_INVALID_ARG, "attention: null pointer");
  if ((c.ld_qkv % 8) || (c.ld_kv % 8) || (c.ld_o % 8) || (c.o_col0 % 8))
    return fail(TSP_ERR_INVALID_ARG, "attention: strides must be multiples of 8 elements");
  if ((long long)c.heads * c.d > c.ld_kv || (long long)c.heads * c.d > c.ld_qkv ||
      c.o_col0 + (long long)c.heads * c.d > c.ld_o)
    return fail(TSP_ERR_INVALID_ARG, "attention: head columns exceed the row width");
  if (c.S > (1ll << 30)) return fail(TSP_ERR_UNSUPPORTED, "attention: S too large");
  AttParams p;
  p.o = static_cast<__nv_bfloat16*>(c.o);
  p.ld_o = c.ld_o;
  p.o_col0 = c.o_col0;
  p.S = c.S;
  p.T = c.T;
  p.C = c.C;
  p.D = c.D;
  p.heads = c.heads;
  p.q_tiles = (int)((c.S + QT - 1) / QT);
  p.natural_order = (c.C % QT == 0) ? 1 : 0;
  p.scale_log2 = 1.4426950408889634f / sqrtf((float)c.d);
  p.status = c.status;
  p.limit_ns = wait_limit_ns();
  return c.d == 64 ? launch_hd<64>(c, p, stream) : launch_hd<128>(c, p, stream);
}

}  // namespace tsp
