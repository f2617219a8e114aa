// attention.cu - causal attention of zigzag query rows against the gathered K/V
// ("Folding Tensor and Sequence Parallelism for Memory-Efficient Transformer
// Training & Inference", section 2, attention layers: FlashAttention after the
// K/V all-gather; zigzag partitioning for causal balance).
//
// One CTA computes two 128-row query tiles (A and B) of one head on the
// 5th-generation tensor cores. Both tiles share every K/V tile the CTA loads.
//   warp 0      TMA: Q_A, Q_B and K_0 (own slot) once, then for each key tile j
//               the pair (V_j, K_{j+1}) into a 2-stage ring of 128B-swizzled shared
//               memory (one full and one empty barrier per pair)
//   warp 1      allocates all 512 TMEM columns; one lane issues, per key tile j,
//                 O_A += P_A V_j,  S_A = Q_A K_{j+1}^T,  O_B += P_B V_j,  S_B = Q_B K_{j+1}^T
//               (S from shared-memory operands; P read from TMEM as the A operand,
//               V as an MN-major shared-memory operand). While one tile's softmax
//               runs, the tensor core works on the other tile's products.
//   warps 2..5  softmax of tile A, warps 6..9 softmax of tile B: one query row per
//               thread (TMEM lane = row), two softmax warps per SM sub-partition so
//               each hides the other's latencies. tcgen05.ld of the S row (four
//               loads in flight), mask by global position, row max (three-input
//               max, 4 chains), P = exp2(s - m) with packed f32x2 argument and sum,
//               rounded to bf16 and written over the first 64 columns of the same S
//               with tcgen05.st; then the epilogue.
// TMEM columns: S_A [0,128) O_A [128,256) S_B [256,384) O_B [384,512); P_X
// occupies the first 64 columns of S_X (two bf16 per column).
//
// Ordering: MMAs issued by one thread execute in order, and tcgen05.commit arrives
// once every earlier MMA of the thread has completed. So S_X(j+1) may overwrite
// the columns P_X(j) is read from right after O_X += P_X(j) V_j is issued, and the
// completion of S_X(j) also tells the softmax that O_X += P_X(j-1) V_{j-1} is done;
// only a tile's last product is committed separately (for its epilogue). Every
// mbarrier operation costs the issuing thread on the order of a hundred cycles, so
// the MMA warp does three waits and three commits per key tile, and waits for the
// next K/V stage while tile A's products run.
//
// Online softmax in base 2 (scores scaled by log2(e)/sqrt(d) inside the exp
// argument). Each row keeps a reference maximum m and sum l; m only moves (and O
// and l are rescaled) when the tile maximum exceeds it by more than 8, so
// P <= 256 and most tiles never touch O. The result is exact softmax: O / l.
//
// Query row r of the rank-major layout is the token at global position pos(r) of
// the zigzag map; key t is visible iff t <= pos(r). A micro-batch of B sequences
// has rank-major [D][B][T] query rows and natural K/V rows b*S + t; the queries of
// sequence b see only its own keys.
//
// CTA order. The (sequence, head) pairs of the call are cut into groups whose K/V
// fit together in a share of L2 (two 64K-token heads; every head of a 16K sequence
// together). Groups run one after the other, so their K/V stay in L2
// across their CTAs. Inside a group the CTAs go query block by query block, every
// pair of the group at each block, and, when the zigzag chunk is a multiple of 256
// tokens, in decreasing position: the longest blocks of every pair start first
// (longest-first over the whole group, not only within one head).
#include "tsp_device.cuh"
#include "tsp_internal.h"

namespace tsp {
namespace {

constexpr int QT = 128;       // query rows per tile (two tiles per CTA)
constexpr int QB = 2 * QT;    // query rows per CTA
constexpr int KT = 128;       // keys per tile
constexpr int STAGES = 2;     // ring of (V_j, K_{j+1}) pairs; K_0 comes with Q
constexpr int THREADS = 320;  // TMA warp, MMA warp, 2 x 4 softmax warps
constexpr uint32_t BOX_BYTES = 128 * 128;  // one TMA box: 128 rows x 64 bf16
constexpr uint32_t TM_S0 = 0, TM_O0 = 128, TM_S1 = 256, TM_O1 = 384;
constexpr uint32_t TMEM_COLS = 512;
constexpr float RESCALE_THRESHOLD = 8.0f;  // log2 units

__device__ __forceinline__ uint32_t tm_s(int t) { return t ? TM_S1 : TM_S0; }
__device__ __forceinline__ uint32_t tm_o(int t) { return t ? TM_O1 : TM_O0; }

template <int HD>
struct Geometry {
  static constexpr int BOXES = HD / 64;  // 64-column boxes per 128-row block
  static constexpr uint32_t TILE_BYTES = 128 * HD * 2;
  // Q_A, Q_B, K_0, then the ring: K slots 0/1 and V slots 0/1
  static constexpr size_t USED = 1024 + (size_t)(3 + 2 * STAGES) * TILE_BYTES + 256;
  // The CTA allocates all 512 TMEM columns, so it must be alone on its SM: ask for
  // more than half of the SM's 228 KB of shared memory.
  static constexpr size_t SMEM = USED > 120 * 1024 ? USED : 120 * 1024;
};

struct AttParams {
  __nv_bfloat16* o;
  long long ld_o;
  long long o_col0;
  float* lse;          // optional: [head][row] base-2 log-sum-exp of the scaled scores
  long long ld_lse;
  long long S, T, C;  // one sequence
  int D;
  int B;               // sequences of the micro-batch
  int heads;
  int q_blocks;        // 256-row query blocks per (sequence, head)
  int group;           // (sequence, head) pairs whose CTAs interleave
  int natural_order;
  // the call's query rows: sharded rows [q_row0, q_end) of the sequence's [D][T]
  // layout (all S rows, or one rank's T rows); the Q, O and lse buffers hold them
  // from their row 0 on (buffer row = sharded row - q_row0)
  long long q_row0, q_end;
  long long q_buf0;    // micro-batch-layout row of the call's first row (r B T for rank r)
  int q_local;         // 1: one rank's rows (longest-first = last local block first)
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

// Row of the micro-batch's [D][B][T] layout that holds row v of sequence `seq`'s
// own [D][T] layout (the identity when B == 1).
__device__ __forceinline__ long long batch_row(long long v, int seq, const AttParams& p) {
  return v + ((v / p.T) * (p.B - 1) + seq) * p.T;
}

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// P = exp2(s * scale - m) for one row of 128 scores: bf16 pairs stored to TMEM
// (64 columns at p_tmem); returns the row sum. The argument and the sum use packed
// f32x2 FMA/ADD (two elements per instruction): the softmax is bound by instruction
// issue, not by the exponential unit (moving part of the exponentials to an FMA-pipe
// polynomial measured slower).
__device__ __forceinline__ float exp_tile(const float (&sc)[KT], uint32_t p_tmem, float scale,
                                          float neg_ref) {
  const uint64_t scale2 = f2_pack(scale, scale), nref2 = f2_pack(neg_ref, neg_ref);
  uint64_t sum2[2] = {0, 0};
#pragma unroll
  for (int c = 0; c < KT; c += 16) {
    uint32_t r[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      float x0, x1;
      f2_unpack(f2_fma(f2_pack(sc[c + 2 * e], sc[c + 2 * e + 1]), scale2, nref2), x0, x1);
      const float p0 = ex2(x0), p1 = ex2(x1);
      sum2[e & 1] = f2_add(sum2[e & 1], f2_pack(p0, p1));
      r[e] = pack_bf16x2(p0, p1);
    }
    tmem_st8(p_tmem + (uint32_t)(c / 2), r);
  }
  const uint64_t s01 = f2_add(sum2[0], sum2[1]);
  float a, b;
  f2_unpack(s01, a, b);
  return a + b;
}

// Number of 128-key tiles the query rows [r0, r0 + QT) need (0 if none is a row).
__device__ __forceinline__ int tiles_needed(long long r0, const AttParams& p) {
  if (r0 >= p.q_end) return 0;
  long long mx = 0;
  if (p.natural_order) {
    mx = row_pos(r0 + QT - 1, p.C, p.T, p.D);
  } else {
    const long long last = min(r0 + QT, p.q_end);
    for (long long r = r0; r < last; ++r) mx = max(mx, row_pos(r, p.C, p.T, p.D));
  }
  return (int)(mx / KT) + 1;
}

// Each SM sub-partition holds 16K registers and 10 warps put three warps on two of
// them, so a thread gets at most 168 registers.
template <int HD>
__global__ void __launch_bounds__(THREADS, 1)
    attention_tcgen05_kernel(const __grid_constant__ CUtensorMap tmQ,
                             const __grid_constant__ CUtensorMap tmK,
                             const __grid_constant__ CUtensorMap tmV, const AttParams p) {
  using G = Geometry<HD>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sQ = smem;                          // tile A, then tile B
  uint8_t* sK0 = sQ + 2 * G::TILE_BYTES;      // K_0
  uint8_t* sK = sK0 + G::TILE_BYTES;          // ring: K_{j+1} in slot j % 2
  uint8_t* sV = sK + STAGES * G::TILE_BYTES;  // ring: V_j in slot j % 2
  uint64_t* bars = reinterpret_cast<uint64_t*>(sV + STAGES * G::TILE_BYTES);
  uint64_t* q_full = bars;               // [1] Q_A, Q_B, K_0
  uint64_t* kv_full = q_full + 1;        // [STAGES] stage j % 2: V_j and K_{j+1}
  uint64_t* kv_empty = kv_full + STAGES; // [STAGES]
  uint64_t* s_full = kv_empty + STAGES;  // [2] per tile: S(j) in TMEM
  uint64_t* p_full = s_full + 2;         // [2] per tile: P(j) in TMEM (4 warps)
  uint64_t* o_done = p_full + 2;         // [2] per tile: its last O += P V complete
  uint64_t* drain = o_done + 2;          // [1]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  // the output row of tile A / B's first row and the head: the softmax warps read
  // them back for their epilogue instead of holding them across the key loop
  long long* out_row0 = reinterpret_cast<long long*>(tmem_slot + 2);  // [2]
  int* out_head = reinterpret_cast<int*>(out_row0 + 2);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // CTA -> group g, query block blk, pair (sequence, head) of the group
  const int pairs = p.heads * p.B;
  const int per_group = p.q_blocks * p.group;
  const int g = (int)(blockIdx.x / (unsigned)per_group);
  const int in_g = min(p.group, pairs - g * p.group);
  const int rem = (int)blockIdx.x - g * per_group;
  const int blk = rem / in_g;
  const int pair = g * p.group + (rem - blk * in_g);
  const int head = pair % p.heads;
  const int seq = pair / p.heads;
  const long long row0 =
      p.q_local ? p.q_row0 + (p.natural_order ? p.q_end - p.q_row0 - (long long)(blk + 1) * QB
                                              : (long long)blk * QB)
      : p.natural_order ? zig_row((long long)(p.q_blocks - 1 - blk) * QB, p.C, p.T, p.D)
                        : (long long)blk * QB;
  const int n_a = tiles_needed(row0, p);
  const int n_b = tiles_needed(row0 + QT, p);
  const int n_tiles = max(n_a, n_b);
  const int col_q = head * HD;  // Q columns inside qkv; K/V columns inside kn/vn
  const int kv_row0 = (int)(seq * p.S);  // first natural K/V row of the sequence

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&kv_full[s], 1);
      mbar_init(&kv_empty[s], 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(&s_full[t], 1);
      mbar_init(&p_full[t], 4);
      mbar_init(&o_done[t], 1);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    // a 128-row tile's rows are contiguous in the micro-batch layout too
    out_row0[0] = batch_row(row0, seq, p) - p.q_buf0;
    out_row0[1] = batch_row(row0 + QT, seq, p) - p.q_buf0;
    *out_head = head;
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
    if (lane == 0 && n_tiles > 0) {
      // ------------------------------------------------------------ TMA producer
      mbar_arrive_expect_tx(q_full, 3 * G::TILE_BYTES);
#pragma unroll
      for (int b = 0; b < G::BOXES; ++b) {
#pragma unroll
        for (int t = 0; t < 2; ++t)
          tma_load_2d(sQ + t * G::TILE_BYTES + b * BOX_BYTES, &tmQ, q_full, col_q + 64 * b,
                      (int)(batch_row(row0 + t * QT, seq, p) - p.q_buf0));
        tma_load_2d(sK0 + b * BOX_BYTES, &tmK, q_full, col_q + 64 * b, kv_row0);
      }
      int last[STAGES];
#pragma unroll
      for (int s = 0; s < STAGES; ++s) last[s] = -1;
      for (int j = 0; j < n_tiles; ++j) {
        // stage j % 2 takes V_j and K_{j+1}; its slots held V_{j-2} and K_{j-1}, both
        // consumed by the MMAs of iteration j-2 (whose commit frees the stage)
        const int st = j % STAGES;
        const uint32_t ph = (uint32_t)((j / STAGES) & 1);
        if (!mbar_wait(&kv_empty[st], ph ^ 1u, wb, SITE_ATT_PRODUCER)) break;
        const bool has_k = j + 1 < n_tiles;
        mbar_arrive_expect_tx(&kv_full[st], (has_k ? 2u : 1u) * G::TILE_BYTES);
#pragma unroll
        for (int b = 0; b < G::BOXES; ++b) {
          tma_load_2d(sV + st * G::TILE_BYTES + b * BOX_BYTES, &tmV, &kv_full[st],
                      col_q + 64 * b, kv_row0 + j * KT);
          if (has_k)
            tma_load_2d(sK + st * G::TILE_BYTES + b * BOX_BYTES, &tmK, &kv_full[st],
                        col_q + 64 * b, kv_row0 + (j + 1) * KT);
        }
        last[st] = (int)ph;
      }
      WaitBound wd{p.status, p.limit_ns, nullptr};
      mbar_wait(q_full, 0, wd, SITE_DRAIN);
      for (int s = 0; s < STAGES; ++s)
        if (last[s] >= 0) mbar_wait(&kv_full[s], (uint32_t)last[s], wd, SITE_DRAIN);
    }
  } else if (warp == 1) {
    if (lane == 0 && n_tiles > 0) {
      // ------------------------------------------------------------ MMA issuer
      const uint32_t idesc_s = make_idesc_bf16(QT, KT, false);
      const uint32_t idesc_o = make_idesc_bf16(QT, HD, true);
      // base descriptors, built once; each MMA adds a compile-time offset (>> 4) to
      // the low word. K-major operands: 16-element K steps are 32 B inside a 128 B
      // swizzle row, 64-element blocks BOX_BYTES apart. V (MN-major): 16-key steps
      // are 2048 B, 64-column blocks BOX_BYTES apart (LBO), 8-row groups 1 KB (SBO).
      const uint64_t dq0 = make_sdesc_sw128(smem_addr(sQ), 16, 1024);
      const uint64_t dk0 = make_sdesc_sw128(smem_addr(sK0), 16, 1024);
      const uint64_t dv0 = make_sdesc_sw128(smem_addr(sV), BOX_BYTES, 1024);
      const uint32_t q_hi = (uint32_t)(dq0 >> 32), k_hi = (uint32_t)(dk0 >> 32);
      const uint32_t v_hi = (uint32_t)(dv0 >> 32);
      constexpr uint32_t TILE16 = G::TILE_BYTES >> 4;
      // S_t = Q_t K_j^T
      auto issue_s = [&](int t, int j) {
        const uint32_t a_lo = (uint32_t)dq0 + (uint32_t)t * TILE16;
        // K_0 in its own slot right before the ring; K_j (j >= 1) in ring slot (j-1) % 2
        const uint32_t b_lo = (uint32_t)dk0 + (j == 0 ? 0u : (uint32_t)(1 + (j - 1) % STAGES) * TILE16);
        const uint32_t d = tmem + tm_s(t);
#pragma unroll
        for (int kk = 0; kk < HD / 16; ++kk) {
          const uint32_t off = (uint32_t)(((kk >> 2) * BOX_BYTES + (kk & 3) * 32) >> 4);
          mma_ss_w(d, a_lo + off, q_hi, b_lo + off, k_hi, idesc_s, kk > 0 ? 1u : 0u);
        }
        mma_commit(&s_full[t]);
      };
      // O_t += P_t V_j; A = P: 16 keys = 8 packed TMEM columns per step
      auto issue_pv = [&](int t, int j) {
        const uint32_t b_lo = (uint32_t)dv0 + (uint32_t)(j % STAGES) * TILE16;
        const uint32_t d = tmem + tm_o(t), a = tmem + tm_s(t);
        const uint32_t first = j > 0 ? 1u : 0u;
#pragma unroll
        for (int kk = 0; kk < KT / 16; ++kk)
          mma_ts_w(d, a + (uint32_t)(kk * 8), b_lo + (uint32_t)(kk * (2048 >> 4)), v_hi, idesc_o,
                   kk > 0 ? 1u : first);
      };
      bool ok = mbar_wait_poll(q_full, 0, wb, SITE_ATT_MMA);
      if (ok) {
        tc_fence_after();
        if (n_a > 0) issue_s(0, 0);
        if (n_b > 0) issue_s(1, 0);
        ok = mbar_wait_poll(&kv_full[0], 0, wb, SITE_ATT_MMA);
      }
      for (int j = 0; ok && j < n_tiles; ++j) {
        // stage j % 2 (V_j, K_{j+1}) has landed
        for (int t = 0; t < 2; ++t) {
          const int nt = t ? n_b : n_a;
          if (j < nt) {
            if (!mbar_wait_poll(&p_full[t], (uint32_t)(j & 1), wb, SITE_ATT_MMA)) {
              ok = false;
              break;
            }
            tc_fence_after();
            issue_pv(t, j);
            if (j + 1 < nt) {
              issue_s(t, j + 1);
            } else {
              mma_commit(&o_done[t]);  // the tile's last product
            }
          }
          // while tile A's products run, wait for the next stage
          if (t == 0 && j + 1 < n_tiles &&
              !mbar_wait_poll(&kv_full[(j + 1) % STAGES], (uint32_t)(((j + 1) / STAGES) & 1), wb,
                         SITE_ATT_MMA)) {
            ok = false;
            break;
          }
        }
        if (!ok) break;
        mma_commit(&kv_empty[j % STAGES]);  // V_j and K_{j+1} are consumed
      }
      mma_commit(drain);
      WaitBound wd{p.status, p.limit_ns, nullptr};
      mbar_wait(drain, 0, wd, SITE_DRAIN);
    }
  } else {
    // -------------------------------------------------------------- softmax
    const int t = (warp - 2) >> 2;  // query tile of this warpgroup: 0 = A, 1 = B
    const int q = warp & 3;         // TMEM lane quarter of this warp
    const int r_local = q * 32 + lane;
    const long long vrow = row0 + t * QT + r_local;  // row in the sequence's own layout
    const bool row_ok = vrow < p.q_end;
    // S < 2^30 (checked at launch): positions fit in int
    const int pos = row_ok ? (int)row_pos(vrow, p.C, p.T, p.D) : -1;
    const uint32_t lane_base = tmem + ((uint32_t)(q * 32) << 16);
    const uint32_t s_tmem = lane_base + tm_s(t);
    const uint32_t o_tmem = lane_base + tm_o(t);
    const int my_tiles = t ? n_b : n_a;
    float m_ref = -INFINITY;  // reference maximum (scaled, log2 units)
    float l = 0.f;
    bool ok = true;
    // every lane waits; the warp goes on only if all lanes saw the phase complete (the
    // bound is rebuilt from the kernel parameters at each wait: nothing of it stays in
    // registers across the key loop)
    auto warp_wait = [&](uint64_t* bar, uint32_t parity) {
      const WaitBound wbs{p.status, p.limit_ns, abort_flag};
      const bool mine = mbar_wait(bar, parity, wbs, SITE_ATT_SOFTMAX);
      return __all_sync(0xffffffffu, mine) != 0;
    };
    for (int j = 0; j < my_tiles; ++j) {
      // S(j) complete also means O += P(j-1) V_{j-1} is complete (in-order MMAs)
      if (!warp_wait(&s_full[t], (uint32_t)(j & 1))) {
        ok = false;
        break;
      }
      tc_fence_after();
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
      const int kv0 = j * KT;
      if (kv0 + KT - 1 > pos) {
#pragma unroll
        for (int e = 0; e < KT; ++e)
          if (kv0 + e > pos) sc[e] = -INFINITY;
      }
      // row maximum: three-input max, 4 independent chains (short dependency chains):
      // sc[0..3] start the chains, 15 steps take 8 scores each (sc[4..123]), and the
      // last four scores close them
      float m4[4] = {sc[0], sc[1], sc[2], sc[3]};
#pragma unroll
      for (int e = 4; e + 8 <= KT; e += 8) {
#pragma unroll
        for (int k = 0; k < 4; ++k) m4[k] = max3f(m4[k], sc[e + k], sc[e + 4 + k]);
      }
      static_assert(KT % 8 == 0, "the tail below covers the last 4 scores");
      const float mraw = max3f(max3f(m4[0], m4[1], sc[KT - 4]), max3f(m4[2], m4[3], sc[KT - 3]),
                               fmaxf(sc[KT - 2], sc[KT - 1]));
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
      // P = exp2(s*scale - m) in bf16 over the first 64 columns of S (masked keys: 0)
      l += exp_tile(sc, s_tmem, p.scale_log2, neg_ref);
      // rescale O (written by the products up to P(j-1) V_{j-1}, complete since S(j)
      // is) before P(j) is handed over; after the exponentials, so that the scores are
      // no longer live: 16 columns at a time
      if (j > 0 && __any_sync(0xffffffffu, rescale && factor != 1.f)) {
#pragma unroll 1
        for (int c = 0; c < HD; c += 16) {
          uint32_t r[16];
          tmem_ld16(o_tmem + c, r);
          tmem_ld_wait();
#pragma unroll
          for (int e = 0; e < 16; ++e) r[e] = __float_as_uint(__uint_as_float(r[e]) * factor);
          tmem_st16(o_tmem + c, r);
        }
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&p_full[t]);
    }
    // ------------------------------------------------------------ epilogue
    if (ok && my_tiles > 0 && warp_wait(&o_done[t], 0u)) {
      tc_fence_after();
      const long long grow = out_row0[t] + r_local;  // row in the micro-batch's layout
      const int ohead = *out_head;
      const float inv = l > 0.f ? 1.f / l : 0.f;
      // log2 of the softmax denominator in the scaled base-2 domain: P_ij is then
      // exp2(s_ij * scale_log2 - lse) for the backward pass
      if (p.lse != nullptr && row_ok) p.lse[(long long)ohead * p.ld_lse + grow] = m_ref + __log2f(l);
      __nv_bfloat16* dst = p.o + grow * p.ld_o + p.o_col0 + ohead * HD;
#pragma unroll
      for (int c = 0; c < HD; c += 32) {
        uint32_t r[32];
        tmem_ld32(o_tmem + c, r);
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
  // each map spans only the call's head columns (heads * d from its base pointer),
  // with the buffer's row stride: the buffers may hold more columns on either side
  const uint64_t rows = (uint64_t)c.S * (uint64_t)p.B;
  const uint64_t cols = (uint64_t)c.heads * (uint64_t)c.d;
  const uint64_t q_rows = p.q_local ? (uint64_t)(p.q_end - p.q_row0) * (uint64_t)p.B : rows;
  tsp_status st = make_tmap_2d_bf16(&tq, c.qkv, cols, q_rows, (uint64_t)c.ld_qkv * 2, 64, QT);
  if (st != TSP_OK) return st;
  st = make_tmap_2d_bf16(&tk, c.kn, cols, rows, (uint64_t)c.ld_kv * 2, 64, KT);
  if (st != TSP_OK) return st;
  st = make_tmap_2d_bf16(&tv, c.vn, cols, rows, (uint64_t)c.ld_kv * 2, 64, KT);
  if (st != TSP_OK) return st;
  auto kernel = attention_tcgen05_kernel<HD>;
  const size_t smem = Geometry<HD>::SMEM;
  TSP_TRY(ensure_smem_limit(reinterpret_cast<const void*>(kernel), (int)smem,
                            "attention: cudaFuncSetAttribute"));
  const long long blocks = (long long)p.q_blocks * p.heads * p.B;
  kernel<<<(unsigned)blocks, THREADS, smem, stream>>>(tq, tk, tv, p);
  cudaError_t e = cudaGetLastError();
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
  const int B = c.B > 0 ? c.B : 1;
  if (c.S * B > (1ll << 30) || (long long)((c.S + QB - 1) / QB) * c.heads * B > (1ll << 31) - 1)
    return fail(TSP_ERR_UNSUPPORTED, "attention: too many rows");
  // with several sequences a 128-row query tile must not straddle two ranks' blocks
  if (B > 1 && c.T % QT)
    return fail(TSP_ERR_UNSUPPORTED, "attention: a micro-batch needs S/D % 128 == 0");
  AttParams p;
  p.o = static_cast<__nv_bfloat16*>(c.o);
  p.ld_o = c.ld_o;
  p.o_col0 = c.o_col0;
  p.lse = c.lse;
  p.ld_lse = c.ld_lse;
  p.S = c.S;
  p.T = c.T;
  p.C = c.C;
  p.D = c.D;
  p.B = B;
  p.heads = c.heads;
  // the call's query rows: every rank's, or rank-local rows [q_row0, q_row0 + q_rows)
  const bool local = c.q_rows > 0;
  // with a micro-batch the range must be one rank's whole block (its rows of every
  // sequence are contiguous in the [D][B][T] layout)
  if (local && (c.q_row0 < 0 || c.q_row0 + c.q_rows > c.S ||
                (B > 1 && (c.q_row0 % c.T || c.q_rows != c.T))))
    return fail(TSP_ERR_INVALID_ARG, "attention: query rows outside the sequence, or not one "
                                     "rank's rows of a micro-batch");
  p.q_local = local ? 1 : 0;
  p.q_row0 = local ? c.q_row0 : 0;
  p.q_end = local ? c.q_row0 + c.q_rows : c.S;
  p.q_buf0 = local ? c.q_row0 * B : 0;  // q_row0 = r T: rank r's block starts at r B T
  p.q_blocks = (int)((p.q_end - p.q_row0 + QB - 1) / QB);
  {
    // pairs per group: their K and V (2 * S * d bf16 each) within 72 MB of the L2,
    // the pairs split evenly over the fewest groups (no short last group, whose
    // longest blocks would start late)
    const long long fit0 = (72LL << 20) / (4LL * c.S * c.d);
    const long long fit = fit0 < 1 ? 1 : fit0;
    const long long pairs = (long long)c.heads * B;
    const long long n_groups = (pairs + fit - 1) / fit;
    p.group = (int)((pairs + n_groups - 1) / n_groups);
  }
  // last-row position = tile maximum; for a rank's rows also whole 256-row blocks
  p.natural_order = (c.C % QB == 0 && (!local || (c.q_row0 % QB == 0 && c.q_rows % QB == 0)))
                        ? 1 : 0;
  p.scale_log2 = 1.4426950408889634f / sqrtf((float)c.d);
  p.status = c.status;
  p.limit_ns = wait_limit_ns();
  return c.d == 64 ? launch_hd<64>(c, p, stream) : launch_hd<128>(c, p, stream);
}

}  // namespace tsp
