// attention_bwd.cu - backward of the causal attention of zigzag query rows against
// the gathered K/V ("Folding Tensor and Sequence Parallelism for Memory-Efficient
// Transformer Training & Inference", section 2, attention layers; the page gives
// the forward only, this is its chain rule).
//
// With s_ij = q_i . k_j (raw), P_ij = exp2(s_ij * scale_log2 - lse_i) (lse from the
// forward, base 2), dP_ij = dO_i . v_j and Delta_i = sum_c dO_ic O_ic:
//     dS_ij = P_ij (dP_ij - Delta_i)
//     dV_j = sum_i P_ij dO_i,   dK_j = scale sum_i dS_ij q_i,   dQ_i = scale sum_j dS_ij k_j
// (scale = 1/sqrt(d)), over visible pairs (key position <= query position).
//
// Two kernels, each a CTA per (128-row tile, head) that keeps its accumulators in
// tensor memory while the other side streams past (no atomics, deterministic):
//   key-side  (dK, dV): the CTA owns 128 keys (natural order) and streams every
//             query tile that sees them (Q, dO, lse, Delta), computing
//             S^T = K Q^T and dP^T = V dO^T, then dV += P^T dO and dK += dS^T Q with
//             P^T and dS^T read from tensor memory as the A operand. Its dK/dV rows
//             are the gradient at the key's owner (the reverse of the all-gather)
//             and are written at the zigzag row of the key.
//   query-side (dQ): the CTA owns 128 query rows (sharded order) and streams the
//             key tiles they see, computing S = Q K^T, dP = dO V^T and
//             dQ += dS K. Its Q and dO rows sit in tensor memory as the A operand
//             of the first two products.
// The query side runs every product on a full 128-wide tile (N = 128 or N = d): a
// tcgen05.mma with M = 128 and K = 16 occupies the tensor pipe for about as long
// with N = 64 as with N = 128 on this part, so a narrower product runs at half
// rate. Its element-wise work is split into two phases that depend on different
// products, and the MMA lane orders its work (S(j+1), dQ(j), dP(j+1), ...) so that
// one phase runs under the products of the other:
//   phase a  (after the scores, which it then releases): P = exp2(s scale_log2 - lse);
//   phase b  (after dP):  dS = P (dP - Delta), stored as bf16 over dP.
// Warps 2..5 and 6..9 (two warpgroups, one accumulator row per thread) take key
// columns [0, 64) and [64, 128) of every tile.
// The key side streams each 128-row query tile as two 64-column halves (score and
// dP^T products with N = 64): warps 2..5 take half 0 and warps 6..9 half 1, so one
// half's element-wise work overlaps the other half's products. It keeps these
// narrower products because its element-wise chain (two exponential-bound phases
// and two tensor-memory round trips per tile) and its two-deep Q/dO ring, which is
// what fits in shared memory beside the owned K and V, leave the tensor pipe idle
// for longer than the halved products cost.
//   warp 0  TMA producer (key side: 2 stages of Q, dO, lse, Delta; query side:
//           3 stages of K, V)
//   warp 1  TMEM allocation (512 columns) and the single MMA-issuing lane
// TMEM columns: key side: dV [0, d), dK [d, 2d), half h: scores [256 + 128h, +64),
// dP^T [320 + 128h, +64), with bf16 P^T / dS^T over the first 32 columns of each.
// Query side: dQ [0, d), bf16 Q [d, 3d/2), bf16 dO [3d/2, 2d), scores [256, 384),
// dP [384, 512) with bf16 dS over [384 + 64g, +32) for warpgroup g.
// MMAs issued by one thread execute in order, so a product may write columns that
// an earlier-issued product reads.
// A micro-batch of B sequences (rank-major [D][B][T] sharded rows, natural K/V rows
// b*S + t) pairs every CTA with one (sequence, head); the CTA order is the forward
// kernel's, with a 48 MB share of L2: (sequence, head) pairs in groups whose K/V fit, and
// inside a group the owned tiles go tile index by tile index across the pairs, the
// longest first.
#include <type_traits>

#include "tsp_device.cuh"
#include "tsp_internal.h"

namespace tsp {
namespace {

constexpr int BT = 128;       // rows of the tile a CTA owns
constexpr int IT = 128;       // rows of a streamed tile
constexpr int GCOLS = 64;     // streamed-tile columns per element-wise warpgroup
constexpr int THREADS = 320;
constexpr uint32_t BOX_BYTES = 128 * 128;  // one TMA box: 128 rows x 64 bf16
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t TM_SC = 256;  // query side: scores S, 128 columns
constexpr uint32_t TM_DP = 384;  // query side: dP, 128 columns
// key side: each streamed tile in two 64-column halves h, scores at
// [256 + 128h, +64) and dP^T at [320 + 128h, +64)
constexpr int HALF = 64;
constexpr int STAGES = 2;
constexpr uint32_t HALF_ROWS_BYTES = HALF * 128;  // 64 rows of a box
__device__ __forceinline__ uint32_t tm_sc(int h) { return 256u + 128u * (uint32_t)h; }
__device__ __forceinline__ uint32_t tm_dp(int h) { return 320u + 128u * (uint32_t)h; }

struct BwdParams {
  __nv_bfloat16* dq;
  __nv_bfloat16* dk;
  __nv_bfloat16* dv;
  long long ld_dqkv;
  const float* lse;
  const float* delta;
  long long ld_stat;
  const __nv_bfloat16* q;     // query-side kernel: owned Q and dO rows, read once
  const __nv_bfloat16* dout;
  long long ld_q, ld_do;
  long long S, T, C;  // one sequence
  int D;
  int B;         // sequences of the micro-batch
  int heads;     // heads of the call
  int group;     // (sequence, head) pairs whose CTAs interleave
  int n_outer;   // owned tiles per (sequence, head)
  int natural;   // zigzag chunk is a multiple of 128: every 128-row tile is one
                 // contiguous run of positions
  float scale_log2;
  float scale;
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
__device__ __forceinline__ long long batch_row(long long v, int seq, const BwdParams& p) {
  return v + ((v / p.T) * (p.B - 1) + seq) * p.T;
}

// CTA -> (owned tile index, sequence, head) in the grouped order described above.
struct CtaPos {
  int tile, seq, head;
};
__device__ __forceinline__ CtaPos cta_pos(const BwdParams& p) {
  const int pairs = p.heads * p.B;
  const int per_group = p.n_outer * p.group;
  const int grp = (int)(blockIdx.x / (unsigned)per_group);
  const int in_g = min(p.group, pairs - grp * p.group);
  const int rem = (int)blockIdx.x - grp * per_group;
  const int tile = rem / in_g;
  const int pair = grp * p.group + (rem - tile * in_g);
  return CtaPos{tile, pair / p.heads, pair % p.heads};
}

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

template <int HD>
struct KeyGeom {
  static constexpr int BOXES = HD / 64;
  static constexpr uint32_t TILE = 128 * HD * 2;
  // K, V, then per stage Q, dO, lse[128], Delta[128]
  static constexpr uint32_t STAGE = 2 * TILE + 1024;
  static constexpr size_t USED = 1024 + 2 * (size_t)TILE + STAGES * (size_t)STAGE + 256;
  // all 512 TMEM columns: one CTA per SM
  static constexpr size_t SMEM = USED > 120 * 1024 ? USED : 120 * 1024;
};

template <int HD>
struct QueryGeom {
  static constexpr int BOXES = HD / 64;
  static constexpr uint32_t TILE = 128 * HD * 2;
  static constexpr int KV_STAGES = 3;
  // per stage K, V (Q and dO live in tensor memory)
  static constexpr uint32_t STAGE = 2 * TILE;
  static constexpr size_t USED = 1024 + KV_STAGES * (size_t)STAGE + 256;
  static constexpr size_t SMEM = USED > 120 * 1024 ? USED : 120 * 1024;
  // TMEM columns of the owned rows as bf16 A operands (two values per column)
  static constexpr uint32_t TM_Q = HD;
  static constexpr uint32_t TM_DO = HD + HD / 2;
};

// K-major operand offset (>> 4) of the kk-th 16-wide K step of a [rows][HD] tile
// stored as 64-column boxes.
__device__ __forceinline__ uint32_t kmajor_step(int kk) {
  return (uint32_t)(((kk >> 2) * BOX_BYTES + (kk & 3) * 32) >> 4);
}

// TMEM column of the bf16 A operand for the kk-th 16-wide step of a streamed
// tile's 128 columns: warpgroup g's 64 values sit in the first 32 columns of its
// own 64-column block.
__device__ __forceinline__ uint32_t packed_step(uint32_t base, int kk) {
  return base + (uint32_t)((kk >> 2) * GCOLS + (kk & 3) * 8);
}

// ============================================================== key side
template <int HD>
__global__ void __launch_bounds__(THREADS, 1)
    attention_bwd_dkv_kernel(const __grid_constant__ CUtensorMap tmQ,
                             const __grid_constant__ CUtensorMap tmDO,
                             const __grid_constant__ CUtensorMap tmK,
                             const __grid_constant__ CUtensorMap tmV, const BwdParams p,
                             int q_col0, int do_col0) {
  using G = KeyGeom<HD>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sK = smem;
  uint8_t* sV = sK + G::TILE;
  uint8_t* sStage = sV + G::TILE;  // stage s: Q, dO, lse, Delta
  uint64_t* bars = reinterpret_cast<uint64_t*>(sStage + STAGES * G::STAGE);
  uint64_t* kv_full = bars;               // [1]
  uint64_t* in_full = kv_full + 1;        // [STAGES]
  uint64_t* in_empty = in_full + STAGES;  // [STAGES]
  uint64_t* s_full = in_empty + STAGES;   // [2] per half
  uint64_t* p_full = s_full + 2;          // [2] per half (4 warps)
  uint64_t* acc_done = p_full + 2;        // [1]
  uint64_t* drain = acc_done + 1;         // [1]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  auto sQ = [&](int st) { return sStage + st * G::STAGE; };
  auto sDO = [&](int st) { return sStage + st * G::STAGE + G::TILE; };
  auto sLse = [&](int st) { return reinterpret_cast<float*>(sStage + st * G::STAGE + 2 * G::TILE); };
  auto sDel = [&](int st) { return sLse(st) + 128; };

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const CtaPos cp = cta_pos(p);
  const int head = cp.head, seq = cp.seq;
  const int kt = cp.tile;  // ascending: most work first
  const long long k0 = (long long)kt * BT;
  const int kv_row0 = (int)(seq * p.S);  // first natural K/V row of the sequence
  const int nq = (int)((p.S + IT - 1) / IT);
  // streamed query tiles: natural order from the diagonal tile on, else every tile
  const int n_inner = p.natural ? nq - kt : nq;
  auto row0_of = [&](int idx) -> long long {
    return p.natural ? zig_row((long long)(kt + idx) * IT, p.C, p.T, p.D) : (long long)idx * IT;
  };

  if (threadIdx.x == 0) {
    mbar_init(kv_full, 1);
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&in_full[s], 1);
      mbar_init(&in_empty[s], 1);
    }
    for (int h = 0; h < 2; ++h) {
      mbar_init(&s_full[h], 1);
      mbar_init(&p_full[h], 4);
    }
    mbar_init(acc_done, 1);
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmDO);
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
  const float* lse_h = p.lse + (long long)head * p.ld_stat;
  const float* del_h = p.delta + (long long)head * p.ld_stat;

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------------ producer
      mbar_arrive_expect_tx(kv_full, 2 * G::TILE);
#pragma unroll
      for (int b = 0; b < G::BOXES; ++b) {
        tma_load_2d(sK + b * BOX_BYTES, &tmK, kv_full, head * HD + 64 * b, kv_row0 + (int)k0);
        tma_load_2d(sV + b * BOX_BYTES, &tmV, kv_full, head * HD + 64 * b, kv_row0 + (int)k0);
      }
      int last[STAGES] = {-1, -1};
      for (int idx = 0; idx < n_inner; ++idx) {
        const int st = idx % STAGES;
        const uint32_t ph = (uint32_t)((idx / STAGES) & 1);
        if (!mbar_wait(&in_empty[st], ph ^ 1u, wb, SITE_BWD_PRODUCER)) break;
        // the tile's rows in the micro-batch layout (contiguous: a 128-row tile never
        // spans two ranks' blocks when B > 1)
        const long long r0 = batch_row(row0_of(idx), seq, p);
        mbar_arrive_expect_tx(&in_full[st], 2 * G::TILE + 1024);
#pragma unroll
        for (int b = 0; b < G::BOXES; ++b) {
          tma_load_2d(sQ(st) + b * BOX_BYTES, &tmQ, &in_full[st], q_col0 + head * HD + 64 * b,
                      (int)r0);
          tma_load_2d(sDO(st) + b * BOX_BYTES, &tmDO, &in_full[st], do_col0 + head * HD + 64 * b,
                      (int)r0);
        }
        bulk_load(sLse(st), lse_h + r0, 512, &in_full[st]);
        bulk_load(sDel(st), del_h + r0, 512, &in_full[st]);
        last[st] = (int)ph;
      }
      WaitBound wd{p.status, p.limit_ns, nullptr};
      mbar_wait(kv_full, 0, wd, SITE_DRAIN);
      for (int s = 0; s < STAGES; ++s)
        if (last[s] >= 0) mbar_wait(&in_full[s], (uint32_t)last[s], wd, SITE_DRAIN);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ------------------------------------------------------------ MMA issuer
      const uint32_t idesc_s = make_idesc_bf16(BT, HALF, false);
      const uint32_t idesc_acc = make_idesc_bf16(BT, HD, true);
      const uint64_t dk0 = make_sdesc_sw128(smem_addr(sK), 16, 1024);
      const uint64_t dv0 = make_sdesc_sw128(smem_addr(sV), 16, 1024);
      const uint64_t dst0 = make_sdesc_sw128(smem_addr(sStage), 16, 1024);            // K-major
      const uint64_t dst0_mn = make_sdesc_sw128(smem_addr(sStage), BOX_BYTES, 1024);  // MN-major
      const uint32_t k_lo = (uint32_t)dk0, k_hi = (uint32_t)(dk0 >> 32);
      const uint32_t v_lo = (uint32_t)dv0, v_hi = (uint32_t)(dv0 >> 32);
      const uint32_t st_lo = (uint32_t)dst0, st_hi = (uint32_t)(dst0 >> 32);
      const uint32_t mn_lo = (uint32_t)dst0_mn, mn_hi = (uint32_t)(dst0_mn >> 32);
      // S^T_h = K Q_h^T and dP^T_h = V dO_h^T (64 query columns of stage st)
      auto issue_sdp = [&](int h, int st) {
        const uint32_t q_lo = st_lo + ((uint32_t)st * G::STAGE + (uint32_t)h * HALF_ROWS_BYTES) / 16;
        const uint32_t o_lo = q_lo + G::TILE / 16;
#pragma unroll
        for (int kk = 0; kk < HD / 16; ++kk)
          mma_ss_w(tmem + tm_sc(h), k_lo + kmajor_step(kk), k_hi, q_lo + kmajor_step(kk), st_hi,
                   idesc_s, kk > 0 ? 1u : 0u);
#pragma unroll
        for (int kk = 0; kk < HD / 16; ++kk)
          mma_ss_w(tmem + tm_dp(h), v_lo + kmajor_step(kk), v_hi, o_lo + kmajor_step(kk), st_hi,
                   idesc_s, kk > 0 ? 1u : 0u);
        mma_commit(&s_full[h]);
      };
      // dV += P^T_h dO_h, dK += dS^T_h Q_h (B MN-major: 16 query rows = 2048 B)
      auto issue_acc = [&](int h, int st, bool first) {
        const uint32_t q_lo = mn_lo + ((uint32_t)st * G::STAGE + (uint32_t)h * HALF_ROWS_BYTES) / 16;
        const uint32_t o_lo = q_lo + G::TILE / 16;
#pragma unroll
        for (int kk = 0; kk < HALF / 16; ++kk)
          mma_ts_w(tmem + 0, tmem + tm_sc(h) + (uint32_t)(kk * 8), o_lo + (uint32_t)(kk * 128),
                   mn_hi, idesc_acc, (first && kk == 0) ? 0u : 1u);
#pragma unroll
        for (int kk = 0; kk < HALF / 16; ++kk)
          mma_ts_w(tmem + HD, tmem + tm_dp(h) + (uint32_t)(kk * 8), q_lo + (uint32_t)(kk * 128),
                   mn_hi, idesc_acc, (first && kk == 0) ? 0u : 1u);
      };
      bool ok = mbar_wait(kv_full, 0, wb, SITE_BWD_MMA) && mbar_wait(&in_full[0], 0, wb, SITE_BWD_MMA);
      if (ok) {
        tc_fence_after();
        issue_sdp(0, 0);
        issue_sdp(1, 0);
      }
      for (int idx = 0; ok && idx < n_inner; ++idx) {
        const int st = idx % STAGES;
        for (int h = 0; h < 2; ++h) {
          if (!mbar_wait(&p_full[h], (uint32_t)(idx & 1), wb, SITE_BWD_MMA)) {
            ok = false;
            break;
          }
          tc_fence_after();
          issue_acc(h, st, idx == 0 && h == 0);
          if (h == 1) mma_commit(&in_empty[st]);
          if (idx + 1 < n_inner) {
            if (h == 0 && !mbar_wait(&in_full[(idx + 1) % STAGES],
                                     (uint32_t)(((idx + 1) / STAGES) & 1), wb, SITE_BWD_MMA)) {
              ok = false;
              break;
            }
            tc_fence_after();
            issue_sdp(h, (idx + 1) % STAGES);
          }
        }
      }
      if (ok) mma_commit(acc_done);
      mma_commit(drain);
      WaitBound wd{p.status, p.limit_ns, nullptr};
      mbar_wait(drain, 0, wd, SITE_DRAIN);
    }
  } else {
    // -------------------------------------------------------------- element-wise
    const int h = (warp - 2) >> 2;  // half of every streamed tile this warpgroup takes
    const int qq = warp & 3;        // TMEM lane quarter
    const int r_local = qq * 32 + lane;
    const long long kp = k0 + r_local;  // key position of this thread's row
    const uint32_t lane_base = tmem + ((uint32_t)(qq * 32) << 16);
    const uint32_t s_t = lane_base + tm_sc(h), d_t = lane_base + tm_dp(h);
    bool ok = true;
    auto warp_wait = [&](uint64_t* bar, uint32_t parity) {
      const bool mine = mbar_wait(bar, parity, wb, SITE_BWD_ELEMENTWISE);
      return __all_sync(0xffffffffu, mine) != 0;
    };
    for (int idx = 0; idx < n_inner; ++idx) {
      const int st = idx % STAGES;
      if (!warp_wait(&s_full[h], (uint32_t)(idx & 1)) ||
          !warp_wait(&in_full[st], (uint32_t)((idx / STAGES) & 1))) {
        ok = false;
        break;
      }
      tc_fence_after();
      // the half's 64 scores and 64 dP values of this key row: one TMEM round trip
      uint32_t s0[32], s1[32], g0[32], g1[32];
      tmem_ld32(s_t, s0);
      tmem_ld32(s_t + 32, s1);
      tmem_ld32(d_t, g0);
      tmem_ld32(d_t + 32, g1);
      const float4* sl4 = reinterpret_cast<const float4*>(sLse(st) + h * HALF);
      const float4* sd4 = reinterpret_cast<const float4*>(sDel(st) + h * HALF);
      const long long r0 = row0_of(idx);
      // natural tiles are contiguous positions; a tile needs masks only where it
      // meets the diagonal (or always, in the general zigzag layout)
      const long long qbase = p.natural ? (long long)(kt + idx) * IT + h * HALF : 0;
      const bool masked = !p.natural || qbase < k0 + BT - 1;
      tmem_ld_wait();
      uint32_t pp[32], dd[32];
      // P^T = exp2(s * scale_log2 - lse[q]), dS^T = P^T (dP^T - Delta[q]) for 32 columns
      auto chunk = [&](const uint32_t (&sv)[32], const uint32_t (&gv)[32], int c0, auto mask_tag) {
        constexpr bool MASK = decltype(mask_tag)::value;
#pragma unroll
        for (int e = 0; e < 32; e += 4) {
          const float4 l4 = sl4[(c0 + e) >> 2], d4 = sd4[(c0 + e) >> 2];
          const float lv[4] = {l4.x, l4.y, l4.z, l4.w};
          const float dl[4] = {d4.x, d4.y, d4.z, d4.w};
#pragma unroll
          for (int u = 0; u < 4; u += 2) {
            float p0 = ex2(fmaf(__uint_as_float(sv[e + u]), p.scale_log2, -lv[u]));
            float p1 = ex2(fmaf(__uint_as_float(sv[e + u + 1]), p.scale_log2, -lv[u + 1]));
            uint64_t ds = f2_mul(f2_pack(p0, p1),
                                 f2_sub(f2_pack(__uint_as_float(gv[e + u]), __uint_as_float(gv[e + u + 1])),
                                        f2_pack(dl[u], dl[u + 1])));
            if constexpr (MASK) {
              bool vis[2];
#pragma unroll
              for (int w = 0; w < 2; ++w) {
                const int col = h * HALF + c0 + e + u + w;
                if (p.natural) {
                  vis[w] = kp <= (long long)(kt + idx) * IT + col;
                } else {
                  const long long r = r0 + col;
                  vis[w] = r < p.S && kp <= row_pos(r, p.C, p.T, p.D);
                }
              }
              float d0, d1;
              f2_unpack(ds, d0, d1);
              p0 = vis[0] ? p0 : 0.f;
              p1 = vis[1] ? p1 : 0.f;
              ds = f2_pack(vis[0] ? d0 : 0.f, vis[1] ? d1 : 0.f);
            }
            float d0, d1;
            f2_unpack(ds, d0, d1);
            pp[(c0 + e + u) >> 1] = pack_bf16x2(p0, p1);
            dd[(c0 + e + u) >> 1] = pack_bf16x2(d0, d1);
          }
        }
      };
      if (masked) {
        chunk(s0, g0, 0, std::true_type{});
        chunk(s1, g1, 32, std::true_type{});
      } else {
        chunk(s0, g0, 0, std::false_type{});
        chunk(s1, g1, 32, std::false_type{});
      }
      tmem_st32(s_t, pp);
      tmem_st32(d_t, dd);
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&p_full[h]);
    }
    // ------------------------------------------------------------ epilogue
    if (ok && warp_wait(acc_done, 0u)) {
      tc_fence_after();
      const bool row_ok = kp < p.S;
      const long long orow = row_ok ? batch_row(zig_row(kp, p.C, p.T, p.D), seq, p) : 0;
      __nv_bfloat16* dvp = p.dv + orow * p.ld_dqkv + head * HD;
      __nv_bfloat16* dkp = p.dk + orow * p.ld_dqkv + head * HD;
#pragma unroll
      for (int c = h * (HD / 2); c < (h + 1) * (HD / 2); c += 32) {
        uint32_t a[32], b[32];
        tmem_ld32(lane_base + (uint32_t)c, a);
        tmem_ld32(lane_base + (uint32_t)(HD + c), b);
        tmem_ld_wait();
        if (row_ok) {
          uint4* v4 = reinterpret_cast<uint4*>(dvp + c);
          uint4* k4 = reinterpret_cast<uint4*>(dkp + c);
#pragma unroll
          for (int w = 0; w < 4; ++w) {
            uint4 x, y;
            x.x = pack_bf16x2(__uint_as_float(a[8 * w + 0]), __uint_as_float(a[8 * w + 1]));
            x.y = pack_bf16x2(__uint_as_float(a[8 * w + 2]), __uint_as_float(a[8 * w + 3]));
            x.z = pack_bf16x2(__uint_as_float(a[8 * w + 4]), __uint_as_float(a[8 * w + 5]));
            x.w = pack_bf16x2(__uint_as_float(a[8 * w + 6]), __uint_as_float(a[8 * w + 7]));
            y.x = pack_bf16x2(__uint_as_float(b[8 * w + 0]) * p.scale, __uint_as_float(b[8 * w + 1]) * p.scale);
            y.y = pack_bf16x2(__uint_as_float(b[8 * w + 2]) * p.scale, __uint_as_float(b[8 * w + 3]) * p.scale);
            y.z = pack_bf16x2(__uint_as_float(b[8 * w + 4]) * p.scale, __uint_as_float(b[8 * w + 5]) * p.scale);
            y.w = pack_bf16x2(__uint_as_float(b[8 * w + 6]) * p.scale, __uint_as_float(b[8 * w + 7]) * p.scale);
            v4[w] = x;
            k4[w] = y;
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

// ============================================================== query side
// The owned Q and dO rows are copied once into tensor memory and serve as the A
// operand of S = Q K^T and dP = dO V^T; only the streamed K/V tiles are read from
// shared memory by the tensor core.
template <int HD>
__global__ void __launch_bounds__(THREADS, 1)
    attention_bwd_dq_kernel(const __grid_constant__ CUtensorMap tmK,
                            const __grid_constant__ CUtensorMap tmV, const BwdParams p,
                            int q_col0, int do_col0) {
  using G = QueryGeom<HD>;
  constexpr int NS = G::KV_STAGES;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sStage = smem;  // stage s: K, V
  uint64_t* bars = reinterpret_cast<uint64_t*>(sStage + NS * G::STAGE);
  uint64_t* a_full = bars;                // [1] Q and dO rows stored in TMEM (8 warps)
  uint64_t* kv_full = a_full + 1;         // [NS]
  uint64_t* kv_empty = kv_full + NS;      // [NS]
  uint64_t* s_full = kv_empty + NS;       // [1] S(j) in TMEM
  uint64_t* dp_full = s_full + 1;         // [1] dP(j) in TMEM
  uint64_t* s_free = dp_full + 1;         // [1] S(j) read by the element-wise warps (8)
  uint64_t* ds_full = s_free + 1;         // [1] dS(j) stored (8 warps)
  uint64_t* acc_done = ds_full + 1;       // [1]
  uint64_t* drain = acc_done + 1;         // [1]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const CtaPos cp = cta_pos(p);
  const int head = cp.head, seq = cp.seq;
  const int blk = cp.tile;
  const int kv_row0 = (int)(seq * p.S);  // first natural K/V row of the sequence
  // natural: query tiles in decreasing position (longest first)
  const long long r0 = p.natural ? zig_row((long long)(p.n_outer - 1 - blk) * BT, p.C, p.T, p.D)
                                 : (long long)blk * BT;
  long long max_pos = 0;
  if (p.natural) {
    max_pos = row_pos(r0 + BT - 1, p.C, p.T, p.D);
  } else {
    const long long last = min(r0 + BT, p.S);
    for (long long r = r0; r < last; ++r) max_pos = max(max_pos, row_pos(r, p.C, p.T, p.D));
  }
  const int n_tiles = (int)(max_pos / IT) + 1;

  if (threadIdx.x == 0) {
    mbar_init(a_full, 8);
    for (int s = 0; s < NS; ++s) {
      mbar_init(&kv_full[s], 1);
      mbar_init(&kv_empty[s], 1);
    }
    mbar_init(s_full, 1);
    mbar_init(dp_full, 1);
    mbar_init(s_free, 8);
    mbar_init(ds_full, 8);
    mbar_init(acc_done, 1);
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
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
      // ------------------------------------------------------------ producer
      int last[NS];
#pragma unroll
      for (int s = 0; s < NS; ++s) last[s] = -1;
      for (int j = 0; j < n_tiles; ++j) {
        const int st = j % NS;
        const uint32_t ph = (uint32_t)((j / NS) & 1);
        if (!mbar_wait(&kv_empty[st], ph ^ 1u, wb, SITE_BWD_PRODUCER)) break;
        mbar_arrive_expect_tx(&kv_full[st], 2 * G::TILE);
        uint8_t* sk = sStage + st * G::STAGE;
#pragma unroll
        for (int b = 0; b < G::BOXES; ++b) {
          tma_load_2d(sk + b * BOX_BYTES, &tmK, &kv_full[st], head * HD + 64 * b, kv_row0 + j * IT);
          tma_load_2d(sk + G::TILE + b * BOX_BYTES, &tmV, &kv_full[st], head * HD + 64 * b,
                      kv_row0 + j * IT);
        }
        last[st] = (int)ph;
      }
      WaitBound wd{p.status, p.limit_ns, nullptr};
      for (int s = 0; s < NS; ++s)
        if (last[s] >= 0) mbar_wait(&kv_full[s], (uint32_t)last[s], wd, SITE_DRAIN);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ------------------------------------------------------------ MMA issuer
      const uint32_t idesc_s = make_idesc_bf16(BT, IT, false);
      const uint32_t idesc_acc = make_idesc_bf16(BT, HD, true);
      const uint64_t dst0 = make_sdesc_sw128(smem_addr(sStage), 16, 1024);
      const uint64_t dst0_mn = make_sdesc_sw128(smem_addr(sStage), BOX_BYTES, 1024);
      const uint32_t st_lo = (uint32_t)dst0, st_hi = (uint32_t)(dst0 >> 32);
      const uint32_t mn_lo = (uint32_t)dst0_mn, mn_hi = (uint32_t)(dst0_mn >> 32);
      // S = Q K^T (128 queries x 128 keys of stage st; A = Q in TMEM)
      auto issue_s = [&](int st) {
        const uint32_t k_lo = st_lo + (uint32_t)st * G::STAGE / 16;
#pragma unroll
        for (int kk = 0; kk < HD / 16; ++kk)
          mma_ts_w(tmem + TM_SC, tmem + G::TM_Q + (uint32_t)(kk * 8), k_lo + kmajor_step(kk),
                   st_hi, idesc_s, kk > 0 ? 1u : 0u);
        mma_commit(s_full);
      };
      // dP = dO V^T (A = dO in TMEM)
      auto issue_dp = [&](int st) {
        const uint32_t v_lo = st_lo + ((uint32_t)st * G::STAGE + G::TILE) / 16;
#pragma unroll
        for (int kk = 0; kk < HD / 16; ++kk)
          mma_ts_w(tmem + TM_DP, tmem + G::TM_DO + (uint32_t)(kk * 8), v_lo + kmajor_step(kk),
                   st_hi, idesc_s, kk > 0 ? 1u : 0u);
        mma_commit(dp_full);
      };
      // dQ += dS K (B MN-major: 16 key rows = 2048 B per K step)
      auto issue_dq = [&](int st, bool first) {
        const uint32_t k_lo = mn_lo + (uint32_t)st * G::STAGE / 16;
#pragma unroll
        for (int kk = 0; kk < IT / 16; ++kk)
          mma_ts_w(tmem + 0, packed_step(tmem + TM_DP, kk), k_lo + (uint32_t)(kk * 128), mn_hi,
                   idesc_acc, (first && kk == 0) ? 0u : 1u);
      };
      bool ok = mbar_wait(a_full, 0, wb, SITE_BWD_MMA) && mbar_wait(&kv_full[0], 0, wb, SITE_BWD_MMA);
      if (ok) {
        tc_fence_after();
        issue_s(0);
        issue_dp(0);
      }
      for (int j = 0; ok && j < n_tiles; ++j) {
        const int st = j % NS;
        const uint32_t ph = (uint32_t)(j & 1);
        if (j + 1 < n_tiles) {
          // next scores as soon as the element-wise warps hold this tile's
          if (!mbar_wait(&kv_full[(j + 1) % NS], (uint32_t)(((j + 1) / NS) & 1), wb, SITE_BWD_MMA) ||
              !mbar_wait(s_free, ph, wb, SITE_BWD_MMA)) {
            ok = false;
            break;
          }
          tc_fence_after();
          issue_s((j + 1) % NS);
        }
        if (!mbar_wait(ds_full, ph, wb, SITE_BWD_MMA)) {
          ok = false;
          break;
        }
        tc_fence_after();
        issue_dq(st, j == 0);
        mma_commit(&kv_empty[st]);
        if (j + 1 < n_tiles) issue_dp((j + 1) % NS);
      }
      if (ok) mma_commit(acc_done);
      mma_commit(drain);
      WaitBound wd{p.status, p.limit_ns, nullptr};
      mbar_wait(drain, 0, wd, SITE_DRAIN);
    }
  } else {
    // -------------------------------------------------------------- element-wise
    const int g = (warp - 2) >> 2;  // key half of every streamed tile this warpgroup takes
    const int qq = warp & 3;
    const int r_local = qq * 32 + lane;
    const long long vrow = r0 + r_local;  // row in the sequence's own layout
    const bool row_ok = vrow < p.S;
    const long long qpos = row_ok ? row_pos(vrow, p.C, p.T, p.D) : -1;
    const long long grow = batch_row(vrow, seq, p);  // row in the micro-batch's layout
    const float lse = row_ok ? p.lse[(long long)head * p.ld_stat + grow] : 0.f;
    const float del = row_ok ? p.delta[(long long)head * p.ld_stat + grow] : 0.f;
    const uint32_t lane_base = tmem + ((uint32_t)(qq * 32) << 16);
    const uint32_t s_t = lane_base + TM_SC + (uint32_t)(g * GCOLS);
    const uint32_t d_t = lane_base + TM_DP + (uint32_t)(g * GCOLS);
    {
      // this thread's row of Q (warpgroup 0) or dO (warpgroup 1) into TMEM, two
      // bf16 values per column, as the A operand of the score / dP products
      const __nv_bfloat16* src = g == 0 ? p.q + grow * p.ld_q + q_col0 + head * HD
                                        : p.dout + grow * p.ld_do + do_col0 + head * HD;
      const uint32_t dst = lane_base + (g == 0 ? G::TM_Q : G::TM_DO);
#pragma unroll
      for (int c = 0; c < HD / 2; c += 32) {
        uint32_t r[32];
        const uint4* s4 = reinterpret_cast<const uint4*>(src + 2 * c);
#pragma unroll
        for (int w = 0; w < 8; ++w) {
          const uint4 v = row_ok ? __ldg(s4 + w) : make_uint4(0u, 0u, 0u, 0u);
          r[4 * w + 0] = v.x;
          r[4 * w + 1] = v.y;
          r[4 * w + 2] = v.z;
          r[4 * w + 3] = v.w;
        }
        tmem_st32(dst + (uint32_t)c, r);
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(a_full);
    }
    bool ok = true;
    auto warp_wait = [&](uint64_t* bar, uint32_t parity) {
      const bool mine = mbar_wait(bar, parity, wb, SITE_BWD_ELEMENTWISE);
      return __all_sync(0xffffffffu, mine) != 0;
    };
    for (int j = 0; j < n_tiles; ++j) {
      const uint32_t ph = (uint32_t)(j & 1);
      if (!warp_wait(s_full, ph)) {
        ok = false;
        break;
      }
      tc_fence_after();
      // ---- phase a: P of this query row for the group's 64 key columns
      float pf[64];
      {
        uint32_t s0[32], s1[32];
        tmem_ld32(s_t, s0);
        tmem_ld32(s_t + 32, s1);
        tmem_ld_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(s_free);
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          pf[c] = ex2(fmaf(__uint_as_float(s0[c]), p.scale_log2, -lse));
          pf[32 + c] = ex2(fmaf(__uint_as_float(s1[c]), p.scale_log2, -lse));
        }
      }
      const long long kbase = (long long)j * IT + g * GCOLS;
      const bool masked = kbase + GCOLS - 1 > qpos;  // some key of the group is in the future
      if (masked) {
#pragma unroll
        for (int c = 0; c < 64; ++c) pf[c] = kbase + c <= qpos ? pf[c] : 0.f;
      }
      // ---- phase b: dS = P (dP - Delta)
      if (!warp_wait(dp_full, ph)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint64_t del2 = f2_pack(del, del);
      uint32_t dd[32];
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        uint32_t gv[32];
        tmem_ld32(d_t + (uint32_t)(32 * half), gv);
        tmem_ld_wait();
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
          const int c = 32 * half + e;
          float d0, d1;
          f2_unpack(f2_mul(f2_pack(pf[c], pf[c + 1]),
                           f2_sub(f2_pack(__uint_as_float(gv[e]), __uint_as_float(gv[e + 1])), del2)),
                    d0, d1);
          dd[c >> 1] = pack_bf16x2(d0, d1);
        }
      }
      tmem_st32(d_t, dd);
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(ds_full);
    }
    // ------------------------------------------------------------ epilogue
    if (ok && warp_wait(acc_done, 0u)) {
      tc_fence_after();
      __nv_bfloat16* dqp = p.dq + grow * p.ld_dqkv + head * HD;
#pragma unroll
      for (int c = g * (HD / 2); c < (g + 1) * (HD / 2); c += 32) {
        uint32_t a[32];
        tmem_ld32(lane_base + (uint32_t)c, a);
        tmem_ld_wait();
        if (row_ok) {
          uint4* q4 = reinterpret_cast<uint4*>(dqp + c);
#pragma unroll
          for (int w = 0; w < 4; ++w) {
            uint4 x;
            x.x = pack_bf16x2(__uint_as_float(a[8 * w + 0]) * p.scale, __uint_as_float(a[8 * w + 1]) * p.scale);
            x.y = pack_bf16x2(__uint_as_float(a[8 * w + 2]) * p.scale, __uint_as_float(a[8 * w + 3]) * p.scale);
            x.z = pack_bf16x2(__uint_as_float(a[8 * w + 4]) * p.scale, __uint_as_float(a[8 * w + 5]) * p.scale);
            x.w = pack_bf16x2(__uint_as_float(a[8 * w + 6]) * p.scale, __uint_as_float(a[8 * w + 7]) * p.scale);
            q4[w] = x;
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

// ============================================================== Delta
// One thread per (row, 8-column chunk); the chunks of a head are consecutive lanes,
// reduced with shuffles.
__global__ void attention_delta_kernel(const uint4* __restrict__ o, const uint4* __restrict__ dout,
                                       long long ld_vec, int heads, int d, long long S,
                                       float* __restrict__ delta, long long ld_stat) {
  const int cph = d / 8;  // chunks per head: 8 or 16, divides 32
  const long long per_row = (long long)heads * cph;
  const long long total = S * per_row;
  for (long long base = (long long)blockIdx.x * blockDim.x; base < total;
       base += (long long)gridDim.x * blockDim.x) {
    const long long i = base + threadIdx.x;
    float acc = 0.f;
    if (i < total) {
      const long long row = i / per_row, c = i - row * per_row;
      const uint4 a = o[row * ld_vec + c], b = dout[row * ld_vec + c];
      const uint32_t ua[4] = {a.x, a.y, a.z, a.w}, ub[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
      for (int w = 0; w < 4; ++w)
        acc += bf16_lo(ua[w]) * bf16_lo(ub[w]) + bf16_hi(ua[w]) * bf16_hi(ub[w]);
    }
    // total is a multiple of cph and blocks are multiples of 32 threads, so the
    // lanes of one head's chunks are all in range or all out of range
    for (int off = 1; off < cph; off <<= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (i < total && (i % cph) == 0) {
      const long long row = i / per_row, head = (i - row * per_row) / cph;
      delta[head * ld_stat + row] = acc;
    }
  }
}

template <int HD>
tsp_status launch_bwd_hd(const AttentionBwdCall& c, const BwdParams& p, cudaStream_t stream) {
  CUtensorMap tq, tdo, tk, tv;
  const uint64_t rows = (uint64_t)c.S * (uint64_t)p.B;
  TSP_TRY(make_tmap_2d_bf16(&tq, c.q, (uint64_t)c.ld_q, rows, (uint64_t)c.ld_q * 2, 64, 128));
  TSP_TRY(make_tmap_2d_bf16(&tdo, c.dout, (uint64_t)c.ld_do, rows, (uint64_t)c.ld_do * 2, 64, 128));
  TSP_TRY(make_tmap_2d_bf16(&tk, c.k, (uint64_t)c.ld_kv, rows, (uint64_t)c.ld_kv * 2, 64, 128));
  TSP_TRY(make_tmap_2d_bf16(&tv, c.v, (uint64_t)c.ld_kv, rows, (uint64_t)c.ld_kv * 2, 64, 128));
  const int tiles = (int)((c.S + 127) / 128);
  const unsigned ctas = (unsigned)((long long)tiles * c.heads * p.B);
  {
    auto kernel = attention_bwd_dkv_kernel<HD>;
    const size_t smem = KeyGeom<HD>::SMEM;
    TSP_TRY(ensure_smem_limit(reinterpret_cast<const void*>(kernel), (int)smem,
                              "attention bwd: cudaFuncSetAttribute"));
    cudaError_t e;
    BwdParams pk = p;
    pk.n_outer = tiles;
    kernel<<<ctas, THREADS, smem, stream>>>(tq, tdo, tk, tv, pk, 0, (int)c.do_col0);
    e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "attention bwd (key side): launch");
  }
  {
    auto kernel = attention_bwd_dq_kernel<HD>;
    const size_t smem = QueryGeom<HD>::SMEM;
    TSP_TRY(ensure_smem_limit(reinterpret_cast<const void*>(kernel), (int)smem,
                              "attention bwd: cudaFuncSetAttribute"));
    cudaError_t e;
    BwdParams pq = p;
    pq.n_outer = tiles;
    kernel<<<ctas, THREADS, smem, stream>>>(tk, tv, pq, 0, (int)c.do_col0);
    e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "attention bwd (query side): launch");
  }
  return TSP_OK;
}

}  // namespace

tsp_status launch_attention_bwd(const AttentionBwdCall& c, cudaStream_t stream) {
  if (c.d != 64 && c.d != 128) return fail(TSP_ERR_UNSUPPORTED, "attention bwd: head_dim 64 or 128");
  if (!c.q || !c.k || !c.v || !c.dout || !c.lse || !c.delta || !c.dq || !c.dk || !c.dv || !c.status)
    return fail(TSP_ERR_INVALID_ARG, "attention bwd: null pointer");
  if ((c.ld_q % 8) || (c.ld_kv % 8) || (c.ld_do % 8) || (c.do_col0 % 8) || (c.ld_dqkv % 8) ||
      (c.ld_stat % 128) || c.ld_stat < c.S * (c.B > 0 ? c.B : 1))
    return fail(TSP_ERR_INVALID_ARG, "attention bwd: bad strides");
  if ((reinterpret_cast<uintptr_t>(c.q) | reinterpret_cast<uintptr_t>(c.dout) |
       reinterpret_cast<uintptr_t>(c.lse) | reinterpret_cast<uintptr_t>(c.delta) |
       reinterpret_cast<uintptr_t>(c.dq) | reinterpret_cast<uintptr_t>(c.dk) |
       reinterpret_cast<uintptr_t>(c.dv)) & 15u)
    return fail(TSP_ERR_INVALID_ARG, "attention bwd: buffers must be 16-byte aligned");
  if ((long long)c.heads * c.d > c.ld_q || (long long)c.heads * c.d > c.ld_kv ||
      c.do_col0 + (long long)c.heads * c.d > c.ld_do || (long long)c.heads * c.d > c.ld_dqkv)
    return fail(TSP_ERR_INVALID_ARG, "attention bwd: head columns exceed the row width");
  const int B = c.B > 0 ? c.B : 1;
  if (c.S * B > (1ll << 30)) return fail(TSP_ERR_UNSUPPORTED, "attention bwd: too many rows");
  if (B > 1 && c.T % 128)
    return fail(TSP_ERR_UNSUPPORTED, "attention bwd: a micro-batch needs S/D % 128 == 0");
  BwdParams p{};
  p.dq = static_cast<__nv_bfloat16*>(c.dq);
  p.dk = static_cast<__nv_bfloat16*>(c.dk);
  p.dv = static_cast<__nv_bfloat16*>(c.dv);
  p.ld_dqkv = c.ld_dqkv;
  p.lse = c.lse;
  p.delta = c.delta;
  p.ld_stat = c.ld_stat;
  p.q = static_cast<const __nv_bfloat16*>(c.q);
  p.dout = static_cast<const __nv_bfloat16*>(c.dout);
  p.ld_q = c.ld_q;
  p.ld_do = c.ld_do;
  p.S = c.S;
  p.T = c.T;
  p.C = c.C;
  p.D = c.D;
  p.B = B;
  p.heads = c.heads;
  {
    // pairs per group: their K and V (2 * S * d bf16 each) within 48 MB of the L2,
    // the pairs split evenly over the fewest groups (no short last group, whose
    // longest blocks would start late)
    const long long fit0 = (48LL << 20) / (4LL * c.S * c.d);
    const long long fit = fit0 < 1 ? 1 : fit0;
    const long long pairs = (long long)c.heads * B;
    const long long n_groups = (pairs + fit - 1) / fit;
    p.group = (int)((pairs + n_groups - 1) / n_groups);
  }
  p.natural = (c.C % 128 == 0) ? 1 : 0;
  p.scale_log2 = 1.4426950408889634f / sqrtf((float)c.d);
  p.scale = 1.0f / sqrtf((float)c.d);
  p.status = c.status;
  p.limit_ns = wait_limit_ns();
  return c.d == 64 ? launch_bwd_hd<64>(c, p, stream) : launch_bwd_hd<128>(c, p, stream);
}

tsp_status launch_attention_delta(const void* o, const void* dout, int64_t ld, int heads, int d,
                                  int64_t S, float* delta, int64_t ld_stat, cudaStream_t stream) {
  if ((ld % 8) || (d != 64 && d != 128) || (long long)heads * d > ld)
    return fail(TSP_ERR_INVALID_ARG, "attention delta: bad shape");
  const long long total = S * heads * (d / 8);
  long long blocks = (total + 255) / 256;
  const long long cap = (long long)sm_count() * 8;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  attention_delta_kernel<<<(unsigned)blocks, 256, 0, stream>>>(
      static_cast<const uint4*>(o), static_cast<const uint4*>(dout), ld / 8, heads, d, S, delta,
      ld_stat);
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? TSP_OK : cuda_fail(e, "attention delta: launch");
}

}  // namespace tsp
