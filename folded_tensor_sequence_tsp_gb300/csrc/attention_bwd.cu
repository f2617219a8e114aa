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
// Both sides run every product on a full 128-wide tile (N = 128 or N = d): a
// tcgen05.mma with M = 128 and K = 16 occupies the tensor pipe for about as long
// with N = 64 as with N = 128 on this part, so a narrower product runs at half
// rate. Each side's element-wise work is split into two phases that depend on
// different products, and the MMA lane orders its work so that one phase runs
// under the products of the other.
// Query side (S(j+1), dQ(j), dP(j+1), ...):
//   phase a  (after the scores, which it then releases): P = exp2(s scale_log2 - lse);
//   phase b  (after dP):  dS = P (dP - Delta), stored as bf16 over dP.
// Key side (dV(j), S^T(j+1), dK(j), dP^T(j+1), ...): two 128-column regions swap
// roles from tile to tile. Tile j's scores land in one; its element-wise warps
// turn them into P^T (bf16, kept in fp32 registers too) in place, then load dP^T(j)
// from the other region, which the MMA lane refills with S^T(j+1) at once, and
// store dS^T(j) beside P^T(j). dV(j) and dK(j) read P^T(j) and dS^T(j) as the A
// operand; dP^T(j+1) then overwrites tile j's region (products execute in issue
// order). The exponentials of tile j+1 run under dV(j), dK(j) and dP^T(j+1), and
// dS^T under S^T(j+1).
// Warps 2..5 and 6..9 (two warpgroups, one accumulator row per thread) take
// columns [0, 64) and [64, 128) of every streamed tile.
//   warp 0  TMA producer (key side: 3 stages of Q and lse, 2 of dO and Delta;
//           query side: 3 stages of K, V)
//   warp 1  TMEM allocation (512 columns) and the single MMA-issuing lane
// TMEM columns: key side: dV [0, d), dK [d, 2d), the two regions [256, 384) and
// [384, 512), warpgroup g's bf16 P^T over [64g, +32) of the scores' region and its
// dS^T over [64g + 32, +32). Query side: dQ [0, d), bf16 Q [d, 3d/2), bf16 dO
// [3d/2, 2d), scores [256, 384), dP [384, 512) with bf16 dS over [384 + 64g, +32)
// for warpgroup g.
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
// key side: two 128-column regions at 256 and 384 that swap roles from one streamed
// tile to the next: tile j's scores (then its packed P^T and dS^T) in tm_s(j), its
// dP^T in tm_g(j) = tm_s(j + 1)
__device__ __forceinline__ uint32_t tm_s(int j) { return (j & 1) ? 384u : 256u; }
__device__ __forceinline__ uint32_t tm_g(int j) { return (j & 1) ? 256u : 384u; }

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
  // Q tiles (with lse) and dO tiles (with Delta) in separate rings: a Q tile is read
  // last by dK, a full tile after its scores, so it gets the deeper ring
  static constexpr int QS = 3;
  static constexpr int OS = 2;
  // lse [QS][128], Delta [OS][128] and the barriers first; K, V, the Q ring and the
  // dO ring from the next 1024-byte boundary
  static constexpr uint32_t SMALL = (QS + OS) * 512 + 256;
  static constexpr uint32_t TILES_OFF = (SMALL + 1023) / 1024 * 1024;
  static constexpr size_t USED = TILES_OFF + (size_t)(2 + QS + OS) * TILE;
  // all 512 TMEM columns: one CTA per SM
  static constexpr size_t SMEM = USED > 120 * 1024 ? USED : 120 * 1024;
};
static_assert(KeyGeom<128>::USED <= 227 * 1024, "key-side shared memory");

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
  // no alignment is assumed for the base: the tiles start at the first 1024-byte
  // boundary after the small buffers, and the check below tests that they fit
  extern __shared__ uint8_t smem_raw[];
  float* sLse = reinterpret_cast<float*>(smem_raw);  // [QS][128]
  float* sDel = sLse + G::QS * 128;                  // [OS][128]
  uint64_t* bars = reinterpret_cast<uint64_t*>(sDel + G::OS * 128);
  uint64_t* kv_full = bars;              // [1]
  uint64_t* q_full = kv_full + 1;        // [QS]
  uint64_t* q_empty = q_full + G::QS;    // [QS]
  uint64_t* o_full = q_empty + G::QS;    // [OS]
  uint64_t* o_empty = o_full + G::OS;    // [OS]
  uint64_t* s_full = o_empty + G::OS;    // scores of the current tile written
  uint64_t* g_full = s_full + 1;         // dP^T of the current tile written
  uint64_t* p_ready = g_full + 1;        // packed P^T stored (8 warps)
  uint64_t* g_taken = p_ready + 1;       // dP^T loaded into registers (8 warps)
  uint64_t* ds_ready = g_taken + 1;      // packed dS^T stored (8 warps)
  uint64_t* acc_done = ds_ready + 1;
  uint64_t* drain = acc_done + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  // the tiles start at the first 1024-byte boundary after the small buffers
  const uint32_t base = smem_addr(smem_raw);
  const uint32_t tiles_off = ((base + G::SMALL + 1023u) & ~1023u) - base;
  if (tiles_off > G::TILES_OFF) {  // the allocation has no room for this base (uniform)
    if (threadIdx.x == 0) record_error(p.status, kStatusUnsupported, SITE_SMEM_LAYOUT);
    return;
  }
  uint8_t* sK = smem_raw + tiles_off;
  uint8_t* sV = sK + G::TILE;
  uint8_t* sQ0 = sV + G::TILE;               // [QS] Q tiles
  uint8_t* sO0 = sQ0 + G::QS * G::TILE;      // [OS] dO tiles

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
    for (int s = 0; s < G::QS; ++s) {
      mbar_init(&q_full[s], 1);
      mbar_init(&q_empty[s], 1);
    }
    for (int s = 0; s < G::OS; ++s) {
      mbar_init(&o_full[s], 1);
      mbar_init(&o_empty[s], 1);
    }
    mbar_init(s_full, 1);
    mbar_init(g_full, 1);
    mbar_init(p_ready, 8);
    mbar_init(g_taken, 8);
    mbar_init(ds_ready, 8);
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
      int q_last[G::QS], o_last[G::OS];
      for (int s = 0; s < G::QS; ++s) q_last[s] = -1;
      for (int s = 0; s < G::OS; ++s) o_last[s] = -1;
      for (int idx = 0; idx < n_inner; ++idx) {
        // the tile's rows in the micro-batch layout (contiguous: a 128-row tile never
        // spans two ranks' blocks when B > 1)
        const long long r0 = batch_row(row0_of(idx), seq, p);
        const int qs = idx % G::QS, os = idx % G::OS;
        const uint32_t qph = (uint32_t)((idx / G::QS) & 1), oph = (uint32_t)((idx / G::OS) & 1);
        if (!mbar_wait(&q_empty[qs], qph ^ 1u, wb, SITE_BWD_PRODUCER)) break;
        mbar_arrive_expect_tx(&q_full[qs], G::TILE + 512);
#pragma unroll
        for (int b = 0; b < G::BOXES; ++b)
          tma_load_2d(sQ0 + qs * G::TILE + b * BOX_BYTES, &tmQ, &q_full[qs],
                      q_col0 + head * HD + 64 * b, (int)r0);
        bulk_load(sLse + qs * 128, lse_h + r0, 512, &q_full[qs]);
        q_last[qs] = (int)qph;
        if (!mbar_wait(&o_empty[os], oph ^ 1u, wb, SITE_BWD_PRODUCER)) break;
        mbar_arrive_expect_tx(&o_full[os], G::TILE + 512);
#pragma unroll
        for (int b = 0; b < G::BOXES; ++b)
          tma_load_2d(sO0 + os * G::TILE + b * BOX_BYTES, &tmDO, &o_full[os],
                      do_col0 + head * HD + 64 * b, (int)r0);
        bulk_load(sDel + os * 128, del_h + r0, 512, &o_full[os]);
        o_last[os] = (int)oph;
      }
      WaitBound wd{p.status, p.limit_ns, nullptr};
      mbar_wait(kv_full, 0, wd, SITE_DRAIN);
      for (int s = 0; s < G::QS; ++s)
        if (q_last[s] >= 0) mbar_wait(&q_full[s], (uint32_t)q_last[s], wd, SITE_DRAIN);
      for (int s = 0; s < G::OS; ++s)
        if (o_last[s] >= 0) mbar_wait(&o_full[s], (uint32_t)o_last[s], wd, SITE_DRAIN);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ------------------------------------------------------------ MMA issuer
      const uint32_t idesc_s = make_idesc_bf16(BT, IT, false);
      const uint32_t idesc_acc = make_idesc_bf16(BT, HD, true);
      const uint64_t dk0 = make_sdesc_sw128(smem_addr(sK), 16, 1024);
      const uint64_t dv0 = make_sdesc_sw128(smem_addr(sV), 16, 1024);
      const uint64_t dq0 = make_sdesc_sw128(smem_addr(sQ0), 16, 1024);            // K-major
      const uint64_t dq0_mn = make_sdesc_sw128(smem_addr(sQ0), BOX_BYTES, 1024);  // MN-major
      const uint64_t do0 = make_sdesc_sw128(smem_addr(sO0), 16, 1024);
      const uint64_t do0_mn = make_sdesc_sw128(smem_addr(sO0), BOX_BYTES, 1024);
      const uint32_t k_lo = (uint32_t)dk0, k_hi = (uint32_t)(dk0 >> 32);
      const uint32_t v_lo = (uint32_t)dv0, v_hi = (uint32_t)(dv0 >> 32);
      const uint32_t kq_hi = (uint32_t)(dq0 >> 32), mn_hi = (uint32_t)(dq0_mn >> 32);
      // S^T(j) = K Q(j)^T and dP^T(j) = V dO(j)^T, one full-width product each
      auto issue_s = [&](int j) {
        const uint32_t q_lo = (uint32_t)dq0 + (uint32_t)(j % G::QS) * (G::TILE / 16);
#pragma unroll
        for (int kk = 0; kk < HD / 16; ++kk)
          mma_ss_w(tmem + tm_s(j), k_lo + kmajor_step(kk), k_hi, q_lo + kmajor_step(kk), kq_hi,
                   idesc_s, kk > 0 ? 1u : 0u);
        mma_commit(s_full);
      };
      auto issue_g = [&](int j) {
        const uint32_t o_lo = (uint32_t)do0 + (uint32_t)(j % G::OS) * (G::TILE / 16);
#pragma unroll
        for (int kk = 0; kk < HD / 16; ++kk)
          mma_ss_w(tmem + tm_g(j), v_lo + kmajor_step(kk), v_hi, o_lo + kmajor_step(kk), kq_hi,
                   idesc_s, kk > 0 ? 1u : 0u);
        mma_commit(g_full);
      };
      // dV += P^T(j) dO(j) and dK += dS^T(j) Q(j): A from tensor memory, B MN-major
      // (16 query rows = 2048 B per K step)
      auto issue_dv = [&](int j) {
        const uint32_t o_lo = (uint32_t)do0_mn + (uint32_t)(j % G::OS) * (G::TILE / 16);
#pragma unroll
        for (int kk = 0; kk < IT / 16; ++kk)
          mma_ts_w(tmem + 0, tmem + packed_step(tm_s(j), kk), o_lo + (uint32_t)(kk * 128), mn_hi,
                   idesc_acc, (j == 0 && kk == 0) ? 0u : 1u);
      };
      auto issue_dk = [&](int j) {
        const uint32_t q_lo = (uint32_t)dq0_mn + (uint32_t)(j % G::QS) * (G::TILE / 16);
#pragma unroll
        for (int kk = 0; kk < IT / 16; ++kk)
          mma_ts_w(tmem + HD, tmem + packed_step(tm_s(j) + 32, kk), q_lo + (uint32_t)(kk * 128),
                   mn_hi, idesc_acc, (j == 0 && kk == 0) ? 0u : 1u);
      };
      auto wait = [&](uint64_t* bar, uint32_t parity) {
        return mbar_wait_poll(bar, parity, wb, SITE_BWD_MMA);
      };
      bool ok = wait(kv_full, 0) && wait(&q_full[0], 0);
      if (ok) {
        tc_fence_after();
        issue_s(0);
      }
      ok = ok && wait(&o_full[0], 0);
      if (ok) {
        tc_fence_after();
        issue_g(0);
      }
      // per tile j: dV(j) once P^T(j) is stored; S^T(j+1) into the dP^T(j) region once
      // the element-wise warps hold dP^T(j); dK(j) once dS^T(j) is stored; dP^T(j+1)
      // into the region of tile j, after dV(j) and dK(j) have read it (in issue order)
      for (int j = 0; ok && j < n_inner; ++j) {
        const uint32_t ph = (uint32_t)(j & 1);
        const bool more = j + 1 < n_inner;
        if (!wait(p_ready, ph)) break;
        tc_fence_after();
        issue_dv(j);
        if (more) {
          if (!wait(g_taken, ph) ||
              !wait(&q_full[(j + 1) % G::QS], (uint32_t)(((j + 1) / G::QS) & 1))) {
            ok = false;
            break;
          }
          tc_fence_after();
          issue_s(j + 1);
        }
        if (!wait(ds_ready, ph)) {
          ok = false;
          break;
        }
        tc_fence_after();
        issue_dk(j);
        mma_commit(&q_empty[j % G::QS]);
        mma_commit(&o_empty[j % G::OS]);
        if (more) {
          if (!wait(&o_full[(j + 1) % G::OS], (uint32_t)(((j + 1) / G::OS) & 1))) {
            ok = false;
            break;
          }
          tc_fence_after();
          issue_g(j + 1);
        }
      }
      if (ok) mma_commit(acc_done);
      mma_commit(drain);
      WaitBound wd{p.status, p.limit_ns, nullptr};
      mbar_wait(drain, 0, wd, SITE_DRAIN);
    }
  } else {
    // -------------------------------------------------------------- element-wise
    const int g = (warp - 2) >> 2;  // query columns [64g, 64g + 64) of every tile
    const int qq = warp & 3;        // TMEM lane quarter
    const int r_local = qq * 32 + lane;
    const long long kp = k0 + r_local;  // key position of this thread's row
    const uint32_t lane_base = tmem + ((uint32_t)(qq * 32) << 16);
    const uint64_t scale2 = f2_pack(p.scale_log2, p.scale_log2);
    bool ok = true;
    auto warp_wait = [&](uint64_t* bar, uint32_t parity) {
      const bool mine = mbar_wait(bar, parity, wb, SITE_BWD_ELEMENTWISE);
      return __all_sync(0xffffffffu, mine) != 0;
    };
    for (int j = 0; j < n_inner; ++j) {
      const uint32_t ph = (uint32_t)(j & 1);
      const int qs = j % G::QS, os = j % G::OS;
      if (!warp_wait(s_full, ph) || !warp_wait(&q_full[qs], (uint32_t)((j / G::QS) & 1))) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t s_t = lane_base + tm_s(j) + (uint32_t)(GCOLS * g);
      const uint32_t g_t = lane_base + tm_g(j) + (uint32_t)(GCOLS * g);
      uint32_t sv[2][32];
      tmem_ld32(s_t, sv[0]);
      tmem_ld32(s_t + 32, sv[1]);
      const float4* sl4 = reinterpret_cast<const float4*>(sLse + qs * 128 + g * GCOLS);
      const long long r0 = row0_of(j);
      // natural tiles are contiguous positions; a tile needs masks only where it
      // meets the diagonal (or always, in the general zigzag layout)
      const long long qbase = p.natural ? (long long)(kt + j) * IT + g * GCOLS : 0;
      const bool masked = !p.natural || qbase < k0 + BT - 1;
      tmem_ld_wait();
      // P^T = exp2(s * scale_log2 - lse[q]), kept in fp32 for dS^T and stored as bf16
      float pf[64];
      uint32_t pp[32];
      auto p_chunk = [&](const uint32_t (&s)[32], int c0, auto mask_tag) {
        constexpr bool MASK = decltype(mask_tag)::value;
#pragma unroll
        for (int e = 0; e < 32; e += 4) {
          const float4 l4 = sl4[(c0 + e) >> 2];
          const uint64_t nl[2] = {f2_pack(-l4.x, -l4.y), f2_pack(-l4.z, -l4.w)};
#pragma unroll
          for (int u = 0; u < 4; u += 2) {
            float x0, x1;
            f2_unpack(f2_fma(f2_pack(__uint_as_float(s[e + u]), __uint_as_float(s[e + u + 1])),
                             scale2, nl[u >> 1]),
                      x0, x1);
            float p0 = ex2(x0), p1 = ex2(x1);
            if constexpr (MASK) {
              bool vis[2];
#pragma unroll
              for (int w = 0; w < 2; ++w) {
                const int col = g * GCOLS + c0 + e + u + w;
                if (p.natural) {
                  vis[w] = kp <= (long long)(kt + j) * IT + col;
                } else {
                  const long long r = r0 + col;
                  vis[w] = r < p.S && kp <= row_pos(r, p.C, p.T, p.D);
                }
              }
              p0 = vis[0] ? p0 : 0.f;
              p1 = vis[1] ? p1 : 0.f;
            }
            pf[c0 + e + u] = p0;
            pf[c0 + e + u + 1] = p1;
            pp[(c0 + e + u) >> 1] = pack_bf16x2(p0, p1);
          }
        }
      };
      if (masked) {
        p_chunk(sv[0], 0, std::true_type{});
        p_chunk(sv[1], 32, std::true_type{});
      } else {
        p_chunk(sv[0], 0, std::false_type{});
        p_chunk(sv[1], 32, std::false_type{});
      }
      tmem_st32(s_t, pp);
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(p_ready);
      if (!warp_wait(g_full, ph) || !warp_wait(&o_full[os], (uint32_t)((j / G::OS) & 1))) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t gv[2][32];
      tmem_ld32(g_t, gv[0]);
      tmem_ld32(g_t + 32, gv[1]);
      tmem_ld_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(g_taken);
      // dS^T = P^T (dP^T - Delta[q]) (zero where P^T is masked to zero)
      const float4* sd4 = reinterpret_cast<const float4*>(sDel + os * 128 + g * GCOLS);
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        uint32_t dd[16];
#pragma unroll
        for (int e = 0; e < 32; e += 4) {
          const float4 d4 = sd4[(32 * c + e) >> 2];
          const uint64_t dl[2] = {f2_pack(d4.x, d4.y), f2_pack(d4.z, d4.w)};
#pragma unroll
          for (int u = 0; u < 4; u += 2) {
            float d0, d1;
            f2_unpack(f2_mul(f2_pack(pf[32 * c + e + u], pf[32 * c + e + u + 1]),
                             f2_sub(f2_pack(__uint_as_float(gv[c][e + u]),
                                            __uint_as_float(gv[c][e + u + 1])),
                                    dl[u >> 1])),
                      d0, d1);
            dd[(e + u) >> 1] = pack_bf16x2(d0, d1);
          }
        }
        tmem_st16(s_t + 32 + 16 * c, dd);
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(ds_ready);
    }
    // ------------------------------------------------------------ epilogue
    if (ok && warp_wait(acc_done, 0u)) {
      tc_fence_after();
      const bool row_ok = kp < p.S;
      const long long orow = row_ok ? batch_row(zig_row(kp, p.C, p.T, p.D), seq, p) : 0;
      __nv_bfloat16* dvp = p.dv + orow * p.ld_dqkv + head * HD;
      __nv_bfloat16* dkp = p.dk + orow * p.ld_dqkv + head * HD;
#pragma unroll
      for (int c = g * (HD / 2); c < (g + 1) * (HD / 2); c += 32) {
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
