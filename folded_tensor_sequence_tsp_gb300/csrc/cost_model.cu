// cost_model.cu - per-device memory, communication and FLOPs of one layer under
// DP, TP, SP, TP+SP and TSP ("Folding Tensor and Sequence Parallelism for
// Memory-Efficient Transformer Training & Inference", section 3, theoretical
// analysis). The page states the comparison in words; the closed forms below are
// written from each scheme's sharding rules for the layer this library computes
// (causal attention with h heads + SwiGLU of width F, S tokens per sequence, a
// micro-batch of B sequences). Host code only: no CUDA call.
//
// Per token the layer keeps boundary activations x and h (2H elements) and inner
// activations q, k, v, o (4H) and a1, a3, g (3F). Weights: 4H^2 + 3HF elements.
// Communication counts what one device receives in one forward of the layer, with
// ring collectives: all-reduce of n elements over g devices = 2 (g-1)/g n received,
// all-gather of n = (g-1)/g n, broadcast of a shard = the shard (non-owners).
// A micro-batch ([TSP] s4: TSP's smaller footprint admits larger micro-batches)
// multiplies every activation term, the activation traffic and the FLOPs by B; the
// weights, and the weight traffic of TSP, serve the whole micro-batch once.
#include <cmath>
#include <cstdint>

#include "tsp.h"
#include "tsp_internal.h"

namespace {

double layer_flops(double S, double H, double F) {
  return 8.0 * S * H * H + 6.0 * S * H * F + 2.0 * H * S * (S + 1.0);
}

}  // namespace

extern "C" tsp_status tsp_cost_model_batched(int scheme, int D, int tp, int64_t S, int batch,
                                             int hidden, int heads, int ffn, tsp_cost* out) {
  using tsp::fail;
  if (!out) return fail(TSP_ERR_INVALID_ARG, "tsp_cost_model: out is NULL");
  if (batch < 1) return fail(TSP_ERR_INVALID_ARG, "tsp_cost_model: batch must be >= 1");
  if (D < 1 || S < 1 || hidden < 1 || heads < 1 || ffn < 1 || hidden % heads)
    return fail(TSP_ERR_INVALID_ARG, "tsp_cost_model: bad layer shape");
  const double s = (double)S, H = hidden, F = ffn, Dd = D;
  const double P = 4.0 * H * H + 3.0 * H * F;  // weight elements of the layer
  const double Ab = 2.0 * H, Ai = 4.0 * H + 3.0 * F;
  const double fl = layer_flops(s, H, F);
  tsp_cost c{};
  switch (scheme) {
    case TSP_SCHEME_DP:  // the whole layer on one device
      c.devices = 1;
      c.weight_elems = P;
      c.act_elems = s * (Ab + Ai);
      c.flops = fl;
      break;
    case TSP_SCHEME_TP:  // weights by heads / ffn columns; x, h replicated
      if (heads % D || ffn % D) return fail(TSP_ERR_UNSUPPORTED, "tsp_cost_model: TP needs heads % D == 0 and ffn % D == 0");
      c.devices = D;
      c.weight_elems = P / Dd;
      c.act_elems = s * Ab + s * Ai / Dd;
      c.comm_act_elems = 2.0 * (2.0 * (Dd - 1.0) / Dd * s * H);  // attention and MLP outputs
      c.flops = fl / Dd;
      break;
    case TSP_SCHEME_SP:  // tokens split, weights replicated, K/V all-gathered
      if (S % D) return fail(TSP_ERR_UNSUPPORTED, "tsp_cost_model: SP needs S % D == 0");
      c.devices = D;
      c.weight_elems = P;
      c.act_elems = s * (Ab + Ai) / Dd;
      c.act_inflight_elems = 2.0 * s * H;
      c.comm_act_elems = (Dd - 1.0) / Dd * 2.0 * s * H;
      c.flops = fl / Dd;
      break;
    case TSP_SCHEME_TP_SP: {  // T x (D/T) grid
      if (tp < 1 || D % tp) return fail(TSP_ERR_INVALID_ARG, "tsp_cost_model: TP+SP needs D % tp == 0");
      const int sg = D / tp;
      if (heads % tp || ffn % tp || S % sg)
        return fail(TSP_ERR_UNSUPPORTED, "tsp_cost_model: TP+SP needs heads % tp, ffn % tp and S % (D/tp) == 0");
      const double T = tp, Sg = sg;
      c.devices = D;
      c.weight_elems = P / T;
      c.act_elems = s * Ab / Sg + s * Ai / Dd;
      c.act_inflight_elems = 2.0 * s * H / T;
      c.comm_act_elems = 2.0 * (2.0 * (T - 1.0) / T * s * H / Sg) + (Sg - 1.0) / Sg * 2.0 * s * H / T;
      c.flops = fl / Dd;
      break;
    }
    case TSP_SCHEME_TSP:  // weights and tokens over the same D devices
      if (heads % D || ffn % D || S % D)
        return fail(TSP_ERR_UNSUPPORTED, "tsp_cost_model: TSP needs heads, ffn and S divisible by D");
      c.devices = D;
      c.weight_elems = P / Dd;
      // a received shard is held while it is used: one attention shard (4H^2/D)
      // during the broadcast iterations, one MLP shard (3HF/D) during the ring steps
      c.weight_inflight_elems = D > 1 ? (4.0 * H * H > 3.0 * H * F ? 4.0 * H * H : 3.0 * H * F) / Dd : 0.0;
      c.act_elems = s * (Ab + Ai) / Dd;
      c.act_inflight_elems = 2.0 * s * H / Dd;  // one head group's full K/V
      c.comm_weight_elems = (Dd - 1.0) / Dd * P;
      c.comm_act_elems = (Dd - 1.0) / Dd * 2.0 * s * H;
      c.flops = fl / Dd;
      break;
    default:
      return fail(TSP_ERR_INVALID_ARG, "tsp_cost_model: unknown scheme");
  }
  const double b = batch;
  c.act_elems *= b;
  c.act_inflight_elems *= b;
  c.comm_act_elems *= b;
  c.flops *= b;
  *out = c;
  return TSP_OK;
}

extern "C" tsp_status tsp_cost_model(int scheme, int D, int tp, int64_t S, int hidden, int heads,
                                     int ffn, tsp_cost* out) {
  return tsp_cost_model_batched(scheme, D, tp, S, 1, hidden, heads, ffn, out);
}

extern "C" tsp_status tsp_cost_max_batch(int scheme, int D, int tp, int64_t S, int hidden,
                                         int heads, int ffn, int layers, double mem_bytes,
                                         int64_t* out) {
  using tsp::fail;
  if (!out) return fail(TSP_ERR_INVALID_ARG, "tsp_cost_max_batch: out is NULL");
  if (layers < 1 || !(mem_bytes >= 0.0) || !std::isfinite(mem_bytes))
    return fail(TSP_ERR_INVALID_ARG, "tsp_cost_max_batch: layers >= 1 and a finite mem_bytes >= 0");
  tsp_cost one;
  tsp_status st = tsp_cost_model_batched(scheme, D, tp, S, 1, hidden, heads, ffn, &one);
  if (st != TSP_OK) return st;
  // bytes(B) = 2 (L (W + B A) + W_inflight + B A_inflight): every layer keeps its
  // weights and activations, one layer's received buffers exist at a time
  const double L = layers;
  const double fixed = 2.0 * (L * one.weight_elems + one.weight_inflight_elems);
  const double per_seq = 2.0 * (L * one.act_elems + one.act_inflight_elems);
  auto fits = [&](double bb) { return fixed + bb * per_seq <= mem_bytes; };
  double bmax = 0.0;
  if (fits(1.0)) {
    bmax = std::floor((mem_bytes - fixed) / per_seq);
    while (bmax > 1.0 && !fits(bmax)) bmax -= 1.0;  // guard the rounding of the division
    while (fits(bmax + 1.0)) bmax += 1.0;
  }
  *out = (int64_t)bmax;
  return TSP_OK;
}
