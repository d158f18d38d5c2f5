// Residency and ring sizing policy: host arithmetic behind the C ABI (no device work).
//
// "F5 M7 — Rolling KV: position-windowed KV residency", sections "Slot pool" (tile the
// link can move during one layer's attention, 0.8 safety, 2..4 slots) and "Auto-adapt
// loop" (a longer tail runs as several position sub-tiles); "T*-aware auto rolling-KV
// spill (HAL #582 P1+, #621 follow-on)", sections "T* — the negligible-drop tail band"
// and "The decision (fit-condition reformulation)".
#include <cmath>

#include "internal.h"

using namespace qps;

namespace {
bool positive(double x) { return std::isfinite(x) && x > 0.0; }
}  // namespace

extern "C" {

qps_status qps_plan_ring(double compute_ms_per_layer, double bw_eff_gbs, double slot_budget_bytes,
                         double per_layer_tail_bytes, int32_t* n_slots, int32_t* tiles_per_layer,
                         double* tile_bytes, double* tile_bytes_max) {
  if (!positive(compute_ms_per_layer) || !positive(bw_eff_gbs) || !positive(slot_budget_bytes))
    return fail(QPS_ERR_INVALID_ARG, "plan_ring: compute time, bandwidth and slot budget must be > 0");
  if (!std::isfinite(per_layer_tail_bytes) || per_layer_tail_bytes < 0.0)
    return fail(QPS_ERR_INVALID_ARG, "plan_ring: per_layer_tail_bytes must be >= 0");
  const double tmax = compute_ms_per_layer * 1e-3 * bw_eff_gbs * 1e9 * 0.8;
  const double slots = std::floor(slot_budget_bytes / tmax);
  const int32_t n = slots < 2.0 ? 2 : (slots > 4.0 ? 4 : (int32_t)slots);
  int32_t tiles = 0;
  double tb = 0.0;
  if (per_layer_tail_bytes > 0.0) {
    const double t = std::ceil(per_layer_tail_bytes / tmax);
    if (t > 2147483647.0) return fail(QPS_ERR_INVALID_ARG, "plan_ring: more than 2^31 tiles per layer");
    tiles = (int32_t)t;
    tb = std::ceil(per_layer_tail_bytes / tiles);
  }
  if (n_slots) *n_slots = n;
  if (tiles_per_layer) *tiles_per_layer = tiles;
  if (tile_bytes) *tile_bytes = tb;
  if (tile_bytes_max) *tile_bytes_max = tmax;
  return QPS_OK;
}

qps_status qps_tail_band(double t_resident_ms, double c_engage_ms, double bw_eff_gbs, double target_drop,
                         double* t_star_bytes) {
  if (!positive(t_resident_ms) || !positive(bw_eff_gbs))
    return fail(QPS_ERR_INVALID_ARG, "tail_band: t_resident_ms and bw_eff_gbs must be > 0");
  if (!std::isfinite(c_engage_ms) || c_engage_ms < 0.0)
    return fail(QPS_ERR_INVALID_ARG, "tail_band: c_engage_ms must be >= 0");
  if (!(target_drop > 0.0 && target_drop < 1.0))
    return fail(QPS_ERR_INVALID_ARG, "tail_band: target_drop must be in (0, 1)");
  if (!t_star_bytes) return fail(QPS_ERR_INVALID_ARG, "tail_band: t_star_bytes is NULL");
  const double t = (target_drop * t_resident_ms - c_engage_ms) * 1e-3 * bw_eff_gbs * 1e9;
  *t_star_bytes = t > 0.0 ? t : 0.0;
  return QPS_OK;
}

qps_status qps_choose_tier(const double* kv_bytes_per_tier, int32_t n_tiers, double budget_bytes,
                           double t_star_bytes, int32_t* tier) {
  if (!kv_bytes_per_tier || n_tiers < 1 || !tier)
    return fail(QPS_ERR_INVALID_ARG, "choose_tier: need >= 1 tier and an output");
  if (!std::isfinite(budget_bytes) || !std::isfinite(t_star_bytes) || t_star_bytes < 0.0)
    return fail(QPS_ERR_INVALID_ARG, "choose_tier: budget and T* must be finite, T* >= 0");
  for (int32_t i = 0; i < n_tiers; ++i) {
    if (kv_bytes_per_tier[i] <= budget_bytes + t_star_bytes) {
      *tier = i;
      return QPS_OK;
    }
  }
  *tier = n_tiers - 1;
  return QPS_OK;
}

}  // extern "C"
