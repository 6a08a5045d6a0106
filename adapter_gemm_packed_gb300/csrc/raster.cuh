// Tile order of the CTA-pair base GEMMs (gemm_2sm.cu, gemm_2sm_w4.cu), chosen on the host: which
// 256x256 output tiles there are, which run as 256x128 halves, and in what raster the persistent
// grid visits them (decoded on the device by decode_pair / decode_item in pair.cuh).  Together with
// those two files this decides the GEMMs' DRAM traffic.
#pragma once

#include <algorithm>

#include "common.cuh"

namespace mlora {

// Work list of the CTA-pair base GEMMs: 256x256 tiles, except that when the last wave would fill at
// most half of the pairs its tiles are split into 256x128 halves, which finish that wave in half
// the time (and give small problems twice the pairs).  Returns the number of pairs to launch.
inline int pair_gemm_items(int n_mtiles, int num_sms, GemmArgs& g) {
  const int n_tiles = ((n_mtiles + 1) / 2) * g.n_tiles_n;
  const int pairs = std::max(1, num_sms / 2);
  const int tail = n_tiles <= pairs ? n_tiles : n_tiles % pairs;
  const bool split = tail > 0 && 2 * tail <= pairs;
  g.n_full_items = split ? n_tiles - tail : n_tiles;
  g.n_items = split ? n_tiles + tail : n_tiles;
  return std::max(1, std::min(g.n_items, pairs));
}

// L2 room for the resident panel of a CTA-pair base GEMM's raster (see decode_pair).
constexpr double RASTER_PANEL_BUDGET = 48.0 * (1 << 20);

// Order and group size of a CTA-pair base GEMM's raster over its m_pairs x n_tiles full tiles
// (K = the main product's reduction length).  Every 256-token pair reads a 256 x K panel of A and
// every output tile a 256 x K panel of B (bf16).  A group of g tiles along one dimension keeps
// its g panels in L2 while it sweeps the other dimension, so that dimension's panels are read
// from HBM once per group: DRAM bytes ~ (resident side, once) + (swept side) x (groups).  The
// resident panels must fit the L2 budget; groups are made equal.  Ties go to output-tile groups
// (the weight stays resident).
inline void set_raster(GemmArgs& g, int K) {
  const double panel = 256.0 * K * 2.0;
  const double budget = RASTER_PANEL_BUDGET;
  const long long m_pairs = (g.n_mtiles + 1) / 2, n_tiles = g.n_tiles_n;
  const long long gmax = std::max(1LL, static_cast<long long>(budget / panel));
  double best = 0.0;
  for (int by_n = 1; by_n >= 0; --by_n) {
    const long long res = by_n ? n_tiles : m_pairs, swept = by_n ? m_pairs : n_tiles;
    const long long groups = (res + std::min(res, gmax) - 1) / std::min(res, gmax);
    const long long gsz = (res + groups - 1) / groups;
    const double bytes = panel * (static_cast<double>(res) + static_cast<double>(swept) * groups);
    if (by_n == 1 || bytes < best) {
      best = bytes;
      g.raster_n = by_n;
      g.group_m = static_cast<int>(gsz);
    }
  }
}

}  // namespace mlora
