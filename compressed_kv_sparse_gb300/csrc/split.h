// Host-side work split of the chunk scorer (no CUDA): the scorer's items are
// (sequence b, query group g, 128-row key tile), numbered
// (b * n_groups + g) * tiles_per + tile. A tile is visited when some row of it
// is visible to the group's last query; a chunk's later queries see more rows
// ("【#3】ds4.c を読み解く" §3: chunks keep absolute positions, so query t of a
// chunk at pos0 sees min((pos0 + t + 1) / ratio, n_comp) compressed rows).
// Splitting the items evenly over the CTAs therefore gives the last CTAs more
// visible tiles than the first; this split gives every CTA an even share of
// the visible tiles instead.
#pragma once

#include <algorithm>
#include <cstdint>
#include <vector>

namespace ds4a {

// Visible key tiles of query group g (queries g * qg .. min(T, (g + 1) qg) - 1)
// of a chunk of T queries at pos0 on a ratio-4 layer with n_comp rows, at most
// tiles_per.
inline uint32_t group_visible_tiles(uint32_t g, uint32_t T, uint32_t qg, uint32_t pos0,
                                    uint32_t n_comp, uint32_t tiles_per, uint32_t rows) {
  const uint32_t last = std::min(T, (g + 1) * qg) - 1;
  const uint32_t vis = std::min((pos0 + last + 1) / 4, n_comp);
  return std::min(tiles_per, (vis + rows - 1) / rows);
}

// Item ranges of `grid` CTAs: CTA j takes items start[j] .. start[j + 1] - 1
// (start has grid + 1 entries; start[grid] = batch * n_groups * tiles_per).
// Every sequence starts at pos0. CTA j's first item is the visible tile of
// rank floor(j V / grid) among the V visible tiles, so the CTAs' visible
// tiles differ by at most one.
inline void split_visible_tiles(uint32_t batch, uint32_t T, uint32_t qg, uint32_t pos0,
                                uint32_t n_comp, uint32_t rows, uint32_t n_groups,
                                uint32_t tiles_per, uint32_t grid, uint32_t *start) {
  std::vector<uint32_t> tg(n_groups);
  uint64_t vb = 0;
  for (uint32_t g = 0; g < n_groups; ++g) {
    tg[g] = group_visible_tiles(g, T, qg, pos0, n_comp, tiles_per, rows);
    vb += tg[g];
  }
  const uint64_t V = vb * batch;
  const uint32_t total = batch * n_groups * tiles_per;
  uint32_t j = 1;
  uint64_t cum = 0;
  start[0] = 0;
  for (uint32_t b = 0; b < batch && j < grid; ++b)
    for (uint32_t g = 0; g < n_groups && j < grid; ++g) {
      const uint32_t n = tg[g];
      while (j < grid && (uint64_t)j * V / grid < cum + n) {
        start[j] = (b * n_groups + g) * tiles_per + (uint32_t)((uint64_t)j * V / grid - cum);
        ++j;
      }
      cum += n;
    }
  for (; j <= grid; ++j) start[j] = total;
}

}  // namespace ds4a
