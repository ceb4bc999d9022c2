// Host build of the kernels' tile scheduler (tg_tile_scheduler.cuh, compiled with the CUDA
// qualifiers defined away) for the CPU tests: prints every unit of every worker as
// "worker w bx by part k_lo k_hi unit", one per line.
// usage: scheduler_driver m_blocks n_blocks workers group k_blocks column_major split_tail sk_tiles
#include <cstdio>
#include <cstdlib>

#include "tg_tile_scheduler.cuh"

int main(int argc, char** argv) {
  if (argc != 9) return 2;
  const uint32_t m = std::atoi(argv[1]), n = std::atoi(argv[2]), P = std::atoi(argv[3]);
  const uint32_t g = std::atoi(argv[4]), kb = std::atoi(argv[5]), col = std::atoi(argv[6]);
  const uint32_t split = std::atoi(argv[7]), tail = std::atoi(argv[8]);
  const uint32_t tiles = m * n - tail;
  uint32_t first = tiles, units = tiles;
  if (split) tg::PersistentTileScheduler::tail_split(tiles, P, first, units);
  for (uint32_t c = 0; c < P; ++c) {
    tg::PersistentTileScheduler s(m, n, g, P, first, units, col, kb, tail);
    for (s.init(c); s.valid(); s.next_tile())
      std::printf("%u %u %u %u %d %u %u %u\n", c, s.current_iter, s.m_idx, s.n_idx, s.part,
                  s.k_lo, s.k_hi, s.linear_idx);
  }
  return 0;
}
