// tg_tile_scheduler.cuh -- the persistent tile scheduler, one instance per warp role.
//
// "[Feature] Introduce tile scheduler #2441" replaces the hand-written
// ``for w in T.unroll(waves): tile_id = sm_num * w + block_id`` loop of
// gemm_tcgen5mma_ws_persistent.py with ``sched = T.PersistentTileScheduler(prefix, m_blocks,
// n_blocks, swizzle_size=group_size)``, ``sched.init(block_id)``, ``while sched.valid():``
// ... ``sched.next_tile()``.  Each role (TMA producer, MMA issuer, epilogue) owns one
// instance; the scheduler holds the only iteration clock: ``current_iter`` is the wave index
// w that drives the pipeline phase and the w & 1 accumulator choice, and ``m_idx``/``n_idx``
// are the tile coordinates.  Because every role's instance is built from the same
// arguments and advanced once per tile, all roles see the same (w, bx, by) sequence.
//
// Linear ids are grid-strided (worker c takes c, c + P, c + 2P, ...) and decoded in the
// grouped order of the page, bx = (t / g) % m_blocks, by = t % g + (t / g) / m_blocks * g,
// which walks panels of g N-tiles top to bottom for L2 reuse.  The page only meets full
// panels (it asserts n_blocks % (2 * group_size) == 0); here the last panel, when
// n_blocks % g != 0, is narrowed to its real width so the decode stays a bijection on
// [0, m_blocks * n_blocks).  With p = t / (m_blocks * g), width = min(g, n_blocks - p * g)
// and u = t - p * m_blocks * g, a tile is (u / width, p * g + u % width); on full panels
// this equals the page's formula term for term.
//
// Tail split (an addition to the page's scheduler): the workers step through *units*, not
// tiles.  Units 0 .. split_from - 1 are the tiles with the same ids; when the last partial
// wave would keep at most half of the workers busy, its tiles (ids split_from .. T - 1) are
// each cut into two half-width units (part 0 = left, part 1 = right half in N), numbered
// split_from + 2 (t - split_from) + part, so that wave takes half a tile's time.  Without a
// split, split_from = total_units = T and every unit is the page's tile (part = -1).
//
// column_major (the page's scheduler option of that name): panels of g M-tiles with ids running
// along M first -- the same decode with the roles of (m_blocks, bx) and (n_blocks, by) swapped.
//
// Stream-K tail (another addition; sk_tiles = R > 0, no half units then): the first
// total_units tiles are whole units on the grid stride as above; the R tiles after them (linear
// ids total_units .. total_units + R - 1, the last partial wave) are split along K.  Their
// k-blocks, numbered tile-major, go to the workers in contiguous ranges, worker c taking
// [floor(c R KB / P), floor((c + 1) R KB / P)); a range is shorter than KB, so it meets at most
// two tail tiles.  The worker whose range holds a tail tile's last k-block owns the tile (part
// 3): it adds the partial sums of the other workers meeting the tile (part 2 units, one at most
// per worker) to its own and stores it.  After its whole tiles a worker walks its contribution
// (the head of the later tile) before the tile it owns (the end of the earlier one), so an
// owner waits only for lower-numbered workers, whose contributions come first in their ranges.
// A tail segment's unit id is total_units + 2c + part - 2; k_lo .. k_hi are its k-blocks.
#pragma once

#include <cstdint>

namespace tg {

struct PersistentTileScheduler {
  uint32_t m_blocks, n_blocks, group, num_workers;
  uint32_t split_from;    // first unit id that is half a tile
  uint32_t total_units;   // units in the traversal
  uint32_t current_iter;  // w: units this worker has already taken
  uint32_t linear_idx;    // worker + w * num_workers
  uint32_t m_idx, n_idx;  // decoded tile (valid only while valid())
  int32_t part;           // -1 whole tile, 0 / 1 left / right half in N; 2 / 3 stream-K
                          // contribution / owned tile
  uint32_t column_major;  // 1: panels of g M-tiles, M fastest
  uint32_t k_blocks;      // k-blocks of a tile
  uint32_t k_lo, k_hi;    // k-blocks of the current unit
  uint32_t sk_tiles;      // R: tiles of the stream-K tail (0: none)
  uint32_t sk_tile;       // index of the current tail tile within the tail (part 2 / 3)
  uint32_t sk_state;      // 0: whole units; 1, 2: at tail segment 0, 1; 3: done
  uint32_t worker;
  uint64_t sk_lo, sk_hi;  // this worker's k-blocks of the tail (tile-major numbering)

  // the page's traversal: every unit a whole tile
  __host__ __device__ PersistentTileScheduler(uint32_t m, uint32_t n, uint32_t g, uint32_t p)
      : PersistentTileScheduler(m, n, g, p, m * n, m * n, 0) {}

  __host__ __device__ PersistentTileScheduler(uint32_t m, uint32_t n, uint32_t g, uint32_t p,
                                              uint32_t first_split, uint32_t units,
                                              uint32_t col_major, uint32_t kb = 0,
                                              uint32_t tail = 0)
      : m_blocks(m), n_blocks(n), group(g), num_workers(p), split_from(first_split),
        total_units(units), current_iter(0), linear_idx(0), m_idx(0), n_idx(0), part(-1),
        column_major(col_major), k_blocks(kb), k_lo(0), k_hi(kb), sk_tiles(tail), sk_tile(0),
        sk_state(0), worker(0), sk_lo(0), sk_hi(0) {}

  // worker c's k-blocks [lo, hi) of an R-tile stream-K tail (tile-major numbering)
  __host__ __device__ static void sk_range(uint32_t c, uint32_t workers, uint32_t tail,
                                           uint32_t kb, uint64_t& lo, uint64_t& hi) {
    const uint64_t total = static_cast<uint64_t>(tail) * kb;
    lo = total * c / workers;
    hi = total * (c + 1) / workers;
  }

  // (split_from, total_units) for T tiles over P workers: split the last partial wave when
  // it holds R tiles with 0 < 2R <= P.
  __host__ __device__ static void tail_split(uint32_t tiles, uint32_t workers,
                                             uint32_t& first_split, uint32_t& units) {
    const uint32_t rem = tiles % workers;
    if (rem == 0 || 2 * rem > workers) {
      first_split = units = tiles;
    } else {
      first_split = tiles - rem;
      units = first_split + 2 * rem;
    }
  }

  __host__ __device__ static void coord(uint32_t t, uint32_t m_blocks, uint32_t n_blocks,
                                        uint32_t group, uint32_t& bx, uint32_t& by) {
    const uint32_t panel_tiles = m_blocks * group;
    const uint32_t p = t / panel_tiles;
    const uint32_t first_col = p * group;
    const uint32_t left = n_blocks - first_col;
    const uint32_t width = left < group ? left : group;
    const uint32_t u = t - p * panel_tiles;
    bx = u / width;
    by = first_col + u % width;
  }

  __host__ __device__ void decode_tile(uint32_t t) {
    if (column_major)
      coord(t, n_blocks, m_blocks, group, n_idx, m_idx);
    else
      coord(t, m_blocks, n_blocks, group, m_idx, n_idx);
  }

  __host__ __device__ void decode() {
    if (linear_idx >= total_units) {
      if (sk_state == 0) sk_enter(0);
      return;
    }
    if (linear_idx < split_from) {
      decode_tile(linear_idx);
      part = -1;
    } else {
      const uint32_t v = linear_idx - split_from;
      decode_tile(split_from + v / 2);
      part = static_cast<int32_t>(v & 1u);
    }
  }

  // Moves to this worker's tail segment ``which`` (0: first, 1: second in walking order), or
  // past the end when it has none.
  __host__ __device__ void sk_enter(uint32_t which) {
    sk_state = 3;
    if (sk_tiles == 0 || sk_lo >= sk_hi) return;
    const uint64_t t0 = sk_lo / k_blocks, t1 = (sk_hi - 1) / k_blocks;
    uint64_t t;
    if (t1 > t0) {                         // the head of t1 (a contribution), then t0's end
      if (which == 0) {
        t = t1;
        k_lo = 0;
        k_hi = static_cast<uint32_t>(sk_hi - t1 * k_blocks);
        part = 2;
      } else if (which == 1) {
        t = t0;
        k_lo = static_cast<uint32_t>(sk_lo - t0 * k_blocks);
        k_hi = k_blocks;
        part = 3;
      } else {
        return;
      }
    } else {                               // one segment, owned iff it holds the last k-block
      if (which != 0) return;
      t = t0;
      k_lo = static_cast<uint32_t>(sk_lo - t0 * k_blocks);
      k_hi = static_cast<uint32_t>(sk_hi - t0 * k_blocks);
      part = k_hi == k_blocks ? 3 : 2;
    }
    sk_tile = static_cast<uint32_t>(t);
    decode_tile(total_units + sk_tile);
    linear_idx = total_units + 2u * worker + static_cast<uint32_t>(part - 2);
    sk_state = which + 1;
  }

  __host__ __device__ void init(uint32_t c) {
    current_iter = 0;
    worker = c;
    linear_idx = c;
    k_lo = 0;
    k_hi = k_blocks;
    sk_state = 0;
    if (sk_tiles) sk_range(c, num_workers, sk_tiles, k_blocks, sk_lo, sk_hi);
    decode();
  }

  // a half-width unit of the tail split (not a whole tile, not a stream-K segment)
  __host__ __device__ bool half_unit() const { return part == 0 || part == 1; }

  __host__ __device__ bool valid() const {
    return sk_state == 0 ? linear_idx < total_units : sk_state < 3;
  }

  __host__ __device__ void next_tile() {
    ++current_iter;
    if (sk_state == 0) {
      linear_idx += num_workers;
      decode();
    } else if (sk_state < 3) {
      sk_enter(sk_state);
    }
  }

  // dynamic persistence (no stream-K tail): the w-th unit of this worker is ``unit``
  __host__ __device__ void jump(uint32_t unit, uint32_t w) {
    current_iter = w;
    linear_idx = unit;
    decode();
  }

  // no further unit for this worker
  __host__ __device__ void finish() {
    linear_idx = total_units;
    sk_state = 3;
  }
};

}  // namespace tg
