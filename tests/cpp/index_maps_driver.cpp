// Test driver: reads one launch configuration per line
//   tile_m tile_n ctas a_rows a_mn b_mn esize swizzled half_cols
// and prints the index maps the host derives for it from the layout helper
// (tiled_tensor_core_02_gb300/csrc/index_maps.hpp), or "error <what>".
#include <iostream>
#include <sstream>
#include <string>

#include "index_maps.hpp"

static void box(const ttc::BoxMap& b) {
  std::cout << ' ' << b.k_inner << ' ' << b.box_inner << ' ' << b.box_outer << ' ' << b.boxes << ' ' << b.box_step
            << ' ' << b.smem_step;
}

int main() {
  std::string line;
  while (std::getline(std::cin, line)) {
    if (line.empty()) continue;
    std::istringstream in(line);
    int tm, tn, ctas, ar, amn, bmn, es, swz, half;
    in >> tm >> tn >> ctas >> ar >> amn >> bmn >> es >> swz >> half;
    try {
      const ttc::TileMaps m = ttc::maps::derive(tm, tn, ctas, ar, amn != 0, bmn != 0, es, swz != 0, half);
      std::cout << m.tile_m << ' ' << m.tile_n << ' ' << m.cta_m << ' ' << m.cta_n;
      box(m.a);
      box(m.b);
      std::cout << ' ' << m.half_n << ' ' << m.cta_n_half;
      box(m.b_half);
      std::cout << ' ' << m.epi_row_step << ' ' << m.tmem_row_step << ' ' << m.epi_chunk << '\n';
    } catch (const std::exception& e) {
      std::cout << "error " << e.what() << '\n';
    }
  }
  return 0;
}
