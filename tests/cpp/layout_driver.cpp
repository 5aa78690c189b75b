// Test driver for include/ttc_layout.hpp: reads commands on stdin, prints
// results on stdout, one line per command.
//   eval <shape> <stride>                  -> the layout's values over its domain
//   crd <shape> <stride> <coord>           -> crd2idx of a hierarchical coordinate
//   compose <sA> <dA> <sB> <dB>            -> "<shape>:<stride> | values"
//   complement <shape> <stride> <m>        -> "<shape>:<stride>"
//   divide <sL> <dL> <sT> <dT>             -> "<shape>:<stride> | values"
//   product <sA> <dA> <sB> <dB>            -> "<shape>:<stride> | values"
//   stripmined <rows> <cols> <threads> <vec> -> "<shape>:<stride> | values"
//   swizzle <B> <off>                      -> Swizzle<B,4,3>(off)
//   zdivide|tdivide <sL> <dL> <t0> <t1>    -> zipped / tiled divide of a rank-2 layout by
//                                            the tilers t0:1, t1:1  ("<shape>:<stride> | values")
//   partition <sT> <dT> <sThr> <dThr> <i>  -> "<offset> | values" of local_partition
// Errors print "error <message>".
#include <iostream>
#include <sstream>
#include <string>

#include "ttc_layout.hpp"

using namespace ttc::layout;

static std::string values(const Layout& l) {
  std::string s;
  for (int64_t i = 0; i < l.size(); ++i) {
    if (i) s += " ";
    s += std::to_string(l(i));
  }
  return s;
}

int main() {
  std::string line;
  while (std::getline(std::cin, line)) {
    std::istringstream in(line);
    std::string cmd;
    in >> cmd;
    try {
      if (cmd == "eval") {
        std::string s, d;
        in >> s >> d;
        std::cout << values(Layout(parse_int_tuple(s), parse_int_tuple(d))) << "\n";
      } else if (cmd == "crd") {
        std::string s, d, c;
        in >> s >> d >> c;
        std::cout << Layout(parse_int_tuple(s), parse_int_tuple(d)).crd2idx(parse_int_tuple(c)) << "\n";
      } else if (cmd == "compose" || cmd == "divide" || cmd == "product") {
        std::string sa, da, sb, db;
        in >> sa >> da >> sb >> db;
        Layout a(parse_int_tuple(sa), parse_int_tuple(da)), b(parse_int_tuple(sb), parse_int_tuple(db));
        Layout r = cmd == "compose" ? composition(a, b) : cmd == "divide" ? logical_divide(a, b) : logical_product(a, b);
        std::cout << to_string(r) << " | " << values(r) << "\n";
      } else if (cmd == "complement") {
        std::string s, d;
        int64_t m;
        in >> s >> d >> m;
        std::cout << to_string(complement(Layout(parse_int_tuple(s), parse_int_tuple(d)), m)) << "\n";
      } else if (cmd == "stripmined") {
        int r, c, t, v;
        in >> r >> c >> t >> v;
        Layout l = stripmined_layout(StripMined{r, c, t, v});
        std::cout << to_string(l) << " | " << values(l) << "\n";
      } else if (cmd == "zdivide" || cmd == "tdivide") {
        std::string sl, dl;
        int64_t t0, t1;
        in >> sl >> dl >> t0 >> t1;
        Layout l(parse_int_tuple(sl), parse_int_tuple(dl));
        std::vector<Layout> tl{Layout(IntTuple(t0), IntTuple(1)), Layout(IntTuple(t1), IntTuple(1))};
        Layout r = cmd == "zdivide" ? zipped_divide(l, tl) : tiled_divide(l, tl);
        std::cout << to_string(r) << " | " << values(r) << "\n";
      } else if (cmd == "partition") {
        std::string st, dt, sh, dh;
        int64_t idx;
        in >> st >> dt >> sh >> dh >> idx;
        Partition pt = local_partition(Layout(parse_int_tuple(st), parse_int_tuple(dt)),
                                       Layout(parse_int_tuple(sh), parse_int_tuple(dh)), idx);
        std::string v;
        for (int64_t i = 0; i < pt.layout.size(); ++i) v += (i ? " " : "") + std::to_string(pt.offset + pt.layout(i));
        std::cout << pt.offset << " | " << v << "\n";
      } else if (cmd == "swizzle") {
        int b;
        uint32_t off;
        in >> b >> off;
        uint32_t y = b == 3 ? SwizzleBytes128{}(off) : b == 2 ? SwizzleBytes64{}(off) : SwizzleBytes32{}(off);
        std::cout << y << "\n";
      } else {
        std::cout << "error unknown command\n";
      }
    } catch (const std::exception& e) {
      std::cout << "error " << e.what() << "\n";
    }
  }
  return 0;
}
