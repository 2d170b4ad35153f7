// Host harness: prints the strided gather's slot arithmetic from the
// library's own header, for a test that checks it against enumeration.
// Output lines: "y0 P r lp value" and "slots P r L value".
#include <cstdio>

#include "common.cuh"

int main() {
  const int parts[4] = {3, 5, 6, 7};
  for (int P : parts) {
    const int apg = ((mla::kPage + P - 1) / P + 7) / 8;
    for (int r = 0; r < P; ++r) {
      for (int lp = 0; lp < 3 * P; ++lp) std::printf("y0 %d %d %d %d\n", P, r, lp, mla::strided_y0(r, P, lp));
      for (int L = 0; L <= 700; ++L)
        std::printf("slots %d %d %d %d\n", P, r, L, mla::strided_slots(L, P, r, apg));
    }
  }
  return 0;
}
