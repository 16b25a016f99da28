// Host check of the decode kernels' CTA split (built by tests/test_cut_host.py
// with nvcc and linked against libpa for the rest of the library): for random
// batches, the kernel's per-CTA walk (cta_first_tile) and the host plan's
// one-pass walk (cta_cuts) must both give the brute-force cut -- CTA i starts
// at the smallest x whose cost of tiles [0, x) reaches floor(i * C(T) / G),
// a tile costing 1 and each segment's first tile w more -- and every range
// must hold a tile.  Prints the number of mismatches; exit status 1 if any.
#include <cstdio>
#include <cstdlib>
#include <vector>

#include "pa_decode.cu"

using namespace pa_split;

static long long brute_cut(const std::vector<int>& lens, int segs, int tk, long long T, int G, int w, int i) {
  if (w == 0) return (long long)i * T / G;
  std::vector<long long> starts;
  long long st = 0;
  for (int L : lens) {
    const long long n = (L + tk - 1) / tk;
    for (int g = 0; g < segs; ++g) {
      starts.push_back(st);
      st += n;
    }
  }
  const long long c = (long long)i * (T + (long long)w * (long long)starts.size()) / G;
  for (long long x = 0; x <= T; ++x) {
    long long below = 0;
    for (long long s0 : starts) below += s0 < x;
    if (x + w * below >= c) return x;
  }
  return -1;
}

int main(int argc, char** argv) {
  const int iters = argc > 1 ? atoi(argv[1]) : 2000;
  srand(12345);
  long long cases = 0, bad = 0;
  for (int it = 0; it < iters; ++it) {
    const int n = 1 + rand() % 12, segs = 1 + rand() % 4, tk = (rand() % 2) ? 64 : 16;
    int w = rand() % 4;
    std::vector<int> lens(n);
    for (auto& L : lens) L = 1 + rand() % ((rand() % 2) ? 300 : 3000);
    long long T = 0;
    for (int L : lens) T += (long long)((L + tk - 1) / tk) * segs;
    int G = 1 + rand() % 40;
    if (G > T) G = (int)T;
    if (w && T < (long long)G * (1 + w)) w = 0;
    Geometry geo{};
    geo.tile_keys = tk;
    geo.segs_per_seq = segs;
    const std::vector<long long> cut = cta_cuts(lens.data(), (uint32_t)n, geo, T, G, w);
    for (int i = 0; i <= G; ++i) {
      const long long d = cta_first_tile(lens.data(), n, segs, tk, T, G, w, i), b = brute_cut(lens, segs, tk, T, G, w, i);
      ++cases;
      if (d != b || cut[i] != b || (i > 0 && cut[i] <= cut[i - 1])) {
        if (bad < 5) printf("case %d, CTA %d: kernel %lld, host %lld, brute force %lld\n", it, i, d, cut[i], b);
        ++bad;
      }
    }
  }
  printf("cases %lld mismatches %lld\n", cases, bad);
  return bad != 0;
}
