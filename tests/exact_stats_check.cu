// Host-side check of the exact row statistics (qe_exact_stats.cuh) that the five-tier rebuild
// kernel uses for the 1-bit tier: reads rows of float32 values and writes, per row, the fast
// path's mean and std (when the row fits its window) and the wide path's, so that a test can
// compare both with the oracle.  The per-lane partial sums of the kernel's warp are emulated
// lane by lane (they are integers, so their order does not matter).
//
//   exact_stats_check IN OUT     IN: int32 n, int32 D, float32 [n][D]
//                                OUT: per row int32 fast_used, float32 m_fast, s_fast, m_wide, s_wide
#include <cstdio>
#include <vector>

#include "qe_exact_stats.cuh"

using namespace qe::xs;

int main(int argc, char** argv) {
  if (argc != 3) return 2;
  FILE* f = fopen(argv[1], "rb");
  if (!f) return 3;
  int n = 0, D = 0;
  if (fread(&n, 4, 1, f) != 1 || fread(&D, 4, 1, f) != 1 || (D != 64 && D != 128)) return 4;
  std::vector<float> x((size_t)n * D);
  if (fread(x.data(), 4, x.size(), f) != x.size()) return 5;
  fclose(f);
  const int lgD = D == 128 ? 7 : 6;
  FILE* o = fopen(argv[2], "wb");
  if (!o) return 6;
  for (int r = 0; r < n; ++r) {
    const float* row = x.data() + (size_t)r * D;
    int E = 0;
    for (int c = 0; c < D; ++c) {
      const Parts p = parts(row[c]);
      if (p.mant && p.ee > E) E = p.ee;
    }
    int used = 1;
    float mf = 0.f, sf = 0.f;
    if (E > 0) {
      long long S = 0;
      u128 Q = 0;
      int bad = 0;
      for (int lane = 0; lane < 32; ++lane) {
        FastAcc a{0, 0, 0};
        for (int c = lane; c < D; c += 32) fast_add(a, row[c], E);
        S += a.s;
        Q += a.q;
        bad |= a.bad;
      }
      if (bad) used = 0;
      else fast_finish(S, Q, E, lgD, mf, sf);
    }
    WideAcc w;
    wide_zero(w);
    for (int c = 0; c < D; ++c) wide_acc(w, row[c]);
    float mw = 0.f, sw = 0.f;
    wide_finish(w, lgD, mw, sw);
    fwrite(&used, 4, 1, o);
    fwrite(&mf, 4, 1, o);
    fwrite(&sf, 4, 1, o);
    fwrite(&mw, 4, 1, o);
    fwrite(&sw, 4, 1, o);
  }
  fclose(o);
  return 0;
}
