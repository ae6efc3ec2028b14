// Host program for tests/test_partition_host.py: the five-tier attention's 32-way unit search
// (search32_unit / search32_narrow from qe_tok.cuh) run on the host, the 32 lanes' tests done in
// a loop.  Input (argv[1]): lines "n x X(0) .. X(n-1)"; output (argv[2]): "u rounds" per line.
#include <cstdio>
#include <vector>
#include "qe_tok.cuh"

int main(int argc, char** argv) {
  if (argc != 3) return 2;
  FILE* in = fopen(argv[1], "r");
  FILE* out = fopen(argv[2], "w");
  if (!in || !out) return 3;
  int n;
  long long x;
  while (fscanf(in, "%d %lld", &n, &x) == 2) {
    std::vector<long long> X(n);
    for (int i = 0; i < n; ++i)
      if (fscanf(in, "%lld", &X[i]) != 1) return 4;
    int lo = 0, hi = n - 1, rounds = 0;
    while (hi > lo) {
      unsigned b = 1u;
      for (int lane = 0; lane < 32; ++lane)
        if (X[qe::search32_unit(lo, hi, lane)] <= x) b |= 1u << lane;
      int m = 31;
      while (!((b >> m) & 1u)) --m;
      qe::search32_narrow(lo, hi, m);
      if (++rounds > 64) return 5;
    }
    fprintf(out, "%d %d\n", lo, rounds);
  }
  fclose(in);
  fclose(out);
  return 0;
}
