// Host program for tests/test_partition_host.py: reads one query per line from argv[1] and
// writes one answer per line to argv[2], computed with the library's partition helpers
// (qe_partition.cuh, compiled for the host).
//   R Cu NW units w      -> x c k          (range_end)
//   Q i nq n             -> floor(i nq / n)
//   S i nq n cb cq       -> tile cost start
//   B loc n nbt          -> bf16 tile index
//   E r n Cu             -> first tile estimate
#include <cstdio>
#include "qe_partition.cuh"

int main(int argc, char** argv) {
  if (argc != 3) return 2;
  FILE* in = fopen(argv[1], "r");
  FILE* out = fopen(argv[2], "w");
  if (!in || !out) return 3;
  char op;
  while (fscanf(in, " %c", &op) == 1) {
    if (op == 'R') {
      long long Cu;
      int NW, units, w;
      if (fscanf(in, "%lld %d %d %d", &Cu, &NW, &units, &w) != 4) return 4;
      const qe::RangeEnd e = qe::range_end(Cu, NW, units, w);
      fprintf(out, "%lld %lld %d\n", e.x, e.c, e.k);
    } else if (op == 'Q') {
      int i, nq, n;
      if (fscanf(in, "%d %d %d", &i, &nq, &n) != 3) return 4;
      fprintf(out, "%d\n", qe::tiles_q_before(i, nq, n));
    } else if (op == 'S') {
      int i, nq, n, cb, cq;
      if (fscanf(in, "%d %d %d %d %d", &i, &nq, &n, &cb, &cq) != 5) return 4;
      fprintf(out, "%lld\n", qe::tile_cost_start(i, nq, n, cb, cq));
    } else if (op == 'B') {
      int loc, n, nbt;
      if (fscanf(in, "%d %d %d", &loc, &n, &nbt) != 3) return 4;
      fprintf(out, "%d\n", qe::bf16_tile_index(loc, n, nbt));
    } else if (op == 'E') {
      long long r, Cu;
      int n;
      if (fscanf(in, "%lld %d %lld", &r, &n, &Cu) != 3) return 4;
      fprintf(out, "%lld\n", qe::first_tile_estimate(r, n, Cu));
    } else {
      return 5;
    }
  }
  fclose(in);
  fclose(out);
  return 0;
}
