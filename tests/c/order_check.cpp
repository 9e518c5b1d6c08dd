// Host check of the attention kernels' work order (chunked_order, compiled for the host): over
// every item index x of a launch, each (tile, head) pair comes out exactly once; tiles run in list
// order within a chunk of heads, and a full chunk's heads of one tile are consecutive items.
// Prints "ok" or the first failing case.
#include <cstdio>
#include <vector>

#include "pg_internal.h"

static int check(int n, int H, int hc) {
  std::vector<int> seen((size_t)n * H, 0);
  int prev_chunk = 0, prev_tile = -1;
  for (int x = 0; x < n * H; ++x) {
    int tile = -1, head = -1;
    pg::chunked_order(x, n, H, hc, tile, head);
    if (tile < 0 || tile >= n || head < 0 || head >= H) {
      printf("out of range: n=%d H=%d hc=%d x=%d -> tile %d head %d\n", n, H, hc, x, tile, head);
      return 1;
    }
    if (seen[(size_t)tile * H + head]++) {
      printf("repeated: n=%d H=%d hc=%d x=%d -> tile %d head %d\n", n, H, hc, x, tile, head);
      return 1;
    }
    const int chunk = head / hc;
    if (chunk < prev_chunk || (chunk == prev_chunk && tile < prev_tile)) {
      printf("order: n=%d H=%d hc=%d x=%d\n", n, H, hc, x);
      return 1;
    }
    if (chunk != prev_chunk) prev_tile = -1;
    prev_chunk = chunk;
    prev_tile = tile;
    if (head % hc != 0 && chunk < H / hc) {
      int t2, h2;
      pg::chunked_order(x - 1, n, H, hc, t2, h2);
      if (t2 != tile || h2 != head - 1) {
        printf("chunk layout: n=%d H=%d hc=%d x=%d\n", n, H, hc, x);
        return 1;
      }
    }
  }
  return 0;
}

int main() {
  int cases = 0;
  const int Hs[] = {1, 2, 8, 32, 40};
  for (int n = 1; n <= 60; n += 7)
    for (int H : Hs)
      for (int hc = 1; hc <= H; hc = hc * 2 + (hc == 1 ? 0 : 1)) {
        if (check(n, H, hc)) return 1;
        ++cases;
      }
  printf("ok %d\n", cases);
  return 0;
}
