// Prints the GEMM launch plan (pair tiles, CTA pairs, leading tiles divided along K),
// the split-tail workspace size, the tiles run as halves and the rows a GEMM that
// quantizes its own activations leaves to the quantize kernel (the leading rows),
// for shapes read from standard input, one "m n k max_clusters workspace_bytes
// halves_ok" per line (workspace_bytes < 0: no workspace).
// Host code only: the plan is inline in the library's internal header.
#include <cstdio>

#include "internal.h"

int main() {
  long long m, n, k, ws;
  int clusters, halves;
  static unsigned char dummy[1];
  while (std::scanf("%lld %lld %lld %d %lld %d", &m, &n, &k, &clusters, &ws, &halves) == 6) {
    const mxk::GemmPlan p = mxk::plan_gemm(m, n, k, clusters, ws < 0 ? nullptr : dummy,
                                           ws < 0 ? 0 : static_cast<size_t>(ws), halves != 0);
    std::printf("%lld %d %d %zu %d %lld\n", static_cast<long long>(p.tiles), p.clusters, p.sk_tiles,
                mxk::split_workspace_bytes(m, n, k), p.half_tiles,
                static_cast<long long>(mxk::qa_lead_rows(m, n, clusters)));
  }
  return 0;
}
