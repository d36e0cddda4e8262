// Host check of the device-side bounds checks' predicates (csrc/checks.h):
// every access the kernels make to C, a stream-K slot or a flag must pass,
// and an access one element outside -- before the block, in a row's pitch
// padding, past the last row, in the neighbouring slot, past the flags --
// must fail. Prints "ok" and exits 0, or names the first failing case.
#include <cstdio>
#include <cstdlib>

#include "checks.h"

using gemm14::c_span_ok;
using gemm14::index_ok;
using gemm14::slot_span_ok;

static int fails = 0;
static void expect(bool got, bool want, const char* what, long a, long b) {
  if (got != want) {
    std::printf("FAIL %s (%ld, %ld): got %d\n", what, a, b, got ? 1 : 0);
    ++fails;
  }
}

int main() {
  // C: M x N block, pitch ldc > N
  const long M = 7, N = 13, ldc = 16;
  for (long r = 0; r < M; ++r)
    for (long c = 0; c < ldc; ++c) {
      const long off = r * ldc + c;
      expect(c_span_ok(off, ldc, M, N, 1), c < N, "c_span width 1", r, c);
      expect(c_span_ok(off, ldc, M, N, 4), c + 4 <= N, "c_span width 4", r, c);
    }
  expect(c_span_ok(-1, ldc, M, N, 1), false, "before C", -1, 0);
  expect(c_span_ok(M * ldc, ldc, M, N, 1), false, "past the last row", M, 0);
  expect(c_span_ok((M - 1) * ldc + N - 1, ldc, M, N, 1), true, "last element", M - 1, N - 1);
  expect(c_span_ok(0, 0, M, N, 1), false, "zero pitch", 0, 0);
  expect(c_span_ok(0, ldc, M, ldc + 1, 1), false, "N above the pitch", 0, 0);
  expect(c_span_ok(0, ldc, M, N, 0), false, "zero width", 0, 0);
  // a 2^31-element C (offsets beyond int32)
  const long big_ld = 32768, big_m = 65600;
  expect(c_span_ok((big_m - 1) * big_ld + 100, big_ld, big_m, 32768, 4), true, "large C", big_m - 1, 100);
  expect(c_span_ok(big_m * big_ld, big_ld, big_m, 32768, 1), false, "large C past end", big_m, 0);

  // slots: 5 slots of 96 elements
  const long S = 96, n = 5;
  for (long s = 0; s < n; ++s) {
    expect(slot_span_ok(s * S, s, S, n, 32), true, "slot start", s, 0);
    expect(slot_span_ok(s * S + S - 32, s, S, n, 32), true, "slot end", s, S - 32);
    expect(slot_span_ok(s * S + S - 31, s, S, n, 32), false, "into the next slot", s, S - 31);
    expect(slot_span_ok(s * S - 1, s, S, n, 1), false, "into the slot before", s, -1);
  }
  expect(slot_span_ok(n * S, n, S, n, 1), false, "slot n", n, 0);
  expect(slot_span_ok(0, -1, S, n, 1), false, "slot -1", -1, 0);
  expect(slot_span_ok(0, 0, S, n, 0), false, "zero width", 0, 0);

  // flags
  expect(index_ok(0, 3), true, "flag 0", 0, 3);
  expect(index_ok(2, 3), true, "flag 2", 2, 3);
  expect(index_ok(3, 3), false, "flag 3", 3, 3);
  expect(index_ok(-1, 3), false, "flag -1", -1, 3);

  if (fails) return 1;
  std::printf("ok\n");
  return 0;
}
