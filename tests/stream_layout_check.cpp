// Host check of the 3- and 6-bit GEMV code-pair schedules (built and run by
// test_gemv_stream_layout.py; needs no GPU).  For each schedule it checks the
// structure (every code placed once, inside its half's mantissa, at the stream
// position it claims) and replays the fast path's arithmetic on random chunks:
// source window -> mask -> OR fp16 1024 -> fp16 decode -> per-class
// accumulation seeded with -1024*sum(x) -> merge by 2^-o, which must equal
// sum_j q_j*x_j from a bit-by-bit unpack, exactly (all values are small
// integers, so double arithmetic is exact).
#include <cmath>
#include <cstdint>
#include <cstdio>
#include <random>

#include "qgemv_stream.h"

using bt::gemv::StreamLayout;
using bt::gemv::StreamPair;

static int fails = 0;
#define CHECK(c, ...) do { if (!(c)) { ++fails; std::printf("FAIL: " __VA_ARGS__); std::printf("\n"); } } while (0)

// fp16 bit pattern -> value, field by field
static double half_value(uint32_t h) {
  const int s = (h >> 15) & 1, e = (h >> 10) & 31, m = h & 1023;
  double v = e == 0 ? std::ldexp(m, -24) : std::ldexp(1024 + m, e - 25);
  return s ? -v : v;
}

template <int BITS>
static uint32_t stream_bits(const uint32_t* w, int pos, int n) {   // n bits from stream bit pos
  uint32_t v = 0;
  for (int i = 0; i < n; ++i) {
    const int b = pos + i;
    v |= ((w[b / 32] >> (b % 32)) & 1u) << i;
  }
  return v;
}

template <int BITS>
static void check() {
  using L = StreamLayout<BITS>;
  int seen[32] = {0};
  for (int i = 0; i < L::n_pairs; ++i) {
    const StreamPair p = L::pair(i);
    CHECK(p.t >= 0 && p.t < 32 * BITS, "b=%d pair %d: source start %d", BITS, i, p.t);
    CHECK(p.lo >= 0 || p.hi >= 0, "b=%d pair %d: empty", BITS, i);
    for (int half = 0; half < 2; ++half) {
      const int j = half ? p.hi : p.lo, o = half ? p.ohi : p.olo;
      if (j < 0) continue;
      CHECK(j < 32, "b=%d pair %d: code %d", BITS, i, j);
      if (j >= 32) continue;
      ++seen[j];
      CHECK(o >= 0 && o + BITS <= 10, "b=%d code %d: offset %d leaves the mantissa", BITS, j, o);
      CHECK(L::offset(L::cls(o)) == o && L::cls(o) < L::n_classes, "b=%d code %d: class of offset %d", BITS, j, o);
      CHECK(j * BITS == p.t + 16 * half + o, "b=%d code %d: stream bit %d, placed at %d", BITS, j, j * BITS,
            p.t + 16 * half + o);
    }
  }
  for (int j = 0; j < 32; ++j) CHECK(seen[j] == 1, "b=%d code %d placed %d times", BITS, j, seen[j]);

  std::mt19937 rng(1234 + BITS);
  for (int trial = 0; trial < 20000; ++trial) {
    uint32_t w[BITS];
    for (int i = 0; i < BITS; ++i) w[i] = rng();
    if (trial == 0) for (int i = 0; i < BITS; ++i) w[i] = 0xFFFFFFFFu;   // every code at its maximum
    if (trial == 1) for (int i = 0; i < BITS; ++i) w[i] = 0u;
    double x[32];
    for (int j = 0; j < 32; ++j) x[j] = (int)(rng() % 17) - 8;
    double want = 0;
    for (int j = 0; j < 32; ++j) want += stream_bits<BITS>(w, j * BITS, BITS) * x[j];

    double acc[L::n_classes] = {};
    for (int i = 0; i < L::n_pairs; ++i) {   // seeds: minus 1024 * x of every code in the class
      const StreamPair p = L::pair(i);
      if (p.lo >= 0) acc[L::cls(p.olo)] -= 1024.0 * x[p.lo];
      if (p.hi >= 0) acc[L::cls(p.ohi)] -= 1024.0 * x[p.hi];
    }
    for (int i = 0; i < L::n_pairs; ++i) {
      const StreamPair p = L::pair(i);
      const int wi = p.t / 32, sh = p.t % 32;
      uint32_t src;
      if (sh == 0) src = w[wi];
      else if (wi + 1 < BITS) src = (uint32_t)((((uint64_t)w[wi + 1] << 32) | w[wi]) >> sh);   // funnel shift
      else src = w[wi] >> sh;
      const uint32_t h = (src & bt::gemv::stream_mask<BITS>(p)) | 0x64006400u;
      if (p.lo >= 0) acc[L::cls(p.olo)] += half_value(h & 0xFFFFu) * x[p.lo];
      if (p.hi >= 0) acc[L::cls(p.ohi)] += half_value(h >> 16) * x[p.hi];
    }
    double got = acc[0];
    for (int c = 1; c < L::n_classes; ++c) got += acc[c] / std::ldexp(1.0, L::offset(c));
    CHECK(got == want, "b=%d trial %d: schedule gives %.1f, unpack gives %.1f", BITS, trial, got, want);
    if (fails > 20) return;
  }
}

int main() {
  check<3>();
  check<6>();
  if (fails) { std::printf("%d failures\n", fails); return 1; }
  std::printf("ok\n");
  return 0;
}
