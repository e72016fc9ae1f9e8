// Code-pair schedules of the fast GEMV path for 3- and 6-bit codes (plain C++,
// usable from host and device code).
//
// A lane's chunk of 32 b-bit codes is a stream of 32*b bits held in b words:
// code j occupies stream bits [j*b, j*b + b), stream bit i being bit i%32 of
// word i/32.  The fast path turns each code into the fp16 value 1024 + 2^o*q:
// a 32-bit "source" window of the stream starting at bit t is masked so that
// each 16-bit half keeps one code at bit offset o (o + b <= 10, inside the
// fp16 mantissa), and every half is ORed with 0x6400 (fp16 1024).  One LOP3
// makes two such values; a source costs one shift unless t is a multiple of
// 32.  Codes are summed into one accumulator per class, a class being one
// offset o (multiplier 2^o).
//
// The schedules were chosen by exhaustive search (an integer program over the
// sources, the code placements and the class sets) for the fewest shifts plus
// LOP3s: per 32 codes, 10 shifts + 16 LOP3s with 3 classes for b = 6, and
// 6 shifts + 18 LOP3s with 4 classes for b = 3.  With one FMA per code and
// the class merge that is 1.9 and 1.8 instructions per code.
#pragma once

#ifdef __CUDACC__
#define BT_HD __host__ __device__
#else
#define BT_HD
#endif

namespace bt {
namespace gemv {

struct StreamPair {
  int t;         // first stream bit of the source window
  int lo, olo;   // code in the low half (-1: none) and its bit offset in that half
  int hi, ohi;   // code in the high half (-1: none) and its bit offset in that half
};

template <int BITS> struct StreamLayout;

// 6-bit codes: offsets 0, 2, 4 (classes x1, x4, x16); every source carries a pair.
template <> struct StreamLayout<6> {
  static constexpr int n_pairs = 16;
  static constexpr int n_classes = 3;
  BT_HD static constexpr int cls(int o) { return o / 2; }
  BT_HD static constexpr int offset(int c) { return 2 * c; }
  BT_HD static constexpr StreamPair pair(int i) {
    constexpr StreamPair tab[n_pairs] = {
        {0, 0, 0, 3, 2},      {4, 1, 2, 4, 4},      {12, 2, 0, 5, 2},     {32, 6, 4, 8, 0},
        {42, 7, 0, 10, 2},    {52, 9, 2, 12, 4},    {64, 11, 2, 14, 4},   {74, 13, 4, 15, 0},
        {96, 16, 0, 19, 2},   {102, 17, 0, 20, 2},  {106, 18, 2, 21, 4},  {128, 22, 4, 24, 0},
        {134, 23, 4, 25, 0},  {152, 26, 4, 28, 0},  {160, 27, 2, 30, 4},  {170, 29, 4, 31, 0}};
    return tab[i];
  }
};

// 3-bit codes: offsets 0, 3, 4, 7 (classes x1, x8, x16, x128); the sources at
// bits 0 and 64 carry one code in each LOP3.
template <> struct StreamLayout<3> {
  static constexpr int n_pairs = 18;
  static constexpr int n_classes = 4;
  BT_HD static constexpr int cls(int o) { return o == 0 ? 0 : o == 3 ? 1 : o == 4 ? 2 : 3; }
  BT_HD static constexpr int offset(int c) { return c == 0 ? 0 : c == 1 ? 3 : c == 2 ? 4 : 7; }
  BT_HD static constexpr StreamPair pair(int i) {
    constexpr StreamPair tab[n_pairs] = {
        {0, 0, 0, -1, 0},     {0, 1, 3, -1, 0},     {2, 2, 4, 6, 0},      {2, 3, 7, 7, 3},
        {8, 4, 4, 8, 0},      {8, 5, 7, 9, 3},      {26, 10, 4, 14, 0},   {26, 11, 7, 15, 3},
        {32, 12, 4, 16, 0},   {32, 13, 7, 17, 3},   {50, 18, 4, 22, 0},   {50, 19, 7, 23, 3},
        {56, 20, 4, 24, 0},   {56, 21, 7, 25, 3},   {64, -1, 0, 28, 4},   {64, -1, 0, 29, 7},
        {74, 26, 4, 30, 0},   {74, 27, 7, 31, 3}};
    return tab[i];
  }
};

// The LOP3 mask of a pair: the low-half code's bits and the high-half code's bits.
template <int BITS>
BT_HD constexpr unsigned stream_mask(const StreamPair& p) {
  return (p.lo >= 0 ? (((1u << BITS) - 1u) << p.olo) : 0u) |
         (p.hi >= 0 ? (((1u << BITS) - 1u) << (16 + p.ohi)) : 0u);
}

}  // namespace gemv
}  // namespace bt
