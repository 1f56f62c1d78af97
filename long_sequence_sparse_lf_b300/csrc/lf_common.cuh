// Shared definitions of the CUDA path: work items, kernel parameters and the
// key-set predicates that both the attention kernel and the key-list
// enumerator use, so that the listed pairs are the pairs attended.
//
// Key set of query i in a head with dilation d, one-sided window w, length L
// and sorted global positions G (Longformer explained, §2: sliding window,
// dilated sliding window, global attention; §4: the patterns combined):
//   band(i) = { i + d*t : |t| <= w, 0 <= i + d*t < L }
//   K(i)    = [0, L) if i in G, else band(i) ∪ G.
// With r = i mod d and t = i div d ("residue space"), band(i) is the plain
// window [t-w, t+w] of the subsequence r, r+d, r+2d, ...
#pragma once

#include <cstdint>
#include <cuda.h>

namespace lf {

constexpr int kMaxDilSlots = 8;     // distinct dilation values per call
constexpr int kBM = 128;            // query rows per tile (MMA M)
constexpr int kBN = 128;            // keys per band block (MMA N)
// Zero padding on each side of a head's row of the bias table: a band
// block's column offsets kpos - t stay within +-(w + kBM + kBN - 2).
constexpr int kBiasPad = 256;
static_assert(kBiasPad >= kBM + kBN - 2, "bias padding too small");
// Length (floats, a multiple of 4) of one shifted copy of a head's padded
// bias row: 2w+1 values and kBiasPad zeros on each side.
__host__ __device__ __forceinline__ int bias_row_len(int w) {
  return (2 * w + 1 + 2 * kBiasPad + 3) & ~3;
}

enum : uint32_t { kStatusTimeout = 1u, kStatusBadItem = 2u };

// One try_wait suspends a waiting thread for at most this long; the host
// turns a timeout into a count of such slices.
constexpr uint32_t kWaitSliceNs = 1024;
__host__ __device__ constexpr uint32_t wait_iters_for(unsigned long long timeout_ns) {
  return (uint32_t)(timeout_ns / kWaitSliceNs) + 1u;
}

// One unit of work of the persistent attention kernel.  A CTA runs two
// 128-row query tiles side by side (tile slots X = 0 and X = 1) over one
// shared stream of 128-key blocks; each block names which slots use it.
//   kind 0 (band pair): slot X holds queries t0 + 128*X .. +127 of residue
//     class r of head bh (residue space, see above).  Block j < nkb holds keys
//     kb0 + 128*j .. +127 (residue space); slot X uses blocks jlo[X]..jhi[X]
//     (empty when jlo > jhi: the slot is absent) and, when present, the ngb
//     gathered global-key blocks j = nkb .. nkb+ngb-1.
//   kind 1 (global rows): both slots hold the gathered global queries
//     r*128 .. r*128+127 of head bh; block j < nkb holds absolute keys
//     kb0 + 128*j .. +127; slot 0 uses the even blocks, slot 1 the odd ones,
//     and slot X writes its partial (O, m, l) as key chunk 2*slot + X.
struct WorkItem {
  int bh;        // b*H + h
  int kind;      // 0: band pair; 1: global rows over a key chunk
  int r;         // band: residue (i mod d); global: gathered-row tile index
  int t0;        // band: first query of slot 0 in residue space
  int kb0;       // first key of block 0 (residue space / absolute position)
  int nkb;       // number of 128-key blocks
  int ngb;       // band: gathered global key blocks; global: 0
  int slot;      // band: dilation slot; global: chunk-pair index
  int jlo[2];    // band: first block used by each tile slot
  int jhi[2];    // band: last band block used by each tile slot (inclusive)
};

// Extra key blocks (the random / strided block patterns, built by the
// kernel instance with extra blocks): a band item may carry, after its band
// and gathered blocks, nx[0] blocks of slot 0 and then nx[1] blocks of slot
// 1, described by XBlock records xlist[xo ..] (xitem[item] = {xo, nx[0],
// nx[1], 0}).  Block j = nkb + ngb + n holds keys kpos0 .. kpos0+127 of the
// item's residue class (residue space); gm marks the columns that are global
// positions (their keys come from the gathered blocks).
struct __align__(16) XBlock {
  uint32_t gm[4];
  int kpos0;
  int pad_[3];
};

// The blocks one tile slot uses in an item, with the slot fixed (its range
// is taken out of the item once, so that walking it needs no indexing):
// band blocks jlo..jhi, the gathered blocks, then the slot's extra blocks
// xa .. xa+xn-1 (none unless given).
struct SlotBlocks {
  int kind, nkb, ngb, jlo, jhi, X, xa, xn;
  __host__ __device__ __forceinline__ SlotBlocks(int kind_, int nkb_, int ngb_, int jlo_, int jhi_,
                                                 int x)
      : kind(kind_), nkb(nkb_), ngb(ngb_), jlo(jlo_), jhi(jhi_), X(x), xa(nkb_ + ngb_), xn(0) {}
  __host__ __device__ __forceinline__ SlotBlocks(const WorkItem& wi, int x)
      : kind(wi.kind), nkb(wi.nkb), ngb(wi.ngb), jlo(x ? wi.jlo[1] : wi.jlo[0]),
        jhi(x ? wi.jhi[1] : wi.jhi[0]), X(x), xa(wi.nkb + wi.ngb), xn(0) {}
  __host__ __device__ __forceinline__ SlotBlocks(const WorkItem& wi, int x, int nx0, int nx1)
      : kind(wi.kind), nkb(wi.nkb), ngb(wi.ngb), jlo(x ? wi.jlo[1] : wi.jlo[0]),
        jhi(x ? wi.jhi[1] : wi.jhi[0]), X(x), xa(wi.nkb + wi.ngb + (x ? nx0 : 0)),
        xn(x ? nx1 : nx0) {}
  __host__ __device__ __forceinline__ int count() const {
    if (kind == 0) return jlo <= jhi ? jhi - jlo + 1 + ngb + xn : 0;
    return nkb > X ? (nkb - X + 1) / 2 : 0;
  }
  __host__ __device__ __forceinline__ int first() const {
    if (kind == 0) return jlo <= jhi ? jlo : -1;
    return nkb > X ? X : -1;
  }
  __host__ __device__ __forceinline__ int next(int j) const {
    if (kind == 0) {
      if (j < jhi) return j + 1;
      if (j < nkb) return ngb > 0 ? nkb : (xn > 0 ? xa : -1);
      if (j < nkb + ngb) return j + 1 < nkb + ngb ? j + 1 : (xn > 0 ? xa : -1);
      return j + 1 < xa + xn ? j + 1 : -1;
    }
    return j + 2 < nkb ? j + 2 : -1;
  }
  __host__ __device__ __forceinline__ bool uses(int j) const {
    if (kind == 0)
      return jlo <= jhi && ((j >= jlo && j <= jhi) || (j >= nkb && j < nkb + ngb) ||
                            (j >= xa && j < xa + xn));
    return j < nkb && (j & 1) == X;
  }
};

// Number of blocks of item `wi` that tile slot X uses (band and gathered
// global blocks; extra blocks are counted apart).
__host__ __device__ __forceinline__ int blk_count(const WorkItem& wi, int X) {
  if (wi.kind == 0) return wi.jlo[X] <= wi.jhi[X] ? wi.jhi[X] - wi.jlo[X] + 1 + wi.ngb : 0;
  return wi.nkb > X ? (wi.nkb - X + 1) / 2 : 0;
}

struct MainParams {
  CUtensorMap tmQ[kMaxDilSlots];   // 4-D views {D, d, L/d, B*H} per dilation slot
  CUtensorMap tmK[kMaxDilSlots];
  CUtensorMap tmV[kMaxDilSlots];
  CUtensorMap tmKp;                // 3-D plain views {D, L, B*H} (global rows)
  CUtensorMap tmVp;
  CUtensorMap tmQg;                // gathered rows {D, NGQ, B*H}, box 128 rows
  CUtensorMap tmKg;                // gathered rows, box NGB rows
  CUtensorMap tmVg;
  int dil[kMaxDilSlots];           // dilation value of each slot
  const WorkItem* items;           // grouped by CTA: CTA c runs items
  const int* cta_begin;            //   [cta_begin[c], cta_begin[c+1]) in order
  int n_items;
  const int32_t* gidx;             // [n_g] sorted global positions
  const uint8_t* is_glob;          // [L] 1 where the position is global
  const int32_t* gcnt;             // [L + 1] number of global positions below x
  int n_g;
  int NGB;                         // rows of one gathered global key block (16..128)
  int NGQ;                         // padded gathered rows per head (multiple of 128)
  int n_chunks;                    // key chunks per global-row tile
  void* out;                       // [B,H,L,D] bf16 or fp32
  int out_f32;
  float* part_o;                   // [(bh*NGQ + g)*n_chunks + c][D] fp32
  float* part_ml;                  // [(bh*NGQ + g)*n_chunks + c][2] (m, l)
  float* lse;                      // [B*H, L]: ln sum_{K(i)} exp(scale q.k), or null
  const int4* xitem;               // [n_items] {xo, nx0, nx1, 0} (extra-block kernel only)
  const XBlock* xlist;             // extra blocks of all items
  const float* rel_bias;           // [H, 4, bias_row_len(w)]: rel_bias/scale, zero-padded,
                                   // copy c shifted by c (the BIAS kernel only)
  int H, L, w;
  float sl2;                       // scale * log2(e)
  unsigned* status;                // device status word
  uint32_t wait_iters;             // bound on every wait, in try_wait slices
};

// ---------------------------------------------------------- predicates

// Residue-space window of query t, clipped to [0, Lr): keys [lo, hi].
__host__ __device__ __forceinline__ void band_window(int t, int w, int Lr, int& lo, int& hi) {
  lo = t - w < 0 ? 0 : t - w;
  hi = t + w > Lr - 1 ? Lr - 1 : t + w;
}

// j in band(i) for absolute positions (both inside [0, L)).
__host__ __device__ __forceinline__ bool in_band_abs(int i, int j, int d, int w) {
  int diff = j - i;
  int ad = diff < 0 ? -diff : diff;
  return ad <= d * w && (diff % d) == 0;
}

// Bits of the columns base .. base+31 that lie in [lo, hi) (bit c - base),
// without branches.
__host__ __device__ __forceinline__ uint32_t range_bits(int lo, int hi, int base) {
  int a = lo - base, b = hi - base;
  a = a < 0 ? 0 : (a > 32 ? 32 : a);
  b = b < 0 ? 0 : (b > 32 ? 32 : b);
  const uint32_t below_b = b >= 32 ? 0xffffffffu : ((1u << b) - 1u);
  const uint32_t below_a = a >= 32 ? 0xffffffffu : ((1u << a) - 1u);
  return below_b & ~below_a;
}

// 16-key chunks c (bit c, c = 0..7) of a 128-key block that overlap the
// columns [lo, hi] / that lie inside them.
__host__ __device__ __forceinline__ uint32_t chunk_overlap_bits(int lo, int hi) {
  if (hi < lo || hi < 0 || lo > 127) return 0u;
  const int a = lo < 0 ? 0 : lo >> 4;
  const int b = hi > 127 ? 7 : hi >> 4;
  return ((1u << (b + 1)) - 1u) & ~((1u << a) - 1u);
}
__host__ __device__ __forceinline__ uint32_t chunk_inside_bits(int lo, int hi) {
  const int a = lo <= 0 ? 0 : (lo + 15) >> 4;
  const int b = hi >= 127 ? 7 : ((hi + 1) >> 4) - 1;
  if (hi < lo || a > b || a > 7 || b < 0) return 0u;
  return ((1u << (b + 1)) - 1u) & ~((1u << a) - 1u);
}

// Number of positions p in [0, L) with p mod d == r.
__host__ __device__ __forceinline__ int residue_len(int L, int d, int r) {
  return r < L ? (L - 1 - r) / d + 1 : 0;
}

}  // namespace lf
