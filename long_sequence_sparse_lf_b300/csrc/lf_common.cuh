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

enum : uint32_t { kStatusTimeout = 1u, kStatusBadItem = 2u };

// One unit of work of the persistent attention kernel.
struct WorkItem {
  int bh;        // b*H + h
  int kind;      // 0: band tile of a head; 1: global-row tile over a key chunk
  int r;         // band: residue (i mod d); global: global-row tile index
  int t0;        // band: first query of the tile in residue space
  int kb0;       // first key of the first key block (residue space for band,
                 // absolute position for global rows); may be negative
  int nkb;       // number of 128-key blocks
  int ngb;       // band: number of gathered global key blocks; global: 0
  int slot;      // band: dilation slot; global: key-chunk index
};

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
  const WorkItem* items;
  int n_items;
  const int32_t* gidx;             // [n_g] sorted global positions
  const uint8_t* is_glob;          // [L] 1 where the position is global
  int n_g;
  int NGB;                         // rows of one gathered global key block (16..128)
  int NGQ;                         // padded gathered rows per head (multiple of 128)
  int n_chunks;                    // key chunks per global-row tile
  void* out;                       // [B,H,L,D] bf16 or fp32
  int out_f32;
  float* part_o;                   // [(bh*NGQ + g)*n_chunks + c][D] fp32
  float* part_ml;                  // [(bh*NGQ + g)*n_chunks + c][2] (m, l)
  int H, L, w;
  float sl2;                       // scale * log2(e)
  unsigned* status;                // device status word
  unsigned long long timeout_ns;   // bound on every wait
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

// Number of positions p in [0, L) with p mod d == r.
__host__ __device__ __forceinline__ int residue_len(int L, int d, int r) {
  return r < L ? (L - 1 - r) / d + 1 : 0;
}

}  // namespace lf
