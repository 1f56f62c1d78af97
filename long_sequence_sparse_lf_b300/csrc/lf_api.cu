// C ABI of the Longformer sparse attention library: argument validation,
// per-shape plans (work lists, global-position tables), tensor-map setup and
// the launch sequence
//     [cast f32->bf16] -> [gather global rows] -> attention -> [combine]
// on the caller's stream.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <map>
#include <memory>
#include <mutex>
#include <queue>
#include <string>
#include <tuple>
#include <vector>


#include "../../include/lfattn.h"
#include "lf_attn_kernel.cuh"
#include "lf_aux_kernels.cuh"
#include "lf_common.cuh"
#include "lf_bwd_tc_kernel.cuh"
#include "lf_gemm_kernel.cuh"
#include "lf_layer_kernels.cuh"

namespace {

using lf::MainParams;
using lf::WorkItem;
using lf::XBlock;

__device__ unsigned g_status_word;

thread_local std::string t_last_error;
std::atomic<uint64_t> g_launches{0};

// ---- per-kernel device-time tracing (events around each library launch)
struct TraceRec {
  const char* name;
  cudaEvent_t e0, e1;
};
std::atomic<int> g_trace_on{0};
std::mutex g_trace_mu;
std::string g_trace_only;   // trace only kernels whose name contains this (empty = all)
std::vector<TraceRec> g_trace;
std::vector<cudaEvent_t> g_event_pool;

cudaEvent_t trace_event() {
  if (!g_event_pool.empty()) {
    cudaEvent_t e = g_event_pool.back();
    g_event_pool.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  cudaEventCreate(&e);
  return e;
}

// Runs `launch` (one kernel launch on `s`) and counts it; while tracing is
// on, brackets it with two events recorded on the same stream.
template <class F>
void traced(const char* name, cudaStream_t s, F&& launch) {
  bool on = g_trace_on.load(std::memory_order_relaxed) != 0;
  if (on) {
    std::lock_guard<std::mutex> lk(g_trace_mu);
    on = g_trace_only.empty() || std::strstr(name, g_trace_only.c_str()) != nullptr;
  }
  if (on) {
    std::lock_guard<std::mutex> lk(g_trace_mu);
    TraceRec r{name, trace_event(), trace_event()};
    cudaEventRecord(r.e0, s);
    launch();
    cudaEventRecord(r.e1, s);
    g_trace.push_back(r);
  } else {
    launch();
  }
  g_launches.fetch_add(1, std::memory_order_relaxed);
}

lf_status fail(lf_status s, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  t_last_error = buf;
  return s;
}

#define LF_CUDA(call)                                                                   \
  do {                                                                                  \
    cudaError_t e_ = (call);                                                            \
    if (e_ != cudaSuccess) {                                                            \
      if (e_ == cudaErrorMemoryAllocation)                                              \
        return fail(LF_ERR_NOMEM, "%s: %s", #call, cudaGetErrorString(e_));             \
      return fail(LF_ERR_CUDA, "%s: %s", #call, cudaGetErrorString(e_));                \
    }                                                                                   \
  } while (0)

// ------------------------------------------------------------ device state

struct DevState {
  bool ready = false;
  int num_sms = 0;
  unsigned* status = nullptr;
  PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
};

std::mutex g_mu;
std::vector<DevState> g_dev;

unsigned long long wait_timeout_ns() {
  static unsigned long long v = [] {
    const char* s = std::getenv("LF_WAIT_TIMEOUT_MS");
    double ms = s ? std::atof(s) : 4000.0;
    if (!(ms >= 0)) ms = 4000.0;
    return static_cast<unsigned long long>(ms * 1e6);
  }();
  return v;
}

lf_status get_dev(DevState** out, int* dev_out) {
  int dev = 0;
  LF_CUDA(cudaGetDevice(&dev));
  std::lock_guard<std::mutex> lk(g_mu);
  if ((int)g_dev.size() <= dev) g_dev.resize(dev + 1);
  DevState& ds = g_dev[dev];
  if (!ds.ready) {
    int major = 0, minor = 0;
    LF_CUDA(cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev));
    LF_CUDA(cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev));
    if (major != 10 || minor != 3)
      return fail(LF_ERR_UNSUPPORTED, "device %d is sm_%d%d; this library is built for sm_103a",
                  dev, major, minor);
    LF_CUDA(cudaDeviceGetAttribute(&ds.num_sms, cudaDevAttrMultiProcessorCount, dev));
    LF_CUDA(cudaGetSymbolAddress(reinterpret_cast<void**>(&ds.status), g_status_word));
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    LF_CUDA(cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                             cudaEnableDefault, &q));
    if (q != cudaDriverEntryPointSuccess || fn == nullptr)
      return fail(LF_ERR_CUDA, "cuTensorMapEncodeTiled entry point not found");
    ds.encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    // The attention kernel hands registers between its warpgroups
    // (setmaxnreg); the split assumes the launch allocation kRegsLaunch.
    for (const void* fn : {reinterpret_cast<const void*>(lf::lf_attn_main_kernel<64>),
                           reinterpret_cast<const void*>(lf::lf_attn_main_kernel<128>),
                           reinterpret_cast<const void*>(lf::lf_attn_main_kernel<64, true>),
                           reinterpret_cast<const void*>(lf::lf_attn_main_kernel<128, true>),
                           reinterpret_cast<const void*>(lf::lf_attn_main_kernel<64, false, true>),
                           reinterpret_cast<const void*>(lf::lf_attn_main_kernel<128, false, true>)}) {
      cudaFuncAttributes fa;
      LF_CUDA(cudaFuncGetAttributes(&fa, fn));
      if (fa.numRegs != (int)lf::kRegsLaunch)
        return fail(LF_ERR_UNSUPPORTED,
                    "attention kernel built with %d registers per thread, expected %u",
                    fa.numRegs, lf::kRegsLaunch);
    }
    LF_CUDA(cudaFuncSetAttribute(lf::lf_attn_main_kernel<64>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)lf::KCfg<64>::SMEM_BYTES));
    LF_CUDA(cudaFuncSetAttribute(lf::lf_attn_main_kernel<128>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)lf::KCfg<128>::SMEM_BYTES));
    LF_CUDA(cudaFuncSetAttribute(lf::lf_attn_main_kernel<64, true>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)lf::KCfg<64>::SMEM_BYTES));
    LF_CUDA(cudaFuncSetAttribute(lf::lf_attn_main_kernel<128, true>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)lf::KCfg<128>::SMEM_BYTES));
    LF_CUDA(cudaFuncSetAttribute(lf::lf_attn_main_kernel<64, false, true>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)lf::KCfg<64>::SMEM_BYTES));
    LF_CUDA(cudaFuncSetAttribute(lf::lf_attn_main_kernel<128, false, true>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)lf::KCfg<128>::SMEM_BYTES));
    ds.ready = true;
  }
  *out = &ds;
  *dev_out = dev;
  return LF_OK;
}

// ------------------------------------------------------------- validation

lf_status check_pattern(int H, int L, int w, const int32_t* dilation, const int32_t* gidx,
                        int n_g) {
  if (H < 1 || L < 1) return fail(LF_ERR_INVALID_ARG, "H=%d and L=%d must be >= 1", H, L);
  if (w < 0) return fail(LF_ERR_INVALID_ARG, "window w=%d must be >= 0", w);
  if (dilation == nullptr) return fail(LF_ERR_INVALID_ARG, "dilation is NULL");
  for (int h = 0; h < H; ++h)
    if (dilation[h] < 1) return fail(LF_ERR_INVALID_ARG, "dilation[%d]=%d < 1", h, dilation[h]);
  if (n_g < 0 || n_g > L) return fail(LF_ERR_INVALID_ARG, "n_global=%d not in [0, L]", n_g);
  if (n_g > 0 && gidx == nullptr) return fail(LF_ERR_INVALID_ARG, "global_idx is NULL");
  for (int g = 0; g < n_g; ++g) {
    if (gidx[g] < 0 || gidx[g] >= L)
      return fail(LF_ERR_INVALID_ARG, "global_idx[%d]=%d out of [0, %d)", g, gidx[g], L);
    if (g > 0 && gidx[g] <= gidx[g - 1])
      return fail(LF_ERR_INVALID_ARG, "global_idx not strictly increasing at %d", g);
  }
  // products such as d*w and H*L must stay inside int32 arithmetic
  for (int h = 0; h < H; ++h)
    if ((long long)dilation[h] * w > (1LL << 28))
      return fail(LF_ERR_UNSUPPORTED, "dilation[%d]*w too large", h);
  if ((long long)H * L > (1LL << 31) - 2) return fail(LF_ERR_UNSUPPORTED, "H*L too large");
  if (L > (1 << 28)) return fail(LF_ERR_UNSUPPORTED, "L=%d too large", L);
  return LF_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// ------------------------------------------------------------------ plans

struct Pattern {
  int H = 0, L = 0, w = 0, n_g = 0;
  std::vector<int32_t> dil, G;
  // extra key blocks per query tile: {T, R, table [H][T][R]}, or empty
  std::vector<int32_t> xkey;
  int32_t* d_G = nullptr;
  uint8_t* d_isg = nullptr;
  int32_t* d_gcnt = nullptr;
  int32_t* d_dil = nullptr;
  std::vector<uint8_t> isg;
  std::vector<int32_t> gcnt;   // [L + 1] number of global positions below x
  // G is a run of consecutive positions G[0] .. G[0] + n_g - 1: the forward
  // then reads the global rows of q, k, v in place, without a gathered copy
  bool g_contig = false;
};

// Global-position tables of a pattern: the flag per position and the prefix
// count, so that the globals inside any window [a, b) are G[gcnt[a] ..
// gcnt[b]) without a search.
void fill_global_tables(Pattern& pt) {
  // (and at least one query tile of rows from G[0] on, so that no box is
  // taller than its tensor)
  pt.g_contig = !pt.G.empty() && pt.L - pt.G[0] >= lf::kBM;
  for (size_t g = 1; g < pt.G.size(); ++g)
    if (pt.G[g] != pt.G[0] + (int32_t)g) pt.g_contig = false;
  pt.isg.assign(pt.L, 0);
  for (int g : pt.G) pt.isg[g] = 1;
  pt.gcnt.assign(pt.L + 1, 0);
  for (int x = 0; x < pt.L; ++x) pt.gcnt[x + 1] = pt.gcnt[x] + pt.isg[x];
}

struct Plan {
  std::shared_ptr<Pattern> pat;
  int B = 0, D = 0;
  int n_slots = 0;
  int slot_dil[lf::kMaxDilSlots] = {0};
  std::vector<int> head_slot;
  int NGB = 16, NGQ = 0, n_gblk = 0, n_chunks = 0;
  std::vector<WorkItem> items;     // grouped by CTA (see cta_begin)
  std::vector<int4> xitem;         // per item {xo, nx0, nx1, 0} (extra blocks; else empty)
  std::vector<XBlock> xlist;       // the extra blocks
  std::vector<int> cta_begin;      // [grid + 1] item ranges per CTA
  int grid = 0;                    // CTAs of the attention kernel
  WorkItem* d_items = nullptr;     // device copy of items, then cta_begin (one allocation,
  int* d_cta = nullptr;            // freed through d_items), then xitem and xlist
  int4* d_xitem = nullptr;
  XBlock* d_xlist = nullptr;
};

using PatKey = std::tuple<int, int, int, int, std::vector<int32_t>, std::vector<int32_t>,
                          std::vector<int32_t>>;
using PlanKey = std::tuple<int, int, int, PatKey>;   // dev, B, D, pattern
std::map<PatKey, std::shared_ptr<Pattern>> g_patterns;
std::map<PlanKey, std::unique_ptr<Plan>> g_plans;

// The extra-block key of a pattern: {T, R, table}, or empty for none.
std::vector<int32_t> xblock_key(int H, const int32_t* xb, int T, int R) {
  std::vector<int32_t> k;
  if (xb == nullptr || T <= 0 || R <= 0) return k;
  k.reserve(2 + (size_t)H * T * R);
  k.push_back(T);
  k.push_back(R);
  k.insert(k.end(), xb, xb + (size_t)H * T * R);
  return k;
}

// Patterns with extra-block tables are cached like the others, but a
// caller may draw a new table every step: past kMaxExtraPatterns of them the
// next new one first evicts them all (see evict_extra_patterns).
constexpr size_t kMaxExtraPatterns = 32;
void evict_extra_patterns();   // needs g_mu held

lf_status get_pattern(int dev, int H, int L, int w, const int32_t* dil, const int32_t* gidx,
                      int n_g, std::shared_ptr<Pattern>* out, const int32_t* xb = nullptr,
                      int T = 0, int R = 0) {
  PatKey key{dev, H, L, w, std::vector<int32_t>(dil, dil + H),
             std::vector<int32_t>(gidx ? gidx : dil, gidx ? gidx + n_g : dil),
             xblock_key(H, xb, T, R)};
  std::lock_guard<std::mutex> lk(g_mu);
  auto it = g_patterns.find(key);
  if (it != g_patterns.end()) {
    *out = it->second;
    return LF_OK;
  }
  if (!std::get<6>(key).empty()) {
    size_t n_extra = 0;
    for (const auto& kv : g_patterns) n_extra += kv.second->xkey.empty() ? 0 : 1;
    if (n_extra >= kMaxExtraPatterns) evict_extra_patterns();
  }
  auto pat = std::make_shared<Pattern>();
  pat->H = H;
  pat->L = L;
  pat->w = w;
  pat->n_g = n_g;
  pat->dil.assign(dil, dil + H);
  if (n_g) pat->G.assign(gidx, gidx + n_g);
  pat->xkey = std::get<6>(key);
  fill_global_tables(*pat);
  LF_CUDA(cudaMalloc(&pat->d_isg, L));
  LF_CUDA(cudaMemcpy(pat->d_isg, pat->isg.data(), L, cudaMemcpyHostToDevice));
  LF_CUDA(cudaMalloc(&pat->d_gcnt, sizeof(int32_t) * (L + 1)));
  LF_CUDA(cudaMemcpy(pat->d_gcnt, pat->gcnt.data(), sizeof(int32_t) * (L + 1),
                     cudaMemcpyHostToDevice));
  LF_CUDA(cudaMalloc(&pat->d_dil, sizeof(int32_t) * H));
  LF_CUDA(cudaMemcpy(pat->d_dil, dil, sizeof(int32_t) * H, cudaMemcpyHostToDevice));
  LF_CUDA(cudaMalloc(&pat->d_G, sizeof(int32_t) * std::max(n_g, 1)));
  if (n_g) LF_CUDA(cudaMemcpy(pat->d_G, gidx, sizeof(int32_t) * n_g, cudaMemcpyHostToDevice));
  g_patterns[key] = pat;
  *out = pat;
  return LF_OK;
}

int ceil_div(int a, int b) { return (a + b - 1) / b; }

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Work list of the attention kernel (see WorkItem): for each (b, h), its
// band pairs of neighbouring 128-query tiles (per residue class), then its
// global-row chunks, so that a head's keys are still in L2 when the global
// rows read them.  The items are then spread over the CTAs longest first,
// each to the least-loaded CTA (a cost per item = the blocks of its busier
// slot, gathered blocks weighted by their width, plus one for the item's
// own loads and epilogue), and stored grouped by CTA.
int item_cost(const WorkItem& wi, int NGB, const int4& xi) {
  int c[2];
  for (int X = 0; X < 2; ++X) {
    const int n = lf::blk_count(wi, X);
    if (wi.kind == 0 && n > 0)
      c[X] = 8 * (n - wi.ngb) + (wi.ngb * NGB + 15) / 16 + 8 * (X ? xi.z : xi.y);   // eighths
    else
      c[X] = 8 * n;
  }
  return std::max(c[0], c[1]) + 8;
}

// The extra key blocks of one query tile (rows ta..tb of residue class r of
// head h, class length Lr): the table's row for the tile, without -1,
// duplicates and blocks that every row already holds in its window;
// appended to xlist with the bits of their global columns.  Returns how many.
int tile_extra_blocks(const Pattern& pt, int h, int d, int r, int Lr, int ta, int tb,
                      std::vector<XBlock>& xlist) {
  if (pt.xkey.empty()) return 0;
  const int T = pt.xkey[0], R = pt.xkey[1];
  const int nqt = ceil_div(ceil_div(pt.L, d), lf::kBM);
  const int rho = r * nqt + ta / lf::kBM;
  const int32_t* row = pt.xkey.data() + 2 + ((size_t)h * T + rho) * R;
  std::vector<int> kbs;
  for (int e = 0; e < R; ++e)
    if (row[e] >= 0) kbs.push_back(row[e]);
  std::sort(kbs.begin(), kbs.end());
  kbs.erase(std::unique(kbs.begin(), kbs.end()), kbs.end());
  int n = 0;
  for (int kb : kbs) {
    const int k0 = kb * lf::kBN, k1 = std::min(k0 + lf::kBN, Lr) - 1;
    if (k0 > k1) continue;
    if (k0 >= tb - pt.w && k1 <= ta + pt.w) continue;   // inside every row's window
    XBlock xb{};
    xb.kpos0 = k0;
    for (int c = 0; c <= k1 - k0; ++c)
      if (pt.isg[r + d * (k0 + c)]) xb.gm[c >> 5] |= 1u << (c & 31);
    xlist.push_back(xb);
    ++n;
  }
  return n;
}

void build_items(Plan& pl, int num_sms) {
  const Pattern& pt = *pl.pat;
  const int H = pt.H, L = pt.L, w = pt.w, n_g = pt.n_g;
  // global key blocks folded into every band tile
  if (n_g > 0) {
    pl.NGB = n_g <= lf::kBN ? ((n_g + 15) / 16) * 16 : lf::kBN;
    pl.n_gblk = ceil_div(n_g, pl.NGB);
    pl.NGQ = ceil_div(n_g, lf::kBM) * lf::kBM;
  } else {
    pl.NGB = 16;
    pl.n_gblk = 0;
    pl.NGQ = 0;
  }
  // key-chunk length of the global-row items: about half a band pair's
  // blocks (of an undilated head), so that they also fill the tail of the
  // schedule.  It depends on (L, w, n_g) only, not on which heads a call
  // holds, so that a head's global rows are summed in the same key chunks
  // whatever heads it is computed with.
  const int pair_blocks =
      ceil_div(std::min(2 * lf::kBM + 2 * w, L), lf::kBN) + pl.n_gblk;
  const int nblocks = ceil_div(L, lf::kBN);
  int n_items1 = 0, CB = 0;
  if (n_g > 0) {
    CB = std::max(2, std::min(nblocks, pair_blocks));
    n_items1 = ceil_div(nblocks, CB);
    CB = ceil_div(nblocks, n_items1);   // even out the chunks
    pl.n_chunks = 2 * n_items1;
  } else {
    pl.n_chunks = 0;
  }
  std::vector<WorkItem> order;
  std::vector<int4> order_x;   // extra blocks of each item, parallel to order
  pl.xlist.clear();
  for (int b = 0; b < pl.B; ++b) {
    for (int h = 0; h < H; ++h) {
      const int bh = b * H + h;
      const int d = pt.dil[h];
      for (int r = 0; r < d; ++r) {
        const int Lr = lf::residue_len(L, d, r);
        for (int t0 = 0; t0 < Lr; t0 += 2 * lf::kBM) {
          // key range [lo, hi] (residue space) of each slot; absent slots have lo > hi
          int lo[2], hi[2];
          bool present[2];
          for (int X = 0; X < 2; ++X) {
            const int ta = t0 + X * lf::kBM;
            const int tb = std::min(ta + lf::kBM - 1, Lr - 1);
            present[X] = ta < Lr;
            if (present[X] && n_g > 0) {
              bool all_global = true;
              for (int t = ta; t <= tb && all_global; ++t) all_global = pt.isg[r + d * t] != 0;
              present[X] = !all_global;
            }
            lo[X] = std::max(ta - w, 0);
            hi[X] = std::min(tb + w, Lr - 1);
          }
          if (!present[0] && !present[1]) continue;
          const int plo = present[0] ? lo[0] : lo[1];
          const int phi = present[1] ? hi[1] : hi[0];
          WorkItem wi{};
          wi.bh = bh;
          wi.kind = 0;
          wi.r = r;
          wi.t0 = t0;
          wi.kb0 = plo;
          wi.nkb = ceil_div(phi - plo + 1, lf::kBN);
          wi.ngb = pl.n_gblk;
          wi.slot = pl.head_slot[h];
          int4 xi = make_int4((int)pl.xlist.size(), 0, 0, 0);
          for (int X = 0; X < 2; ++X) {
            if (present[X]) {
              wi.jlo[X] = (lo[X] - plo) / lf::kBN;
              wi.jhi[X] = (hi[X] - plo) / lf::kBN;
              const int ta = t0 + X * lf::kBM, tb = std::min(ta + lf::kBM - 1, Lr - 1);
              const int nx = tile_extra_blocks(pt, h, d, r, Lr, ta, tb, pl.xlist);
              if (X) xi.z = nx; else xi.y = nx;
            } else {
              wi.jlo[X] = 1;
              wi.jhi[X] = 0;
            }
          }
          order.push_back(wi);
          order_x.push_back(xi);
        }
      }
      for (int gt = 0; gt < pl.NGQ / lf::kBM; ++gt)
        for (int c = 0; c < n_items1; ++c) {
          WorkItem wi{};
          wi.bh = bh;
          wi.kind = 1;
          wi.r = gt;
          wi.t0 = 0;
          wi.kb0 = c * CB * lf::kBN;
          wi.nkb = std::min(CB, nblocks - c * CB);
          wi.ngb = 0;
          wi.slot = c;
          wi.jlo[0] = wi.jlo[1] = 0;
          wi.jhi[0] = wi.jhi[1] = -1;
          order.push_back(wi);
          order_x.push_back(make_int4(0, 0, 0, 0));
        }
    }
  }
  // longest first onto the least-loaded CTA
  const int n = (int)order.size();
  pl.grid = std::max(1, std::min(n, num_sms));
  std::vector<int> idx(n);
  std::vector<int> cost(n);
  for (int x = 0; x < n; ++x) {
    idx[x] = x;
    cost[x] = item_cost(order[x], pl.NGB, order_x[x]);
  }
  std::stable_sort(idx.begin(), idx.end(), [&](int a, int b) { return cost[a] > cost[b]; });
  std::vector<std::vector<int>> per_cta(pl.grid);
  using Load = std::pair<long long, int>;   // (load, cta)
  std::priority_queue<Load, std::vector<Load>, std::greater<Load>> heap;
  for (int c = 0; c < pl.grid; ++c) heap.push({0LL, c});
  for (int x : idx) {
    Load top = heap.top();
    heap.pop();
    per_cta[top.second].push_back(x);
    top.first += cost[x];
    heap.push(top);
  }
  pl.items.clear();
  pl.items.reserve(n);
  pl.xitem.clear();
  pl.cta_begin.assign(pl.grid + 1, 0);
  const bool extra = !pt.xkey.empty();
  for (int c = 0; c < pl.grid; ++c) {
    // keep each CTA's items in list order (head by head, along the keys)
    std::sort(per_cta[c].begin(), per_cta[c].end());
    for (int x : per_cta[c]) {
      pl.items.push_back(order[x]);
      if (extra) pl.xitem.push_back(order_x[x]);
    }
    pl.cta_begin[c + 1] = (int)pl.items.size();
  }
}

// Every block of an item must have a user: the kernel releases a K/V stage
// after its users' products (checked once per plan).
bool items_consistent(const Plan& pl) {
  for (size_t x = 0; x < pl.items.size(); ++x) {
    const WorkItem& wi = pl.items[x];
    const int4 xi = pl.xitem.empty() ? make_int4(0, 0, 0, 0) : pl.xitem[x];
    const lf::SlotBlocks s0(wi, 0, xi.y, xi.z), s1(wi, 1, xi.y, xi.z);
    for (int j = 0; j < wi.nkb + wi.ngb + xi.y + xi.z; ++j)
      if (!s0.uses(j) && !s1.uses(j)) return false;
    if (wi.nkb < 1) return false;
    if (xi.y + xi.z > 0 && (wi.kind != 0 || xi.x < 0 || (size_t)xi.x + xi.y + xi.z > pl.xlist.size()))
      return false;
  }
  return true;
}

lf_status get_plan(int dev, int num_sms, int B, int D, const std::shared_ptr<Pattern>& pat,
                   Plan** out) {
  PatKey pk{dev, pat->H, pat->L, pat->w, pat->dil, pat->G, pat->xkey};
  PlanKey key{dev, B, D, pk};
  std::lock_guard<std::mutex> lk(g_mu);
  auto it = g_plans.find(key);
  if (it != g_plans.end()) {
    *out = it->second.get();
    return LF_OK;
  }
  auto pl = std::make_unique<Plan>();
  pl->pat = pat;
  pl->B = B;
  pl->D = D;
  pl->head_slot.resize(pat->H);
  for (int h = 0; h < pat->H; ++h) {
    int s = 0;
    while (s < pl->n_slots && pl->slot_dil[s] != pat->dil[h]) ++s;
    if (s == pl->n_slots) {
      if (pl->n_slots == lf::kMaxDilSlots)
        return fail(LF_ERR_UNSUPPORTED, "more than %d distinct dilation values",
                    lf::kMaxDilSlots);
      pl->slot_dil[pl->n_slots++] = pat->dil[h];
    }
    pl->head_slot[h] = s;
  }
  build_items(*pl, num_sms);
  if (!items_consistent(*pl)) return fail(LF_ERR_INVALID_ARG, "internal: inconsistent work list");
  {
    const size_t ib = align_up(sizeof(WorkItem) * std::max<size_t>(pl->items.size(), 1), 256);
    const size_t cb = align_up(sizeof(int) * pl->cta_begin.size(), 256);
    const size_t xib = align_up(sizeof(int4) * pl->xitem.size(), 256);
    const size_t xlb = align_up(sizeof(XBlock) * pl->xlist.size(), 256);
    uint8_t* dev_mem = nullptr;
    LF_CUDA(cudaMalloc(reinterpret_cast<void**>(&dev_mem), ib + cb + xib + xlb));
    pl->d_items = reinterpret_cast<WorkItem*>(dev_mem);
    pl->d_cta = reinterpret_cast<int*>(dev_mem + ib);
    if (!pl->items.empty())
      LF_CUDA(cudaMemcpy(pl->d_items, pl->items.data(), sizeof(WorkItem) * pl->items.size(),
                         cudaMemcpyHostToDevice));
    LF_CUDA(cudaMemcpy(pl->d_cta, pl->cta_begin.data(), sizeof(int) * pl->cta_begin.size(),
                       cudaMemcpyHostToDevice));
    if (!pl->xitem.empty()) {
      pl->d_xitem = reinterpret_cast<int4*>(dev_mem + ib + cb);
      LF_CUDA(cudaMemcpy(pl->d_xitem, pl->xitem.data(), sizeof(int4) * pl->xitem.size(),
                         cudaMemcpyHostToDevice));
    }
    if (!pl->xlist.empty()) {
      pl->d_xlist = reinterpret_cast<XBlock*>(dev_mem + ib + cb + xib);
      LF_CUDA(cudaMemcpy(pl->d_xlist, pl->xlist.data(), sizeof(XBlock) * pl->xlist.size(),
                         cudaMemcpyHostToDevice));
    }
  }
  *out = pl.get();
  g_plans[key] = std::move(pl);
  return LF_OK;
}

// ------------------------------------------------------------ tensor maps

lf_status encode(DevState* ds, CUtensorMap* m, const void* base, int rank, const uint64_t* dims,
                 const uint64_t* strides_bytes, const uint32_t* box,
                 CUtensorMapDataType dtype = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                 CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_128B) {
  cuuint64_t gd[5];
  cuuint64_t gs[4];
  cuuint32_t bx[5], es[5];
  for (int i = 0; i < rank; ++i) {
    gd[i] = dims[i];
    bx[i] = box[i];
    es[i] = 1;
  }
  for (int i = 0; i < rank - 1; ++i) gs[i] = strides_bytes[i];
  CUresult r = ds->encode(m, dtype, rank, const_cast<void*>(base), gd,
                          gs, bx, es, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(LF_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
  return LF_OK;
}

// 4-D residue view {D, d, L/d, BH} of a [BH, L, D] bf16 tensor
lf_status map_residue(DevState* ds, CUtensorMap* m, const void* base, int D, int L, int d,
                      int BH, uint32_t box_rows = 128) {
  const uint64_t dims[4] = {(uint64_t)D, (uint64_t)d, (uint64_t)(L / d), (uint64_t)BH};
  const uint64_t st[3] = {(uint64_t)D * 2, (uint64_t)D * 2 * d, (uint64_t)D * 2 * L};
  const uint32_t box[4] = {64, 1, box_rows, 1};
  return encode(ds, m, base, 4, dims, st, box);
}

// 4-D residue view {D, d, L/d, BH} of a [BH, L, D] fp32 tensor, box
// {64, 1, box_rows, 1}, unswizzled (the target of tiled reduce-adds)
lf_status map_residue_f32(DevState* ds, CUtensorMap* m, const void* base, int D, int L, int d,
                          int BH, uint32_t box_rows) {
  const uint64_t dims[4] = {(uint64_t)D, (uint64_t)d, (uint64_t)(L / d), (uint64_t)BH};
  const uint64_t st[3] = {(uint64_t)D * 4, (uint64_t)D * 4 * d, (uint64_t)D * 4 * L};
  const uint32_t box[4] = {64, 1, box_rows, 1};
  return encode(ds, m, base, 4, dims, st, box, CU_TENSOR_MAP_DATA_TYPE_FLOAT32,
                CU_TENSOR_MAP_SWIZZLE_NONE);
}

// 3-D view {D, rows, BH} with a box of `box_rows` rows; consecutive bh lie
// `bh_rows` rows apart (default: rows)
lf_status map_rows(DevState* ds, CUtensorMap* m, const void* base, int D, int rows, int BH,
                   int box_rows, int bh_rows = 0) {
  const uint64_t dims[3] = {(uint64_t)D, (uint64_t)rows, (uint64_t)BH};
  const uint64_t st[2] = {(uint64_t)D * 2, (uint64_t)D * 2 * (bh_rows > 0 ? bh_rows : rows)};
  const uint32_t box[3] = {64, (uint32_t)box_rows, 1};
  return encode(ds, m, base, 3, dims, st, box);
}

// ------------------------------------------------------------------ forward


// Scratch of lf_attn_fwd / lf_attn_fwd_f32: one grow-only buffer per
// (device, stream).  Calls on one stream are ordered, so they can share it;
// a larger need frees the old buffer and allocates a new one, both
// stream-ordered.  lf_plan_cache_clear releases every buffer.
struct Workspace {
  uint8_t* ptr = nullptr;
  size_t bytes = 0;
};
std::map<std::pair<int, cudaStream_t>, Workspace> g_workspaces;

lf_status get_workspace(int dev, cudaStream_t stream, size_t bytes, uint8_t** out) {
  std::lock_guard<std::mutex> lk(g_mu);
  Workspace& w = g_workspaces[{dev, stream}];
  if (w.bytes < bytes) {
    if (w.ptr) LF_CUDA(cudaFreeAsync(w.ptr, stream));
    w.ptr = nullptr;
    w.bytes = 0;
    const size_t grow = align_up(bytes, size_t(1) << 20);
    LF_CUDA(cudaMallocAsync(reinterpret_cast<void**>(&w.ptr), grow, stream));
    w.bytes = grow;
  }
  *out = w.ptr;
  return LF_OK;
}

// Kernel parameters (tensor maps included) of recent calls, keyed by the
// plan and every device address they embed, so that a repeated call encodes
// nothing.
using ParamKey = std::tuple<const Plan*, const void*, const void*, const void*, void*, bool,
                            const uint8_t*, float, float*, const float*>;
// (shared ownership: a call keeps its parameters alive until it has
// launched, even if another thread clears the cache meanwhile)
std::map<ParamKey, std::shared_ptr<MainParams>> g_params;
constexpr size_t kMaxCachedParams = 256;

// Frees every cached pattern that has an extra-block table, with its plans
// and their kernel parameters, after the device has finished all work
// queued so far (an in-flight kernel may still read a plan's work list).
void evict_extra_patterns() {
  cudaDeviceSynchronize();
  for (auto it = g_params.begin(); it != g_params.end();) {
    const Plan* pl = std::get<0>(it->first);
    if (pl != nullptr && !pl->pat->xkey.empty())
      it = g_params.erase(it);
    else
      ++it;
  }
  for (auto it = g_plans.begin(); it != g_plans.end();) {
    if (!it->second->pat->xkey.empty()) {
      if (it->second->d_items) cudaFree(it->second->d_items);
      it = g_plans.erase(it);
    } else {
      ++it;
    }
  }
  for (auto it = g_patterns.begin(); it != g_patterns.end();) {
    Pattern& pt = *it->second;
    if (!pt.xkey.empty()) {
      cudaFree(pt.d_G);
      cudaFree(pt.d_isg);
      cudaFree(pt.d_gcnt);
      cudaFree(pt.d_dil);
      it = g_patterns.erase(it);
    } else {
      ++it;
    }
  }
}

// Kernel parameters of one call: tensor maps of q, k, v (one residue view
// per dilation value) and of the gathered global rows, and the scratch
// addresses.
lf_status build_params(DevState* ds, const Plan& plan, const Pattern& pattern, const void* qb,
                       const void* kb, const void* vb, void* out, bool f32, uint8_t* ws,
                       size_t off_g, size_t off_po, size_t off_pm, float scale, float* lse,
                       const float* rel_bias, MainParams* prm_out) {
  lf_status s = LF_OK;
  const Plan* pl = &plan;
  const Pattern* pat = &pattern;
  const int D = pl->D, L = pat->L, H = pat->H, w = pat->w, n_g = pat->n_g;
  const int BH = pl->B * H;
  MainParams& P = *prm_out;
  std::memset(&P, 0, sizeof(P));
  for (int sl = 0; sl < pl->n_slots; ++sl) {
    const int d = pl->slot_dil[sl];
    P.dil[sl] = d;
    if ((s = map_residue(ds, &P.tmQ[sl], qb, D, L, d, BH)) != LF_OK) return s;
    if ((s = map_residue(ds, &P.tmK[sl], kb, D, L, d, BH)) != LF_OK) return s;
    if ((s = map_residue(ds, &P.tmV[sl], vb, D, L, d, BH)) != LF_OK) return s;
  }
  const size_t g_elems = (size_t)BH * pl->NGQ * D;
  uint16_t* qg = reinterpret_cast<uint16_t*>(ws + off_g);
  uint16_t* kg = qg + g_elems;
  uint16_t* vg = kg + g_elems;
  if (n_g > 0) {
    if ((s = map_rows(ds, &P.tmKp, kb, D, L, BH, lf::kBN)) != LF_OK) return s;
    if ((s = map_rows(ds, &P.tmVp, vb, D, L, BH, lf::kBN)) != LF_OK) return s;
    if (pat->g_contig) {
      // the global rows in place: rows G[0].. of each head (past n_g the
      // kernel masks the keys and drops the query rows; past L the loads
      // read zeros)
      const size_t g0 = (size_t)pat->G[0] * D;
      const int rows = L - pat->G[0];
      const uint16_t* q0 = static_cast<const uint16_t*>(qb) + g0;
      const uint16_t* k0 = static_cast<const uint16_t*>(kb) + g0;
      const uint16_t* v0 = static_cast<const uint16_t*>(vb) + g0;
      if ((s = map_rows(ds, &P.tmQg, q0, D, rows, BH, lf::kBM, L)) != LF_OK) return s;
      if ((s = map_rows(ds, &P.tmKg, k0, D, rows, BH, pl->NGB, L)) != LF_OK) return s;
      if ((s = map_rows(ds, &P.tmVg, v0, D, rows, BH, pl->NGB, L)) != LF_OK) return s;
    } else {
      if ((s = map_rows(ds, &P.tmQg, qg, D, pl->NGQ, BH, lf::kBM)) != LF_OK) return s;
      if ((s = map_rows(ds, &P.tmKg, kg, D, pl->NGQ, BH, pl->NGB)) != LF_OK) return s;
      if ((s = map_rows(ds, &P.tmVg, vg, D, pl->NGQ, BH, pl->NGB)) != LF_OK) return s;
    }
  }
  P.items = pl->d_items;
  P.cta_begin = pl->d_cta;
  P.n_items = (int)pl->items.size();
  P.gidx = pat->d_G;
  P.is_glob = pat->d_isg;
  P.gcnt = pat->d_gcnt;
  P.n_g = n_g;
  P.NGB = pl->NGB;
  P.NGQ = pl->NGQ;
  P.n_chunks = pl->n_chunks;
  P.out = out;
  P.out_f32 = f32 ? 1 : 0;
  P.part_o = reinterpret_cast<float*>(ws + off_po);
  P.part_ml = reinterpret_cast<float*>(ws + off_pm);
  P.H = H;
  P.L = L;
  P.w = w;
  P.sl2 = scale * 1.4426950408889634f;
  P.lse = lse;
  P.rel_bias = rel_bias;
  P.xitem = pl->d_xitem;
  P.xlist = pl->d_xlist;
  P.status = ds->status;
  P.wait_iters = lf::wait_iters_for(wait_timeout_ns());

  return LF_OK;
}

lf_status fwd_impl(const void* q, const void* k, const void* v, void* out, bool f32, int B, int H,
                   int L, int D, int w, const int32_t* dilation, const int32_t* gidx, int n_g,
                   float scale, cudaStream_t stream, float* lse = nullptr,
                   const float* rel_bias = nullptr, const int32_t* xblocks = nullptr, int xT = 0,
                   int xR = 0) {
  t_last_error.clear();
  if (B < 1) return fail(LF_ERR_INVALID_ARG, "B=%d must be >= 1", B);
  lf_status s = check_pattern(H, L, w, dilation, gidx, n_g);
  if (s != LF_OK) return s;
  if (!q || !k || !v || !out) return fail(LF_ERR_INVALID_ARG, "a tensor pointer is NULL");
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out))
    return fail(LF_ERR_INVALID_ARG, "tensor pointers must be 16-byte aligned");
  if (!std::isfinite(scale) || !(scale > 0.f))
    return fail(LF_ERR_INVALID_ARG, "scale must be finite and > 0");
  if (D != 64 && D != 128) return fail(LF_ERR_UNSUPPORTED, "D=%d (supported: 64, 128)", D);
  for (int h = 0; h < H; ++h)
    if (dilation[h] > 1 && L % dilation[h] != 0)
      return fail(LF_ERR_UNSUPPORTED, "L=%d is not a multiple of dilation[%d]=%d", L, h,
                  dilation[h]);
  if ((long long)B * H > (1LL << 30)) return fail(LF_ERR_UNSUPPORTED, "B*H too large");

  DevState* ds = nullptr;
  int dev = 0;
  if ((s = get_dev(&ds, &dev)) != LF_OK) return s;
  std::shared_ptr<Pattern> pat;
  if ((s = get_pattern(dev, H, L, w, dilation, gidx, n_g, &pat, xblocks, xT, xR)) != LF_OK)
    return s;
  Plan* pl = nullptr;
  if ((s = get_plan(dev, ds->num_sms, B, D, pat, &pl)) != LF_OK) return s;
  const bool xb = !pat->xkey.empty();
  if (xb && rel_bias) return fail(LF_ERR_UNSUPPORTED, "extra blocks with a bias table");

  const int BH = B * H;
  const size_t elems = (size_t)BH * L * D;
  // scratch layout
  size_t off = 0;
  const size_t off_cast = off;
  if (f32) off += align_up(3 * elems * 2, 256);
  const size_t off_g = off;
  const size_t g_elems = (size_t)BH * pl->NGQ * D;
  if (n_g > 0) off += align_up(3 * g_elems * 2, 256);
  const size_t off_po = off;
  const size_t n_part = (size_t)BH * pl->NGQ * pl->n_chunks;
  if (n_g > 0) off += align_up(n_part * D * 4, 256);
  const size_t off_pm = off;
  if (n_g > 0) off += align_up(n_part * 2 * 4, 256);
  uint8_t* ws = nullptr;
  if (off > 0 && (s = get_workspace(dev, stream, off, &ws)) != LF_OK) return s;

  const void *qb = q, *kb = k, *vb = v;
  if (f32) {
    uint16_t* cq = reinterpret_cast<uint16_t*>(ws + off_cast);
    const size_t n4 = elems / 4;
    const int threads = 256;
    const int blocks = (int)std::min<size_t>((n4 + threads - 1) / threads, (size_t)ds->num_sms * 8);
    traced("cast_f32_bf16", stream, [&] {
      lf::lf_cast_f32_bf16_kernel<<<blocks, threads, 0, stream>>>(
          reinterpret_cast<const float4*>(q), reinterpret_cast<const float4*>(k),
          reinterpret_cast<const float4*>(v), reinterpret_cast<uint2*>(cq), n4);
    });
    qb = cq;
    kb = cq + elems;
    vb = cq + 2 * elems;
  }

  const ParamKey pkey{pl, qb, kb, vb, out, f32, ws, scale, lse, rel_bias};
  std::shared_ptr<MainParams> cached;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    auto it = g_params.find(pkey);
    if (it != g_params.end()) cached = it->second;
  }
  uint16_t* qg = reinterpret_cast<uint16_t*>(ws + off_g);
  uint16_t* kg = qg + g_elems;
  uint16_t* vg = kg + g_elems;
  if (cached == nullptr) {
    auto fresh = std::make_shared<MainParams>();
    if ((s = build_params(ds, *pl, *pat, qb, kb, vb, out, f32, ws, off_g, off_po, off_pm, scale,
                          lse, rel_bias, fresh.get())) != LF_OK)
      return s;
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_params.size() >= kMaxCachedParams) g_params.clear();
    cached = fresh;
    g_params[pkey] = fresh;
  }
  const MainParams& prm = *cached;

  if (n_g > 0 && !pat->g_contig) {
    const size_t total = (size_t)BH * pl->NGQ * (D / 8);
    const int threads = 256;
    const int blocks = (int)std::max<size_t>(1, std::min<size_t>((total + threads - 1) / threads,
                                                                 (size_t)ds->num_sms * 8));
    traced("gather_globals", stream, [&] {
      lf::lf_gather_globals_kernel<<<blocks, threads, 0, stream>>>(
          reinterpret_cast<const uint4*>(qb), reinterpret_cast<const uint4*>(kb),
          reinterpret_cast<const uint4*>(vb), reinterpret_cast<uint4*>(qg),
          reinterpret_cast<uint4*>(kg), reinterpret_cast<uint4*>(vg), pat->d_G, n_g, pl->NGQ, L,
          D, BH);
    });
  }
  if (prm.n_items > 0) {
    const int grid = pl->grid;
    // the kernel build: plain, with a relative position bias (BIAS: adds the
    // padded table to the window's scores), or with extra key blocks per
    // slot (XB: random / strided block patterns); the plain build is not
    // affected by the others' code
    traced("attn_main", stream, [&] {
      if (D == 64 && xb)
        lf::lf_attn_main_kernel<64, false, true><<<grid, lf::KCfg<64>::THREADS, lf::KCfg<64>::SMEM_BYTES, stream>>>(prm);
      else if (D == 128 && xb)
        lf::lf_attn_main_kernel<128, false, true><<<grid, lf::KCfg<128>::THREADS, lf::KCfg<128>::SMEM_BYTES, stream>>>(prm);
      else if (D == 64 && rel_bias)
        lf::lf_attn_main_kernel<64, true><<<grid, lf::KCfg<64>::THREADS, lf::KCfg<64>::SMEM_BYTES, stream>>>(prm);
      else if (D == 64)
        lf::lf_attn_main_kernel<64><<<grid, lf::KCfg<64>::THREADS, lf::KCfg<64>::SMEM_BYTES, stream>>>(prm);
      else if (rel_bias)
        lf::lf_attn_main_kernel<128, true><<<grid, lf::KCfg<128>::THREADS, lf::KCfg<128>::SMEM_BYTES, stream>>>(prm);
      else
        lf::lf_attn_main_kernel<128><<<grid, lf::KCfg<128>::THREADS, lf::KCfg<128>::SMEM_BYTES, stream>>>(prm);
    });
  }
  if (n_g > 0) {
    const int threads = 256;
    const long long warps = (long long)BH * n_g;
    const int blocks = (int)((warps + threads / 32 - 1) / (threads / 32));
    traced("combine_globals", stream, [&] {
      if (D == 64)
        lf::lf_combine_globals_kernel<64><<<blocks, threads, 0, stream>>>(
            prm.part_o, prm.part_ml, pat->d_G, out, prm.out_f32, n_g, pl->NGQ, pl->n_chunks, L,
            BH, lse);
      else
        lf::lf_combine_globals_kernel<128><<<blocks, threads, 0, stream>>>(
            prm.part_o, prm.part_ml, pat->d_G, out, prm.out_f32, n_g, pl->NGQ, pl->n_chunks, L,
            BH, lse);
    });
  }
  LF_CUDA(cudaGetLastError());
  return LF_OK;
}

// ------------------------------------------------- allocation-free forward
//
// Scratch of lf_attn_fwd_noalloc: one file-scope device array, sized once
// for every GPU that loads the library (see kNoAllocScratchBytes).  It holds,
// per call, the work list, the global-position tables, the gathered global
// rows and the global-row partials.  Host code never names the array as a
// device address; it takes the address from cudaGetSymbolAddress once per
// device (noalloc_scratch below).
constexpr size_t kNoAllocScratchBytes = size_t(32) << 20;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

struct NoAllocDev {
  bool ready = false;
  uint8_t* scratch = nullptr;
};
std::vector<NoAllocDev> g_noalloc_dev;

// Device address of the scratch array on the current device `dev`; looked
// up on the first call for that device.
lf_status noalloc_scratch(int dev, uint8_t** out) {
  std::lock_guard<std::mutex> lk(g_mu);
  if ((int)g_noalloc_dev.size() <= dev) g_noalloc_dev.resize(dev + 1);
  NoAllocDev& nd = g_noalloc_dev[dev];
  if (!nd.ready) {
    void* ptr = nullptr;
    LF_CUDA(cudaGetSymbolAddress(&ptr, g_noalloc_scratch));
    if (ptr == nullptr) return fail(LF_ERR_CUDA, "no device address for the scratch array");
    nd.scratch = static_cast<uint8_t*>(ptr);
    nd.ready = true;
  }
  *out = nd.scratch;
  return LF_OK;
}

lf_status fwd_noalloc_impl(const void* q, const void* k, const void* v, void* out, int B, int H,
                           int L, int D, int w, const int32_t* dilation, const int32_t* gidx,
                           int n_g, float scale, cudaStream_t stream) {
  t_last_error.clear();
  if (B < 1) return fail(LF_ERR_INVALID_ARG, "B=%d must be >= 1", B);
  lf_status s = check_pattern(H, L, w, dilation, gidx, n_g);
  if (s != LF_OK) return s;
  if (!q || !k || !v || !out) return fail(LF_ERR_INVALID_ARG, "a tensor pointer is NULL");
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out))
    return fail(LF_ERR_INVALID_ARG, "tensor pointers must be 16-byte aligned");
  if (!std::isfinite(scale) || !(scale > 0.f))
    return fail(LF_ERR_INVALID_ARG, "scale must be finite and > 0");
  if (D != 64 && D != 128) return fail(LF_ERR_UNSUPPORTED, "D=%d (supported: 64, 128)", D);
  for (int h = 0; h < H; ++h)
    if (dilation[h] > 1 && L % dilation[h] != 0)
      return fail(LF_ERR_UNSUPPORTED, "L=%d is not a multiple of dilation[%d]=%d", L, h,
                  dilation[h]);
  if ((long long)B * H > (1LL << 30)) return fail(LF_ERR_UNSUPPORTED, "B*H too large");

  // the plan, on the host only (the cached plans live in allocated memory)
  Plan pl;
  {
    auto pat = std::make_shared<Pattern>();
    pat->H = H;
    pat->L = L;
    pat->w = w;
    pat->n_g = n_g;
    pat->dil.assign(dilation, dilation + H);
    if (n_g) pat->G.assign(gidx, gidx + n_g);
    fill_global_tables(*pat);
    pl.pat = pat;
  }
  pl.B = B;
  pl.D = D;
  pl.head_slot.resize(H);
  for (int h = 0; h < H; ++h) {
    int sl = 0;
    while (sl < pl.n_slots && pl.slot_dil[sl] != dilation[h]) ++sl;
    if (sl == pl.n_slots) {
      if (pl.n_slots == lf::kMaxDilSlots)
        return fail(LF_ERR_UNSUPPORTED, "more than %d distinct dilation values", lf::kMaxDilSlots);
      pl.slot_dil[pl.n_slots++] = dilation[h];
    }
    pl.head_slot[h] = sl;
  }

  // scratch layout: work list | global positions | global flags | global
  // prefix counts | gathered q, k, v | partial O | partial (m, l); each part
  // 256-byte aligned
  const int BH = B * H;
  DevState* ds = nullptr;
  int dev = 0;
  if ((s = get_dev(&ds, &dev)) != LF_OK) return s;
  build_items(pl, ds->num_sms);
  if (!items_consistent(pl)) return fail(LF_ERR_INVALID_ARG, "internal: inconsistent work list");
  size_t off = 0;
  const size_t off_items = off;
  off += align_up(sizeof(WorkItem) * std::max<size_t>(pl.items.size(), 1), 256);
  const size_t off_cta = off;
  off += align_up(sizeof(int) * pl.cta_begin.size(), 256);
  const size_t off_gidx = off;
  off += align_up(sizeof(int32_t) * std::max(n_g, 1), 256);
  const size_t off_isg = off;
  off += align_up((size_t)L, 256);
  const size_t off_gcnt = off;
  off += align_up(sizeof(int32_t) * ((size_t)L + 1), 256);
  const size_t off_g = off;
  const size_t g_elems = (size_t)BH * pl.NGQ * D;
  if (n_g > 0) off += align_up(3 * g_elems * 2, 256);
  const size_t off_po = off;
  const size_t n_part = (size_t)BH * pl.NGQ * pl.n_chunks;
  if (n_g > 0) off += align_up(n_part * D * 4, 256);
  const size_t off_pm = off;
  if (n_g > 0) off += align_up(n_part * 2 * 4, 256);
  if (off > kNoAllocScratchBytes)
    return fail(LF_ERR_UNSUPPORTED,
                "this problem needs %zu bytes of scratch; the allocation-free entry point has "
                "%zu (use lf_attn_fwd)",
                off, kNoAllocScratchBytes);

  uint8_t* ws = nullptr;
  if ((s = noalloc_scratch(dev, &ws)) != LF_OK) return s;
  // tables into the scratch array (plain copies; nothing needs clearing:
  // every byte the kernels read is written first, by these copies or by the
  // gather kernel and the attention kernel's partial writes)
  WorkItem* d_items = reinterpret_cast<WorkItem*>(ws + off_items);
  int* d_cta = reinterpret_cast<int*>(ws + off_cta);
  int32_t* d_gidx = reinterpret_cast<int32_t*>(ws + off_gidx);
  uint8_t* d_isg = ws + off_isg;
  int32_t* d_gcnt = reinterpret_cast<int32_t*>(ws + off_gcnt);
  if (!pl.items.empty())
    LF_CUDA(cudaMemcpyAsync(d_items, pl.items.data(), sizeof(WorkItem) * pl.items.size(),
                            cudaMemcpyHostToDevice, stream));
  LF_CUDA(cudaMemcpyAsync(d_cta, pl.cta_begin.data(), sizeof(int) * pl.cta_begin.size(),
                          cudaMemcpyHostToDevice, stream));
  if (n_g > 0)
    LF_CUDA(cudaMemcpyAsync(d_gidx, gidx, sizeof(int32_t) * n_g, cudaMemcpyHostToDevice, stream));
  LF_CUDA(cudaMemcpyAsync(d_isg, pl.pat->isg.data(), (size_t)L, cudaMemcpyHostToDevice, stream));
  LF_CUDA(cudaMemcpyAsync(d_gcnt, pl.pat->gcnt.data(), sizeof(int32_t) * ((size_t)L + 1),
                          cudaMemcpyHostToDevice, stream));

  MainParams prm;
  std::memset(&prm, 0, sizeof(prm));
  for (int sl = 0; sl < pl.n_slots; ++sl) {
    const int d = pl.slot_dil[sl];
    prm.dil[sl] = d;
    if ((s = map_residue(ds, &prm.tmQ[sl], q, D, L, d, BH)) != LF_OK) return s;
    if ((s = map_residue(ds, &prm.tmK[sl], k, D, L, d, BH)) != LF_OK) return s;
    if ((s = map_residue(ds, &prm.tmV[sl], v, D, L, d, BH)) != LF_OK) return s;
  }
  uint16_t* qg = reinterpret_cast<uint16_t*>(ws + off_g);
  uint16_t* kg = qg + g_elems;
  uint16_t* vg = kg + g_elems;
  if (n_g > 0) {
    if ((s = map_rows(ds, &prm.tmKp, k, D, L, BH, lf::kBN)) != LF_OK) return s;
    if ((s = map_rows(ds, &prm.tmVp, v, D, L, BH, lf::kBN)) != LF_OK) return s;
    if ((s = map_rows(ds, &prm.tmQg, qg, D, pl.NGQ, BH, lf::kBM)) != LF_OK) return s;
    if ((s = map_rows(ds, &prm.tmKg, kg, D, pl.NGQ, BH, pl.NGB)) != LF_OK) return s;
    if ((s = map_rows(ds, &prm.tmVg, vg, D, pl.NGQ, BH, pl.NGB)) != LF_OK) return s;
  }
  prm.items = d_items;
  prm.cta_begin = d_cta;
  prm.n_items = (int)pl.items.size();
  prm.gidx = d_gidx;
  prm.is_glob = d_isg;
  prm.gcnt = d_gcnt;
  prm.n_g = n_g;
  prm.NGB = pl.NGB;
  prm.NGQ = pl.NGQ;
  prm.n_chunks = pl.n_chunks;
  prm.out = out;
  prm.out_f32 = 0;
  prm.part_o = reinterpret_cast<float*>(ws + off_po);
  prm.part_ml = reinterpret_cast<float*>(ws + off_pm);
  prm.H = H;
  prm.L = L;
  prm.w = w;
  prm.sl2 = scale * 1.4426950408889634f;
  prm.status = ds->status;
  prm.wait_iters = lf::wait_iters_for(wait_timeout_ns());

  if (n_g > 0) {
    const size_t total = (size_t)BH * pl.NGQ * (D / 8);
    const int threads = 256;
    const int blocks = (int)std::max<size_t>(1, std::min<size_t>((total + threads - 1) / threads,
                                                                 (size_t)ds->num_sms * 8));
    lf::lf_gather_globals_kernel<<<blocks, threads, 0, stream>>>(
        reinterpret_cast<const uint4*>(q), reinterpret_cast<const uint4*>(k),
        reinterpret_cast<const uint4*>(v), reinterpret_cast<uint4*>(qg),
        reinterpret_cast<uint4*>(kg), reinterpret_cast<uint4*>(vg), d_gidx, n_g, pl.NGQ, L, D,
        BH);
    g_launches.fetch_add(1, std::memory_order_relaxed);
  }
  if (prm.n_items > 0) {
    const int grid = pl.grid;
    if (D == 64)
      lf::lf_attn_main_kernel<64><<<grid, lf::KCfg<64>::THREADS, lf::KCfg<64>::SMEM_BYTES, stream>>>(prm);
    else
      lf::lf_attn_main_kernel<128><<<grid, lf::KCfg<128>::THREADS, lf::KCfg<128>::SMEM_BYTES, stream>>>(prm);
    g_launches.fetch_add(1, std::memory_order_relaxed);
  }
  if (n_g > 0) {
    const int threads = 256;
    const long long warps = (long long)BH * n_g;
    const int blocks = (int)((warps + threads / 32 - 1) / (threads / 32));
    if (D == 64)
      lf::lf_combine_globals_kernel<64><<<blocks, threads, 0, stream>>>(
          prm.part_o, prm.part_ml, d_gidx, out, 0, n_g, pl.NGQ, pl.n_chunks, L, BH, nullptr);
    else
      lf::lf_combine_globals_kernel<128><<<blocks, threads, 0, stream>>>(
          prm.part_o, prm.part_ml, d_gidx, out, 0, n_g, pl.NGQ, pl.n_chunks, L, BH, nullptr);
    g_launches.fetch_add(1, std::memory_order_relaxed);
  }
  LF_CUDA(cudaGetLastError());
  return LF_OK;
}


// ------------------------------------------------------------ layer forward
//
// The Longformer layer of "基于Block-Sparse Attention的Longformer" §6, with
// the attention read as one softmax over band ∪ G per head (the attention
// above):
//   q, k, v = bf16(x W_qkv^T + b_qkv), split into H heads
//                                              (tcgen05 GEMM, head-split epilogue)
//   a       = attention(q, k, v)               (fwd_impl)
//   x1      = bf16(LN1(x + merge(a)))          (merge_ln1)
//   y       = bf16(LN2(x1 + x1 W_ff^T + b_ff)) (tcgen05 GEMM, LayerNorm epilogue
//                                               over a cluster of CTAs per row block)
// The products accumulate in fp32 in TMEM; only q, k, v, a, x1 and y are
// stored (bf16).

struct LayerWorkspace {
  uint8_t* ptr = nullptr;
  size_t bytes = 0;
};
// kept apart from the attention's scratch, which the layer's attention step
// uses at the same time
std::map<std::pair<int, cudaStream_t>, LayerWorkspace> g_layer_ws;

lf_status get_layer_workspace(int dev, cudaStream_t stream, size_t bytes, uint8_t** out) {
  std::lock_guard<std::mutex> lk(g_mu);
  LayerWorkspace& w = g_layer_ws[{dev, stream}];
  if (w.bytes < bytes) {
    if (w.ptr) LF_CUDA(cudaFreeAsync(w.ptr, stream));
    w.ptr = nullptr;
    w.bytes = 0;
    const size_t grow = align_up(bytes, size_t(1) << 20);
    LF_CUDA(cudaMallocAsync(reinterpret_cast<void**>(&w.ptr), grow, stream));
    w.bytes = grow;
  }
  *out = w.ptr;
  return LF_OK;
}

// Tile width and cluster size of the feed-forward GEMM: a row's hidden
// columns are split over `cluster` CTAs of NT columns (NT fp32 TMEM columns
// each), at most kGemmMaxCluster.
struct FfShape {
  int nt = 0, cluster = 0;
};
FfShape ff_shape(int hidden) {
  if (hidden == 64) return {64, 1};
  if (hidden % 128 == 0 && hidden / 128 <= lf::kGemmMaxCluster) return {128, hidden / 128};
  if (hidden % 256 == 0 && hidden / 256 <= lf::kGemmMaxCluster) return {256, hidden / 256};
  return {};
}

bool g_gemm_smem_set[64][8] = {};

// C = A B^T through lf_gemm_tc_kernel<NT, EPI>: A [M, K], B [N, K] bf16
// row-major (the caller sets P's output maps); grid (N / NT, row tiles):
// B * ceil(L / 128) tiles of one batch element each for EPI 0, ceil(M / 128)
// for EPI 1, with clusters of `cluster` CTAs along the columns.
template <int NT, int EPI, int MH = 1, int ST = 0>
lf_status gemm_tc(DevState* ds, int dev, lf::GemmParams& P, const void* A, const void* Bw,
                  long long M, int N, int K, int cluster, cudaStream_t stream, const char* name) {
  using CF = lf::GemmCfg<NT, MH, ST>;
  lf_status s;
  {
    const uint64_t dims[2] = {(uint64_t)K, (uint64_t)M};
    const uint64_t st[1] = {(uint64_t)K * 2};
    const uint32_t box[2] = {(uint32_t)lf::kGemmBK, (uint32_t)CF::BM};
    if ((s = encode(ds, &P.tmA, A, 2, dims, st, box)) != LF_OK) return s;
  }
  {
    const uint64_t dims[2] = {(uint64_t)K, (uint64_t)N};
    const uint64_t st[1] = {(uint64_t)K * 2};
    const uint32_t box[2] = {(uint32_t)lf::kGemmBK, (uint32_t)NT};
    if ((s = encode(ds, &P.tmB, Bw, 2, dims, st, box)) != LF_OK) return s;
  }
  P.M = (int)M;
  P.K = K;
  P.status = ds->status;
  P.wait_iters = lf::wait_iters_for(wait_timeout_ns());
  {
    std::lock_guard<std::mutex> lk(g_mu);
    const int slot = ST > 0 ? 7 : (MH == 2 ? 6 : (NT == 64 ? 0 : NT == 128 ? 1 : 2) * 2 + EPI);
    if (dev < 64 && !g_gemm_smem_set[dev][slot]) {
      LF_CUDA(cudaFuncSetAttribute(lf::lf_gemm_tc_kernel<NT, EPI, MH, ST>,
                                   cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   (int)CF::SMEM_BYTES));
      g_gemm_smem_set[dev][slot] = true;
    }
  }
  cudaLaunchConfig_t cfg = {};
  const long long row_tiles = (EPI == 0)
                                  ? (long long)P.B * ((P.L + CF::BM - 1) / CF::BM)
                                  : (M + CF::BM - 1) / CF::BM;
  cfg.gridDim = dim3((unsigned)(N / NT), (unsigned)row_tiles, 1);
  cfg.blockDim = dim3(CF::THREADS, 1, 1);
  cfg.dynamicSmemBytes = CF::SMEM_BYTES;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  if (EPI == 1) {
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)cluster;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
  }
  cudaError_t e = cudaSuccess;
  traced(name, stream, [&] { e = cudaLaunchKernelEx(&cfg, lf::lf_gemm_tc_kernel<NT, EPI, MH, ST>, P); });
  if (e != cudaSuccess) return fail(LF_ERR_CUDA, "%s launch: %s", name, cudaGetErrorString(e));
  return LF_OK;
}

lf_status layer_impl(const void* x, const void* w_qkv, const float* b_qkv, const void* w_ff,
                     const float* b_ff, const float* ln1, const float* ln2, void* out, int B, int L,
                     int hidden, int H, int w, const int32_t* dilation, const int32_t* gidx,
                     int n_g, float scale, float eps, cudaStream_t stream) {
  t_last_error.clear();
  if (B < 1 || L < 1 || H < 1 || hidden < 1)
    return fail(LF_ERR_INVALID_ARG, "B=%d, L=%d, H=%d and hidden=%d must be >= 1", B, L, H, hidden);
  if (hidden % H != 0) return fail(LF_ERR_INVALID_ARG, "hidden=%d is not a multiple of H=%d", hidden, H);
  const int D = hidden / H;
  if (D != 64 && D != 128) return fail(LF_ERR_UNSUPPORTED, "head size %d (supported: 64, 128)", D);
  const void* ptrs[8] = {x, w_qkv, b_qkv, w_ff, b_ff, ln1, ln2, out};
  for (const void* q : ptrs) {
    if (q == nullptr) return fail(LF_ERR_INVALID_ARG, "a tensor pointer is NULL");
    if (!aligned16(q)) return fail(LF_ERR_INVALID_ARG, "a tensor pointer is not 16-byte aligned");
  }
  if (!std::isfinite(eps) || !(eps > 0.f)) return fail(LF_ERR_INVALID_ARG, "eps must be finite and > 0");
  if (!std::isfinite(scale) || !(scale > 0.f)) return fail(LF_ERR_INVALID_ARG, "scale must be finite and > 0");
  lf_status s = check_pattern(H, L, w, dilation, gidx, n_g);
  if (s != LF_OK) return s;
  // the LayerNorm kernels hold a row in registers (hidden / 32 values per
  // lane); they are instantiated for these widths
  const int per2 = hidden / 64;
  if (per2 != 1 && per2 != 2 && per2 != 4 && per2 != 6 && per2 != 8 && per2 != 12 &&
      per2 != 16 && per2 != 24 && per2 != 32)
    return fail(LF_ERR_UNSUPPORTED,
                "hidden=%d (supported: 64, 128, 256, 384, 512, 768, 1024, 1536, 2048)", hidden);
  DevState* ds = nullptr;
  int dev = 0;
  if ((s = get_dev(&ds, &dev)) != LF_OK) return s;

  const long long M = (long long)B * L;
  if (M > INT32_MAX) return fail(LF_ERR_UNSUPPORTED, "B*L=%lld tokens is too many", M);
  const FfShape ff = ff_shape(hidden);
  if (ff.nt == 0) return fail(LF_ERR_UNSUPPORTED, "hidden=%d", hidden);
  const size_t act = (size_t)M * hidden;   // elements of one [B, L, hidden] activation
  size_t off = 0;
  const size_t off_qkv = off;              // bf16 3 x [B, H, L, D]
  off += align_up(act * 3 * 2, 256);
  const size_t off_a = off;                // bf16 [B, H, L, D]
  off += align_up(act * 2, 256);
  const size_t off_x1 = off;               // bf16 [M, hidden]
  off += align_up(act * 2, 256);
  uint8_t* ws = nullptr;
  if ((s = get_layer_workspace(dev, stream, off, &ws)) != LF_OK) return s;
  uint16_t* qkv = reinterpret_cast<uint16_t*>(ws + off_qkv);
  uint16_t* a = reinterpret_cast<uint16_t*>(ws + off_a);
  uint16_t* x1 = reinterpret_cast<uint16_t*>(ws + off_x1);

  // q, k, v = bf16(x W_qkv^T + b_qkv), written per head
  {
    lf::GemmParams P;
    std::memset(&P, 0, sizeof(P));
    P.hidden = hidden;
    P.bias = b_qkv;
    P.qkv = qkv;
    P.B = B;
    P.H = H;
    P.L = L;
    P.D = D;
    // 256 x 256 tiles (two accumulators) where the width allows: half the
    // L2 traffic per product of 128 x 128 tiles
    const bool wide = (3 * hidden) % 256 == 0;
    for (int part = 0; part < 3; ++part) {
      const uint64_t dims[3] = {(uint64_t)D, (uint64_t)L, (uint64_t)B * H};
      const uint64_t st[2] = {(uint64_t)D * 2, (uint64_t)D * 2 * L};
      const uint32_t box[3] = {64, (uint32_t)(wide ? 2 * lf::kGemmBM : lf::kGemmBM), 1};
      if ((s = encode(ds, &P.tmO[part], qkv + part * act, 3, dims, st, box)) != LF_OK) return s;
    }
    if (wide)
      s = gemm_tc<256, 0, 2>(ds, dev, P, x, w_qkv, M, 3 * hidden, hidden, 1, stream,
                             "layer_gemm_qkv");
    else if ((3 * hidden) % 128 == 0)
      s = gemm_tc<128, 0>(ds, dev, P, x, w_qkv, M, 3 * hidden, hidden, 1, stream, "layer_gemm_qkv");
    else
      s = gemm_tc<64, 0>(ds, dev, P, x, w_qkv, M, 3 * hidden, hidden, 1, stream, "layer_gemm_qkv");
    if (s != LF_OK) return s;
  }
  if ((s = fwd_impl(qkv, qkv + act, qkv + 2 * act, a, false, B, H, L, D, w, dilation, gidx, n_g,
                    scale, stream)) != LF_OK)
    return s;
  // x1 = bf16(LN1(x + merge(a))): one warp per row, four rows per CTA (small
  // CTAs pack into the register file with less of a tail wave), with the
  // widest vector (VW columns, NJ steps per lane) the width allows
  const int threads = 128;
  const unsigned rows_blocks = (unsigned)((M + threads / 32 - 1) / (threads / 32));
  auto launch_ln1 = [&](auto vw, auto nj) {
    constexpr int VW = decltype(vw)::value, NJ = decltype(nj)::value;
    traced("layer_merge_ln1", stream, [&] {
      lf::lf_layer_merge_ln1_kernel<VW, NJ><<<rows_blocks, threads, 0, stream>>>(
          static_cast<const uint16_t*>(x), a, ln1, x1, B, H, L, D, eps);
    });
  };
  {
    using I = std::integral_constant<int, 1>;
    switch (hidden) {
      case 64: launch_ln1(std::integral_constant<int, 2>{}, I{}); break;
      case 128: launch_ln1(std::integral_constant<int, 4>{}, I{}); break;
      case 256: launch_ln1(std::integral_constant<int, 8>{}, I{}); break;
      case 384: launch_ln1(std::integral_constant<int, 4>{}, std::integral_constant<int, 3>{}); break;
      case 512: launch_ln1(std::integral_constant<int, 8>{}, std::integral_constant<int, 2>{}); break;
      case 768: launch_ln1(std::integral_constant<int, 8>{}, std::integral_constant<int, 3>{}); break;
      case 1024: launch_ln1(std::integral_constant<int, 8>{}, std::integral_constant<int, 4>{}); break;
      case 1536: launch_ln1(std::integral_constant<int, 8>{}, std::integral_constant<int, 6>{}); break;
      default: launch_ln1(std::integral_constant<int, 8>{}, std::integral_constant<int, 8>{}); break;
    }
  }
  // y = bf16(LN2(x1 + x1 W_ff^T + b_ff))
  {
    lf::GemmParams P;
    std::memset(&P, 0, sizeof(P));
    P.hidden = hidden;
    P.bias = b_ff;
    P.resid = x1;
    P.ln = ln2;
    P.out = static_cast<uint16_t*>(out);
    P.eps = eps;
    P.L = L;
    {
      const uint64_t dims[2] = {(uint64_t)hidden, (uint64_t)M};
      const uint64_t st[1] = {(uint64_t)hidden * 2};
      const uint32_t box[2] = {64, (uint32_t)lf::kGemmBM};
      if ((s = encode(ds, &P.tmO[0], out, 2, dims, st, box)) != LF_OK) return s;
    }
    if (ff.nt == 64)
      s = gemm_tc<64, 1>(ds, dev, P, x1, w_ff, M, hidden, hidden, ff.cluster, stream, "layer_gemm_ff_ln2");
    else if (ff.nt == 128)   // two stages: three CTAs per SM, one wave for layer-base
      s = gemm_tc<128, 1, 1, 2>(ds, dev, P, x1, w_ff, M, hidden, hidden, ff.cluster, stream, "layer_gemm_ff_ln2");
    else
      s = gemm_tc<256, 1>(ds, dev, P, x1, w_ff, M, hidden, hidden, ff.cluster, stream, "layer_gemm_ff_ln2");
    if (s != LF_OK) return s;
  }
  LF_CUDA(cudaGetLastError());
  return LF_OK;
}


// ------------------------------------------------------------ backward

// Band tiles of the backward (bh, residue r, first key t0, dilation d), per
// batch size and pattern; plus the backward's own scratch (delta).
// Tiles of the backward kernel (per batch size, pattern and D): band tiles
// of 128 keys per residue class, then the global-key tiles (launched second,
// after the band tiles have stored dK and dV).
struct BwdPlan {
  lf::BtcTile* d_tiles = nullptr;
  int n_band = 0, n_gkey = 0;
  int n_slots = 0;
  int slot_dil[lf::kMaxDilSlots] = {0};
  int dmax = 1;
};
std::map<PlanKey, BwdPlan> g_bwd_plans;
std::map<std::pair<int, cudaStream_t>, LayerWorkspace> g_bwd_ws;
bool g_bwd_smem_set[64] = {false};

// query blocks per global-key tile: the head's rows are split into chunks of
// kBwdGkeyMinBlocks .. kBwdGkeyBlocks blocks, so that a few global keys still
// spread over the GPU
constexpr int kBwdGkeyBlocks = 8, kBwdGkeyMinBlocks = 2;
// resident blocks per SM of the fused prep kernel, per (device, D, global-key
// build); 0 until queried
int g_prep_occ[384] = {};

lf_status bwd_impl(const void* q, const void* k, const void* v, const void* out, const float* lse,
                   const void* dout, float* dq, float* dk, float* dv, int B, int H, int L, int D,
                   int w, const int32_t* dilation, const int32_t* gidx, int n_g, float scale,
                   cudaStream_t stream) {
  t_last_error.clear();
  if (B < 1) return fail(LF_ERR_INVALID_ARG, "B=%d must be >= 1", B);
  lf_status s = check_pattern(H, L, w, dilation, gidx, n_g);
  if (s != LF_OK) return s;
  const void* ptrs[9] = {q, k, v, out, lse, dout, dq, dk, dv};
  for (const void* x : ptrs) {
    if (x == nullptr) return fail(LF_ERR_INVALID_ARG, "a tensor pointer is NULL");
    if (!aligned16(x)) return fail(LF_ERR_INVALID_ARG, "a tensor pointer is not 16-byte aligned");
  }
  if (!std::isfinite(scale) || !(scale > 0.f)) return fail(LF_ERR_INVALID_ARG, "scale must be finite and > 0");
  if (D != 64 && D != 128) return fail(LF_ERR_UNSUPPORTED, "D=%d (supported: 64, 128)", D);
  for (int h = 0; h < H; ++h)
    if (dilation[h] > 1 && L % dilation[h] != 0)
      return fail(LF_ERR_UNSUPPORTED, "L=%d is not a multiple of dilation[%d]=%d", L, h, dilation[h]);
  if ((long long)B * H * L > INT32_MAX) return fail(LF_ERR_UNSUPPORTED, "B*H*L too large");
  DevState* ds = nullptr;
  int dev = 0;
  if ((s = get_dev(&ds, &dev)) != LF_OK) return s;
  std::shared_ptr<Pattern> pat;
  if ((s = get_pattern(dev, H, L, w, dilation, gidx, n_g, &pat)) != LF_OK) return s;
  const int QB = D == 64 ? lf::BtcCfg<64>::QB : lf::BtcCfg<128>::QB;
  const int NGQ = n_g > 0 ? ceil_div(n_g, lf::kBtcKeys) * lf::kBtcKeys : 0;
  BwdPlan* bp = nullptr;
  {
    PatKey pk{dev, H, L, w, pat->dil, pat->G, pat->xkey};
    PlanKey key{dev, B, D, pk};
    std::lock_guard<std::mutex> lk(g_mu);
    auto it = g_bwd_plans.find(key);
    if (it == g_bwd_plans.end()) {
      BwdPlan np;
      std::vector<int> head_slot(H);
      for (int h = 0; h < H; ++h) {
        int sl = 0;
        while (sl < np.n_slots && np.slot_dil[sl] != dilation[h]) ++sl;
        if (sl == np.n_slots) {
          if (np.n_slots == lf::kMaxDilSlots)
            return fail(LF_ERR_UNSUPPORTED, "more than %d distinct dilation values",
                        lf::kMaxDilSlots);
          np.slot_dil[np.n_slots++] = dilation[h];
        }
        head_slot[h] = sl;
        np.dmax = std::max(np.dmax, dilation[h]);
      }
      std::vector<lf::BtcTile> tiles;
      for (int b = 0; b < B; ++b)
        for (int h = 0; h < H; ++h) {
          const int d = dilation[h];
          for (int r = 0; r < d; ++r) {
            const int Lr = lf::residue_len(L, d, r);
            for (int t0 = 0; t0 < Lr; t0 += lf::kBtcKeys)
              tiles.push_back(lf::BtcTile{b * H + h, 0, r, t0, head_slot[h], 0, 0, 0});
          }
        }
      np.n_band = (int)tiles.size();
      // global-key tiles: query chunks short enough for a few waves of
      // resident CTAs (2 per SM at D = 64, 1 at D = 128)
      const int all_blocks = ceil_div(L, QB);
      const long long units = (long long)B * H * ceil_div(std::max(n_g, 1), lf::kBtcKeys) * all_blocks;
      const long long slots = (long long)ds->num_sms * (D == 64 ? 2 : 1);
      const int chunk = (int)std::max<long long>(
          kBwdGkeyMinBlocks, std::min<long long>(kBwdGkeyBlocks, units / (4 * slots)));
      for (int b = 0; b < B && n_g > 0; ++b)
        for (int h = 0; h < H; ++h)
          for (int g0 = 0; g0 < n_g; g0 += lf::kBtcKeys)
            for (int c = 0; c < all_blocks; c += chunk)
              tiles.push_back(lf::BtcTile{b * H + h, 1, 0, g0, head_slot[h], c * QB,
                                          std::min(chunk, all_blocks - c), 0});
      np.n_gkey = (int)tiles.size() - np.n_band;
      LF_CUDA(cudaMalloc(&np.d_tiles, sizeof(lf::BtcTile) * std::max<size_t>(tiles.size(), 1)));
      LF_CUDA(cudaMemcpy(np.d_tiles, tiles.data(), sizeof(lf::BtcTile) * tiles.size(),
                         cudaMemcpyHostToDevice));
      it = g_bwd_plans.emplace(key, np).first;
    }
    bp = &it->second;
  }
  const int BH = B * H;
  const long long rows = (long long)BH * L;
  // workspace: statistics (residue order [BH][stats_bh], gathered global
  // rows [BH][NGQ], natural order [BH][L + pad]) | gathered q, dout, k, v
  // [BH][NGQ][D]
  const long long stats_bh = (long long)L + (long long)lf::kBtcQPad * bp->dmax;
  const size_t off_stats = 0;
  const size_t off_sg = off_stats + align_up((size_t)BH * stats_bh * 16, 256);
  const size_t off_sn = off_sg + align_up((size_t)BH * NGQ * 16 + 16, 256);
  const size_t off_g = off_sn + align_up((size_t)BH * (L + lf::kBtcQPad) * 16, 256);
  const size_t g_elems = (size_t)BH * NGQ * D;
  // few global tokens: the prep kernel does the global-key pairs and sets
  // dq; their dk, dv sums go to dkg, dvg [BH][n_g][D] fp32
  // (and L at least one warp run of rows, so that a block's rows span at
  // most two heads)
  const bool fused_gk = n_g <= lf::kBwdPrepGlobals && L >= 16;
  const size_t gk_elems = fused_gk ? (size_t)BH * n_g * D : 0;
  const size_t off_gk = off_g + align_up(4 * g_elems * 2 + 16, 256);
  const size_t need = off_gk + align_up(2 * gk_elems * 4 + 16, 256);
  uint8_t* ws = nullptr;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    LayerWorkspace& wsp = g_bwd_ws[{dev, stream}];
    if (wsp.bytes < need) {
      if (wsp.ptr) LF_CUDA(cudaFreeAsync(wsp.ptr, stream));
      wsp.ptr = nullptr;
      wsp.bytes = 0;
      LF_CUDA(cudaMallocAsync(reinterpret_cast<void**>(&wsp.ptr), align_up(need, size_t(1) << 20), stream));
      wsp.bytes = align_up(need, size_t(1) << 20);
    }
    ws = wsp.ptr;
  }
  float4* stats = reinterpret_cast<float4*>(ws + off_stats);
  float4* stats_g = reinterpret_cast<float4*>(ws + off_sg);
  float4* stats_n = reinterpret_cast<float4*>(ws + off_sn);
  uint16_t* qg = reinterpret_cast<uint16_t*>(ws + off_g);
  uint16_t* og = qg + g_elems;
  uint16_t* kg = og + g_elems;
  uint16_t* vg = kg + g_elems;
  float* dkg = reinterpret_cast<float*>(ws + off_gk);
  float* dvg = dkg + gk_elems;
  const size_t grad_bytes = (size_t)rows * D * 4;
  // dq is accumulated by every tile: zeroed first, or set by the prep kernel
  // (fused_gk); dk and dv are stored by the band tiles (every key row has
  // one), with the global-key pairs' sums added either there (fused_gk) or
  // by the global-key tiles afterwards
  if (fused_gk) {
    if (gk_elems > 0) LF_CUDA(cudaMemsetAsync(dkg, 0, 2 * gk_elems * 4, stream));
  } else {
    LF_CUDA(cudaMemsetAsync(dq, 0, grad_bytes, stream));
  }

  // kernel parameters: residue views of k, v, q, dout per dilation value,
  // undilated views of q and dout, and the gathered global rows
  lf::BwdTcParams T;
  std::memset(&T, 0, sizeof(T));
  for (int sl = 0; sl < bp->n_slots; ++sl) {
    const int d = bp->slot_dil[sl];
    T.dil[sl] = d;
    if ((s = map_residue(ds, &T.tmK[sl], k, D, L, d, BH)) != LF_OK) return s;
    if ((s = map_residue(ds, &T.tmV[sl], v, D, L, d, BH)) != LF_OK) return s;
    if ((s = map_residue(ds, &T.tmQ[sl], q, D, L, d, BH, QB)) != LF_OK) return s;
    if ((s = map_residue(ds, &T.tmO[sl], dout, D, L, d, BH, QB)) != LF_OK) return s;
    if ((s = map_residue_f32(ds, &T.tmDQ[sl], dq, D, L, d, BH, QB)) != LF_OK) return s;
  }
  if (n_g > 0) {
    if ((s = map_residue(ds, &T.tmQn, q, D, L, 1, BH, QB)) != LF_OK) return s;
    if ((s = map_residue(ds, &T.tmOn, dout, D, L, 1, BH, QB)) != LF_OK) return s;
    if ((s = map_residue_f32(ds, &T.tmDQn, dq, D, L, 1, BH, QB)) != LF_OK) return s;
    if ((s = map_rows(ds, &T.tmQg, qg, D, NGQ, BH, QB)) != LF_OK) return s;
    if ((s = map_rows(ds, &T.tmOg, og, D, NGQ, BH, QB)) != LF_OK) return s;
    if ((s = map_rows(ds, &T.tmKg, kg, D, NGQ, BH, lf::kBtcKeys)) != LF_OK) return s;
    if ((s = map_rows(ds, &T.tmVg, vg, D, NGQ, BH, lf::kBtcKeys)) != LF_OK) return s;
  }
  T.tiles = bp->d_tiles;
  if (fused_gk && n_g > 0) {
    T.dkg = dkg;
    T.dvg = dvg;
    T.is_glob = pat->d_isg;
    T.gcnt = pat->d_gcnt;
  }
  T.stats = stats;
  T.stats_bh = stats_bh;
  T.stats_g = stats_g;
  T.stats_n = stats_n;
  T.gidx = pat->d_G;
  T.n_g = n_g;
  T.NGQ = NGQ;
  T.dq = dq;
  T.dk = dk;
  T.dv = dv;
  T.L = L;
  T.w = w;
  T.scale = scale;
  T.sl2 = scale * 1.4426950408889634f;
  T.status = ds->status;
  T.wait_iters = lf::wait_iters_for(wait_timeout_ns());

  auto launch_all = [&](auto dc) -> lf_status {
    constexpr int DD = decltype(dc)::value;
    using CF = lf::BtcCfg<DD>;
    {
      std::lock_guard<std::mutex> lk(g_mu);
      const int slot = dev * 2 + (DD == 128 ? 1 : 0);
      if (slot < 64 && !g_bwd_smem_set[slot]) {
        LF_CUDA(cudaFuncSetAttribute(lf::lf_bwd_band_tc_kernel<DD>,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)CF::SMEM_BYTES));
        g_bwd_smem_set[slot] = true;
      }
    }
    {
      // blocks per part: the rows, the gathered global rows, the padding
      const int pthreads = 256;
      auto nblk = [&](long long units) {
        return (int)std::max<long long>(
            1, std::min<long long>((units + pthreads - 1) / pthreads, (long long)ds->num_sms * 16));
      };
      // the rows: per thread (plain), or per run of 2 steps a warp
      // (fused_gk)
      int nb1 = nblk((long long)BH * NGQ * (DD / 8));
      int nb2 = nblk((long long)BH * 2 * lf::kBtcQPad);
      // fused_gk: a contiguous range of rows per block, at most L (two
      // heads), a multiple of the warps' 2-step runs.  The blocks of all
      // three parts are sized to be resident at once (one wave): the row
      // blocks all take about the same time, and a second wave of a few of
      // them would double the launch.  The gathered rows and the padding,
      // a few row-slices per thread, take a quarter of their one-pass blocks.
      const long long run_rows = 2 * (32 / (DD / 8));
      long long rpb = run_rows;
      if (fused_gk) {
        nb1 = std::max(1, (nb1 + 3) / 4);
        nb2 = std::max(1, (nb2 + 3) / 4);
        const int gkn = n_g <= 1 ? 0 : n_g <= 2 ? 1 : 2;
        int per_sm = 0;
        {
          std::lock_guard<std::mutex> lk(g_mu);
          const int slot = (dev * 2 + (DD == 128 ? 1 : 0)) * 3 + gkn;
          if (slot < 384 && g_prep_occ[slot] > 0) per_sm = g_prep_occ[slot];
        }
        if (per_sm == 0) {
          const void* fn = gkn == 0   ? (const void*)lf::lf_bwd_tc_prep_kernel<DD, 1>
                           : gkn == 1 ? (const void*)lf::lf_bwd_tc_prep_kernel<DD, 2>
                                      : (const void*)lf::lf_bwd_tc_prep_kernel<DD, 4>;
          LF_CUDA(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, pthreads, 0));
          per_sm = std::max(per_sm, 1);
          std::lock_guard<std::mutex> lk(g_mu);
          const int slot = (dev * 2 + (DD == 128 ? 1 : 0)) * 3 + gkn;
          if (slot < 384) g_prep_occ[slot] = per_sm;
        }
        const long long cap = (long long)ds->num_sms * per_sm;
        const long long target = std::max(cap - nb1 - nb2, std::max(cap / 2, 1LL));
        const long long want = ceil_div(ceil_div(rows, target), run_rows) * run_rows;
        rpb = std::max<long long>(run_rows, std::min<long long>(want, L) / run_rows * run_rows);
      }
      const int nb0 = fused_gk ? (int)ceil_div(rows, rpb) : nblk(rows * (DD / 8));
      traced("bwd_prep", stream, [&] {
        auto args = [&](auto kern) {
          kern<<<nb0 + nb1 + nb2, pthreads, 0, stream>>>(
              reinterpret_cast<const uint4*>(q), reinterpret_cast<const uint4*>(k),
              reinterpret_cast<const uint4*>(v), reinterpret_cast<const uint4*>(out),
              reinterpret_cast<const uint4*>(dout), lse, pat->d_isg, pat->d_dil, pat->d_G, n_g,
              NGQ, H, L, stats_bh, BH, stats, stats_n, stats_g, reinterpret_cast<uint4*>(qg),
              reinterpret_cast<uint4*>(og), reinterpret_cast<uint4*>(kg),
              reinterpret_cast<uint4*>(vg), nb0, nb1, dq, dkg, dvg, w, scale, (int)rpb);
        };
        if (!fused_gk)
          args(lf::lf_bwd_tc_prep_kernel<DD, 0>);
        else if (n_g <= 1)
          args(lf::lf_bwd_tc_prep_kernel<DD, 1>);
        else if (n_g <= 2)
          args(lf::lf_bwd_tc_prep_kernel<DD, 2>);
        else
          args(lf::lf_bwd_tc_prep_kernel<DD, 4>);
      });
    }
    if (bp->n_band > 0)
      traced("bwd_tc_band", stream, [&] {
        lf::lf_bwd_band_tc_kernel<DD><<<(unsigned)bp->n_band, CF::THREADS, CF::SMEM_BYTES,
                                        stream>>>(T);
      });
    if (bp->n_gkey > 0 && !fused_gk) {
      lf::BwdTcParams T2 = T;
      T2.tiles = bp->d_tiles + bp->n_band;
      traced("bwd_tc_global_keys", stream, [&] {
        lf::lf_bwd_band_tc_kernel<DD><<<(unsigned)bp->n_gkey, CF::THREADS, CF::SMEM_BYTES,
                                        stream>>>(T2);
      });
    }
    return LF_OK;
  };
  if (D == 64) s = launch_all(std::integral_constant<int, 64>{});
  else s = launch_all(std::integral_constant<int, 128>{});
  if (s != LF_OK) return s;
  LF_CUDA(cudaGetLastError());
  return LF_OK;
}

// lf_attn_fwd_bias: the zero-padded, 1/scale-scaled, four-way shifted copy
// of the bias table (lf_bias_pad_kernel, into a per-(device, stream)
// workspace), then the forward with the BIAS attention kernel.
std::map<std::pair<int, cudaStream_t>, LayerWorkspace> g_bias_ws;

lf_status bias_fwd_impl(const void* q, const void* k, const void* v, void* out,
                        const float* rel_bias, int B, int H, int L, int D, int w,
                        const int32_t* dilation, const int32_t* gidx, int n_g, float scale,
                        cudaStream_t stream) {
  t_last_error.clear();
  lf_status s = check_pattern(H, L, w, dilation, gidx, n_g);
  if (s != LF_OK) return s;
  if (rel_bias == nullptr || (reinterpret_cast<uintptr_t>(rel_bias) & 3u) != 0)
    return fail(LF_ERR_INVALID_ARG, "rel_bias must be a 4-byte aligned device pointer");
  if (!(scale > 0.f) || !std::isfinite(scale))
    return fail(LF_ERR_INVALID_ARG, "scale=%g must be positive and finite", (double)scale);
  int dev = 0;
  LF_CUDA(cudaGetDevice(&dev));
  if (w > (1 << 24)) return fail(LF_ERR_UNSUPPORTED, "w=%d too large for the bias table", w);
  const size_t rs = 4 * (size_t)lf::bias_row_len(w);
  if ((size_t)H * rs > (size_t)INT32_MAX) return fail(LF_ERR_UNSUPPORTED, "bias table too large");
  float* tbl = nullptr;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    LayerWorkspace& wsp = g_bias_ws[{dev, stream}];
    const size_t need = align_up((size_t)H * rs * 4, 256);
    if (wsp.bytes < need) {
      if (wsp.ptr) LF_CUDA(cudaFreeAsync(wsp.ptr, stream));
      wsp.ptr = nullptr;
      wsp.bytes = 0;
      LF_CUDA(cudaMallocAsync(reinterpret_cast<void**>(&wsp.ptr), need, stream));
      wsp.bytes = need;
    }
    tbl = reinterpret_cast<float*>(wsp.ptr);
  }
  const int n = H * (int)rs;
  traced("bias_pad", stream, [&] {
    lf::lf_bias_pad_kernel<<<(n + 255) / 256, 256, 0, stream>>>(rel_bias, tbl, H, w, 1.0f / scale);
  });
  LF_CUDA(cudaGetLastError());
  return fwd_impl(q, k, v, out, false, B, H, L, D, w, dilation, gidx, n_g, scale, stream, nullptr,
                  tbl);
}

// lf_attn_fwd_blocks: the table's shape and entries are checked here; the
// planner turns each tile's row into extra blocks of its band items.
lf_status blocks_fwd_impl(const void* q, const void* k, const void* v, void* out, int B, int H,
                          int L, int D, int w, const int32_t* dilation, const int32_t* gidx,
                          int n_g, const int32_t* xblocks, int T, int R, float scale,
                          cudaStream_t stream) {
  t_last_error.clear();
  lf_status s = check_pattern(H, L, w, dilation, gidx, n_g);
  if (s != LF_OK) return s;
  if (xblocks == nullptr || T < 1 || R < 1)
    return fail(LF_ERR_INVALID_ARG, "xblocks must be a host table [H, T, R] with T, R >= 1");
  if ((long long)H * T * R > (1LL << 28))
    return fail(LF_ERR_UNSUPPORTED, "extra-block table too large (H*T*R=%lld)",
                (long long)H * T * R);
  for (int h = 0; h < H; ++h) {
    const int d = dilation[h];
    const int nqt = ceil_div(ceil_div(L, d), lf::kBM);
    if ((long long)d * nqt > T)
      return fail(LF_ERR_INVALID_ARG, "T=%d < %d tiles of head %d (dilation %d)", T, d * nqt, h, d);
    const int32_t* tab = xblocks + (size_t)h * T * R;
    for (size_t e = 0; e < (size_t)T * R; ++e)
      if (tab[e] < -1 || tab[e] >= nqt)
        return fail(LF_ERR_INVALID_ARG, "xblocks[%d][%zu]=%d not in [-1, %d)", h, e / R, tab[e],
                    nqt);
  }
  return fwd_impl(q, k, v, out, false, B, H, L, D, w, dilation, gidx, n_g, scale, stream, nullptr,
                  nullptr, xblocks, T, R);
}

}  // namespace

// ------------------------------------------------------- host-buffer forward
//
// lf_attn_fwd_host splits the problem into chunks of whole heads of one
// batch element (each head's attention is independent of the others) and
// pipelines them over two streams of the library: while one chunk is
// computed, the next one's inputs are copied in and the previous one's
// output is copied out, so that the host link, which bounds this call,
// carries data in both directions while the GPU computes.  The streams are
// ordered after the caller's stream at entry, and the caller's stream after
// them at exit.
struct HostPipe {
  bool ready = false;
  cudaStream_t s[2] = {nullptr, nullptr};
  cudaEvent_t fork = nullptr, join[2] = {nullptr, nullptr};
};
std::vector<HostPipe> g_host_pipe;
std::mutex g_host_mu;   // one host-buffer call at a time per process (it blocks anyway)

constexpr int kHostChunks = 8;   // target number of chunks per call

lf_status fwd_host_impl(const void* q, const void* k, const void* v, void* out, bool f32, int B,
                        int H, int L, int D, int w, const int32_t* dilation,
                        const int32_t* gidx, int n_g, float scale, cudaStream_t st) {
  t_last_error.clear();
  if (!q || !k || !v || !out) return fail(LF_ERR_INVALID_ARG, "a host pointer is NULL");
  if (B < 1 || H < 1 || L < 1 || (D != 64 && D != 128))
    return fail(LF_ERR_INVALID_ARG, "bad shape B=%d H=%d L=%d D=%d", B, H, L, D);
  if (dilation == nullptr) return fail(LF_ERR_INVALID_ARG, "dilation is NULL");
  // the whole pattern is checked once here, so that a bad argument fails
  // before any copy
  lf_status s = check_pattern(H, L, w, dilation, gidx, n_g);
  if (s != LF_OK) return s;
  std::lock_guard<std::mutex> hk(g_host_mu);
  int dev = 0;
  LF_CUDA(cudaGetDevice(&dev));
  if ((int)g_host_pipe.size() <= dev) g_host_pipe.resize(dev + 1);
  HostPipe& hp = g_host_pipe[dev];
  if (!hp.ready) {
    for (int x = 0; x < 2; ++x) {
      LF_CUDA(cudaStreamCreateWithFlags(&hp.s[x], cudaStreamNonBlocking));
      LF_CUDA(cudaEventCreateWithFlags(&hp.join[x], cudaEventDisableTiming));
    }
    LF_CUDA(cudaEventCreateWithFlags(&hp.fork, cudaEventDisableTiming));
    hp.ready = true;
  }
  const size_t esz = f32 ? 4 : 2;
  const size_t head = (size_t)L * D * esz;   // bytes of one (b, h) slice
  const size_t bytes = (size_t)B * H * head;
  // heads per chunk: whole heads of one batch element, about kHostChunks
  // chunks in all
  const int per_b = std::max(1, kHostChunks / B);
  const int hc = (H + per_b - 1) / per_b;

  uint8_t* buf = nullptr;
  LF_CUDA(cudaMallocAsync(reinterpret_cast<void**>(&buf), 4 * align_up(bytes, 256), st));
  uint8_t* dq = buf;
  uint8_t* dk = dq + align_up(bytes, 256);
  uint8_t* dv = dk + align_up(bytes, 256);
  uint8_t* dout = dv + align_up(bytes, 256);
  cudaError_t e = cudaEventRecord(hp.fork, st);
  for (int x = 0; x < 2 && e == cudaSuccess; ++x) e = cudaStreamWaitEvent(hp.s[x], hp.fork, 0);
  int chunk = 0;
  for (int b = 0; b < B && e == cudaSuccess && s == LF_OK; ++b) {
    for (int h0 = 0; h0 < H && e == cudaSuccess && s == LF_OK; h0 += hc, ++chunk) {
      const int nh = std::min(hc, H - h0);
      const size_t off = ((size_t)b * H + h0) * head, n = (size_t)nh * head;
      cudaStream_t cs = hp.s[chunk & 1];
      const uint8_t* hq = static_cast<const uint8_t*>(q) + off;
      const uint8_t* hk = static_cast<const uint8_t*>(k) + off;
      const uint8_t* hv = static_cast<const uint8_t*>(v) + off;
      if ((e = cudaMemcpyAsync(dq + off, hq, n, cudaMemcpyHostToDevice, cs)) != cudaSuccess ||
          (e = cudaMemcpyAsync(dk + off, hk, n, cudaMemcpyHostToDevice, cs)) != cudaSuccess ||
          (e = cudaMemcpyAsync(dv + off, hv, n, cudaMemcpyHostToDevice, cs)) != cudaSuccess)
        break;
      s = fwd_impl(dq + off, dk + off, dv + off, dout + off, f32, 1, nh, L, D, w, dilation + h0,
                   gidx, n_g, scale, cs);
      if (s != LF_OK) break;
      e = cudaMemcpyAsync(static_cast<uint8_t*>(out) + off, dout + off, n,
                          cudaMemcpyDeviceToHost, cs);
    }
  }
  // join: the caller's stream waits for both pipeline streams, then frees
  cudaError_t ej = cudaSuccess;
  for (int x = 0; x < 2; ++x) {
    if (ej == cudaSuccess) ej = cudaEventRecord(hp.join[x], hp.s[x]);
    if (ej == cudaSuccess) ej = cudaStreamWaitEvent(st, hp.join[x], 0);
  }
  cudaFreeAsync(buf, st);
  const cudaError_t e2 = cudaStreamSynchronize(st);
  if (s != LF_OK) return s;
  if (e != cudaSuccess) return fail(LF_ERR_CUDA, "copy failed: %s", cudaGetErrorString(e));
  if (ej != cudaSuccess) return fail(LF_ERR_CUDA, "stream join: %s", cudaGetErrorString(ej));
  if (e2 != cudaSuccess) return fail(LF_ERR_CUDA, "stream: %s", cudaGetErrorString(e2));
  return LF_OK;
}

// =================================================================== C ABI

extern "C" {

lf_status lf_attn_fwd(const void* q, const void* k, const void* v, void* out, int B, int H,
                      int L, int D, int w, const int32_t* dilation, const int32_t* global_idx,
                      int n_global, float scale, lf_stream_t stream) {
  try {
    return fwd_impl(q, k, v, out, false, B, H, L, D, w, dilation, global_idx, n_global, scale,
                    static_cast<cudaStream_t>(stream));
  } catch (const std::exception& e) {
    return fail(LF_ERR_NOMEM, "host exception: %s", e.what());
  } catch (...) {
    return fail(LF_ERR_NOMEM, "host exception");
  }
}

lf_status lf_attn_fwd_bias(const void* q, const void* k, const void* v, void* out,
                           const float* rel_bias, int B, int H, int L, int D, int w,
                           const int32_t* dilation, const int32_t* global_idx, int n_global,
                           float scale, lf_stream_t stream) {
  try {
    return bias_fwd_impl(q, k, v, out, rel_bias, B, H, L, D, w, dilation, global_idx, n_global,
                         scale, static_cast<cudaStream_t>(stream));
  } catch (const std::exception& e) {
    return fail(LF_ERR_NOMEM, "host exception: %s", e.what());
  } catch (...) {
    return fail(LF_ERR_NOMEM, "host exception");
  }
}

lf_status lf_attn_fwd_blocks(const void* q, const void* k, const void* v, void* out, int B,
                             int H, int L, int D, int w, const int32_t* dilation,
                             const int32_t* global_idx, int n_global, const int32_t* xblocks,
                             int T, int R, float scale, lf_stream_t stream) {
  try {
    return blocks_fwd_impl(q, k, v, out, B, H, L, D, w, dilation, global_idx, n_global, xblocks,
                           T, R, scale, static_cast<cudaStream_t>(stream));
  } catch (const std::exception& e) {
    return fail(LF_ERR_NOMEM, "host exception: %s", e.what());
  } catch (...) {
    return fail(LF_ERR_NOMEM, "host exception");
  }
}

lf_status lf_attn_fwd_lse(const void* q, const void* k, const void* v, void* out, float* lse,
                          int B, int H, int L, int D, int w, const int32_t* dilation,
                          const int32_t* global_idx, int n_global, float scale,
                          lf_stream_t stream) {
  try {
    if (lse == nullptr || (reinterpret_cast<uintptr_t>(lse) & 15u) != 0)
      return fail(LF_ERR_INVALID_ARG, "lse must be a 16-byte aligned device pointer");
    return fwd_impl(q, k, v, out, false, B, H, L, D, w, dilation, global_idx, n_global, scale,
                    static_cast<cudaStream_t>(stream), lse);
  } catch (const std::exception& e) {
    return fail(LF_ERR_NOMEM, "host exception: %s", e.what());
  } catch (...) {
    return fail(LF_ERR_NOMEM, "host exception");
  }
}

lf_status lf_attn_bwd(const void* q, const void* k, const void* v, const void* out,
                      const float* lse, const void* dout, float* dq, float* dk, float* dv, int B,
                      int H, int L, int D, int w, const int32_t* dilation,
                      const int32_t* global_idx, int n_global, float scale, lf_stream_t stream) {
  try {
    return bwd_impl(q, k, v, out, lse, dout, dq, dk, dv, B, H, L, D, w, dilation, global_idx,
                    n_global, scale, static_cast<cudaStream_t>(stream));
  } catch (const std::exception& e) {
    return fail(LF_ERR_NOMEM, "host exception: %s", e.what());
  } catch (...) {
    return fail(LF_ERR_NOMEM, "host exception");
  }
}

lf_status lf_attn_fwd_f32(const void* q, const void* k, const void* v, void* out, int B, int H,
                          int L, int D, int w, const int32_t* dilation,
                          const int32_t* global_idx, int n_global, float scale,
                          lf_stream_t stream) {
  try {
    return fwd_impl(q, k, v, out, true, B, H, L, D, w, dilation, global_idx, n_global, scale,
                    static_cast<cudaStream_t>(stream));
  } catch (const std::exception& e) {
    return fail(LF_ERR_NOMEM, "host exception: %s", e.what());
  } catch (...) {
    return fail(LF_ERR_NOMEM, "host exception");
  }
}

lf_status lf_layer_fwd(const void* x, const void* w_qkv, const float* b_qkv, const void* w_ff,
                       const float* b_ff, const float* ln1, const float* ln2, void* out, int B,
                       int L, int hidden, int H, int w, const int32_t* dilation,
                       const int32_t* global_idx, int n_global, float scale, float eps,
                       lf_stream_t stream) {
  try {
    return layer_impl(x, w_qkv, b_qkv, w_ff, b_ff, ln1, ln2, out, B, L, hidden, H, w, dilation,
                      global_idx, n_global, scale, eps, static_cast<cudaStream_t>(stream));
  } catch (const std::exception& e) {
    return fail(LF_ERR_NOMEM, "host exception: %s", e.what());
  } catch (...) {
    return fail(LF_ERR_NOMEM, "host exception");
  }
}

lf_status lf_attn_fwd_host(const void* q, const void* k, const void* v, void* out, int is_f32,
                           int B, int H, int L, int D, int w, const int32_t* dilation,
                           const int32_t* global_idx, int n_global, float scale,
                           lf_stream_t stream) {
  try {
    return fwd_host_impl(q, k, v, out, is_f32 != 0, B, H, L, D, w, dilation, global_idx,
                         n_global, scale, static_cast<cudaStream_t>(stream));
  } catch (...) {
    return fail(LF_ERR_NOMEM, "host exception");
  }
}

lf_status lf_attn_pairs(int H, int L, int w, const int32_t* dilation, const int32_t* global_idx,
                        int n_global, int64_t* row_ptr, int32_t* col_idx, int64_t cap,
                        int64_t* total, lf_stream_t stream) {
  try {
    t_last_error.clear();
    lf_status s = check_pattern(H, L, w, dilation, global_idx, n_global);
    if (s != LF_OK) return s;
    if (row_ptr == nullptr || total == nullptr)
      return fail(LF_ERR_INVALID_ARG, "row_ptr and total must not be NULL");
    if (col_idx != nullptr && cap < 0) return fail(LF_ERR_INVALID_ARG, "cap < 0");
    DevState* ds = nullptr;
    int dev = 0;
    if ((s = get_dev(&ds, &dev)) != LF_OK) return s;
    std::shared_ptr<Pattern> pat;
    if ((s = get_pattern(dev, H, L, w, dilation, global_idx, n_global, &pat)) != LF_OK) return s;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const long long n = (long long)H * L;
    const int threads = 256;
    const int blocks = (int)std::min<long long>((n + threads - 1) / threads, ds->num_sms * 16LL);
    // counts are written into row_ptr and scanned in place
    traced("pairs_count", st, [&] {
      lf::lf_pairs_count_kernel<<<blocks, threads, 0, st>>>(pat->d_dil, pat->d_G, pat->d_isg,
                                                           n_global, H, L, w, row_ptr);
    });
    traced("pairs_scan", st, [&] { lf::lf_pairs_scan_kernel<<<1, 1024, 0, st>>>(row_ptr, row_ptr, n); });
    LF_CUDA(cudaGetLastError());
    int64_t tot = 0;
    LF_CUDA(cudaMemcpyAsync(&tot, row_ptr + n, sizeof(int64_t), cudaMemcpyDeviceToHost, st));
    LF_CUDA(cudaStreamSynchronize(st));
    *total = tot;
    if (col_idx == nullptr) return LF_OK;
    if (cap < tot)
      return fail(LF_ERR_INVALID_ARG, "col_idx capacity %lld < %lld pairs", (long long)cap,
                  (long long)tot);
    traced("pairs_fill", st, [&] {
      lf::lf_pairs_fill_kernel<<<blocks, threads, 0, st>>>(pat->d_dil, pat->d_G, pat->d_isg,
                                                          n_global, H, L, w, row_ptr, col_idx);
    });
    LF_CUDA(cudaGetLastError());
    return LF_OK;
  } catch (...) {
    return fail(LF_ERR_NOMEM, "host exception");
  }
}

const char* lf_last_error(void) { return t_last_error.c_str(); }

lf_status lf_attn_get_status(lf_stream_t stream) {
  t_last_error.clear();
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail(LF_ERR_CUDA, "stream: %s", cudaGetErrorString(e));
  unsigned word = 0;
  e = cudaMemcpyFromSymbol(&word, g_status_word, sizeof(word));
  if (e != cudaSuccess) return fail(LF_ERR_CUDA, "status read: %s", cudaGetErrorString(e));
  if (word != 0) {
    unsigned zero = 0;
    cudaMemcpyToSymbol(g_status_word, &zero, sizeof(zero));
    if (word & lf::kStatusTimeout)
      return fail(LF_ERR_TIMEOUT, "a device-side wait ran out (status word 0x%x)", word);
    return fail(LF_ERR_CUDA, "device status word 0x%x", word);
  }
  return LF_OK;
}

void lf_plan_cache_clear(void) {
  std::lock_guard<std::mutex> lk(g_mu);
  cudaDeviceSynchronize();
  g_params.clear();
  for (auto& kv : g_workspaces)
    if (kv.second.ptr) cudaFree(kv.second.ptr);
  g_workspaces.clear();
  for (auto& kv : g_layer_ws)
    if (kv.second.ptr) cudaFree(kv.second.ptr);
  g_layer_ws.clear();
  for (auto& kv : g_bwd_ws)
    if (kv.second.ptr) cudaFree(kv.second.ptr);
  g_bwd_ws.clear();
  for (auto& kv : g_bias_ws)
    if (kv.second.ptr) cudaFree(kv.second.ptr);
  g_bias_ws.clear();
  for (auto& kv : g_bwd_plans) cudaFree(kv.second.d_tiles);
  g_bwd_plans.clear();
  for (auto& kv : g_plans)
    if (kv.second->d_items) cudaFree(kv.second->d_items);
  g_plans.clear();
  for (auto& kv : g_patterns) {
    cudaFree(kv.second->d_G);
    cudaFree(kv.second->d_isg);
    cudaFree(kv.second->d_gcnt);
    cudaFree(kv.second->d_dil);
  }
  g_patterns.clear();
}

uint64_t lf_launch_count(void) { return g_launches.load(); }

void lf_profile_enable(int on) { g_trace_on.store(on ? 1 : 0); }

void lf_profile_only(const char* name) {
  std::lock_guard<std::mutex> lk(g_trace_mu);
  g_trace_only = name ? name : "";
}

void lf_profile_reset(void) {
  std::lock_guard<std::mutex> lk(g_trace_mu);
  for (auto& r : g_trace) {
    cudaEventSynchronize(r.e1);
    g_event_pool.push_back(r.e0);
    g_event_pool.push_back(r.e1);
  }
  g_trace.clear();
}

lf_status lf_profile_query(const char* name, double* total_ms, uint64_t* launches) {
  t_last_error.clear();
  if (total_ms == nullptr || launches == nullptr)
    return fail(LF_ERR_INVALID_ARG, "total_ms and launches must not be NULL");
  std::lock_guard<std::mutex> lk(g_trace_mu);
  double ms = 0.0;
  uint64_t n = 0;
  for (auto& r : g_trace) {
    if (name != nullptr && name[0] != 0 && std::strstr(r.name, name) == nullptr) continue;
    cudaError_t e = cudaEventSynchronize(r.e1);
    if (e != cudaSuccess) return fail(LF_ERR_CUDA, "event: %s", cudaGetErrorString(e));
    float x = 0.f;
    e = cudaEventElapsedTime(&x, r.e0, r.e1);
    if (e != cudaSuccess) return fail(LF_ERR_CUDA, "elapsed: %s", cudaGetErrorString(e));
    ms += x;
    ++n;
  }
  *total_ms = ms;
  *launches = n;
  return LF_OK;
}

lf_status lf_attn_fwd_noalloc(const void* q, const void* k, const void* v, void* out, int B,
                              int H, int L, int D, int w, const int32_t* dilation,
                              const int32_t* global_idx, int n_global, float scale,
                              lf_stream_t stream) {
  try {
    return fwd_noalloc_impl(q, k, v, out, B, H, L, D, w, dilation, global_idx, n_global, scale,
                            static_cast<cudaStream_t>(stream));
  } catch (const std::exception& e) {
    return fail(LF_ERR_NOMEM, "host exception: %s", e.what());
  } catch (...) {
    return fail(LF_ERR_NOMEM, "host exception");
  }
}

lf_status lf_selftest_wait_timeout(int timeout_us, lf_stream_t stream) {
  try {
    t_last_error.clear();
    if (timeout_us < 1 || timeout_us > 1000000)
      return fail(LF_ERR_INVALID_ARG, "timeout_us=%d not in [1, 1000000]", timeout_us);
    DevState* ds = nullptr;
    int dev = 0;
    lf_status s = get_dev(&ds, &dev);
    if (s != LF_OK) return s;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    lf::lf_selftest_wait_kernel<<<1, 32, 0, st>>>(ds->status,
                                                 lf::wait_iters_for(1000ull * (unsigned)timeout_us));
    g_launches.fetch_add(1, std::memory_order_relaxed);
    LF_CUDA(cudaGetLastError());
    return LF_OK;
  } catch (...) {
    return fail(LF_ERR_NOMEM, "host exception");
  }
}

int lf_version(void) { return 100; }

}  // extern "C"
