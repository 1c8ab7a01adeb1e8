// Paged flash-decode over a page list.
//
// Sparse mode: exact attention over the selected pages plus the open tail
// (LOCKS abstract: "attends only the top pages"; blog "Ringkasan spektral per
// halaman": only the top pages are processed).  Dense mode: every page of
// every sequence (the in-library baseline).  Page-LSE mode: the exact
// per-page log-sum-exp that reads every key (the "read-every-key exact-LSE
// oracle" the abstract measures selection against).
//
// Work split: grid (CS * NC, B*Hkv) with thread-block clusters of CS CTAs
// (NC clusters per problem).  The page list of problem bh (sel_pages[0..cnt)
// then the tail pages, or every page) is cut into CS*NC contiguous ranges.  A
// CTA of four warps streams its pages through a shared-memory ring: one thread
// issues 2-D TMA loads (cp.async.bulk.tensor, 64 x 64 bf16 boxes, 128-byte
// swizzle) of the page's K and V tiles (16 KiB each) and an mbarrier with a
// transaction count tells the warps when they have landed.  Warp w owns tokens
// 16w..16w+15 of every page: S = Q K^T on tensor cores (m16n8k16, M = the
// G <= 16 query heads of the group), an online base-2 softmax in registers,
// then O += P V with P reused from the accumulator layout and V fragments read
// by ldmatrix.trans.
//
// Merging partial softmax states (max m, sum l, O): the four warps of a CTA
// in shared memory; then the CTAs of a cluster through distributed shared
// memory, CTA rank c owning output columns [c*128/CS, (c+1)*128/CS).  With a
// page list (one cluster per problem) each CTA pushes its state for those
// columns into their owner's shared memory and arrives on the owner's barrier,
// and each owner merges what it received (nobody reads remote memory, so no
// CTA waits for the others before it exits).  For every page (dense mode)
// each CTA reads the cluster's states after a cluster barrier; with NC > 1
// the clusters of a problem write their partial to the workspace and the last
// cluster to finish (atomic ticket, no waiting) merges them, again one column
// slice per CTA.  The result is o (bf16) and lse (natural log).
//
// 16-token pages (the explainer's §2 "Kernmechanisme" page size): a tile is
// four pages, loaded as four 16-row boxes into the rows 16w..16w+15 that warp
// w already owns, so the inner loop is the 64-token one and each warp masks
// by its own page's length.  The CTA ranges are cut on tile boundaries.
#include "common.cuh"
#include "kernels.h"

namespace locks {

namespace {

constexpr int kWarps = kAttendThreads / 32;
constexpr int kHalfTile = 64 * 128;        // bytes of one 64-row x 64-col bf16 box
constexpr int kTile = 2 * kHalfTile;       // one page-head of K (or V): 16 KiB
constexpr int kStage = 2 * kTile;          // K + V
constexpr int kOStride = 132;              // padded row of the per-warp O buffer (floats)
constexpr int kOctaOff = kWarps * 16 * kOStride * 4;  // CTA-level O [16][128] after the warp buffers
// Sparse mode: what the other CTAs of the cluster push to this one, after the
// stage ring (never aliased): O columns [rank][head][cols], (m, l) [rank][head]
// and the barrier their arrivals complete.
constexpr int kRecvO = 16 * kHeadDim * 4;
constexpr int kRecvMl = 16 * 16 * 8;
constexpr int kRecvBytes = kRecvO + kRecvMl + 16;

__device__ __forceinline__ uint32_t tile_addr(uint32_t base, int row, int chunk16) {
  // 128B swizzle: 16-byte chunk index XOR (row mod 8) within each 128-byte row
  const int half = chunk16 >> 3, cc = chunk16 & 7;
  return base + half * kHalfTile + row * 128 + ((cc ^ (row & 7)) << 4);
}

struct Item {
  int lp;     // logical page, -1 = invalid
  int phys;   // physical page (0 when invalid)
  int len;    // valid tokens in the page (0 when invalid)
};

template <int MODE, int P>
__device__ __forceinline__ Item get_item(const AttendArgs& a, int i, int b, int bh, int L, int ns,
                                         int cnt) {
  Item it;
  int lp, phys = -1;
  bool known = false;  // physical page already given with the selection
  if (MODE == kAttendSparse) {
    if (i < cnt) {
      lp = a.sel_pages[(size_t)bh * a.k_max + i];
      if (a.sel_phys) {  // loaded alongside, not after, the logical page
        phys = a.sel_phys[(size_t)bh * a.k_max + i];
        known = true;
      }
      if (lp < 0 || lp >= ns) {
        set_error(a.err, LOCKS_DEVERR_SEL_PAGE);
        lp = -1;
      }
    } else {
      lp = ns + (i - cnt);
    }
  } else {
    lp = i;
  }
  it.lp = lp;
  it.phys = 0;
  it.len = 0;
  if (lp >= 0) {
    if (!known) phys = a.block_table[(size_t)b * a.max_pages + lp];
    if (phys < 0 || phys >= a.pages_total) {
      set_error(a.err, LOCKS_DEVERR_BLOCK_TABLE);
      it.lp = -1;
    } else {
      it.phys = phys;
      int rem = L - lp * P;
      it.len = rem < P ? rem : P;
    }
  }
  return it;
}

// Tracing builds: this CTA's timestamp for `slot` (0..15) of the page-list modes.
__device__ __forceinline__ void trace_cta(const AttendArgs& a, int slot) {
#if LOCKS_TRACE
  if (threadIdx.x == 0 && a.trace_cta) {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    a.trace_cta[((size_t)blockIdx.y * gridDim.x + blockIdx.x) * 16 + slot] = t;
  }
#else
  (void)a;
  (void)slot;
#endif
}

// Fused mode: the cluster's own page selection.  Lives after the receive area
// of the cluster merge in dynamic shared memory (same offset in every CTA, so
// the candidate lists can be written across the cluster).
struct FusedShared {
  unsigned long long comb[4 * kAttendThreads];  // (key << 32) | ~page; local keys, then the filtered set
  int phys[kAttendThreads];                     // physical page of each local key
  float z[16];                                  // Z_h (natural log) per head
  unsigned long long sel_comb[kFusedMaxK];
  int sel_phys[kFusedMaxK];
  int fsel_lp[kFusedMaxK], fsel_phys[kFusedMaxK];  // the selection, ascending page order
  unsigned long long thresh;
  int f_count;
  unsigned short f_idx[16 * kFusedMaxK];
  uint4 cand[16][kFusedMaxK];  // every CTA's candidates: {comb lo, comb hi, phys, 0}, descending comb
};

__device__ __forceinline__ unsigned long long cand_comb(const uint4& v) {
  return ((unsigned long long)v.y << 32) | v.x;
}

// Group-shared page scores and top-k for one (sequence, KV head) problem,
// computed by the CS CTAs of its cluster (explainer §2 "Group-Shared
// Selection": sigma_j = ln((1/G) sum_h exp(s_hat[h][j] - Z_h)), the k pages of
// largest sigma, ties to the lower page).  CTA c scores pages [c ppc,
// (c+1) ppc) (ppc <= kAttendThreads: one page per thread) and ranks them
// against each other; its k best (key, page, physical page) go to every CTA
// of the cluster.  Every CTA then merges the CS sorted lists the same way: a
// lower bound T on the k-th largest key (the k-th largest of each list's first
// ceil(k / CS) entries) filters the candidates, the survivors are ranked
// against each other, and the k winners are put in ascending page order in
// fs.fsel_lp / fs.fsel_phys.  Called by every thread of every CTA of the
// cluster; cluster barrier phase 1 has been arrived at (not waited on).
__device__ void cluster_select(const AttendArgs& a, int b, int bh, int ns, int k, int CS, uint32_t crank,
                               FusedShared& fs) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int G = a.group;
  const int ppc = (ns + CS - 1) / CS;
  const int j = (int)crank * ppc + tid;
  const bool valid = tid < ppc && j < ns;
  // one round trip: this thread's s_hat row and block-table entry, and the
  // scan partials of up to four heads per warp
  float sv[16];
#pragma unroll
  for (int h = 0; h < 16; ++h) sv[h] = 0.f;
  int phys = -1;
  if (valid) {
    const float* row = a.shat + ((size_t)bh * a.max_pages + j) * G;
    if ((G & 3) == 0) {
#pragma unroll
      for (int h4 = 0; h4 < 4; ++h4) {
        if (4 * h4 < G) {
          const float4 v = __ldcg(reinterpret_cast<const float4*>(row) + h4);
          sv[4 * h4] = v.x;
          sv[4 * h4 + 1] = v.y;
          sv[4 * h4 + 2] = v.z;
          sv[4 * h4 + 3] = v.w;
        }
      }
    } else {
#pragma unroll
      for (int h = 0; h < 16; ++h)
        if (h < G) sv[h] = __ldcg(row + h);
    }
    phys = __ldg(a.block_table + (size_t)b * a.max_pages + j);
  }
  {
    const float2* pb = a.part + (size_t)bh * a.n_scan_chunks * G;
#pragma unroll
    for (int hh = 0; hh < 4; ++hh) {
      const int h = warp + 4 * hh;  // warp-uniform
      if (h < G) {
        float m = -INFINITY, l = 0.f;
        for (int i = lane; i < a.n_scan_chunks; i += 32) {
          const float2 v = __ldcg(pb + (size_t)i * G + h);
          lse2_merge(m, l, v.x, v.y);
        }
#pragma unroll
        for (int o = 16; o; o >>= 1) {
          const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
          const float l2 = __shfl_xor_sync(0xffffffffu, l, o);
          lse2_merge(m, l, m2, l2);
        }
        if (lane == 0) fs.z[h] = (m + fast_log2(l)) * kLn2;
      }
    }
  }
  __syncthreads();
  trace_mark(a.err, kTrTopkLoaded, false);
  trace_cta(a, 2);
  // sigma_j -> order-preserving key; (key, ~page) orders by key, then lower page
  unsigned long long mine = 0ull;
  if (valid) {
    const float log2G = log2f((float)G);
    float y[16];
    float mx = -INFINITY;
#pragma unroll
    for (int h = 0; h < 16; ++h) {
      y[h] = h < G ? fmaf(sv[h], kLog2e, -fs.z[h] * kLog2e) : -INFINITY;
      mx = fmaxf(mx, y[h]);
    }
    float acc = 0.f;
#pragma unroll
    for (int h = 0; h < 16; ++h) acc += h < G ? fast_exp2(y[h] - mx) : 0.f;
    const uint32_t key = orderable_key((mx + fast_log2(acc) - log2G) * kLn2);
    mine = ((unsigned long long)key << 32) | (0xffffffffu - (uint32_t)j);
  }
  fs.comb[tid] = mine;  // zero for a thread without a page: below every real entry
  fs.phys[tid] = phys;
  __syncthreads();
  trace_mark(a.err, kTrSelMinMax, false);
  trace_cta(a, 3);
  // rank among this CTA's pages; the k best go to every CTA of the cluster
  const int n_local = max(0, min(ns - (int)crank * ppc, ppc));
  const int kl = min(k, n_local);
  int rank = kAttendThreads;
  if (valid) {
    rank = 0;
    const ulonglong2* c2 = reinterpret_cast<const ulonglong2*>(fs.comb);
#pragma unroll 8
    for (int v = 0; v < kAttendThreads / 2; ++v) {
      const ulonglong2 x = c2[v];
      rank += (x.x > mine) + (x.y > mine);
    }
  }
  // the CTA's few best pages are likely selected: start bringing their K and
  // V into L2 now, while the cluster agrees on the selection
  if (rank < kFusedPrefetch && rank < kl && phys >= 0 && phys < a.pages_total) {
    const size_t ph = ((size_t)phys * a.num_kv_heads + (size_t)(bh % a.num_kv_heads)) * kPage * kHeadDim;
    prefetch_l2_bulk(a.k_pool16 + ph, kPage * kHeadDim * 2);
    prefetch_l2_bulk(a.v_pool16 + ph, kPage * kHeadDim * 2);
  }
  trace_mark(a.err, kTrSelRadix, false);
  trace_cta(a, 4);
  cluster_wait();  // phase 1: every CTA of the cluster is running and set up
  trace_mark(a.err, kTrSelCompact, false);
  trace_cta(a, 5);
  if (rank < kl) {
    const uint4 rec = make_uint4((uint32_t)mine, (uint32_t)(mine >> 32), (uint32_t)phys, 0u);
    const uint32_t dst = smem_u32(&fs.cand[crank][rank]);
    for (int r = 0; r < CS; ++r) st_dsmem_u4(dsmem_addr(dst, (uint32_t)r), rec);
  }
  cluster_arrive();  // phase 2: release this CTA's candidate stores
  cluster_wait();
  trace_mark(a.err, kTrTopkKeys, false);
  trace_cta(a, 6);
  // ---- merge (identical in every CTA) ----
  // T = the k-th largest of the lists' first m entries (m as large as keeps
  // one entry per thread) is a lower bound on the k-th largest candidate;
  // the candidates >= T are then ranked against each other.
  auto kl_of = [&](int c) { return min(k, max(0, min(ns - c * ppc, ppc))); };
  const int m = min(k, kAttendThreads / CS);
  int usz = 0;
  for (int c = 0; c < CS; ++c) usz += min(m, kl_of(c));
  unsigned long long uv = 0ull;
  if (tid < usz) {
    int t = tid, c = 0;
    while (t >= min(m, kl_of(c))) {
      t -= min(m, kl_of(c));
      ++c;
    }
    uv = cand_comb(fs.cand[c][t]);
  }
  fs.comb[tid] = uv;
  if (tid == 0) fs.f_count = 0;
  __syncthreads();
  unsigned long long T = 0ull;
  if (usz >= k) {
    if (tid < usz) {
      int rk = 0;
      const ulonglong2* c2 = reinterpret_cast<const ulonglong2*>(fs.comb);
#pragma unroll 8
      for (int v = 0; v < kAttendThreads / 2; ++v) {
        const ulonglong2 x = c2[v];
        rk += (x.x > uv) + (x.y > uv);
      }
      if (rk == k - 1) fs.thresh = uv;
    }
    __syncthreads();
    T = fs.thresh;
  }
  trace_mark(a.err, kTrSelPasses, false);
  trace_cta(a, 7);
  // compact the candidates >= T (warp-aggregated slots)
  for (int e0 = 0; e0 < CS * kFusedMaxK; e0 += kAttendThreads) {
    const int e = e0 + tid;
    bool keep = false;
    unsigned long long v = 0ull;
    if (e < CS * kFusedMaxK) {
      const int c = e / kFusedMaxK, p = e % kFusedMaxK;
      if (p < kl_of(c)) {
        v = cand_comb(fs.cand[c][p]);
        keep = v >= T;
      }
    }
    const unsigned msk = __ballot_sync(0xffffffffu, keep);
    int base = 0;
    if (lane == 0 && msk) base = atomicAdd(&fs.f_count, __popc(msk));
    base = __shfl_sync(0xffffffffu, base, 0);
    if (keep) {
      const int slot = base + __popc(msk & ((1u << lane) - 1u));
      fs.comb[slot] = v;
      fs.f_idx[slot] = (unsigned short)e;
    }
  }
  __syncthreads();
  const int nf = fs.f_count;
  for (int f = tid; f < nf; f += kAttendThreads) {
    const unsigned long long v = fs.comb[f];
    int rk = 0;
    for (int f2 = 0; f2 < nf; ++f2) rk += fs.comb[f2] > v;
    if (rk < k) {
      const int e = fs.f_idx[f];
      fs.sel_comb[rk] = v;
      fs.sel_phys[rk] = (int)fs.cand[e / kFusedMaxK][e % kFusedMaxK].z;
    }
  }
  __syncthreads();
  trace_mark(a.err, kTrSelCalls, false);
  trace_cta(a, 8);
  if (tid < k) {
    const int lp = (int)(0xffffffffu - (uint32_t)fs.sel_comb[tid]);
    int pos = 0;
    for (int i = 0; i < k; ++i) pos += (int)(0xffffffffu - (uint32_t)fs.sel_comb[i]) < lp;
    fs.fsel_lp[pos] = lp;
    fs.fsel_phys[pos] = fs.sel_phys[tid];
  }
  __syncthreads();
  trace_mark(a.err, kTrTopkSelected, false);
}

template <int MODE, int STAGES, int P>
__global__ void __launch_bounds__(kAttendThreads) attend_kernel(const __grid_constant__ CUtensorMap tk,
                                                                const __grid_constant__ CUtensorMap tv,
                                                                const AttendArgs a) {
  constexpr int kPPT = kPage / P;                  // pages per 64-token tile: 1 or 4
  constexpr int kTilesPerBatch = kAttendThreads / kPPT;  // tiles whose pages one resolve() covers
  static_assert(kPPT == 1 || kPPT == kWarps, "one page per warp at P = 16");
  static_assert(STAGES <= kTilesPerBatch, "the tiles in flight span at most two resolved batches");
  extern __shared__ uint8_t dyn_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(dyn_raw) + 1023) & ~uintptr_t(1023));
  __shared__ __align__(8) uint64_t bars[STAGES];
  __shared__ float sm_m[kWarps][16], sm_l[kWarps][16];
  __shared__ float2 sm_pl[STAGES][kWarps][16];
  __shared__ float cta_m[16], cta_l[16];
  __shared__ float rk_m[16][16], rk_l[16][16];  // (rank, head) states of the cluster
  __shared__ int s_last;
  // items of this CTA resolved in parallel (one per thread, in batches)
  // (double-buffered so that the next batch can be resolved while the
  // current one is still being consumed)
  __shared__ int it_phys[2][kAttendThreads], it_len[2][kAttendThreads], it_lp[2][kAttendThreads];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, c = lane & 3;
  const int split = blockIdx.x, bh = blockIdx.y;
  const int b = bh / a.num_kv_heads, hkv = bh % a.num_kv_heads;
  const int G = a.group, Hq = a.num_kv_heads * G;

  constexpr bool FUSED = MODE == kAttendFused;
  constexpr bool SPL = MODE == kAttendSparse || FUSED;  // a page list, one cluster per problem
  if (SPL) trace_mark(a.err, kTrAttEnter, true);
  trace_cta(a, 0);
  if (tid == 0) {
    prefetch_tmap(&tk);
    if (MODE != kAttendPageLse) prefetch_tmap(&tv);
    for (int s = 0; s < STAGES; ++s) mbar_init(&bars[s], 1);
    if (SPL) mbar_init(reinterpret_cast<uint64_t*>(smem + STAGES * kStage + kRecvO + kRecvMl), a.cluster);
    fence_mbar_init();
  }
  __syncthreads();
  // page-list modes: every CTA's receive barrier must be initialised before
  // any other CTA of the cluster arrives on it or writes to it (the matching
  // wait comes at the selection or at the merge)
  if (SPL) cluster_arrive();

  // Inside the fused step the step's own inputs (q, lengths, block table, the
  // cache pages) were written before its first kernel started, so they can be
  // read while the selection is still being computed; the selection itself
  // only after the wait.
  if (!a.inputs_early) pdl_wait();

  // Q fragments (rows = heads of the group; rows >= G are zero)
  uint32_t qf[8][4];
  {
    const uint16_t* qb = a.q + ((size_t)b * Hq + (size_t)hkv * G) * kHeadDim;
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
      const int d0 = 16 * kk + 2 * c;
      qf[kk][0] = (g < G) ? __ldg(reinterpret_cast<const uint32_t*>(qb + g * kHeadDim + d0)) : 0u;
      qf[kk][1] = (g + 8 < G) ? __ldg(reinterpret_cast<const uint32_t*>(qb + (g + 8) * kHeadDim + d0)) : 0u;
      qf[kk][2] = (g < G) ? __ldg(reinterpret_cast<const uint32_t*>(qb + g * kHeadDim + d0 + 8)) : 0u;
      qf[kk][3] =
          (g + 8 < G) ? __ldg(reinterpret_cast<const uint32_t*>(qb + (g + 8) * kHeadDim + d0 + 8)) : 0u;
    }
  }
  int L = a.seq_lens[b];
  const int ns_raw = SPL ? a.n_summarized[b] : 0;
  if (SPL && a.inputs_early) {
    // warm L2 with this sequence's block-table row while the selection is
    // still being computed (the entries are looked up right after the wait)
    const char* row = reinterpret_cast<const char*>(a.block_table + (size_t)b * a.max_pages);
    const int lines = (a.max_pages * 4 + 127) / 128;
    for (int li = tid; li < lines; li += kAttendThreads)
      asm volatile("prefetch.global.L2 [%0];\n" ::"l"(row + (size_t)li * 128));
  }

  const uint32_t sbase = smem_u32(smem);
  // bytes one page brings into a stage (K, and V unless page-LSE mode)
  constexpr uint32_t kPageTx = (uint32_t)P * kHeadDim * 2 * (MODE == kAttendPageLse ? 1 : 2);
  int ns = 0, cnt = 0, n_items = 0, n_tail = 0, i0 = 0, i1 = 0, ntile = 0;
  bool sel_needed = false;  // fused mode: more summarised pages than the budget holds
  FusedShared* fsp = reinterpret_cast<FusedShared*>(smem + STAGES * kStage + kRecvBytes);  // fused mode only
  auto clamp_lengths = [&]() {
    if (L < 0 || L > a.max_pages * P) {
      if (tid == 0 && split == 0) set_error(a.err, LOCKS_DEVERR_LENGTHS);
      L = L < 0 ? 0 : a.max_pages * P;
    }
  };
  // pages per CTA: a whole number of tiles
  auto set_range = [&]() {
    const int ipc = ((n_items + a.n_splits - 1) / a.n_splits + kPPT - 1) / kPPT * kPPT;
    i0 = min(n_items, split * ipc);
    i1 = min(n_items, i0 + ipc);
    ntile = (i1 - i0 + kPPT - 1) / kPPT;
  };
  // fused mode, item i: the open tail first (pages ns, ns + 1, ...), then the
  // selected pages in ascending order (all summarised pages when they fit)
  auto fused_item = [&](int i) {
    Item it;
    it.lp = -1;
    it.phys = 0;
    it.len = 0;
    int lp, phys = 0;
    bool lookup = true;
    if (i < n_tail) {
      lp = ns + i;
    } else if (sel_needed) {
      lp = fsp->fsel_lp[i - n_tail];
      phys = fsp->fsel_phys[i - n_tail];
      lookup = false;
    } else {
      lp = i - n_tail;
    }
    if (lookup) phys = a.block_table[(size_t)b * a.max_pages + lp];
    if (phys < 0 || phys >= a.pages_total) {
      set_error(a.err, LOCKS_DEVERR_BLOCK_TABLE);
      return it;
    }
    it.lp = lp;
    it.phys = phys;
    const int rem = L - lp * P;
    it.len = rem < P ? rem : P;
    return it;
  };
  // resolve items [base, base + kAttendThreads) of this CTA: selection entry
  // and block-table entry, all threads at once
  auto resolve = [&](int base) {
    const int i = i0 + base + tid;
    const int buf = (base / kAttendThreads) & 1;
    if (i < i1) {
      Item it;
      if constexpr (FUSED)
        it = fused_item(i);
      else
        it = get_item<MODE, P>(a, i, b, bh, L, ns, cnt);
      it_phys[buf][tid] = it.phys;
      it_len[buf][tid] = it.len;
      it_lp[buf][tid] = it.lp;
    }
  };
  // thread 0 only; the pages of tile t must lie in the resolved batch.
  // Page w of a tile lands in rows 16w.. of each 64-row half-tile (byte
  // offset 2048 w, a multiple of the 1024-byte swizzle period).
  auto issue = [&](int stage, int t) {
    const int np = min(kPPT, i1 - i0 - t * kPPT);
    uint8_t* dst = smem + stage * kStage;
    mbar_arrive_expect_tx(&bars[stage], kPageTx * (uint32_t)np);
    for (int w = 0; w < np; ++w) {
      const int k = t * kPPT + w;
      const int y = (it_phys[(k / kAttendThreads) & 1][k % kAttendThreads] * a.num_kv_heads + hkv) * P;
      uint8_t* d = dst + w * (P * 128);
      tma_load_2d(d, &tk, &bars[stage], 0, y);
      tma_load_2d(d + kHalfTile, &tk, &bars[stage], 64, y);
      if (MODE != kAttendPageLse) {
        tma_load_2d(d + kTile, &tv, &bars[stage], 0, y);
        tma_load_2d(d + kTile + kHalfTile, &tv, &bars[stage], 64, y);
      }
    }
  };
  int n_pre = 0;  // tiles issued before the selection
  if constexpr (FUSED) {
    // the page list's shape depends on the lengths only (inputs of the step)
    clamp_lengths();
    const int n_pages = (L + P - 1) / P;
    const int cap = min(L / P, a.max_pages);
    ns = ns_raw < 0 ? 0 : (ns_raw > cap ? cap : ns_raw);
    sel_needed = a.k_max > 0 && ns > a.k_max;
    cnt = min(a.k_max, ns);
    n_tail = n_pages - ns;
    n_items = n_tail + cnt;
    set_range();
    // the open tail needs no selection: its first tiles load during the wait
    if (i0 + tid < i1 && i0 + tid < n_tail) resolve(0);
    __syncthreads();
    n_pre = min(min(STAGES, ntile), max(0, n_tail - i0));
    if (tid == 0)
      for (int t = 0; t < n_pre; ++t) issue(t, t);
    pdl_wait();
    trace_mark(a.err, kTrAttWait, true);
    trace_cta(a, 1);
    if (sel_needed) cluster_select(a, b, bh, ns, a.k_max, a.cluster, cluster_ctarank(), *fsp);
    if (i0 + tid < i1 && i0 + tid >= n_tail) resolve(0);
    if (cluster_ctarank() == 0) {
      // publish the page list (callers may read it back)
      for (int i = tid; i < cnt; i += kAttendThreads)
        a.sel_pages_out[(size_t)bh * a.k_max + i] = sel_needed ? fsp->fsel_lp[i] : i;
      if (tid == 0) a.sel_count_out[bh] = cnt;
    }
    __syncthreads();
  } else {
    if (a.inputs_early) pdl_wait();
    if (SPL) trace_mark(a.err, kTrAttWait, true);
    clamp_lengths();
    const int n_pages = (L + P - 1) / P;
    int cnt_written = 0;
    if (MODE == kAttendSparse) {
      const int cap = min(L / P, a.max_pages);
      ns = ns_raw < 0 ? 0 : (ns_raw > cap ? cap : ns_raw);
      const int kcap = min(a.k_max, ns);
      if (a.inputs_early) {
        // inside the decode step the top-k writes exactly min(k_max, ns)
        // pages, so the page list is read without first waiting for the
        // count; the count it wrote is loaded alongside and checked
        cnt = kcap;
        cnt_written = a.sel_count[bh];
      } else {
        cnt = a.sel_count[bh];
        if (cnt < 0 || cnt > kcap) {
          if (tid == 0) set_error(a.err, LOCKS_DEVERR_SEL_PAGE);
          cnt = cnt < 0 ? 0 : kcap;
        }
      }
      n_items = cnt + (n_pages - ns);
    } else {
      n_items = n_pages;
    }
    set_range();
    resolve(0);
    if (MODE == kAttendSparse && a.inputs_early && tid == 0 && cnt_written != cnt) set_error(a.err, LOCKS_DEVERR_SEL_PAGE);
    __syncthreads();
  }
  if (SPL) trace_mark(a.err, kTrAttResolved, false);
  trace_cta(a, 9);
  if (tid == 0) {
    for (int s = n_pre; s < STAGES && s < ntile; ++s) issue(s, s);
  }

  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
  bool failed = false;
  int consumed = 0;
  float o[16][4];
#pragma unroll
  for (int i = 0; i < 16; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;

  for (int it = 0; it < ntile; ++it) {
    const int stage = it % STAGES;
    const uint32_t parity = (it / STAGES) & 1;
    // this warp's page (the tile's only page at P = 64)
    const int wk = it * kPPT + (kPPT > 1 ? warp : 0);
    const bool w_in = wk < i1 - i0;
    const int item_len = w_in ? it_len[(wk / kAttendThreads) & 1][wk % kAttendThreads] : 0;
    const int item_lp = kPPT > 1 ? 0 : it_lp[(wk / kAttendThreads) & 1][wk % kAttendThreads];
    const bool ok = mbar_wait(&bars[stage], parity);
    if (__syncthreads_or(!ok)) {
      if (tid == 0) set_error(a.err, kDevErrTimeout);
      failed = true;
      break;
    }
    consumed = it + 1;
    if (SPL && it == 0) trace_mark(a.err, kTrAttFirstData, false);
    if (SPL && it == 0) trace_cta(a, 10);
    const uint32_t kb = sbase + stage * kStage;
    const uint32_t vb = kb + kTile;

    // S = Q K^T for this warp's 16 tokens
    float s[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
    {
      const int mi = lane >> 3;
      const int row = 16 * warp + (mi >> 1) * 8 + (lane & 7);
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        uint32_t b0, b1, b2, b3;
        ldmatrix_x4(b0, b1, b2, b3, tile_addr(kb, row, 2 * kk + (mi & 1)));
        mma_16816(s[0], qf[kk][0], qf[kk][1], qf[kk][2], qf[kk][3], b0, b1);
        mma_16816(s[1], qf[kk][0], qf[kk][1], qf[kk][2], qf[kk][3], b2, b3);
      }
    }
    // valid rows of the tile for this warp: tokens 16w .. 16w + len of its page
    const int len = kPPT > 1 ? 16 * warp + item_len : item_len;
    float tm0 = -INFINITY, tm1 = -INFINITY;
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int tok = 16 * warp + 8 * nt + 2 * c + e;
        const bool valid = tok < len;
        s[nt][e] = valid ? s[nt][e] * a.scale_log2 : -INFINITY;
        s[nt][2 + e] = valid ? s[nt][2 + e] * a.scale_log2 : -INFINITY;
        tm0 = fmaxf(tm0, s[nt][e]);
        tm1 = fmaxf(tm1, s[nt][2 + e]);
      }
    }
    tm0 = fmaxf(tm0, __shfl_xor_sync(0xffffffffu, tm0, 1));
    tm0 = fmaxf(tm0, __shfl_xor_sync(0xffffffffu, tm0, 2));
    tm1 = fmaxf(tm1, __shfl_xor_sync(0xffffffffu, tm1, 1));
    tm1 = fmaxf(tm1, __shfl_xor_sync(0xffffffffu, tm1, 2));

    if (MODE == kAttendPageLse) {
      float p0 = 0.f, p1 = 0.f;
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          p0 += (tm0 == -INFINITY) ? 0.f : fast_exp2(s[nt][e] - tm0);
          p1 += (tm1 == -INFINITY) ? 0.f : fast_exp2(s[nt][2 + e] - tm1);
        }
      p0 += __shfl_xor_sync(0xffffffffu, p0, 1);
      p0 += __shfl_xor_sync(0xffffffffu, p0, 2);
      p1 += __shfl_xor_sync(0xffffffffu, p1, 1);
      p1 += __shfl_xor_sync(0xffffffffu, p1, 2);
      if (c == 0) {
        sm_pl[stage][warp][g] = make_float2(tm0, p0);
        sm_pl[stage][warp][g + 8] = make_float2(tm1, p1);
      }
    } else {
      const float mn0 = fmaxf(m0, tm0), mn1 = fmaxf(m1, tm1);
      const float al0 = (mn0 == -INFINITY) ? 1.f : fast_exp2(m0 - mn0);
      const float al1 = (mn1 == -INFINITY) ? 1.f : fast_exp2(m1 - mn1);
      float p[2][4];
      float ps0 = 0.f, ps1 = 0.f;
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          p[nt][e] = (mn0 == -INFINITY) ? 0.f : fast_exp2(s[nt][e] - mn0);
          p[nt][2 + e] = (mn1 == -INFINITY) ? 0.f : fast_exp2(s[nt][2 + e] - mn1);
          ps0 += p[nt][e];
          ps1 += p[nt][2 + e];
        }
      l0 = l0 * al0 + ps0;
      l1 = l1 * al1 + ps1;
      m0 = mn0;
      m1 = mn1;
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        o[i][0] *= al0;
        o[i][1] *= al0;
        o[i][2] *= al1;
        o[i][3] *= al1;
      }
      // zero V rows past the sequence end (their slots may hold anything)
      if (len < kPage) {
        for (int row = max(len, 16 * warp); row < 16 * warp + 16; ++row) {
          uint8_t* vrow = smem + stage * kStage + kTile + row * 128;
          *reinterpret_cast<uint32_t*>(vrow + lane * 4) = 0u;
          *reinterpret_cast<uint32_t*>(vrow + kHalfTile + lane * 4) = 0u;
        }
        __syncwarp();
      }
      const uint32_t pa0 = pack_bf16(p[0][0], p[0][1]);
      const uint32_t pa1 = pack_bf16(p[0][2], p[0][3]);
      const uint32_t pa2 = pack_bf16(p[1][0], p[1][1]);
      const uint32_t pa3 = pack_bf16(p[1][2], p[1][3]);
      const int mi = lane >> 3;
      const int row = 16 * warp + (mi & 1) * 8 + (lane & 7);
#pragma unroll
      for (int dn = 0; dn < 8; ++dn) {
        uint32_t v0, v1, v2, v3;
        ldmatrix_x4_trans(v0, v1, v2, v3, tile_addr(vb, row, 2 * dn + (mi >> 1)));
        mma_16816(o[2 * dn], pa0, pa1, pa2, pa3, v0, v1);
        mma_16816(o[2 * dn + 1], pa0, pa1, pa2, pa3, v2, v3);
      }
    }

    fence_proxy_async();
    __syncthreads();
    if (MODE == kAttendPageLse) {
      if (kPPT == 1) {
        if (tid < G && item_lp >= 0) {
          float mm = -INFINITY, ll = 0.f;
#pragma unroll
          for (int w = 0; w < kWarps; ++w) lse2_merge(mm, ll, sm_pl[stage][w][tid].x, sm_pl[stage][w][tid].y);
          a.page_lse[((size_t)b * Hq + (size_t)hkv * G + tid) * a.max_pages + item_lp] =
              (mm == -INFINITY) ? -INFINITY : (mm + fast_log2(ll)) * kLn2;
        }
      } else if (tid < kWarps * G) {
        // one page per warp: its own (max, sum) is the page's
        const int w = tid / G, h = tid % G, k = it * kPPT + w;
        const int lp = k < i1 - i0 ? it_lp[(k / kAttendThreads) & 1][k % kAttendThreads] : -1;
        if (lp >= 0) {
          const float2 ml = sm_pl[stage][w][h];
          a.page_lse[((size_t)b * Hq + (size_t)hkv * G + h) * a.max_pages + lp] =
              (ml.x == -INFINITY) ? -INFINITY : (ml.x + fast_log2(ml.y)) * kLn2;
        }
      }
    }
    // next batch of item descriptors once the current one has been issued
    const int nxt = it + STAGES;
    if (nxt % kTilesPerBatch == 0 && nxt < ntile) {
      resolve(nxt * kPPT);
      __syncthreads();
    }
    if (tid == 0 && nxt < ntile) issue(stage, nxt);
  }

  if (failed) {
    // give copies still in flight a bounded time to land before the ring is reused
    if (tid == 0) {
      for (int it = consumed; it < consumed + STAGES && it < ntile; ++it)
        (void)mbar_wait(&bars[it % STAGES], (it / STAGES) & 1);
    }
    __syncthreads();
    m0 = m1 = -INFINITY;
    l0 = l1 = 0.f;
  }
  pdl_launch_dependents();
  if (MODE == kAttendPageLse) return;
  if (SPL) trace_mark(a.err, kTrAttLooped, false);
  trace_cta(a, 11);

  // ---- merge the four warps of this CTA ----
  l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
  l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
  float* so = reinterpret_cast<float*>(smem);              // [kWarps][16][kOStride]
  float* octa = reinterpret_cast<float*>(smem + kOctaOff);  // [16][128]
  if (c == 0) {
    sm_m[warp][g] = m0;
    sm_l[warp][g] = l0;
    sm_m[warp][g + 8] = m1;
    sm_l[warp][g + 8] = l1;
  }
#pragma unroll
  for (int nt = 0; nt < 16; ++nt) {
    const int col = 8 * nt + 2 * c;
    *reinterpret_cast<float2*>(so + (warp * 16 + g) * kOStride + col) = make_float2(o[nt][0], o[nt][1]);
    *reinterpret_cast<float2*>(so + (warp * 16 + g + 8) * kOStride + col) = make_float2(o[nt][2], o[nt][3]);
  }
  __syncthreads();
  // per head: the max over the warps and each warp's rescale factor, once
  __shared__ float sm_f[kWarps][16];
  if (tid < G) {
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) M = fmaxf(M, sm_m[w][tid]);
    float Ls = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      const float f = (M == -INFINITY) ? 0.f : fast_exp2(sm_m[w][tid] - M);
      sm_f[w][tid] = f;
      Ls += sm_l[w][tid] * f;
    }
    cta_m[tid] = M;
    cta_l[tid] = Ls;
  }
  __syncthreads();
  for (int e = tid; e < G * (kHeadDim / 4); e += kAttendThreads) {
    const int h = e / (kHeadDim / 4), d4 = 4 * (e % (kHeadDim / 4));
    float4 O = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      const float f = sm_f[w][h];
      const float4 v = *reinterpret_cast<const float4*>(so + (w * 16 + h) * kOStride + d4);
      O.x = fmaf(v.x, f, O.x);
      O.y = fmaf(v.y, f, O.y);
      O.z = fmaf(v.z, f, O.z);
      O.w = fmaf(v.w, f, O.w);
    }
    *reinterpret_cast<float4*>(octa + h * kHeadDim + d4) = O;
  }
  __syncthreads();

  if (SPL) trace_mark(a.err, kTrAttCtaMerged, false);
  trace_cta(a, 12);
  // ---- merge the CTAs of the cluster through distributed shared memory ----
  const int CS = a.cluster, NC = a.n_splits / a.cluster;
  const uint32_t rank = cluster_ctarank();
  if (SPL) {
    // One cluster per problem.  Each CTA pushes its partial state to the
    // CTAs that own its output columns (rank r owns columns [r*cols,
    // (r+1)*cols)) and arrives on their receive barriers; each CTA then
    // waits for all CS contributions and merges its columns from its own
    // shared memory.  Nobody reads another CTA's memory, so no CTA has to
    // wait for the others before it exits.
    const int cols = kHeadDim / CS;
    float* recv_o = reinterpret_cast<float*>(smem + STAGES * kStage);
    float2* recv_ml = reinterpret_cast<float2*>(smem + STAGES * kStage + kRecvO);
    uint64_t* recv_bar = reinterpret_cast<uint64_t*>(smem + STAGES * kStage + kRecvO + kRecvMl);
    // every CTA's receive barrier is initialised (already waited for when the
    // cluster selected the pages itself)
    if (!(FUSED && sel_needed)) cluster_wait();
    const uint32_t ro = smem_u32(recv_o), rml = smem_u32(recv_ml);
    for (int e = tid; e < G * (kHeadDim / 4); e += kAttendThreads) {
      const int h = e / (kHeadDim / 4), c4 = 4 * (e % (kHeadDim / 4));
      const int dst = c4 / cols, cc = c4 % cols;
      const float4 v = *reinterpret_cast<const float4*>(octa + h * kHeadDim + c4);
      st_dsmem_f4(dsmem_addr(ro + 4 * (((int)rank * G + h) * cols + cc), dst), v);
    }
    for (int e = tid; e < CS * G; e += kAttendThreads) {
      const int dst = e / G, h = e % G;
      st_dsmem_f2(dsmem_addr(rml + 8 * ((int)rank * 16 + h), dst), make_float2(cta_m[h], cta_l[h]));
    }
    __syncthreads();  // the whole CTA's stores precede the release arrivals
    if (tid < CS) mbar_arrive_remote(dsmem_addr(smem_u32(recv_bar), tid));
    if (!mbar_wait_cluster(recv_bar, 0) && tid == 0) set_error(a.err, kDevErrTimeout);
    if (SPL) trace_mark(a.err, kTrAttClusterMerged, false);
    trace_cta(a, 13);
    for (int e = tid; e < G * cols; e += kAttendThreads) {
      const int h = e / cols, cc = e % cols, col = (int)rank * cols + cc;
      float M = -INFINITY;
      for (int rr = 0; rr < CS; ++rr) M = fmaxf(M, recv_ml[rr * 16 + h].x);
      float Ls = 0.f, O = 0.f;
      if (M != -INFINITY) {
        for (int rr = 0; rr < CS; ++rr) {
          const float2 ml = recv_ml[rr * 16 + h];
          const float f = fast_exp2(ml.x - M);
          Ls += ml.y * f;
          O += recv_o[(rr * G + h) * cols + cc] * f;
        }
      }
      const size_t oi = ((size_t)b * Hq + (size_t)hkv * G + h);
      const float val = Ls > 0.f ? O / Ls : 0.f;
      a.out[oi * kHeadDim + col] = __bfloat16_as_ushort(__float2bfloat16_rn(val));
      if (a.lse && col == 0) a.lse[oi] = (Ls > 0.f) ? (M + fast_log2(Ls)) * kLn2 : -INFINITY;
    }
    if (SPL) trace_mark(a.err, kTrAttExit, false);
    trace_cta(a, 14);
    return;
  }
  const int q = split / CS;
  const int cols = kHeadDim / CS, c0 = (int)rank * cols;
  cluster_sync();
  const uint32_t am = smem_u32(cta_m), al = smem_u32(cta_l), ao = smem_u32(octa);
  // every rank's (max, sum) per head, fetched once, all loads in parallel
  for (int e = tid; e < CS * G; e += kAttendThreads) {
    const int rr = e / G, h = e % G;
    rk_m[rr][h] = ld_dsmem(dsmem_addr(am + 4 * h, rr));
    rk_l[rr][h] = ld_dsmem(dsmem_addr(al + 4 * h, rr));
  }
  __syncthreads();
  for (int e = tid; e < G * cols; e += kAttendThreads) {
    const int h = e / cols, col = c0 + e % cols;
    float ov[16];
#pragma unroll
    for (int rr = 0; rr < 16; ++rr) ov[rr] = rr < CS ? ld_dsmem(dsmem_addr(ao + 4 * (h * kHeadDim + col), rr)) : 0.f;
    float M = -INFINITY;
#pragma unroll
    for (int rr = 0; rr < 16; ++rr)
      if (rr < CS) M = fmaxf(M, rk_m[rr][h]);
    float Ls = 0.f, O = 0.f;
    if (M != -INFINITY) {
#pragma unroll
      for (int rr = 0; rr < 16; ++rr) {
        if (rr < CS) {
          const float f = fast_exp2(rk_m[rr][h] - M);
          Ls += rk_l[rr][h] * f;
          O += ov[rr] * f;
        }
      }
    }
    const size_t oi = ((size_t)b * Hq + (size_t)hkv * G + h);
    if (NC == 1) {
      const float val = Ls > 0.f ? O / Ls : 0.f;
      a.out[oi * kHeadDim + col] = __bfloat16_as_ushort(__float2bfloat16_rn(val));
      if (a.lse && col == 0) a.lse[oi] = (Ls > 0.f) ? (M + fast_log2(Ls)) * kLn2 : -INFINITY;
    } else {
      const size_t pi = ((size_t)bh * NC + q) * G + h;
      a.part_o[pi * kHeadDim + col] = O;
      if (rank == 0 && col == c0) a.part_ml[pi] = make_float2(M, Ls);
    }
  }
  if (NC == 1) {
    if (SPL) trace_mark(a.err, kTrAttClusterMerged, false);
    trace_cta(a, 13);
    cluster_sync();  // no CTA leaves while others still read its shared memory
    if (SPL) trace_mark(a.err, kTrAttExit, false);
    trace_cta(a, 14);
    return;
  }

  // ---- several clusters per problem: the last one to finish merges ----
  __threadfence();
  cluster_sync();
  if (rank == 0 && tid == 0) {
    const int last = atomicAdd(a.counters + bh, 1u) == (unsigned)(NC - 1);
    for (int rr = 0; rr < CS; ++rr) st_dsmem(dsmem_addr(smem_u32(&s_last), rr), last);
  }
  cluster_sync();
  if (!s_last) return;
  __threadfence();
  for (int e = tid; e < G * cols; e += kAttendThreads) {
    const int h = e / cols, col = c0 + e % cols;
    const size_t p0 = (size_t)bh * NC * G + h;
    float M = -INFINITY;
    for (int qq = 0; qq < NC; ++qq) M = fmaxf(M, __ldcg(a.part_ml + p0 + (size_t)qq * G).x);
    float Ls = 0.f, O = 0.f;
    if (M != -INFINITY) {
      for (int qq = 0; qq < NC; ++qq) {
        const float2 ml = __ldcg(a.part_ml + p0 + (size_t)qq * G);
        const float f = fast_exp2(ml.x - M);
        Ls += ml.y * f;
        O += __ldcg(a.part_o + (p0 + (size_t)qq * G) * kHeadDim + col) * f;
      }
    }
    const size_t oi = ((size_t)b * Hq + (size_t)hkv * G + h);
    const float val = Ls > 0.f ? O / Ls : 0.f;
    a.out[oi * kHeadDim + col] = __bfloat16_as_ushort(__float2bfloat16_rn(val));
    if (a.lse && col == 0) a.lse[oi] = (Ls > 0.f) ? (M + fast_log2(Ls)) * kLn2 : -INFINITY;
  }
  if (rank == 0 && tid == 0) a.counters[bh] = 0;  // ready for the next call
}

template <int MODE, int STAGES>
size_t smem_bytes() {
  return (size_t)STAGES * kStage + 1024 + (MODE == kAttendSparse ? kRecvBytes : 0) +
         (MODE == kAttendFused ? kRecvBytes + sizeof(FusedShared) : 0);
}

template <int MODE, int STAGES, int P>
cudaError_t launch_mode(const AttendArgs& a, const CUtensorMap& tk, const CUtensorMap& tv, cudaStream_t s,
                        bool pdl) {
  const size_t smem = smem_bytes<MODE, STAGES>();
  auto kern = attend_kernel<MODE, STAGES, P>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  if (a.cluster > 8) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.n_splits, a.batch * a.num_kv_heads, 1);
  cfg.blockDim = dim3(kAttendThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  int na = 0;
  attr[na].id = cudaLaunchAttributeClusterDimension;
  attr[na].val.clusterDim.x = MODE == kAttendPageLse ? 1 : a.cluster;
  attr[na].val.clusterDim.y = 1;
  attr[na].val.clusterDim.z = 1;
  ++na;
  if (pdl) {
    attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
  }
  cfg.attrs = attr;
  cfg.numAttrs = na;
  return cudaLaunchKernelEx(&cfg, kern, tk, tv, a);
}

// How many clusters of cs CTAs of this kernel the device can hold at once
// (0 when it cannot place one).
template <int MODE, int STAGES, int P>
int active_clusters_of(int cs) {
  auto kern = attend_kernel<MODE, STAGES, P>;
  const size_t smem = smem_bytes<MODE, STAGES>();
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess) return 0;
  if (cs > 8 && cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess)
    return 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(cs, 1, 1);
  cfg.blockDim = dim3(kAttendThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = cs;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) {
    (void)cudaGetLastError();
    return 0;
  }
  return n;
}

// Largest cluster size (16, 8, ... 1) the device can place for this kernel.
template <int MODE, int STAGES, int P>
int max_cluster_of() {
  auto kern = attend_kernel<MODE, STAGES, P>;
  const size_t smem = smem_bytes<MODE, STAGES>();
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess) return 1;
  for (int cs = 16; cs > 1; cs /= 2) {
    if (cs > 8 && cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess)
      continue;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(cs, 1, 1);
    cfg.blockDim = dim3(kAttendThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = cs;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) == cudaSuccess && n > 0) return cs;
    (void)cudaGetLastError();
  }
  return 1;
}

constexpr int kSparseStages = 3;
constexpr int kDenseStages = 2;
// fused: two stages keep two CTAs per SM with the selection's shared memory
// (each CTA of a problem's cluster holds about two selected pages)
constexpr int kFusedStages = 2;

// index of a mode in the occupancy caches
int mode_slot(int mode) { return mode == kAttendSparse ? 0 : (mode == kAttendFused ? 2 : 1); }

}  // namespace

int attend_active_clusters(int mode, int cs, int page_size) {
  static int cache[2][3][5][64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64 || cs < 1 || cs > 16) return 1;
  const int m = mode_slot(mode), p16 = page_size == 16 ? 1 : 0;
  if (m == 2 && p16) return 0;
  const int li = 31 - __builtin_clz((unsigned)cs);
  int& slot = cache[p16][m][li][dev];
  if (slot == 0) {
    int n;
    if (p16)
      n = m == 0 ? active_clusters_of<kAttendSparse, kSparseStages, 16>(cs)
                 : active_clusters_of<kAttendDense, kDenseStages, 16>(cs);
    else
      n = m == 0   ? active_clusters_of<kAttendSparse, kSparseStages, kPage>(cs)
          : m == 2 ? active_clusters_of<kAttendFused, kFusedStages, kPage>(cs)
                   : active_clusters_of<kAttendDense, kDenseStages, kPage>(cs);
    slot = n > 0 ? n : -1;
  }
  return slot > 0 ? slot : 0;
}

int attend_max_cluster(int mode, int page_size) {
  static int cache[2][3][64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 8;
  const int m = mode_slot(mode), p16 = page_size == 16 ? 1 : 0;
  if (m == 2 && p16) return 1;
  int& slot = cache[p16][m][dev];
  if (slot == 0) {
    if (p16)
      slot = m == 0 ? max_cluster_of<kAttendSparse, kSparseStages, 16>() : max_cluster_of<kAttendDense, kDenseStages, 16>();
    else
      slot = m == 0   ? max_cluster_of<kAttendSparse, kSparseStages, kPage>()
             : m == 2 ? max_cluster_of<kAttendFused, kFusedStages, kPage>()
                      : max_cluster_of<kAttendDense, kDenseStages, kPage>();
  }
  return slot;
}

template <int P>
cudaError_t launch_page(const AttendArgs& a, const CUtensorMap& tk, const CUtensorMap& tv, int mode,
                        cudaStream_t s, bool pdl) {
  switch (mode) {
    case kAttendSparse: return launch_mode<kAttendSparse, kSparseStages, P>(a, tk, tv, s, pdl);
    case kAttendDense: return launch_mode<kAttendDense, kDenseStages, P>(a, tk, tv, s, pdl);
    case kAttendFused:
      if constexpr (P == kPage) return launch_mode<kAttendFused, kFusedStages, P>(a, tk, tv, s, pdl);
      return cudaErrorInvalidValue;  // 64-token pages only
    default: return launch_mode<kAttendPageLse, kDenseStages, P>(a, tk, tv, s, pdl);
  }
}

cudaError_t launch_attend(const AttendArgs& a, const CUtensorMap& tk, const CUtensorMap& tv, int mode,
                          cudaStream_t s, bool pdl) {
  return a.page_size == 16 ? launch_page<16>(a, tk, tv, mode, s, pdl) : launch_page<kPage>(a, tk, tv, mode, s, pdl);
}

}  // namespace locks
