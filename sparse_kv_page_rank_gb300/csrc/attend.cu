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
// in shared memory; the CTAs of a cluster through distributed shared memory
// (after a cluster barrier, CTA rank c reads every CTA's state for output
// columns [c*128/CS, (c+1)*128/CS)); with NC > 1 the clusters of a problem
// write their partial to the workspace and the last cluster to finish (atomic
// ticket, no waiting) merges them, again one column slice per CTA.  The
// result is o (bf16) and lse (natural log).
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
  int lp;
  if (MODE == kAttendSparse) {
    if (i < cnt) {
      lp = a.sel_pages[(size_t)bh * a.k_max + i];
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
    int phys = a.block_table[(size_t)b * a.max_pages + lp];
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

  if (MODE == kAttendSparse) trace_mark(a.err, kTrAttEnter, true);
  if (tid == 0) {
    prefetch_tmap(&tk);
    if (MODE != kAttendPageLse) prefetch_tmap(&tv);
    for (int s = 0; s < STAGES; ++s) mbar_init(&bars[s], 1);
    if (MODE == kAttendSparse)
      mbar_init(reinterpret_cast<uint64_t*>(smem + STAGES * kStage + kRecvO + kRecvMl), a.cluster);
    fence_mbar_init();
  }
  __syncthreads();
  // sparse mode: every CTA's receive barrier must be initialised before any
  // other CTA of the cluster arrives on it (the matching wait comes at the merge)
  if (MODE == kAttendSparse) cluster_arrive();

  // Inside the fused step the step's own inputs (q, lengths, block table) were
  // written before its first kernel started, so they can be read while the
  // selection is still being computed; the selection itself only after the wait.
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
  const int ns_raw = (MODE == kAttendSparse) ? a.n_summarized[b] : 0;
  if (MODE == kAttendSparse && a.inputs_early) {
    // warm L2 with this sequence's block-table row while the selection is
    // still being computed (the entries are looked up right after the wait)
    const char* row = reinterpret_cast<const char*>(a.block_table + (size_t)b * a.max_pages);
    const int lines = (a.max_pages * 4 + 127) / 128;
    for (int li = tid; li < lines; li += kAttendThreads)
      asm volatile("prefetch.global.L2 [%0];\n" ::"l"(row + (size_t)li * 128));
  }
  if (a.inputs_early) pdl_wait();
  if (MODE == kAttendSparse) trace_mark(a.err, kTrAttWait, true);

  if (L < 0 || L > a.max_pages * P) {
    if (tid == 0 && split == 0) set_error(a.err, LOCKS_DEVERR_LENGTHS);
    L = L < 0 ? 0 : a.max_pages * P;
  }
  const int n_pages = (L + P - 1) / P;
  int ns = 0, cnt = 0, n_items;
  if (MODE == kAttendSparse) {
    const int cap = min(L / P, a.max_pages);
    ns = ns_raw < 0 ? 0 : (ns_raw > cap ? cap : ns_raw);
    cnt = a.sel_count[bh];
    const int kcap = min(a.k_max, ns);
    if (cnt < 0 || cnt > kcap) {
      if (tid == 0) set_error(a.err, LOCKS_DEVERR_SEL_PAGE);
      cnt = cnt < 0 ? 0 : kcap;
    }
    n_items = cnt + (n_pages - ns);
  } else {
    n_items = n_pages;
  }
  // pages per CTA: a whole number of tiles
  const int ipc = ((n_items + a.n_splits - 1) / a.n_splits + kPPT - 1) / kPPT * kPPT;
  const int i0 = min(n_items, split * ipc), i1 = min(n_items, i0 + ipc);
  const int ntile = (i1 - i0 + kPPT - 1) / kPPT;

  const uint32_t sbase = smem_u32(smem);
  // bytes one page brings into a stage (K, and V unless page-LSE mode)
  constexpr uint32_t kPageTx = (uint32_t)P * kHeadDim * 2 * (MODE == kAttendPageLse ? 1 : 2);
  // resolve items [base, base + kAttendThreads) of this CTA: selection entry
  // and block-table entry, all threads at once
  auto resolve = [&](int base) {
    const int i = i0 + base + tid;
    const int buf = (base / kAttendThreads) & 1;
    if (i < i1) {
      const Item it = get_item<MODE, P>(a, i, b, bh, L, ns, cnt);
      it_phys[buf][tid] = it.phys;
      it_len[buf][tid] = it.len;
      it_lp[buf][tid] = it.lp;
    }
  };
  resolve(0);
  __syncthreads();
  if (MODE == kAttendSparse) trace_mark(a.err, kTrAttResolved, false);
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
  if (tid == 0) {
    for (int s = 0; s < STAGES && s < ntile; ++s) issue(s, s);
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
    if (MODE == kAttendSparse && it == 0) trace_mark(a.err, kTrAttFirstData, false);
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
  if (MODE == kAttendSparse) trace_mark(a.err, kTrAttLooped, false);

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

  if (MODE == kAttendSparse) trace_mark(a.err, kTrAttCtaMerged, false);
  // ---- merge the CTAs of the cluster through distributed shared memory ----
  const int CS = a.cluster, NC = a.n_splits / a.cluster;
  const uint32_t rank = cluster_ctarank();
  if (MODE == kAttendSparse) {
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
    cluster_wait();  // every CTA's receive barrier is initialised
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
    if (MODE == kAttendSparse) trace_mark(a.err, kTrAttClusterMerged, false);
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
    if (MODE == kAttendSparse) trace_mark(a.err, kTrAttExit, false);
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
    if (MODE == kAttendSparse) trace_mark(a.err, kTrAttClusterMerged, false);
    cluster_sync();  // no CTA leaves while others still read its shared memory
    if (MODE == kAttendSparse) trace_mark(a.err, kTrAttExit, false);
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
  return (size_t)STAGES * kStage + 1024 + (MODE == kAttendSparse ? kRecvBytes : 0);
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

}  // namespace

int attend_active_clusters(int mode, int cs, int page_size) {
  static int cache[2][2][5][64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64 || cs < 1 || cs > 16) return 1;
  const int m = mode == kAttendSparse ? 0 : 1, p16 = page_size == 16 ? 1 : 0;
  const int li = 31 - __builtin_clz((unsigned)cs);
  int& slot = cache[p16][m][li][dev];
  if (slot == 0) {
    int n;
    if (p16)
      n = mode == kAttendSparse ? active_clusters_of<kAttendSparse, kSparseStages, 16>(cs)
                                : active_clusters_of<kAttendDense, kDenseStages, 16>(cs);
    else
      n = mode == kAttendSparse ? active_clusters_of<kAttendSparse, kSparseStages, kPage>(cs)
                                : active_clusters_of<kAttendDense, kDenseStages, kPage>(cs);
    slot = n > 0 ? n : -1;
  }
  return slot > 0 ? slot : 0;
}

int attend_max_cluster(int mode, int page_size) {
  static int cache[2][2][64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 8;
  const int m = mode == kAttendSparse ? 0 : 1, p16 = page_size == 16 ? 1 : 0;
  int& slot = cache[p16][m][dev];
  if (slot == 0) {
    if (p16)
      slot = mode == kAttendSparse ? max_cluster_of<kAttendSparse, kSparseStages, 16>()
                                   : max_cluster_of<kAttendDense, kDenseStages, 16>();
    else
      slot = mode == kAttendSparse ? max_cluster_of<kAttendSparse, kSparseStages, kPage>()
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
    default: return launch_mode<kAttendPageLse, kDenseStages, P>(a, tk, tv, s, pdl);
  }
}

cudaError_t launch_attend(const AttendArgs& a, const CUtensorMap& tk, const CUtensorMap& tv, int mode,
                          cudaStream_t s, bool pdl) {
  return a.page_size == 16 ? launch_page<16>(a, tk, tv, mode, s, pdl) : launch_page<kPage>(a, tk, tv, mode, s, pdl);
}

}  // namespace locks
