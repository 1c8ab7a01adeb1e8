// Group-shared page scores and top-k page selection.
//
// LOCKS explainer (gist.science), §2 "Group-Shared Selection (GSA)": the
// estimated mass share of each page is averaged over the query heads of a GQA
// group, giving one selection table per KV head; §2 "Reconstructie en
// Selectie": pages are ranked by estimated mass and no candidate key or value
// is read.  With Z_h = ln sum_j exp(s_hat[h][j]) (head h's total estimated
// mass) the score of page j is
//     sigma_j = ln( (1/G) sum_h exp(s_hat[h][j] - Z_h) ),
// and the k = min(k_max, n_summarized) pages of largest sigma are kept, ties
// to the lower page index, written in ascending page order.
//
// Parallel structure (one launch):
//   * grid (n_chunks, B*Hkv); CTA (chunk, bh) owns pages
//     [chunk*chunk_pages, (chunk+1)*chunk_pages) of problem bh;
//   * Z_h from the scan's per-CTA (max, sum) partials (warp per head);
//   * sigma_j for the chunk -> 32-bit order-preserving keys, held in
//     registers (a thread's pages) and in shared memory;
//   * one 2048-bin histogram of the top 11 bits in which the keys differ
//     finds the bin holding the k-th largest key; the keys of that bin are
//     ranked against each other (key descending, page ascending) and the
//     chosen pages are numbered in page order with warp ballots, so the output
//     is already sorted ascending and ties go to lower pages.  A boundary bin
//     of more than 512 keys (many equal keys) falls back to an MSB-first 8-bit
//     radix select over the differing bits and an ordered block scan;
//   * inside the decode step a one-chunk problem also writes each chosen
//     page's physical id, from a block-table row it loads before its
//     grid-dependency wait;
//   * the chunk's candidates go to the workspace; the last CTA of the problem
//     to finish (atomic ticket, no waiting) reruns the same select over all
//     candidates, which are laid out in page order, and writes the page list.
#include "common.cuh"
#include "kernels.h"

namespace locks {

namespace {

constexpr int kWarps = kTopkThreads / 32;

// Block-wide exclusive scan of one int per thread (kTopkThreads threads).
__device__ __forceinline__ int block_exclusive_scan(int v, int* sm_warp, int& total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) sm_warp[warp] = x;
  __syncthreads();
  int base = 0, tot = 0;
#pragma unroll
  for (int w = 0; w < kWarps; ++w) {
    int t = sm_warp[w];
    if (w < warp) base += t;
    tot += t;
  }
  __syncthreads();
  total = tot;
  return base + x - v;
}

struct SelectShared {
  unsigned hist[kWarps][256];  // one row per warp: no atomics shared across warps
  unsigned total[256];
  int warp_tmp[kWarps];
  unsigned wmin[kWarps], wmax[kWarps];
  unsigned bucket;
  unsigned remaining;
};

// Choose the k largest of keys[0..n) (ties -> lower position) and call
// emit(position_in_output, i) for each chosen i, positions in array order.
template <typename Emit>
__device__ void block_select(const uint32_t* keys, int n, int k, SelectShared& sh, Emit emit,
                             int* select_trace_err = nullptr) {
  const int tid = threadIdx.x;
  if (k <= 0 || n <= 0) return;
  uint32_t T = 0;
  unsigned need_eq = 0;
  const bool take_all = k >= n;
  unsigned long long tc0 = trace_clock(), tc1 = tc0, tc2 = tc0;
  int npass = 0;
  if (!take_all) {
    // only the bits below the highest bit where the keys differ need radix
    // passes: the keys' range [min, max] fixes the others
    unsigned lo = 0xffffffffu, hi = 0u;
    for (int i = tid; i < n; i += kTopkThreads) {
      const uint32_t key = keys[i];
      lo = min(lo, key);
      hi = max(hi, key);
    }
    lo = __reduce_min_sync(0xffffffffu, lo);
    hi = __reduce_max_sync(0xffffffffu, hi);
    if ((tid & 31) == 0) {
      sh.wmin[tid >> 5] = lo;
      sh.wmax[tid >> 5] = hi;
    }
    __syncthreads();
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      lo = min(lo, sh.wmin[w]);
      hi = max(hi, sh.wmax[w]);
    }
    const int nbits = (lo == hi) ? 0 : 32 - __clz(lo ^ hi);
    const int passes = (nbits + 7) / 8;
    npass = passes;
    tc1 = trace_clock();
    const uint32_t lowmask = passes >= 4 ? 0xffffffffu : ((1u << (8 * passes)) - 1u);
    uint32_t prefix = lo & ~lowmask, mask = ~lowmask;
    unsigned rem = (unsigned)k;
    for (int shift = 8 * (passes - 1); shift >= 0; shift -= 8) {
      for (int i = tid; i < kWarps * 256; i += kTopkThreads) (&sh.hist[0][0])[i] = 0;
      __syncthreads();
      // histogram of the next digit among keys matching the prefix so far
      const int n_round = (n + kTopkThreads - 1) / kTopkThreads * kTopkThreads;
      for (int i = tid; i < n_round; i += kTopkThreads) {
        unsigned digit = 256u;
        if (i < n) {
          const uint32_t key = keys[i];
          if ((key & mask) == prefix) digit = (key >> shift) & 255u;
        }
        // lanes agreeing with lane 0 (the common case) add once
        const unsigned lead = __shfl_sync(0xffffffffu, digit, 0);
        const unsigned same = __ballot_sync(0xffffffffu, digit == lead);
        unsigned* row = sh.hist[threadIdx.x >> 5];
        if ((threadIdx.x & 31) == 0 && lead < 256u) atomicAdd(&row[lead], __popc(same));
        if (digit != lead && digit < 256u) atomicAdd(&row[digit], 1u);
      }
      __syncthreads();
      for (int bin = tid; bin < 256; bin += kTopkThreads) {
        unsigned t = 0;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) t += sh.hist[w][bin];
        sh.total[bin] = t;
      }
      __syncthreads();
      if (tid < 32) {
        // lane l owns buckets 8l .. 8l+7; count of keys in buckets above its range
        unsigned cnt[8], tot = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) { cnt[i] = sh.total[8 * tid + i]; tot += cnt[i]; }
        unsigned incl = tot;  // sum over lanes >= tid
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          unsigned y = __shfl_down_sync(0xffffffffu, incl, o);
          if (tid + o < 32) incl += y;
        }
        unsigned above = incl - tot;
        if (above < rem && rem <= incl) {
          unsigned run = above;
#pragma unroll
          for (int i = 7; i >= 0; --i) {
            if (run < rem && rem <= run + cnt[i]) {
              sh.bucket = 8 * tid + i;
              sh.remaining = rem - run;
            }
            run += cnt[i];
          }
        }
      }
      __syncthreads();
      prefix |= sh.bucket << shift;
      mask |= 255u << shift;
      rem = sh.remaining;
      __syncthreads();
    }
    T = prefix;
    need_eq = rem;
    tc2 = trace_clock();
  }
  // blocked ranges in array order
  const int ipt = (n + kTopkThreads - 1) / kTopkThreads;
  const int i0 = min(n, tid * ipt), i1 = min(n, i0 + ipt);
  int total;
  int eq_base = 0;
  if (!take_all) {
    int eq = 0;
    for (int i = i0; i < i1; ++i) eq += keys[i] == T;
    eq_base = block_exclusive_scan(eq, sh.warp_tmp, total);
  }
  int takes = 0;
  {
    int e = eq_base;
    for (int i = i0; i < i1; ++i) {
      uint32_t key = keys[i];
      bool t = take_all || key > T || (key == T && (unsigned)e < need_eq);
      if (!take_all && key == T) ++e;
      takes += t;
    }
  }
  int pos = block_exclusive_scan(takes, sh.warp_tmp, total);
  {
    int e = eq_base;
    for (int i = i0; i < i1; ++i) {
      uint32_t key = keys[i];
      bool t = take_all || key > T || (key == T && (unsigned)e < need_eq);
      if (!take_all && key == T) ++e;
      if (t) emit(pos++, i);
    }
  }
  if (tid == 0) {
    const unsigned long long tc3 = trace_clock();
    trace_add(select_trace_err, kTrSelMinMax, tc1 - tc0);
    trace_add(select_trace_err, kTrSelRadix, tc2 - tc1);
    trace_add(select_trace_err, kTrSelCompact, tc3 - tc2);
    trace_add(select_trace_err, kTrSelPasses, (unsigned long long)npass);
    trace_add(select_trace_err, kTrSelCalls, 1ull);
  }
}

// Faster selection for the common case, with the keys in registers: key u
// of thread t is element t + kTopkThreads * u.  One histogram of the top 11
// bits in which the keys differ (2048 bins) finds the bin that holds the
// k-th largest key; keys in higher bins are all taken, and the few keys of
// that boundary bin are ranked against each other (key descending, element
// ascending; one 64-bit word per key, (key, ~element), compared with 16-byte
// loads) to take the rest.  The chosen elements are then numbered in
// element order with warp ballots.  When the boundary bin holds more than
// kBoundaryMax keys (many equal or nearly equal keys) the radix select above
// runs instead, on the same keys in shared memory (`keys_smem`).  Output
// order and ties are as in block_select.
constexpr int kBoundaryMax = kTopkThreads;  // one boundary key per thread
struct __align__(16) FastShared {
  unsigned bins[2048];
  unsigned long long bcomb[kBoundaryMax];  // (key << 32) | ~element; zero past the bin's keys
  unsigned char bwin[kBoundaryMax];
  int wsum[kWarps];
  unsigned wmin[kWarps], wmax[kWarps];
  int cnt[128];  // chosen elements per (u, warp) block, u-major
  int b_bin, b_above, b_cnt;
};

template <int IPT, typename Emit>
__device__ void reg_select(const uint32_t (&kr)[IPT], const uint32_t* keys_smem, int n, int k, SelectShared& sh,
                           FastShared& fs, Emit emit, int* select_trace_err = nullptr) {
  constexpr int E = IPT * kWarps;         // blocks of 32 consecutive elements
  constexpr int EPL = (E + 31) / 32;      // blocks per lane in the prefix sum
  static_assert(E <= 128, "per-block counts must fit");
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (k <= 0 || n <= 0) return;
  if (k >= n) {
    for (int i = tid; i < n; i += kTopkThreads) emit(i, i);
    return;
  }
  const unsigned long long tc0 = trace_clock();
  unsigned lo = 0xffffffffu, hi = 0u;
#pragma unroll
  for (int u = 0; u < IPT; ++u) {
    if (tid + kTopkThreads * u < n) {
      lo = min(lo, kr[u]);
      hi = max(hi, kr[u]);
    }
  }
  lo = __reduce_min_sync(0xffffffffu, lo);
  hi = __reduce_max_sync(0xffffffffu, hi);
  if (lane == 0) {
    fs.wmin[warp] = lo;
    fs.wmax[warp] = hi;
  }
  reinterpret_cast<uint4*>(fs.bins)[tid] = make_uint4(0u, 0u, 0u, 0u);
  fs.bcomb[tid] = 0ull;  // below every real key: padding of the ranking loop
  if (tid == 0) fs.b_cnt = 0;
  __syncthreads();
#pragma unroll
  for (int w = 0; w < kWarps; ++w) {
    lo = min(lo, fs.wmin[w]);
    hi = max(hi, fs.wmax[w]);
  }
  if (lo == hi) {  // all keys equal: the first k elements
    for (int i = tid; i < k; i += kTopkThreads) emit(i, i);
    return;
  }
  // bins: the top 11 of the bits in which the keys differ (monotone in the key)
  const int nbits = 32 - __clz(lo ^ hi);
  const int shift = nbits > 11 ? nbits - 11 : 0;
  unsigned bin[IPT];
#pragma unroll
  for (int u = 0; u < IPT; ++u) {
    bin[u] = (kr[u] - lo) >> shift;
    if (tid + kTopkThreads * u < n) atomicAdd(&fs.bins[bin[u]], 1u);
  }
  __syncthreads();
  // thread t owns bins 4t .. 4t+3; counts above each bin, from the top bin down
  const uint4 c4 = reinterpret_cast<const uint4*>(fs.bins)[tid];
  const unsigned c[4] = {c4.x, c4.y, c4.z, c4.w};
  const unsigned own = c[0] + c[1] + c[2] + c[3];
  unsigned incl = own;  // sum over this lane and the higher lanes of the warp
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned y = __shfl_down_sync(0xffffffffu, incl, o);
    if (lane + o < 32) incl += y;
  }
  if (lane == 0) fs.wsum[warp] = (int)incl;
  __syncthreads();
  unsigned above = incl - own;
#pragma unroll
  for (int w = 0; w < kWarps; ++w)
    if (w > warp) above += (unsigned)fs.wsum[w];
#pragma unroll
  for (int u = 3; u >= 0; --u) {
    if (above < (unsigned)k && (unsigned)k <= above + c[u]) {
      fs.b_bin = 4 * tid + u;
      fs.b_above = (int)above;
    }
    above += c[u];
  }
  __syncthreads();
  const unsigned bstar = (unsigned)fs.b_bin;
  const int need = k - fs.b_above;
  const unsigned m = fs.bins[bstar];
  if (m > (unsigned)kBoundaryMax) {
    block_select(keys_smem, n, k, sh, emit, select_trace_err);
    return;
  }
  // the boundary bin's keys into a short list (one atomic per warp and u)
  int bslot[IPT];
#pragma unroll
  for (int u = 0; u < IPT; ++u) {
    bslot[u] = -1;
    if (kTopkThreads * u >= n) continue;  // uniform over the block
    const bool eq = tid + kTopkThreads * u < n && bin[u] == bstar;
    const unsigned mask = __ballot_sync(0xffffffffu, eq);
    int base = 0;
    if (mask) {
      if (lane == 0) base = atomicAdd(&fs.b_cnt, __popc(mask));
      base = __shfl_sync(0xffffffffu, base, 0);
    }
    bslot[u] = eq ? base + __popc(mask & ((1u << lane) - 1u)) : -1;
    if (eq) fs.bcomb[bslot[u]] = ((unsigned long long)kr[u] << 32) | (0xffffffffu - (uint32_t)(tid + kTopkThreads * u));
  }
  __syncthreads();
  if (tid < (int)m) {
    // rank = keys ahead of this one (larger key, or equal key and lower
    // element); the zero padding up to a multiple of 8 is ahead of nothing
    const unsigned long long mine = fs.bcomb[tid];
    const ulonglong2* bc = reinterpret_cast<const ulonglong2*>(fs.bcomb);
    const int m8 = ((int)m + 7) >> 3;
    int rank = 0;
    for (int v = 0; v < m8; ++v) {
      const ulonglong2 x0 = bc[4 * v], x1 = bc[4 * v + 1], x2 = bc[4 * v + 2], x3 = bc[4 * v + 3];
      rank += (x0.x > mine) + (x0.y > mine) + (x1.x > mine) + (x1.y > mine) + (x2.x > mine) + (x2.y > mine) +
              (x3.x > mine) + (x3.y > mine);
    }
    fs.bwin[tid] = rank < need ? 1 : 0;
  }
  __syncthreads();
  // number the chosen elements in element order: element t + 512u sits in
  // block (u, warp) of 32 consecutive elements, blocks ordered u-major
  bool take[IPT];
#pragma unroll
  for (int u = 0; u < IPT; ++u) {
    take[u] = false;
    if (kTopkThreads * u >= n) {
      if (lane == 0) fs.cnt[u * kWarps + warp] = 0;
      continue;
    }
    take[u] = tid + kTopkThreads * u < n && (bin[u] > bstar || (bslot[u] >= 0 && fs.bwin[bslot[u]]));
    const unsigned mask = __ballot_sync(0xffffffffu, take[u]);
    if (lane == 0) fs.cnt[u * kWarps + warp] = __popc(mask);
  }
  __syncthreads();
  // exclusive prefix over the E block counts, lane l holding blocks
  // EPL*l .. EPL*l + EPL - 1 (every warp computes it)
  int ex[EPL];
  int own2 = 0;
#pragma unroll
  for (int v = 0; v < EPL; ++v) {
    const int e = EPL * lane + v;
    ex[v] = own2;
    own2 += e < E ? fs.cnt[e] : 0;
  }
  int incl2 = own2;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl2, o);
    if (lane >= o) incl2 += y;
  }
#pragma unroll
  for (int v = 0; v < EPL; ++v) ex[v] += incl2 - own2;
#pragma unroll
  for (int u = 0; u < IPT; ++u) {
    if (kTopkThreads * u >= n) break;  // uniform over the block
    const int e = u * kWarps + warp;
    int base = 0;
#pragma unroll
    for (int v = 0; v < EPL; ++v) {
      const int t = __shfl_sync(0xffffffffu, ex[v], e / EPL);
      if (e % EPL == v) base = t;
    }
    const unsigned mask = __ballot_sync(0xffffffffu, take[u]);
    if (take[u]) emit(base + __popc(mask & ((1u << lane) - 1u)), tid + kTopkThreads * u);
  }
  if (tid == 0) {
    trace_add(select_trace_err, kTrSelRadix, trace_clock() - tc0);
    trace_add(select_trace_err, kTrSelCalls, 1ull);
  }
}

// GT: heads per group (compile time; 0 = any G <= 16 at run time).
// Pages per thread at most: s_hat rows of G floats in registers.
constexpr int topk_ipt_max(int gt) { return gt ? (32 / gt < 8 ? 32 / gt : 8) : 2; }

// MULTI: several chunks per problem (candidates, then a merge by the last
// CTA); a problem of one chunk selects straight into the page list.
// Each thread owns IPT pages of the chunk (pages tid + 512 u), whose s_hat
// rows it loads together with the lengths and the scan partials in one round
// trip.  A problem of one chunk takes the smallest IPT that covers its pages:
// the selection's loops are unrolled over IPT, and fewer instructions to
// fetch and fewer registers made the 2048-page top-k 0.85 us faster on GB300.
template <int GT, bool MULTI, int IPT>
__global__ void __launch_bounds__(kTopkThreads, 1) topk_kernel(const TopkArgs a) {
  constexpr int GMAX = GT ? GT : 16;
  static_assert(IPT >= 1 && IPT <= topk_ipt_max(GT), "pages per thread");
  extern __shared__ __align__(16) uint8_t dyn[];
  uint32_t* keys = reinterpret_cast<uint32_t*>(dyn);
  int32_t* idx = reinterpret_cast<int32_t*>(dyn + a.smem_keys * sizeof(uint32_t));
  __shared__ SelectShared sh;
  __shared__ FastShared fsh;
  __shared__ float zsh[16];
  __shared__ int is_last;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int chunk = blockIdx.x, bh = blockIdx.y;
  const int b = bh / a.num_kv_heads;
  const int G = GT ? GT : a.group;

  trace_mark(a.err, kTrTopkEnter, true);
  const int j0 = chunk * a.chunk_pages;
  if (!MULTI && a.sel_phys) {
    // inside the decode step: the block table is an input of the step, so
    // this problem's row loads while the scan is still running (idx is free
    // in a one-chunk problem; thread t keeps the entries of its own pages)
#pragma unroll
    for (int p = 0; p < IPT; ++p) {
      const int j = j0 + tid + kTopkThreads * p;
      if (j < a.max_pages) idx[j - j0] = __ldg(a.block_table + (size_t)b * a.max_pages + j);
    }
  }
  pdl_wait();
  trace_mark(a.err, kTrTopkWait, true);
  // the attention kernel that follows may start its prologue now; it waits
  // for this grid to finish before reading the selection
  pdl_launch_dependents();

  // ---- one round trip: lengths, scan partials (warp h: head h), s_hat rows
  const int L = a.seq_lens[b];
  int ns = a.n_summarized[b];
  // the scan writes one partial per chunk, at most one chunk per SM (152 on
  // GB300): five per lane load them all in the first round trip
  constexpr int kPv = 5;
  float2 pv[kPv];
  const float2* pbase = a.part + (size_t)bh * a.n_scan_chunks * G;
  if (warp < G) {
#pragma unroll
    for (int u = 0; u < kPv; ++u) {
      const int i = lane + 32 * u;
      pv[u] = i < a.n_scan_chunks ? __ldcg(pbase + (size_t)i * G + warp) : make_float2(-INFINITY, 0.f);
    }
  }
  // pages j0 + tid + kTopkThreads * p: a warp reads consecutive rows
  float sv[IPT][GMAX];
  {
    const float* sbase = a.shat + (size_t)bh * a.max_pages * G;
#pragma unroll
    for (int p = 0; p < IPT; ++p) {
      const int j = j0 + tid + kTopkThreads * p;
      const bool in = j < a.max_pages;
      const float* row = sbase + (size_t)j * G;
      if (GT != 0 && GT % 4 == 0) {
#pragma unroll
        for (int h4 = 0; h4 < GMAX / 4; ++h4) {
          const float4 v = in ? __ldcg(reinterpret_cast<const float4*>(row) + h4) : make_float4(0.f, 0.f, 0.f, 0.f);
          sv[p][4 * h4] = v.x;
          sv[p][4 * h4 + 1] = v.y;
          sv[p][4 * h4 + 2] = v.z;
          sv[p][4 * h4 + 3] = v.w;
        }
      } else if (GT == 2) {
        const float2 v = in ? __ldcg(reinterpret_cast<const float2*>(row)) : make_float2(0.f, 0.f);
        sv[p][0] = v.x;
        sv[p][GMAX > 1 ? 1 : 0] = v.y;
      } else {
#pragma unroll
        for (int h = 0; h < GMAX; ++h) sv[p][h] = (in && h < G) ? __ldcg(row + h) : 0.f;
      }
    }
  }

  const int nfull = L < 0 ? 0 : L / a.page_size;
  const int cap = nfull < a.max_pages ? nfull : a.max_pages;
  ns = ns < 0 ? 0 : (ns > cap ? cap : ns);
  const int k = ns < a.k_max ? ns : a.k_max;
  int32_t* sel = a.sel_pages + (size_t)bh * a.k_max;
  int32_t* sphys = (!MULTI && a.sel_phys) ? a.sel_phys + (size_t)bh * a.k_max : nullptr;

  if (ns <= a.k_max) {
    // every summarised page is selected
    if (chunk == 0) {
      for (int i = tid; i < ns; i += kTopkThreads) {
        sel[i] = i;
        if (sphys) sphys[i] = idx[i];  // written by this thread above
      }
      if (tid == 0) a.sel_count[bh] = ns;
    }
    trace_mark(a.err, kTrTopkExit, false);
    return;
  }

  // Z_h (natural log): the remaining partials, then a warp reduction
  if (warp < G) {
    float m = -INFINITY, l = 0.f;
#pragma unroll
    for (int u = 0; u < kPv; ++u) lse2_merge(m, l, pv[u].x, pv[u].y);
    for (int i = lane + 32 * kPv; i < a.n_scan_chunks; i += 32) {
      const float2 v = __ldcg(pbase + (size_t)i * G + warp);
      lse2_merge(m, l, v.x, v.y);
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) {
      const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
      const float l2 = __shfl_xor_sync(0xffffffffu, l, o);
      lse2_merge(m, l, m2, l2);
    }
    if (lane == 0) zsh[warp] = (m + fast_log2(l)) * kLn2;
  }
  __syncthreads();
  trace_mark(a.err, kTrTopkLoaded, false);

  // sigma_j = ln( (1/G) sum_h exp(s_hat[h][j] - Z_h) ) -> order-preserving keys
  const int j1 = min(j0 + a.chunk_pages, ns);
  const int nloc = j1 > j0 ? j1 - j0 : 0;
  uint32_t kr[IPT];  // this thread's keys: page j0 + tid + kTopkThreads * p
  {
    const float log2G = log2f((float)G);
    float zl[GMAX];
#pragma unroll
    for (int h = 0; h < GMAX; ++h) zl[h] = h < G ? zsh[h] * kLog2e : 0.f;
#pragma unroll
    for (int p = 0; p < IPT; ++p) {
      const int jl = tid + kTopkThreads * p;
      if (jl < nloc) {
        float y[GMAX];
        float mx = -INFINITY;
#pragma unroll
        for (int h = 0; h < GMAX; ++h) {
          y[h] = h < G ? fmaf(sv[p][h], kLog2e, -zl[h]) : -INFINITY;
          mx = fmaxf(mx, y[h]);
        }
        float acc = 0.f;
#pragma unroll
        for (int h = 0; h < GMAX; ++h) acc += h < G ? fast_exp2(y[h] - mx) : 0.f;
        kr[p] = orderable_key((mx + fast_log2(acc) - log2G) * kLn2);
        keys[jl] = kr[p];
      } else {
        kr[p] = 0u;
      }
    }
  }
  __syncthreads();
  trace_mark(a.err, kTrTopkKeys, false);

  const int kloc = k < nloc ? k : nloc;
  if constexpr (!MULTI) {
    reg_select<IPT>(kr, keys, nloc, kloc, sh, fsh, [&](int pos, int i) {
      sel[pos] = j0 + i;
      if (sphys) sphys[pos] = idx[i];
    }, a.err);
    if (tid == 0) a.sel_count[bh] = kloc;
    trace_mark(a.err, kTrTopkSelected, false);
    trace_mark(a.err, kTrTopkExit, false);
    return;
  }
  uint32_t* ck = a.cand_key + ((size_t)bh * a.n_chunks + chunk) * a.k_max;
  int32_t* ci = a.cand_idx + ((size_t)bh * a.n_chunks + chunk) * a.k_max;
  const int n_all = a.n_chunks * a.k_max;
  // One call site of the selection.  Every CTA runs it once over its chunk;
  // the last CTA of a problem runs it again over all chunks' candidates,
  // re-executing instructions it has just fetched rather than a second
  // inlined copy that no SM has run yet (cold instruction fetch made that
  // copy about three times slower than the work it does).
  // mode 1: this chunk's candidates; 2: the merge (element i = candidate
  // slot i, page idx[i]).
  int mode = 1;
  int sn = nloc, sk = kloc;
#pragma unroll 1
  for (;;) {
    reg_select<IPT>(kr, keys, sn, sk, sh, fsh, [&](int pos, int i) {
      if (mode == 1) {
        ck[pos] = keys[i];
        ci[pos] = j0 + i;
      } else {
        sel[pos] = idx[i];
      }
    });
    if (mode != 1) break;
    // unused candidate slots get the lowest key (never chosen: the chunks
    // together always offer at least k real candidates)
    for (int j = kloc + tid; j < a.k_max; j += kTopkThreads) {
      ck[j] = 0u;
      ci[j] = -1;
    }
    __threadfence();
    __syncthreads();
    if (tid == 0) {
      unsigned prev = atomicAdd(a.counters + bh, 1u);
      is_last = prev == (unsigned)(a.n_chunks - 1);
    }
    __syncthreads();
    if (!is_last) return;
    __threadfence();
    // every chunk's candidate slots, chunk-major (= page order), in one round trip
    const uint32_t* gk = a.cand_key + (size_t)bh * n_all;
    const int32_t* gi = a.cand_idx + (size_t)bh * n_all;
    if (n_all > IPT * kTopkThreads) {
      // more candidates than registers hold: radix select in shared memory
      for (int i = tid; i < n_all; i += kTopkThreads) {
        keys[i] = __ldcg(gk + i);
        idx[i] = __ldcg(gi + i);
      }
      __syncthreads();
      block_select(keys, n_all, k, sh, [&](int pos, int i) { sel[pos] = idx[i]; });
      break;
    }
#pragma unroll
    for (int u = 0; u < IPT; ++u) {
      const int i = tid + kTopkThreads * u;
      kr[u] = 0u;
      if (i < n_all) {
        kr[u] = __ldcg(gk + i);
        keys[i] = kr[u];
        idx[i] = __ldcg(gi + i);
      }
    }
    sn = n_all;
    sk = k;
    mode = 2;
  }
  if (tid == 0) {
    a.sel_count[bh] = k;
    a.counters[bh] = 0;  // ready for the next call
  }
  trace_mark(a.err, kTrTopkExit, false);
}

}  // namespace

// keys (u32) and their positions (i32)
size_t topk_smem_bytes(size_t keys) { return keys * (sizeof(uint32_t) + sizeof(int32_t)); }

namespace {

template <int GT, bool MULTI, int IPT>
cudaError_t launch_gm(const TopkArgs& a, cudaStream_t s, bool pdl) {
  const size_t smem = topk_smem_bytes(a.smem_keys);
  cudaError_t e =
      cudaFuncSetAttribute(topk_kernel<GT, MULTI, IPT>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.n_chunks, a.batch * a.num_kv_heads, 1);
  cfg.blockDim = dim3(kTopkThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, topk_kernel<GT, MULTI, IPT>, a);
}

template <int GT>
cudaError_t launch_g(const TopkArgs& a, cudaStream_t s, bool pdl) {
  constexpr int kMax = topk_ipt_max(GT);
  if (a.n_chunks > 1) return launch_gm<GT, true, kMax>(a, s, pdl);
  // one chunk: the smallest power of two of pages per thread that covers it
  const int need = (a.max_pages + kTopkThreads - 1) / kTopkThreads;
  if (need <= 1) return launch_gm<GT, false, 1>(a, s, pdl);
  if (need <= 2 || kMax == 2) return launch_gm<GT, false, (kMax < 2 ? kMax : 2)>(a, s, pdl);
  if (need <= 4 || kMax == 4) return launch_gm<GT, false, (kMax < 4 ? kMax : 4)>(a, s, pdl);
  return launch_gm<GT, false, kMax>(a, s, pdl);
}

}  // namespace

int topk_pages_per_cta(int group) {
  const int gt = (group == 1 || group == 2 || group == 4 || group == 8 || group == 16) ? group : 0;
  return topk_ipt_max(gt) * kTopkThreads;
}

cudaError_t launch_topk(const TopkArgs& a, cudaStream_t s, bool pdl) {
  switch (a.group) {
    case 1: return launch_g<1>(a, s, pdl);
    case 2: return launch_g<2>(a, s, pdl);
    case 4: return launch_g<4>(a, s, pdl);
    case 8: return launch_g<8>(a, s, pdl);
    case 16: return launch_g<16>(a, s, pdl);
    default: return launch_g<0>(a, s, pdl);
  }
}

}  // namespace locks
