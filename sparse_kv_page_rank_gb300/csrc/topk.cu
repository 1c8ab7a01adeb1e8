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
//   * sigma_j for the chunk -> 32-bit order-preserving keys in shared memory;
//   * MSB-first 8-bit radix select finds the k-th largest key T and how many
//     keys equal to T to take; an ordered block scan then keeps every key > T
//     and the first such keys == T in page order, so the output is already
//     sorted ascending and ties go to lower pages;
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
  unsigned hist[256];
  int warp_tmp[kWarps];
  unsigned bucket;
  unsigned remaining;
};

// Choose the k largest of keys[0..n) (ties -> lower position) and call
// emit(position_in_output, i) for each chosen i, positions in array order.
template <typename Emit>
__device__ void block_select(const uint32_t* keys, int n, int k, SelectShared& sh, Emit emit) {
  const int tid = threadIdx.x;
  if (k <= 0 || n <= 0) return;
  uint32_t T = 0;
  unsigned need_eq = 0;
  const bool take_all = k >= n;
  if (!take_all) {
    uint32_t prefix = 0, mask = 0;
    unsigned rem = (unsigned)k;
    for (int shift = 24; shift >= 0; shift -= 8) {
      for (int i = tid; i < 256; i += kTopkThreads) sh.hist[i] = 0;
      __syncthreads();
      for (int i = tid; i < n; i += kTopkThreads) {
        uint32_t key = keys[i];
        if ((key & mask) == prefix) atomicAdd(&sh.hist[(key >> shift) & 255u], 1u);
      }
      __syncthreads();
      if (tid < 32) {
        // lane l owns buckets 8l .. 8l+7; count of keys in buckets above its range
        unsigned cnt[8], tot = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) { cnt[i] = sh.hist[8 * tid + i]; tot += cnt[i]; }
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
}

__global__ void __launch_bounds__(kTopkThreads) topk_kernel(const TopkArgs a) {
  extern __shared__ __align__(16) uint8_t dyn[];
  uint32_t* keys = reinterpret_cast<uint32_t*>(dyn);
  int32_t* idx = reinterpret_cast<int32_t*>(dyn + a.smem_keys * sizeof(uint32_t));
  __shared__ SelectShared sh;
  __shared__ float zsh[16];
  __shared__ int is_last;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int chunk = blockIdx.x, bh = blockIdx.y;
  const int b = bh / a.num_kv_heads;
  const int G = a.group;

  pdl_wait();

  const int L = a.seq_lens[b];
  const int nfull = L < 0 ? 0 : L / kPage;
  const int cap = nfull < a.max_pages ? nfull : a.max_pages;
  int ns = a.n_summarized[b];
  ns = ns < 0 ? 0 : (ns > cap ? cap : ns);
  const int k = ns < a.k_max ? ns : a.k_max;
  int32_t* sel = a.sel_pages + (size_t)bh * a.k_max;

  if (ns <= a.k_max) {
    // every summarised page is selected
    if (chunk == 0) {
      for (int i = tid; i < ns; i += kTopkThreads) sel[i] = i;
      if (tid == 0) a.sel_count[bh] = ns;
    }
    pdl_launch_dependents();
    return;
  }

  // Z_h (natural log) from the scan partials
  for (int h = warp; h < G; h += kWarps) {
    float m = -INFINITY, l = 0.f;
    const float2* p = a.part + (size_t)bh * a.n_scan_chunks * G + h;
    for (int i = lane; i < a.n_scan_chunks; i += 32) {
      float2 v = __ldcg(p + (size_t)i * G);
      lse2_merge(m, l, v.x, v.y);
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) {
      float m2 = __shfl_xor_sync(0xffffffffu, m, o);
      float l2 = __shfl_xor_sync(0xffffffffu, l, o);
      lse2_merge(m, l, m2, l2);
    }
    if (lane == 0) zsh[h] = (m + fast_log2(l)) * kLn2;
  }
  __syncthreads();

  const int j0 = chunk * a.chunk_pages;
  const int j1 = min(j0 + a.chunk_pages, ns);
  const int nloc = j1 > j0 ? j1 - j0 : 0;
  const float log2G = log2f((float)G);
  for (int i = tid; i < nloc; i += kTopkThreads) {
    const float* s = a.shat + ((size_t)bh * a.max_pages + j0 + i) * G;
    float y[16];
    float mx = -INFINITY;
#pragma unroll
    for (int h = 0; h < 16; ++h) {
      if (h < G) {
        y[h] = (__ldcg(s + h) - zsh[h]) * kLog2e;
        mx = fmaxf(mx, y[h]);
      }
    }
    float acc = 0.f;
#pragma unroll
    for (int h = 0; h < 16; ++h)
      if (h < G) acc += fast_exp2(y[h] - mx);
    float sigma = (mx + fast_log2(acc) - log2G) * kLn2;
    keys[i] = orderable_key(sigma);
  }
  __syncthreads();

  const int kloc = k < nloc ? k : nloc;
  if (a.n_chunks == 1) {
    block_select(keys, nloc, kloc, sh, [&](int pos, int i) { sel[pos] = j0 + i; });
    if (tid == 0) a.sel_count[bh] = kloc;
    pdl_launch_dependents();
    return;
  }

  uint32_t* ck = a.cand_key + ((size_t)bh * a.n_chunks + chunk) * a.k_max;
  int32_t* ci = a.cand_idx + ((size_t)bh * a.n_chunks + chunk) * a.k_max;
  block_select(keys, nloc, kloc, sh, [&](int pos, int i) {
    ck[pos] = keys[i];
    ci[pos] = j0 + i;
  });
  if (tid == 0) a.cand_cnt[(size_t)bh * a.n_chunks + chunk] = kloc;
  __threadfence();
  __syncthreads();
  if (tid == 0) {
    unsigned prev = atomicAdd(a.counters + bh, 1u);
    is_last = prev == (unsigned)(a.n_chunks - 1);
  }
  __syncthreads();
  if (!is_last) return;
  __threadfence();

  // gather every chunk's candidates, in chunk (= page) order
  int n_all = 0;
  for (int ch = 0; ch < a.n_chunks; ++ch) {
    const int cnt = __ldcg(a.cand_cnt + (size_t)bh * a.n_chunks + ch);
    const uint32_t* sk = a.cand_key + ((size_t)bh * a.n_chunks + ch) * a.k_max;
    const int32_t* si = a.cand_idx + ((size_t)bh * a.n_chunks + ch) * a.k_max;
    for (int i = tid; i < cnt; i += kTopkThreads) {
      keys[n_all + i] = __ldcg(sk + i);
      idx[n_all + i] = __ldcg(si + i);
    }
    n_all += cnt;
  }
  __syncthreads();
  block_select(keys, n_all, k, sh, [&](int pos, int i) { sel[pos] = idx[i]; });
  if (tid == 0) {
    a.sel_count[bh] = k;
    a.counters[bh] = 0;  // ready for the next call
  }
  pdl_launch_dependents();
}

}  // namespace

size_t topk_smem_bytes(size_t keys) { return keys * (sizeof(uint32_t) + sizeof(int32_t)); }

cudaError_t launch_topk(const TopkArgs& a, cudaStream_t s, bool pdl) {
  const size_t smem = topk_smem_bytes(a.smem_keys);
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
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
  return cudaLaunchKernelEx(&cfg, topk_kernel, a);
}

}  // namespace locks
