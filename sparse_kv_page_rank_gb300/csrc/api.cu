// C ABI of liblocks.so: host-side validation, launch planning, workspace
// layout, TMA descriptor encoding and kernel launches.  Nothing here
// allocates device memory or synchronises a stream (except
// locks_get_device_error).
#include <cudaTypedefs.h>

#include <cmath>
#include <cstring>
#include <mutex>

#include "../../include/locks.h"
#include "common.cuh"
#include "kernels.h"

namespace {

using namespace locks;

constexpr size_t kAlign = 256;
size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

int device_sm_count() {
  static int cache[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return 152;
  if (dev < 64 && cache[dev] > 0) return cache[dev];
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 152;
  if (dev < 64) cache[dev] = n;
  return n;
}

struct Plan {
  bool ok = true;  // false: shapes beyond what the launch plan supports
  int G = 0, Hq = 0, BH = 0, k_max = 0;
  int scan_chunk = 0, n_scan = 0, scan_hg = 1;
  int tk_chunk = 0, n_tk = 0;
  size_t tk_keys = 0;
  int sparse_cluster = 1, dense_cluster = 1, dense_nc = 1, lse_splits = 1;
  bool fused = false;     // decode step as scan + one attention kernel that selects the pages itself
  int fused_cluster = 1;
  size_t off_err = 0, off_cnt_tk = 0, off_cnt_att = 0, off_shat = 0, off_part = 0, off_ckey = 0,
         off_cidx = 0, off_sel = 0, off_selcnt = 0, off_selphys = 0, off_pml = 0, off_po = 0, total = 0;
};

locks_status_t check_cache(const locks_cache_t* c, bool need_kv) {
  if (!c) return LOCKS_ERR_INVALID_ARG;
  if (c->batch <= 0 || c->num_kv_heads <= 0 || c->pages_total <= 0 || c->max_pages <= 0)
    return LOCKS_ERR_INVALID_ARG;
  if (c->head_dim != kHeadDim || (c->page_size != kPage && c->page_size != 16)) return LOCKS_ERR_UNSUPPORTED;
  if (need_kv) {
    if (!c->k_pool || !c->v_pool || !c->block_table || !c->seq_lens) return LOCKS_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(c->k_pool) | reinterpret_cast<uintptr_t>(c->v_pool)) & 15)
      return LOCKS_ERR_INVALID_ARG;
  }
  // TMA row coordinate and 32-bit page-head offsets
  // (key rows >= basis rows, since r <= 16 <= P)
  if ((long long)c->pages_total * c->num_kv_heads * c->page_size > 0x7fffffffLL) return LOCKS_ERR_UNSUPPORTED;
  if ((long long)c->max_pages * c->page_size > 0x7fffffffLL) return LOCKS_ERR_UNSUPPORTED;
  return LOCKS_OK;
}

locks_status_t check_params(const locks_cache_t* c, const locks_params_t* p) {
  if (!p) return LOCKS_ERR_INVALID_ARG;
  if (p->num_q_heads <= 0 || p->num_q_heads % c->num_kv_heads) return LOCKS_ERR_INVALID_ARG;
  const int G = p->num_q_heads / c->num_kv_heads;
  if (G > 16) return LOCKS_ERR_UNSUPPORTED;
  if (p->budget_tokens < 0 || (p->flags & ~(LOCKS_FLAG_UNFUSED | LOCKS_FLAG_FUSED)) != 0) return LOCKS_ERR_INVALID_ARG;
  if ((p->flags & LOCKS_FLAG_UNFUSED) && (p->flags & LOCKS_FLAG_FUSED)) return LOCKS_ERR_INVALID_ARG;
  if (!(p->scale >= 0.f) || !std::isfinite(p->scale)) return LOCKS_ERR_INVALID_ARG;
  return LOCKS_OK;
}

locks_status_t check_summary(const locks_summary_t* s, bool for_scan) {
  if (!s || !s->basis_t) return LOCKS_ERR_INVALID_ARG;
  const bool q4 = s->dtype == LOCKS_DTYPE_Q4;
  const bool one = q4 || s->dtype == LOCKS_DTYPE_BF16_PACKED;  // one array of blocks; coeffs unused
  if (!one && !s->coeffs) return LOCKS_ERR_INVALID_ARG;
  if (s->rank < 2 || s->rank > 16 || (s->rank & 1)) return LOCKS_ERR_UNSUPPORTED;
  if (s->dtype != LOCKS_DTYPE_BF16 && s->dtype != LOCKS_DTYPE_F32 && !one) return LOCKS_ERR_INVALID_ARG;
  if (q4 && s->rank > 8) return LOCKS_ERR_UNSUPPORTED;
  if (for_scan && s->dtype == LOCKS_DTYPE_F32) return LOCKS_ERR_UNSUPPORTED;
  if ((reinterpret_cast<uintptr_t>(s->basis_t) | (one ? 0 : reinterpret_cast<uintptr_t>(s->coeffs))) & 15)
    return LOCKS_ERR_INVALID_ARG;
  return LOCKS_OK;
}

float scale_of(const locks_params_t* p) {
  return p->scale > 0.f ? p->scale : 1.0f / std::sqrt((float)kHeadDim);
}

Plan make_plan(const locks_cache_t* c, const locks_params_t* p) {
  Plan pl;
  const int sms = device_sm_count();
  pl.G = p->num_q_heads / c->num_kv_heads;
  pl.Hq = p->num_q_heads;
  pl.BH = c->batch * c->num_kv_heads;
  const int P = c->page_size;
  pl.k_max = std::min(p->budget_tokens / P, c->max_pages);
  const long long BH = pl.BH;
  // attention works in 64-token tiles: one page, or four 16-token pages
  const int ppt = kPage / P;
  const long long max_tiles = (c->max_pages + ppt - 1) / ppt;

  // scan: one CTA per SM, each over a range of pages of one sequence for a
  // block of HG KV heads.  Every (sequence, head block) gets the same number
  // of chunks, at most SMs / blocks of them, so that all CTAs fit in one wave
  // (rounding the chunk size up instead can leave a few full-length CTAs for
  // a second wave, which doubles the scan)
  {
    pl.scan_hg = scan_heads_per_block(c->num_kv_heads);
    const long long blocks = (long long)c->batch * (c->num_kv_heads / pl.scan_hg);
    const long long chunks = std::max<long long>(1, std::min<long long>(sms / blocks, c->max_pages));
    pl.scan_chunk = (int)((c->max_pages + chunks - 1) / chunks);
    pl.n_scan = (c->max_pages + pl.scan_chunk - 1) / pl.scan_chunk;
  }
  // top-k: each CTA scores a fixed chunk of pages (its threads hold the
  // pages' s_hat rows in registers); the last CTA of a problem merges the
  // chunks' candidates (at most 64 chunks)
  {
    const int chunk = topk_pages_per_cta(pl.G);
    const int n = (c->max_pages + chunk - 1) / chunk;
    pl.tk_chunk = chunk;
    pl.n_tk = n;
    pl.tk_keys = std::max<size_t>((size_t)std::min(chunk, c->max_pages), (size_t)n * std::max(pl.k_max, 1));
    if (n > 64 || topk_smem_bytes(pl.tk_keys) > 200 * 1024) pl.ok = false;
  }
  // attention: one thread-block cluster per problem for the sparse step
  // (selected pages + a short tail spread over its CTAs, merged on chip);
  // several clusters per problem for the dense decode, about three resident
  // CTAs per SM
  {
    const long long target = 3LL * sms;
    const int cs_sparse = attend_max_cluster(kAttendSparse, P);
    const int cs_dense = attend_max_cluster(kAttendDense, P);
    const long long items = ((long long)pl.k_max + 2 + ppt - 1) / ppt;  // tiles
    // the largest cluster (up to one CTA per item) with which every
    // problem's cluster is resident at once: one wave, no CTA waits for a slot
    int cs = 1;
    while (cs * 2 <= cs_sparse && cs * 2 <= items) cs *= 2;
    while (cs > 1 && BH > attend_active_clusters(kAttendSparse, cs, P)) cs /= 2;
    pl.sparse_cluster = cs;
    // dense: the (cluster, clusters-per-problem) shape with the most CTAs
    // that still fits in one wave of `target` resident CTAs
    long long best = -1;
    for (int csd = cs_dense; csd >= 1; csd /= 2) {
      if (csd > max_tiles) continue;
      long long nc = target / (BH * csd);
      nc = std::max<long long>(1, std::min<long long>(nc, (max_tiles + csd - 1) / csd));
      const long long ctas = BH * csd * nc;
      // the fullest wave wins; among equals the larger cluster (cheaper
      // on-chip merge), since the loop runs from large to small clusters
      if (ctas <= target && ctas > best) {
        best = ctas;
        pl.dense_cluster = csd;
        pl.dense_nc = (int)nc;
      }
    }
    if (best < 0) {
      pl.dense_cluster = 1;
      pl.dense_nc = 1;
    }
    long long ls = (target + BH - 1) / BH;
    pl.lse_splits = (int)std::max<long long>(1, std::min<long long>(ls, max_tiles));
    // fused step (64-token pages, k <= kFusedMaxK): one cluster per problem
    // whose CTAs score at most one page per thread; sized like the sparse
    // cluster, then raised until the pages fit.  Taken only on request
    // (LOCKS_FLAG_FUSED): the separate top-k, 512 threads per problem,
    // selects faster than the 4-warp attention CTAs do, at every measured
    // problem count (GB300: 8K context with 256 problems, 50.3 us with the
    // separate top-k and 52.0 us fused; 32K with 64 problems, 34.4 and 37.5;
    // 128K with 8 problems, 23.7 and 29.4).
    if (P == kPage && pl.k_max <= kFusedMaxK && (p->flags & LOCKS_FLAG_FUSED)) {
      const int cs_max = attend_max_cluster(kAttendFused, P);
      const long long need = ((long long)c->max_pages + kAttendThreads - 1) / kAttendThreads;
      int csf = 1;
      while (csf * 2 <= cs_max && csf * 2 <= items) csf *= 2;
      while (csf > 1 && BH > attend_active_clusters(kAttendFused, csf, P)) csf /= 2;
      while (csf < need && csf * 2 <= cs_max) csf *= 2;
      if (csf >= need) {
        pl.fused = true;
        pl.fused_cluster = csf;
      }
    }
  }
  size_t off = 0;
  auto take = [&](size_t bytes) {
    size_t o = off;
    off = align_up(off + std::max<size_t>(bytes, 1));
    return o;
  };
  pl.off_err = take(sizeof(int));
  pl.off_cnt_tk = take(sizeof(unsigned) * BH);
  pl.off_cnt_att = take(sizeof(unsigned) * BH);
  pl.off_shat = take(sizeof(float) * BH * c->max_pages * pl.G);
  pl.off_part = take(sizeof(float2) * BH * pl.n_scan * pl.G);
  pl.off_ckey = take(sizeof(uint32_t) * BH * pl.n_tk * std::max(pl.k_max, 1));
  pl.off_cidx = take(sizeof(int32_t) * BH * pl.n_tk * std::max(pl.k_max, 1));
  pl.off_sel = take(sizeof(int32_t) * BH * std::max(pl.k_max, 1));
  pl.off_selcnt = take(sizeof(int32_t) * BH);
  pl.off_selphys = take(sizeof(int32_t) * BH * std::max(pl.k_max, 1));
  pl.off_pml = take(sizeof(float2) * BH * pl.dense_nc * pl.G);
  pl.off_po = take(sizeof(float) * BH * pl.dense_nc * pl.G * kHeadDim);
  pl.total = off;
  return pl;
}

template <typename T>
T* at(void* ws, size_t off) {
  return reinterpret_cast<T*>(static_cast<uint8_t*>(ws) + off);
}

locks_status_t check_ws(void* ws, size_t bytes, const Plan& pl) {
  if (!ws || (reinterpret_cast<uintptr_t>(ws) & (kAlign - 1)) || bytes < pl.total) return LOCKS_ERR_WORKSPACE;
  return LOCKS_OK;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// 2-D view of a pool of 128-column bf16 rows (rows = pages_total * Hkv *
// rows_per_page); 64-column boxes of box_rows rows with 128-byte swizzle.
bool encode_rows(CUtensorMap* m, const void* pool, const locks_cache_t* c, int rows_per_page, int box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {(cuuint64_t)kHeadDim, (cuuint64_t)c->pages_total * c->num_kv_heads * rows_per_page};
  cuuint64_t strides[1] = {(cuuint64_t)kHeadDim * 2};
  cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(pool), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// K or V pool: boxes of one page-head's rows x 64 columns (one page-head is
// two boxes).
bool encode_pool(CUtensorMap* m, const void* pool, const locks_cache_t* c) {
  return encode_rows(m, pool, c, c->page_size, c->page_size);
}

locks_status_t cuda_status(cudaError_t e) { return e == cudaSuccess ? LOCKS_OK : LOCKS_ERR_CUDA; }

// in_step: the top-k inside locks_decode_step, whose attention kernel reads
// the physical pages it writes (one-chunk problems)
locks_status_t run_select(const locks_cache_t* c, const locks_summary_t* s, const locks_params_t* p,
                          const Plan& pl, const void* q, int32_t* sel, int32_t* selcnt, float* page_lse,
                          void* ws, cudaStream_t st, bool in_step = false) {
  ScanArgs sa;
  sa.basis_t = static_cast<const uint16_t*>(s->basis_t);
  sa.coeffs = static_cast<const uint16_t*>(s->coeffs);
  sa.q = static_cast<const uint16_t*>(q);
  sa.block_table = c->block_table;
  sa.seq_lens = c->seq_lens;
  sa.n_summarized = c->n_summarized;
  sa.shat = at<float>(ws, pl.off_shat);
  sa.part = at<float2>(ws, pl.off_part);
  sa.page_lse = page_lse;
  sa.err = at<int>(ws, pl.off_err);
  sa.batch = c->batch;
  sa.num_kv_heads = c->num_kv_heads;
  sa.group = pl.G;
  sa.rank = s->rank;
  sa.max_pages = c->max_pages;
  sa.pages_total = c->pages_total;
  sa.chunk_pages = pl.scan_chunk;
  sa.n_chunks = pl.n_scan;
  sa.scale_log2 = scale_of(p) * kLog2e;
  sa.q4 = s->dtype == LOCKS_DTYPE_Q4 ? 1 : 0;
  sa.packed = s->dtype == LOCKS_DTYPE_BF16_PACKED ? 1 : 0;
  sa.page_size = c->page_size;
  sa.heads_per_block = pl.scan_hg;
  sa.slots = sa.slot_bytes = sa.basis_bytes = sa.coef_bytes = 0;  // set by the launcher
  cudaError_t e = launch_scan(sa, st, true);
  if (e != cudaSuccess) return LOCKS_ERR_CUDA;
  if (!sel) return LOCKS_OK;  // scan only

  TopkArgs ta;
  ta.shat = sa.shat;
  ta.part = sa.part;
  ta.n_scan_chunks = pl.n_scan;
  ta.seq_lens = c->seq_lens;
  ta.n_summarized = c->n_summarized;
  ta.cand_key = at<uint32_t>(ws, pl.off_ckey);
  ta.cand_idx = at<int32_t>(ws, pl.off_cidx);
  ta.counters = at<unsigned>(ws, pl.off_cnt_tk);
  ta.sel_pages = sel;
  ta.sel_count = selcnt;
  ta.block_table = c->block_table;
  ta.sel_phys = in_step && pl.n_tk == 1 ? at<int32_t>(ws, pl.off_selphys) : nullptr;
  ta.err = sa.err;
  ta.batch = c->batch;
  ta.num_kv_heads = c->num_kv_heads;
  ta.group = pl.G;
  ta.max_pages = c->max_pages;
  ta.k_max = pl.k_max;
  ta.chunk_pages = pl.tk_chunk;
  ta.n_chunks = pl.n_tk;
  ta.smem_keys = pl.tk_keys;
  ta.page_size = c->page_size;
  return cuda_status(launch_topk(ta, st, true));
}

locks_status_t run_attend(const locks_cache_t* c, const locks_params_t* p, const Plan& pl, const void* q,
                          int32_t* sel, int32_t* selcnt, void* out, float* lse, float* page_lse,
                          void* ws, int mode, cudaStream_t st, bool inputs_early = false) {
  CUtensorMap tk, tv;
  std::memset(&tk, 0, sizeof(tk));
  std::memset(&tv, 0, sizeof(tv));
  if (!encode_pool(&tk, c->k_pool, c)) return LOCKS_ERR_CUDA;
  if (mode != kAttendPageLse && !encode_pool(&tv, c->v_pool, c)) return LOCKS_ERR_CUDA;
  AttendArgs a;
  a.q = static_cast<const uint16_t*>(q);
  a.block_table = c->block_table;
  a.seq_lens = c->seq_lens;
  a.n_summarized = c->n_summarized;
  a.sel_pages = sel;
  a.sel_count = selcnt;
  // inside the decode step the top-k also wrote the selected pages' physical
  // ids (one-chunk problems), which saves the block-table lookup
  a.sel_phys = (mode == kAttendSparse && inputs_early && pl.n_tk == 1 && ws) ? at<int32_t>(ws, pl.off_selphys)
                                                                             : nullptr;
  a.out = static_cast<uint16_t*>(out);
  a.lse = lse;
  a.page_lse = page_lse;
  a.part_o = ws ? at<float>(ws, pl.off_po) : nullptr;
  a.part_ml = ws ? at<float2>(ws, pl.off_pml) : nullptr;
  a.counters = ws ? at<unsigned>(ws, pl.off_cnt_att) : nullptr;
  a.err = ws ? at<int>(ws, pl.off_err) : nullptr;
  a.batch = c->batch;
  a.num_kv_heads = c->num_kv_heads;
  a.group = pl.G;
  a.max_pages = c->max_pages;
  a.pages_total = c->pages_total;
  a.k_max = pl.k_max;
  a.shat = nullptr;
  a.part = nullptr;
  a.n_scan_chunks = pl.n_scan;
  a.sel_pages_out = nullptr;
  a.sel_count_out = nullptr;
  a.k_pool16 = static_cast<const uint16_t*>(c->k_pool);
  a.v_pool16 = static_cast<const uint16_t*>(c->v_pool);
  a.trace_cta = nullptr;
  if (mode == kAttendSparse) {
    a.cluster = pl.sparse_cluster;
    a.n_splits = pl.sparse_cluster;
  } else if (mode == kAttendFused) {
    a.cluster = pl.fused_cluster;
    a.n_splits = pl.fused_cluster;
    a.shat = at<float>(ws, pl.off_shat);
    a.part = at<float2>(ws, pl.off_part);
    a.sel_pages_out = sel;
    a.sel_count_out = selcnt;
    a.sel_pages = nullptr;
    a.sel_count = nullptr;
  } else if (mode == kAttendDense) {
    a.cluster = pl.dense_cluster;
    a.n_splits = pl.dense_cluster * pl.dense_nc;
  } else {
    a.cluster = 1;
    a.n_splits = pl.lse_splits;
  }
  a.scale_log2 = scale_of(p) * kLog2e;
  a.inputs_early = inputs_early ? 1 : 0;
#if LOCKS_TRACE
  // tracing builds: per-CTA timestamps of the page-list modes go to the end
  // of the workspace (the dense partials' region, the last one) when that
  // region is large enough
  {
    const size_t need = sizeof(unsigned long long) * pl.BH * a.n_splits * 16;
    if (ws && (mode == kAttendSparse || mode == kAttendFused) && pl.total - pl.off_po >= need)
      a.trace_cta = reinterpret_cast<unsigned long long*>(static_cast<uint8_t*>(ws) + pl.total - need);
  }
#endif
  a.page_size = c->page_size;
  return cuda_status(launch_attend(a, tk, tv, mode, st, true));
}

}  // namespace

extern "C" {

const char* locks_status_string(locks_status_t s) {
  switch (s) {
    case LOCKS_OK: return "LOCKS_OK";
    case LOCKS_ERR_INVALID_ARG: return "LOCKS_ERR_INVALID_ARG";
    case LOCKS_ERR_UNSUPPORTED: return "LOCKS_ERR_UNSUPPORTED";
    case LOCKS_ERR_CUDA: return "LOCKS_ERR_CUDA";
    case LOCKS_ERR_WORKSPACE: return "LOCKS_ERR_WORKSPACE";
    case LOCKS_ERR_DEVICE: return "LOCKS_ERR_DEVICE";
  }
  return "LOCKS_ERR_UNKNOWN";
}

locks_status_t locks_workspace_size(const locks_cache_t* cache, const locks_summary_t* summary,
                                    const locks_params_t* params, size_t* bytes) {
  (void)summary;
  if (!bytes) return LOCKS_ERR_INVALID_ARG;
  locks_status_t st = check_cache(cache, false);
  if (st != LOCKS_OK) return st;
  if ((st = check_params(cache, params)) != LOCKS_OK) return st;
  Plan pl = make_plan(cache, params);
  if (!pl.ok) return LOCKS_ERR_UNSUPPORTED;
  *bytes = pl.total;
  return LOCKS_OK;
}

locks_status_t locks_workspace_init(void* ws, size_t bytes, void* stream) {
  if (!ws) return LOCKS_ERR_INVALID_ARG;
  return cuda_status(cudaMemsetAsync(ws, 0, bytes, static_cast<cudaStream_t>(stream)));
}

locks_status_t locks_build_summaries(const locks_cache_t* cache, locks_summary_t* summary,
                                     const int32_t* page_ids, int32_t n, void* ws, size_t ws_bytes,
                                     void* stream) {
  if (!cache || !cache->k_pool) return LOCKS_ERR_INVALID_ARG;
  locks_status_t st = check_cache(cache, false);
  if (st != LOCKS_OK) return st;
  if ((st = check_summary(summary, false)) != LOCKS_OK) return st;
  if (n < 0 || (n > 0 && !page_ids)) return LOCKS_ERR_INVALID_ARG;
  if ((long long)n * cache->num_kv_heads > 0x7fffffffLL) return LOCKS_ERR_INVALID_ARG;
  if (ws && (ws_bytes < sizeof(int) || (reinterpret_cast<uintptr_t>(ws) & (kAlign - 1))))
    return LOCKS_ERR_WORKSPACE;
  BuildArgs a;
  a.k_pool = static_cast<const uint16_t*>(cache->k_pool);
  a.basis_t = summary->basis_t;
  a.coeffs = summary->coeffs;
  a.page_ids = page_ids;
  a.n = n;
  a.num_kv_heads = cache->num_kv_heads;
  a.rank = summary->rank;
  a.pages_total = cache->pages_total;
  a.format = summary->dtype;
  a.err = ws ? static_cast<int*>(ws) : nullptr;  // the error word is at offset 0 of every workspace
  a.page_size = cache->page_size;
  return cuda_status(launch_build(a, static_cast<cudaStream_t>(stream)));
}

locks_status_t locks_select(const locks_cache_t* cache, const locks_summary_t* summary,
                            const locks_params_t* params, const void* q, int32_t* sel_pages,
                            int32_t* sel_count, float* page_lse, void* ws, size_t ws_bytes, void* stream) {
  locks_status_t st = check_cache(cache, false);
  if (st != LOCKS_OK) return st;
  if (!cache->block_table || !cache->seq_lens || !cache->n_summarized) return LOCKS_ERR_INVALID_ARG;
  if ((st = check_params(cache, params)) != LOCKS_OK) return st;
  if ((st = check_summary(summary, true)) != LOCKS_OK) return st;
  if (!q || !sel_pages || !sel_count) return LOCKS_ERR_INVALID_ARG;
  Plan pl = make_plan(cache, params);
  if (!pl.ok) return LOCKS_ERR_UNSUPPORTED;
  if ((st = check_ws(ws, ws_bytes, pl)) != LOCKS_OK) return st;
  return run_select(cache, summary, params, pl, q, sel_pages, sel_count, page_lse, ws,
                    static_cast<cudaStream_t>(stream));
}

locks_status_t locks_page_scores(const locks_cache_t* cache, const locks_summary_t* summary,
                                 const locks_params_t* params, const void* q, float* page_lse, void* ws,
                                 size_t ws_bytes, void* stream) {
  locks_status_t st = check_cache(cache, false);
  if (st != LOCKS_OK) return st;
  if (!cache->block_table || !cache->seq_lens || !cache->n_summarized) return LOCKS_ERR_INVALID_ARG;
  if ((st = check_params(cache, params)) != LOCKS_OK) return st;
  if ((st = check_summary(summary, true)) != LOCKS_OK) return st;
  if (!q || !page_lse) return LOCKS_ERR_INVALID_ARG;
  Plan pl = make_plan(cache, params);
  if (!pl.ok) return LOCKS_ERR_UNSUPPORTED;
  if ((st = check_ws(ws, ws_bytes, pl)) != LOCKS_OK) return st;
  return run_select(cache, summary, params, pl, q, nullptr, nullptr, page_lse, ws,
                    static_cast<cudaStream_t>(stream));
}

locks_status_t locks_sparse_attend(const locks_cache_t* cache, const locks_params_t* params, const void* q,
                                   const int32_t* sel_pages, const int32_t* sel_count, void* out, float* lse,
                                   void* ws, size_t ws_bytes, void* stream) {
  locks_status_t st = check_cache(cache, true);
  if (st != LOCKS_OK) return st;
  if (!cache->n_summarized) return LOCKS_ERR_INVALID_ARG;
  if ((st = check_params(cache, params)) != LOCKS_OK) return st;
  if (!q || !sel_pages || !sel_count || !out) return LOCKS_ERR_INVALID_ARG;
  Plan pl = make_plan(cache, params);
  if (!pl.ok) return LOCKS_ERR_UNSUPPORTED;
  if ((st = check_ws(ws, ws_bytes, pl)) != LOCKS_OK) return st;
  // the sparse mode only reads the page list
  return run_attend(cache, params, pl, q, const_cast<int32_t*>(sel_pages), const_cast<int32_t*>(sel_count), out,
                    lse, nullptr, ws, kAttendSparse, static_cast<cudaStream_t>(stream));
}

locks_status_t locks_decode_step(const locks_cache_t* cache, const locks_summary_t* summary,
                                 const locks_params_t* params, const void* q, void* out, float* lse,
                                 int32_t* sel_pages, int32_t* sel_count, void* ws, size_t ws_bytes,
                                 void* stream) {
  locks_status_t st = check_cache(cache, true);
  if (st != LOCKS_OK) return st;
  if (!cache->n_summarized) return LOCKS_ERR_INVALID_ARG;
  if ((st = check_params(cache, params)) != LOCKS_OK) return st;
  if ((st = check_summary(summary, true)) != LOCKS_OK) return st;
  if (!q || !out || ((sel_pages == nullptr) != (sel_count == nullptr))) return LOCKS_ERR_INVALID_ARG;
  Plan pl = make_plan(cache, params);
  if (!pl.ok) return LOCKS_ERR_UNSUPPORTED;
  if ((st = check_ws(ws, ws_bytes, pl)) != LOCKS_OK) return st;
  int32_t* sel = sel_pages ? sel_pages : at<int32_t>(ws, pl.off_sel);
  int32_t* cnt = sel_count ? sel_count : at<int32_t>(ws, pl.off_selcnt);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (pl.fused) {
    // the scan, then one attention kernel whose clusters select the pages
    if ((st = run_select(cache, summary, params, pl, q, nullptr, nullptr, nullptr, ws, s)) != LOCKS_OK) return st;
    return run_attend(cache, params, pl, q, sel, cnt, out, lse, nullptr, ws, kAttendFused, s, true);
  }
  if ((st = run_select(cache, summary, params, pl, q, sel, cnt, nullptr, ws, s, true)) != LOCKS_OK) return st;
  return run_attend(cache, params, pl, q, sel, cnt, out, lse, nullptr, ws, kAttendSparse, s, true);
}

locks_status_t locks_decode_step_launches(const locks_cache_t* cache, const locks_summary_t* summary,
                                          const locks_params_t* params, int32_t* launches) {
  if (!launches) return LOCKS_ERR_INVALID_ARG;
  locks_status_t st = check_cache(cache, false);
  if (st != LOCKS_OK) return st;
  if ((st = check_params(cache, params)) != LOCKS_OK) return st;
  if ((st = check_summary(summary, true)) != LOCKS_OK) return st;
  Plan pl = make_plan(cache, params);
  if (!pl.ok) return LOCKS_ERR_UNSUPPORTED;
  *launches = pl.fused ? 2 : 3;
  return LOCKS_OK;
}

locks_status_t locks_dense_decode(const locks_cache_t* cache, const locks_params_t* params, const void* q,
                                  void* out, float* lse, void* ws, size_t ws_bytes, void* stream) {
  locks_status_t st = check_cache(cache, true);
  if (st != LOCKS_OK) return st;
  if ((st = check_params(cache, params)) != LOCKS_OK) return st;
  if (!q || !out) return LOCKS_ERR_INVALID_ARG;
  Plan pl = make_plan(cache, params);
  if (!pl.ok) return LOCKS_ERR_UNSUPPORTED;
  if ((st = check_ws(ws, ws_bytes, pl)) != LOCKS_OK) return st;
  return run_attend(cache, params, pl, q, nullptr, nullptr, out, lse, nullptr, ws, kAttendDense,
                    static_cast<cudaStream_t>(stream));
}

locks_status_t locks_exact_page_lse(const locks_cache_t* cache, const locks_params_t* params, const void* q,
                                    float* page_lse, void* stream) {
  if (!cache || !cache->k_pool || !cache->block_table || !cache->seq_lens) return LOCKS_ERR_INVALID_ARG;
  locks_status_t st = check_cache(cache, false);
  if (st != LOCKS_OK) return st;
  if ((reinterpret_cast<uintptr_t>(cache->k_pool) & 15)) return LOCKS_ERR_INVALID_ARG;
  if ((st = check_params(cache, params)) != LOCKS_OK) return st;
  if (!q || !page_lse) return LOCKS_ERR_INVALID_ARG;
  Plan pl = make_plan(cache, params);
  return run_attend(cache, params, pl, q, nullptr, nullptr, nullptr, nullptr, page_lse, nullptr, kAttendPageLse,
                    static_cast<cudaStream_t>(stream));
}

locks_status_t locks_get_device_error(void* ws, int32_t* code, void* stream) {
  if (!ws || !code) return LOCKS_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int v = 0;
  if (cudaMemcpyAsync(&v, ws, sizeof(int), cudaMemcpyDeviceToHost, s) != cudaSuccess) return LOCKS_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return LOCKS_ERR_CUDA;
  if (cudaMemsetAsync(ws, 0, sizeof(int), s) != cudaSuccess) return LOCKS_ERR_CUDA;
  *code = v;
  return v ? LOCKS_ERR_DEVICE : LOCKS_OK;
}

}  // extern "C"
