// Internal launch interface between the C-ABI layer (api.cu) and the kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace locks {

// Summary scan: page-mass estimates s_hat for every summarised page and head.
struct ScanArgs {
  const uint16_t* basis_t;     // bf16 [pages_total][Hkv][r][d]
  const uint16_t* coeffs;      // bf16 [pages_total][Hkv][P][r]
  const uint16_t* q;           // bf16 [B][Hq][d]
  const int32_t* block_table;  // [B][max_pages]
  const int32_t* seq_lens;     // [B]
  const int32_t* n_summarized; // [B]
  float* shat;                 // ws: [B*Hkv][max_pages][G] natural log
  float2* part;                // ws: [B*Hkv][n_chunks][G] (max, sum) of base-2 LSE
  float* page_lse;             // optional [B][Hq][max_pages]
  int* err;
  int batch, num_kv_heads, group, rank, max_pages, pages_total;
  int chunk_pages, n_chunks;
  float scale_log2;            // scale * log2(e)
  int q4;                      // 1: basis_t holds LOCKS_DTYPE_Q4 blocks (coeffs unused)
  int packed;                  // 1: basis_t holds LOCKS_DTYPE_BF16_PACKED blocks (coeffs unused)
  int page_size;               // P: 64 or 16
  int heads_per_block;         // HG: KV heads one CTA scans together (a power of two dividing Hkv, <= 4)
  // set by the launcher: ring of `slots` slots, one page of the head block each
  int slots, slot_bytes, basis_bytes, coef_bytes;
};

// GSA scores + top-k (chunk-local candidates, merged by the last CTA).
struct TopkArgs {
  const float* shat;
  const float2* part;
  int n_scan_chunks;
  const int32_t* seq_lens;
  const int32_t* n_summarized;
  uint32_t* cand_key;   // ws: [B*Hkv][n_chunks][k_max]
  int32_t* cand_idx;    // ws: same
  unsigned* counters;   // ws: [B*Hkv]
  int32_t* sel_pages;   // [B*Hkv][k_max]
  int32_t* sel_count;   // [B*Hkv]
  const int32_t* block_table;  // read before the grid dependency wait when sel_phys is set
  int32_t* sel_phys;    // ws: [B*Hkv][k_max] physical page of each selected page (one-chunk problems), or null
  int* err;
  int batch, num_kv_heads, group, max_pages, k_max;
  int chunk_pages, n_chunks;
  size_t smem_keys;     // capacity (entries) of the dynamic key buffer
  int page_size;
};

// Paged flash-decode over a page list (sparse), every page (dense), or the
// exact per-page LSE of every page (page_lse mode).
struct AttendArgs {
  const uint16_t* q;
  const int32_t* block_table;
  const int32_t* seq_lens;
  const int32_t* n_summarized;
  const int32_t* sel_pages;   // sparse mode only
  const int32_t* sel_count;   // sparse mode only
  const int32_t* sel_phys;    // sparse mode inside the decode step: physical pages of sel_pages, or null
  uint16_t* out;              // bf16 [B][Hq][d]
  float* lse;                 // optional [B][Hq]
  float* page_lse;            // page_lse mode: [B][Hq][max_pages]
  float* part_o;              // ws: [B*Hkv][n_splits][G][d]
  float2* part_ml;            // ws: [B*Hkv][n_splits][G]
  unsigned* counters;         // ws: [B*Hkv]
  int* err;
  int batch, num_kv_heads, group, max_pages, pages_total, k_max;
  int n_splits;               // CTAs per problem = cluster * clusters per problem
  int cluster;                // CTAs per thread-block cluster (1 in page-LSE mode)
  int inputs_early;           // 1: the step's inputs may be read before the grid dependency wait
  float scale_log2;
  int page_size;              // P: 64 (one page per 64-token tile) or 16 (four pages per tile)
  // fused mode only: the scan's page-mass estimates and per-CTA partials,
  // from which the cluster selects the pages itself
  const float* shat;          // ws: [B*Hkv][max_pages][G] natural log
  const float2* part;         // ws: [B*Hkv][n_scan_chunks][G] (max, sum) of base-2 LSE
  int n_scan_chunks;
  const uint16_t* k_pool16;   // fused mode: pool bases for L2 prefetches of likely pages
  const uint16_t* v_pool16;
  int32_t* sel_pages_out;     // fused mode: the page list it selected, [B*Hkv][k_max] (as locks_select)
  int32_t* sel_count_out;     // fused mode: [B*Hkv]
  unsigned long long* trace_cta;  // tracing builds only: per-CTA timestamps [B*Hkv][n_splits][16], or null
};

// kAttendFused: the sparse mode with the group-shared top-k computed inside
// the thread-block cluster from the scan's outputs (64-token pages, k_max <=
// kFusedMaxK, at most kAttendThreads summarised pages per CTA of the cluster).
enum AttendMode { kAttendSparse = 0, kAttendDense = 1, kAttendPageLse = 2, kAttendFused = 3 };
constexpr int kFusedMaxK = 32;
constexpr int kFusedPrefetch = 4;  // each CTA's best pages whose K/V are prefetched into L2 before the merge

// Summary builder.
struct BuildArgs {
  const uint16_t* k_pool;
  void* basis_t;
  void* coeffs;
  const int32_t* page_ids;
  int n, num_kv_heads, rank, pages_total;
  int format;  // LOCKS_DTYPE_BF16 / _F32 (basis_t + coeffs) or _Q4 (packed blocks in basis_t)
  int* err;
  int page_size;
};

cudaError_t launch_scan(const ScanArgs& a, cudaStream_t s, bool pdl);
cudaError_t launch_topk(const TopkArgs& a, cudaStream_t s, bool pdl);
cudaError_t launch_attend(const AttendArgs& a, const CUtensorMap& tk, const CUtensorMap& tv,
                          int mode, cudaStream_t s, bool pdl);
cudaError_t launch_build(const BuildArgs& a, cudaStream_t s);

size_t topk_smem_bytes(size_t keys);
int topk_pages_per_cta(int group);  // pages one top-k CTA scores
int attend_max_cluster(int mode, int page_size);  // largest placeable cluster (<= 16) for that mode
                                                  // (kAttendFused: page_size 64 only)
int attend_active_clusters(int mode, int cs, int page_size);  // clusters of cs CTAs resident at once
// Scan CTA (one per SM): 16 consumer warps + 1 producer warp.
constexpr int kScanWarps = 16;
// KV heads one scan CTA covers: the largest power of two <= 4 dividing Hkv
// (measured on GB300: 4 beats 8 at 128K context and ties elsewhere).
inline int scan_heads_per_block(int num_kv_heads) {
  int hg = 4;
  while (num_kv_heads % hg) hg /= 2;
  return hg;
}
constexpr int kScanThreads = (kScanWarps + 1) * 32;
constexpr int kTopkThreads = 512;
constexpr int kAttendThreads = 128;

}  // namespace locks
