// Summary scan: the page-mass estimate s_hat for every summarised page and
// every query head of a GQA group.
//
// LOCKS explainer (gist.science), §2 "Reconstructie en Selectie": for page j
//   s_hat_j(q) = ln sum_{i in P_j} exp( (V_j^T q) . c_i / sqrt(d) ),
// i.e. project q onto the page basis, rebuild the P within-page logits from
// the coefficients and take their log-sum-exp (LOCKS abstract: "reconstructs
// within-page logits, estimates each page's attention mass by log-sum-exp").
// The summaries are "scanned in full each step" (abstract): this kernel is the
// dominant byte stream of the decode step.
//
// One warp handles one page-head at a time, for all G <= 16 heads of its
// group at once, with two bf16 tensor-core contractions:
//   (1) W^T = Q V_j        m16n8k16, M = heads, N = basis vectors, K = d.
//       The contraction index d is permuted so that each lane's 16-byte load
//       of a basis row (d = 32s+8c .. +8) is exactly its B fragment for two
//       k-steps; the query A fragments use the same permutation.  bf16 x bf16
//       products are exact in the fp32 accumulator.
//   (2) L^T = W^T C_j^T    m16n8k8 (r <= 8) or m16n8k16 (r = 16), M = heads,
//       N = tokens, K = r.  The fp32 W is split into three bf16 terms
//       (hi + mid + lo, 24 bits) so the second product keeps fp32 accuracy.
//       The accumulator of (1) is already in the A-fragment layout of (2), and
//       token n-tile jt, column g is token 8*jt + g, so each coefficient load
//       is one 4-byte word per lane and 128 contiguous bytes per warp.
// Then a base-2 log-sum-exp over the 64 tokens per head (two xor-shuffles
// across the four lanes of a row).  Each CTA also reduces its pages' s_hat
// into a per-head (max, sum) pair, from which the top-k kernel gets the total
// estimated mass Z_h of each head without re-reading every s_hat.
#include "common.cuh"
#include "kernels.h"

namespace locks {

namespace {

struct PageData {
  uint4 bv[4];      // basis row g:   d = 32s + 8c .. +8, s = 0..3
  uint4 bw[4];      // basis row g+8  (r > 8 only)
  uint32_t cb[8];   // coefficients (2c, 2c+1) of token 8*jt + g
  uint32_t cc[8];   // coefficients (2c+8, 2c+9) of token 8*jt + g (r > 8 only)
};

template <bool R16>
__device__ __forceinline__ void load_page(PageData& p, const uint16_t* bas, const uint16_t* coe, int g,
                                          int c, int r) {
  const uint4 z4 = make_uint4(0, 0, 0, 0);
#pragma unroll
  for (int s = 0; s < 4; ++s)
    p.bv[s] = (g < r) ? __ldg(reinterpret_cast<const uint4*>(bas + g * kHeadDim + 32 * s + 8 * c)) : z4;
  if (R16) {
#pragma unroll
    for (int s = 0; s < 4; ++s)
      p.bw[s] = (g + 8 < r)
                    ? __ldg(reinterpret_cast<const uint4*>(bas + (g + 8) * kHeadDim + 32 * s + 8 * c))
                    : z4;
  }
#pragma unroll
  for (int jt = 0; jt < 8; ++jt)
    p.cb[jt] = (2 * c < r) ? __ldg(reinterpret_cast<const uint32_t*>(coe + (8 * jt + g) * r + 2 * c)) : 0u;
  if (R16) {
#pragma unroll
    for (int jt = 0; jt < 8; ++jt)
      p.cc[jt] =
          (2 * c + 8 < r) ? __ldg(reinterpret_cast<const uint32_t*>(coe + (8 * jt + g) * r + 2 * c + 8)) : 0u;
  }
}

// x -> hi + mid + lo with each term a bf16; returned as packed pairs for (x0, x1).
__device__ __forceinline__ void split3(float x0, float x1, uint32_t& hi, uint32_t& mid, uint32_t& lo) {
  float h0 = bf16_round(x0), h1 = bf16_round(x1);
  float r0 = x0 - h0, r1 = x1 - h1;
  float m0 = bf16_round(r0), m1 = bf16_round(r1);
  hi = pack_bf16(h0, h1);
  mid = pack_bf16(m0, m1);
  lo = pack_bf16(r0 - m0, r1 - m1);
}

template <bool G16, bool R16>
__global__ void __launch_bounds__(kScanThreads, 2) scan_kernel(const ScanArgs a) {
  __shared__ float2 red[kScanWarps][16];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, c = lane & 3;
  const int bh = blockIdx.y, chunk = blockIdx.x;
  const int b = bh / a.num_kv_heads, hkv = bh % a.num_kv_heads;
  const int G = a.group, r = a.rank;

  pdl_wait();

  const int L = a.seq_lens[b];
  int ns = a.n_summarized[b];
  const int nfull = L < 0 ? 0 : L / kPage;
  int cap = nfull < a.max_pages ? nfull : a.max_pages;
  if (ns > cap || ns < 0 || L > a.max_pages * kPage) {
    if (threadIdx.x == 0 && chunk == 0) set_error(a.err, LOCKS_DEVERR_LENGTHS);
    ns = ns < 0 ? 0 : (ns > cap ? cap : ns);
  }
  const int j0 = chunk * a.chunk_pages;
  const int j1 = min(j0 + a.chunk_pages, ns);

  // Query A fragments with the permuted contraction index.
  const int Hq = a.num_kv_heads * G;
  uint4 qa[4], qb[4];
  {
    const uint16_t* qrow = a.q + ((size_t)b * Hq + (size_t)hkv * G) * kHeadDim;
#pragma unroll
    for (int s = 0; s < 4; ++s) {
      qa[s] = (g < G) ? __ldg(reinterpret_cast<const uint4*>(qrow + g * kHeadDim + 32 * s + 8 * c))
                      : make_uint4(0, 0, 0, 0);
      qb[s] = (G16 && g + 8 < G)
                  ? __ldg(reinterpret_cast<const uint4*>(qrow + (g + 8) * kHeadDim + 32 * s + 8 * c))
                  : make_uint4(0, 0, 0, 0);
    }
  }

  const size_t ph_stride_b = (size_t)r * kHeadDim;  // elements per page-head of basis
  const size_t ph_stride_c = (size_t)kPage * r;     // elements per page-head of coeffs
  const int32_t* bt = a.block_table + (size_t)b * a.max_pages;

  float zm0 = -INFINITY, zl0 = 0.f, zm1 = -INFINITY, zl1 = 0.f;

  PageData cur, nxt;
  int j = j0 + warp;
  bool have = j < j1;
  bool ok_cur = false;
  if (have) {
    int phys = bt[j];
    ok_cur = phys >= 0 && phys < a.pages_total;
    if (!ok_cur) { if (lane == 0) set_error(a.err, LOCKS_DEVERR_BLOCK_TABLE); phys = 0; }
    size_t ph = (size_t)phys * a.num_kv_heads + hkv;
    load_page<R16>(cur, a.basis_t + ph * ph_stride_b, a.coeffs + ph * ph_stride_c, g, c, r);
  }
  while (have) {
    const int jn = j + kScanWarps;
    const bool have_n = jn < j1;
    bool ok_n = false;
    if (have_n) {
      int phys = bt[jn];
      ok_n = phys >= 0 && phys < a.pages_total;
      if (!ok_n) { if (lane == 0) set_error(a.err, LOCKS_DEVERR_BLOCK_TABLE); phys = 0; }
      size_t ph = (size_t)phys * a.num_kv_heads + hkv;
      load_page<R16>(nxt, a.basis_t + ph * ph_stride_b, a.coeffs + ph * ph_stride_c, g, c, r);
    }

    if (ok_cur) {
      // (1) W^T = Q V  (16 heads x 8 or 16 basis vectors)
      float w0[4] = {0.f, 0.f, 0.f, 0.f}, w1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int s = 0; s < 4; ++s) {
        mma_16816(w0, qa[s].x, qb[s].x, qa[s].y, qb[s].y, cur.bv[s].x, cur.bv[s].y);
        mma_16816(w0, qa[s].z, qb[s].z, qa[s].w, qb[s].w, cur.bv[s].z, cur.bv[s].w);
        if (R16) {
          mma_16816(w1, qa[s].x, qb[s].x, qa[s].y, qb[s].y, cur.bw[s].x, cur.bw[s].y);
          mma_16816(w1, qa[s].z, qb[s].z, qa[s].w, qb[s].w, cur.bw[s].z, cur.bw[s].w);
        }
      }
      // fold scale * log2(e), split into three bf16 terms
      uint32_t h0, m0, l0, h1, m1, l1, h2 = 0, m2 = 0, l2 = 0, h3 = 0, m3 = 0, l3 = 0;
      split3(w0[0] * a.scale_log2, w0[1] * a.scale_log2, h0, m0, l0);
      split3(w0[2] * a.scale_log2, w0[3] * a.scale_log2, h1, m1, l1);
      if (R16) {
        split3(w1[0] * a.scale_log2, w1[1] * a.scale_log2, h2, m2, l2);
        split3(w1[2] * a.scale_log2, w1[3] * a.scale_log2, h3, m3, l3);
      }
      // (2) logits (base-2) for 16 heads x 64 tokens
      float d[8][4];
#pragma unroll
      for (int jt = 0; jt < 8; ++jt) {
        d[jt][0] = d[jt][1] = d[jt][2] = d[jt][3] = 0.f;
        if (R16) {
          mma_16816(d[jt], l0, l1, l2, l3, cur.cb[jt], cur.cc[jt]);
          mma_16816(d[jt], m0, m1, m2, m3, cur.cb[jt], cur.cc[jt]);
          mma_16816(d[jt], h0, h1, h2, h3, cur.cb[jt], cur.cc[jt]);
        } else {
          mma_1688(d[jt], l0, l1, cur.cb[jt]);
          mma_1688(d[jt], m0, m1, cur.cb[jt]);
          mma_1688(d[jt], h0, h1, cur.cb[jt]);
        }
      }
      // base-2 log-sum-exp over the 64 tokens of each head row
      float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
      for (int jt = 0; jt < 8; ++jt) {
        mx0 = fmaxf(mx0, fmaxf(d[jt][0], d[jt][1]));
        if (G16) mx1 = fmaxf(mx1, fmaxf(d[jt][2], d[jt][3]));
      }
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
      if (G16) {
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
      }
      float s0 = 0.f, s1 = 0.f;
#pragma unroll
      for (int jt = 0; jt < 8; ++jt) {
        s0 += fast_exp2(d[jt][0] - mx0) + fast_exp2(d[jt][1] - mx0);
        if (G16) s1 += fast_exp2(d[jt][2] - mx1) + fast_exp2(d[jt][3] - mx1);
      }
      s0 += __shfl_xor_sync(0xffffffffu, s0, 1);
      s0 += __shfl_xor_sync(0xffffffffu, s0, 2);
      if (G16) {
        s1 += __shfl_xor_sync(0xffffffffu, s1, 1);
        s1 += __shfl_xor_sync(0xffffffffu, s1, 2);
      }
      const float e0 = mx0 + fast_log2(s0);
      lse2_merge(zm0, zl0, e0, 1.f);
      float e1 = 0.f;
      if (G16) {
        e1 = mx1 + fast_log2(s1);
        lse2_merge(zm1, zl1, e1, 1.f);
      }
      if (c == 0) {
        float* dst = a.shat + ((size_t)bh * a.max_pages + j) * G;
        if (g < G) dst[g] = e0 * kLn2;
        if (G16 && g + 8 < G) dst[g + 8] = e1 * kLn2;
        if (a.page_lse) {
          float* pl = a.page_lse + ((size_t)b * Hq + (size_t)hkv * G) * a.max_pages + j;
          if (g < G) pl[(size_t)g * a.max_pages] = e0 * kLn2;
          if (G16 && g + 8 < G) pl[(size_t)(g + 8) * a.max_pages] = e1 * kLn2;
        }
      }
    }
    cur = nxt;
    ok_cur = ok_n;
    j = jn;
    have = have_n;
  }

  pdl_launch_dependents();

  if (c == 0) {
    red[warp][g] = make_float2(zm0, zl0);
    if (G16) red[warp][g + 8] = make_float2(zm1, zl1);
  }
  __syncthreads();
  if (threadIdx.x < G) {
    float m = -INFINITY, l = 0.f;
#pragma unroll
    for (int w = 0; w < kScanWarps; ++w) lse2_merge(m, l, red[w][threadIdx.x].x, red[w][threadIdx.x].y);
    a.part[((size_t)bh * a.n_chunks + chunk) * G + threadIdx.x] = make_float2(m, l);
  }
}

template <bool G16, bool R16>
cudaError_t launch_one(const ScanArgs& a, cudaStream_t s, bool pdl) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.n_chunks, a.batch * a.num_kv_heads, 1);
  cfg.blockDim = dim3(kScanThreads, 1, 1);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, scan_kernel<G16, R16>, a);
}

}  // namespace

cudaError_t launch_scan(const ScanArgs& a, cudaStream_t s, bool pdl) {
  const bool g16 = a.group > 8, r16 = a.rank > 8;
  if (g16) return r16 ? launch_one<true, true>(a, s, pdl) : launch_one<true, false>(a, s, pdl);
  return r16 ? launch_one<false, true>(a, s, pdl) : launch_one<false, false>(a, s, pdl);
}

}  // namespace locks
