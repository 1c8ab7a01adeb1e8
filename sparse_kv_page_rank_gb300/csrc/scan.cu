// Summary scan: the page-mass estimate s_hat for every summarised page and
// every query head of a GQA group.
//
// LOCKS explainer (gist.science), §2 "Reconstructie en Selectie": for page j
//   s_hat_j(q) = ln sum_{i in P_j} exp( (V_j^T q) . c_i / sqrt(d) ),
// i.e. project q onto the page basis, rebuild the P within-page logits from
// the coefficients and take their log-sum-exp (LOCKS abstract: "reconstructs
// within-page logits, estimates each page's attention mass by log-sum-exp").
// The summaries are "scanned in full each step" (abstract): this kernel is the
// dominant byte stream of the decode step, so it is built to keep HBM busy.
//
// Memory (warp-specialised): each CTA owns a contiguous range of pages of one
// sequence for a block of HG KV heads (HG the largest power of two <= 4
// dividing the KV-head count), and a ring of S slots in shared memory, one
// page of the block per slot.  The summaries of a physical page are laid out
// head after head, so a page's bases for all HG heads are one contiguous
// range and so are its coefficients: one producer warp fills a slot with two
// TMA bulk copies per page and head block, or one for the quantised format
// and for packed bf16 blocks (basis and coefficients of a page-head together).
// The copy count, not the bytes, limits a TMA read of small pieces (about
// 40 ns per copy per SM measured on GB300, whatever the size up to ~1 KiB), so
// covering HG page-heads per copy is what lets the scan stream at HBM speed.
// The loads carry an L2 evict-first policy: every summary is read once per
// step, and the s_hat rows written here should stay in L2 for the top-k.
// Each of the producer's lanes owns a slot, waits for it to be released and
// refills it, completing on the slot's "full" mbarrier.  Sixteen consumer
// warps only compute: warp w serves head w mod HG of the block and every
// (16 / HG)-th page; it waits on the slot's full barrier and arrives on the
// slot's "empty" barrier, which completes when all HG heads are done.
//
// Compute: one consumer warp per page-head, all G <= 16 heads of the group at
// once, two bf16 tensor-core contractions:
//   (1) W^T = Q V_j        m16n8k16, M = heads, N = basis vectors, K = d.
//       The contraction index d is permuted so that each lane's 16-byte piece
//       of a basis row (d = 32s+8c .. +8) is exactly its B fragment for two
//       k-steps; the query A fragments use the same permutation.  bf16 x bf16
//       products are exact in the fp32 accumulator.
//   (2) L^T = W^T C_j^T    m16n8k8 (r <= 8) or m16n8k16 (r > 8), M = heads,
//       N = tokens, K = r.  The fp32 W is split into two bf16 terms
//       (hi + lo, about 16 bits of W, far inside the 1e-3 relative page-LSE
//       tolerance) so the second product keeps most of fp32's accuracy.  The
//       accumulator of (1) is already in the A-fragment layout of (2);
//       n-tile jt, column g is token 8*jt + g.
// Then a base-2 log-sum-exp over the P tokens per head (P = 64 or 16; at 16
// the first contraction is the same and the second one a quarter as long, so
// a page-head costs nearly as much as at 64 while covering a quarter of the
// tokens: the explainer's §2 "Kernmechanisme" notes that the summary is
// then about 10% of the page's KV bytes).  Each CTA also
// reduces its pages' s_hat into a per-head (max, sum) pair, from which the
// top-k kernel gets the total estimated mass Z_h of each head without
// re-reading every s_hat.
#include "common.cuh"
#include "kernels.h"

namespace locks {

namespace {

// The slot count S is a multiple of the number of warp groups (16 / HG):
// page p goes to slot p mod S and to the warps of group p mod (16 / HG), so
// every slot is always consumed by the same warps, which therefore wait on the
// slot's phases strictly in order.  (With a slot shared by several groups, a
// warp could wait on the parity of a slot's next phase while the current one
// is still incomplete; a parity wait on a phase two ahead returns at once, on
// stale data.)
constexpr int kMaxSlots = 32;  // one producer lane per slot
// ring bytes: one CTA per SM; the quantised format also stages centroid data
constexpr int kRingBytes = 200 * 1024;
constexpr int kRingBytesQ4 = 176 * 1024;

// Quantised format: q . mu is computed for kMuBatch pages of a warp at once
// (one MMA tile, a page per column) instead of page by page; each warp
// stages its pending pages' centroid codes, scales and base LSEs here.
constexpr int kMuBatch = 8;
constexpr int kStageMu = kScanWarps * kMuBatch * 128;        // centroid codes
constexpr int kStageSmu = kScanWarps * kMuBatch * 4;         // centroid scales
constexpr int kStagePend = kScanWarps * kMuBatch * 16 * 4;   // base-2 LSE per head row

// Layout of one slot (a page of a head block) and the ring for these shapes.
struct SlotLayout {
  int basis_bytes;  // per page-head: r rows of 256 B (quantised or packed bf16: the whole block)
  int coef_bytes;   // per page-head: P x r bf16 (quantised or packed bf16: 0, inside the block)
  int slot_bytes;   // HG page-heads
  int slots;
  int smem;         // dynamic shared memory of the kernel
};

SlotLayout slot_layout(int rank, int page_size, int hg, bool q4, bool packed) {
  SlotLayout L;
  L.basis_bytes = q4 ? LOCKS_Q4_BLOCK_BYTES(rank, page_size)
                     : rank * kHeadDim * 2 + (packed ? page_size * rank * 2 : 0);
  L.coef_bytes = q4 || packed ? 0 : page_size * rank * 2;
  L.slot_bytes = hg * (L.basis_bytes + L.coef_bytes);
  const int groups = kScanWarps / hg;
  int s = (q4 ? kRingBytesQ4 : kRingBytes) / L.slot_bytes;
  s = s < kMaxSlots ? s : kMaxSlots;
  s -= s % groups;
  L.slots = s;
  L.smem = s * L.slot_bytes + 128 + (q4 ? kStageMu + kStageSmu + kStagePend : 0);
  return L;
}

// x -> hi + lo, each term a bf16 (truncated; the two keep about 16 bits of
// x), returned as packed pairs for (x0, x1), x0 in the low half.
__device__ __forceinline__ void split2(float x0, float x1, uint32_t& hi, uint32_t& lo) {
  const uint32_t u0 = __float_as_uint(x0) & 0xffff0000u, u1 = __float_as_uint(x1) & 0xffff0000u;
  const float r0 = x0 - __uint_as_float(u0), r1 = x1 - __uint_as_float(u1);
  hi = __byte_perm(u0, u1, 0x7632);
  lo = __byte_perm(__float_as_uint(r0), __float_as_uint(r1), 0x7632);
}

template <int N>
__device__ __forceinline__ float tree_max(const float* v) {
  if constexpr (N == 1) {
    return v[0];
  } else {
    return fmaxf(tree_max<N / 2>(v), tree_max<N / 2>(v + N / 2));
  }
}
template <int N>
__device__ __forceinline__ float tree_sum(const float* v) {
  if constexpr (N == 1) {
    return v[0];
  } else {
    return tree_sum<N / 2>(v) + tree_sum<N / 2>(v + N / 2);
  }
}

// Base-2 log-sum-exp of N values per lane over the lanes of one head (the
// xor masks name the lanes sharing the head; 0 = unused).  When every lane's
// values lie in (-100, 120), 2^v neither overflows nor loses the page's
// mass, and the shared maximum is skipped.
template <int N, int X0, int X1, int X2>
__device__ __forceinline__ float lse2_lanes(float* v) {
  float mx = tree_max<N>(v);
  const bool direct = __all_sync(0xffffffffu, mx > -100.f && mx < 120.f);
  if (!direct) {
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, X0));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, X1));
    if (X2) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, X2));
  } else {
    mx = 0.f;
  }
#pragma unroll
  for (int e = 0; e < N; ++e) v[e] = fast_exp2(v[e] - mx);
  float sm = tree_sum<N>(v);
  sm += __shfl_xor_sync(0xffffffffu, sm, X0);
  sm += __shfl_xor_sync(0xffffffffu, sm, X1);
  if (X2) sm += __shfl_xor_sync(0xffffffffu, sm, X2);
  return mx + fast_log2(sm);
}

// G16: more than 8 heads in the group (both row halves of the MMA tiles).
// R16: rank above 8 (two basis n-tiles, k16 second contraction).
// GRP2: at most 4 heads and rank <= 8: the second contraction packs two
// 32-token groups into one m16n8k16 (rows 0-3 use k 0-7 = coefficients of
// tokens 16jt+n, rows 4-7 use k 8-15 = coefficients of tokens 16jt+8+n),
// which halves its MMAs, exponentials and reductions.
//
// Page-head in shared memory at `slot` -> base-2 LSE for head g (e0) and,
// with G16, head g + 8 (e1).
template <bool G16, bool R16, bool GRP2, int P>
__device__ __forceinline__ void compute_page(uint32_t bas, uint32_t coef, const uint4 (&qa)[4], const uint4 (&qb)[4],
                                             int r, float scale_log2, int lane, float& e0, float& e1) {
  constexpr int NT = P / 8;  // 8-token n-tiles of the page
  const int g = lane >> 2, c = lane & 3;
  const uint4 z4 = make_uint4(0, 0, 0, 0);
  // basis row `row`, 16-byte piece d = 32*s + 8c (linear rows of 256 B)
  auto basis_piece = [&](int row, int s) -> uint32_t { return bas + row * 256 + s * 64 + c * 16; };
  auto coef_word = [&](int jt, int k0) -> uint32_t { return coef + (uint32_t)(((8 * jt + g) * r + k0) * 2); };

  // (1) W^T = Q V  (16 heads x 8 or 16 basis vectors); two accumulators per
  // n-tile halve the dependent MMA chain
  float w0[4] = {0.f, 0.f, 0.f, 0.f}, w1[4] = {0.f, 0.f, 0.f, 0.f};
  float x0[4] = {0.f, 0.f, 0.f, 0.f}, x1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int s = 0; s < 4; ++s) {
    const uint4 bv = (g < r) ? lds128(basis_piece(g, s)) : z4;
    mma_16816(w0, qa[s].x, qb[s].x, qa[s].y, qb[s].y, bv.x, bv.y);
    mma_16816(x0, qa[s].z, qb[s].z, qa[s].w, qb[s].w, bv.z, bv.w);
    if (R16) {
      const uint4 bw = (g + 8 < r) ? lds128(basis_piece(g + 8, s)) : z4;
      mma_16816(w1, qa[s].x, qb[s].x, qa[s].y, qb[s].y, bw.x, bw.y);
      mma_16816(x1, qa[s].z, qb[s].z, qa[s].w, qb[s].w, bw.z, bw.w);
    }
  }
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    w0[e] += x0[e];
    if (R16) w1[e] += x1[e];
  }

  if (GRP2) {
    // rows g < 4 hold heads 0-3 in the k 0-7 half of the A fragment, rows
    // 4-7 the same heads (repeated Q rows) in the k 8-15 half
    uint32_t hh, mm;
    split2(w0[0] * scale_log2, w0[1] * scale_log2, hh, mm);
    const bool lo_half = lane < 16;
    const uint32_t ha0 = lo_half ? hh : 0u, ha2 = lo_half ? 0u : hh;
    const uint32_t ma0 = lo_half ? mm : 0u, ma2 = lo_half ? 0u : mm;
    uint32_t cbv[NT];
#pragma unroll
    for (int jt = 0; jt < NT; ++jt) cbv[jt] = (2 * c < r) ? lds32(coef_word(jt, 2 * c)) : 0u;
    float d[NT / 2][4];
    float v[NT];
#pragma unroll
    for (int jt = 0; jt < NT / 2; ++jt) {
      d[jt][0] = d[jt][1] = d[jt][2] = d[jt][3] = 0.f;
      mma_16816(d[jt], ma0, 0u, ma2, 0u, cbv[2 * jt], cbv[2 * jt + 1]);
      mma_16816(d[jt], ha0, 0u, ha2, 0u, cbv[2 * jt], cbv[2 * jt + 1]);
      v[2 * jt] = d[jt][0];
      v[2 * jt + 1] = d[jt][1];
    }
    e0 = lse2_lanes<NT, 1, 2, 16>(v);
    e1 = 0.f;
    return;
  }

  // fold scale * log2(e), split into two bf16 terms
  uint32_t h0, m0, h1, m1, h2 = 0, m2 = 0, h3 = 0, m3 = 0;
  split2(w0[0] * scale_log2, w0[1] * scale_log2, h0, m0);
  split2(w0[2] * scale_log2, w0[3] * scale_log2, h1, m1);
  if (R16) {
    split2(w1[0] * scale_log2, w1[1] * scale_log2, h2, m2);
    split2(w1[2] * scale_log2, w1[3] * scale_log2, h3, m3);
  }
  uint32_t cb[NT], cc[NT];
#pragma unroll
  for (int jt = 0; jt < NT; ++jt) {
    cb[jt] = (2 * c < r) ? lds32(coef_word(jt, 2 * c)) : 0u;
    cc[jt] = (R16 && 2 * c + 8 < r) ? lds32(coef_word(jt, 2 * c + 8)) : 0u;
  }
  // (2) logits (base-2) for 16 heads x P tokens
  float d[NT][4];
#pragma unroll
  for (int jt = 0; jt < NT; ++jt) {
    d[jt][0] = d[jt][1] = d[jt][2] = d[jt][3] = 0.f;
    if (R16) {
      mma_16816(d[jt], m0, m1, m2, m3, cb[jt], cc[jt]);
      mma_16816(d[jt], h0, h1, h2, h3, cb[jt], cc[jt]);
    } else {
      mma_1688(d[jt], m0, m1, cb[jt]);
      mma_1688(d[jt], h0, h1, cb[jt]);
    }
  }
  // base-2 log-sum-exp over the P tokens of each head row (P / 4 values per
  // lane, four lanes per row)
  float v[2 * NT];
#pragma unroll
  for (int jt = 0; jt < NT; ++jt) {
    v[2 * jt] = d[jt][0];
    v[2 * jt + 1] = d[jt][1];
  }
  e0 = lse2_lanes<2 * NT, 1, 2, 0>(v);
  e1 = 0.f;
  if (G16) {
#pragma unroll
    for (int jt = 0; jt < NT; ++jt) {
      v[2 * jt] = d[jt][2];
      v[2 * jt + 1] = d[jt][3];
    }
    e1 = lse2_lanes<2 * NT, 1, 2, 0>(v);
  }
}

// The same page-head estimate from the quantised, centred format (int4 basis
// codes, int8 centroid and coefficient codes, float32 scales; rank <= 8).
// The block's layout puts what one lane needs side by side: its four basis
// words, its coefficient codes and its two columns' scales are one 16-byte
// load each.  (1) runs on the basis codes in bf16 (exact: small integers),
// each basis vector's and coefficient column's scale is applied in fp32 on
// its column of W, and (2) runs in fp16: a byte code becomes an exact fp16 in
// two instructions per pair, and W is split into two fp16 terms (hi + lo,
// about 22 bits; hi saturates at +-65504, a logit contribution per code unit
// far beyond any softmax-relevant range).  Returns the LSE of the centred
// logits; q . mu shifts every logit of the head alike and is added later
// (mu_batch).
template <bool G16, bool GRP2, int P>
__device__ __forceinline__ void compute_page_q4(uint32_t slot, const uint4 (&qa)[4], const uint4 (&qb)[4], int r,
                                                float scale_log2, int lane, float& e0, float& e1) {
  constexpr int NT = P / 8;
  const int g = lane >> 2, c = lane & 3;
  const int rh = r >> 1;  // column pairs
  const uint32_t coef_off = 64 * r + kHeadDim, sc_off = 64 * r + kHeadDim + P * r;
  // (1) W^T = Q V on the basis codes: row g's words for elements 32s + 8c ..
  // +7, s = 0..3 (a row past the rank reads as all-zero codes)
  const uint4 nib = (g < r) ? lds128(slot + 64 * g + 16 * c) : make_uint4(0x88888888u, 0x88888888u, 0x88888888u,
                                                                            0x88888888u);
  const uint32_t nw[4] = {nib.x, nib.y, nib.z, nib.w};
  float w0[4] = {0.f, 0.f, 0.f, 0.f}, x0[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int s = 0; s < 4; ++s) {
    mma_16816(w0, qa[s].x, qb[s].x, qa[s].y, qb[s].y, u4pair_bf16(nw[s], 0), u4pair_bf16(nw[s], 4));
    mma_16816(x0, qa[s].z, qb[s].z, qa[s].w, qb[s].w, u4pair_bf16(nw[s], 8), u4pair_bf16(nw[s], 12));
  }
  // column 2c of W gets s_v[2c] s_c[2c], column 2c+1 likewise (and the
  // base-2 logit scale); this lane's coefficient codes: tokens g + 8t,
  // columns 2c, 2c+1, two bytes per n-tile t
  const bool has = c < rh;
  const uint4 sc4 = has ? lds128(slot + sc_off + 16 * c) : make_uint4(0u, 0u, 0u, 0u);
  const float f0 = __uint_as_float(sc4.x) * __uint_as_float(sc4.z) * scale_log2;
  const float f1 = __uint_as_float(sc4.y) * __uint_as_float(sc4.w) * scale_log2;
  uint32_t cw[(NT + 1) / 2];
  if constexpr (NT == 8) {
    const uint4 t = has ? lds128(slot + coef_off + 16 * (g * rh + c)) : make_uint4(0x80808080u, 0x80808080u,
                                                                                     0x80808080u, 0x80808080u);
    cw[0] = t.x;
    cw[1] = t.y;
    cw[2] = t.z;
    cw[3] = t.w;
  } else {
    static_assert(NT == 2, "64- or 16-token pages");
    cw[0] = has ? lds32(slot + coef_off + 4 * (g * rh + c)) : 0x80808080u;
  }
  uint32_t cb[NT];  // fp16 pair for n-tile t: (token g + 8t; columns 2c, 2c+1)
#pragma unroll
  for (int u = 0; u < NT / 2; ++u) u8quad_f16(cw[u], cb[2 * u], cb[2 * u + 1]);
  const float wa = (w0[0] + x0[0]) * f0, wb = (w0[1] + x0[1]) * f1;
  const float wc = (w0[2] + x0[2]) * f0, wd = (w0[3] + x0[3]) * f1;

  if (GRP2) {
    uint32_t hh, mm;
    split2_f16(wa, wb, hh, mm);
    const bool lo_half = lane < 16;
    const uint32_t ha0 = lo_half ? hh : 0u, ha2 = lo_half ? 0u : hh;
    const uint32_t ma0 = lo_half ? mm : 0u, ma2 = lo_half ? 0u : mm;
    float d[NT / 2][4];
    float v[NT];
#pragma unroll
    for (int jt = 0; jt < NT / 2; ++jt) {
      d[jt][0] = d[jt][1] = d[jt][2] = d[jt][3] = 0.f;
      mma_16816_f16(d[jt], ma0, 0u, ma2, 0u, cb[2 * jt], cb[2 * jt + 1]);
      mma_16816_f16(d[jt], ha0, 0u, ha2, 0u, cb[2 * jt], cb[2 * jt + 1]);
      v[2 * jt] = d[jt][0];
      v[2 * jt + 1] = d[jt][1];
    }
    e0 = lse2_lanes<NT, 1, 2, 16>(v);
    e1 = 0.f;
    return;
  }

  uint32_t h0, m0, h1, m1;
  split2_f16(wa, wb, h0, m0);
  split2_f16(wc, wd, h1, m1);
  float d[NT][4];
#pragma unroll
  for (int jt = 0; jt < NT; ++jt) {
    d[jt][0] = d[jt][1] = d[jt][2] = d[jt][3] = 0.f;
    mma_1688_f16(d[jt], m0, m1, cb[jt]);
    mma_1688_f16(d[jt], h0, h1, cb[jt]);
  }
  float v[2 * NT];
#pragma unroll
  for (int jt = 0; jt < NT; ++jt) {
    v[2 * jt] = d[jt][0];
    v[2 * jt + 1] = d[jt][1];
  }
  e0 = lse2_lanes<2 * NT, 1, 2, 0>(v);
  e1 = 0.f;
  if (G16) {
#pragma unroll
    for (int jt = 0; jt < NT; ++jt) {
      v[2 * jt] = d[jt][2];
      v[2 * jt + 1] = d[jt][3];
    }
    e1 = lse2_lanes<2 * NT, 1, 2, 0>(v);
  }
}

// q . mu for up to kMuBatch staged pages of one warp: one MMA tile whose
// column n is page n's centroid codes (biased bytes, exact in bf16); lane
// (g, c) ends with the dot products of head rows g and g + 8 with pages 2c
// and 2c + 1 (u[0..1] and u[2..3]).
__device__ __forceinline__ void mu_batch(uint32_t stage_mu, int nb, const uint4 (&qa)[4], const uint4 (&qb)[4],
                                         int lane, float (&u)[4]) {
  const int g = lane >> 2, c = lane & 3;
  float y[4] = {0.f, 0.f, 0.f, 0.f};
  u[0] = u[1] = u[2] = u[3] = 0.f;
#pragma unroll
  for (int s = 0; s < 4; ++s) {
    const uint2 m8 = (g < nb) ? lds64(stage_mu + 128 * g + 32 * s + 8 * c) : make_uint2(0x80808080u, 0x80808080u);
    mma_16816(u, qa[s].x, qb[s].x, qa[s].y, qb[s].y, u8pair_bf16(m8.x, 0), u8pair_bf16(m8.x, 2));
    mma_16816(y, qa[s].z, qb[s].z, qa[s].w, qb[s].w, u8pair_bf16(m8.y, 0), u8pair_bf16(m8.y, 2));
  }
#pragma unroll
  for (int e = 0; e < 4; ++e) u[e] += y[e];
}

template <bool G16, bool R16, bool GRP2, bool Q4, int P>
__global__ void __launch_bounds__(kScanThreads, 1) scan_kernel(const ScanArgs a) {
  extern __shared__ uint8_t ring_raw[];
  __shared__ float2 red[kScanWarps][16];
  __shared__ __align__(8) uint64_t full_bar[kMaxSlots], empty_bar[kMaxSlots];
  __shared__ int slot_ok[kMaxSlots];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, c = lane & 3;
  const int HG = a.heads_per_block, S = a.slots;
  const int ngrp = kScanWarps / HG;  // warp groups; each group serves every HG head of its pages
  const int nhb = a.num_kv_heads / HG;
  const int hblk = blockIdx.y, chunk = blockIdx.x;
  const int b = hblk / nhb, h0 = (hblk % nhb) * HG;
  const int G = a.group, r = a.rank;
  const uint32_t ring = (smem_u32(ring_raw) + 127u) & ~127u;
  const uint32_t slot_bytes = (uint32_t)a.slot_bytes;
  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], (uint32_t)HG);  // one arrival per head of the block
    }
    fence_mbar_init();
  }
  __syncthreads();

  trace_mark(a.err, kTrScanEnter, true);
  trace_mark(a.err, kTrScanLastEnter, false);
  const unsigned long long t_enter = trace_ns();
  pdl_wait();
  trace_mark(a.err, kTrScanWait, true);

  const int L = a.seq_lens[b];
  int ns = a.n_summarized[b];
  const int nfull = L < 0 ? 0 : L / P;
  const int cap = nfull < a.max_pages ? nfull : a.max_pages;
  if (ns > cap || ns < 0 || L > a.max_pages * P) {
    if (threadIdx.x == 0 && chunk == 0) set_error(a.err, LOCKS_DEVERR_LENGTHS);
    ns = ns < 0 ? 0 : (ns > cap ? cap : ns);
  }
  const int j0 = chunk * a.chunk_pages;
  const int j1 = min(j0 + a.chunk_pages, ns);
  const int n = j1 > j0 ? j1 - j0 : 0;  // pages of this CTA

  float zm0 = -INFINITY, zl0 = 0.f, zm1 = -INFINITY, zl1 = 0.f;
  if (warp == kScanWarps) {
    // ---- producer: lane l owns slot l (l < S) and fills pages l, l + S, ...
    // Each lane tests its own slot without blocking, so a released slot is
    // refilled at once whatever the other lanes' slots are doing.
    const int32_t* bt = a.block_table + (size_t)b * a.max_pages;
    const uint32_t bb = (uint32_t)(HG * a.basis_bytes), cb = (uint32_t)(HG * a.coef_bytes);
    // the block-table entries of this lane's first kPre pages, read up front
    constexpr int kPre = 8;
    int pre[kPre];
#pragma unroll
    for (int u = 0; u < kPre; ++u) pre[u] = (lane < S && lane + u * S < n) ? bt[j0 + lane + u * S] : -1;
    // every summary is read once per step: first to leave L2, so that the
    // s_hat rows written here stay there for the top-k
    const uint64_t once = l2_policy_evict_first();
    int p = lane < S ? lane : n;  // next page of this lane
    int u = 0;                    // its round: p = lane + u S
    for (uint32_t spin = 0; __any_sync(0xffffffffu, p < n); ++spin) {
      if (spin == kMbarSpinLimit * 4u) {
        if (lane == 0) set_error(a.err, kDevErrTimeout);
        break;
      }
      const bool ready = p < n && (u == 0 || mbar_test(&empty_bar[lane], (uint32_t)((u - 1) & 1)));
      if (!__any_sync(0xffffffffu, ready)) {
        __nanosleep(64);
        continue;
      }
      if (ready) {
        int phys = -1;
#pragma unroll
        for (int v = 0; v < kPre; ++v)
          if (v == u) phys = pre[v];
        if (u >= kPre) phys = bt[j0 + p];
        const bool valid = phys >= 0 && phys < a.pages_total;
        slot_ok[lane] = valid ? 1 : 0;
        if (valid) {
          // page-heads (phys, h0 .. h0 + HG - 1) are consecutive in both arrays
          const size_t ph = (size_t)phys * a.num_kv_heads + h0;
          const uint32_t slot = ring + lane * slot_bytes;
          mbar_arrive_expect_tx(&full_bar[lane], bb + cb);
          bulk_load_hint(slot, reinterpret_cast<const uint8_t*>(a.basis_t) + ph * a.basis_bytes, bb, &full_bar[lane],
                         once);
          if (!Q4 && cb)  // the two-array bf16 layout: the coefficients separately
            bulk_load_hint(slot + bb, reinterpret_cast<const uint8_t*>(a.coeffs) + ph * a.coef_bytes, cb,
                           &full_bar[lane], once);
        } else {
          mbar_arrive(&full_bar[lane]);
        }
        p += S;
        ++u;
      }
    }
  } else {
    // ---- consumers: warp `warp` serves head hw of the block on the pages of
    // its group
    const int hw = warp % HG, grp = warp / HG;
    const int hkv = h0 + hw, bh = b * a.num_kv_heads + hkv;
    const int Hq = a.num_kv_heads * G;
    uint4 qa[4], qb[4];
    {
      // query A fragments with the permuted contraction index; GRP2: rows
      // 4-7 repeat heads 0-3, so the first contraction already leaves each
      // head's W in both row halves the second one needs
      const uint16_t* qrow = a.q + ((size_t)b * Hq + (size_t)hkv * G) * kHeadDim;
      const int qr = GRP2 ? (g & 3) : g;
#pragma unroll
      for (int s = 0; s < 4; ++s) {
        qa[s] = (qr < G && (!GRP2 || g < 8))
                    ? __ldg(reinterpret_cast<const uint4*>(qrow + qr * kHeadDim + 32 * s + 8 * c))
                    : make_uint4(0, 0, 0, 0);
        qb[s] = (G16 && g + 8 < G)
                    ? __ldg(reinterpret_cast<const uint4*>(qrow + (g + 8) * kHeadDim + 32 * s + 8 * c))
                    : make_uint4(0, 0, 0, 0);
      }
    }
    // this head's basis (or packed block) and coefficients in slot s
    auto head_basis = [&](int s) -> uint32_t { return ring + s * slot_bytes + hw * a.basis_bytes; };
    // (packed bf16 blocks: the coefficients follow the basis rows)
    auto head_coef = [&](int s) -> uint32_t {
      return a.packed ? head_basis(s) + (uint32_t)(r * kHeadDim * 2)
                      : ring + s * slot_bytes + HG * a.basis_bytes + hw * a.coef_bytes;
    };
    unsigned long long cyc_wait = 0, cyc_comp = 0;
    // quantised format: this warp's pending pages (centroid codes, centroid
    // scales and base-2 LSEs per head row), flushed kMuBatch at a time
    const uint32_t stage_end = ring + S * slot_bytes;
    const uint32_t st_mu = stage_end + (uint32_t)(warp * kMuBatch * 128);
    float* st_smu = reinterpret_cast<float*>(ring_raw + (stage_end - smem_u32(ring_raw)) + kStageMu) + warp * kMuBatch;
    float* st_pend = reinterpret_cast<float*>(ring_raw + (stage_end - smem_u32(ring_raw)) + kStageMu + kStageSmu) +
                     warp * kMuBatch * 16;
    int npend = 0, kdone = 0;
    uint32_t vmask = 0;
    auto flush = [&](int nb) {  // warp-uniform
      __syncwarp();
      float u[4];
      mu_batch(st_mu, nb, qa, qb, lane, u);
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const int nn = 2 * c + hh;
        if (nn < nb && ((vmask >> nn) & 1u)) {
          const float sm = st_smu[nn] * a.scale_log2;
          const int j = j0 + grp + ngrp * (kdone + nn);
          const float v0 = st_pend[nn * 16 + g] + u[hh] * sm;
          lse2_merge(zm0, zl0, v0, 1.f);
          float v1 = 0.f;
          if (G16) {
            v1 = st_pend[nn * 16 + g + 8] + u[2 + hh] * sm;
            lse2_merge(zm1, zl1, v1, 1.f);
          }
          float* dst = a.shat + ((size_t)bh * a.max_pages + j) * G;
          if (g < G && (!GRP2 || g < 4)) dst[g] = v0 * kLn2;
          if (G16 && g + 8 < G) dst[g + 8] = v1 * kLn2;
          if (a.page_lse) {
            float* pl = a.page_lse + ((size_t)b * Hq + (size_t)hkv * G) * a.max_pages + j;
            if (g < G && (!GRP2 || g < 4)) pl[(size_t)g * a.max_pages] = v0 * kLn2;
            if (G16 && g + 8 < G) pl[(size_t)(g + 8) * a.max_pages] = v1 * kLn2;
          }
        }
      }
      __syncwarp();  // the staging area is free again
      kdone += nb;
      npend = 0;
      vmask = 0;
    };
    // slot s = p mod S and phase parity (p / S) & 1 of page p, advanced
    // without dividing: S is a multiple of ngrp, so s wraps exactly when p
    // crosses a multiple of S
    int s = grp;
    uint32_t phase = 0;
    for (int p = grp; p < n; p += ngrp, s += ngrp) {
      if (s >= S) {
        s -= S;
        phase ^= 1u;
      }
      const unsigned long long t0 = trace_clock();
      const bool ok = mbar_wait(&full_bar[s], phase);
      const unsigned long long t1 = trace_clock();
      if (__any_sync(0xffffffffu, !ok)) {
        if (lane == 0) set_error(a.err, kDevErrTimeout);
        break;
      }
      const int valid = slot_ok[s];
      float e0 = 0.f, e1 = 0.f;
      if (valid) {
        if (Q4)
          compute_page_q4<G16, GRP2, P>(head_basis(s), qa, qb, r, a.scale_log2, lane, e0, e1);
        else
          compute_page<G16, R16, GRP2, P>(head_basis(s), head_coef(s), qa, qb, r, a.scale_log2, lane, e0, e1);
      }
      if (Q4 && valid) {
        // stage the centroid codes (one word per lane), its scale and the LSEs
        const uint32_t blk = head_basis(s);
        sts32(st_mu + 128 * npend + 4 * lane, lds32(blk + 64 * r + 4 * lane));
        if (lane == 0) st_smu[npend] = __uint_as_float(lds32(blk + 64 * r + kHeadDim + P * r + 8 * r));
        if (c == 0) {
          st_pend[npend * 16 + g] = e0;
          if (G16) st_pend[npend * 16 + g + 8] = e1;
        }
      }
      __syncwarp();  // every lane is done with the slot
      if (lane == 0) mbar_arrive(&empty_bar[s]);
      cyc_wait += t1 - t0;
      cyc_comp += trace_clock() - t1;
      if (Q4) {
        vmask |= (valid ? 1u : 0u) << npend;
        if (!valid && lane == 0 && hw == 0) set_error(a.err, LOCKS_DEVERR_BLOCK_TABLE);
        if (++npend == kMuBatch) flush(kMuBatch);
        continue;
      }
      if (!valid) {
        if (lane == 0 && hw == 0) set_error(a.err, LOCKS_DEVERR_BLOCK_TABLE);
        continue;
      }
      const int j = j0 + p;
      lse2_merge(zm0, zl0, e0, 1.f);
      if (G16) lse2_merge(zm1, zl1, e1, 1.f);
      if (c == 0) {
        float* dst = a.shat + ((size_t)bh * a.max_pages + j) * G;
        if (g < G && (!GRP2 || g < 4)) dst[g] = e0 * kLn2;
        if (G16 && g + 8 < G) dst[g + 8] = e1 * kLn2;
        if (a.page_lse) {
          float* pl = a.page_lse + ((size_t)b * Hq + (size_t)hkv * G) * a.max_pages + j;
          if (g < G && (!GRP2 || g < 4)) pl[(size_t)g * a.max_pages] = e0 * kLn2;
          if (G16 && g + 8 < G) pl[(size_t)(g + 8) * a.max_pages] = e1 * kLn2;
        }
      }
    }
    if (Q4) {
      if (npend > 0) flush(npend);
      // each lane of a head row merged different pages
#pragma unroll
      for (int o = 1; o <= 2; o <<= 1) {
        lse2_merge(zm0, zl0, __shfl_xor_sync(0xffffffffu, zm0, o), __shfl_xor_sync(0xffffffffu, zl0, o));
        if (G16) lse2_merge(zm1, zl1, __shfl_xor_sync(0xffffffffu, zm1, o), __shfl_xor_sync(0xffffffffu, zl1, o));
      }
    }
    if (lane == 0) {
      trace_add(a.err, kTrScanCycWait, cyc_wait);
      trace_add(a.err, kTrScanCycCompute, cyc_comp);
      trace_add(a.err, kTrScanPages, (unsigned long long)((n - grp + ngrp - 1) / ngrp));
    }
    if (c == 0 && (!GRP2 || g < 4)) {
      red[warp][g] = make_float2(zm0, zl0);
      if (G16) red[warp][g + 8] = make_float2(zm1, zl1);
    }
  }

  if (LOCKS_TRACE && lane == 0 && warp < kScanWarps) trace_mark(a.err, kTrScanLoopDone, false);
  pdl_launch_dependents();
  __syncthreads();
  if (threadIdx.x == 0) trace_max(a.err, kTrScanMaxDur, trace_ns() - t_enter);
  // per head of the block: the (max, sum) over its warps' pages
  for (int t = threadIdx.x; t < HG * G; t += kScanThreads) {
    const int hw = t / G, gg = t % G;
    float m = -INFINITY, l = 0.f;
    for (int w = hw; w < kScanWarps; w += HG) lse2_merge(m, l, red[w][gg].x, red[w][gg].y);
    a.part[((size_t)(b * a.num_kv_heads + h0 + hw) * a.n_chunks + chunk) * G + gg] = make_float2(m, l);
  }
  trace_mark(a.err, kTrScanExit, false);
}

template <bool G16, bool R16, bool GRP2, bool Q4, int P>
cudaError_t launch_one(const ScanArgs& a0, cudaStream_t s, bool pdl) {
  ScanArgs a = a0;
  const SlotLayout L = slot_layout(a.rank, P, a.heads_per_block, Q4, a.packed != 0);
  a.slots = L.slots;
  a.slot_bytes = L.slot_bytes;
  a.basis_bytes = L.basis_bytes;
  a.coef_bytes = L.coef_bytes;
  if (L.slots < kScanWarps / a.heads_per_block) return cudaErrorInvalidValue;  // the plan keeps slots large enough
  cudaError_t e = cudaFuncSetAttribute(scan_kernel<G16, R16, GRP2, Q4, P>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, L.smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.n_chunks, a.batch * (a.num_kv_heads / a.heads_per_block), 1);
  cfg.blockDim = dim3(kScanThreads, 1, 1);
  cfg.dynamicSmemBytes = L.smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, scan_kernel<G16, R16, GRP2, Q4, P>, a);
}

template <int P>
cudaError_t launch_page(const ScanArgs& a, cudaStream_t s, bool pdl) {
  const bool g16 = a.group > 8, r16 = a.rank > 8;
  if (a.q4) {  // rank <= 8 (checked by the caller)
    if (g16) return launch_one<true, false, false, true, P>(a, s, pdl);
    if (a.group <= 4) return launch_one<false, false, true, true, P>(a, s, pdl);
    return launch_one<false, false, false, true, P>(a, s, pdl);
  }
  if (g16)
    return r16 ? launch_one<true, true, false, false, P>(a, s, pdl) : launch_one<true, false, false, false, P>(a, s, pdl);
  if (r16) return launch_one<false, true, false, false, P>(a, s, pdl);
  if (a.group <= 4) return launch_one<false, false, true, false, P>(a, s, pdl);
  return launch_one<false, false, false, false, P>(a, s, pdl);
}

}  // namespace

cudaError_t launch_scan(const ScanArgs& a, cudaStream_t s, bool pdl) {
  return a.page_size == 16 ? launch_page<16>(a, s, pdl) : launch_page<kPage>(a, s, pdl);
}

}  // namespace locks
