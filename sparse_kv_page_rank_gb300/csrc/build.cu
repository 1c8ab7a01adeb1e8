// Summary builder: rank-r spectral summary of finalised pages.
//
// LOCKS explainer (gist.science), §2 "Kernmechanisme": when a page is
// finalised (prefill or page crossing) its keys get a small
// eigendecomposition; the top-r eigenvectors are the basis and every token of
// the page keeps its coefficients.  §2 "Implementatie": this happens off the
// critical path of decoding.
//
// For one page-head K (P x d = 64 x 128 or 16 x 128, bf16) the top-r left
// singular vectors are the top-r eigenvectors of the Gram matrix A = K K^T
// (P x P).  Only r <= 16 of P eigenpairs are needed, so one CTA per page-head
// runs
//   1. A = K K^T on tensor cores (m16n8k16, bf16 products exact in fp32;
//      plain fp32 FMAs for the 16 x 16 product of a 16-token page);
//   2. subspace iteration with l = min(r + 8, P) vectors (at P = 16 the
//      whole space, so Rayleigh-Ritz below is exact): X_0 from A times a fixed
//      +-1 pattern, then X <- orth(A X) for a fixed number of steps
//      (modified Gram-Schmidt; deterministic, no early exit);
//   3. Rayleigh-Ritz: T = X^T A X (l x l), eigenpairs of T by a parallel
//      cyclic Jacobi (round-robin pairing, all pairs of a round rotated at
//      once, fixed number of sweeps); U_r = X times the top-r eigenvectors;
//   4. V_r = orthonormalised K^T U_r (d x r), columns whose norm falls to
//      <= 1e-6 of the first one are zero (rank deficit), and C = K V_r,
//      which equals U_r Sigma_r for exact eigenvectors and is the best
//      coefficient matrix for the computed basis in any case.
// Output: basis_t [r][d] (rows = basis vectors, descending singular value)
// and coeffs [P][r], bf16 or fp32.
//
// Quantised format (explainer §2 "Kernmechanisme", Kwantisatie: centred keys, int4 basis,
// int8 coefficients and centroid): the same steps on the centred keys
// K~ = K - 1 mu^T (mu = mean key of the page).  The Gram matrix of K~ is A
// with its row and column means removed (A~_ij = A_ij - m_i - m_j + m, m_i
// the row means of A and m their mean), so the tensor-core product is kept;
// V = K~^T U_r = K^T U_r - mu (1^T U_r) and C = K~ V = K V - 1 (mu^T V).
// Each basis vector, coefficient column and the centroid then get one
// symmetric float32 scale s = max|x| / qmax (qmax 7 for int4, 127 for int8)
// and codes rint(x / s), packed as LOCKS_Q4_BLOCK_BYTES(r, P) bytes.
#include "common.cuh"
#include "kernels.h"

namespace locks {

namespace {

constexpr int kBT = 256;            // threads
constexpr int kBW = kBT / 32;       // warps
constexpr int kKS = 136;            // bf16 row stride of K in shared memory (conflict-free ldmatrix)
template <int P>
constexpr int kAS = P + 1;          // fp32 row stride of A
constexpr int kLmax = 24;           // subspace size limit (r <= 16 -> l <= 24)
constexpr int kXS = kLmax + 1;
constexpr int kVS = kHeadDim + 1;
constexpr int kPowerIters = 8;
constexpr int kJacobiSweeps = 10;

template <int P>
struct BuildSmem {
  uint16_t K[P * kKS];
  float A[P * kAS<P>];
  float X[P * kXS];
  float Y[P * kXS];
  float T[kLmax * kXS];
  float Z[kLmax * kXS];
  float V[16 * kVS];        // basis rows
  float rot[kLmax / 2][2];  // (c, s) per pair of the current round
  int pp[kLmax / 2][2];     // pair members of the current round
  int order[kLmax];
  float red[kBW];
  // quantised format only
  float mu[kHeadDim];  // mean key
  float rm[P];     // row means of A
  float cs[16];        // column sums of U_r, then mu . V_j
  float sv[16], sc[16], smu;
  float grand;
};

// Y = A X  (P x l); A symmetric P x P
template <int P>
__device__ void mul_A(const BuildSmem<P>& s, const float* X, float* Y, int l) {
  for (int e = threadIdx.x; e < P * l; e += kBT) {
    const int i = e / l, j = e % l;
    float acc = 0.f;
#pragma unroll 8
    for (int k = 0; k < P; ++k) acc = fmaf(s.A[i * kAS<P> + k], X[k * kXS + j], acc);
    Y[i * kXS + j] = acc;
  }
}

// Modified Gram-Schmidt on the l columns of X (64 rows) in place; columns
// whose norm vanishes become zero.
__device__ void mgs_cols(float* X, int l, int rows, int stride) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int j = 0; j < l; ++j) {
    // every warp computes the norm of column j redundantly
    float ss = 0.f;
    for (int i = lane; i < rows; i += 32) ss += X[i * stride + j] * X[i * stride + j];
    ss = warp_sum(ss);
    const float inv = ss > 1e-30f ? rsqrtf(ss) : 0.f;
    // warps orthogonalise the later columns against the normalised column j
    for (int jj = j + 1 + warp; jj < l; jj += kBW) {
      float dp = 0.f;
      for (int i = lane; i < rows; i += 32) dp += X[i * stride + j] * X[i * stride + jj];
      dp = warp_sum(dp) * inv * inv;
      for (int i = lane; i < rows; i += 32) X[i * stride + jj] -= dp * X[i * stride + j];
    }
    __syncthreads();
    for (int i = threadIdx.x; i < rows; i += kBT) X[i * stride + j] *= inv;
    __syncthreads();
  }
}

template <int P>
__global__ void __launch_bounds__(kBT) build_kernel(const BuildArgs a) {
  extern __shared__ __align__(16) uint8_t dyn[];
  BuildSmem<P>& s = *reinterpret_cast<BuildSmem<P>*>(dyn);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, c = lane & 3;
  const int item = blockIdx.x;
  const int page_i = item / a.num_kv_heads, hkv = item % a.num_kv_heads;
  const int r = a.rank;
  const int l = min(min(r + 8, kLmax), P);  // even: r and P are

  const int phys = a.page_ids[page_i];
  if (phys < 0 || phys >= a.pages_total) {
    if (tid == 0) set_error(a.err, LOCKS_DEVERR_PAGE_ID);
    return;
  }
  const size_t ph = (size_t)phys * a.num_kv_heads + hkv;
  const uint16_t* kg = a.k_pool + ph * P * kHeadDim;

  // 0. K -> shared memory (bf16, padded rows)
  for (int e = tid; e < P * kHeadDim / 8; e += kBT) {
    const int row = e / 16, col = (e % 16) * 8;
    *reinterpret_cast<uint4*>(&s.K[row * kKS + col]) = __ldg(reinterpret_cast<const uint4*>(kg + row * kHeadDim + col));
  }
  const bool q4 = a.format == LOCKS_DTYPE_Q4;
  if (q4) {
    __syncthreads();  // K is in shared memory
    for (int dd = tid; dd < kHeadDim; dd += kBT) {
      float acc = 0.f;
      for (int i = 0; i < P; ++i) acc += __bfloat162float(__ushort_as_bfloat16(s.K[i * kKS + dd]));
      s.mu[dd] = acc * (1.f / P);
    }
  }
  __syncthreads();

  // 1. A = K K^T : warp w -> rows 16*(w/2).., columns 32*(w%2)..
  // (16-token pages: a 16 x 16 product, one entry per thread in fp32 FMAs;
  // the bf16 products are exact in fp32 either way)
  if constexpr (P != 64) {
    for (int e = tid; e < P * P; e += kBT) {
      const int i = e / P, j = e % P;
      float acc = 0.f;
      for (int k = 0; k < kHeadDim; ++k)
        acc = fmaf(__bfloat162float(__ushort_as_bfloat16(s.K[i * kKS + k])),
                   __bfloat162float(__ushort_as_bfloat16(s.K[j * kKS + k])), acc);
      s.A[i * kAS<P> + j] = acc;
    }
  } else {
    const int mt = warp >> 1, nb = (warp & 1) * 4;
    float acc[4][4] = {};
    const uint32_t kbase = smem_u32(s.K);
    const int mi = lane >> 3;
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
      uint32_t a0, a1, a2, a3;
      {
        const int row = 16 * mt + (mi & 1) * 8 + (lane & 7);
        const int col = 16 * kk + (mi >> 1) * 8;
        ldmatrix_x4(a0, a1, a2, a3, kbase + (row * kKS + col) * 2);
      }
#pragma unroll
      for (int np = 0; np < 2; ++np) {
        uint32_t b0, b1, b2, b3;
        const int row = 8 * (nb + 2 * np) + (mi >> 1) * 8 + (lane & 7);
        const int col = 16 * kk + (mi & 1) * 8;
        ldmatrix_x4(b0, b1, b2, b3, kbase + (row * kKS + col) * 2);
        mma_16816(acc[2 * np], a0, a1, a2, a3, b0, b1);
        mma_16816(acc[2 * np + 1], a0, a1, a2, a3, b2, b3);
      }
    }
#pragma unroll
    for (int nt = 0; nt < 4; ++nt) {
      const int col = 8 * (nb + nt) + 2 * c;
      const int row = 16 * mt + g;
      s.A[row * kAS<P> + col] = acc[nt][0];
      s.A[row * kAS<P> + col + 1] = acc[nt][1];
      s.A[(row + 8) * kAS<P> + col] = acc[nt][2];
      s.A[(row + 8) * kAS<P> + col + 1] = acc[nt][3];
    }
  }
  __syncthreads();
  if (q4) {
    // Gram matrix of the centred keys: remove the row and column means
    for (int i = tid; i < P; i += kBT) {
      float acc = 0.f;
      for (int j = 0; j < P; ++j) acc += s.A[i * kAS<P> + j];
      s.rm[i] = acc * (1.f / P);
    }
    __syncthreads();
    if (tid == 0) {
      float acc = 0.f;
      for (int i = 0; i < P; ++i) acc += s.rm[i];
      s.grand = acc * (1.f / P);
    }
    __syncthreads();
    for (int e = tid; e < P * P; e += kBT) {
      const int i = e / P, j = e % P;
      s.A[i * kAS<P> + j] = s.A[i * kAS<P> + j] - s.rm[i] - s.rm[j] + s.grand;
    }
    __syncthreads();
  }

  // 2. subspace iteration.  Start: A * (fixed +-1 pattern).
  for (int e = tid; e < P * l; e += kBT) {
    const int i = e / l, j = e % l;
    uint32_t h = (uint32_t)(i * 131 + j * 71 + 17);
    h ^= h >> 7;
    h *= 0x9E3779B1u;
    h ^= h >> 15;
    s.Y[i * kXS + j] = (h & 1u) ? 1.f : -1.f;
  }
  __syncthreads();
  mul_A(s, s.Y, s.X, l);
  __syncthreads();
  for (int itn = 0; itn < kPowerIters; ++itn) {
    mgs_cols(s.X, l, P, kXS);
    mul_A(s, s.X, s.Y, l);
    __syncthreads();
    for (int e = tid; e < P * l; e += kBT) s.X[(e / l) * kXS + e % l] = s.Y[(e / l) * kXS + e % l];
    __syncthreads();
  }
  mgs_cols(s.X, l, P, kXS);
  mgs_cols(s.X, l, P, kXS);  // twice: orthonormal to working precision
  mul_A(s, s.X, s.Y, l);
  __syncthreads();

  // 3. T = X^T A X (symmetrised), Z = I
  for (int e = tid; e < l * l; e += kBT) {
    const int i = e / l, j = e % l;
    float t1 = 0.f, t2 = 0.f;
    for (int k = 0; k < P; ++k) {
      t1 = fmaf(s.X[k * kXS + i], s.Y[k * kXS + j], t1);
      t2 = fmaf(s.X[k * kXS + j], s.Y[k * kXS + i], t2);
    }
    s.T[i * kXS + j] = 0.5f * (t1 + t2);
    s.Z[i * kXS + j] = (i == j) ? 1.f : 0.f;
  }
  __syncthreads();

  // parallel cyclic Jacobi on T (l even): round-robin pairing
  const int npair = l / 2;
  for (int sweep = 0; sweep < kJacobiSweeps; ++sweep) {
    for (int rd = 0; rd < l - 1; ++rd) {
      if (tid < npair) {
        int p, q;
        if (tid == 0) {
          p = l - 1;
          q = rd;
        } else {
          p = (rd + tid) % (l - 1);
          q = (rd - tid + (l - 1)) % (l - 1);
        }
        if (p > q) { int t = p; p = q; q = t; }
        const float apq = s.T[p * kXS + q], app = s.T[p * kXS + p], aqq = s.T[q * kXS + q];
        float cs = 1.f, sn = 0.f;
        if (fabsf(apq) > 1e-30f && fabsf(apq) > 1e-9f * (fabsf(app) + fabsf(aqq)) * 1e-3f) {
          const float theta = (aqq - app) / (2.f * apq);
          float t;
          if (fabsf(theta) > 1e15f)
            t = 0.5f / theta;
          else
            t = copysignf(1.f, theta) / (fabsf(theta) + sqrtf(theta * theta + 1.f));
          cs = rsqrtf(t * t + 1.f);
          sn = t * cs;
        }
        s.pp[tid][0] = p;
        s.pp[tid][1] = q;
        s.rot[tid][0] = cs;
        s.rot[tid][1] = sn;
      }
      __syncthreads();
      // T <- J^T T J, block by block (blocks are disjoint)
      for (int e = tid; e < npair * npair; e += kBT) {
        const int bi = e / npair, bj = e % npair;
        const int p = s.pp[bi][0], q = s.pp[bi][1], p2 = s.pp[bj][0], q2 = s.pp[bj][1];
        const float c1 = s.rot[bi][0], s1 = s.rot[bi][1], c2 = s.rot[bj][0], s2 = s.rot[bj][1];
        const float tpp = s.T[p * kXS + p2], tpq = s.T[p * kXS + q2];
        const float tqp = s.T[q * kXS + p2], tqq = s.T[q * kXS + q2];
        // rows: L = J1^T B
        const float lpp = c1 * tpp - s1 * tqp, lpq = c1 * tpq - s1 * tqq;
        const float lqp = s1 * tpp + c1 * tqp, lqq = s1 * tpq + c1 * tqq;
        // columns: L J2
        float npp = c2 * lpp - s2 * lpq, npq = s2 * lpp + c2 * lpq;
        float nqp = c2 * lqp - s2 * lqq, nqq = s2 * lqp + c2 * lqq;
        if (bi == bj) { npq = 0.f; nqp = 0.f; }
        s.T[p * kXS + p2] = npp;
        s.T[p * kXS + q2] = npq;
        s.T[q * kXS + p2] = nqp;
        s.T[q * kXS + q2] = nqq;
      }
      // Z <- Z J
      for (int e = tid; e < l * npair; e += kBT) {
        const int k = e / npair, pi = e % npair;
        const int p = s.pp[pi][0], q = s.pp[pi][1];
        const float cs = s.rot[pi][0], sn = s.rot[pi][1];
        const float zp = s.Z[k * kXS + p], zq = s.Z[k * kXS + q];
        s.Z[k * kXS + p] = cs * zp - sn * zq;
        s.Z[k * kXS + q] = sn * zp + cs * zq;
      }
      __syncthreads();
    }
  }

  // eigenvalues descending -> order
  if (tid == 0) {
    for (int i = 0; i < l; ++i) s.order[i] = i;
    for (int i = 0; i < l; ++i) {
      int best = i;
      for (int j = i + 1; j < l; ++j)
        if (s.T[s.order[j] * kXS + s.order[j]] > s.T[s.order[best] * kXS + s.order[best]]) best = j;
      const int t = s.order[i];
      s.order[i] = s.order[best];
      s.order[best] = t;
    }
  }
  __syncthreads();

  // U_r = X Z[:, order[0..r)]  -> stored in Y (64 x r)
  for (int e = tid; e < P * r; e += kBT) {
    const int i = e / r, j = e % r;
    const int col = s.order[j];
    float acc = 0.f;
    for (int k = 0; k < l; ++k) acc = fmaf(s.X[i * kXS + k], s.Z[k * kXS + col], acc);
    s.Y[i * kXS + j] = acc;
  }
  __syncthreads();

  // 4. V = K^T U_r  (d x r) into s.V as rows [j][d] (centred: minus mu 1^T U_r)
  if (q4) {
    for (int j = warp; j < r; j += kBW) {
      float acc = 0.f;
      for (int i = lane; i < P; i += 32) acc += s.Y[i * kXS + j];
      acc = warp_sum(acc);
      if (lane == 0) s.cs[j] = acc;
    }
    __syncthreads();
  }
  for (int e = tid; e < kHeadDim * r; e += kBT) {
    const int dd = e % kHeadDim, j = e / kHeadDim;
    float acc = 0.f;
    for (int i = 0; i < P; ++i)
      acc = fmaf(__bfloat162float(__ushort_as_bfloat16(s.K[i * kKS + dd])), s.Y[i * kXS + j], acc);
    if (q4) acc -= s.mu[dd] * s.cs[j];
    s.V[j * kVS + dd] = acc;
  }
  __syncthreads();
  // orthonormalise the r rows of V (length d), twice; zero rows that vanish
  for (int pass = 0; pass < 2; ++pass) {
    for (int j = 0; j < r; ++j) {
      float ss = 0.f;
      for (int i = lane; i < kHeadDim; i += 32) ss += s.V[j * kVS + i] * s.V[j * kVS + i];
      ss = warp_sum(ss);
      if (pass == 0 && j == 0 && tid == 0) s.red[0] = sqrtf(ss);  // ~ sigma_1
      float inv = ss > 1e-30f ? rsqrtf(ss) : 0.f;
      for (int jj = j + 1 + warp; jj < r; jj += kBW) {
        float dp = 0.f;
        for (int i = lane; i < kHeadDim; i += 32) dp += s.V[j * kVS + i] * s.V[jj * kVS + i];
        dp = warp_sum(dp) * inv * inv;
        for (int i = lane; i < kHeadDim; i += 32) s.V[jj * kVS + i] -= dp * s.V[j * kVS + i];
      }
      __syncthreads();
      if (pass == 0) {
        // rank deficit: the orthogonalised norm of column j is ~ sigma_j
        if (!(sqrtf(ss) > 1e-6f * s.red[0])) inv = 0.f;
      }
      for (int i = tid; i < kHeadDim; i += kBT) s.V[j * kVS + i] *= inv;
      __syncthreads();
    }
  }

  // C = K V  (64 x r) -> Y  (centred: minus mu . V_j)
  if (q4) {
    for (int j = warp; j < r; j += kBW) {
      float acc = 0.f;
      for (int k = lane; k < kHeadDim; k += 32) acc = fmaf(s.mu[k], s.V[j * kVS + k], acc);
      acc = warp_sum(acc);
      if (lane == 0) s.cs[j] = acc;
    }
    __syncthreads();
  }
  for (int e = tid; e < P * r; e += kBT) {
    const int i = e / r, j = e % r;
    float acc = 0.f;
    for (int k = 0; k < kHeadDim; ++k)
      acc = fmaf(__bfloat162float(__ushort_as_bfloat16(s.K[i * kKS + k])), s.V[j * kVS + k], acc);
    if (q4) acc -= s.cs[j];
    s.Y[i * kXS + j] = acc;
  }
  __syncthreads();

  // store
  if (q4) {
    // one symmetric scale per basis vector (int4), per coefficient column
    // and for the centroid (int8)
    for (int j = warp; j <= r; j += kBW) {
      float av = 0.f, ac = 0.f;
      if (j < r) {
        for (int k = lane; k < kHeadDim; k += 32) av = fmaxf(av, fabsf(s.V[j * kVS + k]));
        for (int i = lane; i < P; i += 32) ac = fmaxf(ac, fabsf(s.Y[i * kXS + j]));
      } else {
        for (int k = lane; k < kHeadDim; k += 32) ac = fmaxf(ac, fabsf(s.mu[k]));
      }
      av = warp_max(av);
      ac = warp_max(ac);
      if (lane == 0) {
        if (j < r) {
          s.sv[j] = av / 7.f;
          s.sc[j] = ac / 127.f;
        } else {
          s.smu = ac / 127.f;
        }
      }
    }
    __syncthreads();
    auto code = [](float x, float sc, float qmax) -> int {
      return sc > 0.f ? (int)fminf(fmaxf(rintf(x / sc), -qmax), qmax) : 0;
    };
    uint8_t* blk = static_cast<uint8_t*>(a.basis_t) + ph * (size_t)LOCKS_Q4_BLOCK_BYTES(r, P);
    // basis: word m of row j holds elements 8m .. 8m+7, element 8m+i at
    // bits 4(i/2) + 16(i%2), as code + 8; it is stored at word 4(m%4) + m/4
    // of the row, so the four words one scan lane reads are adjacent
    uint32_t* bw = reinterpret_cast<uint32_t*>(blk);
    for (int e = tid; e < r * (kHeadDim / 8); e += kBT) {
      const int j = e / (kHeadDim / 8), m = e % (kHeadDim / 8);
      uint32_t w = 0u;
#pragma unroll
      for (int i = 0; i < 8; ++i)
        w |= (uint32_t)(code(s.V[j * kVS + 8 * m + i], s.sv[j], 7.f) + 8) << (4 * (i / 2) + 16 * (i % 2));
      bw[j * (kHeadDim / 8) + 4 * (m % 4) + m / 4] = w;
    }
    for (int k = tid; k < kHeadDim; k += kBT) blk[64 * r + k] = (uint8_t)(code(s.mu[k], s.smu, 127.f) + 128);
    // coefficients: token i, column j at (((i%8) r/2 + j/2) P/8 + i/8) 2 + j%2
    // (the codes of tokens i%8 + 8t, columns 2c and 2c+1, side by side)
    for (int e = tid; e < P * r; e += kBT) {
      const int i = e / r, j = e % r;
      const int at = (((i % 8) * (r / 2) + j / 2) * (P / 8) + i / 8) * 2 + j % 2;
      blk[64 * r + kHeadDim + at] = (uint8_t)(code(s.Y[i * kXS + j], s.sc[j], 127.f) + 128);
    }
    // scales: per column pair t, s_v[2t], s_v[2t+1], s_c[2t], s_c[2t+1]; then s_mu
    float* sco = reinterpret_cast<float*>(blk + 64 * r + kHeadDim + P * r);
    for (int e = tid; e < 2 * r + 1; e += kBT) {
      const int t = e / 4, u = e % 4;
      sco[e] = e == 2 * r ? s.smu : (u < 2 ? s.sv[2 * t + u] : s.sc[2 * t + u - 2]);
    }
  } else if (a.format == LOCKS_DTYPE_F32) {
    float* bo = reinterpret_cast<float*>(a.basis_t) + ph * (size_t)r * kHeadDim;
    float* co = reinterpret_cast<float*>(a.coeffs) + ph * (size_t)P * r;
    for (int e = tid; e < r * kHeadDim; e += kBT) bo[e] = s.V[(e / kHeadDim) * kVS + e % kHeadDim];
    for (int e = tid; e < P * r; e += kBT) co[e] = s.Y[(e / r) * kXS + e % r];
  } else {
    // bf16: two arrays, or one block per page-head (basis rows, then coefficients)
    const bool packed = a.format == LOCKS_DTYPE_BF16_PACKED;
    uint16_t* bo = reinterpret_cast<uint16_t*>(a.basis_t) + ph * (size_t)r * (packed ? kHeadDim + P : kHeadDim);
    uint16_t* co = packed ? bo + r * kHeadDim : reinterpret_cast<uint16_t*>(a.coeffs) + ph * (size_t)P * r;
    for (int e = tid; e < r * kHeadDim; e += kBT)
      bo[e] = __bfloat16_as_ushort(__float2bfloat16_rn(s.V[(e / kHeadDim) * kVS + e % kHeadDim]));
    for (int e = tid; e < P * r; e += kBT)
      co[e] = __bfloat16_as_ushort(__float2bfloat16_rn(s.Y[(e / r) * kXS + e % r]));
  }
}

}  // namespace

namespace {

template <int P>
cudaError_t launch_page(const BuildArgs& a, cudaStream_t st) {
  const size_t smem = sizeof(BuildSmem<P>);
  cudaError_t e = cudaFuncSetAttribute(build_kernel<P>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  build_kernel<P><<<dim3(a.n * a.num_kv_heads), dim3(kBT), smem, st>>>(a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_build(const BuildArgs& a, cudaStream_t st) {
  if (a.n <= 0) return cudaSuccess;
  return a.page_size == 16 ? launch_page<16>(a, st) : launch_page<kPage>(a, st);
}

}  // namespace locks
