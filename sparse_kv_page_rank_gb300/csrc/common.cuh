// Device helpers shared by the LOCKS kernels (sm_103a): inline PTX wrappers for
// warp-level bf16 tensor-core MMA, ldmatrix, mbarrier waits with an iteration
// limit, 2-D TMA tile loads and programmatic dependent launch.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/locks.h"

namespace locks {

constexpr int kHeadDim = 128;
constexpr int kPage = 64;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
// An mbarrier wait gives up after this many polls (each poll blocks in
// hardware for a bounded time slice); the kernel then records
// LOCKS_DEVERR_TIMEOUT-style failure in the error word and returns.
constexpr uint32_t kMbarSpinLimit = 1u << 22;
constexpr int kDevErrTimeout = 0x10;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// D(16x8, f32) += A(16x16, bf16, row) * B(16x8, bf16, col)
__device__ __forceinline__ void mma_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                          uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// D(16x8, f32) += A(16x8, bf16, row) * B(8x8, bf16, col)
__device__ __forceinline__ void mma_1688(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t b0) {
  asm volatile(
      "mma.sync.aligned.m16n8k8.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5}, {%6}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(b0));
}

// The same two shapes with fp16 operands.
__device__ __forceinline__ void mma_16816_f16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                              uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void mma_1688_f16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t b0) {
  asm volatile(
      "mma.sync.aligned.m16n8k8.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5}, {%6}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(b0));
}

__device__ __forceinline__ void ldmatrix_x4(uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3,
                                            uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ void ldmatrix_x4_trans(uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                                  uint32_t& r3, uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

// Two floats -> packed bf16x2 (round to nearest even); `lo` goes to the low half.
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ float bf16_round(float x) {
  return __bfloat162float(__float2bfloat16_rn(x));
}

// Hardware base-2 exponential and logarithm (PTX ex2.approx / lg2.approx).
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float fast_log2(float x) {
  float y;
  asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Monotone map float -> uint32 (larger float, larger key); -0 maps like +0.
__device__ __forceinline__ uint32_t orderable_key(float f) {
  if (f == 0.0f) f = 0.0f;
  uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ void set_error(int* err, int bit) {
  if (err) atomicOr(err, bit);
}

// ---- programmatic dependent launch ------------------------------------------
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;\n" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
}

// ---- mbarrier ----------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(smem_u32(bar)), "r"(count));
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
}
__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(smem_u32(bar)) : "memory");
}
// Non-blocking test: has phase `parity` completed?
__device__ __forceinline__ bool mbar_test(uint64_t* bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(done)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return done != 0;
}
// Wait for phase `parity` to complete; false after kMbarSpinLimit polls.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, uint32_t* polls = nullptr) {
  uint32_t addr = smem_u32(bar);
  for (uint32_t it = 0; it < kMbarSpinLimit; ++it) {
    if (polls) ++*polls;
    uint32_t done;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, "
        "p;\n}\n"
        : "=r"(done)
        : "r"(addr), "r"(parity)
        : "memory");
    if (done) return true;
  }
  return false;
}

// ---- TMA ------------------------------------------------------------------------
__device__ __forceinline__ void tma_load_2d(void* smem_dst, const CUtensorMap* map, uint64_t* bar,
                                            int x, int y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, "
      "{%2, %3}], [%4];\n" ::"r"(smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}

// 1-D bulk copy global -> shared (both 16-byte aligned, size a multiple of 16).
__device__ __forceinline__ void bulk_load(uint32_t smem_dst, const void* gsrc, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n" ::"r"(smem_dst),
      "l"(gsrc), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}
// An L2 cache policy that marks lines as the first to evict (for data read
// once, so that it does not push out data that is read again soon).
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;\n" : "=l"(pol));
  return pol;
}
// bulk_load with an L2 cache policy.
__device__ __forceinline__ void bulk_load_hint(uint32_t smem_dst, const void* gsrc, uint32_t bytes, uint64_t* bar,
                                               uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;\n" ::"r"(
          smem_dst),
      "l"(gsrc), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}
__device__ __forceinline__ void tma_load_2d_u32(uint32_t smem_dst, const CUtensorMap* map, uint64_t* bar, int x,
                                                int y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, "
      "{%2, %3}], [%4];\n" ::"r"(smem_dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}
__device__ __forceinline__ uint32_t lds32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.u32 %0, [%1];\n" : "=r"(v) : "r"(addr));
  return v;
}

// Bulk prefetch of [gsrc, gsrc + bytes) into L2 (16-byte aligned, size a multiple of 16).
__device__ __forceinline__ void prefetch_l2_bulk(const void* gsrc, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;\n" ::"l"(gsrc), "r"(bytes) : "memory");
}

__device__ __forceinline__ void prefetch_tmap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];\n" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// ---- per-thread asynchronous global -> shared copies (LDGSTS) -------------------
__device__ __forceinline__ void cp_async_16(uint32_t smem_addr, const void* gmem) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(smem_addr), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async_4(uint32_t smem_addr, const void* gmem) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;\n" ::"r"(smem_addr), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}
__device__ __forceinline__ uint32_t lds16(uint32_t addr) {
  unsigned short v;
  asm volatile("ld.shared.u16 %0, [%1];\n" : "=h"(v) : "r"(addr));
  return v;
}
__device__ __forceinline__ void sts32(uint32_t addr, uint32_t v) {
  asm volatile("st.shared.u32 [%0], %1;\n" ::"r"(addr), "r"(v) : "memory");
}
__device__ __forceinline__ uint2 lds64(uint32_t addr) {
  uint2 v;
  asm volatile("ld.shared.v2.u32 {%0,%1}, [%2];\n" : "=r"(v.x), "=r"(v.y) : "r"(addr));
  return v;
}
// Integer codes to bf16 without int-to-float conversions: a biased code u
// placed in the low mantissa bits of a fixed exponent is the number
// (2^e + u) exactly, and subtracting (2^e + bias) leaves the code.
// Two 4-bit codes stored as code + 8 in bits sh..sh+3 and sh+16..sh+19 of w:
// bf16 (128 + u) in each half, minus 136 (all exact in bf16).
__device__ __forceinline__ uint32_t u4pair_bf16(uint32_t w, int sh) {
  uint32_t x = ((w >> sh) & 0x000f000fu) | 0x43004300u;
  asm("sub.rn.bf16x2 %0, %0, %1;\n" : "+r"(x) : "r"(0x43084308u));
  return x;
}
// Two 8-bit codes stored as code + 128 in bytes k and k+1 of w: the float
// (2^23 + u) minus (2^23 + 128), then the two floats' upper halves (the
// codes are small integers, exact in bf16).
__device__ __forceinline__ uint32_t u8pair_bf16(uint32_t w, int k) {
  const float lo = __uint_as_float(__byte_perm(w, 0x4b000000u, 0x7650u + k)) - 8388736.f;
  const float hi = __uint_as_float(__byte_perm(w, 0x4b000000u, 0x7651u + k)) - 8388736.f;
  return __byte_perm(__float_as_uint(lo), __float_as_uint(hi), 0x7632u);
}

// Four 8-bit codes stored as code + 128 in the bytes of w -> two fp16 pairs
// (bytes 0, 1 -> lo; bytes 2, 3 -> hi): a byte under the fp16 exponent of
// 1024 is the exact number 1024 + byte, from which 1152 = 1024 + 128 is
// subtracted.
__device__ __forceinline__ void u8quad_f16(uint32_t w, uint32_t& lo, uint32_t& hi) {
  lo = __byte_perm(w, 0x64646464u, 0x4140u);
  hi = __byte_perm(w, 0x64646464u, 0x4342u);
  asm("sub.rn.f16x2 %0, %0, %2;\n sub.rn.f16x2 %1, %1, %2;\n" : "+r"(lo), "+r"(hi) : "r"(0x64806480u));
}
// (x0, x1) -> hi + lo as fp16 pairs (x0 in the low halves): hi rounds x to
// fp16, saturating at +-65504, and lo rounds the remainder (about 22 bits
// of x together).
__device__ __forceinline__ void split2_f16(float x0, float x1, uint32_t& hi, uint32_t& lo) {
  asm("cvt.rn.satfinite.f16x2.f32 %0, %1, %2;\n" : "=r"(hi) : "f"(x1), "f"(x0));
  float h0, h1;
  asm("{\n .reg .f16 a, b;\n mov.b32 {a, b}, %2;\n cvt.f32.f16 %0, a;\n cvt.f32.f16 %1, b;\n}\n"
      : "=f"(h0), "=f"(h1) : "r"(hi));
  asm("cvt.rn.satfinite.f16x2.f32 %0, %1, %2;\n" : "=r"(lo) : "f"(x1 - h1), "f"(x0 - h0));
}

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];\n" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
  return v;
}

// ---- thread-block clusters / distributed shared memory ------------------------------
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;\n" : "=r"(r));
  return r;
}
// Hardware barrier over every CTA of the cluster (all CTAs of a cluster are
// co-scheduled, so it always completes); release/acquire orders shared and
// global memory accesses around it.
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\nbarrier.cluster.wait.acquire.aligned;\n" ::: "memory");
}
// Address of the same shared-memory location in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t dsmem_addr(uint32_t local, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;\n" : "=r"(r) : "r"(local), "r"(rank));
  return r;
}
__device__ __forceinline__ float ld_dsmem(uint32_t addr) {
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];\n" : "=f"(v) : "r"(addr) : "memory");
  return v;
}
__device__ __forceinline__ void st_dsmem(uint32_t addr, int v) {
  asm volatile("st.shared::cluster.u32 [%0], %1;\n" ::"r"(addr), "r"(v) : "memory");
}
__device__ __forceinline__ void st_dsmem_f4(uint32_t addr, float4 v) {
  asm volatile("st.shared::cluster.v4.f32 [%0], {%1, %2, %3, %4};\n" ::"r"(addr), "f"(v.x), "f"(v.y), "f"(v.z),
               "f"(v.w)
               : "memory");
}
__device__ __forceinline__ void st_dsmem_u4(uint32_t addr, uint4 v) {
  asm volatile("st.shared::cluster.v4.u32 [%0], {%1, %2, %3, %4};\n" ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z),
               "r"(v.w)
               : "memory");
}
__device__ __forceinline__ void st_dsmem_f2(uint32_t addr, float2 v) {
  asm volatile("st.shared::cluster.v2.f32 [%0], {%1, %2};\n" ::"r"(addr), "f"(v.x), "f"(v.y) : "memory");
}
// The two halves of cluster_sync, for a barrier whose wait comes much later.
__device__ __forceinline__ void cluster_arrive() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
  asm volatile("barrier.cluster.wait.acquire.aligned;\n" ::: "memory");
}
// Arrive on an mbarrier in another CTA of the cluster (address from
// dsmem_addr); release at cluster scope orders this thread's earlier
// shared-memory stores (and, through a preceding CTA barrier, those of the
// whole CTA) before the arrival.
__device__ __forceinline__ void mbar_arrive_remote(uint32_t bar_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];\n" ::"r"(bar_addr) : "memory");
}
// mbar_wait with acquire at cluster scope (for arrivals from other CTAs).
__device__ __forceinline__ bool mbar_wait_cluster(uint64_t* bar, uint32_t parity) {
  const uint32_t addr = smem_u32(bar);
  for (uint32_t it = 0; it < kMbarSpinLimit; ++it) {
    uint32_t done;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n selp.u32 "
        "%0, 1, 0, p;\n}\n"
        : "=r"(done)
        : "r"(addr), "r"(parity)
        : "memory");
    if (done) return true;
  }
  return false;
}

// ---- optional kernel timeline (build with -DLOCKS_TRACE=1) -------------------------
// Each kernel records %globaltimer (ns) at its first CTA entry, first return
// from the grid-dependency wait, phase ends and last CTA exit, plus summed
// per-warp cycle counts, into 64-bit slots that live in otherwise unused
// bytes of the workspace's first 256-byte block (offset 8, 31 slots).  Start
// slots must be preset to ~0 and the others to 0 by the reader.  Compiled out
// by default.
#ifndef LOCKS_TRACE
#define LOCKS_TRACE 0
#endif
enum TraceSlot {
  kTrScanEnter = 0, kTrScanWait, kTrScanExit,
  kTrTopkEnter, kTrTopkWait, kTrTopkExit,
  kTrAttEnter, kTrAttWait, kTrAttExit,
  kTrScanCycWait, kTrScanCycCompute, kTrScanCycIssue, kTrScanPages,
  kTrTopkLoaded, kTrTopkKeys, kTrTopkSelected,
  kTrAttResolved, kTrAttFirstData, kTrAttLooped, kTrAttCtaMerged, kTrAttClusterMerged,
  kTrScanPolls, kTrSelMinMax, kTrSelRadix, kTrSelCompact, kTrSelPasses, kTrSelCalls,
  kTrScanLastEnter, kTrScanMaxDur, kTrScanLoopDone,
};
__device__ __forceinline__ unsigned long long trace_ns() {
#if LOCKS_TRACE
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
#else
  return 0ull;
#endif
}
__device__ __forceinline__ void trace_max(int* err_word, int slot, unsigned long long v) {
#if LOCKS_TRACE
  if (err_word) atomicMax(reinterpret_cast<unsigned long long*>(reinterpret_cast<char*>(err_word) + 8) + slot, v);
#else
  (void)err_word; (void)slot; (void)v;
#endif
}
__device__ __forceinline__ unsigned long long trace_clock() {
#if LOCKS_TRACE
  return clock64();
#else
  return 0ull;
#endif
}
__device__ __forceinline__ void trace_add(int* err_word, int slot, unsigned long long v) {
#if LOCKS_TRACE
  if (err_word) atomicAdd(reinterpret_cast<unsigned long long*>(reinterpret_cast<char*>(err_word) + 8) + slot, v);
#else
  (void)err_word; (void)slot; (void)v;
#endif
}
__device__ __forceinline__ void trace_mark(int* err_word, int slot, bool is_min) {
#if LOCKS_TRACE
  if (err_word && threadIdx.x == 0) {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    unsigned long long* tr = reinterpret_cast<unsigned long long*>(reinterpret_cast<char*>(err_word) + 8);
    if (is_min) atomicMin(tr + slot, t); else atomicMax(tr + slot, t);
  }
#else
  (void)err_word; (void)slot; (void)is_min;
#endif
}

// ---- warp / block reductions ---------------------------------------------------
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Combine two (max, sum) pairs of a base-2 log-sum-exp: value = m + log2(l).
__device__ __forceinline__ void lse2_merge(float& m, float& l, float m2, float l2) {
  float mn = fmaxf(m, m2);
  if (mn == -INFINITY) return;
  l = l * fast_exp2(m - mn) + l2 * fast_exp2(m2 - mn);
  m = mn;
}

}  // namespace locks
