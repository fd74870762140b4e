// pkv_device.cuh -- device-side helpers shared by the pkv kernels (sm_103a).
//
// Thin inline-PTX wrappers for the primitives the decode kernel is built on:
// mbarrier phases; TMA tensor loads (2-D tiles, 128-byte swizzle) and 1-D bulk
// copies, both global -> shared with completion counted in bytes on an
// mbarrier; ldmatrix and the m16n8k16 bf16 tensor-core product; bf16 packing.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "../../include/pkv.h"

namespace pkv {

constexpr int kHeadDim = PKV_HEAD_DIM;      // 64
constexpr int kPage = PKV_PAGE_SIZE;        // 16 tokens per page
constexpr int kRowBytes = kHeadDim * 2;     // one token's K (or V) row: 128 B
constexpr int kHalfBytes = kPage * kRowBytes;  // one head's K block of a page: 2 KiB
constexpr int kHeadPageBytes = 2 * kHalfBytes; // one head's K+V block of a page: 4 KiB
constexpr unsigned kFull = 0xffffffffu;

// Upper bound on polls of one mbarrier phase before a wait gives up and
// reports PKV_ERR_TIMEOUT (a 4 KiB copy lands in microseconds; this is
// hundreds of milliseconds or more).
constexpr uint32_t kWaitPolls = 1u << 22;

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

// Make mbarrier initialisation visible to the async proxy (bulk copies).
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// Order this thread's earlier generic-proxy shared-memory accesses before
// later async-proxy (bulk copy) accesses of the same memory.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

// The same, called by a whole warp, converged, with warp-uniform arguments:
// one elected lane arrives.
__device__ __forceinline__ void mbar_arrive_expect_tx_elect(uint32_t bar, uint32_t bytes) {
  asm volatile(
      "{\n\t.reg .pred e;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "@e mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n\t}" ::"r"(bar), "r"(bytes)
      : "memory");
}

// Raise the phase's expected transaction bytes without arriving.
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(bar), "r"(parity)
      : "memory");
  return done != 0;
}

// Bounded wait for the phase with the given parity to complete.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity) {
  for (uint32_t i = 0; i < kWaitPolls; ++i)
    if (mbar_try_wait(bar, parity)) return true;
  return false;
}

// 1-D bulk copy global -> shared::cta; completion is counted on `bar` in
// bytes. dst, src and bytes must be multiples of 16.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes,
                                         uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

// 2-D tiled TMA load of a box at (x, y) of `map` into shared memory, called
// by a whole warp, converged, with warp-uniform arguments: one elected lane
// issues the copy (a lone thread issuing was measured to fall far behind when
// other warps kept its SM sub-partition busy).
__device__ __forceinline__ void tma_load_2d_elect(uint32_t dst, const void* map, int x, int y,
                                                  uint32_t bar) {
  asm volatile(
      "{\n\t.reg .pred e;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "@e cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];\n\t}" ::"r"(dst),
      "l"(map), "r"(x), "r"(y), "r"(bar)
      : "memory");
}

// A 2-D tiled TMA load issued by the calling thread, with an L2 cache policy
// (from l2_policy_evict_first): the pages stream through once per launch, so
// they should leave L2 before the small data around them (split pieces,
// tables, query rows) does.
__device__ __forceinline__ void tma_load_2d_hint(uint32_t dst, const void* map, int x, int y,
                                                 uint32_t bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
      "l"(map), "r"(x), "r"(y), "r"(bar), "l"(policy)
      : "memory");
}

__device__ __forceinline__ uint64_t l2_policy_evict_first() {
  uint64_t policy;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(policy));
  return policy;
}

// Four 8x8 b16 matrices from shared memory; lanes 8m..8m+7 give matrix m's row addresses.
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t& r0, uint32_t& r1,
                                              uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

// D = A(16x16, row) * B(16x8, col) + D, bf16 inputs, fp32 accumulate.
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                               uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Two floats -> bf16x2 (round to nearest even), `lo` in the low half.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

__device__ __forceinline__ float2 lds64f(uint32_t addr) {
  float2 v;
  asm volatile("ld.shared.v2.f32 {%0,%1}, [%2];" : "=f"(v.x), "=f"(v.y) : "r"(addr));
  return v;
}

__device__ __forceinline__ uint2 lds64u(uint32_t addr) {
  uint2 v;
  asm volatile("ld.shared.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr));
  return v;
}

// 16 bytes global -> shared without passing through registers, cached in L2
// only (so a word another SM wrote is read from L2, not a stale L1 line).
// Both addresses 16-byte aligned.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}

// Wait until every cp_async16 this thread issued has landed.
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.wait_all;" ::: "memory");
}

__device__ __forceinline__ uint16_t lds16(uint32_t addr) {
  uint16_t v;
  asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(addr));
  return v;
}

__device__ __forceinline__ uint32_t lds32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(addr));
  return v;
}

__device__ __forceinline__ void sts16(uint32_t addr, uint16_t v) {
  asm volatile("st.shared.u16 [%0], %1;" ::"r"(addr), "h"(v) : "memory");
}

__device__ __forceinline__ void sts32(uint32_t addr, uint32_t v) {
  asm volatile("st.shared.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr));
  return v;
}

__device__ __forceinline__ float4 lds128f(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared.v4.f32 {%0,%1,%2,%3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(addr));
  return v;
}

// Two bf16 packed in a 32-bit word -> two floats (exact: a bf16 is the top
// half of a binary32).
__device__ __forceinline__ float2 bf16x2_to_float2(uint32_t w) {
  return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
}

// 2^x via the MUFU approximation (relative error ~2^-22); 2^-inf = 0.
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ double bf16_bits_to_double(uint16_t b) {
  return static_cast<double>(__uint_as_float(static_cast<uint32_t>(b) << 16));
}

// Round a double to the nearest bf16, ties to even, by integer manipulation
// of its IEEE-754 encoding. NaN becomes the quiet NaN 0x7FC0.
__device__ __forceinline__ uint16_t double_to_bf16_rne(double x) {
  const unsigned long long u = static_cast<unsigned long long>(__double_as_longlong(x));
  const uint16_t sign = static_cast<uint16_t>((u >> 48) & 0x8000u);
  const int biased = static_cast<int>((u >> 52) & 0x7ff);
  const unsigned long long frac = u & ((1ull << 52) - 1);
  if (biased == 0x7ff) return frac ? 0x7FC0 : static_cast<uint16_t>(sign | 0x7F80);
  if (biased == 0) return sign;  // |x| < 2^-1022 rounds to zero in bf16
  int e = biased - 1023;
  const unsigned long long sig = frac | (1ull << 52);  // 53-bit significand
  // bits to drop: to 8 significant bits for a normal bf16, more below 2^-126
  const int shift = (e >= -126) ? 45 : 45 + (-126 - e);
  if (shift >= 64) return sign;
  unsigned long long kept = sig >> shift;
  const unsigned long long rem = sig & ((1ull << shift) - 1);
  const unsigned long long half = 1ull << (shift - 1);
  if (rem > half || (rem == half && (kept & 1))) ++kept;
  if (e >= -126) {
    if (kept == (1ull << 8)) {  // carried into the next binade
      kept >>= 1;
      ++e;
    }
    if (e > 127) return static_cast<uint16_t>(sign | 0x7F80);
    return static_cast<uint16_t>(sign | ((e + 127) << 7) | (kept & 0x7f));
  }
  // subnormal bf16 (kept <= 128; 128 is the smallest normal, encoded the same way)
  return static_cast<uint16_t>(sign | kept);
}

// The new key's rotation, shared by the append kernel and the fused decode:
// y0 = x0*c - x1*s, y1 = x1*c + x0*s in fp64, every product and sum rounded
// once (no fused multiply-add), then each rounded once to bf16.
__device__ __forceinline__ void rotate_key_pair(uint16_t k0, uint16_t k1, double c, double s,
                                                uint16_t& y0, uint16_t& y1) {
  const double x0 = bf16_bits_to_double(k0), x1 = bf16_bits_to_double(k1);
  y0 = double_to_bf16_rne(__dsub_rn(__dmul_rn(x0, c), __dmul_rn(x1, s)));
  y1 = double_to_bf16_rne(__dadd_rn(__dmul_rn(x1, c), __dmul_rn(x0, s)));
}

// Key rotation without fp64 arithmetic, rounded exactly as fp64 would round it.
//
// The stored key element is bf16(fl64(fl64(a c) - fl64(b s))): two fp64
// products, their fp64 difference, then round-to-nearest-even to bf16 (the
// arithmetic the oracle and the fp64 append use; y0 takes a = x0, b = x1,
// y1 takes a = x1, b = -x0). fp64 throughput on this part is tiny, so the
// fast path evaluates the same difference in fp32 double-word arithmetic:
// c ~ ch + cl and s ~ sh + sl with |c - ch - cl| <= 2^-48 |c|; a ch = pa + ea
// exactly by an FMA (Dekker's two-product), a cl is one rounded product, and
// Knuth's two-sum keeps the cancellation of pa - pb exact. The result is the
// unevaluated sum f + res, within 2^-42 M of the fp64 difference, where
// M = max(|pa|, |pb|) (error terms: 2^-48 from the split of c, 2^-47 from
// a cl, 2^-46 from each low-order sum, 2^-44 from the last one; the fp64
// difference itself is within 3 2^-53 M of the exact one).
//
// bf16 rounding boundaries are the midpoints between neighbouring bf16
// values. With upper = the top 16 bits of f's magnitude and lower = its
// bottom 16, the nearest boundary is at magnitude (upper << 16) | 0x8000
// (the one below is at least 2^-10 |f| away). When f + res is farther than
// tol = 2^-36 M from it (64x the error bound), f + res, the fp64 difference
// and the exact value all round to the same bf16, which is upper, plus one
// when lower > 0x8000. Otherwise (a near-tie, a zero or subnormal result,
// heavy cancellation, huge or non-finite inputs) the function returns false
// and the caller takes the fp64 route.
__device__ __forceinline__ bool rotated_bf16_fast(float a, float b, float ch, float cl, float sh,
                                                  float sl, uint16_t& y) {
  const float pa = __fmul_rn(a, ch), ea = __fmaf_rn(a, ch, -pa);
  const float pb = __fmul_rn(b, sh), eb = __fmaf_rn(b, sh, -pb);
  const float ta = __fmul_rn(a, cl), tb = __fmul_rn(b, sl);
  // two-sum: s + t = pa - pb exactly
  const float s = __fsub_rn(pa, pb);
  const float sb = __fsub_rn(s, pa);
  const float sa = __fsub_rn(s, sb);
  const float t = __fadd_rn(__fsub_rn(pa, sa), __fsub_rn(-pb, sb));
  const float lo = __fadd_rn(t, __fsub_rn(__fadd_rn(ea, ta), __fadd_rn(eb, tb)));
  // two-sum: f + res = s + lo exactly
  const float f = __fadd_rn(s, lo);
  const float fb = __fsub_rn(f, s);
  const float fa = __fsub_rn(f, fb);
  const float res = __fadd_rn(__fsub_rn(s, fa), __fsub_rn(lo, fb));
  const float m = fmaxf(fabsf(pa), fabsf(pb));
  const float af = fabsf(f);
  const float tol = __fmul_rn(m, 0x1p-36f);
  // (comparisons with NaN are false, so non-finite values fail here too)
  if (!(m <= 0x1p120f) || !(af >= 0x1p-100f) || !(__fmul_rn(af, 0x1p-12f) > tol)) return false;
  const uint32_t u = __float_as_uint(f);
  const uint32_t mag = u & 0x7fffffffu;
  const uint32_t upper = mag >> 16, lower = mag & 0xffffu;
  const float mid = __uint_as_float((upper << 16) | 0x8000u);  // same binade as af: exact difference
  if (!(__fsub_rn(fabsf(__fsub_rn(mid, af)), fabsf(res)) > tol)) return false;
  y = static_cast<uint16_t>(((u >> 16) & 0x8000u) | (upper + (lower > 0x8000u ? 1u : 0u)));
  return true;
}

// Programmatic dependent launch. A kernel launched with programmatic stream
// serialization may start while the kernel before it in the stream is still
// running; grid_dependency_wait() blocks until that kernel has completed and
// its memory operations are visible (a no-op without such a predecessor), so
// every read of data an earlier kernel may write comes after it.
// grid_launch_dependents() lets the next kernel in the stream start early.
__device__ __forceinline__ void grid_dependency_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void grid_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// L2-coherent loads for data another CTA wrote during this launch.
__device__ __forceinline__ float ld_cg(const float* p) { return __ldcg(p); }
__device__ __forceinline__ float2 ld_cg2(const float2* p) { return __ldcg(p); }

}  // namespace pkv
