// Device helpers shared by the two decode-layer kernels (layer.cu: block
// scales as stored, [E, N, K/bs]; decode.cu: k-major block scales
// [E, K/bs, N]): mbarrier, bulk-copy and tensor-copy wrappers, the E2M1 and
// block-scale decoders and the fp16 activation staging helpers.
#pragma once

#include <cuda.h>
#include <cuda_fp16.h>

#include "route_common.cuh"

namespace qmoe {

// ---- PTX helpers --------------------------------------------------------------

__device__ __forceinline__ uint32_t smem_addr(const void *p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_fence_init() { asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory"); }
__device__ __forceinline__ void mbar_expect_tx(uint64_t *bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   smem_addr(dst)),
               "l"(src), "r"(bytes), "r"(smem_addr(bar))
               : "memory");
}
// The same with an L2 eviction-priority policy (createpolicy): the weight
// stream is read once per call, so it is marked evict-first and leaves the
// kernel's code, activations and partial sums in L2 across calls.
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}
__device__ __forceinline__ void bulk_g2s_stream(void *dst, const void *src, uint32_t bytes, uint64_t *bar,
                                                uint64_t pol) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
          smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar)), "l"(pol)
      : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}"
      : "=r"(done)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return done != 0u;
}
// L2 prefetch of a contiguous run (size a multiple of 16 bytes), and of one
// box of a 2-D tensor map: the data is brought into L2 ahead of its copy.
__device__ __forceinline__ void bulk_prefetch_l2(const void *src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}
__device__ __forceinline__ void tensor_prefetch_l2_2d(const CUtensorMap *map, int x, int y) {
  asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(x), "r"(y)
               : "memory");
}
// 2-D tensor copy global -> shared, completion counted on an mbarrier.
__device__ __forceinline__ void tensor_g2s_2d(void *dst, const CUtensorMap *map, int x, int y, uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_addr(bar))
      : "memory");
}
// 16-byte copy global -> shared through the load/store path (not the bulk
// copy engine, so it does not queue behind the weight stream).
__device__ __forceinline__ void cp_async16(void *dst, const void *src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(dst)), "l"(src) : "memory");
}
// Arrive on `bar` once every cp.async this thread issued before has landed
// (the arrival counts against the barrier's expected count).
__device__ __forceinline__ void cp_async_arrive(uint64_t *bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ int ld_acquire(const int32_t *p) {
  int v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// ---- scales and activation helpers -----------------------------------------------

// Raw block scale as fp32 (MXFP4 block scales; NVFP4 ones go through the
// hardware E4M3 conversion).  NVFP4: E4M3 value * 2^-120 (exact); MXFP4:
// 2^(b-127).  `special` is set for codes that need the exact slow path (NaN;
// E8M0 0 / 255).
template <int FMT>
__device__ __forceinline__ float raw_scale(uint32_t b, bool &special) {
  if (FMT == QMOE_NVFP4) {
    special |= (b & 0x7Fu) == 0x7Fu;
    const float f = __uint_as_float((b & 0x7Fu) << 20);
    return (b & 0x80u) ? -f : f;
  } else {
    special |= (b == 0u) || (b == 0xFFu);
    return __uint_as_float(b << 23);
  }
}
template <int FMT>
__device__ __forceinline__ float exact_raw_scale(uint32_t b) {
  if (FMT == QMOE_NVFP4) return e4m3_to_f32(b) * 0x1p-120f;  // NaN stays NaN
  return e8m0_to_f32(b);
}

__device__ __forceinline__ float pow2f(int e) { return __uint_as_float((uint32_t)(127 + e) << 23); }

// x * 2^d for |d| <= 254 (two exact power-of-two steps).
__device__ __forceinline__ float ldexp2(float x, int d) {
  const int h = d / 2;
  return x * pow2f(h) * pow2f(d - h);
}


// Shift that puts the largest |x| (bf16 bits, sign cleared) in [2^14, 2^15).
__device__ __forceinline__ int row_shift(uint32_t m) {
  return m == 0u ? 0 : max(-100, min(100, (int)((m >> 7) & 0xFFu) - 127 - 14));
}

__device__ __forceinline__ uint32_t absmax_bf16x8(const uint4 &v) {
  const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
  uint32_t m = 0;
#pragma unroll
  for (int q = 0; q < 4; ++q) m = max(m, max(w4[q] & 0x7FFFu, (w4[q] >> 16) & 0x7FFFu));
  return m;
}

// 8 bf16 -> 8 fp16 scaled by f (a power of two)
__device__ __forceinline__ uint4 bf16x8_to_f16x8(const uint4 &x4, float f) {
  const uint32_t w4[4] = {x4.x, x4.y, x4.z, x4.w};
  uint32_t o[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const __half2 h = __floats2half2_rn(bf16_to_f32(w4[q] & 0xFFFFu) * f, bf16_to_f32(w4[q] >> 16) * f);
    o[q] = *reinterpret_cast<const uint32_t *>(&h);
  }
  return make_uint4(o[0], o[1], o[2], o[3]);
}

// The 8 E2M1 codes of a word -> 4 f16x2 (byte q -> p[q]; low nibble in the low half).
__device__ __forceinline__ void dec8(uint32_t w, uint32_t (&p)[4]) {
  asm("{ .reg .b8 b0, b1, b2, b3;\n mov.b32 {b0, b1, b2, b3}, %4;\n"
      " cvt.rn.f16x2.e2m1x2 %0, b0;\n cvt.rn.f16x2.e2m1x2 %1, b1;\n"
      " cvt.rn.f16x2.e2m1x2 %2, b2;\n cvt.rn.f16x2.e2m1x2 %3, b3; }"
      : "=r"(p[0]), "=r"(p[1]), "=r"(p[2]), "=r"(p[3])
      : "r"(w));
}
// a[c] += p[c] * x.lo + q[c] * x.hi for the 8 columns c, fp16 operands with
// exact products (fma.rn.f32.f16), fp32 accumulation; x = the fp16 pair of
// two consecutive k rows (p: the word of the first row, q: of the second).
__device__ __forceinline__ void fma16(const uint32_t (&p)[4], const uint32_t (&q)[4], uint32_t x2, float (&a)[8]) {
  asm("{ .reg .f16 x0, x1, l0, h0, l1, h1, l2, h2, l3, h3;\n mov.b32 {x0, x1}, %16;\n"
      " mov.b32 {l0, h0}, %8;\n mov.b32 {l1, h1}, %9;\n mov.b32 {l2, h2}, %10;\n mov.b32 {l3, h3}, %11;\n"
      " fma.rn.f32.f16 %0, l0, x0, %0;\n fma.rn.f32.f16 %1, h0, x0, %1;\n"
      " fma.rn.f32.f16 %2, l1, x0, %2;\n fma.rn.f32.f16 %3, h1, x0, %3;\n"
      " fma.rn.f32.f16 %4, l2, x0, %4;\n fma.rn.f32.f16 %5, h2, x0, %5;\n"
      " fma.rn.f32.f16 %6, l3, x0, %6;\n fma.rn.f32.f16 %7, h3, x0, %7;\n"
      " mov.b32 {l0, h0}, %12;\n mov.b32 {l1, h1}, %13;\n mov.b32 {l2, h2}, %14;\n mov.b32 {l3, h3}, %15;\n"
      " fma.rn.f32.f16 %0, l0, x1, %0;\n fma.rn.f32.f16 %1, h0, x1, %1;\n"
      " fma.rn.f32.f16 %2, l1, x1, %2;\n fma.rn.f32.f16 %3, h1, x1, %3;\n"
      " fma.rn.f32.f16 %4, l2, x1, %4;\n fma.rn.f32.f16 %5, h2, x1, %5;\n"
      " fma.rn.f32.f16 %6, l3, x1, %6;\n fma.rn.f32.f16 %7, h3, x1, %7; }"
      : "+f"(a[0]), "+f"(a[1]), "+f"(a[2]), "+f"(a[3]), "+f"(a[4]), "+f"(a[5]), "+f"(a[6]), "+f"(a[7])
      : "r"(p[0]), "r"(p[1]), "r"(p[2]), "r"(p[3]), "r"(q[0]), "r"(q[1]), "r"(q[2]), "r"(q[3]), "r"(x2));
}

// Two E4M3 bytes (low 16 bits) -> f16x2, exact (every E4M3 value is an f16).
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t two) {
  uint32_t r;
  asm("{ .reg .b16 t; cvt.u16.u32 t, %1; cvt.rn.f16x2.e4m3x2 %0, t; }" : "=r"(r) : "r"(two));
  return r;
}

// The 8 block scales of a thread's column word.  NVFP4: the E4M3 values
// themselves (hardware conversion, NaN codes give NaN); MXFP4: 2^(b-127).
template <int FMT>
__device__ __forceinline__ void block_scales8(uint2 sv, float (&sc)[8]) {
  if constexpr (FMT == QMOE_NVFP4) {
    const uint32_t h[4] = {e4m3x2_to_f16x2(sv.x & 0xFFFFu), e4m3x2_to_f16x2(sv.x >> 16),
                           e4m3x2_to_f16x2(sv.y & 0xFFFFu), e4m3x2_to_f16x2(sv.y >> 16)};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const __half2 v = *reinterpret_cast<const __half2 *>(&h[q]);
      sc[2 * q] = __low2float(v);
      sc[2 * q + 1] = __high2float(v);
    }
    return;
  }
  bool special = false;
#pragma unroll
  for (int c = 0; c < 8; ++c) sc[c] = raw_scale<FMT>(((c < 4 ? sv.x : sv.y) >> (8 * (c & 3))) & 0xFFu, special);
  if (special) {
#pragma unroll
    for (int c = 0; c < 8; ++c) sc[c] = exact_raw_scale<FMT>(((c < 4 ? sv.x : sv.y) >> (8 * (c & 3))) & 0xFFu);
  }
}

}  // namespace qmoe
