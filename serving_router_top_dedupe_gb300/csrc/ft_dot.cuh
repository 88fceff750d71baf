// Dot-product building blocks of the decode GEMV kernels.  Every (token, expert) dot is
// formed the same way in every kernel that uses these: 16-byte chunks strided over the
// lanes, accumulated in FP32 in chunk order, then an xor butterfly across the warp; an FP8
// block's dot product is first summed over the 8 lanes holding it and then scaled once.
#pragma once

#include <cuda_fp16.h>

#include <cstdint>

namespace ft {
namespace dot {

__device__ __forceinline__ uint4 ld_stream(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// ld_stream with an L2 cache policy (see ft::ptx::l2_evict_first).
__device__ __forceinline__ uint4 ld_stream(const void* p, uint64_t pol) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.u32 {%0,%1,%2,%3}, [%4], %5;"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p), "l"(pol));
  return v;
}

// Host-pool reads (mapped pinned memory over the host link): plain coherent loads with
// evict-first L2 policy.  The read-only .nc path is far slower for host memory.
__device__ __forceinline__ uint4 ld_host(const void* p) {
  return __ldcs(reinterpret_cast<const uint4*>(p));
}

__device__ __forceinline__ float ld_cg_f32(const float* p) {
  float v;
  asm volatile("ld.global.cg.f32 %0, [%1];" : "=f"(v) : "l"(p));
  return v;
}

// acc += w.lo*x.lo + w.hi*x.hi, BF16 operands, FP32 accumulation (exact products).
__device__ __forceinline__ float fma2_bf16(uint32_t w, uint32_t x, float acc) {
  asm("{\n\t.reg .b16 wl, wh, xl, xh;\n\t"
      "mov.b32 {wl, wh}, %1;\n\t"
      "mov.b32 {xl, xh}, %2;\n\t"
      "fma.rn.f32.bf16 %0, wl, xl, %0;\n\t"
      "fma.rn.f32.bf16 %0, wh, xh, %0;\n\t}"
      : "+f"(acc)
      : "r"(w), "r"(x));
  return acc;
}

// acc += w.lo*x.lo + w.hi*x.hi, F16 operands, FP32 accumulation (exact products).
__device__ __forceinline__ float fma2_f16(uint32_t w, uint32_t x, float acc) {
  asm("{\n\t.reg .b16 wl, wh, xl, xh;\n\t"
      "mov.b32 {wl, wh}, %1;\n\t"
      "mov.b32 {xl, xh}, %2;\n\t"
      "fma.rn.f32.f16 %0, wl, xl, %0;\n\t"
      "fma.rn.f32.f16 %0, wh, xh, %0;\n\t}"
      : "+f"(acc)
      : "r"(w), "r"(x));
  return acc;
}

// two E4M3 codes (low byte = element 0) -> f16x2 (element 0 in the low half)
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t two) {
  uint32_t r;
  asm("{\n\t.reg .b16 s;\n\tcvt.u16.u32 s, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, s;\n\t}" : "=r"(r) : "r"(two));
  return r;
}

// two E4M3 codes in a 16-bit word (low byte first) -> two floats (low byte in .x)
__device__ __forceinline__ float2 e4m3x2_to_float2(uint16_t two) {
  const uint32_t h2 = e4m3x2_to_f16x2(two);
  return __half22float2(*reinterpret_cast<const __half2*>(&h2));
}

// two E2M1 (FP4) codes in one byte (low nibble = element 0) -> f16x2 (element 0 in the
// low half)
__device__ __forceinline__ uint32_t e2m1x2_to_f16x2(uint32_t byte) {
  uint32_t r;
  asm("{\n\t.reg .b8 s;\n\tcvt.u8.u32 s, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, s;\n\t}" : "=r"(r) : "r"(byte));
  return r;
}

// one 16-element NVFP4 block: E2M1 codes in two 32-bit words (w0: elements 0..7, low byte
// first) . 16 F16 values (xa: 0..7, xb: 8..15) -> the block's partial dot (not scaled)
__device__ __forceinline__ float dot16_e2m1_f16(uint32_t w0, uint32_t w1, uint4 xa, uint4 xb) {
  float d = 0.f;
  d = fma2_f16(e2m1x2_to_f16x2(w0 & 0xffu), xa.x, d);
  d = fma2_f16(e2m1x2_to_f16x2((w0 >> 8) & 0xffu), xa.y, d);
  d = fma2_f16(e2m1x2_to_f16x2((w0 >> 16) & 0xffu), xa.z, d);
  d = fma2_f16(e2m1x2_to_f16x2(w0 >> 24), xa.w, d);
  d = fma2_f16(e2m1x2_to_f16x2(w1 & 0xffu), xb.x, d);
  d = fma2_f16(e2m1x2_to_f16x2((w1 >> 8) & 0xffu), xb.y, d);
  d = fma2_f16(e2m1x2_to_f16x2((w1 >> 16) & 0xffu), xb.z, d);
  d = fma2_f16(e2m1x2_to_f16x2(w1 >> 24), xb.w, d);
  return d;
}

// one 16-element NVFP4 block . 16 FP32 values -> the block's partial dot (not scaled)
__device__ __forceinline__ float dot16_e2m1_f32(uint32_t w0, uint32_t w1, const float* v) {
  float d = 0.f;
  const uint32_t ws[2] = {w0, w1};
#pragma unroll
  for (int q = 0; q < 2; ++q) {
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      const uint32_t h2 = e2m1x2_to_f16x2((ws[q] >> (8 * b)) & 0xffu);
      const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&h2));
      d = fmaf(f.x, v[8 * q + 2 * b], d);
      d = fmaf(f.y, v[8 * q + 2 * b + 1], d);
    }
  }
  return d;
}

// 16 bytes of BF16 weights (8 elements) . 8 BF16 activations
__device__ __forceinline__ float dot_bf16_bf16(uint4 w, uint4 x, float acc) {
  acc = fma2_bf16(w.x, x.x, acc);
  acc = fma2_bf16(w.y, x.y, acc);
  acc = fma2_bf16(w.z, x.z, acc);
  acc = fma2_bf16(w.w, x.w, acc);
  return acc;
}

// 16 bytes of BF16 weights (8 elements) . 8 FP32 values
__device__ __forceinline__ float dot_bf16_f32(uint4 w, const float* v, float acc) {
  const float4 a = *reinterpret_cast<const float4*>(v);
  const float4 b = *reinterpret_cast<const float4*>(v + 4);
  acc = fmaf(__uint_as_float(w.x << 16), a.x, acc);
  acc = fmaf(__uint_as_float(w.x & 0xffff0000u), a.y, acc);
  acc = fmaf(__uint_as_float(w.y << 16), a.z, acc);
  acc = fmaf(__uint_as_float(w.y & 0xffff0000u), a.w, acc);
  acc = fmaf(__uint_as_float(w.z << 16), b.x, acc);
  acc = fmaf(__uint_as_float(w.z & 0xffff0000u), b.y, acc);
  acc = fmaf(__uint_as_float(w.w << 16), b.z, acc);
  acc = fmaf(__uint_as_float(w.w & 0xffff0000u), b.w, acc);
  return acc;
}

// dot_bf16_f32 with the 8 FP32 values given as two float4 (same products, same order)
__device__ __forceinline__ float dot_bf16_f32v(uint4 w, float4 a, float4 b, float acc) {
  acc = fmaf(__uint_as_float(w.x << 16), a.x, acc);
  acc = fmaf(__uint_as_float(w.x & 0xffff0000u), a.y, acc);
  acc = fmaf(__uint_as_float(w.y << 16), a.z, acc);
  acc = fmaf(__uint_as_float(w.y & 0xffff0000u), a.w, acc);
  acc = fmaf(__uint_as_float(w.z << 16), b.x, acc);
  acc = fmaf(__uint_as_float(w.z & 0xffff0000u), b.y, acc);
  acc = fmaf(__uint_as_float(w.w << 16), b.z, acc);
  acc = fmaf(__uint_as_float(w.w & 0xffff0000u), b.w, acc);
  return acc;
}

// one 32-bit word of E4M3 codes (4 elements) . 4 F16 values (as two f16x2 words)
__device__ __forceinline__ float dot4_e4m3_f16(uint32_t w, uint32_t x01, uint32_t x23, float acc) {
  acc = fma2_f16(e4m3x2_to_f16x2(w & 0xffffu), x01, acc);
  acc = fma2_f16(e4m3x2_to_f16x2(w >> 16), x23, acc);
  return acc;
}

// 16 bytes of E4M3 weights (16 elements) . 16 F16 values -> partial (not scaled)
__device__ __forceinline__ float dot_e4m3_f16(uint4 w, uint4 xa, uint4 xb) {
  float d = 0.f;
  d = dot4_e4m3_f16(w.x, xa.x, xa.y, d);
  d = dot4_e4m3_f16(w.y, xa.z, xa.w, d);
  d = dot4_e4m3_f16(w.z, xb.x, xb.y, d);
  d = dot4_e4m3_f16(w.w, xb.z, xb.w, d);
  return d;
}

// 16 bytes of E4M3 weights . 16 FP32 values -> partial (not scaled)
__device__ __forceinline__ float dot_e4m3_f32(uint4 w, const float* v) {
  float d = 0.f;
  const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const float4 xv = *reinterpret_cast<const float4*>(v + 4 * q);
    uint32_t p01 = e4m3x2_to_f16x2(ws[q] & 0xffffu), p23 = e4m3x2_to_f16x2(ws[q] >> 16);
    float2 f01 = __half22float2(*reinterpret_cast<const __half2*>(&p01));
    float2 f23 = __half22float2(*reinterpret_cast<const __half2*>(&p23));
    d = fmaf(f01.x, xv.x, d);
    d = fmaf(f01.y, xv.y, d);
    d = fmaf(f23.x, xv.z, d);
    d = fmaf(f23.y, xv.w, d);
  }
  return d;
}

// dot_e4m3_f32 with the 16 FP32 values given as four float4 (same products, same order)
__device__ __forceinline__ float dot_e4m3_f32v(uint4 w, const float4 (&xv)[4]) {
  float d = 0.f;
  const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    uint32_t p01 = e4m3x2_to_f16x2(ws[q] & 0xffffu), p23 = e4m3x2_to_f16x2(ws[q] >> 16);
    float2 f01 = __half22float2(*reinterpret_cast<const __half2*>(&p01));
    float2 f23 = __half22float2(*reinterpret_cast<const __half2*>(&p23));
    d = fmaf(f01.x, xv[q].x, d);
    d = fmaf(f01.y, xv[q].y, d);
    d = fmaf(f23.x, xv[q].z, d);
    d = fmaf(f23.y, xv[q].w, d);
  }
  return d;
}

// FP8 rows are read as 16-byte chunks strided over the lanes, 32 consecutive chunks per
// step, so the 8 chunks of one 1x128 block sit in the 8 lanes 8m .. 8m+7.  group8_sum adds a
// value over those 8 lanes (xor butterfly, the same sum in each of them): the block's dot
// product, formed before its scale multiplies it once.  groups_sum then adds the 4 groups'
// values (each held by all 8 lanes of its group).
__device__ __forceinline__ float group8_sum(float v) {
  v += __shfl_xor_sync(0xffffffffu, v, 1);
  v += __shfl_xor_sync(0xffffffffu, v, 2);
  v += __shfl_xor_sync(0xffffffffu, v, 4);
  return v;
}

__device__ __forceinline__ float groups_sum(float v) {
  v += __shfl_xor_sync(0xffffffffu, v, 8);
  v += __shfl_xor_sync(0xffffffffu, v, 16);
  return v;
}

// 2^s as a float, for -126 <= s <= 127 (built from the exponent field: exact).
__device__ __forceinline__ float pow2i(int s) { return __uint_as_float((uint32_t)(s + 127) << 23); }

// Activations of the FP8 and FP4 paths enter the products as F16.  BF16 reaches far beyond
// F16's range, so each token is first scaled by an exact power of two 2^-s chosen from its
// largest magnitude: that magnitude lands in [2^14, 2^15), every BF16 value within 2^28 of
// it converts to F16 exactly, and only values below 2^-39 of it are lost.  The finished sum
// is multiplied by 2^s (exact).  `maxbits` is the largest (bf16 bits & 0x7fff) of the token
// (BF16 magnitudes order like their bit patterns).
__device__ __forceinline__ int act_shift(uint32_t maxbits) {
  if (maxbits == 0) return 0;
  const int s = (int)(maxbits >> 7) - 127 - 14;
  return s < -126 ? -126 : (s > 113 ? 113 : s);
}

// max over the 8 BF16 magnitudes of a 16-byte vector and `m` (halfword-wise, then folded)
__device__ __forceinline__ uint32_t bf16x8_maxbits(uint4 v, uint32_t m) {
  const uint32_t k = 0x7fff7fffu;
  uint32_t a = __vmaxu2(__vmaxu2(v.x & k, v.y & k), __vmaxu2(v.z & k, v.w & k));
  a = a > 0xffffu ? max(a >> 16, a & 0xffffu) : a;
  return max(m, a);
}

// 8 BF16 values (one 16-byte vector) times 2^-s, as 8 F16 values
__device__ __forceinline__ uint4 bf16x8_to_f16x8_scaled(uint4 v, float scale) {
  const uint32_t in[4] = {v.x, v.y, v.z, v.w};
  uint32_t o[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    __half2 hh = __floats2half2_rn(__uint_as_float(in[q] << 16) * scale, __uint_as_float(in[q] & 0xffff0000u) * scale);
    o[q] = *reinterpret_cast<uint32_t*>(&hh);
  }
  return make_uint4(o[0], o[1], o[2], o[3]);
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ float silu_mul(float a, float b) { return a / (1.0f + expf(-a)) * b; }

}  // namespace dot
}  // namespace ft
