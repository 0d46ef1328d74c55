// nvr_device.cuh -- device-side building blocks of the NVFP4 router (sm_103a).
//
// * NVFP4 block quantization (the arithmetic of the runtime-gsa section of
//   "nvfp4-megamoe-kernel commit 04cf8ca: dsv4/layers/router.py"), shared by
//   the quantize kernel and the single-launch decode kernel so both produce
//   identical bits.
// * Thin inline-PTX wrappers for mbarriers, TMA, tcgen05 (tensor memory,
//   block-scaled MMA) and packed fp32x2 arithmetic, written from the public
//   PTX ISA description of each instruction.
// * The register top-k list of the router epilogue.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>
#include <cuda_bf16.h>

namespace nvr {

// ------------------------------------------------------------------ constants
constexpr int kBlock = 16;                 // elements per NVFP4 scale block
constexpr float kGsaDivisor = 2688.0f;     // 6 (E2M1 max) * 448 (E4M3 max)

// workspace control words (byte offsets inside the first 256 bytes)
constexpr int kWsStatus = 0;
constexpr int kWsAmaxTicket = 4;
constexpr int kWsDecodeTicket = 8;
// (byte 12 is unused)
constexpr int kWsFusedAmax = 16;           // fused router's in-kernel amax: 5 words (2 maxima, 2 arrivals, generation)
constexpr uint32_t kStatusTimeout = 6;     // == NVR_ERR_TIMEOUT

// ------------------------------------------------------------------ small PTX
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Record a timeout in the workspace status word (first writer wins).
__device__ __forceinline__ void report_timeout(uint32_t* status) {
  if (status) atomicCAS(status, 0u, kStatusTimeout);
}

// ------------------------------------------------------------ fp32x2 packing
__device__ __forceinline__ uint64_t f2_pack(float lo, float hi) {
  return (static_cast<uint64_t>(__float_as_uint(hi)) << 32) | __float_as_uint(lo);
}
__device__ __forceinline__ float f2_lo(uint64_t v) { return __uint_as_float(static_cast<uint32_t>(v)); }
__device__ __forceinline__ float f2_hi(uint64_t v) { return __uint_as_float(static_cast<uint32_t>(v >> 32)); }
__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}

// ----------------------------------------------------- correctly rounded a/b
//
// Division by a value b whose reciprocal rb = RN(1/b) is known, without the
// multi-function unit: q0 = RN(a*rb) is within 1.5 ulp of a/b; one correction
// q1 = RN(q0 + RN(a - b*q0)*rb) brings it within one ulp; a second correction
// then gives exactly RN(a/b) by Markstein's theorem (P. Markstein, "Computation
// of elementary functions on the IBM RISC System/6000 processor", IBM J. Res.
// Dev. 34(1), 1990; restated in Muller et al., Handbook of Floating-Point
// Arithmetic, section on Newton-Raphson division): if rb is within half an ulp
// of 1/b and q within one ulp of a/b, the residual r = a - b*q is exact under
// a fused multiply-add and RN(q + r*rb) = RN(a/b).  Hypotheses: no overflow and
// no underflow of the residual, which hold for b and 1/b in [2^-80, 2^80] and
// |a| >= 2^-100.  For smaller |a| the result is still within a few ulp with the
// right sign; the quantizer only uses such quotients where the code is decided
// by the sign alone (see quant_block16).
__device__ __forceinline__ float div_rn(float a, float b, float rb) {
  float q = __fmul_rn(a, rb);
  float r = __fmaf_rn(-q, b, a);
  q = __fmaf_rn(r, rb, q);
  r = __fmaf_rn(-q, b, a);
  return __fmaf_rn(r, rb, q);
}

// The same on two lanes at once (packed fp32x2 pipe); nb2 = (-b, -b).
__device__ __forceinline__ uint64_t div_rn2(uint64_t a2, uint64_t nb2, uint64_t rb2) {
  uint64_t q = f2_mul(a2, rb2);
  uint64_t r = f2_fma(q, nb2, a2);
  q = f2_fma(r, rb2, q);
  r = f2_fma(q, nb2, a2);
  return f2_fma(r, rb2, q);
}

// Division by a divisor with a short significand: b = d * 2^k with d an odd
// integer <= 15 (every E4M3 scale value, and 6).  Then ONE correction gives
// RN(a/b): q0 = RN(a*rb) is within 2 ulp of a/b; c = q0 + (a - b*q0)*rb
// (residual exact under a fused multiply-add, one rounding in the final fma)
// differs from a/b by at most |a/b - q0| * 2^-24 < 2^-23 ulp.  RN(c) can only
// differ from RN(a/b) if a rounding midpoint M lies within that distance of
// a/b; but a*2^-k - M*d is a nonzero multiple of ulp/2 (a*2^-k lies on a grid
// no finer than ulp(a/b), while M*d is an odd multiple of ulp/2), so
// |a/b - M| >= ulp/(2d) >= ulp/30.  Hypotheses as for div_rn (no overflow,
// a/b not subnormal); a subnormal quotient is < 0.25 and encodes as a signed
// zero whatever its last bits.
__device__ __forceinline__ float div_rn_short(float a, float b, float rb) {
  const float q = __fmul_rn(a, rb);
  const float r = __fmaf_rn(-q, b, a);
  return __fmaf_rn(r, rb, q);
}
__device__ __forceinline__ uint64_t div_rn2_short(uint64_t a2, uint64_t nb2, uint64_t rb2) {
  const uint64_t q = f2_mul(a2, rb2);
  const uint64_t r = f2_fma(q, nb2, a2);
  return f2_fma(r, rb2, q);
}

// ------------------------------------------------------- format conversions
// E4M3 byte of a non-negative fp32 (nearest-even, saturating at 448).
__device__ __forceinline__ uint32_t e4m3_byte(float v) {
  uint16_t h;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(h) : "f"(0.0f), "f"(v));
  return h & 0xFFu;
}

// Value of an E4M3 byte in 0x00..0x7E (exact).
__device__ __forceinline__ float e4m3_value(uint32_t b) {
  const uint32_t e = (b >> 3) & 0xFu, m = b & 7u;
  if (e == 0) return static_cast<float>(m) * 0.001953125f;            // m * 2^-9
  return __uint_as_float(((e + 120u) << 23) | (m << 20));              // (1 + m/8) * 2^(e-7)
}

// Four packed E2M1 bytes from eight fp32 values; element 2j in the low nibble
// of byte j (nearest-even, saturating at 6).
__device__ __forceinline__ uint32_t e2m1_pack8(float v0, float v1, float v2, float v3, float v4,
                                              float v5, float v6, float v7) {
  uint32_t r;
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b2, %6, %5;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b3, %8, %7;\n\t"
      "mov.b32 %0, {b0, b1, b2, b3};\n\t}"
      : "=r"(r)
      : "f"(v0), "f"(v1), "f"(v2), "f"(v3), "f"(v4), "f"(v5), "f"(v6), "f"(v7));
  return r;
}

// ----------------------------------------------------- NVFP4 block quantizer
//
// Per-call constants of the quantizer for one tensor.
struct QuantScale {
  float gsa;     // global scale
  float rgsa;    // RN(1 / gsa)
  int mode;      // 0: gsa == 0 (all zero), 1: fast (Markstein), 2: IEEE divide
};

__device__ __forceinline__ QuantScale make_quant_scale(float amax) {
  QuantScale q;
  q.gsa = __fdiv_rn(amax, kGsaDivisor);
  q.rgsa = q.gsa > 0.0f ? __frcp_rn(q.gsa) : 0.0f;
  // Markstein's hypotheses need gsa and 1/gsa inside [2^-80, 2^80]
  const float lo = 8.27180613e-25f;   // 2^-80
  const float hi = 1.20892582e+24f;   // 2^80
  q.mode = (q.gsa == 0.0f) ? 0 : ((q.gsa >= lo && q.gsa <= hi) ? 1 : 2);
  return q;
}

// One block of input: 16 values widened to fp32, plus the sign of every
// element as nibble masks (bit 4i+3 set when element i, resp. i+8, has its
// sign bit set).  The hardware E2M1 conversion encodes a negative value that
// rounds to zero as +0; the sign masks restore the signed zero (0x8).
struct Block16 {
  float v[16];
  uint32_t neg_lo, neg_hi;
};

// Sign nibble mask of 8 bf16 values held in 4 words (element 2k in the low
// half of word k): gather the high byte of every element with byte permutes,
// split even and odd elements, and move each sign bit to bit 3 / bit 7 of the
// output byte.
__device__ __forceinline__ uint32_t bf16x8_sign_nibbles(uint32_t w0, uint32_t w1, uint32_t w2,
                                                        uint32_t w3) {
  uint32_t t01, t23, ev, od;
  asm("prmt.b32 %0, %1, %2, 0x7531;" : "=r"(t01) : "r"(w0), "r"(w1));   // e0 o1 e2 o3
  asm("prmt.b32 %0, %1, %2, 0x7531;" : "=r"(t23) : "r"(w2), "r"(w3));   // e4 o5 e6 o7
  asm("prmt.b32 %0, %1, %2, 0x6420;" : "=r"(ev) : "r"(t01), "r"(t23));  // e0 e2 e4 e6
  asm("prmt.b32 %0, %1, %2, 0x7531;" : "=r"(od) : "r"(t01), "r"(t23));  // o1 o3 o5 o7
  return ((ev >> 4) & 0x08080808u) | (od & 0x80808080u);
}

// Sign nibble mask of 8 fp32 values.
__device__ __forceinline__ uint32_t f32x8_sign_nibbles(const float* v) {
  uint32_t m = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) m |= (__float_as_uint(v[i]) >> 31) << (4 * i + 3);
  return m;
}

// Quantize 16 fp32 values (one scale block).  Writes 8 bytes of packed codes
// (lo: elements 0-7, hi: 8-15) and returns the E4M3 scale byte.
//   y_i = RN(x_i / gsa); sy = RN(max|y| / 6); byte = E4M3(sy);
//   code_i = E2M1(RN(y_i / dec(byte))) with the sign of x_i (a negative value
//   that rounds to zero is -0, code 0x8); byte == 0 -> all codes 0.
// Exactness of the division shortcuts: y_i is exact whenever |x_i| >= 2^-100
// (mode 1) or always (mode 2).  When |x_i| < 2^-100, |y_i| < 2^-20 and
// |y_i / s| < 2^-11 for every nonzero scale s >= 2^-9, so the code is the
// signed zero whatever the last bits of y_i are.  max|y| / 6 and y / s divide
// by short significands (6 = 3 * 2, s = (8 + m) * 2^(e-10)): div_rn_short.
// `rcp_tab`, when given, holds RN(1 / dec(b)) for every scale byte b in
// 1..126 (the same bits __frcp_rn returns).
__device__ __forceinline__ uint32_t quant_block16(const Block16& blk, const QuantScale& qs,
                                                  uint32_t& codes_lo, uint32_t& codes_hi,
                                                  const float* rcp_tab = nullptr) {
  const float (&x)[16] = blk.v;
  if (qs.mode == 0) { codes_lo = codes_hi = 0; return 0; }
  float y[16];
  if (qs.mode == 1) {
    const uint64_t nb2 = f2_pack(-qs.gsa, -qs.gsa), rb2 = f2_pack(qs.rgsa, qs.rgsa);
#pragma unroll
    for (int i = 0; i < 16; i += 2) {
      const uint64_t q = div_rn2(f2_pack(x[i], x[i + 1]), nb2, rb2);
      y[i] = f2_lo(q);
      y[i + 1] = f2_hi(q);
    }
  } else {
#pragma unroll
    for (int i = 0; i < 16; ++i) y[i] = __fdiv_rn(x[i], qs.gsa);
  }
  float m = 0.0f;
#pragma unroll
  for (int i = 0; i < 16; ++i) m = fmaxf(m, fabsf(y[i]));
  const float r6 = 0.16666667163372039794921875f;       // RN(1/6)
  const float sy = div_rn_short(m, 6.0f, r6);
  const uint32_t byte = e4m3_byte(sy);
  if (byte == 0) { codes_lo = codes_hi = 0; return 0; }
  const float s = e4m3_value(byte);
  const float rs = rcp_tab ? rcp_tab[byte] : __frcp_rn(s);
  const uint64_t ns2 = f2_pack(-s, -s), rs2 = f2_pack(rs, rs);
  float q[16];
#pragma unroll
  for (int i = 0; i < 16; i += 2) {
    const uint64_t v = div_rn2_short(f2_pack(y[i], y[i + 1]), ns2, rs2);
    q[i] = f2_lo(v);
    q[i + 1] = f2_hi(v);
  }
  codes_lo = e2m1_pack8(q[0], q[1], q[2], q[3], q[4], q[5], q[6], q[7]) | blk.neg_lo;
  codes_hi = e2m1_pack8(q[8], q[9], q[10], q[11], q[12], q[13], q[14], q[15]) | blk.neg_hi;
  return byte;
}

// quant_block16 at a fraction of its multiply-adds, same scale byte and
// codes.  Mode 1 only (else quant_block16 itself).
//   byte: RN(max|x| / gsa) = max RN(|x_i| / gsa) (correctly rounded division
//     is monotone), then the same chain as quant_block16;
//   codes: with c = RN(RN(1/gsa) * RN(1/s)) and c_lo/hi = RN(c (1 -/+ 2^-20)),
//     the products P_lo/hi = RN(x c_lo/hi) lie within 5 ulp of x / (gsa s),
//     the exact q = RN(RN(x / gsa) / s) within 2, and the margin is 16 ulp:
//     P_lo <= q <= P_hi in magnitude.  E2M1 rounding is monotone, so where
//     the two code words agree they are the exact codes; otherwise (some q
//     within ~2^-20 of a rounding boundary, e.g. an exact tie) the block is
//     quantized again by quant_block16.  Elements too small for the error
//     bounds (subnormal products) give zero codes on both sides.
__device__ __forceinline__ uint32_t quant_block16_bracket(const Block16& blk, const QuantScale& qs,
                                                          uint32_t& codes_lo, uint32_t& codes_hi,
                                                          const float* rcp_tab = nullptr) {
  if (qs.mode != 1) return quant_block16(blk, qs, codes_lo, codes_hi, rcp_tab);
  const float (&x)[16] = blk.v;
  float m = 0.0f;
#pragma unroll
  for (int i = 0; i < 16; ++i) m = fmaxf(m, fabsf(x[i]));
  const float r6 = 0.16666667163372039794921875f;       // RN(1/6)
  const uint32_t byte = e4m3_byte(div_rn_short(div_rn(m, qs.gsa, qs.rgsa), 6.0f, r6));
  if (byte == 0) { codes_lo = codes_hi = 0; return 0; }
  const float c = __fmul_rn(qs.rgsa, rcp_tab ? rcp_tab[byte] : __frcp_rn(e4m3_value(byte)));
  const float c_lo = __fmul_rn(c, 0.99999904632568359375f);    // 1 - 2^-20
  const float c_hi = __fmul_rn(c, 1.00000095367431640625f);    // 1 + 2^-20
  const uint64_t lo2 = f2_pack(c_lo, c_lo), hi2 = f2_pack(c_hi, c_hi);
  float a[16], b[16];
#pragma unroll
  for (int i = 0; i < 16; i += 2) {
    const uint64_t xp = f2_pack(x[i], x[i + 1]);
    const uint64_t pl = f2_mul(xp, lo2), ph = f2_mul(xp, hi2);
    a[i] = f2_lo(pl); a[i + 1] = f2_hi(pl);
    b[i] = f2_lo(ph); b[i + 1] = f2_hi(ph);
  }
  const uint32_t l0 = e2m1_pack8(a[0], a[1], a[2], a[3], a[4], a[5], a[6], a[7]);
  const uint32_t l1 = e2m1_pack8(a[8], a[9], a[10], a[11], a[12], a[13], a[14], a[15]);
  const uint32_t h0 = e2m1_pack8(b[0], b[1], b[2], b[3], b[4], b[5], b[6], b[7]);
  const uint32_t h1 = e2m1_pack8(b[8], b[9], b[10], b[11], b[12], b[13], b[14], b[15]);
  if ((l0 ^ h0) | (l1 ^ h1)) return quant_block16(blk, qs, codes_lo, codes_hi, rcp_tab);
  codes_lo = l0 | blk.neg_lo;
  codes_hi = l1 | blk.neg_hi;
  return byte;
}

// Widen 8 bf16 (one uint4) to fp32 (exact).
__device__ __forceinline__ void bf16x8_to_f32(const uint4 v, float* out) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    out[2 * i] = __uint_as_float(w[i] << 16);
    out[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

// Load one 16-element block of x (bf16 or fp32) as fp32 with its sign masks.
template <bool kBF16>
__device__ __forceinline__ void load_block16(const void* base, size_t elem_off, Block16& blk) {
  if (kBF16) {
    const uint4* p = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(base) + elem_off);
    const uint4 a = __ldg(p), b = __ldg(p + 1);
    bf16x8_to_f32(a, blk.v);
    bf16x8_to_f32(b, blk.v + 8);
    blk.neg_lo = bf16x8_sign_nibbles(a.x, a.y, a.z, a.w);
    blk.neg_hi = bf16x8_sign_nibbles(b.x, b.y, b.z, b.w);
  } else {
    const float4* p = reinterpret_cast<const float4*>(static_cast<const float*>(base) + elem_off);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float4 a = __ldg(p + i);
      blk.v[4 * i] = a.x; blk.v[4 * i + 1] = a.y; blk.v[4 * i + 2] = a.z; blk.v[4 * i + 3] = a.w;
    }
    blk.neg_lo = f32x8_sign_nibbles(blk.v);
    blk.neg_hi = f32x8_sign_nibbles(blk.v + 8);
  }
}

// The same from shared memory (16-byte aligned rows).
template <bool kBF16>
__device__ __forceinline__ void load_block16_shared(const uint8_t* base, size_t elem_off, Block16& blk) {
  if (kBF16) {
    const uint4* q = reinterpret_cast<const uint4*>(base + elem_off * 2);
    const uint4 a = q[0], b = q[1];
    bf16x8_to_f32(a, blk.v);
    bf16x8_to_f32(b, blk.v + 8);
    blk.neg_lo = bf16x8_sign_nibbles(a.x, a.y, a.z, a.w);
    blk.neg_hi = bf16x8_sign_nibbles(b.x, b.y, b.z, b.w);
  } else {
    const float4* q = reinterpret_cast<const float4*>(base + elem_off * 4);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float4 a = q[i];
      blk.v[4 * i] = a.x; blk.v[4 * i + 1] = a.y; blk.v[4 * i + 2] = a.z; blk.v[4 * i + 3] = a.w;
    }
    blk.neg_lo = f32x8_sign_nibbles(blk.v);
    blk.neg_hi = f32x8_sign_nibbles(blk.v + 8);
  }
}

// Largest |x| bit pattern of a 16-byte vector: non-negative IEEE values order
// like unsigned integers, so the max is taken on the masked bits (exact).
template <bool kBF16>
__device__ __forceinline__ uint32_t absmax_bits16B(const uint4 v) {
  if (kBF16) {
    uint32_t m0, m1, m;
    asm("max.u16x2 %0, %1, %2;" : "=r"(m0) : "r"(v.x & 0x7FFF7FFFu), "r"(v.y & 0x7FFF7FFFu));
    asm("max.u16x2 %0, %1, %2;" : "=r"(m1) : "r"(v.z & 0x7FFF7FFFu), "r"(v.w & 0x7FFF7FFFu));
    asm("max.u16x2 %0, %1, %2;" : "=r"(m) : "r"(m0), "r"(m1));
    const uint32_t lo = m & 0xFFFFu, hi = m >> 16;
    return (lo > hi ? lo : hi) << 16;                   // as fp32 bits
  } else {
    const uint32_t a = max(v.x & 0x7FFFFFFFu, v.y & 0x7FFFFFFFu);
    const uint32_t b = max(v.z & 0x7FFFFFFFu, v.w & 0x7FFFFFFFu);
    return max(a, b);
  }
}

// Byte offset of scale (row r, block c) in the 128x4 tile layout (KB = D/16).
__device__ __forceinline__ size_t sf_tile_offset(int64_t r, int64_t c, int64_t KB) {
  const int64_t atom = (r >> 7) * (KB >> 2) + (c >> 2);
  return static_cast<size_t>(atom * 512 + (r & 31) * 16 + ((r & 127) >> 5) * 4 + (c & 3));
}

// ------------------------------------------------------------ router top-k
// Sorted (best first) list of the K best (key, id) pairs seen so far, with the
// unbiased score carried along.  Order: key descending, then id ascending.
__device__ __forceinline__ bool topk_better(float ka, int ia, float kb, int ib) {
  return ka > kb || (ka == kb && ia < ib);
}

// The epilogue's score: sigmoid(l) = 1 / (1 + exp(-l)), branch-free.
// exp(-l) = 2^t with t = -l*log2(e): t is split Cody-Waite style into its
// float32 rounding t_hi and the rounding error t_lo (computed exactly with a
// fused multiply-add plus the low part of log2(e)); 2^t_hi comes from the
// hardware base-2 exponential (ex2.approx, relative error about 2^-22) and
// 2^t ~= 2^t_hi * (1 + t_lo * ln 2).  The reciprocal uses the hardware
// approximation (__fdividef, within 2 ulp, 0 for a denominator above 2^126).
// The result is within a few ulp of the correctly rounded sigmoid for every
// float32 logit, exact at l = 0 (0.5) and equal to 1 once exp(-l) < 2^-25.
// Below -87 the result is 0 (the true sigmoid is below 2^-125; an infinite
// 2^t_hi would otherwise turn the correction into inf - inf = NaN).
// (W. J. Cody, W. Waite, Software Manual for the Elementary Functions, 1980:
// argument reduction with a split constant.)
__device__ __forceinline__ float sigmoid_f32(float l) {
  const bool tiny = l < -87.0f;
  l = tiny ? -87.0f : l;
  const float kLog2eHi = 1.44269502162933349609375f;      // RN(log2 e)
  const float kLog2eLo = 1.925963033500011079e-8f;        // log2 e - kLog2eHi
  const float t = __fmul_rn(-l, kLog2eHi);
  const float t_lo = __fadd_rn(__fmaf_rn(-l, kLog2eHi, -t), __fmul_rn(-l, kLog2eLo));
  float e;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(e) : "f"(t));
  e = __fmaf_rn(__fmul_rn(e, 0.693147180559945309f), t_lo, e);
  return tiny ? 0.0f : __fdividef(1.0f, __fadd_rn(1.0f, e));
}

// ------------------------------------------------- sorting-network helpers
// Compare-exchange of slots a and b of a (key, id, score) array so that slot a
// holds the better pair (key descending, then id ascending).
template <int N>
__device__ __forceinline__ void cswap(float (&k)[N], int (&i)[N], float (&s)[N], int a, int b) {
  const bool sw = topk_better(k[b], i[b], k[a], i[a]);
  const float tk = sw ? k[b] : k[a], ts = sw ? s[b] : s[a];
  const int ti = sw ? i[b] : i[a];
  k[b] = sw ? k[a] : k[b]; s[b] = sw ? s[a] : s[b]; i[b] = sw ? i[a] : i[b];
  k[a] = tk; s[a] = ts; i[a] = ti;
}

// Sort 8 pairs best-first with the optimal 19-comparator network
// (D. E. Knuth, The Art of Computer Programming vol. 3, section 5.3.4).
__device__ __forceinline__ void sort8(float (&k)[8], int (&i)[8], float (&s)[8]) {
  cswap(k, i, s, 0, 2); cswap(k, i, s, 1, 3); cswap(k, i, s, 4, 6); cswap(k, i, s, 5, 7);
  cswap(k, i, s, 0, 4); cswap(k, i, s, 1, 5); cswap(k, i, s, 2, 6); cswap(k, i, s, 3, 7);
  cswap(k, i, s, 0, 1); cswap(k, i, s, 2, 3); cswap(k, i, s, 4, 5); cswap(k, i, s, 6, 7);
  cswap(k, i, s, 2, 4); cswap(k, i, s, 3, 5);
  cswap(k, i, s, 1, 4); cswap(k, i, s, 3, 6);
  cswap(k, i, s, 1, 2); cswap(k, i, s, 3, 4); cswap(k, i, s, 5, 6);
}


template <int K>
struct TopK {
  float key[K];
  int id[K];
  float sc[K];

  __device__ __forceinline__ void init() {
#pragma unroll
    for (int i = 0; i < K; ++i) { key[i] = -INFINITY; id[i] = 0x7FFFFFFF; sc[i] = 0.0f; }
  }

  // Branch-free insertion (the list lives in registers): walking from the
  // bottom, slot j takes the entry above it when the new pair beats that
  // entry, the new pair when it beats only the current one, else keeps its own.
  __device__ __forceinline__ void push(float k, int i, float s) {
    if (!topk_better(k, i, key[K - 1], id[K - 1])) return;
#pragma unroll
    for (int j = K - 1; j > 0; --j) {
      const bool above = topk_better(k, i, key[j - 1], id[j - 1]);
      const bool here = topk_better(k, i, key[j], id[j]);
      key[j] = above ? key[j - 1] : (here ? k : key[j]);
      id[j] = above ? id[j - 1] : (here ? i : id[j]);
      sc[j] = above ? sc[j - 1] : (here ? s : sc[j]);
    }
    const bool top = topk_better(k, i, key[0], id[0]);
    key[0] = top ? k : key[0];
    id[0] = top ? i : id[0];
    sc[0] = top ? s : sc[0];
  }

  // Warp-uniform insertion: every lane of the warp must call it together
  // (no lane may have left the surrounding loop); lanes with valid == false
  // or a pair that does not qualify keep their list.  When no lane has
  // anything to insert the whole warp skips the work at once.
  __device__ __forceinline__ void push_if(float k, int i, float s, bool valid) {
    const bool ins = valid && topk_better(k, i, key[K - 1], id[K - 1]);
    if (!__any_sync(0xFFFFFFFFu, ins)) return;
#pragma unroll
    for (int j = K - 1; j > 0; --j) {
      const bool above = ins && topk_better(k, i, key[j - 1], id[j - 1]);
      const bool here = ins && topk_better(k, i, key[j], id[j]);
      key[j] = above ? key[j - 1] : (here ? k : key[j]);
      id[j] = above ? id[j - 1] : (here ? i : id[j]);
      sc[j] = above ? sc[j - 1] : (here ? s : sc[j]);
    }
    const bool top = ins && topk_better(k, i, key[0], id[0]);
    key[0] = top ? k : key[0];
    id[0] = top ? i : id[0];
    sc[0] = top ? s : sc[0];
  }

  // Replace the list by the best 8 of (list, b) where b is sorted best-first
  // (K == 8): the element-wise better of list[j] and b[7-j] is a bitonic
  // sequence holding the 8 best; a bitonic half-cleaner cascade sorts it.
  __device__ __forceinline__ void merge_sorted8(const float (&bk)[8], const int (&bi)[8],
                                                const float (&bs)[8]) {
    static_assert(K == 8, "merge_sorted8 needs an 8-entry list");
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const bool keep = topk_better(key[j], id[j], bk[7 - j], bi[7 - j]);
      key[j] = keep ? key[j] : bk[7 - j];
      id[j] = keep ? id[j] : bi[7 - j];
      sc[j] = keep ? sc[j] : bs[7 - j];
    }
#pragma unroll
    for (int d = 4; d > 0; d >>= 1) {
#pragma unroll
      for (int j = 0; j < 8; ++j)
        if ((j & d) == 0) cswap(key, id, sc, j, j + d);
    }
  }

  // The same for any power-of-two K: the element-wise better of list[j] and
  // b[K-1-j] is bitonic and holds the K best; log2(K) half-cleaner stages
  // sort it.
  __device__ __forceinline__ void merge_sorted(const float (&bk)[K], const int (&bi)[K], const float (&bs)[K]) {
    static_assert((K & (K - 1)) == 0, "merge_sorted needs a power-of-two list");
#pragma unroll
    for (int j = 0; j < K; ++j) {
      const bool keep = topk_better(key[j], id[j], bk[K - 1 - j], bi[K - 1 - j]);
      key[j] = keep ? key[j] : bk[K - 1 - j];
      id[j] = keep ? id[j] : bi[K - 1 - j];
      sc[j] = keep ? sc[j] : bs[K - 1 - j];
    }
#pragma unroll
    for (int d = K / 2; d > 0; d >>= 1) {
#pragma unroll
      for (int j = 0; j < K; ++j)
        if ((j & d) == 0) cswap(key, id, sc, j, j + d);
    }
  }

  // Drop the best entry (shift the list up by one; the tail becomes empty).
  __device__ __forceinline__ void pop_front() {
#pragma unroll
    for (int j = 0; j < K - 1; ++j) { key[j] = key[j + 1]; id[j] = id[j + 1]; sc[j] = sc[j + 1]; }
    key[K - 1] = -INFINITY;
    id[K - 1] = 0x7FFFFFFF;
    sc[K - 1] = 0.0f;
  }
};

}  // namespace nvr
