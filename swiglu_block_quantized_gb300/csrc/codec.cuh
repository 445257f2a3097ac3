// codec.cuh -- device-side decoding of Q4_0, Q8_0, PrismML Q2_0 and MLX
// 4-bit affine blocks into fp16 weights.
//
// Codecs (m4-prefill-engine "Releases" page, v0.3.0 and v0.2.3; GGUF for the
// byte layout of Q4_0 / Q8_0):
//   Q4_0  32 weights, 18 B: fp16 d, 16 B of nibbles  w = (q - 8) * d
//   Q8_0  32 weights, 34 B: fp16 d, 32 signed bytes  w = q * d
//   Q2_0 128 weights, 34 B: fp16 d, 32 B of 2-bit codes, w = (q - 1) * d,
//         the reserved code 3 giving +2d.
//   MLX4  32 weights, 20 B: fp16 scale s, fp16 bias b, 16 B of nibbles
//         (code 2i in the low nibble of byte i), w = q * s + b (project page
//         section 4 and Table B: the 20-byte block_mlx_4bit; group size 32).
//
// Every weight is produced with exactly one rounding: the code is placed in
// the fraction field of an fp16 whose exponent makes one fraction step worth
// 1 (so the fp16 holds bias + q exactly), the bias is subtracted exactly with
// an fp16 subtract (the difference is a small integer), and the integer is
// multiplied by d with one round-to-nearest-even fp16 multiply.  The result is
// therefore RNE((q - z) * d), bit for bit, including subnormals and -0.
// MLX4 recovers q the same way and finishes with one fused multiply-add,
// RNE(q * s + b).
//
// A "packed stage" is 8 consecutive blocks of one weight row: 144 B (Q4_0),
// 272 B (Q8_0, Q2_0), 160 B (MLX4), a multiple of 16 bytes so that TMA can
// move it.  It covers KP = 256 (Q4_0, Q8_0, MLX4) or 1024 (Q2_0) weights,
// split into SUB sub-steps of 64 weights each.
#pragma once

#include "common.cuh"

namespace m4q {

template <int C>
struct CodecTraits;

template <>
struct CodecTraits<kQ4_0> {
  static constexpr int B = 32, BB = 18;
};
template <>
struct CodecTraits<kQ8_0> {
  static constexpr int B = 32, BB = 34;
};
template <>
struct CodecTraits<kQ2_0> {
  static constexpr int B = 128, BB = 34;
};
template <>
struct CodecTraits<kMLX4> {
  static constexpr int B = 32, BB = 20;
};

template <int C>
struct Stage {
  static constexpr int B = CodecTraits<C>::B;
  static constexpr int BB = CodecTraits<C>::BB;
  static constexpr int KP = 8 * B;          // weights per packed stage
  static constexpr int KPB = 8 * BB;        // bytes per packed stage (row)
  static constexpr int WORDS = KPB / 4;     // 32-bit words per packed stage
  static constexpr int SUB = KP / 64;       // 64-weight sub-steps per stage
  static_assert(KPB % 16 == 0, "packed stage must be a multiple of 16 bytes");
};

// fp16x2 arithmetic with explicit round-to-nearest-even (never contracted).
__device__ __forceinline__ uint32_t hsub2_rn(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}
__device__ __forceinline__ uint32_t hmul2_rn(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

// a * b + c with one round-to-nearest-even (fused).
__device__ __forceinline__ uint32_t hfma2_rn(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t r;
  asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(c));
  return r;
}

// 16-bit value at an even byte offset of a register-resident byte string.
__device__ __forceinline__ uint32_t u16_at(const uint32_t* w, int off) {
  return (off & 2) ? (w[off >> 2] >> 16) : (w[off >> 2] & 0xFFFFu);
}

// Bytes (off, off+1), off even, spread to [b0, 0, b1, 0].
__device__ __forceinline__ uint32_t spread_pair(const uint32_t* w, int off) {
  return __byte_perm(w[off >> 2], 0u, (off & 2) ? 0x4342u : 0x4140u);
}

// Byte off replicated to [b, 0, b, 0].
__device__ __forceinline__ uint32_t spread_byte(const uint32_t* w, int off) {
  const uint32_t b = (uint32_t)(off & 3);
  return __byte_perm(w[off >> 2], 0u, 0x4040u | (b << 8) | b);
}

// The low half of `dbits` in both halves (a scale or bias for fp16x2 math).
__device__ __forceinline__ uint32_t dup_scale(uint32_t dbits) { return __byte_perm(dbits, 0u, 0x1010u); }

// Biased fp16x2 constants of the decoders, held in registers.  Each code is
// placed with one three-input logic operation, (x & mask) | bias, whose
// mask is its immediate operand; the instruction takes one immediate only,
// and a bias that the compiler sees as a constant makes it split the
// operation in two, so the biases come from an opaque move, once per thread.
// 0x6400 = 1024 (a fraction step of 1 at bit 0), 0x5C00 = 256 (step 1 at
// bit 2), 0x5400 = 64 (bit 4), 0x4C00 = 16 (bit 6).
struct DecK {
  uint32_t b6464;  // (1024, 1024)
  uint32_t b5454;  // (64, 64)
  uint32_t b5c64;  // (1024, 256)  Q2_0 codes 0 and 1 of a byte
  uint32_t b4c54;  // (64, 16)     Q2_0 codes 2 and 3
  uint32_t b5464;  // (1024, 64)   MLX4 low and high nibble of a byte
  uint32_t bff00;  // 0xFF00FF00: Q8_0 bytes of a whole word (see q8_word)
};

__device__ __forceinline__ DecK make_deck() {
  DecK k;
  asm volatile("mov.b32 %0, 0x64006400;" : "=r"(k.b6464));
  asm volatile("mov.b32 %0, 0x54005400;" : "=r"(k.b5454));
  asm volatile("mov.b32 %0, 0x5C006400;" : "=r"(k.b5c64));
  asm volatile("mov.b32 %0, 0x4C005400;" : "=r"(k.b4c54));
  asm volatile("mov.b32 %0, 0x54006400;" : "=r"(k.b5464));
  asm volatile("mov.b32 %0, 0xFF00FF00;" : "=r"(k.bff00));
  return k;
}

// (a & MASK) | c in one instruction.
template <uint32_t MASK>
__device__ __forceinline__ uint32_t and_or(uint32_t a, uint32_t c) {
  uint32_t d;
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(a), "n"(MASK), "r"(c));
  return d;
}
// (a ^ X) | c in one instruction.
template <uint32_t X>
__device__ __forceinline__ uint32_t xor_or(uint32_t a, uint32_t c) {
  uint32_t d;
  asm("lop3.b32 %0, %1, %2, %3, 0xBE;" : "=r"(d) : "r"(a), "n"(X), "r"(c));
  return d;
}

// Q4_0 bytes [b0, 0, b1, 0]: low nibbles -> 1024 + q; high nibbles -> 64 + q.
__device__ __forceinline__ void q4_pair(uint32_t t, uint32_t d2, const DecK& K, uint32_t& lo, uint32_t& hi) {
  lo = hmul2_rn(hsub2_rn(and_or<0x000F000Fu>(t, K.b6464), 0x64086408u), d2);  // - 1032
  hi = hmul2_rn(hsub2_rn(and_or<0x00F000F0u>(t, K.b5454), 0x54805480u), d2);  // - 72
}
// Q8_0 signed bytes [b0, 0, b1, 0]: (q ^ 0x80) = q + 128 -> 1024 + 128 + q.
__device__ __forceinline__ uint32_t q8_pair(uint32_t t, uint32_t d2, const DecK& K) {
  return hmul2_rn(hsub2_rn(xor_or<0x00800080u>(t, K.b6464), 0x64806480u), d2);  // - 1152
}
// Q2_0 byte [v,0,v,0]: codes at bits 0-1, 2-3 -> (1024 + q0, 256 + q1);
// bits 4-5, 6-7 -> (64 + q2, 16 + q3).
__device__ __forceinline__ void q2_byte(uint32_t t, uint32_t d2, const DecK& K, uint32_t& p01, uint32_t& p23) {
  p01 = hmul2_rn(hsub2_rn(and_or<0x000C0003u>(t, K.b5c64), 0x5C046401u), d2);  // -(257, 1025)
  p23 = hmul2_rn(hsub2_rn(and_or<0x00C00030u>(t, K.b4c54), 0x4C405410u), d2);  // -(17, 65)
}

// MLX4 byte [v,0,v,0]: low nibble -> 1024 + q0, high nibble -> 64 + q1;
// subtract the biases exactly, then one fused q * s + b per half.
__device__ __forceinline__ uint32_t mlx_pair(uint32_t t, uint32_t s2, uint32_t b2, const DecK& K) {
  return hfma2_rn(hsub2_rn(and_or<0x00F0000Fu>(t, K.b5464), 0x54006400u), s2, b2);
}

// Whole-word decoders: the four bytes [b0 b1 b2 b3] of one 32-bit word of
// codes, without a byte permute per pair.  The fp16x2 results pair the
// weights of bytes (0, 2) and (1, 3); the caller pairs the activations the
// same way.
// Q4_0: l02 = low nibbles of b0, b2; h02 = high nibbles; l13, h13 for b1, b3.
__device__ __forceinline__ void q4_word(uint32_t w, uint32_t d2, const DecK& K, uint32_t& l02, uint32_t& l13,
                                        uint32_t& h02, uint32_t& h13) {
  const uint32_t v = w >> 8;
  l02 = hmul2_rn(hsub2_rn(and_or<0x000F000Fu>(w, K.b6464), 0x64086408u), d2);
  h02 = hmul2_rn(hsub2_rn(and_or<0x00F000F0u>(w, K.b5454), 0x54805480u), d2);
  l13 = hmul2_rn(hsub2_rn(and_or<0x000F000Fu>(v, K.b6464), 0x64086408u), d2);
  h13 = hmul2_rn(hsub2_rn(and_or<0x00F000F0u>(v, K.b5454), 0x54805480u), d2);
}
// Q8_0: p02 = signed bytes b0, b2; p13 = b1, b3.  One logic operation keeps
// the low byte of each half, flips its bit 7 and sets the exponent:
// ((w & 0x00FF00FF) ^ 0x00800080) | 0x64006400, written as the lookup 0x36
// over (w, 0x9B809B80, 0xFF00FF00): where the third operand is 0 the bit is
// w's, flipped where the second is 1; elsewhere it is the complement of the
// second operand (which holds the complement of the exponent bits).
__device__ __forceinline__ uint32_t q8_bytes02(uint32_t w, const DecK& K) {
  uint32_t d;
  asm("lop3.b32 %0, %1, %2, %3, 0x36;" : "=r"(d) : "r"(w), "n"(0x9B809B80u), "r"(K.bff00));
  return d;
}
__device__ __forceinline__ void q8_word(uint32_t w, uint32_t d2, const DecK& K, uint32_t& p02, uint32_t& p13) {
  p02 = hmul2_rn(hsub2_rn(q8_bytes02(w, K), 0x64806480u), d2);
  p13 = hmul2_rn(hsub2_rn(q8_bytes02(w >> 8, K), 0x64806480u), d2);
}
// MLX4: byte i holds codes 2i (low nibble) and 2i + 1; lo02 = codes of the
// low nibbles of b0, b2, hi02 their high nibbles, lo13 / hi13 for b1, b3.
__device__ __forceinline__ void mlx_word(uint32_t w, uint32_t s2, uint32_t b2, const DecK& K, uint32_t& lo02,
                                         uint32_t& hi02, uint32_t& lo13, uint32_t& hi13) {
  const uint32_t v = w >> 8;
  lo02 = hfma2_rn(hsub2_rn(and_or<0x000F000Fu>(w, K.b6464), 0x64006400u), s2, b2);
  hi02 = hfma2_rn(hsub2_rn(and_or<0x00F000F0u>(w, K.b5454), 0x54005400u), s2, b2);
  lo13 = hfma2_rn(hsub2_rn(and_or<0x000F000Fu>(v, K.b6464), 0x64006400u), s2, b2);
  hi13 = hfma2_rn(hsub2_rn(and_or<0x00F000F0u>(v, K.b5454), 0x54005400u), s2, b2);
}

// MLX4 scale and bias of the block at even byte offset bo, each duplicated
// into both halves.
__device__ __forceinline__ void mlx_scale_bias(const uint32_t* w, int bo, uint32_t& s2, uint32_t& b2) {
  s2 = dup_scale(u16_at(w, bo));
  b2 = dup_scale(u16_at(w, bo + 2));
}

// Decode sub-step j (weights 64j .. 64j+63 of a packed stage) of one row
// into out[i] = fp16x2 (w[64j + 2i], w[64j + 2i + 1]).  `w` holds the row's
// packed stage bytes; j must be a compile-time constant after unrolling.
template <int C>
__device__ __forceinline__ void decode_sub(const uint32_t* w, int j, uint32_t (&out)[32], const DecK& K);

template <>
__device__ __forceinline__ void decode_sub<kQ4_0>(const uint32_t* w, int j, uint32_t (&out)[32],
                                              const DecK& K) {
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int bo = (2 * j + h) * 18;
    const uint32_t d2 = dup_scale(u16_at(w, bo));
#pragma unroll
    for (int p = 0; p < 8; ++p) {
      uint32_t lo, hi;
      q4_pair(spread_pair(w, bo + 2 + 2 * p), d2, K, lo, hi);
      out[16 * h + p] = lo;      // weights 2p, 2p+1 of the block
      out[16 * h + 8 + p] = hi;  // weights 16+2p, 17+2p
    }
  }
}

template <>
__device__ __forceinline__ void decode_sub<kQ8_0>(const uint32_t* w, int j, uint32_t (&out)[32],
                                              const DecK& K) {
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int bo = (2 * j + h) * 34;
    const uint32_t d2 = dup_scale(u16_at(w, bo));
#pragma unroll
    for (int p = 0; p < 16; ++p) out[16 * h + p] = q8_pair(spread_pair(w, bo + 2 + 2 * p), d2, K);
  }
}

template <>
__device__ __forceinline__ void decode_sub<kMLX4>(const uint32_t* w, int j, uint32_t (&out)[32],
                                              const DecK& K) {
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int bo = (2 * j + h) * 20;
    uint32_t s2, b2;
    mlx_scale_bias(w, bo, s2, b2);
#pragma unroll
    for (int p = 0; p < 16; ++p) out[16 * h + p] = mlx_pair(spread_byte(w, bo + 4 + p), s2, b2, K);
  }
}

template <>
__device__ __forceinline__ void decode_sub<kQ2_0>(const uint32_t* w, int j, uint32_t (&out)[32],
                                              const DecK& K) {
  const int bo = (j >> 1) * 34;
  const int cb = bo + 2 + 16 * (j & 1);  // first code byte of this half block
  const uint32_t d2 = dup_scale(u16_at(w, bo));
#pragma unroll
  for (int c = 0; c < 16; ++c) {
    uint32_t p01, p23;
    q2_byte(spread_byte(w, cb + c), d2, K, p01, p23);
    out[2 * c] = p01;
    out[2 * c + 1] = p23;
  }
}

// Half g (0 or 1) of sub-step j: out[i] = fp16x2 (w[64j + 32g + 2i],
// w[64j + 32g + 2i + 1]), i < 16.  j and g must be compile-time constants
// after unrolling.
template <int C, int G>
__device__ __forceinline__ void decode_half(const uint32_t* w, int j, uint32_t (&out)[16], const DecK& K) {
  if constexpr (C == kQ4_0) {
    const int bo = (2 * j + G) * 18;  // block 2j + G
    const uint32_t d2 = dup_scale(u16_at(w, bo));
#pragma unroll
    for (int p = 0; p < 8; ++p) {
      uint32_t lo, hi;
      q4_pair(spread_pair(w, bo + 2 + 2 * p), d2, K, lo, hi);
      out[p] = lo;
      out[8 + p] = hi;
    }
  } else if constexpr (C == kQ8_0) {
    const int bo = (2 * j + G) * 34;
    const uint32_t d2 = dup_scale(u16_at(w, bo));
#pragma unroll
    for (int p = 0; p < 16; ++p) out[p] = q8_pair(spread_pair(w, bo + 2 + 2 * p), d2, K);
  } else if constexpr (C == kMLX4) {
    const int bo = (2 * j + G) * 20;
    uint32_t s2, b2;
    mlx_scale_bias(w, bo, s2, b2);
#pragma unroll
    for (int p = 0; p < 16; ++p) out[p] = mlx_pair(spread_byte(w, bo + 4 + p), s2, b2, K);
  } else {
    const int bo = (j >> 1) * 34;
    const int cb = bo + 2 + 16 * (j & 1) + 8 * G;  // 8 code bytes = 32 weights
    const uint32_t d2 = dup_scale(u16_at(w, bo));
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      uint32_t p01, p23;
      q2_byte(spread_byte(w, cb + c), d2, K, p01, p23);
      out[2 * c] = p01;
      out[2 * c + 1] = p23;
    }
  }
}

}  // namespace m4q
