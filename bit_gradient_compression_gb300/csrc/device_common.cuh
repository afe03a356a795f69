// Device helpers shared by the sender and receiver kernels.
//
// All arithmetic that decides a stored value uses the explicit round-to-
// nearest intrinsics (__fadd_rn, __fmul_rn, __fdiv_rn, __fsqrt_rn): they are
// never contracted into fused multiply-adds, and the library is also built
// with -fmad=false, so every product and sum is rounded on its own as the
// method's fp32 definition states.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "loco_internal.h"

namespace loco {

// Adding 1.5 * 2^23 to a float in [-2^22, 2^22] rounds it to an integer (halves
// to even under round-to-nearest) and leaves that integer, offset by
// 0x4B400000, in the low mantissa bits.  Subtracting the constant back gives
// the integer as a float exactly.
constexpr float kRoundMagic = 12582912.0f;  // 1.5 * 2^23

// Float with bits 0x4B000000 | u (u < 2^23) is 2^23 + u exactly.
constexpr uint32_t kTwo23Bits = 0x4B000000u;

__device__ __forceinline__ float bf16lo_to_f32(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi_to_f32(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Streaming loads/stores: data is touched once, keep it out of L1 and mark it
// evict-first in L2.
__device__ __forceinline__ float4 ld_stream(const float4* p) { return __ldcs(p); }
__device__ __forceinline__ uint4 ld_stream(const uint4* p) { return __ldcs(p); }
__device__ __forceinline__ uint2 ld_stream(const uint2* p) { return __ldcs(p); }
__device__ __forceinline__ uint32_t ld_stream(const uint32_t* p) { return __ldcs(p); }
__device__ __forceinline__ void st_stream(float4* p, float4 v) { __stcs(p, v); }
__device__ __forceinline__ void st_stream(uint2* p, uint2 v) { __stcs(p, v); }
__device__ __forceinline__ void st_stream(uint32_t* p, uint32_t v) { __stcs(p, v); }

// Decode the 8 codes of one 8-element chunk into floats q (exact integers).
//  4 bit: one 32-bit word, element j in nibble j (two's complement).
//  8 bit: two 32-bit words, element j in byte j.
// XOR with the sign bit of each field turns two's complement into an offset
// code (q + 8 or q + 128); OR-ing that under the exponent of 2^23 and
// subtracting 2^23 + offset gives q exactly.
template <int BITS>
struct ChunkCodes;

template <>
struct ChunkCodes<4> {
  uint32_t w;
  __device__ __forceinline__ void load(const uint8_t* base, int64_t e0) {
    w = ld_stream(reinterpret_cast<const uint32_t*>(base + (e0 >> 1)));
  }
  __device__ __forceinline__ void decode(float q[8]) const {
    const uint32_t u = w ^ 0x88888888u;
#pragma unroll
    for (int j = 0; j < 8; ++j)
      q[j] = __fsub_rn(__uint_as_float(kTwo23Bits | ((u >> (4 * j)) & 0xFu)), 8388616.0f);
  }
};

template <>
struct ChunkCodes<8> {
  uint2 w;
  __device__ __forceinline__ void load(const uint8_t* base, int64_t e0) {
    w = ld_stream(reinterpret_cast<const uint2*>(base + e0));
  }
  __device__ __forceinline__ void decode(float q[8]) const {
    const uint32_t u0 = w.x ^ 0x80808080u, u1 = w.y ^ 0x80808080u;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      q[j] = __fsub_rn(__uint_as_float(kTwo23Bits | ((u0 >> (8 * j)) & 0xFFu)), 8388736.0f);
      q[j + 4] = __fsub_rn(__uint_as_float(kTwo23Bits | ((u1 >> (8 * j)) & 0xFFu)), 8388736.0f);
    }
  }
};

// Division by W: for a power of two, multiplying by the exact reciprocal gives
// the same correctly rounded quotient; otherwise an IEEE division.
template <int W>
__device__ __forceinline__ float div_by_ranks(float x) {
  if constexpr ((W & (W - 1)) == 0) {
    return __fmul_rn(x, 1.0f / float(W));
  } else {
    return __fdiv_rn(x, float(W));
  }
}

// Per-element fp32 rank average of Eqn (8), in rank order 0..W-1.
template <int BITS, int W>
__device__ __forceinline__ void decode_mean8(const RankPtrs& rp, int64_t e0, int64_t blk, float out[8]) {
  ChunkCodes<BITS> cw[W];
  float s[W];
#pragma unroll
  for (int w = 0; w < W; ++w) {
    cw[w].load(rp.codes[w], e0);
    s[w] = __ldg(rp.scales[w] + blk);
  }
  float acc[8];
#pragma unroll
  for (int w = 0; w < W; ++w) {
    float q[8];
    cw[w].decode(q);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const float d = __fmul_rn(q[j], s[w]);
      acc[j] = (w == 0) ? d : __fadd_rn(acc[j], d);
    }
  }
#pragma unroll
  for (int j = 0; j < 8; ++j) out[j] = div_by_ranks<W>(acc[j]);
}

}  // namespace loco
