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
__device__ __forceinline__ void st_stream(uint4* p, uint4 v) { __stcs(p, v); }
__device__ __forceinline__ void st_stream(uint2* p, uint2 v) { __stcs(p, v); }
__device__ __forceinline__ void st_stream(uint32_t* p, uint32_t v) { __stcs(p, v); }

// ---------------------------------------------------------------------------
// Asynchronous global -> shared copies (cp.async, 16 bytes per instruction).
// Completion is tracked per thread by commit groups and waited for with the
// hardware cp.async.wait_group; a block barrier then makes every thread's
// copies visible to the others (see pipeline_tiles).  The bytes in flight live
// in shared memory instead of registers, and no thread spins on a flag.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(dst)), "l"(src) : "memory");
}
// 8-byte copy (cached in L1 on the way), both addresses 8-byte aligned.
__device__ __forceinline__ void cp_async8(void* dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(smem_addr(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Bulk (TMA) copy shared -> global of `bytes` (a multiple of 16, both
// addresses 16-byte aligned), issued by one thread.  Completion is tracked by
// bulk groups and waited for with the hardware wait_group instruction.
__device__ __forceinline__ void fence_smem_to_async_proxy() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void bulk_store(void* gdst, const void* ssrc, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(gdst), "r"(smem_addr(ssrc)),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// The shared-memory source of every committed bulk store has been read.
__device__ __forceinline__ void bulk_wait_read_all() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
// The shared-memory source of every committed bulk store but the newest N has been read.
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}
// Every committed bulk store has completed.
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// ---------------------------------------------------------------------------
// Multistage tile pipeline.  The CTA walks tiles blockIdx.x, blockIdx.x +
// gridDim.x, ...; S-1 tiles are in flight (cp.async into their own stage of
// shared memory) while one is consumed.  cp.async.wait_group plus
// __syncthreads make a tile visible to every thread, and the second
// __syncthreads keeps a stage from being refilled before every thread is done
// with it.  Both barriers are reached by all threads of the CTA (the loop
// bounds are uniform), and there is no spin-wait anywhere.
//   issue(stage_base, tile): start the copies of one tile (each thread its share)
//   body(stage_base, tile):  consume one staged tile
// ---------------------------------------------------------------------------
template <int S, typename Issue, typename Body, typename Before, typename After>
__device__ __forceinline__ void pipeline_tiles(uint8_t* sm, size_t stage_bytes, int64_t ntiles, Issue issue, Body body,
                                               Before before, After after) {
#pragma unroll
  for (int s = 0; s < S - 1; ++s) {
    const int64_t tile = blockIdx.x + int64_t(s) * gridDim.x;
    if (tile < ntiles) issue(sm + s * stage_bytes, tile);
    cp_async_commit();
  }
  int cur = 0;
  for (int64_t tile = blockIdx.x; tile < ntiles; tile += gridDim.x) {
    const int64_t ahead = tile + int64_t(S - 1) * gridDim.x;
    const int nxt = (cur == 0) ? S - 1 : cur - 1;
    if (ahead < ntiles) issue(sm + nxt * stage_bytes, ahead);
    cp_async_commit();
    cp_async_wait<S - 1>();
    before(tile);  // runs before the barrier that publishes the tile
    __syncthreads();
    body(sm + cur * stage_bytes, tile);
    __syncthreads();
    after(tile);   // runs after every thread has finished the tile
    cur = (cur + 1 == S) ? 0 : cur + 1;
  }
  cp_async_wait<0>();
}

// Variant for kernels that write a tile's results back into its own stage
// and ship them with bulk (TMA) stores issued by thread 0 (`flush`).  A
// stage is refilled only after those stores have read it: thread 0 waits for
// the reads before the barrier that opens each tile, and the refill copies
// are issued after that barrier.  The tile consumed at step k lives in stage
// k mod S; the refill at step k goes to the previous tile's stage, S-1 tiles
// ahead, so S-1 tiles are in flight as in pipeline_tiles.  Hardware waits
// only, every barrier reached by all threads.
//   flush(stage_base, tile): (thread 0) bulk stores of the tile's results + commit
template <int S, typename Issue, typename Body, typename Flush>
__device__ __forceinline__ void pipeline_tiles_inplace(uint8_t* sm, size_t stage_bytes, int64_t ntiles, Issue issue,
                                                       Body body, Flush flush) {
  static_assert(S >= 2, "one stage computes while the next loads");
  const bool leader = threadIdx.x == 0;
#pragma unroll
  for (int s = 0; s < S - 1; ++s) {
    const int64_t tile = blockIdx.x + int64_t(s) * gridDim.x;
    if (tile < ntiles) issue(sm + s * stage_bytes, tile);
    cp_async_commit();
  }
  int cur = 0;
  for (int64_t tile = blockIdx.x; tile < ntiles; tile += gridDim.x) {
    cp_async_wait<S - 2>();                // this tile's copies have landed
    if (leader) bulk_wait_read_all();      // the previous tile's results have left its stage
    __syncthreads();
    const int prev = (cur == 0) ? S - 1 : cur - 1;
    const int64_t ahead = tile + int64_t(S - 1) * gridDim.x;
    if (ahead < ntiles) issue(sm + prev * stage_bytes, ahead);
    cp_async_commit();
    body(sm + cur * stage_bytes, tile);
    fence_smem_to_async_proxy();           // this thread's results visible to the bulk copy
    __syncthreads();
    if (leader) flush(sm + cur * stage_bytes, tile);
    cur = (cur + 1 == S) ? 0 : cur + 1;
  }
  cp_async_wait<0>();
  if (leader) bulk_wait_all();
}

template <int S, typename Issue, typename Body>
__device__ __forceinline__ void pipeline_tiles(uint8_t* sm, size_t stage_bytes, int64_t ntiles, Issue issue,
                                               Body body) {
  pipeline_tiles<S>(sm, stage_bytes, ntiles, issue, body, [](int64_t) {}, [](int64_t) {});
}

// ---------------------------------------------------------------------------
// Warp-local multistage pipeline.  Warp gw of nw walks its own tiles gw,
// gw + nw, ... (or, with G > 1, groups of G consecutive tiles: G gw ..
// G gw + G-1, then the group nw further on) through S stages of its own shared
// memory (wsm), S-1 tiles in flight while one is consumed.  The warp's lanes
// copy a tile together (cp.async), so cp.async.wait_group (each lane's own
// copies landed) plus __syncwarp (memory ordering among the warp's lanes) make
// it visible to every lane; the __syncwarp also guarantees that the stage
// refilled next, the one consumed in the previous iteration, is no longer
// being read.  No CTA-wide barrier and no spin-wait: warps of a CTA drift
// freely.  Every lane of the warp must run this with the same arguments.
//   issue(stage_base, tile): start this lane's share of the tile's copies
//   body(stage_base, tile):  consume one staged tile
// ---------------------------------------------------------------------------
template <int S, int G = 1, typename Issue, typename Body>
__device__ __forceinline__ void warp_pipeline(uint8_t* wsm, size_t stage_bytes, int64_t gw, int64_t nw, int64_t ntiles,
                                              Issue issue, Body body) {
  static_assert(S >= 2, "one stage computes while the next loads");
  if constexpr (G > 1) {
    static_assert((G & (G - 1)) == 0, "a power-of-two group");
    // this warp's j-th tile
    auto tile_of = [&](int64_t j) { return (gw + (j / G) * nw) * G + (j % G); };
#pragma unroll
    for (int s = 0; s < S - 1; ++s) {
      const int64_t tile = tile_of(s);
      if (tile < ntiles) issue(wsm + s * stage_bytes, tile);
      cp_async_commit();
    }
    int cur = 0;
    for (int64_t j = 0;; ++j) {
      const int64_t tile = tile_of(j);
      if (tile >= ntiles) break;
      cp_async_wait<S - 2>();
      __syncwarp();
      const int prev = (cur == 0) ? S - 1 : cur - 1;
      const int64_t ahead = tile_of(j + S - 1);
      if (ahead < ntiles) issue(wsm + prev * stage_bytes, ahead);
      cp_async_commit();
      body(wsm + cur * stage_bytes, tile);
      cur = (cur + 1 == S) ? 0 : cur + 1;
    }
    cp_async_wait<0>();
  } else {
#pragma unroll
    for (int s = 0; s < S - 1; ++s) {
      const int64_t tile = gw + int64_t(s) * nw;
      if (tile < ntiles) issue(wsm + s * stage_bytes, tile);
      cp_async_commit();
    }
    int cur = 0;
    for (int64_t tile = gw; tile < ntiles; tile += nw) {
      cp_async_wait<S - 2>();  // this lane's copies of `tile` have landed
      __syncwarp();            // ... and every other lane's; the previous stage is free
      const int prev = (cur == 0) ? S - 1 : cur - 1;
      const int64_t ahead = tile + int64_t(S - 1) * nw;
      if (ahead < ntiles) issue(wsm + prev * stage_bytes, ahead);
      cp_async_commit();
      body(wsm + cur * stage_bytes, tile);
      cur = (cur + 1 == S) ? 0 : cur + 1;
    }
    cp_async_wait<0>();
  }
}

// ---------------------------------------------------------------------------
// Packed fp32 pairs.  add.rn.f32x2 / mul.rn.f32x2 / fma.rn.f32x2 (sm_100+)
// each round every lane exactly like the scalar instruction and issue once per
// pair.  A packed multiply whose result feeds a packed add, however, was
// measured to be combined into a single fused multiply-add (one rounding) by
// the code generator even with .rn and -fmad=false.  Where a product feeds a
// sum, it is therefore formed as fma(a, b, z) with z = -0.0 read at run time:
// a + (-0) = a for every a (including +0 and -0 under round-to-nearest), so
// the result is the rounded product, and since z is not known when the code is
// generated the fma can be neither turned back into a multiply nor merged
// with the add that follows.  mul2 is used only where no add consumes it.
// ---------------------------------------------------------------------------
typedef unsigned long long f32x2;

__device__ __forceinline__ f32x2 pk2(float lo, float hi) {
  f32x2 r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ f32x2 pk2u(uint32_t lo, uint32_t hi) {
  f32x2 r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "r"(lo), "r"(hi));
  return r;
}
__device__ __forceinline__ void upk2(f32x2 v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ f32x2 add2(f32x2 a, f32x2 b) {
  f32x2 r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ f32x2 mul2(f32x2 a, f32x2 b) {
  f32x2 r;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ f32x2 sub2(f32x2 a, f32x2 b) {
  f32x2 r;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
// Rounded product a * b per lane; neg_zero2 must hold (-0.0f, -0.0f) at run time.
__device__ __forceinline__ f32x2 prod2(f32x2 a, f32x2 b, f32x2 neg_zero2) {
  f32x2 r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(neg_zero2));
  return r;
}

// ---------------------------------------------------------------------------
// Codes of one E-element chunk of one rank (E*BITS/8 bytes: one 4- or 8-byte
// load), decoded to packed pairs of exact floats f32(q).
//
// XOR with the sign bit of every field turns two's complement into the offset
// code q + 2^(p-1); a byte permute places that byte under the exponent of 2^23
// (bits 0x4B0000xx = 2^23 + xx exactly), and one packed subtraction of
// 2^23 + 2^(p-1) leaves q.  4-bit fields are first split into the even and
// odd nibbles of each byte so every element is one byte.
// ---------------------------------------------------------------------------
template <int BITS, int E>
struct ChunkCodes {
  static constexpr int kWords = E * BITS / 32;  // 32-bit words per rank
  static_assert(kWords == 1 || kWords == 2 || kWords == 4, "one 4-, 8- or 16-byte load per rank");
  uint32_t w[kWords];

  static constexpr int kBytes = kWords * 4;

  __device__ __forceinline__ void load(const uint8_t* base, int64_t e0) {
    const uint8_t* p = base + (e0 * BITS >> 3);
    if constexpr (kWords == 1) {
      w[0] = ld_stream(reinterpret_cast<const uint32_t*>(p));
    } else if constexpr (kWords == 2) {
      const uint2 v = ld_stream(reinterpret_cast<const uint2*>(p));
      w[0] = v.x;
      w[1] = v.y;
    } else {
      const uint4 v = ld_stream(reinterpret_cast<const uint4*>(p));
      w[0] = v.x;
      w[1] = v.y;
      w[2] = v.z;
      w[3] = v.w;
    }
  }

  __device__ __forceinline__ void load_shared(const uint8_t* src) {
    if constexpr (kWords == 1) {
      w[0] = *reinterpret_cast<const uint32_t*>(src);
    } else if constexpr (kWords == 2) {
      const uint2 v = *reinterpret_cast<const uint2*>(src);
      w[0] = v.x;
      w[1] = v.y;
    } else {
      const uint4 v = *reinterpret_cast<const uint4*>(src);
      w[0] = v.x;
      w[1] = v.y;
      w[2] = v.z;
      w[3] = v.w;
    }
  }

  // Elements held by pair j of decode().
  __host__ __device__ static constexpr int pair_lo(int j) { return 2 * j; }
  __host__ __device__ static constexpr int pair_hi(int j) { return 2 * j + 1; }

  // q2[j] holds elements (pair_lo(j), pair_hi(j)) as floats q exactly.
  __device__ __forceinline__ void decode(f32x2 q2[E / 2]) const {
    constexpr uint32_t K = 0x4B000000u;
    if constexpr (BITS == 4) {
      const f32x2 off = pk2(-8388616.0f, -8388616.0f);  // -(2^23 + 8)
#pragma unroll
      for (int i = 0; i < kWords; ++i) {
        const uint32_t u = w[i] ^ 0x88888888u;
        const uint32_t ev = u & 0x0F0F0F0Fu;          // nibbles 0,2,4,6 -> bytes 0..3
        const uint32_t od = (u >> 4) & 0x0F0F0F0Fu;   // nibbles 1,3,5,7 -> bytes 0..3
#pragma unroll
        for (int k = 0; k < 4; ++k)
          q2[4 * i + k] = add2(pk2u(__byte_perm(ev, K, 0x7440 | k), __byte_perm(od, K, 0x7440 | k)), off);
      }
    } else {
      const f32x2 off = pk2(-8388736.0f, -8388736.0f);  // -(2^23 + 128)
#pragma unroll
      for (int i = 0; i < kWords; ++i) {
        const uint32_t u = w[i] ^ 0x80808080u;
        q2[2 * i] = add2(pk2u(__byte_perm(u, K, 0x7440), __byte_perm(u, K, 0x7441)), off);
        q2[2 * i + 1] = add2(pk2u(__byte_perm(u, K, 0x7442), __byte_perm(u, K, 0x7443)), off);
      }
    }
  }
};

__device__ __forceinline__ f32x2 fma2(f32x2 a, f32x2 b, f32x2 c) {
  f32x2 r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}

// ---------------------------------------------------------------------------
// Division of the rank sum by W, correctly rounded like the IEEE division.
//  * W a power of two: the product with the exact reciprocal is the same
//    correctly rounded quotient.
//  * otherwise: the division by a constant known in advance of Brisebarre,
//    Muller and Raina ("Accelerating correctly rounded floating-point division
//    when the divisor is known in advance", IEEE Trans. Computers 53(8),
//    2004): q = fma(x, zh, RN(x*zl)) with zh the binary32 number just below
//    1/W and zl = RN(1/W - zh) > 0, two packed instructions per pair.  For
//    W = 3..15 it equals RN(x/W) for every binary32 x with |x| >= 2^-100
//    (checked exhaustively over all such x); it can differ only where x*zl
//    underflows.  With zl > 0 a zero sum keeps its sign (+-0 / W = +-0).
//    The sums are never that small unless a step is: when every rank's step of
//    the block is 0 or at least 2^-77, every decoded term RN(q*Delta) is 0 or
//    a normal number of magnitude >= 2^-77, hence a multiple of 2^-100, and so
//    is every rounded partial sum (a rounded sum of multiples of 2^-100 stays
//    one), so a nonzero sum has |x| >= 2^-100.  A block with a nonzero step
//    below 2^-77 takes the IEEE division instead.
// ---------------------------------------------------------------------------

// Largest binary32 number not above 1/W (W >= 3, not a power of two).
constexpr float recip_below(int W) {
  float f = 1.0f / float(W);
  if (double(f) > 1.0 / double(W)) {
    double e = 1.0;
    while (e > double(f)) e *= 0.5;  // 2^floor(log2 f)
    f = float(double(f) - e * 1.1920928955078125e-07);  // one unit in the last place below
  }
  return f;
}

template <int W>
struct RankDiv {
  static constexpr bool kPow2 = (W & (W - 1)) == 0;
  static constexpr float zh = kPow2 ? 1.0f / float(W) : recip_below(W);
  static constexpr float zl = kPow2 ? 0.0f : float(1.0 / double(W) - double(zh));
};

// True when every step is 0 or at least 2^-77 (the fast quotient is exact):
// no step's magnitude lies in (0, 2^-77), i.e. none has bits in [1, bits(2^-77)).
template <int W>
__device__ __forceinline__ bool steps_allow_fast_division(const float (&s)[W]) {
  constexpr uint32_t kMinBits = 0x19000000u;  // bits of 2^-77
  uint32_t small = 0;
#pragma unroll
  for (int w = 0; w < W; ++w) small |= uint32_t((__float_as_uint(s[w]) & 0x7FFFFFFFu) - 1u < kMinBits - 1u);
  return small == 0;
}

// Two-constant quotient of a pair (W not a power of two).
template <int W>
__device__ __forceinline__ void div_fast(f32x2 sum, float& lo, float& hi) {
  using D = RankDiv<W>;
  upk2(fma2(sum, pk2(D::zh, D::zh), mul2(sum, pk2(D::zl, D::zl))), lo, hi);
}

// The quotients of E/2 pairs of rank sums (see RankDiv); pair j holds the
// elements (CC::pair_lo(j), CC::pair_hi(j)) of the chunk.
template <int W, int E, typename CC>
__device__ __forceinline__ void div_by_ranks(const f32x2 (&acc)[E / 2], const float (&s)[W], float out[E]) {
  using D = RankDiv<W>;
  if constexpr (D::kPow2) {
#pragma unroll
    for (int j = 0; j < E / 2; ++j) upk2(mul2(acc[j], pk2(D::zh, D::zh)), out[CC::pair_lo(j)], out[CC::pair_hi(j)]);
  } else {
    if (steps_allow_fast_division<W>(s)) {
#pragma unroll
      for (int j = 0; j < E / 2; ++j) div_fast<W>(acc[j], out[CC::pair_lo(j)], out[CC::pair_hi(j)]);
    } else {
#pragma unroll
      for (int j = 0; j < E / 2; ++j) {
        float a, b;
        upk2(acc[j], a, b);
        out[CC::pair_lo(j)] = __fdiv_rn(a, float(W));
        out[CC::pair_hi(j)] = __fdiv_rn(b, float(W));
      }
    }
  }
}

// Per-element fp32 rank average of Eqn (8) for an E-element chunk from its
// W ranks' codes and steps, in rank order 0..W-1:
//   ((d_0 + d_1) + d_2) + ... , d_w = f32(q_w) * Delta_w (rounded), then / W.
// Two elements per instruction: packed products (prod2) and packed sums.
template <int BITS, int W, int E>
__device__ __forceinline__ void mean_of_codes(const ChunkCodes<BITS, E> (&cw)[W], const float (&s)[W], float neg_zero,
                                              float out[E]) {
  const f32x2 z = pk2(neg_zero, neg_zero);
  f32x2 acc[E / 2];
#pragma unroll
  for (int w = 0; w < W; ++w) {
    f32x2 q2[E / 2];
    cw[w].decode(q2);
    const f32x2 s2 = pk2(s[w], s[w]);
#pragma unroll
    for (int j = 0; j < E / 2; ++j) {
      const f32x2 d = prod2(q2[j], s2, z);
      acc[j] = (w == 0) ? d : add2(acc[j], d);
    }
  }
  div_by_ranks<W, E, ChunkCodes<BITS, E>>(acc, s, out);
}

// Same, loading the codes straight from global memory (chunk at e0, block blk).
template <int BITS, int W, int E>
__device__ __forceinline__ void decode_mean(const RankPtrs& rp, int64_t e0, int64_t blk, float out[E]) {
  ChunkCodes<BITS, E> cw[W];
  float s[W];
#pragma unroll
  for (int w = 0; w < W; ++w) {
    cw[w].load(rp.codes[w], e0);
    s[w] = __ldg(rp.scales[w] + blk);
  }
  mean_of_codes<BITS, W, E>(cw, s, rp.neg_zero, out);
}

}  // namespace loco
