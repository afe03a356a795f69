// Sender step of LoCo on one rank's flat gradient bucket.
//
// "LoCo: Low-Bit Communication Adaptor for Large-scale Model Training",
// §3.1 Eqns (1)-(3) and §3.2 Eqns (4)-(7): compensate the gradient with the
// stored error, quantise it blockwise to p bits, pack the codes, and update
// the error as a clipped moving average of the compression error, reset every
// T_c steps.
//
// Mapping: one lane owns 8 consecutive elements (one 16-byte load of bf16
// gradient or two of fp32, two 16-byte loads of the error); a quant block of
// B elements spans B/8 consecutive lanes, so its absmax is a butterfly of
// B/8-lane __shfl_xor_sync steps (max is exact, so the order is irrelevant).
// A warp covers 256 elements.  With only two input streams, direct 16-byte
// loads from enough resident warps keep HBM busy (a shared-memory staged
// variant measured slower: its barriers cost more than it hid).  One pass
// over HBM: read g and e, write e, the packed codes and one step per block.
// No shared memory, no atomics, no inter-CTA communication.
#include "device_common.cuh"

namespace loco {

constexpr int kThreads = 256;

// Eqns (2),(1),(3),(4),(5),(7) for the 8 elements [e0, e0+8) of one lane,
// given their gradient g and previous error e (0 past n).  All 32 lanes of the
// warp must call this together (the absmax is a warp shuffle).  E8 selects
// the 8-bit error storage: the new error is written as int8 codes of step
// Delta/kappa instead of clipped fp32 values.
template <int BITS, int BLOCK, bool E8, bool FIXED>
__device__ __forceinline__ void compress8(const CompressArgs& a, int64_t e0, int64_t n_pad, int lane, const float g[8],
                                          const float e[8]) {
  constexpr int G = BLOCK / 8;  // lanes per quant block
  constexpr float QMAX = float((1 << (BITS - 1)) - 1);
  constexpr float QMIN = -float(1 << (BITS - 1));

  // Eqn (2): compensate; block absmax.
  float h[8];
  float amax = 0.0f;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    h[j] = __fadd_rn(g[j], e[j]);
    amax = fmaxf(amax, fabsf(h[j]));
  }
#pragma unroll
  for (int off = G / 2; off >= 1; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));

  // Scale of Eqn (1) and bounds of the 8-bit error range (Eqn 7).
  float delta, inv;
  if constexpr (FIXED) {
    delta = a.fixed_delta;
    inv = a.fixed_inv;
  } else {
    // An all-zero block, or one whose inverse step qmax/A overflows fp32
    // (A < qmax/FLT_MAX), gets step and inverse 0: every code is 0.
    inv = (amax == 0.0f) ? 0.0f : __fdiv_rn(QMAX, amax);
    if (amax == 0.0f || isinf(inv)) {
      delta = 0.0f;
      inv = 0.0f;
    } else {
      delta = __fdiv_rn(amax, QMAX);
    }
  }
  const float de = __fdiv_rn(delta, a.kappa);
  const float elo = __fmul_rn(-128.0f, de);
  const float ehi = __fmul_rn(127.0f, de);
  float inv_e = __fmul_rn(a.kappa, inv);  // s_e = kappa * s; code 0 if it overflows
  if (isinf(inv_e)) inv_e = 0.0f;

  // Eqns (1),(3),(4),(5),(7) per element.  tq / teq hold the float whose low
  // byte is the two's-complement code (1.5*2^23 + q).
  uint32_t tq[8], teq[8];
  float en[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    float x = __fmul_rn(h[j], inv);
    // Saturation of Round_p-bit.  With the absmax step it is a no-op for finite
    // inputs: |h| <= A and inv = RN(qmax/A) give |x| <= qmax*(1 + 2^-23) < qmax + 1/2,
    // which rounds to at most qmax; only a fixed scale can push x past the range.
    if constexpr (FIXED) x = fminf(fmaxf(x, QMIN), QMAX);
    const float t = __fadd_rn(x, kRoundMagic);  // rint, halves to even
    tq[j] = __float_as_uint(t);
    const float q = __fsub_rn(t, kRoundMagic);
    const float d = __fmul_rn(q, delta);
    const float r = __fsub_rn(h[j], d);
    float v = __fadd_rn(__fmul_rn(a.beta, e[j]), __fmul_rn(a.one_minus_beta, r));
    if constexpr (E8) {
      // Eqn (7): e = Round_8-bit(s_e * e~).
      float xe = __fmul_rn(v, inv_e);
      xe = fminf(fmaxf(xe, -128.0f), 127.0f);
      teq[j] = __float_as_uint(__fadd_rn(xe, kRoundMagic));
    } else {
      v = (v < elo) ? elo : v;
      v = (v > ehi) ? ehi : v;
      en[j] = v;
    }
  }
  // Reset step of Eqn (7): the stored error becomes 0 (a uniform branch).
  if (a.reset) {
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      en[j] = 0.0f;
      teq[j] = 0u;
    }
  }
  // Pack the low bytes / nibbles with byte permutes.
  uint32_t packed[BITS == 4 ? 1 : 2];
  if constexpr (BITS == 8) {
    packed[0] = __byte_perm(__byte_perm(tq[0], tq[1], 0x0040), __byte_perm(tq[2], tq[3], 0x0040), 0x5410);
    packed[1] = __byte_perm(__byte_perm(tq[4], tq[5], 0x0040), __byte_perm(tq[6], tq[7], 0x0040), 0x5410);
  } else {
    // byte k = (code_{2k} & 0xF) | (code_{2k+1} << 4)
    uint32_t b[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) b[k] = (tq[2 * k] & 0xFu) | ((tq[2 * k + 1] << 4) & 0xF0u);
    packed[0] = __byte_perm(__byte_perm(b[0], b[1], 0x0040), __byte_perm(b[2], b[3], 0x0040), 0x5410);
  }
  uint32_t epacked[2] = {0u, 0u};
  if constexpr (E8) {
    epacked[0] = __byte_perm(__byte_perm(teq[0], teq[1], 0x0040), __byte_perm(teq[2], teq[3], 0x0040), 0x5410);
    epacked[1] = __byte_perm(__byte_perm(teq[4], teq[5], 0x0040), __byte_perm(teq[6], teq[7], 0x0040), 0x5410);
  }

  // Stores: codes and the block step inside the padded code range, the error
  // only for elements < n.
  if (e0 < n_pad) {
    if constexpr (BITS == 4)
      st_stream(reinterpret_cast<uint32_t*>(a.codes + (e0 >> 1)), packed[0]);
    else
      st_stream(reinterpret_cast<uint2*>(a.codes + e0), make_uint2(packed[0], packed[1]));
    if ((lane & (G - 1)) == 0) {
      a.scales[e0 / BLOCK] = delta;
      if constexpr (E8) a.err_steps[e0 / BLOCK] = de;
    }
  }
  if constexpr (E8) {
    if (e0 + 8 <= a.n) {
      st_stream(reinterpret_cast<uint2*>(a.err_codes + e0), make_uint2(epacked[0], epacked[1]));
    } else {
#pragma unroll
      for (int j = 0; j < 8; ++j)
        if (e0 + j < a.n) a.err_codes[e0 + j] = int8_t((epacked[j >> 2] >> (8 * (j & 3))) & 0xFFu);
    }
  } else if (e0 + 8 <= a.n) {
    float4* ep = reinterpret_cast<float4*>(a.err + e0);
    st_stream(ep, make_float4(en[0], en[1], en[2], en[3]));
    st_stream(ep + 1, make_float4(en[4], en[5], en[6], en[7]));
  } else {
#pragma unroll
    for (int j = 0; j < 8; ++j)
      if (e0 + j < a.n) a.err[e0 + j] = en[j];
  }
}

// Loads the 8 gradient values of the lane's chunk at e0 (0 past n).
template <bool BF16>
__device__ __forceinline__ void load_grad8(const CompressArgs& a, int64_t e0, float g[8]) {
  if (e0 + 8 <= a.n) {
    if constexpr (BF16) {
      const uint4 raw = ld_stream(reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(a.grad) + e0));
      g[0] = bf16lo_to_f32(raw.x); g[1] = bf16hi_to_f32(raw.x);
      g[2] = bf16lo_to_f32(raw.y); g[3] = bf16hi_to_f32(raw.y);
      g[4] = bf16lo_to_f32(raw.z); g[5] = bf16hi_to_f32(raw.z);
      g[6] = bf16lo_to_f32(raw.w); g[7] = bf16hi_to_f32(raw.w);
    } else {
      const float4* gp = reinterpret_cast<const float4*>(static_cast<const float*>(a.grad) + e0);
      const float4 g0 = ld_stream(gp), g1 = ld_stream(gp + 1);
      g[0] = g0.x; g[1] = g0.y; g[2] = g0.z; g[3] = g0.w;
      g[4] = g1.x; g[5] = g1.y; g[6] = g1.z; g[7] = g1.w;
    }
  } else {
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int64_t i = e0 + j;
      if (i < a.n) {
        if constexpr (BF16)
          g[j] = __uint_as_float(uint32_t(static_cast<const uint16_t*>(a.grad)[i]) << 16);
        else
          g[j] = static_cast<const float*>(a.grad)[i];
      } else {
        g[j] = 0.0f;
      }
    }
  }
}

// Loads the 8 gradient and error values of the lane's chunk at e0 (0 past n).
// With E8 the previous error is decoded from its int8 codes and the block's
// stored step: e = f32(qe) * De (the decompressor of Eqn 2).
template <bool BF16, bool E8, int BLOCK>
__device__ __forceinline__ void load8(const CompressArgs& a, int64_t e0, float g[8], float e[8]) {
  if constexpr (E8) {
    load_grad8<BF16>(a, e0, g);
    const float dprev = (e0 < a.n) ? a.err_steps[e0 / BLOCK] : 0.0f;
    uint32_t w0 = 0, w1 = 0;
    if (e0 + 8 <= a.n) {
      const uint2 v = ld_stream(reinterpret_cast<const uint2*>(a.err_codes + e0));
      w0 = v.x;
      w1 = v.y;
    } else {
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const uint32_t b = (e0 + j < a.n) ? uint32_t(uint8_t(a.err_codes[e0 + j])) : 0u;
        if (j < 4) w0 |= b << (8 * j); else w1 |= b << (8 * (j - 4));
      }
    }
    constexpr uint32_t K = 0x4B000000u;
    const uint32_t u0 = w0 ^ 0x80808080u, u1 = w1 ^ 0x80808080u;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float q0 = __fsub_rn(__uint_as_float(__byte_perm(u0, K, 0x7440 | j)), 8388736.0f);
      const float q1 = __fsub_rn(__uint_as_float(__byte_perm(u1, K, 0x7440 | j)), 8388736.0f);
      e[j] = __fmul_rn(q0, dprev);
      e[j + 4] = __fmul_rn(q1, dprev);
    }
    return;
  }
  if (e0 + 8 <= a.n) {
    if constexpr (BF16) {
      const uint4 raw = ld_stream(reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(a.grad) + e0));
      g[0] = bf16lo_to_f32(raw.x); g[1] = bf16hi_to_f32(raw.x);
      g[2] = bf16lo_to_f32(raw.y); g[3] = bf16hi_to_f32(raw.y);
      g[4] = bf16lo_to_f32(raw.z); g[5] = bf16hi_to_f32(raw.z);
      g[6] = bf16lo_to_f32(raw.w); g[7] = bf16hi_to_f32(raw.w);
    } else {
      const float4* gp = reinterpret_cast<const float4*>(static_cast<const float*>(a.grad) + e0);
      const float4 g0 = ld_stream(gp), g1 = ld_stream(gp + 1);
      g[0] = g0.x; g[1] = g0.y; g[2] = g0.z; g[3] = g0.w;
      g[4] = g1.x; g[5] = g1.y; g[6] = g1.z; g[7] = g1.w;
    }
    const float4* ep = reinterpret_cast<const float4*>(a.err + e0);
    const float4 e0v = ld_stream(ep), e1v = ld_stream(ep + 1);
    e[0] = e0v.x; e[1] = e0v.y; e[2] = e0v.z; e[3] = e0v.w;
    e[4] = e1v.x; e[5] = e1v.y; e[6] = e1v.z; e[7] = e1v.w;
  } else {
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int64_t i = e0 + j;
      if (i < a.n) {
        if constexpr (BF16)
          g[j] = __uint_as_float(uint32_t(static_cast<const uint16_t*>(a.grad)[i]) << 16);
        else
          g[j] = static_cast<const float*>(a.grad)[i];
        e[j] = a.err[i];
      } else {
        g[j] = 0.0f;
        e[j] = 0.0f;
      }
    }
  }
}

// Raw words of one lane's full 8-element chunk, loaded with 16- or 8-byte
// vector loads and decoded only when the chunk is processed, so several
// chunks can be in flight in few registers.  8-bit error storage keeps the
// codes in e[0].x/.y and the block's stored step in e[0].z.
template <bool BF16, bool E8>
struct RawChunk {
  uint4 g[BF16 ? 1 : 2];
  uint4 e[E8 ? 1 : 2];
};

template <bool BF16, bool E8, int BLOCK>
__device__ __forceinline__ void load_raw(const CompressArgs& a, int64_t e0, RawChunk<BF16, E8>& r) {
  const uint4* gp = reinterpret_cast<const uint4*>(static_cast<const uint8_t*>(a.grad) + e0 * (BF16 ? 2 : 4));
  r.g[0] = ld_stream(gp);
  if constexpr (!BF16) r.g[1] = ld_stream(gp + 1);
  if constexpr (E8) {
    const uint2 c = ld_stream(reinterpret_cast<const uint2*>(a.err_codes + e0));
    r.e[0] = make_uint4(c.x, c.y, __float_as_uint(a.err_steps[e0 / BLOCK]), 0u);
  } else {
    const uint4* ep = reinterpret_cast<const uint4*>(a.err + e0);
    r.e[0] = ld_stream(ep);
    r.e[1] = ld_stream(ep + 1);
  }
}

template <bool BF16, bool E8>
__device__ __forceinline__ void unpack_raw(const RawChunk<BF16, E8>& r, float g[8], float e[8]) {
  if constexpr (BF16) {
    g[0] = bf16lo_to_f32(r.g[0].x); g[1] = bf16hi_to_f32(r.g[0].x);
    g[2] = bf16lo_to_f32(r.g[0].y); g[3] = bf16hi_to_f32(r.g[0].y);
    g[4] = bf16lo_to_f32(r.g[0].z); g[5] = bf16hi_to_f32(r.g[0].z);
    g[6] = bf16lo_to_f32(r.g[0].w); g[7] = bf16hi_to_f32(r.g[0].w);
  } else {
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      g[4 * i] = __uint_as_float(r.g[i].x); g[4 * i + 1] = __uint_as_float(r.g[i].y);
      g[4 * i + 2] = __uint_as_float(r.g[i].z); g[4 * i + 3] = __uint_as_float(r.g[i].w);
    }
  }
  if constexpr (E8) {
    constexpr uint32_t K = 0x4B000000u;
    const uint32_t u0 = r.e[0].x ^ 0x80808080u, u1 = r.e[0].y ^ 0x80808080u;
    const float dprev = __uint_as_float(r.e[0].z);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      e[j] = __fmul_rn(__fsub_rn(__uint_as_float(__byte_perm(u0, K, 0x7440 | j)), 8388736.0f), dprev);
      e[j + 4] = __fmul_rn(__fsub_rn(__uint_as_float(__byte_perm(u1, K, 0x7440 | j)), 8388736.0f), dprev);
    }
  } else {
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      e[4 * i] = __uint_as_float(r.e[i].x); e[4 * i + 1] = __uint_as_float(r.e[i].y);
      e[4 * i + 2] = __uint_as_float(r.e[i].z); e[4 * i + 3] = __uint_as_float(r.e[i].w);
    }
  }
}

// Warps walk the bucket's 256-element warp tiles grid-stride, U tiles per
// iteration with all their loads issued before any compute; every lane of a
// warp takes the same trip count, so the shuffles are always full-warp.  A
// lane whose chunk crosses n (only in the last warp tile) loads it element by
// element instead.
template <int BITS, int BLOCK, bool BF16, bool E8, bool FIXED, int U>
__global__ void __launch_bounds__(kThreads) k_compress(const CompressArgs a) {
  const int lane = threadIdx.x & 31;
  const int64_t nb = (a.n + BLOCK - 1) / BLOCK;
  const int64_t n_pad = nb * BLOCK;
  const int64_t ntiles = (n_pad + 255) / 256;
  const int64_t warp0 = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = (int64_t(gridDim.x) * blockDim.x) >> 5;
  for (int64_t tile = warp0; tile < ntiles; tile += U * nwarps) {
    RawChunk<BF16, E8> raw[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t e0 = (tile + u * nwarps) * 256 + lane * 8;
      if (tile + u * nwarps < ntiles && e0 + 8 <= a.n) load_raw<BF16, E8, BLOCK>(a, e0, raw[u]);
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t tu = tile + u * nwarps;
      if (tu < ntiles) {
        const int64_t e0 = tu * 256 + lane * 8;
        float g[8], e[8];
        if (e0 + 8 <= a.n)
          unpack_raw<BF16, E8>(raw[u], g, e);
        else
          load8<BF16, E8, BLOCK>(a, e0, g, e);
        compress8<BITS, BLOCK, E8, FIXED>(a, e0, n_pad, lane, g, e);
      }
    }
  }
}

#ifndef LOCO_COMPRESS_UNROLL
#define LOCO_COMPRESS_UNROLL 2     // fp32 error: 48 bytes per lane per warp tile
#endif
#ifndef LOCO_COMPRESS_UNROLL_E8
#define LOCO_COMPRESS_UNROLL_E8 2  // 8-bit error: 24 bytes per lane per warp tile (issue-bound)
#endif

template <int BITS, int BLOCK, bool BF16, bool E8, bool FIXED>
static cudaError_t launch_t(const CompressArgs& a, cudaStream_t s) {
  constexpr int U = E8 ? LOCO_COMPRESS_UNROLL_E8 : LOCO_COMPRESS_UNROLL;
  const void* fn = reinterpret_cast<const void*>(&k_compress<BITS, BLOCK, BF16, E8, FIXED, U>);
  static const int cap = persistent_grid(fn, kThreads);
  const int64_t nb = (a.n + BLOCK - 1) / BLOCK;
  const int64_t warps_needed = (nb * BLOCK + 255) / 256;
  const int64_t ctas_needed = (warps_needed + kThreads / 32 - 1) / (kThreads / 32);
  const int grid = int(ctas_needed < cap ? ctas_needed : cap);
  k_compress<BITS, BLOCK, BF16, E8, FIXED, U><<<grid, kThreads, 0, s>>>(a);
  return cudaGetLastError();
}

template <int BITS, int BLOCK, bool E8, bool FIXED>
static cudaError_t launch_g(const CompressArgs& a, cudaStream_t s) {
  return a.grad_bf16 ? launch_t<BITS, BLOCK, true, E8, FIXED>(a, s) : launch_t<BITS, BLOCK, false, E8, FIXED>(a, s);
}

template <int BITS, int BLOCK>
static cudaError_t launch_dt(const CompressArgs& a, cudaStream_t s) {
  const bool e8 = a.err_codes != nullptr;
  if (a.fixed) return e8 ? launch_g<BITS, BLOCK, true, true>(a, s) : launch_g<BITS, BLOCK, false, true>(a, s);
  return e8 ? launch_g<BITS, BLOCK, true, false>(a, s) : launch_g<BITS, BLOCK, false, false>(a, s);
}

template <int BITS>
static cudaError_t launch_b(const CompressArgs& a, cudaStream_t s) {
  switch (a.block) {
    case 64: return launch_dt<BITS, 64>(a, s);
    case 128: return launch_dt<BITS, 128>(a, s);
    case 256: return launch_dt<BITS, 256>(a, s);
  }
  return cudaErrorInvalidValue;
}

cudaError_t launch_compress(const CompressArgs& a, cudaStream_t s) {
  return a.bits == 4 ? launch_b<4>(a, s) : launch_b<8>(a, s);
}

}  // namespace loco
