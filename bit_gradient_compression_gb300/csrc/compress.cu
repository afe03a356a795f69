// Sender step of LoCo on one rank's flat gradient bucket.
//
// "LoCo: Low-Bit Communication Adaptor for Large-scale Model Training",
// §3.1 Eqns (1)-(3) and §3.2 Eqns (4)-(7): compensate the gradient with the
// stored error, quantise it blockwise to p bits, pack the codes, and update
// the error as a clipped moving average of the compression error, reset every
// T_c steps.
//
// Mapping: one lane owns EL consecutive elements (8 with the fp32 error: one
// 16-byte load of bf16 gradient or two of fp32, two of the error; 16 with the
// int8 error, whose path is bound by instruction issue rather than HBM); a
// quant block of B elements spans B/EL consecutive lanes, so its absmax is a
// butterfly of __shfl_xor_sync steps (max is exact, so the order is
// irrelevant), and a warp covers 32*EL elements.  With 16 elements per lane a
// warp spans two 256-element blocks whose scales its half-warps compute in the
// same instructions, which halves the per-element cost of the three IEEE
// divisions.  The fp32 arithmetic runs on packed pairs (f32x2).  With only two
// input streams, direct vector loads from enough resident warps keep HBM busy
// (a shared-memory staged variant measured slower: its barriers cost more than
// it hid).  One pass over HBM: read g and e, write e, the packed codes and one
// step per block.  No shared memory, no atomics, no inter-CTA communication.
#include "device_common.cuh"

namespace loco {

constexpr int kThreads = 256;

// Stores NW consecutive 32-bit words with one streaming store (NW = 1, 2, 4).
template <int NW>
__device__ __forceinline__ void st_words(void* p, const uint32_t (&w)[NW]) {
  static_assert(NW == 1 || NW == 2 || NW == 4, "one 4-, 8- or 16-byte store");
  if constexpr (NW == 1)
    st_stream(reinterpret_cast<uint32_t*>(p), w[0]);
  else if constexpr (NW == 2)
    st_stream(reinterpret_cast<uint2*>(p), make_uint2(w[0], w[1]));
  else
    st_stream(reinterpret_cast<uint4*>(p), make_uint4(w[0], w[1], w[2], w[3]));
}

#ifndef LOCO_COMPRESS_E8_CVT
#define LOCO_COMPRESS_E8_CVT 1  // 1: the int8 error code by one saturating round-to-nearest-even conversion
#endif

// Nearest integer to x, halves to even, saturated to [-128, 127] (one
// conversion instruction: a float-to-integer conversion clamps to the range of
// its destination type); the code is the low byte of the result.  Clamping and
// then rounding give the same integer because both bounds are integers.
__device__ __forceinline__ uint32_t rint_sat_s8(float x) {
  uint32_t r;
  asm("cvt.rni.sat.s8.f32 %0, %1;" : "=r"(r) : "f"(x));
  return r;
}

// Low bytes of four words, in order, as one word.
__device__ __forceinline__ uint32_t low_bytes(uint32_t b0, uint32_t b1, uint32_t b2, uint32_t b3) {
  return __byte_perm(__byte_perm(b0, b1, 0x0040), __byte_perm(b2, b3, 0x0040), 0x5410);
}

// Eqns (2),(1),(3),(4),(5),(7) for the EL elements [e0, e0+EL) of one lane,
// given their gradient g and previous error e as EL/2 packed pairs (element
// 2k in the low lane of pair k; 0 past n).  All 32 lanes of the warp must call
// this together (the absmax is a warp shuffle over the BLOCK/EL lanes of a
// block).  E8 selects the 8-bit error storage: the new error is written as
// int8 codes of step Delta/kappa instead of clipped fp32 values.  Every fp32
// multiply and add is one packed instruction per pair with the rounding of the
// scalar one; products that feed an add are formed by prod2.
template <int BITS, int BLOCK, bool E8, bool FIXED, int EL>
__device__ __forceinline__ void compress_chunk(const CompressArgs& a, int64_t e0, int64_t n_pad, int lane,
                                               const f32x2 (&g)[EL / 2], const f32x2 (&e)[EL / 2]) {
  constexpr int P = EL / 2;     // pairs per lane
  constexpr int G = BLOCK / EL;  // lanes per quant block
  static_assert(EL == 8 || EL == 16, "8 or 16 elements per lane");
  static_assert(G >= 1 && G <= 32 && BLOCK % EL == 0, "a lane's elements lie in one block");
  constexpr float QMAX = float((1 << (BITS - 1)) - 1);
  constexpr float QMIN = -float(1 << (BITS - 1));
  const f32x2 z = pk2(a.neg_zero, a.neg_zero);

  // Eqn (2): compensate; block absmax.
  f32x2 h[P];
  float amax = 0.0f;
#pragma unroll
  for (int k = 0; k < P; ++k) {
    h[k] = add2(g[k], e[k]);
    float h0, h1;
    upk2(h[k], h0, h1);
    amax = fmaxf(amax, fmaxf(fabsf(h0), fabsf(h1)));
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
  const float de = (a.kappa_recip != 0.0f) ? __fmul_rn(delta, a.kappa_recip) : __fdiv_rn(delta, a.kappa);
  const float elo = __fmul_rn(-128.0f, de);
  const float ehi = __fmul_rn(127.0f, de);
  float inv_e = __fmul_rn(a.kappa, inv);  // s_e = kappa * s; code 0 if it overflows
  if (isinf(inv_e)) inv_e = 0.0f;

  // Eqns (1),(3),(4),(5),(7) per pair.  tq / teq hold the float whose low
  // byte is the two's-complement code (1.5*2^23 + q).
  const f32x2 inv2 = pk2(inv, inv), delta2 = pk2(delta, delta), inv_e2 = pk2(inv_e, inv_e);
  const f32x2 magic2 = pk2(kRoundMagic, kRoundMagic);
  const f32x2 beta2 = pk2(a.beta, a.beta), omb2 = pk2(a.one_minus_beta, a.one_minus_beta);
  uint32_t tq[EL], teq[EL];
  float en[EL];
#pragma unroll
  for (int k = 0; k < P; ++k) {
    f32x2 x = prod2(h[k], inv2, z);
    // Saturation of Round_p-bit.  With the absmax step it is a no-op for finite
    // inputs: |h| <= A and inv = RN(qmax/A) give |x| <= qmax*(1 + 2^-23) < qmax + 1/2,
    // which rounds to at most qmax; only a fixed scale can push x past the range.
    if constexpr (FIXED) {
      float x0, x1;
      upk2(x, x0, x1);
      x = pk2(fminf(fmaxf(x0, QMIN), QMAX), fminf(fmaxf(x1, QMIN), QMAX));
    }
    const f32x2 t = add2(x, magic2);  // rint, halves to even
    float t0, t1;
    upk2(t, t0, t1);
    tq[2 * k] = __float_as_uint(t0);
    tq[2 * k + 1] = __float_as_uint(t1);
    const f32x2 q = sub2(t, magic2);
    const f32x2 r = sub2(h[k], prod2(q, delta2, z));
    const f32x2 v = add2(prod2(beta2, e[k], z), prod2(omb2, r, z));
    float v0, v1;
    if constexpr (E8) {
      // Eqn (7): e = Round_8-bit(s_e * e~).
      upk2(prod2(v, inv_e2, z), v0, v1);
#if LOCO_COMPRESS_E8_CVT
      teq[2 * k] = rint_sat_s8(v0);
      teq[2 * k + 1] = rint_sat_s8(v1);
#else
      const f32x2 te = add2(pk2(fminf(fmaxf(v0, -128.0f), 127.0f), fminf(fmaxf(v1, -128.0f), 127.0f)), magic2);
      float te0, te1;
      upk2(te, te0, te1);
      teq[2 * k] = __float_as_uint(te0);
      teq[2 * k + 1] = __float_as_uint(te1);
#endif
    } else {
      upk2(v, v0, v1);
      v0 = (v0 < elo) ? elo : v0;
      v0 = (v0 > ehi) ? ehi : v0;
      v1 = (v1 < elo) ? elo : v1;
      v1 = (v1 > ehi) ? ehi : v1;
      en[2 * k] = v0;
      en[2 * k + 1] = v1;
    }
  }
  // Reset step of Eqn (7): the stored error becomes 0 (a uniform branch).
  if (a.reset) {
#pragma unroll
    for (int j = 0; j < EL; ++j) {
      en[j] = 0.0f;
      teq[j] = 0u;
    }
  }
  // Pack the low bytes / nibbles with byte permutes.
  constexpr int CW = EL * BITS / 32;  // code words per lane
  uint32_t packed[CW];
#pragma unroll
  for (int w = 0; w < CW; ++w) {
    if constexpr (BITS == 8) {
      packed[w] = low_bytes(tq[4 * w], tq[4 * w + 1], tq[4 * w + 2], tq[4 * w + 3]);
    } else {
      // byte k = (code_{2k} & 0xF) | (code_{2k+1} << 4): gather the even and odd
      // codes' low bytes, then merge the two words nibble-wise.
      const uint32_t* c = tq + 8 * w;
      const uint32_t ev = low_bytes(c[0], c[2], c[4], c[6]);
      const uint32_t od = low_bytes(c[1], c[3], c[5], c[7]);
      packed[w] = (ev & 0x0F0F0F0Fu) | ((od << 4) & 0xF0F0F0F0u);
    }
  }

  // Stores: codes and the block step inside the padded code range, the error
  // only for elements < n.
  if (e0 < n_pad) {
    st_words<CW>(a.codes + (e0 * BITS >> 3), packed);
    if ((lane & (G - 1)) == 0) {
      a.scales[e0 / BLOCK] = delta;
      if constexpr (E8) a.err_steps[e0 / BLOCK] = de;
    }
  }
  if constexpr (E8) {
    uint32_t epacked[EL / 4];
#pragma unroll
    for (int w = 0; w < EL / 4; ++w) epacked[w] = low_bytes(teq[4 * w], teq[4 * w + 1], teq[4 * w + 2], teq[4 * w + 3]);
    if (e0 + EL <= a.n) {
      st_words<EL / 4>(a.err_codes + e0, epacked);
    } else {
#pragma unroll
      for (int j = 0; j < EL; ++j)
        if (e0 + j < a.n) a.err_codes[e0 + j] = int8_t((epacked[j >> 2] >> (8 * (j & 3))) & 0xFFu);
    }
  } else if (e0 + EL <= a.n) {
    float4* ep = reinterpret_cast<float4*>(a.err + e0);
#pragma unroll
    for (int i = 0; i < EL / 4; ++i) st_stream(ep + i, make_float4(en[4 * i], en[4 * i + 1], en[4 * i + 2], en[4 * i + 3]));
  } else {
#pragma unroll
    for (int j = 0; j < EL; ++j)
      if (e0 + j < a.n) a.err[e0 + j] = en[j];
  }
}

// Gradient and error of a lane chunk that crosses n, element by element (0
// past n).  With E8 the previous error is decoded from its int8 code and the
// block's stored step: e = f32(qe) * De (the decompressor of Eqn 2).
template <bool BF16, bool E8, int BLOCK, int EL>
__device__ __forceinline__ void load_partial(const CompressArgs& a, int64_t e0, f32x2 (&g)[EL / 2],
                                             f32x2 (&e)[EL / 2]) {
  float gs[EL], es[EL];
  const float dprev = (E8 && e0 < a.n) ? a.err_steps[e0 / BLOCK] : 0.0f;
#pragma unroll
  for (int j = 0; j < EL; ++j) {
    const int64_t i = e0 + j;
    gs[j] = 0.0f;
    es[j] = 0.0f;
    if (i < a.n) {
      if constexpr (BF16)
        gs[j] = __uint_as_float(uint32_t(static_cast<const uint16_t*>(a.grad)[i]) << 16);
      else
        gs[j] = static_cast<const float*>(a.grad)[i];
      if constexpr (E8)
        es[j] = __fmul_rn(float(a.err_codes[i]), dprev);
      else
        es[j] = a.err[i];
    }
  }
#pragma unroll
  for (int k = 0; k < EL / 2; ++k) {
    g[k] = pk2(gs[2 * k], gs[2 * k + 1]);
    e[k] = pk2(es[2 * k], es[2 * k + 1]);
  }
}

// Raw words of one lane's full EL-element chunk, loaded with 16-byte (or, for
// 8 int8 codes, 8-byte) vector loads and decoded only when the chunk is
// processed, so several chunks can be in flight in few registers.
template <bool BF16, bool E8, int EL>
struct RawChunk {
  static constexpr int kG = EL * (BF16 ? 2 : 4) / 16;  // 16-byte words of gradient
  uint4 g[kG];
  uint4 e[E8 ? 1 : EL / 4];  // fp32 error, or the int8 codes in the first EL/4 words
  float step;                // block step of the int8 codes
};

template <bool BF16, bool E8, int BLOCK, int EL>
__device__ __forceinline__ void load_raw(const CompressArgs& a, int64_t e0, RawChunk<BF16, E8, EL>& r) {
  const uint4* gp = reinterpret_cast<const uint4*>(static_cast<const uint8_t*>(a.grad) + e0 * (BF16 ? 2 : 4));
#pragma unroll
  for (int i = 0; i < RawChunk<BF16, E8, EL>::kG; ++i) r.g[i] = ld_stream(gp + i);
  if constexpr (E8) {
    if constexpr (EL == 16) {
      r.e[0] = ld_stream(reinterpret_cast<const uint4*>(a.err_codes + e0));
    } else {
      const uint2 c = ld_stream(reinterpret_cast<const uint2*>(a.err_codes + e0));
      r.e[0] = make_uint4(c.x, c.y, 0u, 0u);
    }
    r.step = a.err_steps[e0 / BLOCK];
  } else {
    const uint4* ep = reinterpret_cast<const uint4*>(a.err + e0);
#pragma unroll
    for (int i = 0; i < EL / 4; ++i) r.e[i] = ld_stream(ep + i);
  }
}

template <bool BF16, bool E8, int EL>
__device__ __forceinline__ void unpack_raw(const RawChunk<BF16, E8, EL>& r, float neg_zero, f32x2 (&g)[EL / 2],
                                           f32x2 (&e)[EL / 2]) {
#pragma unroll
  for (int i = 0; i < RawChunk<BF16, E8, EL>::kG; ++i) {
    const uint32_t wv[4] = {r.g[i].x, r.g[i].y, r.g[i].z, r.g[i].w};
    if constexpr (BF16) {
#pragma unroll
      for (int c = 0; c < 4; ++c) g[4 * i + c] = pk2(bf16lo_to_f32(wv[c]), bf16hi_to_f32(wv[c]));
    } else {
      g[2 * i] = pk2u(wv[0], wv[1]);
      g[2 * i + 1] = pk2u(wv[2], wv[3]);
    }
  }
  if constexpr (E8) {
    // e = f32(qe) * De: biased floats 2^23 + 128 + qe from byte permutes, the
    // offset subtracted exactly, then the rounded product.
    constexpr uint32_t K = 0x4B000000u;
    const uint32_t cw[4] = {r.e[0].x, r.e[0].y, r.e[0].z, r.e[0].w};
    const f32x2 off = pk2(8388736.0f, 8388736.0f), dp = pk2(r.step, r.step), z = pk2(neg_zero, neg_zero);
#pragma unroll
    for (int w = 0; w < EL / 4; ++w) {
      const uint32_t u = cw[w] ^ 0x80808080u;
      e[2 * w] = prod2(sub2(pk2u(__byte_perm(u, K, 0x7440), __byte_perm(u, K, 0x7441)), off), dp, z);
      e[2 * w + 1] = prod2(sub2(pk2u(__byte_perm(u, K, 0x7442), __byte_perm(u, K, 0x7443)), off), dp, z);
    }
  } else {
#pragma unroll
    for (int i = 0; i < EL / 4; ++i) {
      e[2 * i] = pk2u(r.e[i].x, r.e[i].y);
      e[2 * i + 1] = pk2u(r.e[i].z, r.e[i].w);
    }
  }
}

// Loads of warp tile t for this lane (a full chunk below n only).
template <bool BF16, bool E8, int BLOCK, int EL>
__device__ __forceinline__ void issue_tile(const CompressArgs& a, int64_t t, int64_t ntiles, int lane,
                                           RawChunk<BF16, E8, EL>& r) {
  const int64_t e0 = t * (32 * EL) + lane * EL;
  if (t < ntiles && e0 + EL <= a.n) load_raw<BF16, E8, BLOCK, EL>(a, e0, r);
}

// Compress this lane's chunk of warp tile t from its loaded words (or, for a
// chunk that crosses n, element by element).
template <int BITS, int BLOCK, bool BF16, bool E8, bool FIXED, int EL>
__device__ __forceinline__ void process_tile(const CompressArgs& a, int64_t t, int64_t n_pad, int lane,
                                             const RawChunk<BF16, E8, EL>& r) {
  const int64_t e0 = t * (32 * EL) + lane * EL;
  f32x2 g[EL / 2], e[EL / 2];
  if (e0 + EL <= a.n)
    unpack_raw<BF16, E8, EL>(r, a.neg_zero, g, e);
  else
    load_partial<BF16, E8, BLOCK, EL>(a, e0, g, e);
  compress_chunk<BITS, BLOCK, E8, FIXED, EL>(a, e0, n_pad, lane, g, e);
}

// Warps walk the bucket's warp tiles (32*EL elements) grid-stride, or in
// groups of G consecutive tiles grid-stride over groups, U tiles per
// iteration with all their loads issued before any compute; every lane of a
// warp takes the same trip count, so the shuffles are always full-warp.  A
// lane whose chunk crosses n (only in the last warp tile) loads it element by
// element instead.  The register budget is the compiler's default for 256
// threads (a minimum-CTA launch bound lets it grow and costs occupancy).
#ifdef LOCO_COMPRESS_MINB  // CTAs per SM the direct-load sender's register budget is fitted for
#define LOCO_COMPRESS_BOUNDS __launch_bounds__(kThreads, LOCO_COMPRESS_MINB)
#else  // the compiler's default budget for 256 threads
#define LOCO_COMPRESS_BOUNDS __launch_bounds__(kThreads)
#endif

#ifndef LOCO_COMPRESS_GROUP
// Consecutive warp tiles each warp takes in turn on buckets of at least
// LOCO_COMPRESS_GROUP_MIN_TILES warp tiles per warp of the resident grid
// (smaller buckets: warp0, warp0 + nwarps, ...; G: G warp0 .. G warp0 + G-1,
// then the group nwarps further on).  Over many tiles the warps drift apart
// and the reads of one DRAM page of g or e arrive from warps far apart in
// time; a group keeps them within one warp.  Groups of 8 against the plain
// order: 0.944 -> 0.966 of the copy rate on the Llama-2-7B bucket, 0.948 ->
// 0.968 at 2^32, 0.957 -> 0.963 at 2^30, TinyLlama 0.943 -> 0.956, Mixtral
// 0.948 -> 0.964 (16: about the same, 32: slower).  (The staged int8-error
// variant measured slower with groups.)
#define LOCO_COMPRESS_GROUP 8
#endif
#ifndef LOCO_COMPRESS_GROUP_MIN_TILES
#define LOCO_COMPRESS_GROUP_MIN_TILES 64
#endif

template <int BITS, int BLOCK, bool BF16, bool E8, bool FIXED, int U, int EL, int G>
__global__ void LOCO_COMPRESS_BOUNDS k_compress(const CompressArgs a) {
  const int lane = threadIdx.x & 31;
  const int64_t nb = (a.n + BLOCK - 1) / BLOCK;
  const int64_t n_pad = nb * BLOCK;
  const int64_t ntiles = (n_pad + 32 * EL - 1) / (32 * EL);
  const int64_t warp0 = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = (int64_t(gridDim.x) * blockDim.x) >> 5;
  if constexpr (G == 1) {
    for (int64_t tile = warp0; tile < ntiles; tile += U * nwarps) {
      RawChunk<BF16, E8, EL> raw[U];
#pragma unroll
      for (int u = 0; u < U; ++u) issue_tile<BF16, E8, BLOCK, EL>(a, tile + u * nwarps, ntiles, lane, raw[u]);
#pragma unroll
      for (int u = 0; u < U; ++u)
        if (tile + u * nwarps < ntiles) process_tile<BITS, BLOCK, BF16, E8, FIXED, EL>(a, tile + u * nwarps, n_pad, lane, raw[u]);
    }
  } else {
    // Groups of G consecutive warp tiles: this warp's j-th tile is tile j % G of
    // group warp0 + (j / G) * nwarps; an iteration takes U consecutive ones.
    static_assert((G & (G - 1)) == 0 && G % U == 0, "a power-of-two group of whole iterations");
    for (int64_t j = 0;; j += U) {
      const int64_t t0 = (warp0 + (j / G) * nwarps) * G + (j % G);
      if (t0 >= ntiles) break;
      RawChunk<BF16, E8, EL> raw[U];
#pragma unroll
      for (int u = 0; u < U; ++u) issue_tile<BF16, E8, BLOCK, EL>(a, t0 + u, ntiles, lane, raw[u]);
#pragma unroll
      for (int u = 0; u < U; ++u)
        if (t0 + u < ntiles) process_tile<BITS, BLOCK, BF16, E8, FIXED, EL>(a, t0 + u, n_pad, lane, raw[u]);
    }
  }
}

// ---------------------------------------------------------------------------
// Staged variant: every warp streams its own full warp tiles (32*EL elements)
// through S stages of its own shared memory (warp_pipeline): the gradient and
// the stored error of a tile are copied in as 16-byte cp.async pieces by the
// warp's lanes, so S-1 tiles per warp are in flight without holding registers.
// The int8 error's block step of a lane's chunk is read one tile ahead into a
// register.  Tiles that reach past n (at most the last one) take the direct
// path above.  Stage layout: the tile's gradient bytes, then its error bytes.
// ---------------------------------------------------------------------------
template <bool BF16, bool E8, int EL>
struct StagedTile {
  static constexpr int WT = 32 * EL;
  static constexpr int GB = WT * (BF16 ? 2 : 4);  // gradient bytes per tile
  static constexpr int EB = WT * (E8 ? 1 : 4);    // error bytes per tile
  static constexpr int kStage = GB + EB;
  static constexpr int GJ = GB / 16 / 32, EJ = EB / 16 / 32;  // 16-byte pieces per lane
  static_assert(GB % 512 == 0 && EB % 512 == 0, "whole pieces for every lane");
};

#ifndef LOCO_COMPRESS_STAGED_MINB
#define LOCO_COMPRESS_STAGED_MINB(e8) 3  // CTAs per SM the register budget is fitted for
#endif

template <int BITS, int BLOCK, bool BF16, bool E8, bool FIXED, int EL, int S>
__global__ void __launch_bounds__(kThreads, LOCO_COMPRESS_STAGED_MINB(E8)) k_compress_staged(const CompressArgs a) {
  extern __shared__ __align__(16) uint8_t sm[];
  using ST = StagedTile<BF16, E8, EL>;
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  uint8_t* wsm = sm + size_t(warp) * S * ST::kStage;
  const int64_t nb = (a.n + BLOCK - 1) / BLOCK;
  const int64_t n_pad = nb * BLOCK;
  const int64_t ntiles = (n_pad + ST::WT - 1) / ST::WT;
  const int64_t nfull = a.n / ST::WT;  // tiles wholly below n
  const int64_t gw = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t nw = (int64_t(gridDim.x) * blockDim.x) >> 5;
  const uint8_t* gsrc = static_cast<const uint8_t*>(a.grad) + 16 * lane;
  const uint8_t* esrc = (E8 ? reinterpret_cast<const uint8_t*>(a.err_codes) : reinterpret_cast<const uint8_t*>(a.err)) +
                        16 * lane;
  auto issue = [&](uint8_t* st, int64_t tile) {
#pragma unroll
    for (int j = 0; j < ST::GJ; ++j) cp_async16(st + 16 * (lane + 32 * j), gsrc + tile * ST::GB + 512 * j);
#pragma unroll
    for (int j = 0; j < ST::EJ; ++j) cp_async16(st + ST::GB + 16 * (lane + 32 * j), esrc + tile * ST::EB + 512 * j);
  };
  float step = 0.0f;
  if constexpr (E8)
    if (gw < nfull) step = a.err_steps[(gw * ST::WT + lane * EL) / BLOCK];
  warp_pipeline<S>(wsm, ST::kStage, gw, nw, nfull, issue, [&](const uint8_t* st, int64_t tile) {
    RawChunk<BF16, E8, EL> r;
    const uint4* gs = reinterpret_cast<const uint4*>(st + lane * (ST::GB / 32));
#pragma unroll
    for (int i = 0; i < RawChunk<BF16, E8, EL>::kG; ++i) r.g[i] = gs[i];
    const uint4* es = reinterpret_cast<const uint4*>(st + ST::GB + lane * (ST::EB / 32));
    if constexpr (E8) {
      if constexpr (EL == 16) {
        r.e[0] = es[0];
      } else {
        const uint2 c = *reinterpret_cast<const uint2*>(es);
        r.e[0] = make_uint4(c.x, c.y, 0u, 0u);
      }
      r.step = step;
      if (tile + nw < nfull) step = a.err_steps[((tile + nw) * ST::WT + lane * EL) / BLOCK];
    } else {
#pragma unroll
      for (int i = 0; i < EL / 4; ++i) r.e[i] = es[i];
    }
    f32x2 g[EL / 2], e[EL / 2];
    unpack_raw<BF16, E8, EL>(r, a.neg_zero, g, e);
    compress_chunk<BITS, BLOCK, E8, FIXED, EL>(a, tile * ST::WT + lane * EL, n_pad, lane, g, e);
  });
  // The tiles that reach past n: direct loads, one warp per tile.
  for (int64_t tile = nfull + gw; tile < ntiles; tile += nw) {
    RawChunk<BF16, E8, EL> r;
    issue_tile<BF16, E8, BLOCK, EL>(a, tile, ntiles, lane, r);
    process_tile<BITS, BLOCK, BF16, E8, FIXED, EL>(a, tile, n_pad, lane, r);
  }
}

#ifndef LOCO_COMPRESS_STAGES
#define LOCO_COMPRESS_STAGES 0     // fp32 error: stages of the staged variant (0: direct loads)
#endif
#ifndef LOCO_COMPRESS_STAGES_E8
#define LOCO_COMPRESS_STAGES_E8 6  // int8 error: stages of the staged variant (0: direct loads)
#endif

#ifndef LOCO_COMPRESS_UNROLL
#define LOCO_COMPRESS_UNROLL 2     // fp32 error: 48 bytes per lane per warp tile
#endif
#ifndef LOCO_COMPRESS_ELEMS
#define LOCO_COMPRESS_ELEMS 8      // fp32 error: elements per lane (memory-bound)
#endif
#ifndef LOCO_COMPRESS_UNROLL_E8
#define LOCO_COMPRESS_UNROLL_E8 1  // 8-bit error, direct loads (LOCO_COMPRESS_STAGES_E8 = 0): warp tiles per iteration
#endif
#ifndef LOCO_COMPRESS_ELEMS_E8
#define LOCO_COMPRESS_ELEMS_E8 16  // 8-bit error: elements per lane; the half-warps compute two blocks' scales at once
#endif

// The direct-load sender with tile groups of G: grid of resident CTAs, at
// most one per CTA-worth of warp tiles.
template <int BITS, int BLOCK, bool BF16, bool E8, bool FIXED, int U, int EL, int G>
static cudaError_t direct_grid(const CompressArgs& a, int* grid) {
  static GridCache cache;
  int cap = 0;
  const cudaError_t e =
      grid_cap(cache, reinterpret_cast<const void*>(&k_compress<BITS, BLOCK, BF16, E8, FIXED, U, EL, G>), kThreads, 0, &cap);
  if (e != cudaSuccess) return e;
  const int64_t nb = (a.n + BLOCK - 1) / BLOCK;
  const int64_t warps_needed = (nb * BLOCK + 32 * EL - 1) / (32 * EL);
  const int64_t ctas_needed = (warps_needed + kThreads / 32 - 1) / (kThreads / 32);
  *grid = int(ctas_needed < cap ? ctas_needed : cap);
  return cudaSuccess;
}

template <int BITS, int BLOCK, bool BF16, bool E8, bool FIXED>
static cudaError_t launch_t(const CompressArgs& a, cudaStream_t s) {
  constexpr int U = E8 ? LOCO_COMPRESS_UNROLL_E8 : LOCO_COMPRESS_UNROLL;
  constexpr int EL = E8 ? LOCO_COMPRESS_ELEMS_E8 : LOCO_COMPRESS_ELEMS;
  constexpr int S = E8 ? LOCO_COMPRESS_STAGES_E8 : LOCO_COMPRESS_STAGES;
  if constexpr (S >= 2) {
    constexpr size_t smem = size_t(kThreads / 32) * S * StagedTile<BF16, E8, EL>::kStage;
    static_assert(smem <= 227 * 1024, "staging area exceeds one CTA's shared memory");
    const void* fn = reinterpret_cast<const void*>(&k_compress_staged<BITS, BLOCK, BF16, E8, FIXED, EL, S>);
    static GridCache cache;
    int cap = 0;
    const cudaError_t e = grid_cap(cache, fn, kThreads, smem, &cap);
    if (e != cudaSuccess) return e;
    const int64_t nb = (a.n + BLOCK - 1) / BLOCK;
    const int64_t warps_needed = (nb * BLOCK + 32 * EL - 1) / (32 * EL);
    const int64_t ctas_needed = (warps_needed + kThreads / 32 - 1) / (kThreads / 32);
    const int grid = int(ctas_needed < cap ? ctas_needed : cap);
    k_compress_staged<BITS, BLOCK, BF16, E8, FIXED, EL, S><<<grid, kThreads, smem, s>>>(a);
    return cudaGetLastError();
  } else {
    constexpr int G = LOCO_COMPRESS_GROUP;
    int grid = 0;
    cudaError_t e = direct_grid<BITS, BLOCK, BF16, E8, FIXED, U, EL, 1>(a, &grid);
    if (e != cudaSuccess) return e;
    if constexpr (G > 1) {
      const int64_t nb = (a.n + BLOCK - 1) / BLOCK;
      const int64_t ntiles = (nb * BLOCK + 32 * EL - 1) / (32 * EL);
      if (ntiles / (int64_t(grid) * (kThreads / 32)) >= LOCO_COMPRESS_GROUP_MIN_TILES) {
        e = direct_grid<BITS, BLOCK, BF16, E8, FIXED, U, EL, G>(a, &grid);
        if (e != cudaSuccess) return e;
        k_compress<BITS, BLOCK, BF16, E8, FIXED, U, EL, G><<<grid, kThreads, 0, s>>>(a);
        return cudaGetLastError();
      }
    }
    k_compress<BITS, BLOCK, BF16, E8, FIXED, U, EL, 1><<<grid, kThreads, 0, s>>>(a);
    return cudaGetLastError();
  }
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
