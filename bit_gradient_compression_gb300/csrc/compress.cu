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
// warp must call this together (the absmax is a warp shuffle).
template <int BITS, int BLOCK>
__device__ __forceinline__ void compress8(const CompressArgs& a, int64_t e0, int64_t n_pad, int lane, const float g[8],
                                          const float e[8]) {
  constexpr int G = BLOCK / 8;  // lanes per quant block
  constexpr float QMAX = float((1 << (BITS - 1)) - 1);
  constexpr float QMIN = -float(1 << (BITS - 1));
  constexpr uint32_t FIELD = (1u << BITS) - 1u;

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
  if (a.fixed) {
    delta = a.fixed_delta;
    inv = a.fixed_inv;
  } else if (amax == 0.0f) {
    delta = 0.0f;
    inv = 0.0f;
  } else {
    delta = __fdiv_rn(amax, QMAX);
    inv = __fdiv_rn(QMAX, amax);
  }
  const float de = __fdiv_rn(delta, a.kappa);
  const float elo = __fmul_rn(-128.0f, de);
  const float ehi = __fmul_rn(127.0f, de);

  // Eqns (1),(3),(4),(5),(7) per element.
  uint32_t packed[BITS == 4 ? 1 : 2] = {};
  float en[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    float x = __fmul_rn(h[j], inv);
    x = fminf(fmaxf(x, QMIN), QMAX);
    const float t = __fadd_rn(x, kRoundMagic);  // rint, halves to even
    const uint32_t code = __float_as_uint(t) & FIELD;
    if constexpr (BITS == 4)
      packed[0] |= code << (4 * j);
    else
      packed[j >> 2] |= code << (8 * (j & 3));
    const float q = __fsub_rn(t, kRoundMagic);
    const float d = __fmul_rn(q, delta);
    const float r = __fsub_rn(h[j], d);
    float v = __fadd_rn(__fmul_rn(a.beta, e[j]), __fmul_rn(a.one_minus_beta, r));
    v = (v < elo) ? elo : v;
    v = (v > ehi) ? ehi : v;
    en[j] = a.reset ? 0.0f : v;
  }

  // Stores: codes and the block step inside the padded code range, the error
  // only for elements < n.
  if (e0 < n_pad) {
    if constexpr (BITS == 4)
      st_stream(reinterpret_cast<uint32_t*>(a.codes + (e0 >> 1)), packed[0]);
    else
      st_stream(reinterpret_cast<uint2*>(a.codes + e0), make_uint2(packed[0], packed[1]));
    if ((lane & (G - 1)) == 0) a.scales[e0 / BLOCK] = delta;
  }
  if (e0 + 8 <= a.n) {
    float4* ep = reinterpret_cast<float4*>(a.err + e0);
    st_stream(ep, make_float4(en[0], en[1], en[2], en[3]));
    st_stream(ep + 1, make_float4(en[4], en[5], en[6], en[7]));
  } else {
#pragma unroll
    for (int j = 0; j < 8; ++j)
      if (e0 + j < a.n) a.err[e0 + j] = en[j];
  }
}

// Loads the 8 gradient and error values of the lane's chunk at e0 (0 past n).
template <bool BF16>
__device__ __forceinline__ void load8(const CompressArgs& a, int64_t e0, float g[8], float e[8]) {
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

// Warps walk the bucket's 256-element warp tiles grid-stride, U tiles per
// iteration with all their loads issued before any compute; every lane of a
// warp takes the same trip count, so the shuffles are always full-warp.
template <int BITS, int BLOCK, bool BF16, int U>
__global__ void __launch_bounds__(kThreads) k_compress(const CompressArgs a) {
  const int lane = threadIdx.x & 31;
  const int64_t nb = (a.n + BLOCK - 1) / BLOCK;
  const int64_t n_pad = nb * BLOCK;
  const int64_t ntiles = (n_pad + 255) / 256;
  const int64_t warp0 = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = (int64_t(gridDim.x) * blockDim.x) >> 5;
  for (int64_t tile = warp0; tile < ntiles; tile += U * nwarps) {
    float g[U][8], e[U][8];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t tu = tile + u * nwarps;
      if (tu < ntiles) load8<BF16>(a, tu * 256 + lane * 8, g[u], e[u]);
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t tu = tile + u * nwarps;
      if (tu < ntiles) compress8<BITS, BLOCK>(a, tu * 256 + lane * 8, n_pad, lane, g[u], e[u]);
    }
  }
}

#ifndef LOCO_COMPRESS_UNROLL
#define LOCO_COMPRESS_UNROLL 2
#endif

template <int BITS, int BLOCK, bool BF16>
static cudaError_t launch_t(const CompressArgs& a, cudaStream_t s) {
  constexpr int U = LOCO_COMPRESS_UNROLL;
  const void* fn = reinterpret_cast<const void*>(&k_compress<BITS, BLOCK, BF16, U>);
  static const int cap = persistent_grid(fn, kThreads);
  const int64_t nb = (a.n + BLOCK - 1) / BLOCK;
  const int64_t warps_needed = (nb * BLOCK + 255) / 256;
  const int64_t ctas_needed = (warps_needed + kThreads / 32 - 1) / (kThreads / 32);
  const int grid = int(ctas_needed < cap ? ctas_needed : cap);
  k_compress<BITS, BLOCK, BF16, U><<<grid, kThreads, 0, s>>>(a);
  return cudaGetLastError();
}

template <int BITS, int BLOCK>
static cudaError_t launch_dt(const CompressArgs& a, cudaStream_t s) {
  return a.grad_bf16 ? launch_t<BITS, BLOCK, true>(a, s) : launch_t<BITS, BLOCK, false>(a, s);
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
