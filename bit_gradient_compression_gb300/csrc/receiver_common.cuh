// Shared machinery of the receiver kernels of LoCo ("LoCo: Low-Bit
// Communication Adaptor for Large-scale Model Training", §3.3 Eqn 8 and §4):
// decode W ranks' packed buckets, average them in fp32, and either store the
// average or feed it straight into an optimizer step without touching HBM.
//
// Mapping: a CTA of 256 threads consumes tiles of 256*E elements staged in
// shared memory by a multistage cp.async pipeline (coalesced 16-byte pieces of
// every input of the tile); thread t owns elements [t*E, t*E + E) of a tile.
// The rank count W is a template parameter so the rank loop unrolls fully.
#pragma once

#include <cuda_bf16.h>

#include "device_common.cuh"

namespace loco {

// E-element vector helpers (E a multiple of 4, 16-byte aligned when full).
template <int E>
__device__ __forceinline__ void load_vec(const float* p, int64_t e0, int64_t n, bool full, float x[E]) {
  if (full) {
#pragma unroll
    for (int i = 0; i < E / 4; ++i) {
      const float4 v = __ldcs(reinterpret_cast<const float4*>(p + e0) + i);
      x[4 * i] = v.x; x[4 * i + 1] = v.y; x[4 * i + 2] = v.z; x[4 * i + 3] = v.w;
    }
  } else {
#pragma unroll
    for (int j = 0; j < E; ++j) x[j] = (e0 + j < n) ? p[e0 + j] : 0.0f;
  }
}

template <int E>
__device__ __forceinline__ void store_vec(float* p, int64_t e0, int64_t n, bool full, const float x[E]) {
  if (full) {
#pragma unroll
    for (int i = 0; i < E / 4; ++i)
      st_stream(reinterpret_cast<float4*>(p + e0) + i, make_float4(x[4 * i], x[4 * i + 1], x[4 * i + 2], x[4 * i + 3]));
  } else {
#pragma unroll
    for (int j = 0; j < E; ++j)
      if (e0 + j < n) p[e0 + j] = x[j];
  }
}

constexpr int kThreads = 256;

// Shared-memory image of one tile of T = 256*E elements: NF fp32 arrays
// (T floats each), W ranks' packed codes (T*BITS/8 bytes each) and W ranks'
// steps (T/block floats each, room for the smallest block of 64).
template <int BITS, int W, int E, int NF>
struct Tile {
  static constexpr int T = kThreads * E;
  static constexpr int kCodeBytes = T * BITS / 8;
  static constexpr int kScaleMax = T / 64;
  static constexpr size_t kFloatBytes = size_t(NF) * T * 4;
  static constexpr size_t kBytes = kFloatBytes + size_t(W) * kCodeBytes + size_t(W) * kScaleMax * 4;
  uint8_t* base;
  __device__ float* f(int arr) const { return reinterpret_cast<float*>(base) + arr * T; }
  __device__ uint8_t* codes(int w) const { return base + kFloatBytes + w * kCodeBytes; }
  __device__ float* scales(int w) const {
    return reinterpret_cast<float*>(base + kFloatBytes + size_t(W) * kCodeBytes) + w * kScaleMax;
  }
};

// Largest stage count <= want (at least 1) for which `min_ctas` CTAs, each
// with S tiles plus `extra` bytes of shared memory, fit on one SM (228 KB,
// 1 KB reserved per CTA); never more than one CTA's 227 KB limit.
template <int BITS, int W, int E, int NF>
constexpr int fit_stages(int want, size_t extra = 0, int min_ctas = 1) {
  int s = want;
  while (s > 1 && (size_t(s) * Tile<BITS, W, E, NF>::kBytes + extra > size_t(227) * 1024 ||
                   size_t(min_ctas) * (size_t(s) * Tile<BITS, W, E, NF>::kBytes + extra + 1024) > size_t(228) * 1024))
    --s;
  return s;
}

// Starts the cp.async copies of tile `tile` into `dst`: every piece is 16
// bytes and consecutive threads take consecutive pieces, so each warp moves
// 512 contiguous bytes per instruction.  nsc = T/block steps per rank.
template <int BITS, int W, int E, int NF>
__device__ __forceinline__ void issue_tile(const Tile<BITS, W, E, NF>& dst, const float* const* farr,
                                           const RankPtrs& rp, int64_t tile, int nsc, int t) {
  using TL = Tile<BITS, W, E, NF>;
  const int64_t e0 = tile * TL::T;
  static_assert((TL::T / 4) % kThreads == 0, "whole 16-byte pieces per thread");
#pragma unroll
  for (int arr = 0; arr < NF; ++arr) {
#pragma unroll
    for (int q = t; q < TL::T / 4; q += kThreads) cp_async16(dst.f(arr) + 4 * q, farr[arr] + e0 + 4 * q);
  }
  constexpr int kCodePieces = TL::kCodeBytes / 16;
#pragma unroll
  for (int p = t; p < W * kCodePieces; p += kThreads) {
    const int w = p / kCodePieces, q = p % kCodePieces;
    cp_async16(dst.codes(w) + 16 * q, rp.codes[w] + tile * TL::kCodeBytes + 16 * q);
  }
  const int sc_pieces = nsc / 4;
  for (int p = t; p < W * sc_pieces; p += kThreads) {
    const int w = p / sc_pieces, q = p - w * sc_pieces;
    cp_async16(dst.scales(w) + 4 * q, rp.scales[w] + tile * nsc + 4 * q);
  }
}

// Rank average of this thread's E elements of a staged tile.
template <int BITS, int W, int E, int NF>
__device__ __forceinline__ void tile_mean(const Tile<BITS, W, E, NF>& tl, int t, int log2_block, float neg_zero,
                                          float out[E]) {
  ChunkCodes<BITS, E> cw[W];
  float sc[W];
  const int blk = (t * E) >> log2_block;
#pragma unroll
  for (int w = 0; w < W; ++w) {
    cw[w].load_shared(tl.codes(w) + (t * E * BITS >> 3));
    sc[w] = tl.scales(w)[blk];
  }
  mean_of_codes<BITS, W, E>(cw, sc, neg_zero, out);
}

// Receiver tiles through the multistage pipeline; elements past the last full
// tile are handled by `tail` in one CTA.  `before`/`after` run for thread-level
// set-up and hand-off around each tile (see pipeline_tiles).
template <int BITS, int W, int E, int NF, int S, typename Body, typename TailFn, typename Before, typename After>
__device__ __forceinline__ void tile_pipeline(const float* const* farr, const RankPtrs& rp, int64_t n, int log2_block,
                                              Body body, TailFn tail, Before before, After after) {
  extern __shared__ __align__(16) uint8_t sm[];
  using TL = Tile<BITS, W, E, NF>;
  const int t = threadIdx.x;
  const int64_t ntiles = n / TL::T;
  const int nsc = TL::T >> log2_block;
  pipeline_tiles<S>(
      sm, TL::kBytes, ntiles,
      [&](uint8_t* st, int64_t tile) { issue_tile<BITS, W, E, NF>(TL{st}, farr, rp, tile, nsc, t); },
      [&](uint8_t* st, int64_t tile) { body(TL{st}, tile * TL::T + int64_t(t) * E); }, before, after);
  if (ntiles * TL::T < n && blockIdx.x == ntiles % gridDim.x) {
    const int64_t e0 = ntiles * TL::T + int64_t(t) * E;
    if (e0 < n) tail(e0);
  }
}

// Same walk with the results written back into the staged fp32 arrays and
// shipped by `flush` (see pipeline_tiles_inplace).
template <int BITS, int W, int E, int NF, int S, typename Body, typename TailFn, typename Flush>
__device__ __forceinline__ void tile_pipeline_inplace(const float* const* farr, const RankPtrs& rp, int64_t n,
                                                      int log2_block, Body body, TailFn tail, Flush flush) {
  extern __shared__ __align__(16) uint8_t sm[];
  using TL = Tile<BITS, W, E, NF>;
  const int t = threadIdx.x;
  const int64_t ntiles = n / TL::T;
  const int nsc = TL::T >> log2_block;
  pipeline_tiles_inplace<S>(
      sm, TL::kBytes, ntiles,
      [&](uint8_t* st, int64_t tile) { issue_tile<BITS, W, E, NF>(TL{st}, farr, rp, tile, nsc, t); },
      [&](uint8_t* st, int64_t tile) { body(TL{st}, tile * TL::T + int64_t(t) * E); },
      [&](uint8_t* st, int64_t tile) { flush(TL{st}, tile); });
  if (ntiles * TL::T < n && blockIdx.x == ntiles % gridDim.x) {
    const int64_t e0 = ntiles * TL::T + int64_t(t) * E;
    if (e0 < n) tail(e0);
  }
}

template <int BITS, int W, int E, int NF, int S, typename Body, typename TailFn>
__device__ __forceinline__ void tile_pipeline(const float* const* farr, const RankPtrs& rp, int64_t n, int log2_block,
                                              Body body, TailFn tail) {
  tile_pipeline<BITS, W, E, NF, S>(farr, rp, n, log2_block, body, tail, [](int64_t) {}, [](int64_t) {});
}

// bf16 copy of E updated parameters (round to nearest even).
template <int E>
__device__ __forceinline__ void store_bf16(uint16_t* dst, int64_t e0, int64_t n, bool full, const float p[E]) {
  uint32_t w[E / 2];
#pragma unroll
  for (int j = 0; j < E / 2; ++j)
    w[j] = uint32_t(__bfloat16_as_ushort(__float2bfloat16_rn(p[2 * j]))) |
           (uint32_t(__bfloat16_as_ushort(__float2bfloat16_rn(p[2 * j + 1]))) << 16);
  if (full) {
#pragma unroll
    for (int i = 0; i < E / 8; ++i)
      st_stream(reinterpret_cast<uint4*>(dst + e0) + i, make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]));
  } else {
#pragma unroll
    for (int j = 0; j < E; ++j)
      if (e0 + j < n) dst[e0 + j] = uint16_t(w[j / 2] >> (16 * (j & 1)));
  }
}

static inline int ilog2_int(int x) {
  int r = 0;
  while ((1 << r) < x) ++r;
  return r;
}

static inline int clamp_grid(int64_t n, int elems_per_cta, int cap) {
  const int64_t need = (n + elems_per_cta - 1) / elems_per_cta;
  return int(need < cap ? need : cap);
}

// Dispatch of a runtime rank count to a template parameter 1..16.
template <template <int> class F, typename... A>
static cudaError_t dispatch_w(int W, A&&... args) {
  switch (W) {
#define LOCO_CASE(w) \
  case w: return F<w>::run(args...);
    LOCO_CASE(1) LOCO_CASE(2) LOCO_CASE(3) LOCO_CASE(4) LOCO_CASE(5) LOCO_CASE(6) LOCO_CASE(7) LOCO_CASE(8)
    LOCO_CASE(9) LOCO_CASE(10) LOCO_CASE(11) LOCO_CASE(12) LOCO_CASE(13) LOCO_CASE(14) LOCO_CASE(15) LOCO_CASE(16)
#undef LOCO_CASE
  }
  return cudaErrorInvalidValue;
}

}  // namespace loco
