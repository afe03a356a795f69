// Receiver side of LoCo: decode W ranks' packed buckets and average them in
// fp32 ("LoCo: Low-Bit Communication Adaptor for Large-scale Model Training",
// §3.3 Eqn 8), optionally feeding the average straight into one Adam(W) step
// (§4 Eqn 9) so that it never touches HBM.
//
// Mapping: a CTA of 256 threads consumes tiles of 256*E elements staged in
// shared memory by a multistage cp.async pipeline (coalesced 16-byte pieces of
// every input of the tile); thread t owns elements [t*E, t*E + E) of a tile.
// The rank count W is a template parameter so the rank loop unrolls fully.
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

// Largest stage count <= want whose tiles fit one CTA's shared memory.
template <int BITS, int W, int E, int NF>
constexpr int fit_stages(int want) {
  int s = want;
  while (s > 1 && size_t(s) * Tile<BITS, W, E, NF>::kBytes > size_t(227) * 1024) --s;
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
__device__ __forceinline__ void tile_mean(const Tile<BITS, W, E, NF>& tl, int t, int log2_block, float out[E]) {
  ChunkCodes<BITS, E> cw[W];
  float sc[W];
  const int blk = (t * E) >> log2_block;
#pragma unroll
  for (int w = 0; w < W; ++w) {
    cw[w].load_shared(tl.codes(w) + (t * E * BITS >> 3));
    sc[w] = tl.scales(w)[blk];
  }
  mean_of_codes<BITS, W, E>(cw, sc, out);
}

// Receiver tiles through the multistage pipeline; elements past the last full
// tile are handled by `tail` in one CTA.
template <int BITS, int W, int E, int NF, int S, typename Body, typename TailFn>
__device__ __forceinline__ void tile_pipeline(const float* const* farr, const RankPtrs& rp, int64_t n, int log2_block,
                                              Body body, TailFn tail) {
  extern __shared__ __align__(16) uint8_t sm[];
  using TL = Tile<BITS, W, E, NF>;
  const int t = threadIdx.x;
  const int64_t ntiles = n / TL::T;
  const int nsc = TL::T >> log2_block;
  pipeline_tiles<S>(
      sm, TL::kBytes, ntiles,
      [&](uint8_t* st, int64_t tile) { issue_tile<BITS, W, E, NF>(TL{st}, farr, rp, tile, nsc, t); },
      [&](uint8_t* st, int64_t tile) { body(TL{st}, tile * TL::T + int64_t(t) * E); });
  if (ntiles * TL::T < n && blockIdx.x == ntiles % gridDim.x) {
    const int64_t e0 = ntiles * TL::T + int64_t(t) * E;
    if (e0 < n) tail(e0);
  }
}

// Receiver average (Eqn 8): codes and steps staged per tile, the mean stored
// straight from registers.
template <int BITS, int W, int E, int S>
__global__ void __launch_bounds__(kThreads) k_decode_reduce(const ReduceArgs a, int log2_block) {
  using TL = Tile<BITS, W, E, 0>;
  const float* none[1] = {nullptr};
  tile_pipeline<BITS, W, E, 0, S>(
      none, a.ranks, a.n, log2_block,
      [&](const TL& tl, int64_t e0) {
        float mean[E];
        tile_mean<BITS, W, E, 0>(tl, threadIdx.x, log2_block, mean);
        store_vec<E>(a.mean, e0, a.n, true, mean);
      },
      [&](int64_t e0) {
        float mean[E];
        decode_mean<BITS, W, E>(a.ranks, e0, e0 >> log2_block, mean);
        store_vec<E>(a.mean, e0, a.n, e0 + E <= a.n, mean);
      });
}

// One Adam(W) update of one element, in the order the header states.
__device__ __forceinline__ void adam_elem(const AdamArgs& a, float g, float& p, float& m, float& v) {
  p = __fsub_rn(p, __fmul_rn(a.lr_wd, p));
  m = __fadd_rn(__fmul_rn(a.beta1, m), __fmul_rn(a.one_minus_beta1, g));
  v = __fadd_rn(__fmul_rn(a.beta2, v), __fmul_rn(a.one_minus_beta2, __fmul_rn(g, g)));
  const float den = a.eps_inside_sqrt ? __fsqrt_rn(__fadd_rn(__fmul_rn(v, a.c2), a.eps))
                                      : __fadd_rn(__fmul_rn(__fsqrt_rn(v), a.c2), a.eps);
  p = __fsub_rn(p, __fmul_rn(a.c1, __fdiv_rn(m, den)));
}

// Receiver average fed to Adam (Eqns 8, 9): param, m, v, codes and steps
// staged per tile; the updated param, m, v stored straight from registers.
template <int BITS, int W, int E, int S>
__global__ void __launch_bounds__(kThreads) k_adam(const AdamArgs a, int log2_block) {
  using TL = Tile<BITS, W, E, 3>;
  const float* farr[3] = {a.param, a.m, a.v};
  tile_pipeline<BITS, W, E, 3, S>(
      farr, a.ranks, a.n, log2_block,
      [&](const TL& tl, int64_t e0) {
        const int t = threadIdx.x;
        float p[E], m[E], v[E], g[E];
#pragma unroll
        for (int q = 0; q < E / 4; ++q) {
          const float4 pv = reinterpret_cast<const float4*>(tl.f(0) + t * E)[q];
          const float4 mv = reinterpret_cast<const float4*>(tl.f(1) + t * E)[q];
          const float4 vv = reinterpret_cast<const float4*>(tl.f(2) + t * E)[q];
          p[4 * q] = pv.x; p[4 * q + 1] = pv.y; p[4 * q + 2] = pv.z; p[4 * q + 3] = pv.w;
          m[4 * q] = mv.x; m[4 * q + 1] = mv.y; m[4 * q + 2] = mv.z; m[4 * q + 3] = mv.w;
          v[4 * q] = vv.x; v[4 * q + 1] = vv.y; v[4 * q + 2] = vv.z; v[4 * q + 3] = vv.w;
        }
        tile_mean<BITS, W, E, 3>(tl, t, log2_block, g);
#pragma unroll
        for (int j = 0; j < E; ++j) adam_elem(a, g[j], p[j], m[j], v[j]);
        store_vec<E>(a.param, e0, a.n, true, p);
        store_vec<E>(a.m, e0, a.n, true, m);
        store_vec<E>(a.v, e0, a.n, true, v);
      },
      [&](int64_t e0) {
        const bool full = e0 + E <= a.n;
        float p[E], m[E], v[E], g[E];
        load_vec<E>(a.param, e0, a.n, full, p);
        load_vec<E>(a.m, e0, a.n, full, m);
        load_vec<E>(a.v, e0, a.n, full, v);
        decode_mean<BITS, W, E>(a.ranks, e0, e0 >> log2_block, g);
#pragma unroll
        for (int j = 0; j < E; ++j) adam_elem(a, g[j], p[j], m[j], v[j]);
        store_vec<E>(a.param, e0, a.n, full, p);
        store_vec<E>(a.m, e0, a.n, full, m);
        store_vec<E>(a.v, e0, a.n, full, v);
      });
}

static int ilog2(int x) {
  int r = 0;
  while ((1 << r) < x) ++r;
  return r;
}

#ifndef LOCO_REDUCE_ELEMS
#define LOCO_REDUCE_ELEMS(bits) (64 / (bits))  // elements per thread chunk: 8 code bytes per rank
#endif
#ifndef LOCO_REDUCE_STAGES
#define LOCO_REDUCE_STAGES 4
#endif
#ifndef LOCO_ADAM_ELEMS
#define LOCO_ADAM_ELEMS(bits) 8
#endif
#ifndef LOCO_ADAM_STAGES
#define LOCO_ADAM_STAGES 2
#endif

template <typename Args, int BITS, int W, bool ADAM>
static cudaError_t launch_w(const Args& a, cudaStream_t s) {
  constexpr int E = ADAM ? LOCO_ADAM_ELEMS(BITS) : LOCO_REDUCE_ELEMS(BITS);
  constexpr int S = ADAM ? fit_stages<BITS, W, E, 3>(LOCO_ADAM_STAGES) : fit_stages<BITS, W, E, 0>(LOCO_REDUCE_STAGES);
  constexpr size_t smem = S * (ADAM ? Tile<BITS, W, E, 3>::kBytes : Tile<BITS, W, E, 0>::kBytes);
  static_assert(smem <= 227 * 1024, "staging area exceeds one CTA's shared memory");
  const void* fn;
  if constexpr (ADAM)
    fn = reinterpret_cast<const void*>(&k_adam<BITS, W, E, S>);
  else
    fn = reinterpret_cast<const void*>(&k_decode_reduce<BITS, W, E, S>);
  static const int cap = [&] {
    cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
    return persistent_grid(fn, kThreads, smem);
  }();
  const int64_t nchunks = (a.n + E - 1) / E;
  const int64_t ctas_needed = (nchunks + kThreads - 1) / kThreads;
  const int grid = int(ctas_needed < cap ? ctas_needed : cap);
  if constexpr (ADAM)
    k_adam<BITS, W, E, S><<<grid, kThreads, smem, s>>>(a, ilog2(a.block));
  else
    k_decode_reduce<BITS, W, E, S><<<grid, kThreads, smem, s>>>(a, ilog2(a.block));
  return cudaGetLastError();
}

template <typename Args, int BITS, bool ADAM>
static cudaError_t launch_bits(const Args& a, cudaStream_t s) {
  switch (a.W) {
#define LOCO_CASE(w) \
  case w: return launch_w<Args, BITS, w, ADAM>(a, s);
    LOCO_CASE(1) LOCO_CASE(2) LOCO_CASE(3) LOCO_CASE(4) LOCO_CASE(5) LOCO_CASE(6) LOCO_CASE(7) LOCO_CASE(8)
    LOCO_CASE(9) LOCO_CASE(10) LOCO_CASE(11) LOCO_CASE(12) LOCO_CASE(13) LOCO_CASE(14) LOCO_CASE(15) LOCO_CASE(16)
#undef LOCO_CASE
  }
  return cudaErrorInvalidValue;
}

cudaError_t launch_decode_reduce(const ReduceArgs& a, cudaStream_t s) {
  return a.bits == 4 ? launch_bits<ReduceArgs, 4, false>(a, s) : launch_bits<ReduceArgs, 8, false>(a, s);
}

cudaError_t launch_adam(const AdamArgs& a, cudaStream_t s) {
  return a.bits == 4 ? launch_bits<AdamArgs, 4, true>(a, s) : launch_bits<AdamArgs, 8, true>(a, s);
}

}  // namespace loco
