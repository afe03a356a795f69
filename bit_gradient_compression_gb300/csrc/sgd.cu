// Receiver average of Eqn (8) fed to one LoCo-SGD step (§4 of "LoCo: Low-Bit
// Communication Adaptor for Large-scale Model Training": theta = theta -
// eta * g~): param, codes and steps staged per tile; the updated param is
// written back into its staged slots and leaves as one bulk (TMA) store per
// tile, the optional bf16 copy straight from registers.
#include "receiver_common.cuh"

namespace loco {

#ifndef LOCO_SGD_ELEMS
#define LOCO_SGD_ELEMS(bits) (64 / (bits))
#endif
#ifndef LOCO_SGD_MIN_CTAS
// CTAs per SM the stage count is fitted for (measured best).  For 9..12 ranks
// of 4-bit codes three CTAs would leave room for one unpipelined stage; two
// CTAs with two stages measured faster there (W = 12: 81 % -> 88 %), and at
// W = 8 (three stages instead of two: 99 % -> 100 %), but not at 13..16 ranks
// (W = 16: 93 % with three CTAs, 87 % with two) nor below 8.
#define LOCO_SGD_MIN_CTAS(bits, w) ((bits) == 4 && (w) >= 8 && (w) <= 12 ? 2 : 3)
#endif
#ifndef LOCO_SGD_STAGES
// Stages wanted; fit_stages takes as many as fit (4-bit codes: 4 at W = 1).
// Four measured faster than three where they fit (4-bit W = 1: 0.95 -> 1.00).
#define LOCO_SGD_STAGES 4
#endif
#ifndef LOCO_SGD_BULK
#define LOCO_SGD_BULK 1  // the updated param written back into the stage and shipped by a bulk (TMA) store (0: direct)
#endif

template <int BITS, int W, int E, int S, bool BF16OUT, bool BULK>
__global__ void __launch_bounds__(kThreads) k_sgd(const SgdArgs a, int log2_block) {
  using TL = Tile<BITS, W, E, 1>;
  const float* farr[1] = {a.param};
  auto body = [&](const TL& tl, int64_t e0) {
    const int t = threadIdx.x;
    float p[E], g[E];
#pragma unroll
    for (int q = 0; q < E / 4; ++q) {
      const float4 pv = reinterpret_cast<const float4*>(tl.f(0) + t * E)[q];
      p[4 * q] = pv.x; p[4 * q + 1] = pv.y; p[4 * q + 2] = pv.z; p[4 * q + 3] = pv.w;
    }
    tile_mean<BITS, W, E, 1>(tl, t, log2_block, a.ranks.neg_zero, g);
#pragma unroll
    for (int j = 0; j < E; ++j) p[j] = __fsub_rn(p[j], __fmul_rn(a.lr, g[j]));
    if constexpr (BULK) {
#pragma unroll
      for (int q = 0; q < E / 4; ++q)
        reinterpret_cast<float4*>(tl.f(0) + t * E)[q] = make_float4(p[4 * q], p[4 * q + 1], p[4 * q + 2], p[4 * q + 3]);
    } else {
      store_vec<E>(a.param, e0, a.n, true, p);
    }
    if constexpr (BF16OUT) store_bf16<E>(a.param_bf16, e0, a.n, true, p);
  };
  auto tail = [&](int64_t e0) {
    const bool full = e0 + E <= a.n;
    float p[E], g[E];
    load_vec<E>(a.param, e0, a.n, full, p);
    decode_mean<BITS, W, E>(a.ranks, e0, e0 >> log2_block, g);
#pragma unroll
    for (int j = 0; j < E; ++j) p[j] = __fsub_rn(p[j], __fmul_rn(a.lr, g[j]));
    store_vec<E>(a.param, e0, a.n, full, p);
    if constexpr (BF16OUT) store_bf16<E>(a.param_bf16, e0, a.n, full, p);
  };
  if constexpr (BULK) {
    tile_pipeline_inplace<BITS, W, E, 1, S>(farr, a.ranks, a.n, log2_block, body, tail,
                                            [&](const TL& tl, int64_t tile) {
                                              bulk_store(a.param + tile * TL::T, tl.f(0), uint32_t(TL::T * 4));
                                              bulk_commit();
                                            });
  } else {
    tile_pipeline<BITS, W, E, 1, S>(farr, a.ranks, a.n, log2_block, body, tail);
  }
}

template <int BITS, bool BF16OUT>
struct SgdLaunch {
  template <int W>
  struct F {
    static cudaError_t run(const SgdArgs& a, cudaStream_t s) {
      constexpr int E = LOCO_SGD_ELEMS(BITS);
      constexpr int S = fit_stages<BITS, W, E, 1>(LOCO_SGD_STAGES, 0, LOCO_SGD_MIN_CTAS(BITS, W));
      constexpr size_t smem = S * Tile<BITS, W, E, 1>::kBytes;
      static_assert(smem <= 227 * 1024, "staging area exceeds one CTA's shared memory");
      constexpr bool BULK = LOCO_SGD_BULK != 0 && S >= 2;  // one stage: no room to refill behind a bulk store
      const void* fn = reinterpret_cast<const void*>(&k_sgd<BITS, W, E, S, BF16OUT, BULK>);
      static GridCache cache;
      int cap = 0;
      const cudaError_t e = grid_cap(cache, fn, kThreads, smem, &cap);
      if (e != cudaSuccess) return e;
      k_sgd<BITS, W, E, S, BF16OUT, BULK><<<clamp_grid(a.n, kThreads * E, cap), kThreads, smem, s>>>(a, ilog2_int(a.block));
      return cudaGetLastError();
    }
  };
};

cudaError_t launch_sgd(const SgdArgs& a, cudaStream_t s) {
  if (a.param_bf16 != nullptr)
    return a.bits == 4 ? dispatch_w<SgdLaunch<4, true>::F>(a.W, a, s) : dispatch_w<SgdLaunch<8, true>::F>(a.W, a, s);
  return a.bits == 4 ? dispatch_w<SgdLaunch<4, false>::F>(a.W, a, s) : dispatch_w<SgdLaunch<8, false>::F>(a.W, a, s);
}

}  // namespace loco
