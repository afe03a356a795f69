// Receiver average of Eqn (8) ("LoCo: Low-Bit Communication Adaptor for
// Large-scale Model Training", §3.3): the W ranks' codes and steps are staged
// per tile, the fp32 mean is stored straight from registers.
#include "receiver_common.cuh"

namespace loco {

#ifndef LOCO_REDUCE_ELEMS
#define LOCO_REDUCE_ELEMS(bits) (64 / (bits))  // elements per thread: 8 code bytes per rank
#endif
#ifndef LOCO_REDUCE_STAGES
#define LOCO_REDUCE_STAGES 4
#endif

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

template <int BITS>
struct DecodeLaunch {
  template <int W>
  struct F {
    static cudaError_t run(const ReduceArgs& a, cudaStream_t s) {
      constexpr int E = LOCO_REDUCE_ELEMS(BITS);
      constexpr int S = fit_stages<BITS, W, E, 0>(LOCO_REDUCE_STAGES);
      constexpr size_t smem = S * Tile<BITS, W, E, 0>::kBytes;
      static_assert(smem <= 227 * 1024, "staging area exceeds one CTA's shared memory");
      const void* fn = reinterpret_cast<const void*>(&k_decode_reduce<BITS, W, E, S>);
      static const int cap = receiver_grid(fn, smem);
      k_decode_reduce<BITS, W, E, S><<<clamp_grid(a.n, kThreads * E, cap), kThreads, smem, s>>>(a, ilog2_int(a.block));
      return cudaGetLastError();
    }
  };
};

cudaError_t launch_decode_reduce(const ReduceArgs& a, cudaStream_t s) {
  return a.bits == 4 ? dispatch_w<DecodeLaunch<4>::F>(a.W, a, s) : dispatch_w<DecodeLaunch<8>::F>(a.W, a, s);
}

}  // namespace loco
