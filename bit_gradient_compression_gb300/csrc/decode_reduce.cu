// Receiver average of Eqn (8) ("LoCo: Low-Bit Communication Adaptor for
// Large-scale Model Training", §3.3): the W ranks' codes and steps are staged
// per tile by the cp.async pipeline.  Where the fp32 output carries most of
// the bytes, each thread writes its E means into a shared-memory output tile
// and one thread stores the whole tile with a bulk (TMA) copy, so the output
// leaves in full, contiguous lines; otherwise threads store directly.
#include "receiver_common.cuh"

namespace loco {

#ifndef LOCO_REDUCE_ELEMS
#define LOCO_REDUCE_ELEMS(bits) (64 / (bits))  // elements per thread: 8 code bytes per rank
#endif
#ifndef LOCO_REDUCE_MIN_CTAS
#define LOCO_REDUCE_MIN_CTAS 3  // CTAs per SM the stage count is fitted for
#endif

// Output path and pipeline depth per configuration, from measurements over
// W = 1..16 at 2^30 elements.  While the fp32 mean dominates the traffic (8-bit
// codes, or 4-bit codes of up to 4 ranks) it is written through a shared-memory
// tile and one bulk copy per tile; with 4-bit codes of more ranks the kernel is
// bound by the per-code decode work, the extra shared-memory pass costs more
// than it saves, and threads store directly with a deeper load pipeline.
#ifndef LOCO_REDUCE_BULK_MAX_W4
#define LOCO_REDUCE_BULK_MAX_W4 4  // largest rank count whose 4-bit mean goes through the bulk store
#endif
#ifndef LOCO_REDUCE_STAGES8
#define LOCO_REDUCE_STAGES8 2
#endif
#ifndef LOCO_REDUCE_STAGES4_BULK
#define LOCO_REDUCE_STAGES4_BULK 3
#endif
#ifndef LOCO_REDUCE_STAGES4_DIRECT
#define LOCO_REDUCE_STAGES4_DIRECT 4
#endif
template <int BITS, int W>
constexpr bool use_bulk_store() {
  return BITS == 8 || W <= LOCO_REDUCE_BULK_MAX_W4;
}
template <int BITS, int W>
constexpr int wanted_stages() {
  return BITS == 8 ? LOCO_REDUCE_STAGES8
                   : (use_bulk_store<BITS, W>() ? LOCO_REDUCE_STAGES4_BULK : LOCO_REDUCE_STAGES4_DIRECT);
}

template <int BITS, int W, int E>
struct DecodeSmem {
  static constexpr bool kBulk = use_bulk_store<BITS, W>();
  static constexpr size_t kOut = kBulk ? size_t(kThreads) * E * 4 : 0;  // one output tile
  static constexpr int S = fit_stages<BITS, W, E, 0>(wanted_stages<BITS, W>(), kOut, LOCO_REDUCE_MIN_CTAS);
  static constexpr size_t kBytes = size_t(S) * Tile<BITS, W, E, 0>::kBytes + kOut;
};

template <int BITS, int W, int E, int S, bool BULK>
__global__ void __launch_bounds__(kThreads) k_decode_reduce(const ReduceArgs a, int log2_block) {
  extern __shared__ __align__(16) uint8_t sm[];
  using TL = Tile<BITS, W, E, 0>;
  float* out = reinterpret_cast<float*>(sm + size_t(S) * TL::kBytes);
  const float* none[1] = {nullptr};
  const bool leader = threadIdx.x == 0;
  tile_pipeline<BITS, W, E, 0, S>(
      none, a.ranks, a.n, log2_block,
      [&](const TL& tl, int64_t e0) {
        float mean[E];
        tile_mean<BITS, W, E, 0>(tl, threadIdx.x, log2_block, a.ranks.neg_zero, mean);
        if constexpr (BULK) {
          float4* o = reinterpret_cast<float4*>(out + threadIdx.x * E);
#pragma unroll
          for (int q = 0; q < E / 4; ++q)
            o[q] = make_float4(mean[4 * q], mean[4 * q + 1], mean[4 * q + 2], mean[4 * q + 3]);
          fence_smem_to_async_proxy();  // make the tile visible to the bulk copy
        } else {
          store_vec<E>(a.mean, e0, a.n, true, mean);
        }
      },
      [&](int64_t e0) {
        float mean[E];
        decode_mean<BITS, W, E>(a.ranks, e0, e0 >> log2_block, mean);
        store_vec<E>(a.mean, e0, a.n, e0 + E <= a.n, mean);
      },
      // before a tile is published: the previous tile's bulk store has read `out`
      [&](int64_t) {
        if constexpr (BULK)
          if (leader) bulk_wait_read_all();
      },
      // after every thread wrote `out`: one thread ships it
      [&](int64_t tile) {
        if constexpr (BULK) {
          if (leader) {
            bulk_store(a.mean + tile * TL::T, out, uint32_t(TL::T * 4));
            bulk_commit();
          }
        }
      });
  if constexpr (BULK)
    if (leader) bulk_wait_all();
}

template <int BITS>
struct DecodeLaunch {
  template <int W>
  struct F {
    static cudaError_t run(const ReduceArgs& a, cudaStream_t s) {
      constexpr int E = LOCO_REDUCE_ELEMS(BITS);
      using SM = DecodeSmem<BITS, W, E>;
      static_assert(SM::kBytes <= 227 * 1024, "staging area exceeds one CTA's shared memory");
      const void* fn = reinterpret_cast<const void*>(&k_decode_reduce<BITS, W, E, SM::S, SM::kBulk>);
      static GridCache cache;
      int cap = 0;
      const cudaError_t e = grid_cap(cache, fn, kThreads, SM::kBytes, &cap);
      if (e != cudaSuccess) return e;
      k_decode_reduce<BITS, W, E, SM::S, SM::kBulk>
          <<<clamp_grid(a.n, kThreads * E, cap), kThreads, SM::kBytes, s>>>(a, ilog2_int(a.block));
      return cudaGetLastError();
    }
  };
};

cudaError_t launch_decode_reduce(const ReduceArgs& a, cudaStream_t s) {
  return a.bits == 4 ? dispatch_w<DecodeLaunch<4>::F>(a.W, a, s) : dispatch_w<DecodeLaunch<8>::F>(a.W, a, s);
}

}  // namespace loco
