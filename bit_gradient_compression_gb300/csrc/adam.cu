// Receiver average of Eqn (8) fed to one Adam(W) step (§4 Eqn 9) of "LoCo:
// Low-Bit Communication Adaptor for Large-scale Model Training": param, m, v,
// codes and steps staged per tile; the updated param, m, v are written back
// into their staged slots and leave as three bulk (TMA) stores per tile (full,
// contiguous lines), the optional bf16 copy of param straight from registers.
#include "receiver_common.cuh"

namespace loco {

#ifndef LOCO_ADAM_ELEMS
#define LOCO_ADAM_ELEMS(bits) 8
#endif
#ifndef LOCO_ADAM_MIN_CTAS
#define LOCO_ADAM_MIN_CTAS 2  // CTAs per SM the stage count is fitted for (measured best)
#endif
#ifndef LOCO_ADAM_STAGES
// Stages wanted; fit_stages takes as many as fit LOCO_ADAM_MIN_CTAS CTAs per
// SM (4 with 4-bit codes up to W = 4, 3 beyond).  Four measured faster than
// three where they fit (4-bit, 2^30 elements: W = 1 0.93 -> 0.95 of the copy
// rate, W = 2 0.98 -> 0.99); two were slower at every W.
#define LOCO_ADAM_STAGES 4
#endif
#ifndef LOCO_ADAM_BULK
#define LOCO_ADAM_BULK 1  // results written back into the stage and shipped by bulk (TMA) stores (0: direct stores)
#endif

// IEEE square root and quotient with a zero operand handled by a select: the
// operation is evaluated on 1 instead and the exact IEEE result put back
// (sqrt(+-0) = +-0; +-0 / d = +-0 for a finite d > 0), so an element whose
// mean gradient has been exactly zero (m = v = 0) does not send its warp down
// the special-value path of the rounded square root or division.  The results
// are those of __fsqrt_rn / __fdiv_rn for every input.  Measured: with 2.5 %
// of the means exactly zero (two ranks' 4-bit codes of Gaussian gradients) the
// step ran at 71 % of the HBM copy rate without the selects and 97 % with them.
__device__ __forceinline__ float sqrt_zsel(float x) {
  const bool z = x == 0.0f;
  const float r = __fsqrt_rn(z ? 1.0f : x);
  return z ? x : r;
}
__device__ __forceinline__ float div_zsel(float n, float d) {
  const bool z = n == 0.0f && d > 0.0f && d < INFINITY;
  const float r = __fdiv_rn(z ? 1.0f : n, d);
  return z ? n : r;
}

// One Adam(W) update of one element, in the order the header states.
__device__ __forceinline__ void adam_elem(const AdamArgs& a, float g, float& p, float& m, float& v) {
  p = __fsub_rn(p, __fmul_rn(a.lr_wd, p));
  m = __fadd_rn(__fmul_rn(a.beta1, m), __fmul_rn(a.one_minus_beta1, g));
  v = __fadd_rn(__fmul_rn(a.beta2, v), __fmul_rn(a.one_minus_beta2, __fmul_rn(g, g)));
  const float den = a.eps_inside_sqrt ? sqrt_zsel(__fadd_rn(__fmul_rn(v, a.c2), a.eps))
                                      : __fadd_rn(__fmul_rn(sqrt_zsel(v), a.c2), a.eps);
  p = __fsub_rn(p, __fmul_rn(a.c1, div_zsel(m, den)));
}

// Three CTAs per SM is what the two-stage staging allows; the bound keeps every
// rank count within the matching register budget (one instantiation otherwise
// took 96 registers and ran at two CTAs per SM).
template <int BITS, int W, int E, int S, bool BF16OUT, bool BULK>
__global__ void __launch_bounds__(kThreads, 3) k_adam(const AdamArgs a, int log2_block) {
  using TL = Tile<BITS, W, E, 3>;
  const float* farr[3] = {a.param, a.m, a.v};
  auto body = [&](const TL& tl, int64_t e0) {
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
    tile_mean<BITS, W, E, 3>(tl, t, log2_block, a.ranks.neg_zero, g);
#pragma unroll
    for (int j = 0; j < E; ++j) adam_elem(a, g[j], p[j], m[j], v[j]);
    if constexpr (BULK) {
      // results back into the thread's own staged slots; thread 0 ships them
#pragma unroll
      for (int q = 0; q < E / 4; ++q) {
        reinterpret_cast<float4*>(tl.f(0) + t * E)[q] = make_float4(p[4 * q], p[4 * q + 1], p[4 * q + 2], p[4 * q + 3]);
        reinterpret_cast<float4*>(tl.f(1) + t * E)[q] = make_float4(m[4 * q], m[4 * q + 1], m[4 * q + 2], m[4 * q + 3]);
        reinterpret_cast<float4*>(tl.f(2) + t * E)[q] = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
      }
    } else {
      store_vec<E>(a.param, e0, a.n, true, p);
      store_vec<E>(a.m, e0, a.n, true, m);
      store_vec<E>(a.v, e0, a.n, true, v);
    }
    if constexpr (BF16OUT) store_bf16<E>(a.param_bf16, e0, a.n, true, p);
  };
  auto tail = [&](int64_t e0) {
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
    if constexpr (BF16OUT) store_bf16<E>(a.param_bf16, e0, a.n, full, p);
  };
  if constexpr (BULK) {
    tile_pipeline_inplace<BITS, W, E, 3, S>(farr, a.ranks, a.n, log2_block, body, tail,
                                            [&](const TL& tl, int64_t tile) {
                                              const int64_t off = tile * TL::T;
                                              bulk_store(a.param + off, tl.f(0), uint32_t(TL::T * 4));
                                              bulk_store(a.m + off, tl.f(1), uint32_t(TL::T * 4));
                                              bulk_store(a.v + off, tl.f(2), uint32_t(TL::T * 4));
                                              bulk_commit();
                                            });
  } else {
    tile_pipeline<BITS, W, E, 3, S>(farr, a.ranks, a.n, log2_block, body, tail);
  }
}

template <int BITS, bool BF16OUT>
struct AdamLaunch {
  template <int W>
  struct F {
    static cudaError_t run(const AdamArgs& a, cudaStream_t s) {
      constexpr int E = LOCO_ADAM_ELEMS(BITS);
      constexpr int S = fit_stages<BITS, W, E, 3>(LOCO_ADAM_STAGES, 0, LOCO_ADAM_MIN_CTAS);
      constexpr size_t smem = S * Tile<BITS, W, E, 3>::kBytes;
      static_assert(smem <= 227 * 1024, "staging area exceeds one CTA's shared memory");
      constexpr bool BULK = LOCO_ADAM_BULK != 0 && S >= 2;  // one stage: no room to refill behind a bulk store
      const void* fn = reinterpret_cast<const void*>(&k_adam<BITS, W, E, S, BF16OUT, BULK>);
      static GridCache cache;
      int cap = 0;
      const cudaError_t e = grid_cap(cache, fn, kThreads, smem, &cap);
      if (e != cudaSuccess) return e;
      k_adam<BITS, W, E, S, BF16OUT, BULK><<<clamp_grid(a.n, kThreads * E, cap), kThreads, smem, s>>>(a, ilog2_int(a.block));
      return cudaGetLastError();
    }
  };
};

cudaError_t launch_adam(const AdamArgs& a, cudaStream_t s) {
  if (a.param_bf16 != nullptr)
    return a.bits == 4 ? dispatch_w<AdamLaunch<4, true>::F>(a.W, a, s) : dispatch_w<AdamLaunch<8, true>::F>(a.W, a, s);
  return a.bits == 4 ? dispatch_w<AdamLaunch<4, false>::F>(a.W, a, s) : dispatch_w<AdamLaunch<8, false>::F>(a.W, a, s);
}

}  // namespace loco
