// Receiver side of LoCo: decode W ranks' packed buckets and average them in
// fp32 ("LoCo: Low-Bit Communication Adaptor for Large-scale Model Training",
// §3.3 Eqn 8), optionally feeding the average straight into one Adam(W) step
// (§4 Eqn 9) so that it never touches HBM.
//
// Mapping: one thread owns E consecutive elements: per rank one 4- or 8-byte
// code load plus one scale load (shared by the B/E threads of a quant block,
// served by L1); all W loads are issued before any decode.
// The rank count W is a template parameter so the rank loop unrolls fully and
// the loads of every rank are in flight together.
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

// Shared-memory staging area of one CTA: S stages, each holding, per thread,
// NF fp32 arrays of E elements (as E/4 16-byte slots, slot-major so a warp's
// 16-byte accesses are contiguous) and W ranks' E-element code chunks.
template <int BITS, int W, int E, int S, int NF>
struct Staging {
  static constexpr int CB = ChunkCodes<BITS, E>::kBytes;
  static constexpr int F4 = E / 4;
  static constexpr size_t kFloatBytes = size_t(S) * NF * F4 * kThreads * 16;
  static constexpr size_t kBytes = kFloatBytes + size_t(S) * W * kThreads * CB;
  __device__ static float4* slot(uint8_t* sm, int stage, int arr, int q, int t) {
    return reinterpret_cast<float4*>(sm) + ((stage * NF + arr) * F4 + q) * kThreads + t;
  }
  __device__ static uint8_t* code(uint8_t* sm, int stage, int w, int t) {
    return sm + kFloatBytes + ((size_t(stage) * W + w) * kThreads + t) * CB;
  }
};

// Receiver average (Eqn 8).  Each thread walks its full E-element chunks
// grid-stride and keeps the codes of its next S-1 chunks in flight through
// cp.async; the one ragged chunk at the end (if any) is decoded from global
// memory by the thread whose stride sequence reaches it.
template <int BITS, int W, int E, int S>
__global__ void __launch_bounds__(kThreads) k_decode_reduce(const ReduceArgs a, int log2_block) {
  extern __shared__ __align__(16) uint8_t sm[];
  using St = Staging<BITS, W, E, S, 0>;
  using CC = ChunkCodes<BITS, E>;
  const int t = threadIdx.x;
  const int64_t nfull = a.n / E;
  const int64_t stride = int64_t(gridDim.x) * kThreads;
  const int64_t c0 = int64_t(blockIdx.x) * kThreads + t;

  auto issue = [&](int stage, int64_t c) {
    if (c < nfull) {
#pragma unroll
      for (int w = 0; w < W; ++w) CC::prefetch(St::code(sm, stage, w, t), a.ranks.codes[w], c * E);
    }
    cp_async_commit();
  };
#pragma unroll
  for (int k = 0; k < S - 1; ++k) issue(k, c0 + k * stride);
  int stage = 0;
  for (int64_t c = c0; c < nfull; c += stride) {
    issue(stage == 0 ? S - 1 : stage - 1, c + (S - 1) * stride);
    cp_async_wait<S - 1>();
    const int64_t e0 = c * E;
    CC cw[W];
    float sc[W];
#pragma unroll
    for (int w = 0; w < W; ++w) {
      cw[w].load_shared(St::code(sm, stage, w, t));
      sc[w] = __ldg(a.ranks.scales[w] + (e0 >> log2_block));
    }
    float mean[E];
    mean_of_codes<BITS, W, E>(cw, sc, mean);
    store_vec<E>(a.mean, e0, a.n, true, mean);
    stage = (stage + 1 == S) ? 0 : stage + 1;
  }
  cp_async_wait<0>();
  if (nfull * E < a.n && c0 == nfull % stride) {
    const int64_t e0 = nfull * E;
    float mean[E];
    decode_mean<BITS, W, E>(a.ranks, e0, e0 >> log2_block, mean);
    store_vec<E>(a.mean, e0, a.n, false, mean);
  }
}

// One Adam(W) update of one element, in the order the header states.
__device__ __forceinline__ void adam_elem(const AdamArgs& a, float g, float& p, float& m, float& v) {
  p = __fsub_rn(p, __fmul_rn(a.lr_wd, p));
  m = __fadd_rn(__fmul_rn(a.beta1, m), __fmul_rn(a.one_minus_beta1, g));
  v = __fadd_rn(__fmul_rn(a.beta2, v), __fmul_rn(a.one_minus_beta2, __fmul_rn(g, g)));
  const float mh = __fdiv_rn(m, a.bc1);
  const float vh = __fdiv_rn(v, a.bc2);
  const float den = a.eps_inside_sqrt ? __fsqrt_rn(__fadd_rn(vh, a.eps)) : __fadd_rn(__fsqrt_rn(vh), a.eps);
  p = __fsub_rn(p, __fmul_rn(a.lr, __fdiv_rn(mh, den)));
}

// Receiver average fed to Adam (Eqns 8, 9).  param, m, v and the W code
// chunks of the next S-1 chunks are staged through cp.async; the updated
// param, m, v go straight back to global memory.
template <int BITS, int W, int E, int S>
__global__ void __launch_bounds__(kThreads) k_adam(const AdamArgs a, int log2_block) {
  extern __shared__ __align__(16) uint8_t sm[];
  using St = Staging<BITS, W, E, S, 3>;
  using CC = ChunkCodes<BITS, E>;
  const int t = threadIdx.x;
  const int64_t nfull = a.n / E;
  const int64_t stride = int64_t(gridDim.x) * kThreads;
  const int64_t c0 = int64_t(blockIdx.x) * kThreads + t;

  auto issue = [&](int stage, int64_t c) {
    if (c < nfull) {
      const int64_t e0 = c * E;
#pragma unroll
      for (int q = 0; q < E / 4; ++q) {
        cp_async16(St::slot(sm, stage, 0, q, t), a.param + e0 + 4 * q);
        cp_async16(St::slot(sm, stage, 1, q, t), a.m + e0 + 4 * q);
        cp_async16(St::slot(sm, stage, 2, q, t), a.v + e0 + 4 * q);
      }
#pragma unroll
      for (int w = 0; w < W; ++w) CC::prefetch(St::code(sm, stage, w, t), a.ranks.codes[w], e0);
    }
    cp_async_commit();
  };
#pragma unroll
  for (int k = 0; k < S - 1; ++k) issue(k, c0 + k * stride);
  int stage = 0;
  for (int64_t c = c0; c < nfull; c += stride) {
    issue(stage == 0 ? S - 1 : stage - 1, c + (S - 1) * stride);
    cp_async_wait<S - 1>();
    const int64_t e0 = c * E;
    float p[E], m[E], v[E], g[E];
#pragma unroll
    for (int q = 0; q < E / 4; ++q) {
      const float4 pv = *St::slot(sm, stage, 0, q, t);
      const float4 mv = *St::slot(sm, stage, 1, q, t);
      const float4 vv = *St::slot(sm, stage, 2, q, t);
      p[4 * q] = pv.x; p[4 * q + 1] = pv.y; p[4 * q + 2] = pv.z; p[4 * q + 3] = pv.w;
      m[4 * q] = mv.x; m[4 * q + 1] = mv.y; m[4 * q + 2] = mv.z; m[4 * q + 3] = mv.w;
      v[4 * q] = vv.x; v[4 * q + 1] = vv.y; v[4 * q + 2] = vv.z; v[4 * q + 3] = vv.w;
    }
    CC cw[W];
    float sc[W];
#pragma unroll
    for (int w = 0; w < W; ++w) {
      cw[w].load_shared(St::code(sm, stage, w, t));
      sc[w] = __ldg(a.ranks.scales[w] + (e0 >> log2_block));
    }
    mean_of_codes<BITS, W, E>(cw, sc, g);
#pragma unroll
    for (int j = 0; j < E; ++j) adam_elem(a, g[j], p[j], m[j], v[j]);
    store_vec<E>(a.param, e0, a.n, true, p);
    store_vec<E>(a.m, e0, a.n, true, m);
    store_vec<E>(a.v, e0, a.n, true, v);
    stage = (stage + 1 == S) ? 0 : stage + 1;
  }
  cp_async_wait<0>();
  if (nfull * E < a.n && c0 == nfull % stride) {
    const int64_t e0 = nfull * E;
    float p[E], m[E], v[E], g[E];
    load_vec<E>(a.param, e0, a.n, false, p);
    load_vec<E>(a.m, e0, a.n, false, m);
    load_vec<E>(a.v, e0, a.n, false, v);
    decode_mean<BITS, W, E>(a.ranks, e0, e0 >> log2_block, g);
#pragma unroll
    for (int j = 0; j < E; ++j) adam_elem(a, g[j], p[j], m[j], v[j]);
    store_vec<E>(a.param, e0, a.n, false, p);
    store_vec<E>(a.m, e0, a.n, false, m);
    store_vec<E>(a.v, e0, a.n, false, v);
  }
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
#define LOCO_ADAM_STAGES 3
#endif

template <typename Args, int BITS, int W, bool ADAM>
static cudaError_t launch_w(const Args& a, cudaStream_t s) {
  constexpr int E = ADAM ? LOCO_ADAM_ELEMS(BITS) : LOCO_REDUCE_ELEMS(BITS);
  constexpr int S = ADAM ? LOCO_ADAM_STAGES : LOCO_REDUCE_STAGES;
  constexpr size_t smem = ADAM ? Staging<BITS, W, E, S, 3>::kBytes : Staging<BITS, W, E, S, 0>::kBytes;
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
