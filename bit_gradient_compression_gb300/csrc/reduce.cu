// Receiver side of LoCo: decode W ranks' packed buckets and average them in
// fp32 ("LoCo: Low-Bit Communication Adaptor for Large-scale Model Training",
// §3.3 Eqn 8), optionally feeding the average straight into one Adam(W) step
// (§4 Eqn 9) so that it never touches HBM.
//
// Mapping: one thread owns 8 consecutive elements: per rank one 4-byte (4-bit)
// or 8-byte (8-bit) code load plus one scale load (shared by the B/8 threads
// of a quant block, served by L1); all W loads are issued before any decode.
// The rank count W is a template parameter so the rank loop unrolls fully and
// the loads of every rank are in flight together.
#include "device_common.cuh"

namespace loco {

template <int BITS, int W>
__global__ void __launch_bounds__(256) k_decode_reduce(const ReduceArgs a, int log2_block) {
  const int64_t nchunks = (a.n + 7) >> 3;
  const int64_t stride = int64_t(gridDim.x) * blockDim.x;
  for (int64_t c = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; c < nchunks; c += stride) {
    const int64_t e0 = c << 3;
    float mean[8];
    decode_mean8<BITS, W>(a.ranks, e0, e0 >> log2_block, mean);
    if (e0 + 8 <= a.n) {
      float4* mp = reinterpret_cast<float4*>(a.mean + e0);
      st_stream(mp, make_float4(mean[0], mean[1], mean[2], mean[3]));
      st_stream(mp + 1, make_float4(mean[4], mean[5], mean[6], mean[7]));
    } else {
#pragma unroll
      for (int j = 0; j < 8; ++j)
        if (e0 + j < a.n) a.mean[e0 + j] = mean[j];
    }
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

template <int BITS, int W>
__global__ void __launch_bounds__(256) k_adam(const AdamArgs a, int log2_block) {
  const int64_t nchunks = (a.n + 7) >> 3;
  const int64_t stride = int64_t(gridDim.x) * blockDim.x;
  for (int64_t c = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; c < nchunks; c += stride) {
    const int64_t e0 = c << 3;
    const bool full = e0 + 8 <= a.n;
    float p[8], m[8], v[8];
    if (full) {
      const float4* pp = reinterpret_cast<const float4*>(a.param + e0);
      const float4* mp = reinterpret_cast<const float4*>(a.m + e0);
      const float4* vp = reinterpret_cast<const float4*>(a.v + e0);
      const float4 p0 = __ldcs(pp), p1 = __ldcs(pp + 1);
      const float4 m0 = __ldcs(mp), m1 = __ldcs(mp + 1);
      const float4 v0 = __ldcs(vp), v1 = __ldcs(vp + 1);
      p[0] = p0.x; p[1] = p0.y; p[2] = p0.z; p[3] = p0.w; p[4] = p1.x; p[5] = p1.y; p[6] = p1.z; p[7] = p1.w;
      m[0] = m0.x; m[1] = m0.y; m[2] = m0.z; m[3] = m0.w; m[4] = m1.x; m[5] = m1.y; m[6] = m1.z; m[7] = m1.w;
      v[0] = v0.x; v[1] = v0.y; v[2] = v0.z; v[3] = v0.w; v[4] = v1.x; v[5] = v1.y; v[6] = v1.z; v[7] = v1.w;
    } else {
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const bool in = e0 + j < a.n;
        p[j] = in ? a.param[e0 + j] : 0.0f;
        m[j] = in ? a.m[e0 + j] : 0.0f;
        v[j] = in ? a.v[e0 + j] : 0.0f;
      }
    }
    float g[8];
    decode_mean8<BITS, W>(a.ranks, e0, e0 >> log2_block, g);
#pragma unroll
    for (int j = 0; j < 8; ++j) adam_elem(a, g[j], p[j], m[j], v[j]);
    if (full) {
      float4* pp = reinterpret_cast<float4*>(a.param + e0);
      float4* mp = reinterpret_cast<float4*>(a.m + e0);
      float4* vp = reinterpret_cast<float4*>(a.v + e0);
      st_stream(pp, make_float4(p[0], p[1], p[2], p[3]));
      st_stream(pp + 1, make_float4(p[4], p[5], p[6], p[7]));
      st_stream(mp, make_float4(m[0], m[1], m[2], m[3]));
      st_stream(mp + 1, make_float4(m[4], m[5], m[6], m[7]));
      st_stream(vp, make_float4(v[0], v[1], v[2], v[3]));
      st_stream(vp + 1, make_float4(v[4], v[5], v[6], v[7]));
    } else {
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        if (e0 + j < a.n) {
          a.param[e0 + j] = p[j];
          a.m[e0 + j] = m[j];
          a.v[e0 + j] = v[j];
        }
      }
    }
  }
}

static int ilog2(int x) {
  int r = 0;
  while ((1 << r) < x) ++r;
  return r;
}

template <typename Args, int BITS, int W, bool ADAM>
static cudaError_t launch_w(const Args& a, cudaStream_t s) {
  const void* fn;
  if constexpr (ADAM)
    fn = reinterpret_cast<const void*>(&k_adam<BITS, W>);
  else
    fn = reinterpret_cast<const void*>(&k_decode_reduce<BITS, W>);
  static const int cap = persistent_grid(fn, 256);
  const int64_t nchunks = (a.n + 7) >> 3;
  const int64_t ctas_needed = (nchunks + 255) / 256;
  const int grid = int(ctas_needed < cap ? ctas_needed : cap);
  if constexpr (ADAM)
    k_adam<BITS, W><<<grid, 256, 0, s>>>(a, ilog2(a.block));
  else
    k_decode_reduce<BITS, W><<<grid, 256, 0, s>>>(a, ilog2(a.block));
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
