// Internal interface between the C ABI (abi.cu) and the kernel launchers.
// Not installed; the public interface is include/loco.h.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

namespace loco {

constexpr int kMaxRanks = 16;

// Everything the sender kernel needs, resolved on the host.
struct CompressArgs {
  const void* grad;
  float* err;          // fp32 error (nullptr with 8-bit storage)
  int8_t* err_codes;   // 8-bit error codes (nullptr with fp32 storage)
  float* err_steps;    // per-block step of the 8-bit error codes
  uint8_t* codes;
  float* scales;
  int64_t n;
  int bits;
  int block;
  int grad_bf16;
  int fixed;          // 1: one fixed step for every block
  float fixed_delta;  // 1/s (host fp32 division)
  float fixed_inv;    // s
  float beta;
  float one_minus_beta;  // 1 - beta, formed once in fp32
  float kappa;
  float kappa_recip;  // 1/kappa when kappa is a power of two (then Delta/kappa = Delta * (1/kappa) exactly), else 0
  int reset;          // this step zeroes the stored error
  float neg_zero;     // -0.0f at run time: addend of the packed products (see device_common.cuh)
};

struct RankPtrs {
  const uint8_t* codes[kMaxRanks];
  const float* scales[kMaxRanks];
  // -0.0f, passed at run time: the addend of the packed product q * Delta
  // (fma(q, Delta, -0) rounds exactly like the product, and a value the code
  // generator cannot see keeps it from merging the product into the rank sum).
  float neg_zero;
};

struct ReduceArgs {
  RankPtrs ranks;
  int W;
  int64_t n;
  int bits;
  int block;
  float* mean;
};

struct AdamArgs {
  RankPtrs ranks;
  int W;
  int64_t n;
  int bits;
  int block;
  float* param;
  float* m;
  float* v;
  uint16_t* param_bf16;  // optional bf16 copy of the updated param (nullptr: none)
  float beta1, beta2;
  float one_minus_beta1, one_minus_beta2;
  float lr_wd;
  float c1;  // lr / (1 - beta1^t)
  float c2;  // 1 / sqrt(1 - beta2^t), or 1 / (1 - beta2^t) with eps inside the root
  float eps;
  int eps_inside_sqrt;
};

struct SgdArgs {
  RankPtrs ranks;
  int W;
  int64_t n;
  int bits;
  int block;
  float* param;
  uint16_t* param_bf16;  // optional bf16 copy of the updated param (nullptr: none)
  float lr;
};

cudaError_t launch_compress(const CompressArgs& a, cudaStream_t s);
cudaError_t launch_decode_reduce(const ReduceArgs& a, cudaStream_t s);
cudaError_t launch_adam(const AdamArgs& a, cudaStream_t s);
cudaError_t launch_sgd(const SgdArgs& a, cudaStream_t s);

// Launch shape of one kernel instantiation, kept per device: resident CTAs per
// SM x SMs of that device (0 = not yet computed there).
struct GridCache {
  static constexpr int kDevices = 64;
  std::atomic<int> cap[kDevices];
};

// Grid cap of a persistent grid-stride kernel on the current device.  The
// first call per device raises the kernel's dynamic shared-memory limit when
// smem_bytes exceeds the 48 KB default and queries occupancy; a failure of
// either is returned (and nothing is cached).  Devices with an ordinal beyond
// GridCache::kDevices are queried on every call.
cudaError_t grid_cap(GridCache& cache, const void* kernel, int threads, size_t smem_bytes, int* cap);

}  // namespace loco
