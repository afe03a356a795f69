// C ABI of libloco (declared in include/loco.h): argument validation,
// derived constants, and dispatch to the kernel launchers.
//
// Every check happens on the host before anything is launched, so a rejected
// call writes nothing.  Device buffers are checked against the extent of the
// allocation they live in (cuMemGetAddressRange, fetched through the runtime's
// driver entry point so the library has no link-time dependency on libcuda):
// a host pointer, a pointer of another device or a buffer shorter than the
// call needs is an argument error, not a memory fault.
#include <cuda.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include "loco.h"
#include "loco_internal.h"

namespace loco {

static thread_local char g_last_error[512] = "";

static loco_status fail(loco_status st, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_last_error, sizeof g_last_error, fmt, ap);
  va_end(ap);
  return st;
}

cudaError_t grid_cap(GridCache& cache, const void* kernel, int threads, size_t smem_bytes, int* cap) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 0 && dev < GridCache::kDevices) {
    const int c = cache.cap[dev].load(std::memory_order_acquire);
    if (c > 0) {
      *cap = c;
      return cudaSuccess;
    }
  }
  // First launch of this kernel on this device: raise its dynamic shared-memory
  // limit there (the attribute belongs to the device's copy of the kernel) and
  // size the persistent grid from this device's SM count and occupancy.
  if (smem_bytes > 48 * 1024) {
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem_bytes));
    if (e != cudaSuccess) return e;
  }
  int sms = 0, per_sm = 0;
  e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, threads, smem_bytes);
  if (e != cudaSuccess) return e;
  if (sms <= 0 || per_sm <= 0) return cudaErrorInvalidConfiguration;
  *cap = sms * per_sm;
  if (dev >= 0 && dev < GridCache::kDevices) cache.cap[dev].store(*cap, std::memory_order_release);
  return cudaSuccess;
}

typedef CUresult (*AddressRangeFn)(CUdeviceptr*, size_t*, CUdeviceptr);

static AddressRangeFn address_range_fn() {
  static AddressRangeFn fn = []() -> AddressRangeFn {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuMemGetAddressRange", &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return nullptr;
    return reinterpret_cast<AddressRangeFn>(p);
  }();
  return fn;
}

// Null and alignment check (no CUDA call).
static loco_status check_ptr(const void* p, size_t align, const char* name) {
  if (p == nullptr) return fail(LOCO_ERR_INVALID_ARG, "%s is NULL", name);
  if (reinterpret_cast<uintptr_t>(p) % align != 0)
    return fail(LOCO_ERR_MISALIGNED, "%s (%p) is not %zu-byte aligned", name, p, align);
  return LOCO_OK;
}

// Checks that [p, p + bytes) is device memory of the current device inside one
// allocation.  name is used in the error text.
static loco_status check_extent(const void* p, size_t bytes, const char* name) {
  cudaPointerAttributes attr;
  cudaError_t e = cudaPointerGetAttributes(&attr, p);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return fail(LOCO_ERR_INVALID_ARG, "%s: cudaPointerGetAttributes failed: %s", name, cudaGetErrorString(e));
  }
  if (attr.type != cudaMemoryTypeDevice && attr.type != cudaMemoryTypeManaged)
    return fail(LOCO_ERR_INVALID_ARG, "%s (%p) is not device memory", name, p);
  int dev = -1;
  cudaGetDevice(&dev);
  if (attr.type == cudaMemoryTypeDevice && attr.device != dev)
    return fail(LOCO_ERR_INVALID_ARG, "%s lives on device %d but device %d is current", name, attr.device, dev);
  AddressRangeFn range = address_range_fn();
  if (range != nullptr) {
    CUdeviceptr base = 0;
    size_t size = 0;
    if (range(&base, &size, reinterpret_cast<CUdeviceptr>(p)) == CUDA_SUCCESS) {
      const uintptr_t lo = reinterpret_cast<uintptr_t>(p);
      if (lo + bytes > uintptr_t(base) + size)
        return fail(LOCO_ERR_INVALID_ARG, "%s: %zu bytes from %p run past the end of its allocation (%zu bytes at %p)",
                    name, bytes, p, size, reinterpret_cast<void*>(base));
    }
  }
  return LOCO_OK;
}

// A list of buffers checked together: every null/alignment rule first, then
// the device-memory and extent rules, so the status does not depend on which
// buffer happens to be listed first.
struct BufCheck {
  const void* p;
  size_t bytes;
  size_t align;
  const char* name;
};

static loco_status check_buffers(const BufCheck* b, int count) {
  for (int i = 0; i < count; ++i) {
    loco_status st = check_ptr(b[i].p, b[i].align, b[i].name);
    if (st != LOCO_OK) return st;
  }
  for (int i = 0; i < count; ++i) {
    loco_status st = check_extent(b[i].p, b[i].bytes, b[i].name);
    if (st != LOCO_OK) return st;
  }
  return LOCO_OK;
}

static bool overlap(const void* a, size_t na, const void* b, size_t nb) {
  const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
  return x < y + nb && y < x + na;
}

static loco_status check_layout(int32_t bits, int32_t block) {
  if (bits != 4 && bits != 8) return fail(LOCO_ERR_UNSUPPORTED, "bits = %d (supported: 4, 8)", bits);
  if (block != 64 && block != 128 && block != 256)
    return fail(LOCO_ERR_UNSUPPORTED, "block = %d (supported: 64, 128, 256)", block);
  return LOCO_OK;
}

static loco_status launch_result(cudaError_t e, const char* what) {
  if (e != cudaSuccess) return fail(LOCO_ERR_CUDA, "%s launch failed: %s", what, cudaGetErrorString(e));
  g_last_error[0] = '\0';
  return LOCO_OK;
}

static loco_status check_ranks(const loco_config* cfg, const uint8_t* const* codes, const float* const* scales,
                               int32_t W, int64_t n, RankPtrs* out, BufCheck* list, int* count) {
  if (codes == nullptr || scales == nullptr) return fail(LOCO_ERR_INVALID_ARG, "codes or scales array is NULL");
  static thread_local char names[2 * kMaxRanks][16];
  const size_t cbytes = size_t(loco_code_bytes(n, cfg->bits, cfg->block));
  const size_t sbytes = size_t(loco_num_blocks(n, cfg->block)) * sizeof(float);
  for (int w = 0; w < W; ++w) {
    snprintf(names[2 * w], 16, "codes[%d]", w);
    snprintf(names[2 * w + 1], 16, "scales[%d]", w);
    list[(*count)++] = BufCheck{codes[w], cbytes, 16, names[2 * w]};
    list[(*count)++] = BufCheck{scales[w], sbytes, 16, names[2 * w + 1]};
    out->codes[w] = codes[w];
    out->scales[w] = scales[w];
  }
  for (int w = W; w < kMaxRanks; ++w) {
    out->codes[w] = nullptr;
    out->scales[w] = nullptr;
  }
  out->neg_zero = -0.0f;
  return LOCO_OK;
}

}  // namespace loco

using namespace loco;

extern "C" {

int64_t loco_num_blocks(int64_t n, int32_t block) {
  if (n <= 0 || n > LOCO_MAX_N || block <= 0) return 0;
  return (n + block - 1) / block;
}

int64_t loco_code_bytes(int64_t n, int32_t bits, int32_t block) {
  if (n <= 0 || n > LOCO_MAX_N || block <= 0 || bits <= 0 || bits > 64) return 0;
  return loco_num_blocks(n, block) * block * bits / 8;
}

loco_status loco_shard_range(int64_t n, int32_t block, int32_t W, int32_t j, int64_t* lo, int64_t* hi) {
  if (lo == nullptr || hi == nullptr) return fail(LOCO_ERR_INVALID_ARG, "lo or hi is NULL");
  if (block != 64 && block != 128 && block != 256)
    return fail(LOCO_ERR_UNSUPPORTED, "block = %d (supported: 64, 128, 256)", block);
  if (n < 0 || n > LOCO_MAX_N)
    return fail(LOCO_ERR_INVALID_ARG, "n = %lld outside [0, LOCO_MAX_N = 2^48]", (long long)n);
  if (W < 1) return fail(LOCO_ERR_INVALID_ARG, "W = %d (need >= 1)", W);
  if (W > kMaxRanks) return fail(LOCO_ERR_UNSUPPORTED, "W = %d (at most %d)", W, kMaxRanks);
  if (j < 0 || j >= W) return fail(LOCO_ERR_INVALID_ARG, "j = %d outside [0, W = %d)", j, W);
  const int64_t unit = int64_t(4) * block;
  const int64_t nu = (n + unit - 1) / unit;
  const int64_t base = nu / W, rem = nu % W;
  const int64_t u0 = j * base + (j < rem ? j : rem);
  const int64_t u1 = (j + 1) * base + (j + 1 < rem ? j + 1 : rem);
  *lo = u0 * unit < n ? u0 * unit : n;
  *hi = u1 * unit < n ? u1 * unit : n;
  g_last_error[0] = '\0';
  return LOCO_OK;
}

const char* loco_status_string(loco_status s) {
  switch (s) {
    case LOCO_OK: return "LOCO_OK";
    case LOCO_ERR_INVALID_ARG: return "LOCO_ERR_INVALID_ARG";
    case LOCO_ERR_UNSUPPORTED: return "LOCO_ERR_UNSUPPORTED";
    case LOCO_ERR_MISALIGNED: return "LOCO_ERR_MISALIGNED";
    case LOCO_ERR_CUDA: return "LOCO_ERR_CUDA";
  }
  return "LOCO_ERR_UNKNOWN";
}

const char* loco_last_error(void) { return g_last_error; }

}  // extern "C"

namespace loco {

// Shared by loco_compress and loco_compress_e8: exactly one of err and
// err_codes is non-null.
static loco_status compress_common(const loco_config* cfg, const void* grad, int32_t grad_dtype, float* err,
                                   int8_t* err_codes, float* err_steps, int64_t n, int64_t step, uint8_t* codes,
                                   float* scales, loco_stream_t stream) {
  if (cfg == nullptr) return fail(LOCO_ERR_INVALID_ARG, "cfg is NULL");
  loco_status st = check_layout(cfg->bits, cfg->block);
  if (st != LOCO_OK) return st;
  if (grad_dtype != LOCO_F32 && grad_dtype != LOCO_BF16)
    return fail(LOCO_ERR_UNSUPPORTED, "grad_dtype = %d (LOCO_F32 or LOCO_BF16)", grad_dtype);
  if (cfg->scale_mode != LOCO_SCALE_ABSMAX && cfg->scale_mode != LOCO_SCALE_FIXED)
    return fail(LOCO_ERR_UNSUPPORTED, "scale_mode = %d", cfg->scale_mode);
  if (!(cfg->beta >= 0.0f && cfg->beta <= 1.0f)) return fail(LOCO_ERR_INVALID_ARG, "beta = %g not in [0, 1]", cfg->beta);
  if (!(cfg->err_scale_mult > 0.0f) || !isfinite(cfg->err_scale_mult))
    return fail(LOCO_ERR_INVALID_ARG, "err_scale_mult (kappa) = %g must be finite and > 0", cfg->err_scale_mult);
  if (cfg->scale_mode == LOCO_SCALE_FIXED && (!(cfg->fixed_scale > 0.0f) || !isfinite(cfg->fixed_scale)))
    return fail(LOCO_ERR_INVALID_ARG, "fixed_scale = %g must be finite and > 0", cfg->fixed_scale);
  if (cfg->reset_period < 0) return fail(LOCO_ERR_INVALID_ARG, "reset_period = %lld < 0", (long long)cfg->reset_period);
  if (n < 0 || n > LOCO_MAX_N)
    return fail(LOCO_ERR_INVALID_ARG, "n = %lld outside [0, LOCO_MAX_N = 2^48]", (long long)n);
  if (step < 1) return fail(LOCO_ERR_INVALID_ARG, "step = %lld (1-based)", (long long)step);
  if (n == 0) return LOCO_OK;

  const bool e8 = err_codes != nullptr || err_steps != nullptr;
  const size_t gbytes = size_t(n) * (grad_dtype == LOCO_BF16 ? 2 : 4);
  const size_t cbytes = size_t(loco_code_bytes(n, cfg->bits, cfg->block));
  const size_t sbytes = size_t(loco_num_blocks(n, cfg->block)) * 4;
  const size_t ebytes = e8 ? size_t(n) : size_t(n) * 4;
  const void* ebuf = e8 ? static_cast<const void*>(err_codes) : static_cast<const void*>(err);
  BufCheck bufs[5] = {{grad, gbytes, 16, "grad"}, {ebuf, ebytes, 16, e8 ? "err_codes" : "err"},
                      {codes, cbytes, 16, "codes"}, {scales, sbytes, 16, "scales"},
                      {err_steps, sbytes, 16, "err_steps"}};
  if ((st = check_buffers(bufs, e8 ? 5 : 4)) != LOCO_OK) return st;
  const int nbufs = e8 ? 5 : 4;
  for (int i = 0; i < nbufs; ++i)
    for (int j = i + 1; j < nbufs; ++j)
      if (overlap(bufs[i].p, bufs[i].bytes, bufs[j].p, bufs[j].bytes))
        return fail(LOCO_ERR_INVALID_ARG, "%s and %s overlap", bufs[i].name, bufs[j].name);

  CompressArgs a;
  a.grad = grad;
  a.err = e8 ? nullptr : err;
  a.err_codes = e8 ? err_codes : nullptr;
  a.err_steps = e8 ? err_steps : nullptr;
  a.codes = codes;
  a.scales = scales;
  a.n = n;
  a.bits = cfg->bits;
  a.block = cfg->block;
  a.grad_bf16 = grad_dtype == LOCO_BF16;
  a.fixed = cfg->scale_mode == LOCO_SCALE_FIXED;
  a.fixed_delta = a.fixed ? 1.0f / cfg->fixed_scale : 0.0f;
  a.fixed_inv = a.fixed ? cfg->fixed_scale : 0.0f;
  a.beta = cfg->beta;
  a.one_minus_beta = 1.0f - cfg->beta;
  a.kappa = cfg->err_scale_mult;
  {
    // A power of two 2^k with 2^-k a normal float: dividing by it is the same
    // real as multiplying by its exact reciprocal, so both round alike.
    int ex = 0;
    const float m = frexpf(a.kappa, &ex);
    a.kappa_recip = (m == 0.5f && ex - 1 >= -126 && ex - 1 <= 126) ? ldexpf(1.0f, 1 - ex) : 0.0f;
  }
  a.reset = cfg->reset_period > 0 && (step % cfg->reset_period) == 0;
  a.neg_zero = -0.0f;
  return launch_result(launch_compress(a, reinterpret_cast<cudaStream_t>(stream)),
                       e8 ? "loco_compress_e8" : "loco_compress");
}

}  // namespace loco

extern "C" {

loco_status loco_compress(const loco_config* cfg, const void* grad, int32_t grad_dtype, float* err, int64_t n,
                          int64_t step, uint8_t* codes, float* scales, loco_stream_t stream) {
  if (n > 0 && err == nullptr) return fail(LOCO_ERR_INVALID_ARG, "err is NULL");
  return compress_common(cfg, grad, grad_dtype, err, nullptr, nullptr, n, step, codes, scales, stream);
}

loco_status loco_compress_e8(const loco_config* cfg, const void* grad, int32_t grad_dtype, int8_t* err_codes,
                             float* err_steps, int64_t n, int64_t step, uint8_t* codes, float* scales,
                             loco_stream_t stream) {
  if (n > 0 && (err_codes == nullptr || err_steps == nullptr))
    return fail(LOCO_ERR_INVALID_ARG, "err_codes or err_steps is NULL");
  return compress_common(cfg, grad, grad_dtype, nullptr, err_codes, err_steps, n, step, codes, scales, stream);
}

loco_status loco_decode_reduce(const loco_config* cfg, const uint8_t* const* codes, const float* const* scales,
                               int32_t W, int64_t n, float* mean, loco_stream_t stream) {
  if (cfg == nullptr) return fail(LOCO_ERR_INVALID_ARG, "cfg is NULL");
  loco_status st = check_layout(cfg->bits, cfg->block);
  if (st != LOCO_OK) return st;
  if (n < 0 || n > LOCO_MAX_N)
    return fail(LOCO_ERR_INVALID_ARG, "n = %lld outside [0, LOCO_MAX_N = 2^48]", (long long)n);
  if (W < 1) return fail(LOCO_ERR_INVALID_ARG, "W = %d (need >= 1)", W);
  if (W > kMaxRanks) return fail(LOCO_ERR_UNSUPPORTED, "W = %d (at most %d)", W, kMaxRanks);
  if (n == 0) return LOCO_OK;
  ReduceArgs a;
  BufCheck bufs[2 * kMaxRanks + 1];
  int nbuf = 0;
  if ((st = check_ranks(cfg, codes, scales, W, n, &a.ranks, bufs, &nbuf)) != LOCO_OK) return st;
  const size_t mbytes = size_t(n) * 4;
  bufs[nbuf++] = BufCheck{mean, mbytes, 16, "mean"};
  if ((st = check_buffers(bufs, nbuf)) != LOCO_OK) return st;
  const size_t cbytes = size_t(loco_code_bytes(n, cfg->bits, cfg->block));
  const size_t sbytes = size_t(loco_num_blocks(n, cfg->block)) * 4;
  for (int w = 0; w < W; ++w)
    if (overlap(mean, mbytes, codes[w], cbytes) || overlap(mean, mbytes, scales[w], sbytes))
      return fail(LOCO_ERR_INVALID_ARG, "mean overlaps the inputs of rank %d", w);
  a.W = W;
  a.n = n;
  a.bits = cfg->bits;
  a.block = cfg->block;
  a.mean = mean;
  return launch_result(launch_decode_reduce(a, reinterpret_cast<cudaStream_t>(stream)), "loco_decode_reduce");
}

}  // extern "C"

namespace loco {

// Shared checks of the fused optimizer entry points: layout, ranks, the
// param/state buffers and their overlaps.  fbufs lists param (+ m, v).
static loco_status check_update(const loco_config* cfg, const uint8_t* const* codes, const float* const* scales,
                                int32_t W, int64_t n, RankPtrs* ranks, const BufCheck* fbufs, int nf,
                                uint16_t* param_bf16) {
  loco_status st;
  BufCheck bufs[2 * kMaxRanks + 4];
  int nbuf = 0;
  if ((st = check_ranks(cfg, codes, scales, W, n, ranks, bufs, &nbuf)) != LOCO_OK) return st;
  const int nranks = nbuf;
  for (int i = 0; i < nf; ++i) bufs[nbuf++] = fbufs[i];
  if (param_bf16 != nullptr) bufs[nbuf++] = BufCheck{param_bf16, size_t(n) * 2, 16, "param_bf16"};
  if ((st = check_buffers(bufs, nbuf)) != LOCO_OK) return st;
  // Outputs (after the ranks' read-only inputs, which may alias each other)
  // must not overlap any other buffer.
  for (int i = nranks; i < nbuf; ++i)
    for (int j = 0; j < nbuf; ++j)
      if (j != i && overlap(bufs[i].p, bufs[i].bytes, bufs[j].p, bufs[j].bytes))
        return fail(LOCO_ERR_INVALID_ARG, "%s overlaps %s", bufs[i].name, bufs[j].name);
  return LOCO_OK;
}

static loco_status check_common(const loco_config* cfg, int32_t W, int64_t n) {
  if (cfg == nullptr) return fail(LOCO_ERR_INVALID_ARG, "cfg is NULL");
  loco_status st = check_layout(cfg->bits, cfg->block);
  if (st != LOCO_OK) return st;
  if (n < 0 || n > LOCO_MAX_N)
    return fail(LOCO_ERR_INVALID_ARG, "n = %lld outside [0, LOCO_MAX_N = 2^48]", (long long)n);
  if (W < 1) return fail(LOCO_ERR_INVALID_ARG, "W = %d (need >= 1)", W);
  if (W > kMaxRanks) return fail(LOCO_ERR_UNSUPPORTED, "W = %d (at most %d)", W, kMaxRanks);
  return LOCO_OK;
}

static loco_status adam_common(const loco_config* cfg, const uint8_t* const* codes, const float* const* scales,
                               int32_t W, int64_t n, float* param, float* m, float* v, uint16_t* param_bf16,
                               const loco_adam_hparams* hp, int64_t t, loco_stream_t stream) {
  if (hp == nullptr) return fail(LOCO_ERR_INVALID_ARG, "hp is NULL");
  loco_status st = check_common(cfg, W, n);
  if (st != LOCO_OK) return st;
  if (t < 1) return fail(LOCO_ERR_INVALID_ARG, "t = %lld (1-based)", (long long)t);
  if (!isfinite(hp->lr) || !isfinite(hp->eps) || !isfinite(hp->weight_decay) || hp->eps < 0.0f)
    return fail(LOCO_ERR_INVALID_ARG, "lr, eps, weight_decay must be finite and eps >= 0");
  if (!(hp->beta1 >= 0.0f && hp->beta1 < 1.0f) || !(hp->beta2 >= 0.0f && hp->beta2 < 1.0f))
    return fail(LOCO_ERR_INVALID_ARG, "beta1 = %g, beta2 = %g must lie in [0, 1)", hp->beta1, hp->beta2);
  if (n == 0) return LOCO_OK;
  AdamArgs a;
  const size_t fbytes = size_t(n) * 4;
  const BufCheck fb[3] = {{param, fbytes, 16, "param"}, {m, fbytes, 16, "m"}, {v, fbytes, 16, "v"}};
  if ((st = check_update(cfg, codes, scales, W, n, &a.ranks, fb, 3, param_bf16)) != LOCO_OK) return st;
  a.W = W;
  a.n = n;
  a.bits = cfg->bits;
  a.block = cfg->block;
  a.param = param;
  a.m = m;
  a.v = v;
  a.param_bf16 = param_bf16;
  a.beta1 = hp->beta1;
  a.beta2 = hp->beta2;
  a.one_minus_beta1 = 1.0f - hp->beta1;
  a.one_minus_beta2 = 1.0f - hp->beta2;
  a.lr_wd = hp->lr * hp->weight_decay;
  a.c1 = hp->lr;
  a.c2 = 1.0f;
  if (hp->bias_correction) {
    const double bc1 = 1.0 - pow(double(hp->beta1), double(t));
    const double bc2 = 1.0 - pow(double(hp->beta2), double(t));
    a.c1 = float(double(hp->lr) / bc1);
    a.c2 = hp->eps_inside_sqrt ? float(1.0 / bc2) : float(1.0 / sqrt(bc2));
  }
  a.eps = hp->eps;
  a.eps_inside_sqrt = hp->eps_inside_sqrt != 0;
  return launch_result(launch_adam(a, reinterpret_cast<cudaStream_t>(stream)),
                       param_bf16 ? "loco_adam_step_bf16" : "loco_adam_step");
}

}  // namespace loco

extern "C" {

loco_status loco_adam_step(const loco_config* cfg, const uint8_t* const* codes, const float* const* scales, int32_t W,
                           int64_t n, float* param, float* m, float* v, const loco_adam_hparams* hp, int64_t t,
                           loco_stream_t stream) {
  return adam_common(cfg, codes, scales, W, n, param, m, v, nullptr, hp, t, stream);
}

loco_status loco_adam_step_bf16(const loco_config* cfg, const uint8_t* const* codes, const float* const* scales,
                                int32_t W, int64_t n, float* param, float* m, float* v, uint16_t* param_bf16,
                                const loco_adam_hparams* hp, int64_t t, loco_stream_t stream) {
  if (n > 0 && param_bf16 == nullptr) return fail(LOCO_ERR_INVALID_ARG, "param_bf16 is NULL");
  return adam_common(cfg, codes, scales, W, n, param, m, v, param_bf16, hp, t, stream);
}

loco_status loco_sgd_step(const loco_config* cfg, const uint8_t* const* codes, const float* const* scales, int32_t W,
                          int64_t n, float* param, uint16_t* param_bf16, float lr, loco_stream_t stream) {
  loco_status st = check_common(cfg, W, n);
  if (st != LOCO_OK) return st;
  if (!isfinite(lr)) return fail(LOCO_ERR_INVALID_ARG, "lr = %g must be finite", lr);
  if (n == 0) return LOCO_OK;
  SgdArgs a;
  const BufCheck fb[1] = {{param, size_t(n) * 4, 16, "param"}};
  if ((st = check_update(cfg, codes, scales, W, n, &a.ranks, fb, 1, param_bf16)) != LOCO_OK) return st;
  a.W = W;
  a.n = n;
  a.bits = cfg->bits;
  a.block = cfg->block;
  a.param = param;
  a.param_bf16 = param_bf16;
  a.lr = lr;
  return launch_result(launch_sgd(a, reinterpret_cast<cudaStream_t>(stream)), "loco_sgd_step");
}

}  // extern "C"
