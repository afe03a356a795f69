/*
 * loco.h — C ABI of libloco, the GB300 (sm_103a) hot path of LoCo gradient
 * compression.
 *
 * Source of the method: "LoCo: Low-Bit Communication Adaptor for Large-scale
 * Model Training" (Xie, Lin, Toh, Zhou; arXiv 2407.04480), HTML body, §3.1
 * (Eqns 1-3), §3.2 (Eqns 4-7), §3.3 (Eqn 8) and §4 (Adam family, Eqn 9).
 *
 * General conventions (apply to every entry point below):
 *  - Every data pointer is DEVICE memory owned by the caller.  The library
 *    allocates nothing, keeps no state between calls and never synchronises
 *    the stream.  Arrays of per-rank pointers (`codes`, `scales`) are HOST
 *    arrays of device pointers; they are read during the call and copied by
 *    value into the kernel launch, so the caller may free them on return.
 *  - Every call is stream ordered: it validates its arguments on the host,
 *    enqueues its kernel(s) on `stream` (NULL = legacy default stream) and
 *    returns.  On any argument error nothing is launched and nothing is
 *    written.  A failed launch returns LOCO_ERR_CUDA and the CUDA error text
 *    is available from loco_last_error().
 *  - Layouts: flat, contiguous, element i of a bucket of n elements.  Quant
 *    block b covers elements [b*block, min((b+1)*block, n)); nb =
 *    ceil(n / block).  Packed codes of block b start at byte
 *    b*block*bits/8.  4-bit codes are two's-complement nibbles, element 2j of
 *    the block in the low nibble of byte j, element 2j+1 in the high nibble.
 *    8-bit codes are int8.  Padding elements of a ragged last block get code 0.
 *  - Alignment: every buffer (grad, err, err_codes, err_steps, codes, scales,
 *    mean, param, m, v, param_bf16) must be 16-byte aligned
 *    (LOCO_ERR_MISALIGNED otherwise).  The receivers stage each rank's steps
 *    with 16-byte copies, so a rank's scales placed at an offset inside a
 *    larger buffer (an exchange buffer, a shard of a bucket) must start on a
 *    16-byte boundary: a shard of a bucket starting at a multiple of 4 quant
 *    blocks does.
 *  - The calls allocate nothing and never synchronise, so they can be captured
 *    in a CUDA graph.  Step counters, the reset decision and the Adam constants
 *    are computed on the host at call time and become part of the captured
 *    launch: a graph captured at step k replays step k.  The first call of each
 *    configuration (bits, block, W, dtype, ...) on each device queries
 *    occupancy and sets the kernel's shared-memory limit on that device; make
 *    it before capturing.
 *  - Arithmetic is IEEE binary32, round to nearest even, every product and
 *    every sum rounded on its own (no product is fused into a following add);
 *    the exact operation order of each step is stated at the
 *    entry point.  Non-finite inputs are outside the contract: no call reads
 *    or writes out of bounds on them, but the values produced are unspecified.
 */
#ifndef LOCO_H
#define LOCO_H

#include <stdint.h>
#include <stddef.h>

/* The entry points below are the only symbols the library exports; every
 * other symbol (kernels, helpers, the statically linked CUDA runtime) is
 * hidden, so the library can share a process with other CUDA code, including
 * another build of itself. */
#if defined(__GNUC__) || defined(__clang__)
#define LOCO_API __attribute__((visibility("default")))
#else
#define LOCO_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Same object as cudaStream_t, declared without the CUDA headers. */
typedef struct CUstream_st* loco_stream_t;

typedef enum {
  LOCO_OK = 0,
  LOCO_ERR_INVALID_ARG = 1,  /* null pointer, n < 0 or n > LOCO_MAX_N, W < 1, step < 1, beta outside [0,1], kappa <= 0, bad scale */
  LOCO_ERR_UNSUPPORTED = 2,  /* bits not in {4,8}, block not in {64,128,256}, W > LOCO_MAX_RANKS, unknown dtype/mode */
  LOCO_ERR_MISALIGNED = 3,   /* a pointer violates the alignment rule above */
  LOCO_ERR_CUDA = 4          /* the kernel launch failed; see loco_last_error() */
} loco_status;

typedef enum { LOCO_F32 = 0, LOCO_BF16 = 1 } loco_dtype;

/* How the quantisation step Delta_b of block b is chosen (the scale s of Eqn 1). */
typedef enum {
  LOCO_SCALE_ABSMAX = 0,  /* Delta_b = A_b / qmax with A_b = max |h_i| over the block's valid elements */
  LOCO_SCALE_FIXED = 1    /* Delta_b = 1/s for every block, s = fixed_scale (the paper's s = 2^19, 2^17; §3.1) */
} loco_scale_mode;

#define LOCO_MAX_RANKS 16

/* Largest bucket a call accepts (2^48 elements, far beyond any device memory);
 * every size the library derives from n then fits in int64_t.  Larger n is
 * LOCO_ERR_INVALID_ARG, and the size helpers below return 0 for it. */
#define LOCO_MAX_N ((int64_t)1 << 48)

/* Sender-side hyper-parameters (§3.1-3.2). */
typedef struct {
  int32_t bits;           /* p of Round_p-bit (Eqn 1): 4 or 8                                    */
  int32_t block;          /* quant block length: 64, 128 or 256 elements                         */
  int32_t scale_mode;     /* loco_scale_mode                                                    */
  float   fixed_scale;    /* s for LOCO_SCALE_FIXED (> 0, finite); ignored for ABSMAX            */
  float   beta;           /* weight of the previous error in the moving average (Eqn 5), [0,1]  */
  float   err_scale_mult; /* kappa = s_e / s (Eqn 7; the paper uses 4 or 6), > 0                 */
  int64_t reset_period;   /* T_c of the periodic reset (Eqn 7; paper 512 or 1024); 0 = never    */
} loco_config;

/* Adam / AdamW hyper-parameters for the fused receiver step (§4, Eqn 9). */
typedef struct {
  float   lr;              /* eta                                                               */
  float   beta1;           /* weight of the previous m: m = beta1*m + (1-beta1)*g               */
  float   beta2;           /* weight of the previous v: v = beta2*v + (1-beta2)*g*g             */
  float   eps;             /* delta                                                             */
  float   weight_decay;    /* decoupled (AdamW) decay; 0 = plain Adam                           */
  int32_t bias_correction; /* 1: bias-corrected step (c1, c2 of loco_adam_step); 0: c1=lr, c2=1  */
  int32_t eps_inside_sqrt; /* 1: 1/sqrt(v+eps) as printed in §4; 0: 1/(sqrt(v)+eps) as in Adam  */
} loco_adam_hparams;

/* nb = ceil(n / block); 0 for n <= 0, n > LOCO_MAX_N or block <= 0. */
LOCO_API int64_t loco_num_blocks(int64_t n, int32_t block);

/* Bytes of packed codes for a bucket of n elements: nb * block * bits / 8; 0 on bad arguments
 * (n <= 0, n > LOCO_MAX_N, bits or block <= 0). */
LOCO_API int64_t loco_code_bytes(int64_t n, int32_t bits, int32_t block);

/*
 * loco_compress — sender side of one LoCo step on one rank's flat gradient bucket.
 * Paper: §3.1 Eqn (2) (compensate), Eqns (1),(3) (low-bit compressor),
 * §3.2 Eqns (4),(5) (moving average of the compression error) and Eqn (7)
 * (error clipping to the 8-bit compressor's range and the periodic reset).
 *
 * Per block b, with qmax = 2^(bits-1)-1, qmin = -2^(bits-1), k = step:
 *   h_i   = f32(g_i) + e_i                                    (Eqn 2)
 *   A_b   = max_i |h_i| over the valid elements
 *   ABSMAX: Delta_b = A_b/qmax, inv_b = qmax/A_b  (both 0 when A_b == 0, or
 *           when qmax/A_b overflows fp32, i.e. A_b < qmax/FLT_MAX)
 *   FIXED:  Delta_b = 1/s,      inv_b = s
 *   q_i   = rint_even(clamp(h_i*inv_b, qmin, qmax))           (Eqns 1, 3)
 *   d_i   = f32(q_i)*Delta_b ;  r_i = h_i - d_i                (Eqn 4)
 *   t_i   = beta*e_i + (1-beta)*r_i                            (Eqn 5; 1-beta formed once in fp32)
 *   De_b  = Delta_b/kappa ; lo = -128*De_b ; hi = 127*De_b
 *   e_i'  = t_i<lo ? lo : (t_i>hi ? hi : t_i)                  (Eqn 7 saturation)
 *   e_i'  = 0 if reset_period > 0 and k % reset_period == 0    (Eqn 7 reset)
 *
 * grad    [n] device, dtype grad_dtype (LOCO_F32 or LOCO_BF16); read only.
 * err     [n] device fp32, in/out: e_{k-1} on entry, e_k on return.  Start a
 *         run with zeros (the paper's e_0 = 0).
 * step    1-based step counter k of this call (>= 1), owned by the caller.
 * codes   [loco_code_bytes(n)] device, out.
 * scales  [nb] device fp32, out: Delta_b (the receiver decodes q*Delta_b).
 * n == 0 is a valid empty call: nothing is launched.
 * grad must not alias err, codes or scales.
 */
LOCO_API loco_status loco_compress(const loco_config* cfg, const void* grad, int32_t grad_dtype,
                          float* err, int64_t n, int64_t step,
                          uint8_t* codes, float* scales, loco_stream_t stream);

/*
 * loco_compress_e8 — loco_compress with the compensation error stored in 8 bits,
 * as the paper keeps it (§3.2 Eqn 7: e_k = compressor(e~_k; s_e, 8) with
 * s_e = kappa*s, decompressed by Eqn 2 before it is added back): one int8 code
 * per element plus one fp32 step per quant block instead of an fp32 error.
 * Codes and scales are bit-identical in format to loco_compress's.
 *
 * Per block b (Delta_b, inv_b, q_i, d_i, r_i as in loco_compress):
 *   e_i    = f32(qe_i) * De_b                        (stored state; zeros to start)
 *   h_i    = f32(g_i) + e_i                           (Eqn 2)
 *   t_i    = beta*e_i + (1-beta)*r_i                  (Eqn 5)
 *   De_b'  = Delta_b/kappa ;  inv_e = kappa*inv_b     (s_e = kappa*s, fp32; 0 if it overflows)
 *   qe_i'  = rint_even(clamp(t_i*inv_e, -128, 127)); 0 on a reset step (Eqn 7)
 * err_codes [n] device int8, in/out (16-byte aligned).
 * err_steps [nb] device fp32, in/out (the De_b; zeros to start).
 * With s_e = 4s..6s the new contribution (1-beta)*r must exceed half a step
 * Delta/(2*kappa) to be stored at all, so beta (weight of the previous error)
 * should be well below 1 with this storage.
 */
LOCO_API loco_status loco_compress_e8(const loco_config* cfg, const void* grad, int32_t grad_dtype,
                             int8_t* err_codes, float* err_steps, int64_t n, int64_t step,
                             uint8_t* codes, float* scales, loco_stream_t stream);

/*
 * loco_decode_reduce — receiver side: decode W ranks' packed buckets and
 * average them in fp32 (§3.3, Eqn 8; the all-to-all variant that never
 * re-compresses a partial sum).
 *
 *   d_{w,i}  = f32(q_{w,i}) * Delta_{w,b}
 *   mean_i   = (((d_{0,i} + d_{1,i}) + d_{2,i}) + ... + d_{W-1,i}) / f32(W)
 *
 * codes[w], scales[w] (host array of W device pointers) hold rank w's output
 * of loco_compress with the same bits/block.  Only cfg->bits and cfg->block
 * are read.  mean [n] device fp32, out; it must not alias any input.
 * 1 <= W <= LOCO_MAX_RANKS.
 */
LOCO_API loco_status loco_decode_reduce(const loco_config* cfg, const uint8_t* const* codes,
                               const float* const* scales, int32_t W, int64_t n,
                               float* mean, loco_stream_t stream);

/*
 * loco_adam_step — loco_decode_reduce fused with one Adam(W) update of the
 * rank's parameters (§4, Eqn 9: the optimizer consumes the averaged low-bit
 * gradient g~ of Eqn 8).  g~_i is formed exactly as in loco_decode_reduce and
 * is never written to memory.  Per element, in this order (Kingma & Ba's Adam
 * with decoupled weight decay; the bias corrections of their Algorithm 1,
 * m_hat = m/(1 - beta1^t) and v_hat = v/(1 - beta2^t), are folded into the
 * step size and the denominator, as torch.optim.AdamW arranges them, except
 * that 1/sqrt(1 - beta2^t) is a rounded factor rather than a divisor; the same
 * update in exact arithmetic, a different rounding in fp32):
 *   p   = p - (lr*wd)*p
 *   m   = beta1*m + (1-beta1)*g~
 *   v   = beta2*v + (1-beta2)*(g~*g~)
 *   den = sqrt(v)*c2 + eps        c2 = 1/sqrt(1 - beta2^t)
 *        (eps_inside_sqrt: den = sqrt(v*c2 + eps), c2 = 1/(1 - beta2^t))
 *   p   = p - c1*(m/den)          c1 = lr/(1 - beta1^t)
 * lr*wd, 1-beta1 and 1-beta2 are formed once in fp32; c1 and c2 once in
 * double from the fp32 hyper-parameters, rounded to fp32 (c1 = lr, c2 = 1
 * without bias correction).  The paper's own convention (beta on the new
 * term, no bias correction, 1/sqrt(v+delta)) is beta1 = 1-0.1,
 * beta2 = 1-beta2_paper, bias_correction = 0, eps_inside_sqrt = 1.
 * param, m, v [n] device fp32, in/out.  t = 1-based optimizer step.
 */
LOCO_API loco_status loco_adam_step(const loco_config* cfg, const uint8_t* const* codes,
                           const float* const* scales, int32_t W, int64_t n,
                           float* param, float* m, float* v,
                           const loco_adam_hparams* hp, int64_t t, loco_stream_t stream);

/*
 * loco_adam_step_bf16 — loco_adam_step that also writes the updated parameters
 * rounded to bf16 (nearest, halves to even) into param_bf16 [n] (device,
 * 16-byte aligned, out): the 16-bit parameter copy a sharded data-parallel job
 * all-gathers after the update (the 16-bit parameters of the Table I memory
 * and communication comparison, §4).  Everything else as loco_adam_step.
 */
LOCO_API loco_status loco_adam_step_bf16(const loco_config* cfg, const uint8_t* const* codes,
                                const float* const* scales, int32_t W, int64_t n,
                                float* param, float* m, float* v, uint16_t* param_bf16,
                                const loco_adam_hparams* hp, int64_t t, loco_stream_t stream);

/*
 * loco_sgd_step — loco_decode_reduce fused with one LoCo-SGD step (§4: the
 * SGD iterate theta_{k+1} = theta_k - eta * g~_k with g~ from Eqn 8):
 *   p = p - lr*g~          (one fp32 product, one fp32 subtraction)
 * g~ is formed exactly as in loco_decode_reduce and never written to memory.
 * param [n] device fp32, in/out.  param_bf16 [n] device, out, or NULL: when
 * given it receives the updated parameters rounded to bf16 (nearest even).
 */
LOCO_API loco_status loco_sgd_step(const loco_config* cfg, const uint8_t* const* codes,
                          const float* const* scales, int32_t W, int64_t n,
                          float* param, uint16_t* param_bf16, float lr, loco_stream_t stream);

/*
 * loco_shard_range — shard j of W of a bucket for the sharded receiver of
 * §3.3 (the all-to-all variant around Eqn 8): every rank compresses its whole
 * bucket, sends the low-bit codes and steps of shard j to rank j, and rank j
 * decodes and averages the W slices it receives (loco_decode_reduce, or a
 * fused optimizer step, on the shard's n_j = hi - lo elements) and updates its
 * part of the parameters.
 *
 * The bucket is cut into units of U = 4*block elements (so every shard starts
 * on a quant-block boundary and its codes and steps start 16-byte aligned in
 * the rank's buffers); with nu = ceil(n / U), shard j holds units
 * [j*base + min(j, rem), (j+1)*base + min(j+1, rem)) where base = nu / W and
 * rem = nu % W, clipped to n.  Shards are contiguous, in rank order, cover
 * [0, n) exactly, and differ in length by at most one unit; when nu < W the
 * last W - nu shards are empty (lo == hi).  Shard j's codes are bytes
 * [lo*bits/8, lo*bits/8 + loco_code_bytes(hi - lo)) of a rank's codes and its
 * steps are floats [lo/block, lo/block + ceil((hi - lo)/block)) of its scales.
 *
 * lo, hi (host, out): element range of shard j.  Errors: NULL lo or hi,
 * n < 0 or n > LOCO_MAX_N, W < 1, j outside [0, W) -> LOCO_ERR_INVALID_ARG;
 * block not in {64, 128, 256} or W > LOCO_MAX_RANKS -> LOCO_ERR_UNSUPPORTED.
 * Host only: no CUDA call.
 */
LOCO_API loco_status loco_shard_range(int64_t n, int32_t block, int32_t W, int32_t j, int64_t* lo, int64_t* hi);

/* Static text for a status code. */
LOCO_API const char* loco_status_string(loco_status s);

/* Text of the last LOCO_ERR_CUDA (or argument error) raised on the calling
 * host thread; "" if none.  Thread local; valid until the next call. */
LOCO_API const char* loco_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* LOCO_H */
