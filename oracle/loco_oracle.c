/*
 * loco_oracle.c — TEST INFRASTRUCTURE ONLY.  A plain, slow, element-by-element
 * CPU statement of what the LoCo hot path computes, used to check the CUDA
 * library.  Only the test suite, the smoke check and the benchmark's CPU
 * baseline load it; no product code path may call it.  It shares no source,
 * header or constant with the CUDA library.
 *
 * Method: "LoCo: Low-Bit Communication Adaptor for Large-scale Model
 * Training" (arXiv 2407.04480), §3.1 Eqns (1)-(3), §3.2 Eqns (4)-(7),
 * §3.3 Eqn (8), §4 Eqn (9).  The displayed equations were lost from the
 * available text; each function states the reading it implements.
 *
 * Precision: IEEE binary32 throughout, round to nearest even, every product
 * and sum a separate rounded operation.  Build with -ffp-contract=off and
 * without -ffast-math (gcc contracts a*b+c into fma by default on aarch64).
 * fp64 appears only in the shadow sum of oracle_decode_reduce and in the
 * bias-correction constants of the Adam step, as stated there.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

/* bf16 -> fp32 is exact: the bf16 bits are the high half of the fp32 bits. */
static float bf16_bits_to_f32(uint16_t b) {
  uint32_t u = ((uint32_t)b) << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return f;
}

/* fp32 -> bf16, round to nearest, halves to even: keep the high 16 bits of
 * u + 0x7FFF + (bit 16 of u).  NaN keeps its sign and becomes a quiet NaN. */
static uint16_t f32_to_bf16_rne(float f) {
  uint32_t u;
  memcpy(&u, &f, sizeof u);
  if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu)) return (uint16_t)((u >> 16) | 0x0040u);
  u += 0x7FFFu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}

/* Round_p-bit of Eqn (1): nearest integer, halves to even (the rounding of
 * torch.round, "the default one in PyTorch", §3.1), saturated to
 * [-2^(p-1), 2^(p-1)-1].  Saturating first and rounding second gives the same
 * integer because both bounds are integers and rounding is monotone. */
static int round_pbit(float x, int bits) {
  float qmax = (float)((1 << (bits - 1)) - 1);
  float qmin = -(float)(1 << (bits - 1));
  if (x < qmin) x = qmin;
  if (x > qmax) x = qmax;
  return (int)nearbyintf(x); /* default rounding mode: nearest, ties to even */
}

/* Read one gradient element as fp32. */
static float grad_at(const void* grad, int grad_is_bf16, int64_t i) {
  if (grad_is_bf16) return bf16_bits_to_f32(((const uint16_t*)grad)[i]);
  return ((const float*)grad)[i];
}

/* Store the p-bit two's-complement code q of element j (index within its
 * block) into the block's packed bytes. */
static void put_code(uint8_t* blk, int bits, int j, int q) {
  if (bits == 8) {
    blk[j] = (uint8_t)(q & 0xFF);
  } else {
    uint8_t nib = (uint8_t)(q & 0xF);
    if (j % 2 == 0)
      blk[j / 2] = (uint8_t)((blk[j / 2] & 0xF0) | nib);
    else
      blk[j / 2] = (uint8_t)((blk[j / 2] & 0x0F) | (nib << 4));
  }
}

/* Read back the code of element j of a block (sign-extended). */
static int get_code(const uint8_t* blk, int bits, int j) {
  if (bits == 8) return (int)(int8_t)blk[j];
  int nib = (j % 2 == 0) ? (blk[j / 2] & 0xF) : (blk[j / 2] >> 4);
  return nib >= 8 ? nib - 16 : nib;
}

/*
 * Sender step of LoCo for the quant blocks [b0, b1) of a bucket of n elements.
 *
 *  §3.1 Eqn (2):  h = g + decompressor(e)           (e stored in fp32 here)
 *  §3.1 Eqns (1),(3): c = Round_p-bit(s*h); s is chosen per block as
 *                 qmax/A_b (A_b = max|h| of the block), or one fixed s for all
 *                 blocks; the decompressor multiplies the code by Delta = 1/s.
 *  §3.2 Eqn (4),(5): error moving average  e~ = beta*e~_prev + (1-beta)*(h-d)
 *  §3.2 Eqn (7):  the error is held within the range of the 8-bit compressor
 *                 of scale s_e = kappa*s, i.e. [-128/s_e, 127/s_e], and set to
 *                 zero every T_c steps.
 *
 * fixed_mode: 0 = per-block absmax, 1 = fixed scale s = fixed_scale.
 * err is updated in place for the elements of the processed blocks.
 * codes holds all blocks' packed codes (block b at byte b*block*bits/8);
 * scales[b] receives Delta_b.
 */
void oracle_compress(int bits, int block, int fixed_mode, float fixed_scale,
                     float beta, float kappa, int64_t reset_period,
                     const void* grad, int grad_is_bf16, float* err, int64_t n,
                     int64_t step, uint8_t* codes, float* scales,
                     int64_t b0, int64_t b1) {
  const float qmax = (float)((1 << (bits - 1)) - 1);
  const float one_minus_beta = 1.0f - beta;
  const int reset = (reset_period > 0) && (step % reset_period == 0);
  const int64_t bytes_per_block = (int64_t)block * bits / 8;
  float h[1024]; /* block <= 1024 */

  for (int64_t b = b0; b < b1; ++b) {
    const int64_t lo = b * block;
    int64_t cnt = n - lo;
    if (cnt > block) cnt = block;

    /* Eqn (2): compensate. */
    for (int64_t j = 0; j < cnt; ++j) {
      float g = grad_at(grad, grad_is_bf16, lo + j);
      h[j] = g + err[lo + j];
    }

    /* Scale of Eqn (1) for this block. */
    float delta, inv;
    if (fixed_mode) {
      delta = 1.0f / fixed_scale;
      inv = fixed_scale;
    } else {
      float amax = 0.0f;
      for (int64_t j = 0; j < cnt; ++j) {
        float a = fabsf(h[j]);
        if (a > amax) amax = a;
      }
      inv = (amax == 0.0f) ? 0.0f : qmax / amax;
      if (amax == 0.0f || isinf(inv)) {
        /* An all-zero block, or one so small that s = qmax/A_b overflows fp32
         * (A_b < qmax/FLT_MAX): no code can represent it; step and inverse 0. */
        delta = 0.0f;
        inv = 0.0f;
      } else {
        delta = amax / qmax;
      }
    }
    scales[b] = delta;

    /* Bounds of the 8-bit error compressor, scale s_e = kappa*s (Eqn 7). */
    const float delta_e = delta / kappa;
    const float e_lo = -128.0f * delta_e;
    const float e_hi = 127.0f * delta_e;

    uint8_t* blk = codes + b * bytes_per_block;
    for (int j = 0; j < block; ++j) {
      if (j >= cnt) { /* ragged tail: padding elements get code 0 */
        put_code(blk, bits, j, 0);
        continue;
      }
      /* Eqns (1),(3): low-bit code. */
      float x = h[j] * inv;
      int q = round_pbit(x, bits);
      put_code(blk, bits, j, q);
      /* Eqn (4): decompressed value and this step's compression error. */
      float d = (float)q * delta;
      float r = h[j] - d;
      /* Eqn (5): moving average with the stored previous error. */
      float prev = err[lo + j];
      float t1 = beta * prev;
      float t2 = one_minus_beta * r;
      float t = t1 + t2;
      /* Eqn (7): saturation of the 8-bit error compressor, then reset. */
      if (t < e_lo) t = e_lo;
      if (t > e_hi) t = e_hi;
      if (reset) t = 0.0f;
      err[lo + j] = t;
    }
  }
}

/*
 * Receiver step, §3.3 Eqn (8): decompress every rank's codes and average them
 * in high precision, for elements [i0, i1) of a bucket.  Each term is
 * f32(q)*Delta; the terms are summed in rank order 0..W-1 in fp32 and the sum
 * is divided by W.  If mean64 is not NULL it receives the same average formed
 * in fp64 from the same fp32 terms (for measuring rounding error).
 */
void oracle_decode_reduce(int bits, int block, const uint8_t* const* codes,
                          const float* const* scales, int W, int64_t i0, int64_t i1,
                          float* mean, double* mean64) {
  const int64_t bytes_per_block = (int64_t)block * bits / 8;
  for (int64_t i = i0; i < i1; ++i) {
    const int64_t b = i / block;
    const int j = (int)(i % block);
    float acc = 0.0f;
    double acc64 = 0.0;
    for (int w = 0; w < W; ++w) {
      int q = get_code(codes[w] + b * bytes_per_block, bits, j);
      float d = (float)q * scales[w][b];
      acc = (w == 0) ? d : acc + d;
      acc64 += (double)d;
    }
    mean[i] = acc / (float)W;
    if (mean64) mean64[i] = acc64 / (double)W;
  }
}

/*
 * Receiver step fused with the optimizer, §4 Eqn (9): the averaged low-bit
 * gradient g~ of Eqn (8) drives one Adam(W) update of param, m, v for the
 * elements [i0, i1).  g~ is formed exactly as in oracle_decode_reduce.
 * The update is Kingma & Ba's Adam with decoupled weight decay.  Their
 * Algorithm 1 divides m by 1 - beta1^t and v by 1 - beta2^t and steps by
 * lr * m_hat / (sqrt(v_hat) + eps); here the two corrections are folded, the
 * first into the step size (c1) and the root of the second into the
 * denominator (c2), the arrangement of torch.optim.AdamW with its division by
 * sqrt(1 - beta2^t) taken as a product with the rounded reciprocal.  In exact
 * arithmetic both are the same update (eps stays outside the corrected root);
 * in fp32 they round differently:
 *   p   = p - (lr*wd)*p
 *   m   = beta1*m + (1-beta1)*g
 *   v   = beta2*v + (1-beta2)*(g*g)
 *   den = sqrt(v)*c2 + eps            with c2 = 1/sqrt(1 - beta2^t)
 *       (eps inside the root:  den = sqrt(v*c2 + eps) with c2 = 1/(1 - beta2^t))
 *   p   = p - c1*(m/den)              with c1 = lr/(1 - beta1^t)
 * c1 and c2 are computed in double from the fp32 hyper-parameters and rounded
 * to fp32 once; without bias correction c1 = lr and c2 = 1.
 */
void oracle_adam_step(int bits, int block, const uint8_t* const* codes,
                      const float* const* scales, int W, int64_t i0, int64_t i1,
                      float* param, float* m, float* v, uint16_t* param_bf16,
                      float lr, float beta1, float beta2, float eps, float wd,
                      int bias_correction, int eps_inside_sqrt, int64_t t) {
  const int64_t bytes_per_block = (int64_t)block * bits / 8;
  const float lr_wd = lr * wd;
  const float omb1 = 1.0f - beta1;
  const float omb2 = 1.0f - beta2;
  float c1 = lr, c2 = 1.0f;
  if (bias_correction) {
    double bc1 = 1.0 - pow((double)beta1, (double)t);
    double bc2 = 1.0 - pow((double)beta2, (double)t);
    c1 = (float)((double)lr / bc1);
    c2 = eps_inside_sqrt ? (float)(1.0 / bc2) : (float)(1.0 / sqrt(bc2));
  }
  for (int64_t i = i0; i < i1; ++i) {
    const int64_t b = i / block;
    const int j = (int)(i % block);
    float acc = 0.0f;
    for (int w = 0; w < W; ++w) {
      int q = get_code(codes[w] + b * bytes_per_block, bits, j);
      float d = (float)q * scales[w][b];
      acc = (w == 0) ? d : acc + d;
    }
    float g = acc / (float)W;

    float p = param[i];
    float decay = lr_wd * p;
    p = p - decay;
    float mi = beta1 * m[i];
    float mg = omb1 * g;
    mi = mi + mg;
    float gg = g * g;
    float vi = beta2 * v[i];
    float vg = omb2 * gg;
    vi = vi + vg;
    float den;
    if (eps_inside_sqrt) {
      float vs = vi * c2;
      float s = vs + eps;
      den = sqrtf(s);
    } else {
      float r = sqrtf(vi);
      float rs = r * c2;
      den = rs + eps;
    }
    float ratio = mi / den;
    float step = c1 * ratio;
    p = p - step;
    param[i] = p;
    m[i] = mi;
    v[i] = vi;
    if (param_bf16) param_bf16[i] = f32_to_bf16_rne(p);
  }
}

/*
 * Receiver step fused with LoCo-SGD, §4: theta_{k+1} = theta_k - eta * g~_k with
 * g~ the average of Eqn (8) (formed as in oracle_decode_reduce), for elements
 * [i0, i1).  If param_bf16 is not NULL it receives the updated parameter
 * rounded to bf16 (nearest, halves to even): the 16-bit copy that the sharded
 * data-parallel setting gathers (the 16-bit parameters of the Table I
 * comparison).
 */
void oracle_sgd_step(int bits, int block, const uint8_t* const* codes,
                     const float* const* scales, int W, int64_t i0, int64_t i1,
                     float* param, uint16_t* param_bf16, float lr) {
  const int64_t bytes_per_block = (int64_t)block * bits / 8;
  for (int64_t i = i0; i < i1; ++i) {
    const int64_t b = i / block;
    const int j = (int)(i % block);
    float acc = 0.0f;
    for (int w = 0; w < W; ++w) {
      int q = get_code(codes[w] + b * bytes_per_block, bits, j);
      float d = (float)q * scales[w][b];
      acc = (w == 0) ? d : acc + d;
    }
    float g = acc / (float)W;
    float step = lr * g;
    float p = param[i] - step;
    param[i] = p;
    if (param_bf16) param_bf16[i] = f32_to_bf16_rne(p);
  }
}

/*
 * Sender step with the compensation error stored in 8 bits, §3.2 Eqn (7) as
 * the paper states it: e_k = compressor(e~_k; s_e, 8) with s_e = kappa*s, and
 * Eqn (2) adds back decompressor(e_{k-1}; s_e).  Per block b the error is kept
 * as int8 codes qe and one step De_b (the decompressor multiplies by it), so
 * the state costs one byte per element (the "additional Psi bytes" of the
 * memory comparison accompanying Table I).
 *
 * Per block b, for the quant blocks [b0, b1):
 *   e_prev_i = f32(qe_i) * De_b                     (stored state, De = 0 at start)
 *   h_i      = g_i + e_prev_i                        (Eqn 2)
 *   Delta_b, inv_b, q_i, d_i = f32(q_i)*Delta_b, r_i = h_i - d_i as in oracle_compress
 *   t_i      = beta*e_prev_i + (1-beta)*r_i          (Eqn 5)
 *   De_b'    = Delta_b / kappa ;  inv_e = kappa * inv_b   (s_e = kappa*s)
 *   qe_i'    = Round_8-bit(t_i * inv_e)              (Eqn 7: nearest, halves to even, [-128,127])
 *   qe_i'    = 0 every T_c steps (reset)
 * err_codes [n] int8 and err_steps [nb] fp32 are updated in place.
 */
void oracle_compress_e8(int bits, int block, int fixed_mode, float fixed_scale,
                        float beta, float kappa, int64_t reset_period,
                        const void* grad, int grad_is_bf16, int8_t* err_codes, float* err_steps,
                        int64_t n, int64_t step, uint8_t* codes, float* scales,
                        int64_t b0, int64_t b1) {
  const float qmax = (float)((1 << (bits - 1)) - 1);
  const float one_minus_beta = 1.0f - beta;
  const int reset = (reset_period > 0) && (step % reset_period == 0);
  const int64_t bytes_per_block = (int64_t)block * bits / 8;
  float h[1024], prev[1024];

  for (int64_t b = b0; b < b1; ++b) {
    const int64_t lo = b * block;
    int64_t cnt = n - lo;
    if (cnt > block) cnt = block;

    /* Eqn (2): compensate with the decompressed 8-bit error. */
    const float de_prev = err_steps[b];
    for (int64_t j = 0; j < cnt; ++j) {
      prev[j] = (float)err_codes[lo + j] * de_prev;
      float g = grad_at(grad, grad_is_bf16, lo + j);
      h[j] = g + prev[j];
    }

    float delta, inv;
    if (fixed_mode) {
      delta = 1.0f / fixed_scale;
      inv = fixed_scale;
    } else {
      float amax = 0.0f;
      for (int64_t j = 0; j < cnt; ++j) {
        float a = fabsf(h[j]);
        if (a > amax) amax = a;
      }
      inv = (amax == 0.0f) ? 0.0f : qmax / amax;
      if (amax == 0.0f || isinf(inv)) {
        delta = 0.0f;
        inv = 0.0f;
      } else {
        delta = amax / qmax;
      }
    }
    scales[b] = delta;

    /* The 8-bit error compressor of scale s_e = kappa*s (Eqn 7); an s_e that
     * overflows fp32 stores code 0, like a zero step. */
    const float de_new = delta / kappa;
    float inv_e = kappa * inv;
    if (isinf(inv_e)) inv_e = 0.0f;
    err_steps[b] = de_new;

    uint8_t* blk = codes + b * bytes_per_block;
    for (int j = 0; j < block; ++j) {
      if (j >= cnt) {
        put_code(blk, bits, j, 0);
        continue;
      }
      float x = h[j] * inv;
      int q = round_pbit(x, bits);
      put_code(blk, bits, j, q);
      float d = (float)q * delta;
      float r = h[j] - d;
      float t1 = beta * prev[j];
      float t2 = one_minus_beta * r;
      float t = t1 + t2;
      float xe = t * inv_e;
      int qe = round_pbit(xe, 8);
      if (reset) qe = 0;
      err_codes[lo + j] = (int8_t)qe;
    }
  }
}
