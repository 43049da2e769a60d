/*
 * kvq_oracle.c -- plain, slow CPU reference of the quantized-KV decode path.
 *
 * TEST INFRASTRUCTURE ONLY.  Only tests/, __graft_entry__.smoke() and the
 * cpu_baseline leg of bench.py may load this library.  It shares no code,
 * header or table with the CUDA library and includes nothing of it.
 *
 * What it computes, and from which passage:
 *   - quantize_group: the round-to-nearest asymmetric quantizer
 *     Q(X) = round((X - z) / s), X' = Q(X) * s + z  (KIVI page, "方法细节",
 *     first formula), with s = (max - min) / (2^b - 1), z = min and the
 *     unsigned range [0, 2^b - 1] with clamping (WindowQuant page §3.3.3,
 *     Eq.14 and Eq.16).  The fp32 expression order below is the library's
 *     documented codec, so codes, scales and zeros are compared bit for bit.
 *   - K per channel over groups of G tokens, V per token over groups of G
 *     channels (KIVI page, "方法细节": per-channel Key, per-token Value).
 *   - dequantization and attention in fp64: a_t = scale * q . k_t,
 *     p = softmax(a), o = sum_t p_t v_t (KIVI page, "背景知识与设计原则",
 *     A = Softmax(t_Q X_K^T), t_O = A X_V; KIVI Algorithm 1 decoding branch,
 *     A = Concat(t_Q Q(X_Kg)^T, t_Q X_Kr^T), t_O = A_g Q(X_Vg) + A_r X_Vr).
 *   - window similarity: cosine between summed window keys and summed text
 *     keys (WindowQuant page §3.2.1, Eq.8, with the library's reading).
 *
 * Compiled with -ffp-contract=off so that no multiply-add is fused.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ---- IEEE binary16 <-> binary32 (compiler's _Float16, round to nearest even) */
static float h2f(uint16_t h) {
  _Float16 v;
  memcpy(&v, &h, sizeof v);
  return (float)v;
}
static uint16_t f2h(float f) {
  _Float16 v = (_Float16)f;
  uint16_t h;
  memcpy(&h, &v, sizeof h);
  return h;
}

float orc_h2f(uint16_t h) { return h2f(h); }
uint16_t orc_f2h(float f) { return f2h(f); }

/* ---- the quantizer: one group of n fp16 values x[i*stride] ---------------- */
void orc_quantize_group(const uint16_t* x, int n, int stride, int bits,
                        uint8_t* code, int code_stride, uint16_t* s_out,
                        uint16_t* z_out) {
  const int qmax = (1 << bits) - 1;
  float mn = h2f(x[0]);
  float mx = mn;
  for (int i = 1; i < n; ++i) {
    float v = h2f(x[(long)i * stride]);
    if (v < mn) mn = v;
    if (v > mx) mx = v;
  }
  float s32 = (mx - mn) / (float)qmax;
  uint16_t s_h = f2h(s32);
  uint16_t z_h = f2h(mn); /* mn is an fp16 value, so this is exact */
  float s = h2f(s_h);
  float z = h2f(z_h);
  for (int i = 0; i < n; ++i) {
    int q = 0;
    if (s != 0.0f) {
      float t = (h2f(x[(long)i * stride]) - z) / s;
      float r = rintf(t);
      if (r < 0.0f) r = 0.0f;
      if (r > (float)qmax) r = (float)qmax;
      q = (int)r;
    }
    code[(long)i * code_stride] = (uint8_t)q;
  }
  *s_out = s_h;
  *z_out = z_h;
}

/* ---- the integer-zero-point quantizer (WindowQuant page §3.3.3) ----------
 * Eq.16: s = (max - min) / (qmax - qmin), z = qmin - round(min / s);
 * Eq.14: Q = clamp(round(x / s) + z, qmin, qmax);
 * Eq.15: X' = s (Q - z);  unsigned range, qmin = 0.
 * s is stored as fp16 and used rounded (as in the KIVI quantizer); z is an
 * integer, stored as a 16-bit two's-complement value in the zero slot, and
 * the codes are computed with exactly the stored s and z, so that Eq.15 of
 * the stored values is the dequantization.  Where Eq.16 is undefined or z
 * would not fit 16 bits the following readings hold:
 *   - a constant group (max = min), or one whose s rounds to 0, takes
 *     s = |min| (exact in fp16); Eq.16 then gives z = -sign(min) and Eq.14
 *     codes 0 for the constant, so Eq.15 gives it back exactly (min = 0:
 *     s = 0, z = 0, codes 0);
 *   - if |round(min / s)| > 32767, s is raised to the smallest fp16 value
 *     for which it is not: a coarser grid, whose step is still below an
 *     fp16 ulp of min.  fp16 inputs give |min| / range < 2^11 and an fp16 s
 *     is at least 2/3 of range / qmax, so this never happens at 2 bits, at
 *     4 bits only with a subnormal s, at 8 bits for groups whose range is
 *     below about |min| / 128. */
static uint16_t f2h_up(float t) { /* smallest fp16 >= t, t >= 0 finite */
  uint16_t h = f2h(t);
  if (h2f(h) < t) ++h;
  return h;
}

void orc_quantize_group_intz(const uint16_t* x, int n, int stride, int bits,
                             uint8_t* code, int code_stride, uint16_t* s_out,
                             uint16_t* z_out) {
  const int qmax = (1 << bits) - 1;
  float mn = h2f(x[0]);
  float mx = mn;
  for (int i = 1; i < n; ++i) {
    float v = h2f(x[(long)i * stride]);
    if (v < mn) mn = v;
    if (v > mx) mx = v;
  }
  float s32 = (mx - mn) / (float)qmax;
  uint16_t s_h = f2h(s32);
  float s = h2f(s_h);
  if (s == 0.0f) {
    s_h = f2h(fabsf(mn));
    s = h2f(s_h);
  }
  float zr = 0.0f; /* round(min / s), an integer */
  if (s != 0.0f) {
    zr = rintf(mn / s);
    if (fabsf(zr) > 32767.0f) {
      s_h = f2h_up(fabsf(mn) / 32767.0f);
      for (int k = 0; k < 8 && fabsf(rintf(mn / h2f(s_h))) > 32767.0f; ++k) ++s_h;
      s = h2f(s_h);
      zr = rintf(mn / s);
    }
  }
  const int z = -(int)zr;
  for (int i = 0; i < n; ++i) {
    int q = 0;
    if (s != 0.0f) {
      float r = rintf(h2f(x[(long)i * stride]) / s) + (float)z;
      if (r < 0.0f) r = 0.0f;
      if (r > (float)qmax) r = (float)qmax;
      q = (int)r;
    }
    code[(long)i * code_stride] = (uint8_t)q;
  }
  *s_out = s_h;
  *z_out = (uint16_t)(int16_t)z;
}

/* K block of G tokens x D channels (row-major [G][D]): one group per channel;
 * intz selects the integer-zero-point quantizer. */
void orc_quantize_k_block(const uint16_t* x, int G, int D, int bits,
                          uint8_t* codes, uint16_t* s, uint16_t* z, int intz) {
  for (int c = 0; c < D; ++c) {
    if (intz) orc_quantize_group_intz(x + c, G, D, bits, codes + c, D, s + c, z + c);
    else orc_quantize_group(x + c, G, D, bits, codes + c, D, s + c, z + c);
  }
}

/* One V token of D channels: one group per G consecutive channels. */
void orc_quantize_v_token(const uint16_t* x, int D, int G, int bits,
                          uint8_t* codes, uint16_t* s, uint16_t* z, int intz) {
  for (int g = 0; g < D / G; ++g) {
    if (intz) orc_quantize_group_intz(x + g * G, G, 1, bits, codes + g * G, 1, s + g, z + g);
    else orc_quantize_group(x + g * G, G, 1, bits, codes + g * G, 1, s + g, z + g);
  }
}

/* ---- packed rows: channel c at bit offset c*bits, LSB first ---------------- */
void orc_pack_row(const uint8_t* codes, int D, int bits, uint8_t* row) {
  memset(row, 0, (size_t)D * bits / 8);
  for (int c = 0; c < D; ++c) {
    int bit = c * bits;
    row[bit / 8] |= (uint8_t)(codes[c] << (bit % 8));
  }
}

void orc_unpack_row(const uint8_t* row, int D, int bits, uint8_t* codes) {
  const int mask = (1 << bits) - 1;
  for (int c = 0; c < D; ++c) {
    int bit = c * bits;
    codes[c] = (uint8_t)((row[bit / 8] >> (bit % 8)) & mask);
  }
}

/* ---- attention of one query over L dense fp64 keys/values ----------------- */
/* out[D] = sum_t p_t V[t], p = softmax(sm_scale * K q); p_out optional [L]. */
void orc_attention_dense(int L, int D, const double* K, const double* V,
                         const double* q, double sm_scale, double* out,
                         double* p_out) {
  for (int c = 0; c < D; ++c) out[c] = 0.0;
  if (L <= 0) return;
  double* a = (double*)malloc(sizeof(double) * (size_t)L);
  double amax = -INFINITY;
  for (int t = 0; t < L; ++t) {
    double dot = 0.0;
    for (int c = 0; c < D; ++c) dot += q[c] * K[(long)t * D + c];
    a[t] = sm_scale * dot;
    if (a[t] > amax) amax = a[t];
  }
  double sum = 0.0;
  for (int t = 0; t < L; ++t) {
    a[t] = exp(a[t] - amax);
    sum += a[t];
  }
  for (int t = 0; t < L; ++t) {
    double p = a[t] / sum;
    if (p_out) p_out[t] = p;
    for (int c = 0; c < D; ++c) out[c] += p * V[(long)t * D + c];
  }
  free(a);
}

/* ---- fp64 dequantization of one code ------------------------------------
 * KIVI float zero point: X' = Q s + z ("方法细节", first formula);
 * integer zero point: X' = s (Q - z) (WindowQuant Eq.15), z the int16 in the
 * zero slot. */
static double dequant_value(int q, uint16_t s_h, uint16_t z_h, int intz) {
  const double s = (double)h2f(s_h);
  if (intz) return s * (double)(q - (int)(int16_t)z_h);
  return (double)q * s + (double)h2f(z_h);
}

/* ---- dequantize one (batch, kv-head) cache into dense fp64 K and V --------
 * Per segment s: codes/scales/zeros point at this head's slice
 * (k_codes [cap][D*bits/8], k_scale/k_zero [cap/G][D], v_codes likewise,
 * v_scale/v_zero [cap][D/Gv]: K groups of G tokens, V groups of Gv
 * channels).  The ring slices are [R][D] fp16.
 * Token order: segment 0 .. n_seg-1 packed tokens, then the ring from its
 * start slot.  Returns the token count L (same for K and V) or -1 if the
 * K and V counts differ. */
int orc_dequant_head(int D, int G, int Gv, int R, int n_seg, const int* bits,
                     const int* intz, const int* nk, const int* nv, const uint8_t* const* kc,
                     const uint16_t* const* ks, const uint16_t* const* kz,
                     const uint8_t* const* vc, const uint16_t* const* vs,
                     const uint16_t* const* vz, const uint16_t* kr,
                     const uint16_t* vr, int nkr, int nvr, int krs, int vrs,
                     double* K, double* V) {
  int Lk = nkr, Lv = nvr;
  for (int s = 0; s < n_seg; ++s) {
    Lk += nk[s];
    Lv += nv[s];
  }
  if (Lk != Lv) return -1;
  uint8_t codes[512];
  int t = 0;
  for (int s = 0; s < n_seg; ++s) {
    const int rb = D * bits[s] / 8;
    for (int u = 0; u < nk[s]; ++u, ++t) {
      orc_unpack_row(kc[s] + (long)u * rb, D, bits[s], codes);
      const int g = u / G;
      for (int c = 0; c < D; ++c)
        K[(long)t * D + c] = dequant_value(codes[c], ks[s][(long)g * D + c], kz[s][(long)g * D + c], intz[s]);
    }
  }
  for (int i = 0; i < nkr; ++i, ++t) {
    const int slot = (krs + i) % R;
    for (int c = 0; c < D; ++c) K[(long)t * D + c] = (double)h2f(kr[(long)slot * D + c]);
  }
  t = 0;
  for (int s = 0; s < n_seg; ++s) {
    const int rb = D * bits[s] / 8;
    for (int u = 0; u < nv[s]; ++u, ++t) {
      orc_unpack_row(vc[s] + (long)u * rb, D, bits[s], codes);
      for (int c = 0; c < D; ++c) {
        const int g = c / Gv;
        V[(long)t * D + c] =
            dequant_value(codes[c], vs[s][(long)u * (D / Gv) + g], vz[s][(long)u * (D / Gv) + g], intz[s]);
      }
    }
  }
  for (int i = 0; i < nvr; ++i, ++t) {
    const int slot = (vrs + i) % R;
    for (int c = 0; c < D; ++c) V[(long)t * D + c] = (double)h2f(vr[(long)slot * D + c]);
  }
  return Lk;
}

/* ---- window similarity (WindowQuant §3.2.1) --------------------------------
 * keys [B][H][M][D] fp16, text [B][H][N][D] fp16.  For batch b and window w:
 * Wv = sum over the window's tokens of the concatenated H*D key vector,
 * Tv = the same sum over the text tokens; cos_bw = Wv.Tv / (|Wv| |Tv|)
 * (0 when a norm is 0).  sim[w] = mean over b of cos_bw.  Sums of fp16
 * values in fp64 are exact for these sizes. */
void orc_window_sims(const uint16_t* keys, const uint16_t* text, int B, int H,
                     int M, int N, int D, int S, double* sim) {
  const int nw = M / S;
  double* Tv = (double*)malloc(sizeof(double) * (size_t)H * D);
  double* Wv = (double*)malloc(sizeof(double) * (size_t)H * D);
  for (int w = 0; w < nw; ++w) sim[w] = 0.0;
  for (int b = 0; b < B; ++b) {
    for (int h = 0; h < H; ++h)
      for (int c = 0; c < D; ++c) {
        double acc = 0.0;
        for (int t = 0; t < N; ++t)
          acc += (double)h2f(text[(((long)b * H + h) * N + t) * D + c]);
        Tv[h * D + c] = acc;
      }
    double tt = 0.0;
    for (int i = 0; i < H * D; ++i) tt += Tv[i] * Tv[i];
    for (int w = 0; w < nw; ++w) {
      for (int h = 0; h < H; ++h)
        for (int c = 0; c < D; ++c) {
          double acc = 0.0;
          for (int t = w * S; t < w * S + S; ++t)
            acc += (double)h2f(keys[(((long)b * H + h) * M + t) * D + c]);
          Wv[h * D + c] = acc;
        }
      double wt = 0.0, ww = 0.0;
      for (int i = 0; i < H * D; ++i) {
        wt += Wv[i] * Tv[i];
        ww += Wv[i] * Wv[i];
      }
      double cosv = (ww > 0.0 && tt > 0.0) ? wt / (sqrt(ww) * sqrt(tt)) : 0.0;
      sim[w] += cosv;
    }
  }
  for (int w = 0; w < nw; ++w) sim[w] = sim[w] / (double)B;
  free(Tv);
  free(Wv);
}
