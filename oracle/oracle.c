/*
 * oracle.c -- float64 CPU oracle of the single-token decode attention block.
 *
 * TEST INFRASTRUCTURE ONLY (see oracle.h): loaded by tests/, smoke() and the
 * CPU baseline of bench.py, never by the CUDA path.  Plain single-threaded
 * float64 loops; each function restates the definition named in oracle.h.
 *
 * Pages cited: [CF] "ClusterFusion框架深度解析" (devpress.csdn.net),
 * [LNA] "大模型推理中的算子融合优化：LayerNorm + Attention" (asdsk.com),
 * [JAX] "解码阶段延迟优化实战" (lpnh.cn).
 */
#include "oracle.h"

#include <math.h>
#include <stdlib.h>

/* [LNA §三 stage 1]: rms = sqrt(sum_sq / hidden_dim + eps); normed = x / rms;
 * then the ln_weight multiply.  Eps sits inside the square root, as in both
 * [LNA §三] and the rsqrt(mean_square + eps) of [JAX §2.2]. */
void orc_rmsnorm(int H, const double* x, const double* g, double eps,
                 double* n) {
  double sum_sq = 0.0;
  for (int i = 0; i < H; ++i) sum_sq += x[i] * x[i];
  double rms = sqrt(sum_sq / (double)H + eps);
  for (int i = 0; i < H; ++i) n[i] = (x[i] / rms) * g[i];
}

/* y = x . W, W [K, N] row-major ([CF §1.1]: torch.mm(hidden_states, W_qkv)). */
void orc_matvec(int K, int N, const double* x, const double* W, double* y) {
  for (int j = 0; j < N; ++j) y[j] = 0.0;
  for (int i = 0; i < K; ++i) {
    const double xi = x[i];
    const double* row = W + (size_t)i * (size_t)N;
    for (int j = 0; j < N; ++j) y[j] += xi * row[j];
  }
}

/* Rotate-half RoPE [LNA §三]: pair (i, i + d/2) turned by pos * theta^(-2i/d). */
void orc_rope(int d, double theta, int pos, double* u) {
  const int half = d / 2;
  for (int i = 0; i < half; ++i) {
    double freq = pow(theta, -2.0 * (double)i / (double)d);
    double phi = (double)pos * freq;
    double c = cos(phi), s = sin(phi);
    double a = u[i], b = u[i + half];
    u[i] = a * c - b * s;
    u[i + half] = b * c + a * s;
  }
}

static double dot(int d, const double* a, const double* b) {
  double s = 0.0;
  for (int i = 0; i < d; ++i) s += a[i] * b[i];
  return s;
}

/* Two-pass softmax attention of a single decode query ([CF §1.1]
 * flash_attention(qkv) stage, written as its definition). */
void orc_attention(int d, int ntok, const double* q, const double* k,
                   ptrdiff_t kstride, const double* v, ptrdiff_t vstride,
                   double* o, double* w) {
  const double scale = 1.0 / sqrt((double)d);
  double* s = (double*)malloc(sizeof(double) * (size_t)ntok);
  double m = -INFINITY;
  for (int t = 0; t < ntok; ++t) {
    s[t] = dot(d, q, k + (ptrdiff_t)t * kstride) * scale;
    if (s[t] > m) m = s[t];
  }
  double sum = 0.0;
  for (int t = 0; t < ntok; ++t) {
    s[t] = exp(s[t] - m);
    sum += s[t];
  }
  for (int i = 0; i < d; ++i) o[i] = 0.0;
  for (int t = 0; t < ntok; ++t) {
    const double wt = s[t] / sum;
    if (w) w[t] = wt;
    const double* vt = v + (ptrdiff_t)t * vstride;
    for (int i = 0; i < d; ++i) o[i] += wt * vt[i];
  }
  free(s);
}

/* Split-KV (flash-decoding) form [CF §3.2]: per-chunk partial statistics,
 * then a max-combine and a rescaled sum-combine.  The page's sum-combine
 * omits the exp(m_c - m) rescale; it is required for the result to equal the
 * softmax, so it is applied here. */
void orc_attention_split(int d, int ntok, const double* q, const double* k,
                         ptrdiff_t kstride, const double* v,
                         ptrdiff_t vstride, int nchunks,
                         const int* chunk_ends, double* o) {
  const double scale = 1.0 / sqrt((double)d);
  double* mc = (double*)malloc(sizeof(double) * (size_t)nchunks);
  double* lc = (double*)malloc(sizeof(double) * (size_t)nchunks);
  double* oc = (double*)malloc(sizeof(double) * (size_t)nchunks * (size_t)d);
  int begin = 0;
  for (int c = 0; c < nchunks; ++c) {
    int end = chunk_ends[c];
    double* occ = oc + (size_t)c * (size_t)d;
    mc[c] = -INFINITY;
    lc[c] = 0.0;
    for (int i = 0; i < d; ++i) occ[i] = 0.0;
    for (int t = begin; t < end; ++t) {
      double st = dot(d, q, k + (ptrdiff_t)t * kstride) * scale;
      if (st > mc[c]) mc[c] = st;
    }
    for (int t = begin; t < end; ++t) {
      double st = dot(d, q, k + (ptrdiff_t)t * kstride) * scale;
      double e = exp(st - mc[c]);
      lc[c] += e;
      const double* vt = v + (ptrdiff_t)t * vstride;
      for (int i = 0; i < d; ++i) occ[i] += e * vt[i];
    }
    begin = end;
  }
  (void)ntok;
  /* ClusterReduce(max) of the statistics ... */
  double m = -INFINITY;
  for (int c = 0; c < nchunks; ++c)
    if (mc[c] > m) m = mc[c];
  /* ... then ClusterReduce(sum) of the rescaled partials. */
  double l = 0.0;
  for (int i = 0; i < d; ++i) o[i] = 0.0;
  for (int c = 0; c < nchunks; ++c) {
    if (lc[c] == 0.0) continue; /* empty chunk */
    double r = exp(mc[c] - m);
    l += lc[c] * r;
    const double* occ = oc + (size_t)c * (size_t)d;
    for (int i = 0; i < d; ++i) o[i] += occ[i] * r;
  }
  for (int i = 0; i < d; ++i) o[i] /= l;
  free(mc);
  free(lc);
  free(oc);
}

int orc_decode_row(const orc_config* c, const double* x, const double* g,
                   const double* wqkv, const double* wo, double* kc,
                   double* vc, int pos, double* out, double* dbg_n,
                   double* dbg_q, double* dbg_k, double* dbg_v,
                   double* dbg_o, double* dbg_proj) {
  const int H = c->hidden, nq = c->n_q_heads, nkv = c->n_kv_heads;
  const int d = c->head_dim, S = c->s_max;
  if (H <= 0 || nq <= 0 || nkv <= 0 || d <= 0 || (d % 2) != 0 ||
      (nq % nkv) != 0 || S <= 0)
    return -1;
  if (pos < 0 || pos >= S) return -1;
  const int C = (nq + 2 * nkv) * d;
  const int group = nq / nkv;

  double* n = (double*)malloc(sizeof(double) * (size_t)H);
  double* y = (double*)malloc(sizeof(double) * (size_t)C);
  double* o = (double*)malloc(sizeof(double) * (size_t)nq * (size_t)d);
  double* proj = (double*)malloc(sizeof(double) * (size_t)H);

  /* 1. RMSNorm [LNA §三 stage 1]. */
  orc_rmsnorm(H, x, g, c->rms_eps, n);
  /* 2. Merged QKV projection [CF §5.1], [LNA §三 stage 2]. */
  orc_matvec(H, C, n, wqkv, y);
  double* q = y;                        /* nq heads  */
  double* k = y + (size_t)nq * d;       /* nkv heads */
  double* v = y + (size_t)(nq + nkv) * d;
  /* 3. RoPE on every query and key head [LNA §三]. */
  for (int h = 0; h < nq; ++h) orc_rope(d, c->rope_theta, pos, q + (size_t)h * d);
  for (int j = 0; j < nkv; ++j) orc_rope(d, c->rope_theta, pos, k + (size_t)j * d);
  /* 4. KV-cache append at slot pos [LNA §三 stage 3]. */
  for (int j = 0; j < nkv; ++j) {
    double* kslot = kc + ((size_t)pos * nkv + j) * d;
    double* vslot = vc + ((size_t)pos * nkv + j) * d;
    for (int i = 0; i < d; ++i) {
      kslot[i] = k[(size_t)j * d + i];
      vslot[i] = v[(size_t)j * d + i];
    }
  }
  /* 5. Attention of each query head over positions 0..pos of its KV head. */
  const ptrdiff_t tstride = (ptrdiff_t)nkv * d;
  for (int h = 0; h < nq; ++h) {
    const int j = h / group;
    orc_attention(d, pos + 1, q + (size_t)h * d, kc + (size_t)j * d, tstride,
                  vc + (size_t)j * d, tstride, o + (size_t)h * d, NULL);
  }
  /* 6. Output projection and residual [CF §3.2], [LNA §一]. */
  orc_matvec(nq * d, H, o, wo, proj);
  for (int i = 0; i < H; ++i) out[i] = x[i] + proj[i];

  if (dbg_n)
    for (int i = 0; i < H; ++i) dbg_n[i] = n[i];
  if (dbg_q)
    for (int i = 0; i < nq * d; ++i) dbg_q[i] = q[i];
  if (dbg_k)
    for (int i = 0; i < nkv * d; ++i) dbg_k[i] = k[i];
  if (dbg_v)
    for (int i = 0; i < nkv * d; ++i) dbg_v[i] = v[i];
  if (dbg_o)
    for (int i = 0; i < nq * d; ++i) dbg_o[i] = o[i];
  if (dbg_proj)
    for (int i = 0; i < H; ++i) dbg_proj[i] = proj[i];
  free(n);
  free(y);
  free(o);
  free(proj);
  return 0;
}

double orc_silu(double z) { return z / (1.0 + exp(-z)); }

int orc_ffn_row(int H, int I, double eps, const double* h, const double* g2,
                const double* wg, const double* wu, const double* wd,
                double* out, double* dbg_n, double* dbg_a, double* dbg_proj) {
  if (H <= 0 || I <= 0) return -1;
  double* n = (double*)malloc(sizeof(double) * (size_t)H);
  double* a = (double*)malloc(sizeof(double) * (size_t)I);
  double* proj = (double*)malloc(sizeof(double) * (size_t)H);
  /* 1. Second RMSNorm [LNA §一], the same form as the first. */
  orc_rmsnorm(H, h, g2, eps, n);
  /* 2. Gate and up projections, SiLU on the gate, elementwise product. */
  for (int i = 0; i < I; ++i) {
    const double* grow = wg + (size_t)i * (size_t)H;
    const double* urow = wu + (size_t)i * (size_t)H;
    double gs = 0.0, us = 0.0;
    for (int k = 0; k < H; ++k) {
      gs += grow[k] * n[k];
      us += urow[k] * n[k];
    }
    a[i] = orc_silu(gs) * us;
  }
  /* 3. Down projection (a . Wd) and residual [LNA §一]. */
  orc_matvec(I, H, a, wd, proj);
  for (int j = 0; j < H; ++j) out[j] = h[j] + proj[j];
  if (dbg_n)
    for (int k = 0; k < H; ++k) dbg_n[k] = n[k];
  if (dbg_a)
    for (int i = 0; i < I; ++i) dbg_a[i] = a[i];
  if (dbg_proj)
    for (int j = 0; j < H; ++j) dbg_proj[j] = proj[j];
  free(n);
  free(a);
  free(proj);
  return 0;
}

/* MLA decode row [CF §5.2], projections as DeepSeek's MLA (see oracle.h). */
int orc_mla_row(const orc_mla_config* c, const double* x, const double* g,
                const double* wq, const double* wdkv, const double* g_kv,
                const double* wukv, const double* wo, double* lc, int pos,
                double* out, double* dbg_q, double* dbg_lat, double* dbg_o,
                double* dbg_proj) {
  const int H = c->hidden, nh = c->n_heads, dn = c->d_nope, dr = c->d_rope;
  const int dv = c->d_v, dc = c->d_latent, S = c->s_max;
  if (H <= 0 || nh <= 0 || dn <= 0 || dr <= 0 || (dr % 2) != 0 || dv <= 0 ||
      dc <= 0 || S <= 0)
    return -1;
  if (pos < 0 || pos >= S) return -1;
  const int dq = dn + dr, dl = dc + dr, ntok = pos + 1;
  const int wcols = nh * (dn + dv);

  double* n = (double*)malloc(sizeof(double) * (size_t)H);
  double* q = (double*)malloc(sizeof(double) * (size_t)nh * dq);
  double* a = (double*)malloc(sizeof(double) * (size_t)dl);
  double* k = (double*)malloc(sizeof(double) * (size_t)ntok * dq);
  double* v = (double*)malloc(sizeof(double) * (size_t)ntok * dv);
  double* s = (double*)malloc(sizeof(double) * (size_t)ntok);
  double* o = (double*)malloc(sizeof(double) * (size_t)nh * dv);
  double* proj = (double*)malloc(sizeof(double) * (size_t)H);

  /* 1. RMSNorm of the hidden row [LNA §三 stage 1]. */
  orc_rmsnorm(H, x, g, c->rms_eps, n);
  /* 2. Query and latent projections. */
  orc_matvec(H, nh * dq, n, wq, q);
  orc_matvec(H, dl, n, wdkv, a);
  /* 3. RMSNorm of the compressed part, RoPE of the position parts. */
  orc_rmsnorm(dc, a, g_kv, c->rms_eps, a);
  orc_rope(dr, c->rope_theta, pos, a + dc);
  for (int h = 0; h < nh; ++h) orc_rope(dr, c->rope_theta, pos, q + (size_t)h * dq + dn);
  /* 4. Append the latent row at slot pos. */
  for (int i = 0; i < dl; ++i) lc[(size_t)pos * dl + i] = a[i];
  /* 5. Per head: keys and values of every position from the latent cache,
   *    then two-pass softmax attention. */
  const double scale = 1.0 / sqrt((double)dq);
  for (int h = 0; h < nh; ++h) {
    const double* wk = wukv + (size_t)h * (dn + dv);  /* column offset of k part */
    const double* wvv = wk + dn;                      /* column offset of v part */
    for (int t = 0; t < ntok; ++t) {
      const double* lt = lc + (size_t)t * dl;
      double* kt = k + (size_t)t * dq;
      double* vt = v + (size_t)t * dv;
      for (int j = 0; j < dn; ++j) kt[j] = 0.0;
      for (int j = 0; j < dv; ++j) vt[j] = 0.0;
      for (int i = 0; i < dc; ++i) {
        const double li = lt[i];
        const double* row = wk + (size_t)i * wcols;
        const double* vrow = wvv + (size_t)i * wcols;
        for (int j = 0; j < dn; ++j) kt[j] += li * row[j];
        for (int j = 0; j < dv; ++j) vt[j] += li * vrow[j];
      }
      for (int j = 0; j < dr; ++j) kt[dn + j] = lt[dc + j];
    }
    const double* qh = q + (size_t)h * dq;
    double m = -INFINITY;
    for (int t = 0; t < ntok; ++t) {
      s[t] = dot(dq, qh, k + (size_t)t * dq) * scale;
      if (s[t] > m) m = s[t];
    }
    double sum = 0.0;
    for (int t = 0; t < ntok; ++t) {
      s[t] = exp(s[t] - m);
      sum += s[t];
    }
    double* oh = o + (size_t)h * dv;
    for (int j = 0; j < dv; ++j) oh[j] = 0.0;
    for (int t = 0; t < ntok; ++t) {
      const double wt = s[t] / sum;
      const double* vt = v + (size_t)t * dv;
      for (int j = 0; j < dv; ++j) oh[j] += wt * vt[j];
    }
  }
  /* 6. Output projection and residual [LNA §一]. */
  orc_matvec(nh * dv, H, o, wo, proj);
  for (int i = 0; i < H; ++i) out[i] = x[i] + proj[i];

  if (dbg_q)
    for (int i = 0; i < nh * dq; ++i) dbg_q[i] = q[i];
  if (dbg_lat)
    for (int i = 0; i < dl; ++i) dbg_lat[i] = a[i];
  if (dbg_o)
    for (int i = 0; i < nh * dv; ++i) dbg_o[i] = o[i];
  if (dbg_proj)
    for (int i = 0; i < H; ++i) dbg_proj[i] = proj[i];
  free(n);
  free(q);
  free(a);
  free(k);
  free(v);
  free(s);
  free(o);
  free(proj);
  return 0;
}
