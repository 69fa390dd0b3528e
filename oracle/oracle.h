/*
 * oracle.h -- float64 CPU oracle of the single-token decode attention block.
 *
 * TEST INFRASTRUCTURE ONLY.  This library is the parity reference for the
 * CUDA path.  Only tests/, __graft_entry__.smoke() and bench.py's CPU
 * baseline may load it.  It shares no code, header, table or constant with
 * the CUDA path, and the CUDA path never calls it.
 *
 * Pages cited (by title and section):
 *   [CF]  "ClusterFusion框架深度解析：LLM推理优化的集群级通信革命"
 *         (devpress.csdn.net)
 *   [LNA] "大模型推理中的算子融合优化：LayerNorm + Attention 的 CUDA Kernel
 *         手写与验证" (asdsk.com)
 *   [JAX] "解码阶段延迟优化实战：基于JAX与XLA的LLM推理加速方案" (lpnh.cn)
 *
 * Every routine is plain float64, single-threaded, with no blocking, fusion
 * or reordering beyond the definition it restates.  Inputs are the storage
 * values converted exactly to double; nothing is rounded in between.
 *
 * Layouts (all row-major, all contiguous):
 *   x, out      [H]                 one batch row of the hidden state
 *   g           [H]                 RMSNorm weight
 *   wqkv        [H, C]              C = (nq + 2*nkv) * d; columns are
 *                                   [Q heads | K heads | V heads], each head
 *                                   d contiguous columns (x . W form)
 *   wo          [nq*d, H]           (attn . W_o form)
 *   kc, vc      [S, nkv, d]         one batch row of the KV cache
 *   wg, wu, wd  [I, H]              FFN weights, one row per intermediate
 *                                   unit (see orc_ffn_row)
 */
#ifndef CF_ORACLE_H
#define CF_ORACLE_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct {
  int hidden;      /* H   */
  int n_q_heads;   /* nq  */
  int n_kv_heads;  /* nkv; nq % nkv == 0 */
  int head_dim;    /* d, even */
  int s_max;       /* S: cache capacity per row */
  double rope_theta;
  double rms_eps;
} orc_config;

/* RMSNorm, [LNA §三 stage 1] and [JAX §2.2]:
 *   n_i = x_i * g_i / sqrt( (1/H) sum_j x_j^2 + eps ).                      */
void orc_rmsnorm(int H, const double* x, const double* g, double eps,
                 double* n);

/* y = x . W with W [K, N] row-major: y_j = sum_i x_i W[i, j].
 * [CF §1.1] (torch.mm(hidden_states, W_qkv)), [CF §5.1] (merged QKV).      */
void orc_matvec(int K, int N, const double* x, const double* W, double* y);

/* RoPE, rotate-half pairing [LNA §三 ("rotate_half")], in place on u[d]:
 *   phi_i = pos * theta^(-2i/d),  i < d/2
 *   u'_i       = u_i cos phi_i - u_{i+d/2} sin phi_i
 *   u'_{i+d/2} = u_{i+d/2} cos phi_i + u_i sin phi_i                         */
void orc_rope(int d, double theta, int pos, double* u);

/* Two-pass softmax attention of one query over ntok keys [CF §1.1]:
 *   s_t = q . k_t / sqrt(d);  w_t = exp(s_t - max s) / sum;  o = sum w_t v_t.
 * Key t sits at k + t*kstride, value t at v + t*vstride.  If w is not NULL
 * the ntok softmax weights are written there.  ntok >= 1.                   */
void orc_attention(int d, int ntok, const double* q, const double* k,
                   ptrdiff_t kstride, const double* v, ptrdiff_t vstride,
                   double* o, double* w);

/* Split-KV form of the same attention [CF §3.2 "在线softmax"]: the ntok keys
 * are cut at chunk_ends[0] < chunk_ends[1] < ... < chunk_ends[nchunks-1]
 * (== ntok); each chunk c yields (m_c, l_c, o_c) with
 *   m_c = max s,  l_c = sum exp(s - m_c),  o_c = sum exp(s - m_c) v_t,
 * and the partials are combined as m = max m_c,
 *   l = sum_c l_c exp(m_c - m),  o = sum_c o_c exp(m_c - m) / l.
 * Empty chunks (equal consecutive ends) contribute nothing.               */
void orc_attention_split(int d, int ntok, const double* q, const double* k,
                         ptrdiff_t kstride, const double* v,
                         ptrdiff_t vstride, int nchunks,
                         const int* chunk_ends, double* o);

/* One batch row of the decode attention block:
 *   n = RMSNorm(x); y = n . Wqkv; q_h, k_g, v_g sliced from y;
 *   RoPE(q_h, pos), RoPE(k_g, pos); kc[pos,g,:] = k_g; vc[pos,g,:] = v_g;
 *   o_h = attention(q_h, kc[0..pos, g(h)], vc[0..pos, g(h)]),
 *         g(h) = h / (nq/nkv)                        [LNA §三, GQA mapping];
 *   out = x + concat_h(o_h) . Wo                     [LNA §一 residual].
 * kc/vc are updated in place (slot pos only).  The dbg_* outputs may each be
 * NULL: dbg_n [H], dbg_q [nq*d] (post-RoPE), dbg_k [nkv*d] (post-RoPE),
 * dbg_v [nkv*d], dbg_o [nq*d], dbg_proj [H] (concat(o) . Wo).
 * Returns 0, or -1 if pos is outside [0, S) or the config is invalid.      */
int orc_decode_row(const orc_config* c, const double* x, const double* g,
                   const double* wqkv, const double* wo, double* kc,
                   double* vc, int pos, double* out, double* dbg_n,
                   double* dbg_q, double* dbg_k, double* dbg_v,
                   double* dbg_o, double* dbg_proj);

/* SiLU, the gate activation of the LLaMA FFN: silu(z) = z / (1 + exp(-z)). */
double orc_silu(double z);

/* The rest of the decoder block for one batch row: the second RMS Norm, the
 * FFN and its residual, in the block order of [LNA §一] ("第二个 RMS Norm、
 * FFN", LLaMA architecture).  The pages name the FFN but not its inner form;
 * the LLaMA FFN is the gated (SwiGLU) one, read here as
 *   n   = RMSNorm(h; g2)                       (as orc_rmsnorm)
 *   a_i = silu( sum_k Wg[i,k] n_k ) * ( sum_k Wu[i,k] n_k ),   i < I
 *   out_j = h_j + sum_i a_i Wd[i,j],                           j < H
 * with Wg, Wu, Wd all [I, H] row-major (row i holds intermediate unit i's
 * weights).  dbg_n [H], dbg_a [I] and dbg_proj [H] (the FFN output before the
 * residual) may each be NULL.  Returns 0, or -1 for a bad shape.           */
int orc_ffn_row(int H, int I, double eps, const double* h, const double* g2,
                const double* wg, const double* wu, const double* wd,
                double* out, double* dbg_n, double* dbg_a, double* dbg_proj);

#ifdef __cplusplus
}
#endif

#endif
