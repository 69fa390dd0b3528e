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

/* The DeepSeek multi-head latent attention (MLA) variant of the decode block
 * [CF §5.2 DeepSeek-MLA特殊处理].  The page gives only the kernel-side
 * adaptation (the latent key/value cache partitioned across clusters, a
 * sparse ClusterReduce); the projections are read as DeepSeek's published MLA
 * with an uncompressed query (the DeepSeek-V2-Lite form):
 *   n     = RMSNorm(x; g)
 *   q     = n . Wq             Wq [H, nh*(dn+dr)]; head h = [q_nope (dn) | q_rope (dr)]
 *   a     = n . Wdkv           Wdkv [H, dc+dr];   a = [c (dc) | kr (dr)]
 *   c'    = RMSNorm(c; g_kv)   (same eps)
 *   q_rope_h <- RoPE(q_rope_h, pos), kr <- RoPE(kr, pos)  (rotate-half over dr)
 *   L[pos] = [c' | kr]         the latent cache row, dc + dr values
 *   for each head h and position t in 0..pos, with Wukv [dc, nh*(dn+dv)]
 *   (head h's columns = [k part (dn) | v part (dv)]):
 *     k_{t,h} = [ L[t, :dc] . Wukv[:, k part of h] | L[t, dc:] ]   (dn + dr)
 *     v_{t,h} =   L[t, :dc] . Wukv[:, v part of h]                 (dv)
 *     o_h     = softmax_t( q_h . k_{t,h} / sqrt(dn + dr) ) . v_{t,h}
 *   out   = x + concat_h(o_h) . Wo                Wo [nh*dv, H]
 * The keys and values are formed per position exactly as defined (no
 * absorption of Wukv into the query or the output).                       */
typedef struct {
  int hidden;      /* H  */
  int n_heads;     /* nh */
  int d_nope;      /* dn: query/key dims without position encoding */
  int d_rope;      /* dr: query/key dims with RoPE (even); the key part is shared by all heads */
  int d_v;         /* dv: value dims per head */
  int d_latent;    /* dc: compressed key/value dims */
  int s_max;       /* S: latent cache capacity per row */
  double rope_theta;
  double rms_eps;
} orc_mla_config;

/* One batch row of the MLA decode block (definition above).  lc [S, dc+dr] is
 * this row's latent cache, updated in place at slot pos only.  The dbg_*
 * outputs may each be NULL: dbg_q [nh*(dn+dr)] (rope parts rotated),
 * dbg_lat [dc+dr] (the new latent row), dbg_o [nh*dv], dbg_proj [H].
 * Returns 0, or -1 if pos is outside [0, S) or the config is invalid.      */
int orc_mla_row(const orc_mla_config* c, const double* x, const double* g,
                const double* wq, const double* wdkv, const double* g_kv,
                const double* wukv, const double* wo, double* lc, int pos,
                double* out, double* dbg_q, double* dbg_lat, double* dbg_o,
                double* dbg_proj);

#ifdef __cplusplus
}
#endif

#endif
