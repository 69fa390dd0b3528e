// cf_unfused.h -- parameters of the three-kernel (unfused) decode step in
// cf_unfused.cu, launched by cf_decode_attn_block_unfused (cf_api.cu).
#pragma once

#include <cuda_runtime.h>

namespace cf {

struct UfParams {
  const void* hidden;    // [B, H]
  const void* ln_w;      // [H]
  const void* w_qkv;     // [H, (nq+2nkv)*D]
  const void* w_o;       // [nq*D, H]
  void* k_cache;         // [B, S, nkv, D]
  void* v_cache;         // [B, S, nkv, D]
  const int* positions;  // [B]
  void* out;             // [B, H]
  float* y;              // [B, (nq+2nkv)*D] projection, fp32 (HBM intermediate; zero
                         // between steps: the attention clears what it read)
  float* part;           // [B, nkv, NS, G, D+4] split partials (o, m, l)
  float* o32;            // [B, nq*D] attention output, fp32 (HBM intermediate)
  float* rinv;           // [B] RMSNorm scales (written by the QKV projection)
  float* acc;            // [B, H] fp32 accumulator, zero between launches
  int* cnt_attn;         // [B * nkv] split counters, zero between launches
  int* cnt_out;          // [B * H/64] output-tile counters, zero between launches
                         // (one per band and batch tile)
  int* errflag;
  int B, H, nq, nkv, D, S;
  int NS;                // position splits per (row, KV head)
  int KS;                // reduction splits of the output projection
  int KS1;               // reduction splits of the QKV projection (adds into y)
  float eps, qk_scale_log2;
  float turn_hi[64], turn_lo[64];  // RoPE turn rates (as in KParams)
};

// Enqueue the three kernels on `st`; returns a CF_* code.
int unfused_launch(const UfParams& p, int dtype, int G, cudaStream_t st);

}  // namespace cf
