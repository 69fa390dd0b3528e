// cf_registry.h -- table of the compiled fused-kernel instances.
#pragma once

namespace cf {

// mode 0: cf_decode_kernel (small batch tiles, CUDA-core projections,
//         sequence split across the cluster);
// mode 1: cf_rows_kernel (batched: tensor-core projections, rows split
//         across the cluster, RPC rows per block).
struct KernelEntry {
  int dtype;       // cf_dtype
  int D;           // head_dim
  int G;           // query heads per KV head
  int BT;          // batch rows per cluster
  const void* fn;  // __global__ function
  int mode = 0;
  int RPC = 0;     // rows per block (mode 1)
  // Only chosen when the caller asks for exactly this batch tile and rows per
  // block (instances kept to measure other cluster sizes, N = BT / RPC).
  bool explicit_only = false;
};

// Each instantiation unit (cf_inst_*.cu) defines one of these.
int registry_f32(const KernelEntry** out);
int registry_f16(const KernelEntry** out);
int registry_bf16(const KernelEntry** out);
int registry_rows(const KernelEntry** out);
int registry_rows_sweep(const KernelEntry** out);

}  // namespace cf
