// cf_registry.h -- table of the compiled fused-kernel instances.
#pragma once

namespace cf {

struct KernelEntry {
  int dtype;       // cf_dtype
  int D;           // head_dim
  int G;           // query heads per KV head
  int BT;          // batch rows per cluster
  const void* fn;  // __global__ function
};

// Each instantiation unit (cf_inst_*.cu) defines one of these.
int registry_f32(const KernelEntry** out);
int registry_f16(const KernelEntry** out);
int registry_bf16(const KernelEntry** out);

}  // namespace cf
