// Fused decode kernel instances with bf16 storage.
#include "cf_kernel.cuh"
#include "cf_registry.h"

namespace cf {
static const KernelEntry kEntries[] = {
    {2, 128, 4, 1, (const void*)&cf_decode_kernel<__nv_bfloat16, 128, 4, 1, 1>},
    {2, 128, 4, 2, (const void*)&cf_decode_kernel<__nv_bfloat16, 128, 4, 2, 1>},
    {2, 128, 1, 1, (const void*)&cf_decode_kernel<__nv_bfloat16, 128, 1, 1, 2>},
    {2, 64, 1, 1, (const void*)&cf_decode_kernel<__nv_bfloat16, 64, 1, 1, 2>},
};
int registry_bf16(const KernelEntry** out) {
  *out = kEntries;
  return (int)(sizeof(kEntries) / sizeof(kEntries[0]));
}
}  // namespace cf
