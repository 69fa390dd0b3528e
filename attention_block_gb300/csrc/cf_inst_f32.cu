// Fused decode kernel instances with fp32 storage.
#include "cf_kernel.cuh"
#include "cf_registry.h"

namespace cf {
static const KernelEntry kEntries[] = {
    {0, 64, 1, 1, (const void*)&cf_decode_kernel<float, 64, 1, 1, 2>},
    {0, 128, 1, 1, (const void*)&cf_decode_kernel<float, 128, 1, 1, 2>},
    {0, 64, 4, 1, (const void*)&cf_decode_kernel<float, 64, 4, 1, 1>},
    {0, 128, 4, 1, (const void*)&cf_decode_kernel<float, 128, 4, 1, 1>},
};
int registry_f32(const KernelEntry** out) {
  *out = kEntries;
  return (int)(sizeof(kEntries) / sizeof(kEntries[0]));
}
}  // namespace cf
