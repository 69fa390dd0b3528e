// Fused decode kernel instances with fp16 storage.
#include "cf_kernel.cuh"
#include "cf_registry.h"

namespace cf {
static const KernelEntry kEntries[] = {
    {1, 128, 1, 1, (const void*)&cf_decode_kernel<__half, 128, 1, 1, 2>},
    {1, 128, 1, 4, (const void*)&cf_decode_kernel<__half, 128, 1, 4, 1>},
    {1, 64, 1, 1, (const void*)&cf_decode_kernel<__half, 64, 1, 1, 2>},
    {1, 64, 1, 4, (const void*)&cf_decode_kernel<__half, 64, 1, 4, 1>},
    {1, 128, 4, 1, (const void*)&cf_decode_kernel<__half, 128, 4, 1, 1>},
    {1, 64, 4, 1, (const void*)&cf_decode_kernel<__half, 64, 4, 1, 1>},
};
int registry_f16(const KernelEntry** out) {
  *out = kEntries;
  return (int)(sizeof(kEntries) / sizeof(kEntries[0]));
}
}  // namespace cf
