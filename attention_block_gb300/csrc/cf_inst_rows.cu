// Batched fused decode kernel instances (fp16 / bf16 storage).
#include "cf_kernel_rows.cuh"
#include "cf_registry.h"

namespace cf {
static const KernelEntry kEntries[] = {
    // dtype, D, G, BT, fn, mode, RPC
    {1, 64, 1, 64, (const void*)&cf_rows_kernel<__half, 64, 1, 64, 16>, 1, 16},
    {1, 64, 1, 32, (const void*)&cf_rows_kernel<__half, 64, 1, 32, 8>, 1, 8},
    {1, 64, 1, 16, (const void*)&cf_rows_kernel<__half, 64, 1, 16, 4>, 1, 4},
    {1, 128, 1, 16, (const void*)&cf_rows_kernel<__half, 128, 1, 16, 4>, 1, 4},
    {1, 128, 4, 16, (const void*)&cf_rows_kernel<__half, 128, 4, 16, 4>, 1, 4},
    {1, 128, 4, 4, (const void*)&cf_rows_kernel<__half, 128, 4, 4, 1>, 1, 1},
    {2, 128, 4, 4, (const void*)&cf_rows_kernel<__nv_bfloat16, 128, 4, 4, 1>, 1, 1},
    {2, 128, 4, 8, (const void*)&cf_rows_kernel<__nv_bfloat16, 128, 4, 8, 2>, 1, 2},
    {2, 128, 4, 16, (const void*)&cf_rows_kernel<__nv_bfloat16, 128, 4, 16, 4>, 1, 4},
    {2, 64, 1, 16, (const void*)&cf_rows_kernel<__nv_bfloat16, 64, 1, 16, 4>, 1, 4},
};
int registry_rows(const KernelEntry** out) {
  *out = kEntries;
  return (int)(sizeof(kEntries) / sizeof(kEntries[0]));
}
}  // namespace cf
