// Batched fused decode kernel instances that differ from the default ones
// only in the cluster size N = BT / RPC: they exist to measure the choice of
// N per head dimension and query-group size (the pages fix it per head
// dimension for Hopper).  Chosen only when a config asks for their exact
// batch tile and rows per block.
#include "cf_kernel_rows.cuh"
#include "cf_registry.h"

namespace cf {
static const KernelEntry kEntries[] = {
    // dtype, D, G, BT, fn, mode, RPC, explicit_only
    {1, 64, 1, 64, (const void*)&cf_rows_kernel<__half, 64, 1, 64, 32>, 1, 32, true},
    {1, 64, 1, 64, (const void*)&cf_rows_kernel<__half, 64, 1, 64, 8>, 1, 8, true},
    {1, 64, 1, 64, (const void*)&cf_rows_kernel<__half, 64, 1, 64, 4>, 1, 4, true},
    {2, 128, 4, 4, (const void*)&cf_rows_kernel<__nv_bfloat16, 128, 4, 4, 4>, 1, 4, true},
    {2, 128, 4, 4, (const void*)&cf_rows_kernel<__nv_bfloat16, 128, 4, 4, 2>, 1, 2, true},
    {2, 128, 4, 8, (const void*)&cf_rows_kernel<__nv_bfloat16, 128, 4, 8, 1>, 1, 1, true},
};
int registry_rows_sweep(const KernelEntry** out) {
  *out = kEntries;
  return (int)(sizeof(kEntries) / sizeof(kEntries[0]));
}
}  // namespace cf
