// Split-decode kernels for one (K format, V format) pair, chosen at compile
// time with -DPA_KT=<pa_type> -DPA_VT=<pa_type>; the build compiles this file
// once per pair, so the nine pairs compile in parallel.  Each unit defines
// lookup_kernel_<K>_<V>, returning the kernel for 1 to 6 n-tiles of 8 query
// rows (6 rows per token: 1, 2, 3-4, 5, 6, 7-8 tokens); 6 to 8 tokens share
// one kernel with two consumer groups.  Each unit also defines
// lookup_rows_tc_kernel_<K>_<V>, the row-tile kernel for 9 to 96 tokens.
#include "pa_rows_tc.cuh"

#if !defined(PA_KT) || !defined(PA_VT)
#error "compile with -DPA_KT=<pa_type> -DPA_VT=<pa_type>"
#endif

#define PA_LOOKUP_NAME_(k, v) lookup_kernel_##k##_##v
#define PA_LOOKUP_NAME(k, v) PA_LOOKUP_NAME_(k, v)

namespace pa_split {

bool PA_LOOKUP_NAME(PA_KT, PA_VT)(int nt, KernelInfo* out) {
  switch (nt) {
    case 1: *out = kernel_info<PA_KT, PA_VT, 1>(); return true;
    case 2: *out = kernel_info<PA_KT, PA_VT, 2>(); return true;
    case 3: *out = kernel_info<PA_KT, PA_VT, 3>(); return true;
    case 4: *out = kernel_info<PA_KT, PA_VT, 4>(); return true;
    // six to eight tokens: two groups of consumer warps, each taking three or
    // four tokens (three n-tiles); measured faster than one group of five or
    // six n-tiles, which five tokens keep
    case 5:
    case 6: *out = kernel_info<PA_KT, PA_VT, 3, 2>(); return true;
    default: return false;
  }
}

#define PA_ROWS_TC_LOOKUP_NAME_(k, v) lookup_rows_tc_kernel_##k##_##v
#define PA_ROWS_TC_LOOKUP_NAME(k, v) PA_ROWS_TC_LOOKUP_NAME_(k, v)

// Row tiles (nine to 96 query tokens) on the fifth-generation tensor core.
bool PA_ROWS_TC_LOOKUP_NAME(PA_KT, PA_VT)(KernelInfo* out) {
  *out = rows_tc_kernel_info<PA_KT, PA_VT>();
  return true;
}

}  // namespace pa_split
