// Split-decode kernels whose K rows are Q4_0 (one translation unit per K
// format, so the formats compile in parallel).  V uses the same format; the
// kernel templates take K and V formats separately.
#include "pa_decode_impl.cuh"

namespace pa_split {

bool lookup_kernel_q4_0(int vt, int nt, KernelInfo* out) {
  if (vt != PA_Q4_0) return false;
  switch (nt) {
    case 1: *out = kernel_info<PA_Q4_0, PA_Q4_0, 1>(); return true;
    case 2: *out = kernel_info<PA_Q4_0, PA_Q4_0, 2>(); return true;
    case 3: *out = kernel_info<PA_Q4_0, PA_Q4_0, 3>(); return true;
    default: return false;
  }
}

}  // namespace pa_split
