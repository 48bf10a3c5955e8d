// head_dim 128 kernels of the split-KV verify attention (one translation unit
// per head_dim, so the library's kernels compile in parallel).
#include "verify_kernel.cuh"

namespace vsk {

KernelFn kernel_d128(bool fp8, int mtw, bool so, bool cl) {
  if (cl) return fp8 ? static_cast<KernelFn>(vsk_kernel<128, true, 1, 1, true, 128, true>)
                     : static_cast<KernelFn>(vsk_kernel<128, false, 1, 1, true, 128, true>);
  if (so) {
    if (mtw == 2) return fp8 ? static_cast<KernelFn>(vsk_kernel<128, true, 2, 1, true>)
                             : static_cast<KernelFn>(vsk_kernel<128, false, 2, 1, true>);
    return fp8 ? static_cast<KernelFn>(vsk_kernel<128, true, 1, 1, true>)
               : static_cast<KernelFn>(vsk_kernel<128, false, 1, 1, true>);
  }
  if (mtw == 2) return fp8 ? static_cast<KernelFn>(vsk_kernel<128, true, 2>) : static_cast<KernelFn>(vsk_kernel<128, false, 2>);
  return fp8 ? static_cast<KernelFn>(vsk_kernel<128, true, 1>) : static_cast<KernelFn>(vsk_kernel<128, false, 1>);
}

}  // namespace vsk
