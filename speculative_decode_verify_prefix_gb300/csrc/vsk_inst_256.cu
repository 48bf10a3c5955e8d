// head_dim 256 kernels of the split-KV verify attention: the one-launch
// kernel, the stream-only kernel, the column-split stream, the tensor-memory
// stream, and the combine kernel of the two-launch forms at every head_dim.
#include "verify_kernel.cuh"

namespace vsk {

KernelFn kernel_d256(bool fp8, int variant) {
  if (variant == 5) return fp8 ? static_cast<KernelFn>(vsk_kernel<256, true, 1, 1, true>)
                               : static_cast<KernelFn>(vsk_kernel<256, false, 1, 1, true>);
  if (variant == 4) return fp8 ? static_cast<KernelFn>(vsk_kernel<256, true, 2, 2>)
                               : static_cast<KernelFn>(vsk_kernel<256, false, 2, 2>);
  if (variant == 3) return fp8 ? static_cast<KernelFn>(vsk_kernel<256, true, 1, 1, false, 256, false, true>)
                               : static_cast<KernelFn>(vsk_kernel<256, false, 1, 1, false, 256, false, true>);
  if (variant == 2) return fp8 ? static_cast<KernelFn>(vsk_kernel<256, true, 1, 2, true, 256, true>)
                               : static_cast<KernelFn>(vsk_kernel<256, false, 1, 2, true, 256, true>);
  if (variant == 1) return fp8 ? static_cast<KernelFn>(vsk_kernel<256, true, 1, 2>)
                               : static_cast<KernelFn>(vsk_kernel<256, false, 1, 2>);
  return fp8 ? static_cast<KernelFn>(vsk_kernel<256, true, 1>) : static_cast<KernelFn>(vsk_kernel<256, false, 1>);
}

KernelFn kernel_tc(bool fp8, int rm) {
  if (rm == 16) return fp8 ? static_cast<KernelFn>(vtc_kernel<256, true, 16>) : static_cast<KernelFn>(vtc_kernel<256, false, 16>);
  return fp8 ? static_cast<KernelFn>(vtc_kernel<256, true, 32>) : static_cast<KernelFn>(vtc_kernel<256, false, 32>);
}

KernelFn kernel_combine(int D, bool fp8) {
  switch (D) {
    case 64: return fp8 ? static_cast<KernelFn>(vsk_combine_kernel<64, true>)
                        : static_cast<KernelFn>(vsk_combine_kernel<64, false>);
    case 128: return fp8 ? static_cast<KernelFn>(vsk_combine_kernel<128, true>)
                         : static_cast<KernelFn>(vsk_combine_kernel<128, false>);
    case 256: return fp8 ? static_cast<KernelFn>(vsk_combine_kernel<256, true>)
                         : static_cast<KernelFn>(vsk_combine_kernel<256, false>);
    default: return nullptr;
  }
}

}  // namespace vsk
