// The rows-on-M tensor-memory stream of head_dim 256 (opt-in form).
#include "verify_tr.cuh"

namespace vsk {

KernelFn kernel_tr(bool fp8, int rm) {
  if (rm == 16) return fp8 ? static_cast<KernelFn>(vtr_kernel<true, 16>) : static_cast<KernelFn>(vtr_kernel<false, 16>);
  return fp8 ? static_cast<KernelFn>(vtr_kernel<true, 32>) : static_cast<KernelFn>(vtr_kernel<false, 32>);
}

}  // namespace vsk
