// One-launch kernels with head_dim D != v_head_dim DV.
#include "verify_kernel.cuh"

namespace vsk {

KernelFn kernel_dv(int D, int DV, bool fp8) {
  (void)D;
  (void)DV;
  (void)fp8;
  return nullptr;
}

}  // namespace vsk
