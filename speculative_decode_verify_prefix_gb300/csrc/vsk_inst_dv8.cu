// One-launch kernels with head_dim D != v_head_dim DV for e4m3 pools (the
// bf16 ones are in vsk_inst_dv.cu).
#include "verify_kernel.cuh"

namespace vsk {

KernelFn kernel_dv8(int D, int DV) {
  if (D == 64 && DV == 128) return vsk_kernel<64, true, 1, 1, false, 128>;
  if (D == 64 && DV == 256) return vsk_kernel<64, true, 1, 1, false, 256>;
  if (D == 128 && DV == 64) return vsk_kernel<128, true, 1, 1, false, 64>;
  if (D == 128 && DV == 256) return vsk_kernel<128, true, 1, 1, false, 256>;
  if (D == 256 && DV == 64) return vsk_kernel<256, true, 1, 1, false, 64>;
  if (D == 256 && DV == 128) return vsk_kernel<256, true, 1, 1, false, 128>;
  return nullptr;
}

}  // namespace vsk
