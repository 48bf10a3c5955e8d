// One-launch kernels with head_dim D != v_head_dim DV, D and DV in
// {64, 128, 256}: bf16 pools here, e4m3 pools in vsk_inst_dv8.cu.
#include "verify_kernel.cuh"

namespace vsk {

KernelFn kernel_dv8(int D, int DV);

KernelFn kernel_dv(int D, int DV, bool fp8) {
  if (fp8) return kernel_dv8(D, DV);
  if (D == 64 && DV == 128) return vsk_kernel<64, false, 1, 1, false, 128>;
  if (D == 64 && DV == 256) return vsk_kernel<64, false, 1, 1, false, 256>;
  if (D == 128 && DV == 64) return vsk_kernel<128, false, 1, 1, false, 64>;
  if (D == 128 && DV == 256) return vsk_kernel<128, false, 1, 1, false, 256>;
  if (D == 256 && DV == 64) return vsk_kernel<256, false, 1, 1, false, 64>;
  if (D == 256 && DV == 128) return vsk_kernel<256, false, 1, 1, false, 128>;
  return nullptr;
}

}  // namespace vsk
