// fp32-input SYRK (placeholder until the split-TF32 kernel lands): every
// launch reports cudaErrorNotSupported, which the host maps to an error.
#include "kernels.cuh"

namespace hk {

size_t syrk_f32_smem_bytes() { return 0; }
cudaError_t syrk_f32_prepare() { return cudaSuccess; }
cudaError_t launch_syrk_f32(const SyrkParams&, int, cudaStream_t) { return cudaErrorNotSupported; }

}  // namespace hk
