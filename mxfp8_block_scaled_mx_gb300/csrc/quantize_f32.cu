// quantize_f32.cu -- the MX quantization launchers for FP32 input (the
// same kernel as for bf16, with 64-column tiles).
#include "quantize_kernel.cuh"

namespace mx {

cudaError_t launch_quantize_f32(const QuantizeParams& p, const CUtensorMap& tmap_x,
                                const CUtensorMap* tmap_r, int num_sms, cudaStream_t stream) {
  return launch_quantize_dense<true>(p, tmap_x, tmap_r, num_sms, stream);
}

cudaError_t launch_quantize_grouped_f32(const QuantizeParams& p, const CUtensorMap& tmap_x,
                                        int num_sms, cudaStream_t stream) {
  return launch_quantize_groups<true>(p, tmap_x, num_sms, stream);
}

}  // namespace mx
