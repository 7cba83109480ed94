// quantize.cu -- the MX quantization launchers for bf16 input (the FP32
// ones are instantiated in their own translation unit, quantize_f32.cu, so
// that the two compile in parallel).
#include "quantize_kernel.cuh"

namespace mx {

cudaError_t launch_quantize(const QuantizeParams& p, const CUtensorMap& tmap_x,
                            const CUtensorMap* tmap_r, int num_sms, cudaStream_t stream) {
  return launch_quantize_dense<false>(p, tmap_x, tmap_r, num_sms, stream);
}

cudaError_t launch_quantize_grouped(const QuantizeParams& p, const CUtensorMap& tmap_x,
                                    int num_sms, cudaStream_t stream) {
  return launch_quantize_groups<false>(p, tmap_x, num_sms, stream);
}

}  // namespace mx
