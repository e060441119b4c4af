// Two-kernel decode path: gate_up and down instantiated for Q5_0, Q5_1, Q5_K, MXFP4,
// F16 and F32 rows (the kernels are in decode_twok.cuh).
#include "decode_twok.cuh"

namespace qre {

cudaError_t launch_gate_up_types_c(const DecodeParams& p, size_t smem, cudaStream_t stream) {
  switch (p.gu_type) {
    case W_Q5_0: return launch_gu_w<W_Q5_0>(p, smem, stream);
    case W_Q5_1: return launch_gu_w<W_Q5_1>(p, smem, stream);
    case W_Q5_K: return launch_gu_w<W_Q5_K>(p, smem, stream);
    case W_MXFP4: return launch_gu_w<W_MXFP4>(p, smem, stream);
    case W_F16: return launch_gu_w<W_F16>(p, smem, stream);
    case W_F32: return launch_gu_w<W_F32>(p, smem, stream);
  }
  return cudaErrorInvalidValue;
}

cudaError_t launch_down_types_c(const DecodeParams& p, size_t smem, cudaStream_t stream) {
  switch (p.dn_type) {
    case W_Q5_0: return launch_dn_w<W_Q5_0, 8>(p, smem, stream);
    case W_Q5_1: return launch_dn_w<W_Q5_1, 8>(p, smem, stream);
    case W_Q5_K: return launch_dn_w<W_Q5_K, 8>(p, smem, stream);
    case W_MXFP4: return launch_dn_w<W_MXFP4, 8>(p, smem, stream);
    case W_F16: return launch_dn_w<W_F16, 16>(p, smem, stream);
    case W_F32: return launch_dn_w<W_F32, 16>(p, smem, stream);
  }
  return cudaErrorInvalidValue;
}

}  // namespace qre
