// Entry points whose tensor-core kernels are not in this build yet.
#include "attn_internal.h"

namespace attn {
cudaError_t launch_bwd_bf16(const BwdArgs&, DeviceStatus*, cudaStream_t) { return cudaErrorNotSupported; }
cudaError_t launch_decode_bf16(const DecodeArgs&, DeviceStatus*, cudaStream_t) { return cudaErrorNotSupported; }
}  // namespace attn
