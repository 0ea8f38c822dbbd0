// placeholder: tensor-core split kernel not yet available
#include "internal.h"
namespace sdv {
bool attn_tc_supported(const AttnParams &) { return false; }
size_t attn_tc_smem_bytes(const AttnParams &) { return 0; }
cudaError_t launch_attn_tc(const AttnParams &, cudaStream_t) { return cudaErrorNotSupported; }
}  // namespace sdv
