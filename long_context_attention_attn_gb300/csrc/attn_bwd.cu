// Backward attention (placeholder until the fused kernel lands).
#include "internal.h"

namespace gb300 {

cudaError_t launch_attn_bwd(const BwdLaunch&, cudaStream_t) { return cudaErrorNotSupported; }

}  // namespace gb300
