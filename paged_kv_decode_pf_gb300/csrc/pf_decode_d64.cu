// head_dim = 64 instantiations of the decode / partition kernel:
// 4 warps per CTA, 4 stages of 16-token K+V tiles (4 KiB) per warp.
#include "pf_partition.cuh"

// Warps per CTA and stages per warp (compile-time tunables).
#ifndef PF_D64_WARPS
#define PF_D64_WARPS 4
#endif
#ifndef PF_D64_STAGES
#define PF_D64_STAGES 4
#endif

namespace pf {

cudaError_t launch_decode_d64(const DecodeParams& p, int group, int mode, cudaStream_t stream) {
    return launch_decode_for_dim<64, PF_D64_WARPS, PF_D64_STAGES>(p, group, mode, stream);
}

}  // namespace pf
