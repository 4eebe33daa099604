// head_dim = 128 instantiations of the decode / partition kernel:
// 4 warps per CTA, 2 stages of 16-token K+V tiles (8 KiB) per warp, three CTAs per SM.
#include "pf_partition.cuh"

// Warps per CTA and stages per warp (compile-time tunables).
#ifndef PF_D128_WARPS
#define PF_D128_WARPS 4
#endif
#ifndef PF_D128_STAGES
#define PF_D128_STAGES 2
#endif

namespace pf {

cudaError_t launch_decode_d128(const DecodeParams& p, int group, int mode, cudaStream_t stream) {
    return launch_decode_for_dim<128, PF_D128_WARPS, PF_D128_STAGES>(p, group, mode, stream);
}

}  // namespace pf
