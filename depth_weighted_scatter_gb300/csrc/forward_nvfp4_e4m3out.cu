// forward_nvfp4_e4m3out.cu -- instantiates the forward kernel for NVFP4 features and an E4M3 output,
// one entry point per channel count (compiled in its own unit to build in parallel).
#include "forward_impl.cuh"

namespace bevpool {

cudaError_t launch_forward_nvfp4_e4m3out(const ForwardArgs &a) {
    switch (a.C) {
        case 64: return launch_forward_t<kDtypeNVFP4, 64, kOutE4M3>(a);
        case 80: return launch_forward_t<kDtypeNVFP4, 80, kOutE4M3>(a);
        case 96: return launch_forward_t<kDtypeNVFP4, 96, kOutE4M3>(a);
        case 128: return launch_forward_t<kDtypeNVFP4, 128, kOutE4M3>(a);
        case 160: return launch_forward_t<kDtypeNVFP4, 160, kOutE4M3>(a);
        case 192: return launch_forward_t<kDtypeNVFP4, 192, kOutE4M3>(a);
        case 256: return launch_forward_t<kDtypeNVFP4, 256, kOutE4M3>(a);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace bevpool
