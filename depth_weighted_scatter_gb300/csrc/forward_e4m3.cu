// forward_e4m3.cu -- instantiates the forward kernel for FP8 E4M3 inputs,
// one entry point per channel count (compiled in its own unit to build in parallel).
#include "forward_impl.cuh"

namespace bevpool {

cudaError_t launch_forward_e4m3(const ForwardArgs &a) {
    switch (a.C) {
        case 8: return launch_forward_t<kDtypeE4M3, 8>(a);
        case 16: return launch_forward_t<kDtypeE4M3, 16>(a);
        case 32: return launch_forward_t<kDtypeE4M3, 32>(a);
        case 64: return launch_forward_t<kDtypeE4M3, 64>(a);
        case 80: return launch_forward_t<kDtypeE4M3, 80>(a);
        case 96: return launch_forward_t<kDtypeE4M3, 96>(a);
        case 128: return launch_forward_t<kDtypeE4M3, 128>(a);
        case 160: return launch_forward_t<kDtypeE4M3, 160>(a);
        case 192: return launch_forward_t<kDtypeE4M3, 192>(a);
        case 256: return launch_forward_t<kDtypeE4M3, 256>(a);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace bevpool
