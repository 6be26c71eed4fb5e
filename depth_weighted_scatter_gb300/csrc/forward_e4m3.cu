// forward_e4m3.cu -- instantiates the forward kernel for FP8 E4M3 inputs and fp16 output,
// one entry point per channel count (compiled in its own unit to build in parallel).
#include "forward_impl.cuh"

namespace bevpool {

cudaError_t launch_forward_e4m3(const ForwardArgs &a) {
    switch (a.C) {
        case 8: return launch_forward_t<kDtypeE4M3, 8, kOutF16>(a);
        case 16: return launch_forward_t<kDtypeE4M3, 16, kOutF16>(a);
        case 32: return launch_forward_t<kDtypeE4M3, 32, kOutF16>(a);
        case 64: return launch_forward_t<kDtypeE4M3, 64, kOutF16>(a);
        case 80: return launch_forward_t<kDtypeE4M3, 80, kOutF16>(a);
        case 96: return launch_forward_t<kDtypeE4M3, 96, kOutF16>(a);
        case 128: return launch_forward_t<kDtypeE4M3, 128, kOutF16>(a);
        case 160: return launch_forward_t<kDtypeE4M3, 160, kOutF16>(a);
        case 192: return launch_forward_t<kDtypeE4M3, 192, kOutF16>(a);
        case 256: return launch_forward_t<kDtypeE4M3, 256, kOutF16>(a);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace bevpool
