// forward_f16_e4m3out.cu -- instantiates the forward kernel for fp16 inputs and an E4M3 output,
// one entry point per channel count (compiled in its own unit to build in parallel).
#include "forward_impl.cuh"

namespace bevpool {

cudaError_t launch_forward_f16_e4m3out(const ForwardArgs &a) {
    switch (a.C) {
        case 16: return launch_forward_t<kDtypeF16, 16, kOutE4M3>(a);
        case 32: return launch_forward_t<kDtypeF16, 32, kOutE4M3>(a);
        case 64: return launch_forward_t<kDtypeF16, 64, kOutE4M3>(a);
        case 80: return launch_forward_t<kDtypeF16, 80, kOutE4M3>(a);
        case 96: return launch_forward_t<kDtypeF16, 96, kOutE4M3>(a);
        case 128: return launch_forward_t<kDtypeF16, 128, kOutE4M3>(a);
        case 160: return launch_forward_t<kDtypeF16, 160, kOutE4M3>(a);
        case 192: return launch_forward_t<kDtypeF16, 192, kOutE4M3>(a);
        case 256: return launch_forward_t<kDtypeF16, 256, kOutE4M3>(a);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace bevpool
