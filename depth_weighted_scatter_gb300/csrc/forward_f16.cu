// forward_f16.cu -- instantiates the forward kernel for fp16 inputs and fp16 output,
// one entry point per channel count (compiled in its own unit to build in parallel).
#include "forward_impl.cuh"

namespace bevpool {

cudaError_t launch_forward_f16(const ForwardArgs &a) {
    switch (a.C) {
        case 8: return launch_forward_t<kDtypeF16, 8, kOutF16>(a);
        case 16: return launch_forward_t<kDtypeF16, 16, kOutF16>(a);
        case 32: return launch_forward_t<kDtypeF16, 32, kOutF16>(a);
        case 64: return launch_forward_t<kDtypeF16, 64, kOutF16>(a);
        case 80: return launch_forward_t<kDtypeF16, 80, kOutF16>(a);
        case 96: return launch_forward_t<kDtypeF16, 96, kOutF16>(a);
        case 128: return launch_forward_t<kDtypeF16, 128, kOutF16>(a);
        case 160: return launch_forward_t<kDtypeF16, 160, kOutF16>(a);
        case 192: return launch_forward_t<kDtypeF16, 192, kOutF16>(a);
        case 256: return launch_forward_t<kDtypeF16, 256, kOutF16>(a);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace bevpool
