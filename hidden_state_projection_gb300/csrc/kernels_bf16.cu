// kernels_bf16.cu -- instances of the streaming kernel for one element type.
#include "launch_impl.cuh"

namespace hsp {

cudaError_t launch_bf16(const LaunchReq &r) {
    if (r.compute == kFmaBf16) {
        if (r.bucket != 0 || r.MT != 1) return cudaErrorInvalidConfiguration;
        return r.RT == 1 ? launch_variant<kFmaBf16, 1, 1, 1, 8>(r) : launch_variant<kFmaBf16, 1, 2, 1, 8>(r);
    }
    return launch_compute<kMmaBf16>(r);
}

}  // namespace hsp
