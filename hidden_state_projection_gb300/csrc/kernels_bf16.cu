// kernels_bf16.cu -- instances of the streaming kernel for one element type.
#include "launch_impl.cuh"

namespace hsp {

cudaError_t launch_bf16(const LaunchReq &r) { return launch_compute<kMmaBf16>(r); }

}  // namespace hsp
