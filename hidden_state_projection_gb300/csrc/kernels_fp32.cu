// kernels_fp32.cu -- instances of the streaming kernel for one element type.
#include "launch_impl.cuh"

namespace hsp {

cudaError_t launch_fp32(const LaunchReq &r) { return launch_compute<kFmaFp32>(r); }

}  // namespace hsp
