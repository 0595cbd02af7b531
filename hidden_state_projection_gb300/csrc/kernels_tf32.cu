// kernels_tf32.cu -- instances of the streaming kernel for one element type.
#include "launch_impl.cuh"

namespace hsp {

cudaError_t launch_tf32(const LaunchReq &r) { return launch_compute<kMmaTf32>(r); }

}  // namespace hsp
