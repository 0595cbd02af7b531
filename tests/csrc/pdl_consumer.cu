// pdl_consumer.cu -- test helper (not part of the library): a kernel that follows
// the projection on the stream with programmatic dependent launch and counts how
// many of the projection's outputs differ from a reference copy at the moment it
// reads them.  With wait = 0 it reads without griddepcontrol.wait (a consumer that
// relies on the producer's trigger order); with wait = 1 it waits first.
#include <cuda_runtime.h>
#include <stdint.h>

__global__ void pdl_consumer_kernel(const uint32_t *out, const uint32_t *ref, int n_words, int wait,
                                    unsigned long long *mismatches) {
    if (wait) asm volatile("griddepcontrol.wait;" ::: "memory");
    int bad = 0;
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n_words; i += gridDim.x * blockDim.x) {
        uint32_t v;
        asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(out + i) : "memory");
        bad += (v != ref[i]);
    }
    if (bad) atomicAdd(mismatches, static_cast<unsigned long long>(bad));
}

extern "C" int pdl_consumer_launch(const void *out, const void *ref, int n_words, int wait, void *mismatches,
                                   void *stream) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(4, 1, 1);
    cfg.blockDim = dim3(256, 1, 1);
    cfg.stream = static_cast<cudaStream_t>(stream);
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    return static_cast<int>(cudaLaunchKernelEx(&cfg, pdl_consumer_kernel, static_cast<const uint32_t *>(out),
                                               static_cast<const uint32_t *>(ref), n_words, wait,
                                               static_cast<unsigned long long *>(mismatches)));
}
