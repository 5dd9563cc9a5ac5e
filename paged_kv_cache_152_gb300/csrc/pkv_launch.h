// pkv_launch.h -- kernel launch with programmatic dependent launch enabled.
//
// The kernel may begin while the previous kernel on the stream is finishing.
// The cache kernels call grid_dependency_wait() (griddepcontrol.wait) before
// touching global memory; the decode kernel reads only the context lengths
// and block tables before it (include/pkv.h states that contract), so results
// are the same as with plain stream ordering.  After a non-kernel operation
// (a copy, an event wait) the launch simply waits as usual.
#ifndef PKV_LAUNCH_H
#define PKV_LAUNCH_H

#include <cuda_runtime.h>

#include "../../include/pkv.h"

namespace pkv {

inline cudaError_t launch_pdl(const void *fn, dim3 grid, dim3 block, size_t smem, pkv_stream_t stream,
                              void **args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = reinterpret_cast<cudaStream_t>(stream);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelExC(&cfg, fn, args);
}

}  // namespace pkv

#endif  // PKV_LAUNCH_H
