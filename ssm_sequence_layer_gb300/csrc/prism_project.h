// Internal declarations of the input-projection kernel (prism_project.cu).
#pragma once

#include "prism_internal.h"

namespace prism {

// Device pointers of one projection call (layouts as in prism.h, prism_project).
struct ProjectArgs {
    const void *X;     // [B,T,D] bf16
    const void *conv;  // [4,D] bf16
    const void *W;     // [N,D] bf16, N = H R (dk + dv + 1)
    void *u, *p;       // [B,H,T,R,dk], [B,H,T,R,dv] bf16
    float *gamma;      // [B,H,T,R]
    void *anchor;      // [B,T,D] bf16 scratch: the convolved input
};

cudaError_t project_prepare();
cudaError_t project_forward(const Shape &s, int D, const ProjectArgs &a, int *d_status, long long wait_ns,
                            KernelTimer &tm);

}  // namespace prism
