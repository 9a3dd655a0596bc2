// k5_adl.cu -- adaptive draft length on the device ("DiffuSpec: Unlocking
// Diffusion Language Models for Speculative Decoding", section 4.3): one
// thread per sequence updates its window from the step's generated (EOS-aware)
// and accepted lengths and writes the next draft length, so a decode loop can
// keep the controller on the stream next to the search and the verification.
#include "sdv_plan.h"

namespace sdv {
namespace {

__global__ void __launch_bounds__(256) adl_kernel(const AdlArgs a) {
    // Launched as a programmatic dependent of the kernel before it on the
    // stream (the draw, in a decode step): wait for that grid and its memory
    // before reading anything.  Then let the next kernel (the next step's
    // pruning pass, which waits for this grid in turn) become resident.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int b = blockIdx.x * blockDim.x + threadIdx.x;
    if (b >= a.B) return;
    const int32_t k = a.k[b];
    if (k < a.kmin || k > a.kmax) {          // left as it is, reported
        if (a.status) atomicOr(reinterpret_cast<unsigned*>(a.status), kStatusBadLength);
        return;
    }
    int32_t* st = a.state + static_cast<int64_t>(b) * adl_state_words(a.W);
    a.k[b] = adl_update(st, a.W, a.kmin, a.kmax, a.up, a.down, k, a.gen_len[b], a.acc_len[b]);
}

}  // namespace

cudaError_t launch_adl(const AdlArgs& a, cudaStream_t s) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>((a.B + 255) / 256));
    cfg.blockDim = dim3(256);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, adl_kernel, a);
}

}  // namespace sdv
