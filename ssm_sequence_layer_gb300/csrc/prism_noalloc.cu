// prism_forward_noalloc: the tensor-core forward with its scratch memory in a fixed array
// compiled into the library, for callers that must not allocate device memory.
//
// Such callers include code running inside a device-memory allocator or pool hook (where a
// nested cudaMalloc would recurse or deadlock), real-time loops whose memory is reserved up
// front and must not grow, and hosts whose policy forbids allocation after start-up.  The
// regular entry points allocate through prism_plan; this one allocates nothing: it uses the
// array below for the segment maps, the segment start states, the per-chunk stash and the
// device status word, and otherwise runs the same kernels as prism_forward's tensor-core path.
#include <cstdio>
#include <mutex>

#include "prism_internal.h"

namespace {

// Scratch of every prism_forward_noalloc call on this device (held from module load to exit).
static __device__ __align__(256) unsigned char g_noalloc_scratch[PRISM_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
void *g_scratch_ptr[kMaxDevices] = {};   // device address of g_noalloc_scratch, per device
int g_sm_count[kMaxDevices] = {};

thread_local char g_noalloc_err[256] = "";

prism_status noalloc_fail(prism_status s, const char *msg)
{
    // reset the runtime's last-error state after a failed CUDA call, so that the error is not
    // reported again by the launch check of a later, unrelated call
    if (s == PRISM_ERR_CUDA) (void)cudaGetLastError();
    snprintf(g_noalloc_err, sizeof(g_noalloc_err), "prism_forward_noalloc: %s", msg);
    prism_set_error_message(g_noalloc_err);
    return s;
}

// once per device, with that device current: resolve the array's device address and set
// the segment kernel's shared-memory attribute
prism_status setup_device(int dev, void **scratch, int *sms)
{
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    if (g_scratch_ptr[dev]) {
        *scratch = g_scratch_ptr[dev];
        *sms = g_sm_count[dev];
        return PRISM_OK;
    }
    int major = 0, minor = 0, count = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return noalloc_fail(PRISM_ERR_CUDA, "cannot query the current device");
    if (major != 10 || minor != 3) return noalloc_fail(PRISM_ERR_ARCH, "the current device is not sm_103");
    void *ptr = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
    if (e != cudaSuccess || !ptr) return noalloc_fail(PRISM_ERR_CUDA, "cudaGetSymbolAddress of the scratch array failed");
    if (prism::tc_prepare() != cudaSuccess) return noalloc_fail(PRISM_ERR_CUDA, "kernel attribute setup failed");
    g_scratch_ptr[dev] = ptr;
    g_sm_count[dev] = count;
    *scratch = ptr;
    *sms = count;
    return PRISM_OK;
}

bool aligned16(const void *p) { return ((uintptr_t)p & 15) == 0; }
bool aligned4(const void *p) { return ((uintptr_t)p & 3) == 0; }

}  // namespace

extern "C" prism_status prism_forward_noalloc(int B, int H, int T, int dk, int dv, int L, const void *q, const void *k,
                                              const void *v, const float *beta, const float *alpha, const void *u,
                                              const float *gamma, const float *eta, const void *conv_w, void *out,
                                              struct CUstream_st *stream, int *device_status)
{
    if (B < 1 || H < 1 || T < 1 || L < 1) return noalloc_fail(PRISM_ERR_INVALID_ARG, "B, H, T and L must be >= 1");
    if ((long long)B * H > 65535) return noalloc_fail(PRISM_ERR_UNSUPPORTED, "B*H must be <= 65535");
    prism::Shape s;
    s.B = B; s.H = H; s.T = T; s.dk = dk; s.dv = dv; s.L = L; s.R = L - 1;
    s.NC = (T + prism::kChunk - 1) / prism::kChunk;
    s.BH = B * H;
    if (!prism::tc_supported(s, PRISM_BF16))
        return noalloc_fail(PRISM_ERR_UNSUPPORTED, "takes the tensor-core shapes only: dk = dv = 64, 1 <= L <= 4");
    if (!q || !k || !v || !beta || !alpha || !conv_w || !out || (s.R > 0 && (!u || !gamma || !eta)))
        return noalloc_fail(PRISM_ERR_INVALID_ARG, "a required tensor pointer is NULL");
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(conv_w) || !aligned16(out) ||
        (s.R > 0 && !aligned16(u)))
        return noalloc_fail(PRISM_ERR_MISALIGNED, "q, k, v, u, conv_w and out must be 16-byte aligned");
    if (!aligned4(beta) || !aligned4(alpha) || (s.R > 0 && (!aligned4(gamma) || !aligned4(eta))))
        return noalloc_fail(PRISM_ERR_MISALIGNED, "gate tensors must be 4-byte aligned");

    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return noalloc_fail(PRISM_ERR_CUDA, "no usable current CUDA device");
    void *scratch = nullptr;
    int sms = 0;
    prism_status st = setup_device(dev, &scratch, &sms);
    if (st != PRISM_OK) return st;

    // The automatic segment count, as prism_forward chooses it, when its scratch fits.  Else one
    // segment per sequence: a single segment starts from S = 0 and writes its outputs directly, so
    // it needs no per-chunk stash, only its map and start state (40 KiB per sequence).
    const size_t avail = (size_t)PRISM_NOALLOC_SCRATCH_BYTES - 256;
    int P = prism::tc_segments(s, sms, 0);
    bool stash = true;
    if (prism::tc_workspace_bytes(s, P) > avail) {
        P = 1;
        stash = false;
    }
    const size_t maps_bytes = (size_t)s.BH * (128 * 64 * 4 + 64 * 64 * 2) + 256;
    if (!stash && maps_bytes > avail)
        return noalloc_fail(PRISM_ERR_UNSUPPORTED,
                            "problem too large for the fixed scratch (one segment per sequence needs 40 KiB "
                            "per sequence; several need 24 KiB more per 64-token chunk; 64 MiB in total)");

    int *d_status = (int *)scratch;
    prism::TcWorkspace w;
    prism::tc_carve(s, P, (char *)scratch + 256, &w);
    if (!stash) {  // never read or written with one segment and no initial state
        w.stash_o = nullptr;
        w.stash_q = nullptr;
    }
    cudaStream_t cs = (cudaStream_t)stream;
    if (cudaMemsetAsync(d_status, 0, sizeof(int), cs) != cudaSuccess)
        return noalloc_fail(PRISM_ERR_CUDA, "clearing the status word failed");
    prism::ForwardArgs a{q, k, v, u, conv_w, beta, alpha, gamma, eta, out};
    prism::KernelTimer timer{};
    timer.on = false;
    timer.reset(cs);
    const cudaError_t e = prism::tc_forward(s, a, false, w, d_status, 0, timer);
    if (e != cudaSuccess) return noalloc_fail(PRISM_ERR_CUDA, cudaGetErrorString(e));
    if (!device_status) return PRISM_OK;

    int word = 0;
    if (cudaStreamSynchronize(cs) != cudaSuccess) return noalloc_fail(PRISM_ERR_CUDA, "stream synchronize failed");
    if (cudaMemcpy(&word, d_status, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
        return noalloc_fail(PRISM_ERR_CUDA, "reading the status word failed");
    *device_status = word;
    if (word == prism::kDevTimeout) return noalloc_fail(PRISM_ERR_TIMEOUT, "a bounded device wait expired");
    if (word != prism::kDevOk) return noalloc_fail(PRISM_ERR_DEVICE, "a device-side check failed");
    return PRISM_OK;
}
