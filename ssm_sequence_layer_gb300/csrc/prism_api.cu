// Host side of the C ABI declared in include/prism.h: argument validation, the
// plan (shape, device, workspace) and the launch sequence on the caller's stream.
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <new>

#include "prism_internal.h"
#include "prism_project.h"

namespace {

thread_local char g_err[512] = "no error";

prism_status fail(prism_status s, const char *fmt, ...)
{
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof(g_err), fmt, ap);
    va_end(ap);
    return s;
}

prism_status cuda_fail(cudaError_t e, const char *what)
{
    // reset the runtime's last-error state, so that a recoverable failure (an allocation that did
    // not fit) is not reported again by the error check after a later call's launches
    (void)cudaGetLastError();
    return fail(PRISM_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

bool aligned(const void *p, size_t a) { return ((uintptr_t)p % a) == 0; }

size_t io_size(prism_dtype io) { return io == PRISM_BF16 ? 2 : 4; }

prism_status check_sizes(int B, int H, int T, int dk, int dv, int L, prism_dtype io)
{
    if (B < 1 || H < 1 || T < 1)
        return fail(PRISM_ERR_INVALID_ARG, "B, H and T must be >= 1 (got B=%d H=%d T=%d)", B, H, T);
    if (L < 1) return fail(PRISM_ERR_INVALID_ARG, "L must be >= 1 (got %d)", L);
    if (io != PRISM_F32 && io != PRISM_BF16) return fail(PRISM_ERR_INVALID_ARG, "unknown io dtype %d", (int)io);
    if ((dk != 64 && dk != 128) || (dv != 64 && dv != 128))
        return fail(PRISM_ERR_UNSUPPORTED, "dk and dv must be 64 or 128 (got dk=%d dv=%d)", dk, dv);
    if (L > 16) return fail(PRISM_ERR_UNSUPPORTED, "L must be <= 16 (got %d)", L);
    const long long BH = (long long)B * H;
    if (BH > 65535) return fail(PRISM_ERR_UNSUPPORTED, "B*H must be <= 65535 (got %lld)", BH);
    if ((long long)T > (1LL << 30)) return fail(PRISM_ERR_UNSUPPORTED, "T too large (%d)", T);
    return PRISM_OK;
}

prism_status check_device(int *device, int *sms)
{
    cudaError_t e = cudaGetDevice(device);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    int major = 0, minor = 0;
    if ((e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, *device))) return cuda_fail(e, "attr");
    if ((e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, *device))) return cuda_fail(e, "attr");
    if ((e = cudaDeviceGetAttribute(sms, cudaDevAttrMultiProcessorCount, *device))) return cuda_fail(e, "attr");
    if (major != 10 || minor != 3)
        return fail(PRISM_ERR_ARCH, "device %d is sm_%d%d; this library is built for sm_103 only", *device, major,
                    minor);
    return PRISM_OK;
}

prism_status check_forward_args(const prism_plan_s *p, const void *q, const void *k, const void *v,
                                const float *beta, const float *alpha, const void *u, const float *gamma,
                                const float *eta, const void *conv_w, int L, const void *out)
{
    if (!p) return fail(PRISM_ERR_INVALID_ARG, "plan is NULL");
    if (L != p->shape.L) return fail(PRISM_ERR_INVALID_ARG, "L=%d differs from the plan's L=%d", L, p->shape.L);
    if (!q || !k || !v || !beta || !alpha || !conv_w || !out)
        return fail(PRISM_ERR_INVALID_ARG, "q, k, v, beta, alpha, conv_w and out must not be NULL");
    if (p->shape.R > 0 && (!u || !gamma || !eta))
        return fail(PRISM_ERR_INVALID_ARG, "u, gamma and eta must not be NULL when L > 1");
    const void *io_ptrs[] = {q, k, v, conv_w, out, p->shape.R > 0 ? u : nullptr};
    const char *io_names[] = {"q", "k", "v", "conv_w", "out", "u"};
    for (int i = 0; i < 6; ++i)
        if (io_ptrs[i] && !aligned(io_ptrs[i], 16))
            return fail(PRISM_ERR_MISALIGNED, "%s is not 16-byte aligned", io_names[i]);
    const void *f_ptrs[] = {beta, alpha, p->shape.R > 0 ? gamma : nullptr, p->shape.R > 0 ? eta : nullptr};
    const char *f_names[] = {"beta", "alpha", "gamma", "eta"};
    for (int i = 0; i < 4; ++i)
        if (f_ptrs[i] && !aligned(f_ptrs[i], 4))
            return fail(PRISM_ERR_MISALIGNED, "%s is not 4-byte aligned", f_names[i]);
    return PRISM_OK;
}

// Byte sizes of the call's tensors, in the order q, k, v, beta, alpha, u, gamma, eta, conv_w, out.
void tensor_bytes(const prism_plan_s *p, size_t nb[10])
{
    const prism::Shape &s = p->shape;
    const size_t e = io_size(p->io), th = (size_t)s.BH * s.T;
    nb[0] = th * s.dk * e;
    nb[1] = th * s.dk * e;
    nb[2] = th * s.dv * e;
    nb[3] = th * 4;
    nb[4] = th * 4;
    nb[5] = th * s.R * s.dk * e;
    nb[6] = th * s.R * 4;
    nb[7] = th * s.R * 4;
    nb[8] = (size_t)s.H * 4 * s.dv * e;
    nb[9] = th * s.dv * io_size(p->out_dtype);
}

// 1 = portable fp32 kernels, 2 = tensor-core path (the segment kernels for dk = dv = 64 and
// L <= 4, the chunk-map kernels for dk = dv = 128 and L <= 16)
bool tensor_core_shape(const prism_plan_s *p)
{
    return prism::tc_supported(p->shape, p->io) || prism::map_supported(p->shape, p->io);
}

int resolve_path(const prism_plan_s *p)
{
    if (p->opt_path == 1) return 1;
    if (p->opt_path == 2) return 2;
    return tensor_core_shape(p) ? 2 : 1;
}

void free_workspaces(prism_plan_s *p)
{
    if (p->ws_simt) cudaFree(p->ws_simt);
    if (p->ws_tc) cudaFree(p->ws_tc);
    if (p->ws_map) cudaFree(p->ws_map);
    if (p->d_status) cudaFree(p->d_status);
    if (p->ws_bwd) cudaFree(p->ws_bwd);
    p->ws_bwd = nullptr;
    p->ws_bwd_bytes = 0;
    p->ws_simt = p->ws_tc = p->ws_map = nullptr;
    p->d_status = nullptr;
}

prism_status ensure_workspace(prism_plan_s *p, int path)
{
    cudaError_t e;
    if (path == 1) {
        if (p->ws_simt) return PRISM_OK;
        const size_t bytes = prism::simt_workspace_bytes(p->shape);
        if ((e = cudaMalloc(&p->ws_simt, bytes)) != cudaSuccess) {
            p->ws_simt = nullptr;
            return cuda_fail(e, "workspace allocation (portable path)");
        }
        p->ws_simt_bytes = bytes;
        prism::simt_carve(p->shape, p->ws_simt, &p->simt);
        return PRISM_OK;
    }
    if (!prism::tc_supported(p->shape, p->io)) {  // chunk-map kernels
        if (p->ws_map) return PRISM_OK;
        const size_t bytes = prism::map_workspace_bytes(p->shape);
        if ((e = cudaMalloc(&p->ws_map, bytes)) != cudaSuccess) {
            p->ws_map = nullptr;
            return cuda_fail(e, "workspace allocation (chunk-map kernels)");
        }
        p->ws_map_bytes = bytes;
        prism::map_carve(p->shape, p->ws_map, &p->mapw);
        return PRISM_OK;
    }
    const int P = prism::tc_segments(p->shape, p->sm_count, p->opt_segments);
    if (p->ws_tc && p->tcw.P == P) return PRISM_OK;
    if (p->ws_tc) {
        cudaFree(p->ws_tc);
        p->ws_tc = nullptr;
        p->ws_tc_bytes = 0;
    }
    const size_t bytes = prism::tc_workspace_bytes(p->shape, P);
    if ((e = cudaMalloc(&p->ws_tc, bytes)) != cudaSuccess) {
        p->ws_tc = nullptr;
        return cuda_fail(e, "workspace allocation (tensor-core path)");
    }
    p->ws_tc_bytes = bytes;
    prism::tc_carve(p->shape, P, p->ws_tc, &p->tcw);
    return PRISM_OK;
}

prism_status check_plan_device(const prism_plan_s *p)
{
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev != p->device)
        return fail(PRISM_ERR_INVALID_ARG, "current device %d differs from the plan's device %d", dev, p->device);
    return PRISM_OK;
}

// The launch sequence of a validated forward on the plan's path.
prism_status run_forward(prism_plan_s *p, const prism::ForwardArgs &a, struct CUstream_st *stream)
{
    prism_status st = check_plan_device(p);
    if (st != PRISM_OK) return st;
    const int path = resolve_path(p);
    if (path == 2 && !tensor_core_shape(p))
        return fail(PRISM_ERR_UNSUPPORTED,
                    "the tensor-core path takes bf16 io with dk = dv = 64 and L <= 4, or dk = dv = 128 and L <= 16");
    if ((st = ensure_workspace(p, path)) != PRISM_OK) return st;
    p->timer.on = p->opt_timing != 0;
    p->timer.reset((cudaStream_t)stream);
    cudaError_t e;
    if (path == 2 && prism::tc_supported(p->shape, p->io))
        e = prism::tc_forward(p->shape, a, p->out_dtype == PRISM_F32, p->tcw, p->d_status, p->opt_wait_ns, p->timer);
    else if (path == 2)
        e = prism::map_forward(p->shape, a, p->out_dtype == PRISM_F32, p->mapw, p->sm_count, p->d_status,
                               p->opt_wait_ns, p->timer);
    else
        e = prism::simt_forward(p->shape, p->io, p->out_dtype, a, p->simt, p->d_status, p->timer);
    if (e != cudaSuccess) return cuda_fail(e, "kernel launch");
    return PRISM_OK;
}

}  // namespace

void prism_set_error_message(const char *msg) { snprintf(g_err, sizeof(g_err), "%s", msg); }

extern "C" {

const char *prism_version(void) { return "0.1.0"; }

const char *prism_last_error_message(void) { return g_err; }

const char *prism_status_string(prism_status s)
{
    switch (s) {
    case PRISM_OK: return "PRISM_OK";
    case PRISM_ERR_INVALID_ARG: return "PRISM_ERR_INVALID_ARG: invalid argument";
    case PRISM_ERR_UNSUPPORTED: return "PRISM_ERR_UNSUPPORTED: unsupported problem size";
    case PRISM_ERR_MISALIGNED: return "PRISM_ERR_MISALIGNED: misaligned tensor";
    case PRISM_ERR_ARCH: return "PRISM_ERR_ARCH: device is not sm_103";
    case PRISM_ERR_CUDA: return "PRISM_ERR_CUDA: CUDA runtime error";
    case PRISM_ERR_TIMEOUT: return "PRISM_ERR_TIMEOUT: a bounded device wait expired";
    case PRISM_ERR_DEVICE: return "PRISM_ERR_DEVICE: a device-side check failed";
    }
    return "unknown prism_status";
}

prism_status prism_plan(int B, int H, int T, int dk, int dv, int L, prism_dtype io, prism_plan_t *out_plan)
{
    if (!out_plan) return fail(PRISM_ERR_INVALID_ARG, "out_plan is NULL");
    *out_plan = nullptr;
    prism_status st = check_sizes(B, H, T, dk, dv, L, io);
    if (st != PRISM_OK) return st;
    int device = 0, sms = 0;
    if ((st = check_device(&device, &sms)) != PRISM_OK) return st;

    prism_plan_s *p = new (std::nothrow) prism_plan_s();
    if (!p) return fail(PRISM_ERR_INVALID_ARG, "out of host memory");
    prism::Shape &s = p->shape;
    s.B = B; s.H = H; s.T = T; s.dk = dk; s.dv = dv; s.L = L; s.R = L - 1;
    s.NC = (T + prism::kChunk - 1) / prism::kChunk;
    s.BH = B * H;
    p->io = io;
    p->out_dtype = io;
    p->device = device;
    p->sm_count = sms;

    cudaError_t e = prism::simt_prepare(s, io);
    if (e == cudaSuccess && prism::tc_supported(s, io)) e = prism::tc_prepare();
    if (e == cudaSuccess && prism::map_supported(s, io)) e = prism::map_prepare();
    if (e == cudaSuccess && io == PRISM_BF16) e = prism::project_prepare();
    if (e == cudaSuccess) e = prism::backward_prepare();
    if (e == cudaSuccess) e = prism::backward_tc_prepare();
    if (e != cudaSuccess) {
        delete p;
        return cuda_fail(e, "kernel attribute setup");
    }
    if ((e = cudaMalloc(&p->d_status, 256)) != cudaSuccess) {
        delete p;
        return cuda_fail(e, "status word allocation");
    }
    if ((e = cudaMemset(p->d_status, 0, sizeof(int))) != cudaSuccess) {
        cudaFree(p->d_status);
        delete p;
        return cuda_fail(e, "status word init");
    }
    // workspace of the path the plan uses by default
    st = ensure_workspace(p, resolve_path(p));
    if (st != PRISM_OK) {
        cudaFree(p->d_status);
        delete p;
        return st;
    }
    for (int i = 0; i < 2 * prism::kMaxTimedKernels; ++i) {
        if ((e = cudaEventCreate(&p->timer.ev[i])) != cudaSuccess) {
            for (int j = 0; j < i; ++j) cudaEventDestroy(p->timer.ev[j]);
            free_workspaces(p);
            delete p;
            return cuda_fail(e, "event creation");
        }
    }
    *out_plan = p;
    return PRISM_OK;
}

prism_status prism_plan_set_option(prism_plan_t p, prism_option opt, long long value)
{
    if (!p) return fail(PRISM_ERR_INVALID_ARG, "plan is NULL");
    switch (opt) {
    case PRISM_OPT_SEGMENTS:
        if (value < 0) return fail(PRISM_ERR_INVALID_ARG, "segments must be >= 0");
        p->opt_segments = value;
        return PRISM_OK;
    case PRISM_OPT_PATH:
        if (value < 0 || value > 2) return fail(PRISM_ERR_INVALID_ARG, "path must be 0, 1 or 2");
        p->opt_path = value;
        return PRISM_OK;
    case PRISM_OPT_WAIT_NS:
        if (value < 0) return fail(PRISM_ERR_INVALID_ARG, "wait bound must be >= 0");
        p->opt_wait_ns = value;
        return PRISM_OK;
    case PRISM_OPT_OUT_DTYPE:
        if (value != PRISM_F32 && value != PRISM_BF16) return fail(PRISM_ERR_INVALID_ARG, "unknown out dtype");
        p->out_dtype = (prism_dtype)value;
        return PRISM_OK;
    case PRISM_OPT_TIMING:
        if (value != 0 && value != 1) return fail(PRISM_ERR_INVALID_ARG, "timing must be 0 or 1");
        p->opt_timing = value;
        return PRISM_OK;
    }
    return fail(PRISM_ERR_INVALID_ARG, "unknown option %d", (int)opt);
}

prism_status prism_forward(prism_plan_t p, const void *q, const void *k, const void *v, const float *beta,
                           const float *alpha, const void *u, const float *gamma, const float *eta,
                           const void *conv_w, int L, void *out, struct CUstream_st *stream)
{
    prism_status st = check_forward_args(p, q, k, v, beta, alpha, u, gamma, eta, conv_w, L, out);
    if (st != PRISM_OK) return st;
    return run_forward(p, prism::ForwardArgs{q, k, v, u, conv_w, beta, alpha, gamma, eta, out}, stream);
}

prism_status prism_forward_state(prism_plan_t p, const void *q, const void *k, const void *v, const float *beta,
                                 const float *alpha, const void *u, const float *gamma, const float *eta,
                                 const void *conv_w, int L, const void *v_hist, const float *S_init, void *out,
                                 float *S_final, void *v_hist_out, struct CUstream_st *stream)
{
    prism_status st = check_forward_args(p, q, k, v, beta, alpha, u, gamma, eta, conv_w, L, out);
    if (st != PRISM_OK) return st;
    const void *sp[] = {v_hist, S_init, S_final, v_hist_out};
    const char *sn[] = {"v_hist", "S_init", "S_final", "v_hist_out"};
    for (int i = 0; i < 4; ++i)
        if (sp[i] && !aligned(sp[i], 16)) return fail(PRISM_ERR_MISALIGNED, "%s is not 16-byte aligned", sn[i]);
    prism::ForwardArgs a{q, k, v, u, conv_w, beta, alpha, gamma, eta, out};
    a.v_hist = v_hist;
    a.S_init = S_init;
    a.S_final = S_final;
    a.v_hist_out = v_hist_out;
    return run_forward(p, a, stream);
}

prism_status prism_forward_nonlinear(prism_plan_t p, const void *q, const void *k, const void *v,
                                     const float *beta, const float *alpha, const void *u, const float *gamma,
                                     const void *p_gain, const void *conv_w, int L, const void *v_hist,
                                     const float *S_init, void *out, float *S_final, void *v_hist_out,
                                     struct CUstream_st *stream)
{
    if (!p) return fail(PRISM_ERR_INVALID_ARG, "plan is NULL");
    const bool lvl = p->shape.R > 0;
    if (lvl && !p_gain) return fail(PRISM_ERR_INVALID_ARG, "p_gain must not be NULL when L > 1");
    // eta is not part of this variant: validate the rest as prism_forward does (gamma stands in
    // for eta's null check)
    prism_status st = check_forward_args(p, q, k, v, beta, alpha, u, gamma, lvl ? gamma : nullptr, conv_w, L, out);
    if (st != PRISM_OK) return st;
    const void *sp[] = {v_hist, S_init, S_final, v_hist_out, lvl ? p_gain : nullptr};
    const char *sn[] = {"v_hist", "S_init", "S_final", "v_hist_out", "p_gain"};
    for (int i = 0; i < 5; ++i)
        if (sp[i] && !aligned(sp[i], 16)) return fail(PRISM_ERR_MISALIGNED, "%s is not 16-byte aligned", sn[i]);
    prism::ForwardArgs a{q, k, v, u, conv_w, beta, alpha, gamma, nullptr, out};
    a.v_hist = v_hist;
    a.S_init = S_init;
    a.S_final = S_final;
    a.v_hist_out = v_hist_out;
    a.p_gain = lvl ? p_gain : nullptr;
    return run_forward(p, a, stream);
}

prism_status prism_project(prism_plan_t p, int D, const void *X, const void *conv_x, const void *W, void *u,
                           void *pg, float *gamma, struct CUstream_st *stream)
{
    if (!p) return fail(PRISM_ERR_INVALID_ARG, "plan is NULL");
    if (p->io != PRISM_BF16) return fail(PRISM_ERR_UNSUPPORTED, "prism_project takes a bf16 plan");
    if (p->shape.R < 1) return fail(PRISM_ERR_INVALID_ARG, "prism_project needs L >= 2 (at least one level)");
    if (D < 64 || D % 64 != 0 || D > 65536)
        return fail(PRISM_ERR_UNSUPPORTED, "D must be a multiple of 64 in [64, 65536] (got %d)", D);
    if (!X || !conv_x || !W || !u || !pg || !gamma)
        return fail(PRISM_ERR_INVALID_ARG, "X, conv_x, W, u, p and gamma must not be NULL");
    const void *ap[] = {X, conv_x, W, u, pg};
    const char *an[] = {"X", "conv_x", "W", "u", "p"};
    for (int i = 0; i < 5; ++i)
        if (!aligned(ap[i], 16)) return fail(PRISM_ERR_MISALIGNED, "%s is not 16-byte aligned", an[i]);
    if (!aligned(gamma, 4)) return fail(PRISM_ERR_MISALIGNED, "gamma is not 4-byte aligned");
    prism_status st = check_plan_device(p);
    if (st != PRISM_OK) return st;
    // the anchor a = ShortConv(X) goes through the plan's staging buffer (B T D bf16)
    const size_t abytes = (size_t)p->shape.B * p->shape.T * D * 2;
    if (p->stage_bytes < abytes) {
        if (p->stage) cudaFree(p->stage);
        p->stage = nullptr;
        p->stage_bytes = 0;
        cudaError_t e = cudaMalloc(&p->stage, abytes);
        if (e != cudaSuccess) return cuda_fail(e, "anchor buffer allocation");
        p->stage_bytes = abytes;
    }
    prism::ProjectArgs a{X, conv_x, W, u, pg, gamma, p->stage};
    p->timer.on = p->opt_timing != 0;
    p->timer.reset((cudaStream_t)stream);
    const cudaError_t e = prism::project_forward(p->shape, D, a, p->d_status, p->opt_wait_ns, p->timer);
    if (e != cudaSuccess) return cuda_fail(e, "kernel launch");
    return PRISM_OK;
}

prism_status prism_decode_step(prism_plan_t p, const void *q, const void *k, const void *v, const float *beta,
                               const float *alpha, const void *u, const float *gamma, const float *eta,
                               const void *conv_w, int L, void *v_hist, float *S, void *out,
                               struct CUstream_st *stream)
{
    if (!p) return fail(PRISM_ERR_INVALID_ARG, "plan is NULL");
    if (L != p->shape.L) return fail(PRISM_ERR_INVALID_ARG, "L=%d differs from the plan's L=%d", L, p->shape.L);
    if (!q || !k || !v || !beta || !alpha || !conv_w || !v_hist || !S || !out)
        return fail(PRISM_ERR_INVALID_ARG, "q, k, v, beta, alpha, conv_w, v_hist, S and out must not be NULL");
    const bool lvl = p->shape.R > 0;
    if (lvl && (!u || !gamma || !eta))
        return fail(PRISM_ERR_INVALID_ARG, "u, gamma and eta must not be NULL when L > 1");
    const void *ap[] = {q, k, v, conv_w, v_hist, S, out, lvl ? u : nullptr};
    const char *an[] = {"q", "k", "v", "conv_w", "v_hist", "S", "out", "u"};
    for (int i = 0; i < 8; ++i)
        if (ap[i] && !aligned(ap[i], 16)) return fail(PRISM_ERR_MISALIGNED, "%s is not 16-byte aligned", an[i]);
    const void *fp[] = {beta, alpha, lvl ? gamma : nullptr, lvl ? eta : nullptr};
    const char *fn[] = {"beta", "alpha", "gamma", "eta"};
    for (int i = 0; i < 4; ++i)
        if (fp[i] && !aligned(fp[i], 4)) return fail(PRISM_ERR_MISALIGNED, "%s is not 4-byte aligned", fn[i]);
    prism_status st = check_plan_device(p);
    if (st != PRISM_OK) return st;
    prism::DecodeArgs a{q, k, v, u, conv_w, beta, alpha, gamma, eta, v_hist, S, out};
    p->timer.on = p->opt_timing != 0;
    p->timer.reset((cudaStream_t)stream);
    const cudaError_t e =
        prism::decode_step(p->shape, p->io, p->out_dtype, a, p->sm_count, p->d_status, p->opt_wait_ns, p->timer);
    if (e != cudaSuccess) return cuda_fail(e, "kernel launch");
    return PRISM_OK;
}

// Both chains' backward.  The linear chain passes eta and deta; the non-linear one p_gain and
// dp_gain (eta and deta null).
static prism_status run_backward(prism_plan_t p, const void *q, const void *k, const void *v, const float *beta,
                                 const float *alpha, const void *u, const float *gamma, const float *eta,
                                 const void *p_gain, const void *conv_w, int L, const void *v_hist,
                                 const float *S_init, const float *dout, const float *dS_final, float *dq, float *dk,
                                 float *dv, float *dbeta, float *dalpha, float *du, float *dgamma, float *deta,
                                 float *dp_gain, float *dconv_w, float *dv_hist, float *dS_init,
                                 struct CUstream_st *stream)
{
    if (!p) return fail(PRISM_ERR_INVALID_ARG, "plan is NULL");
    const bool lvl = p->shape.R > 0, nonlinear = p_gain != nullptr || dp_gain != nullptr;
    if (nonlinear && lvl && (!p_gain || !dp_gain))
        return fail(PRISM_ERR_INVALID_ARG, "p_gain and dp_gain must not be NULL when L > 1");
    // the forward's checks stand for the inputs; dout takes the place of out (gamma stands in
    // for eta's null check in the non-linear chain, which has no eta)
    prism_status st = check_forward_args(p, q, k, v, beta, alpha, u, gamma, nonlinear && lvl ? gamma : eta, conv_w,
                                         L, dout);
    if (st != PRISM_OK) return st;
    if (!dq || !dk || !dv || !dbeta || !dalpha || !dconv_w)
        return fail(PRISM_ERR_INVALID_ARG, "dq, dk, dv, dbeta, dalpha and dconv_w must not be NULL");
    if (lvl && (!du || !dgamma || (!nonlinear && !deta)))
        return fail(PRISM_ERR_INVALID_ARG, "du, dgamma and deta must not be NULL when L > 1");
    const void *ap[] = {v_hist, S_init, dS_final, dv_hist, dS_init, dout, dq, dk, dv, lvl ? du : nullptr,
                        lvl ? p_gain : nullptr, lvl ? dp_gain : nullptr};
    const char *an[] = {"v_hist", "S_init", "dS_final", "dv_hist", "dS_init", "dout", "dq", "dk", "dv", "du",
                        "p_gain", "dp_gain"};
    for (int i = 0; i < 12; ++i)
        if (ap[i] && !aligned(ap[i], 16)) return fail(PRISM_ERR_MISALIGNED, "%s is not 16-byte aligned", an[i]);
    const void *fp[] = {dbeta, dalpha, dconv_w, lvl ? dgamma : nullptr, lvl && !nonlinear ? deta : nullptr};
    const char *fn[] = {"dbeta", "dalpha", "dconv_w", "dgamma", "deta"};
    for (int i = 0; i < 5; ++i)
        if (fp[i] && !aligned(fp[i], 4)) return fail(PRISM_ERR_MISALIGNED, "%s is not 4-byte aligned", fn[i]);
    if ((st = check_plan_device(p)) != PRISM_OK) return st;
    // the chunked tensor-core form wherever it applies, unless the portable kernels are asked for
    const bool chunked = p->opt_path != 1 && prism::backward_tc_supported(p->shape, p->io);
    const size_t bytes =
        chunked ? prism::backward_tc_workspace_bytes(p->shape) : prism::backward_workspace_bytes(p->shape);
    if (p->ws_bwd && p->ws_bwd_bytes < bytes) {
        cudaError_t e = cudaFree(p->ws_bwd);
        p->ws_bwd = nullptr;
        p->ws_bwd_bytes = 0;
        if (e != cudaSuccess) return cuda_fail(e, "backward workspace release");
    }
    if (!p->ws_bwd) {
        cudaError_t e = cudaMalloc(&p->ws_bwd, bytes);
        if (e != cudaSuccess) {
            p->ws_bwd = nullptr;
            return cuda_fail(e, "backward workspace allocation");
        }
        p->ws_bwd_bytes = bytes;
    }
    prism::BackwardArgs a{q, k, v, lvl ? u : nullptr, conv_w, v_hist, beta, alpha, lvl ? gamma : nullptr,
                          lvl && !nonlinear ? eta : nullptr, S_init, dout, dS_final, dq, dk, dv, dbeta, dalpha,
                          lvl ? du : nullptr, lvl ? dgamma : nullptr, lvl && !nonlinear ? deta : nullptr, dconv_w,
                          dv_hist, dS_init};
    a.p_gain = lvl ? p_gain : nullptr;
    a.dp_gain = lvl ? dp_gain : nullptr;
    p->timer.on = p->opt_timing != 0;
    p->timer.reset((cudaStream_t)stream);
    const cudaError_t e = chunked ? prism::backward_tc(p->shape, a, p->ws_bwd, p->d_status, p->opt_wait_ns, p->timer)
                                  : prism::backward(p->shape, p->io, a, p->ws_bwd, p->timer);
    if (e != cudaSuccess) return cuda_fail(e, "kernel launch");
    return PRISM_OK;
}

prism_status prism_backward(prism_plan_t p, const void *q, const void *k, const void *v, const float *beta,
                            const float *alpha, const void *u, const float *gamma, const float *eta,
                            const void *conv_w, int L, const void *v_hist, const float *S_init, const float *dout,
                            const float *dS_final, float *dq, float *dk, float *dv, float *dbeta, float *dalpha,
                            float *du, float *dgamma, float *deta, float *dconv_w, float *dv_hist, float *dS_init,
                            struct CUstream_st *stream)
{
    return run_backward(p, q, k, v, beta, alpha, u, gamma, eta, nullptr, conv_w, L, v_hist, S_init, dout, dS_final,
                        dq, dk, dv, dbeta, dalpha, du, dgamma, deta, nullptr, dconv_w, dv_hist, dS_init, stream);
}

prism_status prism_backward_nonlinear(prism_plan_t p, const void *q, const void *k, const void *v,
                                      const float *beta, const float *alpha, const void *u, const float *gamma,
                                      const void *p_gain, const void *conv_w, int L, const void *v_hist,
                                      const float *S_init, const float *dout, const float *dS_final, float *dq,
                                      float *dk, float *dv, float *dbeta, float *dalpha, float *du, float *dgamma,
                                      float *dp_gain, float *dconv_w, float *dv_hist, float *dS_init,
                                      struct CUstream_st *stream)
{
    if (p && p->shape.R > 0 && (!p_gain || !dp_gain))
        return fail(PRISM_ERR_INVALID_ARG, "p_gain and dp_gain must not be NULL when L > 1");
    return run_backward(p, q, k, v, beta, alpha, u, gamma, nullptr, p_gain, conv_w, L, v_hist, S_init, dout,
                        dS_final, dq, dk, dv, dbeta, dalpha, du, dgamma, nullptr, dp_gain, dconv_w, dv_hist, dS_init,
                        stream);
}

prism_status prism_forward_host(prism_plan_t p, const void *q, const void *k, const void *v, const float *beta,
                                const float *alpha, const void *u, const float *gamma, const float *eta,
                                const void *conv_w, int L, void *out, struct CUstream_st *stream)
{
    if (!p) return fail(PRISM_ERR_INVALID_ARG, "plan is NULL");
    size_t nb[10];
    tensor_bytes(p, nb);
    size_t off[10], total = 0;
    for (int i = 0; i < 10; ++i) {
        off[i] = total;
        total += (nb[i] + 255) & ~(size_t)255;
    }
    if (p->stage_bytes < total) {
        if (p->stage) cudaFree(p->stage);
        p->stage = nullptr;
        p->stage_bytes = 0;
        cudaError_t e = cudaMalloc(&p->stage, total);
        if (e != cudaSuccess) return cuda_fail(e, "staging allocation");
        p->stage_bytes = total;
    }
    const void *src[9] = {q, k, v, beta, alpha, u, gamma, eta, conv_w};
    void *dst[10];
    for (int i = 0; i < 10; ++i) dst[i] = (char *)p->stage + off[i];
    // validate the host pointers like device ones before copying anything
    prism_status st = check_forward_args(p, q, k, v, beta, alpha, u, gamma, eta, conv_w, L, out);
    if (st != PRISM_OK) return st;
    cudaStream_t s = (cudaStream_t)stream;
    for (int i = 0; i < 9; ++i) {
        if (nb[i] == 0 || !src[i]) continue;
        cudaError_t e = cudaMemcpyAsync(dst[i], src[i], nb[i], cudaMemcpyHostToDevice, s);
        if (e != cudaSuccess) return cuda_fail(e, "host-to-device copy");
    }
    const bool lvl = p->shape.R > 0;
    st = prism_forward(p, dst[0], dst[1], dst[2], (const float *)dst[3], (const float *)dst[4],
                       lvl ? dst[5] : nullptr, lvl ? (const float *)dst[6] : nullptr,
                       lvl ? (const float *)dst[7] : nullptr, dst[8], L, dst[9], stream);
    if (st != PRISM_OK) return st;
    cudaError_t e = cudaMemcpyAsync(out, dst[9], nb[9], cudaMemcpyDeviceToHost, s);
    if (e != cudaSuccess) return cuda_fail(e, "device-to-host copy");
    if ((e = cudaStreamSynchronize(s)) != cudaSuccess) return cuda_fail(e, "stream synchronize");
    return PRISM_OK;
}

prism_status prism_plan_destroy(prism_plan_t p)
{
    if (!p) return PRISM_OK;
    for (int i = 0; i < 2 * prism::kMaxTimedKernels; ++i)
        if (p->timer.ev[i]) cudaEventDestroy(p->timer.ev[i]);
    free_workspaces(p);
    cudaError_t e2 = p->stage ? cudaFree(p->stage) : cudaSuccess;
    delete p;
    if (e2 != cudaSuccess) return cuda_fail(e2, "staging free");
    return PRISM_OK;
}

size_t prism_workspace_bytes(prism_plan_t p)
{
    return p ? p->ws_simt_bytes + p->ws_tc_bytes + p->ws_map_bytes + p->ws_bwd_bytes : 0;
}

int prism_plan_kernel_times(prism_plan_t p, prism_kernel_time *out, int max)
{
    if (!p || max < 0 || (max > 0 && !out)) {
        fail(PRISM_ERR_INVALID_ARG, "bad arguments to prism_plan_kernel_times");
        return -1;
    }
    const int n = p->timer.n;
    for (int i = 0; i < n && i < max && i < prism::kMaxTimedKernels; ++i) {
        out[i].name = p->timer.names[i];
        out[i].ms = -1.f;
        if (p->timer.on) {
            float ms = 0.f;
            if (cudaEventElapsedTime(&ms, p->timer.ev[2 * i], p->timer.ev[2 * i + 1]) == cudaSuccess) out[i].ms = ms;
        }
    }
    return n;
}

prism_status prism_plan_last_device_status(prism_plan_t p)
{
    if (!p) return fail(PRISM_ERR_INVALID_ARG, "plan is NULL");
    int word = 0;
    cudaError_t e = cudaMemcpy(&word, p->d_status, sizeof(int), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(e, "status read");
    if (word == prism::kDevOk) return PRISM_OK;
    if ((e = cudaMemset(p->d_status, 0, sizeof(int))) != cudaSuccess) return cuda_fail(e, "status clear");
    if (word == prism::kDevTimeout) return fail(PRISM_ERR_TIMEOUT, "a bounded device wait expired");
    return fail(PRISM_ERR_DEVICE, "device-side check failed (code %d)", word);
}

}  // extern "C"
