// Internal declarations shared by the host library and the kernel files.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/prism.h"

namespace prism {

constexpr int kChunk = 64;  // tokens per chunk of the WY/UT evaluation

// Device status word values (written by kernels, read by prism_plan_last_device_status).
enum DeviceStatus : int {
    kDevOk = 0,
    kDevBounds = 1,   // an internal index check failed
    kDevTimeout = 2,  // a bounded wait expired
};

// Pointers of one forward call (device memory, layouts as in prism.h).  v_hist .. v_hist_out
// carry a sequence across calls and may be null: v_hist [BH][3][dv] (v_{-3}, v_{-2}, v_{-1}, io
// dtype), S_init / S_final [BH][dv][dk] fp32, v_hist_out [BH][3][dv] (the last three tokens of
// [v_hist; v]).  p_gain [BH][T][R][dv] (io dtype), when set, selects the non-linear residual
// variant (eta is then not read).
struct ForwardArgs {
    const void *q, *k, *v, *u, *conv_w;
    const float *beta, *alpha, *gamma, *eta;
    void *out;
    const void *v_hist = nullptr;
    const float *S_init = nullptr;
    float *S_final = nullptr;
    void *v_hist_out = nullptr;
    const void *p_gain = nullptr;
};

// Problem shape shared by all kernels.
struct Shape {
    int B, H, T, dk, dv, L, R, NC, BH;
};

// Workspace of the portable fp32 path: one buffer per intermediate.
struct SimtWorkspace {
    float *X;    // [BH][T][R][dv]   injection factors x_{t,l}
    float *lam;  // [BH][T]          chunk-local cumulative log decay
    float *Tm;   // [BH][NC][C][C]   (I + A)^{-1} per chunk
    float *W;    // [BH][NC*C][dk]   W = T diag(beta Gamma) K
    float *Up;   // [BH][NC*C][dv]   U' = T (diag(beta) V - M X)
    float *S0;   // [BH][NC][dv][dk] state entering each chunk
    float *Vt;   // [BH][NC*C][dv]   V~ = U' - W S0^T
};

// Records CUDA events around each kernel launch of one forward (when enabled) and
// counts the launches.  Events are recorded on the launch stream.
constexpr int kMaxTimedKernels = 16;
struct KernelTimer {
    cudaEvent_t ev[2 * kMaxTimedKernels];
    const char *names[kMaxTimedKernels];
    int n;
    bool on;
    cudaStream_t stream;
    void reset(cudaStream_t s) { n = 0; stream = s; }
    void begin(const char *name)
    {
        if (n < kMaxTimedKernels) {
            names[n] = name;
            if (on) cudaEventRecord(ev[2 * n], stream);
        }
    }
    void end()
    {
        if (on && n < kMaxTimedKernels) cudaEventRecord(ev[2 * n + 1], stream);
        ++n;
    }
};

// Workspace of the tensor-core path.
struct TcWorkspace {
    float *zsum;             // [BH][P][128][64]  segment maps Z = [N; M]
    __half *sstart;          // [BH][P][64][64]   state entering each segment (fp16, fix-up operand)
    void *stash_o;           // [BH][NC][64][64]  o0 per chunk (tracked segments), fp32 or fp16
    __half *stash_q;         // [BH][NC][64][64]  Qhat per chunk (tracked segments)
    int P;                   // segments per sequence
};

bool tc_supported(const Shape &s, prism_dtype io);
int tc_segments(const Shape &s, int sm_count, long long opt);
size_t tc_workspace_bytes(const Shape &s, int P);
void tc_carve(const Shape &s, int P, void *base, TcWorkspace *w);
cudaError_t tc_prepare();
cudaError_t tc_forward(const Shape &s, const ForwardArgs &a, bool out_f32, const TcWorkspace &w, int *d_status,
                       long long wait_ns, KernelTimer &tm);

// Workspace of the chunk-map path (dk = dv = 128): the per-chunk maps, fp16, row-major.
struct MapWorkspace {
    __half *A;  // [BH*NC][128][128]  A_c (state -> state)
    __half *Q;  // [BH*NC][64][128]   Q~   (state -> outputs)
    __half *B;  // [BH*NC][128][128]  B_c (the chunk's own write)
    __half *O;  // [BH*NC][64][128]   O_loc (the chunk's outputs from a zero state)
};

bool map_supported(const Shape &s, prism_dtype io);
size_t map_workspace_bytes(const Shape &s);
void map_carve(const Shape &s, void *base, MapWorkspace *w);
cudaError_t map_prepare();
cudaError_t map_forward(const Shape &s, const ForwardArgs &a, bool out_f32, const MapWorkspace &w, int sm_count,
                        int *d_status, long long wait_ns, KernelTimer &tm);

// v_hist_out = the last three tokens of [v_hist; v] (kernel in prism_state.cu); safe in place
cudaError_t launch_history(const Shape &s, prism_dtype io, const void *v_hist, const void *v, void *v_hist_out,
                           KernelTimer &tm);

// One recurrent step for every (batch, head) (layouts as in prism.h, prism_decode_step).
struct DecodeArgs {
    const void *q, *k, *v, *u, *conv_w;
    const float *beta, *alpha, *gamma, *eta;
    void *v_hist;
    float *S;
    void *out;
};
cudaError_t decode_step(const Shape &s, prism_dtype io, prism_dtype out, const DecodeArgs &a, int sm_count,
                        int *d_status, long long wait_ns, KernelTimer &tm);

// Pointers of one backward call (layouts as in prism.h, prism_backward).  v_hist, S_init,
// dS_final, dv_hist and dS_init may be null; u, gamma, eta, du, dgamma and deta are not read or
// written when R = 0.
struct BackwardArgs {
    const void *q, *k, *v, *u, *conv_w, *v_hist;
    const float *beta, *alpha, *gamma, *eta, *S_init, *dout, *dS_final;
    float *dq, *dk, *dv, *dbeta, *dalpha, *du, *dgamma, *deta, *dconv_w, *dv_hist, *dS_init;
    // the non-linear residual chain: gains [BH T][R][dv] in the io dtype in place of eta, and
    // their cotangent (fp32, same layout) in place of deta; null for the linear chain
    const void *p_gain = nullptr;
    float *dp_gain = nullptr;
};
// token-serial backward (every shape): per-token states and cotangents in the workspace
size_t backward_workspace_bytes(const Shape &s);
cudaError_t backward_prepare();
cudaError_t backward(const Shape &s, prism_dtype io, const BackwardArgs &a, void *ws, KernelTimer &tm);
// the token-local tail shared by both backward forms (prism_backward.cu): chain, gain and convolution
// backwards from dX [BH T][R][dv] and dv = beta z; dH [BH T][dv] and dWp are scratch
int backward_conv_tiles(int T);
cudaError_t backward_token_local(const Shape &s, prism_dtype io, const BackwardArgs &a, float *dX, float *dH,
                                 float *dWp, KernelTimer &tm);
// chunked backward on the tensor cores (prism_bwd_tc.cu; bf16 io, dk = dv = 64, L <= 4): per-chunk
// maps, a chunk-level scan of the states and cotangents, per-chunk cotangent products
bool backward_tc_supported(const Shape &s, prism_dtype io);
size_t backward_tc_workspace_bytes(const Shape &s);
cudaError_t backward_tc_prepare();
cudaError_t backward_tc(const Shape &s, const BackwardArgs &a, void *ws, int *d_status, long long wait_ns,
                        KernelTimer &tm);

size_t simt_workspace_bytes(const Shape &s);
void simt_carve(const Shape &s, void *base, SimtWorkspace *w);
cudaError_t simt_prepare(const Shape &s, prism_dtype io);
cudaError_t simt_forward(const Shape &s, prism_dtype io, prism_dtype out, const ForwardArgs &a,
                         const SimtWorkspace &w, int *d_status, KernelTimer &timer);

}  // namespace prism

// Sets the message prism_last_error_message() returns on the calling thread.
void prism_set_error_message(const char *msg);

struct prism_plan_s {
    prism::Shape shape;
    prism_dtype io;
    int device;
    int sm_count;
    long long opt_segments;
    long long opt_path;
    long long opt_wait_ns;
    long long opt_timing;
    prism_dtype out_dtype;
    prism::KernelTimer timer;
    // device memory (owned): status word, and one workspace per path, allocated on first use
    int *d_status;
    void *ws_simt;
    size_t ws_simt_bytes;
    prism::SimtWorkspace simt;
    void *ws_tc;
    size_t ws_tc_bytes;
    prism::TcWorkspace tcw;
    void *ws_map;
    size_t ws_map_bytes;
    prism::MapWorkspace mapw;
    // workspace of the backward pass (owned, allocated by the first prism_backward)
    void *ws_bwd;
    size_t ws_bwd_bytes;
    // device staging buffers for prism_forward_host (owned, allocated on first use)
    void *stage;
    size_t stage_bytes;
};
