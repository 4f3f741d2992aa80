// fw_internal.cuh -- declarations shared by the translation units of libfw.so.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "fw.h"

namespace fw {

// Device error word values (written by kernels, read by fw_check).
enum : int { kDevErrNone = 0, kDevErrTimeout = 1 };

// Arguments of one prefill call, already validated.
struct PrefillArgs {
    const void *q, *k, *v;
    const float *beta, *lam, *S0;
    const void *k_init;
    void *o;
    float *S_T;
    int64_t n_chains;  // B * H
    int64_t T;
    int d;             // d_k == d_v
    fw_dtype dtype;
    fw_mode mode;
    fw_phi phi;
    float eps;
    unsigned flags;    // FW_FLAG_* bits
    int *err;          // device error word
    long long wait_ns; // limit of every bounded device wait, nanoseconds
    int force_timeout; // testing hook: wait on a barrier nothing arrives on
    int seg_pref;      // two-segment split of few long chains: 0 auto, 1 always, -1 never
    // Set by the chunked launch when it splits each chain at token seg_t0 (> 0):
    int64_t seg_t0;
    void *o_aux;       // outputs of the transition run, bf16 [n_chains][T - seg_t0][d]
    float *s_aux;      // S at the split, S_T from a zero start, transition: fp32 [3][n_chains][d][d]
    // fw_prefill_noalloc: the two-segment workspace comes from this buffer only
    int scratch_only;
    void *scratch;
    size_t scratch_bytes;
};

struct StepArgs {
    const void *q, *k, *v;
    const float *beta, *lam;
    float *S;
    void *o;
    int64_t n_states;
    int d;
    fw_dtype dtype;
    fw_mode mode;
    fw_phi phi;
    float eps;
    unsigned flags;    // FW_FLAG_* bits
};

// Arguments of one Falcon-3 / 3A call (prefill, or a step with T = 1 and
// S0 == S_T == the state), already validated.
struct WindowArgs {
    const void *q, *k, *v;
    const float *beta, *lam, *S0;
    const void *k_init;           // shifted pair of the first token, or NULL
    const float *cx, *cy;         // carried window in (NULL: empty)
    const int *cn;
    void *o;
    float *S_T;
    float *ox, *oy;               // window out (NULL: not wanted)
    int *on;
    int64_t n_chains;
    int64_t T;
    int d;                        // d_k == d_v
    int W;                        // window, 1 .. FW_WINDOW_MAX
    fw_dtype dtype;
    bool inner;                   // Falcon-3A (Falcon-2A with chan)
    bool chan;                    // Falcon-2 / 2A: W = 1, beta [T][d_v] (a step per value column)
    fw_phi phi;
    float eps;
    unsigned flags;
    int *err;                     // device error word
    long long wait_ns;            // limit of every bounded device wait, nanoseconds
};

// Launchers (return a cudaError_t from the launch).
cudaError_t launch_window_prefill(const WindowArgs &a, cudaStream_t s);
cudaError_t launch_window_step(const WindowArgs &a, cudaStream_t s);
cudaError_t launch_recurrent(const PrefillArgs &a, cudaStream_t s);
cudaError_t launch_decode(const StepArgs &a, cudaStream_t s);
// Chunked tensor-core prefill.  supported() tells whether it takes the call.
bool chunked_supported(const PrefillArgs &a);
cudaError_t launch_chunked(const PrefillArgs &a, cudaStream_t s);
// Bytes of workspace the chunked launch's two-segment form takes for this call
// on a device with `sms` SMs (0: the call runs as one segment).
size_t chunked_segment_bytes(const PrefillArgs &a, int sms);
// Device address of the static buffer of fw_prefill_noalloc on device `dev`
// (looked up once per device), or nullptr with the CUDA error in *e.
void *segment_scratch(int dev, cudaError_t *e);
// Chunked tensor-core prefill of the per-channel step (Falcon-2 / 2A).
bool chunked_chan_supported(const PrefillArgs &a);
cudaError_t launch_chunked_chan(const PrefillArgs &a, cudaStream_t s);

// ---- small device helpers ------------------------------------------------

__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }

template <typename T> __device__ __forceinline__ T from_f32(float x);
template <> __device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) {
    return __float2bfloat16_rn(x);
}

// phi(z) = elu(z) + 1 = z + 1 (z > 0), exp(z) (z <= 0); identity otherwise.
__device__ __forceinline__ float apply_phi(int phi, float z) {
    if (phi == FW_PHI_ELU1) return z > 0.f ? z + 1.f : expf(z);
    return z;
}

}  // namespace fw
