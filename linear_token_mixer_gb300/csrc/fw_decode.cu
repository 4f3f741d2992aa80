// fw_decode.cu -- single-token decode step, one pass over the state.
//
// One thread block (256 threads) per state.  The state S (d x d fp32, d_v
// innermost) is streamed once through registers with 128-bit loads and
// stores: a warp covers one row per pass (32 lanes x float4 for d = 128).
// From the old state the block forms, in the same pass, a_j = S[:,j].x and
// c_j = S[:,j].q (partial sums per thread, then a shared-memory reduction over
// row groups), and with n = |x|^2 and x.q from the staged vectors it applies
//     eta = beta / (n + lambda + eps), gamma = 1 - eta lambda,
//     r_j = v_j - a_j,  o_j = gamma c_j + eta r_j (x.q)  (= (S_new^T q)_j),
//     S[i][j] <- gamma S[i][j] + eta x_i r_j,
// the Falcon-1 write and read-after-write of "Fast Weight Attention for
// Continual Learning" paper reading §3.2/§1.4 with the pair (phi(k_prev), v).
// Falcon-1A (§4.3) drops the residual (r = v); Falcon-2 / 2A (§4.2) take beta,
// and so eta and gamma, per value column; FW_FLAG_RBW reads before the write,
// o_j = c_j.  Linear-attention mode: x = phi(k), r = v,
// eta = gamma = 1, read with phi(q) ("Attention is also an FFN" blog §4.1,
// forward_step).
//
// Traffic per state: d*d*4 bytes read + the same written, plus 3 d-vectors.
// The state is read and written with streaming (evict-first) hints since a
// decode batch of states is larger than L2 and is not reused within a step.
#include "fw_internal.cuh"

namespace fw {
namespace {

constexpr int kThreads = 256;

template <int D, typename TIn>
__global__ void __launch_bounds__(kThreads)
decode_kernel(StepArgs a) {
    constexpr int TPR = D / 4;             // threads per row (one float4 each)
    constexpr int RPP = kThreads / TPR;    // rows per pass
    constexpr int NP = D / RPP;            // passes
    const int tid = threadIdx.x;
    const int cq = tid % TPR;
    const int rg = tid / TPR;
    const int64_t s = blockIdx.x;
    const bool falcon = (a.mode != FW_LINATTN);   // eta, gamma
    const bool resid = (a.mode == FW_FALCON1 || a.mode == FW_FALCON2);   // r = v - S^T x
    const bool chan = (a.mode == FW_FALCON2 || a.mode == FW_FALCON2A);   // beta per column
    const bool rbw = (a.flags & FW_FLAG_RBW) != 0;

    float4 *Sp = reinterpret_cast<float4 *>(a.S + s * D * D);
    float4 Sr[NP];
#pragma unroll
    for (int p = 0; p < NP; ++p) Sr[p] = __ldcs(&Sp[(p * RPP + rg) * TPR + cq]);

    __shared__ float xs[D], qs[D], vs[D];
    __shared__ float wsum[D / 32][2];
    __shared__ float4 red[RPP][2][TPR];

    if (tid < D) {
        const TIn *qg = static_cast<const TIn *>(a.q) + s * D;
        const TIn *kg = static_cast<const TIn *>(a.k) + s * D;
        const TIn *vg = static_cast<const TIn *>(a.v) + s * D;
        const float x = apply_phi(a.phi, to_f32(kg[tid]));
        float qv = to_f32(qg[tid]);
        if (!falcon) qv = apply_phi(a.phi, qv);
        xs[tid] = x;
        qs[tid] = qv;
        vs[tid] = to_f32(vg[tid]);
        float n = x * x, xq = x * qv;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            n += __shfl_xor_sync(0xffffffffu, n, off);
            xq += __shfl_xor_sync(0xffffffffu, xq, off);
        }
        if ((tid & 31) == 0) { wsum[tid >> 5][0] = n; wsum[tid >> 5][1] = xq; }
    }
    __syncthreads();

    float n = 0.f, xq = 0.f;
#pragma unroll
    for (int w = 0; w < D / 32; ++w) { n += wsum[w][0]; xq += wsum[w][1]; }
    // eta, gamma of this thread's four value columns cq*4 .. cq*4+3
    float4 eta = make_float4(1.f, 1.f, 1.f, 1.f), gam = eta;
    if (falcon) {
        const float lt = a.lam[s];
        const float den = n + lt + a.eps;
        const float4 b4 = chan ? *reinterpret_cast<const float4 *>(a.beta + s * D + cq * 4)
                               : make_float4(a.beta[s], a.beta[s], a.beta[s], a.beta[s]);
        eta = make_float4(b4.x / den, b4.y / den, b4.z / den, b4.w / den);
        gam = make_float4(1.f - eta.x * lt, 1.f - eta.y * lt, 1.f - eta.z * lt, 1.f - eta.w * lt);
    }

    float4 pa = make_float4(0.f, 0.f, 0.f, 0.f), pc = pa;
#pragma unroll
    for (int p = 0; p < NP; ++p) {
        const int row = p * RPP + rg;
        const float xr = xs[row], qr = qs[row];
        pa.x = fmaf(Sr[p].x, xr, pa.x); pa.y = fmaf(Sr[p].y, xr, pa.y);
        pa.z = fmaf(Sr[p].z, xr, pa.z); pa.w = fmaf(Sr[p].w, xr, pa.w);
        pc.x = fmaf(Sr[p].x, qr, pc.x); pc.y = fmaf(Sr[p].y, qr, pc.y);
        pc.z = fmaf(Sr[p].z, qr, pc.z); pc.w = fmaf(Sr[p].w, qr, pc.w);
    }
    red[rg][0][cq] = pa;
    red[rg][1][cq] = pc;
    __syncthreads();

    float4 A = make_float4(0.f, 0.f, 0.f, 0.f), C = A;
#pragma unroll
    for (int g = 0; g < RPP; ++g) {
        const float4 u = red[g][0][cq], w = red[g][1][cq];
        A.x += u.x; A.y += u.y; A.z += u.z; A.w += u.w;
        C.x += w.x; C.y += w.y; C.z += w.z; C.w += w.w;
    }
    const float4 vv = *reinterpret_cast<const float4 *>(&vs[cq * 4]);
    float4 r;
    if (resid) { r.x = vv.x - A.x; r.y = vv.y - A.y; r.z = vv.z - A.z; r.w = vv.w - A.w; }
    else r = vv;

    if (rg == 0) {
        float4 ov = C;   // read before the write
        if (!rbw) {
            ov.x = fmaf(gam.x, C.x, eta.x * xq * r.x); ov.y = fmaf(gam.y, C.y, eta.y * xq * r.y);
            ov.z = fmaf(gam.z, C.z, eta.z * xq * r.z); ov.w = fmaf(gam.w, C.w, eta.w * xq * r.w);
        }
        TIn *og = static_cast<TIn *>(a.o) + s * D + cq * 4;
        og[0] = from_f32<TIn>(ov.x); og[1] = from_f32<TIn>(ov.y);
        og[2] = from_f32<TIn>(ov.z); og[3] = from_f32<TIn>(ov.w);
    }

#pragma unroll
    for (int p = 0; p < NP; ++p) {
        const int row = p * RPP + rg;
        const float xr = xs[row];
        float4 nv;
        nv.x = fmaf(gam.x, Sr[p].x, eta.x * xr * r.x); nv.y = fmaf(gam.y, Sr[p].y, eta.y * xr * r.y);
        nv.z = fmaf(gam.z, Sr[p].z, eta.z * xr * r.z); nv.w = fmaf(gam.w, Sr[p].w, eta.w * xr * r.w);
        __stcs(&Sp[row * TPR + cq], nv);
    }
}

template <int D, typename TIn>
cudaError_t launch_t(const StepArgs &a, cudaStream_t s) {
    decode_kernel<D, TIn><<<(unsigned)a.n_states, kThreads, 0, s>>>(a);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_decode(const StepArgs &a, cudaStream_t s) {
    if (a.d == 64)
        return a.dtype == FW_F32 ? launch_t<64, float>(a, s) : launch_t<64, __nv_bfloat16>(a, s);
    return a.dtype == FW_F32 ? launch_t<128, float>(a, s) : launch_t<128, __nv_bfloat16>(a, s);
}

}  // namespace fw
