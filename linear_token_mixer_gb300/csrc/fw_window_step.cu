// fw_window_step.cu -- Falcon-3 / 3A single-token decode step, one pass over
// the state.
//
// Two launches.  The window is the carried pairs plus the new pair
// (phi(k_prev), v) ("Fast Weight Attention for Continual Learning" paper
// reading §4.2, §4.3).
//   1. window_prep_kernel: a warp per state forms the window's Gram matrix
//      x_a . x_b and the products x_j . q (warp butterflies); then one lane per
//      state finds mu = lambda_max of the window-average covariance by Jacobi
//      rotations, and gamma = 1 - eta lambda and eta / B.  These 2 + W scalars are parked in
//      the state's own output slot o[s] (at least 128 bytes), which the second
//      launch reads before it writes the output there: no workspace.
//   2. window_step_kernel, one thread block (256 threads) per state, streaming
//      S (d x d fp32, d_v innermost) once through registers with 128-bit loads
//      and stores, as the Falcon-1 step does, with no eigenvalue work on the
//      state's critical path.  From the old state the pass forms the reads
//      a_j = S^T x_j of every window pair and c = S^T q; then, per value column,
//     r_j = y_j - a_j (3A: y_j),  coef_j = (eta / B) r_j,
//     o = gamma c + sum_j coef_j (x_j . q)        (= S_new^T q; RBW: o = c),
//     S <- gamma S + sum_j x_j coef_j^T,
// and the carried window moves on by one pair.
//
// Traffic per state: 2 d^2 * 4 bytes of state plus 2 (W-1) d * 8 bytes of
// carried window in and out and the step's vectors.
#include "fw_window.cuh"

namespace fw {
namespace {

constexpr int kThreads = 256;

// Offset of the scalars parked in o[s]: gamma, eta / B, then x_j . q.
template <typename TIn>
__device__ __forceinline__ float *parked(const WindowArgs &a, int64_t s, int D) {
    return reinterpret_cast<float *>(static_cast<TIn *>(a.o) + s * D);
}

// States per block of the prep launch: a warp per state forms the Gram matrix,
// then one lane per state (a single warp) runs the rotations, so no two lanes
// repeat the same eigenvalue work.
template <int WM> constexpr int prep_states() { return WM <= 4 ? 32 : 16; }

template <int D, int WM, typename TIn>
__global__ void __launch_bounds__(prep_states<WM>() * 32, WM <= 4 ? 2 : 1)
window_prep_kernel(WindowArgs a) {
    constexpr int SPB = prep_states<WM>();
    constexpr int PL = D / 32;   // elements of a row per lane
    __shared__ float gram[SPB][WM * WM + WM + 1];   // window Gram matrix, x_j . q, pairs held
    // the step launch may start now: it streams its state in before it waits for
    // this grid's scalars
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const int W = a.W;
    {
        const int64_t s = (int64_t)blockIdx.x * SPB + w;
        if (s < a.n_chains) {
            const int64_t cs = (int64_t)(W - 1) * D;
            int cn = a.cn ? a.cn[s] : 0;
            cn = cn < 0 ? 0 : (cn > W - 1 ? W - 1 : cn);
            // window rows j = 0 .. W-2: carried slots (held if j >= W-1-cn); row W-1:
            // the new pair's key, phi applied; rows past W are zero
            float x[WM][PL], qv[PL];
#pragma unroll
            for (int j = 0; j < WM; ++j)
#pragma unroll
                for (int e = 0; e < PL; ++e) {
                    const int i = lane + 32 * e;
                    float v = 0.f;
                    if (j < W - 1) {
                        if (a.cx && j >= W - 1 - cn) v = a.cx[s * cs + (int64_t)j * D + i];
                    } else if (j == W - 1) {
                        v = apply_phi(a.phi, to_f32(static_cast<const TIn *>(a.k)[s * D + i]));
                    }
                    x[j][e] = v;
                }
#pragma unroll
            for (int e = 0; e < PL; ++e)
                qv[e] = to_f32(static_cast<const TIn *>(a.q)[s * D + lane + 32 * e]);
            auto wsum = [&](float v) {
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
                return v;
            };
#pragma unroll
            for (int i = 0; i < WM; ++i) {
#pragma unroll
                for (int j = i; j < WM; ++j) {
                    float v = 0.f;
#pragma unroll
                    for (int e = 0; e < PL; ++e) v = fmaf(x[i][e], x[j][e], v);
                    v = wsum(v);
                    if (lane == 0) { gram[w][i * WM + j] = v; gram[w][j * WM + i] = v; }
                }
                float v = 0.f;
#pragma unroll
                for (int e = 0; e < PL; ++e) v = fmaf(x[i][e], qv[e], v);
                v = wsum(v);
                if (lane == 0) gram[w][WM * WM + i] = v;
            }
            if (lane == 0) gram[w][WM * WM + WM] = (float)(cn + 1);   // the carried pairs held, and the new one
        }
    }
    __syncthreads();
    if (w == 0 && lane < SPB) {
        const int64_t s = (int64_t)blockIdx.x * SPB + lane;
        if (s < a.n_chains) {
            float A[WM][WM];
#pragma unroll
            for (int i = 0; i < WM; ++i)
#pragma unroll
                for (int j = 0; j < WM; ++j) A[i][j] = gram[lane][i * WM + j];
            const float nb = gram[lane][WM * WM + WM];
            const float mu = window_max_eig<WM>(A) / nb;
            const float lt = a.lam[s];
            const float eta = a.beta[s] / (mu + lt + a.eps);
            float *sc = parked<TIn>(a, s, D);
            sc[0] = 1.f - eta * lt;
            sc[1] = eta / nb;
#pragma unroll
            for (int j = 0; j < WM; ++j) sc[2 + j] = gram[lane][WM * WM + j];
        }
    }
}

template <int D, int WM, typename TIn, bool INNER>
__global__ void __launch_bounds__(kThreads)
window_step_kernel(WindowArgs a) {
    constexpr int TPR = D / 4;             // threads per row (one float4 each)
    constexpr int RPP = kThreads / TPR;    // rows per pass
    constexpr int NP = D / RPP;            // passes
    constexpr int NR = INNER ? 1 : WM + 1; // reads reduced per column group
    const int tid = threadIdx.x;
    const int cq = tid % TPR, rg = tid / TPR;
    const int64_t s = blockIdx.x;
    const int W = a.W;
    const bool rbw = (a.flags & FW_FLAG_RBW) != 0;

    __shared__ __align__(16) float xs[WM][D];
    __shared__ __align__(16) float ys[WM][D];
    __shared__ float qs[D];
    __shared__ float Eq[WM], scal[2];
    __shared__ float4 red[RPP][NR][TPR];
    __shared__ float4 fin[NR][TPR];

    const int64_t cs = (int64_t)(W - 1) * D;
    int cn = a.cn ? a.cn[s] : 0;
    cn = cn < 0 ? 0 : (cn > W - 1 ? W - 1 : cn);
    // window rows j = 0 .. W-2: carried slots (held if j >= W-1-cn); row W-1:
    // the new pair.  Their loads go out before the state's.
    constexpr int NE = WM * D / kThreads;   // window elements per thread
    float xv[NE], yv[NE];
#pragma unroll
    for (int u = 0; u < NE; ++u) {
        const int e = tid + u * kThreads, j = e / D, i = e % D;
        xv[u] = 0.f;
        yv[u] = 0.f;
        if (j < W - 1) {
            if (a.cx && j >= W - 1 - cn) {
                xv[u] = a.cx[s * cs + e];
                yv[u] = a.cy[s * cs + e];
            }
        } else if (j == W - 1) {
            xv[u] = to_f32(static_cast<const TIn *>(a.k)[s * D + i]);
            yv[u] = to_f32(static_cast<const TIn *>(a.v)[s * D + i]);
        }
    }
    const float qv0 = tid < D ? to_f32(static_cast<const TIn *>(a.q)[s * D + tid]) : 0.f;

    float4 *Sp = reinterpret_cast<float4 *>(a.S_T + s * D * D);
    float4 Sr[NP];
#pragma unroll
    for (int p = 0; p < NP; ++p) Sr[p] = __ldcs(&Sp[(p * RPP + rg) * TPR + cq]);
    // gamma, eta / B and x_j . q from the prep launch, parked in o[s] (read before
    // this block writes the output there).  Launched as its dependent, this grid
    // may start while the prep grid runs: the loads above need nothing from it,
    // and the wait returns once its writes are visible.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const float scv = tid < 2 + WM ? parked<TIn>(a, s, D)[tid] : 0.f;

#pragma unroll
    for (int u = 0; u < NE; ++u) {
        const int e = tid + u * kThreads, j = e / D, i = e % D;
        xs[j][i] = j == W - 1 ? apply_phi(a.phi, xv[u]) : xv[u];
        ys[j][i] = yv[u];
    }
    if (tid < D) qs[tid] = qv0;
    if (tid < 2) scal[tid] = scv;
    else if (tid < 2 + WM) Eq[tid - 2] = scv;
    __syncthreads();

    // reads of the old state (the loads have landed by now)
    float4 pa[WM];
    float4 pc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int j = 0; j < WM; ++j) pa[j] = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int p = 0; p < NP; ++p) {
        const int row = p * RPP + rg;
        const float qv = qs[row];
        pc.x = fmaf(Sr[p].x, qv, pc.x); pc.y = fmaf(Sr[p].y, qv, pc.y);
        pc.z = fmaf(Sr[p].z, qv, pc.z); pc.w = fmaf(Sr[p].w, qv, pc.w);
        if constexpr (!INNER) {
#pragma unroll
            for (int j = 0; j < WM; ++j) {
                if (j < W) {
                    const float xv = xs[j][row];
                    pa[j].x = fmaf(Sr[p].x, xv, pa[j].x); pa[j].y = fmaf(Sr[p].y, xv, pa[j].y);
                    pa[j].z = fmaf(Sr[p].z, xv, pa[j].z); pa[j].w = fmaf(Sr[p].w, xv, pa[j].w);
                }
            }
        }
    }
    red[rg][NR - 1][cq] = pc;
    if constexpr (!INNER) {
#pragma unroll
        for (int j = 0; j < WM; ++j)
            if (j < W) red[rg][j][cq] = pa[j];
    }
    __syncthreads();   // partial reads complete
    // each read's RPP partials are summed once, by the row group whose index it
    // carries, then every thread takes the sums of its column quad
#pragma unroll
    for (int j = rg; j < NR; j += RPP) {
        float4 t = red[0][j][cq];
#pragma unroll
        for (int g = 1; g < RPP; ++g) {
            const float4 u = red[g][j][cq];
            t.x += u.x; t.y += u.y; t.z += u.z; t.w += u.w;
        }
        fin[j][cq] = t;
    }
    __syncthreads();   // sums complete

    const float gam = scal[0], cc = scal[1];
    const float4 C = fin[NR - 1][cq];
    float4 coef[WM];
#pragma unroll
    for (int j = 0; j < WM; ++j) {
        coef[j] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (j < W) {
            float4 r = *reinterpret_cast<const float4 *>(&ys[j][cq * 4]);
            if constexpr (!INNER) {
                const float4 A4 = fin[j][cq];
                r.x -= A4.x; r.y -= A4.y; r.z -= A4.z; r.w -= A4.w;
            }
            coef[j] = make_float4(cc * r.x, cc * r.y, cc * r.z, cc * r.w);
        }
    }

    if (rg == 0) {
        float4 ov = C;   // read before the write
        if (!rbw) {
            ov = make_float4(gam * C.x, gam * C.y, gam * C.z, gam * C.w);
#pragma unroll
            for (int j = 0; j < WM; ++j) {
                if (j < W) {
                    const float e = Eq[j];
                    ov.x = fmaf(coef[j].x, e, ov.x); ov.y = fmaf(coef[j].y, e, ov.y);
                    ov.z = fmaf(coef[j].z, e, ov.z); ov.w = fmaf(coef[j].w, e, ov.w);
                }
            }
        }
        TIn *og = static_cast<TIn *>(a.o) + s * D + cq * 4;
        og[0] = from_f32<TIn>(ov.x); og[1] = from_f32<TIn>(ov.y);
        og[2] = from_f32<TIn>(ov.z); og[3] = from_f32<TIn>(ov.w);
    }

#pragma unroll
    for (int p = 0; p < NP; ++p) {
        const int row = p * RPP + rg;
        float4 nv = make_float4(gam * Sr[p].x, gam * Sr[p].y, gam * Sr[p].z, gam * Sr[p].w);
#pragma unroll
        for (int j = 0; j < WM; ++j) {
            if (j < W) {
                const float xv = xs[j][row];
                nv.x = fmaf(xv, coef[j].x, nv.x); nv.y = fmaf(xv, coef[j].y, nv.y);
                nv.z = fmaf(xv, coef[j].z, nv.z); nv.w = fmaf(xv, coef[j].w, nv.w);
            }
        }
        __stcs(&Sp[row * TPR + cq], nv);
    }

    // the carried window moves on: slot j <- window row j+1
    if (a.ox) {
        for (int e = tid; e < (W - 1) * D; e += kThreads) {
            const int j = e / D, i = e % D;
            a.ox[s * cs + e] = xs[j + 1][i];
            a.oy[s * cs + e] = ys[j + 1][i];
        }
        if (tid == 0) a.on[s] = cn + 1 < W - 1 ? cn + 1 : W - 1;
    }
}

template <int D, int WM, typename TIn, bool INNER>
cudaError_t launch_t(const WindowArgs &a, cudaStream_t s) {
    constexpr int SPB = prep_states<WM>();
    const unsigned nprep = (unsigned)((a.n_chains + SPB - 1) / SPB);
    window_prep_kernel<D, WM, TIn><<<nprep, SPB * 32, 0, s>>>(a);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    // the step grid is the prep grid's programmatic dependent (it waits in-kernel)
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)a.n_chains);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, window_step_kernel<D, WM, TIn, INNER>, a);
}

template <int D, typename TIn>
cudaError_t launch_d(const WindowArgs &a, cudaStream_t s) {
    if (a.W <= 4)
        return a.inner ? launch_t<D, 4, TIn, true>(a, s) : launch_t<D, 4, TIn, false>(a, s);
    return a.inner ? launch_t<D, 8, TIn, true>(a, s) : launch_t<D, 8, TIn, false>(a, s);
}

}  // namespace

cudaError_t launch_window_step(const WindowArgs &a, cudaStream_t s) {
    if (a.d == 64)
        return a.dtype == FW_F32 ? launch_d<64, float>(a, s) : launch_d<64, __nv_bfloat16>(a, s);
    return a.dtype == FW_F32 ? launch_d<128, float>(a, s) : launch_d<128, __nv_bfloat16>(a, s);
}

}  // namespace fw
