// fw_window_step.cu -- Falcon-3 / 3A single-token decode step, one pass over
// the state.
//
// One thread block (256 threads) per state, streaming S (d x d fp32, d_v
// innermost) once through registers with 128-bit loads and stores, as the
// Falcon-1 step does.  The window is the carried pairs plus the new pair
// (phi(k_prev), v) ("Fast Weight Attention for Continual Learning" paper
// reading §4.2, §4.3).  While the state's loads are in flight the block
// stages the window, forms its Gram matrix x_a . x_b and the products
// x_j . q (one warp per product), and one thread finds mu = lambda_max of the
// window-average covariance by Jacobi rotations.  From the old state the
// same pass forms the reads a_j = S^T x_j of every window pair and c = S^T q;
// then, per value column,
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

template <int D, int WM, typename TIn, bool INNER>
__global__ void __launch_bounds__(kThreads)
window_step_kernel(WindowArgs a) {
    constexpr int TPR = D / 4;             // threads per row (one float4 each)
    constexpr int RPP = kThreads / TPR;    // rows per pass
    constexpr int NP = D / RPP;            // passes
    constexpr int NR = INNER ? 1 : WM + 1; // reads reduced per column group
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int cq = tid % TPR, rg = tid / TPR;
    const int64_t s = blockIdx.x;
    const int W = a.W;
    const bool rbw = (a.flags & FW_FLAG_RBW) != 0;

    __shared__ __align__(16) float xs[WM][D];
    __shared__ __align__(16) float ys[WM][D];
    __shared__ float qs[D];
    __shared__ float G[WM][WM], Eq[WM], scal[2];
    __shared__ float4 red[RPP][NR][TPR];

    const int64_t cs = (int64_t)(W - 1) * D;
    int cn = a.cn ? a.cn[s] : 0;
    cn = cn < 0 ? 0 : (cn > W - 1 ? W - 1 : cn);
    // window rows j = 0 .. W-2: carried slots (held if j >= W-1-cn); row W-1:
    // the new pair.  Their loads go out before the state's, so the window's
    // Gram matrix and eigenvalue are formed while the state streams in.
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

#pragma unroll
    for (int u = 0; u < NE; ++u) {
        const int e = tid + u * kThreads, j = e / D, i = e % D;
        xs[j][i] = j == W - 1 ? apply_phi(a.phi, xv[u]) : xv[u];
        ys[j][i] = yv[u];
    }
    if (tid < D) qs[tid] = qv0;
    __syncthreads();

    // Gram matrix of the window (upper triangle) and x_j . q, one warp each
    {
        const int ng = W * (W + 1) / 2;
        for (int it = warp; it < ng + W; it += kThreads / 32) {
            const float *u, *w;
            int ia = 0, ib = 0;
            if (it < ng) {
                int r = it;
                while (r >= W - ia) { r -= W - ia; ++ia; }
                ib = ia + r;
                u = xs[ia];
                w = xs[ib];
            } else {
                ia = it - ng;
                u = xs[ia];
                w = qs;
            }
            float acc = 0.f;
#pragma unroll
            for (int i = lane; i < D; i += 32) acc = fmaf(u[i], w[i], acc);
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
            if (lane == 0) {
                if (it < ng) { G[ia][ib] = acc; G[ib][ia] = acc; }
                else Eq[ia] = acc;
            }
        }
    }

    __syncthreads();   // Gram matrix complete
    // mu, eta, gamma while the state's loads are still in flight
    if (tid == 0) {
        float A[WM][WM];
#pragma unroll
        for (int i = 0; i < WM; ++i)
#pragma unroll
            for (int j = 0; j < WM; ++j) A[i][j] = (i < W && j < W) ? G[i][j] : 0.f;
        const int nb = cn + 1;   // the carried pairs held, and the new one
        const float mu = window_max_eig<WM>(A) / (float)nb;
        const float lt = a.lam[s];
        const float eta = a.beta[s] / (mu + lt + a.eps);
        scal[0] = 1.f - eta * lt;
        scal[1] = eta / (float)nb;
    }
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

    const float gam = scal[0], cc = scal[1];

    float4 C = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int g = 0; g < RPP; ++g) {
        const float4 u = red[g][NR - 1][cq];
        C.x += u.x; C.y += u.y; C.z += u.z; C.w += u.w;
    }
    float4 coef[WM];
#pragma unroll
    for (int j = 0; j < WM; ++j) {
        coef[j] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (j < W) {
            float4 r = *reinterpret_cast<const float4 *>(&ys[j][cq * 4]);
            if constexpr (!INNER) {
                float4 A4 = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                for (int g = 0; g < RPP; ++g) {
                    const float4 u = red[g][j][cq];
                    A4.x += u.x; A4.y += u.y; A4.z += u.z; A4.w += u.w;
                }
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
    window_step_kernel<D, WM, TIn, INNER><<<(unsigned)a.n_chains, kThreads, 0, s>>>(a);
    return cudaGetLastError();
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
