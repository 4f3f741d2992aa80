// fw_window.cuh -- pieces shared by the Falcon-3 / 3A kernels (the window
// write of "Fast Weight Attention for Continual Learning" paper reading §4.2).
#pragma once

#include "fw_internal.cuh"

namespace fw {

// Largest eigenvalue of the symmetric WM x WM matrix A (destroyed), which is
// zero outside the rows and columns of the pairs that exist.  Cyclic Jacobi:
// each rotation J = [[c, s], [-s, c]] on rows / columns (p, q) is chosen so
// that (J^T A J)_pq = 0 (Golub and Van Loan, the symmetric Schur
// decomposition), t = tan(theta) being the smaller root of
// t^2 + 2 tau t - 1 = 0 with tau = (a_qq - a_pp) / (2 a_pq); the two
// diagonal entries move by -t a_pq and +t a_pq.  Sweeps stop once the
// squared off-diagonal mass is below 1e-12 of the squared diagonal, or after
// 12 (window matrices converge in at most five).  Indices are compile-time,
// so A stays in registers.
template <int WM>
__device__ __forceinline__ float window_max_eig(float (&A)[WM][WM]) {
    for (int sweep = 0; sweep < 12; ++sweep) {
        float off = 0.f, dg = 0.f;
#pragma unroll
        for (int p = 0; p < WM; ++p)
#pragma unroll
            for (int q = 0; q < WM; ++q) {
                if (p == q) dg = fmaf(A[p][q], A[p][q], dg);
                else off = fmaf(A[p][q], A[p][q], off);
            }
        if (!(off > 1e-12f * dg)) break;
#pragma unroll
        for (int p = 0; p < WM - 1; ++p)
#pragma unroll
            for (int q = p + 1; q < WM; ++q) {
                const float apq = A[p][q];
                if (apq != 0.f) {
                    // fast reciprocal square root and division (a few ulp): the
                    // rotations stay orthogonal to a few ulp, far inside the
                    // eigenvalue accuracy the step needs
                    const float tau = __fdividef(A[q][q] - A[p][p], 2.f * apq);
                    const float at = fabsf(tau), r = fmaf(tau, tau, 1.f);
                    // for |tau| beyond 1e18, t = 1 / (2 tau) to fp32 precision (and
                    // tau * tau would overflow)
                    const float t = at > 1e18f ? __fdividef(0.5f, tau)
                                               : copysignf(__fdividef(1.f, at + r * rsqrtf(r)), tau);
                    const float c = rsqrtf(fmaf(t, t, 1.f)), s = t * c;
#pragma unroll
                    for (int k = 0; k < WM; ++k) {
                        if (k == p || k == q) continue;
                        const float akp = A[k][p], akq = A[k][q];
                        A[k][p] = A[p][k] = c * akp - s * akq;
                        A[k][q] = A[q][k] = s * akp + c * akq;
                    }
                    A[p][p] -= t * apq;
                    A[q][q] += t * apq;
                    A[p][q] = A[q][p] = 0.f;
                }
            }
    }
    float m = A[0][0];
#pragma unroll
    for (int p = 1; p < WM; ++p) m = fmaxf(m, A[p][p]);
    return m;
}

}  // namespace fw
