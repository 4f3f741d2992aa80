// fw_window.cuh -- pieces shared by the Falcon-3 / 3A kernels (the window
// write of "Fast Weight Attention for Continual Learning" paper reading §4.2).
#pragma once

#include "fw_internal.cuh"

namespace fw {

// Round-robin ("circle") pairing of WM indices: in round r (0 .. WM-2) slot k
// pairs jac_a(r, k) with jac_b(r, k); every round is a perfect matching and a
// sweep of WM-1 rounds meets every pair once.
__host__ __device__ constexpr int jac_a(int n, int r, int k) { return k == 0 ? r : (r + k) % (n - 1); }
__host__ __device__ constexpr int jac_b(int n, int r, int k) {
    return k == 0 ? n - 1 : (r - k + (n - 1)) % (n - 1);
}

// Largest eigenvalue of the symmetric WM x WM matrix A (destroyed), which is
// zero outside the rows and columns of the pairs that exist.  Jacobi
// rotations in the parallel (round-robin) ordering (Golub and Van Loan, the
// symmetric Schur decomposition and its parallel orderings): each round
// rotates WM/2 disjoint index pairs at once, J = [[c, s], [-s, c]] on (p, q)
// chosen so that (J^T A J)_pq = 0, t = tan(theta) being the smaller root of
// t^2 + 2 tau t - 1 = 0 with tau = (a_qq - a_pp) / (2 a_pq); the round's
// rotations commute, so their angles come from the same A and the update is
// A <- J^T A J with J their product.  Sweeps stop once the squared
// off-diagonal mass is below 1e-12 of the squared diagonal, or after 12
// (window matrices converge in at most four).  Indices are compile-time, so A
// stays in registers, and the angles of a round are independent.
template <int WM>
__device__ __forceinline__ float window_max_eig(float (&A)[WM][WM]) {
    if constexpr (WM == 1) {
        return A[0][0];   // a window of one pair: mu = |x|^2
    } else {
    static_assert(WM % 2 == 0, "an even number of slots");
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
        for (int r = 0; r < WM - 1; ++r) {
            float cs[WM / 2], sn[WM / 2];
#pragma unroll
            for (int k = 0; k < WM / 2; ++k) {
                constexpr int n = WM;
                const int a0 = jac_a(n, r, k), b0 = jac_b(n, r, k);
                const int p = a0 < b0 ? a0 : b0, q = a0 < b0 ? b0 : a0;
                const float apq = A[p][q];
                float c = 1.f, s = 0.f;
                if (apq != 0.f) {
                    // fast reciprocal square root and division (a few ulp): the
                    // rotations stay orthogonal to a few ulp, far inside the
                    // eigenvalue accuracy the step needs
                    const float tau = __fdividef(A[q][q] - A[p][p], 2.f * apq);
                    const float at = fabsf(tau), r2 = fmaf(tau, tau, 1.f);
                    // for |tau| beyond 1e18, t = 1 / (2 tau) to fp32 precision (and
                    // tau * tau would overflow)
                    const float t = at > 1e18f ? __fdividef(0.5f, tau)
                                               : copysignf(__fdividef(1.f, at + r2 * rsqrtf(r2)), tau);
                    c = rsqrtf(fmaf(t, t, 1.f));
                    s = t * c;
                }
                cs[k] = c;
                sn[k] = s;
            }
            // A <- A J (columns p, q of every pair), then A <- J^T A (rows)
#pragma unroll
            for (int k = 0; k < WM / 2; ++k) {
                const int a0 = jac_a(WM, r, k), b0 = jac_b(WM, r, k);
                const int p = a0 < b0 ? a0 : b0, q = a0 < b0 ? b0 : a0;
#pragma unroll
                for (int i = 0; i < WM; ++i) {
                    const float aip = A[i][p], aiq = A[i][q];
                    A[i][p] = cs[k] * aip - sn[k] * aiq;
                    A[i][q] = sn[k] * aip + cs[k] * aiq;
                }
            }
#pragma unroll
            for (int k = 0; k < WM / 2; ++k) {
                const int a0 = jac_a(WM, r, k), b0 = jac_b(WM, r, k);
                const int p = a0 < b0 ? a0 : b0, q = a0 < b0 ? b0 : a0;
#pragma unroll
                for (int i = 0; i < WM; ++i) {
                    const float api = A[p][i], aqi = A[q][i];
                    A[p][i] = cs[k] * api - sn[k] * aqi;
                    A[q][i] = sn[k] * api + cs[k] * aqi;
                }
                A[p][q] = A[q][p] = 0.f;
            }
        }
    }
    float m = A[0][0];
#pragma unroll
    for (int p = 1; p < WM; ++p) m = fmaxf(m, A[p][p]);
    return m;
    }
}

}  // namespace fw
