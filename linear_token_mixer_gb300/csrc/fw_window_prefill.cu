// fw_window_prefill.cu -- Falcon-3 / 3A prefill, one token at a time (fp32).
//
// The write of "Fast Weight Attention for Continual Learning" paper reading
// §4.2 (Falcon-3) and §4.3 (Falcon-3A): one gradient step on the average loss
// of the window's pairs,
//     S_t = gamma_t S_{t-1} + c_t sum_{j=0}^{W-1} x_{t-j} r_{t,j}^T,
//     r_{t,j} = y_{t-j} - S_{t-1}^T x_{t-j}   (3A: y_{t-j}),
//     gamma_t = 1 - eta_t lambda_t,  c_t = eta_t / B_t,
//     eta_t = beta_t / (mu_t + lambda_t + eps),
// with mu_t the largest eigenvalue of the window-average key covariance.  A
// pair that does not exist has x = 0, so it drops out of every sum; B_t
// counts the ones that do.
//
// Work split.  The value columns are independent given the window's keys and
// step sizes, so a CTA owns 32 columns of one chain and every column is held
// by four threads, one per quarter of the key rows (the state never leaves
// registers).  Tokens are staged in blocks: the keys of the block's pairs
// (plus the W pairs before it), its queries and its targets go to shared
// memory, and everything that depends on keys alone is formed there for the
// whole block at once: the dot products x_a . x_b of pairs up to W apart,
// q_t . x_{t-j}, the window Gram matrices and their largest eigenvalue (one
// thread per token), eta_t, gamma_t and c_t.  The token loop then only reads
// the state twice per token.
//
// Residual reads by recursion.  Of the W residual reads S_{t-1}^T x_{t-j}
// only the newest pair's (j = 0) is a product with the state: for j >= 1 the
// pair was in token t-1's window too, and expanding S_{t-1} by token t-1's
// write gives
//     S_{t-1}^T x_{t-j} = gamma_{t-1} S_{t-2}^T x_{t-j}
//                         + sum_{j'} (x_{t-1-j'} . x_{t-j}) c_{t-1} r_{t-1,j'},
// where the first term is the previous token's read of the same pair.  The
// read after the write is expanded the same way,
//     o_t = S_t^T q_t = gamma_t S_{t-1}^T q_t + sum_j (x_{t-j} . q_t) c_t r_{t,j}.
// Per token and column this leaves two length-d_k reads and the rank-W write.
// The call's first token has no previous reads and forms all W.
#include "fw_window.cuh"

namespace fw {
namespace {

constexpr int kCG = 32;             // value columns per CTA
constexpr int kThreads = 4 * kCG;   // four threads (key-row quarters) per column

template <int DK, int WM>
struct WinLayout {
    static constexpr int NB = (WM <= 4) ? 32 : 16;  // tokens per staged block
    static constexpr int RQ = DK / 4;               // key rows per thread
    static constexpr int QS = RQ + 4;               // padded quarter: the four
                                                    // quarters start in different banks
    static constexpr int LD = 4 * QS;               // padded row
    static constexpr int NXR = NB + WM;             // key rows: pairs p0-WM .. p0+NB-1
    // offsets in floats
    static constexpr int X = 0;
    static constexpr int Q = X + NXR * LD;
    static constexpr int DOT = Q + NB * LD;          // [NXR][WM] x_r . x_{r-delta}
    static constexpr int E = DOT + NXR * WM;         // [NB][WM]  q_t . x_{t-j}
    static constexpr int M = E + NB * WM;            // [NB][WM][WM] recursion weights
    static constexpr int GAM = M + NB * WM * WM;     // [NB] gamma_t
    static constexpr int CC = GAM + NB;              // [NB] c_t = eta_t / B_t
    static constexpr int BETA = CC + NB;             // [NB]
    static constexpr int LAM = BETA + NB;            // [NB]
    static constexpr int V = LAM + NB;               // [NB][kCG] targets of the CTA's columns
    static constexpr int O = V + NB * kCG;           // [NB][kCG] outputs
    static constexpr int VAL = O + NB * kCG;         // [NXR] 1 if the pair exists
    static constexpr int TOTAL = VAL + NXR;
    static constexpr size_t BYTES = (size_t)TOTAL * sizeof(float);
};

// Position of key element i in a padded row.
template <int RQ>
__device__ __forceinline__ int padded(int i) {
    return (i / RQ) * (RQ + 4) + (i % RQ);
}

__device__ __forceinline__ float4 load4(const float *p) {
    return *reinterpret_cast<const float4 *>(p);
}
__device__ __forceinline__ float4 load4(const __nv_bfloat16 *p) {
    const uint2 u = *reinterpret_cast<const uint2 *>(p);
    const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&u.x));
    const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&u.y));
    return make_float4(a.x, a.y, b.x, b.y);
}

// Dot product of two padded rows (the padding is skipped).
template <int DK>
__device__ __forceinline__ float row_dot(const float *u, const float *w) {
    constexpr int RQ = DK / 4;
    float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f;
#pragma unroll
    for (int qq = 0; qq < 4; ++qq)
#pragma unroll
        for (int m = 0; m < RQ; m += 4) {
            const float4 a = load4(u + qq * (RQ + 4) + m), b = load4(w + qq * (RQ + 4) + m);
            s0 = fmaf(a.x, b.x, s0); s1 = fmaf(a.y, b.y, s1);
            s2 = fmaf(a.z, b.z, s2); s3 = fmaf(a.w, b.w, s3);
        }
    return (s0 + s1) + (s2 + s3);
}

template <int DK, int WM, typename TIn, bool INNER>
__global__ void __launch_bounds__(kThreads, 4)
window_prefill_kernel(WindowArgs a) {
    using L = WinLayout<DK, WM>;
    constexpr int NB = L::NB, RQ = L::RQ, QS = L::QS, LD = L::LD, NXR = L::NXR;
    extern __shared__ __align__(16) float sm[];
    float *X = sm + L::X, *Qs = sm + L::Q, *DOT = sm + L::DOT, *E = sm + L::E,
          *Mw = sm + L::M, *GAM = sm + L::GAM, *CC = sm + L::CC, *BETA = sm + L::BETA,
          *LAM = sm + L::LAM, *V = sm + L::V, *O = sm + L::O, *VAL = sm + L::VAL;

    const int tid = threadIdx.x, qr = tid & 3, cl = tid >> 2;
    const int64_t chain = blockIdx.x;
    const int col0 = blockIdx.y * kCG, col = col0 + cl;
    const int W = a.W;
    const int64_t T = a.T;
    const bool same = (a.flags & FW_FLAG_SAME_PAIR) != 0;
    const bool rbw = (a.flags & FW_FLAG_RBW) != 0;
    const TIn *qg = static_cast<const TIn *>(a.q) + chain * T * DK;
    const TIn *kg = static_cast<const TIn *>(a.k) + chain * T * DK;
    const TIn *vg = static_cast<const TIn *>(a.v) + chain * T * DK;
    const TIn *ki = a.k_init ? static_cast<const TIn *>(a.k_init) + chain * DK : nullptr;
    const float *bg = a.beta + chain * T, *lg = a.lam + chain * T;
    TIn *og = static_cast<TIn *>(a.o) + chain * T * DK;
    const int64_t cs = (int64_t)(W - 1) * DK;   // carried window, per chain
    const float *cx = a.cx ? a.cx + chain * cs : nullptr;
    const float *cy = a.cy ? a.cy + chain * cs : nullptr;
    int cn = a.cn ? a.cn[chain] : 0;
    cn = cn < 0 ? 0 : (cn > W - 1 ? W - 1 : cn);

    float S[RQ];   // S[qr*RQ + m][col]
#pragma unroll
    for (int m = 0; m < RQ; ++m)
        S[m] = a.S0 ? a.S0[chain * DK * DK + (int64_t)(qr * RQ + m) * DK + col] : 0.f;

    // vr[j]: target of pair p - j; pairs before the call come from the carry
    // (pair -j sits in slot W-1-j, held if j <= cn)
    float vr[WM], a_prev[WM], coef_prev[WM];
#pragma unroll
    for (int j = 0; j < WM; ++j) {
        vr[j] = (j >= 1 && j < W && j <= cn && cy) ? cy[(int64_t)(W - 1 - j) * DK + col] : 0.f;
        a_prev[j] = 0.f;
        coef_prev[j] = 0.f;
    }
    float gam_prev = 1.f;

    for (int64_t p0 = 0; p0 < T; p0 += NB) {
        const int nt = (int)(T - p0 < NB ? T - p0 : NB);
        __syncthreads();   // the previous block is read out
        // keys: row r holds pair m = p0 - WM + r, phi applied, 0 if it does not exist
        for (int e = tid; e < NXR * (DK / 4); e += kThreads) {
            const int r = e / (DK / 4), i4 = (e % (DK / 4)) * 4;
            const int64_t m = p0 - WM + r;
            float4 xv = make_float4(0.f, 0.f, 0.f, 0.f);
            bool have = false;
            if (m < 0) {
                const int64_t s = m + W - 1;
                if (cx && s >= 0 && s >= W - 1 - cn) {
                    xv = load4(cx + s * DK + i4);
                    have = true;
                }
            } else if (m < T) {
                const int64_t kk = same ? m : m - 1;
                const TIn *src = kk >= 0 ? kg + kk * DK : ki;
                if (src) {
                    xv = load4(src + i4);
                    xv.x = apply_phi(a.phi, xv.x); xv.y = apply_phi(a.phi, xv.y);
                    xv.z = apply_phi(a.phi, xv.z); xv.w = apply_phi(a.phi, xv.w);
                    have = true;
                }
            }
            *reinterpret_cast<float4 *>(X + r * LD + padded<RQ>(i4)) = xv;
            if (i4 == 0) VAL[r] = have ? 1.f : 0.f;
        }
        for (int e = tid; e < NB * (DK / 4); e += kThreads) {
            const int t = e / (DK / 4), i4 = (e % (DK / 4)) * 4;
            const float4 qv = t < nt ? load4(qg + (p0 + t) * DK + i4) : make_float4(0.f, 0.f, 0.f, 0.f);
            *reinterpret_cast<float4 *>(Qs + t * LD + padded<RQ>(i4)) = qv;
        }
        for (int e = tid; e < NB * kCG; e += kThreads) {
            const int t = e / kCG, c = e % kCG;
            V[e] = t < nt ? to_f32(vg[(p0 + t) * DK + col0 + c]) : 0.f;
        }
        if (tid < NB) {
            BETA[tid] = tid < nt ? bg[p0 + tid] : 0.f;
            LAM[tid] = tid < nt ? lg[p0 + tid] : 0.f;
        }
        __syncthreads();
        // dot products of keys up to W-1 pairs apart, and of queries with the
        // keys of their window
        for (int e = tid; e < (NXR + NB) * W; e += kThreads) {
            const int i = e / W, dl = e % W;
            if (i < NXR) {
                DOT[i * WM + dl] = i - dl >= 0 ? row_dot<DK>(X + i * LD, X + (i - dl) * LD) : 0.f;
            } else {
                const int t = i - NXR;
                E[t * WM + dl] = row_dot<DK>(Qs + t * LD, X + (t + WM - dl) * LD);
            }
        }
        __syncthreads();
        // step size of every token of the block, and the weights of the
        // residual-read recursion, M[t][j][j'] = x_{p-1-j'} . x_{p-j}
        if (tid < nt) {
            const int t = tid, rr = t + WM;   // row of pair p
            float G[WM][WM];
            int nb = 0;
#pragma unroll
            for (int i = 0; i < WM; ++i) {
                if (i < W && VAL[rr - i] != 0.f) ++nb;
#pragma unroll
                for (int j = 0; j < WM; ++j) {
                    const int lo = i < j ? i : j, dl = i < j ? j - i : i - j;
                    G[i][j] = (i < W && j < W) ? DOT[(rr - lo) * WM + dl] : 0.f;
                }
            }
            float eta = 0.f;
            if (nb > 0) {
                const float mu = window_max_eig<WM>(G) / (float)nb;
                eta = BETA[t] / (mu + LAM[t] + a.eps);
            }
            GAM[t] = 1.f - eta * LAM[t];
            CC[t] = nb > 0 ? eta / (float)nb : 0.f;
#pragma unroll
            for (int j = 0; j < WM; ++j)
#pragma unroll
                for (int jp = 0; jp < WM; ++jp) {
                    float w = 0.f;
                    if (j >= 1 && j < W && jp < W) {
                        const int ra = rr - 1 - jp, rb = rr - j;
                        w = ra > rb ? DOT[ra * WM + (ra - rb)] : DOT[rb * WM + (rb - ra)];
                    }
                    Mw[(t * WM + j) * WM + jp] = w;
                }
        }
        __syncthreads();

        for (int t = 0; t < nt; ++t) {
            const int64_t p = p0 + t;
            const int rr = t + WM;
            const float gam = GAM[t], cc = CC[t];
            vr[0] = V[t * kCG + cl];
            const float *xp = X + rr * LD + qr * QS, *qp = Qs + t * LD + qr * QS;
            float xa[RQ];
            float pa0 = 0.f, pa1 = 0.f, pc0 = 0.f, pc1 = 0.f;
#pragma unroll
            for (int m = 0; m < RQ; m += 4) {
                const float4 x4 = load4(xp + m), q4 = load4(qp + m);
                xa[m] = x4.x; xa[m + 1] = x4.y; xa[m + 2] = x4.z; xa[m + 3] = x4.w;
                pa0 = fmaf(S[m], x4.x, pa0); pa1 = fmaf(S[m + 1], x4.y, pa1);
                pa0 = fmaf(S[m + 2], x4.z, pa0); pa1 = fmaf(S[m + 3], x4.w, pa1);
                pc0 = fmaf(S[m], q4.x, pc0); pc1 = fmaf(S[m + 1], q4.y, pc1);
                pc0 = fmaf(S[m + 2], q4.z, pc0); pc1 = fmaf(S[m + 3], q4.w, pc1);
            }
            float pa = pa0 + pa1, pc = pc0 + pc1;
            pa += __shfl_xor_sync(0xffffffffu, pa, 1);
            pc += __shfl_xor_sync(0xffffffffu, pc, 1);
            pa += __shfl_xor_sync(0xffffffffu, pa, 2);
            pc += __shfl_xor_sync(0xffffffffu, pc, 2);

            float aj[WM], coef[WM];
            if constexpr (!INNER) {
                aj[0] = pa;
                if (p == 0) {
                    // no reads of the previous token: form the older pairs' reads
#pragma unroll
                    for (int j = 1; j < WM; ++j) {
                        float s = 0.f;
                        if (j < W) {
                            const float *xj = X + (rr - j) * LD + qr * QS;
#pragma unroll
                            for (int m = 0; m < RQ; ++m) s = fmaf(S[m], xj[m], s);
                            s += __shfl_xor_sync(0xffffffffu, s, 1);
                            s += __shfl_xor_sync(0xffffffffu, s, 2);
                        }
                        aj[j] = s;
                    }
                } else {
                    const float *mt = Mw + t * WM * WM;
#pragma unroll
                    for (int j = 1; j < WM; ++j) {
                        float s = 0.f;
                        if (j < W) {
                            s = gam_prev * a_prev[j - 1];
#pragma unroll
                            for (int jp = 0; jp < WM; ++jp)
                                if (jp < W) s = fmaf(mt[j * WM + jp], coef_prev[jp], s);
                        }
                        aj[j] = s;
                    }
                }
            }
#pragma unroll
            for (int j = 0; j < WM; ++j)
                coef[j] = j < W ? cc * (INNER ? vr[j] : vr[j] - aj[j]) : 0.f;

            if (qr == 0) {
                float ov = pc;   // read before the write
                if (!rbw) {
                    ov = gam * pc;
#pragma unroll
                    for (int j = 0; j < WM; ++j)
                        if (j < W) ov = fmaf(coef[j], E[t * WM + j], ov);
                }
                O[t * kCG + cl] = ov;
            }
            // the write: S = gamma S + sum_j x_{p-j} coef_j
#pragma unroll
            for (int m = 0; m < RQ; ++m) S[m] = fmaf(xa[m], coef[0], gam * S[m]);
#pragma unroll
            for (int j = 1; j < WM; ++j) {
                if (j < W) {
                    const float *xj = X + (rr - j) * LD + qr * QS;
                    const float cj = coef[j];
#pragma unroll
                    for (int m = 0; m < RQ; m += 4) {
                        const float4 x4 = load4(xj + m);
                        S[m] = fmaf(x4.x, cj, S[m]); S[m + 1] = fmaf(x4.y, cj, S[m + 1]);
                        S[m + 2] = fmaf(x4.z, cj, S[m + 2]); S[m + 3] = fmaf(x4.w, cj, S[m + 3]);
                    }
                }
            }
            if (p == T - 1 && a.oy && qr == 0) {
                // carried window out: slot s holds pair T-(W-1)+s = p - (W-2-s)
                for (int s = 0; s < W - 1; ++s) {
                    const int j = W - 2 - s;
                    float y = 0.f;
#pragma unroll
                    for (int jj = 0; jj < WM; ++jj)
                        if (jj == j) y = vr[jj];
                    a.oy[chain * cs + (int64_t)s * DK + col] = VAL[rr - j] != 0.f ? y : 0.f;
                }
            }
#pragma unroll
            for (int j = 0; j < WM; ++j) {
                if constexpr (!INNER) a_prev[j] = aj[j];
                coef_prev[j] = coef[j];
            }
            gam_prev = gam;
#pragma unroll
            for (int j = WM - 1; j >= 1; --j) vr[j] = vr[j - 1];
        }
        __syncthreads();
        for (int e = tid; e < nt * kCG; e += kThreads)
            og[(p0 + e / kCG) * DK + col0 + e % kCG] = from_f32<TIn>(O[e]);
        if (p0 + NB >= T && blockIdx.y == 0 && a.ox) {
            // carried window out, keys: pair T-(W-1)+s sits in row T-(W-1)+s-p0+WM
            for (int e = tid; e < (W - 1) * DK; e += kThreads) {
                const int s = e / DK, i = e % DK;
                const int r = (int)(T - (W - 1) + s - p0) + WM;
                a.ox[chain * cs + e] = VAL[r] != 0.f ? X[r * LD + padded<RQ>(i)] : 0.f;
            }
            if (tid == 0) {
                int n = 0;
                for (int s = 0; s < W - 1; ++s) n += VAL[(int)(T - (W - 1) + s - p0) + WM] != 0.f;
                a.on[chain] = n;
            }
        }
    }

#pragma unroll
    for (int m = 0; m < RQ; ++m)
        a.S_T[chain * DK * DK + (int64_t)(qr * RQ + m) * DK + col] = S[m];
}

template <int DK, int WM, typename TIn, bool INNER>
cudaError_t launch_t(const WindowArgs &a, cudaStream_t s) {
    auto kern = window_prefill_kernel<DK, WM, TIn, INNER>;
    constexpr size_t bytes = WinLayout<DK, WM>::BYTES;
    static_assert(bytes <= 56 * 1024, "four CTAs per SM");
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)bytes);
    if (e != cudaSuccess) return e;
    dim3 grid((unsigned)a.n_chains, DK / kCG);
    kern<<<grid, kThreads, bytes, s>>>(a);
    return cudaGetLastError();
}

template <int DK, typename TIn>
cudaError_t launch_d(const WindowArgs &a, cudaStream_t s) {
    if (a.W <= 4)
        return a.inner ? launch_t<DK, 4, TIn, true>(a, s) : launch_t<DK, 4, TIn, false>(a, s);
    return a.inner ? launch_t<DK, 8, TIn, true>(a, s) : launch_t<DK, 8, TIn, false>(a, s);
}

}  // namespace

cudaError_t launch_window_prefill(const WindowArgs &a, cudaStream_t s) {
    if (a.d == 64)
        return a.dtype == FW_F32 ? launch_d<64, float>(a, s) : launch_d<64, __nv_bfloat16>(a, s);
    return a.dtype == FW_F32 ? launch_d<128, float>(a, s) : launch_d<128, __nv_bfloat16>(a, s);
}

}  // namespace fw
