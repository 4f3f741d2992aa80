// fw_recurrent.cu -- per-token SIMT evaluation of the recurrence (fp32 math).
//
// One thread block per (chain, group of value columns).  The value columns of
// the state evolve independently given x_t, eta_t and gamma_t (the write
// S_t = gamma_t S_{t-1} + eta_t x_t r_t^T acts column by column), so a warp
// owns JW columns outright and its 32 lanes split the key rows.  Per token a
// warp forms, in one batch of butterfly reductions over the key rows, the
// column sums a_j = S[:,j].x_t and c_j = S[:,j].q_t plus |x_t|^2 and x_t.q_t,
// then applies
//     r_j = y_j - a_j,  o_j = gamma c_j + eta r_j (x.q) = (S_t^T q_t)_j,
//     S[i][j] <- gamma S[i][j] + eta x_i r_j,
// i.e. the Falcon-1 write of "Fast Weight Attention for Continual Learning"
// paper reading §3.2/§4.2 on the pair (phi(k_{t-1}), v_t) with x_1 = 0,
// eta_1 = 0 (§4.1) and the read after the write (§1.4).  Falcon-1A (§4.3)
// drops the residual (r = y); Falcon-2 / 2A (§4.2) take beta, and so eta and
// gamma, per value column; with FW_FLAG_SAME_PAIR the pair is
// (phi(k_t), v_t) for every token, and with FW_FLAG_RBW the read is taken
// before the write, o_j = c_j (the §3.3 read / pairing arms).
// Linear-attention mode uses x = phi(k_t), r = v_t, gamma = eta = 1 and reads
// with phi(q_t) ("Attention is also an FFN" blog §2.1).
//
// This kernel serves every shape and dtype (it is the fp32 path and the
// fallback of the chunked tensor-core kernel); the state never leaves
// registers between tokens.
#include "fw_internal.cuh"

namespace fw {
namespace {

constexpr int kJW = 8;     // value columns per warp
constexpr int kNWarp = 4;  // warps per block -> 32 columns per block

// CHAN: Falcon-2 / 2A, a step size per value column (a separate instantiation,
// so the scalar-step modes keep a single division per token).
template <int DK, typename TIn, bool CHAN>
__global__ void __launch_bounds__(kNWarp * 32)
recurrent_kernel(PrefillArgs a) {
    constexpr int RK = DK / 32;                // key rows per lane: i = lane + 32 r
    constexpr int NV = 2 * kJW + 2;            // values reduced per token
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int64_t chain = blockIdx.x;
    const int col0 = (blockIdx.y * kNWarp + warp) * kJW;
    const int64_t T = a.T;
    const bool falcon = (a.mode != FW_LINATTN);                     // eta, gamma, beta, lambda
    const bool resid = (a.mode == FW_FALCON1 || a.mode == FW_FALCON2);   // r = y - S^T x
    constexpr int NB = CHAN ? kJW : 1;                                  // betas per token
    const bool shifted = falcon && !(a.flags & FW_FLAG_SAME_PAIR);  // x_t = phi(k_{t-1})
    const bool rbw = (a.flags & FW_FLAG_RBW) != 0;

    const TIn *q = static_cast<const TIn *>(a.q) + chain * T * DK;
    const TIn *k = static_cast<const TIn *>(a.k) + chain * T * DK;
    const TIn *v = static_cast<const TIn *>(a.v) + chain * T * DK;
    const float *beta = falcon ? a.beta + chain * T * (CHAN ? DK : 1) : nullptr;
    const float *lam = falcon ? a.lam + chain * T : nullptr;
    TIn *o = static_cast<TIn *>(a.o) + chain * T * DK;

    float S[RK][kJW];
#pragma unroll
    for (int r = 0; r < RK; ++r)
#pragma unroll
        for (int c = 0; c < kJW; ++c)
            S[r][c] = a.S0 ? a.S0[chain * DK * DK + (int64_t)(lane + 32 * r) * DK + col0 + c]
                           : 0.f;

    // Pair key carried from the previous token (Falcon-1): x_1 = phi(k_init)
    // if a previous key is given, else 0 with eta_1 = 0.
    float xprev[RK];
    bool have_prev = false;
    if (shifted && a.k_init) {
        const TIn *ki = static_cast<const TIn *>(a.k_init) + chain * DK;
#pragma unroll
        for (int r = 0; r < RK; ++r) xprev[r] = apply_phi(a.phi, to_f32(ki[lane + 32 * r]));
        have_prev = true;
    } else {
#pragma unroll
        for (int r = 0; r < RK; ++r) xprev[r] = 0.f;
    }

    // Register prefetch of the next token's inputs.
    float nq[RK], nk[RK], nv[kJW], nb[NB], nl = 0.f;
    auto load = [&](int64_t t) {
#pragma unroll
        for (int r = 0; r < RK; ++r) {
            nq[r] = to_f32(q[t * DK + lane + 32 * r]);
            nk[r] = to_f32(k[t * DK + lane + 32 * r]);
        }
#pragma unroll
        for (int c = 0; c < kJW; ++c) nv[c] = to_f32(v[t * DK + col0 + c]);
        if (falcon) {
#pragma unroll
            for (int c = 0; c < NB; ++c) nb[c] = CHAN ? beta[t * DK + col0 + c] : beta[t];
            nl = lam[t];
        }
    };
    if (T > 0) load(0);

    for (int64_t t = 0; t < T; ++t) {
        float qv[RK], kt[RK], vv[kJW], bt[NB];
        const float lt = nl;
#pragma unroll
        for (int c = 0; c < NB; ++c) bt[c] = nb[c];
#pragma unroll
        for (int r = 0; r < RK; ++r) { qv[r] = nq[r]; kt[r] = apply_phi(a.phi, nk[r]); }
#pragma unroll
        for (int c = 0; c < kJW; ++c) vv[c] = nv[c];
        if (t + 1 < T) load(t + 1);

        float xs[RK];
#pragma unroll
        for (int r = 0; r < RK; ++r) {
            xs[r] = shifted ? xprev[r] : kt[r];
            if (!falcon) qv[r] = apply_phi(a.phi, qv[r]);
        }

        float red[NV];
#pragma unroll
        for (int c = 0; c < kJW; ++c) {
            float sa = 0.f, sc = 0.f;
#pragma unroll
            for (int r = 0; r < RK; ++r) { sa = fmaf(S[r][c], xs[r], sa); sc = fmaf(S[r][c], qv[r], sc); }
            red[2 * c] = sa;
            red[2 * c + 1] = sc;
        }
        {
            float n = 0.f, xq = 0.f;
#pragma unroll
            for (int r = 0; r < RK; ++r) { n = fmaf(xs[r], xs[r], n); xq = fmaf(xs[r], qv[r], xq); }
            red[2 * kJW] = n;
            red[2 * kJW + 1] = xq;
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1)
#pragma unroll
            for (int i = 0; i < NV; ++i) red[i] += __shfl_xor_sync(0xffffffffu, red[i], off);

        const bool pair = !shifted || (t > 0) || have_prev;
        float eta0 = 1.f, gam0 = 1.f;   // one step size per token (Falcon-2: per column below)
        if (falcon && !CHAN) {
            eta0 = pair ? bt[0] / (red[2 * kJW] + lt + a.eps) : 0.f;
            gam0 = 1.f - eta0 * lt;
        }
        const float xq = red[2 * kJW + 1];
        float outv = 0.f;
#pragma unroll
        for (int c = 0; c < kJW; ++c) {
            float eta = eta0, gam = gam0;
            if constexpr (CHAN) {
                eta = pair ? bt[c] / (red[2 * kJW] + lt + a.eps) : 0.f;
                gam = 1.f - eta * lt;
            }
            const float rc = resid ? vv[c] - red[2 * c] : vv[c];
            const float oc = rbw ? red[2 * c + 1] : fmaf(gam, red[2 * c + 1], eta * rc * xq);
            if (lane == c) outv = oc;
#pragma unroll
            for (int r = 0; r < RK; ++r) S[r][c] = fmaf(gam, S[r][c], (eta * xs[r]) * rc);
        }
        if (lane < kJW) o[t * DK + col0 + lane] = from_f32<TIn>(outv);
        if (shifted) {
#pragma unroll
            for (int r = 0; r < RK; ++r) xprev[r] = kt[r];
        }
    }

#pragma unroll
    for (int r = 0; r < RK; ++r)
#pragma unroll
        for (int c = 0; c < kJW; ++c)
            a.S_T[chain * DK * DK + (int64_t)(lane + 32 * r) * DK + col0 + c] = S[r][c];
}

template <int DK, typename TIn>
cudaError_t launch_t(const PrefillArgs &a, cudaStream_t s) {
    dim3 grid((unsigned)a.n_chains, DK / (kJW * kNWarp));
    if (a.mode == FW_FALCON2 || a.mode == FW_FALCON2A)
        recurrent_kernel<DK, TIn, true><<<grid, kNWarp * 32, 0, s>>>(a);
    else
        recurrent_kernel<DK, TIn, false><<<grid, kNWarp * 32, 0, s>>>(a);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_recurrent(const PrefillArgs &a, cudaStream_t s) {
    if (a.d == 64)
        return a.dtype == FW_F32 ? launch_t<64, float>(a, s) : launch_t<64, __nv_bfloat16>(a, s);
    return a.dtype == FW_F32 ? launch_t<128, float>(a, s) : launch_t<128, __nv_bfloat16>(a, s);
}

}  // namespace fw
