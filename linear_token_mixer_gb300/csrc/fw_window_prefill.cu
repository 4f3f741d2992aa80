// fw_window_prefill.cu -- Falcon-3 / 3A (and Falcon-2 / 2A) prefill, one token
// at a time (fp32).
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
// Work split.  One CTA per chain.  The value columns are independent given
// the window's keys and step sizes: a compute thread holds CPT value columns
// over a slice of the key rows (4 columns x 16 rows at d = 128 for windows up
// to 4 pairs), and the state never leaves registers.  Per token, the
// row-slice lanes of a column group reduce-scatter their partial reads, one
// lane per column runs that column's scalar work, and the write coefficients
// are broadcast back for the rank-W write.  Four producer warps work a block
// of 32 tokens ahead: they bulk-copy the block's keys (with the W pairs
// before it), queries and targets, stage them in shared memory, and form
// everything that depends on keys alone -- the dot products x_a . x_b of
// pairs up to W apart, q_t . x_{t-j}, each token's window Gram matrix and its
// largest eigenvalue, eta_t, gamma_t and c_t -- into the other of two
// buffers.  Buffers change hands through mbarriers whose waits are bounded.
// With a window of one pair and beta per value column (CHAN) the same kernel
// serves Falcon-2 / 2A, the page's per-channel step (§4.2).
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
// Per token and column this leaves two length-d_k reads and the rank-W write,
// issued as packed two-wide fp32 FMAs.  Before the call's first token the
// reads of the pairs already in its window are formed directly (S0^T x), and
// the recursion starts from them with gamma = 1 and no previous write.
#include "fw_window.cuh"
#include "fw_sm100.cuh"

namespace fw {
namespace {

using namespace sm100;

constexpr int kNB = 32;          // tokens per staged block
constexpr int kProducers = 128;  // producer threads (four warps, one per SM sub-partition)
constexpr int kBarProd = 1;      // named barrier of the producer warps

template <int DK, int WM, bool CHAN = false>
struct WinLayout {
    static constexpr int NB = kNB;
    // compute threads: CPT value columns x RPT key rows each; the RG threads
    // of a column group split the key rows.  Four columns per thread halve
    // the shared-memory reads per FMA; a window of up to 8 pairs keeps two,
    // for registers.
    static constexpr int CPT = WM <= 4 ? 4 : 2;
    static constexpr int RG = WM <= 4 ? 8 : 4;
    static constexpr int RPT = DK / RG;
    static constexpr int NCT = (DK / CPT) * RG;
    static constexpr int RQ = RPT;                  // key rows per compute thread
    static constexpr int QS = RQ + 4;               // padded row group: the groups
                                                    // start in different banks
    static constexpr int LD = RG * QS;              // padded row
    static constexpr int NXR = NB + WM;             // key rows: pairs p0-WM .. p0+NB-1
    // one buffer, offsets in floats
    static constexpr int X = 0;
    static constexpr int Q = X + NXR * LD;
    static constexpr int V = Q + NB * LD;            // [NXR][DK] targets, rows as X
    static constexpr int E = V + NXR * DK;           // [NB][WM]  q_t . x_{t-j}
    static constexpr int M = E + NB * WM;            // [NB][WM][WM] recursion weights
    static constexpr int GAM = M + NB * WM * WM;     // [NB] gamma_t
    static constexpr int CC = GAM + NB;              // [NB] c_t = eta_t / B_t
    static constexpr int VAL = CC + NB;              // [NXR] 1 if the pair exists
    static constexpr int BETA = (VAL + NXR + 3) / 4 * 4;   // per-column steps: [NB][DK]
    static constexpr int BUF = BETA + (CHAN ? NB * DK : 0);
    // producer scratch and barriers after the two buffers
    static constexpr int DOT = 2 * BUF;              // [NXR][WM] x_r . x_{r-delta}
    static constexpr int BL = DOT + NXR * WM;        // [NB][2] beta, lambda
    static constexpr int BARS = (BL + 2 * NB + 3) / 4 * 4;   // 5 mbarriers
    // raw input rows as loaded (element type TIn): keys of the block's pairs,
    // its queries, the targets of its pairs
    static constexpr int RAW = BARS + 16;
    template <typename TIn>
    static constexpr size_t raw_bytes() { return (size_t)(2 * NXR + NB) * DK * sizeof(TIn); }
    template <typename TIn>
    static constexpr size_t bytes() { return (size_t)RAW * sizeof(float) + raw_bytes<TIn>(); }
};

// Position of key element i in a padded row (groups of RQ elements, each
// followed by four floats of padding).
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

__device__ __forceinline__ float2 f2(float a, float b) { return make_float2(a, b); }

// N consecutive floats (N = 2 or 4, 8- or 16-byte aligned).
template <int N>
__device__ __forceinline__ void load_n(const float *p, float (&v)[N]) {
    if constexpr (N == 4) {
        const float4 u = *reinterpret_cast<const float4 *>(p);
        v[0] = u.x; v[1] = u.y; v[2] = u.z; v[3] = u.w;
    } else {
        const float2 u = *reinterpret_cast<const float2 *>(p);
        v[0] = u.x; v[1] = u.y;
    }
}
template <int N>
__device__ __forceinline__ void store_n(float *p, const float (&v)[N]) {
    if constexpr (N == 4) *reinterpret_cast<float4 *>(p) = make_float4(v[0], v[1], v[2], v[3]);
    else *reinterpret_cast<float2 *>(p) = make_float2(v[0], v[1]);
}
template <int N>
__device__ __forceinline__ void store_n(__nv_bfloat16 *p, const float (&v)[N]) {
    __nv_bfloat162 *q = reinterpret_cast<__nv_bfloat162 *>(p);
    q[0] = __floats2bfloat162_rn(v[0], v[1]);
    if constexpr (N == 4) q[1] = __floats2bfloat162_rn(v[2], v[3]);
}

template <int DK, int WM, typename TIn, bool INNER, bool CHAN>
__global__ void __launch_bounds__(WinLayout<DK, WM, CHAN>::NCT + kProducers, 1)
window_prefill_kernel(WindowArgs a) {
    using L = WinLayout<DK, WM, CHAN>;
    constexpr int NB = L::NB, RQ = L::RQ, QS = L::QS, LD = L::LD, NXR = L::NXR;
    constexpr int CPT = L::CPT, RG = L::RG, NCT = L::NCT;
    constexpr int NCW = NCT / 32;        // compute warps
    static_assert(2 * CPT == RG, "one reduced value per row-group lane");
    constexpr int NPT = kProducers;      // producer threads
    extern __shared__ __align__(16) float sm[];
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + L::BARS);
    const uint32_t full0 = smem_u32(bars), empty0 = smem_u32(bars + 2), rawbar = smem_u32(bars + 4);

    const int tid = threadIdx.x, lane = tid & 31;
    const int64_t chain = blockIdx.x;
    const int W = a.W;
    const int64_t T = a.T;
    const int64_t nblk = (T + NB - 1) / NB;
    const uint64_t limit = (uint64_t)a.wait_ns;
    const int64_t cs = (int64_t)(W - 1) * DK;   // carried window, per chain
    int cn = a.cn ? a.cn[chain] : 0;
    cn = cn < 0 ? 0 : (cn > W - 1 ? W - 1 : cn);

    if (tid == 0) {
        mbar_init(full0, 1);
        mbar_init(full0 + 8, 1);
        mbar_init(empty0, NCW);
        mbar_init(empty0 + 8, NCW);
        mbar_init(rawbar, 1);
        fence_mbar_init();
    }
    __syncthreads();

    if (tid >= NCT) {
        // ================= producer warps =================
        const int pt = tid - NCT;   // producer thread 0 .. NPT-1
        const bool same = (a.flags & FW_FLAG_SAME_PAIR) != 0;
        const TIn *qg = static_cast<const TIn *>(a.q) + chain * T * DK;
        const TIn *kg = static_cast<const TIn *>(a.k) + chain * T * DK;
        const TIn *vg = static_cast<const TIn *>(a.v) + chain * T * DK;
        const TIn *ki = a.k_init ? static_cast<const TIn *>(a.k_init) + chain * DK : nullptr;
        const float *cx = a.cx ? a.cx + chain * cs : nullptr;
        const float *cy = a.cy ? a.cy + chain * cs : nullptr;
        float *DOT = sm + L::DOT, *BL = sm + L::BL;
        constexpr uint32_t ROWB = DK * sizeof(TIn);
        const int sh = same ? 0 : 1;   // pair m holds key m - sh
        const TIn *rawK = reinterpret_cast<const TIn *>(sm + L::RAW);
        const TIn *rawQ = rawK + NXR * DK, *rawV = rawQ + NB * DK;
        const uint32_t rawK_s = smem_u32(rawK), rawQ_s = smem_u32(rawQ), rawV_s = smem_u32(rawV);
        // bulk copies of block kb's rows that lie inside the sequence: keys
        // (row r <-> key p0 - WM - sh + r), queries, targets (row r <-> pair p0 - WM + r)
        auto issue = [&](int64_t kb) {
            const int64_t p0 = kb * NB;
            const int64_t nt = T - p0 < NB ? T - p0 : NB;
            const int64_t kbase = p0 - WM - sh, vbase = p0 - WM;
            const int64_t klo = kbase > 0 ? kbase : 0, vlo = vbase > 0 ? vbase : 0;
            const int64_t khi = p0 + NB - 1 - sh < T - 1 ? p0 + NB - 1 - sh : T - 1;
            const int64_t vhi = p0 + NB - 1 < T - 1 ? p0 + NB - 1 : T - 1;
            const uint32_t nk = khi >= klo ? (uint32_t)(khi - klo + 1) : 0u;
            const uint32_t nv = vhi >= vlo ? (uint32_t)(vhi - vlo + 1) : 0u;
            mbar_expect_tx(rawbar, (nk + (uint32_t)nt + nv) * ROWB);
            if (nk) bulk_g2s(rawK_s + (uint32_t)(klo - kbase) * ROWB, kg + klo * DK, nk * ROWB, rawbar);
            bulk_g2s(rawQ_s, qg + p0 * DK, (uint32_t)nt * ROWB, rawbar);
            if (nv) bulk_g2s(rawV_s + (uint32_t)(vlo - vbase) * ROWB, vg + vlo * DK, nv * ROWB, rawbar);
        };
        if (pt == 0) issue(0);
        for (int64_t kb = 0; kb < nblk; ++kb) {
            const int b = (int)(kb & 1);
            float *X = sm + b * L::BUF + L::X, *Qs = sm + b * L::BUF + L::Q,
                  *V = sm + b * L::BUF + L::V, *E = sm + b * L::BUF + L::E,
                  *Mw = sm + b * L::BUF + L::M, *GAM = sm + b * L::BUF + L::GAM,
                  *CC = sm + b * L::BUF + L::CC, *VAL = sm + b * L::BUF + L::VAL;
            const int64_t p0 = kb * NB;
            const int nt = (int)(T - p0 < NB ? T - p0 : NB);
            const float bt_l = !CHAN && pt < nt ? a.beta[chain * T + p0 + pt] : 0.f;
            const float lt_l = pt < nt ? a.lam[chain * T + p0 + pt] : 0.f;
            // this block's raw rows (then no copy is in flight), then its
            // buffer; the producer warps agree on the outcome before leaving
            const bool late = !mbar_wait(rawbar, (uint32_t)(kb & 1), limit) ||
                              (kb >= 2 && !mbar_wait(empty0 + 8 * b,
                                                     (uint32_t)(((kb >> 1) + 1) & 1), limit));
            if (bar_or(kBarProd, NPT, late)) {
                if (pt == 0) atomicExch(a.err, kDevErrTimeout);
                return;
            }
            if constexpr (CHAN) {
                // per-column step sizes of the block's tokens, beta[p][j]
                float *BT = sm + b * L::BUF + L::BETA;
                const float *bg = a.beta + (chain * T + p0) * DK;
#pragma unroll 8
                for (int e = pt; e < NB * (DK / 4); e += NPT) {
                    const int t = e / (DK / 4), i4 = (e % (DK / 4)) * 4;
                    *reinterpret_cast<float4 *>(BT + t * DK + i4) =
                        t < nt ? load4(bg + t * DK + i4) : make_float4(0.f, 0.f, 0.f, 0.f);
                }
            }
            // keys: row r holds pair m = p0 - WM + r, phi applied, 0 if it does not exist
#pragma unroll 4
            for (int e = pt; e < NXR * (DK / 4); e += NPT) {
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
                    const TIn *src = m - sh >= 0 ? rawK + r * DK : ki;
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
#pragma unroll 4
            for (int e = pt; e < NB * (DK / 4); e += NPT) {
                const int t = e / (DK / 4), i4 = (e % (DK / 4)) * 4;
                const float4 qv = t < nt ? load4(rawQ + t * DK + i4) : make_float4(0.f, 0.f, 0.f, 0.f);
                *reinterpret_cast<float4 *>(Qs + t * LD + padded<RQ>(i4)) = qv;
            }
            // targets: row r holds the target of pair m = p0 - WM + r (v_m; the
            // carried y for m < 0), 0 where the pair does not exist
#pragma unroll 4
            for (int e = pt; e < NXR * (DK / 4); e += NPT) {
                const int r = e / (DK / 4), i4 = (e % (DK / 4)) * 4;
                const int64_t m = p0 - WM + r;
                float4 vv = make_float4(0.f, 0.f, 0.f, 0.f);
                if (m < 0) {
                    const int64_t s = m + W - 1;
                    if (cy && s >= 0 && s >= W - 1 - cn) vv = load4(cy + s * DK + i4);
                } else if (m < T) {
                    vv = load4(rawV + r * DK + i4);
                }
                *reinterpret_cast<float4 *>(V + r * DK + i4) = vv;
            }
            if (pt < NB) {
                BL[2 * pt] = bt_l;
                BL[2 * pt + 1] = lt_l;
            }
            // the raw rows are read out: prefetch the next block's behind the
            // rest of this block's work
            bar_sync(kBarProd, NPT);
            if (pt == 0 && kb + 1 < nblk) {
                fence_proxy_async();
                issue(kb + 1);
            }
            // dot products of keys up to W-1 pairs apart (DOT, rows as X) and of
            // the queries with their window's keys (E): one product per lane at
            // a time, each lane starting at its own offset along d_k so that the
            // lanes' loads spread over the banks.  The first WM rows repeat the
            // previous block's last WM rows: their products are copied.
            const int r0 = kb == 0 ? 0 : WM;
            if (kb > 0) {
                for (int e = pt; e < WM * WM; e += NPT) DOT[e] = DOT[NB * WM + e];
                bar_sync(kBarProd, NPT);
            }
            for (int it = r0 * WM + pt; it < (NXR + NB) * WM; it += NPT) {
                const int r = it / WM, dl = it - r * WM;
                const float *u = r < NXR ? X + r * LD : Qs + (r - NXR) * LD;
                const int top = r < NXR ? r : r - NXR + WM;   // row of the newest key paired with u
                float s = 0.f;   // 0 outside the window: the compute threads sum over WM slots
                if (dl < W && top - dl >= 0) {
                    const float *w = X + (top - dl) * LD;
                    float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f;
#pragma unroll 8
                    for (int k = 0; k < DK / 4; ++k) {
                        const int i = padded<RQ>(((k + pt) & (DK / 4 - 1)) * 4);
                        const float4 x = load4(u + i), y = load4(w + i);
                        s0 = fmaf(x.x, y.x, s0); s1 = fmaf(x.y, y.y, s1);
                        s2 = fmaf(x.z, y.z, s2); s3 = fmaf(x.w, y.w, s3);
                    }
                    s = (s0 + s1) + (s2 + s3);
                }
                if (r < NXR) DOT[r * WM + dl] = s;
                else E[(r - NXR) * WM + dl] = s;
            }
            bar_sync(kBarProd, NPT);
            // step size of every token of the block (one in every four producer
            // threads: eight per warp), and the weights of the residual-read
            // recursion, M[t][j][j'] = x_{p-1-j'} . x_{p-j}
            if ((pt & 3) == 0 && (pt >> 2) < nt) {
                const int t = pt >> 2, rr = t + WM;   // row of pair p
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
                const float bt = BL[2 * t], lt = BL[2 * t + 1];
                if constexpr (CHAN) {
                    // a step per value column (W = 1, mu = |x|^2): the compute
                    // threads take eta_j = beta_j / (|x|^2 + lambda + eps) from
                    // lambda and the reciprocal denominator
                    GAM[t] = lt;
                    CC[t] = nb > 0 ? 1.f / (G[0][0] + lt + a.eps) : 0.f;
                } else {
                    float eta = 0.f;
                    if (nb > 0) {
                        const float mu = window_max_eig<WM>(G) / (float)nb;
                        eta = bt / (mu + lt + a.eps);
                    }
                    GAM[t] = 1.f - eta * lt;
                    CC[t] = nb > 0 ? eta / (float)nb : 0.f;
                }
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
            bar_sync(kBarProd, NPT);
            if (pt == 0) mbar_arrive(full0 + 8 * b);
            if (kb == nblk - 1 && a.ox) {
                // carried window out, keys: pair T-(W-1)+s sits in row T-(W-1)+s-p0+WM
                for (int e = pt; e < (W - 1) * DK; e += NPT) {
                    const int s = e / DK, i = e % DK;
                    const int r = (int)(T - (W - 1) + s - p0) + WM;
                    const bool held = VAL[r] != 0.f;
                    a.ox[chain * cs + e] = held ? X[r * LD + padded<RQ>(i)] : 0.f;
                    a.oy[chain * cs + e] = held ? V[r * DK + i] : 0.f;
                }
                if (pt == 0) {
                    int n = 0;
                    for (int s = 0; s < W - 1; ++s)
                        n += VAL[(int)(T - (W - 1) + s - p0) + WM] != 0.f;
                    a.on[chain] = n;
                }
            }
        }
        return;
    }

    // ================= compute threads =================
    // thread = (column group, row group rg): columns c0 .. c0 + CPT - 1, key
    // rows rg*RQ .. rg*RQ + RQ - 1, held as pairs of rows so that a float4 of
    // keys feeds two packed FMAs per column
    const int rg = tid % RG, c0 = (tid / RG) * CPT;
    const bool rbw = (a.flags & FW_FLAG_RBW) != 0;
    TIn *og = static_cast<TIn *>(a.o) + chain * T * DK;

    float2 S[CPT][RQ / 2];   // S[c][i] = rows rg*RQ + 2i, 2i + 1 of column c0 + c
#pragma unroll
    for (int m = 0; m < RQ; m += 2) {
        float r0[CPT], r1[CPT];
        if (a.S0) {
            const float *s0 = a.S0 + chain * DK * DK + (int64_t)(rg * RQ + m) * DK + c0;
            load_n<CPT>(s0, r0);
            load_n<CPT>(s0 + DK, r1);
        } else {
#pragma unroll
            for (int c = 0; c < CPT; ++c) r0[c] = r1[c] = 0.f;
        }
#pragma unroll
        for (int c = 0; c < CPT; ++c) S[c][m / 2] = f2(r0[c], r1[c]);
    }

    // lane rg < CPT of a column group keeps column c0 + rg's previous-token
    // reads of its window's pairs and its write coefficients
    float a_prev[WM], coef_prev[WM];
#pragma unroll
    for (int j = 0; j < WM; ++j) {
        a_prev[j] = 0.f;
        coef_prev[j] = 0.f;
    }
    float gam_prev = 1.f;

    for (int64_t kb = 0; kb < nblk; ++kb) {
        const int b = (int)(kb & 1);
        const float *X = sm + b * L::BUF + L::X, *Qs = sm + b * L::BUF + L::Q,
                    *V = sm + b * L::BUF + L::V, *E = sm + b * L::BUF + L::E,
                    *Mw = sm + b * L::BUF + L::M, *GAM = sm + b * L::BUF + L::GAM,
                    *CC = sm + b * L::BUF + L::CC;
        const int64_t p0 = kb * NB;
        const int nt = (int)(T - p0 < NB ? T - p0 : NB);
        if (!mbar_wait(full0 + 8 * b, (uint32_t)((kb >> 1) & 1), limit)) {
            atomicExch(a.err, kDevErrTimeout);
            return;
        }
        if (!INNER && kb == 0) {
            // the first token has no previous reads: form S0^T x of the pairs
            // before it (rows WM-j), so that the recursion starts from them with
            // gamma = 1 and no previous write
#pragma unroll
            for (int j = 1; j < WM; ++j) {
                if (j >= W) continue;   // (compile-time j keeps a_prev in registers)
                const float *xj = X + (WM - j) * LD + rg * QS;
                float2 acc[CPT];
#pragma unroll
                for (int c = 0; c < CPT; ++c) acc[c] = f2(0.f, 0.f);
#pragma unroll
                for (int m = 0; m < RQ; m += 4) {
                    const float4 x4 = load4(xj + m);
#pragma unroll
                    for (int c = 0; c < CPT; ++c) {
                        acc[c] = __ffma2_rn(S[c][m / 2], f2(x4.x, x4.y), acc[c]);
                        acc[c] = __ffma2_rn(S[c][m / 2 + 1], f2(x4.z, x4.w), acc[c]);
                    }
                }
#pragma unroll
                for (int c = 0; c < CPT; ++c) {
                    float r = acc[c].x + acc[c].y;
#pragma unroll
                    for (int off = 1; off < RG; off <<= 1) r += __shfl_xor_sync(0xffffffffu, r, off);
                    if (c == rg) a_prev[j - 1] = r;   // lane rg < CPT keeps column c0 + rg
                }
            }
        }
        for (int t = 0; t < nt; ++t) {
            const int64_t p = p0 + t;
            const int rr = t + WM;
            const float gam = GAM[t], cc = CC[t];
            const float *xp = X + rr * LD + rg * QS, *qp = Qs + t * LD + rg * QS;
            float2 pa[CPT], pc[CPT];
#pragma unroll
            for (int c = 0; c < CPT; ++c) pa[c] = pc[c] = f2(0.f, 0.f);
#pragma unroll
            for (int m = 0; m < RQ; m += 4) {
                const float4 q4 = load4(qp + m);
                if constexpr (!INNER) {
                    const float4 x4 = load4(xp + m);
#pragma unroll
                    for (int c = 0; c < CPT; ++c) {
                        pa[c] = __ffma2_rn(S[c][m / 2], f2(x4.x, x4.y), pa[c]);
                        pa[c] = __ffma2_rn(S[c][m / 2 + 1], f2(x4.z, x4.w), pa[c]);
                    }
                }
#pragma unroll
                for (int c = 0; c < CPT; ++c) {
                    pc[c] = __ffma2_rn(S[c][m / 2], f2(q4.x, q4.y), pc[c]);
                    pc[c] = __ffma2_rn(S[c][m / 2 + 1], f2(q4.z, q4.w), pc[c]);
                }
            }
            // reduce-scatter over the RG row-group lanes of the column group:
            // values 0 .. CPT-1 are the new pair's reads of the CPT columns,
            // CPT .. 2 CPT-1 the query's; lane rg ends with the whole of value rg
            float v[2 * CPT];
#pragma unroll
            for (int c = 0; c < CPT; ++c) {
                v[c] = INNER ? 0.f : pa[c].x + pa[c].y;
                v[CPT + c] = pc[c].x + pc[c].y;
            }
#pragma unroll
            for (int h = RG / 2; h >= 1; h >>= 1) {
                const bool up = (rg & h) != 0;
#pragma unroll
                for (int i = 0; i < h; ++i) {
                    const float send = up ? v[i] : v[i + h];
                    const float keep = up ? v[i + h] : v[i];
                    v[i] = keep + __shfl_xor_sync(0xffffffffu, send, h);
                }
            }
            // lane rg < CPT serves column c0 + rg; its query read sits on lane rg + CPT
            const float rcv = __shfl_xor_sync(0xffffffffu, v[0], CPT);
            float coef_m[WM];
#pragma unroll
            for (int j = 0; j < WM; ++j) coef_m[j] = 0.f;
            float gcol = gam;   // this lane's column: decay, and write coefficient scale
            if (rg < CPT) {
                const int col = c0 + rg;
                const float *mt = Mw + t * WM * WM;
                float ccol = cc;
                if constexpr (CHAN) {   // GAM holds lambda, CC the reciprocal denominator
                    ccol = sm[b * L::BUF + L::BETA + t * DK + col] * cc;
                    gcol = 1.f - ccol * gam;
                }
                // the reads of the older pairs by recursion (descending j, so
                // that a_prev is replaced in place after its last use), the
                // residuals and the write coefficients
#pragma unroll
                for (int j = WM - 1; j >= 0; --j) {
                    const bool in = j < W;   // slot j of the window (else coefficient 0)
                    const float y = V[(rr - j) * DK + col];   // target of pair p - j
                    float aj = 0.f;
                    if constexpr (!INNER) {
                        if (j == 0) {
                            aj = v[0];
                        } else {
                            // M and the previous coefficients are 0 outside the window
                            aj = gam_prev * a_prev[j - 1];
#pragma unroll
                            for (int jp = 0; jp < WM; ++jp)
                                aj = fmaf(mt[j * WM + jp], coef_prev[jp], aj);
                        }
                        a_prev[j] = in ? aj : 0.f;
                    }
                    coef_m[j] = in ? ccol * (y - aj) : 0.f;
                }
                float ov = rcv;   // read before the write
                if (!rbw) {
                    ov *= gcol;
#pragma unroll
                    for (int j = 0; j < WM; ++j) ov = fmaf(coef_m[j], E[t * WM + j], ov);
                }
                og[p * DK + col] = from_f32<TIn>(ov);
#pragma unroll
                for (int j = 0; j < WM; ++j) coef_prev[j] = coef_m[j];
            }
            // every lane of the group takes the coefficients of all CPT columns
            float coef[CPT][WM];
            {
                const int gbase = lane & ~(RG - 1);
#pragma unroll
                for (int c = 0; c < CPT; ++c)
#pragma unroll
                    for (int j = 0; j < WM; ++j)
                        coef[c][j] = __shfl_sync(0xffffffffu, coef_m[j], gbase + c);
            }
            // the write: S = gamma S + sum_j x_{p-j} coef_j (gamma per column with CHAN)
            {
#pragma unroll
                for (int c = 0; c < CPT; ++c) {
                    const float gc = CHAN ? __shfl_sync(0xffffffffu, gcol, (lane & ~(RG - 1)) + c)
                                          : gam;
                    const float2 g2 = f2(gc, gc);
#pragma unroll
                    for (int i = 0; i < RQ / 2; ++i) S[c][i] = __fmul2_rn(S[c][i], g2);
                }
                const float *x0 = X + rr * LD + rg * QS;
#pragma unroll
                for (int m = 0; m < RQ; m += 4) {
#pragma unroll
                    for (int j = 0; j < WM; ++j) {   // slots outside the window add 0
                        const float4 x4 = load4(x0 - j * LD + m);
                        const float2 lo = f2(x4.x, x4.y), hi = f2(x4.z, x4.w);
#pragma unroll
                        for (int c = 0; c < CPT; ++c) {
                            const float2 cf = f2(coef[c][j], coef[c][j]);
                            S[c][m / 2] = __ffma2_rn(lo, cf, S[c][m / 2]);
                            S[c][m / 2 + 1] = __ffma2_rn(hi, cf, S[c][m / 2 + 1]);
                        }
                    }
                }
            }
            gam_prev = gam;
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(empty0 + 8 * b);
    }

#pragma unroll
    for (int m = 0; m < RQ; m += 2) {
        float r0[CPT], r1[CPT];
#pragma unroll
        for (int c = 0; c < CPT; ++c) {
            r0[c] = S[c][m / 2].x;
            r1[c] = S[c][m / 2].y;
        }
        float *s0 = a.S_T + chain * DK * DK + (int64_t)(rg * RQ + m) * DK + c0;
        store_n<CPT>(s0, r0);
        store_n<CPT>(s0 + DK, r1);
    }
}

template <int DK, int WM, typename TIn, bool INNER, bool CHAN = false>
cudaError_t launch_t(const WindowArgs &a, cudaStream_t s) {
    auto kern = window_prefill_kernel<DK, WM, TIn, INNER, CHAN>;
    constexpr size_t bytes = WinLayout<DK, WM, CHAN>::template bytes<TIn>();
    static_assert(bytes <= 227 * 1024, "shared memory of one CTA");
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)bytes);
    if (e != cudaSuccess) return e;
    kern<<<(unsigned)a.n_chains, WinLayout<DK, WM, CHAN>::NCT + kProducers, bytes, s>>>(a);
    return cudaGetLastError();
}

// The window's slots are compile-time (WM = 1, 2, 4 or 8 >= W); slots past W
// carry zero coefficients.
template <int DK, typename TIn>
cudaError_t launch_d(const WindowArgs &a, cudaStream_t s) {
    if (a.W == 1)
        return a.chan ? (a.inner ? launch_t<DK, 1, TIn, true, true>(a, s)
                                 : launch_t<DK, 1, TIn, false, true>(a, s))
                      : (a.inner ? launch_t<DK, 1, TIn, true>(a, s) : launch_t<DK, 1, TIn, false>(a, s));
    if (a.W == 2)
        return a.inner ? launch_t<DK, 2, TIn, true>(a, s) : launch_t<DK, 2, TIn, false>(a, s);
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
