// fw_chunked_chan.cu -- chunked prefill of the per-channel step (Falcon-2 /
// Falcon-2A) for bf16 inputs, d_k = d_v = 128.
//
// "Fast Weight Attention for Continual Learning" paper reading, §4.2: the
// squared error is separable by value dimension, so value channel j takes its
// own step eta_{t,j} = beta_{t,j} / (|x_t|^2 + lambda_t + eps), sharing the
// residual's feature x_t; §4.4: the chunk's Gram matrix is shared by every
// channel, and only the triangular system is modulated per channel.  Our chunk
// form, for one chunk (C = 64 tokens, chunk-local t, s) from state S0, channel j,
// with gamma_t = 1 - eta_t lambda_t, D[t,s] = prod_{i=s+1..t} gamma_i,
// G_t = prod_{i<=t} gamma_i, Gm_t = G_{t-1}, A = X X^T, B = Q X^T, U = X S0[:, j],
// V = Q S0[:, j]:
//   r_t = y_t - Gm_t U_t - sum_{s<t} D[t-1,s] eta_s A[t,s] r_s   (2A: r_t = y_t)
//   o_t = G_t V_t + sum_{s<=t} D[t,s] eta_s B[t,s] r_s
//         (read before the write: Gm_t V_t + sum_{s<t} D[t-1,s] eta_s B[t,s] r_s)
//   S_C[:, j] = G_{C-1} S0[:, j] + X^T (D[C-1, .] eta r).
// The shared matrix products run on tcgen05 (the Gram [X;Q] X^T; U^T = S^T X^T
// and V^T = S^T Q^T with the state transposed in tensor memory, one lane per
// value channel; the state update S^T += Rw^T X).  From the second chunk on, U
// and V do not wait for the state update: with S_{c+1} = diag(G_C) S_c +
// X_c^T Rw_c, U^T(c+1) = (diag(G_C) S_c)^T X_{c+1}^T + Rw_c^T (X_c X_{c+1}^T)
// (V with Q_{c+1}), from a bf16 copy of the pre-scaled state and the cross
// Gram [X_{c+1}; Q_{c+1}] X_c^T formed during chunk c.  Each channel's recurrence
// over the chunk is one thread: the sums over earlier tokens are block-factored
// over blocks of NB tokens, D[t-1, s] = P[t-1] (block totals between) Suf[s] for
// s in an earlier block, so with the weights zhat_s = eta_s r_s brought to the
// end of the last finished block, every cross-block sum is a row of A or B
// against zhat.  Those sums, for a block's eight rows and a warp's 32 channels,
// are one small product (channels x s)(s x tokens) on the warp's tf32 MMAs; the
// older blocks' weights take the previous block's decay on the way into it.
// Inside a block a direct product runs over at most NB - 1 tokens.  At the
// chunk's end zhat is D[C-1, s] eta_s r_s, the state update's weights.  No
// decay product is ever divided (gamma may be zero or negative).
//
// One CTA per chain:
//   warp 0      TMA producer: X (keys shifted one token unless the same-step
//               pair; the row before the sequence reads as zero) and Q tiles,
//               64 x 128 bf16, 128-byte swizzle, in a two-stage ring; the V
//               tile; the chunk's beta rows (64 x 128 fp32, one bulk copy).
//   warp 1      MMA issuer: Gram, cross Gram, U^T / V^T, state update.
//   warp 2      tensor-memory allocation.
//   warps 4-7   staging group: the Gram tile from tensor memory to fp32 A and B
//               in shared memory, 1 / (|x_t|^2 + lambda_t + eps), the fp32
//               state pre-scaled by each channel's chunk decay with its bf16
//               copy, and the cross Gram as bf16 rows in the chunk's Q tile.
//   warps 8-11  channel group (thread j = value channel j = tensor-memory lane
//               j): gates, the recurrence above, the weights, S_T, and the
//               outputs, stored by each thread straight to global memory as
//               they are formed (the four warps write one 256-byte row per
//               token), so no chunk-end store or its wait is on the path.
// Every wait is bounded: on expiry the kernel records an error, the other roles
// stop at their next wait, copies and MMAs in flight are drained, tensor memory
// is freed and the kernel exits.
#include <cudaTypedefs.h>

#include <mutex>

#include "fw_internal.cuh"
#include "fw_sm100.cuh"

namespace fw {
namespace {
using namespace sm100;

constexpr int C = 64;          // chunk length
constexpr int D = 128;         // d_k = d_v
constexpr int NB = 8;          // block of the decay factorisation
constexpr int NTHREADS = 384;
constexpr int SG_W0 = 4, CG_W0 = 8;
constexpr int BAR_SGRP = 1, BAR_CGRP = 2;   // named barriers of the two groups
constexpr int GROUP = 128;
constexpr uint32_t KB = 1024;
constexpr int NST = 2;         // depth of the key/query tile ring

// shared memory (offsets from a 1024-aligned base)
constexpr uint32_t OFF_XQ = 0;             // NST stages of X0 Q0 X1 Q1 (8 KB each)
constexpr uint32_t XQ_X0 = 0, XQ_Q0 = 8 * KB, XQ_X1 = 16 * KB, XQ_Q1 = 24 * KB;
constexpr uint32_t OFF_Y = 64 * KB;        // V tile, two 64-column halves (128-byte swizzle)
constexpr uint32_t OFF_BETA = 80 * KB;     // beta rows of the chunk, fp32 [t][j]
constexpr int ABROW = 68;                  // row stride of A and B (64 + 4: conflict-free columns)
constexpr uint32_t OFF_A = 112 * KB;       // X X^T, fp32 [t][s]
constexpr uint32_t OFF_B = OFF_A + (uint32_t)C * ABROW * 4;   // Q X^T, fp32 [t][s]
constexpr uint32_t OFF_RT = 147 * KB;      // (weights * r)^T, bf16 rows j (K-major A operand)
constexpr uint32_t OFF_Z = OFF_RT + 16 * KB;     // zhat per channel, fp32 rows j of ZROW floats
constexpr int ZROW = 68;                   // 64 + 4 (16-byte groups spread over the banks)
constexpr int HTP = 36;                    // row stride of the H transposes (8 HTP = 8 mod 32: no conflicts)
constexpr uint32_t OFF_HT = OFF_Z + (uint32_t)D * ZROW * 4;    // per channel warp: H_A, H_B [8][HTP]
constexpr uint32_t OFF_VEC = OFF_HT + 4 * 2 * NB * HTP * 4;      // inv[64], lambda[64]
constexpr uint32_t OFF_BAR = OFF_VEC + 512;
constexpr uint32_t OFF_MISC = OFF_BAR + 32 * 8;
constexpr uint32_t SMEM_BYTES = OFF_MISC + 64;
constexpr uint32_t SMEM_ALLOC = SMEM_BYTES + 1024;
static_assert(SMEM_ALLOC <= 227 * KB, "shared memory budget");
static_assert(OFF_VEC % 16 == 0 && OFF_BAR % 8 == 0 && OFF_B + (uint32_t)C * ABROW * 4 <= OFF_RT,
              "alignment and layout");

enum {
    B_FULL0 = 0, B_EMPTY0 = B_FULL0 + NST, B_FULLY = B_EMPTY0 + NST, B_YFREE, B_FULLB, B_BFREE,
    B_GDONE, B_GFREE, B_ABRDY, B_ABFREE, B_SRDY, B_UVDONE, B_RRDY, B_SDONE, B_MDRAIN, B_NEVER,
    B_PATCH, B_SSCL, B_HDONE, B_HRDY, B_COUNT
};
static_assert(B_COUNT <= 32, "barrier area");

// tensor-memory columns (128 lanes x 32 bit); the state is held transposed
// (lane j), with a bf16 copy (two i per column), the A operand of U^T and V^T
constexpr uint32_t COL_G = 0, COL_U = 64, COL_V = 128, COL_SB = 192, COL_S = 256;
// [X_{c+1}; Q_{c+1}] X_c^T, the cross Gram that carries chunk c's state update into
// chunk c+1's U and V
constexpr uint32_t COL_H = 384;
constexpr uint32_t TMEM_COLS = 512;

constexpr uint64_t kDrainNs = 2000000000ull;

// Optional phase timestamps of CTA 0 (instrumented builds only).
#ifdef FW_TRACE
constexpr int kCTraceEv = 32, kCTraceChunks = 64;
__device__ unsigned long long g_ctrace[kCTraceChunks * kCTraceEv];
#define CTRACE(c, ev) \
    do { if (blockIdx.x == 0 && (c) < kCTraceChunks) g_ctrace[(c) * kCTraceEv + (ev)] = globaltimer(); } while (0)
#else
#define CTRACE(c, ev) do { } while (0)
#endif

__device__ __noinline__ bool cwait_slow(uint32_t bar, uint32_t parity, uint64_t limit,
                                        volatile int *abort_flag) {
    const uint64_t t0 = globaltimer();
    for (;;) {
        if (mbar_try_wait_sleep(bar, parity, 100000u)) return true;
        if (*abort_flag) return false;
        if (globaltimer() - t0 > limit) return false;
    }
}

// Bounded wait that also gives up as soon as another role has aborted.
__device__ __forceinline__ bool cwait(uint32_t bar, uint32_t parity, uint64_t limit,
                                      volatile int *abort_flag) {
    if (mbar_try_wait(bar, parity)) return true;
    return cwait_slow(bar, parity, limit, abort_flag);
}

__device__ __forceinline__ void st_row8(uint32_t addr, const float *v) {
    st_shared_v4(addr, pack_bf16(v[0], v[1]), pack_bf16(v[2], v[3]), pack_bf16(v[4], v[5]),
                 pack_bf16(v[6], v[7]));
}

// Eight consecutive columns of one lane, loaded and waited for.
// two 8-column loads, one wait (no memory clobber: tensor memory only)
__device__ __forceinline__ void tmem_ld8x2(uint32_t ta, uint32_t tb, float *va, float *vb) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%16];\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%8,%9,%10,%11,%12,%13,%14,%15}, [%17];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15])
        : "r"(ta), "r"(tb));
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        va[i] = __uint_as_float(r[i]);
        vb[i] = __uint_as_float(r[8 + i]);
    }
}

__device__ __forceinline__ void tmem_ld8(uint32_t taddr, float *v) {
    uint32_t r[8];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7])
        : "r"(taddr)
        : "memory");
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = __uint_as_float(r[i]);
}

template <bool INNER, bool RBW>
__global__ void __launch_bounds__(NTHREADS, 1)
chan_kernel(const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmk,
            const __grid_constant__ CUtensorMap tmv, const PrefillArgs a) {
    extern __shared__ uint8_t smem_raw[];
    // 1024-aligned base, derived from the shared array itself (shared-space loads)
    uint8_t *sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const uint32_t sb = smem_u32(sm);
    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int64_t chain = blockIdx.x;
    const int64_t T = a.T;
    const int nch = (int)((T + C - 1) / C);
    const bool shifted = !(a.flags & FW_FLAG_SAME_PAIR);   // x_t = phi(k_{t-1})
    constexpr bool rbw = RBW;                               // o_t = S_{t-1}^T q_t
    const uint64_t limit = (uint64_t)a.wait_ns;

    volatile int *s_abort = reinterpret_cast<volatile int *>(sm + OFF_MISC);
    volatile uint32_t *s_tmem = reinterpret_cast<volatile uint32_t *>(sm + OFF_MISC + 4);
    auto bar = [&](int i) -> uint32_t { return sb + OFF_BAR + 8u * (uint32_t)i; };
    auto xq = [&](int st) -> uint32_t { return sb + OFF_XQ + (uint32_t)st * 32u * KB; };
    float *inv = reinterpret_cast<float *>(sm + OFF_VEC);
    float *lamv = inv + 64;
    auto fail_now = [&]() {
        *s_abort = 1;
        atomicExch(a.err, kDevErrTimeout);
    };

    if (tid == 0) {
        for (int i = 0; i < B_COUNT; ++i) {
            uint32_t n = 1;
            if (i == B_YFREE || i == B_GFREE || i == B_ABRDY || i == B_ABFREE || i == B_SRDY ||
                i == B_RRDY || i == B_SSCL || i == B_HRDY)
                n = 4;   // one arrival per warp of the publishing group
            if (i == B_BFREE) n = 8;   // the beta rows are read by both groups
            mbar_init(bar(i), n);
        }
        fence_mbar_init();
        *s_abort = 0;
    }
    if (warp == 2) tmem_alloc(sb + OFF_MISC + 4, TMEM_COLS);
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmq);
        tma_prefetch_desc(&tmk);
        tma_prefetch_desc(&tmv);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *s_tmem;

    if (warp == 0) {
        // ================================================================ producer
        if (lane == 0) {
            const int shift = shifted ? 1 : 0;
            int nfill[NST] = {}, ny = 0, nb = 0;
            bool ok = true;
            int cx = 0, cy = 0, cb = 0;
            uint64_t t_last = globaltimer();
            while (cx < nch || cy < nch || cb < nch) {
                bool progressed = false;
                if (cx < nch) {
                    const int b = cx % NST;
                    if (cx < NST || mbar_test(bar(B_EMPTY0 + b), (uint32_t)((cx / NST) - 1) & 1u)) {
                        const uint32_t st = xq(b);
                        const int y = cx * C;
                        const uint32_t full = bar(B_FULL0 + b);
                        mbar_expect_tx(full, 32 * KB);
                        tma_load_3d(st + XQ_X0, &tmk, 0, y - shift, (int)chain, full);
                        tma_load_3d(st + XQ_X1, &tmk, 64, y - shift, (int)chain, full);
                        tma_load_3d(st + XQ_Q0, &tmq, 0, y, (int)chain, full);
                        tma_load_3d(st + XQ_Q1, &tmq, 64, y, (int)chain, full);
                        ++nfill[b];
                        ++cx;
                        progressed = true;
                    }
                }
                if (cy < nch && cy < cx && (cy == 0 || mbar_test(bar(B_YFREE), (uint32_t)(cy - 1) & 1u))) {
                    const int y = cy * C;
                    mbar_expect_tx(bar(B_FULLY), 16 * KB);
                    tma_load_3d(sb + OFF_Y, &tmv, 0, y, (int)chain, bar(B_FULLY));
                    tma_load_3d(sb + OFF_Y + 8 * KB, &tmv, 64, y, (int)chain, bar(B_FULLY));
                    ++ny;
                    ++cy;
                    progressed = true;
                }
                if (cb < nch && cb < cx && (cb == 0 || mbar_test(bar(B_BFREE), (uint32_t)(cb - 1) & 1u))) {
                    // the chunk's beta rows: contiguous [t][j] fp32, 512 B per token,
                    // clipped at the chain's end (rows past T are never read)
                    const int64_t t0 = (int64_t)cb * C;
                    const int rows = (int)((T - t0) < C ? (T - t0) : C);
                    const uint32_t bytes = (uint32_t)rows * (uint32_t)D * 4u;
                    mbar_expect_tx(bar(B_FULLB), bytes);
                    bulk_g2s(sb + OFF_BETA, a.beta + (chain * T + t0) * D, bytes, bar(B_FULLB));
                    ++nb;
                    ++cb;
                    progressed = true;
                }
                if (progressed) {
                    t_last = globaltimer();
                } else {
                    if (*s_abort) { ok = false; break; }
                    if (globaltimer() - t_last > limit) { ok = false; break; }
                    __nanosleep(200);
                }
            }
            if (!ok) fail_now();
            // never leave a copy in flight into this CTA's shared memory
            for (int b = 0; b < NST; ++b)
                if (nfill[b]) mbar_wait(bar(B_FULL0 + b), (uint32_t)(nfill[b] - 1) & 1u, kDrainNs);
            if (ny) mbar_wait(bar(B_FULLY), (uint32_t)(ny - 1) & 1u, kDrainNs);
            if (nb) mbar_wait(bar(B_FULLB), (uint32_t)(nb - 1) & 1u, kDrainNs);
        }
        __syncwarp();
    } else if (warp == 1) {
        // ================================================================ MMA issuer
        if (lane == 0) {
            bool ok = true;
            auto issue_g = [&](int cc) -> bool {   // G = [X; Q] X^T of chunk cc
                if (!cwait(bar(B_FULL0 + cc % NST), (uint32_t)(cc / NST) & 1u, limit, s_abort) ||
                    (cc >= 1 && !cwait(bar(B_GFREE), (uint32_t)(cc - 1) & 1u, limit, s_abort)) ||
                    (cc == 0 && a.k_init && !cwait(bar(B_PATCH), 0u, limit, s_abort)))
                    return false;
                tc_fence_after();
                const uint32_t id = idesc_bf16(128, 64, false, false);
                const uint64_t dx = sdesc_sw128(xq(cc % NST) + XQ_X0, 16, 1024);
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    const uint64_t off = ((kk >> 2) * 16384u + (kk & 3) * 32u) >> 4;
                    mma_bf16(tmem + COL_G, dx + off, dx + off, id, kk > 0);
                }
                mma_commit(bar(B_GDONE));
                return true;
            };
            const uint32_t id64 = idesc_bf16(128, 64, false, false);
            if (nch > 0) ok = issue_g(0);
            // chunk 0's U^T = S0^T X^T (not for the additive write), V^T = S0^T Q^T from
            // the bf16 copy of the initial state
            if (ok && nch > 0) {
                if (!cwait(bar(B_SRDY), 0u, limit, s_abort)) ok = false;
                if (ok) {
                    tc_fence_after();
                    const uint32_t sa = tmem + COL_SB;
                    const uint64_t dxk = sdesc_sw128(xq(0) + XQ_X0, 16, 1024);
                    const uint64_t dqk = sdesc_sw128(xq(0) + XQ_Q0, 16, 1024);
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk) {
                        const uint64_t off = ((kk >> 2) * 16384u + (kk & 3) * 32u) >> 4;
                        if (!INNER) mma_bf16_ta(tmem + COL_U, sa + 8 * kk, dxk + off, id64, kk > 0);
                        mma_bf16_ta(tmem + COL_V, sa + 8 * kk, dqk + off, id64, kk > 0);
                    }
                    mma_commit(bar(B_UVDONE));
                }
            }
            for (int c = 0; c < nch && ok; ++c) {
                const uint32_t st = xq(c % NST);
                const bool more = c + 1 < nch;
                if (more) {
                    const uint32_t stn = xq((c + 1) % NST);
                    // the next chunk's Gram while this chunk's channels run, then the cross
                    // Gram H = [X_{c+1}; Q_{c+1}] X_c^T (its region is free: the staging
                    // group has read the previous one)
                    if (!issue_g(c + 1)) { ok = false; break; }
                    if (c >= 1 && !cwait(bar(B_HRDY), (uint32_t)(c - 1) & 1u, limit, s_abort)) { ok = false; break; }
                    tc_fence_after();
                    {
                        const uint64_t dn = sdesc_sw128(stn + XQ_X0, 16, 1024);
                        const uint64_t dc = sdesc_sw128(st + XQ_X0, 16, 1024);
#pragma unroll
                        for (int kk = 0; kk < 8; ++kk) {
                            const uint64_t off = ((kk >> 2) * 16384u + (kk & 3) * 32u) >> 4;
                            mma_bf16(tmem + COL_H, dn + off, dc + off, id64, kk > 0);
                        }
                        mma_commit(bar(B_HDONE));
                    }
                    // chunk c+1's U and V: S_{c+1} = diag(G_C) S_c + X_c^T Rw_c, so
                    //   U^T = (diag(G_C) S_c)^T X_{c+1}^T + Rw_c^T (X_c X_{c+1}^T)
                    // (V with Q_{c+1}).  The first part from the staging group's bf16 copy
                    // of the pre-scaled state, once this chunk's channels have read U / V;
                    // the second once the weights and H are staged.
                    if (!cwait(bar(B_ABFREE), (uint32_t)c & 1u, limit, s_abort) ||
                        !cwait(bar(B_SSCL), (uint32_t)c & 1u, limit, s_abort)) { ok = false; break; }
                    tc_fence_after();
                    {
                        const uint32_t sa = tmem + COL_SB;
                        const uint64_t dxk = sdesc_sw128(stn + XQ_X0, 16, 1024);
                        const uint64_t dqk = sdesc_sw128(stn + XQ_Q0, 16, 1024);
#pragma unroll
                        for (int kk = 0; kk < 8; ++kk) {
                            const uint64_t off = ((kk >> 2) * 16384u + (kk & 3) * 32u) >> 4;
                            if (!INNER) mma_bf16_ta(tmem + COL_U, sa + 8 * kk, dxk + off, id64, kk > 0);
                            mma_bf16_ta(tmem + COL_V, sa + 8 * kk, dqk + off, id64, kk > 0);
                        }
                    }
                    if (!cwait(bar(B_RRDY), (uint32_t)c & 1u, limit, s_abort) ||
                        !cwait(bar(B_HRDY), (uint32_t)c & 1u, limit, s_abort)) { ok = false; break; }
                    tc_fence_after();
                    {
                        const uint64_t dr = sdesc_sw128(sb + OFF_RT, 16, 1024);
                        const uint64_t dhx = sdesc_sw128(st + XQ_Q0, 16, 1024);   // H rows of X_{c+1}
                        const uint64_t dhq = sdesc_sw128(st + XQ_Q1, 16, 1024);   // H rows of Q_{c+1}
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk) {
                            if (!INNER) mma_bf16(tmem + COL_U, dr + kk * 2, dhx + kk * 2, id64, 1);
                            mma_bf16(tmem + COL_V, dr + kk * 2, dhq + kk * 2, id64, 1);
                        }
                        mma_commit(bar(B_UVDONE));
                        CTRACE(c, 6);
                    }
                } else {
                    if (!cwait(bar(B_RRDY), (uint32_t)c & 1u, limit, s_abort) ||
                        !cwait(bar(B_SSCL), (uint32_t)c & 1u, limit, s_abort)) { ok = false; break; }
                    tc_fence_after();
                }
                // S^T += Rw^T X, onto the state pre-scaled by the chunk's decay
                {
                    const uint32_t id_s = idesc_bf16(128, 128, false, true);
                    const uint64_t dr = sdesc_sw128(sb + OFF_RT, 16, 1024);
                    const uint64_t dx = sdesc_sw128(st + XQ_X0, 16384, 1024);   // X as MN-major B (N = i)
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) mma_bf16(tmem + COL_S, dr + kk * 2, dx + kk * 128, id_s, 1);
                    mma_commit(bar(B_SDONE));
                    mma_commit(bar(B_EMPTY0 + c % NST));
                    CTRACE(c, 7);
                }
            }
            if (!ok) fail_now();
            mma_commit(bar(B_MDRAIN));
            mbar_wait(bar(B_MDRAIN), 0, kDrainNs);
        }
        __syncwarp();
    } else if (warp >= SG_W0 && warp < CG_W0) {
        // ================================================================ staging group
        const int r = tid - SG_W0 * 32;   // == TMEM lane: row r of [X; Q] X^T
        const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
        bool ok = true;
        if (a.force_timeout) {   // testing hook: a wait on a barrier nothing arrives on
            const bool w = cwait(bar(B_NEVER), 0, limit, s_abort);
            if (bar_or(BAR_SGRP, GROUP, !w)) ok = false;
        }
        // chunk 0's first key row is phi(k_init) when one is given (the row before
        // the sequence reads as zero otherwise)
        if (ok && a.k_init && nch > 0) {
            const bool w = cwait(bar(B_FULL0), 0u, limit, s_abort);
            if (bar_or(BAR_SGRP, GROUP, !w)) {
                ok = false;
            } else {
                if (r < 16) {
                    const int hb = r >> 3, c16 = r & 7;
                    const uint4 u = *reinterpret_cast<const uint4 *>(
                        static_cast<const __nv_bfloat16 *>(a.k_init) + chain * D + hb * 64 + c16 * 8);
                    const uint32_t w4[4] = {u.x, u.y, u.z, u.w};
                    float f[8];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float2 p2 = unpack_bf16(w4[e]);
                        f[2 * e] = apply_phi(a.phi, p2.x);
                        f[2 * e + 1] = apply_phi(a.phi, p2.y);
                    }
                    st_row8(xq(0) + (hb ? XQ_X1 : XQ_X0) + (uint32_t)c16 * 16u, f);
                    fence_proxy_async();
                }
                bar_sync(BAR_SGRP, GROUP);
                if (r == 0) mbar_arrive(bar(B_PATCH));
            }
        }
        float *Am = reinterpret_cast<float *>(sm + (r < C ? OFF_A : OFF_B));
        const int t = r & (C - 1);
        // lambda of row t of the next chunk, loaded a chunk ahead so that its global
        // read is not on the staging's path
        auto lam_of = [&](int cc) -> float {
            const int64_t tok = (int64_t)cc * C + t;
            // a volatile read: issued here and kept in its register, not re-read at the use
            return (r < C && cc < nch && tok < T)
                       ? *static_cast<const volatile float *>(a.lam + chain * T + tok) : 0.f;
        };
        float lt_next = lam_of(0);
#pragma unroll 1
        for (int c = 0; c < nch && ok; ++c) {
            const float lt = lt_next;
            lt_next = lam_of(c + 1);
            {
                bool w = cwait(bar(B_GDONE), (uint32_t)c & 1u, limit, s_abort);
                w = w && (c < 1 || cwait(bar(B_ABFREE), (uint32_t)(c - 1) & 1u, limit, s_abort));
                if (bar_or(BAR_SGRP, GROUP, !w)) { ok = false; break; }
            }
            tc_fence_after();
            {
                // the whole row in two 32-column loads and one wait
                float ga[32], gb[32];
                tmem_ld32x2(tmem + lane_base + COL_G, tmem + lane_base + COL_G + 32, ga, gb);
#pragma unroll
                for (int e4 = 0; e4 < 8; ++e4) {
                    *reinterpret_cast<float4 *>(Am + t * ABROW + 4 * e4) =
                        make_float4(ga[4 * e4], ga[4 * e4 + 1], ga[4 * e4 + 2], ga[4 * e4 + 3]);
                    *reinterpret_cast<float4 *>(Am + t * ABROW + 32 + 4 * e4) =
                        make_float4(gb[4 * e4], gb[4 * e4 + 1], gb[4 * e4 + 2], gb[4 * e4 + 3]);
                }
                if (r < C) {   // the diagonal: |x_t|^2
                    const int64_t tok = (int64_t)c * C + t;
                    float n = 0.f;
#pragma unroll
                    for (int e = 0; e < 32; ++e) {
                        n = (e == t) ? ga[e] : n;
                        n = (e + 32 == t) ? gb[e] : n;
                    }
                    // 0 where the token has no pair (past the chain's end, or the first
                    // token of a shifted pairing without k_init): its eta is 0
                    const bool pair = tok < T && (!shifted || tok > 0 || a.k_init != nullptr);
                    inv[t] = pair ? 1.f / (n + lt + a.eps) : 0.f;
                    lamv[t] = lt;
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(bar(B_GFREE));   // this warp's rows of the Gram region are read
                mbar_arrive(bar(B_ABRDY));   // and its rows of A or B are staged
            }
            if (r == 0) CTRACE(c, 8);
            // this chunk's total decay of channel r, and the fp32 state (lane r) pre-scaled
            // by it with a bf16 copy (the A operand of the next chunk's U and V), once the
            // previous chunk's state update is done and this chunk's U and V are formed
            // (they read the previous copy)
            {
                bool w = cwait(bar(B_UVDONE), (uint32_t)c & 1u, limit, s_abort);
                w = w && (c == 0 ? cwait(bar(B_SRDY), 0u, limit, s_abort)
                                 : cwait(bar(B_SDONE), (uint32_t)(c - 1) & 1u, limit, s_abort));
                w = w && cwait(bar(B_FULLB), (uint32_t)c & 1u, limit, s_abort);
                if (bar_or(BAR_SGRP, GROUP, !w)) { ok = false; break; }
            }
            {
                const float *betam = reinterpret_cast<const float *>(sm + OFF_BETA);
                float gtot = 1.f;
#pragma unroll 4
                for (int tt = 0; tt < C; ++tt) {
                    const float eta = betam[tt * D + r] * inv[tt];   // 0 where no pair exists
                    gtot *= 1.f - eta * lamv[tt];
                }
                tc_fence_after();
#pragma unroll 1
                for (int q = 0; q < 4; ++q) {
                    float v[32];
                    tmem_ld32(tmem + lane_base + COL_S + 32 * q, v);
#pragma unroll
                    for (int e = 0; e < 32; ++e) v[e] *= gtot;
                    tmem_st16(tmem + lane_base + COL_S + 32 * q, v);
                    tmem_st16(tmem + lane_base + COL_S + 32 * q + 16, v + 16);
                    float pk[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e) pk[e] = __uint_as_float(pack_bf16(v[2 * e], v[2 * e + 1]));
                    tmem_st16(tmem + lane_base + COL_SB + 16 * q, pk);
                }
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(bar(B_SSCL));
                    mbar_arrive(bar(B_BFREE));
                }
            }
            // H = [X_{c+1}; Q_{c+1}] X_c^T as bf16 K-major rows (row r: r < 64 the next
            // keys', else the next queries') into this chunk's Q tile, which V^T has read
            if (c + 1 < nch) {
                const bool w = cwait(bar(B_HDONE), (uint32_t)c & 1u, limit, s_abort);
                if (bar_or(BAR_SGRP, GROUP, !w)) { ok = false; break; }
                tc_fence_after();
                const uint32_t hb = xq(c % NST) + (r < C ? XQ_Q0 : XQ_Q1);
#pragma unroll 1
                for (int q = 0; q < 4; ++q) {   // 16 columns s at a time
                    float g[16];
                    tmem_ld16(tmem + lane_base + COL_H + 16 * q, g);
                    st_row8(hb + sw128((uint32_t)t, (uint32_t)(2 * q)), g);
                    st_row8(hb + sw128((uint32_t)t, (uint32_t)(2 * q + 1)), g + 8);
                }
                fence_proxy_async();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(B_HRDY));
            }
        }
        if (!ok && r == 0) fail_now();
    } else if (warp >= CG_W0) {
        // ================================================================ channel group
        const int j = tid - CG_W0 * 32;   // value channel == TMEM lane
        const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
        auto gwait = [&](uint32_t bb, uint32_t parity) -> bool {
            const bool w = cwait(bb, parity, limit, s_abort);
            return !bar_or(BAR_CGRP, GROUP, !w);
        };
        const float *Am = reinterpret_cast<const float *>(sm + OFF_A);
        const float *Bm = reinterpret_cast<const float *>(sm + OFF_B);
        const float *betam = reinterpret_cast<const float *>(sm + OFF_BETA);
        float *zrow = reinterpret_cast<float *>(sm + OFF_Z) + j * ZROW;
        const int jw0 = j & ~31;   // first channel of this warp
        float *hts = reinterpret_cast<float *>(sm + OFF_HT) + (j >> 5) * (2 * NB * HTP);
        __nv_bfloat16 *const og = reinterpret_cast<__nv_bfloat16 *>(a.o) + chain * T * D + j;
        // V tile element (t, j): 128-byte swizzled rows, two 64-column halves
        const uint16_t *ysm = reinterpret_cast<const uint16_t *>(sm + OFF_Y + (j >= 64 ? 8 * KB : 0));
        const uint32_t ych = (uint32_t)((j & 63) >> 3), yin = (uint32_t)(j & 7) * 2u;
        bool ok = true;

        // initial state, transposed (thread j holds column j of S): fp32 and bf16
#pragma unroll 1
        for (int q = 0; q < 4; ++q) {   // i = 32q .. 32q+31
            float v[32];
#pragma unroll
            for (int e = 0; e < 32; ++e) v[e] = a.S0 ? a.S0[(chain * D + 32 * q + e) * D + j] : 0.f;
            tmem_st16(tmem + lane_base + COL_S + 32 * q, v);
            tmem_st16(tmem + lane_base + COL_S + 32 * q + 16, v + 16);
            float pk[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) pk[e] = __uint_as_float(pack_bf16(v[2 * e], v[2 * e + 1]));
            tmem_st16(tmem + lane_base + COL_SB + 16 * q, pk);
        }
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(B_SRDY));

#pragma unroll 1
        for (int c = 0; c < nch && ok; ++c) {
            const int64_t tok0 = (int64_t)c * C;
            __nv_bfloat16 *const ot = og + tok0 * D;   // row t of the chunk: ot[t * D]
            const int tlim = T - tok0 < (int64_t)C ? (int)(T - tok0) : C;   // rows past T are not written
            {
                bool w = cwait(bar(B_ABRDY), (uint32_t)c & 1u, limit, s_abort);
                w = w && cwait(bar(B_UVDONE), (uint32_t)c & 1u, limit, s_abort);
                w = w && cwait(bar(B_FULLY), (uint32_t)c & 1u, limit, s_abort);
                w = w && cwait(bar(B_FULLB), (uint32_t)c & 1u, limit, s_abort);
                if (bar_or(BAR_CGRP, GROUP, !w)) { ok = false; break; }
            }
            if (j == 0) CTRACE(c, 0);
            tc_fence_after();
            float gacc = 1.f;   // G of the last token done (running chunk prefix)
            float totp = 1.f;   // total decay of the previous block (this channel)
#pragma unroll 1
            for (int tb = 0; tb < C / NB; ++tb) {
                const int b0 = NB * tb;
                // gates of the block's tokens: eta = beta inv (inv is 0 where no pair
                // exists or past the chain's end), gamma = 1 - eta lambda
                float eta[NB], gam[NB], yv[NB], uv[NB], vv[NB], pre[NB];
                const uint16_t *yrow = ysm + (uint32_t)tb * 512u;   // rows b0 .. b0+7 (1 KB atom)
                float iv[NB], lv[NB];   // the block's shared scalars, two 16-byte loads each
#pragma unroll
                for (int e4 = 0; e4 < NB; e4 += 4) {
                    const float4 i4 = *reinterpret_cast<const float4 *>(inv + b0 + e4);
                    const float4 l4 = *reinterpret_cast<const float4 *>(lamv + b0 + e4);
                    iv[e4] = i4.x; iv[e4 + 1] = i4.y; iv[e4 + 2] = i4.z; iv[e4 + 3] = i4.w;
                    lv[e4] = l4.x; lv[e4 + 1] = l4.y; lv[e4 + 2] = l4.z; lv[e4 + 3] = l4.w;
                }
#pragma unroll
                for (int e = 0; e < NB; ++e) {
                    eta[e] = betam[(b0 + e) * D + j] * iv[e];
                    gam[e] = 1.f - eta[e] * lv[e];
                    // row b0 + e of the swizzled V tile: 128-byte row e of the block's atom
                    yv[e] = __uint_as_float((uint32_t)yrow[(e * 128 + ((ych ^ (uint32_t)e) << 4) + yin) >> 1] << 16);
                    pre[e] = (e == 0 ? 1.f : pre[e - 1]) * gam[e];
                }
                if (INNER) tmem_ld8(tmem + lane_base + COL_V + b0, vv);
                else tmem_ld8x2(tmem + lane_base + COL_U + b0, tmem + lane_base + COL_V + b0, uv, vv);
                if (j == 0 && (tb == 0 || tb == 7)) CTRACE(c, tb == 0 ? 10 : 13);
                // cross-block sums H_A(t) = sum_{s < b0} A[t,s] zhat_s (and H_B with B) for
                // the block's eight rows and this warp's 32 channels, as the transposed
                // product (j x s) (s x t) on the warp's tf32 MMAs: two 16-channel tiles,
                // n = the block's eight tokens, the k steps alternating between two
                // accumulator sets; then through shared memory to one thread per channel.
                // Weights of blocks before the previous one still lack the previous
                // block's decay: they take it on the way in and are stored back.
                float ha[NB], hb[NB];
                {
                    const int g = lane >> 2, t4 = lane & 3;
                    float sc[4];   // decay of channels g + 8 q of this warp
#pragma unroll
                    for (int q = 0; q < 4; ++q) sc[q] = __shfl_sync(0xffffffffu, totp, g + 8 * q);
                    __syncwarp();   // the previous block's weights are in shared memory
                    float xa[2][2][4], xb[2][2][4];   // [k-step parity][channel tile][fragment]
#pragma unroll
                    for (int p = 0; p < 2; ++p)
#pragma unroll
                        for (int mt = 0; mt < 2; ++mt)
#pragma unroll
                            for (int e = 0; e < 4; ++e) { xa[p][mt][e] = 0.f; xb[p][mt][e] = 0.f; }
                    const float *arow = Am + (b0 + g) * ABROW + t4;
                    const float *brow = Bm + (b0 + g) * ABROW + t4;
                    float *zr = reinterpret_cast<float *>(sm + OFF_Z) + (jw0 + g) * ZROW + t4;
                    auto kstep = [&](float (&ya)[2][4], float (&yb)[2][4], int k0, bool stale) {
                        const uint32_t fa[2] = {__float_as_uint(arow[k0]), __float_as_uint(arow[k0 + 4])};
                        const uint32_t fb[2] = {__float_as_uint(brow[k0]), __float_as_uint(brow[k0 + 4])};
#pragma unroll
                        for (int mt = 0; mt < 2; ++mt) {
                            float *zp = zr + 16 * mt * ZROW + k0;
                            // fragment rows g and g + 8 (channels), columns t4 and t4 + 4 (s)
                            float z00 = zp[0], z10 = zp[8 * ZROW], z01 = zp[4], z11 = zp[8 * ZROW + 4];
                            if (stale) {
                                z00 *= sc[2 * mt];
                                z01 *= sc[2 * mt];
                                z10 *= sc[2 * mt + 1];
                                z11 *= sc[2 * mt + 1];
                                zp[0] = z00;
                                zp[4] = z01;
                                zp[8 * ZROW] = z10;
                                zp[8 * ZROW + 4] = z11;
                            }
                            const uint32_t fz[4] = {__float_as_uint(z00), __float_as_uint(z10),
                                                    __float_as_uint(z01), __float_as_uint(z11)};
                            if (!INNER) mma_tf32_16x8x8(ya[mt], fz, fa);
                            mma_tf32_16x8x8(yb[mt], fz, fb);
                        }
                    };
                    int k0 = 0;
#pragma unroll 1
                    for (; k0 + 16 <= b0; k0 += 16) {
                        kstep(xa[0], xb[0], k0, true);
                        kstep(xa[1], xb[1], k0 + 8, k0 + 16 < b0);
                    }
                    if (k0 < b0) kstep(xa[0], xb[0], k0, false);
                    // fragment (channel 16 mt + g + 8 h, token 2 t4 + u) to [token][channel]
#pragma unroll
                    for (int mt = 0; mt < 2; ++mt)
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const int idx = (2 * t4 + (e & 1)) * HTP + 16 * mt + g + 8 * (e >> 1);
                            if (!INNER) hts[idx] = xa[0][mt][e] + xa[1][mt][e];
                            hts[NB * HTP + idx] = xb[0][mt][e] + xb[1][mt][e];
                        }
                    __syncwarp();
#pragma unroll
                    for (int e = 0; e < NB; ++e) {
                        ha[e] = INNER ? 0.f : hts[e * HTP + lane];
                        hb[e] = hts[(NB + e) * HTP + lane];
                    }
                    __syncwarp();
                }
                if (j == 0 && (tb == 0 || tb == 7)) CTRACE(c, tb == 0 ? 11 : 14);
                // the block's tokens in order; w_s = eta_s r_s
                float rr[NB], wv[NB], wr[NB];
#pragma unroll
                for (int tl = 0; tl < NB; ++tl) {
                    const int t = b0 + tl;
                    const float gm = gacc;          // G_{t-1}
                    gacc *= gam[tl];                // G_t
                    const float ct = tl >= 1 ? pre[tl - 1] : 1.f;
                    float ina = 0.f, inb = 0.f;
                    // row t's columns of the block: the strictly lower part and (for the
                    // write-then-read output) the diagonal; the second group of four only
                    // once the row reaches it
                    float arow[NB], brow[NB];
#pragma unroll
                    for (int e4 = 0; e4 < NB; e4 += 4) {
                        if (e4 <= tl) {
                            const float4 a4 = *reinterpret_cast<const float4 *>(Am + t * ABROW + b0 + e4);
                            const float4 b4 = *reinterpret_cast<const float4 *>(Bm + t * ABROW + b0 + e4);
                            arow[e4] = a4.x; arow[e4 + 1] = a4.y; arow[e4 + 2] = a4.z; arow[e4 + 3] = a4.w;
                            brow[e4] = b4.x; brow[e4 + 1] = b4.y; brow[e4 + 2] = b4.z; brow[e4 + 3] = b4.w;
                        }
                    }
                    // wr[s] = D[t-1, s] w_s, carried from the previous token: the older
                    // weights take gamma_{t-1}, the newest enters as w_{t-1}
                    if (tl >= 1) {
#pragma unroll
                        for (int sl = 0; sl < tl - 1; ++sl) wr[sl] *= gam[tl - 1];
                        wr[tl - 1] = wv[tl - 1];
                    }
#pragma unroll
                    for (int sl = 0; sl < tl; ++sl) {   // oldest first: the newest residual enters last
                        if (!INNER) ina = fmaf(arow[sl], wr[sl], ina);
                        inb = fmaf(brow[sl], wr[sl], inb);
                    }
                    if (INNER) rr[tl] = yv[tl];
                    else rr[tl] = yv[tl] - gm * uv[tl] - ct * ha[tl] - ina;
                    wv[tl] = eta[tl] * rr[tl];
                    float o;
                    if (rbw) o = gm * vv[tl] + ct * hb[tl] + inb;
                    else o = gacc * vv[tl] + gam[tl] * (ct * hb[tl] + inb) + brow[tl] * wv[tl];
                    if (t < tlim) ot[t * D] = __float2bfloat16_rn(o);
                }
                if (j == 0 && (tb == 0 || tb == 7)) CTRACE(c, tb == 0 ? 12 : 15);
                // the block is done: its own tokens take the suffix products to its
                // end (earlier weights take its total decay in the next block's sums)
                totp = pre[NB - 1];
                float zb[NB], suf = 1.f;
#pragma unroll
                for (int e = NB - 1; e >= 0; --e) {
                    zb[e] = suf * wv[e];
                    suf *= gam[e];
                }
#pragma unroll
                for (int e4 = 0; e4 < NB; e4 += 4)
                    *reinterpret_cast<float4 *>(zrow + b0 + e4) = make_float4(zb[e4], zb[e4 + 1], zb[e4 + 2], zb[e4 + 3]);
            }
            if (j == 0) CTRACE(c, 1);
            // A, B, inv, V and beta of this chunk are read
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(bar(B_ABFREE));
                mbar_arrive(bar(B_YFREE));
                mbar_arrive(bar(B_BFREE));
            }
            // the weights-times-residuals row as the state update's bf16 A operand,
            // the last block's decay applied to the blocks before it (the staging
            // group pre-scales the fp32 state by the chunk's decay)
#pragma unroll
            for (int c8 = 0; c8 < 8; ++c8) {
                const float f = 8 * c8 < C - NB ? totp : 1.f;
                const float4 z0 = *reinterpret_cast<const float4 *>(zrow + 8 * c8);
                const float4 z1 = *reinterpret_cast<const float4 *>(zrow + 8 * c8 + 4);
                const float z8[8] = {z0.x * f, z0.y * f, z0.z * f, z0.w * f,
                                     z1.x * f, z1.y * f, z1.z * f, z1.w * f};
                st_row8(sb + OFF_RT + sw128((uint32_t)j, (uint32_t)c8), z8);
            }
            fence_proxy_async();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(B_RRDY));
            if (j == 0) CTRACE(c, 2);
            // the last chunk writes S_T once its state update is done (the next chunk's
            // U and V come from the staging group's bf16 copy and the cross Gram)
            if (c + 1 == nch) {
                if (!gwait(bar(B_SDONE), (uint32_t)c & 1u)) { ok = false; break; }
                if (j == 0) CTRACE(c, 3);
                tc_fence_after();
#pragma unroll 1
                for (int q = 0; q < 4; ++q) {
                    float v[32];
                    tmem_ld32(tmem + lane_base + COL_S + 32 * q, v);
#pragma unroll
                    for (int e = 0; e < 32; ++e) a.S_T[(chain * D + 32 * q + e) * D + j] = v[e];
                }
            }
            if (j == 0) CTRACE(c, 4);
        }
        if (!ok && j == 0) fail_now();
    }

    // every role meets here; tensor memory is released last
    tc_fence_before();
    __syncthreads();
    if (warp == 2) {
        tc_fence_after();
        tmem_dealloc(tmem, TMEM_COLS);
    }
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// [n_chains][T][128] bf16 viewed as (d, T, chain): 64 x 64 boxes with the 128-byte
// swizzle for the tile loads.
bool make_map(CUtensorMap *m, const void *ptr, int64_t T, int64_t nc) {
    auto enc = encode_fn();
    if (!enc) return false;
    cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)T, (cuuint64_t)nc};
    cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)T * D * 2};
    cuuint32_t box[3] = {64, (cuuint32_t)C, 1};
    cuuint32_t es[3] = {1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(ptr), dims, strides, box,
               es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

// Falcon-2 / 2A with bf16 inputs, d = 128, phi = identity (phi = elu+1 would round
// phi(k) ~ 1 + k to a bf16 operand and lose the key's varying part).
bool chunked_chan_supported(const PrefillArgs &a) {
    return (a.mode == FW_FALCON2 || a.mode == FW_FALCON2A) && a.phi == FW_PHI_IDENTITY &&
           a.dtype == FW_BF16 && a.d == D && a.T <= (int64_t)INT32_MAX - C &&
           a.n_chains <= (int64_t)INT32_MAX;
}

#ifdef FW_TRACE
extern "C" int fw_debug_read_chan_trace(unsigned long long *dst, int n) {
    if (n > kCTraceChunks * kCTraceEv) n = kCTraceChunks * kCTraceEv;
    return (int)cudaMemcpyFromSymbol(dst, g_ctrace, sizeof(unsigned long long) * n);
}
#endif

cudaError_t launch_chunked_chan(const PrefillArgs &a, cudaStream_t s) {
    CUtensorMap tq, tk, tv;
    if (!make_map(&tq, a.q, a.T, a.n_chains) || !make_map(&tk, a.k, a.T, a.n_chains) ||
        !make_map(&tv, a.v, a.T, a.n_chains))
        return cudaErrorInvalidValue;
    const bool rbw = (a.flags & FW_FLAG_RBW) != 0;
    auto kern = a.mode == FW_FALCON2A ? (rbw ? chan_kernel<true, true> : chan_kernel<true, false>)
                                      : (rbw ? chan_kernel<false, true> : chan_kernel<false, false>);
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)SMEM_ALLOC);
    if (e != cudaSuccess) return e;
    kern<<<(unsigned)a.n_chains, NTHREADS, SMEM_ALLOC, s>>>(tq, tk, tv, a);
    return cudaGetLastError();
}

}  // namespace fw
