// fw_chunked.cu -- chunked tensor-core prefill for bf16 inputs, d_k = d_v = 128.
//
// Follows the three stages the "Fast Weight Attention for Continual Learning"
// paper reading gives for Falcon-1 in §4.4 (WY representation of the chunk's
// rank-one edits: intra-chunk triangular solve, short inter-chunk recurrence
// on a fixed-size state, parallel output materialisation).  The equations are
// our own derivation of that structure.  For one chunk of C = 64 tokens
// (chunk-local indices t, s), starting state S0 and
//   gamma_t = 1 - eta_t lambda_t,  D[t,s] = prod_{i=s+1..t} gamma_i,
//   G_t = prod_{i<=t} gamma_i,     Gm_t = G_{t-1},
//   L[t,s] = D[t-1,s] eta_s (x_t.x_s)  (s < t),   T = (I + L)^{-1},
//   W = T diag(Gm) X,  U = T Y,  R = U - W S0      (the true residuals r_t),
//   P[t,s] = D[t,s] eta_s (q_t.x_s)    (s <= t),
//   O = diag(G) Q S0 + P R,
//   S_C = G_{C-1} S0 + X^T diag(D[C-1,s] eta_s) R.
// D is built from direct running products, never by dividing prefix
// products: gamma may be zero or negative.  Linear attention is the same
// skeleton with x = phi(k_t), q := phi(q_t), eta = gamma = 1 and R = V.
//
// One CTA per chain, warp-specialised so that the key-only work of chunk c+1
// overlaps the state recurrence of chunk c:
//   warp 0      TMA producer: X (keys shifted one token for Falcon-1; the row
//               before the sequence reads as zero), Q, V tiles, 64 x 128 bf16,
//               128-byte swizzle; X/Q in a three-stage ring.
//   warp 1      key-path MMA issuer:  G = [X;Q] X^T, W^T = X^T (T diag Gm)^T,
//               U^T = Y^T T^T.
//   warp 2      state-path MMA issuer: R^T = U^T - S^T W^T, O1^T = S^T Q^T,
//               O2^T = R^T P^T, S += X^T (diag(w) R).
//   warp 3      tensor-memory allocation; in between, the gate warp (norms,
//               eta, gamma and the decay products of each chunk).
//   warps 4-7,  key group (two warps per tensor-memory lane quarter, each
//   12-15       owning half the columns): feature map, L and P from G, the
//               triangular solve, -W^T staging.
//   warps 8-11  state group: R staging, state carry (fp32 in tensor memory,
//               with a bf16 copy in tensor memory as the A operand of R^T and
//               O1^T), outputs o_t = G_t O1_t + O2_t, stored by each thread
//               straight to global memory (the four warps write one 256-byte
//               row per token), so no staging tile or store wait sits on the
//               state path.
// All chunk products are tcgen05 MMAs with M = 128 (transposed forms keep d on
// the M side), bf16 operands and fp32 accumulators in tensor memory.  The
// triangular solve inverts the four 16x16 diagonal blocks by fp32 forward
// substitution on the CUDA cores, then merges them in two levels,
// T_ba = -T_bb L_ba T_aa, on warp-level tf32 MMAs.  With chains on few SMs
// (SPLIT_CARRY) the state carry publishes the bf16 copy before it rescales
// the fp32 state, taking the rescale off the state path's serial chain.
// Every wait is bounded: on expiry the kernel records an error, the other
// roles stop at their next wait, copies and MMAs in flight are drained,
// tensor memory is freed and the kernel exits.
#include <cudaTypedefs.h>

#include <mutex>

#include "fw_internal.cuh"
#include "fw_sm100.cuh"

namespace fw {
namespace {
using namespace sm100;

constexpr int C = 64;        // chunk length
constexpr int D = 128;       // d_k = d_v
constexpr int NTHREADS = 512;
constexpr int KG_W0 = 4;     // first warp of the key group (lane quarters 0..3, column half 0)
constexpr int SG_W0 = 8;     // first warp of the state group
constexpr int KG2_W0 = 12;   // key group, column half 1
constexpr int BAR_KG = 1, BAR_SG = 2;   // named barriers of the two groups
constexpr int BAR_PAIR0 = 3;            // and of the key group's two merge pairs (3, 4)
constexpr int GROUP = 128, KGROUP = 256;

constexpr uint32_t KB = 1024;
constexpr int NST = 3;       // depth of the key/query tile ring (and of the gate blocks)
// shared memory (offsets from a 1024-aligned base)
constexpr uint32_t OFF_XQ0 = 0;         // NST stages of X0 Q0 X1 Q1 (8 KB each)
constexpr uint32_t XQ_X0 = 0, XQ_Q0 = 8 * KB, XQ_X1 = 16 * KB, XQ_Q1 = 24 * KB;
constexpr uint32_t OFF_Y0 = 96 * KB;    // V tile (Falcon-1: the only one; linattn: stage 0)
constexpr uint32_t OFF_Y1 = 112 * KB;   // linattn: V of stage 1; Falcon-1: solve region 0
// Falcon-1 solve regions (16 KB each, alternating by chunk parity): L (fp32 64x64,
// 16-byte-group swizzle), then the bf16 T (K-major rows t) and -T diag(Gm) in its
// two halves once L is dead; the other region holds the fp32 T of the solve.
constexpr uint32_t OFF_PB0 = 128 * KB, OFF_PB1 = 136 * KB;   // P, bf16, K-major rows t
constexpr uint32_t OFF_WTB = 144 * KB;  // -W^T, bf16, rows i (MN-major B operand)
constexpr uint32_t OFF_RA = 160 * KB;   // R^T, bf16, rows j (K-major A operand)
constexpr uint32_t OFF_RB = 176 * KB;   // (diag(w) R)^T, bf16, rows j (K-major A operand)
constexpr uint32_t OFF_TF = 192 * KB;   // Falcon-1: solve region 1; linattn: V of stage 2
constexpr uint32_t OFF_MS = 208 * KB;   // solver scratch: 32 x 32 fp32
constexpr uint32_t OFF_VEC = 212 * KB;  // NST gate blocks
constexpr uint32_t VEC_BYTES = 1792;
constexpr uint32_t V_ETA = 0, V_GAM = 256, V_G = 512, V_GM = 768, V_WC = 1024, V_Q32 = 1280,
                   V_GC = 1536;
constexpr uint32_t OFF_BAR = OFF_VEC + NST * VEC_BYTES;
constexpr uint32_t OFF_MISC = OFF_BAR + 32 * 8;
constexpr uint32_t OFF_SGV = OFF_MISC + 64;    // G_t of the chunk the state group is on
constexpr uint32_t SMEM_BYTES = OFF_SGV + 256;
constexpr uint32_t SMEM_ALLOC = SMEM_BYTES + 1024;
static_assert(SMEM_ALLOC <= 227 * KB, "shared memory budget");

// mbarriers
enum {
    B_FULL0 = 0, B_EMPTY0 = B_FULL0 + NST, B_FULLY = B_EMPTY0 + NST, B_YFREE, B_GGO, B_GDONE,
    B_TRDY, B_WUDONE, B_WRDY, B_GV0, B_PFREE0 = B_GV0 + NST, B_PFREE1, B_SRDY, B_RDONE, B_RRDY,
    B_SDONE, B_OFREE, B_RFREE, B_KDRAIN, B_SDRAIN, B_NEVER, B_SSCL, B_COUNT
};
static_assert(B_COUNT <= 32, "barrier area");

// tensor-memory columns (128 lanes x 32 bit).  The state is held transposed (lane j),
// with a bf16 copy (two i per column) that is the A operand of R and O1.
constexpr uint32_t COL_G = 0, COL_W = 64, COL_R = 128, COL_SB = 192, COL_O1 = 256, COL_O2 = 320,
                   COL_S = 384;
constexpr uint32_t TMEM_COLS = 512;

constexpr uint64_t kDrainNs = 2000000000ull;

// Optional phase timestamps of CTA 0 (instrumented builds only).
#ifdef FW_TRACE
constexpr int kTraceEv = 32, kTraceChunks = 64;
// per-chunk phase stamps, then per-warp stamps of four publications (64 x 4 x 16)
__device__ unsigned long long g_trace[kTraceChunks * kTraceEv + kTraceChunks * 64];
#define TRACE(c, ev) \
    do { if (blockIdx.x == 0 && (c) < kTraceChunks) g_trace[(c) * kTraceEv + (ev)] = globaltimer(); } while (0)
#define TRACEW(c, ev) \
    do { if (blockIdx.x == 0 && (c) < kTraceChunks && (threadIdx.x & 31) == 0) \
        g_trace[kTraceChunks * kTraceEv + ((c) * 4 + (ev)) * 16 + (threadIdx.x >> 5)] = globaltimer(); } while (0)
#else
#define TRACE(c, ev) do { } while (0)
#define TRACEW(c, ev) do { } while (0)
#endif

// fp32 64x64 matrix with its 16-byte groups XOR-swizzled by row (conflict-free
// row writes and tf32 fragment loads); same for the 32x32 scratch.
__device__ __forceinline__ int f64i(int r, int c) { return r * 64 + ((((c >> 2) ^ (r & 15)) << 2) | (c & 3)); }
__device__ __forceinline__ int f32i(int r, int c) { return r * 32 + ((((c >> 2) ^ (r & 7)) << 2) | (c & 3)); }

__device__ __forceinline__ void st_row8_bf16(uint32_t addr, const float *v) {
    st_shared_v4(addr, pack_bf16(v[0], v[1]), pack_bf16(v[2], v[3]), pack_bf16(v[4], v[5]),
                 pack_bf16(v[6], v[7]));
}

__device__ __forceinline__ void unpack8(const uint4 u, float *f) {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        const float2 p = unpack_bf16(w[e]);
        f[2 * e] = p.x;
        f[2 * e + 1] = p.y;
    }
}

// Bounded waits.  The fast path (the phase is already complete) is inline; the
// slow path is one out-of-line function shared by every call site, so that the
// roles' per-chunk code stays short (each role's loop runs once per chunk and
// competes with the other roles for the instruction caches).  A waiting thread is
// parked (issuing nothing) between polls, and gives up on expiry or as soon as
// another role has aborted.
__device__ __noinline__ bool wait_slow(uint32_t bar, uint32_t parity, uint64_t limit,
                                       volatile int *abort_flag) {
    const uint64_t t0 = globaltimer();
    for (;;) {
        if (mbar_try_wait_sleep(bar, parity, 100000u)) return true;
        if (*abort_flag) return false;
        if (globaltimer() - t0 > limit) return false;
    }
}

__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, uint64_t limit,
                                         volatile int *abort_flag) {
    if (mbar_try_wait(bar, parity)) return true;
    return wait_slow(bar, parity, limit, abort_flag);
}

__device__ __forceinline__ bool wait_fast(uint32_t bar, uint32_t parity, uint64_t limit,
                                          volatile int *abort_flag) {
    return wait_bar(bar, parity, limit, abort_flag);
}

// tf32 fragments of a 16x8 A tile / 8x8 B tile of a swizzled fp32 matrix.
// (fp32 bits go in as is: the tf32 MMA reads the top 19 bits of each operand)
__device__ __forceinline__ void frag_a64(const float *M, int r0, int k0, int lane, uint32_t (&a)[4]) {
    const int g = lane >> 2, t = lane & 3;
    a[0] = __float_as_uint(M[f64i(r0 + g, k0 + t)]);
    a[1] = __float_as_uint(M[f64i(r0 + g + 8, k0 + t)]);
    a[2] = __float_as_uint(M[f64i(r0 + g, k0 + t + 4)]);
    a[3] = __float_as_uint(M[f64i(r0 + g + 8, k0 + t + 4)]);
}
__device__ __forceinline__ void frag_b64(const float *M, int k0, int n0, int lane, uint32_t (&b)[2]) {
    const int g = lane >> 2, t = lane & 3;
    b[0] = __float_as_uint(M[f64i(k0 + t, n0 + g)]);
    b[1] = __float_as_uint(M[f64i(k0 + t + 4, n0 + g)]);
}
__device__ __forceinline__ void frag_b32(const float *M, int k0, int n0, int lane, uint32_t (&b)[2]) {
    const int g = lane >> 2, t = lane & 3;
    b[0] = __float_as_uint(M[f32i(k0 + t, n0 + g)]);
    b[1] = __float_as_uint(M[f32i(k0 + t + 4, n0 + g)]);
}

// GATED: eta, gamma and decays (not linear attention); FALCON: the residual
// write (L, T, W).  Each mode is its own instantiation, so no role's loop
// carries another mode's code.
template <bool GATED, bool FALCON, bool SPLIT_CARRY, bool SEGS>
__global__ void __launch_bounds__(NTHREADS, 1)
chunked_kernel(const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmk,
               const __grid_constant__ CUtensorMap tmv,
               const PrefillArgs a) {
    extern __shared__ uint8_t smem_raw[];
    // 1024-aligned base, derived from the shared array itself so that every
    // pointer below stays in the shared address space (plain shared loads)
    uint8_t *sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const uint32_t sb = smem_u32(sm);
    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    // Two-segment form (a.seg_t0 > 0, three CTAs per chain): role 0 runs tokens
    // [0, seg_t0) from S0, role 1 tokens [seg_t0, T) from a zero state, role 2 the
    // same tokens from S = I with zero targets (its outputs are Phi_t^T q_t and its
    // final state Phi_T); segment_fixup_kernel combines them.
    // (SEGS: a separate instantiation, so the one-segment kernels carry none of it)
    const int64_t T_all = a.T;
    constexpr bool segs = SEGS;
    const int role = segs ? (int)((int64_t)blockIdx.x / a.n_chains) : 0;
    const int64_t chain = segs ? (int64_t)blockIdx.x % a.n_chains : (int64_t)blockIdx.x;
    const int64_t t_base = role == 0 ? 0 : a.seg_t0;   // first token of this CTA's segment
    const int64_t T = segs ? (role == 0 ? a.seg_t0 : T_all - a.seg_t0) : T_all;   // its length
    const int nch = (int)((T + C - 1) / C);
    const void *const k_init = role == 0 ? a.k_init : nullptr;
    constexpr bool gated = GATED;                                  // eta, gamma, decays
    constexpr bool falcon = FALCON;                                // residual: L, T, W
    const bool shifted = gated && !(a.flags & FW_FLAG_SAME_PAIR);  // x_t = phi(k_{t-1})
    const bool rbw = (a.flags & FW_FLAG_RBW) != 0;                 // o_t = S_{t-1}^T q_t
    const bool elu = (a.phi == FW_PHI_ELU1);
    const uint64_t limit = (uint64_t)a.wait_ns;

    volatile int *s_abort = reinterpret_cast<volatile int *>(sm + OFF_MISC);
    volatile uint32_t *s_tmem = reinterpret_cast<volatile uint32_t *>(sm + OFF_MISC + 4);
    auto bar = [&](int i) -> uint32_t { return sb + OFF_BAR + 8u * (uint32_t)i; };
    auto vec = [&](int b) -> float * { return reinterpret_cast<float *>(sm + OFF_VEC + b * VEC_BYTES); };
    auto xq = [&](int st) -> uint32_t { return sb + OFF_XQ0 + (uint32_t)st * 32u * KB; };
    // solve region of chunk cc (Falcon-1)
    auto lreg = [&](int cc) -> uint32_t { return (cc & 1) ? OFF_TF : OFF_Y1; };
    // linear attention: V of ring stage st (Falcon-1 keeps its single V tile at OFF_Y0)
    auto yv_of = [&](int st) -> uint32_t { return sb + (st == 0 ? OFF_Y0 : st == 1 ? OFF_Y1 : OFF_TF); };
    auto fail_now = [&]() {
        *s_abort = 1;
        atomicExch(a.err, kDevErrTimeout);
    };

    if (tid == 0) {
        // Falcon-1: T, -W^T and the free Gram region are published by one arrival
        // per key-group warp; R and the state copy by one per state-group warp
        for (int i = 0; i < B_COUNT; ++i) {
            uint32_t n = 1;
            if (falcon && (i == B_TRDY || i == B_WRDY || i == B_GGO)) n = KGROUP / 32;
            if (i == B_SRDY || i == B_SSCL || i == B_RRDY || i == B_RFREE || i == B_OFREE) n = GROUP / 32;
            mbar_init(bar(i), n);
        }
        fence_mbar_init();
        *s_abort = 0;
    }
    if (role == 2) {   // zero targets: the V tiles are never loaded
        const float4 z4 = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int i = tid; i < (int)(16 * KB / 16); i += NTHREADS) {
            reinterpret_cast<float4 *>(sm + OFF_Y0)[i] = z4;
            if (!gated) {
                reinterpret_cast<float4 *>(sm + OFF_Y1)[i] = z4;
                reinterpret_cast<float4 *>(sm + OFF_TF)[i] = z4;
            }
        }
        fence_proxy_async();
    }
    if (warp == 3) tmem_alloc(sb + OFF_MISC + 4, TMEM_COLS);
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
        // ================================================================ TMA producer
        if (lane == 0) {
            const int shift = shifted ? 1 : 0;
            int nfill[NST] = {}, ny = 0;
            bool ok = true;
            // Falcon-1 / 1A: the single V tile of chunk cy can load once the U^T MMA of
            // chunk cy-1 has read the previous one.  The X/Q ring and the V tile are
            // polled independently, so a late V never holds back the ring.
            int cx = 0, cy = 0;
            uint64_t t_last = globaltimer();
            while (cx < nch || (gated && cy < nch)) {
                bool progressed = false;
                if (cx < nch) {
                    const int b = cx % NST;
                    if (cx < NST || mbar_test(bar(B_EMPTY0 + b), (uint32_t)((cx / NST) - 1) & 1u)) {
                        const uint32_t st = xq(b);
                        const int y = (int)(t_base + (int64_t)cx * C);
                        const uint32_t full = bar(B_FULL0 + b);
                        mbar_expect_tx(full, (gated || role == 2) ? 32 * KB : 48 * KB);
                        tma_load_3d(st + XQ_X0, &tmk, 0, y - shift, (int)chain, full);
                        tma_load_3d(st + XQ_X1, &tmk, 64, y - shift, (int)chain, full);
                        tma_load_3d(st + XQ_Q0, &tmq, 0, y, (int)chain, full);
                        tma_load_3d(st + XQ_Q1, &tmq, 64, y, (int)chain, full);
                        if (!gated && role != 2) {
                            const uint32_t yv = yv_of(b);
                            tma_load_3d(yv, &tmv, 0, y, (int)chain, full);
                            tma_load_3d(yv + 8 * KB, &tmv, 64, y, (int)chain, full);
                        }
                        ++nfill[b];
                        TRACE(cx, 19);
                        ++cx;
                        progressed = true;
                    }
                }
                if (gated && cy < nch && cy < cx &&
                    (cy == 0 || mbar_test(bar(B_YFREE), (uint32_t)(cy - 1) & 1u))) {
                    const int y = (int)(t_base + (int64_t)cy * C);
                    if (role == 2) {
                        mbar_arrive(bar(B_FULLY));   // zero targets: the tile stays zero
                    } else {
                        mbar_expect_tx(bar(B_FULLY), 16 * KB);
                        tma_load_3d(sb + OFF_Y0, &tmv, 0, y, (int)chain, bar(B_FULLY));
                        tma_load_3d(sb + OFF_Y0 + 8 * KB, &tmv, 64, y, (int)chain, bar(B_FULLY));
                    }
                    ++ny;
                    ++cy;
                    progressed = true;
                }
                if (progressed) {
                    t_last = globaltimer();
                } else {
                    if (*s_abort) { ok = false; break; }
                    if (globaltimer() - t_last > limit) { ok = false; break; }
                    __nanosleep(100);
                }
            }
            if (!ok) fail_now();
            // never leave a copy in flight into this CTA's shared memory
            for (int b = 0; b < NST; ++b)
                if (nfill[b]) mbar_wait(bar(B_FULL0 + b), (uint32_t)(nfill[b] - 1) & 1u, kDrainNs);
            if (ny) mbar_wait(bar(B_FULLY), (uint32_t)(ny - 1) & 1u, kDrainNs);
        }
        __syncwarp();
    } else if (warp == 1) {
        // ================================================================ key-path MMAs
        if (lane == 0) {
            bool ok = true;
            // G = [X; Q] X^T of chunk cc (rows 0..63: X X^T, rows 64..127: Q X^T)
            auto issue_g = [&](int cc) {
                tc_fence_after();
                const uint32_t id = idesc_bf16(128, 64, false, false);
                const uint64_t dx = sdesc_sw128(xq(cc % NST) + XQ_X0, 16, 1024);
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    const uint64_t off = ((kk >> 2) * 16384u + (kk & 3) * 32u) >> 4;
                    mma_bf16(tmem + COL_G, dx + off, dx + off, id, kk > 0);
                }
                mma_commit(bar(B_GDONE));
                TRACE(cc, 15);
            };
            // chunk cc's Gram may go: its tile has landed and the Gram region is free
            auto g_ready = [&](int cc) -> bool {
                return mbar_test(bar(B_GGO), (uint32_t)cc & 1u) &&
                       mbar_test(bar(B_FULL0 + cc % NST), (uint32_t)(cc / NST) & 1u);
            };
            // With phi = identity the Gram of chunk c+1 is released once chunk c's has
            // been read; it is issued as soon as it can go, ahead of chunk c's W/U
            // when those are not ready yet.
            const bool early = !elu;
            int gnext = 0;   // first chunk whose Gram has not been issued
            for (int c = 0; c < nch && ok; ++c) {
                const int b = c % NST;
                const uint32_t st = xq(b);
                if (gnext == c) {
                    if (!wait_fast(bar(B_GGO), (uint32_t)c & 1u, limit, s_abort) ||
                        !wait_fast(bar(B_FULL0 + b), (uint32_t)(c / NST) & 1u, limit, s_abort)) {
                        ok = false;
                        break;
                    }
                    issue_g(c);
                    ++gnext;
                }
                if (!gated) continue;
                {   // T of chunk c; meanwhile the next Gram, once it can go
                    const uint64_t t0 = globaltimer();
                    for (;;) {
                        if (mbar_test(bar(B_TRDY), (uint32_t)c & 1u)) break;   // W/U first
                        if (early && gnext == c + 1 && gnext < nch && g_ready(gnext)) {
                            issue_g(gnext);
                            ++gnext;
                        }
                        if (mbar_try_wait_sleep(bar(B_TRDY), (uint32_t)c & 1u, 200u)) break;
                        if (*s_abort || globaltimer() - t0 > limit) { ok = false; break; }
                    }
                    if (!ok) break;
                }
                // U^T goes where R^T of chunk c-1 was: its epilogue has read it
                if (!wait_fast(bar(B_FULLY), (uint32_t)c & 1u, limit, s_abort) ||
                    (c >= 1 && !wait_fast(bar(B_RFREE), (uint32_t)(c - 1) & 1u, limit, s_abort))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                {   // -W^T = X^T (-T diag Gm)^T, U^T = Y^T T^T (Falcon-1A: T = I, no W)
                    const uint32_t id = idesc_bf16(128, 64, true, false);
                    const uint64_t dx = sdesc_sw128(st + XQ_X0, 16384, 1024);
                    const uint64_t dtp = sdesc_sw128(sb + lreg(c) + 8 * KB, 16, 1024);
                    const uint64_t dy = sdesc_sw128(sb + OFF_Y0, 8192, 1024);
                    const uint64_t dt = sdesc_sw128(sb + lreg(c), 16, 1024);
                    // two independent accumulator chains, interleaved
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        if (falcon) mma_bf16(tmem + COL_W, dx + kk * 128, dtp + kk * 2, id, kk > 0);
                        mma_bf16(tmem + COL_R, dy + kk * 128, dt + kk * 2, id, kk > 0);
                    }
                    mma_commit(bar(B_WUDONE));
                    mma_commit(bar(B_YFREE));
                    TRACE(c, 16);
                }
            }
            if (!ok) fail_now();
            mma_commit(bar(B_KDRAIN));
            mbar_wait(bar(B_KDRAIN), 0, kDrainNs);
        }
        __syncwarp();
    } else if (warp == 2) {
        // ================================================================ state-path MMAs
        if (lane == 0) {
            bool ok = true;
            for (int c = 0; c < nch && ok; ++c) {
                const int b = c % NST, pi = c & 1;
                const uint32_t st = xq(b);
                // Falcon-1: R first (it needs only W and S); O1 once the output
                // accumulators of chunk c-1 have been read
                if (!wait_fast(bar(B_WRDY), (uint32_t)c & 1u, limit, s_abort) ||
                    !wait_fast(bar(B_SRDY), (uint32_t)c & 1u, limit, s_abort) ||
                    (!gated && c >= 1 && !wait_fast(bar(B_OFREE), (uint32_t)(c - 1) & 1u, limit, s_abort))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t pb = sb + (pi ? OFF_PB1 : OFF_PB0);
                const uint32_t sa = tmem + COL_SB;   // bf16 S^T, A operand: 8 columns per k step
                const uint32_t id_mk = idesc_bf16(128, 64, false, false);
                const uint64_t dq = sdesc_sw128(st + XQ_Q0, 16, 1024);
                const uint64_t dp = sdesc_sw128(pb, 16, 1024);
                const uint64_t dx = sdesc_sw128(st + XQ_X0, 16384, 1024);   // X as MN-major B (N = i)
                if (gated) {
                    // R^T += S^T (-W^T), then O1^T = S^T Q^T.  Falcon-1A: R = U = Y, so
                    // R^T is ready once the key-path MMA warp's U^T is.
                    if (falcon) {
                        const uint32_t id_mm = idesc_bf16(128, 64, false, true);
                        const uint64_t dw = sdesc_sw128(sb + OFF_WTB, 8192, 1024);
#pragma unroll
                        for (int kk = 0; kk < 8; ++kk)
                            mma_bf16_ta(tmem + COL_R, sa + 8 * kk, dw + kk * 128, id_mm, 1);
                        mma_commit(bar(B_RDONE));
                    } else {
                        if (!wait_fast(bar(B_WUDONE), (uint32_t)c & 1u, limit, s_abort)) { ok = false; break; }
                        tc_fence_after();
                        tc_fence_before();
                        mbar_arrive(bar(B_RDONE));
                    }
                    TRACE(c, 0);
                    if (c >= 1 && !wait_fast(bar(B_OFREE), (uint32_t)(c - 1) & 1u, limit, s_abort)) { ok = false; break; }
                    tc_fence_after();
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk)
                        mma_bf16_ta(tmem + COL_O1, sa + 8 * kk,
                                    dq + (((kk >> 2) * 16384u + (kk & 3) * 32u) >> 4), id_mk, kk > 0);
                    TRACE(c, 17);
                    if (!wait_fast(bar(B_RRDY), (uint32_t)c & 1u, limit, s_abort) ||
                        (SPLIT_CARRY && !wait_fast(bar(B_SSCL), (uint32_t)c & 1u, limit, s_abort))) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    // O2^T = R^T P^T;  S^T += (diag(w) R)^T X
                    const uint32_t id_kk = idesc_bf16(128, 64, false, false);
                    const uint64_t dra = sdesc_sw128(sb + OFF_RA, 16, 1024);
                    const uint64_t drb = sdesc_sw128(sb + OFF_RB, 16, 1024);
                    const uint32_t id_s = idesc_bf16(128, 128, false, true);
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        mma_bf16(tmem + COL_S, drb + kk * 2, dx + kk * 128, id_s, 1);
                        mma_bf16(tmem + COL_O2, dra + kk * 2, dp + kk * 2, id_kk, kk > 0);
                    }
                } else {
                    const uint64_t dv = sdesc_sw128(yv_of(b), 8192, 1024);
                    // O1^T = S^T Q^T, O2^T = V^T P^T;  S^T += V^T X
                    const uint32_t id_s = idesc_bf16(128, 128, true, true);
                    const uint32_t id_v = idesc_bf16(128, 64, true, false);
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk) {
                        mma_bf16_ta(tmem + COL_O1, sa + 8 * kk,
                                    dq + (((kk >> 2) * 16384u + (kk & 3) * 32u) >> 4), id_mk, kk > 0);
                        if (kk < 4) {
                            mma_bf16(tmem + COL_S, dv + kk * 128, dx + kk * 128, id_s, 1);
                            mma_bf16(tmem + COL_O2, dv + kk * 128, dp + kk * 2, id_v, kk > 0);
                        }
                    }
                }
                mma_commit(bar(B_SDONE));
                mma_commit(bar(B_PFREE0 + pi));
                mma_commit(bar(B_EMPTY0 + b));
                TRACE(c, 18);
            }
            if (!ok) fail_now();
            mma_commit(bar(B_SDRAIN));
            mbar_wait(bar(B_SDRAIN), 0, kDrainNs);
        }
        __syncwarp();
    } else if (warp == 3) {
        // ================================================================ gates
        // Step sizes and decay products of chunk cc, published in gate block cc % NST
        // as soon as the chunk's keys land: |x_t|^2 straight from the staged X tile,
        // eta_t = beta_t / (|x_t|^2 + lambda_t + eps), gamma_t = 1 - eta_t lambda_t,
        // then the in-chunk prefix and suffix products (division-free).
        // Lane l holds tokens l and l + 32 of the chunk.
        // (Block cc % NST was last read for chunk cc - NST by the key group (L, P,
        // the solve) and the state group (the R epilogue), all of which precede the
        // S MMAs of chunk cc - NST, whose completion released the ring stage chunk
        // cc's keys were loaded into.)
        bool ok = true;
        if (!gated) {   // linear attention: eta = 1, no decay
            for (int b = 0; b < NST; ++b) {
                float *v = vec(b);
                for (int t = lane; t < C; t += 32) {
                    v[V_ETA / 4 + t] = 1.f;
                    v[V_GAM / 4 + t] = 1.f;
                    v[V_G / 4 + t] = 1.f;
                    v[V_GM / 4 + t] = 1.f;
                    v[V_WC / 4 + t] = 1.f;
                    v[V_Q32 / 4 + t] = 1.f;
                }
                if (lane == 0) v[V_GC / 4] = 1.f;
            }
        }
        // beta, lambda of tokens lane and lane + 32, loaded one chunk ahead
        float nb[2] = {0.f, 0.f}, nl[2] = {0.f, 0.f};
        auto load_bl = [&](int cc) {
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                const int64_t tok = (int64_t)cc * C + lane + 32 * u;
                if (gated && cc < nch && tok < T) {
                    nb[u] = a.beta[chain * T_all + t_base + tok];
                    nl[u] = a.lam[chain * T_all + t_base + tok];
                }
            }
        };
        load_bl(0);
#pragma unroll 1
        for (int cc = 0; cc < nch && ok; ++cc) {
            const int b = cc % NST;
            float *vg = vec(b);
            bool w = wait_bar(bar(B_FULL0 + b), (uint32_t)(cc / NST) & 1u, limit, s_abort);
            // chunk 0's first key row is patched with phi(k_init) before the Gram is released
            if (gated && cc == 0 && k_init) w = w && wait_bar(bar(B_GGO), 0u, limit, s_abort);
            if (!__all_sync(0xffffffffu, w)) { ok = false; break; }
            if (lane == 0) TRACE(cc, 21);
            if (gated) {
                const uint32_t xs = xq(b);
                // |x_t|^2: the diagonal of each 16x16 block X_blk X_blk^T, on the warp's
                // bf16 MMAs (fp32 accumulate).  One ldmatrix.x4 gives the A fragment of
                // a 16-wide k step; its row-0..7 / row-8..15 halves are the B fragments
                // of the two 8-column tiles.
                float n[2];
                {
                    const int g = lane >> 2;
                    const int mrow = ((lane >> 3) & 1) * 8 + (lane & 7);   // row within the block
                    const int mchk = lane >> 4;                              // 16-byte chunk within the k step
                    float dg0[4], dg1[4];   // diagonal values held by lanes with t4 == g / 2
#pragma unroll
                    for (int blk = 0; blk < 4; ++blk) {
                        // two accumulators per tile (k halves): dependent chains of 4
                        float d0[2][4] = {}, d1[2][4] = {};
                        const uint32_t r = (uint32_t)(16 * blk + mrow);
#pragma unroll
                        for (int ks = 0; ks < 8; ++ks) {
                            uint32_t f[4];
                            ldmatrix_x4(xs + ((ks >> 2) ? XQ_X1 : XQ_X0) +
                                            sw128(r, (uint32_t)(2 * (ks & 3) + mchk)), f);
                            mma_bf16_16x8x16(d0[ks >> 2], f[0], f[1], f[2], f[3], f[0], f[2]);
                            mma_bf16_16x8x16(d1[ks >> 2], f[0], f[1], f[2], f[3], f[1], f[3]);
                        }
                        // (g, g) of rows 0..7 and (8+g, 8+g) of rows 8..15
                        dg0[blk] = (g & 1) ? d0[0][1] + d0[1][1] : d0[0][0] + d0[1][0];
                        dg1[blk] = (g & 1) ? d1[0][3] + d1[1][3] : d1[0][2] + d1[1][2];
                    }
#pragma unroll
                    for (int u = 0; u < 2; ++u) {
                        const int rr = lane & 15, blk0 = 2 * u + (lane >> 4);
                        const int src = 4 * (rr & 7) + ((rr & 7) >> 1);
                        float v = 0.f;
#pragma unroll
                        for (int blk = 0; blk < 4; ++blk) {
                            const float a0 = __shfl_sync(0xffffffffu, dg0[blk], src);
                            const float a1 = __shfl_sync(0xffffffffu, dg1[blk], src);
                            if (blk == blk0) v = (rr < 8) ? a0 : a1;
                        }
                        n[u] = v;
                    }
                }
                if (lane == 0) TRACE(cc, 22);
                float eta[2], gam[2];
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    const int64_t tok = (int64_t)cc * C + lane + 32 * u;
                    eta[u] = 0.f;
                    gam[u] = 1.f;
                    if (tok < T) {
                        // the same-step pair writes from the first token on
                        const bool pair = !shifted || (t_base + tok > 0) || (k_init != nullptr);
                        eta[u] = pair ? __fdividef(nb[u], n[u] + nl[u] + a.eps) : 0.f;
                        gam[u] = 1.f - eta[u] * nl[u];
                    }
                }
                load_bl(cc + 1);
                // prefix products G_t, Gm_t = G_{t-1}, Q32_t = prod_{32..t} gamma_i
                float g0 = gam[0], g1 = gam[1];
#pragma unroll
                for (int off = 1; off < 32; off <<= 1) {
                    const float u0 = __shfl_up_sync(0xffffffffu, g0, off);
                    const float u1 = __shfl_up_sync(0xffffffffu, g1, off);
                    if (lane >= off) { g0 *= u0; g1 *= u1; }
                }
                const float tot0 = __shfl_sync(0xffffffffu, g0, 31);
                const float q32 = g1;
                g1 *= tot0;
                float e0 = __shfl_up_sync(0xffffffffu, g0, 1);
                float e1 = __shfl_up_sync(0xffffffffu, g1, 1);
                if (lane == 0) { e0 = 1.f; e1 = tot0; }
                // suffix products -> w_s = D[C-1,s] eta_s = eta_s prod_{s<i<C} gamma_i
                float h0 = gam[0], h1 = gam[1];
#pragma unroll
                for (int off = 1; off < 32; off <<= 1) {
                    const float d0 = __shfl_down_sync(0xffffffffu, h0, off);
                    const float d1 = __shfl_down_sync(0xffffffffu, h1, off);
                    if (lane + off < 32) { h0 *= d0; h1 *= d1; }
                }
                const float tot1 = __shfl_sync(0xffffffffu, h1, 0);
                h0 *= tot1;
                float x0 = __shfl_down_sync(0xffffffffu, h0, 1);
                float x1 = __shfl_down_sync(0xffffffffu, h1, 1);
                if (lane == 31) { x0 = tot1; x1 = 1.f; }
                vg[V_ETA / 4 + lane] = eta[0];
                vg[V_ETA / 4 + lane + 32] = eta[1];
                vg[V_GAM / 4 + lane] = gam[0];
                vg[V_GAM / 4 + lane + 32] = gam[1];
                vg[V_G / 4 + lane] = g0;
                vg[V_G / 4 + lane + 32] = g1;
                vg[V_GM / 4 + lane] = e0;
                vg[V_GM / 4 + lane + 32] = e1;
                vg[V_Q32 / 4 + lane + 32] = q32;
                vg[V_WC / 4 + lane] = x0 * eta[0];
                vg[V_WC / 4 + lane + 32] = x1 * eta[1];
                if (lane == 31) vg[V_GC / 4] = g1;
            }
            __syncwarp();
            if (lane == 0) {
                TRACE(cc, 1);
                mbar_arrive(bar(B_GV0 + b));
            }
        }
        if (!ok && lane == 0) fail_now();
    } else if ((warp >= KG_W0 && warp < SG_W0) || warp >= KG2_W0) {
        // ================================================================ key group
        // 8 warps: two per TMEM lane quarter.  Thread (kt, h) owns row kt of the
        // 128-lane tiles and the column half [32h, 32h + 32).
        const int h = (warp >= KG2_W0) ? 1 : 0;
        const int kt = (warp & 3) * 32 + lane;     // TMEM lane of this thread
        const int kidx = h * 128 + kt;             // 0..255 within the group
        const int kw = warp & 3;                   // lane quarter
        const uint32_t lane_base = (uint32_t)(kw * 32) << 16;
        float *Ms = reinterpret_cast<float *>(sm + OFF_MS);
        // L of chunk c and the fp32 T alternate between the two solve regions (the
        // bf16 T of chunk c overwrites L(c) once L is dead, and L(c+1) goes where
        // the fp32 T(c) was, while the W/U products of chunk c still read the bf16 T)
        auto gwait = [&](uint32_t bb, uint32_t parity) -> bool {
            const bool ok = wait_bar(bb, parity, limit, s_abort);
            return !bar_or(BAR_KG, KGROUP, !ok);
        };
        auto gsync = [&]() { bar_sync(BAR_KG, KGROUP); };

        bool ok = true;
        // testing hook: a wait on a barrier nothing arrives on runs out
        if (a.force_timeout && !gwait(bar(B_NEVER), 0)) ok = false;

        // feature map on the loaded tiles of chunk cc and the k_init patch, then
        // release the Gram MMA of chunk cc
        auto prep_go = [&](int cc) -> bool {
            const uint32_t st_ = xq(cc % NST);
            if (!gwait(bar(B_FULL0 + cc % NST), (uint32_t)(cc / NST) & 1u)) return false;
            // ---- feature map on the loaded tiles (row t, a quarter of its 16-byte
            //      chunks per thread), k_init patch
            {
                bool wrote = false;
                if (elu) {
                    const int t = kidx >> 2, qq = kidx & 3;
                    const uint32_t roff = (uint32_t)(t >> 3) * 1024u + (uint32_t)(t & 7) * 128u;
                    for (int which = 0; which < (gated ? 1 : 2); ++which) {
                        const int64_t src = t_base + (int64_t)cc * C + t - ((which == 0 && shifted) ? 1 : 0);
                        if (src < 0 || src >= T_all) continue;
#pragma unroll
                        for (int m = 0; m < 4; ++m) {
                            const int cidx = 4 * qq + m;   // 0..15: block (cidx >> 3), chunk (cidx & 7)
                            const uint32_t row = st_ + (which == 0 ? ((cidx >> 3) ? XQ_X1 : XQ_X0)
                                                                  : ((cidx >> 3) ? XQ_Q1 : XQ_Q0)) + roff;
                            const uint32_t ad = row + (uint32_t)(cidx & 7) * 16u;
                            float f[8];
                            unpack8(ld_shared_v4(ad), f);
#pragma unroll
                            for (int e = 0; e < 8; ++e) f[e] = f[e] > 0.f ? f[e] + 1.f : __expf(f[e]);
                            st_row8_bf16(ad, f);
                        }
                    }
                    wrote = true;
                }
                if (gated && cc == 0 && k_init) {
                    if (kidx < 16) {
                        const int hb = kidx >> 3, c16 = kidx & 7;
                        const uint4 u = *reinterpret_cast<const uint4 *>(
                            static_cast<const __nv_bfloat16 *>(k_init) + chain * D + hb * 64 + c16 * 8);
                        float f[8];
                        unpack8(u, f);
#pragma unroll
                        for (int e = 0; e < 8; ++e) f[e] = apply_phi(a.phi, f[e]);
                        st_row8_bf16(st_ + (hb ? XQ_X1 : XQ_X0) + (uint32_t)c16 * 16u, f);
                    }
                    wrote = true;
                }
                if (wrote) fence_proxy_async();
            }
            gsync();   // mapped tiles (and the k_init row) complete: the Gram MMA may start
            if (falcon ? lane == 0 : kidx == 0) mbar_arrive(bar(B_GGO));
            return true;
        };
        // Without a feature-map pass on the tiles (phi = identity), the Gram MMA of
        // chunk c+1 is released as soon as the Gram of chunk c has been read, so it
        // runs while chunk c's solve and W/U products do.
        const bool early = !elu;
        if (ok) ok = prep_go(0);
        // L and P of chunk cc (L into Lw): waits for the P buffer (chunk cc-2's O2
        // done), the Gram and the gates of chunk cc, then releases the Gram region
        auto lp = [&](int cc, float *Lw) -> bool {
            const float *vg = vec(cc % NST);
            if (kidx == 0) TRACE(cc, 2);
            {
                bool w = cc < 2 || wait_bar(bar(B_PFREE0 + (cc & 1)), (uint32_t)((cc >> 1) - 1) & 1u, limit, s_abort);
                w = w && wait_bar(bar(B_GDONE), (uint32_t)cc & 1u, limit, s_abort);
                w = w && wait_bar(bar(B_GV0 + cc % NST), (uint32_t)(cc / NST) & 1u, limit, s_abort);
                if (bar_or(BAR_KG, KGROUP, !w)) return false;
            }
            tc_fence_after();
            // ---- L and P from G, columns 32h..32h+31 of row kt, in two rolled 16-column
            //      steps from the right.  A half's running product starts from
            //      prod_{i=32}^{u} gamma_i when its row reaches past column 31
            //      (division-free).
            {
                const bool lrow = kt < C;
                if (lrow && !falcon) {
                    // linear attention and Falcon-1A need no L
                } else {
                    const int t = lrow ? kt : kt - C;
                    // last active column: L is strictly lower; P includes the
                    // diagonal, except when the read comes before the write
                    const int top = (lrow || rbw) ? t - 1 : t;
                    float dz = 1.f;
                    if (h == 0 && top >= 32) dz = vg[V_Q32 / 4 + top];
                    const uint32_t pb = sb + ((cc & 1) ? OFF_PB1 : OFF_PB0);
#pragma unroll 1
                    for (int sub = 1; sub >= 0; --sub) {
                        const int col0 = 32 * h + 16 * sub;
                        float g[16];
                        tmem_ld16(tmem + lane_base + COL_G + col0, g);
                        const float4 *eta4 = reinterpret_cast<const float4 *>(vg + V_ETA / 4 + col0);
                        const float4 *gam4 = reinterpret_cast<const float4 *>(vg + V_GAM / 4 + col0);
#pragma unroll
                        for (int q = 3; q >= 0; --q) {
                            const float4 e4 = eta4[q], y4 = gam4[q];
                            const float ev[4] = {e4.x, e4.y, e4.z, e4.w};
                            const float yv[4] = {y4.x, y4.y, y4.z, y4.w};
#pragma unroll
                            for (int e = 3; e >= 0; --e) {
                                const int s2 = 4 * q + e;
                                const bool act = (col0 + s2) <= top;
                                g[s2] = act ? dz * ev[e] * g[s2] : 0.f;
                                if (act) dz *= yv[e];
                            }
                        }
                        if (lrow) {
#pragma unroll
                            for (int q = 0; q < 4; ++q)
                                *reinterpret_cast<float4 *>(Lw + t * 64 + ((((col0 >> 2) + q) ^ (t & 15)) << 2)) =
                                    make_float4(g[4 * q], g[4 * q + 1], g[4 * q + 2], g[4 * q + 3]);
                        } else {
                            st_row8_bf16(pb + sw128((uint32_t)t, (uint32_t)(col0 >> 3)), g);
                            st_row8_bf16(pb + sw128((uint32_t)t, (uint32_t)(col0 >> 3) + 1), g + 8);
                        }
                    }
                }
            }
            tc_fence_before();
            fence_proxy_async();
            if constexpr (falcon) {
                // each warp frees its rows of the Gram region; the phase that follows
                // starts with a group agreement, which orders L and P for every reader
                __syncwarp();
                if (early && cc + 1 < nch && lane == 0) mbar_arrive(bar(B_GGO));
            } else {
                gsync();
                if (early && cc + 1 < nch && kidx == 0) mbar_arrive(bar(B_GGO));   // the Gram region is free
            }
            if (kidx == 0) TRACE(cc, 3);
            return true;
        };
        if (!falcon) {
            // Falcon-1A: T = I.  Its bf16 copy (in both solve regions, which this
            // mode leaves unused) makes the key-path MMA warp's U^T = Y^T T^T the
            // Y^T the state path takes as R^T.
            if (gated) {
                const int t = kidx >> 2, q2 = 2 * (kidx & 3);
#pragma unroll
                for (int h8 = 0; h8 < 2; ++h8) {
                    float e[8];
#pragma unroll
                    for (int u = 0; u < 8; ++u) e[u] = (8 * (q2 + h8) + u == t) ? 1.f : 0.f;
                    const uint32_t off = sw128((uint32_t)t, (uint32_t)(q2 + h8));
                    st_row8_bf16(sb + lreg(0) + off, e);
                    st_row8_bf16(sb + lreg(1) + off, e);
                }
                fence_proxy_async();
            }
#pragma unroll 1
            for (int c = 0; c < nch && ok; ++c) {
                if (c > 0 && !early && !prep_go(c)) { ok = false; break; }
                if (!lp(c, nullptr)) { ok = false; break; }
                if (kidx == 0) {
                    if (gated) mbar_arrive(bar(B_TRDY));   // the (static) T of chunk c
                    mbar_arrive(bar(B_WRDY));
                }
            }
        }
        // Falcon-1 (phi = identity): L/P of chunk c+1 runs while the W/U products of
        // chunk c are in flight
#pragma unroll 1
        for (int c = -1; falcon && c < nch && ok; ++c) {
          // (c = -1 only forms L/P of chunk 0: the loop holds the one copy of lp)
          if (c >= 0) {
            float *vb = vec(c % NST);        // gate block
            const uint32_t tbo = lreg(c);    // L(c), then the bf16 T and -T diag(Gm) of chunk c
            float *Lf = reinterpret_cast<float *>(sm + tbo);
            float *Tf = reinterpret_cast<float *>(sm + lreg(c + 1));
            if (kidx == 0) TRACE(c, 4);
            // ---- T = (I + L)^{-1} in blocks of 16: fp32 forward substitution on the
            //      CUDA cores for the diagonal blocks (a dependent chain of warp-level
            //      tensor MMAs would queue behind the chunk MMAs on the shared tensor
            //      pipe), then T21 = -T22 L21 T11 at 16 -> 32 and 32 -> 64 on
            //      independent warp-level tf32 MMAs.  Tf's blocks above the diagonal
            //      blocks stay zero, so every product runs over whole blocks.
            if (h == 0 && lane < 16) {
                // diagonal block kw, column j, right-looking (the row updates of a step
                // are independent); the rows' 16-byte groups of L four columns at a time
                const int B0 = 16 * kw, j = lane;
                float x[16];
#pragma unroll
                for (int r = 0; r < 16; ++r) x[r] = (r == j) ? 1.f : 0.f;
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    float lk[16][4];
#pragma unroll
                    for (int r = 4 * k + 1; r < 16; ++r) {
                        const float4 v4 = *reinterpret_cast<const float4 *>(
                            Lf + (B0 + r) * 64 + ((((B0 >> 2) + k) ^ r) << 2));
                        lk[r][0] = v4.x; lk[r][1] = v4.y; lk[r][2] = v4.z; lk[r][3] = v4.w;
                    }
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int s2 = 4 * k + e;
#pragma unroll
                        for (int r = s2 + 1; r < 16; ++r) x[r] = fmaf(-lk[r][e], x[s2], x[r]);
                    }
                }
#pragma unroll
                for (int r = 0; r < 16; ++r) Tf[f64i(B0 + r, B0 + j)] = x[r];
            } else if (h == 1) {
                // T[0:16, 16:32] and T[32:48, 48:64] are zero (the merges read them)
                const int r = kt >> 2, c4 = 4 * (kt & 3);
                const int rr = (r < 16) ? r : 16 + r, cc4 = (r < 16) ? 16 + c4 : 48 + c4;
                *reinterpret_cast<float4 *>(Tf + f64i(rr, cc4)) = make_float4(0.f, 0.f, 0.f, 0.f);
            }
            // the first merge of pair p reads only the two diagonal blocks of the warps
            // (kw = 2p, 2p+1) that do it; the zero blocks are read after the next sync
            if (h == 0) {
                if (kw < 2) bar_sync(BAR_PAIR0, 64);
                else bar_sync(BAR_PAIR0 + 1, 64);
            }
            if (kidx == 0) TRACE(c, 5);
            const int gq = lane >> 2, tq = lane & 3;
            float t2b[4];        // phase-2 tile
            if (h == 0) {   // pairs (1,0) and (3,2): warp kw -> pair p, 8-column tile nt
                const int p = kw >> 1, nt = kw & 1;
                const int rb = 16 + 32 * p, cb = 32 * p;
                const int g = gq, t4 = tq;
                float m[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int ks = 0; ks < 2; ++ks) {
                    uint32_t fa[4], fb[2];
                    frag_a64(Lf, rb, cb + 8 * ks, lane, fa);
                    frag_b64(Tf, cb + 8 * ks, cb + 8 * nt, lane, fb);
                    mma_tf32_16x8x8(m, fa, fb);
                }
                float *Mw = Ms + 128 * kw;   // 16 x 8 per warp (the diagonal scratch is free)
                Mw[g * 8 + 2 * t4] = m[0];
                Mw[g * 8 + 2 * t4 + 1] = m[1];
                Mw[(g + 8) * 8 + 2 * t4] = m[2];
                Mw[(g + 8) * 8 + 2 * t4 + 1] = m[3];
                __syncwarp();
                float u[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int ks = 0; ks < 2; ++ks) {
                    uint32_t fa[4], fb[2];
                    frag_a64(Tf, rb, rb + 8 * ks, lane, fa);
                    fb[0] = __float_as_uint(Mw[(8 * ks + t4) * 8 + g]);
                    fb[1] = __float_as_uint(Mw[(8 * ks + t4 + 4) * 8 + g]);
                    mma_tf32_16x8x8(u, fa, fb);
                }
                const int c0 = cb + 8 * nt + 2 * t4;
                Tf[f64i(rb + g, c0)] = -u[0];
                Tf[f64i(rb + g, c0 + 1)] = -u[1];
                Tf[f64i(rb + g + 8, c0)] = -u[2];
                Tf[f64i(rb + g + 8, c0 + 1)] = -u[3];
            }
            gsync();
            if (kidx == 0) TRACE(c, 20);
            // second level: 32x32 tiles, one 16x8 tile per warp: row tile rt, column tile ct
            const int rt = kw >> 1, ct = 2 * (kw & 1) + h;
            {   // M2 = L[32:64, 0:32] T[0:32, 0:32]
                const int g = gq, t4 = tq;
                float m[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int ks = 0; ks < 4; ++ks) {
                    uint32_t fa[4], fb[2];
                    frag_a64(Lf, 32 + 16 * rt, 8 * ks, lane, fa);
                    frag_b64(Tf, 8 * ks, 8 * ct, lane, fb);
                    mma_tf32_16x8x8(m, fa, fb);
                }
                const int c0 = 8 * ct + 2 * t4;
                Ms[f32i(16 * rt + g, c0)] = m[0];
                Ms[f32i(16 * rt + g, c0 + 1)] = m[1];
                Ms[f32i(16 * rt + g + 8, c0)] = m[2];
                Ms[f32i(16 * rt + g + 8, c0 + 1)] = m[3];
            }
            gsync();
            if (kidx == 0) TRACE(c, 30);
            {   // T[32:64, 0:32] = -T[32:64, 32:64] M2
                float u[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int ks = 0; ks < 4; ++ks) {
                    uint32_t fa[4], fb[2];
                    frag_a64(Tf, 32 + 16 * rt, 32 + 8 * ks, lane, fa);
                    frag_b32(Ms, 8 * ks, 8 * ct, lane, fb);
                    mma_tf32_16x8x8(u, fa, fb);
                }
#pragma unroll
                for (int e = 0; e < 4; ++e) t2b[e] = -u[e];
            }
            {   // bf16 T and -T diag(Gm), K-major rows t, where L was (L is dead now)
                const float *gmv = vb + V_GM / 4;
                const int g = gq, t4 = tq;
                const int r2 = 32 + 16 * rt + g, c2 = 8 * ct + 2 * t4;
                auto put_t = [&](int r, int cc, float v0, float v1) {   // bf16 pair (r, cc..cc+1)
                    const uint32_t off = sw128((uint32_t)r, (uint32_t)cc >> 3) + ((uint32_t)(cc & 7) << 1);
                    st_shared_u32(sb + tbo + off, pack_bf16(v0, v1));
                    st_shared_u32(sb + tbo + 8 * KB + off, pack_bf16(-v0 * gmv[cc], -v1 * gmv[cc + 1]));
                };
                put_t(r2, c2, t2b[0], t2b[1]);
                put_t(r2 + 8, c2, t2b[2], t2b[3]);
                // the rest from Tf: row t, columns 16q..16q+15 (rows 32.., columns ..31 are T21 above)
                const int t = kidx >> 2, q = kidx & 3;
                if (t < 32 || q >= 2) {
                    const bool zero = (t < 32 && q >= 2);   // above the diagonal 32-blocks
                    const float4 *gm4 = reinterpret_cast<const float4 *>(gmv) + 4 * q;
                    float tv[16], tp[16];
#pragma unroll
                    for (int e4 = 0; e4 < 4; ++e4) {
                        const float4 v4 = zero ? make_float4(0.f, 0.f, 0.f, 0.f)
                                               : *reinterpret_cast<const float4 *>(Tf + f64i(t, 16 * q + 4 * e4));
                        const float4 g4 = gm4[e4];
                        tv[4 * e4] = v4.x; tv[4 * e4 + 1] = v4.y; tv[4 * e4 + 2] = v4.z; tv[4 * e4 + 3] = v4.w;
                        tp[4 * e4] = -v4.x * g4.x; tp[4 * e4 + 1] = -v4.y * g4.y;
                        tp[4 * e4 + 2] = -v4.z * g4.z; tp[4 * e4 + 3] = -v4.w * g4.w;
                    }
#pragma unroll
                    for (int h8 = 0; h8 < 2; ++h8) {
                        const uint32_t off = sw128((uint32_t)t, (uint32_t)(2 * q + h8));
                        st_row8_bf16(sb + tbo + off, tv + 8 * h8);
                        st_row8_bf16(sb + tbo + 8 * KB + off, tp + 8 * h8);
                    }
                }
            }
            // each warp publishes its part of T (the next phase's leading group
            // agreement keeps L(c+1) from landing on the fp32 T before all have read it)
            fence_proxy_async();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(B_TRDY));
            if (kidx == 0) TRACE(c, 6);
          }
            if (c + 1 < nch && !lp(c + 1, reinterpret_cast<float *>(sm + lreg(c + 1)))) {
                ok = false;   // (for c >= 0: T(c) fp32 is dead)
                break;
            }
            if (c < 0) {
                gsync();   // L(0) complete before the first solve reads it
                continue;
            }

            // ---- -W^T -> bf16 rows i, once W^T(c) is done and R(c-1) has read the old one
            {
                bool w = wait_bar(bar(B_WUDONE), (uint32_t)c & 1u, limit, s_abort);
                w = w && (c < 1 || wait_bar(bar(B_RDONE), (uint32_t)(c - 1) & 1u, limit, s_abort));
                if (bar_or(BAR_KG, KGROUP, !w)) { ok = false; break; }
            }
            if (kidx == 0) TRACE(c, 8);
            tc_fence_after();
            {
                float w[32];
                tmem_ld32(tmem + lane_base + COL_W + 32 * h, w);
#pragma unroll
                for (int c16 = 0; c16 < 4; ++c16)
                    st_row8_bf16(sb + OFF_WTB + sw128(kt, 4 * h + c16), w + 8 * c16);
            }
            tc_fence_before();
            fence_proxy_async();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(B_WRDY));   // each warp its rows of -W^T
            if (kidx == 0) TRACE(c, 9);
        }
        if (!ok && kidx == 0) fail_now();
    } else if (warp >= SG_W0 && warp < KG2_W0) {
        // ================================================================ state group
        const int srow = tid - SG_W0 * 32;         // == TMEM lane of this thread
        // the final state: S_T, or (two segments) this role's slot of the workspace
        float *const sdst = segs ? a.s_aux + (int64_t)role * a.n_chains * D * D : a.S_T;
        const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
        auto gwait = [&](uint32_t bb, uint32_t parity) -> bool {
            const bool ok = wait_bar(bb, parity, limit, s_abort);
            return !bar_or(BAR_SG, GROUP, !ok);
        };
        bool ok = true;

        // bf16 copy of 32 state entries (i = i0 .. i0+31 of column j): the A operand
        // of R and O1 holds two consecutive i per column, the even one low
        auto put_sb = [&](int i0, const float *v) {
            float pk[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) pk[e] = __uint_as_float(pack_bf16(v[2 * e], v[2 * e + 1]));
            tmem_st16(tmem + lane_base + COL_SB + (uint32_t)(i0 / 2), pk);
        };

        // initial state, transposed (this thread holds column j = srow of S):
        // TMEM <- G_{C-1}(chunk 0) S0^T, and the bf16 copy
        float gC0 = 1.f;
        if (gated) {
            if (!gwait(bar(B_GV0), 0)) ok = false;
            else gC0 = vec(0)[V_GC / 4];
        }
        if (ok) {
#pragma unroll 1
            for (int q = 0; q < 4; ++q) {   // i = 32q .. 32q+31
                float v[32];
#pragma unroll
                for (int e = 0; e < 32; ++e)
                    v[e] = role == 2 ? (32 * q + e == srow ? 1.f : 0.f)
                         : (role == 0 && a.S0) ? a.S0[(chain * D + 32 * q + e) * D + srow] : 0.f;
                put_sb(32 * q, v);
#pragma unroll
                for (int e = 0; e < 32; ++e) v[e] *= gC0;
                tmem_st16(tmem + lane_base + COL_S + 32 * q, v);
                tmem_st16(tmem + lane_base + COL_S + 32 * q + 16, v + 16);
            }
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {   // each warp its lanes of the state (bf16 copy, scaled fp32)
                mbar_arrive(bar(B_SRDY));
                if (SPLIT_CARRY) mbar_arrive(bar(B_SSCL));
            }
        }

#pragma unroll 1
        for (int c = 0; c < nch && ok; ++c) {
            const int b = c % NST;   // gate block
            const int64_t tok0 = (int64_t)c * C;
            if (gated) {
                // ---- R^T -> bf16 rows j (A operand) and diag(w)-scaled copy (B operand)
                if (srow == 0) TRACE(c, 31);
                {
                    bool w = wait_bar(bar(B_RDONE), (uint32_t)c & 1u, limit, s_abort);
                    w = w && wait_bar(bar(B_GV0 + b), (uint32_t)(c / NST) & 1u, limit, s_abort);
                    if (bar_or(BAR_SG, GROUP, !w)) { ok = false; break; }
                }
                if (srow == 0) TRACE(c, 10);
                tc_fence_after();
                const float *wc = vec(b) + V_WC / 4;
                if (srow < C)   // the gate warp may recycle this gate block once S(c) is done
                    reinterpret_cast<float *>(sm + OFF_SGV)[srow] =
                        vec(b)[(rbw ? V_GM : V_G) / 4 + srow];   // G_{t-1} for a read before the write
#pragma unroll 1
                for (int q = 0; q < 4; ++q) {   // columns t = 16q .. 16q+15
                    float r[16];
                    tmem_ld16(tmem + lane_base + COL_R + 16 * q, r);
#pragma unroll
                    for (int c8 = 0; c8 < 2; ++c8) {
                        const float4 w0 = *reinterpret_cast<const float4 *>(wc + 16 * q + 8 * c8);
                        const float4 w1 = *reinterpret_cast<const float4 *>(wc + 16 * q + 8 * c8 + 4);
                        const float *rr = r + 8 * c8;
                        const float w8[8] = {rr[0] * w0.x, rr[1] * w0.y, rr[2] * w0.z, rr[3] * w0.w,
                                             rr[4] * w1.x, rr[5] * w1.y, rr[6] * w1.z, rr[7] * w1.w};
                        st_row8_bf16(sb + OFF_RA + sw128(srow, 2 * q + c8), rr);
                        st_row8_bf16(sb + OFF_RB + sw128(srow, 2 * q + c8), w8);
                    }
                }
                // each warp publishes its rows of R (the state carry that follows
                // starts with a group agreement)
                tc_fence_before();
                fence_proxy_async();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(bar(B_RRDY));
                    mbar_arrive(bar(B_RFREE));
                }
                if (srow == 0) TRACE(c, 11);
            }

            // ---- state carry
            const bool last = (c + 1 == nch);
            {
                bool w = wait_bar(bar(B_SDONE), (uint32_t)c & 1u, limit, s_abort);
                if (gated && !last)
                    w = w && wait_bar(bar(B_GV0 + (c + 1) % NST), (uint32_t)((c + 1) / NST) & 1u,
                                      limit, s_abort);
                if (bar_or(BAR_SG, GROUP, !w)) { ok = false; break; }
            }
            if (srow == 0) TRACE(c, 12);
            tc_fence_after();
            const float gC_next = (gated && !last) ? vec((c + 1) % NST)[V_GC / 4] : 1.f;
            if (last) {
#pragma unroll 1
                for (int q = 0; q < 4; ++q) {   // S_T[i][j], consecutive j across the warp
                    float v[32];
                    tmem_ld32(tmem + lane_base + COL_S + 32 * q, v);
#pragma unroll
                    for (int e = 0; e < 32; ++e) sdst[(chain * D + 32 * q + e) * D + srow] = v[e];
                    if (segs && role == 0) {   // and row j of S_mid^T in bf16, for the fix-up's products
                        uint4 *bt = reinterpret_cast<uint4 *>(reinterpret_cast<__nv_bfloat16 *>(
                                        a.s_aux + 3 * a.n_chains * D * D) + (chain * D + srow) * D + 32 * q);
#pragma unroll
                        for (int u = 0; u < 4; ++u)
                            bt[u] = make_uint4(pack_bf16(v[8 * u], v[8 * u + 1]), pack_bf16(v[8 * u + 2], v[8 * u + 3]),
                                               pack_bf16(v[8 * u + 4], v[8 * u + 5]), pack_bf16(v[8 * u + 6], v[8 * u + 7]));
                    }
                }
            } else if constexpr (SPLIT_CARRY) {
                // (few chains: the state path's latency sets the period)
                // the bf16 copy first: the next chunk's R^T and O1 wait only for it
#pragma unroll 1
                for (int q = 0; q < 4; ++q) {
                    float v[32];
                    tmem_ld32(tmem + lane_base + COL_S + 32 * q, v);
                    if (srow == 0 && q == 0) TRACE(c, 23);
                    put_sb(32 * q, v);
                }
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(B_SRDY));   // each warp its lanes
                TRACEW(c, 3);
                if (srow == 0) TRACE(c, 13);
                // then the fp32 state pre-scaled by the next chunk's total decay, which
                // the next chunk's S update waits for (linear attention: no decay)
                if (gated) {
#pragma unroll 1
                    for (int q = 0; q < 4; ++q) {
                        float v[32];
                        tmem_ld32(tmem + lane_base + COL_S + 32 * q, v);
#pragma unroll
                        for (int e = 0; e < 32; ++e) v[e] *= gC_next;
                        tmem_st16(tmem + lane_base + COL_S + 32 * q, v);
                        tmem_st16(tmem + lane_base + COL_S + 32 * q + 16, v + 16);
                    }
                    tmem_st_wait();
                    tc_fence_before();
                    __syncwarp();
                }
                if (lane == 0) mbar_arrive(bar(B_SSCL));
            } else {
                // (many chains: fewer TMEM round trips)
                // one TMEM round trip per 32 columns: the bf16 copy and the fp32 state
                // pre-scaled by the next chunk's total decay (linear attention: no decay)
#pragma unroll 1
                for (int q = 0; q < 4; ++q) {
                    float v[32];
                    tmem_ld32(tmem + lane_base + COL_S + 32 * q, v);
                    if (srow == 0 && q == 0) TRACE(c, 23);
                    put_sb(32 * q, v);
                    if (gated) {
#pragma unroll
                        for (int e = 0; e < 32; ++e) v[e] *= gC_next;
                        tmem_st16(tmem + lane_base + COL_S + 32 * q, v);
                        tmem_st16(tmem + lane_base + COL_S + 32 * q + 16, v + 16);
                    }
                }
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(B_SRDY));   // each warp its lanes
                TRACEW(c, 3);
                if (srow == 0) TRACE(c, 13);
            }

            // ---- outputs o_t = G_t (S0^T q_t) + (P R)_t, bf16, thread j writing column
            //      j of each token's row (rows past T are not written); each warp then
            //      frees its lanes of O1 and O2 for the next chunk's products
            {
                const float *gv = reinterpret_cast<const float *>(sm + OFF_SGV);
                __nv_bfloat16 *ot = role == 2
                    ? reinterpret_cast<__nv_bfloat16 *>(a.o_aux) + (chain * T + tok0) * D + srow
                    : reinterpret_cast<__nv_bfloat16 *>(a.o) + (chain * T_all + t_base + tok0) * D + srow;
                const int tlim = T - tok0 < (int64_t)C ? (int)(T - tok0) : C;
#pragma unroll 1
                for (int h = 0; h < 4; ++h) {   // (a rolled loop: short code beside the other roles')
                    float o1[16], o2[16];
                    tmem_ld16(tmem + lane_base + COL_O1 + 16 * h, o1);
                    tmem_ld16(tmem + lane_base + COL_O2 + 16 * h, o2);
#pragma unroll
                    for (int e4 = 0; e4 < 4; ++e4) {
                        const float4 g4 = gated ? *reinterpret_cast<const float4 *>(gv + 16 * h + 4 * e4)
                                                 : make_float4(1.f, 1.f, 1.f, 1.f);
                        const float gg[4] = {g4.x, g4.y, g4.z, g4.w};
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const int t = 16 * h + 4 * e4 + e;
                            if (t < tlim) ot[t * D] = __float2bfloat16_rn(fmaf(gg[e], o1[4 * e4 + e], o2[4 * e4 + e]));
                        }
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(B_OFREE));   // each warp its lanes of O1, O2
        }
        if (!ok && srow == 0) fail_now();
    }

    // every role meets here; tensor memory is released last
    tc_fence_before();
    __syncthreads();
    if (warp == 3) {
        tc_fence_after();
        tmem_dealloc(tmem, TMEM_COLS);
    }
}

// ---------------------------------------------------------------- two segments
// Second kernel of the two-segment form.  The state map over the second segment is
// affine in its initial state: S_t = Phi_t S_mid + S_t^0, so the true outputs are
// o_t = o_t^0 + S_mid^T (Phi_t^T q_t) (the zero-start run wrote o_t^0 in place, the
// transition run Phi_t^T q_t to the workspace) and S_T = Phi_T S_mid + S_T^0.
// m CTAs per chain, two per SM: CTA k of a chain forms rows k, k + m, ... of S_T
// in fp32, then stages S_mid^T (bf16, written by the first segment's CTA) once and
// takes the chain's 64-token tiles k, k + m, ...: the next tile's Phi_t^T q_t and o
// rows arrive by cp.async into the other of two buffers while a tile is worked on;
// the product runs on warp-level bf16 MMAs (fp32 accumulation) and is added into
// the staged o rows in shared memory, which then go out in whole rows.
constexpr int FX_THREADS = 256, FX_ROWS = 64;
constexpr int FX_LDB = 136;   // bf16 row stride of S_mid^T and the tiles (128 + 8)
constexpr uint32_t FX_TILE = (uint32_t)(FX_ROWS * FX_LDB * 2);
constexpr uint32_t FX_SMEM = (uint32_t)(D * FX_LDB * 2) + 4 * FX_TILE;

__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

__global__ void __launch_bounds__(FX_THREADS, 2)
segment_fixup_kernel(const PrefillArgs a, int m) {
    extern __shared__ __align__(16) uint8_t fsm[];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int64_t n = a.n_chains, T_all = a.T, T1 = T_all - a.seg_t0;
    const float *Smid = a.s_aux, *Sz = a.s_aux + n * D * D, *Phi = a.s_aux + 2 * n * D * D;
    const __nv_bfloat16 *SmidT = reinterpret_cast<const __nv_bfloat16 *>(a.s_aux + 3 * n * D * D);
    const int64_t chain = (int64_t)blockIdx.x / m;
    const int k = (int)((int64_t)blockIdx.x % m);
    // [j][i] = S_mid[i][j]; then two buffers of (Phi_t^T q_t [t][i], o [t][j])
    __nv_bfloat16 *sS = reinterpret_cast<__nv_bfloat16 *>(fsm);
    const uint32_t sS_u = smem_u32(sS), sT_u = sS_u + (uint32_t)(D * FX_LDB * 2);
    auto q_tile = [&](int buf) { return sT_u + (uint32_t)(2 * buf) * FX_TILE; };
    auto o_tile = [&](int buf) { return sT_u + (uint32_t)(2 * buf + 1) * FX_TILE; };
    __nv_bfloat16 *const o_seg = reinterpret_cast<__nv_bfloat16 *>(a.o) + (chain * T_all + a.seg_t0) * D;

    for (int idx = tid; idx < D * 16; idx += FX_THREADS)   // 16-byte pieces of the rows j
        cp_async16(sS_u + (uint32_t)(((idx >> 4) * FX_LDB + 8 * (idx & 15)) * 2),
                   SmidT + (chain * D + (idx >> 4)) * D + 8 * (idx & 15));
    cp_async_commit();
    const int64_t ntile = (T1 + FX_ROWS - 1) / FX_ROWS;
    auto load_tile = [&](int64_t tile, int buf) {   // rows past the segment's end are not read
        const int64_t t0 = tile * FX_ROWS;
        const __nv_bfloat16 *oa = reinterpret_cast<const __nv_bfloat16 *>(a.o_aux) + (chain * T1 + t0) * D;
        const __nv_bfloat16 *oo = o_seg + t0 * D;
        for (int idx = tid; idx < FX_ROWS * 16; idx += FX_THREADS) {
            const int r = idx >> 4, c8 = idx & 15;
            if (t0 + r >= T1) continue;
            const uint32_t off = (uint32_t)((r * FX_LDB + 8 * c8) * 2);
            cp_async16(q_tile(buf) + off, oa + (int64_t)r * D + 8 * c8);
            cp_async16(o_tile(buf) + off, oo + (int64_t)r * D + 8 * c8);
        }
        cp_async_commit();
    };
    if (k < ntile) load_tile(k, 0);

    // S_T = Phi_T S_mid + S_T^0, rows i = k, k + m, ...: thread (row slot, 8 columns);
    // latency-bound, so half the CTAs form it before their tiles and half after
    auto state_rows = [&]() {
        const int j0 = 8 * (tid & 15);
        for (int i = k + m * (tid >> 4); i < D; i += m * (FX_THREADS >> 4)) {
            const float *ph = Phi + (chain * D + i) * D;
            const float *sm0 = Smid + chain * D * D + j0;
            const float4 z0 = *reinterpret_cast<const float4 *>(Sz + (chain * D + i) * D + j0);
            const float4 z1 = *reinterpret_cast<const float4 *>(Sz + (chain * D + i) * D + j0 + 4);
            float acc[8] = {z0.x, z0.y, z0.z, z0.w, z1.x, z1.y, z1.z, z1.w};
#pragma unroll 8
            for (int kk = 0; kk < D; ++kk) {
                const float p = ph[kk];
                const float4 v0 = *reinterpret_cast<const float4 *>(sm0 + (int64_t)kk * D);
                const float4 v1 = *reinterpret_cast<const float4 *>(sm0 + (int64_t)kk * D + 4);
                acc[0] = fmaf(p, v0.x, acc[0]); acc[1] = fmaf(p, v0.y, acc[1]);
                acc[2] = fmaf(p, v0.z, acc[2]); acc[3] = fmaf(p, v0.w, acc[3]);
                acc[4] = fmaf(p, v1.x, acc[4]); acc[5] = fmaf(p, v1.y, acc[5]);
                acc[6] = fmaf(p, v1.z, acc[6]); acc[7] = fmaf(p, v1.w, acc[7]);
            }
            float4 *dst = reinterpret_cast<float4 *>(a.S_T + (chain * D + i) * D + j0);
            dst[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
            dst[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
        }
    };
    if (!(k & 1)) state_rows();

    const int mt = warp & 3, nh = warp >> 2, g = lane >> 2, t4 = lane & 3;
    int buf = 0;
    for (int64_t tile = k; tile < ntile; tile += m, buf ^= 1) {
        if (tile + m < ntile) {
            load_tile(tile + m, buf ^ 1);
            cp_async_wait<1>();
        } else {
            cp_async_wait<0>();
        }
        __syncthreads();   // this tile (and S_mid^T) landed for every thread
        // warp: rows 16 mt .. +15, columns 64 nh .. +63, k = i in 8 steps of 16
        const __nv_bfloat16 *tq = sS + (D + 2 * buf * FX_ROWS) * FX_LDB;   // the q tile of buf
        float acc[8][4];
#pragma unroll
        for (int nt = 0; nt < 8; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[nt][e] = 0.f;
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
            uint32_t fa[4];
            const int ar = 16 * mt + (lane & 7) + 8 * ((lane >> 3) & 1), ac = 16 * ks + 8 * (lane >> 4);
            ldmatrix_x4(smem_u32(tq + ar * FX_LDB + ac), fa);
#pragma unroll
            for (int nt = 0; nt < 8; ++nt) {
                const __nv_bfloat16 *bp = sS + (64 * nh + 8 * nt + g) * FX_LDB + 16 * ks + 2 * t4;
                mma_bf16_16x8x16(acc[nt], fa[0], fa[1], fa[2], fa[3], *reinterpret_cast<const uint32_t *>(bp),
                                 *reinterpret_cast<const uint32_t *>(bp + 8));
            }
        }
        // o_t^0 + the product, in place in the staged o rows (each element one thread's)
        __nv_bfloat16 *to = sS + (D + (2 * buf + 1) * FX_ROWS) * FX_LDB;
#pragma unroll
        for (int nt = 0; nt < 8; ++nt) {
            const int j = 64 * nh + 8 * nt + 2 * t4, r = 16 * mt + g;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                uint32_t *pp = reinterpret_cast<uint32_t *>(to + (r + 8 * h) * FX_LDB + j);
                const float2 f = unpack_bf16(*pp);
                *pp = pack_bf16(f.x + acc[nt][2 * h], f.y + acc[nt][2 * h + 1]);
            }
        }
        __syncthreads();   // the sums are in place; this buffer is free for the prefetch after next
        const int64_t t0 = tile * FX_ROWS;
        for (int idx = tid; idx < FX_ROWS * 16; idx += FX_THREADS) {   // whole rows, 16 bytes a thread
            const int r = idx >> 4, c8 = idx & 15;
            if (t0 + r >= T1) continue;
            *reinterpret_cast<uint4 *>(o_seg + (t0 + r) * D + 8 * c8) =
                *reinterpret_cast<const uint4 *>(to + r * FX_LDB + 8 * c8);
        }
        __syncthreads();   // the rows are out before the next prefetch lands in this buffer
    }
    if (k & 1) state_rows();
    cp_async_wait<0>();   // no copy in flight at exit
}

// Private stream-ordered pool for the two-segment workspace, one per device; it
// keeps its memory between calls.
cudaMemPool_t segment_pool(int dev) {
    static std::mutex m;
    static cudaMemPool_t pools[64] = {};
    if (dev < 0 || dev >= 64) return nullptr;
    std::lock_guard<std::mutex> lock(m);
    if (!pools[dev]) {
        cudaMemPoolProps props = {};
        props.allocType = cudaMemAllocationTypePinned;
        props.location.type = cudaMemLocationTypeDevice;
        props.location.id = dev;
        cudaMemPool_t p = nullptr;
        if (cudaMemPoolCreate(&p, &props) != cudaSuccess) {
            cudaGetLastError();
            return nullptr;
        }
        uint64_t keep = UINT64_MAX;
        cudaMemPoolSetAttribute(p, cudaMemPoolAttrReleaseThreshold, &keep);
        pools[dev] = p;
    }
    return pools[dev];
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

// [n_chains][T][128] bf16 viewed as a 3-D tensor (d, T, chain); 64 x 64 boxes with
// the 128-byte swizzle for the tile loads.
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

// Falcon-1 and Falcon-1A with phi = elu+1 are declined: phi(k) is close to
// 1 + k for small keys, and rounding it to a bf16 MMA operand erases most of
// the key's varying part, which the normalised step and the residual write
// depend on (the per-token kernel keeps it in fp32).  Linear attention
// accumulates phi(k) additively and keeps bf16 operand accuracy.
bool chunked_supported(const PrefillArgs &a) {
    if (a.mode != FW_LINATTN && a.phi == FW_PHI_ELU1) return false;
    // a step per value channel gives every channel its own triangular system:
    // Falcon-2 / 2A run on the per-channel chunked kernel (or the per-token one)
    if (a.mode == FW_FALCON2 || a.mode == FW_FALCON2A) return false;
    return a.dtype == FW_BF16 && a.d == D && a.T <= (int64_t)INT32_MAX - C &&
           a.n_chains <= (int64_t)INT32_MAX;
}

#ifdef FW_TRACE
extern "C" int fw_debug_read_trace(unsigned long long *dst, int n) {
    if (n > kTraceChunks * (kTraceEv + 64)) n = kTraceChunks * (kTraceEv + 64);
    return (int)cudaMemcpyFromSymbol(dst, g_trace, sizeof(unsigned long long) * n);
}
#endif

// The two-segment plan: the split token (0: one segment), the workspace bytes and
// the offset of the states in it.  The chain splits at the chunk boundary nearest
// T/2 when at most a third of the SMs hold a chain and T >= 4096, or as the test
// hook asks.
static int64_t segment_plan(const PrefillArgs &a, int sms, size_t *bytes, size_t *n_o) {
    const int64_t nchk = (a.T + C - 1) / C;
    *bytes = 0;
    *n_o = 0;
    if (a.seg_pref < 0 || nchk < 2 ||
        !(a.seg_pref > 0 || (3 * a.n_chains <= (int64_t)sms && a.T >= 4096)))
        return 0;
    const int64_t t0 = (int64_t)C * (nchk / 2);
    *n_o = (size_t)a.n_chains * (size_t)(a.T - t0) * D * 2;   // a multiple of 256
    // S_mid, S_T from zero and Phi_T in fp32, then S_mid^T in bf16
    *bytes = *n_o + (size_t)3 * (size_t)a.n_chains * D * D * 4 + (size_t)a.n_chains * D * D * 2;
    return t0;
}

size_t chunked_segment_bytes(const PrefillArgs &a, int sms) {
    size_t bytes = 0, n_o = 0;
    segment_plan(a, sms, &bytes, &n_o);
    return bytes;
}

cudaError_t launch_chunked(const PrefillArgs &a, cudaStream_t s) {
    CUtensorMap tq, tk, tv;
    if (!make_map(&tq, a.q, a.T, a.n_chains) || !make_map(&tk, a.k, a.T, a.n_chains) ||
        !make_map(&tv, a.v, a.T, a.n_chains))
        return cudaErrorInvalidValue;
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
        return e;
    // Few long chains: each runs as two segments at once (three CTAs per chain).
    // The workspace comes from the private pool, or (fw_prefill_noalloc) from the
    // static buffer, whose size the API has checked.
    PrefillArgs b = a;
    void *ws = nullptr;   // from the pool: freed after the launches
    size_t need = 0, n_o = 0;
    const int64_t t0 = segment_plan(a, sms, &need, &n_o);
    if (t0 > 0) {
        void *base = nullptr;
        if (a.scratch_only) {
            if (!a.scratch || need > a.scratch_bytes) return cudaErrorInvalidValue;
            base = a.scratch;
        } else {
            cudaMemPool_t pool = segment_pool(dev);
            if (pool && cudaMallocFromPoolAsync(&ws, need, pool, s) == cudaSuccess) {
                base = ws;
            } else {
                cudaGetLastError();   // no workspace: the call runs unsplit
                ws = nullptr;
            }
        }
        if (base) {
            b.seg_t0 = t0;
            b.o_aux = base;
            b.s_aux = reinterpret_cast<float *>(static_cast<char *>(base) + n_o);
        }
    }
    const int64_t ctas = b.seg_t0 > 0 ? 3 * a.n_chains : a.n_chains;
    // With CTAs on at most about 55 % of the SMs (one per SM), the state path's
    // serial chain sets each chain's period, and the decay scaling of the state
    // moves off it (measured crossover between 80 and 96 chains on 152 SMs).
    const bool split = 20 * ctas <= 11 * (int64_t)sms;
    const bool segs = b.seg_t0 > 0;
    auto kern = a.mode == FW_LINATTN
                    ? (segs ? chunked_kernel<false, false, false, true> : chunked_kernel<false, false, false, false>)
              : a.mode == FW_FALCON1
                    ? (split ? (segs ? chunked_kernel<true, true, true, true> : chunked_kernel<true, true, true, false>)
                             : (segs ? chunked_kernel<true, true, false, true> : chunked_kernel<true, true, false, false>))
                    : (split ? (segs ? chunked_kernel<true, false, true, true> : chunked_kernel<true, false, true, false>)
                             : (segs ? chunked_kernel<true, false, false, true> : chunked_kernel<true, false, false, false>));
    if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  (int)SMEM_ALLOC)) == cudaSuccess) {
        kern<<<(unsigned)ctas, NTHREADS, SMEM_ALLOC, s>>>(tq, tk, tv, b);
        e = cudaGetLastError();
    }
    if (e == cudaSuccess && b.seg_t0 > 0) {
        // two CTAs per SM, an equal number per chain
        const int64_t ntile = (a.T - b.seg_t0 + FX_ROWS - 1) / FX_ROWS;
        int64_t m = 2 * (int64_t)sms / a.n_chains;
        if (m > ntile) m = ntile;
        if (m < 1) m = 1;
        e = cudaFuncSetAttribute(segment_fixup_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)FX_SMEM);
        if (e == cudaSuccess) {
            segment_fixup_kernel<<<(unsigned)(a.n_chains * m), FX_THREADS, FX_SMEM, s>>>(b, (int)m);
            e = cudaGetLastError();
        }
    }
    if (ws) {
        const cudaError_t ef = cudaFreeAsync(ws, s);
        if (e == cudaSuccess) e = ef;
    }
    return e;
}

}  // namespace fw
