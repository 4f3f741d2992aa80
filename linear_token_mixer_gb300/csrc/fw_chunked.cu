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
//               128-byte swizzle; X/Q double-buffered.
//   warp 1      key-path MMA issuer:  G = [X;Q] X^T, W^T = X^T (T diag Gm)^T,
//               U^T = Y^T T^T.
//   warp 2      state-path MMA issuer: R^T = U^T - S^T W^T, O1^T = S^T Q^T,
//               O2^T = R^T P^T, S += X^T (diag(w) R).
//   warp 3      tensor-memory allocation.
//   warps 4-7   key group: feature map, gates and decay products, L and P from
//               G, the triangular solve, -W^T staging.
//   warps 8-11  state group: R staging, state carry (fp32 in tensor memory,
//               bf16 copy in shared memory as the MMA operand), outputs
//               o_t = G_t O1_t + O2_t.
// All products are tcgen05 MMAs with M = 128 (transposed forms keep d on the
// M side), bf16 operands in shared memory and fp32 accumulators in tensor
// memory.  The triangular solve runs on warp-level tf32 MMAs: each 16x16
// diagonal block as the exact nilpotent product (I-L)(I+L^2)(I+L^4)(I+L^8),
// then two levels of block merges T_ba = -T_bb L_ba T_aa.  Every
// wait is bounded: on expiry the kernel records an error, the other roles
// stop at their next wait, copies and MMAs in flight are drained, tensor
// memory is freed and the kernel exits.
#include <cudaTypedefs.h>

#include <mutex>

#include "fw_internal.cuh"
#include "fw_sm100.cuh"

namespace fw {
namespace {
using namespace sm100;

constexpr int C = 64;        // chunk length
constexpr int D = 128;       // d_k = d_v
constexpr int NTHREADS = 384;
constexpr int KG_W0 = 4;     // first warp of the key group
constexpr int SG_W0 = 8;     // first warp of the state group
constexpr int BAR_KG = 1, BAR_SG = 2;
constexpr int GROUP = 128;

constexpr uint32_t KB = 1024;
// shared memory (offsets from a 1024-aligned base)
constexpr uint32_t OFF_XQ0 = 0, OFF_XQ1 = 32 * KB;   // X0 Q0 X1 Q1 (8 KB each)
constexpr uint32_t XQ_X0 = 0, XQ_Q0 = 8 * KB, XQ_X1 = 16 * KB, XQ_Q1 = 24 * KB;
constexpr uint32_t OFF_Y0 = 64 * KB;   // V tile (Falcon-1: the only one; linattn: stage 0)
constexpr uint32_t OFF_Y1 = 80 * KB;   // linattn: V of stage 1; Falcon-1: L (fp32), then T
constexpr uint32_t OFF_LF = OFF_Y1;            // L, fp32 64x64, 16-byte-group swizzle
constexpr uint32_t OFF_TB = OFF_Y1;            // T, bf16, K-major rows t (after L is dead)
constexpr uint32_t OFF_TPB = OFF_Y1 + 8 * KB;  // T diag(Gm), bf16
constexpr uint32_t OFF_PB0 = 96 * KB, OFF_PB1 = 104 * KB;   // P, bf16, K-major rows t
constexpr uint32_t OFF_WTB = 112 * KB;  // -W^T, bf16, rows i (MN-major B operand)
constexpr uint32_t OFF_RA = 128 * KB;   // R^T, bf16, rows j (K-major A operand)
constexpr uint32_t OFF_RB = 144 * KB;   // (diag(w) R)^T, bf16, rows j (K-major B operand)
constexpr uint32_t OFF_SB = 160 * KB;   // S, bf16, rows i, two 64-column blocks (16 KB each)
constexpr uint32_t OFF_TF = 192 * KB;   // T, fp32 64x64, swizzled
constexpr uint32_t OFF_MS = 208 * KB;   // solver scratch: 4 x 2 KB per-warp 16x16 pairs, or 32x32
constexpr uint32_t OFF_VEC = 216 * KB;  // two gate blocks of 1536 B
constexpr uint32_t VEC_BYTES = 1536;
constexpr uint32_t V_ETA = 0, V_GAM = 256, V_G = 512, V_GM = 768, V_WC = 1024, V_GC = 1280;
constexpr uint32_t OFF_BAR = OFF_VEC + 2 * VEC_BYTES;
constexpr uint32_t OFF_MISC = OFF_BAR + 32 * 8;
constexpr uint32_t OFF_SGV = OFF_MISC + 64;    // G_t of the chunk the state group is on
constexpr uint32_t SMEM_BYTES = OFF_SGV + 256;
constexpr uint32_t SMEM_ALLOC = SMEM_BYTES + 1024;
static_assert(SMEM_ALLOC <= 227 * KB, "shared memory budget");

// mbarriers
enum {
    B_FULL0 = 0, B_FULL1, B_EMPTY0, B_EMPTY1, B_FULLY, B_YFREE, B_GGO, B_GDONE, B_TRDY,
    B_WUDONE, B_WRDY, B_GV0, B_GV1, B_PFREE0, B_PFREE1, B_SRDY, B_RDONE, B_RRDY, B_SDONE,
    B_OFREE, B_RFREE0, B_RFREE1, B_KDRAIN, B_SDRAIN, B_NEVER, B_COUNT
};
static_assert(B_COUNT <= 32, "barrier area");

// tensor-memory columns (128 lanes x 32 bit)
constexpr uint32_t COL_G = 0, COL_W = 64, COL_R0 = 128, COL_O1 = 256, COL_O2 = 320, COL_S = 384;
constexpr uint32_t TMEM_COLS = 512;

constexpr uint64_t kDrainNs = 2000000000ull;

// Optional phase timestamps of CTA 0 (instrumented builds only).
#ifdef FW_TRACE
constexpr int kTraceEv = 32, kTraceChunks = 64;
__device__ unsigned long long g_trace[kTraceChunks * kTraceEv];
#define TRACE(c, ev) \
    do { if (blockIdx.x == 0 && (c) < kTraceChunks) g_trace[(c) * kTraceEv + (ev)] = globaltimer(); } while (0)
#else
#define TRACE(c, ev) do { } while (0)
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

// Bounded wait for the single-thread roles (producer, MMA issuers): polls
// without parking, so a hand-off is seen as soon as it lands.
__device__ __forceinline__ bool wait_fast(uint32_t bar, uint32_t parity, uint64_t limit,
                                          volatile int *abort_flag) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer();
    for (;;) {
        if (mbar_try_wait(bar, parity)) return true;
        if (*abort_flag) return false;
        if (globaltimer() - t0 > limit) return false;
    }
}

// Bounded wait that also gives up as soon as another role has aborted.
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, uint64_t limit,
                                         volatile int *abort_flag) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer();
    for (;;) {
        // parked until the phase completes (or ~100 us pass): no issue slots spent
        if (mbar_try_wait_sleep(bar, parity, 100000u)) return true;
        if (*abort_flag) return false;
        if (globaltimer() - t0 > limit) return false;
    }
}

// tf32 fragments of a 16x8 A tile / 8x8 B tile of a swizzled fp32 matrix.
__device__ __forceinline__ void frag_a64(const float *M, int r0, int k0, int lane, uint32_t (&a)[4]) {
    const int g = lane >> 2, t = lane & 3;
    a[0] = f2tf32(M[f64i(r0 + g, k0 + t)]);
    a[1] = f2tf32(M[f64i(r0 + g + 8, k0 + t)]);
    a[2] = f2tf32(M[f64i(r0 + g, k0 + t + 4)]);
    a[3] = f2tf32(M[f64i(r0 + g + 8, k0 + t + 4)]);
}
__device__ __forceinline__ void frag_b64(const float *M, int k0, int n0, int lane, uint32_t (&b)[2]) {
    const int g = lane >> 2, t = lane & 3;
    b[0] = f2tf32(M[f64i(k0 + t, n0 + g)]);
    b[1] = f2tf32(M[f64i(k0 + t + 4, n0 + g)]);
}
__device__ __forceinline__ void frag_b32(const float *M, int k0, int n0, int lane, uint32_t (&b)[2]) {
    const int g = lane >> 2, t = lane & 3;
    b[0] = f2tf32(M[f32i(k0 + t, n0 + g)]);
    b[1] = f2tf32(M[f32i(k0 + t + 4, n0 + g)]);
}

__global__ void __launch_bounds__(NTHREADS, 1)
chunked_kernel(const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmk,
               const __grid_constant__ CUtensorMap tmv, const PrefillArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const uint32_t sb = smem_u32(sm);
    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int64_t chain = blockIdx.x;
    const int64_t T = a.T;
    const int nch = (int)((T + C - 1) / C);
    const bool falcon = (a.mode == FW_FALCON1);
    const bool elu = (a.phi == FW_PHI_ELU1);
    const uint64_t limit = (uint64_t)a.wait_ns;

    volatile int *s_abort = reinterpret_cast<volatile int *>(sm + OFF_MISC);
    volatile uint32_t *s_tmem = reinterpret_cast<volatile uint32_t *>(sm + OFF_MISC + 4);
    auto bar = [&](int i) -> uint32_t { return sb + OFF_BAR + 8u * (uint32_t)i; };
    auto vec = [&](int b) -> float * { return reinterpret_cast<float *>(sm + OFF_VEC + b * VEC_BYTES); };
    auto xq = [&](int b) -> uint32_t { return sb + (b ? OFF_XQ1 : OFF_XQ0); };
    auto fail_now = [&]() {
        *s_abort = 1;
        atomicExch(a.err, kDevErrTimeout);
    };

    if (tid == 0) {
        for (int i = 0; i < B_COUNT; ++i) mbar_init(bar(i), 1);
        fence_mbar_init();
        *s_abort = 0;
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
            const int shift = falcon ? 1 : 0;
            int nxq0 = 0, nxq1 = 0, ny = 0;
            bool ok = true;
            for (int c = 0; c < nch && ok; ++c) {
                const int b = c & 1;
                if (c >= 2 && !wait_fast(bar(B_EMPTY0 + b), (uint32_t)((c >> 1) - 1) & 1u, limit, s_abort)) {
                    ok = false;
                    break;
                }
                const uint32_t st = xq(b);
                const int y = c * C;
                const uint32_t full = bar(B_FULL0 + b);
                mbar_expect_tx(full, falcon ? 32 * KB : 48 * KB);
                tma_load_3d(st + XQ_X0, &tmk, 0, y - shift, (int)chain, full);
                tma_load_3d(st + XQ_X1, &tmk, 64, y - shift, (int)chain, full);
                tma_load_3d(st + XQ_Q0, &tmq, 0, y, (int)chain, full);
                tma_load_3d(st + XQ_Q1, &tmq, 64, y, (int)chain, full);
                if (!falcon) {
                    const uint32_t yv = sb + (b ? OFF_Y1 : OFF_Y0);
                    tma_load_3d(yv, &tmv, 0, y, (int)chain, full);
                    tma_load_3d(yv + 8 * KB, &tmv, 64, y, (int)chain, full);
                }
                if (b) ++nxq1; else ++nxq0;
                TRACE(c, 19);
                if (falcon) {
                    if (c >= 1 && !wait_fast(bar(B_YFREE), (uint32_t)(c - 1) & 1u, limit, s_abort)) {
                        ok = false;
                        break;
                    }
                    mbar_expect_tx(bar(B_FULLY), 16 * KB);
                    tma_load_3d(sb + OFF_Y0, &tmv, 0, y, (int)chain, bar(B_FULLY));
                    tma_load_3d(sb + OFF_Y0 + 8 * KB, &tmv, 64, y, (int)chain, bar(B_FULLY));
                    ++ny;
                }
            }
            if (!ok) fail_now();
            // never leave a copy in flight into this CTA's shared memory
            if (nxq0) mbar_wait(bar(B_FULL0), (uint32_t)(nxq0 - 1) & 1u, kDrainNs);
            if (nxq1) mbar_wait(bar(B_FULL1), (uint32_t)(nxq1 - 1) & 1u, kDrainNs);
            if (ny) mbar_wait(bar(B_FULLY), (uint32_t)(ny - 1) & 1u, kDrainNs);
        }
        __syncwarp();
    } else if (warp == 1) {
        // ================================================================ key-path MMAs
        if (lane == 0) {
            bool ok = true;
            for (int c = 0; c < nch && ok; ++c) {
                const int b = c & 1;
                const uint32_t st = xq(b);
                if (!wait_fast(bar(B_GGO), (uint32_t)c & 1u, limit, s_abort)) { ok = false; break; }
                tc_fence_after();
                {   // G = [X; Q] X^T  (rows 0..63: X X^T, rows 64..127: Q X^T)
                    const uint32_t id = idesc_bf16(128, 64, false, false);
                    const uint64_t dx = sdesc_sw128(st + XQ_X0, 16, 1024);
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk) {
                        const uint64_t off = ((kk >> 2) * 16384u + (kk & 3) * 32u) >> 4;
                        mma_bf16(tmem + COL_G, dx + off, dx + off, id, kk > 0);
                    }
                    mma_commit(bar(B_GDONE));
                    TRACE(c, 15);
                }
                if (!falcon) continue;
                if (!wait_fast(bar(B_TRDY), (uint32_t)c & 1u, limit, s_abort) ||
                    !wait_fast(bar(B_FULLY), (uint32_t)c & 1u, limit, s_abort) ||
                    (c >= 2 && !wait_fast(bar(B_RFREE0 + b), (uint32_t)((c >> 1) - 1) & 1u, limit, s_abort))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                {   // -W^T = X^T (-T diag Gm)^T, U^T = Y^T T^T
                    const uint32_t id = idesc_bf16(128, 64, true, false);
                    const uint64_t dx = sdesc_sw128(st + XQ_X0, 16384, 1024);
                    const uint64_t dtp = sdesc_sw128(sb + OFF_TPB, 16, 1024);
                    const uint64_t dy = sdesc_sw128(sb + OFF_Y0, 8192, 1024);
                    const uint64_t dt = sdesc_sw128(sb + OFF_TB, 16, 1024);
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        mma_bf16(tmem + COL_W, dx + kk * 128, dtp + kk * 2, id, kk > 0);
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        mma_bf16(tmem + COL_R0 + 64 * b, dy + kk * 128, dt + kk * 2, id, kk > 0);
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
                const int b = c & 1;
                const uint32_t st = xq(b);
                if (!wait_fast(bar(B_WRDY), (uint32_t)c & 1u, limit, s_abort) ||
                    !wait_fast(bar(B_SRDY), (uint32_t)c & 1u, limit, s_abort) ||
                    (c >= 1 && !wait_fast(bar(B_OFREE), (uint32_t)(c - 1) & 1u, limit, s_abort))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t pb = sb + (b ? OFF_PB1 : OFF_PB0);
                const uint32_t id_mk = idesc_bf16(128, 64, true, false);
                const uint64_t ds = sdesc_sw128(sb + OFF_SB, 16384, 1024);
                const uint64_t dq = sdesc_sw128(st + XQ_Q0, 16, 1024);
                const uint64_t dp = sdesc_sw128(pb, 16, 1024);
                const uint64_t dx = sdesc_sw128(st + XQ_X0, 16384, 1024);
                if (falcon) {
                    // R^T += S^T (-W^T);  O1^T = S^T Q^T
                    const uint32_t id_mm = idesc_bf16(128, 64, true, true);
                    const uint64_t dw = sdesc_sw128(sb + OFF_WTB, 8192, 1024);
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk)
                        mma_bf16(tmem + COL_R0 + 64 * b, ds + kk * 128, dw + kk * 128, id_mm, 1);
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk)
                        mma_bf16(tmem + COL_O1, ds + kk * 128,
                                 dq + (((kk >> 2) * 16384u + (kk & 3) * 32u) >> 4), id_mk, kk > 0);
                    mma_commit(bar(B_RDONE));
                    TRACE(c, 17);
                    if (!wait_fast(bar(B_RRDY), (uint32_t)c & 1u, limit, s_abort)) { ok = false; break; }
                    tc_fence_after();
                    // O2^T = R^T P^T;  S += X^T (diag(w) R)
                    const uint32_t id_kk = idesc_bf16(128, 64, false, false);
                    const uint64_t dra = sdesc_sw128(sb + OFF_RA, 16, 1024);
                    const uint64_t drb = sdesc_sw128(sb + OFF_RB, 16, 1024);
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        mma_bf16(tmem + COL_O2, dra + kk * 2, dp + kk * 2, id_kk, kk > 0);
                    const uint32_t id_s = idesc_bf16(128, 128, true, false);
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        mma_bf16(tmem + COL_S, dx + kk * 128, drb + kk * 2, id_s, 1);
                } else {
                    const uint64_t dv = sdesc_sw128(sb + (b ? OFF_Y1 : OFF_Y0), 8192, 1024);
                    // O1^T = S^T Q^T, O2^T = V^T P^T;  S += X^T V
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk)
                        mma_bf16(tmem + COL_O1, ds + kk * 128,
                                 dq + (((kk >> 2) * 16384u + (kk & 3) * 32u) >> 4), id_mk, kk > 0);
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        mma_bf16(tmem + COL_O2, dv + kk * 128, dp + kk * 2, id_mk, kk > 0);
                    const uint32_t id_s = idesc_bf16(128, 128, true, true);
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        mma_bf16(tmem + COL_S, dx + kk * 128, dv + kk * 128, id_s, 1);
                }
                mma_commit(bar(B_SDONE));
                mma_commit(bar(B_PFREE0 + b));
                mma_commit(bar(B_EMPTY0 + b));
                TRACE(c, 18);
            }
            if (!ok) fail_now();
            mma_commit(bar(B_SDRAIN));
            mbar_wait(bar(B_SDRAIN), 0, kDrainNs);
        }
        __syncwarp();
    } else if (warp >= KG_W0 && warp < SG_W0) {
        // ================================================================ key group
        const int kt = tid - KG_W0 * 32;           // == TMEM lane of this thread
        const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
        float *Lf = reinterpret_cast<float *>(sm + OFF_LF);
        float *Tf = reinterpret_cast<float *>(sm + OFF_TF);
        float *Ms = reinterpret_cast<float *>(sm + OFF_MS);
        const int kw = warp - KG_W0;
        auto gwait = [&](uint32_t bb, uint32_t parity) -> bool {
            const bool ok = wait_bar(bb, parity, limit, s_abort);
            return !bar_or(BAR_KG, GROUP, !ok);
        };
        auto gsync = [&]() { bar_sync(BAR_KG, GROUP); };

        if (!falcon && kt < C) {
            for (int b = 0; b < 2; ++b) {
                float *v = vec(b);
                v[V_ETA / 4 + kt] = 1.f;
                v[V_GAM / 4 + kt] = 1.f;
                v[V_G / 4 + kt] = 1.f;
                v[V_GM / 4 + kt] = 1.f;
                v[V_WC / 4 + kt] = 1.f;
                if (kt == 0) v[V_GC / 4] = 1.f;
            }
        }

        bool ok = true;
        // testing hook: a wait on a barrier nothing arrives on runs out
        if (a.force_timeout && !gwait(bar(B_NEVER), 0)) ok = false;
        // beta, lambda of the next chunk are loaded one chunk ahead (thread t < C)
        float nb = 0.f, nl = 0.f;
        auto load_gates = [&](int cc) {
            const int64_t tok = (int64_t)cc * C + kt;
            if (falcon && kt < C && cc < nch && tok < T) {
                nb = a.beta[chain * T + tok];
                nl = a.lam[chain * T + tok];
            }
        };
        load_gates(0);
#pragma unroll 1
        for (int c = 0; c < nch && ok; ++c) {
            const int b = c & 1;
            const uint32_t st = xq(b);
            float *vb = vec(b);
            if (!gwait(bar(B_FULL0 + b), (uint32_t)(c >> 1) & 1u)) { ok = false; break; }
            if (kt == 0) TRACE(c, 0);

            // ---- feature map on the loaded tiles, k_init patch
            {
                bool wrote = false;
                if (elu) {
                    const int t = kt >> 1, hb = kt & 1;
                    const uint32_t roff = (uint32_t)(t >> 3) * 1024u + (uint32_t)(t & 7) * 128u;
                    for (int which = 0; which < (falcon ? 1 : 2); ++which) {
                        const int64_t src = (int64_t)c * C + t - ((which == 0 && falcon) ? 1 : 0);
                        if (src < 0 || src >= T) continue;
                        const uint32_t row = st + (which == 0 ? (hb ? XQ_X1 : XQ_X0) : (hb ? XQ_Q1 : XQ_Q0)) + roff;
#pragma unroll
                        for (int c16 = 0; c16 < 8; ++c16) {
                            float f[8];
                            unpack8(ld_shared_v4(row + c16 * 16), f);
#pragma unroll
                            for (int e = 0; e < 8; ++e) f[e] = f[e] > 0.f ? f[e] + 1.f : __expf(f[e]);
                            st_row8_bf16(row + c16 * 16, f);
                        }
                    }
                    wrote = true;
                }
                if (falcon && c == 0 && a.k_init) {
                    if (kt < 16) {
                        const int hb = kt >> 3, c16 = kt & 7;
                        const uint4 u = *reinterpret_cast<const uint4 *>(
                            static_cast<const __nv_bfloat16 *>(a.k_init) + chain * D + hb * 64 + c16 * 8);
                        float f[8];
                        unpack8(u, f);
#pragma unroll
                        for (int e = 0; e < 8; ++e) f[e] = apply_phi(a.phi, f[e]);
                        st_row8_bf16(st + (hb ? XQ_X1 : XQ_X0) + (uint32_t)c16 * 16u, f);
                    }
                    wrote = true;
                }
                if (wrote) fence_proxy_async();
            }
            gsync();   // mapped tiles (and the k_init row) complete: the Gram MMA may start
            if (kt == 0) mbar_arrive(bar(B_GGO));

            if (!gwait(bar(B_GDONE), (uint32_t)c & 1u)) { ok = false; break; }
            if (kt == 0) TRACE(c, 2);
            tc_fence_after();
            if (c >= 2 && !gwait(bar(B_PFREE0 + b), (uint32_t)((c >> 1) - 1) & 1u)) { ok = false; break; }
            float g[64];   // row kt of G = [X;Q] X^T
            tmem_ld32(tmem + lane_base + COL_G, g);
            tmem_ld32(tmem + lane_base + COL_G + 32, g + 32);

            // ---- step sizes and decay products of chunk c; |x_t|^2 is G[t,t]
            if (falcon) {
                if (kt < C) {
                    const int t = kt;
                    const int64_t tok = (int64_t)c * C + t;
                    const float bt = nb, lt = nl;
                    load_gates(c + 1);
                    float n = 0.f;
#pragma unroll
                    for (int s2 = 0; s2 < C; ++s2) n = (s2 == t) ? g[s2] : n;
                    float eta = 0.f, gam = 1.f;
                    if (tok < T) {
                        const bool pair = (tok > 0) || (a.k_init != nullptr);
                        eta = pair ? bt / (n + lt + a.eps) : 0.f;
                        gam = 1.f - eta * lt;
                    }
                    vb[V_ETA / 4 + t] = eta;
                    vb[V_GAM / 4 + t] = gam;
                }
                gsync();
                if (kw == 0) {
                    float g0 = vb[V_GAM / 4 + lane], g1 = vb[V_GAM / 4 + lane + 32];
                    float h0 = g0, h1 = g1;
#pragma unroll
                    for (int off = 1; off < 32; off <<= 1) {
                        const float u0 = __shfl_up_sync(0xffffffffu, g0, off);
                        const float u1 = __shfl_up_sync(0xffffffffu, g1, off);
                        const float d0 = __shfl_down_sync(0xffffffffu, h0, off);
                        const float d1 = __shfl_down_sync(0xffffffffu, h1, off);
                        if (lane >= off) { g0 *= u0; g1 *= u1; }
                        if (lane + off < 32) { h0 *= d0; h1 *= d1; }
                    }
                    const float tot0 = __shfl_sync(0xffffffffu, g0, 31);
                    const float tot1 = __shfl_sync(0xffffffffu, h1, 0);
                    g1 *= tot0;
                    h0 *= tot1;
                    float e0 = __shfl_up_sync(0xffffffffu, g0, 1);
                    float e1 = __shfl_up_sync(0xffffffffu, g1, 1);
                    if (lane == 0) { e0 = 1.f; e1 = tot0; }
                    float x0 = __shfl_down_sync(0xffffffffu, h0, 1);
                    float x1 = __shfl_down_sync(0xffffffffu, h1, 1);
                    if (lane == 31) { x0 = tot1; x1 = 1.f; }
                    vb[V_G / 4 + lane] = g0;
                    vb[V_G / 4 + lane + 32] = g1;
                    vb[V_GM / 4 + lane] = e0;
                    vb[V_GM / 4 + lane + 32] = e1;
                    vb[V_WC / 4 + lane] = x0 * vb[V_ETA / 4 + lane];
                    vb[V_WC / 4 + lane + 32] = x1 * vb[V_ETA / 4 + lane + 32];
                    if (lane == 31) vb[V_GC / 4] = g1;
                }
                gsync();
            }
            if (kt == 0) {
                TRACE(c, 1);
                mbar_arrive(bar(B_GV0 + b));
            }

            // ---- L and P from G = [X;Q] X^T
            {
                const float4 *eta4 = reinterpret_cast<const float4 *>(vb + V_ETA / 4);
                const float4 *gam4 = reinterpret_cast<const float4 *>(vb + V_GAM / 4);
                if (kt < C) {
                    if (falcon) {   // L[t,s] = D[t-1,s] eta_s A[t,s], s < t
                        const int t = kt;
                        float dz = 1.f;
#pragma unroll
                        for (int q = 15; q >= 0; --q) {
                            const float4 e4 = eta4[q], y4 = gam4[q];
                            const float ev[4] = {e4.x, e4.y, e4.z, e4.w};
                            const float yv[4] = {y4.x, y4.y, y4.z, y4.w};
#pragma unroll
                            for (int e = 3; e >= 0; --e) {
                                const int s2 = 4 * q + e;
                                const bool act = s2 < t;
                                g[s2] = act ? dz * ev[e] * g[s2] : 0.f;
                                if (act) dz *= yv[e];
                            }
                        }
#pragma unroll
                        for (int q = 0; q < 16; ++q)
                            *reinterpret_cast<float4 *>(Lf + t * 64 + ((q ^ (t & 15)) << 2)) =
                                make_float4(g[4 * q], g[4 * q + 1], g[4 * q + 2], g[4 * q + 3]);
                    }
                } else {   // P[t,s] = D[t,s] eta_s (q_t.x_s), s <= t
                    const int t = kt - C;
                    float dz = 1.f;
#pragma unroll
                    for (int q = 15; q >= 0; --q) {
                        const float4 e4 = eta4[q], y4 = gam4[q];
                        const float ev[4] = {e4.x, e4.y, e4.z, e4.w};
                        const float yv[4] = {y4.x, y4.y, y4.z, y4.w};
#pragma unroll
                        for (int e = 3; e >= 0; --e) {
                            const int s2 = 4 * q + e;
                            const bool act = s2 <= t;
                            g[s2] = act ? dz * ev[e] * g[s2] : 0.f;
                            if (act) dz *= yv[e];
                        }
                    }
                    const uint32_t pb = sb + (b ? OFF_PB1 : OFF_PB0);
#pragma unroll
                    for (int c16 = 0; c16 < 8; ++c16) st_row8_bf16(pb + sw128(t, c16), g + 8 * c16);
                }
            }
            tc_fence_before();
            fence_proxy_async();
            gsync();
            if (kt == 0) TRACE(c, 3);
            if (!falcon) {
                if (kt == 0) mbar_arrive(bar(B_WRDY));
                continue;
            }

            if (kt == 0) TRACE(c, 4);
            // ---- T = (I + L)^{-1} on warp-level tf32 MMAs.  Outputs: fp32 T blocks
            //      needed by later merges (Tf), and the bf16 operands T and
            //      -T diag(Gm) (K-major rows t) written straight from the fragments.
            // bf16 T and -T diag(Gm) live where L does: their writes wait until the
            // last read of L (the second merge level), so fragments are kept here.
            const int gq = lane >> 2, tq = lane & 3;
            const float *gmv = vb + V_GM / 4;
            auto put_t = [&](int r, int c, float v0, float v1) {   // bf16 pair (r, c..c+1)
                const uint32_t off = sw128((uint32_t)r, (uint32_t)c >> 3) + ((uint32_t)(c & 7) << 1);
                st_shared_u32(sb + OFF_TB + off, pack_bf16(v0, v1));
                st_shared_u32(sb + OFF_TPB + off, pack_bf16(-v0 * gmv[c], -v1 * gmv[c + 1]));
            };
            float tdiag[2][4];   // this warp's diagonal block of T (C fragment)
            float tpair[4];      // this warp's tile of T_{10} / T_{32}
            {
                const int g = gq, t4 = tq;
                // diagonal block kw: (I + L)^{-1} = (I - L)(I + L^2)(I + L^4)(I + L^8)
                const int base = 16 * kw;
                float *SA = Ms + kw * 512;        // 16x16 fp32 scratch pair of this warp
                float *SB2 = SA + 256;
                auto sidx = [&](int r, int c) { return r * 16 + ((((c >> 2) ^ (r & 3)) << 2) | (c & 3)); };
                // C fragment (two 8-column tiles) <-> 16x16 scratch
                auto store_c = [&](float *M, const float (&d)[2][4]) {
#pragma unroll
                    for (int nt = 0; nt < 2; ++nt) {
                        M[sidx(g, 8 * nt + 2 * t4)] = d[nt][0];
                        M[sidx(g, 8 * nt + 2 * t4 + 1)] = d[nt][1];
                        M[sidx(g + 8, 8 * nt + 2 * t4)] = d[nt][2];
                        M[sidx(g + 8, 8 * nt + 2 * t4 + 1)] = d[nt][3];
                    }
                };
                // d = Aop(16x16) * Bop(16x16); operands fetched by the given functions
                auto prod = [&](float (&d)[2][4], auto geta, auto getb) {
#pragma unroll
                    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                        for (int e = 0; e < 4; ++e) d[nt][e] = 0.f;
#pragma unroll
                    for (int ks = 0; ks < 2; ++ks) {
                        uint32_t fa[4];
                        fa[0] = f2tf32(geta(g, 8 * ks + t4));
                        fa[1] = f2tf32(geta(g + 8, 8 * ks + t4));
                        fa[2] = f2tf32(geta(g, 8 * ks + t4 + 4));
                        fa[3] = f2tf32(geta(g + 8, 8 * ks + t4 + 4));
#pragma unroll
                        for (int nt = 0; nt < 2; ++nt) {
                            uint32_t fb[2];
                            fb[0] = f2tf32(getb(8 * ks + t4, 8 * nt + g));
                            fb[1] = f2tf32(getb(8 * ks + t4 + 4, 8 * nt + g));
                            mma_tf32_16x8x8(d[nt], fa, fb);
                        }
                    }
                };
                auto Lget = [&](int r, int c) { return Lf[f64i(base + r, base + c)]; };
                auto ImL = [&](int r, int c) { return (r == c ? 1.f : 0.f) - Lf[f64i(base + r, base + c)]; };
                auto SAget = [&](int r, int c) { return SA[sidx(r, c)]; };
                auto SBget = [&](int r, int c) { return SB2[sidx(r, c)]; };
                float d[2][4], p[2][4];
                prod(d, Lget, Lget);                    // L^2
                store_c(SA, d);
                __syncwarp();
                prod(p, ImL, SAget);                    // (I - L) L^2
                // A2 = (I - L) + (I - L) L^2
#pragma unroll
                for (int nt = 0; nt < 2; ++nt) {
                    const int c0 = 8 * nt + 2 * t4;
                    p[nt][0] += ImL(g, c0);     p[nt][1] += ImL(g, c0 + 1);
                    p[nt][2] += ImL(g + 8, c0); p[nt][3] += ImL(g + 8, c0 + 1);
                }
                store_c(SB2, p);
                prod(d, SAget, SAget);                  // L^4
                __syncwarp();
                store_c(SA, d);
                __syncwarp();
                prod(d, SBget, SAget);                  // A2 L^4
#pragma unroll
                for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                    for (int e = 0; e < 4; ++e) p[nt][e] += d[nt][e];   // A3
                prod(d, SAget, SAget);                  // L^8
                __syncwarp();
                store_c(SB2, p);
                store_c(SA, d);
                __syncwarp();
                prod(d, SBget, SAget);                  // A3 L^8
#pragma unroll
                for (int nt = 0; nt < 2; ++nt) {
                    const int c0 = 8 * nt + 2 * t4;
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        d[nt][e] += p[nt][e];   // T_kk
                        tdiag[nt][e] = d[nt][e];
                    }
                    Tf[f64i(base + g, base + c0)] = d[nt][0];
                    Tf[f64i(base + g, base + c0 + 1)] = d[nt][1];
                    Tf[f64i(base + g + 8, base + c0)] = d[nt][2];
                    Tf[f64i(base + g + 8, base + c0 + 1)] = d[nt][3];
                    if ((kw & 1) == 0) {   // zero fp32 block above, inside the 32-block
                        Tf[f64i(base + g, base + 16 + c0)] = 0.f;
                        Tf[f64i(base + g, base + 16 + c0 + 1)] = 0.f;
                        Tf[f64i(base + g + 8, base + 16 + c0)] = 0.f;
                        Tf[f64i(base + g + 8, base + 16 + c0 + 1)] = 0.f;
                    }
                }
            }
            gsync();
            if (kt == 0) TRACE(c, 5);
            {   // pairs (1,0) and (3,2): warp kw -> pair p, 8-column tile nt
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
                    fb[0] = f2tf32(Mw[(8 * ks + t4) * 8 + g]);
                    fb[1] = f2tf32(Mw[(8 * ks + t4 + 4) * 8 + g]);
                    mma_tf32_16x8x8(u, fa, fb);
                }
                const int c0 = cb + 8 * nt + 2 * t4;
                Tf[f64i(rb + g, c0)] = -u[0];
                Tf[f64i(rb + g, c0 + 1)] = -u[1];
                Tf[f64i(rb + g + 8, c0)] = -u[2];
                Tf[f64i(rb + g + 8, c0 + 1)] = -u[3];
#pragma unroll
                for (int e = 0; e < 4; ++e) tpair[e] = -u[e];
            }
            gsync();
            {   // M2 = L[32:64, 0:32] T[0:32, 0:32]
                const int rt = kw >> 1, ch = kw & 1;   // 16-row tile, 16-column half
                const int g = lane >> 2, t4 = lane & 3;
                float m[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
                for (int ks = 0; ks < 4; ++ks) {
                    uint32_t fa[4];
                    frag_a64(Lf, 32 + 16 * rt, 8 * ks, lane, fa);
#pragma unroll
                    for (int n2 = 0; n2 < 2; ++n2) {
                        uint32_t fb[2];
                        frag_b64(Tf, 8 * ks, 16 * ch + 8 * n2, lane, fb);
                        mma_tf32_16x8x8(m[n2], fa, fb);
                    }
                }
#pragma unroll
                for (int n2 = 0; n2 < 2; ++n2) {
                    const int c0 = 16 * ch + 8 * n2 + 2 * t4;
                    Ms[f32i(16 * rt + g, c0)] = m[n2][0];
                    Ms[f32i(16 * rt + g, c0 + 1)] = m[n2][1];
                    Ms[f32i(16 * rt + g + 8, c0)] = m[n2][2];
                    Ms[f32i(16 * rt + g + 8, c0 + 1)] = m[n2][3];
                }
            }
            gsync();
            {   // L is dead: write the bf16 blocks computed so far, zero the upper ones
                const int g = gq, t4 = tq;
                const int base = 16 * kw;
#pragma unroll
                for (int nt = 0; nt < 2; ++nt) {
                    const int c0 = base + 8 * nt + 2 * t4;
                    put_t(base + g, c0, tdiag[nt][0], tdiag[nt][1]);
                    put_t(base + g + 8, c0, tdiag[nt][2], tdiag[nt][3]);
                }
                const int p = kw >> 1, nt = kw & 1;
                const int rb = 16 + 32 * p, c0 = 32 * p + 8 * nt + 2 * t4;
                put_t(rb + g, c0, tpair[0], tpair[1]);
                put_t(rb + g + 8, c0, tpair[2], tpair[3]);
                for (int cb = kw + 1; cb < 4; ++cb) {
                    const int r = base + (lane >> 1), c = 16 * cb + 8 * (lane & 1);
                    st_shared_v4(sb + OFF_TB + sw128((uint32_t)r, (uint32_t)c >> 3), 0u, 0u, 0u, 0u);
                    st_shared_v4(sb + OFF_TPB + sw128((uint32_t)r, (uint32_t)c >> 3), 0u, 0u, 0u, 0u);
                }
            }
            {   // T[32:64, 0:32] = -T[32:64, 32:64] M2  (bf16 operands only)
                const int rt = kw >> 1, ch = kw & 1;
                const int g = gq, t4 = tq;
                float u[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
                for (int ks = 0; ks < 4; ++ks) {
                    uint32_t fa[4];
                    frag_a64(Tf, 32 + 16 * rt, 32 + 8 * ks, lane, fa);
#pragma unroll
                    for (int n2 = 0; n2 < 2; ++n2) {
                        uint32_t fb[2];
                        frag_b32(Ms, 8 * ks, 16 * ch + 8 * n2, lane, fb);
                        mma_tf32_16x8x8(u[n2], fa, fb);
                    }
                }
#pragma unroll
                for (int n2 = 0; n2 < 2; ++n2) {
                    const int c0 = 16 * ch + 8 * n2 + 2 * t4;
                    const int r0 = 32 + 16 * rt + g;
#pragma unroll
                    for (int hh = 0; hh < 2; ++hh) {
                        const int r = r0 + 8 * hh;
                        const float v0 = -u[n2][2 * hh], v1 = -u[n2][2 * hh + 1];
                        const uint32_t off = sw128((uint32_t)r, (uint32_t)c0 >> 3) + ((uint32_t)(c0 & 7) << 1);
                        st_shared_u32(sb + OFF_TB + off, pack_bf16(v0, v1));
                        st_shared_u32(sb + OFF_TPB + off, pack_bf16(-v0 * gmv[c0], -v1 * gmv[c0 + 1]));
                    }
                }
            }
            fence_proxy_async();
            gsync();
            if (kt == 0) { TRACE(c, 6); mbar_arrive(bar(B_TRDY)); }

            // ---- -W^T -> bf16 rows i, once W^T(c) is done and R(c-1) has read the old one
            if (!gwait(bar(B_WUDONE), (uint32_t)c & 1u)) { ok = false; break; }
            if (kt == 0) TRACE(c, 7);
            tc_fence_after();
            if (c >= 1 && !gwait(bar(B_RDONE), (uint32_t)(c - 1) & 1u)) { ok = false; break; }
            if (kt == 0) TRACE(c, 8);
            {
                float w[32];
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    tmem_ld32(tmem + lane_base + COL_W + 32 * h, w);
#pragma unroll
                    for (int c16 = 0; c16 < 4; ++c16)
                        st_row8_bf16(sb + OFF_WTB + sw128(kt, 4 * h + c16), w + 8 * c16);
                }
            }
            tc_fence_before();
            fence_proxy_async();
            gsync();
            if (kt == 0) { TRACE(c, 9); mbar_arrive(bar(B_WRDY)); }
        }
        if (!ok && kt == 0) fail_now();
    } else if (warp >= SG_W0) {
        // ================================================================ state group
        const int srow = tid - SG_W0 * 32;         // == TMEM lane of this thread
        const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
        auto gwait = [&](uint32_t bb, uint32_t parity) -> bool {
            const bool ok = wait_bar(bb, parity, limit, s_abort);
            return !bar_or(BAR_SG, GROUP, !ok);
        };
        auto gsync = [&]() { bar_sync(BAR_SG, GROUP); };
        bool ok = true;

        // initial state: TMEM <- G_{C-1}(chunk 0) S0, bf16 copy for the MMAs
        float gC0 = 1.f;
        if (falcon) {
            if (!gwait(bar(B_GV0), 0)) ok = false;
            else gC0 = vec(0)[V_GC / 4];
        }
        if (ok) {
#pragma unroll 1
            for (int q = 0; q < 8; ++q) {
                float v[16];
                if (a.S0) {
                    const float4 *src = reinterpret_cast<const float4 *>(a.S0 + (chain * D + srow) * D + 16 * q);
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float4 f = src[e];
                        v[4 * e] = f.x; v[4 * e + 1] = f.y; v[4 * e + 2] = f.z; v[4 * e + 3] = f.w;
                    }
                } else {
#pragma unroll
                    for (int e = 0; e < 16; ++e) v[e] = 0.f;
                }
                const uint32_t blk = sb + OFF_SB + (uint32_t)(q >> 2) * 16384u;
                const uint32_t c16 = (uint32_t)((16 * q) & 63) >> 3;
                st_row8_bf16(blk + sw128(srow, c16), v);
                st_row8_bf16(blk + sw128(srow, c16 + 1), v + 8);
#pragma unroll
                for (int e = 0; e < 16; ++e) v[e] *= gC0;
                tmem_st16(tmem + lane_base + COL_S + 16 * q, v);
            }
            tmem_st_wait();
            tc_fence_before();
            fence_proxy_async();
            gsync();
            if (srow == 0) mbar_arrive(bar(B_SRDY));
        }

#pragma unroll 1
        for (int c = 0; c < nch && ok; ++c) {
            const int b = c & 1;
            const int64_t tok0 = (int64_t)c * C;
            if (falcon) {
                // ---- R^T -> bf16 rows j (A operand) and diag(w)-scaled copy (B operand)
                if (!gwait(bar(B_RDONE), (uint32_t)c & 1u) ||
                    !gwait(bar(B_GV0 + b), (uint32_t)(c >> 1) & 1u)) { ok = false; break; }
                if (srow == 0) TRACE(c, 10);
                tc_fence_after();
                const float *wc = vec(b) + V_WC / 4;
                if (srow < C)   // the key group may recycle this gate block once S(c) is done
                    reinterpret_cast<float *>(sm + OFF_SGV)[srow] = vec(b)[V_G / 4 + srow];
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    float r[32];
                    tmem_ld32(tmem + lane_base + COL_R0 + 64 * b + 32 * h, r);
#pragma unroll
                    for (int c16 = 0; c16 < 4; ++c16) {
                        const float4 w0 = *reinterpret_cast<const float4 *>(wc + 32 * h + 8 * c16);
                        const float4 w1 = *reinterpret_cast<const float4 *>(wc + 32 * h + 8 * c16 + 4);
                        const float *rr = r + 8 * c16;
                        const float w8[8] = {rr[0] * w0.x, rr[1] * w0.y, rr[2] * w0.z, rr[3] * w0.w,
                                             rr[4] * w1.x, rr[5] * w1.y, rr[6] * w1.z, rr[7] * w1.w};
                        st_row8_bf16(sb + OFF_RA + sw128(srow, 4 * h + c16), rr);
                        st_row8_bf16(sb + OFF_RB + sw128(srow, 4 * h + c16), w8);
                    }
                }
                tc_fence_before();
                fence_proxy_async();
                gsync();
                if (srow == 0) {
                    TRACE(c, 11);
                    mbar_arrive(bar(B_RRDY));
                    mbar_arrive(bar(B_RFREE0 + b));
                }
            }

            // ---- state carry
            if (!gwait(bar(B_SDONE), (uint32_t)c & 1u)) { ok = false; break; }
            if (srow == 0) TRACE(c, 12);
            tc_fence_after();
            const bool last = (c + 1 == nch);
            float gC_next = 1.f;
            if (falcon && !last) {
                const int b1 = (c + 1) & 1;
                if (!gwait(bar(B_GV0 + b1), (uint32_t)((c + 1) >> 1) & 1u)) { ok = false; break; }
                gC_next = vec(b1)[V_GC / 4];
            }
#pragma unroll 1
            for (int q = 0; q < 8; ++q) {
                float v[16];
                tmem_ld16(tmem + lane_base + COL_S + 16 * q, v);
                if (last) {
                    float4 *dst = reinterpret_cast<float4 *>(a.S_T + (chain * D + srow) * D + 16 * q);
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        dst[e] = make_float4(v[4 * e], v[4 * e + 1], v[4 * e + 2], v[4 * e + 3]);
                } else {
                    const uint32_t blk = sb + OFF_SB + (uint32_t)(q >> 2) * 16384u;
                    const uint32_t c16 = (uint32_t)((16 * q) & 63) >> 3;
                    st_row8_bf16(blk + sw128(srow, c16), v);
                    st_row8_bf16(blk + sw128(srow, c16 + 1), v + 8);
#pragma unroll
                    for (int e = 0; e < 16; ++e) v[e] *= gC_next;
                    tmem_st16(tmem + lane_base + COL_S + 16 * q, v);
                }
            }
            tmem_st_wait();
            tc_fence_before();
            fence_proxy_async();
            gsync();
            if (srow == 0) TRACE(c, 13);
            if (!last && srow == 0) mbar_arrive(bar(B_SRDY));

            // ---- outputs o_t = G_t (S0^T q_t) + (P R)_t.  Lanes j and j^1 swap
            //      halves so each stores a bf16 pair (t, j..j+1): even lanes the
            //      even tokens, odd lanes the odd ones.
            {
                const float *gv = reinterpret_cast<const float *>(sm + OFF_SGV);
                const bool odd = (lane & 1) != 0;
                const int jj = srow & ~1;
                uint32_t *og = reinterpret_cast<uint32_t *>(static_cast<__nv_bfloat16 *>(a.o) +
                                                           (chain * T + tok0) * D + jj);
                const int64_t nvalid = T - tok0;
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    float o1[32], o2[32];
                    tmem_ld32(tmem + lane_base + COL_O1 + 32 * h, o1);
                    tmem_ld32(tmem + lane_base + COL_O2 + 32 * h, o2);
#pragma unroll
                    for (int e = 0; e < 32; e += 2) {
                        const int t = 32 * h + e;
                        const float v0 = falcon ? fmaf(gv[t], o1[e], o2[e]) : o1[e] + o2[e];
                        const float v1 = falcon ? fmaf(gv[t + 1], o1[e + 1], o2[e + 1]) : o1[e + 1] + o2[e + 1];
                        const float other = __shfl_xor_sync(0xffffffffu, odd ? v0 : v1, 1);
                        const int tt = odd ? t + 1 : t;
                        const uint32_t w = odd ? pack_bf16(other, v1) : pack_bf16(v0, other);
                        if (tt < nvalid) og[(int64_t)tt * (D / 2)] = w;
                    }
                }
            }
            tc_fence_before();
            gsync();
            if (srow == 0) { TRACE(c, 14); mbar_arrive(bar(B_OFREE)); }
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

// [n_chains][T][128] bf16 viewed as a 3-D tensor (d, T, chain); 64 x 64 boxes.
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

// Falcon-1 with phi = elu+1 is declined: phi(k) is close to 1 + k for small
// keys, and rounding it to a bf16 MMA operand erases most of the key's varying
// part, which the residual write depends on (the per-token kernel keeps it in
// fp32).  Linear attention accumulates phi(k) additively and keeps bf16
// operand accuracy.
bool chunked_supported(const PrefillArgs &a) {
    if (a.mode == FW_FALCON1 && a.phi == FW_PHI_ELU1) return false;
    return a.dtype == FW_BF16 && a.d == D && a.T <= (int64_t)INT32_MAX - C &&
           a.n_chains <= (int64_t)INT32_MAX;
}

#ifdef FW_TRACE
extern "C" int fw_debug_read_trace(unsigned long long *dst, int n) {
    if (n > kTraceChunks * kTraceEv) n = kTraceChunks * kTraceEv;
    return (int)cudaMemcpyFromSymbol(dst, g_trace, sizeof(unsigned long long) * n);
}
#endif

cudaError_t launch_chunked(const PrefillArgs &a, cudaStream_t s) {
    CUtensorMap tq, tk, tv;
    if (!make_map(&tq, a.q, a.T, a.n_chains) || !make_map(&tk, a.k, a.T, a.n_chains) ||
        !make_map(&tv, a.v, a.T, a.n_chains))
        return cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(chunked_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)SMEM_ALLOC);
    if (e != cudaSuccess) return e;
    chunked_kernel<<<(unsigned)a.n_chains, NTHREADS, SMEM_ALLOC, s>>>(tq, tk, tv, a);
    return cudaGetLastError();
}

}  // namespace fw
