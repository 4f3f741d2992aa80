// fw_api.cu -- the C ABI of libfw.so: argument validation, kernel choice,
// device error word.  See include/fw.h for the contract of every call.
#include <atomic>
#include <cmath>
#include <mutex>

#include "fw_internal.cuh"

namespace fw {
namespace {

// Device error word: set by kernels whose bounded waits run out.
__device__ int g_dev_error;

thread_local int g_last_cuda_error = 0;
constexpr long long kDefaultWaitUs = 2000000;  // 2 s
std::atomic<long long> g_wait_us{kDefaultWaitUs};
std::atomic<int> g_force_timeout{0};
std::atomic<int> g_seg_pref{0};

constexpr int kMaxDevices = 64;
std::mutex g_dev_mu;
int *g_err_ptr[kMaxDevices];
int g_dev_ok[kMaxDevices];  // 0 unknown, 1 ok, -1 not sm_103

int cuda_fail(cudaError_t e) {
    g_last_cuda_error = (int)e;
    return FW_ERR_CUDA;
}

// Resolve (once per device) the device address of the error word and check
// the architecture.  Returns FW_OK or an error.
int device_setup(int **err_ptr) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e);
    if (dev < 0 || dev >= kMaxDevices) return FW_ERR_DEVICE;
    std::lock_guard<std::mutex> lk(g_dev_mu);
    if (g_dev_ok[dev] == 0) {
        int major = 0, minor = 0;
        if ((e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev)) !=
            cudaSuccess)
            return cuda_fail(e);
        if ((e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev)) !=
            cudaSuccess)
            return cuda_fail(e);
        if (major != 10 || minor != 3) {
            g_dev_ok[dev] = -1;
        } else {
            void *p = nullptr;
            if ((e = cudaGetSymbolAddress(&p, g_dev_error)) != cudaSuccess) return cuda_fail(e);
            g_err_ptr[dev] = static_cast<int *>(p);
            g_dev_ok[dev] = 1;
        }
    }
    if (g_dev_ok[dev] < 0) return FW_ERR_DEVICE;
    *err_ptr = g_err_ptr[dev];
    return FW_OK;
}

bool misaligned(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) != 0; }

bool overlaps(const void *a, size_t na, const void *b, size_t nb) {
    if (!a || !b || na == 0 || nb == 0) return false;
    const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return x < y + nb && y < x + na;
}

// Modes with the normalised step and decay (beta, lambda, eps used).
bool gated(fw_mode m) { return m != FW_LINATTN; }

// Modes with a step size per value channel (beta carries a d_v index).
bool per_channel(fw_mode m) { return m == FW_FALCON2 || m == FW_FALCON2A; }

int check_common(const fw_shape *shape, fw_dtype dtype, fw_mode mode, fw_phi phi, float eps,
                 unsigned flags) {
    if (!shape) return FW_ERR_NULL;
    if (shape->B < 1 || shape->H < 1 || shape->T < 1) return FW_ERR_SHAPE;
    if (shape->d_k != 64 && shape->d_k != 128) return FW_ERR_SHAPE;
    if (shape->d_v != shape->d_k) return FW_ERR_SHAPE;
    if (shape->B > (int64_t)1 << 31 || shape->H > (int64_t)1 << 31) return FW_ERR_SHAPE;
    if (shape->B * shape->H > (int64_t)INT32_MAX) return FW_ERR_SHAPE;
    if (dtype != FW_F32 && dtype != FW_BF16) return FW_ERR_DTYPE;
    if (mode != FW_FALCON1 && mode != FW_LINATTN && mode != FW_FALCON1A && mode != FW_FALCON2 &&
        mode != FW_FALCON2A && mode != FW_FALCON3 && mode != FW_FALCON3A)
        return FW_ERR_MODE;
    if (phi != FW_PHI_IDENTITY && phi != FW_PHI_ELU1) return FW_ERR_MODE;
    if (flags & ~(unsigned)(FW_FLAG_RBW | FW_FLAG_SAME_PAIR)) return FW_ERR_MODE;
    if (gated(mode) && !(std::isfinite(eps) && eps >= 0.f)) return FW_ERR_ARG;
    return FW_OK;
}

bool window_mode(fw_mode m) { return m == FW_FALCON3 || m == FW_FALCON3A; }

// Byte extents of a carried window's arrays (x, y, n) for nc chains.
struct WinExtent {
    size_t x, y, n;
};
WinExtent win_extent(int64_t nc, int W, int d) {
    return {(size_t)nc * (size_t)(W - 1) * d * sizeof(float),
            (size_t)nc * (size_t)(W - 1) * d * sizeof(float), (size_t)nc * sizeof(int32_t)};
}

bool win_overlaps(const fw_window *w, const WinExtent &e, const void *p, size_t n) {
    return w && (overlaps(w->x, e.x, p, n) || overlaps(w->y, e.y, p, n) ||
                 overlaps(w->n, e.n, p, n));
}

// Checks of the window arguments shared by fw_window_prefill and
// fw_window_step; `in` and `out` may be NULL.
int check_window(const fw_window *in, const fw_window *out, int W, const WinExtent &e) {
    if (W < 2) return FW_OK;   // nothing carried
    for (const fw_window *w : {in, out}) {
        if (!w) continue;
        if (!w->x || !w->y || !w->n) return FW_ERR_NULL;
        if (misaligned(w->x) || misaligned(w->y) || misaligned(w->n)) return FW_ERR_ALIGN;
    }
    if (out) {
        if (overlaps(out->x, e.x, out->y, e.y) || overlaps(out->x, e.x, out->n, e.n) ||
            overlaps(out->y, e.y, out->n, e.n))
            return FW_ERR_ARG;
        if (in && (win_overlaps(in, e, out->x, e.x) || win_overlaps(in, e, out->y, e.y) ||
                   win_overlaps(in, e, out->n, e.n)))
            return FW_ERR_ARG;
    }
    return FW_OK;
}

}  // namespace
}  // namespace fw

using namespace fw;

namespace {

// fw_prefill_ex and fw_prefill_noalloc (noalloc: the two-segment form's
// workspace from the static buffer, never from the pool)
int prefill_impl(const void *q, const void *k, const void *v, const float *beta,
                 const float *lambda, const float *S0, const void *k_init, void *o, float *S_T,
                 const fw_shape *shape, fw_dtype dtype, fw_mode mode, fw_phi phi, float eps,
                 unsigned flags, fw_algo algo, cudaStream_t stream, bool noalloc) {
    int st = check_common(shape, dtype, mode, phi, eps, flags);
    if (st != FW_OK) return st;
    if (window_mode(mode)) return FW_ERR_MODE;   // fw_window_prefill
    if (algo != FW_ALGO_AUTO && algo != FW_ALGO_RECURRENT && algo != FW_ALGO_CHUNKED)
        return FW_ERR_MODE;
    if (!q || !k || !v || !o || !S_T) return FW_ERR_NULL;
    if (gated(mode) && (!beta || !lambda)) return FW_ERR_NULL;
    if (misaligned(q) || misaligned(k) || misaligned(v) || misaligned(o) || misaligned(S_T) ||
        misaligned(S0) || misaligned(k_init) || (gated(mode) && (misaligned(beta) ||
                                                                   misaligned(lambda))))
        return FW_ERR_ALIGN;

    const int64_t nc = shape->B * shape->H;
    const int d = shape->d_k;
    const size_t esz = dtype == FW_F32 ? 4 : 2;
    const size_t nx = (size_t)nc * (size_t)shape->T * d * esz;
    const size_t ns = (size_t)nc * d * d * sizeof(float);
    const size_t nl = (size_t)nc * (size_t)shape->T * sizeof(float);   // lambda
    const size_t nbl = nl * (per_channel(mode) ? (size_t)d : 1);           // beta
    if (overlaps(o, nx, q, nx) || overlaps(o, nx, k, nx) || overlaps(o, nx, v, nx) ||
        overlaps(o, nx, S0, S0 ? ns : 0) || overlaps(o, nx, S_T, ns))
        return FW_ERR_ARG;
    if (gated(mode) && (overlaps(o, nx, beta, nbl) || overlaps(o, nx, lambda, nl) ||
                        overlaps(S_T, ns, beta, nbl) || overlaps(S_T, ns, lambda, nl)))
        return FW_ERR_ARG;
    if (overlaps(S_T, ns, q, nx) || overlaps(S_T, ns, k, nx) || overlaps(S_T, ns, v, nx))
        return FW_ERR_ARG;
    if (S0 && S0 != S_T && overlaps(S_T, ns, S0, ns)) return FW_ERR_ARG;
    // k_init is read while other chains' outputs are being written
    const size_t nki = (size_t)nc * d * esz;
    if (k_init && (overlaps(o, nx, k_init, nki) || overlaps(S_T, ns, k_init, nki)))
        return FW_ERR_ARG;

    PrefillArgs a;
    a.q = q; a.k = k; a.v = v; a.beta = beta; a.lam = lambda; a.S0 = S0;
    // LINATTN pairs each key with its own value; so do the gated modes with
    // FW_FLAG_SAME_PAIR (then the bit stays set and k_init is unused)
    if (mode == FW_LINATTN) flags &= ~(unsigned)FW_FLAG_SAME_PAIR;
    a.k_init = (gated(mode) && !(flags & FW_FLAG_SAME_PAIR)) ? k_init : nullptr;
    a.o = o; a.S_T = S_T; a.n_chains = nc; a.T = shape->T; a.d = d;
    a.dtype = dtype; a.mode = mode; a.phi = phi; a.eps = eps; a.flags = flags;
    a.wait_ns = g_wait_us.load() * 1000LL;
    a.force_timeout = g_force_timeout.load();
    a.seg_pref = g_seg_pref.load();
    a.seg_t0 = 0; a.o_aux = nullptr; a.s_aux = nullptr;
    a.scratch_only = 0; a.scratch = nullptr; a.scratch_bytes = 0;

    const bool chunk_ok = per_channel(mode) ? chunked_chan_supported(a) : chunked_supported(a);
    if (algo == FW_ALGO_CHUNKED && !chunk_ok) return FW_ERR_UNSUPPORTED;

    st = device_setup(&a.err);
    if (st != FW_OK) return st;

    cudaError_t e;
    if (algo != FW_ALGO_RECURRENT && per_channel(mode) && chunk_ok) {
        // a step per value channel on the chunked tensor-core kernel
        e = launch_chunked_chan(a, stream);
    } else if (algo == FW_ALGO_AUTO && per_channel(mode)) {
        // a step per value column: the staged per-token kernel of the window
        // family with a window of one pair
        WindowArgs w{};
        w.q = q; w.k = k; w.v = v; w.beta = beta; w.lam = lambda; w.S0 = S0;
        w.k_init = a.k_init;
        w.o = o; w.S_T = S_T; w.n_chains = nc; w.T = shape->T; w.d = d; w.W = 1;
        w.dtype = dtype; w.inner = (mode == FW_FALCON2A); w.chan = true; w.phi = phi;
        w.eps = eps; w.flags = flags; w.err = a.err; w.wait_ns = a.wait_ns;
        e = launch_window_prefill(w, stream);
    } else if (algo == FW_ALGO_RECURRENT || !chunk_ok) {
        e = launch_recurrent(a, stream);
    } else {
        if (noalloc) {
            // the two-segment form's workspace: the static buffer, or nothing
            int dev = 0, sms = 0;
            e = cudaGetDevice(&dev);
            if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
            if (e != cudaSuccess) return cuda_fail(e);
            const size_t need = chunked_segment_bytes(a, sms);
            if (need > 0) {
                if (need > (size_t)FW_SCRATCH_BYTES) return FW_ERR_SCRATCH;
                a.scratch = segment_scratch(dev, &e);
                if (!a.scratch) return cuda_fail(e);
                a.scratch_bytes = FW_SCRATCH_BYTES;
            }
            a.scratch_only = 1;
        }
        e = launch_chunked(a, stream);
    }
    if (e != cudaSuccess) return cuda_fail(e);
    return FW_OK;
}

}  // namespace

extern "C" int fw_prefill_ex(const void *q, const void *k, const void *v, const float *beta,
                             const float *lambda, const float *S0, const void *k_init, void *o,
                             float *S_T, const fw_shape *shape, fw_dtype dtype, fw_mode mode,
                             fw_phi phi, float eps, unsigned flags, fw_algo algo,
                             cudaStream_t stream) {
    return prefill_impl(q, k, v, beta, lambda, S0, k_init, o, S_T, shape, dtype, mode, phi, eps,
                        flags, algo, stream, false);
}

extern "C" int fw_prefill_noalloc(const void *q, const void *k, const void *v, const float *beta,
                                  const float *lambda, const float *S0, const void *k_init,
                                  void *o, float *S_T, const fw_shape *shape, fw_dtype dtype,
                                  fw_mode mode, fw_phi phi, float eps, unsigned flags,
                                  fw_algo algo, cudaStream_t stream) {
    return prefill_impl(q, k, v, beta, lambda, S0, k_init, o, S_T, shape, dtype, mode, phi, eps,
                        flags, algo, stream, true);
}

extern "C" int fw_prefill(const void *q, const void *k, const void *v, const float *beta,
                          const float *lambda, const float *S0, void *o, float *S_T,
                          const fw_shape *shape, fw_dtype dtype, fw_mode mode, fw_phi phi,
                          float eps, cudaStream_t stream) {
    return fw_prefill_ex(q, k, v, beta, lambda, S0, nullptr, o, S_T, shape, dtype, mode, phi,
                         eps, 0u, FW_ALGO_AUTO, stream);
}

extern "C" int fw_step_ex(const void *q, const void *k_prev, const void *v, const float *beta,
                          const float *lambda, float *S, void *o, const fw_shape *shape,
                          fw_dtype dtype, fw_mode mode, fw_phi phi, float eps, unsigned flags,
                          cudaStream_t stream) {
    int st = check_common(shape, dtype, mode, phi, eps, flags);
    if (st != FW_OK) return st;
    if (window_mode(mode)) return FW_ERR_MODE;   // fw_window_step
    if (shape->T != 1) return FW_ERR_SHAPE;
    if (!q || !k_prev || !v || !S || !o) return FW_ERR_NULL;
    if (gated(mode) && (!beta || !lambda)) return FW_ERR_NULL;
    if (misaligned(q) || misaligned(k_prev) || misaligned(v) || misaligned(S) || misaligned(o) ||
        (gated(mode) && (misaligned(beta) || misaligned(lambda))))
        return FW_ERR_ALIGN;
    const int64_t ns = shape->B * shape->H;
    const int d = shape->d_k;
    const size_t esz = dtype == FW_F32 ? 4 : 2;
    const size_t nx = (size_t)ns * d * esz;
    const size_t nst = (size_t)ns * d * d * sizeof(float);
    if (overlaps(o, nx, q, nx) || overlaps(o, nx, k_prev, nx) || overlaps(o, nx, v, nx) ||
        overlaps(o, nx, S, nst) || overlaps(S, nst, q, nx) || overlaps(S, nst, k_prev, nx) ||
        overlaps(S, nst, v, nx))
        return FW_ERR_ARG;
    const size_t nb = (size_t)ns * 4 * (per_channel(mode) ? (size_t)d : 1);
    if (gated(mode) && (overlaps(S, nst, beta, nb) || overlaps(S, nst, lambda, ns * 4) ||
                        overlaps(o, nx, beta, nb) || overlaps(o, nx, lambda, ns * 4)))
        return FW_ERR_ARG;

    int *err = nullptr;
    st = device_setup(&err);
    if (st != FW_OK) return st;

    StepArgs a;
    a.q = q; a.k = k_prev; a.v = v; a.beta = beta; a.lam = lambda; a.S = S; a.o = o;
    a.n_states = ns; a.d = d; a.dtype = dtype; a.mode = mode; a.phi = phi; a.eps = eps;
    a.flags = flags & (unsigned)FW_FLAG_RBW;
    cudaError_t e = launch_decode(a, stream);
    if (e != cudaSuccess) return cuda_fail(e);
    return FW_OK;
}

extern "C" int fw_step(const void *q, const void *k_prev, const void *v, const float *beta,
                       const float *lambda, float *S, void *o, const fw_shape *shape,
                       fw_dtype dtype, fw_mode mode, fw_phi phi, float eps,
                       cudaStream_t stream) {
    return fw_step_ex(q, k_prev, v, beta, lambda, S, o, shape, dtype, mode, phi, eps, 0u, stream);
}

extern "C" int fw_window_prefill(const void *q, const void *k, const void *v, const float *beta,
                                 const float *lambda, const float *S0, const void *k_init,
                                 const fw_window *win_in, void *o, float *S_T,
                                 const fw_window *win_out, const fw_shape *shape, int window,
                                 fw_dtype dtype, fw_mode mode, fw_phi phi, float eps,
                                 unsigned flags, cudaStream_t stream) {
    int st = check_common(shape, dtype, mode, phi, eps, flags);
    if (st != FW_OK) return st;
    if (!window_mode(mode)) return FW_ERR_MODE;
    if (window < 1 || window > FW_WINDOW_MAX) return FW_ERR_SHAPE;
    if (!q || !k || !v || !o || !S_T || !beta || !lambda) return FW_ERR_NULL;
    if (misaligned(q) || misaligned(k) || misaligned(v) || misaligned(o) || misaligned(S_T) ||
        misaligned(S0) || misaligned(k_init) || misaligned(beta) || misaligned(lambda))
        return FW_ERR_ALIGN;
    const int64_t nc = shape->B * shape->H;
    const int d = shape->d_k;
    const WinExtent we = win_extent(nc, window, d);
    if ((st = check_window(win_in, win_out, window, we)) != FW_OK) return st;

    const size_t esz = dtype == FW_F32 ? 4 : 2;
    const size_t nx = (size_t)nc * (size_t)shape->T * d * esz;
    const size_t ns = (size_t)nc * d * d * sizeof(float);
    const size_t nl = (size_t)nc * (size_t)shape->T * sizeof(float);
    const size_t nki = (size_t)nc * d * esz;
    if (overlaps(o, nx, q, nx) || overlaps(o, nx, k, nx) || overlaps(o, nx, v, nx) ||
        overlaps(o, nx, S0, S0 ? ns : 0) || overlaps(o, nx, S_T, ns) ||
        overlaps(o, nx, beta, nl) || overlaps(o, nx, lambda, nl) ||
        overlaps(o, nx, k_init, k_init ? nki : 0))
        return FW_ERR_ARG;
    if (overlaps(S_T, ns, q, nx) || overlaps(S_T, ns, k, nx) || overlaps(S_T, ns, v, nx) ||
        overlaps(S_T, ns, beta, nl) || overlaps(S_T, ns, lambda, nl) ||
        overlaps(S_T, ns, k_init, k_init ? nki : 0))
        return FW_ERR_ARG;
    if (S0 && S0 != S_T && overlaps(S_T, ns, S0, ns)) return FW_ERR_ARG;
    const bool carry_in = window > 1 && win_in, carry_out = window > 1 && win_out;
    if (carry_in && (win_overlaps(win_in, we, o, nx) || win_overlaps(win_in, we, S_T, ns)))
        return FW_ERR_ARG;
    if (carry_out) {
        const void *ins[] = {q, k, v, beta, lambda, S0, k_init, o, S_T};
        const size_t nin[] = {nx, nx, nx, nl, nl, S0 ? ns : 0, k_init ? nki : 0, nx, ns};
        for (int i = 0; i < 9; ++i)
            if (win_overlaps(win_out, we, ins[i], nin[i])) return FW_ERR_ARG;
    }

    WindowArgs a;
    a.q = q; a.k = k; a.v = v; a.beta = beta; a.lam = lambda; a.S0 = S0;
    a.k_init = (flags & FW_FLAG_SAME_PAIR) ? nullptr : k_init;
    a.cx = carry_in ? win_in->x : nullptr;
    a.cy = carry_in ? win_in->y : nullptr;
    a.cn = carry_in ? win_in->n : nullptr;
    a.o = o; a.S_T = S_T;
    a.ox = carry_out ? win_out->x : nullptr;
    a.oy = carry_out ? win_out->y : nullptr;
    a.on = carry_out ? win_out->n : nullptr;
    a.n_chains = nc; a.T = shape->T; a.d = d; a.W = window; a.dtype = dtype;
    a.inner = (mode == FW_FALCON3A); a.chan = false; a.phi = phi; a.eps = eps; a.flags = flags;
    a.wait_ns = g_wait_us.load() * 1000LL;

    if ((st = device_setup(&a.err)) != FW_OK) return st;
    cudaError_t e = launch_window_prefill(a, stream);
    if (e != cudaSuccess) return cuda_fail(e);
    return FW_OK;
}

extern "C" int fw_window_step(const void *q, const void *k_prev, const void *v,
                              const float *beta, const float *lambda, float *S,
                              const fw_window *win_in, void *o, const fw_window *win_out,
                              const fw_shape *shape, int window, fw_dtype dtype, fw_mode mode,
                              fw_phi phi, float eps, unsigned flags, cudaStream_t stream) {
    int st = check_common(shape, dtype, mode, phi, eps, flags);
    if (st != FW_OK) return st;
    if (!window_mode(mode)) return FW_ERR_MODE;
    if (flags & ~(unsigned)FW_FLAG_RBW) return FW_ERR_MODE;
    if (shape->T != 1 || window < 1 || window > FW_WINDOW_MAX) return FW_ERR_SHAPE;
    if (!q || !k_prev || !v || !S || !o || !beta || !lambda) return FW_ERR_NULL;
    if (misaligned(q) || misaligned(k_prev) || misaligned(v) || misaligned(S) || misaligned(o) ||
        misaligned(beta) || misaligned(lambda))
        return FW_ERR_ALIGN;
    const int64_t ns = shape->B * shape->H;
    const int d = shape->d_k;
    const WinExtent we = win_extent(ns, window, d);
    if ((st = check_window(win_in, win_out, window, we)) != FW_OK) return st;
    const size_t esz = dtype == FW_F32 ? 4 : 2;
    const size_t nx = (size_t)ns * d * esz;
    const size_t nst = (size_t)ns * d * d * sizeof(float);
    const size_t nl = (size_t)ns * sizeof(float);
    const void *ins[] = {q, k_prev, v, beta, lambda};
    const size_t nin[] = {nx, nx, nx, nl, nl};
    for (int i = 0; i < 5; ++i)
        if (overlaps(o, nx, ins[i], nin[i]) || overlaps(S, nst, ins[i], nin[i]))
            return FW_ERR_ARG;
    if (overlaps(o, nx, S, nst)) return FW_ERR_ARG;
    const bool carry_in = window > 1 && win_in, carry_out = window > 1 && win_out;
    if (carry_in && (win_overlaps(win_in, we, o, nx) || win_overlaps(win_in, we, S, nst)))
        return FW_ERR_ARG;
    if (carry_out) {
        for (int i = 0; i < 5; ++i)
            if (win_overlaps(win_out, we, ins[i], nin[i])) return FW_ERR_ARG;
        if (win_overlaps(win_out, we, o, nx) || win_overlaps(win_out, we, S, nst))
            return FW_ERR_ARG;
    }

    WindowArgs a;
    a.q = q; a.k = k_prev; a.v = v; a.beta = beta; a.lam = lambda; a.S0 = S;
    a.k_init = nullptr;
    a.cx = carry_in ? win_in->x : nullptr;
    a.cy = carry_in ? win_in->y : nullptr;
    a.cn = carry_in ? win_in->n : nullptr;
    a.o = o; a.S_T = S;
    a.ox = carry_out ? win_out->x : nullptr;
    a.oy = carry_out ? win_out->y : nullptr;
    a.on = carry_out ? win_out->n : nullptr;
    a.n_chains = ns; a.T = 1; a.d = d; a.W = window; a.dtype = dtype;
    a.inner = (mode == FW_FALCON3A); a.chan = false; a.phi = phi; a.eps = eps; a.flags = flags;
    a.wait_ns = g_wait_us.load() * 1000LL;

    if ((st = device_setup(&a.err)) != FW_OK) return st;
    cudaError_t e = launch_window_step(a, stream);
    if (e != cudaSuccess) return cuda_fail(e);
    return FW_OK;
}

extern "C" int fw_check(cudaStream_t stream) {
    cudaError_t e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return cuda_fail(e);
    int *err = nullptr;
    int st = device_setup(&err);
    if (st != FW_OK) return st;
    int h = 0;
    if ((e = cudaMemcpy(&h, err, sizeof(int), cudaMemcpyDeviceToHost)) != cudaSuccess)
        return cuda_fail(e);
    if (h != kDevErrNone) {
        const int zero = 0;
        if ((e = cudaMemcpy(err, &zero, sizeof(int), cudaMemcpyHostToDevice)) != cudaSuccess)
            return cuda_fail(e);
        return FW_ERR_TIMEOUT;
    }
    return FW_OK;
}

extern "C" const char *fw_status_string(int status) {
    switch (status) {
    case FW_OK: return "FW_OK";
    case FW_ERR_NULL: return "FW_ERR_NULL: a required pointer is NULL";
    case FW_ERR_SHAPE: return "FW_ERR_SHAPE: unsupported shape";
    case FW_ERR_DTYPE: return "FW_ERR_DTYPE: unknown dtype";
    case FW_ERR_ALIGN: return "FW_ERR_ALIGN: pointer not 16-byte aligned";
    case FW_ERR_MODE: return "FW_ERR_MODE: unknown mode, feature map or algorithm";
    case FW_ERR_CUDA: return "FW_ERR_CUDA: a CUDA call failed";
    case FW_ERR_TIMEOUT: return "FW_ERR_TIMEOUT: a bounded device wait ran out";
    case FW_ERR_UNSUPPORTED: return "FW_ERR_UNSUPPORTED: the chunked kernel does not take this call";
    case FW_ERR_ARG: return "FW_ERR_ARG: invalid eps or overlapping buffers";
    case FW_ERR_DEVICE: return "FW_ERR_DEVICE: the current device is not sm_103";
    case FW_ERR_SCRATCH: return "FW_ERR_SCRATCH: the call needs more than FW_SCRATCH_BYTES of scratch";
    default: return "unknown status";
    }
}

extern "C" int fw_version(void) { return FW_VERSION; }

extern "C" int fw_last_cuda_error(void) { return g_last_cuda_error; }

extern "C" void fw_set_wait_limit_us(long long us) {
    g_wait_us.store(us < 1 ? kDefaultWaitUs : us);
}

extern "C" void fw_debug_force_timeout(int on) { g_force_timeout.store(on ? 1 : 0); }

extern "C" void fw_debug_segment_split(int mode) { g_seg_pref.store(mode > 0 ? 1 : mode < 0 ? -1 : 0); }
