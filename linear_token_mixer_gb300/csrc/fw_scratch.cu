// fw_scratch.cu -- the static device buffer behind fw_prefill_noalloc.
//
// The chunked prefill's two-segment form needs workspace (the transition
// run's outputs and three states per chain).  fw_prefill_ex draws it from a
// stream-ordered pool; fw_prefill_noalloc takes it from this buffer instead,
// so that call allocates nothing.  The buffer sits in its own translation unit,
// so its module (and the memory) loads only when its address is first asked for.
#include <mutex>

#include "fw_internal.cuh"

static __device__ __align__(256) unsigned char g_segment_scratch[FW_SCRATCH_BYTES];

namespace fw {

void *segment_scratch(int dev, cudaError_t *e) {
    static std::mutex m;
    static void *addr[64] = {};
    *e = cudaSuccess;
    if (dev < 0 || dev >= 64) {
        *e = cudaErrorInvalidDevice;
        return nullptr;
    }
    std::lock_guard<std::mutex> lock(m);
    if (!addr[dev]) {
        void *p = nullptr;
        const cudaError_t r = cudaGetSymbolAddress(&p, g_segment_scratch);
        if (r != cudaSuccess) {
            cudaGetLastError();   // not sticky: leave no error behind for later calls
            *e = r;
            return nullptr;
        }
        addr[dev] = p;
    }
    return addr[dev];
}

}  // namespace fw
