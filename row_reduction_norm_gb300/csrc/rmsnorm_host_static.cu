// rmsnorm_host_static.cu -- rmsnorm_fwd_host_static: rmsnorm_fwd_host with
// the library's own device scratch in place of a caller workspace, so the
// call allocates nothing and takes no workspace argument.
//
// The scratch is a file-scope __device__ array: the CUDA runtime places it
// with this translation unit's module (no kernel lives here, so with lazy
// module loading it is claimed when its address is first asked for), and
// each device gets its own copy.  Its address is taken once per device with
// cudaGetSymbolAddress.  Host code apart from the array; the chunked
// pipeline is rmsnorm_fwd_host's, whose per-device streams, events and lock
// also order calls that share this scratch.
#include <cstdint>
#include <mutex>

#include <cuda_runtime.h>

#include "rmsnorm.h"

namespace {

constexpr uint64_t kScratchBytes = 64ull << 20;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

std::mutex g_mu;
void *g_addr[kMaxDevices];

int scratch_of(int dev, void **out) {
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_addr[dev] == nullptr) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_scratch) != cudaSuccess || p == nullptr) {
            (void)cudaGetLastError();
            return RMSNORM_ECUDA;
        }
        g_addr[dev] = p;
    }
    *out = g_addr[dev];
    return RMSNORM_OK;
}

// Rows a chunk of the scratch holds: the weight, then two halves of two (or,
// with a residual, four) parts of whole rows, each on a 256-byte boundary --
// the layout rmsnorm_host_workspace_bytes sizes.
int64_t chunk_rows_of(int64_t hidden, int dtype, int has_residual) {
    const int64_t row_bytes = hidden * (dtype == RMSNORM_BF16 ? 2 : 4);
    int64_t lo = 1, hi = (int64_t)kScratchBytes / row_bytes + 1;
    if (rmsnorm_host_workspace_bytes(1, hidden, dtype, has_residual) > (int64_t)kScratchBytes) return 0;
    while (hi - lo > 1) {   // the largest count whose workspace fits
        const int64_t mid = lo + (hi - lo) / 2;
        const int64_t need = rmsnorm_host_workspace_bytes(mid, hidden, dtype, has_residual);
        if (need > 0 && need <= (int64_t)kScratchBytes)
            lo = mid;
        else
            hi = mid;
    }
    return lo;
}

}  // namespace

extern "C" int rmsnorm_fwd_host_static(const void *x, const void *residual, const void *w, void *y,
                                       void *residual_out, int64_t rows, int64_t hidden, float eps, int dtype,
                                       rmsnorm_stream_t stream) {
    // the op's argument checks first (rows == 0 touches nothing)
    int st = rmsnorm_fwd(nullptr, nullptr, nullptr, nullptr, nullptr, 0, hidden, eps, dtype, stream);
    if (st != RMSNORM_OK) return st;
    if (rows < 0) return RMSNORM_EINVAL;
    if (rows == 0) return RMSNORM_OK;
    const int64_t chunk = chunk_rows_of(hidden, dtype, residual != nullptr ? 1 : 0);
    if (chunk < 1) return RMSNORM_EUNSUPPORTED;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return RMSNORM_ECUDA;
    void *scratch = nullptr;
    if ((st = scratch_of(dev, &scratch)) != RMSNORM_OK) return st;
    return rmsnorm_fwd_host(x, residual, w, y, residual_out, rows, hidden, eps, dtype, scratch, kScratchBytes,
                            chunk, stream);
}
