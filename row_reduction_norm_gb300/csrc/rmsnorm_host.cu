// rmsnorm_host.cu -- rmsnorm_fwd_host: the op on rows that live in host
// memory, streamed through the device in chunks (declared in
// include/rmsnorm.h).  Host code only: every chunk is one rmsnorm_fwd launch
// on device copies in the caller's workspace, so the arithmetic is the
// kernels' and the results are rmsnorm_fwd's, bit for bit.
//
// Pipeline, per device: three streams -- uploads, launches, read-backs --
// and two halves of the workspace.  Chunk i uses half i % 2:
//   uploads:    wait until half's previous read-back is done; copy the
//               chunk's x (and residual) in; record in[half]
//   launches:   wait in[half]; rmsnorm_fwd on the half; record done[half]
//   read-backs: wait done[half]; copy y (and residual_out) out; record
//               out[half]
// so chunk i + 1's uploads run while chunk i is normalised and chunk i - 1
// read back; host-to-device and device-to-host copies go both ways at once.
// The caller's stream orders the call: the uploads wait for the work issued
// on it before the call, and it waits for the last read-backs.  The weight
// is uploaded once per call, after every earlier call's launches on the
// device are done (they may read the same workspace).
#include <cstdint>
#include <cstring>
#include <mutex>

#include <cuda_runtime.h>

#include "rmsnorm.h"

namespace {

constexpr int kMaxDevices = 64;
constexpr int64_t kAlign = 256;

int64_t round_up(int64_t v) { return (v + kAlign - 1) / kAlign * kAlign; }

int elem_bytes(int dtype) { return dtype == RMSNORM_BF16 ? 2 : 4; }

struct Pipe {
    std::mutex mu;
    bool ready = false;
    cudaStream_t up = nullptr, run = nullptr, down = nullptr;
    cudaEvent_t start = nullptr;
    cudaEvent_t in[2] = {nullptr, nullptr};
    cudaEvent_t done[2] = {nullptr, nullptr};
    cudaEvent_t out[2] = {nullptr, nullptr};
};

Pipe g_pipes[kMaxDevices];

// Creates the device's streams and events once (the caller holds P.mu).
int ensure_pipe(Pipe &P) {
    if (P.ready) return RMSNORM_OK;
    const unsigned f = cudaStreamNonBlocking;
    if (cudaStreamCreateWithFlags(&P.up, f) != cudaSuccess || cudaStreamCreateWithFlags(&P.run, f) != cudaSuccess ||
        cudaStreamCreateWithFlags(&P.down, f) != cudaSuccess)
        return RMSNORM_ECUDA;
    cudaEvent_t *all[] = {&P.start, &P.in[0], &P.in[1], &P.done[0], &P.done[1], &P.out[0], &P.out[1]};
    for (cudaEvent_t *e : all)
        if (cudaEventCreateWithFlags(e, cudaEventDisableTiming) != cudaSuccess) return RMSNORM_ECUDA;
    P.ready = true;
    return RMSNORM_OK;
}

// Byte offsets of the workspace's parts: the weight, then per half x, y and,
// with a residual, residual and residual_out, each 256-byte aligned.
struct Layout {
    int64_t chunk_bytes = 0;   // one tensor's chunk
    int64_t w = 0;
    int64_t half[2][4] = {};   // x, y, residual, residual_out
    int64_t total = 0;
};

bool layout_of(int64_t chunk_rows, int64_t row_bytes, bool res, Layout *L) {
    if (chunk_rows > INT64_MAX / 8 / row_bytes) return false;
    L->chunk_bytes = chunk_rows * row_bytes;
    const int64_t part = round_up(L->chunk_bytes);
    int64_t at = round_up(row_bytes);   // the weight first
    L->w = 0;
    const int parts = res ? 4 : 2;
    for (int h = 0; h < 2; ++h) {
        for (int k = 0; k < 4; ++k) L->half[h][k] = -1;
        for (int k = 0; k < parts; ++k) {
            L->half[h][k] = at;
            at += part;
        }
    }
    L->total = at;
    return true;
}

}  // namespace

extern "C" {

int64_t rmsnorm_host_workspace_bytes(int64_t chunk_rows, int64_t hidden, int dtype, int has_residual) {
    if (dtype != RMSNORM_F32 && dtype != RMSNORM_BF16) return RMSNORM_EINVAL;
    if (chunk_rows < 1 || hidden < 1 || (has_residual != 0 && has_residual != 1)) return RMSNORM_EINVAL;
    if (hidden > rmsnorm_max_hidden(dtype)) return RMSNORM_EUNSUPPORTED;
    Layout L;
    if (!layout_of(chunk_rows, hidden * elem_bytes(dtype), has_residual == 1, &L)) return RMSNORM_EINVAL;
    return L.total;
}

int rmsnorm_fwd_host(const void *x, const void *residual, const void *w, void *y, void *residual_out,
                     int64_t rows, int64_t hidden, float eps, int dtype, void *workspace, uint64_t workspace_bytes,
                     int64_t chunk_rows, rmsnorm_stream_t stream) {
    // the op's own argument checks, without touching memory (zero rows)
    int st = rmsnorm_fwd(nullptr, nullptr, nullptr, nullptr, nullptr, 0, hidden, eps, dtype, stream);
    if (st != RMSNORM_OK) return st;
    if (rows < 0 || chunk_rows < 1) return RMSNORM_EINVAL;
    if (rows == 0) return RMSNORM_OK;
    if (x == nullptr || y == nullptr || (residual == nullptr) != (residual_out == nullptr)) return RMSNORM_EINVAL;
    const bool res = residual != nullptr;
    const int64_t row_bytes = hidden * elem_bytes(dtype);
    if (rows > INT64_MAX / row_bytes) return RMSNORM_EINVAL;
    Layout L;
    if (!layout_of(chunk_rows, row_bytes, res, &L)) return RMSNORM_EINVAL;
    if (workspace == nullptr || reinterpret_cast<uintptr_t>(workspace) % kAlign != 0 ||
        workspace_bytes < (uint64_t)L.total)
        return RMSNORM_EINVAL;

    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return RMSNORM_ECUDA;
    Pipe &P = g_pipes[dev];
    std::lock_guard<std::mutex> lk(P.mu);
    if ((st = ensure_pipe(P)) != RMSNORM_OK) return st;

    char *ws = static_cast<char *>(workspace);
    const char *hx = static_cast<const char *>(x);
    const char *hr = static_cast<const char *>(residual);
    char *hy = static_cast<char *>(y);
    char *hh = static_cast<char *>(residual_out);
    cudaStream_t caller = reinterpret_cast<cudaStream_t>(stream);
    bool ok = true;
    auto cu = [&ok](cudaError_t e) { ok = ok && e == cudaSuccess; };

    cu(cudaEventRecord(P.start, caller));
    cu(cudaStreamWaitEvent(P.up, P.start, 0));
    // an earlier call's launches may still read the weight's slot
    cu(cudaStreamWaitEvent(P.up, P.done[0], 0));
    cu(cudaStreamWaitEvent(P.up, P.done[1], 0));
    if (w != nullptr) cu(cudaMemcpyAsync(ws + L.w, w, row_bytes, cudaMemcpyHostToDevice, P.up));

    int64_t i = 0;
    for (int64_t r0 = 0; r0 < rows && ok; r0 += chunk_rows, ++i) {
        const int64_t n = rows - r0 < chunk_rows ? rows - r0 : chunk_rows;
        const int h = (int)(i & 1);
        const int64_t off = r0 * row_bytes, bytes = n * row_bytes;
        char *dx = ws + L.half[h][0], *dy = ws + L.half[h][1];
        char *dr = res ? ws + L.half[h][2] : nullptr, *dh = res ? ws + L.half[h][3] : nullptr;
        // uploads, once this half's previous read-back (hence its launch) is done
        cu(cudaStreamWaitEvent(P.up, P.out[h], 0));
        cu(cudaMemcpyAsync(dx, hx + off, bytes, cudaMemcpyHostToDevice, P.up));
        if (res) cu(cudaMemcpyAsync(dr, hr + off, bytes, cudaMemcpyHostToDevice, P.up));
        cu(cudaEventRecord(P.in[h], P.up));
        // the launch
        cu(cudaStreamWaitEvent(P.run, P.in[h], 0));
        if (!ok) break;
        st = rmsnorm_fwd(dx, dr, w != nullptr ? ws + L.w : nullptr, dy, dh, n, hidden, eps, dtype,
                         reinterpret_cast<rmsnorm_stream_t>(P.run));
        if (st != RMSNORM_OK) break;
        cu(cudaEventRecord(P.done[h], P.run));
        // read-backs
        cu(cudaStreamWaitEvent(P.down, P.done[h], 0));
        cu(cudaMemcpyAsync(hy + off, dy, bytes, cudaMemcpyDeviceToHost, P.down));
        if (res) cu(cudaMemcpyAsync(hh + off, dh, bytes, cudaMemcpyDeviceToHost, P.down));
        cu(cudaEventRecord(P.out[h], P.down));
    }
    // work issued on the caller's stream after this call follows the read-backs
    // (on an error too: whatever was queued still uses the workspace)
    cu(cudaEventRecord(P.in[0], P.up));
    cu(cudaStreamWaitEvent(caller, P.in[0], 0));
    cu(cudaEventRecord(P.done[0], P.run));
    cu(cudaStreamWaitEvent(caller, P.done[0], 0));
    cu(cudaStreamWaitEvent(caller, P.out[0], 0));
    cu(cudaStreamWaitEvent(caller, P.out[1], 0));
    if (st != RMSNORM_OK) return st;
    if (!ok) {
        (void)cudaGetLastError();
        return RMSNORM_ECUDA;
    }
    return RMSNORM_OK;
}

}  // extern "C"
