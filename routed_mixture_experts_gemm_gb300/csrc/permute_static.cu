// moe_permute_static: the token permutation of moe_permute, with its scratch
// taken from a fixed device array inside this library instead of a
// caller-provided workspace, for callers that cannot allocate device memory.
//
// Why some callers cannot allocate: cudaMalloc / cudaFree may synchronise
// the whole device and stall every stream, which a latency-bound decode loop
// cannot afford; and a process whose device memory is owned by another
// framework's pool (a serving runtime's arena, a caching allocator) must not
// take memory behind that pool's back.  Such callers still own and pass the
// inputs and outputs; only the scratch moves into this file.
//
// The scratch is one file-scope array per device (every GPU that loads the
// library holds it until the process exits).  In host code its name is only
// a host-side stand-in, so the host resolves the device address with
// cudaGetSymbolAddress, once per device, with that device current, on the
// first call made on that device; make that first call before any stream
// capture.  Every call shares the array and it keeps the previous call's
// contents: the permutation's first kernel rewrites every scratch entry it
// later reads (per-worker histograms) and resets the completion counter, so
// nothing stale is read.  Calls that overlap on the GPU (other streams,
// other threads) race on the array and must be serialised by the caller.
#include <cuda_runtime.h>

#include <mutex>

#include "gbmoe.h"
#include "internal.h"

namespace gbmoe {
namespace {

constexpr size_t kStaticScratchBytes = size_t(1) << 20;  // 1 MiB
static __device__ __align__(256) unsigned char g_permute_scratch[kStaticScratchBytes];

std::mutex g_scratch_mu;
void* g_scratch_ptr[kMaxDevices];

// Device address of this device's scratch array (nullptr on failure); the
// device must be the current one.
void* scratch_ptr(int device) {
    if (device < 0 || device >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lk(g_scratch_mu);
    if (!g_scratch_ptr[device]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_permute_scratch) != cudaSuccess) return nullptr;
        g_scratch_ptr[device] = p;
    }
    return g_scratch_ptr[device];
}

}  // namespace
}  // namespace gbmoe

using namespace gbmoe;

extern "C" int moe_permute_static(const int32_t* ids_phys, int T, int k, int E_phys,
                                  const uint16_t* x, int H, int32_t* counts, int32_t* offsets,
                                  int32_t* row_to_token, int32_t* flat_to_row, uint16_t* x_perm,
                                  gbmoe_stream_t stream) {
    int64_t N = 0;
    const int st = check_permute_args(ids_phys, T, k, E_phys, x, H, counts, offsets,
                                      row_to_token, flat_to_row, x_perm, &N);
    if (st) return st;
    if (permute_ws_bytes(N, E_phys) > kStaticScratchBytes) return GBMOE_ERR_WORKSPACE;
    const DevCtx* ctx = device_ctx();
    if (!ctx) return GBMOE_ERR_CUDA;
    void* ws = scratch_ptr(ctx->device);
    if (!ws) return GBMOE_ERR_CUDA;
    const cudaError_t e = launch_permute(ids_phys, N, k, E_phys, x, H, counts, offsets,
                                         row_to_token, flat_to_row, x_perm, ws, *ctx,
                                         reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? GBMOE_OK : GBMOE_ERR_CUDA;
}
