// moe_router_topk_noalloc: the router call for callers that cannot allocate
// device memory — for example a host engine that plans all device memory when it
// starts and then calls its plugins from an enqueue path where allocation is not
// allowed, or a service that runs inside a fixed device-memory budget. Such a
// caller has no way to provide moe_router_topk's workspace on demand.
//
// The router's scratch (per-tile counts and probability sums, their scans and
// the device error word) lives here instead, in one file-scope device array of
// kNoAllocScratchBytes. Every GPU that loads libmoe.so holds that array until the
// process exits. The caller still passes every input and output buffer.
//
// Set-up: the first call on a device looks up the array's device address with
// that device current (cudaGetSymbolAddress) and caches it per device; make that
// first call before any stream capture. All calls share the one array and it keeps
// the previous call's contents: the error word is cleared at the start of every
// call and every other scratch region is fully rewritten before it is read. Calls
// that overlap on the GPU (different streams, or different host threads) race on
// the array and must be serialised by the caller.
#include <mutex>

#include "internal.h"

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(32) << 20;  // 32 MiB
constexpr int kMaxDevices = 64;

__device__ __align__(256) uint8_t g_router_scratch[kNoAllocScratchBytes];

void *g_scratch_addr[kMaxDevices];  // device address of g_router_scratch, per device
std::mutex g_scratch_mu;

moe_status scratch_of_current_device(uint8_t **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MOE_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (!g_scratch_addr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_router_scratch) != cudaSuccess || p == nullptr) return MOE_ERR_CUDA;
        g_scratch_addr[dev] = p;
    }
    *out = static_cast<uint8_t *>(g_scratch_addr[dev]);
    return MOE_OK;
}

}  // namespace

extern "C" moe_status moe_router_topk_noalloc(const moe_config *cfg, const void *x, const float *w_r,
                                              const float *b_r, int32_t *topk_idx, float *topk_gate,
                                              int32_t *counts_routed, int32_t *counts_kept,
                                              int32_t *expert_offsets, int32_t *slot_row, int32_t *perm_token,
                                              float *aux, cudaStream_t stream) {
    moe_status st = moe_validate_config(cfg);
    if (st != MOE_OK) return st;
    const moe_config &c = *cfg;
    if (c.routing != MOE_ROUTING_TOKEN_CHOICE) return MOE_ERR_UNSUPPORTED;
    if (!x || !w_r || !topk_idx || !topk_gate || !expert_offsets || !slot_row || !perm_token)
        return MOE_ERR_INVALID_ARG;
    if (c.has_router_bias && !b_r) return MOE_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(x) % 16 || reinterpret_cast<uintptr_t>(w_r) % 16) return MOE_ERR_INVALID_ARG;
    // the router's scratch is the workspace prefix that ends where the hidden buffer starts
    const size_t need = moe::ws_layout(c).hid;
    if (need > kNoAllocScratchBytes) return MOE_ERR_UNSUPPORTED;
    uint8_t *scratch = nullptr;
    if ((st = scratch_of_current_device(&scratch)) != MOE_OK) return st;
    if (cudaMemsetAsync(scratch + moe::ws_layout(c).err, 0, sizeof(uint32_t), stream) != cudaSuccess)
        return MOE_ERR_CUDA;
    moe::RouterOut o{topk_idx, topk_gate, counts_routed, counts_kept, expert_offsets, slot_row, perm_token, aux};
    const cudaError_t e = moe::launch_router(c, x, w_r, c.has_router_bias ? b_r : nullptr, o, scratch, stream);
    return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

// The device error word of the static array (the first word of the router's scratch
// for every config): bounded waits that ran out and out-of-range indices of the calls
// since the last call started. A caller without a workspace has no other way to see
// them, and a call whose wait ran out has unwritten outputs.
extern "C" moe_status moe_router_noalloc_check_error(cudaStream_t stream) {
    uint8_t *scratch = nullptr;
    moe_status st = scratch_of_current_device(&scratch);
    if (st != MOE_OK) return st;
    if (cudaStreamSynchronize(stream) != cudaSuccess) return MOE_ERR_CUDA;
    static_assert(sizeof(uint32_t) <= kNoAllocScratchBytes, "error word inside the array");
    uint32_t word = 0;
    if (cudaMemcpy(&word, scratch, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess) return MOE_ERR_CUDA;
    if (word && cudaMemset(scratch, 0, sizeof(word)) != cudaSuccess) return MOE_ERR_CUDA;
    if (word & moe::kErrTimeout) return MOE_ERR_TIMEOUT;
    if (word & moe::kErrFault) return MOE_ERR_DEVICE_FAULT;
    return MOE_OK;
}
