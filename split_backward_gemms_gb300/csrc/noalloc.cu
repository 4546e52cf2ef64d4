// noalloc.cu — the schedule replay with its activation arena in a static
// device array, for callers that cannot allocate device memory themselves.
//
// Who cannot allocate: code that runs inside a framework or server that
// owns all device memory through its own pool (a custom operator or plugin
// handed only input and output buffers), and latency-critical loops that must
// never call cudaMalloc / cudaFree, which may synchronise the whole device and
// stall every other stream.  Such callers can still pass inputs and outputs;
// this entry point supplies the scratch (the deferred-W activation arena of
// the replay) from a fixed array instead of a caller workspace.
#include <cuda_runtime.h>

#include <mutex>
#include <string>

#include "zb_internal.h"

namespace {

constexpr size_t kStaticArenaBytes = static_cast<size_t>(ZB_STATIC_ARENA_BYTES);

// The arena: one copy per device that uses this entry point, held from its
// first call on that device until the process exits.  Every call shares it.
static __device__ __align__(256) unsigned char g_zb_static_arena[kStaticArenaBytes];

// Device address of the array on the current device.  In host code the
// symbol is only a host-side stand-in; its device address is resolved once
// per device (with that device current) and cached.
void* static_arena_address(std::string* why) {
    static std::mutex mu;
    static void* addr[64] = {nullptr};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) {
        *why = std::string("cudaGetDevice: ") + cudaGetErrorString(e);
        return nullptr;
    }
    if (dev < 0 || dev >= 64) {
        *why = "device ordinal out of range";
        return nullptr;
    }
    std::lock_guard<std::mutex> lk(mu);
    if (!addr[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_zb_static_arena);
        if (e != cudaSuccess || p == nullptr) {
            *why = std::string("cudaGetSymbolAddress(static arena): ") + cudaGetErrorString(e);
            return nullptr;
        }
        addr[dev] = p;
    }
    return addr[dev];
}

}  // namespace

extern "C" zb_status zb_run_stage_schedule_static(const zb_pipeline* pl, const zb_stage_params* stages,
                                                  const void* const* X0, const void* const* dY_last,
                                                  void* const* dX0_out, void* const* Y_last_out,
                                                  const zb_op* ops, size_t n_ops, zb_run_stats* stats,
                                                  void* stream) {
    if (!pl) return zb::fail(ZB_ERR_INVALID_ARG, "pipeline is NULL");
    if (pl->timing) return zb::fail(ZB_ERR_INVALID_ARG, "timing mode creates CUDA events; use zb_run_stage_schedule");
    if (pl->streams > 1)
        return zb::fail(ZB_ERR_INVALID_ARG, "stage-parallel replay uses library streams; use zb_run_stage_schedule");
    size_t need = 0;
    zb_status s = zb_schedule_workspace_size(pl, ops, n_ops, &need, nullptr);
    if (s != ZB_OK) return s;
    if (need > kStaticArenaBytes)
        return zb::fail(ZB_ERR_WORKSPACE, "this op list needs a " + std::to_string(need) +
                                              "-byte arena; the static arena holds " +
                                              std::to_string(kStaticArenaBytes) +
                                              " bytes (use zb_run_stage_schedule with a workspace)");
    std::string why;
    void* arena = static_arena_address(&why);
    if (!arena) return zb::fail(ZB_ERR_CUDA, why);
    // The replay writes every arena buffer before reading it, so the previous
    // call's leftovers need no clearing.
    return zb_run_stage_schedule(pl, stages, X0, dY_last, dX0_out, Y_last_out, ops, n_ops, arena,
                                 kStaticArenaBytes, stats, stream);
}
