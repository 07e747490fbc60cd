// spec_verify_chain_static: chain verification for callers that cannot
// allocate device memory.
//
// Some callers cannot call cudaMalloc at the point where they verify a round:
// code running inside a memory-pool or arena allocator that owns every device
// byte, plug-ins whose host framework forbids allocation on its hot path,
// and callers that must not trigger an allocation's implicit device
// synchronisation mid-stream.  For them this entry point takes its scratch
// memory (the per-request arrival counters, rejection words and per-position
// records that spec_verify_chain keeps in the caller's workspace) from a
// fixed array compiled into this library instead.
//
// The array lives in device memory of every GPU that loads the library and
// stays there until the process exits.  All calls on one GPU share it, so
// calls whose kernels could overlap on the GPU (different streams, or
// different host threads without ordering) race on it: issue them on one
// stream.  It keeps the previous call's contents; each call clears the part
// that must start at zero before launching.
#include <cstdio>
#include <mutex>

#include "kernels.h"
#include "spec_verify.h"

namespace {

constexpr size_t kStaticWsBytes = size_t(1) << 20;  // SPEC_STATIC_WORKSPACE_BYTES
static_assert(kStaticWsBytes == SPEC_STATIC_WORKSPACE_BYTES, "header and library disagree");

static __device__ __align__(256) unsigned char g_static_ws[kStaticWsBytes];

constexpr int kMaxDevices = 64;
void *g_ws_ptr[kMaxDevices];
cudaError_t g_ws_err[kMaxDevices];
std::once_flag g_ws_once[kMaxDevices];

}  // namespace

extern "C" int spec_verify_chain_static(const SpecChainArgs *a, void *stream) {
    // every host-side check comes before the memset below, so a rejected
    // call enqueues nothing
    const int chk = specv::chain_args_check(a);
    if (chk != SPEC_OK) return chk;
    if (a->B == 0) return SPEC_OK;
    const size_t need = spec_workspace_bytes(SPEC_WS_CHAIN, a->B, a->gamma, a->V);
    if (need > kStaticWsBytes) return SPEC_ERR_TOO_LARGE;

    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return SPEC_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return SPEC_ERR_UNSUPPORTED;
    // once per device, with that device current: the array's device address
    std::call_once(g_ws_once[dev], [dev] {
        void *ptr = nullptr;
        g_ws_err[dev] = cudaGetSymbolAddress(&ptr, g_static_ws);
        g_ws_ptr[dev] = ptr;
    });
    if (g_ws_err[dev] != cudaSuccess || g_ws_ptr[dev] == nullptr) return SPEC_ERR_CUDA;

    // status word, arrival counters and rejection words must start at zero
    const size_t zeroed = specv::kWsHeader + 2 * specv::ws_align((size_t)a->B * sizeof(unsigned));
    e = cudaMemsetAsync(g_ws_ptr[dev], 0, zeroed, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return SPEC_ERR_CUDA;
    // the plain chain workspace only: the candidate regions and the
    // full-vocabulary path's state are not part of this array's contract
    return spec_verify_chain(a, g_ws_ptr[dev], need, stream);
}
