// decode_noalloc.cu -- kivi_decode_attend_noalloc: the fused decode with its
// split scratch in a fixed, library-owned device array instead of a
// caller-provided workspace.
//
// Who needs it: callers that cannot allocate device memory at the time they
// decode. Examples are serving runtimes that carve all of HBM into weights and
// KV-cache pages up front and forbid any later allocation (a late cudaMalloc
// can fail there, or stall the whole device while it synchronises), and plain C
// callers that receive device pointers from a framework owning the memory pool
// and have no allocator of their own to get a workspace from.
//
// The scratch is a file-scope __device__ array of KIVI_NOALLOC_SCRATCH_BYTES.
// It exists once per device that loads this library and stays allocated until
// the process exits. Every call on a device uses the same array:
//   * calls whose kernels overlap on that device (e.g. issued on two streams
//     without ordering) race on the scratch and give wrong results -- order them
//     on one stream or with events;
//   * the merge counters at its start must be zero when a call begins: a
//     __device__ array is zero-initialised when the module loads, and every
//     completed call leaves the counters zero; each call writes every partial
//     it later reads, and the array keeps the last call's contents afterwards.
// Host code cannot use the array's name as a device address, so each call
// looks the address up with cudaGetSymbolAddress (with the pointers' device
// current). The lookup is repeated on every call made outside stream capture,
// so a module reloaded after cudaDeviceReset (or after the primary context
// was released and created again) is found at its new address, with its
// counters zero again. Inside a stream capture the call uses the address the
// last uncaptured call on that device found: make one call on each device
// before capturing any stream (that first call may also load the library's
// device code, which a capture must not do).
#include <atomic>

#include "../../include/kivi.h"
#include "kivi_launch.h"

namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[KIVI_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::atomic<void*> g_scratch_addr[kMaxDevices];

// Device address of the scratch array on the current device, or nullptr.
// Looked up afresh outside stream capture; inside a capture, the address the
// last uncaptured lookup on this device found.
void* scratch_address(cudaStream_t stream) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return nullptr;
    }
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(stream, &cs) != cudaSuccess) {
        cudaGetLastError();
        return nullptr;
    }
    if (cs != cudaStreamCaptureStatusNone) return g_scratch_addr[dev].load(std::memory_order_acquire);
    void* addr = nullptr;
    if (cudaGetSymbolAddress(&addr, g_noalloc_scratch) != cudaSuccess || addr == nullptr) {
        cudaGetLastError();
        return nullptr;
    }
    g_scratch_addr[dev].store(addr, std::memory_order_release);
    return addr;
}

}  // namespace

extern "C" kivi_status kivi_decode_attend_noalloc(
    const void* q_f16, const void* kcodes_u8, const float* kscale, const void* kzero_f16,
    const void* vcodes_u8, const float* vscale, const void* vzero_f16, int S_q, int s_cap,
    const void* k_res_f16, const void* v_res_f16, int n_res, int res_cap, int B, int Hq, int Hkv,
    int D, int group_size, int bits, float sm_scale, float* out_f32, kivi_stream_t stream) {
    // Reject work whose split scratch would not fit before touching the device:
    // the need of the exact plan this call takes (its bit width, group size
    // and scale storage), not the largest over all of them.
    const size_t need = kivi::decode_workspace_need(B, Hq, Hkv, S_q, n_res, D, group_size, bits);
    if (need > (size_t)KIVI_NOALLOC_SCRATCH_BYTES) return KIVI_ERR_WORKSPACE;
    void* scratch = nullptr;
    if (need > 0) {
        scratch = scratch_address(reinterpret_cast<cudaStream_t>(stream));
        if (!scratch) return KIVI_ERR_CUDA;
    }
    // All argument checks and launches are those of kivi_decode_attend.
    return kivi_decode_attend(q_f16, kcodes_u8, kscale, kzero_f16, vcodes_u8, vscale, vzero_f16, S_q,
                              s_cap, k_res_f16, v_res_f16, n_res, res_cap, B, Hq, Hkv, D, group_size,
                              bits, sm_scale, out_f32, scratch, need > 0 ? (size_t)KIVI_NOALLOC_SCRATCH_BYTES : 0,
                              stream);
}
