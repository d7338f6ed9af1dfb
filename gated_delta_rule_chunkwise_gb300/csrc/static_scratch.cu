// Library-owned device scratch for ldn_chunk_fwd_noalloc: one statically sized
// __device__ array per device, so that the split variant can run without the
// caller providing (or the library allocating) a workspace.
//
// The array lives in this translation unit's own module.  Under lazy module
// loading (the CUDA default) the runtime loads that module, and so backs the
// array with device memory, when its symbol is first resolved: at the first
// call on a device that needs the scratch.  Under CUDA_MODULE_LOADING=EAGER
// every module loads with the library, so each device the process uses holds
// the 256 MiB from then on.
//
// The first call on a device resolves the address and creates the event
// below; it must not be made while its stream is being captured into a CUDA
// graph (it returns LDN_ERR_UNSUPPORTED and enqueues nothing).  The stream
// must belong to the current device: the lock, the array's address and the
// event are per device.  Outside a capture a stream of another device returns
// LDN_ERR_INVALID_ARG (a capturing stream is not asked for its device: the
// query would invalidate the capture).
//
// All calls of a process on one device share the array.  acquire() takes a
// per-device host lock and makes the caller's stream wait for the event that
// the previous user recorded after its last launch; release() records that
// event on the caller's stream and drops the lock.  Calls on different
// streams therefore use the scratch one after another in device order.  While
// a stream is being captured into a CUDA graph the event is neither waited on
// nor recorded (an event from outside a capture cannot join it): replays of
// such a graph must be ordered with other users of the scratch by the caller.
#include <mutex>

#include "ldn_internal.cuh"

namespace ldn {
namespace {

__device__ __align__(256) uint8_t g_scratch[kStaticScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_lock[kMaxDevices];
void *g_addr[kMaxDevices] = {nullptr};
cudaEvent_t g_done[kMaxDevices] = {nullptr};

bool capturing(cudaStream_t s)
{
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(s, &cs) != cudaSuccess) return false;
    return cs != cudaStreamCaptureStatusNone;
}

}  // namespace

int static_scratch_acquire(cudaStream_t s, uint8_t **ptr, size_t *bytes, int *device)
{
    int dev = 0, sdev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return LDN_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return LDN_ERR_UNSUPPORTED;
    const bool cap = capturing(s);
    // (querying a capturing stream's device invalidates the capture: checked outside captures)
    if (!cap && (cudaStreamGetDevice(s, &sdev) != cudaSuccess || sdev != dev)) return LDN_ERR_INVALID_ARG;
    g_lock[dev].lock();
    if (!g_addr[dev]) {
        if (cap) {   // set-up (symbol resolution, event creation) stays out of captures
            g_lock[dev].unlock();
            return LDN_ERR_UNSUPPORTED;
        }
        void *p = nullptr;
        cudaError_t e = cudaGetSymbolAddress(&p, g_scratch);
        if (e == cudaSuccess) e = cudaEventCreateWithFlags(&g_done[dev], cudaEventDisableTiming);
        if (e != cudaSuccess) {
            g_lock[dev].unlock();
            return LDN_ERR_CUDA;
        }
        g_addr[dev] = p;
    } else if (!cap) {
        if (cudaStreamWaitEvent(s, g_done[dev], 0) != cudaSuccess) {
            g_lock[dev].unlock();
            return LDN_ERR_CUDA;
        }
    }
    *ptr = (uint8_t *)g_addr[dev];
    *bytes = kStaticScratchBytes;
    *device = dev;
    return LDN_OK;
}

cudaError_t static_scratch_release(cudaStream_t s, int device)
{
    cudaError_t e = cudaSuccess;
    if (!capturing(s)) e = cudaEventRecord(g_done[device], s);
    g_lock[device].unlock();
    return e;
}

}  // namespace ldn
