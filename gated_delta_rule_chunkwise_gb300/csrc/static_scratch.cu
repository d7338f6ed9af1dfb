// Library-owned device scratch for ldn_chunk_fwd_noalloc: one statically sized
// __device__ array per device, so that the split variant can run without the
// caller providing (or the library allocating) a workspace.
//
// The array lives in this translation unit's own module, which the CUDA
// runtime loads (and so backs with device memory) only when its symbol is
// first resolved, i.e. at the first ldn_chunk_fwd_noalloc call on a device.
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

cudaError_t static_scratch_acquire(cudaStream_t s, uint8_t **ptr, size_t *bytes, int *device)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    g_lock[dev].lock();
    if (!g_addr[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_scratch);
        if (e == cudaSuccess) e = cudaEventCreateWithFlags(&g_done[dev], cudaEventDisableTiming);
        if (e != cudaSuccess) {
            g_lock[dev].unlock();
            return e;
        }
        g_addr[dev] = p;
    } else if (!capturing(s)) {
        e = cudaStreamWaitEvent(s, g_done[dev], 0);
        if (e != cudaSuccess) {
            g_lock[dev].unlock();
            return e;
        }
    }
    *ptr = (uint8_t *)g_addr[dev];
    *bytes = kStaticScratchBytes;
    *device = dev;
    return cudaSuccess;
}

cudaError_t static_scratch_release(cudaStream_t s, int device)
{
    cudaError_t e = cudaSuccess;
    if (!capturing(s)) e = cudaEventRecord(g_done[device], s);
    g_lock[device].unlock();
    return e;
}

}  // namespace ldn
