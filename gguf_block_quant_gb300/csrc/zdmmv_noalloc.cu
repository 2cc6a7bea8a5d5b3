// zdmmv_noalloc.cu -- the LM-head argmax DMMV for callers that cannot allocate.
//
// zdmmv_dmmv_argmax needs an 8-byte partial per CTA in a caller-provided device
// workspace. Some callers cannot hand one over: an inference engine that plans
// every byte of device memory when it loads a model and treats any later
// allocation as a bug, a plugin running inside a host program that owns all
// device memory, or a latency-critical decode loop that must not call
// cudaMalloc (which can synchronize the device and stall every stream). For
// them, zdmmv_dmmv_argmax_noalloc keeps its scratch in a fixed array that lives
// in this library's device image: the array exists on every GPU that loads the
// library, for as long as the process runs, and is never allocated or freed.
//
// Contract (also in include/zdmmv.h): the array holds kNoAllocSlots partials
// (16 KiB); a launch never uses more CTAs than that, so every row count the
// kernel accepts (1 .. 2^31-1) fits. Every call shares the array and leaves the
// last call's partials in it; nothing has to start at zero, because each launch
// writes every slot it later reads. Two calls that overlap on the GPU (other
// streams, other threads) race on the array and may return wrong results. The
// first call on a device looks up the array's device address
// (cudaGetSymbolAddress) with that device current; make that first call before
// any stream capture.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "zdmmv.h"
#include "zdmmv_device.cuh"
#include "zdmmv_internal.h"

namespace zdmmv {
namespace {

// 2048 partials x 8 bytes = 16 KiB: as many as an argmax launch ever uses
constexpr int kNoAllocSlots = kArgmaxMaxCtas;

// The scratch: one (max bits, row) partial per CTA of a launch.
static __device__ __align__(256) uint2 g_noalloc_argmax_scratch[kNoAllocSlots];

// In host code the array's name is only a host-side handle, not a device
// address; its device address is looked up once per device and kept here.
struct NoAllocDevice {
    bool ready = false;
    uint2 *scratch = nullptr;  // device address of g_noalloc_argmax_scratch
};
constexpr int kMaxDevices = 64;
NoAllocDevice g_noalloc[kMaxDevices];
std::mutex g_noalloc_mu;

cudaError_t noalloc_setup(const NoAllocDevice **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lk(g_noalloc_mu);
    NoAllocDevice &d = g_noalloc[dev];
    if (!d.ready) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_argmax_scratch);  // this device is current
        if (e != cudaSuccess) return e;
        d.scratch = static_cast<uint2 *>(p);
        d.ready = true;
    }
    *out = &d;
    return cudaSuccess;
}

int block_bytes_of(int fmt) { return fmt == kFmtQ8 ? 34 : (fmt == kFmtQ4 ? 18 : 0); }

}  // namespace
}  // namespace zdmmv

using namespace zdmmv;

extern "C" zdmmv_status zdmmv_dmmv_argmax_noalloc(zdmmv_fmt fmt, const void *w, zdmmv_layout layout, int64_t rows,
                                                  int64_t cols, const void *xq, int32_t *argmax_out, float *max_out,
                                                  zdmmv_stream_t stream) {
    const int bb = block_bytes_of(fmt);
    if (bb == 0) return ZDMMV_ERR_FORMAT;
    if (layout != ZDMMV_LAYOUT_GGUF && layout != ZDMMV_LAYOUT_REPACKED) return ZDMMV_ERR_LAYOUT;
    // rows beyond 2^31-1 cannot be reported in the int32 result
    if (rows <= 0 || rows > 0x7fffffff || !tma_shape_ok(fmt, cols)) return ZDMMV_ERR_SHAPE;
    if (!w || !xq || !argmax_out) return ZDMMV_ERR_NULL;
    const auto misaligned = [](const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) != 0; };
    if (misaligned(w, 16) || misaligned(xq, 16) || misaligned(argmax_out, 4) || (max_out && misaligned(max_out, 4)))
        return ZDMMV_ERR_ALIGN;
    const NoAllocDevice *nd = nullptr;
    if (noalloc_setup(&nd) != cudaSuccess) return ZDMMV_ERR_CUDA;
    return launch_argmax_dmmv(fmt, layout, w, rows, cols, xq, argmax_out, max_out, nd->scratch,
                              reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
               ? ZDMMV_OK
               : ZDMMV_ERR_CUDA;
}
