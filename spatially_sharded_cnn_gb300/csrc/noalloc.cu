// noalloc.cu -- depthwise backward for callers that cannot allocate device
// memory (see hc_conv2d_bwd_depthwise_noalloc in hc.h).
//
// The scratch that hc_conv2d_bwd keeps in the caller's workspace lives here in
// one statically sized device array instead.  Host code may not hand the
// array's name to a kernel (on the host it is only a stand-in for the device
// symbol), so the device's real address is looked up with
// cudaGetSymbolAddress, with that device current, and that address is what
// the kernels receive.  It is looked up again on every call made outside a
// stream capture (so an address from before a device reset is never reused);
// a call into a capturing stream uses the address of the device's last such
// lookup.
#include <mutex>

#include "common.cuh"

namespace hc {
namespace {

// 16 MiB: enough for the depthwise scratch of e.g. 8 shards x 256 channels x
// 2 column tiles x 7 images of 7x7 partials (5.7 MB) with room to spare.
constexpr size_t kNoAllocScratchBytes = 16u << 20;

__device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_setup_mu;
void* g_scratch_addr[kMaxDevices];  // per device, filled on first use

size_t round_up256(size_t b) { return (b + 255) & ~(size_t)255; }

// Device address of the scratch array on the current device: looked up now
// unless `st` is capturing, then the device's last looked-up address.
hc_status scratch_on_current_device(cudaStream_t st, void** out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return HC_ERR_CUDA;
    }
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(st, &cs) != cudaSuccess) {
        cudaGetLastError();
        return HC_ERR_CUDA;
    }
    const bool cached = dev >= 0 && dev < kMaxDevices;
    std::lock_guard<std::mutex> lock(g_setup_mu);
    if (cs != cudaStreamCaptureStatusNone) {  // no lookup inside a capture
        if (!cached || !g_scratch_addr[dev]) return HC_ERR_UNSUPPORTED;
        *out = g_scratch_addr[dev];
        return HC_OK;
    }
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) {
        cudaGetLastError();
        return HC_ERR_CUDA;
    }
    if (cached) g_scratch_addr[dev] = p;
    *out = p;
    return HC_OK;
}

bool al16(const void* q) { return ((uintptr_t)q & 15u) == 0; }

}  // namespace
}  // namespace hc

using namespace hc;

extern "C" hc_status hc_conv2d_bwd_depthwise_noalloc(const hc_conv_desc* d, const float* x, const float* w,
                                                     const float* gy, float* gx, float* gw, float* gb,
                                                     float* gw_partials, float* gb_partials, void* stream) {
    static thread_local Plan p;
    hc_status st = make_plan(d, &p);
    if (st) return st;
    if (!x || !w || !gy || !al16(x) || !al16(w) || !al16(gy)) return HC_ERR_INVALID_ARG;
    for (const void* q : {(const void*)gx, (const void*)gw, (const void*)gb, (const void*)gw_partials,
                          (const void*)gb_partials})
        if (q && !al16(q)) return HC_ERR_INVALID_ARG;
    if (!depthwise_supported(d, p)) return HC_ERR_UNSUPPORTED;

    // scratch layout: [shard gw partials][shard gb partials][tile partials]
    const size_t kk = (size_t)d->kh * d->kw;
    const size_t gwp_bytes = round_up256(sizeof(float) * p.Q * d->C_out * kk);
    const size_t gbp_bytes = round_up256(sizeof(float) * p.Q * d->C_out);
    const size_t tile_bytes = round_up256(sizeof(float) * depthwise_bwd_ws_floats(d, p));
    if (gwp_bytes + gbp_bytes + tile_bytes > kNoAllocScratchBytes) return HC_ERR_WORKSPACE;

    void* base = nullptr;
    if ((st = scratch_on_current_device((cudaStream_t)stream, &base))) return st;
    char* s = (char*)base;
    float* gwp = gw_partials ? gw_partials : (float*)s;
    float* gbp = gb_partials ? gb_partials : (float*)(s + gwp_bytes);
    float* tile_part = (float*)(s + gwp_bytes + gbp_bytes);

    cudaStream_t cs = (cudaStream_t)stream;
    traced_begin(cs);
    const bool want_wb = gw || gb || gw_partials || gb_partials;
    return launch_depthwise_bwd(d, p, x, w, gy, gx, tile_part, gwp, gbp, want_wb, cs, nullptr, gw, gb);
}
