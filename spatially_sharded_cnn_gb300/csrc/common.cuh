// common.cuh -- internal declarations shared by the library's translation units.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

#include "hc.h"

namespace hc {

constexpr int kMaxShards = 1024;     // host-side plan
constexpr int kMaxKernelShards = 64; // shards a kernel takes per-shard tables for

// Host-side shard plan (see hc_shard_plan / hc_shard_plan_rows): uniform
// block width Wl (and height Hl); the per-shard halo widths and owned output
// columns (rows).  Shard q = a * S + b of the Sh x S grid holds row block a and
// column block b; Q = Sh * S partials.
struct Plan {
    int S = 0, Wl = 0, Ho = 0, Wo = 0;
    int We = 0;  // widest extended tile: max_r(halo_left + Wl + halo_right)
    int Sh = 1, Hl = 0, Hlo = 0;  // row shards, rows per row block, owned output rows per row block
    int He = 0;                   // tallest extended tile (H with one row shard)
    int Q = 0;                    // Sh * S
    hc_shard_extent ext[kMaxShards];
    hc_shard_extent ext_h[kMaxShards];
};

hc_status make_plan(const hc_conv_desc* d, Plan* p);

// Count of kernel launches issued by the library.
extern std::atomic<unsigned long long> g_launches;

// Per-kernel timing (trace.cu): trace_begin(st) at the start of a launcher,
// trace_launch(name, st) after each of its launches.  Both return at once
// while tracing is off.
extern std::atomic<int> g_trace_on;
void trace_begin(cudaStream_t st);
void trace_launch(const char* name, cudaStream_t st);
inline void traced_begin(cudaStream_t st) {
    if (g_trace_on.load(std::memory_order_relaxed)) trace_begin(st);
}

// After a launch: counts it, records its trace event, and returns HC_ERR_CUDA
// if the launch failed.
inline hc_status launched(const char* name, cudaStream_t st) {
    g_launches.fetch_add(1, std::memory_order_relaxed);
    const hc_status s = cudaPeekAtLastError() == cudaSuccess ? HC_OK : (cudaGetLastError(), HC_ERR_CUDA);
    if (s == HC_OK && g_trace_on.load(std::memory_order_relaxed)) trace_launch(name, st);
    return s;
}

inline unsigned cdiv(long long a, long long b) { return (unsigned)((a + b - 1) / b); }

// Streaming multiprocessors of the current device (looked up once per device),
// or the count hc_set_sm_count imposes.
int device_sm_count();
extern std::atomic<int> g_sm_override;

// Per-device caches (kernel attributes, SM counts, wave sizes, the no-alloc
// scratch address) hold kMaxDevices entries; a device ordinal at or beyond it
// is served without caching (the value is looked up on every call).
constexpr int kMaxDevices = 64;

// Runs `set` (e.g. cudaFuncSetAttribute calls) once for each device the
// library launches on: kernel attributes belong to a device, so a process that
// runs the library on several GPUs needs them set on each.  `set` returns true
// when every call it made succeeded; only then is the device's bit in `done`
// set, so a failed attempt (for example inside a strict stream capture) is
// retried on the next call, and its error is cleared.
template <typename F>
inline void once_per_device(std::atomic<unsigned long long>& done, F&& set) {
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= kMaxDevices) {
        if (!set()) cudaGetLastError();
        return;
    }
    const unsigned long long bit = 1ull << dev;
    if (done.load(std::memory_order_acquire) & bit) return;
    if (set())
        done.fetch_or(bit, std::memory_order_release);
    else
        cudaGetLastError();
}

// TMA descriptor for a tensor of `rank` dims (dims[0] innermost), strides in
// bytes for dims 1..rank-1, zero fill out of bounds.
hc_status make_tmap(CUtensorMap* map, CUtensorMapDataType dtype, int rank, const void* base, const uint64_t* dims,
                    const uint64_t* strides_bytes, const uint32_t* box, CUtensorMapSwizzle swizzle);

// Device status words of the kernels that wait on barriers: returns (and
// clears) the first error recorded since the last call.  Call after the
// stream has been synchronised.
hc_status dw_take_status();
hc_status tc_take_status();
hc_status launch_selftest_timeout(int wait_us, cudaStream_t st);

// GELU, exact form: x * Phi(x), Phi(x) = (1 + erf(x / sqrt 2)) / 2.
__device__ __forceinline__ float gelu_f(float v) { return 0.5f * v * (1.0f + erff(v * 0.70710678118654752f)); }
// d/dx GELU = Phi(x) + x * exp(-x^2 / 2) / sqrt(2 pi)
__device__ __forceinline__ float gelu_d(float v) {
    return 0.5f * (1.0f + erff(v * 0.70710678118654752f)) + v * 0.39894228040143268f * expf(-0.5f * v * v);
}

// fp32 -> three bf16 pieces, the operand format of HC_ALGO_TC_BF16X6:
// p0 = bf16(v), p1 = bf16(v - p0), p2 = bf16(v - p0 - p1); the two differences
// are exact in fp32, and the pieces carry 24 bits of v's significand.
__device__ __forceinline__ void split3(float v, __nv_bfloat16& p0, __nv_bfloat16& p1, __nv_bfloat16& p2) {
    p0 = __float2bfloat16_rn(v);
    const float r = v - __bfloat162float(p0);
    p1 = __float2bfloat16_rn(r);
    p2 = __float2bfloat16_rn(r - __bfloat162float(p1));
}
__device__ __forceinline__ uint32_t pack2(__nv_bfloat16 a, __nv_bfloat16 b) {
    return (uint32_t)__bfloat16_as_ushort(a) | ((uint32_t)__bfloat16_as_ushort(b) << 16);
}
// The pieces of four consecutive values (float4 number i): out[k * ps4 + i] holds
// piece k of all four.
__device__ __forceinline__ void store_pieces4(float4 v, uint2* out, long long i, long long ps4) {
    __nv_bfloat16 a[4], b[4], c[4];
    split3(v.x, a[0], b[0], c[0]);
    split3(v.y, a[1], b[1], c[1]);
    split3(v.z, a[2], b[2], c[2]);
    split3(v.w, a[3], b[3], c[3]);
    out[i] = make_uint2(pack2(a[0], a[1]), pack2(a[2], a[3]));
    out[ps4 + i] = make_uint2(pack2(b[0], b[1]), pack2(b[2], b[3]));
    out[2 * ps4 + i] = make_uint2(pack2(c[0], c[1]), pack2(c[2], c[3]));
}

// ---- kernel launchers (one translation unit each) -------------------------
hc_status launch_halo_gather(const hc_conv_desc* d, const Plan& p, const float* x, float* x_ext, cudaStream_t st);

// direct (any groups, stride, padding)
hc_status launch_direct_fwd(const hc_conv_desc* d, const Plan& p, const float* x, const float* w, const float* b,
                            float* y, cudaStream_t st);
hc_status launch_direct_gx(const hc_conv_desc* d, const Plan& p, const float* w, const float* gy, float* gx,
                           cudaStream_t st);
// per-shard partials gw_part [S][C_out][C_in/g][kh][kw], gb_part [S][C_out] (either may be null), and
// with gw / gb (nullable) the full gradients, the partials summed in shard order
hc_status launch_direct_partials(const hc_conv_desc* d, const Plan& p, const float* x, const float* gy,
                                 float* gw_part, float* gb_part, cudaStream_t st, float* gw = nullptr,
                                 float* gb = nullptr);

// depthwise K x K, stride 1, padding (K-1)/2, 128-column tiles inside a shard
bool depthwise_supported(const hc_conv_desc* d, const Plan& p);
size_t depthwise_bwd_ws_floats(const hc_conv_desc* d, const Plan& p);
// Where a depthwise launch reads x (and grad_output) and which column tiles it
// covers.  pitch: floats per row of those tensors (0: W), xo: the column of a
// row where the block's column 0 sits (the halo-padded layout of one rank:
// pitch W + 2 * kHaloCols, xo = kHaloCols).  tiles: HC_TILES_ALL, _INTERIOR
// (column tiles 1 .. T-2, which read no margin column) or _EDGE (0 and T-1).
// partials (backward): reduce the tile partials to shard partials after the
// launch (the last launch of a split backward).
constexpr int kHaloCols = 4;
struct DwLayout {
    int pitch = 0, xo = 0, tiles = HC_TILES_ALL;
    bool partials = true;
};
hc_status launch_depthwise_fwd(const hc_conv_desc* d, const Plan& p, const float* x, const float* w,
                               const float* b, float* y, cudaStream_t st, const DwLayout& lay = DwLayout());
// tile partials go to ws; then reduced to shard partials gwp / gbp ([S][C][K*K], [S][C])
// gres (nullable, only with gx): added to grad_input in its epilogue (a residual gradient);
// gw / gb (nullable): the full gradients, the shard partials summed in shard order
hc_status launch_depthwise_bwd(const hc_conv_desc* d, const Plan& p, const float* x, const float* w,
                               const float* gy, float* gx, float* tile_part, float* gwp, float* gbp,
                               bool want_weight_grads, cudaStream_t st, const float* gres = nullptr,
                               float* gw = nullptr, float* gb = nullptr, const DwLayout& lay = DwLayout());
// the halo-padded layout of one rank (hc_halo_pad / _pack / _unpack)
// Shard partials of a per-(grid shard, channel) slot table
// tile_part[Q][C][rows][KK + 1] (KK weight terms + the bias): gwp[q][c][k] /
// gbp[q][c] = the slots summed in order, gw / gb (nullable) = those summed over
// q in order.
hc_status launch_shard_partials(const float* tile_part, float* gwp, float* gbp, float* gw, float* gb, int Q, int C,
                                int rows, int KK, cudaStream_t st);

// patchify.cu: weight / bias gradient of a 4x4 stride-4 conv with 3 input
// channels (the ConvNeXt stem) as a direct FP32 reduction, per grid shard.
bool patchify_wgrad_supported(const hc_conv_desc* d, const Plan& p);
size_t patchify_wgrad_ws_floats(const hc_conv_desc* d, const Plan& p);
hc_status launch_patchify_wgrad(const hc_conv_desc* d, const Plan& p, const float* x, const float* gy,
                                float* tile_part, float* gwp, float* gbp, float* gw, float* gb, cudaStream_t st);
hc_status pw_take_status();

hc_status launch_halo_pad(const hc_conv_desc* d, int Wl, const float* x, float* xp, cudaStream_t st);
hc_status launch_halo_pack(const hc_conv_desc* d, int Wl, const float* xp, int side, float* buf, cudaStream_t st);
hc_status launch_halo_unpack(const hc_conv_desc* d, int Wl, const float* buf, int side, float* xp, cudaStream_t st);

// dense conv on tcgen05 (3xTF32 implicit GEMM): groups 1, stride 1, odd k,
// padding (k-1)/2, C_in and C_out multiples of 128
bool tc_supported(const hc_conv_desc* d, const Plan& p);
int tc_wgrad_splits(const hc_conv_desc* d, const Plan& p);
size_t tc_ws_bytes(const hc_conv_desc* d, const Plan& p, int pass);
hc_status launch_tc_fwd(const hc_conv_desc* d, const Plan& p, const float* x, const float* w, const float* b,
                        float* y, void* ws, cudaStream_t st);
// grad_input (if gx) and the per-shard weight-gradient partials gwp (if want_w)
// gbp (nullable, with want_w): the bias-gradient partials, summed in the read of
// grad_output that splits it into the weight gradient's pieces (btmp: scratch).
hc_status launch_tc_bwd(const hc_conv_desc* d, const Plan& p, const float* x, const float* w, const float* gy,
                        float* gx, float* gwp, bool want_w, void* ws, cudaStream_t st, float* gbp = nullptr,
                        float* btmp = nullptr);

// 1x1 conv (stride 1, padding 0, groups 1) on tcgen05 with three bf16 pieces per
// operand (six products, fp32 accuracy); C_in and C_out multiples of 128
// (and k = stride convs as 1x1 convs of the space-to-depth image)
bool bf16_supported(const hc_conv_desc* d, const Plan& p);
// pass 2: the backward pass that takes x's pieces from the forward workspace
size_t bf16_ws_bytes(const hc_conv_desc* d, const Plan& p, int pass);
// gelu_in: the conv's input is GELU(x) (1x1 only): both passes split GELU(x), and
// grad_input is the gradient with respect to GELU(x)
hc_status launch_bf16_fwd(const hc_conv_desc* d, const Plan& p, const float* x, const float* w, const float* b,
                          float* y, void* ws, cudaStream_t st, bool gelu_in = false);
// fwd_ws: the workspace of the forward pass on this desc and x, or NULL to split x here
// gbp (optional): also the bias-gradient partials, with tmp[bias_grad_ws_floats]
// gelu_y (1x1 only): the conv's output y feeds a GELU and gy is the gradient of
// GELU(y): the pass runs on gy * GELU'(gelu_y)
hc_status launch_bf16_bwd(const hc_conv_desc* d, const Plan& p, const float* x, const float* w, const float* gy,
                          float* gx, float* gwp, bool want_w, void* ws, const void* fwd_ws, float* gbp,
                          float* btmp, cudaStream_t st, bool gelu_in = false, const float* gelu_y = nullptr);

// Per-shard bias-gradient partials gbp[S][Co] in two fixed-order stages,
// using tmp[bias_grad_ws_floats(Co, S)].
constexpr int kBiasSlices = 64;
size_t bias_grad_ws_floats(int Co, int S);
// gbp [Sh*S][Co]: row shard a owns output rows [a*own_h, (a+1)*own_h) (the last
// up to Ho), column shard b columns [b*own_w, (b+1)*own_w) (the last up to Wo)
// pieces (optional): also writes the bf16 pieces of gy there (piece k of element
// e at pieces[k * ps + e], ps a multiple of 4) while reading it -- the same sums.
// gelu_y (with pieces): the gradient summed and split is gy * GELU'(gelu_y).
hc_status launch_bias_grad_partials(const float* gy, float* gbp, int N, int Co, int Ho, int Wo, int S, int own_w,
                                    int Sh, int own_h, float* tmp, cudaStream_t st, void* pieces = nullptr,
                                    long long ps = 0, const float* gelu_y = nullptr);

// out[k] = sum over rows r (ascending, in groups of kColumnGroup) of in[r * stride + k];
// tmp holds column_sum_tmp_floats(rows, count) floats.
constexpr int kColumnGroup = 64;
size_t column_sum_tmp_floats(int rows, int count);
hc_status launch_column_sum(const float* in, float* out, int rows, int count, long long stride, float* tmp,
                            cudaStream_t st);

// fixed-order sums
// out[k] = sum_{r < rows} in[r * count + k], r ascending
hc_status launch_sum_rows(const float* in, float* out, int rows, long long count, cudaStream_t st);

}  // namespace hc
