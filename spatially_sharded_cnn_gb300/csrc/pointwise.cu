// pointwise.cu -- the shard-local ops of a ConvNeXt block (the pages' model,
// NVIDIA blog "Perception model training for autonomous vehicles with tensor
// parallelism": ConvNeXt-XL blocks): channels-first LayerNorm over C,
// exact-erf GELU, and layer scale + residual, forward and backward.  None of
// them reads across W, so they need no halo; their parameter gradients are
// per-block partial sums added in block order (deterministic).
//
// Tensors are [N][C][HW] fp32 (NCHW with the spatial dims flattened).
#include "common.cuh"

namespace hc {
namespace {

constexpr int LN_PIX = 32;       // pixels per LayerNorm block
constexpr int LN_PITCH = 33;     // shared-tile row pitch: rows (channels) and columns (pixels) both
                                 // hit 32 distinct banks
constexpr int LN_THREADS = 512;  // 16 channel groups x 32 pixels
constexpr int LN_G = LN_THREADS / 32;

// LayerNorm over C at every (n, pixel): mean, biased variance (two passes over
// the staged tile), y = (x - mean) * rstd * gamma[c] + beta[c].
__global__ void __launch_bounds__(LN_THREADS) ln_fwd_kernel(const float* __restrict__ x, const float* __restrict__ gamma,
                                                            const float* __restrict__ beta, float eps,
                                                            float* __restrict__ y, float* __restrict__ mean,
                                                            float* __restrict__ rstd, int C, long long HW,
                                                            long long blocks_per_image) {
    extern __shared__ float tile[];  // [C][LN_PITCH]
    __shared__ float red[LN_G][LN_PIX];
    __shared__ float stat[2][LN_PIX];
    const long long b = blockIdx.x;
    const int n = (int)(b / blocks_per_image);
    const long long p0 = (b % blocks_per_image) * LN_PIX;
    const int px = threadIdx.x % LN_PIX, g = threadIdx.x / LN_PIX;  // LN_G groups of channels
    const long long p = p0 + px;
    const bool valid = p < HW;
    const float* xb = x + (long long)n * C * HW;
    for (int c = g; c < C; c += LN_G) tile[c * LN_PITCH + px] = valid ? __ldg(xb + (long long)c * HW + p) : 0.0f;
    // mean
    float s = 0.0f;
    for (int c = g; c < C; c += LN_G) s += tile[c * LN_PITCH + px];
    red[g][px] = s;
    __syncthreads();
    if (g == 0) {
        float t = 0.0f;
        for (int k = 0; k < LN_G; k++) t += red[k][px];
        stat[0][px] = t / C;
    }
    __syncthreads();
    const float mu = stat[0][px];
    float v = 0.0f;
    for (int c = g; c < C; c += LN_G) {
        const float d = tile[c * LN_PITCH + px] - mu;
        v = fmaf(d, d, v);
    }
    red[g][px] = v;
    __syncthreads();
    if (g == 0) {
        float t = 0.0f;
        for (int k = 0; k < LN_G; k++) t += red[k][px];
        stat[1][px] = rsqrtf(t / C + eps);
    }
    __syncthreads();
    const float rs = stat[1][px];
    if (valid) {
        float* yb = y + (long long)n * C * HW;
        for (int c = g; c < C; c += LN_G)
            yb[(long long)c * HW + p] = (tile[c * LN_PITCH + px] - mu) * rs * __ldg(gamma + c) + __ldg(beta + c);
        if (g == 0) {
            if (mean) mean[(long long)n * HW + p] = mu;
            if (rstd) rstd[(long long)n * HW + p] = rs;
        }
    }
}

// LayerNorm backward: with xhat = (x - mean) * rstd and g = gy * gamma,
// gx = rstd * (g - mean_c(g) - xhat * mean_c(g * xhat)); the block's partial
// ggamma / gbeta (sums over its pixels of gy * xhat and gy) go to part[b][2][C].
__global__ void __launch_bounds__(LN_THREADS) ln_bwd_kernel(const float* __restrict__ x, const float* __restrict__ gamma,
                                                            const float* __restrict__ mean,
                                                            const float* __restrict__ rstd,
                                                            const float* __restrict__ gy, float* __restrict__ gx,
                                                            float* __restrict__ part, int C, long long HW,
                                                            long long blocks_per_image) {
    extern __shared__ float sm[];  // xhat [C][LN_PITCH], gy [C][LN_PITCH]
    float* th = sm;
    float* tg = sm + C * LN_PITCH;
    __shared__ float red[2][LN_G][LN_PIX];
    __shared__ float stat[2][LN_PIX];
    const long long b = blockIdx.x;
    const int n = (int)(b / blocks_per_image);
    const long long p0 = (b % blocks_per_image) * LN_PIX;
    const int px = threadIdx.x % LN_PIX, g = threadIdx.x / LN_PIX;
    const long long p = p0 + px;
    const bool valid = p < HW;
    const float mu = valid ? __ldg(mean + (long long)n * HW + p) : 0.0f;
    const float rs = valid ? __ldg(rstd + (long long)n * HW + p) : 0.0f;
    const float* xb = x + (long long)n * C * HW;
    const float* gb = gy + (long long)n * C * HW;
    float s1 = 0.0f, s2 = 0.0f;
    for (int c = g; c < C; c += LN_G) {
        const float xh = valid ? (__ldg(xb + (long long)c * HW + p) - mu) * rs : 0.0f;
        const float gv = valid ? __ldg(gb + (long long)c * HW + p) : 0.0f;
        th[c * LN_PITCH + px] = xh;
        tg[c * LN_PITCH + px] = gv;
        const float gg = gv * __ldg(gamma + c);
        s1 += gg;
        s2 = fmaf(gg, xh, s2);
    }
    red[0][g][px] = s1;
    red[1][g][px] = s2;
    __syncthreads();
    if (g == 0) {
        float a = 0.0f, c2 = 0.0f;
        for (int k = 0; k < LN_G; k++) {
            a += red[0][k][px];
            c2 += red[1][k][px];
        }
        stat[0][px] = a / C;
        stat[1][px] = c2 / C;
    }
    __syncthreads();
    const float mg = stat[0][px], mgx = stat[1][px];
    if (valid) {
        float* gxb = gx + (long long)n * C * HW;
        for (int c = g; c < C; c += LN_G) {
            const float xh = th[c * LN_PITCH + px];
            const float gg = tg[c * LN_PITCH + px] * __ldg(gamma + c);
            gxb[(long long)c * HW + p] = rs * (gg - mg - xh * mgx);
        }
    }
    // per-channel partials over this block's pixels (pixel order 0..31)
    if (part) {
        float* pb = part + b * 2 * C;
        for (int c = threadIdx.x; c < C; c += LN_THREADS) {
            float a = 0.0f, bb = 0.0f;
            for (int k = 0; k < LN_PIX; k++) {
                a = fmaf(tg[c * LN_PITCH + k], th[c * LN_PITCH + k], a);
                bb += tg[c * LN_PITCH + k];
            }
            pb[c] = a;
            pb[C + c] = bb;
        }
    }
}

// The same two passes with C = VPT * LN_G known at compile time: every thread
// holds its VPT channels of one pixel in registers (VPT independent loads in
// flight, no shared-memory tile); sums run in the same channel order as
// ln_fwd_kernel's.  (C = 256: 0.44 -> 0.31 ms on a 940 MB tensor.)
template <int VPT>
__global__ void __launch_bounds__(LN_THREADS) ln_fwd_reg_kernel(const float* __restrict__ x,
                                                                const float* __restrict__ gamma,
                                                                const float* __restrict__ beta, float eps,
                                                                float* __restrict__ y, float* __restrict__ mean,
                                                                float* __restrict__ rstd, long long HW,
                                                                long long blocks_per_image) {
    constexpr int C = VPT * LN_G;
    __shared__ float red[LN_G][LN_PIX];
    __shared__ float stat[2][LN_PIX];
    const long long b = blockIdx.x;
    const int n = (int)(b / blocks_per_image);
    const int px = threadIdx.x % LN_PIX, g = threadIdx.x / LN_PIX;
    const long long p = (b % blocks_per_image) * LN_PIX + px;
    const bool valid = p < HW;
    const float* xb = x + (long long)n * C * HW + p;
    float v[VPT];
#pragma unroll
    for (int k = 0; k < VPT; k++) v[k] = valid ? __ldg(xb + (long long)(g + k * LN_G) * HW) : 0.0f;
    float s = 0.0f;
#pragma unroll
    for (int k = 0; k < VPT; k++) s += v[k];
    red[g][px] = s;
    __syncthreads();
    if (g == 0) {
        float t = 0.0f;
        for (int k = 0; k < LN_G; k++) t += red[k][px];
        stat[0][px] = t / C;
    }
    __syncthreads();
    const float mu = stat[0][px];
    float var = 0.0f;
#pragma unroll
    for (int k = 0; k < VPT; k++) {
        const float d = v[k] - mu;
        var = fmaf(d, d, var);
    }
    red[g][px] = var;
    __syncthreads();
    if (g == 0) {
        float t = 0.0f;
        for (int k = 0; k < LN_G; k++) t += red[k][px];
        stat[1][px] = rsqrtf(t / C + eps);
    }
    __syncthreads();
    const float rs = stat[1][px];
    if (valid) {
        float* yb = y + (long long)n * C * HW + p;
#pragma unroll
        for (int k = 0; k < VPT; k++) {
            const int c = g + k * LN_G;
            yb[(long long)c * HW] = (v[k] - mu) * rs * __ldg(gamma + c) + __ldg(beta + c);
        }
        if (g == 0) {
            if (mean) mean[(long long)n * HW + p] = mu;
            if (rstd) rstd[(long long)n * HW + p] = rs;
        }
    }
}

// The backward with C = VPT * LN_G known at compile time, persistent: block b
// takes the 32-pixel groups b, b + gridDim.x, ... in that order (two blocks per
// SM).  Each thread holds its VPT channels of one pixel (x and grad_output: all
// 2 * VPT loads in flight, no shared-memory tile).  The ggamma / gbeta sums of a
// group reduce each channel over the warp's 32 pixels with a fixed shuffle tree
// -- four halving steps (lane bits 4..1) leave lane L one channel,
// (L >> 1) & 15, summed over 16 lanes, and the last step adds lane L ^ 1 --
// and accumulate across the block's groups in one register; the block writes
// one partial row at the end (even lanes the gy * xhat sums, odd lanes the gy
// sums).
template <int VPT>
__global__ void __launch_bounds__(LN_THREADS, 2) ln_bwd_reg_kernel(const float* __restrict__ x,
                                                                   const float* __restrict__ gamma,
                                                                   const float* __restrict__ mean,
                                                                   const float* __restrict__ rstd,
                                                                   const float* __restrict__ gy, float* __restrict__ gx,
                                                                   float* __restrict__ part, int HW,
                                                                   int blocks_per_image, int groups) {
    static_assert(VPT == 16, "the shuffle tree takes 16 channels per thread");
    constexpr int C = VPT * LN_G;
    __shared__ float red[2][LN_G][LN_PIX];
    __shared__ float stat[2][LN_PIX];
    const int px = threadIdx.x % LN_PIX, g = threadIdx.x / LN_PIX;
    const int lane = px;  // a warp is one channel group's 32 pixels
    float acc = 0.0f;     // this lane's channel sum over the block's groups
    for (int grp = blockIdx.x; grp < groups; grp += gridDim.x) {
        const int n = grp / blocks_per_image;
        const int p = (grp - n * blocks_per_image) * LN_PIX + px;
        const bool valid = p < HW;
        const size_t img = (size_t)n * C * HW;  // C * HW < 2^31: offsets inside an image are 32-bit
        const int off = g * HW + p;
        float xh[VPT], gv[VPT];
#pragma unroll
        for (int k = 0; k < VPT; k++) {
            xh[k] = valid ? __ldg(x + img + off + k * LN_G * HW) : 0.0f;
            gv[k] = valid ? __ldg(gy + img + off + k * LN_G * HW) : 0.0f;
        }
        const float mu = valid ? __ldg(mean + (size_t)n * HW + p) : 0.0f;
        const float rs = valid ? __ldg(rstd + (size_t)n * HW + p) : 0.0f;
        float s1 = 0.0f, s2 = 0.0f;
#pragma unroll
        for (int k = 0; k < VPT; k++) {
            xh[k] = valid ? (xh[k] - mu) * rs : 0.0f;
            const float gg = gv[k] * __ldg(gamma + g + k * LN_G);
            s1 += gg;
            s2 = fmaf(gg, xh[k], s2);
        }
        red[0][g][px] = s1;
        red[1][g][px] = s2;
        __syncthreads();
        if (g == 0) {
            float a = 0.0f, c2 = 0.0f;
            for (int k = 0; k < LN_G; k++) {
                a += red[0][k][px];
                c2 += red[1][k][px];
            }
            stat[0][px] = a / C;
            stat[1][px] = c2 / C;
        }
        __syncthreads();  // (the next group writes red only after every thread has read stat)
        const float mg = stat[0][px], mgx = stat[1][px];
        if (valid) {
#pragma unroll
            for (int k = 0; k < VPT; k++) {
                const float gg = gv[k] * __ldg(gamma + g + k * LN_G);
                gx[img + off + k * LN_G * HW] = rs * (gg - mg - xh[k] * mgx);
            }
        }
        if (part) {
#pragma unroll
            for (int k = 0; k < VPT; k++) xh[k] *= gv[k];  // gy * xhat (zero for pixels past HW)
#pragma unroll
            for (int lvl = 0; lvl < 4; lvl++) {
                const int sh = 16 >> lvl, half = 8 >> lvl;
                const bool up = (lane & sh) != 0;
#pragma unroll
                for (int j = 0; j < half; j++) {
                    const float sa = up ? xh[j] : xh[j + half], ka = up ? xh[j + half] : xh[j];
                    const float sb = up ? gv[j] : gv[j + half], kb = up ? gv[j + half] : gv[j];
                    xh[j] = ka + __shfl_xor_sync(0xffffffffu, sa, sh);
                    gv[j] = kb + __shfl_xor_sync(0xffffffffu, sb, sh);
                }
            }
            const float ta = xh[0] + __shfl_xor_sync(0xffffffffu, xh[0], 1);
            const float tb = gv[0] + __shfl_xor_sync(0xffffffffu, gv[0], 1);
            acc += (lane & 1) ? tb : ta;
        }
    }
    if (part) part[blockIdx.x * 2 * C + (lane & 1) * C + g + ((lane >> 1) & 15) * LN_G] = acc;
}

// GELU and its derivative: gelu_f / gelu_d (common.cuh).
__global__ void gelu_fwd_kernel(const float* __restrict__ x, float* __restrict__ y, long long n) {
    const long long n4 = n / 4;
    for (long long q = blockIdx.x * (long long)blockDim.x + threadIdx.x; q < n4; q += (long long)gridDim.x * blockDim.x) {
        const float4 v = __ldg(reinterpret_cast<const float4*>(x) + q);
        reinterpret_cast<float4*>(y)[q] = make_float4(gelu_f(v.x), gelu_f(v.y), gelu_f(v.z), gelu_f(v.w));
    }
    for (long long q = n4 * 4 + blockIdx.x * (long long)blockDim.x + threadIdx.x; q < n;
         q += (long long)gridDim.x * blockDim.x)
        y[q] = gelu_f(__ldg(x + q));
}

__global__ void gelu_bwd_kernel(const float* __restrict__ x, const float* __restrict__ gy, float* __restrict__ gx,
                                long long n) {
    const long long n4 = n / 4;
    for (long long q = blockIdx.x * (long long)blockDim.x + threadIdx.x; q < n4; q += (long long)gridDim.x * blockDim.x) {
        const float4 v = __ldg(reinterpret_cast<const float4*>(x) + q);
        const float4 g = __ldg(reinterpret_cast<const float4*>(gy) + q);
        reinterpret_cast<float4*>(gx)[q] =
            make_float4(g.x * gelu_d(v.x), g.y * gelu_d(v.y), g.z * gelu_d(v.z), g.w * gelu_d(v.w));
    }
    for (long long q = n4 * 4 + blockIdx.x * (long long)blockDim.x + threadIdx.x; q < n;
         q += (long long)gridDim.x * blockDim.x)
        gx[q] = __ldg(gy + q) * gelu_d(__ldg(x + q));
}

// out = res + gamma[c] * branch; one block per (n, c) plane chunk.
// DropPath keep mask with a draw that depends only on (seed, offset, n): the
// value for sample n is output number offset + n of a SplitMix64 generator
// seeded with `seed` (Steele, Lea and Flood, "Fast splittable pseudorandom
// number generators", 2014; finaliser constants of Vigna's public splitmix64),
// so every shard, or device, holding sample n draws the same bits.  Keep iff
// the output's top 24 bits are >= t = floor(p * 2^24); a kept sample's branch
// is scaled by 1 / (1 - p).
__device__ __forceinline__ unsigned long long splitmix64_at(unsigned long long seed, unsigned long long i) {
    unsigned long long z = seed + (i + 1ULL) * 0x9E3779B97F4A7C15ULL;
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
    return z ^ (z >> 31);
}
__global__ void drop_path_mask_kernel(int N, unsigned t, float scale, unsigned long long seed,
                                      unsigned long long offset, float* __restrict__ mask) {
    for (int n = blockIdx.x * blockDim.x + threadIdx.x; n < N; n += gridDim.x * blockDim.x) {
        const unsigned u = (unsigned)(splitmix64_at(seed, offset + (unsigned long long)n) >> 40);
        mask[n] = u >= t ? scale : 0.0f;
    }
}

// Layer scale (+ DropPath) + residual: out = res + mask[n] * gamma[c] * branch,
// mask NULL meaning 1.  Block = (plane n*C + c, chunk of its pixels).
__global__ void ls_fwd_kernel(const float* __restrict__ res, const float* __restrict__ br,
                              const float* __restrict__ gamma, const float* __restrict__ mask,
                              float* __restrict__ out, int C, long long HW, int chunks) {
    const long long plane = blockIdx.x / chunks;
    const int chunk = blockIdx.x % chunks;
    const float gm = __ldg(gamma + plane % C) * (mask ? __ldg(mask + plane / C) : 1.0f);
    const long long b0 = HW * chunk / chunks, b1 = HW * (chunk + 1) / chunks;
    const long long off = plane * HW;
    for (long long q = b0 + threadIdx.x; q < b1; q += blockDim.x) out[off + q] = fmaf(gm, __ldg(br + off + q), __ldg(res + off + q));
}

// gbranch = gamma[c] * gy; partial ggamma of this chunk = sum branch * gy (fixed order).
// Backward: gbranch = mask[n] * gamma[c] * gy; part[plane][chunk] = mask[n] *
// (sum over the chunk of branch * gy), summed over (n, chunk) by ls_reduce_kernel.
__global__ void ls_bwd_kernel(const float* __restrict__ br, const float* __restrict__ gamma,
                              const float* __restrict__ mask, const float* __restrict__ gy, float* __restrict__ gbr,
                              float* __restrict__ part, int C, long long HW, int chunks) {
    __shared__ float red[32];
    const long long plane = blockIdx.x / chunks;
    const int chunk = blockIdx.x % chunks;
    const float m = mask ? __ldg(mask + plane / C) : 1.0f;
    const float gm = __ldg(gamma + plane % C) * m;
    const long long b0 = HW * chunk / chunks, b1 = HW * (chunk + 1) / chunks;
    const long long off = plane * HW;
    float acc = 0.0f;
    for (long long q = b0 + threadIdx.x; q < b1; q += blockDim.x) {
        const float g = __ldg(gy + off + q);
        if (gbr) gbr[off + q] = gm * g;
        acc = fmaf(__ldg(br + off + q), g, acc);
    }
    for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = acc;
    __syncthreads();
    if (threadIdx.x == 0) {
        float t = 0.0f;
        for (int k = 0; k < (int)(blockDim.x >> 5); k++) t += red[k];
        part[blockIdx.x] = m * t;  // [plane][chunk]
    }
}

// ggamma[c] = sum over (n, chunk) of part[(n * C + c) * chunks + chunk], n then chunk ascending.
__global__ void ls_reduce_kernel(const float* __restrict__ part, float* __restrict__ gg, int N, int C, int chunks) {
    const int c = blockIdx.x * blockDim.x + threadIdx.x;
    if (c >= C) return;
    float t = 0.0f;
    for (int n = 0; n < N; n++)
        for (int k = 0; k < chunks; k++) t += part[((long long)n * C + c) * chunks + k];
    gg[c] = t;
}

// y += x
__global__ void add_inplace_kernel(float* __restrict__ y, const float* __restrict__ x, long long n) {
    const long long n4 = n / 4;
    for (long long q = blockIdx.x * (long long)blockDim.x + threadIdx.x; q < n4; q += (long long)gridDim.x * blockDim.x) {
        float4 a = reinterpret_cast<float4*>(y)[q];
        const float4 b = __ldg(reinterpret_cast<const float4*>(x) + q);
        a.x += b.x;
        a.y += b.y;
        a.z += b.z;
        a.w += b.w;
        reinterpret_cast<float4*>(y)[q] = a;
    }
    for (long long q = n4 * 4 + blockIdx.x * (long long)blockDim.x + threadIdx.x; q < n;
         q += (long long)gridDim.x * blockDim.x)
        y[q] += __ldg(x + q);
}

constexpr int LS_CHUNKS = 16;

bool al16(const void* q) { return ((uintptr_t)q & 15u) == 0; }

unsigned grid_elems(long long n) {
    const long long b = (n / 4 + 255) / 256;
    return (unsigned)(b < 1 ? 1 : (b > 152LL * 32 ? 152LL * 32 : b));
}


}  // namespace
}  // namespace hc

using namespace hc;

extern "C" {

hc_status hc_pointwise_workspace_size(int N, int C, long long HW, size_t* bytes) {
    if (N <= 0 || C <= 0 || HW <= 0 || !bytes) return HC_ERR_INVALID_ARG;
    const long long ln_blocks = (long long)N * ((HW + LN_PIX - 1) / LN_PIX);
    if (ln_blocks > 0x7fffffffLL) return HC_ERR_UNSUPPORTED;
    const size_t ln = sizeof(float) * ((size_t)ln_blocks * 2 * C + column_sum_tmp_floats((int)ln_blocks, C) + 64);
    const size_t ls = sizeof(float) * (size_t)N * C * LS_CHUNKS;
    *bytes = ln > ls ? ln : ls;
    return HC_OK;
}

hc_status hc_layernorm_c_fwd(int N, int C, long long HW, const float* x, const float* gamma, const float* beta,
                             float eps, float* y, float* mean, float* rstd, void* stream) {
    traced_begin((cudaStream_t)stream);
    if (N <= 0 || C <= 0 || HW <= 0 || !x || !gamma || !beta || !y || !(eps >= 0.0f)) return HC_ERR_INVALID_ARG;
    const size_t smem = sizeof(float) * (size_t)C * LN_PITCH;
    if (smem > 200 * 1024) return HC_ERR_UNSUPPORTED;
    static std::atomic<unsigned long long> attr{0};
    once_per_device(attr, [&] {
        return cudaFuncSetAttribute(ln_fwd_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024) == cudaSuccess;
    });
    const long long bpi = (HW + LN_PIX - 1) / LN_PIX;
    if (C == 16 * LN_G)
        ln_fwd_reg_kernel<16><<<(unsigned)(N * bpi), LN_THREADS, 0, (cudaStream_t)stream>>>(x, gamma, beta, eps, y,
                                                                                          mean, rstd, HW, bpi);
    else
        ln_fwd_kernel<<<(unsigned)(N * bpi), LN_THREADS, smem, (cudaStream_t)stream>>>(x, gamma, beta, eps, y, mean,
                                                                                     rstd, C, HW, bpi);
    return launched("ln_fwd_kernel", (cudaStream_t)stream);
}

hc_status hc_layernorm_c_bwd(int N, int C, long long HW, const float* x, const float* gamma, const float* mean,
                             const float* rstd, const float* gy, float* gx, float* ggamma, float* gbeta, void* ws,
                             size_t ws_bytes, void* stream) {
    traced_begin((cudaStream_t)stream);
    if (N <= 0 || C <= 0 || HW <= 0 || !x || !gamma || !mean || !rstd || !gy || !gx) return HC_ERR_INVALID_ARG;
    size_t need = 0;
    hc_pointwise_workspace_size(N, C, HW, &need);
    const bool want_p = ggamma || gbeta;
    if (want_p && (ws_bytes < need || !ws || !al16(ws))) return HC_ERR_WORKSPACE;
    const size_t smem = sizeof(float) * (size_t)2 * C * LN_PITCH;
    if (smem > 200 * 1024) return HC_ERR_UNSUPPORTED;
    static std::atomic<unsigned long long> attr{0};
    once_per_device(attr, [&] {
        return cudaFuncSetAttribute(ln_bwd_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024) == cudaSuccess;
    });
    cudaStream_t st = (cudaStream_t)stream;
    const long long bpi = (HW + LN_PIX - 1) / LN_PIX;
    const long long blocks = N * bpi;
    float* part = want_p ? (float*)ws : nullptr;
    long long rows = blocks;  // partial rows: one per block
    if (C == 16 * LN_G && (long long)C * HW < (1LL << 31) && blocks < (1LL << 31)) {
        // persistent, two blocks per SM, one partial row per block
        const long long g = 2LL * device_sm_count();
        rows = blocks < g ? blocks : g;
        ln_bwd_reg_kernel<16><<<(unsigned)rows, LN_THREADS, 0, st>>>(x, gamma, mean, rstd, gy, gx, part, (int)HW,
                                                                    (int)bpi, (int)blocks);
    } else {
        ln_bwd_kernel<<<(unsigned)blocks, LN_THREADS, smem, st>>>(x, gamma, mean, rstd, gy, gx, part, C, HW, bpi);
    }
    hc_status s = launched("ln_bwd_kernel", st);
    if (s || !want_p) return s;
    // part is [rows][2][C]: summed over rows in row order
    float* tmp = part + (size_t)blocks * 2 * C;
    if (ggamma && (s = launch_column_sum(part, ggamma, (int)rows, C, 2 * (long long)C, tmp, st))) return s;
    if (gbeta && (s = launch_column_sum(part + C, gbeta, (int)rows, C, 2 * (long long)C, tmp, st))) return s;
    return HC_OK;
}

hc_status hc_gelu_fwd(long long n, const float* x, float* y, void* stream) {
    traced_begin((cudaStream_t)stream);
    if (n <= 0 || !x || !y || !al16(x) || !al16(y)) return HC_ERR_INVALID_ARG;
    gelu_fwd_kernel<<<grid_elems(n), 256, 0, (cudaStream_t)stream>>>(x, y, n);
    return launched("gelu_fwd_kernel", (cudaStream_t)stream);
}

hc_status hc_gelu_bwd(long long n, const float* x, const float* gy, float* gx, void* stream) {
    traced_begin((cudaStream_t)stream);
    if (n <= 0 || !x || !gy || !gx || !al16(x) || !al16(gy) || !al16(gx)) return HC_ERR_INVALID_ARG;
    gelu_bwd_kernel<<<grid_elems(n), 256, 0, (cudaStream_t)stream>>>(x, gy, gx, n);
    return launched("gelu_bwd_kernel", (cudaStream_t)stream);
}

hc_status hc_add_inplace(long long n, float* y, const float* x, void* stream) {
    traced_begin((cudaStream_t)stream);
    if (n <= 0 || !x || !y || !al16(x) || !al16(y)) return HC_ERR_INVALID_ARG;
    add_inplace_kernel<<<grid_elems(n), 256, 0, (cudaStream_t)stream>>>(y, x, n);
    return launched("add_inplace_kernel", (cudaStream_t)stream);
}

hc_status hc_drop_path_mask(int N, float drop_prob, unsigned long long seed, unsigned long long offset, float* mask,
                            void* stream) {
    traced_begin((cudaStream_t)stream);
    if (N <= 0 || !mask || !(drop_prob >= 0.0f) || !(drop_prob < 1.0f)) return HC_ERR_INVALID_ARG;
    const unsigned t = (unsigned)floor((double)drop_prob * 16777216.0);
    const float scale = 1.0f / (1.0f - drop_prob);
    drop_path_mask_kernel<<<(N + 255) / 256 < 1024 ? (N + 255) / 256 : 1024, 256, 0, (cudaStream_t)stream>>>(
        N, t, scale, seed, offset, mask);
    return launched("drop_path_mask_kernel", (cudaStream_t)stream);
}
hc_status hc_layerscale_droppath_fwd(int N, int C, long long HW, const float* res, const float* branch,
                                     const float* gamma, const float* mask, float* out, void* stream) {
    traced_begin((cudaStream_t)stream);
    if (N <= 0 || C <= 0 || HW <= 0 || !res || !branch || !gamma || !out) return HC_ERR_INVALID_ARG;
    ls_fwd_kernel<<<(unsigned)((long long)N * C * LS_CHUNKS), 256, 0, (cudaStream_t)stream>>>(res, branch, gamma, mask,
                                                                                            out, C, HW, LS_CHUNKS);
    return launched("ls_fwd_kernel", (cudaStream_t)stream);
}
hc_status hc_layerscale_residual_fwd(int N, int C, long long HW, const float* res, const float* branch,
                                     const float* gamma, float* out, void* stream) {
    return hc_layerscale_droppath_fwd(N, C, HW, res, branch, gamma, nullptr, out, stream);
}
hc_status hc_layerscale_droppath_bwd(int N, int C, long long HW, const float* branch, const float* gamma,
                                     const float* mask, const float* gy, float* gbranch, float* ggamma, void* ws,
                                     size_t ws_bytes, void* stream) {
    traced_begin((cudaStream_t)stream);
    if (N <= 0 || C <= 0 || HW <= 0 || !branch || !gamma || !gy || !ggamma) return HC_ERR_INVALID_ARG;
    size_t need = 0;
    hc_pointwise_workspace_size(N, C, HW, &need);
    if (ws_bytes < need || !ws || !al16(ws)) return HC_ERR_WORKSPACE;
    cudaStream_t st = (cudaStream_t)stream;
    float* part = (float*)ws;
    ls_bwd_kernel<<<(unsigned)((long long)N * C * LS_CHUNKS), 256, 0, st>>>(branch, gamma, mask, gy, gbranch, part, C,
                                                                          HW, LS_CHUNKS);
    hc_status s = launched("ls_bwd_kernel", st);
    if (s) return s;
    ls_reduce_kernel<<<(C + 127) / 128, 128, 0, st>>>(part, ggamma, N, C, LS_CHUNKS);
    return launched("ls_reduce_kernel", st);
}
hc_status hc_layerscale_residual_bwd(int N, int C, long long HW, const float* branch, const float* gamma,
                                     const float* gy, float* gbranch, float* ggamma, void* ws, size_t ws_bytes,
                                     void* stream) {
    return hc_layerscale_droppath_bwd(N, C, HW, branch, gamma, nullptr, gy, gbranch, ggamma, ws, ws_bytes, stream);
}

}  // extern "C"
