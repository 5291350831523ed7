// direct.cu -- plain direct convolution for any groups, stride and padding:
// the general path the specialised kernels are measured against, and the one
// used for layouts they do not cover.
//
// Sharding (NVIDIA blog "Perception model training for autonomous vehicles
// with tensor parallelism", design section; kwkr.cn news/18980 section 2.2):
// an output column owned by shard r reads its halo columns directly from the
// neighbouring shards' blocks of x (zeros past the image edge); the weight and
// bias gradients are produced per shard (_Partial) over the shard's own output
// rows and columns (row x column shard grid) and summed afterwards in shard
// order.
#include "common.cuh"

namespace hc {
namespace {

struct ConvDims {
    int N, Ci, H, W, Co, kh, kw, s, p, Cgi, Cgo, Ho, Wo;
};

ConvDims dims_of(const hc_conv_desc* d, const Plan& pl) {
    return ConvDims{d->N, d->C_in, d->H, d->W, d->C_out, d->kh, d->kw, d->stride, d->padding,
                    d->C_in / d->groups, d->C_out / d->groups, pl.Ho, pl.Wo};
}

unsigned grid_for(long long n, int threads) {
    const long long b = (n + threads - 1) / threads;
    return (unsigned)(b < 152LL * 32 ? b : 152LL * 32);
}

// y[n,co,i,j] = b[co] + sum_{ci',u,v} w[co,ci',u,v] * x[n,ci,i*s-p+u,j*s-p+v]
__global__ void direct_fwd_kernel(const float* __restrict__ x, const float* __restrict__ w,
                                  const float* __restrict__ b, float* __restrict__ y, ConvDims D) {
    const long long total = (long long)D.N * D.Co * D.Ho * D.Wo;
    for (long long q = blockIdx.x * (long long)blockDim.x + threadIdx.x; q < total;
         q += (long long)gridDim.x * blockDim.x) {
        const int j = (int)(q % D.Wo);
        const int i = (int)((q / D.Wo) % D.Ho);
        const int co = (int)((q / ((long long)D.Wo * D.Ho)) % D.Co);
        const int n = (int)(q / ((long long)D.Wo * D.Ho * D.Co));
        const int ci0 = (co / D.Cgo) * D.Cgi;
        float acc = b ? __ldg(b + co) : 0.0f;
        for (int cl = 0; cl < D.Cgi; cl++) {
            const float* xp = x + ((long long)n * D.Ci + ci0 + cl) * D.H * D.W;
            const float* wp = w + ((long long)co * D.Cgi + cl) * D.kh * D.kw;
            for (int u = 0; u < D.kh; u++) {
                const int h = i * D.s - D.p + u;
                if (h < 0 || h >= D.H) continue;
                for (int v = 0; v < D.kw; v++) {
                    const int c = j * D.s - D.p + v;
                    if (c < 0 || c >= D.W) continue;
                    acc = fmaf(__ldg(wp + u * D.kw + v), __ldg(xp + (long long)h * D.W + c), acc);
                }
            }
        }
        y[q] = acc;
    }
}

// gx[n,ci,h,c] = sum over (co in the group, u, v) with (h+p-u) and (c+p-v)
// divisible by s of w[co,ci',u,v] * gy[n,co,(h+p-u)/s,(c+p-v)/s]
__global__ void direct_gx_kernel(const float* __restrict__ w, const float* __restrict__ gy, float* __restrict__ gx,
                                 ConvDims D) {
    const long long total = (long long)D.N * D.Ci * D.H * D.W;
    for (long long q = blockIdx.x * (long long)blockDim.x + threadIdx.x; q < total;
         q += (long long)gridDim.x * blockDim.x) {
        const int c = (int)(q % D.W);
        const int h = (int)((q / D.W) % D.H);
        const int ci = (int)((q / ((long long)D.W * D.H)) % D.Ci);
        const int n = (int)(q / ((long long)D.W * D.H * D.Ci));
        const int g = ci / D.Cgi, cl = ci % D.Cgi;
        float acc = 0.0f;
        for (int co = g * D.Cgo; co < (g + 1) * D.Cgo; co++) {
            const float* gp = gy + ((long long)n * D.Co + co) * D.Ho * D.Wo;
            const float* wp = w + ((long long)co * D.Cgi + cl) * D.kh * D.kw;
            for (int u = 0; u < D.kh; u++) {
                const int ti = h + D.p - u;
                if (ti < 0 || ti % D.s) continue;
                const int i = ti / D.s;
                if (i >= D.Ho) continue;
                for (int v = 0; v < D.kw; v++) {
                    const int tj = c + D.p - v;
                    if (tj < 0 || tj % D.s) continue;
                    const int j = tj / D.s;
                    if (j >= D.Wo) continue;
                    acc = fmaf(__ldg(wp + u * D.kw + v), __ldg(gp + (long long)i * D.Wo + j), acc);
                }
            }
        }
        gx[q] = acc;
    }
}

// Small problems (a few thousand outputs would leave most SMs idle, each thread
// running a long serial chain): one warp per output element, its lanes taking
// every 32nd term of the sum; a fixed butterfly adds the lanes' sums.
__global__ void direct_fwd_warp_kernel(const float* __restrict__ x, const float* __restrict__ w,
                                       const float* __restrict__ b, float* __restrict__ y, ConvDims D) {
    const long long total = (long long)D.N * D.Co * D.Ho * D.Wo;
    const int lane = threadIdx.x & 31, KK = D.kh * D.kw, R = D.Cgi * KK;
    const long long warps = ((long long)gridDim.x * blockDim.x) >> 5;
    for (long long q = (blockIdx.x * (long long)blockDim.x + threadIdx.x) >> 5; q < total; q += warps) {
        const int j = (int)(q % D.Wo);
        const int i = (int)((q / D.Wo) % D.Ho);
        const int co = (int)((q / ((long long)D.Wo * D.Ho)) % D.Co);
        const int n = (int)(q / ((long long)D.Wo * D.Ho * D.Co));
        const int ci0 = (co / D.Cgo) * D.Cgi;
        float acc = 0.0f;
        for (int r = lane; r < R; r += 32) {  // r = (ci', u, v)
            const int cl = r / KK, uv = r - cl * KK, u = uv / D.kw, v = uv - u * D.kw;
            const int h = i * D.s - D.p + u, c = j * D.s - D.p + v;
            if (h >= 0 && h < D.H && c >= 0 && c < D.W)
                acc = fmaf(__ldg(w + ((long long)co * D.Cgi + cl) * KK + uv),
                           __ldg(x + (((long long)n * D.Ci + ci0 + cl) * D.H + h) * D.W + c), acc);
        }
        for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
        if (lane == 0) y[q] = acc + (b ? __ldg(b + co) : 0.0f);
    }
}

// direct_gx_kernel's sum with a warp per grad_input element (small problems).
__global__ void direct_gx_warp_kernel(const float* __restrict__ w, const float* __restrict__ gy,
                                      float* __restrict__ gx, ConvDims D) {
    const long long total = (long long)D.N * D.Ci * D.H * D.W;
    const int lane = threadIdx.x & 31, KK = D.kh * D.kw, R = D.Cgo * KK;
    const long long warps = ((long long)gridDim.x * blockDim.x) >> 5;
    for (long long q = (blockIdx.x * (long long)blockDim.x + threadIdx.x) >> 5; q < total; q += warps) {
        const int c = (int)(q % D.W);
        const int h = (int)((q / D.W) % D.H);
        const int ci = (int)((q / ((long long)D.W * D.H)) % D.Ci);
        const int n = (int)(q / ((long long)D.W * D.H * D.Ci));
        const int g = ci / D.Cgi, cl = ci % D.Cgi;
        float acc = 0.0f;
        for (int r = lane; r < R; r += 32) {  // r = (co in the group, u, v)
            const int col = r / KK, uv = r - col * KK, u = uv / D.kw, v = uv - u * D.kw;
            const int co = g * D.Cgo + col;
            const int ti = h + D.p - u, tj = c + D.p - v;
            if (ti < 0 || tj < 0 || ti % D.s || tj % D.s) continue;
            const int i = ti / D.s, j = tj / D.s;
            if (i >= D.Ho || j >= D.Wo) continue;
            acc = fmaf(__ldg(w + ((long long)co * D.Cgi + cl) * KK + uv),
                       __ldg(gy + (((long long)n * D.Co + co) * D.Ho + i) * D.Wo + j), acc);
        }
        for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
        if (lane == 0) gx[q] = acc;
    }
}

// Outputs below which a warp per output is used: about four 256-thread blocks per SM.
constexpr long long kWarpPerOutput = 152LL * 4 * 256;

// Fixed-order block reduction: warp shuffle tree, then warp 0 adds the
// per-warp sums in warp order.  Result valid in thread 0.
__device__ float block_sum(float v, float* red) {
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane == 0) red[warp] = v;
    __syncthreads();
    float t = 0.0f;
    if (threadIdx.x == 0)
        for (int k = 0; k < (int)(blockDim.x >> 5); k++) t += red[k];
    __syncthreads();
    return t;
}

// One block per (weight element, shard): the shard's _Partial gradient
//   gw_part[r, co, ci', u, v] = sum_{n, i, j in own(r)} gy[n,co,i,j] * x[n,ci,i*s-p+u,j*s-p+v]
// Grid shard q = a * S + b: output rows [a*own_h, ...) (the last row shard up to
// Ho) and columns [b*own_w, ...) (the last column shard up to Wo).
struct ShardBox {
    int S, Sh, own_w, own_h;
    __device__ __forceinline__ void of(int q, const ConvDims& D, int& i0, int& i1, int& j0, int& j1) const {
        const int a = q / S, b = q - a * S;
        i0 = a * own_h;
        i1 = (a == Sh - 1) ? D.Ho : i0 + own_h;
        j0 = b * own_w;
        j1 = (b == S - 1) ? D.Wo : j0 + own_w;
        if (i1 < i0) i1 = i0;
        if (j1 < j0) j1 = j0;
    }
};

// One block per weight element (blocks [0, nw)) or output channel (blocks
// [nw, nw + nb)), walking the grid shards q = 0 .. Q-1 in order:
//   gw_part[q, co, ci', u, v] = sum_{n, i, j owned by q} gy[n,co,i,j] * x[n,ci,i*s-p+u,j*s-p+v]
//   gb_part[q, co]            = sum_{n, i, j owned by q} gy[n,co,i,j]
// and, when gw / gb are given, the full gradient: the shard partials added from
// q = 0 up (the order of the library's shard sum).
__global__ void direct_partials_kernel(const float* __restrict__ x, const float* __restrict__ gy,
                                       float* __restrict__ gw_part, float* __restrict__ gb_part,
                                       float* __restrict__ gw, float* __restrict__ gb, ConvDims D, long long wsz,
                                       long long nw, int Q, ShardBox sb) {
    __shared__ float red[32];
    const bool weight = blockIdx.x < nw;
    const long long k = weight ? (long long)blockIdx.x : 0;
    const int v = (int)(k % D.kw);
    const int u = (int)((k / D.kw) % D.kh);
    const int cl = (int)((k / ((long long)D.kw * D.kh)) % D.Cgi);
    const int co = weight ? (int)(k / ((long long)D.kw * D.kh * D.Cgi)) : (int)(blockIdx.x - nw);
    const int ci = (co / D.Cgo) * D.Cgi + cl;
    float total = 0.0f;
    for (int q = 0; q < Q; q++) {
        int i0, i1, j0, j1;
        sb.of(q, D, i0, i1, j0, j1);
        const int nj = j1 - j0, ni = i1 - i0;
        const long long terms = (long long)D.N * ni * nj;
        float acc = 0.0f;
        for (long long t = threadIdx.x; t < terms; t += blockDim.x) {
            const int j = j0 + (int)(t % nj);
            const int i = i0 + (int)((t / nj) % ni);
            const int n = (int)(t / ((long long)nj * ni));
            const float g = __ldg(gy + (((long long)n * D.Co + co) * D.Ho + i) * D.Wo + j);
            if (!weight) {
                acc += g;
                continue;
            }
            const int h = i * D.s - D.p + u, c = j * D.s - D.p + v;
            if (h < 0 || h >= D.H || c < 0 || c >= D.W) continue;
            acc = fmaf(g, __ldg(x + (((long long)n * D.Ci + ci) * D.H + h) * D.W + c), acc);
        }
        const float t = block_sum(acc, red);
        if (threadIdx.x == 0) {
            if (weight)
                gw_part[(long long)q * wsz + k] = t;
            else
                gb_part[(long long)q * D.Co + co] = t;
            total += t;
        }
    }
    if (threadIdx.x == 0) {
        if (weight && gw) gw[k] = total;
        if (!weight && gb) gb[co] = total;
    }
}

}  // namespace

hc_status launch_direct_fwd(const hc_conv_desc* d, const Plan& p, const float* x, const float* w, const float* b,
                            float* y, cudaStream_t st) {
    const ConvDims D = dims_of(d, p);
    const long long total = (long long)D.N * D.Co * D.Ho * D.Wo;
    if (total < kWarpPerOutput)
        direct_fwd_warp_kernel<<<grid_for(total * 32, 256), 256, 0, st>>>(x, w, b, y, D);
    else
        direct_fwd_kernel<<<grid_for(total, 256), 256, 0, st>>>(x, w, b, y, D);
    return launched("direct_fwd_kernel", st);
}

hc_status launch_direct_gx(const hc_conv_desc* d, const Plan& p, const float* w, const float* gy, float* gx,
                           cudaStream_t st) {
    const ConvDims D = dims_of(d, p);
    const long long total = (long long)D.N * D.Ci * D.H * D.W;
    if (total < kWarpPerOutput)
        direct_gx_warp_kernel<<<grid_for(total * 32, 256), 256, 0, st>>>(w, gy, gx, D);
    else
        direct_gx_kernel<<<grid_for(total, 256), 256, 0, st>>>(w, gy, gx, D);
    return launched("direct_gx_kernel", st);
}

hc_status launch_direct_partials(const hc_conv_desc* d, const Plan& p, const float* x, const float* gy,
                                 float* gw_part, float* gb_part, cudaStream_t st, float* gw, float* gb) {
    const ConvDims D = dims_of(d, p);
    const long long wsz = (long long)D.Co * D.Cgi * D.kh * D.kw;
    const ShardBox sb{p.S, p.Sh, p.Wl / d->stride, p.Hlo};
    const long long nw = gw_part ? wsz : 0, nb = gb_part ? D.Co : 0;
    if (nw + nb == 0) return HC_OK;
    if (nw + nb > 0x7fffffffLL) return HC_ERR_UNSUPPORTED;
    direct_partials_kernel<<<(unsigned)(nw + nb), 256, 0, st>>>(x, gy, gw_part, gb_part, gw_part ? gw : nullptr,
                                                               gb_part ? gb : nullptr, D, wsz, nw, p.Q, sb);
    return launched("direct_partials_kernel", st);
}

}  // namespace hc
