// dw.cu -- depthwise K x K convolution (groups = C, stride 1, padding (K-1)/2),
// the ConvNeXt depthwise layer the pages single out for the halo exchange
// (kwkr.cn news/18980 sections 3.2 and 6.2).
//
// Tiling.  A CTA owns one (n, c) plane and one 128-column tile of it; tiles
// never straddle a shard, so a tile at a shard edge takes its halo columns
// from the neighbouring shard's block (the halo exchange of NVIDIA blog
// "Perception model training for autonomous vehicles with tensor
// parallelism", Figure 1), and zeros past the image edge.  The CTA walks down
// the plane in 32-row tiles; each tile plus its halo (32 + K - 1 rows,
// 128 + 8 columns) is staged in shared memory with cp.async, double buffered
// so the next tile streams in while the current one is computed.  Only the
// owned 128 columns are written (the crop).
//
// Each thread computes an 8-row x 4-column block: per input row it reads 12
// floats (three 16-byte shared loads) and issues up to 7 * 4 * K FMAs with the
// plane's K*K weights held in registers.
//
// Backward (one kernel): warps 0-3 compute grad_input (the same stencil over
// the grad_output tile with the kernel flipped); warps 4-7 accumulate the
// weight and bias gradients of the tile's own grad_output elements against
// the input tile, keep them in registers over all the CTA's row tiles, and
// finally reduce them across the four warps (warp shuffles, then a fixed-order
// sum of the per-warp values) into one partial per (shard, c, tile, n).  A
// second kernel sums those partials in a fixed order into the per-shard
// _Partial gradients.
#include "common.cuh"

namespace hc {
namespace {

constexpr int TW = 128;       // tile width (columns)
constexpr int TH = 32;        // tile height (rows)
constexpr int SMW = TW + 8;   // staged row: 4 halo columns on each side
constexpr int FWD_THREADS = 128;
constexpr int BWD_THREADS = 256;

template <int K>
struct Geo {
    static constexpr int P = (K - 1) / 2;
    static constexpr int R = TH + 2 * P;       // staged rows
    static constexpr int TILE = R * SMW;       // floats per staged tile
};

__device__ __forceinline__ void cp_async16(float* smem, const float* gmem, bool valid) {
    const unsigned sa = (unsigned)__cvta_generic_to_shared(smem);
    const int n = valid ? 16 : 0;  // 0 source bytes: the 16 bytes are zero-filled
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(sa), "l"(gmem), "r"(n) : "memory");
}
// A load the compiler cannot repeat later: keeps the K*K weights resident in
// registers instead of re-fetching them inside the unrolled stencil.
__device__ __forceinline__ float ld_keep(const float* p) {
    float v;
    asm volatile("ld.global.nc.f32 %0, [%1];\n" : "=f"(v) : "l"(p));
    return v;
}

__device__ __forceinline__ void bar_all() { asm volatile("bar.sync 0, %0;\n" ::"n"(256) : "memory"); }

__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait1() { asm volatile("cp.async.wait_group 1;\n" ::: "memory"); }

// Stage rows [h0 - P, h0 + TH + P) and columns [c0 - 4, c0 + TW + 4) of one
// plane; everything outside the image is zero.  W is a multiple of 4 and c0 of
// 128, so every 16-byte piece is either fully inside or fully outside.
template <int K>
__device__ __forceinline__ void stage_tile(float* sm, const float* plane, int H, int W, int h0, int c0, int tid,
                                           int nthr) {
    constexpr int P = Geo<K>::P, R = Geo<K>::R, V = SMW / 4;
    for (int q = tid; q < R * V; q += nthr) {
        const int rr = q / V, cc = q - rr * V;
        const int h = h0 - P + rr, c = c0 - 4 + 4 * cc;
        const bool ok = h >= 0 && h < H && c >= 0 && c < W;
        cp_async16(sm + rr * SMW + 4 * cc, ok ? plane + (long long)h * W + c : plane, ok);
    }
}

// acc[r][jj] += sum_{u,v} wt[u][v] * tile[row0 + r + u][4*lane + jj + v - P + 4]
template <int K>
__device__ __forceinline__ void stencil_8x4(const float* sm, int row0, int lane, const float (&wt)[K][K],
                                            float (&acc)[8][4]) {
    constexpr int P = Geo<K>::P;
#pragma unroll
    for (int i = 0; i < 8 + 2 * P; i++) {
        const float4* rp = reinterpret_cast<const float4*>(sm + (row0 + i) * SMW + 4 * lane);
        const float4 a = rp[0], b = rp[1], c = rp[2];
        const float xs[12] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w, c.x, c.y, c.z, c.w};
#pragma unroll
        for (int r = 0; r < 8; r++) {
            const int u = i - r;
            if (u >= 0 && u < K) {
#pragma unroll
                for (int jj = 0; jj < 4; jj++)
#pragma unroll
                    for (int v = 0; v < K; v++) acc[r][jj] = fmaf(wt[u][v], xs[jj + v - P + 4], acc[r][jj]);
            }
        }
    }
}

template <int K>
__global__ void __launch_bounds__(FWD_THREADS, 4) dw_fwd_kernel(const float* __restrict__ x, const float* __restrict__ w,
                                                             const float* __restrict__ bias, float* __restrict__ y,
                                                             int C, int H, int W, int col_tiles) {
    extern __shared__ __align__(16) float smem[];
    constexpr int TILE = Geo<K>::TILE;
    const int plane = blockIdx.x / col_tiles;
    const int c0 = (blockIdx.x - plane * col_tiles) * TW;
    const int c = plane % C;
    const float* xp = x + (long long)plane * H * W;
    float* yp = y + (long long)plane * H * W;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    float wt[K][K];
#pragma unroll
    for (int u = 0; u < K; u++)
#pragma unroll
        for (int v = 0; v < K; v++) wt[u][v] = ld_keep(w + (c * K + u) * K + v);
    const float bv = bias ? __ldg(bias + c) : 0.0f;

    const int ntiles = (H + TH - 1) / TH;
    stage_tile<K>(smem, xp, H, W, 0, c0, tid, FWD_THREADS);
    cp_async_commit();
    for (int t = 0; t < ntiles; t++) {
        if (t + 1 < ntiles) stage_tile<K>(smem + ((t + 1) & 1) * TILE, xp, H, W, (t + 1) * TH, c0, tid, FWD_THREADS);
        cp_async_commit();
        cp_async_wait1();
        __syncthreads();
        const float* sm = smem + (t & 1) * TILE;
        float acc[8][4];
#pragma unroll
        for (int r = 0; r < 8; r++)
#pragma unroll
            for (int jj = 0; jj < 4; jj++) acc[r][jj] = bv;
        stencil_8x4<K>(sm, warp * 8, lane, wt, acc);
#pragma unroll
        for (int r = 0; r < 8; r++) {
            const int h = t * TH + warp * 8 + r;
            if (h < H)
                *reinterpret_cast<float4*>(yp + (long long)h * W + c0 + 4 * lane) =
                    make_float4(acc[r][0], acc[r][1], acc[r][2], acc[r][3]);
        }
        __syncthreads();  // the buffer just read is refilled by the next iteration's prefetch
    }
}

struct BwdArgs {
    const float* x;
    const float* w;
    const float* gy;
    float* gx;
    float* tile_part;
    int N, C, H, W, col_tiles, tiles_per_shard, want_wb;
};

// Both roles run the same staging loop (every thread stages its share of
// both tiles) and meet at the same CTA-wide barriers.
template <int K>
__device__ __forceinline__ void bwd_stage(const BwdArgs& a, float* smem, const float* gp, const float* xp, int t,
                                          int s, int c0) {
    constexpr int TILE = Geo<K>::TILE;
    stage_tile<K>(smem + 2 * s * TILE, gp, a.H, a.W, t * TH, c0, threadIdx.x, BWD_THREADS);
    if (a.want_wb) stage_tile<K>(smem + (2 * s + 1) * TILE, xp, a.H, a.W, t * TH, c0, threadIdx.x, BWD_THREADS);
}

// Warps 0-3: grad_input of the tile = the stencil over the grad_output tile
// with the kernel flipped (gx[h][c] = sum_{u,v} w[K-1-u][K-1-v] gy[h+u-P][c+v-P]).
template <int K>
__device__ __forceinline__ void bwd_gx_role(const BwdArgs& a, float* smem, int plane, int c, int c0) {
    constexpr int TILE = Geo<K>::TILE;
    const float* gp = a.gy + (long long)plane * a.H * a.W;
    const float* xp = a.x + (long long)plane * a.H * a.W;
    float* gxp = a.gx ? a.gx + (long long)plane * a.H * a.W : nullptr;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    float wf[K][K];
#pragma unroll
    for (int u = 0; u < K; u++)
#pragma unroll
        for (int v = 0; v < K; v++) wf[u][v] = ld_keep(a.w + (c * K + (K - 1 - u)) * K + (K - 1 - v));
    const int ntiles = (a.H + TH - 1) / TH;
    bwd_stage<K>(a, smem, gp, xp, 0, 0, c0);
    cp_async_commit();
    for (int t = 0; t < ntiles; t++) {
        if (t + 1 < ntiles) bwd_stage<K>(a, smem, gp, xp, t + 1, (t + 1) & 1, c0);
        cp_async_commit();
        cp_async_wait1();
        bar_all();
        if (gxp) {
            const float* gys = smem + 2 * (t & 1) * TILE;
            float acc[8][4];
#pragma unroll
            for (int r = 0; r < 8; r++)
#pragma unroll
                for (int jj = 0; jj < 4; jj++) acc[r][jj] = 0.0f;
            stencil_8x4<K>(gys, warp * 8, lane, wf, acc);
#pragma unroll
            for (int r = 0; r < 8; r++) {
                const int h = t * TH + warp * 8 + r;
                if (h < a.H)
                    *reinterpret_cast<float4*>(gxp + (long long)h * a.W + c0 + 4 * lane) =
                        make_float4(acc[r][0], acc[r][1], acc[r][2], acc[r][3]);
            }
        }
        bar_all();
    }
}

// Warps 4-7: weight and bias gradients of the tile's own grad_output block,
// gw[u][v] += gy[h][c] * x[h+u-P][c+v-P], kept in registers over all row
// tiles, then reduced across the four warps into one partial.
template <int K>
__device__ __forceinline__ void bwd_gw_role(const BwdArgs& a, float* smem, int plane, int n, int c, int ct, int c0) {
    constexpr int P = Geo<K>::P, TILE = Geo<K>::TILE, KK = K * K;
    const float* gp = a.gy + (long long)plane * a.H * a.W;
    const float* xp = a.x + (long long)plane * a.H * a.W;
    const int wq = (threadIdx.x >> 5) - 4, lane = threadIdx.x & 31;
    float gw[K][K];
#pragma unroll
    for (int u = 0; u < K; u++)
#pragma unroll
        for (int v = 0; v < K; v++) gw[u][v] = 0.0f;
    float gbs = 0.0f;
    const int ntiles = (a.H + TH - 1) / TH;
    bwd_stage<K>(a, smem, gp, xp, 0, 0, c0);
    cp_async_commit();
    for (int t = 0; t < ntiles; t++) {
        if (t + 1 < ntiles) bwd_stage<K>(a, smem, gp, xp, t + 1, (t + 1) & 1, c0);
        cp_async_commit();
        cp_async_wait1();
        bar_all();
        if (a.want_wb) {
            const float* gys = smem + 2 * (t & 1) * TILE;
            const float* xs_t = gys + TILE;
            // own grad_output block: tile rows wq*8 .. wq*8+7, columns 4*lane .. 4*lane+3
            float g[8][4];
#pragma unroll
            for (int r = 0; r < 8; r++) {
                const float4 q = *reinterpret_cast<const float4*>(gys + (P + wq * 8 + r) * SMW + 4 + 4 * lane);
                g[r][0] = q.x;
                g[r][1] = q.y;
                g[r][2] = q.z;
                g[r][3] = q.w;
                gbs += (q.x + q.y) + (q.z + q.w);
            }
#pragma unroll
            for (int i = 0; i < 8 + 2 * P; i++) {
                const float4* rp = reinterpret_cast<const float4*>(xs_t + (wq * 8 + i) * SMW + 4 * lane);
                const float4 p0 = rp[0], p1 = rp[1], p2 = rp[2];
                const float xr[12] = {p0.x, p0.y, p0.z, p0.w, p1.x, p1.y, p1.z, p1.w, p2.x, p2.y, p2.z, p2.w};
#pragma unroll
                for (int r = 0; r < 8; r++) {
                    const int u = i - r;
                    if (u >= 0 && u < K) {
#pragma unroll
                        for (int jj = 0; jj < 4; jj++)
#pragma unroll
                            for (int v = 0; v < K; v++) gw[u][v] = fmaf(g[r][jj], xr[jj + v - P + 4], gw[u][v]);
                    }
                }
            }
        }
        bar_all();
    }
    if (!a.want_wb) return;
    // shuffle tree inside each warp, then the four warp sums in warp order
    float* red = smem;  // [4][KK + 1]; every staged tile has been consumed
#pragma unroll
    for (int u = 0; u < K; u++)
#pragma unroll
        for (int v = 0; v < K; v++) {
            float s = gw[u][v];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
            if (lane == 0) red[wq * (KK + 1) + u * K + v] = s;
        }
    {
        float s = gbs;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
        if (lane == 0) red[wq * (KK + 1) + KK] = s;
    }
    asm volatile("bar.sync 1, 128;\n" ::: "memory");  // the four weight-role warps only
    const int k = threadIdx.x - 128;
    if (k <= KK) {
        const float s = ((red[k] + red[(KK + 1) + k]) + red[2 * (KK + 1) + k]) + red[3 * (KK + 1) + k];
        const int r = ct / a.tiles_per_shard, tt = ct - r * a.tiles_per_shard;
        a.tile_part[((((long long)r * a.C + c) * a.tiles_per_shard + tt) * a.N + n) * (KK + 1) + k] = s;
    }
}

template <int K>
__global__ void __launch_bounds__(BWD_THREADS, 2) dw_bwd_kernel(BwdArgs a) {
    extern __shared__ __align__(16) float smem[];
    const int plane = blockIdx.x / a.col_tiles;
    const int ct = blockIdx.x - plane * a.col_tiles;
    const int n = plane / a.C, c = plane - n * a.C;
    if (threadIdx.x < 128)
        bwd_gx_role<K>(a, smem, plane, c, ct * TW);
    else
        bwd_gw_role<K>(a, smem, plane, n, c, ct, ct * TW);
}

// Shard partials: gwp[r][c][k] = sum over (tile tt, image n) of the tile
// partials, tt then n ascending; gbp[r][c] likewise from the last slot.
__global__ void dw_shard_partials_kernel(const float* __restrict__ tile_part, float* __restrict__ gwp,
                                         float* __restrict__ gbp, int S, int C, int rows, int KK) {
    const long long total = (long long)S * C * (KK + 1);
    for (long long q = blockIdx.x * (long long)blockDim.x + threadIdx.x; q < total;
         q += (long long)gridDim.x * blockDim.x) {
        const int k = (int)(q % (KK + 1));
        const long long rc = q / (KK + 1);  // r * C + c
        const float* src = tile_part + rc * rows * (KK + 1) + k;
        float s = 0.0f;
        for (int m = 0; m < rows; m++) s += src[(long long)m * (KK + 1)];
        if (k < KK) {
            if (gwp) gwp[rc * KK + k] = s;
        } else if (gbp) {
            gbp[rc] = s;
        }
    }
}

int ksize(const hc_conv_desc* d) { return d->kh; }

template <int K>
hc_status fwd_k(const hc_conv_desc* d, const float* x, const float* w, const float* b, float* y, cudaStream_t st) {
    const int col_tiles = d->W / TW;
    const long long blocks = (long long)d->N * d->C_in * col_tiles;
    const size_t smem = 2 * sizeof(float) * Geo<K>::TILE;
    static bool attr = false;
    if (!attr) {
        cudaFuncSetAttribute(dw_fwd_kernel<K>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        attr = true;
    }
    dw_fwd_kernel<K><<<(unsigned)blocks, FWD_THREADS, smem, st>>>(x, w, b, y, d->C_in, d->H, d->W, col_tiles);
    return launched();
}

template <int K>
hc_status bwd_k(const hc_conv_desc* d, const Plan& p, const float* x, const float* w, const float* gy, float* gx,
                float* tile_part, float* gwp, float* gbp, bool want_wb, cudaStream_t st) {
    const int col_tiles = d->W / TW, tps = p.Wl / TW;
    const long long blocks = (long long)d->N * d->C_in * col_tiles;
    const size_t smem = 4 * sizeof(float) * Geo<K>::TILE;
    static bool attr = false;
    if (!attr) {
        cudaFuncSetAttribute(dw_bwd_kernel<K>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        attr = true;
    }
    if (!gx && !want_wb) return HC_OK;
    BwdArgs a{x, w, gy, gx, tile_part, d->N, d->C_in, d->H, d->W, col_tiles, tps, want_wb ? 1 : 0};
    dw_bwd_kernel<K><<<(unsigned)blocks, BWD_THREADS, smem, st>>>(a);
    hc_status s = launched();
    if (s || !want_wb) return s;
    const long long total = (long long)p.S * d->C_in * (K * K + 1);
    const unsigned grid = (unsigned)((total + 255) / 256);
    dw_shard_partials_kernel<<<grid, 256, 0, st>>>(tile_part, gwp, gbp, p.S, d->C_in, tps * d->N, K * K);
    return launched();
}

}  // namespace

bool depthwise_supported(const hc_conv_desc* d, const Plan& p) {
    const int K = d->kh;
    return d->groups == d->C_in && d->C_out == d->C_in && d->kh == d->kw && (K == 3 || K == 5 || K == 7) &&
           d->stride == 1 && d->padding == (K - 1) / 2 && p.Wl % TW == 0 &&
           (long long)d->N * d->C_in * (d->W / TW) < (1LL << 31);
}

size_t depthwise_bwd_ws_floats(const hc_conv_desc* d, const Plan& p) {
    const int K = ksize(d);
    return (size_t)p.S * d->C_in * (p.Wl / TW) * d->N * (K * K + 1);
}

hc_status launch_depthwise_fwd(const hc_conv_desc* d, const Plan& p, const float* x, const float* w,
                               const float* b, float* y, cudaStream_t st) {
    (void)p;
    switch (ksize(d)) {
        case 3: return fwd_k<3>(d, x, w, b, y, st);
        case 5: return fwd_k<5>(d, x, w, b, y, st);
        case 7: return fwd_k<7>(d, x, w, b, y, st);
    }
    return HC_ERR_UNSUPPORTED;
}

hc_status launch_depthwise_bwd(const hc_conv_desc* d, const Plan& p, const float* x, const float* w,
                               const float* gy, float* gx, float* tile_part, float* gwp, float* gbp,
                               bool want_weight_grads, cudaStream_t st) {
    switch (ksize(d)) {
        case 3: return bwd_k<3>(d, p, x, w, gy, gx, tile_part, gwp, gbp, want_weight_grads, st);
        case 5: return bwd_k<5>(d, p, x, w, gy, gx, tile_part, gwp, gbp, want_weight_grads, st);
        case 7: return bwd_k<7>(d, p, x, w, gy, gx, tile_part, gwp, gbp, want_weight_grads, st);
    }
    return HC_ERR_UNSUPPORTED;
}

}  // namespace hc
